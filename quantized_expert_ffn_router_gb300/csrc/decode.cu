// decode.cu -- quantized SwiGLU experts for decode: y = down(silu(gate.x) *
// up.x), int4 (group-scaled) and NVFP4 weights, top-k combine fused.
//
// Sources: "SSD 가중치층으로 35B MoE를 ..." (onedev.kr), "How it works"
// (down(silu(gate(x)) * up(x)) over int4, dedup of the routed experts);
// "NVMe에서 전문가(experts)를 ... 133GB MoE" (molayo1419.me), step 4 (the
// single-token NVFP4 SwiGLU expert kernel built on the hardware e2m1 -> f16x2
// convert); "FreeToken 딥다이브" (fiv.co.kr), design pattern 3 (pairs on the
// host path are masked, each pair computed once).
//
// Two kernels on one stream:
//   gate/up: one CTA per (distinct expert, 16-row block of I).  Each warp owns
//     a row of gate and of up, streams it with 128-bit loads, dequantises in
//     registers, dots it with every token routed to that expert (x staged in
//     shared memory as fp32) and reduces with warp shuffles; h = silu(g)*u
//     goes to the workspace in fp32, one row per (token, rank) pair.
//   down: one CTA per 16-row block of H.  Each warp owns one output row and
//     walks the (distinct expert, 32-element chunk) items of that row, so
//     every expert's down bytes are read once; each token's combine is summed
//     in registers in a fixed order and written once (no atomics).
// Every expert's bytes cross HBM exactly once per call.
#include <cuda_fp16.h>

#include "ft_decode.cuh"

namespace ft {
namespace {

constexpr int kRowsPerCta = 16;  // 8 warps x 2 rows
constexpr int kThreads = 256;
constexpr int kPad = 36;         // floats per 32-element chunk in shared memory (bank spread)
constexpr size_t kSmemLimit = 160 * 1024;

// ------------------------------------------------------------ dequant-dot --
// Dot of one 16-byte chunk (32 codes) with 32 fp32 inputs in shared memory.
// int4: returns sum (q - 8) * x (the group scale is applied by the caller).
__device__ __forceinline__ float dot_int4(const uint4 w, const float* __restrict__ xs) {
  const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float4 xa = *reinterpret_cast<const float4*>(xs + 8 * j);
    const float4 xb = *reinterpret_cast<const float4*>(xs + 8 * j + 4);
    const uint32_t v = wv[j];
    // (0x4B000000 | q) is 2^23 + q exactly; subtracting 2^23 + 8 gives q - 8.
    const float magic = 8388616.0f;
    s0 = fmaf(__uint_as_float(0x4B000000u | (v & 15u)) - magic, xa.x, s0);
    s1 = fmaf(__uint_as_float(0x4B000000u | ((v >> 4) & 15u)) - magic, xa.y, s1);
    s0 = fmaf(__uint_as_float(0x4B000000u | ((v >> 8) & 15u)) - magic, xa.z, s0);
    s1 = fmaf(__uint_as_float(0x4B000000u | ((v >> 12) & 15u)) - magic, xa.w, s1);
    s0 = fmaf(__uint_as_float(0x4B000000u | ((v >> 16) & 15u)) - magic, xb.x, s0);
    s1 = fmaf(__uint_as_float(0x4B000000u | ((v >> 20) & 15u)) - magic, xb.y, s1);
    s0 = fmaf(__uint_as_float(0x4B000000u | ((v >> 24) & 15u)) - magic, xb.z, s0);
    s1 = fmaf(__uint_as_float(0x4B000000u | (v >> 28)) - magic, xb.w, s1);
  }
  return s0 + s1;
}

// Four E2M1 pairs (the bytes of v, low nibble = even element) -> four
// f16x2 via the hardware e2m1x2 -> f16x2 convert (exact: every E2M1 value is
// an f16 value).
__device__ __forceinline__ void e2m1x8_to_h2(uint32_t v, uint32_t h[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(v));
}

__device__ __forceinline__ float2 h2_to_f32(uint32_t h2) {
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}

// E4M3 pair (two bytes, low byte first) -> two fp32 via e4m3x2 -> f16x2.
__device__ __forceinline__ float2 e4m3x2_to_f32(uint32_t two) {
  uint32_t h2;
  const unsigned short b = static_cast<unsigned short>(two);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(b));
  return h2_to_f32(h2);
}

// NVFP4: returns s0 * sum_{i<16} e2m1_i x_i + s1 * sum_{i>=16} e2m1_i x_i,
// s0/s1 the chunk's two E4M3 block scales (packed in `sc`).
__device__ __forceinline__ float dot_nvfp4(const uint4 w, uint32_t sc, const float* __restrict__ xs) {
  const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
  float part[2];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int j = half * 2 + jj;
      const uint32_t v = wv[j];
      const float4 xa = *reinterpret_cast<const float4*>(xs + 8 * j);
      const float4 xb = *reinterpret_cast<const float4*>(xs + 8 * j + 4);
      uint32_t hv[4];
      e2m1x8_to_h2(v, hv);
      const float2 c0 = h2_to_f32(hv[0]);
      const float2 c1 = h2_to_f32(hv[1]);
      const float2 c2 = h2_to_f32(hv[2]);
      const float2 c3 = h2_to_f32(hv[3]);
      s0 = fmaf(c0.x, xa.x, s0);
      s1 = fmaf(c0.y, xa.y, s1);
      s0 = fmaf(c1.x, xa.z, s0);
      s1 = fmaf(c1.y, xa.w, s1);
      s0 = fmaf(c2.x, xb.x, s0);
      s1 = fmaf(c2.y, xb.y, s1);
      s0 = fmaf(c3.x, xb.z, s0);
      s1 = fmaf(c3.y, xb.w, s1);
    }
    part[half] = s0 + s1;
  }
  const float2 s = e4m3x2_to_f32(sc & 0xffffu);
  return fmaf(part[0], s.x, part[1] * s.y);
}

template <int FMT>
__device__ __forceinline__ float chunk_dot(const uint4 w, uint32_t sc, const float* xs) {
  if constexpr (FMT == FT_INT4)
    return dot_int4(w, xs) * __half2float(__ushort_as_half(static_cast<unsigned short>(sc)));
  else
    return dot_nvfp4(w, sc, xs);
}

// Scale word for 32-element chunk c of a row: int4 -> the fp16 group scale;
// NVFP4 -> the two E4M3 block-scale bytes.
template <int FMT>
__device__ __forceinline__ uint32_t load_scale(const uint8_t* srow, int c, int group) {
  if constexpr (FMT == FT_INT4) {
    return __ldg(reinterpret_cast<const unsigned short*>(srow) + (c * 32) / group);
  } else {
    return __ldg(reinterpret_cast<const unsigned short*>(srow) + c);
  }
}

__device__ __forceinline__ float silu(float v) { return v / (1.f + expf(-v)); }

// ------------------------------------------------------------ gate / up ----
template <int FMT, int NT>
__global__ void __launch_bounds__(kThreads) gateup_kernel(DecArgs a) {
  extern __shared__ __align__(16) float xs[];
  __shared__ Groups g;
  build_groups(a, g);
  const int tiles = a.I / kRowsPerCta;
  const int d = blockIdx.x / tiles, rb = blockIdx.x % tiles;
  if (d >= g.nD) return;
  const uint8_t* blk = g.dBlock[d];
  const int p0all = g.dStart[d], npairs = g.dStart[d + 1] - p0all;
  const int HC = a.H / 32;  // 32-element chunks per row
  const int xstride = HC * kPad;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float tsg = 1.f, tsu = 1.f;
  if constexpr (FMT == FT_NVFP4) {
    const int64_t fid = static_cast<int64_t>(a.layer) * a.E + g.dExpert[d];
    tsg = __ldg(a.tscale + 3 * fid + 0);
    tsu = __ldg(a.tscale + 3 * fid + 1);
  }
  const uint64_t srow_bytes = (FMT == FT_INT4) ? static_cast<uint64_t>(a.H / a.group) * 2
                                               : static_cast<uint64_t>(a.H / 16);
  constexpr int kMaxIt = 4;  // H <= 4096
  // The pairs of this expert, NT at a time (more than NT only when one token
  // lists the same expert twice): x of those pairs is staged as fp32.
  for (int c0 = 0; c0 < npairs; c0 += NT) {
    const int p0 = p0all + c0, nt = min(NT, npairs - c0);
    __syncthreads();
    for (int i = threadIdx.x; i < nt * (a.H / 8); i += blockDim.x) {
      const int t = i / (a.H / 8), c8 = i % (a.H / 8);
      const int tok = g.sortedPair[p0 + t] / a.k;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(tok) * a.H) + c8);
      const int kk = c8 * 8;
      float* dst = xs + t * xstride + (kk / 32) * kPad + (kk % 32);
      *reinterpret_cast<float4*>(dst) = make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
      *reinterpret_cast<float4*>(dst + 4) = make_float4(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w));
    }
    __syncthreads();
    for (int rr = 0; rr < 2; ++rr) {
      const int r = rb * kRowsPerCta + warp * 2 + rr;
      const uint8_t* grow = blk + a.off[0] + static_cast<uint64_t>(r) * (a.H / 2);
      const uint8_t* urow = blk + a.off[1] + static_cast<uint64_t>(r) * (a.H / 2);
      const uint8_t* gsrow = blk + a.off[3] + r * srow_bytes;
      const uint8_t* usrow = blk + a.off[4] + r * srow_bytes;
      uint4 wg[kMaxIt], wu[kMaxIt];
      uint32_t sg[kMaxIt], su[kMaxIt];
#pragma unroll
      for (int it = 0; it < kMaxIt; ++it) {
        const int c = lane + 32 * it;
        if (c < HC) {
          wg[it] = __ldg(reinterpret_cast<const uint4*>(grow) + c);
          wu[it] = __ldg(reinterpret_cast<const uint4*>(urow) + c);
          sg[it] = load_scale<FMT>(gsrow, c, a.group);
          su[it] = load_scale<FMT>(usrow, c, a.group);
        }
      }
      float ag[NT], au[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) ag[t] = au[t] = 0.f;
#pragma unroll
      for (int it = 0; it < kMaxIt; ++it) {
        const int c = lane + 32 * it;
        if (c >= HC) break;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (t >= nt) break;
          const float* xc = xs + t * xstride + c * kPad;
          ag[t] += chunk_dot<FMT>(wg[it], sg[it], xc);
          au[t] += chunk_dot<FMT>(wu[it], su[it], xc);
        }
      }
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if (t >= nt) break;
        const float gv = warp_sum(ag[t]) * tsg;
        const float uv = warp_sum(au[t]) * tsu;
        if (lane == 0) {
          const int p = g.sortedPair[p0 + t];
          a.h[static_cast<size_t>(p) * a.I + r] = silu(gv) * uv;
        }
      }
    }
  }
}

// ------------------------------------------------------------------ down ---
template <int FMT, int NT>
__global__ void __launch_bounds__(kThreads) down_kernel(DecArgs a) {
  __shared__ Groups g;
  __shared__ float s_w[kMaxPairs];
  __shared__ int s_tok[kMaxPairs];
  __shared__ float s_tsd[kMaxPairs];
  build_groups(a, g);
  const int IC = a.I / 32;
  const int nV = g.nValid;
  for (int q = threadIdx.x; q < nV; q += blockDim.x) {
    const int p = g.sortedPair[q];
    s_w[q] = a.topk_w[p];
    s_tok[q] = p / a.k;
  }
  for (int d = threadIdx.x; d < g.nD; d += blockDim.x) {
    float ts = 1.f;
    if constexpr (FMT == FT_NVFP4) ts = __ldg(a.tscale + 3 * (static_cast<int64_t>(a.layer) * a.E + g.dExpert[d]) + 2);
    s_tsd[d] = ts;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t srow_bytes = (FMT == FT_INT4) ? static_cast<uint64_t>(a.I / a.group) * 2
                                               : static_cast<uint64_t>(a.I / 16);
  const int items = g.nD * IC;
  for (int rr = 0; rr < 2; ++rr) {
    const int r = blockIdx.x * kRowsPerCta + warp * 2 + rr;
    float acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.f;
    for (int i0 = 0; i0 < items; i0 += 32 * 4) {
      uint4 w[4];
      uint32_t sc[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int it = i0 + u * 32 + lane;
        if (it < items) {
          const int d = it / IC, c = it % IC;
          const uint8_t* blk = g.dBlock[d];
          w[u] = __ldg(reinterpret_cast<const uint4*>(blk + a.off[2] + static_cast<uint64_t>(r) * (a.I / 2)) + c);
          sc[u] = load_scale<FMT>(blk + a.off[5] + r * srow_bytes, c, a.group);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int it = i0 + u * 32 + lane;
        if (it >= items) break;
        const int d = it / IC, c = it % IC;
        const float ts = s_tsd[d];
        for (int q = g.dStart[d]; q < g.dStart[d + 1]; ++q) {
          // h rows are read straight from the workspace (L1-cached)
          const float part = chunk_dot<FMT>(w[u], sc[u], a.h + static_cast<size_t>(g.sortedPair[q]) * a.I + 32 * c);
          const int tok = s_tok[q];
          const float wt = s_w[q] * ts;
#pragma unroll
          for (int t = 0; t < NT; ++t)
            if (t == tok) acc[t] = fmaf(wt, part, acc[t]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (t >= a.T) break;
      const float v = warp_sum(acc[t]);
      if (lane == 0) {
        if (a.out_bf16)
          static_cast<uint16_t*>(a.out)[static_cast<size_t>(t) * a.H + r] = f32_to_bf16(v);
        else
          static_cast<float*>(a.out)[static_cast<size_t>(t) * a.H + r] = v;
      }
    }
  }
}

template <int FMT, int NT>
ft_status launch_decode(const DecArgs& a, cudaStream_t s) {
  const int n = a.T * a.k;
  const size_t xsm = static_cast<size_t>(NT < 8 ? NT : 8) * (a.H / 32) * kPad * sizeof(float);
  static bool attr_done = false;
  if (!attr_done) {
    cudaFuncSetAttribute(gateup_kernel<FMT, (NT < 8 ? NT : 8)>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(kSmemLimit));
    cudaFuncSetAttribute(down_kernel<FMT, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(kSmemLimit));
    attr_done = true;
  }
  const int grid1 = n * (a.I / kRowsPerCta);
  // gate/up stages x for at most 8 tokens at a time (more pairs take passes)
  constexpr int NTX = NT < 8 ? NT : 8;
  gateup_kernel<FMT, NTX><<<grid1, kThreads, xsm, s>>>(a);
  ft_status st = launch_check("experts decode gate/up");
  if (st != FT_OK) return st;
  const int grid2 = a.H / kRowsPerCta;
  down_kernel<FMT, NT><<<grid2, kThreads, 0, s>>>(a);
  return launch_check("experts decode down");
}

}  // namespace

// Prefill (grouped GEMM) lives in prefill.cu.
ft_status experts_prefill(const ft_bank* cache, const ft_bank* pool, int32_t layer, int32_t E,
                          const uint16_t* xp, const float* x_scale, int32_t T, int32_t k,
                          const int32_t* slot_of_expert, const int32_t* offsets, uint16_t* yp, void* ws,
                          size_t ws_bytes, int32_t* dev_status, cudaStream_t s);
size_t experts_prefill_workspace(int32_t T, int32_t k, int32_t H, int32_t I, int32_t E);

}  // namespace ft

extern "C" {

size_t ft_moe_experts_workspace(int32_t mode, int32_t T, int32_t k, int32_t H, int32_t I,
                                int32_t E) {
  if (T <= 0 || k <= 0 || H <= 0 || I <= 0) return 0;
  if (mode == FT_PREFILL) return ft::experts_prefill_workspace(T, k, H, I, E);
  return (static_cast<size_t>(T) * k * I * sizeof(float) + 255) & ~static_cast<size_t>(255);
}

ft_status ft_moe_experts_fwd(const ft_bank* cache, const ft_bank* pool, int32_t layer, int32_t E,
                             const uint16_t* x, const float* x_scale, int32_t T, const int32_t* slot_ids,
                             const int32_t* raw_ids, const float* topk_w, int32_t k, int32_t mode,
                             const int32_t* offsets, void* out, int32_t out_dtype, void* ws,
                             size_t ws_bytes, int32_t* dev_status, void* stream) {
  ft::Layout L;
  ft_status st = ft::check_bank(cache, "experts cache", &L);
  if (st != FT_OK) return st;
  if (pool) {
    ft::Layout Lp;
    if ((st = ft::check_bank(pool, "experts pool", &Lp)) != FT_OK) return st;
    FT_REQUIRE(pool->fmt == cache->fmt && pool->H == cache->H && pool->I == cache->I &&
                   pool->group == cache->group,
               "experts: pool and cache shapes differ");
  }
  FT_REQUIRE(E >= 1 && layer >= 0, "experts: E=%d layer=%d", E, layer);
  FT_REQUIRE(T >= 0 && k >= 1, "experts: T=%d k=%d", T, k);
  FT_REQUIRE(cache->H <= 4096 && cache->I <= 4096, "experts: H, I must be <= 4096");
  cudaStream_t s = ft::as_stream(stream);
  if (mode == FT_PREFILL) {
    FT_REQUIRE(out_dtype == FT_OUT_BF16, "experts prefill: output must be bf16");
    if (T == 0) return FT_OK;
    FT_REQUIRE(x && slot_ids && offsets && out && ws, "experts prefill: NULL pointer");
    return ft::experts_prefill(cache, pool, layer, E, x, x_scale, T, k, slot_ids, offsets,
                               static_cast<uint16_t*>(out), ws, ws_bytes, dev_status, s);
  }
  FT_REQUIRE(mode == FT_DECODE || mode == FT_DECODE_HOST, "experts: unknown mode %d", mode);
  FT_REQUIRE(mode != FT_DECODE_HOST || pool != nullptr, "experts: FT_DECODE_HOST needs the pool");
  FT_REQUIRE(out_dtype == FT_OUT_F32 || out_dtype == FT_OUT_BF16, "experts: bad out_dtype");
  if (T == 0) return FT_OK;
  const int64_t n = static_cast<int64_t>(T) * k;
  FT_REQUIRE(n <= ft::kMaxPairs && T <= ft::kMaxTok, "experts decode: T*k=%lld > %d or T=%d > %d",
             static_cast<long long>(n), ft::kMaxPairs, T, ft::kMaxTok);
  FT_REQUIRE(x && slot_ids && raw_ids && topk_w && out && ws, "experts decode: NULL pointer");
  FT_REQUIRE(reinterpret_cast<uintptr_t>(x) % 16 == 0 && reinterpret_cast<uintptr_t>(ws) % 16 == 0,
             "experts decode: x and ws must be 16-byte aligned");
  FT_REQUIRE(cache->I % ft::kRowsPerCta == 0 && cache->H % ft::kRowsPerCta == 0,
             "experts decode: H and I must be multiples of 16");
  FT_REQUIRE(ws_bytes >= ft_moe_experts_workspace(FT_DECODE, T, k, cache->H, cache->I, E),
             "experts decode: workspace too small");
  const int NT = T <= 1 ? 1 : (T <= 4 ? 4 : 16);
  const size_t xsm = static_cast<size_t>(NT < 8 ? NT : 8) * (cache->H / 32) * ft::kPad * sizeof(float);
  if (xsm > ft::kSmemLimit)
    return ft::fail(FT_ERR_UNSUPPORTED, "experts decode: T*H too large for one pass");
  ft::DecArgs a;
  a.cache = static_cast<const uint8_t*>(cache->base);
  a.cstride = cache->stride;
  a.cblocks = cache->n_blocks;
  a.pool = pool ? static_cast<const uint8_t*>(pool->base) : nullptr;
  a.pstride = pool ? pool->stride : 0;
  a.pblocks = pool ? pool->n_blocks : 0;
  a.tscale = cache->tensor_scale;
  a.fmt = cache->fmt;
  for (int i = 0; i < 6; ++i) a.off[i] = L.off[i];
  a.H = cache->H;
  a.I = cache->I;
  a.group = cache->group;
  a.layer = layer;
  a.E = E;
  a.T = T;
  a.k = k;
  a.x = x;
  a.slot_ids = slot_ids;
  a.raw_ids = raw_ids;
  a.topk_w = topk_w;
  a.h = static_cast<float*>(ws);
  a.out = out;
  a.out_bf16 = (out_dtype == FT_OUT_BF16);
  a.host_only = (mode == FT_DECODE_HOST);
  a.dev_status = dev_status;
  st = ft::decode_streaming(a, s);
  if (st != FT_ERR_UNSUPPORTED) return st;
  if (cache->fmt == FT_INT4) {
    if (NT == 1) return ft::launch_decode<FT_INT4, 1>(a, s);
    if (NT == 4) return ft::launch_decode<FT_INT4, 4>(a, s);
    return ft::launch_decode<FT_INT4, 16>(a, s);
  }
  if (NT == 1) return ft::launch_decode<FT_NVFP4, 1>(a, s);
  if (NT == 4) return ft::launch_decode<FT_NVFP4, 4>(a, s);
  return ft::launch_decode<FT_NVFP4, 16>(a, s);
}

}  // extern "C"
