// permute.cu -- token permutation by expert for the whole-prompt grouped
// expert pass, and the top-k weighted combine back to token order.
//
// Sources: "NVMe에서 전문가(experts)를 스트리밍하여 8GB GPU에서 133GB MoE 모델
// 구동하기" (molayo1419.me), engine step 5 (run the whole prompt through a
// layer's experts at once instead of re-reading every expert per chunk);
// "SSD 가중치층으로 35B MoE를 ..." (onedev.kr), "How it works" (dedup, stack,
// quantized gather); "FreeToken: 让消费级电脑跑起 284B MoE" sec. 6 (partial
// sums merge exactly).
//
// The permutation is a stable counting sort of the T*k pairs by expert in
// three passes over 256-pair chunks: per-chunk histograms, one scan over the
// (expert, chunk) table in expert-major order, and an in-order scatter in
// which the chunk's warps take turns so equal experts keep pair order.
#include <cuda_fp16.h>

#include "ft_common.cuh"

namespace ft {
namespace {

constexpr int kChunk = 256;
constexpr int kMaxE = 4096;

__device__ __forceinline__ uint32_t __halves2half2_bits(float lo, float hi) {
  return static_cast<uint32_t>(__half_as_ushort(__float2half_rn(lo))) |
         (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(hi))) << 16);
}

__global__ void __launch_bounds__(kChunk) perm_count_kernel(const int32_t* __restrict__ ids, int n,
                                                            int E, int nchunks,
                                                            int32_t* __restrict__ counts,
                                                            int32_t* dev_status) {
  extern __shared__ int hist[];
  for (int e = threadIdx.x; e < E; e += kChunk) hist[e] = 0;
  __syncthreads();
  const int p = blockIdx.x * kChunk + threadIdx.x;
  if (p < n) {
    const int e = ids[p];
    if (e >= 0 && e < E)
      atomicAdd(&hist[e], 1);
    else
      record_status(dev_status, FT_ERR_BAD_ID);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kChunk) counts[static_cast<size_t>(e) * nchunks + blockIdx.x] = hist[e];
}

// Exclusive scan of counts[E][nchunks] (expert-major) into base[][], and the
// expert segment offsets.  One CTA; warp w owns a contiguous segment of the
// counts and reads it 32 consecutive counts at a time (coalesced): its total
// first, then, after the warp totals' scan, a running warp-level inclusive
// scan over the segment.
__global__ void __launch_bounds__(1024) perm_scan_kernel(const int32_t* __restrict__ counts,
                                                         int E, int nchunks, int n,
                                                         int32_t* __restrict__ base,
                                                         int32_t* __restrict__ offsets) {
  __shared__ int wsum[32];
  const int N = E * nchunks;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int seg = ((N + 32 * nw - 1) / (32 * nw)) * 32;  // a multiple of 32
  const int lo = min(N, warp * seg), hi = min(N, lo + seg);
  int s = 0;
#pragma unroll 4
  for (int i = lo + lane; i < hi; i += 32) s += counts[i];
  s = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(s)));
  if (lane == 0) wsum[warp] = s;
  __syncthreads();
  if (warp == 0) {
    const int v = lane < nw ? wsum[lane] : 0;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane < nw) wsum[lane] = x - v;  // exclusive
  }
  __syncthreads();
  int carry = wsum[warp];
#pragma unroll 4
  for (int i0 = lo; i0 < hi; i0 += 32) {
    const int i = i0 + lane;
    const int c = i < hi ? counts[i] : 0;
    int x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (i < hi) base[i] = carry + x - c;
    carry += __shfl_sync(0xffffffffu, x, 31);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) offsets[e] = base[static_cast<size_t>(e) * nchunks];
  if (threadIdx.x == 0) offsets[E] = n;
}

__global__ void __launch_bounds__(kChunk) perm_scatter_kernel(const int32_t* __restrict__ ids, int n,
                                                              int k, int E, int nchunks,
                                                              const int32_t* __restrict__ base,
                                                              int32_t* __restrict__ perm,
                                                              int32_t* __restrict__ inv) {
  extern __shared__ int cnt[];
  for (int e = threadIdx.x; e < E; e += kChunk) cnt[e] = base[static_cast<size_t>(e) * nchunks + blockIdx.x];
  __syncthreads();
  const int p = blockIdx.x * kChunk + threadIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int e = -1;
  if (p < n) {
    e = ids[p];
    if (e < 0 || e >= E) e = -1;
  }
  for (int w = 0; w < kChunk / 32; ++w) {
    if (warp == w) {
      const unsigned same = __match_any_sync(0xffffffffu, e);
      const int leader = __ffs(same) - 1;
      const int rank = __popc(same & ((1u << lane) - 1u));
      int b = 0;
      if (e >= 0 && lane == leader) b = cnt[e];
      b = __shfl_sync(0xffffffffu, b, leader);
      if (e >= 0) {
        const int pos = b + rank;
        perm[pos] = p;
        inv[p] = pos;
      }
      __syncwarp();
      if (e >= 0 && lane == leader) cnt[e] = b + __popc(same);
    }
    __syncthreads();
  }
}

// xp[pos] = x[perm[pos] / k], 16 bytes per thread-step.
__global__ void __launch_bounds__(256) gather_kernel(const uint16_t* __restrict__ x, int H, int k,
                                                     const int32_t* __restrict__ perm, int n,
                                                     uint16_t* __restrict__ xp) {
  const int v = H / 8;
  const size_t total = static_cast<size_t>(n) * v;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int pos = static_cast<int>(i / v), c = static_cast<int>(i % v);
    const int t = perm[pos] / k;
    reinterpret_cast<uint4*>(xp + static_cast<size_t>(pos) * H)[c] =
        __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H) + c);
  }
}

// xp[pos] = f16(x[perm[pos] / k] * f), f the power of two that keeps the row
// below 2^15 (1 for ordinary rows), xp_scale[pos] = 1/f.  One warp per row.
__global__ void __launch_bounds__(256) gather_f16_kernel(const uint16_t* __restrict__ x, int H, int k,
                                                         const int32_t* __restrict__ perm, int n,
                                                         uint16_t* __restrict__ xp,
                                                         float* __restrict__ xp_scale) {
  const int lane = threadIdx.x & 31;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  for (int pos = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; pos < n; pos += nw) {
    const int t = perm[pos] / k;
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H);
    float m = 0.f;
    for (int c = lane; c < H / 8; c += 32) {
      const uint4 v = __ldg(src + c);
      m = fmaxf(m, fmaxf(fmaxf(fabsf(bf16_lo(v.x)), fabsf(bf16_hi(v.x))), fmaxf(fabsf(bf16_lo(v.y)), fabsf(bf16_hi(v.y)))));
      m = fmaxf(m, fmaxf(fmaxf(fabsf(bf16_lo(v.z)), fabsf(bf16_hi(v.z))), fmaxf(fabsf(bf16_lo(v.w)), fabsf(bf16_hi(v.w)))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float f = f16_prescale(m);
    uint4* dst = reinterpret_cast<uint4*>(xp + static_cast<size_t>(pos) * H);
    for (int c = lane; c < H / 8; c += 32) {
      const uint4 v = __ldg(src + c);
      uint4 o;
      o.x = __halves2half2_bits(bf16_lo(v.x) * f, bf16_hi(v.x) * f);
      o.y = __halves2half2_bits(bf16_lo(v.y) * f, bf16_hi(v.y) * f);
      o.z = __halves2half2_bits(bf16_lo(v.z) * f, bf16_hi(v.z) * f);
      o.w = __halves2half2_bits(bf16_lo(v.w) * f, bf16_hi(v.w) * f);
      dst[c] = o;
    }
    if (lane == 0) xp_scale[pos] = 1.f / f;
  }
}

// The same gather, one warp per token: the row (H = 256 VPL) is read once
// into registers, its prescale taken once, and written to the k positions
// inv[t, j] of the token's valid pairs.
template <int VPL>
__global__ void __launch_bounds__(128) gather_f16_tok_kernel(const uint16_t* __restrict__ x, int T, int k,
                                                             int E, const int32_t* __restrict__ ids,
                                                             const int32_t* __restrict__ inv,
                                                             uint16_t* __restrict__ xp,
                                                             float* __restrict__ xp_scale) {
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  constexpr int H = 256 * VPL;
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H);
  uint4 v[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) v[i] = __ldg(src + lane + 32 * i);
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    m = fmaxf(m, fmaxf(fmaxf(fabsf(bf16_lo(v[i].x)), fabsf(bf16_hi(v[i].x))),
                       fmaxf(fabsf(bf16_lo(v[i].y)), fabsf(bf16_hi(v[i].y)))));
    m = fmaxf(m, fmaxf(fmaxf(fabsf(bf16_lo(v[i].z)), fabsf(bf16_hi(v[i].z))),
                       fmaxf(fabsf(bf16_lo(v[i].w)), fabsf(bf16_hi(v[i].w)))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float f = f16_prescale(m);
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    uint4 o;
    o.x = __halves2half2_bits(bf16_lo(v[i].x) * f, bf16_hi(v[i].x) * f);
    o.y = __halves2half2_bits(bf16_lo(v[i].y) * f, bf16_hi(v[i].y) * f);
    o.z = __halves2half2_bits(bf16_lo(v[i].z) * f, bf16_hi(v[i].z) * f);
    o.w = __halves2half2_bits(bf16_lo(v[i].w) * f, bf16_hi(v[i].w) * f);
    v[i] = o;
  }
  for (int j = 0; j < k; ++j) {
    const size_t p = static_cast<size_t>(t) * k + j;
    const int e = __ldg(ids + p);
    if (e < 0 || e >= E) continue;  // no position (the count kernel recorded FT_ERR_BAD_ID)
    const int pos = __ldg(inv + p);
    uint4* dst = reinterpret_cast<uint4*>(xp + static_cast<size_t>(pos) * H);
#pragma unroll
    for (int i = 0; i < VPL; ++i) dst[lane + 32 * i] = v[i];
    if (lane == 0) xp_scale[pos] = 1.f / f;
  }
}

// out[t] = host_partial[t] + sum_j w[t,j] * yp[inv[t,j]] (j order, fp32), bf16.
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ yp,
                                                      const int32_t* __restrict__ inv,
                                                      const float* __restrict__ w, int T, int k,
                                                      int H, const float* __restrict__ hp,
                                                      uint16_t* __restrict__ out) {
  const int t = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;  // 8-element column group
  if (t >= T || c * 8 >= H) return;
  float acc[8];
  if (hp) {
    const float4* h4 = reinterpret_cast<const float4*>(hp + static_cast<size_t>(t) * H) + 2 * c;
    const float4 a = h4[0], b = h4[1];
    acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w;
    acc[4] = b.x; acc[5] = b.y; acc[6] = b.z; acc[7] = b.w;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  }
  for (int j = 0; j < k; ++j) {
    const size_t pj = static_cast<size_t>(t) * k + j;
    const float wj = w[pj];
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(yp + static_cast<size_t>(inv[pj]) * H) + c);
    acc[0] = fmaf(wj, bf16_lo(v.x), acc[0]);
    acc[1] = fmaf(wj, bf16_hi(v.x), acc[1]);
    acc[2] = fmaf(wj, bf16_lo(v.y), acc[2]);
    acc[3] = fmaf(wj, bf16_hi(v.y), acc[3]);
    acc[4] = fmaf(wj, bf16_lo(v.z), acc[4]);
    acc[5] = fmaf(wj, bf16_hi(v.z), acc[5]);
    acc[6] = fmaf(wj, bf16_lo(v.w), acc[6]);
    acc[7] = fmaf(wj, bf16_hi(v.w), acc[7]);
  }
  uint4 o;
  o.x = f32_to_bf16(acc[0]) | (static_cast<uint32_t>(f32_to_bf16(acc[1])) << 16);
  o.y = f32_to_bf16(acc[2]) | (static_cast<uint32_t>(f32_to_bf16(acc[3])) << 16);
  o.z = f32_to_bf16(acc[4]) | (static_cast<uint32_t>(f32_to_bf16(acc[5])) << 16);
  o.w = f32_to_bf16(acc[6]) | (static_cast<uint32_t>(f32_to_bf16(acc[7])) << 16);
  reinterpret_cast<uint4*>(out + static_cast<size_t>(t) * H)[c] = o;
}

int sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

// out = a + b elementwise, written as fp32 or bf16: the merge of two fp32
// partial sums over disjoint pair sets (the cache pairs and the host-path
// pairs of one decode layer call).
__global__ void merge_kernel(const float* a, const float* b, int64_t n, void* out,
                             bool bf16) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float v = a[i] + b[i];
    if (bf16) static_cast<uint16_t*>(out)[i] = f32_to_bf16(v);
    else static_cast<float*>(out)[i] = v;
  }
}

}  // namespace
}  // namespace ft

extern "C" {

size_t ft_moe_permute_workspace(int32_t T, int32_t k, int32_t E) {
  if (T <= 0 || k <= 0 || E <= 0) return 0;
  const size_t n = static_cast<size_t>(T) * k;
  const size_t nchunks = (n + ft::kChunk - 1) / ft::kChunk;
  return (2 * nchunks * E * sizeof(int32_t) + 255) & ~static_cast<size_t>(255);
}

ft_status ft_moe_permute(const int32_t* topk_ids, int32_t T, int32_t k, int32_t E,
                         const uint16_t* x, int32_t H, int32_t* perm, int32_t* inv,
                         int32_t* offsets, uint16_t* xp, int32_t xp_format, float* xp_scale,
                         void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
  FT_REQUIRE(T >= 0 && k >= 1, "permute: T=%d k=%d", T, k);
  FT_REQUIRE(E >= 1 && E <= ft::kMaxE, "permute: E %d outside [1, %d]", E, ft::kMaxE);
  const int64_t n64 = static_cast<int64_t>(T) * k;
  FT_REQUIRE(n64 < (1ll << 31), "permute: T*k overflows int32");
  FT_REQUIRE(offsets != nullptr, "permute: offsets is NULL");
  cudaStream_t s = ft::as_stream(stream);
  const int n = static_cast<int>(n64);
  if (n == 0) {
    cudaError_t e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s);
    return e == cudaSuccess ? FT_OK : ft::fail(FT_ERR_CUDA, "permute: %s", cudaGetErrorString(e));
  }
  FT_REQUIRE(topk_ids && perm && inv && ws, "permute: NULL pointer");
  FT_REQUIRE(ws_bytes >= ft_moe_permute_workspace(T, k, E), "permute: workspace %zu < %zu",
             ws_bytes, ft_moe_permute_workspace(T, k, E));
  FT_REQUIRE(xp_format == FT_XP_BF16 || xp_format == FT_XP_F16, "permute: unknown xp_format %d", xp_format);
  if (xp) {
    FT_REQUIRE(xp_format == FT_XP_BF16 || xp_scale != nullptr, "permute: FT_XP_F16 needs xp_scale");
    FT_REQUIRE(x != nullptr && H > 0 && H % 8 == 0, "permute: gather needs x and H %% 8 == 0");
    FT_REQUIRE(reinterpret_cast<uintptr_t>(x) % 16 == 0 && reinterpret_cast<uintptr_t>(xp) % 16 == 0,
               "permute: x and xp must be 16-byte aligned");
  }
  const int nchunks = (n + ft::kChunk - 1) / ft::kChunk;
  int32_t* counts = static_cast<int32_t*>(ws);
  int32_t* base = counts + static_cast<size_t>(nchunks) * E;
  const size_t hsm = sizeof(int) * E;
  ft::perm_count_kernel<<<nchunks, ft::kChunk, hsm, s>>>(topk_ids, n, E, nchunks, counts, dev_status);
  ft_status st = ft::launch_check("permute count");
  if (st != FT_OK) return st;
  ft::perm_scan_kernel<<<1, 1024, 0, s>>>(counts, E, nchunks, n, base, offsets);
  if ((st = ft::launch_check("permute scan")) != FT_OK) return st;
  ft::perm_scatter_kernel<<<nchunks, ft::kChunk, hsm, s>>>(topk_ids, n, k, E, nchunks, base, perm, inv);
  if ((st = ft::launch_check("permute scatter")) != FT_OK) return st;
  if (xp) {
    const size_t total = static_cast<size_t>(n) * (H / 8);
    const int grid = static_cast<int>(std::min<size_t>((total + 255) / 256, static_cast<size_t>(ft::sms()) * 16));
    if (xp_format == FT_XP_BF16) {
      ft::gather_kernel<<<grid, 256, 0, s>>>(x, H, k, perm, n, xp);
    } else {
      // one warp per token (rows of up to 4096 in registers), else one per pair
      const unsigned gt = static_cast<unsigned>((T + 3) / 4);
      switch (H % 256 == 0 ? H / 256 : 0) {
#define FT_GATHER_TOK(V) \
  case V:                \
    ft::gather_f16_tok_kernel<V><<<gt, 128, 0, s>>>(x, T, k, E, topk_ids, inv, xp, xp_scale); \
    break;
        FT_GATHER_TOK(1) FT_GATHER_TOK(2) FT_GATHER_TOK(3) FT_GATHER_TOK(4) FT_GATHER_TOK(5) FT_GATHER_TOK(6)
        FT_GATHER_TOK(7) FT_GATHER_TOK(8) FT_GATHER_TOK(9) FT_GATHER_TOK(10) FT_GATHER_TOK(11)
        FT_GATHER_TOK(12) FT_GATHER_TOK(13) FT_GATHER_TOK(14) FT_GATHER_TOK(15) FT_GATHER_TOK(16)
#undef FT_GATHER_TOK
        default: {
          const int g2 = std::min((n + 7) / 8, ft::sms() * 16);
          ft::gather_f16_kernel<<<g2, 256, 0, s>>>(x, H, k, perm, n, xp, xp_scale);
        }
      }
    }
    if ((st = ft::launch_check("permute gather")) != FT_OK) return st;
  }
  return FT_OK;
}

ft_status ft_moe_combine(const uint16_t* yp, const int32_t* inv, const float* topk_w, int32_t T,
                         int32_t k, int32_t H, const float* host_partial, uint16_t* out,
                         void* stream) {
  FT_REQUIRE(T >= 0 && k >= 1 && H > 0 && H % 8 == 0, "combine: T=%d k=%d H=%d", T, k, H);
  if (T == 0) return FT_OK;
  FT_REQUIRE(yp && inv && topk_w && out, "combine: NULL pointer");
  FT_REQUIRE(reinterpret_cast<uintptr_t>(yp) % 16 == 0 && reinterpret_cast<uintptr_t>(out) % 16 == 0 &&
                 reinterpret_cast<uintptr_t>(host_partial) % 16 == 0,
             "combine: yp, out and host_partial must be 16-byte aligned");
  FT_REQUIRE(T <= 65535, "combine: T %d > 65535", T);
  dim3 grid((H / 8 + 255) / 256, T);
  ft::combine_kernel<<<grid, 256, 0, ft::as_stream(stream)>>>(yp, inv, topk_w, T, k, H,
                                                              host_partial, out);
  return ft::launch_check("combine");
}

ft_status ft_moe_merge_partials(const float* a, const float* b, int64_t n, void* out, int32_t out_dtype,
                                void* stream) {
  FT_REQUIRE(n >= 0, "merge: n < 0");
  FT_REQUIRE(out_dtype == FT_OUT_F32 || out_dtype == FT_OUT_BF16, "merge: bad out_dtype");
  if (n == 0) return FT_OK;
  FT_REQUIRE(a && b && out, "merge: NULL pointer");
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, 65535ll * 16);
  ft::merge_kernel<<<static_cast<unsigned>(blocks), 256, 0, ft::as_stream(stream)>>>(a, b, n, out,
                                                                                     out_dtype == FT_OUT_BF16);
  return ft::launch_check("merge_partials");
}

}  // extern "C"
