// decode2.cu -- the streaming decode experts kernels (T <= 8 tokens).
//
// Decode reads every routed expert's bytes once and does little arithmetic
// per byte, so the whole layer is a race to keep HBM busy.  Each of the two
// kernels runs one CTA per SM; every CTA owns a contiguous slice of the
// work and, before computing anything, issues TMA bulk copies
// (cp.async.bulk) of its whole slice into a shared-memory ring, so the
// layer's bytes are in flight at once.  Warps compute as stages land
// (mbarrier per stage, bounded waits).
//
//   gate/up: units of RA rows of one distinct expert's gate and up matrices.
//     Each warp owns whole rows; lanes split the row in 32-element chunks,
//     dequantise to f16 in registers and accumulate in fp32 with
//     fma.rn.f32.f16 against the token's activations (f16, exact power-of-two
//     prescale per token); a warp-shuffle reduction finishes the row and
//     h = silu(g) * u goes to the workspace in fp32.
//   down: units of RB rows of H, covering every distinct expert's down rows,
//     launched as a programmatic dependent of gate/up: its weight copies are
//     issued before griddepcontrol.wait, so they stream while gate/up still
//     runs.  After the wait the CTA stages h (f16, per-pair prescale) and
//     each warp produces whole output rows, summing all top-k experts of each
//     token in a fixed order (combine fused, no atomics).
//
// int4: a nibble q becomes the f16 value 1 + q/16 by placing it in the
// mantissa; sum (q - 8) a = 16 * sum (1 + q/16) a - 24 * sum a, with sum a per
// 32-element chunk precomputed.  NVFP4: the hardware e2m1x2 -> f16x2 convert,
// one E4M3 scale per 16 elements.  All products are exact; accumulation fp32.
//
// Experts whose block lives in the host pool (the -1 path read in place) are
// never bulk-copied: their rows are read directly with ordinary loads.
//
// Sources: "SSD 가중치층으로 35B MoE를 ..." (onedev.kr), "How it works";
// "NVMe에서 전문가(experts)를 ... 133GB MoE" (molayo1419.me), step 4;
// "FreeToken 딥다이브" (fiv.co.kr), design pattern 3.
#include <cuda_fp16.h>

#include "ft_async.cuh"
#include "ft_decode.cuh"

namespace ft {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kV2Threads = (kConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kMaxStages = 32;
constexpr int kChunkBytes = 80;  // 32 f16 activations + 16 B pad (conflict-free 16-B reads)

struct V2Geo {
  int RA, RB;       // rows per gate/up unit, per down unit
  int sbA, sbB;     // scale bytes per row: gate/up, down
  int stageA;       // bytes of one gate/up stage
  int nsA;          // gate/up ring stages
  int segB;         // bytes of one expert's rows in a down stage
  int ringB;        // bytes of the down ring
  int xbytes;       // activation area of gate/up (T x H/32 chunks)
  int hbytes;       // activation area of down (pairs x I/32 chunks)
};

// ------------------------------------------------------- f16 dequant-dot ---
__device__ __forceinline__ void fma2_f16(float& a0, float& a1, uint32_t w, uint32_t x) {
  asm("{\n .reg .b16 wl, wh, xl, xh;\n mov.b32 {wl, wh}, %2;\n mov.b32 {xl, xh}, %3;\n"
      " fma.rn.f32.f16 %0, wl, xl, %0;\n fma.rn.f32.f16 %1, wh, xh, %1;\n}"
      : "+f"(a0), "+f"(a1)
      : "r"(w), "r"(x));
}

// int4 chunk: sum over 32 codes of (1 + q/16) * a, a in the word-permuted
// order [a0 a4 a1 a5 a2 a6 a3 a7] per 8 codes.
__device__ __forceinline__ float dot_i4_f16(const uint4 w, const uint8_t* xa) {
  const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 xv = *reinterpret_cast<const uint4*>(xa + 16 * j);
    const uint32_t v = wv[j];
    const uint32_t p0 = ((v << 6) & 0x03C003C0u) | 0x3C003C00u;  // codes 0, 4
    const uint32_t p1 = ((v << 2) & 0x03C003C0u) | 0x3C003C00u;  // codes 1, 5
    const uint32_t p2 = ((v >> 2) & 0x03C003C0u) | 0x3C003C00u;  // codes 2, 6
    const uint32_t p3 = ((v >> 6) & 0x03C003C0u) | 0x3C003C00u;  // codes 3, 7
    fma2_f16(s0, s1, p0, xv.x);
    fma2_f16(s0, s1, p1, xv.y);
    fma2_f16(s0, s1, p2, xv.z);
    fma2_f16(s0, s1, p3, xv.w);
  }
  return s0 + s1;
}

__device__ __forceinline__ void e2m1x8(uint32_t v, uint32_t h[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(v));
}

__device__ __forceinline__ float2 e4m3x2_f32(uint32_t two) {
  uint32_t h2;
  const unsigned short b = static_cast<unsigned short>(two);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(b));
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}

// NVFP4 chunk: s0 * sum_{i<16} e2m1_i a_i + s1 * sum_{i>=16} e2m1_i a_i, a in
// natural order.
__device__ __forceinline__ float dot_fp4_f16(const uint4 w, uint32_t sc2, const uint8_t* xa) {
  const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
  float part[2];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int j = half * 2 + jj;
      const uint4 xv = *reinterpret_cast<const uint4*>(xa + 16 * j);
      uint32_t h[4];
      e2m1x8(wv[j], h);
      fma2_f16(s0, s1, h[0], xv.x);
      fma2_f16(s0, s1, h[1], xv.y);
      fma2_f16(s0, s1, h[2], xv.z);
      fma2_f16(s0, s1, h[3], xv.w);
    }
    part[half] = s0 + s1;
  }
  const float2 s = e4m3x2_f32(sc2);
  return fmaf(part[0], s.x, part[1] * s.y);
}

// One 32-element chunk: codes (16 B), its scale bytes, activations (f16 in
// the format's order) and their sum (int4 only).
template <int FMT>
__device__ __forceinline__ float chunk(const uint8_t* codes, const uint8_t* srow, int c, int group,
                                       const uint8_t* xa, float asum) {
  const uint4 w = *reinterpret_cast<const uint4*>(codes + 16 * c);
  if constexpr (FMT == FT_INT4) {
    const float s = __half2float(__ushort_as_half(
        *reinterpret_cast<const unsigned short*>(srow + 2 * ((c * 32) / group))));
    return s * fmaf(16.f, dot_i4_f16(w, xa), -24.f * asum);
  } else {
    const uint32_t sc2 = *reinterpret_cast<const unsigned short*>(srow + 2 * c);
    return dot_fp4_f16(w, sc2, xa);
  }
}

// Convert 32 fp32 activations (times `mul`) to f16 in the format's order,
// write them (64 B) at dst, return their sum as used.
template <int FMT>
__device__ __forceinline__ float pack_chunk(const float* v, float mul, uint8_t* dst) {
  __half hv[32];
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    hv[i] = __float2half_rn(v[i] * mul);
    s += __half2float(hv[i]);
  }
  uint32_t out[16];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      // int4 order per 8 codes: pairs (0,4) (1,5) (2,6) (3,7); NVFP4: (0,1) (2,3) ...
      const int lo = (FMT == FT_INT4) ? 8 * j + m : 8 * j + 2 * m;
      const int hi = (FMT == FT_INT4) ? 8 * j + m + 4 : 8 * j + 2 * m + 1;
      out[4 * j + m] = static_cast<uint32_t>(__half_as_ushort(hv[lo])) |
                       (static_cast<uint32_t>(__half_as_ushort(hv[hi])) << 16);
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<uint4*>(dst + 16 * j) = make_uint4(out[4 * j], out[4 * j + 1], out[4 * j + 2], out[4 * j + 3]);
  return s;
}

// --------------------------------------------------------------- gate/up ---
template <int FMT>
__global__ void __launch_bounds__(kV2Threads, 1) v2_gateup_kernel(DecArgs a, V2Geo geo) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ Groups g;
  __shared__ __align__(8) uint64_t full[kMaxStages];
  __shared__ __align__(8) uint64_t empty[kMaxStages];
  __shared__ float s_inv[kV2MaxTok];
  pdl_launch_dependents();
  if (prior_timeout(a.dev_status)) return;
  build_groups(a, g);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H, HC = H / 32, RA = geo.RA, nsA = geo.nsA;
  uint8_t* ring = sm;
  uint8_t* xsm = sm + static_cast<size_t>(nsA) * geo.stageA;
  float* xsum = reinterpret_cast<float*>(xsm + geo.xbytes);
  if (tid == 0) {
    for (int s = 0; s < nsA; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_barrier_init();
  }
  // activations: per-token prescale, f16 chunks in the format's order, sums
  for (int t = warp; t < a.T; t += kConsumerWarps + 1) {
    float m = 0.f;
    for (int i = lane; i < H; i += 32) m = fmaxf(m, fabsf(bf16_val(a.x[static_cast<size_t>(t) * H + i])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) s_inv[t] = f16_prescale(m);
  }
  __syncthreads();
  for (int i = tid; i < a.T * HC; i += blockDim.x) {
    const int t = i / HC, c = i % HC;
    const uint4* src = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(t) * H + 32 * c);
    float v[32];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 q = __ldg(src + j);
      v[8 * j + 0] = bf16_lo(q.x); v[8 * j + 1] = bf16_hi(q.x);
      v[8 * j + 2] = bf16_lo(q.y); v[8 * j + 3] = bf16_hi(q.y);
      v[8 * j + 4] = bf16_lo(q.z); v[8 * j + 5] = bf16_hi(q.z);
      v[8 * j + 6] = bf16_lo(q.w); v[8 * j + 7] = bf16_hi(q.w);
    }
    xsum[i] = pack_chunk<FMT>(v, s_inv[t], xsm + static_cast<size_t>(i) * kChunkBytes);
  }
  __syncthreads();

  const int upr = a.I / RA;
  const int U = g.nD * upr;
  const int u0 = static_cast<int>(static_cast<long long>(U) * blockIdx.x / gridDim.x);
  const int u1 = static_cast<int>(static_cast<long long>(U) * (blockIdx.x + 1) / gridDim.x);
  const int nu = u1 - u0;
  const uint32_t rowA = static_cast<uint32_t>(H / 2);
  const uint32_t sbA = static_cast<uint32_t>(geo.sbA);

  if (warp == kConsumerWarps) {
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < nu; ++i) {
        const int st = i % nsA;
        if (i >= nsA && !mbar_wait(&empty[st], ((i / nsA) - 1) & 1, a.dev_status)) break;
        const int u = u0 + i, d = u / upr, r0 = (u % upr) * RA;
        const uint8_t* blk = g.dBlock[d];
        if (g.dCached[d]) {
          uint8_t* dst = ring + static_cast<size_t>(st) * geo.stageA;
          mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(geo.stageA));
          bulk_g2s(dst, blk + a.off[0] + r0 * rowA, RA * rowA, &full[st]);
          bulk_g2s(dst + RA * rowA, blk + a.off[1] + r0 * rowA, RA * rowA, &full[st]);
          bulk_g2s(dst + 2 * RA * rowA, blk + a.off[3] + r0 * sbA, RA * sbA, &full[st]);
          bulk_g2s(dst + 2 * RA * rowA + RA * sbA, blk + a.off[4] + r0 * sbA, RA * sbA, &full[st]);
        } else {
          mbar_arrive(&full[st]);
        }
        issued = i + 1;
      }
      // copies still in flight must land before the CTA exits
      for (int i = max(0, issued - nsA); i < issued; ++i)
        if (!mbar_wait(&full[i % nsA], (i / nsA) & 1, a.dev_status)) break;
    }
    return;
  }

  for (int i = 0; i < nu; ++i) {
    const int st = i % nsA;
    if (!mbar_wait(&full[st], (i / nsA) & 1, a.dev_status)) break;
    const int u = u0 + i, d = u / upr, r0 = (u % upr) * RA;
    const bool cached = g.dCached[d] != 0;
    const uint8_t* blk = g.dBlock[d];
    const uint8_t* stg = ring + static_cast<size_t>(st) * geo.stageA;
    float tsg = 1.f, tsu = 1.f;
    if constexpr (FMT == FT_NVFP4) {
      const int64_t fid = static_cast<int64_t>(a.layer) * a.E + g.dExpert[d];
      tsg = __ldg(a.tscale + 3 * fid + 0);
      tsu = __ldg(a.tscale + 3 * fid + 1);
    }
    for (int rr = 0; rr < RA; ++rr) {
      if (((i * RA + rr) & (kConsumerWarps - 1)) != warp) continue;
      const int r = r0 + rr;
      const uint8_t* gc = cached ? stg + rr * rowA : blk + a.off[0] + static_cast<uint64_t>(r) * rowA;
      const uint8_t* uc = cached ? stg + (RA + rr) * rowA : blk + a.off[1] + static_cast<uint64_t>(r) * rowA;
      const uint8_t* gs = cached ? stg + 2 * RA * rowA + rr * sbA : blk + a.off[3] + static_cast<uint64_t>(r) * sbA;
      const uint8_t* us = cached ? stg + 2 * RA * rowA + (RA + rr) * sbA
                                 : blk + a.off[4] + static_cast<uint64_t>(r) * sbA;
      for (int q = g.dStart[d]; q < g.dStart[d + 1]; ++q) {
        const int p = g.sortedPair[q];
        const int t = p / a.k;
        float ag = 0.f, au = 0.f;
        for (int c = lane; c < HC; c += 32) {
          const uint8_t* xa = xsm + static_cast<size_t>(t * HC + c) * kChunkBytes;
          const float xs = xsum[t * HC + c];
          ag += chunk<FMT>(gc, gs, c, a.group, xa, xs);
          au += chunk<FMT>(uc, us, c, a.group, xa, xs);
        }
        ag = warp_sum(ag);
        au = warp_sum(au);
        if (lane == 0) {
          const float inv = 1.f / s_inv[t];
          const float gv = ag * inv * tsg, uv = au * inv * tsu;
          a.h[static_cast<size_t>(p) * a.I + r] = gv / (1.f + expf(-gv)) * uv;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }
}

// ------------------------------------------------------------------ down ---
template <int FMT, int NT>
__global__ void __launch_bounds__(kV2Threads, 1) v2_down_kernel(DecArgs a, V2Geo geo) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ Groups g;
  __shared__ __align__(8) uint64_t full[kMaxStages];
  __shared__ __align__(8) uint64_t empty[kMaxStages];
  __shared__ float s_w[kMaxPairs];
  __shared__ float s_inv[kMaxPairs];
  __shared__ int s_tok[kMaxPairs];
  __shared__ int s_d[kMaxPairs];
  if (prior_timeout(a.dev_status)) return;
  build_groups(a, g);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int I = a.I, IC = I / 32, RB = geo.RB, H = a.H;
  const int nD = g.nD, nV = g.nValid;
  const int stageB = nD * geo.segB;
  const int nsB = max(1, min(kMaxStages, stageB > 0 ? geo.ringB / stageB : 1));
  uint8_t* ring = sm;
  uint8_t* hsm = sm + geo.ringB;
  float* hsum = reinterpret_cast<float*>(hsm + geo.hbytes);
  if (tid == 0) {
    for (int s = 0; s < nsB; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_barrier_init();
  }
  for (int q = tid; q < nV; q += blockDim.x) {
    const int p = g.sortedPair[q];
    s_w[q] = a.topk_w[p];
    s_tok[q] = p / a.k;
  }
  for (int d = tid; d < nD; d += blockDim.x)
    for (int q = g.dStart[d]; q < g.dStart[d + 1]; ++q) s_d[q] = d;
  __syncthreads();

  const int U = H / RB;
  const int u0 = static_cast<int>(static_cast<long long>(U) * blockIdx.x / gridDim.x);
  const int u1 = static_cast<int>(static_cast<long long>(U) * (blockIdx.x + 1) / gridDim.x);
  const int nu = u1 - u0;
  const uint32_t rowB = static_cast<uint32_t>(I / 2);
  const uint32_t sbB = static_cast<uint32_t>(geo.sbB);

  if (warp == kConsumerWarps) {
    // weights do not depend on the previous grid: stream them before its end
    if (lane == 0) {
      int ncached = 0;
      for (int d = 0; d < nD; ++d) ncached += (g.dCached[d] != 0);
      int issued = 0;
      for (int i = 0; i < nu; ++i) {
        const int st = i % nsB;
        if (i >= nsB && !mbar_wait(&empty[st], ((i / nsB) - 1) & 1, a.dev_status)) break;
        const int r0 = (u0 + i) * RB;
        uint8_t* dst = ring + static_cast<size_t>(st) * stageB;
        if (ncached > 0) {
          mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(ncached * geo.segB));
          for (int d = 0; d < nD; ++d) {
            if (!g.dCached[d]) continue;
            const uint8_t* blk = g.dBlock[d];
            bulk_g2s(dst + d * geo.segB, blk + a.off[2] + r0 * rowB, RB * rowB, &full[st]);
            bulk_g2s(dst + d * geo.segB + RB * rowB, blk + a.off[5] + r0 * sbB, RB * sbB, &full[st]);
          }
        } else {
          mbar_arrive(&full[st]);
        }
        issued = i + 1;
      }
      for (int i = max(0, issued - nsB); i < issued; ++i)
        if (!mbar_wait(&full[i % nsB], (i / nsB) & 1, a.dev_status)) break;
    }
    return;
  }

  // h comes from the gate/up grid: wait for it, then stage it as f16 chunks
  pdl_wait();
  for (int q = warp; q < nV; q += kConsumerWarps) {
    const float* hp = a.h + static_cast<size_t>(g.sortedPair[q]) * I;
    float m = 0.f;
    for (int i = lane; i < I; i += 32) m = fmaxf(m, fabsf(hp[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float mul = f16_prescale(m);
    if (lane == 0) s_inv[q] = 1.f / mul;
    for (int c = lane; c < IC; c += 32) {
      float v[32];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 f = *reinterpret_cast<const float4*>(hp + 32 * c + 4 * j);
        v[4 * j] = f.x; v[4 * j + 1] = f.y; v[4 * j + 2] = f.z; v[4 * j + 3] = f.w;
      }
      hsum[q * IC + c] = pack_chunk<FMT>(v, mul, hsm + static_cast<size_t>(q * IC + c) * kChunkBytes);
    }
  }
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");

  for (int i = 0; i < nu; ++i) {
    const int st = i % nsB;
    if (!mbar_wait(&full[st], (i / nsB) & 1, a.dev_status)) break;
    const int r0 = (u0 + i) * RB;
    const uint8_t* stg = ring + static_cast<size_t>(st) * stageB;
    for (int rr = 0; rr < RB; ++rr) {
      if (((i * RB + rr) & (kConsumerWarps - 1)) != warp) continue;
      const int r = r0 + rr;
      float acc[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[t] = 0.f;
      for (int it = lane; it < nV * IC; it += 32) {
        const int q = it / IC, c = it % IC;
        const int d = s_d[q];
        const uint8_t* blk = g.dBlock[d];
        const bool cached = g.dCached[d] != 0;
        const uint8_t* dc = cached ? stg + d * geo.segB + rr * rowB : blk + a.off[2] + static_cast<uint64_t>(r) * rowB;
        const uint8_t* ds = cached ? stg + d * geo.segB + RB * rowB + rr * sbB
                                   : blk + a.off[5] + static_cast<uint64_t>(r) * sbB;
        float part = chunk<FMT>(dc, ds, c, a.group, hsm + static_cast<size_t>(q * IC + c) * kChunkBytes,
                                hsum[q * IC + c]);
        float wq = s_w[q] * s_inv[q];
        if constexpr (FMT == FT_NVFP4)
          wq *= __ldg(a.tscale + 3 * (static_cast<int64_t>(a.layer) * a.E + g.dExpert[d]) + 2);
        const int tok = s_tok[q];
#pragma unroll
        for (int t = 0; t < NT; ++t)
          if (t == tok) acc[t] = fmaf(wq, part, acc[t]);
      }
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if (t >= a.T) break;
        const float v = warp_sum(acc[t]);
        if (lane == 0) {
          if (a.out_bf16)
            static_cast<uint16_t*>(a.out)[static_cast<size_t>(t) * H + r] = f32_to_bf16(v);
          else
            static_cast<float*>(a.out)[static_cast<size_t>(t) * H + r] = v;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }
}

int pow2_rows(int row_bytes_a, int row_bytes_b) {
  for (int r = 1; r <= 16; r *= 2)
    if ((r * row_bytes_a) % 16 == 0 && (r * row_bytes_b) % 16 == 0) return r;
  return 0;
}

template <int FMT, int NT>
ft_status launch_v2(const DecArgs& a, const V2Geo& geo, size_t smemA, size_t smemB, int grid,
                    cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(v2_gateup_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    cudaFuncSetAttribute(v2_down_kernel<FMT, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    attr = true;
  }
  v2_gateup_kernel<FMT><<<grid, kV2Threads, smemA, s>>>(a, geo);
  ft_status st = launch_check("experts decode gate/up (streaming)");
  if (st != FT_OK) return st;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kV2Threads);
  cfg.dynamicSmemBytes = smemB;
  cfg.stream = s;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, v2_down_kernel<FMT, NT>, a, geo);
  if (e != cudaSuccess) return fail(FT_ERR_CUDA, "experts decode down (streaming): %s", cudaGetErrorString(e));
  return launch_check("experts decode down (streaming)");
}

}  // namespace

// Plan and launch the streaming pair of kernels; FT_ERR_UNSUPPORTED when the
// shape does not fit them (the caller then uses the general kernels).
ft_status decode_streaming(const DecArgs& a, cudaStream_t s) {
  const int T = a.T, n = a.T * a.k, H = a.H, I = a.I;
  if (T > kV2MaxTok) return FT_ERR_UNSUPPORTED;
  V2Geo geo;
  geo.sbA = (a.fmt == FT_INT4) ? (H / a.group) * 2 : H / 16;
  geo.sbB = (a.fmt == FT_INT4) ? (I / a.group) * 2 : I / 16;
  const int ra = pow2_rows(H / 2, geo.sbA), rb = pow2_rows(I / 2, geo.sbB);
  if (ra == 0 || rb == 0) return FT_ERR_UNSUPPORTED;
  geo.RA = max(ra, 4);
  geo.RB = max(rb, 2);
  if (I % geo.RA || H % geo.RB) return FT_ERR_UNSUPPORTED;
  geo.stageA = 2 * geo.RA * (H / 2 + geo.sbA);
  geo.segB = geo.RB * (I / 2 + geo.sbB);
  geo.xbytes = T * (H / 32) * kChunkBytes;
  geo.hbytes = n * (I / 32) * kChunkBytes;
  const size_t xsum = static_cast<size_t>(T) * (H / 32) * 4;
  const size_t hsum = static_cast<size_t>(n) * (I / 32) * 4;
  const size_t stageBmax = static_cast<size_t>(n) * geo.segB;
  // shared memory of one SM holds one CTA of each kernel
  const size_t budget = 196 * 1024;
  const size_t fixed = geo.xbytes + xsum + geo.hbytes + hsum;
  if (fixed + geo.stageA + stageBmax > budget) return FT_ERR_UNSUPPORTED;
  const size_t rings = budget - fixed;
  size_t ringA = rings / 2, ringB = rings - ringA;
  if (ringB < stageBmax) {
    ringB = stageBmax;
    ringA = rings - ringB;
  }
  geo.nsA = static_cast<int>(std::min<size_t>(kMaxStages, ringA / geo.stageA));
  if (geo.nsA < 1) return FT_ERR_UNSUPPORTED;
  ringB = std::min<size_t>(ringB, static_cast<size_t>(kMaxStages) * stageBmax);
  ringB = std::max<size_t>(stageBmax, ringB & ~static_cast<size_t>(127));
  geo.ringB = static_cast<int>(ringB);
  const size_t smemA = static_cast<size_t>(geo.nsA) * geo.stageA + geo.xbytes + xsum;
  const size_t smemB = geo.ringB + geo.hbytes + hsum;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = sms > 0 ? sms : 148;
  const int NT = T <= 1 ? 1 : (T <= 2 ? 2 : (T <= 4 ? 4 : 8));
  if (a.fmt == FT_INT4) {
    if (NT == 1) return launch_v2<FT_INT4, 1>(a, geo, smemA, smemB, grid, s);
    if (NT == 2) return launch_v2<FT_INT4, 2>(a, geo, smemA, smemB, grid, s);
    if (NT == 4) return launch_v2<FT_INT4, 4>(a, geo, smemA, smemB, grid, s);
    return launch_v2<FT_INT4, 8>(a, geo, smemA, smemB, grid, s);
  }
  if (NT == 1) return launch_v2<FT_NVFP4, 1>(a, geo, smemA, smemB, grid, s);
  if (NT == 2) return launch_v2<FT_NVFP4, 2>(a, geo, smemA, smemB, grid, s);
  if (NT == 4) return launch_v2<FT_NVFP4, 4>(a, geo, smemA, smemB, grid, s);
  return launch_v2<FT_NVFP4, 8>(a, geo, smemA, smemB, grid, s);
}

}  // namespace ft
