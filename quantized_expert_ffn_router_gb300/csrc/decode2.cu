// decode2.cu -- the pair-major decode experts kernels (T <= 16 tokens).
//
// At decode sizes a layer reads a few MB of expert weights and does little
// arithmetic per byte: the layer is a race against memory latency.  These
// kernels therefore keep every warp independent and put all of a warp's
// weight loads in flight before anything waits:
//
//   gate/up: grid (I / rows per CTA) x (T*k pairs).  A warp owns RPW rows of
//     one (token, rank) pair's expert; each lane loads its 16-byte chunks of
//     those gate and up rows and their scales at once, then converts the
//     token's activations to f16 in registers (exact per-token power-of-two
//     prescale), dots, reduces with shuffles, and lane r writes row r's
//     h = silu(g) * u to the fp32 workspace.  For rows wider than 2048, and
//     when its grid is resident in one wave (one token at 35B shapes), a
//     second form runs one row per warp in 4-warp CTAs, the activations
//     converted once per CTA into shared memory: four times the warps, each
//     with a quarter of the dependent dequant-dot instructions, which is what
//     bounds a one-token layer (same h, bit for bit).
//   down: a programmatic dependent of gate/up, grid (H / rows per CTA) x T.
//     A CTA owns rows of one token's output.  Its lanes first load their
//     chunks of the down rows of the token's k experts (gate/up has already
//     asked L2 for them; they do not depend on h), then griddepcontrol.wait,
//     stage the token's k intermediates in shared memory as f16 (exact
//     power-of-two prescale per pair), and accumulate the top-k weighted sum
//     of every row in a fixed order (the combine is fused, no atomics).  For
//     one-token calls with rows of 9-16 chunks a second form gives each warp
//     one row and splits the pairs over the warp's two halves.
//
// Pairs are not grouped by expert: two pairs of one expert read its rows
// twice, and the second read is served by L2 since both are in flight
// together.  Masked pairs (slot and pool entry both absent) contribute
// nothing.
//
// Dequantisation: an int4 code q in 0..15 is also the E4M3 code of q * 2^-9
// exactly (the subnormals and the first binade of E4M3 are evenly spaced), so
// cvt.rn.f16x2.e4m3x2 turns two nibbles spread to bytes into f16 q * 2^-9, and
// sum (q - 8) a = 512 * sum (q 2^-9) a - 8 * sum a, with sum a per 32-element
// chunk precomputed.  NVFP4 codes go through cvt.rn.f16x2.e2m1x2.  Products
// are exact (fma.rn.f32.f16) and accumulate in fp32.
//
// Experts whose block lives in the host pool (the -1 path read in place) are
// read with the same loads through the host mapping.
//
// Sources: "SSD 가중치층으로 35B MoE를 ..." (onedev.kr), "How it works";
// "NVMe에서 전문가(experts)를 ... 133GB MoE" (molayo1419.me), step 4;
// "FreeToken 딥다이브" (fiv.co.kr), design pattern 3.
#include <cuda_fp16.h>

#include "ft_async.cuh"
#include "ft_decode.cuh"
#include "ft_dequant.cuh"

namespace ft {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kDownLoads = 8;     // down: 16-byte weight loads a lane holds at once

// The block a pair reads: its cache slot, else its pool entry, else none
// (masked).  Bad ids are recorded when `report` is set.
__device__ __forceinline__ const uint8_t* pair_block(const DecArgs& a, int p, bool report) {
  const int e = a.raw_ids[p];
  const int s = a.slot_ids[p];
  if (e < 0 || e >= a.E) {
    if (report) record_status(a.dev_status, FT_ERR_BAD_ID);
    return nullptr;
  }
  if (s >= 0) {
    if (a.host_only) return nullptr;  // a cache pair: the FT_DECODE call on the cache computes it
    if (s < a.cblocks) return a.cache + static_cast<uint64_t>(s) * a.cstride;
    if (report) record_status(a.dev_status, FT_ERR_BAD_ID);
    return nullptr;
  }
  if (a.pool == nullptr) return nullptr;
  const int64_t fid = static_cast<int64_t>(a.layer) * a.E + e;
  if (fid < a.pblocks) return a.pool + static_cast<uint64_t>(fid) * a.pstride;
  if (report) record_status(a.dev_status, FT_ERR_BAD_ID);
  return nullptr;
}

// --------------------------------------------------------------- gate/up ---
// CPL = 32-element chunks per lane (H <= 1024 * CPL), RPW = rows per warp.
template <int FMT, int CPL, int RPW>
__global__ void __launch_bounds__(kThreads, 2) pm_gateup_kernel(DecArgs a, int gshift) {
  // ids and fetched blocks come from earlier kernels: wait for them, and only
  // then let the down kernel (which reads weights before its own wait) start
  pdl_wait();
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int p = blockIdx.y;
  const int H = a.H, HC = H / 32;
  const int r0 = (blockIdx.x * kWarps + warp) * RPW;
  const uint8_t* blk = pair_block(a, p, blockIdx.x == 0 && threadIdx.x == 0);
  if (blk == nullptr) return;  // masked: down skips this pair too
  const uint32_t rowA = static_cast<uint32_t>(H / 2);
  const uint32_t sbA = (FMT == FT_INT4) ? static_cast<uint32_t>((H / a.group) * 2) : static_cast<uint32_t>(H / 16);

  // the token's activations (small, usually in L2) are requested first so
  // they arrive while the weights are still in flight
  const int t = p / a.k;
  uint32_t raw[CPL][16];
#pragma unroll
  for (int j = 0; j < CPL; ++j) {
    const int c = lane + 32 * j;
    if (c < HC) {
      const uint4* src = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(t) * H + 32 * c);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4 q = __ldg(src + u);
        raw[j][4 * u] = q.x; raw[j][4 * u + 1] = q.y; raw[j][4 * u + 2] = q.z; raw[j][4 * u + 3] = q.w;
      }
    }
  }
  // every weight and scale load of this warp goes out next
  uint4 w[RPW][2][CPL];
  uint32_t sc[RPW][2][CPL];
#pragma unroll
  for (int rr = 0; rr < RPW; ++rr)
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const uint8_t* row = blk + a.off[m] + static_cast<uint64_t>(r0 + rr) * rowA;
      const uint8_t* srow = blk + a.off[3 + m] + static_cast<uint64_t>(r0 + rr) * sbA;
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        const int c = lane + 32 * j;
        if (c < HC) {
          w[rr][m][j] = __ldg(reinterpret_cast<const uint4*>(row) + c);
          sc[rr][m][j] = load_scale<FMT>(srow, c, gshift);
        }
      }
    }
  // this CTA's share of the expert's down matrix and scales goes to L2 now,
  // so the down kernel's loads hit L2 (cache slots only; pool entries stay
  // on the host path)
  if (threadIdx.x == 0 && blk >= a.cache && blk < a.cache + a.cblocks * a.cstride) {  // device blocks only
    const uint64_t dbytes = static_cast<uint64_t>(H) * (a.I / 2);
    const uint64_t dsb = (FMT == FT_INT4) ? static_cast<uint64_t>(H) * (a.I / a.group) * 2 : static_cast<uint64_t>(H) * (a.I / 16);
    const uint64_t c0 = (dbytes / gridDim.x + 15) & ~15ull, c1 = (dsb / gridDim.x + 15) & ~15ull;
    const uint64_t o0 = c0 * blockIdx.x, o1 = c1 * blockIdx.x;
    if (o0 < dbytes) l2_prefetch(blk + a.off[2] + o0, static_cast<uint32_t>(min(c0, dbytes - o0)));
    if (o1 < dsb) l2_prefetch(blk + a.off[5] + o1, static_cast<uint32_t>(min(c1, dsb - o1)));
  }
  float ts0 = 1.f, ts1 = 1.f;
  if constexpr (FMT == FT_NVFP4) {
    const int64_t fid = static_cast<int64_t>(a.layer) * a.E + a.raw_ids[p];
    ts0 = __ldg(a.tscale + 3 * fid + 0);
    ts1 = __ldg(a.tscale + 3 * fid + 1);
  }

  // activations -> f16 in registers, exact power-of-two prescale per token
  uint32_t xa[CPL][16];
  float xs[CPL];
  {
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < CPL; ++j)
      if (lane + 32 * j < HC)
#pragma unroll
        for (int i = 0; i < 16; ++i) m = fmaxf(m, fmaxf(fabsf(bf16_lo(raw[j][i])), fabsf(bf16_hi(raw[j][i]))));
    const float mul = f16_prescale(warp_max(m));
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      xs[j] = 0.f;
      if (lane + 32 * j < HC) xs[j] = pack32<FMT>(raw[j], mul, xa[j]);
    }
    const float inv = 1.f / mul;
    ts0 *= inv;
    ts1 *= inv;
  }

  float acc[RPW][2];
#pragma unroll
  for (int rr = 0; rr < RPW; ++rr)
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      float s = 0.f;
#pragma unroll
      for (int j = 0; j < CPL; ++j)
        if (lane + 32 * j < HC) s += chunk_dot<FMT>(w[rr][m][j], sc[rr][m][j], xa[j], xs[j]);
      acc[rr][m] = s;
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr)
#pragma unroll
      for (int m = 0; m < 2; ++m) acc[rr][m] += __shfl_xor_sync(0xffffffffu, acc[rr][m], o);
  if (lane < RPW) {
    float gv = 0.f, uv = 0.f;
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr)
      if (rr == lane) {
        gv = acc[rr][0];
        uv = acc[rr][1];
      }
    gv *= ts0;
    uv *= ts1;
    a.h[static_cast<size_t>(p) * a.I + r0 + lane] = gv / (1.f + expf(-gv)) * uv;
  }
}

// ------------------------------------------------------- gate/up, 1 row ---
// The rows and arithmetic of pm_gateup_kernel with one row per warp and four
// warps per CTA: four times as many warps, each with a quarter of the
// dependent instructions, so that the dequant-dot work (not the memory) no
// longer sets the kernel's length.  The token's activations are converted
// once per CTA into shared memory (16 f16x2 words per chunk in the format's
// order, then the chunk's sum; 80-byte stride, conflict-free 16-byte reads)
// instead of once per warp.  Every h is bit-identical to pm_gateup_kernel's:
// same prescale, same chunk order, same reduction.
constexpr int kG1Warps = 4;
constexpr int kXWords = 20;  // words per staged activation chunk

template <int FMT, int CPL>
__global__ void __launch_bounds__(kG1Warps * 32, CPL <= 2 ? 8 : 5) pm_gateup1_kernel(DecArgs a, int gshift) {
  __shared__ __align__(16) uint32_t xsm[32 * CPL * kXWords];
  __shared__ float s_max[kG1Warps];
  pdl_wait();
  pdl_launch_dependents();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int p = blockIdx.y;
  const int H = a.H, HC = H / 32;
  const int r = blockIdx.x * kG1Warps + warp;
  const uint8_t* blk = pair_block(a, p, blockIdx.x == 0 && tid == 0);
  if (blk == nullptr) return;  // masked (the whole CTA): down skips this pair too
  const uint32_t rowA = static_cast<uint32_t>(H / 2);
  const uint32_t sbA = (FMT == FT_INT4) ? static_cast<uint32_t>((H / a.group) * 2) : static_cast<uint32_t>(H / 16);

  // this thread's activation chunk (chunk tid; 32 * CPL <= 128 chunks) first:
  // it is in L2 and arrives while the weights are in flight
  const int t = p / a.k;
  const bool has_x = tid < HC;
  uint32_t raw[16];
  if (has_x) {
    const uint4* src = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(t) * H + 32 * tid);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint4 q = __ldg(src + u);
      raw[4 * u] = q.x; raw[4 * u + 1] = q.y; raw[4 * u + 2] = q.z; raw[4 * u + 3] = q.w;
    }
  }
  // the warp's gate and up row chunks and scales, all in flight at once
  uint4 w[2][CPL];
  uint32_t sc[2][CPL];
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    const uint8_t* row = blk + a.off[m] + static_cast<uint64_t>(r) * rowA;
    const uint8_t* srow = blk + a.off[3 + m] + static_cast<uint64_t>(r) * sbA;
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      const int c = lane + 32 * j;
      if (c < HC) {
        w[m][j] = __ldg(reinterpret_cast<const uint4*>(row) + c);
        sc[m][j] = load_scale<FMT>(srow, c, gshift);
      }
    }
  }
  // this CTA's share of the expert's down matrix and scales goes to L2 now
  // (cache slots only; pool entries stay on the host path)
  if (tid == 0 && blk >= a.cache && blk < a.cache + a.cblocks * a.cstride) {
    const uint64_t dbytes = static_cast<uint64_t>(H) * (a.I / 2);
    const uint64_t dsb = (FMT == FT_INT4) ? static_cast<uint64_t>(H) * (a.I / a.group) * 2 : static_cast<uint64_t>(H) * (a.I / 16);
    const uint64_t c0 = (dbytes / gridDim.x + 15) & ~15ull, c1 = (dsb / gridDim.x + 15) & ~15ull;
    const uint64_t o0 = c0 * blockIdx.x, o1 = c1 * blockIdx.x;
    if (o0 < dbytes) l2_prefetch(blk + a.off[2] + o0, static_cast<uint32_t>(min(c0, dbytes - o0)));
    if (o1 < dsb) l2_prefetch(blk + a.off[5] + o1, static_cast<uint32_t>(min(c1, dsb - o1)));
  }
  float ts0 = 1.f, ts1 = 1.f;
  if constexpr (FMT == FT_NVFP4) {
    const int64_t fid = static_cast<int64_t>(a.layer) * a.E + a.raw_ids[p];
    ts0 = __ldg(a.tscale + 3 * fid + 0);
    ts1 = __ldg(a.tscale + 3 * fid + 1);
  }

  // activations -> f16 words in shared memory, exact power-of-two prescale
  // from the token's largest magnitude
  float mx = 0.f;
  if (has_x)
#pragma unroll
    for (int i = 0; i < 16; ++i) mx = fmaxf(mx, fmaxf(fabsf(bf16_lo(raw[i])), fabsf(bf16_hi(raw[i]))));
  mx = warp_max(mx);
  if (lane == 0) s_max[warp] = mx;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kG1Warps; ++i) mx = fmaxf(mx, s_max[i]);
  const float mul = f16_prescale(mx);
  if (has_x) {
    uint32_t o[16];
    const float sum = pack32<FMT>(raw, mul, o);
    uint32_t* dst = xsm + tid * kXWords;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<uint4*>(dst + 4 * q) = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
    dst[16] = __float_as_uint(sum);
  }
  __syncthreads();
  const float inv = 1.f / mul;
  ts0 *= inv;
  ts1 *= inv;

  float g = 0.f, u = 0.f;
#pragma unroll
  for (int j = 0; j < CPL; ++j) {
    const int c = lane + 32 * j;
    if (c < HC) {
      const uint32_t* src = xsm + c * kXWords;
      uint32_t xa[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + 4 * q);
        xa[4 * q] = v.x; xa[4 * q + 1] = v.y; xa[4 * q + 2] = v.z; xa[4 * q + 3] = v.w;
      }
      const float asum = __uint_as_float(src[16]);
      g += chunk_dot<FMT>(w[0][j], sc[0][j], xa, asum);
      u += chunk_dot<FMT>(w[1][j], sc[1][j], xa, asum);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    g += __shfl_xor_sync(0xffffffffu, g, o);
    u += __shfl_xor_sync(0xffffffffu, u, o);
  }
  if (lane == 0) {
    g *= ts0;
    u *= ts1;
    a.h[static_cast<size_t>(p) * a.I + r] = g / (1.f + expf(-g)) * u;
  }
}

// ------------------------------------------------------------------ down ---
// LPR lanes per output row (a power of two covering I/32 chunks, CPL chunks
// per lane); a CTA owns 8 * 32 / LPR rows of one token.
template <int FMT, int LPR, int CPL>
__global__ void __launch_bounds__(kThreads, 2) pm_down_kernel(DecArgs a, int gshift) {
  constexpr int kDownPrefetch = kDownLoads / CPL;  // experts whose chunks a lane holds at once
  extern __shared__ __align__(16) uint8_t hsm[];  // [k][I/32] f16 chunks, then [k][I/32] sums
  __shared__ const uint8_t* s_blk[kMaxPairs];
  __shared__ float s_wq[kMaxPairs];
  constexpr int RPWd = 32 / LPR;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.y, k = a.k;
  const int H = a.H, I = a.I, IC = I / 32;
  const int row = (blockIdx.x * kWarps + warp) * RPWd + lane / LPR;
  // the next call (the next layer's router) may start its launch now: it
  // waits for this grid before it reads anything
  pdl_launch_dependents();
  const int sub = lane % LPR;
  const uint32_t rowB = static_cast<uint32_t>(I / 2);
  const uint32_t sbB = (FMT == FT_INT4) ? static_cast<uint32_t>((I / a.group) * 2) : static_cast<uint32_t>(I / 16);
  float* hsum = reinterpret_cast<float*>(hsm + static_cast<size_t>(k) * IC * kChunkBytes);

  // the token's k blocks (gate/up reports bad ids; nothing is reported here)
  for (int j = tid; j < k; j += kThreads) {
    const int p = t * k + j;
    const uint8_t* blk = pair_block(a, p, false);
    s_blk[j] = blk;
    float wq = 0.f;
    if (blk != nullptr) {
      wq = a.topk_w[p];
      if constexpr (FMT == FT_NVFP4)
        wq *= __ldg(a.tscale + 3 * (static_cast<int64_t>(a.layer) * a.E + a.raw_ids[p]) + 2);
    }
    s_wq[j] = wq;
  }
  __syncthreads();

  float acc = 0.f;
  for (int j0 = 0; j0 < k; j0 += kDownPrefetch) {
    // weights first: they do not depend on the previous grid
    uint4 w[kDownPrefetch][CPL];
    uint32_t sc[kDownPrefetch][CPL];
#pragma unroll
    for (int e = 0; e < kDownPrefetch; ++e) {
      const int j = j0 + e;
      const uint8_t* blk = j < k ? s_blk[j] : nullptr;
      if (blk != nullptr) {
        const uint8_t* r = blk + a.off[2] + static_cast<uint64_t>(row) * rowB;
        const uint8_t* sr = blk + a.off[5] + static_cast<uint64_t>(row) * sbB;
#pragma unroll
        for (int m = 0; m < CPL; ++m) {
          const int c = sub + LPR * m;
          if (c < IC) {
            w[e][m] = __ldg(reinterpret_cast<const uint4*>(r) + c);
            sc[e][m] = load_scale<FMT>(sr, c, gshift);
          }
        }
      }
    }
    if (j0 == 0) {
      // h comes from the gate/up grid: wait for it, then stage this token's
      // k rows as f16 chunks (one warp per pair)
      pdl_wait();
      for (int j = warp; j < k; j += kWarps)
        if (s_blk[j] != nullptr) stage_h<FMT>(a, t * k + j, j, hsm, hsum, s_wq);
      __syncthreads();
    }
#pragma unroll
    for (int e = 0; e < kDownPrefetch; ++e) {
      const int j = j0 + e;
      if (j < k && s_blk[j] != nullptr) {
        float s = 0.f;
#pragma unroll
        for (int m = 0; m < CPL; ++m) {
          const int c = sub + LPR * m;
          if (c < IC) {
            const uint8_t* hp = hsm + static_cast<size_t>(j * IC + c) * kChunkBytes;
            uint32_t ha[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint4 v = *reinterpret_cast<const uint4*>(hp + 16 * q);
              ha[4 * q] = v.x; ha[4 * q + 1] = v.y; ha[4 * q + 2] = v.z; ha[4 * q + 3] = v.w;
            }
            s += chunk_dot<FMT>(w[e][m], sc[e][m], ha, hsum[j * IC + c]);
          }
        }
        acc = fmaf(s_wq[j], s, acc);
      }
    }
  }
#pragma unroll
  for (int o = LPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (sub == 0) {
    const size_t idx = static_cast<size_t>(t) * H + row;
    if (a.out_bf16) static_cast<uint16_t*>(a.out)[idx] = f32_to_bf16(acc);
    else static_cast<float*>(a.out)[idx] = acc;
  }
}

// ------------------------------------------------------ down, half pairs ---
// pm_down_kernel with one row per warp and the token's pairs split over the
// warp's two 16-lane halves (half h dots pairs h, h + 2, ...; rows of at
// most 16 chunks), the halves' sums added with one shuffle: twice the warps
// on a grid that would otherwise run one 8-warp CTA per SM or fewer, each
// lane with half the dependent chunk dots.  The staging of h and the weight
// loads before the wait are pm_down_kernel's.
template <int FMT>
__global__ void __launch_bounds__(kThreads, 2) pm_down2_kernel(DecArgs a, int gshift) {
  constexpr int LPR = 16;
  constexpr int NB = kDownLoads;  // pairs whose chunk a lane holds at once
  extern __shared__ __align__(16) uint8_t hsm[];  // [k][I/32] f16 chunks, then [k][I/32] sums
  __shared__ const uint8_t* s_blk[kMaxPairs];
  __shared__ float s_wq[kMaxPairs];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.y, k = a.k;
  const int H = a.H, I = a.I, IC = I / 32;
  const int row = blockIdx.x * kWarps + warp;
  const int half = lane / LPR, sub = lane % LPR;
  // the next call (the next layer's router) may start its launch now: it
  // waits for this grid before it reads anything
  pdl_launch_dependents();
  const uint32_t rowB = static_cast<uint32_t>(I / 2);
  const uint32_t sbB = (FMT == FT_INT4) ? static_cast<uint32_t>((I / a.group) * 2) : static_cast<uint32_t>(I / 16);
  float* hsum = reinterpret_cast<float*>(hsm + static_cast<size_t>(k) * IC * kChunkBytes);

  for (int j = tid; j < k; j += kThreads) {
    const int p = t * k + j;
    const uint8_t* blk = pair_block(a, p, false);
    s_blk[j] = blk;
    float wq = 0.f;
    if (blk != nullptr) {
      wq = a.topk_w[p];
      if constexpr (FMT == FT_NVFP4)
        wq *= __ldg(a.tscale + 3 * (static_cast<int64_t>(a.layer) * a.E + a.raw_ids[p]) + 2);
    }
    s_wq[j] = wq;
  }
  __syncthreads();

  uint4 w[NB];
  uint32_t sc[NB];
  auto load_batch = [&](int j0) {
#pragma unroll
    for (int e = 0; e < NB; ++e) {
      const int j = j0 + 2 * e;
      const uint8_t* blk = j < k ? s_blk[j] : nullptr;
      if (blk != nullptr && sub < IC) {
        w[e] = __ldg(reinterpret_cast<const uint4*>(blk + a.off[2] + static_cast<uint64_t>(row) * rowB) + sub);
        sc[e] = load_scale<FMT>(blk + a.off[5] + static_cast<uint64_t>(row) * sbB, sub, gshift);
      }
    }
  };
  // the first pairs' weights do not depend on the previous grid
  load_batch(half);
  // h comes from the gate/up grid: wait for it, then stage the token's k
  // rows as f16 chunks (one warp per pair)
  pdl_wait();
  for (int j = warp; j < k; j += kWarps)
    if (s_blk[j] != nullptr) stage_h<FMT>(a, t * k + j, j, hsm, hsum, s_wq);
  __syncthreads();

  float acc = 0.f;
  for (int j0 = half; j0 < k; j0 += 2 * NB) {
    if (j0 != half) load_batch(j0);
#pragma unroll
    for (int e = 0; e < NB; ++e) {
      const int j = j0 + 2 * e;
      if (j < k && s_blk[j] != nullptr && sub < IC) {
        const uint8_t* hp = hsm + static_cast<size_t>(j * IC + sub) * kChunkBytes;
        uint32_t ha[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 v = *reinterpret_cast<const uint4*>(hp + 16 * q);
          ha[4 * q] = v.x; ha[4 * q + 1] = v.y; ha[4 * q + 2] = v.z; ha[4 * q + 3] = v.w;
        }
        acc = fmaf(s_wq[j], chunk_dot<FMT>(w[e], sc[e], ha, hsum[j * IC + sub]), acc);
      }
    }
  }
#pragma unroll
  for (int o = LPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  acc += __shfl_xor_sync(0xffffffffu, acc, LPR);  // half 0's pairs + half 1's
  if (lane == 0) {
    const size_t idx = static_cast<size_t>(t) * H + row;
    if (a.out_bf16) static_cast<uint16_t*>(a.out)[idx] = f32_to_bf16(acc);
    else static_cast<float*>(a.out)[idx] = acc;
  }
}

template <int FMT, int CPL, int RPW>
ft_status launch_gateup(const DecArgs& a, int gshift, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.I / (kWarps * RPW), a.T * a.k);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, pm_gateup_kernel<FMT, CPL, RPW>, a, gshift);
  if (e != cudaSuccess) return fail(FT_ERR_CUDA, "experts decode gate/up: %s", cudaGetErrorString(e));
  return launch_check("experts decode gate/up");
}

template <int FMT, int CPL>
ft_status launch_gateup1(const DecArgs& a, int gshift, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.I / kG1Warps, a.T * a.k);
  cfg.blockDim = dim3(kG1Warps * 32);
  cfg.stream = s;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, pm_gateup1_kernel<FMT, CPL>, a, gshift);
  if (e != cudaSuccess) return fail(FT_ERR_CUDA, "experts decode gate/up: %s", cudaGetErrorString(e));
  return launch_check("experts decode gate/up");
}

template <int FMT>
ft_status launch_down2(const DecArgs& a, int gshift, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(a.k) * (a.I / 32) * (kChunkBytes + 4);
  ft_status st = ensure_dyn_smem(reinterpret_cast<const void*>(pm_down2_kernel<FMT>), 200 * 1024,
                                 "experts decode down");
  if (st != FT_OK) return st;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.H / kWarps, a.T);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, pm_down2_kernel<FMT>, a, gshift);
  if (e != cudaSuccess) return fail(FT_ERR_CUDA, "experts decode down: %s", cudaGetErrorString(e));
  return launch_check("experts decode down");
}

template <int FMT, int LPR, int CPL>
ft_status launch_down(const DecArgs& a, int gshift, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(a.k) * (a.I / 32) * (kChunkBytes + 4);
  ft_status st = ensure_dyn_smem(reinterpret_cast<const void*>(pm_down_kernel<FMT, LPR, CPL>), 200 * 1024,
                                 "experts decode down");
  if (st != FT_OK) return st;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.H / (kWarps * (32 / LPR)), a.T);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, pm_down_kernel<FMT, LPR, CPL>, a, gshift);
  if (e != cudaSuccess) return fail(FT_ERR_CUDA, "experts decode down: %s", cudaGetErrorString(e));
  return launch_check("experts decode down");
}

// Which gate/up kernel runs.  Rows wider than 2048 always take the one-row
// kernel: the other form has one row per warp there too, and converts the
// activations in every warp (flash, one token: 23.1 against 28.5 us per
// experts call in a 48-layer graph).  Up to 2048 the one-row kernel runs
// when its grid is resident in one wave (8 CTAs per SM): then it beats four
// rows per warp, whose grid leaves most SMs idle or nearly so (d35b, one
// token: 10.5 against 13.3 us).  Larger calls keep four rows per warp: their
// grids fill the GPU, and the dequant-dot instructions, fewer with four rows
// per warp, bound them (eight tokens: 43.9 against 45.2 us with one row per
// warp, 43.6 with a double-buffered loop over 16 rows per warp).
bool gateup_one_row(const DecArgs& a) {
  const int HC = a.H / 32;
  if (HC > 128 || a.I % kG1Warps != 0) return false;
  return HC > 64 || static_cast<int64_t>(a.I / kG1Warps) * a.T * a.k <= 8ll * device_sm_count();
}

template <int FMT>
ft_status launch_pm(const DecArgs& a, int gshift, cudaStream_t s) {
  const int HC = a.H / 32, IC = a.I / 32;
  ft_status st;
  // gate/up: one row per warp when that grid is resident in one wave
  // (8 CTAs per SM; d35b at one token), else four rows per warp (one for
  // rows wider than 2048): see gateup_one_row.
  if (gateup_one_row(a)) {
    if (HC <= 32) st = launch_gateup1<FMT, 1>(a, gshift, s);
    else if (HC <= 64) st = launch_gateup1<FMT, 2>(a, gshift, s);
    else if (HC <= 96) st = launch_gateup1<FMT, 3>(a, gshift, s);
    else st = launch_gateup1<FMT, 4>(a, gshift, s);
  } else if (HC <= 32) {
    st = launch_gateup<FMT, 1, 4>(a, gshift, s);
  } else {
    st = launch_gateup<FMT, 2, 4>(a, gshift, s);
  }
  if (st != FT_OK) return st;
  // down: with rows of at most 16 chunks and a one-row-per-warp grid that
  // is resident in one wave (2 CTAs per SM), the pairs split over warp
  // halves; else lanes per row
  if (IC <= 16 && IC > 8 && a.k >= 2 && a.H % kWarps == 0 &&
      static_cast<int64_t>(a.H / kWarps) * a.T <= 2ll * device_sm_count())
    return launch_down2<FMT>(a, gshift, s);
  if (IC <= 8) return launch_down<FMT, 8, 1>(a, gshift, s);
  if (IC <= 16) return launch_down<FMT, 16, 1>(a, gshift, s);
  if (IC <= 32) return launch_down<FMT, 32, 1>(a, gshift, s);
  if (IC <= 64) return launch_down<FMT, 32, 2>(a, gshift, s);
  return launch_down<FMT, 32, 4>(a, gshift, s);
}

}  // namespace

// Launch the pair-major kernels; FT_ERR_UNSUPPORTED (with a message) for a
// shape outside them, which the entry point's checks already exclude.
ft_status decode_streaming(const DecArgs& a, cudaStream_t s) {
  const int HC = a.H / 32, IC = a.I / 32;
  const int lpr = IC <= 8 ? 8 : (IC <= 16 ? 16 : 32);
  if (HC > 128 || IC > 128 || a.T * a.k > kMaxPairs || a.T > 65535 ||
      (!gateup_one_row(a) && (HC > 64 || a.I % (kWarps * 4) != 0)) || a.H % (kWarps * (32 / lpr)))
    return fail(FT_ERR_UNSUPPORTED, "experts decode: H=%d I=%d T=%d k=%d outside the decode kernels", a.H, a.I,
                a.T, a.k);
  const int gshift = (a.fmt == FT_INT4) ? (a.group == 32 ? 0 : (a.group == 64 ? 1 : 2)) : 0;
  if (a.fmt == FT_INT4) return launch_pm<FT_INT4>(a, gshift, s);
  return launch_pm<FT_NVFP4>(a, gshift, s);
}

}  // namespace ft
