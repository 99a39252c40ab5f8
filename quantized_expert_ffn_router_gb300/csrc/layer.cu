// layer.cu -- one decode layer call as one kernel: router logits, softmax and
// top-k; the resolve of the top-k ids against the global slot cache with the
// Q16 q* split; the copy of the experts it chose to fetch; the quantized
// SwiGLU experts with the top-k combine.
//
// At decode sizes every step of the layer is short and each depends on the
// one before, so the layer is a chain of latencies, and kernel boundaries
// between the steps cost as much as the steps themselves.  Here one grid of
// one CTA per SM runs the whole chain and the boundaries become three
// grid-wide hand-offs through a counter and a generation word in the
// workspace, each a bounded wait:
//
//   0. before waiting for the previous kernel of the stream, each CTA starts
//      bulk copies of its router rows (rows c, c + G, ...) into shared
//      memory: they are no kernel's output;
//   1. each CTA dots its rows with the tokens and writes the logits; the
//      last CTA to arrive at the counter becomes this call's leader;
//   2. the leader runs the softmax and top-k (one warp per token) and the
//      resolve (dedup, hits, the q* split, recency-ranked fetch choice,
//      victim search, id rewrite; the same device code as
//      ft_moe_resolve_slots), then releases the generation word; meanwhile
//      the other CTAs stage the tokens' activations as f16 chunks;
//   3. when the resolve fetched experts, every CTA copies its share of their
//      blocks from the pool to their slots, then a grid barrier;
//   4. every CTA groups the (token, rank) pairs by distinct expert and starts
//      bulk copies of its output rows of every distinct expert's down matrix
//      (rows [c*H/G, (c+1)*H/G)) and of its share of the gate/up rows (the
//      (expert, row) space cut into G contiguous ranges, each warp a ring of
//      slots), so that a CTA's whole share of the layer's expert bytes is in
//      flight at once; each warp dots its gate/up rows with the tokens of
//      that expert as soon as they land and writes h = silu(g) * u;
//   5. a grid barrier (h complete), then each CTA stages h as f16 chunks and
//      sums the top-k weighted down rows it already holds for every token:
//      out[t, r] = sum_j w[t, j] * (D_e(t,j)[r, :] . h[t, j]) in a fixed order.
//
// The arithmetic of each step is that of the separate entry points: the
// same top-k and resolve code, the dequantise-and-dot of the pair-major
// decode kernels.  Pairs whose expert stays on the host path (slot -1, pool
// given) read the pool in place with plain loads; masked pairs contribute
// nothing.
//
// Every CTA of the grid must be resident at once (the hand-offs wait for all
// of them): the grid is one CTA per SM and is launched cooperatively.
//
// Sources: "FreeToken: 让消费级电脑跑起 284B MoE" (fengjutian.github.io),
// secs. 2 and 6 (router on the GPU; one kernel does dedup, residency, q,
// victims and the id rewrite, with no host crossing inside the layer);
// "FreeToken 딥다이브" (fiv.co.kr), design patterns 2-5; "SSD 가중치층으로
// 35B MoE를 ..." (onedev.kr), "How it works"; "NVMe에서 전문가(experts)를 ...
// 133GB MoE" (molayo1419.me), step 4.
#include "ft_async.cuh"
#include "ft_common.cuh"
#include "ft_decode.cuh"
#include "ft_dequant.cuh"
#include "ft_resolve.cuh"
#include "ft_topk.cuh"

namespace ft {
namespace {

constexpr int kLWarps = 16;
constexpr int kLThreads = kLWarps * 32;
constexpr int kLMaxT = 8;            // tokens per call
constexpr int kLMaxPairs = 128;      // T * k
constexpr int kLMaxE = 512;          // the register top-k
constexpr int kLMaxRouterRows = 4;   // router rows per CTA: E <= 4 * grid
constexpr int kLMaxSegs = 4;         // gate/up row segments (distinct experts) per CTA
constexpr int kXWordsL = 20;         // words per staged activation chunk (16 f16x2 + sum + pad)
constexpr int kLHRep = 8;            // copies of h, so that the workers' reads spread over L2

struct LayerArgs {
  const uint16_t* x;  // [T, H] bf16
  const float* W;     // [E, H] fp32
  int T, H, E, k, renorm, I, gshift, layer, G;
  const uint8_t* cache;
  uint64_t cstride;
  int64_t cblocks;
  const uint8_t* pool;
  uint64_t pstride;
  int64_t pblocks;
  const float* tscale;
  uint64_t off[6];
  uint32_t rowA, sbA;  // bytes of one gate/up code row, of its scale row
  uint32_t rowB, sbB;  // bytes of one down code row, of its scale row
  uint64_t block_bytes;
  int32_t* ids;
  float* wts;
  int32_t* slot_ids;
  int32_t* num_fetch;
  int32_t* fetch_fid;
  int32_t* fetch_slot;
  int max_list;
  void* out;
  int out_bf16;
  ResolveArgs res;
  unsigned long long* bar;  // arrival counter of every hand-off, only ever incremented
  unsigned long long* plan;  // the leader's decisions, each word tagged with this call's generation
  float* logits;          // [E, kLMaxT]: expert e's logits in a 32-byte sector of their own
  float* h;               // kLHRep replicas of [T * k, I] fp32
  size_t h_rep;           // floats between replicas
  int32_t* dev_status;
  uint64_t wait_ns;
  int qg;                 // gate/up rows per unit (scale rows 16-byte aligned)
  int qd;                 // alignment of the down row ranges
  int grows;              // most gate/up rows a CTA owns
  int drows;              // most down rows a CTA owns
  uint32_t dslab;         // one distinct expert's down rows in shared memory
  uint32_t sm_x, sm_r, sm_d, sm_h, sm_bar;
};

// Plan words: [0] nf, then per pair p: [1 + p] expert id | slot << 32 is
// split over two words to keep each word's payload 32 bits: [1 + p] expert,
// [1 + n + p] slot (as uint32), [1 + 2n + p] weight bits, then per fetch i:
// [1 + 3n + i] flat id, [1 + 3n + max_list + i] slot.  Word = tag << 32 | payload.
__device__ __forceinline__ unsigned long long plan_word(uint32_t tag, uint32_t payload) {
  return (static_cast<unsigned long long>(tag) << 32) | payload;
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// A barrier of the workers on a monotonic 64-bit counter: each arrives with a
// release add that it does not wait for, then polls until the counter
// reaches `target` (the value at the call's start plus the arrivals of this
// and the earlier barriers of the call).  Every thread of the CTA calls it;
// true (CTA-uniform) once all have arrived, false on timeout.  Plain writes
// before it are visible after it.
__device__ bool grid_barrier(const LayerArgs& a, unsigned long long target, int* s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(a.bar) : "memory");
    bool ok = true;
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a.bar) : "memory");
    if (v < target) {
      const uint64_t t0 = global_timer_ns();
      for (uint32_t i = 1;; ++i) {
        __nanosleep(20);
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a.bar) : "memory");
        if (v >= target) break;
        if (global_timer_ns() - t0 > a.wait_ns) {
          record_status(a.dev_status, FT_ERR_TIMEOUT);
          ok = false;
          break;
        }
      }
    }
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

__device__ bool mbar_wait_lim(uint64_t* bar, uint32_t parity, int32_t* status, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) {
      record_status(status, FT_ERR_TIMEOUT);
      return false;
    }
  }
}

// A scale word from shared memory (load_scale's layout).
template <int FMT>
__device__ __forceinline__ uint32_t smem_scale(const uint8_t* srow, int c, int gshift) {
  if constexpr (FMT == FT_INT4)
    return reinterpret_cast<const unsigned short*>(srow)[c >> gshift];
  else
    return reinterpret_cast<const unsigned short*>(srow)[c];
}

// The CTA copies `bytes` (a multiple of 16) with plain loads (host memory).
__device__ __forceinline__ void cta_copy(uint8_t* dst, const uint8_t* src, uint32_t bytes) {
  for (uint32_t o = 16u * threadIdx.x; o < bytes; o += 16u * blockDim.x)
    *reinterpret_cast<uint4*>(dst + o) = *reinterpret_cast<const uint4*>(src + o);
}

template <int FMT>
__global__ void __launch_bounds__(kLThreads, 1) layer_kernel(const __grid_constant__ LayerArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ int s_ok, s_leader, s_skip, s_nf, s_nD, s_nseg;
  __shared__ unsigned long long s_base;
  __shared__ float s_part[kLWarps][kLMaxRouterRows * kLMaxT];
  __shared__ float s_xinv[kLMaxT];
  __shared__ int s_pe[kLMaxPairs], s_slot[kLMaxPairs], s_pd[kLMaxPairs];
  __shared__ float s_wq[kLMaxPairs];
  __shared__ int s_dExpert[kLMaxPairs], s_dHost[kLMaxPairs], s_dStart[kLMaxPairs + 1], s_dPairs[kLMaxPairs];
  __shared__ const uint8_t* s_dBlk[kLMaxPairs];
  __shared__ float s_dts[kLMaxPairs][2];
  __shared__ int s_segD[kLMaxSegs], s_segR0[kLMaxSegs], s_segN[kLMaxSegs];
  __shared__ uint32_t s_segOff[kLMaxSegs];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, G = a.G;
  const int T = a.T, H = a.H, E = a.E, k = a.k, I = a.I;
  const int HC = H / 32, IC = I / 32;
  const int n = T * k;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + a.sm_bar);  // [0] router, [1] down, [2..] gate/up segments
  float* wrows = reinterpret_cast<float*>(sm + a.sm_r);
  uint32_t* xsm = reinterpret_cast<uint32_t*>(sm + a.sm_x);

  // ---- 0. this CTA's router rows, before the wait: no kernel writes them
  int nrows = 0;
  for (int e = c; e < E && nrows < kLMaxRouterRows; e += G) ++nrows;
  if (tid == 0) {
    for (int i = 0; i < 2 + kLMaxSegs; ++i) mbar_init(&bars[i], 1);
    fence_barrier_init();
    if (nrows > 0) {
      const uint32_t rb = static_cast<uint32_t>(H) * 4u;
      mbar_arrive_expect_tx(&bars[0], rb * nrows);
      for (int i = 0; i < nrows; ++i)
        bulk_g2s(wrows + static_cast<size_t>(i) * H, a.W + static_cast<size_t>(c + G * i) * H, rb, &bars[0]);
    }
  }
  pdl_wait();  // x, the cache state and the workspace come from earlier kernels
  pdl_launch_dependents();
  if (tid == 0) {
    s_skip = a.dev_status != nullptr && *reinterpret_cast<const volatile int32_t*>(a.dev_status) == FT_ERR_TIMEOUT;
    unsigned long long b;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(b) : "l"(a.bar) : "memory");
    s_base = b;
  }
  __syncthreads();
  const bool router_ok = nrows == 0 || mbar_wait_lim(&bars[0], 0, a.dev_status, a.wait_ns);
  if (s_skip || !router_ok) return;  // an earlier wait gave up: do nothing (no copy is in flight now)
  // the barrier counter grows by at least one every call, so this tag is
  // never that of a word left by an earlier call (nor 0, a cleared word's)
  const unsigned long long base = s_base;
  const uint32_t tag = static_cast<uint32_t>(base) + 1u;

  // ---- 1. logits of this CTA's rows
  {
    const int nch = H / 8;
    for (int t = 0; t < T; ++t) {
      float acc[kLMaxRouterRows] = {0.f, 0.f, 0.f, 0.f};
      for (int ch = tid; ch < nch; ch += kLThreads) {
        const uint4 xv = __ldcg(reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(t) * H) + ch);
        const float xf[8] = {bf16_lo(xv.x), bf16_hi(xv.x), bf16_lo(xv.y), bf16_hi(xv.y),
                             bf16_lo(xv.z), bf16_hi(xv.z), bf16_lo(xv.w), bf16_hi(xv.w)};
#pragma unroll
        for (int i = 0; i < kLMaxRouterRows; ++i) {
          if (i >= nrows) break;
          const float4 w0 = *reinterpret_cast<const float4*>(wrows + static_cast<size_t>(i) * H + 8 * ch);
          const float4 w1 = *reinterpret_cast<const float4*>(wrows + static_cast<size_t>(i) * H + 8 * ch + 4);
          float s = acc[i];
          s = fmaf(xf[0], w0.x, s);
          s = fmaf(xf[1], w0.y, s);
          s = fmaf(xf[2], w0.z, s);
          s = fmaf(xf[3], w0.w, s);
          s = fmaf(xf[4], w1.x, s);
          s = fmaf(xf[5], w1.y, s);
          s = fmaf(xf[6], w1.z, s);
          s = fmaf(xf[7], w1.w, s);
          acc[i] = s;
        }
      }
#pragma unroll
      for (int i = 0; i < kLMaxRouterRows; ++i) {
        if (i >= nrows) break;
        const float v = warp_sum(acc[i]);
        if (lane == 0) s_part[warp][i * T + t] = v;
      }
    }
    __syncthreads();
    if (tid < nrows * T) {
      const int i = tid / T, t = tid % T;
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kLWarps; ++w) v += s_part[w][i * T + t];
      a.logits[static_cast<size_t>(c + G * i) * kLMaxT + t] = v;  // each expert's logits in their own sector
    }
  }
  // ---- 2. CTA 0 leads (the same SM every call, so its code stays in the
  // SM's instruction cache): the others announce their logits with a release
  // add they do not wait for, and CTA 0 waits until all of them have
  const int W = G - 1;  // workers: every CTA but the leader
  s_leader = c == 0;
  __syncthreads();
  if (tid == 0 && c != 0) asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(a.bar) : "memory");
  if (c == 0) {
    if (tid == 0) {
      const unsigned long long goal = s_base + static_cast<unsigned long long>(W);
      unsigned long long v;
      asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a.bar) : "memory");
      s_ok = 1;
      if (v < goal) {
        const uint64_t t0 = global_timer_ns();
        for (uint32_t i = 1;; ++i) {
          __nanosleep(20);
          asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a.bar) : "memory");
          if (v >= goal) break;
          if (global_timer_ns() - t0 > a.wait_ns) {
            record_status(a.dev_status, FT_ERR_TIMEOUT);
            s_ok = 0;
            break;
          }
        }
      }
    }
    __syncthreads();
    if (!s_ok) return;
  }

  unsigned long long* plan = a.plan;
  const int nw_fetch = a.max_list;
  if (s_leader) {
    // softmax + top-k (one warp per token), the resolve, then the plan; the
    // leader takes no part in the expert work
    for (int t = warp; t < T; t += kLWarps)
      topk_any(a.logits + t, nullptr, E, k, a.renorm, s_pe + static_cast<size_t>(t) * k,
               s_wq + static_cast<size_t>(t) * k, kLMaxT);
    __syncthreads();
    for (int p = tid; p < n; p += kLThreads) {
      a.ids[p] = s_pe[p];
      a.wts[p] = s_wq[p];
    }
    ResolveArgs r = a.res;
    r.slot_ids_sm = s_slot;
    r.num_fetch_sm = &s_nf;
    r.ids_sm = s_pe;
    resolve_block(r, sm + a.sm_r);
    __syncthreads();
    const int nf = min(s_nf, a.max_list);
    for (int i = tid; i < 1 + 3 * n + 2 * nw_fetch; i += kLThreads) {
      uint32_t v = 0;
      if (i == 0) v = static_cast<uint32_t>(nf);
      else if (i < 1 + n) v = static_cast<uint32_t>(s_pe[i - 1]);
      else if (i < 1 + 2 * n) v = static_cast<uint32_t>(s_slot[i - 1 - n]);
      else if (i < 1 + 3 * n) v = __float_as_uint(s_wq[i - 1 - 2 * n]);
      else if (i < 1 + 3 * n + nw_fetch) v = (i - 1 - 3 * n < nf) ? static_cast<uint32_t>(a.fetch_fid[i - 1 - 3 * n]) : 0u;
      else v = (i - 1 - 3 * n - nw_fetch < nf) ? static_cast<uint32_t>(a.fetch_slot[i - 1 - 3 * n - nw_fetch]) : 0u;
      st_relaxed_u64(plan + i, plan_word(tag, v));
    }
    return;
  }

  // activations -> f16 chunks in shared memory, one warp per token, with an
  // exact power-of-two prescale from the token's largest magnitude; one pass
  // over x when a lane holds all its chunks (H <= 2048), else two
  for (int t = warp; t < T; t += kLWarps) {
    const uint16_t* xt = a.x + static_cast<size_t>(t) * H;
    auto load16 = [&](int ch, uint32_t (&raw)[16]) {
      const uint4* src = reinterpret_cast<const uint4*>(xt + 32 * ch);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4 q = __ldcg(src + u);
        raw[4 * u] = q.x;
        raw[4 * u + 1] = q.y;
        raw[4 * u + 2] = q.z;
        raw[4 * u + 3] = q.w;
      }
    };
    auto absmax = [](const uint32_t (&raw)[16], float mx) {
#pragma unroll
      for (int m = 0; m < 16; ++m) mx = fmaxf(mx, fmaxf(fabsf(bf16_lo(raw[m])), fabsf(bf16_hi(raw[m]))));
      return mx;
    };
    auto store = [&](int ch, const uint32_t (&raw)[16], float mul) {
      uint32_t o[16];
      const float sum = pack32<FMT>(raw, mul, o);
      uint32_t* dst = xsm + (static_cast<size_t>(t) * HC + ch) * kXWordsL;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(dst + 4 * q) = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
      dst[16] = __float_as_uint(sum);
    };
    uint32_t r0[16], r1[16];
    float mx = 0.f;
    const int c0 = lane, c1 = lane + 32;
    if (c0 < HC) {
      load16(c0, r0);
      mx = absmax(r0, mx);
    }
    if (c1 < HC) {
      load16(c1, r1);
      mx = absmax(r1, mx);
    }
    for (int ch = lane + 64; ch < HC; ch += 32) {  // H > 2048: a first pass for the max
      uint32_t r2[16];
      load16(ch, r2);
      mx = absmax(r2, mx);
    }
    const float mul = f16_prescale(warp_max(mx));
    if (c0 < HC) store(c0, r0, mul);
    if (c1 < HC) store(c1, r1, mul);
    for (int ch = lane + 64; ch < HC; ch += 32) {  // the second read hits L2 again
      uint32_t r2[16];
      load16(ch, r2);
      store(ch, r2, mul);
    }
    if (lane == 0) s_xinv[t] = 1.f / mul;
  }

  // ---- 3. the leader's plan: thread 0 polls the first word (one load per
  // CTA and poll, so that 151 pollers do not crowd the L2 slices the leader
  // is working through); then every word this CTA needs is loaded at once,
  // and reloaded until all carry this call's tag
  {
    const int nwords = 1 + 3 * n;  // the fetch words are read only when nf > 0
    __shared__ int s_expired[2];   // thread 0's timeout verdict, double-buffered by iteration
    bool ok = true;
    const uint64_t t0 = global_timer_ns();
    if (tid == 0) {
      s_ok = 1;
      for (uint32_t it = 0;; ++it) {
        if (static_cast<uint32_t>(ld_relaxed_u64(plan) >> 32) == tag) break;
        if (global_timer_ns() - t0 > a.wait_ns) {
          record_status(a.dev_status, FT_ERR_TIMEOUT);
          s_ok = 0;
          break;
        }
        __nanosleep(100);
      }
    }
    __syncthreads();
    if (!s_ok) return;  // no copy is in flight
    for (uint32_t it = 0;; ++it) {
      if (tid == 0) s_expired[it & 1] = global_timer_ns() - t0 > a.wait_ns;
      bool mine = true;
      if (tid < nwords) {
        const unsigned long long w = ld_relaxed_u64(plan + tid);
        mine = static_cast<uint32_t>(w >> 32) == tag;
        if (mine) {
          const uint32_t v = static_cast<uint32_t>(w);
          if (tid == 0) s_nf = static_cast<int>(v & 0xffffu);
          else if (tid < 1 + n) s_pe[tid - 1] = static_cast<int>(v);
          else if (tid < 1 + 2 * n) s_slot[tid - 1 - n] = static_cast<int>(v);
          else s_wq[tid - 1 - 2 * n] = __uint_as_float(v);
        }
      }
      if (__syncthreads_and(mine)) break;  // also publishes s_expired[it & 1]
      if (s_expired[it & 1]) {
        if (tid == 0) record_status(a.dev_status, FT_ERR_TIMEOUT);
        ok = false;
        break;
      }
      __nanosleep(32);
    }
    if (!ok) return;  // no copy is in flight
  }
  const int nf = s_nf;
  const int wi = c - 1;  // this worker's index
  unsigned long long target = base + static_cast<unsigned long long>(W);  // the logits arrivals

  // ---- 4. fetch (rare): the workers copy the chosen blocks, then a barrier
  if (nf > 0) {
    const uint64_t v16 = a.block_bytes / 16;
    const uint64_t total = v16 * static_cast<uint64_t>(nf);
    const uint64_t b0 = total * wi / W, b1 = total * (wi + 1) / W;
    constexpr int kV = 8;
    for (uint64_t base = b0 + tid; base < b1; base += static_cast<uint64_t>(kLThreads) * kV) {
      uint4 r[kV];
      uint4* dst[kV];
#pragma unroll
      for (int u = 0; u < kV; ++u) {
        const uint64_t v = base + static_cast<uint64_t>(u) * kLThreads;
        dst[u] = nullptr;
        if (v < b1) {
          const int i = static_cast<int>(v / v16);
          const uint64_t o = v % v16;
          const unsigned long long wf = ld_relaxed_u64(plan + 1 + 3 * n + i);
          const unsigned long long ws = ld_relaxed_u64(plan + 1 + 3 * n + nw_fetch + i);
          const int fid = static_cast<int>(static_cast<uint32_t>(wf));
          const int slot = static_cast<int>(static_cast<uint32_t>(ws));
          if (static_cast<uint32_t>(wf >> 32) == tag && static_cast<uint32_t>(ws >> 32) == tag && fid >= 0 &&
              fid < a.pblocks && slot >= 0 && slot < a.cblocks) {
            r[u] = reinterpret_cast<const uint4*>(a.pool + static_cast<uint64_t>(fid) * a.pstride)[o];
            dst[u] = reinterpret_cast<uint4*>(const_cast<uint8_t*>(a.cache) + static_cast<uint64_t>(slot) * a.cstride) + o;
          } else if (o == 0) {
            record_status(a.dev_status, FT_ERR_BAD_ID);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kV; ++u)
        if (dst[u] != nullptr) *dst[u] = r[u];
    }
    fence_proxy_async_global();  // the copies are read by bulk copies below
    target += static_cast<unsigned long long>(W);
    if (!grid_barrier(a, target, &s_ok)) return;
    fence_proxy_async_global();
  }

  // ---- 5. pairs grouped by distinct expert (warp 0, from the plan in shared
  // memory), combine weights and tensor scales
  if (warp == 0 && n <= 32) {
    // one pair per lane: experts matched with match_any, distinct experts
    // numbered by their first pair, pair lists from ranks within each match
    const int p = lane;
    int e = -1, host = 0;
    const uint8_t* blk = nullptr;
    bool bad = false;
    if (p < n) {
      e = s_pe[p];
      const int sl = s_slot[p];
      if (e >= 0 && e < E) {
        if (sl >= 0) {
          if (sl < a.cblocks) blk = a.cache + static_cast<uint64_t>(sl) * a.cstride;
          else bad = true;
        } else {
          const int64_t fid = static_cast<int64_t>(a.layer) * E + e;
          if (fid < a.pblocks) {
            blk = a.pool + static_cast<uint64_t>(fid) * a.pstride;
            host = 1;
          }
        }
      } else {
        bad = true;
      }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0 && wi == 0) record_status(a.dev_status, FT_ERR_BAD_ID);
    const bool valid = blk != nullptr;
    const unsigned same = __match_any_sync(0xffffffffu, valid ? e : -1 - lane);
    const int first = __ffs(same) - 1;
    const bool lead = valid && first == lane;
    const unsigned leads = __ballot_sync(0xffffffffu, lead);
    const unsigned lt = (1u << lane) - 1u;
    const int d = __popc(leads & ((1u << first) - 1u));  // distinct index of this pair's expert
    const int size = __popc(same);
    int incl = lead ? size : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int start = incl - (lead ? size : 0);  // meaningful on leaders
    const int my_start = __shfl_sync(0xffffffffu, start, first);
    float wq = valid ? s_wq[p] : 0.f;
    if (lead) {
      s_dExpert[d] = e;
      s_dBlk[d] = blk;
      s_dHost[d] = host;
      s_dStart[d] = start;
      float t0v = 1.f, t1v = 1.f;
      if constexpr (FMT == FT_NVFP4) {
        const float* ts = a.tscale + 3 * (static_cast<int64_t>(a.layer) * E + e);
        t0v = __ldg(ts);
        t1v = __ldg(ts + 1);
      }
      s_dts[d][0] = t0v;
      s_dts[d][1] = t1v;
    }
    if (valid) {
      s_dPairs[my_start + __popc(same & lt)] = p;
      if constexpr (FMT == FT_NVFP4) wq *= __ldg(a.tscale + 3 * (static_cast<int64_t>(a.layer) * E + e) + 2);
    }
    if (p < n) {
      s_pd[p] = valid ? d : -1;
      s_pe[p] = valid ? e : -1;
      s_wq[p] = wq;
    }
    const int nd = __popc(leads);
    const int nvalid = __popc(__ballot_sync(0xffffffffu, valid));
    if (lane == 0) {
      s_dStart[nd] = nvalid;
      s_nD = nd;
    }
  } else if (warp == 0) {
    __shared__ int s_first[kLMaxPairs], s_leadd[kLMaxPairs];
    __shared__ const uint8_t* s_pblk[kLMaxPairs];
    __shared__ int s_phost[kLMaxPairs];
    int bad = 0;
    for (int p = lane; p < n; p += 32) {
      const int e = s_pe[p];
      const int sl = s_slot[p];
      const uint8_t* blk = nullptr;
      int host = 0;
      if (e >= 0 && e < E) {
        if (sl >= 0) {
          if (sl < a.cblocks) blk = a.cache + static_cast<uint64_t>(sl) * a.cstride;
          else bad = 1;
        } else {
          const int64_t fid = static_cast<int64_t>(a.layer) * E + e;
          if (fid < a.pblocks) {
            blk = a.pool + static_cast<uint64_t>(fid) * a.pstride;
            host = 1;
          }
        }
      } else {
        bad = 1;
      }
      s_pblk[p] = blk;
      s_phost[p] = host;
      if (blk == nullptr) {
        s_pe[p] = -1;
        s_wq[p] = 0.f;
      }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0 && wi == 0) record_status(a.dev_status, FT_ERR_BAD_ID);
    __syncwarp();
    int nd = 0;
    for (int p0 = 0; p0 < n; p0 += 32) {
      const int p = p0 + lane;
      const int e = p < n ? s_pe[p] : -1;
      int first = -1;
      if (e >= 0) {
        for (int q = 0; q < p; ++q)
          if (s_pe[q] == e) {
            first = q;
            break;
          }
        if (first < 0) first = p;
      }
      const bool lead = e >= 0 && first == p;
      const unsigned m = __ballot_sync(0xffffffffu, lead);
      if (lead) {
        const int d = nd + __popc(m & ((1u << lane) - 1u));
        s_dExpert[d] = e;
        s_dBlk[d] = s_pblk[p];
        s_dHost[d] = s_phost[p];
        s_leadd[p] = d;
      }
      if (p < n) s_first[p] = first;
      nd += __popc(m);
    }
    __syncwarp();
    for (int p = lane; p < n; p += 32) s_pd[p] = s_first[p] >= 0 ? s_leadd[s_first[p]] : -1;
    // pair lists per distinct expert, in pair order: each lane counts the
    // pairs of its experts, a warp scan gives the starts
    int cnt[4] = {0, 0, 0, 0};  // nd <= 128: lane l owns d = l + 32 j
    for (int p = 0; p < n; ++p) {
      const int d = s_pd[p];
      if (d >= 0 && (d & 31) == lane) ++cnt[d >> 5];
    }
    int run = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int incl = cnt[j];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int tot = __shfl_sync(0xffffffffu, incl, 31);
      const int d = lane + 32 * j;
      if (d < nd) s_dStart[d] = run + incl - cnt[j];
      run += tot;
    }
    if (lane == 0) s_dStart[nd] = run;
    __syncwarp();
    for (int p0 = 0; p0 < n; p0 += 32) {  // rank of pair p among the pairs of its expert
      const int p = p0 + lane;
      const int d = p < n ? s_pd[p] : -1;
      if (d >= 0) {
        int rk = 0;
        for (int q = 0; q < p; ++q) rk += s_pd[q] == d;
        s_dPairs[s_dStart[d] + rk] = p;
      }
    }
    for (int d = lane; d < nd; d += 32) {
      float t0v = 1.f, t1v = 1.f, t2v = 1.f;
      if constexpr (FMT == FT_NVFP4) {
        const float* ts = a.tscale + 3 * (static_cast<int64_t>(a.layer) * E + s_dExpert[d]);
        t0v = __ldg(ts);
        t1v = __ldg(ts + 1);
        t2v = __ldg(ts + 2);
      }
      s_dts[d][0] = t0v;
      s_dts[d][1] = t1v;
      (void)t2v;
    }
    if constexpr (FMT == FT_NVFP4) {
      for (int p = lane; p < n; p += 32)
        if (s_pd[p] >= 0) s_wq[p] *= __ldg(a.tscale + 3 * (static_cast<int64_t>(a.layer) * E + s_pe[p]) + 2);
    }
    if (lane == 0) s_nD = nd;
  }
  __syncthreads();
  const int nD = s_nD;

  // ---- 6. this worker's bytes: its gate/up rows (units [u0, u1) of the
  // (distinct expert, qg rows) space, cut into segments at expert boundaries)
  // and its down rows [h0, h1) of every distinct expert, all requested at once
  const int upe = I / a.qg;
  const int64_t N = static_cast<int64_t>(nD) * upe;
  const int u0 = static_cast<int>(N * wi / W), u1 = static_cast<int>(N * (wi + 1) / W);
  const int hq = H / a.qd;
  const int h0 = static_cast<int>(static_cast<int64_t>(hq) * wi / W) * a.qd;
  const int h1 = static_cast<int>(static_cast<int64_t>(hq) * (wi + 1) / W) * a.qd;
  const int nr = h1 - h0;
  uint8_t* gsm = sm + a.sm_r;
  uint8_t* dsm = sm + a.sm_d;
  // segment j of this CTA covers the units of distinct expert d0 + j inside
  // [u0, u1); its rows sit at offset (first unit - u0) * qg * 2 * (rowA + sbA)
  if (warp == 0) {
    const int d0 = u1 > u0 ? u0 / upe : 0;
    const int j = lane;
    const int us = max(u0, (d0 + j) * upe), ue = min(u1, (d0 + j + 1) * upe);
    const bool has = j < kLMaxSegs && us < ue;
    if (has) {
      s_segD[j] = d0 + j;
      s_segR0[j] = (us % upe) * a.qg;
      s_segN[j] = (ue - us) * a.qg;
      s_segOff[j] = static_cast<uint32_t>(us - u0) * static_cast<uint32_t>(a.qg) * 2u * (a.rowA + a.sbA);
      const int d = d0 + j;
      if (!s_dHost[d]) {
        const uint32_t rows = static_cast<uint32_t>(ue - us) * static_cast<uint32_t>(a.qg);
        const uint64_t r0 = static_cast<uint64_t>(s_segR0[j]);
        uint8_t* dst = gsm + s_segOff[j];
        const uint8_t* blk = s_dBlk[d];
        mbar_arrive_expect_tx(&bars[2 + j], 2u * rows * (a.rowA + a.sbA));
        bulk_g2s(dst, blk + a.off[0] + r0 * a.rowA, rows * a.rowA, &bars[2 + j]);
        bulk_g2s(dst + rows * a.rowA, blk + a.off[1] + r0 * a.rowA, rows * a.rowA, &bars[2 + j]);
        bulk_g2s(dst + 2u * rows * a.rowA, blk + a.off[3] + r0 * a.sbA, rows * a.sbA, &bars[2 + j]);
        bulk_g2s(dst + 2u * rows * a.rowA + rows * a.sbA, blk + a.off[4] + r0 * a.sbA, rows * a.sbA, &bars[2 + j]);
      }
    }
    const int nseg = __popc(__ballot_sync(0xffffffffu, has));
    if (lane == 0) s_nseg = nseg;
  } else if (warp == 1 && nr > 0) {
    uint32_t nd_dev = 0;
    for (int d = lane; d < nD; d += 32) nd_dev += !s_dHost[d];
    nd_dev = __reduce_add_sync(0xffffffffu, nd_dev);
    if (nd_dev > 0) {
      if (lane == 0) mbar_arrive_expect_tx(&bars[1], nd_dev * static_cast<uint32_t>(nr) * (a.rowB + a.sbB));
      __syncwarp();
      for (int d = lane; d < nD; d += 32) {
        if (s_dHost[d]) continue;
        uint8_t* slab = dsm + static_cast<size_t>(d) * a.dslab;
        const uint8_t* blk = s_dBlk[d];
        bulk_g2s(slab, blk + a.off[2] + static_cast<uint64_t>(h0) * a.rowB, static_cast<uint32_t>(nr) * a.rowB,
                 &bars[1]);
        bulk_g2s(slab + static_cast<size_t>(a.drows) * a.rowB, blk + a.off[5] + static_cast<uint64_t>(h0) * a.sbB,
                 static_cast<uint32_t>(nr) * a.sbB, &bars[1]);
      }
    }
  }
  __syncthreads();
  const int nseg = s_nseg;
  // host-path experts (the pool, read in place): plain loads by the CTA
  bool any_host = false;
  for (int sg = 0; sg < nseg; ++sg) {
    const int d = s_segD[sg];
    if (!s_dHost[d]) continue;
    any_host = true;
    const uint32_t rows = static_cast<uint32_t>(s_segN[sg]);
    const uint64_t r0 = static_cast<uint64_t>(s_segR0[sg]);
    uint8_t* dst = gsm + s_segOff[sg];
    const uint8_t* blk = s_dBlk[d];
    cta_copy(dst, blk + a.off[0] + r0 * a.rowA, rows * a.rowA);
    cta_copy(dst + rows * a.rowA, blk + a.off[1] + r0 * a.rowA, rows * a.rowA);
    cta_copy(dst + 2u * rows * a.rowA, blk + a.off[3] + r0 * a.sbA, rows * a.sbA);
    cta_copy(dst + 2u * rows * a.rowA + rows * a.sbA, blk + a.off[4] + r0 * a.sbA, rows * a.sbA);
  }
  if (nr > 0)
    for (int d = 0; d < nD; ++d) {
      if (!s_dHost[d]) continue;
      any_host = true;
      uint8_t* slab = dsm + static_cast<size_t>(d) * a.dslab;
      cta_copy(slab, s_dBlk[d] + a.off[2] + static_cast<uint64_t>(h0) * a.rowB, static_cast<uint32_t>(nr) * a.rowB);
      cta_copy(slab + static_cast<size_t>(a.drows) * a.rowB, s_dBlk[d] + a.off[5] + static_cast<uint64_t>(h0) * a.sbB,
               static_cast<uint32_t>(nr) * a.sbB);
    }
  if (any_host) __syncthreads();

  // ---- 7. gate/up: warp w takes the CTA's rows w, w + 16, ... as their
  // segment lands, and writes h = silu(g) * u for every pair of that expert
  bool seg_ok = true;
  {
    int sg = 0, base = 0;
    uint32_t waited = 0;
    const int total_rows = (u1 - u0) * a.qg;
    for (int rr = warp; rr < total_rows; rr += kLWarps) {
      while (rr >= base + s_segN[sg]) {
        base += s_segN[sg];
        ++sg;
      }
      const int d = s_segD[sg];
      if (!s_dHost[d] && !((waited >> sg) & 1u)) {
        if (!mbar_wait_lim(&bars[2 + sg], 0, a.dev_status, a.wait_ns)) {
          seg_ok = false;
          break;
        }
        waited |= 1u << sg;
      }
      const uint32_t rows = static_cast<uint32_t>(s_segN[sg]);
      const int q = rr - base;
      const uint8_t* sbase = gsm + s_segOff[sg];
      const uint8_t* grow = sbase + static_cast<size_t>(q) * a.rowA;
      const uint8_t* urow = sbase + static_cast<size_t>(rows) * a.rowA + static_cast<size_t>(q) * a.rowA;
      const uint8_t* gsr = sbase + 2u * rows * a.rowA + static_cast<size_t>(q) * a.sbA;
      const uint8_t* usr = sbase + 2u * rows * a.rowA + rows * a.sbA + static_cast<size_t>(q) * a.sbA;
      const int r = s_segR0[sg] + q;
      const float ts0 = s_dts[d][0], ts1 = s_dts[d][1];
      for (int i = s_dStart[d]; i < s_dStart[d + 1]; ++i) {
        const int p = s_dPairs[i], t = p / k;
        float gacc = 0.f, uacc = 0.f;
        for (int ch = lane; ch < HC; ch += 32) {
          const uint32_t* xs = xsm + (static_cast<size_t>(t) * HC + ch) * kXWordsL;
          uint32_t xa[16];
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            const uint4 v = *reinterpret_cast<const uint4*>(xs + 4 * qq);
            xa[4 * qq] = v.x;
            xa[4 * qq + 1] = v.y;
            xa[4 * qq + 2] = v.z;
            xa[4 * qq + 3] = v.w;
          }
          const float asum = __uint_as_float(xs[16]);
          const uint4 wg = *reinterpret_cast<const uint4*>(grow + 16 * ch);
          const uint4 wu = *reinterpret_cast<const uint4*>(urow + 16 * ch);
          gacc += chunk_dot<FMT>(wg, smem_scale<FMT>(gsr, ch, a.gshift), xa, asum);
          uacc += chunk_dot<FMT>(wu, smem_scale<FMT>(usr, ch, a.gshift), xa, asum);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          gacc += __shfl_xor_sync(0xffffffffu, gacc, o);
          uacc += __shfl_xor_sync(0xffffffffu, uacc, o);
        }
        if (lane < kLHRep) {  // every lane holds the sums: lane j writes replica j
          const float gv = gacc * (ts0 * s_xinv[t]), uv = uacc * (ts1 * s_xinv[t]);
          a.h[a.h_rep * lane + static_cast<size_t>(p) * I + r] = gv / (1.f + expf(-gv)) * uv;
        }
      }
    }
  }
  if (!seg_ok) {
    // wait (bounded) for this CTA's copies still in flight, then leave: the
    // other CTAs' barrier waits run out too
    for (int sg = 0; sg < nseg; ++sg) mbar_wait_lim(&bars[2 + sg], 0, nullptr, a.wait_ns);
    if (nr > 0) mbar_wait_lim(&bars[1], 0, nullptr, a.wait_ns);
    return;
  }

  // ---- 8. h complete on every worker, then the down rows and the combine
  target += static_cast<unsigned long long>(W);
  const bool bar_ok = grid_barrier(a, target, &s_ok);
  bool down_ok = true;
  if (nr > 0) {
    bool dev_down = false;
    for (int d = 0; d < nD; ++d) dev_down |= !s_dHost[d];
    if (dev_down) down_ok = mbar_wait_lim(&bars[1], 0, a.dev_status, a.wait_ns);
  }
  if (!bar_ok || !down_ok || nr == 0) return;
  // h of every valid pair as f16 chunks with an exact power-of-two prescale
  // per pair (absorbed into its combine weight): one pass over h, a warp per
  // pair, each lane holding its chunks (I <= 4096: four chunks a lane)
  uint8_t* hsm = sm + a.sm_h;
  float* hsum = reinterpret_cast<float*>(hsm + static_cast<size_t>(n) * IC * kChunkBytes);
  for (int p = warp; p < n; p += kLWarps) {
    if (s_pd[p] < 0) continue;
    const float* hp = a.h + a.h_rep * (wi % kLHRep) + static_cast<size_t>(p) * I;
    float v[32];
    float m = 0.f;
    for (int ch = lane; ch < IC; ch += 32) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 f = __ldcg(reinterpret_cast<const float4*>(hp + 32 * ch + 4 * q));
        v[4 * q] = f.x;
        v[4 * q + 1] = f.y;
        v[4 * q + 2] = f.z;
        v[4 * q + 3] = f.w;
        m = fmaxf(m, fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w))));
      }
    }
    const float mul = f16_prescale(warp_max(m));
    for (int ch = lane; ch < IC; ch += 32) {
      if (IC > 32) {  // reload: the registers held only the last chunk
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 f = __ldcg(reinterpret_cast<const float4*>(hp + 32 * ch + 4 * q));
          v[4 * q] = f.x;
          v[4 * q + 1] = f.y;
          v[4 * q + 2] = f.z;
          v[4 * q + 3] = f.w;
        }
      }
      uint32_t o[16];
      hsum[static_cast<size_t>(p) * IC + ch] = pack32<FMT>(v, mul, o);
      uint8_t* dst = hsm + (static_cast<size_t>(p) * IC + ch) * kChunkBytes;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(dst + 16 * q) = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
    }
    if (lane == 0) s_wq[p] /= mul;
  }
  __syncthreads();
  // units (row, token): LPR lanes per pair, 32 / LPR pairs at once
  const int LPR = IC <= 8 ? 8 : (IC <= 16 ? 16 : 32);
  const int SPLIT = 32 / LPR;
  const int grp = lane / LPR, sub = lane % LPR;
  for (int u = warp; u < nr * T; u += kLWarps) {
    const int r = u / T, t = u % T;
    float acc = 0.f;
    for (int j = grp; j < k; j += SPLIT) {
      const int p = t * k + j;
      const int d = s_pd[p];
      if (d < 0) continue;
      const uint8_t* slab = dsm + static_cast<size_t>(d) * a.dslab;
      const uint8_t* crow = slab + static_cast<size_t>(r) * a.rowB;
      const uint8_t* srow = slab + static_cast<size_t>(a.drows) * a.rowB + static_cast<size_t>(r) * a.sbB;
      float sacc = 0.f;
      for (int ch = sub; ch < IC; ch += LPR) {
        const uint8_t* hc = hsm + (static_cast<size_t>(p) * IC + ch) * kChunkBytes;
        uint32_t ha[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 vv = *reinterpret_cast<const uint4*>(hc + 16 * q);
          ha[4 * q] = vv.x;
          ha[4 * q + 1] = vv.y;
          ha[4 * q + 2] = vv.z;
          ha[4 * q + 3] = vv.w;
        }
        const uint4 w = *reinterpret_cast<const uint4*>(crow + 16 * ch);
        sacc += chunk_dot<FMT>(w, smem_scale<FMT>(srow, ch, a.gshift), ha, hsum[static_cast<size_t>(p) * IC + ch]);
      }
      acc = fmaf(s_wq[p], sacc, acc);
    }
    // within each lane group first, then across the groups (the pair-major
    // down kernels' order)
    for (int o = LPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    for (int o = LPR; o < 32; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
      const size_t idx = static_cast<size_t>(t) * H + h0 + r;
      if (a.out_bf16) static_cast<uint16_t*>(a.out)[idx] = f32_to_bf16(acc);
      else static_cast<float*>(a.out)[idx] = acc;
    }
  }
}

// Workspace: the counter and the generation word (own 128-byte lines), the
// plan words, the logits, then h.
constexpr size_t kLBarBytes = 256;
size_t layer_plan_bytes(int n, int max_list) {
  return ((static_cast<size_t>(1 + 3 * n + 2 * max_list) * 8) + 255) & ~static_cast<size_t>(255);
}
size_t layer_h_rep_floats(int n, int I) {  // one replica of h, padded to 256 bytes
  return ((static_cast<size_t>(n) * I * sizeof(float) + 255) & ~static_cast<size_t>(255)) / sizeof(float);
}
size_t layer_logits_bytes(int T, int E) {  // [E][kLMaxT]: one 32-byte sector per expert
  (void)T;
  return (static_cast<size_t>(E) * kLMaxT * sizeof(float) + 255) & ~static_cast<size_t>(255);
}

uint64_t g_wait_limit_ns = kWaitLimitNs;

}  // namespace
}  // namespace ft

extern "C" {

size_t ft_moe_decode_layer_workspace(int32_t T, int32_t k, int32_t H, int32_t I, int32_t E) {
  if (T <= 0 || k <= 0 || H <= 0 || I <= 0 || E <= 0) return 0;
  (void)H;
  const size_t hb = ft::layer_h_rep_floats(T * k, I) * sizeof(float) * ft::kLHRep;
  return ft::kLBarBytes + ft::layer_plan_bytes(T * k, T * k) + ft::layer_logits_bytes(T, E) + hb;
}

ft_status ft_set_wait_limit_ns(uint64_t ns) {
  ft::g_wait_limit_ns = ns == 0 ? ft::kWaitLimitNs : ns;
  return FT_OK;
}

ft_status ft_moe_decode_layer(const uint16_t* x, int32_t T, const float* w_router, int32_t k, int32_t renorm,
                              const ft_cache_state* state, int32_t layer, int32_t frac_q16, const ft_bank* cache,
                              const ft_bank* pool, int32_t* topk_ids, float* topk_w, int32_t* slot_ids,
                              int32_t* num_fetch, int32_t* fetch_fid, int32_t* fetch_slot, int32_t max_list,
                              void* out, int32_t out_dtype, void* ws, size_t ws_bytes, int32_t* dev_status,
                              void* stream) {
  using namespace ft;
  Layout L;
  ft_status st = check_bank(cache, "decode layer cache", &L);
  if (st != FT_OK) return st;
  FT_REQUIRE(pool != nullptr, "decode layer: the pool (source of truth) is required");
  {
    Layout Lp;
    if ((st = check_bank(pool, "decode layer pool", &Lp)) != FT_OK) return st;
    FT_REQUIRE(pool->fmt == cache->fmt && pool->H == cache->H && pool->I == cache->I && pool->group == cache->group,
               "decode layer: pool and cache shapes differ");
    FT_REQUIRE(pool->stride % 16 == 0 && reinterpret_cast<uintptr_t>(pool->base) % 16 == 0,
               "decode layer: pool blocks must be 16-byte aligned");
  }
  FT_REQUIRE(state != nullptr, "decode layer: state is NULL");
  const int E = state->E, H = cache->H, I = cache->I;
  FT_REQUIRE(T >= 1 && T <= kLMaxT, "decode layer: T=%d outside [1, %d]", T, kLMaxT);
  FT_REQUIRE(k >= 1 && k <= E && k <= 32 && T * k <= kLMaxPairs, "decode layer: k=%d (T*k <= %d, k <= min(E, 32))",
             k, kLMaxPairs);
  FT_REQUIRE(E >= 1 && E <= kLMaxE, "decode layer: E=%d outside [1, %d]", E, kLMaxE);
  FT_REQUIRE(H <= 4096 && I <= 4096, "decode layer: H, I must be <= 4096");
  FT_REQUIRE(out_dtype == FT_OUT_F32 || out_dtype == FT_OUT_BF16, "decode layer: bad out_dtype");
  FT_REQUIRE(x && w_router && topk_ids && topk_w && slot_ids && out && ws, "decode layer: NULL pointer");
  FT_REQUIRE(reinterpret_cast<uintptr_t>(x) % 16 == 0 && reinterpret_cast<uintptr_t>(w_router) % 16 == 0 &&
                 reinterpret_cast<uintptr_t>(ws) % 256 == 0,
             "decode layer: x and w_router must be 16-byte aligned, ws 256-byte aligned");
  FT_REQUIRE(cache->stride % 16 == 0 && reinterpret_cast<uintptr_t>(cache->base) % 16 == 0,
             "decode layer: cache blocks must be 16-byte aligned");
  FT_REQUIRE(ws_bytes >= ft_moe_decode_layer_workspace(T, k, H, I, E), "decode layer: workspace %zu < %zu", ws_bytes,
             ft_moe_decode_layer_workspace(T, k, H, I, E));
  const int G = device_sm_count();
  FT_REQUIRE(E <= kLMaxRouterRows * G, "decode layer: E=%d > %d router rows per CTA x %d CTAs", E,
             kLMaxRouterRows, G);

  LayerArgs a = {};
  a.x = x;
  a.W = w_router;
  a.T = T;
  a.H = H;
  a.E = E;
  a.k = k;
  a.renorm = renorm ? 1 : 0;
  a.I = I;
  a.gshift = cache->fmt == FT_INT4 ? (cache->group == 32 ? 0 : (cache->group == 64 ? 1 : 2)) : 0;
  a.layer = layer;
  a.G = G;
  a.cache = static_cast<const uint8_t*>(cache->base);
  a.cstride = cache->stride;
  a.cblocks = cache->n_blocks;
  a.pool = static_cast<const uint8_t*>(pool->base);
  a.pstride = pool->stride;
  a.pblocks = pool->n_blocks;
  a.tscale = cache->tensor_scale;
  for (int i = 0; i < 6; ++i) a.off[i] = L.off[i];
  a.rowA = static_cast<uint32_t>(H / 2);
  a.rowB = static_cast<uint32_t>(I / 2);
  if (cache->fmt == FT_INT4) {
    a.sbA = static_cast<uint32_t>(H / cache->group * 2);
    a.sbB = static_cast<uint32_t>(I / cache->group * 2);
  } else {
    a.sbA = static_cast<uint32_t>(H / 16);
    a.sbB = static_cast<uint32_t>(I / 16);
  }
  a.block_bytes = L.total;
  FT_REQUIRE(L.total % 16 == 0, "decode layer: block size %llu not a multiple of 16",
             static_cast<unsigned long long>(L.total));
  // rows per unit so that a unit's scale rows are a multiple of 16 bytes
  auto rows_for = [](uint32_t sb) {
    int q = 1;
    while ((q * sb) % 16 != 0) q *= 2;
    return q;
  };
  a.qg = rows_for(a.sbA);
  a.qd = rows_for(a.sbB);
  FT_REQUIRE(I % a.qg == 0 && H % a.qd == 0, "decode layer: rows do not split into 16-byte scale groups");
  a.ids = topk_ids;
  a.wts = topk_w;
  a.slot_ids = slot_ids;
  a.num_fetch = num_fetch;
  a.fetch_fid = fetch_fid;
  a.fetch_slot = fetch_slot;
  a.max_list = max_list;
  a.out = out;
  a.out_bf16 = out_dtype == FT_OUT_BF16;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  a.bar = reinterpret_cast<unsigned long long*>(w8 + 128);
  const size_t plan_b = layer_plan_bytes(T * k, T * k);
  a.plan = reinterpret_cast<unsigned long long*>(w8 + kLBarBytes);
  a.logits = reinterpret_cast<float*>(w8 + kLBarBytes + plan_b);
  a.h = reinterpret_cast<float*>(w8 + kLBarBytes + plan_b + layer_logits_bytes(T, E));
  a.h_rep = layer_h_rep_floats(T * k, I);
  FT_REQUIRE(max_list >= 0 && max_list <= T * k, "decode layer: max_list %d outside [0, T*k = %d]", max_list, T * k);
  a.dev_status = dev_status;
  a.wait_ns = g_wait_limit_ns;

  // shared memory: x chunks | router rows / resolve / gate-up slots | down slabs | h chunks | barriers
  const void* fn = cache->fmt == FT_INT4 ? reinterpret_cast<const void*>(layer_kernel<FT_INT4>)
                                         : reinterpret_cast<const void*>(layer_kernel<FT_NVFP4>);
  size_t cap = 0;  // dynamic bytes: the per-block opt-in limit less the kernel's static tables
  {
    cudaFuncAttributes fa;
    cudaError_t fe = cudaFuncGetAttributes(&fa, fn);
    if (fe != cudaSuccess) return fail(FT_ERR_CUDA, "decode layer: %s", cudaGetErrorString(fe));
    const size_t optin = static_cast<size_t>(device_smem_optin());
    FT_REQUIRE(optin > fa.sharedSizeBytes + 1024, "decode layer: no shared memory left for the plan");
    cap = optin - fa.sharedSizeBytes - 1024;
  }
  const int n = T * k;
  const int W = G - 1;  // workers: every CTA but the leader
  FT_REQUIRE(W >= 1, "decode layer: needs at least two SMs");
  const size_t xs = static_cast<size_t>(T) * (H / 32) * kXWordsL * 4;
  a.drows = (((H / a.qd) + W - 1) / W) * a.qd;
  a.dslab = static_cast<uint32_t>((static_cast<size_t>(a.drows) * (a.rowB + a.sbB) + 15) & ~static_cast<size_t>(15));
  const size_t ds = static_cast<size_t>(n) * a.dslab;
  const size_t hs = static_cast<size_t>(n) * (I / 32) * (kChunkBytes + 4);
  const int64_t units = static_cast<int64_t>(n) * (I / a.qg);
  a.grows = static_cast<int>((units + W - 1) / W) * a.qg;
  FT_REQUIRE((a.grows + I - 1) / I + 1 <= kLMaxSegs, "decode layer: %d gate/up rows per CTA span too many experts",
             a.grows);
  const size_t gs = static_cast<size_t>(a.grows) * 2 * (a.rowA + a.sbA);
  // region R holds the router rows, then (leader) the resolve's arrays, then
  // (workers) the gate/up rows; the rest is fixed
  const size_t fixed = ((xs + 127) & ~static_cast<size_t>(127)) + ((ds + 127) & ~static_cast<size_t>(127)) +
                       ((hs + 127) & ~static_cast<size_t>(127)) + (2 + kLMaxSegs) * 8;
  const size_t router_bytes = static_cast<size_t>(kLMaxRouterRows) * H * 4;
  size_t rsz = gs > router_bytes ? gs : router_bytes;
  FT_REQUIRE(fixed + rsz <= cap, "decode layer: T=%d k=%d H=%d I=%d needs %zu bytes of shared memory (> %zu)", T, k,
             H, I, fixed + rsz, cap);
  // the leader's resolve uses region R too, staging the slot state in shared
  // memory when it fits in what is left
  ResolveArgs ra;
  size_t res_smem = 0;
  st = resolve_prepare(state, layer, topk_ids, T, k, frac_q16, slot_ids, num_fetch, fetch_fid, fetch_slot, max_list,
                       dev_status, "decode layer", cap - fixed, &ra, &res_smem);
  if (st != FT_OK) return st;
  if (res_smem > rsz) rsz = res_smem;
  a.res = ra;
  size_t off = 0;
  a.sm_r = static_cast<uint32_t>(off);
  off += (rsz + 127) & ~static_cast<size_t>(127);
  a.sm_x = static_cast<uint32_t>(off);
  off += (xs + 127) & ~static_cast<size_t>(127);
  a.sm_d = static_cast<uint32_t>(off);
  off += (ds + 127) & ~static_cast<size_t>(127);
  a.sm_h = static_cast<uint32_t>(off);
  off += (hs + 127) & ~static_cast<size_t>(127);
  a.sm_bar = static_cast<uint32_t>(off);
  off += (2 + kLMaxSegs) * 8;
  FT_REQUIRE(off <= cap, "decode layer: shared memory %zu > %zu", off, cap);

  st = ensure_dyn_smem(fn, static_cast<int>(off), "decode layer");
  if (st != FT_OK) return st;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(kLThreads);
  cfg.dynamicSmemBytes = off;
  cfg.stream = as_stream(stream);
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  at[1].id = cudaLaunchAttributeCooperative;
  at[1].val.cooperative = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  cudaError_t e = cache->fmt == FT_INT4 ? cudaLaunchKernelEx(&cfg, layer_kernel<FT_INT4>, a)
                                        : cudaLaunchKernelEx(&cfg, layer_kernel<FT_NVFP4>, a);
  if (e != cudaSuccess) return fail(FT_ERR_CUDA, "decode layer: %s", cudaGetErrorString(e));
  return launch_check("decode layer");
}

}  // extern "C"
