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
constexpr int kLMaxSlots = 4;        // gate/up slots per warp
constexpr int kXWordsL = 20;         // words per staged activation chunk (16 f16x2 + sum + pad)

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
  uint32_t* ctr;  // arrival counter (wraps to 0 at G)
  uint32_t* gen;  // generation word, advanced once per hand-off
  float* logits;  // [T, E]
  float* h;       // [T * k, I] fp32
  int32_t* dev_status;
  uint64_t wait_ns;
  int qg;               // gate/up rows per unit (scale rows 16-byte aligned)
  int qd;               // alignment of the down row ranges
  int nslot;            // gate/up slots per warp
  uint32_t unit_bytes;  // one slot: qg gate rows, qg up rows, their scales
  int drows;            // most down rows a CTA owns
  uint32_t dslab;       // one distinct expert's down rows in shared memory
  uint32_t sm_x, sm_r, sm_d, sm_h, sm_bar;
};

__device__ __forceinline__ int32_t ld_cg_i32(const int32_t* p) { return __ldcg(p); }

// Wait (thread 0) until the generation word moves past g; false, with
// FT_ERR_TIMEOUT recorded, after limit_ns.
__device__ bool wait_gen(const uint32_t* gen, uint32_t g, uint64_t limit_ns, int32_t* status) {
  if (ld_acquire_gpu(gen) != g) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    __nanosleep(20);
    if (ld_acquire_gpu(gen) != g) return true;
    if ((i & 31u) == 0 && global_timer_ns() - t0 > limit_ns) {
      record_status(status, FT_ERR_TIMEOUT);
      return false;
    }
  }
}

// Every thread of every CTA calls it; true (CTA-uniform) once all G CTAs
// have arrived, false on timeout.  Writes before it (any proxy fenced by the
// caller) are visible to every CTA after it.
__device__ bool grid_barrier(const LayerArgs& a, int* s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t g = ld_acquire_gpu(a.gen);  // cannot move before this CTA arrives
    __threadfence();
    const uint32_t old = atom_inc_acq_rel_gpu(a.ctr, static_cast<uint32_t>(a.G - 1));
    bool ok = true;
    if (old == static_cast<uint32_t>(a.G - 1))
      st_release_gpu(a.gen, g + 1);
    else
      ok = wait_gen(a.gen, g, a.wait_ns, a.dev_status);
    __threadfence();
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
    if ((i & 255u) == 0 && global_timer_ns() - t0 > limit_ns) {
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

// One warp copies `bytes` (a multiple of 16) with plain loads (host memory).
__device__ __forceinline__ void warp_copy(uint8_t* dst, const uint8_t* src, uint32_t bytes, int lane) {
  for (uint32_t o = 16u * lane; o < bytes; o += 16u * 32u)
    *reinterpret_cast<uint4*>(dst + o) = *reinterpret_cast<const uint4*>(src + o);
}

template <int FMT>
__global__ void __launch_bounds__(kLThreads, 1) layer_kernel(const __grid_constant__ LayerArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ int s_ok, s_leader, s_skip, s_nf, s_nD;
  __shared__ uint32_t s_gen, s_dbytes;
  __shared__ float s_part[kLWarps][kLMaxRouterRows * kLMaxT];
  __shared__ float s_xinv[kLMaxT];
  __shared__ int s_pe[kLMaxPairs], s_first[kLMaxPairs], s_leadd[kLMaxPairs], s_phost[kLMaxPairs];
  __shared__ const uint8_t* s_pblk[kLMaxPairs];
  __shared__ int s_pd[kLMaxPairs];  // distinct-expert index of each pair, -1 if masked
  __shared__ float s_wq[kLMaxPairs];
  __shared__ int s_dExpert[kLMaxPairs], s_dHost[kLMaxPairs], s_dStart[kLMaxPairs + 1], s_dPairs[kLMaxPairs];
  __shared__ const uint8_t* s_dBlk[kLMaxPairs];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, G = a.G;
  const int T = a.T, H = a.H, E = a.E, k = a.k, I = a.I;
  const int HC = H / 32, IC = I / 32;
  const int n = T * k;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + a.sm_bar);  // [0] router, [1] down, [2..] gate/up slots
  float* wrows = reinterpret_cast<float*>(sm + a.sm_r);
  uint32_t* xsm = reinterpret_cast<uint32_t*>(sm + a.sm_x);

  // ---- 0. this CTA's router rows, before the wait: no kernel writes them
  int nrows = 0;
  for (int e = c; e < E && nrows < kLMaxRouterRows; e += G) ++nrows;
  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    for (int i = 0; i < kLWarps * a.nslot; ++i) mbar_init(&bars[2 + i], 1);
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
    s_gen = ld_acquire_gpu(a.gen);
    s_dbytes = 0;
  }
  __syncthreads();
  const bool router_ok = nrows == 0 || mbar_wait_lim(&bars[0], 0, a.dev_status, a.wait_ns);
  if (s_skip || !router_ok) return;  // an earlier wait gave up: do nothing (no copy is in flight now)

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
      a.logits[static_cast<size_t>(t) * E + c + G * i] = v;
    }
  }
  // ---- 2. arrival: the last CTA becomes the leader
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const uint32_t old = atom_inc_acq_rel_gpu(a.ctr, static_cast<uint32_t>(G - 1));
    s_leader = old == static_cast<uint32_t>(G - 1);
  }
  __syncthreads();

  // activations -> f16 chunks in shared memory, one warp per token, with an
  // exact power-of-two prescale from the token's largest magnitude
  auto stage_x = [&]() {
    for (int t = warp; t < T; t += kLWarps) {
      const uint16_t* xt = a.x + static_cast<size_t>(t) * H;
      float mx = 0.f;
      for (int ch = lane; ch < HC; ch += 32) {
        const uint4* src = reinterpret_cast<const uint4*>(xt + 32 * ch);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 q = __ldcg(src + u);
          const uint32_t v4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int m = 0; m < 4; ++m) mx = fmaxf(mx, fmaxf(fabsf(bf16_lo(v4[m])), fabsf(bf16_hi(v4[m]))));
        }
      }
      const float mul = f16_prescale(warp_max(mx));
      for (int ch = lane; ch < HC; ch += 32) {
        uint32_t raw[16];
        const uint4* src = reinterpret_cast<const uint4*>(xt + 32 * ch);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 q = __ldcg(src + u);
          raw[4 * u] = q.x;
          raw[4 * u + 1] = q.y;
          raw[4 * u + 2] = q.z;
          raw[4 * u + 3] = q.w;
        }
        uint32_t o[16];
        const float sum = pack32<FMT>(raw, mul, o);
        uint32_t* dst = xsm + (static_cast<size_t>(t) * HC + ch) * kXWordsL;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4*>(dst + 4 * q) = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
        dst[16] = __float_as_uint(sum);
      }
      if (lane == 0) s_xinv[t] = 1.f / mul;
    }
  };

  if (s_leader) {
    // softmax + top-k (one warp per token), then the resolve by the whole CTA
    for (int t = warp; t < T; t += kLWarps)
      topk_any(a.logits + static_cast<size_t>(t) * E, nullptr, E, k, a.renorm, a.ids + static_cast<size_t>(t) * k,
               a.wts + static_cast<size_t>(t) * k);
    __syncthreads();
    resolve_block(a.res, sm + a.sm_r);
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      st_release_gpu(a.gen, s_gen + 1);
    }
    stage_x();
  } else {
    stage_x();
    if (tid == 0) s_ok = wait_gen(a.gen, s_gen, a.wait_ns, a.dev_status);
    __syncthreads();
    if (!s_ok) return;
  }
  __syncthreads();
  if (tid == 0) s_nf = min(ld_cg_i32(a.num_fetch), a.max_list);
  __syncthreads();

  // ---- 3. fetch (rare): every CTA copies its share, then a grid barrier
  const int nf = s_nf;
  if (nf > 0) {
    const uint64_t v16 = a.block_bytes / 16;
    const uint64_t total = v16 * static_cast<uint64_t>(nf);
    const uint64_t b0 = total * c / G, b1 = total * (c + 1) / G;
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
          const int fid = ld_cg_i32(a.fetch_fid + i), slot = ld_cg_i32(a.fetch_slot + i);
          if (fid >= 0 && fid < a.pblocks && slot >= 0 && slot < a.cblocks) {
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
    if (!grid_barrier(a, &s_ok)) return;
    fence_proxy_async_global();
  }

  // ---- 4. pairs grouped by distinct expert (warp 0), combine weights
  if (warp == 0) {
    for (int p = lane; p < n; p += 32) {
      const int e = ld_cg_i32(a.ids + p);
      const int s = ld_cg_i32(a.slot_ids + p);
      const uint8_t* blk = nullptr;
      int host = 0;
      if (e >= 0 && e < E) {
        if (s >= 0) {
          if (s < a.cblocks) blk = a.cache + static_cast<uint64_t>(s) * a.cstride;
          else if (c == 0) record_status(a.dev_status, FT_ERR_BAD_ID);
        } else if (a.pool != nullptr) {
          const int64_t fid = static_cast<int64_t>(a.layer) * E + e;
          if (fid < a.pblocks) {
            blk = a.pool + static_cast<uint64_t>(fid) * a.pstride;
            host = 1;
          }
        }
      } else if (c == 0) {
        record_status(a.dev_status, FT_ERR_BAD_ID);
      }
      s_pe[p] = blk != nullptr ? e : -1;
      s_pblk[p] = blk;
      s_phost[p] = host;
      float wq = 0.f;
      if (blk != nullptr) {
        wq = __ldcg(a.wts + p);
        if constexpr (FMT == FT_NVFP4) wq *= __ldg(a.tscale + 3 * (static_cast<int64_t>(a.layer) * E + e) + 2);
      }
      s_wq[p] = wq;
    }
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
    __syncwarp();
    if (lane == 0) {
      // pair lists in pair order per distinct expert
      for (int d = 0; d <= nd; ++d) s_dStart[d] = 0;
      for (int p = 0; p < n; ++p)
        if (s_pd[p] >= 0) ++s_dStart[s_pd[p] + 1];
      for (int d = 0; d < nd; ++d) s_dStart[d + 1] += s_dStart[d];
      int pos[kLMaxPairs];
      for (int d = 0; d < nd; ++d) pos[d] = s_dStart[d];
      for (int p = 0; p < n; ++p)
        if (s_pd[p] >= 0) s_dPairs[pos[s_pd[p]]++] = p;
      s_nD = nd;
    }
  }
  __syncthreads();
  const int nD = s_nD;

  // this CTA's down rows [h0, h1) of every distinct expert (device blocks by
  // bulk copy now; host blocks by plain loads after gate/up)
  const int hq = H / a.qd;
  const int h0 = static_cast<int>(static_cast<int64_t>(hq) * c / G) * a.qd;
  const int h1 = static_cast<int>(static_cast<int64_t>(hq) * (c + 1) / G) * a.qd;
  const int nr = h1 - h0;
  uint8_t* dsm = sm + a.sm_d;
  if (tid == 0 && nr > 0) {
    uint32_t bytes = 0;
    for (int d = 0; d < nD; ++d)
      if (!s_dHost[d]) bytes += static_cast<uint32_t>(nr) * (a.rowB + a.sbB);
    if (bytes > 0) {
      mbar_arrive_expect_tx(&bars[1], bytes);
      for (int d = 0; d < nD; ++d) {
        if (s_dHost[d]) continue;
        uint8_t* slab = dsm + static_cast<size_t>(d) * a.dslab;
        const uint8_t* blk = s_dBlk[d];
        bulk_g2s(slab, blk + a.off[2] + static_cast<uint64_t>(h0) * a.rowB, static_cast<uint32_t>(nr) * a.rowB, &bars[1]);
        bulk_g2s(slab + static_cast<size_t>(a.drows) * a.rowB, blk + a.off[5] + static_cast<uint64_t>(h0) * a.sbB,
                 static_cast<uint32_t>(nr) * a.sbB, &bars[1]);
      }
    }
    s_dbytes = bytes;
  }

  // ---- gate/up: units (distinct expert, qg rows) in [u0, u1); warp w takes
  // units u0 + w, u0 + w + 16, ... through its ring of slots
  const int upe = I / a.qg;
  const int64_t N = static_cast<int64_t>(nD) * upe;
  const int u0 = static_cast<int>(N * c / G), u1 = static_cast<int>(N * (c + 1) / G);
  const int nmine = (u1 - u0 > warp) ? (u1 - u0 - warp + kLWarps - 1) / kLWarps : 0;
  uint8_t* wslots = sm + a.sm_r + static_cast<size_t>(warp) * a.nslot * a.unit_bytes;
  uint64_t* wbars = &bars[2 + warp * a.nslot];
  const uint32_t cb = static_cast<uint32_t>(a.qg) * a.rowA, sbq = static_cast<uint32_t>(a.qg) * a.sbA;
  auto issue = [&](int j) {  // lane 0: bulk copies of the warp's j-th unit (device blocks only)
    const int u = u0 + warp + kLWarps * j;
    const int d = u / upe, r0 = (u % upe) * a.qg;
    if (s_dHost[d]) return;
    const int slot = j % a.nslot;
    uint8_t* dst = wslots + static_cast<size_t>(slot) * a.unit_bytes;
    const uint8_t* blk = s_dBlk[d];
    mbar_arrive_expect_tx(&wbars[slot], 2 * (cb + sbq));
    bulk_g2s(dst, blk + a.off[0] + static_cast<uint64_t>(r0) * a.rowA, cb, &wbars[slot]);
    bulk_g2s(dst + cb, blk + a.off[1] + static_cast<uint64_t>(r0) * a.rowA, cb, &wbars[slot]);
    bulk_g2s(dst + 2 * cb, blk + a.off[3] + static_cast<uint64_t>(r0) * a.sbA, sbq, &wbars[slot]);
    bulk_g2s(dst + 2 * cb + sbq, blk + a.off[4] + static_cast<uint64_t>(r0) * a.sbA, sbq, &wbars[slot]);
  };
  if (lane == 0)
    for (int j = 0; j < nmine && j < a.nslot; ++j) issue(j);
  __syncwarp();
  uint32_t phase = 0;  // per slot: parity of the next bulk-filled use
  bool timed_out = false;
  for (int j = 0; j < nmine; ++j) {
    const int u = u0 + warp + kLWarps * j;
    const int d = u / upe, r0 = (u % upe) * a.qg;
    const int slot = j % a.nslot;
    uint8_t* src = wslots + static_cast<size_t>(slot) * a.unit_bytes;
    if (s_dHost[d]) {
      const uint8_t* blk = s_dBlk[d];
      warp_copy(src, blk + a.off[0] + static_cast<uint64_t>(r0) * a.rowA, cb, lane);
      warp_copy(src + cb, blk + a.off[1] + static_cast<uint64_t>(r0) * a.rowA, cb, lane);
      warp_copy(src + 2 * cb, blk + a.off[3] + static_cast<uint64_t>(r0) * a.sbA, sbq, lane);
      warp_copy(src + 2 * cb + sbq, blk + a.off[4] + static_cast<uint64_t>(r0) * a.sbA, sbq, lane);
      __syncwarp();
    } else {
      if (!mbar_wait_lim(&wbars[slot], (phase >> slot) & 1u, a.dev_status, a.wait_ns)) {
        timed_out = true;
        break;
      }
      phase ^= 1u << slot;
    }
    float ts0 = 1.f, ts1 = 1.f;
    if constexpr (FMT == FT_NVFP4) {
      const int64_t fid = static_cast<int64_t>(a.layer) * E + s_dExpert[d];
      ts0 = __ldg(a.tscale + 3 * fid + 0);
      ts1 = __ldg(a.tscale + 3 * fid + 1);
    }
    for (int q = 0; q < a.qg; ++q) {
      const uint8_t* grow = src + static_cast<size_t>(q) * a.rowA;
      const uint8_t* urow = src + cb + static_cast<size_t>(q) * a.rowA;
      const uint8_t* gsr = src + 2 * cb + static_cast<size_t>(q) * a.sbA;
      const uint8_t* usr = src + 2 * cb + sbq + static_cast<size_t>(q) * a.sbA;
      for (int i = s_dStart[d]; i < s_dStart[d + 1]; ++i) {
        const int p = s_dPairs[i], t = p / k;
        float g = 0.f, uu = 0.f;
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
          g += chunk_dot<FMT>(wg, smem_scale<FMT>(gsr, ch, a.gshift), xa, asum);
          uu += chunk_dot<FMT>(wu, smem_scale<FMT>(usr, ch, a.gshift), xa, asum);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          g += __shfl_xor_sync(0xffffffffu, g, o);
          uu += __shfl_xor_sync(0xffffffffu, uu, o);
        }
        if (lane == 0) {
          const float gv = g * (ts0 * s_xinv[t]), uv = uu * (ts1 * s_xinv[t]);
          a.h[static_cast<size_t>(p) * I + r0 + q] = gv / (1.f + expf(-gv)) * uv;
        }
      }
    }
    __syncwarp();
    if (lane == 0 && j + a.nslot < nmine) issue(j + a.nslot);
    __syncwarp();
  }
  if (timed_out) {
    // wait (bounded) for this warp's copies still in flight, then leave the
    // barriers to time out in the other CTAs
    for (int s = 0; s < a.nslot; ++s) mbar_wait_lim(&wbars[s], (phase >> s) & 1u, nullptr, a.wait_ns);
  }

  // host blocks' down rows: plain loads into their slabs
  if (nr > 0)
    for (int d = warp; d < nD; d += kLWarps) {
      if (!s_dHost[d]) continue;
      uint8_t* slab = dsm + static_cast<size_t>(d) * a.dslab;
      warp_copy(slab, s_dBlk[d] + a.off[2] + static_cast<uint64_t>(h0) * a.rowB, static_cast<uint32_t>(nr) * a.rowB,
                lane);
      warp_copy(slab + static_cast<size_t>(a.drows) * a.rowB, s_dBlk[d] + a.off[5] + static_cast<uint64_t>(h0) * a.sbB,
                static_cast<uint32_t>(nr) * a.sbB, lane);
    }

  // ---- 5. h complete everywhere, then the down rows and the combine
  const bool bar_ok = grid_barrier(a, &s_ok);
  const bool down_ok = s_dbytes == 0 || mbar_wait_lim(&bars[1], 0, a.dev_status, a.wait_ns);
  if (!bar_ok || !down_ok) return;
  // h of every valid pair as f16 chunks with an exact power-of-two prescale
  // per pair (absorbed into its combine weight)
  uint8_t* hsm = sm + a.sm_h;
  float* hsum = reinterpret_cast<float*>(hsm + static_cast<size_t>(n) * IC * kChunkBytes);
  for (int p = warp; p < n; p += kLWarps) {
    if (s_pd[p] < 0) continue;
    const float* hp = a.h + static_cast<size_t>(p) * I;
    float m = 0.f;
    for (int ch = lane; ch < IC; ch += 32)
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 f = __ldcg(reinterpret_cast<const float4*>(hp + 32 * ch + 4 * q));
        m = fmaxf(m, fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w))));
      }
    const float mul = f16_prescale(warp_max(m));
    for (int ch = lane; ch < IC; ch += 32) {
      float v[32];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 f = __ldcg(reinterpret_cast<const float4*>(hp + 32 * ch + 4 * q));
        v[4 * q] = f.x;
        v[4 * q + 1] = f.y;
        v[4 * q + 2] = f.z;
        v[4 * q + 3] = f.w;
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
      float s = 0.f;
      for (int ch = sub; ch < IC; ch += LPR) {
        const uint8_t* hc = hsm + (static_cast<size_t>(p) * IC + ch) * kChunkBytes;
        uint32_t ha[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 v = *reinterpret_cast<const uint4*>(hc + 16 * q);
          ha[4 * q] = v.x;
          ha[4 * q + 1] = v.y;
          ha[4 * q + 2] = v.z;
          ha[4 * q + 3] = v.w;
        }
        const uint4 w = *reinterpret_cast<const uint4*>(crow + 16 * ch);
        s += chunk_dot<FMT>(w, smem_scale<FMT>(srow, ch, a.gshift), ha, hsum[static_cast<size_t>(p) * IC + ch]);
      }
      acc = fmaf(s_wq[p], s, acc);
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
// logits, then h.
constexpr size_t kLBarBytes = 256;
size_t layer_logits_bytes(int T, int E) {
  return (static_cast<size_t>(T) * E * sizeof(float) + 255) & ~static_cast<size_t>(255);
}

uint64_t g_wait_limit_ns = kWaitLimitNs;

}  // namespace
}  // namespace ft

extern "C" {

size_t ft_moe_decode_layer_workspace(int32_t T, int32_t k, int32_t H, int32_t I, int32_t E) {
  if (T <= 0 || k <= 0 || H <= 0 || I <= 0 || E <= 0) return 0;
  (void)H;
  const size_t hb = (static_cast<size_t>(T) * k * I * sizeof(float) + 255) & ~static_cast<size_t>(255);
  return ft::kLBarBytes + ft::layer_logits_bytes(T, E) + hb;
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
  a.ctr = reinterpret_cast<uint32_t*>(w8);
  a.gen = reinterpret_cast<uint32_t*>(w8 + 128);
  a.logits = reinterpret_cast<float*>(w8 + kLBarBytes);
  a.h = reinterpret_cast<float*>(w8 + kLBarBytes + layer_logits_bytes(T, E));
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
  const size_t xs = static_cast<size_t>(T) * (H / 32) * kXWordsL * 4;
  a.drows = (((H / a.qd) + G - 1) / G) * a.qd;
  a.dslab = static_cast<uint32_t>((static_cast<size_t>(a.drows) * (a.rowB + a.sbB) + 15) & ~static_cast<size_t>(15));
  const size_t ds = static_cast<size_t>(n) * a.dslab;
  const size_t hs = static_cast<size_t>(n) * (I / 32) * (kChunkBytes + 4);
  a.unit_bytes = 2 * (static_cast<uint32_t>(a.qg) * a.rowA + static_cast<uint32_t>(a.qg) * a.sbA);
  const int64_t units = static_cast<int64_t>(n) * (I / a.qg);
  const int per_warp = static_cast<int>(((units + G - 1) / G + kLWarps - 1) / kLWarps);
  // region R holds the router rows, then (leader) the resolve's arrays, then
  // the gate/up slots; the rest is fixed
  const size_t fixed = ((xs + 127) & ~static_cast<size_t>(127)) + ((ds + 127) & ~static_cast<size_t>(127)) +
                       ((hs + 127) & ~static_cast<size_t>(127)) + (2 + kLWarps * kLMaxSlots) * 8;
  const size_t router_bytes = static_cast<size_t>(kLMaxRouterRows) * H * 4;
  int nslot = per_warp < 1 ? 1 : (per_warp > kLMaxSlots ? kLMaxSlots : per_warp);
  while (nslot > 1 && fixed + static_cast<size_t>(kLWarps) * nslot * a.unit_bytes > cap) --nslot;
  size_t rsz = static_cast<size_t>(kLWarps) * nslot * a.unit_bytes;
  if (rsz < router_bytes) rsz = router_bytes;
  FT_REQUIRE(fixed + rsz <= cap, "decode layer: T=%d k=%d H=%d I=%d needs %zu bytes of shared memory (> %zu)", T, k,
             H, I, fixed + rsz, cap);
  a.nslot = nslot;
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
  off += (2 + kLWarps * a.nslot) * 8;
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
