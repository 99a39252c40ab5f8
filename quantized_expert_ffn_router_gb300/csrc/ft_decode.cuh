// ft_decode.cuh -- shared pieces of the decode expert kernels: arguments and
// the per-CTA grouping of (token, rank) pairs by distinct expert.
#pragma once

#include "ft_common.cuh"

namespace ft {

constexpr int kMaxPairs = 256;
constexpr int kMaxTok = 16;
constexpr int kV2MaxTok = 8;

struct DecArgs {
  const uint8_t* cache;
  uint64_t cstride;
  int64_t cblocks;
  const uint8_t* pool;  // may be null
  uint64_t pstride;
  int64_t pblocks;
  const float* tscale;  // [n_fids, 3] or null
  uint64_t off[6];
  int fmt, H, I, group, layer, E, T, k;
  const uint16_t* x;
  const int32_t* slot_ids;
  const int32_t* raw_ids;
  const float* topk_w;
  float* h;             // [T*k, I] fp32
  void* out;
  int out_bf16;
  int host_only;        // 1: only the pairs with slot -1, from the pool (FT_DECODE_HOST)
  int32_t* dev_status;
};

// The pair -> distinct-expert grouping, rebuilt by every CTA in shared memory.
// Distinct experts are numbered in ascending id order; dCached says whether
// the block is a cache slot (device memory) or a pool entry (read in place).
struct Groups {
  int nD;
  int nValid;
  int dStart[kMaxPairs + 1];
  int dExpert[kMaxPairs];
  int dCached[kMaxPairs];
  const uint8_t* dBlock[kMaxPairs];
  int sortedPair[kMaxPairs];  // valid pairs ordered by (distinct expert, pair)
  int sortedTok[kMaxPairs];   // their tokens
  int skip;                   // an earlier bounded wait of this stream gave up
  uintptr_t pairBlock[kMaxPairs];  // scratch: block of each pair, bit 0 = cached
};

// Ascending bitonic sort of 32*V keys held V per lane (element lane*V + v).
template <int V>
__device__ __forceinline__ void warp_bitonic_sort(uint32_t (&x)[V], int lane) {
#pragma unroll
  for (int k = 2; k <= 32 * V; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j < V) {
#pragma unroll
        for (int v = 0; v < V; ++v) {
          const int pv = v ^ j;
          if (pv > v) {
            const bool up = ((lane * V + v) & k) == 0;
            const uint32_t lo = min(x[v], x[pv]), hi = max(x[v], x[pv]);
            x[v] = up ? lo : hi;
            x[pv] = up ? hi : lo;
          }
        }
      } else {
        const int lj = j / V;
        const bool lower = (lane & lj) == 0;
#pragma unroll
        for (int v = 0; v < V; ++v) {
          const uint32_t o = __shfl_xor_sync(0xffffffffu, x[v], lj);
          const bool up = ((lane * V + v) & k) == 0;
          x[v] = (lower == up) ? min(x[v], o) : max(x[v], o);
        }
      }
    }
  }
}

// Warp 0 resolves every pair to its block, sorts the valid pairs by
// (expert id, pair index) and writes the grouping; the rest of the CTA waits
// at one block barrier.  Also reads the status word: returns true (for the
// whole CTA) when an earlier bounded wait of this stream already gave up.
template <int V>
__device__ __forceinline__ bool groups_sorted(const DecArgs& a, Groups& g) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int n = a.T * a.k;
    int32_t st = 0;
    if (lane == 0 && a.dev_status != nullptr) st = *reinterpret_cast<const volatile int32_t*>(a.dev_status);
    uint32_t key[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int p = v * 32 + lane;
      key[v] = 0xffffffffu;
      if (p < n) {
        int e = a.raw_ids[p];
        const int s = a.slot_ids[p];
        const uint8_t* blk = nullptr;
        int cached = 0;
        if (e < 0 || e >= a.E) {
          if (blockIdx.x == 0) record_status(a.dev_status, FT_ERR_BAD_ID);
        } else if (s >= 0) {
          if (a.host_only) {
            // a cache pair: computed by the FT_DECODE call on the cache
          } else if (s < a.cblocks) {
            blk = a.cache + static_cast<uint64_t>(s) * a.cstride;
            cached = 1;
          } else if (blockIdx.x == 0) {
            record_status(a.dev_status, FT_ERR_BAD_ID);
          }
        } else if (a.pool != nullptr) {
          const int64_t fid = static_cast<int64_t>(a.layer) * a.E + e;
          if (fid < a.pblocks)
            blk = a.pool + static_cast<uint64_t>(fid) * a.pstride;
          else if (blockIdx.x == 0)
            record_status(a.dev_status, FT_ERR_BAD_ID);
        }
        g.pairBlock[p] = reinterpret_cast<uintptr_t>(blk) | static_cast<uintptr_t>(cached);
        if (blk != nullptr) key[v] = (static_cast<uint32_t>(e) << 8) | static_cast<uint32_t>(p);
      }
    }
    warp_bitonic_sort<V>(key, lane);
    __syncwarp();
    // element i = lane*V + v; a start flag where the expert id changes
    const uint32_t prev_last = __shfl_up_sync(0xffffffffu, key[V - 1], 1);
    int flags = 0, valid = 0;
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const uint32_t prev = v > 0 ? key[v - 1] : (lane > 0 ? prev_last : 0xffffffffu);
      const bool ok = key[v] != 0xffffffffu;
      valid += ok;
      flags += (ok && (prev == 0xffffffffu || (prev >> 8) != (key[v] >> 8)));
    }
    int incl = flags;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int d = incl - flags - 1;
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const uint32_t kv = key[v];
      if (kv == 0xffffffffu) continue;
      const uint32_t prev = v > 0 ? key[v - 1] : (lane > 0 ? prev_last : 0xffffffffu);
      const int i = lane * V + v;
      const int p = static_cast<int>(kv & 0xffu);
      g.sortedPair[i] = p;
      g.sortedTok[i] = p / a.k;
      if (prev == 0xffffffffu || (prev >> 8) != (kv >> 8)) {
        ++d;
        g.dStart[d] = i;
        g.dExpert[d] = static_cast<int>(kv >> 8);
        g.dBlock[d] = reinterpret_cast<const uint8_t*>(g.pairBlock[p] & ~static_cast<uintptr_t>(1));
        g.dCached[d] = static_cast<int>(g.pairBlock[p] & 1u);
      }
    }
    int nv = valid;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) nv += __shfl_xor_sync(0xffffffffu, nv, o);
    const int nd = __shfl_sync(0xffffffffu, incl, 31);
    if (lane == 0) {
      g.nD = nd;
      g.nValid = nv;
      g.dStart[nd] = nv;
      g.skip = (st == FT_ERR_TIMEOUT);
    }
  }
  __syncthreads();
  return g.skip != 0;
}

// Grouping for any T*k <= kMaxPairs; every thread of the CTA must call it.
__device__ __forceinline__ bool build_groups(const DecArgs& a, Groups& g) {
  const int n = a.T * a.k;
  if (n <= 32) return groups_sorted<1>(a, g);
  if (n <= 64) return groups_sorted<2>(a, g);
  if (n <= 128) return groups_sorted<4>(a, g);
  return groups_sorted<8>(a, g);
}

// The streaming kernels (decode2.cu); FT_ERR_UNSUPPORTED if the shape does
// not fit them.
ft_status decode_streaming(const DecArgs& a, cudaStream_t s);


}  // namespace ft
