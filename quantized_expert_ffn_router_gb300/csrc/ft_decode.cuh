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
};

__device__ __forceinline__ void build_groups(const DecArgs& a, Groups& g) {
  __shared__ int s_e[kMaxPairs];
  __shared__ int s_first[kMaxPairs];
  __shared__ int s_d[kMaxPairs];
  __shared__ const uint8_t* s_blk[kMaxPairs];
  __shared__ int s_cached[kMaxPairs];
  const int n = a.T * a.k;
  for (int p = threadIdx.x; p < n; p += blockDim.x) {
    int e = a.raw_ids[p];
    const int s = a.slot_ids[p];
    const uint8_t* blk = nullptr;
    int cached = 0;
    if (e < 0 || e >= a.E) {
      if (blockIdx.x == 0) record_status(a.dev_status, FT_ERR_BAD_ID);
      e = -1;
    } else if (s >= 0) {
      if (s < a.cblocks) {
        blk = a.cache + static_cast<uint64_t>(s) * a.cstride;
        cached = 1;
      }
      else if (blockIdx.x == 0)
        record_status(a.dev_status, FT_ERR_BAD_ID);
    } else if (a.pool != nullptr) {
      const int64_t fid = static_cast<int64_t>(a.layer) * a.E + e;
      if (fid < a.pblocks)
        blk = a.pool + static_cast<uint64_t>(fid) * a.pstride;
      else if (blockIdx.x == 0)
        record_status(a.dev_status, FT_ERR_BAD_ID);
    }
    if (blk == nullptr) e = -1;  // skipped pair: masked or invalid
    s_e[p] = e;
    s_blk[p] = blk;
    s_cached[p] = cached;
  }
  __syncthreads();
  for (int p = threadIdx.x; p < n; p += blockDim.x) {
    const int e = s_e[p];
    int first = (e >= 0);
    for (int q = 0; q < p && first; ++q) first = (s_e[q] != e);
    s_first[p] = first;
  }
  __syncthreads();
  for (int p = threadIdx.x; p < n; p += blockDim.x) {
    const int e = s_e[p];
    int d = -1;
    if (e >= 0) {
      d = 0;
      for (int q = 0; q < n; ++q) d += (s_first[q] && s_e[q] < e);
    }
    s_d[p] = d;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int nD = 0, nV = 0;
    for (int p = 0; p < n; ++p) {
      nD += s_first[p];
      nV += (s_e[p] >= 0);
    }
    g.nD = nD;
    g.nValid = nV;
  }
  // per-distinct start offsets: count of valid pairs with a smaller d
  for (int p = threadIdx.x; p < n; p += blockDim.x) {
    if (!s_first[p]) continue;
    const int d = s_d[p];
    int start = 0;
    for (int q = 0; q < n; ++q) start += (s_d[q] >= 0 && s_d[q] < d);
    g.dStart[d] = start;
    g.dExpert[d] = s_e[p];
    g.dBlock[d] = s_blk[p];
    g.dCached[d] = s_cached[p];
  }
  __syncthreads();
  if (threadIdx.x == 0) g.dStart[g.nD] = g.nValid;
  for (int p = threadIdx.x; p < n; p += blockDim.x) {
    const int d = s_d[p];
    if (d < 0) continue;
    int r = 0;
    for (int q = 0; q < p; ++q) r += (s_d[q] == d);
    g.sortedPair[g.dStart[d] + r] = p;
  }
  __syncthreads();
}


// The streaming kernels (decode2.cu); FT_ERR_UNSUPPORTED if the shape does
// not fit them.
ft_status decode_streaming(const DecArgs& a, cudaStream_t s);

}  // namespace ft
