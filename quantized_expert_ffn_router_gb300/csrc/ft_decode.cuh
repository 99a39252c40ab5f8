// ft_decode.cuh -- shared pieces of the decode expert kernels: limits and
// arguments.
#pragma once

#include "ft_common.cuh"

namespace ft {

constexpr int kMaxPairs = 256;
constexpr int kMaxTok = 16;

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

// The pair-major decode kernels (decode2.cu).
ft_status decode_streaming(const DecArgs& a, cudaStream_t s);


}  // namespace ft
