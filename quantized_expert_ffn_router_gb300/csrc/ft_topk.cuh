// ft_topk.cuh -- softmax and top-k of one token's router logits by one warp
// (larger logit first, ties to the lower expert id), shared by the router
// kernels and the fused decode layer.
//
// Source: "FreeToken: 让消费级电脑跑起 284B MoE" (fengjutian.github.io),
// sec. 2 (the router runs on the GPU and feeds the hit / miss split).
#pragma once

#include "ft_common.cuh"

namespace ft {
namespace {

// (a before b) in the routing order: larger logit first, ties to the lower id.
__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// One warp per token.  The token's E logits are read once into this warp's
// slice of shared memory (with the running max), then the softmax
// denominator.  Lane l owns the logits e = l (mod 32) and keeps the best of
// its untaken ones; each of the k rounds takes the warp's best (value
// descending, id ascending on ties) and only the winning lane marks it taken
// (a NaN in shared memory, which no comparison ranks first) and rescans its
// own logits for its next best.
__device__ __forceinline__ void lane_best(const float* ls, int E, int lane, float& bv, int& bi) {
  bv = -INFINITY;
  bi = 0x7fffffff;
  for (int e = lane; e < E; e += 32) {
    const float v = ls[e];
    if (ranks_before(v, e, bv, bi)) {
      bv = v;
      bi = e;
    }
  }
}

// Top-k of one token's E logits by one warp; ls is this warp's E floats of
// shared memory.
__device__ __forceinline__ void topk_warp(const float* __restrict__ l, float* ls, int E, int k, int renorm,
                                          int32_t* __restrict__ ids_t, float* __restrict__ wts_t,
                                          int stride = 1) {
  const int lane = threadIdx.x & 31;
  float mx = -INFINITY;
  for (int e = lane; e < E; e += 32) {
    const float v = __ldcg(l + static_cast<size_t>(e) * stride);
    ls[e] = v;
    mx = fmaxf(mx, v);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float z = 0.f;
  for (int e = lane; e < E; e += 32) z += expf(ls[e] - mx);
  z = warp_sum(z);
  float lv;
  int li;
  lane_best(ls, E, lane, lv, li);
  float sel_sum = 0.f;
  float my_w = 0.f;
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    float bv = lv;
    int bi = li;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ranks_before(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    const float p = expf(bv - mx) / z;
    sel_sum += p;
    if (lane == j) {
      my_w = p;
      my_id = bi;
    }
    if (bi == li && bi < E) {  // this lane's best was taken: find its next
      ls[bi] = __int_as_float(0x7fffffff);
      lane_best(ls, E, lane, lv, li);
    }
  }
  if (lane < k) {
    ids_t[lane] = my_id;
    wts_t[lane] = renorm ? my_w / sel_sum : my_w;
  }
}

// The same top-k for E <= 32 * VPL with the token's logits in registers
// (lane l holds e = l, l+32, ...): each round every lane offers its best
// untaken logit as an order-preserving 32-bit key, one redux.sync takes the
// warp's maximum key and a second the lowest expert id among the lanes
// holding it (ties to the lower id, as above).  The softmax denominator is
// summed in the same order as topk_warp, so ids and weights are the same.
// -0 ranks as +0; a NaN logit ranks below every number.
__device__ __forceinline__ uint32_t order_key(float v) {
  if (v != v) return 0u;  // NaN: lowest
  if (v == 0.f) v = 0.f;  // -0 -> +0
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <int VPL>
__device__ __forceinline__ void topk_warp_reg(const float* __restrict__ l, int E, int k, int renorm,
                                              int32_t* __restrict__ ids_t, float* __restrict__ wts_t,
                                              int stride = 1) {
  const int lane = threadIdx.x & 31;
  float v[VPL];
  uint32_t key[VPL];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? __ldcg(l + static_cast<size_t>(e) * stride) : -INFINITY;
    key[i] = e < E ? order_key(v[i]) : 0u;
    if (e < E) mx = fmaxf(mx, v[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float z = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i)
    if (lane + 32 * i < E) z += expf(v[i] - mx);
  z = warp_sum(z);
  uint32_t taken = 0u;
  float sel_sum = 0.f, my_w = 0.f;
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0u;
    int bi = -1;
    float bv = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (lane + 32 * i < E && !((taken >> i) & 1u) && (bi < 0 || key[i] > bk)) {
        bk = key[i];
        bi = i;
        bv = v[i];
      }
    const uint32_t m = __reduce_max_sync(0xffffffffu, bi >= 0 ? bk : 0u);
    const uint32_t cand = (bi >= 0 && bk == m) ? static_cast<uint32_t>(lane + 32 * bi) : 0xffffffffu;
    const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
    const float wv = __shfl_sync(0xffffffffu, bv, static_cast<int>(win & 31u));
    const float p = expf(wv - mx) / z;
    sel_sum += p;
    if (lane == j) {
      my_w = p;
      my_id = static_cast<int>(win);
    }
    if (static_cast<int>(win & 31u) == lane) taken |= 1u << (win >> 5);
  }
  if (lane < k) {
    ids_t[lane] = my_id;
    wts_t[lane] = renorm ? my_w / sel_sum : my_w;
  }
}

// Top-k of one token by one warp: the register form for E <= 512, else the
// shared-memory form (ls: this warp's E floats).  Logit e is l[e * stride].
__device__ __forceinline__ void topk_any(const float* __restrict__ l, float* ls, int E, int k, int renorm,
                                         int32_t* __restrict__ ids_t, float* __restrict__ wts_t, int stride = 1) {
  if (E <= 32) topk_warp_reg<1>(l, E, k, renorm, ids_t, wts_t, stride);
  else if (E <= 64) topk_warp_reg<2>(l, E, k, renorm, ids_t, wts_t, stride);
  else if (E <= 128) topk_warp_reg<4>(l, E, k, renorm, ids_t, wts_t, stride);
  else if (E <= 256) topk_warp_reg<8>(l, E, k, renorm, ids_t, wts_t, stride);
  else if (E <= 512) topk_warp_reg<16>(l, E, k, renorm, ids_t, wts_t, stride);
  else topk_warp(l, ls, E, k, renorm, ids_t, wts_t, stride);
}

}  // namespace
}  // namespace ft
