// decode.cu -- the experts entry point (ft_moe_experts_fwd) and its
// workspace size: host-side checks, then the decode kernels of decode2.cu or
// the prefill grouped GEMM of prefill.cu.
//
// Sources: "SSD 가중치층으로 35B MoE를 ..." (onedev.kr), "How it works"
// (down(silu(gate(x)) * up(x)) over int4, dedup of the routed experts);
// "NVMe에서 전문가(experts)를 ... 133GB MoE" (molayo1419.me), step 4 (the
// single-token NVFP4 SwiGLU expert kernel built on the hardware e2m1 -> f16x2
// convert); "FreeToken 딥다이브" (fiv.co.kr), design pattern 3 (pairs on the
// host path are masked, each pair computed once).
#include "ft_decode.cuh"

namespace ft {

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
  FT_REQUIRE(ws_bytes >= ft_moe_experts_workspace(FT_DECODE, T, k, cache->H, cache->I, E),
             "experts decode: workspace too small");
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
  // every shape these checks admit (H, I <= 4096 and multiples of 32, T <= 16,
  // T*k <= 256) fits the pair-major kernels
  return ft::decode_streaming(a, s);
}

}  // extern "C"
