// layer_buffer.cu -- the whole-layer buffer of prefill: a layer's expert
// blocks copied into a range of cache slots by the copy engine, and the slot
// cache's bookkeeping for it.
//
// Prefill runs every expert of a layer, so the layer's whole expert set is
// held on the GPU: layer l in slots (l%2)*E .., the next layer copied into
// the other half while this one computes, and the last two layers left in
// the cache to seed decode ("FreeToken 딥다이브" (fiv.co.kr), design pattern
// 1; "FreeToken: 让消费级电脑跑起 284B MoE" (fengjutian.github.io), sec. 5).
//
// The copy is one 2-D transfer (E rows of one block each, the banks' strides
// as pitches) on the caller's stream: a DMA engine moves the bytes while the
// SMs run the experts.
#include "ft_common.cuh"

namespace ft {
namespace {

constexpr int kInstallThreads = 1024;
constexpr int kInstallPer = 4;  // experts per thread: E <= 4096
constexpr int kInstallMaxE = kInstallThreads * kInstallPer;

// Install expert e of `layer` (flat id layer*E+e) in slot slot0+e for every e,
// with the end state of installing them one after the other: a copy of the
// flat id in a slot outside the range is dropped (owner -1, usage -1), the
// slot's previous owner is evicted (map -1), the slot takes the flat id with
// usage = the current step; recency and the step are left alone.  Three
// phases: read the old entries, evict, install.  Evictions touch distinct
// entries (a flat id owns at most one slot, a slot one flat id), and every
// map entry an eviction clears for a flat id of this layer is rewritten by
// the install phase.
__global__ void __launch_bounds__(kInstallThreads, 1) install_kernel(int32_t* __restrict__ owner,
                                                                     int32_t* __restrict__ map,
                                                                     int64_t* __restrict__ usage,
                                                                     const int64_t* __restrict__ step, int E,
                                                                     int layer, int slot0) {
  const int base = layer * E;
  int old[kInstallPer], was[kInstallPer];
#pragma unroll
  for (int i = 0; i < kInstallPer; ++i) {
    const int e = threadIdx.x + i * kInstallThreads;
    old[i] = was[i] = -1;
    if (e < E) {
      old[i] = owner[slot0 + e];
      was[i] = map[base + e];
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kInstallPer; ++i) {
    const int e = threadIdx.x + i * kInstallThreads;
    if (e >= E) continue;
    const int s = slot0 + e, fid = base + e;
    if (was[i] >= 0 && (was[i] < slot0 || was[i] >= slot0 + E)) {  // a copy outside the range
      owner[was[i]] = -1;
      usage[was[i]] = -1;
    }
    if (old[i] >= 0 && old[i] != fid) map[old[i]] = -1;
  }
  __syncthreads();
  const int64_t now = *step;
#pragma unroll
  for (int i = 0; i < kInstallPer; ++i) {
    const int e = threadIdx.x + i * kInstallThreads;
    if (e >= E) continue;
    owner[slot0 + e] = base + e;
    map[base + e] = slot0 + e;
    usage[slot0 + e] = now;
  }
}

}  // namespace
}  // namespace ft

extern "C" {

ft_status ft_moe_fetch_layer(const ft_bank* pool, const ft_bank* cache, int32_t layer, int32_t E, int32_t slot0,
                             void* stream) {
  ft::Layout Lp, Lc;
  ft_status s = ft::check_bank(pool, "fetch_layer pool", &Lp);
  if (s != FT_OK) return s;
  s = ft::check_bank(cache, "fetch_layer cache", &Lc);
  if (s != FT_OK) return s;
  FT_REQUIRE(pool->fmt == cache->fmt && pool->H == cache->H && pool->I == cache->I && pool->group == cache->group,
             "fetch_layer: pool and cache shapes differ");
  FT_REQUIRE(E >= 1 && layer >= 0 && slot0 >= 0, "fetch_layer: E=%d layer=%d slot0=%d", E, layer, slot0);
  FT_REQUIRE((static_cast<int64_t>(layer) + 1) * E <= pool->n_blocks,
             "fetch_layer: layer %d's flat ids pass the pool's %lld blocks", layer,
             static_cast<long long>(pool->n_blocks));
  FT_REQUIRE(static_cast<int64_t>(slot0) + E <= cache->n_blocks, "fetch_layer: slots %d..%d pass the cache's %lld",
             slot0, slot0 + E - 1, static_cast<long long>(cache->n_blocks));
  const uint8_t* src = static_cast<const uint8_t*>(pool->base) + static_cast<uint64_t>(layer) * E * pool->stride;
  uint8_t* dst = static_cast<uint8_t*>(const_cast<void*>(cache->base)) + static_cast<uint64_t>(slot0) * cache->stride;
  cudaError_t e = cudaMemcpy2DAsync(dst, cache->stride, src, pool->stride, Lp.total, E, cudaMemcpyDefault,
                                    ft::as_stream(stream));
  if (e != cudaSuccess) return ft::fail(FT_ERR_CUDA, "fetch_layer: %s", cudaGetErrorString(e));
  return FT_OK;
}

ft_status ft_moe_cache_install(const ft_cache_state* st, int32_t layer, int32_t slot0, void* stream) {
  FT_REQUIRE(st != nullptr, "cache_install: state is NULL");
  FT_REQUIRE(st->L > 0 && st->E > 0 && st->S >= 0, "cache_install: bad L/E/S %d/%d/%d", st->L, st->E, st->S);
  FT_REQUIRE(st->E <= ft::kInstallMaxE, "cache_install: E %d > %d", st->E, ft::kInstallMaxE);
  FT_REQUIRE(static_cast<int64_t>(st->L) * st->E < (1ll << 31), "cache_install: L*E overflows int32");
  FT_REQUIRE(layer >= 0 && layer < st->L, "cache_install: layer %d outside [0, %d)", layer, st->L);
  FT_REQUIRE(slot0 >= 0 && static_cast<int64_t>(slot0) + st->E <= st->S,
             "cache_install: slots %d..%d outside the %d slots", slot0, slot0 + st->E - 1, st->S);
  FT_REQUIRE(st->slot_owner && st->map && st->usage && st->step, "cache_install: NULL state array");
  ft::install_kernel<<<1, ft::kInstallThreads, 0, ft::as_stream(stream)>>>(st->slot_owner, st->map, st->usage,
                                                                            st->step, st->E, layer, slot0);
  return ft::launch_check("cache_install");
}

}  // extern "C"
