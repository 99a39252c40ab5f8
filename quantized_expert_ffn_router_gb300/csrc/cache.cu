// cache.cu -- the global slot cache on the device: the Q16 q* split, the
// one-kernel resolve (dedup, residency, q*, recency-ranked fetch choice,
// single-scan K-victim selection, id rewrite) and the fetch copy.
//
// Sources: "FreeToken 딥다이브" (fiv.co.kr), design patterns 2, 3, 5;
// "FreeToken: 让消费级电脑跑起 284B MoE" (fengjutian.github.io), secs. 4, 6.
#include "ft_async.cuh"
#include "ft_common.cuh"
#include "ft_resolve.cuh"
#include "ft_topk.cuh"

namespace ft {
namespace {

constexpr int kResThreads = 1024;

__global__ void split_q16_kernel(const int32_t* __restrict__ m, int32_t n, int32_t phi,
                                 int32_t* __restrict__ out) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    out[i] = split_q16_dev(m[i], phi);
}
// The combined route + resolve call: the router grid leaves each token's
// logits ([E][stride] floats) and this kernel takes their top-k first, one
// warp per token, into ids / wts and a shared-memory copy the resolve reads.
constexpr int kResTopkMax = 16 * 32;  // T * k of the combined call
struct RouteTopk {
  const float* logits;
  int T, E, k, renorm, stride;
  int32_t* ids;
  float* wts;
};

// The arguments stay in the parameter space (__grid_constant__, no local
// copy): the small path, inlined here, reads them as parameter loads, and the
// block-wide body (not inlined, arguments by reference) gets a shared-memory
// copy.
template <bool TOPK>
__global__ void __launch_bounds__(kResThreads, 1) resolve_kernel(const __grid_constant__ ResolveArgs a,
                                                                 const __grid_constant__ RouteTopk r) {
  extern __shared__ __align__(16) unsigned char smem[];
  if (TOPK && threadIdx.x == 0) {
    // the step counter is not the router's output: its last writer finished
    // before the router grid let this kernel start, so it may be fetched now
    asm volatile("prefetch.global.L1 [%0];" ::"l"(a.step));
  }
  pdl_wait();               // ids (or the router logits) come from the previous kernel
  pdl_launch_dependents();  // the next call (fetch) may start its launch now
  __shared__ int32_t s_ids[kResTopkMax];
  const int32_t* ids_sm = nullptr;
  if (TOPK) {
    const int warp = threadIdx.x >> 5;
    if (warp < r.T)  // E <= 512: the register top-k (no shared scratch)
      topk_any(r.logits + warp, nullptr, r.E, r.k, r.renorm, s_ids + warp * r.k, r.wts + warp * r.k, r.stride);
    __syncthreads();
    for (int i = threadIdx.x; i < r.T * r.k; i += blockDim.x) r.ids[i] = s_ids[i];
    ids_sm = s_ids;
  }
  // the small calls inline (the arguments read from the parameter space),
  // the rest in resolve_block, which reads its arguments through a reference:
  // give it a shared-memory copy (one word per thread), not the parameters
  if (a.n <= 32 && !a.prefetch && resolve_small_path(a, ids_sm)) return;
  __shared__ __align__(16) ResolveArgs s_args;
  static_assert(sizeof(ResolveArgs) % 4 == 0, "copied a word at a time");
  if (threadIdx.x < sizeof(ResolveArgs) / 4)
    reinterpret_cast<uint32_t*>(&s_args)[threadIdx.x] = reinterpret_cast<const uint32_t*>(&a)[threadIdx.x];
  __syncthreads();
  resolve_block(s_args, smem, ids_sm, false);
}

// Copy fetched expert blocks pool[fid] -> cache[slot] for i < *num_fetch.
// A grid-stride loop over (fetch index, 32 KiB chunk) items; each thread moves
// eight 16-byte vectors with all loads issued before the stores.
constexpr int kFetchThreads = 256;
constexpr int kFetchVec = 8;

__global__ void __launch_bounds__(kFetchThreads) fetch_kernel(
    const uint8_t* __restrict__ pool, uint64_t pstride, uint8_t* __restrict__ cache,
    uint64_t cstride, uint64_t n16, const int32_t* __restrict__ num_fetch,
    const int32_t* __restrict__ ffid, const int32_t* __restrict__ fslot, int32_t max_list,
    int64_t n_pool, int64_t n_cache, int32_t* dev_status) {
  pdl_wait();               // the fetch list comes from the previous kernel (resolve)
  pdl_launch_dependents();  // the experts call may start its launch now
  const int nf = min(*num_fetch, max_list);
  const uint64_t per = static_cast<uint64_t>(kFetchThreads) * kFetchVec;
  const uint64_t nchunks = (n16 + per - 1) / per;
  const uint64_t items = static_cast<uint64_t>(nf > 0 ? nf : 0) * nchunks;
  for (uint64_t item = blockIdx.x; item < items; item += gridDim.x) {
    const int i = static_cast<int>(item / nchunks);
    const uint64_t c = item % nchunks;
    const int fid = ffid[i], slot = fslot[i];
    if (fid < 0 || fid >= n_pool || slot < 0 || slot >= n_cache) {
      if (c == 0 && threadIdx.x == 0) record_status(dev_status, FT_ERR_BAD_ID);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(pool + static_cast<uint64_t>(fid) * pstride);
    uint4* dst = reinterpret_cast<uint4*>(cache + static_cast<uint64_t>(slot) * cstride);
    uint4 r[kFetchVec];
#pragma unroll
    for (int u = 0; u < kFetchVec; ++u) {
      const uint64_t idx = c * per + static_cast<uint64_t>(u) * kFetchThreads + threadIdx.x;
      if (idx < n16) r[u] = src[idx];
    }
#pragma unroll
    for (int u = 0; u < kFetchVec; ++u) {
      const uint64_t idx = c * per + static_cast<uint64_t>(u) * kFetchThreads + threadIdx.x;
      if (idx < n16) dst[idx] = r[u];
    }
  }
}

}  // namespace

ft_status resolve_prepare(const ft_cache_state* st, int32_t layer, const int32_t* topk_ids, int32_t T,
                          int32_t k, int32_t frac_q16, int32_t* slot_ids, int32_t* num_fetch,
                          int32_t* fetch_fid, int32_t* fetch_slot, int32_t max_list, int32_t* dev_status,
                          const char* what, size_t stage_cap, ResolveArgs* out, size_t* smem_out) {
  FT_REQUIRE(st != nullptr, "%s: state is NULL", what);
  FT_REQUIRE(st->L > 0 && st->E > 0 && st->S >= 0, "%s: bad L/E/S %d/%d/%d", what, st->L, st->E, st->S);
  FT_REQUIRE(st->E <= kResMaxE, "%s: E %d > %d", what, st->E, kResMaxE);
  FT_REQUIRE(static_cast<int64_t>(st->L) * st->E < (1ll << 31), "%s: L*E overflows int32", what);
  FT_REQUIRE(layer >= 0 && layer < st->L, "%s: layer %d outside [0, %d)", what, layer, st->L);
  FT_REQUIRE(T >= 0 && k >= 1, "%s: T=%d k=%d", what, T, k);
  const int64_t n64 = static_cast<int64_t>(T) * k;
  FT_REQUIRE(n64 <= kResMaxN, "%s: T*k = %lld > %d", what, static_cast<long long>(n64), kResMaxN);
  FT_REQUIRE(frac_q16 >= 0 && frac_q16 <= 65536, "%s: frac_q16 %d outside [0, 65536]", what, frac_q16);
  const int n = static_cast<int>(n64);
  const int need = n < st->S ? n : st->S;
  FT_REQUIRE(max_list >= need, "%s: max_list %d < min(T*k, S) = %d", what, max_list, need);
  FT_REQUIRE(st->map && st->recency && st->step && num_fetch && fetch_fid && fetch_slot, "%s: NULL pointer", what);
  FT_REQUIRE(st->S == 0 || (st->slot_owner && st->usage), "%s: NULL slot arrays", what);
  FT_REQUIRE(n == 0 || (topk_ids && slot_ids), "%s: NULL ids", what);
  ResolveArgs& a = *out;
  a.E = st->E;
  a.S = st->S;
  a.layer = layer;
  a.n = n;
  a.phi = frac_q16;
  a.max_list = max_list;
  a.slot_owner = st->slot_owner;
  a.map = st->map;
  a.usage = st->usage;
  a.recency = st->recency;
  a.step = st->step;
  a.ids = topk_ids;
  a.slot_ids = slot_ids;
  a.num_fetch = num_fetch;
  a.fetch_fid = fetch_fid;
  a.fetch_slot = fetch_slot;
  a.dev_status = dev_status;
  a.prefetch = 0;
  a.max_prefetch = 0;
  a.slot_ids_sm = nullptr;
  a.num_fetch_sm = nullptr;
  a.ids_sm = nullptr;
  // the slot state is staged in shared memory when it fits beside the
  // resolve's own arrays (every cache up to ~24k slots at E <= 256)
  const size_t base = resolve_smem_bytes(st->E, n);
  const size_t staged = base + resolve_stage_bytes(st->S);
  a.staged = (st->S > 0 && staged <= stage_cap) ? 1 : 0;
  *smem_out = a.staged ? staged : base;
  return FT_OK;
}

ft_status prefetch_prepare(const ft_cache_state* st, int32_t layer, const int32_t* pred_ids, int32_t T,
                           int32_t k, int32_t max_prefetch, int32_t* num_fetch, int32_t* fetch_fid,
                           int32_t* fetch_slot, int32_t max_list, int32_t* dev_status, size_t stage_cap,
                           ResolveArgs* out, size_t* smem_out) {
  FT_REQUIRE(max_prefetch >= 0, "prefetch: max_prefetch %d < 0", max_prefetch);
  // the resolve's checks, with pred_ids standing in for the (unwritten) slot_ids
  ft_status s = resolve_prepare(st, layer, pred_ids, T, k, 0, const_cast<int32_t*>(pred_ids), num_fetch,
                                fetch_fid, fetch_slot, max_list, dev_status, "prefetch", stage_cap, out,
                                smem_out);
  if (s != FT_OK) return s;
  out->slot_ids = nullptr;
  out->prefetch = 1;
  out->max_prefetch = max_prefetch;
  return FT_OK;
}

}  // namespace ft

namespace {

// One CTA runs a resolve or a prefetch (both set up by *_prepare), chained to
// the previous kernel on the stream by programmatic launch.
ft_status launch_resolve(const ft::ResolveArgs& a, size_t smem, void* stream, const char* what,
                         const ft::RouteTopk* topk = nullptr) {
  if (smem > 48 * 1024) {
    ft_status st = ft::ensure_dyn_smem(reinterpret_cast<const void*>(ft::resolve_kernel<false>),
                                       static_cast<int>(ft::kResSmemCap), what);
    if (st == FT_OK)
      st = ft::ensure_dyn_smem(reinterpret_cast<const void*>(ft::resolve_kernel<true>),
                               static_cast<int>(ft::kResSmemCap), what);
    if (st != FT_OK) return st;
  }
  // every call gets the whole block: the one-warp path of small calls that
  // fetch nothing leaves the rest idle at one barrier, and a call that does
  // fetch scans its slots (staging, minimum, radix select, ordered scan)
  // four times faster than with 256 threads
  const int threads = ft::kResThreads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = ft::as_stream(stream);
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = topk ? cudaLaunchKernelEx(&cfg, ft::resolve_kernel<true>, a, *topk)
                       : cudaLaunchKernelEx(&cfg, ft::resolve_kernel<false>, a, ft::RouteTopk{});
  if (e != cudaSuccess) return ft::fail(FT_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return ft::launch_check(what);
}

}  // namespace

extern "C" {

ft_status ft_moe_split_q16(const int32_t* num_missing, int32_t n, int32_t frac_q16,
                           int32_t* num_fetch, void* stream) {
  FT_REQUIRE(n >= 0, "split_q16: n < 0");
  FT_REQUIRE(frac_q16 >= 0 && frac_q16 <= 65536, "split_q16: frac_q16 %d outside [0, 65536]",
             frac_q16);
  if (n == 0) return FT_OK;
  FT_REQUIRE(num_missing != nullptr && num_fetch != nullptr, "split_q16: NULL pointer");
  const int threads = 256;
  const int blocks = min((n + threads - 1) / threads, 4096);
  ft::split_q16_kernel<<<blocks, threads, 0, ft::as_stream(stream)>>>(num_missing, n, frac_q16,
                                                                     num_fetch);
  return ft::launch_check("split_q16");
}

ft_status ft_moe_resolve_slots(const ft_cache_state* st, int32_t layer, const int32_t* topk_ids,
                               int32_t T, int32_t k, int32_t frac_q16, int32_t* slot_ids,
                               int32_t* num_fetch, int32_t* fetch_fid, int32_t* fetch_slot,
                               int32_t max_list, int32_t* dev_status, void* stream) {
  ft::ResolveArgs a;
  size_t smem = 0;
  ft_status ps = ft::resolve_prepare(st, layer, topk_ids, T, k, frac_q16, slot_ids, num_fetch, fetch_fid,
                                     fetch_slot, max_list, dev_status, "resolve", ft::kResSmemCap, &a, &smem);
  if (ps != FT_OK) return ps;
  return launch_resolve(a, smem, stream, "resolve_slots");
}

ft_status ft_moe_route_resolve(const uint16_t* x, int32_t T, int32_t H, const float* w_router, int32_t E,
                               int32_t k, int32_t renorm, int32_t* topk_ids, float* topk_w, void* route_ws,
                               size_t route_ws_bytes, const ft_cache_state* st, int32_t layer, int32_t frac_q16,
                               int32_t* slot_ids, int32_t* num_fetch, int32_t* fetch_fid, int32_t* fetch_slot,
                               int32_t max_list, int32_t* dev_status, void* stream) {
  // the one-kernel top-k takes T * k <= 32 (the resolve's one-warp shape:
  // at T = 8, k = 8 the resolve runs its block-wide path and the top-k in
  // front of it measured 1.3% slower per decode step than the router's last
  // CTA, against 3.5% faster at T = 1), E <= 512 experts (register top-k)
  // and the state's own E; anything else is the two calls in order
  if (T < 1 || T > 16 || T * k > 32 || E < 1 || E > 512 || k < 1 || k > 32 || k > E || st == nullptr ||
      st->E != E) {
    ft_status s = ft_moe_route(x, T, H, w_router, E, k, renorm, topk_ids, topk_w, route_ws, route_ws_bytes, stream);
    if (s != FT_OK) return s;
    return ft_moe_resolve_slots(st, layer, topk_ids, T, k, frac_q16, slot_ids, num_fetch, fetch_fid, fetch_slot,
                                max_list, dev_status, stream);
  }
  // every check of both calls before anything is launched
  FT_REQUIRE(H >= 8 && H % 8 == 0, "route_resolve: H %d must be a positive multiple of 8", H);
  FT_REQUIRE(x && w_router && topk_ids && topk_w && route_ws, "route_resolve: NULL pointer");
  FT_REQUIRE(route_ws_bytes >= ft_moe_route_workspace(T, E, H), "route_resolve: workspace %zu < %zu",
             route_ws_bytes, ft_moe_route_workspace(T, E, H));
  FT_REQUIRE(reinterpret_cast<uintptr_t>(x) % 16 == 0 && reinterpret_cast<uintptr_t>(w_router) % 16 == 0,
             "route_resolve: x and w_router must be 16-byte aligned");
  ft::ResolveArgs a;
  size_t smem = 0;
  ft_status ps = ft::resolve_prepare(st, layer, topk_ids, T, k, frac_q16, slot_ids, num_fetch, fetch_fid,
                                     fetch_slot, max_list, dev_status, "route_resolve", ft::kResSmemCap, &a, &smem);
  if (ps != FT_OK) return ps;
  const float* logits = nullptr;
  int stride = 0;
  ps = ft::route_rows_logits(x, T, H, w_router, E, route_ws, ft::as_stream(stream), &logits, &stride);
  if (ps != FT_OK) return ps;
  const ft::RouteTopk r{logits, T, E, k, renorm, stride, topk_ids, topk_w};
  return launch_resolve(a, smem, stream, "route_resolve", &r);
}

ft_status ft_moe_prefetch(const ft_cache_state* st, int32_t layer, const int32_t* pred_ids, int32_t T,
                          int32_t k, int32_t max_prefetch, int32_t* num_fetch, int32_t* fetch_fid,
                          int32_t* fetch_slot, int32_t max_list, int32_t* dev_status, void* stream) {
  ft::ResolveArgs a;
  size_t smem = 0;
  ft_status ps = ft::prefetch_prepare(st, layer, pred_ids, T, k, max_prefetch, num_fetch, fetch_fid,
                                      fetch_slot, max_list, dev_status, ft::kResSmemCap, &a, &smem);
  if (ps != FT_OK) return ps;
  return launch_resolve(a, smem, stream, "prefetch");
}

ft_status ft_moe_fetch(const ft_bank* pool, const ft_bank* cache, const int32_t* num_fetch,
                       const int32_t* fetch_fid, const int32_t* fetch_slot, int32_t max_list,
                       int32_t* dev_status, void* stream) {
  ft::Layout Lp, Lc;
  ft_status s = ft::check_bank(pool, "fetch pool", &Lp);
  if (s != FT_OK) return s;
  s = ft::check_bank(cache, "fetch cache", &Lc);
  if (s != FT_OK) return s;
  FT_REQUIRE(pool->fmt == cache->fmt && pool->H == cache->H && pool->I == cache->I &&
                 pool->group == cache->group,
             "fetch: pool and cache shapes differ");
  FT_REQUIRE(max_list >= 0, "fetch: max_list < 0");
  if (max_list == 0) return FT_OK;
  FT_REQUIRE(num_fetch && fetch_fid && fetch_slot, "fetch: NULL pointer");
  const uint64_t n16 = Lp.total / 16;
  const uint64_t per = static_cast<uint64_t>(ft::kFetchThreads) * ft::kFetchVec;
  const uint64_t nchunks = (n16 + per - 1) / per;
  const uint64_t items = nchunks * static_cast<uint64_t>(max_list);
  const int grid = static_cast<int>(std::min<uint64_t>(items, static_cast<uint64_t>(ft::device_sm_count())));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(ft::kFetchThreads);
  cfg.stream = ft::as_stream(stream);
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const uint8_t* src = static_cast<const uint8_t*>(pool->base);
  uint8_t* dst = static_cast<uint8_t*>(const_cast<void*>(cache->base));
  const int64_t npool = pool->n_blocks, ncache = cache->n_blocks;
  cudaError_t e = cudaLaunchKernelEx(&cfg, ft::fetch_kernel, src, pool->stride, dst, cache->stride, n16, num_fetch,
                                     fetch_fid, fetch_slot, max_list, npool, ncache, dev_status);
  if (e != cudaSuccess) return ft::fail(FT_ERR_CUDA, "fetch: %s", cudaGetErrorString(e));
  return ft::launch_check("fetch");
}

}  // extern "C"
