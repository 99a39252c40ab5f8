// rebuild.cu -- runtime rebuild of the global slot cache at a new size.
//
// Sources: "FreeToken: 让消费级电脑跑起 284B MoE" (fengjutian.github.io), sec. 7
// item 1 (the GPU expert cache is rebuilt for a new memory budget at a safe
// point; the host pool is the source of truth, so correctness never depends
// on the cache); "FreeToken 딥다이브" (fiv.co.kr), design pattern 7 (validate
// the new geometry and the budget before destroying anything, refuse a
// rebuild that does not fit).
//
// The old state is only read.  Two kernels on the caller's stream: the first
// empties the new state and copies recency and the step; the second, one CTA
// per old slot, ranks its resident expert among all residents (usage desc,
// slot asc: the order the cache evicts in, reversed) and, if the rank falls
// below the new size, moves the expert's block and state to the slot of that
// rank.
#include "ft_common.cuh"

namespace ft {
namespace {

constexpr int kRbThreads = 256;

__global__ void rebuild_init_kernel(int64_t n_fid, int32_t S_new, int32_t* __restrict__ map_new,
                                    int64_t* __restrict__ recency_new, const int64_t* __restrict__ recency_old,
                                    int32_t* __restrict__ owner_new, int64_t* __restrict__ usage_new,
                                    int64_t* __restrict__ step_new, const int64_t* __restrict__ step_old) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_fid; i += stride) {
    map_new[i] = -1;
    recency_new[i] = recency_old[i];
  }
  for (int64_t d = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; d < S_new; d += stride) {
    owner_new[d] = -1;
    usage_new[d] = -1;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) step_new[0] = step_old[0];
}

__global__ void __launch_bounds__(kRbThreads) rebuild_move_kernel(
    int64_t n_fid, int32_t S_old, const int32_t* __restrict__ owner_old, const int64_t* __restrict__ usage_old,
    int32_t S_new, int32_t* __restrict__ owner_new, int32_t* __restrict__ map_new,
    int64_t* __restrict__ usage_new, const uint8_t* __restrict__ bank_old, uint64_t stride_old,
    uint8_t* __restrict__ bank_new, uint64_t stride_new, uint64_t block_bytes, int32_t* dev_status) {
  __shared__ int s_cnt[kRbThreads / 32];
  const int s = blockIdx.x;
  const int32_t fid = owner_old[s];
  if (fid < 0) return;
  if (fid >= n_fid) {
    if (threadIdx.x == 0) record_status(dev_status, FT_ERR_BAD_ID);
    return;
  }
  const int64_t u = usage_old[s];
  // rank = residents ahead of this one: larger usage, or equal usage and a lower slot
  int cnt = 0;
  for (int j = threadIdx.x; j < S_old; j += kRbThreads) {
    const int32_t o = owner_old[j];
    if (o < 0 || o >= n_fid) continue;
    const int64_t uj = usage_old[j];
    cnt += (uj > u || (uj == u && j < s)) ? 1 : 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if ((threadIdx.x & 31) == 0) s_cnt[threadIdx.x >> 5] = cnt;
  __syncthreads();
  int rank = 0;
#pragma unroll
  for (int w = 0; w < kRbThreads / 32; ++w) rank += s_cnt[w];
  if (rank >= S_new) return;
  if (threadIdx.x == 0) {
    owner_new[rank] = fid;
    usage_new[rank] = u;
    map_new[fid] = rank;
  }
  const uint4* src = reinterpret_cast<const uint4*>(bank_old + static_cast<uint64_t>(s) * stride_old);
  uint4* dst = reinterpret_cast<uint4*>(bank_new + static_cast<uint64_t>(rank) * stride_new);
  const uint64_t n16 = block_bytes / 16;
  for (uint64_t i = threadIdx.x; i < n16; i += kRbThreads) dst[i] = src[i];
}

bool overlaps(const void* a, uint64_t na, const void* b, uint64_t nb) {
  const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
  return na > 0 && nb > 0 && pa < pb + nb && pb < pa + na;
}

}  // namespace
}  // namespace ft

extern "C" {

ft_status ft_moe_cache_rebuild(const ft_cache_state* old_st, const ft_bank* old_cache,
                               const ft_cache_state* new_st, const ft_bank* new_cache, uint64_t budget_bytes,
                               int32_t* dev_status, void* stream) {
  FT_REQUIRE(old_st != nullptr && new_st != nullptr, "cache rebuild: state is NULL");
  ft::Layout Lo, Ln;
  ft_status st = ft::check_bank(old_cache, "cache rebuild old cache", &Lo);
  if (st != FT_OK) return st;
  st = ft::check_bank(new_cache, "cache rebuild new cache", &Ln);
  if (st != FT_OK) return st;
  FT_REQUIRE(old_st->L > 0 && old_st->E > 0 && old_st->S >= 0 && new_st->L > 0 && new_st->E > 0 && new_st->S >= 0,
             "cache rebuild: bad L/E/S");
  FT_REQUIRE(old_st->map && old_st->recency && old_st->step && new_st->map && new_st->recency && new_st->step,
             "cache rebuild: NULL state array");
  FT_REQUIRE(old_st->S == 0 || (old_st->slot_owner && old_st->usage), "cache rebuild: NULL old slot arrays");
  FT_REQUIRE(new_st->S == 0 || (new_st->slot_owner && new_st->usage), "cache rebuild: NULL new slot arrays");
  // the checks a well-formed rebuild can fail: refused, nothing changed
  if (new_st->L != old_st->L || new_st->E != old_st->E)
    return ft::fail(FT_ERR_REJECTED, "cache rebuild: the new state serves L=%d E=%d, the old L=%d E=%d", new_st->L,
                    new_st->E, old_st->L, old_st->E);
  if (new_cache->fmt != old_cache->fmt || new_cache->H != old_cache->H || new_cache->I != old_cache->I ||
      new_cache->group != old_cache->group)
    return ft::fail(FT_ERR_REJECTED, "cache rebuild: the new cache's expert format or shape differs");
  if (new_st->S > new_cache->n_blocks)
    return ft::fail(FT_ERR_REJECTED, "cache rebuild: %d slots but the new bank holds %lld blocks", new_st->S,
                    static_cast<long long>(new_cache->n_blocks));
  const uint64_t S_new = static_cast<uint64_t>(new_st->S);
  const uint64_t need = S_new * new_cache->stride + S_new * (sizeof(int32_t) + sizeof(int64_t));
  if (need > budget_bytes)
    return ft::fail(FT_ERR_REJECTED, "cache rebuild: %llu bytes needed, budget %llu",
                    static_cast<unsigned long long>(need), static_cast<unsigned long long>(budget_bytes));
  const int64_t n_fid = static_cast<int64_t>(old_st->L) * old_st->E;
  const uint64_t S_old = static_cast<uint64_t>(old_st->S);
  const uint64_t bo = static_cast<uint64_t>(old_cache->n_blocks) * old_cache->stride;
  const uint64_t bn = S_new * new_cache->stride;
  // every new range against every old range: the old cache stays intact
  const void* op[6] = {old_cache->base, old_st->map, old_st->recency, old_st->step, old_st->slot_owner, old_st->usage};
  const uint64_t on[6] = {bo, n_fid * 4ull, n_fid * 8ull, 8ull, S_old * 4, S_old * 8};
  const void* np[6] = {new_cache->base, new_st->map, new_st->recency, new_st->step, new_st->slot_owner, new_st->usage};
  const uint64_t nn[6] = {bn, n_fid * 4ull, n_fid * 8ull, 8ull, S_new * 4, S_new * 8};
  for (int i = 0; i < 6; ++i)
    for (int j = 0; j < 6; ++j)
      if (ft::overlaps(np[i], nn[i], op[j], on[j]))
        return ft::fail(FT_ERR_REJECTED, "cache rebuild: the new bank or state overlaps the old");
  cudaStream_t s = ft::as_stream(stream);
  const int64_t span = std::max<int64_t>(n_fid, static_cast<int64_t>(S_new));
  const int init_grid = static_cast<int>(std::min<int64_t>((span + ft::kRbThreads - 1) / ft::kRbThreads, 4096));
  ft::rebuild_init_kernel<<<std::max(init_grid, 1), ft::kRbThreads, 0, s>>>(
      n_fid, new_st->S, new_st->map, new_st->recency, old_st->recency, new_st->slot_owner, new_st->usage,
      new_st->step, old_st->step);
  st = ft::launch_check("cache rebuild init");
  if (st != FT_OK || old_st->S == 0 || new_st->S == 0) return st;
  ft::rebuild_move_kernel<<<old_st->S, ft::kRbThreads, 0, s>>>(
      n_fid, old_st->S, old_st->slot_owner, old_st->usage, new_st->S, new_st->slot_owner, new_st->map,
      new_st->usage, static_cast<const uint8_t*>(old_cache->base), old_cache->stride,
      static_cast<uint8_t*>(const_cast<void*>(new_cache->base)), new_cache->stride, Lo.total, dev_status);
  return ft::launch_check("cache rebuild move");
}

}  // extern "C"
