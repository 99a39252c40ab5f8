// ft_resolve.cuh -- the resolve of a layer's top-k ids against the global
// slot cache, as a device function that one CTA runs (the resolve kernel in
// cache.cu), with its host-side argument checks.
//
// Sources: "FreeToken 딥다이브" (fiv.co.kr), design patterns 2, 3, 5;
// "FreeToken: 让消费级电脑跑起 284B MoE" (fengjutian.github.io), sec. 6 (one
// kernel does dedup, residency, q, victims and the id rewrite).
#pragma once

#include <climits>

#include "ft_common.cuh"

namespace ft {

constexpr int kResMaxE = 4096;
constexpr int kResMaxN = 4096;
constexpr int kResFastVictims = 16;  // up to this many victims: iterated block argmin
constexpr size_t kResSmemCap = 220 * 1024;  // dynamic shared memory the resolve kernel may use

struct ResolveArgs {
  int32_t E, S, layer, n, phi, max_list;
  int32_t staged;  // 1: the victim search reads the slots' usage and hit flags from shared memory
  // 1: a speculative prefetch of predicted ids (no split, cap = max_prefetch,
  // held slots with usage >= step-1 are not victims, no routing bookkeeping,
  // no slot_ids); 0: a resolve
  int32_t prefetch, max_prefetch;
  int32_t* slot_owner;
  int32_t* map;
  int64_t* usage;
  int64_t* recency;
  int64_t* step;
  const int32_t* ids;
  int32_t* slot_ids;
  int32_t* num_fetch;
  int32_t* fetch_fid;
  int32_t* fetch_slot;
  int32_t* dev_status;
  // optional shared-memory copies of slot_ids [n] and num_fetch, for a caller
  // that runs the resolve inside a larger kernel (null: global outputs only)
  int32_t* slot_ids_sm;
  int32_t* num_fetch_sm;
  const int32_t* ids_sm;  // optional shared-memory copy of ids [n], read instead of ids
};

__device__ __forceinline__ int resolve_id(const ResolveArgs& a, int i) { return a.ids_sm ? a.ids_sm[i] : a.ids[i]; }

__host__ __device__ inline size_t resolve_smem_bytes(int E, int n) {
  const int cap = n < E ? n : E;
  // inU[E] slotOf[E] U[cap] M[cap] fe[cap] vs[cap] vs2[cap] | mrec[cap] vu[cap] vu2[cap]
  size_t ints = 2 * static_cast<size_t>(E) + 5 * static_cast<size_t>(cap);
  ints = (ints + 1) & ~static_cast<size_t>(1);
  return ints * 4 + 3 * static_cast<size_t>(cap) * 8;
}

// The victim search's copy of the slot state in shared memory, after the
// arrays above: usage[S] int64, then a hit flag per slot.
__host__ __device__ inline size_t resolve_stage_bytes(int S) {
  return static_cast<size_t>(S) * 8 + ((static_cast<size_t>(S) + 15) & ~static_cast<size_t>(15));
}
// Host: check a prefetch call's arguments the same way (phi unused, no
// slot_ids) and fill the prefetch fields.
ft_status prefetch_prepare(const ft_cache_state* st, int32_t layer, const int32_t* pred_ids, int32_t T,
                           int32_t k, int32_t max_prefetch, int32_t* num_fetch, int32_t* fetch_fid,
                           int32_t* fetch_slot, int32_t max_list, int32_t* dev_status, size_t stage_cap,
                           ResolveArgs* out, size_t* smem_out);
// Host: check a resolve call's arguments and fill its device arguments,
// deciding whether the victim search may stage the slot state in shared
// memory: when the total stays within stage_cap bytes (FT_ERR_INVALID with a
// message when a check fails; `what` names the call).  *smem_out: the
// dynamic shared memory the resolve needs.
ft_status resolve_prepare(const ft_cache_state* st, int32_t layer, const int32_t* topk_ids, int32_t T,
                          int32_t k, int32_t frac_q16, int32_t* slot_ids, int32_t* num_fetch,
                          int32_t* fetch_fid, int32_t* fetch_slot, int32_t max_list, int32_t* dev_status,
                          const char* what, size_t stage_cap, ResolveArgs* out, size_t* smem_out);

namespace {

// The q* split in Q16 fixed point (phi = 2^16 * B_P / B_H).  Fetching f of
// m misses costs max(f*(2^16-phi), (m-f)*phi): the larger of the copy time
// and the host-path time, which run side by side.  The first term grows with
// f and the second falls, so the minimum sits next to their crossing
// f* = m*phi / 2^16.  With m*phi = 2^16*lo + r (0 <= r < 2^16), f = lo costs
// (m-lo)*phi and f = lo+1 costs (lo+1)*(2^16-phi); the second is strictly
// cheaper exactly when r + phi > 2^16, so that is when one more expert is
// fetched (equal costs keep the smaller count).  lo+1 never exceeds m: lo = m
// only at phi = 2^16, where r = 0.  phi == 0 applies no cap.
__device__ __forceinline__ int32_t split_q16_dev(int32_t m, int32_t phi) {
  if (m <= 0) return 0;
  if (phi <= 0) return m;
  const uint64_t prod = static_cast<uint64_t>(m) * static_cast<uint32_t>(phi);
  const uint32_t whole = static_cast<uint32_t>(prod >> 16), frac = static_cast<uint32_t>(prod & 0xffffu);
  return static_cast<int32_t>(whole + (frac + static_cast<uint32_t>(phi) > 65536u ? 1u : 0u));
}
// Is slot s owned by an expert of this call that is already resident (a hit)?
__device__ __forceinline__ bool is_hit_slot(const int32_t* __restrict__ owner, int s, int base,
                                            int E, const int* inU) {
  const int o = owner[s];
  return o >= base && o < base + E && inU[o - base] != 0;
}

__device__ __forceinline__ uint64_t ukey(int64_t u) {
  return static_cast<uint64_t>(u) ^ 0x8000000000000000ull;
}

// The small calls, n <= 32 ids and all valid, start in one warp: lane i
// holds pair i, its expert's slot before the update (map) and, on the first
// lane of each distinct expert (its leader), whether it hits.  When the q*
// split fetches nothing (every distinct expert hits, or the split or the
// evictable slots allow no fetch) the warp finishes the call: the state
// update is the usage of the hit slots and the recency of the distinct
// experts, the outputs are the map lookups.  When it fetches 1 to
// kResFastVictims experts, the warp ranks the misses by (recency desc, id
// asc) and lists the hit slots; the block then takes the victims
// (resolve_small_victims) and the warp installs them (resolve_small_finish).
// Either way the results are those of the general path below.
struct ResSmall {
  int nf, nhit;
  long long now;
  int fe[32];        // the fetched experts, by rank
  int hit[32];       // the slots the hits own (excluded from the victims)
  int vict[kResFastVictims];
  int lane_e[32];    // per pair: its expert
  int lane_slot[32]; // per pair: its slot before the update, -1 for a miss
  int lane_rank[32]; // per pair: its expert's rank among the misses, -1 for a hit
};

// Returns (warp-uniform) 1 when the call is done, 2 when the block goes on
// with the victims, 0 for the general path.
__device__ __forceinline__ int resolve_small(const ResolveArgs& a, ResSmall* sm, const int32_t* ids_sm) {
  const int lane = threadIdx.x & 31;
  const int n = a.n, E = a.E, base = a.layer * a.E;
  const int64_t now = *a.step;
  const int e = lane < n ? (ids_sm ? ids_sm[lane] : resolve_id(a, lane)) : -1;
  const bool bad = lane < n && (e < 0 || e >= E);
  if (__any_sync(0xffffffffu, bad)) return 0;
  const int s = lane < n ? a.map[base + e] : -1;
  const unsigned same = __match_any_sync(0xffffffffu, e);
  const int lead = __ffs(same) - 1;
  const bool leader = lane < n && lane == lead;
  const unsigned hitb = __ballot_sync(0xffffffffu, leader && s >= 0);
  const unsigned missb = __ballot_sync(0xffffffffu, leader && s < 0);
  const int nhit = __popc(hitb), m = __popc(missb);
  const int nf = max(0, min(split_q16_dev(m, a.phi), a.S - nhit));
  if (nf == 0) {
    if (leader) {
      if (s >= 0) a.usage[s] = now;
      a.recency[base + e] = now;
    }
    if (lane < n) {
      a.slot_ids[lane] = s;
      if (a.slot_ids_sm) a.slot_ids_sm[lane] = s;
    }
    for (int i = lane; i < a.max_list; i += 32) {
      a.fetch_fid[i] = -1;
      a.fetch_slot[i] = -1;
    }
    if (lane == 0) {
      *a.num_fetch = 0;
      if (a.num_fetch_sm) *a.num_fetch_sm = 0;
      *a.step = now + 1;
    }
    return 1;
  }
  if (nf > kResFastVictims) return 0;
  const bool miss = leader && s < 0;
  const int64_t rec = miss ? a.recency[base + e] : 0;
  int r = 0;  // this miss's rank: misses before it by (recency desc, id asc)
  for (int j = 0; j < 32; ++j) {
    const int64_t rj = __shfl_sync(0xffffffffu, rec, j);
    const int ej = __shfl_sync(0xffffffffu, e, j);
    if ((missb >> j) & 1u) r += (rj > rec) || (rj == rec && ej < e);
  }
  if (miss && r < nf) sm->fe[r] = e;
  if (leader && s >= 0) sm->hit[__popc(hitb & ((1u << lane) - 1u))] = s;
  const int rank = __shfl_sync(0xffffffffu, miss ? r : -1, lead);  // the pair's expert's rank
  if (lane < n) {
    sm->lane_e[lane] = e;
    sm->lane_slot[lane] = s;
    sm->lane_rank[lane] = rank;
  }
  if (lane == 0) {
    sm->nf = nf;
    sm->nhit = nhit;
    sm->now = now;
  }
  return 2;
}

// The block: nf rounds of a block-wide argmin of (usage, slot) over the
// slots that no hit owns and no earlier round took, which yields the nf
// victims already in (usage asc, slot asc) order.  Every thread calls it.
__device__ __forceinline__ void resolve_small_victims(const ResolveArgs& a, ResSmall* sm) {
  __shared__ long long s_vu[32];
  __shared__ int s_vs[32];
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = (nt + 31) >> 5;
  const int nf = sm->nf, nhit = sm->nhit;
  for (int r = 0; r < nf; ++r) {
    long long bu = LLONG_MAX;
    int bs = INT_MAX;
    for (int s = tid; s < a.S; s += nt) {
      bool skip = false;
      for (int j = 0; j < nhit; ++j) skip |= sm->hit[j] == s;
      for (int j = 0; j < r; ++j) skip |= sm->vict[j] == s;
      if (skip) continue;
      const long long u = a.usage[s];
      if (u < bu || (u == bu && s < bs)) {
        bu = u;
        bs = s;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const long long ou = __shfl_xor_sync(0xffffffffu, bu, o);
      const int os = __shfl_xor_sync(0xffffffffu, bs, o);
      if (ou < bu || (ou == bu && os < bs)) {
        bu = ou;
        bs = os;
      }
    }
    if (lane == 0) {
      s_vu[warp] = bu;
      s_vs[warp] = bs;
    }
    __syncthreads();
    if (warp == 0) {
      bu = lane < nw ? s_vu[lane] : LLONG_MAX;
      bs = lane < nw ? s_vs[lane] : INT_MAX;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const long long ou = __shfl_xor_sync(0xffffffffu, bu, o);
        const int os = __shfl_xor_sync(0xffffffffu, bs, o);
        if (ou < bu || (ou == bu && os < bs)) {
          bu = ou;
          bs = os;
        }
      }
      if (lane == 0) {
        if (bs == INT_MAX) {  // fewer eligible slots than nf: an inconsistent state
          record_status(a.dev_status, FT_ERR_RANGE);
          bs = 0;
        }
        sm->vict[r] = bs;
      }
    }
    __syncthreads();
  }
}

// The warp: evict the victims' owners, install the fetched experts, the
// usage of hit and fetched slots, the recency of every distinct expert,
// then the outputs.
__device__ __forceinline__ void resolve_small_finish(const ResolveArgs& a, const ResSmall* sm) {
  const int lane = threadIdx.x & 31;
  const int n = a.n, base = a.layer * a.E, nf = sm->nf;
  const int64_t now = sm->now;
  if (lane < sm->nhit) a.usage[sm->hit[lane]] = now;
  if (lane < nf) {
    const int old = a.slot_owner[sm->vict[lane]];
    if (old >= 0) a.map[old] = -1;
  }
  __syncwarp();
  if (lane < nf) {
    const int e = sm->fe[lane], v = sm->vict[lane];
    a.slot_owner[v] = base + e;
    a.map[base + e] = v;
    a.usage[v] = now;
  }
  const int e = lane < n ? sm->lane_e[lane] : -1;
  const unsigned same = __match_any_sync(0xffffffffu, e);
  if (lane < n && lane == __ffs(same) - 1) a.recency[base + e] = now;
  if (lane < n) {
    const int s0 = sm->lane_slot[lane], rk = sm->lane_rank[lane];
    const int sl = s0 >= 0 ? s0 : (rk >= 0 && rk < nf ? sm->vict[rk] : -1);
    a.slot_ids[lane] = sl;
    if (a.slot_ids_sm) a.slot_ids_sm[lane] = sl;
  }
  for (int i = lane; i < a.max_list; i += 32) {
    a.fetch_fid[i] = i < nf ? base + sm->fe[i] : -1;
    a.fetch_slot[i] = i < nf ? sm->vict[i] : -1;
  }
  if (lane == 0) {
    *a.num_fetch = nf;
    if (a.num_fetch_sm) *a.num_fetch_sm = nf;
    *a.step = now + 1;
  }
}
// The small path (n <= 32, not a prefetch) as a whole, for a kernel to inline
// so that it reads its arguments straight from the parameter space (through
// the reference of the non-inlined resolve_block every argument read is a
// generic load).  Every thread of the block calls it; returns (block-uniform)
// true when the call is done, false for resolve_block(..., small = false).
__device__ __forceinline__ bool resolve_small_path(const ResolveArgs& a, const int32_t* ids_sm) {
  __shared__ int s_done;
  __shared__ ResSmall s_small;
  if (threadIdx.x < 32) {
    const int done = resolve_small(a, &s_small, ids_sm);
    if (threadIdx.x == 0) s_done = done;
  }
  __syncthreads();
  const int done = s_done;
  if (done == 2) {
    resolve_small_victims(a, &s_small);
    if (threadIdx.x < 32) resolve_small_finish(a, &s_small);
  }
  return done != 0;
}

// The whole resolve call by one CTA (any block size; every thread calls it).
// smem: the dynamic shared memory resolve_prepare asked for.  ids must be
// readable by the CTA (written by an earlier grid, or by this CTA before a
// __syncthreads).
// ids_sm, when not null, is a shared-memory copy of ids [n] that this CTA
// wrote before a __syncthreads, read instead of a.ids / a.ids_sm.  small:
// false when the caller has run the small path (resolve_small_path) already.
__device__ __noinline__ void resolve_block(const ResolveArgs& a, unsigned char* smem, const int32_t* ids_sm = nullptr,
                                          bool small = true) {
  const int E = a.E, n = a.n, S = a.S;
  const int cap = n < E ? n : E;
  int* inU = reinterpret_cast<int*>(smem);
  int* slotOf = inU + E;
  int* U = slotOf + E;
  int* M = U + cap;
  int* fe = M + cap;
  int* vs = fe + cap;
  int* vs2 = vs + cap;
  size_t ints = 2 * static_cast<size_t>(E) + 5 * static_cast<size_t>(cap);
  ints = (ints + 1) & ~static_cast<size_t>(1);
  int64_t* mrec = reinterpret_cast<int64_t*>(smem + ints * 4);
  int64_t* vu = mrec + cap;
  int64_t* vu2 = vu + cap;

  __shared__ int scan_scratch[33];
  __shared__ int s_bad, s_nU, s_m, s_nf, s_cnt;
  __shared__ unsigned int hist[256];
  __shared__ unsigned long long s_kmin, s_kmax, s_prefix;
  __shared__ int s_krem, s_cmin;
  __shared__ long long s_now;

  const int tid = threadIdx.x;
  const int nt = blockDim.x;
  const int base = a.layer * E;

  if (small && n <= 32 && !a.prefetch) {
    __shared__ int s_done;
    __shared__ ResSmall s_small;
    if (tid < 32) {
      const int done = resolve_small(a, &s_small, ids_sm);
      if (tid == 0) s_done = done;
    }
    __syncthreads();
    if (s_done == 1) return;
    if (s_done == 2) {
      resolve_small_victims(a, &s_small);
      if (tid < 32) resolve_small_finish(a, &s_small);
      return;
    }
  }

  for (int e = tid; e < E; e += nt) {
    inU[e] = 0;
    slotOf[e] = -1;
  }
  if (tid == 0) {
    s_bad = 0;
    s_now = *a.step;
  }
  __syncthreads();
  for (int i = tid; i < n; i += nt) {
    const int e = ids_sm ? ids_sm[i] : resolve_id(a, i);
    if (e < 0 || e >= E)
      s_bad = 1;
    else
      inU[e] = 1;
  }
  __syncthreads();
  if (s_bad) {
    if (!a.prefetch)
      for (int i = tid; i < n; i += nt) {
        a.slot_ids[i] = -1;
        if (a.slot_ids_sm) a.slot_ids_sm[i] = -1;
      }
    for (int i = tid; i < a.max_list; i += nt) {
      a.fetch_fid[i] = -1;
      a.fetch_slot[i] = -1;
    }
    if (tid == 0) {
      *a.num_fetch = 0;
      if (a.num_fetch_sm) *a.num_fetch_sm = 0;
      record_status(a.dev_status, FT_ERR_BAD_ID);
    }
    return;
  }

  // 1. U = distinct experts, ascending (ordered compaction over contiguous ranges)
  {
    const int per = (E + nt - 1) / nt;
    const int lo = min(E, tid * per), hi = min(E, lo + per);
    int cnt = 0;
    for (int e = lo; e < hi; ++e) cnt += inU[e];
    int total;
    int off = block_excl_scan(cnt, scan_scratch, &total);
    for (int e = lo; e < hi; ++e)
      if (inU[e]) U[off++] = e;
    if (tid == 0) s_nU = total;
  }
  __syncthreads();
  const int nU = s_nU;

  // 2. hits / misses; misses keep ascending order
  {
    const int per = (nU + nt - 1) / nt;
    const int lo = min(nU, tid * per), hi = min(nU, lo + per);
    int cnt = 0;
    for (int i = lo; i < hi; ++i) {
      const int e = U[i];
      const int s = a.map[base + e];
      slotOf[e] = s;
      cnt += (s < 0);
    }
    int total;
    int off = block_excl_scan(cnt, scan_scratch, &total);
    for (int i = lo; i < hi; ++i) {
      const int e = U[i];
      if (slotOf[e] < 0) {
        M[off] = e;
        mrec[off] = a.recency[base + e];
        ++off;
      }
    }
    if (tid == 0) {
      s_m = total;
      const int nhit = nU - total;
      const int evictable = S - nhit;
      int nf = split_q16_dev(total, a.phi);
      nf = min(nf, evictable);
      s_nf = max(nf, 0);
      s_cnt = 0;
    }
  }
  __syncthreads();
  const int64_t now = s_now;
  // The victim search's view of the slots: whether a slot may not be a victim
  // (a hit; for a prefetch also a held slot with usage >= now-1, which the
  // layer resolved last may still be reading, or an earlier prefetch not yet
  // consumed), and its usage.  When the host found room (a.staged), one
  // coalesced pass copies both into shared memory, so the scans below (several
  // per call) read shared memory, not L2.
  int64_t* su = nullptr;
  unsigned char* shit = nullptr;
  auto blocked_global = [&](int s) -> bool {
    if (is_hit_slot(a.slot_owner, s, base, E, inU)) return true;
    return a.prefetch && a.slot_owner[s] >= 0 && a.usage[s] >= now - 1;
  };
  if (a.prefetch) {
    // a prefetch's count is capped by its eligible slots: count them (and stage)
    if (a.staged) {
      su = reinterpret_cast<int64_t*>(smem + resolve_smem_bytes(E, n));
      shit = reinterpret_cast<unsigned char*>(su + S);
    }
    int c = 0;
    for (int s = tid; s < S; s += nt) {
      const bool b = blocked_global(s);
      if (su) {
        su[s] = a.usage[s];
        shit[s] = b;
      }
      c += b;
    }
    c = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(c)));
    if ((tid & 31) == 0) atomicAdd(&s_cnt, c);
    __syncthreads();
    if (tid == 0) s_nf = max(0, min(min(s_m, a.max_prefetch), S - s_cnt));
    __syncthreads();
  }
  const int m = s_m, nf = s_nf;

  // 3. the fetched misses: rank by (recency desc, id asc)
  for (int j = tid; j < m; j += nt) {
    const int64_t rj = mrec[j];
    const int ej = M[j];
    int r = 0;
    for (int j2 = 0; j2 < m; ++j2) {
      const int64_t r2 = mrec[j2];
      r += (r2 > rj) || (r2 == rj && M[j2] < ej);
    }
    if (r < nf) fe[r] = ej;
  }

  // 4. the victims: the nf smallest (usage, slot) among the slots that may be
  // victims (staged first for a resolve, see above).
  if (nf > 0 && a.staged && !a.prefetch) {
    su = reinterpret_cast<int64_t*>(smem + resolve_smem_bytes(E, n));
    shit = reinterpret_cast<unsigned char*>(su + S);
#pragma unroll 4
    for (int s = tid; s < S; s += nt) {
      su[s] = a.usage[s];
      shit[s] = is_hit_slot(a.slot_owner, s, base, E, inU);
    }
    __syncthreads();
  }
  auto slot_hit = [&](int s) -> bool { return shit ? shit[s] != 0 : blocked_global(s); };
  auto slot_use = [&](int s) -> int64_t { return su ? su[s] : a.usage[s]; };
  if (nf > 0 && nf <= kResFastVictims) {
    // few victims (the usual decode call): nf rounds of a block-wide argmin
    // of (usage, slot) over the eligible slots not taken yet, which yields
    // the nf smallest pairs already in (usage asc, slot asc) order
    __shared__ long long s_wu[32];
    __shared__ int s_ws[32];
    const int lane = tid & 31, warp = tid >> 5, nw = (nt + 31) >> 5;
    for (int r = 0; r < nf; ++r) {
      long long bu = LLONG_MAX;
      int bs = INT_MAX;
      for (int s = tid; s < S; s += nt) {
        if (slot_hit(s)) continue;
        bool taken = false;
        for (int j = 0; j < r; ++j) taken |= vs2[j] == s;
        if (taken) continue;
        const long long u = slot_use(s);
        if (u < bu || (u == bu && s < bs)) {
          bu = u;
          bs = s;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const long long ou = __shfl_xor_sync(0xffffffffu, bu, o);
        const int os = __shfl_xor_sync(0xffffffffu, bs, o);
        if (ou < bu || (ou == bu && os < bs)) {
          bu = ou;
          bs = os;
        }
      }
      if (lane == 0) {
        s_wu[warp] = bu;
        s_ws[warp] = bs;
      }
      __syncthreads();
      if (warp == 0) {
        bu = lane < nw ? s_wu[lane] : LLONG_MAX;
        bs = lane < nw ? s_ws[lane] : INT_MAX;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const long long ou = __shfl_xor_sync(0xffffffffu, bu, o);
          const int os = __shfl_xor_sync(0xffffffffu, bs, o);
          if (ou < bu || (ou == bu && os < bs)) {
            bu = ou;
            bs = os;
          }
        }
        if (lane == 0) {
          if (bs == INT_MAX) {  // fewer eligible slots than nf: an inconsistent state
            record_status(a.dev_status, FT_ERR_RANGE);
            bs = 0;
          }
          vs2[r] = bs;
          vu2[r] = bu;
        }
      }
      __syncthreads();
    }
  } else if (nf > 0) {
    unsigned long long kmin = ~0ull, kmax = 0ull;
    for (int s = tid; s < S; s += nt) {
      if (slot_hit(s)) continue;
      const unsigned long long k = ukey(slot_use(s));
      kmin = min(kmin, k);
      kmax = max(kmax, k);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
      kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    }
    if (tid == 0) {
      s_kmin = ~0ull;
      s_kmax = 0ull;
      s_cmin = 0;
    }
    __syncthreads();
    if ((tid & 31) == 0) {
      atomicMin(&s_kmin, kmin);
      atomicMax(&s_kmax, kmax);
    }
    __syncthreads();
    const unsigned long long gmin = s_kmin, gmax = s_kmax;
    int c = 0;
    for (int s = tid; s < S; s += nt)
      if (!slot_hit(s) && ukey(slot_use(s)) == gmin) ++c;
    c = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(c)));
    if ((tid & 31) == 0 && c != 0) atomicAdd(&s_cmin, c);
    if (tid == 0) {
      s_prefix = 0ull;
      s_krem = nf;
    }
    __syncthreads();
    unsigned long long tau;
    if (s_cmin >= nf || gmax == gmin) {
      tau = gmin;
    } else {
      // radix select over d = key - min, 8 bits per pass from the top digit
      const unsigned long long range = gmax - gmin;
      const int nbits = 64 - __clzll(static_cast<long long>(range));
      for (int shift = ((nbits - 1) / 8) * 8; shift >= 0; shift -= 8) {
        for (int b = tid; b < 256; b += nt) hist[b] = 0;
        __syncthreads();
        const unsigned long long pre = s_prefix;
        // histogram of the digit: one shared-memory add per distinct digit of
        // a warp (slots with close usage share digits, and per-slot adds to
        // one counter would serialise)
        for (int s0 = 0; s0 < S; s0 += nt) {
          const int s = s0 + tid;
          int bin = -1;
          if (s < S && !slot_hit(s)) {
            const unsigned long long d = ukey(slot_use(s)) - gmin;
            const bool match = (shift + 8 >= 64) ? true : ((d >> (shift + 8)) == pre);
            if (match) bin = static_cast<int>((d >> shift) & 255ull);
          }
          const unsigned peers = __match_any_sync(0xffffffffu, bin);
          if (bin >= 0 && (tid & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], static_cast<unsigned>(__popc(peers)));
        }
        __syncthreads();
        if (tid < 32) {
          // the first digit at which the running count reaches krem: lane l
          // sums digits 8l..8l+7, a warp scan gives the lane, that lane the digit
          const int lane = tid;
          unsigned c8[8];
          unsigned loc = 0;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            c8[j] = hist[8 * lane + j];
            loc += c8[j];
          }
          unsigned incl = loc;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
          }
          const int krem = s_krem;
          const unsigned reach = __ballot_sync(0xffffffffu, incl >= static_cast<unsigned>(krem));
          const int first = reach ? __ffs(reach) - 1 : 31;
          if (lane == first) {
            unsigned cum = incl - loc;
            int b = 0;
            for (; b < 8; ++b) {
              if (cum + c8[b] >= static_cast<unsigned>(krem)) break;
              cum += c8[b];
            }
            const int digit = reach ? 8 * lane + b : 256;  // 256: no digit reaches krem (cannot happen)
            s_krem = krem - static_cast<int>(cum);
            s_prefix = (pre << 8) | static_cast<unsigned long long>(digit);
          }
        }
        __syncthreads();
      }
      tau = gmin + s_prefix;
    }
    // keys below tau: all taken (unordered append)
    if (tid == 0) s_cnt = 0;
    __syncthreads();
    for (int s = tid; s < S; s += nt) {
      if (slot_hit(s)) continue;
      const int64_t u = slot_use(s);
      if (ukey(u) < tau) {
        const int p = atomicAdd(&s_cnt, 1);
        if (p < nf) {
          vs[p] = s;
          vu[p] = u;
        }
      }
    }
    __syncthreads();
    const int nless = min(s_cnt, nf);
    const int need = nf - nless;
    // keys equal to tau: the lowest slots first (ordered scan over slots)
    int running = 0;
    for (int t0 = 0; t0 < S && running < need; t0 += nt) {
      const int s = t0 + tid;
      int flag = 0;
      int64_t u = 0;
      if (s < S && !slot_hit(s)) {
        u = slot_use(s);
        flag = (ukey(u) == tau);
      }
      int total;
      const int pos = block_excl_scan(flag, scan_scratch, &total) + running;
      if (flag && pos < need) {
        vs[nless + pos] = s;
        vu[nless + pos] = u;
      }
      running += total;
    }
    __syncthreads();
    // order the victims by (usage asc, slot asc)
    for (int i = tid; i < nf; i += nt) {
      const int64_t ui = vu[i];
      const int si = vs[i];
      int r = 0;
      for (int j = 0; j < nf; ++j) r += (vu[j] < ui) || (vu[j] == ui && vs[j] < si);
      vs2[r] = si;
      vu2[r] = ui;
    }
  }
  __syncthreads();

  // 5. state update (a prefetch routes nothing: hit usage, recency and the
  // step stay as they are)
  if (!a.prefetch)
    for (int i = tid; i < nU; i += nt) {
      const int s = slotOf[U[i]];
      if (s >= 0) a.usage[s] = now;
    }
  for (int i = tid; i < nf; i += nt) {
    const int v = vs2[i];
    const int old = a.slot_owner[v];
    if (old >= 0) a.map[old] = -1;
  }
  __syncthreads();
  for (int i = tid; i < nf; i += nt) {
    const int e = fe[i];
    const int v = vs2[i];
    a.slot_owner[v] = base + e;
    a.map[base + e] = v;
    a.usage[v] = now;
    slotOf[e] = v;
  }
  if (!a.prefetch)
    for (int i = tid; i < nU; i += nt) a.recency[base + U[i]] = now;
  __syncthreads();

  // 6. outputs
  if (!a.prefetch)
    for (int i = tid; i < n; i += nt) {
      const int sl = slotOf[ids_sm ? ids_sm[i] : resolve_id(a, i)];
      a.slot_ids[i] = sl;
      if (a.slot_ids_sm) a.slot_ids_sm[i] = sl;
    }
  for (int i = tid; i < a.max_list; i += nt) {
    a.fetch_fid[i] = (i < nf) ? base + fe[i] : -1;
    a.fetch_slot[i] = (i < nf) ? vs2[i] : -1;
  }
  if (tid == 0) {
    *a.num_fetch = nf;
    if (a.num_fetch_sm) *a.num_fetch_sm = nf;
    if (!a.prefetch) *a.step = now + 1;
  }
}

}  // namespace
}  // namespace ft
