// cache.cu -- the global slot cache on the device: the Q16 q* split, the
// one-kernel resolve (dedup, residency, q*, recency-ranked fetch choice,
// single-scan K-victim selection, id rewrite) and the fetch copy.
//
// Sources: "FreeToken 딥다이브" (fiv.co.kr), design patterns 2, 3, 5;
// "FreeToken: 让消费级电脑跑起 284B MoE" (fengjutian.github.io), secs. 4, 6.
#include "ft_async.cuh"
#include "ft_common.cuh"

namespace ft {
namespace {

constexpr int kResThreads = 1024;
constexpr int kResMaxE = 4096;
constexpr int kResMaxN = 4096;
constexpr size_t kResSmemCap = 220 * 1024;  // dynamic shared memory the resolve kernel may use

// The q* rule in Q16 fixed point: lo = floor(m*phi / 2^16); fetch lo or lo+1,
// whichever gives the smaller slower-branch time max(f*(2^16-phi), (m-f)*phi)
// (ties to lo), capped at m.  phi == 0 applies no cap.  64-bit intermediates.
__device__ __forceinline__ int32_t split_q16_dev(int32_t m, int32_t phi) {
  if (m <= 0) return 0;
  if (phi <= 0) return m;
  const int64_t q = 65536;
  const int64_t M = m, P = phi;
  const int64_t lo = (M * P) >> 16;
  const int64_t c_lo = max(lo * (q - P), (M - lo) * P);
  const int64_t c_hi = max((lo + 1) * (q - P), (M - lo - 1) * P);
  const int64_t f = (c_lo <= c_hi) ? lo : lo + 1;
  return static_cast<int32_t>(min(M, f));
}

__global__ void split_q16_kernel(const int32_t* __restrict__ m, int32_t n, int32_t phi,
                                 int32_t* __restrict__ out) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    out[i] = split_q16_dev(m[i], phi);
}

struct ResolveArgs {
  int32_t E, S, layer, n, phi, max_list;
  int32_t staged;  // 1: the victim search reads the slots' usage and hit flags from shared memory
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
};

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

// Is slot s owned by an expert of this call that is already resident (a hit)?
__device__ __forceinline__ bool is_hit_slot(const int32_t* __restrict__ owner, int s, int base,
                                            int E, const int* inU) {
  const int o = owner[s];
  return o >= base && o < base + E && inU[o - base] != 0;
}

__device__ __forceinline__ uint64_t ukey(int64_t u) {
  return static_cast<uint64_t>(u) ^ 0x8000000000000000ull;
}

// The common small case in one warp: n <= 32 ids, all valid, and the q*
// split fetches nothing (every distinct expert hits, or the split or the
// evictable slots allow no fetch).  Then the state update is only the usage
// of the hit slots and the recency of the distinct experts, and the outputs
// are the map lookups -- the same results as the general path below.
// Returns true (warp-uniform) when it has done the whole call.
__device__ bool resolve_small_no_fetch(const ResolveArgs& a) {
  const int lane = threadIdx.x & 31;
  const int n = a.n, E = a.E, base = a.layer * a.E;
  const int64_t now = *a.step;
  const int e = lane < n ? a.ids[lane] : -1;
  const bool bad = lane < n && (e < 0 || e >= E);
  if (__any_sync(0xffffffffu, bad)) return false;
  const int s = lane < n ? a.map[base + e] : -1;
  const unsigned same = __match_any_sync(0xffffffffu, e);
  const bool leader = lane < n && lane == __ffs(same) - 1;
  const int nhit = __popc(__ballot_sync(0xffffffffu, leader && s >= 0));
  const int m = __popc(__ballot_sync(0xffffffffu, leader && s < 0));
  const int nf = max(0, min(split_q16_dev(m, a.phi), a.S - nhit));
  if (nf > 0) return false;
  if (leader) {
    if (s >= 0) a.usage[s] = now;
    a.recency[base + e] = now;
  }
  if (lane < n) a.slot_ids[lane] = s;
  for (int i = lane; i < a.max_list; i += 32) {
    a.fetch_fid[i] = -1;
    a.fetch_slot[i] = -1;
  }
  if (lane == 0) {
    *a.num_fetch = 0;
    *a.step = now + 1;
  }
  return true;
}

__global__ void __launch_bounds__(kResThreads, 1) resolve_kernel(ResolveArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
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
  pdl_wait();               // ids come from the previous kernel (route)
  pdl_launch_dependents();  // the next call (fetch) may start its launch now

  if (n <= 32) {
    __shared__ int s_done;
    if (tid < 32) {
      const bool done = resolve_small_no_fetch(a);
      if (tid == 0) s_done = done;
    }
    __syncthreads();
    if (s_done) return;
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
    const int e = a.ids[i];
    if (e < 0 || e >= E)
      s_bad = 1;
    else
      inU[e] = 1;
  }
  __syncthreads();
  if (s_bad) {
    for (int i = tid; i < n; i += nt) a.slot_ids[i] = -1;
    for (int i = tid; i < a.max_list; i += nt) {
      a.fetch_fid[i] = -1;
      a.fetch_slot[i] = -1;
    }
    if (tid == 0) {
      *a.num_fetch = 0;
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
    }
  }
  __syncthreads();
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

  // 4. the victims: the nf smallest (usage, slot) among non-hit slots.  Each
  // scan below reads a slot's usage and whether it is a hit; when the host
  // found room (a.staged), one coalesced pass copies both into shared memory
  // first, so the scans (several per call) read shared memory, not L2.
  int64_t* su = nullptr;
  unsigned char* shit = nullptr;
  if (nf > 0 && a.staged) {
    su = reinterpret_cast<int64_t*>(smem + resolve_smem_bytes(E, n));
    shit = reinterpret_cast<unsigned char*>(su + S);
#pragma unroll 4
    for (int s = tid; s < S; s += nt) {
      su[s] = a.usage[s];
      shit[s] = is_hit_slot(a.slot_owner, s, base, E, inU);
    }
    __syncthreads();
  }
  auto slot_hit = [&](int s) -> bool { return shit ? shit[s] != 0 : is_hit_slot(a.slot_owner, s, base, E, inU); };
  auto slot_use = [&](int s) -> int64_t { return su ? su[s] : a.usage[s]; };
  if (nf > 0) {
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
    atomicAdd(&s_cmin, c);
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
        for (int s = tid; s < S; s += nt) {
          if (slot_hit(s)) continue;
          const unsigned long long d = ukey(slot_use(s)) - gmin;
          const bool match = (shift + 8 >= 64) ? true : ((d >> (shift + 8)) == pre);
          if (match) atomicAdd(&hist[(d >> shift) & 255ull], 1u);
        }
        __syncthreads();
        if (tid == 0) {
          int krem = s_krem;
          int b = 0;
          unsigned int cum = 0;
          for (; b < 256; ++b) {
            if (cum + hist[b] >= static_cast<unsigned int>(krem)) break;
            cum += hist[b];
          }
          s_krem = krem - static_cast<int>(cum);
          s_prefix = (pre << 8) | static_cast<unsigned long long>(b);
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

  // 5. state update
  const int64_t now = s_now;
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
  for (int i = tid; i < nU; i += nt) a.recency[base + U[i]] = now;
  __syncthreads();

  // 6. outputs
  for (int i = tid; i < n; i += nt) a.slot_ids[i] = slotOf[a.ids[i]];
  for (int i = tid; i < a.max_list; i += nt) {
    a.fetch_fid[i] = (i < nf) ? base + fe[i] : -1;
    a.fetch_slot[i] = (i < nf) ? vs2[i] : -1;
  }
  if (tid == 0) {
    *a.num_fetch = nf;
    *a.step = now + 1;
  }
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

int g_num_sms = 0;

int num_sms() {
  if (g_num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_num_sms <= 0) g_num_sms = 148;
  }
  return g_num_sms;
}

}  // namespace
}  // namespace ft

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
  FT_REQUIRE(st != nullptr, "resolve: state is NULL");
  FT_REQUIRE(st->L > 0 && st->E > 0 && st->S >= 0, "resolve: bad L/E/S %d/%d/%d", st->L, st->E,
             st->S);
  FT_REQUIRE(st->E <= ft::kResMaxE, "resolve: E %d > %d", st->E, ft::kResMaxE);
  FT_REQUIRE(static_cast<int64_t>(st->L) * st->E < (1ll << 31), "resolve: L*E overflows int32");
  FT_REQUIRE(layer >= 0 && layer < st->L, "resolve: layer %d outside [0, %d)", layer, st->L);
  FT_REQUIRE(T >= 0 && k >= 1, "resolve: T=%d k=%d", T, k);
  const int64_t n64 = static_cast<int64_t>(T) * k;
  FT_REQUIRE(n64 <= ft::kResMaxN, "resolve: T*k = %lld > %d", static_cast<long long>(n64),
             ft::kResMaxN);
  FT_REQUIRE(frac_q16 >= 0 && frac_q16 <= 65536, "resolve: frac_q16 %d outside [0, 65536]",
             frac_q16);
  const int n = static_cast<int>(n64);
  const int need = n < st->S ? n : st->S;
  FT_REQUIRE(max_list >= need, "resolve: max_list %d < min(T*k, S) = %d", max_list, need);
  FT_REQUIRE(st->map && st->recency && st->step && num_fetch && fetch_fid && fetch_slot,
             "resolve: NULL pointer");
  FT_REQUIRE(st->S == 0 || (st->slot_owner && st->usage), "resolve: NULL slot arrays");
  FT_REQUIRE(n == 0 || (topk_ids && slot_ids), "resolve: NULL ids");
  ft::ResolveArgs a;
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
  // the slot state is staged in shared memory when it fits beside the
  // resolve's own arrays (every cache up to ~24k slots at E <= 256)
  size_t smem = ft::resolve_smem_bytes(st->E, n);
  const size_t staged = smem + ft::resolve_stage_bytes(st->S);
  a.staged = (st->S > 0 && staged <= ft::kResSmemCap) ? 1 : 0;
  if (a.staged) smem = staged;
  if (smem > 48 * 1024) {
    static const size_t kMax = ft::kResSmemCap;
    cudaError_t e = cudaFuncSetAttribute(ft::resolve_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kMax));
    if (e != cudaSuccess)
      return ft::fail(FT_ERR_CUDA, "resolve: smem attribute: %s", cudaGetErrorString(e));
  }
  // small calls usually finish in the one-warp path; 256 threads keep the
  // rest cheap to synchronise.  Larger calls get the whole block.
  const int threads = n <= 32 ? 256 : ft::kResThreads;
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, ft::resolve_kernel, a);
  if (e != cudaSuccess) return ft::fail(FT_ERR_CUDA, "resolve_slots: %s", cudaGetErrorString(e));
  return ft::launch_check("resolve_slots");
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
  const int grid = static_cast<int>(std::min<uint64_t>(items, static_cast<uint64_t>(ft::num_sms())));
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
