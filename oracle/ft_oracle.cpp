// ft_oracle.cpp -- plain, slow, single-threaded CPU oracle for the routed,
// quantized expert-FFN MoE layer.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
// call this file; only the tests, the package smoke check and the CPU-baseline
// leg of the benchmark use it.  It shares no code, header, table or constant
// with the CUDA library: every number format is decoded here from its
// definition, and every step is written out in the order the source pages
// describe it.  Floating point is fp64 throughout; integer work is exact.
//
// Sources (page title, section):
//   [FT-KR]  "FreeToken 딥다이브" -- design pattern 2 (q* split in Q16 fixed
//            point and its Python reference), pattern 3 (-1 sentinel and
//            masking), pattern 5 (two LRUs, flat id layer*E+expert).
//   [FT-ZH]  "FreeToken: 让消费级电脑跑起 284B MoE" -- sec. 4 (global slot cache,
//            one slot = one (layer, expert) with gate/up/down), sec. 6 (q*
//            derivation, exact partial-sum merge, one kernel does dedup /
//            residency / q / victims / id rewrite, single-pass K-victim scan).
//   [NVMe]   "NVMe에서 전문가(experts)를 스트리밍하여 8GB GPU에서 133GB MoE" --
//            "Why this model" (2560x640 experts, NVFP4) and engine step 1
//            (expert block gate|up|down|gate_scale|up_scale|down_scale).
//   [Edge0]  "SSD 가중치층으로 35B MoE를 ..." -- "How it works":
//            down(silu(gate(x)) * up(x)) and the dequantised reference.
//
// Parity status of each function is stated beside it; all are pinned by the
// "not gpu" tests except where a function says otherwise.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

// ---------------------------------------------------------------- formats --

// bf16: the upper 16 bits of an IEEE binary32.
double bf16_value(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

// IEEE binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits.
double fp16_value(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0) {
    v = std::ldexp(static_cast<double>(m), -24);  // 2^-14 * m/1024
  } else if (e == 31) {
    v = (m == 0) ? INFINITY : NAN;
  } else {
    v = std::ldexp(1.0 + m / 1024.0, e - 15);
  }
  return sign ? -v : v;
}

// OCP FP4 E2M1: bit 3 sign, bits 2:1 exponent (bias 1), bit 0 mantissa.
// Exponent field 0 is subnormal: 2^(1-1) * (m/2).  No inf / NaN.
double e2m1_value(int code) {
  int sign = (code >> 3) & 1;
  int e = (code >> 1) & 3;
  int m = code & 1;
  double v = (e == 0) ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, e - 1);
  return sign ? -v : v;
}

// OCP FP8 E4M3 ("fn"): bit 7 sign, bits 6:3 exponent (bias 7), bits 2:0
// mantissa.  Exponent 0 is subnormal 2^-6 * m/8.  S.1111.111 is NaN; there is
// no infinity.
double e4m3_value(int code) {
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 0xf;
  int m = code & 7;
  double v;
  if (e == 15 && m == 7) {
    v = NAN;
  } else if (e == 0) {
    v = std::ldexp(static_cast<double>(m), -9);
  } else {
    v = std::ldexp(1.0 + m / 8.0, e - 7);
  }
  return sign ? -v : v;
}

// ----------------------------------------------------------- expert block --
// One expert block holds gate | up | down | gate_scale | up_scale | down_scale
// in that order ([NVMe] engine step 1).  gate and up are [I, H], down is
// [H, I], all row-major with the reduction (K) axis contiguous.  Two 4-bit
// codes share a byte, the low nibble holding the even K index.
//   fmt 0 (int4, group g): code q in 0..15 means (q - 8) * s, s an fp16 scale
//         per g consecutive K elements of a row.
//   fmt 1 (NVFP4): code is E2M1, s an E4M3 scale per 16 K elements, times an
//         fp32 per-tensor scale held outside the block.

enum { FMT_INT4 = 0, FMT_NVFP4 = 1 };

struct Layout {
  size_t off[6];  // gate, up, down, gate_scale, up_scale, down_scale
  size_t total;
};

bool make_layout(int fmt, int H, int I, int g, Layout* L) {
  if (H <= 0 || I <= 0 || (H & 1) || (I & 1)) return false;
  size_t scale_bytes;
  int block;
  if (fmt == FMT_INT4) {
    if (g <= 0 || H % g || I % g) return false;
    block = g;
    scale_bytes = 2;
  } else if (fmt == FMT_NVFP4) {
    if (H % 16 || I % 16) return false;
    block = 16;
    scale_bytes = 1;
  } else {
    return false;
  }
  size_t gate = static_cast<size_t>(I) * H / 2;
  size_t down = static_cast<size_t>(H) * I / 2;
  size_t gs = static_cast<size_t>(I) * (H / block) * scale_bytes;
  size_t ds = static_cast<size_t>(H) * (I / block) * scale_bytes;
  L->off[0] = 0;
  L->off[1] = gate;
  L->off[2] = 2 * gate;
  L->off[3] = 2 * gate + down;
  L->off[4] = L->off[3] + gs;
  L->off[5] = L->off[4] + gs;
  L->total = L->off[5] + ds;
  return true;
}

int nibble(const uint8_t* codes, size_t index) {
  uint8_t b = codes[index >> 1];
  return (index & 1) ? (b >> 4) : (b & 0xf);
}

// Dequantise one [rows, K] matrix of the block into out (row-major, fp64).
void dequant_matrix(int fmt, const uint8_t* codes, const uint8_t* scales,
                    int rows, int K, int g, double tensor_scale, double* out) {
  for (int r = 0; r < rows; ++r) {
    for (int c = 0; c < K; ++c) {
      size_t idx = static_cast<size_t>(r) * K + c;
      int q = nibble(codes, idx);
      double w;
      if (fmt == FMT_INT4) {
        size_t si = static_cast<size_t>(r) * (K / g) + c / g;
        uint16_t sbits = static_cast<uint16_t>(scales[2 * si] | (scales[2 * si + 1] << 8));
        w = (q - 8) * fp16_value(sbits);
      } else {
        size_t si = static_cast<size_t>(r) * (K / 16) + c / 16;
        w = e2m1_value(q) * e4m3_value(scales[si]) * tensor_scale;
      }
      out[idx] = w;
    }
  }
}

double silu(double v) { return v / (1.0 + std::exp(-v)); }

// y[H] = down(silu(gate . x) * (up . x)) for one expert, fp64 ([Edge0]).
void expert_forward(const uint8_t* block, int fmt, int H, int I, int g,
                    const float* tscale3, const double* x, double* y) {
  Layout L;
  make_layout(fmt, H, I, g, &L);
  std::vector<double> G(static_cast<size_t>(I) * H), U(G.size()), D(G.size());
  double ts[3] = {1.0, 1.0, 1.0};
  if (fmt == FMT_NVFP4 && tscale3)
    for (int i = 0; i < 3; ++i) ts[i] = tscale3[i];
  dequant_matrix(fmt, block + L.off[0], block + L.off[3], I, H, g, ts[0], G.data());
  dequant_matrix(fmt, block + L.off[1], block + L.off[4], I, H, g, ts[1], U.data());
  dequant_matrix(fmt, block + L.off[2], block + L.off[5], H, I, g, ts[2], D.data());
  std::vector<double> h(I);
  for (int i = 0; i < I; ++i) {
    double gs = 0.0, us = 0.0;
    for (int c = 0; c < H; ++c) {
      gs += G[static_cast<size_t>(i) * H + c] * x[c];
      us += U[static_cast<size_t>(i) * H + c] * x[c];
    }
    h[i] = silu(gs) * us;
  }
  for (int r = 0; r < H; ++r) {
    double s = 0.0;
    for (int i = 0; i < I; ++i) s += D[static_cast<size_t>(r) * I + i] * h[i];
    y[r] = s;
  }
}

}  // namespace

extern "C" {

// ------------------------------------------------------------ formats API --
double orc_bf16_value(uint16_t b) { return bf16_value(b); }
double orc_fp16_value(uint16_t h) { return fp16_value(h); }
double orc_e2m1_value(int code) { return e2m1_value(code & 0xf); }
double orc_e4m3_value(int code) { return e4m3_value(code & 0xff); }

// Byte offsets of the six parts of one expert block and its total size.
// Returns 0 on success, -1 for an unsupported shape.
int orc_block_layout(int fmt, int H, int I, int g, uint64_t* off6, uint64_t* total) {
  Layout L;
  if (!make_layout(fmt, H, I, g, &L)) return -1;
  for (int i = 0; i < 6; ++i) off6[i] = L.off[i];
  *total = L.total;
  return 0;
}

// Dequantise part `which` (0 gate, 1 up, 2 down) of an expert block.
int orc_dequant(const uint8_t* block, int fmt, int H, int I, int g, int which,
                double tensor_scale, double* out) {
  Layout L;
  if (!make_layout(fmt, H, I, g, &L) || which < 0 || which > 2) return -1;
  int rows = (which == 2) ? H : I;
  int K = (which == 2) ? I : H;
  dequant_matrix(fmt, block + L.off[which], block + L.off[3 + which], rows, K,
                 fmt == FMT_INT4 ? g : 16, tensor_scale, out);
  return 0;
}

// ------------------------------------------------------------- q* split ----
// [FT-KR] pattern 2 and [FT-ZH] sec. 6.  phi = 65536*B_P/B_H in Q16; of m
// missed experts, f are fetched (B_P) and m - f are computed on the host
// path (B_H).  The two branches run side by side, so the step waits for the
// slower one, whose time is proportional to
//   cost(f) = max(f*(65536-phi), (m-f)*phi),
// and the split is the f in [0, m] that minimises it, the smallest such f
// when several tie.  Written here as that definition: every f is tried.
// When phi == 0 the pages apply no cap, and every miss may be fetched.
// Integer arithmetic in 64 bits.
int32_t orc_split_q16(int32_t m, int32_t phi) {
  if (m <= 0) return 0;
  if (phi <= 0) return m;
  const int64_t q = 65536, P = phi;
  int64_t best_f = 0, best_cost = -1;
  for (int64_t f = 0; f <= m; ++f) {
    const int64_t cost = std::max(f * (q - P), (static_cast<int64_t>(m) - f) * P);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_f = f;
    }
  }
  return static_cast<int32_t>(best_f);
}

// The rule over a grid: out[(phi - phi_lo) * (m_max + 1) + m] for every
// m in [0, m_max] and phi in [phi_lo, phi_hi].
void orc_split_q16_grid(int32_t m_max, int32_t phi_lo, int32_t phi_hi, int32_t* out) {
  for (int32_t phi = phi_lo; phi <= phi_hi; ++phi)
    for (int32_t m = 0; m <= m_max; ++m)
      out[static_cast<int64_t>(phi - phi_lo) * (m_max + 1) + m] = orc_split_q16(m, phi);
}

// ---------------------------------------------------------------- route ----
// logits = x . W^T in fp64 from bf16 x [T,H] and fp32 W [E,H]; p = softmax
// over all E experts; top-k by p descending, ties to the lower expert id;
// weights are p at those ids, divided by their sum when renorm != 0.
void orc_route(const uint16_t* x, int T, int H, const float* W, int E, int k,
               int renorm, int32_t* ids, double* wout, double* logits_out) {
  std::vector<double> xd(H), lg(E), p(E);
  std::vector<int> order(E);
  for (int t = 0; t < T; ++t) {
    for (int c = 0; c < H; ++c) xd[c] = bf16_value(x[static_cast<size_t>(t) * H + c]);
    for (int e = 0; e < E; ++e) {
      double s = 0.0;
      for (int c = 0; c < H; ++c) s += xd[c] * static_cast<double>(W[static_cast<size_t>(e) * H + c]);
      lg[e] = s;
      if (logits_out) logits_out[static_cast<size_t>(t) * E + e] = s;
    }
    double mx = lg[0];
    for (int e = 1; e < E; ++e) mx = std::max(mx, lg[e]);
    double z = 0.0;
    for (int e = 0; e < E; ++e) {
      p[e] = std::exp(lg[e] - mx);
      z += p[e];
    }
    for (int e = 0; e < E; ++e) p[e] /= z;
    for (int e = 0; e < E; ++e) order[e] = e;
    std::sort(order.begin(), order.end(), [&](int a, int b) {
      if (p[a] != p[b]) return p[a] > p[b];
      return a < b;
    });
    double sel = 0.0;
    for (int j = 0; j < k; ++j) sel += p[order[j]];
    for (int j = 0; j < k; ++j) {
      ids[static_cast<size_t>(t) * k + j] = order[j];
      wout[static_cast<size_t>(t) * k + j] = renorm ? p[order[j]] / sel : p[order[j]];
    }
  }
}

// -------------------------------------------------------------- resolve ----
// One call resolves the top-k ids of one layer against the global slot
// cache ([FT-KR] patterns 3 and 5, [FT-ZH] secs. 4 and 6).  Flat id
// fid = layer*E + expert.  State: slot_owner[S] (fid or -1), map[L*E] (slot or
// -1), usage[S] (last step the slot was used; -1 when empty), recency[L*E]
// (last step the expert was routed), step (one increment per call).
//   1. U = the distinct experts among ids, ascending.
//   2. hits = {e in U : map[fid] >= 0}; M = U \ hits; m = |M|.
//   3. evictable = S - |hits|; num_fetch = min(split(m, phi), evictable).
//   4. fetched = the first num_fetch of M ordered by (recency desc, id asc).
//   5. victims = the first num_fetch slots not owned by a hit, ordered by
//      (usage asc, slot asc); the i-th fetched expert goes to the i-th victim.
//   6. evict victims' owners, install the fetched experts; usage[slot] = step
//      for every hit and fetched slot; recency[fid] = step for all of U;
//      step += 1.
//   7. slot_ids[t,j] = map[fid(ids[t,j])]: a slot, or -1 for the host path.
// The fetch list holds (fid, slot) for i < num_fetch and -1 after that, up to
// max_list entries.  Returns 0, or -1 (state untouched) for an id outside
// [0, E) or a bad shape.
int orc_resolve(int L, int E, int S, int32_t* slot_owner, int32_t* map,
                int64_t* usage, int64_t* recency, int64_t* step, int layer,
                const int32_t* ids, int T, int k, int32_t phi, int32_t* slot_ids,
                int32_t* num_fetch_out, int32_t* fetch_fid, int32_t* fetch_slot,
                int max_list) {
  if (layer < 0 || layer >= L || E <= 0 || S < 0 || T < 0 || k < 0) return -1;
  if (phi < 0 || phi > 65536) return -1;
  const int n = T * k;
  for (int i = 0; i < n; ++i)
    if (ids[i] < 0 || ids[i] >= E) return -1;
  const int64_t base = static_cast<int64_t>(layer) * E;

  // 1. distinct experts, ascending
  std::vector<int> U(ids, ids + n);
  std::sort(U.begin(), U.end());
  U.erase(std::unique(U.begin(), U.end()), U.end());

  // 2. hits and misses
  std::vector<int> misses;
  std::vector<char> hit_slot(static_cast<size_t>(S), 0);
  int nhit = 0;
  for (int e : U) {
    int32_t s = map[base + e];
    if (s >= 0) {
      hit_slot[s] = 1;
      ++nhit;
    } else {
      misses.push_back(e);
    }
  }
  const int m = static_cast<int>(misses.size());

  // 3. how many to fetch
  int evictable = S - nhit;
  int nf = std::min(orc_split_q16(m, phi), evictable);
  if (nf < 0) nf = 0;

  // 4. which misses: recency descending, then id ascending
  std::vector<int> ranked = misses;
  std::sort(ranked.begin(), ranked.end(), [&](int a, int b) {
    int64_t ra = recency[base + a], rb = recency[base + b];
    if (ra != rb) return ra > rb;
    return a < b;
  });

  // 5. victims: usage ascending, then slot ascending, hit slots excluded
  std::vector<int> cand;
  for (int s = 0; s < S; ++s)
    if (!hit_slot[s]) cand.push_back(s);
  std::sort(cand.begin(), cand.end(), [&](int a, int b) {
    if (usage[a] != usage[b]) return usage[a] < usage[b];
    return a < b;
  });

  // 6. update state
  const int64_t now = *step;
  for (int e : U) {
    int32_t s = map[base + e];
    if (s >= 0) usage[s] = now;
  }
  for (int i = 0; i < nf; ++i) {
    int e = ranked[i];
    int v = cand[i];
    int32_t old = slot_owner[v];
    if (old >= 0) map[old] = -1;
    slot_owner[v] = static_cast<int32_t>(base + e);
    map[base + e] = v;
    usage[v] = now;
  }
  for (int e : U) recency[base + e] = now;
  *step = now + 1;

  // 7. rewrite ids
  for (int i = 0; i < n; ++i) slot_ids[i] = map[base + ids[i]];
  *num_fetch_out = nf;
  for (int i = 0; i < max_list; ++i) {
    fetch_fid[i] = (i < nf) ? static_cast<int32_t>(base + ranked[i]) : -1;
    fetch_slot[i] = (i < nf) ? cand[i] : -1;
  }
  return 0;
}

// n_steps consecutive resolve calls on one layer with one phi; step s reads
// ids + s*T*k and writes slot_ids + s*T*k, num_fetch[s], and max_list fetch
// entries at fetch_fid/fetch_slot + s*max_list.  Returns the first failing
// step's -1, else 0.
int orc_resolve_many(int L, int E, int S, int32_t* slot_owner, int32_t* map, int64_t* usage,
                     int64_t* recency, int64_t* step, int layer, const int32_t* ids, int T,
                     int k, int32_t phi, int n_steps, int32_t* slot_ids, int32_t* num_fetch,
                     int32_t* fetch_fid, int32_t* fetch_slot, int max_list) {
  const int64_t n = static_cast<int64_t>(T) * k;
  for (int s = 0; s < n_steps; ++s) {
    int rc = orc_resolve(L, E, S, slot_owner, map, usage, recency, step, layer, ids + s * n, T, k,
                         phi, slot_ids + s * n, num_fetch + s, fetch_fid + static_cast<int64_t>(s) * max_list,
                         fetch_slot + static_cast<int64_t>(s) * max_list, max_list);
    if (rc != 0) return rc;
  }
  return 0;
}

// ------------------------------------------------------------- prefetch ----
// [NVMe] "Where the time actually goes", speculative copies: layer l+1's router
// run on layer l's MoE input predicts layer l+1's experts, so most of its
// copies can start one layer early, while layer l still computes.  The pages
// give the idea, not the bookkeeping; the reading taken here is a fetch made
// ahead of its resolve, with the resolve's own choice rules:
//   1. U = the distinct predicted experts (pred_ids of `layer`), ascending.
//   2. hits = {e in U : map[fid] >= 0}; M = U \ hits; m = |M|.
//   3. A slot may not be a victim when a predicted hit owns it, or when it is
//      held (owner >= 0) with usage >= step - 1: the last resolve used it at
//      step - 1, so the current layer's experts may still be reading it, and
//      usage == step marks an earlier prefetch or install not yet consumed.
//   4. num = min(m, max_prefetch, eligible slots).
//   5. fetched = the first num of M by (recency desc, id asc); victims = the
//      first num eligible slots by (usage asc, slot asc); the i-th fetched
//      expert goes to the i-th victim.
//   6. Evict the victims' owners (map -1) and install: owner = fid, map =
//      slot, usage = step (the step the next resolve runs at).  Nothing is
//      routed, so recency, the usage of hit slots and the step stay as they
//      are.
// The fetch list has resolve's form: (fid, slot) for i < num, -1 after that,
// up to max_list entries.  Returns 0, or -1 (state untouched) for an id
// outside [0, E), a negative max_prefetch or a bad shape.
// Parity: pinned by a hand-worked trace, brute force over the fetched and
// victim sets on tiny states, and invariants (no busy or hit slot evicted,
// every prefetched expert resident, outputs unchanged).
int orc_prefetch(int L, int E, int S, int32_t* slot_owner, int32_t* map, int64_t* usage,
                 const int64_t* recency, const int64_t* step, int layer, const int32_t* pred_ids,
                 int T, int k, int32_t max_prefetch, int32_t* num_out, int32_t* fetch_fid,
                 int32_t* fetch_slot, int max_list) {
  if (layer < 0 || layer >= L || E <= 0 || S < 0 || T < 0 || k < 0 || max_prefetch < 0) return -1;
  const int n = T * k;
  for (int i = 0; i < n; ++i)
    if (pred_ids[i] < 0 || pred_ids[i] >= E) return -1;
  const int64_t base = static_cast<int64_t>(layer) * E;
  const int64_t now = *step;

  std::vector<int> U(pred_ids, pred_ids + n);
  std::sort(U.begin(), U.end());
  U.erase(std::unique(U.begin(), U.end()), U.end());

  std::vector<char> blocked(static_cast<size_t>(S), 0);
  std::vector<int> misses;
  for (int e : U) {
    const int32_t s = map[base + e];
    if (s >= 0)
      blocked[s] = 1;
    else
      misses.push_back(e);
  }
  for (int s = 0; s < S; ++s)
    if (slot_owner[s] >= 0 && usage[s] >= now - 1) blocked[s] = 1;

  std::vector<int> cand;
  for (int s = 0; s < S; ++s)
    if (!blocked[s]) cand.push_back(s);
  const int m = static_cast<int>(misses.size());
  const int nf = std::min(std::min(m, static_cast<int>(max_prefetch)), static_cast<int>(cand.size()));

  std::vector<int> ranked = misses;
  std::sort(ranked.begin(), ranked.end(), [&](int a, int b) {
    int64_t ra = recency[base + a], rb = recency[base + b];
    if (ra != rb) return ra > rb;
    return a < b;
  });
  std::sort(cand.begin(), cand.end(), [&](int a, int b) {
    if (usage[a] != usage[b]) return usage[a] < usage[b];
    return a < b;
  });

  for (int i = 0; i < nf; ++i) {
    const int e = ranked[i];
    const int v = cand[i];
    const int32_t old = slot_owner[v];
    if (old >= 0) map[old] = -1;
    slot_owner[v] = static_cast<int32_t>(base + e);
    map[base + e] = v;
    usage[v] = now;
  }
  *num_out = nf;
  for (int i = 0; i < max_list; ++i) {
    fetch_fid[i] = (i < nf) ? static_cast<int32_t>(base + ranked[i]) : -1;
    fetch_slot[i] = (i < nf) ? cand[i] : -1;
  }
  return 0;
}

// -------------------------------------------------------------- rebuild ----
// [FT-ZH] sec. 7 item 1 and [FT-KR] design pattern 7: the slot cache is rebuilt
// at a new size at a safe point, after its new geometry has been checked; the
// host pool stays the source of truth, so only performance depends on what
// the rebuilt cache holds.  The pages do not say which experts survive; the
// reading taken here keeps the most recently used ones, the order the cache
// already evicts in: every resident slot (owner >= 0) is ranked by usage,
// larger first, the lower slot first among equal usage; the first
// min(residents, S_new) of that ranking move, in order, to slots 0.., the
// other new slots are empty, every other flat id maps to -1, and recency and
// the step carry over unchanged.  src_of_new[d] is the old slot moved to new
// slot d, or -1.  Returns -1 on an owner outside [0, L*E), else 0.
// Parity: pinned by invariants and by brute force on small states.
int orc_cache_rebuild(int L, int E, int S_old, const int32_t* owner_old, const int64_t* usage_old,
                      int S_new, int32_t* owner_new, int32_t* map_new, int64_t* usage_new,
                      int32_t* src_of_new) {
  const int64_t n_fid = static_cast<int64_t>(L) * E;
  std::vector<int> resident;
  for (int s = 0; s < S_old; ++s) {
    if (owner_old[s] < 0) continue;
    if (owner_old[s] >= n_fid) return -1;
    resident.push_back(s);
  }
  std::stable_sort(resident.begin(), resident.end(), [&](int a, int b) {
    if (usage_old[a] != usage_old[b]) return usage_old[a] > usage_old[b];
    return a < b;
  });
  for (int64_t f = 0; f < n_fid; ++f) map_new[f] = -1;
  for (int d = 0; d < S_new; ++d) {
    owner_new[d] = -1;
    usage_new[d] = -1;
    src_of_new[d] = -1;
  }
  const int keep = std::min(static_cast<int>(resident.size()), S_new);
  for (int d = 0; d < keep; ++d) {
    const int s = resident[d];
    owner_new[d] = owner_old[s];
    usage_new[d] = usage_old[s];
    map_new[owner_old[s]] = d;
    src_of_new[d] = s;
  }
  return 0;
}

// -------------------------------------------------------------- install ----
// [FT-KR] design pattern 1 and [FT-ZH] sec. 5: prefill holds a whole layer's
// experts on the GPU in one half of a two-layer buffer made of the cache's
// first 2E slots (layer l in slots (l%2)*E ..), which then seeds decode.  The
// pages do not spell out the bookkeeping; the reading taken here installs
// expert e of `layer` (flat id layer*E+e) in slot slot0+e, one expert after
// the other in e order: a copy of that flat id held in any other slot is
// dropped (slot emptied, usage -1), the slot's previous owner (another flat
// id) is evicted (its map entry -1), and the slot takes the flat id with
// usage = the current step.  Recency and the step do not change (no routing
// happened).  Returns -1 when layer or the slot range is out of bounds.
// Parity: pinned by a hand-worked example and by invariants.
int orc_cache_install(int L, int E, int S, int32_t* slot_owner, int32_t* map, int64_t* usage,
                      const int64_t* step, int layer, int slot0) {
  if (layer < 0 || layer >= L || slot0 < 0 || static_cast<int64_t>(slot0) + E > S) return -1;
  for (int e = 0; e < E; ++e) {
    const int32_t fid = layer * E + e;
    const int s = slot0 + e;
    const int32_t was = map[fid];
    if (was >= 0 && was != s) {
      slot_owner[was] = -1;
      usage[was] = -1;
      map[fid] = -1;
    }
    const int32_t old = slot_owner[s];
    if (old >= 0 && old != fid) map[old] = -1;
    slot_owner[s] = fid;
    map[fid] = s;
    usage[s] = step[0];
  }
  return 0;
}

// -------------------------------------------------------------- permute ----
// Stable sort of the T*k (token, rank) pairs by expert: expert ascending, then
// token, then rank.  perm[pos] = pair index t*k+j, inv[t*k+j] = pos,
// offsets[e] = first position of expert e, offsets[E] = T*k.
int orc_permute(const int32_t* ids, int T, int k, int E, int32_t* perm,
                int32_t* inv, int32_t* offsets) {
  const int n = T * k;
  for (int i = 0; i < n; ++i)
    if (ids[i] < 0 || ids[i] >= E) return -1;
  std::vector<int> order(n);
  for (int i = 0; i < n; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(),
                   [&](int a, int b) { return ids[a] < ids[b]; });
  for (int pos = 0; pos < n; ++pos) {
    perm[pos] = order[pos];
    inv[order[pos]] = pos;
  }
  for (int e = 0; e <= E; ++e) offsets[e] = 0;
  for (int i = 0; i < n; ++i) offsets[ids[i] + 1] += 1;
  for (int e = 0; e < E; ++e) offsets[e + 1] += offsets[e];
  return 0;
}

// -------------------------------------------------------------- experts ----
// One expert on one fp64 input vector: y = down(silu(gate.x) * up.x).
int orc_expert(const uint8_t* block, int fmt, int H, int I, int g,
               const float* tscale3, const double* x, double* y) {
  Layout L;
  if (!make_layout(fmt, H, I, g, &L)) return -1;
  expert_forward(block, fmt, H, I, g, tscale3, x, y);
  return 0;
}

// The same expert on n input vectors (rows of x, fp64): y[r] = expert(x[r]).
// One dequantisation serves all rows; the per-row arithmetic is expert_forward's.
int orc_expert_batch(const uint8_t* block, int fmt, int H, int I, int g, const float* tscale3,
                     const double* x, int n, double* y) {
  Layout L;
  if (!make_layout(fmt, H, I, g, &L)) return -1;
  std::vector<double> G(static_cast<size_t>(I) * H), U(G.size()), D(G.size());
  double ts[3] = {1.0, 1.0, 1.0};
  if (fmt == FMT_NVFP4 && tscale3)
    for (int i = 0; i < 3; ++i) ts[i] = tscale3[i];
  dequant_matrix(fmt, block + L.off[0], block + L.off[3], I, H, g, ts[0], G.data());
  dequant_matrix(fmt, block + L.off[1], block + L.off[4], I, H, g, ts[1], U.data());
  dequant_matrix(fmt, block + L.off[2], block + L.off[5], H, I, g, ts[2], D.data());
  std::vector<double> h(I);
  for (int r = 0; r < n; ++r) {
    const double* xr = x + static_cast<size_t>(r) * H;
    for (int i = 0; i < I; ++i) {
      double gs = 0.0, us = 0.0;
      for (int c = 0; c < H; ++c) {
        gs += G[static_cast<size_t>(i) * H + c] * xr[c];
        us += U[static_cast<size_t>(i) * H + c] * xr[c];
      }
      h[i] = silu(gs) * us;
    }
    double* yr = y + static_cast<size_t>(r) * H;
    for (int c = 0; c < H; ++c) {
      double acc = 0.0;
      for (int i = 0; i < I; ++i) acc += D[static_cast<size_t>(c) * I + i] * h[i];
      yr[c] = acc;
    }
  }
  return 0;
}

// The routed layer output over a pool bank (the source of truth): for every
// pair (t, j) with include[t*k+j] != 0 (all pairs when include is NULL),
//   out[t] += w[t,j] * expert(layer*E + ids[t,j]) (x[t]),
// summed in j order.  The pool holds one block per flat id at
// pool + fid*stride; tscales holds [L*E, 3] fp32 per-tensor scales (NVFP4).
// Residency never enters: the result is the same for any cache state.
int orc_moe_experts(const uint8_t* pool, uint64_t stride, const float* tscales,
                    int fmt, int H, int I, int g, int layer, int E,
                    const uint16_t* x, int T, const int32_t* ids,
                    const float* w, int k, const uint8_t* include, double* out) {
  Layout L;
  if (!make_layout(fmt, H, I, g, &L) || stride < L.total) return -1;
  std::vector<double> xd(H), y(H);
  for (int t = 0; t < T; ++t) {
    for (int c = 0; c < H; ++c) xd[c] = bf16_value(x[static_cast<size_t>(t) * H + c]);
    double* o = out + static_cast<size_t>(t) * H;
    for (int c = 0; c < H; ++c) o[c] = 0.0;
    for (int j = 0; j < k; ++j) {
      size_t p = static_cast<size_t>(t) * k + j;
      if (include && !include[p]) continue;
      int e = ids[p];
      if (e < 0 || e >= E) return -1;
      int64_t fid = static_cast<int64_t>(layer) * E + e;
      const float* ts = tscales ? tscales + 3 * fid : nullptr;
      expert_forward(pool + static_cast<uint64_t>(fid) * stride, fmt, H, I, g, ts,
                     xd.data(), y.data());
      for (int c = 0; c < H; ++c) o[c] += static_cast<double>(w[p]) * y[c];
    }
  }
  return 0;
}

// The per-row expert outputs of a token-permuted batch (the grouped form):
// yp[pos] = expert(layer*E + e)(x[perm[pos] / k]) for the expert e whose
// segment [offsets[e], offsets[e+1]) holds pos.  Only rows listed in `rows`
// (n_rows of them) are computed, so a sample of a large batch stays cheap.
int orc_grouped_rows(const uint8_t* pool, uint64_t stride, const float* tscales,
                     int fmt, int H, int I, int g, int layer, int E,
                     const uint16_t* x, const int32_t* perm, int k,
                     const int32_t* offsets, const int32_t* rows, int n_rows,
                     double* yp_rows) {
  Layout L;
  if (!make_layout(fmt, H, I, g, &L) || stride < L.total) return -1;
  std::vector<double> xd(H);
  for (int r = 0; r < n_rows; ++r) {
    int pos = rows[r];
    int e = 0;
    while (e < E && !(offsets[e] <= pos && pos < offsets[e + 1])) ++e;
    if (e == E) return -1;
    int t = perm[pos] / k;
    for (int c = 0; c < H; ++c) xd[c] = bf16_value(x[static_cast<size_t>(t) * H + c]);
    int64_t fid = static_cast<int64_t>(layer) * E + e;
    const float* ts = tscales ? tscales + 3 * fid : nullptr;
    expert_forward(pool + static_cast<uint64_t>(fid) * stride, fmt, H, I, g, ts, xd.data(),
                   yp_rows + static_cast<size_t>(r) * H);
  }
  return 0;
}

// --------------------------------------------------------------- combine ---
// out[t] = sum_j w[t,j] * yp[inv[t,j]] in j order (plus host_partial[t] when
// given), fp64.  yp rows are bf16 (the grouped-GEMM output format).
void orc_combine(const uint16_t* yp, const int32_t* inv, const float* w, int T,
                 int k, int H, const float* host_partial, double* out) {
  for (int t = 0; t < T; ++t) {
    double* o = out + static_cast<size_t>(t) * H;
    for (int c = 0; c < H; ++c)
      o[c] = host_partial ? static_cast<double>(host_partial[static_cast<size_t>(t) * H + c]) : 0.0;
    for (int j = 0; j < k; ++j) {
      size_t p = static_cast<size_t>(t) * k + j;
      const uint16_t* row = yp + static_cast<size_t>(inv[p]) * H;
      for (int c = 0; c < H; ++c) o[c] += static_cast<double>(w[p]) * bf16_value(row[c]);
    }
  }
}

}  // extern "C"
