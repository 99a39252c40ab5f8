// prefill.cu -- token-permuted grouped SwiGLU expert GEMM on tcgen05/TMEM.
//
// Sources: "NVMe에서 전문가(experts)를 ... 133GB MoE" (molayo1419.me), engine
// step 5 (the whole prompt goes through a layer's experts at once, so every
// expert's weights are read once per layer); "FreeToken: 让消费级电脑跑起 284B
// MoE" (fengjutian.github.io), sec. 3 (prefill touches nearly every expert
// and is dense compute).
//
// Two launches, each over the work items (128-row weight tile, expert), one
// persistent CTA per SM walking items blockIdx.x, + gridDim.x, ...:
//   gate/up:  Hp[m, i] = f16(2^-4 * silu(g) * u), g = gate[i].x_m, u = up[i].x_m
//   down:     Yp[m, j] = bf16(down[j].h_m)
// for the rows m of the expert's segment of the permuted batch.  The MMA is
// "swap-AB": the weight tile is the M = 128 side, the expert's tokens the N
// side (N <= 256 per pass; longer segments take more passes), so a tile of
// weights is dequantised once for all its tokens.
//
// Operands are f16 (tcgen05.mma kind::f16, fp32 accumulators in TMEM):
//   A: E2M1 codes through the hardware e2m1x2 -> f16x2 convert, times the
//      E4M3 block scale (f16 multiply; exact, the product has <= 6
//      significant bits); the fp32 per-tensor scale is applied in the
//      epilogue.
//   B: the permuted activations in f16 with an exact power-of-two prescale
//      per row (x_scale undoes it), and for down the f16 h written by the
//      gate/up epilogue with a fixed 2^-4 prescale.
//
// Stages.  With few tokens per expert (a launch whose mean segment is at
// most 96 rows: MRG) each stage of the A ring also holds that k-step's token
// tile, which the TMA completes on the same barrier the converters arrive
// on, so an MMA issuer waits and commits once per k-step instead of twice.
// On GB300 an mbarrier poll costs the issuing thread ~200-340 cycles even
// when the phase has completed, against ~130-190 per MMA: at N ~ 48 the
// issuer's loop, not the tensor pipe, sets the pace.  Longer segments keep a
// separate, deeper token ring, which hides the ~1 us that their larger token
// tiles take to arrive from L2.
//
// Roles (640 threads).  Warp 0 lane 0 streams the weights by TMA: E2M1 codes
// in 64-byte-wide boxes (two k-steps, 64-byte swizzle) and E4M3 scales (four
// k-steps per stage).  Warp 2 lane 0 streams the B tiles (tokens), with as
// many stages as the expert's token count leaves room for, so that neither
// stream waits on the other.  Warps 1 and 3 (lane 0) issue the MMAs: an
// issuing thread spends ~126 cycles per tcgen05.mma on fresh operands at any
// N <= 128 (GB300), so two issuers share the work (gate / up; for down, even
// / odd k-steps into two accumulators).  Warps 4..19, two groups of eight, dequantise into the
// 128-byte-swizzled K-major A tiles (gate / up, or even / odd k-steps), half
// a weight row per thread per k-step, and afterwards run the epilogue
// (tcgen05.ld; the four warps of a TMEM lane quarter take every fourth
// 16-token chunk).  Stages are handed over with mbarriers; every wait is
// bounded.
#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "ft_async.cuh"
#include "ft_common.cuh"

namespace ft {
namespace {

constexpr int kBM = 128;        // weight rows per tile (MMA M)
constexpr int kBK = 64;         // K per k-step: one 128-byte row of f16 (four MMAs of K = 16)
constexpr int kRawSteps = 2;    // k-steps per code stage: 64 code bytes per row
constexpr int kScSteps = 4;     // k-steps per scale stage: 16 scale bytes per row
constexpr int kSuper = kScSteps * kBK;  // K must be a multiple of this
constexpr int kNMax = 256;      // tokens per pass (MMA N)
constexpr int kBRows = 64;      // rows per B TMA box
constexpr int kBBytes = 64 * 1024;     // the B (tokens) ring for <= 128 tokens: 4 .. 8 stages
constexpr int kBBytesBig = 96 * 1024;  // ... for more: 3 stages of 256 rows, 4 of 192
constexpr int kBMaxStages = 8;
constexpr int kMrgMeanRows = 96;  // launches with T k <= 96 E put token tiles in the A stages
constexpr int kConvWarps = 16;  // four per SM sub-partition, in two groups of eight
constexpr int kPfThreads = 128 + 32 * kConvWarps;  // + TMA x2, MMA issuer x2
constexpr float kHScale = 0.0625f;  // h is stored as f16(h * 2^-4)

constexpr int kATile = kBM * kBK * 2;                 // 16 KB per matrix per k-step
constexpr int kBBox = kBRows * kBK * 2;               // 8 KB per 64-row B box
constexpr int kRawTile = kBM * kRawSteps * kBK / 2;   // 8 KB per matrix per code stage
constexpr int kScTile = kBM * kScSteps * kBK / 16;    // 2 KB per matrix per scale stage

// Shared memory per CTA (216 KB gate/up, 212 KB down).  Weight codes arrive in
// 64-byte-wide boxes: one TMA row request per 32 B reached about 4.3 TB/s on
// GB300, 64 B about 6.9 TB/s.  The dequantised A ring is three (gate/up) or
// six (down) k-steps deep so that the MMAs of earlier k-steps and the
// conversion of later ones overlap; for experts with more than 128 tokens a
// B stage is larger and arrives from L2 with a microsecond of latency, so one
// A stage (two for down) goes to the B ring instead.  Offsets are computed at
// run time from the layout chosen.
template <int NMAT>
struct PfSmem {
  static constexpr int kAStages = NMAT == 2 ? 3 : 6;
  static constexpr int kAStagesBig = NMAT == 2 ? 2 : 4;
  static constexpr int kRawStages = NMAT == 2 ? 3 : 6;
  static constexpr int kScStages = 2;
  static constexpr int raw_stage = NMAT * kRawTile;
  static constexpr int sc_stage = NMAT * kScTile;
  static constexpr int tail = kRawStages * raw_stage + kScStages * sc_stage;  // raw + scale rings
  static constexpr int total = kAStages * NMAT * kATile + kBBytes + tail;
  static constexpr int kABBudget = total - tail;  // A and token rings
  static constexpr int kAStagesMrg = NMAT == 2 ? 4 : 6;  // A + token stages, at most
  static constexpr int kAStagesMax = kAStagesMrg > kAStages ? kAStagesMrg : kAStages;
  static_assert(kAStagesBig * NMAT * kATile + kBBytesBig + tail <= total, "big-N layout must fit");
};

struct PfArgs {
  const int32_t* offsets;  // [E+1]
  const int32_t* slot_of;  // [E] cache slot of each expert
  int E, K, M, n_rows, layer;
  int tiles;               // 128-row weight tiles per expert (M / 128); work items = tiles * E
  int pmax;                // tokens per pass: 128 (MRG launches) or 256
  int64_t n_blocks;
  const float* x_scale;    // [n_rows] (gate/up only)
  const float* tscale;     // [n_fids, 3]
  uint16_t* out;           // gate/up: Hp f16 [n_rows, M]; down: Yp bf16 [n_rows, M]
  int32_t* dev_status;
};

// Work item it = (expert e, row tile mt): its segment of the permuted batch
// and its cache slot; run is false for an empty segment or an invalid entry
// (recorded once, by the caller that passes report).
struct PfItem {
  int e, mt, row_lo, n_e, slot;
  bool run;
};

__device__ __forceinline__ PfItem pf_item(const PfArgs& a, int it, bool report) {
  PfItem I;
  I.e = it / a.tiles;
  I.mt = it - I.e * a.tiles;
  I.row_lo = a.offsets[I.e];
  I.n_e = a.offsets[I.e + 1] - I.row_lo;
  I.slot = a.slot_of[I.e];
  I.run = I.n_e > 0;
  if (I.run && (I.slot < 0 || I.slot >= a.n_blocks || I.row_lo < 0 || I.row_lo + I.n_e > a.n_rows)) {
    if (report) record_status(a.dev_status, I.slot < 0 ? FT_ERR_UNSUPPORTED : FT_ERR_BAD_ID);
    I.run = false;
  }
  return I;
}

// ----------------------------------------------------------- PTX helpers ---
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// K-major operand in the 128-byte swizzle layout: rows of 128 B, 8-row groups
// 1024 B apart (stride byte offset), version bits 46-47 = 1, layout 2 =
// SWIZZLE_128B.  The tile base is 1024-byte aligned.
__device__ __forceinline__ uint64_t sw128_desc(const void* tile) {
  const uint64_t addr = smem_u32(tile);
  uint64_t d = (addr >> 4) & 0x3FFFull;
  d |= 1ull << 16;                       // leading byte offset (unused for this layout)
  d |= (1024ull >> 4) << 32;             // stride byte offset
  d |= 1ull << 46;                       // descriptor version
  d |= 2ull << 61;                       // SWIZZLE_128B
  return d;
}

// kind::f16 instruction descriptor: fp32 accumulate, f16 A and B, both
// K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t idesc_f16(int n) {
  return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(kBM >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

#define FT_R8(b) "=r"(r[b]), "=r"(r[b + 1]), "=r"(r[b + 2]), "=r"(r[b + 3]), "=r"(r[b + 4]), "=r"(r[b + 5]), "=r"(r[b + 6]), "=r"(r[b + 7])

// 2 x 16 consecutive fp32 TMEM columns of this warp's 32 lanes, both loads in
// flight before one wait.
__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, uint32_t tb, float va[16], float vb[16]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15}, [%32];\n"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%33];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : FT_R8(0), FT_R8(8), FT_R8(16), FT_R8(24)
      : "r"(ta), "r"(tb)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    va[i] = __uint_as_float(r[i]);
    vb[i] = __uint_as_float(r[16 + i]);
  }
}
#undef FT_R8

// E2M1 codes of one 32-bit word (8 codes) times a broadcast f16x2 scale.
__device__ __forceinline__ uint4 dequant8(uint32_t w, uint32_t s2) {
  uint32_t h[4];
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
  uint4 o;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o.x) : "r"(h[0]), "r"(s2));
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o.y) : "r"(h[1]), "r"(s2));
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o.z) : "r"(h[2]), "r"(s2));
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o.w) : "r"(h[3]), "r"(s2));
  return o;
}

// Two E4M3 scale bytes -> {s0, s0} and {s1, s1} as f16x2.
__device__ __forceinline__ void scales2(unsigned short two, uint32_t s2[2]) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(two));
  s2[0] = __byte_perm(h, 0, 0x1010);
  s2[1] = __byte_perm(h, 0, 0x3232);
}

// ---------------------------------------------------------------- kernel ---
// NMAT = 2: gate/up (maps c0,c1 = codes, s0,s1 = scales); NMAT = 1: down.
// MRG: token tiles inside the A stages (see "Stages" above).
template <int NMAT, bool MRG>
__global__ void __launch_bounds__(kPfThreads, 1) pf_kernel(const __grid_constant__ CUtensorMap c0map,
                                                           const __grid_constant__ CUtensorMap c1map,
                                                           const __grid_constant__ CUtensorMap s0map,
                                                           const __grid_constant__ CUtensorMap s1map,
                                                           const __grid_constant__ CUtensorMap bmap,
                                                           PfArgs a) {
  using L = PfSmem<NMAT>;
  constexpr int RS = L::kRawStages, SS = L::kScStages, AS_MAX = L::kAStagesMax;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t raw_full[RS], raw_empty[RS];
  __shared__ __align__(8) uint64_t sc_full[SS], sc_empty[SS];
  __shared__ __align__(8) uint64_t a_full[AS_MAX], a_empty[AS_MAX];
  __shared__ __align__(8) uint64_t b_full[kBMaxStages], b_empty[kBMaxStages];
  __shared__ __align__(8) uint64_t acc_full, acc_empty;
  __shared__ uint32_t s_tmem;

  if (prior_timeout(a.dev_status)) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ksteps = a.K / kBK;
  const int n_items = a.tiles * a.E;
  const int pmax = a.pmax;  // tokens per pass (MMA N <= pmax)
  constexpr uint32_t kCols = 512;  // two accumulators of up to 256 columns
  constexpr int kIss = NMAT == 2 ? 2 : 1;  // MMA issuers that read each k-step's A and B
  // The ring geometry is fixed for the launch (the rings run on from one
  // work item to the next): token stages of pmax / 64 boxes; more than two
  // boxes take the big-N layout.  MRG: a stage is the A tiles then the token
  // tile; otherwise the A ring and the token ring (NB stages) are separate.
  const int nbox_max = pmax / kBRows;
  const int b_stage = nbox_max * kBBox;
  const bool big = nbox_max > 2;
  const int a_stage = NMAT * kATile + (MRG ? b_stage : 0);
  const int AS = MRG ? min(L::kAStagesMrg, L::kABBudget / a_stage) : big ? L::kAStagesBig : L::kAStages;
  const int b_bytes = big ? kBBytesBig : kBBytes;
  const int NB = MRG ? AS : min(kBMaxStages, b_bytes / b_stage);
  uint8_t* const a_base = smem;
  uint8_t* const b_base = MRG ? a_base + NMAT * kATile : a_base + AS * NMAT * kATile;
  const int b_pitch = MRG ? a_stage : b_stage;  // bytes from one token stage to the next
  uint8_t* const raw_base = a_base + L::kABBudget;
  uint8_t* const sc_base = raw_base + RS * L::raw_stage;

  if (tid == 0) {
    for (int s = 0; s < RS; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], kConvWarps);
    }
    for (int s = 0; s < SS; ++s) {
      mbar_init(&sc_full[s], 1);
      mbar_init(&sc_empty[s], kConvWarps);
    }
    for (int s = 0; s < AS; ++s) {
      // the converter warps of a k-step (and with MRG the token producer)
      mbar_init(&a_full[s], (NMAT == 2 ? kConvWarps : kConvWarps / 2) + (MRG ? 1 : 0));
      mbar_init(&a_empty[s], kIss);
    }
    if (!MRG)
      for (int s = 0; s < NB; ++s) {
        mbar_init(&b_full[s], 1);
        mbar_init(&b_empty[s], kIss);
      }
    mbar_init(&acc_full, 2);
    mbar_init(&acc_empty, kConvWarps);
    fence_barrier_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  // Every role walks the same work items (row tile, expert) in the same
  // order, it = blockIdx.x, + gridDim.x, ...; the ring positions and the
  // accumulator's pass count carry over from one item to the next.
  if (warp == 0) {
    // -------------------------------------------------- TMA: weights ---
    if (lane == 0) {
      const CUtensorMap* cm[2] = {&c0map, &c1map};
      const CUtensorMap* sm[2] = {&s0map, &s1map};
      int su = 0, v = 0;  // scale and code stages issued so far
      for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const PfItem I = pf_item(a, it, tid == 0);
        if (!I.run) continue;
        const int n_pass = (I.n_e + pmax - 1) / pmax;
        for (int pass = 0; pass < n_pass; ++pass) {
          for (int kk = 0; kk < ksteps; kk += kRawSteps) {
            if (kk % kScSteps == 0) {
              const int sst = su % SS;
              if (su >= SS && !mbar_wait(&sc_empty[sst], ((su / SS) - 1) & 1, a.dev_status)) goto done_w;
              uint8_t* sc = sc_base + sst * L::sc_stage;
              mbar_arrive_expect_tx(&sc_full[sst], NMAT * kScTile);
              for (int m = 0; m < NMAT; ++m)
                tma_load_3d(sc + m * kScTile, sm[m], (kk / kScSteps) * 16, I.mt * kBM, I.slot, &sc_full[sst]);
              ++su;
            }
            const int rst = v % RS;
            if (v >= RS && !mbar_wait(&raw_empty[rst], ((v / RS) - 1) & 1, a.dev_status)) goto done_w;
            uint8_t* raw = raw_base + rst * L::raw_stage;
            mbar_arrive_expect_tx(&raw_full[rst], NMAT * kRawTile);
            for (int m = 0; m < NMAT; ++m)
              tma_load_3d(raw + m * kRawTile, cm[m], (kk / kRawSteps) * 64, I.mt * kBM, I.slot, &raw_full[rst]);
            ++v;
          }
        }
      }
    done_w:;
    }
  } else if (warp == 2) {
    // --------------------------------------------------- TMA: tokens ---
    if (lane == 0) {
      // ring position kept incrementally: NB is not a compile-time constant
      int bst = 0;
      uint32_t bph = 0;
      bool wrapped = false;
      for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const PfItem I = pf_item(a, it, false);
        if (!I.run) continue;
        const int n_pass = (I.n_e + pmax - 1) / pmax;
        for (int pass = 0; pass < n_pass; ++pass) {
          const int n_valid = min(pmax, I.n_e - pass * pmax);
          const int nbox = (n_valid + kBRows - 1) / kBRows;
          for (int kk = 0; kk < ksteps; ++kk) {
            // MRG: the stage's release is the A stage's, its arrival counts on a_full
            uint64_t* const bfull = MRG ? &a_full[bst] : &b_full[bst];
            if (wrapped && !mbar_wait(MRG ? &a_empty[bst] : &b_empty[bst], bph ^ 1u, a.dev_status)) goto done_b;
            uint8_t* bt = b_base + bst * b_pitch;
            mbar_arrive_expect_tx(bfull, nbox * kBBox);
            for (int bx = 0; bx < nbox; ++bx)
              tma_load_2d(bt + bx * kBBox, &bmap, kk * kBK, I.row_lo + pass * pmax + bx * kBRows, bfull);
            if (++bst == NB) {
              bst = 0;
              bph ^= 1u;
              wrapped = true;
            }
          }
        }
      }
    done_b:;
    }
  } else if (warp == 1 || warp == 3) {
    // ------------------------------------------------------------- MMA ---
    // Two issuing threads: an issuing thread spends ~126 cycles per
    // tcgen05.mma on fresh operands, whatever N is, so two issuers share the
    // work.  gate/up: issuer i owns matrix i.  down: issuer i owns the
    // k-steps kk % 2 == i, into accumulator i (summed in the epilogue).
    const int iss = warp == 1 ? 0 : 1;
    if (lane == 0) {
      bool ok = true;
      int ast = 0, bst = 0, gp = 0;  // gp: passes issued so far (the accumulator's phase)
      uint32_t aph = 0, bph = 0;
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const PfItem I = pf_item(a, it, false);
        if (!I.run) continue;
        const int n_pass = (I.n_e + pmax - 1) / pmax;
        for (int pass = 0; pass < n_pass && ok; ++pass, ++gp) {
          const int n_valid = min(pmax, I.n_e - pass * pmax);
          const int n_mma = (n_valid + 15) & ~15;
          const uint32_t idesc = idesc_f16(n_mma);
          if (gp > 0) {
            if (!mbar_wait(&acc_empty, (gp - 1) & 1, a.dev_status)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          for (int kk = 0; kk < ksteps; ++kk) {
            if (NMAT == 2 || (kk & 1) == iss) {
              if (!mbar_wait(&a_full[ast], aph, a.dev_status) ||
                  (!MRG && !mbar_wait(&b_full[bst], bph, a.dev_status))) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint8_t* at = a_base + ast * a_stage + (NMAT == 2 ? iss * kATile : 0);
              const uint64_t adesc = sw128_desc(at);
              const uint64_t bdesc = sw128_desc(b_base + bst * b_pitch);
              const uint32_t first = NMAT == 2 ? (kk == 0) : (kk == iss);
#pragma unroll
              for (int j = 0; j < kBK / 16; ++j)
                mma_f16(tmem + iss * 256, adesc + 2 * j, bdesc + 2 * j, idesc, (first && j == 0) ? 0u : 1u);
              mma_commit(&a_empty[ast]);
              if (!MRG) mma_commit(&b_empty[bst]);
            }
            if (++ast == AS) {
              ast = 0;
              aph ^= 1u;
            }
            if (++bst == NB) {
              bst = 0;
              bph ^= 1u;
            }
          }
          if (ok) mma_commit(&acc_full);
        }
      }
    }
  } else {
    // --------------------------------------- convert, then the epilogue ---
    // Two groups of eight warps.  gate/up: group g converts matrix g of every
    // k-step; down: group g converts the k-steps kk % 2 == g (the ones MMA
    // issuer g consumes).  In a group, thread (r, hf) converts K half hf of
    // weight row r: lanes 0-7 and 16-23 take half 0, lanes 8-15 and 24-31
    // half 1, so the eight lanes of each shared-memory phase touch eight
    // consecutive rows and, with the 64-byte swizzle of the code tiles and
    // the 128-byte swizzle of the A tiles, distinct banks.  Each stage's codes
    // and scales go to registers at once and the stage is released.  The
    // release is preceded by a proxy fence: the loads are generic-proxy reads
    // and the TMA that refills the stage writes through the async proxy, and
    // the mbarrier hand-off alone does not order the two.  Without the fence
    // a load still outstanding at the arrive could return the next stage's
    // bytes (seen on GB300 as a few weight rows of a tile differing from one
    // run to the next, at 192-token segments).
    const int cwarp = warp - 4;
    const int grp = cwarp >> 3, wc = cwarp & 7;
    const int m = NMAT == 2 ? grp : 0;  // matrix this group converts
    const int r = wc * 16 + (lane & 7) + ((lane >> 4) << 3), hf = (lane >> 3) & 1;
    bool ok = true;
    int ast = 0, u = 0, su = 0, v = 0, gp = 0;
    uint32_t aph = 0;
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      const PfItem I = pf_item(a, it, false);
      if (!I.run) continue;
      const int n_pass = (I.n_e + pmax - 1) / pmax;
      for (int pass = 0; pass < n_pass && ok; ++pass, ++gp) {
        for (int k4 = 0; k4 < ksteps; k4 += kScSteps) {
          const int sst = su % SS;
          if (!mbar_wait(&sc_full[sst], (su / SS) & 1, a.dev_status)) {
            ok = false;
            break;
          }
          ++su;
          const uint4 sc = *reinterpret_cast<const uint4*>(sc_base + sst * L::sc_stage + m * kScTile + r * 16);
          fence_proxy_async_smem();  // the scale words are read before the TMA may refill the stage
          __syncwarp();
          if (lane == 0) mbar_arrive(&sc_empty[sst]);
#pragma unroll
          for (int h2 = 0; h2 < kScSteps / kRawSteps; ++h2) {
            const int rst = v % RS;
            if (!mbar_wait(&raw_full[rst], (v / RS) & 1, a.dev_status)) {
              ok = false;
              break;
            }
            ++v;
            uint4 cw[kRawSteps];
            const uint8_t* raw = raw_base + rst * L::raw_stage + m * kRawTile + r * 64;
#pragma unroll
            for (int jj = 0; jj < kRawSteps; ++jj)
              if (NMAT == 2 || jj == grp)
                cw[jj] = *reinterpret_cast<const uint4*>(raw + (((2 * jj + hf) ^ ((r >> 1) & 3)) << 4));
            fence_proxy_async_smem();  // likewise the code words
            __syncwarp();
            if (lane == 0) mbar_arrive(&raw_empty[rst]);
#pragma unroll
            for (int jj = 0; jj < kRawSteps; ++jj) {
              // k4 and 2 * h2 are even, so this k-step's parity is jj's
              if (NMAT == 2 || jj == grp) {
                const int j4 = h2 * kRawSteps + jj;  // k-step within the scale stage
                if (u >= AS && !mbar_wait(&a_empty[ast], aph ^ 1u, a.dev_status)) {
                  ok = false;
                  break;
                }
                uint8_t* at = a_base + ast * a_stage + m * kATile + r * 128;
                const uint32_t sw = j4 == 0 ? sc.x : j4 == 1 ? sc.y : j4 == 2 ? sc.z : sc.w;
                uint32_t s2[2];
                scales2(static_cast<unsigned short>(hf ? sw >> 16 : sw & 0xffffu), s2);
                const uint32_t words[4] = {cw[jj].x, cw[jj].y, cw[jj].z, cw[jj].w};
#pragma unroll
                for (int w = 0; w < 4; ++w)
                  *reinterpret_cast<uint4*>(at + (((4 * hf + w) ^ (r & 7)) << 4)) = dequant8(words[w], s2[w >> 1]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[ast]);
              }
              ++u;
              if (++ast == AS) {
                ast = 0;
                aph ^= 1u;
              }
            }
            if (!ok) break;
          }
          if (!ok) break;
        }
        if (!ok) break;
        // epilogue of this pass: warp w reads TMEM lanes 32 (w % 4) .. + 31; the
        // four warps of a lane quarter take every fourth 16-token chunk
        if (!mbar_wait_warp(&acc_full, gp & 1, a.dev_status)) {  // one verdict: tcgen05.ld follows
          ok = false;
          break;
        }
        tc_fence_after();
        float ts[2];
        {
          const int64_t fid = static_cast<int64_t>(a.layer) * a.E + I.e;
          ts[0] = __ldg(a.tscale + 3 * fid + (NMAT == 2 ? 0 : 2));
          ts[1] = NMAT == 2 ? __ldg(a.tscale + 3 * fid + 1) : 0.f;
        }
        const int q = warp & 3, part = cwarp >> 2;
        const int n_valid = min(pmax, I.n_e - pass * pmax);
        const int row = I.mt * kBM + q * 32 + lane;  // output column of Hp / Yp
        const size_t m0 = static_cast<size_t>(I.row_lo) + pass * pmax;
        const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16);
        for (int c0 = part * 16; c0 < n_valid; c0 += 64) {
          float v0[16], v1[16];
          tmem_ld16x2(tq + c0, tq + 256 + c0, v0, v1);
          const float xs_l =
              (NMAT == 2 && c0 + (lane & 15) < n_valid) ? __ldg(a.x_scale + m0 + c0 + (lane & 15)) : 0.f;
#pragma unroll
          for (int jj = 0; jj < 16; jj += 2) {
            float o[2];
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              if (NMAT == 2) {
                const float xs = __shfl_sync(0xffffffffu, xs_l, jj + t);
                const float gv = v0[jj + t] * ts[0] * xs, uv = v1[jj + t] * ts[1] * xs;
                o[t] = __fdividef(gv, 1.f + __expf(fminf(-gv, 80.f))) * uv * kHScale;
                if (!(fabsf(o[t]) <= 65504.f) && c0 + jj + t < n_valid) record_status(a.dev_status, FT_ERR_RANGE);
              } else {
                o[t] = (v0[jj + t] + v1[jj + t]) * ts[0] * (1.f / kHScale);
              }
            }
            // lane pairs swap halves so each lane stores two adjacent outputs of
            // one token (even lane: token jj, odd lane: token jj + 1)
            const float mine = (lane & 1) ? o[0] : o[1];
            const float other = __shfl_xor_sync(0xffffffffu, mine, 1);
            const int col = c0 + jj + (lane & 1);
            const float lo = (lane & 1) ? other : o[0], hi = (lane & 1) ? o[1] : other;
            uint32_t pk;
            if (NMAT == 2)
              pk = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(lo))) |
                   (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(hi))) << 16);
            else
              pk = static_cast<uint32_t>(f32_to_bf16(lo)) | (static_cast<uint32_t>(f32_to_bf16(hi)) << 16);
            if (col < n_valid) *reinterpret_cast<uint32_t*>(a.out + (m0 + col) * a.M + (row & ~1)) = pk;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  // A wait that gave up (FT_ERR_TIMEOUT recorded) ends its role's loop with
  // this CTA's TMA copies or MMAs possibly still in flight: let them land
  // (a bounded 200 us) before the TMEM is freed and the CTA exits.
  __shared__ int s_drain;
  if (tid == 0) s_drain = a.dev_status != nullptr && *reinterpret_cast<const volatile int32_t*>(a.dev_status) == FT_ERR_TIMEOUT;
  __syncthreads();
  if (s_drain) {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 200000ull) {
    }
    __syncthreads();
  }
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols) : "memory");
  }
}

// ------------------------------------------------------------ tensor maps ---
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  }
  return fn;
}

// A [n_blocks][rows][inner] byte tensor (codes or scales of one matrix of every
// block in a bank), box {box_inner, 128 rows, 1 block}.
bool map_bank(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t blocks,
              uint64_t block_stride, uint32_t box_inner, CUtensorMapSwizzle swizzle) {
  const cuuint64_t dims[3] = {inner, rows, blocks};
  const cuuint64_t strides[2] = {inner, block_stride};
  const cuuint32_t box[3] = {box_inner, static_cast<cuuint32_t>(kBM), 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A [rows][cols] f16 activation matrix, box {64 cols, 64 rows}, 128-byte swizzle.
bool map_acts(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(kBRows)};
  const cuuint32_t es[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t experts_prefill_workspace(int32_t T, int32_t k, int32_t H, int32_t I, int32_t E) {
  (void)H;
  (void)E;
  return (static_cast<size_t>(T) * k * I * 2 + 255) & ~static_cast<size_t>(255);
}

ft_status experts_prefill(const ft_bank* cache, const ft_bank* pool, int32_t layer, int32_t E,
                          const uint16_t* xp, const float* x_scale, int32_t T, int32_t k,
                          const int32_t* slot_of_expert, const int32_t* offsets, uint16_t* yp, void* ws,
                          size_t ws_bytes, int32_t* dev_status, cudaStream_t s) {
  (void)pool;
  const int H = cache->H, I = cache->I;
  if (cache->fmt != FT_NVFP4) return fail(FT_ERR_UNSUPPORTED, "experts prefill: NVFP4 banks only");
  FT_REQUIRE(H % kSuper == 0 && I % kSuper == 0, "experts prefill: H and I must be multiples of 256");
  FT_REQUIRE(x_scale != nullptr, "experts prefill: x_scale is NULL");
  const int64_t n_rows64 = static_cast<int64_t>(T) * k;
  FT_REQUIRE(n_rows64 < (1ll << 31), "experts prefill: T*k overflows int32");
  FT_REQUIRE(E <= 65535, "experts prefill: E %d > 65535", E);
  FT_REQUIRE(ws_bytes >= experts_prefill_workspace(T, k, H, I, E), "experts prefill: workspace too small");
  FT_REQUIRE(reinterpret_cast<uintptr_t>(xp) % 16 == 0 && reinterpret_cast<uintptr_t>(ws) % 16 == 0,
             "experts prefill: xp and ws must be 16-byte aligned");
  if (encode_fn() == nullptr) return fail(FT_ERR_CUDA, "experts prefill: cuTensorMapEncodeTiled unavailable");
  Layout L;
  layout(cache->fmt, H, I, cache->group, &L);
  const uint8_t* base = static_cast<const uint8_t*>(cache->base);
  const uint64_t nb = static_cast<uint64_t>(cache->n_blocks), st = cache->stride;
  const int n_rows = static_cast<int>(n_rows64);
  uint16_t* hp = static_cast<uint16_t*>(ws);
  CUtensorMap mg, mu, mgs, mus, mx, md, mds, mh;
  bool ok = map_bank(&mg, base + L.off[0], H / 2, I, nb, st, kRawSteps * kBK / 2, CU_TENSOR_MAP_SWIZZLE_64B) &&
            map_bank(&mu, base + L.off[1], H / 2, I, nb, st, kRawSteps * kBK / 2, CU_TENSOR_MAP_SWIZZLE_64B) &&
            map_bank(&mgs, base + L.off[3], H / 16, I, nb, st, 16, CU_TENSOR_MAP_SWIZZLE_NONE) &&
            map_bank(&mus, base + L.off[4], H / 16, I, nb, st, 16, CU_TENSOR_MAP_SWIZZLE_NONE) &&
            map_acts(&mx, xp, H, n_rows) &&
            map_bank(&md, base + L.off[2], I / 2, H, nb, st, kRawSteps * kBK / 2, CU_TENSOR_MAP_SWIZZLE_64B) &&
            map_bank(&mds, base + L.off[5], I / 16, H, nb, st, 16, CU_TENSOR_MAP_SWIZZLE_NONE) &&
            map_acts(&mh, hp, I, n_rows);
  if (!ok) return fail(FT_ERR_INVALID, "experts prefill: tensor map encoding rejected the bank or batch");
  {
    ft_status sa = ensure_dyn_smem(reinterpret_cast<const void*>(pf_kernel<2, false>), PfSmem<2>::total + 1024,
                                   "experts prefill");
    if (sa == FT_OK)
      sa = ensure_dyn_smem(reinterpret_cast<const void*>(pf_kernel<2, true>), PfSmem<2>::total + 1024,
                           "experts prefill");
    if (sa == FT_OK)
      sa = ensure_dyn_smem(reinterpret_cast<const void*>(pf_kernel<1, false>), PfSmem<1>::total + 1024,
                           "experts prefill");
    if (sa == FT_OK)
      sa = ensure_dyn_smem(reinterpret_cast<const void*>(pf_kernel<1, true>), PfSmem<1>::total + 1024,
                           "experts prefill");
    if (sa != FT_OK) return sa;
  }
  PfArgs a;
  a.offsets = offsets;
  a.slot_of = slot_of_expert;
  a.E = E;
  a.n_rows = n_rows;
  a.layer = layer;
  a.n_blocks = cache->n_blocks;
  a.tscale = cache->tensor_scale;
  a.dev_status = dev_status;
  // gate/up: K = H, M = I, output Hp (f16)
  a.K = H;
  a.M = I;
  a.x_scale = x_scale;
  a.out = hp;
  // token tiles inside the A stages when the mean segment is short (passes
  // of 128 tokens), else separate token rings (passes of 256); one CTA per SM
  // walks the (row tile, expert) items
  const bool mrg = static_cast<int64_t>(T) * k <= static_cast<int64_t>(kMrgMeanRows) * E;
  a.pmax = mrg ? 128 : kNMax;
  const int sms = device_sm_count();
  a.tiles = I / kBM;
  const unsigned g1 = static_cast<unsigned>(std::min<int64_t>(static_cast<int64_t>(a.tiles) * E, sms));
  if (mrg)
    pf_kernel<2, true><<<g1, kPfThreads, PfSmem<2>::total + 1024, s>>>(mg, mu, mgs, mus, mx, a);
  else
    pf_kernel<2, false><<<g1, kPfThreads, PfSmem<2>::total + 1024, s>>>(mg, mu, mgs, mus, mx, a);
  ft_status stt = launch_check("experts prefill gate/up");
  if (stt != FT_OK) return stt;
  // down: K = I, M = H, output Yp (bf16)
  a.K = I;
  a.M = H;
  a.x_scale = nullptr;
  a.out = yp;
  a.tiles = H / kBM;
  const unsigned g2 = static_cast<unsigned>(std::min<int64_t>(static_cast<int64_t>(a.tiles) * E, sms));
  if (mrg)
    pf_kernel<1, true><<<g2, kPfThreads, PfSmem<1>::total + 1024, s>>>(md, md, mds, mds, mh, a);
  else
    pf_kernel<1, false><<<g2, kPfThreads, PfSmem<1>::total + 1024, s>>>(md, md, mds, mds, mh, a);
  return launch_check("experts prefill down");
}

}  // namespace ft
