// prefill.cu -- token-permuted grouped SwiGLU expert GEMM on tcgen05/TMEM.
//
// Sources: "NVMe에서 전문가(experts)를 ... 133GB MoE" (molayo1419.me), engine
// step 5 (the whole prompt goes through a layer's experts at once, so every
// expert's weights are read once per layer); "FreeToken: 让消费级电脑跑起 284B
// MoE" (fengjutian.github.io), sec. 3 (prefill touches nearly every expert
// and is dense compute).
//
// Two launches, each one CTA per (128-row weight tile, expert):
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
// Roles (192 threads): warp 0 lane 0 issues TMA (raw codes with the 128-byte
// swizzle so converter threads read them conflict-free, E4M3 scales, and the
// B tiles), warp 1 lane 0 issues the MMAs, warps 2..5 dequantise one weight
// row per thread into the 128-byte-swizzled K-major A tile and afterwards run
// the epilogue (tcgen05.ld, 32 TMEM lanes per warp).  Stages are handed over
// with mbarriers; every wait is bounded.
#include <cuda.h>
#include <cuda_fp16.h>

#include "ft_async.cuh"
#include "ft_common.cuh"

namespace ft {
namespace {

constexpr int kBM = 128;        // weight rows per tile (MMA M)
constexpr int kBK = 64;         // K per k-step: one 128-byte row of f16
constexpr int kSuper = 256;     // K per raw stage: 128 code bytes per row
constexpr int kNMax = 256;      // tokens per pass (MMA N)
constexpr int kBRows = 64;      // rows per B TMA box
constexpr int kStages = 2;      // raw, A and B ring depth
constexpr int kPfThreads = 192;
constexpr float kHScale = 0.0625f;  // h is stored as f16(h * 2^-4)

constexpr int kATile = kBM * kBK * 2;            // 16 KB per matrix per k-step
constexpr int kBTile = kNMax * kBK * 2;          // 32 KB
constexpr int kRawCodes = kBM * (kSuper / 2);    // 16 KB per matrix per raw stage
constexpr int kRawScales = kBM * (kSuper / 16);  // 2 KB

template <int NMAT>
struct PfSmem {
  static constexpr int a_off = 0;
  static constexpr int b_off = a_off + kStages * NMAT * kATile;
  static constexpr int raw_off = b_off + kStages * kBTile;
  static constexpr int raw_codes = 0;                          // within a raw stage
  static constexpr int raw_scales = NMAT * kRawCodes;
  static constexpr int raw_stage = NMAT * (kRawCodes + kRawScales);
  static constexpr int total = raw_off + kStages * raw_stage;
};

struct PfArgs {
  const int32_t* offsets;  // [E+1]
  const int32_t* slot_of;  // [E] cache slot of each expert
  int E, K, M, n_rows, layer;
  int64_t n_blocks;
  const float* x_scale;    // [n_rows] (gate/up only)
  const float* tscale;     // [n_fids, 3]
  uint16_t* out;           // gate/up: Hp f16 [n_rows, M]; down: Yp bf16 [n_rows, M]
  int32_t* dev_status;
};

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

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float v[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

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

// Four E4M3 scale bytes -> four broadcast f16x2 values {s_i, s_i}.
__device__ __forceinline__ void scales4(uint32_t four, uint32_t s2[4]) {
  uint32_t lo, hi;
  const unsigned short b01 = static_cast<unsigned short>(four & 0xffffu);
  const unsigned short b23 = static_cast<unsigned short>(four >> 16);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"(b01));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"(b23));
  s2[0] = __byte_perm(lo, 0, 0x1010);
  s2[1] = __byte_perm(lo, 0, 0x3232);
  s2[2] = __byte_perm(hi, 0, 0x1010);
  s2[3] = __byte_perm(hi, 0, 0x3232);
}

// ---------------------------------------------------------------- kernel ---
// NMAT = 2: gate/up (maps c0,c1 = codes, s0,s1 = scales); NMAT = 1: down.
template <int NMAT>
__global__ void __launch_bounds__(kPfThreads, 1) pf_kernel(const __grid_constant__ CUtensorMap c0map,
                                                           const __grid_constant__ CUtensorMap c1map,
                                                           const __grid_constant__ CUtensorMap s0map,
                                                           const __grid_constant__ CUtensorMap s1map,
                                                           const __grid_constant__ CUtensorMap bmap,
                                                           PfArgs a) {
  using L = PfSmem<NMAT>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t raw_full[kStages], raw_empty[kStages];
  __shared__ __align__(8) uint64_t a_full[kStages], a_empty[kStages];
  __shared__ __align__(8) uint64_t b_full[kStages], b_empty[kStages];
  __shared__ __align__(8) uint64_t acc_full, acc_empty;
  __shared__ uint32_t s_tmem;

  if (prior_timeout(a.dev_status)) return;
  const int e = blockIdx.y, mt = blockIdx.x;
  const int row_lo = a.offsets[e];
  const int n_e = a.offsets[e + 1] - row_lo;
  if (n_e <= 0) return;
  const int slot = a.slot_of[e];
  if (slot < 0 || slot >= a.n_blocks || row_lo < 0 || row_lo + n_e > a.n_rows) {
    if (threadIdx.x == 0) record_status(a.dev_status, slot < 0 ? FT_ERR_UNSUPPORTED : FT_ERR_BAD_ID);
    return;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ksteps = a.K / kBK, supers = a.K / kSuper;
  const int n_pass = (n_e + kNMax - 1) / kNMax;
  constexpr uint32_t kCols = NMAT == 2 ? 512 : 256;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], 4);
      mbar_init(&a_full[s], 4);
      mbar_init(&a_empty[s], 1);
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    mbar_init(&acc_full, 1);
    mbar_init(&acc_empty, 4);
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

  if (warp == 0) {
    // ------------------------------------------------------------- TMA ---
    if (lane == 0) {
      const CUtensorMap* cm[2] = {&c0map, &c1map};
      const CUtensorMap* sm[2] = {&s0map, &s1map};
      for (int pass = 0; pass < n_pass; ++pass) {
        const int n_valid = min(kNMax, n_e - pass * kNMax);
        const int nbox = (n_valid + kBRows - 1) / kBRows;
        for (int s = 0; s < supers; ++s) {
          const int ru = pass * supers + s, rst = ru % kStages;
          if (ru >= kStages && !mbar_wait(&raw_empty[rst], ((ru / kStages) - 1) & 1, a.dev_status)) goto done_tma;
          uint8_t* raw = smem + L::raw_off + rst * L::raw_stage;
          mbar_arrive_expect_tx(&raw_full[rst], NMAT * (kRawCodes + kRawScales));
          for (int m = 0; m < NMAT; ++m) {
            tma_load_3d(raw + L::raw_codes + m * kRawCodes, cm[m], s * (kSuper / 2), mt * kBM, slot, &raw_full[rst]);
            tma_load_3d(raw + L::raw_scales + m * kRawScales, sm[m], s * (kSuper / 16), mt * kBM, slot,
                        &raw_full[rst]);
          }
          for (int j = 0; j < kSuper / kBK; ++j) {
            const int kk = s * (kSuper / kBK) + j;
            const int bu = pass * ksteps + kk, bst = bu % kStages;
            if (bu >= kStages && !mbar_wait(&b_empty[bst], ((bu / kStages) - 1) & 1, a.dev_status)) goto done_tma;
            uint8_t* bt = smem + L::b_off + bst * kBTile;
            mbar_arrive_expect_tx(&b_full[bst], nbox * kBRows * kBK * 2);
            for (int bx = 0; bx < nbox; ++bx)
              tma_load_2d(bt + bx * kBRows * kBK * 2, &bmap, kk * kBK, row_lo + pass * kNMax + bx * kBRows,
                          &b_full[bst]);
          }
        }
      }
    done_tma:;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA ---
    if (lane == 0) {
      bool ok = true;
      for (int pass = 0; pass < n_pass && ok; ++pass) {
        const int n_valid = min(kNMax, n_e - pass * kNMax);
        const int n_mma = (n_valid + 15) & ~15;
        const uint32_t idesc = idesc_f16(n_mma);
        if (pass > 0) {
          if (!mbar_wait(&acc_empty, (pass - 1) & 1, a.dev_status)) break;
          tc_fence_after();
        }
        for (int kk = 0; kk < ksteps; ++kk) {
          const int u = pass * ksteps + kk, st = u % kStages;
          if (!mbar_wait(&a_full[st], (u / kStages) & 1, a.dev_status) ||
              !mbar_wait(&b_full[st], (u / kStages) & 1, a.dev_status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint8_t* at = smem + L::a_off + st * NMAT * kATile;
          const uint64_t bdesc = sw128_desc(smem + L::b_off + st * kBTile);
#pragma unroll
          for (int j = 0; j < kBK / 16; ++j) {
            const uint32_t acc = (kk > 0 || j > 0) ? 1u : 0u;
#pragma unroll
            for (int m = 0; m < NMAT; ++m)
              mma_f16(tmem + m * 256, sw128_desc(at + m * kATile) + 2 * j, bdesc + 2 * j, idesc, acc);
          }
          mma_commit(&a_empty[st]);
          mma_commit(&b_empty[st]);
        }
        if (ok) mma_commit(&acc_full);
      }
    }
  } else {
    // --------------------------------------- convert, then the epilogue ---
    const int r = tid - 64;  // weight row within the tile (0..127)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    float ts[2] = {1.f, 1.f};
    {
      const int64_t fid = static_cast<int64_t>(a.layer) * a.E + e;
      if (NMAT == 2) {
        ts[0] = __ldg(a.tscale + 3 * fid + 0);
        ts[1] = __ldg(a.tscale + 3 * fid + 1);
      } else {
        ts[0] = __ldg(a.tscale + 3 * fid + 2);
      }
    }
    bool ok = true;
    for (int pass = 0; pass < n_pass && ok; ++pass) {
      for (int s = 0; s < supers && ok; ++s) {
        const int ru = pass * supers + s, rst = ru % kStages;
        if (!mbar_wait(&raw_full[rst], (ru / kStages) & 1, a.dev_status)) {
          ok = false;
          break;
        }
        const uint8_t* raw = smem + L::raw_off + rst * L::raw_stage;
        uint4 sc[NMAT];
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
          sc[m] = *reinterpret_cast<const uint4*>(raw + L::raw_scales + m * kRawScales + r * 16);
        for (int j = 0; j < kSuper / kBK; ++j) {
          const int kk = s * (kSuper / kBK) + j;
          const int u = pass * ksteps + kk, ast = u % kStages;
          if (u >= kStages && !mbar_wait(&a_empty[ast], ((u / kStages) - 1) & 1, a.dev_status)) {
            ok = false;
            break;
          }
          uint8_t* at = smem + L::a_off + ast * NMAT * kATile;
#pragma unroll
          for (int m = 0; m < NMAT; ++m) {
            const uint32_t sw = (j == 0) ? sc[m].x : (j == 1) ? sc[m].y : (j == 2) ? sc[m].z : sc[m].w;
            uint32_t s2[4];
            scales4(sw, s2);
            const uint8_t* crow = raw + L::raw_codes + m * kRawCodes + r * 128;
            // the 32 code bytes of this k-step are logical 16-byte chunks 2j, 2j+1
            const uint4 c0 = *reinterpret_cast<const uint4*>(crow + (((2 * j) ^ (r & 7)) << 4));
            const uint4 c1 = *reinterpret_cast<const uint4*>(crow + (((2 * j + 1) ^ (r & 7)) << 4));
            const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            uint8_t* arow = at + m * kATile + r * 128;
#pragma unroll
            for (int w = 0; w < 8; ++w)
              *reinterpret_cast<uint4*>(arow + ((w ^ (r & 7)) << 4)) = dequant8(words[w], s2[w >> 1]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&a_full[ast]);
        }
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(&raw_empty[rst]);
      }
      if (!ok) break;
      // epilogue of this pass
      if (!mbar_wait(&acc_full, pass & 1, a.dev_status)) break;
      tc_fence_after();
      const int n_valid = min(kNMax, n_e - pass * kNMax);
      const int row = mt * kBM + q * 32 + lane;  // output column of Hp / Yp
      for (int c0 = 0; c0 < n_valid; c0 += 16) {
        float v0[16], v1[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + c0, v0);
        if (NMAT == 2) tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + 256 + c0, v1);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const int col = c0 + jj;
          if (col >= n_valid) break;
          const int m = row_lo + pass * kNMax + col;
          if (NMAT == 2) {
            const float xs = __ldg(a.x_scale + m);
            const float gv = v0[jj] * ts[0] * xs, uv = v1[jj] * ts[1] * xs;
            const float hv = gv / (1.f + expf(-gv)) * uv * kHScale;
            if (!(fabsf(hv) <= 65504.f)) record_status(a.dev_status, FT_ERR_RANGE);
            a.out[static_cast<size_t>(m) * a.M + row] = __half_as_ushort(__float2half_rn(hv));
          } else {
            a.out[static_cast<size_t>(m) * a.M + row] = f32_to_bf16(v0[jj] * ts[0] * (1.f / kHScale));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty);
    }
  }
  tc_fence_before();
  __syncthreads();
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
              uint64_t block_stride, uint32_t box_inner, bool swizzle) {
  const cuuint64_t dims[3] = {inner, rows, blocks};
  const cuuint64_t strides[2] = {inner, block_stride};
  const cuuint32_t box[3] = {box_inner, static_cast<cuuint32_t>(kBM), 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
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
  bool ok = map_bank(&mg, base + L.off[0], H / 2, I, nb, st, kSuper / 2, true) &&
            map_bank(&mu, base + L.off[1], H / 2, I, nb, st, kSuper / 2, true) &&
            map_bank(&mgs, base + L.off[3], H / 16, I, nb, st, kSuper / 16, false) &&
            map_bank(&mus, base + L.off[4], H / 16, I, nb, st, kSuper / 16, false) &&
            map_acts(&mx, xp, H, n_rows) &&
            map_bank(&md, base + L.off[2], I / 2, H, nb, st, kSuper / 2, true) &&
            map_bank(&mds, base + L.off[5], I / 16, H, nb, st, kSuper / 16, false) &&
            map_acts(&mh, hp, I, n_rows);
  if (!ok) return fail(FT_ERR_INVALID, "experts prefill: tensor map encoding rejected the bank or batch");
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(pf_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, PfSmem<2>::total + 1024);
    cudaFuncSetAttribute(pf_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, PfSmem<1>::total + 1024);
    attr = true;
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
  pf_kernel<2><<<dim3(I / kBM, E), kPfThreads, PfSmem<2>::total + 1024, s>>>(mg, mu, mgs, mus, mx, a);
  ft_status stt = launch_check("experts prefill gate/up");
  if (stt != FT_OK) return stt;
  // down: K = I, M = H, output Yp (bf16)
  a.K = I;
  a.M = H;
  a.x_scale = nullptr;
  a.out = yp;
  pf_kernel<1><<<dim3(H / kBM, E), kPfThreads, PfSmem<1>::total + 1024, s>>>(md, md, mds, mds, mh, a);
  return launch_check("experts prefill down");
}

}  // namespace ft
