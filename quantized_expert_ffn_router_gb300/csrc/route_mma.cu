// route_mma.cu -- the router logits of long prompts on the tcgen05 tensor
// cores: logits[t, e] = x[t, :] . W[e, :] with x in bf16 and W in fp32.
//
// W is split exactly into three bf16 terms, W = hi + mid + lo: hi is W rounded
// to bf16, mid the remainder rounded to bf16, lo the rest, which then holds no
// more than bf16's 8 significant bits (fp32 has 24).  Every product of a bf16
// x with a bf16 term is exact in fp32.  The tensor core's fp32 accumulation
// truncates what each MMA adds, an error of up to about an ulp of the running
// sum per instruction, always toward zero, so it grows with the number of MMAs
// that feed one accumulator.  Two measures keep that count small: hi's
// products and the (2^8 times smaller) mid + lo products go to accumulators
// of their own, and the hidden axis is split over kRouteSplitK-step slices,
// one CTA each, whose fp32 partial logits the top-k kernel adds in a fixed
// order.  With at most 16 k-steps a slice, hi's accumulator takes at most 64
// MMAs (768 went into one accumulator without these measures).
//
// One CTA per (128-token tile, 128-expert tile, hidden slice), 192 threads:
//   warp 0 (lane 0)  TMA: per 64-wide k-step the token tile [128 x 64] and
//                    the three term tiles [128 x 64], 128-byte swizzle, into
//                    a 3-stage ring (64 KB a stage);
//   warp 1 (lane 0)  tcgen05.mma kind::f16 (bf16 x bf16 -> fp32), M = 128,
//                    N = 128, K = 16: twelve MMAs per k-step into two
//                    accumulators of 128 TMEM columns (hi; mid + lo);
//   warps 2..5       epilogue: tcgen05.ld of their TMEM lane quarter (32
//                    tokens) from both accumulators, their fp32 sum to the
//                    slice's partial logits in global memory.
// Tokens past T are read as zeros by the TMA and never written.
//
// Source: "FreeToken: 让消费级电脑跑起 284B MoE" (fengjutian.github.io), sec. 2
// (the router runs on the GPU; logits, softmax, top-k).
#include <cuda.h>

#include <algorithm>

#include "ft_async.cuh"
#include "ft_common.cuh"

namespace ft {
namespace {

constexpr int kRM = 128;      // tokens per tile (MMA M)
constexpr int kRN = 128;      // experts per tile (MMA N)
constexpr int kRK = 64;       // K per stage: one 128-byte row of bf16
constexpr int kRStages = 3;
constexpr int kRThreads = 192;
constexpr int kRTile = kRM * kRK * 2;  // 16 KB: one 128 x 64 bf16 tile
constexpr int kRStage = 4 * kRTile;    // tokens + three terms
constexpr int kRSmem = kRStages * kRStage + 1024;
constexpr int kRouteSplitK = 16;  // k-steps per hidden slice, at most
constexpr int kRCols = 2 * kRN;   // TMEM columns: the hi and the mid + lo accumulators

__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// K-major operand tile in the 128-byte swizzle layout (rows of 128 B, 8-row
// groups 1024 B apart), descriptor version 1, layout SWIZZLE_128B.
__device__ __forceinline__ uint64_t sw128(const void* tile) {
  const uint64_t addr = smem_u32(tile);
  uint64_t d = (addr >> 4) & 0x3FFFull;
  d |= 1ull << 16;
  d |= (1024ull >> 4) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// kind::f16 instruction descriptor: fp32 D, bf16 A and B (format 1), both
// K-major, N = kRN, M = kRM.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(kRN >> 3) << 17) |
                            (static_cast<uint32_t>(kRM >> 4) << 24);

// Sixteen consecutive TMEM columns of this warp's lane quarter, one per
// register (the caller waits with tcgen05.wait::ld).
__device__ __forceinline__ void tmem_ld16(uint32_t addr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(addr)
      : "memory");
}

__global__ void route_split_kernel(const float* __restrict__ W, size_t n, uint16_t* __restrict__ hi,
                                   uint16_t* __restrict__ mid, uint16_t* __restrict__ lo) {
  pdl_wait();
  pdl_launch_dependents();
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float w = W[i];
    const uint16_t h = f32_to_bf16(w);
    const float r1 = w - bf16_val(h);  // exact: w and bf16(w) share their top bits
    const uint16_t m = f32_to_bf16(r1);
    const float r2 = r1 - bf16_val(m);
    hi[i] = h;
    mid[i] = m;
    lo[i] = f32_to_bf16(r2);
  }
}

__global__ void __launch_bounds__(kRThreads, 1) route_mma_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                  const __grid_constant__ CUtensorMap wmap,
                                                                  int T, int E, int H, float* __restrict__ part0,
                                                                  float* __restrict__ partx) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[kRStages], empty[kRStages], acc_full;
  __shared__ uint32_t s_tmem;
  __shared__ int s_gave_up;  // a wait gave up: copies or MMAs may be in flight at the end
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kRM, n0 = blockIdx.y * kRN;
  const int kall = H / kRK, z = blockIdx.z, nz = gridDim.z;
  const int kbeg = (z * kall) / nz, ksteps = ((z + 1) * kall) / nz - kbeg;
  float* __restrict__ logits = z == 0 ? part0 : partx + static_cast<size_t>(z - 1) * T * E;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&acc_full, 1);
    s_gave_up = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(kRCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = s_tmem;
  pdl_wait();  // x comes from the previous kernel, the terms from the split kernel
  pdl_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      for (int kk = 0; kk < ksteps; ++kk) {
        const int st = kk % kRStages;
        if (kk >= kRStages && !mbar_wait(&empty[st], ((kk / kRStages) - 1) & 1, nullptr)) {
          s_gave_up = 1;
          break;
        }
        uint8_t* stage = smem + st * kRStage;
        mbar_arrive_expect_tx(&full[st], kRStage);
        const int kc = (kbeg + kk) * kRK;
        tma_2d(stage, &xmap, kc, m0, &full[st]);
        for (int t = 0; t < 3; ++t) tma_2d(stage + (1 + t) * kRTile, &wmap, kc, t * E + n0, &full[st]);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = true;
      for (int kk = 0; kk < ksteps; ++kk) {
        const int st = kk % kRStages;
        if (!mbar_wait(&full[st], (kk / kRStages) & 1, nullptr)) {
          ok = false;
          s_gave_up = 1;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint8_t* stage = smem + st * kRStage;
        const uint64_t ad = sw128(stage);
#pragma unroll
        for (int t = 0; t < 3; ++t) {
          const uint64_t bd = sw128(stage + (1 + t) * kRTile);
          const uint32_t dst = t == 0 ? tmem : tmem + kRN;  // hi | mid + lo
#pragma unroll
          for (int j = 0; j < kRK / 16; ++j) {
            const uint32_t acc = (kk > 0 || t > 1 || j > 0) ? 1u : 0u;
            asm volatile(
                "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(dst),
                "l"(ad + 2 * j), "l"(bd + 2 * j), "r"(kIdesc), "r"(acc)
                : "memory");
          }
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         smem_u32(&empty[st]))
                     : "memory");
      }
      if (ok)
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         smem_u32(&acc_full))
                     : "memory");
    }
  } else {
    // warps 2..5: TMEM lane quarter q = warp % 4, token m0 + 32 q + lane
    if (!mbar_wait_warp(&acc_full, 0, nullptr)) {  // one verdict per warp: tcgen05.ld follows
      s_gave_up = 1;
    } else {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int q = warp & 3;
      const int t = m0 + q * 32 + lane;
      const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16);
      for (int c0 = 0; c0 < kRN; c0 += 16) {
        uint32_t r[16], u[16];
        tmem_ld16(tq + c0, r);
        tmem_ld16(tq + kRN + c0, u);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (t < T) {
          float4* dst = reinterpret_cast<float4*>(logits + static_cast<size_t>(t) * E + n0 + c0);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            float o[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) o[c] = __uint_as_float(r[4 * v + c]) + __uint_as_float(u[4 * v + c]);
            dst[v] = make_float4(o[0], o[1], o[2], o[3]);
          }
        }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (s_gave_up) {  // let this CTA's copies and MMAs still in flight land (bounded)
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 200000ull) {
    }
    __syncthreads();
  }
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kRCols) : "memory");
  }
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn route_encode_fn() {
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

// [rows][cols] bf16, box {64 cols, 128 rows}, 128-byte swizzle; rows past the
// end read as zeros.
bool map_bf16(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kRK), static_cast<cuuint32_t>(kRM)};
  const cuuint32_t es[2] = {1, 1};
  return route_encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool route_mma_fits(int T, int E, int H) { return T > 16 && E % kRN == 0 && H % kRK == 0 && H >= kRK; }

// Hidden slices of the tensor-core path: at most kRouteSplitK k-steps each.
int route_mma_slices(int H) { return (H / kRK + kRouteSplitK - 1) / kRouteSplitK; }

size_t route_mma_terms_bytes(int E, int H) {
  return (static_cast<size_t>(3) * E * H * 2 + 255) & ~static_cast<size_t>(255);
}

// Bytes the tensor-core path keeps in the route workspace after the logits:
// the three bf16 terms of W, then the partial logits [T, E] fp32 of every
// hidden slice but the first (0 when the shape does not take that path).
size_t route_mma_split_bytes(int T, int E, int H) {
  if (!route_mma_fits(T, E, H)) return 0;
  const size_t part = static_cast<size_t>(route_mma_slices(H) - 1) * T * E * sizeof(float);
  return route_mma_terms_bytes(E, H) + ((part + 255) & ~static_cast<size_t>(255));
}

// The partial logits [T, E] fp32 of x [T, H] bf16 and W [E, H] fp32, one per
// hidden slice: the first slice's in `logits`, the others' after W's three
// bf16 terms in `extra` (route_mma_split_bytes); their sum is the logits.
// Both launches are programmatic dependents of the previous kernel on the
// stream.  Returns the number of slices in *slices.
// Where the partial logits of the slices after the first begin in `extra`.
float* route_mma_partials(void* extra, int E, int H) {
  return reinterpret_cast<float*>(static_cast<uint8_t*>(extra) + route_mma_terms_bytes(E, H));
}

ft_status route_mma_logits(const uint16_t* x, int T, int H, const float* W, int E, float* logits, void* extra,
                           int* slices, cudaStream_t s) {
  void* terms = extra;
  const int nz = route_mma_slices(H);
  float* partx = route_mma_partials(extra, E, H);
  *slices = nz;
  if (route_encode_fn() == nullptr) return fail(FT_ERR_CUDA, "route: cuTensorMapEncodeTiled unavailable");
  uint16_t* hi = static_cast<uint16_t*>(terms);
  const size_t n = static_cast<size_t>(E) * H;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(std::min<size_t>((n + 255) / 256, 4u * static_cast<size_t>(device_sm_count()))));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, route_split_kernel, W, n, hi, hi + n, hi + 2 * n);
    if (e != cudaSuccess) return fail(FT_ERR_CUDA, "route split: %s", cudaGetErrorString(e));
  }
  CUtensorMap xmap, wmap;
  if (!map_bf16(&xmap, x, H, T) || !map_bf16(&wmap, hi, H, static_cast<uint64_t>(3) * E))
    return fail(FT_ERR_INVALID, "route: tensor map encoding rejected x or the router terms");
  ft_status st = ensure_dyn_smem(reinterpret_cast<const void*>(route_mma_kernel), kRSmem, "route");
  if (st != FT_OK) return st;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((T + kRM - 1) / kRM, E / kRN, nz);
  cfg.blockDim = dim3(kRThreads);
  cfg.dynamicSmemBytes = kRSmem;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, route_mma_kernel, xmap, wmap, T, E, H, logits, partx);
  if (e != cudaSuccess) return fail(FT_ERR_CUDA, "route logits: %s", cudaGetErrorString(e));
  return launch_check("route logits");
}

}  // namespace ft
