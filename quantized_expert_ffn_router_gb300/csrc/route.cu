// route.cu -- the router on the GPU: logits = x . W^T (fp32 accumulation),
// softmax over all experts, top-k by probability (ties to the lower id).
//
// Source: "FreeToken: 让消费级电脑跑起 284B MoE" (fengjutian.github.io),
// sec. 2 (the router runs on the GPU and feeds the hit / miss split).
//
// Two logits kernels: a weight-streaming GEMV for small token counts (one CTA
// per expert row) and a tiled SIMT GEMM for long prompts.  Then one warp per
// token does the softmax and the top-k selection, launched as a programmatic
// dependent so it is resident before the logits are done.
#include "ft_async.cuh"
#include "ft_common.cuh"
#include "ft_topk.cuh"

namespace ft {
namespace {

constexpr int kGemvMaxT = 16;
constexpr int kRouteMaxK = 32;
constexpr int kRouteMaxE = 4096;

// The arrival counter's own 256 bytes at the start of the workspace: the same
// offset for every T, so a workspace sized for one T serves any smaller T.
constexpr size_t kRouteCounterBytes = 256;

// Logits of the one-kernel path (T <= 16): [E][kRowsT(T)], every expert's
// logits in a 32-byte sector (or two) of their own, since each is written by
// a different CTA and partial writes from many SMs to one sector would queue
// behind each other.  The tiled path keeps [T][E].
__host__ __device__ constexpr int route_row_stride(int T) { return T <= 8 ? 8 : 16; }

size_t route_logits_bytes(int T, int E) {
  const size_t n = T <= kGemvMaxT ? static_cast<size_t>(E) * route_row_stride(T) : static_cast<size_t>(T) * E;
  return (n * sizeof(float) + 255) & ~static_cast<size_t>(255);
}

// Small token counts: one CTA per expert row, its 8 warps splitting the
// hidden axis, so the whole router matrix is requested by the whole GPU at
// once; partial sums meet in shared memory (fixed order).  The last CTA to
// finish (an arrival counter after the logits in the workspace, back at zero
// when the call ends) then runs the softmax and top-k of every token.
// TAIL = false: the logits only (the combined route + resolve call takes the
// top-k in its resolve kernel, which waits for this whole grid anyway).

template <int TMAX, bool TAIL = true>
__global__ void __launch_bounds__(256) route_rows_kernel(const uint16_t* __restrict__ x, int T, int H,
                                                         const float* __restrict__ W, int E,
                                                         float* __restrict__ logits, unsigned* counter,
                                                         int k, int renorm, int32_t* __restrict__ ids,
                                                         float* __restrict__ wts) {
  extern __shared__ float lsm[];  // last CTA: [min(T, 8)][E] logits
  __shared__ float part[8][TMAX];
  __shared__ int s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x;
  const float4* wrow = reinterpret_cast<const float4*>(W + static_cast<size_t>(e) * H);
  const int nch = H / 8;  // 8-element chunks
  // The router weights are no kernel's output: the first chunks are
  // requested before the wait for the previous kernel, so they arrive while
  // it finishes (the previous layer's experts, started early by its
  // programmatic launch).
  float4 wa[2], wb[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int c = warp * 32 + u * 256 + lane;
    if (c < nch) {
      wa[u] = __ldg(wrow + 2 * c);
      wb[u] = __ldg(wrow + 2 * c + 1);
    }
  }
  pdl_wait();               // x may come from the previous kernel in the stream
  pdl_launch_dependents();  // the next call (resolve) may start its launch now
  float acc[TMAX];
#pragma unroll
  for (int t = 0; t < TMAX; ++t) acc[t] = 0.f;
  for (int c0 = warp * 32; c0 < nch; c0 += 256 * 2) {
    if (c0 != warp * 32) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int c = c0 + u * 256 + lane;
        if (c < nch) {
          wa[u] = __ldg(wrow + 2 * c);
          wb[u] = __ldg(wrow + 2 * c + 1);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int c = c0 + u * 256 + lane;
      if (c >= nch) break;
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (t >= T) break;
        const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H) + c);
        float s = acc[t];
        s = fmaf(bf16_lo(xv.x), wa[u].x, s);
        s = fmaf(bf16_hi(xv.x), wa[u].y, s);
        s = fmaf(bf16_lo(xv.y), wa[u].z, s);
        s = fmaf(bf16_hi(xv.y), wa[u].w, s);
        s = fmaf(bf16_lo(xv.z), wb[u].x, s);
        s = fmaf(bf16_hi(xv.z), wb[u].y, s);
        s = fmaf(bf16_lo(xv.w), wb[u].z, s);
        s = fmaf(bf16_hi(xv.w), wb[u].w, s);
        acc[t] = s;
      }
    }
  }
#pragma unroll
  for (int t = 0; t < TMAX; ++t) {
    if (t >= T) break;
    const float v = warp_sum(acc[t]);
    if (lane == 0) part[warp][t] = v;
  }
  __syncthreads();
  if (threadIdx.x < T) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) v += part[w][threadIdx.x];
    logits[static_cast<size_t>(e) * route_row_stride(T) + threadIdx.x] = v;
  }
  if (!TAIL) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    // the arrival releases this CTA's logits (written before the barrier
    // above) and, for the last CTA, acquires every other CTA's: one
    // acquire-release atomic instead of a fence on each side
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.inc.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(counter), "r"(gridDim.x - 1)
                 : "memory");
    s_last = old == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  for (int t = warp; t < T; t += 8)
    topk_any(logits + t, lsm + static_cast<size_t>(warp) * E, E, k, renorm,
             ids + static_cast<size_t>(t) * k, wts + static_cast<size_t>(t) * k, route_row_stride(T));
}

// Tiled SIMT GEMM: a 64-token x 64-expert tile per CTA, 256 threads with 4x4
// outputs each, K staged 32 at a time through shared memory.
constexpr int kTM = 64, kTN = 64, kTK = 32;

__global__ void __launch_bounds__(256) route_tiled_kernel(const uint16_t* __restrict__ x, int T,
                                                          int H, const float* __restrict__ W,
                                                          int E, float* __restrict__ logits) {
  __shared__ float xs[kTK][kTM + 4];
  __shared__ float ws[kTK][kTN + 4];
  const int t0 = blockIdx.y * kTM, e0 = blockIdx.x * kTN;
  const int tid = threadIdx.x;
  const int tr = (tid / 16) * 4, tc = (tid % 16) * 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < H; k0 += kTK) {
    // x tile: 64 rows x 32 k as bf16 -> 256 threads x 8 elements
    {
      const int row = tid / 4, kk = (tid % 4) * 8;
      const int t = t0 + row;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (t < T) v = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H + k0 + kk));
      xs[kk + 0][row] = bf16_lo(v.x);
      xs[kk + 1][row] = bf16_hi(v.x);
      xs[kk + 2][row] = bf16_lo(v.y);
      xs[kk + 3][row] = bf16_hi(v.y);
      xs[kk + 4][row] = bf16_lo(v.z);
      xs[kk + 5][row] = bf16_hi(v.z);
      xs[kk + 6][row] = bf16_lo(v.w);
      xs[kk + 7][row] = bf16_hi(v.w);
    }
    // W tile: 64 experts x 32 k fp32 -> 256 threads x 2 float4
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int idx = tid + u * 256;
      const int row = idx / 8, kk = (idx % 8) * 4;
      const int e = e0 + row;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e < E) v = __ldg(reinterpret_cast<const float4*>(W + static_cast<size_t>(e) * H + k0 + kk));
      ws[kk + 0][row] = v.x;
      ws[kk + 1][row] = v.y;
      ws[kk + 2][row] = v.z;
      ws[kk + 3][row] = v.w;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kTK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = xs[kk][tr + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = ws[kk][tc + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + tr + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tc + j;
      if (e < E) logits[static_cast<size_t>(t) * E + e] = acc[i][j];
    }
  }
}

// One warp per token.  With nx > 0 the logits come in 1 + nx partial sums
// (logits, then partx's [nx][T][E]); the warp adds them in slice order over
// its own row of `logits` (no other warp reads or writes that row) before the
// top-k reads it back.
__global__ void __launch_bounds__(256) route_topk_kernel(float* __restrict__ logits, int T,
                                                         int E, int k, int renorm,
                                                         int32_t* __restrict__ ids,
                                                         float* __restrict__ wts,
                                                         const float* __restrict__ partx, int nx) {
  extern __shared__ float lsm[];  // [warps][E]
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + warp;
  if (t >= T) return;
  float* row = logits + static_cast<size_t>(t) * E;
  if (nx > 0) {
    const size_t plane = static_cast<size_t>(T) * E;
    const float* px = partx + static_cast<size_t>(t) * E;
    for (int e = lane; e < E; e += 32) {
      float v = row[e];
      for (int z = 0; z < nx; ++z) v += px[z * plane + e];
      row[e] = v;
    }
    __syncwarp();  // the row's sums, written by every lane, before any lane reads them
  }
  topk_any(row, lsm + static_cast<size_t>(warp) * E, E, k, renorm, ids + static_cast<size_t>(t) * k,
           wts + static_cast<size_t>(t) * k);
}


// Host: launch route_rows_kernel (T <= kGemvMaxT), logits and top-k in one
// kernel; the arrival counter is the first word of ws, the logits follow it.
ft_status launch_rows(const uint16_t* x, int T, int H, const float* W, int E, int k, int renorm,
                      int32_t* ids, float* wts, void* ws, cudaStream_t s) {
  unsigned* counter = static_cast<unsigned*>(ws);
  float* logits = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kRouteCounterBytes);
  const size_t smem = static_cast<size_t>(T < 8 ? T : 8) * E * sizeof(float);
  {
    const int mx = 8 * kRouteMaxE * static_cast<int>(sizeof(float));
    ft_status st = ensure_dyn_smem(reinterpret_cast<const void*>(route_rows_kernel<1>), mx, "route");
    if (st == FT_OK) st = ensure_dyn_smem(reinterpret_cast<const void*>(route_rows_kernel<4>), mx, "route");
    if (st == FT_OK) st = ensure_dyn_smem(reinterpret_cast<const void*>(route_rows_kernel<16>), mx, "route");
    if (st != FT_OK) return st;
  }
  cudaLaunchConfig_t rc = {};
  rc.gridDim = dim3(E);
  rc.blockDim = dim3(256);
  rc.dynamicSmemBytes = smem;
  rc.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  rc.attrs = at;
  rc.numAttrs = 1;
  cudaError_t le;
  if (T <= 1)
    le = cudaLaunchKernelEx(&rc, route_rows_kernel<1>, x, T, H, W, E, logits, counter, k, renorm, ids, wts);
  else if (T <= 4)
    le = cudaLaunchKernelEx(&rc, route_rows_kernel<4>, x, T, H, W, E, logits, counter, k, renorm, ids, wts);
  else
    le = cudaLaunchKernelEx(&rc, route_rows_kernel<16>, x, T, H, W, E, logits, counter, k, renorm, ids, wts);
  if (le != cudaSuccess) return fail(FT_ERR_CUDA, "route: %s", cudaGetErrorString(le));
  return launch_check("route");
}

}  // namespace

// Logits only, for T <= 16: [E][route_row_stride(T)] floats at ws + 256
// (the layout the top-k of the combined route + resolve call reads), one CTA
// per expert row, launched as a programmatic dependent of the previous kernel.
ft_status route_rows_logits(const uint16_t* x, int T, int H, const float* W, int E, void* ws, cudaStream_t s,
                            const float** logits_out, int* stride_out) {
  float* logits = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kRouteCounterBytes);
  cudaLaunchConfig_t rc = {};
  rc.gridDim = dim3(E);
  rc.blockDim = dim3(256);
  rc.dynamicSmemBytes = 0;
  rc.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  rc.attrs = at;
  rc.numAttrs = 1;
  cudaError_t le;
  unsigned* counter = static_cast<unsigned*>(ws);  // untouched without the tail
  if (T <= 1)
    le = cudaLaunchKernelEx(&rc, route_rows_kernel<1, false>, x, T, H, W, E, logits, counter, 1, 0,
                            static_cast<int32_t*>(nullptr), static_cast<float*>(nullptr));
  else if (T <= 4)
    le = cudaLaunchKernelEx(&rc, route_rows_kernel<4, false>, x, T, H, W, E, logits, counter, 1, 0,
                            static_cast<int32_t*>(nullptr), static_cast<float*>(nullptr));
  else
    le = cudaLaunchKernelEx(&rc, route_rows_kernel<16, false>, x, T, H, W, E, logits, counter, 1, 0,
                            static_cast<int32_t*>(nullptr), static_cast<float*>(nullptr));
  if (le != cudaSuccess) return fail(FT_ERR_CUDA, "route logits: %s", cudaGetErrorString(le));
  *logits_out = logits;
  *stride_out = route_row_stride(T);
  return launch_check("route logits");
}

}  // namespace ft

extern "C" {

size_t ft_moe_route_workspace(int32_t T, int32_t E, int32_t H) {
  if (T <= 0 || E <= 0 || H <= 0) return 0;
  // the arrival counter, the logits, then (long prompts on the tensor cores)
  // the router's three bf16 terms
  return ft::kRouteCounterBytes + ft::route_logits_bytes(T, E) + ft::route_mma_split_bytes(T, E, H);
}

ft_status ft_moe_route(const uint16_t* x, int32_t T, int32_t H, const float* w_router, int32_t E,
                       int32_t k, int32_t renorm, int32_t* topk_ids, float* topk_w, void* ws,
                       size_t ws_bytes, void* stream) {
  FT_REQUIRE(T >= 0, "route: T < 0");
  FT_REQUIRE(E >= 1 && E <= 4096, "route: E %d outside [1, 4096]", E);
  FT_REQUIRE(k >= 1 && k <= E && k <= ft::kRouteMaxK, "route: k %d outside [1, min(E, 32)]", k);
  FT_REQUIRE(H >= 8 && H % 8 == 0, "route: H %d must be a positive multiple of 8", H);
  if (T == 0) return FT_OK;
  FT_REQUIRE(x && w_router && topk_ids && topk_w && ws, "route: NULL pointer");
  FT_REQUIRE(ws_bytes >= ft_moe_route_workspace(T, E, H), "route: workspace %zu < %zu", ws_bytes,
             ft_moe_route_workspace(T, E, H));
  FT_REQUIRE(reinterpret_cast<uintptr_t>(x) % 16 == 0 && reinterpret_cast<uintptr_t>(w_router) % 16 == 0,
             "route: x and w_router must be 16-byte aligned");
  cudaStream_t s = ft::as_stream(stream);
  float* logits = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + ft::kRouteCounterBytes);
  if (T <= ft::kGemvMaxT)  // logits and top-k in one kernel
    return ft::launch_rows(x, T, H, w_router, E, k, renorm, topk_ids, topk_w, ws, s);
  ft_status st;
  int slices = 1;
  float* partx = nullptr;
  if (ft::route_mma_fits(T, E, H)) {  // tensor cores: the split terms and partial logits follow the logits
    void* extra = static_cast<uint8_t*>(ws) + ft::kRouteCounterBytes + ft::route_logits_bytes(T, E);
    st = ft::route_mma_logits(x, T, H, w_router, E, logits, extra, &slices, s);
    partx = ft::route_mma_partials(extra, E, H);
  } else {
    FT_REQUIRE(H % ft::kTK == 0, "route: H %d must be a multiple of 32 for T > 16", H);
    dim3 grid((E + ft::kTN - 1) / ft::kTN, (T + ft::kTM - 1) / ft::kTM);
    ft::route_tiled_kernel<<<grid, 256, 0, s>>>(x, T, H, w_router, E, logits);
    st = ft::launch_check("route logits");
  }
  if (st != FT_OK) return st;
  // the top-k grid starts while the logits grid drains (programmatic launch)
  // one warp per token, each with E logits in shared memory (<= 32 KB per CTA)
  const int warps = E <= 1024 ? 8 : 2;
  const int nx = slices - 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((T + warps - 1) / warps);
  cfg.blockDim = dim3(32 * warps);
  cfg.dynamicSmemBytes = static_cast<size_t>(warps) * E * sizeof(float);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const float* px = partx;
  cudaError_t e = cudaLaunchKernelEx(&cfg, ft::route_topk_kernel, logits, T, E, k, renorm, topk_ids, topk_w, px, nx);
  if (e != cudaSuccess) return ft::fail(FT_ERR_CUDA, "route topk: %s", cudaGetErrorString(e));
  return ft::launch_check("route topk");
}

}  // extern "C"
