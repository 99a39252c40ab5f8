// ft_common.cuh -- shared helpers of the CUDA library (host error plumbing,
// device status words, bf16/f16 bit helpers, block-wide scans, the expert
// block layout).  Nothing here is shared with the CPU oracle.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ft_moe.h"

namespace ft {

// ------------------------------------------------------------------ host ---
void set_error(const char* fmt, ...);
ft_status fail(ft_status code, const char* fmt, ...);
ft_status launch_check(const char* what);

struct Layout {
  uint64_t off[6];  // gate, up, down, gate_scale, up_scale, down_scale
  uint64_t total;
  int32_t block;    // K elements per scale: group (int4) or 16 (NVFP4)
};
// Fills L; false for an unsupported (fmt, H, I, group).
bool layout(int32_t fmt, int32_t H, int32_t I, int32_t group, Layout* L);

// Host-side validation of a bank descriptor against an expected shape.
ft_status check_bank(const ft_bank* b, const char* name, Layout* L);

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// The current device's SM count, and its per-block shared-memory limit
// (opt-in), each looked up once per device.
int device_sm_count();
int device_smem_optin();
// The router logits of long prompts on the tensor cores (route_mma.cu): the
// shapes it takes, the workspace its split router terms and partial logits
// need, the launch (partial logits per hidden slice; *slices of them).
bool route_mma_fits(int T, int E, int H);
size_t route_mma_split_bytes(int T, int E, int H);
float* route_mma_partials(void* extra, int E, int H);
ft_status route_mma_logits(const uint16_t* x, int T, int H, const float* W, int E, float* logits, void* extra,
                           int* slices, cudaStream_t s);
// The router logits alone for T <= 16 (route.cu), in the workspace of
// ft_moe_route: *logits_out = [E][*stride_out] floats, token t's logit of
// expert e at e * stride + t.
ft_status route_rows_logits(const uint16_t* x, int T, int H, const float* W, int E, void* ws, cudaStream_t s,
                            const float** logits_out, int* stride_out);

// Raise a kernel's dynamic shared memory limit to `bytes` on the current
// device, once per (kernel, device); FT_ERR_CUDA if the device refuses.
ft_status ensure_dyn_smem(const void* kernel, int bytes, const char* what);

#define FT_REQUIRE(cond, ...)                                   \
  do {                                                          \
    if (!(cond)) return ::ft::fail(FT_ERR_INVALID, __VA_ARGS__); \
  } while (0)

// ---------------------------------------------------------------- device ---
__device__ __forceinline__ void record_status(int32_t* st, int32_t code) {
  if (st != nullptr) atomicCAS(st, 0, code);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16_val(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// Round-to-nearest-even fp32 -> bf16 bits (NaN kept quiet).
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return static_cast<uint16_t>((u >> 16) | 0x40);
  u += 0x7fffu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

// Power-of-two factor that keeps |v| * factor below 2^16 in f16 (1 when it
// already is): exact scaling, undone by the caller with 1/factor.
__device__ __forceinline__ float f16_prescale(float amax) {
  if (!(amax < 32768.f)) {
    if (!isfinite(amax)) return 1.f;
    return ldexpf(1.f, 14 - ilogbf(amax));
  }
  return 1.f;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Exclusive block-wide scan of one int per thread.  `scratch` holds at least
// 33 ints of shared memory; every thread of the block must call it.
__device__ __forceinline__ int block_excl_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int w = (lane < nw) ? scratch[lane] : 0;
    int s = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    scratch[lane] = s - w;
    if (lane == 31) scratch[32] = s;
  }
  __syncthreads();
  int res = scratch[wid] + x - v;
  *total = scratch[32];
  __syncthreads();
  return res;
}

}  // namespace ft
