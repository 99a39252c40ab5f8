// ft_dequant.cuh -- the decode experts' dequantise-and-dot arithmetic, shared
// by the pair-major kernels (decode2.cu) and the fused decode layer
// (layer.cu): 4-bit codes to f16 through the hardware FP8/FP4 converts,
// exact f16 products accumulated in fp32, activations packed as f16 chunks
// with an exact power-of-two prescale.
//
// An int4 code q in 0..15 is also the E4M3 code of q * 2^-9 exactly (the
// subnormals and the first binade of E4M3 are evenly spaced), so
// cvt.rn.f16x2.e4m3x2 turns two nibbles spread to bytes into f16 q * 2^-9, and
// sum (q - 8) a = 512 * sum (q 2^-9) a - 8 * sum a, with sum a per 32-element
// chunk precomputed.  NVFP4 codes go through cvt.rn.f16x2.e2m1x2.
//
// Sources: "SSD 가중치층으로 35B MoE를 ..." (onedev.kr), "How it works";
// "NVMe에서 전문가(experts)를 ... 133GB MoE" (molayo1419.me), step 4.
#pragma once

#include <cuda_fp16.h>

#include "ft_decode.cuh"

namespace ft {
namespace {

constexpr int kChunkBytes = 80;   // 32 f16 values + 16 B pad (conflict-free 16-byte reads)

// ----------------------------------------------------------- conversions ---
__device__ __forceinline__ uint32_t cvt_e4m3x2(uint32_t two_bytes) {
  uint32_t h;
  const unsigned short b = static_cast<unsigned short>(two_bytes);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(b));
  return h;
}

// 8 int4 codes of a word -> f16 q * 2^-9 in the pairs (c0,c2) (c4,c6) (c1,c3) (c5,c7).
__device__ __forceinline__ void int4x8(uint32_t v, uint32_t h[4]) {
  const uint32_t lo = v & 0x0F0F0F0Fu, hi = (v >> 4) & 0x0F0F0F0Fu;
  h[0] = cvt_e4m3x2(lo);
  h[1] = cvt_e4m3x2(lo >> 16);
  h[2] = cvt_e4m3x2(hi);
  h[3] = cvt_e4m3x2(hi >> 16);
}

// 8 E2M1 codes of a word -> f16 in the pairs (c0,c1) (c2,c3) (c4,c5) (c6,c7).
__device__ __forceinline__ void e2m1x8(uint32_t v, uint32_t h[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(v));
}

// a0 += w.lo * x.lo, a1 += w.hi * x.hi in fp32 (f16 operands, exact products).
__device__ __forceinline__ void fma2_f16(float& a0, float& a1, uint32_t w, uint32_t x) {
  asm("{\n .reg .b16 wl, wh, xl, xh;\n mov.b32 {wl, wh}, %2;\n mov.b32 {xl, xh}, %3;\n"
      " fma.rn.f32.f16 %0, wl, xl, %0;\n fma.rn.f32.f16 %1, wh, xh, %1;\n}"
      : "+f"(a0), "+f"(a1)
      : "r"(w), "r"(x));
}

// The scale word of one chunk: int4 -> its fp16 group scale; NVFP4 -> its two
// E4M3 block scales (16 elements each) in the low 16 bits.
template <int FMT>
__device__ __forceinline__ uint32_t load_scale(const uint8_t* srow, int c, int gshift) {
  if constexpr (FMT == FT_INT4)
    return __ldg(reinterpret_cast<const unsigned short*>(srow) + (c >> gshift));
  else
    return __ldg(reinterpret_cast<const unsigned short*>(srow) + c);
}

// One 32-element chunk: 16 bytes of codes, the chunk's scale word, 16 f16x2
// activation words in the format's order and (int4) the sum of those values.
template <int FMT>
__device__ __forceinline__ float chunk_dot(const uint4 w, uint32_t sc, const uint32_t* xa, float asum) {
  const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
  if constexpr (FMT == FT_INT4) {
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t h[4];
      int4x8(wv[j], h);
      fma2_f16(s0, s1, h[0], xa[4 * j + 0]);
      fma2_f16(s2, s3, h[1], xa[4 * j + 1]);
      fma2_f16(s0, s1, h[2], xa[4 * j + 2]);
      fma2_f16(s2, s3, h[3], xa[4 * j + 3]);
    }
    const float s = __half2float(__ushort_as_half(static_cast<unsigned short>(sc)));
    return s * fmaf(512.f, (s0 + s1) + (s2 + s3), -8.f * asum);
  } else {
    float p0 = 0.f, p1 = 0.f, q0 = 0.f, q1 = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t h[4];
      e2m1x8(wv[j], h);
      float& a0 = (j < 2) ? p0 : q0;
      float& a1 = (j < 2) ? p1 : q1;
      fma2_f16(a0, a1, h[0], xa[4 * j + 0]);
      fma2_f16(a0, a1, h[1], xa[4 * j + 1]);
      fma2_f16(a0, a1, h[2], xa[4 * j + 2]);
      fma2_f16(a0, a1, h[3], xa[4 * j + 3]);
    }
    const uint32_t h2 = cvt_e4m3x2(sc);
    const float2 s = __half22float2(*reinterpret_cast<const __half2*>(&h2));
    return fmaf(p0 + p1, s.x, (q0 + q1) * s.y);
  }
}

// Element i of a chunk: from 32 fp32 values or from 16 bf16x2 words.
__device__ __forceinline__ float elem(const float* v, int i) { return v[i]; }
__device__ __forceinline__ float elem(const uint32_t* b, int i) {
  return (i & 1) ? bf16_hi(b[i >> 1]) : bf16_lo(b[i >> 1]);
}

// 32 values (times `mul`) -> 16 f16x2 words in the format's order; returns
// the sum of the f16 values as used.
template <int FMT, typename V>
__device__ __forceinline__ float pack32(const V* v, float mul, uint32_t* out) {
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      // int4 pairs per 8 codes: (0,2) (4,6) (1,3) (5,7); NVFP4: (0,1) (2,3) (4,5) (6,7)
      const int lo = (FMT == FT_INT4) ? 8 * j + ((m & 1) ? 4 : 0) + ((m & 2) ? 1 : 0) : 8 * j + 2 * m;
      const int hi = (FMT == FT_INT4) ? lo + 2 : lo + 1;
      const __half a = __float2half_rn(elem(v, lo) * mul), b = __float2half_rn(elem(v, hi) * mul);
      s += __half2float(a) + __half2float(b);
      out[4 * j + m] = static_cast<uint32_t>(__half_as_ushort(a)) | (static_cast<uint32_t>(__half_as_ushort(b)) << 16);
    }
  }
  return s;
}

__device__ __forceinline__ float warp_max(float m) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  return m;
}

// One warp stages pair p's intermediate row (I fp32 values from the gate/up
// grid) in shared memory as slot j: f16 chunks in the format's order at
// hsm + (j*IC + c)*kChunkBytes, their sums in hsum[j*IC + c], with an exact
// power-of-two prescale from the row's largest magnitude, which s_wq[j]
// (the pair's combine weight) absorbs.
template <int FMT>
__device__ __forceinline__ void stage_h(const DecArgs& a, int p, int j, uint8_t* hsm, float* hsum, float* s_wq) {
  const int lane = threadIdx.x & 31;
  const int I = a.I, IC = I / 32;
  const float* hp = a.h + static_cast<size_t>(p) * I;
  float v[32];
  float m = 0.f;
  if (lane < IC) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 f = *reinterpret_cast<const float4*>(hp + 32 * lane + 4 * q);
      v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) m = fmaxf(m, fabsf(v[i]));
  }
  for (int c = lane + 32; c < IC; c += 32) {  // I > 1024: a first pass for the max
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 f = *reinterpret_cast<const float4*>(hp + 32 * c + 4 * q);
      m = fmaxf(m, fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w))));
    }
  }
  const float mul = f16_prescale(warp_max(m));
  if (lane == 0) s_wq[j] /= mul;
  uint32_t o[16];
  if (lane < IC) {
    hsum[j * IC + lane] = pack32<FMT>(v, mul, o);
    uint8_t* dst = hsm + static_cast<size_t>(j * IC + lane) * kChunkBytes;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<uint4*>(dst + 16 * q) = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
  }
  for (int c = lane + 32; c < IC; c += 32) {  // the second read hits L1
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 f = *reinterpret_cast<const float4*>(hp + 32 * c + 4 * q);
      v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
    }
    hsum[j * IC + c] = pack32<FMT>(v, mul, o);
    uint8_t* dst = hsm + static_cast<size_t>(j * IC + c) * kChunkBytes;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<uint4*>(dst + 16 * q) = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
  }
}

}  // namespace
}  // namespace ft
