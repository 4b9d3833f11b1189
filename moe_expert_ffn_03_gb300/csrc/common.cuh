// Device helpers shared by the kernels of libmoeffn (sm_103a only).
//
// MX quantization: one power-of-two scale per 32 consecutive values and 8-bit
// E4M3 elements (page "Efficient MoE Training for Biological Foundation
// Models", section "MoE训练的瓶颈与TE的对应能力"); the scale rule and rounding
// are the readings stated in include/moe_ffn.h.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/moe_ffn.h"

namespace moe {

// ---- device error word (workspace offset 0): int32 code, int32 site ----------
enum ErrSite : int {
  SITE_ROUTE = 100,
  SITE_PERMUTE = 200,
  SITE_QUANT = 300,
  SITE_COMBINE = 400,
  SITE_GEMM_PRODUCER = 500,
  SITE_GEMM_MMA = 510,
  SITE_GEMM_MMA_ACC = 520,
  SITE_GEMM_EPILOGUE = 530,
  SITE_GEMM_DRAIN = 540,
};

__device__ __forceinline__ void report_error(int* err, int code, int site) {
  if (err != nullptr && atomicCAS(err, 0, code) == 0) atomicExch(err + 1, site);
}

// ---- MX scale layout ----------------------------------------------------------
// Scale byte of (row r, 32-block b) of a [rows][K] MX tensor in the MMA tile
// layout: 128x4 scale atoms of 512 bytes, atom (r/128, b/4) at
// ((r/128)*(K/128) + b/4)*512, inside it byte (r%32)*16 + ((r/32)%4)*4 + b%4.
__host__ __device__ __forceinline__ size_t sf_offset(size_t r, size_t b, size_t K) {
  return (((r >> 7) * (K >> 7) + (b >> 2)) << 9) + ((r & 31) << 4) + (((r >> 5) & 3) << 2) + (b & 3);
}

// ---- MX quantization of one block of 32 values -----------------------------------
// amax over |x| taken on float bit patterns (|x| bits order like the values,
// and NaN/Inf patterns sit above every finite one).
__device__ __forceinline__ uint32_t abs_bits(float v) { return __float_as_uint(v) & 0x7FFFFFFFu; }

// Scale code c = e + 127 for the smallest e with amax <= 448*2^e, clamped to
// e >= -127 (448 = 1.75*2^8: e = floor(log2 amax) - 8, plus one when the
// significand exceeds 1.75); 255 for a non-finite block.
__device__ __forceinline__ uint32_t mx_scale_code(uint32_t amax_bits) {
  const uint32_t ef = amax_bits >> 23;
  if (ef == 255u) return 255u;
  const int c = int(ef) - 8 + int((amax_bits & 0x7FFFFFu) > 0x600000u);
  return c < 0 ? 0u : uint32_t(c);
}

// 2^(127 - c) as a float (c <= 254).
__device__ __forceinline__ float mx_inv_scale(uint32_t c) { return __uint_as_float((254u - c) << 23); }

// Two floats -> two E4M3 codes (round to nearest even, saturate to +-448);
// `lo` lands in the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Quantize 32 floats (already loaded) to 32 codes packed in 8 words; returns the scale code.
__device__ __forceinline__ uint32_t mx_quant32(const float* v, uint32_t* q) {
  uint32_t amax = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = max(amax, abs_bits(v[i]));
  const uint32_t c = mx_scale_code(amax);
  if (c == 255u) {
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = 0x7F7F7F7Fu;
    return c;
  }
  const float m = mx_inv_scale(c);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t a = cvt_e4m3x2(v[4 * i + 0] * m, v[4 * i + 1] * m);
    const uint32_t b = cvt_e4m3x2(v[4 * i + 2] * m, v[4 * i + 3] * m);
    q[i] = a | (b << 16);
  }
  return c;
}

// One value quantized with a known scale code (for blocks reduced across lanes).
__device__ __forceinline__ uint32_t mx_quant1(float v, uint32_t c) {
  if (c == 255u) return 0x7Fu;
  return cvt_e4m3x2(v * mx_inv_scale(c), 0.0f) & 0xFFu;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void load_bf16x32(const __nv_bfloat16* p, float (&v)[32]) {
  const uint4* p4 = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 w = p4[i];
    v[8 * i + 0] = bf16_lo(w.x); v[8 * i + 1] = bf16_hi(w.x);
    v[8 * i + 2] = bf16_lo(w.y); v[8 * i + 3] = bf16_hi(w.y);
    v[8 * i + 4] = bf16_lo(w.z); v[8 * i + 5] = bf16_hi(w.z);
    v[8 * i + 6] = bf16_lo(w.w); v[8 * i + 7] = bf16_hi(w.w);
  }
}

__device__ __forceinline__ void store_codes32(uint8_t* p, const uint32_t (&q)[8]) {
  uint4* p4 = reinterpret_cast<uint4*>(p);
  p4[0] = make_uint4(q[0], q[1], q[2], q[3]);
  p4[1] = make_uint4(q[4], q[5], q[6], q[7]);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: every bounded wait gives up after this

}  // namespace moe
