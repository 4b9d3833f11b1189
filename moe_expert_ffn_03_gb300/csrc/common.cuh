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
  SITE_ROUTER_DW = 600,
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

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// mx_quant32 for 32 bf16 values packed two per word (value 2i in the low half
// of w[i]).  The block max is taken on the 16-bit |x| patterns of both halves
// at once; codes and scale are bit-identical to mx_quant32 on the same values.
__device__ __forceinline__ uint32_t mx_quant32_bf16(const uint32_t* w, uint32_t* q) {
  uint32_t mx = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) mx = __vmaxu2(mx, w[i] & 0x7FFF7FFFu);
  const uint32_t c = mx_scale_code(max(mx << 16, mx & 0xFFFF0000u));
  if (c == 255u) {
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = 0x7F7F7F7Fu;
    return c;
  }
  const float m = mx_inv_scale(c);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t a = cvt_e4m3x2(bf16_lo(w[2 * i]) * m, bf16_hi(w[2 * i]) * m);
    const uint32_t b = cvt_e4m3x2(bf16_lo(w[2 * i + 1]) * m, bf16_hi(w[2 * i + 1]) * m);
    q[i] = a | (b << 16);
  }
  return c;
}

// Two adjacent columns of 32 rows at once: word i of the column pair is
// p[i * stride] (low half = left column).  Codes of the left column go to
// q_lo, of the right one to q_hi; returns both scale codes (left in bits 0-7,
// right in bits 8-15).  Bit-identical to mx_quant32 on each column.
__device__ __forceinline__ uint32_t mx_quant32_bf16_colpair(const uint32_t* p, int stride, uint32_t* q_lo,
                                                            uint32_t* q_hi) {
  uint32_t mx = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) mx = __vmaxu2(mx, p[i * stride] & 0x7FFF7FFFu);
  const uint32_t c_lo = mx_scale_code(mx << 16), c_hi = mx_scale_code(mx & 0xFFFF0000u);
  const float m_lo = mx_inv_scale(c_lo == 255u ? 0u : c_lo), m_hi = mx_inv_scale(c_hi == 255u ? 0u : c_hi);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t w0 = p[(4 * i + 0) * stride], w1 = p[(4 * i + 1) * stride];
    const uint32_t w2 = p[(4 * i + 2) * stride], w3 = p[(4 * i + 3) * stride];
    q_lo[i] = cvt_e4m3x2(bf16_lo(w0) * m_lo, bf16_lo(w1) * m_lo) |
              (cvt_e4m3x2(bf16_lo(w2) * m_lo, bf16_lo(w3) * m_lo) << 16);
    q_hi[i] = cvt_e4m3x2(bf16_hi(w0) * m_hi, bf16_hi(w1) * m_hi) |
              (cvt_e4m3x2(bf16_hi(w2) * m_hi, bf16_hi(w3) * m_hi) << 16);
  }
  if (c_lo == 255u) {
#pragma unroll
    for (int i = 0; i < 8; ++i) q_lo[i] = 0x7F7F7F7Fu;
  }
  if (c_hi == 255u) {
#pragma unroll
    for (int i = 0; i < 8; ++i) q_hi[i] = 0x7F7F7F7Fu;
  }
  return c_lo | (c_hi << 8);
}

// Per-tensor FP8 scale of a tensor with max |v| = amax (float bits):
// s = 448 / amax rounded to float32 (IEEE division), 1 for an all-zero tensor.
__device__ __forceinline__ float t8_scale(uint32_t amax_bits) {
  const float a = __uint_as_float(amax_bits);
  return a == 0.0f ? 1.0f : __fdiv_rn(448.0f, a);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// 32 bytes at p from 8 words in one 256-bit store (p 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t* q) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(q[0]), "r"(q[1]), "r"(q[2]),
               "r"(q[3]), "r"(q[4]), "r"(q[5]), "r"(q[6]), "r"(q[7]) : "memory");
}
// 32 bytes at p into 8 words in one 256-bit load (p 32-byte aligned).
__device__ __forceinline__ void ld_global_v8(const void* p, uint32_t* q) {
  asm volatile("ld.global.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3]), "=r"(q[4]), "=r"(q[5]), "=r"(q[6]), "=r"(q[7])
               : "l"(p));
}
__host__ __device__ __forceinline__ bool aligned32(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 31u) == 0;
}

// 32 codes at p (32-byte offset inside its tensor): one 256-bit store when the tensor's base
// is 32-byte aligned (v8), else two 16-byte stores.
__device__ __forceinline__ void store_codes32(uint8_t* p, const uint32_t (&q)[8], bool v8) {
  if (v8) {
    st_global_v8(p, q);
    return;
  }
  uint4* p4 = reinterpret_cast<uint4*>(p);
  p4[0] = make_uint4(q[0], q[1], q[2], q[3]);
  p4[1] = make_uint4(q[4], q[5], q[6], q[7]);
}

// 16-byte global -> shared copy that bypasses registers (cp.async, L1 not
// allocated).  valid == false writes 16 zero bytes and reads nothing.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(valid ? 16 : 0)
               : "memory");
}

// Waits for all of this thread's cp.async copies (a hardware wait, not a spin loop).
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: every bounded wait gives up after this

// ---- programmatic dependent launch --------------------------------------------------
// A kernel launched with programmatic stream serialization (launch_pdl) may start while
// the kernel before it in the stream is still running.  pdl_wait() returns once that
// kernel has completed and its memory operations are visible; every such kernel calls
// it before its first access to global memory that an earlier kernel may write or read.
// pdl_launch_dependents() lets the next kernel's CTAs be scheduled once every CTA of
// this one has called it or exited.  Both are no-ops in a kernel launched without the
// attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- mbarriers (this CTA's shared memory) ----------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

}  // namespace moe
