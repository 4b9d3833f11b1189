// bf16 transposes for the bf16 training path (page "Efficient MoE Training for
// Biological Foundation Models", section "运行要求、基准与验证步骤": the recipe
// trains in BF16 or in MXFP8).  Every GEMM of the engine takes both operands
// K-major; the backward GEMMs contract over H (dgrad of the down projection),
// over 2I (dgrad of gate_up) and over each expert's tokens (weight gradients),
// so the weights and the permuted activations are also needed transposed.  In
// the MXFP8 path the same copies come out of the quantizers along the other
// axis; here they are plain bf16.
//
// One CTA per 128x128 tile of src[batch]: the tile is staged in shared memory
// with cp.async (rows gathered through src_map when given, -1 -> zero row),
// then every thread writes two transposed rows of 32 values (64 contiguous
// bytes each).  HBM-bound: 2 B read and 2 B written per element.  The byte
// transpose below serves the per-tensor FP8 path the same way.
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int TT = 128;                 // tile edge
constexpr int TP = TT + 8;              // bf16 per shared row (16 B pad)

// S: StackedSrc (one tensor of batch matrices; with src_map its matrix 0 is the gather
// source) or ExpertSrc (one pointer per matrix: each expert's own weight tensor).
template <typename S>
__global__ void __launch_bounds__(256, 6) transpose_bf16_kernel(
    S src, const int* __restrict__ src_map, int64_t n_src_rows, int rows, int cols,
    const int* __restrict__ split_sizes, int E, __nv_bfloat16* __restrict__ out, int* err) {
  __shared__ __align__(16) __nv_bfloat16 tile[TT * TP];
  __shared__ int s_rows_used;
  const int row0 = blockIdx.x * TT;
  const int col0 = blockIdx.y * TT;
  const int64_t batch = blockIdx.z;
  const int c16 = threadIdx.x & 15, rbase = threadIdx.x >> 4;
  int sr[TT / 16];
  if (src_map != nullptr) {
#pragma unroll
    for (int it = 0; it < TT / 16; ++it) sr[it] = src_map[row0 + rbase + 16 * it];
  }
  if (split_sizes != nullptr) {
    if (threadIdx.x < 32) {
      int acc = 0;
      for (int e = threadIdx.x; e < E; e += 32) acc += (split_sizes[e] + 127) & ~127;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
      if (threadIdx.x == 0) s_rows_used = acc;
    }
    __syncthreads();
    if (row0 >= s_rows_used) return;                  // rows past the padded segments
  }
  const __nv_bfloat16* mat = src.mat(src_map != nullptr ? 0 : batch);
#pragma unroll
  for (int it = 0; it < TT / 16; ++it) {
    const int r = rbase + 16 * it;
    int64_t s;
    if (src_map != nullptr) {
      s = sr[it];
      if (s >= n_src_rows) {
        report_error(err, MOE_ERR_DEVICE_BOUNDS, SITE_QUANT + 20);
        s = -1;
      }
    } else {
      s = row0 + r;
    }
    const bool valid = s >= 0;
    cp_async16(&tile[r * TP + c16 * 8], valid ? static_cast<const void*>(mat + s * cols + col0 + c16 * 8) : mat,
               valid);
  }
  cp_async_wait_all();
  __syncthreads();
  // task: columns (c, c+1) x rows rb*32 .. rb*32+31 -- one per thread
  const int c = 2 * (threadIdx.x & 63), rb = threadIdx.x >> 6;
  const uint32_t* p = reinterpret_cast<const uint32_t*>(&tile[(rb * 32) * TP + c]);
  uint32_t lo[16], hi[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t w0 = p[(2 * i) * (TP / 2)], w1 = p[(2 * i + 1) * (TP / 2)];
    lo[i] = __byte_perm(w0, w1, 0x5410);               // column c: rows 2i, 2i+1
    hi[i] = __byte_perm(w0, w1, 0x7632);               // column c+1
  }
  const int64_t orow = batch * cols + col0 + c;        // row of the transposed tensor
  uint4* d0 = reinterpret_cast<uint4*>(out + orow * rows + row0 + rb * 32);
  uint4* d1 = reinterpret_cast<uint4*>(out + (orow + 1) * rows + row0 + rb * 32);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    d0[q] = make_uint4(lo[4 * q], lo[4 * q + 1], lo[4 * q + 2], lo[4 * q + 3]);
    d1[q] = make_uint4(hi[4 * q], hi[4 * q + 1], hi[4 * q + 2], hi[4 * q + 3]);
  }
}

// Byte transpose of E4M3 codes (the per-tensor FP8 path: a scale per tensor does not
// depend on the axis, so the along-token operands are the row codes transposed).
// Tile 128x128 bytes; thread (column c, half h) reads 64 rows of column c from
// shared memory and writes them as 64 contiguous bytes of transposed row c.
__global__ void __launch_bounds__(256) transpose_u8_kernel(const uint8_t* __restrict__ src, int rows, int cols,
                                                           const int* __restrict__ split_sizes, int E,
                                                           uint8_t* __restrict__ out) {
  __shared__ __align__(16) uint8_t tile[TT * (TT + 16)];
  __shared__ int s_rows_used;
  const int row0 = blockIdx.x * TT;
  const int col0 = blockIdx.y * TT;
  const int64_t batch = blockIdx.z;
  if (split_sizes != nullptr) {
    if (threadIdx.x < 32) {
      int acc = 0;
      for (int e = threadIdx.x; e < E; e += 32) acc += (split_sizes[e] + 127) & ~127;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
      if (threadIdx.x == 0) s_rows_used = acc;
    }
    __syncthreads();
    if (row0 >= s_rows_used) return;
  }
  constexpr int P = TT + 16;                           // bytes per shared row
  const uint8_t* base = src + (batch * rows + row0) * int64_t(cols) + col0;
#pragma unroll
  for (int it = 0; it < 4; ++it) {                     // 128 rows x 8 chunks of 16 B
    const int i = threadIdx.x + 256 * it;
    const int r = i >> 3, c16 = i & 7;
    cp_async16(&tile[r * P + c16 * 16], base + int64_t(r) * cols + c16 * 16, true);
  }
  cp_async_wait_all();
  __syncthreads();
  const int c = threadIdx.x & 127, h = threadIdx.x >> 7;
  uint32_t w[16];
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const int r = 64 * h + 4 * q;
    w[q] = uint32_t(tile[r * P + c]) | (uint32_t(tile[(r + 1) * P + c]) << 8) |
           (uint32_t(tile[(r + 2) * P + c]) << 16) | (uint32_t(tile[(r + 3) * P + c]) << 24);
  }
  uint4* d = reinterpret_cast<uint4*>(out + (batch * cols + col0 + c) * int64_t(rows) + row0 + 64 * h);
#pragma unroll
  for (int q = 0; q < 4; ++q) d[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
}

}  // namespace

cudaError_t launch_transpose_u8(const uint8_t* src, int batch, int rows, int cols, const int* split_sizes, int E,
                                uint8_t* out, cudaStream_t st) {
  dim3 grid(rows / TT, cols / TT, batch);
  transpose_u8_kernel<<<grid, 256, 0, st>>>(src, rows, cols, split_sizes, E, out);
  return cudaGetLastError();
}

cudaError_t launch_transpose_bf16(const void* src, const int* src_map, int64_t n_src_rows, int batch, int rows,
                                  int cols, const int* split_sizes, int E, void* out, int* err, cudaStream_t st) {
  dim3 grid(rows / TT, cols / TT, batch);
  const StackedSrc s{static_cast<const __nv_bfloat16*>(src), int64_t(rows) * cols};
  transpose_bf16_kernel<<<grid, 256, 0, st>>>(s, src_map, n_src_rows, rows, cols, split_sizes, E,
                                              static_cast<__nv_bfloat16*>(out), err);
  return cudaGetLastError();
}

cudaError_t launch_transpose_bf16_experts(const ExpertSrc& src, int batch, int rows, int cols, void* out,
                                          cudaStream_t st) {
  dim3 grid(rows / TT, cols / TT, batch);
  transpose_bf16_kernel<<<grid, 256, 0, st>>>(src, nullptr, 0, rows, cols, nullptr, 0,
                                              static_cast<__nv_bfloat16*>(out), nullptr);
  return cudaGetLastError();
}

}  // namespace moe
