// MXFP8 quantization kernels: bf16 -> E4M3 codes + power-of-two scales, one
// scale per 32 consecutive values along the consuming GEMM's K axis (page
// "Efficient MoE Training for Biological Foundation Models", sections
// "MoE训练的瓶颈与TE的对应能力" and "MXFP8与融合MLP").  All kernels here are
// HBM-bound: each bf16 element is read once and its code written once (k
// times for the scattered token rows).
#include "kernels.cuh"

namespace moe {

// ---------------------------------------------------------------------------------
// Rowwise: blocks of 32 along the contiguous axis.  One warp per source row;
// lane l takes blocks l, l+32, ... so a warp reads 2 KB contiguous per step.
// SCATTER: source row s (a token) is written to the k rows row_of[s*k + j]
// (the permuted rows); otherwise to row s itself.
// ---------------------------------------------------------------------------------
template <bool SCATTER>
__global__ void __launch_bounds__(256) quant_rowwise_kernel(
    const __nv_bfloat16* __restrict__ src, int64_t n_rows, int cols,
    const int* __restrict__ row_of, int k, int64_t cap,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, int* err) {
  const int lane = threadIdx.x & 31;
  const int64_t s = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (s >= n_rows) return;
  const int nblk = cols >> 5;
  int64_t dst[8];
  int nd = 1;
  if (SCATTER) {
    nd = k;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k) {
        const int r = row_of[s * k + j];
        if (r < 0 || r >= cap) {
          report_error(err, MOE_ERR_DEVICE_BOUNDS, SITE_QUANT + 1);
          return;
        }
        dst[j] = r;
      }
    }
  } else {
    dst[0] = s;
  }
  for (int b = lane; b < nblk; b += 32) {
    float v[32];
    load_bf16x32(src + s * cols + (int64_t)b * 32, v);
    uint32_t q[8];
    const uint32_t c = mx_quant32(v, q);
    for (int j = 0; j < nd; ++j) {
      store_codes32(codes + dst[j] * cols + (int64_t)b * 32, q);
      scales[sf_offset(dst[j], b, cols)] = uint8_t(c);
    }
  }
}

// Zero codes and zero scale codes for the padding rows of every expert segment
// (rows split_sizes[e] .. roundup(split_sizes[e],128)-1 of segment e).
__global__ void __launch_bounds__(256) fill_pad_rows_kernel(
    const int* __restrict__ split_sizes, int E, int cols,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  __shared__ int seg_start;
  const int e = blockIdx.x;
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int i = 0; i < e; ++i) acc += (split_sizes[i] + 127) & ~127;
    seg_start = acc;
  }
  __syncthreads();
  const int m = split_sizes[e];
  const int npad = ((m + 127) & ~127) - m;
  const int64_t r0 = int64_t(seg_start) + m;
  const int vec_per_row = cols >> 4;                 // uint4 per row
  for (int64_t i = threadIdx.x; i < int64_t(npad) * vec_per_row; i += blockDim.x) {
    const int64_t r = r0 + i / vec_per_row;
    const int c = int(i % vec_per_row);
    reinterpret_cast<uint4*>(codes + r * cols)[c] = make_uint4(0, 0, 0, 0);
  }
  const int nblk = cols >> 5;
  for (int64_t i = threadIdx.x; i < int64_t(npad) * nblk; i += blockDim.x) {
    const int64_t r = r0 + i / nblk;
    scales[sf_offset(r, i % nblk, cols)] = 0;
  }
}

// ---------------------------------------------------------------------------------
// Colwise: blocks of 32 along the row axis, output transposed.  One CTA per
// 128x128 tile: the tile is staged in shared memory with 16-byte loads, then
// thread (column c, row block rb) reduces 32 rows, quantizes them and writes
// 32 contiguous codes of the transposed row c.  The tile's scales form exactly
// one 512-byte atom of the transposed tensor.
//   src row of tile row r: src_map ? src_map[r] (-1 -> zero row) : batch*rows + r
//   split_sizes (optional): rows at or past the padded total are skipped.
// ---------------------------------------------------------------------------------
constexpr int QC_TILE = 128;
constexpr int QC_PITCH = QC_TILE + 8;                // bf16 per smem row (16 B pad)

__global__ void __launch_bounds__(256) quant_colwise_kernel(
    const __nv_bfloat16* __restrict__ src, const int* __restrict__ src_map, int64_t n_src_rows,
    int rows, int cols, const int* __restrict__ split_sizes, int E,
    uint8_t* __restrict__ codes_t, uint8_t* __restrict__ scales_t, int* err) {
  __shared__ __align__(16) __nv_bfloat16 tile[QC_TILE * QC_PITCH];
  __shared__ __align__(16) uint8_t sc_atom[512];
  __shared__ int s_rows_used;
  const int row0 = blockIdx.x * QC_TILE;
  const int col0 = blockIdx.y * QC_TILE;
  const int64_t batch = blockIdx.z;
  if (split_sizes != nullptr) {
    if (threadIdx.x == 0) {
      int acc = 0;
      for (int e = 0; e < E; ++e) acc += (split_sizes[e] + 127) & ~127;
      s_rows_used = acc;
    }
    __syncthreads();
    if (row0 >= s_rows_used) return;
  }
  // stage: 128 rows x 256 bytes = 16 uint4 per row; all eight loads of a thread in flight together
#pragma unroll
  for (int it = 0; it < QC_TILE * 16 / 256; ++it) {
    const int i = threadIdx.x + it * 256;
    const int r = i >> 4, c16 = i & 15;
    int64_t sr;
    if (src_map != nullptr) {
      sr = src_map[row0 + r];
      if (sr >= n_src_rows) {
        report_error(err, MOE_ERR_DEVICE_BOUNDS, SITE_QUANT + 2);
        sr = -1;
      }
    } else {
      sr = batch * rows + row0 + r;
    }
    uint4 w = make_uint4(0, 0, 0, 0);
    if (sr >= 0) w = reinterpret_cast<const uint4*>(src + sr * cols + col0)[c16];
    *reinterpret_cast<uint4*>(&tile[r * QC_PITCH + c16 * 8]) = w;
  }
  __syncthreads();
  const int c = threadIdx.x & 127;
  const int64_t drow = batch * cols + col0 + c;      // row of the transposed tensor
  for (int rb = threadIdx.x >> 7; rb < 4; rb += 2) {
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __bfloat162float(tile[(rb * 32 + i) * QC_PITCH + c]);
    uint32_t q[8];
    const uint32_t sc = mx_quant32(v, q);
    store_codes32(codes_t + drow * rows + row0 + rb * 32, q);
    sc_atom[((c & 31) << 4) + (((c >> 5) & 3) << 2) + rb] = uint8_t(sc);
  }
  __syncthreads();
  // the tile's scales are exactly one 512-byte atom of the transposed tensor
  if (threadIdx.x < 32) {
    const int64_t atom = ((batch * cols + col0) >> 7) * (rows >> 7) + (row0 >> 7);
    reinterpret_cast<uint4*>(scales_t + (atom << 9))[threadIdx.x] = reinterpret_cast<const uint4*>(sc_atom)[threadIdx.x];
  }
}

// ---------------------------------------------------------------------------------
// Both orientations from one read: a 128x128 tile of src[batch] is staged once;
// thread tasks then quantize (row, 32-column block) pairs into codes[rows][cols]
// and (column, 32-row block) pairs into codes_t[cols][rows].  Each bf16 weight is
// read once and both MX copies written: 2 B in, 2*(1 + 1/32) B out per element.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) quant_dual_kernel(
    const __nv_bfloat16* __restrict__ src, int rows, int cols, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales, uint8_t* __restrict__ codes_t, uint8_t* __restrict__ scales_t) {
  __shared__ __align__(16) __nv_bfloat16 tile[QC_TILE * QC_PITCH];
  __shared__ __align__(16) uint8_t sc_row[512];
  __shared__ __align__(16) uint8_t sc_col[512];
  const int row0 = blockIdx.x * QC_TILE;
  const int col0 = blockIdx.y * QC_TILE;
  const int64_t batch = blockIdx.z;
  const int64_t srow0 = batch * rows + row0;
#pragma unroll
  for (int it = 0; it < QC_TILE * 16 / 256; ++it) {
    const int i = threadIdx.x + it * 256;
    const int r = i >> 4, c16 = i & 15;
    const uint4 w = reinterpret_cast<const uint4*>(src + (srow0 + r) * cols + col0)[c16];
    *reinterpret_cast<uint4*>(&tile[r * QC_PITCH + c16 * 8]) = w;
  }
  __syncthreads();
  // rowwise: task = (row r, block b), 128 x 4
  for (int task = threadIdx.x; task < QC_TILE * 4; task += blockDim.x) {
    const int r = task >> 2, b = task & 3;
    float v[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 w = *reinterpret_cast<const uint4*>(&tile[r * QC_PITCH + b * 32 + i * 8]);
      v[8 * i + 0] = bf16_lo(w.x); v[8 * i + 1] = bf16_hi(w.x);
      v[8 * i + 2] = bf16_lo(w.y); v[8 * i + 3] = bf16_hi(w.y);
      v[8 * i + 4] = bf16_lo(w.z); v[8 * i + 5] = bf16_hi(w.z);
      v[8 * i + 6] = bf16_lo(w.w); v[8 * i + 7] = bf16_hi(w.w);
    }
    uint32_t q[8];
    const uint32_t sc = mx_quant32(v, q);
    const int64_t drow = srow0 + r;
    store_codes32(codes + drow * cols + col0 + b * 32, q);
    sc_row[((r & 31) << 4) + (((r >> 5) & 3) << 2) + b] = uint8_t(sc);
  }
  // colwise: task = (column c, row block rb), 128 x 4
  for (int task = threadIdx.x; task < QC_TILE * 4; task += blockDim.x) {
    const int c = task & 127, rb = task >> 7;
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __bfloat162float(tile[(rb * 32 + i) * QC_PITCH + c]);
    uint32_t q[8];
    const uint32_t sc = mx_quant32(v, q);
    const int64_t drow = batch * cols + col0 + c;
    store_codes32(codes_t + drow * rows + row0 + rb * 32, q);
    sc_col[((c & 31) << 4) + (((c >> 5) & 3) << 2) + rb] = uint8_t(sc);
  }
  __syncthreads();
  // each orientation's scales of this tile are exactly one 512-byte atom
  if (threadIdx.x < 32) {
    const int64_t atom = (srow0 >> 7) * (cols >> 7) + (col0 >> 7);
    reinterpret_cast<uint4*>(scales + (atom << 9))[threadIdx.x] = reinterpret_cast<const uint4*>(sc_row)[threadIdx.x];
  } else if (threadIdx.x < 64) {
    const int64_t atom = ((batch * cols + col0) >> 7) * (rows >> 7) + (row0 >> 7);
    reinterpret_cast<uint4*>(scales_t + (atom << 9))[threadIdx.x - 32] =
        reinterpret_cast<const uint4*>(sc_col)[threadIdx.x - 32];
  }
}

// ---------------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------------
cudaError_t launch_quant_rowwise(const void* src, int64_t n_rows, int cols, const int* row_of, int k,
                                 int64_t cap, uint8_t* codes, uint8_t* scales, int* err, cudaStream_t st) {
  if (n_rows == 0) return cudaSuccess;
  const int64_t threads = n_rows * 32;
  const unsigned grid = unsigned((threads + 255) / 256);
  if (row_of != nullptr)
    quant_rowwise_kernel<true><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(src), n_rows, cols,
                                                     row_of, k, cap, codes, scales, err);
  else
    quant_rowwise_kernel<false><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(src), n_rows, cols,
                                                      nullptr, 1, cap, codes, scales, err);
  return cudaGetLastError();
}

cudaError_t launch_fill_pad_rows(const int* split_sizes, int E, int cols, uint8_t* codes, uint8_t* scales,
                                 cudaStream_t st) {
  fill_pad_rows_kernel<<<E, 256, 0, st>>>(split_sizes, E, cols, codes, scales);
  return cudaGetLastError();
}

cudaError_t launch_quant_colwise(const void* src, const int* src_map, int64_t n_src_rows, int batch, int rows,
                                 int cols, const int* split_sizes, int E, uint8_t* codes_t, uint8_t* scales_t,
                                 int* err, cudaStream_t st) {
  dim3 grid(rows / QC_TILE, cols / QC_TILE, batch);
  quant_colwise_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(src), src_map, n_src_rows, rows,
                                             cols, split_sizes, E, codes_t, scales_t, err);
  return cudaGetLastError();
}

cudaError_t launch_quant_dual(const void* src, int batch, int rows, int cols, uint8_t* codes, uint8_t* scales,
                              uint8_t* codes_t, uint8_t* scales_t, cudaStream_t st) {
  dim3 grid(rows / QC_TILE, cols / QC_TILE, batch);
  quant_dual_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(src), rows, cols, codes, scales, codes_t,
                                          scales_t);
  return cudaGetLastError();
}

}  // namespace moe
