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
// Destination rows of source row s (a token):
//   ROW_SELF     row s itself;
//   ROW_GIVEN    the k rows row_of[s*k + j] (the permuted rows);
//   ROW_PERMUTE  the k rows the permutation assigns, computed here from the routing's
//                per-expert token masks and their group prefix sums (row = padded start
//                of expert e + base[e][g] + tokens of e below s in s's 32-token group),
//                and written to row_of, src_of and prob_perm on the way.
// v8_src / v8_dst: src / codes are 32-byte aligned (256-bit loads / stores).
// ---------------------------------------------------------------------------------
enum RowMode { ROW_SELF = 0, ROW_GIVEN = 1, ROW_PERMUTE = 2 };

// Zero codes and zero scale codes (scales may be null: codes only) for the padding
// rows of every expert segment (rows split_sizes[e] .. roundup(split_sizes[e],128)-1
// of segment e); with src_of / prob_perm also src -1 and probability 0 there.
// Slice `slice` of expert e clears padding rows slice, slice + FP_SLICES, ...
constexpr int FP_SLICES = 16;

__device__ __forceinline__ void fill_pad_rows_block(const int* __restrict__ split_sizes, int E, int cols,
                                                    int64_t cap, uint8_t* __restrict__ codes,
                                                    uint8_t* __restrict__ scales, int* __restrict__ src_of,
                                                    float* __restrict__ prob_perm, int* err, int e, int slice) {
  __shared__ int seg_start;
  if (threadIdx.x < 32) {
    int acc = 0;
    for (int i = threadIdx.x; i < e; i += 32) acc += (split_sizes[i] + 127) & ~127;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
    if (threadIdx.x == 0) seg_start = acc;
  }
  __syncthreads();
  const int m = split_sizes[e];
  const int npad = ((m + 127) & ~127) - m;
  const int64_t r0 = int64_t(seg_start) + m;
  if (m < 0 || r0 + npad > cap) {
    if (threadIdx.x == 0 && slice == 0) report_error(err, MOE_ERR_DEVICE_BOUNDS, SITE_QUANT + 2);
    return;
  }
  const int vec_per_row = cols >> 4;                 // uint4 per row
  const int nblk = cols >> 5;
  for (int pr = slice; pr < npad; pr += FP_SLICES) {
    const int64_t r = r0 + pr;
    uint4* row = reinterpret_cast<uint4*>(codes + r * cols);
    for (int c = threadIdx.x; c < vec_per_row; c += blockDim.x) row[c] = make_uint4(0, 0, 0, 0);
    if (scales != nullptr)
      for (int b = threadIdx.x; b < nblk; b += blockDim.x) scales[sf_offset(r, b, cols)] = 0;
    if (src_of != nullptr && threadIdx.x == 0) {
      src_of[r] = -1;
      prob_perm[r] = 0.f;
    }
  }
}

// pad_split (optional): blocks past the token blocks zero the padding rows of every
// segment (FP_SLICES blocks per expert); ROW_PERMUTE always has them.
template <int MODE>
__global__ void __launch_bounds__(256) quant_rowwise_kernel(
    const __nv_bfloat16* __restrict__ src, int64_t n_rows, int cols,
    const int* __restrict__ row_of, int k, int64_t cap,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, int* err, bool v8_src, bool v8_dst,
    const int* __restrict__ pad_split, int pad_E, int token_blocks, PermuteRows pr) {
  pdl_wait();                 // may start early (programmatic stream serialization)
  pdl_launch_dependents();
  if (pad_split != nullptr && int(blockIdx.x) >= token_blocks) {
    const int pb = blockIdx.x - token_blocks;
    fill_pad_rows_block(pad_split, pad_E, cols, cap, codes, scales, MODE == ROW_PERMUTE ? pr.src_of : nullptr,
                        pr.prob_perm, err, pb / FP_SLICES, pb % FP_SLICES);
    return;
  }
  const int lane = threadIdx.x & 31;
  __shared__ int seg_start[kMaxExperts];
  if (MODE == ROW_PERMUTE) {
    // padded segment starts: lane l holds experts 8l .. 8l+7
    if (threadIdx.x < 32) {
      int v[8], local = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = 8 * lane + i;
        v[i] = e < pr.E ? (pr.split_sizes[e] + 127) & ~127 : 0;
        local += v[i];
      }
      int incl = local;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += o;
      }
      int run = incl - local;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = 8 * lane + i;
        if (e < pr.E) seg_start[e] = run;
        run += v[i];
      }
    }
    __syncthreads();
  }
  const int64_t s = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (s >= n_rows) return;
  const int nblk = cols >> 5;
  // lane j < k finds the destination row of slot j; every lane then takes all k by
  // shuffles here, where the whole warp is present (fewer than 32 lanes enter the
  // block loop below when cols < 1024)
  int nd = 1;
  int dst[8];
  if (MODE != ROW_SELF) {
    nd = k;
    int my_dst = -1;
    bool bad = false;
    if (lane < k) {
      if (MODE == ROW_GIVEN) {
        my_dst = row_of[s * k + lane];
      } else {
        const int e = pr.idx[s * k + lane];
        if (e >= 0 && e < pr.E) {
          const int64_t gi = int64_t(e) * pr.G + (s >> 5);
          const uint32_t m = pr.masks[gi];
          const uint32_t bit = 1u << (s & 31);
          if (m & bit) my_dst = seg_start[e] + pr.bases[gi] + __popc(m & (bit - 1u));
        }
      }
      bad = my_dst < 0 || my_dst >= cap;
      if (MODE == ROW_PERMUTE) {
        pr.row_of[s * k + lane] = bad ? -1 : my_dst;
        if (!bad) {
          pr.src_of[my_dst] = int(s);
          pr.prob_perm[my_dst] = pr.prob[s * k + lane];
        }
      }
    }
    if (__any_sync(0xFFFFFFFFu, bad)) {
      if (lane == 0) report_error(err, MOE_ERR_DEVICE_BOUNDS, SITE_QUANT + 1);
      return;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) dst[j] = __shfl_sync(0xFFFFFFFFu, my_dst, j);
  }
  for (int b = lane; b < nblk; b += 32) {
    uint32_t w[16];
    const __nv_bfloat16* blk = src + s * cols + (int64_t)b * 32;
    if (v8_src) {
      ld_global_v8(blk, w);
      ld_global_v8(blk + 16, w + 8);
    } else {
      const uint4* p4 = reinterpret_cast<const uint4*>(blk);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 x = p4[i];
        w[4 * i + 0] = x.x;
        w[4 * i + 1] = x.y;
        w[4 * i + 2] = x.z;
        w[4 * i + 3] = x.w;
      }
    }
    uint32_t q[8];
    const uint32_t c = mx_quant32_bf16(w, q);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < nd) {
        const int64_t row = MODE != ROW_SELF ? int64_t(dst[j]) : s;
        store_codes32(codes + row * cols + (int64_t)b * 32, q, v8_dst);
        scales[sf_offset(row, b, cols)] = uint8_t(c);
      }
    }
  }
}

__global__ void __launch_bounds__(256) fill_pad_rows_kernel(
    const int* __restrict__ split_sizes, int E, int cols, int64_t cap,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, int* err) {
  pdl_wait();                 // may start early (programmatic stream serialization)
  pdl_launch_dependents();
  fill_pad_rows_block(split_sizes, E, cols, cap, codes, scales, nullptr, nullptr, err, blockIdx.x, blockIdx.y);
}

// ---------------------------------------------------------------------------------
// Colwise: blocks of 32 along the row axis, output transposed.  One CTA per tile of
// 128 rows x 64 columns.  Warp 0 fetches the tile's rows with 32 four-row TMA
// gathers (tile::gather4: one instruction per four source rows, wherever they lie;
// a padding row's index points one past the source, and the copy fills it with
// zeros), then thread (column pair c, row block rb) reduces 32 rows of two columns,
// quantizes them and writes 32 contiguous codes to each of the transposed rows c
// and c+1.  The small tiles keep twelve CTAs' loads (192 KB) in flight per SM.
// The tile's scales are half of a 512-byte atom of the transposed tensor: bytes
// 0..7 (the atom's first 64 columns) or 8..15 of each of its 16-byte rows.
//   src row of tile row r: src_map ? src_map[r] (-1 -> zero row) : batch*rows + r
//   split_sizes (optional): row tiles at or past the padded total are skipped.
// ---------------------------------------------------------------------------------
constexpr int QC_TILE = 128;
constexpr int QC_PITCH = QC_TILE + 8;                // bf16 per smem row of the dual kernel (16 B pad)
constexpr int QG_ROWS = 128, QG_COLS = 64;           // gathered tile
constexpr int QG_THREADS = 2 * QG_COLS;              // (column pair, row block) tasks: 32 x 4

__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* map, int x, const int (&y)[4],
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y[0]), "r"(y[1]), "r"(y[2]),
        "r"(y[3]), "r"(smem_u32(bar))
      : "memory");
}

__global__ void __launch_bounds__(QG_THREADS, 12) quant_colwise_kernel(
    const __grid_constant__ CUtensorMap src_rows, const int* __restrict__ src_map, int n_src_rows, int rows,
    int cols, const int* __restrict__ split_sizes, int E, uint8_t* __restrict__ codes_t,
    uint8_t* __restrict__ scales_t, int* err, bool v8, uint64_t wait_limit_ns) {
  pdl_wait();                 // may start early (programmatic stream serialization)
  pdl_launch_dependents();
  __shared__ __align__(1024) __nv_bfloat16 tile[QG_ROWS * QG_COLS];
  __shared__ __align__(16) uint8_t sc_half[256];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int s_rows_used;
  const int row0 = blockIdx.x * QG_ROWS;
  const int col0 = blockIdx.y * QG_COLS;
  const int64_t batch = blockIdx.z;
  if (threadIdx.x < 32) {
    int acc = rows;
    if (split_sizes != nullptr) {
      acc = 0;
      for (int e = threadIdx.x; e < E; e += 32) acc += (split_sizes[e] + 127) & ~127;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
    }
    if (threadIdx.x == 0) {
      s_rows_used = acc;
      mbar_init(&bar, 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
  }
  __syncthreads();
  if (row0 >= s_rows_used) return;
  if (threadIdx.x < 32) {
    // lane l gathers tile rows 4l .. 4l+3
    int y[4];
    if (src_map != nullptr) {
      const int4 s4 = reinterpret_cast<const int4*>(src_map + row0)[threadIdx.x];
      y[0] = s4.x;
      y[1] = s4.y;
      y[2] = s4.z;
      y[3] = s4.w;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (y[j] >= n_src_rows) {
          report_error(err, MOE_ERR_DEVICE_BOUNDS, SITE_QUANT + 2);
          y[j] = -1;
        }
        if (y[j] < 0) y[j] = n_src_rows;       // past the source: zeros
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) y[j] = int(batch * rows) + row0 + 4 * int(threadIdx.x) + j;
    }
    if (threadIdx.x == 0) mbar_arrive_expect_tx(&bar, QG_ROWS * QG_COLS * 2);
    __syncwarp();
    tma_gather4(tile + threadIdx.x * 4 * QG_COLS, &src_rows, col0, y, &bar);
  }
  // bounded wait for the tile (the only copies this CTA issues)
  if (!mbar_try_wait(&bar, 0)) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(&bar, 0)) {
      if (globaltimer_ns() - t0 > wait_limit_ns) {
        report_error(err, MOE_ERR_DEVICE_TIMEOUT, SITE_QUANT + 3);
        return;
      }
    }
  }
  const int c = 2 * (threadIdx.x & 31), rb = threadIdx.x >> 5;
  const uint32_t* p = reinterpret_cast<const uint32_t*>(&tile[(rb * 32) * QG_COLS + c]);
  uint32_t q_lo[8], q_hi[8];
  const uint32_t sc = mx_quant32_bf16_colpair(p, QG_COLS / 2, q_lo, q_hi);
  const int64_t drow = batch * cols + col0 + c;          // row of the transposed tensor
  store_codes32(codes_t + drow * rows + row0 + rb * 32, q_lo, v8);
  store_codes32(codes_t + (drow + 1) * rows + row0 + rb * 32, q_hi, v8);
  // atom byte of (column cc of the atom's 128, row block rb): 16 (cc & 31) + 4 ((cc >> 5) & 3) + rb;
  // here (cc >> 5) & 3 = 2 [col0 & 64] + (c >> 5), so the tile fills 8 bytes of each 16-byte row
  sc_half[((c & 31) << 3) + ((c >> 5) << 2) + rb] = uint8_t(sc);
  sc_half[(((c + 1) & 31) << 3) + (((c + 1) >> 5) << 2) + rb] = uint8_t(sc >> 8);
  __syncthreads();
  if (threadIdx.x < 32) {
    const int64_t atom = ((batch * cols + col0) >> 7) * (rows >> 7) + (row0 >> 7);
    *reinterpret_cast<uint2*>(scales_t + (atom << 9) + (threadIdx.x << 4) + ((col0 & 64) >> 3)) =
        reinterpret_cast<const uint2*>(sc_half)[threadIdx.x];
  }
}

// ---------------------------------------------------------------------------------
// Both orientations from one read: a 128x128 tile of src[batch] is staged once;
// thread tasks then quantize (row, 32-column block) pairs into codes[rows][cols]
// and (column, 32-row block) pairs into codes_t[cols][rows].  Each bf16 weight is
// read once and both MX copies written: 2 B in, 2*(1 + 1/32) B out per element.
// ---------------------------------------------------------------------------------
// Src: StackedSrc (src[batch] of one tensor) or ExpertSrc (one pointer per matrix).
// codes_t == nullptr: the rowwise orientation only.
template <class Src>
__global__ void __launch_bounds__(256, 6) quant_dual_kernel(
    const __grid_constant__ Src src, int rows, int cols, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales, uint8_t* __restrict__ codes_t, uint8_t* __restrict__ scales_t, bool v8) {
  pdl_wait();                 // may start early (programmatic stream serialization)
  pdl_launch_dependents();
  __shared__ __align__(16) __nv_bfloat16 tile[QC_TILE * QC_PITCH];
  __shared__ __align__(16) uint8_t sc_row[512];
  __shared__ __align__(16) uint8_t sc_col[512];
  const int row0 = blockIdx.x * QC_TILE;
  const int col0 = blockIdx.y * QC_TILE;
  const int64_t batch = blockIdx.z;
  const int64_t srow0 = batch * rows + row0;         // row of the stacked outputs
  {
    const __nv_bfloat16* m = src.mat(batch);
    const int c16 = threadIdx.x & 15, rbase = threadIdx.x >> 4;
#pragma unroll
    for (int it = 0; it < QC_TILE / 16; ++it) {
      const int r = rbase + 16 * it;
      cp_async16(&tile[r * QC_PITCH + c16 * 8], m + int64_t(row0 + r) * cols + col0 + c16 * 8, true);
    }
  }
  cp_async_wait_all();
  __syncthreads();
  // rowwise: task = (row r, block b), 128 x 4
  for (int task = threadIdx.x; task < QC_TILE * 4; task += blockDim.x) {
    const int r = task >> 2, b = task & 3;
    const uint32_t* p = reinterpret_cast<const uint32_t*>(&tile[r * QC_PITCH + b * 32]);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 x = reinterpret_cast<const uint4*>(p)[i];
      w[4 * i + 0] = x.x;
      w[4 * i + 1] = x.y;
      w[4 * i + 2] = x.z;
      w[4 * i + 3] = x.w;
    }
    uint32_t q[8];
    const uint32_t sc = mx_quant32_bf16(w, q);
    const int64_t drow = srow0 + r;
    store_codes32(codes + drow * cols + col0 + b * 32, q, v8);
    sc_row[((r & 31) << 4) + (((r >> 5) & 3) << 2) + b] = uint8_t(sc);
  }
  // colwise: task = (columns c, c+1) x 32-row block rb -- one per thread
  if (codes_t != nullptr) {
    const int c = 2 * (threadIdx.x & 63), rb = threadIdx.x >> 6;
    const uint32_t* p = reinterpret_cast<const uint32_t*>(&tile[(rb * 32) * QC_PITCH + c]);
    uint32_t q_lo[8], q_hi[8];
    const uint32_t sc = mx_quant32_bf16_colpair(p, QC_PITCH / 2, q_lo, q_hi);
    const int64_t drow = batch * cols + col0 + c;
    store_codes32(codes_t + drow * rows + row0 + rb * 32, q_lo, v8);
    store_codes32(codes_t + (drow + 1) * rows + row0 + rb * 32, q_hi, v8);
    sc_col[((c & 31) << 4) + (((c >> 5) & 3) << 2) + rb] = uint8_t(sc);
    sc_col[(((c + 1) & 31) << 4) + ((((c + 1) >> 5) & 3) << 2) + rb] = uint8_t(sc >> 8);
  }
  __syncthreads();
  // each orientation's scales of this tile are exactly one 512-byte atom
  if (threadIdx.x < 32) {
    const int64_t atom = (srow0 >> 7) * (cols >> 7) + (col0 >> 7);
    reinterpret_cast<uint4*>(scales + (atom << 9))[threadIdx.x] = reinterpret_cast<const uint4*>(sc_row)[threadIdx.x];
  } else if (threadIdx.x < 64 && codes_t != nullptr) {
    const int64_t atom = ((batch * cols + col0) >> 7) * (rows >> 7) + (row0 >> 7);
    reinterpret_cast<uint4*>(scales_t + (atom << 9))[threadIdx.x - 32] =
        reinterpret_cast<const uint4*>(sc_col)[threadIdx.x - 32];
  }
}

// ---------------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------------
cudaError_t launch_quant_rowwise(const void* src, int64_t n_rows, int cols, const int* row_of, int k,
                                 int64_t cap, uint8_t* codes, uint8_t* scales, int* err, cudaStream_t st,
                                 const int* pad_split, int pad_E) {
  if (n_rows == 0 && pad_split == nullptr) return cudaSuccess;
  const int64_t token_blocks = (n_rows * 32 + 255) / 256;
  const unsigned grid = unsigned(token_blocks + (pad_split != nullptr ? int64_t(pad_E) * FP_SLICES : 0));
  const bool v8s = aligned32(src), v8d = aligned32(codes);
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(src);
  if (row_of != nullptr)
    launch_pdl(quant_rowwise_kernel<ROW_GIVEN>, dim3(grid), dim3(256), 0, st,
               x, n_rows, cols, row_of, k, cap, codes, scales, err, v8s, v8d, pad_split, pad_E, int(token_blocks),
               PermuteRows{});
  else
    launch_pdl(quant_rowwise_kernel<ROW_SELF>, dim3(grid), dim3(256), 0, st,
               x, n_rows, cols, nullptr, 1, cap, codes, scales, err, v8s, v8d, pad_split, pad_E, int(token_blocks),
               PermuteRows{});
  return cudaGetLastError();
}

cudaError_t launch_permute_quant_rows(const void* x, int T, int H, int k, int64_t cap, const PermuteRows& p,
                                      uint8_t* codes, uint8_t* scales, int* err, cudaStream_t st) {
  if (p.E < 1 || p.E > kMaxExperts || k < 1 || k > 8) return cudaErrorInvalidValue;
  const int64_t token_blocks = (int64_t(T) * 32 + 255) / 256;
  const unsigned grid = unsigned(token_blocks + int64_t(p.E) * FP_SLICES);
  launch_pdl(quant_rowwise_kernel<ROW_PERMUTE>, dim3(grid), dim3(256), 0, st,
             static_cast<const __nv_bfloat16*>(x), T, H, nullptr, k, cap, codes, scales, err, aligned32(x),
             aligned32(codes), p.split_sizes, p.E, int(token_blocks), p);
  return cudaGetLastError();
}

cudaError_t launch_fill_pad_rows(const int* split_sizes, int E, int cols, int64_t cap, uint8_t* codes,
                                 uint8_t* scales, int* err, cudaStream_t st) {
  launch_pdl(fill_pad_rows_kernel, dim3(E, FP_SLICES), dim3(256), 0, st,
             split_sizes, E, cols, cap, codes, scales, err);
  return cudaGetLastError();
}

cudaError_t launch_quant_colwise(const void* src, const int* src_map, int64_t n_src_rows, int batch, int rows,
                                 int cols, const int* split_sizes, int E, uint8_t* codes_t, uint8_t* scales_t,
                                 int* err, cudaStream_t st) {
  if (rows <= 0 || cols <= 0 || batch <= 0) return cudaSuccess;
  // row coordinates of the gathers (and the one-past-the-end zero row) are 32-bit
  if (n_src_rows >= (int64_t(1) << 31) - 1 || rows % QG_ROWS != 0 || cols % QG_COLS != 0)
    return cudaErrorInvalidValue;
  CUtensorMap m;
  if (!encode_gather_rows_map(&m, src, n_src_rows, cols, QG_COLS)) return cudaErrorInvalidValue;
  dim3 grid(rows / QG_ROWS, cols / QG_COLS, batch);
  launch_pdl(quant_colwise_kernel, dim3(grid), dim3(QG_THREADS), 0, st,
             m, src_map, int(n_src_rows), rows, cols, split_sizes, E, codes_t, scales_t, err, aligned32(codes_t),
             kWaitLimitNs);
  return cudaGetLastError();
}

cudaError_t launch_quant_dual(const void* src, int batch, int rows, int cols, uint8_t* codes, uint8_t* scales,
                              uint8_t* codes_t, uint8_t* scales_t, cudaStream_t st) {
  dim3 grid(rows / QC_TILE, cols / QC_TILE, batch);
  const StackedSrc s{static_cast<const __nv_bfloat16*>(src), int64_t(rows) * cols};
  launch_pdl(quant_dual_kernel<StackedSrc>, dim3(grid), dim3(256), 0, st,
             s, rows, cols, codes, scales, codes_t, scales_t, aligned32(codes) && aligned32(codes_t));
  return cudaGetLastError();
}

cudaError_t launch_quant_dual_experts(const ExpertSrc& src, int batch, int rows, int cols, uint8_t* codes,
                                      uint8_t* scales, uint8_t* codes_t, uint8_t* scales_t, cudaStream_t st) {
  dim3 grid(rows / QC_TILE, cols / QC_TILE, batch);
  launch_pdl(quant_dual_kernel<ExpertSrc>, dim3(grid), dim3(256), 0, st,
             src, rows, cols, codes, scales, codes_t, scales_t, aligned32(codes) && aligned32(codes_t));
  return cudaGetLastError();
}

}  // namespace moe
