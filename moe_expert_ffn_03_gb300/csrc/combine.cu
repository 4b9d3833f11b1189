// Unpermute + combine: out[t] = sum over slots j of y[row_of[t][j]] (optionally
// times prob[t][j]), f32 sum in slot order, rounded to bf16.  The router
// probability is already applied by ScaledSwiGLU, so the layer calls it with
// prob = NULL (page "Efficient MoE Training for Biological Foundation Models",
// section "MXFP8与融合MLP").  HBM-bound: k*H*2 bytes read, H*2 written per token.
#include "kernels.cuh"

namespace moe {

// V8: y and out 32-byte aligned, 16 bf16 per lane and step with 256-bit loads and stores;
// otherwise 8 with 16-byte ones.
template <bool V8>
__global__ void __launch_bounds__(256) combine_kernel(
    const __nv_bfloat16* __restrict__ y, const int* __restrict__ row_of, const float* __restrict__ prob,
    int T, int k, int H, int64_t cap, __nv_bfloat16* __restrict__ out, int* err) {
  pdl_wait();                 // may start early (programmatic stream serialization)
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  int rows[8];
  float p[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    rows[j] = 0;
    p[j] = 1.f;
    if (j < k) {
      rows[j] = row_of[t * k + j];
      if (prob != nullptr) p[j] = prob[t * k + j];
      if (rows[j] < 0 || rows[j] >= cap) {
        report_error(err, MOE_ERR_DEVICE_BOUNDS, SITE_COMBINE + 1);
        return;
      }
    }
  }
  constexpr int W = V8 ? 8 : 4;                      // 32-bit words (two bf16 each) per lane and step
  const int nvec = H / (2 * W);
  for (int c = lane; c < nvec; c += 32) {
    float acc[2 * W];
#pragma unroll
    for (int i = 0; i < 2 * W; ++i) acc[i] = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k) {
        uint32_t w[W];
        const __nv_bfloat16* src = y + int64_t(rows[j]) * H + int64_t(c) * 2 * W;
        if (V8) {
          ld_global_v8(src, w);
        } else {
          const uint4 v = *reinterpret_cast<const uint4*>(src);
          w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
        }
#pragma unroll
        for (int i = 0; i < W; ++i) {
          acc[2 * i] += p[j] * bf16_lo(w[i]);
          acc[2 * i + 1] += p[j] * bf16_hi(w[i]);
        }
      }
    }
    uint32_t o[W];
#pragma unroll
    for (int i = 0; i < W; ++i) o[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
    __nv_bfloat16* dst = out + t * H + int64_t(c) * 2 * W;
    if (V8) st_global_v8(dst, o);
    else *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// dprob[t][j] = sum over N-tiles of the per-tile partial row sums at row_of[t][j]
// (fixed tile order: deterministic, no float atomics).
__global__ void __launch_bounds__(256) dprob_reduce_kernel(
    const float* __restrict__ dp_part, int n_tiles, int64_t cap, const int* __restrict__ row_of, int64_t R,
    float* __restrict__ dprob, int* err) {
  pdl_wait();                 // may start early (programmatic stream serialization)
  pdl_launch_dependents();
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= R) return;
  const int r = row_of[i];
  if (r < 0 || r >= cap) {
    report_error(err, MOE_ERR_DEVICE_BOUNDS, SITE_COMBINE + 2);
    return;
  }
  float acc = 0.f;
  for (int n = 0; n < n_tiles; ++n) acc += dp_part[int64_t(n) * cap + r];
  dprob[i] = acc;
}

// The same sums by permuted row, for rows with many partials (the Mixtral-shaped 224; the
// token-ordered kernel above is as fast for few).  A block holds 32 rows and its eight warps
// split the partials: warp w sums n = w, w + 8, ... of its lane's row (a warp's loads are 128
// contiguous bytes), then warp 0 adds the eight sums in warp order (a fixed order:
// deterministic), finds the row's slot j among row_of[src_of[r]][*] and writes
// dprob[src_of[r]][j].  Rows past the padded total and padding rows (src_of = -1) write nothing.
constexpr int DPR_WARPS = 8;
__global__ void __launch_bounds__(32 * DPR_WARPS) dprob_reduce_rows_kernel(
    const float* __restrict__ dp_part, int n_tiles, int64_t cap, const int* __restrict__ split_sizes, int E,
    const int* __restrict__ src_of, const int* __restrict__ row_of, int k, int T, float* __restrict__ dprob,
    int* err) {
  pdl_wait();                 // may start early (programmatic stream serialization)
  pdl_launch_dependents();
  __shared__ int64_t total_s;
  __shared__ float part[DPR_WARPS][32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (w == 0) {
    int64_t acc = 0;
    for (int e = lane; e < E; e += 32) acc += (split_sizes[e] + 127) & ~127;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
    if (lane == 0) total_s = acc;
  }
  __syncthreads();
  const int64_t r = int64_t(blockIdx.x) * 32 + lane;
  const bool valid = r < total_s && r < cap;
  float acc = 0.f;
  if (valid) {
    int n = w;
    for (; n + 3 * DPR_WARPS < n_tiles; n += 4 * DPR_WARPS) {
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = dp_part[int64_t(n + j * DPR_WARPS) * cap + r];
#pragma unroll
      for (int j = 0; j < 4; ++j) acc += v[j];
    }
    for (; n < n_tiles; n += DPR_WARPS) acc += dp_part[int64_t(n) * cap + r];
  }
  part[w][lane] = acc;
  __syncthreads();
  if (w != 0 || !valid) return;
  float sum = part[0][lane];
#pragma unroll
  for (int i = 1; i < DPR_WARPS; ++i) sum += part[i][lane];
  const int t = src_of[r];
  if (t < 0) return;
  if (t >= T) {
    report_error(err, MOE_ERR_DEVICE_BOUNDS, SITE_COMBINE + 4);
    return;
  }
  int j = 0;
  while (j < k && row_of[int64_t(t) * k + j] != r) ++j;
  if (j == k) {
    report_error(err, MOE_ERR_DEVICE_BOUNDS, SITE_COMBINE + 5);
    return;
  }
  dprob[int64_t(t) * k + j] = sum;
}

// bf16 path: x_perm[row_of[t][j]] = x[t] (one warp per token, 16-byte copies).
__global__ void __launch_bounds__(256) gather_rows_kernel(const __nv_bfloat16* __restrict__ x,
                                                          const int* __restrict__ row_of, int T, int k, int H,
                                                          int64_t cap, __nv_bfloat16* __restrict__ x_perm, int* err) {
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  const uint4* src = reinterpret_cast<const uint4*>(x + t * H);
  for (int j = 0; j < k; ++j) {
    const int r = row_of[t * k + j];
    if (r < 0 || r >= cap) {
      report_error(err, MOE_ERR_DEVICE_BOUNDS, SITE_COMBINE + 3);
      continue;
    }
    uint4* dst = reinterpret_cast<uint4*>(x_perm + int64_t(r) * H);
    for (int c = lane; c < H / 8; c += 32) dst[c] = src[c];
  }
}

// Zero the padding rows (split_sizes[e] .. roundup(split_sizes[e],128)-1 of segment e)
// of a permuted buffer whose rows are row_bytes long (a multiple of 16).
__global__ void __launch_bounds__(256) zero_pad_rows_kernel(const int* __restrict__ split_sizes, int E,
                                                            int64_t row_bytes, uint8_t* __restrict__ buf) {
  __shared__ int seg_start;
  const int e = blockIdx.x;
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int i = 0; i < e; ++i) acc += (split_sizes[i] + 127) & ~127;
    seg_start = acc;
  }
  __syncthreads();
  const int m = split_sizes[e];
  const int64_t n16 = (((m + 127) & ~127) - m) * (row_bytes / 16);
  uint4* p = reinterpret_cast<uint4*>(buf + (int64_t(seg_start) + m) * row_bytes);
  for (int64_t i = int64_t(blockIdx.y) * blockDim.x + threadIdx.x; i < n16; i += int64_t(gridDim.y) * blockDim.x)
    p[i] = make_uint4(0, 0, 0, 0);
}

cudaError_t launch_gather_rows(const void* x, const int* row_of, const int* split_sizes, int T, int k, int H, int E,
                               int64_t cap, void* x_perm, int* err, cudaStream_t st) {
  gather_rows_kernel<<<unsigned((int64_t(T) * 32 + 255) / 256), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(x), row_of, T, k, H, cap, static_cast<__nv_bfloat16*>(x_perm), err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  zero_pad_rows_kernel<<<dim3(E, 8), 256, 0, st>>>(split_sizes, E, int64_t(H) * 2, static_cast<uint8_t*>(x_perm));
  return cudaGetLastError();
}

cudaError_t launch_combine(const void* y, const int* row_of, const float* prob, int T, int k, int H, int64_t cap,
                           void* out, int* err, cudaStream_t st) {
  const int64_t threads = int64_t(T) * 32;
  const unsigned grid = unsigned((threads + 255) / 256);
  const __nv_bfloat16* yb = static_cast<const __nv_bfloat16*>(y);
  __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(out);
  if (aligned32(y) && aligned32(out) && H % 16 == 0)
    launch_pdl(combine_kernel<true>, dim3(grid), dim3(256), 0, st,
               yb, row_of, prob, T, k, H, cap, ob, err);
  else
    launch_pdl(combine_kernel<false>, dim3(grid), dim3(256), 0, st,
               yb, row_of, prob, T, k, H, cap, ob, err);
  return cudaGetLastError();
}

cudaError_t launch_dprob_reduce(const float* dp_part, int n_tiles, int64_t cap, const int* split_sizes, int E,
                                const int* src_of, const int* row_of, int k, int T, float* dprob, int* err,
                                cudaStream_t st) {
  if (src_of != nullptr && n_tiles >= 64) {
    launch_pdl(dprob_reduce_rows_kernel, dim3(unsigned((cap + 31) / 32)), dim3(32 * DPR_WARPS), 0, st,
               dp_part, n_tiles, cap, split_sizes, E, src_of, row_of, k, T, dprob, err);
  } else {
    const int64_t R = int64_t(T) * k;
    launch_pdl(dprob_reduce_kernel, dim3(unsigned((R + 255) / 256)), dim3(256), 0, st,
               dp_part, n_tiles, cap, row_of, R, dprob, err);
  }
  return cudaGetLastError();
}

}  // namespace moe
