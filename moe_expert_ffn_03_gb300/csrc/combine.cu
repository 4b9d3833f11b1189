// Unpermute + combine: out[t] = sum over slots j of y[row_of[t][j]] (optionally
// times prob[t][j]), f32 sum in slot order, rounded to bf16.  The router
// probability is already applied by ScaledSwiGLU, so the layer calls it with
// prob = NULL (page "Efficient MoE Training for Biological Foundation Models",
// section "MXFP8与融合MLP").  HBM-bound: k*H*2 bytes read, H*2 written per token.
#include "kernels.cuh"

namespace moe {

__global__ void __launch_bounds__(256) combine_kernel(
    const __nv_bfloat16* __restrict__ y, const int* __restrict__ row_of, const float* __restrict__ prob,
    int T, int k, int H, int64_t cap, __nv_bfloat16* __restrict__ out, int* err) {
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
  const int nvec = H >> 3;                            // 8 bf16 per 16-byte vector
  for (int c = lane; c < nvec; c += 32) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k) {
        const uint4 w = reinterpret_cast<const uint4*>(y + int64_t(rows[j]) * H)[c];
        acc[0] += p[j] * bf16_lo(w.x); acc[1] += p[j] * bf16_hi(w.x);
        acc[2] += p[j] * bf16_lo(w.y); acc[3] += p[j] * bf16_hi(w.y);
        acc[4] += p[j] * bf16_lo(w.z); acc[5] += p[j] * bf16_hi(w.z);
        acc[6] += p[j] * bf16_lo(w.w); acc[7] += p[j] * bf16_hi(w.w);
      }
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    reinterpret_cast<uint4*>(out + t * H)[c] = o;
  }
}

// dprob[t][j] = sum over N-tiles of the per-tile partial row sums at row_of[t][j]
// (fixed tile order: deterministic, no float atomics).
__global__ void __launch_bounds__(256) dprob_reduce_kernel(
    const float* __restrict__ dp_part, int n_tiles, int64_t cap, const int* __restrict__ row_of, int64_t R,
    float* __restrict__ dprob, int* err) {
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

cudaError_t launch_combine(const void* y, const int* row_of, const float* prob, int T, int k, int H, int64_t cap,
                           void* out, int* err, cudaStream_t st) {
  const int64_t threads = int64_t(T) * 32;
  combine_kernel<<<unsigned((threads + 255) / 256), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(y), row_of, prob, T, k, H, cap, static_cast<__nv_bfloat16*>(out), err);
  return cudaGetLastError();
}

cudaError_t launch_dprob_reduce(const float* dp_part, int n_tiles, int64_t cap, const int* row_of, int64_t R,
                                float* dprob, int* err, cudaStream_t st) {
  dprob_reduce_kernel<<<unsigned((R + 255) / 256), 256, 0, st>>>(dp_part, n_tiles, cap, row_of, R, dprob, err);
  return cudaGetLastError();
}

}  // namespace moe
