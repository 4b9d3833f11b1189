// Linear router on both sides: logits = x W_r^T, and the backward through the
// top-k softmax (page "英伟达开源MoE加速神器", section "三板斧": tokens are
// routed to a few experts; page "Efficient MoE Training for Biological
// Foundation Models", section "MXFP8与融合MLP": the router probabilities scale
// the SwiGLU output).  The forward runs on the tensor cores; the backward
// kernels run on the CUDA cores with fixed summation orders (deterministic
// results):
//   forward                 logits = x W_r^T on the tensor cores (router_fwd_tc_kernel,
//                           gemm.cu): 128 tokens per CTA, N = roundup(E, 16), bf16
//                           operands, f32 logits (rows and columns past T and E masked);
//   router_dlogits_kernel   one warp per token, straight-through top-k softmax;
//   router_dx_kernel        dx[t] += sum_e dl[t][e] W_r[e] (bf16 in place);
//   dW_r                    dl^T x on the tensor cores (router_dw_tc_kernel): dl split
//                           into two bf16 terms hi + lo by the dlogits kernel, f32
//                           accumulation per token chunk, chunks summed in chunk order
//                           by router_dw_reduce_kernel.
#include <cstdio>

#include "kernels.cuh"

namespace moe {

// One warp per token.  renormalize: dl[e_j] = p_j (dp_j - sum_i p_i dp_i), 0 elsewhere;
// plain softmax: dl[e] = s_e (g_e - sum_j p_j dp_j) with g the dprob scattered to idx.
// Also dl as two bf16 terms for the tensor cores, [T][N] with zeros in columns E..N-1:
// hi = bf16(dl), lo = bf16(dl - hi) (dl - hi is exact in f32).
__global__ void __launch_bounds__(256) router_dlogits_kernel(const float* __restrict__ logits,
                                                             const int* __restrict__ idx,
                                                             const float* __restrict__ prob,
                                                             const float* __restrict__ dprob, int T, int E, int k,
                                                             int renorm, float* __restrict__ dl,
                                                             __nv_bfloat16* __restrict__ dl_hi,
                                                             __nv_bfloat16* __restrict__ dl_lo, int N, int* err) {
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  float pdp = 0.f;
  for (int j = 0; j < k; ++j) pdp += prob[t * k + j] * dprob[t * k + j];
  const float* lrow = logits + t * E;
  float m = -INFINITY, z = 0.f;
  if (!renorm) {
    for (int e = lane; e < E; e += 32) m = fmaxf(m, lrow[e]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    for (int e = lane; e < E; e += 32) z += expf(lrow[e] - m);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, off);
  }
  for (int e = lane; e < N; e += 32) {
    float v = 0.f;
    if (e < E) {
      float g = 0.f, pe = 0.f;
      bool sel = false;
      for (int j = 0; j < k; ++j) {
        const int ej = idx[t * k + j];
        if (ej < 0 || ej >= E) {
          report_error(err, MOE_ERR_DEVICE_BOUNDS, SITE_ROUTE + 1);
          continue;
        }
        if (ej == e) {
          sel = true;
          g = dprob[t * k + j];
          pe = prob[t * k + j];
        }
      }
      if (renorm) v = sel ? pe * (g - pdp) : 0.f;
      else v = expf(lrow[e] - m) / z * (g - pdp);
      dl[t * E + e] = v;
    }
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    dl_hi[t * N + e] = hi;
    dl_lo[t * N + e] = __float2bfloat16_rn(v - __bfloat162float(hi));
  }
}

// One warp per token: dx[t][h..h+7] = bf16(float(dx) + sum over the experts with a
// non-zero dl (the k selected ones when renormalizing) of dl * W_r[e][h..h+7]).
__global__ void __launch_bounds__(256) router_dx_kernel(const float* __restrict__ dl, const int* __restrict__ idx,
                                                        const __nv_bfloat16* __restrict__ w, int T, int H, int E,
                                                        int k, int renorm, __nv_bfloat16* __restrict__ dx) {
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  const int n = renorm ? k : E;
  for (int c = lane; c < H / 8; c += 32) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int j = 0; j < n; ++j) {
      const int e = renorm ? idx[t * k + j] : j;
      if (e < 0 || e >= E) continue;
      const float s = dl[t * E + e];
      const uint4 wv = *reinterpret_cast<const uint4*>(w + int64_t(e) * H + c * 8);
      acc[0] += s * bf16_lo(wv.x); acc[1] += s * bf16_hi(wv.x);
      acc[2] += s * bf16_lo(wv.y); acc[3] += s * bf16_hi(wv.y);
      acc[4] += s * bf16_lo(wv.z); acc[5] += s * bf16_hi(wv.z);
      acc[6] += s * bf16_lo(wv.w); acc[7] += s * bf16_hi(wv.w);
    }
    uint4* p = reinterpret_cast<uint4*>(dx + t * H) + c;
    const uint4 o = *p;
    uint4 r;
    r.x = pack_bf16x2(bf16_lo(o.x) + acc[0], bf16_hi(o.x) + acc[1]);
    r.y = pack_bf16x2(bf16_lo(o.y) + acc[2], bf16_hi(o.y) + acc[3]);
    r.z = pack_bf16x2(bf16_lo(o.z) + acc[4], bf16_hi(o.z) + acc[5]);
    r.w = pack_bf16x2(bf16_lo(o.w) + acc[6], bf16_hi(o.w) + acc[7]);
    *p = r;
  }
}

__global__ void __launch_bounds__(256) router_dw_reduce_kernel(const float* __restrict__ partial, int64_t n,
                                                               int chunks, float* __restrict__ dw) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float s = 0.f;
  for (int c = 0; c < chunks; ++c) s += partial[int64_t(c) * n + i];
  dw[i] = s;
}

// Workspace of the router backward: chunk partials [max chunks][E][H] f32, then dl as
// bf16 hi and lo terms [T][N] each.
static size_t al256(size_t b) { return (b + 255) & ~size_t(255); }
size_t router_ws_bytes(int T, int E, int H) {
  return al256(size_t(router_dw_max_chunks(H)) * E * H * sizeof(float)) +
         2 * al256(size_t(T) * router_dw_cols(E) * sizeof(__nv_bfloat16));
}

cudaError_t launch_router_fwd(const void* x, const void* w, int T, int H, int E, float* logits, int* err,
                              cudaStream_t st, char* msg, size_t msg_len) {
  // 128 tokens per CTA, N = roundup(E, 16) on single-CTA tensor-core MMAs (gemm.cu)
  const cudaError_t e = launch_router_fwd_tc(x, w, T, H, E, logits, err, st);
  if (e != cudaSuccess && msg != nullptr) snprintf(msg, msg_len, "router logits launch failed: %s", cudaGetErrorString(e));
  return e;
}

cudaError_t launch_router_bwd(const void* x, const void* w, const float* logits, const int* idx, const float* prob,
                              const float* dprob, int T, int H, int E, int k, int renorm, float* dl, void* dx,
                              float* dw, void* ws, int* err, cudaStream_t st) {
  const int N = router_dw_cols(E);
  const int max_chunks = router_dw_max_chunks(H);
  uint8_t* base = static_cast<uint8_t*>(ws);
  float* partial = reinterpret_cast<float*>(base);
  const size_t off_hi = al256(size_t(max_chunks) * E * H * sizeof(float));
  __nv_bfloat16* dl_hi = reinterpret_cast<__nv_bfloat16*>(base + off_hi);
  __nv_bfloat16* dl_lo = reinterpret_cast<__nv_bfloat16*>(base + off_hi + al256(size_t(T) * N * 2));
  const unsigned warps_grid = unsigned((int64_t(T) * 32 + 255) / 256);
  router_dlogits_kernel<<<warps_grid, 256, 0, st>>>(logits, idx, prob, dprob, T, E, k, renorm, dl, dl_hi, dl_lo, N,
                                                   err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  router_dx_kernel<<<warps_grid, 256, 0, st>>>(dl, idx, static_cast<const __nv_bfloat16*>(w), T, H, E, k, renorm,
                                              static_cast<__nv_bfloat16*>(dx));
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  int chunks = 0;
  e = launch_router_dw_tc(x, dl_hi, dl_lo, T, H, E, partial, max_chunks, &chunks, err, st);
  if (e != cudaSuccess) return e;
  const int64_t n = int64_t(E) * H;
  router_dw_reduce_kernel<<<unsigned((n + 255) / 256), 256, 0, st>>>(partial, n, chunks, dw);
  return cudaGetLastError();
}

}  // namespace moe
