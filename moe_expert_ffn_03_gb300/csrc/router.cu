// Linear router on both sides: logits = x W_r^T, and the backward through the
// top-k softmax (page "英伟达开源MoE加速神器", section "三板斧": tokens are
// routed to a few experts; page "Efficient MoE Training for Biological
// Foundation Models", section "MXFP8与融合MLP": the router probabilities scale
// the SwiGLU output).  N = E is small (<= 256), so these are bandwidth-bound
// CUDA-core kernels with fixed summation orders (deterministic results):
//   router_fwd_kernel       32 tokens x all experts per CTA, x and W_r chunks in
//                           shared memory, fp32 sums in ascending h;
//   router_dlogits_kernel   one warp per token, straight-through top-k softmax;
//   router_dx_kernel        dx[t] += sum_e dl[t][e] W_r[e] (bf16 in place);
//   router_dw_partial/reduce dW_r = dl^T x over fixed token chunks, summed in
//                           chunk order.
#include "kernels.cuh"

namespace moe {

constexpr int RT_TOK = 32;       // tokens per CTA of the forward
constexpr int RT_HC = 128;       // hidden chunk
constexpr int RT_XP = RT_TOK + 1;

template <int EPT>
__global__ void __launch_bounds__(256) router_fwd_kernel(const __nv_bfloat16* __restrict__ x,
                                                         const __nv_bfloat16* __restrict__ w, int T, int H, int E,
                                                         float* __restrict__ logits) {
  extern __shared__ __align__(16) float rsm[];
  float* xs = rsm;                                                     // [RT_HC][RT_XP]
  __nv_bfloat16* ws = reinterpret_cast<__nv_bfloat16*>(rsm + RT_HC * RT_XP);  // [E][RT_HC]
  const int t0 = blockIdx.x * RT_TOK;
  const int tl = threadIdx.x & 31, eg = threadIdx.x >> 5;
  float acc[EPT];
#pragma unroll
  for (int j = 0; j < EPT; ++j) acc[j] = 0.f;
  for (int h0 = 0; h0 < H; h0 += RT_HC) {
    __syncthreads();
    for (int i = threadIdx.x; i < RT_TOK * (RT_HC / 8); i += 256) {
      const int r = i / (RT_HC / 8), c8 = i % (RT_HC / 8);
      const int t = t0 + r;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (t < T) v = *reinterpret_cast<const uint4*>(x + int64_t(t) * H + h0 + c8 * 8);
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        xs[(c8 * 8 + 2 * q) * RT_XP + r] = bf16_lo(wv[q]);
        xs[(c8 * 8 + 2 * q + 1) * RT_XP + r] = bf16_hi(wv[q]);
      }
    }
    for (int i = threadIdx.x; i < E * (RT_HC / 8); i += 256) {
      const int e = i / (RT_HC / 8), c8 = i % (RT_HC / 8);
      *reinterpret_cast<uint4*>(ws + e * RT_HC + c8 * 8) =
          *reinterpret_cast<const uint4*>(w + int64_t(e) * H + h0 + c8 * 8);
    }
    __syncthreads();
    for (int h = 0; h < RT_HC; ++h) {
      const float xv = xs[h * RT_XP + tl];
#pragma unroll
      for (int j = 0; j < EPT; ++j) {
        const int e = eg + 8 * j;
        if (e < E) acc[j] += xv * __bfloat162float(ws[e * RT_HC + h]);
      }
    }
  }
  const int t = t0 + tl;
  if (t < T) {
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      const int e = eg + 8 * j;
      if (e < E) logits[int64_t(t) * E + e] = acc[j];
    }
  }
}

// One warp per token.  renormalize: dl[e_j] = p_j (dp_j - sum_i p_i dp_i), 0 elsewhere;
// plain softmax: dl[e] = s_e (g_e - sum_j p_j dp_j) with g the dprob scattered to idx.
__global__ void __launch_bounds__(256) router_dlogits_kernel(const float* __restrict__ logits,
                                                             const int* __restrict__ idx,
                                                             const float* __restrict__ prob,
                                                             const float* __restrict__ dprob, int T, int E, int k,
                                                             int renorm, float* __restrict__ dl, int* err) {
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
  for (int e = lane; e < E; e += 32) {
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
    float v;
    if (renorm) v = sel ? pe * (g - pdp) : 0.f;
    else v = expf(lrow[e] - m) / z * (g - pdp);
    dl[t * E + e] = v;
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

constexpr int RT_DW_CHUNKS = 8;

// partial[c][e][h] = sum over the tokens of chunk c of dl[t][e] * x[t][h]; CTA = 32
// hidden columns x all experts of one token chunk.
template <int EPT>
__global__ void __launch_bounds__(256) router_dw_partial_kernel(const float* __restrict__ dl,
                                                                const __nv_bfloat16* __restrict__ x, int T, int H,
                                                                int E, float* __restrict__ partial) {
  const int h = blockIdx.x * 32 + (threadIdx.x & 31);
  const int eg = threadIdx.x >> 5;
  const int c = blockIdx.y;
  const int per = (T + RT_DW_CHUNKS - 1) / RT_DW_CHUNKS;
  const int ta = c * per, tb = min(T, ta + per);
  float acc[EPT];
#pragma unroll
  for (int j = 0; j < EPT; ++j) acc[j] = 0.f;
  for (int t = ta; t < tb; ++t) {
    const float xv = __bfloat162float(x[int64_t(t) * H + h]);
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      const int e = eg + 8 * j;
      if (e < E) acc[j] += dl[int64_t(t) * E + e] * xv;
    }
  }
#pragma unroll
  for (int j = 0; j < EPT; ++j) {
    const int e = eg + 8 * j;
    if (e < E) partial[(int64_t(c) * E + e) * H + h] = acc[j];
  }
}

__global__ void __launch_bounds__(256) router_dw_reduce_kernel(const float* __restrict__ partial, int64_t n,
                                                               float* __restrict__ dw) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float s = 0.f;
  for (int c = 0; c < RT_DW_CHUNKS; ++c) s += partial[int64_t(c) * n + i];
  dw[i] = s;
}

namespace {
template <template <int> class K, typename... A>
cudaError_t dispatch_ept(int E, dim3 grid, size_t smem, cudaStream_t st, A... args) {
  auto go = [&](auto kernel) {
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
      if (e != cudaSuccess) return e;
    }
    kernel<<<grid, 256, smem, st>>>(args...);
    return cudaGetLastError();
  };
  const int ept = (E + 7) / 8;
  if (ept <= 1) return go(K<1>::fn);
  if (ept <= 2) return go(K<2>::fn);
  if (ept <= 4) return go(K<4>::fn);
  if (ept <= 8) return go(K<8>::fn);
  if (ept <= 16) return go(K<16>::fn);
  return go(K<32>::fn);
}
template <int EPT>
struct FwdK {
  static constexpr auto fn = router_fwd_kernel<EPT>;
};
template <int EPT>
struct DwK {
  static constexpr auto fn = router_dw_partial_kernel<EPT>;
};
}  // namespace

size_t router_partial_bytes(int E, int H) { return size_t(RT_DW_CHUNKS) * E * H * sizeof(float); }

cudaError_t launch_router_fwd(const void* x, const void* w, int T, int H, int E, float* logits, cudaStream_t st) {
  const size_t smem = size_t(RT_HC) * RT_XP * sizeof(float) + size_t(E) * RT_HC * sizeof(__nv_bfloat16);
  dim3 grid((T + RT_TOK - 1) / RT_TOK);
  return dispatch_ept<FwdK>(E, grid, smem, st, static_cast<const __nv_bfloat16*>(x),
                            static_cast<const __nv_bfloat16*>(w), T, H, E, logits);
}

cudaError_t launch_router_bwd(const void* x, const void* w, const float* logits, const int* idx, const float* prob,
                              const float* dprob, int T, int H, int E, int k, int renorm, float* dl, void* dx,
                              float* dw, float* partial, int* err, cudaStream_t st) {
  const unsigned warps_grid = unsigned((int64_t(T) * 32 + 255) / 256);
  router_dlogits_kernel<<<warps_grid, 256, 0, st>>>(logits, idx, prob, dprob, T, E, k, renorm, dl, err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  router_dx_kernel<<<warps_grid, 256, 0, st>>>(dl, idx, static_cast<const __nv_bfloat16*>(w), T, H, E, k, renorm,
                                              static_cast<__nv_bfloat16*>(dx));
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = dispatch_ept<DwK>(E, dim3(H / 32, RT_DW_CHUNKS), 0, st, static_cast<const float*>(dl),
                        static_cast<const __nv_bfloat16*>(x), T, H, E, partial);
  if (e != cudaSuccess) return e;
  const int64_t n = int64_t(E) * H;
  router_dw_reduce_kernel<<<unsigned((n + 255) / 256), 256, 0, st>>>(partial, n, dw);
  return cudaGetLastError();
}

}  // namespace moe
