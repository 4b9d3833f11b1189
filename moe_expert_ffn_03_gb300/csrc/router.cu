// Linear router on both sides: logits = x W_r^T, and the backward through the
// top-k softmax (page "英伟达开源MoE加速神器", section "三板斧": tokens are
// routed to a few experts; page "Efficient MoE Training for Biological
// Foundation Models", section "MXFP8与融合MLP": the router probabilities scale
// the SwiGLU output).  The forward runs on the tensor cores; the backward
// kernels run on the CUDA cores with fixed summation orders (deterministic
// results):
//   forward                 logits = x W_r^T on the tensor cores: the grouped GEMM
//                           engine with bf16 operands, one segment of T rows,
//                           N = E, f32 logits (rows and columns past T and E masked);
//   router_dlogits_kernel   one warp per token, straight-through top-k softmax;
//   router_dx_kernel        dx[t] += sum_e dl[t][e] W_r[e] (bf16 in place);
//   router_dw_partial/reduce dW_r = dl^T x over fixed token chunks, summed in
//                           chunk order; each chunk's CTA stages 16-token
//                           slices of dl and x in shared memory and keeps a
//                           4x4 block of outputs per thread.
#include "kernels.cuh"

namespace moe {

__host__ __device__ inline int router_et(int E) { return E <= 8 ? 8 : E <= 16 ? 16 : E <= 32 ? 32 : 64; }

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

// dW_r tiles: ET experts x (4096 / ET) hidden columns per CTA, 256 threads with a
// 4 x 4 block each; tokens in slices of RT_DW_TS staged in shared memory.  The
// number of token chunks depends on E and H only (it sizes the workspace): enough
// CTAs to fill the GPU a few times over, between 8 and 64.
constexpr int RT_DW_TS = 16;

inline int router_dw_chunks(int E, int H) {
  const int et = router_et(E), ht = 4096 / et;
  const int tiles = ((H + ht - 1) / ht) * ((E + et - 1) / et);
  const int c = (600 + tiles - 1) / tiles;
  return c < 8 ? 8 : c > 64 ? 64 : c;
}

// partial[c][e][h] = sum over the tokens of chunk c (ascending) of dl[t][e] * x[t][h].
template <int ET>
__global__ void __launch_bounds__(256) router_dw_partial_kernel(const float* __restrict__ dl,
                                                                const __nv_bfloat16* __restrict__ x, int T, int H,
                                                                int E, int chunks, float* __restrict__ partial) {
  constexpr int HT = 4096 / ET;              // hidden columns of the tile
  constexpr int TH = HT / 4;                 // threads along h (4 columns each)
  __shared__ __align__(16) float dls[RT_DW_TS][ET];
  __shared__ __align__(16) __nv_bfloat16 xs[RT_DW_TS][HT];
  const int h0 = blockIdx.x * HT, e0 = blockIdx.y * ET, c = blockIdx.z;
  const int hg = threadIdx.x % TH, eg = threadIdx.x / TH;   // columns h0+4hg.., experts e0+4eg..
  const int per = (T + chunks - 1) / chunks;
  const int ta = min(T, c * per), tb = min(T, ta + per);
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int ts = ta; ts < tb; ts += RT_DW_TS) {
    __syncthreads();
    // dl slice: RT_DW_TS rows x ET floats (zero past T or E)
    for (int i = threadIdx.x; i < RT_DW_TS * ET; i += 256) {
      const int r = i / ET, e = i % ET;
      const int t = ts + r;
      dls[r][e] = (t < tb && e0 + e < E) ? dl[int64_t(t) * E + e0 + e] : 0.f;
    }
    // x slice: RT_DW_TS rows x HT bf16, 8 at a time (H is a multiple of 8)
    for (int i = threadIdx.x; i < RT_DW_TS * (HT / 8); i += 256) {
      const int r = i / (HT / 8), c8 = i % (HT / 8);
      const int t = ts + r, h = h0 + c8 * 8;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (t < tb && h < H) v = *reinterpret_cast<const uint4*>(x + int64_t(t) * H + h);
      *reinterpret_cast<uint4*>(&xs[r][c8 * 8]) = v;
    }
    __syncthreads();
#pragma unroll 4
    for (int r = 0; r < RT_DW_TS; ++r) {
      const float4 d = *reinterpret_cast<const float4*>(&dls[r][4 * eg]);
      const uint2 xv = *reinterpret_cast<const uint2*>(&xs[r][4 * hg]);
      const float xf[4] = {bf16_lo(xv.x), bf16_hi(xv.x), bf16_lo(xv.y), bf16_hi(xv.y)};
      const float df[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] += df[i] * xf[j];
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = e0 + 4 * eg + i;
    const int h = h0 + 4 * hg;
    if (e >= E || h >= H) continue;
    *reinterpret_cast<float4*>(partial + (int64_t(c) * E + e) * H + h) =
        make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
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

size_t router_partial_bytes(int E, int H) { return size_t(router_dw_chunks(E, H)) * E * H * sizeof(float); }

cudaError_t launch_router_fwd(const void* x, const void* w, int T, int H, int E, float* logits, int* err,
                              cudaStream_t st, char* msg, size_t msg_len) {
  // one segment of T rows (E = 1 in the grouped engine's terms), N = the router's experts
  GemmArgs g{};
  g.mode = 0;
  g.E = 1;
  g.split_sizes = nullptr;
  g.rows_limit = T;
  g.K = H;
  g.N = E;
  g.n_tiles = (E + 255) / 256;
  g.b_rows_per_expert = E;
  g.cap = (int64_t(T) + 127) / 128 * 128;
  g.out_f32 = logits;
  g.ldo = E;
  g.err = err;
  return launch_grouped_gemm(EPI_B16_F32_OUT, g, x, T, H, w, E, H, (g.cap / 128) * g.n_tiles, st, msg, msg_len);
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
  const int chunks = router_dw_chunks(E, H);
  const int et = router_et(E), ht = 4096 / et;
  const dim3 grid(unsigned((H + ht - 1) / ht), unsigned((E + et - 1) / et), unsigned(chunks));
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  switch (et) {
    case 8: router_dw_partial_kernel<8><<<grid, 256, 0, st>>>(dl, xb, T, H, E, chunks, partial); break;
    case 16: router_dw_partial_kernel<16><<<grid, 256, 0, st>>>(dl, xb, T, H, E, chunks, partial); break;
    case 32: router_dw_partial_kernel<32><<<grid, 256, 0, st>>>(dl, xb, T, H, E, chunks, partial); break;
    default: router_dw_partial_kernel<64><<<grid, 256, 0, st>>>(dl, xb, T, H, E, chunks, partial); break;
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t n = int64_t(E) * H;
  router_dw_reduce_kernel<<<unsigned((n + 255) / 256), 256, 0, st>>>(partial, n, chunks, dw);
  return cudaGetLastError();
}

}  // namespace moe
