// Top-k routing and the expert-major permutation (page "英伟达开源MoE加速神器",
// section "三板斧": tokens go to a few of many experts; page "Efficient MoE
// Training for Biological Foundation Models", section "GroupedLinear": the
// grouped call takes the tokens collected per expert plus split_sizes).
//
// Deterministic without sorting or atomics:
//   1. route_topk_kernel: one warp per 32-token group selects the top-k
//      experts of each token by exact logit comparisons and writes, per expert
//      e and group g, the 32-bit ballot mask[e][g] of the group's tokens that
//      picked e.
//   2. permute_scan_kernel: one CTA per expert scans popc(mask[e][g]) over g:
//      base[e][g] = tokens of e in groups before g; split_sizes[e] = total.
//   3. permute_scatter_kernel: row of (t, slot) = padded start of e +
//      base[e][g] + popc(mask[e][g] & lanes below t) -- ascending token order
//      inside every expert segment.
#include "kernels.cuh"

namespace moe {

constexpr int kMaxK = 8;
constexpr int kMaxE = 256;

__device__ __forceinline__ bool better(float va, int ea, float vb, int eb) {
  return va > vb || (va == vb && ea < eb);
}

__global__ void __launch_bounds__(256) route_topk_kernel(
    const float* __restrict__ logits, int T, int E, int k, int renorm,
    int* __restrict__ idx, float* __restrict__ prob, uint32_t* __restrict__ masks, int G) {
  const int lane = threadIdx.x & 31;
  const int g = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (g >= G) return;
  const int nchunk = (E + 31) >> 5;                    // <= 8 logits per lane
  int my_sel[kMaxK];
#pragma unroll
  for (int s = 0; s < kMaxK; ++s) my_sel[s] = -1;
  for (int i = 0; i < 32; ++i) {
    const int t = g * 32 + i;
    if (t >= T) break;                                 // warp-uniform
    float v[8];
    unsigned taken = 0;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int e = lane + 32 * c;
      v[c] = (c < nchunk && e < E) ? logits[(int64_t)t * E + e] : -INFINITY;
    }
    int sel_e[kMaxK];
    float sel_v[kMaxK];
#pragma unroll
    for (int s = 0; s < kMaxK; ++s) {
      sel_e[s] = -1;
      sel_v[s] = -INFINITY;
      if (s < k) {
        float bv = -INFINITY;
        int be = 0x7FFFFFFF;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int e = lane + 32 * c;
          if (c < nchunk && e < E && !((taken >> c) & 1u) && better(v[c], e, bv, be)) {
            bv = v[c];
            be = e;
          }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
          const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, off);
          if (better(ov, oe, bv, be)) {
            bv = ov;
            be = oe;
          }
        }
        sel_e[s] = be;
        sel_v[s] = bv;
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
      }
    }
    // probabilities: softmax of the selected logits (renorm) or of all E
    const float m = sel_v[0];
    float den = 0.f;
    if (renorm) {
#pragma unroll
      for (int s = 0; s < kMaxK; ++s)
        if (s < k) den += expf(sel_v[s] - m);
    } else {
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int e = lane + 32 * c;
        if (c < nchunk && e < E) den += expf(v[c] - m);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xFFFFFFFFu, den, off);
    }
#pragma unroll
    for (int s = 0; s < kMaxK; ++s) {
      if (s < k && lane == s) {
        idx[(int64_t)t * k + s] = sel_e[s];
        prob[(int64_t)t * k + s] = expf(sel_v[s] - m) / den;
      }
      if (lane == i) my_sel[s] = (s < k) ? sel_e[s] : -1;
    }
  }
  // ballot masks: bit l of mask[e][g] = token g*32+l picked expert e
  for (int e = 0; e < E; ++e) {
    bool pick = false;
#pragma unroll
    for (int s = 0; s < kMaxK; ++s) pick |= (my_sel[s] == e);
    const unsigned msk = __ballot_sync(0xFFFFFFFFu, pick);
    if (lane == 0) masks[(int64_t)e * G + g] = msk;
  }
}

// One CTA per expert: exclusive scan over groups of popc(mask).
__global__ void __launch_bounds__(1024) permute_scan_kernel(
    const uint32_t* __restrict__ masks, int G, int* __restrict__ bases, int* __restrict__ split_sizes) {
  __shared__ int warp_sums[32];
  __shared__ int carry_s;
  const int e = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) carry_s = 0;
  __syncthreads();
  for (int g0 = 0; g0 < G; g0 += 1024) {
    const int g = g0 + threadIdx.x;
    const int cnt = (g < G) ? __popc(masks[(int64_t)e * G + g]) : 0;
    int incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int ws = warp_sums[lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xFFFFFFFFu, ws, off);
        if (lane >= off) ws += o;
      }
      warp_sums[lane] = ws;                           // inclusive over warps
    }
    __syncthreads();
    const int carry = carry_s;
    const int excl = carry + (warp > 0 ? warp_sums[warp - 1] : 0) + incl - cnt;
    if (g < G) bases[(int64_t)e * G + g] = excl;
    __syncthreads();
    if (threadIdx.x == 0) carry_s = carry + warp_sums[31];
    __syncthreads();
  }
  if (threadIdx.x == 0) split_sizes[e] = carry_s;
}

// Rows of every (token, slot); padding rows of each segment get src -1, prob 0.
__global__ void __launch_bounds__(256) permute_scatter_kernel(
    const int* __restrict__ idx, const float* __restrict__ prob, int T, int k, int E, int G,
    const uint32_t* __restrict__ masks, const int* __restrict__ bases, const int* __restrict__ split_sizes,
    int* __restrict__ row_of, int* __restrict__ src_of, float* __restrict__ prob_perm, int token_blocks,
    int* err) {
  __shared__ int seg_start[kMaxE + 1];
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int e = 0; e < E; ++e) {
      seg_start[e] = acc;
      acc += (split_sizes[e] + 127) & ~127;
    }
    seg_start[E] = acc;
  }
  __syncthreads();
  if (int(blockIdx.x) < token_blocks) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    const int g = t >> 5, l = t & 31;
    for (int s = 0; s < k; ++s) {
      const int e = idx[(int64_t)t * k + s];
      if (e < 0 || e >= E) {
        report_error(err, MOE_ERR_DEVICE_BOUNDS, SITE_PERMUTE + 1);
        continue;
      }
      const uint32_t msk = masks[(int64_t)e * G + g];
      const int row = seg_start[e] + bases[(int64_t)e * G + g] + __popc(msk & ((1u << l) - 1u));
      row_of[(int64_t)t * k + s] = row;
      src_of[row] = t;
      prob_perm[row] = prob[(int64_t)t * k + s];
    }
  } else {
    const int e = blockIdx.x - token_blocks;
    const int r0 = seg_start[e] + split_sizes[e];
    for (int r = r0 + threadIdx.x; r < seg_start[e + 1]; r += blockDim.x) {
      src_of[r] = -1;
      prob_perm[r] = 0.f;
    }
  }
}

cudaError_t launch_route_permute(const float* logits, int T, int E, int k, int renorm, int* idx, float* prob,
                                 uint32_t* masks, int* bases, int* split_sizes, int* row_of, int* src_of,
                                 float* prob_perm, int* err, cudaStream_t st) {
  const int G = (T + 31) / 32;
  route_topk_kernel<<<(G * 32 + 255) / 256, 256, 0, st>>>(logits, T, E, k, renorm, idx, prob, masks, G);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  permute_scan_kernel<<<E, 1024, 0, st>>>(masks, G, bases, split_sizes);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int token_blocks = (T + 255) / 256;
  permute_scatter_kernel<<<token_blocks + E, 256, 0, st>>>(idx, prob, T, k, E, G, masks, bases, split_sizes,
                                                           row_of, src_of, prob_perm, token_blocks, err);
  return cudaGetLastError();
}

}  // namespace moe
