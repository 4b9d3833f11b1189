// Top-k routing and the expert-major permutation (page "英伟达开源MoE加速神器",
// section "三板斧": tokens go to a few of many experts; page "Efficient MoE
// Training for Biological Foundation Models", section "GroupedLinear": the
// grouped call takes the tokens collected per expert plus split_sizes).
//
// Deterministic without sorting (the results never depend on the order of atomics):
//   1. route_topk_kernel: one thread per token keeps its k best (logit,
//      expert) pairs in a sorted register list (exact comparisons, ties to the
//      lower expert id); the warp then writes, per expert e and 32-token group
//      g, the bit mask[e][g] of the group's tokens that picked e.  With 32 or
//      more experts and masks past the one-launch bound, route_topk_quad_kernel
//      does the same with four lanes per token.
//   2. the per-expert scan of popc(mask[e][g]) over g: base[e][g] = tokens of e
//      in groups before g; split_sizes[e] = total.  While the masks hold at most
//      16384 words, the block of route_topk_kernel that takes the last ticket
//      (one atomicInc per block) runs it in the same launch; past that bound,
//      permute_scan_kernel, one CTA per expert.
//   3. the rows: row of (t, slot) = padded start of e + base[e][g] +
//      popc(mask[e][g] & lanes below t) -- ascending token order inside every
//      expert segment.  The row quantizer computes them while it gathers x
//      (quantize.cu); permute_scatter_kernel writes the maps alone.
#include "kernels.cuh"

namespace moe {

constexpr int kMaxK = 8;
constexpr int kMaxE = kMaxExperts;

// Total order of (logit, expert): larger logit first, ties to the lower expert id.
// A NaN logit ranks below every number (-inf included) and NaNs tie among
// themselves, so a row with fewer than k non-NaN logits still fills its k slots
// with real experts (the NaN ones, lowest ids first).  +0 and -0 tie.
__device__ __forceinline__ bool better(float va, int ea, float vb, int eb) {
  const bool na = va != va, nb = vb != vb;
  if (na != nb) return nb;
  if (!na && va != vb) return va > vb;
  return ea < eb;
}

constexpr int RT_THREADS = 128;
// Top-k and the per-expert scan as one launch (the last block scans) while the masks are
// at most RS_SCAN_MAX_WORDS words; larger ones get the scan kernel with one CTA per expert.
constexpr int RS_THREADS = 512;
constexpr int RS_SCAN_MAX_WORDS = 16384;

// Bubble (v, e) into the sorted list (best first); the last entry falls off.
__device__ __forceinline__ void topk_insert(float v, int e, float (&sv)[kMaxK], int (&se)[kMaxK]) {
#pragma unroll
  for (int s = 0; s < kMaxK; ++s) {
    if (better(v, e, sv[s], se[s])) {
      const float tv = sv[s];
      const int te = se[s];
      sv[s] = v;
      se[s] = e;
      v = tv;
      e = te;
    }
  }
}

// Exclusive scan over groups g of popc(mask[e][g]) for the experts e = warp, warp + nwarps, ...
// (one warp per expert, 128 groups a step, 4 consecutive groups a lane): base[e][g] and
// split_sizes[e].  Loads bypass L1: the masks were written by other blocks of this launch.
__device__ __forceinline__ void scan_experts_by_warps(const uint32_t* masks, int G, int E, int warp, int nwarps,
                                                      int lane, int* bases, int* split_sizes) {
  for (int e = warp; e < E; e += nwarps) {
    const uint32_t* m = masks + (int64_t)e * G;
    int* b = bases + (int64_t)e * G;
    int carry = 0;
    for (int g0 = 0; g0 < G; g0 += 128) {
      int c[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int g = g0 + 4 * lane + i;
        c[i] = g < G ? __popc(__ldcg(m + g)) : 0;
      }
      const int local = c[0] + c[1] + c[2] + c[3];
      int incl = local;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += o;
      }
      int run = carry + incl - local;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int g = g0 + 4 * lane + i;
        if (g < G) b[g] = run;
        run += c[i];
      }
      carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (lane == 0) split_sizes[e] = carry;
  }
}

// NT threads a block, one token a thread.  With SCAN the block that finishes last (a
// ticket taken after each block's masks are written and fenced) also runs the per-expert
// scan, so top-k and scan are one launch; atomicInc wraps the ticket back to 0 at the
// last block, ready for the next launch.  Nothing waits on another block.
template <int NT, bool SCAN>
__global__ void __launch_bounds__(NT) route_topk_kernel(
    const float* __restrict__ logits, int T, int E, int k, int renorm,
    int* __restrict__ idx, float* __restrict__ prob, uint32_t* __restrict__ masks, int G, int* err,
    unsigned* ticket, int* __restrict__ bases, int* __restrict__ split_sizes) {
  pdl_wait();                 // may start early (programmatic stream serialization)
  pdl_launch_dependents();
  __shared__ uint32_t smask[NT / 32][kMaxE];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int t = blockIdx.x * NT + threadIdx.x;
  const int g = t >> 5;                                // the warp's 32-token group
  if (g < G) {                                         // warp-uniform
    for (int e = lane; e < E; e += 32) smask[w][e] = 0u;
    __syncwarp();
    if (t < T) {
      float sv[kMaxK];
      int se[kMaxK];
#pragma unroll
      for (int s = 0; s < kMaxK; ++s) {
        sv[s] = __int_as_float(0x7FFFFFFF);            // NaN with the largest id: below every real entry
        se[s] = 0x7FFFFFFF;
      }
      const float* row = logits + (int64_t)t * E;
      if ((E & 3) == 0) {
        const float4* row4 = reinterpret_cast<const float4*>(row);
        for (int e4 = 0; e4 < (E >> 2); ++e4) {
          const float4 q = row4[e4];
          topk_insert(q.x, 4 * e4 + 0, sv, se);
          topk_insert(q.y, 4 * e4 + 1, sv, se);
          topk_insert(q.z, 4 * e4 + 2, sv, se);
          topk_insert(q.w, 4 * e4 + 3, sv, se);
        }
      } else {
        for (int e = 0; e < E; ++e) topk_insert(row[e], e, sv, se);
      }
      // probabilities: softmax of the selected logits (renorm) or of all E
      const float m = sv[0];
      float den = 0.f;
      if (renorm) {
#pragma unroll
        for (int s = 0; s < kMaxK; ++s)
          if (s < k) den += expf(sv[s] - m);
      } else {
        for (int e = 0; e < E; ++e) den += expf(row[e] - m);
      }
#pragma unroll
      for (int s = 0; s < kMaxK; ++s) {
        if (s < k) {
          // k <= E, so the list holds k real experts; the check keeps a broken invariant
          // from turning into a shared-memory access out of bounds
          if (se[s] < 0 || se[s] >= E) {
            report_error(err, MOE_ERR_DEVICE_BOUNDS, SITE_ROUTE);
            idx[(int64_t)t * k + s] = -1;
            prob[(int64_t)t * k + s] = 0.f;
            continue;
          }
          idx[(int64_t)t * k + s] = se[s];
          prob[(int64_t)t * k + s] = expf(sv[s] - m) / den;
          atomicOr(&smask[w][se[s]], 1u << lane);
        }
      }
    }
    __syncwarp();
    // bit l of mask[e][g] = token g*32+l picked expert e
    for (int e = lane; e < E; e += 32) masks[(int64_t)e * G + g] = smask[w][e];
  }
  if (SCAN) {
    __shared__ bool last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last = atomicInc(ticket, gridDim.x - 1) == gridDim.x - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();
    scan_experts_by_warps(masks, G, E, w, NT / 32, lane, bases, split_sizes);
  }
}

// Many experts: four lanes per token.  Lane s of a token's quad keeps the sorted top-k of
// experts s, s+4, s+8, ... (ascending, so a quad reads 16 contiguous bytes at a time), then
// two shuffle rounds merge the quad's lists (partner lane ^1, then ^2): every lane ends with
// the token's k best in the total order, the same list one lane over all E would hold, so
// idx and the renormalised probabilities equal route_topk_kernel's bit for bit; without
// renormalisation lane 0 sums the row's exponentials in expert order, as that kernel does.
// A 128-thread block is one 32-token group; its masks are gathered in shared memory.
constexpr int RQ_THREADS = 128;                      // 32 tokens x 4 lanes
__global__ void __launch_bounds__(RQ_THREADS) route_topk_quad_kernel(
    const float* __restrict__ logits, int T, int E, int k, int renorm,
    int* __restrict__ idx, float* __restrict__ prob, uint32_t* __restrict__ masks, int G, int* err) {
  pdl_wait();                 // may start early (programmatic stream serialization)
  pdl_launch_dependents();
  __shared__ uint32_t smask[kMaxE];
  const int lane = threadIdx.x & 31, sub = lane & 3;
  const int tl = threadIdx.x >> 2;                   // token of this quad inside the group (0..31)
  const int g = blockIdx.x;
  const int t = g * 32 + tl;
  for (int e = threadIdx.x; e < E; e += RQ_THREADS) smask[e] = 0u;
  __syncthreads();
  float sv[kMaxK];
  int se[kMaxK];
#pragma unroll
  for (int s = 0; s < kMaxK; ++s) {
    sv[s] = __int_as_float(0x7FFFFFFF);              // NaN with the largest id: below every real entry
    se[s] = 0x7FFFFFFF;
  }
  const float* row = logits + (int64_t)t * E;
  if (t < T) {
#pragma unroll 4
    for (int e = sub; e < E; e += 4) topk_insert(row[e], e, sv, se);
  }
#pragma unroll
  for (int m = 1; m <= 2; m <<= 1) {
    float pv[kMaxK];
    int pe[kMaxK];
#pragma unroll
    for (int s = 0; s < kMaxK; ++s) {
      pv[s] = __shfl_xor_sync(0xFFFFFFFFu, sv[s], m);
      pe[s] = __shfl_xor_sync(0xFFFFFFFFu, se[s], m);
    }
#pragma unroll
    for (int s = 0; s < kMaxK; ++s)
      if (s < k) topk_insert(pv[s], pe[s], sv, se);
  }
  if (t < T && sub == 0) {
    const float m = sv[0];
    float den = 0.f;
    if (renorm) {
#pragma unroll
      for (int s = 0; s < kMaxK; ++s)
        if (s < k) den += expf(sv[s] - m);
    } else {
      for (int e = 0; e < E; ++e) den += expf(row[e] - m);
    }
#pragma unroll
    for (int s = 0; s < kMaxK; ++s) {
      if (s < k) {
        if (se[s] < 0 || se[s] >= E) {
          report_error(err, MOE_ERR_DEVICE_BOUNDS, SITE_ROUTE);
          idx[(int64_t)t * k + s] = -1;
          prob[(int64_t)t * k + s] = 0.f;
          continue;
        }
        idx[(int64_t)t * k + s] = se[s];
        prob[(int64_t)t * k + s] = expf(sv[s] - m) / den;
        atomicOr(&smask[se[s]], 1u << tl);
      }
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += RQ_THREADS) masks[(int64_t)e * G + g] = smask[e];
}

// One CTA per expert: exclusive scan over groups of popc(mask).
__global__ void __launch_bounds__(1024) permute_scan_kernel(
    const uint32_t* __restrict__ masks, int G, int* __restrict__ bases, int* __restrict__ split_sizes) {
  pdl_wait();                 // may start early (programmatic stream serialization)
  pdl_launch_dependents();
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
  pdl_wait();                 // may start early (programmatic stream serialization)
  pdl_launch_dependents();
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
        row_of[(int64_t)t * k + s] = -1;                // later kernels' row checks catch the slot
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

// Ballot masks of given expert ids (the routing-free permutation): warp w of a CTA takes
// the 32-token group g; bit l of mask[e][g] = token g*32+l has a slot with expert e.
// An id outside 0..E-1 is recorded and its slot skipped (the scatter marks it -1).
__global__ void __launch_bounds__(RT_THREADS) idx_masks_kernel(const int* __restrict__ idx, int T, int E, int k,
                                                               uint32_t* __restrict__ masks, int G, int* err) {
  pdl_wait();                 // may start early (programmatic stream serialization)
  pdl_launch_dependents();
  __shared__ uint32_t smask[RT_THREADS / 32][kMaxE];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int t = blockIdx.x * RT_THREADS + threadIdx.x;
  const int g = t >> 5;
  if (g >= G) return;                                  // warp-uniform
  for (int e = lane; e < E; e += 32) smask[w][e] = 0u;
  __syncwarp();
  if (t < T) {
    for (int s = 0; s < k; ++s) {
      const int e = idx[(int64_t)t * k + s];
      if (e < 0 || e >= E) {
        report_error(err, MOE_ERR_DEVICE_BOUNDS, SITE_ROUTE + 1);
        continue;
      }
      atomicOr(&smask[w][e], 1u << lane);
    }
  }
  __syncwarp();
  for (int e = lane; e < E; e += 32) masks[(int64_t)e * G + g] = smask[w][e];
}

cudaError_t launch_permute_from_idx(const int* idx, const float* prob, int T, int E, int k, uint32_t* masks,
                                    int* bases, int* split_sizes, int* row_of, int* src_of, float* prob_perm,
                                    int* err, cudaStream_t st) {
  const int G = (T + 31) / 32;
  launch_pdl(idx_masks_kernel, dim3((G * 32 + RT_THREADS - 1) / RT_THREADS), dim3(RT_THREADS), 0, st,
             idx, T, E, k, masks, G, err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  launch_pdl(permute_scan_kernel, dim3(E), dim3(1024), 0, st,
             masks, G, bases, split_sizes);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int token_blocks = (T + 255) / 256;
  launch_pdl(permute_scatter_kernel, dim3(token_blocks + E), dim3(256), 0, st,
             idx, prob, T, k, E, G, masks, bases, split_sizes, row_of, src_of, prob_perm, token_blocks, err);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------
bool route_scan_fused(int T, int E) { return int64_t(E) * ((int64_t(T) + 31) / 32) <= RS_SCAN_MAX_WORDS; }

cudaError_t launch_route_scan(const float* logits, int T, int E, int k, int renorm, int* idx, float* prob,
                              uint32_t* masks, int* bases, int* split_sizes, unsigned* ticket, int* err,
                              cudaStream_t st) {
  const int G = (T + 31) / 32;
  if (route_scan_fused(T, E)) {
    launch_pdl(route_topk_kernel<RS_THREADS, true>, dim3((G * 32 + RS_THREADS - 1) / RS_THREADS), dim3(RS_THREADS),
               0, st,
               logits, T, E, k, renorm, idx, prob, masks, G, err, ticket, bases, split_sizes);
    return cudaGetLastError();
  }
  if (E >= 32)
    launch_pdl(route_topk_quad_kernel, dim3(G), dim3(RQ_THREADS), 0, st,
               logits, T, E, k, renorm, idx, prob, masks, G, err);
  else
    launch_pdl(route_topk_kernel<RT_THREADS, false>, dim3((G * 32 + RT_THREADS - 1) / RT_THREADS), dim3(RT_THREADS),
               0, st,
               logits, T, E, k, renorm, idx, prob, masks, G, err, nullptr, nullptr, nullptr);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  launch_pdl(permute_scan_kernel, dim3(E), dim3(1024), 0, st,
             masks, G, bases, split_sizes);
  return cudaGetLastError();
}

cudaError_t launch_route_permute(const float* logits, int T, int E, int k, int renorm, int* idx, float* prob,
                                 uint32_t* masks, int* bases, int* split_sizes, int* row_of, int* src_of,
                                 float* prob_perm, unsigned* ticket, int* err, cudaStream_t st) {
  const int G = (T + 31) / 32;
  cudaError_t e = launch_route_scan(logits, T, E, k, renorm, idx, prob, masks, bases, split_sizes, ticket, err, st);
  if (e != cudaSuccess) return e;
  const int token_blocks = (T + 255) / 256;
  launch_pdl(permute_scatter_kernel, dim3(token_blocks + E), dim3(256), 0, st,
             idx, prob, T, k, E, G, masks, bases, split_sizes, row_of, src_of, prob_perm, token_blocks, err);
  return cudaGetLastError();
}

}  // namespace moe
