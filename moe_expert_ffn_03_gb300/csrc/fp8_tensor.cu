// Per-tensor FP8 with dynamic scaling (page "英伟达开源MoE加速神器", section
// "3. Transformer Engine：FP8 训练加速": the Hopper FP8 recipe scales each
// tensor by its current range; page "Efficient MoE Training for Biological
// Foundation Models", section "MoE训练的瓶颈与TE的对应能力": FP8 keeps one scale
// per tensor where MXFP8 keeps one per 32 values).
//
// One scale per operand tensor of each expert's GEMM: s = 448 / amax (float32,
// IEEE division; 1 for an all-zero tensor), code = RNE_E4M3(v * s) saturating.
// The amax kernels keep the maximum as float bits (non-negative floats order
// like their bit patterns), so atomicMax on them is exact and order-free.
// All kernels are HBM-bound: the amax passes read their input once, the
// quantize passes read it once more and write one byte per element.
#include "kernels.cuh"

namespace moe {
namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;

// max of the |v| patterns of 8 packed bf16 values, both halves at once
__device__ __forceinline__ uint32_t vmax_abs8(uint32_t m2, const uint4& v) {
  m2 = __vmaxu2(m2, v.x & 0x7FFF7FFFu);
  m2 = __vmaxu2(m2, v.y & 0x7FFF7FFFu);
  m2 = __vmaxu2(m2, v.z & 0x7FFF7FFFu);
  return __vmaxu2(m2, v.w & 0x7FFF7FFFu);
}

// the larger half of a packed max, as the float bits of that bf16 value
__device__ __forceinline__ uint32_t halves_max(uint32_t m2) { return max(m2 << 16, m2 & 0xFFFF0000u); }

// 8 packed bf16 values times s -> 8 E4M3 codes (value 0 in the low byte)
__device__ __forceinline__ uint2 t8_codes8(const uint4& v, float s) {
  uint2 q;
  q.x = cvt_e4m3x2(bf16_lo(v.x) * s, bf16_hi(v.x) * s) | (cvt_e4m3x2(bf16_lo(v.y) * s, bf16_hi(v.y) * s) << 16);
  q.y = cvt_e4m3x2(bf16_lo(v.z) * s, bf16_hi(v.z) * s) | (cvt_e4m3x2(bf16_lo(v.w) * s, bf16_hi(v.w) * s) << 16);
  return q;
}

// ---- amax over each expert's routed token rows of x -------------------------------
// One warp per token (8 tokens per warp, 8 warps per block): the row max is
// raised into the block's per-expert maxima in shared memory for each of the
// token's k experts, and the block then raises the global ones.
constexpr int AT_WARPS = 8, AT_TOKENS_PER_WARP = 8;

__global__ void __launch_bounds__(AT_WARPS * 32) t8_amax_tokens_kernel(
    const __nv_bfloat16* __restrict__ x, int T, int H, const int* __restrict__ idx, int k, int E,
    uint32_t* __restrict__ amax, int* err) {
  __shared__ uint32_t s_amax[256];
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_amax[e] = 0u;
  __syncthreads();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int t0 = (blockIdx.x * AT_WARPS + w) * AT_TOKENS_PER_WARP;
  for (int i = 0; i < AT_TOKENS_PER_WARP; ++i) {
    const int t = t0 + i;
    if (t >= T) break;                                // warp-uniform
    const uint4* row = reinterpret_cast<const uint4*>(x + int64_t(t) * H);
    uint32_t m2 = 0;
#pragma unroll 4
    for (int c = lane; c < H / 8; c += 32) m2 = vmax_abs8(m2, row[c]);
    const uint32_t m = __reduce_max_sync(kFull, halves_max(m2));
    if (lane < k) {
      const int e = idx[int64_t(t) * k + lane];
      if (e < 0 || e >= E)
        report_error(err, MOE_ERR_DEVICE_BOUNDS, SITE_QUANT + 10);
      else
        atomicMax(&s_amax[e], m);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (s_amax[e] != 0u) atomicMax(&amax[e], s_amax[e]);
}

// ---- codes of x's token rows, scattered to the k permuted rows ----------------------
// One warp per token; lane j < k holds slot j's row and scale (shuffled to the
// warp once).  A warp writes 256 contiguous codes of a row per store step.
__global__ void __launch_bounds__(256) t8_quant_tokens_kernel(
    const __nv_bfloat16* __restrict__ x, int T, int H, const int* __restrict__ idx, const int* __restrict__ row_of,
    int k, int E, int64_t cap, const uint32_t* __restrict__ amax, uint8_t* __restrict__ codes, int* err) {
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  int my_row = 0;
  float my_s = 1.0f;
  bool bad = false;
  if (lane < k) {
    const int e = idx[t * k + lane];
    const int r = row_of[t * k + lane];
    bad = e < 0 || e >= E || r < 0 || r >= cap;
    if (!bad) {
      my_row = r;
      my_s = t8_scale(amax[e]);
    }
  }
  if (__any_sync(kFull, bad)) {
    if (lane == 0) report_error(err, MOE_ERR_DEVICE_BOUNDS, SITE_QUANT + 11);
    return;
  }
  int rows[8];
  float sc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    rows[j] = __shfl_sync(kFull, my_row, j);
    sc[j] = __shfl_sync(kFull, my_s, j);
  }
  const uint4* src = reinterpret_cast<const uint4*>(x + t * H);
  for (int c = lane; c < H / 8; c += 32) {
    const uint4 v = src[c];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < k) *reinterpret_cast<uint2*>(codes + int64_t(rows[j]) * H + int64_t(c) * 8) = t8_codes8(v, sc[j]);
  }
}

// ---- per-slice amax and codes of a batch of tensors (the experts' weights) -------------
// Src: StackedSrc or ExpertSrc (one pointer per expert's tensor).
template <class Src>
__global__ void __launch_bounds__(256) t8_amax_batches_kernel(const __grid_constant__ Src src, int64_t per_batch,
                                                              uint32_t* __restrict__ amax) {
  __shared__ uint32_t s_warp[8];
  const int64_t b = blockIdx.y;
  const uint4* p = reinterpret_cast<const uint4*>(src.mat(b));
  const int64_t n = per_batch / 8;
  uint32_t m2 = 0;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x)
    m2 = vmax_abs8(m2, p[i]);
  const uint32_t m = __reduce_max_sync(kFull, halves_max(m2));
  if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    const uint32_t v = __reduce_max_sync(kFull, threadIdx.x < blockDim.x / 32 ? s_warp[threadIdx.x] : 0u);
    if (threadIdx.x == 0 && v != 0u) atomicMax(&amax[b], v);
  }
}

template <class Src>
__global__ void __launch_bounds__(256) t8_quant_batches_kernel(const __grid_constant__ Src src, int64_t per_batch,
                                                               const uint32_t* __restrict__ amax,
                                                               uint8_t* __restrict__ codes) {
  const int64_t b = blockIdx.y;
  const float s = t8_scale(amax[b]);
  const uint4* p = reinterpret_cast<const uint4*>(src.mat(b));
  uint2* q = reinterpret_cast<uint2*>(codes + b * per_batch);
  const int64_t n = per_batch / 8;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x)
    q[i] = t8_codes8(p[i], s);
}

// ---- codes of a permuted-row tensor, one scale per expert segment ------------------
// Block (row block mb, column chunk): warp 0 finds the expert whose padded
// segment holds row block mb (a warp scan over the padded block counts); row
// blocks past the padded total are skipped.
constexpr int QS_COLS = 1024;

__global__ void __launch_bounds__(256) t8_quant_segments_kernel(const __nv_bfloat16* __restrict__ src,
                                                                const int* __restrict__ split_sizes, int E, int cols,
                                                                const uint32_t* __restrict__ amax,
                                                                uint8_t* __restrict__ codes) {
  __shared__ int s_e;
  const int mb = blockIdx.x;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int base = 0, found = -1;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int nb = e < E ? (split_sizes[e] + 127) >> 7 : 0;
      int incl = nb;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += o;
      }
      const bool hit = nb > 0 && base + incl - nb <= mb && mb < base + incl;
      const uint32_t msk = __ballot_sync(kFull, hit);
      if (msk != 0u) {
        found = e0 + __ffs(msk) - 1;
        break;
      }
      base += __shfl_sync(kFull, incl, 31);
    }
    if (lane == 0) s_e = found;
  }
  __syncthreads();
  const int e = s_e;
  if (e < 0) return;
  const float s = t8_scale(amax[e]);
  const int c0 = blockIdx.y * QS_COLS;
  const int wcols = min(QS_COLS, cols - c0) / 8;       // uint4 per row in this chunk
  for (int i = threadIdx.x; i < 128 * wcols; i += blockDim.x) {
    const int r = i / wcols, c = i - r * wcols;
    const int64_t off = (int64_t(mb) * 128 + r) * cols + c0 + int64_t(c) * 8;
    *reinterpret_cast<uint2*>(codes + off) = t8_codes8(*reinterpret_cast<const uint4*>(src + off), s);
  }
}

}  // namespace

cudaError_t launch_t8_amax_tokens(const void* x, int T, int H, const int* idx, int k, int E, uint32_t* amax,
                                  int* err, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int per_block = AT_WARPS * AT_TOKENS_PER_WARP;
  t8_amax_tokens_kernel<<<(T + per_block - 1) / per_block, AT_WARPS * 32, 0, st>>>(
      static_cast<const __nv_bfloat16*>(x), T, H, idx, k, E, amax, err);
  return cudaGetLastError();
}

cudaError_t launch_t8_quant_tokens(const void* x, int T, int H, const int* idx, const int* row_of, int k, int E,
                                   int64_t cap, const uint32_t* amax, uint8_t* codes, int* err, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int64_t threads = int64_t(T) * 32;
  t8_quant_tokens_kernel<<<unsigned((threads + 255) / 256), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(x), T, H, idx, row_of, k, E, cap, amax, codes, err);
  return cudaGetLastError();
}

namespace {
template <class Src>
cudaError_t amax_batches(const Src& src, int batch, int64_t per_batch, uint32_t* amax, cudaStream_t st) {
  const int64_t chunks = (per_batch / 8 + 255) / 256;
  const dim3 grid(unsigned(chunks < 1024 ? chunks : 1024), unsigned(batch));
  t8_amax_batches_kernel<Src><<<grid, 256, 0, st>>>(src, per_batch, amax);
  return cudaGetLastError();
}
template <class Src>
cudaError_t quant_batches(const Src& src, int batch, int64_t per_batch, const uint32_t* amax, uint8_t* codes,
                          cudaStream_t st) {
  const int64_t chunks = (per_batch / 8 + 255) / 256;
  const dim3 grid(unsigned(chunks < 2048 ? chunks : 2048), unsigned(batch));
  t8_quant_batches_kernel<Src><<<grid, 256, 0, st>>>(src, per_batch, amax, codes);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_t8_amax_batches(const void* src, int batch, int64_t per_batch, uint32_t* amax, cudaStream_t st) {
  return amax_batches(StackedSrc{static_cast<const __nv_bfloat16*>(src), per_batch}, batch, per_batch, amax, st);
}

cudaError_t launch_t8_quant_batches(const void* src, int batch, int64_t per_batch, const uint32_t* amax,
                                    uint8_t* codes, cudaStream_t st) {
  return quant_batches(StackedSrc{static_cast<const __nv_bfloat16*>(src), per_batch}, batch, per_batch, amax, codes,
                       st);
}

cudaError_t launch_t8_amax_experts(const ExpertSrc& src, int batch, int64_t per_batch, uint32_t* amax,
                                   cudaStream_t st) {
  return amax_batches(src, batch, per_batch, amax, st);
}

cudaError_t launch_t8_quant_experts(const ExpertSrc& src, int batch, int64_t per_batch, const uint32_t* amax,
                                    uint8_t* codes, cudaStream_t st) {
  return quant_batches(src, batch, per_batch, amax, codes, st);
}

cudaError_t launch_t8_quant_segments(const void* src, const int* split_sizes, int E, int64_t cap, int cols,
                                     const uint32_t* amax, uint8_t* codes, cudaStream_t st) {
  const dim3 grid(unsigned(cap / 128), unsigned((cols + QS_COLS - 1) / QS_COLS));
  t8_quant_segments_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(src), split_sizes, E, cols, amax,
                                                 codes);
  return cudaGetLastError();
}

}  // namespace moe
