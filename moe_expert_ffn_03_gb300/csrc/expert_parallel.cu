// Expert-parallel dispatch and combine (page "英伟达开源MoE加速神器：一行代码，微调快3.7倍",
// section "三板斧", expert parallelism: the experts are spread over the GPUs and an
// All-to-All sends each token to the GPU of its expert and brings the result back; page
// "Efficient MoE Training for Biological Foundation Models", section
// "运行要求、基准与验证步骤": the recipe runs with EP = 8 and DP x EP = #GPUs).
//
// Experts are laid out over G ranks in contiguous blocks: rank r owns experts
// r*E/G .. (r+1)*E/G - 1.  After moe_route_permute a rank's (token, slot) rows are
// already expert-major, hence grouped by destination rank; the pack kernel writes
// them densely (no segment padding) into the send buffer: row pos of (t, j) is the
// expert's unpadded start plus the row's rank inside its expert, i.e. row_of[t][j]
// minus the expert's padded start plus its unpadded start.  Each send row carries
// x[t] (bf16), its probability and its expert id local to the destination rank; the
// kernel also counts the rows per destination rank (the All-to-All split sizes) and
// keeps pos for the combine of the rows that come back.
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int EP_WARPS = 8;
constexpr int kMaxE = 256;

__global__ void __launch_bounds__(32 * EP_WARPS) ep_pack_kernel(
    const __nv_bfloat16* __restrict__ x, const int* __restrict__ idx, const float* __restrict__ prob,
    const int* __restrict__ row_of, const int* __restrict__ split_sizes, int T, int H, int E, int k, int G,
    __nv_bfloat16* __restrict__ send_x, float* __restrict__ send_prob, int* __restrict__ send_eid,
    int* __restrict__ pos_of, int* __restrict__ rank_counts, int* err) {
  __shared__ int pad_start[kMaxE], start[kMaxE];
  if (threadIdx.x == 0) {
    int acc = 0, acc_pad = 0;
    for (int e = 0; e < E; ++e) {
      start[e] = acc;
      pad_start[e] = acc_pad;
      acc += split_sizes[e];
      acc_pad += (split_sizes[e] + 127) & ~127;
    }
    if (blockIdx.x == 0) {
      const int per = E / G;
      for (int r = 0; r < G; ++r) {
        int c = 0;
        for (int e = r * per; e < (r + 1) * per; ++e) c += split_sizes[e];
        rank_counts[r] = c;
      }
    }
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t pair = int64_t(blockIdx.x) * EP_WARPS + warp;       // (token, slot) = (pair / k, pair % k)
  if (pair >= int64_t(T) * k) return;
  const int t = int(pair / k);
  const int e = idx[pair];
  const int r = row_of[pair];
  if (e < 0 || e >= E || r < pad_start[e] || r - pad_start[e] >= split_sizes[e]) {
    if (lane == 0) {
      report_error(err, MOE_ERR_DEVICE_BOUNDS, SITE_PERMUTE + 10);
      pos_of[pair] = -1;
    }
    return;
  }
  const int pos = start[e] + (r - pad_start[e]);
  if (lane == 0) {
    pos_of[pair] = pos;
    send_prob[pos] = prob[pair];
    send_eid[pos] = e % (E / G);
  }
  // the row: H bf16 = H/8 chunks of 16 bytes
  const uint4* src = reinterpret_cast<const uint4*>(x + int64_t(t) * H);
  uint4* dst = reinterpret_cast<uint4*>(send_x + int64_t(pos) * H);
  for (int c = lane; c < H / 8; c += 32) dst[c] = src[c];
}

// out[i] = src[map[i]] (map entries outside 0..n_src-1 give 0 and are recorded).
__global__ void gather_f32_kernel(const float* __restrict__ src, int64_t n_src, const int* __restrict__ map,
                                  int64_t n, float* __restrict__ out, int* err) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int m = map[i];
  if (m < 0 || m >= n_src) {
    report_error(err, MOE_ERR_DEVICE_BOUNDS, SITE_COMBINE + 10);
    out[i] = 0.f;
    return;
  }
  out[i] = src[m];
}

}  // namespace

cudaError_t launch_ep_pack(const void* x, const int* idx, const float* prob, const int* row_of,
                           const int* split_sizes, int T, int H, int E, int k, int G, void* send_x, float* send_prob,
                           int* send_eid, int* pos_of, int* rank_counts, int* err, cudaStream_t st) {
  const int64_t pairs = int64_t(T) * k;
  const int64_t grid = (pairs + EP_WARPS - 1) / EP_WARPS;
  ep_pack_kernel<<<unsigned(grid), 32 * EP_WARPS, 0, st>>>(
      static_cast<const __nv_bfloat16*>(x), idx, prob, row_of, split_sizes, T, H, E, k, G,
      static_cast<__nv_bfloat16*>(send_x), send_prob, send_eid, pos_of, rank_counts, err);
  return cudaGetLastError();
}

cudaError_t launch_gather_f32(const float* src, int64_t n_src, const int* map, int64_t n, float* out, int* err,
                              cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  gather_f32_kernel<<<unsigned((n + 255) / 256), 256, 0, st>>>(src, n_src, map, n, out, err);
  return cudaGetLastError();
}

}  // namespace moe
