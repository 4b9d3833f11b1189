// Launchers of the libmoeffn kernels (internal; the public interface is the C
// ABI in include/moe_ffn.h, implemented in api.cu).
#pragma once

#include <cuda.h>

#include <utility>

#include "common.cuh"

namespace moe {

// Launch with programmatic stream serialization: the kernel may begin (and run up to its
// pdl_wait()) while the previous kernel in the stream finishes.  Only for kernels that call
// pdl_wait() before touching global memory an earlier kernel may write or read.  A grid of
// more than kPdlMaxCtas CTAs runs in many waves, and starting its first one early gains
// nothing: it is launched the ordinary way (pdl_wait() then returns at once).
constexpr int64_t kPdlMaxCtas = 2048;
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = int64_t(grid.x) * grid.y * grid.z <= kPdlMaxCtas ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Per-thread text of the last host-side error, returned by moe_last_error_message().
constexpr size_t kLastErrorBytes = 512;
char* last_error_buffer();
// The size checks every layer entry point applies (T, H, I, E, k, the row capacity);
// on failure the message names the offending field.
moe_status check_layer_dims(const moe_dims* d);
// Rows of every permuted buffer for valid dims: roundup(T*k, 128) + 128*E.
int64_t rows_capacity(const moe_dims* d);

// Sources of a batch of bf16 [rows][cols] matrices: one stacked tensor, or one
// pointer per matrix (each expert's own weight tensor), passed by value.
constexpr int kMaxExpertPtrs = 256;
struct StackedSrc {
  const __nv_bfloat16* base;
  int64_t per;                                 // elements per matrix
  __device__ __forceinline__ const __nv_bfloat16* mat(int64_t b) const { return base + b * per; }
};
struct ExpertSrc {
  const __nv_bfloat16* p[kMaxExpertPtrs];
  __device__ __forceinline__ const __nv_bfloat16* mat(int64_t b) const { return p[b]; }
};

// pad_split (optional, with pad_E experts): the same launch also zeroes the padding rows of
// every segment of the permuted output (what launch_fill_pad_rows does).
cudaError_t launch_quant_rowwise(const void* src, int64_t n_rows, int cols, const int* row_of, int k, int64_t cap,
                                 uint8_t* codes, uint8_t* scales, int* err, cudaStream_t st,
                                 const int* pad_split = nullptr, int pad_E = 0);
cudaError_t launch_fill_pad_rows(const int* split_sizes, int E, int cols, int64_t cap, uint8_t* codes,
                                 uint8_t* scales, int* err, cudaStream_t st);
// The expert-major permutation, finished while x is quantized: the routing's outputs
// (idx, prob, the per-expert token masks [E][G] with their group prefix sums and
// split_sizes) in, row_of / src_of / prob_perm out.
constexpr int kMaxExperts = 256;
struct PermuteRows {
  const int* idx;
  const float* prob;
  const uint32_t* masks;
  const int* bases;
  const int* split_sizes;
  int E, G;
  int* row_of;
  int* src_of;
  float* prob_perm;
};
// x bf16 [T][H] -> MX codes/scales of the permuted rows [cap][H] (padding rows zero, src
// -1, prob 0) and the permutation maps, in one launch.
cudaError_t launch_permute_quant_rows(const void* x, int T, int H, int k, int64_t cap, const PermuteRows& p,
                                      uint8_t* codes, uint8_t* scales, int* err, cudaStream_t st);
// Tensor map for tile::gather4 loads of a bf16 [rows][cols] tensor (box: one row of
// box_cols elements); false when the driver's encoder is missing or refuses it.
bool encode_gather_rows_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_cols);
cudaError_t launch_quant_colwise(const void* src, const int* src_map, int64_t n_src_rows, int batch, int rows,
                                 int cols, const int* split_sizes, int E, uint8_t* codes_t, uint8_t* scales_t,
                                 int* err, cudaStream_t st);
cudaError_t launch_quant_dual(const void* src, int batch, int rows, int cols, uint8_t* codes, uint8_t* scales,
                              uint8_t* codes_t, uint8_t* scales_t, cudaStream_t st);
// codes_t / scales_t may be null (rows only)
cudaError_t launch_quant_dual_experts(const ExpertSrc& src, int batch, int rows, int cols, uint8_t* codes,
                                      uint8_t* scales, uint8_t* codes_t, uint8_t* scales_t, cudaStream_t st);
// Router backward workspace (chunk partials of dW_r and dl as bf16 hi + lo) and the
// tensor-core dW_r launch (partial [chunks][E][H]; *chunks_used chunks written).
size_t router_ws_bytes(int T, int E, int H);
int router_dw_cols(int E);
int router_dw_max_chunks(int H);
// Router logits [T][E] f32 = x [T][H] . W_r [E][H]^T on the tensor cores (bf16 operands).
cudaError_t launch_router_fwd_tc(const void* x, const void* w, int T, int H, int E, float* logits, int* err,
                                 cudaStream_t st);
cudaError_t launch_router_dw_tc(const void* x, const void* dl_hi, const void* dl_lo, int T, int H, int E,
                                float* partial, int max_chunks, int* chunks_used, int* err, cudaStream_t st);
cudaError_t launch_router_fwd(const void* x, const void* w, int T, int H, int E, float* logits, int* err,
                              cudaStream_t st, char* msg, size_t msg_len);
cudaError_t launch_router_bwd(const void* x, const void* w, const float* logits, const int* idx, const float* prob,
                              const float* dprob, int T, int H, int E, int k, int renorm, float* dl, void* dx,
                              float* dw, void* ws, int* err, cudaStream_t st);
// Top-k routing plus the per-expert scan of the token masks (masks [E][G], bases [E][G],
// split_sizes [E]).  One launch while E*ceil(T/32) <= 16384 (the last block to finish
// scans; `ticket` is a zero-initialised counter the launch returns to zero), else two.
bool route_scan_fused(int T, int E);
// The ticket of launch_route_scan: word 8 of a workspace's 256-byte error region (the
// error code and site are words 0 and 1), zero from the workspace's zero fill.
inline unsigned* route_ticket(int* err) { return reinterpret_cast<unsigned*>(err + 8); }
cudaError_t launch_route_scan(const float* logits, int T, int E, int k, int renorm, int* idx, float* prob,
                              uint32_t* masks, int* bases, int* split_sizes, unsigned* ticket, int* err,
                              cudaStream_t st);
// launch_route_scan, then the permutation maps alone (row_of, src_of, prob_perm).
cudaError_t launch_route_permute(const float* logits, int T, int E, int k, int renorm, int* idx, float* prob,
                                 uint32_t* masks, int* bases, int* split_sizes, int* row_of, int* src_of,
                                 float* prob_perm, unsigned* ticket, int* err, cudaStream_t st);
// The permutation of moe_route_permute for given expert ids idx [T][k] and probabilities.
cudaError_t launch_permute_from_idx(const int* idx, const float* prob, int T, int E, int k, uint32_t* masks,
                                    int* bases, int* split_sizes, int* row_of, int* src_of, float* prob_perm,
                                    int* err, cudaStream_t st);
// Expert parallelism: pack the (token, slot) rows of x by destination rank (see expert_parallel.cu).
cudaError_t launch_ep_pack(const void* x, const int* idx, const float* prob, const int* row_of,
                           const int* split_sizes, int T, int H, int E, int k, int G, void* send_x, float* send_prob,
                           int* send_eid, int* pos_of, int* rank_counts, int* err, cudaStream_t st);
cudaError_t launch_gather_f32(const float* src, int64_t n_src, const int* map, int64_t n, float* out, int* err,
                              cudaStream_t st);
cudaError_t launch_gather_rows(const void* x, const int* row_of, const int* split_sizes, int T, int k, int H, int E,
                               int64_t cap, void* x_perm, int* err, cudaStream_t st);
cudaError_t launch_combine(const void* y, const int* row_of, const float* prob, int T, int k, int H, int64_t cap,
                           void* out, int* err, cudaStream_t st);
// Per-tensor FP8 (one scale per expert operand tensor): amax reductions and E4M3 codes.
cudaError_t launch_t8_amax_tokens(const void* x, int T, int H, const int* idx, int k, int E, uint32_t* amax,
                                  int* err, cudaStream_t st);
cudaError_t launch_t8_quant_tokens(const void* x, int T, int H, const int* idx, const int* row_of, int k, int E,
                                   int64_t cap, const uint32_t* amax, uint8_t* codes, int* err, cudaStream_t st);
cudaError_t launch_t8_amax_batches(const void* src, int batch, int64_t per_batch, uint32_t* amax, cudaStream_t st);
cudaError_t launch_t8_quant_batches(const void* src, int batch, int64_t per_batch, const uint32_t* amax,
                                    uint8_t* codes, cudaStream_t st);
cudaError_t launch_t8_amax_experts(const ExpertSrc& src, int batch, int64_t per_batch, uint32_t* amax,
                                   cudaStream_t st);
cudaError_t launch_t8_quant_experts(const ExpertSrc& src, int batch, int64_t per_batch, const uint32_t* amax,
                                    uint8_t* codes, cudaStream_t st);
cudaError_t launch_t8_quant_segments(const void* src, const int* split_sizes, int E, int64_t cap, int cols,
                                     const uint32_t* amax, uint8_t* codes, cudaStream_t st);
// out[b*cols + c][r] = src row (b, r) column c for a batch of [rows][cols] bf16 matrices
// (rows, cols multiples of 128); with src_map, row r of the single matrix comes from
// src[src_map[r]] (-1: a zero row); with split_sizes, row tiles past the padded
// segments are skipped.
cudaError_t launch_transpose_bf16(const void* src, const int* src_map, int64_t n_src_rows, int batch, int rows,
                                  int cols, const int* split_sizes, int E, void* out, int* err, cudaStream_t st);
// the same for one bf16 [rows][cols] matrix per expert (src.p[b]), out stacked [batch][cols][rows]
cudaError_t launch_transpose_bf16_experts(const ExpertSrc& src, int batch, int rows, int cols, void* out,
                                          cudaStream_t st);
// out[b*cols + c][r] = src[b][r][c] for uint8 [batch][rows][cols] (multiples of 128);
// with split_sizes, row tiles past the padded segments are skipped.
cudaError_t launch_transpose_u8(const uint8_t* src, int batch, int rows, int cols, const int* split_sizes, int E,
                                uint8_t* out, cudaStream_t st);
// dprob[t][j] = the fixed-order sum of the down dgrad's per-tile partial row sums at
// row_of[t][j]; with src_of (and split_sizes) and many partials it reduces by permuted row.
cudaError_t launch_dprob_reduce(const float* dp_part, int n_tiles, int64_t cap, const int* split_sizes, int E,
                                const int* src_of, const int* row_of, int k, int T, float* dprob, int* err,
                                cudaStream_t st);

// ---- grouped block-scaled MXFP8 GEMM (tcgen05) ------------------------------------
// C[M][N] = A[M][K] * B[N][K]^T, both operands K-major MX tensors.
//   mode 0 (grouped rows): A rows are the permuted token rows, split into
//     128-row blocks per expert segment (from split_sizes); B = expert e's
//     weight rows.  K fixed.
//   mode 1 (grouped K, weight gradients): for each expert e an independent
//     [M][N] output with K = the expert's padded token range of A and B.
// EPI_BF16 .. EPI_BWD_SWIGLU take MXFP8 operands (block-scaled MMA); the B16 kinds take
// bf16 operands (kind::f16 MMA, no scales): plain bf16 output, or ScaledSwiGLU with a
// bf16 `a` written to out [cap][I].  The T8 kinds take per-tensor scaled E4M3 operands
// (kind::f8f6f4 MMA, no block scales): the accumulator is multiplied by
// 1 / (s_a[e] * s_b[e]) with s = 448 / amax of the expert's operand tensors, then a
// plain bf16 output, or ScaledSwiGLU with a bf16 `a` in out [cap][I] and the amax of
// every expert's bf16 `a` raised into amax_out[e].
enum Epilogue : int {
  EPI_BF16 = 0,
  EPI_FWD_SWIGLU = 1,
  EPI_BWD_SWIGLU = 2,
  EPI_B16_OUT = 3,
  EPI_B16_FWD_SWIGLU = 4,
  EPI_T8_OUT = 5,
  EPI_T8_FWD_SWIGLU = 6,
  EPI_B16_BWD_SWIGLU = 7,    // bf16 operands; SwiGLU backward writing bf16 dH to out [cap][2I] and out_t [2I][cap]
  EPI_T8_BWD_SWIGLU = 8,     // per-tensor E4M3 operands; SwiGLU backward writing bf16 dH to out [cap][2I]
                             // and raising every expert's amax of dH into amax_out
};

struct GemmArgs {
  int mode;
  int E;
  const int* split_sizes;
  int K;                     // mode 0 contraction length (multiple of 128)
  int N;                     // output columns (per expert in mode 1); SwiGLU epilogues: I
  int M;                     // mode 1: output rows per expert (multiple of 128)
  int n_tiles;               // tiles along N
  int64_t b_rows_per_expert; // mode 0: rows of B per expert
  int64_t cap;               // permuted row capacity
  const uint8_t* sfa;        // tile-layout scales of A
  const uint8_t* sfb;        // tile-layout scales of B
  int64_t sfa_K;             // K of A's scale layout
  int64_t sfb_K;             // K of B's scale layout
  // epilogue operands
  __nv_bfloat16* out;        // EPI_BF16 output
  int64_t ldo;
  __nv_bfloat16* out_t;      // EPI_B16_BWD_SWIGLU: dH transposed [2I][cap]
  const float* prob_perm;    // SwiGLU epilogues
  uint8_t* q_row;            // rowwise MX output (codes) [cap][q_row_K]
  uint8_t* q_row_s;
  int64_t q_row_K;
  uint8_t* q_col;            // colwise MX output (codes) [cols][cap], optional
  uint8_t* q_col_s;
  __nv_bfloat16* gu;         // saved g,u [cap][2I]: written by FWD (optional), read by BWD
  float* dp_part;            // BWD: [n_tiles][cap] partial row sums of dA*silu(g)*u
  int I;
  const uint32_t* amax_a;    // T8 kinds: per-expert amax (float bits) of A's and B's tensors
  const uint32_t* amax_b;
  uint32_t* amax_out;        // EPI_T8_FWD_SWIGLU: per-expert amax of the bf16 `a` (raised, not set)
  int64_t rows_limit;        // mode 0 with split_sizes == nullptr: one segment of this many rows (E = 1)
  int* err;
  bool out_v8;               // set by launch_grouped_gemm: out, out_t and gu are 32-byte aligned (256-bit stores)
  uint64_t wait_limit_ns;    // bound of every mbarrier wait (0: the default kWaitLimitNs)
  int selftest_no_loads;     // self-test only: the producer issues nothing, so the waits run out
};

// The GEMM epilogues' MX quantizers (row-wise along cols, and along rows into the
// transposed [cols][rows] tensor) applied to a caller's f32 [rows][cols] tensor
// (rows, cols multiples of 128), one 32 x 32 block per warp as an epilogue warp
// holds it.
cudaError_t launch_epilogue_quant_selftest(const float* src, int rows, int cols, uint8_t* codes, uint8_t* scales,
                                           uint8_t* codes_t, uint8_t* scales_t, cudaStream_t st);

// The MXFP8 MMA issue ceiling: one launch of SMs/2 CTA pairs, each issuing k_steps
// K steps of the GEMM's MMAs (M=256, N=256, K=128 per step, with its scale copies)
// on resident zero operands; *pairs = the pairs launched.  err: device error word.
cudaError_t launch_mma_rate_selftest(int k_steps, int* err, int* pairs, cudaStream_t st);

// b_experts (host array of E pointers, E <= 128; the bf16 forward kinds only): B is one
// [b_rows][b_K] matrix per expert instead of the stacked tensor B (then a.b_rows_per_expert = 0).
cudaError_t launch_grouped_gemm(int epi, const GemmArgs& a, const void* A, int64_t a_rows, int64_t a_K,
                                const void* B, int64_t b_rows, int64_t b_K, int64_t max_tiles, cudaStream_t st,
                                char* msg, size_t msg_len, const void* const* b_experts = nullptr);

}  // namespace moe
