/*
 * moe_ffn.h -- C ABI of the GB300 (sm_103a) grouped MXFP8 MoE expert FFN.
 *
 * The library computes the Mixture-of-Experts expert FFN as one grouped
 * operation instead of a per-expert loop: top-k routing, an expert-major
 * permutation driven by per-expert token counts (split_sizes), MXFP8
 * quantization, a grouped gate_up GEMM with ScaledSwiGLU fused into its
 * epilogue, a grouped down GEMM, the combine, and the matching backward
 * (dgrad and wgrad).
 *
 * Sources.  Page "Efficient MoE Training for Biological Foundation Models"
 * (summary of the NVIDIA technical blog on the BioNeMo MoE recipe):
 *   - section "GroupedLinear：把逐专家循环改成一次分组GEMM": one grouped call
 *     takes the tokens collected per expert plus split_sizes; every expert
 *     keeps its own weight; gate_up has out_features = 2*intermediate,
 *     bias=False;
 *   - section "MXFP8与融合MLP：减少显存并跳过独立量化步骤": gate_up ->
 *     ScaledSwiGLU (SwiGLU times the router probabilities) -> down, with
 *     quantization, SwiGLU and the probability scaling fused, forward and
 *     backward;
 *   - section "MoE训练的瓶颈与TE的对应能力": MXFP8 holds values in 8 bits with
 *     one scale per 32 consecutive values; 16-bit master weights are
 *     quantized before each low-precision GEMM.
 * Page "英伟达开源MoE加速神器：一行代码，微调快3.7倍", section "三板斧": each
 * token goes to a few of many experts; the expert FFN is the compute bulk.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the
 *     library allocates nothing and keeps no state beyond a per-process
 *     cache of the driver entry point that encodes TMA descriptors.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  No call synchronises the host except
 *     moe_get_device_error.  split_sizes is never read on the host.
 *   - Host-checkable errors (sizes, alignment, null pointers) return before
 *     anything is launched.  Errors detected by a kernel (a bounded wait
 *     that ran out, an index out of range) are recorded in the workspace
 *     error word and read with moe_get_device_error; kernels never trap.
 *   - bf16 means IEEE bfloat16 stored as 2 bytes; f32 is IEEE float.
 *   - Every pointer must be 16-byte aligned.
 *
 * Sizes: T tokens (>= 1), H hidden, I intermediate (H and I multiples of
 * 128), E experts (1..256), k experts per token (1..min(E, 8)).
 * R = T*k routed rows.  Permuted buffers have CAP = moe_rows_capacity()
 * rows: the expert segments are laid out expert-major from row 0, segment e
 * has roundup(split_sizes[e], 128) rows (rows past split_sizes[e] are zero
 * padding), and CAP bounds the padded total for every routing.
 *
 * MXFP8 tensors.  An MX tensor is (codes, scales):
 *   codes  uint8 E4M3 (sign, 4 exponent bits with bias 7, 3 mantissa bits,
 *          max 448, 0x7F/0xFF NaN), row-major [rows][K];
 *   scales uint8 power-of-two exponents c (scale = 2^(c-127), 255 = NaN),
 *          one per 32 consecutive elements along K, in the MMA tile layout:
 *          the scale of (row r, block b = k/32) is stored at byte
 *              ((r/128)*(K/128) + b/4)*512 + (r%32)*16 + ((r/32)%4)*4 + b%4
 *          (rows a multiple of 128, K a multiple of 128).  A batch of
 *          matrices [B][rows][K] uses the same formula on [B*rows][K].
 *   Quantization rule: e = smallest integer with amax <= 448*2^e (no element
 *   saturates), clamped to [-127,127], all-zero block -> code 0; elements
 *   are x*2^-e rounded to nearest-even E4M3 (subnormals and the sign of
 *   zero kept); a block holding NaN/Inf gets scale 255 and codes 0x7F.
 *   The page fixes "8 bits" and "one scale per 32 consecutive values"; the
 *   E4M3 element, the power-of-two scale and this rounding rule are the
 *   readings this library implements.
 */
#ifndef MOE_FFN_H
#define MOE_FFN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,     /* a size or pointer argument is out of range */
  MOE_ERR_UNSUPPORTED = 2,     /* a valid configuration this build does not handle */
  MOE_ERR_ALIGNMENT = 3,       /* a pointer is not 16-byte aligned */
  MOE_ERR_WORKSPACE = 4,       /* workspace missing or smaller than moe_workspace_size */
  MOE_ERR_CUDA = 5,            /* a CUDA runtime/driver call failed (launch, attribute, TMA encode) */
  MOE_ERR_DEVICE_TIMEOUT = 6,  /* (device) a bounded wait inside a kernel ran out */
  MOE_ERR_DEVICE_BOUNDS = 7    /* (device) an index read from device data was out of range */
} moe_status;

typedef void* moe_stream_t;    /* a cudaStream_t */

typedef struct moe_dims {
  int32_t T;            /* tokens */
  int32_t H;            /* hidden size, multiple of 128 */
  int32_t I;            /* intermediate size, multiple of 128 (gate_up has 2*I outputs) */
  int32_t E;            /* experts, 1..256 */
  int32_t k;            /* experts per token, 1..min(E,8) */
  int32_t renormalize;  /* 1: prob = softmax over the k selected logits; 0: softmax over all E */
} moe_dims;

/* Human-readable name of a status code (static string). */
const char* moe_status_string(moe_status s);

/* Text of the last host-side error on the calling thread ("" if none). */
const char* moe_last_error_message(void);

/* Rows of every permuted buffer: roundup(T*k, 128) + 128*E.  Host only. */
size_t moe_rows_capacity(const moe_dims* d);

/* Bytes of workspace needed for these sizes by moe_route_permute and the
 * forward calls (training = 0), also by grouped_mlp_bwd and moe_router_bwd
 * (training = 1), and also by grouped_mlp_bwd_bf16 (training = 2) or by
 * grouped_mlp_bwd_fp8_tensor (training = 3).  The workspace is caller memory,
 * 256-byte aligned, zero-filled once before first use (that clears the device
 * error word and the block counter of the routing launch, which every routing
 * call leaves at zero again); it may be reused by later calls on the same
 * stream, not by calls running at the same time on other streams.  Returns 0
 * for invalid sizes or training outside 0..3.  Host only. */
size_t moe_workspace_size(const moe_dims* d, int32_t training);

/*
 * mxfp8_quantize -- bf16 -> MX tensor (the quantize step before each GEMM;
 * page "Efficient MoE Training for Biological Foundation Models", section
 * "MoE训练的瓶颈与TE的对应能力").  Used for the 16-bit master weights, once
 * per optimizer step.
 *   src     bf16 [batch][rows][cols], row-major.
 *   axis 0: blocks of 32 along cols -> codes [batch][rows][cols],
 *           scales in the tile layout of [batch*rows][cols].
 *   axis 1: blocks of 32 along rows -> codes [batch][cols][rows] (each
 *           matrix transposed), scales in the tile layout of [batch*cols][rows].
 *   rows and cols multiples of 128, batch >= 1.
 */
moe_status mxfp8_quantize(const void* src, int32_t batch, int32_t rows, int32_t cols, int32_t axis,
                          uint8_t* codes, uint8_t* scales, moe_stream_t stream);

/*
 * mxfp8_quantize_dual -- both results of mxfp8_quantize (axis 0 into
 * codes/scales, axis 1 into codes_t/scales_t) from ONE read of src.  This is
 * the training-time weight quantization: the forward GEMMs consume W blocked
 * along its columns, the backward (dgrad) GEMMs consume W^T blocked along its
 * rows (page "Efficient MoE Training for Biological Foundation Models",
 * section "MoE训练的瓶颈与TE的对应能力": 16-bit master weights are quantized
 * before the low-precision GEMMs).  Same sizes, layouts and errors as
 * mxfp8_quantize; batch <= 65535.
 */
moe_status mxfp8_quantize_dual(const void* src, int32_t batch, int32_t rows, int32_t cols,
                               uint8_t* codes, uint8_t* scales, uint8_t* codes_t, uint8_t* scales_t,
                               moe_stream_t stream);

/*
 * moe_route_permute -- top-k routing, expert-major permutation, gather and
 * quantization of the tokens (page "Efficient MoE Training for Biological
 * Foundation Models", section "GroupedLinear": tokens are collected per
 * expert, split_sizes counts them; page "英伟达开源MoE加速神器", section
 * "三板斧": each token is routed to a few experts).
 *   logits      f32 [T][E]
 *   x           bf16 [T][H]
 *   idx         out int32 [T][k]: top-k experts by logit, descending, ties to
 *               the lower expert index (+0 and -0 tie).  A NaN logit ranks
 *               below every number, -inf included, and NaNs tie among
 *               themselves, so every row selects k distinct experts; a row
 *               that selects a NaN logit gets NaN probabilities.
 *   prob        out f32 [T][k]: softmax of the selected logits (see renormalize)
 *   split_sizes out int32 [E]: tokens per expert (sum = T*k)
 *   row_of      out int32 [T][k]: permuted row of (token, slot); inside an
 *               expert segment rows follow ascending token index
 *   src_of      out int32 [CAP]: source token of each row, -1 on padding
 *               (rows past the padded total are not written)
 *   prob_perm   out f32 [CAP]: prob of each row, 0 on padding
 *   xq,xq_scale out MX [CAP][H] of x rows, blocks along H (padding rows zero)
 *   xq_col,xq_col_scale  optional (both NULL or both set): MX [H][CAP], x
 *               permuted and quantized in blocks of 32 rows along the token
 *               axis (blocks start at segment starts; padding is zero) --
 *               the B operand of the gate_up weight gradient.
 *   workspace   >= moe_workspace_size(d, xq_col != NULL) bytes.
 */
moe_status moe_route_permute(const moe_dims* d, const float* logits, const void* x,
                             int32_t* idx, float* prob, int32_t* split_sizes,
                             int32_t* row_of, int32_t* src_of, float* prob_perm,
                             uint8_t* xq, uint8_t* xq_scale, uint8_t* xq_col, uint8_t* xq_col_scale,
                             void* workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * moe_route -- the routing and permutation of moe_route_permute without the
 * gather and quantization of x: idx, prob, split_sizes, row_of, src_of and
 * prob_perm exactly as moe_route_permute writes them.  An expert-parallel
 * rank (moe_ep_pack) needs only these on the tokens' side.  workspace as for
 * moe_route_permute with training = 0.
 */
moe_status moe_route(const moe_dims* d, const float* logits, int32_t* idx, float* prob, int32_t* split_sizes,
                     int32_t* row_of, int32_t* src_of, float* prob_perm, void* workspace, size_t workspace_bytes,
                     moe_stream_t stream);

/*
 * moe_permute -- moe_route_permute for rows whose experts are already known
 * (page "Efficient MoE Training for Biological Foundation Models", section
 * "GroupedLinear": the grouped call receives the tokens collected per expert
 * together with split_sizes).  idx int32 [T][k] holds expert ids in 0..E-1 and
 * prob f32 [T][k] their probabilities; the stable expert-major permutation
 * (ascending row inside each segment, segments padded to 128 rows), the MX
 * codes of x rows and, optionally, of x along tokens are those moe_route_permute
 * produces for the same idx.  An expert-parallel rank calls it on the rows it
 * received (k = 1, idx = their local expert ids).  An id outside 0..E-1 is
 * recorded in the workspace error word and its slot skipped (row_of -1).
 * Arguments otherwise as moe_route_permute.
 */
moe_status moe_permute(const moe_dims* d, const int32_t* idx, const float* prob, const void* x, int32_t* split_sizes,
                       int32_t* row_of, int32_t* src_of, float* prob_perm, uint8_t* xq, uint8_t* xq_scale,
                       uint8_t* xq_col, uint8_t* xq_col_scale, void* workspace, size_t workspace_bytes,
                       moe_stream_t stream);

/*
 * moe_ep_pack -- the send side of the expert-parallel dispatch (page
 * "英伟达开源MoE加速神器：一行代码，微调快3.7倍", section "三板斧": experts are
 * spread over the GPUs and an All-to-All takes each token to its expert's GPU).
 * The E experts are laid out over `world` ranks in contiguous blocks (rank r owns
 * experts r*E/world .. (r+1)*E/world - 1; world divides E).  From the routing of
 * moe_route (idx, prob, row_of, split_sizes of this rank's T tokens) it writes the
 * T*k rows densely in expert-major order, which groups them by destination rank:
 *   send_x     out bf16 [T*k][H]: row pos of (t, j) = x[t], where pos = the number
 *              of rows of experts before idx[t][j] plus the row's rank inside its
 *              expert (ascending token order)
 *   send_prob  out f32 [T*k]: prob[t][j] at pos
 *   send_eid   out int32 [T*k]: idx[t][j] modulo E/world (the destination's local id)
 *   pos_of     out int32 [T][k]: pos of every (t, j) (the combine's row map)
 *   rank_counts out int32 [world]: rows for each destination rank (the split sizes
 *              of the All-to-All)
 * workspace as for moe_route (its error word records inconsistent inputs).
 */
moe_status moe_ep_pack(const moe_dims* d, int32_t world, const void* x, const int32_t* idx, const float* prob,
                       const int32_t* row_of, const int32_t* split_sizes, void* send_x, float* send_prob,
                       int32_t* send_eid, int32_t* pos_of, int32_t* rank_counts, void* workspace,
                       size_t workspace_bytes, moe_stream_t stream);

/*
 * moe_gather_f32 -- out[i] = src[map[i]] for i < n (f32); a map entry outside
 * 0..n_src-1 gives 0 and is recorded in the error word at `workspace` (any
 * layer workspace).  The expert-parallel combine takes the returned dprob rows
 * back to [T][k] with it (map = pos_of).
 */
moe_status moe_gather_f32(const float* src, int64_t n_src, const int32_t* map, int64_t n, float* out,
                          void* workspace, moe_stream_t stream);

/*
 * grouped_mlp_fwd -- grouped gate_up GEMM + ScaledSwiGLU + grouped down GEMM
 * (page "Efficient MoE Training for Biological Foundation Models", sections
 * "GroupedLinear" and "MXFP8与融合MLP").  One launch per GEMM covers every
 * expert; the tile schedule is derived on the device from split_sizes.
 *   xq,xq_scale   MX [CAP][H] from moe_route_permute
 *   split_sizes   int32 [E] (device)
 *   prob_perm     f32 [CAP]
 *   wgu_q,wgu_s   MX [E][2I][H] (mxfp8_quantize axis 0 of W_gu; rows 0..I-1
 *                 gate, I..2I-1 up)
 *   wd_q,wd_s     MX [E][H][I]  (mxfp8_quantize axis 0 of W_d)
 *   y             out bf16 [CAP][H]: expert output of every row (padding 0)
 *   saved_gu      optional out bf16 [CAP][2I]: g (cols 0..I-1) and u (I..2I-1)
 *                 as bf16, for the backward
 *   aq_col,aq_col_scale  optional out MX [I][CAP]: a = silu(g)*u*p quantized
 *                 along tokens, for the down weight gradient
 *   Epilogue of the gate_up GEMM: a = silu(g)*u*prob_perm[row], quantized
 *   rowwise along I into the workspace; no f32/bf16 copy of a is stored.
 */
moe_status grouped_mlp_fwd(const moe_dims* d, const uint8_t* xq, const uint8_t* xq_scale,
                           const int32_t* split_sizes, const float* prob_perm,
                           const uint8_t* wgu_q, const uint8_t* wgu_s,
                           const uint8_t* wd_q, const uint8_t* wd_s,
                           void* y, void* saved_gu, uint8_t* aq_col, uint8_t* aq_col_scale,
                           void* workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * moe_gather_rows -- bf16 path: x_perm[row_of[t][j]] = x[t] for every (token,
 * slot); padding rows of each expert segment are zeroed.  x bf16 [T][H],
 * row_of and split_sizes from moe_route_permute, x_perm out bf16 [CAP][H].
 * workspace: as for grouped_mlp_fwd (its error word records bad rows).
 */
moe_status moe_gather_rows(const moe_dims* d, const void* x, const int32_t* row_of, const int32_t* split_sizes,
                           void* x_perm, void* workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * grouped_mlp_fwd_bf16 -- the same grouped gate_up GEMM + ScaledSwiGLU + grouped
 * down GEMM with bf16 operands and no quantization (page "Efficient MoE
 * Training for Biological Foundation Models", section "运行要求、基准与验证步骤":
 * the recipe runs in BF16 or in MXFP8).  tcgen05 kind::f16 MMA, f32 accumulate.
 *   x_perm   bf16 [CAP][H] (moe_gather_rows); split_sizes, prob_perm as for
 *            grouped_mlp_fwd; w_gu bf16 [E][2I][H], w_d bf16 [E][H][I] (the master
 *            weights as they are);
 *   a_perm   out bf16 [CAP][I]: a = silu(g)*u*p rounded to bf16 (the down
 *            GEMM's input);
 *   y        out bf16 [CAP][H];
 *   saved_gu out bf16 [CAP][2I] or NULL: g and u for grouped_mlp_bwd_bf16.
 */
moe_status grouped_mlp_fwd_bf16(const moe_dims* d, const void* x_perm, const int32_t* split_sizes,
                                const float* prob_perm, const void* w_gu, const void* w_d, void* a_perm, void* y,
                                void* saved_gu, void* workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * moe_transpose_bf16 -- dst[b][c][r] = src[b][r][c] for bf16 [batch][rows][cols]
 * (rows, cols multiples of 128; 1 <= batch <= 65535).  The bf16 training path
 * takes W_gu^T [E][H][2I] and W_d^T [E][I][H] from it, once per step, the way the
 * MXFP8 path takes its transposed weight copies from mxfp8_quantize_dual.
 */
moe_status moe_transpose_bf16(const void* src, int32_t batch, int32_t rows, int32_t cols, void* dst,
                              moe_stream_t stream);

/*
 * moe_transpose_bf16_experts -- moe_transpose_bf16 for weights held as one
 * tensor per expert (page "Efficient MoE Training for Biological Foundation
 * Models", section "GroupedLinear": every expert keeps its own weight, weight0,
 * weight1, ...).  src is a HOST array of E device pointers, each to a bf16
 * [rows][cols] matrix (16-byte aligned; read during the call only); dst is the
 * stacked transposed tensor [E][cols][rows] that grouped_mlp_bwd_bf16 reads.
 * rows, cols multiples of 128; 1 <= E <= 256.
 */
moe_status moe_transpose_bf16_experts(const void* const* src, int32_t E, int32_t rows, int32_t cols, void* dst,
                                      moe_stream_t stream);

/*
 * grouped_mlp_fwd_bf16_experts -- grouped_mlp_fwd_bf16 on one weight tensor per
 * expert (page "Efficient MoE Training for Biological Foundation Models",
 * section "GroupedLinear": GroupedLinear keeps weight0, weight1, ... and the
 * grouped call applies each expert's own matrix to its split of the tokens).
 * w_gu and w_d are HOST arrays of E device pointers (read during the call):
 * w_gu[e] bf16 [2I][H] (rows 0..I-1 gate, I..2I-1 up), w_d[e] bf16 [H][I], each
 * 16-byte aligned.  The GEMMs read each expert's tensor where it is, through one
 * TMA descriptor per expert; results are bit-identical to grouped_mlp_fwd_bf16
 * on the same weights stacked.  E <= 128 (MOE_ERR_UNSUPPORTED above).  Other
 * arguments, outputs and errors as grouped_mlp_fwd_bf16.
 */
moe_status grouped_mlp_fwd_bf16_experts(const moe_dims* d, const void* x_perm, const int32_t* split_sizes,
                                        const float* prob_perm, const void* const* w_gu, const void* const* w_d,
                                        void* a_perm, void* y, void* saved_gu, void* workspace,
                                        size_t workspace_bytes, moe_stream_t stream);

/*
 * grouped_mlp_bwd_bf16 -- backward of grouped_mlp_fwd_bf16 (no quantization;
 * every stored tensor bf16, every GEMM a tcgen05 kind::f16 MMA with f32
 * accumulation).  The steps are those of grouped_mlp_bwd: dY = dout gathered
 * to rows; dA = dY*W_d with the SwiGLU backward fused (dg = dA*p*u*silu'(g),
 * du = dA*p*silu(g), dp = sum dA*silu(g)*u), writing dH = [dg|du] as bf16 rows
 * and transposed; dW_d = dY^T*a and dW_gu = dH^T*x over each expert's tokens;
 * dX = dH*W_gu.
 *   dout            bf16 [T][H]
 *   split_sizes, row_of, src_of, prob_perm: from moe_route_permute
 *   saved_gu        bf16 [CAP][2I]: the saved_gu output of grouped_mlp_fwd_bf16
 *   x_perm, a_perm  bf16 [CAP][H], [CAP][I]: from moe_gather_rows and
 *                   grouped_mlp_fwd_bf16
 *   w_guT, w_dT     bf16 [E][H][2I], [E][I][H]: moe_transpose_bf16 of W_gu, W_d
 *   dx_perm         out bf16 [CAP][H]; combine it with moe_unpermute_combine
 *   dwgu, dwd       out bf16 [E][2I][H], [E][H][I] (zeros for experts without tokens)
 *   dprob           out f32 [T][k]
 *   workspace       moe_workspace_size(d, 2) bytes (holds dY, dH and x, a transposed)
 */
moe_status grouped_mlp_bwd_bf16(const moe_dims* d, const void* dout, const int32_t* split_sizes,
                                const int32_t* row_of, const int32_t* src_of, const float* prob_perm,
                                const void* saved_gu, const void* x_perm, const void* a_perm, const void* w_guT,
                                const void* w_dT, void* dx_perm, void* dwgu, void* dwd, float* dprob, void* workspace,
                                size_t workspace_bytes, moe_stream_t stream);

/*
 * mxfp8_quantize_experts -- mxfp8_quantize_dual for weights held as one tensor
 * per expert (page "Efficient MoE Training for Biological Foundation Models",
 * section "GroupedLinear": every expert keeps its own weight tensor, weight0,
 * weight1, ...).  w is a HOST array of E device pointers, each to a bf16
 * [rows][cols] row-major matrix, 16-byte aligned; the results are the stacked
 * tensors of mxfp8_quantize_dual with batch = E, so the grouped GEMMs read
 * them unchanged.  codes_t/scales_t may both be NULL (forward-only: the
 * rowwise copy alone).  1 <= E <= 256; the pointers are read during the call
 * only.
 */
moe_status mxfp8_quantize_experts(const void* const* w, int32_t E, int32_t rows, int32_t cols, uint8_t* codes,
                                  uint8_t* scales, uint8_t* codes_t, uint8_t* scales_t, moe_stream_t stream);

/*
 * Per-tensor FP8 with dynamic scaling (page "英伟达开源MoE加速神器", section
 * "3. Transformer Engine：FP8 训练加速": the Hopper recipe scales every tensor by
 * its current range; page "Efficient MoE Training for Biological Foundation
 * Models", section "MoE训练的瓶颈与TE的对应能力": FP8 keeps one scale per tensor
 * where MXFP8 keeps one per 32 values).  The tensors are the operands of each
 * expert's GEMMs: expert e's token rows of x, its W_gu[e] and W_d[e], and its
 * rows of the activation a.  For such a tensor with amax = max |v|:
 *   s = 448 / amax rounded to float32 (s = 1 for an all-zero tensor),
 *   code = E4M3 of the float32 product v * s, nearest-even, saturating to
 *   +-448 (sign of zero kept); value = code / s.
 * The amax arrays are float32 [E] on the device, non-negative; the calls that
 * fill them first set them to zero.  Tensors holding NaN or Inf are outside
 * this path.
 */

/*
 * fp8_tensor_quantize -- per-slice amax and E4M3 codes of src bf16
 * [batch][rows][cols] (cols a multiple of 8): amax out float32 [batch],
 * codes out uint8 [batch][rows][cols] (the same layout).  For the weights:
 * W_gu as batch E, rows 2I, cols H; W_d as batch E, rows H, cols I.  Device
 * pointers 16-byte aligned.
 */
moe_status fp8_tensor_quantize(const void* src, int batch, int rows, int cols, uint8_t* codes, float* amax,
                               moe_stream_t stream);

/*
 * fp8_tensor_quantize_experts -- fp8_tensor_quantize for one weight tensor per
 * expert: w is a HOST array of E device pointers (bf16 [rows][cols] each,
 * 16-byte aligned), 1 <= E <= 256; codes out stacked uint8 [E][rows][cols],
 * amax out float32 [E].
 */
moe_status fp8_tensor_quantize_experts(const void* const* w, int32_t E, int32_t rows, int32_t cols, uint8_t* codes,
                                       float* amax, moe_stream_t stream);

/*
 * moe_fp8_tensor_quantize_tokens -- the x operand of the per-tensor path:
 * amax_x[e] = max |x[t][h]| over the tokens t routed to e, then for every
 * (token, slot j) with expert e = idx[t][j] the codes of x[t] * s_x[e] in
 * permuted row row_of[t][j] of xq (uint8 [CAP][H]); padding rows of every
 * segment get zero codes.  idx, row_of, split_sizes from moe_route_permute;
 * amax_x out float32 [E]; workspace as for grouped_mlp_fwd (its error word
 * records out-of-range experts or rows).
 */
moe_status moe_fp8_tensor_quantize_tokens(const moe_dims* d, const void* x, const int32_t* idx,
                                          const int32_t* row_of, const int32_t* split_sizes, uint8_t* xq,
                                          float* amax_x, void* workspace, size_t workspace_bytes,
                                          moe_stream_t stream);

/*
 * grouped_mlp_fwd_fp8_tensor -- the grouped gate_up GEMM + ScaledSwiGLU +
 * grouped down GEMM on per-tensor FP8 operands: tcgen05 kind::f8f6f4 MMA
 * (E4M3 x E4M3, no block scales), f32 accumulate, the accumulator multiplied
 * by 1/(s_a[e] * s_b[e]) in the epilogue.
 *   xq, amax_x      from moe_fp8_tensor_quantize_tokens
 *   split_sizes, prob_perm from moe_route_permute
 *   wgu_q, amax_gu  fp8_tensor_quantize of W_gu; wd_q, amax_d of W_d
 *   a_perm          out bf16 [CAP][I]: a = silu(g)*u*p rounded to bf16 (the
 *                   activation is stored because its scale needs the
 *                   tensor's amax before any element is quantized)
 *   aq              out uint8 [CAP][I]: codes of a with s_a[e]
 *   amax_a          out float32 [E]: amax of every expert's rows of a_perm
 *   y               out bf16 [CAP][H]; combine with moe_unpermute_combine;
 *   saved_gu        out bf16 [CAP][2I] or NULL: g and u for grouped_mlp_bwd_fp8_tensor.
 */
moe_status grouped_mlp_fwd_fp8_tensor(const moe_dims* d, const uint8_t* xq, const float* amax_x,
                                      const int32_t* split_sizes, const float* prob_perm, const uint8_t* wgu_q,
                                      const float* amax_gu, const uint8_t* wd_q, const float* amax_d, void* a_perm,
                                      uint8_t* aq, float* amax_a, void* y, void* saved_gu, void* workspace,
                                      size_t workspace_bytes, moe_stream_t stream);

/*
 * grouped_mlp_bwd_fp8_tensor -- backward of grouped_mlp_fwd_fp8_tensor with
 * straight-through per-tensor quantizers (one dynamic scale per expert operand
 * tensor; E4M3 for the gradients too).  A per-tensor scale does not depend on
 * the axis, so the operands of the weight-gradient GEMMs are the forward's codes
 * and dY's and dH's codes, transposed.  Steps: dY = dout gathered, its amax per
 * expert and codes; dA = dY*W_d (kind::f8f6f4) with the SwiGLU backward fused,
 * writing dH in bf16 and raising each expert's amax of dH; dH codes; dW_d =
 * dY^T*a and dW_gu = dH^T*x over each expert's tokens; dX = dH*W_gu.
 *   dout            bf16 [T][H]
 *   idx, split_sizes, row_of, prob_perm: from moe_route_permute
 *   saved_gu        bf16 [CAP][2I]: the saved_gu output of grouped_mlp_fwd_fp8_tensor
 *   xq, amax_x      from moe_fp8_tensor_quantize_tokens
 *   aq, amax_a      from grouped_mlp_fwd_fp8_tensor
 *   wgu_q, amax_gu, wd_q, amax_d: fp8_tensor_quantize of W_gu, W_d
 *   dx_perm         out bf16 [CAP][H]; combine it with moe_unpermute_combine
 *   dwgu, dwd       out bf16 [E][2I][H], [E][H][I] (zeros for experts without tokens)
 *   dprob           out f32 [T][k]
 *   workspace       moe_workspace_size(d, 3) bytes
 */
moe_status grouped_mlp_bwd_fp8_tensor(const moe_dims* d, const void* dout, const int32_t* idx,
                                      const int32_t* split_sizes, const int32_t* row_of, const float* prob_perm,
                                      const void* saved_gu, const uint8_t* xq, const float* amax_x,
                                      const uint8_t* aq, const float* amax_a, const uint8_t* wgu_q,
                                      const float* amax_gu, const uint8_t* wd_q, const float* amax_d, void* dx_perm,
                                      void* dwgu, void* dwd, float* dprob, void* workspace, size_t workspace_bytes,
                                      moe_stream_t stream);

/*
 * grouped_mlp_bwd -- backward of grouped_mlp_fwd with straight-through
 * quantizers (page "Efficient MoE Training for Biological Foundation
 * Models", section "MXFP8与融合MLP": the fused op has a matching backward).
 *   dout          bf16 [T][H]: gradient of the combined output
 *   split_sizes, row_of, src_of, prob_perm: from moe_route_permute
 *   saved_gu      bf16 [CAP][2I] from grouped_mlp_fwd
 *   aq_col,aq_col_scale  MX [I][CAP] from grouped_mlp_fwd
 *   xq_col,xq_col_scale  MX [H][CAP] from moe_route_permute
 *   wguT_q,wguT_s MX [E][H][2I] (mxfp8_quantize axis 1 of W_gu)
 *   wdT_q,wdT_s   MX [E][I][H]  (mxfp8_quantize axis 1 of W_d)
 *   dx_perm       out bf16 [CAP][H]: input gradient of every row; combine
 *                 it with moe_unpermute_combine to get dx [T][H]
 *   dwgu          out bf16 [E][2I][H]; dwd out bf16 [E][H][I] (zeros for
 *                 experts without tokens)
 *   dprob         out f32 [T][k]: gradient of prob
 * Steps: dY = dout gathered to rows and quantized along H and along tokens;
 * dA = dY*W_d (GEMM, K=H) with the SwiGLU backward fused in its epilogue
 * (dg = dA*p*u*silu'(g), du = dA*p*silu(g), dp = sum dA*silu(g)*u), writing
 * dH = [dg|du] quantized along 2I and along tokens; dW_d = dY^T*a (K = each
 * expert's tokens); dX = dH*W_gu (K = 2I); dW_gu = dH^T*x (K = tokens).
 */
moe_status grouped_mlp_bwd(const moe_dims* d, const void* dout,
                           const int32_t* split_sizes, const int32_t* row_of, const int32_t* src_of,
                           const float* prob_perm, const void* saved_gu,
                           const uint8_t* aq_col, const uint8_t* aq_col_scale,
                           const uint8_t* xq_col, const uint8_t* xq_col_scale,
                           const uint8_t* wguT_q, const uint8_t* wguT_s,
                           const uint8_t* wdT_q, const uint8_t* wdT_s,
                           void* dx_perm, void* dwgu, void* dwd, float* dprob,
                           void* workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * moe_unpermute_combine -- out[t] = sum over j of y_perm[row_of[t][j]]
 * (times prob[t][j] when prob != NULL), f32 sum in slot order, rounded to
 * bf16.  With the probability already applied in ScaledSwiGLU, prob is NULL
 * (page "Efficient MoE Training for Biological Foundation Models", section
 * "MXFP8与融合MLP").  Also combines dx_perm into dx.
 *   y_perm bf16 [CAP][H], row_of int32 [T][k], prob f32 [T][k] or NULL,
 *   out bf16 [T][H].
 */
moe_status moe_unpermute_combine(const moe_dims* d, const void* y_perm, const int32_t* row_of,
                                 const float* prob, void* out, moe_stream_t stream);

/*
 * moe_router_fwd -- router logits of a linear router: logits[t][e] =
 * sum_h x[t][h] * w_r[e][h] (page "英伟达开源MoE加速神器", section "三板斧":
 * each token is routed to a few experts; the pages give no router formula, a
 * bias-free linear map is the reading).  Computed on the tensor cores: bf16
 * products, f32 accumulation (the order of the partial sums is the MMA's).
 *   x bf16 [T][H], 16-byte aligned; w_r bf16 [E][H], 16-byte aligned;
 *   logits out f32 [T][E].
 *   workspace: the layer's workspace (moe_workspace_size of any mode); its
 *   error word records device-side failures (moe_get_device_error).
 */
moe_status moe_router_fwd(const moe_dims* d, const void* x, const void* w_r, float* logits, void* workspace,
                          size_t workspace_bytes, moe_stream_t stream);

/*
 * moe_router_bwd -- gradient of the router from dprob (grouped_mlp_bwd),
 * through the top-k softmax with the selection held fixed (page "Efficient
 * MoE Training for Biological Foundation Models", section "MXFP8与融合MLP":
 * the probabilities scale the SwiGLU output, so their gradient reaches the
 * router).
 *   renormalize=1: dlogits[t][e_j] = p_j (dp_j - sum_i p_i dp_i), 0 elsewhere;
 *   renormalize=0: dlogits[t][e] = s_e (g_e - sum_j p_j dp_j), s = softmax of the
 *                  row, g = dprob scattered to idx.
 *   logits f32 [T][E], idx int32 [T][k], prob f32 [T][k] (from
 *   moe_route_permute), dprob f32 [T][k]; dlogits out f32 [T][E];
 *   dx in/out bf16 [T][H]: dx[t] += sum_e dlogits[t][e] w_r[e] (f32 sum, one
 *   rounding to bf16); dw_r out f32 [E][H] = dlogits^T x on the tensor cores
 *   (dlogits as two bf16 terms hi + lo, float32-level accuracy), per fixed
 *   token chunk, the chunks summed in chunk order (deterministic).
 *   workspace: as for grouped_mlp_bwd (moe_workspace_size with training).
 */
moe_status moe_router_bwd(const moe_dims* d, const void* x, const void* w_r, const float* logits,
                          const int32_t* idx, const float* prob, const float* dprob, float* dlogits,
                          void* dx, float* dw_r, void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* moe_selftest_wait_timeout -- exercises the device-side failure path without
 * faulting anything.  One launch of the grouped GEMM kernel over a single
 * 128x256x128 tile whose producer is told to issue no loads: the MMA, scale
 * copy and epilogue warps wait for data that never comes, each wait runs out
 * after limit_ns (1 ms .. 2 s), the kernel records MOE_ERR_DEVICE_TIMEOUT and a
 * site id, frees its tensor memory and returns.  Synchronises `stream` and
 * returns the recorded *code and *site (expected: MOE_ERR_DEVICE_TIMEOUT and a
 * site in 500..599).  scratch: >= 96 KB of device memory, 256-byte aligned,
 * overwritten.  The context stays usable afterwards. */
moe_status moe_selftest_wait_timeout(void* scratch, size_t scratch_bytes, int64_t limit_ns, int32_t* code,
                                     int32_t* site, moe_stream_t stream);

/*
 * moe_workspace_tensor -- where an intermediate tensor of the layer sits in a
 * workspace of moe_workspace_size(d, training) bytes, for callers that want to
 * inspect it (the tests compare these against the oracle).  The pages have no
 * counterpart: these are the quantized operands the fused ops of page
 * "Efficient MoE Training for Biological Foundation Models", section
 * "MXFP8与融合MLP", keep internal.  *offset = byte offset from the workspace
 * start (256-aligned), *bytes = size.  Layouts as documented for MX tensors:
 *   MOE_WS_A_CODES / _SCALES        a = silu(g)*u*p, rows along I [CAP][I]
 *                                   (written by grouped_mlp_fwd)
 *   MOE_WS_DY_CODES / _SCALES       dY = dout gathered to rows, along H [CAP][H]
 *   MOE_WS_DY_COL_CODES / _SCALES   dY along tokens, transposed [H][CAP]
 *   MOE_WS_DH_CODES / _SCALES       dH = [dg | du], rows along 2I [CAP][2I]
 *   MOE_WS_DH_COL_CODES / _SCALES   dH along tokens, transposed [2I][CAP]
 * (the DY and DH tensors are written by grouped_mlp_bwd and exist only for
 * training >= 1).  Contents are valid after the writing call completes and
 * until the next call that writes the same workspace.  Host only.
 */
enum moe_ws_tensor {
  MOE_WS_A_CODES = 0, MOE_WS_A_SCALES = 1,
  MOE_WS_DY_CODES = 2, MOE_WS_DY_SCALES = 3, MOE_WS_DY_COL_CODES = 4, MOE_WS_DY_COL_SCALES = 5,
  MOE_WS_DH_CODES = 6, MOE_WS_DH_SCALES = 7, MOE_WS_DH_COL_CODES = 8, MOE_WS_DH_COL_SCALES = 9
};
moe_status moe_workspace_tensor(const moe_dims* d, int32_t training, int32_t which, size_t* offset, size_t* bytes);

/*
 * moe_selftest_epilogue_quant -- runs the MX quantizers of the GEMM epilogues
 * (the ones that write a after ScaledSwiGLU and dH after the SwiGLU backward;
 * page "Efficient MoE Training for Biological Foundation Models", section
 * "MXFP8与融合MLP": quantization is fused into the grouped MLP) on a caller's
 * float32 tensor, so that their codes can be checked bit for bit on inputs with
 * full 24-bit significands.  Each warp holds one 32x32 block the way an
 * epilogue warp holds its accumulator columns (lane = row).
 *   src      f32 [rows][cols] (rows, cols multiples of 128)
 *   codes, scales      out MX [rows][cols], blocks of 32 along cols (codes
 *                      32-byte aligned: each row block is one 256-bit store)
 *   codes_t, scales_t  out MX [cols][rows], blocks of 32 along rows
 *                      (the tensor transposed, as the along-token copies)
 */
moe_status moe_selftest_epilogue_quant(const float* src, int32_t rows, int32_t cols, uint8_t* codes,
                                       uint8_t* scales, uint8_t* codes_t, uint8_t* scales_t, moe_stream_t stream);

/*
 * moe_selftest_mma_issue -- the tensor pipe's MXFP8 issue ceiling for the GEMM's
 * instruction mix, a measurement aid with no counterpart in the pages.  One
 * launch of SMs/2 CTA pairs (one CTA per SM); in each pair one thread issues
 * k_steps K steps, each three scale-factor copies (tcgen05.cp) and four
 * tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale of M=256, N=256, K=32,
 * on operands resident in shared memory (zeros), with no loads and no
 * epilogue.  FLOPs of the launch = *pairs * k_steps * 2*256*256*128; time it
 * with events on `stream`.  scratch >= 256 bytes, 256-byte aligned, zeroed by
 * the caller: its first 8 bytes are a device error word (moe_get_device_error).
 */
moe_status moe_selftest_mma_issue(int32_t k_steps, void* scratch, size_t scratch_bytes, int32_t* pairs,
                                  moe_stream_t stream);

/* Read (and keep) the device error word of a workspace: *code is a
 * moe_status (MOE_OK if none), *site identifies the kernel and wait.
 * Synchronises `stream`. */
moe_status moe_get_device_error(const void* workspace, int32_t* code, int32_t* site, moe_stream_t stream);

/* Zero the device error word of a workspace (asynchronous on stream). */
moe_status moe_clear_device_error(void* workspace, moe_stream_t stream);

/*
 * moe_route_permute_noalloc -- moe_route_permute for callers that cannot
 * allocate device memory for the library.  The pages have no counterpart of
 * this entry point; it is an interface addition of this library.
 *
 * Some callers own no allocator they may use here: a plugin inside a host
 * framework that hands over only the layer's inputs and outputs, or a serving
 * loop whose memory is planned at start-up and where a cudaMalloc (which can
 * synchronise the device) is not allowed.  They cannot supply the workspace
 * that moe_route_permute needs for its two permutation tables (a 32-bit ballot
 * mask and a 32-bit running count per expert and 32-token group), so this
 * variant takes them from a fixed array compiled into the library.
 *
 * Arguments and results are exactly those of moe_route_permute, minus the
 * workspace.  Limits: everything moe_route_permute accepts, and in addition
 * E * ceil(T/32) <= 262144 (for example T = 32768 tokens with E up to 256
 * experts); larger sizes return MOE_ERR_UNSUPPORTED with a message naming the
 * limit.  The array takes 2 MiB + 256 bytes of device memory on every GPU
 * that loads the library, held until the process exits.  The call allocates
 * nothing.
 *
 * The first call on each device looks up the array's device address with that
 * device current and caches it with the id of the device's context; a call
 * under a new context (after cudaDeviceReset) looks it up again.  Make the
 * first call on a device, and the first after a reset, before any stream
 * capture.  All calls share the one array and each call rewrites it (only its
 * error word is cleared at the start of a call): calls whose kernels overlap on
 * the GPU -- different streams, or threads without ordering between them --
 * race and corrupt each other's permutation, so order them.  The array's own
 * error word cannot be read through this interface; instead a (token, slot)
 * that the kernels had to skip is marked -1 in idx and row_of (no valid input
 * produces one: every row selects k real experts, NaN logits included).
 */
moe_status moe_route_permute_noalloc(const moe_dims* d, const float* logits, const void* x,
                                     int32_t* idx, float* prob, int32_t* split_sizes,
                                     int32_t* row_of, int32_t* src_of, float* prob_perm,
                                     uint8_t* xq, uint8_t* xq_scale, uint8_t* xq_col, uint8_t* xq_col_scale,
                                     moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FFN_H */
