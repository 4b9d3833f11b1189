// C ABI of libmoeffn (declared and documented in include/moe_ffn.h): argument
// checks, workspace layout and the launch sequence of every entry point.
#include <cstdarg>
#include <cstdio>

#include "kernels.cuh"

using namespace moe;

namespace {

thread_local char g_msg[kLastErrorBytes] = "";

moe_status fail(moe_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return s;
}

moe_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

int64_t capacity(const moe_dims* d) { return round_up(int64_t(d->T) * d->k, 128) + 128 * int64_t(d->E); }

moe_status check_dims(const moe_dims* d) {
  if (d == nullptr) return fail(MOE_ERR_INVALID_ARG, "dims is NULL");
  if (d->T < 1) return fail(MOE_ERR_INVALID_ARG, "T=%d must be >= 1", d->T);
  if (d->H < 128 || d->H % 128) return fail(MOE_ERR_UNSUPPORTED, "H=%d must be a positive multiple of 128", d->H);
  if (d->I < 128 || d->I % 128) return fail(MOE_ERR_UNSUPPORTED, "I=%d must be a positive multiple of 128", d->I);
  if (d->E < 1 || d->E > 256) return fail(MOE_ERR_UNSUPPORTED, "E=%d must be in 1..256", d->E);
  if (d->k < 1 || d->k > 8 || d->k > d->E) return fail(MOE_ERR_UNSUPPORTED, "k=%d must be in 1..min(E,8)", d->k);
  if (d->H > 65536 || d->I > 65536) return fail(MOE_ERR_UNSUPPORTED, "H and I must be <= 65536");
  const int64_t cap = capacity(d);
  if (cap > (int64_t(1) << 30)) return fail(MOE_ERR_UNSUPPORTED, "T*k too large (row capacity %lld)", (long long)cap);
  if (int64_t(d->E) * 2 * d->I > (int64_t(1) << 30) || int64_t(d->E) * d->H > (int64_t(1) << 30))
    return fail(MOE_ERR_UNSUPPORTED, "E*2I or E*H too large for 32-bit TMA coordinates");
  return MOE_OK;
}

struct WsLayout {
  size_t err, masks, bases, aq, aq_s;
  size_t dyq, dyq_s, dyqc, dyqc_s, dhq, dhq_s, dhqc, dhqc_s, dp, rpart;
  size_t dy16, dy16c, dh16, dh16c, x16c, a16c;   // bf16 training: dY, dH and x, a transposed
  // per-tensor FP8 training: dY codes (rows, transposed), dH (bf16, codes, transposed codes),
  // x and a codes transposed, the weights' codes transposed, per-expert amax of dY and dH
  size_t t8dy, t8dyc, t8dh16, t8dh, t8dhc, t8xc, t8ac, t8wdT, t8wguT, t8amax;
  size_t total;
};

// mode 0: forward; 1: MXFP8 training; 2: bf16 training (the MXFP8 buffers plus bf16 ones);
// 3: per-tensor FP8 training (the MXFP8 buffers plus per-tensor ones)
WsLayout ws_layout(const moe_dims* d, int mode) {
  const bool training = mode != 0;
  WsLayout w{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) & ~size_t(255);
    return o;
  };
  const size_t cap = size_t(capacity(d));
  const size_t G = size_t((d->T + 31) / 32);
  const size_t H = size_t(d->H), I = size_t(d->I), E = size_t(d->E);
  w.err = take(256);
  w.masks = take(E * G * 4);
  w.bases = take(E * G * 4);
  w.aq = take(cap * I);
  w.aq_s = take(cap * I / 32);
  if (training) {
    const size_t ntI = (I + 255) / 256;             // 256-column tiles of the SwiGLU-backward GEMM
    w.dyq = take(cap * H);
    w.dyq_s = take(cap * H / 32);
    w.dyqc = take(H * cap);
    w.dyqc_s = take(H * cap / 32);
    w.dhq = take(cap * 2 * I);
    w.dhq_s = take(cap * 2 * I / 32);
    w.dhqc = take(2 * I * cap);
    w.dhqc_s = take(2 * I * cap / 32);
    w.dp = take(ntI * 4 * cap * 4);                 // one partial row sum per 64-column group
    w.rpart = take(router_ws_bytes(d->T, d->E, d->H));  // router backward: dW_r partials, dl hi/lo
  }
  if (mode == 3) {
    w.t8dy = take(cap * H);
    w.t8dyc = take(H * cap);
    w.t8dh16 = take(cap * 2 * I * 2);
    w.t8dh = take(cap * 2 * I);
    w.t8dhc = take(2 * I * cap);
    w.t8xc = take(H * cap);
    w.t8ac = take(I * cap);
    w.t8wdT = take(E * I * H);
    w.t8wguT = take(E * H * 2 * I);
    w.t8amax = take(2 * E * 4);
  }
  if (mode == 2) {
    w.dy16 = take(cap * H * 2);
    w.dy16c = take(H * cap * 2);
    w.dh16 = take(cap * 2 * I * 2);
    w.dh16c = take(2 * I * cap * 2);
    w.x16c = take(H * cap * 2);
    w.a16c = take(I * cap * 2);
  }
  w.total = off;
  return w;
}

moe_status check_ws(const moe_dims* d, const void* ws, size_t bytes, int mode) {
  if (ws == nullptr) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return fail(MOE_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  const size_t need = ws_layout(d, mode).total;
  if (bytes < need) return fail(MOE_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", bytes, need);
  return MOE_OK;
}

#define REQUIRE_PTR(p)                                                                         \
  do {                                                                                         \
    if ((p) == nullptr) return fail(MOE_ERR_INVALID_ARG, "%s is NULL", #p);                   \
    if (!al16(p)) return fail(MOE_ERR_ALIGNMENT, "%s is not 16-byte aligned", #p);            \
  } while (0)

#define CUDA_TRY(expr, what)                                                                   \
  do {                                                                                         \
    cudaError_t e_ = (expr);                                                                   \
    if (e_ != cudaSuccess) return cuda_fail(e_, what);                                         \
  } while (0)

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

}  // namespace

char* moe::last_error_buffer() { return g_msg; }
moe_status moe::check_layer_dims(const moe_dims* d) { return check_dims(d); }
int64_t moe::rows_capacity(const moe_dims* d) { return capacity(d); }

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_ALIGNMENT: return "MOE_ERR_ALIGNMENT";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT";
    case MOE_ERR_DEVICE_BOUNDS: return "MOE_ERR_DEVICE_BOUNDS";
  }
  return "MOE_ERR_UNKNOWN";
}

const char* moe_last_error_message(void) { return g_msg; }

size_t moe_rows_capacity(const moe_dims* d) {
  if (check_dims(d) != MOE_OK) return 0;
  return size_t(capacity(d));
}

size_t moe_workspace_size(const moe_dims* d, int32_t training) {
  if (check_dims(d) != MOE_OK) return 0;
  if (training < 0 || training > 3) return 0;
  return ws_layout(d, training).total;
}

moe_status mxfp8_quantize(const void* src, int32_t batch, int32_t rows, int32_t cols, int32_t axis,
                          uint8_t* codes, uint8_t* scales, moe_stream_t stream) {
  g_msg[0] = 0;
  REQUIRE_PTR(src);
  REQUIRE_PTR(codes);
  REQUIRE_PTR(scales);
  if (batch < 1 || rows < 128 || cols < 128 || rows % 128 || cols % 128)
    return fail(MOE_ERR_UNSUPPORTED, "batch=%d rows=%d cols=%d: need batch>=1 and rows, cols multiples of 128",
                batch, rows, cols);
  if (axis != 0 && axis != 1) return fail(MOE_ERR_INVALID_ARG, "axis=%d must be 0 or 1", axis);
  if (int64_t(batch) * rows > (int64_t(1) << 31) / 1 || int64_t(batch) * cols > (int64_t(1) << 31))
    return fail(MOE_ERR_UNSUPPORTED, "tensor too large");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (axis == 0) {
    const int64_t n = int64_t(batch) * rows;
    CUDA_TRY(launch_quant_rowwise(src, n, cols, nullptr, 1, n, codes, scales, nullptr, st), "quant_rowwise");
  } else {
    CUDA_TRY(launch_quant_colwise(src, nullptr, int64_t(batch) * rows, batch, rows, cols, nullptr, 0, codes, scales,
                                  nullptr, st),
             "quant_colwise");
  }
  return MOE_OK;
}

moe_status mxfp8_quantize_dual(const void* src, int32_t batch, int32_t rows, int32_t cols, uint8_t* codes,
                               uint8_t* scales, uint8_t* codes_t, uint8_t* scales_t, moe_stream_t stream) {
  g_msg[0] = 0;
  REQUIRE_PTR(src);
  REQUIRE_PTR(codes);
  REQUIRE_PTR(scales);
  REQUIRE_PTR(codes_t);
  REQUIRE_PTR(scales_t);
  if (batch < 1 || rows < 128 || cols < 128 || rows % 128 || cols % 128)
    return fail(MOE_ERR_UNSUPPORTED, "batch=%d rows=%d cols=%d: need batch>=1 and rows, cols multiples of 128",
                batch, rows, cols);
  if (int64_t(batch) * rows > (int64_t(1) << 31) || int64_t(batch) * cols > (int64_t(1) << 31) || batch > 65535)
    return fail(MOE_ERR_UNSUPPORTED, "tensor too large");
  CUDA_TRY(launch_quant_dual(src, batch, rows, cols, codes, scales, codes_t, scales_t,
                             static_cast<cudaStream_t>(stream)),
           "quant_dual");
  return MOE_OK;
}

}  // extern "C"

namespace {
// The host array of per-expert weight pointers, checked and copied into a kernel parameter table.
moe_status expert_table(const void* const* w, int32_t E, ExpertSrc* tbl) {
  if (w == nullptr) return fail(MOE_ERR_INVALID_ARG, "the expert pointer array is NULL");
  if (E < 1 || E > kMaxExpertPtrs) return fail(MOE_ERR_UNSUPPORTED, "E=%d must be in 1..%d", E, kMaxExpertPtrs);
  for (int e = 0; e < E; ++e) {
    if (w[e] == nullptr) return fail(MOE_ERR_INVALID_ARG, "the weight pointer of expert %d is NULL", e);
    if (!al16(w[e])) return fail(MOE_ERR_ALIGNMENT, "the weight of expert %d is not 16-byte aligned", e);
    tbl->p[e] = static_cast<const __nv_bfloat16*>(w[e]);
  }
  for (int e = E; e < kMaxExpertPtrs; ++e) tbl->p[e] = nullptr;
  return MOE_OK;
}
}  // namespace

extern "C" {

moe_status mxfp8_quantize_experts(const void* const* w, int32_t E, int32_t rows, int32_t cols, uint8_t* codes,
                                  uint8_t* scales, uint8_t* codes_t, uint8_t* scales_t, moe_stream_t stream) {
  g_msg[0] = 0;
  REQUIRE_PTR(codes);
  REQUIRE_PTR(scales);
  if ((codes_t == nullptr) != (scales_t == nullptr))
    return fail(MOE_ERR_INVALID_ARG, "codes_t and scales_t must both be given or both be NULL");
  if (codes_t != nullptr) {
    REQUIRE_PTR(codes_t);
    REQUIRE_PTR(scales_t);
  }
  if (rows < 128 || cols < 128 || rows % 128 || cols % 128)
    return fail(MOE_ERR_UNSUPPORTED, "rows=%d cols=%d: need multiples of 128", rows, cols);
  if (int64_t(E) * rows > (int64_t(1) << 31) || int64_t(E) * cols > (int64_t(1) << 31))
    return fail(MOE_ERR_UNSUPPORTED, "tensor too large");
  ExpertSrc tbl;
  moe_status s = expert_table(w, E, &tbl);
  if (s != MOE_OK) return s;
  CUDA_TRY(launch_quant_dual_experts(tbl, E, rows, cols, codes, scales, codes_t, scales_t,
                                     static_cast<cudaStream_t>(stream)),
           "quant_dual (per-expert pointers)");
  return MOE_OK;
}

moe_status fp8_tensor_quantize_experts(const void* const* w, int32_t E, int32_t rows, int32_t cols, uint8_t* codes,
                                       float* amax, moe_stream_t stream) {
  g_msg[0] = 0;
  REQUIRE_PTR(codes);
  if (amax == nullptr) return fail(MOE_ERR_INVALID_ARG, "amax is NULL");
  if (rows < 1 || cols < 8 || cols % 8)
    return fail(MOE_ERR_UNSUPPORTED, "rows=%d cols=%d: need rows >= 1 and cols a multiple of 8", rows, cols);
  ExpertSrc tbl;
  moe_status s = expert_table(w, E, &tbl);
  if (s != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t per = int64_t(rows) * cols;
  uint32_t* am = reinterpret_cast<uint32_t*>(amax);
  CUDA_TRY(cudaMemsetAsync(am, 0, sizeof(uint32_t) * size_t(E), st), "clear amax");
  CUDA_TRY(launch_t8_amax_experts(tbl, E, per, am, st), "per-tensor amax (per-expert pointers)");
  CUDA_TRY(launch_t8_quant_experts(tbl, E, per, am, codes, st), "per-tensor quantize (per-expert pointers)");
  return MOE_OK;
}

moe_status moe_route_permute(const moe_dims* d, const float* logits, const void* x, int32_t* idx, float* prob,
                             int32_t* split_sizes, int32_t* row_of, int32_t* src_of, float* prob_perm,
                             uint8_t* xq, uint8_t* xq_scale, uint8_t* xq_col, uint8_t* xq_col_scale,
                             void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  g_msg[0] = 0;
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  REQUIRE_PTR(logits);
  REQUIRE_PTR(x);
  REQUIRE_PTR(idx);
  REQUIRE_PTR(prob);
  REQUIRE_PTR(split_sizes);
  REQUIRE_PTR(row_of);
  REQUIRE_PTR(src_of);
  REQUIRE_PTR(prob_perm);
  REQUIRE_PTR(xq);
  REQUIRE_PTR(xq_scale);
  if ((xq_col == nullptr) != (xq_col_scale == nullptr))
    return fail(MOE_ERR_INVALID_ARG, "xq_col and xq_col_scale must both be set or both be NULL");
  if (xq_col != nullptr) {
    REQUIRE_PTR(xq_col);
    REQUIRE_PTR(xq_col_scale);
  }
  s = check_ws(d, workspace, workspace_bytes, false);
  if (s != MOE_OK) return s;
  const WsLayout w = ws_layout(d, false);
  int* err = at<int>(workspace, w.err);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t cap = capacity(d);
  uint32_t* masks = at<uint32_t>(workspace, w.masks);
  int* bases = at<int>(workspace, w.bases);
  CUDA_TRY(launch_route_scan(logits, d->T, d->E, d->k, d->renormalize, idx, prob, masks, bases, split_sizes,
                             route_ticket(err), err, st),
           "route + scan");
  const PermuteRows pr{idx, prob, masks, bases, split_sizes, d->E, (d->T + 31) / 32, row_of, src_of, prob_perm};
  CUDA_TRY(launch_permute_quant_rows(x, d->T, d->H, d->k, cap, pr, xq, xq_scale, err, st),
           "permutation + gather_quant_rowwise + padding rows");
  if (xq_col != nullptr)
    CUDA_TRY(launch_quant_colwise(x, src_of, d->T, 1, int(cap), d->H, split_sizes, d->E, xq_col, xq_col_scale, err,
                                  st),
             "gather_quant_colwise");
  return MOE_OK;
}

moe_status moe_route(const moe_dims* d, const float* logits, int32_t* idx, float* prob, int32_t* split_sizes,
                     int32_t* row_of, int32_t* src_of, float* prob_perm, void* workspace, size_t workspace_bytes,
                     moe_stream_t stream) {
  g_msg[0] = 0;
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  REQUIRE_PTR(logits);
  REQUIRE_PTR(idx);
  REQUIRE_PTR(prob);
  REQUIRE_PTR(split_sizes);
  REQUIRE_PTR(row_of);
  REQUIRE_PTR(src_of);
  REQUIRE_PTR(prob_perm);
  s = check_ws(d, workspace, workspace_bytes, false);
  if (s != MOE_OK) return s;
  const WsLayout w = ws_layout(d, false);
  int* err = at<int>(workspace, w.err);
  CUDA_TRY(launch_route_permute(logits, d->T, d->E, d->k, d->renormalize, idx, prob, at<uint32_t>(workspace, w.masks),
                                at<int>(workspace, w.bases), split_sizes, row_of, src_of, prob_perm,
                                route_ticket(err), err, static_cast<cudaStream_t>(stream)),
           "route");
  return MOE_OK;
}

moe_status moe_permute(const moe_dims* d, const int32_t* idx, const float* prob, const void* x, int32_t* split_sizes,
                       int32_t* row_of, int32_t* src_of, float* prob_perm, uint8_t* xq, uint8_t* xq_scale,
                       uint8_t* xq_col, uint8_t* xq_col_scale, void* workspace, size_t workspace_bytes,
                       moe_stream_t stream) {
  g_msg[0] = 0;
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  REQUIRE_PTR(idx);
  REQUIRE_PTR(prob);
  REQUIRE_PTR(x);
  REQUIRE_PTR(split_sizes);
  REQUIRE_PTR(row_of);
  REQUIRE_PTR(src_of);
  REQUIRE_PTR(prob_perm);
  REQUIRE_PTR(xq);
  REQUIRE_PTR(xq_scale);
  if ((xq_col == nullptr) != (xq_col_scale == nullptr))
    return fail(MOE_ERR_INVALID_ARG, "xq_col and xq_col_scale must both be set or both be NULL");
  if (xq_col != nullptr) {
    REQUIRE_PTR(xq_col);
    REQUIRE_PTR(xq_col_scale);
  }
  s = check_ws(d, workspace, workspace_bytes, false);
  if (s != MOE_OK) return s;
  const WsLayout w = ws_layout(d, false);
  int* err = at<int>(workspace, w.err);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t cap = capacity(d);
  CUDA_TRY(launch_permute_from_idx(idx, prob, d->T, d->E, d->k, at<uint32_t>(workspace, w.masks),
                                   at<int>(workspace, w.bases), split_sizes, row_of, src_of, prob_perm, err, st),
           "permute");
  CUDA_TRY(launch_quant_rowwise(x, d->T, d->H, row_of, d->k, cap, xq, xq_scale, err, st, split_sizes, d->E),
           "gather_quant_rowwise + padding rows");
  if (xq_col != nullptr)
    CUDA_TRY(launch_quant_colwise(x, src_of, d->T, 1, int(cap), d->H, split_sizes, d->E, xq_col, xq_col_scale, err,
                                  st),
             "gather_quant_colwise");
  return MOE_OK;
}

moe_status moe_ep_pack(const moe_dims* d, int32_t world, const void* x, const int32_t* idx, const float* prob,
                       const int32_t* row_of, const int32_t* split_sizes, void* send_x, float* send_prob,
                       int32_t* send_eid, int32_t* pos_of, int32_t* rank_counts, void* workspace,
                       size_t workspace_bytes, moe_stream_t stream) {
  g_msg[0] = 0;
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  if (world < 1 || world > d->E || d->E % world != 0)
    return fail(MOE_ERR_UNSUPPORTED, "world=%d must divide E=%d", world, d->E);
  REQUIRE_PTR(x);
  REQUIRE_PTR(idx);
  REQUIRE_PTR(prob);
  REQUIRE_PTR(row_of);
  REQUIRE_PTR(split_sizes);
  REQUIRE_PTR(send_x);
  REQUIRE_PTR(send_prob);
  REQUIRE_PTR(send_eid);
  REQUIRE_PTR(pos_of);
  REQUIRE_PTR(rank_counts);
  s = check_ws(d, workspace, workspace_bytes, false);
  if (s != MOE_OK) return s;
  const WsLayout w = ws_layout(d, false);
  CUDA_TRY(launch_ep_pack(x, idx, prob, row_of, split_sizes, d->T, d->H, d->E, d->k, world, send_x, send_prob,
                          send_eid, pos_of, rank_counts, at<int>(workspace, w.err), static_cast<cudaStream_t>(stream)),
           "expert-parallel pack");
  return MOE_OK;
}

moe_status moe_gather_f32(const float* src, int64_t n_src, const int32_t* map, int64_t n, float* out,
                          void* workspace, moe_stream_t stream) {
  g_msg[0] = 0;
  if (n < 0 || n_src < 0) return fail(MOE_ERR_INVALID_ARG, "negative size");
  if (n == 0) return MOE_OK;
  if (src == nullptr || map == nullptr || out == nullptr || workspace == nullptr)
    return fail(MOE_ERR_INVALID_ARG, "src, map, out and workspace must be non-NULL");
  if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(map)) & 3u)
    return fail(MOE_ERR_ALIGNMENT, "src, map and out must be 4-byte aligned");
  CUDA_TRY(launch_gather_f32(src, n_src, map, n, out, static_cast<int*>(workspace),
                             static_cast<cudaStream_t>(stream)),
           "gather f32");
  return MOE_OK;
}

moe_status grouped_mlp_fwd(const moe_dims* d, const uint8_t* xq, const uint8_t* xq_scale, const int32_t* split_sizes,
                           const float* prob_perm, const uint8_t* wgu_q, const uint8_t* wgu_s, const uint8_t* wd_q,
                           const uint8_t* wd_s, void* y, void* saved_gu, uint8_t* aq_col, uint8_t* aq_col_scale,
                           void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  g_msg[0] = 0;
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  REQUIRE_PTR(xq);
  REQUIRE_PTR(xq_scale);
  REQUIRE_PTR(split_sizes);
  REQUIRE_PTR(prob_perm);
  REQUIRE_PTR(wgu_q);
  REQUIRE_PTR(wgu_s);
  REQUIRE_PTR(wd_q);
  REQUIRE_PTR(wd_s);
  REQUIRE_PTR(y);
  if (saved_gu != nullptr) REQUIRE_PTR(saved_gu);
  if ((aq_col == nullptr) != (aq_col_scale == nullptr))
    return fail(MOE_ERR_INVALID_ARG, "aq_col and aq_col_scale must both be set or both be NULL");
  if (aq_col != nullptr) {
    REQUIRE_PTR(aq_col);
    REQUIRE_PTR(aq_col_scale);
  }
  s = check_ws(d, workspace, workspace_bytes, false);
  if (s != MOE_OK) return s;
  const WsLayout w = ws_layout(d, false);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t cap = capacity(d);
  const int H = d->H, I = d->I, E = d->E;

  GemmArgs g1{};
  g1.mode = 0;
  g1.E = E;
  g1.split_sizes = split_sizes;
  g1.K = H;
  g1.N = I;
  g1.n_tiles = I / 128;
  g1.b_rows_per_expert = 2 * int64_t(I);
  g1.cap = cap;
  g1.sfa = xq_scale;
  g1.sfb = wgu_s;
  g1.sfa_K = H;
  g1.sfb_K = H;
  g1.prob_perm = prob_perm;
  g1.q_row = at<uint8_t>(workspace, w.aq);
  g1.q_row_s = at<uint8_t>(workspace, w.aq_s);
  g1.q_row_K = I;
  g1.q_col = aq_col;
  g1.q_col_s = aq_col_scale;
  g1.gu = static_cast<__nv_bfloat16*>(saved_gu);
  g1.I = I;
  g1.err = at<int>(workspace, w.err);
  CUDA_TRY(launch_grouped_gemm(EPI_FWD_SWIGLU, g1, xq, cap, H, wgu_q, int64_t(E) * 2 * I, H, (cap / 128) * g1.n_tiles,
                               st, g_msg, sizeof(g_msg)),
           "grouped gate_up GEMM");

  GemmArgs g2{};
  g2.mode = 0;
  g2.E = E;
  g2.split_sizes = split_sizes;
  g2.K = I;
  g2.N = H;
  g2.n_tiles = (H + 255) / 256;
  g2.b_rows_per_expert = H;
  g2.cap = cap;
  g2.sfa = g1.q_row_s;
  g2.sfb = wd_s;
  g2.sfa_K = I;
  g2.sfb_K = I;
  g2.out = static_cast<__nv_bfloat16*>(y);
  g2.ldo = H;
  g2.I = I;
  g2.err = g1.err;
  CUDA_TRY(launch_grouped_gemm(EPI_BF16, g2, g1.q_row, cap, I, wd_q, int64_t(E) * H, I, (cap / 128) * g2.n_tiles, st,
                               g_msg, sizeof(g_msg)),
           "grouped down GEMM");
  return MOE_OK;
}

moe_status moe_gather_rows(const moe_dims* d, const void* x, const int32_t* row_of, const int32_t* split_sizes,
                           void* x_perm, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  g_msg[0] = 0;
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  REQUIRE_PTR(x);
  REQUIRE_PTR(row_of);
  REQUIRE_PTR(split_sizes);
  REQUIRE_PTR(x_perm);
  s = check_ws(d, workspace, workspace_bytes, false);
  if (s != MOE_OK) return s;
  const WsLayout w = ws_layout(d, false);
  CUDA_TRY(launch_gather_rows(x, row_of, split_sizes, d->T, d->k, d->H, d->E, capacity(d), x_perm,
                              at<int>(workspace, w.err), static_cast<cudaStream_t>(stream)),
           "gather rows");
  return MOE_OK;
}

moe_status grouped_mlp_fwd_bf16(const moe_dims* d, const void* x_perm, const int32_t* split_sizes,
                                const float* prob_perm, const void* w_gu, const void* w_d, void* a_perm, void* y,
                                void* saved_gu, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  g_msg[0] = 0;
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  REQUIRE_PTR(x_perm);
  REQUIRE_PTR(split_sizes);
  REQUIRE_PTR(prob_perm);
  REQUIRE_PTR(w_gu);
  REQUIRE_PTR(w_d);
  REQUIRE_PTR(a_perm);
  REQUIRE_PTR(y);
  s = check_ws(d, workspace, workspace_bytes, false);
  if (s != MOE_OK) return s;
  const WsLayout w = ws_layout(d, false);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t cap = capacity(d);
  const int H = d->H, I = d->I, E = d->E;
  GemmArgs g1{};
  g1.mode = 0;
  g1.E = E;
  g1.split_sizes = split_sizes;
  g1.K = H;
  g1.N = I;
  g1.n_tiles = I / 128;
  g1.b_rows_per_expert = 2 * int64_t(I);
  g1.cap = cap;
  g1.prob_perm = prob_perm;
  g1.out = static_cast<__nv_bfloat16*>(a_perm);
  g1.ldo = I;
  g1.gu = static_cast<__nv_bfloat16*>(saved_gu);
  g1.I = I;
  g1.err = at<int>(workspace, w.err);
  if (saved_gu != nullptr && !al16(saved_gu)) return fail(MOE_ERR_ALIGNMENT, "saved_gu is not 16-byte aligned");
  CUDA_TRY(launch_grouped_gemm(EPI_B16_FWD_SWIGLU, g1, x_perm, cap, H, w_gu, int64_t(E) * 2 * I, H,
                               (cap / 128) * g1.n_tiles, st, g_msg, sizeof(g_msg)),
           "bf16 grouped gate_up GEMM");
  GemmArgs g2{};
  g2.mode = 0;
  g2.E = E;
  g2.split_sizes = split_sizes;
  g2.K = I;
  g2.N = H;
  g2.n_tiles = (H + 255) / 256;
  g2.b_rows_per_expert = H;
  g2.cap = cap;
  g2.out = static_cast<__nv_bfloat16*>(y);
  g2.ldo = H;
  g2.I = I;
  g2.err = g1.err;
  CUDA_TRY(launch_grouped_gemm(EPI_B16_OUT, g2, a_perm, cap, I, w_d, int64_t(E) * H, I, (cap / 128) * g2.n_tiles,
                               st, g_msg, sizeof(g_msg)),
           "bf16 grouped down GEMM");
  return MOE_OK;
}

moe_status fp8_tensor_quantize(const void* src, int32_t batch, int32_t rows, int32_t cols, uint8_t* codes,
                               float* amax, moe_stream_t stream) {
  g_msg[0] = 0;
  REQUIRE_PTR(src);
  REQUIRE_PTR(codes);
  if (amax == nullptr) return fail(MOE_ERR_INVALID_ARG, "amax is NULL");
  if (batch < 1 || rows < 1 || cols < 8 || cols % 8)
    return fail(MOE_ERR_UNSUPPORTED, "batch=%d rows=%d cols=%d: need batch, rows >= 1 and cols a multiple of 8",
                batch, rows, cols);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t per = int64_t(rows) * cols;
  uint32_t* am = reinterpret_cast<uint32_t*>(amax);
  CUDA_TRY(cudaMemsetAsync(am, 0, sizeof(uint32_t) * size_t(batch), st), "clear amax");
  CUDA_TRY(launch_t8_amax_batches(src, batch, per, am, st), "per-tensor amax");
  CUDA_TRY(launch_t8_quant_batches(src, batch, per, am, codes, st), "per-tensor quantize");
  return MOE_OK;
}

moe_status moe_fp8_tensor_quantize_tokens(const moe_dims* d, const void* x, const int32_t* idx,
                                          const int32_t* row_of, const int32_t* split_sizes, uint8_t* xq,
                                          float* amax_x, void* workspace, size_t workspace_bytes,
                                          moe_stream_t stream) {
  g_msg[0] = 0;
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  REQUIRE_PTR(x);
  REQUIRE_PTR(idx);
  REQUIRE_PTR(row_of);
  REQUIRE_PTR(split_sizes);
  REQUIRE_PTR(xq);
  if (amax_x == nullptr) return fail(MOE_ERR_INVALID_ARG, "amax_x is NULL");
  s = check_ws(d, workspace, workspace_bytes, false);
  if (s != MOE_OK) return s;
  const WsLayout w = ws_layout(d, false);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* err = at<int>(workspace, w.err);
  uint32_t* am = reinterpret_cast<uint32_t*>(amax_x);
  CUDA_TRY(cudaMemsetAsync(am, 0, sizeof(uint32_t) * size_t(d->E), st), "clear amax_x");
  CUDA_TRY(launch_t8_amax_tokens(x, d->T, d->H, idx, d->k, d->E, am, err, st), "per-expert amax of x");
  CUDA_TRY(launch_t8_quant_tokens(x, d->T, d->H, idx, row_of, d->k, d->E, capacity(d), am, xq, err, st),
           "per-tensor quantize of x rows");
  CUDA_TRY(launch_fill_pad_rows(split_sizes, d->E, d->H, capacity(d), xq, nullptr, err, st), "padding rows of xq");
  return MOE_OK;
}

moe_status grouped_mlp_fwd_fp8_tensor(const moe_dims* d, const uint8_t* xq, const float* amax_x,
                                      const int32_t* split_sizes, const float* prob_perm, const uint8_t* wgu_q,
                                      const float* amax_gu, const uint8_t* wd_q, const float* amax_d, void* a_perm,
                                      uint8_t* aq, float* amax_a, void* y, void* saved_gu, void* workspace,
                                      size_t workspace_bytes, moe_stream_t stream) {
  g_msg[0] = 0;
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  REQUIRE_PTR(xq);
  REQUIRE_PTR(split_sizes);
  REQUIRE_PTR(prob_perm);
  REQUIRE_PTR(wgu_q);
  REQUIRE_PTR(wd_q);
  REQUIRE_PTR(a_perm);
  REQUIRE_PTR(aq);
  REQUIRE_PTR(y);
  if (amax_x == nullptr || amax_gu == nullptr || amax_d == nullptr || amax_a == nullptr)
    return fail(MOE_ERR_INVALID_ARG, "an amax array is NULL");
  s = check_ws(d, workspace, workspace_bytes, false);
  if (s != MOE_OK) return s;
  const WsLayout w = ws_layout(d, false);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t cap = capacity(d);
  const int H = d->H, I = d->I, E = d->E;
  uint32_t* am_a = reinterpret_cast<uint32_t*>(amax_a);
  CUDA_TRY(cudaMemsetAsync(am_a, 0, sizeof(uint32_t) * size_t(E), st), "clear amax_a");
  GemmArgs g1{};
  g1.mode = 0;
  g1.E = E;
  g1.split_sizes = split_sizes;
  g1.K = H;
  g1.N = I;
  g1.n_tiles = I / 128;
  g1.b_rows_per_expert = 2 * int64_t(I);
  g1.cap = cap;
  g1.prob_perm = prob_perm;
  g1.out = static_cast<__nv_bfloat16*>(a_perm);
  g1.ldo = I;
  g1.I = I;
  g1.amax_a = reinterpret_cast<const uint32_t*>(amax_x);
  g1.amax_b = reinterpret_cast<const uint32_t*>(amax_gu);
  g1.amax_out = am_a;
  g1.gu = static_cast<__nv_bfloat16*>(saved_gu);
  if (saved_gu != nullptr && !al16(saved_gu)) return fail(MOE_ERR_ALIGNMENT, "saved_gu is not 16-byte aligned");
  g1.err = at<int>(workspace, w.err);
  CUDA_TRY(launch_grouped_gemm(EPI_T8_FWD_SWIGLU, g1, xq, cap, H, wgu_q, int64_t(E) * 2 * I, H,
                               (cap / 128) * g1.n_tiles, st, g_msg, sizeof(g_msg)),
           "per-tensor FP8 grouped gate_up GEMM");
  CUDA_TRY(launch_t8_quant_segments(a_perm, split_sizes, E, cap, I, am_a, aq, st), "per-tensor quantize of a");
  GemmArgs g2{};
  g2.mode = 0;
  g2.E = E;
  g2.split_sizes = split_sizes;
  g2.K = I;
  g2.N = H;
  g2.n_tiles = (H + 255) / 256;
  g2.b_rows_per_expert = H;
  g2.cap = cap;
  g2.out = static_cast<__nv_bfloat16*>(y);
  g2.ldo = H;
  g2.I = I;
  g2.amax_a = am_a;
  g2.amax_b = reinterpret_cast<const uint32_t*>(amax_d);
  g2.err = g1.err;
  CUDA_TRY(launch_grouped_gemm(EPI_T8_OUT, g2, aq, cap, I, wd_q, int64_t(E) * H, I, (cap / 128) * g2.n_tiles, st,
                               g_msg, sizeof(g_msg)),
           "per-tensor FP8 grouped down GEMM");
  return MOE_OK;
}

moe_status moe_transpose_bf16(const void* src, int32_t batch, int32_t rows, int32_t cols, void* dst,
                              moe_stream_t stream) {
  g_msg[0] = 0;
  REQUIRE_PTR(src);
  REQUIRE_PTR(dst);
  if (batch < 1 || batch > 65535 || rows < 128 || cols < 128 || rows % 128 || cols % 128)
    return fail(MOE_ERR_UNSUPPORTED, "batch=%d rows=%d cols=%d: need 1 <= batch <= 65535 and rows, cols multiples "
                "of 128", batch, rows, cols);
  if (int64_t(batch) * rows > (int64_t(1) << 31) || int64_t(batch) * cols > (int64_t(1) << 31))
    return fail(MOE_ERR_UNSUPPORTED, "tensor too large");
  CUDA_TRY(launch_transpose_bf16(src, nullptr, int64_t(batch) * rows, batch, rows, cols, nullptr, 0, dst, nullptr,
                                 static_cast<cudaStream_t>(stream)),
           "transpose");
  return MOE_OK;
}

moe_status moe_transpose_bf16_experts(const void* const* src, int32_t E, int32_t rows, int32_t cols, void* dst,
                                      moe_stream_t stream) {
  g_msg[0] = 0;
  REQUIRE_PTR(dst);
  if (rows < 128 || cols < 128 || rows % 128 || cols % 128)
    return fail(MOE_ERR_UNSUPPORTED, "rows=%d cols=%d: need multiples of 128", rows, cols);
  if (int64_t(E) * rows > (int64_t(1) << 31) || int64_t(E) * cols > (int64_t(1) << 31))
    return fail(MOE_ERR_UNSUPPORTED, "tensor too large");
  ExpertSrc tbl;
  moe_status s = expert_table(src, E, &tbl);
  if (s != MOE_OK) return s;
  CUDA_TRY(launch_transpose_bf16_experts(tbl, E, rows, cols, dst, static_cast<cudaStream_t>(stream)),
           "transpose (per-expert pointers)");
  return MOE_OK;
}

moe_status grouped_mlp_fwd_bf16_experts(const moe_dims* d, const void* x_perm, const int32_t* split_sizes,
                                        const float* prob_perm, const void* const* w_gu, const void* const* w_d,
                                        void* a_perm, void* y, void* saved_gu, void* workspace,
                                        size_t workspace_bytes, moe_stream_t stream) {
  g_msg[0] = 0;
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  REQUIRE_PTR(x_perm);
  REQUIRE_PTR(split_sizes);
  REQUIRE_PTR(prob_perm);
  REQUIRE_PTR(a_perm);
  REQUIRE_PTR(y);
  if (saved_gu != nullptr) REQUIRE_PTR(saved_gu);
  if (d->E > 128) return fail(MOE_ERR_UNSUPPORTED, "E=%d: per-expert weight tensors take E <= 128", d->E);
  ExpertSrc tgu, td;                               // checks the pointer arrays (NULL, alignment)
  s = expert_table(w_gu, d->E, &tgu);
  if (s != MOE_OK) return s;
  s = expert_table(w_d, d->E, &td);
  if (s != MOE_OK) return s;
  s = check_ws(d, workspace, workspace_bytes, false);
  if (s != MOE_OK) return s;
  const WsLayout w = ws_layout(d, false);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t cap = capacity(d);
  const int H = d->H, I = d->I, E = d->E;
  GemmArgs g1{};
  g1.mode = 0;
  g1.E = E;
  g1.split_sizes = split_sizes;
  g1.K = H;
  g1.N = I;
  g1.n_tiles = I / 128;
  g1.b_rows_per_expert = 0;                        // B rows inside each expert's own tensor
  g1.cap = cap;
  g1.prob_perm = prob_perm;
  g1.out = static_cast<__nv_bfloat16*>(a_perm);
  g1.ldo = I;
  g1.gu = static_cast<__nv_bfloat16*>(saved_gu);
  g1.I = I;
  g1.err = at<int>(workspace, w.err);
  CUDA_TRY(launch_grouped_gemm(EPI_B16_FWD_SWIGLU, g1, x_perm, cap, H, w_gu[0], 2 * int64_t(I), H,
                               (cap / 128) * g1.n_tiles, st, g_msg, sizeof(g_msg), w_gu),
           "bf16 grouped gate_up GEMM (per-expert weights)");
  GemmArgs g2{};
  g2.mode = 0;
  g2.E = E;
  g2.split_sizes = split_sizes;
  g2.K = I;
  g2.N = H;
  g2.n_tiles = (H + 255) / 256;
  g2.b_rows_per_expert = 0;
  g2.cap = cap;
  g2.out = static_cast<__nv_bfloat16*>(y);
  g2.ldo = H;
  g2.I = I;
  g2.err = g1.err;
  CUDA_TRY(launch_grouped_gemm(EPI_B16_OUT, g2, a_perm, cap, I, w_d[0], H, I, (cap / 128) * g2.n_tiles, st, g_msg,
                               sizeof(g_msg), w_d),
           "bf16 grouped down GEMM (per-expert weights)");
  return MOE_OK;
}

moe_status grouped_mlp_bwd_bf16(const moe_dims* d, const void* dout, const int32_t* split_sizes,
                                const int32_t* row_of, const int32_t* src_of, const float* prob_perm,
                                const void* saved_gu, const void* x_perm, const void* a_perm, const void* w_guT,
                                const void* w_dT, void* dx_perm, void* dwgu, void* dwd, float* dprob, void* workspace,
                                size_t workspace_bytes, moe_stream_t stream) {
  g_msg[0] = 0;
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  REQUIRE_PTR(dout);
  REQUIRE_PTR(split_sizes);
  REQUIRE_PTR(row_of);
  REQUIRE_PTR(src_of);
  REQUIRE_PTR(prob_perm);
  REQUIRE_PTR(saved_gu);
  REQUIRE_PTR(x_perm);
  REQUIRE_PTR(a_perm);
  REQUIRE_PTR(w_guT);
  REQUIRE_PTR(w_dT);
  REQUIRE_PTR(dx_perm);
  REQUIRE_PTR(dwgu);
  REQUIRE_PTR(dwd);
  REQUIRE_PTR(dprob);
  s = check_ws(d, workspace, workspace_bytes, 2);
  if (s != MOE_OK) return s;
  const WsLayout w = ws_layout(d, 2);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t cap = capacity(d);
  const int H = d->H, I = d->I, E = d->E, k = d->k;
  int* err = at<int>(workspace, w.err);
  void* dy = at<uint8_t>(workspace, w.dy16);
  void* dyc = at<uint8_t>(workspace, w.dy16c);
  __nv_bfloat16* dh = at<__nv_bfloat16>(workspace, w.dh16);
  __nv_bfloat16* dhc = at<__nv_bfloat16>(workspace, w.dh16c);
  void* xc = at<uint8_t>(workspace, w.x16c);
  void* ac = at<uint8_t>(workspace, w.a16c);
  float* dp = at<float>(workspace, w.dp);

  // dY rows (gathered dout) and dY, x, a along tokens (transposed) for the weight gradients
  CUDA_TRY(launch_gather_rows(dout, row_of, split_sizes, d->T, k, H, E, cap, dy, err, st), "dout gather rows");
  CUDA_TRY(launch_transpose_bf16(dout, src_of, d->T, 1, int(cap), H, split_sizes, E, dyc, err, st),
           "dout gather transposed");
  CUDA_TRY(launch_transpose_bf16(x_perm, nullptr, cap, 1, int(cap), H, split_sizes, E, xc, err, st), "x transposed");
  CUDA_TRY(launch_transpose_bf16(a_perm, nullptr, cap, 1, int(cap), I, split_sizes, E, ac, err, st), "a transposed");

  // down dgrad + SwiGLU backward: dA = dY * W_d -> dH bf16 (rows and transposed), dp partials
  GemmArgs g3{};
  g3.mode = 0;
  g3.E = E;
  g3.split_sizes = split_sizes;
  g3.K = H;
  g3.N = I;
  g3.n_tiles = (I + 255) / 256;
  g3.b_rows_per_expert = I;
  g3.cap = cap;
  g3.prob_perm = prob_perm;
  g3.out = dh;
  g3.ldo = 2 * int64_t(I);
  g3.out_t = dhc;
  g3.gu = const_cast<__nv_bfloat16*>(static_cast<const __nv_bfloat16*>(saved_gu));
  g3.dp_part = dp;
  g3.I = I;
  g3.err = err;
  CUDA_TRY(launch_grouped_gemm(EPI_B16_BWD_SWIGLU, g3, dy, cap, H, w_dT, int64_t(E) * I, H, (cap / 128) * g3.n_tiles,
                               st, g_msg, sizeof(g_msg)),
           "bf16 down dgrad GEMM");
  CUDA_TRY(launch_dprob_reduce(dp, g3.n_tiles * 4, cap, split_sizes, E, src_of, row_of, k, d->T, dprob, err, st),
           "dprob reduce");

  // down wgrad: dW_d[e] = dY_e^T a_e (K = the expert's tokens)
  GemmArgs g4{};
  g4.mode = 1;
  g4.E = E;
  g4.split_sizes = split_sizes;
  g4.M = H;
  g4.N = I;
  g4.n_tiles = (I + 255) / 256;
  g4.cap = cap;
  g4.out = static_cast<__nv_bfloat16*>(dwd);
  g4.ldo = I;
  g4.I = I;
  g4.err = err;
  CUDA_TRY(launch_grouped_gemm(EPI_B16_OUT, g4, dyc, H, cap, ac, I, cap, int64_t(E) * (H / 128) * g4.n_tiles, st,
                               g_msg, sizeof(g_msg)),
           "bf16 down wgrad GEMM");

  // gate_up dgrad: dX = dH * W_gu (K = 2I)
  GemmArgs g5{};
  g5.mode = 0;
  g5.E = E;
  g5.split_sizes = split_sizes;
  g5.K = 2 * I;
  g5.N = H;
  g5.n_tiles = (H + 255) / 256;
  g5.b_rows_per_expert = H;
  g5.cap = cap;
  g5.out = static_cast<__nv_bfloat16*>(dx_perm);
  g5.ldo = H;
  g5.I = I;
  g5.err = err;
  CUDA_TRY(launch_grouped_gemm(EPI_B16_OUT, g5, dh, cap, 2 * int64_t(I), w_guT, int64_t(E) * H, 2 * int64_t(I),
                               (cap / 128) * g5.n_tiles, st, g_msg, sizeof(g_msg)),
           "bf16 gate_up dgrad GEMM");

  // gate_up wgrad: dW_gu[e] = dH_e^T x_e (K = the expert's tokens)
  GemmArgs g6{};
  g6.mode = 1;
  g6.E = E;
  g6.split_sizes = split_sizes;
  g6.M = 2 * I;
  g6.N = H;
  g6.n_tiles = (H + 255) / 256;
  g6.cap = cap;
  g6.out = static_cast<__nv_bfloat16*>(dwgu);
  g6.ldo = H;
  g6.I = I;
  g6.err = err;
  CUDA_TRY(launch_grouped_gemm(EPI_B16_OUT, g6, dhc, 2 * int64_t(I), cap, xc, H, cap,
                               int64_t(E) * (2 * I / 128) * g6.n_tiles, st, g_msg, sizeof(g_msg)),
           "bf16 gate_up wgrad GEMM");
  return MOE_OK;
}

moe_status grouped_mlp_bwd_fp8_tensor(const moe_dims* d, const void* dout, const int32_t* idx,
                                      const int32_t* split_sizes, const int32_t* row_of, const float* prob_perm,
                                      const void* saved_gu, const uint8_t* xq, const float* amax_x,
                                      const uint8_t* aq, const float* amax_a, const uint8_t* wgu_q,
                                      const float* amax_gu, const uint8_t* wd_q, const float* amax_d, void* dx_perm,
                                      void* dwgu, void* dwd, float* dprob, void* workspace, size_t workspace_bytes,
                                      moe_stream_t stream) {
  g_msg[0] = 0;
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  REQUIRE_PTR(dout);
  REQUIRE_PTR(idx);
  REQUIRE_PTR(split_sizes);
  REQUIRE_PTR(row_of);
  REQUIRE_PTR(prob_perm);
  REQUIRE_PTR(saved_gu);
  REQUIRE_PTR(xq);
  REQUIRE_PTR(aq);
  REQUIRE_PTR(wgu_q);
  REQUIRE_PTR(wd_q);
  REQUIRE_PTR(dx_perm);
  REQUIRE_PTR(dwgu);
  REQUIRE_PTR(dwd);
  REQUIRE_PTR(dprob);
  if (amax_x == nullptr || amax_a == nullptr || amax_gu == nullptr || amax_d == nullptr)
    return fail(MOE_ERR_INVALID_ARG, "an amax array is NULL");
  s = check_ws(d, workspace, workspace_bytes, 3);
  if (s != MOE_OK) return s;
  const WsLayout w = ws_layout(d, 3);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t cap = capacity(d);
  const int H = d->H, I = d->I, E = d->E, k = d->k;
  int* err = at<int>(workspace, w.err);
  uint8_t* dyq = at<uint8_t>(workspace, w.t8dy);
  uint8_t* dyqc = at<uint8_t>(workspace, w.t8dyc);
  __nv_bfloat16* dh16 = at<__nv_bfloat16>(workspace, w.t8dh16);
  uint8_t* dhq = at<uint8_t>(workspace, w.t8dh);
  uint8_t* dhqc = at<uint8_t>(workspace, w.t8dhc);
  uint8_t* xqc = at<uint8_t>(workspace, w.t8xc);
  uint8_t* aqc = at<uint8_t>(workspace, w.t8ac);
  uint8_t* wdT = at<uint8_t>(workspace, w.t8wdT);
  uint8_t* wguT = at<uint8_t>(workspace, w.t8wguT);
  uint32_t* am_dy = at<uint32_t>(workspace, w.t8amax);
  uint32_t* am_dh = am_dy + E;
  float* dp = at<float>(workspace, w.dp);

  // dY: per-expert amax of the routed dout rows, codes in rows and transposed
  CUDA_TRY(cudaMemsetAsync(am_dy, 0, 2 * sizeof(uint32_t) * size_t(E), st), "clear amax of dY, dH");
  CUDA_TRY(launch_t8_amax_tokens(dout, d->T, H, idx, k, E, am_dy, err, st), "per-expert amax of dY");
  CUDA_TRY(launch_t8_quant_tokens(dout, d->T, H, idx, row_of, k, E, cap, am_dy, dyq, err, st),
           "per-tensor quantize of dY rows");
  CUDA_TRY(launch_fill_pad_rows(split_sizes, E, H, cap, dyq, nullptr, err, st), "padding rows of dY");
  CUDA_TRY(launch_transpose_u8(dyq, 1, int(cap), H, split_sizes, E, dyqc, st), "dY codes transposed");
  // the weights' codes transposed (a per-tensor scale does not depend on the axis)
  CUDA_TRY(launch_transpose_u8(wd_q, E, H, I, nullptr, 0, wdT, st), "W_d codes transposed");
  CUDA_TRY(launch_transpose_u8(wgu_q, E, 2 * I, H, nullptr, 0, wguT, st), "W_gu codes transposed");

  // down dgrad + SwiGLU backward: dH in bf16 and its per-expert amax, dp partials
  GemmArgs g3{};
  g3.mode = 0;
  g3.E = E;
  g3.split_sizes = split_sizes;
  g3.K = H;
  g3.N = I;
  g3.n_tiles = (I + 255) / 256;
  g3.b_rows_per_expert = I;
  g3.cap = cap;
  g3.prob_perm = prob_perm;
  g3.out = dh16;
  g3.ldo = 2 * int64_t(I);
  g3.gu = const_cast<__nv_bfloat16*>(static_cast<const __nv_bfloat16*>(saved_gu));
  g3.dp_part = dp;
  g3.I = I;
  g3.amax_a = am_dy;
  g3.amax_b = reinterpret_cast<const uint32_t*>(amax_d);
  g3.amax_out = am_dh;
  g3.err = err;
  CUDA_TRY(launch_grouped_gemm(EPI_T8_BWD_SWIGLU, g3, dyq, cap, H, wdT, int64_t(E) * I, H, (cap / 128) * g3.n_tiles,
                               st, g_msg, sizeof(g_msg)),
           "per-tensor FP8 down dgrad GEMM");
  CUDA_TRY(launch_dprob_reduce(dp, g3.n_tiles * 4, cap, split_sizes, E, nullptr, row_of, k, d->T, dprob, err, st),
           "dprob reduce");
  // dH codes with its expert's scale, rows and transposed; x and a codes transposed
  CUDA_TRY(launch_t8_quant_segments(dh16, split_sizes, E, cap, 2 * I, am_dh, dhq, st), "per-tensor quantize of dH");
  CUDA_TRY(launch_transpose_u8(dhq, 1, int(cap), 2 * I, split_sizes, E, dhqc, st), "dH codes transposed");
  CUDA_TRY(launch_transpose_u8(xq, 1, int(cap), H, split_sizes, E, xqc, st), "x codes transposed");
  CUDA_TRY(launch_transpose_u8(aq, 1, int(cap), I, split_sizes, E, aqc, st), "a codes transposed");

  // down wgrad: dW_d[e] = dY_e^T a_e (K = the expert's tokens)
  GemmArgs g4{};
  g4.mode = 1;
  g4.E = E;
  g4.split_sizes = split_sizes;
  g4.M = H;
  g4.N = I;
  g4.n_tiles = (I + 255) / 256;
  g4.cap = cap;
  g4.out = static_cast<__nv_bfloat16*>(dwd);
  g4.ldo = I;
  g4.I = I;
  g4.amax_a = am_dy;
  g4.amax_b = reinterpret_cast<const uint32_t*>(amax_a);
  g4.err = err;
  CUDA_TRY(launch_grouped_gemm(EPI_T8_OUT, g4, dyqc, H, cap, aqc, I, cap, int64_t(E) * (H / 128) * g4.n_tiles, st,
                               g_msg, sizeof(g_msg)),
           "per-tensor FP8 down wgrad GEMM");

  // gate_up dgrad: dX = dH * W_gu (K = 2I)
  GemmArgs g5{};
  g5.mode = 0;
  g5.E = E;
  g5.split_sizes = split_sizes;
  g5.K = 2 * I;
  g5.N = H;
  g5.n_tiles = (H + 255) / 256;
  g5.b_rows_per_expert = H;
  g5.cap = cap;
  g5.out = static_cast<__nv_bfloat16*>(dx_perm);
  g5.ldo = H;
  g5.I = I;
  g5.amax_a = am_dh;
  g5.amax_b = reinterpret_cast<const uint32_t*>(amax_gu);
  g5.err = err;
  CUDA_TRY(launch_grouped_gemm(EPI_T8_OUT, g5, dhq, cap, 2 * int64_t(I), wguT, int64_t(E) * H, 2 * int64_t(I),
                               (cap / 128) * g5.n_tiles, st, g_msg, sizeof(g_msg)),
           "per-tensor FP8 gate_up dgrad GEMM");

  // gate_up wgrad: dW_gu[e] = dH_e^T x_e (K = the expert's tokens)
  GemmArgs g6{};
  g6.mode = 1;
  g6.E = E;
  g6.split_sizes = split_sizes;
  g6.M = 2 * I;
  g6.N = H;
  g6.n_tiles = (H + 255) / 256;
  g6.cap = cap;
  g6.out = static_cast<__nv_bfloat16*>(dwgu);
  g6.ldo = H;
  g6.I = I;
  g6.amax_a = am_dh;
  g6.amax_b = reinterpret_cast<const uint32_t*>(amax_x);
  g6.err = err;
  CUDA_TRY(launch_grouped_gemm(EPI_T8_OUT, g6, dhqc, 2 * int64_t(I), cap, xqc, H, cap,
                               int64_t(E) * (2 * I / 128) * g6.n_tiles, st, g_msg, sizeof(g_msg)),
           "per-tensor FP8 gate_up wgrad GEMM");
  return MOE_OK;
}

moe_status grouped_mlp_bwd(const moe_dims* d, const void* dout, const int32_t* split_sizes, const int32_t* row_of,
                           const int32_t* src_of, const float* prob_perm, const void* saved_gu, const uint8_t* aq_col,
                           const uint8_t* aq_col_scale, const uint8_t* xq_col, const uint8_t* xq_col_scale,
                           const uint8_t* wguT_q, const uint8_t* wguT_s, const uint8_t* wdT_q, const uint8_t* wdT_s,
                           void* dx_perm, void* dwgu, void* dwd, float* dprob, void* workspace,
                           size_t workspace_bytes, moe_stream_t stream) {
  g_msg[0] = 0;
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  REQUIRE_PTR(dout);
  REQUIRE_PTR(split_sizes);
  REQUIRE_PTR(row_of);
  REQUIRE_PTR(src_of);
  REQUIRE_PTR(prob_perm);
  REQUIRE_PTR(saved_gu);
  REQUIRE_PTR(aq_col);
  REQUIRE_PTR(aq_col_scale);
  REQUIRE_PTR(xq_col);
  REQUIRE_PTR(xq_col_scale);
  REQUIRE_PTR(wguT_q);
  REQUIRE_PTR(wguT_s);
  REQUIRE_PTR(wdT_q);
  REQUIRE_PTR(wdT_s);
  REQUIRE_PTR(dx_perm);
  REQUIRE_PTR(dwgu);
  REQUIRE_PTR(dwd);
  REQUIRE_PTR(dprob);
  s = check_ws(d, workspace, workspace_bytes, true);
  if (s != MOE_OK) return s;
  const WsLayout w = ws_layout(d, true);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t cap = capacity(d);
  const int H = d->H, I = d->I, E = d->E, k = d->k;
  int* err = at<int>(workspace, w.err);
  uint8_t* dyq = at<uint8_t>(workspace, w.dyq);
  uint8_t* dyq_s = at<uint8_t>(workspace, w.dyq_s);
  uint8_t* dyqc = at<uint8_t>(workspace, w.dyqc);
  uint8_t* dyqc_s = at<uint8_t>(workspace, w.dyqc_s);
  uint8_t* dhq = at<uint8_t>(workspace, w.dhq);
  uint8_t* dhq_s = at<uint8_t>(workspace, w.dhq_s);
  uint8_t* dhqc = at<uint8_t>(workspace, w.dhqc);
  uint8_t* dhqc_s = at<uint8_t>(workspace, w.dhqc_s);
  float* dp = at<float>(workspace, w.dp);

  // dY rows: gathered dout quantized along H (dgrad) and along tokens (wgrad)
  CUDA_TRY(launch_quant_rowwise(dout, d->T, H, row_of, k, cap, dyq, dyq_s, err, st, split_sizes, E),
           "dout gather_quant_rowwise + padding rows");
  CUDA_TRY(launch_quant_colwise(dout, src_of, d->T, 1, int(cap), H, split_sizes, E, dyqc, dyqc_s, err, st),
           "dout gather_quant_colwise");

  // down dgrad + fused SwiGLU backward: dA = dY * W_d -> dH (both axes), dp partials
  GemmArgs g3{};
  g3.mode = 0;
  g3.E = E;
  g3.split_sizes = split_sizes;
  g3.K = H;
  g3.N = I;
  g3.n_tiles = (I + 255) / 256;
  g3.b_rows_per_expert = I;
  g3.cap = cap;
  g3.sfa = dyq_s;
  g3.sfb = wdT_s;
  g3.sfa_K = H;
  g3.sfb_K = H;
  g3.prob_perm = prob_perm;
  g3.q_row = dhq;
  g3.q_row_s = dhq_s;
  g3.q_row_K = 2 * int64_t(I);
  g3.q_col = dhqc;
  g3.q_col_s = dhqc_s;
  g3.gu = const_cast<__nv_bfloat16*>(static_cast<const __nv_bfloat16*>(saved_gu));
  g3.dp_part = dp;
  g3.I = I;
  g3.err = err;
  CUDA_TRY(launch_grouped_gemm(EPI_BWD_SWIGLU, g3, dyq, cap, H, wdT_q, int64_t(E) * I, H, (cap / 128) * g3.n_tiles,
                               st, g_msg, sizeof(g_msg)),
           "down dgrad GEMM");
  CUDA_TRY(launch_dprob_reduce(dp, g3.n_tiles * 4, cap, split_sizes, E, src_of, row_of, k, d->T, dprob, err, st),
           "dprob reduce");

  // down wgrad: dW_d[e] = dY_e^T a_e, K = the expert's tokens
  GemmArgs g4{};
  g4.mode = 1;
  g4.E = E;
  g4.split_sizes = split_sizes;
  g4.M = H;
  g4.N = I;
  g4.n_tiles = (I + 255) / 256;
  g4.cap = cap;
  g4.sfa = dyqc_s;
  g4.sfb = aq_col_scale;
  g4.sfa_K = cap;
  g4.sfb_K = cap;
  g4.out = static_cast<__nv_bfloat16*>(dwd);
  g4.ldo = I;
  g4.I = I;
  g4.err = err;
  CUDA_TRY(launch_grouped_gemm(EPI_BF16, g4, dyqc, H, cap, aq_col, I, cap, int64_t(E) * (H / 128) * g4.n_tiles, st,
                               g_msg, sizeof(g_msg)),
           "down wgrad GEMM");

  // gate_up dgrad: dX = dH * W_gu (K = 2I)
  GemmArgs g5{};
  g5.mode = 0;
  g5.E = E;
  g5.split_sizes = split_sizes;
  g5.K = 2 * I;
  g5.N = H;
  g5.n_tiles = (H + 255) / 256;
  g5.b_rows_per_expert = H;
  g5.cap = cap;
  g5.sfa = dhq_s;
  g5.sfb = wguT_s;
  g5.sfa_K = 2 * int64_t(I);
  g5.sfb_K = 2 * int64_t(I);
  g5.out = static_cast<__nv_bfloat16*>(dx_perm);
  g5.ldo = H;
  g5.I = I;
  g5.err = err;
  CUDA_TRY(launch_grouped_gemm(EPI_BF16, g5, dhq, cap, 2 * int64_t(I), wguT_q, int64_t(E) * H, 2 * int64_t(I),
                               (cap / 128) * g5.n_tiles, st, g_msg, sizeof(g_msg)),
           "gate_up dgrad GEMM");

  // gate_up wgrad: dW_gu[e] = dH_e^T x_e, K = the expert's tokens
  GemmArgs g6{};
  g6.mode = 1;
  g6.E = E;
  g6.split_sizes = split_sizes;
  g6.M = 2 * I;
  g6.N = H;
  g6.n_tiles = (H + 255) / 256;
  g6.cap = cap;
  g6.sfa = dhqc_s;
  g6.sfb = xq_col_scale;
  g6.sfa_K = cap;
  g6.sfb_K = cap;
  g6.out = static_cast<__nv_bfloat16*>(dwgu);
  g6.ldo = H;
  g6.I = I;
  g6.err = err;
  CUDA_TRY(launch_grouped_gemm(EPI_BF16, g6, dhqc, 2 * int64_t(I), cap, xq_col, H, cap,
                               int64_t(E) * (2 * I / 128) * g6.n_tiles, st, g_msg, sizeof(g_msg)),
           "gate_up wgrad GEMM");
  return MOE_OK;
}

moe_status moe_unpermute_combine(const moe_dims* d, const void* y_perm, const int32_t* row_of, const float* prob,
                                 void* out, moe_stream_t stream) {
  g_msg[0] = 0;
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  REQUIRE_PTR(y_perm);
  REQUIRE_PTR(row_of);
  REQUIRE_PTR(out);
  if (prob != nullptr && (reinterpret_cast<uintptr_t>(prob) & 3u))
    return fail(MOE_ERR_ALIGNMENT, "prob is not 4-byte aligned");
  CUDA_TRY(launch_combine(y_perm, row_of, prob, d->T, d->k, d->H, capacity(d), out, nullptr,
                          static_cast<cudaStream_t>(stream)),
           "combine");
  return MOE_OK;
}

moe_status moe_router_fwd(const moe_dims* d, const void* x, const void* w_r, float* logits, void* workspace,
                          size_t workspace_bytes, moe_stream_t stream) {
  g_msg[0] = 0;
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  REQUIRE_PTR(x);
  REQUIRE_PTR(w_r);
  REQUIRE_PTR(logits);
  s = check_ws(d, workspace, workspace_bytes, false);
  if (s != MOE_OK) return s;
  const WsLayout w = ws_layout(d, false);
  CUDA_TRY(launch_router_fwd(x, w_r, d->T, d->H, d->E, logits, at<int>(workspace, w.err),
                             static_cast<cudaStream_t>(stream), g_msg, sizeof(g_msg)),
           "router fwd");
  return MOE_OK;
}

moe_status moe_router_bwd(const moe_dims* d, const void* x, const void* w_r, const float* logits, const int32_t* idx,
                          const float* prob, const float* dprob, float* dlogits, void* dx, float* dw_r,
                          void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  g_msg[0] = 0;
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  REQUIRE_PTR(x);
  REQUIRE_PTR(w_r);
  REQUIRE_PTR(logits);
  REQUIRE_PTR(idx);
  REQUIRE_PTR(prob);
  REQUIRE_PTR(dprob);
  REQUIRE_PTR(dlogits);
  REQUIRE_PTR(dx);
  REQUIRE_PTR(dw_r);
  s = check_ws(d, workspace, workspace_bytes, true);
  if (s != MOE_OK) return s;
  const WsLayout w = ws_layout(d, true);
  CUDA_TRY(launch_router_bwd(x, w_r, logits, idx, prob, dprob, d->T, d->H, d->E, d->k, d->renormalize, dlogits, dx,
                             dw_r, at<uint8_t>(workspace, w.rpart), at<int>(workspace, w.err),
                             static_cast<cudaStream_t>(stream)),
           "router bwd");
  return MOE_OK;
}

moe_status moe_selftest_wait_timeout(void* scratch, size_t scratch_bytes, int64_t limit_ns, int32_t* code,
                                     int32_t* site, moe_stream_t stream) {
  g_msg[0] = 0;
  constexpr size_t kNeed = 96 * 1024;
  if (scratch == nullptr || code == nullptr || site == nullptr)
    return fail(MOE_ERR_INVALID_ARG, "scratch, code and site must be non-NULL");
  if ((reinterpret_cast<uintptr_t>(scratch) & 255u) != 0) return fail(MOE_ERR_ALIGNMENT, "scratch must be 256-byte aligned");
  if (scratch_bytes < kNeed) return fail(MOE_ERR_WORKSPACE, "scratch needs %zu bytes", kNeed);
  if (limit_ns < 1000000 || limit_ns > 2000000000) return fail(MOE_ERR_INVALID_ARG, "limit_ns must be in [1 ms, 2 s]");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // layout: [0,256) error word, [256,512) split_sizes, [4 KB, +16 KB) A codes 128x128,
  // [20 KB, +32 KB) B codes 256x128, [52 KB, +512) A scales, [53 KB, +1 KB) B scales
  uint8_t* base = static_cast<uint8_t*>(scratch);
  CUDA_TRY(cudaMemsetAsync(scratch, 0, kNeed, st), "clear scratch");
  static const int32_t one_expert_rows = 128;
  CUDA_TRY(cudaMemcpyAsync(base + 256, &one_expert_rows, sizeof(int32_t), cudaMemcpyHostToDevice, st),
           "split_sizes");
  GemmArgs g{};
  g.mode = 0;
  g.E = 1;
  g.split_sizes = reinterpret_cast<const int*>(base + 256);
  g.K = 128;
  g.N = 256;
  g.n_tiles = 1;
  g.b_rows_per_expert = 256;
  g.cap = 128;
  g.sfa = base + 52 * 1024;
  g.sfb = base + 53 * 1024;
  g.sfa_K = 128;
  g.sfb_K = 128;
  g.out = reinterpret_cast<__nv_bfloat16*>(base + 60 * 1024);   // 128 x 128 bf16 would fit; never written
  g.ldo = 128;
  g.err = reinterpret_cast<int*>(base);
  g.wait_limit_ns = uint64_t(limit_ns);
  g.selftest_no_loads = 1;
  CUDA_TRY(launch_grouped_gemm(EPI_BF16, g, base + 4 * 1024, 128, 128, base + 20 * 1024, 256, 128, 1, st, g_msg,
                               sizeof(g_msg)),
           "self-test GEMM");
  int32_t h[2] = {0, 0};
  CUDA_TRY(cudaMemcpyAsync(h, scratch, sizeof(h), cudaMemcpyDeviceToHost, st), "read error word");
  CUDA_TRY(cudaStreamSynchronize(st), "synchronize");
  *code = h[0];
  *site = h[1];
  return MOE_OK;
}

moe_status moe_workspace_tensor(const moe_dims* d, int32_t training, int32_t which, size_t* offset, size_t* bytes) {
  g_msg[0] = 0;
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  if (offset == nullptr || bytes == nullptr) return fail(MOE_ERR_INVALID_ARG, "offset and bytes must be non-NULL");
  if (training < 0 || training > 3) return fail(MOE_ERR_INVALID_ARG, "training=%d must be in 0..3", training);
  const WsLayout w = ws_layout(d, training);
  const size_t cap = size_t(capacity(d));
  const size_t H = size_t(d->H), I = size_t(d->I);
  size_t off = 0, n = 0;
  switch (which) {
    case MOE_WS_A_CODES: off = w.aq; n = cap * I; break;
    case MOE_WS_A_SCALES: off = w.aq_s; n = cap * I / 32; break;
    case MOE_WS_DY_CODES: off = w.dyq; n = cap * H; break;
    case MOE_WS_DY_SCALES: off = w.dyq_s; n = cap * H / 32; break;
    case MOE_WS_DY_COL_CODES: off = w.dyqc; n = H * cap; break;
    case MOE_WS_DY_COL_SCALES: off = w.dyqc_s; n = H * cap / 32; break;
    case MOE_WS_DH_CODES: off = w.dhq; n = cap * 2 * I; break;
    case MOE_WS_DH_SCALES: off = w.dhq_s; n = cap * 2 * I / 32; break;
    case MOE_WS_DH_COL_CODES: off = w.dhqc; n = 2 * I * cap; break;
    case MOE_WS_DH_COL_SCALES: off = w.dhqc_s; n = 2 * I * cap / 32; break;
    default: return fail(MOE_ERR_INVALID_ARG, "unknown workspace tensor %d", which);
  }
  if (which >= MOE_WS_DY_CODES && training == 0)
    return fail(MOE_ERR_INVALID_ARG, "the backward tensors exist only in a training workspace (training >= 1)");
  *offset = off;
  *bytes = n;
  return MOE_OK;
}

moe_status moe_selftest_epilogue_quant(const float* src, int32_t rows, int32_t cols, uint8_t* codes, uint8_t* scales,
                                       uint8_t* codes_t, uint8_t* scales_t, moe_stream_t stream) {
  g_msg[0] = 0;
  REQUIRE_PTR(src);
  REQUIRE_PTR(codes);
  REQUIRE_PTR(scales);
  REQUIRE_PTR(codes_t);
  REQUIRE_PTR(scales_t);
  if (reinterpret_cast<uintptr_t>(codes) & 31u) return fail(MOE_ERR_ALIGNMENT, "codes must be 32-byte aligned");
  if (rows < 128 || cols < 128 || rows % 128 || cols % 128 || int64_t(rows) * cols > (int64_t(1) << 31))
    return fail(MOE_ERR_UNSUPPORTED, "rows=%d cols=%d: need multiples of 128, rows*cols <= 2^31", rows, cols);
  CUDA_TRY(launch_epilogue_quant_selftest(src, rows, cols, codes, scales, codes_t, scales_t,
                                          static_cast<cudaStream_t>(stream)),
           "epilogue quantizer self-test");
  return MOE_OK;
}

moe_status moe_selftest_mma_issue(int32_t k_steps, void* scratch, size_t scratch_bytes, int32_t* pairs,
                                  moe_stream_t stream) {
  g_msg[0] = 0;
  if (scratch == nullptr || pairs == nullptr) return fail(MOE_ERR_INVALID_ARG, "scratch and pairs must be non-NULL");
  if ((reinterpret_cast<uintptr_t>(scratch) & 255u) != 0) return fail(MOE_ERR_ALIGNMENT, "scratch must be 256-byte aligned");
  if (scratch_bytes < 256) return fail(MOE_ERR_WORKSPACE, "scratch needs 256 bytes");
  if (k_steps < 1 || k_steps > (1 << 24)) return fail(MOE_ERR_INVALID_ARG, "k_steps=%d must be in 1..2^24", k_steps);
  int p = 0;
  CUDA_TRY(launch_mma_rate_selftest(k_steps, static_cast<int*>(scratch), &p, static_cast<cudaStream_t>(stream)),
           "MMA issue self-test");
  *pairs = p;
  return MOE_OK;
}

moe_status moe_get_device_error(const void* workspace, int32_t* code, int32_t* site, moe_stream_t stream) {
  g_msg[0] = 0;
  if (workspace == nullptr || code == nullptr || site == nullptr)
    return fail(MOE_ERR_INVALID_ARG, "workspace, code and site must be non-NULL");
  int32_t h[2] = {0, 0};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CUDA_TRY(cudaMemcpyAsync(h, workspace, sizeof(h), cudaMemcpyDeviceToHost, st), "read error word");
  CUDA_TRY(cudaStreamSynchronize(st), "synchronize");
  *code = h[0];
  *site = h[1];
  return MOE_OK;
}

moe_status moe_clear_device_error(void* workspace, moe_stream_t stream) {
  g_msg[0] = 0;
  if (workspace == nullptr) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
  CUDA_TRY(cudaMemsetAsync(workspace, 0, 8, static_cast<cudaStream_t>(stream)), "clear error word");
  return MOE_OK;
}

}  // extern "C"
