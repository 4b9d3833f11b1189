// moe_route_permute_noalloc: the routing/permutation entry point for callers
// that cannot hand the library any device memory of its own.
//
// Who needs it: code whose device memory is owned and planned by someone else
// and that has no way to pass a workspace through -- for example a plugin
// inside a host framework that exposes only the layer's inputs and outputs, or
// a serving loop whose memory is fixed at start-up and where a cudaMalloc
// (which can synchronise the device) is not acceptable.  Those callers still
// pass every input and output; the two scratch tables of the permutation (one
// 32-bit ballot mask and one 32-bit running count per expert and 32-token
// group) come from a fixed array compiled into this library instead.
//
// The array is file-scope device memory: every GPU that loads the library
// keeps it (kNoallocScratchBytes) until the process exits.  Host code cannot
// use the array's name as a device address, so the first call on each device
// asks the runtime for the address (cudaGetSymbolAddress, with that device
// current) and remembers it; that first call should therefore come before any
// stream capture.  Every call shares the same array: calls whose kernels
// overlap on the GPU (different streams or host threads without ordering)
// race on it.  Nothing here allocates.
#include <atomic>
#include <cstdio>

#include "kernels.cuh"

namespace {

constexpr size_t kNoallocMaxExpertGroups = 262144;  // E * ceil(T/32)
constexpr size_t kNoallocErrBytes = 256;
constexpr size_t kNoallocScratchBytes = kNoallocErrBytes + 2 * 4 * kNoallocMaxExpertGroups;  // 2 MiB + 256 B

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<unsigned char*> g_scratch_addr[kMaxDevices];

moe_status nfail(moe_status s, const char* what) {
  snprintf(moe::last_error_buffer(), moe::kLastErrorBytes, "%s", what);
  return s;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device address of the scratch array on the current device (set up once per device).
moe_status scratch_address(unsigned char** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return nfail(MOE_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return nfail(MOE_ERR_UNSUPPORTED, "device ordinal >= 64");
  unsigned char* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
    if (e != cudaSuccess || addr == nullptr) {
      snprintf(moe::last_error_buffer(), moe::kLastErrorBytes, "cudaGetSymbolAddress of the scratch array failed: %s",
               cudaGetErrorString(e));
      return MOE_ERR_CUDA;
    }
    p = static_cast<unsigned char*>(addr);
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_route_permute_noalloc(const moe_dims* d, const float* logits, const void* x,
                                                int32_t* idx, float* prob, int32_t* split_sizes, int32_t* row_of,
                                                int32_t* src_of, float* prob_perm, uint8_t* xq, uint8_t* xq_scale,
                                                uint8_t* xq_col, uint8_t* xq_col_scale, moe_stream_t stream) {
  moe::last_error_buffer()[0] = 0;
  if (d == nullptr) return nfail(MOE_ERR_INVALID_ARG, "dims is NULL");
  if (d->T < 1 || d->H < 128 || d->H % 128 || d->I < 128 || d->I % 128 || d->E < 1 || d->E > 256 || d->k < 1 ||
      d->k > 8 || d->k > d->E || d->H > 65536)
    return nfail(MOE_ERR_UNSUPPORTED, "sizes outside the supported range (see moe_route_permute)");
  const size_t groups = size_t(d->E) * size_t((d->T + 31) / 32);
  if (groups > kNoallocMaxExpertGroups) {
    snprintf(moe::last_error_buffer(), moe::kLastErrorBytes,
             "E*ceil(T/32) = %zu exceeds the built-in scratch limit of %zu; use moe_route_permute with a workspace",
             groups, kNoallocMaxExpertGroups);
    return MOE_ERR_UNSUPPORTED;
  }
  const void* ptrs[] = {logits, x, idx, prob, split_sizes, row_of, src_of, prob_perm, xq, xq_scale};
  for (const void* p : ptrs) {
    if (p == nullptr) return nfail(MOE_ERR_INVALID_ARG, "a required pointer is NULL");
    if (!al16(p)) return nfail(MOE_ERR_ALIGNMENT, "a pointer is not 16-byte aligned");
  }
  if ((xq_col == nullptr) != (xq_col_scale == nullptr))
    return nfail(MOE_ERR_INVALID_ARG, "xq_col and xq_col_scale must both be set or both be NULL");
  if (xq_col != nullptr && (!al16(xq_col) || !al16(xq_col_scale)))
    return nfail(MOE_ERR_ALIGNMENT, "xq_col or xq_col_scale is not 16-byte aligned");

  unsigned char* base = nullptr;
  moe_status s = scratch_address(&base);
  if (s != MOE_OK) return s;
  int* err = reinterpret_cast<int*>(base);
  uint32_t* masks = reinterpret_cast<uint32_t*>(base + kNoallocErrBytes);
  int* bases = reinterpret_cast<int*>(base + kNoallocErrBytes + 4 * kNoallocMaxExpertGroups);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t cap = ((int64_t(d->T) * d->k + 127) / 128) * 128 + 128 * int64_t(d->E);
  // the masks and bases are fully rewritten by every call; only the error word starts at zero
  cudaError_t e = cudaMemsetAsync(err, 0, 8, st);
  if (e == cudaSuccess)
    e = moe::launch_route_permute(logits, d->T, d->E, d->k, d->renormalize, idx, prob, masks, bases, split_sizes,
                                  row_of, src_of, prob_perm, err, st);
  if (e == cudaSuccess) e = moe::launch_quant_rowwise(x, d->T, d->H, row_of, d->k, cap, xq, xq_scale, err, st);
  if (e == cudaSuccess) e = moe::launch_fill_pad_rows(split_sizes, d->E, d->H, xq, xq_scale, st);
  if (e == cudaSuccess && xq_col != nullptr)
    e = moe::launch_quant_colwise(x, src_of, d->T, 1, int(cap), d->H, split_sizes, d->E, xq_col, xq_col_scale, err,
                                  st);
  if (e != cudaSuccess) {
    snprintf(moe::last_error_buffer(), moe::kLastErrorBytes, "launch failed: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}
