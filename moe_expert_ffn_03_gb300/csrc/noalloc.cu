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
// current) and remembers it together with the id of the device's current
// context; a later call under another context (after cudaDeviceReset, which
// unloads the module) looks the address up again.  That look-up happens on a
// call, so the first call on a device (and the first after a reset) should
// come before any stream capture.  Every call shares the same array: calls
// whose kernels overlap on the GPU (different streams or host threads without
// ordering) race on it.  Nothing here allocates.
#include <cuda.h>

#include <cstdio>
#include <mutex>

#include "kernels.cuh"

namespace {

constexpr size_t kNoallocMaxExpertGroups = 262144;  // E * ceil(T/32)
constexpr size_t kNoallocErrBytes = 256;
constexpr size_t kNoallocScratchBytes = kNoallocErrBytes + 2 * 4 * kNoallocMaxExpertGroups;  // 2 MiB + 256 B

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchSlot {
  unsigned long long ctx_id;   // id of the context the address belongs to (0: none yet)
  unsigned char* addr;
};
ScratchSlot g_slots[kMaxDevices];
std::mutex g_slots_mutex;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Id of the calling thread's current context (the runtime's primary context of the
// current device once the runtime has been used on it); 0 if it cannot be read.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

moe_status nfail(moe_status s, const char* what) {
  snprintf(moe::last_error_buffer(), moe::kLastErrorBytes, "%s", what);
  return s;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device address of the scratch array on the current device, looked up once per device
// and context.
moe_status scratch_address(unsigned char** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return nfail(MOE_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return nfail(MOE_ERR_UNSUPPORTED, "device ordinal >= 64");
  // make the runtime's primary context of this device current on this thread (it is the
  // current device already; since CUDA 12 this also initialises the context), so that the
  // context id below is the one the address belongs to
  e = cudaSetDevice(dev);
  if (e != cudaSuccess) return nfail(MOE_ERR_CUDA, cudaGetErrorString(e));
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_slots_mutex);
  ScratchSlot& slot = g_slots[dev];
  if (slot.addr == nullptr || ctx == 0 || slot.ctx_id != ctx) {
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
    if (e != cudaSuccess || addr == nullptr) {
      snprintf(moe::last_error_buffer(), moe::kLastErrorBytes, "cudaGetSymbolAddress of the scratch array failed: %s",
               cudaGetErrorString(e));
      return MOE_ERR_CUDA;
    }
    slot.addr = static_cast<unsigned char*>(addr);
    slot.ctx_id = ctx;
  }
  *out = slot.addr;
  return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_route_permute_noalloc(const moe_dims* d, const float* logits, const void* x,
                                                int32_t* idx, float* prob, int32_t* split_sizes, int32_t* row_of,
                                                int32_t* src_of, float* prob_perm, uint8_t* xq, uint8_t* xq_scale,
                                                uint8_t* xq_col, uint8_t* xq_col_scale, moe_stream_t stream) {
  moe::last_error_buffer()[0] = 0;
  // the checks of moe_route_permute (the message names the field), then the scratch limit
  const moe_status dims_ok = moe::check_layer_dims(d);
  if (dims_ok != MOE_OK) return dims_ok;
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
  const int64_t cap = moe::rows_capacity(d);
  // the masks and bases are fully rewritten by every call; the error word and the routing
  // launch's block ticket start at zero
  cudaError_t e = cudaMemsetAsync(err, 0, 64, st);
  if (e == cudaSuccess)
    e = moe::launch_route_scan(logits, d->T, d->E, d->k, d->renormalize, idx, prob, masks, bases, split_sizes,
                               moe::route_ticket(err), err, st);
  if (e == cudaSuccess) {
    const moe::PermuteRows pr{idx, prob, masks, bases, split_sizes, d->E, (d->T + 31) / 32, row_of, src_of,
                              prob_perm};
    e = moe::launch_permute_quant_rows(x, d->T, d->H, d->k, cap, pr, xq, xq_scale, err, st);
  }
  if (e == cudaSuccess && xq_col != nullptr)
    e = moe::launch_quant_colwise(x, src_of, d->T, 1, int(cap), d->H, split_sizes, d->E, xq_col, xq_col_scale, err,
                                  st);
  if (e != cudaSuccess) {
    snprintf(moe::last_error_buffer(), moe::kLastErrorBytes, "launch failed: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}
