// Global top-W selection for callers that cannot allocate device memory.
//
// gdnbeam_select_topw needs a temporary device buffer from its caller. Some
// callers cannot provide one: a plugin that a host framework calls with only
// its input and output tensors and no workspace, or a process whose device
// memory is entirely reserved by another allocator. For them this file keeps
// a fixed scratch area inside the library itself, a file-scope device array
// that exists on every GPU where the library is loaded, for the life of the
// process. The selection it runs is the same as gdnbeam_select_topw's.
#include <atomic>

#include "common.cuh"
#include "launchers.h"

namespace {

// Largest scratch one call may use; select sizes needing more are refused.
constexpr size_t kStaticSelectBytes = (size_t)16 << 20;  // 16 MiB

static __device__ __align__(256) unsigned char g_select_scratch[kStaticSelectBytes];

// Device address of g_select_scratch on each device, resolved on the first
// call made with that device current. The host-side name of the array is not
// a device address; only this resolved pointer is handed to kernels. Host
// threads making their first call at once may both resolve it; they store
// the same value, and the atomic makes that well defined.
constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices] = {};

int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDNBEAM_ECUDA;
  void* p = g_scratch_addr[dev].load(std::memory_order_relaxed);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_select_scratch) != cudaSuccess || !p) return GDNBEAM_ECUDA;
    g_scratch_addr[dev].store(p, std::memory_order_relaxed);
  }
  *out = p;
  return GDNBEAM_OK;
}

}  // namespace

extern "C" size_t gdnbeam_select_noalloc_max_bytes(void) { return kStaticSelectBytes; }

extern "C" int gdnbeam_select_topw_noalloc(int R, int W_t, int W_next, int V, int dtype,
                                           const void* logits, const float* lse, const float* cum,
                                           const float* bias, int32_t* parents, int32_t* tokens,
                                           float* cum_next, gdnbeam_stream_t stream) {
  if (R < 1 || W_t < 1 || W_next < 1 || V < 2 || !logits || !lse || !parents || !tokens ||
      !cum_next)
    return GDNBEAM_EINVAL;
  if (dtype != GDNBEAM_F32 && dtype != GDNBEAM_BF16) return GDNBEAM_EUNSUPPORTED;
  if ((long long)W_t * V >= (1ll << 31) || (long long)W_next > (long long)W_t * V)
    return GDNBEAM_EINVAL;
  // The whole call must fit the fixed scratch area.
  if (gdnbeam::select_scratch_bytes(R, W_t, W_next, V) > kStaticSelectBytes)
    return GDNBEAM_EWORKSPACE;
  void* scratch = nullptr;
  int st = scratch_address(&scratch);
  if (st) return st;
  return gdnbeam::launch_select(R, W_t, W_next, V, dtype, logits, lse, cum, bias, nullptr,
                                parents, tokens, cum_next, scratch, gdnbeam::error_word(),
                                (cudaStream_t)stream);
}
