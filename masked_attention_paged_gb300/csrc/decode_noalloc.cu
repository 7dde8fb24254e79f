// decode_noalloc.cu -- paged_decode_attn for callers that cannot allocate
// device memory.
//
// paged_decode_attn needs a caller-supplied workspace for its split-K
// partial results.  Some callers have no way to provide one: a plugin whose
// host framework hands it only input and output pointers and owns every
// other byte of device memory, or a loop whose memory budget is fixed at
// start-up and must not grow or call an allocator (an allocation can also
// synchronise the device, which a latency-bound loop cannot afford).  This
// entry point serves them with scratch memory that is part of the library
// itself: a file-scope device array of kNoAllocScratchBytes, created when the
// library's code is loaded onto a GPU and held by every GPU that loads it
// until the process exits.  The entry point allocates and frees nothing.
//
// The array is shared by every call on a device and keeps what the last call
// left in it.  The partial results are fully rewritten before they are read,
// so only the status word at its head needs clearing, which each call does on
// its stream before launching.  Two calls whose kernels overlap on the GPU
// (different streams, or different host threads without ordering) race on the
// array and produce wrong results; callers must order them.
#include <cuda.h>

#include <mutex>

#include "internal.h"
#include "libattn.h"

namespace {

// 20 MiB: the 64-sequence, 32-head, D 128 decode with up to 8192-token
// contexts (width 513 blocks) needs 9.51 MB including the status block.
constexpr size_t kNoAllocScratchBytes = size_t(20) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

// The array's device address belongs to the context the library's code was
// loaded into: a device reset (or any new primary context) loads it again,
// possibly elsewhere.  So the address is remembered together with the unique
// id of the context it was looked up in, and looked up again when the
// current context's id differs.
struct ScratchAddr {
  unsigned long long ctx_id;
  void* addr;
};

std::mutex g_setup_mu;
ScratchAddr g_scratch[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (0 when it cannot be had).
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
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// With the device current: translate the array's host-side name into its
// device address, once per (device, context).  The host-side symbol is only a
// handle; a kernel must never be given it directly.
attn_status scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  const unsigned long long id = current_context_id();
  std::lock_guard<std::mutex> lock(g_setup_mu);
  ScratchAddr& s = g_scratch[dev];
  if (s.addr == nullptr || id == 0 || s.ctx_id != id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return ATTN_ERR_CUDA;
    s.addr = p;
    // the lookup made the device's primary context current if none was
    s.ctx_id = current_context_id();
  }
  *out = s.addr;
  return ATTN_OK;
}

}  // namespace

extern "C" attn_status paged_decode_attn_noalloc(const attn_tensor* q, const attn_kv_cache* cache,
                                                 const int32_t* block_table, int64_t bt_stride, int32_t max_blocks,
                                                 const int32_t* ctx_lens, float scale, const attn_tensor* out,
                                                 float* lse, uint32_t* device_status, cudaStream_t stream) {
  if (q == nullptr || cache == nullptr || q->ndim != 3 || max_blocks <= 0) return ATTN_ERR_INVALID_ARG;
  if (q->shape[0] < 0 || q->shape[0] > 65535 || q->shape[1] <= 0 || q->shape[1] > 65535)
    return ATTN_ERR_INVALID_ARG;
  const size_t need = paged_decode_workspace_size(static_cast<int32_t>(q->shape[0]),
                                                  static_cast<int32_t>(q->shape[1]), max_blocks, cache->block_size,
                                                  cache->head_dim);
  if (need == 0) return ATTN_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return ATTN_ERR_WORKSPACE;  // larger than the built-in scratch
  // the scratch address is the current device's: the work must go there too
  int dev = -1, stream_dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaStreamGetDevice(stream, &stream_dev) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (stream_dev != dev) return ATTN_ERR_INVALID_ARG;
  void* scratch = nullptr;
  attn_status st = scratch_for_current_device(&scratch);
  if (st != ATTN_OK) return st;
  // the previous call's status must not leak into this one
  if (cudaMemsetAsync(scratch, 0, sizeof(uint32_t), stream) != cudaSuccess) return ATTN_ERR_CUDA;
  st = paged_decode_attn(q, cache, block_table, bt_stride, max_blocks, ctx_lens, scale, out, lse, scratch,
                         kNoAllocScratchBytes, stream);
  if (st != ATTN_OK) return st;
  if (device_status != nullptr &&
      cudaMemcpyAsync(device_status, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}
