// noalloc.cu — dllm_block_qkv_rope_write_noalloc: the fused projection call
// for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library scratch memory: code that runs
// while another component owns the device allocator (a plugin host that only
// passes input and output buffers), code with a fixed memory budget reserved
// at start-up that forbids any allocation on the serving path, or code that
// is itself called from a context where cudaMalloc is not allowed.  For them
// this entry point uses a fixed scratch array that lives in the library's own
// device memory instead of the caller's workspace.
//
// The scratch array is a file-scope __device__ variable: every GPU that loads
// the library holds kNoAllocScratchBytes of it until the process exits.  In
// host code its name is only a host-side stand-in, so its device address is
// looked up once per device with cudaGetSymbolAddress (with that device
// current) and cached; that lookup happens on the first call on each device,
// so the first call on a device should come before any stream capture.  The
// cached address belongs to the device's current context: after a
// cudaDeviceReset the library's module is loaded again and the array may move,
// so a process that resets a device must not call this entry point on that
// device again (the cached address would be stale).
//
// All calls share the array and it keeps the last call's contents.  A call
// writes every scale and partial tile before it reads it, and the counters
// at the start of the array (zero when the library is loaded) are set back
// to zero by every call, so nothing needs clearing between calls; but two
// calls whose GPU work overlaps (different streams, no ordering between
// them) race on the array.
#include <mutex>

#include "dllm.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t{8} << 20;  // 8 MiB: counters, row scales, stream-K partial tiles
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once per device).
dllm_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DLLM_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();  // clear the failed lookup's error: later, unrelated calls must not report it
      return DLLM_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return DLLM_OK;
}

}  // namespace

extern "C" dllm_status dllm_block_qkv_rope_write_noalloc(const dllm_layer_desc* desc, const dllm_batch* batch,
                                                         const void* x_block, const void* rms_gain,
                                                         const void* w_packed, const float* rope_table,
                                                         int32_t rope_max_pos, const dllm_cache* cache,
                                                         void* q_block, void* stream) {
  size_t need = 0;
  const dllm_status st = dllm_workspace_size(desc, batch, DLLM_OP_BLOCK_QKV_ROPE_WRITE, &need);
  if (st != DLLM_OK) return st;
  if (need > kNoAllocScratchBytes) return DLLM_ERR_WORKSPACE_TOO_SMALL;  // beyond the fixed scratch
  void* scratch = nullptr;
  const dllm_status ss = scratch_address(&scratch);
  if (ss != DLLM_OK) return ss;
  return dllm_block_qkv_rope_write(desc, batch, x_block, rms_gain, w_packed, rope_table, rope_max_pos, cache, q_block,
                                   scratch, kNoAllocScratchBytes, stream);
}
