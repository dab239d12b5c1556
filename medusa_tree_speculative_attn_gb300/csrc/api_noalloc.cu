// mt_tree_attn_paged_noalloc: tree attention with the workspace taken from a
// fixed array that the library reserves in device memory, for callers that
// must not allocate on the calling path.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds kNoallocScratchBytes for it until the process exits.  Host
// code cannot use the array's name as a device address, so the first call on
// each device (with that device current) asks the runtime for the address
// with cudaGetSymbolAddress and keeps it; that first call should therefore
// come before any stream capture.  The address is kept for the life of the
// process: a cudaDeviceReset after the first call on a device may move the
// array, so this entry point is not supported across a device reset.  All
// calls on a device share the one array: calls whose kernels overlap on the
// GPU race with each other, so callers serialise them (one stream, or events).
#include <mutex>

#include "../../include/medusa_tree.h"

namespace {

constexpr size_t kNoallocScratchBytes = size_t(64) << 20;  // 64 MiB per device
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device (set up once per device).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MT_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MT_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MT_OK;
}

}  // namespace

extern "C" int mt_tree_attn_paged_noalloc(const mt_attn_desc* desc, const void* q, const void* k_new,
                                          const void* v_new, void* k_cache, void* v_cache,
                                          const int32_t* block_tables, const int32_t* seq_lens,
                                          const int32_t* tree_parents, const int32_t* tree_depths,
                                          const mt_rope* rope, void* out, int32_t* device_status,
                                          cudaStream_t stream) {
  const size_t need = mt_tree_attn_workspace_size(desc);
  if (need == 0)  // an invalid descriptor: the workspace call reports why, launching nothing
    return mt_tree_attn_paged(desc, q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens, tree_parents,
                              tree_depths, rope, out, nullptr, 0, stream);
  if (need > kNoallocScratchBytes) return MT_ERR_UNSUPPORTED;  // workspace exceeds the fixed array
  void* scratch = nullptr;
  int st = scratch_address(&scratch);
  if (st != MT_OK) return st;
  // the status word must start at zero; every other workspace byte is
  // written by the call before it is read
  if (cudaMemsetAsync(scratch, 0, sizeof(int32_t), stream) != cudaSuccess) return MT_ERR_CUDA;
  st = mt_tree_attn_paged(desc, q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens, tree_parents,
                          tree_depths, rope, out, scratch, kNoallocScratchBytes, stream);
  if (st != MT_OK) return st;
  if (device_status &&
      cudaMemcpyAsync(device_status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice, stream) !=
          cudaSuccess)
    return MT_ERR_CUDA;
  return MT_OK;
}
