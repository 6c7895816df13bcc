// Allocation-free variant of ba_select.
//
// Some callers cannot allocate device memory when they run the selection:
// a serving engine that reserves the whole GPU heap for its own pool at
// start-up and forbids cudaMalloc afterwards, or a plugin that runs inside a
// host framework without access to that framework's allocator.  Such callers
// cannot provide the scratch buffer ba_select needs.  ba_select_noalloc uses
// a fixed scratch array compiled into this library instead.
//
// The array is a file-scope __device__ object, so every GPU that loads the
// library holds BA_SELECT_STATIC_SCRATCH_BYTES of it until the process exits.
// Host code cannot use the array's name as a device address; its address is
// looked up once per device with cudaGetSymbolAddress, with that device
// current, on the first call made on that device.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/ba.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_select_scratch[BA_SELECT_STATIC_SCRATCH_BYTES];

std::mutex g_lock;
void *g_scratch_addr[kMaxDevices] = {};

// Address of this device's copy of the scratch array (set up on first use).
int scratch_for_current_device(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return BA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> guard(g_lock);
  if (g_scratch_addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_select_scratch) != cudaSuccess || p == nullptr)
      return BA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return BA_OK;
}

}  // namespace

extern "C" int ba_select_noalloc(const void *q, const void *k, int batch, int heads, int seqlen,
                                 int head_dim, int block, int kappa, float beta, int sort_mode,
                                 int sort_window, int32_t *perm_q, int32_t *perm_k,
                                 int32_t *block_idx, uint32_t *block_mask, float *block_scores,
                                 ba_stream_t stream) {
  const size_t need = ba_select_workspace_size(batch, heads, seqlen, head_dim, block, kappa,
                                               sort_mode, sort_window);
  if (need > static_cast<size_t>(BA_SELECT_STATIC_SCRATCH_BYTES)) return BA_ERR_WORKSPACE;
  // the scratch address is per device: the stream must belong to the
  // current device (else the kernels would be given another GPU's array)
  if (stream != nullptr) {
    int cur = 0, sdev = 0;
    if (cudaGetDevice(&cur) != cudaSuccess ||
        cudaStreamGetDevice(reinterpret_cast<cudaStream_t>(stream), &sdev) != cudaSuccess)
      return BA_ERR_CUDA;
    if (sdev != cur) return BA_ERR_INVALID_ARG;
  }
  void *scratch = nullptr;
  const int st = scratch_for_current_device(&scratch);
  if (st != BA_OK) return st;
  // Nothing in the scratch array has to start at zero: every kernel of the
  // selection writes each scratch element before it reads it.
  return ba_select(q, k, batch, heads, seqlen, head_dim, block, kappa, beta, sort_mode,
                   sort_window, perm_q, perm_k, block_idx, block_mask, block_scores, scratch,
                   static_cast<size_t>(BA_SELECT_STATIC_SCRATCH_BYTES), stream);
}
