// tq_decode_noalloc: tq_decode with its workspace in a fixed device array.
//
// For callers that cannot hand the decode a device buffer: a plain C host
// with no device allocator of its own, or a serving loop that must not call
// cudaMalloc between steps (it can synchronise the device and can fail under
// memory pressure). The workspace lives in a file-scope __device__ array of
// TQ_DECODE_NOALLOC_SCRATCH_BYTES; nothing here, and nothing tq_decode does,
// allocates device or host memory.
//
// The array sits in this translation unit alone, so its module (and its
// device memory) is only loaded by processes that call this entry point.

#include <atomic>
#include <mutex>

#include <cuda_runtime.h>

#include "tq.h"

namespace {

static __device__ __align__(256) unsigned char g_scratch[TQ_DECODE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_ptr[kMaxDevices];
std::mutex g_setup_mutex;

// Address of the current device's copy of g_scratch, looked up once per
// device (the lookup loads this module on that device).
tq_status scratch_for_current_device(void** ptr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return TQ_ERR_UNSUPPORTED;
  void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (p) {
    *ptr = p;
    return TQ_OK;
  }
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
      cudaGetLastError();   // the failed lookup must not poison the caller's next check
      return TQ_ERR_CUDA;
    }
    g_scratch_ptr[dev].store(p, std::memory_order_release);
  }
  *ptr = p;
  return TQ_OK;
}

}  // namespace

extern "C" tq_status tq_decode_noalloc(const tq_config* cfg, const tq_codebook* cb, const void* q, int q_dtype,
                                       const void* cache, long long num_blocks, const int* block_table,
                                       int bt_stride, const int* seq_lens, int batch, int max_seq_len,
                                       float scale, void* out, int out_dtype, unsigned int* dev_status,
                                       tq_stream_t stream) {
  if (!cfg) return TQ_ERR_INVALID_ARG;
  const size_t need = tq_decode_workspace_size(cfg, batch, max_seq_len);
  if (need == 0)   // bad configuration or sizes: let tq_decode name the error (it launches nothing)
    return tq_decode(cfg, cb, q, q_dtype, cache, num_blocks, block_table, bt_stride, seq_lens, batch,
                     max_seq_len, scale, out, out_dtype, nullptr, 0, dev_status, stream);
  if (need > static_cast<size_t>(TQ_DECODE_NOALLOC_SCRATCH_BYTES)) return TQ_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const tq_status st = scratch_for_current_device(&scratch);
  if (st != TQ_OK) return st;
  return tq_decode(cfg, cb, q, q_dtype, cache, num_blocks, block_table, bt_stride, seq_lens, batch, max_seq_len,
                   scale, out, out_dtype, scratch, static_cast<size_t>(TQ_DECODE_NOALLOC_SCRATCH_BYTES),
                   dev_status, stream);
}
