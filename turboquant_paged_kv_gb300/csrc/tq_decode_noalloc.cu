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

#include <cuda_runtime.h>

#include "tq.h"

namespace {

static __device__ __align__(256) unsigned char g_scratch[TQ_DECODE_NOALLOC_SCRATCH_BYTES];

// Device address of g_scratch in the context current on the calling thread.
// In host code the name g_scratch is only a stand-in for the symbol, never a
// device address. The address is looked up on every call, not cached: it
// belongs to one context and to this module's copy in it, so a cached value
// would dangle after a context reset, or name another caller's memory when a
// different context is current on the same device. Once the module is loaded
// (the first call in a context does that) the look-up is a host-side table
// read that allocates nothing.
tq_status scratch_for_current_context(void** ptr) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
    cudaGetLastError();   // the failed look-up must not poison the caller's next check
    return TQ_ERR_CUDA;
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
  const tq_status st = scratch_for_current_context(&scratch);
  if (st != TQ_OK) return st;
  return tq_decode(cfg, cb, q, q_dtype, cache, num_blocks, block_table, bt_stride, seq_lens, batch, max_seq_len,
                   scale, out, out_dtype, scratch, static_cast<size_t>(TQ_DECODE_NOALLOC_SCRATCH_BYTES),
                   dev_status, stream);
}
