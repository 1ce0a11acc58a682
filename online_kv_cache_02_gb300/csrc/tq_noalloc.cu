// Decode attention for callers that cannot allocate device memory.
//
// Some callers have no way to call cudaMalloc at the point where they run
// decode: code inside a custom allocator or memory pool, a runtime that has
// handed every byte of the device to its own arena, or an embedding that only
// passes pointers it already owns.  For them this file keeps the decode
// workspace (query projections and split-K partials) in one fixed-size array
// that lives in the library image on every device that loads the library, and
// runs the ordinary three-stage decode with it.  The caller still passes the
// inputs, the caches and the output buffer.
//
// The array is not zero-initialised per call and is shared by every call on a
// device: the decode stages write every byte they later read, so nothing has
// to start at zero, but two calls whose work overlaps on the GPU (different
// streams, or different host threads) race on it.

#include "tq_internal.h"

#include <cuda_runtime.h>

#include <mutex>

namespace {

// Fixed workspace: 16 MiB on every device that loads the library, held until exit.
constexpr size_t kScratchBytes = TQ_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 128;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the array on the current device.  In host code the
// array's name only stands for the symbol; the address a kernel may use comes
// from cudaGetSymbolAddress, taken once per device with that device current.
tq_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return TQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();
      return TQ_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return TQ_OK;
}

}  // namespace

extern "C" tq_status tq_decode_attention_noalloc(const tq_ctx* ctx, const void* q, tq_dtype dtype, int batch,
                                                 int num_q_heads, int num_kv_heads, const int32_t* seq_lens,
                                                 int max_seq_len, const int32_t* block_table,
                                                 int max_pages_per_seq, int num_pages, const void* k_cache,
                                                 const void* v_cache, int chunk_tokens, float softmax_scale,
                                                 float* out, void* stream) {
  if (!ctx) return TQ_ERR_INVALID_ARG;
  void* ws = nullptr;
  tq_status st = scratch_address(&ws);
  if (st != TQ_OK) return st;
  // The ordinary decode checks the workspace the sizes need against the
  // array's capacity and returns TQ_ERR_WORKSPACE, launching nothing, when
  // they need more.
  return tq_decode_attention_ex(ctx, q, dtype, batch, num_q_heads, num_kv_heads, seq_lens, max_seq_len,
                                block_table, max_pages_per_seq, num_pages, k_cache, v_cache, chunk_tokens,
                                softmax_scale, out, ws, kScratchBytes, TQ_STAGE_ALL, stream);
}
