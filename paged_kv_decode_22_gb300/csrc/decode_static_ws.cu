// pkd_paged_decode_attention_static_ws: decode attention for callers that
// cannot allocate device memory.
//
// The ordinary entry point takes the split-context scratch ("workspace") from
// the caller.  Some callers have no way to provide it: code that runs where
// cudaMalloc is forbidden or unsafe (inside a latency-critical serving loop
// that must never hit the allocator, a runtime whose device memory is owned
// and pre-carved by another component, or a plugin that gets only the input
// and output pointers of an operator).  This entry point serves them with a
// scratch array compiled into the library as a file-scope __device__ array of
// PKD_STATIC_WORKSPACE_BYTES bytes.  Every GPU that loads the library holds
// that array until the process exits.
//
// Set-up: the first call on each device (with that device current) looks up
// the array's device address with cudaGetSymbolAddress and caches it; later
// calls on that device reuse it.  Make that first call before any stream
// capture.  Host code never hands the array's name itself to a kernel: in
// host code that name is only a host-side stand-in for the device symbol.
//
// Sharing: all calls on a device use the same array, and it keeps whatever
// the previous call left.  No part of it has to start at zero: every value a
// call reads from it was written earlier in that same call.  Calls whose work
// overlaps on the GPU (for example on two streams at once) race on the array
// and corrupt each other's results; the caller must order them.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/pkd.h"
#include "internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_ws[PKD_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_static_ws_addr[kMaxDevices];

// Device address of g_static_ws on the current device (set up once per
// device).  Called after the plan has checked the device.
pkd_status static_ws_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return pkd::record_cuda_error(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return PKD_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_static_ws_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_ws);
    if (e != cudaSuccess) return pkd::record_cuda_error(e, "cudaGetSymbolAddress(static workspace)");
    if (p == nullptr) return pkd::record_cuda_error(cudaErrorInvalidSymbol, "cudaGetSymbolAddress(static workspace)");
    g_static_ws_addr[dev] = p;
  }
  *out = g_static_ws_addr[dev];
  return PKD_OK;
}

}  // namespace

extern "C" PKD_API pkd_status pkd_paged_decode_attention_static_ws(
    void* out, const void* q, const void* key_cache, const void* value_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int max_context_len, int num_seqs, int num_heads, int num_kv_heads, int head_size,
    int block_size, int num_blocks, float scale, pkd_dtype dtype, int partition_size,
    uint32_t* device_status, void* stream) {
  // Arguments and the device first (the plan checks the device), then the
  // scratch array's address.
  if (!out || !q || !key_cache || !value_cache || !block_tables || !context_lens)
    return PKD_ERR_NULL;
  size_t need = 0;
  pkd_status st = pkd_decode_plan(num_seqs, num_heads, num_kv_heads, head_size, block_size,
                                  max_context_len, partition_size, nullptr, nullptr, nullptr,
                                  &need);
  if (st != PKD_OK) return st;
  if (need > (size_t)PKD_STATIC_WORKSPACE_BYTES) return PKD_ERR_WORKSPACE;
  void* ws = nullptr;
  st = static_ws_address(&ws);
  if (st != PKD_OK) return st;
  return pkd_paged_decode_attention(out, q, key_cache, value_cache, block_tables,
                                    max_blocks_per_seq, context_lens, max_context_len, num_seqs,
                                    num_heads, num_kv_heads, head_size, block_size, num_blocks,
                                    scale, dtype, partition_size, ws,
                                    (size_t)PKD_STATIC_WORKSPACE_BYTES, device_status, stream);
}
