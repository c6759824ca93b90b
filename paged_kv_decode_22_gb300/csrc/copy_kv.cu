// Row copies between the paged KV pool and contiguous token-major tensors.
//
//  gather_cached_kv ("Memcpy kernel for flash attention", vLLM pull request
//  29): dst[t] = pool[slot_mapping[t]], for K and V.
//  reshape_and_cache (the cache_ops.cache step named in the notes of pull
//  request 2744): pool[slot_mapping[t]] = src[t], for K and V.
//
// In the [num_blocks][block_size][num_heads][head_size] layout a slot's row
// of num_heads * head_size elements is contiguous, so both directions are
// plain row copies.  One CTA copies one token's K row (blockIdx.y = 0) or V
// row (blockIdx.y = 1) with 16-byte streaming loads and stores, five in
// flight per thread (a 40-head x 128 row of 640 chunks is one round of 128
// threads).
#include "common.cuh"
#include "internal.h"

namespace pkd {
namespace {

constexpr int kThreads = 128;
constexpr int kInflight = 5;

__device__ __forceinline__ void copy_row(char* dst, const char* src, int n16) {
  for (int i0 = threadIdx.x; i0 < n16; i0 += kThreads * kInflight) {
    uint4 r[kInflight];
#pragma unroll
    for (int k = 0; k < kInflight; ++k) {
      const int i = i0 + k * kThreads;
      if (i < n16) r[k] = ld_stream(src + (size_t)i * 16);
    }
#pragma unroll
    for (int k = 0; k < kInflight; ++k) {
      const int i = i0 + k * kThreads;
      if (i < n16) st_stream(dst + (size_t)i * 16, r[k]);
    }
  }
}

__global__ void __launch_bounds__(kThreads) gather_kernel(const CopyArgs a) {
  prefetch_l2_lines(a.slots + blockIdx.x, 8, 0, 1, 1);   // this CTA's slot, while the previous grid drains
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x;
  const bool is_v = blockIdx.y != 0;
  const size_t row_bytes = (size_t)a.row_elems * 2;
  const int n16 = (int)(row_bytes / 16);
  char* dst = static_cast<char*>(is_v ? a.dst_v : a.dst_k) + (size_t)t * row_bytes;
  const long long slot = a.slots[t];
  if (slot < 0 || slot >= (long long)a.num_blocks * a.block_size) {
    for (int i = threadIdx.x; i < n16; i += kThreads)
      st_stream(dst + (size_t)i * 16, make_uint4(0, 0, 0, 0));
    if (!is_v && threadIdx.x == 0) flag(a.status, PKD_DEV_BAD_SLOT);
    return;
  }
  const char* src = static_cast<const char*>(is_v ? a.src_v : a.src_k) + (size_t)slot * row_bytes;
  copy_row(dst, src, n16);
}

__global__ void __launch_bounds__(kThreads) scatter_kernel(const CopyArgs a) {
  prefetch_l2_lines(a.slots + blockIdx.x, 8, 0, 1, 1);   // this CTA's slot, while the previous grid drains
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x;
  const bool is_v = blockIdx.y != 0;
  const size_t row_bytes = (size_t)a.row_elems * 2;
  const int n16 = (int)(row_bytes / 16);
  const long long slot = a.slots[t];
  if (slot < 0) return;  // padding token: not stored
  if (slot >= (long long)a.num_blocks * a.block_size) {
    if (!is_v && threadIdx.x == 0) flag(a.status, PKD_DEV_BAD_SLOT);
    return;
  }
  const char* src = static_cast<const char*>(is_v ? a.src_v : a.src_k) + (size_t)t * row_bytes;
  char* dst = static_cast<char*>(is_v ? a.dst_v : a.dst_k) + (size_t)slot * row_bytes;
  copy_row(dst, src, n16);
}

}  // namespace

cudaError_t launch_gather(const CopyArgs& a, cudaStream_t st) {
  return launch_pdl(gather_kernel, dim3(a.num_tokens, 2), dim3(kThreads), 0, st, a);
}

cudaError_t launch_scatter(const CopyArgs& a, cudaStream_t st) {
  return launch_pdl(scatter_kernel, dim3(a.num_tokens, 2), dim3(kThreads), 0, st, a);
}

}  // namespace pkd
