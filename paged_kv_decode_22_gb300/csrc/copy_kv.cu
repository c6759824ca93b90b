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
// row (blockIdx.y = 1).
//
// Copies of at most kBulkMaxRows rows of up to 32 KB: a one-warp CTA whose
// first lane moves the row with two bulk copies, global -> shared
// (completing on an mbarrier) and shared -> global.  More rows, or larger
// ones: 16-byte streaming loads and stores, five in flight per thread (a
// 40-head x 128 row of 640 chunks is one round of 128 threads).  Measured on
// 40 x 128 fp16 rows, bulk against 16-byte loads: 19-31 % (gather) and
// 12-22 % (scatter) faster up to 512 rows (T <= 256); at 1024 rows equal
// (gather) and 3 % slower (scatter); at 2048 rows 8-11 % slower; at 4096
// equal.
#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

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

// Copies of at most kBulkMaxRows rows of at most kBulkRowMax bytes go
// through shared memory by bulk copies (a row within the default 48 KB of
// dynamic shared memory).
constexpr uint32_t kBulkRowMax = 32 * 1024;
constexpr long long kBulkMaxRows = 512;

// One row per one-warp CTA, in the direction SCATTER names; slots outside the
// pool are handled as in gather_kernel (zero row, status bit) and
// scatter_kernel (negative: padding, skipped; past the pool: status bit).
template <bool SCATTER>
__global__ void __launch_bounds__(32) copy_bulk_kernel(const CopyArgs a) {
  extern __shared__ __align__(128) uint8_t row_buf[];
  __shared__ uint64_t bar;
  prefetch_l2_lines(a.slots + blockIdx.x, 8, 0, 1, 1);   // this CTA's slot, while the previous grid drains
  if (threadIdx.x == 0) {
    sm100::mbar_init(&bar, 1);
    sm100::fence_barrier_init();
  }
  __syncwarp();
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x;
  const bool is_v = blockIdx.y != 0;
  const uint32_t row_bytes = (uint32_t)a.row_elems * 2;
  const long long slot = a.slots[t];
  if (slot < 0 || slot >= (long long)a.num_blocks * a.block_size) {
    if constexpr (!SCATTER) {
      char* dst = static_cast<char*>(is_v ? a.dst_v : a.dst_k) + (size_t)t * row_bytes;
      for (uint32_t i = threadIdx.x; i < row_bytes / 16; i += 32)
        st_stream(dst + (size_t)i * 16, make_uint4(0, 0, 0, 0));
    }
    if (!is_v && threadIdx.x == 0 && (!SCATTER || slot >= 0)) flag(a.status, PKD_DEV_BAD_SLOT);
    return;
  }
  const size_t src_row = SCATTER ? (size_t)t : (size_t)slot;
  const size_t dst_row = SCATTER ? (size_t)slot : (size_t)t;
  const char* src = static_cast<const char*>(is_v ? a.src_v : a.src_k) + src_row * row_bytes;
  char* dst = static_cast<char*>(is_v ? a.dst_v : a.dst_k) + dst_row * row_bytes;
  if (threadIdx.x == 0) {
    sm100::mbar_arrive_expect_tx(&bar, row_bytes);
    sm100::bulk_load(row_buf, src, row_bytes, &bar);
    if (sm100::mbar_wait(&bar, 0)) {
      sm100::bulk_store(dst, row_buf, row_bytes);
      sm100::bulk_commit();
      sm100::bulk_wait_read_all();   // the buffer is read before the CTA exits
    } else {
      flag(a.status, PKD_DEV_TIMEOUT);
      sm100::mbar_wait(&bar, 0, 100000000ull);   // let the load land before the CTA exits
    }
  }
}

bool bulk_fits(const CopyArgs& a) {
  return (uint32_t)a.row_elems * 2 <= kBulkRowMax && 2LL * a.num_tokens <= kBulkMaxRows;
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
  if (bulk_fits(a))
    return launch_pdl(copy_bulk_kernel<false>, dim3(a.num_tokens, 2), dim3(32),
                      (size_t)a.row_elems * 2, st, a);
  return launch_pdl(gather_kernel, dim3(a.num_tokens, 2), dim3(kThreads), 0, st, a);
}

cudaError_t launch_scatter(const CopyArgs& a, cudaStream_t st) {
  if (bulk_fits(a))
    return launch_pdl(copy_bulk_kernel<true>, dim3(a.num_tokens, 2), dim3(32),
                      (size_t)a.row_elems * 2, st, a);
  return launch_pdl(scatter_kernel, dim3(a.num_tokens, 2), dim3(kThreads), 0, st, a);
}

}  // namespace pkd
