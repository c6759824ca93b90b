// Device-side helpers shared by the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/pkd.h"

namespace pkd {

// Round two floats to the 16-bit format (nearest-even) and pack them.
template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&b);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// Programmatic dependent launch.  Every kernel is launched so that the next
// kernel in the stream may start while its CTAs drain; each kernel therefore
// waits, before its first global-memory read or write (L2 prefetches, which
// read nothing, may come earlier), until the previous grid has completed and
// its writes are visible, and then lets its own dependents launch.  Without
// the launch attribute both instructions do nothing.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Asks L2 for the cache lines of the byte range [base, base + bytes): the
// lines first, first + step, first + 2 step, ... of the range, at most
// `count` of them, spread over the CTA's threads.  A prefetch reads no value
// into the SM, so it may be issued before pdl_wait(): the lines are then on
// their way while the previous grid drains, and a later load still sees that
// grid's writes, which are made in L2.  Every address lies inside the range.
__device__ __forceinline__ void prefetch_l2_lines(const void* base, size_t bytes, long long first,
                                                  long long step, int count) {
  if (bytes == 0) return;
  const uintptr_t b = reinterpret_cast<uintptr_t>(base);
  const uintptr_t start = b & ~uintptr_t(127);
  const long long lines = (long long)((b + bytes - start + 127) / 128);
  for (int k = threadIdx.x; k < count; k += blockDim.x) {
    const long long l = first + (long long)k * step;
    if (l >= lines) break;
    const uintptr_t p = l == 0 ? b : start + (uintptr_t)l * 128;
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
  }
}

__device__ __forceinline__ void flag(uint32_t* status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

// 16-byte global load that bypasses L1 allocation (streamed data).
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// 16-byte global store with the streaming (evict-first) hint.
__device__ __forceinline__ void st_stream(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// A context length is usable when it fits the grid and the block table.
__device__ __forceinline__ bool len_ok(int L, int max_context_len, int max_blocks_per_seq,
                                       int block_size) {
  return L >= 0 && L <= max_context_len &&
         (long long)L <= (long long)max_blocks_per_seq * block_size;
}

// Row of the split-context workspace holding the partial result of query
// head h of sequence s over context partition p.  Rows are ordered
// [sequence][KV head][partition][head within the group], so the partials of
// one (sequence, KV head, partition) unit form one contiguous block.
__device__ __forceinline__ size_t partial_row(int s, int h, int p, int num_heads, int num_kv_heads,
                                              int num_partitions) {
  const int g = num_heads / num_kv_heads;
  const int hk = h / g;
  return (((size_t)s * num_kv_heads + hk) * num_partitions + p) * g + (h - hk * g);
}

constexpr float kLog2e = 1.4426950408889634f;

// 2^x by the hardware approximation (ex2.approx.ftz: relative error about
// 2^-22, results below 2^-126 flushed to zero, 2^-inf = 0).  Softmax
// weights need no more.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------- packed f32 pairs
// Two floats in one 64-bit register pair, operated on by the paired FP32
// instructions (one issue slot for two lanes' worth of arithmetic).
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
  return make_float2(a, b);
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

}  // namespace pkd
