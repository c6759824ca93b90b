// Decode attention over a paged KV cache on the CUDA cores (query-group
// sizes below 4, head_size 64, and partitions the tensor-core path does not
// take).
//
// One CTA of 4 warps handles one (sequence, KV head, head chunk, context
// partition).  It computes, for the GC query heads of the chunk,
//     out[s,h,:] = softmax_t(scale * q[s,h,:] . K[t,:]) @ V[t,:]
// over the partition's tokens, reading each K/V row of the shared KV head
// once for all GC heads (the group sharing of "Optimize MQA Kernel", vLLM
// pull request 452).  The query chunk is loaded once per CTA and kept in
// registers, so no thread group re-reads it per token (the point of
// "Optimizes the single_query_cached_kv_attention kernel", pull request 420).
//
// Latency: the context length, the partition's block ids (into shared
// memory) and the query are requested together at entry, so only one global
// round trip precedes the first K/V load.  Table entries of the partition past
// the sequence end are read with the others but never used.  K and V reach
// shared memory by TMA: each warp owns a ring of 2 stages, one stage being
// the K and V rows of 8 consecutive tokens of one block (two boxes, 4 KB at
// head_size 128), so a warp keeps up to 8 KB of loads in flight while it
// computes, with two TMA instructions per 8 tokens.  The small ring (32 KB
// per CTA) lets many CTAs share an SM, the next call's among them.  Rows a box brings in
// past the partition end or the sequence end are masked (their V is read as
// zero: cache slots past the end may hold anything, NaN included); boxes of
// out-of-range block ids read an out-of-bounds row, which TMA fills with zeros.
//
// Lane layout: D/8 lanes share one token row, each holding 8 consecutive
// elements (one 16-byte load of K and one of V per token), so a warp row
// covers 32/(D/8) tokens with fully coalesced 256-byte (D=128) rows.  Each
// warp runs its own online softmax over the tokens it loads; the four warps
// are merged through shared memory at the end.
//
// Arithmetic per 8-token box: q . k with mixed-precision FMAs (16-bit
// operands, fp32 accumulation: exact products, no conversions); the per-lane
// partial dots of a lane's rows are summed across the row's lanes by a
// halving butterfly, after which each lane holds one row's logit, so one
// exponential per lane covers the box; the running rescale runs only when
// the maximum moves; p, rounded to the input's 16-bit type (as the
// tensor-core path's P operand is), is broadcast to the lanes of its row and
// accumulated into o with the same mixed-precision FMA.  l sums the unrounded
// fp32 p.
//
// Output: with one partition the CTA writes `out` directly; otherwise it
// writes the unnormalised partial (o, m, l) that lse_reduce.cu merges.
#include <cuda.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace pkd {
namespace {

using namespace sm100;

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kRows = 8;        // tokens per warp iteration = rows of one TMA box
constexpr int kStages = 2;      // ring depth per warp
constexpr int kMaxIds = 1024;   // block ids staged in shared memory per pass

template <int D>
struct Ring {
  static constexpr int box = kRows * D * 2;           // K (or V) rows of one stage
  static constexpr int stage = 2 * box;
  static constexpr int bytes = kWarps * kStages * stage + 128;   // + alignment slack
};

// Dot product of 8 16-bit elements of k and q with fp32 accumulation: each
// product of two 16-bit values is exact in fp32, so the mixed-precision FMA
// gives the same result as converting both operands first.
template <bool BF16>
__device__ __forceinline__ float dot8(const uint4& k, const uint4& q) {
  float d = 0.f;
  const uint32_t kk[4] = {k.x, k.y, k.z, k.w};
  const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (BF16)
      asm("{\n\t.reg .b16 kl, kh, ql, qh;\n\t"
          "mov.b32 {kl, kh}, %1;\n\tmov.b32 {ql, qh}, %2;\n\t"
          "fma.rn.f32.bf16 %0, kl, ql, %0;\n\tfma.rn.f32.bf16 %0, kh, qh, %0;\n\t}"
          : "+f"(d) : "r"(kk[i]), "r"(qq[i]));
    else
      asm("{\n\t.reg .b16 kl, kh, ql, qh;\n\t"
          "mov.b32 {kl, kh}, %1;\n\tmov.b32 {ql, qh}, %2;\n\t"
          "fma.rn.f32.f16 %0, kl, ql, %0;\n\tfma.rn.f32.f16 %0, kh, qh, %0;\n\t}"
          : "+f"(d) : "r"(kk[i]), "r"(qq[i]));
  }
  return d;
}

// acc[i] += p * v[i] for 8 16-bit elements of v, p a 16-bit probability in
// the low half of `p16` (the same rounding of p as the tensor-core path's P
// operand), fp32 accumulation.
template <bool BF16>
__device__ __forceinline__ void axpy8(float (&acc)[8], uint32_t p16, const uint4& v) {
  const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (BF16)
      asm("{\n\t.reg .b16 vl, vh, p, pz;\n\t"
          "mov.b32 {vl, vh}, %2;\n\tmov.b32 {p, pz}, %3;\n\t"
          "fma.rn.f32.bf16 %0, p, vl, %0;\n\tfma.rn.f32.bf16 %1, p, vh, %1;\n\t}"
          : "+f"(acc[2 * i]), "+f"(acc[2 * i + 1]) : "r"(vv[i]), "r"(p16));
    else
      asm("{\n\t.reg .b16 vl, vh, p, pz;\n\t"
          "mov.b32 {vl, vh}, %2;\n\tmov.b32 {p, pz}, %3;\n\t"
          "fma.rn.f32.f16 %0, p, vl, %0;\n\tfma.rn.f32.f16 %1, p, vh, %1;\n\t}"
          : "+f"(acc[2 * i]), "+f"(acc[2 * i + 1]) : "r"(vv[i]), "r"(p16));
  }
}

// Sums over the TPG lanes of a token row of U per-lane partial dot products
// (one per row u of the lane's sub-row), by a halving butterfly: each step
// trades half of the remaining values with the partner lane.  Lane `part`
// ends with the full sum of row u = part / (TPG / U).
template <int TPG, int U>
__device__ __forceinline__ float reduce_rows(const float (&d)[U], int part) {
  if constexpr (U == 4) {
    static_assert(TPG == 16, "U = 4 rows per lane goes with 16 lanes per row");
    const bool b3 = part & 8, b2 = part & 4;
    float w0 = (b3 ? d[2] : d[0]) + __shfl_xor_sync(0xffffffffu, b3 ? d[0] : d[2], 8);
    float w1 = (b3 ? d[3] : d[1]) + __shfl_xor_sync(0xffffffffu, b3 ? d[1] : d[3], 8);
    float w = (b2 ? w1 : w0) + __shfl_xor_sync(0xffffffffu, b2 ? w0 : w1, 4);
    w += __shfl_xor_sync(0xffffffffu, w, 2);
    return w + __shfl_xor_sync(0xffffffffu, w, 1);
  } else {
    static_assert(U == 2 && TPG == 8, "U = 2 rows per lane goes with 8 lanes per row");
    const bool b2 = part & 4;
    float w = (b2 ? d[1] : d[0]) + __shfl_xor_sync(0xffffffffu, b2 ? d[0] : d[1], 4);
    w += __shfl_xor_sync(0xffffffffu, w, 2);
    return w + __shfl_xor_sync(0xffffffffu, w, 1);
  }
}

template <bool BF16, int D, int GC>
__global__ void __launch_bounds__(kThreads)
    decode_simt_kernel(const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap, const DecodeArgs a) {
  constexpr int TPG = D / 8;       // lanes per token row
  constexpr int SUBS = 32 / TPG;   // token rows per warp row
  constexpr int U = kRows / SUBS;  // rows per lane per iteration
  static_assert(U * SUBS == kRows, "one box per warp iteration");
  extern __shared__ __align__(128) uint8_t ring_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ring_raw) + 127) &
                                             ~uintptr_t(127));
  __shared__ uint64_t full[kWarps][kStages];

  __shared__ float red_m[kWarps][GC];
  __shared__ float red_l[kWarps][GC];
  __shared__ __align__(16) float red_o[kWarps][GC][D];
  __shared__ int ids[kMaxIds];

  const int s = blockIdx.z;
  const int g = a.num_heads / a.num_kv_heads;
  const int n_chunks = g / GC;
  const int hk = blockIdx.y / n_chunks;
  const int h0 = hk * g + (blockIdx.y % n_chunks) * GC;
  const int p = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / TPG, part = lane % TPG;
  const bool single = a.num_partitions == 1;
  const int H = a.num_heads;
  const int lb = __ffs(a.block_size) - 1;  // block_size is a power of two
  const int bmask = a.block_size - 1;
  const int t0 = p * a.partition_size;
  const int32_t* bt = a.block_tables + (size_t)s * a.max_blocks_per_seq;

  const int tab_tokens = a.max_blocks_per_seq << lb;
  const int blk_first = t0 >> lb;   // first block of the partition
  const int blk_end = t0 < tab_tokens ? ((min(t0 + a.partition_size, tab_tokens) - 1) >> lb) + 1 : blk_first;
  const uint16_t* qp0 = reinterpret_cast<const uint16_t*>(a.q) + ((size_t)s * H + h0) * D;
  // The entry loads below, requested into L2 while the previous grid drains.
  prefetch_l2_lines(a.context_lens + s, 4, 0, 1, 1);
  prefetch_l2_lines(bt + blk_first, (size_t)min(blk_end - blk_first, kMaxIds) * 4, 0, 1, kThreads);
  prefetch_l2_lines(qp0, (size_t)GC * D * 2, 0, 1, kThreads);
  if (threadIdx.x == 0) {
    for (int w = 0; w < kWarps; ++w)
      for (int i = 0; i < kStages; ++i) mbar_init(&full[w][i], 1);
    fence_barrier_init();
  }
  pdl_wait();
  pdl_launch_dependents();
  // ---- entry: length, block ids of this partition (first pass) and q together
  const int L = a.context_lens[s];
  {
    const int n = min(blk_end - blk_first, kMaxIds);
    for (int i = threadIdx.x; i < n; i += kThreads) ids[i] = __ldg(bt + blk_first + i);
  }

  const float qscale = a.scale * kLog2e;
  uint4 qw[GC];
  {
    const uint16_t* qp = qp0 + part * 8;
#pragma unroll
    for (int j = 0; j < GC; ++j) qw[j] = *reinterpret_cast<const uint4*>(qp + (size_t)j * D);
  }

  const bool lok = len_ok(L, a.max_context_len, a.max_blocks_per_seq, a.block_size);
  if (!lok && p == 0 && blockIdx.y == 0 && threadIdx.x == 0) flag(a.status, PKD_DEV_BAD_LEN);
  if (!lok || t0 >= L) {
    // Nothing to attend to.  Unsplit: write the zero row here.  Split: the
    // reduction reads context_lens itself and writes zeros.
    if (single) {
      uint32_t* o = reinterpret_cast<uint32_t*>(a.out);
      for (int i = threadIdx.x; i < GC * D / 2; i += kThreads)
        o[(((size_t)s * H + h0) * D) / 2 + i] = 0u;
    }
    return;
  }
  const int t1 = min(t0 + a.partition_size, L);

  // ALiBi: logit += slope_j * (t - L + 1), in the same log2 units as q.
  float slope[GC];
#pragma unroll
  for (int j = 0; j < GC; ++j) slope[j] = a.alibi ? a.alibi[h0 + j] * kLog2e : 0.f;

  float m[GC], l[GC], acc[GC][8];
#pragma unroll
  for (int j = 0; j < GC; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[j][i] = 0.f;
  }

  bool bad = false;

  // Blocks [pb0, pb0 + kMaxIds) of the partition have their ids in shared memory.
  int pb0 = blk_first;
  __syncthreads();

  uint8_t* wring = ring + warp * kStages * Ring<D>::stage;
  const int oob_row = a.num_blocks << lb;   // first row past the pool: TMA zero fill
  uint32_t wi_issue = 0, wi_use = 0;        // this warp's ring counters
  bool ok_wait = true;

  // Request the K and V rows of tokens [tb, tb + 8) into the next stage.
  auto issue = [&](int tb) {
    const int st = wi_issue % kStages;
    if (lane == 0) {
      const int id = ids[(tb >> lb) - pb0];
      const bool in_range = id >= 0 && id < a.num_blocks;
      bad |= !in_range;
      const int row = in_range ? (id << lb) + (tb & bmask) : oob_row;
      uint8_t* dst = wring + st * Ring<D>::stage;
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&full[warp][st], Ring<D>::stage);
      tma_load_3d(dst, &kmap, &full[warp][st], 0, hk, row);
      tma_load_3d(dst + Ring<D>::box, &vmap, &full[warp][st], 0, hk, row);
    }
    ++wi_issue;
  };

  // Row of the box whose logit this lane holds after the row reduction (see
  // reduce_rows), and the lane holding row u's logit for this lane's sub-row.
  constexpr int kRowLanes = TPG / U;                 // lanes that end with the same row
  const int u_mine = part / kRowLanes;
  const int r_mine = u_mine * SUBS + sub;

  auto consume = [&](int tb) {
    const int st = wi_use % kStages;
    ok_wait = __all_sync(0xffffffffu, ok_wait && mbar_wait(&full[warp][st], (wi_use / kStages) & 1));
    ++wi_use;
    if (!ok_wait) return;
    const int id = ids[(tb >> lb) - pb0];
    const bool in_range = id >= 0 && id < a.num_blocks;
    // Rows [0, nvalid) of the box are attended (warp-uniform).  Boxes of bad
    // ids were zero-filled by TMA; rows past the sequence end inside a good
    // block may hold anything (NaN included), so their V is zeroed here.
    const int nvalid = in_range ? min(kRows, t1 - tb) : 0;
    uint8_t* src = wring + st * Ring<D>::stage;
    if (in_range && nvalid < kRows) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int r = u * SUBS + sub;
        if (r >= nvalid)
          *reinterpret_cast<uint4*>(src + Ring<D>::box + r * D * 2 + part * 16) = make_uint4(0, 0, 0, 0);
      }
      __syncwarp();
    }
    uint4 kw[U], vw[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int r = u * SUBS + sub;
      kw[u] = *reinterpret_cast<const uint4*>(src + r * D * 2 + part * 16);
      vw[u] = *reinterpret_cast<const uint4*>(src + Ring<D>::box + r * D * 2 + part * 16);
    }
    const bool row_ok = r_mine < nvalid;
    const float pos = (float)(tb + r_mine - (L - 1));   // ALiBi distance to the query
#pragma unroll
    for (int j = 0; j < GC; ++j) {
      float d[U];
#pragma unroll
      for (int u = 0; u < U; ++u) d[u] = dot8<BF16>(kw[u], qw[j]);
      float x = reduce_rows<TPG, U>(d, part);
      x = row_ok ? fmaf(x, qscale, slope[j] * pos) : -INFINITY;
      // Maximum over the 8 rows: they differ in lane bits 2..4.
      float mx = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float m_new = fmaxf(m[j], mx);
      if (m_new == -INFINITY) continue;  // nothing valid seen by this warp yet
      if (m_new != m[j]) {               // warp-uniform: rescale only when the maximum moves
        const float alpha = fast_exp2(m[j] - m_new);
        l[j] *= alpha;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[j][i] *= alpha;
        m[j] = m_new;
      }
      const float pr = fast_exp2(x - m_new);   // 0 for masked rows
      l[j] += pr;
      const uint32_t p16 = pack2<BF16>(pr, 0.f);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t pu = __shfl_sync(0xffffffffu, p16, sub * TPG + u * kRowLanes);
        axpy8<BF16>(acc[j], pu, vw[u]);
      }
    }
  };

  // Passes of up to kMaxIds blocks (one pass unless the partition is huge).
  // Warp w takes the 8-token groups w, w + 4, w + 8, ... of the pass.
  for (;;) {
    const int pass_t0 = max(t0, pb0 << lb);
    const int pass_t1 = min(t1, (pb0 + kMaxIds) << lb);
    const int n_it = pass_t1 > pass_t0 + warp * kRows
                         ? (pass_t1 - pass_t0 - warp * kRows + kWarps * kRows - 1) / (kWarps * kRows)
                         : 0;
    auto tok = [&](int k) { return pass_t0 + (k * kWarps + warp) * kRows; };
    for (int k = 0; k < n_it && k < kStages; ++k) issue(tok(k));
    for (int k = 0; k < n_it && ok_wait; ++k) {
      consume(tok(k));
      __syncwarp();
      if (ok_wait && k + kStages < n_it) issue(tok(k + kStages));
    }
    if (pass_t1 >= t1) break;
    // Stage the next pass's block ids (the barrier also makes a timed-out
    // warp's decision to stop common to the CTA).
    if (__syncthreads_or(!ok_wait)) {
      ok_wait = false;
      break;
    }
    pb0 += kMaxIds;
    const int n = min(blk_end - pb0, kMaxIds);
    for (int i = threadIdx.x; i < n; i += kThreads) ids[i] = __ldg(bt + pb0 + i);
    __syncthreads();
  }
  if (!ok_wait) {
    // A bounded wait gave up: report it, and let this warp's loads land
    // before the CTA can exit.
    if (lane == 0) {
      flag(a.status, PKD_DEV_TIMEOUT);
      for (uint32_t w = wi_use; w < wi_issue; ++w)
        mbar_wait(&full[warp][w % kStages], (w / kStages) & 1, 100000000ull);
    }
    __syncwarp();
  }

  // Merge the token rows of each warp: m is already warp-uniform; each lane's
  // l covers the rows it held a logit for (the rows differ in lane bits 2..4,
  // lanes differing in bits 0..1 hold copies), each lane's acc the rows of
  // its sub-row.
#pragma unroll
  for (int j = 0; j < GC; ++j) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) l[j] += __shfl_xor_sync(0xffffffffu, l[j], off);
#pragma unroll
    for (int off = TPG; off < 32; off <<= 1) {
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[j][i] += __shfl_xor_sync(0xffffffffu, acc[j][i], off);
    }
    if (lane == 0) {
      red_m[warp][j] = m[j];
      red_l[warp][j] = l[j];
    }
    if (sub == 0) {
      float4* dst = reinterpret_cast<float4*>(&red_o[warp][j][part * 8]);
      dst[0] = make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
      dst[1] = make_float4(acc[j][4], acc[j][5], acc[j][6], acc[j][7]);
    }
  }
  const bool any_bad = __syncthreads_or(bad || !ok_wait);
  if (any_bad && threadIdx.x == 0) flag(a.status, PKD_DEV_BAD_BLOCK);

  // Merge the warps and write the result: two output elements per thread.
  for (int idx = threadIdx.x; idx < GC * D / 2; idx += kThreads) {
    const int j = (2 * idx) / D, d = (2 * idx) % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w][j]);
    float n0 = 0.f, n1 = 0.f, den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float c = exp2f(red_m[w][j] - M);
        n0 = fmaf(c, red_o[w][j][d], n0);
        n1 = fmaf(c, red_o[w][j][d + 1], n1);
        den = fmaf(c, red_l[w][j], den);
      }
    }
    const int h = h0 + j;
    if (single) {
      const bool zero = any_bad || den == 0.f;
      const float inv = zero ? 0.f : 1.f / den;
      reinterpret_cast<uint32_t*>(a.out)[(((size_t)s * H + h) * D + d) / 2] =
          pack2<BF16>(n0 * inv, n1 * inv);
    } else {
      const size_t sp = partial_row(s, h, p, H, a.num_kv_heads, a.num_partitions);
      *reinterpret_cast<float2*>(&a.ws_o[sp * D + d]) = make_float2(n0, n1);
      if (d == 0) {
        a.ws_m[sp] = M;
        a.ws_l[sp] = any_bad ? -1.f : den;
      }
    }
  }
}

template <bool BF16, int D, int GC>
cudaError_t launch_g(const DecodeArgs& a, const CUtensorMap& km, const CUtensorMap& vm,
                     cudaStream_t st) {
  static std::atomic<bool> attr_set[64];   // setting it twice from two threads is harmless
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(decode_simt_kernel<BF16, D, GC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Ring<D>::bytes);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true, std::memory_order_release);
  }
  const int g = a.num_heads / a.num_kv_heads;
  dim3 grid(a.num_partitions, a.num_kv_heads * (g / GC), a.num_seqs);
  return launch_pdl(decode_simt_kernel<BF16, D, GC>, grid, dim3(kThreads), Ring<D>::bytes, st,
                    km, vm, a);
}

template <bool BF16, int D>
cudaError_t launch_d(const DecodeArgs& a, cudaStream_t st) {
  CUtensorMap km, vm;
  const long long rows = (long long)a.num_blocks * a.block_size;
  if (!make_kv_map(&km, a.key_cache, BF16, D, a.num_kv_heads, rows, D, kRows, false) ||
      !make_kv_map(&vm, a.value_cache, BF16, D, a.num_kv_heads, rows, D, kRows, false))
    return cudaErrorInvalidValue;
  switch (simt_heads_per_cta(a.num_heads / a.num_kv_heads)) {
    case 4: return launch_g<BF16, D, 4>(a, km, vm, st);
    case 3: return launch_g<BF16, D, 3>(a, km, vm, st);
    case 2: return launch_g<BF16, D, 2>(a, km, vm, st);
    default: return launch_g<BF16, D, 1>(a, km, vm, st);
  }
}

}  // namespace

int simt_heads_per_cta(int group) {
  for (int c : {4, 2, 3, 1})
    if (group % c == 0) return c;
  return 1;
}

cudaError_t launch_decode_simt(const DecodeArgs& a, cudaStream_t st) {
  if (a.head_size == 128) return a.is_bf16 ? launch_d<true, 128>(a, st) : launch_d<false, 128>(a, st);
  return a.is_bf16 ? launch_d<true, 64>(a, st) : launch_d<false, 64>(a, st);
}

}  // namespace pkd
