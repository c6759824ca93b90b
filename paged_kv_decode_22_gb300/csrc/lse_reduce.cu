// Log-sum-exp merge of split-context partial results.
//
// Each context partition of a (sequence, head) left an unnormalised partial
// output o_p, its logit maximum m_p (log2 domain) and its exponent sum l_p.
// The merge is
//     M = max_p m_p,   w_p = 2^(m_p - M),
//     out = (sum_p w_p o_p) / (sum_p w_p l_p),
// equal to the unsplit softmax result.  This is the second step of the
// split-context form behind the "Paged attention V2" column of the
// kernel-latency tables in "[Performance] Support MQA/GQA in decode phase by
// using FlashAttention" (vLLM pull request 2744).
//
// One warp per (sequence, head); each lane owns D/32 consecutive elements.
// The number of partitions of sequence s is recomputed from context_lens, so
// partitions past the end of a short sequence are never read.
#include "common.cuh"
#include "internal.h"

namespace pkd {
namespace {

constexpr int kWarps = 4;

template <bool BF16, int D>
__global__ void __launch_bounds__(kWarps * 32) lse_reduce_kernel(const DecodeArgs a) {
  constexpr int E = D / 32;  // elements per lane (2 or 4)
  pdl_wait();
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.num_heads;
  const long long sh = (long long)blockIdx.x * kWarps + warp;
  if (sh >= (long long)a.num_seqs * H) return;
  const int s = (int)(sh / H);
  const int P = a.num_partitions;

  const int L = a.context_lens[s];
  const bool lok = len_ok(L, a.max_context_len, a.max_blocks_per_seq, a.block_size);
  const int n_p = lok ? (L + a.partition_size - 1) / a.partition_size : 0;
  // Partials of (s, h) sit g rows apart, one per partition.
  const int g = H / a.num_kv_heads;
  const size_t row0 = partial_row(s, (int)(sh - (long long)s * H), 0, H, a.num_kv_heads, P);
  const float* ms = a.ws_m + row0;
  const float* ls = a.ws_l + row0;

  float M = -INFINITY;
  bool bad = false;
  for (int p = lane; p < n_p; p += 32) {
    M = fmaxf(M, ms[(size_t)p * g]);
    bad |= ls[(size_t)p * g] < 0.f;
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  bad = __any_sync(0xffffffffu, bad);

  float acc[E];
#pragma unroll
  for (int i = 0; i < E; ++i) acc[i] = 0.f;
  float den = 0.f;
  if (!bad && M != -INFINITY) {
    const float* os = a.ws_o + row0 * D + lane * E;
    for (int p = 0; p < n_p; ++p) {
      const float w = exp2f(ms[(size_t)p * g] - M);
      den = fmaf(w, ls[(size_t)p * g], den);
      if constexpr (E == 4) {
        const float4 o = *reinterpret_cast<const float4*>(os + (size_t)p * g * D);
        acc[0] = fmaf(w, o.x, acc[0]);
        acc[1] = fmaf(w, o.y, acc[1]);
        acc[2] = fmaf(w, o.z, acc[2]);
        acc[3] = fmaf(w, o.w, acc[3]);
      } else {
        const float2 o = *reinterpret_cast<const float2*>(os + (size_t)p * g * D);
        acc[0] = fmaf(w, o.x, acc[0]);
        acc[1] = fmaf(w, o.y, acc[1]);
      }
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  uint32_t* out = reinterpret_cast<uint32_t*>(a.out) + (sh * D + lane * E) / 2;
#pragma unroll
  for (int i = 0; i < E / 2; ++i) out[i] = pack2<BF16>(acc[2 * i] * inv, acc[2 * i + 1] * inv);
}

// Stream form: the tiles of (sequence s, KV head) sit at positions
// [A, A + n) of the position list (each pair's tiles, then empty positions
// when its last tile is partial), CTA b held [T b / G, T (b + 1) / G).  A pair
// cut by a range edge left partials: CTA b0 (holding position A; the pair
// begins inside its range) in slot 2 b0 + 1, and every later CTA up to b1
// (holding A + n - 1) whose range is not empty in slot 2b.  One column of
// blocks per range edge (kMergeWarps heads per block, a warp per head); the
// column of the pair's first cut (b0 + 1) merges it.
constexpr int kMergeWarps = 8;
constexpr int kMergeChunk = 8;    // partial slots loaded at once

__device__ __forceinline__ int cta_of(long long t, long long T, int G) {   // holder of tile t
  return (int)(((t + 1) * G - 1) / T);
}

template <bool BF16>
__global__ void __launch_bounds__(kMergeWarps * 32) stream_merge_kernel(const DecodeArgs a) {
  constexpr int D = 128, E = 4;   // lane: 4 consecutive elements of d
  pdl_wait();
  pdl_launch_dependents();
  const int4 dsc = a.ws_desc[blockIdx.x];
  const long long A = dsc.x, T = dsc.w;
  const int n = dsc.y;
  if (n == 0) return;                        // no pair cut at this edge
  const int G = a.stream_ctas;
  const int b0 = cta_of(A, T, G);
  if ((int)blockIdx.x != b0 + 1) return;     // merged by the block of its first cut
  const int b1 = cta_of(A + n - 1, T, G);
  const int g = a.num_heads / a.num_kv_heads;
  const long long row0 = (long long)dsc.z * g;   // output row of head 0 of the pair
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int first_slot = 2 * b0 + 1;
  const int j = blockIdx.y * kMergeWarps + warp;
  if (j < g) {
    float acc[E] = {0.f, 0.f, 0.f, 0.f};
    float den = 0.f, M = -INFINITY;
    bool bad = false;
    for (int c0 = b0; c0 <= b1; c0 += kMergeChunk) {
      // Lanes < kMergeChunk: the partial row of CTA c0 + lane (-1: none).
      int r = -1;
      const int b = c0 + lane;
      if (lane < kMergeChunk && b <= b1 &&
          (b == b0 || (T * b) / G < (T * (b + 1)) / G))   // range not empty
        r = (b == b0 ? first_slot : 2 * b) * g + j;
      float m = -INFINITY, l = 0.f;
      if (r >= 0) {
        m = a.ws_m[r];
        l = a.ws_l[r];
      }
      float4 o[kMergeChunk];
#pragma unroll
      for (int k = 0; k < kMergeChunk; ++k) {
        const int rk = __shfl_sync(0xffffffffu, r, k);
        o[k] = rk >= 0 ? *reinterpret_cast<const float4*>(a.ws_o + (size_t)rk * D + lane * E)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      bad |= l < 0.f;
      float cm = m;
#pragma unroll
      for (int off = 4; off >= 1; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
      cm = __shfl_sync(0xffffffffu, cm, 0);
      const float Mn = fmaxf(M, cm);
      const float sc = M == -INFINITY ? 0.f : exp2f(M - Mn);
      const float w = r >= 0 ? exp2f(m - Mn) : 0.f;
      float wl = w * l;
#pragma unroll
      for (int off = 4; off >= 1; off >>= 1) wl += __shfl_xor_sync(0xffffffffu, wl, off);
      den = fmaf(den, sc, __shfl_sync(0xffffffffu, wl, 0));
      acc[0] *= sc; acc[1] *= sc; acc[2] *= sc; acc[3] *= sc;
#pragma unroll
      for (int k = 0; k < kMergeChunk; ++k) {
        const float wk = __shfl_sync(0xffffffffu, w, k);
        acc[0] = fmaf(wk, o[k].x, acc[0]);
        acc[1] = fmaf(wk, o[k].y, acc[1]);
        acc[2] = fmaf(wk, o[k].z, acc[2]);
        acc[3] = fmaf(wk, o[k].w, acc[3]);
      }
      M = Mn;
    }
    bad = __any_sync(0xffffffffu, bad);
    const float inv = den > 0.f ? 1.f / den : 0.f;
    uint32_t* out = reinterpret_cast<uint32_t*>(a.out) + ((row0 + j) * D + lane * E) / 2;
#pragma unroll
    for (int i = 0; i < E / 2; ++i)   // a bad block anywhere zeroes the row
      out[i] = bad ? 0u : pack2<BF16>(acc[2 * i] * inv, acc[2 * i + 1] * inv);
  }
}

template <bool BF16>
cudaError_t launch_sm(const DecodeArgs& a, cudaStream_t st) {
  const int g = a.num_heads / a.num_kv_heads;
  return launch_pdl(stream_merge_kernel<BF16>,
                    dim3(a.stream_ctas, (g + kMergeWarps - 1) / kMergeWarps),
                    dim3(kMergeWarps * 32), 0, st, a);
}

template <bool BF16, int D>
cudaError_t launch_r(const DecodeArgs& a, cudaStream_t st) {
  const long long rows = (long long)a.num_seqs * a.num_heads;
  const unsigned blocks = (unsigned)((rows + kWarps - 1) / kWarps);
  return launch_pdl(lse_reduce_kernel<BF16, D>, dim3(blocks), dim3(kWarps * 32), 0, st, a);
}

}  // namespace

cudaError_t launch_stream_merge(const DecodeArgs& a, cudaStream_t st) {
  if (a.head_size != 128) return cudaErrorInvalidValue;   // the tensor-core path only
  return a.is_bf16 ? launch_sm<true>(a, st) : launch_sm<false>(a, st);
}

cudaError_t launch_lse_reduce(const DecodeArgs& a, cudaStream_t st) {
  if (a.head_size == 128) return a.is_bf16 ? launch_r<true, 128>(a, st) : launch_r<false, 128>(a, st);
  return a.is_bf16 ? launch_r<true, 64>(a, st) : launch_r<false, 64>(a, st);
}

}  // namespace pkd
