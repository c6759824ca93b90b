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

template <bool BF16, int D>
cudaError_t launch_r(const DecodeArgs& a, cudaStream_t st) {
  const long long rows = (long long)a.num_seqs * a.num_heads;
  const unsigned blocks = (unsigned)((rows + kWarps - 1) / kWarps);
  return launch_pdl(lse_reduce_kernel<BF16, D>, dim3(blocks), dim3(kWarps * 32), 0, st, a);
}

}  // namespace

cudaError_t launch_lse_reduce(const DecodeArgs& a, cudaStream_t st) {
  if (a.head_size == 128) return a.is_bf16 ? launch_r<true, 128>(a, st) : launch_r<false, 128>(a, st);
  return a.is_bf16 ? launch_r<true, 64>(a, st) : launch_r<false, 64>(a, st);
}

}  // namespace pkd
