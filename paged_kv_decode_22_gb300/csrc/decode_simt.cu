// Decode attention over a paged KV cache on the CUDA cores (query-group
// sizes below 4, and head_size / block_size combinations the tensor-core
// path does not take).
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
// Lane layout: D/8 lanes share one token row, each holding 8 consecutive
// elements (one 16-byte load of K and one of V per token), so a warp row
// covers 32/(D/8) tokens with fully coalesced 256-byte (D=128) rows.  Each
// warp runs its own online softmax over the tokens it loads; the four warps
// are merged through shared memory at the end.  Block ids are fetched one
// iteration ahead so the id load never sits in front of the K/V loads.
//
// Output: with one partition the CTA writes `out` directly; otherwise it
// writes the unnormalised partial (o, m, l) that lse_reduce.cu merges.
#include "common.cuh"
#include "internal.h"

namespace pkd {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kUnroll = 4;

template <bool BF16, int D, int GC>
__global__ void __launch_bounds__(kThreads) decode_simt_kernel(const DecodeArgs a) {
  constexpr int TPG = D / 8;       // lanes per token row
  constexpr int SUBS = 32 / TPG;   // token rows per warp row
  constexpr int WT = SUBS * kUnroll;
  constexpr int CT = kWarps * WT;  // tokens per CTA iteration

  __shared__ float red_m[kWarps][GC];
  __shared__ float red_l[kWarps][GC];
  __shared__ __align__(16) float red_o[kWarps][GC][D];

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

  const int L = a.context_lens[s];
  const bool lok = len_ok(L, a.max_context_len, a.max_blocks_per_seq, a.block_size);
  if (!lok && p == 0 && blockIdx.y == 0 && threadIdx.x == 0) flag(a.status, PKD_DEV_BAD_LEN);
  const int t0 = p * a.partition_size;
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
  const int lb = __ffs(a.block_size) - 1;  // block_size is a power of two
  const int bmask = a.block_size - 1;

  // Query chunk: 8 elements per lane and head, pre-scaled so exp2 can be used.
  const float qscale = a.scale * kLog2e;
  float qr[GC][8];
  {
    const uint16_t* qp =
        reinterpret_cast<const uint16_t*>(a.q) + ((size_t)s * H + h0) * D + part * 8;
#pragma unroll
    for (int j = 0; j < GC; ++j) {
      uint4 w = *reinterpret_cast<const uint4*>(qp + (size_t)j * D);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float2 f = unpack2<BF16>(ww[i]);
        qr[j][2 * i] = f.x * qscale;
        qr[j][2 * i + 1] = f.y * qscale;
      }
    }
  }

  float m[GC], l[GC], acc[GC][8];
#pragma unroll
  for (int j = 0; j < GC; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[j][i] = 0.f;
  }

  const int32_t* bt = a.block_tables + (size_t)s * a.max_blocks_per_seq;
  const size_t slot_stride = (size_t)a.num_kv_heads * D;  // elements per cache slot
  const uint16_t* kbase = reinterpret_cast<const uint16_t*>(a.key_cache) + (size_t)hk * D + part * 8;
  const uint16_t* vbase = reinterpret_cast<const uint16_t*>(a.value_cache) + (size_t)hk * D + part * 8;
  bool bad = false;

  int ids[kUnroll];
  int base = t0 + warp * WT;
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int t = base + u * SUBS + sub;
    ids[u] = t < t1 ? __ldg(bt + (t >> lb)) : 0;
  }

  for (; base < t1; base += CT) {
    // Issue this iteration's K/V loads, then prefetch the next iteration's ids.
    uint4 kr[kUnroll], vr[kUnroll];
    bool ok[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int t = base + u * SUBS + sub;
      const int id = ids[u];
      const bool in_range = id >= 0 && id < a.num_blocks;
      ok[u] = t < t1 && in_range;
      bad |= (t < t1) && !in_range;
      if (ok[u]) {
        const size_t row = ((size_t)id << lb) + (t & bmask);
        kr[u] = ld_stream(kbase + row * slot_stride);
        vr[u] = ld_stream(vbase + row * slot_stride);
      } else {
        kr[u] = make_uint4(0, 0, 0, 0);
        vr[u] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int t = base + CT + u * SUBS + sub;
      ids[u] = t < t1 ? __ldg(bt + (t >> lb)) : 0;
    }

    float kf[kUnroll][8], vf[kUnroll][8];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t kw[4] = {kr[u].x, kr[u].y, kr[u].z, kr[u].w};
      const uint32_t vw[4] = {vr[u].x, vr[u].y, vr[u].z, vr[u].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float2 fk = unpack2<BF16>(kw[i]);
        float2 fv = unpack2<BF16>(vw[i]);
        kf[u][2 * i] = fk.x;
        kf[u][2 * i + 1] = fk.y;
        vf[u][2 * i] = fv.x;
        vf[u][2 * i + 1] = fv.y;
      }
    }

#pragma unroll
    for (int j = 0; j < GC; ++j) {
      float x[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        float d = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) d = fmaf(qr[j][i], kf[u][i], d);
        x[u] = d;
      }
#pragma unroll
      for (int off = TPG / 2; off >= 1; off >>= 1) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) x[u] += __shfl_xor_sync(0xffffffffu, x[u], off);
      }
      float mx = -INFINITY;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (!ok[u]) x[u] = -INFINITY;
        mx = fmaxf(mx, x[u]);
      }
#pragma unroll
      for (int off = TPG; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_new = fmaxf(m[j], mx);
      if (m_new == -INFINITY) continue;  // nothing valid seen by this warp yet
      const float alpha = exp2f(m[j] - m_new);
      m[j] = m_new;
      l[j] *= alpha;
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[j][i] *= alpha;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const float pu = exp2f(x[u] - m_new);  // 0 for masked tokens
        l[j] += pu;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[j][i] = fmaf(pu, vf[u][i], acc[j][i]);
      }
    }
  }

  // Merge the token rows (subs) of each warp: m is already warp-uniform.
#pragma unroll
  for (int j = 0; j < GC; ++j) {
#pragma unroll
    for (int off = TPG; off < 32; off <<= 1) {
      l[j] += __shfl_xor_sync(0xffffffffu, l[j], off);
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
  const bool any_bad = __syncthreads_or(bad);
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
      const size_t sp = ((size_t)s * H + h) * a.num_partitions + p;
      *reinterpret_cast<float2*>(&a.ws_o[sp * D + d]) = make_float2(n0, n1);
      if (d == 0) {
        a.ws_m[sp] = M;
        a.ws_l[sp] = any_bad ? -1.f : den;
      }
    }
  }
}

template <bool BF16, int D>
cudaError_t launch_d(const DecodeArgs& a, cudaStream_t st) {
  const int g = a.num_heads / a.num_kv_heads;
  int gc = 1;
  for (int c : {4, 2, 3, 1}) {
    if (g % c == 0) {
      gc = c;
      break;
    }
  }
  dim3 grid(a.num_partitions, a.num_kv_heads * (g / gc), a.num_seqs);
  switch (gc) {
    case 4: decode_simt_kernel<BF16, D, 4><<<grid, kThreads, 0, st>>>(a); break;
    case 3: decode_simt_kernel<BF16, D, 3><<<grid, kThreads, 0, st>>>(a); break;
    case 2: decode_simt_kernel<BF16, D, 2><<<grid, kThreads, 0, st>>>(a); break;
    default: decode_simt_kernel<BF16, D, 1><<<grid, kThreads, 0, st>>>(a); break;
  }
  return cudaGetLastError();
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
