// Prefill over a paged KV cache on the 5th-generation tensor cores: a chunk
// of new query tokens per sequence attends causally to the cache up to each
// query's own position.  The review comments of "[Performance] Support
// MQA/GQA in decode phase by using FlashAttention" (vLLM pull request 2744)
// note that the KV-cache attention kernel serves prefill as well, with or
// without a cached prefix; this is that generalisation, shaped for prefill.
//
// Work unit = (sequence, KV head, tile of QT = 128 / g chunk queries): its
// 128 rows are the (query, head) pairs r = query * g + head, so all g heads
// of a query share every K/V tile.  A persistent grid of one CTA per SM walks
// the units, dealt round-robin; inside the CTA:
//   warps 0, 3 K producers (half 0 and the unit's Q tile; half 1): TMA boxes of one block x
//              64 columns into a ring of 32 KB stages, block ids one tile
//              ahead, out-of-range blocks from an out-of-bounds row (zeros).
//   warp 1     V producer, same boxes into its own ring.
//   warp 2     MMA issuer (one thread):
//                S = Q K^T   M = 128 rows, N = 128 tokens, K = head_size,
//                            A = Q (shared memory), B = K tile, into TMEM;
//                O += P V    M = 128 rows, N = head_size, K = 128 tokens,
//                            A = P (TMEM, written by the softmax), B = V tile.
//   warps 4-7  softmax: thread = TMEM lane = one row.  Its 128 logits of a
//              tile are in registers, so the row maximum and sum need no
//              other thread.  p = 2^(x - m_ref) with a reference maximum
//              m_ref that moves only when a logit passes it by more than 8
//              (log2 units); then l and the row of O (in TMEM) are rescaled.
//              P goes back into TMEM as 16-bit pairs over the first 64
//              columns of the tile's S buffer, the A operand of P V.
// TMEM: S double-buffered (2 x 128 columns), O double-buffered by unit
// parity (2 x 128), 512 columns.
#include <cuda.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "schedule.cuh"
#include "sm100.cuh"

namespace pkd {
namespace {

using namespace sm100;

constexpr int TT = 128;                  // tokens per tile (= MMA N of S)
constexpr int HD = 128;                  // head_size of this path
constexpr int ROWS = 128;                // (query, head) rows per unit (= MMA M)
constexpr int TILE_BYTES = TT * HD * 2;  // one K or V tile, 32 KB
constexpr int Q_BYTES = ROWS * HD * 2;   // one Q tile, 32 KB
constexpr int NK = 2, NV = 2;            // ring stages
constexpr int kPfTable = 128;            // sequences whose lengths and chunk bounds sit in shared memory
constexpr int kThreads = 256;            // 8 warps
constexpr int kSoftmaxThreads = 128;
constexpr int kNoBlock = -2147483647 - 1;
constexpr float kHeadroom = 8.f;         // log2 units: p < 2^8 between rescales

constexpr int off_q = 0;
constexpr int off_k = off_q + 2 * Q_BYTES;
constexpr int off_v = off_k + NK * TILE_BYTES;
constexpr int off_misc = off_v + NV * TILE_BYTES;

struct Misc {
  uint64_t k_full[NK], k_empty[NK], v_full[NV], v_empty[NV];
  uint64_t q_full[2], q_empty[2], s_full[2], p_full[2], pv_done[2], o_full[2], o_empty[2], drain;
  uint32_t tmem_base;
  int abort;
  int k_bad[NK];      // per K stage: token offset of the tile's first bad block id, or -1
  int tab_L[kPfTable];        // context_lens, with at most kPfTable sequences
  int tab_qs[kPfTable + 1];   // query_start, likewise
};
constexpr int kMiscBytes = 1280;
static_assert(sizeof(Misc) <= kMiscBytes, "misc area too small");
constexpr int kSmemBytes = off_misc + kMiscBytes + 1024;   // + alignment slack
static_assert(kSmemBytes <= 232448, "above the shared memory of one CTA");

__device__ __forceinline__ void set_abort(Misc& ms, uint32_t* status) {
  ms.abort = 1;
  flag(status, PKD_DEV_TIMEOUT);
}

// ---------------------------------------------------------------- schedule
// A sequence's units are its query tiles of q_per_unit queries; a chunk
// longer than the context or than max_query_len (or an invalid length) has
// none.  q0, q1 = query_start[s], query_start[s + 1].
__device__ __forceinline__ bool chunk_rows_ok(const DecodeArgs& a, int q0, int q1) {
  return 0 <= q0 && q0 <= q1 && q1 <= a.num_q_tokens;   // rows inside q / out
}

__device__ __forceinline__ int prefill_parts(const DecodeArgs& a, int q0, int q1, int L) {
  const int n = q1 - q0;
  return (chunk_rows_ok(a, q0, q1) && len_ok(L, a.max_context_len, a.max_blocks_per_seq, a.block_size) &&
          n > 0 && n <= L && n <= a.max_query_len)
             ? (n + a.q_per_unit - 1) / a.q_per_unit
             : 0;
}

// Unit (sequence s, KV head hk, query tile p): its queries and the cache
// range up to the last one's position; ntiles = 0 when the chunk has no
// such tile.  Lengths and chunk bounds come from the shared-memory table
// when it holds them.
__device__ __forceinline__ UnitInfo unit_at(const Misc& ms, const DecodeArgs& a, int s, int hk,
                                            int p) {
  UnitInfo ui;
  ui.s = s;
  ui.hk = hk;
  ui.p = p;
  ui.slot = -1;
  const bool tab = a.num_seqs <= kPfTable;
  ui.L = tab ? ms.tab_L[s] : a.context_lens[s];
  ui.lok = len_ok(ui.L, a.max_context_len, a.max_blocks_per_seq, a.block_size);
  const int q0 = tab ? ms.tab_qs[s] : a.query_start[s];
  const int q1 = tab ? ms.tab_qs[s + 1] : a.query_start[s + 1];
  if (p < prefill_parts(a, q0, q1, ui.L)) {
    const int n = q1 - q0, i0 = p * a.q_per_unit;
    ui.nq = min(a.q_per_unit, n - i0);
    ui.qrow0 = q0 + i0;
    ui.pos0 = ui.L - n + i0;
    ui.t0 = 0;
    ui.t1 = ui.pos0 + ui.nq;
    ui.ntiles = (ui.t1 + TT - 1) / TT;
  } else {
    ui.ntiles = 0;
  }
  return ui;
}

// The table, and zero rows (with the length status bit) for chunks that
// cannot be attended: an invalid length, or longer than the context.  Every
// thread calls this; it ends with __syncthreads().
__device__ __forceinline__ void prefill_setup(Misc& ms, const DecodeArgs& a) {
  if (a.num_seqs <= kPfTable)
    for (int i = threadIdx.x; i <= a.num_seqs; i += kThreads) {
      if (i < a.num_seqs) ms.tab_L[i] = a.context_lens[i];
      ms.tab_qs[i] = a.query_start[i];
    }
  for (int sq = blockIdx.x; sq < a.num_seqs; sq += gridDim.x) {
    const int L = a.context_lens[sq];
    const int q0 = a.query_start[sq], q1 = a.query_start[sq + 1], n = q1 - q0;
    if (!chunk_rows_ok(a, q0, q1)) {     // rows outside q / out: nothing can be written
      if (threadIdx.x == 0) flag(a.status, PKD_DEV_BAD_LEN);
    } else if (n > 0 && prefill_parts(a, q0, q1, L) == 0) {
      if (threadIdx.x == 0) flag(a.status, PKD_DEV_BAD_LEN);
      uint32_t* o = reinterpret_cast<uint32_t*>(a.out) + (size_t)q0 * a.num_heads * a.head_size / 2;
      const size_t words = (size_t)n * a.num_heads * a.head_size / 2;
      for (size_t i = threadIdx.x; i < words; i += kThreads) o[i] = 0u;
    }
  }
  __syncthreads();
}

// Units of one CTA: unit u of S * Hk * P, dealt round-robin (consecutive
// query tiles of a causal chunk differ in cost; dealing spreads them), later
// (heavier) tiles first.
struct PfCursor {
  long long next, end;
  int stride;
  __device__ __forceinline__ void begin(const DecodeArgs& a) {
    next = blockIdx.x;
    stride = gridDim.x;
    end = (long long)a.num_seqs * a.num_kv_heads * a.num_partitions;
  }
  __device__ __forceinline__ bool step(const Misc& ms, const DecodeArgs& a, UnitInfo& ui) {
    const int per = a.num_partitions;
    while (next < end) {
      const int v = (int)next;
      next += stride;
      const int pp = per - 1 - v % per, sh = v / per;
      const int hk = sh % a.num_kv_heads, s = sh / a.num_kv_heads;
      ui = unit_at(ms, a, s, hk, pp);
      if (ui.ntiles) return true;
    }
    return false;
  }
};

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap,
                      const __grid_constant__ CUtensorMap qmap, const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  uint8_t* qbuf = sm + off_q;
  uint8_t* kbuf = sm + off_k;
  uint8_t* vbuf = sm + off_v;
  Misc& ms = *reinterpret_cast<Misc*>(sm + off_misc);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = a.num_heads / a.num_kv_heads;
  // A K stage is free once the MMA is done with it and the softmax has read
  // the stage's bad-block entry (without that arrival a stage could be
  // refilled before the softmax checks it).
  constexpr uint32_t kMmaCount = 1;

  // ---------------------------------------------------------------- setup
  prefetch_schedule_inputs(a);
  if (threadIdx.x == 0) {
    for (int i = 0; i < NK; ++i) {
      mbar_init(&ms.k_full[i], 1);
      mbar_init(&ms.k_empty[i], kMmaCount + kSoftmaxThreads);
      ms.k_bad[i] = -1;
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(&ms.v_full[i], 1);
      mbar_init(&ms.v_empty[i], kMmaCount);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ms.q_full[i], 1);
      mbar_init(&ms.q_empty[i], 1);
      mbar_init(&ms.s_full[i], 1);
      mbar_init(&ms.p_full[i], kSoftmaxThreads);
      mbar_init(&ms.pv_done[i], 1);
      mbar_init(&ms.o_full[i], 1);
      mbar_init(&ms.o_empty[i], kSoftmaxThreads);
    }
    mbar_init(&ms.drain, 1);
    ms.abort = 0;
    fence_barrier_init();
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    tma_prefetch_desc(&qmap);
  }
  if (warp == 2) {
    tmem_alloc(&ms.tmem_base, 512);
    tmem_relinquish();
  }
  pdl_wait();
  pdl_launch_dependents();
  prefill_setup(ms, a);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;

  if (warp == 0 || warp == 1 || warp == 3) {
    // ============================================================ producers
    // Warp 0 issues K's first 64-column half (and owns the stage's barrier
    // bookkeeping and the Q loads), warp 3 K's second half in parallel, warp
    // 1 both halves of V.
    const bool is_v = warp == 1;
    const bool primary = warp != 3;
    const int half_mask = warp == 0 ? 1 : warp == 3 ? 2 : 3;   // 64-column halves issued
    const int B = a.block_size;
    const int R = B < TT ? B : TT;            // rows per TMA box
    const int nbox = TT / R;                  // boxes per tile and 64-column half
    const int oob_row = a.num_blocks * B;     // first row past the pool: zero fill
    const CUtensorMap* map = is_v ? &vmap : &kmap;
    uint8_t* ring = is_v ? vbuf : kbuf;
    const int nst = is_v ? NV : NK;
    uint64_t* full = is_v ? ms.v_full : ms.k_full;
    uint64_t* empty = is_v ? ms.v_empty : ms.k_empty;
    const bool issuer = lane < 2 * nbox && ((half_mask >> (lane / nbox)) & 1);
    const int my_box = lane % nbox, my_half = lane / nbox;
    auto load_raw = [&](const UnitInfo& t, int tj) {
      int raw = kNoBlock;
      if (lane < nbox) {
        const int ts = tj * TT;
        const int tok0 = B <= TT ? ts + lane * B : ts;
        if (tok0 < t.t1) raw = __ldg(a.block_tables + (size_t)t.s * a.max_blocks_per_seq + tok0 / B);
      }
      return raw;
    };
    PfCursor cur;
    cur.begin(a);
    UnitInfo ui;
    bool have = cur.step(ms, a, ui);
    int jl = 0;
    int raw = have ? load_raw(ui, 0) : kNoBlock;
    uint32_t jk = 0, un = 0;
    bool ok = true;
    while (have) {
      UnitInfo nui = ui;
      bool nhave = true;
      int njl = jl + 1;
      if (njl >= ui.ntiles) {
        nhave = cur.step(ms, a, nui);
        njl = 0;
      }
      const int nraw = nhave ? load_raw(nui, njl) : kNoBlock;
      if (!is_v && primary && jl == 0 && lane == 0) {
        const int qb = un & 1;
        ok = mbar_wait(&ms.q_empty[qb], ((un >> 1) & 1) ^ 1);
        if (ok) {
          // Rows (query, head) of the unit: box {64, g, QT} over q [T][H][D].
          mbar_arrive_expect_tx(&ms.q_full[qb], (uint32_t)(g * a.q_per_unit * 256));
          tma_load_3d(qbuf + qb * Q_BYTES, &qmap, &ms.q_full[qb], 0, ui.hk * g, ui.qrow0);
          tma_load_3d(qbuf + qb * Q_BYTES + ROWS * 128, &qmap, &ms.q_full[qb], 64, ui.hk * g,
                      ui.qrow0);
        }
      }
      const int ts = jl * TT;
      const bool bad = raw != kNoBlock && (raw < 0 || raw >= a.num_blocks);
      const int row = (raw != kNoBlock && !bad) ? raw * B + (B <= TT ? 0 : ts % B) : oob_row;
      const uint32_t bad_lanes = __ballot_sync(0xffffffffu, bad);   // lanes < nbox: boxes in token order
      const int st = jk % nst;
      if (lane == 0) {
        ok = ok && mbar_wait(&empty[st], ((jk / nst) & 1) ^ 1);
        if (ok && primary) {
          if (!is_v) {
            ms.k_bad[st] = bad_lanes ? (__ffs(bad_lanes) - 1) * R : -1;
            if (bad_lanes) flag(a.status, PKD_DEV_BAD_BLOCK);
          }
          mbar_arrive_expect_tx(&full[st], TILE_BYTES);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const int r = __shfl_sync(0xffffffffu, row, my_box);
      if (issuer) {
        uint8_t* dst = ring + st * TILE_BYTES + my_half * TT * 128 + my_box * R * 128;
        tma_load_3d(dst, map, &full[st], my_half * 64, ui.hk, r);
      }
      ++jk;
      if (njl == 0) ++un;
      have = nhave;
      ui = nui;
      jl = njl;
      raw = nraw;
    }
    if (!ok && lane == 0) {
      set_abort(ms, a.status);
      for (uint32_t j = (jk >= (uint32_t)nst ? jk - nst : 0); j < jk; ++j)
        mbar_wait(&full[j % nst], (j / nst) & 1, 100000000ull);
    }
  } else if (warp == 2) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_f16(ROWS, TT, BF16, false, false);
      const uint32_t id_o = idesc_f16(ROWS, HD, BF16, false, true);
      const uint32_t qaddr = smem_u32(qbuf), kaddr = smem_u32(kbuf), vaddr = smem_u32(vbuf);
      uint32_t j = 0, un = 0;
      bool ok = true;
      // The pending P V: its tile, unit, and whether it opens / closes the unit.
      int pv_j = -1;
      uint32_t pv_u = 0;
      bool pv_first = false, pv_last = false;
      auto issue_pv = [&]() {
        const uint32_t jp = (uint32_t)pv_j;
        const int vs = jp % NV, b = jp & 1, ub = pv_u & 1;
        ok = ok && mbar_wait(&ms.v_full[vs], (jp / NV) & 1);
        ok = ok && mbar_wait(&ms.p_full[b], (jp >> 1) & 1);
        // The unit's O buffer was last read by the finalisation of unit pv_u - 2.
        if (pv_first) ok = ok && mbar_wait(&ms.o_empty[ub], ((pv_u >> 1) & 1) ^ 1);
        if (!ok) return;
        tc_fence_after();
        const uint32_t d = tmem + 256 + ub * 128;
#pragma unroll
        for (int k = 0; k < TT / 16; ++k) {
          const uint64_t bd = smem_desc(vaddr + vs * TILE_BYTES + k * 2048, TT * 128, 1024,
                                        kSwizzle128B);
          mma_f16_ts(d, tmem + b * 128 + k * 8, bd, id_o, !(pv_first && k == 0));
        }
        mma_commit(&ms.v_empty[vs]);
        mma_commit(&ms.pv_done[b]);
        if (pv_last) mma_commit(&ms.o_full[ub]);
      };
      PfCursor cur;
      cur.begin(a);
      UnitInfo ui;
      while (ok && cur.step(ms, a, ui)) {
        const int qb = un & 1;
        ok = ok && mbar_wait(&ms.q_full[qb], (un >> 1) & 1);
        for (int jl = 0; jl < ui.ntiles && ok; ++jl, ++j) {
          const int ks = j % NK, b = j & 1;
          ok = mbar_wait(&ms.k_full[ks], (j / NK) & 1);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d = tmem + b * 128;
#pragma unroll
          for (int k = 0; k < HD / 16; ++k) {
            const uint64_t ad = smem_desc(qaddr + qb * Q_BYTES + (k >> 2) * ROWS * 128 + (k & 3) * 32,
                                          16, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(kaddr + ks * TILE_BYTES + (k >> 2) * TT * 128 + (k & 3) * 32,
                                          16, 1024, kSwizzle128B);
            mma_f16(d, ad, bd, id_s, k > 0);
          }
          mma_commit(&ms.s_full[b]);
          mma_commit(&ms.k_empty[ks]);
          if (jl == ui.ntiles - 1) mma_commit(&ms.q_empty[qb]);
          if (pv_j >= 0) issue_pv();
          pv_j = (int)j;
          pv_u = un;
          pv_first = jl == 0;
          pv_last = jl == ui.ntiles - 1;
        }
        ++un;
      }
      if (ok && pv_j >= 0) issue_pv();
      if (!ok) set_abort(ms, a.status);
      mma_commit(&ms.drain);
      mbar_wait(&ms.drain, 0, 100000000ull);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ============================================================ softmax / epilogue
    const int wq = warp & 3;                   // TMEM lane quadrant
    const int row = wq * 32 + lane;            // this thread's row of S, P and O
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    const float qscale = a.scale * kLog2e;
    const int H = a.num_heads;
    const int qi = row / g, hj = row - qi * g; // row = (chunk query qi, head hj of the group)
    const bool alibi = a.alibi != nullptr;
    uint32_t j = 0, u = 0, u_fin = 0;   // u_fin: units whose output is written
    bool ok = true;
    // A unit's output is written after the next unit's first P, so its last
    // P V runs while that tile's softmax does: the pending write's state.
    bool pend = false, pend_valid = false;
    int pend_ub = 0;
    float pend_inv = 0.f;
    uint4* pend_dst = nullptr;
    auto finalize = [&]() {
      ok = ok && mbar_wait(&ms.o_full[pend_ub], (u_fin >> 1) & 1);
      if (!ok) return;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        float v[32];
        tmem_ld32(lane_addr + 256 + pend_ub * 128 + c * 32, v);
        if (pend_valid) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            pend_dst[c * 4 + i] = make_uint4(pack2<BF16>(v[8 * i] * pend_inv, v[8 * i + 1] * pend_inv),
                                             pack2<BF16>(v[8 * i + 2] * pend_inv, v[8 * i + 3] * pend_inv),
                                             pack2<BF16>(v[8 * i + 4] * pend_inv, v[8 * i + 5] * pend_inv),
                                             pack2<BF16>(v[8 * i + 6] * pend_inv, v[8 * i + 7] * pend_inv));
        }
      }
      tc_fence_before();
      mbar_arrive(&ms.o_empty[pend_ub]);
      pend = false;
      ++u_fin;
    };
    PfCursor cur;
    cur.begin(a);
    UnitInfo ui;
    while (ok && cur.step(ms, a, ui)) {
      const int ub = u & 1;
      const bool valid_row = qi < ui.nq;
      const int pos = valid_row ? ui.pos0 + qi : -1;      // last visible token
      const float slope = alibi && valid_row ? a.alibi[ui.hk * g + hj] * kLog2e : 0.f;
      float m_ref = valid_row ? -INFINITY : INFINITY;       // +inf: p = 0, never rescales
      float l = 0.f;
      int bad_from = 0x7fffffff;
      for (int jl = 0; jl < ui.ntiles; ++jl, ++j) {
        const int b = j & 1, ks = j % NK;
        const int ts = jl * TT;
        ok = ok && mbar_wait(&ms.s_full[b], (j >> 1) & 1);
        ok = ok && mbar_wait(&ms.k_full[ks], (j / NK) & 1);
        if (!ok) break;
        tc_fence_after();
        {
          const int kb = ms.k_bad[ks];
          if (kb >= 0) bad_from = min(bad_from, ts + kb);
        }
        mbar_arrive(&ms.k_empty[ks]);
        // This row's logits for the tile, log2 units, masked past the query.
        float x[TT];
#pragma unroll
        for (int c = 0; c < TT / 32; ++c) {
          float v[32];
          tmem_ld32(lane_addr + b * 128 + c * 32, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) x[c * 32 + i] = v[i];
        }
        // Logits in log2 units are x * sc: without ALiBi the scale folds into
        // the exponent's FMA (sc = scale * log2 e > 0: the maximum of x is the
        // maximum of the logits); with ALiBi x carries the scale and the bias.
        const bool fold = !alibi && qscale > 0.f;
        const float sc = fold ? qscale : 1.f;
        if (!fold) {
#pragma unroll
          for (int i = 0; i < TT; ++i) {
            const int t = ts + i;
            x[i] = t <= pos ? fmaf(x[i], qscale, slope * (float)(t - pos)) : -INFINITY;
          }
        } else if (ts + TT - 1 > pos) {         // the tile passes this row's query
#pragma unroll
          for (int i = 0; i < TT; ++i) x[i] = ts + i <= pos ? x[i] : -INFINITY;
        }
        // Row maximum: 8 independent chains, then a 3-level tree.
        float m8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) m8[k] = x[k];
#pragma unroll
        for (int i = 8; i < TT; i += 8)
#pragma unroll
          for (int k = 0; k < 8; ++k) m8[k] = fmaxf(m8[k], x[i + k]);
        const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                               fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))) * sc;
        float alpha = 1.f;
        if (mx > m_ref + kHeadroom) {
          const float m_new = fmaxf(m_ref, mx);
          alpha = m_ref == -INFINITY ? 0.f : fast_exp2(m_ref - m_new);
          l *= alpha;
          m_ref = m_new;
        }
        // Rows whose reference moved rescale their O (accumulated in TMEM by
        // the previous tiles' P V) once the last of those has completed.
        if (__any_sync(0xffffffffu, alpha != 1.f && jl > 0)) {
          const uint32_t jp = j - 1;
          ok = ok && mbar_wait(&ms.pv_done[jp & 1], (jp >> 1) & 1);
          tc_fence_after();
          const uint32_t o_addr = lane_addr + 256 + ub * 128;
#pragma unroll
          for (int c = 0; c < HD / 32; ++c) {
            float v[32];
            uint32_t w[32];
            tmem_ld32(o_addr + c * 32, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(v[i] * alpha);
            tmem_st32(o_addr + c * 32, w);
          }
          tmem_wait_st();
        }
        // P = 2^(x * sc - m_ref), 16-bit pairs over the S buffer's first 64
        // columns; the row sum in 8 independent chains.
        float l8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t w[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float p0 = fast_exp2(fmaf(x[c * 64 + 2 * i], sc, -m_ref));
            const float p1 = fast_exp2(fmaf(x[c * 64 + 2 * i + 1], sc, -m_ref));
            l8[(2 * i) & 7] += p0;
            l8[(2 * i + 1) & 7] += p1;
            w[i] = pack2<BF16>(p0, p1);
          }
          tmem_st32(lane_addr + b * 128 + c * 32, w);
        }
        l += ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
        // Cache slots past the sequence end inside a loaded block may hold
        // anything (NaN included): zero those V rows before P V reads them
        // (thread `row` clears token row `row` of the tile).
        if (ts + TT > ui.L) {
          const int vs = j % NV;
          ok = ok && mbar_wait(&ms.v_full[vs], (j / NV) & 1);
          if (ok && ts + row >= ui.L) {
            uint4* v0 = reinterpret_cast<uint4*>(vbuf + vs * TILE_BYTES + row * 128);
            uint4* v1 = reinterpret_cast<uint4*>(vbuf + vs * TILE_BYTES + TT * 128 + row * 128);
#pragma unroll
            for (int i = 0; i < 8; ++i) v0[i] = v1[i] = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&ms.p_full[b]);
        if (pend) finalize();   // the previous unit's output, its last P V now done
      }
      if (!ok) break;
      // ---------------------------------------------------------- finalise unit
      // (written after the next unit's first P, or after the last unit)
      pend = true;
      pend_ub = ub;
      pend_valid = valid_row;
      pend_inv = !valid_row || pos >= bad_from || l == 0.f ? 0.f : 1.f / l;
      pend_dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) +
                                          ((size_t)(ui.qrow0 + qi) * H + ui.hk * g + hj) * HD);
      ++u;
    }
    if (ok && pend) finalize();
    if (!ok && threadIdx.x == 128) set_abort(ms, a.status);
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Maximum dynamic shared memory, set once per device and kernel.
template <bool BF16>
cudaError_t prepare() {
  static std::atomic<bool> attr_set[64];   // setting it twice from two threads is harmless
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(prefill_tc_kernel<BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true, std::memory_order_release);
  }
  return cudaSuccess;
}

template <bool BF16>
cudaError_t launch_t(const DecodeArgs& a, cudaStream_t st) {
  CUtensorMap km, vm, qm;
  const long long rows = (long long)a.num_blocks * a.block_size;
  const int box_rows = a.block_size < TT ? a.block_size : TT;
  const int g = a.num_heads / a.num_kv_heads;
  if (!make_kv_map(&km, a.key_cache, BF16, HD, a.num_kv_heads, rows, 64, box_rows, true) ||
      !make_kv_map(&vm, a.value_cache, BF16, HD, a.num_kv_heads, rows, 64, box_rows, true) ||
      !make_q_chunk_map(&qm, a.q, BF16, HD, a.num_heads, a.num_q_tokens, g, a.q_per_unit))
    return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaError_t e = prepare<BF16>();
  if (e != cudaSuccess) return e;
  const long long units = (long long)a.num_seqs * a.num_kv_heads * a.num_partitions;
  const int grid = (int)(units < sms ? units : sms);
  return launch_pdl(prefill_tc_kernel<BF16>, dim3(grid), dim3(kThreads), kSmemBytes, st, km, vm,
                    qm, a);
}

}  // namespace

int prefill_rows_queries_per_unit(int group) { return group >= 1 && group <= ROWS ? ROWS / group : 0; }

cudaError_t launch_prefill_rows(const DecodeArgs& a, cudaStream_t st) {
  const int g = a.num_heads / a.num_kv_heads;
  if (a.head_size != HD || g < 1 || g > 64 || a.q_per_unit != prefill_rows_queries_per_unit(g))
    return cudaErrorInvalidValue;
  return a.is_bf16 ? launch_t<true>(a, st) : launch_t<false>(a, st);
}

}  // namespace pkd
