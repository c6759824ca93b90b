// Prefill over a paged KV cache on the 5th-generation tensor cores: a chunk
// of new query tokens per sequence attends causally to the cache up to each
// query's own position.  The review comments of "[Performance] Support
// MQA/GQA in decode phase by using FlashAttention" (vLLM pull request 2744)
// note that the KV-cache attention kernel serves prefill as well, with or
// without a cached prefix; this is that generalisation, shaped for prefill.
//
// Query tile = QT = 128 / g chunk queries of one (sequence, KV head): its 128
// rows are the (query, head) pairs r = query * g + head, so all g heads of a
// query share every K/V tile.  Two kernels, both persistent (one CTA per
// SM, units dealt round-robin, heaviest first):
//   warps 0, 3 K producers (half 0 and the unit's Q tiles; half 1): TMA boxes
//              of one block x 64 columns into a ring of 32 KB stages, block
//              ids one tile ahead, out-of-range blocks from an
//              out-of-bounds row (zeros).
//   warp 1     V producer, same boxes into its own ring.
//   warp 2     MMA issuer (one thread):
//                S = Q K^T   M = 128 rows, N = 128 tokens, K = head_size,
//                            A = Q (shared memory), B = K tile, into TMEM;
//                O += P V    M = 128 rows, N = head_size, K = 128 tokens,
//                            A = P (TMEM, written by the softmax), B = V tile.
//   softmax    thread = TMEM lane = one row.  The row's 128 logits of a
//              tile are in registers, so its maximum and sum need no other
//              thread.  p = 2^(x - m_ref) with a reference maximum m_ref
//              that moves only when a logit passes it by more than 8 (log2
//              units); then l and the row of O (in TMEM) are rescaled.  P
//              goes back into TMEM as 16-bit pairs over the first 64
//              columns of the tile's S.
// Single kernel (8 warps, softmax warps 4-7): a unit is one query tile; S
// double-buffered by tile parity and O by unit parity (512 TMEM columns),
// so a unit's output is written after the next unit's first P.
// Paired kernel (12 warps): a unit is TWO consecutive query tiles (slots A
// and B) of one (sequence, KV head) and every K/V tile serves both, so a
// tile carries twice the MMA work it costs in TMA boxes and a CTA switches
// units half as often.  TMEM holds S_A, S_B, O_A, O_B; the MMA order per
// K/V tile is S_A S_B | P_A V, next S_A | P_B V, next S_B, so that each
// slot's next S runs while the softmax works on the other slot.  Warps 4-7
// run slot A's softmax and warps 8-11 slot B's, each at its own pace (the
// pattern of FlashAttention-4's two softmax warpgroups).  Per tile a thread
// loads its 128 logits with one TMEM load, takes the maximum with
// three-input max instructions, and scales and sums on packed f32 pairs;
// it settles the K stage's bookkeeping after handing over P.  The
// producers' path from a stage's release to its TMA issue holds no warp
// exchange.  A unit whose second tile does not exist (the last of an odd
// count) runs slot A only.
// Each kernel has two instantiations: FOLD (no ALiBi, scale above 0: the
// scale folds into the exponent's FMA and only tiles that pass a query are
// masked) and the general one (every logit scaled, ALiBi bias added), so
// the loop that every tile runs in the common case holds no bias code.
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
constexpr int ROWS = 128;                // (query, head) rows per query tile (= MMA M)
constexpr int TILE_BYTES = TT * HD * 2;  // one K or V tile, 32 KB
constexpr int Q_BYTES = ROWS * HD * 2;   // one Q tile, 32 KB
constexpr int NV = 2;                    // V ring stages (K: Layout::NK)
constexpr int kPfTable = 128;            // sequences whose lengths and chunk bounds sit in shared memory
constexpr int kThreads = 256;            // single kernel: 8 warps
constexpr int kThreadsPair = 384;        // paired kernel: 12 warps (two softmax warpgroups)
constexpr int kSoftmaxThreads = 128;
constexpr int kNoBlock = -2147483647 - 1;
constexpr float kHeadroom = 8.f;         // log2 units: p < 2^8 between rescales
constexpr int kPairMinTokens = 1024;     // paired kernel from this many visible tokens per query
// TMEM columns of slot x's S and O.
__host__ __device__ constexpr uint32_t col_s(int x) { return x ? 128u : 0u; }
__host__ __device__ constexpr uint32_t col_o(int x) { return x ? 384u : 256u; }

// Shared memory: two Q tiles (the single kernel's by unit parity, the
// paired kernel's slots A and B), the K ring, the V ring, then the barriers.
template <bool PAIR>
struct Layout {
  static constexpr int NK = PAIR ? 3 : 2;   // K ring stages
  static constexpr int off_q = 0;
  static constexpr int off_k = off_q + 2 * Q_BYTES;
  static constexpr int off_v = off_k + NK * TILE_BYTES;
  // Single kernel: a query tile's output, staged for its TMA store.
  static constexpr int off_stage = off_v + NV * TILE_BYTES;
  static constexpr int off_misc = off_stage + (PAIR ? 0 : Q_BYTES);
};

// Lengths and chunk bounds, in shared memory when there are at most
// kPfTable sequences.
struct PfTab {
  int L[kPfTable];        // context_lens
  int qs[kPfTable + 1];   // query_start
  int parts[kPfTable];    // query tiles of the sequence (prefill_parts)
};

constexpr int kMiscBytes = 1792;          // single kernel
constexpr int kMiscBytesPair = 1792;      // paired kernel
struct MiscPair {
  uint64_t k_full[Layout<true>::NK], k_empty[Layout<true>::NK], v_full[NV], v_empty[NV];
  // per slot (A, B)
  uint64_t q_full[2], q_empty[2], s_full[2], p_full[2], pv_done[2], o_full[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int k_bad[Layout<true>::NK];      // per K stage: token offset of the tile's first bad block id, or -1
  PfTab tab;
};
static_assert(sizeof(MiscPair) <= kMiscBytesPair, "misc area too small");

struct MiscSingle {
  uint64_t k_full[Layout<false>::NK], k_empty[Layout<false>::NK], v_full[NV], v_empty[NV];
  uint64_t q_full[2], q_empty[2], s_full[2], p_full[2], pv_done[2], o_full[2], o_empty[2], drain;
  uint64_t stage_full, stage_free;   // the output stage: rows written; read by the last store
  uint32_t tmem_base;
  int abort;
  int k_bad[Layout<false>::NK];      // per K stage: token offset of the tile's first bad block id, or -1
  PfTab tab;
};
static_assert(sizeof(MiscSingle) <= kMiscBytes, "misc area too small");

template <bool PAIR>
constexpr int smem_bytes() {
  return Layout<PAIR>::off_misc + (PAIR ? kMiscBytesPair : kMiscBytes) + 1024;   // + alignment slack
}
static_assert(smem_bytes<true>() <= 232448 && smem_bytes<false>() <= 232448,
              "above the shared memory of one CTA");

template <class M>
__device__ __forceinline__ void set_abort(M& ms, uint32_t* status) {
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
__device__ __forceinline__ UnitInfo unit_at(const PfTab& tab, const DecodeArgs& a, int s, int hk,
                                            int p) {
  UnitInfo ui;
  ui.s = s;
  ui.hk = hk;
  ui.p = p;
  ui.slot = -1;
  const bool in_tab = a.num_seqs <= kPfTable;
  ui.L = in_tab ? tab.L[s] : a.context_lens[s];
  const int q0 = in_tab ? tab.qs[s] : a.query_start[s];
  const int q1 = in_tab ? tab.qs[s + 1] : a.query_start[s + 1];
  const int parts = in_tab ? tab.parts[s] : prefill_parts(a, q0, q1, ui.L);
  ui.lok = parts > 0;
  if (p < parts) {
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
__device__ __forceinline__ void prefill_setup(PfTab& tab, const DecodeArgs& a) {
  const int nthreads = blockDim.x;
  if (a.num_seqs <= kPfTable)
    for (int i = threadIdx.x; i <= a.num_seqs; i += nthreads) {
      tab.qs[i] = a.query_start[i];
      if (i < a.num_seqs) {
        tab.L[i] = a.context_lens[i];
        tab.parts[i] = prefill_parts(a, a.query_start[i], a.query_start[i + 1], a.context_lens[i]);
      }
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
      for (size_t i = threadIdx.x; i < words; i += nthreads) o[i] = 0u;
    }
  }
  __syncthreads();
}

// Units of one CTA: unit u of S * Hk * P, dealt round-robin (consecutive
// query tiles of a causal chunk differ in cost; dealing spreads them), later
// (heavier) tiles first.
// Round-robin walk over unit indices v = blockIdx.x + k * gridDim.x, v =
// (s * Hk + hk) * per + r, kept as its parts (r, hk, s) while s < S: one
// step adds the stride's parts (from the launch arguments) with carries, no
// division.
struct UnitWalk {
  int r, hk, s;
  __device__ __forceinline__ void begin(const DecodeArgs& a, int per) {
    const int v = blockIdx.x;
    r = v % per;
    hk = (v / per) % a.num_kv_heads;
    s = (v / per) / a.num_kv_heads;
  }
  __device__ __forceinline__ bool more(const DecodeArgs& a) const { return s < a.num_seqs; }
  __device__ __forceinline__ void advance(const DecodeArgs& a, int per) {
    r += a.walk_dr;
    const int c = r >= per;
    if (c) r -= per;
    hk += a.walk_dhk + c;
    const int c2 = hk >= a.num_kv_heads;
    if (c2) hk -= a.num_kv_heads;
    s += a.walk_ds + c2;
  }
};

struct SingleCursor {
  UnitWalk w;
  __device__ __forceinline__ void begin(const DecodeArgs& a) { w.begin(a, a.num_partitions); }
  __device__ __forceinline__ bool step(const PfTab& tab, const DecodeArgs& a, UnitInfo& ui) {
    const int per = a.num_partitions;
    while (w.more(a)) {
      const int pp = per - 1 - w.r, hk = w.hk, s = w.s;
      w.advance(a, per);
      ui = unit_at(tab, a, s, hk, pp);
      if (ui.ntiles) return true;
    }
    return false;
  }
};

// A row's logits x of the tile at token ts, in log2 units and masked past
// the query's position pos.  When the scale folds into the exponent's FMA
// (fold: no ALiBi and a scale above 0) only a tile that passes the query is
// touched; otherwise each visible logit is scaled and gets the bias slope *
// (t - pos) (slope 0 without ALiBi).  FOLD instantiates a kernel for the
// folded case alone (the host launches it for exactly that case), so the
// common kernel carries no bias code in the loop that every tile runs.
template <bool FOLD>
__device__ __forceinline__ void mask_logits(float (&x)[TT], bool fold, float qscale, float slope,
                                            int ts, int pos) {
  if (!FOLD && !fold) {
#pragma unroll
    for (int i = 0; i < TT; ++i) {
      const int t = ts + i;
      x[i] = t <= pos ? fmaf(x[i], qscale, slope * (float)(t - pos)) : -INFINITY;
    }
  } else if (ts + TT - 1 > pos) {            // the tile passes this row's query
#pragma unroll
    for (int i = 0; i < TT; ++i) x[i] = ts + i <= pos ? x[i] : -INFINITY;
  }
}

template <bool BF16, bool FOLD>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_single_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap,
                      const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap omap, const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  uint8_t* qbuf = sm + Layout<false>::off_q;
  uint8_t* kbuf = sm + Layout<false>::off_k;
  uint8_t* vbuf = sm + Layout<false>::off_v;
  uint8_t* stage = sm + Layout<false>::off_stage;
  MiscSingle& ms = *reinterpret_cast<MiscSingle*>(sm + Layout<false>::off_misc);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = a.num_heads / a.num_kv_heads;
  // A K stage is free once the MMA is done with it and the softmax has read
  // the stage's bad-block entry (without that arrival a stage could be
  // refilled before the softmax checks it).
  constexpr uint32_t kMmaCount = 1;

  // ---------------------------------------------------------------- setup
  prefetch_schedule_inputs(a);
  if (threadIdx.x == 0) {
    for (int i = 0; i < Layout<false>::NK; ++i) {
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
    mbar_init(&ms.stage_full, kSoftmaxThreads);
    mbar_init(&ms.stage_free, 1);
    ms.abort = 0;
    fence_barrier_init();
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    tma_prefetch_desc(&omap);
    tma_prefetch_desc(&qmap);
  }
  if (warp == 2) {
    tmem_alloc(&ms.tmem_base, 512);
    tmem_relinquish();
  }
  pdl_wait();
  pdl_launch_dependents();
  prefill_setup(ms.tab, a);
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
    const int nst = is_v ? NV : Layout<false>::NK;
    uint64_t* full = is_v ? ms.v_full : ms.k_full;
    uint64_t* empty = is_v ? ms.v_empty : ms.k_empty;
    const bool issuer = lane < 2 * nbox && ((half_mask >> (lane / nbox)) & 1);
    const int my_box = lane % nbox, my_half = lane / nbox;
    auto load_raw = [&](const UnitInfo& t, int tj) {
      int raw = kNoBlock;
      if (lane < 2 * nbox) {
        const int ts = tj * TT;
        const int tok0 = B <= TT ? ts + my_box * B : ts;
        if (tok0 < t.t1) raw = __ldg(a.block_tables + (size_t)t.s * a.max_blocks_per_seq + tok0 / B);
      }
      return raw;
    };
    SingleCursor cur;
    cur.begin(a);
    UnitInfo ui;
    bool have = cur.step(ms.tab, a, ui);
    int jl = 0;
    int raw = have ? load_raw(ui, 0) : kNoBlock;
    uint32_t jk = 0, un = 0;
    bool ok = true;
    while (have) {
      UnitInfo nui = ui;
      bool nhave = true;
      int njl = jl + 1;
      if (njl >= ui.ntiles) {
        nhave = cur.step(ms.tab, a, nui);
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
      // lanes < nbox: boxes in token order
      const uint32_t bad_lanes = __ballot_sync(0xffffffffu, bad && lane < nbox);
      const int st = jk % nst;
      // Every lane polls the stage barrier, and each issuer lane holds its
      // own box's row: nothing on the way from the stage's release to the
      // TMA issue is a warp exchange.  The stage's transaction count may
      // go below zero until lane 0's expect-tx arrives; its one pending
      // arrival keeps the phase open until then.
      ok = ok && mbar_wait(&empty[st], ((jk / nst) & 1) ^ 1);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      if (issuer) {
        uint8_t* dst = ring + st * TILE_BYTES + my_half * TT * 128 + my_box * R * 128;
        tma_load_3d(dst, map, &full[st], my_half * 64, ui.hk, row);
      }
      if (lane == 0 && primary) {
        if (!is_v) {
          ms.k_bad[st] = bad_lanes ? (__ffs(bad_lanes) - 1) * R : -1;
          if (bad_lanes) flag(a.status, PKD_DEV_BAD_BLOCK);
        }
        mbar_arrive_expect_tx(&full[st], TILE_BYTES);
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
      SingleCursor cur;
      cur.begin(a);
      UnitInfo ui;
      while (ok && cur.step(ms.tab, a, ui)) {
        const int qb = un & 1;
        ok = ok && mbar_wait(&ms.q_full[qb], (un >> 1) & 1);
        for (int jl = 0; jl < ui.ntiles && ok; ++jl, ++j) {
          const int ks = j % Layout<false>::NK, b = j & 1;
          ok = mbar_wait(&ms.k_full[ks], (j / Layout<false>::NK) & 1);
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
    bool pend = false, pend_valid = false, pend_whole = false;
    int pend_ub = 0, pend_hk = 0, pend_qrow0 = 0;
    float pend_inv = 0.f;
    uint4* pend_dst = nullptr;
    // A unit's output rows.  A whole query tile goes through shared memory:
    // each thread writes its row there (128-byte swizzled, the layout of the
    // output tensor map's two {64, g, QT} boxes) and one thread stores the
    // tile with two TMA stores, so the warpgroup's load/store path is not
    // left with 16 global stores a thread in front of its next waits.  A
    // partial tile (the end of a chunk) is written row by row.
    uint32_t n_whole = 0;   // whole tiles stored through the stage
    auto finalize = [&]() {
      ok = ok && mbar_wait(&ms.o_full[pend_ub], (u_fin >> 1) & 1);
      if (!ok) return;
      tc_fence_after();
      if (pend_whole) {
        // The stage is free once the previous tile's store has read it.
        if (threadIdx.x == 128) {
          bulk_wait_read_all();
          mbar_arrive(&ms.stage_free);
        }
        ok = mbar_wait(&ms.stage_free, n_whole & 1);
        if (!ok) return;
      }
      // A rolled loop: this code runs once per unit, and unrolled it would
      // take instruction-cache room from the loop every tile runs.
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        float v[32];
        tmem_ld32(lane_addr + 256 + pend_ub * 128 + c * 32, v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 w = make_uint4(pack2<BF16>(v[8 * i] * pend_inv, v[8 * i + 1] * pend_inv),
                                     pack2<BF16>(v[8 * i + 2] * pend_inv, v[8 * i + 3] * pend_inv),
                                     pack2<BF16>(v[8 * i + 4] * pend_inv, v[8 * i + 5] * pend_inv),
                                     pack2<BF16>(v[8 * i + 6] * pend_inv, v[8 * i + 7] * pend_inv));
          if (pend_whole) {
            // 16-byte chunk ch of this row's 64-column half (c >> 1).
            const int ch = (c & 1) * 4 + i;
            *reinterpret_cast<uint4*>(stage + (c >> 1) * Q_BYTES / 2 + row * 128 +
                                      ((ch ^ (row & 7)) << 4)) = w;
          } else if (pend_valid) {
            pend_dst[c * 4 + i] = w;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&ms.o_empty[pend_ub]);
      if (pend_whole) {
        fence_proxy_async_smem();   // the stage's writes, before the TMA reads them
        mbar_arrive(&ms.stage_full);
        if (threadIdx.x == 128) {
          ok = mbar_wait(&ms.stage_full, n_whole & 1);
          if (ok) {
            tma_store_3d(&omap, stage, 0, pend_hk * g, pend_qrow0);
            tma_store_3d(&omap, stage + Q_BYTES / 2, 64, pend_hk * g, pend_qrow0);
            bulk_commit();
          }
        }
        ++n_whole;
      }
      pend = false;
      ++u_fin;
    };
    SingleCursor cur;
    cur.begin(a);
    UnitInfo ui;
    while (ok && cur.step(ms.tab, a, ui)) {
      const int ub = u & 1;
      const bool valid_row = qi < ui.nq;
      const int pos = valid_row ? ui.pos0 + qi : -1;      // last visible token
      const float slope = alibi && valid_row ? a.alibi[ui.hk * g + hj] * kLog2e : 0.f;
      float m_ref = valid_row ? -INFINITY : INFINITY;       // +inf: p = 0, never rescales
      float l = 0.f;
      int bad_from = 0x7fffffff;
      for (int jl = 0; jl < ui.ntiles; ++jl, ++j) {
        const int b = j & 1, ks = j % Layout<false>::NK;
        const int ts = jl * TT;
        ok = ok && mbar_wait(&ms.s_full[b], (j >> 1) & 1);
        if (!ok) break;
        tc_fence_after();
        // This row's logits for the tile, log2 units, masked past the query.
        float x[TT];
        tmem_ld128(lane_addr + b * 128, x);
        // Logits in log2 units are x * sc: folded (no ALiBi, sc = scale *
        // log2 e > 0: the maximum of x is the maximum of the logits), or x
        // carries the scale and the bias.
        const bool fold = FOLD || (!alibi && qscale > 0.f);
        const float sc = fold ? qscale : 1.f;
        mask_logits<FOLD>(x, fold, qscale, slope, ts, pos);
        // Row maximum: 8 independent chains of three-input maxima, then a
        // tree.
        float m8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) m8[k] = fmaxf(x[k], x[8 + k]);
#pragma unroll
        for (int i = 16; i < TT; i += 16)
#pragma unroll
          for (int k = 0; k < 8; ++k) m8[k] = fmax3(m8[k], x[i + k], x[i + 8 + k]);
        const float mx = fmaxf(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], fmax3(m8[5], m8[6], m8[7]))) * sc;
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
#pragma unroll 1   // rare: kept out of the instruction cache's way
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
        // columns.  The scaling and the row sum run on packed pairs (one
        // instruction for two values), the sum in 4 independent pair chains.
        const uint64_t sc2 = f2_pack(sc, sc), nm2 = f2_pack(-m_ref, -m_ref);
        uint64_t l2[4] = {0, 0, 0, 0};
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t w[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float2 es = f2_unpack(f2_fma(f2_pack(x[c * 64 + 2 * i], x[c * 64 + 2 * i + 1]), sc2, nm2));
            const uint64_t p2 = f2_pack(fast_exp2(es.x), fast_exp2(es.y));
            l2[i & 3] = f2_add(l2[i & 3], p2);
            const float2 ps = f2_unpack(p2);
            w[i] = pack2<BF16>(ps.x, ps.y);
          }
          tmem_st32(lane_addr + b * 128 + c * 32, w);
        }
        {
          const float2 lt = f2_unpack(f2_add(f2_add(l2[0], l2[1]), f2_add(l2[2], l2[3])));
          l += lt.x + lt.y;
        }
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
        // The K stage's bad-block entry, then the stage's release (the
        // MMA's commit is its other arrival), off the path from S to P.
        ok = ok && mbar_wait(&ms.k_full[ks], (j / Layout<false>::NK) & 1);
        if (ok) {
          const int kb = ms.k_bad[ks];
          if (kb >= 0) bad_from = min(bad_from, ts + kb);
        }
        mbar_arrive(&ms.k_empty[ks]);
        if (!ok) break;
        if (pend) finalize();   // the previous unit's output, its last P V now done
      }
      if (!ok) break;
      // ---------------------------------------------------------- finalise unit
      // (written after the next unit's first P, or after the last unit)
      pend = true;
      pend_ub = ub;
      pend_valid = valid_row;
      pend_whole = ui.nq == a.q_per_unit;
      pend_hk = ui.hk;
      pend_qrow0 = ui.qrow0;
      pend_inv = !valid_row || pos >= bad_from || l == 0.f ? 0.f : 1.f / l;
      pend_dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) +
                                          ((size_t)(ui.qrow0 + qi) * H + ui.hk * g + hj) * HD);
      ++u;
    }
    if (ok && pend) finalize();
    if (threadIdx.x == 128) bulk_wait_all();   // every output store done before the CTA exits
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

// A unit: query tiles 2pp (slot A) and 2pp + 1 (slot B) of one (sequence,
// KV head), walked over the K/V tiles up to the later tile's last query.
struct PairUnit {
  int s, hk, L, t1, ntiles;
  bool hasB;
  int qrow0[2], nq[2], pos0[2];   // per slot: first packed q row, queries, first position
};

// Units of one CTA: unit u of S * Hk * ceil(P / 2), dealt round-robin
// (consecutive query tiles of a causal chunk differ in cost; dealing spreads
// them), later (heavier) pairs first.
struct PairCursor {
  UnitWalk w;
  __device__ __forceinline__ void begin(const DecodeArgs& a) { w.begin(a, (a.num_partitions + 1) / 2); }
  __device__ __forceinline__ bool step(const PfTab& tab, const DecodeArgs& a, PairUnit& pu) {
    const int per = (a.num_partitions + 1) / 2;
    while (w.more(a)) {
      const int pp = per - 1 - w.r, hk = w.hk, s = w.s;
      w.advance(a, per);
      const UnitInfo ua = unit_at(tab, a, s, hk, 2 * pp);
      if (ua.ntiles == 0) continue;   // no tile 2pp, so no tile 2pp + 1 either
      const UnitInfo ub = unit_at(tab, a, s, hk, 2 * pp + 1);
      pu.s = s;
      pu.hk = hk;
      pu.L = ua.L;
      pu.hasB = ub.ntiles > 0;
      pu.t1 = pu.hasB ? ub.t1 : ua.t1;
      pu.ntiles = pu.hasB ? ub.ntiles : ua.ntiles;
      pu.qrow0[0] = ua.qrow0;
      pu.nq[0] = ua.nq;
      pu.pos0[0] = ua.pos0;
      pu.qrow0[1] = pu.hasB ? ub.qrow0 : 0;
      pu.nq[1] = pu.hasB ? ub.nq : 0;
      pu.pos0[1] = pu.hasB ? ub.pos0 : 0;
      return true;
    }
    return false;
  }
};

template <bool BF16, bool FOLD>
__global__ void __launch_bounds__(kThreadsPair, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap,
                      const __grid_constant__ CUtensorMap qmap, const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  uint8_t* qbuf = sm + Layout<true>::off_q;
  uint8_t* kbuf = sm + Layout<true>::off_k;
  uint8_t* vbuf = sm + Layout<true>::off_v;
  MiscPair& ms = *reinterpret_cast<MiscPair*>(sm + Layout<true>::off_misc);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = a.num_heads / a.num_kv_heads;

  // ---------------------------------------------------------------- setup
  prefetch_schedule_inputs(a);
  if (threadIdx.x == 0) {
    for (int i = 0; i < Layout<true>::NK; ++i) {
      // Freed by the MMA (after the tile's last S) and by the softmax, which
      // reads the stage's bad-block entry: without its arrival a stage could
      // be refilled before the softmax has checked it.
      mbar_init(&ms.k_full[i], 1);
      mbar_init(&ms.k_empty[i], 1 + 2 * kSoftmaxThreads);
      ms.k_bad[i] = -1;
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(&ms.v_full[i], 1);
      mbar_init(&ms.v_empty[i], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&ms.q_full[x], 1);
      mbar_init(&ms.q_empty[x], 1);
      mbar_init(&ms.s_full[x], 1);
      mbar_init(&ms.p_full[x], kSoftmaxThreads);
      mbar_init(&ms.pv_done[x], 1);
      mbar_init(&ms.o_full[x], 1);
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
  prefill_setup(ms.tab, a);
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
    const int nst = is_v ? NV : Layout<true>::NK;
    uint64_t* full = is_v ? ms.v_full : ms.k_full;
    uint64_t* empty = is_v ? ms.v_empty : ms.k_empty;
    const bool issuer = lane < 2 * nbox && ((half_mask >> (lane / nbox)) & 1);
    const int my_box = lane % nbox, my_half = lane / nbox;
    auto load_raw = [&](const PairUnit& t, int tj) {
      int raw = kNoBlock;
      if (lane < 2 * nbox) {
        const int ts = tj * TT;
        const int tok0 = B <= TT ? ts + my_box * B : ts;
        if (tok0 < t.t1) raw = __ldg(a.block_tables + (size_t)t.s * a.max_blocks_per_seq + tok0 / B);
      }
      return raw;
    };
    PairCursor cur;
    cur.begin(a);
    PairUnit pu;
    bool have = cur.step(ms.tab, a, pu);
    int jl = 0;
    int raw = have ? load_raw(pu, 0) : kNoBlock;
    uint32_t jk = 0, un = 0, unb = 0;   // tiles, units, units with slot B
    bool ok = true;
    while (have) {
      PairUnit npu = pu;
      bool nhave = true;
      int njl = jl + 1;
      if (njl >= pu.ntiles) {
        nhave = cur.step(ms.tab, a, npu);
        njl = 0;
      }
      const int nraw = nhave ? load_raw(npu, njl) : kNoBlock;
      if (!is_v && primary && jl == 0 && lane == 0) {
        // The unit's query tiles: box {64, g, QT} (rows (query, head)) over
        // q [T][H][D], two 64-column halves per slot.
        const uint32_t qbytes = (uint32_t)(g * a.q_per_unit * 256);
        ok = mbar_wait(&ms.q_empty[0], (un & 1) ^ 1);
        if (ok) {
          mbar_arrive_expect_tx(&ms.q_full[0], qbytes);
          tma_load_3d(qbuf, &qmap, &ms.q_full[0], 0, pu.hk * g, pu.qrow0[0]);
          tma_load_3d(qbuf + ROWS * 128, &qmap, &ms.q_full[0], 64, pu.hk * g, pu.qrow0[0]);
        }
        if (ok && pu.hasB) {
          ok = mbar_wait(&ms.q_empty[1], (unb & 1) ^ 1);
          if (ok) {
            mbar_arrive_expect_tx(&ms.q_full[1], qbytes);
            tma_load_3d(qbuf + Q_BYTES, &qmap, &ms.q_full[1], 0, pu.hk * g, pu.qrow0[1]);
            tma_load_3d(qbuf + Q_BYTES + ROWS * 128, &qmap, &ms.q_full[1], 64, pu.hk * g,
                        pu.qrow0[1]);
          }
        }
      }
      const int ts = jl * TT;
      const bool bad = raw != kNoBlock && (raw < 0 || raw >= a.num_blocks);
      const int row = (raw != kNoBlock && !bad) ? raw * B + (B <= TT ? 0 : ts % B) : oob_row;
      // lanes < nbox: boxes in token order
      const uint32_t bad_lanes = __ballot_sync(0xffffffffu, bad && lane < nbox);
      const int st = jk % nst;
      // Every lane polls the stage barrier, and each issuer lane holds its
      // own box's row: nothing on the way from the stage's release to the
      // TMA issue is a warp exchange.  The stage's transaction count may
      // go below zero until lane 0's expect-tx arrives; its one pending
      // arrival keeps the phase open until then.
      ok = ok && mbar_wait(&empty[st], ((jk / nst) & 1) ^ 1);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      if (issuer) {
        uint8_t* dst = ring + st * TILE_BYTES + my_half * TT * 128 + my_box * R * 128;
        tma_load_3d(dst, map, &full[st], my_half * 64, pu.hk, row);
      }
      if (lane == 0 && primary) {
        if (!is_v) {
          ms.k_bad[st] = bad_lanes ? (__ffs(bad_lanes) - 1) * R : -1;
          if (bad_lanes) flag(a.status, PKD_DEV_BAD_BLOCK);
        }
        mbar_arrive_expect_tx(&full[st], TILE_BYTES);
      }
      ++jk;
      if (njl == 0) {
        ++un;
        if (pu.hasB) ++unb;
      }
      have = nhave;
      pu = npu;
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
      uint32_t j = 0, jb = 0, un = 0, unb = 0;   // tiles (slot B's separately), units
      bool ok = true;
      // S_X(tile jj) = Q_X K^T into slot X's S columns.
      auto issue_s = [&](int x, uint32_t jj) {
        const int ks = jj % Layout<true>::NK;
        const uint32_t d = tmem + col_s(x);
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint64_t ad = smem_desc(qaddr + x * Q_BYTES + (k >> 2) * ROWS * 128 + (k & 3) * 32,
                                        16, 1024, kSwizzle128B);
          const uint64_t bd = smem_desc(kaddr + ks * TILE_BYTES + (k >> 2) * TT * 128 + (k & 3) * 32,
                                        16, 1024, kSwizzle128B);
          mma_f16(d, ad, bd, id_s, k > 0);
        }
        mma_commit(&ms.s_full[x]);
      };
      // O_X += P_X V (tile jj; `first`: the unit's first tile overwrites O_X).
      auto issue_pv = [&](int x, uint32_t jj, bool first) {
        const int vs = jj % NV;
        const uint32_t d = tmem + col_o(x);
#pragma unroll
        for (int k = 0; k < TT / 16; ++k) {
          const uint64_t bd = smem_desc(vaddr + vs * TILE_BYTES + k * 2048, TT * 128, 1024,
                                        kSwizzle128B);
          mma_f16_ts(d, tmem + col_s(x) + k * 8, bd, id_o, !(first && k == 0));
        }
        mma_commit(&ms.pv_done[x]);
      };
      PairCursor cur;
      cur.begin(a);
      PairUnit pu;
      while (ok && cur.step(ms.tab, a, pu)) {
        const int nt = pu.ntiles;
        const bool hb = pu.hasB;
        // The unit's first S of each slot.
        ok = mbar_wait(&ms.q_full[0], un & 1);
        if (ok && hb) ok = mbar_wait(&ms.q_full[1], unb & 1);
        ok = ok && mbar_wait(&ms.k_full[j % Layout<true>::NK], (j / Layout<true>::NK) & 1);
        if (!ok) break;
        tc_fence_after();
        issue_s(0, j);
        if (hb) issue_s(1, j);
        mma_commit(&ms.k_empty[j % Layout<true>::NK]);
        if (nt == 1) {
          mma_commit(&ms.q_empty[0]);
          if (hb) mma_commit(&ms.q_empty[1]);
        }
        for (int jl = 0; jl < nt && ok; ++jl) {
          const uint32_t jj = j + jl;
          const bool more = jl + 1 < nt;
          // Slot A: P_A V, then (the S_A columns free again) the next S_A.
          ok = mbar_wait(&ms.v_full[jj % NV], (jj / NV) & 1) &&
               mbar_wait(&ms.p_full[0], jj & 1);
          if (!ok) break;
          tc_fence_after();
          issue_pv(0, jj, jl == 0);
          if (jl == nt - 1) mma_commit(&ms.o_full[0]);
          if (more) {
            ok = mbar_wait(&ms.k_full[(jj + 1) % Layout<true>::NK], ((jj + 1) / Layout<true>::NK) & 1);
            if (!ok) break;
            tc_fence_after();
            issue_s(0, jj + 1);
          }
          // Slot B likewise.
          if (hb) {
            ok = mbar_wait(&ms.p_full[1], (jb + jl) & 1);
            if (!ok) break;
            tc_fence_after();
            issue_pv(1, jj, jl == 0);
            if (jl == nt - 1) mma_commit(&ms.o_full[1]);
            if (more) issue_s(1, jj + 1);
          }
          mma_commit(&ms.v_empty[jj % NV]);
          if (more) {
            mma_commit(&ms.k_empty[(jj + 1) % Layout<true>::NK]);
            if (jl + 2 == nt) {   // the unit's last S of each slot
              mma_commit(&ms.q_empty[0]);
              if (hb) mma_commit(&ms.q_empty[1]);
            }
          }
        }
        j += nt;
        if (hb) jb += nt;
        ++un;
        if (hb) ++unb;
      }
      if (!ok) set_abort(ms, a.status);
      mma_commit(&ms.drain);
      mbar_wait(&ms.drain, 0, 100000000ull);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ============================================================ softmax / epilogue
    // Warpgroup x (warps 4-7: slot A, warps 8-11: slot B) works on its own
    // slot's tiles: thread = TMEM lane = one row, the row's 128 logits of a
    // tile in its registers.  The two warpgroups are coupled only through
    // the MMA order, so on every SM sub-partition one warp's exponentials
    // overlap the other's TMEM loads and reductions.
    const int wq = warp & 3;                   // TMEM lane quadrant
    const int x = (warp - 4) >> 2;             // slot of this warpgroup
    const int row = wq * 32 + lane;            // this thread's row of S, P and O
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    const uint32_t s_addr = lane_addr + col_s(x), o_addr = lane_addr + col_o(x);
    const float qscale = a.scale * kLog2e;
    const int H = a.num_heads;
    const int qi = row / g, hj = row - qi * g; // row = (tile query qi, head hj of the group)
    const bool alibi = a.alibi != nullptr;
    const bool fold = FOLD || (!alibi && qscale > 0.f);
    const float sc = fold ? qscale : 1.f;
    uint32_t j = 0, jx = 0, ux = 0;            // tiles of all units, tiles and units of this slot
    bool ok = true;
    PairCursor cur;
    cur.begin(a);
    PairUnit pu;
    while (ok && cur.step(ms.tab, a, pu)) {
      // Slot B of a unit without a second query tile has no work, but its
      // warpgroup still releases every K stage the unit uses.
      const bool mine = x == 0 || pu.hasB;
      const bool valid = mine && qi < pu.nq[x];
      const int pos = valid ? pu.pos0[x] + qi : -1;         // last visible token
      const float slope = alibi && valid ? a.alibi[pu.hk * g + hj] * kLog2e : 0.f;
      float m_ref = valid ? -INFINITY : INFINITY;           // +inf: p = 0, never rescales
      float l = 0.f;
      int bad_from = 0x7fffffff;
      for (int jl = 0; jl < pu.ntiles; ++jl, ++j) {
        const int ks = j % Layout<true>::NK;
        const int ts = jl * TT;
        // The K stage's bad-block entry, then the stage's release (the
        // MMA's commit is its other arrival).  A slot with work does this
        // after handing over the tile's P, off the path from S to P.
        auto release_k = [&]() {
          ok = ok && mbar_wait(&ms.k_full[ks], (j / Layout<true>::NK) & 1);
          if (ok) {
            const int kb = ms.k_bad[ks];
            if (kb >= 0) bad_from = min(bad_from, ts + kb);
          }
          mbar_arrive(&ms.k_empty[ks]);
        };
        if (!mine) {
          release_k();
          if (!ok) break;
          continue;
        }
        ok = ok && mbar_wait(&ms.s_full[x], jx & 1);
        if (!ok) break;
        tc_fence_after();
        // This row's logits for the tile in one TMEM load, log2 units,
        // masked past the query: folded (no ALiBi, sc = scale * log2 e > 0:
        // the maximum of xv is the maximum of the logits), or xv carries the
        // scale and the bias.
        float xv[TT];
        tmem_ld128(s_addr, xv);
        mask_logits<FOLD>(xv, fold, qscale, slope, ts, pos);
        float m8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) m8[k] = fmaxf(xv[k], xv[8 + k]);
#pragma unroll
        for (int i = 16; i < TT; i += 16)
#pragma unroll
          for (int k = 0; k < 8; ++k) m8[k] = fmax3(m8[k], xv[i + k], xv[i + 8 + k]);
        const float mx = fmaxf(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], fmax3(m8[5], m8[6], m8[7]))) * sc;
        float alpha = 1.f;
        if (mx > m_ref + kHeadroom) {
          const float m_new = fmaxf(m_ref, mx);
          alpha = m_ref == -INFINITY ? 0.f : fast_exp2(m_ref - m_new);
          l *= alpha;
          m_ref = m_new;
        }
        // P = 2^(xv * sc - m_ref), 16-bit pairs over the S buffer's first 64
        // columns (half h's into columns [32h, 32h + 32), which held only
        // first-half logits).  The scaling and the row sum run on packed
        // pairs (one instruction for two values), the sum in 4 independent
        // pair chains.
        const uint64_t sc2 = f2_pack(sc, sc), nm2 = f2_pack(-m_ref, -m_ref);
        uint64_t l2[4] = {0, 0, 0, 0};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 es = f2_unpack(f2_fma(f2_pack(xv[32 * c + 2 * i], xv[32 * c + 2 * i + 1]), sc2, nm2));
            const uint64_t p2 = f2_pack(fast_exp2(es.x), fast_exp2(es.y));
            l2[i & 3] = f2_add(l2[i & 3], p2);
            const float2 ps = f2_unpack(p2);
            w[i] = pack2<BF16>(ps.x, ps.y);
          }
          tmem_st16(s_addr + c * 16, w);
        }
        {
          const float2 lt = f2_unpack(f2_add(f2_add(l2[0], l2[1]), f2_add(l2[2], l2[3])));
          l += lt.x + lt.y;
        }
        // Rows whose reference moved rescale their O (accumulated in TMEM by
        // the slot's previous P V) once that P V has completed, before this
        // tile's P V: after the exponentials, when the logits no longer
        // hold registers.
        if (__any_sync(0xffffffffu, alpha != 1.f && jl > 0)) {
          ok = ok && mbar_wait(&ms.pv_done[x], (jx - 1) & 1);
          tc_fence_after();
#pragma unroll 1   // rare: kept out of the instruction cache's way
          for (int c = 0; c < HD / 16; ++c) {
            float v[16];
            uint32_t w[16];
            tmem_ld16(o_addr + c * 16, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(v[i] * alpha);
            tmem_st16(o_addr + c * 16, w);
          }
          tmem_wait_st();
        }
        // Cache slots past the sequence end inside a loaded block may hold
        // anything (NaN included): slot A's warpgroup zeroes those V rows
        // before its P V, the first to read the tile (thread `row` clears
        // token row `row`).
        if (x == 0 && ts + TT > pu.L) {
          const int vs = j % NV;
          ok = ok && mbar_wait(&ms.v_full[vs], (j / NV) & 1);
          if (ok && ts + row >= pu.L) {
            uint4* v0 = reinterpret_cast<uint4*>(vbuf + vs * TILE_BYTES + row * 128);
            uint4* v1 = reinterpret_cast<uint4*>(vbuf + vs * TILE_BYTES + TT * 128 + row * 128);
#pragma unroll
            for (int i = 0; i < 8; ++i) v0[i] = v1[i] = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&ms.p_full[x]);
        release_k();
        if (!ok) break;
        ++jx;
      }
      if (!ok) break;
      if (!mine) continue;
      // ---------------------------------------------------------- finish the unit
      // Wait for the slot's last P V, then write this row of O / l.  The
      // next unit's first P V (which overwrites O) waits for this
      // warpgroup's next P, so O is read before it is reused.
      ok = mbar_wait(&ms.o_full[x], ux & 1);
      if (!ok) break;
      tc_fence_after();
      const float inv = !valid || pos >= bad_from || l == 0.f ? 0.f : 1.f / l;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) +
                                            ((size_t)(valid ? pu.qrow0[x] + qi : 0) * H +
                                             pu.hk * g + hj) * HD);
      // A rolled loop over 32-column pieces: this runs once per unit, and
      // unrolled it would take instruction-cache room from the tile loop.
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        float v[32];
        tmem_ld32(o_addr + c * 32, v);
        if (valid) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[c * 4 + i] = make_uint4(pack2<BF16>(v[8 * i] * inv, v[8 * i + 1] * inv),
                                        pack2<BF16>(v[8 * i + 2] * inv, v[8 * i + 3] * inv),
                                        pack2<BF16>(v[8 * i + 4] * inv, v[8 * i + 5] * inv),
                                        pack2<BF16>(v[8 * i + 6] * inv, v[8 * i + 7] * inv));
        }
      }
      tc_fence_before();
      ++ux;
    }
    if (!ok) set_abort(ms, a.status);
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
template <bool BF16, bool FOLD, bool PAIR>
cudaError_t prepare() {
  static std::atomic<bool> attr_set[64];   // setting it twice from two threads is harmless
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
    e = PAIR ? cudaFuncSetAttribute(prefill_pair_kernel<BF16, FOLD>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes<true>())
             : cudaFuncSetAttribute(prefill_single_kernel<BF16, FOLD>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes<false>());
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true, std::memory_order_release);
  }
  return cudaSuccess;
}

// The paired kernel halves the K/V loads and the unit switches per query
// tile but single-buffers Q, S and O, so each switch costs a pipeline
// bubble: it pays when units are long.  It is taken for chunks of two or
// more query tiles whose queries see at least kPairMinTokens cache tokens on
// average by the host's bounds (a chunk over a long cached prefix): a
// 256-token chunk after 3840 cached tokens runs in 149 us against 171 on the
// single kernel, while 1024-token prompts without prefix ran 237 -> 298 us
// on the paired kernel's first version.
template <bool BF16, bool FOLD>
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
  const bool pair = a.num_partitions >= 2 && a.max_context_len - a.max_query_len / 2 >= kPairMinTokens;
  cudaError_t e = pair ? prepare<BF16, FOLD, true>() : prepare<BF16, FOLD, false>();
  if (e != cudaSuccess) return e;
  const int per = pair ? (a.num_partitions + 1) / 2 : a.num_partitions;
  const long long units = (long long)a.num_seqs * a.num_kv_heads * per;
  const int grid = (int)(units < sms ? units : sms);
  DecodeArgs la = a;
  la.walk_dr = grid % per;
  la.walk_dhk = (grid / per) % a.num_kv_heads;
  la.walk_ds = (grid / per) / a.num_kv_heads;
  if (pair)
    return launch_pdl(prefill_pair_kernel<BF16, FOLD>, dim3(grid), dim3(kThreadsPair), smem_bytes<true>(),
                      st, km, vm, qm, la);
  CUtensorMap om;   // the output, boxes like the query tiles'
  if (!make_q_chunk_map(&om, a.out, BF16, HD, a.num_heads, a.num_q_tokens, g, a.q_per_unit))
    return cudaErrorInvalidValue;
  return launch_pdl(prefill_single_kernel<BF16, FOLD>, dim3(grid), dim3(kThreads), smem_bytes<false>(), st,
                    km, vm, qm, om, la);
}

}  // namespace

int prefill_rows_queries_per_unit(int group) { return group >= 1 && group <= ROWS ? ROWS / group : 0; }

cudaError_t launch_prefill_rows(const DecodeArgs& a, cudaStream_t st) {
  const int g = a.num_heads / a.num_kv_heads;
  if (a.head_size != HD || g < 1 || g > 64 || a.q_per_unit != prefill_rows_queries_per_unit(g))
    return cudaErrorInvalidValue;
  // The scale folds into the exponent's FMA when it is above 0 and there is
  // no bias.
  if (a.alibi == nullptr && a.scale > 0.f)
    return a.is_bf16 ? launch_t<true, true>(a, st) : launch_t<false, true>(a, st);
  return a.is_bf16 ? launch_t<true, false>(a, st) : launch_t<false, false>(a, st);
}

}  // namespace pkd
