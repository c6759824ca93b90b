// Decode attention over a paged KV cache on the 5th-generation tensor cores
// (tcgen05 MMA, accumulators in TMEM), K/V staged by TMA.  Used when a KV head
// is shared by 4..64 query heads (GQA / MQA) with head_size 128: then
// q K^T and p V are real dense contractions of a tile of 128 cached tokens
// against the whole query group, which is why the group sharing of
// "Optimize MQA Kernel" (vLLM pull request 452) and the GQA case of
// "[Performance] Support MQA/GQA in decode phase by using FlashAttention"
// (pull request 2744) map onto them.
//
// Work unit = (sequence s, KV head, context partition).  A persistent grid of
// one CTA per SM walks its units round-robin; inside the CTA, warps are
// specialised and linked by mbarriers so the K/V stream never stops at unit
// boundaries:
//   warps 0, 6 producers (K and q; V): read block ids one tile ahead and
//              issue the TMA loads of a 128-token tile from up to 32 lanes
//              at once (one box per block and 64-column half) into rings of
//              32 KB stages.  Blocks past the partition end (and
//              out-of-range ids) are loaded from an out-of-bounds
//              coordinate, which TMA fills with zeros without touching
//              memory.
//   warp 1     MMA issuer (one thread): S^T = K q^T (M = 128 tokens,
//              N = group padded to 16) into TMEM, then O^T = V^T P^T
//              (M = 128 = head_size, K = 128 tokens).
//   warps 2-5  softmax / epilogue (thread = TMEM lane = token row of S and
//              d row of O): online softmax with per-tile maxima shared
//              through shared memory, P written (16-bit) for the second MMA,
//              O accumulated in registers with the running rescale, and the
//              final (or partial, for split context) result written.
// Shared-memory operands use the 128-byte swizzled canonical layouts: K, q and
// P K-major, V MN-major (head_size contiguous).
//
// Split context comes in three forms.  Workspace form: each unit writes its
// partial (o, m, l) to global memory and lse_reduce merges them in a second
// launch.  Cluster form (small grids): the P partitions of one (sequence, KV
// head) are the P CTAs of one thread-block cluster, one unit each; they keep
// their partials in shared memory and merge them over distributed shared
// memory before the kernel ends, so there is neither workspace nor merge
// launch.  Stream form: every CTA takes an equal share of all tiles, and the
// pairs cut at share edges are merged by a second launch.  The form is a
// template argument (plain -- unsplit or workspace --, cluster, stream), so
// each instantiation holds only its own form's code: on short calls the
// instruction footprint is part of the time.
#include <cuda.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "schedule.cuh"
#include "sm100.cuh"

namespace pkd {
namespace {

using namespace sm100;

constexpr int TT = 128;                 // tokens per tile (= MMA M for S)
static_assert(TT == kStreamTile, "the stream form's positions are this kernel's tiles");
constexpr int HD = 128;                 // head_size of this path (= MMA M for O)
constexpr int TILE_BYTES = TT * HD * 2; // one K or V tile, 32 KB
constexpr int kSoftmaxThreads = 128;   // one softmax warpgroup
constexpr int kNoBlock = -2147483647 - 1;  // "no block here" marker of the producers
constexpr uint32_t kSoftmaxBar = 1;     // named barrier id of softmax group 0 (group 1: 2)
constexpr int kMaxCluster = 16;         // partitions merged inside one cluster, at most

// K stages recycle as soon as S = K q^T has run; V stages only after P V,
// which waits for the softmax, so V gets the deeper ring where shared memory
// allows only five stages.
__host__ __device__ constexpr int k_stages(int npad) { return npad <= 16 ? 3 : 2; }
__host__ __device__ constexpr int v_stages(int npad) { return npad <= 48 ? 3 : 2; }
// The NPAD columns of S and O (the query group padded to a multiple of 16)
// are split between NPAD / 16 softmax warpgroups of 16 columns each.
__host__ __device__ constexpr int sm_groups(int npad) { return npad / 16; }
__host__ __device__ constexpr int threads_of(int npad) { return 64 + 128 * sm_groups(npad) + 32; }
__host__ __device__ constexpr int tmem_cols(int npad) {
  return 4 * npad <= 32 ? 32 : 4 * npad <= 64 ? 64 : 4 * npad <= 128 ? 128 : 256;
}

template <int NPAD>
struct SmemLayout {
  static constexpr int NK = k_stages(NPAD);
  static constexpr int NV = v_stages(NPAD);
  static constexpr int QB = NPAD * HD * 2;   // one q (or P) buffer
  static constexpr int off_k = 0;
  static constexpr int off_v = off_k + NK * TILE_BYTES;
  static constexpr int off_q = off_v + NV * TILE_BYTES;
  static constexpr int off_p = off_q + 2 * QB;
  static constexpr int off_misc = off_p + 2 * QB;
  static constexpr int misc_bytes = 13824;
  static constexpr int bytes = off_misc + misc_bytes;
};

struct Misc {
  uint64_t k_full[3], k_empty[3], v_full[3], v_empty[3];
  uint64_t q_full[2], q_empty[2], s_full[2], p_full[2], o_full[2], drain;
  uint32_t tmem_base;
  int abort;
  int k_bad[3];                 // per K stage: token offset of the tile's first bad block id, or -1
  alignas(16) float red[2][4][64];   // per-warp tile maxima
  alignas(16) float m_run[2][64];    // reference maxima (log2 domain), per unit parity
  alignas(16) float alpha[2][64];    // rescale factor of each tile parity
  float lsum[4][64];            // per-warp exponent sums at finalisation
  alignas(16) float inv_l[64];       // 1 / sum (0 for a bad unit)
  alignas(16) float slope[2][64];    // ALiBi slopes of the unit's columns (log2 units)
  float sum_l[64];                   // sum written to the workspace
  SchedSmem sched;                   // work-unit schedule
};

static_assert(sizeof(Misc) <= SmemLayout<16>::misc_bytes, "misc area too small");

__device__ __forceinline__ void set_abort(Misc& ms, uint32_t* status) {
  ms.abort = 1;
  flag(status, PKD_DEV_TIMEOUT);
}

// Maximum over the 32 lanes of each of 16 per-lane values, by a butterfly
// that halves the values each step (16 shuffles instead of 80).  Lane l ends
// with the result for value (l >> 1) & 15.
__device__ __forceinline__ float warp_max16(const float (&v)[16], int lane) {
  float w8[8], w4[4], w2[2];
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    w8[i] = fmaxf(b4 ? v[8 + i] : v[i], __shfl_xor_sync(0xffffffffu, b4 ? v[i] : v[8 + i], 16));
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w4[i] = fmaxf(b3 ? w8[4 + i] : w8[i], __shfl_xor_sync(0xffffffffu, b3 ? w8[i] : w8[4 + i], 8));
#pragma unroll
  for (int i = 0; i < 2; ++i)
    w2[i] = fmaxf(b2 ? w4[2 + i] : w4[i], __shfl_xor_sync(0xffffffffu, b2 ? w4[i] : w4[2 + i], 4));
  float w1 = fmaxf(b1 ? w2[1] : w2[0], __shfl_xor_sync(0xffffffffu, b1 ? w2[0] : w2[1], 2));
  return fmaxf(w1, __shfl_xor_sync(0xffffffffu, w1, 1));
}

// Same butterfly for sums: lane l ends with the sum of value (l >> 1) & 15.
__device__ __forceinline__ float warp_sum16(const float (&v)[16], int lane) {
  float w8[8], w4[4], w2[2];
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    w8[i] = (b4 ? v[8 + i] : v[i]) + __shfl_xor_sync(0xffffffffu, b4 ? v[i] : v[8 + i], 16);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w4[i] = (b3 ? w8[4 + i] : w8[i]) + __shfl_xor_sync(0xffffffffu, b3 ? w8[i] : w8[4 + i], 8);
#pragma unroll
  for (int i = 0; i < 2; ++i)
    w2[i] = (b2 ? w4[2 + i] : w4[i]) + __shfl_xor_sync(0xffffffffu, b2 ? w4[i] : w4[2 + i], 4);
  float w1 = (b1 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? w2[0] : w2[1], 2);
  return w1 + __shfl_xor_sync(0xffffffffu, w1, 1);
}

template <bool BF16, int NPAD, int FORM>
__global__ void __launch_bounds__(threads_of(NPAD), 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap,
                     const __grid_constant__ CUtensorMap qmap, const DecodeArgs a) {
  using LY = SmemLayout<NPAD>;
  constexpr int NK = LY::NK, NV = LY::NV;
  constexpr int GROUPS = sm_groups(NPAD);
  constexpr int kThreads = threads_of(NPAD);
  constexpr int kVWarp = 2 + 4 * GROUPS;     // V producer (warp 0 produces K and q)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  uint8_t* kbuf = sm + LY::off_k;
  uint8_t* vbuf = sm + LY::off_v;
  uint8_t* qbuf = sm + LY::off_q;
  uint8_t* pbuf = sm + LY::off_p;
  Misc& ms = *reinterpret_cast<Misc*>(sm + LY::off_misc);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = a.num_heads / a.num_kv_heads;

  // ---------------------------------------------------------------- setup
  prefetch_schedule_inputs<FORM>(a);
  if (threadIdx.x == 0) {
    for (int i = 0; i < NK; ++i) {
      mbar_init(&ms.k_full[i], 1);
      mbar_init(&ms.k_empty[i], 1 + kSoftmaxThreads * GROUPS);
      ms.k_bad[i] = -1;
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(&ms.v_full[i], 1);
      mbar_init(&ms.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ms.q_full[i], 1);
      mbar_init(&ms.q_empty[i], 1);
      mbar_init(&ms.s_full[i], 1);
      mbar_init(&ms.p_full[i], kSoftmaxThreads * GROUPS);
      mbar_init(&ms.o_full[i], 1);
    }
    mbar_init(&ms.drain, 1);
    ms.abort = 0;
    fence_barrier_init();
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    tma_prefetch_desc(&qmap);
  }
  // P buffers start at zero: rows of padded heads are never written again.
  for (int i = threadIdx.x; i < 2 * LY::QB / 16; i += kThreads)
    reinterpret_cast<uint4*>(pbuf)[i] = make_uint4(0, 0, 0, 0);
  for (int i = threadIdx.x; i < 128; i += kThreads) ms.m_run[i >> 6][i & 63] = -INFINITY;
  if (warp == 1) {
    tmem_alloc(&ms.tmem_base, tmem_cols(NPAD));
    tmem_relinquish();
  }
  pdl_wait();
  pdl_launch_dependents();
  schedule_setup<FORM>(ms.sched, a, kThreads);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;

  if (warp == 0 || warp == kVWarp) {
    // ============================================================ producers
    const bool is_v = warp == kVWarp;
    const int B = a.block_size;
    const int R = B < TT ? B : TT;            // rows per TMA box
    const int nbox = TT / R;                  // boxes per tile and 64-column half
    const int oob_row = a.num_blocks * B;     // first row past the pool: zero fill
    const CUtensorMap* map = is_v ? &vmap : &kmap;
    uint8_t* ring = is_v ? vbuf : kbuf;
    const int nst = is_v ? NV : NK;
    uint64_t* full = is_v ? ms.v_full : ms.k_full;
    uint64_t* empty = is_v ? ms.v_empty : ms.k_empty;
    const uint64_t policy = policy_evict_first();
    const bool issuer = lane < 2 * nbox;      // lane issues box (lane % nbox) of half (lane / nbox)
    const int my_box = lane % nbox, my_half = lane / nbox;

    // Raw block id of box `lane` of tile tj (lanes < nbox), kNoBlock if the
    // box lies past the partition end.  The loaded value is first used one
    // tile later, so its latency hides behind the current tile's issue.
    auto load_raw = [&](const UnitInfo& t, int tj) {
      int raw = kNoBlock;
      if (lane < nbox) {
        const int ts = t.t0 + tj * TT;
        const int tok0 = B <= TT ? ts + lane * B : ts;
        if (tok0 < t.t1) raw = __ldg(a.block_tables + (size_t)t.s * a.max_blocks_per_seq + tok0 / B);
      }
      return raw;
    };
    UnitCursor cur = cursor_begin<FORM>(ms.sched, a);
    UnitInfo ui;
    bool have = cursor_next<TT, FORM>(cur, ms.sched, a, ui);
    int jl = 0;
    int raw = have ? load_raw(ui, 0) : kNoBlock;
    uint32_t jk = 0, un = 0;
    bool ok = true;
    while (have) {
      UnitInfo nui = ui;
      bool nhave = true;
      int njl = jl + 1;
      if (njl >= ui.ntiles) {
        nhave = cursor_next<TT, FORM>(cur, ms.sched, a, nui);
        njl = 0;
      }
      const int nraw = nhave ? load_raw(nui, njl) : kNoBlock;
      if (!is_v && jl == 0 && lane == 0) {
        const int qb = un & 1;
        ok = mbar_wait(&ms.q_empty[qb], ((un >> 1) & 1) ^ 1);
        if (ok) {
          mbar_arrive_expect_tx(&ms.q_full[qb], LY::QB);
          const int row0 = ui.s * a.num_heads + ui.hk * g;
          tma_load_2d(qbuf + qb * LY::QB, &qmap, &ms.q_full[qb], 0, row0);
          tma_load_2d(qbuf + qb * LY::QB + NPAD * 128, &qmap, &ms.q_full[qb], 64, row0);
        }
      }
      const int ts = ui.t0 + jl * TT;
      const bool bad = raw != kNoBlock && (raw < 0 || raw >= a.num_blocks);
      const int row = (raw != kNoBlock && !bad) ? raw * B + (B <= TT ? 0 : ts % B) : oob_row;
      const uint32_t bad_lanes = __ballot_sync(0xffffffffu, bad);   // lanes < nbox: boxes in token order
      const int st = jk % nst;
      if (lane == 0) {
        ok = ok && mbar_wait(&empty[st], ((jk / nst) & 1) ^ 1);
        if (ok) {
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
      if (issuer)
        tma_load_3d_hint(ring + st * TILE_BYTES + my_half * TT * 128 + my_box * R * 128, map,
                         &full[st], my_half * 64, ui.hk, r, policy);
      ++jk;
      if (njl == 0) ++un;
      have = nhave;
      ui = nui;
      jl = njl;
      raw = nraw;
    }
    if (!ok && lane == 0) {
      set_abort(ms, a.status);
      // Let armed loads land before the CTA can exit.
      for (uint32_t j = (jk >= (uint32_t)nst ? jk - nst : 0); j < jk; ++j)
        mbar_wait(&full[j % nst], (j / nst) & 1, 100000000ull);
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_f16(128, NPAD, BF16, false, false);
      const uint32_t id_o = idesc_f16(128, NPAD, BF16, true, false);
      const uint32_t kaddr = smem_u32(kbuf), vaddr = smem_u32(vbuf);
      const uint32_t qaddr = smem_u32(qbuf), paddr = smem_u32(pbuf);
      uint32_t j = 0, un = 0;
      int prev = -1;
      bool ok = true;
      auto issue_pv = [&](uint32_t jp) {
        const int vs = jp % NV, b = jp & 1;
        ok = ok && mbar_wait(&ms.v_full[vs], (jp / NV) & 1);
        ok = ok && mbar_wait(&ms.p_full[b], (jp >> 1) & 1);
        if (!ok) return;
        tc_fence_after();
        const uint32_t d = tmem + 2 * NPAD + b * NPAD;
#pragma unroll
        for (int k = 0; k < TT / 16; ++k) {
          const uint64_t ad = smem_desc(vaddr + vs * TILE_BYTES + k * 2048, TT * 128, 1024,
                                        kSwizzle128B);
          const uint64_t bd = smem_desc(paddr + b * LY::QB + (k >> 2) * NPAD * 128 + (k & 3) * 32,
                                        16, 1024, kSwizzle128B);
          mma_f16(d, ad, bd, id_o, k > 0);
        }
        mma_commit(&ms.o_full[b]);
        mma_commit(&ms.v_empty[vs]);
      };
      UnitCursor cur = cursor_begin<FORM>(ms.sched, a);
      UnitInfo ui;
      while (ok && cursor_next<TT, FORM>(cur, ms.sched, a, ui)) {
        // The softmax warps finish the previous unit only after its last P V:
        // issue that one before this unit's first S.
        if (prev >= 0) {
          issue_pv((uint32_t)prev);
          prev = -1;
        }
        const int qb = un & 1;
        ok = ok && mbar_wait(&ms.q_full[qb], (un >> 1) & 1);
        for (int jl = 0; jl < ui.ntiles && ok; ++jl, ++j) {
          const int ks = j % NK, b = j & 1;
          ok = mbar_wait(&ms.k_full[ks], (j / NK) & 1);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d = tmem + b * NPAD;
#pragma unroll
          for (int k = 0; k < HD / 16; ++k) {
            const uint64_t ad = smem_desc(kaddr + ks * TILE_BYTES + (k >> 2) * TT * 128 + (k & 3) * 32,
                                          16, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(qaddr + qb * LY::QB + (k >> 2) * NPAD * 128 + (k & 3) * 32,
                                          16, 1024, kSwizzle128B);
            mma_f16(d, ad, bd, id_s, k > 0);
          }
          mma_commit(&ms.s_full[b]);
          mma_commit(&ms.k_empty[ks]);
          if (jl == ui.ntiles - 1) mma_commit(&ms.q_empty[qb]);
          if (prev >= 0) issue_pv((uint32_t)prev);
          prev = (int)j;
        }
        ++un;
      }
      if (ok && prev >= 0) issue_pv((uint32_t)prev);
      if (!ok) set_abort(ms, a.status);
      // Drain: every MMA issued above has completed once this arrives.
      mma_commit(&ms.drain);
      mbar_wait(&ms.drain, 0, 100000000ull);
    }
    __syncwarp();
  } else {
    // ============================================================ softmax / epilogue
    // Softmax warpgroup grp handles the 16 columns [hbase, hbase + 16) of
    // S and O (query heads of the group): their probabilities, P rows, O
    // columns and output rows, with its own
    // named barrier.  Columns are independent, so the warpgroups never wait
    // for each other.
    //
    // Reference maxima: the exponentials of a tile use the running reference
    // m_run of each column, p = 2^(x - m_run).  A tile only moves m_run
    // (cross-thread maxima, rescale factor alpha, a second barrier) when one
    // of its logits passes m_run + kHeadroom, which after the first tile of
    // a unit is rare, so p stays below 2^kHeadroom and the result is the
    // same softmax.  Padded columns hold m_run = +inf: their p is 0 and they
    // never ask for a rescale.
    constexpr int HPG = 16;
    constexpr float kHeadroom = 8.f;
    static_assert(NPAD == HPG * GROUPS, "one softmax warpgroup per 16 columns");
    const int grp = (warp - 2) >> 2;
    const int hbase = grp * HPG;
    const uint32_t bar = kSoftmaxBar + grp;
    const int et = threadIdx.x - 64 - kSoftmaxThreads * grp;   // thread within the warpgroup
    const bool leader = et == 0;
    const int wq = warp & 3;                   // TMEM lane quadrant of this warp
    const int row = wq * 32 + lane;            // token row of S, d row of O
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    const float qscale = a.scale * kLog2e;
    const bool single = a.num_partitions == 1;
    const bool fused = form_fused<FORM>(a);    // one unit, merged over the cluster
    const int H = a.num_heads;
    const int group_heads = max(0, min(HPG, g - hbase));    // decode: valid heads of this warpgroup
    // This thread's element (column hbase + hl, token row) of the K-major,
    // 128-byte swizzled P^T operand sits at p_row ^ ((hl & 7) << 4), plus
    // hl * 128: the swizzle XORs the 16-byte chunk index ((row & 63) >> 3)
    // with the row's index mod 8, hbase is a multiple of 16, and bits 4..6
    // of everything else are zero.
    const uint32_t p_row = (uint32_t)((row >> 6) * NPAD * 128 + hbase * 128 +
                                      (((row & 63) >> 3) << 4) + ((row & 7) << 1));
    float o_acc[HPG], l_part[HPG];
#pragma unroll
    for (int h = 0; h < HPG; ++h) o_acc[h] = l_part[h] = 0.f;
    uint32_t j = 0;
    uint32_t resc = 0;     // bit (tile & 1): that tile moved m_run (factors in ms.alpha)
    bool ok = true;

    // o += (the tile's P V), rescaled first when the tile moved m_run.
    auto accumulate_o = [&](uint32_t jo) {
      const int b = jo & 1;
      ok = ok && mbar_wait(&ms.o_full[b], (jo >> 1) & 1);
      if (!ok) return;
      tc_fence_after();
      float v[HPG];
      tmem_ld16(lane_addr + 2 * NPAD + b * NPAD + hbase, v);
      if ((resc >> b) & 1) {
#pragma unroll
        for (int i = 0; i < HPG; i += 4) {
          const float4 al = *reinterpret_cast<const float4*>(&ms.alpha[b][hbase + i]);
          o_acc[i] = fmaf(o_acc[i], al.x, v[i]);
          o_acc[i + 1] = fmaf(o_acc[i + 1], al.y, v[i + 1]);
          o_acc[i + 2] = fmaf(o_acc[i + 2], al.z, v[i + 2]);
          o_acc[i + 3] = fmaf(o_acc[i + 3], al.w, v[i + 3]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < HPG; ++i) o_acc[i] += v[i];
      }
      tc_fence_before();
    };

    UnitCursor cur = cursor_begin<FORM>(ms.sched, a);
    UnitInfo ui, nx;
    const bool alibi = a.alibi != nullptr;
    // Per-unit state of this warpgroup's columns in buffer ub: reference
    // maxima (-inf; +inf for padded columns) and ALiBi slopes.  The next
    // unit's is written before the current unit's last barrier, so units
    // need no barrier of their own to start.
    auto setup_unit = [&](const UnitInfo& v, int ub) {
      if (et < HPG) {
        const int c = hbase + et;
        ms.m_run[ub][c] = et < group_heads ? -INFINITY : INFINITY;
        if (alibi && et < group_heads) ms.slope[ub][c] = a.alibi[v.hk * g + c] * kLog2e;
      }
    };
    bool have = cursor_next<TT, FORM>(cur, ms.sched, a, ui);
    if (have) setup_unit(ui, 0);
    named_barrier(bar, kSoftmaxThreads);
    uint32_t u = 0;                    // units done by this warpgroup
    while (ok && have) {
      const int ub = u & 1;
      const int h0 = ui.hk * g;
      const int my_heads = group_heads;   // valid columns of this warpgroup
      float* const m_run = ms.m_run[ub];
      const float* const slope = ms.slope[ub];
      bool unit_bad = false;
      // Every wait below is bounded; a thread that gives up keeps taking part
      // in the group barriers, which combine the flag so the group stops together.
      for (int jl = 0; jl < ui.ntiles; ++jl, ++j) {
        const int b = j & 1, ks = j % NK, vs = j % NV;
        const int ts = ui.t0 + jl * TT;
        const bool valid = ts + row < ui.t1;
        ok = ok && mbar_wait(&ms.s_full[b], (j >> 1) & 1);
        ok = ok && mbar_wait(&ms.k_full[ks], (j / NK) & 1);
        tc_fence_after();
        unit_bad |= ms.k_bad[ks] >= 0;
        mbar_arrive(&ms.k_empty[ks]);
        // Logits of the tile in log2 units (masked: -inf).
        float xs[HPG];
        tmem_ld16(lane_addr + b * NPAD + hbase, xs);
        if (alibi) {
          const float pos = (float)(ts + row - (ui.L - 1));   // ALiBi distance to the query
#pragma unroll
          for (int i = 0; i < HPG; i += 4) {
            const float4 sl = *reinterpret_cast<const float4*>(&slope[hbase + i]);
            xs[i] = valid ? fmaf(sl.x, pos, xs[i] * qscale) : -INFINITY;
            xs[i + 1] = valid ? fmaf(sl.y, pos, xs[i + 1] * qscale) : -INFINITY;
            xs[i + 2] = valid ? fmaf(sl.z, pos, xs[i + 2] * qscale) : -INFINITY;
            xs[i + 3] = valid ? fmaf(sl.w, pos, xs[i + 3] * qscale) : -INFINITY;
          }
        } else if (ts + TT <= ui.t1) {           // every row of the tile is attended
#pragma unroll
          for (int i = 0; i < HPG; ++i) xs[i] *= qscale;
        } else {
#pragma unroll
          for (int i = 0; i < HPG; ++i) xs[i] = valid ? xs[i] * qscale : -INFINITY;
        }
        // Does a logit pass its column's reference by more than the headroom?
        float over = -INFINITY;
#pragma unroll
        for (int i = 0; i < HPG; i += 4) {
          const float4 mr = *reinterpret_cast<const float4*>(&m_run[hbase + i]);
          over = fmaxf(over, fmaxf(fmaxf(xs[i] - mr.x, xs[i + 1] - mr.y),
                                   fmaxf(xs[i + 2] - mr.z, xs[i + 3] - mr.w)));
        }
        if (named_barrier_or(bar, kSoftmaxThreads, over > kHeadroom || !ok)) {
          // Rare: move the references to the tile maxima (or stop together).
          ok = named_barrier_and(bar, kSoftmaxThreads, ok);
          if (!ok) break;
          const float m = warp_max16(xs, lane);
          if ((lane & 1) == 0) ms.red[b][wq][hbase + ((lane >> 1) & 15)] = m;
          named_barrier(bar, kSoftmaxThreads);
          if (et < my_heads) {
            const int h = hbase + et;
            const float mt = fmaxf(fmaxf(ms.red[b][0][h], ms.red[b][1][h]),
                                   fmaxf(ms.red[b][2][h], ms.red[b][3][h]));
            const float m_old = m_run[h];
            const float m_new = fmaxf(m_old, mt);
            ms.alpha[b][h] = m_new == -INFINITY ? 1.f : fast_exp2(m_old - m_new);
            m_run[h] = m_new;
          } else if (et < HPG) {
            ms.alpha[b][hbase + et] = 1.f;
          }
          named_barrier(bar, kSoftmaxThreads);
#pragma unroll
          for (int i = 0; i < HPG; i += 4) {
            const float4 al = *reinterpret_cast<const float4*>(&ms.alpha[b][hbase + i]);
            l_part[i] *= al.x;
            l_part[i + 1] *= al.y;
            l_part[i + 2] *= al.z;
            l_part[i + 3] *= al.w;
          }
          resc |= 1u << b;
        } else {
          resc &= ~(1u << b);
        }
        // Probabilities: written 16-bit into the P^T operand, summed per thread.
        const uint32_t pb = smem_u32(pbuf + b * LY::QB) + p_row;
#pragma unroll
        for (int i = 0; i < HPG; i += 2) {
          const float2 mr = *reinterpret_cast<const float2*>(&m_run[hbase + i]);
          const float p0 = fast_exp2(xs[i] - mr.x);       // 0 for masked rows and padded columns
          const float p1 = fast_exp2(xs[i + 1] - mr.y);
          l_part[i] += p0;
          l_part[i + 1] += p1;
          const uint32_t pk = pack2<BF16>(p0, p1);
          if (i < my_heads) st_shared_u16((pb ^ ((i & 7) << 4)) + i * 128, (uint16_t)pk);
          if (i + 1 < my_heads)
            st_shared_u16((pb ^ (((i + 1) & 7) << 4)) + (i + 1) * 128, (uint16_t)(pk >> 16));
        }
        // Cache slots past the sequence end inside a loaded block may hold
        // anything (NaN included): zero those V rows before P V reads them.
        // (Warpgroup 0 does it; the others' arrivals on p_full come after
        // theirs, and P V waits for all of them.)
        if (ts + TT > ui.L && grp == 0) {
          ok = ok && mbar_wait(&ms.v_full[vs], (j / NV) & 1);
          if (ok && ts + row >= ui.L) {
            uint4* v0 = reinterpret_cast<uint4*>(vbuf + vs * TILE_BYTES + row * 128);
            uint4* v1 = reinterpret_cast<uint4*>(vbuf + vs * TILE_BYTES + TT * 128 + row * 128);
#pragma unroll
            for (int i = 0; i < 8; ++i) v0[i] = v1[i] = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&ms.p_full[b]);
        if (jl > 0) accumulate_o(j - 1);
        if (jl == ui.ntiles - 1) accumulate_o(j);
      }
      // ---------------------------------------------------------- finalise unit
      // The warpgroup's P rows are idle now (the unit's last P V has
      // completed): four pieces of 16 x 128 bytes (2 buffers x 2 slabs) that
      // stage a cluster partial, 4 whole fp32 rows per piece.
      auto piece = [&](int q) { return pbuf + (q >> 1) * LY::QB + (q & 1) * NPAD * 128 + hbase * 128; };
      // Workspace or cluster partial (unnormalised), or a whole result.  In
      // the stream form a unit cut by the CTA's range edge is a partial in
      // its slot; every other unit is whole.
      const bool partial = form_stream<FORM>(a) ? ui.slot >= 0 : !single;
      const size_t unit_row =
          form_stream<FORM>(a) ? (size_t)ui.slot * g
                   : (((size_t)ui.s * a.num_kv_heads + ui.hk) * a.num_partitions + ui.p) * g;
      if (partial) {
        if (fused) {
#pragma unroll
          for (int hl = 0; hl < HPG; ++hl)
            if (hl < my_heads) reinterpret_cast<float*>(piece(hl >> 2))[(hl & 3) * HD + row] = o_acc[hl];
        } else {
          // Workspace rows straight from registers: a warp writes 128
          // consecutive bytes of a row per store.
          float* const wo = a.ws_o + (unit_row + hbase) * HD + row;
#pragma unroll
          for (int hl = 0; hl < HPG; ++hl)
            if (hl < my_heads) wo[hl * HD] = o_acc[hl];
        }
      }
      const bool have_next = cursor_next<TT, FORM>(cur, ms.sched, a, nx);
      if (have_next) setup_unit(nx, ub ^ 1);
      {
        const float t = warp_sum16(l_part, lane);
        if ((lane & 1) == 0) ms.lsum[wq][hbase + ((lane >> 1) & 15)] = t;
      }
      ok = named_barrier_and(bar, kSoftmaxThreads, ok);
      if (!ok) break;
      if (partial) {
        if (et < my_heads) {
          const int h = hbase + et;
          const float den = ms.lsum[0][h] + ms.lsum[1][h] + ms.lsum[2][h] + ms.lsum[3][h];
          const float l = unit_bad ? -1.f : den;        // < 0 marks a bad block
          if (fused) {
            ms.sum_l[h] = l;
          } else {
            a.ws_m[unit_row + h] = m_run[h];
            a.ws_l[unit_row + h] = l;
          }
        }
        if (fused) break;   // the cluster merge reads the staged partial
      } else {
        if (et < my_heads) {
          const int h = hbase + et;
          const float den = ms.lsum[0][h] + ms.lsum[1][h] + ms.lsum[2][h] + ms.lsum[3][h];
          ms.inv_l[h] = unit_bad || den == 0.f ? 0.f : 1.f / den;
        }
        named_barrier(bar, kSoftmaxThreads);
        // Output rows straight from registers: a warp writes 64 consecutive
        // bytes of a row per store.
        uint16_t* const dst = reinterpret_cast<uint16_t*>(a.out) + ((size_t)ui.s * H + h0 + hbase) * HD + row;
#pragma unroll
        for (int hl = 0; hl < HPG; ++hl)
          if (hl < my_heads) dst[hl * HD] = (uint16_t)pack2<BF16>(o_acc[hl] * ms.inv_l[hbase + hl], 0.f);
      }
#pragma unroll
      for (int h = 0; h < HPG; ++h) o_acc[h] = l_part[h] = 0.f;
      ui = nx;
      have = have_next;
      ++u;
    }
    if (!ok && leader) set_abort(ms, a.status);
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols(NPAD));
  }

  // ---------------------------------------------------------------- cluster merge
  // Fused split context: the CTAs of the cluster are the partitions of one
  // (sequence, KV head), and each has left its partial in shared memory: the
  // unnormalised o rows (fp32, in its P buffers), the maxima m (log2 domain)
  // and the sums l (negative for a bad block).  Heads are dealt round-robin
  // to the ranks; a warp merges one head, each lane 4 columns of d:
  //     M = max_p m_p,  w_p = 2^(m_p - M),  out = sum_p w_p o_p / sum_p w_p l_p.
  if (form_fused<FORM>(a)) {
    cluster_sync();
    constexpr int HPG = NPAD / GROUPS, PER = HPG / 4;   // staging: PER rows per piece
    const int P = a.num_partitions;
    const uint32_t rank = cluster_ctarank();
    const int s = blockIdx.y / a.num_kv_heads;
    const int hk = blockIdx.y - s * a.num_kv_heads;
    const int L = a.context_lens[s];
    const int np = parts_of(a, L);
    if (rank == 0 && hk == 0 && threadIdx.x == 0 &&
        !len_ok(L, a.max_context_len, a.max_blocks_per_seq, a.block_size))
      flag(a.status, PKD_DEV_BAD_LEN);
    for (int h = (int)rank + P * warp; h < g; h += P * (kThreads / 32)) {
      const int grp = h / HPG, hl = h - grp * HPG, q = hl / PER;
      const uint8_t* row = pbuf + (q >> 1) * LY::QB + (q & 1) * NPAD * 128 + grp * HPG * 128 +
                           (hl - q * PER) * HD * 4 + lane * 16;
      float m[kMaxCluster], l[kMaxCluster];
      float M = -INFINITY;
      bool bad = false;
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r) {
        if (r < np) {
          m[r] = ld_dsmem(dsmem_addr(&ms.m_run[0][h], r));
          l[r] = ld_dsmem(dsmem_addr(&ms.sum_l[h], r));
          M = fmaxf(M, m[r]);
          bad |= l[r] < 0.f;
        }
      }
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      float den = 0.f;
      if (!bad && M != -INFINITY) {
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) {
          if (r < np) {
            const float w = exp2f(m[r] - M);
            const float4 o = ld_dsmem4(dsmem_addr(row, r));
            den = fmaf(w, l[r], den);
            acc.x = fmaf(w, o.x, acc.x);
            acc.y = fmaf(w, o.y, acc.y);
            acc.z = fmaf(w, o.z, acc.z);
            acc.w = fmaf(w, o.w, acc.w);
          }
        }
      }
      const float inv = den > 0.f ? 1.f / den : 0.f;
      uint2 v;
      v.x = pack2<BF16>(acc.x * inv, acc.y * inv);
      v.y = pack2<BF16>(acc.z * inv, acc.w * inv);
      const size_t orow = (size_t)s * a.num_heads + (size_t)hk * g + h;
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + orow * HD + lane * 4) = v;
    }
    cluster_sync();   // every rank's shared memory stays until all have read it
  }
}

// ---------------------------------------------------------------- host side

int pad_group(int g) { return (g + 15) / 16 * 16; }

// Kernel attributes, set once per device: the dynamic shared memory and
// clusters of up to 16 CTAs.
template <bool BF16, int NPAD, int FORM>
cudaError_t prepare(int* smem_out) {
  const int smem = SmemLayout<NPAD>::bytes + 1024;
  *smem_out = smem;
  static std::atomic<bool> attr_set[64];   // setting it twice from two threads is harmless
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || attr_set[dev].load(std::memory_order_acquire)) return cudaSuccess;
  if ((e = cudaFuncSetAttribute(decode_tc_kernel<BF16, NPAD, FORM>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(decode_tc_kernel<BF16, NPAD, FORM>,
                                cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
    return e;
  attr_set[dev].store(true, std::memory_order_release);
  return cudaSuccess;
}

void cluster_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute (&attr)[2], dim3 grid,
                    int threads, int smem, int cluster, cudaStream_t st) {
  *cfg = {};
  cfg->gridDim = grid;
  cfg->blockDim = dim3(threads);
  cfg->dynamicSmemBytes = smem;
  cfg->stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg->attrs = attr;
  cfg->numAttrs = 2;
}

template <bool BF16, int NPAD>
cudaError_t launch_t(const DecodeArgs& a, cudaStream_t st) {
  CUtensorMap km, vm, qm;
  const long long rows = (long long)a.num_blocks * a.block_size;
  const int box_rows = a.block_size < TT ? a.block_size : TT;
  if (!make_kv_map(&km, a.key_cache, BF16, HD, a.num_kv_heads, rows, 64, box_rows, true) ||
      !make_kv_map(&vm, a.value_cache, BF16, HD, a.num_kv_heads, rows, 64, box_rows, true) ||
      !make_rows_map(&qm, a.q, BF16, HD, (long long)a.num_seqs * a.num_heads, 64, NPAD))
    return cudaErrorInvalidValue;
  int smem = 0;
  cudaError_t e;
  if (a.fused) {
    // One cluster of P CTAs per (sequence, KV head).
    if ((e = prepare<BF16, NPAD, kFormCluster>(&smem)) != cudaSuccess) return e;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    cluster_config(&cfg, attr, dim3(a.num_partitions, a.num_seqs * a.num_kv_heads),
                   threads_of(NPAD), smem, a.num_partitions, st);
    return cudaLaunchKernelEx(&cfg, decode_tc_kernel<BF16, NPAD, kFormCluster>, km, vm, qm, a);
  }
  if (a.stream) {
    if ((e = prepare<BF16, NPAD, kFormStream>(&smem)) != cudaSuccess) return e;
    return launch_pdl(decode_tc_kernel<BF16, NPAD, kFormStream>, dim3(a.stream_ctas),
                      dim3(threads_of(NPAD)), smem, st, km, vm, qm, a);
  }
  if ((e = prepare<BF16, NPAD, kFormPlain>(&smem)) != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long units = (long long)a.num_seqs * a.num_kv_heads * a.num_partitions;
  const int grid = (int)(units < sms ? units : sms);
  return launch_pdl(decode_tc_kernel<BF16, NPAD, kFormPlain>, dim3(grid), dim3(threads_of(NPAD)),
                    smem, st, km, vm, qm, a);
}

// Co-resident clusters of `cluster` CTAs, cached per device and cluster size.
template <int NPAD>
int capacity_t(int cluster) {
  static std::atomic<int> cache[64][kMaxCluster + 1];   // value + 1; 0 = not yet queried
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::atomic<int>& c = cache[dev][cluster];
  if (c.load(std::memory_order_relaxed) == 0) {
    int smem = 0, n = 0;
    if (prepare<true, NPAD, kFormCluster>(&smem) == cudaSuccess) {
      cudaLaunchConfig_t cfg;
      cudaLaunchAttribute attr[2];
      cluster_config(&cfg, attr, dim3(cluster), threads_of(NPAD), smem, cluster, nullptr);
      if (cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel<true, NPAD, kFormCluster>, &cfg) !=
          cudaSuccess) {
        cudaGetLastError();   // a refused query only means "no cluster launch"
        n = 0;
      }
    }
    c.store(n + 1, std::memory_order_relaxed);
  }
  return c.load(std::memory_order_relaxed) - 1;
}

template <bool BF16>
cudaError_t launch_b(const DecodeArgs& a, cudaStream_t st) {
  switch (pad_group(a.num_heads / a.num_kv_heads)) {
    case 16: return launch_t<BF16, 16>(a, st);
    case 32: return launch_t<BF16, 32>(a, st);
    case 48: return launch_t<BF16, 48>(a, st);
    case 64: return launch_t<BF16, 64>(a, st);
  }
  return cudaErrorNotSupported;
}

}  // namespace

bool decode_tc_supported(int head_size, int group, int block_size) {
  return head_size == HD && group >= 4 && group <= 64 && block_size >= 8 && tma_available();
}

int decode_tc_tile() { return TT; }
int decode_tc_sched_max() { return kSchedMax; }

int decode_tc_cluster_capacity(int group, int cluster) {
  if (cluster < 2 || cluster > kMaxCluster || group < 4 || group > 64) return 0;
  switch (pad_group(group)) {
    case 16: return capacity_t<16>(cluster);
    case 32: return capacity_t<32>(cluster);
    case 48: return capacity_t<48>(cluster);
    case 64: return capacity_t<64>(cluster);
  }
  return 0;
}

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t st) {
  return a.is_bf16 ? launch_b<true>(a, st) : launch_b<false>(a, st);
}

}  // namespace pkd
