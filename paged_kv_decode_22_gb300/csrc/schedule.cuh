// Work units of the persistent decode kernels and their schedule.
//
// A unit is (sequence s, KV head, context partition p): the tokens
// [p * partition_size, min((p + 1) * partition_size, L_s)) of one KV head,
// processed in tiles of TT tokens.  With at most kSchedMax sequences every
// CTA builds, in shared memory, the per-sequence count of non-empty units
// and their prefix sum, numbers the non-empty units densely (sequence, then
// KV head, then partition) and takes an equal contiguous range of them, so
// empty partitions of short sequences cost nothing and the load is even.
// With more sequences CTAs take units round-robin and skip the empty ones.
// In the cluster form of the tensor-core kernel each CTA takes the single
// unit its grid position names (x = partition, y = sequence * Hk + KV head).
// In the stream form the prefix counts positions -- each (sequence, KV
// head) pair's 128-token tiles, followed by kStreamTailCost empty positions
// when its last tile is partial -- and CTA b takes the positions
// [T b / G, T (b + 1) / G): a unit is the run of its tiles inside one pair,
// and only a CTA's first and last units can be cut short (partials in slots
// 2b and 2b + 1).
#pragma once

#include "common.cuh"
#include "internal.h"

namespace pkd {

constexpr int kSchedMax = 1024;

// The split-context form of a decode launch: read from the arguments at run
// time, or fixed by a kernel instantiation, so that an instantiation holds
// only its own form's code (a kernel's instruction footprint is part of a
// short call's time).
constexpr int kFormRuntime = -1, kFormPlain = 0, kFormCluster = 1, kFormStream = 2;
template <int FORM>
__device__ __forceinline__ bool form_stream(const DecodeArgs& a) {
  return FORM == kFormRuntime ? a.stream != 0 : FORM == kFormStream;
}
template <int FORM>
__device__ __forceinline__ bool form_fused(const DecodeArgs& a) {
  return FORM == kFormRuntime ? a.fused != 0 : FORM == kFormCluster;
}

struct SchedSmem {
  int total;
  int L[kSchedMax];        // context length of each sequence
  int pre[kSchedMax + 1];  // units (stream: positions) of the sequences before s
  // Stream form: this CTA's range [next, end) of the tile list and the
  // (sequence, KV head, offset, positions per pair) of its first tile,
  // found once by the set-up for every role's cursor.
  int start[6];            // next, end, s, hk, off, np
};

struct UnitInfo {
  int s, hk, p, L, t0, t1, ntiles;
  bool lok;
  int slot;   // stream form: workspace slot of a partial unit, -1 for a whole one
  // Prefill (its own schedule) only: the unit's queries are chunk queries
  // [p * QT, p * QT + nq) of sequence s, stored from packed row qrow0 on;
  // the first sits at position pos0, query c at pos0 + c.
  int qrow0, nq, pos0;
};

// Stream form: empty positions after each pair of a sequence of length L.
__device__ __forceinline__ int stream_pad(int L) {
  return L % kStreamTile ? kStreamTailCost : 0;
}

__device__ __forceinline__ int parts_of(const DecodeArgs& a, int L) {
  return (len_ok(L, a.max_context_len, a.max_blocks_per_seq, a.block_size) && L > 0)
             ? (L + a.partition_size - 1) / a.partition_size
             : 0;
}

template <int TT>
__device__ __forceinline__ UnitInfo unit_info(const DecodeArgs& a, int u) {
  UnitInfo ui;
  const int P = a.num_partitions;
  ui.p = u % P;
  const int sh = u / P;
  ui.hk = sh % a.num_kv_heads;
  ui.s = sh / a.num_kv_heads;
  ui.slot = -1;
  ui.L = a.context_lens[ui.s];
  ui.lok = len_ok(ui.L, a.max_context_len, a.max_blocks_per_seq, a.block_size);
  ui.t0 = ui.p * a.partition_size;
  ui.t1 = min(ui.t0 + a.partition_size, ui.L);
  ui.ntiles = (ui.lok && ui.t0 < ui.L) ? (ui.t1 - ui.t0 + TT - 1) / TT : 0;
  return ui;
}

struct UnitCursor {
  long long next, end;
  bool dense;
  int s, hk, p, np;   // dense: position of the last unit returned (np < 0: none yet);
                      // stream: position of the next tile (np = positions per pair of s)
};

template <int FORM = kFormRuntime>
__device__ __forceinline__ UnitCursor cursor_begin(const SchedSmem& sc, const DecodeArgs& a) {
  UnitCursor c;
  c.dense = !form_fused<FORM>(a) && a.num_seqs <= kSchedMax;
  c.s = c.hk = c.p = 0;
  c.np = -1;
  if (form_stream<FORM>(a)) {
    // Stream form: an equal contiguous range of the sequence-major tile
    // list, starting on the tile the set-up found.
    c.next = sc.start[0];
    c.end = sc.start[1];
    c.s = sc.start[2];
    c.hk = sc.start[3];
    c.p = sc.start[4];
    c.np = sc.start[5];
  } else if (form_fused<FORM>(a)) {
    // Cluster launch: grid (P, S * Hk), one unit per CTA, partition = x.
    c.next = (long long)blockIdx.y * a.num_partitions + blockIdx.x;
    c.end = c.next + 1;
  } else if (c.dense) {
    const long long total = sc.total;
    c.next = total * blockIdx.x / gridDim.x;
    c.end = total * (blockIdx.x + 1) / gridDim.x;
  } else {
    c.next = blockIdx.x;
    c.end = (long long)a.num_seqs * a.num_kv_heads * a.num_partitions;
  }
  return c;
}

template <int TT, int FORM = kFormRuntime>
__device__ __forceinline__ bool cursor_next(UnitCursor& c, const SchedSmem& sc,
                                            const DecodeArgs& a, UnitInfo& ui) {
  if (form_stream<FORM>(a)) {
    // Units are the runs of the CTA's range over one pair's tiles; np =
    // positions per pair of sequence s (its tiles and empty positions).
    while (c.next < c.end) {
      if (c.np < 0) {
        const int t = (int)c.next;
        int lo = 0, hi = a.num_seqs - 1;   // last s with pre[s] <= t
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (sc.pre[mid] <= t) lo = mid; else hi = mid - 1;
        }
        c.s = lo;
        c.np = (sc.pre[lo + 1] - sc.pre[lo]) / a.num_kv_heads;
        const int r = t - sc.pre[lo];
        c.hk = r / c.np;
        c.p = r - c.hk * c.np;
      }
      const int nt = c.np - stream_pad(sc.L[c.s]);   // tiles of the pair
      const int off = c.p;
      if (off < nt) {
        const int n = (int)min((long long)(nt - off), c.end - c.next);
        ui.s = c.s;
        ui.hk = c.hk;
        ui.p = 0;
        ui.L = sc.L[c.s];
        ui.lok = true;
        ui.t0 = off * TT;
        ui.t1 = min(ui.L, (off + n) * TT);
        ui.ntiles = n;
        // A cut pair that began before the range is its first unit (slot
        // 2b); one that begins inside runs past the range end (2b + 1).
        ui.slot = (off > 0 || off + n < nt)
                      ? 2 * (int)blockIdx.x +
                            (c.next - off >= (long long)sc.total * blockIdx.x / gridDim.x)
                      : -1;
        c.next += n;
        c.p += n;
        return true;
      }
      // The pair's empty positions: step to the next pair.
      c.next += c.np - off;
      if (c.next < c.end) {
        c.p = 0;
        if (++c.hk == a.num_kv_heads) {
          c.hk = 0;
          do { ++c.s; } while (sc.pre[c.s + 1] == sc.pre[c.s]);
          c.np = (sc.pre[c.s + 1] - sc.pre[c.s]) / a.num_kv_heads;
        }
      }
    }
    return false;
  }
  if (c.dense) {
    if (c.next >= c.end) return false;
    const int j = (int)c.next++;
    if (c.np < 0) {
      // First unit: binary search for the last s with pre[s] <= j.
      int lo = 0, hi = a.num_seqs - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sc.pre[mid] <= j) lo = mid; else hi = mid - 1;
      }
      c.s = lo;
      c.np = (sc.pre[lo + 1] - sc.pre[lo]) / a.num_kv_heads;   // units per KV head
      const int r = j - sc.pre[lo];
      c.hk = r / c.np;
      c.p = r - c.hk * c.np;
    } else if (++c.p == c.np) {
      // Later units follow in (sequence, KV head, partition) order; sequences
      // without units have pre[s + 1] == pre[s] and are stepped over.
      c.p = 0;
      if (++c.hk == a.num_kv_heads) {
        c.hk = 0;
        do { ++c.s; } while (sc.pre[c.s + 1] == sc.pre[c.s]);
        c.np = (sc.pre[c.s + 1] - sc.pre[c.s]) / a.num_kv_heads;
      }
    }
    ui.s = c.s;
    ui.L = sc.L[c.s];
    ui.hk = c.hk;
    ui.p = c.p;
    ui.lok = true;
    ui.t0 = ui.p * a.partition_size;
    ui.t1 = min(ui.t0 + a.partition_size, ui.L);
    ui.ntiles = (ui.t1 - ui.t0 + TT - 1) / TT;
    return true;
  }
  while (c.next < c.end) {
    ui = unit_info<TT>(a, (int)c.next);
    c.next += gridDim.x;
    if (ui.ntiles) return true;
  }
  return false;
}

// L2 prefetch, issued before pdl_wait(), of what a persistent kernel reads
// first: the context lengths (all of them when every CTA builds the
// schedule, else a share) and, in the persistent forms, the used head of
// every block-table row (ceil(max_context_len / block_size) entries), row s
// by CTA s mod G; in the cluster form the CTA's own length and partition.
template <int FORM = kFormRuntime>
__device__ __forceinline__ void prefetch_schedule_inputs(const DecodeArgs& a) {
  const int S = a.num_seqs, B = a.block_size, mbps = a.max_blocks_per_seq;
  if (form_fused<FORM>(a)) {
    const int s = blockIdx.y / a.num_kv_heads;
    const long long b0 = (long long)blockIdx.x * a.partition_size / B;
    prefetch_l2_lines(a.context_lens + s, 4, 0, 1, 1);
    if (b0 < mbps) {
      const long long nb = min((long long)(a.partition_size + B - 1) / B + 1, (long long)mbps - b0);
      prefetch_l2_lines(a.block_tables + (size_t)s * mbps + b0, (size_t)nb * 4, 0, 1, 64);
    }
    return;
  }
  if (S <= kSchedMax)
    prefetch_l2_lines(a.context_lens, (size_t)S * 4, 0, 1, 64);
  else
    prefetch_l2_lines(a.context_lens, (size_t)S * 4, blockIdx.x, gridDim.x, 64);
  if (a.query_start) prefetch_l2_lines(a.query_start, (size_t)(S + 1) * 4, 0, 1, 64);
  const long long used = min((long long)mbps, ((long long)a.max_context_len + B - 1) / B);
  for (int s = blockIdx.x; s < S; s += gridDim.x)
    prefetch_l2_lines(a.block_tables + (size_t)s * mbps, (size_t)used * 4, 0, 1, 1024);
}

// Build the schedule (when dense) and zero the output rows of sequences that
// have nothing to attend to (unsplit plans; the merge writes them when
// split), setting the length status bit for invalid lengths.  Every thread
// of the CTA calls this; it ends with __syncthreads().
template <int FORM = kFormRuntime>
__device__ __forceinline__ void schedule_setup(SchedSmem& sc, const DecodeArgs& a, int nthreads) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (form_fused<FORM>(a)) {   // one unit per CTA; the cluster merge handles empty sequences
    __syncthreads();
    return;
  }
  if (a.num_seqs <= kSchedMax) {
    for (int i = threadIdx.x; i < a.num_seqs; i += nthreads) {
      const int L = a.context_lens[i];
      sc.L[i] = L;
      const int n = parts_of(a, L);
      sc.pre[i + 1] = (form_stream<FORM>(a) && n > 0 ? n + stream_pad(L) : n) * a.num_kv_heads;
    }
    __syncthreads();
    if (warp == 0) {
      int carry = 0;
      for (int base = 0; base < a.num_seqs; base += 32) {
        int v = base + lane < a.num_seqs ? sc.pre[base + lane + 1] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int n = __shfl_up_sync(0xffffffffu, v, o);
          if (lane >= o) v += n;
        }
        if (base + lane < a.num_seqs) sc.pre[base + lane + 1] = v + carry;
        carry += __shfl_sync(0xffffffffu, v, 31);
      }
      if (lane == 0) {
        sc.pre[0] = 0;
        sc.total = carry;
      }
    }
    if (form_stream<FORM>(a) && warp == 0) {
      // This CTA's range of the tile list and its first tile, for every
      // role's cursor, and the pair cut by the range's left edge, for the
      // merge launch (warp 0 wrote the prefix).
      __syncwarp();
      if (lane == 0) {
        const long long T = sc.total;
        const int t = (int)(T * blockIdx.x / gridDim.x);
        const int te = (int)(T * (blockIdx.x + 1) / gridDim.x);
        int lo = 0, np = 1, hk = 0, off = 0;
        if (t < T) {
          int hi = a.num_seqs - 1;   // last s with pre[s] <= t (a sequence with entries)
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (sc.pre[mid] <= t) lo = mid; else hi = mid - 1;
          }
          np = (sc.pre[lo + 1] - sc.pre[lo]) / a.num_kv_heads;
          const int r = t - sc.pre[lo];
          hk = r / np;
          off = r - hk * np;
        }
        sc.start[0] = t;
        sc.start[1] = te;
        sc.start[2] = lo;
        sc.start[3] = hk;
        sc.start[4] = off;
        sc.start[5] = np;
        int4 d = make_int4(0, 0, 0, (int)T);
        if (blockIdx.x > 0 && t < T) {
          const int nt = np - stream_pad(sc.L[lo]);
          if (off > 0 && off < nt)   // inside the pair's tiles
            d = make_int4(sc.pre[lo] + hk * np, nt, lo * a.num_kv_heads + hk, (int)T);
        }
        a.ws_desc[blockIdx.x] = d;
      }
    }
  }
  for (int sq = blockIdx.x; sq < a.num_seqs; sq += gridDim.x) {
    const int L = a.num_seqs <= kSchedMax ? sc.L[sq] : a.context_lens[sq];
    if (parts_of(a, L) == 0) {
      if (!len_ok(L, a.max_context_len, a.max_blocks_per_seq, a.block_size) && threadIdx.x == 0)
        flag(a.status, PKD_DEV_BAD_LEN);
      if (a.num_partitions == 1) {
        uint32_t* o = reinterpret_cast<uint32_t*>(a.out) + (size_t)sq * a.num_heads * a.head_size / 2;
        for (int i = threadIdx.x; i < a.num_heads * a.head_size / 2; i += nthreads) o[i] = 0u;
      }
    }
  }
  __syncthreads();
}

}  // namespace pkd
