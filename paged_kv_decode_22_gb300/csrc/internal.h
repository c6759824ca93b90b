// Internal host-side interface between the C ABI (api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/pkd.h"

namespace pkd {

// Records a failed CUDA call for pkd_last_error() on this host thread and
// returns PKD_ERR_CUDA.
pkd_status record_cuda_error(cudaError_t e, const char* what);

// Launch with programmatic stream serialization (see pdl_wait in common.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Arguments of one decode-attention launch, already validated on the host.
// Stream form: a (sequence, KV head) pair whose last tile is partial counts
// this many more positions in the tile list than it has tiles -- what ending
// such a unit costs, in tile times (its last P V waits for a V tile that
// lands late) -- so that CTAs whose share ends more of them take fewer tiles.
constexpr int kStreamTailCost = 2;
constexpr int kStreamTile = 128;   // tokens per tile of the stream form (its partition size)

struct DecodeArgs {
  void* out;
  const void* q;
  const void* key_cache;
  const void* value_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int max_blocks_per_seq;
  int max_context_len;
  int num_seqs;
  int num_heads;
  int num_kv_heads;
  int head_size;
  int block_size;
  int num_blocks;
  float scale;
  const float* alibi;   // [num_heads] ALiBi slopes, or nullptr
  int is_bf16;
  int partition_size;   // tokens per partition (multiple of 64)
  int num_partitions;   // 1 = write `out` directly
  int fused;            // tensor-core path only: the partitions of one (sequence,
                        // KV head) form one thread-block cluster and are merged
                        // through distributed shared memory (no workspace)
  int stream;           // tensor-core path only: CTA b takes positions [T b / G, T (b + 1) / G)
                        // of the list of all (sequence, KV head) pairs in order, each pair
                        // its tiles then, when its last tile is partial, kStreamTailCost
                        // empty positions (partition_size = 128, num_partitions = 1); a
                        // unit cut by a range edge leaves a partial in slot 2b (the pair
                        // began before the CTA's range) or 2b + 1 (it begins inside)
  int stream_ctas;      // stream: G, the grid size
  int4* ws_desc;        // stream: [G] the (sequence, KV head) cut by the left edge of CTA
                        // b's range, written by CTA b: {position A of its first tile, tiles n,
                        // s * Hk + hk, total positions T}; n = 0 when no pair is cut there
  const int32_t* query_start;   // prefill: [S + 1] cumulative chunk lengths (nullptr: decode)
  int q_per_unit;       // prefill: query tokens per work unit
  // prefill: the grid stride gridDim.x written as (ds * Hk + dhk) * per + dr,
  // per the units per (sequence, KV head) of the launched kernel (set by the
  // launch, so that a CTA's walk over its units needs no division)
  int walk_dr, walk_dhk, walk_ds;
  int max_query_len;    // prefill: longer chunks are invalid (zero rows)
  int num_q_tokens;     // prefill: rows of q and out (query_start[S])
  float* ws_o;          // [S][Hk][P][H/Hk][D] unnormalised partial outputs
  float* ws_m;          // [S][Hk][P][H/Hk] partial maxima (log2 domain)
  float* ws_l;          // [S][Hk][P][H/Hk] partial sums; < 0 marks a bad block
  uint32_t* status;
};

struct CopyArgs {
  void* dst_k;
  void* dst_v;
  const void* src_k;
  const void* src_v;
  const int64_t* slots;
  int num_tokens;
  int row_elems;    // num_heads * head_size
  int block_size;
  int num_blocks;
  uint32_t* status;
};

// TMA tensor maps (tmap.cu).  KV map: 3-D {head_size, num_kv_heads, rows}
// over a cache viewed as [rows][num_kv_heads][head_size]; rows map: 2-D
// {cols, rows}, 128-byte swizzle.
bool tma_available();
bool make_kv_map(CUtensorMap* map, const void* cache, bool bf16, int head_size, int num_kv_heads,
                 long long rows, int box_cols, int box_rows, bool swizzle128);
bool make_rows_map(CUtensorMap* map, const void* base, bool bf16, int cols, long long rows,
                   int box_cols, int box_rows);
// Query chunks: 3-D {head_size, num_heads, tokens} over q [tokens][H][D],
// box {64, box_heads, box_tokens}, 128-byte swizzle.
bool make_q_chunk_map(CUtensorMap* map, const void* q, bool bf16, int head_size, int num_heads,
                      long long tokens, int box_heads, int box_tokens);

cudaError_t launch_decode_simt(const DecodeArgs& a, cudaStream_t st);
int simt_heads_per_cta(int group);
cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t st);
bool decode_tc_supported(int head_size, int group, int block_size);
int decode_tc_tile();
int decode_tc_sched_max();   // sequences the in-kernel tile prefix holds
// Clusters of `cluster` CTAs of the tensor-core kernel for query-group size
// `group` that the current device holds at once (0: cannot launch).
int decode_tc_cluster_capacity(int group, int cluster);
// Prefill on the row-per-thread tensor-core kernel (128 (query, head) rows
// per unit, S and O in TMEM): query tokens per unit and the launch.
int prefill_rows_queries_per_unit(int group);
cudaError_t launch_prefill_rows(const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_lse_reduce(const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_stream_merge(const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_gather(const CopyArgs& a, cudaStream_t st);
cudaError_t launch_selftest_wait(uint32_t* status, long long limit_ns, cudaStream_t st);
cudaError_t launch_scatter(const CopyArgs& a, cudaStream_t st);

}  // namespace pkd
