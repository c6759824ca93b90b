// C ABI of the library (declared in include/pkd.h): argument validation,
// launch planning and dispatch.  Allocates nothing and never synchronises.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/pkd.h"
#include "internal.h"

namespace {

thread_local char g_last_error[256] = "";

pkd_status cuda_fail(cudaError_t e, const char* what) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", what, cudaGetErrorName(e),
                cudaGetErrorString(e));
  return PKD_ERR_CUDA;
}

}  // namespace

namespace pkd {
pkd_status record_cuda_error(cudaError_t e, const char* what) { return cuda_fail(e, what); }
}  // namespace pkd

namespace {

struct DeviceInfo {
  int sms = 0;
  int major = 0;
  int minor = 0;
};

// Per-device attributes, queried once per device and cached (the first
// query is made under a lock; later calls read the cache after an acquire
// load of its ready flag).
pkd_status device_info(DeviceInfo* out) {
  static DeviceInfo cache[64];
  static std::atomic<bool> ready[64];
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return PKD_ERR_DEVICE;
  if (!ready[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(mu);
    if (!ready[dev].load(std::memory_order_relaxed)) {
      DeviceInfo n;
      if ((e = cudaDeviceGetAttribute(&n.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
          (e = cudaDeviceGetAttribute(&n.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
          (e = cudaDeviceGetAttribute(&n.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute");
      cache[dev] = n;
      ready[dev].store(true, std::memory_order_release);
    }
  }
  const DeviceInfo& d = cache[dev];
  *out = d;
  if (d.major != 10 || d.minor != 3) return PKD_ERR_DEVICE;  // built for sm_103a only
  return PKD_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool pow2_in(int v, int lo, int hi) { return v >= lo && v <= hi && (v & (v - 1)) == 0; }

constexpr int kPartitionQuantum = 64;   // partitions are whole 64-token tiles
constexpr int kTargetCtasPerSm = 2;     // split until about this many CTAs per SM

constexpr int kMaxCluster = 16;         // partitions merged inside one cluster, at most
constexpr double kClusterMergeCost = 0.5;   // in-cluster merge, in tiles

struct Plan {
  int partition_size = kPartitionQuantum;
  int num_partitions = 1;
  int path = PKD_PATH_SIMT;
  bool fused = false;                   // tensor-core split merged inside clusters
  int stream_ctas = 0;                  // > 0: tensor-core stream form on that many CTAs
  size_t ws_bytes = 0;
  size_t off_m = 0, off_l = 0, off_desc = 0;
};

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

pkd_status check_decode_sizes(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                              int max_context_len) {
  if (num_seqs < 1 || num_seqs > 65535 || num_heads < 1 || num_kv_heads < 1 ||
      max_context_len < 0)
    return PKD_ERR_SHAPE;
  if (num_heads % num_kv_heads != 0) return PKD_ERR_SHAPE;
  if (num_kv_heads * (num_heads / num_kv_heads) > 65535) return PKD_ERR_SHAPE;
  if (head_size != 64 && head_size != 128) return PKD_ERR_UNSUPPORTED;
  return PKD_OK;
}

// Tiles-per-CTA estimate of the persistent tensor-core kernel for P
// partitions: CTAs take units round-robin, so the busiest CTA handles
// ceil(units * P / ctas) units of ceil(tiles / P) tiles; each unit costs about
// a quarter tile of fixed work and a split adds the merge launch.
double tc_cost(long long units, int tiles, int P, int ctas) {
  const long long per_cta = (units * P + ctas - 1) / ctas;
  const int tiles_per_unit = (tiles + P - 1) / P;
  return (double)per_cta * tiles_per_unit + 0.25 * per_cta + (P > 1 ? 2.0 : 0.0);
}

// A split into P partitions is merged inside thread-block clusters (one
// cluster of P CTAs per (sequence, KV head), no workspace, no merge launch)
// when all the clusters fit on the device at once.
bool cluster_fits(long long units, int group, int P) {
  if (P < 2 || P > kMaxCluster || units > 65535) return false;
  const int cap = pkd::decode_tc_cluster_capacity(group, P);
  return cap > 0 && units <= cap;
}

double tc_cluster_cost(int tiles, int P) {
  return (double)((tiles + P - 1) / P) + 0.25 + kClusterMergeCost;
}

// Stream form: every CTA takes an equal share of all tiles, at most two more
// units than units / ctas (its range edges), and a merge launch follows.
double tc_stream_cost(long long units, int tiles, int ctas) {
  return (double)units * tiles / ctas + 0.25 * ((double)units / ctas + 2.0) + 2.0;
}

// The stream form builds its tile prefix in shared memory (at most 1024
// sequences) and counts tiles in 32-bit integers.
bool stream_fits(int num_seqs, int num_kv_heads, int max_tiles) {
  return num_seqs <= pkd::decode_tc_sched_max() &&
         (long long)num_seqs * num_kv_heads * (max_tiles + pkd::kStreamTailCost) < (1LL << 30);
}

pkd_status make_plan(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                     int max_context_len, int block_size, int partition_size, Plan* plan) {
  pkd_status st = check_decode_sizes(num_seqs, num_heads, num_kv_heads, head_size, max_context_len);
  if (st != PKD_OK) return st;
  if (partition_size < PKD_PARTITION_STREAM) return PKD_ERR_SHAPE;
  DeviceInfo dev;
  if ((st = device_info(&dev)) != PKD_OK) return st;
  const int g = num_heads / num_kv_heads;
  Plan p;
  const int tc_tile = pkd::decode_tc_tile();
  const bool tc = pkd::decode_tc_supported(head_size, g, block_size) &&
                  (partition_size <= 0 || partition_size % tc_tile == 0);
  p.path = tc ? PKD_PATH_TC : PKD_PATH_SIMT;
  const int quantum = tc ? tc_tile : kPartitionQuantum;
  const int max_tiles = std::max(1, (max_context_len + quantum - 1) / quantum);
  const long long units = (long long)num_seqs * num_kv_heads;
  bool stream = false;
  if (partition_size == PKD_PARTITION_STREAM) {
    if (!tc || !stream_fits(num_seqs, num_kv_heads, max_tiles)) return PKD_ERR_UNSUPPORTED;
    stream = true;
  } else if (partition_size > 0) {
    if (partition_size % kPartitionQuantum) return PKD_ERR_SHAPE;
    p.partition_size = partition_size;
  } else if (tc) {
    int best = 1;
    double best_cost = tc_cost(units, max_tiles, 1, dev.sms);
    for (int P = 2; P <= max_tiles && P <= 64; ++P) {
      const double c = cluster_fits(units, g, P) ? tc_cluster_cost(max_tiles, P)
                                                 : tc_cost(units, max_tiles, P, dev.sms);
      if (c < best_cost * 0.97) {
        best_cost = c;
        best = P;
      }
    }
    p.partition_size = ((max_tiles + best - 1) / best) * quantum;
    stream = stream_fits(num_seqs, num_kv_heads, max_tiles) &&
             tc_stream_cost(units, max_tiles, dev.sms) < best_cost * 0.97;
  } else {
    const long long units = (long long)num_seqs * num_kv_heads * (g / pkd::simt_heads_per_cta(g));
    const long long target = (long long)kTargetCtasPerSm * dev.sms;
    long long parts = units >= target ? 1 : (target + units - 1) / units;
    parts = std::min<long long>(parts, max_tiles);
    const int tiles = (int)((max_tiles + parts - 1) / parts);
    p.partition_size = tiles * quantum;
  }
  if (stream) {
    // One tile per partition in the prefix; 2 partial slots and one
    // range-edge descriptor per CTA.
    p.partition_size = pkd::kStreamTile;
    p.num_partitions = 1;
    p.stream_ctas = dev.sms;
    const size_t rows = (size_t)2 * dev.sms * g;
    p.off_m = align256(rows * head_size * sizeof(float));
    p.off_l = p.off_m + align256(rows * sizeof(float));
    p.off_desc = p.off_l + align256(rows * sizeof(float));
    p.ws_bytes = p.off_desc + align256((size_t)dev.sms * sizeof(int4));
    *plan = p;
    return PKD_OK;
  }
  p.num_partitions = std::max(1, (max_context_len + p.partition_size - 1) / p.partition_size);
  if (p.num_partitions > 65535) return PKD_ERR_SHAPE;
  p.fused = tc && cluster_fits((long long)num_seqs * num_kv_heads, g, p.num_partitions);
  if (p.num_partitions > 1 && !p.fused) {
    const size_t rows = (size_t)num_seqs * num_heads * p.num_partitions;
    p.off_m = align256(rows * head_size * sizeof(float));
    p.off_l = p.off_m + align256(rows * sizeof(float));
    p.ws_bytes = p.off_l + align256(rows * sizeof(float));
  }
  *plan = p;
  return PKD_OK;
}

}  // namespace

extern "C" {

pkd_status pkd_decode_plan(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                           int block_size, int max_context_len, int partition_size,
                           int* out_partition_size, int* out_num_partitions, int* out_path,
                           size_t* out_workspace_bytes) {
  if (!pow2_in(block_size, 8, 256)) return PKD_ERR_UNSUPPORTED;
  Plan p;
  pkd_status st = make_plan(num_seqs, num_heads, num_kv_heads, head_size, max_context_len,
                            block_size, partition_size, &p);
  if (st != PKD_OK) return st;
  if (out_partition_size) *out_partition_size = p.partition_size;
  if (out_num_partitions) *out_num_partitions = p.num_partitions;
  if (out_path)
    *out_path = p.fused ? PKD_PATH_TC_CLUSTER : p.stream_ctas > 0 ? PKD_PATH_TC_STREAM : p.path;
  if (out_workspace_bytes) *out_workspace_bytes = p.ws_bytes;
  return PKD_OK;
}

size_t pkd_decode_workspace_bytes(int num_seqs, int num_heads, int head_size,
                                  int max_context_len) {
  // The largest workspace of the library's own plan (partition_size 0) over
  // every KV-head count (a divisor of num_heads) and block size.
  size_t worst = 0;
  bool any = false;
  for (int hk = 1; hk <= num_heads; ++hk) {
    if (num_heads % hk) continue;
    for (int bs = 8; bs <= 256; bs *= 2) {
      Plan p;
      if (make_plan(num_seqs, num_heads, hk, head_size, max_context_len, bs, 0, &p) != PKD_OK)
        continue;
      any = true;
      worst = std::max(worst, p.ws_bytes);
    }
  }
  return any ? worst : 0;
}

pkd_status pkd_paged_decode_attention(void* out, const void* q, const void* key_cache,
                                      const void* value_cache, const int32_t* block_tables,
                                      int max_blocks_per_seq, const int32_t* context_lens,
                                      int max_context_len, int num_seqs, int num_heads,
                                      int num_kv_heads, int head_size, int block_size,
                                      int num_blocks, float scale, pkd_dtype dtype,
                                      int partition_size, void* workspace,
                                      size_t workspace_bytes, uint32_t* device_status,
                                      void* stream) {
  return pkd_paged_decode_attention_ex(out, q, key_cache, value_cache, block_tables,
                                       max_blocks_per_seq, context_lens, max_context_len, num_seqs,
                                       num_heads, num_kv_heads, head_size, block_size, num_blocks,
                                       scale, nullptr, dtype, partition_size, workspace,
                                       workspace_bytes, device_status, stream);
}

pkd_status pkd_paged_decode_attention_ex(void* out, const void* q, const void* key_cache,
                                         const void* value_cache, const int32_t* block_tables,
                                         int max_blocks_per_seq, const int32_t* context_lens,
                                         int max_context_len, int num_seqs, int num_heads,
                                         int num_kv_heads, int head_size, int block_size,
                                         int num_blocks, float scale, const float* alibi_slopes,
                                         pkd_dtype dtype, int partition_size, void* workspace,
                                         size_t workspace_bytes, uint32_t* device_status,
                                         void* stream) {
  if (!out || !q || !key_cache || !value_cache || !block_tables || !context_lens)
    return PKD_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(alibi_slopes) & 3u) != 0) return PKD_ERR_ALIGN;
  if (dtype != PKD_FP16 && dtype != PKD_BF16) return PKD_ERR_UNSUPPORTED;
  if (!pow2_in(block_size, 8, 256)) return PKD_ERR_UNSUPPORTED;
  if (num_blocks < 1 || max_blocks_per_seq < 1) return PKD_ERR_SHAPE;
  if ((long long)num_blocks * block_size > 0x7fffffffLL) return PKD_ERR_SHAPE;
  if ((long long)max_blocks_per_seq * block_size > 0x7fff0000LL) return PKD_ERR_SHAPE;
  if (!aligned16(out) || !aligned16(q) || !aligned16(key_cache) || !aligned16(value_cache))
    return PKD_ERR_ALIGN;
  Plan plan;
  pkd_status st = make_plan(num_seqs, num_heads, num_kv_heads, head_size, max_context_len,
                            block_size, partition_size, &plan);
  if (st != PKD_OK) return st;
  if (plan.ws_bytes > 0) {
    if (!workspace || workspace_bytes < plan.ws_bytes) return PKD_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PKD_ERR_ALIGN;
  }

  pkd::DecodeArgs a = {};
  a.out = out;
  a.q = q;
  a.key_cache = key_cache;
  a.value_cache = value_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.max_context_len = max_context_len;
  a.num_seqs = num_seqs;
  a.num_heads = num_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_size = head_size;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.scale = scale;
  a.alibi = alibi_slopes;
  a.is_bf16 = dtype == PKD_BF16;
  a.partition_size = plan.partition_size;
  a.num_partitions = plan.num_partitions;
  a.fused = plan.fused ? 1 : 0;
  a.stream = plan.stream_ctas > 0 ? 1 : 0;
  a.stream_ctas = plan.stream_ctas;
  char* ws = static_cast<char*>(workspace);
  const bool use_ws = plan.ws_bytes > 0;
  a.ws_o = use_ws ? reinterpret_cast<float*>(ws) : nullptr;
  a.ws_m = use_ws ? reinterpret_cast<float*>(ws + plan.off_m) : nullptr;
  a.ws_l = use_ws ? reinterpret_cast<float*>(ws + plan.off_l) : nullptr;
  a.ws_desc = a.stream ? reinterpret_cast<int4*>(ws + plan.off_desc) : nullptr;
  a.status = device_status;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = plan.path == PKD_PATH_TC ? pkd::launch_decode_tc(a, s) : pkd::launch_decode_simt(a, s);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  if (a.stream) {
    e = pkd::launch_stream_merge(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "stream merge launch");
  } else if (use_ws) {
    e = pkd::launch_lse_reduce(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "lse_reduce launch");
  }
  return PKD_OK;
}

pkd_status pkd_selftest_bounded_wait(uint32_t* device_status, long long limit_ns, void* stream) {
  if (!device_status) return PKD_ERR_NULL;
  if (limit_ns < 1000 || limit_ns > 1000000000LL) return PKD_ERR_SHAPE;
  DeviceInfo dev;
  pkd_status st = device_info(&dev);
  if (st != PKD_OK) return st;
  cudaError_t e = pkd::launch_selftest_wait(device_status, limit_ns, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKD_OK : cuda_fail(e, "self-test launch");
}

pkd_status pkd_paged_prefill_attention(void* out, const void* q, const void* key_cache,
                                       const void* value_cache, const int32_t* block_tables,
                                       int max_blocks_per_seq, const int32_t* context_lens,
                                       const int32_t* query_start, int num_query_tokens,
                                       int max_query_len, int max_context_len, int num_seqs,
                                       int num_heads, int num_kv_heads, int head_size,
                                       int block_size, int num_blocks, float scale,
                                       const float* alibi_slopes, pkd_dtype dtype,
                                       uint32_t* device_status, void* stream) {
  if (!out || !q || !key_cache || !value_cache || !block_tables || !context_lens || !query_start)
    return PKD_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(alibi_slopes) & 3u) != 0) return PKD_ERR_ALIGN;
  if (dtype != PKD_FP16 && dtype != PKD_BF16) return PKD_ERR_UNSUPPORTED;
  if (!pow2_in(block_size, 8, 256)) return PKD_ERR_UNSUPPORTED;
  pkd_status st = check_decode_sizes(num_seqs, num_heads, num_kv_heads, head_size, max_context_len);
  if (st != PKD_OK) return st;
  const int g = num_heads / num_kv_heads;
  if (head_size != 128 || g > 64) return PKD_ERR_UNSUPPORTED;
  if (num_query_tokens < 0 || max_query_len < 0 || num_blocks < 1 || max_blocks_per_seq < 1)
    return PKD_ERR_SHAPE;
  if ((long long)num_blocks * block_size > 0x7fffffffLL) return PKD_ERR_SHAPE;
  if ((long long)max_blocks_per_seq * block_size > 0x7fff0000LL) return PKD_ERR_SHAPE;
  if ((long long)num_query_tokens * num_heads > 0x7fffffffLL) return PKD_ERR_SHAPE;
  if (!aligned16(out) || !aligned16(q) || !aligned16(key_cache) || !aligned16(value_cache))
    return PKD_ERR_ALIGN;
  DeviceInfo dev;
  if ((st = device_info(&dev)) != PKD_OK) return st;
  if (!pkd::tma_available()) return PKD_ERR_UNSUPPORTED;
  if (num_query_tokens == 0 || max_query_len == 0) return PKD_OK;   // no query rows

  const int qt = pkd::prefill_rows_queries_per_unit(g);
  const long long tiles = ((long long)max_query_len + qt - 1) / qt;
  if (tiles > 65535) return PKD_ERR_SHAPE;
  pkd::DecodeArgs a = {};
  a.out = out;
  a.q = q;
  a.key_cache = key_cache;
  a.value_cache = value_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.max_context_len = max_context_len;
  a.num_seqs = num_seqs;
  a.num_heads = num_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_size = head_size;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.scale = scale;
  a.alibi = alibi_slopes;
  a.is_bf16 = dtype == PKD_BF16;
  a.partition_size = max_context_len;   // unused by prefill: one range per query tile
  a.num_partitions = (int)tiles;        // query tiles per sequence, at most
  a.query_start = query_start;
  a.q_per_unit = qt;
  a.max_query_len = max_query_len;
  a.num_q_tokens = num_query_tokens;
  a.status = device_status;
  cudaError_t e = pkd::launch_prefill_rows(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKD_OK : cuda_fail(e, "prefill launch");
}

static pkd_status copy_common(const void* a, const void* b, const void* c, const void* d,
                              const int64_t* slots, int num_tokens, int num_heads, int head_size,
                              int block_size, int num_blocks, pkd_dtype dtype) {
  if (num_tokens < 0 || num_heads < 1 || head_size < 8 || head_size % 8 || block_size < 1 ||
      num_blocks < 1)
    return PKD_ERR_SHAPE;
  if (dtype != PKD_FP16 && dtype != PKD_BF16) return PKD_ERR_UNSUPPORTED;
  if ((long long)num_heads * head_size > 0x7fffffffLL / 2) return PKD_ERR_SHAPE;
  if (num_tokens == 0) return PKD_OK;
  if (!a || !b || !c || !d || !slots) return PKD_ERR_NULL;
  if (!aligned16(a) || !aligned16(b) || !aligned16(c) || !aligned16(d)) return PKD_ERR_ALIGN;
  DeviceInfo dev;
  return device_info(&dev);
}

pkd_status pkd_gather_cached_kv(void* key_out, void* value_out, const void* key_cache,
                                const void* value_cache, const int64_t* slot_mapping,
                                int num_tokens, int num_heads, int head_size, int block_size,
                                int num_blocks, pkd_dtype dtype, uint32_t* device_status,
                                void* stream) {
  pkd_status st = copy_common(key_out, value_out, key_cache, value_cache, slot_mapping, num_tokens,
                              num_heads, head_size, block_size, num_blocks, dtype);
  if (st != PKD_OK || num_tokens == 0) return st;
  pkd::CopyArgs a{key_out, value_out, key_cache, value_cache, slot_mapping, num_tokens,
                  num_heads * head_size, block_size, num_blocks, device_status};
  cudaError_t e = pkd::launch_gather(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKD_OK : cuda_fail(e, "gather launch");
}

pkd_status pkd_reshape_and_cache(const void* key, const void* value, void* key_cache,
                                 void* value_cache, const int64_t* slot_mapping, int num_tokens,
                                 int num_heads, int head_size, int block_size, int num_blocks,
                                 pkd_dtype dtype, uint32_t* device_status, void* stream) {
  pkd_status st = copy_common(key_cache, value_cache, key, value, slot_mapping, num_tokens,
                              num_heads, head_size, block_size, num_blocks, dtype);
  if (st != PKD_OK || num_tokens == 0) return st;
  pkd::CopyArgs a{key_cache, value_cache, key, value, slot_mapping, num_tokens,
                  num_heads * head_size, block_size, num_blocks, device_status};
  cudaError_t e = pkd::launch_scatter(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKD_OK : cuda_fail(e, "reshape_and_cache launch");
}

const char* pkd_status_string(pkd_status status) {
  switch (status) {
    case PKD_OK: return "ok";
    case PKD_ERR_NULL: return "a required pointer is NULL";
    case PKD_ERR_SHAPE: return "sizes inconsistent or out of range";
    case PKD_ERR_UNSUPPORTED: return "head_size, block_size or dtype not supported";
    case PKD_ERR_WORKSPACE: return "workspace missing or too small";
    case PKD_ERR_ALIGN: return "a tensor pointer is not 16-byte aligned (workspace: 256)";
    case PKD_ERR_CUDA: return "a CUDA call or launch failed";
    case PKD_ERR_DEVICE: return "current device is not an sm_103 GPU";
  }
  return "unknown status";
}

const char* pkd_last_error(void) { return g_last_error; }

int pkd_version(void) { return 100; }

}  // extern "C"
