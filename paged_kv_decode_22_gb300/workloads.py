"""Seeded synthetic inputs for paged decode attention and gather_cached_kv.

This module only draws random numbers and stores them in the 16-bit formats
the kernels read.  It holds none of the attention or gather arithmetic: both
the CUDA path (through the tests and the bench) and the CPU oracle receive the
arrays built here, and neither side imports the other.

Workload shapes follow the vLLM pull-request pages the library is built from:
the kernel-latency tables of "[Performance] Support MQA/GQA in decode phase by
using FlashAttention" (64 query / 8 KV heads, bf16, context 1024 and 4096,
batch 1..256), the gather table of "Memcpy kernel for flash attention"
(40 heads, head_size 128, block_size 8, 1024 blocks, fp16, 64..2048 tokens),
the LLaMA-13B latency run of "Optimizes the single_query_cached_kv_attention
kernel" (batch 8, fp16) and the StarCoder run of "Optimize MQA Kernel"
(48 query heads sharing 1 KV head).

Value recipe: q, K and V are N(0, 1) float32 draws rounded to nearest-even
into fp16 or bf16.  Physical block ids are a seeded permutation of the pool,
so no two sequences share a block.  With ``poison=True`` every cache slot no
sequence references (unused blocks, the tail of each last block) holds NaN,
and block-table padding holds -1, so a kernel that reads them is caught.
Large pools copy windows of a 16 Mi-value table of normal draws at seeded
random offsets (one window per block) instead of drawing every value.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "f32_to_bf16_bits", "f32_to_f16_bits", "DecodeCase", "GatherCase", "PrefillCase",
    "make_decode_case", "make_gather_case", "make_prefill_case", "decode_configs",
    "gather_sweep", "prefill_configs", "NAN_BITS",
]

# Quiet-NaN bit patterns used to poison memory that no sequence references.
NAN_BITS = {"fp16": np.uint16(0x7E00), "bf16": np.uint16(0x7FC0)}

_TABLE_VALUES = 1 << 24  # size of the normal-draw table used for big pools


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    nan = (u & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
    r = np.where(nan, np.uint32(0x7FC0), r)
    return r.astype(np.uint16)


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to IEEE half (nearest, ties to even); return bits."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def _to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    if dtype == "fp16":
        return f32_to_f16_bits(x)
    raise ValueError(f"unknown dtype {dtype!r}")


def _normal_bits(rng: np.random.Generator, n: int, dtype: str) -> np.ndarray:
    return _to_bits(rng.standard_normal(n, dtype=np.float32), dtype)


def _pool_bits(rng, num_blocks: int, block_elems: int, dtype: str) -> np.ndarray:
    """[num_blocks, block_elems] 16-bit normal values."""
    total = num_blocks * block_elems
    if total <= _TABLE_VALUES:
        return _normal_bits(rng, total, dtype).reshape(num_blocks, block_elems)
    table = _normal_bits(rng, _TABLE_VALUES, dtype)
    table = np.concatenate([table, table[:block_elems]])
    windows = np.lib.stride_tricks.sliding_window_view(table, block_elems)
    starts = rng.integers(0, _TABLE_VALUES, size=num_blocks)
    return windows[starts]


@dataclass
class DecodeCase:
    """Inputs of one paged decode-attention call (host arrays, 16-bit bits)."""
    name: str
    dtype: str                 # "fp16" or "bf16"
    q: np.ndarray              # uint16 [S, H, D]
    key_cache: np.ndarray      # uint16 [NB, B, Hk, D]
    value_cache: np.ndarray    # uint16 [NB, B, Hk, D]
    block_tables: np.ndarray   # int32 [S, MB]
    context_lens: np.ndarray   # int32 [S]
    scale: float
    num_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    num_blocks: int
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.q.shape[0])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.context_lens.size else 0

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])


def make_decode_case(*, seed: int, num_seqs: int, num_heads: int, num_kv_heads: int,
                     head_size: int, block_size: int, num_blocks: int, context_lens,
                     dtype: str, poison: bool = True, scale: float | None = None,
                     max_blocks_per_seq: int | None = None, name: str = "") -> DecodeCase:
    """Build a seeded paged decode-attention case.

    ``context_lens`` is a sequence of per-sequence lengths.  Each sequence gets
    ceil(L / block_size) distinct physical blocks taken in order from one
    seeded permutation of the pool.
    """
    rng = np.random.default_rng(seed)
    lens = np.asarray(context_lens, dtype=np.int64).reshape(num_seqs)
    need = -(-lens // block_size)
    if need.sum() > num_blocks:
        raise ValueError(f"pool of {num_blocks} blocks too small for {int(need.sum())}")
    mb = int(max_blocks_per_seq or max(1, int(need.max(initial=1))))
    perm = rng.permutation(num_blocks).astype(np.int32)
    tables = np.full((num_seqs, mb), -1 if poison else 0, dtype=np.int32)
    pos = 0
    for s in range(num_seqs):
        n = int(need[s])
        tables[s, :n] = perm[pos:pos + n]
        pos += n

    q = _normal_bits(rng, num_seqs * num_heads * head_size, dtype).reshape(
        num_seqs, num_heads, head_size)
    block_elems = block_size * num_kv_heads * head_size
    kc = _pool_bits(rng, num_blocks, block_elems, dtype)
    vc = _pool_bits(rng, num_blocks, block_elems, dtype)
    shape = (num_blocks, block_size, num_kv_heads, head_size)
    kc = kc.reshape(shape)
    vc = vc.reshape(shape)
    if poison:
        used = np.zeros(num_blocks, dtype=bool)
        used[perm[:pos]] = True
        nanb = NAN_BITS[dtype]
        kc[~used] = nanb
        vc[~used] = nanb
        for s in range(num_seqs):
            n, L = int(need[s]), int(lens[s])
            if n and L % block_size:
                last = tables[s, n - 1]
                kc[last, L % block_size:] = nanb
                vc[last, L % block_size:] = nanb
    return DecodeCase(
        name=name or f"decode_s{num_seqs}_h{num_heads}_{num_kv_heads}",
        dtype=dtype, q=q, key_cache=kc, value_cache=vc, block_tables=tables,
        context_lens=lens.astype(np.int32),
        scale=float(scale if scale is not None else 1.0 / np.sqrt(head_size)),
        num_heads=num_heads, num_kv_heads=num_kv_heads, head_size=head_size,
        block_size=block_size, num_blocks=num_blocks, meta={"seed": seed})


@dataclass
class GatherCase:
    """Inputs of one gather_cached_kv call."""
    name: str
    dtype: str
    key_cache: np.ndarray      # uint16 [NB, B, H, D]
    value_cache: np.ndarray
    slot_mapping: np.ndarray   # int64 [T]
    num_heads: int
    head_size: int
    block_size: int
    num_blocks: int

    @property
    def num_tokens(self) -> int:
        return int(self.slot_mapping.shape[0])


def make_gather_case(*, seed: int, num_tokens: int, num_heads: int, head_size: int,
                     block_size: int, num_blocks: int, dtype: str, name: str = "") -> GatherCase:
    """Random pool plus ``num_tokens`` distinct slots drawn from it."""
    rng = np.random.default_rng(seed)
    nslots = num_blocks * block_size
    if num_tokens > nslots:
        raise ValueError("more tokens than slots")
    slots = rng.choice(nslots, size=num_tokens, replace=False).astype(np.int64)
    block_elems = block_size * num_heads * head_size
    shape = (num_blocks, block_size, num_heads, head_size)
    kc = _pool_bits(rng, num_blocks, block_elems, dtype).reshape(shape)
    vc = _pool_bits(rng, num_blocks, block_elems, dtype).reshape(shape)
    return GatherCase(name=name or f"gather_t{num_tokens}", dtype=dtype, key_cache=kc,
                      value_cache=vc, slot_mapping=slots, num_heads=num_heads,
                      head_size=head_size, block_size=block_size, num_blocks=num_blocks)


# ---------------------------------------------------------------------------
# The workloads.  Seed convention: 1000 * workload id + sweep index.

@dataclass
class PrefillCase:
    """Inputs of one paged prefill call: a DecodeCase's cache, tables and
    lengths, plus the packed chunk queries."""
    base: DecodeCase           # its q is unused
    q: np.ndarray              # uint16 [T, H, D], T = query_start[-1]
    query_start: np.ndarray    # int32 [S + 1], cumulative chunk lengths

    @property
    def query_lens(self) -> np.ndarray:
        return np.diff(self.query_start)


def make_prefill_case(*, seed: int, num_seqs: int, num_heads: int, num_kv_heads: int,
                      head_size: int, block_size: int, num_blocks: int, context_lens,
                      query_lens, dtype: str, poison: bool = True,
                      name: str = "") -> PrefillCase:
    """A seeded paged cache (as make_decode_case) and, for each sequence s,
    query_lens[s] new query tokens packed token-major into q [T, H, D]."""
    base = make_decode_case(seed=seed, num_seqs=num_seqs, num_heads=num_heads,
                            num_kv_heads=num_kv_heads, head_size=head_size,
                            block_size=block_size, num_blocks=num_blocks,
                            context_lens=context_lens, dtype=dtype, poison=poison,
                            name=name or f"prefill_s{num_seqs}_h{num_heads}_{num_kv_heads}")
    qlens = np.asarray(query_lens, dtype=np.int64).reshape(num_seqs)
    if np.any(qlens < 0):
        raise ValueError("query lengths must be >= 0")
    starts = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    rng = np.random.default_rng(seed + 7919)
    T = int(starts[-1])
    q = _normal_bits(rng, T * num_heads * head_size, dtype).reshape(T, num_heads, head_size)
    return PrefillCase(base=base, q=q, query_start=starts)


def decode_configs():
    """Decode-attention workloads as {name: kwargs for make_decode_case}."""
    out = {}
    out["tiny_mha"] = dict(seed=1000, num_seqs=2, num_heads=4, num_kv_heads=4, head_size=64,
                           block_size=16, num_blocks=16, context_lens=[17, 40], dtype="fp16")
    out["llama13b_mha_b8_ctx256"] = dict(
        seed=2000, num_seqs=8, num_heads=40, num_kv_heads=40, head_size=128, block_size=16,
        num_blocks=2048, context_lens=[256] * 8, dtype="fp16")
    for i, s in enumerate((1, 4, 16, 64, 256)):
        out[f"gqa_ctx1024_b{s}"] = dict(
            seed=3000 + i, num_seqs=s, num_heads=64, num_kv_heads=8, head_size=128,
            block_size=16, num_blocks=256 * 1024 // 16, context_lens=[1024] * s, dtype="bf16")
    for i, s in enumerate((1, 4, 16, 64, 256)):
        out[f"gqa_ctx4096_b{s}"] = dict(
            seed=4000 + i, num_seqs=s, num_heads=64, num_kv_heads=8, head_size=128,
            block_size=16, num_blocks=256 * 4096 // 16, context_lens=[4096] * s, dtype="bf16")
    for i, s in enumerate((1, 4, 16, 64, 256)):
        out[f"gqa_ctx4096_bs256_b{s}"] = dict(
            seed=4100 + i, num_seqs=s, num_heads=64, num_kv_heads=8, head_size=128,
            block_size=256, num_blocks=256 * 4096 // 256, context_lens=[4096] * s, dtype="bf16")
    lens = np.random.default_rng(5000).integers(128, 8192, size=64, endpoint=True)
    out["mqa_ragged_b64"] = dict(
        seed=5001, num_seqs=64, num_heads=48, num_kv_heads=1, head_size=128, block_size=16,
        num_blocks=40000, context_lens=lens.tolist(), dtype="fp16")
    return out


def prefill_configs():
    """Prefill workloads as {name: kwargs for make_prefill_case}: the 128-token
    prompts of the end-to-end throughput runs in "[Performance] Support
    MQA/GQA in decode phase by using FlashAttention" (7B models with 32 MHA
    heads), and 64/8-head GQA chunks with and without a long cached prefix."""
    return {
        "prefill_mha32_prompt128_b16": dict(
            seed=6000, num_seqs=16, num_heads=32, num_kv_heads=32, head_size=128, block_size=16,
            num_blocks=16 * 128 // 16 + 8, context_lens=[128] * 16, query_lens=[128] * 16,
            dtype="fp16"),
        "prefill_gqa_prompt1024_b8": dict(
            seed=6001, num_seqs=8, num_heads=64, num_kv_heads=8, head_size=128, block_size=16,
            num_blocks=8 * 1024 // 16 + 8, context_lens=[1024] * 8, query_lens=[1024] * 8,
            dtype="bf16"),
        "prefill_gqa_chunk256_ctx4096_b4": dict(
            seed=6002, num_seqs=4, num_heads=64, num_kv_heads=8, head_size=128, block_size=16,
            num_blocks=4 * 4096 // 16 + 8, context_lens=[4096] * 4, query_lens=[256] * 4,
            dtype="bf16"),
    }


def gather_sweep():
    """gather_cached_kv workloads as {name: kwargs for make_gather_case}."""
    return {f"gather_t{t}": dict(seed=2100 + i, num_tokens=t, num_heads=40, head_size=128,
                                 block_size=8, num_blocks=1024, dtype="fp16")
            for i, t in enumerate((64, 128, 256, 512, 1024, 2048))}
