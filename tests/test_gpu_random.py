"""Seeded random shapes on the GPU against the CPU oracle.

Decode: random query-group sizes, KV-head counts, head sizes, block sizes,
dtypes and ragged lengths (with the edge lengths 0, 1 and one block +- 1
mixed in), each run in the library's own plan and in the forced forms that
the shape admits (stream, fixed partitions of 128 and 256 tokens).  Prefill:
random layouts and chunk mixes (prompts, chunks over a prefix, one-token
chunks, empty chunks), each run in both kernels.  The cases are fixed by
their seeds, so a failure reproduces; they add shape combinations that the
hand-picked layouts of the other tests do not reach.

Tolerances as in the other tests: decode max |err| <= 1e-2 and mean <= 1e-3;
prefill the same with one output ulp at |ref| on the max bound.
"""
import functools

import numpy as np
import pytest

from oracle.paged_attention import paged_decode_attention as oracle_decode
from paged_kv_decode_22_gb300.workloads import make_decode_case

from .gpu_util import DeviceCase, assert_close, assert_close_ulp, run_decode
from .test_gpu_prefill import _case as prefill_case
from .test_gpu_prefill import _oracle as prefill_oracle
from .test_gpu_prefill import _run as prefill_run

pytestmark = pytest.mark.gpu

DECODE_SEEDS = list(range(7100, 7132))
PREFILL_SEEDS = list(range(7200, 7216))


def _decode_shape(seed):
    rng = np.random.default_rng(seed)
    dtype = ["fp16", "bf16"][int(rng.integers(2))]
    D = [64, 128, 128, 128][int(rng.integers(4))]
    Hk = [1, 2, 4, 8][int(rng.integers(4))]
    g = [1, 2, 3, 4, 5, 6, 8, 12, 16, 24, 32, 48, 64][int(rng.integers(13))]
    while Hk * g > 128:
        Hk //= 2
    B = [8, 16, 32, 64, 128, 256][int(rng.integers(6))]
    S = int(rng.integers(1, 33))
    special = [0, 1, B - 1, B, B + 1, 127, 128, 129]
    lens = [int(rng.choice(special)) if rng.random() < 0.3 else int(rng.integers(1, 2600))
            for _ in range(S)]
    if max(lens) == 0:
        lens[0] = 1
    return dict(dtype=dtype, head_size=D, num_kv_heads=Hk, num_heads=Hk * g, block_size=B,
                num_seqs=S, context_lens=lens)


@pytest.mark.parametrize("seed", DECODE_SEEDS)
def test_random_decode_matches_oracle(seed):
    from paged_kv_decode_22_gb300 import ops
    sh = _decode_shape(seed)
    B = sh["block_size"]
    need = sum(-(-L // B) for L in sh["context_lens"])
    c = make_decode_case(seed=seed, num_blocks=need + 8, **sh)
    dc = DeviceCase(c)
    ref = oracle_decode(c.q, c.key_cache, c.value_cache, c.block_tables, c.context_lens, c.scale,
                        c.dtype)
    ran = 0
    for ps in (0, -1, 128, 256):
        try:
            plan = ops.decode_plan(c.num_seqs, c.num_heads, c.num_kv_heads, c.head_size, B,
                                   c.max_context_len, ps)
        except ops.PkdError:
            continue   # a form this shape does not admit (the stream form needs the TC path)
        got, status = run_decode(dc, partition_size=ps)
        assert status == 0, (sh, ps)
        assert_close(got, ref, f"seed {seed} {sh} partition_size {ps} plan {plan}")
        ran += 1
    assert ran >= 2   # the library's plan and at least one fixed split


def _prefill_shape(seed):
    rng = np.random.default_rng(seed)
    dtype = ["fp16", "bf16"][int(rng.integers(2))]
    Hk = [1, 2, 4, 8][int(rng.integers(4))]
    g = [1, 2, 4, 5, 8, 16, 32, 64][int(rng.integers(8))]
    while Hk * g > 128:
        Hk //= 2
    B = [8, 16, 32, 64, 128, 256][int(rng.integers(6))]
    S = int(rng.integers(1, 7))
    chunks = []
    for _ in range(S):
        kind = int(rng.integers(4))
        if kind == 0:     # a prompt without prefix
            L = int(rng.integers(1, 700))
            n = L
        else:             # a chunk over a cached prefix: empty, one token, or up to 300
            L = int(rng.integers(1, 2600))
            if kind == 1:
                n = 0 if rng.random() < 0.3 else 1
            else:
                n = int(rng.integers(1, min(L, 300) + 1))
        chunks.append((L, n))
    if all(n == 0 for _, n in chunks):
        chunks[0] = (chunks[0][0], min(chunks[0][0], 33))
    return dtype, Hk * g, Hk, B, chunks


@functools.lru_cache(maxsize=1)
def _prefill_case_and_ref(seed):
    dtype, H, Hk, B, chunks = _prefill_shape(seed)
    c = prefill_case(seed, H, Hk, B, dtype, chunks)
    return (dtype, H, Hk, B, chunks), c, prefill_oracle(c)


# form varies fastest, so both kernels run on one seed's cached case in turn
@pytest.mark.parametrize("form", ["single", "pair"])
@pytest.mark.parametrize("seed", PREFILL_SEEDS)
def test_random_prefill_matches_oracle(form, seed):
    (dtype, H, Hk, B, chunks), c, ref = _prefill_case_and_ref(seed)
    got, status = prefill_run(c, form=form)
    assert status == 0
    assert_close_ulp(got, ref, dtype, f"seed {seed} H{H}/{Hk} B{B} {dtype} {chunks} {form}")
