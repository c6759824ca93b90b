"""Helpers for the GPU tests: upload seeded host cases, run the C ABI, compare."""
from __future__ import annotations

import numpy as np
import torch

from oracle.formats import decode_bits

ATOL_MAX = 1e-2   # max |gpu - oracle| over compared elements (fp16/bf16 output)
ATOL_MEAN = 1e-3  # mean |gpu - oracle| over compared elements

TORCH_DT = {"fp16": torch.float16, "bf16": torch.bfloat16}


def up(a: np.ndarray, dtype: str | None = None, device="cuda"):
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
    if dtype is not None:
        t = t.view(TORCH_DT[dtype])
    return t.to(device)


def down_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class DeviceCase:
    """A DecodeCase uploaded to the GPU."""

    def __init__(self, c):
        self.c = c
        self.q = up(c.q, c.dtype)
        self.kc = up(c.key_cache, c.dtype)
        self.vc = up(c.value_cache, c.dtype)
        self.bt = up(c.block_tables)
        self.cl = up(c.context_lens)


def run_decode(dc: DeviceCase, *, partition_size=0, max_context_len=None, block_tables=None,
               context_lens=None, scale=None):
    from paged_kv_decode_22_gb300 import ops
    c = dc.c
    out = torch.full(c.q.shape, float("nan"), dtype=TORCH_DT[c.dtype], device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.paged_decode_attention(
        out, dc.q, dc.kc, dc.vc, dc.bt if block_tables is None else block_tables,
        dc.cl if context_lens is None else context_lens,
        c.max_context_len if max_context_len is None else max_context_len,
        c.scale if scale is None else scale, partition_size=partition_size,
        device_status=status)
    torch.cuda.synchronize()
    return decode_bits(down_bits(out), c.dtype), int(status.item())


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    assert err.max() <= ATOL_MAX, f"{what}: max|err| {err.max():.3e} > {ATOL_MAX}"
    assert err.mean() <= ATOL_MEAN, f"{what}: mean|err| {err.mean():.3e} > {ATOL_MEAN}"
    return float(err.max()), float(err.mean())


# One unit in the last place of the 16-bit output type, relative to the
# magnitude: 2^-7 (bf16, 8 significant bits) and 2^-10 (fp16, 11).
ULP_REL = {"bf16": 2.0 ** -7, "fp16": 2.0 ** -10}


# Elements compared by assert_close_ulp, and how many of them were above the
# fixed 1e-2 bound (passing only through the one-ulp allowance); the test
# session prints both at its end.
ULP_ALLOWANCE_USE = {"compared": 0, "needed": 0}


def assert_close_ulp(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = ""):
    """assert_close with one output ulp at |ref| added to the max bound: the
    final rounding of a large result (and the 16-bit probability operand)
    is that large on its own.  Prefill's first queries attend to a few
    tokens, so their outputs reach |v| itself."""
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    ULP_ALLOWANCE_USE["compared"] += err.size
    ULP_ALLOWANCE_USE["needed"] += int((err > ATOL_MAX).sum())
    excess = err - ULP_REL[dtype] * np.abs(ref)
    assert excess.max() <= ATOL_MAX, f"{what}: max(|err| - ulp) {excess.max():.3e} > {ATOL_MAX}"
    assert err.mean() <= ATOL_MEAN, f"{what}: mean|err| {err.mean():.3e} > {ATOL_MEAN}"
    return float(err.max()), float(err.mean())


def sample_pairs(c, n: int, seed: int = 0):
    """n distinct (s, h) pairs, always including the first and last sequence and head."""
    rng = np.random.default_rng(seed)
    S, H = c.num_seqs, c.num_heads
    picks = {(0, 0), (S - 1, H - 1), (S - 1, 0), (0, H - 1)}
    while len(picks) < min(n, S * H):
        picks.add((int(rng.integers(S)), int(rng.integers(H))))
    return sorted(picks)
