"""gather_cached_kv and reshape_and_cache on the GPU: bit-exact against the oracle."""
import numpy as np
import pytest
import torch

from oracle.cache import cache_kv
from oracle.gather import gather_cached_kv as oracle_gather
from paged_kv_decode_22_gb300.workloads import gather_sweep, make_gather_case

from .gpu_util import down_bits, up

pytestmark = pytest.mark.gpu


def _run_gather(g, slots=None):
    from paged_kv_decode_22_gb300 import ops
    slots = g.slot_mapping if slots is None else slots
    dt = torch.float16 if g.dtype == "fp16" else torch.bfloat16
    kc, vc = up(g.key_cache, g.dtype), up(g.value_cache, g.dtype)
    T = len(slots)
    ko = torch.full((T, g.num_heads, g.head_size), float("nan"), dtype=dt, device="cuda")
    vo = torch.full_like(ko, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.gather_cached_kv(ko, vo, kc, vc, up(np.asarray(slots, np.int64)), device_status=status)
    torch.cuda.synchronize()
    return down_bits(ko), down_bits(vo), int(status.item())


@pytest.mark.parametrize("name", sorted(gather_sweep()))
def test_gather_sweep_bit_exact(name):
    g = make_gather_case(name=name, **gather_sweep()[name])
    k, v, status = _run_gather(g)
    rk, rv = oracle_gather(g.key_cache, g.value_cache, g.slot_mapping)
    assert status == 0
    np.testing.assert_array_equal(k, rk)
    np.testing.assert_array_equal(v, rv)


# 50 tokens are 100 rows: rows of 16 B up to 32 KB take the bulk-copy kernel
# (128 x 128 x 2 B is its largest row); 136 heads give 34 KB rows, which take
# the 16-byte-load kernel, as do the sweep's gathers of more than 256 tokens.
@pytest.mark.parametrize("H,D,B,dtype", [(1, 8, 1, "fp16"), (3, 24, 5, "bf16"),
                                         (8, 128, 16, "bf16"), (40, 128, 8, "fp16"),
                                         (128, 128, 4, "bf16"), (136, 128, 2, "fp16")])
def test_gather_odd_shapes_and_invalid_slots(H, D, B, dtype):
    g = make_gather_case(seed=4, num_tokens=50, num_heads=H, head_size=D, block_size=B,
                         num_blocks=64, dtype=dtype)
    slots = g.slot_mapping.copy()
    slots[[3, 17]] = [-1, 64 * B]
    k, v, status = _run_gather(g, slots)
    rk, rv = oracle_gather(g.key_cache, g.value_cache, slots)
    assert status == 2
    np.testing.assert_array_equal(k, rk)
    np.testing.assert_array_equal(v, rv)


def test_gather_empty_is_a_no_op():
    g = make_gather_case(seed=5, num_tokens=1, num_heads=2, head_size=8, block_size=4,
                         num_blocks=2, dtype="fp16")
    k, v, status = _run_gather(g, np.zeros(0, np.int64))
    assert k.shape == (0, 2, 8) and status == 0


@pytest.mark.parametrize("T", [256, 257])
def test_copies_at_the_kernel_boundary(T):
    # 256 tokens (512 rows) are the most the bulk-copy kernel takes; 257 go
    # to the 16-byte-load kernels.  Both directions, with a bad slot each.
    from paged_kv_decode_22_gb300 import ops
    g = make_gather_case(seed=9, num_tokens=T, num_heads=40, head_size=128, block_size=8,
                         num_blocks=64, dtype="fp16")
    slots = g.slot_mapping.copy()
    slots[T - 1] = 64 * 8 + 1
    k, v, status = _run_gather(g, slots)
    rk, rv = oracle_gather(g.key_cache, g.value_cache, slots)
    assert status == 2
    np.testing.assert_array_equal(k, rk)
    np.testing.assert_array_equal(v, rv)
    rng = np.random.default_rng(T)
    key = rng.integers(0, 0x7C00, (T, 40, 128), dtype=np.uint16)
    val = rng.integers(0, 0x7C00, (T, 40, 128), dtype=np.uint16)
    slots[0] = -1
    kc, vc = up(g.key_cache, "fp16"), up(g.value_cache, "fp16")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.reshape_and_cache(up(key, "fp16"), up(val, "fp16"), kc, vc, up(slots), device_status=st)
    torch.cuda.synchronize()
    rk, rv = cache_kv(key, val, g.key_cache, g.value_cache, slots)
    assert int(st.item()) == 2
    np.testing.assert_array_equal(down_bits(kc), rk)
    np.testing.assert_array_equal(down_bits(vc), rv)


# 200 tokens (400 rows) take the bulk-copy kernel, 700 the 16-byte-load one.
@pytest.mark.parametrize("T", [200, 700])
@pytest.mark.parametrize("H,D,B,dtype", [(40, 128, 8, "fp16"), (8, 128, 16, "bf16"),
                                         (3, 16, 3, "fp16")])
def test_reshape_and_cache_bit_exact(H, D, B, dtype, T):
    from paged_kv_decode_22_gb300 import ops
    nb = max(64, -(-(T + 100) // B))
    g = make_gather_case(seed=6, num_tokens=T, num_heads=H, head_size=D, block_size=B,
                         num_blocks=nb, dtype=dtype)
    rng = np.random.default_rng(2)
    key = rng.integers(0, 0x7C00, (T, H, D), dtype=np.uint16)   # finite fp16/bf16 patterns
    val = rng.integers(0, 0x7C00, (T, H, D), dtype=np.uint16)
    slots = g.slot_mapping.copy()
    slots[[0, 5]] = [-1, nb * B + 2]
    kc, vc = up(g.key_cache, dtype), up(g.value_cache, dtype)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.reshape_and_cache(up(key, dtype), up(val, dtype), kc, vc, up(slots),
                          device_status=status)
    torch.cuda.synchronize()
    rk, rv = cache_kv(key, val, g.key_cache, g.value_cache, slots)
    assert int(status.item()) == 2
    np.testing.assert_array_equal(down_bits(kc), rk)
    np.testing.assert_array_equal(down_bits(vc), rv)
