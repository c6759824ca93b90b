"""Every instantiation of the tensor-core decode kernel against the oracle.

The kernel is compiled once per (16-bit type, padded query group, split
form), so that each instantiation holds only its own form's code.  This
runs each of the 32 on a small ragged case: the padded groups 16, 32, 48
and 64, fp16 and bf16, and the four forms -- unsplit, split through the
workspace and the merge launch, split inside a thread-block cluster, and the
stream form -- each checked through decode_plan to be the one that runs.
Tolerances as in the other decode tests (max |err| <= 1e-2, mean <= 1e-3).
"""
import pytest

from oracle.paged_attention import paged_decode_attention as oracle_attention
from paged_kv_decode_22_gb300.workloads import make_decode_case

from .gpu_util import DeviceCase, assert_close, run_decode

pytestmark = pytest.mark.gpu

# padded group -> (H, Hk): groups 8, 32, 40 and 64
GROUPS = {16: (32, 4), 32: (64, 2), 48: (40, 1), 64: (64, 1)}
LENS = [700, 1, 300, 0, 513]
PS = 128   # partitions of the split forms


def _case(npad, dtype):
    H, Hk = GROUPS[npad]
    need = sum(-(-L // 16) for L in LENS)
    return make_decode_case(seed=900 + npad + (dtype == "bf16"), num_seqs=len(LENS), num_heads=H,
                            num_kv_heads=Hk, head_size=128, block_size=16, num_blocks=need + 4,
                            context_lens=LENS, dtype=dtype)


def _form_args(c, form):
    """(partition_size, max_context_len, expected path, expected partitions > 1)."""
    from paged_kv_decode_22_gb300 import ops
    if form == "unsplit":
        return 1024, c.max_context_len, ops.PATH_TC, False
    if form == "workspace":   # more partitions than a cluster holds
        return PS, 17 * PS, ops.PATH_TC, True
    if form == "cluster":
        return PS, c.max_context_len, ops.PATH_TC_CLUSTER, True
    return -1, c.max_context_len, ops.PATH_TC_STREAM, False


@pytest.mark.parametrize("form", ["unsplit", "workspace", "cluster", "stream"])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("npad", [16, 32, 48, 64])
def test_every_instantiation_matches_oracle(npad, dtype, form):
    from paged_kv_decode_22_gb300 import ops
    c = _case(npad, dtype)
    ps, max_ctx, path, split = _form_args(c, form)
    _, npart, got_path, _ = ops.decode_plan(c.num_seqs, c.num_heads, c.num_kv_heads, c.head_size,
                                           c.block_size, max_ctx, ps)
    if form == "cluster" and got_path != path:
        pytest.skip("the device holds too few clusters of this size for the case")
    assert got_path == path and (npart > 1) == split, (form, npart, got_path)
    got, status = run_decode(DeviceCase(c), partition_size=ps, max_context_len=max_ctx)
    assert status == 0
    ref = oracle_attention(c.q, c.key_cache, c.value_cache, c.block_tables, c.context_lens,
                           c.scale, c.dtype)
    assert_close(got, ref, f"npad {npad} {dtype} {form} (P {npart})")
    assert (got[LENS.index(0)] == 0).all()   # the empty sequence: zero rows
