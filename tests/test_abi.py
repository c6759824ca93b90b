"""The C-ABI library loads, exports what include/pkd.h declares, and rejects
bad host arguments before touching the GPU (these run without a GPU)."""
import ctypes

import pytest

from paged_kv_decode_22_gb300 import _lib

NULL = None
FAKE = ctypes.c_void_p(0x10000)        # 16-byte aligned, never dereferenced
MISALIGNED = ctypes.c_void_p(0x10008)


@pytest.fixture(scope="module")
def lib():
    import os
    if not os.path.exists(_lib.LIB_PATH):
        from paged_kv_decode_22_gb300 import build
        build.build()
    return _lib.lib()


def test_every_declared_symbol_is_exported(lib):
    names = _lib.exported_names()
    assert set(names) >= {"pkd_paged_decode_attention", "pkd_gather_cached_kv",
                          "pkd_reshape_and_cache", "pkd_decode_plan", "pkd_status_string",
                          "pkd_last_error", "pkd_version"}
    for n in names:
        assert hasattr(lib, n), n


def test_header_constants_match_the_binding():
    """Every #define of include/pkd.h that the binding mirrors has the same value."""
    import re
    text = open(_lib.HEADER).read()
    defs = {m.group(1): int(m.group(2)) for m in
            re.finditer(r"#define\s+PKD_(\w+)\s+\(?(-?\d+)u?\)?", text)}
    mirrored = {"PATH_SIMT": _lib.PATH_SIMT, "PATH_TC": _lib.PATH_TC,
                "PATH_TC_CLUSTER": _lib.PATH_TC_CLUSTER, "PATH_TC_STREAM": _lib.PATH_TC_STREAM,
                "PARTITION_STREAM": _lib.PARTITION_STREAM, "DEV_BAD_BLOCK": _lib.DEV_BAD_BLOCK,
                "DEV_BAD_SLOT": _lib.DEV_BAD_SLOT, "DEV_BAD_LEN": _lib.DEV_BAD_LEN,
                "DEV_TIMEOUT": _lib.DEV_TIMEOUT}
    for name, value in mirrored.items():
        assert defs.get(name) == value, (name, defs.get(name), value)


def test_selftest_rejects_bad_arguments_on_host(lib):
    assert lib.pkd_selftest_bounded_wait(NULL, 1000000, NULL) == 1
    assert lib.pkd_selftest_bounded_wait(FAKE, 10, NULL) == 2
    assert lib.pkd_selftest_bounded_wait(FAKE, 2 * 10**9, NULL) == 2


def test_version_and_status_strings(lib):
    assert lib.pkd_version() >= 100
    for code in range(8):
        assert lib.pkd_status_string(code)
    assert lib.pkd_status_string(99) == b"unknown status"
    assert lib.pkd_last_error() == b""


def _decode(lib, **kw):
    a = dict(out=FAKE, q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, mb=4, cl=FAKE, maxctx=64, S=2, H=8,
             Hk=2, D=128, B=16, NB=16, scale=0.1, dtype=1, ps=0, ws=NULL, wsb=0, st=NULL,
             stream=NULL)
    a.update(kw)
    return lib.pkd_paged_decode_attention(a["out"], a["q"], a["kc"], a["vc"], a["bt"], a["mb"],
                                          a["cl"], a["maxctx"], a["S"], a["H"], a["Hk"], a["D"],
                                          a["B"], a["NB"], a["scale"], a["dtype"], a["ps"],
                                          a["ws"], a["wsb"], a["st"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(out=NULL), 1), (dict(q=NULL), 1), (dict(bt=NULL), 1), (dict(cl=NULL), 1),
    (dict(dtype=5), 3), (dict(B=12), 3), (dict(B=4), 3), (dict(B=512), 3),
    (dict(NB=0), 2), (dict(mb=0), 2), (dict(q=MISALIGNED), 5), (dict(kc=MISALIGNED), 5),
    (dict(H=6, Hk=4), 2), (dict(S=0), 2), (dict(S=70000), 2), (dict(maxctx=-1), 2),
    (dict(D=96), 3), (dict(NB=1 << 28, B=16), 2), (dict(ps=-2), 2),
])
def test_decode_rejects_bad_arguments_on_host(lib, kw, code):
    assert _decode(lib, **kw) == code


def test_decode_ex_rejects_misaligned_alibi_slopes(lib):
    st = lib.pkd_paged_decode_attention_ex(FAKE, FAKE, FAKE, FAKE, FAKE, 4, FAKE, 64, 2, 8, 2, 128,
                                           16, 16, 0.1, ctypes.c_void_p(0x10002), 1, 0, NULL, 0,
                                           NULL, NULL)
    assert st == 5
    assert lib.pkd_paged_decode_attention_ex(NULL, FAKE, FAKE, FAKE, FAKE, 4, FAKE, 64, 2, 8, 2,
                                             128, 16, 16, 0.1, NULL, 1, 0, NULL, 0, NULL,
                                             NULL) == 1


def _copy(lib, fn, **kw):
    a = dict(d0=FAKE, d1=FAKE, s0=FAKE, s1=FAKE, slots=FAKE, T=4, H=40, D=128, B=8, NB=16,
             dtype=0, st=NULL, stream=NULL)
    a.update(kw)
    return getattr(lib, fn)(a["d0"], a["d1"], a["s0"], a["s1"], a["slots"], a["T"], a["H"],
                            a["D"], a["B"], a["NB"], a["dtype"], a["st"], a["stream"])


@pytest.mark.parametrize("fn", ["pkd_gather_cached_kv", "pkd_reshape_and_cache"])
@pytest.mark.parametrize("kw,code", [
    (dict(T=0, d0=NULL, slots=NULL), 0),   # empty input: nothing to do, no GPU needed
    (dict(d0=NULL), 1), (dict(slots=NULL), 1), (dict(T=-1), 2), (dict(D=12), 2),
    (dict(B=0), 2), (dict(NB=0), 2), (dict(dtype=2), 3), (dict(s1=MISALIGNED), 5),
])
def test_copies_reject_bad_arguments_on_host(lib, fn, kw, code):
    assert _copy(lib, fn, **kw) == code


def test_binding_raises_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        _lib.lib()


def test_workspace_bytes_is_zero_without_a_device_or_for_bad_sizes(lib):
    # Pure host answer: no sm_103 device (or invalid sizes) means no plan.
    import torch
    assert lib.pkd_decode_workspace_bytes(4, 63, 128, 4096) == 0 or torch.cuda.is_available()
    assert lib.pkd_decode_workspace_bytes(0, 64, 128, 4096) == 0
    assert lib.pkd_decode_workspace_bytes(4, 64, 96, 4096) == 0
    if not torch.cuda.is_available():
        assert lib.pkd_decode_workspace_bytes(4, 64, 128, 4096) == 0
