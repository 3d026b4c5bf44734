"""CPU checks of the C ABI: the library builds, loads, exports every symbol
include/kvc.h declares, and rejects bad arguments on the host before any
device work (no GPU is touched by these tests)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from eviction_kvc_score_gb300 import build
    path = build.build()
    return C.CDLL(path)


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "kvc.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvc_[a-z_]+)\s*\(", text)))


def test_header_declares_the_five_path_calls():
    syms = declared_symbols()
    for name in ("kvc_score", "kvc_mba_budget", "kvc_topk_select", "kvc_compact",
                 "kvc_channel_prune"):
        assert name in syms


def test_every_declared_symbol_is_exported(lib):
    missing = [s for s in declared_symbols() if not hasattr(lib, s)]
    assert not missing, missing


def test_bounds_checking_build_exports_the_same_abi():
    """The KVC_DEBUG_BOUNDS variant is the same C ABI with extra device checks."""
    from eviction_kvc_score_gb300 import build
    dbg = C.CDLL(build.build(debug_bounds=True))
    missing = [s for s in declared_symbols() if not hasattr(dbg, s)]
    assert not missing, missing


def test_binding_exposes_the_same_names(lib):
    from eviction_kvc_score_gb300 import kvc
    for s in declared_symbols():
        assert hasattr(kvc, s), s


def _shape(kvc, **kw):
    base = dict(n_layers=2, n_q_heads=8, n_kv_heads=2, head_dim=128, seq_len=1000, window=32,
                dtype="bf16")
    base.update(kw)
    return kvc.shape(**base)


def test_host_side_validation_rejects_bad_arguments(lib):
    from eviction_kvc_score_gb300 import kvc
    L = kvc._lib
    nul = C.c_void_p(0)
    fake = C.c_void_p(0x1000)
    for bad in (dict(seq_len=32), dict(n_q_heads=7), dict(head_dim=0), dict(window=0),
                dict(dtype=5)):
        s = _shape(kvc, **bad)
        if bad.get("dtype") == 5:
            s.dtype = 5
        rc = L.kvc_score(C.byref(s), fake, fake, fake, fake, 1 << 20, nul)
        assert rc == -1, bad
        assert kvc.kvc_last_error()
    s = _shape(kvc)
    # NULL tensors and misaligned pointers are argument errors
    assert L.kvc_score(C.byref(s), nul, fake, fake, fake, 1 << 20, nul) == -1
    assert L.kvc_score(C.byref(s), C.c_void_p(0x1001), fake, fake, fake, 1 << 20, nul) == -1
    # too-small workspace
    assert L.kvc_score(C.byref(s), fake, fake, fake, fake, 16, nul) == -5
    # budget arguments: floor above the prefix, total below L*floor, bad mass
    assert L.kvc_mba_budget(C.byref(s), fake, 9, 10, 10_000, 2000, fake, fake, fake, 4096, nul) == -1
    assert L.kvc_mba_budget(C.byref(s), fake, 9, 10, 100, 64, fake, fake, fake, 4096, nul) == -1
    assert L.kvc_mba_budget(C.byref(s), fake, 11, 10, 1000, 64, fake, fake, fake, 4096, nul) == -1
    assert L.kvc_mba_budget(C.byref(s), fake, 9, 0, 1000, 64, fake, fake, fake, 4096, nul) == -1
    assert L.kvc_topk_select(C.byref(s), fake, fake, 0, fake, fake, 4096, nul) == -1
    # more layers than the budgets' one-thread-per-layer block holds
    big = _shape(kvc, n_layers=1025)
    assert L.kvc_mba_budget(C.byref(big), fake, 9, 10, 100_000, 64, fake, fake, fake, 4096,
                            nul) == -2
    assert "1024" in kvc.kvc_last_error()
    assert L.kvc_channel_prune(C.byref(s), fake, fake, C.c_double(1.0), fake, fake, 10, fake,
                               4096, nul) == -1


def test_value_channel_prune_rejects_bad_arguments(lib):
    """kvc_channel_prune_value refuses NULL tensors, misaligned inputs, a
    lambda that keeps no channel and a small workspace before any launch."""
    from eviction_kvc_score_gb300 import kvc
    L = kvc._lib
    nul = C.c_void_p(0)
    fake = C.c_void_p(0x1000)
    s = _shape(kvc)

    def call(q=fake, k=fake, v=fake, v_out=fake, bud=fake, lam=0.3, chan=fake, vp=fake, ws=fake,
             ws_bytes=1 << 30):
        return L.kvc_channel_prune_value(C.byref(s), q, k, v, v_out, bud, C.c_double(lam), nul,
                                         chan, vp, 1 << 20, ws, ws_bytes, nul)
    assert call(q=nul) == -1
    assert call(v=nul) == -1
    assert call(chan=nul) == -1
    assert call(k=C.c_void_p(0x1008)) == -1                 # not 16-byte aligned
    assert call(lam=1.0) == -1 and call(lam=-0.1) == -1     # keeps no channel / invalid
    assert call(ws_bytes=64) == -5
    assert call(ws=C.c_void_p(0x1010)) == -5                # workspace not 256-byte aligned
    assert "kvc_channel_prune_value" in kvc.kvc_last_error()
    # the flags entry point: unknown flag bits are refused before anything else runs
    assert L.kvc_channel_prune_value_ex(C.byref(s), fake, fake, fake, fake, fake, C.c_double(0.3),
                                        nul, fake, fake, 1 << 20, 0x2, fake, 1 << 30, nul) == -1
    assert "flags" in kvc.kvc_last_error()


def test_keep_channels_and_workspace_size(lib):
    from eviction_kvc_score_gb300 import kvc
    assert kvc.kvc_keep_channels(0.4, 128) == 76
    assert kvc.kvc_keep_channels(0.5, 64) == 32
    assert kvc.kvc_keep_channels(1.0, 64) == 0
    s = _shape(kvc)
    n = kvc.kvc_workspace_size(s, 100)
    assert n >= 256 and n % 256 == 0
    assert kvc.kvc_status_string(-5)


def test_oracle_and_library_share_no_code():
    """The oracle never imports the package and the package never imports the
    oracle; only the input generators are shared."""
    pkg = os.path.join(ROOT, "eviction_kvc_score_gb300")
    imp = re.compile(r"^\s*(from\s+oracle|import\s+oracle|#\s*include\s*[<\"].*oracle)", re.M)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                assert not imp.search(open(os.path.join(dirpath, f)).read()), f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c")):
            text = open(os.path.join(ROOT, "oracle", f)).read()
            assert "eviction_kvc_score_gb300" not in text and "kvc.h" not in text, f
