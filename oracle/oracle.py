"""ctypes front end for the fp64 CPU oracle in oracle.c.

TEST INFRASTRUCTURE ONLY: imported by the test-suite, the package smoke check
and the benchmark's CPU-baseline leg.  The product library never imports this
module, and this module never imports the product package.

All arrays are numpy; inputs are passed as their raw bytes (fp32, or bf16
carried in uint16), so the oracle sees exactly the bytes the GPU sees.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, OpenMP when available)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB)
    return _LIB


class Shape(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("n_q_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32),
                ("seq_len", C.c_int32), ("window", C.c_int32), ("dtype", C.c_int32)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = C.CDLL(build())
            p, i32, i64, u32, d = C.c_void_p, C.c_int32, C.c_int64, C.c_uint32, C.c_double
            sp = C.POINTER(Shape)
            sig = {
                "ora_num_threads": (C.c_int, []),
                "ora_set_num_threads": (None, [C.c_int]),
                "ora_score_unit": (C.c_int, [sp, p, p, C.c_int, C.c_int, p]),
                "ora_score": (C.c_int, [sp, p, p, p]),
                "ora_mba": (i64, [i64, p, u32, u32]),
                "ora_mba_all": (C.c_int, [sp, p, u32, u32, p]),
                "ora_mba_all_f32": (C.c_int, [sp, p, u32, u32, p]),
                "ora_budget": (C.c_int, [C.c_int, C.c_int, p, i64, i64, i64, p]),
                "ora_topk": (i64, [i64, p, i64, p]),
                "ora_topk_all": (C.c_int, [sp, p, p, i64, p]),
                "ora_topk_all_f32": (C.c_int, [sp, p, p, i64, p]),
                "ora_pool": (C.c_int, [sp, p, i32, i32, p]),
                "ora_pool_f32": (C.c_int, [sp, p, i32, i32, p]),
                "ora_compact_rows": (i64, [sp, p]),
                "ora_philox4x32_10": (None, [p, p, p]),
                "ora_keyformer_uniform": (d, [C.c_uint64, i64, i64, i64]),
                "ora_score_keyformer": (C.c_int, [sp, p, p, C.c_uint64, d, p]),
                "ora_head_budget": (C.c_int, [C.c_int, C.c_int, p, p, i64, p]),
                "ora_topk_heads": (C.c_int, [sp, p, p, i64, p]),
                "ora_threshold_select": (C.c_int, [sp, p, C.c_float, i64, p, p]),
                "ora_compact_heads": (i64, [sp, p, p, p, i64, p]),
                "ora_compact": (i64, [sp, p, p, p, i64, p]),
                "ora_keep_channels": (i32, [d, i32]),
                "ora_channel_prune": (C.c_int, [sp, p, p, d, p, p, p]),
                "ora_channel_prune_query": (C.c_int, [sp, p, p, p, d, p, p, p]),
                "ora_value_scores": (C.c_int, [sp, p, p, p, p]),
                "ora_channel_prune_value": (C.c_int, [sp, p, p, p, d, p, p]),
                "ora_compress": (C.c_int, [sp, p, p, p, u32, u32, i64, i64, d, i64,
                                           p, p, p, p, p, p, p, p]),
            }
            for name, (res, args) in sig.items():
                f = getattr(_lib, name)
                f.restype = res
                f.argtypes = args
        return _lib


# --- helpers ----------------------------------------------------------------

def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def raw(x) -> np.ndarray:
    """Contiguous raw-bytes view of a tensor/array: fp32 stays float32, bf16
    becomes its uint16 bit pattern."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16)
            return x.numpy()
    except ImportError:
        pass
    return np.ascontiguousarray(x)


def shape_of(n_layers, n_q_heads, n_kv_heads, head_dim, seq_len, window, dtype) -> Shape:
    return Shape(n_layers, n_q_heads, n_kv_heads, head_dim, seq_len, window,
                 0 if dtype in ("f32", 0) else 1)


def _check(rc, what):
    if rc < 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")
    return rc


def num_threads() -> int:
    return lib().ora_num_threads()


def set_num_threads(n: int) -> None:
    lib().ora_set_num_threads(int(n))


def score_unit(s: Shape, q, k, layer: int, kv_head: int) -> np.ndarray:
    qa, ka = raw(q), raw(k)
    c = np.empty(s.seq_len, dtype=np.float64)
    _check(lib().ora_score_unit(C.byref(s), _ptr(qa), _ptr(ka), layer, kv_head, _ptr(c)), "score")
    return c


def score(s: Shape, q, k) -> np.ndarray:
    qa, ka = raw(q), raw(k)
    c = np.empty((s.n_layers, s.n_kv_heads, s.seq_len), dtype=np.float64)
    _check(lib().ora_score(C.byref(s), _ptr(qa), _ptr(ka), _ptr(c)), "score")
    return c


def mba(c, num=9, den=10) -> int:
    c = np.ascontiguousarray(c, dtype=np.float64)
    return _check(lib().ora_mba(c.size, _ptr(c), num, den), "mba")


def mba_all(s: Shape, scores, num=9, den=10) -> np.ndarray:
    out = np.empty((s.n_layers, s.n_kv_heads), dtype=np.int32)
    if scores.dtype == np.float32:
        sc = np.ascontiguousarray(scores)
        _check(lib().ora_mba_all_f32(C.byref(s), _ptr(sc), num, den, _ptr(out)), "mba")
    else:
        sc = np.ascontiguousarray(scores, dtype=np.float64)
        _check(lib().ora_mba_all(C.byref(s), _ptr(sc), num, den, _ptr(out)), "mba")
    return out


def budget(mba_lk, prefix: int, total: int, floor: int) -> np.ndarray:
    m = np.ascontiguousarray(mba_lk, dtype=np.int32)
    L, H = m.shape
    out = np.empty(L, dtype=np.int32)
    _check(lib().ora_budget(L, H, _ptr(m), prefix, total, floor, _ptr(out)), "budget")
    return out


def topk(c, P: int, B: int) -> np.ndarray:
    c = np.ascontiguousarray(c, dtype=np.float64)
    idx = np.empty(max(1, min(max(B, 0), P)), dtype=np.int32)
    n = _check(lib().ora_topk(P, _ptr(c), B, _ptr(idx)), "topk")
    return idx[:n]


def topk_all(s: Shape, scores, budget_l, k_max: int) -> np.ndarray:
    b = np.ascontiguousarray(budget_l, dtype=np.int32)
    idx = np.full((s.n_layers, s.n_kv_heads, max(k_max, 1)), -1, dtype=np.int32)
    if scores.dtype == np.float32:
        sc = np.ascontiguousarray(scores)
        _check(lib().ora_topk_all_f32(C.byref(s), _ptr(sc), _ptr(b), k_max, _ptr(idx)), "topk")
    else:
        sc = np.ascontiguousarray(scores, dtype=np.float64)
        _check(lib().ora_topk_all(C.byref(s), _ptr(sc), _ptr(b), k_max, _ptr(idx)), "topk")
    return idx


def pool(s: Shape, scores, kernel: int, mode: int = 0) -> np.ndarray:
    """SnapKV pooling of the prefix scores (mode 0 average, 1 max); fp64
    [L][H_kv][T], window positions copied unchanged."""
    out = np.empty((s.n_layers, s.n_kv_heads, s.seq_len), dtype=np.float64)
    if scores.dtype == np.float32:
        sc = np.ascontiguousarray(scores)
        _check(lib().ora_pool_f32(C.byref(s), _ptr(sc), kernel, mode, _ptr(out)), "pool")
    else:
        sc = np.ascontiguousarray(scores, dtype=np.float64)
        _check(lib().ora_pool(C.byref(s), _ptr(sc), kernel, mode, _ptr(out)), "pool")
    return out


def head_budget(mba_lk, budget_l, prefix: int) -> np.ndarray:
    """Per-head split of each layer's H_kv * B_l tokens by MBA: [L][H_kv]."""
    m = np.ascontiguousarray(mba_lk, dtype=np.int32)
    b = np.ascontiguousarray(budget_l, dtype=np.int32)
    L, H = m.shape
    out = np.empty((L, H), dtype=np.int32)
    _check(lib().ora_head_budget(L, H, _ptr(m), _ptr(b), prefix, _ptr(out)), "head_budget")
    return out


def topk_heads(s: Shape, scores, head_budget_lk, k_max: int) -> np.ndarray:
    hb = np.ascontiguousarray(head_budget_lk, dtype=np.int32)
    idx = np.full((s.n_layers, s.n_kv_heads, max(k_max, 1)), -1, dtype=np.int32)
    sc = np.ascontiguousarray(scores, dtype=np.float64)
    _check(lib().ora_topk_heads(C.byref(s), _ptr(sc), _ptr(hb), k_max, _ptr(idx)), "topk_heads")
    return idx


def threshold_select(s: Shape, scores_f32, tau: float, k_max: int):
    """Returns (idx [L][H_kv][k_max] (-1 past the count), counts [L][H_kv],
    overflowed)."""
    sc = np.ascontiguousarray(scores_f32, dtype=np.float32)
    idx = np.full((s.n_layers, s.n_kv_heads, max(k_max, 1)), -1, dtype=np.int32)
    cnt = np.empty((s.n_layers, s.n_kv_heads), dtype=np.int32)
    rc = _check(lib().ora_threshold_select(C.byref(s), _ptr(sc), float(tau), k_max, _ptr(idx),
                                           _ptr(cnt)), "threshold_select")
    return idx, cnt, bool(rc)


def compact_heads(s: Shape, x, idx, counts, k_max: int) -> np.ndarray:
    xa = raw(x)
    ix = np.ascontiguousarray(idx, dtype=np.int32)
    c = np.ascontiguousarray(counts, dtype=np.int32)
    P = s.seq_len - s.window
    n = np.minimum(np.clip(c, 0, P), k_max).astype(np.int64)
    rows = int((n + s.window).sum())
    out = np.empty((rows, s.head_dim), dtype=xa.dtype)
    got = _check(lib().ora_compact_heads(C.byref(s), _ptr(xa), _ptr(ix), _ptr(c), k_max, _ptr(out)),
                 "compact_heads")
    assert got == rows
    return out


def philox4x32_10(counter, key) -> list:
    c = (C.c_uint32 * 4)(*[int(x) & 0xFFFFFFFF for x in counter])
    k = (C.c_uint32 * 2)(*[int(x) & 0xFFFFFFFF for x in key])
    o = (C.c_uint32 * 4)()
    lib().ora_philox4x32_10(c, k, o)
    return list(o)


def keyformer_uniform(seed: int, unit: int, row: int, key: int) -> float:
    return lib().ora_keyformer_uniform(int(seed), int(unit), int(row), int(key))


def score_keyformer(s: Shape, q, k, seed: int, tau: float) -> np.ndarray:
    """Keyformer window scores with Gumbel noise and temperature: fp64
    [L][H_kv][T]."""
    qa, ka = raw(q), raw(k)
    c = np.empty((s.n_layers, s.n_kv_heads, s.seq_len), dtype=np.float64)
    _check(lib().ora_score_keyformer(C.byref(s), _ptr(qa), _ptr(ka), int(seed), float(tau),
                                     _ptr(c)), "score_keyformer")
    return c


def compact_rows(s: Shape, budget_l) -> int:
    b = np.ascontiguousarray(budget_l, dtype=np.int32)
    return _check(lib().ora_compact_rows(C.byref(s), _ptr(b)), "compact")


def compact(s: Shape, x, idx, budget_l, k_max: int) -> np.ndarray:
    """Returns the packed rows as a raw array [rows][D] (float32 or uint16)."""
    xa = raw(x)
    b = np.ascontiguousarray(budget_l, dtype=np.int32)
    ix = np.ascontiguousarray(idx, dtype=np.int32)
    rows = compact_rows(s, b)
    out = np.empty((rows, s.head_dim), dtype=xa.dtype)
    _check(lib().ora_compact(C.byref(s), _ptr(xa), _ptr(ix), _ptr(b), k_max, _ptr(out)), "compact")
    return out


def keep_channels(lam: float, D: int) -> int:
    return lib().ora_keep_channels(float(lam), int(D))


def channel_prune(s: Shape, k_out, budget_l, lam: float):
    """Returns (chan [L][H_kv][keep], norms [L][H_kv][D] fp64, k_pruned raw)."""
    ka = raw(k_out)
    b = np.ascontiguousarray(budget_l, dtype=np.int32)
    keep = keep_channels(lam, s.head_dim)
    P = s.seq_len - s.window
    n = np.clip(b, 0, P).astype(np.int64)
    chan = np.empty((s.n_layers, s.n_kv_heads, max(keep, 1)), dtype=np.int32)
    norms = np.empty((s.n_layers, s.n_kv_heads, s.head_dim), dtype=np.float64)
    kp = np.empty(int(s.n_kv_heads * n.sum() * max(keep, 1)), dtype=ka.dtype)
    _check(lib().ora_channel_prune(C.byref(s), _ptr(ka), _ptr(b), float(lam), _ptr(chan),
                                   _ptr(norms), _ptr(kp)), "channel_prune")
    return chan, norms, kp


def channel_prune_query(s: Shape, q, k_out, budget_l, lam: float):
    """ThinK query-driven criterion.  Returns (chan [L][H_kv][keep],
    scores [L][H_kv][D] fp64, k_pruned raw)."""
    qa, ka = raw(q), raw(k_out)
    b = np.ascontiguousarray(budget_l, dtype=np.int32)
    keep = keep_channels(lam, s.head_dim)
    P = s.seq_len - s.window
    n = np.clip(b, 0, P).astype(np.int64)
    chan = np.empty((s.n_layers, s.n_kv_heads, max(keep, 1)), dtype=np.int32)
    sc = np.empty((s.n_layers, s.n_kv_heads, s.head_dim), dtype=np.float64)
    kp = np.empty(int(s.n_kv_heads * n.sum() * max(keep, 1)), dtype=ka.dtype)
    _check(lib().ora_channel_prune_query(C.byref(s), _ptr(qa), _ptr(ka), _ptr(b), float(lam),
                                         _ptr(chan), _ptr(sc), _ptr(kp)), "channel_prune_query")
    return chan, sc, kp


def value_scores(s: Shape, q, k, v) -> np.ndarray:
    """THINKV channel scores: [L][H_kv][D] fp64, the squared norm of each
    column of the window rows' attention output softmax(QK^T/sqrt(D)) V."""
    qa, ka, va = raw(q), raw(k), raw(v)
    out = np.empty((s.n_layers, s.n_kv_heads, s.head_dim), dtype=np.float64)
    _check(lib().ora_value_scores(C.byref(s), _ptr(qa), _ptr(ka), _ptr(va), _ptr(out)),
           "value_scores")
    return out


def channel_prune_value(s: Shape, score_v, v_out, budget_l, lam: float):
    """THINKV selection on given channel scores ([L][H_kv][D], fp64 or fp32
    widened exactly) and copy of the kept prefix rows' channels.  Returns
    (chan [L][H_kv][keep], v_pruned raw)."""
    sv = np.ascontiguousarray(score_v, dtype=np.float64)
    va = raw(v_out)
    b = np.ascontiguousarray(budget_l, dtype=np.int32)
    keep = keep_channels(lam, s.head_dim)
    P = s.seq_len - s.window
    n = np.clip(b, 0, P).astype(np.int64)
    chan = np.empty((s.n_layers, s.n_kv_heads, max(keep, 1)), dtype=np.int32)
    vp = np.empty(max(1, int(s.n_kv_heads * n.sum() * max(keep, 1))), dtype=va.dtype)
    _check(lib().ora_channel_prune_value(C.byref(s), _ptr(sv), _ptr(va), _ptr(b), float(lam),
                                         _ptr(chan), _ptr(vp)), "channel_prune_value")
    return chan, vp[: int(s.n_kv_heads * n.sum() * keep)]


def compress(s: Shape, q, k, v, total: int, floor: int, k_max: int,
             num=9, den=10, lam=None):
    """The whole path for one prompt.  Returns a dict of numpy outputs."""
    qa, ka, va = raw(q), raw(k), raw(v)
    L, H, T, W, D = s.n_layers, s.n_kv_heads, s.seq_len, s.window, s.head_dim
    P = T - W
    scores = np.empty((L, H, T), dtype=np.float64)
    mba_o = np.empty((L, H), dtype=np.int32)
    bud = np.empty(L, dtype=np.int32)
    idx = np.full((L, H, max(k_max, 1)), -1, dtype=np.int32)
    cap_rows = H * (min(total, L * P) + L * W + 1)
    k_out = np.empty((cap_rows, D), dtype=ka.dtype)
    v_out = np.empty((cap_rows, D), dtype=va.dtype)
    keep = keep_channels(lam, D) if lam is not None else 1
    chan = np.empty((L, H, max(keep, 1)), dtype=np.int32)
    k_pr = np.empty(max(1, H * min(total, L * P) * keep), dtype=ka.dtype)
    rc = lib().ora_compress(C.byref(s), _ptr(qa), _ptr(ka), _ptr(va), num, den, total, floor,
                            -1.0 if lam is None else float(lam), k_max,
                            _ptr(scores), _ptr(mba_o), _ptr(bud), _ptr(idx),
                            _ptr(k_out), _ptr(v_out), _ptr(chan), _ptr(k_pr))
    _check(rc, "compress")
    rows = compact_rows(s, bud)
    n = np.clip(bud, 0, P).astype(np.int64)
    out = dict(scores=scores, mba=mba_o, budget=bud, idx=idx,
               k_out=k_out[:rows], v_out=v_out[:rows])
    if lam is not None:
        out["chan"] = chan
        out["k_pruned"] = k_pr[: int(H * n.sum() * keep)]
    return out
