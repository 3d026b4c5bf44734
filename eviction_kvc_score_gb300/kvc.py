"""Python binding of libkvc (include/kvc.h): argument marshalling only.

Every function here forwards device pointers, sizes and the current CUDA
stream to the C ABI; all compression work runs in the library's CUDA kernels.
There is no CPU fallback: importing this module raises if libkvc.so has not
been built, and calls raise KvcError on any non-zero status.

Tensors are torch tensors on the GPU (torch provides device memory and
streams only).
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# KVC_LIBRARY selects another build of the same ABI, e.g. the bounds-checking
# libkvc_debug.so
LIB_PATH = os.environ.get("KVC_LIBRARY") or os.path.join(_HERE, "libkvc.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libkvc.so is missing at {LIB_PATH}: build it with "
        "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")

_lib = C.CDLL(LIB_PATH)

KVC_OK = 0
KVC_F32, KVC_BF16 = 0, 1
DEV_TIMEOUT, DEV_BAD_SCORE, DEV_BAD_BUDGET, DEV_OUT_CAPACITY = 0x1, 0x2, 0x4, 0x8
VALUE_REUSE_SCORE_STATS = 0x1   # kvc_channel_prune_value_ex flag
DEV_INVARIANT = 0x10   # bounds-checking builds only


class KvcError(RuntimeError):
    def __init__(self, fn, code, msg):
        super().__init__(f"{fn} failed with status {code}: {msg}")
        self.code = code


class KvcShape(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("n_q_heads", C.c_int32), ("n_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("seq_len", C.c_int32), ("window", C.c_int32),
                ("dtype", C.c_int32)]


_p, _sz, _i32, _i64, _u32, _d = C.c_void_p, C.c_size_t, C.c_int32, C.c_int64, C.c_uint32, C.c_double
_sp = C.POINTER(KvcShape)
_SIGS = {
    "kvc_workspace_size": (_sz, [_sp, _i32]),
    "kvc_workspace_init": (C.c_int, [_p, _sz, _p]),
    "kvc_workspace_status": (C.c_int, [_p, _sz, C.POINTER(_u32), _p]),
    "kvc_score": (C.c_int, [_sp, _p, _p, _p, _p, _sz, _p]),
    "kvc_score_noalloc": (C.c_int, [_sp, _p, _p, _p, _p, _p]),
    "kvc_score_keyformer": (C.c_int, [_sp, _p, _p, C.c_uint64, _d, _p, _p, _sz, _p]),
    "kvc_compress_host": (C.c_int, [_sp, _p, _p, _p, _p, _p, _u32, _u32, _i64, _i32, _i32, _p, _p, _p,
                                    _p, _p, _p, _i64, _p, _sz, _p, _p]),
    "kvc_mba_budget": (C.c_int, [_sp, _p, _u32, _u32, _i64, _i32, _p, _p, _p, _sz, _p]),
    "kvc_topk_select": (C.c_int, [_sp, _p, _p, _i32, _p, _p, _sz, _p]),
    "kvc_pool_scores": (C.c_int, [_sp, _p, _i32, _i32, _p, _p, _sz, _p]),
    "kvc_head_budget": (C.c_int, [_sp, _p, _p, _p, _p, _sz, _p]),
    "kvc_topk_select_heads": (C.c_int, [_sp, _p, _p, _i32, _p, _p, _sz, _p]),
    "kvc_threshold_select": (C.c_int, [_sp, _p, C.c_float, _i32, _p, _p, _p, _sz, _p]),
    "kvc_compact_heads": (C.c_int, [_sp, _p, _p, _p, _p, _i32, _p, _p, _i64, _p, _sz, _p]),
    "kvc_compact": (C.c_int, [_sp, _p, _p, _p, _p, _i32, _p, _p, _i64, _p, _sz, _p]),
    "kvc_channel_prune": (C.c_int, [_sp, _p, _p, _d, _p, _p, _i64, _p, _sz, _p]),
    "kvc_channel_prune_query": (C.c_int, [_sp, _p, _p, _p, _d, _p, _p, _i64, _p, _sz, _p]),
    "kvc_channel_prune_value": (C.c_int, [_sp, _p, _p, _p, _p, _p, _d, _p, _p, _p, _i64, _p, _sz,
                                          _p]),
    "kvc_channel_prune_value_ex": (C.c_int, [_sp, _p, _p, _p, _p, _p, _d, _p, _p, _p, _i64,
                                             C.c_uint32, _p, _sz, _p]),
    "kvc_keep_channels": (_i32, [_d, _i32]),
    "kvc_status_string": (C.c_char_p, [C.c_int]),
    "kvc_last_error": (C.c_char_p, []),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args


def _check(fn, rc):
    if rc != KVC_OK:
        raise KvcError(fn, rc, _lib.kvc_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libkvc takes device tensors")
    if not t.is_contiguous():
        raise ValueError("libkvc takes contiguous tensors")
    return C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def shape(n_layers, n_q_heads, n_kv_heads, head_dim, seq_len, window, dtype) -> KvcShape:
    if isinstance(dtype, torch.dtype):
        dt = KVC_F32 if dtype == torch.float32 else KVC_BF16
    else:
        dt = KVC_F32 if dtype in ("f32", KVC_F32) else KVC_BF16
    return KvcShape(n_layers, n_q_heads, n_kv_heads, head_dim, seq_len, window, dt)


def shape_of(wl) -> KvcShape:
    """KvcShape of a workloads.Workload."""
    return shape(wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.seq_len, wl.window,
                 wl.dtype)


# --- the C ABI, one Python function per entry point -------------------------

def kvc_workspace_size(s: KvcShape, k_max: int = 0) -> int:
    n = _lib.kvc_workspace_size(C.byref(s), int(k_max))
    if n == 0:
        raise KvcError("kvc_workspace_size", -1, _lib.kvc_last_error().decode())
    return n


def kvc_workspace_init(ws: torch.Tensor, stream=None) -> None:
    _check("kvc_workspace_init", _lib.kvc_workspace_init(_ptr(ws), ws.numel(), _stream(stream)))


def kvc_workspace_status(ws: torch.Tensor, stream=None) -> int:
    out = _u32(0)
    _check("kvc_workspace_status",
           _lib.kvc_workspace_status(_ptr(ws), ws.numel(), C.byref(out), _stream(stream)))
    return out.value


def kvc_score(s: KvcShape, q_obs, k, scores, ws, stream=None) -> None:
    _check("kvc_score", _lib.kvc_score(C.byref(s), _ptr(q_obs), _ptr(k), _ptr(scores), _ptr(ws),
                                       ws.numel(), _stream(stream)))


def kvc_score_noalloc(s: KvcShape, q_obs, k, scores, dev_status=None, stream=None) -> None:
    """kvc_score without a workspace, for callers that may not allocate device
    memory: scratch comes from a fixed array inside the library (see kvc.h).
    Calls that overlap on the GPU race on that array; keep them on one
    stream."""
    _check("kvc_score_noalloc", _lib.kvc_score_noalloc(
        C.byref(s), _ptr(q_obs), _ptr(k), _ptr(scores), _ptr(dev_status), _stream(stream)))


def _hptr(t: torch.Tensor):
    if t.is_cuda or not t.is_pinned():
        raise ValueError("kvc_compress_host takes pinned host tensors for q/k/v")
    return C.c_void_p(t.data_ptr())


def kvc_compress_host(s: KvcShape, q_host, k_host, v_host, q_dev, k_dev, mass_num: int,
                      mass_den: int, total_budget: int, layer_floor: int, k_max: int, scores, mba,
                      budget, idx, k_out, v_out, ws, stream=None, copy_stream=None) -> None:
    """Whole default path from pinned host Q/K/V: K copied layer by layer on
    copy_stream while earlier layers are scored on stream; V rows read in
    place through the device mapping."""
    if copy_stream is None:
        raise ValueError("kvc_compress_host needs a copy stream")
    _check("kvc_compress_host", _lib.kvc_compress_host(
        C.byref(s), _hptr(q_host), _hptr(k_host), _hptr(v_host), _ptr(q_dev), _ptr(k_dev),
        int(mass_num), int(mass_den), int(total_budget), int(layer_floor), int(k_max),
        _ptr(scores), _ptr(mba), _ptr(budget), _ptr(idx), _ptr(k_out), _ptr(v_out),
        k_out.shape[0], _ptr(ws), ws.numel(), _stream(stream), _stream(copy_stream)))


def kvc_score_keyformer(s: KvcShape, q_obs, k, seed: int, tau: float, scores, ws,
                        stream=None) -> None:
    """Keyformer window scores: Gumbel-noised logits, temperature tau."""
    _check("kvc_score_keyformer", _lib.kvc_score_keyformer(
        C.byref(s), _ptr(q_obs), _ptr(k), int(seed) & 0xFFFFFFFFFFFFFFFF, float(tau),
        _ptr(scores), _ptr(ws), ws.numel(), _stream(stream)))


def kvc_mba_budget(s: KvcShape, scores, mass_num: int, mass_den: int, total_budget: int,
                   layer_floor: int, mba, budget, ws, stream=None) -> None:
    _check("kvc_mba_budget", _lib.kvc_mba_budget(
        C.byref(s), _ptr(scores), int(mass_num), int(mass_den), int(total_budget),
        int(layer_floor), _ptr(mba), _ptr(budget), _ptr(ws), ws.numel(), _stream(stream)))


def kvc_topk_select(s: KvcShape, scores, budget, k_max: int, idx, ws, stream=None) -> None:
    _check("kvc_topk_select", _lib.kvc_topk_select(
        C.byref(s), _ptr(scores), _ptr(budget), int(k_max), _ptr(idx), _ptr(ws), ws.numel(),
        _stream(stream)))


def kvc_pool_scores(s: KvcShape, scores, kernel: int, mode: int, pooled, ws, stream=None) -> None:
    """SnapKV 1D pooling of the prefix scores (mode 0 average, 1 max)."""
    _check("kvc_pool_scores", _lib.kvc_pool_scores(
        C.byref(s), _ptr(scores), int(kernel), int(mode), _ptr(pooled), _ptr(ws), ws.numel(),
        _stream(stream)))


def kvc_head_budget(s: KvcShape, mba, budget, head_budget, ws, stream=None) -> None:
    """Per-head split of each layer's budget by MBA (head_budget [L][H_kv])."""
    _check("kvc_head_budget", _lib.kvc_head_budget(
        C.byref(s), _ptr(mba), _ptr(budget), _ptr(head_budget), _ptr(ws), ws.numel(),
        _stream(stream)))


def kvc_topk_select_heads(s: KvcShape, scores, head_budget, k_max: int, idx, ws,
                          stream=None) -> None:
    _check("kvc_topk_select_heads", _lib.kvc_topk_select_heads(
        C.byref(s), _ptr(scores), _ptr(head_budget), int(k_max), _ptr(idx), _ptr(ws), ws.numel(),
        _stream(stream)))


def kvc_threshold_select(s: KvcShape, scores, tau: float, k_max: int, idx, counts, ws,
                         stream=None) -> None:
    """Keep every prefix position whose score is >= tau (plus the window)."""
    _check("kvc_threshold_select", _lib.kvc_threshold_select(
        C.byref(s), _ptr(scores), float(tau), int(k_max), _ptr(idx), _ptr(counts), _ptr(ws),
        ws.numel(), _stream(stream)))


def kvc_compact_heads(s: KvcShape, k, v, idx, counts, k_max: int, k_out, v_out, ws,
                      stream=None) -> None:
    _check("kvc_compact_heads", _lib.kvc_compact_heads(
        C.byref(s), _ptr(k), _ptr(v), _ptr(idx), _ptr(counts), int(k_max), _ptr(k_out),
        _ptr(v_out), k_out.shape[0], _ptr(ws), ws.numel(), _stream(stream)))


def kvc_compact(s: KvcShape, k, v, idx, budget, k_max: int, k_out, v_out, ws, stream=None) -> None:
    _check("kvc_compact", _lib.kvc_compact(
        C.byref(s), _ptr(k), _ptr(v), _ptr(idx), _ptr(budget), int(k_max), _ptr(k_out),
        _ptr(v_out), k_out.shape[0], _ptr(ws), ws.numel(), _stream(stream)))


def kvc_channel_prune(s: KvcShape, k_out, budget, lam: float, chan, k_pruned, ws,
                      stream=None) -> None:
    _check("kvc_channel_prune", _lib.kvc_channel_prune(
        C.byref(s), _ptr(k_out), _ptr(budget), float(lam), _ptr(chan), _ptr(k_pruned),
        k_pruned.numel(), _ptr(ws), ws.numel(), _stream(stream)))


def kvc_channel_prune_query(s: KvcShape, q_obs, k_out, budget, lam: float, chan, k_pruned, ws,
                            stream=None) -> None:
    """ThinK query-driven key-channel criterion (window-query x kept-key norms)."""
    _check("kvc_channel_prune_query", _lib.kvc_channel_prune_query(
        C.byref(s), _ptr(q_obs), _ptr(k_out), _ptr(budget), float(lam), _ptr(chan),
        _ptr(k_pruned), k_pruned.numel(), _ptr(ws), ws.numel(), _stream(stream)))


def kvc_channel_prune_value(s: KvcShape, q_obs, k, v, v_out, budget, lam: float, chan, v_pruned,
                            ws, value_scores=None, stream=None, reuse_score_stats=False) -> None:
    """THINKV: rank value channels by the squared column norms of the window
    rows' attention output and keep the top floor((1-lam) D) of the kept
    prefix rows of v_out (see kvc.h).  reuse_score_stats: take the window
    rows' softmax normalisers the last kvc_score over the same shape, q_obs
    and k left in ws (kvc_channel_prune_value_ex, KVC_VALUE_REUSE_SCORE_STATS)."""
    if reuse_score_stats:
        kvc_channel_prune_value_ex(s, q_obs, k, v, v_out, budget, lam, chan, v_pruned,
                                   VALUE_REUSE_SCORE_STATS, ws, value_scores, stream)
        return
    _check("kvc_channel_prune_value", _lib.kvc_channel_prune_value(
        C.byref(s), _ptr(q_obs), _ptr(k), _ptr(v), _ptr(v_out), _ptr(budget), float(lam),
        _ptr(value_scores), _ptr(chan), _ptr(v_pruned), v_pruned.numel(), _ptr(ws), ws.numel(),
        _stream(stream)))


def kvc_channel_prune_value_ex(s: KvcShape, q_obs, k, v, v_out, budget, lam: float, chan,
                               v_pruned, flags: int, ws, value_scores=None, stream=None) -> None:
    """kvc_channel_prune_value with flags (VALUE_REUSE_SCORE_STATS; see kvc.h)."""
    _check("kvc_channel_prune_value_ex", _lib.kvc_channel_prune_value_ex(
        C.byref(s), _ptr(q_obs), _ptr(k), _ptr(v), _ptr(v_out), _ptr(budget), float(lam),
        _ptr(value_scores), _ptr(chan), _ptr(v_pruned), v_pruned.numel(), int(flags), _ptr(ws),
        ws.numel(), _stream(stream)))


def kvc_keep_channels(lam: float, head_dim: int) -> int:
    return int(_lib.kvc_keep_channels(float(lam), int(head_dim)))


def kvc_status_string(code: int) -> str:
    return _lib.kvc_status_string(int(code)).decode()


def kvc_last_error() -> str:
    return _lib.kvc_last_error().decode()


# --- buffers for one prompt -------------------------------------------------

@dataclass
class Buffers:
    """Device buffers for the whole path on one prompt shape.  Output row
    capacity is sized for the largest packed result the budgets allow:
    H_kv * (min(total, L*P) + L*W) rows."""
    shape: KvcShape
    k_max: int
    ws: torch.Tensor
    scores: torch.Tensor
    mba: torch.Tensor
    budget: torch.Tensor
    idx: torch.Tensor
    k_out: torch.Tensor
    v_out: torch.Tensor
    chan: Optional[torch.Tensor] = None
    k_pruned: Optional[torch.Tensor] = None
    keep: int = 0
    pooled: Optional[torch.Tensor] = None


def alloc_buffers(s: KvcShape, total_budget: int, k_max: int, lam: Optional[float] = None,
                  device="cuda") -> Buffers:
    L, H, T, W, D = s.n_layers, s.n_kv_heads, s.seq_len, s.window, s.head_dim
    P = T - W
    dt = torch.float32 if s.dtype == KVC_F32 else torch.bfloat16
    ws_bytes = kvc_workspace_size(s, k_max)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
    kept_rows = min(int(total_budget), L * P)
    rows = H * (kept_rows + L * W)
    b = Buffers(
        shape=s, k_max=int(k_max), ws=ws,
        scores=torch.empty((L, H, T), dtype=torch.float32, device=device),
        mba=torch.empty((L, H), dtype=torch.int32, device=device),
        budget=torch.empty(L, dtype=torch.int32, device=device),
        idx=torch.empty((L, H, max(1, int(k_max))), dtype=torch.int32, device=device),
        k_out=torch.empty((rows, D), dtype=dt, device=device),
        v_out=torch.empty((rows, D), dtype=dt, device=device))
    if lam is not None:
        b.keep = kvc_keep_channels(lam, D)
        b.chan = torch.empty((L, H, max(1, b.keep)), dtype=torch.int32, device=device)
        b.k_pruned = torch.empty(max(1, H * kept_rows * b.keep), dtype=dt, device=device)
    kvc_workspace_init(ws)
    return b


def compress(b: Buffers, q_obs, k, v, total_budget: int, layer_floor: int, mass_num: int = 9,
             mass_den: int = 10, lam: Optional[float] = None, stream=None,
             pool_kernel: int = 0, pool_mode: int = 0, think: str = "magnitude") -> None:
    """Enqueue the whole path: score -> MBA/budget -> (pool ->) top-K -> compact
    (-> channel prune when lam is given, by key magnitude or, with
    think="query", by the query-driven criterion).  pool_kernel > 1 pools the
    scores before top-K (MBA stays on the raw scores).  Asynchronous on
    `stream`."""
    s = b.shape
    kvc_score(s, q_obs, k, b.scores, b.ws, stream)
    kvc_mba_budget(s, b.scores, mass_num, mass_den, total_budget, layer_floor, b.mba, b.budget,
                   b.ws, stream)
    sel = b.scores
    if pool_kernel > 1:
        if getattr(b, "pooled", None) is None:
            b.pooled = torch.empty_like(b.scores)
        kvc_pool_scores(s, b.scores, pool_kernel, pool_mode, b.pooled, b.ws, stream)
        sel = b.pooled
    kvc_topk_select(s, sel, b.budget, b.k_max, b.idx, b.ws, stream)
    kvc_compact(s, k, v, b.idx, b.budget, b.k_max, b.k_out, b.v_out, b.ws, stream)
    if lam is not None:
        if think == "query":
            kvc_channel_prune_query(s, q_obs, b.k_out, b.budget, lam, b.chan, b.k_pruned, b.ws,
                                    stream)
        elif think == "magnitude":
            kvc_channel_prune(s, b.k_out, b.budget, lam, b.chan, b.k_pruned, b.ws, stream)
        else:
            raise ValueError(f"unknown ThinK criterion {think!r}")
