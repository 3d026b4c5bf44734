"""The bounds-checking build (libkvc_debug.so, compiled with KVC_DEBUG_BOUNDS):
its kernels verify their outputs' invariants and record KVC_DEV_INVARIANT in
the status word instead of trapping.  On valid inputs it must give the release
build's bytes with a clean status; on a planted violation (caller indices out
of order) it must set the bit, where the release build copies as told.

The debug library runs in a child process (KVC_LIBRARY selects it), so this
process keeps the release library."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from eviction_kvc_score_gb300 import workloads as wk

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys
import numpy as np, torch
from eviction_kvc_score_gb300 import kvc, workloads as wk
wl = wk.ZIGZAG_32K.scaled(n_layers=3, n_kv_heads=2, n_q_heads=8, seq_len=2100,
                          total_budget=3 * 400, layer_floor=50, think_lambda=0.4)
torch.cuda.set_device(0)
x = wk.make_inputs(wl, 91, device="cuda")
total, floor = wl.budget_args()
b = kvc.alloc_buffers(kvc.shape_of(wl), total, wl.k_max, lam=wl.think_lambda)
kvc.compress(b, x["q"], x["k"], x["v"], total, floor, wl.mass_num, wl.mass_den,
             lam=wl.think_lambda)
torch.cuda.synchronize()
import hashlib
def digest(t):
    return hashlib.sha256(t.contiguous().cpu().view(torch.uint8).numpy().tobytes()).hexdigest()
n = b.budget.cpu().clamp(0, wl.prefix_len).tolist()
rows = wl.n_kv_heads * (sum(n) + wl.n_layers * wl.window)
out = {"status": kvc.kvc_workspace_status(b.ws),
       "digest": {"scores": digest(b.scores), "mba": digest(b.mba), "budget": digest(b.budget),
                  "idx": [digest(b.idx[l, :, : n[l]]) for l in range(wl.n_layers)],
                  "k_out": digest(b.k_out[:rows]), "v_out": digest(b.v_out[:rows]),
                  "chan": digest(b.chan),
                  "k_pruned": digest(b.k_pruned[: wl.n_kv_heads * sum(n) * b.keep])}}
# planted: descending caller indices for the compaction
s1 = kvc.shape(1, 2, 2, 16, 300, 4, "f32")
ws = torch.empty(kvc.kvc_workspace_size(s1, 50), dtype=torch.uint8, device="cuda")
kvc.kvc_workspace_init(ws)
kk = torch.randn((1, 2, 300, 16), device="cuda")
idx = torch.arange(50, 0, -1, dtype=torch.int32, device="cuda").repeat(2, 1).view(1, 2, 50)
k_out = torch.empty((2 * (50 + 4), 16), device="cuda")
v_out = torch.empty_like(k_out)
kvc.kvc_compact(s1, kk, kk, idx, torch.tensor([50], dtype=torch.int32, device="cuda"), 50,
                k_out, v_out, ws)
out["planted_status"] = kvc.kvc_workspace_status(ws)
print(json.dumps(out))
"""


def _run(lib):
    env = dict(os.environ)
    if lib:
        env["KVC_LIBRARY"] = lib
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    from eviction_kvc_score_gb300 import build
    return build.LIB, build.build(debug_bounds=True)


def test_debug_build_matches_release_and_flags_planted_violation(libs):
    from eviction_kvc_score_gb300 import kvc
    rel, dbg = _run(None), _run(libs[1])
    # valid inputs: clean status, the same outputs
    assert rel["status"] == 0 and dbg["status"] == 0
    assert rel["digest"] == dbg["digest"]
    # planted descending indices: flagged by the checks, copied by the release build
    assert dbg["planted_status"] & kvc.DEV_INVARIANT
    assert not rel["planted_status"] & kvc.DEV_INVARIANT
