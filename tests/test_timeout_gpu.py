"""A device wait that runs out.  With KVC_TEST_SKIP_ARRIVE=1 the odd CTA of
every SM pair withholds one arrival in score pass 1 (a barrier that nothing
completes), so the pair's bounded waits (1 s) expire: the call must record
KVC_DEV_TIMEOUT in the workspace status word, return within seconds, and
leave the context usable -- the next call, without the knob, gives the
oracle's scores."""
import time

import numpy as np
import pytest
import torch

from eviction_kvc_score_gb300 import workloads as wk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def test_withheld_arrival_times_out_and_context_recovers(monkeypatch):
    from eviction_kvc_score_gb300 import kvc
    from oracle import oracle as O

    wl = wk.ZIGZAG_32K.scaled(n_layers=1, n_kv_heads=2, n_q_heads=8, seq_len=1500,
                              total_budget=300, layer_floor=40, temperature=None)
    x = wk.make_inputs(wl, 41, device="cuda")
    s = kvc.shape_of(wl)
    total, _ = wl.budget_args()
    b = kvc.alloc_buffers(s, total, wl.k_max)
    monkeypatch.setenv("KVC_SCORE_IMPL", "tc")
    monkeypatch.setenv("KVC_TEST_SKIP_ARRIVE", "1")
    t0 = time.time()
    kvc.kvc_score(s, x["q"], x["k"], b.scores, b.ws)
    torch.cuda.synchronize()
    took = time.time() - t0
    assert kvc.kvc_workspace_status(b.ws) & kvc.DEV_TIMEOUT
    assert took < 30.0

    monkeypatch.delenv("KVC_TEST_SKIP_ARRIVE")
    kvc.kvc_workspace_init(b.ws)
    kvc.kvc_score(s, x["q"], x["k"], b.scores, b.ws)
    torch.cuda.synchronize()
    assert kvc.kvc_workspace_status(b.ws) == 0
    ora = O.score(O.shape_of(wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim,
                             wl.seq_len, wl.window, wl.dtype), x["q"], x["k"])
    got = b.scores.double().cpu().numpy()
    assert (np.abs(got - ora) <= 1e-3 * ora + 1e-30).all()
