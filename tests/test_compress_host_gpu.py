"""kvc_compress_host: the default path fed from pinned host buffers (K copied
layer by layer against the scoring, V rows read in place through the device
mapping).  Scores against the oracle within 1e-3 relative; MBA, budgets, top-K
and compacted bytes bit-exact against the oracle run on the GPU's own scores;
two calls in a row on the same buffers give the same bytes."""
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


def K():
    from eviction_kvc_score_gb300 import kvc
    return kvc


def O():
    from oracle import oracle
    return oracle


CASES = {
    "bf16_tc": (wk.ZIGZAG_32K.scaled(n_layers=3, n_kv_heads=2, n_q_heads=8, seq_len=2100,
                                     total_budget=3 * 400, layer_floor=50,
                                     temperature=(0.3, 3.0)), 61),
    "f32_simt": (wk.ZIGZAG_32K.scaled(n_layers=2, n_kv_heads=2, n_q_heads=4, head_dim=80,
                                      seq_len=333, window=8, total_budget=2 * 60, layer_floor=10,
                                      temperature=None, dtype="f32"), 62),
}


def _run(wl, x):
    kvc = K()
    total, floor = wl.budget_args()
    b = kvc.alloc_buffers(kvc.shape_of(wl), total, wl.k_max)
    hin = {k: x[k].cpu().pin_memory() for k in ("q", "k", "v")}
    q_dev, k_dev = torch.empty_like(x["q"]), torch.empty_like(x["k"])
    copy_stream = torch.cuda.Stream()
    kvc.kvc_compress_host(b.shape, hin["q"], hin["k"], hin["v"], q_dev, k_dev, wl.mass_num,
                          wl.mass_den, total, floor, b.k_max, b.scores, b.mba, b.budget, b.idx,
                          b.k_out, b.v_out, b.ws, copy_stream=copy_stream)
    torch.cuda.synchronize()
    assert kvc.kvc_workspace_status(b.ws) == 0
    return b, hin, q_dev, k_dev, copy_stream


@pytest.mark.parametrize("name", list(CASES))
def test_compress_host_matches_oracle(name):
    wl, seed = CASES[name]
    x = wk.make_inputs(wl, seed, device="cuda")
    b, *_ = _run(wl, x)
    o = O()
    s = o.shape_of(wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.seq_len, wl.window,
                   wl.dtype)
    want = o.score(s, x["q"], x["k"])
    got = b.scores.cpu().numpy().astype(np.float64)
    assert (np.abs(got - want) <= 1e-3 * want + 1e-30).all()
    total, floor = wl.budget_args()
    sc = b.scores.cpu().numpy()
    mba = o.mba_all(s, sc, wl.mass_num, wl.mass_den)
    assert np.array_equal(mba, b.mba.cpu().numpy())
    bud = o.budget(mba, wl.prefix_len, total, floor)
    assert np.array_equal(bud, b.budget.cpu().numpy())
    idx = o.topk_all(s, sc, bud, wl.k_max)
    gi = b.idx.cpu().numpy()
    for l in range(wl.n_layers):
        assert np.array_equal(gi[l, :, : bud[l]], idx[l, :, : bud[l]])
    rows = o.compact_rows(s, bud)
    assert np.array_equal(o.raw(b.k_out[:rows]), o.compact(s, x["k"], idx, bud, wl.k_max))
    assert np.array_equal(o.raw(b.v_out[:rows]), o.compact(s, x["v"], idx, bud, wl.k_max))


def test_compress_host_twice_in_a_row():
    kvc = K()
    wl, seed = CASES["bf16_tc"]
    x = wk.make_inputs(wl, seed, device="cuda")
    b, hin, q_dev, k_dev, cs = _run(wl, x)
    first = (b.k_out.clone(), b.v_out.clone(), b.idx.clone())
    total, floor = wl.budget_args()
    kvc.kvc_compress_host(b.shape, hin["q"], hin["k"], hin["v"], q_dev, k_dev, wl.mass_num,
                          wl.mass_den, total, floor, b.k_max, b.scores, b.mba, b.budget, b.idx,
                          b.k_out, b.v_out, b.ws, copy_stream=cs)
    torch.cuda.synchronize()
    assert torch.equal(first[0], b.k_out) and torch.equal(first[1], b.v_out)
    assert torch.equal(first[2], b.idx)


def test_compress_host_rejects_unmapped_or_device_inputs():
    kvc = K()
    wl, seed = CASES["f32_simt"]
    x = wk.make_inputs(wl, seed, device="cuda")
    total, floor = wl.budget_args()
    b = kvc.alloc_buffers(kvc.shape_of(wl), total, wl.k_max)
    cs = torch.cuda.Stream()
    pinned = {k: x[k].cpu().pin_memory() for k in ("q", "k")}
    with pytest.raises(ValueError):   # pageable V: refused by the binding
        kvc.kvc_compress_host(b.shape, pinned["q"], pinned["k"], x["v"].cpu(), x["q"], x["k"],
                              9, 10, total, floor, b.k_max, b.scores, b.mba, b.budget, b.idx,
                              b.k_out, b.v_out, b.ws, copy_stream=cs)
    with pytest.raises(ValueError):
        kvc.kvc_compress_host(b.shape, pinned["q"], pinned["k"], x["v"], x["q"], x["k"], 9, 10,
                              total, floor, b.k_max, b.scores, b.mba, b.budget, b.idx, b.k_out,
                              b.v_out, b.ws, copy_stream=cs)


def test_compress_host_from_two_threads_with_separate_buffers():
    """Two prompts driven from two host threads on one device, each with its
    own staging buffers, streams and workspace, several calls each: both
    match the oracle (the calls keep no shared per-device state)."""
    import threading
    kvc = K()
    o = O()
    cases = [(CASES["bf16_tc"][0], 71),
             (CASES["bf16_tc"][0].scaled(n_layers=2, seq_len=3000, total_budget=2 * 500), 72)]
    runs = []
    for wl, seed in cases:
        x = wk.make_inputs(wl, seed, device="cuda")
        total, floor = wl.budget_args()
        b = kvc.alloc_buffers(kvc.shape_of(wl), total, wl.k_max)
        hin = {k: x[k].cpu().pin_memory() for k in ("q", "k", "v")}
        runs.append(dict(wl=wl, x=x, b=b, hin=hin, q_dev=torch.empty_like(x["q"]),
                         k_dev=torch.empty_like(x["k"]), stream=torch.cuda.Stream(),
                         copy_stream=torch.cuda.Stream()))
    torch.cuda.synchronize()
    errors = []

    def drive(r):
        try:
            wl, b, hin = r["wl"], r["b"], r["hin"]
            total, floor = wl.budget_args()
            for _ in range(3):
                kvc.kvc_compress_host(b.shape, hin["q"], hin["k"], hin["v"], r["q_dev"],
                                      r["k_dev"], wl.mass_num, wl.mass_den, total, floor,
                                      b.k_max, b.scores, b.mba, b.budget, b.idx, b.k_out,
                                      b.v_out, b.ws, stream=r["stream"],
                                      copy_stream=r["copy_stream"])
            r["stream"].synchronize()
        except Exception as e:       # surfaced in the main thread
            errors.append(e)

    th = [threading.Thread(target=drive, args=(r,)) for r in runs]
    for t in th:
        t.start()
    for t in th:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for r in runs:
        wl, b, x = r["wl"], r["b"], r["x"]
        assert kvc.kvc_workspace_status(b.ws) == 0
        s = o.shape_of(wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.seq_len,
                       wl.window, wl.dtype)
        want = o.score(s, x["q"], x["k"])
        got = b.scores.cpu().numpy().astype(np.float64)
        assert (np.abs(got - want) <= 1e-3 * want + 1e-30).all()
        total, floor = wl.budget_args()
        sc = b.scores.cpu().numpy()
        mba = o.mba_all(s, sc, wl.mass_num, wl.mass_den)
        bud = o.budget(mba, wl.prefix_len, total, floor)
        assert np.array_equal(bud, b.budget.cpu().numpy())
        idx = o.topk_all(s, sc, bud, wl.k_max)
        rows = o.compact_rows(s, bud)
        assert np.array_equal(o.raw(b.k_out[:rows]), o.compact(s, x["k"], idx, bud, wl.k_max))
        assert np.array_equal(o.raw(b.v_out[:rows]), o.compact(s, x["v"], idx, bud, wl.k_max))
