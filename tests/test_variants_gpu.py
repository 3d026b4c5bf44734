"""GPU parity of the optional allocation/selection variants against the
oracle, stage-isolated on the GPU's own fp32 scores (bit-exact: integer and
index work and byte copies):
  per-head budgets inside a layer (kvc_head_budget), top-K with per-head
  budgets (kvc_topk_select_heads), threshold selection with the recent window
  (kvc_threshold_select) and compaction with per-head counts
  (kvc_compact_heads)."""
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


def oshape(wl):
    return O().shape_of(wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.seq_len,
                        wl.window, wl.dtype)


CASES = {
    "bf16_rows512": (wk.ZIGZAG_32K.scaled(
        n_layers=3, n_kv_heads=4, n_q_heads=16, seq_len=3000, total_budget=3 * 500,
        layer_floor=60, temperature=(0.3, 3.0)), 51),
    "f32_odd": (wk.ZIGZAG_32K.scaled(
        n_layers=2, n_kv_heads=3, n_q_heads=6, head_dim=80, seq_len=700, window=16,
        total_budget=2 * 200, layer_floor=20, temperature=None, dtype="f32"), 52),
}


def _scores_and_budgets(wl, seed):
    kvc = K()
    x = wk.make_inputs(wl, seed, device="cuda")
    s = kvc.shape_of(wl)
    P = wl.seq_len - wl.window
    ws = torch.empty(kvc.kvc_workspace_size(s, P), dtype=torch.uint8, device="cuda")
    kvc.kvc_workspace_init(ws)
    L, H, T = wl.n_layers, wl.n_kv_heads, wl.seq_len
    sc = torch.empty((L, H, T), device="cuda")
    mba = torch.empty((L, H), dtype=torch.int32, device="cuda")
    bud = torch.empty(L, dtype=torch.int32, device="cuda")
    total, floor = wl.budget_args()
    kvc.kvc_score(s, x["q"], x["k"], sc, ws)
    kvc.kvc_mba_budget(s, sc, wl.mass_num, wl.mass_den, total, floor, mba, bud, ws)
    return kvc, s, ws, x, sc, mba, bud


def _check_compaction(wl, x, idx, counts, k_max, k_out, v_out):
    o = O()
    s = oshape(wl)
    ci = counts.cpu().numpy()
    ii = idx.cpu().numpy()
    want_k = o.compact_heads(s, x["k"], ii, ci, k_max)
    want_v = o.compact_heads(s, x["v"], ii, ci, k_max)
    rows = want_k.shape[0]
    assert np.array_equal(o.raw(k_out[:rows]), want_k), "K"
    assert np.array_equal(o.raw(v_out[:rows]), want_v), "V"


@pytest.mark.parametrize("name", list(CASES))
def test_head_budget_topk_compact(name):
    wl, seed = CASES[name]
    kvc, s, ws, x, sc, mba, bud = _scores_and_budgets(wl, seed)
    o = O()
    L, H, P, W, D = wl.n_layers, wl.n_kv_heads, wl.seq_len - wl.window, wl.window, wl.head_dim
    hb = torch.empty((L, H), dtype=torch.int32, device="cuda")
    kvc.kvc_head_budget(s, mba, bud, hb, ws)
    torch.cuda.synchronize()
    want = o.head_budget(mba.cpu().numpy(), bud.cpu().numpy(), P)
    assert np.array_equal(hb.cpu().numpy(), want)
    assert np.array_equal(want.sum(axis=1), H * bud.cpu().numpy().astype(np.int64))
    k_max = int(want.max())
    idx = torch.full((L, H, k_max), -1, dtype=torch.int32, device="cuda")
    kvc.kvc_topk_select_heads(s, sc, hb, k_max, idx, ws)
    torch.cuda.synchronize()
    widx = o.topk_heads(s_o := oshape(wl), sc.cpu().numpy(), want, k_max)
    gi = idx.cpu().numpy()
    for l in range(L):
        for h in range(H):
            n = want[l, h]
            assert np.array_equal(gi[l, h, :n], widx[l, h, :n]), (l, h)
    rows = int((want + W).sum())
    dt = x["k"].dtype
    k_out = torch.empty((rows, D), dtype=dt, device="cuda")
    v_out = torch.empty((rows, D), dtype=dt, device="cuda")
    kvc.kvc_compact_heads(s, x["k"], x["v"], idx, hb, k_max, k_out, v_out, ws)
    torch.cuda.synchronize()
    assert kvc.kvc_workspace_status(ws) == 0
    _check_compaction(wl, x, idx, hb, k_max, k_out, v_out)


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("tau_mult", [0.0, 1.0, 4.0, 1e9])
def test_threshold_select_compact(name, tau_mult):
    wl, seed = CASES[name]
    kvc, s, ws, x, sc, _, _ = _scores_and_budgets(wl, seed)
    o = O()
    L, H, T, W, D = wl.n_layers, wl.n_kv_heads, wl.seq_len, wl.window, wl.head_dim
    P = T - W
    tau = float(np.float32(tau_mult / T))
    idx = torch.full((L, H, P), -1, dtype=torch.int32, device="cuda")
    cnt = torch.empty((L, H), dtype=torch.int32, device="cuda")
    kvc.kvc_threshold_select(s, sc, tau, P, idx, cnt, ws)
    torch.cuda.synchronize()
    assert kvc.kvc_workspace_status(ws) == 0
    widx, wcnt, over = o.threshold_select(oshape(wl), sc.cpu().numpy(), tau, P)
    assert not over
    assert np.array_equal(cnt.cpu().numpy(), wcnt)
    gi = idx.cpu().numpy()
    for l in range(L):
        for h in range(H):
            n = wcnt[l, h]
            assert np.array_equal(gi[l, h, :n], widx[l, h, :n]), (l, h)
    rows = int((wcnt + W).sum())
    dt = x["k"].dtype
    k_out = torch.empty((max(rows, 1), D), dtype=dt, device="cuda")
    v_out = torch.empty((max(rows, 1), D), dtype=dt, device="cuda")
    kvc.kvc_compact_heads(s, x["k"], x["v"], idx, cnt, P, k_out, v_out, ws)
    torch.cuda.synchronize()
    assert kvc.kvc_workspace_status(ws) == 0
    _check_compaction(wl, x, idx, cnt, P, k_out, v_out)


def test_threshold_overflow_sets_status_and_keeps_first():
    kvc = K()
    wl, seed = CASES["f32_odd"]
    kvc, s, ws, x, sc, _, _ = _scores_and_budgets(wl, seed)
    L, H, T, W = wl.n_layers, wl.n_kv_heads, wl.seq_len, wl.window
    P = T - W
    k_max = 37
    idx = torch.full((L, H, k_max), -1, dtype=torch.int32, device="cuda")
    cnt = torch.empty((L, H), dtype=torch.int32, device="cuda")
    kvc.kvc_threshold_select(s, sc, 0.0, k_max, idx, cnt, ws)
    torch.cuda.synchronize()
    assert kvc.kvc_workspace_status(ws) & kvc.DEV_BAD_BUDGET
    assert (cnt == P).all()
    assert (idx == torch.arange(k_max, device="cuda", dtype=torch.int32)).all()


def test_full_32k_variants_sampled():
    """On the 32-layer 32K workload: per-head budgets over every layer, top-K
    on sampled heads, threshold selection over every head."""
    wl = wk.ZIGZAG_32K
    kvc, s, ws, x, sc, mba, bud = _scores_and_budgets(wl, wk.seed_for(2))
    o = O()
    L, H, T, W = wl.n_layers, wl.n_kv_heads, wl.seq_len, wl.window
    P = T - W
    hb = torch.empty((L, H), dtype=torch.int32, device="cuda")
    kvc.kvc_head_budget(s, mba, bud, hb, ws)
    torch.cuda.synchronize()
    want = o.head_budget(mba.cpu().numpy(), bud.cpu().numpy(), P)
    assert np.array_equal(hb.cpu().numpy(), want)
    k_max = int(want.max())
    idx = torch.full((L, H, k_max), -1, dtype=torch.int32, device="cuda")
    kvc.kvc_topk_select_heads(s, sc, hb, k_max, idx, ws)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    scn = sc.cpu().numpy()
    for _ in range(4):
        l, h = int(rng.integers(L)), int(rng.integers(H))
        n = int(want[l, h])
        ref = o.topk(scn[l, h].astype(np.float64), P, n)
        assert np.array_equal(idx[l, h, :n].cpu().numpy(), ref)
    tau = float(np.float32(4.0 / T))
    tidx = torch.full((L, H, P), -1, dtype=torch.int32, device="cuda")
    cnt = torch.empty((L, H), dtype=torch.int32, device="cuda")
    kvc.kvc_threshold_select(s, sc, tau, P, tidx, cnt, ws)
    torch.cuda.synchronize()
    widx, wcnt, _ = o.threshold_select(oshape(wl), scn, tau, P)
    assert np.array_equal(cnt.cpu().numpy(), wcnt)
    gi = tidx.cpu().numpy()
    for l in range(L):
        for h in range(H):
            assert np.array_equal(gi[l, h, :wcnt[l, h]], widx[l, h, :wcnt[l, h]])
    assert kvc.kvc_workspace_status(ws) == 0
