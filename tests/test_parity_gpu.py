"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle.

Rules (the oracle's scores are fp64; the GPU accumulates in fp32):
  scores       |c_gpu - c_ora| <= 1e-3 * c_ora + 1e-30 element by element,
               and every head's scores sum to 1 within 1e-5;
  MBA, budget, top-K indices, compacted K/V bytes, ThinK channels and pruned
  bytes: bit-exact against the oracle run on the GPU's own fp32 scores
  (stage-isolated) -- these are integer / byte decisions on identical inputs;
  ThinK channels may differ only where the oracle's two boundary norms are
  equal to within 1e-9 relative (the GPU sums squares in a float-float pair);
  end to end (oracle scores vs GPU scores): top-K may differ only at
  positions whose oracle score is within 1e-3 relative of the head's B-th
  largest oracle score, MBA only where the oracle's crossing mass is within
  1e-5 relative of the threshold.
"""
import math
import os

import numpy as np
import pytest
import torch

from eviction_kvc_score_gb300 import workloads as wk

pytestmark = pytest.mark.gpu

SCORE_RTOL = 1e-3
SCORE_ATOL = 1e-30


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


def run_gpu(wl, x, lam=None, impl=None):
    kvc = K()
    old = os.environ.get("KVC_SCORE_IMPL")
    if impl:
        os.environ["KVC_SCORE_IMPL"] = impl
    try:
        s = kvc.shape_of(wl)
        total, floor = wl.budget_args()
        b = kvc.alloc_buffers(s, total, wl.k_max, lam=lam)
        kvc.compress(b, x["q"], x["k"], x["v"], total, floor, wl.mass_num, wl.mass_den, lam=lam)
        torch.cuda.synchronize()
    finally:
        if impl:
            if old is None:
                os.environ.pop("KVC_SCORE_IMPL", None)
            else:
                os.environ["KVC_SCORE_IMPL"] = old
    assert kvc.kvc_workspace_status(b.ws) == 0
    return b


def assert_scores_close(gpu, ora):
    gpu = np.asarray(gpu, dtype=np.float64)
    bad = np.abs(gpu - ora) > SCORE_RTOL * ora + SCORE_ATOL
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{bad.sum()} scores out of tolerance, first at {tuple(i)}: "
                             f"gpu {gpu[tuple(i)]!r} oracle {ora[tuple(i)]!r}")


def check_discrete_stages(wl, x, b, lam=None, heads=None):
    """Oracle stages 2..6 on the GPU's own fp32 scores must match bit for bit."""
    o = O()
    s = oshape(wl)
    total, floor = wl.budget_args()
    sc = b.scores.cpu().numpy()
    mba = o.mba_all(s, sc, wl.mass_num, wl.mass_den)
    assert np.array_equal(mba, b.mba.cpu().numpy()), "MBA"
    bud = o.budget(mba, wl.prefix_len, total, floor)
    assert np.array_equal(bud, b.budget.cpu().numpy()), "budget"
    assert bud.sum() == min(total, wl.n_layers * wl.prefix_len) and bud.min() >= floor
    idx = o.topk_all(s, sc, bud, wl.k_max)
    gi = b.idx.cpu().numpy()
    for l in range(wl.n_layers):
        assert np.array_equal(gi[l, :, : bud[l]], idx[l, :, : bud[l]]), f"top-K layer {l}"
    rows = o.compact_rows(s, bud)
    assert np.array_equal(o.raw(b.k_out[:rows]), o.compact(s, x["k"], idx, bud, wl.k_max)), "K"
    assert np.array_equal(o.raw(b.v_out[:rows]), o.compact(s, x["v"], idx, bud, wl.k_max)), "V"
    if lam is not None:
        chan, norms, kp = o.channel_prune(s, o.raw(b.k_out[:rows]), bud, lam)
        gchan = b.chan.cpu().numpy()
        for l in range(wl.n_layers):
            for h in range(wl.n_kv_heads):
                if not np.array_equal(gchan[l, h], chan[l, h]):
                    # only a near-tie at the keep boundary may differ
                    srt = np.sort(norms[l, h])[::-1]
                    kth, nxt = srt[b.keep - 1], srt[b.keep]
                    assert abs(kth - nxt) <= 1e-9 * kth, f"ThinK channels layer {l} head {h}"
        if np.array_equal(gchan, chan):
            assert np.array_equal(kp, o.raw(b.k_pruned[: kp.size])), "pruned K"
    return bud


# --------------------------------------------------------------------------
# small cases: oracle over every unit
SMALL = {
    "tc_d128_rows512_ragged": (wk.ZIGZAG_32K.scaled(
        n_layers=2, n_kv_heads=2, n_q_heads=8, seq_len=1500, total_budget=2 * 300,
        layer_floor=40, temperature=(0.3, 3.0)), None, 31),
    "tc_d64_rows128": (wk.ZIGZAG_32K.scaled(
        n_layers=3, n_kv_heads=3, n_q_heads=6, head_dim=64, seq_len=777, window=64,
        total_budget=3 * 100, layer_floor=20), None, 32),
    "tc_rows48_tail16": (wk.ZIGZAG_32K.scaled(
        n_layers=2, n_kv_heads=2, n_q_heads=6, seq_len=300, window=16, total_budget=2 * 50,
        layer_floor=5, temperature=None), None, 33),
    "tc_rows256_think": (wk.ZIGZAG_32K.scaled(
        n_layers=2, n_kv_heads=2, n_q_heads=8, seq_len=4100, window=64,
        total_budget=2 * 820, layer_floor=102, temperature=None), 0.4, 34),
    # 384 window rows: the second 256-row job of a tile is half padding (the
    # odd CTA's rows), so pass 1 skips that CTA's share and pass 2 has a
    # warpgroup with no real columns; T = 2000 leaves a ragged last tile
    "tc_rows384_pad_job": (wk.ZIGZAG_32K.scaled(
        n_layers=2, n_kv_heads=2, n_q_heads=8, seq_len=2000, window=96,
        total_budget=2 * 380, layer_floor=30, temperature=(0.5, 2.0)), None, 37),
    "tiny_mha_f32": (wk.TINY, None, wk.seed_for(0)),
    "simt_odd_dim": (wk.ZIGZAG_32K.scaled(
        n_layers=2, n_kv_heads=2, n_q_heads=4, head_dim=80, seq_len=333, window=8,
        total_budget=2 * 60, layer_floor=10, temperature=None), 0.25, 35),
    "prefix_of_one": (wk.ZIGZAG_32K.scaled(
        n_layers=2, n_kv_heads=1, n_q_heads=2, seq_len=33, window=32, total_budget=2,
        layer_floor=0, temperature=None), None, 36),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_small_parity(name):
    wl, lam, seed = SMALL[name]
    x = wk.make_inputs(wl, seed, device="cuda")
    b = run_gpu(wl, x, lam=lam)
    ora = O().score(oshape(wl), x["q"], x["k"])
    assert_scores_close(b.scores.cpu().numpy(), ora)
    np.testing.assert_allclose(b.scores.double().sum(-1).cpu().numpy(), 1.0, atol=1e-5)
    check_discrete_stages(wl, x, b, lam=lam)


@pytest.mark.parametrize("name", ["tc_d128_rows512_ragged", "tc_rows48_tail16"])
def test_simt_path_matches_oracle_on_bf16(name):
    wl, lam, seed = SMALL[name]
    x = wk.make_inputs(wl, seed, device="cuda")
    b = run_gpu(wl, x, lam=lam, impl="simt")
    assert_scores_close(b.scores.cpu().numpy(), O().score(oshape(wl), x["q"], x["k"]))
    check_discrete_stages(wl, x, b, lam=lam)


def test_end_to_end_against_oracle_chain():
    """Oracle's own chain (its fp64 scores) vs the GPU chain, with the
    near-tie allowances."""
    wl, _, seed = SMALL["tc_d128_rows512_ragged"]
    x = wk.make_inputs(wl, seed, device="cuda")
    b = run_gpu(wl, x)
    o = O()
    total, floor = wl.budget_args()
    ref = o.compress(oshape(wl), x["q"], x["k"], x["v"], total, floor, wl.k_max)
    assert_scores_close(b.scores.cpu().numpy(), ref["scores"])
    gm = b.mba.cpu().numpy()
    for (l, h), m in np.ndenumerate(ref["mba"]):
        if gm[l, h] != m:
            c = np.sort(ref["scores"][l, h])[::-1]
            cum = np.cumsum(c)
            thr = 0.9 * cum[-1]
            assert abs(cum[m - 1] - thr) <= 1e-5 * thr or abs(cum[gm[l, h] - 1] - thr) <= 1e-5 * thr
    if np.array_equal(gm, ref["mba"]):
        assert np.array_equal(b.budget.cpu().numpy(), ref["budget"])
    bud = b.budget.cpu().numpy()
    gi = b.idx.cpu().numpy()
    P = wl.prefix_len
    for l in range(wl.n_layers):
        n = bud[l]
        for h in range(wl.n_kv_heads):
            oi = set(o.topk(ref["scores"][l, h, :P], P, n).tolist())
            diff = oi ^ set(gi[l, h, :n].tolist())
            if diff:
                kth = np.sort(ref["scores"][l, h, :P])[::-1][n - 1]
                for j in diff:
                    assert abs(ref["scores"][l, h, j] - kth) <= 1e-3 * kth


def test_runs_are_deterministic():
    wl, lam, seed = SMALL["tc_rows256_think"]
    x = wk.make_inputs(wl, seed, device="cuda")
    a = run_gpu(wl, x, lam=lam)
    b = run_gpu(wl, x, lam=lam)
    for f in ("scores", "mba", "budget", "chan"):
        assert torch.equal(getattr(a, f), getattr(b, f)), f
    n = a.budget.cpu().clamp(0, wl.prefix_len).tolist()
    for l in range(wl.n_layers):          # entries past n_l are never written
        assert torch.equal(a.idx[l, :, : n[l]], b.idx[l, :, : n[l]])
    rows = wl.n_kv_heads * (sum(n) + wl.n_layers * wl.window)
    assert torch.equal(a.k_out[:rows], b.k_out[:rows]) and torch.equal(a.v_out[:rows], b.v_out[:rows])
    used = wl.n_kv_heads * sum(n) * a.keep
    assert torch.equal(a.k_pruned[:used], b.k_pruned[:used])


# --------------------------------------------------------------------------
# discrete stages on constructed score vectors (edge cases)
def _stage_buffers(L, H, T, W, k_max, dtype=torch.float32):
    kvc = K()
    s = kvc.shape(L, H, H, 16, T, W, "f32")
    ws = torch.empty(kvc.kvc_workspace_size(s, k_max), dtype=torch.uint8, device="cuda")
    kvc.kvc_workspace_init(ws)
    return kvc, s, ws


def test_uniform_scores_ties_and_mba():
    L, H, T, W = 2, 3, 1000, 10
    kvc, s, ws = _stage_buffers(L, H, T, W, 500)
    sc = torch.full((L, H, T), 1.0 / T, device="cuda")
    mba = torch.empty((L, H), dtype=torch.int32, device="cuda")
    bud = torch.empty(L, dtype=torch.int32, device="cuda")
    kvc.kvc_mba_budget(s, sc, 9, 10, 2 * 200, 50, mba, bud, ws)
    idx = torch.full((L, H, 500), -1, dtype=torch.int32, device="cuda")
    kvc.kvc_topk_select(s, sc, bud, 500, idx, ws)
    torch.cuda.synchronize()
    assert (mba == math.ceil(0.9 * T)).all()
    assert bud.tolist() == [200, 200]
    for l in range(L):
        for h in range(H):
            assert idx[l, h, :200].tolist() == list(range(200))
    assert kvc.kvc_workspace_status(ws) == 0


def test_one_hot_all_zero_and_extreme_budgets():
    L, H, T, W = 3, 2, 600, 20
    P = T - W
    kvc, s, ws = _stage_buffers(L, H, T, W, P)
    sc = torch.zeros((L, H, T), device="cuda")
    sc[0, :, 17] = 1.0
    sc[1, 0, 5] = 0.5
    sc[1, 0, 6] = 0.5
    mba = torch.empty((L, H), dtype=torch.int32, device="cuda")
    bud = torch.empty(L, dtype=torch.int32, device="cuda")
    kvc.kvc_mba_budget(s, sc, 9, 10, 10 * P, 0, mba, bud, ws)   # total >= L*P: keep all
    torch.cuda.synchronize()
    assert mba[0].tolist() == [1, 1] and mba[1].tolist() == [2, 0] and mba[2].tolist() == [0, 0]
    assert bud.tolist() == [P] * L
    b2 = torch.tensor([0, P, 7], dtype=torch.int32, device="cuda")
    idx = torch.full((L, H, P), -1, dtype=torch.int32, device="cuda")
    kvc.kvc_topk_select(s, sc, b2, P, idx, ws)
    torch.cuda.synchronize()
    assert (idx[0] == -1).all()                                   # nothing kept
    assert idx[1, 0].tolist() == list(range(P))                   # everything kept
    assert idx[2, 0, :7].tolist() == list(range(7))               # all-zero ties
    assert kvc.kvc_workspace_status(ws) == 0


def test_device_status_flags():
    L, H, T, W = 1, 1, 300, 4
    kvc, s, ws = _stage_buffers(L, H, T, W, 50)
    sc = torch.full((L, H, T), 1.0 / T, device="cuda")
    sc[0, 0, 3] = -0.5
    mba = torch.empty((L, H), dtype=torch.int32, device="cuda")
    bud = torch.empty(L, dtype=torch.int32, device="cuda")
    kvc.kvc_mba_budget(s, sc, 9, 10, 40, 0, mba, bud, ws)
    assert kvc.kvc_workspace_status(ws) & kvc.DEV_BAD_SCORE
    kvc.kvc_workspace_init(ws)
    idx = torch.empty((L, H, 50), dtype=torch.int32, device="cuda")
    kvc.kvc_topk_select(s, torch.rand((L, H, T), device="cuda"),
                        torch.tensor([80], dtype=torch.int32, device="cuda"), 50, idx, ws)
    assert kvc.kvc_workspace_status(ws) & kvc.DEV_BAD_BUDGET
    kvc.kvc_workspace_init(ws)
    kk = torch.randn((L, H, T, 16), device="cuda")
    k_out = torch.empty((10, 16), device="cuda")
    v_out = torch.empty((10, 16), device="cuda")
    kvc.kvc_compact(s, kk, kk, idx, torch.tensor([20], dtype=torch.int32, device="cuda"), 50,
                    k_out, v_out, ws)
    st = kvc.kvc_workspace_status(ws)
    assert st & kvc.DEV_OUT_CAPACITY


def test_rejects_undersized_workspace_before_launch():
    kvc = K()
    wl, _, seed = SMALL["tc_rows48_tail16"]
    s = kvc.shape_of(wl)
    x = wk.make_inputs(wl, seed, device="cuda")
    ws = torch.zeros(512, dtype=torch.uint8, device="cuda")
    sc = torch.empty((wl.n_layers, wl.n_kv_heads, wl.seq_len), device="cuda")
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_score(s, x["q"], x["k"], sc, ws)
    assert e.value.code == -5


# --------------------------------------------------------------------------
# full-size workloads, in the launch configuration the benchmark times
def _sampled_units(wl, rng, n):
    units = [(l, h) for l in range(wl.n_layers) for h in range(wl.n_kv_heads)]
    pick = rng.choice(len(units), size=min(n, len(units)), replace=False)
    return [units[i] for i in sorted(pick)]


def _check_units(wl, x, b, units):
    o = O()
    s = oshape(wl)
    sc = b.scores
    for (l, h) in units:
        q1 = x["q"][l: l + 1].cpu()
        k1 = x["k"][l: l + 1].cpu()
        s1 = o.shape_of(1, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.seq_len, wl.window,
                        wl.dtype)
        ref = o.score_unit(s1, q1, k1, 0, h)
        assert_scores_close(sc[l, h].cpu().numpy(), ref)


def _check_compaction_heads(wl, b, x, bud, heads):
    """Compacted rows of the sampled heads equal the oracle's copy for that
    head (its K/V, the GPU's indices)."""
    o = O()
    P, W = wl.prefix_len, wl.window
    n = np.clip(bud, 0, P).astype(np.int64)
    offs = np.concatenate([[0], np.cumsum(wl.n_kv_heads * (n + W))])
    gi = b.idx
    for (l, h) in heads:
        s1 = o.shape_of(1, wl.group, 1, wl.head_dim, wl.seq_len, W, wl.dtype)
        r0 = int(offs[l] + h * (n[l] + W))
        idx1 = gi[l, h: h + 1].cpu().numpy()[None]
        for name, out in (("k", b.k_out), ("v", b.v_out)):
            src = x[name][l, h].cpu()[None, None]
            ref = o.compact(s1, src, idx1, np.array([bud[l]], dtype=np.int32), wl.k_max)
            assert np.array_equal(o.raw(out[r0: r0 + n[l] + W]), ref), (name, l, h)


def test_full_llama3_8b_single_layer_16k():
    wl = wk.LLAMA3_8B_LAYER
    x = wk.make_inputs(wl, wk.seed_for(1), device="cuda")
    b = run_gpu(wl, x)
    _check_units(wl, x, b, [(0, h) for h in range(wl.n_kv_heads)])
    check_discrete_stages(wl, x, b)


def test_full_zigzag_32k_sampled():
    wl = wk.ZIGZAG_32K
    x = wk.make_inputs(wl, wk.seed_for(2), device="cuda")
    b = run_gpu(wl, x)
    rng = np.random.default_rng(2)
    _check_units(wl, x, b, _sampled_units(wl, rng, 3))
    o = O()
    s = oshape(wl)
    total, floor = wl.budget_args()
    sc = b.scores.cpu().numpy()
    np.testing.assert_allclose(sc.astype(np.float64).sum(-1), 1.0, atol=1e-5)
    mba = o.mba_all(s, sc)
    assert np.array_equal(mba, b.mba.cpu().numpy())
    bud = o.budget(mba, wl.prefix_len, total, floor)
    assert np.array_equal(bud, b.budget.cpu().numpy())
    assert bud.sum() == total and bud.min() >= floor and len(set(bud.tolist())) > 1
    idx = o.topk_all(s, sc, bud, wl.k_max)
    gi = b.idx.cpu().numpy()
    for l in range(wl.n_layers):
        assert np.array_equal(gi[l, :, : bud[l]], idx[l, :, : bud[l]])
    _check_compaction_heads(wl, b, x, bud, _sampled_units(wl, rng, 4))


def test_full_think_128k_sampled():
    wl = wk.THINK_128K
    x = wk.make_inputs(wl, wk.seed_for(4), device="cuda")
    lam = wl.think_lambda
    b = run_gpu(wl, x, lam=lam)
    rng = np.random.default_rng(4)
    _check_units(wl, x, b, _sampled_units(wl, rng, 1))
    o = O()
    s = oshape(wl)
    total, floor = wl.budget_args()
    sc = b.scores.cpu().numpy()
    mba = o.mba_all(s, sc)
    assert np.array_equal(mba, b.mba.cpu().numpy())
    bud = o.budget(mba, wl.prefix_len, total, floor)
    assert np.array_equal(bud, b.budget.cpu().numpy())
    idx = o.topk_all(s, sc, bud, wl.k_max)
    gi = b.idx.cpu().numpy()
    for l in range(wl.n_layers):
        assert np.array_equal(gi[l, :, : bud[l]], idx[l, :, : bud[l]])
    heads = _sampled_units(wl, rng, 3)
    _check_compaction_heads(wl, b, x, bud, heads)
    # ThinK on the sampled heads: oracle over that head's compacted keys
    P, W, D = wl.prefix_len, wl.window, wl.head_dim
    n = np.clip(bud, 0, P).astype(np.int64)
    offs = np.concatenate([[0], np.cumsum(wl.n_kv_heads * (n + W))])
    keep = b.keep
    gchan = b.chan.cpu().numpy()
    poffs = np.concatenate([[0], np.cumsum(wl.n_kv_heads * n * keep)])
    for (l, h) in heads:
        r0 = int(offs[l] + h * (n[l] + W))
        blk = o.raw(b.k_out[r0: r0 + n[l] + W])
        s1 = o.shape_of(1, wl.group, 1, D, wl.seq_len, W, wl.dtype)
        chan, norms, kp = o.channel_prune(s1, blk, np.array([bud[l]], dtype=np.int32), lam)
        assert np.array_equal(chan[0, 0], gchan[l, h])
        p0 = int(poffs[l] + h * n[l] * keep)
        assert np.array_equal(kp, o.raw(b.k_pruned[p0: p0 + n[l] * keep]))
    # the outlier channels (x8) are among the kept channels of every head
    kf = x["k"]
    for (l, h) in heads:
        outl = torch.topk(kf[l, h, :P].float().abs().mean(0), wl.outlier_channels).indices
        assert set(outl.tolist()) <= set(gchan[l, h].tolist())


def test_ragged_mistral_batch_sampled():
    batch = wk.ragged_mistral_batch(wk.seed_for(3))
    rng = np.random.default_rng(3)
    o = O()
    for wl in (min(batch, key=lambda w: w.seq_len), max(batch, key=lambda w: w.seq_len)):
        x = wk.make_inputs(wl, wk.seed_for(3) + wl.seq_len, device="cuda")
        b = run_gpu(wl, x)
        _check_units(wl, x, b, _sampled_units(wl, rng, 1))
        s = oshape(wl)
        total, floor = wl.budget_args()
        sc = b.scores.cpu().numpy()
        mba = o.mba_all(s, sc)
        assert np.array_equal(mba, b.mba.cpu().numpy())
        bud = o.budget(mba, wl.prefix_len, total, floor)
        assert np.array_equal(bud, b.budget.cpu().numpy())
        idx = o.topk_all(s, sc, bud, wl.k_max)
        gi = b.idx.cpu().numpy()
        for l in range(wl.n_layers):
            assert np.array_equal(gi[l, :, : bud[l]], idx[l, :, : bud[l]])
        _check_compaction_heads(wl, b, x, bud, _sampled_units(wl, rng, 2))
        del x, b
        torch.cuda.empty_cache()
