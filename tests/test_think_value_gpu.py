"""GPU parity of the optional THINKV value-channel criterion
(kvc_channel_prune_value; ThinK page, appendix "Value cache pruning
strategy") against the oracle, on every (layer, KV head) unit:

  value scores   |s_gpu - s_ora| <= VALUE_RTOL * s_ora per channel, s_ora the
                 oracle's fp64 squared column norms of the window rows'
                 attention output (VALUE_RTOL per path, see below) -- or, for a
                 channel whose output column cancels (o_r[d] = sum_j p_rj v_jd
                 near 0 against its terms: few window rows), VALUE_RTOL * m_ora,
                 m_ora the same squared norm of the magnitudes it sums,
                 sum_r (sum_j p_rj |v_jd|)^2 (the oracle's value score on |V|);
                 m_ora = s_ora when nothing cancels;
  stage-isolated the oracle's selection on the GPU's own fp32 value scores
                 gives the GPU's channels and pruned bytes bit for bit;
  end to end     the GPU's channels equal the oracle's (from its fp64 scores)
                 except where a channel in the symmetric difference has an
                 oracle score within the two channels' tolerances of the
                 head's keep-th score.
"""
import os

import numpy as np
import pytest
import torch

from eviction_kvc_score_gb300 import workloads as wk

pytestmark = pytest.mark.gpu

# Both paths form each probability in fp32 from the exact row normaliser
# (ex2.approx, ~2^-22 relative).  CUDA cores: fp32 products and sums over at
# most a few 10^5 terms per output (relative error ~ sqrt(T) 2^-24 < 1e-4).
# Tensor cores: each probability enters the product with V as two bf16 terms
# (p_hi + p_lo carries ~16 significant bits, 2^-17 relative), bf16 x bf16
# products are exact in the fp32 accumulator, so the same 1e-4 bound holds.
VALUE_RTOL = {"simt": 1e-4, "tc": 1e-4}


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
    # tensor-core shape: bf16, D=128, 512 window rows, ragged last tile
    "bf16_d128_rows512": (wk.ZIGZAG_32K.scaled(
        n_layers=2, n_kv_heads=2, n_q_heads=8, seq_len=1500, total_budget=2 * 300,
        layer_floor=40, temperature=(0.3, 3.0), think_lambda=0.4), 41),
    # 384 rows: the second 256-row job is half padding
    "bf16_d128_rows384": (wk.ZIGZAG_32K.scaled(
        n_layers=2, n_kv_heads=2, n_q_heads=8, seq_len=2000, window=96,
        total_budget=2 * 380, layer_floor=30, temperature=None, think_lambda=0.3), 42),
    # 48 rows, one tile only partly visible
    "bf16_d128_rows48": (wk.ZIGZAG_32K.scaled(
        n_layers=2, n_kv_heads=2, n_q_heads=6, seq_len=300, window=16, total_budget=2 * 50,
        layer_floor=5, temperature=None, think_lambda=0.5), 43),
    # CUDA-core shapes
    "bf16_d64": (wk.ZIGZAG_32K.scaled(
        n_layers=2, n_kv_heads=3, n_q_heads=6, head_dim=64, seq_len=777, window=64,
        total_budget=2 * 100, layer_floor=20, think_lambda=0.4), 44),
    "f32_mha": (wk.TINY.scaled(think_lambda=0.25), 45),
    "f32_d80": (wk.ZIGZAG_32K.scaled(
        n_layers=2, n_kv_heads=2, n_q_heads=4, head_dim=80, seq_len=333, window=8,
        total_budget=2 * 60, layer_floor=10, temperature=None, dtype="f32",
        think_lambda=0.25), 46),
}


def path_of(wl):
    tc = (wl.dtype == "bf16" and wl.head_dim == 128 and wl.group * wl.window <= 512
          and os.environ.get("KVC_SCORE_IMPL", "auto") != "simt")
    return "tc" if tc else "simt"


def run_value(wl, x):
    """Default chain, then THINKV on its compacted values."""
    kvc = K()
    lam = wl.think_lambda
    total, floor = wl.budget_args()
    b = kvc.alloc_buffers(kvc.shape_of(wl), total, wl.k_max)
    kvc.compress(b, x["q"], x["k"], x["v"], total, floor, wl.mass_num, wl.mass_den)
    L, H, D = wl.n_layers, wl.n_kv_heads, wl.head_dim
    keep = kvc.kvc_keep_channels(lam, D)
    kept_rows = min(total, L * wl.prefix_len)
    b.v_scores = torch.full((L, H, D), float("nan"), device="cuda")
    b.v_chan = torch.full((L, H, keep), -1, dtype=torch.int32, device="cuda")
    b.v_pruned = torch.empty(max(1, H * kept_rows * keep), dtype=x["v"].dtype, device="cuda")
    kvc.kvc_channel_prune_value(b.shape, x["q"], x["k"], x["v"], b.v_out, b.budget, lam,
                                b.v_chan, b.v_pruned, b.ws, value_scores=b.v_scores)
    torch.cuda.synchronize()
    assert kvc.kvc_workspace_status(b.ws) == 0
    b.v_keep = keep
    return b


def value_tolerance(wl, x, gs, ref_scores, rtol):
    """Per-channel tolerance: rtol * s_ora, widened to rtol * m_ora (the squared
    norm of the magnitudes, computed per layer only where needed) for channels
    whose output column cancels."""
    o = O()
    tol = rtol * ref_scores
    bad = np.abs(gs - ref_scores) > tol
    for l in sorted(set(np.argwhere(bad)[:, 0].tolist())):
        s1 = o.shape_of(1, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.seq_len, wl.window,
                        wl.dtype)
        mag = o.value_scores(s1, x["q"][l:l + 1], x["k"][l:l + 1], x["v"][l:l + 1].abs())[0]
        tol[l] = np.maximum(tol[l], rtol * mag)
    return tol


def check_value(wl, x, b, ref_scores, rtol):
    o = O()
    s = oshape(wl)
    lam = wl.think_lambda
    gs = b.v_scores.double().cpu().numpy()
    tol = value_tolerance(wl, x, gs, ref_scores, rtol)
    bad = np.abs(gs - ref_scores) > tol
    assert not bad.any(), (f"{bad.sum()} value scores out of tolerance, worst relative "
                           f"{(np.abs(gs - ref_scores) / ref_scores).max():.2e}")
    bud = b.budget.cpu().numpy()
    rows = o.compact_rows(s, bud)
    v_out = o.raw(b.v_out[:rows])
    # stage-isolated: the oracle's selection on the GPU's own scores
    chan_g, vp_g = o.channel_prune_value(s, b.v_scores.cpu().numpy(), v_out, bud, lam)
    gchan = b.v_chan.cpu().numpy()
    assert np.array_equal(gchan, chan_g), "channels on the GPU's scores"
    assert np.array_equal(o.raw(b.v_pruned[: vp_g.size]), vp_g), "pruned V bytes"
    # end to end: the oracle's own fp64 scores, near-ties allowed
    chan_o, _ = o.channel_prune_value(s, ref_scores, v_out, bud, lam)
    keep = b.v_keep
    n_diff = 0
    for l in range(wl.n_layers):
        for h in range(wl.n_kv_heads):
            diff = np.setxor1d(gchan[l, h], chan_o[l, h])
            if diff.size:
                kc = np.argsort(-ref_scores[l, h], kind="stable")[keep - 1]
                kth = ref_scores[l, h, kc]
                assert np.all(np.abs(ref_scores[l, h, diff] - kth) <= tol[l, h, diff] + tol[l, h, kc]), \
                    (l, h)
                n_diff += diff.size
    return n_diff


@pytest.mark.parametrize("name", list(CASES))
def test_value_channels_match_oracle(name):
    wl, seed = CASES[name]
    x = wk.make_inputs(wl, seed, device="cuda")
    b = run_value(wl, x)
    ref = O().value_scores(oshape(wl), x["q"], x["k"], x["v"])
    check_value(wl, x, b, ref, VALUE_RTOL[path_of(wl)])


def test_value_cuda_core_path_on_tensor_core_shape():
    wl, seed = CASES["bf16_d128_rows512"]
    x = wk.make_inputs(wl, seed, device="cuda")
    old = os.environ.get("KVC_SCORE_IMPL")
    os.environ["KVC_SCORE_IMPL"] = "simt"
    try:
        b = run_value(wl, x)
    finally:
        if old is None:
            os.environ.pop("KVC_SCORE_IMPL", None)
        else:
            os.environ["KVC_SCORE_IMPL"] = old
    ref = O().value_scores(oshape(wl), x["q"], x["k"], x["v"])
    check_value(wl, x, b, ref, VALUE_RTOL["simt"])


def test_value_full_llama3_layer_16k_all_units():
    wl = wk.LLAMA3_8B_LAYER.scaled(think_lambda=0.3)
    x = wk.make_inputs(wl, wk.seed_for(1), device="cuda")
    b = run_value(wl, x)
    ref = O().value_scores(oshape(wl), x["q"], x["k"], x["v"])
    check_value(wl, x, b, ref, VALUE_RTOL[path_of(wl)])


def test_value_runs_are_deterministic():
    wl, seed = CASES["bf16_d128_rows512"]
    x = wk.make_inputs(wl, seed, device="cuda")
    a = run_value(wl, x)
    b = run_value(wl, x)
    assert torch.equal(a.v_scores, b.v_scores) and torch.equal(a.v_chan, b.v_chan)
    assert torch.equal(a.v_pruned, b.v_pruned)


def test_value_full_zigzag_32k_all_units():
    """The 32-layer 32K prompt in the benchmark's launch configuration: every
    unit's value scores against the oracle's fp64 definition."""
    wl = wk.ZIGZAG_32K.scaled(think_lambda=0.3)
    x = wk.make_inputs(wl, wk.seed_for(2), device="cuda")
    b = run_value(wl, x)
    ref = O().value_scores(oshape(wl), x["q"], x["k"], x["v"])
    check_value(wl, x, b, ref, VALUE_RTOL[path_of(wl)])


def test_value_full_think_128k_sampled_layers():
    """The 128K prompt (32 layers, the benchmark's launch configuration): the
    GPU runs every layer; two layers' value scores (all their heads) are
    checked against the oracle run on those layers alone, and the channels and
    pruned bytes of every head against the oracle's selection on the GPU's own
    scores."""
    wl = wk.THINK_128K.scaled(think_lambda=0.3)
    x = wk.make_inputs(wl, wk.seed_for(4), device="cuda")
    b = run_value(wl, x)
    o = O()
    gs = b.v_scores.double().cpu().numpy()
    for l in (0, 17):
        s1 = o.shape_of(1, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.seq_len, wl.window,
                        wl.dtype)
        ref = o.value_scores(s1, x["q"][l:l + 1], x["k"][l:l + 1], x["v"][l:l + 1])[0]
        rtol = VALUE_RTOL[path_of(wl)]
        assert np.all(np.abs(gs[l] - ref) <= rtol * ref), l   # 512 rows: no cancellation
    s = oshape(wl)
    bud = b.budget.cpu().numpy()
    rows = o.compact_rows(s, bud)
    chan_g, vp_g = o.channel_prune_value(s, b.v_scores.cpu().numpy(), o.raw(b.v_out[:rows]), bud,
                                         wl.think_lambda)
    assert np.array_equal(b.v_chan.cpu().numpy(), chan_g)
    assert np.array_equal(o.raw(b.v_pruned[: vp_g.size]), vp_g)


@pytest.mark.parametrize("case", ["budget_zero_and_full", "window_one", "prefix_of_one"])
def test_value_edge_cases(case):
    """Degenerate budgets and shapes: a layer keeping no prefix row (its
    channels are still chosen, its pruned block is empty) next to one keeping
    the whole prefix; a one-row window; a one-token prefix."""
    kvc = K()
    o = O()
    if case == "budget_zero_and_full":
        wl = wk.ZIGZAG_32K.scaled(n_layers=2, n_kv_heads=2, n_q_heads=8, seq_len=700,
                                  total_budget=0, layer_floor=0, temperature=None,
                                  think_lambda=0.25)
        budgets = [0, 700 - 128]
    elif case == "window_one":
        wl = wk.ZIGZAG_32K.scaled(n_layers=2, n_kv_heads=2, n_q_heads=4, seq_len=900, window=1,
                                  total_budget=2 * 100, layer_floor=10, temperature=None,
                                  think_lambda=0.5)
        budgets = [60, 140]
    else:
        wl = wk.ZIGZAG_32K.scaled(n_layers=2, n_kv_heads=1, n_q_heads=2, seq_len=33, window=32,
                                  total_budget=2, layer_floor=0, temperature=None,
                                  think_lambda=0.4)
        budgets = [1, 1]
    x = wk.make_inputs(wl, 47, device="cuda")
    s = kvc.shape_of(wl)
    L, H, D, P = wl.n_layers, wl.n_kv_heads, wl.head_dim, wl.prefix_len
    ws = torch.empty(kvc.kvc_workspace_size(s, P), dtype=torch.uint8, device="cuda")
    kvc.kvc_workspace_init(ws)
    bud = torch.tensor(budgets, dtype=torch.int32, device="cuda")
    k_max = max(1, max(min(b, P) for b in budgets))
    idx = torch.empty((L, H, k_max), dtype=torch.int32, device="cuda")
    scores = torch.empty((L, H, wl.seq_len), device="cuda")
    kvc.kvc_score(s, x["q"], x["k"], scores, ws)
    kvc.kvc_topk_select(s, scores, bud, k_max, idx, ws)
    rows = H * sum(min(b, P) + wl.window for b in budgets)
    k_out = torch.empty((rows, D), dtype=x["k"].dtype, device="cuda")
    v_out = torch.empty_like(k_out)
    kvc.kvc_compact(s, x["k"], x["v"], idx, bud, k_max, k_out, v_out, ws)
    keep = kvc.kvc_keep_channels(wl.think_lambda, D)
    chan = torch.full((L, H, keep), -1, dtype=torch.int32, device="cuda")
    vp = torch.empty(max(1, H * sum(min(b, P) for b in budgets) * keep), dtype=x["v"].dtype,
                     device="cuda")
    vsc = torch.empty((L, H, D), device="cuda")
    kvc.kvc_channel_prune_value(s, x["q"], x["k"], x["v"], v_out, bud, wl.think_lambda, chan, vp,
                                ws, value_scores=vsc)
    torch.cuda.synchronize()
    assert kvc.kvc_workspace_status(ws) == 0
    ref = o.value_scores(oshape(wl), x["q"], x["k"], x["v"])
    rtol = VALUE_RTOL[path_of(wl)]
    gs = vsc.double().cpu().numpy()
    assert np.all(np.abs(gs - ref) <= value_tolerance(wl, x, gs, ref, rtol))
    bnp = bud.cpu().numpy()
    chan_g, vp_g = o.channel_prune_value(oshape(wl), vsc.cpu().numpy(), o.raw(v_out), bnp,
                                         wl.think_lambda)
    assert np.array_equal(chan.cpu().numpy(), chan_g)
    assert np.array_equal(o.raw(vp[: vp_g.size]), vp_g)


def test_value_reuses_the_score_statistics():
    """kvc_channel_prune_value_ex with KVC_VALUE_REUSE_SCORE_STATS after the
    default path's kvc_score gives bit-identical value scores, channels and
    pruned bytes without its own statistics pass; with no matching kvc_score
    recorded for the workspace (a fresh workspace, a Keyformer score, a reset)
    it is refused."""
    kvc = K()
    wl, seed = CASES["bf16_d128_rows512"]
    x = wk.make_inputs(wl, seed, device="cuda")
    b = run_value(wl, x)   # compress (kvc_score on b.ws), then THINKV with its own statistics
    kvc.kvc_score(b.shape, x["q"], x["k"], b.scores, b.ws)   # the record for b.ws
    vs = torch.full_like(b.v_scores, float("nan"))
    ch = torch.full_like(b.v_chan, -1)
    vp = torch.zeros_like(b.v_pruned)
    kvc.kvc_channel_prune_value(b.shape, x["q"], x["k"], x["v"], b.v_out, b.budget,
                                wl.think_lambda, ch, vp, b.ws, value_scores=vs,
                                reuse_score_stats=True)
    torch.cuda.synchronize()
    assert kvc.kvc_workspace_status(b.ws) == 0
    assert torch.equal(vs, b.v_scores) and torch.equal(ch, b.v_chan)
    assert torch.equal(vp, b.v_pruned)
    # another shape's or another tensor's statistics are not taken
    with pytest.raises(RuntimeError):
        kvc.kvc_channel_prune_value(b.shape, x["q"].clone(), x["k"], x["v"], b.v_out, b.budget,
                                    wl.think_lambda, ch, vp, b.ws, reuse_score_stats=True)
    # a Keyformer score rewrites the statistics: refused until the next kvc_score
    kvc.kvc_score_keyformer(b.shape, x["q"], x["k"], 7, 1.0, b.scores, b.ws)
    with pytest.raises(RuntimeError):
        kvc.kvc_channel_prune_value(b.shape, x["q"], x["k"], x["v"], b.v_out, b.budget,
                                    wl.think_lambda, ch, vp, b.ws, reuse_score_stats=True)
    # a fresh workspace has no statistics
    ws2 = torch.empty_like(b.ws)
    kvc.kvc_workspace_init(ws2)
    with pytest.raises(RuntimeError):
        kvc.kvc_channel_prune_value(b.shape, x["q"], x["k"], x["v"], b.v_out, b.budget,
                                    wl.think_lambda, ch, vp, ws2, reuse_score_stats=True)
    # the CUDA-core path reuses its own statistics, and statistics of the
    # other path (another row split) are refused
    old = os.environ.get("KVC_SCORE_IMPL")
    try:
        os.environ["KVC_SCORE_IMPL"] = "simt"
        with pytest.raises(RuntimeError):   # the record is the tensor-core score's... none now
            kvc.kvc_channel_prune_value(b.shape, x["q"], x["k"], x["v"], b.v_out, b.budget,
                                        wl.think_lambda, ch, vp, b.ws, reuse_score_stats=True)
        kvc.kvc_score(b.shape, x["q"], x["k"], b.scores, b.ws)
        ref_s = torch.empty_like(vs)
        kvc.kvc_channel_prune_value(b.shape, x["q"], x["k"], x["v"], b.v_out, b.budget,
                                    wl.think_lambda, ch, vp, b.ws, value_scores=ref_s)
        kvc.kvc_score(b.shape, x["q"], x["k"], b.scores, b.ws)
        vs2 = torch.full_like(vs, float("nan"))
        kvc.kvc_channel_prune_value(b.shape, x["q"], x["k"], x["v"], b.v_out, b.budget,
                                    wl.think_lambda, ch, vp, b.ws, value_scores=vs2,
                                    reuse_score_stats=True)
        torch.cuda.synchronize()
        assert torch.equal(vs2, ref_s)
        os.environ["KVC_SCORE_IMPL"] = "tc"
        with pytest.raises(RuntimeError):   # recorded for the CUDA-core split
            kvc.kvc_channel_prune_value(b.shape, x["q"], x["k"], x["v"], b.v_out, b.budget,
                                        wl.think_lambda, ch, vp, b.ws, reuse_score_stats=True)
    finally:
        if old is None:
            os.environ.pop("KVC_SCORE_IMPL", None)
        else:
            os.environ["KVC_SCORE_IMPL"] = old

