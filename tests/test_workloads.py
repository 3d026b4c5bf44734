"""CPU checks of the seeded input generators that both the CUDA path and the
oracle consume (eviction_kvc_score_gb300/workloads.py): the bytes are a
function of the seed alone, the layouts are the documented ones, and each
generator knob produces the structure it names (mixed window queries, outlier
key channels, planted keys, per-layer temperatures, the ragged batch's
lengths and budgets)."""
import math

import torch

from eviction_kvc_score_gb300 import workloads as wk


def _small_zigzag(**kw):
    args = dict(n_layers=2, n_kv_heads=2, n_q_heads=8, seq_len=512, window=16,
                total_budget=2 * 100, layer_floor=10)
    args.update(kw)
    return wk.ZIGZAG_32K.scaled(**args)


def test_inputs_are_a_function_of_the_seed_and_have_the_documented_layout():
    for wl in (wk.TINY, _small_zigzag()):
        a = wk.make_inputs(wl, 7)
        b = wk.make_inputs(wl, 7)
        c = wk.make_inputs(wl, 8)
        L, Hq, Hkv, D, T, W = (wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim,
                               wl.seq_len, wl.window)
        assert a["q"].shape == (L, Hq, W, D) and a["q"].is_contiguous()
        assert a["k"].shape == (L, Hkv, T, D) and a["v"].shape == (L, Hkv, T, D)
        for name in ("q", "k", "v"):
            assert a[name].dtype == wl.torch_dtype
            assert torch.equal(a[name], b[name]), (wl.name, name)
            assert not torch.equal(a[name], c[name]), (wl.name, name)
        assert wk.make_inputs(wl, 7, with_v=False)["v"] is None


def test_mixed_queries_are_convex_combinations_of_their_heads_keys():
    """With the mix weight at 1 every window query of KV head h is a convex
    combination of h's prefix keys, so each coordinate lies within the range
    of that coordinate over those keys (up to the final bf16 rounding)."""
    wl = _small_zigzag(mix_weight=1.0, temperature=None)
    x = wk.make_inputs(wl, 3)
    G, P = wl.group, wl.prefix_len
    q, k = x["q"].float(), x["k"].float()
    for l in range(wl.n_layers):
        for h in range(wl.n_kv_heads):
            lo = k[l, h, :P].min(dim=0).values
            hi = k[l, h, :P].max(dim=0).values
            qh = q[l, h * G:(h + 1) * G].reshape(-1, wl.head_dim)
            slack = 1e-2 * (hi - lo).abs().max()
            assert bool((qh >= lo - slack).all() and (qh <= hi + slack).all()), (l, h)


def test_outlier_channels_are_the_loudest():
    wl = _small_zigzag(temperature=None)
    k = wk.make_inputs(wl, 5)["k"].float()
    for l in range(wl.n_layers):
        for h in range(wl.n_kv_heads):
            norms = k[l, h].pow(2).mean(dim=0).sqrt()          # per channel
            top = torch.topk(norms, wl.outlier_channels).values
            rest = torch.sort(norms, descending=True).values[wl.outlier_channels:]
            # unit-variance channels have RMS near 1, the scaled ones near 8
            assert float(rest.max()) < 1.5
            assert float(top.min()) > 0.5 * wl.outlier_scale


def test_planted_keys_are_three_times_the_mean_window_query():
    wl = wk.TINY
    x = wk.make_inputs(wl, 11)
    G = wl.group
    for l in range(wl.n_layers):
        for h in range(wl.n_kv_heads):
            qm = x["q"][l, h * G:(h + 1) * G].reshape(-1, wl.head_dim).float().mean(dim=0)
            pos = x["planted"][l, h]
            assert pos.numel() == wl.planted and len(set(pos.tolist())) == wl.planted
            assert bool((pos < wl.prefix_len).all())
            for p in pos.tolist():
                assert torch.allclose(x["k"][l, h, p].float(), 3.0 * qm, rtol=1e-5, atol=1e-6)


def test_temperatures_divide_each_layers_queries():
    """The per-layer temperatures lie in their log-uniform range, and dividing
    by them sets each layer's query scale: std(q_l) * tau_l is about the same
    for every layer while std(q_l) itself spreads with tau."""
    base = _small_zigzag(dtype="f32", n_layers=6, temperature=(0.3, 3.0))
    x = wk.make_inputs(base, 4)
    taus = x["tau"]
    lo, hi = base.temperature
    assert taus.shape == (base.n_layers,) and bool(((taus >= lo) & (taus <= hi)).all())
    raw = torch.stack([x["q"][l].std() for l in range(base.n_layers)])
    scaled = raw * taus
    assert float(scaled.max() / scaled.min()) < 1.5
    assert float(raw.max() / raw.min()) > 0.8 * float(taus.max() / taus.min()) / 1.5


def test_ragged_batch_lengths_and_budgets():
    a = wk.ragged_mistral_batch(wk.seed_for(3))
    b = wk.ragged_mistral_batch(wk.seed_for(3))
    assert [w.seq_len for w in a] == [w.seq_len for w in b]
    assert len(a) == 8
    for w in a:
        assert 4096 <= w.seq_len <= 65536
        assert (w.n_layers, w.n_q_heads, w.n_kv_heads, w.head_dim, w.window) == (32, 32, 8, 128, 64)
        mean_b = math.floor(0.2 * w.seq_len)
        assert w.total_budget == 32 * mean_b and w.layer_floor == mean_b // 8
        total, floor = w.budget_args()
        assert w.k_max == min(w.prefix_len, total - 31 * floor)
    assert len({w.seq_len for w in a}) > 1
