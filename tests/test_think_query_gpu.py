"""GPU parity of the optional ThinK query-driven key-channel criterion
(kvc_channel_prune_query) against the oracle, stage-isolated: the oracle ranks
the channels of the GPU's own compacted keys with the same window queries.
Channels are bit-exact except where the oracle's two boundary scores are within
1e-9 relative (the GPU sums squares in float-float pairs); pruned bytes are
exact whenever the channels agree."""
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


def _run(wl, seed, lam):
    kvc = K()
    x = wk.make_inputs(wl, seed, device="cuda")
    total, floor = wl.budget_args()
    b = kvc.alloc_buffers(kvc.shape_of(wl), total, wl.k_max, lam=lam)
    kvc.compress(b, x["q"], x["k"], x["v"], total, floor, wl.mass_num, wl.mass_den, lam=lam,
                 think="query")
    torch.cuda.synchronize()
    assert kvc.kvc_workspace_status(b.ws) == 0
    return x, b


def _check_heads(o, s_full, wl, x, b, lam, heads):
    bud = b.budget.cpu().numpy()
    P, W, D = wl.seq_len - wl.window, wl.window, wl.head_dim
    G = wl.n_q_heads // wl.n_kv_heads
    n = np.clip(bud, 0, P).astype(np.int64)
    offs = np.concatenate([[0], np.cumsum(wl.n_kv_heads * (n + W))])
    keep = b.keep
    poffs = np.concatenate([[0], np.cumsum(wl.n_kv_heads * n * keep)])
    gchan = b.chan.cpu().numpy()
    qn = o.raw(x["q"])
    for (l, h) in heads:
        r0 = int(offs[l] + h * (n[l] + W))
        blk = o.raw(b.k_out[r0: r0 + n[l] + W])
        s1 = o.shape_of(1, G, 1, D, wl.seq_len, W, wl.dtype)
        q1 = np.ascontiguousarray(qn[l, h * G:(h + 1) * G])
        chan, sc, kp = o.channel_prune_query(s1, q1, blk, np.array([bud[l]], dtype=np.int32), lam)
        if not np.array_equal(chan[0, 0], gchan[l, h]):
            srt = np.sort(sc[0, 0])[::-1]
            kth, nxt = srt[keep - 1], srt[keep]
            assert abs(kth - nxt) <= 1e-9 * kth, f"query-driven channels layer {l} head {h}"
            continue
        p0 = int(poffs[l] + h * n[l] * keep)
        assert np.array_equal(kp, o.raw(b.k_pruned[p0: p0 + n[l] * keep])), f"pruned K {l},{h}"


CASES = {
    "bf16_tc_rows256": (wk.ZIGZAG_32K.scaled(
        n_layers=2, n_kv_heads=2, n_q_heads=8, seq_len=4100, window=64,
        total_budget=2 * 820, layer_floor=102, temperature=None), 0.4, 41),
    "f32_odd_dim": (wk.ZIGZAG_32K.scaled(
        n_layers=2, n_kv_heads=2, n_q_heads=4, head_dim=80, seq_len=333, window=8,
        total_budget=2 * 60, layer_floor=10, temperature=None, dtype="f32"), 0.25, 42),
    "bf16_d64_mix": (wk.LLAMA3_8B_LAYER.scaled(
        n_layers=2, seq_len=2048, n_q_heads=8, n_kv_heads=2, head_dim=64), 0.5, 43),
}


@pytest.mark.parametrize("name", list(CASES))
def test_query_driven_small(name):
    wl, lam, seed = CASES[name]
    x, b = _run(wl, seed, lam)
    heads = [(l, h) for l in range(wl.n_layers) for h in range(wl.n_kv_heads)]
    _check_heads(O(), oshape(wl), wl, x, b, lam, heads)


def test_query_driven_differs_from_magnitude_when_queries_ignore_a_channel():
    """Zeroing one channel of every window query makes that channel's
    query-driven score zero: it must drop out although its keys are large."""
    kvc = K()
    wl, lam, seed = CASES["bf16_d64_mix"]
    x = wk.make_inputs(wl, seed, device="cuda")
    x["q"][..., 7] = 0
    x["k"][..., 7] *= 16
    total, floor = wl.budget_args()
    b = kvc.alloc_buffers(kvc.shape_of(wl), total, wl.k_max, lam=lam)
    kvc.compress(b, x["q"], x["k"], x["v"], total, floor, lam=lam, think="query")
    chan_q = b.chan.clone()
    kvc.kvc_channel_prune(b.shape, b.k_out, b.budget, lam, b.chan, b.k_pruned, b.ws)
    torch.cuda.synchronize()
    assert (chan_q != 7).all()
    assert (b.chan == 7).any(dim=-1).all()


def test_query_driven_full_128k_sampled():
    wl = wk.THINK_128K
    lam = wl.think_lambda
    x, b = _run(wl, wk.seed_for(4), lam)
    rng = np.random.default_rng(44)
    heads = [(int(rng.integers(wl.n_layers)), int(rng.integers(wl.n_kv_heads))) for _ in range(3)]
    _check_heads(O(), oshape(wl), wl, x, b, lam, heads)


def test_query_driven_rejects_bad_arguments():
    kvc = K()
    s = kvc.shape(1, 2, 1, 16, 100, 4, "f32")
    ws = torch.empty(kvc.kvc_workspace_size(s, 10), dtype=torch.uint8, device="cuda")
    kvc.kvc_workspace_init(ws)
    q = torch.zeros((1, 2, 4, 16), device="cuda")
    k_out = torch.zeros((14, 16), device="cuda")
    bud = torch.tensor([10], dtype=torch.int32, device="cuda")
    chan = torch.empty((1, 1, 16), dtype=torch.int32, device="cuda")
    kp = torch.empty(160, device="cuda")
    with pytest.raises(kvc.KvcError):
        kvc.kvc_channel_prune_query(s, q, k_out, bud, 1.5, chan, kp, ws)     # keeps no channel
    with pytest.raises(kvc.KvcError):
        kvc.kvc_channel_prune_query(s, None, k_out, bud, 0.5, chan, kp, ws)  # NULL query
