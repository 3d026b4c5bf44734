"""GPU parity of the optional Keyformer scores (Gumbel-noised logits with a
temperature, counter-based Philox draws) against the fp64 oracle, which draws
the same noise from its own Philox4x32-10: scores within 1e-3 relative (the
GPU works in fp32), every head's scores sum to 1 within 1e-5, top-K on the
GPU's scores bit-exact against the oracle's selection on the same scores."""
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


def _gpu_scores(wl, x, seed, tau):
    kvc = K()
    s = kvc.shape_of(wl)
    ws = torch.empty(kvc.kvc_workspace_size(s, max(wl.k_max, 1)), dtype=torch.uint8, device="cuda")
    kvc.kvc_workspace_init(ws)
    sc = torch.empty((wl.n_layers, wl.n_kv_heads, wl.seq_len), device="cuda")
    kvc.kvc_score_keyformer(s, x["q"], x["k"], seed, tau, sc, ws)
    torch.cuda.synchronize()
    assert kvc.kvc_workspace_status(ws) == 0
    return sc, ws


CASES = {
    "f32_mha": (wk.TINY.scaled(n_layers=2, seq_len=600, window=16), 101),
    "bf16_gqa_rows512": (wk.ZIGZAG_32K.scaled(
        n_layers=1, n_kv_heads=2, n_q_heads=8, seq_len=1200, temperature=None), 102),
    # tensor-core path with one 256-row job per tile (two warpgroups per job
    # in pass 1), D = 64, ragged last tile
    "bf16_d64_rows256": (wk.ZIGZAG_32K.scaled(
        n_layers=2, n_kv_heads=2, n_q_heads=4, head_dim=64, seq_len=900, window=64,
        total_budget=2 * 100, layer_floor=20, temperature=None), 104),
    "bf16_odd_dim": (wk.ZIGZAG_32K.scaled(
        n_layers=2, n_kv_heads=2, n_q_heads=4, head_dim=80, seq_len=333, window=8,
        total_budget=2 * 60, layer_floor=10, temperature=None), 103),
    # tensor-core path, 400 window rows (W = 100, not a multiple of 4): the
    # second 256-row job is partly padding and the causal edge crosses the
    # four-row groups whose noise blocks pass 2 shares across lanes; ragged
    # last tile
    "bf16_rows400_w100": (wk.ZIGZAG_32K.scaled(
        n_layers=1, n_kv_heads=2, n_q_heads=8, seq_len=3001, window=100,
        total_budget=2 * 500, layer_floor=40, temperature=None), 105),
    # 384 rows, D = 64: the odd CTA's rows of the second job are all padding
    "bf16_d64_rows384": (wk.ZIGZAG_32K.scaled(
        n_layers=1, n_kv_heads=2, n_q_heads=16, head_dim=64, seq_len=1000, window=48,
        total_budget=2 * 200, layer_floor=20, temperature=None), 106),
}


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("tau", [0.5, 1.0, 4.0])
def test_keyformer_scores_match_oracle(name, tau):
    wl, seed = CASES[name]
    x = wk.make_inputs(wl, seed, device="cuda")
    sc, _ = _gpu_scores(wl, x, 2024 + seed, tau)
    want = O().score_keyformer(oshape(wl), x["q"], x["k"], 2024 + seed, tau)
    got = sc.cpu().numpy().astype(np.float64)
    bad = np.abs(got - want) > 1e-3 * want + 1e-30
    assert not bad.any(), (np.argwhere(bad)[:3], got[bad][:3], want[bad][:3])
    np.testing.assert_allclose(got.sum(-1), 1.0, atol=1e-5)


def test_keyformer_seed_determinism_and_selection():
    kvc, o = K(), O()
    wl, seed = CASES["bf16_gqa_rows512"]
    wl = wl.scaled(total_budget=300, layer_floor=100)
    x = wk.make_inputs(wl, seed, device="cuda")
    a, ws = _gpu_scores(wl, x, 7, 1.0)
    b, _ = _gpu_scores(wl, x, 7, 1.0)
    c, _ = _gpu_scores(wl, x, 8, 1.0)
    assert torch.equal(a, b) and not torch.equal(a, c)
    # top-K on the noisy scores: bit-exact against the oracle's selection on
    # the same fp32 scores
    s = kvc.shape_of(wl)
    bud = torch.tensor([300], dtype=torch.int32, device="cuda")
    idx = torch.full((1, wl.n_kv_heads, 300), -1, dtype=torch.int32, device="cuda")
    kvc.kvc_topk_select(s, a, bud, 300, idx, ws)
    torch.cuda.synchronize()
    want = o.topk_all(oshape(wl), a.cpu().numpy(), np.array([300], np.int32), 300)
    assert np.array_equal(idx.cpu().numpy(), want)


def test_keyformer_full_llama3_layer_16k():
    """One Llama-3-8B-shaped layer, T = 16384, 8 KV heads x 512 window rows:
    every unit against the oracle."""
    wl = wk.LLAMA3_8B_LAYER
    x = wk.make_inputs(wl, wk.seed_for(1), device="cuda")
    sc, _ = _gpu_scores(wl, x, 11, 1.0)
    want = O().score_keyformer(oshape(wl), x["q"], x["k"], 11, 1.0)
    got = sc.cpu().numpy().astype(np.float64)
    assert (np.abs(got - want) <= 1e-3 * want + 1e-30).all()


def test_keyformer_tensor_core_and_cuda_core_paths_agree(monkeypatch):
    """The same draws through both implementations: scores within 1e-3 of
    each other element by element (both are within 1e-3 of the oracle)."""
    wl, seed = CASES["bf16_gqa_rows512"]
    x = wk.make_inputs(wl, seed, device="cuda")
    monkeypatch.setenv("KVC_SCORE_IMPL", "tc")
    a, _ = _gpu_scores(wl, x, 5, 2.0)
    monkeypatch.setenv("KVC_SCORE_IMPL", "simt")
    b, _ = _gpu_scores(wl, x, 5, 2.0)
    a, b = a.double(), b.double()
    assert ((a - b).abs() <= 2e-3 * b + 1e-30).all()


def test_keyformer_rejects_bad_tau():
    kvc = K()
    wl, seed = CASES["f32_mha"]
    x = wk.make_inputs(wl, seed, device="cuda")
    s = kvc.shape_of(wl)
    ws = torch.empty(kvc.kvc_workspace_size(s, 1), dtype=torch.uint8, device="cuda")
    sc = torch.empty((wl.n_layers, wl.n_kv_heads, wl.seq_len), device="cuda")
    for tau in [0.0, -1.0, float("nan"), 1e31]:
        with pytest.raises(kvc.KvcError):
            kvc.kvc_score_keyformer(s, x["q"], x["k"], 1, tau, sc, ws)
