"""GPU parity of the optional SnapKV score pooling (average or max over an odd
1D kernel, window positions copied) and of top-K run on the pooled scores.

Max mode is exact.  Average mode sums at most `kernel` fp32 terms left to
right and divides once, so each output is within (kernel + 1) * 2^-24
relative of the fp64 mean of the same fp32 inputs.  Top-K indices on the
pooled scores are bit-exact against the oracle run on the GPU's own pooled
fp32 values.
"""
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


def _pool_case(L, H, T, W, kernel, mode, seed):
    kvc, ora = K(), O()
    g = torch.Generator().manual_seed(seed)
    # heavy-tailed positive scores with a run of exact ties
    sc = torch.rand((L, H, T), generator=g, dtype=torch.float64) ** 6
    sc[..., 100:140] = 0.25
    sc = (sc / sc.sum(-1, keepdim=True)).float()
    s = kvc.shape(L, H, H, 16, T, W, "f32")
    ws = torch.empty(kvc.kvc_workspace_size(s, 1), dtype=torch.uint8, device="cuda")
    kvc.kvc_workspace_init(ws)
    dev = sc.cuda()
    out = torch.full_like(dev, float("nan"))
    kvc.kvc_pool_scores(s, dev, kernel, mode, out, ws)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    want = ora.pool(ora.shape_of(L, H, H, 16, T, W, "f32"), sc.numpy(), kernel, mode)
    return kvc, s, ws, out, got, want


@pytest.mark.parametrize("kernel", [1, 3, 7, 15, 31, 255])
@pytest.mark.parametrize("mode", [0, 1])
def test_pool_matches_oracle(kernel, mode):
    L, H, T, W = 2, 3, 5000, 37           # 5 tiles of 1024 with a ragged tail
    *_, got, want = _pool_case(L, H, T, W, kernel, mode, 100 + kernel)
    if mode == 1:
        np.testing.assert_array_equal(got, want)
    else:
        np.testing.assert_allclose(got, want, rtol=(kernel + 1) * 2.0 ** -24, atol=0)
    np.testing.assert_array_equal(got[..., T - W:], want[..., T - W:])


def test_pool_identity_and_prefix_shorter_than_kernel():
    *_, got, want = _pool_case(1, 2, 300, 290, 1, 0, 7)
    np.testing.assert_array_equal(got, want)
    *_, got2, want2 = _pool_case(1, 2, 300, 290, 31, 0, 7)   # P = 10 < kernel
    np.testing.assert_allclose(got2, want2, rtol=32 * 2.0 ** -24, atol=0)


def test_pool_many_heads_beyond_one_grid_row():
    # more (layer, head) pairs than one launch row holds: the blocks loop
    *_, got, want = _pool_case(70000, 1, 40, 3, 5, 1, 11)
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("kernel,mode", [(7, 0), (7, 1), (31, 0)])
def test_topk_on_pooled_scores_bit_exact(kernel, mode):
    L, H, T, W = 3, 4, 6000, 64
    P = T - W
    kvc, s, ws, out, got, _ = _pool_case(L, H, T, W, kernel, mode, 300 + kernel)
    ora = O()
    budget = torch.tensor([0, 777, P], dtype=torch.int32, device="cuda")
    idx = torch.full((L, H, P), -1, dtype=torch.int32, device="cuda")
    kvc.kvc_topk_select(s, out, budget, P, idx, ws)
    torch.cuda.synchronize()
    assert kvc.kvc_workspace_status(ws) == 0
    want = ora.topk_all(ora.shape_of(L, H, H, 16, T, W, "f32"), out.cpu().numpy(),
                        budget.cpu().numpy(), P)
    for l, n in enumerate(budget.tolist()):
        np.testing.assert_array_equal(idx[l, :, :n].cpu().numpy(), want[l, :, :n])


def test_pool_of_gpu_scores_end_to_end():
    """Pooling the GPU's window scores agrees with pooling the oracle's fp64
    scores to the score tolerance (a mean or max of values that are each
    within 1e-3 relative is itself within 1e-3 relative)."""
    kvc, ora = K(), O()
    wl = wk.Workload("pool_e2e", n_layers=2, n_q_heads=8, n_kv_heads=2, head_dim=128,
                     seq_len=1500, window=48, dtype="bf16", total_budget=600, layer_floor=16)
    x = wk.make_inputs(wl, 4242, device="cuda")
    s = kvc.shape_of(wl)
    ws = torch.empty(kvc.kvc_workspace_size(s, wl.k_max), dtype=torch.uint8, device="cuda")
    kvc.kvc_workspace_init(ws)
    sc = torch.empty((wl.n_layers, wl.n_kv_heads, wl.seq_len), device="cuda")
    kvc.kvc_score(s, x["q"], x["k"], sc, ws)
    out = torch.empty_like(sc)
    kvc.kvc_pool_scores(s, sc, 7, 0, out, ws)
    torch.cuda.synchronize()
    os_ = ora.shape_of(wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.seq_len,
                       wl.window, wl.dtype)
    want = ora.pool(os_, ora.score(os_, x["q"], x["k"]), 7, 0)
    got = out.cpu().numpy().astype(np.float64)
    assert (np.abs(got - want) <= 1e-3 * want + 1e-30).all()


def test_pool_rejects_bad_arguments():
    kvc = K()
    s = kvc.shape(1, 1, 1, 16, 100, 4, "f32")
    ws = torch.empty(kvc.kvc_workspace_size(s, 1), dtype=torch.uint8, device="cuda")
    sc = torch.rand((1, 1, 100), device="cuda")
    out = torch.empty_like(sc)
    for kernel, mode, code in [(2, 0, -1), (0, 0, -1), (257, 0, -2), (3, 2, -1)]:
        with pytest.raises(kvc.KvcError) as e:
            kvc.kvc_pool_scores(s, sc, kernel, mode, out, ws)
        assert e.value.code == code
    with pytest.raises(kvc.KvcError):
        kvc.kvc_pool_scores(s, sc, 3, 0, sc, ws)
