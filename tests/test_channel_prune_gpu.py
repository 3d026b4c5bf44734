"""GPU parity of the ThinK key-channel magnitude criterion (kvc_channel_prune)
on synthetic compacted keys, over the shapes the kernel's code paths split on:
head dims of 1, 2, 4 and 8 channel groups of 32 per lane, partial groups
(D = 40, 96, 200), fp32 and bf16, keep = D and keep = a few channels, layer
counts above 32 (the head's row offsets are summed over earlier layers by a
warp), empty and one-row heads, and long heads whose rows span many warps.

Rules ("ThinK: Thinner Key Cache by Query-Driven Pruning", "Magnitude-based
pruning"): channels bit-exact against the oracle's fp64 ranking except where
the oracle's two boundary norms are within 1e-9 relative (the GPU sums squares
in float-float pairs); the pruned bytes exact whenever the channels agree.  An
output buffer too small for the result raises KVC_DEV_OUT_CAPACITY and holds
exactly the leading elements that fit."""
import numpy as np
import pytest
import torch

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


# name: (L, H, D, T, W, dtype, budgets (None: seeded random in [0, P]), lambda)
CASES = {
    "d64_bf16_40_layers": (40, 2, 64, 300, 8, "bf16", None, 0.5),
    "d256_f32": (3, 2, 256, 500, 16, "f32", [0, 484, 37], 0.25),
    "d40_bf16_keep4": (2, 3, 40, 200, 8, "bf16", [150, 1], 0.9),
    "d200_bf16_keep_all": (2, 2, 200, 400, 32, "bf16", [368, 100], 0.0),
    "d96_f32": (2, 2, 96, 300, 8, "f32", [292, 50], 0.6),
    "d16_f32_one_group": (2, 2, 16, 100, 4, "f32", [96, 3], 0.5),
    "d128_bf16_long_heads": (2, 4, 128, 9000, 128, "bf16", [8872, 4000], 0.4),
}


def _make(name, seed=0):
    L, H, D, T, W, dt, budgets, lam = CASES[name]
    P = T - W
    g = np.random.default_rng(seed)
    bud = np.asarray(budgets if budgets is not None else g.integers(0, P + 1, size=L),
                     dtype=np.int32)
    rows = int(H * (np.clip(bud, 0, P).sum() + L * W))
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    # per-channel scales spread the norms apart, so near-ties are rare
    scale = torch.from_numpy(g.uniform(0.2, 3.0, size=D).astype(np.float32))
    k_out = (torch.from_numpy(g.standard_normal((rows, D)).astype(np.float32)) * scale).to(tdt)
    return L, H, D, T, W, dt, bud, lam, k_out.cuda()


def _run(name, capacity_short=0):
    kvc, o = K(), O()
    L, H, D, T, W, dt, bud, lam, k_out = _make(name)
    s = kvc.shape(L, H, H, D, T, W, dt)
    os_ = o.shape_of(L, H, H, D, T, W, dt)
    keep = kvc.kvc_keep_channels(lam, D)
    P = T - W
    total = int(H * np.clip(bud, 0, P).sum() * keep)
    ws = torch.empty(kvc.kvc_workspace_size(s, 1), dtype=torch.uint8, device="cuda")
    kvc.kvc_workspace_init(ws)
    chan = torch.full((L, H, keep), -1, dtype=torch.int32, device="cuda")
    kp = torch.zeros(max(1, total - capacity_short), dtype=k_out.dtype, device="cuda")
    kvc.kvc_channel_prune(s, k_out, torch.from_numpy(bud).cuda(), lam, chan, kp, ws)
    torch.cuda.synchronize()
    st = kvc.kvc_workspace_status(ws)
    ochan, norms, okp = o.channel_prune(os_, o.raw(k_out), bud, lam)
    return keep, chan.cpu().numpy(), kp, st, ochan, norms, okp


@pytest.mark.parametrize("name", list(CASES))
def test_channel_prune_matches_oracle(name):
    kvc, o = K(), O()
    keep, gchan, kp, st, ochan, norms, okp = _run(name)
    assert st == 0
    L, H = gchan.shape[:2]
    for l in range(L):
        for h in range(H):
            if not np.array_equal(gchan[l, h], ochan[l, h]):
                srt = np.sort(norms[l, h])[::-1]
                kth, nxt = srt[keep - 1], srt[keep]
                assert abs(kth - nxt) <= 1e-9 * kth, (name, l, h)
    if np.array_equal(gchan, ochan):
        assert np.array_equal(o.raw(kp[: okp.size]), okp), name
    # chosen channels strictly ascending and in range, every head
    assert np.all(np.diff(gchan, axis=-1) > 0) and gchan.min() >= 0


def test_channel_prune_reports_short_output():
    o = O()
    keep, gchan, kp, st, ochan, norms, okp = _run("d128_bf16_long_heads", capacity_short=1000)
    from eviction_kvc_score_gb300 import kvc
    assert st & kvc.DEV_OUT_CAPACITY
    assert np.array_equal(gchan, ochan)
    n = kp.numel()
    assert np.array_equal(o.raw(kp)[:n], okp[:n])
