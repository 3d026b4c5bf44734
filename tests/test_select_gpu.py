"""GPU parity of MBA, the layer budgets and top-K on synthetic score rows fed
straight to kvc_mba_budget / kvc_topk_select, against the oracle run on the
same fp32 scores (bit-exact: these are integer decisions on identical inputs).

Sources: blog post "ZigZagKV, KVCache 80% compression near-lossless",
sections "ZigZagKV's new observations" (MBA: fewest tokens reaching the mass
fraction), "ZigZagKV space allocation" (budgets) and "SnapKV" (top-K).

The rows cover the selection kernels' code paths: rows kept in shared memory
and rows read from global memory (T above 36,864), 16-byte aligned rows and
rows that are not (T not a multiple of 4), crossing buckets whose keys
overflow the per-warp gather lists (near-uniform scores), rows above 2^20
scores (64-bit bucket sums), heavy ties at the selection boundary, mass
fractions from 1/2 to 1, and crossings that sit exactly on a first-digit
bucket border."""
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


def _rows(kind, L, H, T, seed):
    """Non-negative fp32 rows summing to about 1 (column means of softmax
    rows do), in distributions that stress different buckets."""
    g = np.random.default_rng(seed)
    if kind == "lognormal":        # spread over many octaves
        x = np.exp(g.normal(0.0, 2.0, size=(L, H, T)))
    elif kind == "near_uniform":   # one first-digit bucket holds nearly every score
        x = 1.0 + 1e-3 * g.random((L, H, T))
    elif kind == "ties":           # a few distinct values, many equal keys
        x = g.integers(1, 5, size=(L, H, T)).astype(np.float64)
    elif kind == "heavy_tail":     # a few large scores and a flat floor
        x = g.pareto(1.2, size=(L, H, T)) + 1e-3
    else:
        raise ValueError(kind)
    x = x / x.sum(axis=-1, keepdims=True)
    return torch.from_numpy(x.astype(np.float32))


# name: (distribution, L, H, T, W, num, den)
CASES = {
    "cached_aligned_lognormal": ("lognormal", 3, 2, 32768, 128, 9, 10),
    "cached_unaligned_heavy_tail": ("heavy_tail", 2, 3, 10001, 17, 9, 10),
    "cached_near_uniform_overflow": ("near_uniform", 2, 2, 30000, 64, 9, 10),
    "cached_ties_half": ("ties", 2, 2, 5000, 8, 1, 2),
    "uncached_aligned_lognormal": ("lognormal", 2, 2, 65536, 128, 99, 100),
    "uncached_unaligned_near_uniform": ("near_uniform", 1, 2, 40003, 3, 9, 10),
    "uncached_ties_all_mass": ("ties", 1, 2, 50000, 100, 1, 1),
    "above_2p20_lognormal": ("lognormal", 1, 1, (1 << 20) + 3, 1000, 9, 10),
}


@pytest.mark.parametrize("name", list(CASES))
def test_mba_budget_topk_match_oracle(name):
    kvc, o = K(), O()
    kind, L, H, T, W, num, den = CASES[name]
    P = T - W
    sc = _rows(kind, L, H, T, seed=len(name))
    s = kvc.shape(L, H, H, 64, T, W, "f32")
    floor = min(P, 16)
    total = L * floor + (L * P - L * floor) // 3
    k_max = P
    ws = torch.empty(kvc.kvc_workspace_size(s, k_max), dtype=torch.uint8, device="cuda")
    kvc.kvc_workspace_init(ws)
    scd = sc.cuda()
    mba = torch.empty((L, H), dtype=torch.int32, device="cuda")
    bud = torch.empty(L, dtype=torch.int32, device="cuda")
    kvc.kvc_mba_budget(s, scd, num, den, total, floor, mba, bud, ws)
    idx = torch.full((L, H, k_max), -1, dtype=torch.int32, device="cuda")
    kvc.kvc_topk_select(s, scd, bud, k_max, idx, ws)
    torch.cuda.synchronize()
    assert kvc.kvc_workspace_status(ws) == 0
    c = sc.double().numpy()
    want_mba = np.array([[o.mba(c[l, h], num, den) for h in range(H)] for l in range(L)])
    assert np.array_equal(mba.cpu().numpy(), want_mba), name
    want_bud = o.budget(want_mba, P, total, floor)
    assert np.array_equal(bud.cpu().numpy(), want_bud), name
    got = idx.cpu().numpy()
    for l in range(L):
        B = int(want_bud[l])
        for h in range(H):
            assert np.array_equal(got[l, h, :B], o.topk(c[l, h], P, B)), (name, l, h)
            assert (got[l, h, B:] == -1).all(), (name, l, h)


@pytest.mark.parametrize("T", [1000, 40000])
def test_topk_every_budget_shape_on_ties(T):
    """Budgets 1, a tie-splitting middle value, P - 1 and P on rows of four
    distinct values: the kept ties are the lowest positions."""
    kvc, o = K(), O()
    L, H, W = 4, 1, 8
    P = T - W
    sc = _rows("ties", L, H, T, seed=T)
    s = kvc.shape(L, H, H, 64, T, W, "f32")
    ws = torch.empty(kvc.kvc_workspace_size(s, P), dtype=torch.uint8, device="cuda")
    kvc.kvc_workspace_init(ws)
    budgets = [1, P // 3 + 1, P - 1, P]
    idx = torch.full((L, H, P), -1, dtype=torch.int32, device="cuda")
    kvc.kvc_topk_select(s, sc.cuda(), torch.tensor(budgets, dtype=torch.int32, device="cuda"), P,
                        idx, ws)
    torch.cuda.synchronize()
    assert kvc.kvc_workspace_status(ws) == 0
    c = sc.double().numpy()
    got = idx.cpu().numpy()
    for l, B in enumerate(budgets):
        assert np.array_equal(got[l, 0, :B], o.topk(c[l, 0], P, B)), (T, B)


def _f32(e, w):
    """The fp32 value w * 2^(e - 150) (w the 24-bit significand with its
    leading one), from its bits."""
    return np.array([(e << 23) | (w - (1 << 23))], dtype=np.uint32).view(np.float32)[0]


def _boundary_rows(T=1000):
    """Two rows whose 90% crossing sits exactly on the border between two
    first-digit buckets (all scores of a bucket share exponent and top four
    significand bits).  In "low" the top bucket's scores carry a set last
    significand bit and its mass is exactly 9x the rest, so the whole top
    bucket is needed (MBA 90) while any mass estimate that drops low bits
    puts the crossing one bucket lower; "high" mirrors it (the lower bucket
    carries the low bits; the crossing takes one score from it, MBA 91)."""
    z = [np.float32(0.0)]
    low = ([_f32(120, 2**23 + 1)] * 90 + [_f32(119, 2**23)] * 20 + [_f32(100, 10 * 2**20)] +
           z * (T - 111))
    high = [_f32(120, 2**23)] * 90 + [_f32(119, 2**23 + 1)] * 20 + z * (T - 110)
    g = np.random.default_rng(11)
    return {name: np.array(r, dtype=np.float32)[g.permutation(T)]
            for name, r in (("low", low), ("high", high))}


def test_mba_crossing_on_a_bucket_boundary():
    kvc, o = K(), O()
    rows = _boundary_rows()
    sc = torch.from_numpy(np.stack([rows["low"], rows["high"]])[:, None, :].copy())
    L, H, T, W = 2, 1, sc.shape[-1], 8
    P = T - W
    s = kvc.shape(L, H, H, 64, T, W, "f32")
    ws = torch.empty(kvc.kvc_workspace_size(s, P), dtype=torch.uint8, device="cuda")
    kvc.kvc_workspace_init(ws)
    scd = sc.cuda()
    mba = torch.empty((L, H), dtype=torch.int32, device="cuda")
    bud = torch.empty(L, dtype=torch.int32, device="cuda")
    kvc.kvc_mba_budget(s, scd, 9, 10, 2 * 100, 10, mba, bud, ws)
    idx = torch.full((L, H, P), -1, dtype=torch.int32, device="cuda")
    kvc.kvc_topk_select(s, scd, bud, P, idx, ws)
    torch.cuda.synchronize()
    assert kvc.kvc_workspace_status(ws) == 0
    c = sc.double().numpy()
    want = [o.mba(c[l, 0], 9, 10) for l in range(L)]
    assert want == [90, 91]                      # the rows are what they claim to be
    assert mba[:, 0].tolist() == want
    want_bud = o.budget(np.array(want, dtype=np.int32)[:, None], P, 2 * 100, 10)
    assert bud.tolist() == want_bud.tolist()
    got = idx.cpu().numpy()
    for l in range(L):
        B = int(want_bud[l])
        assert np.array_equal(got[l, 0, :B], o.topk(c[l, 0], P, B)), l


@pytest.mark.parametrize("T", [3000, 40000])
def test_negative_zero_scores_count_as_zero(T):
    """-0.0 and +0.0 are the same score: MBA with the whole mass counts the
    positive scores, and a budget reaching into the zeros keeps the
    lowest-index zeros whatever their sign."""
    kvc, o = K(), O()
    L, H, W = 2, 1, 8
    P = T - W
    g = np.random.default_rng(T + 5)
    x = np.zeros((L, H, T), dtype=np.float32)
    npos = 500
    for l in range(L):
        pos = g.choice(P, size=npos, replace=False)
        v = np.exp(g.normal(0.0, 1.0, size=npos))
        x[l, 0, pos] = (v / v.sum()).astype(np.float32)
    neg = (x == 0) & (g.random(x.shape) < 0.5)
    x[neg] = np.float32(-0.0)
    assert np.signbit(x).sum() > 0
    s = kvc.shape(L, H, H, 64, T, W, "f32")
    ws = torch.empty(kvc.kvc_workspace_size(s, P), dtype=torch.uint8, device="cuda")
    kvc.kvc_workspace_init(ws)
    scd = torch.from_numpy(x).cuda()
    c = x.astype(np.float64)
    for num, den in ((1, 1), (9, 10)):
        mba = torch.empty((L, H), dtype=torch.int32, device="cuda")
        bud = torch.empty(L, dtype=torch.int32, device="cuda")
        kvc.kvc_mba_budget(s, scd, num, den, L * 100, 10, mba, bud, ws)
        torch.cuda.synchronize()
        want = [o.mba(c[l, 0], num, den) for l in range(L)]
        assert mba[:, 0].tolist() == want, (num, den)
    assert want[0] <= npos
    budgets = [npos + 300, npos - 1]
    idx = torch.full((L, H, P), -1, dtype=torch.int32, device="cuda")
    kvc.kvc_topk_select(s, scd, torch.tensor(budgets, dtype=torch.int32, device="cuda"), P, idx,
                        ws)
    torch.cuda.synchronize()
    assert kvc.kvc_workspace_status(ws) == 0
    got = idx.cpu().numpy()
    for l, B in enumerate(budgets):
        assert np.array_equal(got[l, 0, :B], o.topk(c[l, 0], P, B)), (T, B)


@pytest.mark.parametrize("L,H,T", [(32, 2, 600), (33, 2, 600), (40, 3, 700), (1024, 1, 300)])
def test_budgets_across_layer_counts(L, H, T):
    """The layer budgets are computed by the last MBA block: one lane per
    layer for up to 32 layers, block-wide sums beyond (up to the 1024-layer
    limit).  Budgets tight enough that the cap at P and the largest-remainder
    leftovers both occur; MBA, budgets and top-K against the oracle."""
    kvc, o = K(), O()
    W = 8
    P = T - W
    sc = _rows("lognormal", L, H, T, seed=L * 7 + H)
    s = kvc.shape(L, H, H, 64, T, W, "f32")
    floor = 5
    for total in (L * floor + 7, (L * P * 3) // 4 + 1):
        ws = torch.empty(kvc.kvc_workspace_size(s, P), dtype=torch.uint8, device="cuda")
        kvc.kvc_workspace_init(ws)
        scd = sc.cuda()
        mba = torch.empty((L, H), dtype=torch.int32, device="cuda")
        bud = torch.empty(L, dtype=torch.int32, device="cuda")
        kvc.kvc_mba_budget(s, scd, 9, 10, total, floor, mba, bud, ws)
        idx = torch.full((L, H, P), -1, dtype=torch.int32, device="cuda")
        kvc.kvc_topk_select(s, scd, bud, P, idx, ws)
        torch.cuda.synchronize()
        assert kvc.kvc_workspace_status(ws) == 0
        c = sc.double().numpy()
        want_mba = np.array([[o.mba(c[l, h], 9, 10) for h in range(H)] for l in range(L)])
        assert np.array_equal(mba.cpu().numpy(), want_mba), (L, total)
        want_bud = o.budget(want_mba, P, total, floor)
        got_bud = bud.cpu().numpy()
        assert np.array_equal(got_bud, want_bud), (L, total)
        assert int(got_bud.sum()) == total
        got = idx.cpu().numpy()
        for l in range(0, L, max(1, L // 16)):
            B = int(want_bud[l])
            for h in range(H):
                assert np.array_equal(got[l, h, :B], o.topk(c[l, h], P, B)), (L, total, l, h)


@pytest.mark.parametrize("Hkv", [8, 40])
def test_head_budgets_beyond_one_warp(Hkv):
    """kvc_head_budget runs one thread per KV head: 40 heads take two warps of
    block-wide sums."""
    kvc, o = K(), O()
    L, T, W = 3, 800, 16
    P = T - W
    g = np.random.default_rng(Hkv)
    mba = torch.from_numpy(g.integers(0, P, size=(L, Hkv)).astype(np.int32)).cuda()
    bud = torch.from_numpy(np.array([P // 3, P - 1, 7], dtype=np.int32)).cuda()
    s = kvc.shape(L, Hkv, Hkv, 64, T, W, "f32")
    ws = torch.empty(kvc.kvc_workspace_size(s, P), dtype=torch.uint8, device="cuda")
    kvc.kvc_workspace_init(ws)
    hb = torch.empty((L, Hkv), dtype=torch.int32, device="cuda")
    kvc.kvc_head_budget(s, mba, bud, hb, ws)
    torch.cuda.synchronize()
    want = o.head_budget(mba.cpu().numpy(), bud.cpu().numpy(), P)
    assert np.array_equal(hb.cpu().numpy(), want)


@pytest.mark.parametrize("L,H,T", [(25, 8, 3000), (50, 4, 3000), (25, 8, 30000), (50, 4, 30000),
                                   (25, 8, 3001), (25, 8, 30001)])
def test_more_heads_than_sms(L, H, T):
    """200 heads: more than one wave of 1024-thread blocks on a GB300 (152
    SMs), so MBA runs as 512-thread blocks, two per SM, for rows up to 36,864
    scores (rows of 3,000 held in shared memory, rows of 30,000 read from L2);
    one lane per layer (25) and block-wide sums (50) for the budgets; rows
    whose length is not a multiple of four take the scalar visits."""
    kvc, o = K(), O()
    W = 16
    P = T - W
    sc = _rows("lognormal", L, H, T, seed=L * H + T)
    s = kvc.shape(L, H, H, 64, T, W, "f32")
    floor = 8
    total = L * floor + (L * P - L * floor) // 5
    ws = torch.empty(kvc.kvc_workspace_size(s, P), dtype=torch.uint8, device="cuda")
    kvc.kvc_workspace_init(ws)
    scd = sc.cuda()
    mba = torch.empty((L, H), dtype=torch.int32, device="cuda")
    bud = torch.empty(L, dtype=torch.int32, device="cuda")
    kvc.kvc_mba_budget(s, scd, 9, 10, total, floor, mba, bud, ws)
    idx = torch.full((L, H, P), -1, dtype=torch.int32, device="cuda")
    kvc.kvc_topk_select(s, scd, bud, P, idx, ws)
    torch.cuda.synchronize()
    assert kvc.kvc_workspace_status(ws) == 0
    c = sc.double().numpy()
    want_mba = np.array([[o.mba(c[l, h], 9, 10) for h in range(H)] for l in range(L)])
    assert np.array_equal(mba.cpu().numpy(), want_mba)
    want_bud = o.budget(want_mba, P, total, floor)
    assert np.array_equal(bud.cpu().numpy(), want_bud)
    got = idx.cpu().numpy()
    for l in range(0, L, 3):
        B = int(want_bud[l])
        for h in range(H):
            assert np.array_equal(got[l, h, :B], o.topk(c[l, h], P, B)), (l, h)
