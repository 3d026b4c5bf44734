"""kvc_score_noalloc: the score entry point for callers that may not allocate
device memory (hosts that pass a plugin only its inputs and outputs and own
all device memory themselves).  Its scratch is a fixed array inside the
library that every call reuses, so it must give the oracle's scores, and the
very same bits as kvc_score with a caller workspace, call after call -- also
right after a call of another shape has left different row statistics in that
array.

This file is collected last on purpose, and it builds and loads the library
itself, so it passes both alone in a fresh process and after the others."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

RTOL = 1e-3      # the score tolerance used by the parity tests
ATOL = 1e-30


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    from eviction_kvc_score_gb300 import kvc as k
    return k


def _cases():
    from eviction_kvc_score_gb300 import workloads as wk
    return {
        # tensor cores: 512 window rows, ragged last tile
        "bf16_tensor_core": wk.ZIGZAG_32K.scaled(n_layers=3, n_kv_heads=2, n_q_heads=8,
                                                 seq_len=5000, total_budget=3 * 500,
                                                 layer_floor=50),
        # CUDA cores: fp32 inputs
        "f32_cuda_core": wk.TINY,
    }


def _other(wl):
    """A shape whose split differs from wl's (other row padding, other slot
    count, other unit count): its call leaves different row statistics in the
    shared array."""
    from eviction_kvc_score_gb300 import workloads as wk
    if wl.dtype == "bf16":
        return wk.ZIGZAG_32K.scaled(n_layers=1, n_kv_heads=5, n_q_heads=10, seq_len=20000,
                                    window=96, total_budget=900, layer_floor=100)
    return wk.TINY.scaled(n_layers=2, n_kv_heads=3, n_q_heads=3, seq_len=3000, window=50)


def _oracle_scores(wl, x):
    from oracle import oracle as O
    s = O.shape_of(wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.seq_len,
                   wl.window, wl.dtype)
    return O.score(s, x["q"], x["k"])


@pytest.mark.parametrize("case", ["bf16_tensor_core", "f32_cuda_core"])
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(kvc, case):
    from eviction_kvc_score_gb300 import workloads as wk
    wl = _cases()[case]
    x = wk.make_inputs(wl, 77, device="cuda")
    s = kvc.shape_of(wl)
    ws = torch.empty(kvc.kvc_workspace_size(s, 0), dtype=torch.uint8, device="cuda")
    kvc.kvc_workspace_init(ws)
    ref = torch.empty((wl.n_layers, wl.n_kv_heads, wl.seq_len), device="cuda")
    kvc.kvc_score(s, x["q"], x["k"], ref, ws)
    ora = _oracle_scores(wl, x)

    other = _other(wl)
    xo = wk.make_inputs(other, 78, device="cuda")
    so = kvc.shape_of(other)
    out_o = torch.empty((other.n_layers, other.n_kv_heads, other.seq_len), device="cuda")

    status = torch.ones(1, dtype=torch.int32, device="cuda")
    for _ in range(2):                      # two calls in a row share the array
        out = torch.full_like(ref, float("nan"))
        kvc.kvc_score_noalloc(s, x["q"], x["k"], out, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0      # zeroed by the call, no device error
        # same kernels on the same split: the very same bits as kvc_score
        assert torch.equal(out, ref)
        got = out.double().cpu().numpy()
        assert (np.abs(got - ora) <= RTOL * ora + ATOL).all()
        # a call of another shape rewrites the array before the next one
        kvc.kvc_score_noalloc(so, xo["q"], xo["k"], out_o, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
    np.testing.assert_allclose(out_o.double().sum(-1).cpu().numpy(), 1.0, atol=1e-5)
    assert kvc.kvc_workspace_status(ws) == 0


def test_noalloc_rejects_shapes_beyond_its_scratch(kvc):
    # 4096 (layer, head) units x 512 window rows need far more than 8 MiB of
    # row statistics; the call must refuse before touching the GPU.
    s = kvc.shape(128, 128, 32, 128, 4096, 128, "bf16")
    fake = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_score_noalloc(s, fake, fake, torch.empty(1, device="cuda"))
    assert e.value.code == -2
    assert "static buffer" in kvc.kvc_last_error()


def test_noalloc_rejects_a_misaligned_status_word(kvc):
    # the kernels OR bits into the status word with 32-bit atomics: a word
    # that is not 4-byte aligned is refused before anything is launched
    from eviction_kvc_score_gb300 import workloads as wk
    wl = wk.TINY
    x = wk.make_inputs(wl, 5, device="cuda")
    out = torch.empty((wl.n_layers, wl.n_kv_heads, wl.seq_len), device="cuda")
    word = torch.zeros(8, dtype=torch.uint8, device="cuda")[1:5]
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_score_noalloc(kvc.shape_of(wl), x["q"], x["k"], out, word)
    assert e.value.code == -1
    assert "4-byte aligned" in kvc.kvc_last_error()
