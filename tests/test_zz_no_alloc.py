"""kvc_score_noalloc: the score entry point for callers that may not allocate
device memory (hosts that pass a plugin only its inputs and outputs and own
all device memory themselves).  Its scratch is a fixed array inside the
library; it must give the same scores as kvc_score with a caller workspace,
call after call, since every call reuses that array.

This file is collected last on purpose, and it builds and loads the library
itself, so it passes both alone in a fresh process and after the others."""
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


def _close(a, b):
    return bool(((a.double() - b.double()).abs() <= RTOL * b.double().abs() + ATOL).all())


@pytest.mark.parametrize("case", ["bf16_tensor_core", "f32_cuda_core"])
def test_noalloc_matches_workspace_entry_point_twice(kvc, case):
    from eviction_kvc_score_gb300 import workloads as wk
    if case == "bf16_tensor_core":
        wl = wk.ZIGZAG_32K.scaled(n_layers=3, n_kv_heads=2, n_q_heads=8, seq_len=5000,
                                  total_budget=3 * 500, layer_floor=50)
    else:
        wl = wk.TINY
    x = wk.make_inputs(wl, 77, device="cuda")
    s = kvc.shape_of(wl)
    ws = torch.empty(kvc.kvc_workspace_size(s, 0), dtype=torch.uint8, device="cuda")
    kvc.kvc_workspace_init(ws)
    ref = torch.empty((wl.n_layers, wl.n_kv_heads, wl.seq_len), device="cuda")
    kvc.kvc_score(s, x["q"], x["k"], ref, ws)
    status = torch.ones(1, dtype=torch.int32, device="cuda")
    for _ in range(2):                      # two calls in a row share the array
        out = torch.full_like(ref, float("nan"))
        kvc.kvc_score_noalloc(s, x["q"], x["k"], out, status)
        torch.cuda.synchronize()
        assert _close(out, ref)
        assert int(status.item()) == 0      # zeroed by the call, no device error
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
