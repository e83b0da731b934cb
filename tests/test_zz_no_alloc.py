"""The allocation-free LayerNorm backward (for callers that cannot allocate
device memory; it uses the library's fixed device scratch) must give what the
allocating entry point gives, call after call.  Collected last on purpose."""
import numpy as np
import pytest
import torch

from scratch_gpt_step_train_b300 import kernels as K

pytestmark = pytest.mark.gpu


def _case(N, C, dtype, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    x = (torch.randn(N, C, generator=g, device="cuda") * 1.3 + 0.2).to(dtype)
    w = (1 + 0.1 * torch.randn(C, generator=g, device="cuda")).to(dtype)
    b = (0.1 * torch.randn(C, generator=g, device="cuda")).to(dtype)
    dy = torch.randn(N, C, generator=g, device="cuda").to(dtype)
    dx0 = torch.randn(N, C, generator=g, device="cuda").to(dtype)
    dw0 = torch.randn(C, generator=g, device="cuda")
    db0 = torch.randn(C, generator=g, device="cuda")
    y = torch.empty_like(x)
    mean = torch.empty(N, device="cuda")
    rstd = torch.empty(N, device="cuda")
    K.layernorm_forward(y, mean, rstd, x, w, b)
    return x, w, dy, dx0, dw0, db0, mean, rstd


@pytest.mark.parametrize("N,C", [(16384, 768), (300, 1600), (37, 200)], ids=["124M", "1558M-width", "ragged"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
def test_noalloc_matches_allocating_entry_twice(N, C, dtype):
    x, w, dy, dx0, dw0, db0, mean, rstd = _case(N, C, dtype, 1)
    ref = (dx0.clone(), dw0.clone(), db0.clone())
    K.layernorm_backward(ref[0], ref[1], ref[2], dy, x, w, mean, rstd)
    for _ in range(2):  # the shared array keeps the previous call's contents
        out = (dx0.clone(), dw0.clone(), db0.clone())
        K.layernorm_backward_noalloc(out[0], out[1], out[2], dy, x, w, mean, rstd)
        torch.cuda.synchronize()
        # the same kernels in the same fixed order: identical bits (which is
        # inside any tolerance the other LayerNorm tests use)
        for a, r in zip(out, ref):
            assert torch.equal(a, r)


def test_noalloc_rejects_rows_wider_than_its_scratch():
    # rejected before any work is queued, so the buffers' contents do not matter
    N, C = 8, 2056
    x, dy, dx = (torch.zeros(N, C, device="cuda") for _ in range(3))
    w, dw, db = (torch.zeros(C, device="cuda") for _ in range(3))
    mean, rstd = torch.zeros(N, device="cuda"), torch.ones(N, device="cuda")
    with pytest.raises(Exception) as e:
        K.layernorm_backward_noalloc(dx, dw, db, dy, x, w, mean, rstd)
    assert getattr(e.value, "code", None) == -1
