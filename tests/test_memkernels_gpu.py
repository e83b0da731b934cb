"""Parity of the memory-bound kernels of the step against the oracle (fp64),
at the full GPT-2 124M micro-batch (B=16, T=1024, C=768, V=50257) and at
small ragged shapes: embedding forward/backward, LayerNorm forward/backward,
bias gradient, fused softmax cross-entropy (loss + dlogits in place).

Gathers and scatters are checked bit-exactly: the embedding forward in fp32 is
one fp32 add (the fp32 build of the oracle does the same add), and the
embedding backward is fed small integers, whose sums are exact in any order.
"""
import numpy as np
import pytest
import torch

from oracle.pyoracle import Ops
from scratch_gpt_step_train_b300 import inputs
from scratch_gpt_step_train_b300 import kernels as K
from parity import assert_close

pytestmark = pytest.mark.gpu
ops = Ops("double")
ops32 = Ops("float")
FULL = dict(B=16, T=1024, C=768, V=50257)


def _t(x, dtype):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dtype).cuda()


def _np(t):
    return t.double().cpu().numpy()


# ------------------------------------------------------------------ embedding

@pytest.mark.parametrize("B,T,C,V", [(2, 37, 40, 100), (16, 1024, 768, 50257)], ids=["small", "full"])
def test_encoder_forward_fp32_bit_exact(B, T, C, V):
    rng = np.random.default_rng(0)
    wte = rng.normal(0, 0.02, (V, C)).astype(np.float32)
    wpe = rng.normal(0, 0.02, (T, C)).astype(np.float32)
    tok = inputs.zipf_batches(1, 1, B, T, V)[0][0]
    out = torch.empty(B, T, C, device="cuda")
    err = K.encoder_forward(out, torch.from_numpy(tok).cuda(), _t(wte, torch.float32),
                            _t(wpe, torch.float32), V)
    ref = ops32.encoder_forward(tok, wte, wpe)
    assert np.array_equal(out.cpu().numpy(), ref)
    assert int(err[0]) == 0


def test_encoder_forward_bf16_and_range_flag():
    B, T, C, V = 4, 64, 128, 1000
    rng = np.random.default_rng(1)
    wte = _t(rng.normal(0, 0.02, (V, C)), torch.bfloat16)
    wpe = _t(rng.normal(0, 0.02, (T, C)), torch.bfloat16)
    tok = inputs.uniform_batch(2, B, T, V)[0]
    out = torch.empty(B, T, C, dtype=torch.bfloat16, device="cuda")
    err = K.encoder_forward(out, torch.from_numpy(tok).cuda(), wte, wpe, V)
    ref = ops.encoder_forward(tok, _np(wte), _np(wpe))
    # one RNE rounding to bf16 (unit roundoff 2^-8) of the exact fp32 sum
    assert np.all(np.abs(_np(out) - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-30)
    assert int(err[0]) == 0
    bad = tok.copy()
    bad[1, 5] = V
    err = K.encoder_forward(out, torch.from_numpy(bad).cuda(), wte, wpe, V)
    assert int(err[0]) & 1


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_encoder_backward_full_size_exact_indexing(dtype):
    """integer-valued dx: every row sum is exact, so any misrouted row shows"""
    B, T, C, V = FULL["B"], FULL["T"], FULL["C"], FULL["V"]
    Vp = ((V + 127) // 128) * 128
    tok = inputs.zipf_batches(2, 1, B, T, V)[0][0]
    rng = np.random.default_rng(3)
    dx = rng.integers(-4, 5, (B, T, C)).astype(np.float32)
    dwte0 = rng.integers(-3, 4, (Vp, C)).astype(np.float32)
    dwpe0 = rng.integers(-3, 4, (T, C)).astype(np.float32)
    dwte = torch.from_numpy(dwte0).cuda()
    dwpe = torch.from_numpy(dwpe0).cuda()
    K.encoder_backward(dwte, dwpe, _t(dx, dtype), torch.from_numpy(tok).cuda())
    rwte, rwpe = ops.encoder_backward(dx.astype(np.float64), tok, Vp)
    assert np.array_equal(dwte.cpu().numpy(), dwte0 + rwte)
    assert np.array_equal(dwpe.cpu().numpy(), dwpe0 + rwpe)


def test_encoder_backward_heavy_tokens_in_every_scan_block():
    """Zipf tokens relabelled by a seeded permutation: the tokens with more
    than one 32-row chunk lie all over [0, Vp), in every 1024-token block of
    the bucket scan; integer-valued dx, so the sums are exact"""
    B, T, C, V = 8, 1024, 256, 50257
    Vp = ((V + 127) // 128) * 128
    tok = inputs.zipf_batches(6, 1, B, T, V)[0][0]
    perm = np.random.default_rng(7).permutation(V).astype(tok.dtype)
    tok = perm[tok]
    counts = np.bincount(tok.ravel(), minlength=Vp)
    heavy = np.nonzero(counts > 32)[0]
    assert len(np.unique(heavy // 1024)) >= 5  # the case this test is for
    rng = np.random.default_rng(8)
    dx = rng.integers(-4, 5, (B, T, C)).astype(np.float32)
    dwte = torch.zeros(Vp, C, device="cuda")
    dwpe = torch.zeros(T, C, device="cuda")
    K.encoder_backward(dwte, dwpe, _t(dx, torch.float32), torch.from_numpy(tok).cuda())
    rwte, rwpe = ops.encoder_backward(dx.astype(np.float64), tok, Vp)
    assert np.array_equal(dwte.cpu().numpy(), rwte)
    assert np.array_equal(dwpe.cpu().numpy(), rwpe)


def test_encoder_backward_real_values_and_determinism():
    B, T, C, V = 8, 200, 64, 300
    Vp = 384
    tok = inputs.zipf_batches(4, 1, B, T, V)[0][0]  # long buckets for the head ids
    dx = np.random.default_rng(5).normal(0, 1, (B, T, C)).astype(np.float32)
    outs = []
    for _ in range(2):
        dwte = torch.zeros(Vp, C, device="cuda")
        dwpe = torch.zeros(T, C, device="cuda")
        K.encoder_backward(dwte, dwpe, _t(dx, torch.float32), torch.from_numpy(tok).cuda())
        outs.append((dwte.cpu().numpy(), dwpe.cpu().numpy()))
    rwte, rwpe = ops.encoder_backward(dx.astype(np.float64), tok, Vp)
    assert_close(outs[0][0], rwte, 1e-6, "dwte")
    assert_close(outs[0][1], rwpe, 1e-6, "dwpe")
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])


# ------------------------------------------------------------------ layernorm

def _ln_inputs(N, C, seed):
    rng = np.random.default_rng(seed)
    x = rng.normal(0.2, 1.3, (N, C))
    w = rng.normal(1, 0.1, C)
    b = rng.normal(0, 0.1, C)
    return x, w, b


@pytest.mark.parametrize("N,C", [(37, 200), (16384, 768), (300, 1600), (8192, 1024)],
                         ids=["small", "full", "c1600", "c1024"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_layernorm_forward(N, C, dtype):
    x, w, b = _ln_inputs(N, C, 1)
    xt, wt, bt = _t(x, dtype), _t(w, dtype), _t(b, dtype)
    out = torch.empty(N, C, dtype=dtype, device="cuda")
    mean = torch.empty(N, device="cuda")
    rstd = torch.empty(N, device="cuda")
    K.layernorm_forward(out, mean, rstd, xt, wt, bt)
    ref, rm, rr = ops.layernorm_forward(_np(xt), _np(wt), _np(bt))
    if dtype == torch.float32:
        assert_close(_np(out), ref, 1e-5, "y")
    else:
        assert np.all(np.abs(_np(out) - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5)
    assert np.abs(mean.double().cpu().numpy() - rm).max() <= 1e-5
    assert np.all(np.abs(rstd.double().cpu().numpy() - rr) <= 1e-5 * rr)


@pytest.mark.parametrize("mode", ["accum", "overwrite_dxsum"])
@pytest.mark.parametrize("N,C", [(37, 200), (16384, 768), (300, 1600), (8192, 1024)],
                         ids=["small", "full", "c1600", "c1024"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_layernorm_backward(N, C, dtype, mode):
    x, w, b = _ln_inputs(N, C, 2)
    rng = np.random.default_rng(3)
    dy = rng.normal(0, 1, (N, C))
    dx0 = rng.normal(0, 1, (N, C))
    xt, wt, bt, dyt = _t(x, dtype), _t(w, dtype), _t(b, dtype), _t(dy, dtype)
    out = torch.empty(N, C, dtype=dtype, device="cuda")
    mean = torch.empty(N, device="cuda")
    rstd = torch.empty(N, device="cuda")
    K.layernorm_forward(out, mean, rstd, xt, wt, bt)
    accumulate = mode == "accum"
    dx = _t(dx0, dtype)
    dx0r = _np(dx) if accumulate else np.zeros((N, C))
    dw0 = rng.normal(0, 1, C).astype(np.float32)
    db0 = rng.normal(0, 1, C).astype(np.float32)
    dw = torch.from_numpy(dw0).cuda()
    db = torch.from_numpy(db0).cuda()
    dxsum = None
    if not accumulate:
        ds0 = rng.normal(0, 1, C).astype(np.float32)
        dxsum = torch.from_numpy(ds0).cuda()
    K.layernorm_backward(dx, dw, db, dyt, xt, wt, mean, rstd, dxsum=dxsum, accumulate=accumulate)
    _, rm, rr = ops.layernorm_forward(_np(xt), _np(wt), _np(bt))
    rdx, rdw, rdb = ops.layernorm_backward(_np(dyt), _np(xt), _np(wt), rm, rr)
    tol = 1e-4 if dtype == torch.float32 else 1e-2
    assert_close(_np(dx) - dx0r, rdx, tol, "dx")
    assert_close(dw.double().cpu().numpy() - dw0, rdw, 1e-4, "dw")
    assert_close(db.double().cpu().numpy() - db0, rdb, 1e-4, "db")
    if dxsum is not None:
        # dxsum is the column sum of the rows as written (dx itself is checked
        # against the oracle above): exact up to fp32 summation, whose error is
        # at most about N * 2^-24 * sum|dx| per column
        st = _np(dx)
        got = dxsum.double().cpu().numpy() - ds0.astype(np.float64)
        bound = (N + 8) * 2.0 ** -24 * np.abs(st).sum(0) + 2.0 ** -24 * np.abs(ds0) * 4
        assert np.all(np.abs(got - st.sum(0)) <= bound), "dxsum"


# -------------------------------------------------------------- bias gradient

@pytest.mark.parametrize("N,OC", [(37, 200), (16384, 2304), (16384, 3072), (8192, 3072), (8192, 4096)],
                         ids=["small", "qkv", "fc", "qkv350M", "fc350M"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_bias_grad(N, OC, dtype):
    rng = np.random.default_rng(4)
    dout = _t(rng.normal(0, 1, (N, OC)), dtype)
    db0 = rng.normal(0, 1, OC).astype(np.float32)
    db = torch.from_numpy(db0).cuda()
    K.bias_grad(db, dout)
    # the oracle's linear backward with a single input column: its bias
    # gradient is the column sum of dout
    d64 = _np(dout)
    _, _, rdb = ops.matmul_backward(d64, np.ones((N, 1)), np.ones((OC, 1)))
    assert_close(db.double().cpu().numpy() - db0, rdb, 1e-5, "db")


# ------------------------------------------------------------- cross-entropy

@pytest.mark.parametrize("N,V", [(37, 1000), (16384, 50257)], ids=["small", "full"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_crossentropy_fused(N, V, dtype):
    Vp = ((V + 127) // 128) * 128
    g = torch.Generator(device="cuda").manual_seed(5)
    logits = (torch.randn(N, Vp, generator=g, device="cuda") * 2.0).to(dtype)
    logits[:, V:] = 0
    tgt = torch.from_numpy(inputs.zipf_batches(6, 1, 1, N, V)[0][1].reshape(-1)).cuda()
    rows = np.sort(np.random.default_rng(7).choice(N, min(N, 64), replace=False))
    z = _np(logits[torch.from_numpy(rows).cuda()])
    losses = torch.empty(N, device="cuda")
    dloss = 1.0 / N
    err = K.crossentropy(logits, losses, tgt, V, dloss)
    probs, rloss = ops.crossentropy_forward(z, tgt.cpu().numpy()[rows], V)
    rd = ops.crossentropy_backward(probs, tgt.cpu().numpy()[rows], dloss, V)
    got_l = losses.double().cpu().numpy()[rows]
    assert np.all(np.abs(got_l - rloss) <= 1e-4 * np.abs(rloss) + 1e-5)
    got_d = _np(logits[torch.from_numpy(rows).cuda()])
    assert np.all(got_d[:, V:] == 0)
    if dtype == torch.float32:
        # the kernel's fast exp is good to a few ulp (relative 1e-5 is loose for it)
        assert np.all(np.abs(got_d - rd) <= 1e-5 * np.abs(rd) + 1e-6 * dloss)
    else:
        assert np.all(np.abs(got_d - rd) <= 2.0 ** -8 * np.abs(rd) + 1e-6 * dloss)
    assert int(err[0]) == 0


# ------------------------------------------------------------ elementwise GELU

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_gelu_forward(dtype):
    """the recompute path's GELU (odd length: vector body plus scalar tail)"""
    x = np.random.default_rng(9).normal(0, 2.5, 100003)
    xt = _t(x, dtype)
    out = torch.empty_like(xt)
    K.gelu_forward(out, xt)
    xin = _np(xt)
    ref = ops.gelu_forward(xin)
    got = _np(out)
    # fp32: a few ulp of the sigmoid-form evaluation; bf16: plus one rounding.
    # The oracle evaluates the tanh form, whose 1 + tanh(u) cancels in fp64 in
    # the far negative tail (it returns 0 below x ~ -5.7): its own absolute
    # error, about 2^-52 |x|, is part of the bar.
    rel = 4e-6 if dtype == torch.float32 else 2.0 ** -8 + 4e-6
    assert np.all(np.abs(got - ref) <= rel * np.abs(ref) + 2.0 ** -50 * np.abs(xin) + 1e-30)


# ------------------------------------------------ stochastic rounding (-w 0)

def test_stochastic_round_bf16_bit_exact():
    from oracle.pyoracle import stochastic_round_bf16 as oracle_sr
    rng = np.random.default_rng(31)
    x = (rng.normal(0, 1, 300001) * np.exp(rng.uniform(-30, 30, 300001))).astype(np.float32)
    x[:6] = [np.nan, np.inf, -np.inf, 0.0, -0.0, 3.3e38]
    xt = torch.from_numpy(x).cuda()
    out = torch.empty(x.size, dtype=torch.bfloat16, device="cuda")
    seed, k0 = 0x5352000000000001, 123456789012
    K.stochastic_round_bf16(out, xt, seed, k0)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, oracle_sr(x, seed, k0))
