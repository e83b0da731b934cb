"""Parity of causal attention (forward and backward) against the oracle's
attention (fp64) on the same bf16-rounded qkv.

bf16 path (tensor cores, head size 64): the probabilities P pass through bf16
before the P.V product and the output is rounded to bf16, so the forward's
per-element bound is 2^-8 (sum_j a_ij |v_j|) + 2^-8 |o_i| (a = the exact
attention weights); the backward's per-element bound is derived the same way
in _bwd_bound.  fp32 path: rel 1e-4 (see tests/parity.py)."""
import numpy as np
import pytest
import torch

from oracle.pyoracle import Ops
from scratch_gpt_step_train_b300 import kernels as K
from parity import assert_close

pytestmark = pytest.mark.gpu
ops = Ops("double")


def _qkv(B, T, C, seed, qscale=1.0, dtype=torch.bfloat16):
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 1, (B, T, 3 * C))
    x[..., :C] *= qscale
    t = torch.from_numpy(x.astype(np.float32)).to(dtype).cuda()
    return t, t.double().cpu().numpy()


def _fwd(qkv, B, T, C, H):
    out = torch.empty(B, T, C, dtype=qkv.dtype, device="cuda")
    lse = torch.empty(B, H, T, dtype=torch.float32, device="cuda")
    K.attention_forward(out, lse, qkv, B, T, C, H)
    torch.cuda.synchronize()
    return out, lse


def _lse_ref(q64, att, C, H):
    """lse_t = s_tt - log(a_tt): the diagonal score is always in the softmax"""
    B, T, _ = q64.shape
    hd = C // H
    out = np.zeros((B, H, T))
    for h in range(H):
        q = q64[..., h * hd:(h + 1) * hd]
        k = q64[..., C + h * hd:C + (h + 1) * hd]
        s = (q * k).sum(-1) / np.sqrt(hd)
        d = np.diagonal(att[:, h], axis1=1, axis2=2)
        out[:, h] = s - np.log(d)
    return out


SHAPES = [(2, 200, 192, 3), (1, 128, 64, 1), (3, 37, 128, 2), (1, 300, 64, 1)]


@pytest.mark.parametrize("B,T,C,H", SHAPES, ids=["ragged", "one-tile", "short", "three-tiles"])
@pytest.mark.parametrize("qscale", [1.0, 4.0], ids=["mild", "peaky"])
def test_attention_forward_bf16(B, T, C, H, qscale):
    qkv, q64 = _qkv(B, T, C, 1, qscale)
    out, lse = _fwd(qkv, B, T, C, H)
    ref, att = ops.attention_forward(q64, H)
    a = q64.copy()
    a[..., 2 * C:] = np.abs(a[..., 2 * C:])
    refabs, _ = ops.attention_forward(a, H)
    got = out.double().cpu().numpy()
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * (refabs + np.abs(ref)) + 1e-7)
    assert np.abs(lse.double().cpu().numpy() - _lse_ref(q64, att, C, H)).max() < 2e-4


@pytest.mark.parametrize("B,T,C,H", SHAPES[:3], ids=["ragged", "one-tile", "short"])
def test_attention_forward_fp32(B, T, C, H):
    qkv, q64 = _qkv(B, T, C, 2, 1.0, torch.float32)
    out, lse = _fwd(qkv, B, T, C, H)
    ref, att = ops.attention_forward(q64, H)
    assert_close(out.double().cpu().numpy(), ref, 1e-4, "out")
    assert np.abs(lse.double().cpu().numpy() - _lse_ref(q64, att, C, H)).max() < 1e-4


# GPT-2 widths at the micro-batch each is trained with: (C, H, B), T = 1024
FULL_WIDTHS = [(768, 12, 16), (1600, 25, 16), (1024, 16, 8)]
FULL_IDS = ["124M", "1558M", "350M"]


@pytest.mark.parametrize("C,H,B", FULL_WIDTHS, ids=FULL_IDS)
def test_attention_forward_full_size_sampled(C, H, B):
    """GPT-2 124M, 350M and 1558M widths at their micro-batches x 1024: the
    oracle recomputes one sequence (every head)"""
    T = 1024
    qkv, _ = _qkv(B, T, C, 3)
    out, lse = _fwd(qkv, B, T, C, H)
    b = 9 % B
    q64 = qkv[b:b + 1].double().cpu().numpy()
    ref, att = ops.attention_forward(q64, H)
    a = q64.copy()
    a[..., 2 * C:] = np.abs(a[..., 2 * C:])
    refabs, _ = ops.attention_forward(a, H)
    got = out[b:b + 1].double().cpu().numpy()
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * (refabs + np.abs(ref)) + 1e-7)
    assert np.abs(lse[b:b + 1].double().cpu().numpy() - _lse_ref(q64, att, C, H)).max() < 2e-4


def _bwd(qkv, dout, out, lse, B, T, C, H):
    dqkv = torch.full_like(qkv, float("nan"))
    K.attention_backward(dqkv, dout, qkv, out, lse, B, T, C, H)
    torch.cuda.synchronize()
    return dqkv


U = 2.0 ** -8  # unit roundoff of bf16 (8-bit significand, round to nearest even)


def _bwd_bound(q64, dout64, att, C, H):
    """Per-element bound on |GPU - oracle| of the bf16 backward, derived from
    its arithmetic (exact attention weights a, exact dP = dO V^T, D = dO.o,
    dS = a (dP - D)):
      * O from the forward carries its bound eO = u (a|V| + |o|), so
        D = dO.O is off by dD = |dO|.eO;
      * P = exp(S - lse) in fp32 (relative error eps_p, covering the forward's
        log-sum-exp), rounded to bf16 for P^T dO (u);
      * dS = P (dP - D) carries a dD + (eps_p + 2u)|dS| (P's and dS's own
        roundings) before dQ = dS K / sqrt(hd) and dK = dS^T Q / sqrt(hd);
      * fp32 accumulation over at most T terms (T 2^-24 of the |.| products),
        and every output rounded to bf16 (u |ref|)."""
    B, T, _ = q64.shape
    hd = C // H
    sc = 1.0 / np.sqrt(hd)
    eps_p = 2.0 ** -12
    acc = T * 2.0 ** -24
    bound = np.zeros((B, T, 3 * C))
    for b in range(B):
        for h in range(H):
            cs = slice(h * hd, (h + 1) * hd)
            q, k, v = (q64[b, :, off + h * hd:off + (h + 1) * hd] for off in (0, C, 2 * C))
            do = dout64[b, :, cs]
            a = att[b, h]
            o = a @ v
            e_o = U * (a @ np.abs(v) + np.abs(o))
            d_d = (np.abs(do) * e_o).sum(-1)
            dp = do @ v.T
            ds = a * (dp - (a * dp).sum(-1, keepdims=True))
            e_ds = a * (d_d[:, None] + hd * 2.0 ** -24 * (np.abs(do) @ np.abs(v).T)) + \
                (eps_p + 2 * U) * np.abs(ds)
            dq, dk, dv = sc * ds @ k, sc * ds.T @ q, a.T @ do
            bound[b, :, cs] = sc * (e_ds @ np.abs(k)) + acc * sc * (np.abs(ds) @ np.abs(k)) + \
                U * np.abs(dq)
            bound[b, :, C + h * hd:C + (h + 1) * hd] = sc * (e_ds.T @ np.abs(q)) + \
                acc * sc * (np.abs(ds).T @ np.abs(q)) + U * np.abs(dk)
            bound[b, :, 2 * C + h * hd:2 * C + (h + 1) * hd] = \
                (U + eps_p + acc) * (a.T @ np.abs(do)) + U * np.abs(dv)
    return bound + 1e-7


def _check_bwd_bf16(got, ref, q64, dout64, att, C, H, what):
    """every element of dQ, dK, dV within the bound derived above"""
    bnd = _bwd_bound(q64, dout64, att, C, H)
    r = np.abs(got - ref) / bnd
    worst = np.unravel_index(np.argmax(r), r.shape)
    assert r.max() <= 1.0, (what, "worst at (b, t, column)", worst, r.max())


@pytest.mark.parametrize("B,T,C,H", SHAPES, ids=["ragged", "one-tile", "short", "three-tiles"])
def test_attention_backward_bf16(B, T, C, H):
    qkv, q64 = _qkv(B, T, C, 4, 2.0)
    out, lse = _fwd(qkv, B, T, C, H)
    dout = torch.from_numpy(np.random.default_rng(5).normal(0, 1, (B, T, C)).astype(np.float32))
    dout = dout.to(torch.bfloat16).cuda()
    dqkv = _bwd(qkv, dout, out, lse, B, T, C, H)
    _, att = ops.attention_forward(q64, H)
    ref = ops.attention_backward(dout.double().cpu().numpy(), q64, att, H)
    got = dqkv.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    _check_bwd_bf16(got, ref, q64, dout.double().cpu().numpy(), att, C, H, (B, T, C, H))


@pytest.mark.parametrize("B,T,C,H", SHAPES[:3], ids=["ragged", "one-tile", "short"])
def test_attention_backward_fp32(B, T, C, H):
    qkv, q64 = _qkv(B, T, C, 6, 1.0, torch.float32)
    out, lse = _fwd(qkv, B, T, C, H)
    dout = torch.from_numpy(np.random.default_rng(7).normal(0, 1, (B, T, C)).astype(np.float32)).cuda()
    dqkv = _bwd(qkv, dout, out, lse, B, T, C, H)
    _, att = ops.attention_forward(q64, H)
    ref = ops.attention_backward(dout.double().cpu().numpy(), q64, att, H)
    assert_close(dqkv.double().cpu().numpy(), ref, 1e-4, "dqkv")


@pytest.mark.parametrize("C,H,B", FULL_WIDTHS, ids=FULL_IDS)
def test_attention_backward_full_size_sampled(C, H, B):
    """the 124M, 350M and 1558M widths at their micro-batches x 1024; the
    oracle recomputes one sequence (every head), each element against the
    bound"""
    T = 1024
    qkv, _ = _qkv(B, T, C, 8)
    out, lse = _fwd(qkv, B, T, C, H)
    dout = (torch.randn(B, T, C, generator=torch.Generator(device="cuda").manual_seed(9),
                        device="cuda")).to(torch.bfloat16)
    dqkv = _bwd(qkv, dout, out, lse, B, T, C, H)
    b = 13 % B
    q64 = qkv[b:b + 1].double().cpu().numpy()
    d64 = dout[b:b + 1].double().cpu().numpy()
    _, att = ops.attention_forward(q64, H)
    ref = ops.attention_backward(d64, q64, att, H)
    _check_bwd_bf16(dqkv[b:b + 1].double().cpu().numpy(), ref, q64, d64, att, C, H, "full")


def test_attention_backward_deterministic():
    B, T, C, H = 2, 300, 128, 2
    qkv, _ = _qkv(B, T, C, 10)
    out, lse = _fwd(qkv, B, T, C, H)
    dout = torch.randn(B, T, C, device="cuda").to(torch.bfloat16)
    a = _bwd(qkv, dout, out, lse, B, T, C, H)
    b = _bwd(qkv, dout, out, lse, B, T, C, H)
    assert torch.equal(a, b)
