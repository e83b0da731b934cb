"""Whole-step parity of GPT-2 124M at micro-batch 4 x 1024 against the fp64
oracle, through the C-ABI.

Workload: L=12, H=12, C=768, V=50257 (padded to 50304), T=1024, B=4; weights
from seed 1; tokens i.i.d. Zipf(1.1) from seed 2, the stream continuing from
step to step, targets = next token; AdamW lr 6e-4, b1 0.9, b2 0.95, eps 1e-8,
wd 0.1, clip 1.0; one micro-batch per step.

Expected values were written by oracle/make_golden_124M.py (it calls only the
oracle and the token generator): tests/golden/gpt2_124M_B4T1024.npz holds the
fp64 oracle's 20 steps, gpt2_124M_B4T1024_f32.npz the fp32 build's first 10.

fp32 mode, 10 steps (rel 1e-4 read per tensor as ||d||_2 <= 1e-4 ||ref||_2
and max|d| <= 1e-4 max|ref|):
  * the loss and the gradient norm each update sees, at every step (from the
    second step under the bar below);
  * at step 1 (both sides hold the same weights): sampled logits, every
    element of the small gradient tensors and 8192 sampled elements of each
    large one, and every tensor's L2 norm and max |.|;
  * at step 10 the same quantities against max(1e-4, 4 x the fp32 oracle's
    error at step 10): after the first update two fp32 evaluations hold
    different weights (AdamW's first step moves every weight by lr in the
    direction of its gradient's sign however small the gradient, so one whose
    gradient is rounding noise moves by lr either way), and the fp32 oracle
    measures how far a plain fp32 evaluation of the definition drifts.
bf16 mode, 20 steps: |loss - oracle loss| <= 2e-2 at every step.
"""
import os

import numpy as np
import pytest

from oracle.pyoracle import TENSOR_NAMES
from scratch_gpt_step_train_b300 import inputs
from scratch_gpt_step_train_b300.gpt2 import BF16, FP32, GPT2

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
G64 = os.path.join(HERE, "golden", "gpt2_124M_B4T1024.npz")
G32 = os.path.join(HERE, "golden", "gpt2_124M_B4T1024_f32.npz")
CFG = dict(L=12, H=12, C=768, V=50257, T=1024, B=4)
HP = dict(lr=6e-4, b1=0.9, b2=0.95, eps=1e-8, wd=0.1, clip=1.0)


def _load(p):
    d = np.load(p)
    return {k: d[k] for k in d.files}


def _offsets(gm):
    """canonical offsets of the 16 tensors (the order the library and the
    oracle both document)"""
    L, C, T, Vp = CFG["L"], CFG["C"], CFG["T"], gm.Vp
    sizes = [Vp * C, T * C, L * C, L * C, L * 3 * C * C, L * 3 * C, L * C * C, L * C, L * C,
             L * C, L * 4 * C * C, L * 4 * C, L * C * 4 * C, L * C, C, C]
    off = np.concatenate([[0], np.cumsum(sizes)])
    return {k: slice(int(off[i]), int(off[i + 1])) for i, k in enumerate(TENSOR_NAMES)}


def _err(got, ref, ref_max):
    """(||d||_2 / ||ref||_2, max|d| / max|ref|) with max|ref| over the whole
    tensor when only a sample is compared"""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    d = got - ref
    nr = np.linalg.norm(ref)
    return (np.linalg.norm(d) / nr if nr > 0 else np.linalg.norm(d),
            np.abs(d).max() / ref_max if ref_max > 0 else np.abs(d).max())


def _bar(e32, tol=1e-4, factor=4.0):
    return max(tol, factor * max(e32)) if e32 is not None else tol


def _golden(p, how):
    if not os.path.exists(p):
        pytest.fail(f"stored oracle values missing: run oracle/make_golden_124M.py {how}")
    return _load(p)


@pytest.fixture(scope="module")
def g64():
    return _golden(G64, "")


@pytest.fixture(scope="module")
def g32():
    return _golden(G32, "--real float")


def test_fp32_124M_ten_steps(g64, g32):
    gm = GPT2(**CFG, seed=1, mode=FP32)
    sl = _offsets(gm)
    stream = inputs.ZipfStream(2, CFG["B"], CFG["T"], CFG["V"])
    BT = CFG["B"] * CFG["T"]
    for s in range(1, 11):
        tok, tgt = stream.next()
        assert int(tok.astype(np.int64).sum()) == int(g64["tok_sum"][s - 1])
        if s in (1, 10):
            gm.forward(tok, None)
            lg = gm.get_logits().reshape(BT, CFG["V"])[g64["lrow"]][:, g64["lcol"]]
            ref = g64[f"logit{s}"]
            e32 = None if s == 1 else _err(g32[f"logit{s}"], ref, g64[f"lmax{s}"].max())
            e = _err(lg, ref, g64[f"lmax{s}"].max())
            assert max(e) <= _bar(e32), (s, "logits", e, e32)
        gm.zero_grad()
        loss = gm.forward(tok, tgt, sync_loss=True)
        lo = g64["loss"][s - 1]
        e32 = None if s == 1 else (abs(g32["loss"][s - 1] - lo) / abs(lo),)
        assert abs(loss - lo) <= _bar(e32) * abs(lo), (s, loss, lo, e32)
        gm.backward()
        g = gm.get_grads()
        for j, k in enumerate(TENSOR_NAMES):
            gk = g[sl[k]].astype(np.float64)
            tn = (np.linalg.norm(gk), np.abs(gk).max())
            rn = (g64["gnorm"][s - 1, j], g64["gmax"][s - 1, j])
            e32 = None
            if s > 1:
                fn = (g32["gnorm"][s - 1, j], g32["gmax"][s - 1, j])
                e32 = tuple(abs(a - b) / b for a, b in zip(fn, rn))
            for a, b, what in zip(tn, rn, ("norm", "max")):
                assert abs(a - b) <= _bar(e32) * b, (s, k, what, a, b, e32)
            if s in (1, 10):
                idx = g64["idx_" + k]
                ref = g64[f"grad{s}_{k}"]
                e = _err(gk[idx], ref, g64["gmax"][s - 1, j])
                e32 = None if s == 1 else _err(g32[f"grad{s}_{k}"], ref, g64["gmax"][s - 1, j])
                assert max(e) <= _bar(e32), (s, k, e, e32)
        norm = gm.adamw_step(**HP)
        no = g64["norm"][s - 1]
        e32 = None if s == 1 else (abs(g32["norm"][s - 1] - no) / no,)
        assert abs(norm - no) <= _bar(e32) * no, (s, norm, no, e32)


def test_bf16_124M_twenty_steps(g64):
    gm = GPT2(**CFG, seed=1, mode=BF16)
    stream = inputs.ZipfStream(2, CFG["B"], CFG["T"], CFG["V"])
    worst = 0.0
    for s in range(1, 21):
        tok, tgt = stream.next()
        gm.zero_grad()
        loss = gm.forward(tok, tgt, sync_loss=True)
        gm.backward()
        gm.adamw_step(**HP)
        d = abs(loss - g64["loss"][s - 1])
        worst = max(worst, d)
        assert d <= 2e-2, (s, loss, g64["loss"][s - 1])
    assert np.isfinite(worst)
