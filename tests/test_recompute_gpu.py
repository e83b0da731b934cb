"""Activation recompute ("Karpathy reproduces GPT-2 (1.6B) in llm.c",
"Parameter guide" -r 1 / -r 2): the GELU output, and then also the LayerNorm
outputs, are not kept per layer but recomputed in the backward.

fp32 mode: a recompute run is bit for bit the run without recompute (the
recomputation reruns the forward's own kernels on the same inputs).  bf16 mode:
the recompute path takes GELU from the rounded pre-activation, so it is checked
against the fp64 oracle (the bf16 loss bar) and for determinism, and it must
use less memory."""
import numpy as np
import pytest

from oracle.pyoracle import Model
from scratch_gpt_step_train_b300 import inputs
from scratch_gpt_step_train_b300.gpt2 import (BF16, FP32, GPT2, RECOMPUTE_GELU, RECOMPUTE_LN,
                                              workspace_bytes)

pytestmark = pytest.mark.gpu
CFG = dict(L=2, H=2, C=128, V=300, T=64, B=2)
HP = dict(lr=1e-3, b1=0.9, b2=0.95, eps=1e-8, wd=0.1, clip=1.0)


def _run(mode, steps=2, accum=2, seed=1):
    gm = GPT2(**CFG, seed=seed, mode=mode)
    out = []
    for s in range(steps):
        gm.zero_grad()
        for a in range(accum):
            tok, tgt = inputs.uniform_batch(700 + 10 * s + a, CFG["B"], CFG["T"], CFG["V"])
            out.append(gm.forward(tok, tgt, sync_loss=True))
            gm.backward()
        out.append(gm.get_grads())
        out.append(gm.adamw_step(**HP))
    out.append(gm.get_params())
    return out


@pytest.mark.parametrize("flag", [RECOMPUTE_GELU, RECOMPUTE_LN], ids=["gelu", "gelu+ln"])
def test_fp32_recompute_is_bit_identical(flag):
    ref = _run(FP32)
    got = _run(FP32 | flag)
    assert len(ref) == len(got)
    for a, b in zip(got, ref):
        assert np.array_equal(np.asarray(a), np.asarray(b))


def test_recompute_saves_memory():
    args = [CFG[k] for k in ("L", "H", "C", "V", "T", "B")]
    base = workspace_bytes(*args, BF16)
    gelu = workspace_bytes(*args, BF16 | RECOMPUTE_GELU)
    ln = workspace_bytes(*args, BF16 | RECOMPUTE_LN)
    BT, C, L = CFG["B"] * CFG["T"], CFG["C"], CFG["L"]
    assert base - gelu >= (L - 1) * BT * 4 * C * 2
    assert gelu - ln >= 2 * (L - 1) * BT * C * 2


@pytest.mark.parametrize("flag", [RECOMPUTE_GELU, RECOMPUTE_LN], ids=["gelu", "gelu+ln"])
def test_bf16_recompute_tracks_the_oracle_and_is_deterministic(flag):
    om = Model(**CFG, seed=1)
    runs = []
    for _ in range(2):
        gm = GPT2(**CFG, seed=1, mode=BF16 | flag)
        gm.set_params(om.params())
        stream = inputs.ZipfStream(2, CFG["B"], CFG["T"], CFG["V"], 1.1)
        losses = []
        for step in range(8):
            tok, tgt = stream.next()
            gm.zero_grad()
            losses.append(gm.forward(tok, tgt, sync_loss=True))
            gm.backward()
            gm.adamw_step(**HP)
        runs.append((losses, gm.get_params()))
    assert runs[0][0] == runs[1][0] and np.array_equal(runs[0][1], runs[1][1])
    stream = inputs.ZipfStream(2, CFG["B"], CFG["T"], CFG["V"], 1.1)
    for step in range(8):
        tok, tgt = stream.next()
        om.zero_grad()
        lo = om.forward(tok, tgt)
        om.backward()
        om.adamw_step(**HP)
        assert abs(runs[0][0][step] - lo) <= 2e-2, (step, runs[0][0][step], lo)
