"""Parameters without fp32 master weights ("Karpathy reproduces GPT-2 (1.6B)
in llm.c", "Parameter guide" -w 0): bf16 parameters, AdamW in fp32 with
stochastic rounding back to bf16 (the rule of gpt2k_stochastic_round_bf16,
stream seed ^ 0x5352000000000000, counter (t-1)*N + i)."""
import numpy as np
import pytest

from oracle.pyoracle import DECAYED, TENSOR_NAMES, Model, Ops
from scratch_gpt_step_train_b300 import inputs
from scratch_gpt_step_train_b300.gpt2 import BF16, GPT2, NO_MASTER, workspace_bytes

pytestmark = pytest.mark.gpu
CFG = dict(L=2, H=2, C=128, V=300, T=64, B=2)
HP = dict(lr=1e-3, b1=0.9, b2=0.95, eps=1e-8, wd=0.1, clip=0.0)
ops = Ops("double")


def _bf16_floor_ceil(x):
    """the two bf16 magnitudes around |x| (as float64), same sign"""
    b = np.asarray(x, np.float32).view(np.uint32)
    lo = ((b >> 16) << 16).view(np.float32).astype(np.float64)
    hi = (((b >> 16) + 1) << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    return lo, hi


def test_no_master_saves_four_bytes_per_parameter():
    args = [CFG[k] for k in ("L", "H", "C", "V", "T", "B")]
    gm = GPT2(**CFG, seed=1, mode=BF16 | NO_MASTER)
    saved = workspace_bytes(*args, BF16) - workspace_bytes(*args, BF16 | NO_MASTER)
    assert 4 * gm.n <= saved <= 4 * gm.n + 256


def test_no_master_adamw_step_against_the_oracle():
    gm = GPT2(**CFG, seed=1, mode=BF16 | NO_MASTER)
    om = Model(**CFG, seed=1)  # only for the tensor layout
    sl = om.tensor_slices()
    tok, tgt = inputs.uniform_batch(41, CFG["B"], CFG["T"], CFG["V"])
    w0 = gm.get_params().astype(np.float64)
    # parameters are bf16 values
    assert np.array_equal(w0.astype(np.float32).view(np.uint32) & 0xFFFF, np.zeros(w0.size, np.uint32))
    for step in range(2):
        gm.zero_grad()
        gm.forward(tok, tgt)
        gm.backward()
        g = gm.get_grads().astype(np.float64)
        m0, v0, t0 = gm.get_opt_state()
        w0 = gm.get_params().astype(np.float64)
        gm.adamw_step(**HP)
        w1 = gm.get_params().astype(np.float64)
        m1, v1, t1 = gm.get_opt_state()
        assert t1 == t0 + 1
        ref_w, ref_m, ref_v = np.empty_like(w0), np.empty_like(w0), np.empty_like(w0)
        for name in TENSOR_NAMES:
            s = sl[name]
            ref_w[s], ref_m[s], ref_v[s] = ops.adamw(
                w0[s], m0[s], v0[s], g[s], 1.0, HP["lr"], HP["b1"], HP["b2"], HP["eps"],
                HP["wd"], name in DECAYED, t1)
        # moments: fp32 evaluation of the same update (m = b1 m0 + (1-b1) g can
        # cancel: its rounding error is relative to the terms)
        assert np.all(np.abs(m1 - ref_m) <= 1e-6 * (np.abs(m0) + np.abs(g)) + 1e-30)
        assert np.all(np.abs(v1 - ref_v) <= 1e-5 * np.abs(ref_v) + 1e-18)
        # parameters: one of the two bf16 neighbours of the exact update (with
        # the fp32 evaluation's slack at the grid points)
        lo, hi = _bf16_floor_ceil(ref_w * (1 - 1e-6 * np.sign(ref_w)))
        lo2, hi2 = _bf16_floor_ceil(ref_w * (1 + 1e-6 * np.sign(ref_w)))
        ok = (w1 == lo) | (w1 == hi) | (w1 == lo2) | (w1 == hi2)
        assert np.all(ok), np.flatnonzero(~ok)[:10]
        # unbiased: among moved parameters, rounding up happens as often as
        # the exact values' mean position inside their bf16 interval predicts
        lo, hi = _bf16_floor_ceil(ref_w)
        f = np.where(hi != lo, (np.abs(ref_w) - np.abs(lo)) / np.abs(hi - lo), 0.0)
        moving = (f > 1e-3) & (f < 1 - 1e-3)
        up = np.mean(w1[moving] == hi[moving])
        n = moving.sum()
        assert n > 1000
        assert abs(up - f[moving].mean()) < 5 * np.sqrt(0.25 / n)


def test_no_master_training_is_deterministic_and_tracks_the_oracle():
    om = Model(**CFG, seed=1)
    runs = []
    for _ in range(2):
        gm = GPT2(**CFG, seed=1, mode=BF16 | NO_MASTER)
        gm.set_params(om.params())
        stream = inputs.ZipfStream(2, CFG["B"], CFG["T"], CFG["V"], 1.1)
        losses = []
        for step in range(8):
            tok, tgt = stream.next()
            gm.zero_grad()
            losses.append(gm.forward(tok, tgt, sync_loss=True))
            gm.backward()
            gm.adamw_step(**dict(HP, clip=1.0))
        runs.append((losses, gm.get_params()))
    assert runs[0][0] == runs[1][0] and np.array_equal(runs[0][1], runs[1][1])
    stream = inputs.ZipfStream(2, CFG["B"], CFG["T"], CFG["V"], 1.1)
    for step in range(8):
        tok, tgt = stream.next()
        om.zero_grad()
        lo = om.forward(tok, tgt)
        om.backward()
        om.adamw_step(**dict(HP, clip=1.0))
        assert abs(runs[0][0][step] - lo) <= 2e-2, (step, runs[0][0][step], lo)
