"""Checkpoint/resume and update skipping on loss / gradient-norm spikes.

The pages' run saves checkpoints (-n) and resumes bit-exactly (-y 1), and skips
the update on transient instabilities (-sl 5.0 -sg 5.0) ("Karpathy reproduces
GPT-2 (1.6B) in llm.c", "Training").  Resume is checked bit for bit against
the uninterrupted run; the detector's z-scores are recomputed here from the
recorded step losses and gradient norms."""
import os

import numpy as np
import pytest

from scratch_gpt_step_train_b300 import inputs
from scratch_gpt_step_train_b300.gpt2 import BF16, FP32, GPT2, NO_MASTER, GPT2Error

pytestmark = pytest.mark.gpu
CFG = dict(L=2, H=2, C=128, V=300, T=64, B=2)  # head size 64: tensor-core attention in bf16
HP = dict(lr=1e-3, b1=0.9, b2=0.95, eps=1e-8, wd=0.1, clip=1.0)


def _batches(n, seed):
    return [inputs.uniform_batch(seed + i, CFG["B"], CFG["T"], CFG["V"]) for i in range(n)]


def _step(gm, micro, hp=HP):
    gm.zero_grad()
    for tok, tgt in micro:
        gm.forward(tok, tgt)
        gm.backward()
    return gm.adamw_step(**hp)


def _state(gm):
    m, v, t = gm.get_opt_state()
    return gm.get_params(), m, v, t


@pytest.mark.parametrize("mode", [FP32, BF16, BF16 | NO_MASTER], ids=["fp32", "bf16", "bf16-nomaster"])
def test_resume_from_checkpoint_is_bit_exact(tmp_path, mode):
    steps = [_batches(2, 100 + 10 * i) for i in range(5)]
    a = GPT2(**CFG, seed=1, mode=mode)
    a.set_spike_skip(1e9, 1e9, 2)  # detector on (never fires): its window is saved too
    path = os.fspath(tmp_path / "ckpt.bin")
    for i, micro in enumerate(steps):
        _step(a, micro)
        if i == 2:
            a.save_checkpoint(path)
    ref = _state(a)
    ref_info = a.last_step_info()
    b = GPT2(**CFG, seed=7, mode=mode)  # another init: everything comes from the file
    b.load_checkpoint(path)
    for micro in steps[3:]:
        _step(b, micro)
    got = _state(b)
    for x, y in zip(got[:3], ref[:3]):
        assert np.array_equal(x, y)
    assert got[3] == ref[3] == 5
    info = b.last_step_info()
    assert info[0] == ref_info[0] and np.float32(info[1]) == np.float32(ref_info[1])
    assert np.float32(info[2]) == np.float32(ref_info[2])


def test_checkpoint_errors(tmp_path):
    a = GPT2(**CFG, seed=1)
    path = os.fspath(tmp_path / "a.bin")
    a.save_checkpoint(path)
    other = GPT2(**dict(CFG, C=192, H=3), seed=1)
    with pytest.raises(GPT2Error) as e:
        other.load_checkpoint(path)
    assert e.value.code == -1
    bad = tmp_path / "bad.bin"
    bad.write_bytes(b"not a checkpoint" * 8)
    with pytest.raises(GPT2Error) as e:
        a.load_checkpoint(os.fspath(bad))
    assert e.value.code == -8
    trunc = tmp_path / "trunc.bin"
    trunc.write_bytes(open(path, "rb").read()[:1000])
    with pytest.raises(GPT2Error) as e:
        a.load_checkpoint(os.fspath(trunc))
    assert e.value.code == -8
    with pytest.raises(GPT2Error) as e:
        a.load_checkpoint(os.fspath(tmp_path / "missing.bin"))
    assert e.value.code == -8


def _z(hist, x):
    h = np.asarray(hist, np.float64)
    sd = h.std()
    return (x - h.mean()) / sd


def test_gradient_norm_spike_skips_the_update():
    gm = GPT2(**CFG, seed=1)
    w = 4
    gm.set_spike_skip(0.0, 5.0, w)  # gradient-norm criterion only
    norms = []
    for i in range(w + 2):
        norms.append(_step(gm, _batches(1, 300 + i)))
        skipped, zl, zg = gm.last_step_info()
        if i < w:
            assert not skipped and np.isnan(zg)
        else:
            assert zg == pytest.approx(_z(norms[-w - 1:-1], norms[-1]), rel=1e-4, abs=1e-4)
            assert skipped == (zg > 5.0)
    before = _state(gm)
    # a spike: this step's gradients scaled by 100 before the update
    gm.zero_grad()
    tok, tgt = _batches(1, 400)[0]
    gm.forward(tok, tgt)
    gm.backward()
    gm.set_grads(gm.get_grads() * 100.0)
    n = gm.adamw_step(**HP)
    skipped, zl, zg = gm.last_step_info()
    assert skipped and zg > 5.0
    assert zg == pytest.approx(_z(norms[-w:], n), rel=1e-4)
    after = _state(gm)
    for x, y in zip(after[:3], before[:3]):
        assert np.array_equal(x, y)
    assert after[3] == before[3]


def test_loss_spike_skips_the_update():
    """lr = 0 keeps the parameters fixed, so each batch's loss is known in
    advance: the window holds three ordinary batches, then the batch with the
    highest loss arrives"""
    gm = GPT2(**CFG, seed=3)
    cand = _batches(12, 500)
    losses = [gm.forward(t, y, sync_loss=True) for t, y in cand]
    order = np.argsort(losses)
    window = [cand[i] for i in order[:3]]
    spike = cand[order[-1]]
    gm.set_spike_skip(1e-3, 0.0, 3)  # loss criterion only, any rise above the window fires
    hp = dict(HP, lr=0.0)
    for micro in window:
        _step(gm, [micro], hp)
        assert not gm.last_step_info()[0]
    p0 = gm.get_params()
    t0 = gm.get_opt_state()[2]
    _step(gm, [spike], hp)
    skipped, zl, zg = gm.last_step_info()
    want = _z([losses[i] for i in order[:3]], losses[order[-1]])
    assert zl == pytest.approx(want, rel=1e-3)
    assert skipped == (want > 1e-3) and skipped
    assert np.array_equal(gm.get_params(), p0) and gm.get_opt_state()[2] == t0
