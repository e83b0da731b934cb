"""GPU parity of the whole training step, through the C-ABI, against the CPU
oracle (fp64 build) on the same seeded inputs.

fp32 mode: loss, logits, per-position losses and every gradient tensor within
rel 1e-4 (see tests/parity.py for the reading of "rel"); AdamW updates checked
step by step with the oracle's state injected before each step.  bf16 mode:
|loss difference| <= 2e-2 at every one of the first 20 steps.
"""
import numpy as np
import pytest

from oracle.pyoracle import Model
from scratch_gpt_step_train_b300 import inputs
from scratch_gpt_step_train_b300.gpt2 import BF16, FP32, GPT2, GPT2Error
from parity import assert_close, compare_tensors, key_bias_mask, rel_err

pytestmark = pytest.mark.gpu

TOY = dict(L=2, H=2, C=16, V=2, T=3)
TINY = dict(L=2, H=2, C=32, V=64, T=8, B=2)
# head size 64 as in every GPT-2 size; ragged against 64/128-row tiles
MID = dict(L=2, H=3, C=192, V=1000, T=97, B=3)


def _perturbed_params(om, seed):
    """oracle init + noise on every tensor (no degenerate biases / gains);
    padded vocabulary rows stay 0"""
    rng = np.random.default_rng(seed)
    p = om.params()
    for name, s in om.tensor_slices().items():
        p[s] += rng.normal(0, 0.05 if name.startswith("ln") else 0.02, s.stop - s.start)
    sl = om.tensor_slices()["wte"]
    wte = p[sl].reshape(om.Vp, om.C)
    wte[om.V:] = 0
    p[sl] = wte.reshape(-1)
    p = p.astype(np.float32).astype(np.float64)
    om.set_params(p)
    return p


def _pair(cfg, mode=FP32, seed=0, perturb=None):
    om = Model(**cfg, seed=seed)
    gm = GPT2(**cfg, seed=seed, mode=mode)
    if perturb is not None:
        p = _perturbed_params(om, perturb)
        gm.set_params(p)
    return om, gm


def test_init_matches_oracle():
    cfg = dict(L=2, H=3, C=192, V=1000, T=97, B=1)
    om = Model(**cfg, seed=1234)
    gm = GPT2(**cfg, seed=1234)
    ref = om.params().astype(np.float32)
    got = gm.get_params()
    # same counter-based draws; the two sides' double log/cos may differ in the
    # last bit of a double, which can move the fp32 rounding by one ulp
    ulp = np.spacing(np.abs(ref)).astype(np.float32)
    assert np.all(np.abs(got - ref) <= ulp)
    assert np.mean(got == ref) > 0.999


@pytest.mark.parametrize("cfg", [TINY, MID, dict(TOY, B=12)], ids=["tiny", "mid", "toy"])
def test_fp32_forward_backward(cfg):
    om, gm = _pair(cfg, FP32, seed=3, perturb=5)
    tok, tgt = inputs.uniform_batch(7, cfg["B"], cfg["T"], cfg["V"])
    # logits (forward without targets)
    om.forward(tok, None)
    gm.forward(tok.copy(), None)
    assert_close(gm.get_logits(), om.logits(), 1e-4, "logits")
    # loss, per-position losses, gradients
    ref_loss = om.forward(tok, tgt)
    om.zero_grad()
    om.backward()
    gm.zero_grad()
    loss = gm.forward(tok, tgt, sync_loss=True)
    assert abs(loss - ref_loss) <= 1e-4 * abs(ref_loss)
    assert_close(gm.get_losses(), om.losses(), 1e-4, "losses")
    gm.backward()
    compare_tensors(gm.get_grads(), om.grads(), om, 1e-4, "grad")


def _stepwise(cfg, n_steps, n_accum, hp, mode=FP32, tol=1e-4, perturb=9):
    """Each step: inject the oracle's params and AdamW state into the GPU, run
    n_accum micro-batches + one AdamW step on both sides, compare."""
    om, gm = _pair(cfg, mode, seed=2, perturb=perturb)
    keep = key_bias_mask(om)
    stream = inputs.ZipfStream(11, cfg["B"], cfg["T"], cfg["V"], 1.1)
    norms = []
    for step in range(n_steps):
        p0 = om.params()
        gm.set_params(p0)
        gm.set_opt_state(om.m(), om.v(), om.step_count())
        om.zero_grad()
        gm.zero_grad()
        for _ in range(n_accum):
            tok, tgt = stream.next()
            lo = om.forward(tok, tgt)
            om.backward()
            lg = gm.forward(tok, tgt, sync_loss=True)
            assert abs(lg - lo) <= tol * abs(lo), (step, lg, lo)
            gm.backward()
        compare_tensors(gm.get_grads(), om.grads(), om, tol, f"step {step} grad")
        rc, no = om.adamw_step(**hp)
        ng = gm.adamw_step(**hp)
        assert rc == 0
        assert abs(ng - no) <= tol * no
        norms.append(no)
        got = gm.get_params()
        ref = om.params()
        assert_close(got[keep], ref[keep], tol, f"step {step} params")
        m, v, t = gm.get_opt_state()
        assert t == om.step_count()
        assert_close(m[keep], om.m()[keep], tol, f"step {step} m")
        assert_close(v[keep], om.v()[keep], tol, f"step {step} v")
    return norms


def test_fp32_toy_50_adamw_steps_stepwise():
    """the toy binary GPT, lr 1e-2, wd 0, torch-default betas/eps, no clip"""
    cfg = dict(TOY, B=12)
    om, gm = _pair(cfg, FP32, seed=0)
    o32 = Model(**cfg, seed=0, real="float")
    keep = key_bias_mask(om)
    tok, tgt = inputs.toy_windows(0)
    hp = dict(lr=1e-2, b1=0.9, b2=0.999, eps=1e-8, wd=0.0, clip=0.0)
    for step in range(50):
        gm.set_params(om.params())
        gm.set_opt_state(om.m(), om.v(), om.step_count())
        o32.set_params(om.params())
        om.zero_grad()
        gm.zero_grad()
        o32.zero_grad()
        lo = om.forward(tok, tgt)
        om.backward()
        o32.forward(tok, tgt)
        o32.backward()
        lg = gm.forward(tok, tgt, sync_loss=True)
        gm.backward()
        assert abs(lg - lo) <= 1e-4 * abs(lo)
        compare_tensors(gm.get_grads(), om.grads(), om, 1e-4, f"step {step} grad",
                        f32_vec=o32.grads(), widen=("lnfb",))
        om.adamw_step(**hp)
        gm.adamw_step(**hp)
        assert_close(gm.get_params()[keep], om.params()[keep], 1e-4, f"step {step} params")


def _table(model_params, gpu=True):
    """P(next = 1 | state) for the 8 states of the toy at the last position"""
    states = inputs.toy_states()
    if gpu:
        gm = GPT2(**TOY, B=8, seed=0)
        gm.set_params(model_params)
        gm.forward(states, None)
        z = gm.get_logits()[:, -1, :]
    else:
        om = Model(**TOY, B=8, seed=0)
        om.set_params(model_params)
        om.forward(states, None)
        z = om.logits()[:, -1, :]
    z = z.astype(np.float64)
    return 1 / (1 + np.exp(z[:, 0] - z[:, 1]))


def test_toy_transition_table_gpu():
    cfg = dict(TOY, B=12)
    gm = GPT2(**cfg, seed=0)
    om = Model(**cfg, seed=0)
    p0 = gm.get_params()
    a0 = _table(p0, gpu=True)
    assert np.abs(a0 - _table(p0.astype(np.float64), gpu=False)).max() < 1e-5
    assert np.all(np.abs(a0 - 0.5) < 0.1)
    tok, tgt = inputs.toy_windows(0)
    losses = []
    for _ in range(50):
        gm.zero_grad()
        losses.append(gm.forward(tok, tgt, sync_loss=True))
        gm.backward()
        gm.adamw_step(1e-2, 0.9, 0.999, 1e-8, 0.0, 0.0)
    p50 = gm.get_params()
    a50 = _table(p50, gpu=True)
    assert np.abs(a50 - _table(p50.astype(np.float64), gpu=False)).max() < 1e-5
    assert losses[-1] < losses[0] - 0.05
    # arrows move toward the empirical next-bit frequency of the seen states
    states = [int("".join(map(str, r)), 2) for r in tok]
    for s in range(8):
        nxt = [tgt[i, -1] for i in range(len(states)) if states[i] == s]
        if nxt and abs(np.mean(nxt) - 0.5) >= 0.3:
            f = float(np.mean(nxt))
            assert abs(a50[s] - f) < abs(a0[s] - f) - 0.1


# the GPT-2 1558M layer width (C=1600, 25 heads of 64, 4C=6400) and the 350M
# one (C=1024, 16 heads), the full vocabulary, two layers, one sequence of 128
# tokens
WIDTHS = {"1558M": dict(L=2, H=25, C=1600, V=50257, T=128, B=1),
          "350M": dict(L=2, H=16, C=1024, V=50257, T=128, B=1)}
WIDE_HP = dict(lr=6e-4, b1=0.9, b2=0.95, eps=1e-8, wd=0.1, clip=1.0)


@pytest.mark.parametrize("width", sorted(WIDTHS))
def test_fp32_wide_two_steps(width):
    """fp32 mode against the fp64 oracle from the same init and Zipf tokens,
    two AdamW steps: logits, loss and the norm each update saw at rel 1e-4;
    every gradient tensor at rel 1e-4 at the first step.  From the second
    step the weights of any two fp32 evaluations differ (AdamW's first step
    moves every weight by lr in the direction of its gradient's sign, however
    small the gradient, so a gradient that is rounding noise moves its weight
    by lr either way), and each gradient tensor is held to
    max(1e-4, 4 x the error of the fp32 build of the oracle run alongside)."""
    WIDE = WIDTHS[width]
    om = Model(**WIDE, seed=1)
    o32 = Model(**WIDE, seed=1, real="float")
    gm = GPT2(**WIDE, seed=1, mode=FP32)
    gm.set_params(om.params())
    o32.set_params(om.params())
    stream = inputs.ZipfStream(2, WIDE["B"], WIDE["T"], WIDE["V"])
    for step in range(2):
        tok, tgt = stream.next()
        om.forward(tok, None)
        gm.forward(tok, None)
        assert_close(gm.get_logits(), om.logits(), 1e-4, f"step {step} logits")
        for m in (om, o32):
            m.zero_grad()
        lo = om.forward(tok, tgt)
        om.backward()
        o32.forward(tok, tgt)
        o32.backward()
        gm.zero_grad()
        lg = gm.forward(tok, tgt, sync_loss=True)
        assert abs(lg - lo) <= 1e-4 * abs(lo), (step, lg, lo)
        gm.backward()
        widen = () if step == 0 else tuple(om.tensor_slices())
        compare_tensors(gm.get_grads(), om.grads(), om, 1e-4, f"step {step} grad",
                        f32_vec=o32.grads(), widen=widen)
        rc, no = om.adamw_step(**WIDE_HP)
        o32.adamw_step(**WIDE_HP)
        ng = gm.adamw_step(**WIDE_HP)
        assert rc == 0 and abs(ng - no) <= 1e-4 * no, (step, ng, no)


@pytest.mark.parametrize("width", sorted(WIDTHS))
def test_bf16_wide_two_steps(width):
    """bf16-mixed mode at the same shapes: |loss difference| <= 2e-2 per step"""
    WIDE = WIDTHS[width]
    om = Model(**WIDE, seed=1)
    gm = GPT2(**WIDE, seed=1, mode=BF16)
    gm.set_params(om.params())
    stream = inputs.ZipfStream(2, WIDE["B"], WIDE["T"], WIDE["V"])
    for step in range(2):
        tok, tgt = stream.next()
        om.zero_grad()
        lo = om.forward(tok, tgt)
        om.backward()
        om.adamw_step(**WIDE_HP)
        gm.zero_grad()
        lg = gm.forward(tok, tgt, sync_loss=True)
        gm.backward()
        gm.adamw_step(**WIDE_HP)
        assert abs(lg - lo) <= 2e-2, (step, lg, lo)


def test_fp32_accum_clip_decay_stepwise():
    """two micro-batches per step, clip active, weight decay on 2-D weights"""
    hp = dict(lr=3e-3, b1=0.9, b2=0.95, eps=1e-8, wd=0.1, clip=0.05)
    norms = _stepwise(MID, 3, 2, hp)
    assert all(n > 0.05 for n in norms)  # the clip was active


def test_bf16_loss_trajectory_20_steps():
    """bf16-mixed vs the fp64 oracle from the same init and tokens"""
    cfg = dict(L=2, H=3, C=192, V=1000, T=64, B=4)
    om = Model(**cfg, seed=1)
    gm = GPT2(**cfg, seed=1, mode=BF16)
    gm.set_params(om.params())
    stream = inputs.ZipfStream(2, cfg["B"], cfg["T"], cfg["V"], 1.1)
    hp = dict(lr=1e-3, b1=0.9, b2=0.95, eps=1e-8, wd=0.1, clip=1.0)
    worst = 0.0
    for step in range(20):
        tok, tgt = stream.next()
        om.zero_grad()
        lo = om.forward(tok, tgt)
        om.backward()
        om.adamw_step(**hp)
        gm.zero_grad()
        lg = gm.forward(tok, tgt, sync_loss=True)
        gm.backward()
        gm.adamw_step(**hp)
        worst = max(worst, abs(lg - lo))
        assert abs(lg - lo) <= 2e-2, (step, lg, lo)
    assert np.isfinite(worst)


@pytest.mark.parametrize("mode", [FP32, BF16], ids=["fp32", "bf16"])
def test_bitwise_determinism(mode):
    cfg = MID
    tok, tgt = inputs.zipf_batches(4, 1, cfg["B"], cfg["T"], cfg["V"])[0]
    out = []
    for _ in range(2):
        gm = GPT2(**cfg, seed=5, mode=mode)
        for _ in range(2):
            gm.zero_grad()
            gm.forward(tok, tgt)
            gm.backward()
            gm.forward(tok, tgt)
            gm.backward()
            gm.adamw_step(1e-3)
        gm.forward(tok, tgt)
        gm.backward()
        out.append((gm.get_params(), gm.get_grads(), gm.get_loss()))
    assert np.array_equal(out[0][0], out[1][0])
    assert np.array_equal(out[0][1], out[1][1])
    assert out[0][2] == out[1][2]


def test_host_and_device_token_paths_agree():
    import torch
    cfg = TINY
    tok, tgt = inputs.uniform_batch(3, cfg["B"], cfg["T"], cfg["V"])
    gm = GPT2(**cfg, seed=1)
    l_host = gm.forward(tok, tgt, sync_loss=True)
    l_dev = gm.forward(torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda(), sync_loss=True)
    assert l_host == l_dev


def test_errors_are_reported():
    cfg = TINY
    gm = GPT2(**cfg, seed=1)
    tok, tgt = inputs.uniform_batch(3, cfg["B"], cfg["T"], cfg["V"])
    with pytest.raises(GPT2Error) as e:
        gm.backward()
    assert e.value.code == -4
    bad = tok.copy()
    bad[1, 3] = cfg["V"]  # out of range
    with pytest.raises(GPT2Error) as e:
        gm.forward(bad, tgt, sync_loss=True)
    assert e.value.code == -5
    badt = tgt.copy()
    badt[0, 0] = -1
    with pytest.raises(GPT2Error) as e:
        gm.forward(tok, badt, sync_loss=True)
    assert e.value.code == -5
    # the handle stays usable
    gm.zero_grad()
    gm.forward(tok, tgt, sync_loss=True)
    gm.backward()
    p0 = gm.get_params()
    g = gm.get_grads()
    g[17] = np.nan
    gm.set_grads(g)
    rc, n = gm.adamw_step_rc(1e-3)
    assert rc == -6 and not np.isfinite(n)
    assert np.array_equal(gm.get_params(), p0)
    m, v, t = gm.get_opt_state()
    assert t == 0 and not m.any() and not v.any()
    # adamw without accumulated gradients
    gm.zero_grad()
    rc, _ = gm.adamw_step_rc(1e-3)
    assert rc == -4


def test_bf16_gradients_near_the_oracle():
    """bf16-mixed mode, one forward/backward at the mid shape (head size 64:
    the tensor-core attention and products, the fc bias gradient out of the
    fcproj product's epilogue, the batched column sums): every gradient
    tensor within a relative L2 error of 5e-2 of the fp64 oracle, and the
    bias and LayerNorm tensors (summed by the batched column sums) within the
    same bar.  The bar: every stored activation and gradient is rounded to
    bf16 (relative 2^-8); a 2-layer model stores about a dozen of them on any
    path from the loss to a parameter, a few percent at most."""
    om, gm = _pair(MID, BF16, seed=3, perturb=5)
    tok, tgt = inputs.uniform_batch(7, MID["B"], MID["T"], MID["V"])
    om.zero_grad()
    om.forward(tok, tgt)
    om.backward()
    gm.zero_grad()
    gm.forward(tok, tgt, sync_loss=True)
    gm.backward()
    got, ref = om.split(gm.get_grads().astype(np.float64)), om.split(om.grads())
    errs = {k: float(np.linalg.norm(got[k] - ref[k]) / np.linalg.norm(ref[k])) for k in ref}
    assert all(np.isfinite(v) for v in errs.values()), errs
    assert max(errs.values()) <= 5e-2, errs
