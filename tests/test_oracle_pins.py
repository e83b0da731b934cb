"""Pins for the CPU oracle (no GPU): each test checks the oracle against
something other than itself -- a library implementation of the same math,
finite differences, closed forms, invariants, the pages' printed numbers, and
brute force on the binary toy.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle.pyoracle import DECAYED, TENSOR_NAMES, Model, Ops, param_count
from scratch_gpt_step_train_b300 import inputs
import torch_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TINY = dict(L=2, H=2, C=32, V=64, T=8, B=2)


def _perturbed(m: Model, seed: int):
    """init + noise on every tensor, so that no parameter is degenerate
    (non-zero biases, LayerNorm gains away from 1); pad rows stay 0."""
    rng = np.random.default_rng(seed)
    p = m.params()
    sl = m.tensor_slices()
    for name in TENSOR_NAMES:
        s = sl[name]
        p[s] += rng.normal(0, 0.05 if name.startswith("ln") else 0.02, s.stop - s.start)
    wte = p[sl["wte"]].reshape(m.Vp, m.C)
    wte[m.V:] = 0
    p[sl["wte"]] = wte.reshape(-1)
    m.set_params(p)
    return p


def _batch(seed, B, T, V):
    return inputs.uniform_batch(seed, B, T, V)


# ---------------------------------------------------------------- page values

def test_param_count_matches_page():
    """num_parameters printed for the d48 model in the 1558M run log."""
    g = json.load(open(os.path.join(GOLDEN, "page_values.json")))
    n = param_count(48, 1600, 50304, 1024)
    assert n == g["num_parameters_1558M"]["value"]
    assert 2 * n == g["param_bytes_bf16_1558M"]["value"]


def test_padded_vocab_matches_page():
    from oracle.pyoracle import padded_vocab
    g = json.load(open(os.path.join(GOLDEN, "page_values.json")))
    assert padded_vocab(50257) == g["padded_vocab"]["value"]


# ---------------------------------------------------- library cross-check (torch)

@pytest.mark.parametrize("cfg", [TINY, dict(L=1, H=4, C=64, V=300, T=13, B=3)])
def test_forward_backward_vs_torch(cfg):
    m = Model(**cfg, seed=11)
    p = _perturbed(m, 5)
    tok, tgt = _batch(3, cfg["B"], cfg["T"], cfg["V"])
    loss = m.forward(tok, tgt)
    m.zero_grad()
    m.backward()
    tp = torch_ref.to_torch(m.split(p))
    logits, tloss = torch_ref.forward(tp, tok, tgt, cfg["L"], cfg["H"], cfg["C"], cfg["V"])
    tloss.backward()
    assert abs(loss - tloss.item()) <= 1e-12 * abs(loss)
    np.testing.assert_allclose(m.logits(), logits.detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(m.probs().sum(-1), 1.0, atol=1e-12)
    g = m.split(m.grads())
    for k in TENSOR_NAMES:
        ref = tp[k].grad.numpy()
        scale = max(np.abs(ref).max(), 1e-30)
        assert np.abs(g[k] - ref).max() <= 1e-10 * scale, k


def test_adamw_accum_clip_vs_torch():
    """two micro-batches, global clip active, decay mask; three steps."""
    cfg = TINY
    m = Model(**cfg, seed=7)
    p = _perturbed(m, 9)
    tp = torch_ref.to_torch(m.split(p))
    hp = dict(lr=1e-2, b1=0.9, b2=0.95, eps=1e-8, wd=0.1)
    opt = torch_ref.make_optimizer(tp, **hp)
    for step in range(3):
        m.zero_grad()
        opt.zero_grad()
        batches = [_batch(100 + 2 * step + i, cfg["B"], cfg["T"], cfg["V"]) for i in range(2)]
        tl = 0
        for tok, tgt in batches:
            m.forward(tok, tgt)
            m.backward()
            _, loss = torch_ref.forward(tp, tok, tgt, cfg["L"], cfg["H"], cfg["C"], cfg["V"])
            tl = tl + loss / 2
        tl.backward()
        clip = 0.05  # small enough to be active
        rc, norm = m.adamw_step(**hp, clip=clip)
        tnorm = torch_ref.clip_and_step(tp, opt, clip)
        assert rc == 0
        assert norm > clip
        assert abs(norm - tnorm) <= 1e-12 * tnorm
        got = m.split(m.params())
        for k in TENSOR_NAMES:
            ref = tp[k].detach().numpy()
            assert np.abs(got[k] - ref).max() <= 1e-12 * max(np.abs(ref).max(), 1e-30), k


# ------------------------------------------------------------ finite differences

def _fd_check(m, tok, tgt, idx, rel_h=1e-3, tol=1e-7):
    """Central differences with one Richardson step (error O(h^4)):
    D(h) = (f(w+h)-f(w-h))/2h,  estimate = (4 D(h/2) - D(h)) / 3."""
    m.forward(tok, tgt)
    m.zero_grad()
    m.backward()
    g = m.grads()
    worst = 0.0
    scale = np.abs(g).max()

    def central(i, w0, h):
        m.set_param(i, w0 + h)
        lp = m.forward(tok, tgt)
        m.set_param(i, w0 - h)
        lm = m.forward(tok, tgt)
        m.set_param(i, w0)
        return (lp - lm) / (2 * h)

    for i in idx:
        i = int(i)
        w0 = m.get_param(i)
        h = rel_h * max(1.0, abs(w0))
        fd = (4 * central(i, w0, h / 2) - central(i, w0, h)) / 3
        err = abs(fd - g[i]) / (abs(g[i]) + 1e-3 * scale)
        worst = max(worst, err)
    assert worst < tol, worst


def test_finite_differences_tiny():
    m = Model(**TINY, seed=3)
    _perturbed(m, 4)
    tok, tgt = _batch(8, TINY["B"], TINY["T"], TINY["V"])
    rng = np.random.default_rng(0)
    idx = []
    for name, s in m.tensor_slices().items():
        n = s.stop - s.start
        if name == "wte":
            # real rows (first V*C entries) plus a few padded-row entries
            idx += list(s.start + rng.choice(TINY["V"] * TINY["C"], 24, replace=False))
            idx += list(s.start + TINY["V"] * TINY["C"] + rng.choice(n - TINY["V"] * TINY["C"], 4))
        else:
            idx += list(s.start + rng.choice(n, min(n, 16), replace=False))
    _fd_check(m, tok, tgt, idx)


def test_finite_differences_toy_every_parameter():
    m = Model(L=2, H=2, C=16, V=2, T=3, B=12, seed=0)
    _perturbed(m, 1)
    tok, tgt = inputs.toy_windows(0)
    sl = m.tensor_slices()
    real_wte = range(sl["wte"].start, sl["wte"].start + 2 * 16)
    idx = list(real_wte) + list(range(sl["wpe"].start, m.n))
    _fd_check(m, tok, tgt, idx)


# -------------------------------------------------------------------- invariants

def test_causal_exactness():
    """changing tokens after position t leaves logits at <= t bit-identical"""
    m = Model(**TINY, seed=2)
    _perturbed(m, 2)
    tok, tgt = _batch(1, TINY["B"], TINY["T"], TINY["V"])
    m.forward(tok, tgt)
    a = m.logits().copy()
    t0 = 3
    tok2 = tok.copy()
    tok2[:, t0 + 1:] = (tok2[:, t0 + 1:] + 7) % TINY["V"]
    m.forward(tok2, tgt)
    b = m.logits()
    assert np.array_equal(a[:, :t0 + 1], b[:, :t0 + 1])
    assert not np.array_equal(a[:, t0 + 1:], b[:, t0 + 1:])


def test_layernorm_moments(ops64):
    rng = np.random.default_rng(0)
    x = rng.normal(0.3, 2.0, (17, 96))
    y, mean, rstd = ops64.layernorm_forward(x, np.ones(96), np.zeros(96))
    var = x.var(axis=1)
    np.testing.assert_allclose(y.mean(1), 0, atol=1e-13)
    np.testing.assert_allclose(y.var(1), var / (var + 1e-5), rtol=1e-12)
    np.testing.assert_allclose(mean, x.mean(1), rtol=1e-13)


def test_layernorm_vs_torch(ops64):
    rng = np.random.default_rng(1)
    x = rng.normal(0, 1.5, (9, 40))
    w, b = rng.normal(1, 0.1, 40), rng.normal(0, 0.1, 40)
    dy = rng.normal(0, 1, x.shape)
    y, mean, rstd = ops64.layernorm_forward(x, w, b)
    dx, dw, db = ops64.layernorm_backward(dy, x, w, mean, rstd)
    tx, tw, tb = (torch.tensor(a, requires_grad=True) for a in (x, w, b))
    ty = torch.nn.functional.layer_norm(tx, (40,), tw, tb, eps=1e-5)
    ty.backward(torch.tensor(dy))
    np.testing.assert_allclose(y, ty.detach().numpy(), atol=1e-13)
    np.testing.assert_allclose(dx, tx.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dw, tw.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(db, tb.grad.numpy(), atol=1e-12)


def test_gelu_special_values(ops64):
    x = np.array([0.0, 1.0, -1.0, 10.0, -10.0, 3.0])
    y = ops64.gelu_forward(x)
    assert y[0] == 0.0
    # odd/even split: gelu(x) - gelu(-x) = x
    np.testing.assert_allclose(y[1] - y[2], 1.0, atol=1e-15)
    np.testing.assert_allclose(y[3], 10.0, atol=1e-12)
    np.testing.assert_allclose(y[4], 0.0, atol=1e-12)
    np.testing.assert_allclose(ops64.gelu_backward(np.array([0.0]), np.array([1.0])), 0.5)
    t = torch.nn.functional.gelu(torch.tensor(x), approximate="tanh").numpy()
    np.testing.assert_allclose(y, t, atol=1e-15)


def test_dlogits_rows_sum_to_zero(ops64):
    rng = np.random.default_rng(0)
    logits = rng.normal(0, 3, (6, 256))
    tgt = rng.integers(0, 200, 6)
    probs, losses = ops64.crossentropy_forward(logits, tgt, 200)
    d = ops64.crossentropy_backward(probs, tgt, 1 / 6, 200)
    np.testing.assert_allclose(d.sum(1), 0, atol=1e-16)
    assert np.all(d[:, 200:] == 0)
    ref = torch.nn.functional.cross_entropy(torch.tensor(logits[:, :200]), torch.tensor(tgt),
                                            reduction="none").numpy()
    np.testing.assert_allclose(losses, ref, rtol=1e-13)


def test_padded_rows_stay_zero_and_batch_permutation():
    m = Model(**TINY, seed=4)
    tok, tgt = _batch(5, TINY["B"], TINY["T"], TINY["V"])
    for _ in range(3):
        m.zero_grad()
        m.forward(tok, tgt)
        m.backward()
        m.adamw_step(1e-2, 0.9, 0.95, 1e-8, 0.1, 1.0)
    wte = m.split(m.params())["wte"]
    assert np.all(wte[TINY["V"]:] == 0)
    m.zero_grad()
    l1 = m.forward(tok, tgt)
    m.backward()
    g1 = m.grads()
    los1 = m.losses()
    m.zero_grad()
    l2 = m.forward(tok[::-1].copy(), tgt[::-1].copy())
    m.backward()
    g2 = m.grads()
    assert abs(l1 - l2) <= 1e-14 * abs(l1)
    np.testing.assert_array_equal(m.losses()[::-1], los1)
    np.testing.assert_allclose(g1, g2, rtol=0, atol=1e-13 * np.abs(g1).max())


# ------------------------------------------------------------------ closed forms

def test_adamw_scalar_closed_form(ops64):
    """constant gradient: mhat = g, vhat = g^2 exactly, so
    w_t = w0 (1-lr wd)^t - lr s sum_{k<t} (1-lr wd)^k with s = g/(|g|+eps)."""
    lr, wd, eps, g = 0.01, 0.1, 1e-8, -0.37
    w, m_, v = np.array([0.5]), np.zeros(1), np.zeros(1)
    for t in range(1, 21):
        w, m_, v = ops64.adamw(w, m_, v, np.array([g]), 1.0, lr, 0.9, 0.95, eps, wd, 1, t)
        r = 1 - lr * wd
        s = g / (abs(g) + eps)
        closed = 0.5 * r ** t - lr * s * sum(r ** k for k in range(t))
        assert abs(w[0] - closed) < 1e-13
    # decay off: no shrink term
    w, m_, v = ops64.adamw(np.array([0.5]), np.zeros(1), np.zeros(1), np.array([g]), 1.0, lr,
                           0.9, 0.95, eps, wd, 0, 1)
    assert abs(w[0] - (0.5 - lr * g / (abs(g) + eps))) < 1e-15


def test_clip_post_norm_equals_min():
    """after the step, m = (1-b1) * s * g/n_accum, so its norm / (1-b1) is the
    post-clip gradient norm = min(n, clip)."""
    for clip in (0.01, 1e3):
        m = Model(**TINY, seed=6)
        tok, tgt = _batch(2, TINY["B"], TINY["T"], TINY["V"])
        m.zero_grad()
        for _ in range(2):  # two micro-batches of the same data
            m.forward(tok, tgt)
            m.backward()
        rc, n = m.adamw_step(1e-3, 0.9, 0.95, 1e-8, 0.0, clip)
        post = np.linalg.norm(m.m()) / (1 - 0.9)
        assert rc == 0
        assert abs(post - min(n, clip)) <= 1e-12 * min(n, clip)


def test_nonfinite_norm_skips_update():
    m = Model(**TINY, seed=6)
    tok, tgt = _batch(2, TINY["B"], TINY["T"], TINY["V"])
    m.zero_grad()
    m.forward(tok, tgt)
    m.backward()
    p0 = m.params()
    g = m.grads()
    g[123] = np.inf
    m.set_grads(g)
    rc, n = m.adamw_step(1e-3, 0.9, 0.95, 1e-8, 0.1, 1.0)
    assert rc == -6 and not np.isfinite(n)
    np.testing.assert_array_equal(m.params(), p0)
    assert m.step_count() == 0 and np.all(m.m() == 0)


@pytest.mark.parametrize("C,T,B", [(768, 128, 2), (1600, 64, 2)])
def test_init_loss_closed_form(C, T, B):
    """At init lnf rows have unit variance, so each real logit is ~N(0, C*0.02^2)
    given the row, and the log-sum-exp over V logits is ln V + C*0.02^2/2 up to
    a relative spread ~sqrt((e^{sigma^2}-1)/V).  The mean loss adds -logit[tgt],
    whose mean over n positions has std sigma/sqrt(n)."""
    V = 50257
    m = Model(L=1, H=C // 64, C=C, V=V, T=T, B=B, seed=1)
    tok, tgt = inputs.zipf_batches(2, 1, B, T, V)[0]
    loss = m.forward(tok, tgt)
    logits = m.logits().reshape(-1, V)
    zt = logits[np.arange(B * T), tgt.reshape(-1)]
    lse = m.losses().reshape(-1) + zt
    sigma2 = C * 0.02 ** 2
    closed = math.log(V) + sigma2 / 2
    assert abs(lse.mean() - closed) < 0.01
    assert abs(loss - closed) < 4 * math.sqrt(sigma2 / (B * T)) + 0.01
    if C == 1600:
        g = json.load(open(os.path.join(GOLDEN, "page_values.json")))
        for key in ("init_val_loss_1558M", "step1_loss_1558M"):
            assert abs(g[key]["value"] - closed) < 0.05


def test_init_distribution():
    """init draws: N(0, 0.02) for matrices, 0.02/sqrt(2L) for the two residual
    projections, zeros for biases and padded rows, ones for LN gains."""
    from scipy import stats
    m = Model(L=2, H=2, C=64, V=1000, T=32, B=1, seed=123)
    p = m.split(m.params())
    for k in ("wte", "qkvw", "fcw", "wpe"):
        x = p[k][:1000] if k == "wte" else p[k]
        x = x.reshape(-1)
        assert abs(x.std() - 0.02) < 0.02 * 5 / math.sqrt(2 * x.size)
        assert stats.kstest(x / 0.02, "norm").pvalue > 1e-4
    for k in ("projw", "fcprojw"):
        x = p[k].reshape(-1)
        assert stats.kstest(x / (0.02 / math.sqrt(4)), "norm").pvalue > 1e-4
    assert np.all(p["wte"][1000:] == 0)
    for k in ("qkvb", "projb", "fcb", "fcprojb", "ln1b", "ln2b", "lnfb"):
        assert np.all(p[k] == 0)
    for k in ("ln1w", "ln2w", "lnfw"):
        assert np.all(p[k] == 1)
    # values are fp32-representable
    allp = m.params()
    assert np.array_equal(allp, allp.astype(np.float32).astype(np.float64))
    # a different seed gives different draws
    m2 = Model(L=2, H=2, C=64, V=1000, T=32, B=1, seed=124)
    assert not np.array_equal(m2.params(), allp)


# --------------------------------------------------------------- toy binary GPT

TOY = dict(L=2, H=2, C=16, V=2, T=3)


def _arrows(params, real="double"):
    """P(next = 1 | state) at the last position, for all 8 states at once."""
    m = Model(**TOY, B=8, seed=0, real=real)
    m.set_params(params)
    m.forward(inputs.toy_states(), None)
    return m.logits()[:, -1, :]


def _softmax1(z):
    return 1 / (1 + np.exp(z[:, 0] - z[:, 1]))


def test_toy_transition_table_brute_force_and_training():
    m = Model(**TOY, B=12, seed=0)
    tok, tgt = inputs.toy_windows(0)
    p0 = m.params()
    a0 = _softmax1(_arrows(p0))
    # init: logits ~ N(0, 16*0.02^2), so each arrow is 0.5 within a few 0.03
    assert np.all(np.abs(a0 - 0.5) < 0.1)
    # brute force: each state alone (B=1) gives the same arrow as the batch
    for s, state in enumerate(inputs.toy_states()):
        m1 = Model(**TOY, B=1, seed=0)
        m1.set_params(p0)
        m1.forward(state[None, :], None)
        assert abs(_softmax1(m1.logits()[:, -1, :])[0] - a0[s]) < 1e-15
    # 50 steps, lr 1e-2, wd 0, torch AdamW defaults otherwise, no clipping
    tp = torch_ref.to_torch(m.split(p0))
    opt = torch_ref.make_optimizer(tp, 1e-2, 0.9, 0.999, 1e-8, 0.0)
    losses = []
    for step in range(50):
        m.zero_grad()
        losses.append(m.forward(tok, tgt))
        m.backward()
        assert m.adamw_step(1e-2, 0.9, 0.999, 1e-8, 0.0, 0.0)[0] == 0
        opt.zero_grad()
        _, tl = torch_ref.forward(tp, tok, tgt, TOY["L"], TOY["H"], TOY["C"], TOY["V"])
        tl.backward()
        torch_ref.clip_and_step(tp, opt, 0.0)
        if step == 9:
            ref = torch.cat([tp[k].detach().reshape(-1) for k in TENSOR_NAMES]).numpy()
            assert np.abs(m.params() - ref).max() < 1e-11
    a50 = _softmax1(_arrows(m.params()))
    ref = torch.cat([tp[k].detach().reshape(-1) for k in TENSOR_NAMES]).numpy()
    a50_torch = _softmax1(_arrows(ref))
    # The key-bias gradient is zero in exact arithmetic (a shift shared by all
    # keys cancels in the softmax); both sides get rounding noise there, which
    # Adam's normalisation turns into 1e-13-sized steps.  This toy's training
    # is sensitive enough that those differences grow to ~1e-6 by step 50.
    np.testing.assert_allclose(a50, a50_torch, atol=1e-5)
    assert losses[-1] < losses[0] - 0.05
    # arrows move toward the empirical next-bit frequency of each seen state
    states = [int("".join(map(str, r)), 2) for r in tok]
    for s in range(8):
        nxt = [tgt[i, -1] for i in range(len(states)) if states[i] == s]
        if not nxt:
            continue
        f = float(np.mean(nxt))
        if abs(f - 0.5) >= 0.3:
            assert abs(a50[s] - f) < abs(a0[s] - f) - 0.1, (s, f, a0[s], a50[s])


# ------------------------------------------------ stochastic rounding (-w 0)

def test_splitmix64_published_first_output():
    from oracle.pyoracle import splitmix64
    # the first output of SplitMix64 seeded with 0 (Steele, Lea & Flood 2014)
    assert splitmix64(0, 0) == 0xE220A8397B1DCDAF


def test_stochastic_round_bf16_oracle():
    from oracle.pyoracle import splitmix64, stochastic_round_bf16
    rng = np.random.default_rng(21)
    x = (rng.normal(0, 1, 4096) * np.exp(rng.uniform(-20, 20, 4096))).astype(np.float32)
    bits = x.view(np.uint32)
    top = (bits >> 16).astype(np.uint32)
    seed, k0 = 12345, 777
    out = stochastic_round_bf16(x, seed, k0).astype(np.uint32)
    # always one of the two bf16 neighbours of |x| (sign-magnitude)
    assert np.all((out == top) | (out == top + 1))
    # the decision follows the published generator: up iff f + r >= 2^16
    for i in range(0, 4096, 97):
        r = splitmix64(seed, k0 + i) >> 48
        f = int(bits[i]) & 0xFFFF
        assert int(out[i]) == int(top[i]) + (1 if f + r >= 65536 else 0)
    # values on the bf16 grid stay put; NaN -> quiet NaN; inf stays inf
    grid = (top.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(stochastic_round_bf16(grid, seed, k0).astype(np.uint32), top)
    sp = np.array([np.nan, np.inf, -np.inf, 0.0, -0.0], np.float32)
    assert list(stochastic_round_bf16(sp, 1)) == [0x7FC0, 0x7F80, 0xFF80, 0x0000, 0x8000]
    # unbiased: 1 + 2^-9 lies a quarter of the way from 1 to 1 + 2^-7
    n = 200000
    y = stochastic_round_bf16(np.full(n, 1.0 + 2.0 ** -9, np.float32), 99, 0)
    up = np.mean(y == 0x3F81)
    assert np.all((y == 0x3F80) | (y == 0x3F81))
    assert abs(up - 0.25) < 4 * np.sqrt(0.25 * 0.75 / n)
