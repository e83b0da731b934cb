"""ctypes wrapper around the plain-C oracle (test infrastructure only).

The C source (gpt2_oracle.c) holds all the arithmetic; this module only moves
numpy arrays in and out.  Its per-op functions mirror the layer functions of
the CPU trainer described in "Karpathy's llm.c: understanding LLM training
from scratch in C/CUDA", section "Code anatomy -- CPU version train_gpt2.c".
"""
import ctypes as ct
import os

import numpy as np

from . import build as _build

TENSOR_NAMES = ["wte", "wpe", "ln1w", "ln1b", "qkvw", "qkvb", "projw", "projb",
                "ln2w", "ln2b", "fcw", "fcb", "fcprojw", "fcprojb", "lnfw", "lnfb"]
DECAYED = {"wte", "wpe", "qkvw", "projw", "fcw", "fcprojw"}

_libs = {}


def _lib(real="double"):
    if real in _libs:
        return _libs[real]
    _build.build()
    lib = ct.CDLL(_build.lib_path(real))
    R = ct.c_double if real == "double" else ct.c_float
    pR = ct.POINTER(R)
    pI = ct.POINTER(ct.c_int)
    pD = ct.POINTER(ct.c_double)
    sz = ct.c_size_t
    i = ct.c_int
    sig = {
        "og_create": (ct.c_void_p, [i, i, i, i, i, i, ct.c_uint64]),
        "og_destroy": (None, [ct.c_void_p]),
        "og_num_params": (sz, [ct.c_void_p]),
        "og_padded_V": (i, [ct.c_void_p]),
        "og_param_count": (sz, [i, i, i, i]),
        "og_padded_vocab": (i, [i]),
        "og_normal_sample": (ct.c_float, [ct.c_uint64, ct.c_uint64, ct.c_double]),
        "og_forward": (ct.c_double, [ct.c_void_p, pI, pI]),
        "og_backward": (i, [ct.c_void_p]),
        "og_zero_grad": (None, [ct.c_void_p]),
        "og_adamw_step": (i, [ct.c_void_p] + [ct.c_double] * 6 + [pD]),
        "og_get_params": (None, [ct.c_void_p, pD]),
        "og_set_params": (None, [ct.c_void_p, pD]),
        "og_get_grads": (None, [ct.c_void_p, pD]),
        "og_set_grads": (None, [ct.c_void_p, pD]),
        "og_get_m": (None, [ct.c_void_p, pD]),
        "og_get_v": (None, [ct.c_void_p, pD]),
        "og_get_param": (ct.c_double, [ct.c_void_p, sz]),
        "og_set_param": (None, [ct.c_void_p, sz, ct.c_double]),
        "og_set_n_accum": (None, [ct.c_void_p, i]),
        "og_get_step": (i, [ct.c_void_p]),
        "og_get_logits": (None, [ct.c_void_p, pD]),
        "og_get_probs": (None, [ct.c_void_p, pD]),
        "og_get_losses": (None, [ct.c_void_p, pD]),
        "og_get_lnf": (None, [ct.c_void_p, pD]),
        "og_tensor_offset": (sz, [ct.c_void_p, i]),
        "og_tensor_size": (sz, [ct.c_void_p, i]),
        "og_encoder_forward": (None, [pR, pI, pR, pR, i, i, i]),
        "og_encoder_backward": (None, [pR, pR, pR, pI, i, i, i]),
        "og_layernorm_forward": (None, [pR, pR, pR, pR, pR, pR, i, i]),
        "og_layernorm_backward": (None, [pR, pR, pR, pR, pR, pR, pR, pR, i, i]),
        "og_matmul_forward": (None, [pR, pR, pR, pR, i, i, i]),
        "og_matmul_backward": (None, [pR, pR, pR, pR, pR, pR, i, i, i]),
        "og_attention_forward": (None, [pR, pR, pR, i, i, i, i]),
        "og_attention_backward": (None, [pR, pR, pR, pR, i, i, i, i]),
        "og_gelu_forward": (None, [pR, pR, sz]),
        "og_gelu_backward": (None, [pR, pR, pR, sz]),
        "og_crossentropy_forward": (None, [pR, pR, pR, pI, i, i, i]),
        "og_crossentropy_backward": (None, [pR, pR, pI, R, i, i, i]),
        "og_sumsq": (R, [pR, sz]),
        "og_adamw": (None, [pR, pR, pR, pR, sz, R, R, R, R, R, R, i, i]),
        "og_stochastic_round_bf16": (None, [ct.POINTER(ct.c_uint16), ct.POINTER(ct.c_float), sz,
                                            ct.c_uint64, ct.c_uint64]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    lib._np_real = np.float64 if real == "double" else np.float32
    lib._R = R
    _libs[real] = lib
    return lib


def _p(a, ctype):
    return a.ctypes.data_as(ct.POINTER(ctype))


def _ints(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, _p(a, ct.c_int)


def padded_vocab(V):
    return _lib().og_padded_vocab(V)


def param_count(L, C, Vp, T):
    return _lib().og_param_count(L, C, Vp, T)


def normal_sample(seed, i, std):
    return _lib().og_normal_sample(seed, i, std)


class Ops:
    """Per-layer oracle functions on numpy arrays (float64 or float32 build)."""

    def __init__(self, real="double"):
        self.lib = _lib(real)
        self.dt = self.lib._np_real
        self.R = self.lib._R

    def _a(self, x):
        return np.ascontiguousarray(x, dtype=self.dt)

    def _pp(self, a):
        return None if a is None else _p(a, self.R)

    def encoder_forward(self, tok, wte, wpe):
        B, T = tok.shape
        C = wte.shape[1]
        wte, wpe = self._a(wte), self._a(wpe)
        tok, ptok = _ints(tok)
        out = np.zeros((B, T, C), self.dt)
        self.lib.og_encoder_forward(self._pp(out), ptok, self._pp(wte), self._pp(wpe), B, T, C)
        return out

    def encoder_backward(self, dout, tok, Vp, Tmax=None):
        B, T, C = dout.shape
        dout = self._a(dout)
        tok, ptok = _ints(tok)
        dwte = np.zeros((Vp, C), self.dt)
        dwpe = np.zeros((Tmax or T, C), self.dt)
        self.lib.og_encoder_backward(self._pp(dwte), self._pp(dwpe), self._pp(dout), ptok, B, T, C)
        return dwte, dwpe

    def layernorm_forward(self, x, w, b):
        x, w, b = self._a(x), self._a(w), self._a(b)
        N, C = x.reshape(-1, x.shape[-1]).shape
        out = np.zeros_like(x)
        mean = np.zeros(N, self.dt)
        rstd = np.zeros(N, self.dt)
        self.lib.og_layernorm_forward(self._pp(out), self._pp(mean), self._pp(rstd), self._pp(x),
                                      self._pp(w), self._pp(b), N, C)
        return out, mean, rstd

    def layernorm_backward(self, dout, x, w, mean, rstd):
        dout, x, w, mean, rstd = map(self._a, (dout, x, w, mean, rstd))
        N, C = x.reshape(-1, x.shape[-1]).shape
        dx = np.zeros_like(x)
        dw = np.zeros(C, self.dt)
        db = np.zeros(C, self.dt)
        self.lib.og_layernorm_backward(self._pp(dx), self._pp(dw), self._pp(db), self._pp(dout),
                                       self._pp(x), self._pp(w), self._pp(mean), self._pp(rstd),
                                       N, C)
        return dx, dw, db

    def matmul_forward(self, x, w, bias=None):
        x, w = self._a(x), self._a(w)
        bias = None if bias is None else self._a(bias)
        N, C = x.reshape(-1, x.shape[-1]).shape
        OC = w.shape[0]
        out = np.zeros((N, OC), self.dt)
        self.lib.og_matmul_forward(self._pp(out), self._pp(x), self._pp(w), self._pp(bias), N, C, OC)
        return out

    def matmul_backward(self, dout, x, w, with_bias=True):
        dout, x, w = map(self._a, (dout, x, w))
        N, C = x.reshape(-1, x.shape[-1]).shape
        OC = w.shape[0]
        dx = np.zeros((N, C), self.dt)
        dw = np.zeros((OC, C), self.dt)
        db = np.zeros(OC, self.dt) if with_bias else None
        self.lib.og_matmul_backward(self._pp(dx), self._pp(dw), self._pp(db), self._pp(dout),
                                    self._pp(x), self._pp(w), N, C, OC)
        return dx, dw, db

    def attention_forward(self, qkv, H):
        qkv = self._a(qkv)
        B, T, C3 = qkv.shape
        C = C3 // 3
        out = np.zeros((B, T, C), self.dt)
        att = np.zeros((B, H, T, T), self.dt)
        self.lib.og_attention_forward(self._pp(out), self._pp(att), self._pp(qkv), B, T, C, H)
        return out, att

    def attention_backward(self, dout, qkv, att, H):
        dout, qkv, att = map(self._a, (dout, qkv, att))
        B, T, C3 = qkv.shape
        C = C3 // 3
        dqkv = np.zeros_like(qkv)
        self.lib.og_attention_backward(self._pp(dqkv), self._pp(dout), self._pp(qkv),
                                       self._pp(att), B, T, C, H)
        return dqkv

    def gelu_forward(self, x):
        x = self._a(x)
        out = np.zeros_like(x)
        self.lib.og_gelu_forward(self._pp(out), self._pp(x), x.size)
        return out

    def gelu_backward(self, x, dout):
        x, dout = self._a(x), self._a(dout)
        dx = np.zeros_like(x)
        self.lib.og_gelu_backward(self._pp(dx), self._pp(x), self._pp(dout), x.size)
        return dx

    def crossentropy_forward(self, logits, tgt, V):
        logits = self._a(logits)
        N, Vp = logits.shape
        tgt, ptgt = _ints(tgt)
        probs = np.zeros_like(logits)
        losses = np.zeros(N, self.dt)
        self.lib.og_crossentropy_forward(self._pp(probs), self._pp(losses), self._pp(logits), ptgt,
                                         N, V, Vp)
        return probs, losses

    def crossentropy_backward(self, probs, tgt, dloss, V):
        probs = self._a(probs)
        N, Vp = probs.shape
        tgt, ptgt = _ints(tgt)
        d = np.zeros_like(probs)
        self.lib.og_crossentropy_backward(self._pp(d), self._pp(probs), ptgt, dloss, N, V, Vp)
        return d

    def adamw(self, w, m, v, g, gscale, lr, b1, b2, eps, wd, decay, t):
        w, m, v, g = (np.array(a, dtype=self.dt, copy=True) for a in (w, m, v, g))
        self.lib.og_adamw(self._pp(w), self._pp(m), self._pp(v), self._pp(g), w.size, gscale,
                          lr, b1, b2, eps, wd, int(decay), int(t))
        return w, m, v


def stochastic_round_bf16(x, seed, k0=0):
    """bf16 bit patterns (uint16) of the oracle's stochastic rounding of the
    fp32 array x with SplitMix64 counters k0, k0+1, ..."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    out = np.empty(x.size, np.uint16)
    _lib("double").og_stochastic_round_bf16(out.ctypes.data_as(ct.POINTER(ct.c_uint16)),
                                            x.ctypes.data_as(ct.POINTER(ct.c_float)), x.size,
                                            int(seed), int(k0))
    return out


def splitmix64(seed, j):
    """output number j of SplitMix64 seeded with `seed`, as the oracle computes
    it (for pins)"""
    z = (seed + (j + 1) * 0x9E3779B97F4A7C15) % 2 ** 64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) % 2 ** 64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) % 2 ** 64
    return z ^ (z >> 31)


class Model:
    """The oracle's whole GPT-2 (one training micro-step at a time)."""

    def __init__(self, L, H, C, V, T, B, seed, real="double"):
        self.lib = _lib(real)
        self.L, self.H, self.C, self.V, self.T, self.B = L, H, C, V, T, B
        self.h = self.lib.og_create(L, H, C, V, T, B, seed)
        if not self.h:
            raise ValueError("oracle: bad dimensions")
        self.Vp = self.lib.og_padded_V(self.h)
        self.n = self.lib.og_num_params(self.h)

    def __del__(self):
        h = getattr(self, "h", None)
        if h:
            self.lib.og_destroy(h)
            self.h = None

    def _vec(self, fn, n=None):
        out = np.zeros(self.n if n is None else n, np.float64)
        fn(self.h, _p(out, ct.c_double))
        return out

    def params(self):
        return self._vec(self.lib.og_get_params)

    def set_params(self, p):
        p = np.ascontiguousarray(p, dtype=np.float64)
        assert p.size == self.n
        self.lib.og_set_params(self.h, _p(p, ct.c_double))

    def grads(self):
        return self._vec(self.lib.og_get_grads)

    def set_grads(self, g):
        g = np.ascontiguousarray(g, dtype=np.float64)
        assert g.size == self.n
        self.lib.og_set_grads(self.h, _p(g, ct.c_double))

    def m(self):
        return self._vec(self.lib.og_get_m)

    def v(self):
        return self._vec(self.lib.og_get_v)

    def get_param(self, i):
        return self.lib.og_get_param(self.h, i)

    def set_param(self, i, x):
        self.lib.og_set_param(self.h, i, x)

    def step_count(self):
        return self.lib.og_get_step(self.h)

    def forward(self, tokens, targets=None):
        tokens, pt = _ints(tokens)
        assert tokens.size == self.B * self.T
        if targets is None:
            return self.lib.og_forward(self.h, pt, None)
        targets, pg = _ints(targets)
        return self.lib.og_forward(self.h, pt, pg)

    def backward(self):
        rc = self.lib.og_backward(self.h)
        if rc != 0:
            raise RuntimeError("oracle: backward without a forward with targets")

    def zero_grad(self):
        self.lib.og_zero_grad(self.h)

    def set_n_accum(self, n):
        self.lib.og_set_n_accum(self.h, n)

    def adamw_step(self, lr, b1, b2, eps, wd, clip):
        norm = ct.c_double(0.0)
        rc = self.lib.og_adamw_step(self.h, lr, b1, b2, eps, wd, clip, ct.byref(norm))
        return rc, norm.value

    def logits(self):
        return self._vec(self.lib.og_get_logits, self.B * self.T * self.V).reshape(
            self.B, self.T, self.V)

    def probs(self):
        return self._vec(self.lib.og_get_probs, self.B * self.T * self.V).reshape(
            self.B, self.T, self.V)

    def losses(self):
        return self._vec(self.lib.og_get_losses, self.B * self.T).reshape(self.B, self.T)

    def lnf(self):
        return self._vec(self.lib.og_get_lnf, self.B * self.T * self.C).reshape(
            self.B, self.T, self.C)

    def tensor_slices(self):
        """name -> slice of the canonical vector"""
        out = {}
        for k, name in enumerate(TENSOR_NAMES):
            o = self.lib.og_tensor_offset(self.h, k)
            s = self.lib.og_tensor_size(self.h, k)
            out[name] = slice(o, o + s)
        return out

    def split(self, vec):
        """canonical vector -> dict of shaped arrays"""
        L, C, T, Vp = self.L, self.C, self.T, self.Vp
        shapes = {"wte": (Vp, C), "wpe": (T, C), "ln1w": (L, C), "ln1b": (L, C),
                  "qkvw": (L, 3 * C, C), "qkvb": (L, 3 * C), "projw": (L, C, C),
                  "projb": (L, C), "ln2w": (L, C), "ln2b": (L, C), "fcw": (L, 4 * C, C),
                  "fcb": (L, 4 * C), "fcprojw": (L, C, 4 * C), "fcprojb": (L, C),
                  "lnfw": (C,), "lnfb": (C,)}
        sl = self.tensor_slices()
        return {k: vec[sl[k]].reshape(shapes[k]) for k in TENSOR_NAMES}
