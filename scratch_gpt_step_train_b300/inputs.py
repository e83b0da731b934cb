"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module draws token ids only; it holds none of the model's arithmetic.

* Zipf tokens stand in for the FineWeb-Edu shards the 1558M run trains on
  ("Karpathy reproduces GPT-2 (1.6B) in llm.c", section "Training"), which are
  not available here: ids are i.i.d. with p(k) proportional to (k+1)^-s over
  [0, V), drawn by inverse CDF from numpy's default_rng(seed).  Each
  micro-batch takes B*(T+1) consecutive draws laid out as [B, T+1]; tokens are
  [:, :T] and targets [:, 1:].  Successive micro-batches continue the stream.
* The binary toy follows "BabyGPT: a minimal GPT as a finite-state Markov
  chain": two tokens, context 3, 12 windows of a 15-bit stream whose ones
  have probability 0.8 (the page's own 15-bit string has 12 ones out of 15).
"""
import numpy as np


def zipf_cdf(V: int = 50257, s: float = 1.1) -> np.ndarray:
    w = (np.arange(1, V + 1, dtype=np.float64)) ** (-s)
    cdf = np.cumsum(w)
    return cdf / cdf[-1]


class ZipfStream:
    """Endless stream of (tokens, targets) micro-batches, int32 [B, T]."""

    def __init__(self, seed: int, B: int, T: int, V: int = 50257, s: float = 1.1):
        self.rng = np.random.default_rng(seed)
        self.cdf = zipf_cdf(V, s)
        self.B, self.T, self.V = B, T, V

    def next(self):
        u = self.rng.random(self.B * (self.T + 1))
        ids = np.searchsorted(self.cdf, u, side="right")
        ids = np.minimum(ids, self.V - 1).astype(np.int32).reshape(self.B, self.T + 1)
        return np.ascontiguousarray(ids[:, :-1]), np.ascontiguousarray(ids[:, 1:])


def zipf_batches(seed: int, n: int, B: int, T: int, V: int = 50257, s: float = 1.1):
    st = ZipfStream(seed, B, T, V, s)
    return [st.next() for _ in range(n)]


def uniform_batch(seed: int, B: int, T: int, V: int):
    """Uniform ids over [0, V) (used for small parity shapes)."""
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, V, size=(B, T + 1), dtype=np.int64).astype(np.int32)
    return np.ascontiguousarray(ids[:, :-1]), np.ascontiguousarray(ids[:, 1:])


def toy_bits(seed: int = 0, n: int = 15, p_one: float = 0.8) -> np.ndarray:
    return (np.random.default_rng(seed).random(n) < p_one).astype(np.int32)


def toy_windows(seed: int = 0, T: int = 3):
    """12 windows (for 15 bits, T=3): tokens bits[i:i+T], targets bits[i+1:i+T+1]."""
    bits = toy_bits(seed)
    n = len(bits) - T
    tok = np.stack([bits[i:i + T] for i in range(n)]).astype(np.int32)
    tgt = np.stack([bits[i + 1:i + T + 1] for i in range(n)]).astype(np.int32)
    return tok, tgt


def toy_states(T: int = 3) -> np.ndarray:
    """All 2^T binary contexts; row s holds the bits of s, most significant first."""
    s = np.arange(2 ** T)
    return np.stack([(s >> (T - 1 - i)) & 1 for i in range(T)], axis=1).astype(np.int32)
