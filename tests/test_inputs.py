"""The seeded synthetic inputs follow their stated recipe: Zipf(s) ids drawn by
inverse CDF (closed-form head probability, empirical frequencies within
binomial bounds), targets the next token of the same draw, streams that
continue across micro-batches, and the binary toy's 12 windows of a 15-bit
stream ("BabyGPT: a minimal GPT as a finite-state Markov chain")."""
import numpy as np

from scratch_gpt_step_train_b300 import inputs


def test_zipf_cdf_closed_form():
    V, s = 50257, 1.1
    cdf = inputs.zipf_cdf(V, s)
    h = np.sum(np.arange(1, V + 1, dtype=np.float64) ** -s)
    assert abs(cdf[0] - 1.0 / h) < 1e-15 and cdf[-1] == 1.0
    assert np.all(np.diff(cdf) > 0)
    assert abs(cdf[0] - 0.139) < 1e-3  # the head id's probability at V=50257, s=1.1


def test_zipf_stream_statistics_and_layout():
    B, T, V = 16, 1024, 50257
    st = inputs.ZipfStream(2, B, T, V)
    tok, tgt = st.next()
    assert tok.dtype == np.int32 and tok.shape == (B, T) and tgt.shape == (B, T)
    assert tok.min() >= 0 and tok.max() < V
    assert np.array_equal(tok[:, 1:], tgt[:, :-1])  # targets are the next token
    n = B * (T + 1)
    p0 = inputs.zipf_cdf(V)[0]
    ids = np.concatenate([tok, tgt[:, -1:]], axis=1)
    k0 = int((ids == 0).sum())
    sd = np.sqrt(n * p0 * (1 - p0))
    assert abs(k0 - n * p0) < 5 * sd
    # the same seed gives the same stream; the next batch continues it
    again = inputs.ZipfStream(2, B, T, V)
    t2, g2 = again.next()
    assert np.array_equal(t2, tok) and np.array_equal(g2, tgt)
    nxt = st.next()[0]
    assert not np.array_equal(nxt, tok)
    assert np.array_equal(inputs.zipf_batches(2, 2, B, T, V)[1][0], nxt)


def test_toy_windows():
    bits = inputs.toy_bits(0)
    assert bits.shape == (15,) and set(np.unique(bits)) <= {0, 1}
    tok, tgt = inputs.toy_windows(0)
    assert tok.shape == (12, 3) and tgt.shape == (12, 3)
    for i in range(12):
        assert np.array_equal(tok[i], bits[i:i + 3]) and np.array_equal(tgt[i], bits[i + 1:i + 4])
    states = inputs.toy_states(3)
    assert states.shape == (8, 3)
    assert [int("".join(map(str, r)), 2) for r in states] == list(range(8))
