"""Write the stored expected values of the GPT-2 124M whole-step parity test.

Test infrastructure: this script calls only the oracle (oracle/pyoracle.py,
fp64 build) and the seeded token generator (scratch_gpt_step_train_b300/
inputs.py, which holds none of the model's arithmetic).  Nothing it stores
comes from the CUDA library.

Workload (GPT-2 124M: L=12, H=12, C=768, V=50257 padded to 50304, T=1024,
B=4, weights from seed 1, tokens i.i.d. Zipf(1.1) from seed 2 with the stream
continuing from step to step, targets = next token; AdamW lr 6e-4, b1 0.9,
b2 0.95, eps 1e-8, wd 0.1, clip 1.0).  Twenty steps, one micro-batch each:
zero_grad, forward with targets, backward, AdamW.

Stored (tests/golden/gpt2_124M_B4T1024.npz):
  loss[s], norm[s]            mean loss of step s+1 and the global gradient
                              norm its update saw (before clipping)
  gnorm[s, k], gmax[s, k]     L2 norm and max |.| of gradient tensor k
  tok_sum[s]                  sum of the step's token ids (generator check)
  idx_<name>                  sampled canonical offsets within tensor <name>:
                              every element of tensors up to 65536 elements,
                              8192 seeded draws (sorted, unique) otherwise
  grad1_<name>, grad10_<name> the sampled gradient elements at steps 1 and 10
  param10_<name>              the sampled parameters after the tenth update
  lrow, lcol                  32 sampled rows (of B*T) and 1024 sampled columns
                              (of V) of the logits
  logit1, logit10             the sampled logits at steps 1 and 10 (the
                              forward of that step, before its update)
  lmax1, lmax10               max |logit| of each sampled row over all V

With --real float the same script runs the fp32 build of the oracle for the
first ten steps and writes the same quantities to gpt2_124M_B4T1024_f32.npz:
how far a plain fp32 evaluation of the step drifts from the fp64 one along
the trajectory (after the first update two fp32 evaluations no longer hold
the same weights), which sets the test's bar from the second step on.

Run it on the CPU (about 70 minutes on 8 cores, 30 more for --real float):
    OMP_NUM_THREADS=8 python -m oracle.make_golden_124M [--real float]
"""
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle.pyoracle import TENSOR_NAMES, Model  # noqa: E402
from scratch_gpt_step_train_b300.inputs import ZipfStream  # noqa: E402

CFG = dict(L=12, H=12, C=768, V=50257, T=1024, B=4, wseed=1, tseed=2)
HP = dict(lr=6e-4, b1=0.9, b2=0.95, eps=1e-8, wd=0.1, clip=1.0)
STEPS = 20
SNAP = (1, 10)
OUT = os.path.join(ROOT, "tests", "golden", "gpt2_124M_B4T1024.npz")
OUT_F32 = os.path.join(ROOT, "tests", "golden", "gpt2_124M_B4T1024_f32.npz")


def sample_offsets(sizes, seed=7, full_upto=65536, n=8192):
    rng = np.random.default_rng(seed)
    out = {}
    for k in TENSOR_NAMES:
        s = sizes[k]
        if s <= full_upto:
            out[k] = np.arange(s, dtype=np.int64)
        else:
            out[k] = np.unique(rng.integers(0, s, size=n, dtype=np.int64))
    return out


def main(real="double"):
    c = CFG
    steps, out = (STEPS, OUT) if real == "double" else (10, OUT_F32)
    t0 = time.time()
    m = Model(c["L"], c["H"], c["C"], c["V"], c["T"], c["B"], c["wseed"], real=real)
    sl = m.tensor_slices()
    sizes = {k: sl[k].stop - sl[k].start for k in TENSOR_NAMES}
    idx = sample_offsets(sizes)
    rng = np.random.default_rng(11)
    BT = c["B"] * c["T"]
    lrow = np.sort(rng.choice(BT, size=32, replace=False)).astype(np.int64)
    lcol = np.sort(rng.choice(c["V"], size=1024, replace=False)).astype(np.int64)
    stream = ZipfStream(c["tseed"], c["B"], c["T"])
    res = {"loss": np.zeros(steps), "norm": np.zeros(steps),
           "gnorm": np.zeros((steps, 16)), "gmax": np.zeros((steps, 16)),
           "tok_sum": np.zeros(steps, np.int64), "lrow": lrow, "lcol": lcol}
    for k in TENSOR_NAMES:
        res["idx_" + k] = idx[k]
    for s in range(1, steps + 1):
        tok, tgt = stream.next()
        res["tok_sum"][s - 1] = int(tok.astype(np.int64).sum())
        m.zero_grad()
        loss = m.forward(tok, tgt)
        res["loss"][s - 1] = loss
        if s in SNAP:
            lg = m.logits().reshape(BT, c["V"])[lrow]
            res[f"logit{s}"] = lg[:, lcol].astype(np.float32)
            res[f"lmax{s}"] = np.abs(lg).max(axis=1)
        m.backward()
        g = m.grads()
        for j, k in enumerate(TENSOR_NAMES):
            gk = g[sl[k]]
            res["gnorm"][s - 1, j] = np.linalg.norm(gk)
            res["gmax"][s - 1, j] = np.abs(gk).max()
            if s in SNAP:
                res[f"grad{s}_{k}"] = gk[idx[k]].astype(np.float32)
        del g
        rc, norm = m.adamw_step(HP["lr"], HP["b1"], HP["b2"], HP["eps"], HP["wd"], HP["clip"])
        if rc != 0:
            raise RuntimeError(f"oracle AdamW step {s} returned {rc}")
        res["norm"][s - 1] = norm
        if s == 10 and real == "double":
            p = m.params()
            for k in TENSOR_NAMES:
                res[f"param10_{k}"] = p[sl[k]][idx[k]].astype(np.float32)
            del p
        print(f"step {s:2d}  loss {loss:.6f}  norm {norm:.6f}  ({time.time() - t0:.0f} s)",
              flush=True)
    tmp = out + ".tmp.npz"
    np.savez_compressed(tmp, **res)
    os.replace(tmp, out)
    print("wrote", out, flush=True)


if __name__ == "__main__":
    main("float" if "--real" in sys.argv and sys.argv[sys.argv.index("--real") + 1] == "float"
         else "double")
