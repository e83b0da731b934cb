"""Data-parallel step with the optimizer update sharded over the ranks
("Karpathy reproduces GPT-2 (1.6B) in llm.c", "Training": one process per
GPU, gradients averaged over the ranks).

CPU part: two gloo ranks drive dp.DataParallel over a stand-in model whose
shard update is the oracle's AdamW; after three steps each rank's parameters
must equal, bit for bit, one process updating the whole vector with the
gradient summed over both ranks' micro-batches and divided by their total
count.  GPU part: the same split done on one GPU by two handles (each updating
its half, the halves then exchanged) equals the plain whole-vector step bit
for bit, in fp32, bf16 and bf16 without master weights; and DataParallel over
a one-rank NCCL group equals the plain step."""
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from scratch_gpt_step_train_b300.dp import DataParallel, shard_bounds

HP = dict(lr=1e-2, b1=0.9, b2=0.95, eps=1e-8, wd=0.1, clip=1.0)
N_PARAMS = 1000  # ragged over two ranks: slices [0, 512) and [512, 1000)
MICRO = 2
STEPS = 3


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_shard_bounds_cover_and_align():
    for n in (0, 1, 63, 64, 1000, 124475904):
        for world in (1, 2, 3, 8):
            b = shard_bounds(n, world)
            assert len(b) == world and b[0][0] == 0 and b[-1][1] == n
            for (lo, hi), (lo2, _) in zip(b, b[1:]):
                assert hi == lo2
            for lo, hi in b:
                assert 0 <= lo <= hi <= n
                assert (lo % 64 == 0 or lo == n) and (hi % 64 == 0 or hi == n)
    assert shard_bounds(10, 4) == [(0, 10), (10, 10), (10, 10), (10, 10)]


class OracleShardModel:
    """Stand-in for a GPT2 handle: fp64 CPU vectors, the update of a slice
    done by the oracle's AdamW, the clip scale from the norm of the whole
    summed gradient divided by the micro-batch count.  With shard=(lo, hi) it
    holds the moments of that slice alone, as a ZeRO-1 handle does."""

    def __init__(self, n, seed, shard=None):
        from oracle.pyoracle import Ops
        self.ops = Ops("double")
        g = torch.Generator().manual_seed(seed)
        self.n = n
        self.shard = tuple(shard) if shard is not None else (0, n)
        ns = self.shard[1] - self.shard[0]
        self.w = torch.randn(n, generator=g, dtype=torch.float64) * 0.02
        self.m = torch.zeros(ns, dtype=torch.float64)
        self.v = torch.zeros(ns, dtype=torch.float64)
        self.g = torch.zeros(n, dtype=torch.float64)
        self.count = 0
        self.dcount = None
        self.t = 0

    def zero_grad(self):
        self.g.zero_()
        self.count = 0

    def accumulate(self, grad):
        self.g += grad
        self.count += 1

    def grads_tensor(self):
        return self.g

    def param_tensors(self):
        return self.w, None

    def grad_count(self):
        return self.count

    def set_grad_count(self, c):
        self.count = c

    def set_grad_count_device(self, t):
        self.dcount = t  # read by the next update, then dropped

    def adamw_step_shard(self, lo, hi, lr, b1, b2, eps, wd, clip):
        count = int(self.dcount.item()) if self.dcount is not None else self.count
        self.dcount = None
        norm = float(torch.sqrt((self.g * self.g).sum())) / count
        if not np.isfinite(norm):  # the library's GPT2_ERR_NONFINITE: nothing updated
            raise FloatingPointError("gradient norm is not finite")
        sc = (1.0 / count) * (clip / norm if clip > 0 and norm > clip else 1.0)
        self.t += 1
        s0 = self.shard[0]
        assert self.shard == (0, self.n) or self.shard == (lo, hi)
        if hi > lo:
            w, m, v = self.ops.adamw(self.w[lo:hi].numpy(), self.m[lo - s0:hi - s0].numpy(),
                                     self.v[lo - s0:hi - s0].numpy(), self.g[lo:hi].numpy(), sc,
                                     lr, b1, b2, eps, wd, True, self.t)
            self.w[lo:hi] = torch.from_numpy(w)
            self.m[lo - s0:hi - s0] = torch.from_numpy(m)
            self.v[lo - s0:hi - s0] = torch.from_numpy(v)
        return norm


def _micro_grad(rank, step, k, n=N_PARAMS):
    g = torch.Generator().manual_seed(1000 * rank + 10 * step + k)
    return torch.randn(n, generator=g, dtype=torch.float64)


def _micro_count(rank, uneven):
    return MICRO + rank if uneven else MICRO


def _gloo_rank(rank, world, port, q, n=N_PARAMS, uneven=False):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        # each rank holds the moments of its own slice only (ZeRO-1)
        model = OracleShardModel(n, seed=5, shard=shard_bounds(n, world)[rank])
        dp = DataParallel(model)
        norms = []
        for step in range(STEPS):
            model.zero_grad()
            for k in range(_micro_count(rank, uneven)):
                model.accumulate(_micro_grad(rank, step, k, n))
            norms.append(dp.step(**HP))
        q.put((rank, model.w.numpy().copy(), model.m.numpy().copy(), norms))
    finally:
        dist.destroy_process_group()


def _run_gloo(world, n, uneven=False):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gloo_rank, args=(r, world, port, q, n, uneven))
             for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(world):
        rank, w, m, norms = q.get(timeout=120)
        got[rank] = (w, m, norms)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return got


@pytest.mark.parametrize("world,n,uneven", [(3, 1000, False), (4, 10, False), (3, 1000, True)],
                         ids=["3-ranks", "4-ranks-empty-shards", "3-ranks-uneven-micro-batches"])
def test_data_parallel_gloo_more_ranks(world, n, uneven):
    """three ranks (ragged last slice), four ranks over 10 parameters (one
    64-aligned slice holds everything, the other ranks update nothing but still
    take part), and three ranks with 2, 3 and 4 micro-batches (the divisor is
    their sum): every rank ends with the one-process result; the all-reduce of
    more than two ranks may add in another order, hence a tolerance"""
    got = _run_gloo(world, n, uneven)
    ref = OracleShardModel(n, seed=5)
    for step in range(STEPS):
        ref.zero_grad()
        total = torch.zeros(n, dtype=torch.float64)
        for r in range(world):
            for k in range(_micro_count(r, uneven)):
                total += _micro_grad(r, step, k, n)
        ref.g.copy_(total)
        ref.set_grad_count(sum(_micro_count(r, uneven) for r in range(world)))
        ref.adamw_step_shard(0, n, **HP)
    bounds = shard_bounds(n, world)
    for r in range(world):
        w, m, norms = got[r]
        np.testing.assert_allclose(w, ref.w.numpy(), rtol=1e-12, atol=1e-15)
        lo, hi = bounds[r]
        assert m.size == hi - lo  # the rank holds its slice of the moments alone
        np.testing.assert_allclose(m, ref.m.numpy()[lo:hi], rtol=1e-12, atol=1e-15)
        assert all(got[q][2] == norms for q in range(world))  # one summed gradient everywhere


def _gloo_rank_poisoned(rank, world, port, q):
    """rank 1 feeds a NaN into step 1's gradient; every rank must see the step
    fail, clear its gradients and go on"""
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        model = OracleShardModel(N_PARAMS, seed=5, shard=shard_bounds(N_PARAMS, world)[rank])
        dp = DataParallel(model)
        failed = []
        for step in range(STEPS):
            model.zero_grad()
            for k in range(MICRO):
                g = _micro_grad(rank, step, k)
                if step == 1 and rank == 1 and k == 0:
                    g[7] = float("nan")
                model.accumulate(g)
            try:
                dp.step(**HP)
                failed.append(False)
            except FloatingPointError:
                failed.append(True)
        q.put((rank, model.w.numpy().copy(), failed))
    finally:
        dist.destroy_process_group()


def test_data_parallel_gloo_non_finite_step_fails_on_every_rank():
    """a non-finite gradient on one rank reaches every rank through the
    all-reduce: the step fails alike everywhere, updates nothing, and after
    zero_grad the next step equals one process that skipped it"""
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gloo_rank_poisoned, args=(r, world, port, q))
             for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(world):
        rank, w, failed = q.get(timeout=120)
        got[rank] = (w, failed)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    ref = OracleShardModel(N_PARAMS, seed=5)
    for step in range(STEPS):
        if step == 1:
            continue
        ref.zero_grad()
        per_rank = []
        for r in range(world):  # each rank's own sum, then the two ranks' (the all-reduce)
            acc = torch.zeros(N_PARAMS, dtype=torch.float64)
            for k in range(MICRO):
                acc += _micro_grad(r, step, k)
            per_rank.append(acc)
        ref.g.copy_(per_rank[0] + per_rank[1])
        ref.set_grad_count(world * MICRO)
        ref.adamw_step_shard(0, N_PARAMS, **HP)
    for r in range(world):
        w, failed = got[r]
        assert failed == [False, True, False]
        assert np.array_equal(w, ref.w.numpy())


def test_data_parallel_gloo_two_ranks_equals_one_process():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gloo_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(world):
        rank, w, m, norms = q.get(timeout=120)
        got[rank] = (w, m, norms)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0

    ref = OracleShardModel(N_PARAMS, seed=5)
    ref_norms = []
    for step in range(STEPS):
        ref.zero_grad()
        per_rank = []
        for r in range(world):
            acc = torch.zeros(N_PARAMS, dtype=torch.float64)
            for k in range(MICRO):
                acc += _micro_grad(r, step, k)
            per_rank.append(acc)
        ref.g.copy_(per_rank[0] + per_rank[1])
        ref.set_grad_count(world * MICRO)
        ref_norms.append(ref.adamw_step_shard(0, N_PARAMS, **HP))
    bounds = shard_bounds(N_PARAMS, world)
    for r in range(world):
        w, m, norms = got[r]
        assert np.array_equal(w, ref.w.numpy())  # every slice, after the exchange
        lo, hi = bounds[r]
        assert np.array_equal(m, ref.m.numpy()[lo:hi])  # this rank's optimizer shard
        assert norms == ref_norms


# ---------------------------------------------------------------------------
# GPU
# ---------------------------------------------------------------------------
CFG = dict(L=2, H=2, C=128, V=300, T=64, B=2)


def _gpu_modes():
    from scratch_gpt_step_train_b300.gpt2 import BF16, FP32, NO_MASTER
    return [FP32, BF16, BF16 | NO_MASTER]


def _batch(seed):
    from scratch_gpt_step_train_b300 import inputs
    return inputs.uniform_batch(seed, CFG["B"], CFG["T"], CFG["V"])


def _micro(gm, seed):
    tok, tgt = _batch(seed)
    gm.forward(tok, tgt)
    gm.backward()


@pytest.mark.gpu
@pytest.mark.parametrize("mi", [0, 1, 2], ids=["fp32", "bf16", "bf16-nomaster"])
def test_sharded_update_on_two_handles_equals_whole_step(mi):
    from scratch_gpt_step_train_b300.gpt2 import GPT2
    mode = _gpu_modes()[mi]
    a = GPT2(**CFG, seed=3, mode=mode)
    r = [GPT2(**CFG, seed=3, mode=mode) for _ in range(2)]
    n = a.n
    bounds = shard_bounds(n, 2)
    for step in range(3):
        # the reference: one micro-batch, count 1
        a.zero_grad()
        _micro(a, 40 + step)
        na = a.adamw_step(**HP)
        # two "ranks" with the same micro-batch: the summed gradient is exactly
        # twice it and the count is 2, so the update is the same to the bit
        for h in r:
            h.zero_grad()
            _micro(h, 40 + step)
        g0, g1 = r[0].grads_tensor(), r[1].grads_tensor()
        s = g0 + g1
        g0.copy_(s)
        g1.copy_(s)
        norms = []
        for h, (lo, hi) in zip(r, bounds):
            h.set_grad_count(h.grad_count() * 2)
            norms.append(h.adamw_step_shard(lo, hi, **HP))
        for i, (lo, hi) in enumerate(bounds):
            for dst, src in zip(r[1 - i].param_tensors(), r[i].param_tensors()):
                if src is not None:
                    dst[lo:hi].copy_(src[lo:hi])
        torch.cuda.synchronize()
        assert norms[0] == norms[1] == na
    pa = a.get_params()
    ma, va, ta = a.get_opt_state()
    for i, h in enumerate(r):
        assert np.array_equal(h.get_params(), pa)
        m, v, t = h.get_opt_state()
        lo, hi = bounds[i]
        assert t == ta == 3
        assert np.array_equal(m[lo:hi], ma[lo:hi]) and np.array_equal(v[lo:hi], va[lo:hi])
    if mi > 0:  # the bf16 compute copies too
        pb = a.param_tensors()[1]
        for h in r:
            assert torch.equal(h.param_tensors()[1].view(torch.int16), pb.view(torch.int16))


@pytest.mark.gpu
def test_data_parallel_nccl_one_rank_equals_plain_step():
    from scratch_gpt_step_train_b300.gpt2 import BF16, GPT2
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0,
                            world_size=1, device_id=torch.device("cuda:0"))
    try:
        a = GPT2(**CFG, seed=9, mode=BF16)
        b = GPT2(**CFG, seed=9, mode=BF16)
        dp = DataParallel(b)
        for step in range(3):
            for h in (a, b):
                h.zero_grad()
                _micro(h, 70 + 2 * step)
                _micro(h, 71 + 2 * step)
            na = a.adamw_step(**HP)
            nb = dp.step(**HP)
            assert na == nb
        torch.cuda.synchronize()
        assert np.array_equal(a.get_params(), b.get_params())
    finally:
        dist.destroy_process_group()


def _slice_adamw_oracle(w, m, v, g, lo, hi, sc, t, offsets, hp):
    """the oracle's AdamW over the canonical slice [lo, hi), tensor by tensor
    (decay on the 2-D weights only)"""
    from oracle.pyoracle import DECAYED, TENSOR_NAMES, Ops
    ops = Ops("double")
    w, m, v = (np.array(a, np.float64) for a in (w, m, v))
    for name in TENSOR_NAMES:
        a, b = max(lo, offsets[name].start), min(hi, offsets[name].stop)
        if a >= b:
            continue
        i, j = a - lo, b - lo
        w[i:j], m[i:j], v[i:j] = ops.adamw(w[i:j], m[i:j], v[i:j], g[a:b], sc, hp["lr"],
                                           hp["b1"], hp["b2"], hp["eps"], hp["wd"],
                                           name in DECAYED, t)
    return w, m, v


@pytest.mark.gpu
@pytest.mark.parametrize("mi", [0, 1], ids=["fp32", "bf16"])
def test_zero1_shard_handles_against_the_oracle(mi):
    """Two ZeRO-1 handles on one GPU, each holding the moments (and in bf16
    mode the fp32 master) of its half only: the workspace shrinks by the
    slices it does not hold; over three steps each rank's update of its slice
    (master, m, v) matches the oracle's AdamW applied to the same summed
    gradient, state and clip scale at rel 1e-4, the bf16 copy of the slice is
    the master rounded to nearest even, and after the gather both handles hold
    the same parameters"""
    from oracle.pyoracle import Model
    from parity import assert_close
    from scratch_gpt_step_train_b300.gpt2 import GPT2, workspace_bytes
    mode = _gpu_modes()[mi]
    full = workspace_bytes(**CFG, mode=mode)
    r = []
    probe = GPT2(**CFG, seed=3, mode=mode)
    n = probe.n
    bounds = shard_bounds(n, 2)
    probe.close()
    for lo, hi in bounds:
        saved = (n - (hi - lo)) * (12 if mi else 8)  # m, v (+ the fp32 master in bf16 mode)
        assert abs(full - workspace_bytes(**CFG, mode=mode, shard=(lo, hi)) - saved) < 1024
        r.append(GPT2(**CFG, seed=3, mode=mode, shard=(lo, hi)))
    offsets = Model(**CFG, seed=3).tensor_slices()
    count = torch.tensor([2], dtype=torch.int32, device="cuda")
    for step in range(3):
        for h in r:
            h.zero_grad()
            _micro(h, 40 + step)
        s = r[0].grads_tensor() + r[1].grads_tensor()
        for h in r:
            h.grads_tensor().copy_(s)
        torch.cuda.synchronize()
        gsum = s.double().cpu().numpy()
        norm = np.linalg.norm(gsum) / 2
        sc = 0.5 * (HP["clip"] / norm if norm > HP["clip"] else 1.0)
        before = [(h.get_shard_master(), *h.get_opt_state()[:2]) for h in r]
        for h, (lo, hi), (w0, m0, v0) in zip(r, bounds, before):
            h.set_grad_count_device(count)
            ng = h.adamw_step_shard(lo, hi, **HP)
            assert abs(ng - norm) <= 1e-5 * norm
            w1, m1, v1 = _slice_adamw_oracle(w0, m0, v0, gsum, lo, hi, sc, step + 1, offsets, HP)
            m, v, t = h.get_opt_state()
            assert t == step + 1 and m.size == hi - lo
            assert_close(h.get_shard_master(), w1, 1e-4, f"step {step} master [{lo}, {hi})")
            assert_close(m, m1, 1e-4, f"step {step} m")
            assert_close(v, v1, 1e-4, f"step {step} v")
            assert h.grad_count() == 1  # the device count served one update, the host's is kept
            if mi:
                bf = h.param_tensors()[1][lo:hi].float().cpu()
                rne = torch.from_numpy(h.get_shard_master()).to(torch.bfloat16).float()
                assert torch.equal(bf, rne)
        # the all-gather: each handle's slice into the other
        for i, (lo, hi) in enumerate(bounds):
            src = r[i].param_tensors()[1 if mi else 0]
            r[1 - i].param_tensors()[1 if mi else 0][lo:hi].copy_(src[lo:hi])
    torch.cuda.synchronize()
    assert np.array_equal(r[0].get_params(), r[1].get_params())
    with pytest.raises(Exception):
        r[0].adamw_step(**HP)  # a sharded handle updates its slice only


def test_shard_step_argument_errors_are_host_checks():
    """the C-ABI rejects unaligned or out-of-range slices before any launch
    (checked here through a null handle, which needs no GPU)"""
    from scratch_gpt_step_train_b300.gpt2 import lib
    L = lib()
    assert L.gpt2_adamw_step_shard(None, 0, 4, 1e-3, 0.9, 0.95, 1e-8, 0.1, 1.0, None) == -1
    assert L.gpt2_set_grad_count(None, 2) == -1
    assert L.gpt2_set_grad_count_device(None, None) == -1
    assert L.gpt2_create_shard(None, 2, 2, 64, 100, 16, 2, 0, 0, 0, 4, None, 0, None) == -1


def test_zero1_workspace_sizes():
    """a rank's workspace drops the moments (and in bf16 mode the master) of
    the slices it does not hold; bad slices are rejected with size 0"""
    from scratch_gpt_step_train_b300.gpt2 import BF16, FP32, workspace_bytes
    shape = dict(L=12, H=12, C=768, V=50257, T=1024, B=16)
    n = 124475904
    for mode, per in ((FP32, 8), (BF16, 12)):
        full = workspace_bytes(**shape, mode=mode)
        for world in (2, 8):
            lo, hi = shard_bounds(n, world)[world - 1]
            d = full - workspace_bytes(**shape, mode=mode, shard=(lo, hi))
            assert abs(d - per * (n - (hi - lo))) < 1024
    assert workspace_bytes(**shape, mode=BF16, shard=(2, 64)) == 0  # unaligned
    assert workspace_bytes(**shape, mode=BF16, shard=(64, 0)) == 0  # empty the wrong way
    assert workspace_bytes(**shape, mode=BF16, shard=(0, n + 4)) == 0  # beyond N
