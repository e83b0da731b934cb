"""Data-parallel training step over torch.distributed, the optimizer update
sharded across the ranks (ZeRO-1 style) -- "Karpathy reproduces GPT-2 (1.6B)
in llm.c", "Training": one process per GPU, gradients averaged over the ranks.

One process per GPU, each with its own GPT2 handle of the same shape and
parameters.  A step is: every rank runs its micro-batches (forward +
backward); then DataParallel.step() sums the gradient vectors of all ranks in
place (all-reduce), sets the divisor to the micro-batch count summed over the
ranks, lets every
rank update its own slice of the canonical parameter vector (the clip and the
norm from the whole summed gradient, identical on every rank), and exchanges
the updated slices (each rank broadcasts its slice of the fp32 master and of
the bf16 copy).  With NCCL the collectives run on the GPU; the class only
needs the handle's interface below, so it runs as well on CPU tensors with
gloo (which is how its logic is tested without several GPUs).

Model interface: .n, grads_tensor(), param_tensors() -> (master or None,
bf16 or None), grad_count(), set_grad_count(c), adamw_step_shard(lo, hi, lr,
b1, b2, eps, wd, clip) -> gradient norm.
"""
from contextlib import nullcontext

import torch
import torch.distributed as dist


def shard_bounds(n, world, align=64):
    """[lo, hi) slices of range(n), one per rank: equal chunks (a multiple of
    `align` elements, so that every slice starts 16-byte aligned), the last
    ones shorter or empty"""
    chunk = -(-n // world)
    chunk = -(-chunk // align) * align
    return [(min(n, r * chunk), min(n, (r + 1) * chunk)) for r in range(world)]


class DataParallel:
    def __init__(self, model, group=None):
        self.model = model
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.bounds = shard_bounds(model.n, self.world)
        self.grads = model.grads_tensor()
        if self.grads is None:
            raise ValueError("the model's gradient buffer is not addressable as a tensor")
        self.params = [t for t in model.param_tensors() if t is not None]

    def _global(self, r):
        return r if self.group is None else dist.get_global_rank(self.group, r)

    def step(self, lr, b1=0.9, b2=0.95, eps=1e-8, wd=0.1, clip=1.0):
        """all-reduce the gradients, update this rank's slice, exchange the
        slices; returns the global gradient norm"""
        # the collectives are ordered after the handle's kernels on its stream
        s = getattr(self.model, "stream", None)
        with torch.cuda.stream(s) if s is not None else nullcontext():
            dist.all_reduce(self.grads, op=dist.ReduceOp.SUM, group=self.group)
            # the divisor: micro-batches summed over the ranks (they may differ)
            count = torch.tensor([self.model.grad_count()], dtype=torch.int64,
                                 device=self.grads.device)
            dist.all_reduce(count, op=dist.ReduceOp.SUM, group=self.group)
            self.model.set_grad_count(int(count.item()))
            lo, hi = self.bounds[self.rank]
            norm = self.model.adamw_step_shard(lo, hi, lr, b1, b2, eps, wd, clip)
            for r, (a, b) in enumerate(self.bounds):
                if b > a:
                    for t in self.params:
                        dist.broadcast(t[a:b], src=self._global(r), group=self.group)
        return norm
