"""Data-parallel training step over torch.distributed, the optimizer state
sharded across the ranks (ZeRO-1) -- "Karpathy reproduces GPT-2 (1.6B) in
llm.c", "Training": one process per GPU, gradients averaged over the ranks,
optimizer state sharded (-z 1).

One process per GPU, each with its own GPT2 handle of the same shape and
parameters, created for its own slice of the canonical parameter vector
(GPT2(..., shard=shard_bounds(n, world)[rank])): the handle then holds the
AdamW moments, and in bf16 mode the fp32 master, of that slice alone.  A step
is: every rank runs its micro-batches (forward + backward); then
DataParallel.step()
  1. sums the gradient vectors of all ranks in place (all-reduce),
  2. sums the ranks' micro-batch counts into a device word (a one-element
     all-reduce) that the update reads on the device (no host round trip),
  3. lets every rank update its own slice (the clip and the norm come from
     the whole summed gradient, identical on every rank),
  4. gathers the updated slices of the parameters the forward reads (the bf16
     copy in bf16 mode, the fp32 parameters in fp32 mode) into every rank
     (one all-gather).
All of it is enqueued on the handle's stream; with NCCL the collectives run on
the GPU.  The class needs only the handle's interface below, so it runs as
well on CPU tensors with gloo (which is how its logic is tested without
several GPUs).

Model interface: .n, .shard (its [lo, hi), (0, n) for an unsharded handle),
grads_tensor(), param_tensors() -> (fp32 parameters or None, bf16 copy or
None), grad_count(), set_grad_count_device(int32 tensor), adamw_step_shard(lo,
hi, lr, b1, b2, eps, wd, clip) -> gradient norm.

After a step that fails (a non-finite norm raises on every rank alike) the
gradient buffer holds the all-reduced sum: call zero_grad before the next
micro-batches.
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
        lo, hi = self.bounds[self.rank]
        shard = tuple(getattr(model, "shard", (0, model.n)))
        if shard != (0, model.n) and shard != (lo, hi):
            raise ValueError(f"the handle holds the slice {shard}; rank {self.rank} of "
                             f"{self.world} updates {(lo, hi)}")
        self.grads = model.grads_tensor()
        if self.grads is None:
            raise ValueError("the model's gradient buffer is not addressable as a tensor")
        master, bf16 = model.param_tensors()
        # the parameters the forward reads: the bf16 copy, else the fp32 ones
        self.params = bf16 if bf16 is not None else master
        if self.params is None:
            raise ValueError("the model's parameters are not addressable as a tensor")
        chunk = self.bounds[0][1] - self.bounds[0][0]
        dev = self.params.device
        self.send = torch.zeros(chunk, dtype=self.params.dtype, device=dev)
        self.recv = torch.empty(self.world * chunk, dtype=self.params.dtype, device=dev)
        self.count = torch.zeros(1, dtype=torch.int32, device=self.grads.device)

    def step(self, lr, b1=0.9, b2=0.95, eps=1e-8, wd=0.1, clip=1.0):
        """all-reduce the gradients and the micro-batch count, update this
        rank's slice, gather the slices; returns the global gradient norm"""
        s = getattr(self.model, "stream", None)
        with torch.cuda.stream(s) if s is not None else nullcontext():
            dist.all_reduce(self.grads, op=dist.ReduceOp.SUM, group=self.group)
            # the divisor: micro-batches summed over the ranks (they may differ)
            self.count.fill_(self.model.grad_count())
            dist.all_reduce(self.count, op=dist.ReduceOp.SUM, group=self.group)
            self.model.set_grad_count_device(self.count)
            lo, hi = self.bounds[self.rank]
            norm = self.model.adamw_step_shard(lo, hi, lr, b1, b2, eps, wd, clip)
            # rank r's slice lands at r * chunk = its canonical offset
            self.send[:hi - lo].copy_(self.params[lo:hi])
            dist.all_gather_into_tensor(self.recv, self.send, group=self.group)
            self.params.copy_(self.recv[:self.model.n])
        return norm
