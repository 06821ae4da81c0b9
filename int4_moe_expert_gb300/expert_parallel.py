"""Expert parallelism: one MoE layer's routed experts split over several GPUs.

The pages' tiered residency (reader.mx, "25GB 内存上运行 GLM 5.2 744B",
section 13 "五级专家驻留") keeps disjoint expert sets on the GPUs of one tier.
Here rank r of W owns the routed experts e with r*E//W <= e < (r+1)*E//W
(the rule the library applies to a handle made with ep_size=W, ep_rank=r;
``include/moe.h``, "Expert parallelism").  Every rank holds the router and
computes the whole selection, so the ranks agree on it without an exchange;
each rank's call writes its partial output

    y_r = sum over the top-K slots whose expert rank r owns of w_k d_k
          (+ the shared expert, and x with the pre-norm residual, on rank 0),

and the layer's y is the sum of the partials: one all-reduce of y[T, H], the
only collective on the path.  This module is host plumbing around the
library: which experts' weights a rank loads, the handle, and the reduction
through ``torch.distributed`` (NCCL between GPUs, gloo on CPU).
"""
from __future__ import annotations

from . import MoeLayer, make_config


def owned_range(n_experts: int, ep_size: int, ep_rank: int) -> tuple[int, int]:
    """[lo, hi): the routed experts rank ep_rank of ep_size computes."""
    if not (1 <= ep_size <= n_experts and 0 <= ep_rank < ep_size):
        raise ValueError(f"ep_size={ep_size}, ep_rank={ep_rank} with {n_experts} experts")
    return ep_rank * n_experts // ep_size, (ep_rank + 1) * n_experts // ep_size


def reduce_partials(y, group=None):
    """Sum the ranks' partial outputs in place (every rank ends with the layer's y)."""
    import torch.distributed as dist
    dist.all_reduce(y, op=dist.ReduceOp.SUM, group=group)
    return y


class ExpertParallelLayer:
    """This rank's part of a layer: the router, its own routed experts, and the
    shared expert on rank 0.  ``slabs``/``scales`` hold either all E experts or
    only this rank's (hi - lo rows); only the owned rows go to the device."""

    def __init__(self, cfg_kwargs: dict, router_w, router_b, slabs, scales, sh_slab=None,
                 sh_scale=None, *, ep_size: int, ep_rank: int, max_tokens: int = 1, device=None,
                 group=None):
        E = cfg_kwargs["E"]
        self.lo, self.hi = owned_range(E, ep_size, ep_rank)
        self.ep_size, self.ep_rank, self.group = ep_size, ep_rank, group
        n_own = self.hi - self.lo
        if len(slabs) == E:
            slabs, scales = slabs[self.lo:self.hi], scales[self.lo:self.hi]
        elif len(slabs) != n_own:
            raise ValueError(f"slabs: {len(slabs)} rows, need {E} or this rank's {n_own}")
        rows = [e - self.lo if self.lo <= e < self.hi else None for e in range(E)]
        cfg = make_config(**cfg_kwargs, ep_size=ep_size, ep_rank=ep_rank)
        shared = ep_rank == 0 and cfg.n_shared
        self.layer = MoeLayer(cfg, router_w, router_b, slabs, scales, sh_slab if shared else None,
                              sh_scale if shared else None, max_tokens=max_tokens, device=device,
                              expert_rows=rows)
        self.handle = self.layer.handle

    def forward_partial(self, x, y=None, stream=None):
        """This rank's partial output y_r (no collective)."""
        return self.layer.forward(x, y, stream)

    def forward(self, x, y=None, stream=None):
        """The layer's output: this rank's partial, then the all-reduce over the group."""
        return reduce_partials(self.forward_partial(x, y, stream), self.group)

    def close(self):
        self.layer.close()
