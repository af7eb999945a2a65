"""Load-balancing loss over a data-parallel batch.

When the tokens of one batch are split across ranks, each rank's router sees
only its shard, so the per-expert statistics of the load-balancing loss must
be combined before the loss is formed: the Qwen2-MoE code walkthrough
(jsqmd.com), section 5.2 (the multi-GPU aux-loss bug), all-reduces the mean
probabilities and the selection frequencies across ranks.  Here the raw sums
are all-reduced instead of the means, which gives the exact full-batch loss
also when the ranks hold different numbers of tokens.

This is the only exchange the layer has; the layer itself needs none (every
token is routed and computed on its own rank).
"""
from __future__ import annotations


def global_aux_loss(psum, count, tokens: int, k: int, group=None):
    """``E * sum_i f_i P_i`` over the tokens of every rank in ``group``.

    psum   [E] per-expert sum of router probabilities over this rank's tokens
           (``moe_router_topk``'s ``psum`` output), any float tensor
    count  [E] slots routed to each expert on this rank, before capacity drops
    tokens this rank's token count
    Returns a float64 scalar tensor, identical on every rank."""
    import torch
    import torch.distributed as dist

    E = psum.numel()
    stats = torch.cat([psum.detach().to("cpu", torch.float64).reshape(-1),
                       count.detach().to("cpu", torch.float64).reshape(-1),
                       torch.tensor([float(tokens)], dtype=torch.float64)])
    if dist.is_available() and dist.is_initialized():
        backend = dist.get_backend(group)
        if backend == "nccl":
            dev = torch.device("cuda", torch.cuda.current_device())
            s = stats.to(dev)
            dist.all_reduce(s, op=dist.ReduceOp.SUM, group=group)
            stats = s.cpu()
        else:
            dist.all_reduce(stats, op=dist.ReduceOp.SUM, group=group)
    P = stats[:E] / stats[2 * E]
    f = stats[E:2 * E] / (stats[2 * E] * k)
    return E * (f * P).sum()
