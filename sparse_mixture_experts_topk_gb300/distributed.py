"""Load-balancing loss over a data-parallel batch.

When the tokens of one batch are split across ranks, each rank's router sees
only its shard, so the per-expert statistics of the load-balancing loss must
be combined before the loss is formed: the Qwen2-MoE code walkthrough
(jsqmd.com), section 5.2 (the multi-GPU aux-loss bug), all-reduces the mean
probabilities and the selection frequencies across ranks.  Here the raw sums
are all-reduced instead of the means, which gives the exact full-batch
statistics also when the ranks hold different numbers of tokens; the loss is
then formed from them by the library's ``moe_aux_loss`` kernel, like the
single-GPU loss.

This is the only exchange the layer has; the layer itself needs none (every
token is routed and computed on its own rank).
"""
from __future__ import annotations


def reduce_aux_stats(psum, count, tokens: int, group=None):
    """All-reduce (sum) this rank's load-balancing statistics over ``group``.

    psum   [E] per-expert sum of router probabilities over this rank's tokens
           (``moe_router_topk``'s ``psum`` output), any float tensor
    count  [E] slots routed to each expert on this rank, before capacity drops
    tokens this rank's token count
    Returns ``(psum_total [E] float64, count_total [E] int64, tokens_total)``
    as CPU tensors and an int, identical on every rank.  Without an
    initialised process group the local values are returned."""
    import torch
    import torch.distributed as dist

    E = psum.numel()
    stats = torch.cat([psum.detach().to("cpu", torch.float64).reshape(-1),
                       count.detach().to("cpu", torch.float64).reshape(-1),
                       torch.tensor([float(tokens)], dtype=torch.float64)])
    if dist.is_available() and dist.is_initialized():
        if dist.get_backend(group) == "nccl":
            s = stats.to(torch.device("cuda", torch.cuda.current_device()))
            dist.all_reduce(s, op=dist.ReduceOp.SUM, group=group)
            stats = s.cpu()
        else:
            dist.all_reduce(stats, op=dist.ReduceOp.SUM, group=group)
    # counts and tokens are integers; their fp64 sums are exact below 2^53
    return stats[:E].clone(), stats[E:2 * E].round().to(torch.int64), int(round(float(stats[2 * E])))


def global_aux_loss(psum, count, tokens: int, k: int, group=None, stream=None):
    """``E * sum_i f_i P_i`` over the tokens of every rank in ``group``: the
    statistics are all-reduced (``reduce_aux_stats``), then the loss is formed
    on the current CUDA device by ``moe_aux_loss``.  Returns a one-element fp32
    device tensor, the same on every rank."""
    import torch
    import sparse_mixture_experts_topk_gb300 as moe

    ps, cnt, n = reduce_aux_stats(psum, count, tokens, group)
    E = ps.numel()
    dev = torch.device("cuda", torch.cuda.current_device())
    ps_d = ps.to(torch.float32).to(dev)
    cnt_d = cnt.to(torch.int32).to(dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    # H and F do not enter the loss; 8 is the smallest valid width
    d = moe.make_desc(n, 8, E, k, 8)
    moe.moe_aux_loss(d, ps_d, cnt_d, loss, stream)
    return loss
