"""Data-parallel load-balancing loss.  With two gloo ranks on the CPU: the
sharded statistics, all-reduced, are the full batch's statistics and give the
oracle's full-batch loss; a rank that dies before the collective makes the
survivor fail with a timeout instead of hanging.  On the GPU: the loss formed
from the reduced statistics by the library's kernel matches the oracle."""
import datetime
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _shard_stats(rank, world, T, E, k):
    from oracle import moe_oracle as O
    rng = np.random.default_rng(11)
    l = rng.standard_normal((T, E)) * 1.5 + np.linspace(1, 0, E)[None, :]
    bounds = [0, 37, T] if world == 2 else [0, T]        # unequal shards
    lo, hi = bounds[rank], bounds[rank + 1]
    ids, w, p = O.route(l[lo:hi], k)
    count = np.bincount(ids.reshape(-1), minlength=E)
    full_ids, _, full_p = O.route(l, k)
    full = O.aux_loss(full_p, np.bincount(full_ids.reshape(-1), minlength=E), k)
    return p.sum(0), count, hi - lo, full


def _worker(rank, world, port, q, die):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=10))
    from sparse_mixture_experts_topk_gb300.distributed import reduce_aux_stats
    from oracle import moe_oracle as O
    T, E, k = 100, 8, 2
    psum, count, n, full = _shard_stats(rank, world, T, E, k)
    if die and rank == 1:
        os._exit(0)                      # leaves between steps, before the collective
    try:
        ps, cnt, tot = reduce_aux_stats(torch.from_numpy(psum), torch.from_numpy(count), n)
        L = O.aux_loss_from_psum(ps.numpy(), cnt.numpy(), tot, k)
        q.put((rank, "ok", float(L), full, tot, cnt.tolist()))
    except Exception as ex:              # the survivor's collective must fail, not hang
        q.put((rank, "error", type(ex).__name__, full, None, None))
    try:
        dist.destroy_process_group()
    except Exception:
        pass


def _run(world, die):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q, die)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(60)
        assert not p.is_alive()
    out = []
    while not q.empty():
        out.append(q.get())
    return out


def test_sharded_aux_equals_full_batch():
    res = _run(2, die=False)
    assert len(res) == 2
    _, _, _, full_count = _full_stats(100, 8, 2)
    for rank, status, L, full, tot, cnt in res:
        assert status == "ok"
        assert tot == 100 and cnt == full_count.tolist()
        assert L == pytest.approx(full, rel=1e-12)


def _full_stats(T, E, k):
    from oracle import moe_oracle as O
    rng = np.random.default_rng(11)
    l = rng.standard_normal((T, E)) * 1.5 + np.linspace(1, 0, E)[None, :]
    ids, _, p = O.route(l, k)
    return l, p, ids, np.bincount(ids.reshape(-1), minlength=E)


def test_single_process_without_group_is_local_stats():
    from sparse_mixture_experts_topk_gb300.distributed import reduce_aux_stats
    psum, count, n, full = _shard_stats(0, 1, 100, 8, 2)
    ps, cnt, tot = reduce_aux_stats(torch.from_numpy(psum), torch.from_numpy(count), n)
    assert tot == n and np.array_equal(cnt.numpy(), count)
    assert np.array_equal(ps.numpy(), psum)


def test_dead_rank_gives_error_not_hang():
    res = _run(2, die=True)
    assert len(res) == 1
    rank, status, what = res[0][:3]
    assert rank == 0 and status == "error"


@pytest.mark.gpu
def test_global_aux_loss_on_device_matches_oracle():
    """One process, no group: the statistics go to the library's loss kernel."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mixture_experts_topk_gb300 import build
    from sparse_mixture_experts_topk_gb300.distributed import global_aux_loss
    build.build()
    psum, count, n, full = _shard_stats(0, 1, 100, 8, 2)
    L = global_aux_loss(torch.from_numpy(psum), torch.from_numpy(count), n, 2)
    torch.cuda.synchronize()
    assert L.is_cuda and float(L.item()) == pytest.approx(full, rel=1e-5)
