"""The multi-process host path on CPU: two gloo ranks, rows sharded contiguously.

Rows are independent, so each rank's shard computed alone and gathered must
equal the whole batch computed in one process (here with the oracle, on the CPU),
and the timing reduction must return the slowest rank's value.
"""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

from top_kl_distill_gb300 import dist as D  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    from oracle import vloss_oracle as O
    from top_kl_distill_gb300 import workloads as W
    try:
        dist.init_process_group("gloo", rank=rank, world_size=ws)
        assert D.world() == (ws, rank, rank)
        w = W.WORKLOADS["ce_tiny"]
        r0, r1, ls, le = D.window_shard(w.ntok, rank, ws, w.loss_start, w.loss_end)
        assert (r0, r1) == D.shard(w.ntok, rank, ws)
        x = W.logits(w, r0, r1, threads=1)
        lab = W.labels(w, r0, r1)
        loss, lse, grad, local_mean = O.ce_fused(x, lab, ls, le, w.scale)
        gmean = D.global_window_mean(torch.tensor([local_mean], dtype=torch.float32), le - ls,
                                     w.loss_end - w.loss_start)
        mine = torch.from_numpy(np.concatenate([loss, lse, grad.ravel()]).astype(np.float64))
        sizes = [torch.zeros(1, dtype=torch.int64) for _ in range(ws)]
        dist.all_gather(sizes, torch.tensor([mine.numel()]))
        big = int(max(int(n) for n in sizes))          # gloo gathers equal sizes: pad, then trim
        padded = torch.zeros(big, dtype=torch.float64)
        padded[:mine.numel()] = mine
        parts = [torch.zeros(big, dtype=torch.float64) for _ in sizes]
        dist.all_gather(parts, padded)
        parts = [p[:int(n)] for p, n in zip(parts, sizes)]
        slowest = D.max_over_ranks(1.5 + rank, "cpu")
        dist.barrier()
        q.put((rank, [p.numpy() for p in parts], slowest, float(gmean[0])))
    except Exception as e:  # report to the parent instead of hanging it
        q.put((rank, repr(e), None, None))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


def test_shard_bounds():
    for ntok in (0, 1, 7, 64, 1000):
        for ws in (1, 2, 3, 8):
            spans = [D.shard(ntok, r, ws) for r in range(ws)]
            assert spans[0][0] == 0 and spans[-1][1] == ntok
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        D.shard(10, 2, 2)


@pytest.mark.parametrize("ws", [2, 3])
def test_gloo_ranks_match_one_process(ws):
    """Each rank's shard computed alone and gathered equals the batch computed in one
    process; the window mean from the ranks' part means (one all-reduce) equals the
    batch's mean; the timing reduction returns the slowest rank."""
    from oracle import vloss_oracle as O
    from top_kl_distill_gb300 import workloads as W
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(ws):
        rank, parts, slowest, gmean = q.get(timeout=120)
        assert slowest is not None, parts
        got[rank] = (parts, slowest, gmean)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w = W.WORKLOADS["ce_tiny"]
    x = W.logits(w, threads=1)
    loss, lse, grad, mean = O.ce_fused(x, W.labels(w), w.loss_start, w.loss_end, w.scale)
    for rank in range(ws):
        parts, slowest, gmean = got[rank]
        assert slowest == 1.5 + (ws - 1)
        assert abs(gmean - mean) <= 1e-6 * abs(mean), (gmean, mean)   # fp32 part means, as a device gives
        r = [D.shard(w.ntok, i, ws) for i in range(ws)]
        for i, (r0, r1) in enumerate(r):
            n = r1 - r0
            p = parts[i]
            assert np.array_equal(p[:n], loss[r0:r1])
            assert np.array_equal(p[n:2 * n], lse[r0:r1])
            assert np.array_equal(p[2 * n:].reshape(n, w.V), grad[r0:r1])


def test_window_shard_covers_the_window_once():
    for ntok, ls, le in [(64, 8, 64), (10, 0, 0), (7, 3, 4), (1000, 0, 1000)]:
        for ws in (1, 2, 3, 5, 8):
            total = 0
            for rank in range(ws):
                r0, r1, a, b = D.window_shard(ntok, rank, ws, ls, le)
                assert 0 <= a <= b <= r1 - r0
                assert (r0 + a, r0 + b) == (max(ls, r0), max(min(le, r1), max(ls, r0))) or a == b
                total += b - a
            assert total == le - ls
    with pytest.raises(ValueError):
        D.window_shard(10, 0, 2, 5, 11)


def test_global_mean_alone_and_empty_window():
    t = torch.tensor([2.5])
    assert float(D.global_window_mean(t, 4, 4)[0]) == 2.5     # not distributed: the local mean itself
    assert float(D.global_window_mean(t, 0, 0)[0]) == 0.0
