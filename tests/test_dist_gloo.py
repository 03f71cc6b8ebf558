"""Multi-rank paths on CPU with gloo ranks: bench.py's timing reduction (max elapsed over
ranks, sum of units), and data parallelism over one optimizer step's rows (each rank's row
block scaled by the step's global N, the step result reduced across ranks) against the
unsharded step."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, lr = bench.dist_env()
    bench.barrier(w)
    el, units = bench.reduce_timing(1.0 + rank, 100.0 * (rank + 1), w)
    q.put((r, w, el, units))
    dist.destroy_process_group()


def test_reduce_timing_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out == [(0, 2, 2.0, 300.0), (1, 2, 2.0, 300.0)]


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_timing(3.5, 42.0, 1) == (3.5, 42.0)


def _dp_worker(rank, world, port, q, name="tiny"):
    # each rank plans the whole batch, runs (with the oracle, on the CPU) its exec-order token
    # ranges of every optimizer step (dp_exec_ranges), scaled by the step's global N, and
    # reduces the step result; the reduced result must be the unsharded step's
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import math
    import numpy as np
    from oracle import advantage as OA
    from oracle import loss as OL
    from rl_post_token_gb300 import step as S
    from rl_post_token_gb300 import workloads as W

    if name == "compaction":  # 4/8/4 rows padded for `world` GPUs, short rows, small V
        wl = W.make_workload("compaction", V=512, row_tokens=16, seed=5)
        wl.plan = dict(wl.plan, n_gpus=world, micro=1)
    else:
        wl = W.make_workload("tiny", rows=24, seed=5, mini=12, micro=4)
    z = W.logits_to_host(W.make_logits(wl, "cpu"))
    adv = OA.broadcast_to_tokens(OA.group_advantage(wl.rewards, wl.group_size, np.float32(1e-6), True),
                                 wl.row_rollout, wl.row_len)
    logp = OL.loss_fwd_bwd(z, wl.target, None, adv, wl.mask, wl.eps, want_grad=False)["logp_tok"]
    old = logp + wl.old_noise
    bp = S.plan_batch(wl.plan, wl.row_len, wl.row_valid, wl.seg_counts)
    # exec-order inputs: a padding row reads its source row's inputs with the mask off
    if bp.tok_src is None:
        src = np.arange(z.shape[0])
        real = np.ones(z.shape[0], bool)
    else:
        ts = np.asarray(bp.tok_src)
        real = ts >= 0
        src = np.where(real, ts, -1 - ts)
    zx, yx, ox, ax = z[src], wl.target[src], old[src], adv[src]
    mx = (wl.mask[src] != 0) & real
    out = []
    for s in range(bp.n_steps):
        c0, c1 = int(bp.plan["step_chunk_off"][s]), int(bp.plan["step_chunk_off"][s + 1])
        a, b = int(bp.exec_tok_off[c0]), int(bp.exec_tok_off[c1])
        N = int(mx[a:b].sum())
        idx = np.concatenate([np.arange(t0, t1) for t0, t1 in S.dp_exec_ranges(bp, s, rank, world)] or
                             [np.zeros(0, np.int64)]).astype(np.int64)
        mine = OL.loss_fwd_bwd(zx[idx], yx[idx], ox[idx], ax[idx], mx[idx], wl.eps, 1.0 / max(N, 1))
        res = dict(loss_sum=math.fsum(mine["loss_tok"]), n_valid=int(mx[idx].sum()),
                   n_clipped=int((mine["clipped"] & mx[idx]).sum()), n_nonfinite=0, n_tokens=int(idx.size),
                   status=0, kernel_flags=0)
        got = S.dp_allreduce_step_result(res, N)
        full = OL.loss_fwd_bwd(zx[a:b], yx[a:b], ox[a:b], ax[a:b], mx[a:b], wl.eps, 1.0 / max(N, 1))
        want = OL.finish_step(full["loss_tok"], mx[a:b], full["clipped"])
        out.append((got, want, N, b - a))
    q.put((rank, out))
    dist.destroy_process_group()


@pytest.mark.parametrize("name, world", [("tiny", 2), ("tiny", 3), ("compaction", 2)])
def test_data_parallel_step_reduces_to_the_unsharded_step(name, world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_dp_worker, args=(r, world, port, q, name)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sorted(res) == list(range(world))
    for r in range(world):
        assert len(res[r]) == (2 if name == "tiny" else 1)  # optimizer steps
        for k, (got, want, N, T) in enumerate(res[r]):
            assert got == res[0][k][0]  # identical on every rank
            assert got["n_valid"] == want["n_valid"] == N
            assert got["n_clipped"] == want["n_clipped"] and got["n_tokens"] == T
            assert got["clipfrac"] == want["clipfrac"]
            assert abs(got["loss"] - want["loss"]) <= 1e-12 * max(abs(want["loss_sum"]) / max(N, 1), 1e-300)
            assert got["status"] == 0 and got["kernel_flags"] == 0


def test_dp_row_blocks_and_combine():
    from rl_post_token_gb300 import _lib
    from rl_post_token_gb300 import step as S
    for n in range(0, 12):
        for world in range(1, 5):
            blocks = [S.dp_row_block(n, r, world) for r in range(world)]
            assert blocks[0][0] == 0 and blocks[-1][1] == n
            assert all(blocks[i][1] == blocks[i + 1][0] for i in range(world - 1))
            sizes = [b - a for a, b in blocks]
            assert max(sizes) - min(sizes) <= 1 and sizes == sorted(sizes, reverse=True)
    with pytest.raises(ValueError):
        S.dp_row_block(4, 2, 2)
    base = dict(loss_sum=1.5, n_valid=3, n_clipped=1, n_nonfinite=0, n_tokens=4, status=0, kernel_flags=0)
    r = S.combine_step_results([base, dict(base, loss_sum=-0.5, n_valid=2)], divisor=5)
    assert r["loss"] == 1.0 / 5 and r["n_valid"] == 5 and r["clipfrac"] == 2 / 5 and r["status"] == 0
    skip = dict(base, status=_lib.STEP_SKIPPED_NONFINITE, n_nonfinite=1, kernel_flags=2)
    err = dict(base, status=_lib.ERR_N_MISMATCH, kernel_flags=4)
    assert S.combine_step_results([base, skip], 6)["status"] == _lib.STEP_SKIPPED_NONFINITE
    both = S.combine_step_results([skip, err, dict(base, status=_lib.ERR_KERNEL)], 6)
    assert both["status"] == _lib.ERR_N_MISMATCH and both["kernel_flags"] == 6 and both["n_nonfinite"] == 1
    assert S.combine_step_results([], 0)["loss"] == 0.0


@pytest.mark.parametrize("name, world", [("tiny", 2), ("qwen_step", 3), ("dynamic", 4), ("compaction", 4),
                                         ("compaction", 2)])
def test_dp_exec_ranges_partition_every_step(name, world):
    # the ranks' ranges cover each optimizer step's exec tokens exactly once; a compaction plan
    # gives each rank the rows its row_gpu slots name (each padded group split evenly)
    import numpy as np
    from rl_post_token_gb300 import step as S
    from rl_post_token_gb300 import workloads as W
    ov = {"n_gpus": world, "micro": 1} if name == "compaction" else {}
    wl = W.make_workload(name)
    plan = dict(wl.plan, **ov)
    bp = S.plan_batch(plan, wl.row_len, wl.row_valid, wl.seg_counts)
    p = bp.plan
    for s in range(bp.n_steps):
        c0, c1 = int(p["step_chunk_off"][s]), int(p["step_chunk_off"][s + 1])
        t_lo, t_hi = int(bp.exec_tok_off[c0]), int(bp.exec_tok_off[c1])
        covered = np.zeros(t_hi - t_lo, np.int32)
        per_rank_rows = []
        for r in range(world):
            rows = 0
            for a, b in S.dp_exec_ranges(bp, s, r, world):
                assert t_lo <= a < b <= t_hi
                covered[a - t_lo:b - t_lo] += 1
                rows += b - a
            per_rank_rows.append(rows)
        assert (covered == 1).all()
        if name == "compaction":
            # every row has the same length here, so equal token counts mean equal row counts
            assert len(set(per_rank_rows)) == 1
            gpu = np.asarray(p["row_gpu"][:int(p["n_rows"])])
            off = np.concatenate([[0], np.cumsum(bp.row_len[np.asarray(p["row_src"][:int(p["n_rows"])])])])
            for r in range(world):
                want = [(int(off[j]), int(off[j + 1])) for j in np.nonzero(gpu == r)[0]]
                got = [(x, y) for a, b in S.dp_exec_ranges(bp, s, r, world) for x, y in
                       zip(range(a, b, 1024), range(a + 1024, b + 1, 1024))]
                assert got == want


def test_dp_exec_ranges_compaction_needs_its_gpu_count():
    from rl_post_token_gb300 import step as S
    from rl_post_token_gb300 import workloads as W
    wl = W.make_workload("compaction")  # planned for 4 GPUs
    bp = S.plan_batch(wl.plan, wl.row_len, wl.row_valid, wl.seg_counts)
    with pytest.raises(ValueError):
        S.dp_exec_ranges(bp, 0, 0, 2)
