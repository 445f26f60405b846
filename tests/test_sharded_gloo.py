"""Sharded (2-rank, gloo, CPU) step: tensors partitioned across ranks, the
non-finite flag combined with all-reduce(MAX), each rank updating its own
tensors with the oracle.  The union of the shards must equal the unsharded
oracle step, and a non-finite gradient on one rank must make both skip."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


SIZES = [1000, 4096, 257, 3000, 17, 640]
HYPER = (1e-3, 0.9, 0.999, 1e-8, 0.01)


def _inputs():
    rng = np.random.default_rng(123)
    master = [(rng.standard_normal(n) * 0.02).astype(np.float32) for n in SIZES]
    grads = []
    for step in range(4):
        g = [(rng.standard_normal(n) * 1e-5 * 65536).astype(np.float16).view(np.uint16)
             for n in SIZES]
        if step == 1:
            g[2][256] = 0x7C00          # +inf in tensor 2 only
        grads.append(g)
    return master, grads


def _rank(rank, world, port, q):
    import torch
    import torch.distributed as dist

    import oracle as O
    from loss_scaling_master_gb300.sharded import combine_found_inf, partition_tensors
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = partition_tensors(SIZES, world)[rank]
    master, grads = _inputs()
    p = [master[i].copy() for i in mine]
    m = [np.zeros_like(x) for x in p]
    v = [np.zeros_like(x) for x in p]
    scale, tracker, step = 65536.0, 0, 0
    flags = []
    for g in grads:
        gs = [g[i].copy() for i in mine]
        local = O.unscale_check(gs, "f16", scale)
        fi = torch.tensor([local], dtype=torch.int32)
        combine_found_inf(fi)
        flags.append((local, int(fi.item())))
        step = O.adamw_master_step(p, m, v, gs, "f16", None, scale, int(fi.item()), step, *HYPER)
        scale, tracker, _ = O.update_scale(scale, tracker, int(fi.item()), 2.0, 0.5, 2)
    q.put((rank, mine, p, m, v, flags, scale, tracker, step))
    dist.barrier()
    dist.destroy_process_group()


def test_partition_is_balanced_and_complete():
    from loss_scaling_master_gb300.sharded import partition_tensors
    for world in (1, 2, 3, 4):
        parts = partition_tensors(SIZES, world)
        assert sorted(i for p in parts for i in p) == list(range(len(SIZES)))
        loads = [sum(SIZES[i] for i in p) for p in parts]
        assert max(loads) - min(loads) <= max(SIZES)


def test_two_rank_gloo_step_matches_unsharded():
    import oracle as O
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    master, grads = _inputs()
    p = [x.copy() for x in master]
    m = [np.zeros_like(x) for x in p]
    v = [np.zeros_like(x) for x in p]
    scale, tracker, step = 65536.0, 0, 0
    for g in grads:
        fi = O.unscale_check([x.copy() for x in g], "f16", scale)
        step = O.adamw_master_step(p, m, v, [x.copy() for x in g], "f16", None, scale, fi, step,
                                   *HYPER)
        scale, tracker, _ = O.update_scale(scale, tracker, fi, 2.0, 0.5, 2)
    owner_of_inf = [r for r in res if 2 in r[1]][0][0]
    for rank, mine, pr, mr, vr, flags, sc, tr, st in res:
        assert (sc, tr, st) == (scale, tracker, step) == (65536.0, 0, 3)
        assert [f[1] for f in flags] == [0, 1, 0, 0]           # combined: everyone skips step 2
        assert flags[1][0] == int(rank == owner_of_inf)        # locally only the owner saw it
        for k, i in enumerate(mine):
            assert np.array_equal(pr[k], p[i]) and np.array_equal(mr[k], m[i])
            assert np.array_equal(vr[k], v[i])


MAX_NORM = 1e-4      # below the global norm of these gradients (~9.5e-4): clipping is active


def _rank_clip(rank, world, port, q):
    import torch
    import torch.distributed as dist

    import oracle as O
    from loss_scaling_master_gb300.sharded import (combine_found_inf, combine_grad_sumsq,
                                                   partition_tensors)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = partition_tensors(SIZES, world)[rank]
    master, grads = _inputs()
    p = [master[i].copy() for i in mine]
    m = [np.zeros_like(x) for x in p]
    v = [np.zeros_like(x) for x in p]
    scale, tracker, step = 65536.0, 0, 0
    sums = []
    for g in grads:
        gs = [g[i].copy() for i in mine]
        fi = torch.tensor([O.unscale_check(gs, "f16", scale)], dtype=torch.int32)
        combine_found_inf(fi)
        ss = torch.tensor([O.grad_sumsq(gs, "f16", scale)], dtype=torch.float64)
        combine_grad_sumsq(ss)
        sums.append(float(ss.item()))
        clip = O.clip_coef(float(ss.item()), MAX_NORM)
        step = O.adamw_master_step(p, m, v, gs, "f16", None, scale, int(fi.item()), step, *HYPER,
                                   clip=clip)
        scale, tracker, _ = O.update_scale(scale, tracker, int(fi.item()), 2.0, 0.5, 2)
    q.put((rank, mine, p, m, v, sums, scale, tracker, step))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_gloo_clipped_step_uses_the_global_norm():
    """With clipping, the ranks' sums of squares are summed (all-reduce SUM):
    both ranks see the global sum and clip by the global norm, and the union
    of the shards matches the unsharded clipped step.  The global sum adds
    the ranks' partial sums in another order than the unsharded sum, so it
    and the states are compared within rel 1e-12 and rel 1e-6."""
    import oracle as O
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_clip, args=(r, world, port, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    master, grads = _inputs()
    p = [x.copy() for x in master]
    m = [np.zeros_like(x) for x in p]
    v = [np.zeros_like(x) for x in p]
    scale, tracker, step = 65536.0, 0, 0
    sums, clips = [], []
    for g in grads:
        fi = O.unscale_check([x.copy() for x in g], "f16", scale)
        ss = O.grad_sumsq([x.copy() for x in g], "f16", scale)
        sums.append(ss)
        clips.append(O.clip_coef(ss, MAX_NORM))
        step = O.adamw_master_step(p, m, v, [x.copy() for x in g], "f16", None, scale, fi, step,
                                   *HYPER, clip=clips[-1])
        scale, tracker, _ = O.update_scale(scale, tracker, fi, 2.0, 0.5, 2)
    assert all(c < 1.0 for k, c in enumerate(clips) if k != 1)     # clipping is active
    for rank, mine, pr, mr, vr, rs, sc, tr, st in res:
        assert (sc, tr, st) == (scale, tracker, step)
        for k in (0, 2, 3):                                       # step 2 is skipped (inf)
            assert abs(rs[k] - sums[k]) <= 1e-12 * sums[k]
        for k, i in enumerate(mine):
            for got, ref in ((pr[k], p[i]), (mr[k], m[i]), (vr[k], v[i])):
                rms = np.sqrt(np.mean(ref.astype(np.float64) ** 2))
                np.testing.assert_allclose(got, ref, rtol=1e-6, atol=1e-6 * rms)
