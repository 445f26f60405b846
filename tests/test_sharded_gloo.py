"""Sharded (2- and 4-rank, gloo, CPU) step: tensors partitioned across ranks,
the non-finite flag combined with all-reduce(MAX), each rank updating its own
tensors with the oracle.  The union of the shards must equal the unsharded
oracle step, and a non-finite gradient on one rank must make all skip."""
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


@pytest.mark.parametrize("world", [2, 4, 7])      # 7 ranks for 6 tensors: one rank owns none
def test_gloo_step_matches_unsharded(world):
    import oracle as O
    port = _free_port()
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


@pytest.mark.parametrize("world", [2, 4, 7])
def test_gloo_clipped_step_uses_the_global_norm(world):
    """With clipping, the ranks' sums of squares are summed (all-reduce SUM):
    every rank sees the global sum and clips by the global norm, and the union
    of the shards matches the unsharded clipped step.  The global sum adds
    the ranks' partial sums in another order than the unsharded sum, so it
    and the states are compared within rel 1e-12 and rel 1e-6."""
    import oracle as O
    port = _free_port()
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


# ------------------------------------------------ flat (FSDP-style) shards
FLAT_SHAPES = [(1000,), (64, 64), (257,), (200, 200), (17,), (640,)]
FLAT_FP8 = [None, 0, None, 1, None, None]          # global FP8 index of each 2-D weight


def test_partition_flat_covers_everything_once_on_row_and_vector_boundaries():
    from loss_scaling_master_gb300.sharded import partition_flat
    sizes = [int(np.prod(s)) for s in FLAT_SHAPES]
    for world in (1, 2, 3, 4, 7):
        parts = partition_flat(FLAT_SHAPES, world)
        assert len(parts) == world
        flat = [(t, b, e) for p in parts for (t, b, e) in p]
        # in flat order, contiguous, each tensor covered exactly once
        pos = 0
        offs = np.concatenate([[0], np.cumsum(sizes)])
        for t, b, e in flat:
            assert offs[t] + b == pos and e > b
            pos = offs[t] + e
        assert pos == offs[-1]
        for t, b, e in flat:
            s = FLAT_SHAPES[t]
            for x in (b, e):
                if len(s) == 2:
                    assert x % s[1] == 0 and ((x // s[1]) % 16 == 0 or x == sizes[t]), (t, x)
                else:
                    assert x % 8 == 0 or x == sizes[t], (t, x)
        # balanced to within one cut unit of the even share
        loads = [sum(e - b for _, b, e in p) for p in parts]
        assert max(loads) - min(loads) <= 2 * 16 * 200 + 8


def _flat_inputs():
    rng = np.random.default_rng(77)
    sizes = [int(np.prod(s)) for s in FLAT_SHAPES]
    master = [(rng.standard_normal(n) * 0.02).astype(np.float32) for n in sizes]
    grads = []
    for step in range(4):
        g = [(rng.standard_normal(n) * 1e-5 * 65536).astype(np.float16).view(np.uint16)
             for n in sizes]
        if step == 1:
            g[3][150 * 200 + 7] = 0x7C00     # +inf in the second rank's rows of the FP8 weight
        grads.append(g)
    return master, grads


def _rank_flat(rank, world, port, q):
    import torch
    import torch.distributed as dist

    import oracle as O
    from loss_scaling_master_gb300.sharded import (combine_amax, combine_found_inf,
                                                   partition_flat)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    pieces = partition_flat(FLAT_SHAPES, world)[rank]
    master, grads = _flat_inputs()
    p = [master[t][b:e].copy() for t, b, e in pieces]
    m = [np.zeros_like(x) for x in p]
    v = [np.zeros_like(x) for x in p]
    bf = [np.zeros(x.size, np.uint16) for x in p]
    slots = [FLAT_FP8[t] if FLAT_FP8[t] is not None else -1 for t, _, _ in pieces]
    scale, tracker, step = 65536.0, 0, 0
    fp8 = {}
    for g in grads:
        gs = [g[t][b:e].copy() for t, b, e in pieces]
        fi = torch.tensor([O.unscale_check(gs, "f16", scale)], dtype=torch.int32)
        combine_found_inf(fi)
        amax = np.zeros(2, np.float32)
        step = O.adamw_master_step(p, m, v, gs, "f16", bf, scale, int(fi.item()), step, *HYPER,
                                   amax_slot=slots, amax=amax)
        at = torch.from_numpy(amax.copy())
        combine_amax(at)                      # the global amax of every FP8 weight
        if not int(fi.item()):
            for k, (t, b, e) in enumerate(pieces):
                if FLAT_FP8[t] is None:
                    continue
                cols = FLAT_SHAPES[t][1]
                q_, qt, inv, _ = O.fp8_quant_tensorwise(bf[k], "bf16", (e - b) // cols, cols,
                                                        "e4m3fn", amax=float(at[FLAT_FP8[t]]))
                fp8[t] = (b // cols, q_, qt, inv)
        scale, tracker, _ = O.update_scale(scale, tracker, int(fi.item()), 2.0, 0.5, 2)
    q.put((rank, pieces, p, m, v, bf, fp8, scale, tracker, step))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_gloo_flat_shards_match_unsharded(world):
    """A weight with an FP8 copy spans several ranks (two of two, four of
    four).  Each rank updates its flat slice, folds the amax of its rows, and
    the amax array is all-reduced (MAX) before the cast: the union of the
    ranks' bands of FP8 rows, of their column slices of the transposed copy,
    and of master, m, v and bf16 equals the unsharded oracle step bit for bit,
    and an inf in one rank's rows makes all skip."""
    import oracle as O
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_flat, args=(r, world, port, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    master, grads = _flat_inputs()
    fp8_shapes = [s if FLAT_FP8[i] is not None else None for i, s in enumerate(FLAT_SHAPES)]
    orc = O.AmpStepOracle(master, "f16", *HYPER, 65536.0, 2.0, 0.5, 2, fp8_shapes=fp8_shapes)
    for g in grads:
        orc.run([x.copy() for x in g])
    assert orc.step == 3 and orc.scale == 65536.0
    spans = {}
    for rank, pieces, p, m, v, bf, fp8, sc, tr, st in res:
        assert (sc, tr, st) == (orc.scale, orc.tracker, orc.step)
        for k, (t, b, e) in enumerate(pieces):
            spans.setdefault(t, []).append(rank)
            assert np.array_equal(p[k].view(np.uint32), orc.master[t][b:e].view(np.uint32))
            assert np.array_equal(m[k].view(np.uint32), orc.exp_avg[t][b:e].view(np.uint32))
            assert np.array_equal(v[k].view(np.uint32), orc.exp_avg_sq[t][b:e].view(np.uint32))
            assert np.array_equal(bf[k], orc.bf16[t][b:e])
    assert sorted(spans[3]) == list(range(world))          # the FP8 weight spans the ranks
    for t, shp in enumerate(FLAT_SHAPES):
        if FLAT_FP8[t] is None:
            continue
        rows, cols = shp
        full, full_t = np.zeros((rows, cols), np.uint8), np.zeros((cols, rows), np.uint8)
        for rank, _, _, _, _, _, fp8, *_ in res:
            if t in fp8:
                r0, q_, qt, inv = fp8[t]
                nr = q_.size // cols
                full[r0:r0 + nr] = q_.reshape(nr, cols)
                full_t[:, r0:r0 + nr] = qt.reshape(cols, nr)
                assert inv == orc.inv_scale[FLAT_FP8[t]]       # one scale for the whole weight
        assert np.array_equal(full.ravel(), orc.fp8[t])
        assert np.array_equal(full_t.ravel(), orc.fp8_t[t])
