"""AmpOptimizerStep(data_parallel=True) on the GPU: two or four ranks
(processes on the one visible GPU, exchanging over gloo through the host, so no
kernel waits on another rank's kernel) each step the tensors they own.  The non-finite flag
and, with clipping, the sum of squares are all-reduced between the check and
the update; the union of the shards must equal the unsharded oracle step, and
an inf in one rank's gradients must make every rank skip."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu

SIZES = [1000, 4096, 257, 3000, 17, 640]
HYPER = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
MAX_NORM = 1e-4          # the global norm of these gradients is ~9.5e-4


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _inputs():
    rng = np.random.default_rng(321)
    master = [(rng.standard_normal(n) * 0.02).astype(np.float32) for n in SIZES]
    grads = []
    for step in range(4):
        g = [(rng.standard_normal(n) * 1e-5 * 65536).astype(np.float16).view(np.uint16)
             for n in SIZES]
        if step == 1:
            g[2][256] = 0x7C00          # +inf in tensor 2 only
        grads.append(g)
    return master, grads


def _rank(rank, world, port, clip, q):
    import torch
    import torch.distributed as dist

    import loss_scaling_master_gb300 as A
    from loss_scaling_master_gb300.sharded import partition_tensors
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dev = torch.device("cuda:0")
    mine = partition_tensors(SIZES, world)[rank]
    master, grads = _inputs()
    P = [torch.from_numpy(master[i].copy()).to(dev) for i in mine]
    G = [torch.empty(SIZES[i], dtype=torch.float16, device=dev) for i in mine]
    st = A.AmpOptimizerStep(P, G, **HYPER, init_scale=65536.0, growth_interval=2,
                            max_norm=MAX_NORM if clip else None, data_parallel=True)
    states = []
    for g in grads:
        for t, i in zip(G, mine):
            t.copy_(torch.from_numpy(g[i].view(np.int16).copy()).view(torch.float16))
        st.step()
        states.append(st.state())
    out = ([p.cpu().numpy() for p in P], [m.cpu().numpy() for m in st.exp_avg],
           [v.cpu().numpy() for v in st.exp_avg_sq])
    st.check()
    st.close()
    q.put((rank, mine, states, out))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4, 7])      # 7 ranks for 6 tensors: one rank owns none
@pytest.mark.parametrize("clip", [False, True])
def test_ranks_on_one_gpu_match_the_unsharded_step(clip, world):
    import oracle as O
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, clip, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    res = [q.get(timeout=300) for _ in range(world)]
    for pr in procs:
        pr.join(timeout=120)
        assert pr.exitcode == 0
    master, grads = _inputs()
    p = [x.copy() for x in master]
    m = [np.zeros_like(x) for x in p]
    v = [np.zeros_like(x) for x in p]
    scale, tracker, step, trace = 65536.0, 0, 0, []
    for g in grads:
        fi = O.unscale_check([x.copy() for x in g], "f16", scale)
        c = O.clip_coef(O.grad_sumsq([x.copy() for x in g], "f16", scale), MAX_NORM) \
            if clip else None
        step = O.adamw_master_step(p, m, v, [x.copy() for x in g], "f16", None, scale, fi, step,
                                   HYPER["lr"], HYPER["beta1"], HYPER["beta2"], HYPER["eps"],
                                   HYPER["weight_decay"], clip=c)
        scale, tracker, _ = O.update_scale(scale, tracker, fi, 2.0, 0.5, 2)
        trace.append((scale, tracker, step))
    assert trace[1] == (32768.0, 0, 1)                      # the inf step is skipped
    for rank, mine, states, (pr, mr, vr) in res:
        assert [(s["scale"], s["growth_tracker"], s["step"]) for s in states] == trace
        for k, i in enumerate(mine):
            for got, ref in ((pr[k], p[i]), (mr[k], m[i]), (vr[k], v[i])):
                if clip:    # the global sum of squares adds the ranks' partial sums
                    rms = np.sqrt(np.mean(ref.astype(np.float64) ** 2))
                    np.testing.assert_allclose(got, ref, rtol=1e-6, atol=1e-6 * rms)
                else:
                    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


# ------------------------------------------------ flat (FSDP-style) shards
FLAT_SHAPES = [(1000,), (64, 64), (257,), (200, 200), (17,), (640,)]
FLAT_FP8 = [None, 0, None, 1, None, None]          # global FP8 index of each 2-D weight


def _flat_inputs():
    rng = np.random.default_rng(78)
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

    import loss_scaling_master_gb300 as A
    from loss_scaling_master_gb300.sharded import partition_flat
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dev = torch.device("cuda:0")
    pieces = partition_flat(FLAT_SHAPES, world)[rank]
    master, grads = _flat_inputs()
    P = [torch.from_numpy(master[t][b:e].copy()).to(dev) for t, b, e in pieces]
    G = [torch.empty(e - b, dtype=torch.float16, device=dev) for t, b, e in pieces]
    shapes = [((e - b) // FLAT_SHAPES[t][1], FLAT_SHAPES[t][1]) if FLAT_FP8[t] is not None
              else None for t, b, e in pieces]
    st = A.AmpOptimizerStep(P, G, **HYPER, init_scale=65536.0, growth_interval=2,
                            fp8_shapes=shapes, fp8_slots=[FLAT_FP8[t] for t, _, _ in pieces],
                            n_fp8_total=2, data_parallel=True)
    first = [q_.view(torch.uint8).cpu().numpy().copy() for q_ in st.fp8]
    states = []
    for g in grads:
        for tt, (t, b, e) in zip(G, pieces):
            tt.copy_(torch.from_numpy(g[t][b:e].view(np.int16).copy()).view(torch.float16))
        st.step()
        states.append(st.state())
    out = dict(p=[x.cpu().numpy() for x in P], bf=[x.view(torch.int16).cpu().numpy().view(np.uint16)
                                                  for x in st.bf16],
               q=[x.view(torch.uint8).cpu().numpy() for x in st.fp8],
               qt=[x.view(torch.uint8).cpu().numpy() for x in st.fp8_t],
               inv=st.inv_scale.cpu().numpy(), first=first)
    st.check()
    st.close()
    q.put((rank, pieces, shapes, states, out))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_flat_shards_on_one_gpu_match_the_unsharded_step(world):
    """Flat shards through AmpOptimizerStep(fp8_slots=..., data_parallel=True):
    a weight with an FP8 copy spans every rank (bands of 16-row multiples); each rank's amax of its rows
    is all-reduced (MAX) before the cast, from the first working copies on.
    The union of the bands of FP8 rows, of the column slices of the
    transposed copy, and of master and bf16 equals the unsharded oracle step
    bit for bit; every rank holding rows of a weight has the whole weight's
    inv_scale."""
    import oracle as O
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_flat, args=(r, world, port, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    res = [q.get(timeout=300) for _ in range(world)]
    for pr in procs:
        pr.join(timeout=120)
        assert pr.exitcode == 0
    master, grads = _flat_inputs()
    fp8_shapes = [s if FLAT_FP8[i] is not None else None for i, s in enumerate(FLAT_SHAPES)]
    orc = O.AmpStepOracle(master, "f16", HYPER["lr"], HYPER["beta1"], HYPER["beta2"],
                          HYPER["eps"], HYPER["weight_decay"], 65536.0, 2.0, 0.5, 2,
                          fp8_shapes=fp8_shapes)
    first = {t: orc.fp8[t].copy() for t in (1, 3)}          # the first working copies
    trace = []
    for g in grads:
        orc.run([x.copy() for x in g])
        trace.append((orc.scale, orc.tracker, orc.step))
    assert trace[1] == (32768.0, 0, 1)                       # the inf step is skipped
    full = {t: np.zeros(FLAT_SHAPES[t], np.uint8) for t in (1, 3)}
    full_t = {t: np.zeros(FLAT_SHAPES[t][::-1], np.uint8) for t in (1, 3)}
    full0 = {t: np.zeros(FLAT_SHAPES[t], np.uint8) for t in (1, 3)}
    owners = {}
    for rank, pieces, shapes, states, out in res:
        assert [(s["scale"], s["growth_tracker"], s["step"]) for s in states] == trace
        j = 0
        for k, (t, b, e) in enumerate(pieces):
            assert np.array_equal(out["p"][k].view(np.uint32), orc.master[t][b:e].view(np.uint32))
            assert np.array_equal(out["bf"][k], orc.bf16[t][b:e])
            if shapes[k] is None:
                continue
            owners.setdefault(t, set()).add(rank)
            r0, nr = b // FLAT_SHAPES[t][1], shapes[k][0]
            full[t][r0:r0 + nr] = out["q"][j]
            full_t[t][:, r0:r0 + nr] = out["qt"][j]
            full0[t][r0:r0 + nr] = out["first"][j]
            j += 1
        for t in {t for (t, _, _), sh in zip(pieces, shapes) if sh is not None}:
            assert out["inv"][FLAT_FP8[t]] == orc.inv_scale[FLAT_FP8[t]]   # the owners' bands
    assert owners[3] == set(range(world))
    for t in (1, 3):
        assert np.array_equal(full[t].ravel(), orc.fp8[t])
        assert np.array_equal(full_t[t].ravel(), orc.fp8_t[t])
        assert np.array_equal(full0[t].ravel(), first[t])


# ------------------- flat shards: ranks with no FP8 weight, and an empty rank
# case: (shapes, global FP8 index per tensor, world, (tensor, element, step) of a +inf)
CASES = {
    # both FP8 weights fall inside rank 0's slice; ranks 1-3 hold plain tensors only
    "no_fp8": ([(64, 64), (128, 64), (20000,), (20000,)], [0, 1, None, None], 4, (3, 15000, 2)),
    # the 32-row weight is cut in two 16-row bands; rank 1's slice is empty
    "empty_rank": ([(32, 64), (16,)], [0, None], 3, (1, 5, 2)),
}


def _case_inputs(case):
    shapes, _, _, (ti, ei, si) = CASES[case]
    rng = np.random.default_rng(79)
    sizes = [int(np.prod(s)) for s in shapes]
    master = [(rng.standard_normal(n) * 0.02).astype(np.float32) for n in sizes]
    grads = []
    for step in range(4):
        g = [(rng.standard_normal(n) * 1e-5 * 65536).astype(np.float16).view(np.uint16)
             for n in sizes]
        if step == si:
            g[ti][ei] = 0x7C00
        grads.append(g)
    return master, grads


def _rank_case(rank, world, port, q, case):
    import torch
    import torch.distributed as dist

    import loss_scaling_master_gb300 as A
    from loss_scaling_master_gb300.sharded import partition_flat
    shapes_all, fp8_all, _, _ = CASES[case]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(0)
    dev = torch.device("cuda:0")
    pieces = partition_flat(shapes_all, world)[rank]
    master, grads = _case_inputs(case)
    P = [torch.from_numpy(master[t][b:e].copy()).to(dev) for t, b, e in pieces]
    G = [torch.empty(e - b, dtype=torch.float16, device=dev) for t, b, e in pieces]
    shapes = [((e - b) // shapes_all[t][1], shapes_all[t][1]) if fp8_all[t] is not None
              else None for t, b, e in pieces]
    st = A.AmpOptimizerStep(P, G, **HYPER, init_scale=65536.0, growth_interval=2,
                            fp8_shapes=shapes, fp8_slots=[fp8_all[t] for t, _, _ in pieces],
                            n_fp8_total=sum(x is not None for x in fp8_all), data_parallel=True)
    states = []
    for g in grads:
        for tt, (t, b, e) in zip(G, pieces):
            tt.copy_(torch.from_numpy(g[t][b:e].view(np.int16).copy()).view(torch.float16))
        st.step()
        states.append(st.state())
    out = dict(p=[x.cpu().numpy() for x in P],
               bf=[x.view(torch.int16).cpu().numpy().view(np.uint16) for x in st.bf16],
               q=[x.view(torch.uint8).cpu().numpy() for x in st.fp8],
               qt=[x.view(torch.uint8).cpu().numpy() for x in st.fp8_t],
               inv=st.inv_scale.cpu().numpy())
    st.check()
    st.close()
    q.put((rank, pieces, states, out))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("case", sorted(CASES))
def test_flat_shards_with_ranks_holding_no_fp8_weight_or_nothing(case):
    """Flat shards where some ranks hold no FP8 weight ("no_fp8": three of
    four ranks hold plain tensors only) or nothing at all ("empty_rank": the
    middle one of three slices is empty).  Every rank still takes part in the
    found_inf and amax exchanges, from the first working copies on, so no
    collective waits for it; an inf on one rank makes every rank skip; every
    piece equals the unsharded oracle step bit for bit, the FP8 bands, their
    transposed slices and the owners' inv_scale too."""
    import oracle as O
    shapes_all, fp8_all, world, _ = CASES[case]
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_case, args=(r, world, port, q, case)) for r in range(world)]
    for pr in procs:
        pr.start()
    res = [q.get(timeout=300) for _ in range(world)]
    for pr in procs:
        pr.join(timeout=120)
        assert pr.exitcode == 0
    master, grads = _case_inputs(case)
    fp8_shapes = [s if fp8_all[i] is not None else None for i, s in enumerate(shapes_all)]
    orc = O.AmpStepOracle(master, "f16", HYPER["lr"], HYPER["beta1"], HYPER["beta2"],
                          HYPER["eps"], HYPER["weight_decay"], 65536.0, 2.0, 0.5, 2,
                          fp8_shapes=fp8_shapes)
    trace = []
    for g in grads:
        orc.run([x.copy() for x in g])
        trace.append((orc.scale, orc.tracker, orc.step))
    assert trace[2][2] == trace[1][2]                         # the inf step is skipped
    full = {t: np.zeros(shapes_all[t], np.uint8) for t in range(len(shapes_all))
            if fp8_all[t] is not None}
    full_t = {t: np.zeros(shapes_all[t][::-1], np.uint8) for t in full}
    holders = {t: set() for t in full}
    for rank, pieces, states, out in res:
        assert [(s["scale"], s["growth_tracker"], s["step"]) for s in states] == trace
        j = 0
        for k, (t, b, e) in enumerate(pieces):
            assert np.array_equal(out["p"][k].view(np.uint32), orc.master[t][b:e].view(np.uint32))
            assert np.array_equal(out["bf"][k], orc.bf16[t][b:e])
            if fp8_all[t] is None:
                continue
            holders[t].add(rank)
            cols = shapes_all[t][1]
            r0, nr = b // cols, (e - b) // cols
            full[t][r0:r0 + nr] = out["q"][j].reshape(nr, cols)
            full_t[t][:, r0:r0 + nr] = out["qt"][j].reshape(cols, nr)
            assert out["inv"][fp8_all[t]] == orc.inv_scale[fp8_all[t]]
            j += 1
    for t in full:
        assert np.array_equal(full[t].ravel(), orc.fp8[t])
        assert np.array_equal(full_t[t].ravel(), orc.fp8_t[t])
    if case == "no_fp8":
        assert set().union(*holders.values()) == {0}
    else:
        assert holders[0] == {0, 2} and not [p for r, p, _, _ in res if r == 1][0]
