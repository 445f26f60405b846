"""Bounds and coverage checks that stand in for a memory sanitizer.

* Every size 0 ... 67 (plus 255-257, 1000, 4096) in one list, 16-byte aligned
  and not, through the check and the AdamW step, against the oracle.
* Canaries: every output is a view into a larger buffer whose 64 elements
  before and after it (and a misaligning lead) are pre-filled with a pattern;
  after the calls the pattern must be intact, the outputs equal to the oracle,
  and the read-only inputs unchanged."""
import numpy as np
import pytest
import torch

import oracle as O
from parity_helpers import to_device, to_host_bits

pytestmark = pytest.mark.gpu

GUARD = 64
SMALL = list(range(68)) + [255, 256, 257, 1000, 4096]
_INT = {torch.float32: (torch.int32, 0x7FA5A5A5), torch.float16: (torch.int16, -0x5A5B),
        torch.bfloat16: (torch.int16, -0x5A5B), torch.uint8: (torch.uint8, 0xA5),
        torch.int32: (torch.int32, 0x7FA5A5A5)}


@pytest.fixture(scope="module")
def A():
    from loss_scaling_master_gb300 import build as B
    B.build()
    import loss_scaling_master_gb300 as pkg
    pkg.load()
    assert torch.cuda.is_available()
    return pkg


@pytest.fixture(scope="module")
def dev(A):
    return torch.device("cuda:0")


class Guarded:
    """A device view of n elements inside a buffer with canary-filled margins."""

    def __init__(self, n, dtype, dev, lead=0, shape=None):
        self.n, self.lead = n, lead
        self.buf = torch.empty(GUARD + lead + n + GUARD, dtype=dtype, device=dev)
        it, self.canary = _INT[dtype]
        self.ibuf = self.buf.view(it)
        self.ibuf.fill_(self.canary)
        v = self.buf[GUARD + lead:GUARD + lead + n]
        self.view = v.view(*shape) if shape is not None else v

    def intact(self) -> bool:
        b = self.ibuf.cpu()
        lo, hi = GUARD + self.lead, GUARD + self.lead + self.n
        return bool((b[:lo] == self.canary).all()) and bool((b[hi:] == self.canary).all())


def _grads(rng, sizes, sigma):
    return [(rng.standard_normal(n) * sigma).astype(np.float16).view(np.uint16) for n in sizes]


@pytest.mark.parametrize("lead", [0, 1])
def test_every_small_size_through_check_and_adamw(A, dev, lead):
    rng = np.random.default_rng(70 + lead)
    sizes = SMALL
    master = [(rng.standard_normal(n) * 0.02).astype(np.float32) for n in sizes]
    P = [Guarded(n, torch.float32, dev, lead) for n in sizes]
    M = [Guarded(n, torch.float32, dev, lead) for n in sizes]
    V = [Guarded(n, torch.float32, dev, lead) for n in sizes]
    G = [Guarded(n, torch.float16, dev, lead) for n in sizes]
    B = [Guarded(n, torch.bfloat16, dev, lead) for n in sizes]
    for g, m in zip(P, master):
        g.view.copy_(torch.from_numpy(m))
    for g in M + V:
        g.view.zero_()
    lists = [A.amp_tensor_list_create([g.view for g in X]) for X in (P, M, V, G, B)]
    scale = torch.tensor([1024.0], device=dev)
    fi = torch.zeros(1, dtype=torch.int32, device=dev)
    step = torch.zeros(1, dtype=torch.int32, device=dev)
    rp, rm, rv = [m.copy() for m in master], [np.zeros(n, np.float32) for n in sizes], \
        [np.zeros(n, np.float32) for n in sizes]
    rb = [np.zeros(n, np.uint16) for n in sizes]
    rstep = 0
    hyper = (1e-3, 0.9, 0.999, 1e-8, 0.01)
    for k in range(4):
        gh = _grads(rng, sizes, 1e-3 * 1024)
        if k == 2:                                  # a planted inf at the tail of size 67
            gh[67][66] = 0x7C00
        for g, h in zip(G, gh):
            g.view.copy_(to_device(h, "f16", dev))
        fi.zero_()
        A.amp_unscale_check(lists[3], scale, fi)
        expect = O.unscale_check([h.copy() for h in gh], "f16", 1024.0)
        assert int(fi.item()) == expect == (1 if k == 2 else 0)
        A.amp_adamw_master_step(*lists, scale, fi, step, *hyper)
        rstep = O.adamw_master_step(rp, rm, rv, gh, "f16", rb, 1024.0, expect, rstep, *hyper)
        torch.cuda.synchronize()
        assert int(step.item()) == rstep
        for i, n in enumerate(sizes):
            assert np.array_equal(to_host_bits(P[i].view).view(np.uint32), rp[i].view(np.uint32)), (k, n)
            assert np.array_equal(to_host_bits(M[i].view).view(np.uint32), rm[i].view(np.uint32)), (k, n)
            assert np.array_equal(to_host_bits(V[i].view).view(np.uint32), rv[i].view(np.uint32)), (k, n)
            assert np.array_equal(to_host_bits(B[i].view), rb[i]), (k, n)
            assert np.array_equal(to_host_bits(G[i].view), gh[i]), (k, n)   # read only
    assert all(g.intact() for X in (P, M, V, G, B) for g in X)
    for L in lists:
        L.close()


@pytest.mark.parametrize("lead", [0, 1])
def test_fp8_outputs_stay_in_their_extent(A, dev, lead):
    """Tensorwise (single and list) and rowwise casts, with transposed copies,
    on tile-aligned and ragged shapes: no byte outside any output changes."""
    rng = np.random.default_rng(80 + lead)
    shapes = [(1, 1), (3, 5), (17, 31), (128, 128), (127, 129), (256, 384), (300, 520)]
    xs = [O.encode("bf16", rng.standard_normal(r * c).astype(np.float32)) for r, c in shapes]
    X = [Guarded(r * c, torch.bfloat16, dev, lead, (r, c)) for r, c in shapes]
    for g, h in zip(X, xs):
        g.view.copy_(to_device(h, "bf16", dev).view(g.view.shape))
    # single-tensor tensorwise and rowwise
    for (r, c), g, h in zip(shapes, X, xs):
        q = Guarded(r * c, torch.uint8, dev, lead)
        qt = Guarded(r * c, torch.uint8, dev, lead)
        inv = Guarded(1, torch.float32, dev)
        am = Guarded(1, torch.float32, dev)
        A.fp8_quant_tensorwise(g.view, "e4m3fn", q.view, qt.view, inv.view, am.view, rows=r, cols=c)
        rq, rqt, rinv, ramax = O.fp8_quant_tensorwise(h, "bf16", r, c, "e4m3fn")
        torch.cuda.synchronize()
        assert np.array_equal(to_host_bits(q.view), rq) and np.array_equal(to_host_bits(qt.view), rqt)
        assert all(t.intact() for t in (q, qt, inv, am, g)), (r, c)
        vec = {k: Guarded(n, torch.float32, dev) for k, n in
               (("ar", r), ("sr", r), ("ir", r), ("ac", c), ("sc", c), ("ic", c))}
        q2 = Guarded(r * c, torch.uint8, dev, lead)
        qt2 = Guarded(r * c, torch.uint8, dev, lead)
        A.fp8_quant_rowwise(g.view, "e5m2", q2.view, qt2.view, vec["ar"].view, vec["sr"].view,
                            vec["ir"].view, vec["ac"].view, vec["sc"].view, vec["ic"].view)
        ref = O.fp8_quant_rowwise(h, "bf16", r, c, "e5m2")
        torch.cuda.synchronize()
        assert np.array_equal(to_host_bits(q2.view), ref["q"])
        assert np.array_equal(to_host_bits(qt2.view), ref["q_t"])
        assert all(t.intact() for t in [q2, qt2] + list(vec.values())), (r, c)
    # the list form over all shapes at once
    Q = [Guarded(r * c, torch.uint8, dev, lead, (r, c)) for r, c in shapes]
    QT = [Guarded(r * c, torch.uint8, dev, lead, (c, r)) for r, c in shapes]
    LX = A.amp_tensor_list_create([g.view for g in X], two_d=True)
    LQ = A.amp_tensor_list_create([g.view.view(torch.float8_e4m3fn) for g in Q], two_d=True)
    LQT = A.amp_tensor_list_create([g.view.view(torch.float8_e4m3fn) for g in QT], two_d=True)
    amax = Guarded(len(shapes), torch.float32, dev)
    inv = Guarded(len(shapes), torch.float32, dev)
    ram = [float(np.abs(O.decode("bf16", h)).max()) for h in xs]
    amax.view.copy_(torch.tensor(ram))
    A.fp8_quant_tensorwise_list(LX, LQ, LQT, "e4m3fn", amax.view, inv.view)
    torch.cuda.synchronize()
    for i, ((r, c), h) in enumerate(zip(shapes, xs)):
        rq, rqt, _, _ = O.fp8_quant_tensorwise(h, "bf16", r, c, "e4m3fn", amax=ram[i])
        assert np.array_equal(to_host_bits(Q[i].view).ravel(), rq), (r, c)
        assert np.array_equal(to_host_bits(QT[i].view).ravel(), rqt), (r, c)
    assert all(t.intact() for t in Q + QT + X + [amax, inv])
    for L in (LX, LQ, LQT):
        L.close()


def test_inplace_unscale_stays_in_extent(A, dev):
    rng = np.random.default_rng(90)
    G = [Guarded(n, torch.float16, dev, 1) for n in SMALL]
    gh = _grads(rng, SMALL, 100.0)
    for g, h in zip(G, gh):
        g.view.copy_(to_device(h, "f16", dev))
    L = A.amp_tensor_list_create([g.view for g in G])
    fi = torch.zeros(1, dtype=torch.int32, device=dev)
    A.amp_unscale_check(L, torch.tensor([8.0], device=dev), fi, inplace=True)
    ref = [h.copy() for h in gh]
    assert int(fi.item()) == O.unscale_check(ref, "f16", 8.0, inplace=True) == 0
    torch.cuda.synchronize()
    for g, r in zip(G, ref):
        assert np.array_equal(to_host_bits(g.view), r)
    assert all(g.intact() for g in G)
    L.close()
