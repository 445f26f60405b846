"""CUDA path (through the C ABI) vs the CPU oracle, element by element, on
seeded inputs that span several chunks/tiles, ragged tails, misaligned
tensors and the method's degenerate cases."""
import numpy as np
import pytest
import torch

import oracle as O
from parity_helpers import (assert_bf16_close, assert_state_close, bit_identical_fraction,
                            to_device, to_host_bits)

pytestmark = pytest.mark.gpu

RAGGED = [1, 7, 8, 9, 63, 64, 67, 255, 256, 257, 1000, 4096, 16383, 16384, 16385, 40000]


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


def _grads_host(rng, sizes, dt, sigma=1.0):
    out = []
    for n in sizes:
        x = (rng.standard_normal(n) * sigma).astype(np.float32)
        if dt == "f32":
            out.append(x)
        elif dt == "f16":
            out.append(x.astype(np.float16).view(np.uint16))
        else:
            out.append(O.encode("bf16", x))
    return out


def _device_views(host_list, dt, device, misalign: bool):
    """Device tensors holding host_list; with misalign, packed back to back
    in one buffer with a 1-element lead, so most bases are not 16-byte aligned."""
    if not misalign:
        return [to_device(h, dt, device) for h in host_list]
    flat = np.concatenate([np.zeros(1, host_list[0].dtype)] + list(host_list))
    buf = to_device(flat, dt, device)
    views, off = [], 1
    for h in host_list:
        views.append(buf[off:off + h.size])
        off += h.size
    return views


def _inf_bits(dt, val):
    if dt == "f32":
        return np.float32(val)
    if dt == "f16":
        return np.array([val], np.float16).view(np.uint16)[0]
    return O.encode("bf16", np.array([val], np.float32))[0]


# ------------------------------------------------------------ unscale / check
@pytest.mark.parametrize("dt", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("misalign", [False, True])
def test_unscale_check_parity(A, dev, dt, misalign):
    rng = np.random.default_rng(10)
    sizes = RAGGED
    base = _grads_host(rng, sizes, dt, sigma=3.0)
    cases = []
    for scale in (65536.0, 1.0, 2.0 ** -20, 1e-35, 0.0, np.inf, np.nan, -4.0):
        cases.append((scale, None))
    for site in ((len(sizes) - 1, sizes[-1] - 1, np.inf), (5, 0, np.nan), (9, 256, -np.inf),
                 (13, 16383, np.inf), (14, 16384, np.nan)):
        cases.append((65536.0, site))
    for scale, site in cases:
        hl = [h.copy() for h in base]
        if site is not None:
            hl[site[0]][site[1]] = _inf_bits(dt, site[2])
        tensors = _device_views(hl, dt, dev, misalign)
        L = A.amp_tensor_list_create(tensors)
        for start in (0, 1):
            fi = torch.tensor([start], dtype=torch.int32, device=dev)
            s = torch.tensor([scale], dtype=torch.float32, device=dev)
            A.amp_unscale_check(L, s, fi)
            expect = O.unscale_check([h.copy() for h in hl], dt, float(np.float32(scale)),
                                     found_inf=start)
            assert int(fi.item()) == expect, (dt, misalign, scale, site, start)
        L.close()


@pytest.mark.parametrize("dt", ["f16", "bf16", "f32"])
def test_unscale_inplace_parity(A, dev, dt):
    rng = np.random.default_rng(11)
    hl = _grads_host(rng, RAGGED, dt, sigma=1e3)
    hl[3][2] = _inf_bits(dt, np.nan)
    for scale in (65536.0, 3.0, 1e-3):
        tensors = _device_views(hl, dt, dev, misalign=True)
        L = A.amp_tensor_list_create(tensors)
        fi = torch.zeros(1, dtype=torch.int32, device=dev)
        A.amp_unscale_check(L, torch.tensor([scale], device=dev), fi, inplace=True)
        ref = [h.copy() for h in hl]
        expect = O.unscale_check(ref, dt, scale, inplace=True)
        assert int(fi.item()) == expect == 1
        for t, r in zip(tensors, ref):
            got = to_host_bits(t)
            if dt == "f32":
                # an fp32 product with a NaN operand is NaN; IEEE 754 leaves
                # its payload open, so NaN positions are compared, bits elsewhere
                nan = np.isnan(r)
                assert np.array_equal(np.isnan(got), nan)
                assert np.array_equal(got[~nan].view(np.uint32), r[~nan].view(np.uint32))
            else:
                assert np.array_equal(got, r)
        L.close()


# ------------------------------------------------------------ scale machine
def test_update_scale_parity(A, dev):
    rng = np.random.default_rng(12)
    for interval, growth, backoff, init in ((2, 2.0, 0.5, 65536.0), (10, 2.0, 0.5, 65536.0),
                                            (1, 2.0, 0.5, 2.0 ** 126), (3, 1.0, 1.0, 1.0),
                                            (5, 3.0, 0.25, 1000.0)):
        s = torch.tensor([init], dtype=torch.float32, device=dev)
        t = torch.zeros(1, dtype=torch.int32, device=dev)
        fi = torch.zeros(1, dtype=torch.int32, device=dev)
        amax = torch.full((5,), 7.0, device=dev)
        rs, rt = float(np.float32(init)), 0
        for k in range(60):
            flag = int(rng.random() < 0.15)
            fi.fill_(flag)
            A.amp_update_scale(s, t, fi, growth, backoff, interval, amax=amax, n_amax=5)
            ram = np.full(5, 7.0, np.float32)
            rs, rt, rfi = O.update_scale(rs, rt, flag, growth, backoff, interval, ram)
            assert float(s.item()) == rs and int(t.item()) == rt and int(fi.item()) == rfi == 0
            assert not amax.any()
            amax.fill_(7.0)


# ------------------------------------------------------------------- AdamW
def _adamw_case(A, dev, gdt, misalign, sizes, steps, hyper, scales, skip_at, slots, seed):
    rng = np.random.default_rng(seed)
    n = len(sizes)
    master_h = [(rng.standard_normal(k) * 0.02).astype(np.float32) for k in sizes]
    mk = lambda hs, dt: _device_views(hs, dt, dev, misalign)
    P = mk(master_h, "f32")
    M = mk([np.zeros(k, np.float32) for k in sizes], "f32")
    V = mk([np.zeros(k, np.float32) for k in sizes], "f32")
    G = mk(_grads_host(rng, sizes, gdt), gdt)
    Bf = mk([np.zeros(k, np.uint16) for k in sizes], "bf16")
    LP, LM, LV, LG, LB = (A.amp_tensor_list_create(x) for x in (P, M, V, G, Bf))
    n_slots = max(slots) + 1 if slots else 0
    if slots:
        A.amp_tensor_list_set_amax_slots(LB, slots)
    amax = torch.zeros(max(n_slots, 1), device=dev)
    step = torch.zeros(1, dtype=torch.int32, device=dev)
    fi = torch.zeros(1, dtype=torch.int32, device=dev)
    s_dev = torch.zeros(1, device=dev)
    rp = [x.copy() for x in master_h]
    rm = [np.zeros(k, np.float32) for k in sizes]
    rv = [np.zeros(k, np.float32) for k in sizes]
    rb = [np.zeros(k, np.uint16) for k in sizes]
    rstep = 0
    for k in range(steps):
        S = scales[k % len(scales)]
        gh = _grads_host(rng, sizes, gdt, sigma=1e-3 * S)
        for t, h in zip(G, gh):
            t.copy_(to_device(h, gdt, dev))
        skip = int(k in skip_at)
        fi.fill_(skip)
        s_dev.fill_(S)
        amax.zero_()
        A.amp_adamw_master_step(LP, LM, LV, LG, LB, s_dev, fi, step, *hyper,
                                amax=amax if slots else None)
        ram = np.zeros(max(n_slots, 1), np.float32)
        rstep = O.adamw_master_step(rp, rm, rv, gh, gdt, rb, float(np.float32(S)), skip, rstep,
                                    *hyper, amax_slot=slots, amax=ram)
        assert int(step.item()) == rstep
        if slots:
            assert np.array_equal(to_host_bits(amax)[:n_slots].view(np.uint32),
                                  ram[:n_slots].view(np.uint32))
    ident = []
    for i in range(n):
        gp, gm, gv = to_host_bits(P[i]), to_host_bits(M[i]), to_host_bits(V[i])
        assert_state_close(gp, rp[i], f"master[{i}]")
        assert_state_close(gm, rm[i], f"exp_avg[{i}]")
        assert_state_close(gv, rv[i], f"exp_avg_sq[{i}]")
        assert_bf16_close(to_host_bits(Bf[i]), rb[i], f"bf16[{i}]")
        ident += [bit_identical_fraction(gp, rp[i]), bit_identical_fraction(gm, rm[i]),
                  bit_identical_fraction(gv, rv[i])]
    for L in (LP, LM, LV, LG, LB):
        L.close()
    return min(ident)


@pytest.mark.parametrize("gdt", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("misalign", [False, True])
def test_adamw_parity(A, dev, gdt, misalign):
    sizes = RAGGED + [3 * 16384 + 5]
    slots = [-1] * len(sizes)
    slots[4], slots[13], slots[-1] = 0, 1, 2
    ident = _adamw_case(A, dev, gdt, misalign, sizes, steps=6,
                        hyper=(1e-3, 0.9, 0.999, 1e-8, 0.01), scales=[65536.0, 1024.0, 3.0],
                        skip_at={2}, slots=slots, seed=20)
    # same operation order on both sides: expect bit-identical fp32 state
    assert ident == 1.0, f"fp32 state not bit-identical (min fraction {ident})"


def test_adamw_gpt2_hyper_no_scale(A, dev):
    """bf16 grads, S fixed 1.0, lr 3e-4, betas (0.9, 0.95), wd 0.1."""
    ident = _adamw_case(A, dev, "bf16", False, [768, 50257, 3 * 768 * 10], steps=10,
                        hyper=(3e-4, 0.9, 0.95, 1e-8, 0.1), scales=[1.0], skip_at=set(),
                        slots=None, seed=21)
    assert ident == 1.0


def test_adamw_bf16_emission_exhaustive_rounding_classes(A, dev):
    """lr = 0 and wd = 0 leave p unchanged, so the bf16 copy is RNE(p) for
    every fp32 p of the rounding-class sweep (ties, near-ties, subnormals,
    inf, NaN, signed zeros)."""
    hi = np.arange(1 << 20, dtype=np.uint64) << 12
    lows = np.array([0, 1, 0x7FF, 0x800, 0x801, 0xFFF], np.uint64)
    p = (hi[:, None] | lows[None, :]).astype(np.uint32).ravel().view(np.float32)
    P = [to_device(p, "f32", dev)]
    M = [torch.zeros(p.size, device=dev)]
    V = [torch.zeros(p.size, device=dev)]
    G = [torch.zeros(p.size, dtype=torch.float16, device=dev)]
    B = [torch.empty(p.size, dtype=torch.bfloat16, device=dev)]
    Ls = [A.amp_tensor_list_create(x) for x in (P, M, V, G, B)]
    step = torch.zeros(1, dtype=torch.int32, device=dev)
    A.amp_adamw_master_step(*Ls, None, None, step, 0.0, 0.9, 0.999, 1e-8, 0.0)
    got = to_host_bits(B[0])
    ref = O.encode("bf16", p)
    assert np.array_equal(got, ref)
    gp = to_host_bits(P[0])
    nan = np.isnan(p)
    assert np.array_equal(gp[~nan].view(np.uint32), p[~nan].view(np.uint32))
    for L in Ls:
        L.close()


@pytest.mark.parametrize("misalign", [False, True])
def test_emit_bf16_parity(A, dev, misalign):
    """amp_emit_bf16: the bf16 working copy of the masters (the rounding-class
    sweep in one tensor, ragged sizes around the chunk, specials at tails)
    equals the oracle's RNE encoder, and the amax folded for slot tensors is
    max|bf16| by the oracle's decoder, NaN propagating."""
    rng = np.random.default_rng(23)
    hi = np.arange(1 << 16, dtype=np.uint64) << 16
    lows = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF], np.uint64)
    sweep = (hi[:, None] | lows[None, :]).astype(np.uint32).ravel().view(np.float32)
    sweep = sweep[np.isfinite(sweep)]
    sizes = RAGGED + [3 * 16384 + 5]
    master_h = [(rng.standard_normal(k) * 0.02).astype(np.float32) for k in sizes] + [sweep]
    master_h[9][256] = np.inf           # +inf in a tail element
    master_h[12][16382] = -np.inf
    master_h[13][0] = np.nan            # NaN: its slot's amax is NaN
    master_h[5][3] = 3.0e38             # rounds to bf16 inf
    slots = [-1] * len(master_h)
    for j, i in enumerate((4, 9, 13, 15, len(master_h) - 1)):
        slots[i] = j
    P = _device_views(master_h, "f32", dev, misalign)
    B = _device_views([np.zeros(h.size, np.uint16) for h in master_h], "bf16", dev, misalign)
    LP, LB = A.amp_tensor_list_create(P), A.amp_tensor_list_create(B)
    A.amp_tensor_list_set_amax_slots(LB, slots)
    amax = torch.zeros(5, device=dev)
    A.amp_emit_bf16(LP, LB, amax)
    got_amax = to_host_bits(amax).view(np.uint32)
    for i, h in enumerate(master_h):
        ref = O.encode("bf16", h)
        assert np.array_equal(to_host_bits(B[i]), ref), i
        assert np.array_equal(to_host_bits(P[i]).view(np.uint32), h.view(np.uint32)), i
        if slots[i] >= 0:
            mag = np.abs(O.decode("bf16", ref))
            want = np.float32(np.nan) if np.isnan(mag).any() else np.float32(mag.max())
            if np.isnan(want):
                assert np.isnan(got_amax.view(np.float32)[slots[i]]), i
            else:
                assert got_amax[slots[i]] == want.view(np.uint32), i
    with pytest.raises(A.AmpError):               # slots but no amax buffer
        A.amp_emit_bf16(LP, LB, None)
    LP.close()
    LB.close()


# -------------------------------------------------------------------- FP8
FP8_SHAPES = [(1, 1), (3, 5), (17, 31), (128, 128), (127, 129), (256, 384), (129, 136),
              (300, 520), (64, 4096), (384, 256)]


def _x_host(rng, rows, cols, xdt, outliers=True):
    x = rng.standard_normal(rows * cols).astype(np.float32)
    if outliers and x.size > 10:
        idx = rng.choice(x.size, size=max(1, x.size // 1000), replace=False)
        x[idx] *= 100
    if xdt == "f32":
        return x
    if xdt == "f16":
        return x.astype(np.float16).view(np.uint16)
    return O.encode("bf16", x)


def _run_quant(A, dev, xh, xdt, rows, cols, fmt, with_t, amax_given=None, skip=None,
               misalign=False):
    x = _device_views([xh], xdt, dev, misalign)[0]
    out = torch.full((rows * cols,), 0xA5, dtype=torch.uint8, device=dev)
    out_t = torch.full((rows * cols,), 0x5A, dtype=torch.uint8, device=dev) if with_t else None
    inv = torch.zeros(1, device=dev)
    amax = torch.tensor([amax_given if amax_given is not None else -1.0], device=dev)
    sk = None if skip is None else torch.tensor([skip], dtype=torch.int32, device=dev)
    A.fp8_quant_tensorwise(x, fmt, out, out_t, inv, amax, amax_given=amax_given is not None,
                           skip_if=sk, rows=rows, cols=cols)
    return (to_host_bits(out), None if out_t is None else to_host_bits(out_t),
            to_host_bits(inv)[0], to_host_bits(amax)[0])


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
@pytest.mark.parametrize("xdt", ["bf16", "f16", "f32"])
def test_fp8_quant_parity(A, dev, fmt, xdt):
    rng = np.random.default_rng(30)
    for rows, cols in FP8_SHAPES:
        xh = _x_host(rng, rows, cols, xdt)
        for with_t in (True, False):
            for misalign in ((False, True) if rows * cols > 8 else (False,)):
                q, qt, inv, am = _run_quant(A, dev, xh, xdt, rows, cols, fmt, with_t,
                                            misalign=misalign)
                rq, rqt, rinv, ram = O.fp8_quant_tensorwise(xh, xdt, rows, cols, fmt,
                                                            transposed=with_t)
                key = (rows, cols, with_t, misalign)
                assert am == np.float32(ram), key
                assert np.float32(inv).view(np.uint32) == np.float32(rinv).view(np.uint32), key
                assert np.array_equal(q, rq), key
                if with_t:
                    assert np.array_equal(qt, rqt), key


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
def test_fp8_quant_degenerate_cases(A, dev, fmt):
    rng = np.random.default_rng(31)
    # all-zero tensor: amax clamps to EPS, all bytes zero
    z = np.zeros(256 * 128, np.uint16)
    q, qt, inv, am = _run_quant(A, dev, z, "bf16", 256, 128, fmt, True)
    rq, rqt, rinv, _ = O.fp8_quant_tensorwise(z, "bf16", 256, 128, fmt)
    assert am == 0.0 and not q.any() and not qt.any() and inv == np.float32(rinv)
    # given amax (delayed-style): values beyond it saturate; inf saturates
    xh = _x_host(rng, 128, 256, "f32")
    xh[5] = np.inf
    xh[77] = -np.inf
    for given in (0.5, 3.0, 1e-20):
        q, qt, inv, _ = _run_quant(A, dev, xh, "f32", 128, 256, fmt, True, amax_given=given)
        rq, rqt, rinv, _ = O.fp8_quant_tensorwise(xh, "f32", 128, 256, fmt, amax=given)
        assert np.array_equal(q, rq) and np.array_equal(qt, rqt) and inv == np.float32(rinv)
    # a NaN input: amax is NaN, every byte is the NaN code
    xn = _x_host(rng, 128, 128, "bf16")
    xn[1000] = 0x7FC1
    q, qt, inv, am = _run_quant(A, dev, xn, "bf16", 128, 128, fmt, True)
    rq, rqt, rinv, ram = O.fp8_quant_tensorwise(xn, "bf16", 128, 128, fmt)
    assert np.isnan(am) and np.isnan(ram) and np.isnan(inv) and np.isnan(rinv)
    assert np.array_equal(q, rq) and np.array_equal(qt, rqt)
    # amax = inf: finite values go to signed zero, the infinite one to NaN
    xi = _x_host(rng, 128, 128, "f32")
    xi[3] = -np.inf
    q, qt, inv, am = _run_quant(A, dev, xi, "f32", 128, 128, fmt, True)
    rq, rqt, rinv, ram = O.fp8_quant_tensorwise(xi, "f32", 128, 128, fmt)
    assert np.isinf(am) and np.array_equal(q, rq) and np.array_equal(qt, rqt)
    # empty tensor
    q, qt, inv, am = _run_quant(A, dev, np.zeros(0, np.uint16), "bf16", 0, 7, fmt, True)
    assert am == 0.0 and inv == np.float32(O.fp8_quant_tensorwise(np.zeros(0, np.uint16), "bf16",
                                                                  0, 7, fmt)[2])
    # skip flag set: nothing written, the amax output included
    q, qt, inv, am = _run_quant(A, dev, xh, "f32", 128, 256, fmt, True, amax_given=1.0, skip=1)
    assert np.all(q == 0xA5) and np.all(qt == 0x5A) and inv == 0.0
    q, qt, inv, am = _run_quant(A, dev, xh, "f32", 128, 256, fmt, True, skip=1)
    assert np.all(q == 0xA5) and np.all(qt == 0x5A) and inv == 0.0 and am == -1.0


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
def test_fp8_cast_rounding_classes(A, dev, fmt):
    """With amax = fp8_max the scale is exactly 1, so each byte is the
    saturating RNE cast of the fp32 input itself: every sign / exponent /
    kept-fraction combination with round and sticky bits clear, set and tied."""
    hi = np.arange(1 << 20, dtype=np.uint64) << 12
    lows = np.array([0, 1, 0x7FF, 0x800, 0x801, 0xFFF], np.uint64)
    x = (hi[:, None] | lows[None, :]).astype(np.uint32).ravel().view(np.float32)
    cols = 4096
    rows = x.size // cols
    x = x[:rows * cols]
    fmax = O.fmt_max(fmt)
    q, qt, inv, _ = _run_quant(A, dev, x, "f32", rows, cols, fmt, True, amax_given=fmax)
    rq, rqt, rinv, _ = O.fp8_quant_tensorwise(x, "f32", rows, cols, fmt, amax=fmax)
    assert inv == 1.0 == rinv
    assert np.array_equal(q, rq)
    assert np.array_equal(qt, rqt)


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
@pytest.mark.parametrize("xdt", ["bf16", "f16", "f32"])
def test_fp8_quant_list_parity(A, dev, fmt, xdt):
    tdt = torch.float8_e4m3fn if fmt == "e4m3fn" else torch.float8_e5m2
    rng = np.random.default_rng(32)
    shapes = [(128, 256), (1024, 512), (127, 129), (384, 128), (64, 4096)]
    xs_h = [_x_host(rng, r, c, xdt) for r, c in shapes]
    X = [to_device(h, xdt, dev).view(r, c) for h, (r, c) in zip(xs_h, shapes)]
    Q = [torch.empty((r, c), dtype=tdt, device=dev) for r, c in shapes]
    QT = [torch.empty((c, r), dtype=tdt, device=dev) for r, c in shapes]
    LX, LQ, LQT = (A.amp_tensor_list_create(t, two_d=True) for t in (X, Q, QT))
    dec = (lambda h: h) if xdt == "f32" else (lambda h: O.decode(xdt, h))
    amax_h = np.array([np.abs(dec(h)).max() for h in xs_h], np.float32)
    amax_h[1] *= 0.5     # a given amax below the data: saturation path
    amax = torch.from_numpy(amax_h).to(dev)
    inv = torch.zeros(len(shapes), device=dev)
    for skip in (1, 0):
        fi = torch.tensor([skip], dtype=torch.int32, device=dev)
        A.fp8_quant_tensorwise_list(LX, LQ, LQT, fmt, amax, inv, skip_if=fi)
        if skip:
            assert not inv.any()
    for i, (r, c) in enumerate(shapes):
        rq, rqt, rinv, _ = O.fp8_quant_tensorwise(xs_h[i], xdt, r, c, fmt,
                                                  amax=float(amax_h[i]))
        assert np.array_equal(to_host_bits(Q[i].view(torch.uint8)).ravel(), rq), i
        assert np.array_equal(to_host_bits(QT[i].view(torch.uint8)).ravel(), rqt), i
        assert to_host_bits(inv)[i] == np.float32(rinv)
    for L in (LX, LQ, LQT):
        L.close()


# ------------------------------------------------------------ composition
@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
def test_amp_step_composition_with_fp8(A, dev, fmt):
    """The four calls of a step, with FP8 weights and an inf at step 3,
    against the oracle's step in the pages' order."""
    from loss_scaling_master_gb300 import AmpOptimizerStep
    rng = np.random.default_rng(40)
    shapes = [(96, 256), (300,), (128, 136), (1000,), (256, 512)]
    fp8_shapes = [s if len(s) == 2 else None for s in shapes]
    sizes = [int(np.prod(s)) for s in shapes]
    master = [(rng.standard_normal(n) * 0.02).astype(np.float32) for n in sizes]
    G = [torch.empty(n, dtype=torch.float16, device=dev) for n in sizes]
    hyper = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    st = AmpOptimizerStep([torch.from_numpy(m.copy()).to(dev) for m in master], G,
                          init_scale=65536.0, growth_interval=2, fp8_shapes=fp8_shapes,
                          fp8_format=fmt, **hyper)
    orc = O.AmpStepOracle(master, "f16", hyper["lr"], hyper["beta1"], hyper["beta2"],
                          hyper["eps"], hyper["weight_decay"], 65536.0, 2.0, 0.5, 2,
                          fp8_shapes=fp8_shapes, fp8_format=fmt)
    for i, sh in enumerate(fp8_shapes):              # the first working copies
        assert np.array_equal(to_host_bits(st.bf16[i]), orc.bf16[i]), i
        if sh is not None:
            j = orc.slots[i]
            assert np.array_equal(to_host_bits(st.fp8[j].view(torch.uint8)).ravel(), orc.fp8[i])
            assert np.array_equal(to_host_bits(st.fp8_t[j].view(torch.uint8)).ravel(), orc.fp8_t[i])
            assert to_host_bits(st.inv_scale)[j] == orc.inv_scale[j]
    assert not to_host_bits(st.amax).any()
    for k in range(1, 8):
        gh = [(rng.standard_normal(n) * 1e-4 * orc.scale).astype(np.float16).view(np.uint16)
              for n in sizes]
        if k == 3:
            gh[2][135] = 0x7C00
        for t, h in zip(G, gh):
            t.copy_(to_device(h, "f16", dev))
        st.step()
        orc.run(gh)
        s = st.state()
        assert (s["scale"], s["growth_tracker"], s["step"], s["found_inf"]) == \
            (orc.scale, orc.tracker, orc.step, 0), k
    for i in range(len(shapes)):
        assert np.array_equal(to_host_bits(st.master[i]).view(np.uint32),
                              orc.master[i].view(np.uint32))
        assert np.array_equal(to_host_bits(st.bf16[i]), orc.bf16[i])
    j = 0
    for i, sh in enumerate(fp8_shapes):
        if sh is None:
            continue
        assert np.array_equal(to_host_bits(st.fp8[j].view(torch.uint8)).ravel(), orc.fp8[i])
        assert np.array_equal(to_host_bits(st.fp8_t[j].view(torch.uint8)).ravel(), orc.fp8_t[i])
        assert to_host_bits(st.inv_scale)[j] == orc.inv_scale[orc.slots[i]]
        j += 1
    st.close()


@pytest.mark.parametrize("mode", ["dynamic", "delayed", "clip", "sr", "health", "sr_fp8",
                                  "sr_delayed", "sr_clip"])
def test_graph_replay_matches_eager(A, dev, mode):
    """The step captured once in a CUDA graph (with its programmatic launch
    edges) and replayed gives the same bits as the eager calls, including a
    skipped step, for every form of the step."""
    from loss_scaling_master_gb300 import AmpOptimizerStep
    rng = np.random.default_rng(41)
    shapes = [(128, 256), (777,), (256, 384)]
    fp8_shapes = [s if len(s) == 2 else None for s in shapes]
    sizes = [int(np.prod(s)) for s in shapes]
    master = [(rng.standard_normal(n) * 0.02).astype(np.float32) for n in sizes]
    hyper = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    opts = {"dynamic": {}, "delayed": {"fp8_scaling": "delayed", "amax_history_len": 2},
            "clip": {"max_norm": 0.05}, "sr": {"sr_seed": 77, "fp8_shapes": None},
            "health": {"min_scale": 600.0}, "sr_fp8": {"sr_seed": 78},
            "sr_delayed": {"sr_seed": 79, "fp8_scaling": "delayed", "amax_history_len": 2},
            "sr_clip": {"sr_seed": 80, "max_norm": 0.05}}[mode]
    kw = dict(fp8_shapes=fp8_shapes)
    kw.update(opts)
    mk = lambda: AmpOptimizerStep([torch.from_numpy(m.copy()).to(dev) for m in master],
                                  [torch.empty(n, dtype=torch.float16, device=dev) for n in sizes],
                                  init_scale=1024.0, growth_interval=3, **kw, **hyper)
    eager, graphed = mk(), mk()
    graphed.capture_graph()
    for k in range(6):
        gh = [(rng.standard_normal(n) * 1e-3 * 1024).astype(np.float16).view(np.uint16)
              for n in sizes]
        if k == 2:
            gh[1][776] = 0x7E00
        for st in (eager, graphed):
            for t, h in zip(st.grads, gh):
                t.copy_(to_device(h, "f16", dev))
            st.step()
        torch.cuda.synchronize()
        assert eager.state() == graphed.state()
    for a, b in zip(eager.master + eager.exp_avg + eager.exp_avg_sq + eager.bf16,
                    graphed.master + graphed.exp_avg + graphed.exp_avg_sq + graphed.bf16):
        assert torch.equal(a.view(torch.int16 if a.element_size() == 2 else torch.int32),
                           b.view(torch.int16 if b.element_size() == 2 else torch.int32))
    for a, b in zip(eager.fp8 + eager.fp8_t, graphed.fp8 + graphed.fp8_t):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    if eager.n_fp8:
        assert torch.equal(eager.inv_scale, graphed.inv_scale)
    if mode == "health":
        assert eager.health() == graphed.health() == 2       # 1024 halved below 600 at the skip
    eager.close()
    graphed.close()


# ------------------------------------------------------ grad-norm clipping
@pytest.mark.parametrize("dt", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("misalign", [False, True])
def test_grad_norm_parity_and_determinism(A, dev, dt, misalign):
    """Sum of squared unscaled gradients vs the oracle's fp64 sequential sum.
    Tolerance: squares of 16-bit values are exact in fp32; a chain of four
    fused multiply-adds plus the pair add costs <= 4 ulp, the compensated
    per-thread sum <= 2 ulp, every later addition is fp64 (6 ulp of fp32 =
    3.6e-7, plus 2 ulp when 1/S is not a power of two); rel 1e-6 bounds it.
    Repeated calls are bit-identical."""
    rng = np.random.default_rng(50)
    for scale in (65536.0, 1.0, 1000.0):
        hl = _grads_host(rng, RAGGED + [3 * 16384 + 5], dt, sigma=0.01 * scale)
        tensors = _device_views(hl, dt, dev, misalign)
        L = A.amp_tensor_list_create(tensors)
        fi = torch.zeros(1, dtype=torch.int32, device=dev)
        ss = torch.zeros(1, dtype=torch.float64, device=dev)
        A.amp_unscale_check_norm(L, torch.tensor([scale], device=dev), fi, ss)
        first = ss.item()
        A.amp_unscale_check_norm(L, torch.tensor([scale], device=dev), fi, ss)
        assert ss.item() == first
        ref = O.grad_sumsq(hl, dt, scale)
        assert abs(first - ref) <= 1e-6 * ref, (scale, first, ref)
        assert int(fi.item()) == 0
        hl[3][1] = _inf_bits(dt, np.inf)
        bad = _device_views(hl, dt, dev, misalign)
        Lb = A.amp_tensor_list_create(bad)
        A.amp_unscale_check_norm(Lb, torch.tensor([scale], device=dev), fi, ss)
        assert int(fi.item()) == 1 and not np.isfinite(ss.item())
        L.close()
        Lb.close()


@pytest.mark.parametrize("gdt,with_fp8", [("f16", False), ("bf16", False), ("f32", False),
                                          ("f16", True)])
def test_clipped_step_composition(A, dev, gdt, with_fp8, monkeypatch):
    """AmpOptimizerStep with max_norm vs the oracle's step with clipping, over
    steps where the factor is < 1, = 1 and a skipped step; every grad dtype,
    and once with FP8 weights cast after the clipped update.

    The clip factor comes from a sum of squares that matches the oracle within
    a tolerance, so the GPU's bf16 copy may differ from the oracle's by the
    allowed 1 ulp.  The FP8 cast after it is exact given its input, so on
    every step that is not skipped the FP8 bytes, the transposed bytes and
    inv_scale are compared with the oracle's quantizer run on the GPU's own
    bf16 copy, and the GPU's folded amax with max|bf16| of that copy."""
    from loss_scaling_master_gb300 import AmpOptimizerStep
    from loss_scaling_master_gb300 import step as step_mod
    snap = {}
    real_update = step_mod.A.amp_update_scale

    def spy_update(*args, amax=None, **kw):
        if amax is not None:
            snap["amax"] = amax.clone()      # enqueued on the step's stream, before the clear
        return real_update(*args, amax=amax, **kw)

    monkeypatch.setattr(step_mod.A, "amp_update_scale", spy_update)
    rng = np.random.default_rng(51)
    sizes = [1000, 4096, 257, 40000]
    fp8_shapes = [None, (64, 64), None, (200, 200)] if with_fp8 else None
    master = [(rng.standard_normal(n) * 0.02).astype(np.float32) for n in sizes]
    hyper = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[gdt]
    st = AmpOptimizerStep([torch.from_numpy(m.copy()).to(dev) for m in master],
                          [torch.empty(n, dtype=tdt, device=dev) for n in sizes],
                          init_scale=65536.0, growth_interval=3, max_norm=0.5,
                          fp8_shapes=fp8_shapes, **hyper)
    orc = O.AmpStepOracle(master, gdt, hyper["lr"], hyper["beta1"], hyper["beta2"], hyper["eps"],
                          hyper["weight_decay"], 65536.0, 2.0, 0.5, 3, max_norm=0.5,
                          fp8_shapes=fp8_shapes)
    for k in range(6):
        sigma = (1e-2 if k % 2 == 0 else 1e-5) * orc.scale      # clipped, then unclipped
        gh = [(rng.standard_normal(n) * sigma).astype(np.float32) for n in sizes]
        gh = [g.astype(np.float16).view(np.uint16) if gdt == "f16" else
              (O.encode("bf16", g) if gdt == "bf16" else g) for g in gh]
        if k == 3:
            gh[2][100] = _inf_bits(gdt, np.inf)
        for t, h in zip(st.grads, gh):
            t.copy_(to_device(h, gdt, dev))
        st.step()
        orc.run(gh)
        s = st.state()
        assert (s["scale"], s["growth_tracker"], s["step"]) == (orc.scale, orc.tracker, orc.step)
        if k != 3:
            assert abs(np.sqrt(st.grad_sumsq.item()) - orc.grad_norm) <= 1e-6 * orc.grad_norm
        if with_fp8 and k != 3:
            gpu_amax = to_host_bits(snap["amax"])
            n_cmp, j = 0, 0
            for i, sh in enumerate(fp8_shapes):
                if sh is None:
                    continue
                gb = to_host_bits(st.bf16[i])
                assert_bf16_close(gb, orc.bf16[i], f"bf16[{i}] step {k}")
                mag = np.abs(O.decode("bf16", gb))
                ref_amax = np.float32(np.nan) if np.isnan(mag).any() else mag.max()
                assert gpu_amax[j].view(np.uint32) == np.float32(ref_amax).view(np.uint32), (k, i)
                q, qt, inv, _ = O.fp8_quant_tensorwise(gb, "bf16", sh[0], sh[1], "e4m3fn",
                                                       1e-12, True, amax=float(gpu_amax[j]))
                assert np.array_equal(to_host_bits(st.fp8[j].view(torch.uint8)).ravel(), q), (k, i)
                assert np.array_equal(to_host_bits(st.fp8_t[j].view(torch.uint8)).ravel(), qt), (k, i)
                assert to_host_bits(st.inv_scale)[j].view(np.uint32) == \
                    np.float32(inv).view(np.uint32), (k, i)
                n_cmp += 1
                j += 1
            assert n_cmp == 2
    for i in range(len(sizes)):
        assert_state_close(to_host_bits(st.master[i]), orc.master[i], f"master[{i}]")
        assert_state_close(to_host_bits(st.exp_avg[i]), orc.exp_avg[i], f"exp_avg[{i}]")
        assert_state_close(to_host_bits(st.exp_avg_sq[i]), orc.exp_avg_sq[i], f"exp_avg_sq[{i}]")
        assert_bf16_close(to_host_bits(st.bf16[i]), orc.bf16[i], f"bf16[{i}]")
    st.close()


# ------------------------------------------------------ delayed FP8 scaling
@pytest.mark.parametrize("hist_len,fmt", [(1, "e4m3fn"), (3, "e4m3fn"), (3, "e5m2")])
@pytest.mark.parametrize("gdt", ["f16", "bf16", "f32"])
def test_delayed_fp8_step_composition(A, dev, hist_len, gdt, fmt):
    """AdamW + bf16 + FP8 in one pass with the delayed scale vs the oracle's
    step: full tiles (vector path), ragged edge tiles and a tensor whose
    column count breaks 16-byte rows (element path), a skipped step."""
    from loss_scaling_master_gb300 import AmpOptimizerStep
    rng = np.random.default_rng(70 + hist_len)
    shapes = [(256, 512), (300,), (96, 256), (128, 136), (1000,), (130, 52), (384, 128)]
    fp8_shapes = [s if len(s) == 2 else None for s in shapes]
    sizes = [int(np.prod(s)) for s in shapes]
    master = [(rng.standard_normal(n) * 0.02).astype(np.float32) for n in sizes]
    hyper = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[gdt]
    st = AmpOptimizerStep([torch.from_numpy(m.copy()).to(dev) for m in master],
                          [torch.empty(n, dtype=tdt, device=dev) for n in sizes],
                          init_scale=4096.0, growth_interval=3, fp8_shapes=fp8_shapes,
                          fp8_scaling="delayed", amax_history_len=hist_len, fp8_format=fmt,
                          **hyper)
    orc = O.AmpStepOracle(master, gdt, hyper["lr"], hyper["beta1"], hyper["beta2"], hyper["eps"],
                          hyper["weight_decay"], 4096.0, 2.0, 0.5, 3, fp8_shapes=fp8_shapes,
                          fp8_scaling="delayed", hist_len=hist_len, fp8_format=fmt)

    def check_fp8():
        j = 0
        for i, sh in enumerate(fp8_shapes):
            if sh is None:
                continue
            assert np.array_equal(to_host_bits(st.fp8[j].view(torch.uint8)).ravel(), orc.fp8[i]), i
            assert np.array_equal(to_host_bits(st.fp8_t[j].view(torch.uint8)).ravel(), orc.fp8_t[i]), i
            assert to_host_bits(st.inv_scale)[j] == orc.inv_scale[orc.slots[i]], i
            j += 1
        assert np.array_equal(to_host_bits(st.amax_history), orc.hist)

    torch.cuda.synchronize()
    for i in range(len(shapes)):                     # the first working copies (amp_emit_bf16)
        assert np.array_equal(to_host_bits(st.bf16[i]), orc.bf16[i]), i
    check_fp8()                                      # the seeding cast
    for k in range(6):
        sigma = 1e-3 * orc.scale
        gh = [(rng.standard_normal(n) * sigma).astype(np.float32) for n in sizes]
        gh = [g.astype(np.float16).view(np.uint16) if gdt == "f16" else
              (O.encode("bf16", g) if gdt == "bf16" else g) for g in gh]
        if k == 3:
            gh[3][17] = _inf_bits(gdt, np.inf)
        for t, h in zip(st.grads, gh):
            t.copy_(to_device(h, gdt, dev))
        st.step()
        orc.run(gh)
        s = st.state()
        assert (s["scale"], s["growth_tracker"], s["step"]) == (orc.scale, orc.tracker, orc.step)
        check_fp8()
    for i in range(len(shapes)):
        assert np.array_equal(to_host_bits(st.master[i]).view(np.uint32), orc.master[i].view(np.uint32))
        assert np.array_equal(to_host_bits(st.exp_avg[i]).view(np.uint32), orc.exp_avg[i].view(np.uint32))
        assert np.array_equal(to_host_bits(st.bf16[i]), orc.bf16[i])
    st.close()


# ----------------------------------------------------------- rowwise FP8
def _run_rowwise(A, dev, xh, xdt, rows, cols, fmt, with_t, skip=None, misalign=False):
    x = _device_views([xh], xdt, dev, misalign)[0].view(rows, cols)
    o = {"q": torch.full((rows * cols,), 0xA5, dtype=torch.uint8, device=dev)}
    o.update({k: torch.full((rows,), -1.0, device=dev) for k in ("amax_row", "scale_row", "inv_row")})
    if with_t:
        o["q_t"] = torch.full((rows * cols,), 0x5A, dtype=torch.uint8, device=dev)
        o.update({k: torch.full((cols,), -1.0, device=dev) for k in ("amax_col", "scale_col", "inv_col")})
    sk = None if skip is None else torch.tensor([skip], dtype=torch.int32, device=dev)
    A.fp8_quant_rowwise(x, fmt, o["q"], o.get("q_t"), o["amax_row"], o["scale_row"], o["inv_row"],
                        o.get("amax_col"), o.get("scale_col"), o.get("inv_col"), skip_if=sk)
    return {k: to_host_bits(v) for k, v in o.items()}


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
@pytest.mark.parametrize("xdt", ["bf16", "f16", "f32"])
def test_fp8_rowwise_parity(A, dev, fmt, xdt):
    rng = np.random.default_rng(90)
    for rows, cols in FP8_SHAPES:
        xh = _x_host(rng, rows, cols, xdt)
        if rows > 3:                       # a zero row: its scale clamps to EPS
            if xdt == "f32":
                xh.reshape(rows, cols)[2] = 0
            else:
                xh.reshape(rows, cols)[2] = 0
        for with_t in (True, False):
            for misalign in ((False, True) if rows * cols > 8 else (False,)):
                got = _run_rowwise(A, dev, xh, xdt, rows, cols, fmt, with_t, misalign=misalign)
                ref = O.fp8_quant_rowwise(xh, xdt, rows, cols, fmt, transposed=with_t)
                key = (rows, cols, with_t, misalign)
                for k in ref:
                    if ref[k].dtype == np.float32:
                        assert np.array_equal(got[k].view(np.uint32), ref[k].view(np.uint32)), (k, key)
                    else:
                        assert np.array_equal(got[k], ref[k]), (k, key)


@pytest.mark.parametrize("xdt", ["bf16", "f32"])
@pytest.mark.parametrize("rows,cols", [(8256, 2056), (16, 76800), (76800, 8)])
def test_fp8_rowwise_strip_walks(A, dev, xdt, rows, cols):
    """The maxima pass gives each column strip S CTAs, each taking every S-th
    tile row of its strip: [8256, 2056] gives every CTA several tiles with a
    ragged last tile row and a ragged last strip in the same walk; [16, 76800]
    has more strips than CTAs fit at once (S = 1); [76800, 8] has one narrow
    strip and hundreds of CTAs on it.  Every byte and scale equals the
    oracle's."""
    rng = np.random.default_rng(93)
    xh = _x_host(rng, rows, cols, xdt)
    got = _run_rowwise(A, dev, xh, xdt, rows, cols, "e4m3fn", True)
    ref = O.fp8_quant_rowwise(xh, xdt, rows, cols, "e4m3fn")
    _assert_same(got, ref, f"rowwise strips {rows}x{cols}")


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
def test_fp8_rowwise_degenerate(A, dev, fmt):
    rng = np.random.default_rng(91)
    rows, cols = 256, 384
    xh = _x_host(rng, rows, cols, "f32")
    xh[5 * cols + 7] = np.nan            # row 5 and column 7 become NaN; others unaffected
    xh[9 * cols + 100] = -np.inf         # row 9 and column 100: amax inf
    got = _run_rowwise(A, dev, xh, "f32", rows, cols, fmt, True)
    ref = O.fp8_quant_rowwise(xh, "f32", rows, cols, fmt)
    assert np.array_equal(got["q"], ref["q"]) and np.array_equal(got["q_t"], ref["q_t"])
    for k in ("amax_row", "scale_row", "inv_row", "amax_col", "scale_col", "inv_col"):
        g, r = got[k], ref[k]
        assert np.array_equal(np.isnan(g), np.isnan(r)), k
        assert np.array_equal(g[~np.isnan(r)], r[~np.isnan(r)]), k
    skipped = _run_rowwise(A, dev, xh, "f32", rows, cols, fmt, True, skip=1)
    assert np.all(skipped["q"] == 0xA5) and np.all(skipped["q_t"] == 0x5A)
    assert np.all(skipped["amax_row"] == -1.0) and np.all(skipped["inv_col"] == -1.0)


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
@pytest.mark.parametrize("xdt", ["bf16", "f16"])
def test_fp8_rowwise_nonfinite_16bit(A, dev, fmt, xdt):
    """16-bit x with NaNs of both signs and several payloads, +-inf,
    subnormals and -0: the rows and columns they touch get NaN or zero scales
    and (canonical) NaN bytes; every other row and column is unaffected."""
    rng = np.random.default_rng(150)
    rows, cols = 384, 512
    xh = _x_host(rng, rows, cols, xdt).reshape(rows, cols).copy()
    if xdt == "bf16":
        specials = [0x7FC0, 0xFFC0, 0x7F81, 0xFFFF, 0x7F80, 0xFF80, 0x0001, 0x807F, 0x8000]
    else:
        specials = [0x7E00, 0xFE00, 0x7C01, 0xFFFF, 0x7C00, 0xFC00, 0x0001, 0x83FF, 0x8000]
    for v in specials:
        i, j = rng.integers(0, rows), rng.integers(0, cols)
        xh[i, j] = v
    xh[200, :] = specials[6]            # a row of subnormals only
    xh[:, 300] = specials[8]            # a column of -0 only
    xh = xh.ravel()
    got = _run_rowwise(A, dev, xh, xdt, rows, cols, fmt, True)
    ref = O.fp8_quant_rowwise(xh, xdt, rows, cols, fmt)
    _assert_same(got, ref, "rowwise nonfinite")


# ------------------------------------------------------ stochastic rounding
@pytest.mark.parametrize("misalign", [False, True])
def test_adamw_stochastic_rounding_parity(A, dev, misalign):
    """The bf16 copy rounded stochastically with the Philox4x32-10 stream of
    each element: bit-identical to the oracle's (same published generator,
    written separately) over several steps with a skip; the master state is
    the RNE step's."""
    rng = np.random.default_rng(95)
    sizes = [1, 7, 257, 4096, 16385, 40000]
    seed = 0x1234_5678_9ABC_DEF0
    master_h = [(rng.standard_normal(k) * 0.02).astype(np.float32) for k in sizes]
    P = _device_views(master_h, "f32", dev, misalign)
    M = _device_views([np.zeros(k, np.float32) for k in sizes], "f32", dev, misalign)
    V = _device_views([np.zeros(k, np.float32) for k in sizes], "f32", dev, misalign)
    G = _device_views(_grads_host(rng, sizes, "f16"), "f16", dev, misalign)
    B = _device_views([np.zeros(k, np.uint16) for k in sizes], "bf16", dev, misalign)
    Ls = [A.amp_tensor_list_create(x) for x in (P, M, V, G, B)]
    A.amp_tensor_list_set_amax_slots(Ls[4], [0, -1, -1, 1, -1, 2])
    amax = torch.zeros(3, device=dev)
    step = torch.zeros(1, dtype=torch.int32, device=dev)
    fi = torch.zeros(1, dtype=torch.int32, device=dev)
    rp, rm, rv = [x.copy() for x in master_h], [np.zeros(k, np.float32) for k in sizes], \
        [np.zeros(k, np.float32) for k in sizes]
    rb = [np.zeros(k, np.uint16) for k in sizes]
    rstep = 0
    for k in range(4):
        gh = _grads_host(rng, sizes, "f16", sigma=1e-3 * 1024)
        for t, h in zip(G, gh):
            t.copy_(to_device(h, "f16", dev))
        skip = int(k == 2)
        fi.fill_(skip)
        amax.zero_()
        A.amp_adamw_master_step_sr(*Ls, torch.tensor([1024.0], device=dev), fi, step,
                                   1e-3, 0.9, 0.999, 1e-8, 0.01, seed, amax=amax)
        ram = np.zeros(3, np.float32)
        rstep = O.adamw_master_step(rp, rm, rv, gh, "f16", rb, 1024.0, skip, rstep, 1e-3, 0.9,
                                    0.999, 1e-8, 0.01, amax_slot=[0, -1, -1, 1, -1, 2], amax=ram,
                                    sr_seed=seed)
        assert int(step.item()) == rstep
        assert np.array_equal(to_host_bits(amax).view(np.uint32), ram.view(np.uint32))
    for i in range(len(sizes)):
        assert np.array_equal(to_host_bits(P[i]).view(np.uint32), rp[i].view(np.uint32))
        assert np.array_equal(to_host_bits(B[i]), rb[i]), i
    for L in Ls:
        L.close()


def test_stochastic_rounding_unbiased_on_gpu(A, dev):
    """E[bf16_sr(p)] = p: the mean of the stochastically rounded copy of a
    constant master over 4M elements sits within 5 sigma of the master."""
    n = 1 << 22
    p = torch.full((n,), 1.0 + 1e-3, device=dev)
    Ls = [A.amp_tensor_list_create([t]) for t in
          (p, torch.zeros(n, device=dev), torch.zeros(n, device=dev),
           torch.zeros(n, dtype=torch.float16, device=dev),
           torch.empty(n, dtype=torch.bfloat16, device=dev))]
    step = torch.zeros(1, dtype=torch.int32, device=dev)
    # lr = 0, wd = 0: p stays, the copy is SR(p)
    A.amp_adamw_master_step_sr(*Ls, None, None, step, 0.0, 0.9, 0.999, 1e-8, 0.0, 42)
    b = Ls[4].tensors[0].float().double()
    lo, hi = 1.0, 1.0 + 2.0 ** -7
    frac = (float(np.float32(1.0 + 1e-3)) - lo) / (hi - lo)
    assert set(torch.unique(b).tolist()) <= {lo, hi}
    sigma = (hi - lo) * np.sqrt(frac * (1 - frac) / n)
    assert abs(b.mean().item() - float(np.float32(1.0 + 1e-3))) < 5 * sigma
    for L in Ls:
        L.close()


# ------------------------------------------- stochastic rounding of FP8 copies
@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
@pytest.mark.parametrize("xdt", ["bf16", "f16", "f32"])
def test_fp8_list_stochastic_parity(A, dev, fmt, xdt):
    """fp8_quant_tensorwise_list_sr: every byte of both layouts and every
    inv_scale equal to the oracle's stochastic quantizer (same published
    generator, written separately), on full, ragged and misaligned-row tiles,
    with NaN, inf, zeros and values in the FP8 subnormal range; a set skip flag
    writes nothing; the tensor word of the random counter is the list index."""
    rng = np.random.default_rng(160)
    shapes = [(128, 128), (127, 129), (256, 384), (33, 40), (1, 1), (130, 52)]
    seed, t = 0xDEADBEEF_0BADF00D, 13
    xs, xh = [], []
    for (r, c) in shapes:
        h = _x_host(rng, r, c, xdt)
        if r * c > 64:
            flat = h.reshape(-1)
            flat[3] = _inf_bits(xdt, np.inf)
            flat[5] = _inf_bits(xdt, -np.inf) if r != 33 else flat[5]
            flat[7] = _inf_bits(xdt, np.nan) if (r, c) == (256, 384) else flat[7]
            if xdt == "f32":
                flat[9] = np.float32(1e-30)
        xh.append(h)
        xs.append(to_device(h, xdt, dev).view(r, c))
    LX = A.amp_tensor_list_create(xs, True)
    tdt = torch.float8_e4m3fn if fmt == "e4m3fn" else torch.float8_e5m2
    Q = [torch.full((r, c), 0x5A, dtype=torch.uint8, device=dev).view(tdt) for r, c in shapes]
    QT = [torch.full((c, r), 0xA5, dtype=torch.uint8, device=dev).view(tdt) for r, c in shapes]
    LQ, LQT = A.amp_tensor_list_create(Q, True), A.amp_tensor_list_create(QT, True)
    # amax per tensor from the oracle's quantizer (the list takes it as given)
    amax_h = np.array([O.fp8_quant_tensorwise(h, xdt, r, c, fmt)[3] for h, (r, c) in
                       zip(xh, shapes)], np.float32)
    amax_h[1] = 0.75 * amax_h[1]                        # a delayed amax: values saturate
    amax = torch.from_numpy(amax_h).to(dev)
    inv = torch.zeros(len(shapes), device=dev)
    step = torch.tensor([t], dtype=torch.int32, device=dev)
    skip = torch.ones(1, dtype=torch.int32, device=dev)
    A.fp8_quant_tensorwise_list_sr(LX, LQ, LQT, fmt, amax, inv, seed, step, skip_if=skip)
    torch.cuda.synchronize()
    assert all(int(q.view(torch.uint8).unique().item()) == 0x5A for q in Q)
    A.fp8_quant_tensorwise_list_sr(LX, LQ, LQT, fmt, amax, inv, seed, step)
    for j, (h, (r, c)) in enumerate(zip(xh, shapes)):
        q, qt, rinv, _ = O.fp8_quant_tensorwise_sr(h, xdt, r, c, fmt, seed, t, j,
                                                   amax=float(amax_h[j]))
        assert np.array_equal(to_host_bits(Q[j].view(torch.uint8)).ravel(), q), (j, r, c)
        assert np.array_equal(to_host_bits(QT[j].view(torch.uint8)).ravel(), qt), (j, r, c)
        gi = to_host_bits(inv)[j]
        if np.isnan(rinv):                    # an fp32 NaN's payload is open: by position
            assert np.isnan(gi), j
        else:
            assert gi.view(np.uint32) == np.float32(rinv).view(np.uint32), j
    for L in (LX, LQ, LQT):
        L.close()


@pytest.mark.parametrize("mode,fmt", [("dynamic", "e4m3fn"), ("dynamic", "e5m2"),
                                      ("delayed", "e4m3fn"), ("delayed", "e5m2")])
def test_stochastic_step_composition(A, dev, mode, fmt):
    """AmpOptimizerStep(sr_seed) with FP8 weights, dynamic or delayed scaling,
    against the oracle's step with the same seed: master, m, v, the bf16 copy,
    the FP8 bytes of both layouts and inv_scale bit-identical over several
    steps with a skip."""
    from loss_scaling_master_gb300 import AmpOptimizerStep
    rng = np.random.default_rng(161)
    shapes = [(256, 512), (300,), (96, 256), (128, 136), (1000,), (130, 52)]
    fp8_shapes = [s if len(s) == 2 else None for s in shapes]
    sizes = [int(np.prod(s)) for s in shapes]
    master = [(rng.standard_normal(n) * 0.02).astype(np.float32) for n in sizes]
    hyper = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    seed = 0x5EED_0000_1234_5678
    st = AmpOptimizerStep([torch.from_numpy(m.copy()).to(dev) for m in master],
                          [torch.empty(n, dtype=torch.float16, device=dev) for n in sizes],
                          init_scale=4096.0, growth_interval=3, fp8_shapes=fp8_shapes,
                          fp8_scaling=mode, amax_history_len=2, fp8_format=fmt, sr_seed=seed,
                          **hyper)
    orc = O.AmpStepOracle(master, "f16", hyper["lr"], hyper["beta1"], hyper["beta2"], hyper["eps"],
                          hyper["weight_decay"], 4096.0, 2.0, 0.5, 3, fp8_shapes=fp8_shapes,
                          fp8_scaling=mode, hist_len=2, fp8_format=fmt, sr_seed=seed)
    for k in range(5):
        gh = [(rng.standard_normal(n) * 1e-3 * orc.scale).astype(np.float16).view(np.uint16)
              for n in sizes]
        if k == 2:
            gh[3][17] = 0x7C00
        for t, h in zip(st.grads, gh):
            t.copy_(to_device(h, "f16", dev))
        st.step()
        orc.run(gh)
        s = st.state()
        assert (s["scale"], s["growth_tracker"], s["step"]) == (orc.scale, orc.tracker, orc.step)
        for i, sh in enumerate(fp8_shapes):
            assert np.array_equal(to_host_bits(st.bf16[i]), orc.bf16[i]), (k, i)
            if sh is None:
                continue
            j = orc.slots[i]
            assert np.array_equal(to_host_bits(st.fp8[j].view(torch.uint8)).ravel(), orc.fp8[i]), (k, i)
            assert np.array_equal(to_host_bits(st.fp8_t[j].view(torch.uint8)).ravel(),
                                  orc.fp8_t[i]), (k, i)
            assert to_host_bits(st.inv_scale)[j] == orc.inv_scale[j], (k, i)
    for i in range(len(shapes)):
        assert np.array_equal(to_host_bits(st.master[i]).view(np.uint32), orc.master[i].view(np.uint32))
        assert np.array_equal(to_host_bits(st.exp_avg_sq[i]).view(np.uint32),
                              orc.exp_avg_sq[i].view(np.uint32))
    st.close()


def test_stochastic_step_with_clipping(A, dev, monkeypatch):
    """AmpOptimizerStep(sr_seed, max_norm) with FP8 weights: the master state
    within the clipped step's tolerance, the bf16 copy within 1 ulp of the
    oracle's (its clip factor comes from a tolerance-checked sum of squares),
    and on every step that is not skipped the FP8 bytes equal the oracle's
    stochastic quantizer run on the GPU's own bf16 copy with the GPU's amax."""
    from loss_scaling_master_gb300 import AmpOptimizerStep
    from loss_scaling_master_gb300 import step as step_mod
    snap = {}
    real_update = step_mod.A.amp_update_scale

    def spy_update(*args, amax=None, **kw):
        if amax is not None:
            snap["amax"] = amax.clone()
        return real_update(*args, amax=amax, **kw)

    monkeypatch.setattr(step_mod.A, "amp_update_scale", spy_update)
    rng = np.random.default_rng(162)
    sizes = [1000, 4096, 257, 40000]
    fp8_shapes = [None, (64, 64), None, (200, 200)]
    master = [(rng.standard_normal(n) * 0.02).astype(np.float32) for n in sizes]
    hyper = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    seed = 77
    st = AmpOptimizerStep([torch.from_numpy(m.copy()).to(dev) for m in master],
                          [torch.empty(n, dtype=torch.float16, device=dev) for n in sizes],
                          init_scale=65536.0, growth_interval=3, max_norm=0.5,
                          fp8_shapes=fp8_shapes, sr_seed=seed, **hyper)
    orc = O.AmpStepOracle(master, "f16", hyper["lr"], hyper["beta1"], hyper["beta2"], hyper["eps"],
                          hyper["weight_decay"], 65536.0, 2.0, 0.5, 3, max_norm=0.5,
                          fp8_shapes=fp8_shapes, sr_seed=seed)
    for k in range(5):
        sigma = (1e-2 if k % 2 == 0 else 1e-5) * orc.scale
        gh = [(rng.standard_normal(n) * sigma).astype(np.float16).view(np.uint16) for n in sizes]
        if k == 3:
            gh[2][100] = 0x7C00
        for t, h in zip(st.grads, gh):
            t.copy_(to_device(h, "f16", dev))
        st.step()
        orc.run(gh)
        s = st.state()
        assert (s["scale"], s["growth_tracker"], s["step"]) == (orc.scale, orc.tracker, orc.step)
        if k == 3:
            continue
        gpu_amax = to_host_bits(snap["amax"])
        for i, sh in enumerate(fp8_shapes):
            gb = to_host_bits(st.bf16[i])
            assert_bf16_close(gb, orc.bf16[i], f"bf16[{i}] step {k}")
            if sh is None:
                continue
            j = orc.slots[i]
            q, qt, inv, _ = O.fp8_quant_tensorwise_sr(gb, "bf16", sh[0], sh[1], "e4m3fn", seed,
                                                      s["step"], j, amax=float(gpu_amax[j]))
            assert np.array_equal(to_host_bits(st.fp8[j].view(torch.uint8)).ravel(), q), (k, i)
            assert np.array_equal(to_host_bits(st.fp8_t[j].view(torch.uint8)).ravel(), qt), (k, i)
    for i in range(len(sizes)):
        assert_state_close(to_host_bits(st.master[i]), orc.master[i], f"master[{i}]")
    st.close()


@pytest.mark.parametrize("fmt,tdt", [("e4m3fn", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_fp8_stochastic_unbiased_on_gpu(A, dev, fmt, tdt):
    """E[fp8_sr(y)] = y: a constant [2048, 2048] bf16 matrix whose scaled value
    falls between two FP8 neighbours; the mean of the dequantized bytes over
    its 4M elements sits within 5 sigma of the scaled value."""
    n = 2048
    xval = 0.3                                         # bf16 0.30078125; amax given as 1.0
    x = torch.full((n, n), xval, dtype=torch.bfloat16, device=dev)
    q = torch.empty((n, n), dtype=tdt, device=dev)
    LX, LQ = A.amp_tensor_list_create([x], True), A.amp_tensor_list_create([q], True)
    amax = torch.ones(1, device=dev)
    inv = torch.zeros(1, device=dev)
    step = torch.tensor([5], dtype=torch.int32, device=dev)
    A.fp8_quant_tensorwise_list_sr(LX, LQ, None, fmt, amax, inv, 4242, step)
    fmax = O.fmt_max(fmt)
    y = float(np.float32(np.float32(x[0, 0].item()) * np.float32(fmax)))
    d = q.float().double()
    grid = torch.arange(128, dtype=torch.uint8).view(tdt).float().double().cpu().numpy()
    grid = np.unique(grid[np.isfinite(grid)])
    j = np.searchsorted(grid, y, side="right") - 1
    lo, hi = grid[j], grid[j + 1]
    assert set(torch.unique(d).tolist()) <= {lo, hi}
    p = (y - lo) / (hi - lo)
    sigma = (hi - lo) * np.sqrt(p * (1 - p) / d.numel())
    assert 0.05 < p < 0.95
    assert abs(d.mean().item() - y) < 5 * sigma
    LX.close()
    LQ.close()


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
def test_fp8_stochastic_rule_dense_over_fp32_patterns(A, dev, fmt):
    """The stochastic FP8 rule on 4M fp32 bit patterns spread (odd stride, so
    the low fraction bits vary) over every magnitude where the rounding has a
    non-zero chance of going up: the FP8 subnormal range, the normal binades,
    the clamp above fp8_max; every other pattern negative, and NaN and
    infinities planted.  f32 input with amax = fp8_max gives a cast scale of
    exactly 1, so the cast rounds these patterns themselves; every byte of
    both layouts equals the oracle's."""
    rows, cols = 2048, 2048
    n = rows * cols
    lo, hi = 0x2F000000, 0x47800000          # 2^-33 .. 2^16: past both formats' ranges
    k = np.arange(n, dtype=np.uint64)
    bits = (lo + (k * 97) % (hi - lo)).astype(np.uint32)
    bits[1::2] |= np.uint32(0x80000000)
    bits[[10, 11, 12]] = np.array([0x7F800000, 0xFF800000, 0x7FC00001], np.uint32)
    x = bits.view(np.float32)
    fmax = O.fmt_max(fmt)
    tdt = torch.float8_e4m3fn if fmt == "e4m3fn" else torch.float8_e5m2
    xd = torch.from_numpy(x.copy()).to(dev).view(rows, cols)
    q = torch.empty((rows, cols), dtype=tdt, device=dev)
    qt = torch.empty((cols, rows), dtype=tdt, device=dev)
    LX, LQ, LQT = (A.amp_tensor_list_create([t], True) for t in (xd, q, qt))
    amax = torch.tensor([fmax], dtype=torch.float32, device=dev)
    inv = torch.zeros(1, device=dev)
    seed, step = 0x0123456789ABCDEF, 77
    A.fp8_quant_tensorwise_list_sr(LX, LQ, LQT, fmt, amax, inv, seed,
                                   torch.tensor([step], dtype=torch.int32, device=dev))
    rq, rqt, rinv, _ = O.fp8_quant_tensorwise_sr(x, "f32", rows, cols, fmt, seed, step, 0,
                                                 amax=fmax)
    assert rinv == 1.0 and to_host_bits(inv)[0] == 1.0
    assert np.array_equal(to_host_bits(q.view(torch.uint8)).ravel(), rq)
    assert np.array_equal(to_host_bits(qt.view(torch.uint8)).ravel(), rqt)
    for L in (LX, LQ, LQT):
        L.close()


# --------------------------------------------------------- checkpoint / resume
def test_delayed_scaling_without_fp8_weights_is_the_plain_step(A, dev):
    """A set given fp8_shapes with no FP8 weight in it (a data-parallel shard
    can own none) and delayed scaling steps exactly as the plain dynamic step:
    nothing to cast, no history; master, m, v, bf16 and the scaler state equal
    the plain step's bit for bit through a skipped step."""
    from loss_scaling_master_gb300 import AmpOptimizerStep
    rng = np.random.default_rng(111)
    sizes = [1000, 4097, 300]
    master = [(rng.standard_normal(n) * 0.02).astype(np.float32) for n in sizes]
    grads = []
    for k in range(3):
        g = [(rng.standard_normal(n) * 1e-5 * 1024).astype(np.float16).view(np.uint16)
             for n in sizes]
        if k == 1:
            g[2][7] = 0x7C00
        grads.append(g)
    runs = []
    for kw in (dict(fp8_shapes=[None, None, None], fp8_scaling="delayed"), dict()):
        P = [to_device(m, "f32", dev) for m in master]
        G = [torch.empty(n, dtype=torch.float16, device=dev) for n in sizes]
        st = AmpOptimizerStep(P, G, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                              weight_decay=0.01, init_scale=1024.0, growth_interval=2, **kw)
        assert st.fp8_scaling == "dynamic" and st.n_fp8 == 0
        trace = []
        for g in grads:
            for t, h in zip(G, g):
                t.copy_(to_device(h, "f16", dev))
            st.step()
            s = st.state()
            trace.append((s["scale"], s["growth_tracker"], s["step"]))
        runs.append((trace, [to_host_bits(x) for x in st.master + st.exp_avg + st.exp_avg_sq],
                     [to_host_bits(x) for x in st.bf16]))
        st.check()
        st.close()
    assert runs[0][0] == runs[1][0] and runs[0][0][1][2] == runs[0][0][0][2]
    for a, b in zip(runs[0][1] + runs[0][2], runs[1][1] + runs[1][2]):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


@pytest.mark.parametrize("fp8_scaling", ["dynamic", "delayed"])
def test_checkpoint_resume_is_bit_identical(A, dev, fp8_scaling):
    """Save the state after 3 steps, restore it into a fresh step object and
    continue: the resumed run equals the uninterrupted one bit for bit."""
    from loss_scaling_master_gb300 import AmpOptimizerStep
    rng = np.random.default_rng(101)
    shapes = [(128, 256), (300,), (256, 384)]
    fp8_shapes = [s if len(s) == 2 else None for s in shapes]
    sizes = [int(np.prod(s)) for s in shapes]
    master = [(rng.standard_normal(n) * 0.02).astype(np.float32) for n in sizes]
    grads = [[(rng.standard_normal(n) * 1e-3 * 1024).astype(np.float16).view(np.uint16) for n in sizes]
             for _ in range(6)]
    grads[4][1][7] = 0x7C00                                        # a skipped step after resume
    hyper = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)

    def make():
        return AmpOptimizerStep([torch.from_numpy(m.copy()).to(dev) for m in master],
                                [torch.empty(n, dtype=torch.float16, device=dev) for n in sizes],
                                init_scale=1024.0, growth_interval=2, fp8_shapes=fp8_shapes,
                                fp8_scaling=fp8_scaling, amax_history_len=2, **hyper)

    def run(st, gs):
        for g in gs:
            for t, h in zip(st.grads, g):
                t.copy_(to_device(h, "f16", dev))
            st.step()

    whole = make()
    run(whole, grads)
    first = make()
    run(first, grads[:3])
    ckpt = first.state_dict()
    first.close()
    resumed = make()
    resumed.load_state_dict(ckpt)
    run(resumed, grads[3:])
    a, b = whole.state_dict(), resumed.state_dict()
    for k in a:
        if a[k] is None:
            continue
        xs, ys = (a[k], b[k]) if isinstance(a[k], list) else ([a[k]], [b[k]])
        for x, y in zip(xs, ys):
            assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), k
    whole.close()
    resumed.close()


# ------------------------------------------------------ bounded waits
def test_bounded_wait_gives_up_and_context_survives(A, dev):
    """A wait on a barrier that nothing completes ends after its time limit
    with an error status instead of hanging; the GPU keeps working."""
    import time
    err = torch.full((1,), -1, dtype=torch.int32, device=dev)
    t0 = time.perf_counter()
    A.amp_selftest_bounded_wait(err, 0.05)
    torch.cuda.synchronize()
    assert int(err.item()) == 1
    assert time.perf_counter() - t0 < 5.0
    x = torch.arange(1000, device=dev, dtype=torch.float32)
    assert float(x.sum().item()) == 499500.0               # the context is fine


def test_list_check_ok_after_steps(A, dev):
    from loss_scaling_master_gb300 import AmpOptimizerStep
    st = AmpOptimizerStep([torch.zeros(5000, device=dev)], [torch.zeros(5000, dtype=torch.float16, device=dev)],
                          lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
    for _ in range(3):
        st.step()
    A.amp_tensor_list_check(st.L_master)
    st.check()
    st.close()


# ------------------------------------------------------ empty tensors and lists
@pytest.mark.parametrize("fp8_scaling", ["dynamic", "delayed"])
def test_empty_tensors_in_the_step(A, dev, fp8_scaling):
    """Tensors with no elements among the parameters, including empty FP8
    weights of shape [0, 128] and [128, 0]: the step runs, every non-empty
    tensor matches the oracle bit for bit, and the empty FP8 weights get the
    inv_scale of amax 0 (the EPS floor of [FP8] §2)."""
    from loss_scaling_master_gb300 import AmpOptimizerStep
    rng = np.random.default_rng(41)
    shapes = [(0,), (96, 256), (0, 128), (300,), (128, 0), (0,), (128, 136)]
    fp8_shapes = [s if len(s) == 2 else None for s in shapes]
    sizes = [int(np.prod(s)) for s in shapes]
    master = [(rng.standard_normal(n) * 0.02).astype(np.float32) for n in sizes]
    G = [torch.empty(n, dtype=torch.float16, device=dev) for n in sizes]
    hyper = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    st = AmpOptimizerStep([torch.from_numpy(m.copy()).to(dev) for m in master], G,
                          init_scale=65536.0, growth_interval=2, fp8_shapes=fp8_shapes,
                          fp8_scaling=fp8_scaling, **hyper)
    orc = O.AmpStepOracle(master, "f16", hyper["lr"], hyper["beta1"], hyper["beta2"],
                          hyper["eps"], hyper["weight_decay"], 65536.0, 2.0, 0.5, 2,
                          fp8_shapes=fp8_shapes, fp8_scaling=fp8_scaling)
    for k in range(1, 6):
        gh = [(rng.standard_normal(n) * 1e-4 * orc.scale).astype(np.float16).view(np.uint16)
              for n in sizes]
        if k == 3:
            gh[3][299] = 0x7C00
        for t, h in zip(G, gh):
            t.copy_(to_device(h, "f16", dev))
        st.step()
        orc.run(gh)
        s = st.state()
        assert (s["scale"], s["growth_tracker"], s["step"], s["found_inf"]) == \
            (orc.scale, orc.tracker, orc.step, 0), k
    st.check()
    for i, n in enumerate(sizes):
        assert np.array_equal(to_host_bits(st.master[i]).view(np.uint32),
                              orc.master[i].view(np.uint32)), i
        assert np.array_equal(to_host_bits(st.bf16[i]), orc.bf16[i]), i
    inv = to_host_bits(st.inv_scale)
    j = 0
    for i, sh in enumerate(fp8_shapes):
        if sh is None:
            continue
        assert np.array_equal(to_host_bits(st.fp8[j].view(torch.uint8)).ravel(), orc.fp8[i])
        assert np.array_equal(to_host_bits(st.fp8_t[j].view(torch.uint8)).ravel(), orc.fp8_t[i])
        assert inv[j].view(np.uint32) == np.float32(orc.inv_scale[orc.slots[i]]).view(np.uint32), (i, inv[j])
        if sizes[i] == 0:
            assert inv[j] == np.float32(1e-12 / 448.0)
        j += 1
    st.close()


def test_lists_with_no_tensors(A, dev):
    """Every list entry point accepts a list of no tensors: the check leaves
    found_inf alone, the norm is 0, and the AdamW step (nothing to update)
    still advances the step counter unless skipped, as the oracle does."""
    E = [A.amp_tensor_list_create([], dtype=d) for d in ("f32", "f32", "f32", "f16", "bf16")]
    X8 = A.amp_tensor_list_create([], two_d=True, dtype="bf16")
    Q8 = A.amp_tensor_list_create([], two_d=True, dtype="e4m3fn")
    QT = A.amp_tensor_list_create([], two_d=True, dtype="e4m3fn")
    scale = torch.tensor([1024.0], device=dev)
    fi = torch.zeros(1, dtype=torch.int32, device=dev)
    step = torch.zeros(1, dtype=torch.int32, device=dev)
    sumsq = torch.full((1,), -1.0, dtype=torch.float64, device=dev)
    A.amp_unscale_check(E[3], scale, fi)
    A.amp_unscale_check_norm(E[3], scale, fi, sumsq)
    A.amp_adamw_master_step(*E, scale, fi, step, 1e-3, 0.9, 0.999, 1e-8, 0.01)
    fi.fill_(1)
    A.amp_adamw_master_step(*E, scale, fi, step, 1e-3, 0.9, 0.999, 1e-8, 0.01)
    amax = torch.zeros(1, device=dev)
    inv = torch.zeros(1, device=dev)
    A.fp8_quant_tensorwise_list(X8, Q8, QT, "e4m3fn", amax, inv)
    torch.cuda.synchronize()
    rstep = O.adamw_master_step([], [], [], [], "f16", None, 1024.0, 0, 0, 1e-3, 0.9, 0.999, 1e-8, 0.01)
    rstep = O.adamw_master_step([], [], [], [], "f16", None, 1024.0, 1, rstep, 1e-3, 0.9, 0.999, 1e-8, 0.01)
    assert int(step.item()) == rstep == 1
    assert float(sumsq.item()) == 0.0
    A.amp_tensor_list_check(E[0])
    for L in E + [X8, Q8, QT]:
        L.close()


def test_list_host_copies_round_trip(A, dev):
    """amp_tensor_list_copy_from_host / _to_host move every tensor of a list
    (empty ones included) byte for byte, from pageable and page-locked memory."""
    rng = np.random.default_rng(42)
    sizes = [0, 1, 7, 16385, 0, 100003]
    for pinned in (False, True):
        D = [torch.empty(n, dtype=torch.float16, device=dev) for n in sizes]
        L = A.amp_tensor_list_create(D)
        src = [torch.from_numpy(rng.integers(0, 1 << 16, n, dtype=np.uint16).view(np.int16).copy())
               for n in sizes]
        dst = [torch.full((n,), -1, dtype=torch.int16) for n in sizes]
        if pinned:
            src = [t.pin_memory() for t in src]
            dst = [t.pin_memory() for t in dst]
        A.amp_tensor_list_copy_from_host(L, [t if t.numel() else None for t in src])
        torch.cuda.synchronize()
        for d, s in zip(D, src):
            assert torch.equal(d.cpu().view(torch.int16), s)
        A.amp_tensor_list_copy_to_host(L, dst)
        torch.cuda.synchronize()
        for d, s in zip(dst, src):
            assert torch.equal(d, s)
        L.close()


def test_huge_page_host_buffer_feeds_a_list(A, dev):
    """pinned_empty (huge-page mapping registered with CUDA) as the host side of
    amp_tensor_list_copy_from_host: one buffer viewed per tensor, as the e2e
    feed uses it; every byte arrives, and the buffer closes cleanly."""
    from loss_scaling_master_gb300.hostmem import pinned_empty
    rng = np.random.default_rng(43)
    sizes = [1, 1000, 0, (1 << 21) + 5, 8]
    buf = pinned_empty(sum(sizes), torch.float16)
    host = buf.tensor
    assert host.numel() == sum(sizes) and host.dtype == torch.float16
    host.view(torch.int16).copy_(torch.from_numpy(
        rng.integers(0, 1 << 16, sum(sizes), dtype=np.uint16).view(np.int16)))
    D = [torch.empty(n, dtype=torch.float16, device=dev) for n in sizes]
    L = A.amp_tensor_list_create(D)
    ptrs, off = [], 0
    for n in sizes:
        ptrs.append(host.data_ptr() + 2 * off if n else None)
        off += n
    A.amp_tensor_list_copy_from_host(L, ptrs)
    torch.cuda.synchronize()
    off = 0
    for d, n in zip(D, sizes):
        assert torch.equal(d.cpu().view(torch.int16), host[off:off + n].view(torch.int16))
        off += n
    L.close()
    del host
    buf.close()
    assert buf.tensor is None


# ------------------------------------------------------ monitoring
def test_read_state_and_scale_health(A, dev):
    """amp_read_state copies the scaler state to host memory; amp_scale_health
    sets bit 2 once the scale has halved below min_scale and bit 1 for a
    non-finite scale, into page-locked host memory the host polls."""
    from loss_scaling_master_gb300 import AmpOptimizerStep
    n = 3000
    G = [torch.zeros(n, dtype=torch.float16, device=dev)]
    st = AmpOptimizerStep([torch.zeros(n, device=dev)], G, lr=1e-3, beta1=0.9, beta2=0.999,
                          eps=1e-8, weight_decay=0.0, init_scale=8.0, growth_interval=1000,
                          min_scale=1.0)
    G[0][17] = float("inf")                       # every step overflows: S halves each time
    seen = []
    for k in range(5):
        st.step()
        torch.cuda.synchronize()
        seen.append(st.health())
    assert seen == [0, 0, 0, 2, 2]                # 4, 2, 1, 0.5, 0.25
    s = st.state()
    assert s == {"scale": 0.25, "growth_tracker": 0, "step": 0, "found_inf": 0}
    out = A.ScalerState()
    bad = torch.tensor([float("nan")], device=dev)
    A.amp_read_state(bad, st.growth_tracker, None, None, out)
    health = torch.zeros(1, dtype=torch.int32).pin_memory()
    A.amp_scale_health(bad, 1.0, health)
    torch.cuda.synchronize()
    assert np.isnan(out.scale) and out.growth_tracker == 0 and int(health[0]) == 1
    st.close()


# ------------------------------------------------------ every AdamW instantiation
@pytest.mark.parametrize("gdt", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("emit", ["none", "rne", "sr"])
def test_adamw_every_grad_dtype_and_copy_mode(A, dev, gdt, emit):
    """Each (grad dtype) x (no copy, RNE bf16 copy, stochastic bf16 copy) form
    of the update, aligned and misaligned, over chunk-spanning ragged sizes
    with a skipped step: master, m, v and the copy bit-identical to the oracle."""
    rng = np.random.default_rng(100 + len(gdt) + len(emit))
    sizes = [1, 9, 2047, 2049, 16383, 16385, 3 * 16384 + 5]
    seed = 0xC0FFEE
    for misalign in (False, True):
        master_h = [(rng.standard_normal(k) * 0.02).astype(np.float32) for k in sizes]
        P = _device_views(master_h, "f32", dev, misalign)
        M = _device_views([np.zeros(k, np.float32) for k in sizes], "f32", dev, misalign)
        V = _device_views([np.zeros(k, np.float32) for k in sizes], "f32", dev, misalign)
        G = _device_views(_grads_host(rng, sizes, gdt), gdt, dev, misalign)
        B = _device_views([np.zeros(k, np.uint16) for k in sizes], "bf16", dev, misalign) \
            if emit != "none" else None
        LP, LM, LV, LG = (A.amp_tensor_list_create(x) for x in (P, M, V, G))
        LB = A.amp_tensor_list_create(B) if B is not None else None
        step = torch.zeros(1, dtype=torch.int32, device=dev)
        fi = torch.zeros(1, dtype=torch.int32, device=dev)
        rp, rm, rv = [x.copy() for x in master_h], [np.zeros(k, np.float32) for k in sizes], \
            [np.zeros(k, np.float32) for k in sizes]
        rb = [np.zeros(k, np.uint16) for k in sizes] if B is not None else None
        rstep = 0
        S = 512.0
        for k in range(3):
            gh = _grads_host(rng, sizes, gdt, sigma=1e-3 * S)
            for t, h in zip(G, gh):
                t.copy_(to_device(h, gdt, dev))
            skip = int(k == 1)
            fi.fill_(skip)
            sd = torch.tensor([S], device=dev)
            hyper = (1e-3, 0.9, 0.999, 1e-8, 0.01)
            if emit == "sr":
                A.amp_adamw_master_step_sr(LP, LM, LV, LG, LB, sd, fi, step, *hyper, seed)
            else:
                A.amp_adamw_master_step(LP, LM, LV, LG, LB, sd, fi, step, *hyper)
            rstep = O.adamw_master_step(rp, rm, rv, gh, gdt, rb, S, skip, rstep, *hyper,
                                        sr_seed=seed if emit == "sr" else None)
            assert int(step.item()) == rstep
        for i in range(len(sizes)):
            key = (gdt, emit, misalign, sizes[i])
            assert np.array_equal(to_host_bits(P[i]).view(np.uint32), rp[i].view(np.uint32)), key
            assert np.array_equal(to_host_bits(M[i]).view(np.uint32), rm[i].view(np.uint32)), key
            assert np.array_equal(to_host_bits(V[i]).view(np.uint32), rv[i].view(np.uint32)), key
            if B is not None:
                assert np.array_equal(to_host_bits(B[i]), rb[i]), key
        for L in (LP, LM, LV, LG, LB):
            if L is not None:
                L.close()


def test_two_steps_on_two_streams_concurrently(A, dev):
    """Two independent optimizer steps (own lists, own scaler state), each on
    its own stream, enqueued alternately with no host sync in between: both
    end bit-identical to the oracle (per-list scratch, stream-ordered launches)."""
    from loss_scaling_master_gb300 import AmpOptimizerStep
    rng = np.random.default_rng(110)
    streams = [torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)]
    cases = []
    for c in range(2):
        shapes = [(96, 256), (3000,), (200, 136)] if c == 0 else [(50000,), (128, 128)]
        fp8_shapes = [s if len(s) == 2 else None for s in shapes]
        sizes = [int(np.prod(s)) for s in shapes]
        master = [(rng.standard_normal(n) * 0.02).astype(np.float32) for n in sizes]
        hyper = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
        with torch.cuda.stream(streams[c]):
            st = AmpOptimizerStep([torch.from_numpy(m.copy()).to(dev) for m in master],
                                  [torch.zeros(n, dtype=torch.float16, device=dev) for n in sizes],
                                  init_scale=1024.0, growth_interval=2, fp8_shapes=fp8_shapes,
                                  fp8_scaling="delayed" if c == 1 else "dynamic",
                                  stream=streams[c], **hyper)
        orc = O.AmpStepOracle(master, "f16", hyper["lr"], hyper["beta1"], hyper["beta2"],
                              hyper["eps"], hyper["weight_decay"], 1024.0, 2.0, 0.5, 2,
                              fp8_shapes=fp8_shapes,
                              fp8_scaling="delayed" if c == 1 else "dynamic")
        cases.append((st, orc, sizes, fp8_shapes))
    torch.cuda.synchronize()
    grads = [[[(rng.standard_normal(n) * 1e-3 * 1024).astype(np.float16).view(np.uint16)
               for n in sizes] for _ in range(4)] for (_, _, sizes, _) in cases]
    dev_grads = [[[to_device(h, "f16", dev) for h in g] for g in per] for per in grads]
    torch.cuda.synchronize()
    for k in range(4):
        for c, (st, orc, sizes, _) in enumerate(cases):
            with torch.cuda.stream(streams[c]):
                for t, h in zip(st.grads, dev_grads[c][k]):
                    t.copy_(h)
            st.step(stream=streams[c])
    torch.cuda.synchronize()
    for c, (st, orc, sizes, fp8_shapes) in enumerate(cases):
        for k in range(4):
            orc.run(grads[c][k])
        s = st.state()
        assert (s["scale"], s["growth_tracker"], s["step"]) == (orc.scale, orc.tracker, orc.step)
        for i in range(len(sizes)):
            assert np.array_equal(to_host_bits(st.master[i]).view(np.uint32),
                                  orc.master[i].view(np.uint32)), (c, i)
            assert np.array_equal(to_host_bits(st.bf16[i]), orc.bf16[i]), (c, i)
        j = 0
        for i, sh in enumerate(fp8_shapes):
            if sh is None:
                continue
            assert np.array_equal(to_host_bits(st.fp8[j].view(torch.uint8)).ravel(), orc.fp8[i])
            assert np.array_equal(to_host_bits(st.fp8_t[j].view(torch.uint8)).ravel(), orc.fp8_t[i])
            j += 1
        st.close()


# ----------------------------------------------------------- group-wise FP8
def _run_groupwise(A, dev, xh, xdt, rows, cols, fmt, group, with_t, skip=None, misalign=False):
    x = _device_views([xh], xdt, dev, misalign)[0].view(rows, cols)
    ngc, ngr = -(-cols // group), -(-rows // group)
    o = {"q": torch.full((rows * cols,), 0xA5, dtype=torch.uint8, device=dev)}
    o.update({k: torch.full((rows * ngc,), -1.0, device=dev) for k in ("amax_rg", "scale_rg", "inv_rg")})
    if with_t:
        o["q_t"] = torch.full((rows * cols,), 0x5A, dtype=torch.uint8, device=dev)
        o.update({k: torch.full((cols * ngr,), -1.0, device=dev) for k in ("amax_cg", "scale_cg", "inv_cg")})
    sk = None if skip is None else torch.tensor([skip], dtype=torch.int32, device=dev)
    A.fp8_quant_groupwise(x, fmt, group, o["q"], o.get("q_t"), o["amax_rg"], o["scale_rg"],
                          o["inv_rg"], o.get("amax_cg"), o.get("scale_cg"), o.get("inv_cg"),
                          skip_if=sk)
    return {k: to_host_bits(v) for k, v in o.items()}


def _assert_same(got, ref, key):
    """Bytes bit for bit; fp32 bit for bit except NaN, whose payload IEEE 754
    leaves open for arithmetic results, so NaNs are compared by position."""
    for k in ref:
        if ref[k].dtype == np.float32:
            g, r = got[k].view(np.float32), ref[k]
            nan = np.isnan(r)
            assert np.array_equal(np.isnan(g), nan), (k, key)
            assert np.array_equal(g[~nan].view(np.uint32), r[~nan].view(np.uint32)), (k, key)
        else:
            assert np.array_equal(got[k], ref[k]), (k, key)


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
@pytest.mark.parametrize("xdt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("group", [32, 64, 128])
def test_fp8_groupwise_parity(A, dev, fmt, xdt, group):
    rng = np.random.default_rng(120 + group)
    for rows, cols in FP8_SHAPES:
        xh = _x_host(rng, rows, cols, xdt)
        if rows > 3:                       # a zero row: its groups clamp to EPS
            xh.reshape(rows, cols)[2] = 0
        for with_t in (True, False):
            for misalign in ((False, True) if rows * cols > 8 else (False,)):
                got = _run_groupwise(A, dev, xh, xdt, rows, cols, fmt, group, with_t,
                                     misalign=misalign)
                ref = O.fp8_quant_groupwise(xh, xdt, rows, cols, fmt, group, transposed=with_t)
                _assert_same(got, ref, (rows, cols, with_t, misalign))


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
@pytest.mark.parametrize("xdt,group", [("bf16", 128), ("f16", 64)])
def test_fp8_groupwise_many_tiles_per_cta(A, dev, fmt, xdt, group):
    """More tiles than one wave of CTAs, full tiles and ragged edge tiles
    mixed, twice in a row on one matrix."""
    rng = np.random.default_rng(150)
    rows, cols = 4096 + 80, 2048 + 8               # 33 x 17 tiles, a ragged row and column
    xh = _x_host(rng, rows, cols, xdt)
    ref = O.fp8_quant_groupwise(xh, xdt, rows, cols, fmt, group, transposed=True)
    for _ in range(2):
        got = _run_groupwise(A, dev, xh, xdt, rows, cols, fmt, group, True)
        _assert_same(got, ref, (rows, cols))


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
def test_fp8_groupwise_scale_over_many_amax_values(A, dev, fmt):
    """The kernel forms group scales with fp32 divisions (equal to the fp64
    recipe rounded to fp32, see its header); check that against the oracle's
    fp64 formula for 2^16 group maxima spread over every fp32 exponent,
    subnormals, values around EPS, zero, inf and NaN: each row group of a
    [2^16, 128] fp32 matrix holds one such value, all else zero."""
    rng = np.random.default_rng(130)
    n = 1 << 16
    bits = rng.integers(0, 0x7F800000, n, dtype=np.uint32)
    bits[:64] = [0, 1, 0x00400000, 0x007FFFFF, 0x00800000, 0x7F7FFFFF, 0x7F800000, 0x7FC00000] * 8
    eps = 1e-12
    near = np.float32(eps).view(np.uint32)
    bits[64:96] = near + np.arange(-16, 16, dtype=np.int64).astype(np.uint32)
    vals = bits.view(np.float32)
    x = np.zeros((n, 128), np.float32)
    x[np.arange(n), rng.integers(0, 128, n)] = vals * np.where(rng.random(n) < 0.5, -1, 1).astype(np.float32)
    xh = x.ravel()
    got = _run_groupwise(A, dev, xh, "f32", n, 128, fmt, 128, True)
    ref = O.fp8_quant_groupwise(xh, "f32", n, 128, fmt, 128, eps=eps)
    _assert_same(got, ref, "amax sweep")


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
def test_scale_formula_dense_where_it_is_tightest(A, dev, fmt):
    """The kernels form scale = fp8_max / amax and inv_scale = amax / fp8_max
    with IEEE fp32 divisions in place of the fp64 recipe rounded to fp32; the
    argument for equality is tightest where amax / fp8_max is exact, i.e. where
    amax's significand is a multiple of 7 (fp8_max = 7 * 2^k).  Every fp32
    significand m with m % 7 in {0, 1, 2, 5, 6} (the multiples and their two
    neighbours on each side) at the smallest normal exponent, at 2^-20, 2^0,
    2^20 and 2^127, and every subnormal pattern with that residue (where the
    EPS floor decides), as single-element rows of the per-row quantizer: amax,
    scale, inv_scale and the byte equal the oracle's fp64 formula."""
    m = np.arange(1 << 23, 1 << 24, dtype=np.uint32)
    m = m[np.isin(m % 7, [0, 1, 2, 5, 6])] - np.uint32(1 << 23)
    sub = np.arange(1, 1 << 23, dtype=np.uint32)
    sub = sub[np.isin(sub % 7, [0, 1, 2, 5, 6])]
    for e in (-126, -20, 0, 20, 127, None):
        bits = sub if e is None else (np.uint32(e + 127) << np.uint32(23)) | m
        x = bits.view(np.float32)
        rows = x.size
        got = _run_rowwise(A, dev, x, "f32", rows, 1, fmt, False)
        ref = O.fp8_quant_rowwise(x, "f32", rows, 1, fmt, transposed=False)
        _assert_same(got, ref, ("dense scale", e))


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
@pytest.mark.parametrize("xdt", ["bf16", "f16"])
@pytest.mark.parametrize("group", [32, 64, 128])
def test_fp8_groupwise_nonfinite_16bit(A, dev, fmt, xdt, group):
    """16-bit x with NaNs of both signs and several payloads, +-inf,
    subnormals and -0 planted in some full tiles, the others left finite:
    group maxima (NaN above inf), the NaN / zero scales they give, and the NaN
    bytes (canonical) in both layouts."""
    rng = np.random.default_rng(140 + group)
    rows, cols = 384, 512
    xh = _x_host(rng, rows, cols, xdt).reshape(rows, cols).copy()
    if xdt == "bf16":
        specials = [0x7FC0, 0xFFC0, 0x7F81, 0xFFFF, 0x7F80, 0xFF80, 0x0001, 0x807F, 0x8000]
    else:
        specials = [0x7E00, 0xFE00, 0x7C01, 0xFFFF, 0x7C00, 0xFC00, 0x0001, 0x83FF, 0x8000]
    # tiles (0, 0), (1, 2) and (2, 3) get specials; tile (1, 1) holds only
    # subnormals and -0; the rest stays finite
    for (tr, tc) in ((0, 0), (1, 2), (2, 3)):
        for v in specials:
            i, j = rng.integers(0, 128, 2)
            xh[128 * tr + i, 128 * tc + j] = v
    xh[128:256, 128:256] = np.where(rng.random((128, 128)) < 0.5, specials[6], specials[7])
    xh[130, 130] = specials[8]
    xh = xh.ravel()
    for with_t in (True, False):
        got = _run_groupwise(A, dev, xh, xdt, rows, cols, fmt, group, with_t)
        ref = O.fp8_quant_groupwise(xh, xdt, rows, cols, fmt, group, transposed=with_t)
        _assert_same(got, ref, ("nonfinite", with_t))


def test_binding_rejects_short_or_mistyped_buffers(A, dev):
    """Undersized outputs and wrongly typed scalars raise in the binding, before
    a launch could write past them."""
    x = torch.zeros(256, 256, dtype=torch.bfloat16, device=dev)
    q = torch.empty(256 * 256, dtype=torch.uint8, device=dev)
    short = torch.empty(256 * 256 - 1, dtype=torch.uint8, device=dev)
    f = torch.empty(1, device=dev)
    with pytest.raises(ValueError, match="out_t"):
        A.fp8_quant_tensorwise(x, "e4m3fn", q, short, f, f)
    with pytest.raises(ValueError, match="amax"):
        A.fp8_quant_tensorwise(x, "e4m3fn", q, None, f, torch.empty(1, dtype=torch.float64,
                                                                     device=dev))
    r = torch.empty(256, device=dev)
    with pytest.raises(ValueError, match="scale_col"):
        A.fp8_quant_rowwise(x, "e4m3fn", q, q, r, r, r, r, r[:255], r)
    g = torch.empty(256 * 2, device=dev)
    with pytest.raises(ValueError, match="inv_rg"):
        A.fp8_quant_groupwise(x, "e4m3fn", 128, q, None, g, g, g[:511])
    with pytest.raises(ValueError, match="found_inf"):
        A.amp_update_scale(f, torch.zeros(1, dtype=torch.int32, device=dev),
                           torch.zeros(1, dtype=torch.int64, device=dev), 2.0, 0.5, 10)
    torch.cuda.synchronize()


def test_fp8_groupwise_skip_writes_nothing(A, dev):
    rng = np.random.default_rng(131)
    xh = _x_host(rng, 256, 384, "bf16")
    got = _run_groupwise(A, dev, xh, "bf16", 256, 384, "e4m3fn", 128, True, skip=1)
    assert np.all(got["q"] == 0xA5) and np.all(got["q_t"] == 0x5A)
    assert np.all(got["amax_rg"] == -1.0) and np.all(got["inv_cg"] == -1.0)


def test_many_tensors_in_one_list(A, dev):
    """3000 tensors (sizes 0..40 plus a few over a chunk) in one list through
    the check and the AdamW step: the per-list tables of a large ragged list."""
    rng = np.random.default_rng(140)
    sizes = list(rng.integers(0, 41, 3000))
    sizes[100], sizes[2000] = 16385, 40001
    master_h = [(rng.standard_normal(k) * 0.02).astype(np.float32) for k in sizes]
    P = _device_views(master_h, "f32", dev, True)
    M = _device_views([np.zeros(k, np.float32) for k in sizes], "f32", dev, True)
    V = _device_views([np.zeros(k, np.float32) for k in sizes], "f32", dev, True)
    gh = _grads_host(rng, sizes, "bf16", sigma=1e-3)
    G = _device_views(gh, "bf16", dev, True)
    B = _device_views([np.zeros(k, np.uint16) for k in sizes], "bf16", dev, True)
    Ls = [A.amp_tensor_list_create(x) for x in (P, M, V, G, B)]
    fi = torch.zeros(1, dtype=torch.int32, device=dev)
    step = torch.zeros(1, dtype=torch.int32, device=dev)
    A.amp_unscale_check(Ls[3], None, fi)
    assert int(fi.item()) == O.unscale_check([h.copy() for h in gh], "bf16", 1.0) == 0
    A.amp_adamw_master_step(*Ls, None, fi, step, 1e-3, 0.9, 0.95, 1e-8, 0.1)
    rp = [x.copy() for x in master_h]
    rm = [np.zeros(k, np.float32) for k in sizes]
    rv = [np.zeros(k, np.float32) for k in sizes]
    rb = [np.zeros(k, np.uint16) for k in sizes]
    O.adamw_master_step(rp, rm, rv, gh, "bf16", rb, None, 0, 0, 1e-3, 0.9, 0.95, 1e-8, 0.1)
    torch.cuda.synchronize()
    for i in range(len(sizes)):
        assert np.array_equal(to_host_bits(P[i]).view(np.uint32), rp[i].view(np.uint32)), i
        assert np.array_equal(to_host_bits(B[i]), rb[i]), i
    for L in Ls:
        L.close()


def test_amax_fold_propagates_nan_and_inf(A, dev):
    """The amax the AdamW pass folds from the bf16 copy: a NaN master makes the
    slot NaN, an infinite one makes it inf, as the oracle's max does."""
    sizes = [5000, 5000, 5000]
    master_h = [np.full(k, 0.5, np.float32) for k in sizes]
    master_h[0][1234] = np.nan
    master_h[1][4999] = np.inf
    P = _device_views(master_h, "f32", dev, False)
    M = _device_views([np.zeros(k, np.float32) for k in sizes], "f32", dev, False)
    V = _device_views([np.zeros(k, np.float32) for k in sizes], "f32", dev, False)
    gh = [np.zeros(k, np.uint16) for k in sizes]
    G = _device_views(gh, "f16", dev, False)
    B = _device_views([np.zeros(k, np.uint16) for k in sizes], "bf16", dev, False)
    Ls = [A.amp_tensor_list_create(x) for x in (P, M, V, G, B)]
    A.amp_tensor_list_set_amax_slots(Ls[4], [0, 1, 2])
    amax = torch.zeros(3, device=dev)
    step = torch.zeros(1, dtype=torch.int32, device=dev)
    A.amp_adamw_master_step(*Ls, None, None, step, 1e-3, 0.9, 0.999, 1e-8, 0.0, amax=amax)
    ram = np.zeros(3, np.float32)
    rp = [x.copy() for x in master_h]
    O.adamw_master_step(rp, [np.zeros(k, np.float32) for k in sizes],
                        [np.zeros(k, np.float32) for k in sizes], gh, "f16",
                        [np.zeros(k, np.uint16) for k in sizes], None, 0, 0, 1e-3, 0.9, 0.999,
                        1e-8, 0.0, amax_slot=[0, 1, 2], amax=ram)
    got = to_host_bits(amax)
    assert np.isnan(got[0]) and np.isnan(ram[0])
    assert got[1] == ram[1] == np.inf
    assert got[2] == ram[2]
    for L in Ls:
        L.close()
