"""Pins of the CPU oracle against what the pages and the mathematics fix.

Nothing here compares the oracle with itself: every expected value is either
printed on the pages (fixtures under tests/golden/, each with its citation),
a closed form, an independent library routine (numpy / torch CPU casts,
torch.optim.AdamW), an invariant, or brute force on tiny inputs.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from workloads import amp_config, host_grads, host_master

F32 = np.float32


def f32(x):
    return np.float32(x)


# ------------------------------------------------------------------ formats
def test_format_constants(golden):
    g = golden("format_constants.json")
    assert O.fmt_max("f16") == g["max"]["f16"]
    assert O.fmt_max("e4m3fn") == g["max"]["e4m3fn"]
    assert O.fmt_max("e5m2") == g["max"]["e5m2"]
    def two_digits(v):            # the pages print these to two significant digits
        return float(f"{v:.1e}")
    assert two_digits(O.fmt_max("bf16")) == g["max"]["bf16_approx"]
    # smallest positive normal: exponent field 1, fraction 0
    assert two_digits(O.decode("f16", np.array([0x0400]))[0]) == g["min_normal_approx"]["f16"]
    assert two_digits(O.decode("bf16", np.array([0x0080]))[0]) == g["min_normal_approx"]["bf16"]
    # bit layouts: the fraction width sets the spacing just above 1.0
    for dt, (s, e, m) in g["layouts"].items():
        one = {"f16": 0x3C00, "bf16": 0x3F80}[dt]
        assert O.decode(dt, np.array([one + 1]))[0] - 1.0 == 2.0 ** -m
        # exponent width: max exponent field gives inf (IEEE specials)
        assert np.isinf(O.decode(dt, np.array([((1 << e) - 1) << m]))[0])


def test_decode_f16_exhaustive_vs_numpy():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = O.decode("f16", bits)
    ref = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


@pytest.mark.parametrize("dt,tdt", [("bf16", torch.bfloat16), ("e4m3fn", torch.float8_e4m3fn),
                                     ("e5m2", torch.float8_e5m2)])
def test_decode_exhaustive_vs_torch(dt, tdt):
    n = 1 << (16 if dt == "bf16" else 8)
    bits = np.arange(n, dtype=np.uint32).astype(np.uint16 if dt == "bf16" else np.uint8)
    ours = O.decode(dt, bits)
    tb = torch.from_numpy(bits.view(np.int16) if dt == "bf16" else bits.view(np.int8))
    ref = tb.view(tdt).to(torch.float32).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _rounding_class_sweep():
    """All 2^20 values of the top 20 bits of an fp32 pattern, each with the
    low 12 bits in {0, 1, 0x7FF, 0x800, 0x801, 0xFFF}: every sign, exponent and
    kept-fraction combination of the 8/16-bit formats, with the round bit and
    the sticky bits below it both clear, set and at the tie."""
    hi = (np.arange(1 << 20, dtype=np.uint64) << 12)
    lows = np.array([0, 1, 0x7FF, 0x800, 0x801, 0xFFF], np.uint64)
    return (hi[:, None] | lows[None, :]).astype(np.uint32).ravel().view(np.float32)


@pytest.fixture(scope="module")
def sweep():
    return _rounding_class_sweep()


def test_encode_f16_vs_numpy(sweep):
    ours = O.encode("f16", sweep)
    with np.errstate(over="ignore", invalid="ignore"):
        ref = sweep.astype(np.float16)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours.view(np.float16)), nan)
    assert np.all(ours[nan] == 0x7E00)            # canonical NaN reading
    assert np.array_equal(ours[~nan], ref[~nan].view(np.uint16))


def test_encode_bf16_vs_torch(sweep):
    ours = O.encode("bf16", sweep)
    ref = torch.from_numpy(sweep).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(sweep)
    assert np.all(ours[nan] == 0x7FC0)
    assert np.array_equal(ours[~nan], ref[~nan])


@pytest.mark.parametrize("dt,tdt", [("e4m3fn", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_encode_fp8_vs_torch_in_range(sweep, dt, tdt):
    """On the range the quantizer feeds the encoder (|y| <= fp8_max after the
    clamp) the oracle's RNE encoder agrees bit for bit with torch's cast."""
    m = O.fmt_max(dt)
    x = sweep[np.abs(sweep) <= m]
    ours = O.encode(dt, x)
    ref = torch.from_numpy(x).to(tdt).view(torch.int8).numpy().view(np.uint8)
    assert np.array_equal(ours, ref)


def test_encode_fp8_overflow_and_specials():
    # e4m3fn has no infinity: beyond the largest finite value rounding overflows to NaN
    assert O.encode("e4m3fn", np.array([448.0, 464.0, 465.0, np.inf, np.nan], F32)).tolist() == \
        [0x7E, 0x7E, 0x7F, 0x7F, 0x7F]
    # e5m2: IEEE-like; 61440 is the tie between 57344 and 2^16 -> even -> inf
    assert O.encode("e5m2", np.array([57344.0, 61439.0, 61440.0, -np.inf, np.nan], F32)).tolist() == \
        [0x7B, 0x7B, 0x7C, 0xFC, 0x7E]
    # signed zeros and the smallest subnormals
    assert O.encode("e4m3fn", np.array([-0.0, 2.0 ** -9, -2.0 ** -10, 2.0 ** -10 * 1.0001], F32)).tolist() == \
        [0x80, 0x01, 0x80, 0x01]


# -------------------------------------------------------- worked examples
def test_fp16_small_update_lost(golden):
    g = golden("fp16_small_update_example.json")
    w = O.encode("f16", np.array([g["w0"]], F32))
    u = O.decode("f16", O.encode("f16", np.array([g["update"]], F32)))
    s = O.decode("f16", w)[0] + u[0]            # fp32 sum of the two fp16 values
    res = O.decode("f16", O.encode("f16", np.array([s], F32)))[0]
    assert res == g["fp16_result"]
    spacing = O.decode("f16", w + 1)[0] - O.decode("f16", w)[0]
    assert abs(spacing - g["fp16_spacing_at_w0_approx"]) < 0.1 * g["fp16_spacing_at_w0_approx"]
    # the fp32 master keeps it
    assert f32(g["w0"]) + f32(g["update"]) != f32(g["w0"])


def test_bf16_master_copy_example(golden):
    g = golden("master_weight_bf16_example.json")
    w0, d = f32(g["w0"]), f32(g["delta"])
    w_bits = O.encode("bf16", np.array([w0], F32))
    assert O.decode("bf16", w_bits)[0] - O.decode("bf16", w_bits - 1)[0] == g["bf16_spacing_at_w0"]
    assert O.decode("bf16", w_bits - 1)[0] == g["bf16_next_below_w0"]
    master, bf_only = w0, O.decode("bf16", w_bits)[0]
    copies, only = [], []
    for _ in range(g["steps"]):
        master = F32(master + d)                     # fp32 master update
        copies.append(float(O.decode("bf16", O.encode("bf16", np.array([master], F32)))[0]))
        bf_only = O.decode("bf16", O.encode("bf16", np.array([F32(bf_only + d)], F32)))[0]
        only.append(float(bf_only))
    assert copies == g["bf16_copy_of_fp32_master"]
    assert only == g["bf16_only_parameter"]


def test_bf16_master_copy_example_through_adamw(golden):
    """Same example driven by the oracle's AdamW: a constant gradient with
    wd = 0 gives the bias-corrected update lr * g / (|g| + eps) = lr every
    step, so lr = 0.001 reproduces the page's -0.001 per step."""
    g = golden("master_weight_bf16_example.json")
    master = [np.array([g["w0"]], F32)]
    m, v = [np.zeros(1, F32)], [np.zeros(1, F32)]
    bf = [np.zeros(1, np.uint16)]
    step, copies, masters = 0, [], []
    for _ in range(g["steps"]):
        grads = [np.array([1.0], F32)]
        step = O.adamw_master_step(master, m, v, grads, "f32", bf, None, 0, step,
                                   -g["delta"], 0.9, 0.999, 1e-12, 0.0)
        copies.append(float(O.decode("bf16", bf[0])[0]))
        masters.append(float(master[0][0]))
    assert copies == g["bf16_copy_of_fp32_master"]
    for k, mv in enumerate(masters, 1):   # closed form 1.25 - 0.001 k, to fp32 rounding
        assert abs(mv - (g["w0"] + k * g["delta"])) <= 4 * 2.0 ** -23 * 1.25
    assert step == g["steps"]


# ---------------------------------------------------------- scale machine
def _run_trace(init, interval, inf_steps, steps):
    s, t, opt = init, 0, 0
    rows = []
    for k in range(1, steps + 1):
        fi = int(k in inf_steps)
        opt += 0 if fi else 1
        s, t, fi_after = O.update_scale(s, t, fi, 2.0, 0.5, interval)
        assert fi_after == 0
        rows.append((s, t, opt, bool(fi)))
    return rows


def test_scaler_trace_tiny(golden):
    tr = golden("scaler_traces.json")["traces"]["tiny_interval2_inf_at_2"]
    rows = _run_trace(tr["init_scale"], tr["growth_interval"], tr["inf_steps"], tr["steps"])
    assert [r[0] for r in rows] == tr["scale"]
    assert [r[1] for r in rows] == tr["tracker"]
    assert [r[3] for r in rows] == tr["skipped"]


def test_scaler_trace_interval10(golden):
    tr = golden("scaler_traces.json")["traces"]["interval10_inf_at_7_27_47"]
    rows = _run_trace(tr["init_scale"], tr["growth_interval"], tr["inf_steps"], tr["steps"])
    grew = [k for k in range(2, tr["steps"] + 1) if rows[k - 1][0] > rows[k - 2][0]]
    assert grew == tr["growth_at"]
    assert rows[-1][0] == tr["final_scale"] and rows[-1][1] == tr["final_tracker"]


def test_scaler_growth_overflow_keeps_scale_and_clears_amax():
    big = float(np.finfo(np.float32).max)
    amax = np.array([3.0, 5.0], F32)
    s, t, fi = O.update_scale(big, 0, 0, 2.0, 0.5, 1, amax)
    assert s == big and t == 0 and fi == 0 and np.all(amax == 0)


# --------------------------------------------------------- unscale / check
def test_unscale_check_detects_and_unscales():
    S = 65536.0
    g = [np.array([1.0, -2.0, 0.5], np.float16).view(np.uint16).copy(),
         (np.arange(257, dtype=np.float16) * np.float16(0.25)).view(np.uint16).copy()]
    assert O.unscale_check([a.copy() for a in g], "f16", S) == 0
    for val in (np.inf, -np.inf, np.nan):
        h = [a.copy() for a in g]
        h[1][256] = np.array([val], np.float16).view(np.uint16)[0]     # tail element
        assert O.unscale_check(h, "f16", S) == 1
    # never cleared: an incoming flag survives a clean list
    assert O.unscale_check([a.copy() for a in g], "f16", S, found_inf=1) == 1
    # S = 0: 1/S = inf, so even 0 * inf = NaN is non-finite
    assert O.unscale_check([np.zeros(4, np.uint16)], "f16", 0.0) == 1
    # finite fp16 times a huge 1/S overflows fp32
    assert O.unscale_check([np.array([65504.0], np.float16).view(np.uint16)], "f16", 1e-35) == 1
    # in place: the stored value becomes fp16(g / S)
    h = [a.copy() for a in g]
    O.unscale_check(h, "f16", S, inplace=True)
    np.testing.assert_array_equal(h[0].view(np.float16).astype(np.float64),
                                  (g[0].view(np.float16).astype(np.float64) / S)
                                  .astype(np.float16).astype(np.float64))


# ------------------------------------------------------------------ AdamW
def _adamw_oracle(p0, grads_seq, lr, b1, b2, eps, wd, gdt="f32", scale=None):
    master = [p.copy() for p in p0]
    m = [np.zeros_like(p) for p in p0]
    v = [np.zeros_like(p) for p in p0]
    step = 0
    for g in grads_seq:
        step = O.adamw_master_step(master, m, v, g, gdt, None, scale, 0, step, lr, b1, b2, eps, wd)
    return master, m, v, step


def test_adamw_first_step_closed_form():
    """t = 1 from m = v = 0: m_hat = g and v_hat = g^2 exactly, so
    p1 = p0 (1 - lr wd) - lr g / (|g| + eps)."""
    rng = np.random.default_rng(1)
    p0 = [rng.standard_normal(1000).astype(F32)]
    g = [rng.standard_normal(1000).astype(F32) * F32(1e-3)]
    lr, wd, eps = 1e-3, 0.01, 1e-8
    p, m, v, step = _adamw_oracle(p0, [g], lr, 0.9, 0.999, eps, wd)
    p0d, gd = p0[0].astype(np.float64), g[0].astype(np.float64)
    exact = p0d * (1 - lr * wd) - lr * gd / (np.abs(gd) + eps)
    # fp32 rounding of each term: relative to the size of the terms, not of
    # their difference (p0 (1 - lr wd) and lr can nearly cancel)
    assert np.all(np.abs(p[0] - exact) <= 1e-6 * (np.abs(p0d) + lr))
    np.testing.assert_allclose(m[0], 0.1 * gd, rtol=1e-6)
    np.testing.assert_allclose(v[0], 0.001 * gd * gd, rtol=1e-6)
    assert step == 1


def test_adamw_pure_decay_closed_form():
    """g = 0: both moments stay 0, the Adam term vanishes and each step only
    multiplies by the fp32 factor (1 - lr wd): p_t = p0 * decay^t in fp32."""
    p0 = [np.array([1.0, -0.5, 3.0e-3, 0.0], F32)]
    lr, wd, T = 1e-2, 0.1, 25
    p, m, v, _ = _adamw_oracle(p0, [[np.zeros(4, F32)]] * T, lr, 0.9, 0.95, 1e-8, wd)
    expect = p0[0].copy()
    decay = F32(1.0 - lr * wd)
    for _ in range(T):
        expect = (expect * decay).astype(F32)
    assert np.array_equal(p[0], expect)
    assert not m[0].any() and not v[0].any()


def test_adamw_matches_torch_optim():
    """Independent library: torch.optim.AdamW on CPU fp32, 10 steps."""
    rng = np.random.default_rng(7)
    sizes = [1000, 4096, 257]
    p0 = [rng.standard_normal(n).astype(F32) * F32(0.02) for n in sizes]
    gseq = [[rng.standard_normal(n).astype(F32) * F32(1e-3) for n in sizes] for _ in range(10)]
    hp = dict(lr=3e-4, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1)
    p, m, v, _ = _adamw_oracle(p0, gseq, hp["lr"], *hp["betas"], hp["eps"], hp["weight_decay"])
    tp = [torch.nn.Parameter(torch.from_numpy(x.copy())) for x in p0]
    opt = torch.optim.AdamW(tp, foreach=False, fused=False, **hp)
    for gs in gseq:
        for t, g in zip(tp, gs):
            t.grad = torch.from_numpy(g.copy())
        opt.step()
    for i, t in enumerate(tp):
        st = opt.state[t]
        for ours, ref in ((p[i], t.detach().numpy()), (m[i], st["exp_avg"].numpy()),
                          (v[i], st["exp_avg_sq"].numpy())):
            floor = 1e-6 * np.sqrt(np.mean(ref.astype(np.float64) ** 2))
            err = np.abs(ours.astype(np.float64) - ref)
            assert np.all(err <= 1e-6 * np.maximum(np.abs(ours), np.abs(ref)) + floor)


def test_adamw_skip_changes_nothing():
    rng = np.random.default_rng(3)
    master = [rng.standard_normal(300).astype(F32)]
    m, v = [rng.standard_normal(300).astype(F32)], [rng.random(300).astype(F32)]
    bf = [np.full(300, 0x1234, np.uint16)]
    snap = [a[0].copy() for a in (master, m, v, bf)]
    amax = np.array([7.0], F32)
    st = O.adamw_master_step(master, m, v, [np.full(300, 0x3C00, np.uint16)], "f16", bf, 65536.0,
                             1, 5, 1e-3, 0.9, 0.999, 1e-8, 0.01, amax_slot=[0], amax=amax)
    assert st == 5 and amax[0] == 7.0
    for a, s in zip((master, m, v, bf), snap):
        assert np.array_equal(a[0], s)


def test_adamw_bf16_emit_and_amax():
    rng = np.random.default_rng(4)
    master = [rng.standard_normal(n).astype(F32) for n in (100, 37)]
    m = [np.zeros_like(x) for x in master]
    v = [np.zeros_like(x) for x in master]
    bf = [np.zeros(x.size, np.uint16) for x in master]
    amax = np.zeros(1, F32)
    O.adamw_master_step(master, m, v, [np.zeros(x.size, F32) for x in master], "f32", bf, None,
                        0, 0, 1e-3, 0.9, 0.999, 1e-8, 0.0, amax_slot=[-1, 0], amax=amax)
    ref = [torch.from_numpy(x).to(torch.bfloat16) for x in master]
    for b, r in zip(bf, ref):
        assert np.array_equal(b, r.view(torch.int16).numpy().view(np.uint16))
    assert amax[0] == ref[1].abs().max().float().item()


# ----------------------------------------------------------- FP8 quantizer
@pytest.mark.parametrize("fmt,top", [("e4m3fn", 0x7E), ("e5m2", 0x7B)])
def test_quant_amax_maps_to_fp8_max(fmt, top):
    rng = np.random.default_rng(11)
    x = rng.standard_normal((33, 70)).astype(F32)
    x[5, 7] = -np.abs(x).max() * 3          # unique largest magnitude, negative
    x[20, 69] = -x[5, 7]                    # and its positive twin
    q, qt, inv, amax = O.fp8_quant_tensorwise(x.ravel(), "f32", 33, 70, fmt)
    q = q.reshape(33, 70)
    assert amax == np.abs(x).max()
    assert q[5, 7] == (top | 0x80) and q[20, 69] == top
    deq = O.decode(fmt, q) * inv
    assert np.max(np.abs(deq)) == pytest.approx(amax, rel=1e-6)
    assert np.array_equal(qt.reshape(70, 33), q.T)       # the column-major copy


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
def test_quant_zero_tensor_uses_eps(fmt):
    q, qt, inv, amax = O.fp8_quant_tensorwise(np.zeros(64 * 32, np.uint16), "bf16", 64, 32, fmt,
                                              eps=1e-12)
    assert amax == 0.0 and not q.any() and not qt.any()
    assert inv == F32(1e-12 / O.fmt_max(fmt))


@pytest.mark.parametrize("fmt,tdt", [("e4m3fn", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
@pytest.mark.parametrize("shape", [(1, 1), (3, 5), (17, 31), (64, 130)])
def test_quant_vs_torch_ops(fmt, tdt, shape):
    """Tiny tensors: torch CPU ops (abs-max, fp64 scale, fp32 multiply,
    clamp, library fp8 cast) give the same bytes and inv_scale."""
    rng = np.random.default_rng(shape[0] * 100 + shape[1])
    x = (rng.standard_normal(shape) * 10 ** rng.uniform(-3, 3)).astype(F32)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16).ravel()
    q, qt, inv, amax = O.fp8_quant_tensorwise(bits, "bf16", *shape, fmt)
    mx = float(torch.finfo(tdt).max)
    am = xb.float().abs().max()
    sc = mx / am.double().clamp(min=1e-12)
    ref = (xb.float() * sc).clamp(-mx, mx).to(tdt).view(torch.int8).numpy().view(np.uint8)
    assert amax == am.item()
    assert np.array_equal(q, ref.ravel())
    assert inv == sc.reciprocal().float().item()
    assert np.array_equal(qt.reshape(shape[1], shape[0]), ref.T)


@pytest.mark.parametrize("fmt,tdt", [("e4m3fn", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_quant_amax_propagates_nan(fmt, tdt):
    """[FP8] §2 takes amax = x.abs().max(), which propagates NaN: one NaN makes
    the amax, the scale and so every output NaN, as torch's own ops give."""
    rng = np.random.default_rng(12)
    x = rng.standard_normal((9, 20)).astype(F32)
    x[4, 13] = np.nan
    xb = torch.from_numpy(x).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16).ravel()
    q, qt, inv, amax = O.fp8_quant_tensorwise(bits, "bf16", 9, 20, fmt)
    mx = float(torch.finfo(tdt).max)
    am = xb.float().abs().max()
    sc = mx / am.double().clamp(min=1e-12)
    ref = (xb.float() * sc).clamp(-mx, mx).to(tdt).float().numpy()
    assert np.isnan(am.item()) and np.isnan(amax) and np.isnan(inv)
    assert np.isnan(ref).all()
    assert np.isnan(O.decode(fmt, q)).all() and np.isnan(O.decode(fmt, qt)).all()


def test_quant_dequant_error_bound():
    """RNE error: |deq - x| <= half the fp8 spacing at |x*scale|, mapped back."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal(4096).astype(F32)
    q, _, inv, amax = O.fp8_quant_tensorwise(x, "f32", 64, 64, "e4m3fn", transposed=False)
    y = np.abs(x.astype(np.float64) * F32(448.0 / amax))
    e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
    half_spacing = 0.5 * 2.0 ** (e - 3)
    err = np.abs(O.decode("e4m3fn", q).astype(np.float64) - x.astype(np.float64) * F32(448.0 / amax))
    assert np.all(err <= half_spacing * (1 + 1e-6))


# ------------------------------------------------------------ composition
def test_tiny_config_trace_through_oracle_step(golden):
    """Config 'tiny': the composed step reproduces the hand-derived scaler
    trace, skips exactly step 2 and leaves the state untouched there."""
    cfg = amp_config("tiny")
    tr = golden("scaler_traces.json")["traces"]["tiny_interval2_inf_at_2"]
    orc = O.AmpStepOracle(host_master(cfg), cfg.grad_dtype, cfg.lr, cfg.beta1, cfg.beta2, cfg.eps,
                          cfg.weight_decay, cfg.init_scale, cfg.growth_factor, cfg.backoff_factor,
                          cfg.growth_interval)
    for k in range(1, cfg.steps + 1):
        before = [x.copy() for x in orc.master]
        fi = orc.run(host_grads(cfg, k, orc.scale))
        assert bool(fi) == tr["skipped"][k - 1]
        if fi:
            assert all(np.array_equal(a, b) for a, b in zip(before, orc.master))
        assert orc.scale == tr["scale"][k - 1] and orc.tracker == tr["tracker"][k - 1]
        assert orc.step == tr["optimizer_step"][k - 1]


# --------------------------------------------------- grad-norm clipping
def test_grad_norm_closed_form():
    """Constant gradients c (fp16, scaled by S = 2^k): norm = |c| sqrt(N)."""
    S = 1024.0
    sizes = [100, 300, 24]
    c = np.float16(3.0)
    grads = [np.full(n, c, np.float16).view(np.uint16) for n in sizes]
    ss = O.grad_sumsq(grads, "f16", S)
    assert ss == (3.0 / S) ** 2 * sum(sizes)
    assert O.clip_coef(ss, 1e9) == 1.0
    assert O.clip_coef(0.0, 1.0) == 1.0
    assert np.isnan(O.clip_coef(float("nan"), 1.0))


def test_clip_matches_torch_clip_grad_norm():
    """Independent library: unscale, torch.nn.utils.clip_grad_norm_, then
    torch.optim.AdamW, vs the oracle's fused clip + AdamW over 5 steps."""
    rng = np.random.default_rng(9)
    sizes = [1000, 4096, 257]
    S = 4096.0
    p0 = [rng.standard_normal(n).astype(F32) * F32(0.02) for n in sizes]
    hp = dict(lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01)
    max_norm = 0.05
    gseq = [[(rng.standard_normal(n) * 1e-3 * S).astype(np.float16).view(np.uint16) for n in sizes]
            for _ in range(5)]
    master = [x.copy() for x in p0]
    m = [np.zeros_like(x) for x in p0]
    v = [np.zeros_like(x) for x in p0]
    step = 0
    tp = [torch.nn.Parameter(torch.from_numpy(x.copy())) for x in p0]
    opt = torch.optim.AdamW(tp, foreach=False, fused=False, **hp)
    for gs in gseq:
        ss = O.grad_sumsq(gs, "f16", S)
        coef = O.clip_coef(ss, max_norm)
        assert coef < 1.0
        step = O.adamw_master_step(master, m, v, gs, "f16", None, S, 0, step, hp["lr"],
                                   *hp["betas"], hp["eps"], hp["weight_decay"], clip=coef)
        for t, g in zip(tp, gs):
            t.grad = torch.from_numpy(g.view(np.float16).astype(np.float32) / np.float32(S))
        tn = torch.nn.utils.clip_grad_norm_(tp, max_norm, foreach=False)
        assert abs(float(tn) - np.sqrt(ss)) <= 1e-6 * np.sqrt(ss)
        opt.step()
    for i, t in enumerate(tp):
        ref = t.detach().numpy()
        floor = 1e-6 * np.sqrt(np.mean(ref.astype(np.float64) ** 2))
        assert np.all(np.abs(master[i].astype(np.float64) - ref)
                      <= 1e-6 * np.maximum(np.abs(master[i]), np.abs(ref)) + floor)


def test_clip_factor_one_is_the_unclipped_step():
    rng = np.random.default_rng(10)
    p0 = [rng.standard_normal(500).astype(F32)]
    g = [rng.standard_normal(500).astype(F32)]
    a = _adamw_oracle(p0, [g], 1e-3, 0.9, 0.999, 1e-8, 0.01)
    master = [p0[0].copy()]
    m, v = [np.zeros(500, F32)], [np.zeros(500, F32)]
    O.adamw_master_step(master, m, v, g, "f32", None, None, 0, 0, 1e-3, 0.9, 0.999, 1e-8, 0.01,
                        clip=1.0)
    assert np.array_equal(master[0], a[0][0]) and np.array_equal(m[0], a[1][0])


# ------------------------------------------------------ delayed FP8 scaling
@pytest.mark.parametrize("hist_len", [1, 3])
def test_delayed_scaling_uses_previous_amax(hist_len):
    """'第20章 量化与混合精度训练' §20.5.9: the scale of a step comes from the
    amax of earlier steps.  With history length H the cast of step t uses the
    max of the amaxes of the last H non-skipped steps' bf16 copies (the
    initial copy counting as the first); a skipped step leaves it unchanged."""
    rng = np.random.default_rng(60)
    shapes = [(64, 96), None, (32, 40)]
    sizes = [64 * 96, 300, 32 * 40]
    master = [(rng.standard_normal(n) * 0.02).astype(F32) for n in sizes]
    orc = O.AmpStepOracle(master, "f16", 1e-2, 0.9, 0.999, 1e-8, 0.0, 1024.0, 2.0, 0.5, 100,
                          fp8_shapes=shapes, fp8_scaling="delayed", hist_len=hist_len)
    amaxes = {0: [np.abs(O.decode("bf16", orc.bf16[0])).max()],
              2: [np.abs(O.decode("bf16", orc.bf16[2])).max()]}
    for k in range(5):
        g = [(rng.standard_normal(n) * 1e-3 * 1024).astype(np.float16).view(np.uint16) for n in sizes]
        if k == 2:
            g[1][5] = 0x7C00
        inv_before = orc.inv_scale.copy()
        fi = orc.run(g)
        for i, slot in ((0, 0), (2, 1)):
            if fi:
                assert orc.inv_scale[slot] == inv_before[slot]
                continue
            used = max(amaxes[i][-hist_len:])
            assert orc.inv_scale[slot] == np.float32(1.0 / (448.0 / max(float(used), 1e-12)))
            amaxes[i].append(np.abs(O.decode("bf16", orc.bf16[i])).max())
        assert fi == (k == 2)
    for i, slot in ((0, 0), (2, 1)):
        want = list(reversed(amaxes[i][-hist_len:]))
        want += [0.0] * (hist_len - len(want))
        assert np.array_equal(orc.hist[slot], np.array(want, F32))


# ----------------------------------------------------------- rowwise FP8
@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
def test_rowwise_reduces_to_tensorwise(fmt):
    """One row: the row scale is the tensor scale; one column: the column
    scale of the transposed copy is the tensor scale (the pinned quantizer)."""
    rng = np.random.default_rng(80)
    x = (rng.standard_normal(333) * 7).astype(F32)
    r = O.fp8_quant_rowwise(x, "f32", 1, 333, fmt)
    q, qt, inv, amax = O.fp8_quant_tensorwise(x, "f32", 1, 333, fmt)
    assert np.array_equal(r["q"], q) and r["inv_row"][0] == np.float32(inv) and r["amax_row"][0] == amax
    c = O.fp8_quant_rowwise(x, "f32", 333, 1, fmt)
    assert np.array_equal(c["q_t"], qt) and c["inv_col"][0] == np.float32(inv)


@pytest.mark.parametrize("fmt,top", [("e4m3fn", 0x7E), ("e5m2", 0x7B)])
def test_rowwise_each_row_and_column_reaches_fp8_max(fmt, top):
    rng = np.random.default_rng(81)
    rows, cols = 37, 53
    x = (rng.standard_normal((rows, cols)) * 10 ** rng.uniform(-3, 3, size=(rows, 1))).astype(F32)
    r = O.fp8_quant_rowwise(x.ravel(), "f32", rows, cols, fmt)
    q = r["q"].reshape(rows, cols)
    qt = r["q_t"].reshape(cols, rows)
    for i in range(rows):
        j = int(np.argmax(np.abs(x[i])))
        assert q[i, j] & 0x7F == top
    for j in range(cols):
        i = int(np.argmax(np.abs(x[:, j])))
        assert qt[j, i] & 0x7F == top
    # a row scaled by a power of two keeps its bytes (its scale follows it)
    y = x.copy()
    y[4] *= 8.0
    r2 = O.fp8_quant_rowwise(y.ravel(), "f32", rows, cols, fmt)
    assert np.array_equal(r2["q"].reshape(rows, cols)[4], q[4])


@pytest.mark.parametrize("fmt,tdt", [("e4m3fn", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_rowwise_vs_torch_ops(fmt, tdt):
    rng = np.random.default_rng(82)
    rows, cols = 24, 40
    xb = torch.from_numpy((rng.standard_normal((rows, cols)) * 3).astype(F32)).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16).ravel()
    r = O.fp8_quant_rowwise(bits, "bf16", rows, cols, fmt)
    mx = float(torch.finfo(tdt).max)
    for dim, key, qk in ((1, "row", "q"), (0, "col", "q_t")):
        am = xb.float().abs().amax(dim=dim, keepdim=True)
        sc = mx / am.double().clamp(min=1e-12)
        ref = (xb.float() * sc).clamp(-mx, mx).to(tdt).view(torch.int8).numpy().view(np.uint8)
        if dim == 0:
            ref = ref.T
        assert np.array_equal(r[qk], ref.ravel())
        assert np.array_equal(r["inv_" + key], sc.reciprocal().float().numpy().ravel())
        assert np.array_equal(r["amax_" + key], am.numpy().ravel())


# --------------------------------------------------------- group-wise FP8
@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
@pytest.mark.parametrize("rows,cols", [(5, 7), (33, 64)])
def test_groupwise_with_one_group_is_rowwise(fmt, rows, cols):
    """A group at least as long as a row (a column) is the whole row (column):
    the group-wise quantizer then reduces to the row-wise one."""
    rng = np.random.default_rng(83)
    x = (rng.standard_normal(rows * cols) * 2).astype(F32)
    g = O.fp8_quant_groupwise(x, "f32", rows, cols, fmt, group=max(rows, cols) + 3)
    r = O.fp8_quant_rowwise(x, "f32", rows, cols, fmt)
    assert np.array_equal(g["q"], r["q"]) and np.array_equal(g["q_t"], r["q_t"])
    for a, b in (("amax_rg", "amax_row"), ("scale_rg", "scale_row"), ("inv_rg", "inv_row"),
                 ("amax_cg", "amax_col"), ("scale_cg", "scale_col"), ("inv_cg", "inv_col")):
        assert np.array_equal(g[a].view(np.uint32), r[b].view(np.uint32)), a


@pytest.mark.parametrize("fmt,tdt", [("e4m3fn", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
@pytest.mark.parametrize("group", [4, 32, 128])
def test_groupwise_vs_torch_ops(fmt, tdt, group):
    """Each group of `group` elements (the last one ragged) through torch CPU
    ops: abs-max, fp64 scale with the EPS floor, fp32 multiply by the scale
    rounded to fp32, clamp, library fp8 cast; rows for the row-major bytes,
    columns for the transposed copy ("第20章" §20.5.18 g128 layout)."""
    rng = np.random.default_rng(84)
    rows, cols = 70, 150
    x = rng.standard_normal((rows, cols)) * 10 ** rng.uniform(-2, 2, size=(rows, 1))
    x[3, :] = 0.0                                   # an all-zero row: its groups clamp to EPS
    xb = torch.from_numpy(x.astype(F32)).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16).ravel()
    r = O.fp8_quant_groupwise(bits, "bf16", rows, cols, fmt, group=group)
    mx = float(torch.finfo(tdt).max)
    xf = xb.float()

    def ref(m):               # m: [n, L] -> bytes, amax, inv per group along dim 1
        q = torch.empty(m.shape, dtype=torch.uint8)
        am, inv = [], []
        for i in range(m.shape[0]):
            for j0 in range(0, m.shape[1], group):
                seg = m[i, j0:j0 + group]
                a = seg.abs().max()
                sc = mx / a.double().clamp(min=1e-12)
                q[i, j0:j0 + group] = (seg * sc.float()).clamp(-mx, mx).to(tdt).view(torch.uint8)
                am.append(a.item())
                inv.append(sc.reciprocal().float().item())
        return q.numpy().ravel(), np.array(am, F32), np.array(inv, F32)

    q, am, inv = ref(xf)
    assert np.array_equal(r["q"], q)
    assert np.array_equal(r["amax_rg"], am) and np.array_equal(r["inv_rg"], inv)
    qt, amt, invt = ref(xf.T.contiguous())
    assert np.array_equal(r["q_t"], qt)
    assert np.array_equal(r["amax_cg"], amt) and np.array_equal(r["inv_cg"], invt)


# ---------------------------------------------------- stochastic rounding
def test_philox_known_answers():
    """Philox4x32-10 known-answer vectors of its authors' reference release
    (Salmon et al., 'Parallel random numbers: as easy as 1, 2, 3', SC 2011)."""
    kat = [([0, 0, 0, 0], [0, 0], [0x6627e8d5, 0xe169c58d, 0xbc57ac4c, 0x9b00dbd8]),
           ([0xffffffff] * 4, [0xffffffff] * 2, [0x408f276d, 0x41c83b0e, 0xa20bc7c6, 0x6d5451fd]),
           ([0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344], [0xa4093822, 0x299f31d0],
            [0xd16cfe09, 0x94fdcceb, 0x5001e420, 0x24126ea1])]
    for ctr, key, want in kat:
        assert O.philox4x32_10(ctr, key).tolist() == want


def test_stochastic_rounding_is_unbiased_and_on_grid():
    """'第20章 量化与混合精度训练' §20.5.14: round down or up with probability
    proportional to the distance; the expected value is the input."""
    p = np.full(200000, np.float32(1.0 + 1e-3), np.float32)        # between two bf16 values
    lo, hi = 1.0, 1.0 + 2.0 ** -7
    b = O.bf16_stochastic(p, seed=1234, step=1, tensor=0)
    vals = O.decode("bf16", b).astype(np.float64)
    assert set(np.unique(vals)) <= {lo, hi}
    frac_up = np.mean(vals == hi)
    want = (float(p[0]) - lo) / (hi - lo)
    assert abs(frac_up - want) < 5 * np.sqrt(want * (1 - want) / p.size)
    assert abs(vals.mean() - float(p[0])) < 5 * (hi - lo) * np.sqrt(want * (1 - want) / p.size)
    # exact grid values, zeros, inf and NaN are left as RNE leaves them
    special = np.array([1.25, -0.0, 0.0, np.inf, -np.inf, np.nan, 65536.0], np.float32)
    assert np.array_equal(O.bf16_stochastic(special, 7, 3, 1), O.encode("bf16", special))
    # negative values mirror positive ones (rounding away from zero is "up")
    q = O.bf16_stochastic(-p[:1000], 1234, 1, 0)
    assert np.array_equal(q & 0x7FFF, b[:1000])


def test_stochastic_rounding_probability_is_exact():
    """Over all 2^16 values of the 16 random bits, the fraction that rounds
    away from zero is exactly (|p| - |lo|) / (|hi| - |lo|), lo and hi the
    neighbouring bf16 values, computed here in fp64 from their decoded values;
    values on the bf16 grid never move."""
    u = np.arange(1 << 16, dtype=np.uint32)
    for pv in [1.0 + 1e-3, 1.25, -3.3e-5, 3.0e38, 1.0e-40, -7.77e5, 2.0 ** -133]:
        p = np.float32(pv)
        out = np.array([O.lib().orc_bf16_stochastic(float(p), int(k)) for k in u], np.uint16)
        mag = abs(float(p))
        # bf16 values next to |p|: decode every bf16 magnitude and bracket |p|
        grid = O.decode("bf16", np.arange(0x7F80, dtype=np.uint16)).astype(np.float64)
        j = np.searchsorted(grid, mag, side="right") - 1
        lo = grid[j]
        hi = grid[j + 1] if j + 1 < grid.size else np.inf
        vals = np.abs(O.decode("bf16", out).astype(np.float64))
        assert set(np.unique(vals)) <= {lo, hi}, pv
        n_up = int(np.sum(vals == hi))
        if mag == lo:
            assert n_up == 0, pv
        else:
            assert n_up == (mag - lo) / (hi - lo) * 65536, pv
        assert np.all(np.signbit(O.decode("bf16", out)) == np.signbit(p)), pv


@pytest.mark.parametrize("fp8_scaling", ["dynamic", "delayed"])
def test_step_oracle_stream_ids_are_only_labels(fp8_scaling):
    """AmpStepOracle's explicit random-stream words (for a subset of a larger
    set): given the words it would derive itself, the run is identical; given
    other words, the stochastically rounded copies change while master, m and
    v do not (the streams feed only the roundings)."""
    rng = np.random.default_rng(5)
    shapes = [(64, 96), None, (32, 48)]
    master = [(rng.standard_normal(64 * 96) * 0.02).astype(np.float32),
              (rng.standard_normal(300) * 0.02).astype(np.float32),
              (rng.standard_normal(32 * 48) * 0.02).astype(np.float32)]
    grads = [(rng.standard_normal(m.size) * 1e-3 * 1024).astype(np.float16).view(np.uint16)
             for m in master]
    hyper = (1e-3, 0.9, 0.999, 1e-8, 0.01, 1024.0, 2.0, 0.5, 10)
    own = [0 | (1 << 30), 0, 1 | (1 << 30)] if fp8_scaling == "delayed" else [0, 1, 2]

    def run(**kw):
        o = O.AmpStepOracle(master, "f16", *hyper, fp8_shapes=shapes, fp8_scaling=fp8_scaling,
                            sr_seed=99, **kw)
        for _ in range(2):
            o.run([g.copy() for g in grads])
        return o

    a, b = run(), run(sr_tensor_ids=own, sr_fp8_ids=[0, 1])
    c = run(sr_tensor_ids=[x + 5 for x in own], sr_fp8_ids=[7, 8])
    for i in range(3):
        assert np.array_equal(a.bf16[i], b.bf16[i])
        assert np.array_equal(a.master[i], c.master[i]) and np.array_equal(a.exp_avg_sq[i],
                                                                           c.exp_avg_sq[i])
    assert all(np.array_equal(a.fp8[i], b.fp8[i]) for i in (0, 2))
    assert not np.array_equal(a.bf16[0], c.bf16[0])
    assert not np.array_equal(a.fp8[2], c.fp8[2])


def test_adamw_with_stochastic_rounding_keeps_master_and_rounds_copy():
    rng = np.random.default_rng(62)
    p0 = [rng.standard_normal(5000).astype(F32) * F32(0.02)]
    g = [rng.standard_normal(5000).astype(F32) * F32(1e-3)]
    m1, v1 = [np.zeros(5000, F32)], [np.zeros(5000, F32)]
    m2, v2 = [np.zeros(5000, F32)], [np.zeros(5000, F32)]
    a, b = [p0[0].copy()], [p0[0].copy()]
    ba, bb = [np.zeros(5000, np.uint16)], [np.zeros(5000, np.uint16)]
    O.adamw_master_step(a, m1, v1, g, "f32", ba, None, 0, 0, 1e-3, 0.9, 0.999, 1e-8, 0.01)
    O.adamw_master_step(b, m2, v2, g, "f32", bb, None, 0, 0, 1e-3, 0.9, 0.999, 1e-8, 0.01,
                        sr_seed=99)
    assert np.array_equal(a[0], b[0]) and np.array_equal(m1[0], m2[0])      # state unchanged
    assert np.array_equal(bb[0], O.bf16_stochastic(b[0], 99, 1, 0))         # step t = 1, tensor 0
    d = bf16_ulp_steps(ba[0], bb[0])
    assert d.max() <= 1 and 0 < np.mean(d) < 1


def bf16_ulp_steps(a, b):
    key = lambda x: np.where(x & 0x8000, -(x.astype(np.int64) & 0x7FFF), x.astype(np.int64) & 0x7FFF)
    return np.abs(key(a) - key(b))


# --------------------------------------------- stochastic rounding of FP8
def _torch_fp8_grid(tdt):
    """Ascending finite non-negative magnitudes of an FP8 format, decoded by
    torch's own casts (independent of the oracle's decoder)."""
    v = torch.arange(128, dtype=torch.uint8).view(tdt).float().numpy().astype(np.float64)
    return np.unique(v[np.isfinite(v)])


FP8_SR_VALUES = {
    # normal range, binade edges, the largest gap, ties, the subnormal range
    "e4m3fn": [1.0 + 1e-3, 1.0625, 1.1, 255.9, 447.0, 300.1, 0.015625 + 1e-6, 0.0017, 2.0 ** -9 * 0.7,
               -3.3, -0.123, 1.0e-30],
    "e5m2": [1.0 + 1e-3, 1.125, 1.3, 57000.0, 40000.5, 0.000061, 2.0 ** -16 * 0.3, -7.7, -1.0e-6,
             3.0e-20],
}


@pytest.mark.parametrize("fmt,tdt", [("e4m3fn", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_fp8_stochastic_probability_is_exact(fmt, tdt):
    """'第20章 量化与混合精度训练' §20.5.14: round to the neighbour away from
    zero with probability equal to the distance ratio.  Over all 2^16 values
    of the 16 random bits, the count that rounds to hi is floor(2^16 * (|y| -
    lo) / (hi - lo)), with lo < |y| < hi the FP8 neighbours from torch's own
    decode and the ratio computed here in fp64: the ratio itself when it is a
    multiple of 2^-16 (checked on such values), else truncated."""
    grid = _torch_fp8_grid(tdt)
    u = np.arange(1 << 16, dtype=np.uint32)
    vals = list(FP8_SR_VALUES[fmt])
    # values whose ratio is an exact multiple of 2^-16: lo + m * gap / 2^16
    for j, m in ((20, 1), (40, 12345), (90, 65535), (100, 32768)):
        vals.append(float(grid[j] + m * (grid[j + 1] - grid[j]) / 65536))
    for yv in vals:
        y = np.float32(yv)
        a = abs(float(y))
        j = np.searchsorted(grid, a, side="right") - 1
        lo, hi = grid[j], grid[j + 1]
        ratio = (a - lo) / (hi - lo)
        out = O.fp8_stochastic(fmt, np.full(u.size, y), u)
        dec = torch.from_numpy(out).view(tdt).float().numpy().astype(np.float64)
        assert set(np.unique(np.abs(dec))) <= {lo, hi}, yv
        n_up = int(np.sum(np.abs(dec) == hi)) if hi != lo else 0
        assert n_up == int(np.floor(ratio * 65536)), (yv, n_up, ratio)
        if ratio * 65536 == np.floor(ratio * 65536):
            assert n_up == ratio * 65536, yv                    # the exact probability
        # hi exactly for the lowest n_up values of u
        assert np.all(np.abs(dec[:n_up]) == hi) and np.all(np.abs(dec[n_up:]) == lo), yv
        assert np.all(np.signbit(dec) == np.signbit(y)) or lo == 0.0, yv


@pytest.mark.parametrize("fmt,tdt", [("e4m3fn", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_fp8_stochastic_is_unbiased_and_keeps_grid(fmt, tdt):
    """The mean of many draws is the input (within 5 sigma); grid values,
    zeros and the saturation of [FP8] §2's clamp are as the RNE cast gives
    them for every random word; NaN is the canonical NaN."""
    rng = np.random.default_rng(7)
    grid = _torch_fp8_grid(tdt)
    for yv in (1.0 + 1e-3, 3.14159, -0.0123, 0.7 * grid[1]):
        y = np.float32(yv)
        u = rng.integers(0, 2 ** 16, 400000, dtype=np.uint64).astype(np.uint32)
        out = O.fp8_stochastic(fmt, np.full(u.size, y), u)
        dec = torch.from_numpy(out).view(tdt).float().numpy().astype(np.float64)
        a = abs(float(y))
        j = np.searchsorted(grid, a, side="right") - 1
        lo, hi = grid[j], grid[j + 1]
        assert set(np.unique(np.abs(dec))) <= {lo, hi}, yv
        p = (a - lo) / (hi - lo)
        sd = (hi - lo) * np.sqrt(p * (1 - p) / u.size)
        # the probability is truncated to a multiple of 2^-16: low by < 2^-16 * gap
        assert abs(dec.mean() - float(y)) <= 5 * sd + (hi - lo) / 65536, yv
    fmax = O.fmt_max(fmt)
    special = np.array([grid[5], -grid[40], grid[-1], 0.0, -0.0, fmax * 1.5, -np.inf, np.inf,
                        np.nan], np.float32)
    want = O.encode(fmt, np.clip(special, -fmax, fmax))                 # RNE of the clamp
    for u in (0, 1, 2 ** 15, 2 ** 16 - 1):
        got = O.fp8_stochastic(fmt, special, np.full(special.size, u, np.uint32))
        assert np.array_equal(got, want), u
    # torch's cast agrees on the saturated and on-grid values (NaN: canonical code)
    tq = torch.from_numpy(np.clip(special[:-1], -fmax, fmax)).to(tdt).view(torch.uint8).numpy()
    assert np.array_equal(want[:-1], tq)
    assert want[-1] == {"e4m3fn": 0x7F, "e5m2": 0x7E}[fmt]


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
def test_fp8_quant_sr_reduces_to_rne_on_grid(fmt):
    """With amax = fp8_max the scale is exactly 1, so x on the FP8 grid stays
    on it: the stochastic quantizer then equals the RNE one byte for byte, for
    any seed; its amax and inv_scale equal the RNE quantizer's for any x."""
    codes = np.arange(256, dtype=np.uint8)
    vals = O.decode(fmt, codes)
    vals = vals[np.isfinite(vals)]
    x = O.encode("bf16", vals)                    # every FP8 value is exact in bf16
    rows, cols = 1, x.size
    fmax = O.fmt_max(fmt)
    q0, qt0, inv0, _ = O.fp8_quant_tensorwise(x, "bf16", rows, cols, fmt, amax=fmax)
    for seed in (1, 99):
        q1, qt1, inv1, _ = O.fp8_quant_tensorwise_sr(x, "bf16", rows, cols, fmt, seed, 3, 0,
                                                     amax=fmax)
        assert np.array_equal(q0, q1) and np.array_equal(qt0, qt1) and inv0 == inv1
    rng = np.random.default_rng(8)
    y = O.encode("bf16", rng.standard_normal(40 * 24).astype(F32))
    a0 = O.fp8_quant_tensorwise(y, "bf16", 40, 24, fmt)
    a1 = O.fp8_quant_tensorwise_sr(y, "bf16", 40, 24, fmt, 5, 2, 1)
    assert a0[2] == a1[2] and a0[3] == a1[3]
    # out_t holds the same bytes transposed (one draw per element)
    assert np.array_equal(a1[1].reshape(24, 40).T.ravel(), a1[0])
    # each byte is the RNE byte or the neighbour on the other side of the
    # scaled value x * s32 (fp32 product, s32 = fp8_max / amax rounded to fp32)
    s32 = np.float32(O.fmt_max(fmt) / np.float64(a0[3]))
    exact = (O.decode("bf16", y) * s32).astype(np.float64)
    d0 = O.decode(fmt, a0[0]).astype(np.float64)
    d1 = O.decode(fmt, a1[0]).astype(np.float64)
    assert np.all((d1 == d0) | (np.sign(d1 - exact) == -np.sign(d0 - exact)))
    assert np.any(d1 != d0)


def test_fp8_random_stream_is_apart_from_bf16_stream():
    """The FP8 draws of element k are the 16-bit half (k%8)%2 (low first) of
    Philox output word (k%8)/2 at counter {k/8, step, tensor | 2^31}; the
    bf16 copy's draws use the same layout at {k/8, step, tensor}, tensor
    below 2^31: no counter of one stream is a counter of the other."""
    seed, step, tensor = 0x0123456789ABCDEF, 9, 4
    bits = O.sr8_bits(seed, step, tensor, 0, 24)
    key = [seed & 0xFFFFFFFF, seed >> 32]

    def halves(w):
        out = []
        for g in range(3):
            for word in O.philox4x32_10([g, 0, step, w], key):
                out += [int(word) & 0xFFFF, int(word) >> 16]
        return np.array(out, np.uint32)
    assert bits.tolist() == halves(tensor | 0x80000000).tolist()
    assert not np.array_equal(bits, halves(tensor))
