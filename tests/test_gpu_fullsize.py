"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (AmpOptimizerStep over the whole parameter set).

* GPT-2-small set (124,356,864 params, bf16 grads, S = 1): every element,
  all 10 steps.
* 1B Llama set (1,235,814,400 params, fp16 grads, dynamic S, inf/-inf/NaN at
  steps 7/27/47): the scaler trace every step, and master/m/v/bf16 on sampled
  elements (each tensor's ends, chunk boundaries, random positions and the
  planted non-finite sites), which the oracle computes one by one - the update
  is element-wise once found_inf is known.
* FP8 sweep (bf16 [4096,4096], [8192,8192], [16384,5120] and an all-zero
  [4096,4096], e4m3fn and e5m2): every byte of both layouts; the same matrices
  with per-row / per-column scales and with 128-wide group scales (bf16, and
  widened to fp32), every byte and every scale.
* 8B Llama-3 set, the bench's own state (flat buffers, FP8 weights), with
  dynamic and with delayed FP8 scaling: 3 steps; two FP8 weights and a norm
  vector in full through the oracle (bf16, amax or amax history, inv_scale,
  row-major and transposed bytes), sampled elements elsewhere.  The same
  state with both copies rounded stochastically: three tensors in full.
"""
import numpy as np
import pytest
import torch

import oracle as O
from parity_helpers import (assert_bf16_close, assert_state_close, bit_identical_fraction,
                            to_device, to_host_bits)
from workloads import (FP8_SWEEP_SHAPES, FP8_SWEEP_ZERO_SHAPE, amp_config, device_fill_normal,
                       device_generator, fp8_sweep_host, host_grads, host_master, injection_site,
                       tensor_sigmas)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    from loss_scaling_master_gb300 import build as B
    B.build()
    import loss_scaling_master_gb300 as pkg
    pkg.load()
    assert torch.cuda.is_available()
    return pkg


def _step_obj(A, cfg, master_dev, grads_dev, fp8_shapes=None):
    return A.AmpOptimizerStep(master_dev, grads_dev, lr=cfg.lr, beta1=cfg.beta1, beta2=cfg.beta2,
                              eps=cfg.eps, weight_decay=cfg.weight_decay,
                              init_scale=cfg.init_scale, growth_factor=cfg.growth_factor,
                              backoff_factor=cfg.backoff_factor,
                              growth_interval=cfg.growth_interval, fp8_shapes=fp8_shapes)


def _oracle(cfg, master_host, fp8_shapes=None):
    return O.AmpStepOracle(master_host, cfg.grad_dtype, cfg.lr, cfg.beta1, cfg.beta2, cfg.eps,
                           cfg.weight_decay, cfg.init_scale, cfg.growth_factor,
                           cfg.backoff_factor, cfg.growth_interval, fp8_shapes=fp8_shapes)


def test_gpt2_small_full_parity(A):
    dev = torch.device("cuda:0")
    cfg = amp_config("gpt2_small")
    mh = host_master(cfg)
    st = _step_obj(A, cfg, [torch.from_numpy(m).to(dev) for m in mh],
                   [torch.empty(s.numel, dtype=torch.bfloat16, device=dev) for s in cfg.specs])
    orc = _oracle(cfg, mh)
    for k in range(1, cfg.steps + 1):
        gh = host_grads(cfg, k, orc.scale)
        for t, h in zip(st.grads, gh):
            t.copy_(to_device(h, "bf16", dev))
        st.step()
        orc.run(gh)
        s = st.state()
        assert (s["scale"], s["growth_tracker"], s["step"]) == (orc.scale, orc.tracker, orc.step)
    ident = []
    for i in range(len(cfg.specs)):
        for got, ref, nm in ((st.master[i], orc.master[i], "master"),
                             (st.exp_avg[i], orc.exp_avg[i], "exp_avg"),
                             (st.exp_avg_sq[i], orc.exp_avg_sq[i], "exp_avg_sq")):
            g = to_host_bits(got)
            assert_state_close(g, ref, f"{nm}[{cfg.specs[i].name}]")
            ident.append(bit_identical_fraction(g, ref))
        assert_bf16_close(to_host_bits(st.bf16[i]), orc.bf16[i], f"bf16[{cfg.specs[i].name}]")
    assert min(ident) == 1.0
    st.check()                      # no bounded wait gave up
    st.close()


def _sample_indices(n, rng, k=48):
    idx = {0, n - 1, n // 2}
    for b in range(16384, n, 16384 * 97):
        idx.update((b - 1, b))
    idx.update(rng.integers(0, n, size=min(k, n)).tolist())
    return np.array(sorted(i for i in idx if 0 <= i < n), np.int64)


def test_llama_1b_sampled_parity(A):
    dev = torch.device("cuda:0")
    cfg = amp_config("llama_1b")
    sig = tensor_sigmas(cfg, 0)
    gen = device_generator(dev, 0, 3)
    master = [device_fill_normal(torch.empty(s.numel, device=dev), cfg.master_sigma, gen)
              for s in cfg.specs]
    grads = [torch.empty(s.numel, dtype=torch.float16, device=dev) for s in cfg.specs]
    rng = np.random.default_rng(77)
    sites = {k: injection_site(cfg, k, 0) for k in cfg.inject}
    samples = []
    for i, s in enumerate(cfg.specs):
        ix = set(_sample_indices(s.numel, rng).tolist())
        ix.update(e for (t, e, _) in sites.values() if t == i)
        samples.append(torch.tensor(sorted(ix), dtype=torch.int64, device=dev))
    take = lambda ts: [to_host_bits(t.index_select(0, ix)) for t, ix in zip(ts, samples)]
    orc = _oracle(cfg, take(master))
    st = _step_obj(A, cfg, master, grads)
    gen_g = device_generator(dev, 0, 4)
    for k in range(1, cfg.steps + 1):
        for i, g in enumerate(grads):
            device_fill_normal(g, float(sig[i] * orc.scale), gen_g)
        if k in sites:
            t, e, val = sites[k]
            grads[t][e] = val
        gh = take(grads)
        st.step()
        fi = orc.run(gh)
        assert fi == int(k in sites)
        s = st.state()
        assert (s["scale"], s["growth_tracker"], s["step"]) == (orc.scale, orc.tracker, orc.step), k
    assert orc.step == cfg.steps - len(sites)
    for nm, got, ref in (("master", st.master, orc.master), ("exp_avg", st.exp_avg, orc.exp_avg),
                         ("exp_avg_sq", st.exp_avg_sq, orc.exp_avg_sq)):
        for i, g in enumerate(take(got)):
            assert_state_close(g, ref[i], f"{nm}[{cfg.specs[i].name}]")
            assert bit_identical_fraction(g, ref[i]) == 1.0
    for i, b in enumerate(take(st.bf16)):
        assert_bf16_close(b, orc.bf16[i], f"bf16[{cfg.specs[i].name}]")
    st.check()                      # no bounded wait gave up
    st.close()


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
def test_fp8_sweep_full_parity(A, fmt):
    dev = torch.device("cuda:0")
    shapes = FP8_SWEEP_SHAPES + [FP8_SWEEP_ZERO_SHAPE]
    for j, (r, c) in enumerate(shapes):
        xh = fp8_sweep_host(r, c, seed=0, zero=(j == len(FP8_SWEEP_SHAPES)))
        x = to_device(xh, "bf16", dev).view(r, c)
        out = torch.empty((r, c), dtype=torch.uint8, device=dev)
        out_t = torch.empty((c, r), dtype=torch.uint8, device=dev)
        inv = torch.zeros(1, device=dev)
        amax = torch.zeros(1, device=dev)
        A.fp8_quant_tensorwise(x, fmt, out, out_t, inv, amax)
        rq, rqt, rinv, ramax = O.fp8_quant_tensorwise(xh, "bf16", r, c, fmt)
        assert to_host_bits(amax)[0] == np.float32(ramax)
        assert to_host_bits(inv)[0] == np.float32(rinv)
        assert np.array_equal(to_host_bits(out).ravel(), rq), (r, c)
        assert np.array_equal(to_host_bits(out_t).ravel(), rqt), (r, c)
        del x, out, out_t


@pytest.mark.parametrize("fp8_scaling", ["dynamic", "delayed"])
def test_llama3_8b_bench_state_parity(A, fp8_scaling):
    import bench
    dev = torch.device("cuda:0")
    torch.cuda.empty_cache()
    st, info = bench.build_step("llama3_8b", dev, seed=1234, fp8_scaling=fp8_scaling)
    cfg = info["cfg"]
    names = [s.name for s in cfg.specs]
    full = [names.index(n) for n in ("l0.k", "l31.gate", "l5.ffn_norm")]
    rng = np.random.default_rng(88)
    samples = {i: torch.tensor(_sample_indices(s.numel, rng), dtype=torch.int64, device=dev)
               for i, s in enumerate(cfg.specs) if i not in full}
    order = full + sorted(samples)
    init = [to_host_bits(st.master[i]) if i in full
            else to_host_bits(st.master[i].index_select(0, samples[i])) for i in order]
    gh = [to_host_bits(st.grads[i]) if i in full
          else to_host_bits(st.grads[i].index_select(0, samples[i])) for i in order]
    fp8_shapes = [(cfg.specs[i].rows, cfg.specs[i].cols) if (i in full and cfg.specs[i].fp8)
                  else None for i in order]
    orc = O.AmpStepOracle(init, cfg.grad_dtype, cfg.lr, cfg.beta1, cfg.beta2, cfg.eps,
                          cfg.weight_decay, cfg.init_scale, cfg.growth_factor, cfg.backoff_factor,
                          cfg.growth_interval, fp8_shapes=fp8_shapes, fp8_scaling=fp8_scaling)
    for k in range(3):
        st.step()
        assert orc.run(gh) == 0
        s = st.state()
        assert (s["scale"], s["growth_tracker"], s["step"]) == (orc.scale, orc.tracker, orc.step)
    fp8_index = {}
    j = 0
    for i, s in enumerate(cfg.specs):
        if s.fp8:
            fp8_index[i] = j
            j += 1
    for pos, i in enumerate(order):
        sel = (lambda t: to_host_bits(t)) if i in full else \
            (lambda t, ix=samples[i]: to_host_bits(t.index_select(0, ix)))
        for nm, got, ref in (("master", st.master[i], orc.master[pos]),
                             ("exp_avg", st.exp_avg[i], orc.exp_avg[pos]),
                             ("exp_avg_sq", st.exp_avg_sq[i], orc.exp_avg_sq[pos])):
            g = sel(got)
            assert_state_close(g, ref, f"{nm}[{names[i]}]")
            assert bit_identical_fraction(g, ref) == 1.0
        assert_bf16_close(sel(st.bf16[i]), orc.bf16[pos], f"bf16[{names[i]}]")
        if fp8_shapes[pos] is not None:
            q = st.fp8[fp8_index[i]].view(torch.uint8)
            qt = st.fp8_t[fp8_index[i]].view(torch.uint8)
            assert np.array_equal(to_host_bits(q).ravel(), orc.fp8[pos]), names[i]
            assert np.array_equal(to_host_bits(qt).ravel(), orc.fp8_t[pos]), names[i]
            assert to_host_bits(st.inv_scale)[fp8_index[i]] == orc.inv_scale[orc.slots[pos]]
            if fp8_scaling == "delayed":
                assert np.array_equal(to_host_bits(st.amax_history)[fp8_index[i]],
                                      orc.hist[orc.slots[pos]])
    st.check()                      # no bounded wait gave up
    st.close()
    del st, info
    torch.cuda.empty_cache()


@pytest.mark.parametrize("fp8_scaling", ["dynamic", "delayed"])
def test_llama3_8b_bench_state_stochastic_parity(A, fp8_scaling):
    """The bench's 8B state with both copies rounded stochastically (its
    --sr-seed line), 3 steps.  Two FP8 weights and a norm vector go whole
    through the oracle, whose random counters take the tensor words the whole
    set's lists give them: the bf16 copy the list position (delayed step: the
    plain-list position, or FP8 index | 2^30), the FP8 copy the FP8 index.
    master, m, v, bf16, both FP8 layouts and inv_scale equal the oracle's bit
    for bit."""
    import bench
    dev = torch.device("cuda:0")
    torch.cuda.empty_cache()
    seed = 0x5EED0F5EED
    st, info = bench.build_step("llama3_8b", dev, seed=1234, fp8_scaling=fp8_scaling,
                                sr_seed=seed)
    cfg = info["cfg"]
    names = [s.name for s in cfg.specs]
    full = [names.index(n) for n in ("l0.k", "l0.v", "l5.ffn_norm")]
    plain = [i for i, s in enumerate(cfg.specs) if not s.fp8]
    fp8 = [i for i, s in enumerate(cfg.specs) if s.fp8]
    if fp8_scaling == "delayed":
        ids = [fp8.index(i) | (1 << 30) if cfg.specs[i].fp8 else plain.index(i) for i in full]
    else:
        ids = list(full)
    fp8_shapes = [(cfg.specs[i].rows, cfg.specs[i].cols) if cfg.specs[i].fp8 else None
                  for i in full]
    orc = O.AmpStepOracle([to_host_bits(st.master[i]) for i in full], cfg.grad_dtype, cfg.lr,
                          cfg.beta1, cfg.beta2, cfg.eps, cfg.weight_decay, cfg.init_scale,
                          cfg.growth_factor, cfg.backoff_factor, cfg.growth_interval,
                          fp8_shapes=fp8_shapes, fp8_scaling=fp8_scaling, sr_seed=seed,
                          sr_tensor_ids=ids,
                          sr_fp8_ids=[fp8.index(i) for i in full if cfg.specs[i].fp8])
    gh = [to_host_bits(st.grads[i]) for i in full]
    for _ in range(3):
        st.step()
        assert orc.run(gh) == 0
        s = st.state()
        assert (s["scale"], s["growth_tracker"], s["step"]) == (orc.scale, orc.tracker, orc.step)
    for pos, i in enumerate(full):
        for got, ref in ((st.master[i], orc.master[pos]), (st.exp_avg[i], orc.exp_avg[pos]),
                         (st.exp_avg_sq[i], orc.exp_avg_sq[pos])):
            assert np.array_equal(to_host_bits(got).view(np.uint32), ref.view(np.uint32)), names[i]
        assert np.array_equal(to_host_bits(st.bf16[i]), orc.bf16[pos]), names[i]
        if cfg.specs[i].fp8:
            j = fp8.index(i)
            assert np.array_equal(to_host_bits(st.fp8[j].view(torch.uint8)).ravel(),
                                  orc.fp8[pos]), names[i]
            assert np.array_equal(to_host_bits(st.fp8_t[j].view(torch.uint8)).ravel(),
                                  orc.fp8_t[pos]), names[i]
            assert to_host_bits(st.inv_scale)[j] == orc.inv_scale[orc.slots[pos]]
    st.check()
    st.close()
    del st, info
    torch.cuda.empty_cache()


def test_fp8_sweep_rowwise_full_parity(A):
    """The sweep matrices with per-row / per-column scales, every byte and scale."""
    dev = torch.device("cuda:0")
    for j, (r, c) in enumerate(FP8_SWEEP_SHAPES + [FP8_SWEEP_ZERO_SHAPE]):
        xh = fp8_sweep_host(r, c, seed=0, zero=(j == len(FP8_SWEEP_SHAPES)))
        x = to_device(xh, "bf16", dev).view(r, c)
        o = {"q": torch.empty(r * c, dtype=torch.uint8, device=dev),
             "q_t": torch.empty(r * c, dtype=torch.uint8, device=dev)}
        o.update({k: torch.empty(r, device=dev) for k in ("amax_row", "scale_row", "inv_row")})
        o.update({k: torch.empty(c, device=dev) for k in ("amax_col", "scale_col", "inv_col")})
        A.fp8_quant_rowwise(x, "e4m3fn", o["q"], o["q_t"], o["amax_row"], o["scale_row"],
                            o["inv_row"], o["amax_col"], o["scale_col"], o["inv_col"])
        ref = O.fp8_quant_rowwise(xh, "bf16", r, c, "e4m3fn")
        for k in ref:
            g = to_host_bits(o[k])
            assert np.array_equal(g.view(np.uint8) if g.dtype == np.uint8 else g.view(np.uint32),
                                  ref[k] if ref[k].dtype == np.uint8 else ref[k].view(np.uint32)), (k, r, c)
        del x, o


@pytest.mark.parametrize("xdt", ["bf16", "f32"])
@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
def test_fp8_sweep_groupwise_full_parity(A, fmt, xdt):
    """The sweep matrices with g128 group scales (the bench's group size),
    every byte and scale, both directions; as bf16 (tiles held in registers)
    and widened exactly to fp32 (tiles staged in shared memory)."""
    dev = torch.device("cuda:0")
    G = 128
    for j, (r, c) in enumerate(FP8_SWEEP_SHAPES + [FP8_SWEEP_ZERO_SHAPE]):
        xh = fp8_sweep_host(r, c, seed=0, zero=(j == len(FP8_SWEEP_SHAPES)))
        if xdt == "f32":
            xh = (xh.astype(np.uint32) << 16).view(np.float32)
        x = to_device(xh, xdt, dev).view(r, c)
        ngc, ngr = -(-c // G), -(-r // G)
        o = {"q": torch.empty(r * c, dtype=torch.uint8, device=dev),
             "q_t": torch.empty(r * c, dtype=torch.uint8, device=dev)}
        o.update({k: torch.empty(r * ngc, device=dev) for k in ("amax_rg", "scale_rg", "inv_rg")})
        o.update({k: torch.empty(c * ngr, device=dev) for k in ("amax_cg", "scale_cg", "inv_cg")})
        A.fp8_quant_groupwise(x, fmt, G, o["q"], o["q_t"], o["amax_rg"], o["scale_rg"],
                              o["inv_rg"], o["amax_cg"], o["scale_cg"], o["inv_cg"])
        ref = O.fp8_quant_groupwise(xh, xdt, r, c, fmt, G)
        for k in ref:
            g = to_host_bits(o[k])
            assert np.array_equal(g.view(np.uint8) if g.dtype == np.uint8 else g.view(np.uint32),
                                  ref[k] if ref[k].dtype == np.uint8 else ref[k].view(np.uint32)), (k, r, c)
        del x, o


def test_over_2g_element_tensors(A):
    """Largest sizes: one tensor of 2^31 + 12,345 elements through AdamW, and a
    [2^16 + 128, 2^15 + 64] matrix (over 2^31 elements) through the FP8 cast
    with its transposed copy - byte offsets past 2^31 and 2^32.  Checked at
    sampled elements around and beyond the 32-bit boundaries."""
    dev = torch.device("cuda:0")
    torch.cuda.empty_cache()
    n = (1 << 31) + 12345
    gen = device_generator(dev, 5, 9)
    p = device_fill_normal(torch.empty(n, device=dev), 0.02, gen)
    g = device_fill_normal(torch.empty(n, dtype=torch.float16, device=dev), 10.0, gen)
    m = torch.zeros(n, device=dev)
    v = torch.zeros(n, device=dev)
    b = torch.empty(n, dtype=torch.bfloat16, device=dev)
    idx = torch.tensor([0, 1, (1 << 31) - 1, 1 << 31, (1 << 31) + 1, n - 8, n - 1] +
                       torch.randint(0, n, (64,), generator=torch.Generator().manual_seed(3)).tolist(),
                       dtype=torch.int64, device=dev)
    p0, g0 = to_host_bits(p[idx]), to_host_bits(g[idx])
    Ls = [A.amp_tensor_list_create([t]) for t in (p, m, v, g, b)]
    step = torch.zeros(1, dtype=torch.int32, device=dev)
    A.amp_adamw_master_step(*Ls, torch.tensor([1024.0], device=dev), None, step,
                            1e-3, 0.9, 0.999, 1e-8, 0.01)
    rp, rm, rv, rb = [p0.copy()], [np.zeros(idx.numel(), np.float32)], [np.zeros(idx.numel(), np.float32)], \
        [np.zeros(idx.numel(), np.uint16)]
    O.adamw_master_step(rp, rm, rv, [g0], "f16", rb, 1024.0, 0, 0, 1e-3, 0.9, 0.999, 1e-8, 0.01)
    assert np.array_equal(to_host_bits(p[idx]).view(np.uint32), rp[0].view(np.uint32))
    assert np.array_equal(to_host_bits(v[idx]).view(np.uint32), rv[0].view(np.uint32))
    assert np.array_equal(to_host_bits(b[idx]), rb[0])
    for L in Ls:
        L.close()
    del p, g, m, v, b, Ls
    torch.cuda.empty_cache()

    rows, cols = (1 << 16) + 128, (1 << 15) + 64
    x = device_fill_normal(torch.empty((rows, cols), dtype=torch.bfloat16, device=dev), 1.0, gen)
    q = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
    qt = torch.empty((cols, rows), dtype=torch.uint8, device=dev)
    inv = torch.zeros(1, device=dev)
    amax = torch.zeros(1, device=dev)
    A.fp8_quant_tensorwise(x, "e4m3fn", q, qt, inv, amax)
    am = float(to_host_bits(amax)[0])
    assert am == float(x.abs().max().float().item())
    rsel = torch.tensor([0, 1, rows // 2, rows - 2, rows - 1], device=dev)
    csel = torch.tensor([0, 7, cols // 2, cols - 65, cols - 1], device=dev)
    xs = x[rsel][:, csel].contiguous()
    rq, _, rinv, _ = O.fp8_quant_tensorwise(to_host_bits(xs).ravel(), "bf16", 5, 5, "e4m3fn",
                                            transposed=False, amax=am)
    assert np.array_equal(to_host_bits(q[rsel][:, csel]).ravel(), rq)
    assert np.array_equal(to_host_bits(qt[csel][:, rsel]).T.ravel(), rq)
    assert to_host_bits(inv)[0] == np.float32(rinv)
