"""Seeded synthetic workloads for the mixed-precision optimizer step.

This module is shared by the CPU oracle side and the CUDA side of the tests and
by ``bench.py``.  It holds parameter-set shapes, hyper-parameters and seeded
random inputs only - none of the method's arithmetic (no unscale, no
optimizer, no quantization).  Casting a freshly drawn gradient to its storage
dtype (fp16 / bf16) is part of producing the input, done with numpy / torch
library casts.

Parameter sets (shapes follow the named model families; linear weights are
stored [out_features, in_features] as nn.Linear does):

* ``tiny``        3 fp32 tensors [1000], [4096], [257]
* ``gpt2_small``  124,356,864 params in 100 tensors
* ``llama_1b``    1,235,814,400 params in 146 tensors (tied embedding)
* ``llama3_8b``   8,030,261,248 params in 291 tensors; its 224 linear
                  weights (6,979,321,856 params) also get FP8 copies
* ``fp8_sweep``   bf16 matrices [4096,4096], [8192,8192], [16384,5120] and an
                  all-zero [4096,4096], N(0,1) with 0.1 % outliers x100
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class TensorSpec:
    name: str
    rows: int
    cols: int = 1          # 1 => a 1-D vector of length ``rows``
    fp8: bool = False      # linear weight that also gets an e4m3fn copy

    @property
    def numel(self) -> int:
        return self.rows * self.cols


def tiny_specs():
    return [TensorSpec("t0", 1000), TensorSpec("t1", 4096), TensorSpec("t2", 257)]


def gpt2_small_specs():
    d, v, ctx, L = 768, 50257, 1024, 12
    s = [TensorSpec("wte", v, d), TensorSpec("wpe", ctx, d)]
    for i in range(L):
        p = f"h{i}."
        s += [TensorSpec(p + "ln_1.w", d), TensorSpec(p + "ln_1.b", d),
              TensorSpec(p + "attn.c_attn.w", d, 3 * d), TensorSpec(p + "attn.c_proj.w", d, d),
              TensorSpec(p + "ln_2.w", d), TensorSpec(p + "ln_2.b", d),
              TensorSpec(p + "mlp.c_fc.w", d, 4 * d), TensorSpec(p + "mlp.c_proj.w", 4 * d, d)]
    s += [TensorSpec("ln_f.w", d), TensorSpec("ln_f.b", d)]
    return s


def _llama_specs(hidden, layers, ffn, vocab, kv_width, tied, fp8_linear):
    s = [TensorSpec("embed", vocab, hidden)]
    for i in range(layers):
        p = f"l{i}."
        s += [TensorSpec(p + "attn_norm", hidden),
              TensorSpec(p + "q", hidden, hidden, fp8_linear),
              TensorSpec(p + "k", kv_width, hidden, fp8_linear),
              TensorSpec(p + "v", kv_width, hidden, fp8_linear),
              TensorSpec(p + "o", hidden, hidden, fp8_linear),
              TensorSpec(p + "ffn_norm", hidden),
              TensorSpec(p + "gate", ffn, hidden, fp8_linear),
              TensorSpec(p + "up", ffn, hidden, fp8_linear),
              TensorSpec(p + "down", hidden, ffn, fp8_linear)]
    s += [TensorSpec("final_norm", hidden)]
    if not tied:
        s += [TensorSpec("lm_head", vocab, hidden)]
    return s


def llama_1b_specs():
    # hidden 2048, 16 layers, ffn 8192, vocab 128256; 32 q / 8 kv heads of 64
    return _llama_specs(2048, 16, 8192, 128256, 512, tied=True, fp8_linear=False)


def llama3_8b_specs():
    # hidden 4096, 32 layers, GQA 32 q / 8 kv heads of 128, ffn 14336, vocab 128256
    return _llama_specs(4096, 32, 14336, 128256, 1024, tied=False, fp8_linear=True)


FP8_SWEEP_SHAPES = [(4096, 4096), (8192, 8192), (16384, 5120)]
FP8_SWEEP_ZERO_SHAPE = (4096, 4096)


@dataclass
class AmpConfig:
    name: str
    specs: list
    grad_dtype: str           # "f16" | "bf16" | "f32"
    steps: int
    lr: float
    beta1: float
    beta2: float
    eps: float
    weight_decay: float
    init_scale: float
    growth_factor: float
    backoff_factor: float
    growth_interval: int
    grad_sigma: object        # float, or "loguniform" (per tensor 10**U(-8,-2))
    master_sigma: float = 0.02
    # step (1-based) -> (tensor index or None for seeded, element or None, value)
    inject: dict = field(default_factory=dict)
    fp8_weights: bool = False


def amp_config(name: str) -> AmpConfig:
    if name == "tiny":
        return AmpConfig("tiny", tiny_specs(), "f16", 4, 1e-3, 0.9, 0.999, 1e-8, 0.01,
                         65536.0, 2.0, 0.5, 2, 1e-5, inject={2: (2, 256, np.inf)})
    if name == "gpt2_small":
        return AmpConfig("gpt2_small", gpt2_small_specs(), "bf16", 10, 3e-4, 0.9, 0.95, 1e-8,
                         0.1, 1.0, 1.0, 1.0, 2000, 1e-3)
    if name == "llama_1b":
        return AmpConfig("llama_1b", llama_1b_specs(), "f16", 50, 1e-3, 0.9, 0.999, 1e-8, 0.01,
                         65536.0, 2.0, 0.5, 10, "loguniform",
                         inject={7: (None, None, np.inf), 27: (None, None, -np.inf),
                                 47: (None, None, np.nan)})
    if name == "llama3_8b":
        return AmpConfig("llama3_8b", llama3_8b_specs(), "f16", 20, 1e-3, 0.9, 0.999, 1e-8, 0.01,
                         65536.0, 2.0, 0.5, 2000, 1e-4, fp8_weights=True)
    if name == "llama3_8b_2layers":
        # two decoder layers of the 8B set (no embedding / head): a profiling-size
        # case of the same kernels (436,224,000 params, all linear weights FP8)
        specs = [s for s in llama3_8b_specs() if s.name.startswith(("l0.", "l1."))]
        return AmpConfig("llama3_8b_2layers", specs, "f16", 20, 1e-3, 0.9, 0.999, 1e-8, 0.01,
                         65536.0, 2.0, 0.5, 2000, 1e-4, fp8_weights=True)
    raise KeyError(name)


def tensor_sigmas(cfg: AmpConfig, seed: int = 0) -> np.ndarray:
    """Per-tensor gradient standard deviation (true, unscaled)."""
    n = len(cfg.specs)
    if cfg.grad_sigma == "loguniform":
        rng = np.random.default_rng([seed, 0x5167])
        return 10.0 ** rng.uniform(-8.0, -2.0, size=n)
    return np.full(n, float(cfg.grad_sigma))


def injection_site(cfg: AmpConfig, step: int, seed: int = 0):
    """(tensor, element, value) of the non-finite value planted at ``step``, or None."""
    if step not in cfg.inject:
        return None
    t, e, val = cfg.inject[step]
    rng = np.random.default_rng([seed, 0x1AF, step])
    if t is None:
        t = int(rng.integers(0, len(cfg.specs)))
    if e is None:
        e = int(rng.integers(0, cfg.specs[t].numel))
    return t, e, val


# ------------------------------------------------------------------ numpy (host) side
def host_master(cfg: AmpConfig, seed: int = 0):
    """fp32 master weights ~ N(0, master_sigma), one array per tensor."""
    rng = np.random.default_rng([seed, 0xA57E])
    return [(rng.standard_normal(s.numel) * cfg.master_sigma).astype(np.float32)
            for s in cfg.specs]


def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def host_grads(cfg: AmpConfig, step: int, scale: float, seed: int = 0):
    """Scaled low-precision gradients of one step: dtype(N(0, sigma_t) * S).
    16-bit dtypes are returned as uint16 bit patterns, f32 as float32."""
    rng = np.random.default_rng([seed, 0x6AD, step])
    sig = tensor_sigmas(cfg, seed)
    out = []
    for i, s in enumerate(cfg.specs):
        g = rng.standard_normal(s.numel) * (sig[i] * scale)
        if cfg.grad_dtype == "f16":
            out.append(g.astype(np.float16).view(np.uint16))
        elif cfg.grad_dtype == "bf16":
            out.append(_to_bf16_bits(g.astype(np.float32)))
        else:
            out.append(g.astype(np.float32))
    site = injection_site(cfg, step, seed)
    if site is not None:
        t, e, val = site
        if cfg.grad_dtype == "f16":
            out[t][e] = np.array([val], np.float16).view(np.uint16)[0]
        elif cfg.grad_dtype == "bf16":
            out[t][e] = _to_bf16_bits(np.array([val], np.float32))[0]
        else:
            out[t][e] = np.float32(val)
    return out


def fp8_sweep_host(rows: int, cols: int, seed: int = 0, zero: bool = False,
                   outlier_frac: float = 1e-3, outlier_mult: float = 100.0) -> np.ndarray:
    """bf16 bit patterns of an N(0,1) matrix with a fraction of positions x100."""
    if zero:
        return np.zeros(rows * cols, np.uint16)
    rng = np.random.default_rng([seed, 0xF8, rows, cols])
    x = rng.standard_normal(rows * cols).astype(np.float32)
    k = max(1, int(round(outlier_frac * x.size)))
    idx = rng.choice(x.size, size=k, replace=False)
    x[idx] *= outlier_mult
    return _to_bf16_bits(x)


# ------------------------------------------------------------------ torch (device) side
def device_generator(device, seed: int, salt: int):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1000003 + salt) & 0x7FFFFFFFFFFFFFFF)
    return g


def device_fill_normal(t, sigma: float, gen):
    """In-place N(0, sigma) fill of an fp32 tensor, or of a 16-bit tensor via
    an fp32 draw cast to its dtype (chunked to bound the fp32 temporary)."""
    import torch
    flat = t.view(-1)
    if t.dtype == torch.float32:
        flat.normal_(0.0, sigma, generator=gen)
        return t
    step = 1 << 27
    for s in range(0, flat.numel(), step):
        e = min(flat.numel(), s + step)
        tmp = torch.empty(e - s, dtype=torch.float32, device=t.device)
        tmp.normal_(0.0, sigma, generator=gen)
        flat[s:e].copy_(tmp)
    return t


def device_fill_sweep(x, gen, outlier_frac: float = 1e-3, outlier_mult: float = 100.0):
    """The sweep's matrix on the device: N(0,1) drawn in fp32, a seeded
    fraction of positions (0.1 %, sign kept) multiplied by 100, then rounded
    to x's dtype, as fp8_sweep_host does on the host."""
    import torch
    tmp = torch.empty(x.numel(), dtype=torch.float32, device=x.device)
    tmp.normal_(0.0, 1.0, generator=gen)
    k = max(1, int(round(outlier_frac * tmp.numel())))
    idx = torch.randint(0, tmp.numel(), (k,), generator=gen, device=x.device).unique()
    tmp[idx] *= outlier_mult
    x.view(-1).copy_(tmp)
    return x
