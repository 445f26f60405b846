"""CPU oracle for the mixed-precision optimizer step - TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and
this package imports nothing from the product: the two sides share only the
seeded input generators in ``workloads/``.

The arithmetic lives in ``oracle.c`` (plain C, single-threaded, its own
number-format converters); this module only marshals numpy arrays into it.
16-bit and 8-bit floating-point buffers travel as raw bit patterns
(``uint16`` / ``uint8`` arrays); fp32 buffers as ``float32``.

Dtype names: ``"f32"``, ``"f16"``, ``"bf16"``, ``"e4m3fn"``, ``"e5m2"``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_CODES = {"f32": 0, "f16": 1, "bf16": 2, "e4m3fn": 3, "e5m2": 4}
_lock = threading.Lock()
_lib = None

P = ctypes.c_void_p
I64P = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, no CUDA)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC",
                               "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.orc_fmt_max.restype = ctypes.c_double
            L.orc_fmt_max.argtypes = [ctypes.c_int]
            L.orc_decode.argtypes = [ctypes.c_int, P, P, ctypes.c_int64]
            L.orc_encode.argtypes = [ctypes.c_int, P, P, ctypes.c_int64]
            L.orc_unscale_check.argtypes = [ctypes.c_int, P, I64P, ctypes.c_int,
                                            ctypes.c_float, P, ctypes.c_int]
            L.orc_update_scale.argtypes = [P, P, P, ctypes.c_float, ctypes.c_float,
                                           ctypes.c_int32, P, ctypes.c_int]
            L.orc_adamw_master_step.argtypes = (
                [ctypes.c_int, P, P, P, P, ctypes.c_int, P, I64P, P, ctypes.c_int32, P]
                + [ctypes.c_double] * 5 + [P, P])
            L.orc_grad_sumsq.restype = ctypes.c_double
            L.orc_grad_sumsq.argtypes = [ctypes.c_int, P, I64P, ctypes.c_int, ctypes.c_float]
            L.orc_clip_coef.restype = ctypes.c_float
            L.orc_clip_coef.argtypes = [ctypes.c_double, ctypes.c_double]
            L.orc_adamw_master_step_clip.argtypes = (
                [ctypes.c_int, P, P, P, P, ctypes.c_int, P, I64P, P, ctypes.c_int32, P]
                + [ctypes.c_double] * 5 + [P, P, ctypes.c_float])
            L.orc_adamw_master_step_ex.argtypes = (
                [ctypes.c_int, P, P, P, P, ctypes.c_int, P, I64P, P, ctypes.c_int32, P]
                + [ctypes.c_double] * 5 + [P, P, ctypes.c_float, ctypes.c_int, ctypes.c_uint64])
            L.orc_philox4x32_10.argtypes = [P, P, P]
            L.orc_bf16_stochastic.restype = ctypes.c_uint16
            L.orc_bf16_stochastic.argtypes = [ctypes.c_float, ctypes.c_uint32]
            L.orc_bf16_stochastic_list.argtypes = [P, P, ctypes.c_int64, ctypes.c_uint64,
                                                   ctypes.c_int32, ctypes.c_int32]
            L.orc_fp8_quant_rowwise.argtypes = [P, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                                ctypes.c_int, ctypes.c_double] + [P] * 8
            L.orc_fp8_quant_groupwise.argtypes = [P, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                                  ctypes.c_int64, ctypes.c_int, ctypes.c_double] + [P] * 8
            L.orc_fp8_quant_tensorwise.argtypes = [P, ctypes.c_int, ctypes.c_int64,
                                                   ctypes.c_int64, ctypes.c_int,
                                                   ctypes.c_double, P, P, P, P, ctypes.c_int]
            L.orc_fp8_quant_tensorwise_sr.argtypes = [P, ctypes.c_int, ctypes.c_int64,
                                                      ctypes.c_int64, ctypes.c_int,
                                                      ctypes.c_double, P, P, P, P, ctypes.c_int,
                                                      ctypes.c_uint64, ctypes.c_int32,
                                                      ctypes.c_int32]
            L.orc_fp8_stochastic.restype = ctypes.c_uint8
            L.orc_fp8_stochastic.argtypes = [ctypes.c_int, ctypes.c_float, ctypes.c_uint32]
            L.orc_fp8_stochastic_list.argtypes = [ctypes.c_int, P, P, P, ctypes.c_int64]
            L.orc_sr8_bits_list.argtypes = [ctypes.c_uint64, ctypes.c_int32, ctypes.c_int32,
                                            ctypes.c_int64, ctypes.c_int64, P]
            L.orc_adamw_master_step_ids.argtypes = (
                [ctypes.c_int, P, P, P, P, ctypes.c_int, P, I64P, P, ctypes.c_int32, P]
                + [ctypes.c_double] * 5 + [P, P, ctypes.c_float, ctypes.c_int, ctypes.c_uint64,
                                           P])
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle buffers must be C-contiguous"
    return a.ctypes.data_as(P)


def _ptr_array(arrs):
    return (P * max(1, len(arrs)))(*[(_ptr(a) if a is not None else None) for a in arrs])


def _numels(arrs):
    return (ctypes.c_int64 * max(1, len(arrs)))(*[a.size for a in arrs])


def _bits_dtype(dt: str):
    return {"f32": np.float32, "f16": np.uint16, "bf16": np.uint16,
            "e4m3fn": np.uint8, "e5m2": np.uint8}[dt]


# ---------------------------------------------------------------- converters
def fmt_max(dt: str) -> float:
    """Largest finite magnitude of a format, from its bit-layout definition."""
    return lib().orc_fmt_max(_CODES[dt])


def decode(dt: str, bits: np.ndarray) -> np.ndarray:
    """Raw bit patterns of format ``dt`` -> float32 values."""
    bits = np.ascontiguousarray(bits, dtype=_bits_dtype(dt))
    out = np.empty(bits.shape, np.float32)
    lib().orc_decode(_CODES[dt], _ptr(bits), _ptr(out), bits.size)
    return out


def encode(dt: str, x: np.ndarray) -> np.ndarray:
    """float32 values -> round-to-nearest-even bit patterns of format ``dt``
    (overflow: infinity, or NaN for e4m3fn; NaN: positive canonical NaN)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, _bits_dtype(dt))
    lib().orc_encode(_CODES[dt], _ptr(x), _ptr(out), x.size)
    return out


# ------------------------------------------------------------------ the step
def unscale_check(grads, dt: str, scale: float, found_inf: int = 0, inplace: bool = False) -> int:
    """OR of !isfinite(g * (1/S)) over every element of every tensor."""
    fi = np.array([found_inf], np.int32)
    lib().orc_unscale_check(len(grads), _ptr_array(grads), _numels(grads), _CODES[dt],
                            ctypes.c_float(scale), _ptr(fi), int(inplace))
    return int(fi[0])


def update_scale(scale: float, tracker: int, found_inf: int, growth: float, backoff: float,
                 interval: int, amax: np.ndarray | None = None):
    """One pass of the dynamic scale state machine. Returns (scale, tracker, found_inf)
    and zeroes ``amax`` in place when given."""
    s = np.array([scale], np.float32)
    t = np.array([tracker], np.int32)
    f = np.array([found_inf], np.int32)
    n = 0 if amax is None else amax.size
    lib().orc_update_scale(_ptr(s), _ptr(t), _ptr(f), ctypes.c_float(growth),
                           ctypes.c_float(backoff), int(interval),
                           _ptr(amax) if n else None, n)
    return float(s[0]), int(t[0]), int(f[0])


def grad_sumsq(grads, dt: str, scale: float) -> float:
    """fp64 sum over all elements of (g * (1/S))^2, in element order."""
    return float(lib().orc_grad_sumsq(len(grads), _ptr_array(grads), _numels(grads), _CODES[dt],
                                      ctypes.c_float(scale)))


def clip_coef(sumsq: float, max_norm: float) -> float:
    """fp32 min(1, max_norm / (sqrt(sumsq) + 1e-6))."""
    return float(lib().orc_clip_coef(sumsq, max_norm))


def adamw_master_step(master, exp_avg, exp_avg_sq, grads, gdt: str, bf16_out, scale,
                      found_inf: int, step: int, lr, beta1, beta2, eps, wd,
                      amax_slot=None, amax: np.ndarray | None = None,
                      clip: float | None = None, sr_seed: int | None = None,
                      sr_ids=None) -> int:
    """FP32-master AdamW over a tensor list (in place); returns the new step count.
    ``scale`` None means S = 1. ``bf16_out`` is a list of uint16 arrays or None.
    ``clip`` is the fp32 gradient clipping factor (None: no clipping).
    ``sr_seed``: round the bf16 copy stochastically; ``sr_ids`` the tensor
    word of each tensor's random counter (None: its list index)."""
    n = len(master)
    sc = None if scale is None else np.array([scale], np.float32)
    st = np.array([step], np.int32)
    slots = None if amax_slot is None else np.ascontiguousarray(amax_slot, np.int32)
    args = [n, _ptr_array(master), _ptr_array(exp_avg), _ptr_array(exp_avg_sq),
            _ptr_array(grads), _CODES[gdt], _ptr_array(bf16_out) if bf16_out else None,
            _numels(master), _ptr(sc) if sc is not None else None, int(found_inf), _ptr(st),
            lr, beta1, beta2, eps, wd,
            _ptr(slots) if slots is not None else None,
            _ptr(amax) if amax is not None else None]
    if sr_seed is not None:
        ids = None if sr_ids is None else np.ascontiguousarray(sr_ids, np.int32)
        lib().orc_adamw_master_step_ids(*args, ctypes.c_float(1.0 if clip is None else clip), 1,
                                        ctypes.c_uint64(sr_seed),
                                        _ptr(ids) if ids is not None else None)
    elif clip is None:
        lib().orc_adamw_master_step(*args)
    else:
        lib().orc_adamw_master_step_clip(*args, ctypes.c_float(clip))
    return int(st[0])


def philox4x32_10(ctr, key):
    c = np.ascontiguousarray(ctr, np.uint32)
    k = np.ascontiguousarray(key, np.uint32)
    o = np.zeros(4, np.uint32)
    lib().orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(o))
    return o


def bf16_stochastic(p: np.ndarray, seed: int, step: int, tensor: int) -> np.ndarray:
    """Stochastically rounded bf16 bits of fp32 p, random bits from the counter
    {element group, step, tensor} and key seed."""
    p = np.ascontiguousarray(p, np.float32)
    out = np.empty(p.size, np.uint16)
    lib().orc_bf16_stochastic_list(_ptr(p), _ptr(out), p.size, seed, step, tensor)
    return out


def fp8_quant_tensorwise(x: np.ndarray, xdt: str, rows: int, cols: int, fp8: str,
                         eps: float = 1e-12, transposed: bool = True, amax: float | None = None):
    """Returns (q [rows*cols] uint8, q_t [cols*rows] uint8 or None, inv_scale, amax)."""
    x = np.ascontiguousarray(x)
    assert x.size == rows * cols
    out = np.empty(rows * cols, np.uint8)
    out_t = np.empty(rows * cols, np.uint8) if transposed else None
    inv = np.zeros(1, np.float32)
    am = np.array([0.0 if amax is None else amax], np.float32)
    lib().orc_fp8_quant_tensorwise(_ptr(x), _CODES[xdt], rows, cols, _CODES[fp8], eps,
                                   _ptr(out), _ptr(out_t) if out_t is not None else None,
                                   _ptr(inv), _ptr(am), int(amax is not None))
    return out, out_t, float(inv[0]), float(am[0])


def fp8_stochastic(fp8: str, y: np.ndarray, u: np.ndarray) -> np.ndarray:
    """Stochastic rounding of fp32 values y (already scaled) to FP8 bytes with
    16 random bits each (hi exactly when u < floor(2^16 * distance ratio))."""
    y = np.ascontiguousarray(y, np.float32)
    u = np.ascontiguousarray(u, np.uint32)
    assert y.shape == u.shape
    out = np.empty(y.shape, np.uint8)
    lib().orc_fp8_stochastic_list(_CODES[fp8], _ptr(y), _ptr(u), _ptr(out), y.size)
    return out


def sr8_bits(seed: int, step: int, tensor: int, k0: int, n: int) -> np.ndarray:
    """The 16 random bits of elements k0 .. k0+n-1 of FP8 tensor `tensor` at `step`."""
    out = np.empty(n, np.uint32)
    lib().orc_sr8_bits_list(ctypes.c_uint64(seed), step, tensor, k0, n, _ptr(out))
    return out


def fp8_quant_tensorwise_sr(x: np.ndarray, xdt: str, rows: int, cols: int, fp8: str,
                            seed: int, step: int, tensor: int, eps: float = 1e-12,
                            transposed: bool = True, amax: float | None = None):
    """fp8_quant_tensorwise with the stochastic cast (same amax / inv_scale).
    Returns (q, q_t or None, inv_scale, amax)."""
    x = np.ascontiguousarray(x)
    assert x.size == rows * cols
    out = np.empty(rows * cols, np.uint8)
    out_t = np.empty(rows * cols, np.uint8) if transposed else None
    inv = np.zeros(1, np.float32)
    am = np.array([0.0 if amax is None else amax], np.float32)
    lib().orc_fp8_quant_tensorwise_sr(_ptr(x), _CODES[xdt], rows, cols, _CODES[fp8], eps,
                                      _ptr(out), _ptr(out_t) if out_t is not None else None,
                                      _ptr(inv), _ptr(am), int(amax is not None),
                                      ctypes.c_uint64(seed), step, tensor)
    return out, out_t, float(inv[0]), float(am[0])


def fp8_quant_groupwise(x: np.ndarray, xdt: str, rows: int, cols: int, fp8: str, group: int,
                        eps: float = 1e-12, transposed: bool = True):
    """One scale per `group` consecutive elements of a row for the row-major
    bytes, per `group` consecutive rows of a column for the transposed copy.
    Returns a dict of q, amax/scale/inv per row group ([rows, ceil(cols/group)])
    and, transposed, q_t and amax/scale/inv per column group
    ([cols, ceil(rows/group)])."""
    x = np.ascontiguousarray(x)
    assert x.size == rows * cols and group >= 1
    ngc, ngr = -(-cols // group), -(-rows // group)
    r = {"q": np.empty(rows * cols, np.uint8), "amax_rg": np.empty(rows * ngc, np.float32),
         "scale_rg": np.empty(rows * ngc, np.float32), "inv_rg": np.empty(rows * ngc, np.float32)}
    if transposed:
        r.update(q_t=np.empty(rows * cols, np.uint8), amax_cg=np.empty(cols * ngr, np.float32),
                 scale_cg=np.empty(cols * ngr, np.float32), inv_cg=np.empty(cols * ngr, np.float32))
    g = lambda k: _ptr(r[k]) if k in r else None
    lib().orc_fp8_quant_groupwise(_ptr(x), _CODES[xdt], rows, cols, group, _CODES[fp8], eps,
                                  g("q"), g("q_t"), g("amax_rg"), g("scale_rg"), g("inv_rg"),
                                  g("amax_cg"), g("scale_cg"), g("inv_cg"))
    return r


def fp8_quant_rowwise(x: np.ndarray, xdt: str, rows: int, cols: int, fp8: str,
                      eps: float = 1e-12, transposed: bool = True):
    """Per-row scales for the row-major bytes, per-column scales for the
    transposed copy.  Returns a dict of q, q_t, amax/scale/inv per row and col."""
    x = np.ascontiguousarray(x)
    assert x.size == rows * cols
    r = {"q": np.empty(rows * cols, np.uint8),
         "amax_row": np.empty(rows, np.float32), "scale_row": np.empty(rows, np.float32),
         "inv_row": np.empty(rows, np.float32)}
    if transposed:
        r.update(q_t=np.empty(rows * cols, np.uint8), amax_col=np.empty(cols, np.float32),
                 scale_col=np.empty(cols, np.float32), inv_col=np.empty(cols, np.float32))
    g = lambda k: _ptr(r[k]) if k in r else None
    lib().orc_fp8_quant_rowwise(_ptr(x), _CODES[xdt], rows, cols, _CODES[fp8], eps, g("q"),
                                g("q_t"), g("amax_row"), g("scale_row"), g("inv_row"),
                                g("amax_col"), g("scale_col"), g("inv_col"))
    return r


class AmpStepOracle:
    """One optimizer step in the pages' order, composed from the functions above:

    1. unscale + non-finite check of the scaled gradients (found_inf),
    2. skip-or-step: FP32-master AdamW emitting the bf16 working copy,
    3. for FP8 weights, tensorwise e4m3fn quantization of the bf16 copy
       (row-major + transposed) from the amax folded in step 2,
    4. the scale state machine, which also clears found_inf and amax.
    """

    def __init__(self, master, grad_dtype, lr, beta1, beta2, eps, weight_decay,
                 init_scale, growth_factor, backoff_factor, growth_interval,
                 emit_bf16=True, fp8_shapes=None, fp8_eps=1e-12, max_norm=None,
                 fp8_scaling="dynamic", hist_len=1, fp8_format="e4m3fn", sr_seed=None,
                 sr_tensor_ids=None, sr_fp8_ids=None):
        self.master = [np.array(m, np.float32, copy=True) for m in master]
        self.exp_avg = [np.zeros_like(m) for m in self.master]
        self.exp_avg_sq = [np.zeros_like(m) for m in self.master]
        self.bf16 = [np.zeros(m.size, np.uint16) for m in self.master] if emit_bf16 else None
        self.gdt = grad_dtype
        self.hyper = (lr, beta1, beta2, eps, weight_decay)
        self.scale, self.tracker, self.step, self.found_inf = float(init_scale), 0, 0, 0
        self.growth, self.backoff, self.interval = growth_factor, backoff_factor, growth_interval
        # fp8_shapes: per tensor (rows, cols) or None; FP8 slots numbered in order
        self.fp8_shapes = fp8_shapes
        self.slots = None
        self.fp8_eps = fp8_eps
        # format of the FP8 weight copies ("FP8训练：量化、自动微分、Torchao" §3:
        # e4m3fn for weights and activations, e5m2 for gradients; both offered)
        self.fp8_format = fp8_format
        self.max_norm = max_norm
        self.grad_norm = None
        # Stochastic rounding ("第20章 量化与混合精度训练" §20.5.14) of the copies
        # each step emits: the bf16 copy and the FP8 weights cast from it.  The
        # first working copies, made before any step, keep round-to-nearest.
        self.sr_seed = sr_seed
        # Tensor words of the random counters, for tensors that are a subset of
        # a larger set: sr_tensor_ids per tensor for its bf16 copy (default:
        # the list position; in the delayed step the plain-list position p, or
        # j | 2^30 for FP8 weight j), sr_fp8_ids per FP8 slot for its FP8 copy
        # (default: the slot).
        self.sr_tensor_ids = None if sr_tensor_ids is None else list(sr_tensor_ids)
        self.sr_fp8_ids = None if sr_fp8_ids is None else list(sr_fp8_ids)
        if fp8_shapes is not None:
            self.slots, k = [], 0
            for sh in fp8_shapes:
                self.slots.append(k if sh is not None else -1)
                k += sh is not None
            self.amax = np.zeros(max(k, 1), np.float32)
            self.fp8 = [None] * len(master)
            self.fp8_t = [None] * len(master)
            self.inv_scale = np.zeros(max(k, 1), np.float32)
        else:
            self.amax = None
        # The working copies exist before the first step: the model's bf16
        # parameters are the master rounded to bf16 ("从 AMP 到 Mixed
        # Precision", "PyTorch AMP 与 FP32 Master Weights", mode B), and the
        # FP8 weights are cast from that copy with its own amax
        # ("FP8训练：量化、自动微分、Torchao" §2).
        # Delayed scaling ("第20章 量化与混合精度训练" §20.5.9): each FP8 weight
        # keeps the amax of its last hist_len steps (newest first) and is cast
        # with the scale of their maximum.  At construction there is no
        # previous step, so the history starts from the amax of that first
        # bf16 copy.
        self.fp8_scaling = fp8_scaling
        self.hist_len = hist_len
        if fp8_scaling == "delayed":
            assert fp8_shapes is not None and emit_bf16
            self.hist = np.zeros((max(k, 1), hist_len), np.float32)
        if emit_bf16:
            for i in range(len(self.master)):
                self.bf16[i] = encode("bf16", self.master[i])
        if fp8_shapes is not None:
            for i, sh in enumerate(fp8_shapes):
                if sh is None:
                    continue
                q, qt, inv, am = fp8_quant_tensorwise(self.bf16[i], "bf16", sh[0], sh[1],
                                                      self.fp8_format, self.fp8_eps, True)
                s_ = self.slots[i]
                self.fp8[i], self.fp8_t[i], self.inv_scale[s_] = q, qt, inv
                if fp8_scaling == "delayed":
                    self.hist[s_, 0] = am

    def run(self, grads):
        """Apply one step with the given scaled gradients; returns found_inf."""
        fi = unscale_check(grads, self.gdt, self.scale, found_inf=self.found_inf)
        self.found_inf = fi
        clip = None
        if self.max_norm is not None:
            ss = grad_sumsq(grads, self.gdt, self.scale)
            self.grad_norm = float(np.sqrt(ss))
            clip = clip_coef(ss, self.max_norm)
        sr_ids = None
        if self.sr_seed is not None and self.sr_tensor_ids is not None:
            sr_ids = self.sr_tensor_ids
        elif self.sr_seed is not None and self.fp8_scaling == "delayed":
            # the delayed step walks the plain tensors and the FP8 weights as
            # two lists: plain tensor p draws as p, FP8 weight j as j | 2^30
            sr_ids, p_idx = [], 0
            for sh, sl in zip(self.fp8_shapes, self.slots):
                if sh is None:
                    sr_ids.append(p_idx)
                    p_idx += 1
                else:
                    sr_ids.append(sl | (1 << 30))
        self.step = adamw_master_step(self.master, self.exp_avg, self.exp_avg_sq, grads,
                                      self.gdt, self.bf16, self.scale, fi, self.step,
                                      *self.hyper, amax_slot=self.slots, amax=self.amax,
                                      clip=clip, sr_seed=self.sr_seed, sr_ids=sr_ids)
        if self.fp8_shapes is not None and not fi:
            for i, sh in enumerate(self.fp8_shapes):
                if sh is None:
                    continue
                s = self.slots[i]
                if self.fp8_scaling == "delayed":
                    h = self.hist[s]
                    a = float("nan") if np.isnan(h).any() else float(h.max())
                else:
                    a = float(self.amax[s])
                if self.sr_seed is None:
                    q, qt, inv, _ = fp8_quant_tensorwise(self.bf16[i], "bf16", sh[0], sh[1],
                                                         self.fp8_format, self.fp8_eps, True,
                                                         amax=a)
                else:
                    w = s if self.sr_fp8_ids is None else self.sr_fp8_ids[s]
                    q, qt, inv, _ = fp8_quant_tensorwise_sr(self.bf16[i], "bf16", sh[0], sh[1],
                                                            self.fp8_format, self.sr_seed,
                                                            self.step, w, self.fp8_eps, True,
                                                            amax=a)
                self.fp8[i], self.fp8_t[i], self.inv_scale[s] = q, qt, inv
        if self.fp8_scaling == "delayed" and not fi:
            self.hist[:, 1:] = self.hist[:, :-1].copy()
            self.hist[:, 0] = self.amax[:self.hist.shape[0]]
        self.scale, self.tracker, self.found_inf = update_scale(
            self.scale, self.tracker, self.found_inf, self.growth, self.backoff,
            self.interval, self.amax)
        return fi
