"""ctypes binding of libampfp8.so (declared in include/ampfp8.h).

Argument marshalling only: every function here passes device pointers,
sizes and a stream handle straight to the C entry point of the same name and
raises ``AmpError`` on a non-OK status.  PyTorch supplies device memory and
streams; no computation of the step happens in Python.  There is no fallback:
if the shared library is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libampfp8.so")

AMP_OK = 0
STATUS = {0: "AMP_OK", -1: "AMP_EINVAL", -2: "AMP_EDTYPE", -4: "AMP_ECUDA", -5: "AMP_ENOMEM",
          -6: "AMP_ETIMEOUT"}
DT = {"f32": 1, "f16": 2, "bf16": 3, "e4m3fn": 4, "e5m2": 5}
_TORCH_DT = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16",
             torch.float8_e4m3fn: "e4m3fn", torch.float8_e5m2: "e5m2"}

# every symbol include/ampfp8.h declares
EXPORTS = ("amp_tensor_list_create", "amp_tensor_list_set_amax_slots", "amp_tensor_list_destroy",
           "amp_tensor_list_check", "amp_selftest_bounded_wait",
           "amp_tensor_list_copy_from_host", "amp_tensor_list_copy_to_host",
           "amp_read_state", "amp_scale_health", "fp8_quant_groupwise",
           "amp_unscale_check", "amp_unscale_check_norm", "amp_adamw_master_step", "amp_emit_bf16",
           "amp_adamw_master_step_clip", "amp_adamw_master_step_sr",
           "amp_adamw_master_step_clip_sr", "amp_adamw_master_step_fp8_delayed_sr",
           "fp8_quant_tensorwise_list_sr",
           "amp_adamw_master_step_noalloc", "amp_noalloc_check",
           "amp_adamw_master_step_fp8_delayed", "amp_update_scale_fp8_history",
           "fp8_quant_tensorwise", "fp8_quant_tensorwise_list", "fp8_quant_rowwise",
           "amp_update_scale",
           "amp_last_error", "amp_abi_version")


class AmpError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} -> {STATUS.get(status, status)}: {msg}")
        self.status = status


class amp_adamw_hyper(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double)]


_lock = threading.Lock()
_lib = None
P = ctypes.c_void_p


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libampfp8.so and declare its prototypes (raises if not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(path)
        i32, i64, dbl, flt = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_float
        L.amp_tensor_list_create.argtypes = [i32, P, P, P, i32, P, ctypes.POINTER(P)]
        L.amp_tensor_list_set_amax_slots.argtypes = [P, P, P]
        L.amp_tensor_list_destroy.argtypes = [P]
        L.amp_unscale_check.argtypes = [P, P, P, i32, P]
        L.amp_tensor_list_check.argtypes = [P, P]
        L.amp_tensor_list_copy_from_host.argtypes = [P, P, P]
        L.amp_tensor_list_copy_to_host.argtypes = [P, P, P]
        L.amp_read_state.argtypes = [P, P, P, P, P, P]
        L.amp_scale_health.argtypes = [P, flt, P, P]
        L.fp8_quant_groupwise.argtypes = [P, i32, i64, i64, i64, i32, dbl] + [P] * 10
        L.amp_noalloc_check.argtypes = [P]
        L.amp_selftest_bounded_wait.argtypes = [P, dbl, P]
        L.amp_adamw_master_step.argtypes = [P, P, P, P, P, P, P, P,
                                            ctypes.POINTER(amp_adamw_hyper), P, P]
        L.amp_unscale_check_norm.argtypes = [P, P, P, P, P]
        L.amp_emit_bf16.argtypes = [P, P, P, P]
        L.amp_adamw_master_step_clip.argtypes = [P, P, P, P, P, P, P, P,
                                                 ctypes.POINTER(amp_adamw_hyper), P, P, dbl, P]
        L.amp_adamw_master_step_sr.argtypes = [P, P, P, P, P, P, P, P,
                                               ctypes.POINTER(amp_adamw_hyper), P,
                                               ctypes.c_uint64, P]
        L.amp_adamw_master_step_clip_sr.argtypes = [P, P, P, P, P, P, P, P,
                                                    ctypes.POINTER(amp_adamw_hyper), P, P, dbl,
                                                    ctypes.c_uint64, P]
        L.amp_adamw_master_step_fp8_delayed_sr.argtypes = (
            [P] * 12 + [i32, dbl, P, i32, P, P, P, P, P, ctypes.POINTER(amp_adamw_hyper),
                        ctypes.c_uint64, P])
        L.fp8_quant_tensorwise_list_sr.argtypes = [P, P, P, i32, dbl, P, P, P, ctypes.c_uint64,
                                                   P, P]
        L.amp_adamw_master_step_noalloc.argtypes = [i32, P, P, P, P, i32, P, P, P, P, P, P,
                                                    ctypes.POINTER(amp_adamw_hyper), P, P]
        L.amp_adamw_master_step_fp8_delayed.argtypes = [P] * 12 + [i32, dbl, P, i32, P, P, P, P,
                                                                  P, ctypes.POINTER(amp_adamw_hyper),
                                                                  P]
        L.amp_update_scale_fp8_history.argtypes = [P, P, P, flt, flt, ctypes.c_int32, P, P, i32,
                                                   i32, P]
        L.fp8_quant_tensorwise.argtypes = [P, i32, i64, i64, i32, dbl, P, P, P, P, i32, P, P]
        L.fp8_quant_rowwise.argtypes = [P, i32, i64, i64, i32, dbl] + [P] * 10
        L.fp8_quant_tensorwise_list.argtypes = [P, P, P, i32, dbl, P, P, P, P]
        L.amp_update_scale.argtypes = [P, P, P, flt, flt, ctypes.c_int32, P, i32, P]
        for name in EXPORTS[:-2]:
            getattr(L, name).restype = ctypes.c_int
        L.amp_last_error.restype = ctypes.c_char_p
        L.amp_last_error.argtypes = []
        L.amp_abi_version.restype = ctypes.c_int
        L.amp_abi_version.argtypes = []
        _lib = L
        return L


def _check(fn: str, st: int):
    if st != AMP_OK:
        raise AmpError(fn, st, load().amp_last_error().decode(errors="replace"))


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return P(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _buf(t, what: str, dtype=None, numel: int = 1, itemsize: int | None = None,
         host_ok: bool = False):
    """Pointer of a buffer the library reads or writes, after checking that it
    is a contiguous CUDA tensor (or page-locked host memory where host_ok) of
    the expected dtype (or item size) with at least `numel` elements, so a
    wrong buffer fails here instead of faulting on the device."""
    if t is None:
        return None
    if not t.is_contiguous() or not (t.is_cuda or (host_ok and t.is_pinned())):
        raise ValueError(f"{what}: needs a contiguous "
                         + ("CUDA or page-locked host" if host_ok else "CUDA") + " tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{what}: dtype {t.dtype}, expected {dtype}")
    if itemsize is not None and t.element_size() != itemsize:
        raise ValueError(f"{what}: {t.element_size()}-byte elements, expected {itemsize}")
    if t.numel() < numel:
        raise ValueError(f"{what}: {t.numel()} elements, at least {numel} needed")
    return P(t.data_ptr())


_F32, _F64, _I32 = torch.float32, torch.float64, torch.int32


def _step_bufs(scale, found_inf, step):
    """scale (fp32, may be None for S = 1), found_inf and the step counter (int32)."""
    return (_buf(scale, "scale", _F32), _buf(found_inf, "found_inf", _I32),
            _buf(step, "step", _I32))


def dtype_name(t: torch.Tensor) -> str:
    return _TORCH_DT[t.dtype]


class TensorList:
    """Owner of an ``amp_tensor_list`` handle; keeps its tensors alive."""

    def __init__(self, handle, tensors, dtype: str, two_d: bool):
        self.handle, self.tensors, self.dtype, self.two_d = handle, tensors, dtype, two_d
        self.slots = None   # amax slots, once set

    def __len__(self):
        return len(self.tensors)

    def close(self):
        if self.handle:
            h, self.handle = self.handle, None
            _check("amp_tensor_list_destroy", load().amp_tensor_list_destroy(h))

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def amp_tensor_list_create(tensors, two_d: bool = False, dtype: str | None = None,
                           stream=None) -> TensorList:
    """Describe contiguous device tensors as one list (2-D lists keep their
    [rows, cols] shapes for the FP8 kernels)."""
    tensors = list(tensors)
    if dtype is None:
        if not tensors:
            raise ValueError("empty list needs an explicit dtype")
        dtype = dtype_name(tensors[0])
    n = len(tensors)
    for t in tensors:
        if not t.is_cuda or not t.is_contiguous() or dtype_name(t) != dtype:
            raise ValueError("every tensor must be a contiguous CUDA tensor of the list dtype")
        if two_d and t.dim() != 2:
            raise ValueError("2-D list needs 2-D tensors")
    ptrs = (P * max(n, 1))(*[t.data_ptr() for t in tensors])
    if two_d:
        rows = (ctypes.c_int64 * max(n, 1))(*[t.shape[0] for t in tensors])
        cols = (ctypes.c_int64 * max(n, 1))(*[t.shape[1] for t in tensors])
    else:
        rows = (ctypes.c_int64 * max(n, 1))(*[t.numel() for t in tensors])
        cols = None
    h = P()
    _check("amp_tensor_list_create",
           load().amp_tensor_list_create(n, ptrs, rows, cols, DT[dtype], _stream(stream),
                                         ctypes.byref(h)))
    return TensorList(h, tensors, dtype, two_d)


def amp_tensor_list_set_amax_slots(lst: TensorList, slots, stream=None):
    slots = [int(s) for s in slots]
    if len(slots) != len(lst):
        raise ValueError(f"{len(slots)} slots for a list of {len(lst)} tensors")
    arr = (ctypes.c_int32 * max(len(lst), 1))(*slots)
    _check("amp_tensor_list_set_amax_slots",
           load().amp_tensor_list_set_amax_slots(lst.handle, arr, _stream(stream)))
    lst.slots = slots


def _n_entries(x: TensorList) -> int:
    """amax / inv_scale entries a list cast reads and writes: one per tensor,
    or up to the largest slot when x has slots."""
    if x.slots is not None and any(s >= 0 for s in x.slots):
        if min(x.slots) < 0:
            raise ValueError("every tensor of a cast list with slots needs a slot >= 0")
        return max(x.slots) + 1
    return len(x)


def amp_tensor_list_destroy(lst: TensorList):
    lst.close()


def amp_tensor_list_check(lst: TensorList, stream=None):
    """Raise AmpError(AMP_ETIMEOUT) if a kernel's bounded wait gave up (synchronises)."""
    _check("amp_tensor_list_check", load().amp_tensor_list_check(lst.handle, _stream(stream)))


def _host_ptrs(items, n: int):
    """Host addresses of numpy arrays / CPU tensors / ints (None for empty tensors)."""
    items = list(items)
    if len(items) != n:
        raise ValueError(f"{len(items)} host buffers for a list of {n} tensors")
    vals = []
    for x in items:
        if x is None or isinstance(x, int):
            vals.append(x)
        elif hasattr(x, "ctypes"):
            vals.append(x.ctypes.data)
        else:
            if x.is_cuda:
                raise ValueError("host buffers must be in host memory")
            vals.append(x.data_ptr())
    return (P * max(n, 1))(*vals)


def amp_tensor_list_copy_from_host(lst: TensorList, host, stream=None):
    """One H2D cudaMemcpyAsync per tensor from the host buffers (kept alive by
    the caller until the copies are done)."""
    _check("amp_tensor_list_copy_from_host",
           load().amp_tensor_list_copy_from_host(lst.handle, _host_ptrs(host, len(lst)),
                                                 _stream(stream)))


def amp_tensor_list_copy_to_host(lst: TensorList, host, stream=None):
    _check("amp_tensor_list_copy_to_host",
           load().amp_tensor_list_copy_to_host(lst.handle, _host_ptrs(host, len(lst)),
                                               _stream(stream)))


class ScalerState(ctypes.Structure):
    """amp_scaler_state: the scaler and step state read back by amp_read_state."""
    _fields_ = [("scale", ctypes.c_float), ("growth_tracker", ctypes.c_int32),
                ("step", ctypes.c_int32), ("found_inf", ctypes.c_int32)]


def amp_read_state(scale, growth_tracker, step, found_inf, host_out, stream=None):
    """Enqueue the D2H copy of {scale, tracker, step, found_inf} into host_out:
    a ScalerState, or the address of one (page-locked for asynchrony)."""
    out = host_out if isinstance(host_out, int) else ctypes.addressof(host_out)
    _check("amp_read_state",
           load().amp_read_state(_buf(scale, "scale", _F32), _buf(growth_tracker, "growth_tracker", _I32),
                                 _buf(step, "step", _I32), _buf(found_inf, "found_inf", _I32), out,
                                 _stream(stream)))


def amp_scale_health(scale, min_scale: float, health, stream=None):
    """Sticky health bits of the loss scale into health (device or page-locked host int32)."""
    _check("amp_scale_health",
           load().amp_scale_health(_buf(scale, "scale", _F32), float(min_scale),
                                   _buf(health, "health", _I32, host_ok=True), _stream(stream)))


def amp_noalloc_check(stream=None):
    """amp_tensor_list_check for the allocation-free AdamW entry point (synchronises)."""
    _check("amp_noalloc_check", load().amp_noalloc_check(_stream(stream)))


def amp_selftest_bounded_wait(err, limit_seconds: float = 0.05, stream=None):
    _check("amp_selftest_bounded_wait",
           load().amp_selftest_bounded_wait(_buf(err, "err", _I32), float(limit_seconds),
                                            _stream(stream)))


def amp_unscale_check(grads: TensorList, scale, found_inf, inplace: bool = False, stream=None):
    _check("amp_unscale_check",
           load().amp_unscale_check(grads.handle, _buf(scale, "scale", _F32),
                                    _buf(found_inf, "found_inf", _I32), int(inplace),
                                    _stream(stream)))


def amp_unscale_check_norm(grads: TensorList, scale, found_inf, grad_sumsq, stream=None):
    """As amp_unscale_check, and grad_sumsq (fp64 device scalar) = sum of
    squared unscaled gradients."""
    _check("amp_unscale_check_norm",
           load().amp_unscale_check_norm(grads.handle, _buf(scale, "scale", _F32),
                                         _buf(found_inf, "found_inf", _I32),
                                         _buf(grad_sumsq, "grad_sumsq", _F64), _stream(stream)))


def amp_adamw_master_step_clip(master: TensorList, exp_avg: TensorList, exp_avg_sq: TensorList,
                               grads: TensorList, bf16_out: TensorList | None, scale, found_inf,
                               step, lr: float, beta1: float, beta2: float, eps: float,
                               weight_decay: float, grad_sumsq, max_norm: float, amax=None,
                               stream=None):
    h = amp_adamw_hyper(lr, beta1, beta2, eps, weight_decay)
    _check("amp_adamw_master_step_clip",
           load().amp_adamw_master_step_clip(master.handle, exp_avg.handle, exp_avg_sq.handle,
                                             grads.handle, bf16_out.handle if bf16_out else None,
                                             *_step_bufs(scale, found_inf, step),
                                             ctypes.byref(h), _buf(amax, "amax", _F32),
                                             _buf(grad_sumsq, "grad_sumsq", _F64),
                                             float(max_norm), _stream(stream)))


def amp_adamw_master_step_clip_sr(master: TensorList, exp_avg: TensorList,
                                  exp_avg_sq: TensorList, grads: TensorList, bf16_out: TensorList,
                                  scale, found_inf, step, lr: float, beta1: float, beta2: float,
                                  eps: float, weight_decay: float, grad_sumsq, max_norm: float,
                                  seed: int, amax=None, stream=None):
    h = amp_adamw_hyper(lr, beta1, beta2, eps, weight_decay)
    _check("amp_adamw_master_step_clip_sr",
           load().amp_adamw_master_step_clip_sr(master.handle, exp_avg.handle, exp_avg_sq.handle,
                                                grads.handle, bf16_out.handle,
                                                *_step_bufs(scale, found_inf, step),
                                                ctypes.byref(h), _buf(amax, "amax", _F32),
                                                _buf(grad_sumsq, "grad_sumsq", _F64),
                                                float(max_norm), ctypes.c_uint64(seed),
                                                _stream(stream)))


def amp_adamw_master_step_sr(master: TensorList, exp_avg: TensorList, exp_avg_sq: TensorList,
                             grads: TensorList, bf16_out: TensorList, scale, found_inf, step,
                             lr: float, beta1: float, beta2: float, eps: float,
                             weight_decay: float, seed: int, amax=None, stream=None):
    h = amp_adamw_hyper(lr, beta1, beta2, eps, weight_decay)
    _check("amp_adamw_master_step_sr",
           load().amp_adamw_master_step_sr(master.handle, exp_avg.handle, exp_avg_sq.handle,
                                           grads.handle, bf16_out.handle,
                                           *_step_bufs(scale, found_inf, step), ctypes.byref(h),
                                           _buf(amax, "amax", _F32), ctypes.c_uint64(seed),
                                           _stream(stream)))


def amp_adamw_master_step(master: TensorList, exp_avg: TensorList, exp_avg_sq: TensorList,
                          grads: TensorList, bf16_out: TensorList | None, scale, found_inf, step,
                          lr: float, beta1: float, beta2: float, eps: float,
                          weight_decay: float, amax=None, stream=None):
    h = amp_adamw_hyper(lr, beta1, beta2, eps, weight_decay)
    _check("amp_adamw_master_step",
           load().amp_adamw_master_step(master.handle, exp_avg.handle, exp_avg_sq.handle,
                                        grads.handle, bf16_out.handle if bf16_out else None,
                                        *_step_bufs(scale, found_inf, step),
                                        ctypes.byref(h), _buf(amax, "amax", _F32),
                                        _stream(stream)))


def amp_emit_bf16(master: TensorList, bf16_out: TensorList, amax=None, stream=None):
    """bf16_out = RNE(master), folding max|bf16| into amax[slot] for tensors
    with an amax slot."""
    if len(master) != len(bf16_out):
        raise ValueError("master and bf16_out differ in tensor count")
    _check("amp_emit_bf16",
           load().amp_emit_bf16(master.handle, bf16_out.handle, _buf(amax, "amax", _F32),
                                _stream(stream)))


def amp_adamw_master_step_noalloc(master, exp_avg, exp_avg_sq, grads, bf16_out, scale,
                                  found_inf, step, lr: float, beta1: float, beta2: float,
                                  eps: float, weight_decay: float, amax_slots=None, amax=None,
                                  stream=None):
    """Allocation-free AdamW step over plain lists of contiguous device tensors
    (no list handles); see include/ampfp8.h for its limits.  Every list must
    hold one tensor per parameter with master's element counts: master, m, v
    fp32, bf16_out bf16, the gradients one dtype among f32/f16/bf16; amax
    must hold every slot named.  A mismatch raises ValueError before the call,
    since the library sees only pointers and would write out of bounds."""
    master = list(master)
    n = len(master)
    lists = {"master": master, "exp_avg": list(exp_avg), "exp_avg_sq": list(exp_avg_sq),
             "grads": list(grads)}
    if bf16_out is not None:
        lists["bf16_out"] = list(bf16_out)
    sizes = [t.numel() for t in master]
    for name, ts in lists.items():
        if len(ts) != n:
            raise ValueError(f"{name}: {len(ts)} tensors, master has {n}")
        for i, t in enumerate(ts):
            if t.numel() != sizes[i]:
                raise ValueError(f"{name}[{i}]: {t.numel()} elements, master[{i}] has {sizes[i]}")
    want = {"master": (torch.float32,), "exp_avg": (torch.float32,),
            "exp_avg_sq": (torch.float32,), "bf16_out": (torch.bfloat16,),
            "grads": (torch.float32, torch.float16, torch.bfloat16)}
    for name, ts in lists.items():
        for i, t in enumerate(ts):
            if t.dtype not in want[name]:
                raise ValueError(f"{name}[{i}]: dtype {t.dtype}, expected one of {want[name]}")
    gdts = {t.dtype for t in lists["grads"]}
    if len(gdts) > 1:
        raise ValueError(f"grads: mixed dtypes {sorted(map(str, gdts))}; one dtype is needed")
    if amax_slots is not None:
        amax_slots = [int(x) for x in amax_slots]
        if len(amax_slots) != n:
            raise ValueError(f"amax_slots: {len(amax_slots)} entries for {n} tensors")
        top = max(amax_slots, default=-1)
        if top >= 0 and bf16_out is not None and (amax is None or top >= amax.numel()):
            raise ValueError(f"amax_slots name slot {top}; amax holds "
                             f"{0 if amax is None else amax.numel()}")
    for name, ts in lists.items():
        if any(not t.is_cuda or not t.is_contiguous() for t in ts):
            raise ValueError(f"{name}: every tensor must be a contiguous CUDA tensor")

    def arr(ts):
        return (P * max(n, 1))(*[t.data_ptr() for t in ts])

    numel = (ctypes.c_int64 * max(n, 1))(*sizes)
    slots = None if amax_slots is None else (ctypes.c_int32 * max(n, 1))(*amax_slots)
    h = amp_adamw_hyper(lr, beta1, beta2, eps, weight_decay)
    _check("amp_adamw_master_step_noalloc",
           load().amp_adamw_master_step_noalloc(
               n, arr(master), arr(lists["exp_avg"]), arr(lists["exp_avg_sq"]),
               arr(lists["grads"]), DT[dtype_name(lists["grads"][0])] if n else DT["f32"],
               arr(lists["bf16_out"]) if bf16_out is not None else None, numel, slots,
               *_step_bufs(scale, found_inf, step), ctypes.byref(h), _buf(amax, "amax", _F32),
               _stream(stream)))


def amp_adamw_master_step_fp8_delayed(plain, fp8_group, fp8_out: TensorList,
                                      fp8_t_out: TensorList | None, fp8_dtype: str,
                                      amax_history, hist_len: int, amax, inv_scale, scale,
                                      found_inf, step, lr: float, beta1: float, beta2: float,
                                      eps: float, weight_decay: float, fp8_eps: float = 1e-12,
                                      stream=None):
    """plain / fp8_group: (master, exp_avg, exp_avg_sq, grads, bf16_out) TensorLists;
    the FP8 group's lists are 2-D."""
    h = amp_adamw_hyper(lr, beta1, beta2, eps, weight_decay)
    _check("amp_adamw_master_step_fp8_delayed",
           load().amp_adamw_master_step_fp8_delayed(
               *[x.handle for x in plain], *[x.handle for x in fp8_group], fp8_out.handle,
               fp8_t_out.handle if fp8_t_out else None, DT[fp8_dtype], fp8_eps,
               _buf(amax_history, "amax_history", _F32, len(fp8_out) * int(hist_len)),
               int(hist_len), _buf(amax, "amax", _F32, len(fp8_out)),
               _buf(inv_scale, "inv_scale", _F32, len(fp8_out)),
               *_step_bufs(scale, found_inf, step), ctypes.byref(h), _stream(stream)))


def amp_adamw_master_step_fp8_delayed_sr(plain, fp8_group, fp8_out: TensorList,
                                         fp8_t_out: TensorList | None, fp8_dtype: str,
                                         amax_history, hist_len: int, amax, inv_scale, scale,
                                         found_inf, step, lr: float, beta1: float, beta2: float,
                                         eps: float, weight_decay: float, seed: int,
                                         fp8_eps: float = 1e-12, stream=None):
    """amp_adamw_master_step_fp8_delayed with the bf16 and FP8 copies rounded
    stochastically (Philox4x32-10 with this 64-bit seed)."""
    h = amp_adamw_hyper(lr, beta1, beta2, eps, weight_decay)
    _check("amp_adamw_master_step_fp8_delayed_sr",
           load().amp_adamw_master_step_fp8_delayed_sr(
               *[x.handle for x in plain], *[x.handle for x in fp8_group], fp8_out.handle,
               fp8_t_out.handle if fp8_t_out else None, DT[fp8_dtype], fp8_eps,
               _buf(amax_history, "amax_history", _F32, len(fp8_out) * int(hist_len)),
               int(hist_len), _buf(amax, "amax", _F32, len(fp8_out)),
               _buf(inv_scale, "inv_scale", _F32, len(fp8_out)),
               *_step_bufs(scale, found_inf, step), ctypes.byref(h), ctypes.c_uint64(seed),
               _stream(stream)))


def amp_update_scale_fp8_history(scale, growth_tracker, found_inf, growth_factor: float,
                                 backoff_factor: float, growth_interval: int, amax,
                                 amax_history, n_fp8: int, hist_len: int, stream=None):
    _check("amp_update_scale_fp8_history",
           load().amp_update_scale_fp8_history(_buf(scale, "scale", _F32),
                                               _buf(growth_tracker, "growth_tracker", _I32),
                                               _buf(found_inf, "found_inf", _I32), growth_factor,
                                               backoff_factor, int(growth_interval),
                                               _buf(amax, "amax", _F32, int(n_fp8)),
                                               _buf(amax_history, "amax_history", _F32,
                                                    int(n_fp8) * int(hist_len)),
                                               int(n_fp8), int(hist_len), _stream(stream)))


def fp8_quant_tensorwise(x: torch.Tensor, fp8_dtype: str, out: torch.Tensor, out_t, inv_scale,
                         amax, amax_given: bool = False, eps: float = 1e-12, skip_if=None,
                         stream=None, rows: int | None = None, cols: int | None = None):
    """x is [rows, cols] row-major (a 1-D tensor is one row unless rows/cols say otherwise)."""
    if rows is None:
        rows, cols = (x.shape[0], x.shape[1]) if x.dim() == 2 else (1, x.numel())
    _check("fp8_quant_tensorwise",
           load().fp8_quant_tensorwise(_buf(x, "x", numel=rows * cols), DT[dtype_name(x)], rows,
                                       cols, DT[fp8_dtype], eps,
                                       _buf(out, "out", itemsize=1, numel=rows * cols),
                                       _buf(out_t, "out_t", itemsize=1, numel=rows * cols),
                                       _buf(inv_scale, "inv_scale", _F32),
                                       _buf(amax, "amax", _F32), int(amax_given),
                                       _buf(skip_if, "skip_if", _I32),
                                       _stream(stream)))


def fp8_quant_rowwise(x: torch.Tensor, fp8_dtype: str, out, out_t, amax_row, scale_row,
                      inv_scale_row, amax_col=None, scale_col=None, inv_scale_col=None,
                      eps: float = 1e-12, skip_if=None, stream=None):
    """x is [rows, cols]; per-row scales for out, per-column scales for out_t."""
    rows, cols = x.shape
    _check("fp8_quant_rowwise",
           load().fp8_quant_rowwise(_buf(x, "x", numel=rows * cols), DT[dtype_name(x)], rows, cols,
                                    DT[fp8_dtype], eps,
                                    _buf(out, "out", itemsize=1, numel=rows * cols),
                                    _buf(out_t, "out_t", itemsize=1, numel=rows * cols),
                                    *[_buf(t, n, _F32, rows) for t, n in
                                      ((amax_row, "amax_row"), (scale_row, "scale_row"),
                                       (inv_scale_row, "inv_scale_row"))],
                                    *[_buf(t, n, _F32, cols) for t, n in
                                      ((amax_col, "amax_col"), (scale_col, "scale_col"),
                                       (inv_scale_col, "inv_scale_col"))],
                                    _buf(skip_if, "skip_if", _I32), _stream(stream)))


def fp8_quant_groupwise(x: torch.Tensor, fp8_dtype: str, group: int, out, out_t, amax_rg,
                        scale_rg, inv_rg, amax_cg=None, scale_cg=None, inv_cg=None,
                        eps: float = 1e-12, skip_if=None, stream=None):
    """x is [rows, cols]; one scale per `group` elements of a row for out, per
    `group` rows of a column for out_t ([cols, rows])."""
    rows, cols = x.shape
    g = max(int(group), 1)
    n_rg, n_cg = rows * -(-cols // g), cols * -(-rows // g)
    _check("fp8_quant_groupwise",
           load().fp8_quant_groupwise(_buf(x, "x", numel=rows * cols), DT[dtype_name(x)], rows,
                                      cols, int(group), DT[fp8_dtype], eps,
                                      _buf(out, "out", itemsize=1, numel=rows * cols),
                                      _buf(out_t, "out_t", itemsize=1, numel=rows * cols),
                                      *[_buf(t, n, _F32, n_rg) for t, n in
                                        ((amax_rg, "amax_rg"), (scale_rg, "scale_rg"),
                                         (inv_rg, "inv_rg"))],
                                      *[_buf(t, n, _F32, n_cg) for t, n in
                                        ((amax_cg, "amax_cg"), (scale_cg, "scale_cg"),
                                         (inv_cg, "inv_cg"))],
                                      _buf(skip_if, "skip_if", _I32), _stream(stream)))


def fp8_quant_tensorwise_list(x: TensorList, out: TensorList, out_t: TensorList | None,
                              fp8_dtype: str, amax, inv_scale, eps: float = 1e-12, skip_if=None,
                              stream=None):
    _check("fp8_quant_tensorwise_list",
           load().fp8_quant_tensorwise_list(x.handle, out.handle, out_t.handle if out_t else None,
                                            DT[fp8_dtype], eps,
                                            _buf(amax, "amax", _F32, _n_entries(x)),
                                            _buf(inv_scale, "inv_scale", _F32, _n_entries(x)),
                                            _buf(skip_if, "skip_if", _I32), _stream(stream)))


def fp8_quant_tensorwise_list_sr(x: TensorList, out: TensorList, out_t: TensorList | None,
                                 fp8_dtype: str, amax, inv_scale, seed: int, step,
                                 eps: float = 1e-12, skip_if=None, stream=None):
    """fp8_quant_tensorwise_list with stochastically rounded FP8 bytes; step is
    the device step counter whose value keys the random draws."""
    _check("fp8_quant_tensorwise_list_sr",
           load().fp8_quant_tensorwise_list_sr(x.handle, out.handle,
                                               out_t.handle if out_t else None, DT[fp8_dtype],
                                               eps, _buf(amax, "amax", _F32, _n_entries(x)),
                                               _buf(inv_scale, "inv_scale", _F32, _n_entries(x)),
                                               _buf(skip_if, "skip_if", _I32),
                                               ctypes.c_uint64(seed), _buf(step, "step", _I32),
                                               _stream(stream)))


def amp_update_scale(scale, growth_tracker, found_inf, growth_factor: float,
                     backoff_factor: float, growth_interval: int, amax=None, n_amax: int = 0,
                     stream=None):
    _check("amp_update_scale",
           load().amp_update_scale(_buf(scale, "scale", _F32),
                                   _buf(growth_tracker, "growth_tracker", _I32),
                                   _buf(found_inf, "found_inf", _I32),
                                   growth_factor, backoff_factor, int(growth_interval),
                                   _buf(amax, "amax", _F32, int(n_amax)), int(n_amax),
                                   _stream(stream)))


def amp_last_error() -> str:
    return load().amp_last_error().decode(errors="replace")


def amp_abi_version() -> int:
    return load().amp_abi_version()
