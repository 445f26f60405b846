"""Shared helpers of the GPU parity tests: tolerances stated by the method's
accuracy contract, and host<->device marshalling of raw bit patterns."""
import numpy as np
import torch

# Contract: found_inf, scale, tracker, step, skip, FP8 bytes and inv_scale
# bit-exact; fp32 master/m/v within rel 1e-6 (floor 1e-6 * rms of the tensor
# for values that cross zero); the bf16 copy within 1 bf16 ulp.
STATE_RTOL = 1e-6
BF16_ULP = 1

_BITS = {torch.float32: (np.uint32, torch.int32), torch.float16: (np.uint16, torch.int16),
         torch.bfloat16: (np.uint16, torch.int16), torch.float8_e4m3fn: (np.uint8, torch.uint8),
         torch.float8_e5m2: (np.uint8, torch.uint8), torch.int32: (np.int32, torch.int32),
         torch.uint8: (np.uint8, torch.uint8)}
_NPDT = {"f32": (np.float32, torch.float32), "f16": (np.uint16, torch.float16),
         "bf16": (np.uint16, torch.bfloat16)}


def to_host_bits(t: torch.Tensor) -> np.ndarray:
    """Device tensor -> host numpy array of its raw bits (float32 stays float32)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.float32:
        return t.numpy().copy()
    npdt, idt = _BITS[t.dtype]
    return t.view(idt).numpy().view(npdt).copy()


def to_device(bits: np.ndarray, dt: str, device) -> torch.Tensor:
    """Host bits/values of dtype name dt ('f32' | 'f16' | 'bf16') -> device tensor."""
    npdt, tdt = _NPDT[dt]
    a = np.ascontiguousarray(bits, npdt)
    if dt == "f32":
        return torch.from_numpy(a.copy()).to(device)
    return torch.from_numpy(a.view(np.int16).copy()).to(device).view(tdt)


def assert_state_close(got: np.ndarray, ref: np.ndarray, what: str):
    """rel 1e-6, floor 1e-6 * rms(ref); NaN matches NaN."""
    g = got.astype(np.float64)
    r = ref.astype(np.float64)
    both_nan = np.isnan(g) & np.isnan(r)
    fin = np.isfinite(r)
    rms = np.sqrt(np.mean(r[fin] ** 2)) if fin.any() else 0.0
    err = np.abs(g - r)
    ok = both_nan | (g == r) | (err <= STATE_RTOL * np.maximum(np.abs(g), np.abs(r)) + 1e-6 * rms)
    if not ok.all():
        i = int(np.flatnonzero(~ok)[0])
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outside rel 1e-6; first at "
                             f"{i}: got {got[i]!r} ref {ref[i]!r}")


def bf16_ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in representable bf16 steps between two bit-pattern arrays
    (sign-magnitude mapped onto a monotone integer line)."""
    def key(x):
        x = x.astype(np.int64)
        return np.where(x & 0x8000, -(x & 0x7FFF), x & 0x7FFF)
    return np.abs(key(a) - key(b))


def assert_bf16_close(got: np.ndarray, ref: np.ndarray, what: str):
    nan_g = (got & 0x7FFF) > 0x7F80
    nan_r = (ref & 0x7FFF) > 0x7F80
    assert np.array_equal(nan_g, nan_r), f"{what}: NaN positions differ"
    d = bf16_ulp_distance(got[~nan_r], ref[~nan_r])
    if d.size and d.max() > BF16_ULP:
        raise AssertionError(f"{what}: max bf16 distance {int(d.max())} ulp")


def bit_identical_fraction(got: np.ndarray, ref: np.ndarray) -> float:
    g = got.view(np.uint32) if got.dtype == np.float32 else got
    r = ref.view(np.uint32) if ref.dtype == np.float32 else ref
    return float(np.mean(g == r)) if g.size else 1.0
