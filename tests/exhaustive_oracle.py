"""Oracle side of the exhaustive sweeps over all 2^32 fp32 bit patterns.

Run in worker processes started with the ``spawn`` method (they import numpy
and the oracle only, never CUDA).  Pattern k of the sweep is the fp32 whose
bits are the unsigned integer k."""
import numpy as np

import oracle as O


def patterns(lo: int, n: int) -> np.ndarray:
    return np.arange(lo, lo + n, dtype=np.uint32).view(np.float32)


def fp8_cast(args):
    """Quantizer bytes of patterns [lo, lo+n) with amax = fp8_max, i.e. scale
    exactly 1: the saturating RNE cast of each pattern itself ([FP8] §2)."""
    fmt, lo, n = args
    q, _, _, _ = O.fp8_quant_tensorwise(patterns(lo, n), "f32", 1, n, fmt, transposed=False,
                                        amax=O.fmt_max(fmt))
    return q


def bf16_copy(args):
    """RNE bf16 of patterns [lo, lo+n): the working copy of an unchanged master."""
    lo, n = args
    return O.encode("bf16", patterns(lo, n))
