"""Worker of the exhaustive encoder pin (spawned processes; CPU only): the
oracle's RNE encoder against torch's casts on a range of fp32 patterns."""
import numpy as np

import oracle as O

# NaN bit patterns by definition of each format: all-ones exponent with a
# non-zero fraction (binary16, bfloat16, e5m2); S.1111.111 for e4m3fn
_NAN = {"f16": lambda b: (b & 0x7C00 == 0x7C00) & (b & 0x03FF != 0),
        "bf16": lambda b: (b & 0x7F80 == 0x7F80) & (b & 0x007F != 0),
        "e5m2": lambda b: (b & 0x7C == 0x7C) & (b & 0x03 != 0),
        "e4m3fn": lambda b: b & 0x7F == 0x7F}


def compare(args):
    fmt, lo, n = args
    import torch
    torch.set_num_threads(1)
    x = np.arange(lo, lo + n, dtype=np.uint32).view(np.float32)
    ours = O.encode(fmt, x)
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "e4m3fn": torch.float8_e4m3fn,
           "e5m2": torch.float8_e5m2}[fmt]
    it = torch.int16 if fmt in ("f16", "bf16") else torch.uint8
    npdt = np.uint16 if fmt in ("f16", "bf16") else np.uint8
    ref = torch.from_numpy(x).to(tdt).view(it).numpy().view(npdt)
    isnan = _NAN[fmt]
    nan_o, nan_r = isnan(ours), isnan(ref)
    bad = (nan_o != nan_r) | (~nan_o & (ours != ref))
    idx = np.flatnonzero(bad)
    return int(idx.size), [(hex(lo + int(i)), hex(int(ours[i])), hex(int(ref[i]))) for i in idx[:5]]
