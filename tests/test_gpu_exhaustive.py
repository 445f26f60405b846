"""Exhaustive parity over all 2^32 fp32 bit patterns, GPU path against the oracle.

* FP8 cast ([FP8] §2, §3): the quantizer with amax = fp8_max has scale exactly
  1, so its bytes are the saturating round-to-nearest-even cast of each fp32
  pattern itself: every sign, exponent, subnormal, tie, overflow, inf and NaN.
* BF16 working copy ([MP] "PyTorch AMP and FP32 master weights"): with lr = 0,
  weight decay 0 and zero gradients the AdamW step leaves every master value
  unchanged, so the emitted copy is RNE(p) for every fp32 pattern p.

The sweep runs in chunks of 2^28 patterns; the oracle's share of each chunk is
split over spawned worker processes (tests/exhaustive_oracle.py)."""
import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

from parity_helpers import to_host_bits

pytestmark = pytest.mark.gpu

CHUNK = 1 << 28
SIDE = 1 << 14            # each chunk is quantized as a [2^14, 2^14] matrix


@pytest.fixture(scope="module")
def A():
    from loss_scaling_master_gb300 import build as B
    B.build()
    import loss_scaling_master_gb300 as pkg
    pkg.load()
    assert torch.cuda.is_available()
    return pkg


@pytest.fixture(scope="module")
def pool():
    ctx = mp.get_context("spawn")
    n = max(2, min(16, os.cpu_count() or 2))
    with ctx.Pool(n) as p:
        yield p, n


def _device_patterns(lo: int, n: int, dev) -> torch.Tensor:
    k = torch.arange(lo, lo + n, dtype=torch.int64, device=dev)
    k = torch.where(k >= (1 << 31), k - (1 << 32), k)
    return k.to(torch.int32).view(torch.float32)


def _oracle_chunk(pool, fn, lo, n, extra=()):
    p, workers = pool
    sub = n // workers
    assert sub * workers == n
    parts = p.map(fn, [(*extra, lo + w * sub, sub) for w in range(workers)])
    return np.concatenate(parts)


def _first_mismatches(got, ref, lo, k=5):
    idx = np.flatnonzero(got != ref)[:k]
    return [(hex(lo + int(i)), hex(int(got[i])), hex(int(ref[i]))) for i in idx]


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
def test_fp8_cast_all_fp32_patterns(A, pool, fmt):
    import exhaustive_oracle as X
    dev = torch.device("cuda:0")
    fmax = {"e4m3fn": 448.0, "e5m2": 57344.0}[fmt]
    out = torch.empty(CHUNK, dtype=torch.uint8, device=dev)
    inv = torch.zeros(1, device=dev)
    amax = torch.tensor([fmax], device=dev)
    for lo in range(0, 1 << 32, CHUNK):
        x = _device_patterns(lo, CHUNK, dev)
        A.fp8_quant_tensorwise(x, fmt, out, None, inv, amax, amax_given=True, rows=SIDE, cols=SIDE)
        got = to_host_bits(out)
        del x
        ref = _oracle_chunk(pool, X.fp8_cast, lo, CHUNK, (fmt,))
        assert np.array_equal(got, ref), _first_mismatches(got, ref, lo)
        assert float(inv.item()) == 1.0


def test_bf16_copy_all_fp32_patterns(A, pool):
    import exhaustive_oracle as X
    dev = torch.device("cuda:0")
    P = torch.empty(CHUNK, dtype=torch.float32, device=dev)
    M = torch.zeros(CHUNK, device=dev)
    V = torch.zeros(CHUNK, device=dev)
    G = torch.zeros(CHUNK, dtype=torch.float16, device=dev)
    B = torch.empty(CHUNK, dtype=torch.bfloat16, device=dev)
    Ls = [A.amp_tensor_list_create([t]) for t in (P, M, V, G, B)]
    step = torch.zeros(1, dtype=torch.int32, device=dev)
    try:
        for lo in range(0, 1 << 32, CHUNK):
            P.copy_(_device_patterns(lo, CHUNK, dev))
            A.amp_adamw_master_step(*Ls, None, None, step, 0.0, 0.9, 0.999, 1e-8, 0.0)
            got = to_host_bits(B)
            ref = _oracle_chunk(pool, X.bf16_copy, lo, CHUNK)
            assert np.array_equal(got, ref), _first_mismatches(got, ref, lo)
        A.amp_tensor_list_check(Ls[0])
        assert int(step.item()) == (1 << 32) // CHUNK
    finally:
        for L in Ls:
            L.close()
