"""The oracle's encoders over all 2^32 fp32 bit patterns against independent
library casts: torch's binary16, bfloat16, e4m3fn and e5m2 conversions
(round to nearest even; overflow to inf, or to NaN for e4m3fn, which has no
infinity).  The binary16 cast is also checked against numpy's on 6.3 M
rounding-class patterns in the pins; here torch's is used because numpy's
float16 conversion takes minutes over 2^32 values.  NaN outputs are compared
as NaN (the oracle writes canonical NaNs, the libraries keep payloads).  CPU
only, split over spawned worker processes."""
import multiprocessing as mp
import os

import pytest

pytestmark = pytest.mark.slow

CHUNK = 1 << 23


@pytest.fixture(scope="module")
def pool():
    ctx = mp.get_context("spawn")
    n = max(2, min(16, os.cpu_count() or 2))
    with ctx.Pool(n) as p:
        yield p


@pytest.mark.parametrize("fmt", ["f16", "bf16", "e4m3fn", "e5m2"])
def test_encoder_matches_library_on_every_fp32_pattern(pool, fmt):
    import exhaustive_encode_worker as W
    res = pool.map(W.compare, [(fmt, lo, CHUNK) for lo in range(0, 1 << 32, CHUNK)])
    bad = sum(r[0] for r in res)
    examples = [e for r in res for e in r[1]][:10]
    assert bad == 0, (fmt, bad, examples)
