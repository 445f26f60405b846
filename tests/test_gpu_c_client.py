"""The C ABI used from plain C: a C program (tests/c_client/amp_c_client.c,
built with gcc against include/ampfp8.h and libampfp8.so) runs the tiny
configuration with an FP8 weight, with dynamic FP8 scaling and, from the
first working copies it emits itself, with delayed scaling; its outputs must
equal the oracle's bit for bit."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle as O
from workloads import amp_config, host_grads, host_master

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("mode", ["dynamic", "delayed"])
def test_plain_c_client_matches_oracle(tmp_path, mode):
    from loss_scaling_master_gb300 import build as B
    lib = B.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = str(tmp_path / "amp_c_client")
    cc = shutil.which("gcc") or "cc"
    subprocess.check_call([cc, "-std=c11", "-O1", os.path.join(ROOT, "tests", "c_client", "amp_c_client.c"),
                           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                           "-L", os.path.dirname(lib), "-lampfp8", "-L", os.path.join(cuda, "lib64"),
                           "-lcudart", "-Wl,-rpath," + os.path.dirname(lib) + ":" +
                           os.path.join(cuda, "lib64"), "-o", exe])
    cfg = amp_config("tiny")
    shapes = [None, (64, 64), None]                          # tensor 1 (4096) is an FP8 weight
    masters = host_master(cfg)
    orc = O.AmpStepOracle(masters, "f16", cfg.lr, cfg.beta1, cfg.beta2, cfg.eps, cfg.weight_decay,
                          cfg.init_scale, cfg.growth_factor, cfg.backoff_factor,
                          cfg.growth_interval, fp8_shapes=shapes, fp8_scaling=mode, hist_len=1)
    grads, fi = [], []
    for k in range(1, cfg.steps + 1):
        g = host_grads(cfg, k, orc.scale)
        grads.append(g)
        fi.append(orc.run(g))
    with open(tmp_path / "in.bin", "wb") as f:
        f.write(np.array([len(masters), cfg.steps], np.int32).tobytes())
        for s, sh in zip(cfg.specs, shapes):
            f.write(np.array([s.numel, sh[0] if sh else 0, sh[1] if sh else 0], np.int64).tobytes())
        for m in masters:
            f.write(m.tobytes())
        for g in grads:
            for t in g:
                f.write(t.tobytes())
    out = subprocess.run([exe, str(tmp_path / "in.bin"), str(tmp_path / "out.bin")]
                         + (["delayed"] if mode == "delayed" else []),
                         capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    raw = open(tmp_path / "out.bin", "rb").read()
    off = 0

    def take(dtype, count):
        nonlocal off
        a = np.frombuffer(raw, dtype=dtype, count=count, offset=off)
        off += a.nbytes
        return a
    assert take(np.int32, cfg.steps).tolist() == fi
    assert take(np.float32, 1)[0] == orc.scale
    assert take(np.int32, 1)[0] == orc.tracker and take(np.int32, 1)[0] == orc.step
    for i, s in enumerate(cfg.specs):
        for ref in (orc.master[i], orc.exp_avg[i], orc.exp_avg_sq[i]):
            assert np.array_equal(take(np.uint32, s.numel), ref.view(np.uint32))
        assert np.array_equal(take(np.uint16, s.numel), orc.bf16[i])
    for i, sh in enumerate(shapes):
        if sh is None:
            continue
        assert np.array_equal(take(np.uint8, cfg.specs[i].numel), orc.fp8[i])
        assert np.array_equal(take(np.uint8, cfg.specs[i].numel), orc.fp8_t[i])
        assert take(np.float32, 1)[0] == orc.inv_scale[orc.slots[i]]
    assert off == len(raw)
