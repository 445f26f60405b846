"""Host logic: the synthetic parameter sets have the sizes the configs name."""
import numpy as np

from workloads import (amp_config, gpt2_small_specs, host_grads, injection_site,
                       llama3_8b_specs, llama_1b_specs, tiny_specs)


def _count(specs):
    return sum(s.numel for s in specs), len(specs)


def test_param_set_sizes():
    assert _count(tiny_specs()) == (5353, 3)
    assert _count(gpt2_small_specs()) == (124_356_864, 100)
    assert _count(llama_1b_specs()) == (1_235_814_400, 146)
    assert _count(llama3_8b_specs()) == (8_030_261_248, 291)
    fp8 = [s for s in llama3_8b_specs() if s.fp8]
    assert len(fp8) == 224 and sum(s.numel for s in fp8) == 6_979_321_856
    two = amp_config("llama3_8b_2layers").specs
    assert _count(two) == (436_224_000, 18) and sum(s.numel for s in two if s.fp8) == 436_207_616


def test_injection_sites_are_seeded_and_in_range():
    cfg = amp_config("llama_1b")
    sites = {k: injection_site(cfg, k) for k in (7, 27, 47)}
    assert sites == {k: injection_site(cfg, k) for k in (7, 27, 47)}
    for k, (t, e, v) in sites.items():
        assert 0 <= e < cfg.specs[t].numel
    assert np.isposinf(sites[7][2]) and np.isneginf(sites[27][2]) and np.isnan(sites[47][2])
    assert injection_site(cfg, 8) is None


def test_tiny_grads_plant_inf_at_step_2_tail():
    cfg = amp_config("tiny")
    g = host_grads(cfg, 2, 65536.0)
    assert g[2][256] == 0x7C00
    assert all(np.isfinite(x.view(np.float16)).all() for x in host_grads(cfg, 1, 65536.0))
