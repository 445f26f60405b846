"""The allocation-free AdamW entry point against the handle-based one.

amp_adamw_master_step_noalloc serves callers that cannot allocate device
memory (an arena-owning runtime, a loop that must not take cudaMalloc's
device synchronisation, a GPU run nearly full, a plain-C caller without
handle lifetimes).  It keeps its tables in a fixed device array built into
the library instead of cudaMalloc'd handles.  This test calls it through the
C ABI and checks its outputs against amp_adamw_master_step on the same inputs,
on two calls in a row (the second reuses the array the first left behind).
The file sorts last so a stop-at-first-failure run has run everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

from parity_helpers import assert_bf16_close, assert_state_close, to_host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    from loss_scaling_master_gb300 import build as B
    B.build()
    import loss_scaling_master_gb300 as pkg
    pkg.load()
    assert torch.cuda.is_available()
    return pkg


def _state(dev, sizes, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    p = [(torch.randn(n, generator=g) * 0.02).to(dev) for n in sizes]
    return p, [torch.zeros(n, device=dev) for n in sizes], [torch.zeros(n, device=dev) for n in sizes], \
        [torch.empty(n, dtype=torch.bfloat16, device=dev) for n in sizes]


def test_noalloc_matches_handle_path_two_calls(A):
    dev = torch.device("cuda:0")
    sizes = [1, 257, 4096, 16384, 16385, 40000, 3 * 16384 + 7]
    slots = [-1, 0, -1, 1, -1, 2, -1]
    hyper = (1e-3, 0.9, 0.999, 1e-8, 0.01)
    pa, ma, va, ba = _state(dev, sizes, 1)
    pb, mb, vb, bb = [t.clone() for t in pa], [t.clone() for t in ma], [t.clone() for t in va], \
        [t.clone() for t in ba]
    LP, LM, LV, LB = (A.amp_tensor_list_create(x) for x in (pa, ma, va, ba))
    A.amp_tensor_list_set_amax_slots(LB, slots)
    scale = torch.tensor([65536.0], device=dev)
    fi = torch.zeros(1, dtype=torch.int32, device=dev)
    step_a = torch.zeros(1, dtype=torch.int32, device=dev)
    step_b = torch.zeros(1, dtype=torch.int32, device=dev)
    gen = torch.Generator(device="cpu").manual_seed(2)
    for call in range(2):
        grads = [(torch.randn(n, generator=gen) * 1e-4 * 65536).half().to(dev) for n in sizes]
        LG = A.amp_tensor_list_create(grads)
        amax_a = torch.zeros(3, device=dev)
        amax_b = torch.zeros(3, device=dev)
        A.amp_adamw_master_step(LP, LM, LV, LG, LB, scale, fi, step_a, *hyper, amax=amax_a)
        A.amp_adamw_master_step_noalloc(pb, mb, vb, grads, bb, scale, fi, step_b, *hyper,
                                        amax_slots=slots, amax=amax_b)
        torch.cuda.synchronize()
        A.amp_noalloc_check()
        A.amp_tensor_list_check(LP)
        LG.close()
        assert int(step_a.item()) == int(step_b.item()) == call + 1
        assert np.array_equal(to_host_bits(amax_a).view(np.uint32), to_host_bits(amax_b).view(np.uint32))
        for i in range(len(sizes)):
            assert_state_close(to_host_bits(pb[i]), to_host_bits(pa[i]), f"master[{i}] call {call}")
            assert_state_close(to_host_bits(mb[i]), to_host_bits(ma[i]), f"exp_avg[{i}] call {call}")
            assert_state_close(to_host_bits(vb[i]), to_host_bits(va[i]), f"exp_avg_sq[{i}] call {call}")
            assert_bf16_close(to_host_bits(bb[i]), to_host_bits(ba[i]), f"bf16[{i}] call {call}")
    for L in (LP, LM, LV, LB):
        L.close()


def test_noalloc_rejects_sizes_beyond_its_array(A):
    L = A.load()
    from loss_scaling_master_gb300._lib import DT, amp_adamw_hyper
    P = ctypes.c_void_p
    dummy = torch.zeros(4, dtype=torch.int32, device="cuda:0")
    h = amp_adamw_hyper(1e-3, 0.9, 0.999, 1e-8, 0.0)
    n = 1025                                            # over the tensor limit
    ptrs = (P * n)(*([dummy.data_ptr()] * n))
    numel = (ctypes.c_int64 * n)(*([1] * n))
    st = L.amp_adamw_master_step_noalloc(n, ptrs, ptrs, ptrs, ptrs, DT["f32"], None, numel, None,
                                         None, None, P(dummy.data_ptr()), ctypes.byref(h), None,
                                         None)
    assert st == -1 and b"limit" in L.amp_last_error()
    n = 1                                               # over the chunk limit
    numel = (ctypes.c_int64 * 1)(524288 * 16384 + 1)
    st = L.amp_adamw_master_step_noalloc(n, ptrs, ptrs, ptrs, ptrs, DT["f32"], None, numel, None,
                                         None, None, P(dummy.data_ptr()), ctypes.byref(h), None,
                                         None)
    assert st == -1 and b"limit" in L.amp_last_error()
