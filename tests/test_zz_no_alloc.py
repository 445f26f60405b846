"""The allocation-free AdamW entry point against the handle-based one and the
oracle.

amp_adamw_master_step_noalloc serves callers that cannot allocate device
memory (an arena-owning runtime, a loop that must not take cudaMalloc's
device synchronisation, a GPU run nearly full, a plain-C caller without
handle lifetimes).  It keeps its tables in a fixed device array built into
the library instead of cudaMalloc'd handles.  These tests call it through the
C ABI and check its outputs against amp_adamw_master_step on the same inputs
and against the CPU oracle, on calls in a row that reuse the array the call
before left behind (a larger table, then a smaller one), with every gradient
dtype, with and without the bf16 copy, on a side stream, on a skipped step, on
an empty parameter list, and on a stream that is capturing a graph (refused).
The file sorts last so a stop-at-first-failure run has run everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from parity_helpers import assert_bf16_close, assert_state_close, to_device, to_host_bits

pytestmark = pytest.mark.gpu

HYPER = (1e-3, 0.9, 0.999, 1e-8, 0.01)


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


def _grads_host(rng, sizes, gdt, sigma):
    out = []
    for n in sizes:
        x = (rng.standard_normal(n) * sigma).astype(np.float32)
        out.append(x if gdt == "f32" else
                   x.astype(np.float16).view(np.uint16) if gdt == "f16" else O.encode("bf16", x))
    return out


def test_noalloc_matches_handle_path_two_calls(A):
    dev = torch.device("cuda:0")
    sizes = [1, 257, 4096, 16384, 16385, 40000, 3 * 16384 + 7]
    slots = [-1, 0, -1, 1, -1, 2, -1]
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
        A.amp_adamw_master_step(LP, LM, LV, LG, LB, scale, fi, step_a, *HYPER, amax=amax_a)
        A.amp_adamw_master_step_noalloc(pb, mb, vb, grads, bb, scale, fi, step_b, *HYPER,
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


@pytest.mark.parametrize("gdt", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("with_bf16", [True, False])
def test_noalloc_matches_oracle_and_handle_path(A, gdt, with_bf16):
    """Three calls in a row on a side stream - a large table, then a smaller
    one, then a skipped step - against the oracle (bit-identical fp32 state,
    the same step counter and amax) and against the handle-based entry point."""
    dev = torch.device("cuda:0")
    rng = np.random.default_rng(90)
    big = [7, 16384, 16385, 40000, 3 * 16384 + 5, 1000]
    small = big[:3]
    side = torch.cuda.Stream(device=dev)
    for sizes, skip in ((big, 0), (small, 0), (small, 1)):
        n = len(sizes)
        master_h = [(rng.standard_normal(k) * 0.02).astype(np.float32) for k in sizes]
        gh = _grads_host(rng, sizes, gdt, 1e-3 * 1024.0)
        slots = [i % 2 if with_bf16 else -1 for i in range(n)]
        slots[0] = -1
        P = [to_device(h, "f32", dev) for h in master_h]
        M = [torch.zeros(k, device=dev) for k in sizes]
        V = [torch.zeros(k, device=dev) for k in sizes]
        G = [to_device(h, gdt, dev) for h in gh]
        B = [torch.zeros(k, dtype=torch.bfloat16, device=dev) for k in sizes] if with_bf16 else None
        P2, M2, V2 = [t.clone() for t in P], [t.clone() for t in M], [t.clone() for t in V]
        B2 = [t.clone() for t in B] if with_bf16 else None
        scale = torch.tensor([1024.0], device=dev)
        fi = torch.full((1,), skip, dtype=torch.int32, device=dev)
        step = torch.full((1,), 4, dtype=torch.int32, device=dev)
        step2 = step.clone()
        amax = torch.zeros(2, device=dev)
        amax2 = torch.zeros(2, device=dev)
        torch.cuda.synchronize()
        A.amp_adamw_master_step_noalloc(P, M, V, G, B, scale, fi, step, *HYPER,
                                        amax_slots=slots if with_bf16 else None,
                                        amax=amax if with_bf16 else None, stream=side)
        lists = [A.amp_tensor_list_create(x) for x in (P2, M2, V2, G)]
        LB = A.amp_tensor_list_create(B2) if with_bf16 else None
        if with_bf16:
            A.amp_tensor_list_set_amax_slots(LB, slots)
        A.amp_adamw_master_step(*lists, LB, scale, fi, step2, *HYPER,
                                amax=amax2 if with_bf16 else None)
        torch.cuda.synchronize()
        A.amp_noalloc_check(stream=side)

        rm = [np.zeros(k, np.float32) for k in sizes]
        rv = [np.zeros(k, np.float32) for k in sizes]
        rp = [h.copy() for h in master_h]
        rb = [np.zeros(k, np.uint16) for k in sizes] if with_bf16 else None
        ram = np.zeros(2, np.float32)
        rstep = O.adamw_master_step(rp, rm, rv, gh, gdt, rb, 1024.0, skip, 4, *HYPER,
                                    amax_slot=slots if with_bf16 else None,
                                    amax=ram if with_bf16 else None)
        assert int(step.item()) == int(step2.item()) == rstep == 4 + (1 - skip)
        if with_bf16:
            assert np.array_equal(to_host_bits(amax).view(np.uint32), ram.view(np.uint32))
            assert np.array_equal(to_host_bits(amax2).view(np.uint32), ram.view(np.uint32))
        for i in range(n):
            for got, ref in ((P[i], rp[i]), (M[i], rm[i]), (V[i], rv[i])):
                assert np.array_equal(to_host_bits(got).view(np.uint32), ref.view(np.uint32)), i
            for got, other in ((P[i], P2[i]), (M[i], M2[i]), (V[i], V2[i])):
                assert torch.equal(got.view(torch.int32), other.view(torch.int32)), i
            if with_bf16:
                assert np.array_equal(to_host_bits(B[i]), rb[i]), i
                assert torch.equal(B[i].view(torch.int16), B2[i].view(torch.int16)), i
            if skip:   # nothing written on a skipped step
                assert np.array_equal(to_host_bits(P[i]).view(np.uint32),
                                      master_h[i].view(np.uint32)), i
        for L in lists + ([LB] if LB else []):
            L.close()


def test_noalloc_empty_list_and_capture_refusal(A):
    """An empty parameter list only advances the step counter (as the
    handle-based call does); a call on a stream that is capturing a graph is
    refused with AMP_EINVAL and enqueues nothing, and the capture survives."""
    dev = torch.device("cuda:0")
    fi = torch.zeros(1, dtype=torch.int32, device=dev)
    step = torch.zeros(1, dtype=torch.int32, device=dev)
    A.amp_adamw_master_step_noalloc([], [], [], [], None, None, fi, step, *HYPER)
    torch.cuda.synchronize()
    assert int(step.item()) == 1
    A.amp_noalloc_check()

    p, m, v, b = _state(dev, [300], 3)
    g = [torch.zeros(300, dtype=torch.float16, device=dev)]
    before = p[0].clone()
    s = torch.cuda.Stream(device=dev)
    graph = torch.cuda.CUDAGraph()
    err = None
    with torch.cuda.graph(graph, stream=s):
        try:
            A.amp_adamw_master_step_noalloc(p, m, v, g, b, None, fi, step, *HYPER, stream=s)
        except A.AmpError as e:
            err = e
        fi.add_(0)       # some captured work, so the graph is not empty
    assert err is not None and err.status == -1 and "captur" in str(err)
    torch.cuda.synchronize()
    assert torch.equal(p[0], before) and int(step.item()) == 1
    graph.replay()
    torch.cuda.synchronize()
    A.amp_noalloc_check()


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
    numel = (ctypes.c_int64 * 1)(2 ** 63 - 1)           # ceil must not overflow int64
    st = L.amp_adamw_master_step_noalloc(n, ptrs, ptrs, ptrs, ptrs, DT["f32"], None, numel, None,
                                         None, None, P(dummy.data_ptr()), ctypes.byref(h), None,
                                         None)
    assert st == -1 and b"limit" in L.amp_last_error()
