"""The C-ABI library loads, exports every symbol include/ampfp8.h declares,
and rejects invalid arguments with a status before touching the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from loss_scaling_master_gb300 import build as B
    B.build()
    import loss_scaling_master_gb300 as pkg
    return pkg.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "ampfp8.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:amp_status|const char \*|int)\s*\*?\s*(\w+)\s*\(",
                                 src, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) == 29, names
    from loss_scaling_master_gb300._lib import EXPORTS
    assert sorted(EXPORTS) == names
    for n in names:
        assert hasattr(lib, n), n


def test_abi_version(lib):
    assert lib.amp_abi_version() == 11


def test_invalid_arguments_return_status(lib):
    from loss_scaling_master_gb300._lib import DT, amp_adamw_hyper
    EINVAL, EDTYPE = -1, -2
    P = ctypes.c_void_p
    assert lib.amp_unscale_check(None, None, None, 0, None) == EINVAL
    assert b"NULL" in lib.amp_last_error()
    h = amp_adamw_hyper(1e-3, 0.9, 0.999, 1e-8, 0.0)
    assert lib.amp_adamw_master_step(None, None, None, None, None, None, None, None,
                                     ctypes.byref(h), None, None) == EINVAL
    assert lib.amp_update_scale(None, None, None, 2.0, 0.5, 10, None, 0, None) == EINVAL
    assert lib.amp_emit_bf16(None, None, None, None) == EINVAL
    dummy = P(16)
    assert lib.amp_update_scale(dummy, dummy, dummy, 2.0, 0.5, 0, None, 0, None) == EINVAL
    assert lib.amp_update_scale(dummy, dummy, dummy, 2.0, 0.5, 1, None, 3, None) == EINVAL
    # fp8 quant: negative size, bad eps, unsupported dtypes
    assert lib.fp8_quant_tensorwise(dummy, DT["bf16"], -1, 4, DT["e4m3fn"], 1e-12, dummy, None,
                                    dummy, dummy, 0, None, None) == EINVAL
    assert lib.fp8_quant_tensorwise(dummy, DT["bf16"], 4, 4, DT["e4m3fn"], 0.0, dummy, None,
                                    dummy, dummy, 0, None, None) == EINVAL
    assert lib.fp8_quant_tensorwise(dummy, DT["e4m3fn"], 4, 4, DT["e4m3fn"], 1e-12, dummy, None,
                                    dummy, dummy, 0, None, None) == EDTYPE
    assert lib.fp8_quant_tensorwise(dummy, DT["bf16"], 4, 4, DT["f16"], 1e-12, dummy, None,
                                    dummy, dummy, 0, None, None) == EDTYPE
    # list creation: negative n, NULL arrays, negative size, NULL pointer of a non-empty tensor
    out = P()
    assert lib.amp_tensor_list_create(-1, None, None, None, DT["f32"], None, ctypes.byref(out)) == EINVAL
    assert lib.amp_tensor_list_create(1, None, None, None, DT["f32"], None, ctypes.byref(out)) == EINVAL
    ptrs = (P * 1)(None)
    neg = (ctypes.c_int64 * 1)(-5)
    one = (ctypes.c_int64 * 1)(7)
    assert lib.amp_tensor_list_create(1, ptrs, neg, None, DT["f32"], None, ctypes.byref(out)) == EINVAL
    assert lib.amp_tensor_list_create(1, ptrs, one, None, DT["f32"], None, ctypes.byref(out)) == EINVAL
    # shapes past the launch arithmetic: a side >= 2^48, rows * cols past int64
    big = (ctypes.c_int64 * 1)(1 << 48)
    huge = (ctypes.c_int64 * 1)((1 << 40) + 1)
    assert lib.amp_tensor_list_create(1, (P * 1)(dummy), big, None, DT["f32"], None,
                                      ctypes.byref(out)) == EINVAL
    assert lib.amp_tensor_list_create(1, (P * 1)(dummy), huge, huge, DT["f32"], None,
                                      ctypes.byref(out)) == EINVAL
    assert b"too large" in lib.amp_last_error()
    # a shape that passes those limits but whose chunk table would pass 2^31
    # entries fails before the table grows (no host allocation of it)
    vast = (ctypes.c_int64 * 1)(1 << 45)
    assert lib.amp_tensor_list_create(1, (P * 1)(dummy), vast, None, DT["f32"], None,
                                      ctypes.byref(out)) == EINVAL
    assert b"too large" in lib.amp_last_error()
    assert lib.fp8_quant_tensorwise(dummy, DT["bf16"], (1 << 40) + 1, (1 << 40) + 1, DT["e4m3fn"],
                                    1e-12, dummy, None, dummy, dummy, 0, None, None) == EINVAL
    assert lib.fp8_quant_rowwise(dummy, DT["bf16"], 0, 1 << 48, DT["e4m3fn"], 1e-12, dummy, None,
                                 dummy, dummy, dummy, None, None, None, None, None) == EINVAL
    assert lib.amp_tensor_list_create(1, ptrs, one, None, 99, None, ctypes.byref(out)) == EDTYPE
    assert not out.value


def test_binding_rejects_host_tensors_and_bad_buffers():
    """The Python binding checks every buffer it hands to the library (device,
    contiguity, dtype, size) and raises before any call reaches the GPU."""
    import torch

    import loss_scaling_master_gb300 as A
    x = torch.zeros(4, 4, dtype=torch.bfloat16)          # host memory
    q = torch.empty(16, dtype=torch.uint8)
    f = torch.empty(1, dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA"):
        A.fp8_quant_tensorwise(x, "e4m3fn", q, None, f, f)
    with pytest.raises(ValueError, match="CUDA"):
        A.amp_tensor_list_create([torch.zeros(3)])
    with pytest.raises(ValueError, match="CUDA"):
        A.amp_update_scale(f, torch.zeros(1, dtype=torch.int32), torch.zeros(1, dtype=torch.int32),
                           2.0, 0.5, 10)
    with pytest.raises(ValueError, match="contiguous"):
        A.fp8_quant_rowwise(torch.zeros(4, 8, dtype=torch.bfloat16)[:, ::2], "e4m3fn", q, None,
                            f, f, f)


def test_noalloc_binding_rejects_mismatched_lists():
    """The allocation-free AdamW binding hands the library bare pointers, so it
    checks every list against master (count, element counts, dtypes), one
    gradient dtype, and that amax holds every named slot, before any call."""
    import torch

    import loss_scaling_master_gb300 as A
    sizes = [5, 17]
    f32 = lambda: [torch.zeros(k) for k in sizes]
    g16 = [torch.zeros(k, dtype=torch.float16) for k in sizes]
    b16 = [torch.zeros(k, dtype=torch.bfloat16) for k in sizes]
    hyper = (1e-3, 0.9, 0.999, 1e-8, 0.0)
    i32 = torch.zeros(1, dtype=torch.int32)

    def call(master=None, m=None, v=None, g=None, b="default", **kw):
        A.amp_adamw_master_step_noalloc(master or f32(), m or f32(), v or f32(), g or g16,
                                        b16 if b == "default" else b, None, i32, i32, *hyper,
                                        **kw)

    with pytest.raises(ValueError, match="exp_avg: 1 tensors"):
        call(m=[torch.zeros(5)])
    with pytest.raises(ValueError, match=r"exp_avg_sq\[1\]: 16 elements"):
        call(v=[torch.zeros(5), torch.zeros(16)])
    with pytest.raises(ValueError, match=r"grads\[0\]: 4 elements"):
        call(g=[torch.zeros(4, dtype=torch.float16), g16[1]])
    with pytest.raises(ValueError, match=r"bf16_out\[1\]: 3 elements"):
        call(b=[b16[0], torch.zeros(3, dtype=torch.bfloat16)])
    with pytest.raises(ValueError, match=r"exp_avg\[0\]: dtype"):
        call(m=[torch.zeros(5, dtype=torch.float64), torch.zeros(17)])
    with pytest.raises(ValueError, match=r"bf16_out\[0\]: dtype"):
        call(b=[torch.zeros(5, dtype=torch.float16), b16[1]])
    with pytest.raises(ValueError, match=r"grads\[1\]: dtype"):
        call(g=[g16[0], torch.zeros(17, dtype=torch.int16)])
    with pytest.raises(ValueError, match="mixed dtypes"):
        call(g=[g16[0], torch.zeros(17, dtype=torch.bfloat16)])
    with pytest.raises(ValueError, match="amax_slots: 1 entries"):
        call(amax_slots=[0], amax=torch.zeros(2))
    with pytest.raises(ValueError, match="slot 2; amax holds 2"):
        call(amax_slots=[0, 2], amax=torch.zeros(2))
    with pytest.raises(ValueError, match="slot 0; amax holds 0"):
        call(amax_slots=[0, -1])
    with pytest.raises(ValueError, match="CUDA"):        # well-formed lists, host memory
        call(amax_slots=[0, 1], amax=torch.zeros(2))
