"""The C-ABI library on the CPU: it loads, exports every declared entry point,
and rejects bad arguments before touching a GPU."""
import ctypes

import numpy as np
import pytest

from verify_matvec_gb300 import build, cbq


@pytest.fixture(scope="module")
def lib():
    build.build()
    return cbq.load()


def test_every_header_function_is_exported(lib):
    names = cbq.header_functions()
    assert len(names) >= 19
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(cbq._SIGS), "binding and header disagree"


def test_status_strings(lib):
    for st in (0, -1, -2, -3, -4):
        assert lib.cbq_status_string(st).decode().startswith("CBQ_")
    assert b"unknown" in lib.cbq_status_string(7)


def test_argument_errors_need_no_gpu(lib):
    P = ctypes.c_void_p
    dummy = P(16)
    h = ctypes.c_void_p()
    EINVAL = cbq.CBQ_EINVAL
    # bad shapes / null pointers are rejected before any CUDA call
    assert lib.cbq_weights_create(None, 4, 64, 0, None, ctypes.byref(h)) == EINVAL
    assert lib.cbq_weights_create(dummy, 4, 48, 0, None, ctypes.byref(h)) == EINVAL
    assert lib.cbq_weights_create(dummy, 0, 64, 0, None, ctypes.byref(h)) == EINVAL
    assert lib.cbq_weights_create(dummy, 4, 64, 0, None, None) == EINVAL
    assert lib.cbq_quantize_act(None, 64, 1, dummy, dummy, None) == EINVAL
    assert lib.cbq_quantize_act(dummy, 40, 1, dummy, dummy, None) == EINVAL
    assert lib.cbq_quantize_act(dummy, 64, 0, dummy, dummy, None) == EINVAL
    assert lib.cbq_matvec(None, dummy, 1, dummy, None) == EINVAL
    assert lib.cbq_matvec_q(None, dummy, dummy, 1, dummy, None) == EINVAL
    assert lib.cbq_moe_create(dummy, dummy, 0, 64, 64, 0, None, ctypes.byref(h)) == EINVAL
    assert lib.cbq_moe_create(dummy, dummy, 4, 60, 64, 0, None, ctypes.byref(h)) == EINVAL
    assert lib.cbq_moe_create(dummy, dummy, 1, (1 << 20) + 32, 64, 0, None, ctypes.byref(h)) == EINVAL  # H cap
    assert lib.cbq_moe_create(dummy, dummy, 1, 64, (1 << 20) + 32, 0, None, ctypes.byref(h)) == EINVAL  # F cap
    assert lib.cbq_moe_matvec(None, dummy, 1, dummy, dummy, 1, 1, dummy, None) == EINVAL
    assert lib.cbq_weights_destroy(None) == EINVAL
    assert lib.cbq_moe_destroy(None) == EINVAL
    assert lib.cbq_weights_get_error(None, None, ctypes.byref(ctypes.c_uint())) == EINVAL
    assert lib.cbq_moe_get_error(None, None, ctypes.byref(ctypes.c_uint())) == EINVAL
    assert lib.cbq_weights_get_error(dummy, None, None) == EINVAL                            # no output word
    assert lib.cbq_moe_get_error(dummy, None, None) == EINVAL
    assert lib.cbq_moe_debug_stall(None, 1) == EINVAL
    assert lib.cbq_moe_set_shared(None, dummy, dummy, 0, None) == EINVAL
    assert lib.cbq_moe_set_shared(None, None, None, 0, None) == EINVAL
    assert lib.cbq_router_topk(None, 1, 8, 2, dummy, dummy, None) == EINVAL
    assert lib.cbq_router_topk(dummy, 1, 0, 1, dummy, dummy, None) == EINVAL                      # E < 1
    assert lib.cbq_router_topk(dummy, 1, 4, 5, dummy, dummy, None) == EINVAL                      # topk > E
    assert lib.cbq_router_topk(dummy, 1, cbq.CBQ_ROUTER_MAX_E + 1, 2, dummy, dummy, None) == EINVAL
    assert lib.cbq_router_topk(dummy, 0, 8, 2, dummy, dummy, None) == EINVAL                      # no token
    assert lib.cbq_moe_matvec_logits(None, dummy, 1, dummy, 2, 1, dummy, None) == EINVAL
    assert lib.cbq_matmat(None, dummy, 8, dummy, None) == EINVAL
    assert lib.cbq_debug_mmq_block_dots(None, dummy, 8, dummy, None) == EINVAL
    aligned = ctypes.c_void_p(0x1000)
    assert lib.cbq_quantize_weights(None, 4, 64, aligned, None) == EINVAL                      # no weights
    assert lib.cbq_quantize_weights(aligned, 4, 64, None, None) == EINVAL                      # no output
    assert lib.cbq_quantize_weights(aligned, 0, 64, aligned, None) == EINVAL                   # M < 1
    assert lib.cbq_quantize_weights(aligned, 4, 48, aligned, None) == EINVAL                   # K % 32
    assert lib.cbq_quantize_weights(aligned, 4, 0, aligned, None) == EINVAL                    # K < 32
    assert lib.cbq_quantize_weights(ctypes.c_void_p(0x1004), 4, 64, aligned, None) == EINVAL  # w not 16-aligned
    assert lib.cbq_quantize_weights(aligned, 4, 64, ctypes.c_void_p(0x1001), None) == EINVAL  # odd output
    assert lib.cbq_debug_mmq_stall(None, 1) == EINVAL
    far = ctypes.c_void_p(0x100000)
    assert lib.cbq_hc_sinkhorn(None, 4, 20, far, None) == EINVAL                               # no logits
    assert lib.cbq_hc_sinkhorn(aligned, 4, 20, None, None) == EINVAL                           # no output
    assert lib.cbq_hc_sinkhorn(aligned, 0, 20, far, None) == EINVAL                            # n < 1
    assert lib.cbq_hc_sinkhorn(aligned, cbq.CBQ_HC_MAX_N + 1, 20, far, None) == EINVAL         # n too large
    assert lib.cbq_hc_sinkhorn(aligned, 4, -1, far, None) == EINVAL                            # iters < 0
    assert lib.cbq_hc_sinkhorn(aligned, 4, cbq.CBQ_HC_MAX_ITERS + 1, far, None) == EINVAL      # too many rounds
    assert lib.cbq_hc_sinkhorn(ctypes.c_void_p(0x1008), 4, 20, far, None) == EINVAL            # not 16-aligned
    assert lib.cbq_hc_sinkhorn(aligned, 4, 20, ctypes.c_void_p(0x1040), None) == EINVAL        # overlaps, not in place


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(cbq, "_lib", None)
    monkeypatch.setattr(cbq, "LIB_PATH", str(tmp_path / "libcbq.so"))
    with pytest.raises(ImportError):
        cbq.load()
