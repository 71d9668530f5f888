"""The C ABI without a GPU: the library builds, loads and exports every entry point declared in
include/drafthead.h, and rejects bad arguments on the host before any CUDA call.

Every call below fails validation, so no kernel is launched and no pointer is dereferenced
(the fake addresses are never touched).
"""
import ctypes
import os
import re

import pytest

from bit_draft_lm_gb300 import build as dh_build
from bit_draft_lm_gb300 import drafthead as dh

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "drafthead.h")

A16 = 0x10000          # fake, 16-byte aligned address (never dereferenced)
A256 = 0x20000


@pytest.fixture(scope="module")
def lib():
    dh_build.build()
    return dh.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dh_\w+)\s*\(", text)))


def test_header_symbols_exported(lib):
    names = _declared()
    assert "dh_draft_head_coarse_topk" in names and "dh_quantize_pack_int2" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(dh.SIGNATURES), "binding and header disagree"


def test_packed_bytes_page_shape(lib):
    assert dh.dh_packed_bytes(124160, 5120, 128, 2) == 178_790_400
    assert dh.dh_packed_bytes(124160, 5120, 64, 2) == 158_924_800 + 2 * 124160 * 80 * 2
    assert dh.dh_packed_bytes(124160, 5120, 128, 4) == 124160 * 2560 + 2 * 124160 * 40 * 2
    assert dh.dh_packed_bytes(10, 100, 128, 2) == 0
    assert dh.dh_packed_bytes(10, 1024, 96, 2) == 0
    assert dh.dh_workspace_bytes(8, 124160, 5120, 8, 16) >= 256


def _quant(lib, W=A16, N=64, K=1024, G=128, packed=A16, S=A16, ZS=A16, bits=2):
    f = lib.dh_quantize_pack_int2 if bits == 2 else lib.dh_quantize_pack_int4
    return f(W, N, K, G, packed, S, ZS, None)


def test_quantize_validation(lib):
    assert _quant(lib, W=None) == dh.DH_ERR_NULL
    assert "NULL" in dh.dh_last_error()
    assert _quant(lib, G=96) == dh.DH_ERR_PARAM
    assert _quant(lib, K=1000) == dh.DH_ERR_SHAPE
    assert _quant(lib, K=256 + 512) == dh.DH_ERR_SHAPE          # not a multiple of 4*G
    assert _quant(lib, K=640, bits=4) == dh.DH_ERR_SHAPE         # int4 needs K % (2G)
    assert _quant(lib, N=0) == dh.DH_ERR_SHAPE
    assert _quant(lib, W=A16 + 2) == dh.DH_ERR_ALIGN


def _coarse(lib, x=A16, M=1, K=1024, packed=A16, S=A16, ZS=A16, N=8192, G=128, bits=2,
            kcand=8, cv=A16, ci=A16, y=None, ws=A256, wsb=256):
    return lib.dh_draft_head_coarse_topk(x, M, K, packed, S, ZS, N, G, bits, kcand, cv, ci, y, ws,
                                         wsb, None)


def test_coarse_validation(lib):
    assert _coarse(lib, x=None) == dh.DH_ERR_NULL
    assert _coarse(lib, cv=None) == dh.DH_ERR_NULL
    assert _coarse(lib, bits=3) == dh.DH_ERR_PARAM
    assert _coarse(lib, G=32) == dh.DH_ERR_PARAM
    assert _coarse(lib, kcand=0) == dh.DH_ERR_PARAM
    assert _coarse(lib, kcand=65) == dh.DH_ERR_PARAM
    assert _coarse(lib, M=0) == dh.DH_ERR_SHAPE
    assert _coarse(lib, M=5000) == dh.DH_ERR_SHAPE
    assert _coarse(lib, N=0) == dh.DH_ERR_SHAPE
    assert _coarse(lib, K=1536) == dh.DH_ERR_SHAPE              # not a multiple of 8*G
    assert _coarse(lib, K=6144) == dh.DH_ERR_SHAPE              # above the supported K
    assert _coarse(lib, x=A16 + 8) == dh.DH_ERR_ALIGN
    assert _coarse(lib, packed=A16 + 4) == dh.DH_ERR_ALIGN
    assert _coarse(lib, cv=A16 + 2) == dh.DH_ERR_ALIGN
    assert _coarse(lib, ws=None) == dh.DH_ERR_WORKSPACE
    assert _coarse(lib, ws=A256 + 64) == dh.DH_ERR_WORKSPACE
    assert _coarse(lib, wsb=16) == dh.DH_ERR_WORKSPACE
    assert "workspace" in dh.dh_last_error()


def _rerank(lib, x=A16, M=1, K=1024, W=A16, N=8192, cv=A16, ci=A16, ncand=1024, R=16, rr=A16,
            rl=A16, am=A16, y=None, ws=A256, wsb=256):
    return lib.dh_draft_head_rerank_argmax(x, M, K, W, N, cv, ci, ncand, R, rr, rl, am, y, ws,
                                           wsb, None)


def test_rerank_validation(lib):
    assert _rerank(lib, W=None) == dh.DH_ERR_NULL
    assert _rerank(lib, am=None) == dh.DH_ERR_NULL
    assert _rerank(lib, R=0) == dh.DH_ERR_PARAM
    assert _rerank(lib, R=257) == dh.DH_ERR_PARAM
    assert _rerank(lib, ncand=8, R=16) == dh.DH_ERR_SHAPE        # rerank > ncand
    assert _rerank(lib, K=1001) == dh.DH_ERR_SHAPE
    assert _rerank(lib, M=0) == dh.DH_ERR_SHAPE
    assert _rerank(lib, W=A16 + 8) == dh.DH_ERR_ALIGN
    assert _rerank(lib, rr=A16 + 1) == dh.DH_ERR_ALIGN
    assert _rerank(lib, wsb=0) == dh.DH_ERR_WORKSPACE


def test_status_validation(lib):
    word = ctypes.c_uint32(0)
    assert lib.dh_workspace_status(None, 256, ctypes.addressof(word), None) == dh.DH_ERR_NULL
    assert lib.dh_workspace_status(A256, 0, ctypes.addressof(word), None) == dh.DH_ERR_WORKSPACE


def test_last_error_cleared_by_success_path_message(lib):
    _coarse(lib, G=7)
    assert "G=7" in dh.dh_last_error()


def test_workspace_bytes_sizes(lib):
    """Up to 16 hidden rows the workspace is the 256-byte header; beyond, the tensor-core pass
    keeps its scratch after it: x as the MMA operand (80 x K x 2 B), group sums (80 x K/64 x 4 B)
    and exponents (80 x 4 B), each rounded up to 256 B."""
    assert dh.dh_workspace_bytes(1, 124160, 5120, 8, 16) == 256
    assert dh.dh_workspace_bytes(16, 124160, 5120, 8, 16) == 256
    r = lambda v: (v + 255) // 256 * 256
    assert dh.dh_workspace_bytes(72, 124160, 5120, 8, 16) == \
        256 + r(80 * 5120 * 2) + r(80 * 80 * 4) + r(80 * 4) + r(256 * 128 * 80 * 4)
    assert dh.dh_workspace_bytes(0, 124160, 5120, 8, 16) == 0


def test_fp8_and_topk_validation(lib):
    f = lib.dh_quantize_pack_int2_fp8
    assert f(A16, None, 64, 1024, 128, A16, A16, A16, None) == dh.DH_ERR_NULL
    assert f(None, A16, 64, 1024, 128, A16, A16, A16, None) == dh.DH_ERR_NULL
    assert f(A16, A16, 64, 1000, 128, A16, A16, A16, None) == dh.DH_ERR_SHAPE
    assert f(A16, A16 + 2, 64, 1024, 128, A16, A16, A16, None) == dh.DH_ERR_ALIGN
    g = lib.dh_draft_head_rerank_argmax_fp8
    args = [A16, 1, 1024, A16, A16, 8192, A16, A16, 1024, 16, A16, A16, A16, None, A256, 256, None]
    bad = list(args); bad[3] = None
    assert g(*bad) == dh.DH_ERR_NULL
    bad = list(args); bad[4] = None
    assert g(*bad) == dh.DH_ERR_NULL
    bad = list(args); bad[9] = 0
    assert g(*bad) == dh.DH_ERR_PARAM
    bad = list(args); bad[3] = A16 + 8
    assert g(*bad) == dh.DH_ERR_ALIGN
    t = lib.dh_topk_only_logits
    assert t(None, A16, 1, 16, 8192, A16, None) == dh.DH_ERR_NULL
    assert t(A16, A16, 0, 16, 8192, A16, None) == dh.DH_ERR_SHAPE
    assert t(A16, A16, 1, 0, 8192, A16, None) == dh.DH_ERR_SHAPE
    assert t(A16 + 2, A16, 1, 16, 8192, A16, None) == dh.DH_ERR_ALIGN


def test_host_call_validation(lib):
    h = lib.dh_draft_head_host
    args = [A16, 1, 1024, A16, A16, A16, A16, A16, 8192, 128, 2, 8, 16, A16, A16, A16, A16, A16,
            A16, A16, A16, A256, 256, None]
    bad = list(args); bad[0] = None
    assert h(*bad) == dh.DH_ERR_NULL
    bad = list(args); bad[18] = None
    assert h(*bad) == dh.DH_ERR_NULL
    bad = list(args); bad[1] = 0
    assert h(*bad) == dh.DH_ERR_SHAPE
    bad = list(args); bad[12] = 300
    assert h(*bad) == dh.DH_ERR_SHAPE
    bad = list(args); bad[3] = A16 + 4
    assert h(*bad) == dh.DH_ERR_ALIGN


def test_argmax_call_validation(lib):
    """dh_draft_head_argmax rejects bad arguments before anything is launched (every case here
    fails validation: the addresses are not real device memory)."""
    f = lib.dh_draft_head_argmax
    args = [A16, 1, 1024, A16, A16, A16, A16, 8192, 128, 2, 8, 16, A16, A16, A16, A16, A16, None,
            A256, 256, None]
    bad = list(args); bad[6] = None      # W
    assert f(*bad) == dh.DH_ERR_NULL
    bad = list(args); bad[3] = None      # packed
    assert f(*bad) == dh.DH_ERR_NULL
    bad = list(args); bad[11] = 0        # rerank
    assert f(*bad) == dh.DH_ERR_PARAM
    bad = list(args); bad[9] = 3         # bits
    assert f(*bad) == dh.DH_ERR_PARAM
    bad = list(args); bad[6] = A16 + 2   # W misaligned
    assert f(*bad) == dh.DH_ERR_ALIGN
    bad = list(args); bad[19] = 128      # smaller than the 256-byte header
    assert f(*bad) == dh.DH_ERR_WORKSPACE


def test_host_plan_validation(lib):
    """dh_host_plan_create rejects bad arguments before any CUDA call and leaves *plan NULL;
    dh_host_plan_run rejects a NULL plan; dh_host_plan_destroy ignores NULL."""
    f = lib.dh_host_plan_create
    args = [A16, 1, 1024, A16, A16, A16, A16, A16, 8192, 128, 2, 8, 16, A16, A16, A16, A16, A16,
            A16, A16, A16, A256, 256]
    plan = ctypes.c_void_p(0x1234)
    bad = list(args); bad[0] = None      # x_host
    assert f(*bad, ctypes.byref(plan)) == dh.DH_ERR_NULL and plan.value is None
    assert f(*args, None) == dh.DH_ERR_NULL
    bad = list(args); bad[18] = None     # argmax_host
    assert f(*bad, ctypes.byref(plan)) == dh.DH_ERR_NULL
    bad = list(args); bad[1] = 0         # M
    assert f(*bad, ctypes.byref(plan)) == dh.DH_ERR_SHAPE
    bad = list(args); bad[12] = 300      # rerank
    assert f(*bad, ctypes.byref(plan)) == dh.DH_ERR_SHAPE
    bad = list(args); bad[3] = A16 + 4   # x_dev misaligned
    assert f(*bad, ctypes.byref(plan)) == dh.DH_ERR_ALIGN
    assert lib.dh_host_plan_run(None, None) == dh.DH_ERR_NULL
    lib.dh_host_plan_destroy(None)


def test_binding_rejects_host_tensors_and_bad_dtypes(lib):
    """The Python binding refuses CPU tensors, non-bf16 inputs and mis-shaped outputs before it
    calls into the library (the CPU-tensor guard of the page's plug-in tests)."""
    import torch
    x = torch.zeros(1, 1024, dtype=torch.bfloat16)
    W = torch.zeros(8192, 1024, dtype=torch.bfloat16)
    packed = torch.zeros(8192, 256, dtype=torch.uint8)
    S = torch.zeros(8192, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        dh.dh_draft_head_coarse_topk(x, packed, S, S, 8192)
    with pytest.raises(ValueError, match="CUDA tensor"):
        dh.dh_draft_head_argmax(x, packed, S, S, W)
    cv = torch.zeros(1, 1024, dtype=torch.float32)
    ci = torch.zeros(1, 1024, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        dh.dh_draft_head_rerank_argmax(x, W, cv, ci, 16)
    with pytest.raises(ValueError, match="bf16"):
        dh.dh_draft_head_rerank_argmax(x.float(), W, cv, ci, 16)
    with pytest.raises(ValueError, match="bf16"):
        dh.dh_quantize_pack_int2(W.float())
