"""Python binding of the C ABI in include/drafthead.h (argument marshalling only).

Every function here has the name of the C entry point it calls, takes torch CUDA tensors for
the device buffers, checks dtype / shape / contiguity, and passes raw pointers and the current
CUDA stream to libdrafthead.so. PyTorch provides device memory and streams; every step of the
draft head runs in the library's CUDA kernels. If the library has not been built the binding
raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdrafthead.so")

DH_OK = 0
DH_ERR_NULL = -1
DH_ERR_SHAPE = -2
DH_ERR_ALIGN = -3
DH_ERR_PARAM = -4
DH_ERR_WORKSPACE = -5
DH_ERR_CUDA = -6
DH_ERR_DEVICE = -7
DH_DEV_WAIT_TIMEOUT = 0x1
DH_DEV_BAD_ID = 0x2
BLOCK_ROWS = 64

# C entry points and their argument types, in header order.
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
_SZ = ctypes.c_size_t
SIGNATURES = {
    "dh_quantize_pack_int2": ([_P, _I64, _I64, _I, _P, _P, _P, _P], _I),
    "dh_quantize_pack_int4": ([_P, _I64, _I64, _I, _P, _P, _P, _P], _I),
    "dh_packed_bytes": ([_I64, _I64, _I, _I], _SZ),
    "dh_workspace_bytes": ([_I64, _I64, _I64, _I, _I], _SZ),
    "dh_draft_head_coarse_topk": ([_P, _I64, _I64, _P, _P, _P, _I64, _I, _I, _I, _P, _P, _P, _P,
                                   _SZ, _P], _I),
    "dh_draft_head_rerank_argmax": ([_P, _I64, _I64, _P, _I64, _P, _P, _I64, _I, _P, _P, _P, _P,
                                     _P, _SZ, _P], _I),
    "dh_draft_head_argmax": ([_P, _I64, _I64, _P, _P, _P, _P, _I64, _I, _I, _I, _I, _P, _P, _P,
                              _P, _P, _P, _P, _SZ, _P], _I),
    "dh_draft_head_rerank_argmax_noalloc": ([_P, _I64, _I64, _P, _I64, _P, _P, _I64, _I, _P,
                                             _P, _P, _P, _P], _I),
    "dh_draft_head_host": ([_P, _I64, _I64, _P, _P, _P, _P, _P, _I64, _I, _I, _I, _I, _P, _P, _P,
                            _P, _P, _P, _P, _P, _P, _SZ, _P], _I),
    "dh_host_plan_create": ([_P, _I64, _I64, _P, _P, _P, _P, _P, _I64, _I, _I, _I, _I, _P, _P,
                             _P, _P, _P, _P, _P, _P, _P, _SZ, _P], _I),
    "dh_host_plan_run": ([_P, _P], _I),
    "dh_host_plan_destroy": ([_P], None),
    "dh_topk_only_logits": ([_P, _P, _I64, _I, _I64, _P, _P], _I),
    "dh_quantize_pack_int2_fp8": ([_P, _P, _I64, _I64, _I, _P, _P, _P, _P], _I),
    "dh_draft_head_rerank_argmax_fp8": ([_P, _I64, _I64, _P, _P, _I64, _P, _P, _I64, _I, _P, _P,
                                         _P, _P, _P, _SZ, _P], _I),
    "dh_argmax_shard_keys": ([_P, _P, _I64, _I, _I64, _P, _P], _I),
    "dh_argmax_merge": ([_P, _I, _I64, _P, _P, _P], _I),
    "dh_argmax_shard_keys_host": ([_P, _P, _I64, _I, _I64, _P], _I),
    "dh_argmax_merge_host": ([_P, _I, _I64, _P, _P], _I),
    "dh_workspace_status": ([_P, _SZ, _P, _P], _I),
    "dh_last_error": ([], ctypes.c_char_p),
}

_lib = None


class DraftHeadError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"status {status}: {message}")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m bit_draft_lm_gb300.build` (nvcc, sm_103a)")
        h = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            f = getattr(h, name)
            f.argtypes = args
            f.restype = res
        _lib = h
    return _lib


def dh_last_error() -> str:
    return lib().dh_last_error().decode()


def _check(rc: int):
    if rc != DH_OK:
        raise DraftHeadError(rc, dh_last_error())


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dev(t: Optional[torch.Tensor], name: str, dtype, shape=None) -> int:
    if t is None:
        return 0
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t.data_ptr()


def _bf16(t: torch.Tensor, name: str) -> torch.Tensor:
    if t.dtype in (torch.int16, torch.uint16):
        return t.view(torch.bfloat16)
    if t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must hold bf16 values (torch.bfloat16), got {t.dtype}")
    return t


def dh_packed_bytes(N: int, K: int, G: int, bits: int) -> int:
    return int(lib().dh_packed_bytes(N, K, G, bits))


def dh_workspace_bytes(M: int, N: int, K: int, kcand: int, rerank: int) -> int:
    return int(lib().dh_workspace_bytes(M, N, K, kcand, rerank))


def new_workspace(M: int, N: int, K: int, kcand: int, rerank: int,
                  device="cuda") -> torch.Tensor:
    """A zero-filled workspace for these sizes (the caching allocator aligns to 512 bytes)."""
    n = dh_workspace_bytes(M, N, K, kcand, rerank)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def _quantize(fn, bits, W, G, packed, S, ZS, stream):
    W = _bf16(W, "W")
    N, K = W.shape
    per = 8 // bits
    dev = W.device
    if packed is None:
        packed = torch.empty(N, K // per, dtype=torch.uint8, device=dev)
    if S is None:
        S = torch.empty(N, K // G, dtype=torch.bfloat16, device=dev)
    if ZS is None:
        ZS = torch.empty(N, K // G, dtype=torch.bfloat16, device=dev)
    S, ZS = _bf16(S, "S"), _bf16(ZS, "ZS")
    _check(fn(_dev(W, "W", torch.bfloat16), N, K, G,
              _dev(packed, "packed", torch.uint8, (N, K // per)),
              _dev(S, "S", torch.bfloat16, (N, K // G)), _dev(ZS, "ZS", torch.bfloat16, (N, K // G)),
              _stream(stream)))
    return packed, S, ZS


def dh_quantize_pack_int2(W: torch.Tensor, G: int = 128, packed=None, S=None, ZS=None,
                          stream=None) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    return _quantize(lib().dh_quantize_pack_int2, 2, W, G, packed, S, ZS, stream)


def dh_quantize_pack_int4(W: torch.Tensor, G: int = 128, packed=None, S=None, ZS=None,
                          stream=None) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    return _quantize(lib().dh_quantize_pack_int4, 4, W, G, packed, S, ZS, stream)


def dh_draft_head_coarse_topk(x: torch.Tensor, packed: torch.Tensor, S: torch.Tensor,
                              ZS: torch.Tensor, N: int, G: int = 128, bits: int = 2,
                              kcand: int = 8, cand_val=None, cand_id=None, y_coarse=None,
                              workspace=None, stream=None):
    """-> (cand_val f32 [M, nblk*kcand], cand_id i32 [M, nblk*kcand])."""
    x = _bf16(x, "x")
    M, K = x.shape
    nblk = (N + BLOCK_ROWS - 1) // BLOCK_ROWS
    dev = x.device
    if cand_val is None:
        cand_val = torch.empty(M, nblk * kcand, dtype=torch.float32, device=dev)
    if cand_id is None:
        cand_id = torch.empty(M, nblk * kcand, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = new_workspace(M, N, K, kcand, 1, dev)
    if y_coarse is not None:
        y_coarse = _bf16(y_coarse, "y_coarse")
    _check(lib().dh_draft_head_coarse_topk(
        _dev(x, "x", torch.bfloat16), M, K, _dev(packed, "packed", torch.uint8),
        _dev(_bf16(S, "S"), "S", torch.bfloat16), _dev(_bf16(ZS, "ZS"), "ZS", torch.bfloat16),
        N, G, bits, kcand,
        _dev(cand_val, "cand_val", torch.float32, (M, nblk * kcand)),
        _dev(cand_id, "cand_id", torch.int32, (M, nblk * kcand)),
        _dev(y_coarse, "y_coarse", torch.bfloat16, (M, N)),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream)))
    return cand_val, cand_id


def dh_draft_head_rerank_argmax(x: torch.Tensor, W: torch.Tensor, cand_val: torch.Tensor,
                                cand_id: torch.Tensor, rerank: int = 16, rr_id=None,
                                rr_logit=None, argmax_id=None, y_coarse=None, workspace=None,
                                stream=None):
    """-> (rr_id i32 [M, R], rr_logit f32 [M, R], argmax_id i32 [M])."""
    x = _bf16(x, "x")
    W = _bf16(W, "W")
    M, K = x.shape
    N = W.shape[0]
    ncand = cand_val.shape[1]
    dev = x.device
    if rr_id is None:
        rr_id = torch.empty(M, rerank, dtype=torch.int32, device=dev)
    if rr_logit is None:
        rr_logit = torch.empty(M, rerank, dtype=torch.float32, device=dev)
    if argmax_id is None:
        argmax_id = torch.empty(M, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = new_workspace(M, N, K, 1, rerank, dev)
    if y_coarse is not None:
        y_coarse = _bf16(y_coarse, "y_coarse")
    _check(lib().dh_draft_head_rerank_argmax(
        _dev(x, "x", torch.bfloat16), M, K, _dev(W, "W", torch.bfloat16, (N, K)), N,
        _dev(cand_val, "cand_val", torch.float32, (M, ncand)),
        _dev(cand_id, "cand_id", torch.int32, (M, ncand)), ncand, rerank,
        _dev(rr_id, "rr_id", torch.int32, (M, rerank)),
        _dev(rr_logit, "rr_logit", torch.float32, (M, rerank)),
        _dev(argmax_id, "argmax_id", torch.int32, (M,)),
        _dev(y_coarse, "y_coarse", torch.bfloat16, (M, N)),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream)))
    return rr_id, rr_logit, argmax_id


def dh_draft_head_argmax(x: torch.Tensor, packed: torch.Tensor, S: torch.Tensor,
                         ZS: torch.Tensor, W: torch.Tensor, G: int = 128, bits: int = 2,
                         kcand: int = 8, rerank: int = 16, cand_val=None, cand_id=None,
                         rr_id=None, rr_logit=None, argmax_id=None, y_coarse=None,
                         workspace=None, stream=None):
    """Coarse pass, global top-R, exact rerank and argmax in one call (the coarse and rerank
    kernels, validated together). -> (rr_id i32 [M, R], rr_logit f32 [M, R], argmax_id i32 [M],
    cand_val, cand_id)."""
    x = _bf16(x, "x")
    W = _bf16(W, "W")
    M, K = x.shape
    N = W.shape[0]
    nblk = (N + BLOCK_ROWS - 1) // BLOCK_ROWS
    dev = x.device
    if cand_val is None:
        cand_val = torch.empty(M, nblk * kcand, dtype=torch.float32, device=dev)
    if cand_id is None:
        cand_id = torch.empty(M, nblk * kcand, dtype=torch.int32, device=dev)
    if rr_id is None:
        rr_id = torch.empty(M, rerank, dtype=torch.int32, device=dev)
    if rr_logit is None:
        rr_logit = torch.empty(M, rerank, dtype=torch.float32, device=dev)
    if argmax_id is None:
        argmax_id = torch.empty(M, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = new_workspace(M, N, K, kcand, rerank, dev)
    if y_coarse is not None:
        y_coarse = _bf16(y_coarse, "y_coarse")
    _check(lib().dh_draft_head_argmax(
        _dev(x, "x", torch.bfloat16), M, K, _dev(packed, "packed", torch.uint8),
        _dev(_bf16(S, "S"), "S", torch.bfloat16), _dev(_bf16(ZS, "ZS"), "ZS", torch.bfloat16),
        _dev(W, "W", torch.bfloat16, (N, K)), N, G, bits, kcand, rerank,
        _dev(cand_val, "cand_val", torch.float32, (M, nblk * kcand)),
        _dev(cand_id, "cand_id", torch.int32, (M, nblk * kcand)),
        _dev(rr_id, "rr_id", torch.int32, (M, rerank)),
        _dev(rr_logit, "rr_logit", torch.float32, (M, rerank)),
        _dev(argmax_id, "argmax_id", torch.int32, (M,)),
        _dev(y_coarse, "y_coarse", torch.bfloat16, (M, N)),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream)))
    return rr_id, rr_logit, argmax_id, cand_val, cand_id


def dh_draft_head_rerank_argmax_noalloc(x: torch.Tensor, W: torch.Tensor,
                                        cand_val: torch.Tensor, cand_id: torch.Tensor,
                                        rerank: int = 16, rr_id=None, rr_logit=None,
                                        argmax_id=None, y_coarse=None, stream=None):
    """dh_draft_head_rerank_argmax without a workspace: the library's fixed device scratch is
    used instead (for callers that cannot allocate). Outputs are allocated here only when not
    given. -> (rr_id i32 [M, R], rr_logit f32 [M, R], argmax_id i32 [M])."""
    x = _bf16(x, "x")
    W = _bf16(W, "W")
    M, K = x.shape
    N = W.shape[0]
    ncand = cand_val.shape[1]
    dev = x.device
    if rr_id is None:
        rr_id = torch.empty(M, rerank, dtype=torch.int32, device=dev)
    if rr_logit is None:
        rr_logit = torch.empty(M, rerank, dtype=torch.float32, device=dev)
    if argmax_id is None:
        argmax_id = torch.empty(M, dtype=torch.int32, device=dev)
    if y_coarse is not None:
        y_coarse = _bf16(y_coarse, "y_coarse")
    _check(lib().dh_draft_head_rerank_argmax_noalloc(
        _dev(x, "x", torch.bfloat16), M, K, _dev(W, "W", torch.bfloat16, (N, K)), N,
        _dev(cand_val, "cand_val", torch.float32, (M, ncand)),
        _dev(cand_id, "cand_id", torch.int32, (M, ncand)), ncand, rerank,
        _dev(rr_id, "rr_id", torch.int32, (M, rerank)),
        _dev(rr_logit, "rr_logit", torch.float32, (M, rerank)),
        _dev(argmax_id, "argmax_id", torch.int32, (M,)),
        _dev(y_coarse, "y_coarse", torch.bfloat16, (M, N)), _stream(stream)))
    return rr_id, rr_logit, argmax_id


def dh_quantize_pack_int2_fp8(W8: torch.Tensor, row_scale: torch.Tensor, G: int = 128,
                              packed=None, S=None, ZS=None, stream=None):
    """FP8 head (e4m3 rows [N, K] as uint8 or float8_e4m3fn, fp32 per-row scale [N]) ->
    (packed, S, ZS) of the values e4m3 * scale."""
    if W8.dtype == torch.float8_e4m3fn:
        W8 = W8.view(torch.uint8)
    N, K = W8.shape
    dev = W8.device
    if packed is None:
        packed = torch.empty(N, K // 4, dtype=torch.uint8, device=dev)
    if S is None:
        S = torch.empty(N, K // G, dtype=torch.bfloat16, device=dev)
    if ZS is None:
        ZS = torch.empty(N, K // G, dtype=torch.bfloat16, device=dev)
    _check(lib().dh_quantize_pack_int2_fp8(
        _dev(W8, "W8", torch.uint8, (N, K)), _dev(row_scale, "row_scale", torch.float32, (N,)),
        N, K, G, _dev(packed, "packed", torch.uint8, (N, K // 4)),
        _dev(S, "S", torch.bfloat16, (N, K // G)), _dev(ZS, "ZS", torch.bfloat16, (N, K // G)),
        _stream(stream)))
    return packed, S, ZS


def dh_draft_head_rerank_argmax_fp8(x, W8, row_scale, cand_val, cand_id, rerank, rr_id=None,
                                    rr_logit=None, argmax_id=None, y_coarse=None,
                                    workspace=None, stream=None):
    """dh_draft_head_rerank_argmax against e4m3 rows times their per-row scale."""
    if W8.dtype == torch.float8_e4m3fn:
        W8 = W8.view(torch.uint8)
    x = _bf16(x, "x")
    M, K = x.shape
    N = W8.shape[0]
    ncand = cand_val.shape[1]
    dev = x.device
    rr_id = rr_id if rr_id is not None else torch.empty(M, rerank, dtype=torch.int32, device=dev)
    rr_logit = rr_logit if rr_logit is not None else torch.empty(M, rerank, dtype=torch.float32,
                                                                  device=dev)
    argmax_id = argmax_id if argmax_id is not None else torch.empty(M, dtype=torch.int32, device=dev)
    if workspace is None:
        raise ValueError("workspace is required (new_workspace)")
    _check(lib().dh_draft_head_rerank_argmax_fp8(
        _dev(x, "x", torch.bfloat16), M, K, _dev(W8, "W8", torch.uint8, (N, K)),
        _dev(row_scale, "row_scale", torch.float32, (N,)), N,
        _dev(cand_val, "cand_val", torch.float32, (M, ncand)),
        _dev(cand_id, "cand_id", torch.int32, (M, ncand)), ncand, rerank,
        _dev(rr_id, "rr_id", torch.int32, (M, rerank)),
        _dev(rr_logit, "rr_logit", torch.float32, (M, rerank)),
        _dev(argmax_id, "argmax_id", torch.int32, (M,)),
        _dev(y_coarse, "y_coarse", torch.bfloat16, (M, N)),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream)))
    return rr_id, rr_logit, argmax_id


def dh_topk_only_logits(rr_id: torch.Tensor, rr_logit: torch.Tensor, N: int, y=None,
                        stream=None) -> torch.Tensor:
    """bf16 [M, N] logits for a top-K caller: -inf except the reranked entries (their exact
    logit rounded to bf16)."""
    M, R = rr_id.shape
    if y is None:
        y = torch.empty(M, N, dtype=torch.bfloat16, device=rr_id.device)
    _check(lib().dh_topk_only_logits(_dev(rr_id, "rr_id", torch.int32, (M, R)),
                                     _dev(rr_logit, "rr_logit", torch.float32, (M, R)), M, R, N,
                                     _dev(_bf16(y, "y"), "y", torch.bfloat16, (M, N)),
                                     _stream(stream)))
    return y


def _host(t: Optional[torch.Tensor], name: str, dtype, shape=None) -> int:
    if t is None:
        return 0
    if t.is_cuda:
        raise ValueError(f"{name} must be a host tensor")
    if t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t.data_ptr()


def vocab_shard(N: int, world: int, rank: int) -> Tuple[int, int]:
    """Vocab rows [n0, n1) of `rank`'s shard: the ceil(N/64) candidate blocks split as evenly as
    possible in rank order, so that no 64-row block straddles two shards."""
    nblk = (N + BLOCK_ROWS - 1) // BLOCK_ROWS
    b0, b1 = rank * nblk // world, (rank + 1) * nblk // world
    return min(N, BLOCK_ROWS * b0), min(N, BLOCK_ROWS * b1)


def dh_argmax_shard_keys(rr_id: torch.Tensor, rr_logit: torch.Tensor, id_offset: int,
                         keys=None, stream=None) -> torch.Tensor:
    """int64 [M] keys of a shard's reranked lists (rr_id shard-local, id_offset = the shard's first
    vocab row): the largest key over all shards names the global argmax. Device tensors run the
    library's kernel on the stream; host tensors its host routine."""
    M, R = rr_id.shape
    if keys is None:
        keys = torch.empty(M, dtype=torch.int64, device=rr_id.device)
    if rr_id.is_cuda:
        _check(lib().dh_argmax_shard_keys(_dev(rr_id, "rr_id", torch.int32, (M, R)),
                                          _dev(rr_logit, "rr_logit", torch.float32, (M, R)), M, R,
                                          id_offset, _dev(keys, "keys", torch.int64, (M,)),
                                          _stream(stream)))
    else:
        _check(lib().dh_argmax_shard_keys_host(_host(rr_id, "rr_id", torch.int32, (M, R)),
                                               _host(rr_logit, "rr_logit", torch.float32, (M, R)),
                                               M, R, id_offset,
                                               _host(keys, "keys", torch.int64, (M,))))
    return keys


def dh_argmax_merge(keys: torch.Tensor, argmax_id=None, logit=None, stream=None):
    """keys int64 [P, M] (P shards' keys, or [1, M] after a MAX all-reduce) -> (argmax_id int32 [M],
    logit float32 [M]): the global argmax vocab id and its reranked logit."""
    P, M = keys.shape
    dev = keys.device
    if argmax_id is None:
        argmax_id = torch.empty(M, dtype=torch.int32, device=dev)
    if logit is None:
        logit = torch.empty(M, dtype=torch.float32, device=dev)
    if keys.is_cuda:
        _check(lib().dh_argmax_merge(_dev(keys, "keys", torch.int64, (P, M)), P, M,
                                     _dev(argmax_id, "argmax_id", torch.int32, (M,)),
                                     _dev(logit, "logit", torch.float32, (M,)), _stream(stream)))
    else:
        _check(lib().dh_argmax_merge_host(_host(keys, "keys", torch.int64, (P, M)), P, M,
                                          _host(argmax_id, "argmax_id", torch.int32, (M,)),
                                          _host(logit, "logit", torch.float32, (M,))))
    return argmax_id, logit


def merge_argmax_across_ranks(rr_id: torch.Tensor, rr_logit: torch.Tensor, id_offset: int,
                              group=None):
    """The exchange of the vocabulary-sharded head: this rank's keys, one MAX all-reduce over the
    process group (NCCL for device tensors, gloo for host tensors), then the decode. Returns
    (argmax_id [M] global vocab ids, logit [M]), the same on every rank."""
    import torch.distributed as dist
    keys = dh_argmax_shard_keys(rr_id, rr_logit, id_offset)
    dist.all_reduce(keys, op=dist.ReduceOp.MAX, group=group)
    return dh_argmax_merge(keys.view(1, -1))


def dh_workspace_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronises the stream and returns the workspace status word (0 = no kernel failure)."""
    word = ctypes.c_uint32(0)
    rc = lib().dh_workspace_status(_dev(workspace, "workspace", torch.uint8), workspace.numel(),
                                   ctypes.addressof(word), _stream(stream))
    if rc not in (DH_OK, DH_ERR_DEVICE):
        _check(rc)
    return int(word.value)


class DraftHead:
    """A quantised draft head on one GPU: the bf16 weight W[N, K] (kept for the exact rerank)
    plus its int2/int4 packing, and a workspace; calling it runs the whole path for x[M, K]."""

    def __init__(self, W: torch.Tensor, G: int = 128, bits: int = 2, kcand: int = 8,
                 rerank: int = 16, max_tokens: int = 72):
        W = _bf16(W, "W")
        if not W.is_cuda:
            raise ValueError("W must be a CUDA tensor")
        self.W, self.G, self.bits, self.kcand, self.rerank = W, G, bits, kcand, rerank
        self.N, self.K = W.shape
        quant = dh_quantize_pack_int2 if bits == 2 else dh_quantize_pack_int4
        self.packed, self.S, self.ZS = quant(W, G)
        self.workspace = new_workspace(max_tokens, self.N, self.K, kcand, rerank, W.device)
        self.max_tokens = max_tokens
        nblk = (self.N + BLOCK_ROWS - 1) // BLOCK_ROWS
        dev = W.device
        self._cv = torch.empty(max_tokens, nblk * kcand, dtype=torch.float32, device=dev)
        self._ci = torch.empty(max_tokens, nblk * kcand, dtype=torch.int32, device=dev)
        self._rr = torch.empty(max_tokens, rerank, dtype=torch.int32, device=dev)
        self._rl = torch.empty(max_tokens, rerank, dtype=torch.float32, device=dev)
        self._am = torch.empty(max_tokens, dtype=torch.int32, device=dev)

    def infer(self, x_host: torch.Tensor, stream=None):
        """End-to-end call from any host tensor: x_host (bf16 [M, K], pageable or pinned) is
        copied into this head's pinned staging buffer, then the call runs through call_host (the
        library's host-memory plan: copy in, coarse pass, rerank, results out and the
        synchronisation, all native). Returns pinned host tensors argmax [M], rr_id [M, R] and
        rr_logit [M, R], views of buffers the next call with the same M overwrites."""
        M = x_host.shape[0]
        if M < 1 or M > self.max_tokens:
            raise ValueError(f"M={M} outside 1..max_tokens={self.max_tokens}")
        if getattr(self, "_stage", None) is None:
            self._stage = torch.empty(self.max_tokens, self.K, dtype=torch.bfloat16,
                                      pin_memory=True)
        st = self._stage[:M]
        st.copy_(_bf16(x_host, "x_host"))
        return self.call_host(st, stream)

    def call_host(self, x_host: torch.Tensor, stream=None, plan: bool = True):
        """The same end-to-end call through the library's host-memory entry points: copy in,
        coarse pass, rerank, results out and the synchronisation all happen in native code.
        plan=True (default): a dh_host_plan prepared on the first call per (M, x_host) and run
        with dh_host_plan_run; plan=False: dh_draft_head_host with every argument each call.
        Returns pinned host tensors (argmax [M], rr_id [M, R], rr_logit [M, R]), views of
        buffers the next call with the same M overwrites."""
        M, R = x_host.shape[0], self.rerank
        sh = _stream(stream)
        key = (M, x_host.data_ptr())
        cached = self._host_calls.get(key) if hasattr(self, "_host_calls") else None
        if cached is None:
            if M < 1 or M > self.max_tokens:
                raise ValueError(f"M={M} outside 1..max_tokens={self.max_tokens}")
            xb = _bf16(x_host, "x_host")
            if xb.is_cuda or not xb.is_contiguous() or tuple(xb.shape) != (M, self.K):
                raise ValueError("x_host must be a contiguous host tensor [M, K]")
            if not hasattr(self, "_host_bufs"):
                dev, n = self.W.device, self.max_tokens * (1 + 2 * R)
                # results back to back (argmax, rr_id, rr_logit) on both sides
                self._host_bufs = (
                    torch.empty(self.max_tokens, self.K, dtype=torch.bfloat16, device=dev),
                    torch.empty(n, dtype=torch.int32, device=dev),
                    torch.empty(n, dtype=torch.int32, pin_memory=True))
                self._host_calls = {}
            x_dev, d_out, h_out = self._host_bufs
            d_am, d_rr, d_rl = d_out[:M], d_out[M:M + M * R], d_out[M + M * R:M + 2 * M * R]
            h_am = h_out[:M]
            h_rr = h_out[M:M + M * R].view(M, R)
            h_rl = h_out[M + M * R:M + 2 * M * R].view(torch.float32).view(M, R)
            ws = self.workspace
            args = (xb.data_ptr(), M, self.K, x_dev.data_ptr(), self.packed.data_ptr(),
                    self.S.data_ptr(), self.ZS.data_ptr(), self.W.data_ptr(), self.N, self.G,
                    self.bits, self.kcand, R, self._cv.data_ptr(), self._ci.data_ptr(),
                    d_rr.data_ptr(), d_rl.data_ptr(), d_am.data_ptr(), h_am.data_ptr(),
                    h_rr.data_ptr(), h_rl.data_ptr(), ws.data_ptr(), ws.numel())
            handle = ctypes.c_void_p()
            _check(lib().dh_host_plan_create(*args, ctypes.byref(handle)))
            # x_host is kept alive with its pointer; the plan is freed with this object
            cached = (args, (h_am, h_rr, h_rl), x_host, handle)
            self._host_calls[key] = cached
        if plan:
            _check(lib().dh_host_plan_run(cached[3], sh))
        else:
            _check(lib().dh_draft_head_host(*cached[0], sh))
        return cached[1]

    def __del__(self):
        calls = getattr(self, "_host_calls", None)
        if calls and _lib is not None:
            for c in calls.values():
                try:
                    _lib.dh_host_plan_destroy(c[3])
                except Exception:
                    pass
            calls.clear()

    def __call__(self, x: torch.Tensor, y_coarse=None, stream=None):
        """x bf16 [M, K] on the device -> dict of argmax [M], rr_id [M, R], rr_logit [M, R],
        cand_val, cand_id."""
        if x.shape[0] > self.max_tokens:
            raise ValueError(f"M={x.shape[0]} > max_tokens={self.max_tokens}")
        M = x.shape[0]
        rr, rl, am, cv, ci = dh_draft_head_argmax(
            x, self.packed, self.S, self.ZS, self.W, self.G, self.bits, self.kcand, self.rerank,
            cand_val=self._cv[:M], cand_id=self._ci[:M], rr_id=self._rr[:M],
            rr_logit=self._rl[:M], argmax_id=self._am[:M], y_coarse=y_coarse,
            workspace=self.workspace, stream=stream)
        return {"argmax": am, "rr_id": rr, "rr_logit": rl, "cand_val": cv, "cand_id": ci}
