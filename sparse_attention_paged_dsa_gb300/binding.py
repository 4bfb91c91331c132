"""Thin Python front-end of ``libdsa_indexer.so`` (argument marshalling only).

Every function here checks tensor dtypes, shapes and devices, then calls the
C entry point of the same name with raw device pointers and the current
torch CUDA stream.  All indexer arithmetic runs in the library's CUDA
kernels; if the library has not been built, ``load()`` raises instead of
falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdsa_indexer.so")

HEADS, HEAD_DIM, PAGE_ENTRIES, PAGE_TOKENS = 32, 64, 64, 256
WORKSPACE_HEADER_BYTES = 256

DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_WORKSPACE, DSA_ERR_CUDA = range(5)
DEVERR_SEQ_LEN_CLAMPED, DEVERR_BAD_PAGE, DEVERR_WAIT_TIMEOUT = 0x1, 0x2, 0x4

_lib = None


class DsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = load()
        msg = lib.dsa_status_string(status).decode()
        if status == DSA_ERR_CUDA:
            msg += ": " + lib.dsa_indexer_last_cuda_error().decode()
        super().__init__(f"{where}: {msg} (status {status})")
        self.status = status


def load():
    """Load the CUDA library (built by ``build.build()``); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    p, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    st = ctypes.c_int
    lib.dsa_indexer_workspace_size.argtypes = [i32, i64, i32]
    lib.dsa_indexer_workspace_size.restype = sz
    lib.dsa_indexer_workspace_init.argtypes = [p, sz, p]
    lib.dsa_indexer_workspace_init.restype = st
    lib.dsa_indexer_scores.argtypes = [p, p, p, i64, p, p, i32, i64, p, p, sz, p]
    lib.dsa_indexer_scores.restype = st
    lib.dsa_indexer_topk.argtypes = [p, p, i32, i64, i32, p, p, sz, p]
    lib.dsa_indexer_topk.restype = st
    lib.dsa_indexer_fused.argtypes = [p, p, p, i64, p, p, i32, i64, i32, p, p, p, sz, p]
    lib.dsa_indexer_fused.restype = st
    lib.dsa_indexer_scores_fp8.argtypes = [p, p, p, p, i64, p, p, i32, i64, p, p, sz, p]
    lib.dsa_indexer_scores_fp8.restype = st
    lib.dsa_indexer_fused_fp8.argtypes = [p, p, p, p, i64, p, p, i32, i64, i32, p, p, p, sz, p]
    lib.dsa_indexer_fused_fp8.restype = st
    lib.dsa_indexer_workspace_size_mtp.argtypes = [i32, i32, i64, i32]
    lib.dsa_indexer_workspace_size_mtp.restype = sz
    lib.dsa_indexer_scores_mtp.argtypes = [p, p, p, i64, p, p, i32, i32, i64, p, p, sz, p]
    lib.dsa_indexer_scores_mtp.restype = st
    lib.dsa_indexer_topk_mtp.argtypes = [p, p, i32, i32, i64, i32, p, p, sz, p]
    lib.dsa_indexer_topk_mtp.restype = st
    lib.dsa_indexer_fused_mtp.argtypes = [p, p, p, i64, p, p, i32, i32, i64, i32, p, p, p, sz, p]
    lib.dsa_indexer_fused_mtp.restype = st
    lib.dsa_indexer_qw_proj_workspace_size.argtypes = [i32, i64]
    lib.dsa_indexer_qw_proj_workspace_size.restype = sz
    lib.dsa_indexer_qw_proj.argtypes = [p, p, p, i32, i64, p, p, p, sz, p]
    lib.dsa_indexer_qw_proj.restype = st
    lib.dsa_sparse_mla_workspace_size.argtypes = [i32, i32]
    lib.dsa_sparse_mla_workspace_size.restype = sz
    lib.dsa_sparse_mla_decode.argtypes = [p, p, i64, p, p, i32, i64, p, i32, ctypes.c_float, p, p, p, sz, p]
    lib.dsa_sparse_mla_decode.restype = st
    lib.dsa_indexer_get_error.argtypes = [p, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int, p]
    lib.dsa_indexer_get_error.restype = st
    lib.dsa_status_string.argtypes = [st]
    lib.dsa_status_string.restype = ctypes.c_char_p
    lib.dsa_indexer_last_cuda_error.argtypes = []
    lib.dsa_indexer_last_cuda_error.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, name, dtypes, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


_BF16 = (torch.bfloat16, torch.int16, torch.uint16) if hasattr(torch, "uint16") else (torch.bfloat16, torch.int16)


def workspace_size(batch: int, max_context: int, k: int = 1) -> int:
    return int(load().dsa_indexer_workspace_size(batch, max_context, k))


def new_workspace(batch: int, max_context: int, k: int = 1, device="cuda") -> torch.Tensor:
    """A zeroed workspace of the size every entry point accepts for this shape."""
    n = workspace_size(batch, max_context, k)
    if n == 0:
        raise ValueError("invalid shape for a workspace")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def _check(status: int, where: str):
    if status != DSA_OK:
        raise DsaError(status, where)


def _score_args(q, w, key_pool, page_table, seq_lens, max_context):
    B = q.shape[0]
    _need(q, "q", _BF16, (B, HEADS, HEAD_DIM))
    _need(w, "w", (torch.float32,), (B, HEADS))
    _need(key_pool, "key_pool", _BF16)
    if key_pool.dim() != 3 or tuple(key_pool.shape[1:]) != (PAGE_ENTRIES, HEAD_DIM):
        raise ValueError(f"key_pool must be [num_pages, 64, 64], got {tuple(key_pool.shape)}")
    _need(page_table, "page_table", (torch.int32,), (B, max_context // PAGE_TOKENS))
    _need(seq_lens, "seq_lens", (torch.int32,), (B,))
    return B


def dsa_indexer_scores(q, w, key_pool, page_table, seq_lens, max_context: int, scores=None, workspace=None):
    """Scores [B, max_context/4] fp32: live scores, -inf elsewhere."""
    B = _score_args(q, w, key_pool, page_table, seq_lens, max_context)
    M = max_context // 4
    if scores is None:
        scores = torch.empty((B, M), dtype=torch.float32, device=q.device)
    _need(scores, "scores", (torch.float32,), (B, M))
    if workspace is None:
        workspace = torch.zeros(WORKSPACE_HEADER_BYTES, dtype=torch.uint8, device=q.device)
    st = load().dsa_indexer_scores(_ptr(q), _ptr(w), _ptr(key_pool), key_pool.shape[0], _ptr(page_table),
                                   _ptr(seq_lens), B, max_context, _ptr(scores), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(q.device))
    _check(st, "dsa_indexer_scores")
    return scores


def dsa_indexer_topk(scores, seq_lens, max_context: int, k: int, topk_idx=None, workspace=None):
    """Top-k positions [B, k] int32 of each row's live scores (ascending, -1 padded)."""
    B = scores.shape[0]
    _need(scores, "scores", (torch.float32,), (B, max_context // 4))
    _need(seq_lens, "seq_lens", (torch.int32,), (B,))
    if topk_idx is None:
        topk_idx = torch.empty((B, k), dtype=torch.int32, device=scores.device)
    _need(topk_idx, "topk_idx", (torch.int32,), (B, k))
    if workspace is None:
        workspace = torch.zeros(WORKSPACE_HEADER_BYTES, dtype=torch.uint8, device=scores.device)
    st = load().dsa_indexer_topk(_ptr(scores), _ptr(seq_lens), B, max_context, k, _ptr(topk_idx), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(scores.device))
    _check(st, "dsa_indexer_topk")
    return topk_idx


def dsa_indexer_fused(q, w, key_pool, page_table, seq_lens, max_context: int, k: int, topk_idx=None,
                      scores=None, workspace=None):
    """Scores + top-k in one call; ``scores`` None keeps the full-width row unwritten."""
    B = _score_args(q, w, key_pool, page_table, seq_lens, max_context)
    if topk_idx is None:
        topk_idx = torch.empty((B, k), dtype=torch.int32, device=q.device)
    _need(topk_idx, "topk_idx", (torch.int32,), (B, k))
    if scores is not None:
        _need(scores, "scores", (torch.float32,), (B, max_context // 4))
    if workspace is None:
        workspace = new_workspace(B, max_context, k, q.device)
    st = load().dsa_indexer_fused(_ptr(q), _ptr(w), _ptr(key_pool), key_pool.shape[0], _ptr(page_table),
                                  _ptr(seq_lens), B, max_context, k, _ptr(topk_idx), _ptr(scores),
                                  _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(q.device))
    _check(st, "dsa_indexer_fused")
    return topk_idx


_FP8 = tuple(t for t in (torch.uint8, getattr(torch, "float8_e4m3fn", None)) if t is not None)


def _fp8_args(q, w, key_codes, key_scales, page_table, seq_lens, max_context):
    B = q.shape[0]
    _need(q, "q", _BF16, (B, HEADS, HEAD_DIM))
    _need(w, "w", (torch.float32,), (B, HEADS))
    _need(key_codes, "key_codes", _FP8)
    if key_codes.dim() != 3 or tuple(key_codes.shape[1:]) != (PAGE_ENTRIES, HEAD_DIM):
        raise ValueError(f"key_codes must be [num_pages, 64, 64], got {tuple(key_codes.shape)}")
    _need(key_scales, "key_scales", (torch.float32,), (key_codes.shape[0], PAGE_ENTRIES))
    _need(page_table, "page_table", (torch.int32,), (B, max_context // PAGE_TOKENS))
    _need(seq_lens, "seq_lens", (torch.int32,), (B,))
    return B


def dsa_indexer_scores_fp8(q, w, key_codes, key_scales, page_table, seq_lens, max_context: int, scores=None,
                           workspace=None):
    """Scores on the fp8 key cache (e4m3 codes + per-key fp32 scale), as ``dsa_indexer_scores``."""
    B = _fp8_args(q, w, key_codes, key_scales, page_table, seq_lens, max_context)
    M = max_context // 4
    if scores is None:
        scores = torch.empty((B, M), dtype=torch.float32, device=q.device)
    _need(scores, "scores", (torch.float32,), (B, M))
    if workspace is None:
        workspace = torch.zeros(WORKSPACE_HEADER_BYTES, dtype=torch.uint8, device=q.device)
    st = load().dsa_indexer_scores_fp8(_ptr(q), _ptr(w), _ptr(key_codes), _ptr(key_scales), key_codes.shape[0],
                                       _ptr(page_table), _ptr(seq_lens), B, max_context, _ptr(scores),
                                       _ptr(workspace), workspace.numel() * workspace.element_size(),
                                       _stream(q.device))
    _check(st, "dsa_indexer_scores_fp8")
    return scores


def dsa_indexer_fused_fp8(q, w, key_codes, key_scales, page_table, seq_lens, max_context: int, k: int,
                          topk_idx=None, scores=None, workspace=None):
    """Scores + top-k on the fp8 key cache, as ``dsa_indexer_fused``."""
    B = _fp8_args(q, w, key_codes, key_scales, page_table, seq_lens, max_context)
    if topk_idx is None:
        topk_idx = torch.empty((B, k), dtype=torch.int32, device=q.device)
    _need(topk_idx, "topk_idx", (torch.int32,), (B, k))
    if scores is not None:
        _need(scores, "scores", (torch.float32,), (B, max_context // 4))
    if workspace is None:
        workspace = new_workspace(B, max_context, k, q.device)
    st = load().dsa_indexer_fused_fp8(_ptr(q), _ptr(w), _ptr(key_codes), _ptr(key_scales), key_codes.shape[0],
                                      _ptr(page_table), _ptr(seq_lens), B, max_context, k, _ptr(topk_idx),
                                      _ptr(scores), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                      _stream(q.device))
    _check(st, "dsa_indexer_fused_fp8")
    return topk_idx


def _mtp_args(q, w, key_pool, page_table, seq_lens, max_context):
    if q.dim() != 4:
        raise ValueError(f"q must be [batch, next_n, 32, 64], got {tuple(q.shape)}")
    B, Q = q.shape[0], q.shape[1]
    _need(q, "q", _BF16, (B, Q, HEADS, HEAD_DIM))
    _need(w, "w", (torch.float32,), (B, Q, HEADS))
    _need(key_pool, "key_pool", _BF16)
    if key_pool.dim() != 3 or tuple(key_pool.shape[1:]) != (PAGE_ENTRIES, HEAD_DIM):
        raise ValueError(f"key_pool must be [num_pages, 64, 64], got {tuple(key_pool.shape)}")
    _need(page_table, "page_table", (torch.int32,), (B, max_context // PAGE_TOKENS))
    _need(seq_lens, "seq_lens", (torch.int32,), (B,))
    return B, Q


def workspace_size_mtp(batch: int, next_n: int, max_context: int, k: int = 1) -> int:
    return int(load().dsa_indexer_workspace_size_mtp(batch, next_n, max_context, k))


def dsa_indexer_scores_mtp(q, w, key_pool, page_table, seq_lens, max_context: int, scores=None, workspace=None):
    """Scores [B, next_n, max_context/4] for next_n query tokens per request (q [B, next_n, 32, 64])."""
    B, Q = _mtp_args(q, w, key_pool, page_table, seq_lens, max_context)
    M = max_context // 4
    if scores is None:
        scores = torch.empty((B, Q, M), dtype=torch.float32, device=q.device)
    _need(scores, "scores", (torch.float32,), (B, Q, M))
    if workspace is None:
        workspace = torch.zeros(WORKSPACE_HEADER_BYTES, dtype=torch.uint8, device=q.device)
    st = load().dsa_indexer_scores_mtp(_ptr(q), _ptr(w), _ptr(key_pool), key_pool.shape[0], _ptr(page_table),
                                       _ptr(seq_lens), B, Q, max_context, _ptr(scores), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(q.device))
    _check(st, "dsa_indexer_scores_mtp")
    return scores


def dsa_indexer_topk_mtp(scores, seq_lens, max_context: int, k: int, topk_idx=None, workspace=None):
    """Top-k [B, next_n, k] of each token's row (token j sees seq_len - (next_n - 1 - j) tokens)."""
    if scores.dim() != 3:
        raise ValueError(f"scores must be [batch, next_n, max_context/4], got {tuple(scores.shape)}")
    B, Q = scores.shape[0], scores.shape[1]
    _need(scores, "scores", (torch.float32,), (B, Q, max_context // 4))
    _need(seq_lens, "seq_lens", (torch.int32,), (B,))
    if topk_idx is None:
        topk_idx = torch.empty((B, Q, k), dtype=torch.int32, device=scores.device)
    _need(topk_idx, "topk_idx", (torch.int32,), (B, Q, k))
    if workspace is None:
        workspace = torch.zeros(WORKSPACE_HEADER_BYTES, dtype=torch.uint8, device=scores.device)
    st = load().dsa_indexer_topk_mtp(_ptr(scores), _ptr(seq_lens), B, Q, max_context, k, _ptr(topk_idx),
                                     _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream(scores.device))
    _check(st, "dsa_indexer_topk_mtp")
    return topk_idx


def dsa_indexer_fused_mtp(q, w, key_pool, page_table, seq_lens, max_context: int, k: int, topk_idx=None,
                          scores=None, workspace=None):
    """Scores + top-k for next_n query tokens per request; ``scores`` None keeps the rows unwritten."""
    B, Q = _mtp_args(q, w, key_pool, page_table, seq_lens, max_context)
    if topk_idx is None:
        topk_idx = torch.empty((B, Q, k), dtype=torch.int32, device=q.device)
    _need(topk_idx, "topk_idx", (torch.int32,), (B, Q, k))
    if scores is not None:
        _need(scores, "scores", (torch.float32,), (B, Q, max_context // 4))
    if workspace is None:
        n = workspace_size_mtp(B, Q, max_context, k)
        if n == 0:
            raise ValueError("invalid shape for a workspace")
        workspace = torch.zeros(n, dtype=torch.uint8, device=q.device)
    st = load().dsa_indexer_fused_mtp(_ptr(q), _ptr(w), _ptr(key_pool), key_pool.shape[0], _ptr(page_table),
                                      _ptr(seq_lens), B, Q, max_context, k, _ptr(topk_idx), _ptr(scores),
                                      _ptr(workspace), workspace.numel() * workspace.element_size(),
                                      _stream(q.device))
    _check(st, "dsa_indexer_fused_mtp")
    return topk_idx


def qw_proj_workspace_size(batch: int, d_model: int) -> int:
    return int(load().dsa_indexer_qw_proj_workspace_size(batch, d_model))


def dsa_indexer_qw_proj(x, w_q, w_w, q_out=None, w_out=None, workspace=None):
    """q [B, 32, 64] bf16 and w [B, 32] fp32 from the bf16 hidden state x [B, d] (fp32 accumulate)."""
    if x.dim() != 2:
        raise ValueError(f"x must be [batch, d_model], got {tuple(x.shape)}")
    B, d = x.shape
    _need(x, "x", _BF16, (B, d))
    _need(w_q, "w_q", _BF16, (HEADS * HEAD_DIM, d))
    _need(w_w, "w_w", _BF16, (HEADS, d))
    if q_out is None:
        q_out = torch.empty((B, HEADS, HEAD_DIM), dtype=torch.bfloat16, device=x.device)
    _need(q_out, "q_out", _BF16, (B, HEADS, HEAD_DIM))
    if w_out is None:
        w_out = torch.empty((B, HEADS), dtype=torch.float32, device=x.device)
    _need(w_out, "w_out", (torch.float32,), (B, HEADS))
    if workspace is None:
        n = qw_proj_workspace_size(B, d)
        if n == 0:
            raise ValueError("invalid shape for the projection")
        workspace = torch.zeros(n, dtype=torch.uint8, device=x.device)
    st = load().dsa_indexer_qw_proj(_ptr(x), _ptr(w_q), _ptr(w_w), B, d, _ptr(q_out), _ptr(w_out), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(x.device))
    _check(st, "dsa_indexer_qw_proj")
    return q_out, w_out


MLA_HEADS, MLA_DIM, MLA_DV, MLA_MAX_TOPK = 64, 576, 512, 2048


def sparse_mla_workspace_size(batch: int, k: int) -> int:
    return int(load().dsa_sparse_mla_workspace_size(batch, k))


def dsa_sparse_mla_decode(q, kv_cache, page_table, seq_lens, max_context: int, topk_idx, sm_scale: float,
                          out=None, lse=None, workspace=None):
    """o [B, 64, 512] fp32 and lse [B, 64] fp32: attention of q [B, 64, 576] bf16 over the
    paged cache entries kv_cache [P, 64, 576] bf16 that topk_idx [B, k] selects."""
    if q.dim() != 3:
        raise ValueError(f"q must be [batch, 64, 576], got {tuple(q.shape)}")
    B = q.shape[0]
    _need(q, "q", _BF16, (B, MLA_HEADS, MLA_DIM))
    _need(kv_cache, "kv_cache", _BF16)
    if kv_cache.dim() != 3 or tuple(kv_cache.shape[1:]) != (PAGE_ENTRIES, MLA_DIM):
        raise ValueError(f"kv_cache must be [num_pages, 64, 576], got {tuple(kv_cache.shape)}")
    _need(page_table, "page_table", (torch.int32,), (B, max_context // PAGE_TOKENS))
    _need(seq_lens, "seq_lens", (torch.int32,), (B,))
    if topk_idx.dim() != 2 or topk_idx.shape[0] != B:
        raise ValueError(f"topk_idx must be [batch, k], got {tuple(topk_idx.shape)}")
    k = topk_idx.shape[1]
    _need(topk_idx, "topk_idx", (torch.int32,), (B, k))
    if out is None:
        out = torch.empty((B, MLA_HEADS, MLA_DV), dtype=torch.float32, device=q.device)
    _need(out, "out", (torch.float32,), (B, MLA_HEADS, MLA_DV))
    if lse is None:
        lse = torch.empty((B, MLA_HEADS), dtype=torch.float32, device=q.device)
    _need(lse, "lse", (torch.float32,), (B, MLA_HEADS))
    if workspace is None:
        n = sparse_mla_workspace_size(B, k)
        if n == 0:
            raise ValueError("invalid shape for the sparse MLA decode")
        workspace = torch.zeros(n, dtype=torch.uint8, device=q.device)
    st = load().dsa_sparse_mla_decode(_ptr(q), _ptr(kv_cache), kv_cache.shape[0], _ptr(page_table), _ptr(seq_lens),
                                      B, max_context, _ptr(topk_idx), k, float(sm_scale), _ptr(out), _ptr(lse),
                                      _ptr(workspace), workspace.numel() * workspace.element_size(),
                                      _stream(q.device))
    _check(st, "dsa_sparse_mla_decode")
    return out, lse


def get_error(workspace, clear: bool = True) -> int:
    """Read (and by default clear) the sticky device error word; synchronises the stream."""
    code = ctypes.c_uint32(0)
    st = load().dsa_indexer_get_error(_ptr(workspace), ctypes.byref(code), int(bool(clear)),
                                      _stream(workspace.device))
    _check(st, "dsa_indexer_get_error")
    return int(code.value)


def to_device(case, device="cuda"):
    """Copy an ``inputs.IndexerCase`` to device tensors (q, w, key_pool, page_table, seq_lens)."""
    q = torch.from_numpy(case.q.view("int16")).to(device).view(torch.bfloat16)
    w = torch.from_numpy(case.w).to(device)
    pool = torch.from_numpy(case.key_pool.view("int16")).to(device).view(torch.bfloat16)
    table = torch.from_numpy(case.page_table).to(device)
    seq = torch.from_numpy(case.seq_lens).to(device)
    return q, w, pool, table, seq


def to_device_fp8(case, device="cuda"):
    """Device copies of an fp8 case's key codes (uint8) and key scales (fp32)."""
    if case.key_codes is None or case.key_scales is None:
        raise ValueError("case has no fp8 key cache (see inputs.with_fp8_keys)")
    return torch.from_numpy(case.key_codes).to(device), torch.from_numpy(case.key_scales).to(device)
