"""Thin ctypes binding of ``libpkv.so`` (the C ABI in ``include/pkv.h``).

Argument marshalling only: every step of the sampler, the write-back and the
page fill runs in the library's CUDA kernels.  PyTorch supplies device memory
and the current stream.  The functions keep the C names without the ``pkv_``
prefix and raise ``PkvError`` on a negative status.  There is no CPU fallback:
if ``libpkv.so`` has not been built (``__graft_entry__.build()``) every call
raises.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

PKV_OK, PKV_EINVAL, PKV_ENOSPC, PKV_ECUDA, PKV_EUNSUPPORTED = 0, -1, -2, -3, -4
PKV_FP32, PKV_BF16 = 0, 1
PKV_MAX_VOCAB_FP32, PKV_MAX_VOCAB_BF16 = 262144, 524288
ST_NONFINITE, ST_ALL_NEG_INF, ST_ROW_OOB, ST_COL_OOB, ST_BAD_UNIFORM, ST_NOSPC = 1, 2, 4, 8, 16, 32
ST_TIMEOUT = 64
ST_TOKEN_CAP = 128
FL_COUNT, FL_ALIGN, FL_RANGE, FL_DUPLICATE = 1, 2, 4, 8

_lock = threading.Lock()
_lib = None


class PkvError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"pkv error {code}: {message}")
        self.code = code


def load() -> ctypes.CDLL:
    """Load libpkv.so (raises if it is missing: there is no fallback path)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing; build it with "
                                   "`python -c 'import __graft_entry__ as g; g.build()'`")
            lib = ctypes.CDLL(LIB_PATH)
            vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
            lib.pkv_last_error.restype = ctypes.c_char_p
            lib.pkv_last_error.argtypes = []
            lib.pkv_version.restype = i32
            lib.pkv_version.argtypes = []
            lib.pkv_sample_workspace_bytes.restype = sz
            lib.pkv_sample_workspace_bytes.argtypes = [i32, i32, i32]
            lib.pkv_sample_batch_noalloc.restype = i32
            lib.pkv_sample_batch_noalloc.argtypes = [vp, i32, i32, i32, i64, vp, vp, vp, vp, vp,
                                                     vp, i64, i64, vp, vp, vp, vp, vp]
            lib.pkv_decode_tail.restype = i32
            lib.pkv_decode_tail.argtypes = [vp, i32, i32, i32, i64, vp, vp, vp, vp, vp, vp, i64,
                                            i64, vp, vp, vp, vp, sz, vp, vp, vp, i32, i32, vp,
                                            i64, vp, i64, i64, vp, vp]
            lib.pkv_sample_workspace_init.restype = i32
            lib.pkv_sample_workspace_init.argtypes = [vp, sz, vp]
            lib.pkv_sample_batch_ex.restype = i32
            lib.pkv_sample_batch_ex.argtypes = [vp, i32, i32, i32, i64, vp, vp, vp, vp, vp, vp,
                                                vp, i64, i64, vp, vp, vp, vp, vp, sz, vp]
            lib.pkv_sample_batch.restype = i32
            lib.pkv_sample_batch.argtypes = [vp, i32, i32, i32, i64, vp, vp, vp, vp, vp, vp,
                                             i64, i64, vp, vp, vp, vp, vp, sz, vp]
            lib.pkv_writeback_tokens.restype = i32
            lib.pkv_writeback_tokens.argtypes = [vp, vp, vp, i32, vp, i64, i64, vp, vp]
            lib.pkv_alloc_pages.restype = i32
            lib.pkv_alloc_pages.argtypes = [vp, vp, i32, i32, i64, vp, vp, vp, vp]
            lib.pkv_fill_page_table.restype = i32
            lib.pkv_fill_page_table.argtypes = [vp, vp, vp, i32, i32, vp, i64, vp, i64, i64,
                                                vp, vp, vp]
            lib.pkv_free_pages.restype = i32
            lib.pkv_free_pages.argtypes = [vp, vp, vp, i32, i32, vp, i64, i64, vp, i64, i64,
                                           vp, vp, vp]
            lib.pkv_prepare_step.restype = i32
            lib.pkv_prepare_step.argtypes = [vp, vp, vp, i32, i32, vp, i64, vp, i64, i64, vp,
                                             i64, i64, vp, vp, vp, i64, vp, vp, vp, vp]
            lib.pkv_philox_uniforms.restype = i32
            lib.pkv_philox_uniforms.argtypes = [ctypes.c_uint64, ctypes.c_uint64, i32, vp, vp]
            lib.pkv_check_free_list.restype = i32
            lib.pkv_check_free_list.argtypes = [vp, i64, i32, i64, i64, vp, i64, vp, vp]
            _lib = lib
    return _lib


def last_error() -> str:
    return load().pkv_last_error().decode()


def version() -> int:
    return load().pkv_version()


def _check(rc: int) -> None:
    if rc != PKV_OK:
        raise PkvError(rc, last_error())


def _dev(t: Optional[torch.Tensor], dtype: torch.dtype, name: str, n: Optional[int] = None):
    """Device pointer of a contiguous CUDA tensor of the given dtype (or None)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if n is not None and t.numel() < n:
        raise ValueError(f"{name} has {t.numel()} elements, needs {n}")
    return t.data_ptr()


def _stream(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


_workspaces = {}


def sample_workspace_bytes(B: int, V: int, dtype: torch.dtype) -> int:
    """pkv_sample_workspace_bytes for a [B, V] batch of ``dtype`` logits."""
    code = PKV_BF16 if dtype == torch.bfloat16 else PKV_FP32
    return int(load().pkv_sample_workspace_bytes(int(B), int(V), code))


def sample_workspace_init(workspace: torch.Tensor, stream=None) -> None:
    """pkv_sample_workspace_init: readies a new workspace (zeroes its header)."""
    if workspace.dtype != torch.uint8 or not workspace.is_cuda or not workspace.is_contiguous():
        raise TypeError("workspace must be a contiguous uint8 CUDA tensor")
    _check(load().pkv_sample_workspace_init(workspace.data_ptr(), workspace.numel(),
                                            _stream(stream, workspace.device)))


def _workspace(device: torch.device, nbytes: int) -> torch.Tensor:
    """A cached, zero-initialised uint8 device buffer of at least ``nbytes``
    (replaced by a larger one as needed).

    Calls on different streams of one device must pass their own workspace.
    """
    key = (device.type, device.index)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def sample_batch(logits: torch.Tensor, temperature: Optional[torch.Tensor] = None,
                 top_k: Optional[torch.Tensor] = None, top_p: Optional[torch.Tensor] = None,
                 uniform: Optional[torch.Tensor] = None,
                 out_tokens: Optional[torch.Tensor] = None,
                 token_pool: Optional[torch.Tensor] = None,
                 wb_rows: Optional[torch.Tensor] = None, wb_cols: Optional[torch.Tensor] = None,
                 probs_out: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                 workspace: Optional[torch.Tensor] = None, stream=None,
                 min_p: Optional[torch.Tensor] = None) -> torch.Tensor:
    """pkv_sample_batch: one int32 token per row of ``logits`` [B, V]
    (pkv_sample_batch_ex when ``min_p`` is given).

    ``logits`` is fp32 or bf16 with unit column stride (any row stride).
    ``workspace`` (a uint8 CUDA tensor, initialised once with
    sample_workspace_init or zeroed) defaults to a buffer cached per device.
    Returns ``out_tokens`` (allocated here if not given).  See include/pkv.h.
    """
    lib = load()
    if logits.dim() != 2 or not logits.is_cuda:
        raise ValueError("logits must be a 2-D CUDA tensor")
    if logits.stride(1) != 1:
        raise ValueError("logits must have unit column stride")
    if logits.dtype == torch.bfloat16:
        dcode = PKV_BF16
    elif logits.dtype == torch.float32:
        dcode = PKV_FP32
    else:
        raise TypeError(f"logits dtype {logits.dtype} is not fp32 or bf16")
    B, V = logits.shape
    if out_tokens is None:
        out_tokens = torch.empty(B, dtype=torch.int32, device=logits.device)
    pool_rows = pool_cols = 0
    if token_pool is not None:
        if token_pool.dim() != 2:
            raise ValueError("token_pool must be 2-D")
        pool_rows, pool_cols = token_pool.shape
    need = int(lib.pkv_sample_workspace_bytes(B, V, dcode))
    if workspace is None:
        workspace = _workspace(logits.device, need)
    if workspace.dtype != torch.uint8 or not workspace.is_cuda or not workspace.is_contiguous():
        raise TypeError("workspace must be a contiguous uint8 CUDA tensor")
    head = (logits.data_ptr(), dcode, B, V, logits.stride(0),
            _dev(temperature, torch.float32, "temperature", B),
            _dev(top_k, torch.int32, "top_k", B), _dev(top_p, torch.float32, "top_p", B))
    if min_p is not None:
        call = lambda *rest: lib.pkv_sample_batch_ex(  # noqa: E731
            *head, _dev(min_p, torch.float32, "min_p", B), *rest)
    else:
        call = lambda *rest: lib.pkv_sample_batch(*head, *rest)  # noqa: E731
    rc = call(
        _dev(uniform, torch.float32, "uniform", B), _dev(out_tokens, torch.int32, "out_tokens", B),
        _dev(token_pool, torch.int32, "token_pool"), pool_rows, pool_cols,
        _dev(wb_rows, torch.int32, "wb_rows", B), _dev(wb_cols, torch.int64, "wb_cols", B),
        _dev(probs_out, torch.float32, "probs_out", B * V), _dev(status, torch.int32, "status", 1),
        workspace.data_ptr(), workspace.numel(), _stream(stream, logits.device))
    _check(rc)
    return out_tokens


def sample_batch_noalloc(logits: torch.Tensor, temperature: Optional[torch.Tensor] = None,
                         top_k: Optional[torch.Tensor] = None,
                         top_p: Optional[torch.Tensor] = None,
                         uniform: Optional[torch.Tensor] = None,
                         out_tokens: torch.Tensor = None,
                         token_pool: Optional[torch.Tensor] = None,
                         wb_rows: Optional[torch.Tensor] = None,
                         wb_cols: Optional[torch.Tensor] = None,
                         probs_out: Optional[torch.Tensor] = None,
                         status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """pkv_sample_batch_noalloc: sample_batch with the library's own static
    scratch; ``out_tokens`` (int32 [B], on the logits' device) is required, so
    that nothing is allocated.  See include/pkv.h."""
    lib = load()
    if logits.dim() != 2 or not logits.is_cuda or logits.stride(1) != 1:
        raise ValueError("logits must be a 2-D CUDA tensor with unit column stride")
    if logits.dtype == torch.bfloat16:
        dcode = PKV_BF16
    elif logits.dtype == torch.float32:
        dcode = PKV_FP32
    else:
        raise TypeError(f"logits dtype {logits.dtype} is not fp32 or bf16")
    if out_tokens is None:
        raise ValueError("out_tokens is required")
    B, V = logits.shape
    pool_rows = pool_cols = 0
    if token_pool is not None:
        if token_pool.dim() != 2:
            raise ValueError("token_pool must be 2-D")
        pool_rows, pool_cols = token_pool.shape
    rc = lib.pkv_sample_batch_noalloc(
        logits.data_ptr(), dcode, B, V, logits.stride(0),
        _dev(temperature, torch.float32, "temperature", B),
        _dev(top_k, torch.int32, "top_k", B), _dev(top_p, torch.float32, "top_p", B),
        _dev(uniform, torch.float32, "uniform", B), _dev(out_tokens, torch.int32, "out_tokens", B),
        _dev(token_pool, torch.int32, "token_pool"), pool_rows, pool_cols,
        _dev(wb_rows, torch.int32, "wb_rows", B), _dev(wb_cols, torch.int64, "wb_cols", B),
        _dev(probs_out, torch.float32, "probs_out", B * V), _dev(status, torch.int32, "status", 1),
        _stream(stream, logits.device))
    _check(rc)
    return out_tokens


def decode_tail(logits: torch.Tensor, temperature, top_k, top_p, uniform,
                out_tokens: torch.Tensor, token_pool, wb_rows, wb_cols,
                cached_len: torch.Tensor, device_len: torch.Tensor, table_idx: torch.Tensor,
                page_size: int, free_slots: torch.Tensor, page_table: torch.Tensor,
                total_out: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """pkv_decode_tail: sample_batch (with its write-back) and fill_page_table
    of one decode step in one call.  Returns ``out_tokens``."""
    lib = load()
    if logits.dim() != 2 or not logits.is_cuda or logits.stride(1) != 1:
        raise ValueError("logits must be a 2-D CUDA tensor with unit column stride")
    if logits.dtype == torch.bfloat16:
        dcode = PKV_BF16
    elif logits.dtype == torch.float32:
        dcode = PKV_FP32
    else:
        raise TypeError(f"logits dtype {logits.dtype} is not fp32 or bf16")
    B, V = logits.shape
    pool_rows = pool_cols = 0
    if token_pool is not None:
        pool_rows, pool_cols = token_pool.shape
    if page_table.dim() != 2:
        raise ValueError("page_table must be 2-D")
    need = int(lib.pkv_sample_workspace_bytes(B, V, dcode))
    if workspace is None:
        workspace = _workspace(logits.device, need)
    fb = cached_len.numel()
    rc = lib.pkv_decode_tail(
        logits.data_ptr(), dcode, B, V, logits.stride(0),
        _dev(temperature, torch.float32, "temperature", B),
        _dev(top_k, torch.int32, "top_k", B), _dev(top_p, torch.float32, "top_p", B),
        _dev(uniform, torch.float32, "uniform", B), _dev(out_tokens, torch.int32, "out_tokens", B),
        _dev(token_pool, torch.int32, "token_pool"), pool_rows, pool_cols,
        _dev(wb_rows, torch.int32, "wb_rows", B), _dev(wb_cols, torch.int64, "wb_cols", B),
        _dev(status, torch.int32, "status", 1), workspace.data_ptr(), workspace.numel(),
        _dev(cached_len, torch.int32, "cached_len", fb),
        _dev(device_len, torch.int32, "device_len", fb),
        _dev(table_idx, torch.int32, "table_idx", fb), fb, int(page_size),
        _dev(free_slots, torch.int32, "free_slots"), free_slots.numel(),
        _dev(page_table, torch.int32, "page_table"), page_table.shape[0], page_table.shape[1],
        _dev(total_out, torch.int64, "total_out", 1), _stream(stream, logits.device))
    _check(rc)
    return out_tokens


def writeback_tokens(tokens: torch.Tensor, rows: torch.Tensor, cols: torch.Tensor,
                     token_pool: torch.Tensor, status: Optional[torch.Tensor] = None,
                     stream=None) -> None:
    """pkv_writeback_tokens: token_pool[rows[b], cols[b]] = tokens[b] (cols < 0 skipped)."""
    lib = load()
    B = tokens.numel()
    R, C = token_pool.shape
    rc = lib.pkv_writeback_tokens(
        _dev(tokens, torch.int32, "tokens"), _dev(rows, torch.int32, "rows", B),
        _dev(cols, torch.int64, "cols", B), B, _dev(token_pool, torch.int32, "token_pool"),
        R, C, _dev(status, torch.int32, "status", 1), _stream(stream, token_pool.device))
    _check(rc)


def alloc_pages(cached_len, device_len, page_size: int, free_count: int) -> dict:
    """pkv_alloc_pages on host int32 arrays; returns first_page, num_pages, offset, total.

    Raises PkvError(PKV_ENOSPC) when the total exceeds free_count.
    """
    lib = load()
    c = torch.as_tensor(cached_len, dtype=torch.int32).contiguous().cpu()
    d = torch.as_tensor(device_len, dtype=torch.int32).contiguous().cpu()
    B = c.numel()
    first = torch.empty(B, dtype=torch.int32)
    num = torch.empty(B, dtype=torch.int32)
    off = torch.empty(B, dtype=torch.int64)
    total = torch.zeros(1, dtype=torch.int64)
    rc = lib.pkv_alloc_pages(c.data_ptr(), d.data_ptr(), B, int(page_size), int(free_count),
                             first.data_ptr(), num.data_ptr(), off.data_ptr(), total.data_ptr())
    out = {"first_page": first, "num_pages": num, "offset": off, "total": int(total[0])}
    _check(rc)
    return out


def fill_page_table(cached_len: torch.Tensor, device_len: torch.Tensor, table_idx: torch.Tensor,
                    page_size: int, free_slots: torch.Tensor, page_table: torch.Tensor,
                    total_out: Optional[torch.Tensor] = None,
                    status: Optional[torch.Tensor] = None, stream=None) -> None:
    """pkv_fill_page_table: allocate from the front of ``free_slots`` and fill ``page_table``."""
    lib = load()
    B = cached_len.numel()
    R, C = page_table.shape
    rc = lib.pkv_fill_page_table(
        _dev(cached_len, torch.int32, "cached_len", B), _dev(device_len, torch.int32, "device_len", B),
        _dev(table_idx, torch.int32, "table_idx", B), B, int(page_size),
        _dev(free_slots, torch.int32, "free_slots"), free_slots.numel(),
        _dev(page_table, torch.int32, "page_table"), R, C,
        _dev(total_out, torch.int64, "total_out", 1), _dev(status, torch.int32, "status", 1),
        _stream(stream, page_table.device))
    _check(rc)


def prepare_step(cached_len: torch.Tensor, device_len: torch.Tensor, table_idx: torch.Tensor,
                 page_size: int, free_slots: torch.Tensor, page_table: torch.Tensor,
                 token_pool: torch.Tensor, max_tokens: int,
                 positions: Optional[torch.Tensor] = None,
                 input_ids: Optional[torch.Tensor] = None,
                 out_loc: Optional[torch.Tensor] = None,
                 total_pages: Optional[torch.Tensor] = None,
                 total_tokens: Optional[torch.Tensor] = None,
                 status: Optional[torch.Tensor] = None, stream=None):
    """pkv_prepare_step: allocate and fill this step's pages, pack the
    positions [cached_len, device_len) and gather input_ids / out_loc at
    (table_idx, position).  Returns (positions, input_ids, out_loc,
    total_pages, total_tokens) as device tensors; the first three hold
    ``max_tokens`` entries, of which the first total_tokens are the step's."""
    lib = load()
    B = cached_len.numel()
    dev = page_table.device
    R, C = page_table.shape
    PR, PC = token_pool.shape
    n = int(max_tokens)

    def out(t, dtype, k):
        return t if t is not None else torch.empty(k, dtype=dtype, device=dev)

    positions = out(positions, torch.int32, n)
    input_ids = out(input_ids, torch.int32, n)
    out_loc = out(out_loc, torch.int32, n)
    total_pages = out(total_pages, torch.int64, 1)
    total_tokens = out(total_tokens, torch.int64, 1)
    rc = lib.pkv_prepare_step(
        _dev(cached_len, torch.int32, "cached_len", B), _dev(device_len, torch.int32, "device_len", B),
        _dev(table_idx, torch.int32, "table_idx", B), B, int(page_size),
        _dev(free_slots, torch.int32, "free_slots"), free_slots.numel(),
        _dev(page_table, torch.int32, "page_table"), R, C,
        _dev(token_pool, torch.int32, "token_pool"), PR, PC,
        _dev(positions, torch.int32, "positions", n), _dev(input_ids, torch.int32, "input_ids", n),
        _dev(out_loc, torch.int32, "out_loc", n), n,
        _dev(total_pages, torch.int64, "total_pages", 1),
        _dev(total_tokens, torch.int64, "total_tokens", 1),
        _dev(status, torch.int32, "status", 1), _stream(stream, dev))
    _check(rc)
    return positions, input_ids, out_loc, total_pages, total_tokens


def philox_uniforms(seed: int, offset: int, B: int, out: Optional[torch.Tensor] = None,
                    device=None, stream=None) -> torch.Tensor:
    """pkv_philox_uniforms: the B float32 uniforms of call ``offset`` under
    ``seed``, generated on the device."""
    if out is None:
        out = torch.empty(int(B), dtype=torch.float32,
                          device=device if device is not None else "cuda")
    rc = load().pkv_philox_uniforms(int(seed) & ((1 << 64) - 1), int(offset) & ((1 << 64) - 1),
                                    int(B), _dev(out, torch.float32, "out", int(B)),
                                    _stream(stream, out.device))
    _check(rc)
    return out


def free_pages(table_idx: torch.Tensor, begin: torch.Tensor, end: torch.Tensor, page_size: int,
               page_table: torch.Tensor, free_slots: torch.Tensor, free_count: int,
               total_out: Optional[torch.Tensor] = None,
               status: Optional[torch.Tensor] = None, stream=None) -> None:
    """pkv_free_pages: append page_table[t, b:e:ps] of every request after the
    ``free_count`` live entries of ``free_slots`` (whose length is the capacity)."""
    lib = load()
    B = table_idx.numel()
    R, C = page_table.shape
    rc = lib.pkv_free_pages(
        _dev(table_idx, torch.int32, "table_idx", B), _dev(begin, torch.int32, "begin", B),
        _dev(end, torch.int32, "end", B), B, int(page_size),
        _dev(page_table, torch.int32, "page_table"), R, C,
        _dev(free_slots, torch.int32, "free_slots"), int(free_count), free_slots.numel(),
        _dev(total_out, torch.int64, "total_out", 1), _dev(status, torch.int32, "status", 1),
        _stream(stream, page_table.device))
    _check(rc)


def check_free_list(free_slots: torch.Tensor, free_count: int, page_size: int, num_pages: int,
                    cache_pages: int, bitmap: torch.Tensor, result: torch.Tensor,
                    stream=None) -> None:
    """pkv_check_free_list: OR the FL_* bits of the first ``free_count`` entries
    into ``result`` (zeroed first); ``bitmap`` is int32 scratch of
    ceil(num_pages / 32) words."""
    lib = load()
    rc = lib.pkv_check_free_list(
        _dev(free_slots, torch.int32, "free_slots"), int(free_count), int(page_size),
        int(num_pages), int(cache_pages), _dev(bitmap, torch.int32, "bitmap"), bitmap.numel(),
        _dev(result, torch.int32, "result", 1), _stream(stream, result.device))
    _check(rc)
