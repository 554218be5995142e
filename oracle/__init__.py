"""ctypes front end of the CPU oracle (``oracle.cpp``).

TEST INFRASTRUCTURE ONLY.  The oracle is the plain fp64 definition of the
decode-step tail that the CUDA library is checked against.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package; the library itself never does, and it shares no code with it.

Every function cites the passage of "mini-sglang from Scratch" it follows in
``oracle.cpp``.  Arrays are numpy or CPU torch tensors; results are numpy.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
# A prebuilt oracle library to load instead (the mutant test of
# tests/test_oracle_mutants.py loads copies with one planted mistake each).
_LIB_OVERRIDE = os.environ.get("PKV_ORACLE_LIB")
_lock = threading.Lock()
_lib = None

DTYPE_FP32 = 0
DTYPE_BF16 = 1


def build(force: bool = False) -> str:
    """Compile oracle.cpp into liboracle.so with the host C++ compiler."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread",
               _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            if _LIB_OVERRIDE:
                lib = ctypes.CDLL(_LIB_OVERRIDE)
            else:
                build()
                lib = ctypes.CDLL(_LIB_PATH)
            vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
            lib.oracle_sample.argtypes = [vp, i32, i32, i32, i64, vp, vp, vp, vp,
                                          vp, vp, vp, vp, vp, vp, i32]
            lib.oracle_sample.restype = i32
            lib.oracle_sample_ex.argtypes = [vp, i32, i32, i32, i64, vp, vp, vp, vp, vp,
                                             vp, vp, vp, vp, vp, vp, vp, i32]
            lib.oracle_sample_ex.restype = i32
            lib.oracle_writeback.argtypes = [vp, vp, vp, i32, vp, i64, i64]
            lib.oracle_writeback.restype = i32
            lib.oracle_alloc_pages.argtypes = [vp, vp, i32, i32, i64, vp, vp, vp, vp]
            lib.oracle_alloc_pages.restype = i32
            lib.oracle_fill_page_table.argtypes = [vp, vp, vp, i32, i32, vp, i64,
                                                   vp, i64, i64, vp, vp]
            lib.oracle_fill_page_table.restype = i32
            lib.oracle_free_pages.argtypes = [vp, vp, vp, i32, i32, vp, i64, i64, vp, i64,
                                              i64, vp, vp]
            lib.oracle_free_pages.restype = i32
            lib.oracle_check_free_list.argtypes = [vp, i64, i32, i64, i64]
            lib.oracle_check_free_list.restype = i32
            lib.oracle_philox4x64.argtypes = [vp, vp, vp]
            lib.oracle_philox4x64.restype = None
            lib.oracle_uniforms.argtypes = [ctypes.c_uint64, ctypes.c_uint64, i32, vp]
            lib.oracle_uniforms.restype = None
            lib.oracle_prepare_step.argtypes = [vp, vp, vp, i32, i32, vp, i64, vp, i64, i64,
                                                vp, i64, i64, vp, vp, vp, i64, vp, vp, vp]
            lib.oracle_prepare_step.restype = i32
            _lib = lib
    return _lib


def _np(x, dtype):
    """Contiguous numpy copy/view of a numpy array or CPU torch tensor."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=dtype))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def logits_bits(logits):
    """(raw array, dtype code) for fp32 or bf16 logits.

    bf16 tensors are passed as their raw 16-bit patterns; numpy has no bf16.
    """
    if hasattr(logits, "detach"):
        import torch

        t = logits.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16), DTYPE_BF16
        if t.dtype == torch.float32:
            return t.numpy(), DTYPE_FP32
        raise TypeError(f"logits dtype {t.dtype} is not fp32 or bf16")
    a = np.ascontiguousarray(logits)
    if a.dtype == np.float32:
        return a, DTYPE_FP32
    if a.dtype == np.uint16:
        return a, DTYPE_BF16
    raise TypeError(f"logits dtype {a.dtype} is not float32 or uint16 (bf16 bits)")


def sample(logits, temperature=None, top_k=None, top_p=None, uniform=None,
           want_probs: bool = False, threads: int = 1, min_p=None) -> dict:
    """Sample one token per row of ``logits`` [B, V] (fp32 or bf16).

    ``temperature=None`` is the all-greedy batch; rows with temperature <= 0
    are greedy.  ``top_k`` / ``top_p`` / ``min_p`` None mean "off".  Returns a
    dict with ``tokens`` (int32), ``probs`` (fp64 [B, V] or None),
    ``topp_margin``, ``cdf_margin``, ``minp_margin``, ``kept`` and
    ``row_status``.
    """
    lib = _load()
    bits, dcode = logits_bits(logits)
    if bits.ndim != 2:
        raise ValueError("logits must be [B, V]")
    B, V = bits.shape
    t = _np(temperature, np.float32)
    k = _np(top_k, np.int32)
    p = _np(top_p, np.float32)
    u = _np(uniform, np.float32)
    if t is not None and u is None:
        raise ValueError("uniform is required unless the batch is all greedy")
    tokens = np.empty(B, np.int32)
    probs = np.empty((B, V), np.float64) if want_probs else None
    tm = np.empty(B, np.float64)
    cm = np.empty(B, np.float64)
    kept = np.empty(B, np.int32)
    st = np.empty(B, np.int32)
    mp = _np(min_p, np.float32)
    mm = np.empty(B, np.float64)
    lib.oracle_sample_ex(_ptr(bits), dcode, B, V, V, _ptr(t), _ptr(k), _ptr(p), _ptr(mp),
                         _ptr(u), _ptr(tokens), _ptr(probs), _ptr(tm), _ptr(cm), _ptr(mm),
                         _ptr(kept), _ptr(st), int(threads))
    return {"tokens": tokens, "probs": probs, "topp_margin": tm, "cdf_margin": cm,
            "minp_margin": mm, "kept": kept, "row_status": st}


def writeback(tokens, rows, cols, pool: np.ndarray) -> int:
    """token_pool[rows[b], cols[b]] = tokens[b] in place; returns status bits."""
    lib = _load()
    tok = _np(tokens, np.int32)
    r = _np(rows, np.int32)
    c = _np(cols, np.int64)
    if pool.dtype != np.int32 or not pool.flags.c_contiguous:
        raise TypeError("pool must be a C-contiguous int32 array")
    R, C = pool.shape
    return int(lib.oracle_writeback(_ptr(tok), _ptr(r), _ptr(c), len(tok), _ptr(pool), R, C))


def alloc_pages(cached_len, device_len, page_size: int, free_count: int) -> dict:
    """Per-request first page, page count and free-list offset, plus the total."""
    lib = _load()
    c = _np(cached_len, np.int32)
    d = _np(device_len, np.int32)
    B = len(c)
    first = np.empty(B, np.int32)
    num = np.empty(B, np.int32)
    off = np.empty(B, np.int64)
    total = np.zeros(1, np.int64)
    rc = lib.oracle_alloc_pages(_ptr(c), _ptr(d), B, int(page_size), int(free_count),
                                _ptr(first), _ptr(num), _ptr(off), _ptr(total))
    return {"rc": int(rc), "first_page": first, "num_pages": num, "offset": off,
            "total": int(total[0])}


def fill_page_table(cached_len, device_len, table_idx, page_size: int, free_slots,
                    page_table: np.ndarray) -> dict:
    """Allocate from the front of ``free_slots`` and fill ``page_table`` in place."""
    lib = _load()
    c = _np(cached_len, np.int32)
    d = _np(device_len, np.int32)
    t = _np(table_idx, np.int32)
    fs = _np(free_slots, np.int32)
    if page_table.dtype != np.int32 or not page_table.flags.c_contiguous:
        raise TypeError("page_table must be a C-contiguous int32 array")
    R, C = page_table.shape
    total = np.zeros(1, np.int64)
    status = np.zeros(1, np.int32)
    rc = lib.oracle_fill_page_table(_ptr(c), _ptr(d), _ptr(t), len(c), int(page_size),
                                    _ptr(fs), len(fs), _ptr(page_table), R, C,
                                    _ptr(total), _ptr(status))
    return {"rc": int(rc), "total": int(total[0]), "status": int(status[0])}


def free_pages(table_idx, begin, end, page_size: int, page_table: np.ndarray, free_slots,
               free_count: int) -> dict:
    """Batched lazy free: append page_table[t, b:e:ps] of every request to the
    free list.  ``free_slots`` is an int32 array of the list's capacity whose
    first ``free_count`` entries are live; it is updated in place."""
    lib = _load()
    t = _np(table_idx, np.int32)
    b = _np(begin, np.int32)
    e = _np(end, np.int32)
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    if not isinstance(free_slots, np.ndarray) or free_slots.dtype != np.int32 \
            or not free_slots.flags.c_contiguous:
        raise TypeError("free_slots must be a C-contiguous int32 array")
    R, C = pt.shape
    total = np.zeros(1, np.int64)
    status = np.zeros(1, np.int32)
    rc = lib.oracle_free_pages(_ptr(t), _ptr(b), _ptr(e), len(t), int(page_size), _ptr(pt), R, C,
                               _ptr(free_slots), int(free_count), len(free_slots),
                               _ptr(total), _ptr(status))
    return {"rc": int(rc), "total": int(total[0]), "status": int(status[0])}


def check_free_list(free_slots, page_size: int, num_pages: int, cache_pages: int) -> int:
    """Integrity bits of a free list: 1 count, 2 alignment, 4 range, 8 duplicate."""
    lib = _load()
    fs = _np(free_slots, np.int32)
    return int(lib.oracle_check_free_list(_ptr(fs), len(fs), int(page_size), int(num_pages),
                                          int(cache_pages)))


def prepare_step(cached_len, device_len, table_idx, page_size: int, free_slots,
                 page_table: np.ndarray, token_pool, max_tokens: int) -> dict:
    """The step before the model: allocate and fill the new pages of every
    request in ``page_table`` (in place), then pack the positions
    [cached_len, device_len) in batch order and gather ``input_ids`` from the
    token pool and ``out_loc`` from the page table at (table_idx, position).
    Returns the three packed int32 arrays (length = the token count when it
    is at most ``max_tokens``, else empty), the totals, status bits and rc."""
    lib = _load()
    c = _np(cached_len, np.int32)
    d = _np(device_len, np.int32)
    t = _np(table_idx, np.int32)
    fs = _np(free_slots, np.int32)
    pool = _np(token_pool, np.int32)
    if page_table.dtype != np.int32 or not page_table.flags.c_contiguous:
        raise TypeError("page_table must be a C-contiguous int32 array")
    R, C = page_table.shape
    PR, PC = pool.shape
    cap = max(int(max_tokens), 0)
    pos = np.full(cap, -7, np.int32)
    ids = np.full(cap, -7, np.int32)
    loc = np.full(cap, -7, np.int32)
    pages = np.zeros(1, np.int64)
    ntok = np.zeros(1, np.int64)
    status = np.zeros(1, np.int32)
    rc = lib.oracle_prepare_step(_ptr(c), _ptr(d), _ptr(t), len(c), int(page_size), _ptr(fs),
                                 len(fs), _ptr(page_table), R, C, _ptr(pool), PR, PC, _ptr(pos),
                                 _ptr(ids), _ptr(loc), int(max_tokens), _ptr(pages), _ptr(ntok),
                                 _ptr(status))
    n = int(ntok[0]) if rc == 0 else 0
    return {"rc": int(rc), "positions": pos[:n], "input_ids": ids[:n], "out_loc": loc[:n],
            "total_pages": int(pages[0]), "total_tokens": int(ntok[0]), "status": int(status[0])}


def philox4x64(counter, key) -> np.ndarray:
    """One Philox-4x64-10 block: four 64-bit words for a 4-word counter and a
    2-word key."""
    lib = _load()
    c = np.ascontiguousarray(np.asarray(counter, dtype=np.uint64))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint64))
    out = np.empty(4, np.uint64)
    lib.oracle_philox4x64(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniforms(seed: int, offset: int, B: int) -> np.ndarray:
    """The B float32 uniforms of call ``offset`` under ``seed`` (one per row)."""
    lib = _load()
    u = np.empty(B, np.float32)
    lib.oracle_uniforms(int(seed) & ((1 << 64) - 1), int(offset) & ((1 << 64) - 1), int(B), _ptr(u))
    return u
