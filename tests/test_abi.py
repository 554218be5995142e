"""CPU tests of the C ABI: the library loads, exports every symbol that
include/pkv.h declares, rejects bad arguments on the host before any launch,
and its host-side page allocation matches the oracle."""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from paged_kv_gb300 import pkv, workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = pkv.load()
    names = declared_functions()
    assert "pkv_sample_batch" in names and "pkv_fill_page_table" in names
    for name in names:
        assert hasattr(lib, name), f"{name} is declared in pkv.h but not exported"


def test_binding_types_every_declared_function():
    # The ctypes binding declares argument and result types for every entry
    # point of pkv.h (an untyped call would pass 64-bit values as int).
    lib = pkv.load()
    for name in declared_functions():
        fn = getattr(lib, name)
        assert fn.argtypes is not None, f"{name}: no argtypes in paged_kv_gb300/pkv.py"
        assert fn.restype is not None, f"{name}: no restype in paged_kv_gb300/pkv.py"


def test_binding_constants_match_the_header():
    text = open(HEADER).read()
    for name in ("PKV_MAX_VOCAB_FP32", "PKV_MAX_VOCAB_BF16"):
        m = re.search(r"#define\s+%s\s+(\d+)" % name, text)
        assert m is not None and int(m.group(1)) == getattr(pkv, name), name


def test_version_and_workspace():
    lib = pkv.load()
    assert pkv.version() == 310
    # A 256-byte header, then per (row, chunk) one
    # 3216-byte record and 16 KB of slice histograms (8 warps x 1024 16-bit
    # counts); the mixed batch's rows are 8 chunks of 20480 bf16.
    fixed = 256
    per = 3216 + 8 * 1024 * 2
    assert lib.pkv_sample_workspace_bytes(256, 151936, 1) == fixed + 256 * 8 * per
    assert lib.pkv_sample_workspace_bytes(1024, 256000, 1) == fixed + 1024 * 16 * per
    # fp32 rows have no count-histogram items, so no slice histograms: the
    # nucleus batch's rows are 15 chunks of 10240 fp32.
    assert lib.pkv_sample_workspace_bytes(256, 151936, 0) == fixed + 256 * 15 * 3216
    assert lib.pkv_sample_workspace_bytes(0, 100, 1) == 0
    assert lib.pkv_sample_workspace_bytes(4, 0, 1) == 0
    assert lib.pkv_sample_workspace_bytes(4, 100, 7) == 0


def test_sample_batch_requires_a_workspace():
    lib = pkv.load()
    p = ctypes.c_void_p(256)
    need = lib.pkv_sample_workspace_bytes(256, 151936, 1)
    common = (p, 1, 256, 151936, 151936, None, None, None, None, p, None, 0, 0,
              None, None, None, None)
    rc = lib.pkv_sample_batch(*common, None, 0, None)
    assert rc == pkv.PKV_EINVAL and "workspace" in pkv.last_error()
    rc = lib.pkv_sample_batch(*common, p, need - 1, None)
    assert rc == pkv.PKV_EINVAL and "workspace" in pkv.last_error()
    rc = lib.pkv_sample_batch(*common, ctypes.c_void_p(264), need, None)
    assert rc == pkv.PKV_EINVAL and "aligned" in pkv.last_error()


def test_workspace_init_validates_before_any_launch():
    lib = pkv.load()
    assert lib.pkv_sample_workspace_init(None, 4096, None) == pkv.PKV_EINVAL
    assert "NULL" in pkv.last_error()
    assert lib.pkv_sample_workspace_init(ctypes.c_void_p(256), 255, None) == pkv.PKV_EINVAL
    assert "header" in pkv.last_error()
    assert lib.pkv_sample_workspace_init(ctypes.c_void_p(264), 4096, None) == pkv.PKV_EINVAL
    assert "aligned" in pkv.last_error()


def test_host_validation_launches_nothing():
    lib = pkv.load()
    # NULL logits / out_tokens, bad sizes: rejected before any CUDA call.
    rc = lib.pkv_sample_batch(None, 1, 4, 100, 100, None, None, None, None, 1, None, 0, 0,
                              None, None, None, None, None, 0, None)
    assert rc == pkv.PKV_EINVAL and "logits" in pkv.last_error()
    dummy = ctypes.c_void_p(16)
    rc = lib.pkv_sample_batch(dummy, 1, 0, 100, 100, None, None, None, None, dummy, None, 0,
                              0, None, None, None, None, None, 0, None)
    assert rc == pkv.PKV_EINVAL
    rc = lib.pkv_sample_batch(dummy, 1, 4, 100, 99, None, None, None, None, dummy, None, 0, 0,
                              None, None, None, None, None, 0, None)
    assert rc == pkv.PKV_EINVAL and "row_stride" in pkv.last_error()
    rc = lib.pkv_sample_batch(dummy, 7, 4, 100, 100, None, None, None, None, dummy, None, 0,
                              0, None, None, None, None, None, 0, None)
    assert rc == pkv.PKV_EINVAL
    rc = lib.pkv_sample_batch(dummy, 1, 4, 100, 100, dummy, None, None, None, dummy, None, 0,
                              0, None, None, None, None, None, 0, None)
    assert rc == pkv.PKV_EINVAL and "uniform" in pkv.last_error()
    rc = lib.pkv_sample_batch(dummy, 1, 4, 100, 100, None, None, None, None, dummy, dummy, 4,
                              8, None, None, None, None, None, 0, None)
    assert rc == pkv.PKV_EINVAL and "wb_rows" in pkv.last_error()
    rc = lib.pkv_sample_batch(dummy, 0, 4, 300000, 300000, None, None, None, None, dummy,
                              None, 0, 0, None, None, None, None, None, 0, None)
    assert rc == pkv.PKV_EUNSUPPORTED
    rc = lib.pkv_fill_page_table(dummy, dummy, dummy, 5000, 4, dummy, 10, dummy, 4, 4, None,
                                 None, None)
    assert rc == pkv.PKV_EINVAL
    rc = lib.pkv_fill_page_table(dummy, dummy, dummy, 4, 0, dummy, 10, dummy, 4, 4, None,
                                 None, None)
    assert rc == pkv.PKV_EINVAL and "page_size" in pkv.last_error()
    rc = lib.pkv_writeback_tokens(None, dummy, dummy, 3, dummy, 2, 2, None, None)
    assert rc == pkv.PKV_EINVAL


def test_free_path_host_validation_launches_nothing():
    lib = pkv.load()
    d = ctypes.c_void_p(16)
    # B outside [0, 4096], page_size < 1, count above capacity, NULL pointers.
    assert lib.pkv_free_pages(d, d, d, -1, 4, d, 4, 4, d, 0, 8, None, None, None) == pkv.PKV_EINVAL
    assert lib.pkv_free_pages(d, d, d, 5000, 4, d, 4, 4, d, 0, 8, None, None, None) == pkv.PKV_EINVAL
    assert lib.pkv_free_pages(d, d, d, 2, 0, d, 4, 4, d, 0, 8, None, None, None) == pkv.PKV_EINVAL
    assert "page_size" in pkv.last_error()
    assert lib.pkv_free_pages(d, d, d, 2, 4, d, 4, 4, d, 9, 8, None, None, None) == pkv.PKV_EINVAL
    assert "capacity" in pkv.last_error()
    assert lib.pkv_free_pages(d, None, d, 2, 4, d, 4, 4, d, 0, 8, None, None, None) == pkv.PKV_EINVAL
    assert lib.pkv_free_pages(d, d, d, 2, 4, d, 0, 4, d, 0, 8, None, None, None) == pkv.PKV_EINVAL
    # The integrity check: NULL result, pool above 2^31 entries, bitmap too small.
    assert lib.pkv_check_free_list(d, 4, 4, 4, 0, d, 1, None, None) == pkv.PKV_EINVAL
    assert lib.pkv_check_free_list(d, 4, 64, 1 << 26, 0, d, 1 << 21, d, None) == pkv.PKV_EINVAL
    assert "2^31" in pkv.last_error()
    assert lib.pkv_check_free_list(d, 4, 4, 100, 0, d, 3, d, None) == pkv.PKV_EINVAL
    assert "bitmap" in pkv.last_error()
    assert lib.pkv_check_free_list(d, -1, 4, 4, 0, d, 1, d, None) == pkv.PKV_EINVAL
    assert lib.pkv_check_free_list(d, 4, 4, -4, 0, d, 1, d, None) == pkv.PKV_EINVAL


def test_sample_batch_ex_validates_like_the_plain_call():
    lib = pkv.load()
    d = ctypes.c_void_p(16)
    # (logits, dt, B, V, stride, T, k, p, min_p, u, out, pool, rows, cols, wb_rows, wb_cols,
    #  probs, status, workspace, workspace_bytes, stream)
    f = lib.pkv_sample_batch_ex
    assert f(None, 1, 4, 100, 100, None, None, None, d, None, d, None, 0, 0, None, None, None,
             None, None, 0, None) == pkv.PKV_EINVAL and "logits" in pkv.last_error()
    assert f(d, 1, 4, 100, 99, None, None, None, d, None, d, None, 0, 0, None, None, None, None,
             None, 0, None) == pkv.PKV_EINVAL and "row_stride" in pkv.last_error()
    assert f(d, 1, 4, 100, 100, d, None, None, d, None, d, None, 0, 0, None, None, None, None,
             None, 0, None) == pkv.PKV_EINVAL and "uniform" in pkv.last_error()
    # A valid call without a workspace is refused before any launch.
    assert f(d, 1, 4, 100, 100, None, None, None, d, None, d, None, 0, 0, None, None, None, None,
             None, 0, None) == pkv.PKV_EINVAL and "workspace" in pkv.last_error()


def test_prepare_step_host_validation_launches_nothing():
    lib = pkv.load()
    d = ctypes.c_void_p(16)
    f = lib.pkv_prepare_step
    ok = dict(cached=d, device=d, table=d, B=2, ps=4, free=d, nfree=8, pt=d, ptr=4, ptc=16,
              pool=d, pr=4, pc=16, pos=d, ids=d, loc=d, cap=32)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["cached"], a["device"], a["table"], a["B"], a["ps"], a["free"], a["nfree"],
                 a["pt"], a["ptr"], a["ptc"], a["pool"], a["pr"], a["pc"], a["pos"], a["ids"],
                 a["loc"], a["cap"], None, None, None, None)

    assert call(B=-1) == pkv.PKV_EINVAL
    assert call(B=5000) == pkv.PKV_EINVAL
    assert call(ps=0) == pkv.PKV_EINVAL and "page_size" in pkv.last_error()
    assert call(cap=-1) == pkv.PKV_EINVAL and "max_tokens" in pkv.last_error()
    assert call(cap=1 << 31) == pkv.PKV_EINVAL
    assert call(pool=None) == pkv.PKV_EINVAL and "token_pool" in pkv.last_error()
    assert call(pr=0) == pkv.PKV_EINVAL
    assert call(loc=None) == pkv.PKV_EINVAL and "output" in pkv.last_error()
    assert call(table=None) == pkv.PKV_EINVAL
    assert call(ptc=0) == pkv.PKV_EINVAL


def test_philox_uniforms_host_validation_launches_nothing():
    lib = pkv.load()
    d = ctypes.c_void_p(16)
    assert lib.pkv_philox_uniforms(42, 0, -1, d, None) == pkv.PKV_EINVAL
    assert lib.pkv_philox_uniforms(42, 0, 65536, d, None) == pkv.PKV_EINVAL
    assert lib.pkv_philox_uniforms(42, 0, 4, None, None) == pkv.PKV_EINVAL
    assert lib.pkv_philox_uniforms(42, 0, 0, None, None) == pkv.PKV_OK


@pytest.mark.parametrize("name", ["pr1", "mixed", "nucleus", "large"])
def test_host_alloc_pages_matches_oracle(name):
    w = workloads.make(name) if name in ("pr1",) else workloads.make(name, B=64, V=64)
    host = pkv.alloc_pages(w.cached_len, w.device_len, w.page_size, len(w.free_slots))
    ref = oracle.alloc_pages(w.cached_len, w.device_len, w.page_size, len(w.free_slots))
    assert ref["rc"] == 0
    np.testing.assert_array_equal(host["first_page"].numpy(), ref["first_page"])
    np.testing.assert_array_equal(host["num_pages"].numpy(), ref["num_pages"])
    np.testing.assert_array_equal(host["offset"].numpy(), ref["offset"])
    assert host["total"] == ref["total"]


def test_host_alloc_pages_pins_and_errors():
    res = pkv.alloc_pages([6], [9], 4, 10)  # one page: logical page 2
    assert res["first_page"].tolist() == [2] and res["num_pages"].tolist() == [1]
    with pytest.raises(pkv.PkvError) as e:
        pkv.alloc_pages([0, 0], [9, 9], 4, 5)
    assert e.value.code == pkv.PKV_ENOSPC
    with pytest.raises(pkv.PkvError) as e:
        pkv.alloc_pages([-1], [3], 4, 5)
    assert e.value.code == pkv.PKV_EINVAL
    with pytest.raises(pkv.PkvError):
        pkv.alloc_pages([0], [3], 0, 5)
    assert pkv.alloc_pages([], [], 4, 0)["total"] == 0


def test_binding_refuses_cpu_tensors():
    import torch

    with pytest.raises(ValueError):
        pkv.sample_batch(torch.zeros(2, 8))
