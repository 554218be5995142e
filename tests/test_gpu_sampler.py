"""GPU parity of pkv_sample_batch against the CPU oracle (through the C ABI).

Small shapes span several CTAs, ragged row tails, V below the warp width,
the unaligned (scalar-load) path, ties at the argmax / top-k / top-p
boundaries, -inf logits and every parameter extreme; the five workloads run
at full size in the launch configuration the benchmark times.
"""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gb300 import pkv, workloads
from parity import check_sampler

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _d(x):
    return None if x is None else x.to(DEV)


def gpu_sample(logits, t=None, k=None, p=None, u=None, probs=False, pool=None, rows=None,
               cols=None):
    L = logits if logits.is_cuda else logits.to(DEV)
    B, V = L.shape
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    q = torch.full((B, V), -1.0, dtype=torch.float32, device=DEV) if probs else None
    tok = pkv.sample_batch(L, _d(t), _d(k), _d(p), _d(u), probs_out=q, status=status,
                           token_pool=pool, wb_rows=_d(rows), wb_cols=_d(cols))
    torch.cuda.synchronize()
    return tok.cpu().numpy(), (q.cpu().numpy() if probs else None), int(status.item())


def test_page_example_rows():
    # "The engine and the sampler", section "Tests": [5,4,3,0,0,0] with
    # top_k=2, top_p=0.5 and a greedy row, over a grid of uniforms.
    logits = torch.tensor([[5.0, 4.0, 3.0, 0.0, 0.0, 0.0]] * 3)
    t = torch.tensor([1.0, 1.0, 0.0])
    k = torch.tensor([2, -1, -1], dtype=torch.int32)
    p = torch.tensor([1.0, 0.5, 1.0])
    q0 = 1.0 / (1.0 + np.exp(-1.0))
    for uu in np.linspace(0.0, 0.999, 37):
        u = torch.full((3,), float(uu))
        tok, q, st = gpu_sample(logits, t, k, p, u, probs=True)
        assert st == 0
        assert tok[0] == (0 if uu < q0 else 1) or abs(uu - q0) < 1e-5
        assert tok[1] == 0 and tok[2] == 0
        assert abs(q[0, 0] - q0) < 1e-5 and abs(q[0, 1] - (1 - q0)) < 1e-5
        assert q[1, 0] == 1.0


def test_pr1_workload_with_probs_and_writeback():
    w = workloads.pr1()
    pool = torch.zeros(w.pool_shape, dtype=torch.int32, device=DEV)
    tok, q, st = gpu_sample(w.logits, w.temperature, w.top_k, w.top_p, w.uniform, probs=True,
                            pool=pool, rows=w.wb_rows, cols=w.wb_cols)
    assert st == 0
    check_sampler(w.logits, w.temperature, w.top_k, w.top_p, w.uniform, tok, q)
    want = np.zeros(w.pool_shape, np.int32)
    oracle.writeback(tok, w.wb_rows, w.wb_cols, want)
    np.testing.assert_array_equal(pool.cpu().numpy(), want)


SHAPES = [(1, 1), (3, 5), (2, 31), (4, 33), (5, 1000), (3, 4097), (2, 20000), (2, 70001)]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("B,V", SHAPES)
@pytest.mark.parametrize("discrete", [False, True])
def test_random_shapes(dtype, B, V, discrete):
    seed = 7 * V + B + (1 if discrete else 0) + (3 if dtype == torch.bfloat16 else 0)
    logits = workloads.random_rows(B, V, dtype, seed=seed, discrete=discrete)
    t, k, p, u = workloads.random_params(B, seed=seed + 1, k_values=(-1, 1, 2, V - 1, V, V + 5, 20),
                                         p_values=(1.0, 1e-6, 0.5, 0.9, 0.95))
    tok, q, st = gpu_sample(logits, t, k, p, u, probs=True)
    assert st == 0
    check_sampler(logits, t, k, p, u, tok, q)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_every_row_kind_in_one_batch(dtype):
    # Rows cycle through greedy, top-k only, top-p only, both, neither.
    B, V = 40, 50000
    logits = workloads.random_rows(B, V, dtype, seed=11, scale=3.0)
    t = torch.tensor([0.0, 0.8, 1.2, 0.5, 1.0] * 8)
    k = torch.tensor([-1, 50, -1, 20, -1] * 8, dtype=torch.int32)
    p = torch.tensor([1.0, 1.0, 0.9, 0.95, 1.0] * 8)
    u = torch.rand(B, generator=torch.Generator().manual_seed(12))
    tok, q, st = gpu_sample(logits, t, k, p, u, probs=True)
    assert st == 0
    check_sampler(logits, t, k, p, u, tok, q)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_batch_beyond_the_cost_order(dtype):
    # More rows than the stream kernel orders by cost (4096): items are then
    # taken in row order from one queue.
    B, V = 5000, 4096
    seed = 31 + (1 if dtype == torch.bfloat16 else 0)
    logits = workloads.random_rows(B, V, dtype, seed=seed)
    t, k, p, u = workloads.random_params(B, seed=seed + 2, k_values=(-1, 1, 20, 300, V),
                                         p_values=(1.0, 0.5, 0.9, 0.95))
    tok, _, st = gpu_sample(logits, t, k, p, u)
    assert st == 0
    stats = check_sampler(logits, t, k, p, u, tok, None)
    _every_row_checked(stats, B)


def test_maximum_batch():
    B, V = 65535, 40
    logits = workloads.random_rows(B, V, torch.bfloat16, seed=41, discrete=True)
    t, k, p, u = workloads.random_params(B, seed=42, k_values=(-1, 1, 5, V),
                                         p_values=(1.0, 0.5, 0.9))
    tok, _, st = gpu_sample(logits, t, k, p, u)
    assert st == 0
    stats = check_sampler(logits, t, k, p, u, tok, None)
    _every_row_checked(stats, B)


@pytest.mark.parametrize("dtype,V", [(torch.float32, pkv.PKV_MAX_VOCAB_FP32),
                                     (torch.bfloat16, pkv.PKV_MAX_VOCAB_BF16)])
def test_rows_at_the_vocab_limit(dtype, V):
    # Greedy, top-k, top-p, top-k with top-p, and plain rows at the largest V.
    logits = workloads.random_rows(5, V, dtype, seed=51, scale=2.0)
    t = torch.tensor([0.0, 0.9, 1.1, 0.7, 1.0])
    k = torch.tensor([-1, 40, -1, 500, -1], dtype=torch.int32)
    p = torch.tensor([1.0, 1.0, 0.9, 0.8, 1.0])
    u = torch.rand(5, generator=torch.Generator().manual_seed(52))
    tok, q, st = gpu_sample(logits, t, k, p, u, probs=True)
    assert st == 0
    stats = check_sampler(logits, t, k, p, u, tok, q)
    _every_row_checked(stats, 5)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_unaligned_rows_take_the_scalar_path(dtype):
    B, V = 6, 3001
    base = workloads.random_rows(B, V + 1, dtype, seed=21)
    base_d = base.to(DEV)
    # Row stride V + 1 is not a multiple of 16 bytes; the first view also
    # starts one element in.
    for lo in (1, 0):
        view = base_d[:, lo:lo + V]
        assert view.stride(0) == V + 1
        t, k, p, u = workloads.random_params(B, seed=22 + lo)
        tok, q, st = gpu_sample(view, t, k, p, u, probs=True)
        assert st == 0
        check_sampler(base[:, lo:lo + V].contiguous(), t, k, p, u, tok, q)


def test_all_greedy_batch_with_ties():
    w = workloads.greedy()
    L = w.logits[:, :50000].contiguous()
    tok, q, st = gpu_sample(L, probs=True)
    assert st == 0
    np.testing.assert_array_equal(tok, np.argmax(L.float().numpy(), axis=1))


def test_ties_at_topk_and_topp_boundaries():
    # Many equal logits straddle the k-th position and the top-p cut.
    B, V = 8, 9000
    g = torch.Generator().manual_seed(31)
    x = torch.randint(0, 6, (B, V), generator=g).to(torch.float32)
    t = torch.full((B,), 1.0)
    k = torch.tensor([3, 100, 2000, 8999, -1, -1, 700, 1], dtype=torch.int32)
    p = torch.tensor([1.0, 1.0, 0.5, 0.3, 0.5, 0.77, 0.9, 1.0])
    u = torch.rand(B, generator=g)
    for dtype in (torch.float32, torch.bfloat16):
        L = x.to(dtype)
        tok, q, st = gpu_sample(L, t, k, p, u, probs=True)
        assert st == 0
        check_sampler(L, t, k, p, u, tok, q)


def test_neg_inf_and_extremes():
    B, V = 6, 3000
    x = workloads.random_rows(B, V, torch.float32, seed=41)
    x[0, ::2] = float("-inf")
    x[1, :] = float("-inf")
    x[1, 1234] = 0.5                     # a single finite logit
    x[2, 100:] = float("-inf")           # k larger than the finite count
    t = torch.tensor([1.0, 0.7, 1.0, 1e-7, 5.0, 1.0])
    k = torch.tensor([-1, -1, 500, -1, 3, 1], dtype=torch.int32)
    p = torch.tensor([0.9, 1.0, 1.0, 1.0, 1e-6, 1.0])
    u = torch.tensor([0.3, 0.999, 0.5, 0.7, 0.0, 0.9999])
    tok, q, st = gpu_sample(x, t, k, p, u, probs=True)
    assert st == 0
    check_sampler(x, t, k, p, u, tok, q)


def test_error_rows_set_status_and_skip_writes():
    B, V = 4, 1000
    x = workloads.random_rows(B, V, torch.float32, seed=51)
    x[0, 7] = float("nan")
    x[1, :] = float("-inf")
    x[2, 3] = float("inf")
    t = torch.tensor([1.0, 1.0, 1.0, 1.0])
    u = torch.tensor([0.5, 0.5, 0.5, 1.5])
    pool = torch.zeros((4, 8), dtype=torch.int32, device=DEV)
    rows = torch.arange(4, dtype=torch.int32)
    cols = torch.tensor([1, 2, 3, 4], dtype=torch.int64)
    tok, _, st = gpu_sample(x, t, None, None, u, pool=pool, rows=rows, cols=cols)
    ores = oracle.sample(x, t, None, None, u)
    np.testing.assert_array_equal(tok[:3], [-1, -1, -1])
    assert st == (1 | 2 | 16)
    assert tok[3] == ores["tokens"][3]  # u clamped below 1
    got = pool.cpu().numpy()
    assert got[0, 1] == 0 and got[1, 2] == 0 and got[2, 3] == 0 and got[3, 4] == tok[3]
    # greedy NaN row
    tok, _, st = gpu_sample(x[:1], None)
    assert tok[0] == -1 and st == 1


def test_writeback_bounds_and_skip():
    B, V = 4, 256
    x = workloads.random_rows(B, V, torch.bfloat16, seed=61)
    pool = torch.zeros((3, 5), dtype=torch.int32, device=DEV)
    rows = torch.tensor([0, 7, 1, 2], dtype=torch.int32)
    cols = torch.tensor([0, 1, 9, -1], dtype=torch.int64)
    tok, _, st = gpu_sample(x, None, pool=pool, rows=rows, cols=cols)
    assert st == (4 | 8)
    want = np.zeros((3, 5), np.int32)
    want[0, 0] = tok[0]
    np.testing.assert_array_equal(pool.cpu().numpy(), want)


def test_deterministic_across_calls():
    w = workloads.mixed(B=32)
    a, _, _ = gpu_sample(w.logits, w.temperature, w.top_k, w.top_p, w.uniform)
    b, _, _ = gpu_sample(w.logits, w.temperature, w.top_k, w.top_p, w.uniform)
    np.testing.assert_array_equal(a, b)


def test_workspace_header_is_checked_and_repaired():
    # A workspace whose header was never initialised (here: both ticket
    # counters past every item) hands out no queued item, so the rows those
    # items belong to have stale records: their tokens are -1 with status bit
    # 64 and nothing is written back for them.  Rows the kernel starts on
    # without a ticket (the first item of every producer) may still be
    # settled, and then exactly.  The call leaves the header reset, and the
    # next call on it is exact.
    w = workloads.mixed(B=400, V=32768)
    B, V = w.logits.shape
    ws = torch.zeros(pkv.sample_workspace_bytes(B, V, w.logits.dtype), dtype=torch.uint8,
                     device=DEV)
    hdr = ws[:16].view(torch.int32)
    hdr[0] = 0x7FFFFF00  # ticket (main queue)
    hdr[2] = 7           # calls
    hdr[3] = 0x7FFFFF00  # ticket (count-histogram queue)
    L = w.logits.to(DEV)
    args = (_d(w.temperature), _d(w.top_k), _d(w.top_p), _d(w.uniform))
    pool = torch.zeros((B, 64), dtype=torch.int32, device=DEV)
    rows = torch.arange(B, dtype=torch.int32)
    cols = torch.zeros(B, dtype=torch.int64)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    tok = pkv.sample_batch(L, *args, token_pool=pool, wb_rows=_d(rows), wb_cols=_d(cols),
                           status=status, workspace=ws)
    torch.cuda.synchronize()
    tok = tok.cpu().numpy()
    failed = tok == -1
    assert failed.any()
    assert int(status.item()) & pkv.ST_TIMEOUT
    written = pool.cpu().numpy()[:, 0]
    assert (written[failed] == 0).all()
    ok = np.nonzero(~failed)[0]
    if len(ok):
        sub = lambda x: None if x is None else x[ok]  # noqa: E731
        check_sampler(w.logits[ok], sub(w.temperature), sub(w.top_k), sub(w.top_p),
                      sub(w.uniform), tok[ok])
    assert hdr.cpu().tolist()[:4] == [0, 0, 8, 0]
    status.zero_()
    tok = pkv.sample_batch(L, *args, status=status, workspace=ws)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    check_sampler(w.logits, w.temperature, w.top_k, w.top_p, w.uniform, tok.cpu().numpy())


def test_workspace_init_readies_a_dirty_buffer():
    w = workloads.mixed(B=16, V=20000)
    B, V = w.logits.shape
    ws = torch.full((pkv.sample_workspace_bytes(B, V, w.logits.dtype),), 0xA5, dtype=torch.uint8,
                    device=DEV)
    pkv.sample_workspace_init(ws)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    tok = pkv.sample_batch(w.logits.to(DEV), _d(w.temperature), _d(w.top_k), _d(w.top_p),
                           _d(w.uniform), status=status, workspace=ws)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    check_sampler(w.logits, w.temperature, w.top_k, w.top_p, w.uniform, tok.cpu().numpy())


# ---------------------------------------------------------------- full-size workloads


def _full(name, rows_checked=None, probs_rows=32):
    w = workloads.make(name)
    L = w.logits.to(DEV)
    B, V = L.shape
    pool = torch.zeros(w.pool_shape, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    tok = pkv.sample_batch(L, _d(w.temperature), _d(w.top_k), _d(w.top_p), _d(w.uniform),
                           token_pool=pool, wb_rows=_d(w.wb_rows), wb_cols=_d(w.wb_cols),
                           status=status)
    torch.cuda.synchronize()
    tok = tok.cpu().numpy()
    assert int(status.item()) == 0
    sel = np.arange(B) if rows_checked is None else rows_checked
    sub = lambda x: None if x is None else x[sel]  # noqa: E731
    stats = check_sampler(w.logits[sel], sub(w.temperature), sub(w.top_k), sub(w.top_p),
                          sub(w.uniform), tok[sel])
    # The fused write-back equals a scatter of the GPU's own tokens.
    want = np.zeros(w.pool_shape, np.int32)
    oracle.writeback(tok, w.wb_rows, w.wb_cols, want)
    np.testing.assert_array_equal(pool.cpu().numpy(), want)
    # Kept-set probabilities on a subset of rows, through the debug output.
    pr = sel[:probs_rows]
    q = torch.empty((len(pr), V), dtype=torch.float32, device=DEV)
    sub2 = lambda x: None if x is None else x[pr].to(DEV)  # noqa: E731
    tok2 = pkv.sample_batch(L[torch.as_tensor(pr, device=DEV)], sub2(w.temperature),
                            sub2(w.top_k), sub2(w.top_p), sub2(w.uniform), probs_out=q)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(tok2.cpu().numpy(), tok[pr])
    sub3 = lambda x: None if x is None else x[pr]  # noqa: E731
    check_sampler(w.logits[pr], sub3(w.temperature), sub3(w.top_k), sub3(w.top_p),
                  sub3(w.uniform), tok[pr], q.cpu().numpy())
    return stats


def _every_row_checked(stats, B):
    # Every row is either exact (greedy or sampled) or excused and validated.
    assert stats["greedy"] + stats["exact"] + stats["validated"] == B, stats
    assert stats["validated"] == (stats["excused_cdf"] + stats["excused_topp"]
                                  + stats["excused_minp"]), stats


def test_full_greedy():
    stats = _full("greedy")
    assert stats["greedy"] == 64


def test_full_mixed():
    stats = _full("mixed")
    _every_row_checked(stats, 256)
    assert stats["exact"] + stats["greedy"] >= 200, stats


def test_full_nucleus():
    stats = _full("nucleus")
    _every_row_checked(stats, 256)
    assert stats["exact"] >= 200, stats


def test_full_large_every_row():
    stats = _full("large", probs_rows=16)
    _every_row_checked(stats, 1024)
    assert stats["exact"] >= 900, stats
