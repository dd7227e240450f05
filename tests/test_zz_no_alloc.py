"""RMSNorm backward without any device allocation, checked against the entry
point that takes a caller-provided scratch buffer.

Some callers of this library cannot allocate device memory: a host
application that reserves the GPU's whole memory budget up front and forbids
further allocation, or a latency-critical loop in which a cudaMalloc (which can
synchronise the device) is not acceptable.  mt_op_rmsnorm_bwd_noalloc serves
them from a fixed array inside the library.  The file name makes pytest
collect it last, so a run that stops at the first failure has run every other
test before this one.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

hms = pytest.importorskip("host_memory_streamed_gb300")
from host_memory_streamed_gb300 import _lib  # noqa: E402

DEV = "cuda"


def _rel(a, b):
    a, b = a.double(), b.double()
    return float((a - b).norm() / b.norm().clamp_min(1e-300))


def _inputs(rows, d, seed):
    g = torch.Generator().manual_seed(seed)
    bf = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16).to(DEV)
    x, dy, dres = bf(rows, d), bf(rows, d), bf(rows, d)
    w = (1 + 0.1 * torch.randn(d, generator=g)).to(torch.bfloat16).to(DEV)
    rstd = torch.rsqrt(x.float().pow(2).mean(-1) + 1e-5).contiguous()
    return dy, x, w, rstd, dres


def _ptr(t):
    return None if t is None else t.data_ptr()


def _with_caller_scratch(dy, x, w, rstd, dres, stream=None):
    L = _lib.lib()
    rows, d = x.shape
    dx = torch.empty_like(x)
    dg = torch.empty(d, device=DEV, dtype=torch.bfloat16)
    scratch = torch.empty(L.mt_op_rmsnorm_bwd_scratch_floats(rows, d), device=DEV)
    rc = L.mt_op_rmsnorm_bwd(dy.data_ptr(), x.data_ptr(), w.data_ptr(), rstd.data_ptr(), _ptr(dres),
                             dx.data_ptr(), dg.data_ptr(), scratch.data_ptr(), rows, d, stream)
    assert rc == 0, L.mt_op_last_error()
    return dx, dg


def _without_allocation(dy, x, w, rstd, dres, stream=None):
    L = _lib.lib()
    rows, d = x.shape
    dx = torch.empty_like(x)
    dg = torch.empty(d, device=DEV, dtype=torch.bfloat16)
    rc = L.mt_op_rmsnorm_bwd_noalloc(dy.data_ptr(), x.data_ptr(), w.data_ptr(), rstd.data_ptr(), _ptr(dres),
                                     dx.data_ptr(), dg.data_ptr(), rows, d, stream)
    assert rc == 0, L.mt_op_last_error()
    return dx, dg


def test_noalloc_matches_caller_scratch_on_two_calls_in_a_row():
    # two calls with different shapes: the second must not see the first's scratch contents
    for rows, d, seed in ((1000, 5120, 1), (4096, 1024, 2)):
        args = _inputs(rows, d, seed)
        ref_dx, ref_dg = _with_caller_scratch(*args)
        dx, dg = _without_allocation(*args)
        torch.cuda.synchronize()
        assert _rel(dx, ref_dx) <= 4e-3 and _rel(dg, ref_dg) <= 4e-3
        assert torch.equal(dx, ref_dx) and torch.equal(dg, ref_dg)  # same kernels, same order


def test_noalloc_at_exactly_its_limit():
    """ceil(rows/64) * d == 4,194,304 floats, the whole fixed array: accepted,
    and identical to the caller-scratch entry point."""
    rows, d = 64 * 1024, 4096
    args = _inputs(rows, d, 3)
    ref_dx, ref_dg = _with_caller_scratch(*args)
    dx, dg = _without_allocation(*args)
    torch.cuda.synchronize()
    assert torch.equal(dx, ref_dx) and torch.equal(dg, ref_dg)


def test_noalloc_on_a_side_stream_without_residual():
    """dres = NULL, both calls on a non-default stream: still identical."""
    dy, x, w, rstd, _ = _inputs(700, 2048, 4)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ref_dx, ref_dg = _with_caller_scratch(dy, x, w, rstd, None, side.cuda_stream)
        dx, dg = _without_allocation(dy, x, w, rstd, None, side.cuda_stream)
    side.synchronize()
    assert torch.equal(dx, ref_dx) and torch.equal(dg, ref_dg)


def test_noalloc_rejects_widths_beyond_the_kernels_plan():
    L = _lib.lib()
    t = torch.zeros(8, device=DEV, dtype=torch.bfloat16)
    rc = L.mt_op_rmsnorm_bwd_noalloc(t.data_ptr(), t.data_ptr(), t.data_ptr(), t.data_ptr(), None, t.data_ptr(),
                                     t.data_ptr(), 1, 1 << 20, None)
    assert rc == _lib.MT_EINVAL
    assert b"widest row" in L.mt_op_last_error()


def test_noalloc_rejects_row_counts_that_would_overflow():
    L = _lib.lib()
    t = torch.zeros(8, device=DEV, dtype=torch.bfloat16)
    rc = L.mt_op_rmsnorm_bwd_noalloc(t.data_ptr(), t.data_ptr(), t.data_ptr(), t.data_ptr(), None, t.data_ptr(),
                                     t.data_ptr(), (1 << 63) - 1, 8, None)
    assert rc == _lib.MT_EINVAL


def test_noalloc_rejects_sizes_beyond_its_fixed_scratch():
    L = _lib.lib()
    rows, d = 64 * 1025, 4096  # ceil(rows/64) * d = 4,198,400 > 4,194,304
    t = torch.zeros(8, device=DEV, dtype=torch.bfloat16)
    rc = L.mt_op_rmsnorm_bwd_noalloc(t.data_ptr(), t.data_ptr(), t.data_ptr(), t.data_ptr(), None, t.data_ptr(),
                                     t.data_ptr(), rows, d, None)
    assert rc == _lib.MT_EINVAL
    assert b"exceeds the fixed scratch" in L.mt_op_last_error()
