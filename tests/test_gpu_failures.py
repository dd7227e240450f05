"""Failure detection without a GPU fault.

Device side: the library's spin-waits are bounded by %globaltimer and report
through a status word; the wait probe makes one such wait run out on purpose
(a barrier nothing arrives on) and the context must stay usable.  Host side:
a failure injected into one host component (loader, D2H, accumulator, Adam)
aborts the step with MT_EINTERNAL, a stalled loader makes the compute
thread's bounded wait return MT_ETIMEDOUT; either way the handle still hands
out its tiles, refuses further steps, frees cleanly, and a fresh handle on the
same device trains as before."""
import time

import pytest
import torch

import mt_inputs

pytestmark = pytest.mark.gpu

hms = pytest.importorskip("host_memory_streamed_gb300")
from host_memory_streamed_gb300 import _lib, ops  # noqa: E402

SHAPE = mt_inputs.PRESETS["tiny"]


def _one_step(**kw):
    m = hms.StreamedDecoder.from_shape(SHAPE, **kw)
    m.load_weights(mt_inputs.model_weights(SHAPE))
    loss = m.train_step(mt_inputs.step_tokens(SHAPE, 1))
    w = m.weights()
    m.close()
    return loss, w


def test_device_wait_probe_times_out_and_context_stays_usable():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    ops.wait_probe(status, 50_000_000)  # 50 ms
    torch.cuda.synchronize()
    assert int(status.item()) == _lib.MT_STATUS_WAIT_PROBE
    assert time.time() - t0 < 30
    g = torch.Generator().manual_seed(3)
    A = torch.randn(300, 128, generator=g).to(torch.bfloat16)
    B = torch.randn(200, 128, generator=g).to(torch.bfloat16)
    out = torch.empty(300, 200, dtype=torch.bfloat16, device="cuda")
    ops.gemm(A.cuda(), B.cuda(), out)
    torch.cuda.synchronize()
    ref = A.double() @ B.double().T
    assert float((out.cpu().double() - ref).norm() / ref.norm()) < 4e-3


@pytest.mark.parametrize("what", [_lib.MT_INJECT_LOADER_FAIL, _lib.MT_INJECT_D2H_FAIL, _lib.MT_INJECT_ACCUM_FAIL,
                                  _lib.MT_INJECT_ADAM_FAIL])
def test_injected_host_failure_aborts_the_step_cleanly(what):
    ref_loss, ref_w = _one_step()
    m = hms.StreamedDecoder.from_shape(SHAPE)
    m.load_weights(mt_inputs.model_weights(SHAPE))
    m.debug_inject(what, 2)
    tokens = mt_inputs.step_tokens(SHAPE, 1)
    with pytest.raises(hms.MtError) as ei:
        m.train_step(tokens)
    assert ei.value.code == _lib.MT_EINTERNAL and "injected" in str(ei.value)
    m.weights()  # the tiles are still readable
    with pytest.raises(hms.MtError) as e2:
        m.train_step(tokens)
    assert e2.value.code == _lib.MT_ESTATE
    m.close()
    loss, w = _one_step()
    assert loss == ref_loss
    for n in ref_w["layers"][0]:
        assert torch.equal(w["layers"][0][n], ref_w["layers"][0][n]), n


def test_loader_stall_times_out_on_the_host():
    m = hms.StreamedDecoder.from_shape(SHAPE, timeout_ms=1500)
    m.load_weights(mt_inputs.model_weights(SHAPE))
    m.debug_inject(_lib.MT_INJECT_LOADER_STALL, 2)
    t0 = time.time()
    with pytest.raises(hms.MtError) as ei:
        m.train_step(mt_inputs.step_tokens(SHAPE, 1))
    assert ei.value.code == _lib.MT_ETIMEDOUT
    assert time.time() - t0 < 60
    m.close()
    loss, _ = _one_step()
    assert loss == loss  # a fresh handle steps normally


def test_an_injection_arms_one_step_only():
    """An injection whose visit is never reached expires with its step."""
    m = hms.StreamedDecoder.from_shape(SHAPE)
    m.load_weights(mt_inputs.model_weights(SHAPE))
    m.debug_inject(_lib.MT_INJECT_LOADER_FAIL, 10_000)
    m.train_step(mt_inputs.step_tokens(SHAPE, 1))
    m.debug_inject(_lib.MT_INJECT_NONE, 0)
    m.train_step(mt_inputs.step_tokens(SHAPE, 2))
    m.close()


def test_adam_failure_after_an_async_step_returns_is_reported():
    """MT_ASYNC_ADAM: a step may return before its Adam updates finish; an
    injected Adam failure then surfaces at the next call that waits for them
    (mt_sync here), never silently."""
    m = hms.StreamedDecoder.from_shape(SHAPE, flags=_lib.MT_ASYNC_ADAM)
    m.load_weights(mt_inputs.model_weights(SHAPE))
    m.debug_inject(_lib.MT_INJECT_ADAM_FAIL, 2)
    tokens = mt_inputs.step_tokens(SHAPE, 1)
    with pytest.raises(hms.MtError) as ei:
        m.train_step(tokens)
        m.sync()
    assert ei.value.code == _lib.MT_EINTERNAL and "injected" in str(ei.value)
    m.weights()  # the tiles are still readable
    with pytest.raises(hms.MtError):
        m.train_step(tokens)
    m.close()
