"""Where BF16 storage alone puts the gradients, with no kernel involved (CPU).

The target fixes the GEMMs as BF16 tensor-core GEMMs, so the normalised
activations and q/k/v reach the tensor cores as BF16.  The storage-precision
model (tests/precision_model.py: the step in FP32, rounded to BF16 exactly
where the library stores BF16) is compared with the FP64 oracle on a proxy of
the 14B width: d_model 5120 with N(0, 0.02) weights (score standard deviation
near 2, as in the 14B-shaped workload), two layers, 200 tokens, with fewer
heads, a narrow MLP and a small vocabulary so that the test runs in seconds.

Any implementation with those storage points lands past the normwise 2e-2
bound on the last layer's attention-side gradients at this width; keeping
the normalised activations and q/k/v in FP32 brings every gradient within
it; at the 1.3B width (d 2048) BF16 storage stays within it.  This pins, on
the CPU, why the full-width 14B and 7B checks on the GPU report an expected
failure while naming both the library's and this model's errors.
"""
import pytest

import mt_inputs
import oracle
from oracle import OracleConfig
from tests import parity
from tests import precision_model as pm

GRAD_RTOL, GRAD_COS = 2e-2, 0.999


def _errors(name, drop=()):
    s = mt_inputs.PRESETS[name].with_(n_layers=2, batch=1, seq=200, vocab=1024, n_heads=8, n_kv_heads=2,
                                      ffn=1024)
    cfg = OracleConfig.from_shape(s)
    params = mt_inputs.model_weights(s, gain_jitter=0.1)
    tokens = mt_inputs.step_tokens(s, 1)
    _, gref = oracle.model_loss_and_grads(params, tokens, cfg)
    _, g = pm.Model(pm.ALL - set(drop)).loss_and_grads(params, tokens, cfg)
    return {n: (c, r) for n, c, r in parity.grad_report(g, gref)}


@pytest.fixture(scope="module")
def width_5120():
    return _errors("14b"), _errors("14b", drop=("n", "qkv"))


def test_bf16_storage_exceeds_the_bound_at_width_5120(width_5120):
    """All storage points in BF16: the last layer's q/k projections (and its
    attention norm gain) land past 2e-2, though still with cosine >= 0.999."""
    err, _ = width_5120
    worst = max(err, key=lambda n: err[n][1])
    assert err[worst][1] > GRAD_RTOL, err[worst]
    assert worst in ("layers.1.wq", "layers.1.wk", "layers.1.g1"), worst
    assert err["layers.1.wq"][1] > GRAD_RTOL and err["layers.1.wk"][1] > GRAD_RTOL
    assert min(c for c, _ in err.values()) >= GRAD_COS


def test_fp32_norm_outputs_and_qkv_meet_the_bound_at_width_5120(width_5120):
    """The same step with only the normalised activations and q/k/v kept in
    FP32 (every other storage point still BF16): every gradient within 2e-2.
    The excess comes from those two tensor-core operands."""
    _, err = width_5120
    worst = max(err, key=lambda n: err[n][1])
    assert err[worst][1] <= GRAD_RTOL, (worst, err[worst])


def test_bf16_storage_meets_the_bound_at_width_2048():
    """At the 1.3B width every gradient meets the bound with every storage
    point in BF16."""
    err = _errors("1.3b")
    worst = max(err, key=lambda n: err[n][1])
    assert err[worst][1] <= GRAD_RTOL and min(c for c, _ in err.values()) >= GRAD_COS, (worst, err[worst])
