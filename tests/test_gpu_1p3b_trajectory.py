"""Ten streamed training steps at the 1.3B workload's width against the oracle.

The 1.3B-shaped decoder (d 2048, 16 heads x 128, ffn 5632, vocab 32000) at
reduced depth and token count (2 layers, block recompute every 2 layers,
2 x 136 tokens): the library and the oracle each run their own ten-step
trajectory from the same BF16 weights on the same token batches, and at every
step the loss and every gradient tensor must meet the step tolerances (loss
relative error <= 1e-2; each gradient cosine >= 0.999 and normwise relative
error <= 2e-2).  Adam makes the two trajectories drift apart only by the
rounding of updated BF16 weights, which this checks stays within those
tolerances over the steps.  Named to be collected before the slow full-size
cases.
"""
import pytest
import torch

import mt_inputs
import oracle
from oracle import OracleConfig
from tests import parity

pytestmark = pytest.mark.gpu

hms = pytest.importorskip("host_memory_streamed_gb300")

STEPS = 10


def test_ten_step_trajectory_at_1p3b_width_matches_oracle():
    s = mt_inputs.PRESETS["1.3b"].with_(n_layers=2, ckpt_every=2, batch=2, seq=136)
    cfg = OracleConfig.from_shape(s)
    params = mt_inputs.model_weights(s, gain_jitter=0.1)
    m = hms.StreamedDecoder.from_shape(s)
    state = None
    losses = []
    try:
        m.load_weights(params)
        for n in range(1, STEPS + 1):
            tok = mt_inputs.step_tokens(s, n)
            loss = m.train_step(tok)
            g_lib = m.grads()
            loss_ref, grads, params, state = oracle.train_step(params, state, tok, n, cfg)
            losses.append((loss, loss_ref))
            assert abs(loss - loss_ref) <= parity.LOSS_RTOL * abs(loss_ref), (n, loss, loss_ref)
            rep = parity.grad_report(g_lib, grads)
            worst = max(r for _, _, r in rep)
            print(f"step {n}: loss {loss:.6f} oracle {loss_ref:.6f}; worst gradient rel {worst:.4f}")
            bad = [(name, c, r) for name, c, r in rep if not (c >= parity.GRAD_COS and r <= parity.GRAD_RTOL)]
            assert not bad, (n, bad)
            del g_lib, grads
        assert m.step == STEPS
    finally:
        m.close()
    # the two trajectories stay together to the end
    assert abs(losses[-1][0] - losses[-1][1]) <= parity.LOSS_RTOL * abs(losses[-1][1])
