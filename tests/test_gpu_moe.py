"""MoE MLP on the device (routing, counting sort, gather, the grouped expert
GEMMs, combine and their backward) against the FP64 MoE oracle."""
import pytest
import torch

from oracle import moe

pytestmark = pytest.mark.gpu

hms = pytest.importorskip("host_memory_streamed_gb300")
from host_memory_streamed_gb300 import ops  # noqa: E402

D = torch.float64
DEV = "cuda"


def rel(a, b):
    a, b = a.to(D).cpu(), b.to(D).cpu()
    return float((a - b).norm() / b.norm().clamp_min(1e-300))


def cos(a, b):
    a, b = a.to(D).cpu().reshape(-1), b.to(D).cpu().reshape(-1)
    return float(a @ b / (a.norm() * b.norm()).clamp_min(1e-300))


@pytest.mark.parametrize("N,E,k", [(300, 8, 2), (1000, 64, 4), (37, 5, 5), (128, 256, 8)])
def test_route_and_sort(N, E, k):
    g = torch.Generator().manual_seed(N + E + k)
    logits = torch.randn(N, E, generator=g)
    logits[0, :] = 0.5  # one token whose logits all tie: the lower ids win
    idx, gates, order, pos, offsets = ops.moe_route(logits.to(DEV), k)
    torch.cuda.synchronize()
    _, idx_ref, gates_ref = moe.moe_route(logits.to(D), torch.eye(E, dtype=D), k)  # x = logits, W_r = I
    assert torch.equal(idx.cpu().long(), idx_ref)
    assert torch.allclose(gates.cpu().to(D), gates_ref, rtol=1e-5, atol=1e-7)
    flat = idx.cpu().reshape(-1).long()
    order, pos, offsets = order.cpu().long(), pos.cpu().long(), offsets.cpu().long()
    assert torch.equal(offsets, torch.cat([torch.zeros(1, dtype=torch.long), torch.bincount(flat, minlength=E).cumsum(0)]))
    assert torch.equal(pos[order], torch.arange(N * k))
    for e in range(E):
        seg = order[offsets[e]:offsets[e + 1]]
        assert torch.all(flat[seg] == e) and torch.all(seg[1:] > seg[:-1])  # stable: pair order kept


def _moe_weights(E, d, Fh, seed):
    g = torch.Generator().manual_seed(seed)
    wr = (torch.randn(E, d, generator=g) * 0.3).to(torch.bfloat16)
    wg = (torch.randn(E, Fh, d, generator=g) * 0.05).to(torch.bfloat16)
    wu = (torch.randn(E, Fh, d, generator=g) * 0.05).to(torch.bfloat16)
    wd = (torch.randn(E, d, Fh, generator=g) * 0.05).to(torch.bfloat16)
    wgu = torch.stack([wg, wu], dim=2).reshape(E, 2 * Fh, d)  # gate/up rows interleaved
    experts = [{"wg": wg[e].to(D), "wu": wu[e].to(D), "wd": wd[e].to(D)} for e in range(E)]
    return wr, wgu, wd, experts


@pytest.mark.parametrize("N,E,k,d,Fh", [(256, 8, 2, 128, 96), (200, 16, 4, 64, 136)])
def test_moe_mlp_matches_oracle(N, E, k, d, Fh):
    wr, wgu, wd, experts = _moe_weights(E, d, Fh, N + E)
    g = torch.Generator().manual_seed(5)
    x = torch.randn(N, d, generator=g).to(torch.bfloat16)
    dy = (torch.randn(N, d, generator=g) * 0.1).to(torch.bfloat16)
    y, saved = ops.moe_mlp_forward(x.to(DEV), wr.to(DEV), wgu.to(DEV), wd.to(DEV), k)
    dx, dwr, dwgu, dwd = ops.moe_mlp_backward(dy.to(DEV), x.to(DEV), wr.to(DEV), wgu.to(DEV), wd.to(DEV), k, saved)
    torch.cuda.synchronize()
    y_ref, cache = moe.moe_mlp_forward(x.to(D), wr.to(D), experts, k)
    # the selection is an integer decision: both sides must have made the same one
    assert torch.equal(saved["idx"].cpu().long(), cache["idx"])
    dx_ref, dwr_ref, dex_ref = moe.moe_mlp_backward(dy.to(D), x.to(D), wr.to(D), experts, k, cache)
    assert rel(y, y_ref) < 1e-2
    for mine, ref in [(dx, dx_ref), (dwr, dwr_ref)]:
        assert cos(mine, ref) > 0.999 and rel(mine, ref) < 2e-2
    dwg_ref = torch.stack([e["wg"] for e in dex_ref])
    dwu_ref = torch.stack([e["wu"] for e in dex_ref])
    dwd_ref = torch.stack([e["wd"] for e in dex_ref])
    dwgu_ref = torch.stack([dwg_ref, dwu_ref], dim=2).reshape(E, 2 * Fh, d)
    for mine, ref in [(dwgu, dwgu_ref), (dwd, dwd_ref)]:
        assert cos(mine, ref) > 0.999 and rel(mine, ref) < 2e-2


def test_moe_mlp_deterministic():
    N, E, k, d, Fh = 256, 8, 2, 128, 96
    wr, wgu, wd, _ = _moe_weights(E, d, Fh, 77)
    x = torch.randn(N, d, generator=torch.Generator().manual_seed(78)).to(torch.bfloat16).to(DEV)
    dy = torch.randn(N, d, generator=torch.Generator().manual_seed(79)).to(torch.bfloat16).to(DEV)
    outs = []
    for _ in range(2):
        y, saved = ops.moe_mlp_forward(x, wr.to(DEV), wgu.to(DEV), wd.to(DEV), k)
        grads = ops.moe_mlp_backward(dy, x, wr.to(DEV), wgu.to(DEV), wd.to(DEV), k, saved)
        outs.append([y] + list(grads))
    torch.cuda.synchronize()
    for a, b in zip(*outs):
        assert torch.equal(a, b)


# ------------------------------------------------------------------ padded routing and grouped GEMMs
@pytest.mark.parametrize("N,E,k", [(300, 8, 2), (128, 256, 8), (1000, 64, 4)])
def test_route_padded(N, E, k):
    """row_align = 64: the same stable order per expert as the unpadded sort,
    each expert's range padded to a multiple of 64 with order = -1."""
    g = torch.Generator().manual_seed(7 * N + E)
    logits = torch.randn(N, E, generator=g).to(DEV)
    idx, _, order, pos, offsets = ops.moe_route(logits, k, row_align=64)
    idx1, _, order1, _, offsets1 = ops.moe_route(logits, k)
    torch.cuda.synchronize()
    assert torch.equal(idx.cpu(), idx1.cpu())
    flat = idx.cpu().reshape(-1).long()
    counts = torch.bincount(flat, minlength=E)
    off, order, pos = offsets.cpu().long(), order.cpu().long(), pos.cpu().long()
    o1, f1 = order1.cpu().long(), offsets1.cpu().long()
    assert order.numel() == N * k + 63 * E
    assert torch.equal(off, torch.cat([torch.zeros(1, dtype=torch.long), ((counts + 63) // 64 * 64).cumsum(0)]))
    for e in range(E):
        assert torch.equal(order[off[e]:off[e] + counts[e]], o1[f1[e]:f1[e + 1]])
        assert torch.all(order[off[e] + counts[e]:off[e + 1]] == -1)
    assert torch.all(order[off[E]:] == -1)
    assert torch.equal(order[pos], torch.arange(N * k))


def _padded_offsets(counts, align=64):
    run, out = 0, [0]
    for c in counts:
        run += (c + align - 1) // align * align
        out.append(run)
    return torch.tensor(out, dtype=torch.int32)


@pytest.mark.parametrize("counts,N,K,b_mn", [
    ([0, 300, 1, 0, 64, 513, 0, 7], 200, 128, False),
    ([0, 300, 1, 0, 64, 513, 0, 7], 136, 192, True),
    ([1000], 96, 64, False),
    ([0] * 7 + [5], 384, 272, True),
])
def test_grouped_rows_gemm(counts, N, K, b_mn):
    """One launch over every group's rows against an FP64 product per group;
    rows past the last group are not written."""
    G = len(counts)
    off = _padded_offsets(counts)
    R = int(off[-1]) + 100
    g = torch.Generator().manual_seed(sum(counts) + N + K)
    A = torch.randn(R, K, generator=g).to(torch.bfloat16)
    B = (torch.randn(G, K, N, generator=g) if b_mn else torch.randn(G, N, K, generator=g)).to(torch.bfloat16)
    out = torch.full((R, N), 7.0, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ops.gemm_grouped_rows(A.to(DEV), B.to(DEV), off.to(DEV), out, b_mn=b_mn, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    out = out.cpu()
    for e in range(G):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 > r0:
            ref = A[r0:r1].to(D) @ (B[e].to(D) if b_mn else B[e].to(D).T)
            assert rel(out[r0:r1], ref) < 4e-3, e
    assert torch.all(out[int(off[-1]):] == 7.0)


@pytest.mark.parametrize("counts,M,N", [
    ([0, 300, 1, 0, 64, 513, 0, 7], 128, 96),
    ([1000], 256, 320),
    ([0, 0, 3], 192, 64),
])
def test_grouped_k_gemm(counts, M, N):
    """Weight-gradient grouping: C_g = A_g^T B_g over each group's (zero-padded)
    rows in one launch; a group without rows gets an exact zero block."""
    G = len(counts)
    off = _padded_offsets(counts)
    R = int(off[-1]) + 64
    g = torch.Generator().manual_seed(sum(counts) + M + N)
    A = torch.randn(R, M, generator=g).to(torch.bfloat16)
    B = torch.randn(R, N, generator=g).to(torch.bfloat16)
    for e, c in enumerate(counts):  # the padding rows of a routed buffer are zero
        A[int(off[e]) + c:int(off[e + 1])] = 0
        B[int(off[e]) + c:int(off[e + 1])] = 0
    out = torch.full((G, M, N), 7.0, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ops.gemm_grouped_k(A.to(DEV), B.to(DEV), off.to(DEV), out, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    out = out.cpu()
    for e in range(G):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 == r0:
            assert torch.all(out[e] == 0), e
        else:
            assert rel(out[e], A[r0:r1].to(D).T @ B[r0:r1].to(D)) < 4e-3, e


def test_moe_mlp_empty_experts_get_zero_gradients():
    """64 tokens, top-1 of 64 experts: most experts receive no row; their
    gradients are exactly zero and the rest match the oracle."""
    N, E, k, d, Fh = 64, 64, 1, 64, 64
    wr, wgu, wd, experts = _moe_weights(E, d, Fh, 91)
    g = torch.Generator().manual_seed(92)
    x = torch.randn(N, d, generator=g).to(torch.bfloat16)
    dy = (torch.randn(N, d, generator=g) * 0.1).to(torch.bfloat16)
    y, saved = ops.moe_mlp_forward(x.to(DEV), wr.to(DEV), wgu.to(DEV), wd.to(DEV), k)
    dx, dwr, dwgu, dwd = ops.moe_mlp_backward(dy.to(DEV), x.to(DEV), wr.to(DEV), wgu.to(DEV), wd.to(DEV), k, saved)
    torch.cuda.synchronize()
    y_ref, cache = moe.moe_mlp_forward(x.to(D), wr.to(D), experts, k)
    assert torch.equal(saved["idx"].cpu().long(), cache["idx"])
    used = torch.bincount(cache["idx"].reshape(-1), minlength=E) > 0
    assert not bool(used.all())
    assert torch.all(dwgu.cpu()[~used] == 0) and torch.all(dwd.cpu()[~used] == 0)
    dx_ref, dwr_ref, dex_ref = moe.moe_mlp_backward(dy.to(D), x.to(D), wr.to(D), experts, k, cache)
    assert rel(y, y_ref) < 1e-2
    dwd_ref = torch.stack([e["wd"] for e in dex_ref])
    # top-1: the gate is a softmax over one selected logit, identically 1, so
    # the router gets no gradient at all (on both sides, exactly)
    assert torch.all(dwr_ref == 0) and torch.all(dwr.cpu() == 0)
    for mine, ref in [(dx, dx_ref), (dwd, dwd_ref)]:
        assert cos(mine, ref) > 0.999 and rel(mine, ref) < 2e-2


# ------------------------------------------------------------------ MoE layers in the streamed step
def _moe_shape(E, k):
    import mt_inputs
    return mt_inputs.PRESETS["tiny"].with_(n_experts=E, top_k=k, ffn=136)


def _moe_run(s, steps=1, flags=0):
    import mt_inputs
    m = hms.StreamedDecoder.from_shape(s, flags=flags)
    params = mt_inputs.model_weights(s, gain_jitter=0.1)
    m.load_weights(params)
    out = {"params0": params, "loss": [], "w": [], "g": [], "mv": []}
    for n in range(1, steps + 1):
        out["loss"].append(m.train_step(mt_inputs.step_tokens(s, n)))
        out["w"].append(m.weights())
        out["g"].append(m.grads())
        out["mv"].append(m.moments())
    m.close()
    return out


def test_moe_step_with_every_expert_matches_oracle():
    """k = E: every token uses every expert, so no selection is involved and
    the step must match the oracle within the library's usual tolerances."""
    import mt_inputs
    from oracle import OracleConfig
    from tests import parity
    s = _moe_shape(8, 8)
    cfg = OracleConfig.from_shape(s)
    r = _moe_run(s)
    loss, grads = moe.moe_model_loss_and_grads(r["params0"], mt_inputs.step_tokens(s, 1), cfg, s.top_k)
    assert abs(r["loss"][0] - loss) <= parity.LOSS_RTOL * abs(loss)
    parity.assert_grads_close(r["g"][0], grads)
    m, v = r["mv"][0]
    parity.assert_adam_matches(r["w"][0], r["params0"], r["g"][0], m, v, 1, cfg)


def test_moe_step_top2_streamed_equals_resident_and_loss_close():
    """Top-2 of 16 experts: streamed == resident bit for bit (routing is
    deterministic), and the loss is the oracle's (a near-tie routed
    differently moves the loss by far less than the tolerance)."""
    import mt_inputs
    from oracle import OracleConfig
    from tests import parity
    s = _moe_shape(16, 2)
    a = _moe_run(s, steps=2)
    b = _moe_run(s, steps=2, flags=hms.MT_RESIDENT)
    assert a["loss"] == b["loss"]
    for (n, x), (_, y) in zip(parity.flat_named(a["w"][-1]), parity.flat_named(b["w"][-1])):
        assert torch.equal(x, y), n
    cfg = OracleConfig.from_shape(s)
    loss, _ = moe.moe_model_loss_and_grads(a["params0"], mt_inputs.step_tokens(s, 1), cfg, s.top_k)
    assert abs(a["loss"][0] - loss) <= parity.LOSS_RTOL * abs(loss)
