"""Pins of the MoE oracle (oracle/moe.py) against things other than itself."""
import math

import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import moe

D = torch.float64


def _weights(E, d, Fh, seed):
    g = torch.Generator().manual_seed(seed)
    wr = torch.randn(E, d, generator=g, dtype=D) * 0.5
    experts = [{"wg": torch.randn(Fh, d, generator=g, dtype=D) * 0.2,
                "wu": torch.randn(Fh, d, generator=g, dtype=D) * 0.2,
                "wd": torch.randn(d, Fh, generator=g, dtype=D) * 0.2} for _ in range(E)]
    return wr, experts


def _library_forward(x, wr, experts, k):
    """The same block written with torch.nn.functional and autograd-friendly
    ops: per token, gather the chosen experts' weights (no index_add_)."""
    s = F.linear(x, wr)
    idx = torch.sort(-s.detach(), dim=1, stable=True).indices[:, :k]
    g = torch.softmax(s.gather(1, idx), dim=1)
    Wg = torch.stack([e["wg"] for e in experts])  # [E, F, d]
    Wu = torch.stack([e["wu"] for e in experts])
    Wd = torch.stack([e["wd"] for e in experts])  # [E, d, F]
    out = torch.zeros_like(x)
    for j in range(k):
        e = idx[:, j]
        gate = torch.einsum("nfd,nd->nf", Wg[e], x)
        up = torch.einsum("nfd,nd->nf", Wu[e], x)
        out = out + g[:, j:j + 1] * torch.einsum("ndf,nf->nd", Wd[e], F.silu(gate) * up)
    return out


@pytest.mark.parametrize("E,k", [(8, 2), (6, 3), (4, 4)])
def test_moe_grads_match_autograd_of_library_forward(E, k):
    N, d, Fh = 40, 24, 20
    wr, experts = _weights(E, d, Fh, 1 + E + k)
    x = torch.randn(N, d, generator=torch.Generator().manual_seed(7), dtype=D)
    dy = torch.randn(N, d, generator=torch.Generator().manual_seed(8), dtype=D)
    y, cache = moe.moe_mlp_forward(x, wr, experts, k)
    dx, dwr, dex = moe.moe_mlp_backward(dy, x, wr, experts, k, cache)
    xl = x.clone().requires_grad_(True)
    wrl = wr.clone().requires_grad_(True)
    exl = [{n: t.clone().requires_grad_(True) for n, t in e.items()} for e in experts]
    yl = _library_forward(xl, wrl, exl, k)
    assert torch.allclose(y, yl.detach(), rtol=1e-12, atol=1e-12)
    (yl * dy).sum().backward()
    assert torch.allclose(dx, xl.grad, rtol=1e-10, atol=1e-12)
    assert torch.allclose(dwr, wrl.grad, rtol=1e-10, atol=1e-12)
    for mine, theirs in zip(dex, exl):
        for n in ("wg", "wu", "wd"):
            assert torch.allclose(mine[n], theirs[n].grad, rtol=1e-10, atol=1e-12), n


def test_moe_finite_differences():
    """Central differences of the oracle's own forward along random directions
    of (x, W_r, experts), small enough that no token's selection changes."""
    E, k, N, d, Fh = 6, 2, 16, 12, 10
    wr, experts = _weights(E, d, Fh, 21)
    x = torch.randn(N, d, generator=torch.Generator().manual_seed(22), dtype=D)
    dy = torch.randn(N, d, generator=torch.Generator().manual_seed(23), dtype=D)
    y, cache = moe.moe_mlp_forward(x, wr, experts, k)
    dx, dwr, dex = moe.moe_mlp_backward(dy, x, wr, experts, k, cache)
    gen = torch.Generator().manual_seed(24)
    for _ in range(3):
        ux = torch.randn(x.shape, generator=gen, dtype=D)
        ur = torch.randn(wr.shape, generator=gen, dtype=D)
        ue = [{n: torch.randn(t.shape, generator=gen, dtype=D) for n, t in e.items()} for e in experts]
        h = 1e-6

        def f(sign):
            ex = [{n: t + sign * h * ue[i][n] for n, t in e.items()} for i, e in enumerate(experts)]
            yy, c = moe.moe_mlp_forward(x + sign * h * ux, wr + sign * h * ur, ex, k)
            assert torch.equal(c["idx"], cache["idx"])  # the selection did not move
            return float((yy * dy).sum())

        fd = (f(1) - f(-1)) / (2 * h)
        an = float((dx * ux).sum() + (dwr * ur).sum() +
                   sum(float((dex[i][n] * ue[i][n]).sum()) for i in range(E) for n in ("wg", "wu", "wd")))
        assert abs(fd - an) <= 1e-6 * abs(an) + 1e-9, (fd, an)


def test_single_expert_is_the_dense_swiglu_mlp():
    """E = k = 1: the gate is 1 and the block is the dense SwiGLU MLP."""
    N, d, Fh = 10, 16, 12
    wr, experts = _weights(1, d, Fh, 31)
    x = torch.randn(N, d, generator=torch.Generator().manual_seed(32), dtype=D)
    y, _ = moe.moe_mlp_forward(x, wr, experts, 1)
    e = experts[0]
    dense = oracle.swiglu(x @ e["wg"].T, x @ e["wu"].T) @ e["wd"].T
    assert torch.allclose(y, dense, rtol=1e-13, atol=1e-15)


def test_relabelling_experts_changes_nothing():
    """Permuting the experts together with the router rows gives the same
    output (the routing depends on the logits, not on the labels)."""
    E, k, N, d, Fh = 7, 3, 30, 16, 12
    wr, experts = _weights(E, d, Fh, 41)
    x = torch.randn(N, d, generator=torch.Generator().manual_seed(42), dtype=D)
    perm = torch.randperm(E, generator=torch.Generator().manual_seed(43))
    y, c = moe.moe_mlp_forward(x, wr, experts, k)
    y2, c2 = moe.moe_mlp_forward(x, wr[perm], [experts[int(i)] for i in perm], k)
    assert torch.allclose(y, y2, rtol=1e-13, atol=1e-15)
    assert torch.equal(perm[c2["idx"]], c["idx"])
    assert torch.allclose(c["gates"].sum(1), torch.ones(N, dtype=D))


def test_ties_go_to_the_lower_expert_id():
    x = torch.ones(1, 4, dtype=D)
    wr = torch.tensor([[0.0] * 4, [1.0] * 4, [1.0] * 4, [0.5] * 4], dtype=D)  # logits 0, 4, 4, 2
    _, idx, gates = moe.moe_route(x, wr, 3)
    assert idx.tolist() == [[1, 2, 3]]
    e = math.exp(-2.0)
    assert torch.allclose(gates, torch.tensor([[1 / (2 + e), 1 / (2 + e), e / (2 + e)]], dtype=D))


def _layer_setup(E, k, seed):
    import mt_inputs
    from oracle import OracleConfig
    s = mt_inputs.PRESETS["tiny"].with_(n_layers=1, d_model=64, n_heads=4, n_kv_heads=2, head_dim=16, ffn=48,
                                        vocab=50, batch=2, seq=10)
    cfg = OracleConfig.from_shape(s)
    lw = {n: t.to(D) for n, t in mt_inputs.layer_weights(s, 0, gain_jitter=0.1).items()}
    wr, experts = _weights(E, s.d_model, s.ffn, seed)
    x = torch.randn(s.batch, s.seq, s.d_model, generator=torch.Generator().manual_seed(seed + 1), dtype=D)
    cos, sin = oracle.rope_cos_sin(s.seq, s.head_dim, s.rope_theta)
    return s, cfg, lw, wr, experts, x, cos, sin


def test_moe_layer_with_one_expert_is_the_dense_layer():
    """E = k = 1 with the dense layer's own MLP as the expert: the MoE layer's
    output and every gradient equal the dense layer's."""
    s, cfg, lw, wr, _, x, cos, sin = _layer_setup(1, 1, 51)
    mw = {n: lw[n] for n in ("g1", "wq", "wk", "wv", "wo", "g2")}
    mw["wr"] = wr
    mw["experts"] = [{"wg": lw["wg"], "wu": lw["wu"], "wd": lw["wd"]}]
    y_dense, c_dense = oracle.layer_forward(x, lw, cfg, cos, sin)
    y_moe, c_moe = moe.moe_layer_forward(x, mw, cfg, cos, sin, 1)
    assert torch.allclose(y_moe, y_dense, rtol=1e-13, atol=1e-14)
    dy = torch.randn(x.shape, generator=torch.Generator().manual_seed(52), dtype=D)
    dx_d, g_d = oracle.layer_backward(dy, c_dense, lw, cfg, cos, sin)
    dx_m, g_m = moe.moe_layer_backward(dy, c_moe, mw, cfg, cos, sin, 1)
    assert torch.allclose(dx_m, dx_d, rtol=1e-11, atol=1e-13)
    for n in ("g1", "wq", "wk", "wv", "wo", "g2"):
        assert torch.allclose(g_m[n], g_d[n], rtol=1e-11, atol=1e-13), n
    for n in ("wg", "wu", "wd"):
        assert torch.allclose(g_m["experts"][0][n], g_d[n], rtol=1e-11, atol=1e-13), n
    assert torch.all(g_m["wr"] == 0)  # one expert, gate identically 1


def test_moe_layer_finite_differences():
    """Directional central differences of the MoE layer over all its weights
    and its input, small enough that no token's expert selection moves."""
    E, k = 5, 2
    s, cfg, lw, wr, experts, x, cos, sin = _layer_setup(E, k, 61)
    mw = {n: lw[n] for n in ("g1", "wq", "wk", "wv", "wo", "g2")}
    mw["wr"], mw["experts"] = wr, experts
    dy = torch.randn(x.shape, generator=torch.Generator().manual_seed(62), dtype=D)
    _, c = moe.moe_layer_forward(x, mw, cfg, cos, sin, k)
    dx, g = moe.moe_layer_backward(dy, c, mw, cfg, cos, sin, k)
    gen = torch.Generator().manual_seed(63)
    names = ("g1", "wq", "wk", "wv", "wo", "g2", "wr")
    for _ in range(2):
        ux = torch.randn(x.shape, generator=gen, dtype=D)
        uw = {n: torch.randn(mw[n].shape, generator=gen, dtype=D) for n in names}
        ue = [{n: torch.randn(t.shape, generator=gen, dtype=D) for n, t in e.items()} for e in experts]
        h = 1e-6

        def f(sign):
            w2 = {n: mw[n] + sign * h * uw[n] for n in names}
            w2["experts"] = [{n: t + sign * h * ue[i][n] for n, t in e.items()} for i, e in enumerate(experts)]
            y, c2 = moe.moe_layer_forward(x + sign * h * ux, w2, cfg, cos, sin, k)
            assert torch.equal(c2["moe"]["idx"], c["moe"]["idx"])
            return float((y * dy).sum())

        fd = (f(1) - f(-1)) / (2 * h)
        an = float((dx * ux).sum()) + sum(float((g[n] * uw[n]).sum()) for n in names) + \
            sum(float((g["experts"][i][n] * ue[i][n]).sum()) for i in range(E) for n in ("wg", "wu", "wd"))
        assert abs(fd - an) <= 1e-6 * abs(an) + 1e-9, (fd, an)


def test_moe_model_with_one_expert_is_the_dense_model():
    """A whole model of single-expert MoE layers (the dense MLP as the expert)
    has the dense model's loss and gradients."""
    import mt_inputs
    from oracle import OracleConfig
    s = mt_inputs.PRESETS["tiny"].with_(n_layers=2, d_model=64, n_heads=4, n_kv_heads=2, head_dim=16, ffn=48,
                                        vocab=50, batch=2, seq=10)
    cfg = OracleConfig.from_shape(s)
    params = mt_inputs.model_weights(s, gain_jitter=0.1)
    tokens = mt_inputs.step_tokens(s, 1)
    loss, grads = oracle.model_loss_and_grads(params, tokens, cfg)
    mp = dict(params, layers=[{**{n: lw[n] for n in ("g1", "wq", "wk", "wv", "wo", "g2")},
                               "wr": torch.zeros(1, s.d_model, dtype=torch.bfloat16),
                               "experts": [{"wg": lw["wg"], "wu": lw["wu"], "wd": lw["wd"]}]}
                              for lw in params["layers"]])
    loss_m, grads_m = moe.moe_model_loss_and_grads(mp, tokens, cfg, 1)
    assert abs(loss_m - loss) <= 1e-12 * abs(loss)
    assert torch.allclose(grads_m["embed"]["E"], grads["embed"]["E"], rtol=1e-10, atol=1e-14)
    for gl_m, gl in zip(grads_m["layers"], grads["layers"]):
        for n in ("g1", "wq", "wk", "wv", "wo", "g2"):
            assert torch.allclose(gl_m[n], gl[n], rtol=1e-10, atol=1e-14), n
        for n in ("wg", "wu", "wd"):
            assert torch.allclose(gl_m["experts"][0][n], gl[n], rtol=1e-10, atol=1e-14), n
