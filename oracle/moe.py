"""CPU oracle of a mixture-of-experts MLP block (FP64).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only ``tests/`` may
import it; the library never does.

The pages name the model of MegaTrain's largest run (gpt-oss 120B, a
mixture-of-experts decoder; author's blog, the single-H200 run; podcast
transcript, the 120B GPT-OSS run), list dedicated MoE optimisations among
planned work (author's blog, planned projects) and note that the stateless
layer templates may need redesign for MoE (engineersofai.com breakdown,
limitations), but give no formula for the MoE layer.  This file takes the
plainest reading of a top-k MoE MLP, stated here so that the kernels have a
definition to match:

* router logits ``s = x W_r^T`` (``W_r`` [E, d], no bias);
* per token, the k experts with the largest logits; ties go to the lower
  expert index (a stable order, so the selection is a function of ``s``);
* gates ``g = softmax`` over the k selected logits (they sum to 1);
* ``y = sum_j g_j * f_{e_j}(x)`` with every expert a SwiGLU MLP,
  ``f_e(x) = W_d[e] (silu(W_g[e] x) * W_u[e] x)``, no biases.

The selection is piecewise constant, so the gradient flows through the gates
and the experts only.  Everything is FP64 and unblocked: each expert runs on
the rows routed to it, gathered with ``index_select`` and scattered back with
``index_add_``.

Parity status: pinned by ``tests/test_oracle_moe_pins.py`` (autograd of a
separately written forward, finite differences of the block and of the whole
MoE decoder layer, the single-expert block equal to the dense SwiGLU MLP and
the single-expert layer equal to the dense decoder layer, invariance under
relabelling the experts, the tie order).
"""
from __future__ import annotations

import torch

from .decoder import (OracleConfig, causal_gqa_attention, causal_gqa_attention_backward, head_loss_and_backward,
                      head_weight, rms_norm, rms_norm_backward, rope, rope_backward, rope_cos_sin, swiglu,
                      swiglu_backward)

__all__ = ["moe_route", "moe_mlp_forward", "moe_mlp_backward", "moe_layer_forward", "moe_layer_backward",
           "moe_model_loss_and_grads"]


def moe_route(x, wr, k):
    """x [N, d], wr [E, d] -> (logits [N, E], expert ids [N, k], gates [N, k]).

    Expert ids per token in descending logit order, ties to the lower id.
    """
    s = x @ wr.T
    E = s.shape[1]
    # stable descending order: sort by (-logit, id)
    order = torch.sort(-s, dim=1, stable=True).indices
    idx = order[:, :k]
    sel = s.gather(1, idx)
    gates = torch.softmax(sel, dim=1)
    assert idx.shape[1] == k <= E
    return s, idx, gates


def moe_mlp_forward(x, wr, experts, k):
    """y = sum_j g_j f_{e_j}(x) for x [N, d]; ``experts`` is a list of dicts
    with 'wg', 'wu' [F, d] and 'wd' [d, F].  Returns (y, cache)."""
    N, d = x.shape
    s, idx, gates = moe_route(x, wr, k)
    y = torch.zeros_like(x)
    per_expert = []
    for e, ew in enumerate(experts):
        tok, slot = (idx == e).nonzero(as_tuple=True)  # rows routed to e, and which of their k slots
        xe = x.index_select(0, tok)
        gate, up = xe @ ew["wg"].T, xe @ ew["wu"].T
        a = swiglu(gate, up)
        fe = a @ ew["wd"].T
        y.index_add_(0, tok, fe * gates[tok, slot][:, None])
        per_expert.append((tok, slot, xe, gate, up, a, fe))
    return y, {"s": s, "idx": idx, "gates": gates, "per_expert": per_expert}


def moe_mlp_backward(dy, x, wr, experts, k, cache):
    """Gradients of sum(dy * y): returns (dx, dwr, [{'wg','wu','wd'}] per expert)."""
    idx, gates = cache["idx"], cache["gates"]
    N, d = x.shape
    dx = torch.zeros_like(x)
    dg = torch.zeros_like(gates)  # d loss / d gate[n, j]
    dexperts = []
    for e, ew in enumerate(experts):
        tok, slot, xe, gate, up, a, fe = cache["per_expert"][e]
        dye = dy.index_select(0, tok)
        dg[tok, slot] = (dye * fe).sum(1)
        dfe = dye * gates[tok, slot][:, None]  # gradient of this expert's output
        dwd = dfe.T @ a
        da = dfe @ ew["wd"]
        dgate, dup = swiglu_backward(da, gate, up)
        dwg = dgate.T @ xe
        dwu = dup.T @ xe
        dx.index_add_(0, tok, dgate @ ew["wg"] + dup @ ew["wu"])
        dexperts.append({"wg": dwg, "wu": dwu, "wd": dwd})
    # softmax over the selected logits: ds_j = g_j (dg_j - sum_i g_i dg_i)
    dsel = gates * (dg - (gates * dg).sum(1, keepdim=True))
    ds = torch.zeros(N, wr.shape[0], dtype=x.dtype)
    ds.scatter_(1, idx, dsel)
    dwr = ds.T @ x
    dx += ds @ wr
    return dx, dwr, dexperts


# ----------------------------------------------------------------------------
# One MoE decoder layer: the dense layer's attention half, then the MoE MLP
# ----------------------------------------------------------------------------

def moe_layer_forward(x, lw, cfg: OracleConfig, cos, sin, k):
    """x [B, S, d] -> x' = h + MoE(n2), h = x + W_o attn(n1), n2 = RMSNorm(h; g2).

    ``lw``: g1, wq, wk, wv, wo, g2, wr [E, d] and ``experts`` (a list of
    {wg, wu, wd}).  Returns x' and the cache for ``moe_layer_backward``.
    """
    B, S, d = x.shape
    Hq, Hkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    n1, rstd1 = rms_norm(x, lw["g1"], cfg.rms_eps)
    qr = rope((n1 @ lw["wq"].T).reshape(B, S, Hq, hd), cos, sin)
    kr = rope((n1 @ lw["wk"].T).reshape(B, S, Hkv, hd), cos, sin)
    v = (n1 @ lw["wv"].T).reshape(B, S, Hkv, hd)
    o, probs = causal_gqa_attention(qr, kr, v)
    o2 = o.reshape(B, S, Hq * hd)
    h = x + o2 @ lw["wo"].T
    n2, rstd2 = rms_norm(h, lw["g2"], cfg.rms_eps)
    y, mc = moe_mlp_forward(n2.reshape(B * S, d), lw["wr"], lw["experts"], k)
    x_out = h + y.reshape(B, S, d)
    cache = dict(x=x, n1=n1, rstd1=rstd1, qr=qr, kr=kr, v=v, probs=probs, o2=o2, h=h, n2=n2, rstd2=rstd2, moe=mc)
    return x_out, cache


def moe_layer_backward(dx_out, c, lw, cfg: OracleConfig, cos, sin, k):
    """Backward of ``moe_layer_forward``: (dx, grads named as in ``lw``, the
    experts' gradients as a list under 'experts')."""
    B, S, d = dx_out.shape
    Hq, Hkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim

    def wgrad(dy, xin):
        return dy.reshape(-1, dy.shape[-1]).T @ xin.reshape(-1, xin.shape[-1])

    g = {}
    dn2, g["wr"], g["experts"] = moe_mlp_backward(dx_out.reshape(B * S, d), c["n2"].reshape(B * S, d), lw["wr"],
                                                 lw["experts"], k, c["moe"])
    dh_n, g["g2"] = rms_norm_backward(dn2.reshape(B, S, d), c["h"], lw["g2"], c["rstd2"])
    dh = dx_out + dh_n
    g["wo"] = wgrad(dh, c["o2"])
    do = (dh @ lw["wo"]).reshape(B, S, Hq, hd)
    dqr, dkr, dv = causal_gqa_attention_backward(do, c["qr"], c["kr"], c["v"], c["probs"])
    dq = rope_backward(dqr, cos, sin).reshape(B, S, Hq * hd)
    dk = rope_backward(dkr, cos, sin).reshape(B, S, Hkv * hd)
    dv = dv.reshape(B, S, Hkv * hd)
    g["wq"] = wgrad(dq, c["n1"])
    g["wk"] = wgrad(dk, c["n1"])
    g["wv"] = wgrad(dv, c["n1"])
    dn1 = dq @ lw["wq"] + dk @ lw["wk"] + dv @ lw["wv"]
    dx_n, g["g1"] = rms_norm_backward(dn1, c["x"], lw["g1"], c["rstd1"])
    return dh + dx_n, g


def moe_model_loss_and_grads(params, tokens, cfg: OracleConfig, k, dtype=torch.float64):
    """``model_loss_and_grads`` of a decoder whose layers are all MoE layers
    (``params["layers"][i]`` as ``moe_layer_forward`` takes them); the
    embedding, the final norm, the LM head (tied or not) and the loss as in
    the dense model."""
    f = lambda t: t.to(dtype)
    p = {"embed": {n: f(t) for n, t in params["embed"].items()},
         "layers": [{n: ([{m: f(u) for m, u in e.items()} for e in t] if n == "experts" else f(t))
                     for n, t in lw.items()} for lw in params["layers"]],
         "head": {n: f(t) for n, t in params["head"].items()}}
    tokens = tokens.long()
    inp, tgt = tokens[:, :-1], tokens[:, 1:]
    S = inp.shape[1]
    cos, sin = rope_cos_sin(S, cfg.head_dim, cfg.rope_theta, dtype)
    x = p["embed"]["E"][inp]
    caches = []
    for lw in p["layers"]:
        x, c = moe_layer_forward(x, lw, cfg, cos, sin, k)
        caches.append(c)
    tied = "wh" not in p["head"]
    loss, dx, head_g = head_loss_and_backward(x, {"gf": p["head"]["gf"], "wh": head_weight(p)}, tgt, cfg)
    layer_g = [None] * len(p["layers"])
    for i in reversed(range(len(p["layers"]))):
        dx, layer_g[i] = moe_layer_backward(dx, caches[i], p["layers"][i], cfg, cos, sin, k)
    dE = torch.zeros_like(p["embed"]["E"])
    dE.index_add_(0, inp.reshape(-1), dx.reshape(-1, cfg.d_model))
    if tied:
        dE += head_g.pop("wh")
    return float(loss), {"embed": {"E": dE}, "layers": layer_g, "head": head_g}

