"""CPU oracle of one MegaTrain training step: decoder forward, backward, Adam.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module.  The product path
(``host_memory_streamed_gb300``) never imports, calls or links it and shares
no code, table or constant generator with it.

What it computes is the plain definition of the training step that the
layer-streamed schedule must reproduce (streaming, recompute and the
three-stream pipeline change only *where* and *when* things run; MegaTrain
paper summary (paperlayer.ai), §3 "Execution workflow"; hyper.ai summary,
方法 "Method" ¶2):

* a Llama-style decoder (RMSNorm, rotate-half RoPE, causal GQA attention,
  SwiGLU MLP, no biases; embedding and LM head untied, or tied: one matrix
  used for both, see ``head_weight``) on token ids
  ``tokens[B, S+1]``; inputs ``tokens[:, :S]``, targets ``tokens[:, 1:]``;
* the mean next-token cross-entropy over the B*S targets;
* its gradient with respect to every weight, written out by hand;
* one bias-corrected Adam step whose persistent state is BF16 weights, BF16
  gradients and FP32 moments and nothing else (12 bytes per parameter, no FP32
  master copy; paperlayer.ai summary §2 "Training memory"; author's blog,
  the 12x accounting; podcast transcript, the Adam bias-correction remark).

Precision: every activation, gradient and reduction is FP64 (``torch.float64``
on the CPU) and never rounded; the only roundings are the ones the pages fix:
weights are BF16 values (upcast exactly), the stored gradient is BF16, the
Adam moments are FP32 and the updated weight is BF16 (round to nearest even).
``dtype=torch.float32`` runs the same code in FP32 for the timed CPU baseline.

Library primitives used as single steps: ``torch.matmul``, ``exp``, ``log``,
``sqrt``, ``sigmoid``, ``logsumexp``, ``softmax``, ``index_add_``.  There is no
blocking, fusion or reordering: attention materialises the full score matrix
of one (batch, head) pair, the LM head materialises all logits.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(finite differences, library special cases, closed forms and invariants).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

__all__ = [
    "OracleConfig",
    "round_to_bf16",
    "round_to_fp32",
    "rms_norm",
    "rms_norm_backward",
    "rope_cos_sin",
    "rope",
    "rope_backward",
    "causal_gqa_attention",
    "causal_gqa_attention_backward",
    "attention_rows",
    "attention_key_grads",
    "swiglu",
    "swiglu_backward",
    "layer_forward",
    "layer_backward",
    "layer_tail_rows",
    "head_loss_and_backward",
    "head_weight",
    "model_forward_loss",
    "model_loss_and_grads",
    "adam_update",
    "train_step",
]


@dataclass(frozen=True)
class OracleConfig:
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rms_eps: float = 1e-5
    rope_theta: float = 1e4
    lr: float = 1e-4
    beta1: float = 0.9
    beta2: float = 0.95
    adam_eps: float = 1e-8
    weight_decay: float = 0.0

    @staticmethod
    def from_shape(s) -> "OracleConfig":
        return OracleConfig(
            s.n_layers, s.d_model, s.n_heads, s.n_kv_heads, s.head_dim, s.ffn, s.vocab,
            s.rms_eps, s.rope_theta, s.lr, s.beta1, s.beta2, s.adam_eps, s.weight_decay,
        )


# ----------------------------------------------------------------------------
# Rounding
# ----------------------------------------------------------------------------

def round_to_bf16(x: torch.Tensor) -> torch.Tensor:
    """Round FP64 values to the nearest BF16 value (ties to even), as FP64.

    BF16 keeps 8 significant bits.  With x = m * 2**e, 0.5 <= |m| < 1
    (``frexp``), the BF16 value is round_half_even(m * 256) / 256 * 2**e; the
    product m * 256 is exact in FP64, so the only rounding is the one asked for.
    Subnormal BF16 inputs do not occur in this model and are not special-cased.
    """
    x = x.to(torch.float64)
    m, e = torch.frexp(x)
    r = torch.round(m * 256.0) / 256.0  # torch.round rounds half to even
    return torch.ldexp(r, e.to(torch.float64))


def round_to_fp32(x: torch.Tensor) -> torch.Tensor:
    """FP64 -> nearest FP32 (IEEE cast, ties to even), returned as FP64."""
    return x.to(torch.float32).to(torch.float64)


# ----------------------------------------------------------------------------
# RMSNorm: y = x / sqrt(mean(x^2) + eps) * g
# ----------------------------------------------------------------------------

def rms_norm(x, g, eps):
    """RMSNorm over the last axis. Returns (y, rstd) with rstd = 1/sqrt(ms + eps)."""
    ms = (x * x).mean(dim=-1, keepdim=True)
    rstd = 1.0 / torch.sqrt(ms + eps)
    return x * rstd * g, rstd


def rms_norm_backward(dy, x, g, rstd):
    """Gradients of y = x * rstd(x) * g.

    With xhat = x * rstd and n the row length:
      dg = sum_rows(dy * xhat)
      dx = rstd * (dy*g - xhat * mean(dy*g*xhat))
    """
    xhat = x * rstd
    dyg = dy * g
    n = x.shape[-1]
    dx = rstd * (dyg - xhat * (dyg * xhat).sum(dim=-1, keepdim=True) / n)
    dg = (dy * xhat).reshape(-1, n).sum(dim=0)
    return dx, dg


# ----------------------------------------------------------------------------
# Rotary position embedding, rotate-half form, position = index within sequence
# ----------------------------------------------------------------------------

def rope_cos_sin(seq, head_dim, theta, dtype=torch.float64):
    """cos/sin tables [seq, head_dim/2] of angle s * theta**(-2i/head_dim)."""
    i = torch.arange(head_dim // 2, dtype=torch.float64)
    inv_freq = theta ** (-2.0 * i / head_dim)
    s = torch.arange(seq, dtype=torch.float64)
    ang = s[:, None] * inv_freq[None, :]
    return torch.cos(ang).to(dtype), torch.sin(ang).to(dtype)


def rope(x, cos, sin):
    """x [B, S, H, hd] -> (x1 cos - x2 sin, x2 cos + x1 sin) with x = [x1 | x2]."""
    h = x.shape[-1] // 2
    x1, x2 = x[..., :h], x[..., h:]
    c = cos[None, :, None, :]
    s = sin[None, :, None, :]
    return torch.cat([x1 * c - x2 * s, x2 * c + x1 * s], dim=-1)


def rope_backward(dy, cos, sin):
    """Transpose of the rotation: (dy1 cos + dy2 sin, dy2 cos - dy1 sin)."""
    h = dy.shape[-1] // 2
    d1, d2 = dy[..., :h], dy[..., h:]
    c = cos[None, :, None, :]
    s = sin[None, :, None, :]
    return torch.cat([d1 * c + d2 * s, d2 * c - d1 * s], dim=-1)


# ----------------------------------------------------------------------------
# Causal grouped-query attention
# ----------------------------------------------------------------------------

def _kv_head(h, n_heads, n_kv_heads):
    return h * n_kv_heads // n_heads


def causal_gqa_attention(q, k, v):
    """softmax(q k^T / sqrt(hd) + causal mask) v, query head h reading kv head h*Hkv/Hq.

    q [B, S, Hq, hd]; k, v [B, S, Hkv, hd].  Returns o [B, S, Hq, hd] and the
    list of probability matrices P[b][h] ([S, S]) for the backward pass.
    """
    B, S, Hq, hd = q.shape
    Hkv = k.shape[2]
    scale = 1.0 / math.sqrt(hd)
    mask = torch.ones(S, S, dtype=torch.bool).triu(1)  # key index > query index
    o = torch.empty_like(q)
    probs = []
    for b in range(B):
        pb = []
        for h in range(Hq):
            j = _kv_head(h, Hq, Hkv)
            scores = (q[b, :, h, :] @ k[b, :, j, :].T) * scale
            scores = scores.masked_fill(mask, float("-inf"))
            p = torch.softmax(scores, dim=-1)
            o[b, :, h, :] = p @ v[b, :, j, :]
            pb.append(p)
        probs.append(pb)
    return o, probs


def causal_gqa_attention_backward(do, q, k, v, probs):
    """Gradients through o = P v, P = softmax(scores), scores = q k^T * scale.

    dP = dO v^T; dScores = P * (dP - rowsum(P * dP)); dq = dScores k * scale;
    dk = dScores^T q * scale; dv = P^T dO.  Key/value gradients of the query
    heads that share a kv head are summed.
    """
    B, S, Hq, hd = q.shape
    Hkv = k.shape[2]
    scale = 1.0 / math.sqrt(hd)
    dq = torch.zeros_like(q)
    dk = torch.zeros_like(k)
    dv = torch.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            j = _kv_head(h, Hq, Hkv)
            p = probs[b][h]
            dob = do[b, :, h, :]
            dp = dob @ v[b, :, j, :].T
            ds = p * (dp - (p * dp).sum(dim=-1, keepdim=True))
            dq[b, :, h, :] = (ds @ k[b, :, j, :]) * scale
            dk[b, :, j, :] += (ds.T @ q[b, :, h, :]) * scale
            dv[b, :, j, :] += p.T @ dob
    return dq, dk, dv


def attention_rows(q, k, v, rows, do=None):
    """The same causal attention for selected query rows of one head.

    q [S, hd] (one query head), k, v [S, hd] (its kv head); for each row i in
    ``rows``: scores over keys 0..i, o_i = softmax(scores) v, lse_i =
    logsumexp(scores); with ``do`` [S, hd], also dq_i = (P * (dP - rowsum(P*dP))) k * scale.
    Cost O(len(rows) * S * hd): usable at long sequences.  Returns (o, lse, dq)
    stacked over ``rows`` (dq is None without ``do``).
    """
    hd = q.shape[-1]
    scale = 1.0 / math.sqrt(hd)
    os_, ls_, dq_ = [], [], []
    for i in rows:
        sc = (k[: i + 1] @ q[i]) * scale
        lse = torch.logsumexp(sc, dim=0)
        p = torch.exp(sc - lse)
        os_.append(p @ v[: i + 1])
        ls_.append(lse)
        if do is not None:
            dp = v[: i + 1] @ do[i]
            ds = p * (dp - (p * dp).sum())
            dq_.append((ds @ k[: i + 1]) * scale)
    dq = torch.stack(dq_) if do is not None else None
    return torch.stack(os_), torch.stack(ls_), dq


def attention_key_grads(qs, k, v, dos, j):
    """dk_j and dv_j of key position j of one kv head.

    qs [G, S, hd] and dos [G, S, hd]: the query heads that read this kv head
    and their output gradients; k, v [S, hd].  Sums over every query row
    i >= j of every head in the group: dv_j = sum P_ij dO_i and
    dk_j = sum dS_ij q_i * scale with P, dS of the full causal rows i.
    Cost O(G * (S - j) * S * hd).
    """
    G, S, hd = qs.shape
    scale = 1.0 / math.sqrt(hd)
    mask = torch.arange(S)[None, :] > torch.arange(j, S)[:, None]  # key > query
    dk = torch.zeros(hd, dtype=k.dtype)
    dv = torch.zeros(hd, dtype=v.dtype)
    for g in range(G):
        qi = qs[g, j:]
        sc = (qi @ k.T) * scale
        sc = sc.masked_fill(mask, float("-inf"))
        p = torch.softmax(sc, dim=-1)
        dp = dos[g, j:] @ v.T
        ds = p * (dp - (p * dp).sum(dim=-1, keepdim=True))
        dv += p[:, j] @ dos[g, j:]
        dk += (ds[:, j] @ qi) * scale
    return dk, dv


# ----------------------------------------------------------------------------
# SwiGLU: a = silu(gate) * up, silu(x) = x * sigmoid(x)
# ----------------------------------------------------------------------------

def swiglu(gate, up):
    return gate * torch.sigmoid(gate) * up


def swiglu_backward(da, gate, up):
    sg = torch.sigmoid(gate)
    silu = gate * sg
    dsilu = sg * (1.0 + gate * (1.0 - sg))
    return da * up * dsilu, da * silu


# ----------------------------------------------------------------------------
# One decoder layer
# ----------------------------------------------------------------------------

def _f(t, dtype):
    return t.to(dtype)


def layer_forward(x, lw, cfg: OracleConfig, cos, sin):
    """x [B, S, d] -> x' = h + W_d(silu(W_g n2) * W_u n2), h = x + W_o attn(n1).

    ``lw`` maps g1, wq, wk, wv, wo, g2, wg, wu, wd to tensors of the compute
    dtype.  Returns x' and the cache the backward pass needs.
    """
    B, S, d = x.shape
    Hq, Hkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    n1, rstd1 = rms_norm(x, lw["g1"], cfg.rms_eps)
    q = (n1 @ lw["wq"].T).reshape(B, S, Hq, hd)
    k = (n1 @ lw["wk"].T).reshape(B, S, Hkv, hd)
    v = (n1 @ lw["wv"].T).reshape(B, S, Hkv, hd)
    qr = rope(q, cos, sin)
    kr = rope(k, cos, sin)
    o, probs = causal_gqa_attention(qr, kr, v)
    o2 = o.reshape(B, S, Hq * hd)
    h = x + o2 @ lw["wo"].T
    n2, rstd2 = rms_norm(h, lw["g2"], cfg.rms_eps)
    gate = n2 @ lw["wg"].T
    up = n2 @ lw["wu"].T
    a = swiglu(gate, up)
    x_out = h + a @ lw["wd"].T
    cache = dict(x=x, n1=n1, rstd1=rstd1, qr=qr, kr=kr, v=v, probs=probs, o2=o2,
                 h=h, n2=n2, rstd2=rstd2, gate=gate, up=up, a=a)
    return x_out, cache


def layer_backward(dx_out, c, lw, cfg: OracleConfig, cos, sin):
    """Backward of ``layer_forward``: returns (dx, grads dict with the names of lw)."""
    B, S, d = dx_out.shape
    Hq, Hkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    g = {}

    def wgrad(dy, xin):  # dW = dy^T x over all tokens
        return dy.reshape(-1, dy.shape[-1]).T @ xin.reshape(-1, xin.shape[-1])

    # x_out = h + a Wd^T
    dh = dx_out.clone()
    g["wd"] = wgrad(dx_out, c["a"])
    da = dx_out @ lw["wd"]
    dgate, dup = swiglu_backward(da, c["gate"], c["up"])
    g["wg"] = wgrad(dgate, c["n2"])
    g["wu"] = wgrad(dup, c["n2"])
    dn2 = dgate @ lw["wg"] + dup @ lw["wu"]
    dh_n, g["g2"] = rms_norm_backward(dn2, c["h"], lw["g2"], c["rstd2"])
    dh = dh + dh_n
    # h = x + o Wo^T
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


def layer_tail_rows(x, dy_tail, lw, cfg: OracleConfig, cos, sin, t0):
    """One decoder layer on one sequence whose output gradient is zero before row t0.

    x [S, d]: the layer input of one sequence; dy_tail [S - t0, d]: dL/dx' on
    rows t0..S-1 (rows before t0 carry no gradient).  By causality, rows t0..
    of x' need the queries of those rows and the keys and values of every row,
    and the gradient reaches rows before t0 only through their keys and
    values, so the result equals ``layer_forward`` / ``layer_backward`` with
    dy zero-padded, at a cost of O(S (d (2 Hkv hd) + (S - t0) Hq hd) +
    (S - t0) d (Hq hd + 3 ffn)) instead of O(S^2 Hq hd + S d ffn).
    ``cos``/``sin`` are the tables of all S positions.  Returns (x' on rows
    t0.., dL/dx on all S rows, weight gradients named as in ``lw``).
    """
    S, d = x.shape
    R = S - t0
    Hq, Hkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    scale = 1.0 / math.sqrt(hd)
    ct, st = cos[t0:], sin[t0:]
    # forward: normalised input of every row, keys/values of every row
    n1, rstd1 = rms_norm(x, lw["g1"], cfg.rms_eps)
    k = rope((n1 @ lw["wk"].T).reshape(1, S, Hkv, hd), cos, sin)[0]
    v = (n1 @ lw["wv"].T).reshape(S, Hkv, hd)
    n1t = n1[t0:]
    q = rope((n1t @ lw["wq"].T).reshape(1, R, Hq, hd), ct, st)[0]
    mask = torch.arange(S)[None, :] > torch.arange(t0, S)[:, None]  # key index > query index
    o = torch.empty(R, Hq, hd, dtype=x.dtype)
    probs = []
    for h in range(Hq):
        j = _kv_head(h, Hq, Hkv)
        sc = ((q[:, h] @ k[:, j].T) * scale).masked_fill(mask, float("-inf"))
        p = torch.softmax(sc, dim=-1)
        o[:, h] = p @ v[:, j]
        probs.append(p)
    o2 = o.reshape(R, Hq * hd)
    hh = x[t0:] + o2 @ lw["wo"].T
    n2, rstd2 = rms_norm(hh, lw["g2"], cfg.rms_eps)
    gate = n2 @ lw["wg"].T
    up = n2 @ lw["wu"].T
    a = swiglu(gate, up)
    y = hh + a @ lw["wd"].T
    # backward
    g = {}
    dy = dy_tail
    g["wd"] = dy.T @ a
    dgate, dup = swiglu_backward(dy @ lw["wd"], gate, up)
    g["wg"] = dgate.T @ n2
    g["wu"] = dup.T @ n2
    dh_n, g["g2"] = rms_norm_backward(dgate @ lw["wg"] + dup @ lw["wu"], hh, lw["g2"], rstd2)
    dh = dy + dh_n
    g["wo"] = dh.T @ o2
    do = (dh @ lw["wo"]).reshape(R, Hq, hd)
    dq = torch.empty(R, Hq, hd, dtype=x.dtype)
    dk = torch.zeros(S, Hkv, hd, dtype=x.dtype)
    dv = torch.zeros(S, Hkv, hd, dtype=x.dtype)
    for h in range(Hq):
        j = _kv_head(h, Hq, Hkv)
        p = probs[h]
        dp = do[:, h] @ v[:, j].T
        ds = p * (dp - (p * dp).sum(dim=-1, keepdim=True))
        dq[:, h] = (ds @ k[:, j]) * scale
        dk[:, j] += (ds.T @ q[:, h]) * scale
        dv[:, j] += p.T @ do[:, h]
    dq = rope_backward(dq[None], ct, st)[0].reshape(R, Hq * hd)
    dk = rope_backward(dk[None], cos, sin)[0].reshape(S, Hkv * hd)
    dv = dv.reshape(S, Hkv * hd)
    g["wq"] = dq.T @ n1t
    g["wk"] = dk.T @ n1
    g["wv"] = dv.T @ n1
    dn1 = dk @ lw["wk"] + dv @ lw["wv"]
    dn1[t0:] += dq @ lw["wq"]
    dx, g["g1"] = rms_norm_backward(dn1, x, lw["g1"], rstd1)
    dx[t0:] += dh
    return y, dx, g


# ----------------------------------------------------------------------------
# Final norm + LM head + mean cross-entropy
# ----------------------------------------------------------------------------

def head_loss_and_backward(x, hw, tgt, cfg: OracleConfig):
    """loss = mean_t [logsumexp(z_t) - z_t[y_t]], z = RMSNorm(x; gf) W_h^T.

    Returns (loss, dx, {'gf': dgf, 'wh': dW_h}).  dz = (softmax(z) - onehot(y)) / N.
    """
    B, S, d = x.shape
    N = B * S
    nf, rstd = rms_norm(x, hw["gf"], cfg.rms_eps)
    nf2 = nf.reshape(N, d)
    z = nf2 @ hw["wh"].T
    y = tgt.reshape(N).long()
    lse = torch.logsumexp(z, dim=-1)
    loss = (lse - z.gather(1, y[:, None])[:, 0]).mean()
    dz = torch.softmax(z, dim=-1)
    dz[torch.arange(N), y] -= 1.0
    dz /= N
    grads = {"wh": dz.T @ nf2}
    dnf = (dz @ hw["wh"]).reshape(B, S, d)
    dx, grads["gf"] = rms_norm_backward(dnf, x, hw["gf"], rstd)
    return loss, dx, grads


# ----------------------------------------------------------------------------
# Whole model
# ----------------------------------------------------------------------------

def head_weight(p):
    """The LM head's weight: its own W_h, or the embedding E when the model ties
    them (``params["head"]`` then holds only the final norm gain).  The pages'
    host store keeps tied embedding and head states in one shared region
    (paperlayer.ai summary §A.1, tied embeddings); mathematically the one
    matrix E is used twice, as the token embedding and as W_h."""
    return p["head"]["wh"] if "wh" in p["head"] else p["embed"]["E"]


def _cast_params(params, dtype):
    return {
        "embed": {k: _f(v, dtype) for k, v in params["embed"].items()},
        "layers": [{k: _f(v, dtype) for k, v in lw.items()} for lw in params["layers"]],
        "head": {k: _f(v, dtype) for k, v in params["head"].items()},
    }


def model_forward_loss(params, tokens, cfg: OracleConfig, dtype=torch.float64):
    """Forward pass only: the mean next-token cross-entropy (a Python float)."""
    p = _cast_params(params, dtype)
    tokens = tokens.long()
    inp, tgt = tokens[:, :-1], tokens[:, 1:]
    S = inp.shape[1]
    cos, sin = rope_cos_sin(S, cfg.head_dim, cfg.rope_theta, dtype)
    x = p["embed"]["E"][inp]
    for lw in p["layers"]:
        x, _ = layer_forward(x, lw, cfg, cos, sin)
    nf, _ = rms_norm(x, p["head"]["gf"], cfg.rms_eps)
    z = nf.reshape(-1, cfg.d_model) @ head_weight(p).T
    y = tgt.reshape(-1)
    return float((torch.logsumexp(z, dim=-1) - z.gather(1, y[:, None])[:, 0]).mean())


def model_loss_and_grads(params, tokens, cfg: OracleConfig, dtype=torch.float64):
    """Loss and the gradient of every weight, in the structure of ``params``.

    The layer caches of the whole forward pass are kept (the plain definition;
    which activations the GPU keeps or recomputes does not change the result).
    """
    p = _cast_params(params, dtype)
    tokens = tokens.long()
    inp, tgt = tokens[:, :-1], tokens[:, 1:]
    S = inp.shape[1]
    cos, sin = rope_cos_sin(S, cfg.head_dim, cfg.rope_theta, dtype)
    x = p["embed"]["E"][inp]
    caches = []
    for lw in p["layers"]:
        x, c = layer_forward(x, lw, cfg, cos, sin)
        caches.append(c)
    tied = "wh" not in p["head"]
    loss, dx, head_g = head_loss_and_backward(x, {"gf": p["head"]["gf"], "wh": head_weight(p)}, tgt, cfg)
    layer_g = [None] * len(p["layers"])
    for i in reversed(range(len(p["layers"]))):
        dx, layer_g[i] = layer_backward(dx, caches[i], p["layers"][i], cfg, cos, sin)
    dE = torch.zeros_like(p["embed"]["E"])
    dE.index_add_(0, inp.reshape(-1), dx.reshape(-1, cfg.d_model))
    if tied:  # E is used twice: its gradient is the sum of both uses' (chain rule)
        dE += head_g.pop("wh")
    grads = {"embed": {"E": dE}, "layers": layer_g, "head": head_g}
    return float(loss), grads


# ----------------------------------------------------------------------------
# Adam on the host tile (BF16 w, BF16 g, FP32 m and v)
# ----------------------------------------------------------------------------

def adam_update(w, g, m, v, step, cfg: OracleConfig, dtype=torch.float64):
    """One bias-corrected Adam(W) step in the PyTorch convention.

    m <- b1 m + (1-b1) g;  v <- b2 v + (1-b2) g^2;
    mhat = m / (1-b1^t);  vhat = v / (1-b2^t);
    w <- w - lr * (mhat / (sqrt(vhat) + eps) + wd * w)

    Inputs: w and g hold BF16 values, m and v FP32 values (any float dtype).
    The arithmetic is in ``dtype`` (FP64 for parity, FP32 for the timed CPU
    baseline); the results are stored as the tile stores them: m, v rounded
    to FP32 and w rounded to BF16 (ties to even).  Returns (w_new, m_new,
    v_new) as FP64 tensors holding those rounded values.
    """
    w = w.to(dtype)
    g = g.to(dtype)
    m = m.to(dtype)
    v = v.to(dtype)
    t = float(step)
    m_new = cfg.beta1 * m + (1.0 - cfg.beta1) * g
    v_new = cfg.beta2 * v + (1.0 - cfg.beta2) * g * g
    mhat = m_new / (1.0 - cfg.beta1 ** t)
    vhat = v_new / (1.0 - cfg.beta2 ** t)
    w_new = w - cfg.lr * (mhat / (torch.sqrt(vhat) + cfg.adam_eps) + cfg.weight_decay * w)
    return round_to_bf16(w_new), round_to_fp32(m_new), round_to_fp32(v_new)


def train_step(params, state, tokens, step, cfg: OracleConfig, dtype=torch.float64):
    """One full step: loss, grads, grads rounded to BF16, Adam on every tensor.

    ``state`` has the structure of ``params`` with (m, v) pairs per tensor, or
    None for zero moments.  Returns (loss, grads_fp, new_params, new_state),
    where new_params hold BF16 values as FP64 tensors.
    """
    loss, grads = model_loss_and_grads(params, tokens, cfg, dtype)

    def upd(w, gr, mv):
        gb = round_to_bf16(gr.to(torch.float64))
        if mv is None:
            mv = (torch.zeros_like(gb), torch.zeros_like(gb))
        return adam_update(w, gb, mv[0], mv[1], step, cfg)

    new_p = {"embed": {}, "layers": [], "head": {}}
    new_s = {"embed": {}, "layers": [], "head": {}}
    for part in ("embed", "head"):
        for k, w in params[part].items():
            st = None if state is None else state[part][k]
            wn, mn, vn = upd(w, grads[part][k], st)
            new_p[part][k] = wn
            new_s[part][k] = (mn, vn)
    for i, lw in enumerate(params["layers"]):
        pl, sl = {}, {}
        for k, w in lw.items():
            st = None if state is None else state["layers"][i][k]
            wn, mn, vn = upd(w, grads["layers"][i][k], st)
            pl[k], sl[k] = wn, (mn, vn)
        new_p["layers"].append(pl)
        new_s["layers"].append(sl)
    return loss, grads, new_p, new_s
