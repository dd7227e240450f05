"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test ties one oracle function to a library routine that computes the same
special case, to a closed form, to an invariant of the mathematics, or to
finite differences of the oracle's own forward pass.  Together they are chosen
so that a dropped term, a wrong sign or index, or a transposed operand in the
oracle fails at least one of them.
"""
import math
from fractions import Fraction

import pytest
import torch
import torch.nn.functional as F

import mt_inputs
import oracle
from oracle import OracleConfig

D = torch.float64


@pytest.fixture(autouse=True)
def _fp64_default_dtype():
    """The pins build FP64 tensors by default; restore the caller's default after each test."""
    old = torch.get_default_dtype()
    torch.set_default_dtype(torch.float64)
    yield
    torch.set_default_dtype(old)


def _tiny(**kw):
    s = mt_inputs.PRESETS["tiny"].with_(**kw)
    return s, OracleConfig.from_shape(s)


# ---------------------------------------------------------------- rounding

def test_round_to_bf16_matches_torch_cast_on_fp32_values():
    g = torch.Generator().manual_seed(0)
    x = (torch.randn(100000, generator=g, dtype=torch.float32) * torch.exp(torch.randn(100000, generator=g) * 5).float())
    ref = x.to(torch.bfloat16).to(D)  # torch's cast is round-to-nearest-even from fp32
    assert torch.equal(oracle.round_to_bf16(x.to(D)), ref)


def test_round_to_bf16_ties_to_even():
    one = 1.0
    ulp = 2.0 ** -7
    vals = torch.tensor([one + ulp / 2, one + 1.5 * ulp, -(one + ulp / 2), 3.0 * 2 ** -20])
    out = oracle.round_to_bf16(vals)
    assert out.tolist() == [1.0, one + 2 * ulp, -1.0, 3.0 * 2 ** -20]


# ---------------------------------------------------------------- RMSNorm

def test_rms_norm_matches_library_and_autograd():
    g = torch.Generator().manual_seed(1)
    x = torch.randn(5, 7, 48, generator=g)
    w = 1 + 0.3 * torch.randn(48, generator=g)
    y, rstd = oracle.rms_norm(x, w, 1e-5)
    assert torch.allclose(y, F.rms_norm(x, (48,), w, 1e-5), rtol=1e-13, atol=1e-13)
    dy = torch.randn_like(x)
    xa = x.clone().requires_grad_()
    wa = w.clone().requires_grad_()
    F.rms_norm(xa, (48,), wa, 1e-5).backward(dy)
    dx, dg = oracle.rms_norm_backward(dy, x, w, rstd)
    assert torch.allclose(dx, xa.grad, rtol=1e-12, atol=1e-12)
    assert torch.allclose(dg, wa.grad, rtol=1e-12, atol=1e-12)


def test_rms_norm_scale_invariant_without_eps():
    g = torch.Generator().manual_seed(2)
    x = torch.randn(3, 16, generator=g)
    w = torch.randn(16, generator=g)
    y1, _ = oracle.rms_norm(x, w, 0.0)
    y2, _ = oracle.rms_norm(7.5 * x, w, 0.0)
    assert torch.allclose(y1, y2, rtol=1e-14, atol=1e-14)
    # unit mean square after normalisation with unit gains
    y, _ = oracle.rms_norm(x, torch.ones(16), 0.0)
    assert torch.allclose((y * y).mean(-1), torch.ones(3), rtol=1e-14)


# ---------------------------------------------------------------- RoPE

def test_rope_two_dims_is_plain_rotation_by_position():
    # head_dim 2: one pair, inverse frequency theta**0 = 1, angle = position
    cos, sin = oracle.rope_cos_sin(4, 2, 1e4)
    x = torch.tensor([1.0, 0.5]).reshape(1, 1, 1, 2).repeat(1, 4, 1, 1)
    y = oracle.rope(x, cos, sin)
    for s in range(4):
        R = torch.tensor([[math.cos(s), -math.sin(s)], [math.sin(s), math.cos(s)]])
        assert torch.allclose(y[0, s, 0], R @ torch.tensor([1.0, 0.5]), rtol=0, atol=1e-15)


def test_rope_frequency_of_each_pair():
    # head_dim 4 with theta 1e4: pair 0 turns by s, pair 1 by s * 1e4**(-2/4) = s/100;
    # the pairs are (x[0], x[2]) and (x[1], x[3]) in the rotate-half form.
    cos, sin = oracle.rope_cos_sin(300, 4, 1e4)
    x = torch.zeros(1, 300, 1, 4)
    x[..., 1] = 1.0  # unit vector in pair 1's first coordinate
    y = oracle.rope(x, cos, sin)
    s = torch.arange(300, dtype=D)
    assert torch.allclose(y[0, :, 0, 1], torch.cos(s / 100), atol=1e-14)
    assert torch.allclose(y[0, :, 0, 3], torch.sin(s / 100), atol=1e-14)
    assert torch.all(y[0, :, 0, 0] == 0) and torch.all(y[0, :, 0, 2] == 0)


def test_rope_preserves_norm_relative_position_and_adjoint():
    g = torch.Generator().manual_seed(3)
    S, hd = 40, 16
    cos, sin = oracle.rope_cos_sin(S, hd, 1e4)
    q = torch.randn(1, S, 1, hd, generator=g)
    y = oracle.rope(q, cos, sin)
    assert torch.allclose(y.norm(dim=-1), q.norm(dim=-1), rtol=1e-13)
    # <R_a q, R_b k> depends only on a - b
    qv = torch.randn(hd, generator=g)
    kv = torch.randn(hd, generator=g)
    Q = qv.reshape(1, 1, 1, hd).repeat(1, S, 1, 1)
    K = kv.reshape(1, 1, 1, hd).repeat(1, S, 1, 1)
    rq, rk = oracle.rope(Q, cos, sin)[0, :, 0], oracle.rope(K, cos, sin)[0, :, 0]
    assert abs(float(rq[10] @ rk[3]) - float(rq[27] @ rk[20])) < 1e-12
    # backward is the transpose of the forward map
    a = torch.randn(2, S, 3, hd, generator=g)
    b = torch.randn(2, S, 3, hd, generator=g)
    lhs = (oracle.rope(a, cos, sin) * b).sum()
    rhs = (a * oracle.rope_backward(b, cos, sin)).sum()
    assert abs(float(lhs - rhs)) < 1e-11


# ---------------------------------------------------------------- attention

@pytest.mark.parametrize("Hq,Hkv,hd,S", [(4, 4, 16, 9), (6, 2, 8, 13), (5, 1, 32, 7)])
def test_attention_matches_library_sdpa_and_its_autograd(Hq, Hkv, hd, S):
    g = torch.Generator().manual_seed(4)
    B = 2
    q = torch.randn(B, S, Hq, hd, generator=g)
    k = torch.randn(B, S, Hkv, hd, generator=g)
    v = torch.randn(B, S, Hkv, hd, generator=g)
    o, probs = oracle.causal_gqa_attention(q, k, v)
    qa, ka, va = (t.transpose(1, 2).clone().requires_grad_() for t in (q, k, v))
    ref = F.scaled_dot_product_attention(qa, ka, va, is_causal=True, enable_gqa=True)
    assert torch.allclose(o, ref.transpose(1, 2), rtol=1e-12, atol=1e-12)
    do = torch.randn_like(o)
    ref.backward(do.transpose(1, 2))
    dq, dk, dv = oracle.causal_gqa_attention_backward(do, q, k, v, probs)
    assert torch.allclose(dq, qa.grad.transpose(1, 2), rtol=1e-11, atol=1e-12)
    assert torch.allclose(dk, ka.grad.transpose(1, 2), rtol=1e-11, atol=1e-12)
    assert torch.allclose(dv, va.grad.transpose(1, 2), rtol=1e-11, atol=1e-12)


def test_attention_special_cases():
    g = torch.Generator().manual_seed(5)
    # one token: softmax over one key, o = v
    q = torch.randn(2, 1, 4, 8, generator=g)
    k = torch.randn(2, 1, 2, 8, generator=g)
    v = torch.randn(2, 1, 2, 8, generator=g)
    o, probs = oracle.causal_gqa_attention(q, k, v)
    assert torch.allclose(o, v.repeat_interleave(2, dim=2), rtol=0, atol=0)
    # GQA equals MHA on kv heads repeated Hq/Hkv times (head h reads kv head h // group)
    q = torch.randn(1, 11, 6, 8, generator=g)
    k = torch.randn(1, 11, 3, 8, generator=g)
    v = torch.randn(1, 11, 3, 8, generator=g)
    o1, probs = oracle.causal_gqa_attention(q, k, v)
    o2, _ = oracle.causal_gqa_attention(q, k.repeat_interleave(2, 2), v.repeat_interleave(2, 2))
    assert torch.allclose(o1, o2, rtol=0, atol=1e-15)
    # rows of P sum to 1 and row i puts no weight on keys after i
    p = probs[0][3]
    assert torch.allclose(p.sum(-1), torch.ones(11), rtol=1e-14)
    assert torch.all(p.triu(1) == 0)
    # first query attends to the first key only
    assert torch.allclose(o1[0, 0], v[0, 0].repeat_interleave(2, 0).reshape(6, 8), atol=1e-15)


def test_attention_row_functions_agree_with_full_matrix():
    """The per-row and per-key forms (for long sequences) give the full-matrix
    oracle's output, lse, dq, dk and dv."""
    g = torch.Generator().manual_seed(41)
    S, hd, G = 37, 16, 3
    q = torch.randn(1, S, G, hd, generator=g)
    k = torch.randn(1, S, 1, hd, generator=g)
    v = torch.randn(1, S, 1, hd, generator=g)
    do = torch.randn(1, S, G, hd, generator=g)
    o, probs = oracle.causal_gqa_attention(q, k, v)
    dq, dk, dv = oracle.causal_gqa_attention_backward(do, q, k, v, probs)
    rows = [0, 5, 36]
    for h in range(G):
        o_r, lse_r, dq_r = oracle.attention_rows(q[0, :, h], k[0, :, 0], v[0, :, 0], rows, do[0, :, h])
        assert torch.allclose(o_r, o[0, rows, h], atol=1e-13)
        assert torch.allclose(dq_r, dq[0, rows, h], atol=1e-12)
        sc = (q[0, :, h] @ k[0, :, 0].T) / math.sqrt(hd)
        sc = sc.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
        assert torch.allclose(lse_r, torch.logsumexp(sc, -1)[rows], atol=1e-13)
    for j in (0, 20, 36):
        dk_j, dv_j = oracle.attention_key_grads(q[0].permute(1, 0, 2), k[0, :, 0], v[0, :, 0],
                                                do[0].permute(1, 0, 2), j)
        assert torch.allclose(dk_j, dk[0, j, 0], atol=1e-12)
        assert torch.allclose(dv_j, dv[0, j, 0], atol=1e-12)


@pytest.mark.parametrize("t0", [0, 23, 36])
def test_layer_tail_rows_equals_full_layer_with_zero_padded_gradient(t0):
    """The tail-rows layer (for long sequences) reproduces layer_forward and
    layer_backward exactly when dL/dx' is zero before row t0."""
    cfg = OracleConfig(n_layers=1, d_model=32, n_heads=4, n_kv_heads=2, head_dim=8, ffn=40, vocab=16,
                       rms_eps=1e-5, rope_theta=1e4, lr=1e-4, beta1=0.9, beta2=0.95, adam_eps=1e-8,
                       weight_decay=0.0)
    g = torch.Generator().manual_seed(43)
    S = 37
    shapes = dict(g1=(32,), wq=(32, 32), wk=(16, 32), wv=(16, 32), wo=(32, 32), g2=(32,), wg=(40, 32),
                  wu=(40, 32), wd=(32, 40))
    lw = {k: (1 + 0.3 * torch.randn(sh, generator=g)) if len(sh) == 1 else 0.3 * torch.randn(sh, generator=g)
          for k, sh in shapes.items()}
    x = torch.randn(1, S, 32, generator=g)
    dy = torch.randn(1, S, 32, generator=g)
    dy[:, :t0] = 0
    cos, sin = oracle.rope_cos_sin(S, 8, 1e4)
    y_ref, c = oracle.layer_forward(x, lw, cfg, cos, sin)
    dx_ref, g_ref = oracle.layer_backward(dy, c, lw, cfg, cos, sin)
    y, dx, gr = oracle.layer_tail_rows(x[0], dy[0, t0:], lw, cfg, cos, sin, t0)
    assert torch.allclose(y, y_ref[0, t0:], atol=1e-12)
    assert torch.allclose(dx, dx_ref[0], atol=1e-12)
    for k in shapes:
        assert torch.allclose(gr[k], g_ref[k], atol=1e-11), k


# ---------------------------------------------------------------- SwiGLU

def test_swiglu_matches_library_and_autograd():
    g = torch.Generator().manual_seed(6)
    a = torch.randn(20, 30, generator=g) * 3
    b = torch.randn(20, 30, generator=g)
    assert torch.allclose(oracle.swiglu(a, b), F.silu(a) * b, rtol=1e-14, atol=1e-15)
    aa, ba = a.clone().requires_grad_(), b.clone().requires_grad_()
    d = torch.randn(20, 30, generator=g)
    (F.silu(aa) * ba).backward(d)
    da, db = oracle.swiglu_backward(d, a, b)
    assert torch.allclose(da, aa.grad, rtol=1e-13, atol=1e-14)
    assert torch.allclose(db, ba.grad, rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- head / CE

def test_head_matches_library_cross_entropy_and_autograd():
    s, cfg = _tiny(n_layers=0, vocab=50, d_model=24, batch=3, seq=5)
    g = torch.Generator().manual_seed(7)
    x = torch.randn(3, 5, 24, generator=g)
    hw = {"gf": 1 + 0.2 * torch.randn(24, generator=g), "wh": 0.3 * torch.randn(50, 24, generator=g)}
    tgt = torch.randint(0, 50, (3, 5), generator=g)
    loss, dx, grads = oracle.head_loss_and_backward(x, hw, tgt, cfg)
    xa = x.clone().requires_grad_()
    ga = hw["gf"].clone().requires_grad_()
    wa = hw["wh"].clone().requires_grad_()
    ref = F.cross_entropy(F.linear(F.rms_norm(xa, (24,), ga, 1e-5), wa).reshape(-1, 50), tgt.reshape(-1))
    ref.backward()
    assert abs(float(loss) - float(ref.detach())) < 1e-13
    assert torch.allclose(dx, xa.grad, rtol=1e-11, atol=1e-14)
    assert torch.allclose(grads["gf"], ga.grad, rtol=1e-11, atol=1e-14)
    assert torch.allclose(grads["wh"], wa.grad, rtol=1e-11, atol=1e-14)
    # each row of dz sums to zero, so the rows of dW_h sum to zero
    assert torch.allclose(grads["wh"].sum(0), torch.zeros(24), atol=1e-14)


def test_head_single_token_vocab_has_zero_loss():
    s, cfg = _tiny(n_layers=0, vocab=1, d_model=8)
    g = torch.Generator().manual_seed(8)
    x = torch.randn(2, 4, 8, generator=g)
    hw = {"gf": torch.ones(8), "wh": torch.randn(1, 8, generator=g)}
    loss, dx, grads = oracle.head_loss_and_backward(x, hw, torch.zeros(2, 4, dtype=torch.long), cfg)
    assert float(loss) == 0.0
    assert torch.all(dx == 0) and torch.all(grads["wh"] == 0)


# ---------------------------------------------------------------- whole model

def _library_model_loss(params, tokens, cfg):
    """The same decoder written with library routines (autograd-capable)."""
    inp, tgt = tokens[:, :-1].long(), tokens[:, 1:].long()
    B, S = inp.shape
    cos, sin = oracle.rope_cos_sin(S, cfg.head_dim, cfg.rope_theta)
    x = F.embedding(inp, params["embed"]["E"])
    for lw in params["layers"]:
        n = F.rms_norm(x, (cfg.d_model,), lw["g1"], cfg.rms_eps)
        q = oracle.rope(F.linear(n, lw["wq"]).reshape(B, S, cfg.n_heads, cfg.head_dim), cos, sin)
        k = oracle.rope(F.linear(n, lw["wk"]).reshape(B, S, cfg.n_kv_heads, cfg.head_dim), cos, sin)
        v = F.linear(n, lw["wv"]).reshape(B, S, cfg.n_kv_heads, cfg.head_dim)
        o = F.scaled_dot_product_attention(q.transpose(1, 2), k.transpose(1, 2), v.transpose(1, 2),
                                           is_causal=True, enable_gqa=True).transpose(1, 2)
        h = x + F.linear(o.reshape(B, S, -1), lw["wo"])
        n2 = F.rms_norm(h, (cfg.d_model,), lw["g2"], cfg.rms_eps)
        x = h + F.linear(F.silu(F.linear(n2, lw["wg"])) * F.linear(n2, lw["wu"]), lw["wd"])
    nf = F.rms_norm(x, (cfg.d_model,), params["head"]["gf"], cfg.rms_eps)
    return F.cross_entropy(F.linear(nf, params["head"]["wh"]).reshape(-1, cfg.vocab), tgt.reshape(-1))


def _as_f64(params, requires_grad=False):
    f = lambda t: t.to(D).clone().requires_grad_(requires_grad)
    return {"embed": {k: f(v) for k, v in params["embed"].items()},
            "layers": [{k: f(v) for k, v in lw.items()} for lw in params["layers"]],
            "head": {k: f(v) for k, v in params["head"].items()}}


def _flat(tree):
    out = [tree["embed"]["E"]]
    for lw in tree["layers"]:
        out += [lw[k] for k in mt_inputs.LAYER_TENSORS]
    out += [tree["head"]["gf"], tree["head"]["wh"]]
    return out


def _gqa_tiny():
    return _tiny(n_heads=4, n_kv_heads=2, head_dim=32, d_model=128, ffn=200, vocab=97, seq=24)


@pytest.mark.parametrize("which", ["tiny", "gqa"])
def test_model_grads_match_autograd_of_library_forward(which):
    s, cfg = _tiny() if which == "tiny" else _gqa_tiny()
    params = mt_inputs.model_weights(s, gain_jitter=0.1)
    tokens = mt_inputs.step_tokens(s, 1)
    loss, grads = oracle.model_loss_and_grads(params, tokens, cfg)
    p = _as_f64(params, requires_grad=True)
    ref = _library_model_loss(p, tokens, cfg)
    ref.backward()
    assert abs(loss - float(ref.detach())) < 1e-12 * abs(loss)
    for mine, theirs in zip(_flat(grads), _flat(p)):
        err = (mine - theirs.grad).norm() / theirs.grad.norm()
        assert err < 1e-10, err


@pytest.mark.parametrize("which", ["tiny", "gqa"])
def test_tied_model_grads_match_autograd_of_library_forward(which):
    """Tied embedding and LM head: autograd through the library's forward with
    one leaf tensor used both as the embedding table and as the head weight
    accumulates both uses into its gradient; the oracle's tied dE must match."""
    s, cfg = _tiny() if which == "tiny" else _gqa_tiny()
    params = mt_inputs.tied(mt_inputs.model_weights(s, gain_jitter=0.1))
    tokens = mt_inputs.step_tokens(s, 2)
    loss, grads = oracle.model_loss_and_grads(params, tokens, cfg)
    assert set(grads["head"]) == {"gf"}
    p = _as_f64(params, requires_grad=True)
    ref = _library_model_loss(dict(p, head={"gf": p["head"]["gf"], "wh": p["embed"]["E"]}), tokens, cfg)
    ref.backward()
    assert abs(loss - float(ref.detach())) < 1e-12 * abs(loss)
    pairs = [(grads["embed"]["E"], p["embed"]["E"]), (grads["head"]["gf"], p["head"]["gf"])]
    for gl, pl in zip(grads["layers"], p["layers"]):
        pairs += [(gl[k], pl[k]) for k in mt_inputs.LAYER_TENSORS]
    for mine, theirs in pairs:
        err = (mine - theirs.grad).norm() / theirs.grad.norm()
        assert err < 1e-10, err
    # the tied gradient of E is the untied embedding gradient plus the untied head gradient
    untied = dict(params, head={"gf": params["head"]["gf"], "wh": params["embed"]["E"]})
    _, gu = oracle.model_loss_and_grads(untied, tokens, cfg)
    assert torch.allclose(grads["embed"]["E"], gu["embed"]["E"] + gu["head"]["wh"], rtol=0, atol=1e-14)


def test_tied_model_grad_finite_differences():
    """Central differences along random directions of (E, gf) in the tied model:
    a perturbation of E moves both the embedding lookups and the logits."""
    s, cfg = _tiny(n_layers=1, d_model=64, n_heads=2, n_kv_heads=1, head_dim=32, ffn=96, vocab=61, seq=12)
    params = _as_f64(mt_inputs.tied(mt_inputs.model_weights(s, gain_jitter=0.1)))
    tokens = mt_inputs.step_tokens(s, 4)
    _, grads = oracle.model_loss_and_grads(params, tokens, cfg)
    gen = torch.Generator().manual_seed(13)
    for trial in range(3):
        uE = torch.randn(params["embed"]["E"].shape, generator=gen, dtype=D)
        ug = torch.randn(params["head"]["gf"].shape, generator=gen, dtype=D)
        nrm = math.sqrt(float((uE * uE).sum() + (ug * ug).sum()))
        uE, ug = uE / nrm, ug / nrm
        h = 1e-5

        def at(sign):
            q = _as_f64(params)
            q["embed"]["E"].add_(sign * h * uE)
            q["head"]["gf"].add_(sign * h * ug)
            return oracle.model_forward_loss(q, tokens, cfg)

        fd = (at(1) - at(-1)) / (2 * h)
        an = float((grads["embed"]["E"] * uE).sum() + (grads["head"]["gf"] * ug).sum())
        assert abs(fd - an) <= 1e-6 * abs(an) + 1e-11, (fd, an)


def test_model_grad_finite_differences():
    """Central differences of the oracle's own forward, in FP64.

    Random directions over all weights at once (<grad, u> against
    (L(w+hu) - L(w-hu)) / 2h) and single coordinates of every tensor.
    """
    s, cfg = _tiny(n_layers=2, d_model=64, n_heads=2, n_kv_heads=1, head_dim=32, ffn=96, vocab=61, seq=12)
    params = mt_inputs.model_weights(s, gain_jitter=0.1)
    params = _as_f64(params)
    tokens = mt_inputs.step_tokens(s, 3)
    loss, grads = oracle.model_loss_and_grads(params, tokens, cfg)
    flat_p, flat_g = _flat(params), _flat(grads)
    gen = torch.Generator().manual_seed(9)

    def shifted(delta):
        out = _as_f64(params)
        for t, d_ in zip(_flat(out), delta):
            t.add_(d_)
        return out

    for trial in range(3):
        u = [torch.randn(t.shape, generator=gen) for t in flat_p]
        nrm = math.sqrt(sum(float((x * x).sum()) for x in u))
        u = [x / nrm for x in u]
        h = 1e-5
        lp = oracle.model_forward_loss(shifted([h * x for x in u]), tokens, cfg)
        lm = oracle.model_forward_loss(shifted([-h * x for x in u]), tokens, cfg)
        fd = (lp - lm) / (2 * h)
        an = sum(float((gg * x).sum()) for gg, x in zip(flat_g, u))
        assert abs(fd - an) <= 1e-6 * abs(an) + 1e-11, (fd, an)

    # two coordinates of every tensor (the largest-gradient entry and one random entry)
    for ti, (t, gt) in enumerate(zip(flat_p, flat_g)):
        idxs = [int(gt.abs().argmax()), int(torch.randint(0, t.numel(), (1,), generator=gen))]
        for idx in idxs:
            h = 1e-6
            delta = [torch.zeros_like(x) for x in flat_p]
            delta[ti].view(-1)[idx] = h
            lp = oracle.model_forward_loss(shifted(delta), tokens, cfg)
            delta[ti].view(-1)[idx] = -h
            lm = oracle.model_forward_loss(shifted(delta), tokens, cfg)
            fd = (lp - lm) / (2 * h)
            an = float(gt.view(-1)[idx])
            assert abs(fd - an) <= 1e-6 * abs(an) + 1e-9, (ti, idx, fd, an)


def test_zero_output_projections_make_layers_identity():
    """With W_o = W_d = 0 every layer passes x through, so the loss is the
    closed form embed -> RMSNorm -> LM head -> cross-entropy."""
    s, cfg = _tiny()
    params = mt_inputs.model_weights(s)
    for lw in params["layers"]:
        lw["wo"] = torch.zeros_like(lw["wo"])
        lw["wd"] = torch.zeros_like(lw["wd"])
    tokens = mt_inputs.step_tokens(s, 2)
    loss, grads = oracle.model_loss_and_grads(params, tokens, cfg)
    inp, tgt = tokens[:, :-1].long(), tokens[:, 1:].long()
    E = params["embed"]["E"].to(D)
    nf = F.rms_norm(F.embedding(inp, E), (s.d_model,), params["head"]["gf"].to(D), 1e-5)
    ref = F.cross_entropy((nf @ params["head"]["wh"].to(D).T).reshape(-1, s.vocab), tgt.reshape(-1))
    assert abs(loss - float(ref)) < 1e-12
    # nothing flows into the attention / MLP inputs when their outputs are zeroed
    for lg in grads["layers"]:
        for k in ("wq", "wk", "wv", "wg", "wu", "g1", "g2"):
            assert torch.all(lg[k] == 0)


def test_loss_at_init_is_near_log_vocab():
    s, cfg = _tiny()
    loss = oracle.model_forward_loss(mt_inputs.model_weights(s), mt_inputs.step_tokens(s, 1), cfg)
    # small logits (std ~ 0.02 * sqrt(d) = 0.32): loss ~ ln V + sigma^2 / 2
    assert math.log(s.vocab) - 0.05 < loss < math.log(s.vocab) + 0.15


def test_recompute_changes_nothing():
    """Re-running a layer's forward from its input gives the same cache (the
    schedule's recompute is a pure function of x and the weights)."""
    s, cfg = _tiny()
    params = _as_f64(mt_inputs.model_weights(s))
    tokens = mt_inputs.step_tokens(s, 1)
    cos, sin = oracle.rope_cos_sin(s.seq, s.head_dim, s.rope_theta)
    x = params["embed"]["E"][tokens[:, :-1].long()]
    y1, c1 = oracle.layer_forward(x, params["layers"][0], cfg, cos, sin)
    y2, c2 = oracle.layer_forward(x.clone(), params["layers"][0], cfg, cos, sin)
    assert torch.equal(y1, y2) and torch.equal(c1["a"], c2["a"])


# ---------------------------------------------------------------- Adam

def test_adam_first_step_is_lr_times_sign():
    s, cfg = _tiny()
    w = torch.tensor([0.5, -0.25, 0.0078125, 3.0, 0.125]).to(torch.bfloat16).to(D)
    g = torch.tensor([1e-3, -2e-5, 0.0, 7.0, -1e-6]).to(torch.bfloat16).to(D)
    z = torch.zeros(5)
    wn, m, v = oracle.adam_update(w, g, z, z, 1, cfg)
    # m = (1-b1) g, v = (1-b2) g^2, mhat = g, vhat = g^2: update = lr * g / (|g| + eps)
    expect = oracle.round_to_bf16(w - cfg.lr * g / (g.abs() + cfg.adam_eps))
    assert torch.equal(wn, expect)
    assert wn[2] == w[2]  # zero gradient leaves the weight unchanged
    step = oracle.round_to_bf16(w - cfg.lr * torch.sign(g))
    big = g.abs() > 1e-4
    assert torch.equal(wn[big], step[big])
    assert torch.allclose(m, 0.1 * g, rtol=1e-7)
    assert torch.allclose(v, 0.05 * g * g, rtol=1e-7)


def test_adam_fp32_arithmetic_first_step_is_lr_times_sign():
    """The FP32 arithmetic of the timed CPU baseline reaches the same closed
    form at t = 1: update = lr * sign(g) where |g| >> eps, none where g = 0."""
    s, cfg = _tiny()
    w = torch.tensor([0.5, -0.25, 0.0078125, 3.0, 0.125]).to(torch.bfloat16).to(D)
    g = torch.tensor([1e-3, -2e-5, 0.0, 7.0, -1e-6]).to(torch.bfloat16).to(D)
    z = torch.zeros(5)
    wn, m, v = oracle.adam_update(w, g, z, z, 1, cfg, dtype=torch.float32)
    assert wn[2] == w[2]
    big = g.abs() > 1e-4
    assert torch.equal(wn[big], oracle.round_to_bf16(w - cfg.lr * torch.sign(g))[big])
    w64, _, _ = oracle.adam_update(w, g, z, z, 1, cfg)
    ulp = torch.ldexp(torch.ones_like(w64), torch.frexp(w64)[1] - 8)
    assert ((wn - w64).abs() <= ulp).all()


def test_adam_two_steps_exact_rationals():
    """Two Adam steps on three elements, worked in exact rational arithmetic
    (eps = 0 so the square roots are exact for these perfect-square inputs)."""
    cfg = OracleConfig(0, 1, 1, 1, 1, 1, 1, lr=Fraction(1, 64).__float__(), beta1=0.5, beta2=0.75,
                       adam_eps=0.0)
    g1 = [Fraction(4), Fraction(-2), Fraction(1)]
    g2 = [Fraction(10), Fraction(2), Fraction(-1)]  # 3*g1^2 + 4*g2^2 = 7 r^2 keeps vhat square
    w0 = [Fraction(1), Fraction(1, 2), Fraction(-3, 4)]
    b1, b2, lr = Fraction(1, 2), Fraction(3, 4), Fraction(1, 64)
    m = [Fraction(0)] * 3
    v = [Fraction(0)] * 3
    w = list(w0)
    for t, g in ((1, g1), (2, g2)):
        m = [b1 * mi + (1 - b1) * gi for mi, gi in zip(m, g)]
        v = [b2 * vi + (1 - b2) * gi * gi for vi, gi in zip(v, g)]
        # hand-evaluated bias corrections: 1-b1^t, 1-b2^t
        c1, c2 = 1 - b1 ** t, 1 - b2 ** t
        upd = []
        for mi, vi, wi in zip(m, v, w):
            vh = vi / c2
            # sqrt of a rational perfect square
            num, den = vh.numerator, vh.denominator
            r = Fraction(math.isqrt(num), math.isqrt(den))
            assert r * r == vh
            upd.append(wi - lr * (mi / c1) / r)
        w = upd
    # feed the oracle the same sequence
    wt = torch.tensor([float(x) for x in w0])
    mt = torch.zeros(3)
    vt = torch.zeros(3)
    for t, g in ((1, g1), (2, g2)):
        wt, mt, vt = oracle.adam_update(wt, torch.tensor([float(x) for x in g]), mt, vt, t, cfg)
    assert wt.tolist() == [float(oracle.round_to_bf16(torch.tensor([float(x)]))[0]) for x in w]
    assert mt.tolist() == [float(x) for x in m]
    assert vt.tolist() == [float(x) for x in v]


def test_train_step_applies_adam_to_bf16_rounded_grads():
    s, cfg = _tiny()
    params = mt_inputs.model_weights(s)
    tokens = mt_inputs.step_tokens(s, 1)
    loss, grads, new_p, new_s = oracle.train_step(params, None, tokens, 1, cfg)
    gq = oracle.round_to_bf16(grads["layers"][1]["wq"])
    w = params["layers"][1]["wq"].to(D)
    expect = oracle.round_to_bf16(w - cfg.lr * gq / (gq.abs() + cfg.adam_eps))
    assert torch.equal(new_p["layers"][1]["wq"], expect)
    # embedding rows of tokens that never appear get no update (0 / (0 + eps) = 0)
    used = torch.zeros(s.vocab, dtype=torch.bool)
    used[tokens[:, :-1].long().reshape(-1)] = True
    E0 = params["embed"]["E"].to(D)
    assert torch.equal(new_p["embed"]["E"][~used], E0[~used])


def test_precision_model_without_rounding_is_the_oracle_in_fp32():
    """The storage-precision model (tests/precision_model.py) with every
    rounding point off is the same step in FP32: its loss and gradients match
    the FP64 oracle to FP32 accuracy, and switching all points on moves the
    gradients by about the BF16 scale."""
    from tests import parity, precision_model as pm
    s = mt_inputs.PRESETS["tiny"].with_(batch=1, seq=48)
    cfg = OracleConfig.from_shape(s)
    params = mt_inputs.model_weights(s, gain_jitter=0.1)
    tokens = mt_inputs.step_tokens(s, 1)
    loss_ref, gref = oracle.model_loss_and_grads(params, tokens, cfg)
    loss, g = pm.Model(()).loss_and_grads(params, tokens, cfg)
    assert abs(loss - loss_ref) < 1e-5 * abs(loss_ref)
    assert max(r for _, _, r in parity.grad_report(g, gref)) < 1e-4
    _, gb = pm.Model(pm.ALL).loss_and_grads(params, tokens, cfg)
    worst = max(r for _, _, r in parity.grad_report(gb, gref))
    assert 1e-3 < worst < 5e-2
