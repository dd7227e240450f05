"""Comparison helpers shared by the GPU parity tests (test code, not product).

Tolerances are the ones the target sets for the training step:
  * loss: relative error <= 1e-2;
  * every tensor's gradient: cosine >= 0.999 and normwise relative error <= 2e-2;
  * updated weights: within 1 BF16 ulp of the oracle's Adam update applied in
    BF16.  Read as (i) the oracle's Adam applied to the library's own BF16
    gradients matches the library's new weights within 1 ulp everywhere
    (or, where the update cancels the weight, within the FP32 error bound of
    the host's subtraction: ``adam_weight_tol``), and
    (ii) against the oracle's own gradients, within 1 ulp wherever the two
    gradients have the same sign and the oracle gradient is not negligible
    (|g| > 1e-3 * rms(g)); elsewhere a 2-ulp move is expected and only counted.
"""
from __future__ import annotations

import math

import torch

import mt_inputs
import oracle

LOSS_RTOL = 1e-2
GRAD_COS = 0.999
GRAD_RTOL = 2e-2
D = torch.float64


def flat_named(tree):
    out = [("embed.E", tree["embed"]["E"])]
    for i, lw in enumerate(tree["layers"]):
        if "experts" in lw:  # MoE layer
            for k in ("g1", "wq", "wk", "wv", "wo", "g2", "wr"):
                out.append((f"layers.{i}.{k}", lw[k]))
            for e, ew in enumerate(lw["experts"]):
                for k in ("wg", "wu", "wd"):
                    out.append((f"layers.{i}.experts.{e}.{k}", ew[k]))
            continue
        for k in mt_inputs.LAYER_TENSORS:
            out.append((f"layers.{i}.{k}", lw[k]))
    out.append(("head.gf", tree["head"]["gf"]))
    if "wh" in tree["head"]:  # absent with tied embeddings (E is the head's weight)
        out.append(("head.wh", tree["head"]["wh"]))
    return out


def grad_report(lib_grads, ora_grads):
    """Per tensor: (name, cosine, normwise relative error)."""
    rep = []
    for (n, a), (_, b) in zip(flat_named(lib_grads), flat_named(ora_grads)):
        a = a.to(D).reshape(-1)
        b = b.to(D).reshape(-1)
        nb = float(b.norm())
        na = float(a.norm())
        if nb == 0.0:
            rep.append((n, 1.0 if na == 0.0 else 0.0, 0.0 if na == 0.0 else math.inf))
            continue
        cos = float(a @ b) / max(na * nb, 1e-300)
        rel = float((a - b).norm()) / nb
        rep.append((n, cos, rel))
    return rep


def assert_grads_close(lib_grads, ora_grads):
    bad = [(n, c, r) for n, c, r in grad_report(lib_grads, ora_grads) if not (c >= GRAD_COS and r <= GRAD_RTOL)]
    assert not bad, f"gradient tensors outside cos>={GRAD_COS}, rel<={GRAD_RTOL}: {bad[:8]}"


def bf16_ulp(x):
    """Spacing of BF16 numbers at |x| (8 significant bits)."""
    x = x.to(D).abs()
    _, e = torch.frexp(torch.where(x == 0, torch.full_like(x, 2.0 ** -126), x))
    return torch.ldexp(torch.ones_like(x), (e - 8).to(D))


def adam_weight_tol(we, w0):
    """Allowed |w_lib - w_oracle| for one Adam update of BF16 weights.

    1 BF16 ulp of the expected weight, or, where the update nearly cancels the
    weight (w - lr*u with lr*u ~ w), the FP32 error bound of that subtraction:
    the host computes the update in FP32 (reading A7), whose operands carry
    <= 2^-24 relative rounding each, i.e. a few FP32 ulps of |w0|.
    """
    return torch.maximum(bf16_ulp(we), 4 * 2.0 ** -24 * w0.to(D).abs())


def fp32_hyper(cfg):
    """The oracle config with Adam hyper-parameters rounded to FP32, as the C-ABI receives them."""
    import dataclasses
    f = lambda x: float(torch.tensor(x, dtype=torch.float32))
    return dataclasses.replace(cfg, lr=f(cfg.lr), beta1=f(cfg.beta1), beta2=f(cfg.beta2), adam_eps=f(cfg.adam_eps),
                               weight_decay=f(cfg.weight_decay))


def assert_adam_matches(lib_w_new, lib_w_old, lib_g, lib_m, lib_v, step, cfg, m_old=None, v_old=None):
    """Reading (i): the oracle's Adam on the library's BF16 gradients."""
    cfg = fp32_hyper(cfg)
    for (n, wn), (_, wo), (_, g), (_, m), (_, v) in zip(flat_named(lib_w_new), flat_named(lib_w_old),
                                                         flat_named(lib_g), flat_named(lib_m), flat_named(lib_v)):
        mo = torch.zeros_like(g, dtype=D) if m_old is None else dict(flat_named(m_old))[n]
        vo = torch.zeros_like(g, dtype=D) if v_old is None else dict(flat_named(v_old))[n]
        we, me, ve = oracle.adam_update(wo, g, mo, vo, step, cfg)
        diff = (wn.to(D) - we).abs()
        tol = adam_weight_tol(we, wo)
        assert torch.all(diff <= tol), f"{n}: {int((diff > tol).sum())} weights beyond 1 BF16 ulp"
        # FP32 moments: within a few FP32 ulps of the larger of the two terms
        gd = g.to(D)
        assert torch.all((m.to(D) - me).abs() <= 4 * 2.0 ** -24 * (cfg.beta1 * mo.to(D).abs() + (1 - cfg.beta1) * gd.abs())), \
            f"{n}: first moment"
        assert torch.all((v.to(D) - ve).abs() <= 4 * 2.0 ** -24 * (cfg.beta2 * vo.to(D) + (1 - cfg.beta2) * gd * gd)), \
            f"{n}: second moment"


def adam_vs_oracle_grads(lib_w_new, lib_w_old, ora_grads, step, cfg):
    """Reading (ii): fraction of weights within 1 ulp where the comparison is meaningful."""
    total = ok = excluded = 0
    worst = []
    for (n, wn), (_, wo), (_, go) in zip(flat_named(lib_w_new), flat_named(lib_w_old), flat_named(ora_grads)):
        gb = oracle.round_to_bf16(go.to(D))
        z = torch.zeros_like(gb)
        we, _, _ = oracle.adam_update(wo, gb, z, z, step, cfg)
        diff = (wn.to(D) - we).abs()
        ulp = bf16_ulp(we)
        rms = float(go.to(D).pow(2).mean().sqrt()) if go.numel() else 0.0
        meaningful = go.to(D).abs() > 1e-3 * rms
        within = diff <= ulp
        total += int(meaningful.sum())
        ok += int((within & meaningful).sum())
        excluded += int((~meaningful).sum())
        if int((~within & meaningful).sum()):
            worst.append((n, int((~within & meaningful).sum())))
    return ok, total, excluded, worst
