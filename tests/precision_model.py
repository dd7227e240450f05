"""CPU model of the library's storage precision (test infrastructure).

The training step written out again in FP32 with BF16 rounding at the points
where the GPU path stores BF16 between kernels (reading A10: BF16 storage,
FP32 arithmetic), each point switchable:

  n      RMSNorm outputs (the GEMM A operands n1, n2, nf)
  qkv    q, k (after RoPE) and v
  P      attention probabilities used for P V
  o      attention output
  res    residual stream h and the layer output
  mlp    gate, up and the SwiGLU activation
  bwd    every gradient tensor passed between kernels (dz, dnf, dx, da, dgu, dn, dO, dqkv)
  dS     P and dS in the attention backward
  grad   the stored weight gradients

Comparing its gradients with the FP64 oracle's tells how far *any*
implementation with these storage points must land from the oracle, so that
the GPU path's own error can be told apart from the precision model's:

    python -m tests.precision_model 14b [seq]

prints, for the full-width two-layer model, the worst normwise relative
gradient errors with all points on and with each point alone.  Only
``tests/`` uses this module; it shares nothing with the library.
"""
from __future__ import annotations

import math
import os
import sys

import torch

import mt_inputs
import oracle
from oracle import OracleConfig

F = torch.float32
ALL = frozenset({"n", "qkv", "P", "o", "res", "mlp", "bwd", "dS", "grad"})


class Model:
    def __init__(self, active):
        self.active = frozenset(active)

    def rb(self, x, key):
        return x.to(torch.bfloat16).to(F) if key in self.active else x

    @staticmethod
    def rms(x, g, eps):
        r = torch.rsqrt((x * x).mean(-1, keepdim=True) + eps)
        return x * r * g, r

    @staticmethod
    def rms_bwd(dy, x, g, r):
        xh = x * r
        dyg = dy * g
        return r * (dyg - xh * (dyg * xh).mean(-1, keepdim=True)), (dy * xh).sum(0)

    @staticmethod
    def rope(x, c, s):  # x [S, H, hd]
        h = x.shape[-1] // 2
        x1, x2 = x[..., :h], x[..., h:]
        return torch.cat([x1 * c[:, None] - x2 * s[:, None], x2 * c[:, None] + x1 * s[:, None]], -1)

    @staticmethod
    def rope_bwd(d, c, s):
        h = d.shape[-1] // 2
        d1, d2 = d[..., :h], d[..., h:]
        return torch.cat([d1 * c[:, None] + d2 * s[:, None], d2 * c[:, None] - d1 * s[:, None]], -1)

    def layer_fwd(self, x, w, cfg, c, s):
        rb = self.rb
        S = x.shape[0]
        Hq, Hkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
        n1, r1 = self.rms(x, w["g1"], cfg.rms_eps)
        n1 = rb(n1, "n")
        q = rb(self.rope((n1 @ w["wq"].T).reshape(S, Hq, hd), c, s), "qkv")
        k = rb(self.rope((n1 @ w["wk"].T).reshape(S, Hkv, hd), c, s), "qkv")
        v = rb((n1 @ w["wv"].T).reshape(S, Hkv, hd), "qkv")
        sc = 1 / math.sqrt(hd)
        mask = torch.ones(S, S, dtype=torch.bool).triu(1)
        o = torch.empty(S, Hq, hd, dtype=F)
        lse = torch.empty(Hq, S, dtype=F)
        for h in range(Hq):
            j = h * Hkv // Hq
            z = ((q[:, h] @ k[:, j].T) * sc).masked_fill(mask, -float("inf"))
            m = z.max(-1, keepdim=True).values
            p = torch.exp(z - m)
            l = p.sum(-1, keepdim=True)
            o[:, h] = (rb(p, "P") @ v[:, j]) / l
            lse[h] = (m + torch.log(l))[:, 0]
        o = rb(o.reshape(S, -1), "o")
        hh = rb(x + o @ w["wo"].T, "res")
        n2, r2 = self.rms(hh, w["g2"], cfg.rms_eps)
        n2 = rb(n2, "n")
        gate, up = n2 @ w["wg"].T, n2 @ w["wu"].T
        a = rb(gate * torch.sigmoid(gate) * up, "mlp")
        gate, up = rb(gate, "mlp"), rb(up, "mlp")
        xo = rb(hh + a @ w["wd"].T, "res")
        return xo, dict(x=x, n1=n1, r1=r1, q=q, k=k, v=v, o=o, lse=lse, h=hh, n2=n2, r2=r2, gate=gate, up=up, a=a)

    def layer_bwd(self, dxo, C, w, cfg, c, s):
        rb = self.rb
        S = dxo.shape[0]
        Hq, Hkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
        g = {"wd": rb(dxo.T @ C["a"], "grad")}
        da = rb(dxo @ w["wd"], "bwd")
        sg = torch.sigmoid(C["gate"])
        dgate = rb(da * C["up"] * sg * (1 + C["gate"] * (1 - sg)), "bwd")
        dup = rb(da * C["gate"] * sg, "bwd")
        g["wg"] = rb(dgate.T @ C["n2"], "grad")
        g["wu"] = rb(dup.T @ C["n2"], "grad")
        dn2 = rb(dgate @ w["wg"] + dup @ w["wu"], "bwd")
        dhn, dg2 = self.rms_bwd(dn2, C["h"], w["g2"], C["r2"])
        g["g2"] = rb(dg2, "grad")
        dh = rb(dxo + dhn, "bwd")
        g["wo"] = rb(dh.T @ C["o"], "grad")
        do = rb(dh @ w["wo"], "bwd").reshape(S, Hq, hd)
        o3 = C["o"].reshape(S, Hq, hd)
        sc = 1 / math.sqrt(hd)
        mask = torch.ones(S, S, dtype=torch.bool).triu(1)
        dq = torch.empty(S, Hq, hd, dtype=F)
        dk = torch.zeros(S, Hkv, hd, dtype=F)
        dv = torch.zeros(S, Hkv, hd, dtype=F)
        for h in range(Hq):
            j = h * Hkv // Hq
            z = (C["q"][:, h] @ C["k"][:, j].T) * sc
            p = torch.exp(z - C["lse"][h][:, None]).masked_fill(mask, 0)
            delta = (do[:, h] * o3[:, h]).sum(-1, keepdim=True)
            ds = p * (do[:, h] @ C["v"][:, j].T - delta)
            pb, dsb = rb(p, "dS"), rb(ds, "dS")
            dv[:, j] += pb.T @ do[:, h]
            dk[:, j] += dsb.T @ C["q"][:, h] * sc
            dq[:, h] = dsb @ C["k"][:, j] * sc
        dq = rb(self.rope_bwd(dq, c, s).reshape(S, -1), "bwd")
        dk = rb(self.rope_bwd(dk, c, s).reshape(S, -1), "bwd")
        dv = rb(dv.reshape(S, -1), "bwd")
        g["wq"] = rb(dq.T @ C["n1"], "grad")
        g["wk"] = rb(dk.T @ C["n1"], "grad")
        g["wv"] = rb(dv.T @ C["n1"], "grad")
        dn1 = rb(dq @ w["wq"] + dk @ w["wk"] + dv @ w["wv"], "bwd")
        dxn, dg1 = self.rms_bwd(dn1, C["x"], w["g1"], C["r1"])
        g["g1"] = rb(dg1, "grad")
        return rb(dh + dxn, "bwd"), g

    def loss_and_grads(self, params, tokens, cfg):
        """One sequence (tokens [1, S+1]); returns (loss, grads in the oracle's structure)."""
        rb = self.rb
        p = {"embed": {"E": params["embed"]["E"].to(F)},
             "layers": [{k: v.to(F) for k, v in lw.items()} for lw in params["layers"]],
             "head": {k: v.to(F) for k, v in params["head"].items()}}
        inp, tgt = tokens[0, :-1].long(), tokens[0, 1:].long()
        S = inp.shape[0]
        c, s = oracle.rope_cos_sin(S, cfg.head_dim, cfg.rope_theta, F)
        x = p["embed"]["E"][inp]
        caches = []
        for w in p["layers"]:
            x, C = self.layer_fwd(x, w, cfg, c, s)
            caches.append(C)
        nf, rf = self.rms(x, p["head"]["gf"], cfg.rms_eps)
        nf = rb(nf, "n")
        z = nf @ p["head"]["wh"].T
        loss = float((torch.logsumexp(z, -1) - z.gather(1, tgt[:, None])[:, 0]).mean())
        dz = torch.softmax(z, -1)
        dz[torch.arange(S), tgt] -= 1
        dz = rb(dz / S, "bwd")
        dnf = rb(dz @ p["head"]["wh"], "bwd")
        gh = {"wh": rb(dz.T @ nf, "grad")}
        dx, dgf = self.rms_bwd(dnf, x, p["head"]["gf"], rf)
        gh["gf"] = rb(dgf, "grad")
        dx = rb(dx, "bwd")
        lg = [None] * len(p["layers"])
        for i in reversed(range(len(p["layers"]))):
            dx, lg[i] = self.layer_bwd(dx, caches[i], p["layers"][i], cfg, c, s)
        dE = torch.zeros_like(p["embed"]["E"]).index_add_(0, inp, dx)
        return loss, {"embed": {"E": rb(dE, "grad")}, "layers": lg, "head": gh}


def main(argv):
    from tests import parity
    torch.set_num_threads(os.cpu_count() or 1)
    name = argv[1] if len(argv) > 1 else "14b"
    seq = int(argv[2]) if len(argv) > 2 else 200
    s = mt_inputs.PRESETS[name].with_(n_layers=2, batch=1, seq=seq)
    cfg = OracleConfig.from_shape(s)
    params = mt_inputs.model_weights(s, gain_jitter=0.1)
    tokens = mt_inputs.step_tokens(s, 1)
    loss_ref, gref = oracle.model_loss_and_grads(params, tokens, cfg)
    for active in [ALL] + [{k} for k in sorted(ALL)]:
        loss, g = Model(active).loss_and_grads(params, tokens, cfg)
        worst = sorted(parity.grad_report(g, gref), key=lambda r: -r[2])[:4]
        print(f"{'all' if active == ALL else sorted(active)[0]:5s} loss rel {abs(loss - loss_ref) / loss_ref:.2e}  " +
              "  ".join(f"{n} {r:.4f}" for n, c, r in worst), flush=True)


if __name__ == "__main__":
    main(sys.argv)
