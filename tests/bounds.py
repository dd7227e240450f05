"""Element-wise error bounds for the kernel parity tests (test code, not product).

Each bound is |gpu - oracle| <= bound, element by element, where the oracle
is FP64 on the same BF16 inputs and the bound follows from the precisions the
kernels compute and store in:

* one BF16 rounding of a value y (round to nearest even, 8 significant bits)
  moves it by at most u = 2^-8 |y| (half a unit in the last place, relative
  to the smallest value of the binade);
* an FP32 sum of n terms t_k (BF16 inputs make every product of two of them
  exact in FP32) is off by at most acc(n) * sum |t_k| with acc(n) = n 2^-23,
  the worst case of n roundings (or truncations) of 2^-23 each;
* the attention kernels exponentiate FP32 scores with the SFU's exp2 and the
  log-sum-exp carried from the forward; together with the FP32 score error
  this perturbs every probability by a relative E_S = 1e-4 at most at the
  tested scales (|score| < 40).

Every bound below is the first-order sum of those terms along the kernel's
chain of roundings, times a safety factor MARGIN = 2.  A plausible kernel
mistake (a wrong row block, a dropped causal mask, a wrong GQA head, a
missing gain) moves elements by O(|y|), far outside these bounds, while a
norm over 10^5 elements could hide it.
"""
from __future__ import annotations

import math

import torch

D = torch.float64
U = 2.0 ** -8      # BF16 unit roundoff (8 significant bits)
E_S = 1e-4         # relative error of an attention probability
MARGIN = 2.0


def acc(n):
    """Worst-case relative error of an FP32 sum of n terms (w.r.t. sum |terms|)."""
    return n * 2.0 ** -23


def check(got, ref, bound, what):
    """Assert |got - ref| <= bound element-wise; report the worst element."""
    got = got.to(D).cpu()
    ref = ref.to(D).cpu()
    bound = bound.to(D).cpu()
    err = (got - ref).abs()
    bad = err > bound
    if bool(bad.any()):
        ratio = err / bound.clamp_min(1e-300)
        i = int(ratio.reshape(-1).argmax())
        idx = [int(x) for x in torch.unravel_index(torch.tensor(i), ratio.shape)]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.numel()} elements outside the bound; worst at "
                             f"{idx}: got {float(got.reshape(-1)[i]):.6g}, oracle {float(ref.reshape(-1)[i]):.6g}, "
                             f"bound {float(bound.reshape(-1)[i]):.3g}")


# ------------------------------------------------------------------ GEMM epilogues
def gemm_err(A, B, K):
    """FP32 accumulator of A @ B^T (BF16 operands): acc(K) |A| @ |B|^T."""
    return acc(K) * (A.to(D).abs() @ B.to(D).abs().T)


def store_bf16(ref, err_in):
    """A value with input error err_in, then rounded to BF16."""
    return MARGIN * (U * ref.abs() + err_in)


# ------------------------------------------------------------------ RMSNorm
def rmsnorm_fwd(y_ref, x, g, rstd):
    """y = bf16(x * rstd * g): the FP32 sum of squares (acc(d)) moves rstd by
    acc(d)/2 relative, rsqrt adds a few 2^-23; then one BF16 rounding."""
    d = x.shape[-1]
    rel_in = acc(d) + 4 * 2.0 ** -23
    return MARGIN * (U * y_ref.abs() + rel_in * (x.to(D).abs() * rstd.to(D)[:, None] * g.to(D).abs()))


def rmsnorm_bwd(dx_ref, dg_ref, dy, x, g, rstd, dres):
    """dx = bf16(dres + r (dy g - x r m)), m = mean(dy g x r) (FP32 over d, in
    a butterfly and a warp-order sum), dg = bf16(sum over rows of dy x r)
    (FP32, per block of rows, then over the blocks).  rstd is the library's (its
    relative error, < 1e-6 as tested, enters through r and r^2)."""
    dy, x, g, r = dy.to(D), x.to(D), g.to(D), rstd.to(D)[:, None]
    rows, d = x.shape
    terms = (dy * g * x * r).abs()
    m_err = acc(d) * terms.mean(-1, keepdim=True) + 2e-6 * terms.mean(-1, keepdim=True)
    m_abs = terms.mean(-1, keepdim=True)
    res = dres.to(D).abs() if dres is not None else 0.0
    dx_in = (4 * 2.0 ** -23 + 2e-6) * (res + r * (dy * g).abs() + r * r * x.abs() * m_abs) + r * r * x.abs() * m_err
    dg_terms = (dy * x * r).abs().sum(0)
    dg_in = (acc(rows) + 2e-6) * dg_terms
    return store_bf16(dx_ref, dx_in), store_bf16(dg_ref, dg_in)


# ------------------------------------------------------------------ SwiGLU backward
def swiglu_bwd(dg_ref, du_ref, da, gate, up, da_err=None):
    """dgate = da * up * silu'(gate), dup = da * silu(gate) in FP32 from BF16
    gate/up (and da, exact or with error da_err), then BF16.  silu' = s (1 +
    gate (1 - s)) cancels near gate = -1.28: its FP32 error is a few 2^-23
    of s (1 + |gate|)."""
    da, gate, up = da.to(D), gate.to(D), up.to(D)
    s = torch.sigmoid(gate)
    dsilu_abs = s * (1 + gate.abs())
    silu = gate * s
    e = 8 * 2.0 ** -23
    in_g = e * (da * up).abs() * dsilu_abs
    in_u = e * (da * silu).abs()
    if da_err is not None:
        in_g = in_g + da_err * (up * s * (1 + gate * (1 - s))).abs()
        in_u = in_u + da_err * silu.abs()
    return store_bf16(dg_ref, in_g), store_bf16(du_ref, in_u)


# ------------------------------------------------------------------ cross-entropy
def cross_entropy_dz(dz_ref, z, tgt, inv_n):
    """dz = bf16((softmax(z) - onehot) * inv_n) with FP32 exp and log-sum-exp:
    each probability off by a few 2^-23 times (1 + |z|)."""
    z = z.to(D)
    p = torch.softmax(z, -1)
    e = 16 * 2.0 ** -23 * (1 + z.abs().amax(-1, keepdim=True))
    return store_bf16(dz_ref, e * p * inv_n)


# ------------------------------------------------------------------ embedding backward
def embedding_bwd(dE_ref, tok, dx, V):
    """dE[v] = bf16(FP32 sum of the BF16 rows of dx with token v)."""
    tok = tok.long()
    mag = torch.zeros(V, dx.shape[1], dtype=D).index_add_(0, tok, dx.to(D).abs())
    cnt = torch.bincount(tok, minlength=V).to(D)[:, None]
    return store_bf16(dE_ref, acc(1) * cnt.clamp_min(1) * mag)


# ------------------------------------------------------------------ attention
def attention_head(q, k, v, do, scale=None):
    """Bounds for one query head against its K/V head (FP64, full S x S).

    Forward: P is rounded to BF16 as the PV product's operand, so
      |do| <= U * (P @ |v|) + E_S * (P @ |v|) + acc(S) (P @ |v|), then BF16.
    Backward (delta = rowsum(dO o) uses the library's BF16 o, whose bound is
    the forward's): dS = P (dP - delta) is rounded to BF16 for both products,
      |d dS| <= U |dS| + P (|d delta| + acc(hd) |dO| |v|^T) + E_S P |dP - delta|,
      |d dq| <= scale |d dS| @ |k| + acc(S) scale |dS| @ |k|, then BF16,
      |d dk| <= scale |d dS|^T @ |q| + acc(S) scale |dS|^T @ |q| (per head),
      |d dv| <= (U + E_S + acc(S)) P^T @ |dO| (per head).
    Returns the reference pieces and the pre-rounding error terms; dk/dv are
    per-head contributions to be summed over the group, then rounded."""
    q, k, v, do = q.to(D), k.to(D), v.to(D), do.to(D)
    S, hd = q.shape
    scale = scale if scale is not None else 1.0 / math.sqrt(hd)
    s = (q @ k.T) * scale
    s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
    P = torch.softmax(s, -1)
    o = P @ v
    Pv = P @ v.abs()
    bo = MARGIN * ((U + E_S + acc(S)) * Pv + U * o.abs())
    dP = do @ v.T
    delta = (do * o).sum(-1, keepdim=True)
    dS = P * (dP - delta)
    d_delta = (do.abs() * bo).sum(-1, keepdim=True) + acc(hd) * (do * o).abs().sum(-1, keepdim=True)
    d_dS = U * dS.abs() + P * (d_delta + acc(hd) * (do.abs() @ v.abs().T)) + E_S * P * (dP - delta).abs()
    kab, qab = k.abs(), q.abs()
    dq = scale * (dS @ k)
    e_dq = scale * (d_dS @ kab) + acc(S) * scale * (dS.abs() @ kab)
    dk = scale * (dS.T @ q)
    e_dk = scale * (d_dS.T @ qab) + acc(S) * scale * (dS.abs().T @ qab)
    dv = P.T @ do
    e_dv = (U + E_S + acc(S)) * (P.T @ do.abs())
    return dict(o=o, bo=bo, dq=dq, e_dq=e_dq, bdq=MARGIN * (e_dq + U * dq.abs()), dk=dk, e_dk=e_dk, dv=dv, e_dv=e_dv)


def attention_row(q, k, v, do, i, scale=None):
    """The same bounds for one query row i of a long sequence (keys 0..i)."""
    q, k, v, do = q.to(D), k.to(D), v.to(D), do.to(D)
    hd = q.shape[1]
    scale = scale if scale is not None else 1.0 / math.sqrt(hd)
    kk, vv = k[:i + 1], v[:i + 1]
    p = torch.softmax((kk @ q[i]) * scale, -1)
    o = p @ vv
    Pv = p @ vv.abs()
    bo = MARGIN * ((U + E_S + acc(i + 1)) * Pv + U * o.abs())
    dP = vv @ do[i]
    delta = float(do[i] @ o)
    dS = p * (dP - delta)
    d_delta = float(do[i].abs() @ bo) + acc(hd) * float((do[i] * o).abs().sum())
    d_dS = U * dS.abs() + p * (d_delta + acc(hd) * (vv.abs() @ do[i].abs())) + E_S * p * (dP - delta).abs()
    dq = scale * (dS @ kk)
    e_dq = scale * (d_dS @ kk.abs()) + acc(i + 1) * scale * (dS.abs() @ kk.abs())
    return bo, MARGIN * (e_dq + U * dq.abs())


def attention_key(qs, k, v, dos, j, scale=None):
    """Bounds on dk_j and dv_j (summed over the query heads qs [G, S, hd] that
    share this K/V head) from every query i >= j."""
    qs, k, v, dos = qs.to(D), k.to(D), v.to(D), dos.to(D)
    G, S, hd = qs.shape
    scale = scale if scale is not None else 1.0 / math.sqrt(hd)
    e_dk = torch.zeros(hd, dtype=D)
    e_dv = torch.zeros(hd, dtype=D)
    dk = torch.zeros(hd, dtype=D)
    dv = torch.zeros(hd, dtype=D)
    causal = torch.ones(S - j, S, dtype=torch.bool)
    causal = causal.triu(j + 1)  # row r (query j + r) sees keys <= j + r
    for h in range(G):
        q, do = qs[h, j:], dos[h, j:]
        s = (q @ k.T) * scale
        s = s.masked_fill(causal, float("-inf"))
        P = torch.softmax(s, -1)
        o = P @ v
        Pv = P @ v.abs()
        bo = MARGIN * ((U + E_S + acc(S)) * Pv + U * o.abs())
        pj = P[:, j]
        dPj = do @ v[j]
        delta = (do * o).sum(-1)
        dSj = pj * (dPj - delta)
        d_delta = (do.abs() * bo).sum(-1) + acc(hd) * (do * o).abs().sum(-1)
        d_dSj = U * dSj.abs() + pj * (d_delta + acc(hd) * (do.abs() @ v[j].abs())) + E_S * pj * (dPj - delta).abs()
        dk += scale * (dSj @ q)
        e_dk += scale * (d_dSj @ q.abs()) + acc(S * G) * scale * (dSj.abs() @ q.abs())
        dv += pj @ do
        e_dv += (U + E_S + acc(S * G)) * (pj @ do.abs())
    return MARGIN * (e_dk + U * dk.abs()), MARGIN * (e_dv + U * dv.abs())
