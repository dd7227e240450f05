"""Each sm_103a kernel through the C-ABI (include/mt_ops.h) against the CPU
oracle's function for the same step (FP64) on the same seeded BF16 inputs."""
import math

import pytest
import torch

import oracle
from tests import bounds

pytestmark = pytest.mark.gpu

hms = pytest.importorskip("host_memory_streamed_gb300")
from host_memory_streamed_gb300 import _lib, ops  # noqa: E402

D = torch.float64
DEV = "cuda"


def rel(a, b):
    a = a.to(D).cpu()
    b = b.to(D).cpu()
    return float((a - b).norm() / b.norm().clamp_min(1e-300))


def rnd(shape, gen, scale=1.0):
    return (torch.randn(shape, generator=gen) * scale).to(torch.bfloat16)


def rope_tables(S, hd, theta=1e4):
    c, s = oracle.rope_cos_sin(S, hd, theta)
    return c.float().to(DEV).contiguous(), s.float().to(DEV).contiguous()


# ------------------------------------------------------------------ GEMM
GEMM_SHAPES = [(128, 256, 64), (300, 688, 256), (129, 264, 72), (1, 8, 8), (513, 1032, 1376), (2048, 1536, 512)]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_gemm_store_and_fp32(M, N, K):
    g = torch.Generator().manual_seed(M * 7 + N)
    A, B = rnd((M, K), g), rnd((N, K), g)
    ref = A.to(D) @ B.to(D).T
    C32 = torch.empty(M, N, device=DEV)
    ops.gemm(A.to(DEV), B.to(DEV), C32, _lib.EPI_F32)
    Cb = torch.empty(M, N, device=DEV, dtype=torch.bfloat16)
    ops.gemm(A.to(DEV), B.to(DEV), Cb, _lib.EPI_STORE_BF16)
    torch.cuda.synchronize()
    # FP32 accumulation of K exact BF16 products: error ~ sqrt(K) * 2^-24 * |terms|
    bound = 1e-5 * math.sqrt(K) * (A.to(D).abs() @ B.to(D).abs().T) + 1e-30
    assert torch.all((C32.cpu().to(D) - ref).abs() <= bound)
    assert torch.equal(Cb.cpu(), C32.cpu().to(torch.bfloat16))  # BF16 output = RNE of the FP32 accumulator


def test_gemm_residual_accumulate_swiglu_rope():
    g = torch.Generator().manual_seed(3)
    M, N, K, S, hd = 384, 512, 256, 96, 128
    A, B, R = rnd((M, K), g), rnd((N, K), g), rnd((M, N), g)
    Ad, Bd = A.to(DEV), B.to(DEV)
    ref = A.to(D) @ B.to(D).T
    err = bounds.gemm_err(A, B, K)  # the FP32 accumulator's error, element-wise
    out = torch.empty(M, N, device=DEV, dtype=torch.bfloat16)
    ops.gemm(Ad, Bd, out, _lib.EPI_RESIDUAL_BF16, residual=R.to(DEV))
    assert rel(out, ref + R.to(D)) < 4e-3
    bounds.check(out, ref + R.to(D), bounds.store_bf16(ref + R.to(D), err), "residual epilogue")
    acc = torch.full((M, N), 0.5, device=DEV)
    ops.gemm(Ad, Bd, acc, _lib.EPI_F32_ACCUMULATE)
    assert rel(acc, ref + 0.5) < 1e-6
    bounds.check(acc, ref + 0.5, bounds.MARGIN * (err + 2.0 ** -23 * (ref + 0.5).abs()), "FP32 += epilogue")
    a = torch.empty(M, N // 2, device=DEV, dtype=torch.bfloat16)
    gu = torch.empty(M, N, device=DEV, dtype=torch.bfloat16)
    ops.gemm(Ad, Bd, a, _lib.EPI_SWIGLU, out2=gu)
    a_ref = oracle.swiglu(ref[:, 0::2], ref[:, 1::2])
    assert rel(a, a_ref) < 4e-3
    assert rel(gu, ref) < 4e-3
    gt, up = ref[:, 0::2], ref[:, 1::2]
    sg = torch.sigmoid(gt)
    a_in = (sg * (1 + gt * (1 - sg))).abs() * up.abs() * err[:, 0::2] + (gt * sg).abs() * err[:, 1::2] + \
        8 * 2.0 ** -23 * a_ref.abs()
    bounds.check(a, a_ref, bounds.store_bf16(a_ref, a_in), "SwiGLU epilogue")
    bounds.check(gu, ref, bounds.store_bf16(ref, err), "SwiGLU epilogue's stored gate/up")
    cos, sin = rope_tables(S, hd)
    ro = torch.empty(M, N, device=DEV, dtype=torch.bfloat16)
    ops.gemm(Ad, Bd, ro, _lib.EPI_ROPE, rope_cos=cos, rope_sin=sin, rope_cols=3 * hd, head_dim=hd, seq=S)
    torch.cuda.synchronize()
    c64, s64 = oracle.rope_cos_sin(S, hd, 1e4)
    B_, S_ = M // S, S
    x = ref[:, :3 * hd].reshape(B_, S_, 3, hd)
    expect = torch.cat([oracle.rope(x, c64, s64).reshape(M, 3 * hd), ref[:, 3 * hd:]], 1)
    assert rel(ro, expect) < 4e-3
    # rotated columns: |cos| e_1 + |sin| e_2 from the accumulator, a few FP32
    # roundings of the products (and of the FP32 tables), then BF16
    h = hd // 2
    e = err[:, :3 * hd].reshape(B_, S_, 3, hd)
    xa = x.abs()
    ca, sa = c64.abs()[None, :, None, :], s64.abs()[None, :, None, :]
    e_rot = torch.cat([ca * e[..., :h] + sa * e[..., h:], ca * e[..., h:] + sa * e[..., :h]], -1) + \
        8 * 2.0 ** -23 * torch.cat([ca * xa[..., :h] + sa * xa[..., h:], ca * xa[..., h:] + sa * xa[..., :h]], -1)
    e_all = torch.cat([e_rot.reshape(M, 3 * hd), err[:, 3 * hd:]], 1)
    bounds.check(ro, expect, bounds.store_bf16(expect, e_all), "RoPE epilogue")


@pytest.mark.parametrize("M,N,K", [(300, 344, 256), (256, 688, 512), (33, 40, 64)])
def test_gemm_swiglu_backward_epilogue(M, N, K):
    """da = dY W (FP32 accumulator) and, in the same epilogue, the SwiGLU
    backward against the stored (gate, up) pairs."""
    g = torch.Generator().manual_seed(M + N + K)
    dY, W = rnd((M, K), g), rnd((N, K), g, 0.1)
    gu = rnd((M, 2 * N), g, 2.0)
    dgu = torch.empty(M, 2 * N, device=DEV, dtype=torch.bfloat16)
    ops.gemm(dY.to(DEV), W.to(DEV), dgu, _lib.EPI_SWIGLU_BWD, residual=gu.to(DEV))
    torch.cuda.synchronize()
    da = dY.to(D) @ W.to(D).T
    dg, du = oracle.swiglu_backward(da, gu.to(D)[:, 0::2], gu.to(D)[:, 1::2])
    assert rel(dgu.cpu()[:, 0::2], dg) < 4e-3
    assert rel(dgu.cpu()[:, 1::2], du) < 4e-3
    bg, bu = bounds.swiglu_bwd(dg, du, da, gu[:, 0::2], gu[:, 1::2], da_err=bounds.gemm_err(dY, W, K))
    bounds.check(dgu.cpu()[:, 0::2], dg, bg, "SwiGLU-backward epilogue dgate")
    bounds.check(dgu.cpu()[:, 1::2], du, bu, "SwiGLU-backward epilogue dup")


# Both kernels (single CTA for M <= 128, CTA pairs with 256 x 256 tiles above)
# in all four operand layouts, with ragged M, N and K tails and partial tiles
# (MN-major operands need M resp. N to be a multiple of 8).
LAYOUT_SHAPES = [(128, 264, 72), (120, 136, 64), (296, 520, 200), (256, 256, 64), (1000, 776, 1032),
                 (2304, 2048, 512)]


@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (True, False), (False, True), (True, True)])
@pytest.mark.parametrize("M,N,K", LAYOUT_SHAPES)
def test_gemm_operand_layouts(M, N, K, a_mn, b_mn):
    g = torch.Generator().manual_seed(M + 3 * N + 7 * K + 2 * a_mn + b_mn)
    A, B = rnd((M, K), g), rnd((N, K), g)
    ref = A.to(D) @ B.to(D).T
    Ad = (A.T.contiguous() if a_mn else A).to(DEV)
    Bd = (B.T.contiguous() if b_mn else B).to(DEV)
    C32 = torch.empty(M, N, device=DEV)
    ops.gemm_layout(Ad, Bd, C32, a_mn=a_mn, b_mn=b_mn, epilogue=_lib.EPI_F32)
    acc = torch.full((M, N), 0.25, device=DEV)
    ops.gemm_layout(Ad, Bd, acc, a_mn=a_mn, b_mn=b_mn, epilogue=_lib.EPI_F32_ACCUMULATE)
    status = torch.zeros(1, device=DEV, dtype=torch.int32)
    Cb = torch.empty(M, N, device=DEV, dtype=torch.bfloat16)
    ops.gemm_layout(Ad, Bd, Cb, a_mn=a_mn, b_mn=b_mn, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    bound = 1e-5 * math.sqrt(K) * (A.to(D).abs() @ B.to(D).abs().T) + 1e-30
    assert torch.all((C32.cpu().to(D) - ref).abs() <= bound)
    assert torch.all((acc.cpu().to(D) - (ref + 0.25)).abs() <= bound + 1e-7)
    assert torch.equal(Cb.cpu(), C32.cpu().to(torch.bfloat16))


def test_gemm_rejects_bad_arguments():
    A = torch.zeros(16, 12, device=DEV, dtype=torch.bfloat16)
    C = torch.zeros(16, 16, device=DEV, dtype=torch.bfloat16)
    with pytest.raises(RuntimeError, match="multiple of 8"):
        ops.gemm(A, A[:, :12], C)


def test_gemm_deterministic():
    g = torch.Generator().manual_seed(5)
    A, B = rnd((1000, 2048), g).to(DEV), rnd((3000, 2048), g).to(DEV)
    c1 = torch.empty(1000, 3000, device=DEV)
    c2 = torch.empty(1000, 3000, device=DEV)
    ops.gemm(A, B, c1, _lib.EPI_F32)
    ops.gemm(A, B, c2, _lib.EPI_F32)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)


# ------------------------------------------------------------------ attention
# S % 4 == 0 brings whole query blocks' lse/delta by bulk copy in the dK/dV
# kernel and stages ragged ones by thread: 512 (all whole, GQA 4), 452 and 200
# (whole blocks, then a ragged one), 333 / 257 / 1 (all staged).  The
# backward kernels start their CTAs in chunks of 256 / (query blocks) rows of
# the grid, the forward in chunks of 128 / (query blocks): 180 query heads and
# 90 kv-head rows over three query blocks (chunks of 85 and 42 rows) leave a
# short last chunk in every kernel.
ATTN = [(2, 128, 4, 4, 64), (1, 200, 4, 2, 128), (2, 333, 6, 2, 64), (1, 1, 2, 1, 128), (1, 257, 10, 2, 128),
        (1, 64, 8, 1, 64), (2, 512, 8, 2, 128), (1, 452, 4, 1, 128), (2, 300, 90, 45, 64)]


def _attn_inputs(B, S, Hq, Hkv, hd, seed):
    g = torch.Generator().manual_seed(seed)
    ld = (Hq + 2 * Hkv) * hd
    qkv = rnd((B * S, ld), g)
    do = rnd((B * S, Hq * hd), g)
    return qkv, do


@pytest.mark.parametrize("B,S,Hq,Hkv,hd", ATTN)
def test_attention_forward_backward_vs_oracle(B, S, Hq, Hkv, hd):
    qkv, do = _attn_inputs(B, S, Hq, Hkv, hd, seed=B * 1000 + S + Hq)
    T, ld = B * S, qkv.shape[1]
    qd = qkv.to(DEV)
    o = torch.empty(T, Hq * hd, device=DEV, dtype=torch.bfloat16)
    lse = torch.empty(B * Hq * S, device=DEV)
    ops.attention_fwd(qd, B, S, Hq, Hkv, hd, o, lse)
    delta = torch.empty(B * Hq * S, device=DEV)
    dqkv = torch.zeros(T, ld, device=DEV, dtype=torch.bfloat16)
    ops.attention_bwd(qd, B, S, Hq, Hkv, hd, o, lse, do.to(DEV), delta, dqkv)
    torch.cuda.synchronize()
    x = qkv.to(D)
    q = x[:, :Hq * hd].reshape(B, S, Hq, hd)
    k = x[:, Hq * hd:(Hq + Hkv) * hd].reshape(B, S, Hkv, hd)
    v = x[:, (Hq + Hkv) * hd:].reshape(B, S, Hkv, hd)
    o_ref, probs = oracle.causal_gqa_attention(q, k, v)
    assert rel(o, o_ref.reshape(T, -1)) < 5e-3
    # log-sum-exp of each score row, from the oracle's scores
    scale = 1 / math.sqrt(hd)
    lse_ref = torch.empty(B, Hq, S, dtype=D)
    for b in range(B):
        for h in range(Hq):
            j = h * Hkv // Hq
            sc = (q[b, :, h] @ k[b, :, j].T) * scale
            sc = sc.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
            lse_ref[b, h] = torch.logsumexp(sc, -1)
    assert (lse.cpu().to(D) - lse_ref.reshape(-1)).abs().max() < 1e-4
    dq, dk, dv = oracle.causal_gqa_attention_backward(do.to(D).reshape(B, S, Hq, hd), q, k, v, probs)
    got = dqkv.cpu().to(D)
    for name, a, b_ in (("dq", got[:, :Hq * hd], dq), ("dk", got[:, Hq * hd:(Hq + Hkv) * hd], dk),
                        ("dv", got[:, (Hq + Hkv) * hd:], dv)):
        b_ = b_.reshape(T, -1)
        if float(b_.norm()) < 1e-12:  # S = 1: the softmax is constant, dq = dk = 0 exactly
            assert float(a.abs().max()) < 1e-2 * float(do.to(D).abs().max()), name
        else:
            assert rel(a, b_) < 1e-2, (name, rel(a, b_))
    # element-wise: every output, query head and key head against its bound
    _attention_elementwise(o.cpu().to(D), got, q, k, v, do.to(D).reshape(B, S, Hq, hd), o_ref, dq, dk, dv)


def _attention_elementwise(o, got, q, k, v, do, o_ref, dq, dk, dv, rope=None):
    """|gpu - oracle| <= bound for o, dq, dk, dv, element by element (bounds
    from tests/bounds.py: BF16 P and dS operands, FP32 sums, BF16 outputs).
    rope = (cos, sin): the backward's outputs are the inverse-rotated grads."""
    B, S, Hq, hd = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    T = B * S
    bo = torch.empty(B, S, Hq, hd, dtype=D)
    e_dq = torch.empty(B, S, Hq, hd, dtype=D)
    e_dk = torch.zeros(B, S, Hkv, hd, dtype=D)
    e_dv = torch.zeros(B, S, Hkv, hd, dtype=D)
    for b in range(B):
        for h in range(Hq):
            j = h // G
            r = bounds.attention_head(q[b, :, h], k[b, :, j], v[b, :, j], do[b, :, h])
            bo[b, :, h] = r["bo"]
            e_dq[b, :, h] = r["e_dq"]
            e_dk[b, :, j] += r["e_dk"]
            e_dv[b, :, j] += r["e_dv"]
    bounds.check(o, o_ref.reshape(T, -1), bo.reshape(T, -1), "attention o")
    dq, dk, dv = dq.reshape(B, S, Hq, hd), dk.reshape(B, S, Hkv, hd), dv.reshape(B, S, Hkv, hd)
    if rope is not None:
        c, s_ = rope
        h2 = hd // 2
        ca, sa = c.abs()[None, :, None, :], s_.abs()[None, :, None, :]

        def rot_err(e, x):
            xa = x.abs()
            return torch.cat([ca * e[..., :h2] + sa * e[..., h2:], ca * e[..., h2:] + sa * e[..., :h2]], -1) + \
                8 * 2.0 ** -23 * torch.cat([ca * xa[..., :h2] + sa * xa[..., h2:],
                                            ca * xa[..., h2:] + sa * xa[..., :h2]], -1)
        e_dq, e_dk = rot_err(e_dq, dq), rot_err(e_dk, dk)
        dq, dk = oracle.rope_backward(dq, c, s_), oracle.rope_backward(dk, c, s_)
    for name, a, ref, e in (("dq", got[:, :Hq * hd], dq, e_dq), ("dk", got[:, Hq * hd:(Hq + Hkv) * hd], dk, e_dk),
                            ("dv", got[:, (Hq + Hkv) * hd:], dv, e_dv)):
        ref = ref.reshape(T, -1)
        bounds.check(a, ref, bounds.MARGIN * (e.reshape(T, -1) + bounds.U * ref.abs()), f"attention {name}")


def test_attention_backward_with_rope_gives_unrotated_grads():
    B, S, Hq, Hkv, hd = 2, 150, 4, 2, 128
    qkv, do = _attn_inputs(B, S, Hq, Hkv, hd, seed=11)
    T, ld = B * S, qkv.shape[1]
    cos, sin = rope_tables(S, hd)
    qd = qkv.to(DEV)
    o = torch.empty(T, Hq * hd, device=DEV, dtype=torch.bfloat16)
    lse = torch.empty(B * Hq * S, device=DEV)
    ops.attention_fwd(qd, B, S, Hq, Hkv, hd, o, lse)
    dqkv = torch.zeros(T, ld, device=DEV, dtype=torch.bfloat16)
    ops.attention_bwd(qd, B, S, Hq, Hkv, hd, o, lse, do.to(DEV), torch.empty(B * Hq * S, device=DEV), dqkv,
                      cos, sin)
    torch.cuda.synchronize()
    x = qkv.to(D)
    q = x[:, :Hq * hd].reshape(B, S, Hq, hd)
    k = x[:, Hq * hd:(Hq + Hkv) * hd].reshape(B, S, Hkv, hd)
    v = x[:, (Hq + Hkv) * hd:].reshape(B, S, Hkv, hd)
    _, probs = oracle.causal_gqa_attention(q, k, v)
    dq, dk, _ = oracle.causal_gqa_attention_backward(do.to(D).reshape(B, S, Hq, hd), q, k, v, probs)
    c64, s64 = oracle.rope_cos_sin(S, hd, 1e4)
    got = dqkv.cpu().to(D)
    assert rel(got[:, :Hq * hd], oracle.rope_backward(dq, c64, s64).reshape(T, -1)) < 1e-2
    assert rel(got[:, Hq * hd:(Hq + Hkv) * hd], oracle.rope_backward(dk, c64, s64).reshape(T, -1)) < 1e-2
    o_ref, _ = oracle.causal_gqa_attention(q, k, v)
    _, _, dv = oracle.causal_gqa_attention_backward(do.to(D).reshape(B, S, Hq, hd), q, k, v, probs)
    _attention_elementwise(o.cpu().to(D), got, q, k, v, do.to(D).reshape(B, S, Hq, hd), o_ref, dq, dk, dv,
                           rope=(c64, s64))


def test_attention_backward_deterministic():
    B, S, Hq, Hkv, hd = 1, 700, 10, 2, 128
    qkv, do = _attn_inputs(B, S, Hq, Hkv, hd, seed=12)
    T, ld = B * S, qkv.shape[1]
    qd, dod = qkv.to(DEV), do.to(DEV)
    o = torch.empty(T, Hq * hd, device=DEV, dtype=torch.bfloat16)
    lse = torch.empty(B * Hq * S, device=DEV)
    ops.attention_fwd(qd, B, S, Hq, Hkv, hd, o, lse)
    outs = []
    for _ in range(2):
        d = torch.zeros(T, ld, device=DEV, dtype=torch.bfloat16)
        ops.attention_bwd(qd, B, S, Hq, Hkv, hd, o, lse, dod, torch.empty(B * Hq * S, device=DEV), d)
        outs.append(d)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])


# ------------------------------------------------------------------ RMSNorm / SwiGLU / CE / embedding / transpose
@pytest.mark.parametrize("rows,d", [(256, 256), (1000, 5120), (77, 64), (130, 8192)])
def test_rmsnorm_vs_oracle(rows, d):
    g = torch.Generator().manual_seed(rows + d)
    x, w = rnd((rows, d), g), (1 + 0.1 * torch.randn(d, generator=g)).to(torch.bfloat16)
    dy, dres = rnd((rows, d), g), rnd((rows, d), g)
    y = torch.empty(rows, d, device=DEV, dtype=torch.bfloat16)
    rstd = torch.empty(rows, device=DEV)
    ops.rmsnorm_fwd(x.to(DEV), w.to(DEV), y, rstd, 1e-5)
    dx = torch.empty_like(y)
    dg = torch.empty(d, device=DEV, dtype=torch.bfloat16)
    ops.rmsnorm_bwd(dy.to(DEV), x.to(DEV), w.to(DEV), rstd, dres.to(DEV), dx, dg)
    torch.cuda.synchronize()
    yr, rr = oracle.rms_norm(x.to(D), w.to(D), 1e-5)
    dxr, dgr = oracle.rms_norm_backward(dy.to(D), x.to(D), w.to(D), rr)
    assert rel(y, yr) < 4e-3
    assert rel(rstd, rr.reshape(-1)) < 1e-6
    assert rel(dx, dxr + dres.to(D)) < 4e-3
    assert rel(dg, dgr) < 4e-3
    assert float(((rstd.cpu().to(D) - rr.reshape(-1)) / rr.reshape(-1)).abs().max()) < 1e-6
    bounds.check(y, yr, bounds.rmsnorm_fwd(yr, x, w, rstd.cpu()), "rmsnorm y")
    bdx, bdg = bounds.rmsnorm_bwd(dxr + dres.to(D), dgr, dy, x, w, rstd.cpu(), dres)
    bounds.check(dx, dxr + dres.to(D), bdx, "rmsnorm dx")
    bounds.check(dg, dgr, bdg, "rmsnorm dg")


@pytest.mark.parametrize("rows,f", [(256, 688), (300, 5632), (5, 7)])
def test_swiglu_backward_vs_oracle(rows, f):
    g = torch.Generator().manual_seed(rows + f)
    gu, da = rnd((rows, 2 * f), g, 2.0), rnd((rows, f), g)
    dgu = torch.empty(rows, 2 * f, device=DEV, dtype=torch.bfloat16)
    ops.swiglu_bwd(da.to(DEV), gu.to(DEV), dgu)
    torch.cuda.synchronize()
    dg, du = oracle.swiglu_backward(da.to(D), gu.to(D)[:, 0::2], gu.to(D)[:, 1::2])
    assert rel(dgu.cpu()[:, 0::2], dg) < 4e-3
    assert rel(dgu.cpu()[:, 1::2], du) < 4e-3
    bg, bu = bounds.swiglu_bwd(dg, du, da, gu[:, 0::2], gu[:, 1::2])
    bounds.check(dgu.cpu()[:, 0::2], dg, bg, "swiglu backward dgate")
    bounds.check(dgu.cpu()[:, 1::2], du, bu, "swiglu backward dup")


@pytest.mark.parametrize("rows,V", [(256, 1024), (64, 152064), (10, 40)])
def test_cross_entropy_vs_oracle(rows, V):
    g = torch.Generator().manual_seed(rows + V)
    z = torch.randn(rows, V, generator=g) * 3
    y = torch.randint(0, V, (rows,), generator=g, dtype=torch.int32)
    dz = torch.empty(rows, V, device=DEV, dtype=torch.bfloat16)
    lr = torch.empty(rows, device=DEV)
    st = torch.zeros(1, device=DEV, dtype=torch.int32)
    ops.cross_entropy(z.to(DEV), y.to(DEV), 1.0 / rows, dz, lr, st)
    torch.cuda.synchronize()
    zd = z.to(D)
    lref = torch.logsumexp(zd, -1) - zd.gather(1, y.long()[:, None])[:, 0]
    assert (lr.cpu().to(D) - lref).abs().max() < 1e-5 * max(1.0, float(lref.abs().max()))
    p = torch.softmax(zd, -1)
    p[torch.arange(rows), y.long()] -= 1
    assert rel(dz, p / rows) < 4e-3
    bounds.check(dz, p / rows, bounds.cross_entropy_dz(p / rows, z, y, 1.0 / rows), "cross-entropy dz")
    assert int(st.item()) == 0


def test_embedding_forward_exact_backward_deterministic_sum():
    g = torch.Generator().manual_seed(21)
    V, d, T = 1000, 256, 512
    E = rnd((V, d), g)
    tok = torch.randint(0, V, (T,), generator=g, dtype=torch.int32)
    x = torch.empty(T, d, device=DEV, dtype=torch.bfloat16)
    st = torch.zeros(1, device=DEV, dtype=torch.int32)
    ops.embedding_fwd(tok.to(DEV), E.to(DEV), x, st)
    dx = rnd((T, d), g)
    order = torch.argsort(tok.long() * T + torch.arange(T))
    off = torch.zeros(V + 1, dtype=torch.int32)
    off[1:] = torch.cumsum(torch.bincount(tok.long(), minlength=V), 0).int()
    dE = torch.empty(V, d, device=DEV, dtype=torch.bfloat16)
    ops.embedding_bwd(off.to(DEV), order.int().to(DEV), dx.to(DEV), dE)
    torch.cuda.synchronize()
    assert torch.equal(x.cpu(), E[tok.long()])
    ref = torch.zeros(V, d, dtype=D).index_add_(0, tok.long(), dx.to(D))
    assert rel(dE, ref) < 4e-3
    bounds.check(dE, ref, bounds.embedding_bwd(ref, tok, dx, V), "embedding backward")
    assert torch.all(dE.cpu()[torch.bincount(tok.long(), minlength=V) == 0] == 0)
    bad = tok.clone()
    bad[3] = V + 5
    ops.embedding_fwd(bad.to(DEV), E.to(DEV), x, st)
    torch.cuda.synchronize()
    assert int(st.item()) != 0


@pytest.mark.parametrize("r,c", [(100, 70), (4096, 5120), (64, 64), (1, 9), (130, 257)])
def test_transpose_exact(r, c):
    g = torch.Generator().manual_seed(r + c)
    x = rnd((r, c), g).to(DEV)
    y = torch.empty(c, r, device=DEV, dtype=torch.bfloat16)
    ops.transpose(x, y)
    torch.cuda.synchronize()
    assert torch.equal(y, x.T)


def _attention_vs_oracle(qkv, B, S, Hq, Hkv, hd):
    T = B * S
    qd = qkv.to(DEV)
    o = torch.empty(T, Hq * hd, device=DEV, dtype=torch.bfloat16)
    lse = torch.empty(B * Hq * S, device=DEV)
    st = torch.zeros(1, device=DEV, dtype=torch.int32)
    ops.attention_fwd(qd, B, S, Hq, Hkv, hd, o, lse, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    x = qkv.to(D)
    q = x[:, :Hq * hd].reshape(B, S, Hq, hd)
    k = x[:, Hq * hd:(Hq + Hkv) * hd].reshape(B, S, Hkv, hd)
    v = x[:, (Hq + Hkv) * hd:].reshape(B, S, Hkv, hd)
    o_ref, _ = oracle.causal_gqa_attention(q, k, v)
    return rel(o, o_ref.reshape(T, -1))


def test_attention_rescale_in_part_of_a_warp():
    """Half of one warp's query rows meet a key, in a later key block, whose
    score exceeds their running maximum by far more than 2^8, the other half
    do not: the running-maximum rescale then happens for some lanes of a warp
    only, which the kernel must handle as one warp."""
    B, S, Hq, Hkv, hd = 1, 512, 2, 1, 128
    g = torch.Generator().manual_seed(31)
    qkv = torch.randn(B * S, (Hq + 2 * Hkv) * hd, generator=g) * 0.5
    u = torch.randn(hd, generator=g)
    u = u / u.norm()
    for r in range(400, 416):  # query rows in key block 3, lanes 16..31 of the warp owning rows 384..415
        qkv[r, :hd] = 4.0 * u
    qkv[300, Hq * hd:(Hq + 1) * hd] = 4.0 * u  # key 300 (block 2) aligns with them: score 16/sqrt(128) * ... >> 2^8 in exp
    qkv[300, Hq * hd:(Hq + 1) * hd] *= 8.0
    assert _attention_vs_oracle(qkv.to(torch.bfloat16), B, S, Hq, Hkv, hd) < 5e-3


def test_attention_long_sequence_step_scale():
    """Activations at the scale the decoder produces (std ~1.4) over 16 key blocks."""
    B, S, Hq, Hkv, hd = 1, 2048, 4, 2, 128
    g = torch.Generator().manual_seed(32)
    qkv = (torch.randn(B * S, (Hq + 2 * Hkv) * hd, generator=g) * 1.4).to(torch.bfloat16)
    assert _attention_vs_oracle(qkv, B, S, Hq, Hkv, hd) < 5e-3


@pytest.mark.parametrize("n", [8, 4096, 1 << 20, 1000003])
def test_flag_nonfinite(n):
    """The device non-finite check: clean data leaves the flag at 0; one NaN,
    +Inf or -Inf anywhere (first, middle, in the ragged tail, last) sets it."""
    L = _lib.lib()
    g = torch.Generator().manual_seed(n)
    x = rnd((n,), g).to(DEV)
    flag = torch.zeros(1, device=DEV, dtype=torch.int32)
    assert L.mt_op_flag_nonfinite(x.data_ptr(), n, flag.data_ptr(), None) == 0
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    for pos in sorted({0, n // 2, n - 1, (n // 8) * 8 if n % 8 else n - 1}):
        for bad in (float("nan"), float("inf"), float("-inf")):
            y = x.clone()
            y[pos] = bad
            flag.zero_()
            assert L.mt_op_flag_nonfinite(y.data_ptr(), n, flag.data_ptr(), None) == 0
            torch.cuda.synchronize()
            assert int(flag.item()) == 1, (pos, bad)
