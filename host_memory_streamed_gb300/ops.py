"""Per-kernel entry points (include/mt_ops.h) on torch CUDA tensors.

Argument marshalling only: each call checks dtypes/devices, passes raw device
pointers and the current CUDA stream to libmt.so and returns.
"""
from __future__ import annotations

import torch

from . import _lib


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _chk(rc):
    if rc != 0:
        raise RuntimeError(_lib.lib().mt_op_last_error().decode())


def _need(t, dtype, name):
    if t is None:
        return
    if not t.is_cuda or t.dtype != dtype:
        raise TypeError(f"{name} must be a CUDA {dtype} tensor")


F32, BF16, I32 = torch.float32, torch.bfloat16, torch.int32


def gemm(A, B, out, epilogue=_lib.EPI_STORE_BF16, residual=None, out2=None, rope_cos=None, rope_sin=None,
         rope_cols=0, head_dim=0, seq=1, status=None):
    """out = epilogue(A @ B^T); A [M, K], B [N, K] BF16 (row strides may exceed K)."""
    _need(A, BF16, "A")
    _need(B, BF16, "B")
    _need(out, F32 if epilogue in (_lib.EPI_F32, _lib.EPI_F32_ACCUMULATE) else BF16, "out")
    _need(residual, BF16, "residual")
    _need(out2, BF16, "out2")
    _need(rope_cos, F32, "rope_cos")
    _need(rope_sin, F32, "rope_sin")
    _need(status, I32, "status")
    M, K = A.shape
    N = B.shape[0]
    _chk(_lib.lib().mt_op_gemm(A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), M, N, K, epilogue,
                               out.data_ptr(), out.stride(0), _ptr(residual),
                               residual.stride(0) if residual is not None else 0, _ptr(out2),
                               out2.stride(0) if out2 is not None else 0, _ptr(rope_cos), _ptr(rope_sin),
                               rope_cols, head_dim, seq, _ptr(status), _stream()))


def gemm_layout(A, B, out, a_mn=False, b_mn=False, epilogue=_lib.EPI_STORE_BF16, residual=None, status=None):
    """out = epilogue(op(A) @ op(B)^T) with A stored [M, K] (or [K, M] when a_mn)
    and B stored [N, K] (or [K, N] when b_mn): the weight-gradient and
    data-gradient layouts of the backward pass."""
    _need(A, BF16, "A")
    _need(B, BF16, "B")
    _need(out, F32 if epilogue in (_lib.EPI_F32, _lib.EPI_F32_ACCUMULATE) else BF16, "out")
    _need(residual, BF16, "residual")
    _need(status, I32, "status")
    M, K = (A.shape[1], A.shape[0]) if a_mn else (A.shape[0], A.shape[1])
    N = B.shape[1] if b_mn else B.shape[0]
    layout = (_lib.GEMM_A_MN if a_mn else 0) | (_lib.GEMM_B_MN if b_mn else 0)
    _chk(_lib.lib().mt_op_gemm_layout(A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), M, N, K, layout,
                                      epilogue, out.data_ptr(), out.stride(0), _ptr(residual),
                                      residual.stride(0) if residual is not None else 0, _ptr(status), _stream()))


def wait_probe(status, limit_ns):
    """Launch the failure-detection probe: a bounded wait that must run out
    and record MT_STATUS_WAIT_PROBE in ``status`` (device int32)."""
    _need(status, I32, "status")
    _chk(_lib.lib().mt_op_wait_probe(status.data_ptr(), int(limit_ns), _stream()))


def gemm_grouped_rows(A, B, offsets, out, b_mn=False, epilogue=_lib.EPI_STORE_BF16, residual=None, out2=None,
                      status=None):
    """One launch, per group g: out[r] = epilogue(A[r] @ B[g]^T) for the rows r
    in offsets[g] .. offsets[g+1] (device int32 [G + 1]).  A [R, K]; B [G, N, K]
    (or [G, K, N] when b_mn); out has A's rows (SwiGLU: N/2 columns, SwiGLU
    backward: 2N columns against residual = the gate/up pairs)."""
    _need(A, BF16, "A")
    _need(B, BF16, "B")
    _need(offsets, I32, "offsets")
    _need(out, F32 if epilogue in (_lib.EPI_F32, _lib.EPI_F32_ACCUMULATE) else BF16, "out")
    _need(residual, BF16, "residual")
    _need(out2, BF16, "out2")
    _need(status, I32, "status")
    G = B.shape[0]
    K, N = (B.shape[1], B.shape[2]) if b_mn else (B.shape[2], B.shape[1])
    if B.stride(0) != B.shape[1] * B.stride(1) or offsets.numel() != G + 1:
        raise ValueError("gemm_grouped_rows: B must stack its groups contiguously, offsets must have G + 1 entries")
    _chk(_lib.lib().mt_op_gemm_grouped(A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(1), A.shape[0], N, K,
                                       _lib.GEMM_B_MN if b_mn else 0, _lib.GEMM_GROUP_ROWS, offsets.data_ptr(), G,
                                       epilogue, out.data_ptr(), out.stride(0), _ptr(residual),
                                       residual.stride(0) if residual is not None else 0, _ptr(out2),
                                       out2.stride(0) if out2 is not None else 0, _ptr(status), _stream()))


def gemm_grouped_k(A, B, offsets, out, epilogue=_lib.EPI_STORE_BF16, status=None):
    """One launch, per group g: out[g] = A[rows]^T @ B[rows] over the rows
    offsets[g] .. offsets[g+1] (each a multiple of 64 long; an empty group
    gives zeros).  A [R, M], B [R, N], out [G, M, N]."""
    _need(A, BF16, "A")
    _need(B, BF16, "B")
    _need(offsets, I32, "offsets")
    _need(out, F32 if epilogue in (_lib.EPI_F32, _lib.EPI_F32_ACCUMULATE) else BF16, "out")
    _need(status, I32, "status")
    G, M, N = out.shape
    if out.stride(0) != M * out.stride(1) or offsets.numel() != G + 1:
        raise ValueError("gemm_grouped_k: out must stack its groups contiguously, offsets must have G + 1 entries")
    _chk(_lib.lib().mt_op_gemm_grouped(A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), M, N, A.shape[0],
                                       _lib.GEMM_A_MN | _lib.GEMM_B_MN, _lib.GEMM_GROUP_K, offsets.data_ptr(), G,
                                       epilogue, out.data_ptr(), out.stride(1), None, 0, None, 0, _ptr(status),
                                       _stream()))


def attention_fwd(qkv, batch, seq, n_heads, n_kv_heads, head_dim, o, lse, status=None):
    _need(qkv, BF16, "qkv")
    _need(o, BF16, "o")
    _need(lse, F32, "lse")
    _chk(_lib.lib().mt_op_attention_fwd(qkv.data_ptr(), qkv.stride(0), batch, seq, n_heads, n_kv_heads, head_dim,
                                        o.data_ptr(), o.stride(0), lse.data_ptr(), _ptr(status), _stream()))


def attention_bwd(qkv, batch, seq, n_heads, n_kv_heads, head_dim, o, lse, dout, delta, dqkv, rope_cos=None,
                  rope_sin=None, status=None):
    for t, dt, n in ((qkv, BF16, "qkv"), (o, BF16, "o"), (lse, F32, "lse"), (dout, BF16, "dout"),
                     (delta, F32, "delta"), (dqkv, BF16, "dqkv"), (rope_cos, F32, "rope_cos"),
                     (rope_sin, F32, "rope_sin")):
        _need(t, dt, n)
    _chk(_lib.lib().mt_op_attention_bwd(qkv.data_ptr(), qkv.stride(0), batch, seq, n_heads, n_kv_heads, head_dim,
                                        o.data_ptr(), o.stride(0), lse.data_ptr(), dout.data_ptr(), delta.data_ptr(),
                                        dqkv.data_ptr(), _ptr(rope_cos), _ptr(rope_sin), _ptr(status), _stream()))


def rmsnorm_fwd(x, g, y, rstd, eps):
    for t, dt, n in ((x, BF16, "x"), (g, BF16, "g"), (y, BF16, "y"), (rstd, F32, "rstd")):
        _need(t, dt, n)
    rows, d = x.shape
    _chk(_lib.lib().mt_op_rmsnorm_fwd(x.data_ptr(), g.data_ptr(), y.data_ptr(), rstd.data_ptr(), rows, d, eps,
                                      _stream()))


def rmsnorm_bwd(dy, x, g, rstd, dres, dx, dg):
    for t, dt, n in ((dy, BF16, "dy"), (x, BF16, "x"), (g, BF16, "g"), (rstd, F32, "rstd"), (dres, BF16, "dres"),
                     (dx, BF16, "dx"), (dg, BF16, "dg")):
        _need(t, dt, n)
    rows, d = x.shape
    L = _lib.lib()
    scratch = torch.empty(L.mt_op_rmsnorm_bwd_scratch_floats(rows, d), dtype=torch.float32, device=x.device)
    _chk(L.mt_op_rmsnorm_bwd(dy.data_ptr(), x.data_ptr(), g.data_ptr(), rstd.data_ptr(), _ptr(dres), dx.data_ptr(),
                             dg.data_ptr(), scratch.data_ptr(), rows, d, _stream()))


def swiglu_bwd(da, gu, dgu):
    for t, n in ((da, "da"), (gu, "gu"), (dgu, "dgu")):
        _need(t, BF16, n)
    rows, f = da.shape
    _chk(_lib.lib().mt_op_swiglu_bwd(da.data_ptr(), gu.data_ptr(), dgu.data_ptr(), rows, f, _stream()))


def transpose(src, dst):
    _need(src, BF16, "src")
    _need(dst, BF16, "dst")
    r, c = src.shape
    _chk(_lib.lib().mt_op_transpose(src.data_ptr(), r, c, src.stride(0), dst.data_ptr(), dst.stride(0), _stream()))


def cross_entropy(z, tgt, inv_n, dz, loss_rows, status=None):
    for t, dt, n in ((z, F32, "z"), (tgt, I32, "tgt"), (dz, BF16, "dz"), (loss_rows, F32, "loss_rows"),
                     (status, I32, "status")):
        _need(t, dt, n)
    rows, V = z.shape
    _chk(_lib.lib().mt_op_cross_entropy(z.data_ptr(), rows, V, tgt.data_ptr(), inv_n, dz.data_ptr(),
                                        loss_rows.data_ptr(), _ptr(status), _stream()))


def embedding_fwd(tok, E, x, status=None):
    for t, dt, n in ((tok, I32, "tok"), (E, BF16, "E"), (x, BF16, "x"), (status, I32, "status")):
        _need(t, dt, n)
    V, d = E.shape
    _chk(_lib.lib().mt_op_embedding_fwd(tok.data_ptr(), E.data_ptr(), x.data_ptr(), tok.numel(), d, V, _ptr(status),
                                        _stream()))


def embedding_bwd(row_offsets, positions, dx, dE):
    for t, dt, n in ((row_offsets, I32, "row_offsets"), (positions, I32, "positions"), (dx, BF16, "dx"),
                     (dE, BF16, "dE")):
        _need(t, dt, n)
    V, d = dE.shape
    _chk(_lib.lib().mt_op_embedding_bwd(row_offsets.data_ptr(), positions.data_ptr(), dx.data_ptr(), dE.data_ptr(),
                                        V, d, _stream()))


# ------------------------------------------------------------------ mixture of experts
def moe_route(logits, k, row_align=1):
    """FP32 router logits [N, E] -> (idx [N, k], gates [N, k], order [R], pos [N k], offsets [E + 1]).

    Each expert's positions are padded to a multiple of row_align (order = -1
    there); R = N k + (row_align - 1) E."""
    _need(logits, F32, "logits")
    N, E = logits.shape
    dev = logits.device
    R = int(_lib.lib().mt_op_moe_rows_capacity(N * k, E, row_align))
    if R < 0:
        raise ValueError("moe_route: row_align must be in 1 .. 256")
    idx = torch.empty(N, k, device=dev, dtype=I32)
    gates = torch.empty(N, k, device=dev, dtype=F32)
    order = torch.empty(R, device=dev, dtype=I32)
    pos = torch.empty(N * k, device=dev, dtype=I32)
    offsets = torch.empty(E + 1, device=dev, dtype=I32)
    scratch = torch.empty(int(_lib.lib().mt_op_moe_sort_scratch_ints(N * k, E)), device=dev, dtype=I32)
    _chk(_lib.lib().mt_op_moe_route(logits.data_ptr(), N, E, k, row_align, idx.data_ptr(), gates.data_ptr(),
                                    order.data_ptr(), pos.data_ptr(), offsets.data_ptr(), scratch.data_ptr(),
                                    _stream()))
    return idx, gates, order, pos, offsets


def moe_zero_pads(order, buf):
    """buf[i] = 0 for the padding rows (order[i] = -1)."""
    _need(buf, BF16, "buf")
    _chk(_lib.lib().mt_op_moe_zero_pads(order.data_ptr(), order.numel(), buf.shape[1], buf.data_ptr(), _stream()))


def moe_gather(x, order, k):
    _need(x, BF16, "x")
    P, d = order.numel(), x.shape[1]
    xp = torch.empty(P, d, device=x.device, dtype=BF16)
    _chk(_lib.lib().mt_op_moe_gather(x.data_ptr(), x.stride(0), order.data_ptr(), k, P, d, xp.data_ptr(), _stream()))
    return xp


def moe_combine(yp, pos, gates, residual=None):
    _need(yp, BF16, "yp")
    N, k = gates.shape
    d = yp.shape[1]
    out = torch.empty(N, d, device=yp.device, dtype=BF16)
    _chk(_lib.lib().mt_op_moe_combine(yp.data_ptr(), pos.data_ptr(), gates.data_ptr(), N, k, d, _ptr(residual),
                                      out.data_ptr(), _stream()))
    return out


def moe_combine_bwd(dy, yp, pos, gates):
    N, k = gates.shape
    d = dy.shape[1]
    dyp = torch.empty(yp.shape[0], d, device=dy.device, dtype=BF16)
    dgates = torch.empty(N, k, device=dy.device, dtype=F32)
    _chk(_lib.lib().mt_op_moe_combine_bwd(dy.data_ptr(), yp.data_ptr(), pos.data_ptr(), gates.data_ptr(), N, k, d,
                                          dyp.data_ptr(), dgates.data_ptr(), _stream()))
    return dyp, dgates


def moe_gate_bwd(idx, gates, dgates, E):
    N, k = gates.shape
    ds = torch.empty(N, E, device=gates.device, dtype=BF16)
    _chk(_lib.lib().mt_op_moe_gate_bwd(idx.data_ptr(), gates.data_ptr(), dgates.data_ptr(), N, E, k, ds.data_ptr(),
                                       _stream()))
    return ds


def moe_scatter_bwd(dxp, pos, N, k, dres=None):
    d = dxp.shape[1]
    dx = torch.empty(N, d, device=dxp.device, dtype=BF16)
    _chk(_lib.lib().mt_op_moe_scatter_bwd(dxp.data_ptr(), pos.data_ptr(), N, k, d, _ptr(dres), dx.data_ptr(),
                                          _stream()))
    return dx


def moe_mlp_forward(x, wr, wgu, wd, k):
    """The MoE MLP on the device from the pieces above and the grouped tcgen05
    GEMM, with no host read of the routing: x [N, d] BF16, wr [E, d], wgu
    [E, 2F, d] (gate/up rows interleaved), wd [E, d, F].  Returns (y [N, d]
    BF16, saved tensors for the backward).  Each expert's rows are padded to a
    multiple of 64 with zero rows (the weight-gradient GEMM's K block)."""
    N, d = x.shape
    E, twoF, _ = wgu.shape
    Fh = twoF // 2
    logits = torch.empty(N, E, device=x.device, dtype=F32)
    gemm(x, wr, logits, _lib.EPI_F32)
    idx, gates, order, pos, offsets = moe_route(logits, k, row_align=64)
    xp = moe_gather(x, order, k)
    R = order.numel()
    ap = torch.empty(R, Fh, device=x.device, dtype=BF16)
    gup = torch.empty(R, twoF, device=x.device, dtype=BF16)
    yp = torch.empty(R, d, device=x.device, dtype=BF16)
    gemm_grouped_rows(xp, wgu, offsets, ap, epilogue=_lib.EPI_SWIGLU, out2=gup)
    gemm_grouped_rows(ap, wd, offsets, yp)
    y = moe_combine(yp, pos, gates)
    return y, dict(idx=idx, gates=gates, order=order, pos=pos, offsets=offsets, xp=xp, ap=ap, gup=gup, yp=yp)


def moe_mlp_backward(dy, x, wr, wgu, wd, k, saved):
    """Gradients of the MoE MLP: (dx, dwr, dwgu [E, 2F, d], dwd [E, d, F]).
    Every expert GEMM is one grouped launch; experts without rows get zero
    gradients."""
    N, d = x.shape
    E, twoF, _ = wgu.shape
    offsets, order = saved["offsets"], saved["order"]
    dyp, dgates = moe_combine_bwd(dy, saved["yp"], saved["pos"], saved["gates"])
    moe_zero_pads(order, dyp)
    R = order.numel()
    dgup = torch.empty(R, twoF, device=x.device, dtype=BF16)
    dxp = torch.empty(R, d, device=x.device, dtype=BF16)
    dwgu = torch.empty_like(wgu)
    dwd = torch.empty_like(wd)
    gemm_grouped_k(dyp, saved["ap"], offsets, dwd)
    gemm_grouped_rows(dyp, wd, offsets, dgup, b_mn=True, epilogue=_lib.EPI_SWIGLU_BWD, residual=saved["gup"])
    gemm_grouped_k(dgup, saved["xp"], offsets, dwgu)
    gemm_grouped_rows(dgup, wgu, offsets, dxp, b_mn=True)
    ds = moe_gate_bwd(saved["idx"], saved["gates"], dgates, E)
    dwr = torch.empty_like(wr)
    gemm_layout(ds, x, dwr, a_mn=True, b_mn=True)
    dx_router = torch.empty(N, d, device=x.device, dtype=BF16)
    gemm_layout(ds, wr, dx_router, b_mn=True)
    dx = moe_scatter_bwd(dxp, saved["pos"], N, k, dres=dx_router)
    return dx, dwr, dwgu, dwd