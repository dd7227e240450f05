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


def gemm(A, B, out, epilogue=_lib.EPI_STORE_BF16, residual=None, out2=None, rope_cos=None, rope_sin=None,
         rope_cols=0, head_dim=0, seq=1, status=None):
    """out = epilogue(A @ B^T); A [M, K], B [N, K] BF16 (row strides may exceed K)."""
    _need(A, torch.bfloat16, "A")
    _need(B, torch.bfloat16, "B")
    M, K = A.shape
    N = B.shape[0]
    _chk(_lib.lib().mt_op_gemm(A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), M, N, K, epilogue,
                               out.data_ptr(), out.stride(0), _ptr(residual),
                               residual.stride(0) if residual is not None else 0, _ptr(out2),
                               out2.stride(0) if out2 is not None else 0, _ptr(rope_cos), _ptr(rope_sin),
                               rope_cols, head_dim, seq, _ptr(status), _stream()))


def attention_fwd(qkv, batch, seq, n_heads, n_kv_heads, head_dim, o, lse):
    _need(qkv, torch.bfloat16, "qkv")
    _chk(_lib.lib().mt_op_attention_fwd(qkv.data_ptr(), qkv.stride(0), batch, seq, n_heads, n_kv_heads, head_dim,
                                        o.data_ptr(), o.stride(0), lse.data_ptr(), _stream()))


def attention_bwd(qkv, batch, seq, n_heads, n_kv_heads, head_dim, o, lse, dout, delta, dqkv, rope_cos=None,
                  rope_sin=None):
    _chk(_lib.lib().mt_op_attention_bwd(qkv.data_ptr(), qkv.stride(0), batch, seq, n_heads, n_kv_heads, head_dim,
                                        o.data_ptr(), o.stride(0), lse.data_ptr(), dout.data_ptr(), delta.data_ptr(),
                                        dqkv.data_ptr(), _ptr(rope_cos), _ptr(rope_sin), _stream()))


def rmsnorm_fwd(x, g, y, rstd, eps):
    rows, d = x.shape
    _chk(_lib.lib().mt_op_rmsnorm_fwd(x.data_ptr(), g.data_ptr(), y.data_ptr(), rstd.data_ptr(), rows, d, eps,
                                      _stream()))


def rmsnorm_bwd(dy, x, g, rstd, dres, dx, dg):
    rows, d = x.shape
    L = _lib.lib()
    scratch = torch.empty(L.mt_op_rmsnorm_bwd_scratch_floats(rows, d), dtype=torch.float32, device=x.device)
    _chk(L.mt_op_rmsnorm_bwd(dy.data_ptr(), x.data_ptr(), g.data_ptr(), rstd.data_ptr(), _ptr(dres), dx.data_ptr(),
                             dg.data_ptr(), scratch.data_ptr(), rows, d, _stream()))


def swiglu_bwd(da, gu, dgu):
    rows, f = da.shape
    _chk(_lib.lib().mt_op_swiglu_bwd(da.data_ptr(), gu.data_ptr(), dgu.data_ptr(), rows, f, _stream()))


def transpose(src, dst):
    r, c = src.shape
    _chk(_lib.lib().mt_op_transpose(src.data_ptr(), r, c, src.stride(0), dst.data_ptr(), dst.stride(0), _stream()))


def cross_entropy(z, tgt, inv_n, dz, loss_rows, status=None):
    rows, V = z.shape
    _chk(_lib.lib().mt_op_cross_entropy(z.data_ptr(), rows, V, tgt.data_ptr(), inv_n, dz.data_ptr(),
                                        loss_rows.data_ptr(), _ptr(status), _stream()))


def embedding_fwd(tok, E, x, status=None):
    V, d = E.shape
    _chk(_lib.lib().mt_op_embedding_fwd(tok.data_ptr(), E.data_ptr(), x.data_ptr(), tok.numel(), d, V, _ptr(status),
                                        _stream()))


def embedding_bwd(row_offsets, positions, dx, dE):
    V, d = dE.shape
    _chk(_lib.lib().mt_op_embedding_bwd(row_offsets.data_ptr(), positions.data_ptr(), dx.data_ptr(), dE.data_ptr(),
                                        V, d, _stream()))
