// Tile layouts and the stateless layer template.
//
// A template is the kernel sequence of one decoder layer (or of the
// embedding / head) with no weight pointers of its own: Bind computes views
// into whichever device buffer currently holds the tile (pointer arithmetic
// over the tile's static offsets, no copy), and the same sequence runs on it
// (MegaTrain paperlayer.ai summary §A.4 "GPU Compute Dispatch"; hyper.ai
// summary 方法 ¶6: templates hold the compute kernels but no persistent
// weight pointers; a Bind primitive maps views of the streaming buffer into
// the template's input slots).  Because the host tile layout equals the
// device view layout, Bind needs no gather kernel.
#include <algorithm>
#include <cstring>
#include <stdexcept>

#include "runtime.h"

namespace mt {

const TensorSlot& TileLayout::slot(const char* n) const {
  for (const auto& t : tensors)
    if (t.name == n) return t;
  throw std::runtime_error(std::string("no tensor ") + n);
}

bool TileLayout::has(const char* n) const {
  for (const auto& t : tensors)
    if (t.name == n) return true;
  return false;
}

Dims dims_of(const mt_config& c) {
  Dims d;
  d.L = c.n_layers;
  d.d = c.d_model;
  d.Hq = c.n_heads;
  d.Hkv = c.n_kv_heads;
  d.hd = c.head_dim;
  d.f = c.ffn;
  d.V = c.vocab;
  d.B = c.batch;
  d.S = c.seq;
  d.T = (long)c.batch * c.seq;
  d.Tc = (c.mlp_chunk_rows > 0 && c.mlp_chunk_rows < d.T) ? (long)c.mlp_chunk_rows : d.T;
  d.Dq = c.n_heads * c.head_dim;
  d.Dqkv = (c.n_heads + 2 * c.n_kv_heads) * c.head_dim;
  d.E = c.n_experts > 0 ? c.n_experts : 0;
  d.k = d.E ? c.top_k : 0;
  return d;
}

TileLayout make_layout(TileKind kind, const Dims& d, bool tied) {
  TileLayout L;
  L.kind = kind;
  auto add = [&](const char* n, int64_t r, int64_t c) {
    TensorSlot s;
    s.name = n;
    s.ndim = c ? 2 : 1;
    s.shape[0] = r;
    s.shape[1] = c;
    s.numel = c ? r * c : r;
    L.tensors.push_back(s);
  };
  if (kind == kTileEmbed) {
    add("E", d.V, d.d);
    if (tied) add("gf", d.d, 0);
  } else if (kind == kTileLayer) {
    add("g1", d.d, 0);
    add("wqkv", d.Dqkv, d.d);
    add("wo", d.d, d.Dq);
    add("g2", d.d, 0);
    if (d.E) {  // MoE: router, then the experts stacked (expert e's rows at e * rows-per-expert)
      add("wr", d.E, d.d);
      add("wgu", (int64_t)d.E * 2L * d.f, d.d);
      add("wd", (int64_t)d.E * d.d, d.f);
    } else {
      add("wgu", 2L * d.f, d.d);
      add("wd", d.d, d.f);
    }
  } else {
    add("gf", d.d, 0);
    add("wh", d.V, d.d);
  }
  int64_t off = 0;
  for (auto& t : L.tensors) {
    t.offset = off;
    off = align_up(off + t.numel * 2, kTensorAlign);
    L.n_params += t.numel;
  }
  L.w_bytes = align_up(off, kPage);
  L.mv_bytes = 2 * L.w_bytes;
  L.off_w = 0;
  L.off_g = L.w_bytes;
  L.off_m = 2 * L.w_bytes;
  L.off_v = 2 * L.w_bytes + L.mv_bytes;
  L.tile_bytes = 2 * L.w_bytes + 2 * L.mv_bytes;
  return L;
}

LayerView bind_layer(const TileLayout& lay, void* base) {
  auto p = [&](const char* n) { return reinterpret_cast<bf16*>(static_cast<uint8_t*>(base) + lay.slot(n).offset); };
  LayerView v{p("g1"), p("wqkv"), p("wo"), p("g2"), p("wgu"), p("wd")};
  if (lay.has("wr")) v.wr = p("wr");
  return v;
}

HeadView bind_head(const TileLayout& lay, void* base) {
  auto p = [&](const char* n) { return reinterpret_cast<bf16*>(static_cast<uint8_t*>(base) + lay.slot(n).offset); };
  // tied embeddings: the head's weight is the embedding table itself
  return HeadView{p("gf"), lay.has("wh") ? p("wh") : p("E")};
}

// ------------------------------------------------------------------ template
int LayerTemplate::gemm(const GemmArgs& g) const {
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (stats->time_gemms) {
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    cudaEventRecord(e0, s);
  }
  const int rc = launch_gemm(g, s);
  if (stats->time_gemms) {
    cudaEventRecord(e1, s);
    stats->gemm_events->push_back(e0);
    stats->gemm_events->push_back(e1);
    stats->gemm_event_flops->push_back(2.0 * g.M * g.N * g.K);
  }
  stats->kernels += 1;
  stats->gemms += 1;
  stats->gemm_flops += 2.0 * g.M * g.N * g.K;
  trace(g.a_mn || g.b_mn ? "gemm (MN-major operand)" : "gemm");
  return rc;
}

// One grouped launch (an MoE layer's expert GEMMs); the statistics count the
// FLOPs of the `rows` routed rows (padding and skipped tiles excluded).
int LayerTemplate::gemm_grouped(const GemmArgs& g, const int32_t* offsets, int groups, int mode, long rows) const {
  const int rc = launch_gemm_grouped(g, offsets, groups, mode, s);
  const double flops = mode == kGemmGroupRows ? 2.0 * rows * g.N * g.K : 2.0 * g.M * g.N * rows;
  stats->kernels += 1;
  stats->gemms += 1;
  stats->gemm_flops += flops;
  trace("grouped gemm");
  return rc;
}

namespace {
GemmArgs mk(const bf16* A, long lda, const bf16* B, long ldb, int M, int N, int K, int epi, void* C, long ldc,
            int* status) {
  GemmArgs g;
  g.A = A;
  g.lda = lda;
  g.B = B;
  g.ldb = ldb;
  g.M = M;
  g.N = N;
  g.K = K;
  g.epi = epi;
  g.C = C;
  g.ldc = ldc;
  g.status = status;
  return g;
}
}  // namespace

int LayerTemplate::forward(const LayerView& w, LayerActs& a, bf16* x_out, bool keep_gu) const {
  const Dims& D = dm;
  const long T = D.T;
  int rc = 0;
  launch_rmsnorm_fwd(a.x, w.g1, a.n1, a.rstd1, T, D.d, eps, s);
  trace("rmsnorm_fwd");
  // qkv = n1 Wqkv^T with rotate-half RoPE on the q and k columns
  GemmArgs g = mk(a.n1, D.d, w.wqkv, D.d, (int)T, D.Dqkv, D.d, kEpiRope, a.qkv, D.Dqkv, ws->status);
  g.rope_cos = ws->rope_cos;
  g.rope_sin = ws->rope_sin;
  g.rope_cols = (D.Hq + D.Hkv) * D.hd;
  g.head_dim = D.hd;
  g.seq = D.S;
  rc |= gemm(g);
  AttnArgs at;
  at.qkv = a.qkv;
  at.ldqkv = D.Dqkv;
  at.batch = D.B;
  at.seq = D.S;
  at.n_heads = D.Hq;
  at.n_kv_heads = D.Hkv;
  at.head_dim = D.hd;
  at.o = a.o;
  at.ldo = D.Dq;
  at.lse = a.lse;
  at.status = ws->status;
  rc |= launch_attn_fwd(at, s);
  trace("attention_fwd");
  // h = x + o Wo^T
  g = mk(a.o, D.Dq, w.wo, D.Dq, (int)T, D.d, D.Dq, kEpiResidualBf16, a.h, D.d, ws->status);
  g.R = a.x;
  g.ldr = D.d;
  rc |= gemm(g);
  launch_rmsnorm_fwd(a.h, w.g2, a.n2, a.rstd2, T, D.d, eps, s);
  trace("rmsnorm_fwd");
  if (D.E) {
    stats->kernels += 3;
    return rc | moe_forward(w, a, x_out);
  }
  if (D.Tc < T) {
    // chunked MLP: the gate/up activations of one row chunk at a time.  An
    // internals-only pass (for backward) stops here: backward recomputes the
    // MLP chunk by chunk.
    if (x_out) {
      for (long c0 = 0; c0 < T; c0 += D.Tc) {
        const int rows = (int)std::min(D.Tc, T - c0);
        g = mk(a.n2 + c0 * D.d, D.d, w.wgu, D.d, rows, 2 * D.f, D.d, kEpiSwiGLU, a.a, D.f, ws->status);
        rc |= gemm(g);
        g = mk(a.a, D.f, w.wd, D.f, rows, D.d, D.f, kEpiResidualBf16, x_out + c0 * D.d, D.d, ws->status);
        g.R = a.h + c0 * D.d;
        g.ldr = D.d;
        rc |= gemm(g);
      }
    }
    stats->kernels += 3;
    return rc;
  }
  // a = silu(n2 Wg^T) * (n2 Wu^T) from interleaved gate/up rows
  g = mk(a.n2, D.d, w.wgu, D.d, (int)T, 2 * D.f, D.d, kEpiSwiGLU, a.a, D.f, ws->status);
  if (keep_gu) {
    g.C2 = a.gu;
    g.ldc2 = 2L * D.f;
  }
  rc |= gemm(g);
  // x_out = h + a Wd^T (skipped when only the internals are recomputed for backward)
  if (x_out) {
    g = mk(a.a, D.f, w.wd, D.f, (int)T, D.d, D.f, kEpiResidualBf16, x_out, D.d, ws->status);
    g.R = a.h;
    g.ldr = D.d;
    rc |= gemm(g);
  }
  stats->kernels += 3;
  return rc;
}

int LayerTemplate::backward(const LayerView& w, const LayerActs& a, const bf16* dx_out, bf16* dx_in,
                            const LayerView& gv) const {
  const Dims& D = dm;
  const long T = D.T;
  const Workspace& W = *ws;
  int rc = 0;
  // Weight gradient dW[N, K] = dY[T, N]^T X[T, K]: both operands read MN-major
  // (T is the contraction, N and K contiguous), no transpose pass.
  auto wgrad = [&](const bf16* dY, int N, const bf16* X, int K, bf16* dW) {
    GemmArgs g = mk(dY, N, X, K, N, K, (int)T, kEpiStoreBf16, dW, K, W.status);
    g.a_mn = true;
    g.b_mn = true;
    rc |= gemm(g);
  };
  // Data gradient dX[T, K] = dY[T, N] W[N, K]: W read MN-major.
  auto dgrad = [&](const bf16* dY, int N, const bf16* Wm, int K, bf16* dX) {
    GemmArgs g = mk(dY, N, Wm, K, (int)T, K, N, kEpiStoreBf16, dX, K, W.status);
    g.b_mn = true;
    rc |= gemm(g);
  };

  if (D.E) {
    rc |= moe_backward(w, a, dx_out, gv);
  } else if (D.Tc < T) {
    rc |= mlp_backward_chunked(w, a, dx_out, gv);
  } else {
  // x_out = h + a Wd^T
  wgrad(dx_out, D.d, a.a, D.f, gv.wd);
  // da = dx_out Wd (Wd read MN-major), and in the same epilogue the SwiGLU
  // backward: dgu = (da * up * silu'(gate), da * silu(gate)) from the stored gate/up
  {
    GemmArgs g = mk(dx_out, D.d, w.wd, D.f, (int)T, D.f, D.d, kEpiSwiGLUBwd, W.dgu, 2L * D.f, W.status);
    g.b_mn = true;
    g.R = a.gu;
    g.ldr = 2L * D.f;
    rc |= gemm(g);
  }
  wgrad(W.dgu, 2 * D.f, a.n2, D.d, gv.wgu);
  dgrad(W.dgu, 2 * D.f, w.wgu, D.d, W.dn);
  }
  // dh = dx_out + RMSNorm2^T dn2 ; dg2
  {
    const long parts = launch_rmsnorm_bwd(W.dn, a.h, w.g2, a.rstd2, dx_out, W.dh, W.dg_partial, T, D.d, s);
    trace("rmsnorm_bwd");
    launch_colsum_bf16(W.dg_partial, parts, D.d, gv.g2, s);
  }
  // h = x + o Wo^T
  wgrad(W.dh, D.d, a.o, D.Dq, gv.wo);
  dgrad(W.dh, D.d, w.wo, D.Dq, W.dout);
  AttnArgs at;
  at.qkv = a.qkv;
  at.ldqkv = D.Dqkv;
  at.batch = D.B;
  at.seq = D.S;
  at.n_heads = D.Hq;
  at.n_kv_heads = D.Hkv;
  at.head_dim = D.hd;
  at.o = a.o;
  at.ldo = D.Dq;
  at.lse = a.lse;
  at.dout = W.dout;
  at.delta = W.delta;
  at.dqkv = W.dqkv;
  at.rope_cos = W.rope_cos;
  at.rope_sin = W.rope_sin;
  at.status = W.status;
  rc |= launch_attn_bwd(at, s);
  trace("attention_bwd");
  wgrad(W.dqkv, D.Dqkv, a.n1, D.d, gv.wqkv);
  dgrad(W.dqkv, D.Dqkv, w.wqkv, D.d, W.dn);
  {
    const long parts = launch_rmsnorm_bwd(W.dn, a.x, w.g1, a.rstd1, W.dh, dx_in, W.dg_partial, T, D.d, s);
    trace("rmsnorm_bwd");
    launch_colsum_bf16(W.dg_partial, parts, D.d, gv.g1, s);
  }
  stats->kernels += 7;  // 2 x (rmsnorm bwd + colsum), attention delta + dK/dV + dQ
  return rc;
}

// ------------------------------------------------------------------ MoE layers
// The MLP half of an MoE decoder layer: router logits n2 W_r^T (FP32), top-k
// routing and the stable sort of the (token, slot) pairs by expert (each
// expert's rows padded to a multiple of 64 with zero rows), the routed rows of
// n2 gathered, the experts' gate/up (+SwiGLU) and down GEMMs as one grouped
// launch each (the per-expert row counts stay on the device), and the
// gate-weighted combine with the residual h.
int LayerTemplate::moe_forward(const LayerView& w, LayerActs& a, bf16* x_out) const {
  const Dims& D = dm;
  const long T = D.T;
  const int E = D.E, k = D.k, F = D.f, d = D.d;
  const long P = T * k, R = moe_rows_capacity(P, E, kMoeRowAlign);
  int rc = 0;
  rc |= gemm(mk(a.n2, d, w.wr, d, (int)T, E, d, kEpiF32, a.moe_logits, E, ws->status));
  rc |= launch_moe_topk(a.moe_logits, T, E, k, a.moe_idx, a.moe_gates, s) ? 1 : 0;
  rc |= launch_moe_sort(a.moe_idx, P, E, kMoeRowAlign, ws->moe_scratch, a.moe_order, a.moe_pos, a.moe_off, s) ? 1 : 0;
  rc |= launch_moe_gather(a.n2, d, a.moe_order, k, R, d, a.moe_xp, s) ? 1 : 0;
  stats->kernels += 5;
  trace("moe routing");
  GemmArgs g = mk(a.moe_xp, d, w.wgu, d, (int)R, 2 * F, d, kEpiSwiGLU, a.moe_ap, F, ws->status);
  g.C2 = a.moe_gup;
  g.ldc2 = 2L * F;
  rc |= gemm_grouped(g, a.moe_off, E, kGemmGroupRows, P);
  rc |= gemm_grouped(mk(a.moe_ap, F, w.wd, F, (int)R, d, F, kEpiStoreBf16, a.moe_yp, d, ws->status), a.moe_off, E,
                     kGemmGroupRows, P);
  if (x_out) {
    rc |= launch_moe_combine(a.moe_yp, a.moe_pos, a.moe_gates, T, k, d, a.h, x_out, s) ? 1 : 0;
    stats->kernels += 1;
  }
  return rc;
}

// Backward of moe_forward (its internals recomputed for this visit): dn2 into
// ws->dn; the experts' and the router's weight gradients into gv.  Every
// expert GEMM is one grouped launch; experts that received no row get zero
// gradients from the grouped weight-gradient GEMM itself.
int LayerTemplate::moe_backward(const LayerView& w, const LayerActs& a, const bf16* dx_out,
                                const LayerView& gv) const {
  const Dims& D = dm;
  const long T = D.T;
  const int E = D.E, k = D.k, F = D.f, d = D.d;
  const long P = T * k, R = moe_rows_capacity(P, E, kMoeRowAlign);
  const Workspace& W = *ws;
  int rc = 0;
  rc |= launch_moe_combine_bwd(dx_out, a.moe_yp, a.moe_pos, a.moe_gates, T, k, d, W.moe_dyp, W.moe_dgates, s) ? 1 : 0;
  rc |= launch_moe_zero_pads(a.moe_order, R, d, W.moe_dyp, s) ? 1 : 0;  // the padding rows enter the K sums
  stats->kernels += 2;
  // dW_d[e] = dY_e^T A_e over each expert's rows (both operands MN-major)
  GemmArgs g = mk(W.moe_dyp, d, a.moe_ap, F, d, F, (int)R, kEpiStoreBf16, gv.wd, F, W.status);
  g.a_mn = g.b_mn = true;
  rc |= gemm_grouped(g, a.moe_off, E, kGemmGroupK, P);
  // da = dY W_d[e] and, in the epilogue, the SwiGLU backward against the kept gate/up pairs
  g = mk(W.moe_dyp, d, w.wd, F, (int)R, F, d, kEpiSwiGLUBwd, W.moe_dgup, 2L * F, W.status);
  g.b_mn = true;
  g.R = a.moe_gup;
  g.ldr = 2L * F;
  rc |= gemm_grouped(g, a.moe_off, E, kGemmGroupRows, P);
  // dW_gu[e] = dGU_e^T Xp_e
  g = mk(W.moe_dgup, 2L * F, a.moe_xp, d, 2 * F, d, (int)R, kEpiStoreBf16, gv.wgu, d, W.status);
  g.a_mn = g.b_mn = true;
  rc |= gemm_grouped(g, a.moe_off, E, kGemmGroupK, P);
  // dXp = dGU W_gu[e]
  g = mk(W.moe_dgup, 2L * F, w.wgu, d, (int)R, d, 2 * F, kEpiStoreBf16, W.moe_dxp, d, W.status);
  g.b_mn = true;
  rc |= gemm_grouped(g, a.moe_off, E, kGemmGroupRows, P);
  // router: ds = softmax backward over the selected logits; dW_r = ds^T n2; dn2 += ds W_r
  rc |= launch_moe_gate_bwd(a.moe_idx, a.moe_gates, W.moe_dgates, T, E, k, W.moe_ds, s) ? 1 : 0;
  g = mk(W.moe_ds, E, a.n2, d, E, d, (int)T, kEpiStoreBf16, gv.wr, d, W.status);
  g.a_mn = g.b_mn = true;
  rc |= gemm(g);
  g = mk(W.moe_ds, E, w.wr, d, (int)T, d, E, kEpiStoreBf16, W.moe_dn2r, d, W.status);
  g.b_mn = true;
  rc |= gemm(g);
  rc |= launch_moe_scatter_bwd(W.moe_dxp, a.moe_pos, T, k, d, W.moe_dn2r, W.dn, s) ? 1 : 0;
  stats->kernels += 2;
  return rc;
}

// MLP backward over row chunks (long sequences): per chunk, recompute the
// gate/up GEMM (the forward kept no [T, 2 ffn] activations), then
//   dW_d  += dx_out^T a          (FP32, accumulated across chunks)
//   dgu    = SwiGLU'(dx_out W_d)  (fused into the GEMM epilogue)
//   dW_gu += dgu^T n2             (FP32)
//   dn2    = dgu W_gu
// and finally the two FP32 gradients are rounded into the BF16 tile.
int LayerTemplate::mlp_backward_chunked(const LayerView& w, const LayerActs& a, const bf16* dx_out,
                                        const LayerView& gv) const {
  const Dims& D = dm;
  const long T = D.T;
  const Workspace& W = *ws;
  int rc = 0;
  for (long c0 = 0; c0 < T; c0 += D.Tc) {
    const int rows = (int)std::min(D.Tc, T - c0);
    const int acc = c0 == 0 ? kEpiF32 : kEpiF32Accumulate;
    const bf16* n2 = a.n2 + c0 * D.d;
    const bf16* dy = dx_out + c0 * D.d;
    GemmArgs g = mk(n2, D.d, w.wgu, D.d, rows, 2 * D.f, D.d, kEpiSwiGLU, a.a, D.f, W.status);
    g.C2 = a.gu;
    g.ldc2 = 2L * D.f;
    rc |= gemm(g);
    g = mk(dy, D.d, a.a, D.f, D.d, D.f, rows, acc, W.dwd_f32, D.f, W.status);
    g.a_mn = true;
    g.b_mn = true;
    rc |= gemm(g);
    g = mk(dy, D.d, w.wd, D.f, rows, D.f, D.d, kEpiSwiGLUBwd, W.dgu, 2L * D.f, W.status);
    g.b_mn = true;
    g.R = a.gu;
    g.ldr = 2L * D.f;
    rc |= gemm(g);
    g = mk(W.dgu, 2L * D.f, n2, D.d, 2 * D.f, D.d, rows, acc, W.dwgu_f32, D.d, W.status);
    g.a_mn = true;
    g.b_mn = true;
    rc |= gemm(g);
    g = mk(W.dgu, 2L * D.f, w.wgu, D.d, rows, D.d, 2 * D.f, kEpiStoreBf16, W.dn + c0 * D.d, D.d, W.status);
    g.b_mn = true;
    rc |= gemm(g);
  }
  launch_f32_to_bf16(W.dwd_f32, gv.wd, (long)D.d * D.f, s);
  trace("f32_to_bf16");
  launch_f32_to_bf16(W.dwgu_f32, gv.wgu, 2L * D.f * D.d, s);
  trace("f32_to_bf16");
  stats->kernels += 2;
  return rc;
}

int LayerTemplate::head(const HeadView& w, const bf16* x_L, bf16* dx_L, const HeadView& gv) const {
  const Dims& D = dm;
  const long T = D.T;
  const Workspace& W = *ws;
  int rc = 0;
  launch_rmsnorm_fwd(x_L, w.gf, W.nf, W.rstd_f, T, D.d, eps, s);
  launch_zero(W.dwh_f32, sizeof(float) * (size_t)D.V * D.d, s);
  stats->kernels += 1;
  const float inv_n = loss_scale / (float)T;
  for (long r0 = 0; r0 < T; r0 += W.head_chunk) {
    const long rows = (T - r0) < W.head_chunk ? (T - r0) : W.head_chunk;
    const bf16* nf = W.nf + r0 * D.d;
    rc |= gemm(mk(nf, D.d, w.wh, D.d, (int)rows, D.V, D.d, kEpiF32, W.z, D.V, W.status));
    launch_cross_entropy(W.z, rows, D.V, W.tgt + r0, inv_n, W.dz, W.loss_rows + r0, W.status, s);
    trace("cross_entropy");
    // d nf = dz W_h  (W_h [V, d] read MN-major)
    GemmArgs g = mk(W.dz, D.V, w.wh, D.d, (int)rows, D.d, D.V, kEpiStoreBf16, W.dnf + r0 * D.d, D.d, W.status);
    g.b_mn = true;
    rc |= gemm(g);
    // dW_h += dz^T nf  (both operands MN-major, the chunk's tokens are the contraction)
    g = mk(W.dz, D.V, nf, D.d, D.V, D.d, (int)rows, kEpiF32Accumulate, W.dwh_f32, D.d, W.status);
    g.a_mn = true;
    g.b_mn = true;
    rc |= gemm(g);
    stats->kernels += 1;
  }
  launch_f32_to_bf16(W.dwh_f32, gv.wh, (long)D.V * D.d, s);
  trace("f32_to_bf16");
  launch_mean_loss(W.loss_rows, T, inv_n, W.loss, s);
  trace("mean_loss");
  {
    const long parts = launch_rmsnorm_bwd(W.dnf, x_L, w.gf, W.rstd_f, nullptr, dx_L, W.dg_partial, T, D.d, s);
    launch_colsum_bf16(W.dg_partial, parts, D.d, gv.gf, s);
  }
  stats->kernels += 4;
  return rc;
}

int LayerTemplate::embed_fwd(const bf16* E, bf16* x0) const {
  launch_embed_fwd(ws->inp, E, x0, dm.T, dm.d, dm.V, ws->status, s);
  trace("embed_fwd");
  stats->kernels += 1;
  return 0;
}

int LayerTemplate::embed_bwd_rows(const bf16* dx0, bf16* out, int U) const {
  launch_embed_bwd_rows(ws->emb_off, ws->emb_pos, ws->emb_rows, U, dx0, out, dm.d, s);
  trace("embed_bwd_rows");
  stats->kernels += 1;
  return 0;
}

int LayerTemplate::embed_bwd(const bf16* dx0, bf16* dE) const {
  launch_embed_bwd(ws->emb_off, ws->emb_pos, dx0, dE, dm.V, dm.d, s);
  trace("embed_bwd");
  stats->kernels += 1;
  return 0;
}

}  // namespace mt
