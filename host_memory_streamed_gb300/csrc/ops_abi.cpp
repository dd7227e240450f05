// C-ABI wrappers of the individual device kernels (declared in include/mt_ops.h).
// They take device pointers and a cudaStream_t passed as void*, launch one
// kernel sequence and return without synchronising.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/mt_ops.h"
#include "kernels.h"

static_assert((int)MT_STATUS_WAIT_PROBE == (int)mt::kStatusWaitProbe, "wait-probe status code");

namespace {
thread_local std::string g_op_error;
int op_fail(const char* msg) {
  g_op_error = msg ? msg : "unknown error";
  return MT_EINVAL;
}
// 16-byte aligned (NULL counts as aligned: null checks are separate)
bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
constexpr int64_t kMaxGridRows = 0x7fffffff;  // one CTA per row: grid.x limit
int op_cuda(int rc, const char* what) {
  if (rc == 0) return MT_OK;
  g_op_error = std::string(what) + ": launch failed (" + (rc == -4 ? mt::last_launch_error() : "bad descriptor or attributes") + ")";
  return MT_ECUDA;
}
}  // namespace

namespace mt {
void set_op_error(const std::string& msg) { g_op_error = msg; }
}  // namespace mt

extern "C" {

const char* mt_op_last_error(void) { return g_op_error.c_str(); }

int mt_op_gemm(const void* A, int64_t lda, const void* B, int64_t ldb, int32_t M, int32_t N, int32_t K,
               int32_t epilogue, void* C, int64_t ldc, const void* R, int64_t ldr, void* C2, int64_t ldc2,
               const float* rope_cos, const float* rope_sin, int32_t rope_cols, int32_t head_dim, int32_t seq,
               int32_t* status, void* stream) {
  mt::GemmArgs g;
  g.A = static_cast<const mt::bf16*>(A);
  g.lda = lda;
  g.B = static_cast<const mt::bf16*>(B);
  g.ldb = ldb;
  g.M = M;
  g.N = N;
  g.K = K;
  g.epi = epilogue;
  g.C = C;
  g.ldc = ldc;
  g.R = static_cast<const mt::bf16*>(R);
  g.ldr = ldr;
  g.C2 = static_cast<mt::bf16*>(C2);
  g.ldc2 = ldc2;
  g.rope_cos = rope_cos;
  g.rope_sin = rope_sin;
  g.rope_cols = rope_cols;
  g.head_dim = head_dim;
  g.seq = seq;
  g.status = status;
  if (!A || !B) return op_fail("gemm: null A or B");
  if (const char* e = mt::gemm_check(g)) return op_fail(e);
  return op_cuda(mt::launch_gemm(g, static_cast<cudaStream_t>(stream)), "gemm");
}

int mt_op_gemm_layout(const void* A, int64_t lda, const void* B, int64_t ldb, int32_t M, int32_t N, int32_t K,
                      int32_t layout, int32_t epilogue, void* C, int64_t ldc, const void* R, int64_t ldr,
                      int32_t* status, void* stream) {
  mt::GemmArgs g;
  g.A = static_cast<const mt::bf16*>(A);
  g.lda = lda;
  g.B = static_cast<const mt::bf16*>(B);
  g.ldb = ldb;
  g.M = M;
  g.N = N;
  g.K = K;
  g.a_mn = (layout & 1) != 0;
  g.b_mn = (layout & 2) != 0;
  g.epi = epilogue;
  g.C = C;
  g.ldc = ldc;
  g.R = static_cast<const mt::bf16*>(R);
  g.ldr = ldr;
  g.status = status;
  if (layout & ~3) return op_fail("gemm: layout must be a combination of MT_GEMM_A_MN and MT_GEMM_B_MN");
  if (epilogue == MT_EPI_SWIGLU || epilogue == MT_EPI_ROPE) return op_fail("gemm_layout: use mt_op_gemm for SwiGLU/RoPE");
  if (!A || !B) return op_fail("gemm: null A or B");
  if (const char* e = mt::gemm_check(g)) return op_fail(e);
  return op_cuda(mt::launch_gemm(g, static_cast<cudaStream_t>(stream)), "gemm");
}

int mt_op_gemm_grouped(const void* A, int64_t lda, const void* B, int64_t ldb, int32_t M, int32_t N, int32_t K,
                       int32_t layout, int32_t grouping, const int32_t* offsets, int32_t groups, int32_t epilogue,
                       void* C, int64_t ldc, const void* R, int64_t ldr, void* C2, int64_t ldc2, int32_t* status,
                       void* stream) {
  mt::GemmArgs g;
  g.A = static_cast<const mt::bf16*>(A);
  g.lda = lda;
  g.B = static_cast<const mt::bf16*>(B);
  g.ldb = ldb;
  g.M = M;
  g.N = N;
  g.K = K;
  g.a_mn = (layout & 1) != 0;
  g.b_mn = (layout & 2) != 0;
  g.epi = epilogue;
  g.C = C;
  g.ldc = ldc;
  g.R = static_cast<const mt::bf16*>(R);
  g.ldr = ldr;
  g.C2 = static_cast<mt::bf16*>(C2);
  g.ldc2 = ldc2;
  g.status = status;
  if (layout & ~3) return op_fail("gemm: layout must be a combination of MT_GEMM_A_MN and MT_GEMM_B_MN");
  if (!A || !B) return op_fail("gemm: null A or B");
  if (const char* e = mt::gemm_grouped_check(g, offsets, groups, grouping)) return op_fail(e);
  return op_cuda(mt::launch_gemm_grouped(g, offsets, groups, grouping, static_cast<cudaStream_t>(stream)),
                 "grouped gemm");
}

}  // extern "C"

extern "C" {

int mt_op_attention_fwd(const void* qkv, int64_t ldqkv, int32_t batch, int32_t seq, int32_t n_heads,
                        int32_t n_kv_heads, int32_t head_dim, void* o, int64_t ldo, float* lse, int32_t* status,
                        void* stream) {
  mt::AttnArgs a;
  a.qkv = static_cast<const mt::bf16*>(qkv);
  a.ldqkv = ldqkv;
  a.batch = batch;
  a.seq = seq;
  a.n_heads = n_heads;
  a.n_kv_heads = n_kv_heads;
  a.head_dim = head_dim;
  a.o = static_cast<mt::bf16*>(o);
  a.ldo = ldo;
  a.lse = lse;
  a.status = status;
  if (const char* e = mt::attn_check(a)) return op_fail(e);
  return op_cuda(mt::launch_attn_fwd(a, static_cast<cudaStream_t>(stream)), "attention forward");
}

int mt_op_attention_bwd(const void* qkv, int64_t ldqkv, int32_t batch, int32_t seq, int32_t n_heads,
                        int32_t n_kv_heads, int32_t head_dim, const void* o, int64_t ldo, const float* lse,
                        const void* dout, float* delta, void* dqkv, const float* rope_cos, const float* rope_sin,
                        int32_t* status, void* stream) {
  mt::AttnArgs a;
  a.qkv = static_cast<const mt::bf16*>(qkv);
  a.ldqkv = ldqkv;
  a.batch = batch;
  a.seq = seq;
  a.n_heads = n_heads;
  a.n_kv_heads = n_kv_heads;
  a.head_dim = head_dim;
  a.o = const_cast<mt::bf16*>(static_cast<const mt::bf16*>(o));
  a.ldo = ldo;
  a.lse = const_cast<float*>(lse);
  a.dout = static_cast<const mt::bf16*>(dout);
  a.delta = delta;
  a.dqkv = static_cast<mt::bf16*>(dqkv);
  a.rope_cos = rope_cos;
  a.rope_sin = rope_sin;
  a.status = status;
  if (const char* e = mt::attn_check(a)) return op_fail(e);
  if (!dout || !delta || !dqkv) return op_fail("attention backward: null dout, delta or dqkv");
  if ((reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(dqkv)) & 15)
    return op_fail("attention backward: dout and dqkv must be 16-byte aligned");
  if ((rope_cos == nullptr) != (rope_sin == nullptr)) return op_fail("attention backward: cos and sin go together");
  return op_cuda(mt::launch_attn_bwd(a, static_cast<cudaStream_t>(stream)), "attention backward");
}

int mt_op_rmsnorm_fwd(const void* x, const void* g, void* y, float* rstd, int64_t rows, int32_t d, float eps,
                      void* stream) {
  if (d <= 0 || d % 8) return op_fail("rmsnorm: d must be a positive multiple of 8");
  if (rows < 0 || rows > kMaxGridRows) return op_fail("rmsnorm: rows must be in 0 .. 2^31 - 1");
  if (rows > 0 && (!x || !g || !y || !rstd)) return op_fail("rmsnorm: null x, g, y or rstd");
  if (!al16(x) || !al16(g) || !al16(y)) return op_fail("rmsnorm: x, g and y must be 16-byte aligned");
  mt::launch_rmsnorm_fwd(static_cast<const mt::bf16*>(x), static_cast<const mt::bf16*>(g),
                         static_cast<mt::bf16*>(y), rstd, rows, d, eps, static_cast<cudaStream_t>(stream));
  return op_cuda(cudaPeekAtLastError() == cudaSuccess ? 0 : -1, "rmsnorm forward");
}

int64_t mt_op_rmsnorm_bwd_scratch_floats(int64_t rows, int32_t d) {
  if (rows < 0 || d <= 0) return -1;
  const int64_t parts = rows / mt::kRmsRowsPerBlock + (rows % mt::kRmsRowsPerBlock != 0);
  if (parts > INT64_MAX / d) return -1;
  return parts * (int64_t)d;
}

int mt_op_rmsnorm_bwd(const void* dy, const void* x, const void* g, const float* rstd, const void* dres, void* dx,
                      void* dg, float* scratch, int64_t rows, int32_t d, void* stream) {
  if (d <= 0 || d % 8 || rows < 0) return op_fail("rmsnorm: d must be a positive multiple of 8 and rows >= 0");
  if (!dg || (rows > 0 && (!dy || !x || !g || !rstd || !dx || !scratch)))
    return op_fail("rmsnorm backward: null dy, x, g, rstd, dx, dg or scratch");
  if (!al16(dy) || !al16(x) || !al16(g) || !al16(dres) || !al16(dx))
    return op_fail("rmsnorm backward: dy, x, g, dres and dx must be 16-byte aligned");
  if (d > mt::rmsnorm_bwd_max_d()) return op_fail("rmsnorm backward: d exceeds the widest row this device takes");
  auto s = static_cast<cudaStream_t>(stream);
  const long parts = mt::launch_rmsnorm_bwd(static_cast<const mt::bf16*>(dy), static_cast<const mt::bf16*>(x),
                                            static_cast<const mt::bf16*>(g), rstd,
                                            static_cast<const mt::bf16*>(dres), static_cast<mt::bf16*>(dx), scratch,
                                            rows, d, s);
  mt::launch_colsum_bf16(scratch, parts, d, static_cast<mt::bf16*>(dg), s);
  return op_cuda(cudaPeekAtLastError() == cudaSuccess ? 0 : -1, "rmsnorm backward");
}

int mt_op_flag_nonfinite(const void* p, int64_t n, int32_t* flag, void* stream) {
  if (n < 0 || !flag || (n > 0 && (!p || (reinterpret_cast<uintptr_t>(p) & 15))))
    return op_fail("flag_nonfinite: n >= 0, a flag and a 16-byte aligned p are required");
  mt::launch_flag_nonfinite(static_cast<const mt::bf16*>(p), n, flag, static_cast<cudaStream_t>(stream));
  return op_cuda(cudaPeekAtLastError() == cudaSuccess ? 0 : -1, "flag_nonfinite");
}

int mt_op_swiglu_bwd(const void* da, const void* gu, void* dgu, int64_t rows, int32_t f, void* stream) {
  if (f <= 0 || rows < 0) return op_fail("swiglu: f must be positive and rows >= 0");
  if (rows > 0 && (!da || !gu || !dgu)) return op_fail("swiglu: null da, gu or dgu");
  if (f % 8 == 0 && (!al16(da) || !al16(gu) || !al16(dgu)))
    return op_fail("swiglu: with f % 8 == 0, da, gu and dgu must be 16-byte aligned");
  mt::launch_swiglu_bwd(static_cast<const mt::bf16*>(da), static_cast<const mt::bf16*>(gu),
                        static_cast<mt::bf16*>(dgu), rows, f, static_cast<cudaStream_t>(stream));
  return op_cuda(cudaPeekAtLastError() == cudaSuccess ? 0 : -1, "swiglu backward");
}

int mt_op_transpose(const void* src, int64_t rows, int64_t cols, int64_t lds, void* dst, int64_t ldd,
                    void* stream) {
  if (rows < 0 || cols < 0 || lds < cols || ldd < rows) return op_fail("transpose: bad shape or leading dimension");
  if (rows > 0 && cols > 0 && (!src || !dst)) return op_fail("transpose: null src or dst");
  mt::launch_transpose(static_cast<const mt::bf16*>(src), rows, cols, lds, static_cast<mt::bf16*>(dst), ldd,
                       static_cast<cudaStream_t>(stream));
  return op_cuda(cudaPeekAtLastError() == cudaSuccess ? 0 : -1, "transpose");
}

int mt_op_cross_entropy(const float* z, int64_t rows, int32_t vocab, const int32_t* tgt, float inv_n, void* dz,
                        float* loss_rows, int32_t* status, void* stream) {
  if (vocab <= 0) return op_fail("cross entropy: vocab must be positive");
  if (rows < 0 || rows > kMaxGridRows) return op_fail("cross entropy: rows must be in 0 .. 2^31 - 1");
  if (rows > 0 && (!z || !tgt || !dz || !loss_rows)) return op_fail("cross entropy: null z, tgt, dz or loss_rows");
  if (!al16(z) || !al16(dz)) return op_fail("cross entropy: z and dz must be 16-byte aligned");
  mt::launch_cross_entropy(z, rows, vocab, tgt, inv_n, static_cast<mt::bf16*>(dz), loss_rows, status,
                           static_cast<cudaStream_t>(stream));
  return op_cuda(cudaPeekAtLastError() == cudaSuccess ? 0 : -1, "cross entropy");
}

int mt_op_embedding_fwd(const int32_t* tok, const void* E, void* x, int64_t T, int32_t d, int32_t V,
                        int32_t* status, void* stream) {
  if (d <= 0 || d % 8 || V <= 0) return op_fail("embedding: d must be a positive multiple of 8 and V positive");
  if (T < 0 || T > kMaxGridRows) return op_fail("embedding: T must be in 0 .. 2^31 - 1");
  if (T > 0 && (!tok || !E || !x)) return op_fail("embedding: null tok, E or x");
  if (!al16(E) || !al16(x)) return op_fail("embedding: E and x must be 16-byte aligned");
  mt::launch_embed_fwd(tok, static_cast<const mt::bf16*>(E), static_cast<mt::bf16*>(x), T, d, V, status,
                       static_cast<cudaStream_t>(stream));
  return op_cuda(cudaPeekAtLastError() == cudaSuccess ? 0 : -1, "embedding forward");
}

int mt_op_embedding_bwd(const int32_t* row_offsets, const int32_t* positions, const void* dx, void* dE, int32_t V,
                        int32_t d, void* stream) {
  if (d <= 0 || d % 8 || V <= 0) return op_fail("embedding: d must be a positive multiple of 8 and V positive");
  if (!row_offsets || !positions || !dx || !dE) return op_fail("embedding backward: null pointer");
  if (!al16(dx) || !al16(dE)) return op_fail("embedding backward: dx and dE must be 16-byte aligned");
  mt::launch_embed_bwd(row_offsets, positions, static_cast<const mt::bf16*>(dx), static_cast<mt::bf16*>(dE), V, d,
                       static_cast<cudaStream_t>(stream));
  return op_cuda(cudaPeekAtLastError() == cudaSuccess ? 0 : -1, "embedding backward");
}

int mt_op_wait_probe(int32_t* status, int64_t limit_ns, void* stream) {
  if (!status || limit_ns < 1000000 || limit_ns > 5000000000LL)
    return op_fail("wait probe: status required, limit between 1 ms and 5 s");
  return op_cuda(mt::launch_wait_probe(status, (uint64_t)limit_ns, static_cast<cudaStream_t>(stream)), "wait probe");
}

int64_t mt_op_moe_sort_scratch_ints(int64_t P, int32_t E) { return mt::moe_sort_scratch_ints(P, E); }

int64_t mt_op_moe_rows_capacity(int64_t P, int32_t E, int32_t row_align) {
  if (P < 0 || E < 1 || row_align < 1 || row_align > 256) return -1;
  return mt::moe_rows_capacity(P, E, row_align);
}

int mt_op_moe_route(const float* logits, int64_t N, int32_t E, int32_t k, int32_t row_align, int32_t* idx,
                    float* gates, int32_t* order, int32_t* pos, int32_t* offsets, int32_t* scratch, void* stream) {
  if (const char* e = mt::moe_check(N, E, k, 8)) return op_fail(e);
  if (row_align < 1 || row_align > 256) return op_fail("moe route: row_align must be in 1 .. 256");
  if (!logits || !idx || !gates || !order || !pos || !offsets || !scratch) return op_fail("moe route: null pointer");
  auto s = static_cast<cudaStream_t>(stream);
  if (mt::launch_moe_topk(logits, N, E, k, idx, gates, s)) return op_cuda(-4, "moe top-k");
  return op_cuda(mt::launch_moe_sort(idx, N * k, E, row_align, scratch, order, pos, offsets, s), "moe sort");
}

int mt_op_moe_zero_pads(const int32_t* order, int64_t P_rows, int32_t d, void* buf, void* stream) {
  if (P_rows <= 0 || d <= 0 || d % 8 || !order || !buf) return op_fail("moe zero pads: bad shape");
  if (!al16(buf)) return op_fail("moe zero pads: buf must be 16-byte aligned");
  return op_cuda(mt::launch_moe_zero_pads(order, P_rows, d, static_cast<mt::bf16*>(buf),
                                          static_cast<cudaStream_t>(stream)),
                 "moe zero pads");
}

int mt_op_moe_gather(const void* x, int64_t ldx, const int32_t* order, int32_t k, int64_t P, int32_t d, void* xp,
                     void* stream) {
  if (P <= 0 || k < 1 || d <= 0 || d % 8 || ldx % 8 || ldx < d) return op_fail("moe gather: bad shape");
  if (!x || !order || !xp) return op_fail("moe gather: null x, order or xp");
  if (!al16(x) || !al16(xp)) return op_fail("moe gather: x and xp must be 16-byte aligned");
  return op_cuda(mt::launch_moe_gather(static_cast<const mt::bf16*>(x), ldx, order, k, P, d,
                                       static_cast<mt::bf16*>(xp), static_cast<cudaStream_t>(stream)),
                 "moe gather");
}

int mt_op_moe_combine(const void* yp, const int32_t* pos, const float* gates, int64_t N, int32_t k, int32_t d,
                      const void* res, void* out, void* stream) {
  if (const char* e = mt::moe_check(N, k, k, d)) return op_fail(e);
  if (!yp || !pos || !gates || !out) return op_fail("moe combine: null yp, pos, gates or out");
  return op_cuda(mt::launch_moe_combine(static_cast<const mt::bf16*>(yp), pos, gates, N, k, d,
                                        static_cast<const mt::bf16*>(res), static_cast<mt::bf16*>(out),
                                        static_cast<cudaStream_t>(stream)),
                 "moe combine");
}

int mt_op_moe_combine_bwd(const void* dy, const void* yp, const int32_t* pos, const float* gates, int64_t N, int32_t k,
                          int32_t d, void* dyp, float* dgates, void* stream) {
  if (const char* e = mt::moe_check(N, k, k, d)) return op_fail(e);
  if (!dy || !yp || !pos || !gates || !dyp || !dgates) return op_fail("moe combine backward: null pointer");
  return op_cuda(mt::launch_moe_combine_bwd(static_cast<const mt::bf16*>(dy), static_cast<const mt::bf16*>(yp), pos,
                                            gates, N, k, d, static_cast<mt::bf16*>(dyp), dgates,
                                            static_cast<cudaStream_t>(stream)),
                 "moe combine backward");
}

int mt_op_moe_gate_bwd(const int32_t* idx, const float* gates, const float* dgates, int64_t N, int32_t E, int32_t k,
                       void* ds, void* stream) {
  if (const char* e = mt::moe_check(N, E, k, 8)) return op_fail(e);
  if (!idx || !gates || !dgates || !ds) return op_fail("moe gate backward: null pointer");
  return op_cuda(mt::launch_moe_gate_bwd(idx, gates, dgates, N, E, k, static_cast<mt::bf16*>(ds),
                                         static_cast<cudaStream_t>(stream)),
                 "moe gate backward");
}

int mt_op_moe_scatter_bwd(const void* dxp, const int32_t* pos, int64_t N, int32_t k, int32_t d, const void* dres,
                          void* dx, void* stream) {
  if (const char* e = mt::moe_check(N, k, k, d)) return op_fail(e);
  if (!dxp || !pos || !dx) return op_fail("moe scatter backward: null dxp, pos or dx");
  return op_cuda(mt::launch_moe_scatter_bwd(static_cast<const mt::bf16*>(dxp), pos, N, k, d,
                                            static_cast<const mt::bf16*>(dres), static_cast<mt::bf16*>(dx),
                                            static_cast<cudaStream_t>(stream)),
                 "moe scatter backward");
}

}  // extern "C"
