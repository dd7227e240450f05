/*
 * mt_ops.h -- per-kernel C-ABI of libmt.so (device pointers, no allocation).
 *
 * These entry points expose the individual sm_103a kernels that the training
 * step (mt.h) chains together, so that each can be checked on its own.  All
 * pointers are DEVICE pointers owned by the caller; `stream` is a
 * cudaStream_t passed as void* (NULL = legacy default stream).  Calls are
 * asynchronous: they enqueue work and return.  Arguments are validated on the
 * host: an unsupported shape, alignment or mode returns MT_EINVAL before
 * anything is launched, with the reason in mt_op_last_error() (per thread).
 * Buffers the kernels move in 16-byte vectors must be 16-byte aligned (the
 * RMSNorm rows and gain, the SwiGLU buffers when f % 8 == 0, the embedding
 * table and rows, cross-entropy's z and dz, the attention buffers, the GEMM
 * operands).  The elementwise kernels (RMSNorm, SwiGLU, transpose,
 * cross-entropy, embedding forward) take zero rows or tokens: they launch
 * nothing over rows and return MT_OK, and their row buffers may then be NULL
 * (RMSNorm's gain gradient dg [d] is still written, as zeros).  GEMM and
 * attention take non-empty shapes only.  Row counts that index the grid (one
 * CTA per row) must be below 2^31.
 * A launch failure returns MT_ECUDA.  Kernels that can detect a problem at
 * run time (a bounded wait that expired, a token id out of range) write a
 * nonzero code into *status (device int, first error sticks) when `status`
 * is not NULL.
 */
#ifndef MT_OPS_H
#define MT_OPS_H
#include <stdint.h>

#include "mt.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Epilogue modes of mt_op_gemm. */
enum {
  MT_EPI_STORE_BF16 = 0,   /* C = acc (BF16) */
  MT_EPI_RESIDUAL_BF16 = 1,/* C = R + acc (BF16; R has C's shape) */
  MT_EPI_F32 = 2,          /* C = acc (FP32) */
  MT_EPI_F32_ACCUMULATE = 3,/* C += acc (FP32) */
  MT_EPI_SWIGLU = 4,       /* columns (2j, 2j+1) are (gate, up): C[:, j] = silu(gate)*up (BF16, N/2 cols);
                              C2, when not NULL, receives the BF16 gate/up values themselves */
  MT_EPI_ROPE = 5,         /* C = acc (BF16) with rotate-half RoPE applied to columns < rope_cols,
                              heads of head_dim columns, position = row % seq */
  MT_EPI_SWIGLU_BWD = 6    /* acc = da, the gradient of a = silu(gate) * up (N columns); R = the BF16
                              (gate, up) pairs [M, 2N] interleaved; C (BF16, [M, 2N]) receives
                              (da * up * silu'(gate), da * silu(gate)) at columns (2j, 2j+1) */
};

const char* mt_op_last_error(void);

/*
 * C[M, N] = epilogue(A[M, K] * B[N, K]^T), BF16 operands, FP32 accumulation
 * on the tcgen05 tensor cores.  The decoder's projections are nn.Linear
 * weights [out, in] (MegaTrain page summaries: dense Llama-style layers whose
 * weights stream per layer), so y = x W^T is mt_op_gemm(A=x, B=W).
 * Requirements: K % 8 == 0, lda/ldb/ldc/ldr/ldc2 % 8 == 0, all base pointers
 * 16-byte aligned; row-major with the given leading dimensions (elements).
 */
int mt_op_gemm(const void* A, int64_t lda, const void* B, int64_t ldb, int32_t M, int32_t N, int32_t K,
               int32_t epilogue, void* C, int64_t ldc, const void* R, int64_t ldr, void* C2, int64_t ldc2,
               const float* rope_cos, const float* rope_sin, int32_t rope_cols, int32_t head_dim, int32_t seq,
               int32_t* status, void* stream);


/* Operand layouts of mt_op_gemm_layout. */
enum { MT_GEMM_A_MN = 1, /* A stored [K, M] (M contiguous), leading dimension lda >= M */
       MT_GEMM_B_MN = 2  /* B stored [K, N] (N contiguous), leading dimension ldb >= N */ };

/*
 * mt_op_gemm with either operand stored MN-major, read as such by the tensor
 * cores (no transpose pass): the backward GEMMs of a linear layer,
 * dW = dY^T X (both operands MN-major) and dX = dY W (B MN-major).
 * Epilogues MT_EPI_STORE_BF16, MT_EPI_RESIDUAL_BF16, MT_EPI_F32,
 * MT_EPI_F32_ACCUMULATE.  Same alignment rules as mt_op_gemm.
 */
int mt_op_gemm_layout(const void* A, int64_t lda, const void* B, int64_t ldb, int32_t M, int32_t N, int32_t K,
                      int32_t layout, int32_t epilogue, void* C, int64_t ldc, const void* R, int64_t ldr,
                      int32_t* status, void* stream);

/* Groupings of mt_op_gemm_grouped. */
enum { MT_GEMM_GROUP_ROWS = 1, MT_GEMM_GROUP_K = 2 };

/*
 * One launch for a GEMM per group (the experts of a mixture-of-experts layer)
 * whose sizes are only known on the device: offsets (device int32
 * [groups + 1], non-decreasing, groups 1..256) give each group's first row of
 * a shared buffer.  No host synchronisation.  Values outside the operand are
 * clamped to it, so no offsets can make the kernel read or write out of
 * bounds.
 *
 * MT_GEMM_GROUP_ROWS (layout 0 or MT_GEMM_B_MN): for every group g and row r
 *   in offsets[g] .. offsets[g+1]:  C[r] = epilogue(A[r] B_g^T).
 *   A [M, K] K-major (M = the buffer's rows, all groups); B_g is group g's
 *   block of a stacked B: rows g*N .. g*N + N of a K-major [groups*N, K] B, or
 *   (MT_GEMM_B_MN) rows g*K .. g*K + K of a [groups*K, N] B.  C, R, C2 have
 *   A's rows.  Epilogues MT_EPI_STORE_BF16, MT_EPI_F32, MT_EPI_F32_ACCUMULATE,
 *   MT_EPI_SWIGLU (C2 optional), MT_EPI_SWIGLU_BWD.
 * MT_GEMM_GROUP_K (layout MT_GEMM_A_MN | MT_GEMM_B_MN): for every group g,
 *   C[g*M .. g*M + M) = A_g^T B_g, where A is stored [K, M], B stored [K, N]
 *   (K = the buffer's rows, all groups) and A_g, B_g are their rows
 *   offsets[g] .. offsets[g+1].  Each group's row count must be a multiple
 *   of 64 (pad with zero rows: mt_op_moe_route with row_align 64); a group
 *   without rows gets a zero block.  Epilogues MT_EPI_STORE_BF16, MT_EPI_F32,
 *   MT_EPI_F32_ACCUMULATE.  This is the weight gradient of every expert in
 *   one launch.
 * Alignment rules as mt_op_gemm.  Errors: MT_EINVAL for unsupported
 * arguments (nothing launched), MT_ECUDA for a failed launch.
 */
int mt_op_gemm_grouped(const void* A, int64_t lda, const void* B, int64_t ldb, int32_t M, int32_t N, int32_t K,
                       int32_t layout, int32_t grouping, const int32_t* offsets, int32_t groups, int32_t epilogue,
                       void* C, int64_t ldc, const void* R, int64_t ldr, void* C2, int64_t ldc2, int32_t* status,
                       void* stream);

/*
 * Causal grouped-query attention forward (flash style, one pass over keys).
 * qkv: [batch*seq, ldqkv] BF16 rows (token t = b*seq + s) holding n_heads query
 * heads, then n_kv_heads key heads, then n_kv_heads value heads, head_dim
 * columns each (q, k already rotated).  Query head h reads kv head
 * h*n_kv_heads/n_heads.  o: [batch*seq, ldo] BF16; lse: FP32
 * [batch, n_heads, seq] natural-log log-sum-exp of each score row (scores
 * scaled by 1/sqrt(head_dim)).  head_dim 64 or 128; n_heads % n_kv_heads == 0;
 * batch, seq > 0; ldqkv, ldo multiples of 8 and at least the row widths;
 * qkv and o 16-byte aligned (TMA); otherwise MT_EINVAL before any launch.
 * A wait inside the kernel that runs out writes a nonzero code to *status.
 */
int mt_op_attention_fwd(const void* qkv, int64_t ldqkv, int32_t batch, int32_t seq, int32_t n_heads,
                        int32_t n_kv_heads, int32_t head_dim, void* o, int64_t ldo, float* lse, int32_t* status,
                        void* stream);

/*
 * Attention backward: given o, lse from the forward and dout (layout of o),
 * writes dqkv (layout of qkv) = gradients w.r.t. q, k, v.  delta: FP32 scratch
 * [batch, n_heads, seq] (overwritten).  When rope_cos/rope_sin ([seq,
 * head_dim/2] FP32) are given, dq and dk are passed back through the inverse
 * rotate-half rotation (gradient w.r.t. the unrotated projections).
 * Deterministic: no atomics, fixed accumulation order.  The forward's
 * argument rules apply, and dout and dqkv must be non-null and 16-byte
 * aligned, delta non-null, rope_cos and rope_sin both given or both NULL;
 * otherwise MT_EINVAL before any launch.
 */
int mt_op_attention_bwd(const void* qkv, int64_t ldqkv, int32_t batch, int32_t seq, int32_t n_heads,
                        int32_t n_kv_heads, int32_t head_dim, const void* o, int64_t ldo, const float* lse,
                        const void* dout, float* delta, void* dqkv, const float* rope_cos, const float* rope_sin,
                        int32_t* status, void* stream);

/* y = x * rsqrt(mean(x^2) + eps) * g over rows of d (d % 8 == 0); rstd: FP32 [rows]. */
int mt_op_rmsnorm_fwd(const void* x, const void* g, void* y, float* rstd, int64_t rows, int32_t d, float eps,
                      void* stream);
/* FP32 scratch elements mt_op_rmsnorm_bwd needs: ceil(rows/64) * d; -1 when
 * rows < 0, d <= 0 or the product does not fit in int64. */
int64_t mt_op_rmsnorm_bwd_scratch_floats(int64_t rows, int32_t d);
/*
 * dx = dres + d(rmsnorm)/dx^T dy (dres may be NULL); dg [d] BF16 = sum over rows
 * of dy * x * rstd, reduced in a fixed order (per block of rows, then over the
 * blocks).  d % 8 == 0; rows wider than 8192 keep d floats in shared memory per
 * block, so d beyond what the device's shared memory holds (about 58K on this
 * part) returns MT_EINVAL.
 */
int mt_op_rmsnorm_bwd(const void* dy, const void* x, const void* g, const float* rstd, const void* dres, void* dx,
                      void* dg, float* scratch, int64_t rows, int32_t d, void* stream);
/* SwiGLU backward on interleaved (gate, up) columns: gu, dgu [rows, 2f]; da [rows, f]. */
int mt_op_swiglu_bwd(const void* da, const void* gu, void* dgu, int64_t rows, int32_t f, void* stream);
/* dst[c, r] = src[r, c] (BF16). */
int mt_op_transpose(const void* src, int64_t rows, int64_t cols, int64_t lds, void* dst, int64_t ldd,
                    void* stream);
/*
 * Row-wise cross-entropy of FP32 logits z [rows, vocab] against tgt [rows]:
 * loss_rows[r] = logsumexp(z_r) - z_r[tgt_r]; dz (BF16) = (softmax(z_r) -
 * onehot(tgt_r)) * inv_n.  An out-of-range target sets *status.
 */
int mt_op_cross_entropy(const float* z, int64_t rows, int32_t vocab, const int32_t* tgt, float inv_n, void* dz,
                        float* loss_rows, int32_t* status, void* stream);
/* x[t] = E[tok[t]] ([V, d] BF16); out-of-range ids give zeros and set *status. */
int mt_op_embedding_fwd(const int32_t* tok, const void* E, void* x, int64_t T, int32_t d, int32_t V,
                        int32_t* status, void* stream);
/*
 * dE[v] = sum of dx[positions[k]] for k in [row_offsets[v], row_offsets[v+1])
 * in ascending k, for every v < V (rows with no token become zero): a
 * deterministic scatter-add given the token positions grouped by id.
 */
int mt_op_embedding_bwd(const int32_t* row_offsets, const int32_t* positions, const void* dx, void* dE, int32_t V,
                        int32_t d, void* stream);

/*
 * RMSNorm backward that allocates nothing (no counterpart in the MegaTrain
 * pages: it exists for callers of this library).  Same inputs, outputs and
 * results as mt_op_rmsnorm_bwd, but without the caller-provided scratch
 * buffer.  It is meant for callers that cannot allocate device memory: code
 * embedded in a host application that reserves the GPU's memory budget up
 * front and forbids further allocation, or latency-critical loops where a
 * cudaMalloc/cudaFree (which can synchronise the device) is not acceptable.
 *
 * The gain-gradient partial sums go to a fixed array in the library's own
 * device memory (16 MiB, 4,194,304 floats) that every GPU loading the library
 * keeps until the process exits.  The call requires ceil(rows/64) * d <=
 * 4,194,304 and d within mt_op_rmsnorm_bwd's limit, and returns MT_EINVAL
 * otherwise, before launching anything (message in mt_op_last_error()).
 * It calls no cudaMalloc, cudaFree or allocating library routine.  The first
 * call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  All calls share the one array: each overwrites
 * the part it reads, but calls that overlap on the GPU (other streams, or
 * other host threads without ordering) race and must be serialised.
 */
int mt_op_rmsnorm_bwd_noalloc(const void* dy, const void* x, const void* g, const float* rstd, const void* dres,
                              void* dx, void* dg, int64_t rows, int32_t d, void* stream);

/*
 * Failure-detection probe.  Every spin-wait in the library's kernels is
 * bounded by %globaltimer and, on expiry, records a code in the kernel's
 * device status word and returns instead of hanging (a context that stays
 * usable).  This probe exercises that path on purpose: one warp waits, for
 * limit_ns (1 ms .. 5 s), on an mbarrier that nothing arrives on, then writes
 * MT_STATUS_WAIT_PROBE (7) into *status (device int32, first error sticks)
 * and exits.  MT_EINVAL for a null status or a limit out of range.
 */
enum { MT_STATUS_WAIT_PROBE = 7 };
int mt_op_wait_probe(int32_t* status, int64_t limit_ns, void* stream);

/*
 * *flag = 1 if any of the n BF16 values at p (16-byte aligned) is NaN or Inf;
 * *flag is left as it is otherwise (the caller zeroes it).  The device check
 * behind MT_DIRECT_GRADS (no counterpart in the pages: their host copy of each
 * gradient slab is where a non-finite value would be seen).
 */
int mt_op_flag_nonfinite(const void* p, int64_t n, int32_t* flag, void* stream);

/*
 * Mixture-of-experts MLP pieces (the expert GEMMs run on mt_op_gemm_grouped,
 * or mt_op_gemm / mt_op_gemm_layout over each expert's rows).  MegaTrain's
 * largest run trains an MoE model (author's blog, the single-H200 gpt-oss
 * 120B run; podcast transcript, the 120B GPT-OSS run); the pages give no
 * formula for the MoE layer, so this is the plainest top-k reading.  N
 * tokens, E experts (1..256),
 * top k (1..min(8, E)), pairs p = n*k + j (P = N*k), d a multiple of 8.
 * Routing: per token the k largest router logits (ties to the lower expert
 * id), gates = softmax over them; the pairs are then sorted by expert, stably.
 *
 * mt_op_moe_route: logits FP32 [N, E] -> idx int32 [N, k], gates FP32 [N, k],
 *   order int32 [R] (pair at each position, -1 at padding), pos int32 [P]
 *   (position of each pair), offsets int32 [E + 1] (first position of each
 *   expert; offsets[E] = the positions used); scratch:
 *   mt_op_moe_sort_scratch_ints(P, E) int32 values.  Each expert's positions
 *   are padded to a multiple of row_align (1..256; 1 = no padding, R = P; 64
 *   for the grouped weight-gradient GEMM); R = mt_op_moe_rows_capacity(P, E,
 *   row_align) = P + (row_align - 1) E.
 * mt_op_moe_gather: xp[i] = x[order[i] / k] for i < P rows (BF16 rows, x rows
 *   ldx apart), a zero row where order[i] = -1.
 * mt_op_moe_zero_pads: buf[i] = 0 for the rows i < P_rows with order[i] = -1.
 * mt_op_moe_combine: out[n] = res[n] + sum_j gates[n, j] yp[pos[n k + j]]
 *   (BF16 rows, FP32 sums in slot order; res may be NULL).
 * mt_op_moe_combine_bwd: dyp[pos[p]] = gates[p] dy[n] (BF16),
 *   dgates[p] = <dy[n], yp[pos[p]]> (FP32).
 * mt_op_moe_gate_bwd: ds [N, E] BF16 = softmax backward over the selected
 *   logits (g_j (dg_j - sum_i g_i dg_i) at the selected experts, 0 elsewhere).
 * mt_op_moe_scatter_bwd: dx[n] = dres[n] + sum_j dxp[pos[n k + j]] (dres may be NULL).
 */
int64_t mt_op_moe_sort_scratch_ints(int64_t P, int32_t E);
int64_t mt_op_moe_rows_capacity(int64_t P, int32_t E, int32_t row_align);
int mt_op_moe_route(const float* logits, int64_t N, int32_t E, int32_t k, int32_t row_align, int32_t* idx,
                    float* gates, int32_t* order, int32_t* pos, int32_t* offsets, int32_t* scratch, void* stream);
int mt_op_moe_zero_pads(const int32_t* order, int64_t P_rows, int32_t d, void* buf, void* stream);
int mt_op_moe_gather(const void* x, int64_t ldx, const int32_t* order, int32_t k, int64_t P, int32_t d, void* xp,
                     void* stream);
int mt_op_moe_combine(const void* yp, const int32_t* pos, const float* gates, int64_t N, int32_t k, int32_t d,
                      const void* res, void* out, void* stream);
int mt_op_moe_combine_bwd(const void* dy, const void* yp, const int32_t* pos, const float* gates, int64_t N, int32_t k,
                          int32_t d, void* dyp, float* dgates, void* stream);
int mt_op_moe_gate_bwd(const int32_t* idx, const float* gates, const float* dgates, int64_t N, int32_t E, int32_t k,
                       void* ds, void* stream);
int mt_op_moe_scatter_bwd(const void* dxp, const int32_t* pos, int64_t N, int32_t k, int32_t d, const void* dres,
                          void* dx, void* stream);

#ifdef __cplusplus
}
#endif
#endif
