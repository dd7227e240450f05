// Launch interfaces of the sm_103a kernels that make up one decoder layer's
// forward, recompute and backward, plus the embedding and LM-head steps.
// All tensors are row-major; BF16 unless stated; `rows` counts tokens.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace mt {

using bf16 = __nv_bfloat16;

// Device status word codes (the first error sticks: written with atomicCAS).
enum : int {
  kStatusOk = 0,
  kStatusGemmTimeout = 1,
  kStatusAttnBadShape = 2,
  kStatusIndexOutOfRange = 3,
  kStatusNonFinite = 4,
  kStatusAttnFwdTimeout = 5,
  kStatusAttnBwdTimeout = 6,
  kStatusWaitProbe = 7,  // the wait probe's bounded wait ran out (its expected outcome)
};

// Failure-detection probe: one warp waits, bounded by limit_ns of
// %globaltimer, on an mbarrier that nothing arrives on, then records
// kStatusWaitProbe in *status and exits.
int launch_wait_probe(int* status, uint64_t limit_ns, cudaStream_t s);

// ----------------------------------------------------------------- GEMM
enum EpiMode : int {
  kEpiStoreBf16 = 0,      // C(bf16) = acc
  kEpiResidualBf16 = 1,   // C(bf16) = R + acc
  kEpiF32 = 2,            // C(f32) = acc
  kEpiF32Accumulate = 3,  // C(f32) += acc
  kEpiSwiGLU = 4,         // columns (2j, 2j+1) = (gate, up): C[:, j] = silu(gate) * up; C2 = gu (optional)
  kEpiRope = 5,           // C(bf16) = acc, rotate-half RoPE on columns < rope_cols
  kEpiSwiGLUBwd = 6,      // acc = da[:, j]; R = gu [M, 2N] (gate, up interleaved); C[:, 2j | 2j+1] = (dgate, dup)
};

struct GemmArgs {
  const bf16* A = nullptr;  // [M, K] (a_mn: stored [K, M]), leading dimension lda
  long lda = 0;
  const bf16* B = nullptr;  // [N, K] (b_mn: stored [K, N]), leading dimension ldb
  long ldb = 0;
  bool a_mn = false, b_mn = false;
  int M = 0, N = 0, K = 0;
  int epi = kEpiStoreBf16;
  void* C = nullptr;
  long ldc = 0;
  const bf16* R = nullptr;
  long ldr = 0;
  bf16* C2 = nullptr;
  long ldc2 = 0;
  const float* rope_cos = nullptr;  // [seq, head_dim/2]
  const float* rope_sin = nullptr;
  int rope_cols = 0;
  int head_dim = 0;
  int seq = 1;
  int* status = nullptr;
};

// 0 when the launches just issued succeeded; otherwise -4, keeping the CUDA
// error's text for last_launch_error() (thread-local).
int launch_result();
const char* last_launch_error();

// Returns a message when the arguments are unsupported, else nullptr.
const char* gemm_check(const GemmArgs& g);
// 0 on success; negative on a launch or descriptor error.
int launch_gemm(const GemmArgs& g, cudaStream_t stream);

// Grouped GEMM: one launch for a GEMM per group (the experts of an MoE layer)
// whose row counts live on the device, offsets [groups + 1] (int32, first row
// of each group, non-decreasing; values are clamped to the operand).
//   kGemmGroupRows  C[r] = epi(A[r] B_g^T) for r in offsets[g] .. offsets[g+1]:
//                   A [M, K] K-major holds every group's rows; B is group-
//                   stacked, [groups * N, K] K-major or [groups * K, N]
//                   MN-major; C (and R, C2) rows are A's rows.
//   kGemmGroupK     C[g*M .. g*M + M) = A_g^T B_g with A stored [K, M] and B
//                   stored [K, N] (both MN-major), A_g and B_g their rows
//                   offsets[g] .. offsets[g+1]; every group's row count is a
//                   multiple of 64 (zero rows as padding); an empty group's C
//                   block is zero.
enum GemmGroup : int { kGemmGroupRows = 1, kGemmGroupK = 2 };
const char* gemm_grouped_check(const GemmArgs& g, const int32_t* offsets, int groups, int mode);
int launch_gemm_grouped(const GemmArgs& g, const int32_t* offsets, int groups, int mode, cudaStream_t stream);

// ----------------------------------------------------------------- attention
struct AttnArgs {
  const bf16* qkv = nullptr;  // [B*S, ldqkv]: q heads, then k heads, then v heads (head_dim each)
  long ldqkv = 0;
  int batch = 0, seq = 0, n_heads = 0, n_kv_heads = 0, head_dim = 0;
  bf16* o = nullptr;  // [B*S, ldo], head h at column h*head_dim
  long ldo = 0;
  float* lse = nullptr;  // [B, n_heads, S] natural-log row sums of exp(scores)
  // backward
  const bf16* dout = nullptr;  // dO, layout of o
  float* delta = nullptr;      // [B, n_heads, S] scratch: rowsum(dO * O)
  bf16* dqkv = nullptr;        // gradient w.r.t. the rotated q, k and v, layout of qkv
  // rotate-half RoPE tables [seq, head_dim/2]; when set, the backward applies
  // the inverse rotation so dqkv holds gradients w.r.t. the unrotated q, k.
  const float* rope_cos = nullptr;
  const float* rope_sin = nullptr;
  int* status = nullptr;
};
const char* attn_check(const AttnArgs& a);
int launch_attn_fwd(const AttnArgs& a, cudaStream_t stream);
// tcgen05/TMEM forward (attention_tc.cu); same contract as launch_attn_fwd.
int launch_attn_fwd_tc(const AttnArgs& a, cudaStream_t stream);
// tcgen05/TMEM backward: dK/dV then dQ (attention_tc.cu); delta must already hold rowsum(dO * O).
int launch_attn_bwd_tc_main(const AttnArgs& a, cudaStream_t stream);
int launch_attn_bwd(const AttnArgs& a, cudaStream_t stream);

// ----------------------------------------------------------------- elementwise
// y = x * rsqrt(mean(x^2) + eps) * g ; rstd[r] saved for the backward.
void launch_rmsnorm_fwd(const bf16* x, const bf16* g, bf16* y, float* rstd, long rows, int d, float eps,
                        cudaStream_t s);
// dx = dres + rstd * (dy*g - xhat * mean(dy*g*xhat)), xhat = x*rstd.
// dg_partial[blk, d] = sum over the rows of block blk of dy * xhat; returns
// the number of blocks (partial rows), at most ceil(rows / kRmsRowsPerBlock)
// (the scratch callers provide); reduce them with launch_colsum_bf16.
constexpr int kRmsRowsPerBlock = 64;
long launch_rmsnorm_bwd(const bf16* dy, const bf16* x, const bf16* g, const float* rstd, const bf16* dres,
                        bf16* dx, float* dg_partial, long rows, int d, cudaStream_t s);
// Largest d the backward launches on this device (its shared-memory plan for
// d > 8192 keeps d floats per block).
long rmsnorm_bwd_max_d();
// out[c] = bf16(sum_p partial[p, c]) in a fixed order.
void launch_colsum_bf16(const float* partial, long nparts, int d, bf16* out, cudaStream_t s);
// gu [rows, 2f] interleaved (gate, up); da [rows, f] -> dgu [rows, 2f] interleaved.
void launch_swiglu_bwd(const bf16* da, const bf16* gu, bf16* dgu, long rows, int f, cudaStream_t s);
// dst[c, r] = src[r, c]
void launch_transpose(const bf16* src, long rows, long cols, long lds, bf16* dst, long ldd, cudaStream_t s);
// x[t] = E[tok[t]]; out-of-range ids set status and produce zeros.
void launch_embed_fwd(const int32_t* tok, const bf16* E, bf16* x, long T, int d, int V, int* status,
                      cudaStream_t s);
// dE[v] = sum over t in pos[off[v] .. off[v+1]) of dx[t] (ascending t), zeros elsewhere.
// Compact embedding gradient: out[u] = sum of dx rows of token id rows[u], u < U.
void launch_embed_bwd_rows(const int32_t* off, const int32_t* pos, const int32_t* rows, int U, const bf16* dx,
                           bf16* out, int d, cudaStream_t s);
void launch_embed_bwd(const int32_t* off, const int32_t* pos, const bf16* dx, bf16* dE, int V, int d,
                      cudaStream_t s);
// Row-wise cross-entropy on FP32 logits z [rows, V]:
// loss_rows[r] = logsumexp(z_r) - z_r[tgt_r];  dz_r = (softmax(z_r) - onehot(tgt_r)) * inv_n  (bf16)
void launch_cross_entropy(const float* z, long rows, int V, const int32_t* tgt, float inv_n, bf16* dz,
                          float* loss_rows, int* status, cudaStream_t s);
// out[0] = sum(loss_rows[0..n)) * inv_n, fixed-order reduction.
void launch_mean_loss(const float* loss_rows, long n, float inv_n, float* out, cudaStream_t s);
void launch_f32_to_bf16(const float* src, bf16* dst, long n, cudaStream_t s);
void launch_zero(void* p, size_t bytes, cudaStream_t s);
// status |= kStatusNonFinite when any of the n BF16 values is NaN or Inf.
void launch_check_finite(const bf16* p, long n, int* status, cudaStream_t s);
// *flag = 1 if any of the n values is NaN or Inf (p 16-byte aligned).
void launch_flag_nonfinite(const bf16* p, long n, int* flag, cudaStream_t s);

// ----------------------------------------------------------------- mixture of experts (moe.cu)
// N tokens, E experts (<= 256), top k (<= 8), pairs p = n*k + j, P = N*k.
const char* moe_check(long N, int E, int k, int d);
// idx[n, j], gates[n, j] from FP32 router logits [N, E]: k largest, ties to the lower id; softmax over them.
int launch_moe_topk(const float* logits, long N, int E, int k, int32_t* idx, float* gates, cudaStream_t s);
// Stable counting sort of the pairs by expert: order[i] = pair at position i,
// pos[p] = position of pair p, offsets[e] = first position of expert e.  Each
// expert's positions are padded to a multiple of row_align (order = -1 at the
// padding; offsets[E] = the padded total); order holds
// moe_rows_capacity(P, E, row_align) entries.  row_align = 1: no padding.
long moe_sort_scratch_ints(long P, int E);
long moe_rows_capacity(long P, int E, int row_align);
int launch_moe_sort(const int32_t* idx, long P, int E, int row_align, int32_t* scratch, int32_t* order,
                    int32_t* pos, int32_t* offsets, cudaStream_t s);
// xp[i] = x[order[i] / k] for i < P (rows of d BF16 values; x rows ldx apart);
// a zero row where order[i] < 0.
int launch_moe_gather(const bf16* x, long ldx, const int32_t* order, int k, long P, int d, bf16* xp,
                      cudaStream_t s);
// out[n] = res[n] + sum_j gates[n, j] yp[pos[n k + j]] (res may be null).
int launch_moe_combine(const bf16* yp, const int32_t* pos, const float* gates, long N, int k, int d, const bf16* res,
                       bf16* out, cudaStream_t s);
// dyp[pos[p]] = gates[p] dy[n]; dgates[p] = <dy[n], yp[pos[p]]>.
int launch_moe_combine_bwd(const bf16* dy, const bf16* yp, const int32_t* pos, const float* gates, long N, int k,
                           int d, bf16* dyp, float* dgates, cudaStream_t s);
// ds [N, E] (BF16): softmax backward over the selected logits, zero elsewhere.
int launch_moe_gate_bwd(const int32_t* idx, const float* gates, const float* dgates, long N, int E, int k, bf16* ds,
                        cudaStream_t s);
// buf[i] = 0 (d BF16 values) for the rows i < P_rows with order[i] < 0.
int launch_moe_zero_pads(const int32_t* order, long P_rows, int d, bf16* buf, cudaStream_t s);
// dx[n] = dres[n] + sum_j dxp[pos[n k + j]] (dres may be null).
int launch_moe_scatter_bwd(const bf16* dxp, const int32_t* pos, long N, int k, int d, const bf16* dres, bf16* dx,
                           cudaStream_t s);

}  // namespace mt
