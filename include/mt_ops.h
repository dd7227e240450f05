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
  MT_EPI_ROPE = 5          /* C = acc (BF16) with rotate-half RoPE applied to columns < rope_cols,
                              heads of head_dim columns, position = row % seq */
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

#ifdef __cplusplus
}
#endif
#endif
