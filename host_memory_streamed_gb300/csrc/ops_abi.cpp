// C-ABI wrappers of the individual device kernels (declared in include/mt_ops.h).
// They take device pointers and a cudaStream_t passed as void*, launch one
// kernel sequence and return without synchronising.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <string>

#include "../../include/mt_ops.h"
#include "kernels.h"

namespace {
thread_local std::string g_op_error;
int op_fail(const char* msg) {
  g_op_error = msg ? msg : "unknown error";
  return MT_EINVAL;
}
int op_cuda(int rc, const char* what) {
  if (rc == 0) return MT_OK;
  g_op_error = std::string(what) + ": launch failed (" + cudaGetErrorString(cudaGetLastError()) + ")";
  return MT_ECUDA;
}
}  // namespace

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
  if (const char* e = mt::gemm_check(g)) return op_fail(e);
  return op_cuda(mt::launch_gemm(g, static_cast<cudaStream_t>(stream)), "gemm");
}

}  // extern "C"
