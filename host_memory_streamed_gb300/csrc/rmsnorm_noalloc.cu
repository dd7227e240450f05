// RMSNorm backward for callers that cannot allocate device memory.
//
// mt_op_rmsnorm_bwd needs a caller-provided FP32 scratch buffer for the
// per-block partial sums of the gain gradient.  Some callers cannot provide
// one: code embedded in a host application that reserves the whole GPU memory
// budget up front and forbids further allocation, or a latency-critical loop
// in which a cudaMalloc/cudaFree (which can synchronise the device) is not
// acceptable.  mt_op_rmsnorm_bwd_noalloc runs the same kernels with the
// scratch held in a fixed array in this library's own device memory instead.
//
// The array below lives in every GPU that loads the library for as long as
// the process runs.  Every call shares it; each call overwrites the part it
// uses before reading it, so nothing from an earlier call leaks into a result.
// Calls that overlap on the GPU (different streams, or different host threads
// without ordering) race on the array and must be serialised by the caller.
#include <cuda_runtime.h>

#include <cstdint>
#include <map>
#include <mutex>
#include <string>

#include "../../include/mt_ops.h"
#include "kernels.h"

namespace mt {
namespace {

// Largest scratch (in floats) one call may use: ceil(rows / 64) * d <= this.
constexpr long kNoAllocScratchFloats = 4L << 20;  // 16 MiB

static __device__ __align__(256) float g_rmsnorm_scratch[kNoAllocScratchFloats];

// Device address of the array for the current device, looked up once per device.
float* scratch_for_current_device(int* err) {
  static std::mutex mu;
  static std::map<int, float*> addr;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    *err = 1;
    return nullptr;
  }
  std::lock_guard<std::mutex> g(mu);
  auto it = addr.find(dev);
  if (it != addr.end()) return it->second;
  void* p = nullptr;
  const cudaError_t rc = cudaGetSymbolAddress(&p, g_rmsnorm_scratch);
  if (rc != cudaSuccess || p == nullptr) {
    *err = 2;
    return nullptr;
  }
  addr[dev] = static_cast<float*>(p);
  return static_cast<float*>(p);
}

}  // namespace

// Message for mt_op_last_error() (defined with the other per-kernel entry points).
void set_op_error(const std::string& msg);

}  // namespace mt

extern "C" int mt_op_rmsnorm_bwd_noalloc(const void* dy, const void* x, const void* g, const float* rstd,
                                         const void* dres, void* dx, void* dg, int64_t rows, int32_t d,
                                         void* stream) {
  if (d <= 0 || d % 8 || rows < 0) {
    mt::set_op_error("rmsnorm (no-alloc): d must be a positive multiple of 8 and rows >= 0");
    return MT_EINVAL;
  }
  if (!dg || (rows > 0 && (!dy || !x || !g || !rstd || !dx))) {
    mt::set_op_error("rmsnorm (no-alloc): null dy, x, g, rstd, dx or dg");
    return MT_EINVAL;
  }
  if ((reinterpret_cast<uintptr_t>(dy) | reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(g) |
       reinterpret_cast<uintptr_t>(dres) | reinterpret_cast<uintptr_t>(dx)) & 15) {
    mt::set_op_error("rmsnorm (no-alloc): dy, x, g, dres and dx must be 16-byte aligned");
    return MT_EINVAL;
  }
  if (d > mt::rmsnorm_bwd_max_d()) {
    mt::set_op_error("rmsnorm (no-alloc): d = " + std::to_string(d) + " exceeds the widest row this device takes (" +
                     std::to_string(mt::rmsnorm_bwd_max_d()) + ")");
    return MT_EINVAL;
  }
  // partial-sum rows, computed without overflow for any rows >= 0
  const int64_t nparts = rows / mt::kRmsRowsPerBlock + (rows % mt::kRmsRowsPerBlock != 0);
  if (nparts > mt::kNoAllocScratchFloats / d) {
    mt::set_op_error("rmsnorm (no-alloc): ceil(rows/64) * d exceeds the fixed scratch of " +
                     std::to_string(mt::kNoAllocScratchFloats) +
                     " floats; use mt_op_rmsnorm_bwd with a caller buffer");
    return MT_EINVAL;
  }
  int err = 0;
  float* scratch = mt::scratch_for_current_device(&err);
  if (!scratch) {
    mt::set_op_error("rmsnorm (no-alloc): cudaGetSymbolAddress of the scratch array failed");
    return MT_ECUDA;
  }
  auto s = static_cast<cudaStream_t>(stream);
  // the kernel writes at most nparts partial rows (fewer when its grid is capped at one wave)
  const long parts = mt::launch_rmsnorm_bwd(static_cast<const mt::bf16*>(dy), static_cast<const mt::bf16*>(x),
                                            static_cast<const mt::bf16*>(g), rstd,
                                            static_cast<const mt::bf16*>(dres), static_cast<mt::bf16*>(dx), scratch,
                                            rows, d, s);
  mt::launch_colsum_bf16(scratch, parts, d, static_cast<mt::bf16*>(dg), s);
  if (cudaPeekAtLastError() != cudaSuccess) {
    mt::set_op_error(std::string("rmsnorm (no-alloc): launch failed: ") + cudaGetErrorString(cudaGetLastError()));
    return MT_ECUDA;
  }
  return MT_OK;
}
