// Mixture-of-experts MLP: the routing and data-movement kernels around the
// per-expert GEMMs (which run on the library's tcgen05 GEMM over the rows
// routed to each expert).
//
// Definition (the pages name gpt-oss 120B as an MoE model but give no formula;
// the plainest top-k reading): router logits s = x W_r^T; per token the k
// experts with the largest logits, ties to the lower expert id; gates =
// softmax over the k selected logits; y = sum_j gate_j * expert_{e_j}(x).
//
// Every kernel here is deterministic: the pairs (token n, slot j), p = n*k + j,
// are ordered by expert with a stable counting sort (per-block histograms, an
// exclusive scan in expert-major order, stable ranks inside each block), and
// every reduction over a token's k slots runs in slot order.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace mt {

namespace {

constexpr int kMoeSortBlock = 1024;  // pairs per block of the counting sort

__device__ __forceinline__ float bf(const bf16 v) { return __bfloat162float(v); }

// (value, id) comparison of the selection: larger value first, ties to the lower id.
__device__ __forceinline__ bool moe_better(float v, int i, float w, int j) {
  return v > w || (v == w && i < j);
}

// One warp per token: k rounds of a warp arg-max over the E logits (E <= 256,
// at most 8 per lane), then the softmax over the selected logits.
__global__ void moe_topk_kernel(const float* __restrict__ logits, long N, int E, int k, int32_t* __restrict__ idx,
                                float* __restrict__ gates) {
  const long n = ((long)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x & 31;
  if (n >= N) return;
  float v[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int e = q * 32 + lane;
    const float l = e < E ? logits[n * E + e] : -INFINITY;
    v[q] = l == l ? l : -INFINITY;  // a NaN logit (the step is lost anyway) ranks as -inf
  }
  unsigned taken = 0;  // bit q: expert q*32 + lane already selected
  float sel_v[8];
  int sel_i[8];
  for (int r = 0; r < k; ++r) {
    // this lane's best candidate among the experts not yet selected
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = q * 32 + lane;
      if (e < E && !((taken >> q) & 1u) && (bi == 0x7fffffff || moe_better(v[q], e, bv, bi))) {
        bv = v[q];
        bi = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (moe_better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    sel_v[r] = bv;
    sel_i[r] = bi;  // k <= E: some expert is always left
    // the winner leaves its lane's candidates
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (q * 32 + lane == bi) taken |= 1u << q;
  }
  if (lane == 0) {
    const float m = sel_v[0];
    float sum = 0.f;
    for (int r = 0; r < k; ++r) sum += __expf(sel_v[r] - m);
    const float inv = 1.f / sum;
    for (int r = 0; r < k; ++r) {
      idx[n * k + r] = sel_i[r];
      gates[n * k + r] = __expf(sel_v[r] - m) * inv;
    }
  }
}

// Counting sort, pass 1: counts[b * E + e] = pairs of block b routed to e.
__global__ void moe_hist_kernel(const int32_t* __restrict__ idx, long P, int E, int32_t* __restrict__ counts) {
  extern __shared__ int32_t h[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
  __syncthreads();
  const long p0 = (long)blockIdx.x * kMoeSortBlock;
  for (int t = threadIdx.x; t < kMoeSortBlock; t += blockDim.x) {
    const long p = p0 + t;
    if (p < P) atomicAdd(&h[idx[p]], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) counts[(long)blockIdx.x * E + e] = h[e];
}

// Pass 2 (one block): base[b * E + e] = position of the first pair of (e, b)
// in expert-major order; offsets[e] = first position of expert e.  Each
// expert's range is padded to a multiple of row_align positions (order = -1
// there); offsets[E] = the padded total.
__global__ void moe_scan_kernel(const int32_t* __restrict__ counts, int nblk, int E, int row_align,
                                int32_t* __restrict__ base, int32_t* __restrict__ offsets) {
  if (threadIdx.x != 0) return;  // nblk * E is small (thousands): one thread keeps the order plain
  int32_t run = 0;
  for (int e = 0; e < E; ++e) {
    offsets[e] = run;
    for (int b = 0; b < nblk; ++b) {
      base[(long)b * E + e] = run;
      run += counts[(long)b * E + e];
    }
    run = (run + row_align - 1) / row_align * row_align;
  }
  offsets[E] = run;
}

// Pass 3: one warp per block walks its pairs in index order, 32 at a time;
// pairs of the same expert inside a group of 32 are ranked by lane, and a
// per-expert running count carries the ranks across groups.
__global__ void moe_place_kernel(const int32_t* __restrict__ idx, long P, int E, const int32_t* __restrict__ base,
                                 int32_t* __restrict__ order, int32_t* __restrict__ pos) {
  extern __shared__ int32_t run[];
  const int lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) run[e] = 0;
  __syncwarp();
  const long p0 = (long)blockIdx.x * kMoeSortBlock;
  for (int c = 0; c < kMoeSortBlock; c += 32) {
    const long p = p0 + c + lane;
    const bool ok = p < P;
    const int e = ok ? idx[p] : -1 - lane;  // out-of-range lanes match nobody
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(same & ((1u << lane) - 1u));
    int r0 = 0;
    if (ok) r0 = run[e];
    __syncwarp();
    if (ok) {
      const int at = base[(long)blockIdx.x * E + e] + r0 + rank;
      pos[p] = at;
      order[at] = (int32_t)p;
      if (rank == 0) run[e] = r0 + __popc(same);
    }
    __syncwarp();
  }
}

// xp[i] = x[order[i] / k], a zero row where order[i] < 0 (padding): 16-byte
// copies, one warp per row.
__global__ void moe_gather_kernel(const bf16* __restrict__ x, long ldx, const int32_t* __restrict__ order, int k,
                                  long P, int d, bf16* __restrict__ xp) {
  const long i = ((long)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x & 31;
  if (i >= P) return;
  const int32_t o = order[i];
  uint4* dst = reinterpret_cast<uint4*>(xp + i * (long)d);
  if (o < 0) {
    for (int c = lane; c < d / 8; c += 32) dst[c] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(x + (long)(o / k) * ldx);
  for (int c = lane; c < d / 8; c += 32) dst[c] = src[c];
}

// buf[i] = 0 for the padding rows (order[i] < 0), one warp per row.
__global__ void moe_zero_pads_kernel(const int32_t* __restrict__ order, long P, int d, bf16* __restrict__ buf) {
  const long i = ((long)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x & 31;
  if (i >= P || order[i] >= 0) return;
  uint4* dst = reinterpret_cast<uint4*>(buf + i * (long)d);
  for (int c = lane; c < d / 8; c += 32) dst[c] = make_uint4(0u, 0u, 0u, 0u);
}

// out[n] = res[n] + sum_j gates[n, j] * yp[pos[n*k + j]] (FP32, slot order).
__global__ void moe_combine_kernel(const bf16* __restrict__ yp, const int32_t* __restrict__ pos,
                                   const float* __restrict__ gates, long N, int k, int d,
                                   const bf16* __restrict__ res, bf16* __restrict__ out) {
  const long n = blockIdx.x;
  if (n >= N) return;
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    float acc = res ? bf(res[n * d + c]) : 0.f;
    for (int j = 0; j < k; ++j) acc += gates[n * k + j] * bf(yp[(long)pos[n * k + j] * d + c]);
    out[n * d + c] = __float2bfloat16_rn(acc);
  }
}

// Backward of the combine, one block per token:
//   dyp[pos[p]] = gates[p] * dy[n],  dgates[p] = <dy[n], yp[pos[p]]> (fixed-order block sum).
__global__ void moe_combine_bwd_kernel(const bf16* __restrict__ dy, const bf16* __restrict__ yp,
                                       const int32_t* __restrict__ pos, const float* __restrict__ gates, long N,
                                       int k, int d, bf16* __restrict__ dyp, float* __restrict__ dgates) {
  __shared__ float red[32];
  const long n = blockIdx.x;
  if (n >= N) return;
  for (int j = 0; j < k; ++j) {
    const long p = n * k + j;
    const long at = pos[p];
    const float g = gates[p];
    float dot = 0.f;
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
      const float dv = bf(dy[n * d + c]);
      dyp[at * d + c] = __float2bfloat16_rn(g * dv);
      dot += dv * bf(yp[at * d + c]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = dot;
    __syncthreads();
    if (threadIdx.x == 0) {
      float s = 0.f;
      for (int w = 0; w < (int)(blockDim.x / 32); ++w) s += red[w];
      dgates[p] = s;
    }
    __syncthreads();
  }
}

// Softmax backward over the selected logits, one thread per token:
// ds[n, e_j] = g_j (dg_j - sum_i g_i dg_i), zero for the experts not selected.
__global__ void moe_gate_bwd_kernel(const int32_t* __restrict__ idx, const float* __restrict__ gates,
                                    const float* __restrict__ dgates, long N, int E, int k, bf16* __restrict__ ds) {
  const long n = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  for (int e = 0; e < E; ++e) ds[n * E + e] = __float2bfloat16_rn(0.f);
  float dot = 0.f;
  for (int j = 0; j < k; ++j) dot += gates[n * k + j] * dgates[n * k + j];
  for (int j = 0; j < k; ++j)
    ds[n * E + idx[n * k + j]] = __float2bfloat16_rn(gates[n * k + j] * (dgates[n * k + j] - dot));
}

// dx[n] = dres[n] + sum_j dxp[pos[n*k + j]] (FP32, slot order).
__global__ void moe_scatter_bwd_kernel(const bf16* __restrict__ dxp, const int32_t* __restrict__ pos, long N, int k,
                                       int d, const bf16* __restrict__ dres, bf16* __restrict__ dx) {
  const long n = blockIdx.x;
  if (n >= N) return;
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    float acc = dres ? bf(dres[n * d + c]) : 0.f;
    for (int j = 0; j < k; ++j) acc += bf(dxp[(long)pos[n * k + j] * d + c]);
    dx[n * d + c] = __float2bfloat16_rn(acc);
  }
}

}  // namespace

const char* moe_check(long N, int E, int k, int d) {
  if (N <= 0 || d <= 0) return "moe: empty shape";
  if (N * (long)k + 255L * E > 0x7fffffffL) return "moe: too many (token, slot) pairs for int32 positions";
  if (E < 1 || E > 256) return "moe: 1 <= n_experts <= 256";
  if (k < 1 || k > 8 || k > E) return "moe: 1 <= top_k <= min(8, n_experts)";
  if (d % 8) return "moe: d_model must be a multiple of 8";
  return nullptr;
}

int launch_moe_topk(const float* logits, long N, int E, int k, int32_t* idx, float* gates, cudaStream_t s) {
  moe_topk_kernel<<<(unsigned)((N * 32 + 255) / 256), 256, 0, s>>>(logits, N, E, k, idx, gates);
  return launch_result();
}

long moe_sort_scratch_ints(long P, int E) { return ((P + kMoeSortBlock - 1) / kMoeSortBlock) * (long)E * 2; }

long moe_rows_capacity(long P, int E, int row_align) { return P + (long)(row_align - 1) * E; }

int launch_moe_sort(const int32_t* idx, long P, int E, int row_align, int32_t* scratch, int32_t* order,
                    int32_t* pos, int32_t* offsets, cudaStream_t s) {
  const int nblk = (int)((P + kMoeSortBlock - 1) / kMoeSortBlock);
  int32_t* counts = scratch;
  int32_t* base = scratch + (long)nblk * E;
  if (row_align > 1 &&
      cudaMemsetAsync(order, 0xff, sizeof(int32_t) * moe_rows_capacity(P, E, row_align), s) != cudaSuccess)
    return launch_result();
  moe_hist_kernel<<<nblk, 256, E * sizeof(int32_t), s>>>(idx, P, E, counts);
  moe_scan_kernel<<<1, 32, 0, s>>>(counts, nblk, E, row_align, base, offsets);
  moe_place_kernel<<<nblk, 32, E * sizeof(int32_t), s>>>(idx, P, E, base, order, pos);
  return launch_result();
}

int launch_moe_zero_pads(const int32_t* order, long P_rows, int d, bf16* buf, cudaStream_t s) {
  moe_zero_pads_kernel<<<(unsigned)((P_rows * 32 + 255) / 256), 256, 0, s>>>(order, P_rows, d, buf);
  return launch_result();
}

int launch_moe_gather(const bf16* x, long ldx, const int32_t* order, int k, long P, int d, bf16* xp,
                      cudaStream_t s) {
  moe_gather_kernel<<<(unsigned)((P * 32 + 255) / 256), 256, 0, s>>>(x, ldx, order, k, P, d, xp);
  return launch_result();
}

int launch_moe_combine(const bf16* yp, const int32_t* pos, const float* gates, long N, int k, int d, const bf16* res,
                       bf16* out, cudaStream_t s) {
  moe_combine_kernel<<<(unsigned)N, 256, 0, s>>>(yp, pos, gates, N, k, d, res, out);
  return launch_result();
}

int launch_moe_combine_bwd(const bf16* dy, const bf16* yp, const int32_t* pos, const float* gates, long N, int k,
                           int d, bf16* dyp, float* dgates, cudaStream_t s) {
  moe_combine_bwd_kernel<<<(unsigned)N, 256, 0, s>>>(dy, yp, pos, gates, N, k, d, dyp, dgates);
  return launch_result();
}

int launch_moe_gate_bwd(const int32_t* idx, const float* gates, const float* dgates, long N, int E, int k, bf16* ds,
                        cudaStream_t s) {
  moe_gate_bwd_kernel<<<(unsigned)((N + 255) / 256), 256, 0, s>>>(idx, gates, dgates, N, E, k, ds);
  return launch_result();
}

int launch_moe_scatter_bwd(const bf16* dxp, const int32_t* pos, long N, int k, int d, const bf16* dres, bf16* dx,
                           cudaStream_t s) {
  moe_scatter_bwd_kernel<<<(unsigned)N, 256, 0, s>>>(dxp, pos, N, k, d, dres, dx);
  return launch_result();
}

}  // namespace mt
