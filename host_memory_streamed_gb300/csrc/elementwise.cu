// HBM-bound kernels of the decoder step: RMSNorm forward/backward, SwiGLU
// backward, transposes, embedding gather / deterministic scatter, row-wise
// cross-entropy, reductions.  128-bit (8 x BF16) vectorised, coalesced access;
// FP32 arithmetic; every reduction runs in a fixed order so results are
// bit-reproducible run to run.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cfloat>
#include <map>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace mt {

namespace {

__device__ __forceinline__ void unpack8(const uint4& w, float* f) {
  f[0] = __uint_as_float(w.x << 16);
  f[1] = __uint_as_float(w.x & 0xFFFF0000u);
  f[2] = __uint_as_float(w.y << 16);
  f[3] = __uint_as_float(w.y & 0xFFFF0000u);
  f[4] = __uint_as_float(w.z << 16);
  f[5] = __uint_as_float(w.z & 0xFFFF0000u);
  f[6] = __uint_as_float(w.w << 16);
  f[7] = __uint_as_float(w.w & 0xFFFF0000u);
}
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&p);
}
__device__ __forceinline__ uint4 pack8(const float* f) {
  return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// Block-wide sum with a fixed reduction tree (deterministic).
template <int THREADS>
__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x / 32, l = threadIdx.x % 32;
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
  if (w == 0) {
    t = l < THREADS / 32 ? red[l] : 0.f;
    t = warp_sum(t);
    if (l == 0) red[0] = t;
  }
  __syncthreads();
  t = red[0];
  __syncthreads();
  return t;
}

// ---------------------------------------------------------------- RMSNorm
// One block per row; d % 8 == 0; each thread owns d/8/THREADS (ceil) vectors.
constexpr int RMS_THREADS = 256;

__global__ void __launch_bounds__(RMS_THREADS) rmsnorm_fwd_kernel(const bf16* __restrict__ x, const bf16* __restrict__ g,
                                                              bf16* __restrict__ y, float* __restrict__ rstd, int d,
                                                              float eps) {
  __shared__ float red[32];
  const long row = blockIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(x + row * d);
  const uint4* gr = reinterpret_cast<const uint4*>(g);
  uint4* yr = reinterpret_cast<uint4*>(y + row * d);
  const int nv = d / 8;
  float ss = 0.f;
  for (int i = threadIdx.x; i < nv; i += RMS_THREADS) {
    float f[8];
    unpack8(xr[i], f);
#pragma unroll
    for (int j = 0; j < 8; ++j) ss += f[j] * f[j];
  }
  ss = block_sum<RMS_THREADS>(ss, red);
  const float r = rsqrtf(ss / (float)d + eps);
  if (threadIdx.x == 0) rstd[row] = r;
  for (int i = threadIdx.x; i < nv; i += RMS_THREADS) {
    float f[8], w[8];
    unpack8(xr[i], f);
    unpack8(gr[i], w);
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] = f[j] * r * w[j];
    yr[i] = pack8(f);
  }
}

// Backward: one block handles kRmsRowsPerBlock rows; per-column dg partials of
// the block go to dg_partial[blockIdx.x, :] (summed later in fixed order).
__global__ void __launch_bounds__(RMS_THREADS) rmsnorm_bwd_kernel(const bf16* __restrict__ dy,
                                                              const bf16* __restrict__ x, const bf16* __restrict__ g,
                                                              const float* __restrict__ rstd,
                                                              const bf16* __restrict__ dres, bf16* __restrict__ dx,
                                                              float* __restrict__ dg_partial, long rows, int d) {
  __shared__ float red[32];
  extern __shared__ float dg_acc[];  // d floats
  const int nv = d / 8;
  for (int c = threadIdx.x; c < d; c += RMS_THREADS) dg_acc[c] = 0.f;
  __syncthreads();
  const long r0 = (long)blockIdx.x * kRmsRowsPerBlock;
  const long r1 = min(rows, r0 + kRmsRowsPerBlock);
  const uint4* gr = reinterpret_cast<const uint4*>(g);
  for (long row = r0; row < r1; ++row) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + row * d);
    const uint4* dyr = reinterpret_cast<const uint4*>(dy + row * d);
    const float r = rstd[row];
    float dot = 0.f;
    for (int i = threadIdx.x; i < nv; i += RMS_THREADS) {
      float xf[8], df[8], wf[8];
      unpack8(xr[i], xf);
      unpack8(dyr[i], df);
      unpack8(gr[i], wf);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float xh = xf[j] * r;
        dot += df[j] * wf[j] * xh;
        dg_acc[i * 8 + j] += df[j] * xh;  // each column owned by one thread: no race
      }
    }
    dot = block_sum<RMS_THREADS>(dot, red) / (float)d;
    uint4* dxr = reinterpret_cast<uint4*>(dx + row * d);
    const uint4* rr = dres ? reinterpret_cast<const uint4*>(dres + row * d) : nullptr;
    for (int i = threadIdx.x; i < nv; i += RMS_THREADS) {
      float xf[8], df[8], wf[8], out[8];
      unpack8(xr[i], xf);
      unpack8(dyr[i], df);
      unpack8(gr[i], wf);
      float rf[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (rr) unpack8(rr[i], rf);
#pragma unroll
      for (int j = 0; j < 8; ++j) out[j] = rf[j] + r * (df[j] * wf[j] - xf[j] * r * dot);
      dxr[i] = pack8(out);
    }
  }
  __syncthreads();
  for (int c = threadIdx.x; c < d; c += RMS_THREADS) dg_partial[(long)blockIdx.x * d + c] = dg_acc[c];
}

// Backward with the columns held in registers: each thread owns VPT 16-byte
// vectors (8 columns each) of every row, vector i = threadIdx.x + k*blockDim.x
// for k < VPT, so the gain and the block's gain-gradient sums for those
// columns stay in registers for all of the block's rows.  The grid is one
// wave (every block resident at once), each block taking an equal run of
// rows_per_block >= kRmsRowsPerBlock rows, so no partial wave idles the
// memory system at the end.  A block's rows go two at a time; with PREFETCH (one vector per
// thread, where the registers allow it) the next pair's dy, x and dres
// vectors are requested before the current pair is reduced, so loads stay in
// flight while the block waits on its reduction barrier.  The
// two rows' dot products are reduced together (warp butterfly, then the
// warps' sums in warp order from a double-buffered shared slot: one barrier
// per pair of rows).  No shared-memory accumulator and no barrier per row,
// unlike rmsnorm_bwd_kernel, which remains for rows wider than
// kRmsBwdRegMaxVectors vectors.
constexpr int kRmsBwdRegMaxVectors = 1024;  // d <= 8192

template <int VPT>
struct RmsPair {
  uint4 dy[2][VPT], x[2][VPT], r[2][VPT];
  float rs[2];
};

template <int VPT>
__device__ __forceinline__ void rms_load_pair(RmsPair<VPT>& p, const bf16* __restrict__ dy,
                                              const bf16* __restrict__ x, const float* __restrict__ rstd,
                                              const bf16* __restrict__ dres, long row, int nr, int nv) {
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const long off = (row + j) * (long)nv;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int i = threadIdx.x + k * blockDim.x;
      const bool ok = i < nv && j < nr;
      p.dy[j][k] = ok ? reinterpret_cast<const uint4*>(dy)[off + i] : zero;
      p.x[j][k] = ok ? reinterpret_cast<const uint4*>(x)[off + i] : zero;
      p.r[j][k] = (ok && dres) ? reinterpret_cast<const uint4*>(dres)[off + i] : zero;
    }
  }
  p.rs[0] = nr > 0 ? rstd[row] : 0.f;
  p.rs[1] = nr > 1 ? rstd[row + 1] : 0.f;
}

template <int VPT, bool PREFETCH>
__global__ void __launch_bounds__(VPT == 1 ? 640 : (VPT == 2 ? 384 : 256)) rmsnorm_bwd_rows_kernel(
    const bf16* __restrict__ dy, const bf16* __restrict__ x, const bf16* __restrict__ g,
    const float* __restrict__ rstd, const bf16* __restrict__ dres, bf16* __restrict__ dx,
    float* __restrict__ dg_partial, long rows, int d, long rows_per_block) {
  __shared__ float red[2][2][32];  // [buffer][row of the pair][warp]
  const int nv = d / 8;
  const int nthreads = blockDim.x;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, nwarps = nthreads / 32;
  const uint4* gr = reinterpret_cast<const uint4*>(g);
  float wf[VPT][8], acc[VPT][8];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int i = threadIdx.x + k * nthreads;
    if (i < nv) {
      unpack8(gr[i], wf[k]);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) wf[k][e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[k][e] = 0.f;
  }
  const long r0 = (long)blockIdx.x * rows_per_block;
  const long r1 = min(rows, r0 + rows_per_block);
  auto pair_rows = [&](long row) { return row >= r1 ? 0 : (row + 1 < r1 ? 2 : 1); };
  RmsPair<VPT> cur, nxt;
  if (PREFETCH) rms_load_pair<VPT>(cur, dy, x, rstd, dres, r0, pair_rows(r0), nv);
  int buf = 0;
  for (long row = r0; row < r1; row += 2) {
    const int nr = pair_rows(row);
    if (PREFETCH)
      rms_load_pair<VPT>(nxt, dy, x, rstd, dres, row + 2, pair_rows(row + 2), nv);
    else
      rms_load_pair<VPT>(cur, dy, x, rstd, dres, row, nr, nv);
    float dot[2] = {0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        float xf[8], df[8];
        unpack8(cur.x[j][k], xf);
        unpack8(cur.dy[j][k], df);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float xh = xf[e] * cur.rs[j];
          dot[j] += df[e] * wf[k][e] * xh;
          acc[k][e] += df[e] * xh;  // zero for a missing second row (dy = 0)
        }
      }
    }
    dot[0] = warp_sum(dot[0]);
    dot[1] = warp_sum(dot[1]);
    if (lane == 0) {
      red[buf][0][warp] = dot[0];
      red[buf][1][warp] = dot[1];
    }
    __syncthreads();
    float t0 = 0.f, t1 = 0.f;
    for (int w = 0; w < nwarps; ++w) {
      t0 += red[buf][0][w];
      t1 += red[buf][1][w];
    }
    // the next pair writes the other buffer; this one is rewritten only after
    // the next pair's barrier, which every thread reaches after reading it
    buf ^= 1;
    const float mean[2] = {t0 / (float)d, t1 / (float)d};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (j >= nr) break;
      const long off = (row + j) * (long)nv;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int i = threadIdx.x + k * nthreads;
        if (i >= nv) continue;
        float xf[8], df[8], rf[8], out[8];
        unpack8(cur.x[j][k], xf);
        unpack8(cur.dy[j][k], df);
        unpack8(cur.r[j][k], rf);
#pragma unroll
        for (int e = 0; e < 8; ++e) out[e] = rf[e] + cur.rs[j] * (df[e] * wf[k][e] - xf[e] * cur.rs[j] * mean[j]);
        reinterpret_cast<uint4*>(dx)[off + i] = pack8(out);
      }
    }
    if (PREFETCH) cur = nxt;
  }
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int i = threadIdx.x + k * nthreads;
    if (i < nv) {
      float4* dst = reinterpret_cast<float4*>(dg_partial + (long)blockIdx.x * d + (long)i * 8);
      dst[0] = make_float4(acc[k][0], acc[k][1], acc[k][2], acc[k][3]);
      dst[1] = make_float4(acc[k][4], acc[k][5], acc[k][6], acc[k][7]);
    }
  }
}

// out[c] = sum_p partial[p, c] in a fixed order: the parts split into
// kColsumSlices consecutive slices, each summed in ascending order by one warp
// over 32 adjacent columns (128-byte loads), then the slice sums in slice
// order.  One block per 32 columns.
constexpr int kColsumSlices = 8;
__global__ void __launch_bounds__(32 * kColsumSlices) colsum_bf16_kernel(const float* __restrict__ partial,
                                                                       long nparts, int d, bf16* __restrict__ out) {
  __shared__ float acc[kColsumSlices][32];
  const int lane = threadIdx.x & 31, sl = threadIdx.x >> 5;
  const int c = blockIdx.x * 32 + lane;
  const long per = (nparts + kColsumSlices - 1) / kColsumSlices;
  const long p0 = sl * per, p1 = min(nparts, p0 + per);
  float v = 0.f;
  if (c < d) {
#pragma unroll 8
    for (long p = p0; p < p1; ++p) v += partial[p * d + c];
  }
  acc[sl][lane] = v;
  __syncthreads();
  if (sl == 0 && c < d) {
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < kColsumSlices; ++k) t += acc[k][lane];
    out[c] = __float2bfloat16_rn(t);
  }
}

// ---------------------------------------------------------------- SwiGLU backward
// gu: [rows, 2f] with (gate, up) interleaved; da: [rows, f]; dgu like gu.
__global__ void swiglu_bwd_kernel(const bf16* __restrict__ da, const bf16* __restrict__ gu, bf16* __restrict__ dgu,
                                  long rows, int f) {
  // one thread per 8 outputs of `da` (16 interleaved values)
  const long nvec_row = f / 8;
  const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= rows * nvec_row) return;
  const long row = i / nvec_row, v = i % nvec_row;
  float a8[8], g16[16];
  unpack8(reinterpret_cast<const uint4*>(da + row * f)[v], a8);
  const uint4* gp = reinterpret_cast<const uint4*>(gu + row * 2L * f) + 2 * v;
  unpack8(gp[0], g16);
  unpack8(gp[1], g16 + 8);
  float out[16];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float gt = g16[2 * j], up = g16[2 * j + 1];
    const float sg = 1.0f / (1.0f + __expf(-gt));
    const float silu = gt * sg;
    out[2 * j] = a8[j] * up * sg * (1.0f + gt * (1.0f - sg));
    out[2 * j + 1] = a8[j] * silu;
  }
  uint4* dp = reinterpret_cast<uint4*>(dgu + row * 2L * f) + 2 * v;
  dp[0] = pack8(out);
  dp[1] = pack8(out + 8);
}

// Scalar tail for f % 8 != 0 columns (used when f is not a multiple of 8).
__global__ void swiglu_bwd_scalar_kernel(const bf16* __restrict__ da, const bf16* __restrict__ gu,
                                         bf16* __restrict__ dgu, long rows, int f) {
  const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= rows * f) return;
  const long row = i / f, j = i % f;
  const float a = __bfloat162float(da[row * f + j]);
  const float gt = __bfloat162float(gu[row * 2L * f + 2 * j]);
  const float up = __bfloat162float(gu[row * 2L * f + 2 * j + 1]);
  const float sg = 1.0f / (1.0f + __expf(-gt));
  dgu[row * 2L * f + 2 * j] = __float2bfloat16_rn(a * up * sg * (1.0f + gt * (1.0f - sg)));
  dgu[row * 2L * f + 2 * j + 1] = __float2bfloat16_rn(a * gt * sg);
}

// ---------------------------------------------------------------- transpose
// 64 x 64 tiles through shared memory; 256 threads; 16-byte loads/stores when
// the tile is interior and aligned, element-wise at the edges.
constexpr int TP = 64;
__global__ void __launch_bounds__(256) transpose_kernel(const bf16* __restrict__ src, long rows, long cols, long lds,
                                                        bf16* __restrict__ dst, long ldd) {
  __shared__ bf16 tile[TP][TP + 8];
  const long r0 = (long)blockIdx.y * TP, c0 = (long)blockIdx.x * TP;
  const bool interior = (r0 + TP <= rows) && (c0 + TP <= cols) && (lds % 8 == 0) && (ldd % 8 == 0);
  if (interior) {
    for (int i = threadIdx.x; i < TP * TP / 8; i += 256) {
      const int r = i / (TP / 8), cv = i % (TP / 8);
      const uint4 w = *reinterpret_cast<const uint4*>(src + (r0 + r) * lds + c0 + cv * 8);
      const bf16* e = reinterpret_cast<const bf16*>(&w);
#pragma unroll
      for (int j = 0; j < 8; ++j) tile[r][cv * 8 + j] = e[j];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < TP * TP / 8; i += 256) {
      const int c = i / (TP / 8), rv = i % (TP / 8);
      uint4 w;
      bf16* e = reinterpret_cast<bf16*>(&w);
#pragma unroll
      for (int j = 0; j < 8; ++j) e[j] = tile[rv * 8 + j][c];
      *reinterpret_cast<uint4*>(dst + (c0 + c) * ldd + r0 + rv * 8) = w;
    }
  } else {
    for (int i = threadIdx.x; i < TP * TP; i += 256) {
      const int r = i / TP, c = i % TP;
      if (r0 + r < rows && c0 + c < cols) tile[r][c] = src[(r0 + r) * lds + c0 + c];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < TP * TP; i += 256) {
      const int c = i / TP, r = i % TP;
      if (r0 + r < rows && c0 + c < cols) dst[(c0 + c) * ldd + r0 + r] = tile[r][c];
    }
  }
}

// ---------------------------------------------------------------- embedding
__global__ void embed_fwd_kernel(const int32_t* __restrict__ tok, const bf16* __restrict__ E, bf16* __restrict__ x,
                                 long T, int d, int V, int* status) {
  const long t = blockIdx.x;
  const int id = tok[t];
  const bool ok = id >= 0 && id < V;
  if (!ok && threadIdx.x == 0) set_status(status, kStatusIndexOutOfRange);
  const uint4* src = reinterpret_cast<const uint4*>(E + (long)(ok ? id : 0) * d);
  uint4* dst = reinterpret_cast<uint4*>(x + t * d);
  for (int i = threadIdx.x; i < d / 8; i += blockDim.x) dst[i] = ok ? src[i] : make_uint4(0, 0, 0, 0);
}

// dE[v] = sum of dx rows listed for v (ascending positions), written for every v.
__global__ void embed_bwd_kernel(const int32_t* __restrict__ off, const int32_t* __restrict__ pos,
                                 const bf16* __restrict__ dx, bf16* __restrict__ dE, int V, int d) {
  const long v = blockIdx.x;
  const int b = off[v], e = off[v + 1];
  uint4* out = reinterpret_cast<uint4*>(dE + v * d);
  for (int i = threadIdx.x; i < d / 8; i += blockDim.x) {
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int k = b; k < e; ++k) {
      float f[8];
      unpack8(reinterpret_cast<const uint4*>(dx + (long)pos[k] * d)[i], f);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] += f[j];
    }
    out[i] = pack8(acc);
  }
}

// Only the vocabulary rows that occur among the step's tokens: out[u] = sum of
// the dx rows listed for rows[u] (ascending positions), u < U, packed densely.
__global__ void embed_bwd_rows_kernel(const int32_t* __restrict__ off, const int32_t* __restrict__ pos,
                                      const int32_t* __restrict__ rows, const bf16* __restrict__ dx,
                                      bf16* __restrict__ out, int d) {
  const long u = blockIdx.x;
  const int v = rows[u];
  const int b = off[v], e = off[v + 1];
  uint4* o = reinterpret_cast<uint4*>(out + u * d);
  for (int i = threadIdx.x; i < d / 8; i += blockDim.x) {
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int k = b; k < e; ++k) {
      float f[8];
      unpack8(reinterpret_cast<const uint4*>(dx + (long)pos[k] * d)[i], f);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] += f[j];
    }
    o[i] = pack8(acc);
  }
}

// ---------------------------------------------------------------- cross-entropy
constexpr int CE_THREADS = 512;
// One block per row.  Pass 1: per-thread online (max, sum) over a strided
// slice, combined in a fixed tree; pass 2: dz = (exp(z - lse) - onehot) * inv_n.
__global__ void __launch_bounds__(CE_THREADS) cross_entropy_kernel(const float* __restrict__ z, int V,
                                                                   const int32_t* __restrict__ tgt, float inv_n,
                                                                   bf16* __restrict__ dz, float* __restrict__ loss_rows,
                                                                   int* status) {
  __shared__ float sm[CE_THREADS / 32], ss[CE_THREADS / 32];
  const long row = blockIdx.x;
  const float* zr = z + row * (long)V;
  float m = -FLT_MAX, s = 0.f;
  const bool vec = (V % 4) == 0;
  if (vec) {
    const float4* z4 = reinterpret_cast<const float4*>(zr);
    for (int i = threadIdx.x; i < V / 4; i += CE_THREADS) {
      const float4 q = z4[i];
      const float mx = fmaxf(fmaxf(q.x, q.y), fmaxf(q.z, q.w));
      if (mx > m) {
        s *= __expf(m - mx);
        m = mx;
      }
      s += __expf(q.x - m) + __expf(q.y - m) + __expf(q.z - m) + __expf(q.w - m);
    }
  } else {
    for (int i = threadIdx.x; i < V; i += CE_THREADS) {
      const float q = zr[i];
      if (q > m) {
        s *= __expf(m - q);
        m = q;
      }
      s += __expf(q - m);
    }
  }
  // warp combine
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const float mm = fmaxf(m, m2);
    s = s * __expf(m - mm) + s2 * __expf(m2 - mm);
    m = mm;
  }
  const int w = threadIdx.x / 32, l = threadIdx.x % 32;
  if (l == 0) {
    sm[w] = m;
    ss[w] = s;
  }
  __syncthreads();
  if (w == 0) {
    m = l < CE_THREADS / 32 ? sm[l] : -FLT_MAX;
    s = l < CE_THREADS / 32 ? ss[l] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
      const float mm = fmaxf(m, m2);
      s = s * __expf(m - mm) + s2 * __expf(m2 - mm);
      m = mm;
    }
    if (l == 0) {
      sm[0] = m;
      ss[0] = s;
    }
  }
  __syncthreads();
  const float lse = sm[0] + __logf(ss[0]);
  int y = tgt[row];
  if (y < 0 || y >= V) {
    if (threadIdx.x == 0) set_status(status, kStatusIndexOutOfRange);
    y = 0;
  }
  if (threadIdx.x == 0) loss_rows[row] = lse - zr[y];
  bf16* dr = dz + row * (long)V;
  if (vec && (V % 8) == 0) {
    const float4* z4 = reinterpret_cast<const float4*>(zr);
    for (int i = threadIdx.x; i < V / 8; i += CE_THREADS) {
      const float4 a = z4[2 * i], b = z4[2 * i + 1];
      float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        f[j] = __expf(f[j] - lse);
        if (i * 8 + j == y) f[j] -= 1.0f;
        f[j] *= inv_n;
      }
      reinterpret_cast<uint4*>(dr)[i] = pack8(f);
    }
  } else {
    for (int i = threadIdx.x; i < V; i += CE_THREADS) {
      float p = __expf(zr[i] - lse);
      if (i == y) p -= 1.0f;
      dr[i] = __float2bfloat16_rn(p * inv_n);
    }
  }
}

constexpr int LOSS_THREADS = 1024;
__global__ void __launch_bounds__(LOSS_THREADS) mean_loss_kernel(const float* __restrict__ loss_rows, long n,
                                                                 float inv_n, float* out) {
  __shared__ float red[32];
  // FP64 would be nicer but is slow on this part; pairwise-ish fixed order in FP32 is plenty for a mean.
  float s = 0.f;
  for (long i = threadIdx.x; i < n; i += LOSS_THREADS) s += loss_rows[i];
  s = block_sum<LOSS_THREADS>(s, red);
  if (threadIdx.x == 0) out[0] = s * inv_n;
}

__global__ void f32_to_bf16_kernel(const float* __restrict__ src, bf16* __restrict__ dst, long n) {
  const long i = ((long)blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (i + 8 <= n) {
    const float4 a = reinterpret_cast<const float4*>(src + i)[0], b = reinterpret_cast<const float4*>(src + i)[1];
    float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    *reinterpret_cast<uint4*>(dst + i) = pack8(f);
  } else {
    for (long j = i; j < n; ++j) dst[j] = __float2bfloat16_rn(src[j]);
  }
}

__global__ void check_finite_kernel(const bf16* __restrict__ p, long n, int* status) {
  long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  bool bad = false;
  for (; i < n; i += (long)gridDim.x * blockDim.x) {
    const unsigned short b = reinterpret_cast<const unsigned short*>(p)[i];
    if ((b & 0x7F80u) == 0x7F80u) bad = true;  // exponent all ones: Inf or NaN
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x % 32) == 0) set_status(status, kStatusNonFinite);
}

// *flag = 1 when any of the n BF16 values holds NaN or Inf (exponent bits all
// ones); 16-byte loads, grid-strided.  Every writer stores the same value.
__global__ void flag_nonfinite_kernel(const bf16* __restrict__ p, long n, int* flag) {
  const long nvec = n / 8;
  const uint4* v = reinterpret_cast<const uint4*>(p);
  bool bad = false;
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += (long)gridDim.x * blockDim.x) {
    const uint4 q = v[i];
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
      bad |= ((w[k] & 0x7F80u) == 0x7F80u) | ((w[k] & 0x7F800000u) == 0x7F800000u);
  }
  if (blockIdx.x == 0)
    for (long i = nvec * 8 + threadIdx.x; i < n; i += blockDim.x)
      bad |= (reinterpret_cast<const unsigned short*>(p)[i] & 0x7F80u) == 0x7F80u;
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x % 32) == 0) *flag = 1;
}

inline unsigned blocks_for(long n, int per) { return (unsigned)((n + per - 1) / per); }

// Failure-detection probe (see launch_wait_probe): the barrier expects one
// arrival and gets none, so phase 0 never completes and the bounded wait
// must run out.
__global__ void wait_probe_kernel(int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0 && !mbar_wait_for(&bar, 0, limit_ns)) set_status(status, kStatusWaitProbe);
}

}  // namespace

void launch_rmsnorm_fwd(const bf16* x, const bf16* g, bf16* y, float* rstd, long rows, int d, float eps,
                        cudaStream_t s) {
  if (rows <= 0) return;
  rmsnorm_fwd_kernel<<<(unsigned)rows, RMS_THREADS, 0, s>>>(x, g, y, rstd, d, eps);
}

long rmsnorm_bwd_max_d() {
  static long maxd = -1;
  static std::once_flag once;
  std::call_once(once, [] {
    // widths the register kernel takes need no dynamic shared memory; beyond
    // them rmsnorm_bwd_kernel keeps d floats in shared memory
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      optin = 48 * 1024;
    const long smem_d = ((long)optin - 32 * (long)sizeof(float)) / (long)sizeof(float) / 8 * 8;
    maxd = std::max<long>(smem_d, 8L * kRmsBwdRegMaxVectors);
  });
  return maxd;
}

namespace {
// Blocks of a register-kernel variant, at a given block size, that fit on the
// device at once (0 when the device cannot say).
template <int VPT, bool PF>
int resident_rows_blocks(int threads) {
  static std::mutex mu;
  static std::map<int, int> cache;
  std::lock_guard<std::mutex> g(mu);
  auto it = cache.find(threads);
  if (it != cache.end()) return it->second;
  int dev = 0, sms = 0, per = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, rmsnorm_bwd_rows_kernel<VPT, PF>, threads, 0) !=
          cudaSuccess)
    sms = per = 0;
  return cache[threads] = sms * per;
}

template <int VPT, bool PF>
long launch_rows_variant(const bf16* dy, const bf16* x, const bf16* g, const float* rstd, const bf16* dres, bf16* dx,
                         float* dg_partial, long rows, int d, cudaStream_t s) {
  const int nv = d / 8;
  const int threads = (nv + VPT * 32 - 1) / (VPT * 32) * 32;
  // one block per kRmsRowsPerBlock rows at most (the scratch the callers size),
  // and no more blocks than are resident at once at this block size
  long nb = (rows + kRmsRowsPerBlock - 1) / kRmsRowsPerBlock;
  const int wave = resident_rows_blocks<VPT, PF>(threads);
  if (wave > 0 && nb > wave) nb = wave;
  const long rpb = (rows + nb - 1) / nb;
  nb = (rows + rpb - 1) / rpb;
  rmsnorm_bwd_rows_kernel<VPT, PF><<<(unsigned)nb, threads, 0, s>>>(dy, x, g, rstd, dres, dx, dg_partial, rows, d,
                                                                     rpb);
  return nb;
}
}  // namespace

long launch_rmsnorm_bwd(const bf16* dy, const bf16* x, const bf16* g, const float* rstd, const bf16* dres,
                        bf16* dx, float* dg_partial, long rows, int d, cudaStream_t s) {
  if (rows <= 0) return 0;
  const int nv = d / 8;
  if (nv <= 640) return launch_rows_variant<1, true>(dy, x, g, rstd, dres, dx, dg_partial, rows, d, s);
  if (nv <= 768) return launch_rows_variant<2, false>(dy, x, g, rstd, dres, dx, dg_partial, rows, d, s);
  if (nv <= kRmsBwdRegMaxVectors)
    return launch_rows_variant<4, false>(dy, x, g, rstd, dres, dx, dg_partial, rows, d, s);
  const unsigned nb = blocks_for(rows, kRmsRowsPerBlock);
  const size_t shm = (size_t)d * sizeof(float);
  if (shm > 48 * 1024) cudaFuncSetAttribute(rmsnorm_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)shm);
  rmsnorm_bwd_kernel<<<nb, RMS_THREADS, shm, s>>>(dy, x, g, rstd, dres, dx, dg_partial, rows, d);
  return nb;
}

void launch_colsum_bf16(const float* partial, long nparts, int d, bf16* out, cudaStream_t s) {
  colsum_bf16_kernel<<<blocks_for(d, 32), 32 * kColsumSlices, 0, s>>>(partial, nparts, d, out);
}

void launch_swiglu_bwd(const bf16* da, const bf16* gu, bf16* dgu, long rows, int f, cudaStream_t s) {
  if (rows <= 0) return;
  if (f % 8 == 0) {
    const long n = rows * (f / 8);
    swiglu_bwd_kernel<<<blocks_for(n, 256), 256, 0, s>>>(da, gu, dgu, rows, f);
  } else {
    const long n = rows * (long)f;
    swiglu_bwd_scalar_kernel<<<blocks_for(n, 256), 256, 0, s>>>(da, gu, dgu, rows, f);
  }
}

void launch_transpose(const bf16* src, long rows, long cols, long lds, bf16* dst, long ldd, cudaStream_t s) {
  if (rows <= 0 || cols <= 0) return;
  dim3 grid(blocks_for(cols, TP), blocks_for(rows, TP));
  transpose_kernel<<<grid, 256, 0, s>>>(src, rows, cols, lds, dst, ldd);
}

void launch_embed_fwd(const int32_t* tok, const bf16* E, bf16* x, long T, int d, int V, int* status,
                      cudaStream_t s) {
  if (T <= 0) return;
  embed_fwd_kernel<<<(unsigned)T, 128, 0, s>>>(tok, E, x, T, d, V, status);
}

void launch_embed_bwd_rows(const int32_t* off, const int32_t* pos, const int32_t* rows, int U, const bf16* dx,
                           bf16* out, int d, cudaStream_t s) {
  if (U > 0) embed_bwd_rows_kernel<<<(unsigned)U, 128, 0, s>>>(off, pos, rows, dx, out, d);
}

void launch_embed_bwd(const int32_t* off, const int32_t* pos, const bf16* dx, bf16* dE, int V, int d,
                      cudaStream_t s) {
  embed_bwd_kernel<<<(unsigned)V, 128, 0, s>>>(off, pos, dx, dE, V, d);
}

void launch_cross_entropy(const float* z, long rows, int V, const int32_t* tgt, float inv_n, bf16* dz,
                          float* loss_rows, int* status, cudaStream_t s) {
  if (rows <= 0) return;
  cross_entropy_kernel<<<(unsigned)rows, CE_THREADS, 0, s>>>(z, V, tgt, inv_n, dz, loss_rows, status);
}

void launch_mean_loss(const float* loss_rows, long n, float inv_n, float* out, cudaStream_t s) {
  mean_loss_kernel<<<1, LOSS_THREADS, 0, s>>>(loss_rows, n, inv_n, out);
}

void launch_f32_to_bf16(const float* src, bf16* dst, long n, cudaStream_t s) {
  if (n <= 0) return;
  f32_to_bf16_kernel<<<blocks_for((n + 7) / 8, 256), 256, 0, s>>>(src, dst, n);
}

void launch_zero(void* p, size_t bytes, cudaStream_t s) {
  if (bytes) cudaMemsetAsync(p, 0, bytes, s);
}

void launch_check_finite(const bf16* p, long n, int* status, cudaStream_t s) {
  if (n <= 0) return;
  unsigned nb = blocks_for(n, 256);
  if (nb > 152u * 16u) nb = 152u * 16u;
  check_finite_kernel<<<nb, 256, 0, s>>>(p, n, status);
}

void launch_flag_nonfinite(const bf16* p, long n, int* flag, cudaStream_t s) {
  if (n <= 0) return;
  unsigned nb = blocks_for((n + 7) / 8, 256);
  if (nb > 152u * 8u) nb = 152u * 8u;
  flag_nonfinite_kernel<<<nb, 256, 0, s>>>(p, n, flag);
}

int launch_wait_probe(int* status, uint64_t limit_ns, cudaStream_t s) {
  wait_probe_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return launch_result();
}

}  // namespace mt
