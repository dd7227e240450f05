// Causal grouped-query flash attention, forward and backward.
//
// Forward (per (batch, query head), 128 queries per CTA, 8 warps x 16 rows):
// stream 64-key blocks of K and V through double-buffered shared memory
// (cp.async, XOR-swizzled rows so ldmatrix is conflict-free), S = Q K^T on
// the tensor cores (mma.sync m16n8k16 BF16 -> FP32), online softmax in base 2
// with quad shuffles for the row max / sum, P re-used from the accumulator
// registers as the A operand of O += P V.  Stores O (BF16) and the row
// log-sum-exp (natural log, FP32) for the backward pass.
//
// Backward, deterministic (no atomics):
//   1. delta[row] = sum(dO * O) per (token, head);
//   2. dK/dV: one CTA per 128-key block of one kv head; it loops over the
//      query heads of its group and over the query blocks at or after the
//      diagonal in a fixed order, recomputing P^T = exp(S^T - lse) and
//      accumulating dV += P^T dO and dK += dS^T Q in registers;
//   3. dQ: one CTA per 128-query block of one query head, looping over key
//      blocks, dQ += dS K.
// dK and dQ leave through the inverse rotate-half RoPE rotation, so the
// gradient lands on the unrotated q/k projections.
//
// MegaTrain names "Attention and MLP kernels" inside its stateless templates
// (paperlayer.ai summary §A.4) without giving them; this design is the
// library's own.  Query head h reads kv head h * Hkv / Hq.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"

namespace mt {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct AttnDev {
  const bf16* qkv;
  long ld;
  int B, S, Hq, Hkv;
  bf16* o;
  long ldo;
  float* lse;
  const bf16* dout;
  const float* delta;
  bf16* dqkv;
  const float* cos_t;
  const float* sin_t;
  float scale;  // 1/sqrt(hd)
};

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

// Byte address of 16-byte chunk `ch` of row `row` in a swizzled [rows][HD] BF16 tile.
template <int HD>
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int row, int ch) {
  return base + row * (HD * 2) + ((ch ^ (row & 7)) << 4);
}

// Asynchronously copy rows [row0, row0 + nrows) of a head slice (row stride
// ld elements) into a swizzled shared tile; rows >= S are zero-filled.
template <int HD, int NT>
__device__ __forceinline__ void load_rows(bf16* s, const bf16* g, long ld, int row0, int nrows, int S) {
  constexpr int CPR = HD / 8;
  const uint32_t base = smem_u32(s);
  for (int i = threadIdx.x; i < nrows * CPR; i += NT) {
    const int r = i / CPR, c = i % CPR;
    const int gr = row0 + r;
    const bool ok = gr < S;
    const bf16* src = g + (long)(ok ? gr : 0) * ld + c * 8;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(tile_addr<HD>(base, r, c)), "l"(src),
                 "r"(ok ? 16 : 0)
                 : "memory");
  }
}

// A-operand fragments (16 rows x 16 k) from a swizzled tile: rows r0..r0+15, k chunk pair kk.
template <int HD>
__device__ __forceinline__ void lda_frag(uint32_t base, int r0, int kk, int lane, uint32_t (&a)[4]) {
  ldsm_x4(tile_addr<HD>(base, r0 + (lane & 15), 2 * kk + (lane >> 4)), a[0], a[1], a[2], a[3]);
}
// B-operand fragments for two n8 blocks (rows n0..n0+15 of the tile are the
// n index), k chunk pair kk: (b0,b1) for rows n0..+7 and (b2,b3) for n0+8..+15.
template <int HD>
__device__ __forceinline__ void ldb_frag(uint32_t base, int n0, int kk, int lane, uint32_t& b0, uint32_t& b1,
                                         uint32_t& b2, uint32_t& b3) {
  ldsm_x4(tile_addr<HD>(base, n0 + (lane & 7) + ((lane >> 4) << 3), 2 * kk + ((lane >> 3) & 1)), b0, b1, b2, b3);
}
// B-operand fragments where tile rows are the k index (keys/queries) and the
// n index runs along HD: k rows k0..k0+15, hd columns 16*nd2 .. +15.
template <int HD>
__device__ __forceinline__ void ldb_frag_t(uint32_t base, int k0, int nd2, int lane, uint32_t& b0, uint32_t& b1,
                                           uint32_t& b2, uint32_t& b3) {
  ldsm_x4_t(tile_addr<HD>(base, k0 + (lane & 7) + (((lane >> 3) & 1) << 3), 2 * nd2 + (lane >> 4)), b0, b1, b2, b3);
}

// ------------------------------------------------------------------ forward
template <int HD>
__global__ void __launch_bounds__(256) attn_fwd_kernel(AttnDev a) {
  constexpr int BM = 128, BN = 64, NT = 256;
  extern __shared__ __align__(128) uint8_t smem[];
  bf16* sQ = reinterpret_cast<bf16*>(smem);
  bf16* sK = sQ + BM * HD;
  bf16* sV = sK + 2 * BN * HD;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane >> 2, t = lane & 3;
  const int qb = gridDim.x - 1 - blockIdx.x;
  const int b = blockIdx.y / a.Hq, h = blockIdx.y % a.Hq;
  const int kvh = h * a.Hkv / a.Hq;
  const int S = a.S;
  const int q0 = qb * BM;
  const long tok0 = (long)b * S;
  const bf16* Qg = a.qkv + tok0 * a.ld + (long)h * HD;
  const bf16* Kg = a.qkv + tok0 * a.ld + (long)(a.Hq + kvh) * HD;
  const bf16* Vg = a.qkv + tok0 * a.ld + (long)(a.Hq + a.Hkv + kvh) * HD;
  const float sl2 = a.scale * kLog2e;

  load_rows<HD, NT>(sQ, Qg, a.ld, q0, BM, S);
  cp_async_commit();
  const int n_kb = min((S + BN - 1) / BN, (q0 + BM + BN - 1) / BN);
  load_rows<HD, NT>(sK, Kg, a.ld, 0, BN, S);
  load_rows<HD, NT>(sV, Vg, a.ld, 0, BN, S);
  cp_async_commit();

  cp_async_wait<1>();
  __syncthreads();
  const uint32_t qbase = smem_u32(sQ);
  uint32_t qf[HD / 16][4];
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) lda_frag<HD>(qbase, warp * 16, kk, lane, qf[kk]);

  float o[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
  const int row_a = q0 + warp * 16 + g, row_b = row_a + 8;

  for (int kb = 0; kb < n_kb; ++kb) {
    const int buf = kb & 1;
    if (kb + 1 < n_kb) {
      load_rows<HD, NT>(sK + (buf ^ 1) * BN * HD, Kg, a.ld, (kb + 1) * BN, BN, S);
      load_rows<HD, NT>(sV + (buf ^ 1) * BN * HD, Vg, a.ld, (kb + 1) * BN, BN, S);
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const uint32_t kbase = smem_u32(sK + buf * BN * HD);
    const uint32_t vbase = smem_u32(sV + buf * BN * HD);

    float s[BN / 8][4];
#pragma unroll
    for (int i = 0; i < BN / 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
      for (int nb2 = 0; nb2 < BN / 16; ++nb2) {
        uint32_t b0, b1, b2, b3;
        ldb_frag<HD>(kbase, nb2 * 16, kk, lane, b0, b1, b2, b3);
        mma16816(s[2 * nb2], qf[kk], b0, b1);
        mma16816(s[2 * nb2 + 1], qf[kk], b2, b3);
      }
    }
    // scale to base 2, causal mask, row max
    const int key0 = kb * BN;
    const bool need_mask = key0 + BN - 1 > q0 + warp * 16;
    float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
    for (int nb = 0; nb < BN / 8; ++nb) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = s[nb][e] * sl2;
        if (need_mask) {
          const int key = key0 + nb * 8 + 2 * t + (e & 1);
          const int row = e < 2 ? row_a : row_b;
          if (key > row) v = -INFINITY;
        }
        s[nb][e] = v;
      }
      mx_a = fmaxf(mx_a, fmaxf(s[nb][0], s[nb][1]));
      mx_b = fmaxf(mx_b, fmaxf(s[nb][2], s[nb][3]));
    }
    mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
    mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
    mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
    mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
    const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
    const float base_a = mn_a == -INFINITY ? 0.f : mn_a;
    const float base_b = mn_b == -INFINITY ? 0.f : mn_b;
    const float alpha_a = exp2f(m_a - base_a), alpha_b = exp2f(m_b - base_b);
    m_a = mn_a;
    m_b = mn_b;
    float rs_a = 0.f, rs_b = 0.f;
#pragma unroll
    for (int nb = 0; nb < BN / 8; ++nb) {
      s[nb][0] = exp2f(s[nb][0] - base_a);
      s[nb][1] = exp2f(s[nb][1] - base_a);
      s[nb][2] = exp2f(s[nb][2] - base_b);
      s[nb][3] = exp2f(s[nb][3] - base_b);
      rs_a += s[nb][0] + s[nb][1];
      rs_b += s[nb][2] + s[nb][3];
    }
    l_a = l_a * alpha_a + rs_a;
    l_b = l_b * alpha_b + rs_b;
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) {
      o[i][0] *= alpha_a;
      o[i][1] *= alpha_a;
      o[i][2] *= alpha_b;
      o[i][3] *= alpha_b;
    }
    // O += P V
#pragma unroll
    for (int kk2 = 0; kk2 < BN / 16; ++kk2) {
      uint32_t pa[4];
      pa[0] = pack_bf16x2(s[2 * kk2][0], s[2 * kk2][1]);
      pa[1] = pack_bf16x2(s[2 * kk2][2], s[2 * kk2][3]);
      pa[2] = pack_bf16x2(s[2 * kk2 + 1][0], s[2 * kk2 + 1][1]);
      pa[3] = pack_bf16x2(s[2 * kk2 + 1][2], s[2 * kk2 + 1][3]);
#pragma unroll
      for (int nd2 = 0; nd2 < HD / 16; ++nd2) {
        uint32_t b0, b1, b2, b3;
        ldb_frag_t<HD>(vbase, kk2 * 16, nd2, lane, b0, b1, b2, b3);
        mma16816(o[2 * nd2], pa, b0, b1);
        mma16816(o[2 * nd2 + 1], pa, b2, b3);
      }
    }
    __syncthreads();
  }
  // finalize
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
  const float inv_a = 1.f / l_a, inv_b = 1.f / l_b;
  if (row_a < S) {
    bf16* dst = a.o + (tok0 + row_a) * a.ldo + (long)h * HD;
#pragma unroll
    for (int nd = 0; nd < HD / 8; ++nd)
      *reinterpret_cast<uint32_t*>(dst + nd * 8 + 2 * t) = pack_bf16x2(o[nd][0] * inv_a, o[nd][1] * inv_a);
    if (t == 0) a.lse[((long)b * a.Hq + h) * S + row_a] = (m_a + log2f(l_a)) * kLn2;
  }
  if (row_b < S) {
    bf16* dst = a.o + (tok0 + row_b) * a.ldo + (long)h * HD;
#pragma unroll
    for (int nd = 0; nd < HD / 8; ++nd)
      *reinterpret_cast<uint32_t*>(dst + nd * 8 + 2 * t) = pack_bf16x2(o[nd][2] * inv_b, o[nd][3] * inv_b);
    if (t == 0) a.lse[((long)b * a.Hq + h) * S + row_b] = (m_b + log2f(l_b)) * kLn2;
  }
}

// ------------------------------------------------------------------ backward: delta
template <int HD>
__global__ void attn_delta_kernel(AttnDev a) {
  // one group of HD/8 threads per (token, head) row
  constexpr int G = HD / 8;
  const long gid = ((long)blockIdx.x * blockDim.x + threadIdx.x);
  const long row = gid / G;
  const int c = gid % G;
  const long T = (long)a.B * a.S;
  float acc = 0.f;
  const bool ok = row < T * a.Hq;
  long tok = 0;
  int h = 0;
  if (ok) {
    tok = row / a.Hq;
    h = row % a.Hq;
    const uint4 x = *reinterpret_cast<const uint4*>(a.dout + tok * a.ldo + (long)h * HD + c * 8);
    const uint4 y = *reinterpret_cast<const uint4*>(a.o + tok * a.ldo + (long)h * HD + c * 8);
    const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc += __uint_as_float(xs[j] << 16) * __uint_as_float(ys[j] << 16);
      acc += __uint_as_float(xs[j] & 0xFFFF0000u) * __uint_as_float(ys[j] & 0xFFFF0000u);
    }
  }
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o, G);
  if (ok && c == 0) {
    const long b = tok / a.S, s = tok % a.S;
    const_cast<float*>(a.delta)[(b * a.Hq + h) * a.S + s] = acc;
  }
}

// Inverse rotate-half RoPE on the 16 x HD accumulator fragment of one warp
// (rows row_a, row_b = positions), then BF16 store at dst rows.
template <int HD>
__device__ __forceinline__ void store_rows_rope_bwd(float (&acc)[HD / 8][4], float scale, const AttnDev& a,
                                                    bool rope, int pos_a, int pos_b, bf16* dst_a, bf16* dst_b,
                                                    int t) {
#pragma unroll
  for (int nd = 0; nd < HD / 8; ++nd)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nd][e] *= scale;
  if (rope) {
#pragma unroll
    for (int nd = 0; nd < HD / 16; ++nd) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = nd * 8 + 2 * t + (e & 1);  // < HD/2
        const int pos = e < 2 ? pos_a : pos_b;
        const float c = a.cos_t[(long)pos * (HD / 2) + i], sn = a.sin_t[(long)pos * (HD / 2) + i];
        const float d1 = acc[nd][e], d2 = acc[nd + HD / 16][e];
        acc[nd][e] = d1 * c + d2 * sn;
        acc[nd + HD / 16][e] = d2 * c - d1 * sn;
      }
    }
  }
  if (dst_a) {
#pragma unroll
    for (int nd = 0; nd < HD / 8; ++nd)
      *reinterpret_cast<uint32_t*>(dst_a + nd * 8 + 2 * t) = pack_bf16x2(acc[nd][0], acc[nd][1]);
  }
  if (dst_b) {
#pragma unroll
    for (int nd = 0; nd < HD / 8; ++nd)
      *reinterpret_cast<uint32_t*>(dst_b + nd * 8 + 2 * t) = pack_bf16x2(acc[nd][2], acc[nd][3]);
  }
}

// ------------------------------------------------------------------ backward: dK, dV
template <int HD>
__global__ void __launch_bounds__(256) attn_bwd_dkdv_kernel(AttnDev a) {
  constexpr int BN = 128, BM = 64, NT = 256;
  extern __shared__ __align__(128) uint8_t smem[];
  bf16* sK = reinterpret_cast<bf16*>(smem);
  bf16* sV = sK + BN * HD;
  bf16* sQ = sV + BN * HD;      // 2 buffers
  bf16* sdO = sQ + 2 * BM * HD;  // 2 buffers
  float* sL = reinterpret_cast<float*>(sdO + 2 * BM * HD);  // 2 x BM, log2 units
  float* sD = sL + 2 * BM;                                   // 2 x BM
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane >> 2, t = lane & 3;
  const int kb = blockIdx.x;
  const int b = blockIdx.y / a.Hkv, kvh = blockIdx.y % a.Hkv;
  const int S = a.S;
  const int k0 = kb * BN;
  const long tok0 = (long)b * S;
  const int G = a.Hq / a.Hkv;
  const float sl2 = a.scale * kLog2e;

  load_rows<HD, NT>(sK, a.qkv + tok0 * a.ld + (long)(a.Hq + kvh) * HD, a.ld, k0, BN, S);
  load_rows<HD, NT>(sV, a.qkv + tok0 * a.ld + (long)(a.Hq + a.Hkv + kvh) * HD, a.ld, k0, BN, S);
  cp_async_commit();

  float dk[HD / 8][4], dv[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) {
    dk[i][0] = dk[i][1] = dk[i][2] = dk[i][3] = 0.f;
    dv[i][0] = dv[i][1] = dv[i][2] = dv[i][3] = 0.f;
  }
  const uint32_t kbase = smem_u32(sK), vbase = smem_u32(sV);
  const int key_a = k0 + warp * 16 + g, key_b = key_a + 8;
  const int qb_first = k0 / BM;
  const int n_qb = (S + BM - 1) / BM;
  const int per_head = n_qb - qb_first;
  const int total = per_head * G;

  auto issue = [&](int it, int buf) {
    const int h = kvh * G + it / per_head;
    const int q0 = (qb_first + it % per_head) * BM;
    load_rows<HD, NT>(sQ + buf * BM * HD, a.qkv + tok0 * a.ld + (long)h * HD, a.ld, q0, BM, S);
    load_rows<HD, NT>(sdO + buf * BM * HD, a.dout + tok0 * a.ldo + (long)h * HD, a.ldo, q0, BM, S);
    for (int i = threadIdx.x; i < BM; i += NT) {
      const int q = q0 + i;
      const long idx = ((long)b * a.Hq + h) * S + q;
      sL[buf * BM + i] = q < S ? a.lse[idx] * kLog2e : INFINITY;
      sD[buf * BM + i] = q < S ? a.delta[idx] : 0.f;
    }
  };
  if (total > 0) issue(0, 0);
  cp_async_commit();

  for (int it = 0; it < total; ++it) {
    const int buf = it & 1;
    if (it + 1 < total) issue(it + 1, buf ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const int q0 = (qb_first + it % per_head) * BM;
    const uint32_t qbase = smem_u32(sQ + buf * BM * HD), obase = smem_u32(sdO + buf * BM * HD);
    const float* L = sL + buf * BM;
    const float* Dd = sD + buf * BM;

    // S^T = K_w Q^T and dP^T = V_w dO^T  (16 keys x BM queries)
    float st[BM / 8][4], dpt[BM / 8][4];
#pragma unroll
    for (int i = 0; i < BM / 8; ++i) {
      st[i][0] = st[i][1] = st[i][2] = st[i][3] = 0.f;
      dpt[i][0] = dpt[i][1] = dpt[i][2] = dpt[i][3] = 0.f;
    }
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
      uint32_t ka[4], va[4];
      lda_frag<HD>(kbase, warp * 16, kk, lane, ka);
      lda_frag<HD>(vbase, warp * 16, kk, lane, va);
#pragma unroll
      for (int nb2 = 0; nb2 < BM / 16; ++nb2) {
        uint32_t b0, b1, b2, b3;
        ldb_frag<HD>(qbase, nb2 * 16, kk, lane, b0, b1, b2, b3);
        mma16816(st[2 * nb2], ka, b0, b1);
        mma16816(st[2 * nb2 + 1], ka, b2, b3);
        ldb_frag<HD>(obase, nb2 * 16, kk, lane, b0, b1, b2, b3);
        mma16816(dpt[2 * nb2], va, b0, b1);
        mma16816(dpt[2 * nb2 + 1], va, b2, b3);
      }
    }
    // P^T, dS^T
#pragma unroll
    for (int nb = 0; nb < BM / 8; ++nb) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int qi = nb * 8 + 2 * t + (e & 1);
        const int q = q0 + qi;
        const int key = e < 2 ? key_a : key_b;
        float p = exp2f(st[nb][e] * sl2 - L[qi]);
        if (key > q || q >= S) p = 0.f;
        st[nb][e] = p;
        dpt[nb][e] = p * (dpt[nb][e] - Dd[qi]);
      }
    }
    // dV += P^T dO ; dK += dS^T Q
#pragma unroll
    for (int kk2 = 0; kk2 < BM / 16; ++kk2) {
      uint32_t pa[4], sa[4];
      pa[0] = pack_bf16x2(st[2 * kk2][0], st[2 * kk2][1]);
      pa[1] = pack_bf16x2(st[2 * kk2][2], st[2 * kk2][3]);
      pa[2] = pack_bf16x2(st[2 * kk2 + 1][0], st[2 * kk2 + 1][1]);
      pa[3] = pack_bf16x2(st[2 * kk2 + 1][2], st[2 * kk2 + 1][3]);
      sa[0] = pack_bf16x2(dpt[2 * kk2][0], dpt[2 * kk2][1]);
      sa[1] = pack_bf16x2(dpt[2 * kk2][2], dpt[2 * kk2][3]);
      sa[2] = pack_bf16x2(dpt[2 * kk2 + 1][0], dpt[2 * kk2 + 1][1]);
      sa[3] = pack_bf16x2(dpt[2 * kk2 + 1][2], dpt[2 * kk2 + 1][3]);
#pragma unroll
      for (int nd2 = 0; nd2 < HD / 16; ++nd2) {
        uint32_t b0, b1, b2, b3;
        ldb_frag_t<HD>(obase, kk2 * 16, nd2, lane, b0, b1, b2, b3);
        mma16816(dv[2 * nd2], pa, b0, b1);
        mma16816(dv[2 * nd2 + 1], pa, b2, b3);
        ldb_frag_t<HD>(qbase, kk2 * 16, nd2, lane, b0, b1, b2, b3);
        mma16816(dk[2 * nd2], sa, b0, b1);
        mma16816(dk[2 * nd2 + 1], sa, b2, b3);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  const long ldg = a.ld;
  bf16* dka = key_a < S ? a.dqkv + (tok0 + key_a) * ldg + (long)(a.Hq + kvh) * HD : nullptr;
  bf16* dkb = key_b < S ? a.dqkv + (tok0 + key_b) * ldg + (long)(a.Hq + kvh) * HD : nullptr;
  bf16* dva = key_a < S ? a.dqkv + (tok0 + key_a) * ldg + (long)(a.Hq + a.Hkv + kvh) * HD : nullptr;
  bf16* dvb = key_b < S ? a.dqkv + (tok0 + key_b) * ldg + (long)(a.Hq + a.Hkv + kvh) * HD : nullptr;
  const bool rope = a.cos_t != nullptr;
  store_rows_rope_bwd<HD>(dk, a.scale, a, rope, key_a < S ? key_a : 0, key_b < S ? key_b : 0, dka, dkb, t);
  store_rows_rope_bwd<HD>(dv, 1.0f, a, false, 0, 0, dva, dvb, t);
}

// ------------------------------------------------------------------ backward: dQ
template <int HD>
__global__ void __launch_bounds__(256) attn_bwd_dq_kernel(AttnDev a) {
  constexpr int BM = 128, BN = 64, NT = 256;
  extern __shared__ __align__(128) uint8_t smem[];
  bf16* sQ = reinterpret_cast<bf16*>(smem);
  bf16* sdO = sQ + BM * HD;
  bf16* sK = sdO + BM * HD;  // 2 buffers
  bf16* sV = sK + 2 * BN * HD;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane >> 2, t = lane & 3;
  const int qb = gridDim.x - 1 - blockIdx.x;
  const int b = blockIdx.y / a.Hq, h = blockIdx.y % a.Hq;
  const int kvh = h * a.Hkv / a.Hq;
  const int S = a.S;
  const int q0 = qb * BM;
  const long tok0 = (long)b * S;
  const float sl2 = a.scale * kLog2e;
  const bf16* Kg = a.qkv + tok0 * a.ld + (long)(a.Hq + kvh) * HD;
  const bf16* Vg = a.qkv + tok0 * a.ld + (long)(a.Hq + a.Hkv + kvh) * HD;

  load_rows<HD, NT>(sQ, a.qkv + tok0 * a.ld + (long)h * HD, a.ld, q0, BM, S);
  load_rows<HD, NT>(sdO, a.dout + tok0 * a.ldo + (long)h * HD, a.ldo, q0, BM, S);
  cp_async_commit();
  const int n_kb = min((S + BN - 1) / BN, (q0 + BM + BN - 1) / BN);
  load_rows<HD, NT>(sK, Kg, a.ld, 0, BN, S);
  load_rows<HD, NT>(sV, Vg, a.ld, 0, BN, S);
  cp_async_commit();

  const int row_a = q0 + warp * 16 + g, row_b = row_a + 8;
  const long lrow = ((long)b * a.Hq + h) * S;
  const float L_a = row_a < S ? a.lse[lrow + row_a] * kLog2e : INFINITY;
  const float L_b = row_b < S ? a.lse[lrow + row_b] * kLog2e : INFINITY;
  const float D_a = row_a < S ? a.delta[lrow + row_a] : 0.f;
  const float D_b = row_b < S ? a.delta[lrow + row_b] : 0.f;
  const uint32_t qbase = smem_u32(sQ), obase = smem_u32(sdO);

  float dq[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) dq[i][0] = dq[i][1] = dq[i][2] = dq[i][3] = 0.f;

  for (int kb = 0; kb < n_kb; ++kb) {
    const int buf = kb & 1;
    if (kb + 1 < n_kb) {
      load_rows<HD, NT>(sK + (buf ^ 1) * BN * HD, Kg, a.ld, (kb + 1) * BN, BN, S);
      load_rows<HD, NT>(sV + (buf ^ 1) * BN * HD, Vg, a.ld, (kb + 1) * BN, BN, S);
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const uint32_t kbase = smem_u32(sK + buf * BN * HD), vbase = smem_u32(sV + buf * BN * HD);
    float s[BN / 8][4], dp[BN / 8][4];
#pragma unroll
    for (int i = 0; i < BN / 8; ++i) {
      s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
      dp[i][0] = dp[i][1] = dp[i][2] = dp[i][3] = 0.f;
    }
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
      uint32_t qa[4], oa[4];
      lda_frag<HD>(qbase, warp * 16, kk, lane, qa);
      lda_frag<HD>(obase, warp * 16, kk, lane, oa);
#pragma unroll
      for (int nb2 = 0; nb2 < BN / 16; ++nb2) {
        uint32_t b0, b1, b2, b3;
        ldb_frag<HD>(kbase, nb2 * 16, kk, lane, b0, b1, b2, b3);
        mma16816(s[2 * nb2], qa, b0, b1);
        mma16816(s[2 * nb2 + 1], qa, b2, b3);
        ldb_frag<HD>(vbase, nb2 * 16, kk, lane, b0, b1, b2, b3);
        mma16816(dp[2 * nb2], oa, b0, b1);
        mma16816(dp[2 * nb2 + 1], oa, b2, b3);
      }
    }
    const int key0 = kb * BN;
#pragma unroll
    for (int nb = 0; nb < BN / 8; ++nb) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = key0 + nb * 8 + 2 * t + (e & 1);
        const int row = e < 2 ? row_a : row_b;
        float p = exp2f(s[nb][e] * sl2 - (e < 2 ? L_a : L_b));
        if (key > row) p = 0.f;
        s[nb][e] = p * (dp[nb][e] - (e < 2 ? D_a : D_b));  // dS
      }
    }
    // dQ += dS K
#pragma unroll
    for (int kk2 = 0; kk2 < BN / 16; ++kk2) {
      uint32_t sa[4];
      sa[0] = pack_bf16x2(s[2 * kk2][0], s[2 * kk2][1]);
      sa[1] = pack_bf16x2(s[2 * kk2][2], s[2 * kk2][3]);
      sa[2] = pack_bf16x2(s[2 * kk2 + 1][0], s[2 * kk2 + 1][1]);
      sa[3] = pack_bf16x2(s[2 * kk2 + 1][2], s[2 * kk2 + 1][3]);
#pragma unroll
      for (int nd2 = 0; nd2 < HD / 16; ++nd2) {
        uint32_t b0, b1, b2, b3;
        ldb_frag_t<HD>(kbase, kk2 * 16, nd2, lane, b0, b1, b2, b3);
        mma16816(dq[2 * nd2], sa, b0, b1);
        mma16816(dq[2 * nd2 + 1], sa, b2, b3);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  bf16* da = row_a < S ? a.dqkv + (tok0 + row_a) * a.ld + (long)h * HD : nullptr;
  bf16* db = row_b < S ? a.dqkv + (tok0 + row_b) * a.ld + (long)h * HD : nullptr;
  store_rows_rope_bwd<HD>(dq, a.scale, a, a.cos_t != nullptr, row_a < S ? row_a : 0, row_b < S ? row_b : 0, da,
                          db, t);
}

template <int HD>
constexpr int fwd_smem() {
  return (128 * HD + 4 * 64 * HD) * 2;
}
template <int HD>
constexpr int dkdv_smem() {
  return (2 * 128 * HD + 4 * 64 * HD) * 2 + 4 * 64 * 4;
}
template <int HD>
constexpr int dq_smem() {
  return (2 * 128 * HD + 4 * 64 * HD) * 2;
}

AttnDev to_dev(const AttnArgs& x) {
  AttnDev a;
  a.qkv = x.qkv;
  a.ld = x.ldqkv;
  a.B = x.batch;
  a.S = x.seq;
  a.Hq = x.n_heads;
  a.Hkv = x.n_kv_heads;
  a.o = x.o;
  a.ldo = x.ldo;
  a.lse = x.lse;
  a.dout = x.dout;
  a.delta = x.delta;
  a.dqkv = x.dqkv;
  a.cos_t = x.rope_cos;
  a.sin_t = x.rope_sin;
  a.scale = 1.0f / sqrtf((float)x.head_dim);
  return a;
}

template <int HD>
int fwd_impl(const AttnArgs& x, cudaStream_t s) {
  static bool init = false;
  if (!init) {
    cudaFuncSetAttribute(attn_fwd_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, fwd_smem<HD>());
    init = true;
  }
  AttnDev a = to_dev(x);
  dim3 grid((x.seq + 127) / 128, x.batch * x.n_heads);
  attn_fwd_kernel<HD><<<grid, 256, fwd_smem<HD>(), s>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

template <int HD>
int bwd_impl(const AttnArgs& x, cudaStream_t s) {
  AttnDev a = to_dev(x);
  const long rows = (long)x.batch * x.seq * x.n_heads;
  const long threads = rows * (HD / 8);
  attn_delta_kernel<HD><<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(a);
  if (cudaPeekAtLastError() != cudaSuccess) return -4;
  return launch_attn_bwd_tc_main(x, s);
}

}  // namespace

const char* attn_check(const AttnArgs& x) {
  if (x.head_dim != 64 && x.head_dim != 128) return "attention: head_dim must be 64 or 128";
  if (x.batch <= 0 || x.seq <= 0 || x.n_heads <= 0 || x.n_kv_heads <= 0) return "attention: empty shape";
  if (x.n_heads % x.n_kv_heads) return "attention: n_heads must be a multiple of n_kv_heads";
  if (x.ldqkv % 8 || x.ldo % 8) return "attention: leading dimensions must be multiples of 8";
  if (x.ldqkv < (long)(x.n_heads + 2 * x.n_kv_heads) * x.head_dim) return "attention: ldqkv too small";
  if (x.ldo < (long)x.n_heads * x.head_dim) return "attention: ldo too small";
  if (!x.qkv || !x.o || !x.lse) return "attention: null q/k/v, o or lse";
  if ((reinterpret_cast<uintptr_t>(x.qkv) | reinterpret_cast<uintptr_t>(x.o)) & 15) return "attention: misaligned";
  return nullptr;
}

int launch_attn_fwd(const AttnArgs& x, cudaStream_t s) {
  if (attn_check(x)) return -1;
  return launch_attn_fwd_tc(x, s);
}

int launch_attn_bwd(const AttnArgs& x, cudaStream_t s) {
  if (attn_check(x)) return -1;
  if (!x.dout || !x.delta || !x.dqkv) return -1;
  if ((reinterpret_cast<uintptr_t>(x.dout) | reinterpret_cast<uintptr_t>(x.dqkv)) & 15) return -1;
  return x.head_dim == 128 ? bwd_impl<128>(x, s) : bwd_impl<64>(x, s);
}

}  // namespace mt
