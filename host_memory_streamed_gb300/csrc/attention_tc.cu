// Causal grouped-query flash attention forward on the 5th-generation tensor
// cores: S = Q K^T and O += P V with tcgen05.mma, S and O accumulated in
// TMEM, Q/K/V tiles brought in by TMA.
//
// One CTA per (128 queries, query head, batch), started longest causal row
// first within chunks of a few heads (causal_cta_order); 10 warps:
//   warp 0      TMA: Q once; K and V blocks of 128 keys into a 3-stage ring
//               (one tensor map over the packed q|k|v projection buffer).
//   warp 1      MMA (one thread): S_j = Q K_j^T into TMEM buffer j%2; once
//               the softmax has written P_j (BF16, over S_j's first 64
//               columns) O_{j%2} += P_j V_j with P read from TMEM as the A
//               operand and V as an MN-major operand straight from its
//               [keys][head_dim] tile; then S_{j+2} into the same buffer.
//   warps 2..9  softmax in two groups of four warps: group 0 takes the even
//               key blocks, group 1 the odd ones, each with its own running
//               maximum, row sum and O accumulator in TMEM, so that one
//               group's exponentials overlap the tensor core's work on the
//               other group's block.  Thread <-> query row (TMEM lane); each
//               thread reads its whole score row, takes the maximum and
//               exponentiates all 128 keys (f32x2 arithmetic, SFU exp2).  A
//               group's maximum is only moved (and its O rescaled in TMEM)
//               when it grows by more than a factor 2^8.  At the end the two
//               groups' (max, sum) pairs meet in shared memory and each group
//               writes half of the output columns from both accumulators.
// Every mbarrier wait is bounded; on expiry the kernel records
// kStatusAttnFwdTimeout in the status word and unwinds.
//
// MegaTrain's templates hold "Attention and MLP kernels" (paperlayer.ai
// summary §A.4) without specifying them; this kernel is the library's own.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"

namespace mt {

// Defined in gemm.cu: 2-D BF16 tensor map with 64-column x box_rows boxes, 128-byte swizzle.
bool make_tmap_bf16(CUtensorMap* m, const void* base, long rows, long cols, long ld, int box_rows);

namespace {

constexpr int TA_BM = 128, TA_BN = 128, TA_THREADS = 320;
constexpr int kSoftmaxWarps = 8;  // barriers the softmax warps arrive on count warps (one arrival each)
constexpr float kLog2eF = 1.4426950408889634f;
constexpr float kLn2F = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8

// Order of the CTAs of a causal grid whose x is the block along the sequence
// (x = 0 the longest causal work) and whose y is a row of blocks that share
// operands (a head or a kv-head group).  The block scheduler starts CTAs in
// linear block order; taken row by row, every row's longest CTA would start
// up to one row's span late and the kernel would end on one of them.  The
// grid is cut into chunks of `chunk` rows and, within a chunk, walks
// x-major: the x = 0 CTAs of all its rows first, then x = 1, ...  So the
// longest CTAs of a chunk start first and short ones fill the end, while the
// CTAs running at one time still come from a few rows, whose shared
// operands stay in L2.  chunk = 1 is plain row-by-row order.
__device__ __forceinline__ void causal_cta_order(int chunk, int& x, int& y) {
  const int nx = (int)gridDim.x, ny = (int)gridDim.y;
  const int lin = (int)blockIdx.y * nx + (int)blockIdx.x;  // < nx * ny
  const int y0 = lin / (chunk * nx) * chunk;              // first row of this CTA's chunk
  const int cy = min(chunk, ny - y0);                     // rows in the chunk (the last may be short)
  const int idx = lin - y0 * nx;                          // < cy * nx
  x = idx / cy;
  y = y0 + idx % cy;
}

// Rows per chunk for a grid of nx x ny CTAs: about `ctas` CTAs per chunk, at
// least one row.  The backward kernels take 256 (1.7 waves of one CTA per
// SM): their longest CTAs run hundreds of key or query blocks and need the
// wider chunk to balance.  The forward's CTAs are short, and 128 (fewer
// heads' K/V in L2 at a time) measured faster at every width tried.
inline int causal_chunk_rows(int nx, int ny, int ctas) {
  return std::max(1, std::min(ny, ctas / std::max(1, nx)));
}

template <int HD>
struct TaCfg {
  static constexpr int BOX = 128 * 128;          // one 64-column box of 128 rows, bytes
  static constexpr int Q_BYTES = 128 * HD * 2;   // HD/64 boxes
  static constexpr int KV_BYTES = 128 * HD * 2;  // K or V block
  static constexpr int STAGES = 3;               // K/V ring depth
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;             // STAGES blocks
  static constexpr int OFF_V = OFF_K + STAGES * KV_BYTES;   // STAGES blocks
  static constexpr int OFF_BAR = OFF_V + STAGES * KV_BYTES;  // the final (max, sum) exchange reuses the K ring
  static constexpr int SMEM = OFF_BAR + 256 + 1024;         // barriers + alignment slack
};

struct TaParams {
  int B, S, Hq, Hkv;
  bf16* o;
  long ldo;
  float* lse;
  float sl2;  // softmax scale * log2(e)
  int chunk;  // rows of the grid per chunk of the CTA order (causal_cta_order)
  int* status;
};

__device__ __forceinline__ uint32_t pack2bf(float a, float b) {
  __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&p);
}

// ---- FP32 pairs: one f32x2 instruction does the work of two scalar ones.
__device__ __forceinline__ uint64_t f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2split(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

template <int HD>
__global__ void __launch_bounds__(TA_THREADS, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, TaParams p) {
  using C = TaCfg<HD>;
  constexpr int NS = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bar + 0;
  uint64_t* kv_full = bar + 1;           // [NS]
  uint64_t* kv_empty = bar + 1 + NS;     // [NS]
  uint64_t* s_full = bar + 1 + 2 * NS;   // [2] S_j in TMEM buffer j & 1
  uint64_t* p_full = bar + 3 + 2 * NS;   // [2] P_j stored over S_j, O_{j&1} rescaled (the group's 4 warps)
  uint64_t* pv_done = bar + 5 + 2 * NS;  // [2] O_{j&1} += P_j V_j done
  uint64_t* o_full = bar + 7 + 2 * NS;   // every MMA done
  uint64_t* ml_ready = bar + 8 + 2 * NS; // both groups' (m, l) of every row in shared memory (8 warps)
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bar + 9 + 2 * NS);
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  int bx, by;
  causal_cta_order(p.chunk, bx, by);
  const int qb = gridDim.x - 1 - bx;  // longest causal rows first
  const int b = by / p.Hq, h = by % p.Hq;
  const int kvh = h * p.Hkv / p.Hq;
  const int S = p.S;
  const int q0 = qb * TA_BM;
  const int n_kb = min((S + TA_BN - 1) / TA_BN, (q0 + TA_BM + TA_BN - 1) / TA_BN);
  const int row0 = b * S;  // token row of position 0 in the packed buffer
  const int colQ = h * HD, colK = (p.Hq + kvh) * HD, colV = (p.Hq + p.Hkv + kvh) * HD;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(q_full, 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], kSoftmaxWarps / 2);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(o_full, 1);
    mbar_init(ml_ready, kSoftmaxWarps);
    fence_barrier_init();
    tma_prefetch_desc(&tm_qkv);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // S_j at 128 * (j & 1); the two groups' O accumulators at 256 and 256 + HD
  auto tO = [&](int g) { return tmem + 256u + (uint32_t)(g * HD); };

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, C::Q_BYTES);
#pragma unroll
      for (int i = 0; i < HD / 64; ++i) tma_load_2d(sQ + i * C::BOX, &tm_qkv, colQ + 64 * i, row0 + q0, q_full);
      int pend[NS];
      for (int s = 0; s < NS; ++s) pend[s] = -1;
      for (int j = 0; j < n_kb && !abort_flag; ++j) {
        const int s = j % NS;
        if (j >= NS && !mbar_wait(&kv_empty[s], ((j / NS) - 1) & 1)) {
          set_status(p.status, kStatusAttnFwdTimeout * 1000 + 100 + min(j, 99));
          abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&kv_full[s], 2 * C::KV_BYTES);
#pragma unroll
        for (int i = 0; i < HD / 64; ++i) {
          tma_load_2d(sK + s * C::KV_BYTES + i * C::BOX, &tm_qkv, colK + 64 * i, row0 + j * TA_BN, &kv_full[s]);
          tma_load_2d(sV + s * C::KV_BYTES + i * C::BOX, &tm_qkv, colV + 64 * i, row0 + j * TA_BN, &kv_full[s]);
        }
        pend[s] = (j / NS) & 1;
      }
      // every issued load must land before exit
      if (!mbar_wait(q_full, 0)) set_status(p.status, kStatusAttnFwdTimeout * 1000 + 200);
      for (int s = 0; s < NS; ++s)
        if (pend[s] >= 0 && !mbar_wait(&kv_full[s], (uint32_t)pend[s]))
          set_status(p.status, kStatusAttnFwdTimeout * 1000 + 300 + s);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_qk = idesc_bf16_f32(128, 128);
      const uint32_t id_pv = idesc_bf16_f32(128, HD) | (1u << 16);  // P (TMEM) x V (MN-major)
      int site = 0;
      bool ok = mbar_wait(q_full, 0);
      if (!ok) site = 400;
      auto issue_qk = [&](int j) {
        const int s = j % NS;
        if (!mbar_wait(&kv_full[s], (j / NS) & 1)) {
          site = 500 + min(j, 99);
          return false;
        }
        tc_fence_after();
        const uint64_t da = smem_desc_kmajor_sw128(sQ), db = smem_desc_kmajor_sw128(sK + s * C::KV_BYTES);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          tc_mma_bf16(tmem + 128u * (uint32_t)(j & 1), da + desc_step(kk, C::BOX), db + desc_step(kk, C::BOX), id_qk,
                      kk > 0 ? 1u : 0u);
        tc_commit(&s_full[j & 1]);
        return true;
      };
      if (ok) ok = issue_qk(0);
      if (ok && n_kb > 1) ok = issue_qk(1);
      for (int j = 0; ok && j < n_kb; ++j) {
        const int g = j & 1;
        if (!mbar_wait(&p_full[g], (j >> 1) & 1)) {
          site = 600 + min(j, 99);
          ok = false;
          break;
        }
        tc_fence_after();
        const int s = j % NS;
        const uint64_t vdesc = smem_desc_mnmajor_sw128(sV + s * C::KV_BYTES, C::BOX);
        const uint32_t pa = tmem + 128u * (uint32_t)g;
#pragma unroll
        for (int kk = 0; kk < TA_BN / 16; ++kk)
          tc_mma_bf16_ts(tO(g), pa + kk * 8, vdesc + (uint64_t)(kk * (2048 >> 4)), id_pv, (j >= 2 || kk > 0) ? 1u : 0u);
        tc_commit(&kv_empty[s]);
        tc_commit(&pv_done[g]);
        // S_{j+2} overwrites P_j: issued after the MMAs that read it
        if (j + 2 < n_kb && !issue_qk(j + 2)) {
          ok = false;
          break;
        }
      }
      if (ok) {
        tc_commit(o_full);
      } else {
        set_status(p.status, kStatusAttnFwdTimeout * 1000 + site);
        abort_flag = 1;
      }
    }
  } else {
    // softmax warps: group g = 0 (warps 2..5) takes the even key blocks, g = 1
    // (warps 6..9) the odd ones; thread <-> query row r (TMEM lane r), all
    // 128 keys of its group's blocks, its own running maximum, row sum and O
    // accumulator.  While one group exponentiates, the tensor core works on
    // the other group's blocks.
    const int quarter = warp & 3;
    const int g = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const int qrow = q0 + r;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tOg = tO(g) + lane_off;
    float m = -INFINITY, l = 0.f;  // running maximum (raw score units) and row sum of this group's blocks
    bool ok = true;
    int site = 0;
    for (int j = g; j < n_kb; j += 2) {
      const uint32_t tS = tmem + 128u * (uint32_t)g + lane_off;
      if (!mbar_wait_warp(&s_full[g], (j >> 1) & 1)) {
        site = 700 + min(j, 99);
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t x[TA_BN];
#pragma unroll
      for (int c = 0; c < TA_BN / 64; ++c)
        tmem_ld_32x32b_x64(tS + c * 64, *reinterpret_cast<uint32_t(*)[64]>(x + c * 64));
      tmem_wait_ld_regs(x);
      const int k0 = j * TA_BN;
      if (k0 + TA_BN - 1 > q0) {  // block touches the diagonal
#pragma unroll
        for (int c = 0; c < TA_BN; ++c)
          if (k0 + c > qrow) x[c] = __float_as_uint(-INFINITY);
      }
      float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
      for (int c = 0; c < TA_BN; c += 4) {
        mxa = fmax3(mxa, __uint_as_float(x[c]), __uint_as_float(x[c + 1]));
        mxb = fmax3(mxb, __uint_as_float(x[c + 2]), __uint_as_float(x[c + 3]));
      }
      const float mx = fmaxf(mxa, mxb);
      // scores are raw q.k; probabilities exp2((x - m) * scale * log2 e)
      const float m_new = fmaxf(m, mx);
      const bool rescale = (m == -INFINITY) || ((m_new - m) * p.sl2 > kRescaleThreshold);
      float alpha = 1.f;
      if (rescale) {
        alpha = (m == -INFINITY) ? 0.f : ex2_approx((m - m_new) * p.sl2);
        m = m_new;
      }
      const float nb = (m == -INFINITY) ? 0.f : -m * p.sl2;
      const uint64_t sl2x2 = f2(p.sl2, p.sl2), nbx2 = f2(nb, nb);
      // two packed partial row sums: four independent chains of adds
      uint64_t acc[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
      // P_j as packed BF16 pairs over the first 64 columns of S_j (this warp's
      // own lanes, already read), one half of the keys at a time; the register
      // arrays are indexed with constants only
      auto exp_half = [&](auto half) {
        constexpr int K0 = decltype(half)::value * (TA_BN / 2);
        uint32_t pk[TA_BN / 4];
#pragma unroll
        for (int e = 0; e < TA_BN / 4; ++e) {
          const uint64_t t =
              fma2(f2(__uint_as_float(x[K0 + 2 * e]), __uint_as_float(x[K0 + 2 * e + 1])), sl2x2, nbx2);
          float t0, t1;
          f2split(t, t0, t1);
          const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
          acc[e & 1] = add2(acc[e & 1], f2(p0, p1));
          pk[e] = pack2bf(p0, p1);
        }
        tmem_st_32x32b_x32(tS + decltype(half)::value * 32, pk);
      };
      exp_half(std::integral_constant<int, 0>{});
      exp_half(std::integral_constant<int, 1>{});
      float a0, a1, b0, b1;
      f2split(acc[0], a0, a1);
      f2split(acc[1], b0, b1);
      l = l * alpha + ((a0 + a1) + (b0 + b1));
      // O_g holds the sum over this group's earlier blocks; tcgen05.ld/st are
      // warp-collective, so the whole warp rescales when any of its rows must
      // (alpha = 1 for the others), after the previous P V into O_g is done.
      if (__any_sync(0xffffffffu, rescale && j >= 2)) {
        if (!mbar_wait_warp(&pv_done[g], ((j - 2) >> 1) & 1)) {
          site = 900 + min(j, 99);
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tOg + c * 32, v);
          tmem_wait_ld_regs(v);
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
          tmem_st_32x32b_x32(tOg + c * 32, v);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(&p_full[g]);
    }
    ok = __all_sync(0xffffffffu, ok);
    if (ok && !mbar_wait_warp(o_full, 0)) {
      site = 999;
      ok = false;
    }
    // The two groups' (m, l) meet in shared memory (the K ring is free once
    // every MMA is done); each group then writes half of the output columns.
    float* sML = reinterpret_cast<float*>(sK);  // [2 groups][m, l][128 rows]
    if (ok) {
      sML[g * 256 + r] = m;
      sML[g * 256 + 128 + r] = l;
      mbar_arrive_warp(ml_ready);
      if (!mbar_wait_warp(ml_ready, 0)) {
        site = 998;
        ok = false;
      }
    }
    if (ok) {
      tc_fence_after();
      const float m0 = sML[r], l0 = sML[128 + r], m1 = sML[256 + r], l1 = sML[384 + r];
      const float mm = fmaxf(m0, m1);
      // a group that saw no key of this row (or no block at all) contributes nothing
      const float c0 = (m0 == -INFINITY) ? 0.f : ex2_approx((m0 - mm) * p.sl2);
      const float c1 = (m1 == -INFINITY) ? 0.f : ex2_approx((m1 - mm) * p.sl2);
      const float lt = l0 * c0 + l1 * c1;
      const float inv = 1.f / lt;
      const float w0 = c0 * inv, w1 = c1 * inv;
      const bool valid = qrow < S;
      bf16* dst = p.o + (long)(row0 + qrow) * p.ldo + (long)h * HD + g * (HD / 2);
#pragma unroll
      for (int c = 0; c < HD / 64; ++c) {
        uint32_t va[32], vb[32];
        tmem_ld_32x32b_x32(tO(0) + lane_off + g * (HD / 2) + c * 32, va);
        tmem_ld_32x32b_x32(tO(1) + lane_off + g * (HD / 2) + c * 32, vb);
        tmem_wait_ld_regs(va);
        tmem_wait_ld_regs(vb);
        float f[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          // select, not multiply: an O accumulator that was never written holds garbage
          const float o0 = __uint_as_float(va[e]) * w0;
          f[e] = (c1 != 0.f) ? fmaf(__uint_as_float(vb[e]), w1, o0) : o0;
        }
        if (valid) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            d4[q] = make_uint4(pack2bf(f[8 * q], f[8 * q + 1]), pack2bf(f[8 * q + 2], f[8 * q + 3]),
                               pack2bf(f[8 * q + 4], f[8 * q + 5]), pack2bf(f[8 * q + 6], f[8 * q + 7]));
        }
      }
      if (valid && g == 0) p.lse[((long)b * p.Hq + h) * S + qrow] = mm * (p.sl2 * kLn2F) + logf(lt);
    } else {
      set_status(p.status, kStatusAttnFwdTimeout * 1000 + site);
      abort_flag = 1;
    }
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int HD>
int launch_tc(const AttnArgs& x, cudaStream_t s) {
  using C = TaCfg<HD>;
  static bool init = false;
  if (!init) {
    if (cudaFuncSetAttribute(attn_fwd_tc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
        cudaSuccess)
      return -2;
    init = true;
  }
  CUtensorMap tm;
  const long T = (long)x.batch * x.seq;
  if (!make_tmap_bf16(&tm, x.qkv, T, (long)(x.n_heads + 2 * x.n_kv_heads) * HD, x.ldqkv, 128)) return -3;
  TaParams p;
  p.B = x.batch;
  p.S = x.seq;
  p.Hq = x.n_heads;
  p.Hkv = x.n_kv_heads;
  p.o = x.o;
  p.ldo = x.ldo;
  p.lse = x.lse;
  p.sl2 = kLog2eF / sqrtf((float)HD);
  p.status = x.status;
  dim3 grid((x.seq + TA_BM - 1) / TA_BM, x.batch * x.n_heads);
  p.chunk = causal_chunk_rows((int)grid.x, (int)grid.y, 128);
  attn_fwd_tc_kernel<HD><<<grid, TA_THREADS, C::SMEM, s>>>(tm, p);
  return launch_result();
}

}  // namespace

int launch_attn_fwd_tc(const AttnArgs& x, cudaStream_t s) {
  if (attn_check(x)) return -1;
  return x.head_dim == 128 ? launch_tc<128>(x, s) : launch_tc<64>(x, s);
}

}  // namespace mt

// ============================================================================
// Backward on the tensor cores (deterministic, no atomics).
//
// Both kernels work on 128 x 128 score blocks, so every tcgen05.mma has
// N = 128 (narrower MMAs were bound by shared-memory operand bandwidth), and
// keep the BF16 probabilities / score gradients in TMEM, written in place
// over the FP32 scores they came from, where the tensor core reads them as
// its A operand (tcgen05.mma with A in TMEM: lane = row, 32-bit column j =
// elements 2j and 2j+1 of the row).
//
// dK/dV kernel: one CTA per (128-key block, kv head, batch).  K and V of the
// block stay in shared memory; the TMA warp streams 128-query blocks of Q and
// dO (2 stages) for every query head of the group, in a fixed order.  Per
// query block (TMEM: S^T 0..127, dP^T 128..255, dV, dK accumulators above):
//   S^T = K Q^T, dP^T = V dO^T
//   P^T = exp(S^T * scale - lse[q])          -> BF16 over S^T's columns
//   dS^T = P^T * (dP^T - delta[q])           -> BF16 over dP^T's columns
//   dV += P^T dO, dK += dS^T Q               (dO, Q read MN-major from the
//                                             tiles used K-major above)
// The tensor core runs dV_i, S^T_{i+1}, dK_i, dP^T_{i+1} in that order, so
// each score block is overwritten only after its probabilities were used.
// dQ kernel: one CTA per (128-query block, query head, batch), streaming
// 128-key blocks of K (3 stages) and V (2 stages): S = Q K^T, dP = dO V^T
// (two TMEM buffers), dS = P * (dP - delta) -> BF16 over dP's columns,
// dQ += dS K.  S is released as soon as every softmax thread holds its row in
// registers, so S_{j+1} and dP_{j+1} run while the softmax works on block j.
// dK and dQ are scaled by 1/sqrt(hd) and leave through the inverse RoPE
// rotation when tables are given.
// ============================================================================
namespace mt {
namespace {

constexpr int TB_THREADS = 320;  // TMA warp, MMA warp, 8 softmax warps (two per TMEM lane group)

struct TbParams {
  int B, S, Hq, Hkv;
  const float* lse;
  const float* delta;
  bf16* dqkv;
  long ld;  // of dqkv (= ld of qkv)
  const float* cos_t;
  const float* sin_t;
  float sl2;    // scale * log2(e)
  float scale;  // 1/sqrt(hd)
  int ld_bulk;  // lse/delta rows 16-byte aligned (S % 4 == 0): whole query blocks arrive by bulk copy
  int chunk_kv;  // rows per chunk of the dK/dV grid's CTA order (causal_cta_order)
  int chunk_q;   // the same for the dQ grid
  int* status;
};

// 32 lanes x 16 consecutive 32-bit TMEM columns.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// Half of an accumulator row held by one of the two warps that share a TMEM
// lane group: columns [h*W, h*W+W) and [HD/2 + h*W, +W) with W = HD/4, so the
// rotate-half pairs (i, i + HD/2) stay in one thread.  Scales, applies the
// inverse RoPE rotation when tables are given, stores BF16.
template <int HD>
__device__ __forceinline__ void store_half_row(uint32_t taddr, int h, float scale, bool rope, const float* cs,
                                               const float* sn, bf16* dst) {
  constexpr int W = HD / 4;
  float a[W], c2[W];
  if constexpr (W == 32) {
    uint32_t r0[32], r1[32];
    tmem_ld_32x32b_x32(taddr + h * W, r0);
    tmem_ld_32x32b_x32(taddr + HD / 2 + h * W, r1);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < W; ++e) {
      a[e] = __uint_as_float(r0[e]) * scale;
      c2[e] = __uint_as_float(r1[e]) * scale;
    }
  } else {
    uint32_t r0[16], r1[16];
    tmem_ld_32x32b_x16(taddr + h * W, r0);
    tmem_ld_32x32b_x16(taddr + HD / 2 + h * W, r1);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < W; ++e) {
      a[e] = __uint_as_float(r0[e]) * scale;
      c2[e] = __uint_as_float(r1[e]) * scale;
    }
  }
  if (rope) {
#pragma unroll
    for (int e = 0; e < W; ++e) {
      const int i = h * W + e;
      const float c = cs[i], sv = sn[i];
      const float d1 = a[e], d2 = c2[e];
      a[e] = d1 * c + d2 * sv;
      c2[e] = d2 * c - d1 * sv;
    }
  }
  if (dst) {
    uint4* d0 = reinterpret_cast<uint4*>(dst + h * W);
    uint4* d1 = reinterpret_cast<uint4*>(dst + HD / 2 + h * W);
#pragma unroll
    for (int q = 0; q < W / 8; ++q) {
      d0[q] = make_uint4(pack2bf(a[q * 8], a[q * 8 + 1]), pack2bf(a[q * 8 + 2], a[q * 8 + 3]),
                         pack2bf(a[q * 8 + 4], a[q * 8 + 5]), pack2bf(a[q * 8 + 6], a[q * 8 + 7]));
      d1[q] = make_uint4(pack2bf(c2[q * 8], c2[q * 8 + 1]), pack2bf(c2[q * 8 + 2], c2[q * 8 + 3]),
                         pack2bf(c2[q * 8 + 4], c2[q * 8 + 5]), pack2bf(c2[q * 8 + 6], c2[q * 8 + 7]));
    }
  }
}

// Probabilities / score gradients of one half row (64 columns), packed BF16
// pairs (even column in the low half), into TMEM columns [col, col + 32).
__device__ __forceinline__ void tmem_st_packed32(uint32_t taddr, const uint32_t (&v)[32]) {
  tmem_st_32x32b_x32(taddr, v);
}

template <int HD>
struct TkvCfg {
  static constexpr int BOX = 128 * 128;      // one 64-column box of 128 rows, bytes
  static constexpr int TILE = 128 * HD * 2;  // 128 rows x HD columns (HD / 64 boxes)
  static constexpr int QSTAGES = 2;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE;
  static constexpr int OFF_Q = OFF_V + TILE;                 // QSTAGES tiles
  static constexpr int OFF_DO = OFF_Q + QSTAGES * TILE;      // QSTAGES tiles
  static constexpr int OFF_LD = OFF_DO + QSTAGES * TILE;     // [QSTAGES][lse 128 | delta 128]
  static constexpr int OFF_BAR = OFF_LD + QSTAGES * 256 * 4;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
};

template <int HD>
__global__ void __launch_bounds__(TB_THREADS, 1)
    attn_bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_do,
                            TbParams p) {
  using C = TkvCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sdO = smem + C::OFF_DO;
  float* sLD = reinterpret_cast<float*>(smem + C::OFF_LD);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bar + 0;
  uint64_t* qd_full = bar + 1;    // [2]
  uint64_t* qd_empty = bar + 3;   // [2]
  uint64_t* st_full = bar + 5;    // S^T of the current block computed
  uint64_t* dpt_full = bar + 6;   // dP^T of the current block computed
  uint64_t* p_ready = bar + 7;    // P^T stored (256 softmax threads)
  uint64_t* ds_ready = bar + 8;   // dS^T stored (256)
  uint64_t* ld_ready = bar + 9;   // lse/delta of a ragged block staged by the softmax threads (256)
  uint64_t* acc_full = bar + 13;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bar + 14);
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  int kb, gy;  // key block (0 = the most query blocks) and (batch, kv head) row
  causal_cta_order(p.chunk_kv, kb, gy);
  const int b = gy / p.Hkv, kvh = gy % p.Hkv;
  const int S = p.S;
  const int k0 = kb * 128;
  const int row0 = b * S;
  const int G = p.Hq / p.Hkv;
  const int qb_first = kb;
  const int n_qb = (S + 127) / 128;
  const int per_head = n_qb - qb_first;
  const int total = per_head * G;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&qd_full[i], 1);
      mbar_init(&qd_empty[i], 1);
    }
    mbar_init(ld_ready, kSoftmaxWarps);
    mbar_init(st_full, 1);
    mbar_init(dpt_full, 1);
    mbar_init(p_ready, kSoftmaxWarps);
    mbar_init(ds_ready, kSoftmaxWarps);
    mbar_init(acc_full, 1);
    fence_barrier_init();
    tma_prefetch_desc(&tm_qkv);
    tma_prefetch_desc(&tm_do);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t tST = tmem, tDPT = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + HD;

  auto head_of = [&](int it) { return kvh * G + it / per_head; };
  auto q0_of = [&](int it) { return (qb_first + it % per_head) * 128; };
  // lse and delta of a whole query block come with its Q and dO tiles (bulk
  // copies); a ragged last block is staged by the softmax threads
  auto bulk_ld = [&](int q0) { return p.ld_bulk && q0 + 128 <= S; };

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(kv_full, 2 * C::TILE);
#pragma unroll
      for (int i = 0; i < HD / 64; ++i) {
        tma_load_2d(sK + i * C::BOX, &tm_qkv, (p.Hq + kvh) * HD + 64 * i, row0 + k0, kv_full);
        tma_load_2d(sV + i * C::BOX, &tm_qkv, (p.Hq + p.Hkv + kvh) * HD + 64 * i, row0 + k0, kv_full);
      }
      int pend[2] = {-1, -1};
      for (int it = 0; it < total && !abort_flag; ++it) {
        const int st = it & 1;
        if (it >= 2 && !mbar_wait(&qd_empty[st], ((it >> 1) - 1) & 1)) {
          set_status(p.status, kStatusAttnBwdTimeout);
          abort_flag = 1;
          break;
        }
        const int h = head_of(it), q0 = q0_of(it);
        const bool bulk = bulk_ld(q0);
        mbar_arrive_expect_tx(&qd_full[st], 2 * C::TILE + (bulk ? 1024 : 0));
#pragma unroll
        for (int i = 0; i < HD / 64; ++i) {
          tma_load_2d(sQ + st * C::TILE + i * C::BOX, &tm_qkv, h * HD + 64 * i, row0 + q0, &qd_full[st]);
          tma_load_2d(sdO + st * C::TILE + i * C::BOX, &tm_do, h * HD + 64 * i, row0 + q0, &qd_full[st]);
        }
        if (bulk) {
          const long idx = ((long)b * p.Hq + h) * S + q0;
          bulk_load_1d(sLD + st * 256, p.lse + idx, 512, &qd_full[st]);
          bulk_load_1d(sLD + st * 256 + 128, p.delta + idx, 512, &qd_full[st]);
        }
        pend[st] = (it >> 1) & 1;
      }
      if (!mbar_wait(kv_full, 0)) set_status(p.status, kStatusAttnBwdTimeout);
      for (int s = 0; s < 2; ++s)
        if (pend[s] >= 0 && !mbar_wait(&qd_full[s], (uint32_t)pend[s])) set_status(p.status, kStatusAttnBwdTimeout);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(128, 128);                // K/V [keys][hd] x Q/dO [q][hd]^T
      const uint32_t id_acc = idesc_bf16_f32(128, HD) | (1u << 16);  // P^T/dS^T (TMEM) x dO/Q (MN-major)
      bool ok = mbar_wait(kv_full, 0);
      // S^T (or dP^T with V, dO) of block it into TMEM columns dst
      auto issue_scores = [&](int it, const uint8_t* sA, const uint8_t* sB, uint32_t dst) {
        const int qs = it & 1;
        const uint64_t da = smem_desc_kmajor_sw128(sA), db = smem_desc_kmajor_sw128(sB + qs * C::TILE);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          tc_mma_bf16(dst, da + desc_step(kk, C::BOX), db + desc_step(kk, C::BOX), id_s, kk > 0 ? 1u : 0u);
      };
      // acc += (TMEM operand at src) x (tile of block it, MN-major)
      auto issue_acc = [&](int it, uint32_t src, const uint8_t* sB, uint32_t acc) {
        const int qs = it & 1;
        const uint64_t bd = smem_desc_mnmajor_sw128(sB + qs * C::TILE, C::BOX);
#pragma unroll
        for (int kk = 0; kk < 128 / 16; ++kk)  // queries 64.. sit at columns 96..127
          tc_mma_bf16_ts(acc, src + kk * 8 + (kk >= 4 ? 64 : 0), bd + (uint64_t)(kk * (2048 >> 4)), id_acc,
                         (it > 0 || kk > 0) ? 1u : 0u);
      };
      if (ok && total > 0) {
        ok = mbar_wait(&qd_full[0], 0);
        if (ok) {
          tc_fence_after();
          issue_scores(0, sK, sQ, tST);
          tc_commit(st_full);
          issue_scores(0, sV, sdO, tDPT);
          tc_commit(dpt_full);
        }
      }
      for (int it = 0; ok && it < total; ++it) {
        const uint32_t ph = it & 1;
        if (!mbar_wait(p_ready, ph)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_acc(it, tST, sdO, tdV);  // dV += P^T dO
        const bool more = it + 1 < total;
        if (more) {
          if (!mbar_wait(&qd_full[(it + 1) & 1], ((it + 1) >> 1) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_scores(it + 1, sK, sQ, tST);  // runs after dV_it has read P^T
          tc_commit(st_full);
        }
        if (!mbar_wait(ds_ready, ph)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_acc(it, tDPT, sQ, tdK);  // dK += dS^T Q
        tc_commit(&qd_empty[it & 1]);
        if (more) {
          issue_scores(it + 1, sV, sdO, tDPT);  // runs after dK_it has read dS^T
          tc_commit(dpt_full);
        }
      }
      if (ok) {
        tc_commit(acc_full);
      } else {
        set_status(p.status, kStatusAttnBwdTimeout);
        abort_flag = 1;
      }
    }
  } else {
    // softmax warps 2..9: thread <-> key row r, half hf of the 128 query columns
    const int quarter = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const int tid = (warp - 2) * 32 + lane;  // 0..255
    const int key = k0 + r;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    bool ok = true;
    int staged = 0;  // ragged blocks staged so far (ld_ready's phase)
    for (int it = 0; it < total; ++it) {
      const int st = it & 1;
      const uint32_t ph = it & 1;
      const int h = head_of(it), q0 = q0_of(it);
      float* ld = sLD + st * 256;
      if (bulk_ld(q0)) {
        // the block's Q/dO barrier also covers its lse/delta copies
        if (!mbar_wait_warp(&qd_full[st], (it >> 1) & 1)) {
          ok = false;
          break;
        }
      } else {
        // stage lse and delta of the 128 queries once for all rows; queries
        // past the end get lse = +inf (P = 0) and delta = 0.  The slot's
        // previous block (it - 2) has been read by every softmax thread: this
        // thread has seen dP^T of block it - 1, which the MMA warp issues only
        // after all dS^T of block it - 2 are stored.  No copy targets it: the
        // TMA fills a slot only for whole blocks.
        const int t = tid & 127, q = q0 + t;
        const long idx = ((long)b * p.Hq + h) * S + q;
        if (tid < 128)
          ld[t] = q < S ? p.lse[idx] : INFINITY;
        else
          ld[128 + t] = q < S ? p.delta[idx] : 0.f;
        mbar_arrive_warp(ld_ready);
        if (!mbar_wait_warp(ld_ready, staged & 1)) {
          ok = false;
          break;
        }
        ++staged;
      }
      if (!mbar_wait_warp(st_full, ph)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[64];
      tmem_ld_32x32b_x64(tST + lane_off + hf * 64, sv);  // one wide load: less TMEM traffic contention
      tmem_wait_ld_regs(sv);
      // Queries past the sequence end have lse = +inf (P = 0) and delta = 0;
      // only the diagonal block (q0 == k0) needs the key > query mask.
      const bool diag = q0 == k0;
      const float4* lse4 = reinterpret_cast<const float4*>(ld + hf * 64);
      float pf[64];
      uint32_t pk[32];
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const float4 l4 = lse4[c4];
        const float lv[4] = {l4.x * kLog2eF, l4.y * kLog2eF, l4.z * kLog2eF, l4.w * kLog2eF};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = c4 * 4 + e;
          float pr = ex2_approx(fmaf(__uint_as_float(sv[c]), p.sl2, -lv[e]));
          if (diag && key > q0 + hf * 64 + c) pr = 0.f;
          pf[c] = pr;
        }
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) pk[j] = pack2bf(pf[2 * j], pf[2 * j + 1]);
      // P^T over the first 32 of this half's own 64 S^T columns (half 0:
      // 0..31, half 1: 96..127): no other thread reads them, so no barrier
      tmem_st_packed32(tST + lane_off + hf * 96, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(p_ready);
      // dS^T = P^T * (dP^T - delta)
      if (!mbar_wait_warp(dpt_full, ph)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float4* del4 = reinterpret_cast<const float4*>(ld + 128 + hf * 64);
      {
        uint32_t dp[64];
        tmem_ld_32x32b_x64(tDPT + lane_off + hf * 64, dp);
        tmem_wait_ld_regs(dp);
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 d4 = del4[c4];
          const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
          const int c = c4 * 4;
          pk[c / 2] = pack2bf(pf[c] * (__uint_as_float(dp[c]) - dv[0]), pf[c + 1] * (__uint_as_float(dp[c + 1]) - dv[1]));
          pk[c / 2 + 1] =
              pack2bf(pf[c + 2] * (__uint_as_float(dp[c + 2]) - dv[2]), pf[c + 3] * (__uint_as_float(dp[c + 3]) - dv[3]));
        }
      }
      tmem_st_packed32(tDPT + lane_off + hf * 96, pk);  // dS^T likewise over this half's dP^T columns
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(ds_ready);
    }
    ok = __all_sync(0xffffffffu, ok);
    if (ok && mbar_wait_warp(acc_full, 0)) {
      tc_fence_after();
      const bool valid = key < S;
      const bool rope = p.cos_t != nullptr;
      const int pos = valid ? key : 0;
      const float* cs = rope ? p.cos_t + (long)pos * (HD / 2) : nullptr;
      const float* sn = rope ? p.sin_t + (long)pos * (HD / 2) : nullptr;
      bf16* dk = valid ? p.dqkv + (long)(row0 + key) * p.ld + (long)(p.Hq + kvh) * HD : nullptr;
      bf16* dv = valid ? p.dqkv + (long)(row0 + key) * p.ld + (long)(p.Hq + p.Hkv + kvh) * HD : nullptr;
      store_half_row<HD>(tdK + lane_off, hf, p.scale, rope, cs, sn, dk);
      store_half_row<HD>(tdV + lane_off, hf, 1.0f, false, nullptr, nullptr, dv);
    } else {
      set_status(p.status, kStatusAttnBwdTimeout);
      abort_flag = 1;
    }
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int HD>
struct TdqCfg {
  static constexpr int BOX = 128 * 128;      // one 64-column box of 128 rows, bytes
  static constexpr int TILE = 128 * HD * 2;  // 128 rows x HD columns
  // K is read by S_j and, last, by dQ_j; V only by dP_j, which runs a whole
  // score block earlier.  Separate rings let V_j be refilled as soon as dP_j
  // is done, and give K a third stage.
  static constexpr int KSTAGES = 3, VSTAGES = 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = OFF_Q + TILE;
  static constexpr int OFF_K = OFF_DO + TILE;             // KSTAGES tiles
  static constexpr int OFF_V = OFF_K + KSTAGES * TILE;    // VSTAGES tiles
  static constexpr int OFF_BAR = OFF_V + VSTAGES * TILE;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
};

template <int HD>
__global__ void __launch_bounds__(TB_THREADS, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_do,
                          TbParams p) {
  using C = TdqCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sdO = smem + C::OFF_DO;
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  constexpr int NK = C::KSTAGES, NV = C::VSTAGES;
  uint64_t* q_full = bar + 0;
  uint64_t* k_full = bar + 1;                 // [NK]
  uint64_t* k_empty = bar + 1 + NK;           // [NK]
  uint64_t* v_full = bar + 1 + 2 * NK;        // [NV]
  uint64_t* v_empty = bar + 1 + 2 * NK + NV;  // [NV]
  uint64_t* s_full = bar + 1 + 2 * NK + 2 * NV;   // S of the current block computed
  uint64_t* s_read = bar + 2 + 2 * NK + 2 * NV;   // every softmax warp holds its S row in registers
  uint64_t* dp_full = bar + 3 + 2 * NK + 2 * NV;  // [2] dP of block j in TMEM buffer j & 1
  // [2] dS_j stored (over dP buffer j & 1).  Two barriers: the softmax may
  // finish block j + 1 before the MMA thread starts waiting for block j.
  uint64_t* ds_ready = bar + 5 + 2 * NK + 2 * NV;
  uint64_t* acc_full = bar + 7 + 2 * NK + 2 * NV;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bar + 8 + 2 * NK + 2 * NV);
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  int bx, by;
  causal_cta_order(p.chunk_q, bx, by);
  const int qb = gridDim.x - 1 - bx;  // longest causal rows first
  const int b = by / p.Hq, h = by % p.Hq;
  const int kvh = h * p.Hkv / p.Hq;
  const int S = p.S;
  const int q0 = qb * 128;
  const int row0 = b * S;
  const int n_kb = qb + 1;  // key blocks 0..qb (128-aligned, same as the query blocks)

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(q_full, 1);
    for (int i = 0; i < NK; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_read, kSoftmaxWarps);
    for (int i = 0; i < 2; ++i) mbar_init(&dp_full[i], 1);
    mbar_init(&ds_ready[0], kSoftmaxWarps);
    mbar_init(&ds_ready[1], kSoftmaxWarps);
    mbar_init(acc_full, 1);
    fence_barrier_init();
    tma_prefetch_desc(&tm_qkv);
    tma_prefetch_desc(&tm_do);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // TMEM columns: S 0, dP[2] 128 / 256 (dS over them), dQ 384 (HD columns)
  const uint32_t tS = tmem, tdQ = tmem + 384;
  auto tDP = [&](int j) { return tmem + 128u + 128u * (uint32_t)(j & 1); };

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, 2 * C::TILE);
#pragma unroll
      for (int i = 0; i < HD / 64; ++i) {
        tma_load_2d(sQ + i * C::BOX, &tm_qkv, h * HD + 64 * i, row0 + q0, q_full);
        tma_load_2d(sdO + i * C::BOX, &tm_do, h * HD + 64 * i, row0 + q0, q_full);
      }
      int pk[NK], pv[NV];
      for (int s = 0; s < NK; ++s) pk[s] = -1;
      for (int s = 0; s < NV; ++s) pv[s] = -1;
      for (int j = 0; j < n_kb && !abort_flag; ++j) {
        const int sk = j % NK, sv = j % NV;
        if (j >= NK && !mbar_wait(&k_empty[sk], ((j / NK) - 1) & 1)) {
          set_status(p.status, kStatusAttnBwdTimeout);
          abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&k_full[sk], C::TILE);
#pragma unroll
        for (int i = 0; i < HD / 64; ++i)
          tma_load_2d(sK + sk * C::TILE + i * C::BOX, &tm_qkv, (p.Hq + kvh) * HD + 64 * i, row0 + j * 128,
                      &k_full[sk]);
        pk[sk] = (j / NK) & 1;
        if (j >= NV && !mbar_wait(&v_empty[sv], ((j / NV) - 1) & 1)) {
          set_status(p.status, kStatusAttnBwdTimeout);
          abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&v_full[sv], C::TILE);
#pragma unroll
        for (int i = 0; i < HD / 64; ++i)
          tma_load_2d(sV + sv * C::TILE + i * C::BOX, &tm_qkv, (p.Hq + p.Hkv + kvh) * HD + 64 * i, row0 + j * 128,
                      &v_full[sv]);
        pv[sv] = (j / NV) & 1;
      }
      if (!mbar_wait(q_full, 0)) set_status(p.status, kStatusAttnBwdTimeout);
      for (int s = 0; s < NK; ++s)
        if (pk[s] >= 0 && !mbar_wait(&k_full[s], (uint32_t)pk[s])) set_status(p.status, kStatusAttnBwdTimeout);
      for (int s = 0; s < NV; ++s)
        if (pv[s] >= 0 && !mbar_wait(&v_full[s], (uint32_t)pv[s])) set_status(p.status, kStatusAttnBwdTimeout);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(128, 128);
      const uint32_t id_dq = idesc_bf16_f32(128, HD) | (1u << 16);  // dS (TMEM) x K (MN-major)
      bool ok = mbar_wait(q_full, 0);
      // scores of block j: A (Q or dO) x B-tile^T into TMEM columns dst
      auto issue_scores = [&](const uint8_t* sA, const uint8_t* sBt, uint32_t dst) {
        const uint64_t da = smem_desc_kmajor_sw128(sA), db = smem_desc_kmajor_sw128(sBt);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          tc_mma_bf16(dst, da + desc_step(kk, C::BOX), db + desc_step(kk, C::BOX), id_s, kk > 0 ? 1u : 0u);
      };
      auto issue_s = [&](int j) {
        if (!mbar_wait(&k_full[j % NK], (j / NK) & 1)) return false;
        tc_fence_after();
        issue_scores(sQ, sK + (j % NK) * C::TILE, tS);
        tc_commit(s_full);
        return true;
      };
      // dP_j into buffer j & 1, whose dS_{j-2} the dQ MMAs issued before have read
      auto issue_dp = [&](int j) {
        if (!mbar_wait(&v_full[j % NV], (j / NV) & 1)) return false;
        tc_fence_after();
        issue_scores(sdO, sV + (j % NV) * C::TILE, tDP(j));
        tc_commit(&dp_full[j & 1]);
        tc_commit(&v_empty[j % NV]);
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok) ok = issue_dp(0);
      for (int j = 0; ok && j < n_kb; ++j) {
        // S_{j+1} once every softmax thread holds S_j in registers, dP_{j+1}
        // into the other buffer: both run while the softmax works on block j
        if (!mbar_wait(s_read, j & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (j + 1 < n_kb && (!issue_s(j + 1) || !issue_dp(j + 1))) {
          ok = false;
          break;
        }
        if (!mbar_wait(&ds_ready[j & 1], (j >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t src = tDP(j);
        const uint64_t kd = smem_desc_mnmajor_sw128(sK + (j % NK) * C::TILE, C::BOX);
#pragma unroll
        for (int kk = 0; kk < 128 / 16; ++kk)  // keys 64.. sit at columns 96..127
          tc_mma_bf16_ts(tdQ, src + kk * 8 + (kk >= 4 ? 64 : 0), kd + (uint64_t)(kk * (2048 >> 4)), id_dq,
                         (j > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&k_empty[j % NK]);
      }
      if (ok) {
        tc_commit(acc_full);
      } else {
        set_status(p.status, kStatusAttnBwdTimeout);
        abort_flag = 1;
      }
    }
  } else {
    // softmax warps 2..9: thread <-> query row r, half hf of the 128 key columns
    const int quarter = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const int qrow = q0 + r;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const bool valid = qrow < S;
    const long li = ((long)b * p.Hq + h) * S + (valid ? qrow : 0);
    const float L2 = valid ? p.lse[li] * kLog2eF : INFINITY;
    const float Dr = valid ? p.delta[li] : 0.f;
    bool ok = true;
    for (int j = 0; j < n_kb; ++j) {
      const uint32_t tD = tDP(j);
      if (!mbar_wait_warp(s_full, j & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[64];
      tmem_ld_32x32b_x64(tS + lane_off + hf * 64, sv);  // one wide load: less TMEM traffic contention
      tmem_wait_ld_regs(sv);
      tc_fence_before();
      mbar_arrive_warp(s_read);  // S_{j+1} may overwrite S_j
      // Rows past the sequence end have L2 = +inf (P = 0); only the diagonal
      // block (key block j == query block) needs the key > query mask.
      const int k0 = j * 128;
      const bool diag = j == qb;
      float pf[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        float pr = ex2_approx(fmaf(__uint_as_float(sv[c]), p.sl2, -L2));
        if (diag && k0 + hf * 64 + c > qrow) pr = 0.f;
        pf[c] = pr;
      }
      if (!mbar_wait_warp(&dp_full[j & 1], (j >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t pk[32];
      {
        uint32_t dp[64];
        tmem_ld_32x32b_x64(tD + lane_off + hf * 64, dp);
        tmem_wait_ld_regs(dp);
#pragma unroll
        for (int e = 0; e < 32; ++e)
          pk[e] = pack2bf(pf[2 * e] * (__uint_as_float(dp[2 * e]) - Dr), pf[2 * e + 1] * (__uint_as_float(dp[2 * e + 1]) - Dr));
      }
      // dS over the first 32 of this half's own 64 dP columns (half 0: 0..31,
      // half 1: 96..127), which this thread has read: no barrier
      tmem_st_packed32(tD + lane_off + hf * 96, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(&ds_ready[j & 1]);
    }
    ok = __all_sync(0xffffffffu, ok);
    if (ok && mbar_wait_warp(acc_full, 0)) {
      tc_fence_after();
      const bool rope = p.cos_t != nullptr;
      const int pos = valid ? qrow : 0;
      const float* cs = rope ? p.cos_t + (long)pos * (HD / 2) : nullptr;
      const float* sn = rope ? p.sin_t + (long)pos * (HD / 2) : nullptr;
      bf16* dq = valid ? p.dqkv + (long)(row0 + qrow) * p.ld + (long)h * HD : nullptr;
      store_half_row<HD>(tdQ + lane_off, hf, p.scale, rope, cs, sn, dq);
    } else {
      set_status(p.status, kStatusAttnBwdTimeout);
      abort_flag = 1;
    }
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int HD>
int launch_bwd_tc(const AttnArgs& x, cudaStream_t s) {
  using A = TkvCfg<HD>;
  using Bq = TdqCfg<HD>;
  static bool init = false;
  if (!init) {
    if (cudaFuncSetAttribute(attn_bwd_dkdv_tc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, A::SMEM) !=
            cudaSuccess ||
        cudaFuncSetAttribute(attn_bwd_dq_tc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, Bq::SMEM) !=
            cudaSuccess)
      return -2;
    init = true;
  }
  const long T = (long)x.batch * x.seq;
  const long cols = (long)(x.n_heads + 2 * x.n_kv_heads) * HD;
  CUtensorMap tm_qkv, tm_do;
  if (!make_tmap_bf16(&tm_qkv, x.qkv, T, cols, x.ldqkv, 128) ||
      !make_tmap_bf16(&tm_do, x.dout, T, (long)x.n_heads * HD, x.ldo, 128))
    return -3;
  TbParams p;
  p.B = x.batch;
  p.S = x.seq;
  p.Hq = x.n_heads;
  p.Hkv = x.n_kv_heads;
  p.lse = x.lse;
  p.delta = x.delta;
  p.dqkv = x.dqkv;
  p.ld = x.ldqkv;
  p.cos_t = x.rope_cos;
  p.sin_t = x.rope_sin;
  p.scale = 1.0f / sqrtf((float)HD);
  p.sl2 = p.scale * kLog2eF;
  p.ld_bulk = x.seq % 4 == 0 && (reinterpret_cast<uintptr_t>(x.lse) & 15) == 0 &&
              (reinterpret_cast<uintptr_t>(x.delta) & 15) == 0;
  p.status = x.status;
  dim3 g1((x.seq + 127) / 128, x.batch * x.n_kv_heads);
  dim3 g2((x.seq + 127) / 128, x.batch * x.n_heads);
  p.chunk_kv = causal_chunk_rows((int)g1.x, (int)g1.y, 256);
  p.chunk_q = causal_chunk_rows((int)g2.x, (int)g2.y, 256);
  attn_bwd_dkdv_tc_kernel<HD><<<g1, TB_THREADS, A::SMEM, s>>>(tm_qkv, tm_do, p);
  attn_bwd_dq_tc_kernel<HD><<<g2, TB_THREADS, Bq::SMEM, s>>>(tm_qkv, tm_do, p);
  return launch_result();
}

}  // namespace

int launch_attn_bwd_tc_main(const AttnArgs& x, cudaStream_t s) {
  return x.head_dim == 128 ? launch_bwd_tc<128>(x, s) : launch_bwd_tc<64>(x, s);
}

}  // namespace mt
