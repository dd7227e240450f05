// Causal grouped-query flash attention forward on the 5th-generation tensor
// cores: S = Q K^T and O += P V with tcgen05.mma, S and O accumulated in
// TMEM, Q/K/V tiles brought in by TMA.
//
// One CTA per (128 queries, query head, batch); 6 warps:
//   warp 0      TMA: Q once; K and V blocks of 128 keys into a 2-stage ring
//               (one tensor map over the packed q|k|v projection buffer).
//   warp 1      MMA (one thread): S_j = Q K_j^T into TMEM buffer j%2, then,
//               once the softmax has written P_j, O += P_j V_j (V read as an
//               MN-major operand straight from its [keys][head_dim] tile).
//   warps 2..5  softmax: each thread owns one query row (its TMEM lane), so
//               the row max and row sum need no shuffles.  P_j is written to
//               shared memory in the 128-byte-swizzled K-major layout the
//               tensor core reads as its A operand.  The running maximum is
//               only moved (and O rescaled in TMEM) when it grows by more than
//               a factor 2^8, so O is rarely touched; the final O / l and the
//               log-sum-exp use whichever maximum was kept.
// Every mbarrier wait is bounded; on expiry the kernel records
// kStatusGemmTimeout in the status word and unwinds.
//
// MegaTrain's templates hold "Attention and MLP kernels" (paperlayer.ai
// summary §A.4) without specifying them; this kernel is the library's own.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace mt {

// Defined in gemm.cu: 2-D BF16 tensor map with 64-column x box_rows boxes, 128-byte swizzle.
bool make_tmap_bf16(CUtensorMap* m, const void* base, long rows, long cols, long ld, int box_rows);

namespace {

constexpr int TA_BM = 128, TA_BN = 128, TA_THREADS = 192;
constexpr float kLog2eF = 1.4426950408889634f;
constexpr float kLn2F = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8

template <int HD>
struct TaCfg {
  static constexpr int BOX = 128 * 128;          // one 64-column box of 128 rows, bytes
  static constexpr int Q_BYTES = 128 * HD * 2;   // HD/64 boxes
  static constexpr int KV_BYTES = 128 * HD * 2;  // K or V block
  static constexpr int P_BYTES = 128 * 128 * 2;  // two 64-key boxes
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;            // 2 stages
  static constexpr int OFF_V = OFF_K + 2 * KV_BYTES;       // 2 stages
  static constexpr int OFF_P = OFF_V + 2 * KV_BYTES;       // 2 buffers
  static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;        // barriers + alignment slack
};

struct TaParams {
  int B, S, Hq, Hkv;
  bf16* o;
  long ldo;
  float* lse;
  float sl2;  // softmax scale * log2(e)
  int* status;
};

__device__ __forceinline__ uint32_t pack2bf(float a, float b) {
  __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&p);
}

template <int HD>
__global__ void __launch_bounds__(TA_THREADS, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, TaParams p) {
  using C = TaCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sP = smem + C::OFF_P;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bar + 0;
  uint64_t* kv_full = bar + 1;   // [2]
  uint64_t* kv_empty = bar + 3;  // [2]
  uint64_t* s_full = bar + 5;    // [2]
  uint64_t* p_full = bar + 7;    // [2]
  uint64_t* pv_done = bar + 9;   // [2]
  uint64_t* o_full = bar + 11;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bar + 12);
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int qb = gridDim.x - 1 - blockIdx.x;  // longest causal rows first
  const int b = blockIdx.y / p.Hq, h = blockIdx.y % p.Hq;
  const int kvh = h * p.Hkv / p.Hq;
  const int S = p.S;
  const int q0 = qb * TA_BM;
  const int n_kb = min((S + TA_BN - 1) / TA_BN, (q0 + TA_BM + TA_BN - 1) / TA_BN);
  const int row0 = b * S;  // token row of position 0 in the packed buffer
  const int colQ = h * HD, colK = (p.Hq + kvh) * HD, colV = (p.Hq + p.Hkv + kvh) * HD;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(o_full, 1);
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
  const uint32_t tO = tmem + 256;

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, C::Q_BYTES);
#pragma unroll
      for (int i = 0; i < HD / 64; ++i) tma_load_2d(sQ + i * C::BOX, &tm_qkv, colQ + 64 * i, row0 + q0, q_full);
      int pend[2] = {-1, -1};
      for (int j = 0; j < n_kb && !abort_flag; ++j) {
        const int s = j & 1;
        if (j >= 2 && !mbar_wait(&kv_empty[s], ((j >> 1) - 1) & 1)) {
          set_status(p.status, kStatusGemmTimeout);
          abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&kv_full[s], 2 * C::KV_BYTES);
#pragma unroll
        for (int i = 0; i < HD / 64; ++i) {
          tma_load_2d(sK + s * C::KV_BYTES + i * C::BOX, &tm_qkv, colK + 64 * i, row0 + j * TA_BN, &kv_full[s]);
          tma_load_2d(sV + s * C::KV_BYTES + i * C::BOX, &tm_qkv, colV + 64 * i, row0 + j * TA_BN, &kv_full[s]);
        }
        pend[s] = (j >> 1) & 1;
      }
      // every issued load must land before exit
      if (!mbar_wait(q_full, 0)) set_status(p.status, kStatusGemmTimeout);
      for (int s = 0; s < 2; ++s)
        if (pend[s] >= 0 && !mbar_wait(&kv_full[s], (uint32_t)pend[s])) set_status(p.status, kStatusGemmTimeout);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_qk = idesc_bf16_f32(128, 128);
      const uint32_t id_pv = idesc_bf16_f32(128, HD) | (1u << 16);  // B (V) MN-major
      bool ok = mbar_wait(q_full, 0);
      auto issue_qk = [&](int j) {
        const int s = j & 1;
        if (!mbar_wait(&kv_full[s], (j >> 1) & 1)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const int box = kk >> 2, off = (kk & 3) * 32;
          const uint64_t a = smem_desc_kmajor_sw128(sQ + box * C::BOX + off);
          const uint64_t bb = smem_desc_kmajor_sw128(sK + s * C::KV_BYTES + box * C::BOX + off);
          tc_mma_bf16((tmem + 128u * (uint32_t)s), a, bb, id_qk, kk > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[s]);
        return true;
      };
      if (ok) ok = issue_qk(0);
      for (int j = 0; ok && j < n_kb; ++j) {
        const int s = j & 1;
        if (j + 1 < n_kb && !issue_qk(j + 1)) {
          ok = false;
          break;
        }
        if (!mbar_wait(&p_full[s], (j >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t vdesc = smem_desc_mnmajor_sw128(sV + s * C::KV_BYTES, C::BOX);
#pragma unroll
        for (int kk = 0; kk < TA_BN / 16; ++kk) {
          const int box = kk >> 2, off = (kk & 3) * 32;
          const uint64_t a = smem_desc_kmajor_sw128(sP + s * C::P_BYTES + box * C::BOX + off);
          tc_mma_bf16(tO, a, vdesc + (uint64_t)(kk * (2048 >> 4)), id_pv, (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&kv_empty[s]);
        tc_commit(&pv_done[s]);
      }
      if (ok) {
        tc_commit(o_full);
      } else {
        set_status(p.status, kStatusGemmTimeout);
        abort_flag = 1;
      }
    }
  } else {
    // softmax warps: thread <-> query row r (TMEM lane r)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int qrow = q0 + r;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kb; ++j) {
      const int s = j & 1;
      if (!mbar_wait(&s_full[s], (j >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[TA_BN];
#pragma unroll
      for (int c = 0; c < TA_BN / 32; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32((tmem + 128u * (uint32_t)s) + lane_off + c * 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) x[c * 32 + e] = __uint_as_float(v[e]) * p.sl2;
      }
      const int k0 = j * TA_BN;
      float mx = -INFINITY;
      if (k0 + TA_BN - 1 > q0) {  // block touches the diagonal
#pragma unroll
        for (int c = 0; c < TA_BN; ++c)
          if (k0 + c > qrow) x[c] = -INFINITY;
      }
#pragma unroll
      for (int c = 0; c < TA_BN; ++c) mx = fmaxf(mx, x[c]);
      const float m_new = fmaxf(m, mx);
      const bool rescale = (m == -INFINITY) || (m_new > m + kRescaleThreshold);
      float alpha = 1.f;
      if (rescale) {
        alpha = (m == -INFINITY) ? 0.f : exp2f(m - m_new);
        m = m_new;
      }
      const float base = (m == -INFINITY) ? 0.f : m;
      // the P buffer is free once PV_{j-2} completed
      if (j >= 2 && !mbar_wait(&pv_done[s], ((j >> 1) - 1) & 1)) {
        ok = false;
        break;
      }
      float rs = 0.f;
      uint8_t* prow = sP + s * C::P_BYTES + r * 128;
#pragma unroll
      for (int c16 = 0; c16 < TA_BN / 8; ++c16) {  // 16-byte chunks of 8 keys
        float e8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          e8[e] = exp2f(x[c16 * 8 + e] - base);
          rs += e8[e];
        }
        const int box = c16 >> 3, cc = c16 & 7;
        uint4 w = make_uint4(pack2bf(e8[0], e8[1]), pack2bf(e8[2], e8[3]), pack2bf(e8[4], e8[5]),
                             pack2bf(e8[6], e8[7]));
        *reinterpret_cast<uint4*>(prow + box * C::BOX + ((cc ^ (r & 7)) << 4)) = w;
      }
      l = l * alpha + rs;
      if (rescale && j > 0) {
        // O holds sum_{i<j} P_i V_i: wait for PV_{j-1}, then scale this row in TMEM
        if (!mbar_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tO + lane_off + c * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
          tmem_st_32x32b_x32(tO + lane_off + c * 32, v);
        }
        tmem_wait_st();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[s]);
    }
    if (ok && mbar_wait(o_full, 0)) {
      tc_fence_after();
      const float inv = 1.f / l;
      const bool valid = qrow < S;
      bf16* dst = p.o + (long)(row0 + qrow) * p.ldo + (long)h * HD;
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tO + lane_off + c * 32, v);
        tmem_wait_ld();
        if (valid) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float* f = reinterpret_cast<const float*>(v + q * 8);
            d4[q] = make_uint4(pack2bf(f[0] * inv, f[1] * inv), pack2bf(f[2] * inv, f[3] * inv),
                               pack2bf(f[4] * inv, f[5] * inv), pack2bf(f[6] * inv, f[7] * inv));
          }
        }
      }
      if (valid) p.lse[((long)b * p.Hq + h) * S + qrow] = (m + log2f(l)) * kLn2F;
    } else {
      set_status(p.status, kStatusGemmTimeout);
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
  attn_fwd_tc_kernel<HD><<<grid, TA_THREADS, C::SMEM, s>>>(tm, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace

int launch_attn_fwd_tc(const AttnArgs& x, cudaStream_t s) {
  if (attn_check(x)) return -1;
  return x.head_dim == 128 ? launch_tc<128>(x, s) : launch_tc<64>(x, s);
}

}  // namespace mt
