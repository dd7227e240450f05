// BF16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM), fed by TMA.
//
//   C[M, N] = epilogue( A[M, K] * B[N, K]^T )      (both operands K-major)
//
// This is the one dense contraction of the decoder step: the QKV, O, gate-up
// and down projections in forward, their data and weight gradients in
// backward, and the LM head (MegaTrain paper summary (paperlayer.ai), §A.4
// "GPU Compute Dispatch": the layer templates hold the attention and MLP
// kernels; the kernels themselves are this library's own design).
//
// Two kernels with the same warp roles, persistent over output tiles:
//   gemm_bf16_tcgen05_pair_kernel (every GEMM with M > 128): clusters of two
//     CTAs on two SMs share one 256 x 256 tile; each CTA stages its 128 rows
//     of A and its half of B (6-stage ring), the even CTA issues
//     tcgen05.mma.cta_group::2 (M=256, N=256, K=16) and its commits arrive on
//     both CTAs' barriers.  Per SM 32 KB of operands per 64-wide K block.
//   gemm_bf16_tcgen05_kernel (M <= 128, or no pair placeable): one CTA per SM,
//     128 x 256 tiles, tcgen05.mma M=128, N=256, K=16, 4-stage ring.
// Warp roles (both):
//   warp 0      TMA producer: 128-byte-swizzled boxes into the stage ring.
//   warp 1      MMA issuer: one elected thread issues the MMAs into one of two
//               TMEM accumulators (2 x 256 FP32 columns), commits stage
//               release and accumulator-ready.
//   warps 2..5  epilogue: tcgen05.ld of one accumulator row per thread, fused
//               epilogue (bf16 / fp32 store, residual add, SwiGLU on
//               interleaved gate/up columns, the SwiGLU backward through a
//               per-warp shared-memory transpose, rotate-half RoPE, fp32 +=),
//               16-byte stores.  The second accumulator lets the epilogue of
//               tile i overlap the main loop of tile i+1.
// Every mbarrier wait is bounded (2 s); on expiry the kernel records
// kStatusGemmTimeout in the status word and unwinds.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace mt {

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int A_STAGE = BM * BK * 2;  // 16 KB
constexpr int B_STAGE = BN * BK * 2;  // 32 KB
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 2 * BN;  // two FP32 accumulators
constexpr int GROUP_M = 16;        // tile raster: 16 M-tiles share each B panel
// Per epilogue warp a 32 x 33 float block for transposing an accumulator chunk.
constexpr int XPOSE_BYTES = 4 * 32 * 33 * 4;
constexpr int SMEM_USED = STAGES * (A_STAGE + B_STAGE) + 1024 /*align*/ + 256 /*barriers*/ + XPOSE_BYTES;
// Launch with the whole 227 KB (one CTA per SM either way); the unused tail
// keeps every tensor-core read of the last stage inside the allocation.
constexpr int SMEM_BYTES = 232448 - 256;  // 227 KB less room for the static shared variables
static_assert(SMEM_USED <= SMEM_BYTES, "shared memory plan exceeds 227 KB");

// CTA-pair variant (cta_group::2): a cluster of two CTAs on two SMs computes
// one 256 x 256 output tile.  Each CTA stages its 128 rows of A and its 128
// rows (half) of B per K block; the leading CTA's single MMA thread issues
// M = 256, N = 256 MMAs that read both CTAs' stages, and each CTA's TMEM
// receives its 128 rows of the tile.  Per SM this moves 32 KB of operands per
// K block instead of 48 KB for the same 128 x 256 x 64 of work.
constexpr int PM = 256;                // pair tile rows (128 per CTA)
constexpr int PHALF = 128;             // rows of A and of B staged per CTA
constexpr int P_STAGES = 6;
constexpr int P_A_STAGE = PHALF * BK * 2;  // 16 KB
constexpr int P_B_STAGE = PHALF * BK * 2;  // 16 KB
constexpr int P_GROUP_M = 8;           // pair-tile raster: 8 M-tiles share each B panel
// Grouped launches (one GEMM per expert of a mixture-of-experts layer in one
// launch) keep the group's row offsets and tile prefix in shared memory.
constexpr int kMaxGroups = 256;
constexpr int P_GROUP_TABLE = 2 * (kMaxGroups + 4) * 4;
constexpr int P_SMEM_USED = P_STAGES * (P_A_STAGE + P_B_STAGE) + 1024 + 256 + XPOSE_BYTES + P_GROUP_TABLE;
static_assert(P_SMEM_USED <= SMEM_BYTES, "pair shared memory plan exceeds 227 KB");

// Grouping of a pair launch (a compile-time kernel parameter):
//   kGroupNone  one GEMM.
//   kGroupM     per group g the rows offsets[g] .. offsets[g+1] of A (K-major,
//               one buffer for all groups) times group g's B (stacked: rows
//               g*N .. of a K-major B, K rows g*K .. of an MN-major B); C rows
//               are A's rows.  Tiles past a group's last row are computed and
//               not stored.
//   kGroupK     per group g, C[g*M .. g*M + M) = A_g^T B_g where A_g, B_g are
//               the rows offsets[g] .. offsets[g+1] of two MN-major operands
//               (the K range of group g).  A group with no rows stores zeros.
//               Every group's row count must be a multiple of 64 (one K block)
//               or its last block reads the next group's rows.
enum : int { kGroupNone = 0, kGroupM = 1, kGroupK = 2 };
static_assert((int)kGroupM == (int)kGemmGroupRows && (int)kGroupK == (int)kGemmGroupK, "grouping codes");

struct EpiParams {
  int M, N, K;
  int mode;
  void* C;
  long ldc;
  const __nv_bfloat16* R;
  long ldr;
  __nv_bfloat16* C2;
  long ldc2;
  const float* rope_cos;
  const float* rope_sin;
  int rope_cols;
  int head_dim;
  int seq;
  int* status;
  const int32_t* group_off;  // grouped launches: [groups + 1] row offsets on the device
  int groups;
};

__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int& tm, int& tn, int group_m = GROUP_M) {
  const int per_group = group_m * num_n;
  const int group = tile / per_group;
  const int first_m = group * group_m;
  const int gsize = min(num_m - first_m, group_m);
  const int r = tile - group * per_group;
  tm = first_m + r % gsize;
  tn = r / gsize;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

// Store 32 FP32 values as BF16 at dst[0..31] (dst 16-byte aligned) for the
// columns that are < ncols_valid.
__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float* v, int ncols_valid) {
  if (ncols_valid >= 32) {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 w;
      w.x = pack_bf16(v[q * 8 + 0], v[q * 8 + 1]);
      w.y = pack_bf16(v[q * 8 + 2], v[q * 8 + 3]);
      w.z = pack_bf16(v[q * 8 + 4], v[q * 8 + 5]);
      w.w = pack_bf16(v[q * 8 + 6], v[q * 8 + 7]);
      d[q] = w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)  // constant indices keep v in registers
      if (j < ncols_valid) dst[j] = __float2bfloat16_rn(v[j]);
  }
}

__device__ __forceinline__ void epilogue_chunk(const EpiParams& p, int row, int col0, float* v) {
  // `v` holds accumulator columns col0 .. col0+31 of output row `row`.
  const int nvalid = min(32, p.N - col0);
  if (row >= p.M || nvalid <= 0) return;
  switch (p.mode) {
    case kEpiStoreBf16: {
      store_bf16x32(reinterpret_cast<__nv_bfloat16*>(p.C) + (long)row * p.ldc + col0, v, nvalid);
      break;
    }
    case kEpiResidualBf16: {
      const __nv_bfloat16* r = p.R + (long)row * p.ldr + col0;
      if (nvalid >= 32) {
        const uint4* r4 = reinterpret_cast<const uint4*>(r);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 w = r4[q];
          v[q * 8 + 0] += bf16_lo(w.x); v[q * 8 + 1] += bf16_hi(w.x);
          v[q * 8 + 2] += bf16_lo(w.y); v[q * 8 + 3] += bf16_hi(w.y);
          v[q * 8 + 4] += bf16_lo(w.z); v[q * 8 + 5] += bf16_hi(w.z);
          v[q * 8 + 6] += bf16_lo(w.w); v[q * 8 + 7] += bf16_hi(w.w);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < nvalid) v[j] += __bfloat162float(r[j]);
      }
      store_bf16x32(reinterpret_cast<__nv_bfloat16*>(p.C) + (long)row * p.ldc + col0, v, nvalid);
      break;
    }
    case kEpiF32: {
      float* c = reinterpret_cast<float*>(p.C) + (long)row * p.ldc + col0;
      if (nvalid >= 32) {
        float4* c4 = reinterpret_cast<float4*>(c);
#pragma unroll
        for (int q = 0; q < 8; ++q) c4[q] = make_float4(v[q * 4], v[q * 4 + 1], v[q * 4 + 2], v[q * 4 + 3]);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < nvalid) c[j] = v[j];
      }
      break;
    }
    case kEpiF32Accumulate: {
      float* c = reinterpret_cast<float*>(p.C) + (long)row * p.ldc + col0;
      if (nvalid >= 32) {
        float4* c4 = reinterpret_cast<float4*>(c);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float4 o = c4[q];
          c4[q] = make_float4(o.x + v[q * 4], o.y + v[q * 4 + 1], o.z + v[q * 4 + 2], o.w + v[q * 4 + 3]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < nvalid) c[j] += v[j];
      }
      break;
    }
    case kEpiSwiGLU: {
      // Columns alternate gate, up: output a[row, col/2] = silu(gate) * up.
      if (p.C2) store_bf16x32(p.C2 + (long)row * p.ldc2 + col0, v, nvalid);
      float a[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float g = v[2 * j], u = v[2 * j + 1];
        a[j] = g / (1.0f + __expf(-g)) * u;
      }
      __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.C) + (long)row * p.ldc + col0 / 2;
      const int na = nvalid / 2;
      if (na >= 16) {
        uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint4 w;
          w.x = pack_bf16(a[q * 8 + 0], a[q * 8 + 1]);
          w.y = pack_bf16(a[q * 8 + 2], a[q * 8 + 3]);
          w.z = pack_bf16(a[q * 8 + 4], a[q * 8 + 5]);
          w.w = pack_bf16(a[q * 8 + 6], a[q * 8 + 7]);
          d[q] = w;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (j < na) dst[j] = __float2bfloat16_rn(a[j]);
      }
      break;
    }
    default:
      break;
  }
}

// Epilogue of one output tile: thread `row` of the tile reads its TMEM lane
// (tbase already points at lane quarter*32, accumulator column 0), applies the
// epilogue mode and stores columns tn*BN .. tn*BN + BN - 1.
__device__ __forceinline__ void store_tile(const EpiParams& p, uint32_t tbase, int row, int tn, float* xpose) {
  if (p.mode == kEpiSwiGLUBwd) {
    // One row per thread does not coalesce: each lane would read its row's
    // gate/up pairs and write dgate/dup 64 KB away from its neighbours'.  The
    // warp's 32 x 32 block of da goes through shared memory (row stride 33
    // floats: conflict-free both ways) and comes back as 4 consecutive
    // columns of one row per lane, so 8 lanes cover 128 contiguous bytes of
    // R and of C.  All eight loads of a chunk are issued before any use.
    const int lane = threadIdx.x & 31;
    const int row0 = row - lane;
    const int sub = lane & 7;
    auto grad = [](float da, float gt, float up, float& dg, float& du) {
      const float sg = 1.0f / (1.0f + __expf(-gt));
      dg = da * up * sg * (1.0f + gt * (1.0f - sg));
      du = da * gt * sg;
    };
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(tbase + c * 32, r);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) xpose[lane * 33 + e] = __uint_as_float(r[e]);
      __syncwarp();
      const int col = tn * BN + c * 32 + 4 * sub;  // this lane's first da column
      const int nv = min(4, p.N - col);
      uint4 g[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int grow = row0 + 4 * i + (lane >> 3);
        g[i] = make_uint4(0u, 0u, 0u, 0u);
        if (grow < p.M && nv == 4) g[i] = *reinterpret_cast<const uint4*>(p.R + (long)grow * p.ldr + 2 * col);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int rr = 4 * i + (lane >> 3);
        const int grow = row0 + rr;
        if (grow >= p.M || nv <= 0) continue;
        const float* dav = xpose + rr * 33 + 4 * sub;
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.C) + (long)grow * p.ldc + 2 * col;
        if (nv == 4) {
          const uint32_t ws[4] = {g[i].x, g[i].y, g[i].z, g[i].w};
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float dg, du;
            grad(dav[e], bf16_lo(ws[e]), bf16_hi(ws[e]), dg, du);
            o[e] = pack_bf16(dg, du);
          }
          *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
        } else {
          const __nv_bfloat16* gp = p.R + (long)grow * p.ldr + 2 * col;
          for (int e = 0; e < nv; ++e) {
            float dg, du;
            grad(dav[e], __bfloat162float(gp[2 * e]), __bfloat162float(gp[2 * e + 1]), dg, du);
            dst[2 * e] = __float2bfloat16_rn(dg);
            dst[2 * e + 1] = __float2bfloat16_rn(du);
          }
        }
      }
      __syncwarp();  // the next chunk overwrites this warp's block
    }
  } else if (p.mode == kEpiRope && tn * BN < p.rope_cols) {
    // rotate-half RoPE: columns j and j + hd/2 of each head form a pair.
    // The row's cos/sin for frequencies j .. j+31 are loaded once (16-byte
    // loads) and serve every head of the tile.
    const int hd = p.head_dim;
    const int s = row % p.seq;
    for (int j = 0; j < hd / 2; j += 32) {
      float cs[32], sn[32];
      if (row < p.M) {
        const float4* c4 = reinterpret_cast<const float4*>(p.rope_cos + (long)s * (hd / 2) + j);
        const float4* s4 = reinterpret_cast<const float4*>(p.rope_sin + (long)s * (hd / 2) + j);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 a = c4[q], b = s4[q];
          cs[4 * q] = a.x, cs[4 * q + 1] = a.y, cs[4 * q + 2] = a.z, cs[4 * q + 3] = a.w;
          sn[4 * q] = b.x, sn[4 * q + 1] = b.y, sn[4 * q + 2] = b.z, sn[4 * q + 3] = b.w;
        }
      }
      for (int h0 = 0; h0 < BN; h0 += hd) {
        uint32_t lo_r[32], hi_r[32];
        tmem_ld_32x32b_x32(tbase + h0 + j, lo_r);
        tmem_ld_32x32b_x32(tbase + h0 + hd / 2 + j, hi_r);
        tmem_wait_ld();
        float lo[32], hi[32];
        const int gcol = tn * BN + h0 + j;
        if (row < p.M && gcol < p.rope_cols) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float x1 = __uint_as_float(lo_r[e]), x2 = __uint_as_float(hi_r[e]);
            lo[e] = x1 * cs[e] - x2 * sn[e];
            hi[e] = x2 * cs[e] + x1 * sn[e];
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            lo[e] = __uint_as_float(lo_r[e]);
            hi[e] = __uint_as_float(hi_r[e]);
          }
        }
        EpiParams q = p;
        q.mode = kEpiStoreBf16;
        epilogue_chunk(q, row, gcol, lo);
        epilogue_chunk(q, row, gcol + hd / 2, hi);
      }
    }
  } else {
    EpiParams q = p;
    if (q.mode == kEpiRope) q.mode = kEpiStoreBf16;
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(tbase + c * 32, r);
      tmem_wait_ld();
      float v[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
      epilogue_chunk(q, row, tn * BN + c * 32, v);
    }
  }
}

// A_MN / B_MN: the operand is stored MN-major ([K][M] resp. [K][N], M or N
// contiguous) instead of K-major.  MN-major tiles arrive as 64-column TMA
// boxes (8 KB each, 128-byte swizzle) stacked along M/N.
template <bool A_MN, bool B_MN>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_bf16_tcgen05_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                             EpiParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * B_STAGE);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tempty + 2);
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int num_m = (p.M + BM - 1) / BM;
  const int num_n = (p.N + BN - 1) / BN;
  const int num_tiles = num_m * num_n;
  const int num_k = (p.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
    }
    fence_barrier_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int pending[STAGES];
      for (int s = 0; s < STAGES; ++s) pending[s] = -1;
      for (int tile = blockIdx.x; tile < num_tiles && !abort_flag; tile += gridDim.x) {
        int tm, tn;
        tile_coords(tile, num_m, num_n, tm, tn);
        for (int kb = 0; kb < num_k; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1)) {
            set_status(p.status, kStatusGemmTimeout);
            abort_flag = 1;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], A_STAGE + B_STAGE);
          if (A_MN) {
#pragma unroll
            for (int i = 0; i < BM / 64; ++i)
              tma_load_2d(sA + stage * A_STAGE + i * (64 * BK * 2), &tmap_a, tm * BM + 64 * i, kb * BK, &full[stage]);
          } else {
            tma_load_2d(sA + stage * A_STAGE, &tmap_a, kb * BK, tm * BM, &full[stage]);
          }
          if (B_MN) {
#pragma unroll
            for (int i = 0; i < BN / 64; ++i)
              tma_load_2d(sB + stage * B_STAGE + i * (64 * BK * 2), &tmap_b, tn * BN + 64 * i, kb * BK, &full[stage]);
          } else {
            tma_load_2d(sB + stage * B_STAGE, &tmap_b, kb * BK, tn * BN, &full[stage]);
          }
          pending[stage] = (int)phase;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Drain: a load issued into a stage the MMA warp never consumed (abort
      // path) must still land before the CTA exits.
      for (int s = 0; s < STAGES; ++s)
        if (pending[s] >= 0 && !mbar_wait(&full[s], (uint32_t)pending[s])) set_status(p.status, kStatusGemmTimeout);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(BM, BN) | (A_MN ? (1u << 15) : 0u) | (B_MN ? (1u << 16) : 0u);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int tile = blockIdx.x; tile < num_tiles && !abort_flag; tile += gridDim.x) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1)) {
          set_status(p.status, kStatusGemmTimeout);
          abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        bool ok = true;
        for (int kb = 0; kb < num_k; ++kb) {
          if (!mbar_wait(&full[stage], phase)) {
            set_status(p.status, kStatusGemmTimeout);
            abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = A_MN ? smem_desc_mnmajor_sw128(sA + stage * A_STAGE, 64 * BK * 2)
                                      : smem_desc_kmajor_sw128(sA + stage * A_STAGE);
          const uint64_t bdesc = B_MN ? smem_desc_mnmajor_sw128(sB + stage * B_STAGE, 64 * BK * 2)
                                      : smem_desc_kmajor_sw128(sB + stage * B_STAGE);
          // one K step of 16: K-major advances 32 bytes inside the swizzle
          // atom; MN-major advances two 8-row groups (2048 bytes)
          constexpr uint64_t a_step = A_MN ? (2048 >> 4) : (32 >> 4);
          constexpr uint64_t b_step = B_MN ? (2048 >> 4) : (32 >> 4);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            tc_mma_bf16(d_tmem, adesc + a_step * kk, bdesc + b_step * kk, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
    }
  } else {
    // Epilogue warps 2..5: warp w reads TMEM lanes 32*(w%4) .. +31.
    const int quarter = warp & 3;
    float* xpose = reinterpret_cast<float*>(sB + STAGES * B_STAGE + 256) + (warp - 2) * 32 * 33;
    const int row_in_tile = quarter * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      int tm, tn;
      tile_coords(tile, num_m, num_n, tm, tn);
      if (!mbar_wait_warp(&tfull[acc], acc_phase)) {
        set_status(p.status, kStatusGemmTimeout);
        abort_flag = 1;
        break;
      }
      tc_fence_after();
      const int row = tm * BM + row_in_tile;
      const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
      store_tile(p, tbase, row, tn, xpose);
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// One output tile of a pair launch: where its operands start, how many K
// blocks it takes and where its rows go.
struct PairJob {
  int tn;       // N tile: output columns tn*BN ..
  int a_m0;     // first of the tile's 256 rows of A (a row of K-major A, a column of MN-major A)
  int b_n0;     // first of the tile's 256 rows of B (likewise)
  int k0;       // first K of both operands' blocks (0 for K-major A; a group's first row for kGroupK)
  int b_k0;     // first K of B's blocks when it differs (an MN-major B stacked along K)
  int nk;       // K blocks
  int c_row0;   // output row of the tile's first row
  int row_lim;  // output rows >= row_lim are computed and not stored
};

// Group g's clamped row offsets; rows = max(off[g+1] - off[g], 0).  The
// clamp to [0, cap] keeps every load and store of a grouped launch inside
// its operands whatever the device-computed offsets hold.
template <int GROUP>
__device__ __forceinline__ int group_tiles(int rows, int num_m, int num_n) {
  return GROUP == kGroupM ? ((rows + PM - 1) / PM) * num_n : num_m * num_n;
}

// Grouped launches: one warp fills s_off[0..groups] (clamped offsets) and
// s_tstart[0..groups] (exclusive prefix of the groups' tile counts; the last
// entry is the launch's tile count).  Lane l holds groups 8l .. 8l+7.
template <int GROUP>
__device__ __forceinline__ void load_group_table(const EpiParams& p, int num_m, int num_n, int* s_off,
                                                 int* s_tstart) {
  const int lane = threadIdx.x & 31;
  const int cap = GROUP == kGroupM ? p.M : p.K;
  auto clamped = [&](int g) { return min(max(p.group_off[g], 0), cap); };
  int cnt[8];
  int sum = 0;
  int prev = lane * 8 < p.groups ? clamped(lane * 8) : 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int g = lane * 8 + q;
    int t = 0;
    if (g < p.groups) {
      const int next = clamped(g + 1);
      s_off[g] = prev;
      t = group_tiles<GROUP>(max(next - prev, 0), num_m, num_n);
      prev = next;
    }
    cnt[q] = t;
    sum += t;
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  int run = incl - sum;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int g = lane * 8 + q;
    if (g < p.groups) s_tstart[g] = run;
    run += cnt[q];
  }
  if (lane == 31) s_tstart[p.groups] = incl;
  if (lane == 0) s_off[p.groups] = clamped(p.groups);
}

template <int GROUP, bool B_MN>
__device__ __forceinline__ PairJob pair_job(int tile, const EpiParams& p, const int* s_off, const int* s_tstart,
                                            int num_m, int num_n, int num_k) {
  PairJob j;
  int tm, tn;
  if constexpr (GROUP == kGroupNone) {
    tile_coords(tile, num_m, num_n, tm, tn, P_GROUP_M);
    j.a_m0 = tm * PM;
    j.b_n0 = tn * BN;
    j.k0 = j.b_k0 = 0;
    j.nk = num_k;
    j.c_row0 = tm * PM;
    j.row_lim = p.M;
  } else {
    // the group holding this tile: s_tstart[lo] <= tile < s_tstart[hi]
    // (groups without tiles share their start with the next group)
    int lo = 0, hi = p.groups;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_tstart[mid] <= tile)
        lo = mid;
      else
        hi = mid;
    }
    const int g = lo;
    const int r0 = s_off[g], rows = max(s_off[g + 1] - r0, 0);
    if constexpr (GROUP == kGroupM) {
      tile_coords(tile - s_tstart[g], (rows + PM - 1) / PM, num_n, tm, tn, P_GROUP_M);
      j.a_m0 = r0 + tm * PM;
      j.b_n0 = (B_MN ? 0 : g * p.N) + tn * BN;
      j.k0 = 0;
      j.b_k0 = B_MN ? g * p.K : 0;
      j.nk = num_k;
      j.c_row0 = j.a_m0;
      j.row_lim = r0 + rows;
    } else {
      tile_coords(tile - s_tstart[g], num_m, num_n, tm, tn, P_GROUP_M);
      j.a_m0 = tm * PM;
      j.b_n0 = tn * BN;
      j.k0 = j.b_k0 = r0;
      j.nk = (rows + BK - 1) / BK;
      j.c_row0 = g * p.M + tm * PM;
      j.row_lim = g * p.M + p.M;
    }
  }
  j.tn = tn;
  return j;
}

// The CTA-pair kernel.  Roles per CTA as in gemm_bf16_tcgen05_kernel; the
// MMA warp of the odd CTA only takes part in the TMEM allocation.
//   full[s]    leading CTA only: the leader's producer arms it with both
//              CTAs' bytes, both producers' loads complete on it.
//   empty[s]   both CTAs: the MMA commit arrives on both (multicast).
//   tfull[a]   both CTAs: accumulator a ready (multicast commit).
//   tempty[a]  leading CTA only: the 8 epilogue warps of the pair arrive.
// Every wait is bounded; after a timeout each role stops, records
// kStatusGemmTimeout and both CTAs still meet at the final cluster barrier.
template <bool A_MN, bool B_MN, int GROUP>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    gemm_bf16_tcgen05_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                                  const __grid_constant__ CUtensorMap tmap_b, EpiParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + P_STAGES * P_A_STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + P_STAGES * P_B_STAGE);
  uint64_t* empty = full + P_STAGES;
  uint64_t* tfull = empty + P_STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(done + 1);
  int* s_off = reinterpret_cast<int*>(sB + P_STAGES * P_B_STAGE + 256 + XPOSE_BYTES);  // grouped only
  int* s_tstart = s_off + kMaxGroups + 4;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1;
  const int num_clusters = gridDim.x >> 1;
  const int num_m = (p.M + PM - 1) / PM;  // kGroupM: not used (per group)
  const int num_n = (p.N + BN - 1) / BN;
  const int num_k = (p.K + BK - 1) / BK;  // kGroupK: not used (per group)

  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 8);
    }
    mbar_init(done, 1);
    fence_barrier_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_holder, TMEM_COLS);
    tmem_relinquish_pair();
  }
  if constexpr (GROUP != kGroupNone)
    if (warp == 2) load_group_table<GROUP>(p, num_m, num_n, s_off, s_tstart);
  tc_fence_before();
  cluster_sync();  // barriers initialised in both CTAs before any remote use (and the group table filled)
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int num_tiles = GROUP == kGroupNone ? num_m * num_n : s_tstart[p.groups];

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int pending[P_STAGES];
      for (int s = 0; s < P_STAGES; ++s) pending[s] = -1;
      const int row0 = (int)rank * PHALF;
      bool ok = true;
      for (int tile = cluster; tile < num_tiles && ok; tile += num_clusters) {
        const PairJob jb = pair_job<GROUP, B_MN>(tile, p, s_off, s_tstart, num_m, num_n, num_k);
        for (int kb = 0; kb < jb.nk; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1)) {
            set_status(p.status, kStatusGemmTimeout);
            ok = false;
            break;
          }
          const uint32_t bar = mapa_shared(smem_u32(&full[stage]), 0);
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * (P_A_STAGE + P_B_STAGE));
          uint8_t* a_dst = sA + stage * P_A_STAGE;
          uint8_t* b_dst = sB + stage * P_B_STAGE;
          const int ka = jb.k0 + kb * BK, kbb = jb.b_k0 + kb * BK;
          if (A_MN) {
#pragma unroll
            for (int i = 0; i < PHALF / 64; ++i)
              tma_load_2d_pair(a_dst + i * (64 * BK * 2), &tmap_a, jb.a_m0 + row0 + 64 * i, ka, bar);
          } else {
            tma_load_2d_pair(a_dst, &tmap_a, ka, jb.a_m0 + row0, bar);
          }
          if (B_MN) {
#pragma unroll
            for (int i = 0; i < PHALF / 64; ++i)
              tma_load_2d_pair(b_dst + i * (64 * BK * 2), &tmap_b, jb.b_n0 + row0 + 64 * i, kbb, bar);
          } else {
            tma_load_2d_pair(b_dst, &tmap_b, kbb, jb.b_n0 + row0, bar);
          }
          pending[stage] = (int)phase;
          if (++stage == P_STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Tail: every load of this CTA has landed once the MMA released its
      // stage.  After a timeout here the remaining loads were issued more
      // than the wait limit ago.
      for (int s = 0; s < P_STAGES; ++s)
        if (pending[s] >= 0 && !mbar_wait(&empty[s], (uint32_t)pending[s])) {
          set_status(p.status, kStatusGemmTimeout);
          break;
        }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      const uint32_t idesc = idesc_bf16_f32(PM, BN) | (A_MN ? (1u << 15) : 0u) | (B_MN ? (1u << 16) : 0u);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      bool issued = false;  // any MMA at all (a grouped launch may leave a cluster without work)
      for (int tile = cluster; tile < num_tiles && ok; tile += num_clusters) {
        // only kGroupK has a per-tile K; a group without rows has none, and its
        // tiles skip the accumulator altogether (the epilogue stores zeros)
        const int nk = GROUP == kGroupK ? pair_job<GROUP, B_MN>(tile, p, s_off, s_tstart, num_m, num_n, num_k).nk
                                        : num_k;
        if (GROUP == kGroupK && nk == 0) continue;
        if (!mbar_wait_cluster(&tempty[acc], acc_phase ^ 1)) {
          set_status(p.status, kStatusGemmTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_cluster(&full[stage], phase)) {
            set_status(p.status, kStatusGemmTimeout);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = A_MN ? smem_desc_mnmajor_sw128(sA + stage * P_A_STAGE, 64 * BK * 2)
                                      : smem_desc_kmajor_sw128(sA + stage * P_A_STAGE);
          const uint64_t bdesc = B_MN ? smem_desc_mnmajor_sw128(sB + stage * P_B_STAGE, 64 * BK * 2)
                                      : smem_desc_kmajor_sw128(sB + stage * P_B_STAGE);
          constexpr uint64_t a_step = A_MN ? (2048 >> 4) : (32 >> 4);
          constexpr uint64_t b_step = B_MN ? (2048 >> 4) : (32 >> 4);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc_mma_bf16_pair(d_tmem, adesc + a_step * kk, bdesc + b_step * kk, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          issued = true;
          tc_commit_pair_mc(&empty[stage], 0x3);
          if (++stage == P_STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit_pair_mc(&tfull[acc], 0x3);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      // Every MMA issued above has completed (and stopped reading both CTAs'
      // shared memory and writing their TMEM) once this commit arrives.
      if (issued) {
        tc_commit_pair(done);
        if (!mbar_wait(done, 0)) set_status(p.status, kStatusGemmTimeout);
      }
    }
  } else {
    const int quarter = warp & 3;
    const int row_in_tile = (int)rank * PHALF + quarter * 32 + lane;
    float* xpose = reinterpret_cast<float*>(sB + P_STAGES * P_B_STAGE + 256) + (warp - 2) * 32 * 33;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = cluster; tile < num_tiles; tile += num_clusters) {
      const PairJob jb = pair_job<GROUP, B_MN>(tile, p, s_off, s_tstart, num_m, num_n, num_k);
      if (GROUP == kGroupK && jb.nk == 0) {
        // a group without rows: the product is zero; no accumulator was used
        EpiParams q = p;
        q.M = jb.row_lim;
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0.f;
          epilogue_chunk(q, jb.c_row0 + row_in_tile, jb.tn * BN + c * 32, v);
        }
        continue;
      }
      if (!mbar_wait_warp(&tfull[acc], acc_phase)) {
        set_status(p.status, kStatusGemmTimeout);
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
      if constexpr (GROUP == kGroupNone) {
        store_tile(p, tbase, jb.c_row0 + row_in_tile, jb.tn, xpose);
      } else {
        EpiParams q = p;
        q.M = jb.row_lim;
        store_tile(q, tbase, jb.c_row0 + row_in_tile, jb.tn, xpose);
      }
      tc_fence_before();
      if (leader)
        mbar_arrive_warp(&tempty[acc]);
      else
        mbar_arrive_warp_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before();
  cluster_sync();  // no CTA leaves while its peer may still touch its shared memory
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// Row-major BF16 matrix [rows, cols] with leading dimension ld (elements),
// boxes of 64 columns x box_rows rows, 128-byte swizzle, zero fill outside.
// K-major operands use rows = M/N, cols = K, box_rows = BM/BN; MN-major
// operands use rows = K, cols = M/N, box_rows = BK.
bool make_tmap(CUtensorMap* m, const void* base, long rows, long cols, long ld, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

}  // namespace

namespace {
thread_local const char* g_launch_err = "no error";
}

int launch_result() {
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) return 0;
  g_launch_err = cudaGetErrorString(e);
  return -4;
}

const char* last_launch_error() { return g_launch_err; }

bool make_tmap_bf16(CUtensorMap* m, const void* base, long rows, long cols, long ld, int box_rows) {
  return make_tmap(m, base, rows, cols, ld, box_rows);
}

const char* gemm_check(const GemmArgs& g) {
  if (g.M <= 0 || g.N <= 0 || g.K <= 0) return "gemm: M, N and K must be positive";
  // K is the contiguous dimension of a K-major operand; with both operands
  // MN-major it is the outer one and any K works (the last block reads zeros)
  if (g.K % 8 && !(g.a_mn && g.b_mn)) return "gemm: K must be a multiple of 8 (16-byte TMA rows)";
  if (g.lda % 8 || g.ldb % 8) return "gemm: lda/ldb must be multiples of 8 elements";
  if (g.lda < (g.a_mn ? g.M : g.K) || g.ldb < (g.b_mn ? g.N : g.K)) return "gemm: lda/ldb smaller than a row";
  if ((reinterpret_cast<uintptr_t>(g.A) | reinterpret_cast<uintptr_t>(g.B)) & 15) return "gemm: A/B not 16-byte aligned";
  if (!g.C) return "gemm: null output";
  if (reinterpret_cast<uintptr_t>(g.C) & 15) return "gemm: C not 16-byte aligned";
  if (g.ldc % 8) return "gemm: ldc must be a multiple of 8";
  switch (g.epi) {
    case kEpiStoreBf16:
    case kEpiF32:
    case kEpiF32Accumulate:
      break;
    case kEpiResidualBf16:
      if (!g.R || (reinterpret_cast<uintptr_t>(g.R) & 15) || g.ldr % 8) return "gemm: bad residual operand";
      break;
    case kEpiSwiGLUBwd:
      if (!g.R || (reinterpret_cast<uintptr_t>(g.R) & 15) || g.ldr % 8 || g.ldr < 2L * g.N)
        return "gemm: SwiGLU backward needs the gate/up pairs R [M, 2N]";
      if (g.ldc < 2L * g.N) return "gemm: SwiGLU backward writes C [M, 2N]";
      break;
    case kEpiSwiGLU:
      if (g.N % 2) return "gemm: SwiGLU needs an even N";
      if (g.C2 && ((reinterpret_cast<uintptr_t>(g.C2) & 15) || g.ldc2 % 8)) return "gemm: bad SwiGLU gu output";
      break;
    case kEpiRope:
      if (!(g.head_dim == 64 || g.head_dim == 128)) return "gemm: RoPE head_dim must be 64 or 128";
      if (g.rope_cols % g.head_dim) return "gemm: rope_cols must be a multiple of head_dim";
      if (!g.rope_cos || !g.rope_sin || g.seq <= 0) return "gemm: RoPE tables missing";
      if ((reinterpret_cast<uintptr_t>(g.rope_cos) | reinterpret_cast<uintptr_t>(g.rope_sin)) & 15)
        return "gemm: RoPE tables must be 16-byte aligned";
      break;
    default:
      return "gemm: unknown epilogue";
  }
  return nullptr;
}

namespace {

// Clusters of two that fit on the device at once (one CTA per SM; SMs left
// over by an odd GPC stay idle), or 0 when no pair can be placed.
template <bool A_MN, bool B_MN, int GROUP = kGroupNone>
int pair_clusters() {
  static int n = -1;
  static std::once_flag once;
  std::call_once(once, [] {
    auto* k = gemm_bf16_tcgen05_pair_kernel<A_MN, B_MN, GROUP>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) != cudaSuccess) {
      n = 0;
      return;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * num_sms(), 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    int c = 0;
    n = cudaOccupancyMaxActiveClusters(&c, k, &cfg) == cudaSuccess ? c : 0;
    cudaGetLastError();
  });
  return n;
}

template <bool A_MN, bool B_MN, int GROUP = kGroupNone>
int launch_pair(const CUtensorMap& ta, const CUtensorMap& tb, const EpiParams& p, int clusters, cudaStream_t s) {
  gemm_bf16_tcgen05_pair_kernel<A_MN, B_MN, GROUP><<<2 * clusters, THREADS, SMEM_BYTES, s>>>(ta, tb, p);
  return launch_result();
}

template <bool A_MN, bool B_MN>
int gemm_pair(const GemmArgs& g, const EpiParams& p, cudaStream_t s) {
  const int avail = pair_clusters<A_MN, B_MN>();
  if (avail <= 0) return 1;  // not placeable: the caller uses the single-CTA kernel
  CUtensorMap ta, tb;
  if (A_MN ? !make_tmap(&ta, g.A, g.K, g.M, g.lda, BK) : !make_tmap(&ta, g.A, g.M, g.K, g.lda, PHALF)) return -3;
  if (B_MN ? !make_tmap(&tb, g.B, g.K, g.N, g.ldb, BK) : !make_tmap(&tb, g.B, g.N, g.K, g.ldb, PHALF)) return -3;
  const int tiles = ((g.M + PM - 1) / PM) * ((g.N + BN - 1) / BN);
  return launch_pair<A_MN, B_MN>(ta, tb, p, tiles < avail ? tiles : avail, s);
}

EpiParams epi_params(const GemmArgs& g) {
  EpiParams p;
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.mode = g.epi;
  p.C = g.C;
  p.ldc = g.ldc;
  p.R = g.R;
  p.ldr = g.ldr;
  p.C2 = g.C2;
  p.ldc2 = g.ldc2;
  p.rope_cos = g.rope_cos;
  p.rope_sin = g.rope_sin;
  p.rope_cols = g.rope_cols;
  p.head_dim = g.head_dim;
  p.seq = g.seq;
  p.status = g.status;
  p.group_off = nullptr;
  p.groups = 0;
  return p;
}

template <bool A_MN, bool B_MN, int GROUP>
int grouped_pair(const CUtensorMap& ta, const CUtensorMap& tb, const EpiParams& p, long max_tiles, cudaStream_t s) {
  const int avail = pair_clusters<A_MN, B_MN, GROUP>();
  if (avail <= 0) return -2;
  return launch_pair<A_MN, B_MN, GROUP>(ta, tb, p, (int)(max_tiles < avail ? max_tiles : avail), s);
}

}  // namespace

const char* gemm_grouped_check(const GemmArgs& g, const int32_t* offsets, int groups, int mode) {
  if (const char* e = gemm_check(g)) return e;
  if (!offsets || (reinterpret_cast<uintptr_t>(offsets) & 3)) return "grouped gemm: offsets missing or misaligned";
  if (groups < 1 || groups > kMaxGroups) return "grouped gemm: 1 <= groups <= 256";
  if (mode == kGemmGroupRows) {
    if (g.a_mn) return "grouped gemm (rows): A must be K-major";
    if (g.epi == kEpiRope || g.epi == kEpiResidualBf16) return "grouped gemm (rows): no RoPE or residual epilogue";
    if ((long)groups * (g.b_mn ? g.K : g.N) > 0x7fffffffL) return "grouped gemm (rows): stacked B too tall";
  } else if (mode == kGemmGroupK) {
    if (!g.a_mn || !g.b_mn) return "grouped gemm (K): both operands must be MN-major";
    if (g.epi != kEpiStoreBf16 && g.epi != kEpiF32 && g.epi != kEpiF32Accumulate)
      return "grouped gemm (K): store or FP32 epilogues only";
    if ((long)groups * g.M > 0x7fffffffL) return "grouped gemm (K): stacked C too tall";
  } else {
    return "grouped gemm: unknown grouping";
  }
  return nullptr;
}

int launch_gemm_grouped(const GemmArgs& g, const int32_t* offsets, int groups, int mode, cudaStream_t stream) {
  if (gemm_grouped_check(g, offsets, groups, mode)) return -1;
  EpiParams p = epi_params(g);
  p.group_off = offsets;
  p.groups = groups;
  const long num_n = (g.N + BN - 1) / BN;
  CUtensorMap ta, tb;
  if (mode == kGemmGroupRows) {
    // A [M, K]: every group's rows; B stacked per group along N (K-major) or K (MN-major)
    if (!make_tmap(&ta, g.A, g.M, g.K, g.lda, PHALF)) return -3;
    if (g.b_mn ? !make_tmap(&tb, g.B, (long)groups * g.K, g.N, g.ldb, BK)
               : !make_tmap(&tb, g.B, (long)groups * g.N, g.K, g.ldb, PHALF))
      return -3;
    const long max_tiles = ((g.M + PM - 1) / PM + groups) * num_n;  // each group adds at most one partial M tile
    return g.b_mn ? grouped_pair<false, true, kGroupM>(ta, tb, p, max_tiles, stream)
                  : grouped_pair<false, false, kGroupM>(ta, tb, p, max_tiles, stream);
  }
  // A stored [K, M], B stored [K, N]: K = every group's rows
  if (!make_tmap(&ta, g.A, g.K, g.M, g.lda, BK) || !make_tmap(&tb, g.B, g.K, g.N, g.ldb, BK)) return -3;
  const long tiles = (long)groups * ((g.M + PM - 1) / PM) * num_n;
  return grouped_pair<true, true, kGroupK>(ta, tb, p, tiles, stream);
}

int launch_gemm(const GemmArgs& g, cudaStream_t stream) {
  if (gemm_check(g)) return -1;
  static bool attr_done = false;
  if (!attr_done) {
    bool ok = cudaFuncSetAttribute(gemm_bf16_tcgen05_kernel<false, false>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) == cudaSuccess;
    ok &= cudaFuncSetAttribute(gemm_bf16_tcgen05_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               SMEM_BYTES) == cudaSuccess;
    ok &= cudaFuncSetAttribute(gemm_bf16_tcgen05_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               SMEM_BYTES) == cudaSuccess;
    ok &= cudaFuncSetAttribute(gemm_bf16_tcgen05_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               SMEM_BYTES) == cudaSuccess;
    if (!ok) return -2;
    attr_done = true;
  }
  const EpiParams p = epi_params(g);
  // More than one 128-row tile of M: CTA pairs (256 x 256 tiles).
  if (g.M > BM) {
    int rc;
    if (!g.a_mn && !g.b_mn)
      rc = gemm_pair<false, false>(g, p, stream);
    else if (g.a_mn && !g.b_mn)
      rc = gemm_pair<true, false>(g, p, stream);
    else if (!g.a_mn && g.b_mn)
      rc = gemm_pair<false, true>(g, p, stream);
    else
      rc = gemm_pair<true, true>(g, p, stream);
    if (rc <= 0) return rc;
  }
  CUtensorMap ta, tb;
  if (g.a_mn ? !make_tmap(&ta, g.A, g.K, g.M, g.lda, BK) : !make_tmap(&ta, g.A, g.M, g.K, g.lda, BM)) return -3;
  if (g.b_mn ? !make_tmap(&tb, g.B, g.K, g.N, g.ldb, BK) : !make_tmap(&tb, g.B, g.N, g.K, g.ldb, BN)) return -3;
  const int tiles = ((g.M + BM - 1) / BM) * ((g.N + BN - 1) / BN);
  const int grid = tiles < num_sms() ? tiles : num_sms();
  if (!g.a_mn && !g.b_mn)
    gemm_bf16_tcgen05_kernel<false, false><<<grid, THREADS, SMEM_BYTES, stream>>>(ta, tb, p);
  else if (g.a_mn && !g.b_mn)
    gemm_bf16_tcgen05_kernel<true, false><<<grid, THREADS, SMEM_BYTES, stream>>>(ta, tb, p);
  else if (!g.a_mn && g.b_mn)
    gemm_bf16_tcgen05_kernel<false, true><<<grid, THREADS, SMEM_BYTES, stream>>>(ta, tb, p);
  else
    gemm_bf16_tcgen05_kernel<true, true><<<grid, THREADS, SMEM_BYTES, stream>>>(ta, tb, p);
  return launch_result();
}

}  // namespace mt
