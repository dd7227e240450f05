// Causal grouped-query flash attention: argument checks, the launch entry
// points, and the one HBM-bound step of the backward pass,
//   delta[b, h, s] = sum_d dO[token, h, d] * O[token, h, d],
// that the tensor-core backward kernels (attention_tc.cu) read per query row.
// Forward and backward proper run on tcgen05 in attention_tc.cu; the
// backward is deterministic (no atomics).  Query head h reads kv head
// h * Hkv / Hq.
//
// MegaTrain names "Attention and MLP kernels" inside its stateless templates
// (paperlayer.ai summary §A.4) without giving them; this design is the
// library's own.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace mt {

namespace {

// One group of HD/8 threads per (token, head) row: 16-byte loads of dO and O,
// FP32 products, shuffle reduction inside the group.
template <int HD>
__global__ void attn_delta_kernel(const bf16* dout, const bf16* o, long ldo, int B, int S, int Hq, float* delta) {
  constexpr int G = HD / 8;
  const long gid = ((long)blockIdx.x * blockDim.x + threadIdx.x);
  const long row = gid / G;
  const int c = gid % G;
  const long T = (long)B * S;
  float acc = 0.f;
  const bool ok = row < T * Hq;
  long tok = 0;
  int h = 0;
  if (ok) {
    tok = row / Hq;
    h = row % Hq;
    const uint4 x = *reinterpret_cast<const uint4*>(dout + tok * ldo + (long)h * HD + c * 8);
    const uint4 y = *reinterpret_cast<const uint4*>(o + tok * ldo + (long)h * HD + c * 8);
    const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc += __uint_as_float(xs[j] << 16) * __uint_as_float(ys[j] << 16);
      acc += __uint_as_float(xs[j] & 0xFFFF0000u) * __uint_as_float(ys[j] & 0xFFFF0000u);
    }
  }
#pragma unroll
  for (int off = G / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, G);
  if (ok && c == 0) {
    const long b = tok / S, s = tok % S;
    delta[(b * Hq + h) * S + s] = acc;
  }
}

template <int HD>
int bwd_impl(const AttnArgs& x, cudaStream_t s) {
  const long rows = (long)x.batch * x.seq * x.n_heads;
  const long threads = rows * (HD / 8);
  attn_delta_kernel<HD><<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(x.dout, x.o, x.ldo, x.batch, x.seq,
                                                                         x.n_heads, x.delta);
  if (launch_result() != 0) return -4;
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
