// CPU Adam on host tiles: BF16 weights and gradients, FP32 moments, no FP32
// master copy (MegaTrain paperlayer.ai summary §2 "Training memory": 12 bytes
// per parameter; §3 "Execution workflow": Adam runs on the CPU because it is
// compute-light and I/O-heavy; author's blog: "a string of additions,
// subtractions, multiplications, and divisions").
//
// Plain C++ loops over contiguous ranges, compiled with -O3 -fno-math-errno
// so the compiler vectorises them for the host ISA (NEON/SVE on Grace,
// SSE/AVX on x86) without intrinsics; IEEE FP32 semantics are kept
// (no fast-math).
#include <cmath>
#include <cstdint>
#include <cstring>

#include "runtime.h"

namespace mt {

static inline float bf16_bits_to_f32(uint16_t b) {
  const uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// Round-to-nearest-even FP32 -> BF16 bit pattern (finite inputs).
static inline uint16_t f32_to_bf16_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

void adam_range(uint16_t* __restrict__ w, const uint16_t* __restrict__ g, float* __restrict__ m,
                float* __restrict__ v, size_t n, const AdamHyper& h) {
  const float b1 = h.beta1, b2 = h.beta2;
  const float omb1 = 1.0f - b1, omb2 = 1.0f - b2;
  const double t = static_cast<double>(h.step);
  const float bc1 = static_cast<float>(1.0 - std::pow(static_cast<double>(b1), t));
  const float bc2 = static_cast<float>(1.0 - std::pow(static_cast<double>(b2), t));
  const float lr = h.lr, eps = h.eps, wd = h.weight_decay;
  // bias corrections as multiplications (1/(1-b^t) once per call): two fewer
  // divisions per element; the rounding differs from dividing by < 1 FP32 ulp
  const float ibc1 = 1.0f / bc1, ibc2 = 1.0f / bc2;
  for (size_t i = 0; i < n; ++i) {
    const float gi = bf16_bits_to_f32(g[i]);
    const float mi = b1 * m[i] + omb1 * gi;
    const float vi = b2 * v[i] + omb2 * gi * gi;
    m[i] = mi;
    v[i] = vi;
    const float mhat = mi * ibc1;
    const float vhat = vi * ibc2;
    const float wi = bf16_bits_to_f32(w[i]);
    const float upd = mhat / (std::sqrt(vhat) + eps) + wd * wi;
    w[i] = f32_to_bf16_bits(wi - lr * upd);
  }
}

// Copy BF16 gradient bits from a pinned slab into the tile's G section and
// report whether any value is NaN or Inf (exponent bits all ones).
bool copy_grad_check_finite(uint16_t* __restrict__ dst, const uint16_t* __restrict__ src, size_t n) {
  uint32_t bad = 0;
  for (size_t i = 0; i < n; ++i) {
    const uint16_t b = src[i];
    dst[i] = b;
    bad |= static_cast<uint32_t>((b & 0x7F80u) == 0x7F80u);
  }
  return bad == 0;
}

// dst += src (BF16 gradients of another micro-batch): the sum in FP32, rounded
// to nearest even; reports whether src holds a NaN or Inf.
bool add_grad_check_finite(uint16_t* __restrict__ dst, const uint16_t* __restrict__ src, size_t n) {
  uint32_t bad = 0;
  for (size_t i = 0; i < n; ++i) {
    const uint16_t b = src[i];
    bad |= static_cast<uint32_t>((b & 0x7F80u) == 0x7F80u);
    dst[i] = f32_to_bf16_bits(bf16_bits_to_f32(dst[i]) + bf16_bits_to_f32(b));
  }
  return bad == 0;
}

}  // namespace mt

extern "C" int mt_adam_host(uint16_t* w, const uint16_t* g, float* m, float* v, size_t n, int64_t t, float lr,
                            float beta1, float beta2, float eps, float weight_decay) {
  if (t < 1 || (n && (!w || !g || !m || !v))) return -1;
  mt::AdamHyper h{lr, beta1, beta2, eps, weight_decay, t};
  mt::adam_range(w, g, m, v, n, h);
  return 0;
}
