// Host-side structures of the layer-streamed training runtime.
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include "../../include/mt.h"
#include "kernels.h"

namespace mt {

constexpr int64_t kPage = 4096;     // tile section alignment (single-burst DMA of page-aligned blocks)
constexpr int64_t kTensorAlign = 256;  // sub-tensor alignment inside a section

inline int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

struct AdamHyper {
  float lr, beta1, beta2, eps, weight_decay;
  int64_t step;
};
void adam_range(uint16_t* w, const uint16_t* g, float* m, float* v, size_t n, const AdamHyper& h);
bool copy_grad_check_finite(uint16_t* dst, const uint16_t* src, size_t n);
bool add_grad_check_finite(uint16_t* dst, const uint16_t* src, size_t n);

// ------------------------------------------------------------------ tiles
enum TileKind { kTileEmbed = 0, kTileLayer = 1, kTileHead = 2 };

struct TensorSlot {
  std::string name;
  int ndim;
  int64_t shape[2];
  int64_t offset;  // bytes inside the W section
  int64_t numel;
};

struct TileLayout {
  TileKind kind;
  std::vector<TensorSlot> tensors;
  int64_t n_params = 0;
  int64_t w_bytes = 0;  // W section bytes (page multiple); G section identical
  int64_t mv_bytes = 0; // M (and V) section bytes (page multiple)
  int64_t off_w = 0, off_g = 0, off_m = 0, off_v = 0;
  int64_t tile_bytes = 0;
  const TensorSlot& slot(const char* n) const;
  bool has(const char* n) const;
};

// MoE layers pad each expert's permuted rows to a multiple of this (one K
// block of the grouped weight-gradient GEMM).
constexpr int kMoeRowAlign = 64;

struct Dims {
  int L, d, Hq, Hkv, hd, f, V, B, S;
  int E = 0, k = 0;  // MoE layers: experts and experts per token (E = 0: dense)
  long T;       // B*S
  long Tc;      // rows per MLP chunk (T when the MLP runs on the whole step at once)
  int Dq;       // Hq*hd
  int Dqkv;     // (Hq + 2 Hkv) * hd
};

Dims dims_of(const mt_config& c);
// tied: the embedding tile also holds the final norm gain and serves as the LM
// head's weight (there is no head tile).
TileLayout make_layout(TileKind kind, const Dims& d, bool tied = false);

// ------------------------------------------------------------------ device workspace
// Bound views of one layer tile (weights in a streamed buffer, or gradients
// in a gradient buffer): pointers only, no storage (the "Bind" of a template).
struct LayerView {
  bf16 *g1, *wqkv, *wo, *g2, *wgu, *wd;
  bf16* wr = nullptr;  // MoE layers: router [E, d]; wgu/wd then stack the experts
};
struct HeadView {
  bf16 *gf, *wh;
};
LayerView bind_layer(const TileLayout& lay, void* base);
HeadView bind_head(const TileLayout& lay, void* base);

// Activations of one layer pass.
struct LayerActs {
  bf16* x;       // input (not owned: checkpoint or block buffer)
  bf16* n1;
  float* rstd1;
  bf16* qkv;
  bf16* o;
  float* lse;
  bf16* h;
  bf16* n2;
  float* rstd2;
  bf16* gu;      // may be null in plain forward
  bf16* a;
  // MoE layers: router logits, routing, the permuted rows and the experts' outputs
  float* moe_logits = nullptr;  // [T, E]
  int32_t *moe_idx = nullptr, *moe_order = nullptr, *moe_pos = nullptr, *moe_off = nullptr;
  float* moe_gates = nullptr;   // [T, k]
  bf16 *moe_xp = nullptr, *moe_ap = nullptr, *moe_gup = nullptr, *moe_yp = nullptr;
};

struct Workspace {
  // backward scratch
  bf16 *dx_a, *dx_b;    // ping-pong dx between layers
  bf16 *dh, *dgu, *dn, *dout, *dqkv;
  float* delta;
  float* dg_partial;
  float *dwd_f32, *dwgu_f32;  // FP32 W_d / W_gu gradients accumulated over MLP row chunks (chunked MLP only)
  // head
  bf16* nf;
  float* rstd_f;
  float* z;        // [chunk, V] FP32 logits
  bf16* dz;        // [chunk, V]
  bf16* dnf;       // [T, d]
  float* dwh_f32;  // [V, d]
  float* loss_rows;
  float* loss;     // [1]
  // tokens
  int32_t* inp;    // [T]
  int32_t* tgt;    // [T]
  int32_t* emb_off;  // [V+1]
  int32_t* emb_pos;  // [T]
  int32_t* emb_rows; // [min(T, V)] token ids that occur in the step, ascending
  int32_t* tokens_dev;  // [B, S+1] (device-token entry point)
  float *rope_cos, *rope_sin;  // [S, hd/2]
  int* status;
  int* grad_flags;  // [3 L + 8]: one non-finite flag per gradient visit (direct gradient landing)
  long head_chunk;  // rows per LM-head chunk
  // MoE backward scratch
  bf16 *moe_dyp = nullptr, *moe_dgup = nullptr, *moe_dxp = nullptr, *moe_ds = nullptr, *moe_dn2r = nullptr;
  float* moe_dgates = nullptr;
  int32_t* moe_scratch = nullptr;  // counting-sort scratch
};

// Counts what the launch sequences issued (for the step statistics).
struct LaunchStats {
  int64_t kernels = 0;
  int64_t gemms = 0;
  double gemm_flops = 0;
  double gemm_ms = 0;
  bool time_gemms = false;
  std::vector<cudaEvent_t>* gemm_events = nullptr;  // pairs
  std::vector<double>* gemm_event_flops = nullptr;
};

// The stateless layer template: the kernel sequences of one decoder layer,
// parameterised only by bound views and workspace pointers.
struct LayerTemplate {
  Dims dm;
  float eps;
  cudaStream_t s;
  const Workspace* ws;
  LaunchStats* stats;

  // Optional debugging hook called after every kernel launch with its name
  // (used by MT_TRACE to wait for and report each kernel).
  float loss_scale = 1.f;  // the head's cross-entropy is scaled by loss_scale / tokens (micro-batches)
  void (*trace_fn)(void* ctx, const char* kernel) = nullptr;
  void* trace_ctx = nullptr;
  void trace(const char* kernel) const {
    if (trace_fn) trace_fn(trace_ctx, kernel);
  }

  int gemm(const GemmArgs& g) const;
  int gemm_grouped(const GemmArgs& g, const int32_t* offsets, int groups, int mode, long rows) const;
  // x -> x_out (x_out == nullptr: stop after the MLP activation).  keep_gu: also
  // store the gate/up pre-activations (needed by backward).
  int forward(const LayerView& w, LayerActs& a, bf16* x_out, bool keep_gu) const;
  // Given the layer's forward activations and dx_out, write dx_in and the
  // layer's gradients into gv (BF16, tile layout).
  int backward(const LayerView& w, const LayerActs& a, const bf16* dx_out, bf16* dx_in, const LayerView& gv) const;
  int mlp_backward_chunked(const LayerView& w, const LayerActs& a, const bf16* dx_out, const LayerView& gv) const;
  // MoE layers: the MLP half from n2 (and h for the residual) to x_out, and its
  // backward from dx_out to dn2 in ws->dn; the per-expert row counts stay on
  // the device (grouped GEMMs), so neither synchronises with the host.
  int moe_forward(const LayerView& w, LayerActs& a, bf16* x_out) const;
  int moe_backward(const LayerView& w, const LayerActs& a, const bf16* dx_out, const LayerView& gv) const;
  // Final norm + LM head + cross-entropy, forward and backward in chunks.
  int head(const HeadView& w, const bf16* x_L, bf16* dx_L, const HeadView& gv) const;
  int embed_fwd(const bf16* E, bf16* x0) const;
  int embed_bwd(const bf16* dx0, bf16* dE) const;
  // Gradient rows of the U token ids in ws->emb_rows only, packed [U, d].
  int embed_bwd_rows(const bf16* dx0, bf16* out, int U) const;
};

}  // namespace mt
