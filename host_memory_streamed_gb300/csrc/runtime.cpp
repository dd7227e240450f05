// The layer-streamed training step: host-authoritative tiles, two device
// weight buffers, three CUDA streams ordered by events, CPU worker threads.
//
//   caller thread   compute stream: waits Weights-Ready[v], binds the tile in
//                   buffer b, launches the template's kernels, records
//                   Buffer-Free[v] and (for backward visits) Grads-Done[v].
//   loader thread   H2D stream: for each visit that needs a tile, waits for the
//                   buffer's previous user to be done (Buffer-Free), then has
//                   the packer threads copy the pageable tile into one of two
//                   pinned staging chunks while the other chunk's DMA runs,
//                   and records Weights-Ready[v].
//   d2h thread      D2H stream: after Grads-Done[v], copies the gradient buffer
//                   (layers alternate two; the head and the embedding rows use
//                   a third) into free pinned slabs (24 x 64 MiB by default)
//                   and records Grads-Evacuated[v] so the compute stream may
//                   reuse the buffer.
//   accumulator     copies each landed slab into the tile's G section, returns
//                   the slab, and hands the slab's range to the Adam pool.
//   Adam pool       updates W, M, V of each landed range while the GPU keeps
//                   working on earlier layers.
//
// MegaTrain sources: paperlayer.ai summary §3 (execution workflow, three
// streams, background gradient evacuation), §A.1 (layer-contiguous tiles,
// pinned slab recycling, two pinned staging buffers), §A.2 (ComputeStream /
// WeightStream / GradStream; weights-ready, backward-done and buffer-free
// events), §A.3 (flat-buffer streaming with one copy per layer, pinned
// gradient slabs (12 there) with a background accumulator, preallocated
// workspaces),
// §A.4 (stateless templates, ping-pong binding, no CUDA graphs); hyper.ai
// summary 方法 ¶2-6 (block recompute order, JIT packer thread, Weights-Ready
// event before Bind); author's blog (per-block F/W/G figure).
//
// Replica group (n_replicas >= 2): one process per GPU, every process mapping
// one shared-memory segment that holds a control block and all host tiles.
// Each replica runs the step above on its own batch; its accumulator adds a
// gradient chunk into the shared G only when the chunk's turn counter says
// replicas 0 .. r-1 have added theirs, and the last replica's Adam pool
// updates each chunk once its own addition is in.  Each tile's finished
// update is published in the control block, and every replica's loader waits
// for it before uploading that tile for the next step.
#include <atomic>
#include <chrono>
#include <cmath>
#include <condition_variable>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <deque>
#include <functional>
#include <map>
#include <memory>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include <nvtx3/nvToolsExt.h>
#include <errno.h>
#include <fcntl.h>
#include <sys/mman.h>
#include <sys/resource.h>
#include <sys/stat.h>
#include <sys/syscall.h>
#include <unistd.h>

#include "runtime.h"

namespace {
// NVTX ranges for timeline profilers (no-ops unless one is attached): one per
// visit on the compute thread, per weight upload on the loader thread, per
// gradient evacuation on the D2H thread, per accumulated slab and per Adam task.
struct NvtxRange {
  explicit NvtxRange(const char* fmt, int a = 0, int b = 0) {
    char name[64];
    std::snprintf(name, sizeof name, fmt, a, b);
    nvtxRangePushA(name);
  }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
const char* const kVisitRangeFmt[] = {"embed fwd", "layer fwd %d (tile %d)", "head", "recompute %d (tile %d)",
                                      "layer bwd %d (tile %d)", "embed bwd"};
}  // namespace

namespace mt {
namespace {

using Clock = std::chrono::steady_clock;

double ms_since(Clock::time_point t0) {
  return std::chrono::duration<double, std::milli>(Clock::now() - t0).count();
}

struct MtError {
  int code;
  std::string msg;
};

// ------------------------------------------------------------------ small thread pool
class Pool {
 public:
  // nice > 0 lowers the workers' scheduling priority (Linux niceness of each
  // worker thread), so that work on the step's critical path preempts them.
  explicit Pool(int n, int nice = 0) {
    for (int i = 0; i < n; ++i)
      th_.emplace_back([this, nice] {
        if (nice > 0) setpriority(PRIO_PROCESS, (id_t)syscall(SYS_gettid), nice);
        run();
      });
  }
  ~Pool() {
    {
      std::lock_guard<std::mutex> g(mu_);
      stop_ = true;
    }
    cv_.notify_all();
    for (auto& t : th_) t.join();
  }
  // Tasks run in ascending key order (equal keys in submission order).
  void submit(std::function<void()> f, int key = 0) {
    {
      std::lock_guard<std::mutex> g(mu_);
      q_[key].push_back(std::move(f));
      ++queued_;
      ++pending_;
    }
    cv_.notify_one();
  }
  // Wait until every submitted task finished; false on timeout.
  bool wait_idle(int64_t timeout_ms) {
    std::unique_lock<std::mutex> g(mu_);
    return done_cv_.wait_for(g, std::chrono::milliseconds(timeout_ms), [this] { return pending_ == 0; });
  }
  int size() const { return (int)th_.size(); }

 private:
  void run() {
    while (true) {
      std::function<void()> f;
      {
        std::unique_lock<std::mutex> g(mu_);
        cv_.wait(g, [this] { return stop_ || queued_ > 0; });
        if (stop_ && queued_ == 0) return;
        auto it = q_.begin();
        f = std::move(it->second.front());
        it->second.pop_front();
        if (it->second.empty()) q_.erase(it);
        --queued_;
      }
      f();
      {
        std::lock_guard<std::mutex> g(mu_);
        if (--pending_ == 0) done_cv_.notify_all();
      }
    }
  }
  std::vector<std::thread> th_;
  std::map<int, std::deque<std::function<void()>>> q_;
  std::mutex mu_;
  std::condition_variable cv_, done_cv_;
  int64_t pending_ = 0, queued_ = 0;
  bool stop_ = false;
};

// ------------------------------------------------------------------ schedule
enum VisitKind { kEmbedFwd, kLayerFwd, kHead, kRecompute, kLayerBwd, kEmbedBwd };
static_assert(kEmbedFwd == MT_VISIT_EMBED_FWD && kLayerFwd == MT_VISIT_LAYER_FWD && kHead == MT_VISIT_HEAD &&
                  kRecompute == MT_VISIT_RECOMPUTE && kLayerBwd == MT_VISIT_LAYER_BWD && kEmbedBwd == MT_VISIT_EMBED_BWD,
              "visit kinds of the C-ABI");

struct Visit {
  VisitKind kind;
  int tile;
  int layer;
  int buf = -1;        // device weight buffer (-1: none)
  bool h2d = false;    // stream the tile into buf before this visit
  int prev_user = -1;  // previous visit that used buf
  bool grads = false;
  int gbuf = -1;
  int prev_gbuf_user = -1;
};

// keep_from: layers keep_from .. L-1 keep their internals from the forward
// (their backward visits recompute nothing); layers 0 .. keep_from-1 form the
// checkpoint blocks of K layers.
std::vector<Visit> build_schedule(int L, int K, int keep_from, bool single_buffer, int head_tile) {
  std::vector<Visit> v;
  v.push_back({kEmbedFwd, 0, -1});
  for (int i = 0; i < L; ++i) v.push_back({kLayerFwd, i + 1, i});
  v.push_back({kHead, head_tile, -1});
  for (int j = L - 1; j >= keep_from; --j) v.push_back({kLayerBwd, j + 1, j});
  const int nblk = (keep_from + K - 1) / K;
  for (int b = nblk - 1; b >= 0; --b) {
    const int s = b * K, e = std::min(keep_from, s + K);
    for (int j = s; j < e - 1; ++j) v.push_back({kRecompute, j + 1, j});
    for (int j = e - 1; j >= s; --j) v.push_back({kLayerBwd, j + 1, j});
  }
  v.push_back({kEmbedBwd, 0, -1});
  // buffer assignment with residency reuse
  int held[2] = {-1, -1}, last_user[2] = {-1, -1}, prev_buf = 1;
  int glast[3] = {-1, -1, -1}, gnext = 0;
  for (int i = 0; i < (int)v.size(); ++i) {
    Visit& x = v[i];
    if (x.kind != kEmbedBwd) {
      int b = -1;
      for (int c = 0; c < (single_buffer ? 1 : 2); ++c)
        if (held[c] == x.tile) b = c;
      if (b < 0) {
        b = single_buffer ? 0 : (prev_buf ^ 1);
        x.h2d = true;
        held[b] = x.tile;
      }
      x.buf = b;
      x.prev_user = last_user[b];
      last_user[b] = i;
      prev_buf = b;
    }
    x.grads = (x.kind == kHead || x.kind == kLayerBwd || x.kind == kEmbedBwd);
    if (x.grads) {
      // Layers alternate between gradient buffers 0 and 1; the head (its
      // gradient is several layers' worth and takes that long to leave) and
      // the compact embedding rows use buffer 2, so no layer waits for the
      // head's gradient to be evacuated.
      const int g = x.kind == kLayerBwd ? gnext : 2;
      x.gbuf = g;
      x.prev_gbuf_user = glast[g];
      glast[g] = i;
      if (x.kind == kLayerBwd) gnext ^= 1;
    }
  }
  return v;
}

// ------------------------------------------------------------------ device arena plan
struct Plan {
  int64_t total = 0;
  int64_t add(int64_t bytes) {
    const int64_t off = total;
    total = align_up(total + std::max<int64_t>(bytes, 1), 256);
    return off;
  }
};

struct ActsSizes {
  int64_t n1, rstd, qkv, o, lse, h, n2, gu, a, x;
  int64_t moe_logits, moe_pairs_i32, moe_rows_i32, moe_off, moe_gates, moe_xp, moe_ap, moe_gup, moe_yp;  // MoE only
  int64_t total;
};

ActsSizes acts_sizes(const Dims& D) {
  ActsSizes s;
  s.x = align_up(D.T * D.d * 2, 256);
  s.n1 = s.x;
  s.rstd = align_up(D.T * 4, 256);
  s.qkv = align_up(D.T * D.Dqkv * 2, 256);
  s.o = align_up(D.T * D.Dq * 2, 256);
  s.lse = align_up((int64_t)D.B * D.Hq * D.S * 4, 256);
  s.h = s.x;
  s.n2 = s.x;
  s.gu = D.E ? 0 : align_up(D.Tc * 2L * D.f * 2, 256);  // one MLP row chunk (the whole step when unchunked)
  s.a = D.E ? 0 : align_up(D.Tc * (int64_t)D.f * 2, 256);
  const int64_t P = D.T * (int64_t)D.k;  // (token, slot) pairs of an MoE layer
  const int64_t R = D.E ? moe_rows_capacity(P, D.E, kMoeRowAlign) : 0;  // permuted rows, padding included
  s.moe_logits = align_up(D.T * (int64_t)D.E * 4, 256);
  s.moe_pairs_i32 = align_up(P * 4, 256);
  s.moe_rows_i32 = align_up(R * 4, 256);
  s.moe_off = align_up((D.E + 1) * 4L, 256);
  s.moe_gates = s.moe_pairs_i32;
  s.moe_xp = align_up(R * D.d * 2, 256);
  s.moe_ap = align_up(R * D.f * 2, 256);
  s.moe_gup = align_up(R * 2L * D.f * 2, 256);
  s.moe_yp = s.moe_xp;
  const int64_t moe = D.E ? s.moe_logits + 2 * s.moe_pairs_i32 + s.moe_rows_i32 + s.moe_off + s.moe_gates +
                                s.moe_xp + s.moe_ap + s.moe_gup + s.moe_yp
                          : 0;
  s.total = s.n1 + 2 * s.rstd + s.qkv + s.o + s.lse + s.h + s.n2 + s.gu + s.a + moe;
  return s;
}

LayerActs carve_acts(uint8_t* p, const Dims& D, bf16* x) {
  const ActsSizes s = acts_sizes(D);
  LayerActs a;
  a.x = x;
  a.n1 = reinterpret_cast<bf16*>(p);
  p += s.n1;
  a.rstd1 = reinterpret_cast<float*>(p);
  p += s.rstd;
  a.qkv = reinterpret_cast<bf16*>(p);
  p += s.qkv;
  a.o = reinterpret_cast<bf16*>(p);
  p += s.o;
  a.lse = reinterpret_cast<float*>(p);
  p += s.lse;
  a.h = reinterpret_cast<bf16*>(p);
  p += s.h;
  a.n2 = reinterpret_cast<bf16*>(p);
  p += s.n2;
  a.rstd2 = reinterpret_cast<float*>(p);
  p += s.rstd;
  a.gu = reinterpret_cast<bf16*>(p);
  p += s.gu;
  a.a = reinterpret_cast<bf16*>(p);
  p += s.a;
  if (D.E) {
    a.moe_logits = reinterpret_cast<float*>(p);
    p += s.moe_logits;
    a.moe_idx = reinterpret_cast<int32_t*>(p);
    p += s.moe_pairs_i32;
    a.moe_order = reinterpret_cast<int32_t*>(p);
    p += s.moe_rows_i32;
    a.moe_pos = reinterpret_cast<int32_t*>(p);
    p += s.moe_pairs_i32;
    a.moe_off = reinterpret_cast<int32_t*>(p);
    p += s.moe_off;
    a.moe_gates = reinterpret_cast<float*>(p);
    p += s.moe_gates;
    a.moe_xp = reinterpret_cast<bf16*>(p);
    p += s.moe_xp;
    a.moe_ap = reinterpret_cast<bf16*>(p);
    p += s.moe_ap;
    a.moe_gup = reinterpret_cast<bf16*>(p);
    p += s.moe_gup;
    a.moe_yp = reinterpret_cast<bf16*>(p);
  }
  return a;
}

long head_chunk_rows(const Dims& D) {
  // keep the FP32 logits of one chunk near 2 GiB, at most T, a multiple of 128
  long rows = (long)((2LL << 30) / ((int64_t)D.V * 4));
  rows = std::max(128L, rows / 128 * 128);
  return std::min(rows, D.T);
}

// Workspace layout (shared by the byte count and by init).
Workspace carve_ws(uint8_t* base, const Dims& D, Plan& P) {
  const long T = D.T;
  const long hc = head_chunk_rows(D);
  const int64_t td = T * D.d * 2;
  auto at = [&](int64_t bytes) { return base ? base + P.add(bytes) : (P.add(bytes), nullptr); };
  Workspace w{};
  w.dx_a = reinterpret_cast<bf16*>(at(td));
  w.dx_b = reinterpret_cast<bf16*>(at(td));
  w.dh = reinterpret_cast<bf16*>(at(td));
  w.dgu = reinterpret_cast<bf16*>(at(D.E ? 0 : D.Tc * 2L * D.f * 2));
  w.dn = reinterpret_cast<bf16*>(at(td));
  w.dout = reinterpret_cast<bf16*>(at(T * (int64_t)D.Dq * 2));
  w.dqkv = reinterpret_cast<bf16*>(at(T * (int64_t)D.Dqkv * 2));
  w.delta = reinterpret_cast<float*>(at((int64_t)D.B * D.Hq * D.S * 4));
  w.dg_partial = reinterpret_cast<float*>(at(((T + kRmsRowsPerBlock - 1) / kRmsRowsPerBlock) * (int64_t)D.d * 4));
  const bool chunked = D.Tc < T;
  w.dwd_f32 = chunked ? reinterpret_cast<float*>(at((int64_t)D.d * D.f * 4)) : nullptr;
  w.dwgu_f32 = chunked ? reinterpret_cast<float*>(at(2LL * D.f * D.d * 4)) : nullptr;
  w.nf = reinterpret_cast<bf16*>(at(td));
  w.rstd_f = reinterpret_cast<float*>(at(T * 4));
  w.z = reinterpret_cast<float*>(at(hc * (int64_t)D.V * 4));
  w.dz = reinterpret_cast<bf16*>(at(hc * (int64_t)D.V * 2));
  w.dnf = reinterpret_cast<bf16*>(at(td));
  w.dwh_f32 = reinterpret_cast<float*>(at((int64_t)D.V * D.d * 4));
  w.loss_rows = reinterpret_cast<float*>(at(T * 4));
  w.loss = reinterpret_cast<float*>(at(256));
  w.inp = reinterpret_cast<int32_t*>(at(T * 4));
  w.tgt = reinterpret_cast<int32_t*>(at(T * 4));
  w.emb_off = reinterpret_cast<int32_t*>(at(((int64_t)D.V + 1) * 4));
  w.emb_pos = reinterpret_cast<int32_t*>(at(T * 4));
  w.emb_rows = reinterpret_cast<int32_t*>(at(std::min<int64_t>(T, D.V) * 4));
  w.tokens_dev = reinterpret_cast<int32_t*>(at((int64_t)D.B * (D.S + 1) * 4));
  w.rope_cos = reinterpret_cast<float*>(at((int64_t)D.S * (D.hd / 2) * 4));
  w.rope_sin = reinterpret_cast<float*>(at((int64_t)D.S * (D.hd / 2) * 4));
  w.status = reinterpret_cast<int*>(at(256));
  w.grad_flags = reinterpret_cast<int*>(at((3LL * D.L + 8) * 4));  // more than the visits of any schedule
  w.head_chunk = hc;
  if (D.E) {
    const int64_t P = T * (int64_t)D.k, R = moe_rows_capacity(P, D.E, kMoeRowAlign);
    w.moe_dyp = reinterpret_cast<bf16*>(at(R * D.d * 2));
    w.moe_dgup = reinterpret_cast<bf16*>(at(R * 2L * D.f * 2));
    w.moe_dxp = reinterpret_cast<bf16*>(at(R * D.d * 2));
    w.moe_ds = reinterpret_cast<bf16*>(at(T * (int64_t)D.E * 2));
    w.moe_dn2r = reinterpret_cast<bf16*>(at(td));
    w.moe_dgates = reinterpret_cast<float*>(at(P * 4));
    w.moe_scratch = reinterpret_cast<int32_t*>(at(moe_sort_scratch_ints(P, D.E) * 4));
  }
  return w;
}

}  // namespace
}  // namespace mt

// ====================================================================== replica group control block
namespace mt {
constexpr int kMaxReplicas = 64;
constexpr uint64_t kGroupMagic = 0x3170756f72477453ull;

// At the start of the shared segment; the turn counters [n_chunks], the
// published Adam steps [tiles] and the loaded flags [tiles] follow it.  All
// counters are read and written with atomic builtins (lock-free, address-free
// on both host architectures), so they work across processes.
struct GroupHeader {
  uint64_t magic;
  int64_t total_bytes, n_chunks, slab_bytes, n_tiles;
  int32_t n_replicas, ready, attached, failed;
  int64_t steps_done;      // step completions of all replicas, cumulative
  int64_t nonfinite_step;  // s + 1 once group step s has seen a non-finite loss or gradient
  int64_t emb_turn;        // embedding rows of step s: replica r adds once it reads s * n + r
  int64_t barrier_count;   // mt_replica_barrier arrivals, cumulative
  float loss[2][kMaxReplicas];  // each replica's scaled loss, by step parity
};

template <class T>
inline T aload(const T* p) { return __atomic_load_n(p, __ATOMIC_ACQUIRE); }
template <class T>
inline void astore(T* p, T v) { __atomic_store_n(p, v, __ATOMIC_RELEASE); }
template <class T>
inline T aadd(T* p, T v) { return __atomic_add_fetch(p, v, __ATOMIC_ACQ_REL); }
}  // namespace mt

// ====================================================================== the handle
struct mt_model {
  mt_config cfg{};
  mt::Dims D{};
  int device = 0;
  int K = 1;
  bool resident_mode = false, store_acts = false, single_buffer = false, debug = false, time_kernels = false;
  int keep_from = 0;  // first layer whose internals stay on the device (L: none); stored[i - keep_from]
  bool trace = false;
  bool visit_log = false;
  bool tied = false;   // MT_TIE_EMBEDDINGS: the head's weight is tile 0's E
  int head_tile = 0;   // tile the head visit streams (L + 1, or 0 when tied)
  bool undrained = false;
  std::vector<mt::TileLayout> layouts;  // per tile
  std::vector<uint8_t*> tiles;
  std::vector<uint8_t> w_loaded;
  int64_t step = 0;
  std::string err;
  bool broken = false;

  // device
  uint8_t* arena = nullptr;
  size_t arena_bytes = 0;
  int64_t arena_used = 0;
  cudaStream_t s_comp = nullptr, s_h2d = nullptr, s_d2h = nullptr;
  uint8_t* wbuf[2] = {nullptr, nullptr};
  uint8_t* gbuf[3] = {nullptr, nullptr, nullptr};  // layers alternate 0/1; head and embedding rows use 2
  int64_t gbuf_bytes[3] = {0, 0, 0};
  uint8_t* resident = nullptr;
  std::vector<int64_t> resident_off;
  std::vector<mt::bf16*> ckpt, blockbuf;
  mt::bf16* xtmp[2] = {nullptr, nullptr};
  std::vector<mt::LayerActs> stored;
  mt::LayerActs acts{};
  mt::Workspace ws{};
  int64_t max_w_bytes = 0;

  // host pinned
  uint8_t* stage[2] = {nullptr, nullptr};
  int64_t stage_bytes = 0;
  std::vector<uint8_t*> slabs;
  int64_t slab_bytes = 0;
  float* pinned_scalars = nullptr;  // [0] loss, [1] status bits
  int32_t* pinned_tok = nullptr;    // inp | tgt | emb_off | emb_pos | emb_rows
  int emb_u = 0;                    // number of distinct token ids of the step (rows of the compact dE)
  // micro-batches of the current step: pass micro_index of micro_count; gradients
  // of later passes add into the tile's G, Adam runs on the last pass only
  int micro_index = 0, micro_count = 1;
  bool grads_only = false;  // mt_train_step_grads: no pass is the last (no Adam, no step advance)
  bool last_pass() const { return !grads_only && micro_index + 1 == micro_count; }

  // schedule + events
  std::vector<mt::Visit> visits;
  int n_grad_visits = 0;
  int last_grad_visit = -1;
  std::vector<cudaEvent_t> ev_ready, ev_free, ev_grads, ev_d2h;
  std::vector<cudaEvent_t> ev_wait_a, ev_wait_b, ev_h2d_a, ev_h2d_b, ev_d2h_a, ev_d2h_b;
  std::vector<cudaEvent_t> ev_vis_a, ev_vis_b;  // first / last kernel of each visit on the compute stream
  cudaEvent_t ev_stage[2] = {nullptr, nullptr};
  std::vector<cudaEvent_t> ev_slab;
  cudaEvent_t ev_t0 = nullptr, ev_t1 = nullptr;
  // MT_TIME_KERNELS timeline: an event pair around every H2D and D2H chunk copy
  std::vector<cudaEvent_t> tl_h2d, tl_d2h;
  std::vector<int> tl_h2d_visit, tl_d2h_visit;
  int tl_h2d_n = 0;
  std::atomic<int> tl_d2h_n{0};

  // host handshakes
  std::mutex mu;
  std::condition_variable cv;
  std::vector<char> rec_ready, rec_free, rec_d2h, rec_h2d_timed, rec_d2h_timed, rec_wait_timed;
  std::vector<double> host_wait_ready_ms, host_wait_gbuf_ms;  // compute thread's waits per visit (MT_VISIT_LOG)
  std::atomic<bool> abort_flag{false};
  std::atomic<bool> nonfinite{false};
  std::atomic<int> worker_code{0};
  std::string worker_msg;
  // host-side fault injection (mt_debug_inject): fires once, in the next step
  std::atomic<int> inject_what{MT_INJECT_NONE};
  std::atomic<int> inject_visit{0};

  // threads
  std::unique_ptr<mt::Pool> adam_pool, pack_pool, acc_pool;
  std::thread loader, d2h, accum;
  bool stop_threads = false;
  int64_t step_gen = 0;
  std::deque<int> d2h_q;
  struct AccJob {
    int slab, visit, tile;
    int64_t off, bytes;
    bool last;
    bool rows;  // compact embedding gradient: the slab holds whole rows of emb_rows, from row off / (2 d)
    bool direct;  // MT_DIRECT_GRADS: the chunk was copied straight into the tile's G (slab memory unused)
  };
  std::deque<AccJob> acc_q;
  std::vector<int> free_slabs;
  int acc_tiles_done = 0;
  std::atomic<int64_t> adam_us{0};
  // Adam tasks not yet finished, per tile (MT_ASYNC_ADAM: a step may return
  // with some pending; a tile's are waited for before it is uploaded or read)
  bool async_adam = false;
  // MT_DIRECT_GRADS: the tiles' G sections are page-locked and gradient
  // chunks land in them directly; a device check flags non-finite values of
  // each gradient visit (grad_flags, copied to pinned_flags before the chunks)
  bool direct_grads = false;
  // a model's own host tiles: one anonymous mapping (nullptr in a replica group)
  uint8_t* tile_map = nullptr;
  size_t tile_map_bytes = 0;
  // page-locked range of each tile (MT_DIRECT_GRADS: its G section; MT_DIRECT_WEIGHTS: its W
  // section; both: W and G as one range), nullptr where nothing is registered
  std::vector<uint8_t*> host_reg;
  bool direct_weights = false;
  int* grad_flags = nullptr;     // device [visits]
  int* pinned_flags = nullptr;   // host, pinned [visits]
  std::mutex adam_mu;
  std::condition_variable adam_cv;
  std::vector<int> adam_pending;
  std::chrono::steady_clock::time_point last_grads_landed;

  // replica group (n_replicas >= 2); micro_index / micro_count are rank / n
  struct Group {
    int rank = 0, n = 0;
    uint8_t* base = nullptr;  // the mapped segment
    size_t bytes = 0;
    mt::GroupHeader* h = nullptr;
    int64_t* turn = nullptr;       // per gradient chunk
    int64_t* adam_done = nullptr;  // per tile: s + 1 once step s's update of the tile has finished
    int32_t* loaded = nullptr;     // per tile: W loaded by some replica
    std::vector<int64_t> chunk_base;  // first chunk index of each tile
    int64_t s = 0;                    // group steps run (the current step while one runs)
    int64_t barriers = 0;             // mt_replica_barrier calls of this replica
    std::vector<int64_t> final_val;   // last replica: value to publish once the tile's Adam tasks finish
  } grp;
  bool group() const { return grp.n >= 2; }

  // stats
  mt_step_stats stats{};
  mt::LaunchStats ls;
  std::vector<cudaEvent_t> gemm_events;
  std::vector<double> gemm_event_flops;
};

namespace mt {
namespace {

thread_local std::string g_init_error;

#define MT_CK(call)                                                                                    \
  do {                                                                                                 \
    cudaError_t e__ = (call);                                                                          \
    if (e__ != cudaSuccess) throw MtError{MT_ECUDA, std::string(#call) + ": " + cudaGetErrorString(e__)}; \
  } while (0)

void worker_fail(mt_model* m, const MtError& e) {
  {
    std::lock_guard<std::mutex> g(m->mu);
    if (m->worker_code == 0) {
      m->worker_code = e.code;
      m->worker_msg = e.msg;
    }
    m->abort_flag = true;
  }
  if (m->group()) astore(&m->grp.h->failed, 1);  // the other replicas' waits fail too
  m->cv.notify_all();
}

// True once for the armed injection `what` at the first visit >= its visit.
bool inject_now(mt_model* m, int what, int visit) {
  if (m->inject_what.load() != what || visit < m->inject_visit.load()) return false;
  int expected = what;
  return m->inject_what.compare_exchange_strong(expected, MT_INJECT_NONE);
}

MtError injected(const char* where, int visit) {
  return MtError{MT_EINTERNAL, std::string("injected ") + where + " failure at visit " + std::to_string(visit)};
}

void check_abort(mt_model* m) {
  if (m->abort_flag) {
    std::lock_guard<std::mutex> g(m->mu);
    throw MtError{m->worker_code ? m->worker_code.load() : MT_EINTERNAL, "step aborted: " + m->worker_msg};
  }
}

void wait_event(mt_model* m, cudaEvent_t e, const char* what) {
  const auto t0 = Clock::now();
  while (true) {
    const cudaError_t r = cudaEventQuery(e);
    if (r == cudaSuccess) return;
    if (r != cudaErrorNotReady) throw MtError{MT_ECUDA, std::string(what) + ": " + cudaGetErrorString(r)};
    check_abort(m);
    if (ms_since(t0) > (double)m->cfg.timeout_ms) throw MtError{MT_ETIMEDOUT, std::string("timed out waiting for ") + what};
    std::this_thread::sleep_for(std::chrono::microseconds(20));
  }
}

// Wait (bounded) for everything enqueued on a stream so far; false on timeout or error.
bool drain_stream(cudaStream_t st, int64_t timeout_ms) {
  cudaEvent_t e;
  if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return false;
  bool ok = cudaEventRecord(e, st) == cudaSuccess;
  const auto t0 = Clock::now();
  while (ok) {
    const cudaError_t r = cudaEventQuery(e);
    if (r == cudaSuccess) break;
    if (r != cudaErrorNotReady || ms_since(t0) > (double)timeout_ms) ok = false;
    else std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
  cudaEventDestroy(e);
  return ok;
}

void wait_flag(mt_model* m, std::vector<char>& vec, int i, const char* what) {
  std::unique_lock<std::mutex> g(m->mu);
  const bool ok = m->cv.wait_for(g, std::chrono::milliseconds(m->cfg.timeout_ms),
                                 [&] { return vec[i] != 0 || m->abort_flag.load(); });
  if (m->abort_flag)
    throw MtError{m->worker_code ? m->worker_code.load() : MT_EINTERNAL,
                  std::string("aborted while waiting for ") + what + ": " + m->worker_msg};
  if (!ok) throw MtError{MT_ETIMEDOUT, std::string("timed out waiting for ") + what};
}

void set_flag(mt_model* m, std::vector<char>& vec, int i) {
  {
    std::lock_guard<std::mutex> g(m->mu);
    vec[i] = 1;
  }
  m->cv.notify_all();
}

// ------------------------------------------------------------------ replica group waits and turns
// Bounded poll of a condition in the shared control block; fails at once when
// another replica has failed or this replica's step was aborted.
template <class F>
void group_wait(mt_model* m, F ready, const char* what) {
  const auto t0 = Clock::now();
  for (int spin = 0; !ready(); ++spin) {
    if (aload(&m->grp.h->failed))
      throw MtError{MT_EINTERNAL, std::string("another replica of the group failed (waiting for ") + what + ")"};
    check_abort(m);
    if (ms_since(t0) > (double)m->cfg.timeout_ms)
      throw MtError{MT_ETIMEDOUT, std::string("timed out waiting for ") + what};
    if (spin < 64) std::this_thread::yield();
    else std::this_thread::sleep_for(std::chrono::microseconds(20));
  }
}

void group_set_nonfinite(mt_model* m) {
  m->nonfinite = true;
  if (m->group()) astore(&m->grp.h->nonfinite_step, m->grp.s + 1);
}

// Whether this step has seen a non-finite value on this replica or, in a
// group, on any replica whose contribution this one has waited for.
bool step_nonfinite(mt_model* m) {
  return m->nonfinite || (m->group() && aload(&m->grp.h->nonfinite_step) == m->grp.s + 1);
}

int64_t* group_chunk_turn(mt_model* m, int tile, int64_t off) {
  return m->grp.turn + m->grp.chunk_base[tile] + off / m->slab_bytes;
}

// Replica r may write a gradient chunk of step s once the chunk's counter reads
// s * n + r (replicas 0 .. r-1 have added theirs); it then sets s * n + r + 1.
void group_take_turn(mt_model* m, int64_t* slot) {
  const int64_t want = m->grp.s * m->grp.n + m->grp.rank;
  group_wait(m, [&] { return aload(slot) >= want; }, "the previous replica's gradient chunk");
  if (aload(slot) != want) throw MtError{MT_EINTERNAL, "replica group: a gradient turn counter is ahead of this step"};
}

void group_pass_turn(mt_model* m, int64_t* slot) {
  astore(slot, m->grp.s * m->grp.n + m->grp.rank + 1);
}

// Last replica: every Adam task of `tile` for this step has been submitted;
// publish the tile's update once they have finished.
void group_tile_final(mt_model* m, int tile) {
  std::lock_guard<std::mutex> g(m->adam_mu);
  if (m->adam_pending[tile] == 0) astore(&m->grp.adam_done[tile], m->grp.s + 1);
  else m->grp.final_val[tile] = m->grp.s + 1;
}

// Wait until the last replica has published the update of `tile` (-1: every
// tile) for the steps before group step v.
void group_wait_adam(mt_model* m, int tile, int64_t v) {
  const int lo = tile < 0 ? 0 : tile, hi = tile < 0 ? (int)m->tiles.size() : tile + 1;
  for (int t = lo; t < hi; ++t)
    group_wait(m, [&] { return aload(&m->grp.adam_done[t]) >= v; }, "the Adam update of a tile (last replica)");
}

// Multi-threaded pageable -> pinned copy (the JIT packer).
void pack_copy(mt_model* m, uint8_t* dst, const uint8_t* src, int64_t n) {
  const int nt = m->pack_pool->size();
  const int64_t piece = align_up((n + nt - 1) / nt, 4096);
  if (nt <= 1 || n < (8 << 20)) {
    std::memcpy(dst, src, (size_t)n);
    return;
  }
  for (int64_t off = 0; off < n; off += piece) {
    const int64_t c = std::min(piece, n - off);
    m->pack_pool->submit([=] { std::memcpy(dst + off, src + off, (size_t)c); });
  }
  if (!m->pack_pool->wait_idle(m->cfg.timeout_ms)) throw MtError{MT_ETIMEDOUT, "packer copy timed out"};
}

// Every Adam task goes through here: counted per tile, queued with the tile
// index as its priority (the next step uploads tiles in index order, so the
// tile needed first is updated first).
void submit_adam_task(mt_model* m, int tile, std::function<void()> fn) {
  {
    std::lock_guard<std::mutex> g(m->adam_mu);
    ++m->adam_pending[tile];
  }
  m->adam_pool->submit(
      [m, tile, fn = std::move(fn)] {
        NvtxRange range("adam (tile %d)", tile);
        fn();
        std::lock_guard<std::mutex> g(m->adam_mu);
        if (--m->adam_pending[tile] == 0) {
          m->adam_cv.notify_all();
          if (m->group() && m->grp.final_val[tile]) {
            astore(&m->grp.adam_done[tile], m->grp.final_val[tile]);
            m->grp.final_val[tile] = 0;
          }
        }
      },
      tile);
}

// Bounded wait until tile `tile` has no Adam task pending (all tiles: -1).
void wait_adam(mt_model* m, int tile) {
  std::unique_lock<std::mutex> g(m->adam_mu);
  auto idle = [&] {
    if (tile >= 0) return m->adam_pending[tile] == 0;
    for (int c : m->adam_pending)
      if (c) return false;
    return true;
  };
  if (!m->adam_cv.wait_for(g, std::chrono::milliseconds(m->cfg.timeout_ms), idle))
    throw MtError{MT_ETIMEDOUT, "timed out waiting for the Adam update of tile " + std::to_string(tile)};
}

// Entry points that read or overwrite tiles wait for their pending Adam
// tasks (tile, or -1 for all).  A failure of a task that ran after its step
// returned is reported by the next waiting call that can fail.
int settle_adam(mt_model* m, int tile, bool report_failure) {
  if (!m->async_adam && !m->group()) return MT_OK;
  try {
    if (m->group()) group_wait_adam(m, tile, m->grp.s);
    else wait_adam(m, tile);
  } catch (const MtError& e) {
    m->err = e.msg;
    m->broken = true;
    return e.code;
  }
  if (report_failure && m->abort_flag && m->worker_code) {
    m->err = "an Adam update that ran after its step returned failed: " + m->worker_msg;
    m->broken = true;
    return m->worker_code;
  }
  return MT_OK;
}

// ------------------------------------------------------------------ loader (H2D stream)
void loader_main(mt_model* m) {
  cudaSetDevice(m->device);
  int64_t gen = 0;
  while (true) {
    int64_t gs = 0;  // group step of this step
    {
      std::unique_lock<std::mutex> g(m->mu);
      m->cv.wait(g, [&] { return m->stop_threads || m->step_gen > gen; });
      if (m->stop_threads) return;
      gen = m->step_gen;
      gs = m->grp.s;
    }
    try {
      int si = 0;
      for (int v = 0; v < (int)m->visits.size(); ++v) {
        const Visit& x = m->visits[v];
        if (!x.h2d) continue;
        if (inject_now(m, MT_INJECT_LOADER_FAIL, v)) throw injected("loader", v);
        if (inject_now(m, MT_INJECT_LOADER_STALL, v)) {
          // stop without an error: the compute thread's Weights-Ready wait runs
          // out; leave once the step has aborted (bounded in any case)
          std::unique_lock<std::mutex> g(m->mu);
          m->cv.wait_for(g, std::chrono::milliseconds(4 * m->cfg.timeout_ms),
                         [&] { return m->abort_flag.load() || m->stop_threads; });
          break;
        }
        NvtxRange range("h2d visit %d (tile %d)", v, x.tile);
        if (x.prev_user >= 0) {
          wait_flag(m, m->rec_free, x.prev_user, "buffer free");
          MT_CK(cudaStreamWaitEvent(m->s_h2d, m->ev_free[x.prev_user], 0));
        }
        if (m->group()) group_wait_adam(m, x.tile, gs);  // the previous step's update, on the last replica
        else if (m->async_adam) wait_adam(m, x.tile);  // the previous step's update of this tile
        MT_CK(cudaEventRecord(m->ev_h2d_a[v], m->s_h2d));
        const TileLayout& lay = m->layouts[x.tile];
        const uint8_t* src = m->tiles[x.tile] + lay.off_w;
        uint8_t* dst = m->wbuf[x.buf];
        const int64_t n = lay.w_bytes;
        // Staged: a packer copy into one of the two pinned staging chunks, then its
        // DMA.  Direct (MT_DIRECT_WEIGHTS): the DMA reads the page-locked W section
        // itself, chunk by chunk, so nothing on the host touches the bytes.
        for (int64_t off = 0; off < n; off += m->stage_bytes) {
          const int64_t c = std::min(m->stage_bytes, n - off);
          const uint8_t* from = src + off;
          const int k = si & 1;
          if (!m->direct_weights) {
            ++si;
            wait_event(m, m->ev_stage[k], "pinned staging buffer");
            pack_copy(m, m->stage[k], src + off, c);
            from = m->stage[k];
          }
          const int tl = m->time_kernels && 2 * m->tl_h2d_n + 1 < (int)m->tl_h2d.size() ? m->tl_h2d_n++ : -1;
          if (tl >= 0) {
            m->tl_h2d_visit[tl] = v;
            MT_CK(cudaEventRecord(m->tl_h2d[2 * tl], m->s_h2d));
          }
          MT_CK(cudaMemcpyAsync(dst + off, from, (size_t)c, cudaMemcpyHostToDevice, m->s_h2d));
          if (tl >= 0) MT_CK(cudaEventRecord(m->tl_h2d[2 * tl + 1], m->s_h2d));
          if (!m->direct_weights) MT_CK(cudaEventRecord(m->ev_stage[k], m->s_h2d));
        }
        MT_CK(cudaEventRecord(m->ev_h2d_b[v], m->s_h2d));
        MT_CK(cudaEventRecord(m->ev_ready[v], m->s_h2d));
        if (m->trace) std::fprintf(stderr, "[mt trace] loader: tile %d for visit %d enqueued\n", x.tile, v);
        m->rec_h2d_timed[v] = 1;
        set_flag(m, m->rec_ready, v);
      }
    } catch (const MtError& e) {
      worker_fail(m, e);
    }
  }
}

// ------------------------------------------------------------------ D2H stream + slabs
int acquire_slab(mt_model* m) {
  std::unique_lock<std::mutex> g(m->mu);
  const bool ok = m->cv.wait_for(g, std::chrono::milliseconds(m->cfg.timeout_ms),
                                 [&] { return !m->free_slabs.empty() || m->abort_flag.load(); });
  if (m->abort_flag) throw MtError{MT_EINTERNAL, "aborted"};
  if (!ok) throw MtError{MT_ETIMEDOUT, "timed out waiting for a free gradient slab"};
  const int s = m->free_slabs.back();
  m->free_slabs.pop_back();
  return s;
}

void d2h_main(mt_model* m) {
  cudaSetDevice(m->device);
  while (true) {
    int v;
    {
      std::unique_lock<std::mutex> g(m->mu);
      m->cv.wait(g, [&] { return m->stop_threads || !m->d2h_q.empty(); });
      if (m->stop_threads) return;
      v = m->d2h_q.front();
      m->d2h_q.pop_front();
    }
    try {
      check_abort(m);
      if (inject_now(m, MT_INJECT_D2H_FAIL, v)) throw injected("D2H", v);
      const Visit& x = m->visits[v];
      const TileLayout& lay = m->layouts[x.tile];
      NvtxRange range("d2h visit %d (tile %d)", v, x.tile);
      MT_CK(cudaStreamWaitEvent(m->s_d2h, m->ev_grads[v], 0));
      MT_CK(cudaEventRecord(m->ev_d2h_a[v], m->s_d2h));
      const uint8_t* src = m->gbuf[x.gbuf];
      // the embedding gradient leaves compact (rows of the step's token ids), in whole rows per slab
      const bool rows = x.kind == kEmbedBwd;
      const int64_t row_b = 2LL * m->D.d;
      const int64_t n = rows ? (int64_t)m->emb_u * row_b : lay.w_bytes;
      const int64_t chunk = rows ? m->slab_bytes / row_b * row_b : m->slab_bytes;
      // Direct landing (first pass of a step): the chunks go into the tile's
      // page-locked G and the slab is only a token bounding the chunks in
      // flight; the visit's device non-finite flag travels first.
      const bool direct = m->direct_grads && !rows && m->micro_index == 0;
      uint8_t* gdst = m->tiles[x.tile] + lay.off_g;
      if (direct)
        MT_CK(cudaMemcpyAsync(m->pinned_flags + v, m->grad_flags + v, sizeof(int), cudaMemcpyDeviceToHost, m->s_d2h));
      for (int64_t off = 0; off < n; off += chunk) {
        const int64_t c = std::min(chunk, n - off);
        const int s = acquire_slab(m);
        int tl = -1;
        if (m->time_kernels) {
          tl = m->tl_d2h_n++;
          if (2 * tl + 1 >= (int)m->tl_d2h.size()) tl = -1;
        }
        if (tl >= 0) {
          m->tl_d2h_visit[tl] = v;
          MT_CK(cudaEventRecord(m->tl_d2h[2 * tl], m->s_d2h));
        }
        MT_CK(cudaMemcpyAsync(direct ? gdst + off : m->slabs[s], src + off, (size_t)c, cudaMemcpyDeviceToHost,
                              m->s_d2h));
        if (tl >= 0) MT_CK(cudaEventRecord(m->tl_d2h[2 * tl + 1], m->s_d2h));
        MT_CK(cudaEventRecord(m->ev_slab[s], m->s_d2h));
        {
          std::lock_guard<std::mutex> g(m->mu);
          m->acc_q.push_back({s, v, x.tile, off, c, off + c >= n, rows, direct});
        }
        m->cv.notify_all();
      }
      MT_CK(cudaEventRecord(m->ev_d2h_b[v], m->s_d2h));
      MT_CK(cudaEventRecord(m->ev_d2h[v], m->s_d2h));
      m->rec_d2h_timed[v] = 1;
      set_flag(m, m->rec_d2h, v);
    } catch (const MtError& e) {
      worker_fail(m, e);
    }
  }
}

// Adam on the elements of tile `tile` whose BF16 gradients occupy bytes
// [g_off, g_off + g_bytes) of its G section (one landed gradient slab): the
// update is elementwise, so each slab is updated as soon as it lands.
void submit_adam_range(mt_model* m, int tile, int64_t g_off, int64_t g_bytes) {
  const TileLayout& lay = m->layouts[tile];
  uint8_t* base = m->tiles[tile];
  const AdamHyper h{m->cfg.lr, m->cfg.beta1, m->cfg.beta2, m->cfg.adam_eps, m->cfg.weight_decay, m->step + 1};
  const int64_t lo_b = g_off, hi_b = g_off + g_bytes;
  for (const auto& t : lay.tensors) {
    // element range of this tensor inside [lo_b, hi_b)
    const int64_t e0 = std::max<int64_t>(0, (lo_b - t.offset + 1) / 2);
    const int64_t e1 = std::min<int64_t>(t.numel, (hi_b - t.offset) / 2);
    if (e1 <= e0) continue;
    const int64_t n = e1 - e0;
    const int64_t piece = std::max<int64_t>(1 << 18, (n + m->adam_pool->size() - 1) / m->adam_pool->size());
    for (int64_t b = e0; b < e1; b += piece) {
      const int64_t c = std::min(piece, e1 - b);
      uint16_t* w = reinterpret_cast<uint16_t*>(base + lay.off_w + t.offset) + b;
      const uint16_t* g = reinterpret_cast<const uint16_t*>(base + lay.off_g + t.offset) + b;
      float* mm = reinterpret_cast<float*>(base + lay.off_m + 2 * t.offset) + b;
      float* vv = reinterpret_cast<float*>(base + lay.off_v + 2 * t.offset) + b;
      submit_adam_task(m, tile, [=] {
        const auto t0 = Clock::now();
        adam_range(w, g, mm, vv, (size_t)c, h);
        m->adam_us += (int64_t)(ms_since(t0) * 1000.0);
      });
    }
  }
}

// Embedding rows whose gradient is zero this step (token ids that do not occur):
// zero their G rows and, when the loss is finite, run Adam on them (g = 0).
// Submitted once the loss is known (the head's gradient lands).  The embedding
// W was streamed for the forward before the head ran and the backward does
// not read it, so these rows may be updated mid-step.
void submit_untouched_embed(mt_model* m) {
  if (m->micro_index > 0) return;  // later micro-batches add into the rows the first one set
  // with micro-batches one dense embedding update at the end; none for gradients only
  const bool update = m->micro_count == 1 && !m->grads_only;
  const TileLayout& lay = m->layouts[0];
  const TensorSlot& E = lay.slot("E");
  const int d = m->D.d, V = m->D.V;
  uint8_t* base = m->tiles[0];
  const int32_t* off = m->pinned_tok + 2 * m->D.T;  // emb_off [V + 1]
  const AdamHyper h{m->cfg.lr, m->cfg.beta1, m->cfg.beta2, m->cfg.adam_eps, m->cfg.weight_decay, m->step + 1};
  constexpr int kRowsPerTask = 64;
  for (int v0 = 0; v0 < V; v0 += kRowsPerTask) {
    const int v1 = std::min(V, v0 + kRowsPerTask);
    submit_adam_task(m, 0, [=] {
      const auto t0 = Clock::now();
      for (int v = v0; v < v1; ++v) {
        if (off[v + 1] > off[v]) continue;
        const int64_t e = (int64_t)v * d;
        uint16_t* g = reinterpret_cast<uint16_t*>(base + lay.off_g + E.offset) + e;
        std::memset(g, 0, sizeof(uint16_t) * d);
        if (!update || m->nonfinite) continue;
        adam_range(reinterpret_cast<uint16_t*>(base + lay.off_w + E.offset) + e, g,
                   reinterpret_cast<float*>(base + lay.off_m + 2 * E.offset) + e,
                   reinterpret_cast<float*>(base + lay.off_v + 2 * E.offset) + e, (size_t)d, h);
      }
      m->adam_us += (int64_t)(ms_since(t0) * 1000.0);
    });
  }
}

// Tied embeddings, once the head's gradient has landed in tile 0's G: Adam on
// gf and on E's rows that no token of the step uses (their gradient is the
// head's alone and is complete).  The other rows wait for their embedding
// gradient (submit_adam_embed_rows).
void submit_tied_head_adam(mt_model* m) {
  const TileLayout& lay = m->layouts[0];
  const TensorSlot& E = lay.slot("E");
  const TensorSlot& gf = lay.slot("gf");
  submit_adam_range(m, 0, gf.offset, 2 * gf.numel);
  const int d = m->D.d, V = m->D.V;
  uint8_t* base = m->tiles[0];
  const int32_t* off = m->pinned_tok + 2 * m->D.T;  // emb_off [V + 1]
  const AdamHyper h{m->cfg.lr, m->cfg.beta1, m->cfg.beta2, m->cfg.adam_eps, m->cfg.weight_decay, m->step + 1};
  constexpr int kRowsPerTask = 64;
  for (int v0 = 0; v0 < V; v0 += kRowsPerTask) {
    const int v1 = std::min(V, v0 + kRowsPerTask);
    submit_adam_task(m, 0, [=] {
      const auto t0 = Clock::now();
      for (int v = v0; v < v1; ++v) {
        if (off[v + 1] > off[v]) continue;
        const int64_t e = (int64_t)v * d;
        adam_range(reinterpret_cast<uint16_t*>(base + lay.off_w + E.offset) + e,
                   reinterpret_cast<const uint16_t*>(base + lay.off_g + E.offset) + e,
                   reinterpret_cast<float*>(base + lay.off_m + 2 * E.offset) + e,
                   reinterpret_cast<float*>(base + lay.off_v + 2 * E.offset) + e, (size_t)d, h);
      }
      m->adam_us += (int64_t)(ms_since(t0) * 1000.0);
    });
  }
}

// One slab of the compact embedding gradient: rows u0 .. u0 + nrows of the
// step's token ids.  Scatter each row into the tile's G section and check it
// is finite (accumulator pool); the rows' Adam then goes to the Adam pool.
void accumulate_embed_rows(mt_model* m, const mt_model::AccJob& j, std::atomic<bool>& fin, bool add) {
  const TileLayout& lay = m->layouts[j.tile];
  const TensorSlot& E = lay.slot("E");
  const int d = m->D.d;
  const int64_t row_b = 2LL * d;
  const int64_t u0 = j.off / row_b, nrows = j.bytes / row_b;
  const int32_t* rows = m->pinned_tok + 3 * m->D.T + m->D.V + 1;  // emb_rows
  uint8_t* base = m->tiles[j.tile];
  const uint16_t* src = reinterpret_cast<const uint16_t*>(m->slabs[j.slab]);
  const int nt = m->acc_pool->size();
  const int64_t per = std::max<int64_t>(16, (nrows + nt - 1) / nt);
  for (int64_t a = 0; a < nrows; a += per) {
    const int64_t b = std::min(nrows, a + per);
    m->acc_pool->submit([=, &fin] {
      for (int64_t k = a; k < b; ++k) {
        uint16_t* g = reinterpret_cast<uint16_t*>(base + lay.off_g + E.offset) + (int64_t)rows[u0 + k] * d;
        const bool okr = add ? add_grad_check_finite(g, src + k * d, (size_t)d)
                             : copy_grad_check_finite(g, src + k * d, (size_t)d);
        if (!okr) fin = false;
      }
    });
  }
}

// Adam on the embedding rows rows[u0 .. u0 + nrows) whose gradients just landed.
void submit_adam_embed_rows(mt_model* m, int tile, int64_t u0, int64_t nrows) {
  const TileLayout& lay = m->layouts[tile];
  const TensorSlot& E = lay.slot("E");
  const int d = m->D.d;
  const int32_t* rows = m->pinned_tok + 3 * m->D.T + m->D.V + 1;
  uint8_t* base = m->tiles[tile];
  const AdamHyper h{m->cfg.lr, m->cfg.beta1, m->cfg.beta2, m->cfg.adam_eps, m->cfg.weight_decay, m->step + 1};
  const int64_t per = std::max<int64_t>(8, (1 << 18) / d);
  for (int64_t a = 0; a < nrows; a += per) {
    const int64_t b = std::min(nrows, a + per);
    submit_adam_task(m, tile, [=] {
      const auto t0 = Clock::now();
      for (int64_t k = a; k < b; ++k) {
        const int64_t e = (int64_t)rows[u0 + k] * d;
        adam_range(reinterpret_cast<uint16_t*>(base + lay.off_w + E.offset) + e,
                   reinterpret_cast<const uint16_t*>(base + lay.off_g + E.offset) + e,
                   reinterpret_cast<float*>(base + lay.off_m + 2 * E.offset) + e,
                   reinterpret_cast<float*>(base + lay.off_v + 2 * E.offset) + e, (size_t)d, h);
      }
      m->adam_us += (int64_t)(ms_since(t0) * 1000.0);
    });
  }
}

void accum_main(mt_model* m) {
  cudaSetDevice(m->device);
  while (true) {
    mt_model::AccJob j;
    {
      std::unique_lock<std::mutex> g(m->mu);
      m->cv.wait(g, [&] { return m->stop_threads || !m->acc_q.empty(); });
      if (m->stop_threads) return;
      j = m->acc_q.front();
      m->acc_q.pop_front();
    }
    try {
      NvtxRange range("accumulate visit %d (tile %d)", j.visit, j.tile);
      wait_event(m, m->ev_slab[j.slab], "gradient slab copy");
      if (inject_now(m, MT_INJECT_ACCUM_FAIL, j.visit)) throw injected("accumulator", j.visit);
      const bool head = m->visits[j.visit].kind == kHead;
      if (head && j.off == 0) {
        if (!std::isfinite(m->pinned_scalars[0])) group_set_nonfinite(m);
        if (!m->tied) submit_untouched_embed(m);
      }
      if (j.rows) {
        // replica group: the rows of replica r add once replicas 0 .. r-1 have added all of theirs
        if (m->group()) group_take_turn(m, &m->grp.h->emb_turn);
        std::atomic<bool> fin{true};
        accumulate_embed_rows(m, j, fin, m->tied || m->micro_index > 0);
        if (!m->acc_pool->wait_idle(m->cfg.timeout_ms)) throw MtError{MT_ETIMEDOUT, "gradient accumulation timed out"};
        if (!fin) group_set_nonfinite(m);
        if (m->group() && j.last) {
          if (m->grp.rank == 0) wait_adam(m, 0);  // the zeroed rows that no token of this replica uses
          group_pass_turn(m, &m->grp.h->emb_turn);
        }
        if (!step_nonfinite(m) && m->last_pass()) {
          if (m->micro_count == 1) {
            submit_adam_embed_rows(m, j.tile, j.off / (2LL * m->D.d), j.bytes / (2LL * m->D.d));
          } else if (j.last) {  // every row may have been touched by some micro-batch: one dense update
            if (m->tied) {  // E and gf: the whole tile
              submit_adam_range(m, j.tile, 0, m->layouts[j.tile].w_bytes);
            } else {
              const TensorSlot& E = m->layouts[j.tile].slot("E");
              submit_adam_range(m, j.tile, E.offset, 2 * E.numel);
            }
          }
        }
        if (m->group() && j.last && m->last_pass()) group_tile_final(m, j.tile);
        {
          std::lock_guard<std::mutex> g(m->mu);
          m->free_slabs.push_back(j.slab);
          if (j.last) {
            m->acc_tiles_done += 1;
            m->last_grads_landed = Clock::now();
          }
        }
        m->cv.notify_all();
        continue;
      }
      const TileLayout& lay = m->layouts[j.tile];
      int64_t* turn = m->group() ? group_chunk_turn(m, j.tile, j.off) : nullptr;
      if (turn) group_take_turn(m, turn);
      if (j.direct) {
        // already in the tile; the device flag (copied before the chunks) says whether it is finite
        if (m->pinned_flags[j.visit]) group_set_nonfinite(m);
      } else {
        uint16_t* dst = reinterpret_cast<uint16_t*>(m->tiles[j.tile] + lay.off_g + j.off);
        const uint16_t* src = reinterpret_cast<const uint16_t*>(m->slabs[j.slab]);
        // the copy (and NaN/Inf scan) of one slab is split over the accumulator pool
        const int64_t n = j.bytes / 2;
        const int nt = m->acc_pool->size();
        const bool add = m->micro_index > 0;
        const int64_t piece = std::max<int64_t>(1 << 18, align_up((n + nt - 1) / nt, 2048));
        std::atomic<bool> fin{true};
        for (int64_t b = 0; b < n; b += piece) {
          const int64_t c = std::min(piece, n - b);
          m->acc_pool->submit([=, &fin] {
            const bool okc = add ? add_grad_check_finite(dst + b, src + b, (size_t)c)
                                 : copy_grad_check_finite(dst + b, src + b, (size_t)c);
            if (!okc) fin = false;
          });
        }
        if (!m->acc_pool->wait_idle(m->cfg.timeout_ms)) throw MtError{MT_ETIMEDOUT, "gradient accumulation timed out"};
        if (!fin) group_set_nonfinite(m);
      }
      if (turn) group_pass_turn(m, turn);
      {
        std::lock_guard<std::mutex> g(m->mu);
        m->free_slabs.push_back(j.slab);
      }
      m->cv.notify_all();
      if (!step_nonfinite(m) && m->last_pass()) {
        if (inject_now(m, MT_INJECT_ADAM_FAIL, j.visit)) {
          const int v = j.visit;
          submit_adam_task(m, j.tile, [m, v] { worker_fail(m, injected("Adam", v)); });
        } else if (!(head && m->tied)) {
          submit_adam_range(m, j.tile, j.off, j.bytes);
        } else if (j.last && m->micro_count == 1) {
          // tied: E's rows wait for their embedding gradient unless no token
          // of the step uses them; gf is complete with the head's gradient
          submit_tied_head_adam(m);
        }
      }
      if (m->group() && j.last && m->last_pass()) group_tile_final(m, j.tile);
      if (j.last) {
        {
          std::lock_guard<std::mutex> g(m->mu);
          m->acc_tiles_done += 1;
          m->last_grads_landed = Clock::now();
        }
        m->cv.notify_all();
      }
    } catch (const MtError& e) {
      worker_fail(m, e);
    }
  }
}

// ------------------------------------------------------------------ host token preprocessing
// tokens [B, S+1] -> inp [T], tgt [T], and the positions of every token id in
// ascending order (counting sort) for the deterministic embedding scatter.
void prepare_tokens(mt_model* m, const int32_t* tokens) {
  const Dims& D = m->D;
  const long T = D.T;
  int32_t* inp = m->pinned_tok;
  int32_t* tgt = inp + T;
  int32_t* off = tgt + T;
  int32_t* pos = off + D.V + 1;
  for (int b = 0; b < D.B; ++b)
    for (int s = 0; s < D.S; ++s) {
      inp[(long)b * D.S + s] = tokens[(long)b * (D.S + 1) + s];
      tgt[(long)b * D.S + s] = tokens[(long)b * (D.S + 1) + s + 1];
    }
  for (long t = 0; t < T; ++t)
    if (inp[t] < 0 || inp[t] >= D.V || tgt[t] < 0 || tgt[t] >= D.V)
      throw MtError{MT_EINVAL, "token id out of range [0, vocab)"};
  std::memset(off, 0, sizeof(int32_t) * (D.V + 1));
  for (long t = 0; t < T; ++t) off[inp[t] + 1] += 1;
  for (int v = 0; v < D.V; ++v) off[v + 1] += off[v];
  std::vector<int32_t> cur(off, off + D.V);
  for (long t = 0; t < T; ++t) pos[cur[inp[t]]++] = (int32_t)t;
  // token ids that occur in the step: the only rows of dE that can be nonzero
  int32_t* rows = pos + T;
  int u = 0;
  for (int v = 0; v < D.V; ++v)
    if (off[v + 1] > off[v]) rows[u++] = v;
  m->emb_u = u;
  const size_t bytes = sizeof(int32_t) * (size_t)(2 * T + D.V + 1 + T);
  // ws.inp, tgt, emb_off, emb_pos are not contiguous in the arena: copy each.
  MT_CK(cudaMemcpyAsync(m->ws.inp, inp, sizeof(int32_t) * T, cudaMemcpyHostToDevice, m->s_comp));
  MT_CK(cudaMemcpyAsync(m->ws.tgt, tgt, sizeof(int32_t) * T, cudaMemcpyHostToDevice, m->s_comp));
  MT_CK(cudaMemcpyAsync(m->ws.emb_off, off, sizeof(int32_t) * (D.V + 1), cudaMemcpyHostToDevice, m->s_comp));
  MT_CK(cudaMemcpyAsync(m->ws.emb_pos, pos, sizeof(int32_t) * T, cudaMemcpyHostToDevice, m->s_comp));
  MT_CK(cudaMemcpyAsync(m->ws.emb_rows, rows, sizeof(int32_t) * u, cudaMemcpyHostToDevice, m->s_comp));
  (void)bytes;
}

// ------------------------------------------------------------------ FLOP accounting
// layer_fwd: one layer's forward; layer_internal: the internals that a
// backward visit recomputes (for a dense layer the forward without the down
// projection, whose output the backward does not need; an MoE layer recomputes
// its experts' outputs too, for the gate gradient); head_fwd: the LM head's
// forward.  Attention counts the causal half of QK^T and PV; a backward counts
// as two forwards (the usual convention for the model FLOPs).  MoE layers count
// the router and k experts per token (not the rows padding each expert's
// group to a multiple of 64).
struct Flops {
  double layer_fwd, layer_internal, head_fwd;
};
Flops flop_model(const Dims& D) {
  const double T = (double)D.T;
  const double attn_lin = (double)D.d * D.Dqkv + (double)D.Dq * D.d;
  const double mlp = D.E ? D.k * 3.0 * D.d * D.f + (double)D.d * D.E : 3.0 * D.d * D.f;
  const double attn = 4.0 * D.B * D.Hq * D.hd * ((double)D.S * (D.S + 1) / 2.0);
  const double fwd = 2.0 * T * (attn_lin + mlp) + attn;
  const double down = D.E ? 0.0 : 2.0 * T * (double)D.f * D.d;
  return Flops{fwd, fwd - down, 2.0 * T * (double)D.d * D.V};
}

// ------------------------------------------------------------------ the step
bf16* x_fwd_loc(mt_model* m, int i) {
  if (i < m->D.L && i >= m->keep_from) return m->stored[i - m->keep_from].x;
  return (i < m->keep_from && i % m->K == 0) ? m->ckpt[i / m->K] : m->xtmp[i % 2];
}

// Replica group, once this replica's gradients are all in the shared tiles:
// wait for every replica to get there, then take the global loss (the
// replicas' scaled losses summed in rank order, as mt_train_step_micro sums
// its micro-batches) and the group's non-finite verdict for the step.
void group_finish_step(mt_model* m) {
  auto& g = m->grp;
  const int64_t s = g.s;
  g.h->loss[s & 1][g.rank] = m->pinned_scalars[0];
  aadd(&g.h->steps_done, (int64_t)1);
  group_wait(m, [&] { return aload(&g.h->steps_done) >= (s + 1) * g.n; }, "every replica to finish the step");
  float loss = 0.f;
  for (int r = 0; r < g.n; ++r) loss += g.h->loss[s & 1][r];
  m->pinned_scalars[0] = loss;
  if (aload(&g.h->nonfinite_step) == s + 1) m->nonfinite = true;
}

int run_step(mt_model* m, const int32_t* tokens_host, const int32_t* tokens_dev, size_t n_tokens, float* loss_out) {
  const Dims& D = m->D;
  if (m->broken) {
    m->err = "handle is unusable after an earlier CUDA or internal error: " + m->err;
    return MT_ESTATE;
  }
  if (n_tokens != (size_t)D.B * (D.S + 1)) {
    m->err = "n_tokens must equal batch * (seq + 1)";
    return MT_EINVAL;
  }
  for (size_t t = 0; t < m->tiles.size(); ++t)
    if (!(m->group() ? aload(&m->grp.loaded[t]) != 0 : m->w_loaded[t] != 0)) {
      m->err = "tile " + std::to_string(t) + " has no weights loaded";
      return MT_ESTATE;
    }
  if (m->group() && aload(&m->grp.h->failed)) {
    m->err = "a replica of the group failed; the group is unusable";
    m->broken = true;
    return MT_ESTATE;
  }
  const auto wall0 = Clock::now();
  int code = MT_OK;
  try {
    MT_CK(cudaSetDevice(m->device));
    std::vector<int32_t> host_tok;
    if (tokens_dev) {
      host_tok.resize(n_tokens);
      MT_CK(cudaMemcpyAsync(host_tok.data(), tokens_dev, n_tokens * 4, cudaMemcpyDeviceToHost, m->s_comp));
      MT_CK(cudaStreamSynchronize(m->s_comp));
      tokens_host = host_tok.data();
    }
    if (m->async_adam) {
      // The previous step's embedding Adam reads that step's token tables,
      // which this step overwrites; and a deferred task that failed fails
      // this call before the per-step state is reset.
      wait_adam(m, 0);
      check_abort(m);
    }
    // reset per-step state
    {
      std::lock_guard<std::mutex> g(m->mu);
      std::fill(m->rec_ready.begin(), m->rec_ready.end(), 0);
      std::fill(m->rec_free.begin(), m->rec_free.end(), 0);
      std::fill(m->rec_d2h.begin(), m->rec_d2h.end(), 0);
      std::fill(m->rec_h2d_timed.begin(), m->rec_h2d_timed.end(), 0);
      std::fill(m->rec_d2h_timed.begin(), m->rec_d2h_timed.end(), 0);
      std::fill(m->rec_wait_timed.begin(), m->rec_wait_timed.end(), 0);
      std::fill(m->host_wait_ready_ms.begin(), m->host_wait_ready_ms.end(), 0.0);
      std::fill(m->host_wait_gbuf_ms.begin(), m->host_wait_gbuf_ms.end(), 0.0);
      m->abort_flag = false;
      m->worker_code = 0;
      m->worker_msg.clear();
      m->acc_tiles_done = 0;
      m->tl_h2d_n = 0;
      m->tl_d2h_n = 0;
      m->d2h_q.clear();
      m->acc_q.clear();
    }
    if (m->micro_index == 0 || m->group()) m->nonfinite = false;
    m->adam_us = 0;
    m->ls = LaunchStats{};
    m->ls.time_gemms = m->time_kernels;
    m->ls.gemm_events = &m->gemm_events;
    m->ls.gemm_event_flops = &m->gemm_event_flops;
    m->pinned_scalars[0] = 0.f;
    m->pinned_scalars[1] = 0.f;

    prepare_tokens(m, tokens_host);
    MT_CK(cudaMemsetAsync(m->ws.status, 0, sizeof(int), m->s_comp));
    if (m->resident_mode)
      for (size_t t = 0; t < m->tiles.size(); ++t)
        MT_CK(cudaMemcpyAsync(m->resident + m->resident_off[t], m->tiles[t] + m->layouts[t].off_w,
                              (size_t)m->layouts[t].w_bytes, cudaMemcpyHostToDevice, m->s_comp));
    if (m->direct_grads)
      MT_CK(cudaMemsetAsync(m->ws.grad_flags, 0, sizeof(int) * m->visits.size(), m->s_comp));
    MT_CK(cudaEventRecord(m->ev_t0, m->s_comp));
    const auto t_ev0 = Clock::now();
    {
      std::lock_guard<std::mutex> g(m->mu);
      m->step_gen += 1;
    }
    m->cv.notify_all();

    LayerTemplate tmpl{D, m->cfg.rms_eps, m->s_comp, &m->ws, &m->ls};
    tmpl.loss_scale = 1.0f / (float)m->micro_count;  // the loss is the mean over every micro-batch's tokens
    if (m->trace) {
      tmpl.trace_ctx = m;
      tmpl.trace_fn = [](void* ctx, const char* kernel) {
        mt_model* mm = static_cast<mt_model*>(ctx);
        const auto t0 = Clock::now();
        MT_CK(cudaEventRecord(mm->ev_t1, mm->s_comp));
        wait_event(mm, mm->ev_t1, kernel);
        int st = 0;
        MT_CK(cudaMemcpy(&st, mm->ws.status, sizeof(int), cudaMemcpyDeviceToHost));
        std::fprintf(stderr, "[mt trace]   %-26s %9.3f ms  status %d\n", kernel, ms_since(t0), st);
        if (st != 0) throw MtError{MT_ETIMEDOUT, std::string("device status ") + std::to_string(st) + " after " + kernel};
      };
    }
    bf16* dx_cur = m->ws.dx_a;
    bf16* dx_nxt = m->ws.dx_b;
    for (int v = 0; v < (int)m->visits.size(); ++v) {
      check_abort(m);
      const Visit& x = m->visits[v];
      NvtxRange range(kVisitRangeFmt[x.kind], x.layer, x.tile);
      if (m->trace)
        std::fprintf(stderr, "[mt trace] visit %d (tile %d, layer %d, buffer %d, h2d %d) starts\n", v, x.tile,
                     x.layer, x.buf, (int)x.h2d);
      uint8_t* wb = nullptr;
      if (x.buf >= 0) {
        if (m->resident_mode) {
          wb = m->resident + m->resident_off[x.tile];
        } else {
          if (x.h2d) {
            const auto tw = Clock::now();
            wait_flag(m, m->rec_ready, v, "weights ready");
            m->host_wait_ready_ms[v] = ms_since(tw);
            MT_CK(cudaEventRecord(m->ev_wait_a[v], m->s_comp));
            MT_CK(cudaStreamWaitEvent(m->s_comp, m->ev_ready[v], 0));
            MT_CK(cudaEventRecord(m->ev_wait_b[v], m->s_comp));
            m->rec_wait_timed[v] = 1;
          }
          wb = m->wbuf[x.buf];
        }
      }
      uint8_t* gb = nullptr;
      if (x.grads) {
        if (x.prev_gbuf_user >= 0) {
          const auto tw = Clock::now();
          wait_flag(m, m->rec_d2h, x.prev_gbuf_user, "gradient buffer evacuated");
          m->host_wait_gbuf_ms[v] = ms_since(tw);
          MT_CK(cudaStreamWaitEvent(m->s_comp, m->ev_d2h[x.prev_gbuf_user], 0));
        }
        gb = m->gbuf[x.gbuf];
      }
      const TileLayout& lay = m->layouts[x.tile];
      int rc = 0;
      MT_CK(cudaEventRecord(m->ev_vis_a[v], m->s_comp));
      switch (x.kind) {
        case kEmbedFwd:
          rc = tmpl.embed_fwd(reinterpret_cast<bf16*>(wb + lay.slot("E").offset), x_fwd_loc(m, 0));
          break;
        case kLayerFwd: {
          const int i = x.layer;
          const bool kept = i >= m->keep_from;
          LayerActs a = kept ? m->stored[i - m->keep_from] : m->acts;
          a.x = x_fwd_loc(m, i);
          rc = tmpl.forward(bind_layer(lay, wb), a, x_fwd_loc(m, i + 1), kept);
          break;
        }
        case kHead:
          rc = tmpl.head(bind_head(lay, wb), x_fwd_loc(m, D.L), dx_cur, bind_head(lay, gb));
          MT_CK(cudaMemcpyAsync(m->pinned_scalars, m->ws.loss, sizeof(float), cudaMemcpyDeviceToHost, m->s_comp));
          break;
        case kRecompute: {
          const int j = x.layer, s = j / m->K * m->K;
          LayerActs a = m->acts;
          a.x = (j == s) ? m->ckpt[s / m->K] : m->blockbuf[j - s - 1];
          rc = tmpl.forward(bind_layer(lay, wb), a, m->blockbuf[j - s], false);
          break;
        }
        case kLayerBwd: {
          const int j = x.layer;
          LayerActs a;
          if (j >= m->keep_from) {
            a = m->stored[j - m->keep_from];
          } else {
            const int s = j / m->K * m->K;
            a = m->acts;
            a.x = (j == s) ? m->ckpt[s / m->K] : m->blockbuf[j - s - 1];
            rc = tmpl.forward(bind_layer(lay, wb), a, nullptr, true);  // internals only
          }
          rc |= tmpl.backward(bind_layer(lay, wb), a, dx_cur, dx_nxt, bind_layer(lay, gb));
          std::swap(dx_cur, dx_nxt);
          break;
        }
        case kEmbedBwd:  // compact: the rows of the step's token ids, packed from the buffer start
          rc = tmpl.embed_bwd_rows(dx_cur, reinterpret_cast<bf16*>(gb), m->emb_u);
          break;
      }
      if (rc != 0) throw MtError{MT_ECUDA, std::string("kernel launch failed: ") + last_launch_error()};
      MT_CK(cudaPeekAtLastError());
      MT_CK(cudaEventRecord(m->ev_vis_b[v], m->s_comp));
      if (x.buf >= 0 && !m->resident_mode) {
        MT_CK(cudaEventRecord(m->ev_free[v], m->s_comp));
        set_flag(m, m->rec_free, v);
      }
      if (m->trace) {
        // debugging: finish this visit, report its time and the device status
        const auto t0 = Clock::now();
        MT_CK(cudaEventRecord(m->ev_t1, m->s_comp));
        wait_event(m, m->ev_t1, "traced visit");
        int st = 0;
        MT_CK(cudaMemcpy(&st, m->ws.status, sizeof(int), cudaMemcpyDeviceToHost));
        static const char* kind_name[] = {"embed_fwd", "layer_fwd", "head", "recompute", "layer_bwd", "embed_bwd"};
        std::fprintf(stderr, "[mt trace] visit %d %s tile %d layer %d: %.3f ms after issue, status %d\n", v,
                     kind_name[x.kind], x.tile, x.layer, ms_since(t0), st);
        if (st != 0)
          throw MtError{MT_ETIMEDOUT, "device status " + std::to_string(st) + " after visit " + std::to_string(v) +
                                          " (" + kind_name[x.kind] + ", layer " + std::to_string(x.layer) + ")"};
      }
      if (x.grads) {
        if (m->debug)
          launch_check_finite(reinterpret_cast<bf16*>(gb),
                              x.kind == kEmbedBwd ? (int64_t)m->emb_u * D.d : lay.w_bytes / 2, m->ws.status,
                              m->s_comp);
        if (m->direct_grads && x.kind != kEmbedBwd && m->micro_index == 0)
          launch_flag_nonfinite(reinterpret_cast<bf16*>(gb), lay.w_bytes / 2, m->grad_flags + v, m->s_comp);
        MT_CK(cudaEventRecord(m->ev_grads[v], m->s_comp));
        {
          std::lock_guard<std::mutex> g(m->mu);
          m->d2h_q.push_back(v);
        }
        m->cv.notify_all();
      }
    }
    MT_CK(cudaEventRecord(m->ev_t1, m->s_comp));
    MT_CK(cudaMemcpyAsync(m->pinned_scalars + 1, m->ws.status, sizeof(int), cudaMemcpyDeviceToHost, m->s_comp));
    wait_event(m, m->ev_t1, "compute stream");
    MT_CK(cudaStreamSynchronize(m->s_comp));
    const auto t_compute_done = Clock::now();
    const int status = *reinterpret_cast<int*>(m->pinned_scalars + 1);
    // drain the gradient path and Adam
    wait_flag(m, m->rec_d2h, m->last_grad_visit, "last gradient evacuation");
    {
      std::unique_lock<std::mutex> g(m->mu);
      const bool ok = m->cv.wait_for(g, std::chrono::milliseconds(m->cfg.timeout_ms),
                                     [&] { return m->acc_tiles_done >= m->n_grad_visits || m->abort_flag.load(); });
      if (m->abort_flag) throw MtError{m->worker_code ? m->worker_code.load() : MT_EINTERNAL, m->worker_msg};
      if (!ok) throw MtError{MT_ETIMEDOUT, "timed out waiting for gradient accumulation"};
    }
    const auto t_grads_done = Clock::now();
    if (m->group()) group_finish_step(m);
    // MT_ASYNC_ADAM: the step returns with Adam tasks still running; each
    // tile's finish before it is uploaded again or read through the API
    if (!m->async_adam && !m->adam_pool->wait_idle(m->cfg.timeout_ms))
      throw MtError{MT_ETIMEDOUT, "timed out waiting for Adam"};
    if (m->group() && !m->async_adam) group_wait_adam(m, -1, m->grp.s + 1);
    const auto adam_end = Clock::now();
    check_abort(m);
    MT_CK(cudaStreamSynchronize(m->s_h2d));
    MT_CK(cudaStreamSynchronize(m->s_d2h));

    // statistics
    mt_step_stats& st = m->stats;
    st = mt_step_stats{};
    st.loss = m->pinned_scalars[0];
    float f = 0.f;
    MT_CK(cudaEventElapsedTime(&f, m->ev_t0, m->ev_t1));
    st.gpu_compute_ms = f;
    for (int v = 0; v < (int)m->visits.size(); ++v) {
      if (m->rec_h2d_timed[v] && cudaEventElapsedTime(&f, m->ev_h2d_a[v], m->ev_h2d_b[v]) == cudaSuccess) st.h2d_ms += f;
      if (m->rec_d2h_timed[v] && cudaEventElapsedTime(&f, m->ev_d2h_a[v], m->ev_d2h_b[v]) == cudaSuccess) st.d2h_ms += f;
      if (m->rec_wait_timed[v] && cudaEventElapsedTime(&f, m->ev_wait_a[v], m->ev_wait_b[v]) == cudaSuccess)
        st.wait_weights_ms += f;
      float gap = 0.f;
      if (v > 0 && cudaEventElapsedTime(&gap, m->ev_vis_b[v - 1], m->ev_vis_a[v]) == cudaSuccess) st.visit_gap_ms += gap;
      if (m->visit_log) {
        static const char* kind_name[] = {"embed_fwd", "layer_fwd", "head", "recompute", "layer_bwd", "embed_bwd"};
        float run = 0.f, ww = 0.f, end = 0.f, d2h_a = -1.f, d2h_b = -1.f;
        cudaEventElapsedTime(&run, m->ev_vis_a[v], m->ev_vis_b[v]);
        cudaEventElapsedTime(&end, m->ev_t0, m->ev_vis_b[v]);
        if (m->rec_wait_timed[v]) cudaEventElapsedTime(&ww, m->ev_wait_a[v], m->ev_wait_b[v]);
        if (m->rec_d2h_timed[v]) {
          cudaEventElapsedTime(&d2h_a, m->ev_t0, m->ev_d2h_a[v]);
          cudaEventElapsedTime(&d2h_b, m->ev_t0, m->ev_d2h_b[v]);
        }
        std::fprintf(stderr,
                     "[mt visit] %3d %-9s layer %3d  gap %7.3f ms  run %8.3f ms  stream wait weights %7.3f ms  "
                     "host wait weights %7.3f ms  host wait grad buffer %7.3f ms  ends at %8.2f ms  "
                     "gradient copy %8.2f .. %8.2f ms\n",
                     v, kind_name[m->visits[v].kind], m->visits[v].layer, gap, run, ww, m->host_wait_ready_ms[v],
                     m->host_wait_gbuf_ms[v], end, d2h_a, d2h_b);
      }
      const Visit& x = m->visits[v];
      if (x.h2d && !m->resident_mode) st.h2d_bytes += m->layouts[x.tile].w_bytes;
      if (x.grads) st.d2h_bytes += x.kind == kEmbedBwd ? 2LL * m->emb_u * D.d : m->layouts[x.tile].w_bytes;
    }
    cudaGetLastError();
    for (size_t i = 0; i + 1 < m->gemm_events.size(); i += 2) {
      if (cudaEventElapsedTime(&f, m->gemm_events[i], m->gemm_events[i + 1]) == cudaSuccess) st.gemm_ms += f;
      cudaEventDestroy(m->gemm_events[i]);
      cudaEventDestroy(m->gemm_events[i + 1]);
    }
    for (double fl : m->gemm_event_flops) st.gemm_flops += fl;
    m->gemm_events.clear();
    m->gemm_event_flops.clear();
    st.gemm_launches = m->ls.gemms;
    st.kernel_launches = m->ls.kernels;
    st.adam_ms = m->adam_us.load() / 1000.0;
    st.adam_tail_ms = std::chrono::duration<double, std::milli>(adam_end - m->last_grads_landed).count();
    const Flops fm = flop_model(D);
    // executed: every forward visit and boundary recompute in full, every
    // backward visit's internal recompute (when activations are not stored),
    // each layer's backward, and the head's forward and backward once
    int n_fwd = 0, n_internal = 0;
    for (const auto& x : m->visits) {
      if (x.kind == kLayerFwd || x.kind == kRecompute) ++n_fwd;
      if (x.kind == kLayerBwd && x.layer < m->keep_from) ++n_internal;
    }
    st.flops_model = (int64_t)(3.0 * (D.L * fm.layer_fwd + fm.head_fwd));
    st.flops_executed = (int64_t)(n_fwd * fm.layer_fwd + n_internal * fm.layer_internal + 2.0 * D.L * fm.layer_fwd +
                                  3.0 * fm.head_fwd);
    st.arena_high_water = m->arena_used;
    if (status != 0) {
      if (status == kStatusGemmTimeout)
        throw MtError{MT_ETIMEDOUT, "a device-side bounded wait expired (GEMM pipeline)"};
      if (status == kStatusAttnFwdTimeout || status == kStatusAttnBwdTimeout || status / 1000 == kStatusAttnFwdTimeout ||
          status / 1000 == kStatusAttnBwdTimeout)
        throw MtError{MT_ETIMEDOUT, "a device-side bounded wait expired (attention pipeline, code " +
                                        std::to_string(status) + ")"};
      if (status == kStatusNonFinite) {
        m->nonfinite = true;
      } else {
        throw MtError{MT_EINVAL, "device status " + std::to_string(status) + " (index out of range)"};
      }
    }
    if (m->last_pass() || m->group()) m->step += 1;
    if (m->group()) m->grp.s += 1;
    st.step = m->step;
    st.step_ms = ms_since(wall0);
    auto span = [](Clock::time_point a, Clock::time_point b) {
      return std::chrono::duration<double, std::milli>(b - a).count();
    };
    st.host_pre_ms = span(wall0, t_ev0);
    st.tail_grads_ms = span(t_compute_done, t_grads_done);
    if (m->visit_log)
      std::fprintf(stderr, "[mt visit] compute stream ends at %8.2f ms; host: all gradients accumulated %.2f ms "
                           "and Adam done %.2f ms after the compute stream was seen finished\n",
                   st.gpu_compute_ms, st.tail_grads_ms, span(t_compute_done, adam_end));
    st.tail_adam_ms = span(t_grads_done, adam_end);
    st.tail_rest_ms = span(adam_end, Clock::now());
    if (loss_out) *loss_out = m->pinned_scalars[0];
    if (m->nonfinite) {
      m->err = "non-finite loss or gradient; Adam skipped from the first affected tile on";
      code = MT_ENONFINITE;
    }
  } catch (const MtError& e) {
    m->err = e.msg;
    code = e.code;
    // stop the workers' part of this step and bring the streams to rest
    worker_fail(m, e);
    const bool drained = drain_stream(m->s_comp, m->cfg.timeout_ms) & drain_stream(m->s_h2d, m->cfg.timeout_ms) &
                         drain_stream(m->s_d2h, m->cfg.timeout_ms);
    if (!drained) {
      m->err += " (streams did not drain within the timeout; the handle keeps its buffers until mt_free)";
      m->undrained = true;
    }
    m->adam_pool->wait_idle(m->cfg.timeout_ms);
    if (code != MT_EINVAL) m->broken = true;
  }
  m->inject_what = MT_INJECT_NONE;  // an injection arms one step only
  return code;
}

// ------------------------------------------------------------------ init helpers
const char* validate(const mt_config& c) {
  if (c.n_layers < 1 || c.d_model < 8 || c.n_heads < 1 || c.n_kv_heads < 1 || c.ffn < 8 || c.vocab < 8 ||
      c.batch < 1 || c.seq < 1)
    return "dimensions must be positive";
  if (c.head_dim != 64 && c.head_dim != 128) return "head_dim must be 64 or 128";
  if (c.n_heads % c.n_kv_heads) return "n_heads must be a multiple of n_kv_heads";
  if (c.d_model % 8 || c.ffn % 8 || c.vocab % 8) return "d_model, ffn and vocab must be multiples of 8";
  if (((int64_t)c.batch * c.seq) % 8) return "batch * seq must be a multiple of 8";
  if (c.ckpt_every < 1) return "ckpt_every must be >= 1";
  if (c.mlp_chunk_rows < 0 || c.mlp_chunk_rows % 128) return "mlp_chunk_rows must be a multiple of 128 (0 = unchunked)";
  if (c.n_experts < 0 || c.n_experts > 256 || c.n_experts % 8)
    return "n_experts must be 0 (dense) or a multiple of 8 up to 256";
  if (c.n_experts > 0) {
    if (c.top_k < 1 || c.top_k > 8 || c.top_k > c.n_experts) return "top_k must be in 1 .. min(8, n_experts)";
    if (c.ffn % 8) return "MoE layers need ffn (the expert width) to be a multiple of 8";
    if ((int64_t)c.batch * c.seq * c.top_k + 63LL * c.n_experts > 0x7fffffffLL)
      return "MoE layers: batch * seq * top_k (plus padding) must fit int32 row positions";
    if (c.mlp_chunk_rows > 0 && c.mlp_chunk_rows < (int64_t)c.batch * c.seq)
      return "mlp_chunk_rows does not apply to MoE layers";
  }
  if (c.keep_layers < 0) return "keep_layers must be >= 0";
  if (c.n_replicas < 0 || c.n_replicas > kMaxReplicas) return "n_replicas must be in 0 .. 64";
  if (c.n_replicas >= 2) {
    if (c.replica_rank < 0 || c.replica_rank >= c.n_replicas) return "replica_rank must be in 0 .. n_replicas - 1";
    const size_t len = strnlen(c.replica_name, sizeof(c.replica_name));
    if (len == 0 || len == sizeof(c.replica_name)) return "replica_name must be a non-empty NUL-terminated name";
    for (size_t i = 0; i < len; ++i) {
      const char ch = c.replica_name[i];
      if (!((ch >= 'a' && ch <= 'z') || (ch >= 'A' && ch <= 'Z') || (ch >= '0' && ch <= '9') || ch == '_' ||
            ch == '-' || ch == '.'))
        return "replica_name may hold letters, digits, '_', '-' and '.' only";
    }
    if (c.flags & MT_RESIDENT) return "a replica group streams its weights: MT_RESIDENT does not apply";
    if (c.flags & MT_TIE_EMBEDDINGS) return "a replica group does not support MT_TIE_EMBEDDINGS";
  }
  if (c.mlp_chunk_rows > 0 && c.mlp_chunk_rows < (int64_t)c.batch * c.seq &&
      ((c.flags & MT_STORE_ACTS) || c.keep_layers > 0))
    return "a chunked MLP keeps no per-layer gate/up activations: not combinable with MT_STORE_ACTS or keep_layers";
  if (c.grad_slab_bytes > 0 && align_up(c.grad_slab_bytes, kPage) < 2LL * c.d_model)
    return "grad_slab_bytes must hold one embedding row (2 * d_model bytes)";
  if (!(c.rms_eps > 0) || !(c.rope_theta > 0) || !(c.lr >= 0) || !(c.beta1 >= 0 && c.beta1 < 1) ||
      !(c.beta2 >= 0 && c.beta2 < 1) || !(c.adam_eps >= 0))
    return "bad hyper-parameter";
  return nullptr;
}

mt_config with_defaults(const mt_config& in) {
  mt_config c = in;
  // Adam is bound by host memory bandwidth well before every core is busy;
  // three quarters of the hardware threads leave cores and bandwidth to the
  // packers and the gradient accumulator.
  if (c.n_adam_threads <= 0) c.n_adam_threads = std::max(1u, std::thread::hardware_concurrency() * 3 / 4);
  if (c.n_pack_threads <= 0) c.n_pack_threads = 8;
  if (c.n_grad_slabs <= 0) c.n_grad_slabs = 24;  // 1.5 GiB pinned at 64 MiB: absorbs the LM head's gradient burst
  if (c.grad_slab_bytes <= 0) c.grad_slab_bytes = 64ll << 20;
  if (c.stage_bytes <= 0) c.stage_bytes = 64ll << 20;
  if (c.timeout_ms <= 0) c.timeout_ms = 60000;
  c.grad_slab_bytes = align_up(c.grad_slab_bytes, kPage);
  c.stage_bytes = align_up(c.stage_bytes, kPage);
  return c;
}

// First layer that keeps its internals on the device (n_layers: none).
int keep_from_of(const mt_config& c) {
  if (c.flags & MT_STORE_ACTS) return 0;
  return std::max(0, c.n_layers - std::max(0, c.keep_layers));
}

// Lay out the device arena; with base == nullptr only the byte count is computed.
int64_t plan_arena(mt_model* m, uint8_t* base) {
  const Dims& D = m->D;
  Plan P;
  auto at = [&](int64_t bytes) -> uint8_t* {
    const int64_t off = P.add(bytes);
    return base ? base + off : nullptr;
  };
  const int64_t xb = D.T * D.d * 2;
  for (int b = 0; b < 2; ++b) m->wbuf[b] = at(m->max_w_bytes);
  for (int b = 0; b < 3; ++b) m->gbuf[b] = at(m->gbuf_bytes[b]);
  if (m->resident_mode) {
    int64_t tot = 0;
    m->resident_off.assign(m->layouts.size(), 0);
    for (size_t t = 0; t < m->layouts.size(); ++t) {
      m->resident_off[t] = tot;
      tot += m->layouts[t].w_bytes;
    }
    m->resident = at(tot);
  }
  const ActsSizes as = acts_sizes(D);
  m->ckpt.clear();
  m->blockbuf.clear();
  m->stored.clear();
  // kept layers: their input and internals, one set each
  for (int i = m->keep_from; i < D.L; ++i) {
    uint8_t* x = at(xb);
    uint8_t* p = at(as.total);
    m->stored.push_back(base ? carve_acts(p, D, reinterpret_cast<bf16*>(x)) : LayerActs{});
  }
  // recomputed layers: their block checkpoints, the block buffers and one
  // shared set of internals
  if (m->keep_from > 0) {
    for (int i = 0; i < (m->keep_from + m->K - 1) / m->K; ++i) m->ckpt.push_back(reinterpret_cast<bf16*>(at(xb)));
    for (int i = 0; i < std::min(m->K, m->keep_from) - 1; ++i) m->blockbuf.push_back(reinterpret_cast<bf16*>(at(xb)));
    uint8_t* p = at(as.total);
    if (base) m->acts = carve_acts(p, D, nullptr);
  }
  for (int b = 0; b < 2; ++b) m->xtmp[b] = reinterpret_cast<bf16*>(at(xb));
  uint8_t* wsbase = base ? base + P.total : nullptr;
  Plan Pw;
  Workspace w = carve_ws(wsbase, D, Pw);
  P.total += Pw.total;
  if (base) m->ws = w;
  return P.total;
}

void build_layouts(mt_model* m) {
  m->layouts.clear();
  m->tied = m->cfg.flags & MT_TIE_EMBEDDINGS;
  m->layouts.push_back(make_layout(kTileEmbed, m->D, m->tied));
  for (int i = 0; i < m->D.L; ++i) m->layouts.push_back(make_layout(kTileLayer, m->D));
  if (!m->tied) m->layouts.push_back(make_layout(kTileHead, m->D));
  m->head_tile = m->tied ? 0 : m->D.L + 1;
  m->max_w_bytes = 0;
  for (const auto& l : m->layouts) m->max_w_bytes = std::max(m->max_w_bytes, l.w_bytes);
  int64_t layer_bytes = 0;
  for (int i = 1; i <= m->D.L; ++i) layer_bytes = std::max(layer_bytes, m->layouts[i].w_bytes);
  m->gbuf_bytes[0] = m->gbuf_bytes[1] = layer_bytes;
  m->gbuf_bytes[2] =
      std::max<int64_t>(m->layouts[m->head_tile].w_bytes, std::min<int64_t>(m->D.T, m->D.V) * 2LL * m->D.d);
}

void parallel_zero(uint8_t* p, int64_t n, int nthreads) {
  std::vector<std::thread> th;
  const int64_t piece = align_up((n + nthreads - 1) / nthreads, kPage);
  for (int64_t off = 0; off < n; off += piece) {
    const int64_t c = std::min(piece, n - off);
    th.emplace_back([=] { std::memset(p + off, 0, (size_t)c); });
  }
  for (auto& t : th) t.join();
}

// Replica group: map the shared segment (control block, then every tile on a
// page boundary) and point the tiles into it.  Replica 0 creates it (fresh
// shared memory reads as zeros, so the tiles start zeroed) and removes the
// name once all n replicas have attached; the others open it once it exists
// with the expected size and its control block is marked ready.
void group_attach(mt_model* m) {
  auto& g = m->grp;
  const mt_config& c = m->cfg;
  const int rank = c.replica_rank, n = c.n_replicas;  // the handle's group fields are set once attached
  const int64_t nt = (int64_t)m->layouts.size();
  g.chunk_base.assign(nt + 1, 0);
  for (int64_t t = 0; t < nt; ++t)
    g.chunk_base[t + 1] = g.chunk_base[t] + (m->layouts[t].w_bytes + m->slab_bytes - 1) / m->slab_bytes;
  const int64_t n_chunks = g.chunk_base[nt];
  const int64_t head = align_up((int64_t)sizeof(GroupHeader) + 8 * n_chunks + 12 * nt, kPage);
  std::vector<int64_t> tile_off(nt);
  int64_t total = head;
  for (int64_t t = 0; t < nt; ++t) {
    tile_off[t] = total;
    total += align_up(m->layouts[t].tile_bytes, kPage);
  }
  const std::string name = std::string("/") + c.replica_name;
  const auto t0 = Clock::now();
  auto expired = [&] { return ms_since(t0) > (double)c.timeout_ms; };
  int fd = -1;
  if (rank == 0) {
    shm_unlink(name.c_str());  // a leftover of a group that never finished attaching
    fd = shm_open(name.c_str(), O_CREAT | O_EXCL | O_RDWR, 0600);
    if (fd < 0) throw MtError{MT_ENOMEM, "shm_open(" + name + "): " + std::strerror(errno)};
    if (ftruncate(fd, (off_t)total) != 0) {
      const int e = errno;
      close(fd);
      shm_unlink(name.c_str());
      throw MtError{MT_ENOMEM, "sizing the replica group's shared memory to " + std::to_string(total) +
                                   " bytes: " + std::strerror(e)};
    }
  } else {
    while (true) {
      fd = shm_open(name.c_str(), O_RDWR, 0);
      if (fd >= 0) {
        struct stat st {};
        if (fstat(fd, &st) == 0 && st.st_size == (off_t)total) break;
        close(fd);
        fd = -1;
      }
      if (expired())
        throw MtError{MT_ETIMEDOUT, "replica " + std::to_string(rank) + ": no shared segment " + name + " of " +
                                        std::to_string(total) + " bytes appeared (is replica 0 running with the "
                                        "same config?)"};
      std::this_thread::sleep_for(std::chrono::milliseconds(1));
    }
  }
  void* p = mmap(nullptr, (size_t)total, PROT_READ | PROT_WRITE, MAP_SHARED, fd, 0);
  const int map_errno = errno;
  close(fd);
  if (p == MAP_FAILED) {
    if (rank == 0) shm_unlink(name.c_str());
    throw MtError{MT_ENOMEM, std::string("mapping the replica group's shared memory: ") + std::strerror(map_errno)};
  }
  g.base = static_cast<uint8_t*>(p);
  g.bytes = (size_t)total;
  madvise(p, (size_t)total, MADV_HUGEPAGE);  // as for a model's own tiles; shared memory may decline
  g.h = reinterpret_cast<GroupHeader*>(g.base);
  g.turn = reinterpret_cast<int64_t*>(g.base + sizeof(GroupHeader));
  g.adam_done = g.turn + n_chunks;
  g.loaded = reinterpret_cast<int32_t*>(g.adam_done + nt);
  g.final_val.assign(nt, 0);
  GroupHeader* h = g.h;
  if (rank == 0) {
    h->total_bytes = total;
    h->n_chunks = n_chunks;
    h->slab_bytes = m->slab_bytes;
    h->n_tiles = nt;
    h->n_replicas = n;
    h->magic = kGroupMagic;
    astore(&h->ready, 1);
  } else {
    while (!aload(&h->ready)) {
      if (expired()) throw MtError{MT_ETIMEDOUT, "replica group: the control block was never marked ready"};
      std::this_thread::sleep_for(std::chrono::milliseconds(1));
    }
    if (h->magic != kGroupMagic || h->total_bytes != total || h->n_chunks != n_chunks ||
        h->slab_bytes != m->slab_bytes || h->n_tiles != nt || h->n_replicas != n)
      throw MtError{MT_EINVAL, "replica group: this replica's config differs from replica 0's"};
  }
  if (aadd(&h->attached, 1) > n)
    throw MtError{MT_EINVAL, "replica group: more replicas attached than n_replicas (a reused replica_name?)"};
  if (rank == 0) {
    while (aload(&h->attached) < n) {
      if (expired()) {
        shm_unlink(name.c_str());
        throw MtError{MT_ETIMEDOUT, "replica group: only " + std::to_string(aload(&h->attached)) + " of " +
                                        std::to_string(n) + " replicas attached"};
      }
      std::this_thread::sleep_for(std::chrono::milliseconds(1));
    }
    shm_unlink(name.c_str());
  }
  for (int64_t t = 0; t < nt; ++t) m->tiles[t] = g.base + tile_off[t];
  m->micro_index = rank;  // replica r adds its gradients as micro-batch r of the group's step
  m->micro_count = n;
  g.rank = rank;
  g.n = n;
}

// Size of a transparent huge page on this host (2 MiB when the kernel does not say).
int64_t huge_page_bytes() {
  int64_t v = 0;
  if (FILE* f = std::fopen("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size", "r")) {
    long long x = 0;
    if (std::fscanf(f, "%lld", &x) == 1) v = x;
    std::fclose(f);
  }
  return v >= kPage && (v & (v - 1)) == 0 ? v : (2LL << 20);
}

// Host tiles of a model of its own: one anonymous mapping holding every tile
// on a page boundary, started on a huge-page boundary and advised for
// transparent huge pages (where the kernel grants them: fewer translations for
// the CPU Adam workers' streaming and shorter page lists for the DMA engines'
// in-place copies).  First touch, which zeroes, is spread over threads.
void alloc_tiles(mt_model* m) {
  const int64_t huge = huge_page_bytes();
  std::vector<int64_t> off(m->layouts.size());
  int64_t total = 0;
  for (size_t t = 0; t < m->layouts.size(); ++t) {
    off[t] = total;
    total += align_up(m->layouts[t].tile_bytes, kPage);
  }
  const size_t map_bytes = (size_t)(total + huge);
  void* p = mmap(nullptr, map_bytes, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
  if (p == MAP_FAILED)
    throw MtError{MT_ENOMEM, "host tile allocation of " + std::to_string(total) + " bytes failed"};
  m->tile_map = static_cast<uint8_t*>(p);
  m->tile_map_bytes = map_bytes;
  uint8_t* base = reinterpret_cast<uint8_t*>(align_up((int64_t)reinterpret_cast<uintptr_t>(p), huge));
  madvise(base, (size_t)total, MADV_HUGEPAGE);  // advisory: a refusal leaves ordinary pages
  for (size_t t = 0; t < m->layouts.size(); ++t) {
    m->tiles[t] = base + off[t];
    parallel_zero(m->tiles[t], m->layouts[t].tile_bytes, std::min(16, m->cfg.n_adam_threads));
  }
}

void destroy(mt_model* m) {
  if (!m) return;
  {
    std::lock_guard<std::mutex> g(m->mu);
    m->stop_threads = true;
    m->abort_flag = true;
  }
  m->cv.notify_all();
  if (m->loader.joinable()) m->loader.join();
  if (m->d2h.joinable()) m->d2h.join();
  if (m->accum.joinable()) m->accum.join();
  m->adam_pool.reset();
  m->pack_pool.reset();
  m->acc_pool.reset();
  bool drained = true;
  if (m->s_comp) drained &= drain_stream(m->s_comp, m->cfg.timeout_ms);
  if (m->s_h2d) drained &= drain_stream(m->s_h2d, m->cfg.timeout_ms);
  if (m->s_d2h) drained &= drain_stream(m->s_d2h, m->cfg.timeout_ms);
  if (!drained || m->undrained) {
    // work may still be running against the pinned buffers: leak them rather than free memory in use
    std::fprintf(stderr, "mt_free: streams still busy after %lld ms; pinned buffers are leaked\n",
                 (long long)m->cfg.timeout_ms);
    delete m;  // the tile mapping (page-locked in parts) is leaked with the buffers
    return;
  }
  auto kill = [](std::vector<cudaEvent_t>& v) {
    for (auto e : v)
      if (e) cudaEventDestroy(e);
    v.clear();
  };
  kill(m->ev_ready);
  kill(m->ev_free);
  kill(m->ev_grads);
  kill(m->ev_d2h);
  kill(m->ev_wait_a);
  kill(m->ev_wait_b);
  kill(m->ev_h2d_a);
  kill(m->ev_h2d_b);
  kill(m->ev_d2h_a);
  kill(m->ev_d2h_b);
  kill(m->ev_vis_a);
  kill(m->ev_vis_b);
  kill(m->ev_slab);
  kill(m->gemm_events);
  kill(m->tl_h2d);
  kill(m->tl_d2h);
  for (auto& e : m->ev_stage)
    if (e) cudaEventDestroy(e);
  if (m->ev_t0) cudaEventDestroy(m->ev_t0);
  if (m->ev_t1) cudaEventDestroy(m->ev_t1);
  for (auto& s : m->stage)
    if (s) cudaFreeHost(s);
  for (auto s : m->slabs)
    if (s) cudaFreeHost(s);
  if (m->pinned_scalars) cudaFreeHost(m->pinned_scalars);
  if (m->pinned_tok) cudaFreeHost(m->pinned_tok);
  if (m->pinned_flags) cudaFreeHost(m->pinned_flags);
  for (uint8_t* r : m->host_reg)
    if (r) cudaHostUnregister(r);
  if (m->grp.base) munmap(m->grp.base, m->grp.bytes);
  if (m->tile_map) munmap(m->tile_map, m->tile_map_bytes);
  delete m;
}

void init_model(mt_model* m, const mt_config& cin, void* arena, size_t arena_bytes, void* sc, void* sh, void* sd) {
  if (const char* e = validate(cin)) throw MtError{MT_EINVAL, e};
  m->cfg = with_defaults(cin);
  m->D = dims_of(m->cfg);
  m->K = m->cfg.ckpt_every;
  m->resident_mode = m->cfg.flags & MT_RESIDENT;
  m->store_acts = m->cfg.flags & MT_STORE_ACTS;
  m->async_adam = m->cfg.flags & MT_ASYNC_ADAM;
  m->direct_grads = m->cfg.flags & MT_DIRECT_GRADS;
  m->direct_weights = m->cfg.flags & MT_DIRECT_WEIGHTS;
  m->keep_from = keep_from_of(m->cfg);
  m->single_buffer = m->cfg.flags & MT_NO_DOUBLE_BUFFER;
  m->debug = m->cfg.flags & MT_DEBUG_CHECKS;
  m->time_kernels = m->cfg.flags & MT_TIME_KERNELS;
  m->trace = m->cfg.flags & MT_TRACE;
  m->visit_log = m->cfg.flags & MT_VISIT_LOG;
  if (!sc || !sh || !sd || sc == sh || sc == sd || sh == sd)
    throw MtError{MT_EINVAL, "three distinct CUDA streams are required"};
  MT_CK(cudaGetDevice(&m->device));
  m->s_comp = static_cast<cudaStream_t>(sc);
  m->s_h2d = static_cast<cudaStream_t>(sh);
  m->s_d2h = static_cast<cudaStream_t>(sd);
  build_layouts(m);
  m->adam_pending.assign(m->layouts.size(), 0);
  const int64_t need = plan_arena(m, nullptr);
  if (!arena || (reinterpret_cast<uintptr_t>(arena) & 255)) throw MtError{MT_EINVAL, "device arena must be 256-byte aligned"};
  if ((int64_t)arena_bytes < need)
    throw MtError{MT_ENOMEM, "device arena too small: need " + std::to_string(need) + " bytes"};
  m->arena = static_cast<uint8_t*>(arena);
  m->arena_bytes = arena_bytes;
  m->arena_used = plan_arena(m, m->arena);

  // visit schedule
  m->visits = build_schedule(m->D.L, m->K, m->keep_from, m->single_buffer, m->head_tile);
  if (m->resident_mode)
    for (auto& x : m->visits) x.h2d = false;
  const int nv = (int)m->visits.size();
  m->n_grad_visits = 0;
  for (int v = 0; v < nv; ++v)
    if (m->visits[v].grads) {
      ++m->n_grad_visits;
      m->last_grad_visit = v;
    }
  auto mk = [&](std::vector<cudaEvent_t>& vec, bool timing) {
    vec.assign(nv, nullptr);
    for (auto& e : vec) MT_CK(cudaEventCreateWithFlags(&e, timing ? cudaEventDefault : cudaEventDisableTiming));
  };
  mk(m->ev_ready, false);
  mk(m->ev_free, false);
  mk(m->ev_grads, false);
  mk(m->ev_d2h, false);
  mk(m->ev_wait_a, true);
  mk(m->ev_wait_b, true);
  mk(m->ev_h2d_a, true);
  mk(m->ev_h2d_b, true);
  mk(m->ev_d2h_a, true);
  mk(m->ev_d2h_b, true);
  mk(m->ev_vis_a, true);
  mk(m->ev_vis_b, true);
  for (auto& e : m->ev_stage) MT_CK(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
  MT_CK(cudaEventCreate(&m->ev_t0));
  MT_CK(cudaEventCreate(&m->ev_t1));
  m->rec_ready.assign(nv, 0);
  m->rec_free.assign(nv, 0);
  m->rec_d2h.assign(nv, 0);
  m->rec_h2d_timed.assign(nv, 0);
  m->rec_d2h_timed.assign(nv, 0);
  m->rec_wait_timed.assign(nv, 0);
  m->host_wait_ready_ms.assign(nv, 0.0);
  m->host_wait_gbuf_ms.assign(nv, 0.0);

  // host tiles: pageable, page aligned, zeroed (first touch spread over threads)
  m->tiles.assign(m->layouts.size(), nullptr);
  m->w_loaded.assign(m->layouts.size(), 0);
  m->slab_bytes = std::min<int64_t>(m->cfg.grad_slab_bytes, m->max_w_bytes);
  if (m->cfg.n_replicas >= 2) {
    group_attach(m);
  } else {
    alloc_tiles(m);
  }
  // pinned staging, slabs, scalars, token buffers
  m->stage_bytes = std::min<int64_t>(m->cfg.stage_bytes, m->max_w_bytes);
  for (auto& s : m->stage)
    if (cudaHostAlloc(reinterpret_cast<void**>(&s), (size_t)m->stage_bytes, cudaHostAllocDefault) != cudaSuccess)
      throw MtError{MT_ENOMEM, "pinned staging allocation failed"};
  m->slabs.assign(m->cfg.n_grad_slabs, nullptr);
  m->ev_slab.assign(m->cfg.n_grad_slabs, nullptr);
  for (int i = 0; i < m->cfg.n_grad_slabs; ++i) {
    if (cudaHostAlloc(reinterpret_cast<void**>(&m->slabs[i]), (size_t)m->slab_bytes, cudaHostAllocDefault) !=
        cudaSuccess)
      throw MtError{MT_ENOMEM, "pinned gradient slab allocation failed"};
    MT_CK(cudaEventCreateWithFlags(&m->ev_slab[i], cudaEventDisableTiming));
    m->free_slabs.push_back(i);
  }
  MT_CK(cudaHostAlloc(reinterpret_cast<void**>(&m->pinned_scalars), 256, cudaHostAllocDefault));
  if (m->time_kernels) {
    // one event pair per chunk copy of a step, both directions
    int64_t nh = 0, nd = 0;
    for (const auto& x : m->visits) {
      const int64_t wb = m->layouts[x.tile].w_bytes;
      if (x.h2d) nh += (wb + m->stage_bytes - 1) / m->stage_bytes;
      if (x.grads) {
        const int64_t row_b = 2LL * m->D.d;
        const int64_t rows_chunk = std::max<int64_t>(1, m->slab_bytes / row_b) * row_b;
        nd += x.kind == kEmbedBwd ? (std::min<int64_t>(m->D.T, m->D.V) * row_b + rows_chunk - 1) / rows_chunk
                                  : (wb + m->slab_bytes - 1) / m->slab_bytes;
      }
    }
    m->tl_h2d.assign(2 * nh, nullptr);
    m->tl_d2h.assign(2 * nd, nullptr);
    m->tl_h2d_visit.assign(nh, -1);
    m->tl_d2h_visit.assign(nd, -1);
    for (auto& e : m->tl_h2d) MT_CK(cudaEventCreate(&e));
    for (auto& e : m->tl_d2h) MT_CK(cudaEventCreate(&e));
  }
  if (m->direct_grads || m->direct_weights) {
    // page-lock the sections the DMA engines read (W) or write (G) in place
    m->host_reg.assign(m->tiles.size(), nullptr);
    for (size_t t = 0; t < m->tiles.size(); ++t) {
      const TileLayout& lay = m->layouts[t];
      const int64_t lo = m->direct_weights ? lay.off_w : lay.off_g;
      const int64_t hi = m->direct_grads ? lay.off_m : lay.off_w + lay.w_bytes;
      if (cudaHostRegister(m->tiles[t] + lo, (size_t)(hi - lo), cudaHostRegisterDefault) != cudaSuccess) {
        cudaGetLastError();
        throw MtError{MT_ENOMEM, "could not page-lock tile " + std::to_string(t) + " for direct copies"};
      }
      m->host_reg[t] = m->tiles[t] + lo;
    }
  }
  if (m->direct_grads) {
    m->grad_flags = m->ws.grad_flags;
    MT_CK(cudaHostAlloc(reinterpret_cast<void**>(&m->pinned_flags), sizeof(int) * (3 * m->D.L + 8),
                        cudaHostAllocDefault));
  }
  const size_t ntok = (size_t)(3 * m->D.T + m->D.V + 1 + std::min<int64_t>(m->D.T, m->D.V));
  MT_CK(cudaHostAlloc(reinterpret_cast<void**>(&m->pinned_tok), ntok * sizeof(int32_t), cudaHostAllocDefault));

  // RoPE tables (rotate-half; angle = s * theta^(-2i/hd)), computed in double
  {
    const int half = m->D.hd / 2;
    std::vector<float> c((size_t)m->D.S * half), s((size_t)m->D.S * half);
    for (int p = 0; p < m->D.S; ++p)
      for (int i = 0; i < half; ++i) {
        const double ang = (double)p * std::pow((double)m->cfg.rope_theta, -2.0 * i / m->D.hd);
        c[(size_t)p * half + i] = (float)std::cos(ang);
        s[(size_t)p * half + i] = (float)std::sin(ang);
      }
    MT_CK(cudaMemcpy(m->ws.rope_cos, c.data(), c.size() * 4, cudaMemcpyHostToDevice));
    MT_CK(cudaMemcpy(m->ws.rope_sin, s.data(), s.size() * 4, cudaMemcpyHostToDevice));
  }
  // zero the gradient buffers once (alignment padding is never written)
  for (int b = 0; b < 3; ++b) MT_CK(cudaMemset(m->gbuf[b], 0, (size_t)m->gbuf_bytes[b]));
  MT_CK(cudaDeviceSynchronize());

  // Adam is background work for the step (it only has to finish by its end);
  // packing weights and draining gradient slabs gate the GPU, so they win.
  m->adam_pool.reset(new Pool(m->cfg.n_adam_threads, 10));
  m->pack_pool.reset(new Pool(m->cfg.n_pack_threads));
  m->acc_pool.reset(new Pool(std::max(1, std::min(8, m->cfg.n_adam_threads))));
  m->loader = std::thread(loader_main, m);
  m->d2h = std::thread(d2h_main, m);
  m->accum = std::thread(accum_main, m);
}

}  // namespace
}  // namespace mt

// ====================================================================== C-ABI
using mt::MtError;

extern "C" {

int32_t mt_plan_schedule(int32_t n_layers, int32_t ckpt_every, int32_t keep_layers, uint32_t flags, mt_visit* out,
                         int32_t cap) {
  if (n_layers < 1 || ckpt_every < 1 || keep_layers < 0 || cap < 0) return MT_EINVAL;
  const bool tied = flags & MT_TIE_EMBEDDINGS;
  const int keep_from = (flags & MT_STORE_ACTS) ? 0 : std::max(0, n_layers - keep_layers);
  const auto v = mt::build_schedule(n_layers, ckpt_every, keep_from, flags & MT_NO_DOUBLE_BUFFER,
                                    tied ? 0 : n_layers + 1);
  for (int i = 0; out && i < (int)v.size() && i < cap; ++i) {
    const mt::Visit& x = v[i];
    out[i] = mt_visit{(int32_t)x.kind, x.tile, x.layer, x.buf, x.h2d ? 1 : 0, x.prev_user, x.gbuf, x.prev_gbuf_user};
  }
  return (int32_t)v.size();
}

int64_t mt_required_device_bytes(const mt_config* cfg) {
  if (!cfg) return MT_EINVAL;
  if (const char* e = mt::validate(*cfg)) {
    mt::g_init_error = e;
    return MT_EINVAL;
  }
  mt_model tmp;
  tmp.cfg = mt::with_defaults(*cfg);
  tmp.D = mt::dims_of(tmp.cfg);
  tmp.K = tmp.cfg.ckpt_every;
  tmp.resident_mode = tmp.cfg.flags & MT_RESIDENT;
  tmp.store_acts = tmp.cfg.flags & MT_STORE_ACTS;
  tmp.keep_from = mt::keep_from_of(tmp.cfg);
  mt::build_layouts(&tmp);
  return mt::plan_arena(&tmp, nullptr);
}

int mt_init_model(const mt_config* cfg, void* device_arena, size_t arena_bytes, void* stream_comp, void* stream_h2d,
                  void* stream_d2h, mt_model** out) {
  if (!cfg || !out) {
    mt::g_init_error = "null argument";
    return MT_EINVAL;
  }
  *out = nullptr;
  mt_model* m = new (std::nothrow) mt_model();
  if (!m) return MT_ENOMEM;
  try {
    mt::init_model(m, *cfg, device_arena, arena_bytes, stream_comp, stream_h2d, stream_d2h);
  } catch (const MtError& e) {
    mt::g_init_error = e.msg;
    if (m->grp.h) mt::astore(&m->grp.h->failed, 1);  // the other replicas stop waiting for this one
    mt::destroy(m);
    return e.code;
  } catch (const std::exception& e) {
    mt::g_init_error = e.what();
    if (m->grp.h) mt::astore(&m->grp.h->failed, 1);
    mt::destroy(m);
    return MT_EINTERNAL;
  }
  *out = m;
  return MT_OK;
}

int mt_debug_inject(mt_model* m, int32_t what, int32_t visit) {
  if (!m || what < MT_INJECT_NONE || what > MT_INJECT_LOADER_STALL || visit < 0) return MT_EINVAL;
  m->inject_visit = visit;
  m->inject_what = what;
  return MT_OK;
}

int mt_tile_count(const mt_model* m) { return m ? (int)m->layouts.size() : MT_EINVAL; }

static void fill_tile_desc(const mt::TileLayout& L, mt_tile_desc* out) {
  std::memset(out, 0, sizeof(*out));
  out->kind = L.kind;
  out->n_tensors = (int)L.tensors.size();
  out->n_params = L.n_params;
  out->w_bytes = L.w_bytes;
  out->tile_bytes = L.tile_bytes;
  for (size_t i = 0; i < L.tensors.size() && i < 8; ++i) {
    const auto& t = L.tensors[i];
    std::strncpy(out->tensors[i].name, t.name.c_str(), 15);
    out->tensors[i].ndim = t.ndim;
    out->tensors[i].shape[0] = t.shape[0];
    out->tensors[i].shape[1] = t.shape[1];
    out->tensors[i].offset = t.offset;
    out->tensors[i].numel = t.numel;
  }
}

int mt_tile_info(const mt_model* m, int tile, mt_tile_desc* out) {
  if (!m || !out || tile < 0 || tile >= (int)m->layouts.size()) return MT_EINVAL;
  fill_tile_desc(m->layouts[tile], out);
  return MT_OK;
}

int mt_plan_tile_info(const mt_config* cfg, int tile, mt_tile_desc* out) {
  if (!cfg) {
    mt::g_init_error = "null config";
    return MT_EINVAL;
  }
  if (const char* e = mt::validate(*cfg)) {
    mt::g_init_error = e;
    return MT_EINVAL;
  }
  try {
    mt_model tmp;
    tmp.cfg = mt::with_defaults(*cfg);
    tmp.D = mt::dims_of(tmp.cfg);
    mt::build_layouts(&tmp);
    const int n = (int)tmp.layouts.size();
    if (tile < 0 || tile >= n) {
      mt::g_init_error = "tile index out of range";
      return MT_EINVAL;
    }
    if (out) fill_tile_desc(tmp.layouts[tile], out);
    return n;
  } catch (const std::exception& e) {
    mt::g_init_error = e.what();
    return MT_EINTERNAL;
  }
}

static int part_span(mt_model* m, int tile, int part, size_t nbytes, int64_t* off, int64_t* n) {
  if (!m || tile < 0 || tile >= (int)m->layouts.size()) {
    if (m) m->err = "tile index out of range";
    return MT_EINVAL;
  }
  const auto& L = m->layouts[tile];
  switch (part) {
    case MT_PART_W: *off = L.off_w; *n = L.w_bytes; break;
    case MT_PART_G: *off = L.off_g; *n = L.w_bytes; break;
    case MT_PART_M: *off = L.off_m; *n = L.mv_bytes; break;
    case MT_PART_V: *off = L.off_v; *n = L.mv_bytes; break;
    default: m->err = "bad part"; return MT_EINVAL;
  }
  if ((int64_t)nbytes != *n) {
    m->err = "nbytes must equal the part size " + std::to_string(*n);
    return MT_EINVAL;
  }
  return MT_OK;
}

int mt_load_layer_tile(mt_model* m, int tile, int part, const void* src, size_t nbytes) {
  int64_t off, n;
  if (int rc = part_span(m, tile, part, nbytes, &off, &n)) return rc;
  if (!src) {
    m->err = "null source";
    return MT_EINVAL;
  }
  if (int rc = mt::settle_adam(m, tile, false)) return rc;
  std::memcpy(m->tiles[tile] + off, src, (size_t)n);
  if (part == MT_PART_W) {
    m->w_loaded[tile] = 1;
    if (m->group()) mt::astore(&m->grp.loaded[tile], 1);
  }
  return MT_OK;
}

int mt_get_layer_tile(mt_model* m, int tile, int part, void* dst, size_t nbytes) {
  int64_t off, n;
  if (int rc = part_span(m, tile, part, nbytes, &off, &n)) return rc;
  if (!dst) {
    m->err = "null destination";
    return MT_EINVAL;
  }
  if (int rc = mt::settle_adam(m, tile, false)) return rc;
  std::memcpy(dst, m->tiles[tile] + off, (size_t)n);
  return MT_OK;
}

int mt_train_step(mt_model* m, const int32_t* tokens, size_t n_tokens, float* loss_out) {
  if (!m || !tokens) return MT_EINVAL;
  return mt::run_step(m, tokens, nullptr, n_tokens, loss_out);
}

int mt_train_step_device_tokens(mt_model* m, const int32_t* tokens_dev, size_t n_tokens, float* loss_out) {
  if (!m || !tokens_dev) return MT_EINVAL;
  return mt::run_step(m, nullptr, tokens_dev, n_tokens, loss_out);
}

namespace {
// Entry points whose accumulation or update pattern a replica group does not have.
int refuse_in_group(mt_model* m, const char* what) {
  m->err = std::string(what) + " is not available to a replica of a group (each group step is one mt_train_step "
                               "on every replica)";
  return MT_ESTATE;
}
}  // namespace

int mt_train_step_grads(mt_model* m, const int32_t* tokens, size_t n_tokens, float* loss_out) {
  if (!m || !tokens) return MT_EINVAL;
  if (m->group()) return refuse_in_group(m, "mt_train_step_grads");
  m->grads_only = true;
  const int code = mt::run_step(m, tokens, nullptr, n_tokens, loss_out);
  m->grads_only = false;
  return code;
}

int mt_apply_adam(mt_model* m) {
  using namespace mt;
  if (!m) return MT_EINVAL;
  if (m->group()) return refuse_in_group(m, "mt_apply_adam");
  if (m->broken) {
    m->err = "handle is unusable after an earlier CUDA or internal error: " + m->err;
    return MT_ESTATE;
  }
  if (int rc = settle_adam(m, -1, true)) return rc;
  for (size_t t = 0; t < m->tiles.size(); ++t) submit_adam_range(m, (int)t, 0, m->layouts[t].w_bytes);
  if (!m->adam_pool->wait_idle(m->cfg.timeout_ms)) {
    m->err = "timed out waiting for Adam";
    m->broken = true;
    return MT_ETIMEDOUT;
  }
  m->step += 1;
  return MT_OK;
}

int mt_train_step_micro(mt_model* m, const int32_t* tokens, size_t n_tokens, int32_t n_micro, float* loss_out) {
  if (!m || !tokens || n_micro < 1) return MT_EINVAL;
  if (m->group()) return refuse_in_group(m, "mt_train_step_micro");
  const size_t per = (size_t)m->D.B * (m->D.S + 1);
  if (n_tokens != per * (size_t)n_micro) {
    m->err = "n_tokens must equal n_micro * batch * (seq + 1)";
    return MT_EINVAL;
  }
  mt_step_stats tot{};
  float loss = 0.f;
  int code = MT_OK;
  for (int k = 0; k < n_micro; ++k) {
    m->micro_index = k;
    m->micro_count = n_micro;
    float l = 0.f;
    code = mt::run_step(m, tokens + (size_t)k * per, nullptr, per, &l);
    const mt_step_stats& s = m->stats;
    for (double mt_step_stats::*f : {&mt_step_stats::step_ms, &mt_step_stats::gpu_compute_ms, &mt_step_stats::h2d_ms,
                                     &mt_step_stats::d2h_ms, &mt_step_stats::wait_weights_ms, &mt_step_stats::adam_ms,
                                     &mt_step_stats::gemm_ms, &mt_step_stats::gemm_flops, &mt_step_stats::visit_gap_ms,
                                     &mt_step_stats::host_pre_ms, &mt_step_stats::tail_grads_ms,
                                     &mt_step_stats::tail_adam_ms, &mt_step_stats::tail_rest_ms})
      tot.*f += s.*f;
    for (int64_t mt_step_stats::*f : {&mt_step_stats::gemm_launches, &mt_step_stats::kernel_launches,
                                      &mt_step_stats::h2d_bytes, &mt_step_stats::d2h_bytes,
                                      &mt_step_stats::flops_executed, &mt_step_stats::flops_model})
      tot.*f += s.*f;
    tot.adam_tail_ms = s.adam_tail_ms;
    tot.arena_high_water = s.arena_high_water;
    if (code != MT_OK) break;
    loss += l;
  }
  m->micro_index = 0;
  m->micro_count = 1;
  tot.loss = loss;
  tot.step = m->step;
  m->stats = tot;
  if (loss_out) *loss_out = loss;
  return code;
}

int mt_layer_pass(mt_model* m, int layer, const void* x_in, const void* dx_out, void* x_out, void* dx_in) {
  using namespace mt;
  if (!m) return MT_EINVAL;
  const Dims& D = m->D;
  if (layer < 0 || layer >= D.L || !x_in) {
    m->err = "mt_layer_pass: layer out of range or null x_in";
    return MT_EINVAL;
  }
  if (m->broken) {
    m->err = "handle is unusable after an earlier CUDA or internal error: " + m->err;
    return MT_ESTATE;
  }
  const int tile = layer + 1;
  if (int rc = settle_adam(m, tile, true)) return rc;
  if (!m->w_loaded[tile]) {
    m->err = "tile " + std::to_string(tile) + " has no weights loaded";
    return MT_ESTATE;
  }
  int code = MT_OK;
  try {
    MT_CK(cudaSetDevice(m->device));
    const TileLayout& lay = m->layouts[tile];
    uint8_t* wb = m->resident_mode ? m->resident + m->resident_off[tile] : m->wbuf[0];
    MT_CK(cudaMemsetAsync(m->ws.status, 0, sizeof(int), m->s_comp));
    MT_CK(cudaMemcpyAsync(wb, m->tiles[tile] + lay.off_w, (size_t)lay.w_bytes, cudaMemcpyHostToDevice, m->s_comp));
    LaunchStats ls;
    LayerTemplate tmpl{D, m->cfg.rms_eps, m->s_comp, &m->ws, &ls};
    LayerActs a = layer >= m->keep_from ? m->stored[layer - m->keep_from] : m->acts;
    a.x = reinterpret_cast<bf16*>(const_cast<void*>(x_in));
    int rc = tmpl.forward(bind_layer(lay, wb), a, reinterpret_cast<bf16*>(x_out), dx_out != nullptr);
    if (dx_out) {
      bf16* dxi = dx_in ? reinterpret_cast<bf16*>(dx_in) : m->ws.dx_b;
      rc |= tmpl.backward(bind_layer(lay, wb), a, reinterpret_cast<const bf16*>(dx_out), dxi,
                          bind_layer(lay, m->gbuf[0]));
    }
    if (rc != 0) throw MtError{MT_ECUDA, std::string("kernel launch failed: ") + last_launch_error()};
    // bounded wait for the kernels, then plain copies of the results
    MT_CK(cudaEventRecord(m->ev_t1, m->s_comp));
    wait_event(m, m->ev_t1, "layer pass");
    MT_CK(cudaStreamSynchronize(m->s_comp));
    int st = 0;
    MT_CK(cudaMemcpy(&st, m->ws.status, sizeof(int), cudaMemcpyDeviceToHost));
    if (dx_out && st == 0)
      MT_CK(cudaMemcpy(m->tiles[tile] + lay.off_g, m->gbuf[0], (size_t)lay.w_bytes, cudaMemcpyDeviceToHost));
    if (st != 0) {
      if (st == kStatusNonFinite) throw MtError{MT_ENONFINITE, "non-finite value in the layer pass"};
      throw MtError{MT_ETIMEDOUT, "device status " + std::to_string(st) + " in the layer pass"};
    }
  } catch (const MtError& e) {
    m->err = e.msg;
    code = e.code;
    if (!drain_stream(m->s_comp, m->cfg.timeout_ms)) {
      m->err += " (compute stream did not drain within the timeout)";
      m->undrained = true;
    }
    if (code != MT_EINVAL && code != MT_ENONFINITE) m->broken = true;
  }
  return code;
}

int mt_get_step_stats(const mt_model* m, mt_step_stats* out) {
  if (!m || !out) return MT_EINVAL;
  *out = m->stats;
  return MT_OK;
}

int64_t mt_get_step(const mt_model* m) { return m ? m->step : MT_EINVAL; }

int mt_replica_barrier(mt_model* m) {
  using namespace mt;
  if (!m) return MT_EINVAL;
  if (!m->group()) return MT_OK;
  try {
    const int64_t k = ++m->grp.barriers;
    GroupHeader* h = m->grp.h;
    aadd(&h->barrier_count, (int64_t)1);
    group_wait(m, [&] { return aload(&h->barrier_count) >= k * m->grp.n; }, "every replica to reach the barrier");
  } catch (const MtError& e) {
    m->err = e.msg;
    return e.code;
  }
  return MT_OK;
}

int mt_set_step(mt_model* m, int64_t step) {
  if (!m || step < 0) return MT_EINVAL;
  if (int rc = mt::settle_adam(m, -1, false)) return rc;
  m->step = step;
  return MT_OK;
}

int64_t mt_get_timeline(const mt_model* m, mt_interval* out, int64_t cap) {
  if (!m || cap < 0) return MT_EINVAL;
  if (!m->time_kernels) return 0;
  std::vector<mt_interval> iv;
  auto add = [&](int32_t kind, int32_t visit, cudaEvent_t a, cudaEvent_t b) {
    float t0 = 0.f, t1 = 0.f;
    if (cudaEventElapsedTime(&t0, m->ev_t0, a) == cudaSuccess && cudaEventElapsedTime(&t1, m->ev_t0, b) == cudaSuccess)
      iv.push_back(mt_interval{kind, visit, (double)t0, (double)t1});
    else
      cudaGetLastError();
  };
  for (int v = 0; v < (int)m->visits.size(); ++v) add(MT_SPAN_COMPUTE, v, m->ev_vis_a[v], m->ev_vis_b[v]);
  for (int k = 0; k < m->tl_h2d_n; ++k) add(MT_SPAN_H2D, m->tl_h2d_visit[k], m->tl_h2d[2 * k], m->tl_h2d[2 * k + 1]);
  const int nd = std::min<int>(m->tl_d2h_n.load(), (int)m->tl_d2h_visit.size());
  for (int k = 0; k < nd; ++k) add(MT_SPAN_D2H, m->tl_d2h_visit[k], m->tl_d2h[2 * k], m->tl_d2h[2 * k + 1]);
  for (int64_t i = 0; out && i < (int64_t)iv.size() && i < cap; ++i) out[i] = iv[i];
  return (int64_t)iv.size();
}

int mt_sync(mt_model* m) {
  if (!m) return MT_EINVAL;
  return mt::settle_adam(m, -1, true);
}

const char* mt_last_error(const mt_model* m) { return m ? m->err.c_str() : mt::g_init_error.c_str(); }

void mt_free(mt_model* m) { mt::destroy(m); }

}  // extern "C"
