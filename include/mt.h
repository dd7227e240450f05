/*
 * mt.h -- C-ABI of libmt.so: one layer-streamed decoder training step on one
 * GPU with the host as the authoritative store (MegaTrain).
 *
 * Where each operation comes from (page titles of the MegaTrain sources):
 *  - host memory holds all persistent state; the GPU is a transient compute
 *    engine: paperlayer.ai summary "MegaTrain: Full Precision Training of
 *    100B+ Parameter Large Language Models on a Single GPU", Abstract and §3
 *    "Execution workflow";
 *  - one contiguous 4 KB-aligned tile per layer holding BF16 weights, BF16
 *    gradients and FP32 Adam moments (12 bytes/parameter): paperlayer.ai §2
 *    "Training memory", §A.1 "Layer-Contiguous Tiling"; hyper.ai summary,
 *    方法 (Method) ¶5;
 *  - streaming through two device buffers on three CUDA streams ordered by
 *    Weights-Ready / Buffer-Free / Grads-Done events, a CPU packer thread
 *    filling pinned staging buffers, gradient slabs with a background
 *    accumulator: paperlayer.ai §A.2, §A.3; hyper.ai 方法 ¶3-5;
 *  - stateless layer templates bound to streamed buffers (Bind):
 *    paperlayer.ai §A.4; hyper.ai 方法 ¶6;
 *  - block checkpoints and recompute in backward: paperlayer.ai §3; hyper.ai
 *    方法 ¶2; author's blog "How to Train 100B+ Large Models on a Single GPU",
 *    the F/W/G block figure;
 *  - Adam on CPU threads: paperlayer.ai §3 "Execution workflow", §A.
 *
 * Conventions
 *  - Tiles: index 0 = embedding (E [V, d]), 1..L = decoder layers,
 *    L+1 = head (final RMSNorm gain g_f [d], LM head W_h [V, d]).
 *  - Each tile is one page-aligned host block with four sections in this
 *    order: W (BF16), G (BF16), M (FP32), V (FP32); each section starts on a
 *    4096-byte boundary.  Inside W (and identically inside G) the tensors of
 *    the tile follow in the order given by mt_tile_info, each on a 256-byte
 *    boundary.  M and V hold one FP32 per parameter in the same order and
 *    offsets x2.
 *  - Layer tile tensors: g1 [d], wqkv [(Hq+2Hkv)*hd, d] (rows: all q heads,
 *    then k heads, then v heads), wo [d, Hq*hd], g2 [d], wgu [2f, d] whose row
 *    2j is gate row j and row 2j+1 is up row j, wd [d, f].  Matrices are
 *    nn.Linear [out, in], row-major.
 *  - Tokens: int32 [B, S+1]; row b trains on inputs tokens[b, :S] and targets
 *    tokens[b, 1:]; the loss is the mean over the B*S targets.
 *
 * Ownership: the caller owns every pointer it passes (config, tokens, src,
 * dst, device arena, streams) and keeps the arena and streams alive until
 * mt_free.  The library copies what it needs and keeps no caller pointer
 * except the arena and the streams.  The library owns the host tiles, the
 * pinned staging buffers, the gradient slabs, its events and its threads.
 *
 * Errors: every call returns 0 (MT_OK) or a negative MT_E* code; the text is
 * in mt_last_error(handle) (or mt_last_error(NULL) for failures before a
 * handle exists).  No C++ exception crosses this boundary.  After MT_ECUDA or
 * MT_EINTERNAL the handle accepts only mt_get_layer_tile, mt_last_error and
 * mt_free.
 */
#ifndef MT_H
#define MT_H
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  MT_OK = 0,
  MT_EINVAL = -1,      /* bad config, size, tile index or argument */
  MT_ENOMEM = -2,      /* host allocation / pinning failed, or the arena is too small */
  MT_ECUDA = -3,       /* a CUDA call failed */
  MT_ETIMEDOUT = -4,   /* a bounded wait (host event poll or device mbarrier) expired */
  MT_ESTATE = -5,      /* call not allowed in the handle's state */
  MT_ENONFINITE = -6,  /* the loss or a gradient is NaN/Inf: Adam is not applied to any gradient chunk
                          that lands after the first non-finite value is seen; a non-finite loss is seen
                          before any gradient lands, so then no weight is updated */
  MT_EINTERNAL = -7    /* a worker thread failed */
};

/* mt_config.flags */
enum {
  MT_RESIDENT = 1u << 0,          /* upload every tile's W once; no streaming (test path) */
  MT_STORE_ACTS = 1u << 1,        /* keep every layer's internals from forward; no recompute (keep_layers =
                                     n_layers) */
  MT_NO_DOUBLE_BUFFER = 1u << 2,  /* one device weight buffer: no H2D/compute overlap (ablation) */
  MT_DEBUG_CHECKS = 1u << 3,      /* NaN/Inf scan of every gradient tile; host event-order asserts */
  MT_TIME_KERNELS = 1u << 4,      /* CUDA-event timing of every GEMM launch (mt_get_step_stats) */
  MT_TRACE = 1u << 5,             /* debugging: wait for every visit (layer pass) to finish, print its kind,
                                     layer, time and the device status word to stderr, stop at the first
                                     nonzero status */
  MT_VISIT_LOG = 1u << 6,         /* after each step print one line per visit to stderr: the compute-stream
                                     gap before it, its compute-stream time, and how long the stream and the
                                     issuing host thread waited for its weights and its gradient buffer */
  MT_ASYNC_ADAM = 1u << 8,        /* mt_train_step returns once the step's gradients have landed in their tiles
                                     and leaves the Adam updates still running on the CPU workers; each
                                     tile's update finishes before the next step uploads that tile and
                                     before any call reads or writes it (mt_get_layer_tile,
                                     mt_load_layer_tile, mt_layer_pass, mt_apply_adam, mt_set_step;
                                     mt_sync waits for all).  Updates run lowest tile first, the order in
                                     which the next step needs them, so the host's memory bandwidth, which
                                     the backward's gradient traffic saturates, finishes the updates of the
                                     upper layers during the next forward (paperlayer.ai summary §3: CPU
                                     updates run concurrently with the GPU).  The results are those of the
                                     synchronous step, bit for bit. */
  MT_DIRECT_GRADS = 1u << 9,      /* gradient chunks of the first (or only) micro-batch land straight in the
                                     tiles' G sections, which mt_init_model page-locks, instead of passing
                                     through the pinned slabs and the accumulator's copy: half the host
                                     memory traffic of the gradient path, and no host copy between the D2H
                                     stream and the device gradient buffers' reuse.  A device check flags
                                     non-finite gradients per visit (the slab path checks on the host).
                                     Later micro-batches and the embedding rows keep the slab path. */
  MT_DIRECT_WEIGHTS = 1u << 10,   /* each upload's DMA reads the tile's W section in place, which
                                     mt_init_model page-locks, instead of a packer copy into the two
                                     pinned staging chunks followed by their DMA: a third of the host
                                     memory traffic of the weight path, and no host thread on it.  The
                                     tile's bytes must not change while its copy is queued, which the
                                     step already guarantees (its Adam update finishes before the
                                     upload is enqueued, MT_ASYNC_ADAM included).  With MT_DIRECT_GRADS
                                     the W and G sections are page-locked as one range per tile. */
  MT_TIE_EMBEDDINGS = 1u << 7     /* the LM head's weight is the embedding table E (paperlayer.ai summary
                                     §A.1, tied embeddings: one shared host region, update readiness
                                     tracked).  Tile 0 holds E and the final norm gain gf; there is no head
                                     tile (mt_tile_count = L + 1).  The head's visit streams tile 0 and binds
                                     W_h to its E (one device address); its dense dW_h lands in tile 0's G and
                                     the embedding rows' gradient is added to it.  E's rows that no token of
                                     the step uses are updated once the head's gradient has landed, the rest
                                     once their embedding gradient has been added. */
};

/* Tile parts for load/get. */
enum { MT_PART_W = 0, MT_PART_G = 1, MT_PART_M = 2, MT_PART_V = 3 };

typedef struct {
  int32_t n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn, vocab;
  float rms_eps, rope_theta; /* 1e-5, 1e4 */
  int32_t batch, seq;        /* tokens per step = batch * seq */
  int32_t ckpt_every;        /* K: keep the input of every K-th layer; recompute inside blocks of K */
  float lr, beta1, beta2, adam_eps, weight_decay;
  int32_t n_adam_threads;    /* CPU Adam workers (0 = 3/4 of the hardware threads) */
  int32_t n_pack_threads;    /* CPU threads copying pageable tiles into pinned staging (0 = 8) */
  int32_t n_grad_slabs;      /* pinned gradient slabs (0 = 24) */
  int64_t grad_slab_bytes;   /* bytes per gradient slab (0 = 64 MiB) */
  int64_t stage_bytes;       /* bytes per pinned H2D staging chunk (0 = 64 MiB); two chunks ping-pong */
  int64_t timeout_ms;        /* bound of every host wait (0 = 60000) */
  uint32_t flags;
  int64_t mlp_chunk_rows;    /* run the MLP (gate/up, SwiGLU, down and their backward) over row chunks of
                                this many tokens, a multiple of 128, so that its [tokens, 2 ffn]
                                activations exist one chunk at a time (long sequences); the W_gu and W_d
                                gradients then accumulate in FP32 across chunks.  0 = the whole step at
                                once.  Not combinable with MT_STORE_ACTS. */
  int32_t n_experts;         /* 0: dense decoder layers.  > 0: every layer's MLP is a top-k mixture of
                                n_experts SwiGLU experts of width ffn (a multiple of 8, at most 256):
                                router logits x W_r^T, per token the top_k largest (ties to the lower
                                expert id), gates = softmax over them, output = the gate-weighted sum of
                                the chosen experts.  A layer tile then holds g1, wqkv, wo, g2, wr
                                [n_experts, d], wgu [n_experts * 2 ffn, d] (each expert's gate/up rows
                                interleaved) and wd [n_experts * d, ffn].  Not combinable with
                                mlp_chunk_rows. */
  int32_t top_k;             /* experts per token (1 .. min(8, n_experts)); ignored when n_experts = 0 */
  int32_t keep_layers;       /* the last keep_layers decoder layers keep their internals (normalised
                                inputs, q/k/v, attention output and log-sum-exp, residual, gate/up and
                                SwiGLU activations) in device memory from their forward to their
                                backward, so their backward visits recompute nothing; the other layers
                                follow the ckpt_every block schedule.  Checkpointing trades device memory
                                for recompute (hyper.ai summary, 实验 ablation: checkpoint interval 1
                                cuts the largest batch 96 -> 32); a device with the memory for every
                                layer's internals needs no recompute.  0 = every layer recomputed;
                                >= n_layers = every layer kept (as MT_STORE_ACTS).  Each kept layer adds
                                its stored set to mt_required_device_bytes.  Not combinable with
                                mlp_chunk_rows. */
  int32_t replica_rank;      /* replica group: this process's rank, 0 .. n_replicas - 1 */
  int32_t n_replicas;        /* 0 or 1: a model of its own.  2 .. 64: one of n_replicas data-parallel
                                replicas of ONE model, one process per GPU, each training on its own
                                batch of batch x seq tokens (the future multi-GPU work of the MegaTrain
                                pages: author's blog, planned projects).  The replicas map one
                                shared-memory segment (replica_name) that holds every host tile, so W,
                                M and V exist once on the host.  Each replica streams the weights from
                                it; its gradient chunks are summed into the shared G in rank order,
                                replica r adding a chunk once replicas 0 .. r-1 have added theirs, with
                                each replica's cross-entropy scaled by 1 / n_replicas: the additions of
                                mt_train_step_micro with micro-batch r = replica r, so the result is that
                                call's bit for bit.  The last replica runs Adam on each chunk as it
                                completes (paperlayer.ai summary §A.3: a background accumulator drains
                                the gradient slabs and the CPU update overlaps the backward); every
                                replica's next upload of a tile waits for its update.  mt_train_step
                                returns the loss of the global batch (every replica's mean, averaged)
                                on every replica, after all have finished the step, and MT_ENONFINITE on
                                every replica if any saw a non-finite value.  Every replica calls
                                mt_init_model with the same config apart from replica_rank;
                                mt_init_model returns once all have attached.  Tiles are written
                                (mt_load_layer_tile) by one replica while no step runs, and read
                                (mt_get_layer_tile) while no replica runs a step: the replicas meet at
                                mt_replica_barrier.  A failure on
                                one replica makes the others' waits fail (MT_EINTERNAL) and leaves every
                                handle of the group unusable.  Not combinable with MT_RESIDENT or
                                MT_TIE_EMBEDDINGS; mt_train_step_micro, mt_train_step_grads and
                                mt_apply_adam return MT_ESTATE. */
  char replica_name[48];     /* the group's shared-memory name (letters, digits, '_', '-', '.'; NUL
                                terminated), new for each group: replica 0 creates the segment and
                                removes the name once every replica has attached */
} mt_config;

typedef struct mt_model mt_model;

typedef struct {
  char name[16];
  int32_t ndim;
  int64_t shape[2];
  int64_t offset; /* byte offset inside the W (or G) section */
  int64_t numel;
} mt_tensor_desc;

typedef struct {
  int32_t kind;      /* 0 embed, 1 layer, 2 head */
  int32_t n_tensors;
  int64_t n_params;
  int64_t w_bytes;   /* bytes of the W section (== G section); M, V sections are 2x */
  int64_t tile_bytes;/* whole host tile */
  mt_tensor_desc tensors[8];
} mt_tile_desc;

typedef struct {
  double loss;
  double step_ms;          /* host wall time of mt_train_step */
  double gpu_compute_ms;   /* compute-stream time between the first and last event of the step */
  double h2d_ms, d2h_ms;   /* summed copy time on the H2D / D2H streams (events) */
  double wait_weights_ms;  /* compute-stream time spent waiting for Weights-Ready */
  double adam_ms;          /* summed wall time of Adam tasks (all workers) */
  double adam_tail_ms;     /* wall time from the last Grads-Done to the end of Adam */
  double gemm_ms;          /* summed GEMM kernel time (MT_TIME_KERNELS) */
  double gemm_flops;       /* FLOPs of those GEMM launches */
  int64_t gemm_launches;
  int64_t kernel_launches; /* kernels launched by the step */
  int64_t h2d_bytes, d2h_bytes;
  int64_t flops_executed;  /* matmul FLOPs of the schedule: forward visits and boundary recomputes in full,
                              each backward visit's internal recompute without the down projection, each
                              layer's backward at 2x its forward, the head's forward + backward once */
  int64_t flops_model;     /* 6 * N_linear * T + causal-attention FLOPs (3x forward) */
  int64_t arena_high_water;
  int64_t step;            /* Adam step counter after this step */
  double visit_gap_ms;     /* compute-stream time between the end of one visit's kernels and the start of
                              the next one's: stream waits plus idle time while the host was behind */
  double host_pre_ms;      /* host wall time from the call to the first compute-stream event */
  double tail_grads_ms;    /* from the compute stream's end to the last gradient landing in its tile */
  double tail_adam_ms;     /* from there to the end of the last Adam task */
  double tail_rest_ms;     /* from there to the return (stream drains, statistics) */
} mt_step_stats;

/* Device bytes the handle needs in its arena for this config (>0), or a negative MT_E* code. */
int64_t mt_required_device_bytes(const mt_config* cfg);

/*
 * Host tile layout of this config without a handle (no GPU involved), to size
 * host memory before mt_init_model: fills *out (if not NULL) with the
 * description mt_tile_info gives for tile `tile` once the handle exists, and
 * returns the number of tiles (> 0).  The tile store is the pages' 12 bytes
 * per parameter (BF16 W and G, FP32 M and V) plus section and sub-tensor
 * alignment (paperlayer.ai §2 "Training memory", §A.1 "Layer-Contiguous
 * Tiling").  MT_EINVAL for an invalid config or a tile index outside
 * [0, tiles); the text is in mt_last_error(NULL).
 */
int mt_plan_tile_info(const mt_config* cfg, int tile, mt_tile_desc* out);

/*
 * Create a handle.  device_arena: a device allocation of at least
 * mt_required_device_bytes(cfg) bytes, 256-byte aligned; stream_*:
 * cudaStream_t values (compute, host-to-device, device-to-host), distinct and
 * non-blocking w.r.t. each other.  Allocates the host tiles (zeroed), the
 * pinned staging buffers and gradient slabs, starts the worker threads.
 * Every tile's W must be loaded (mt_load_layer_tile, part W) before the
 * first mt_train_step.
 */
int mt_init_model(const mt_config* cfg, void* device_arena, size_t arena_bytes, void* stream_comp,
                  void* stream_h2d, void* stream_d2h, mt_model** out);

/* One visit of the streamed schedule (mt_plan_schedule). */
enum {
  MT_VISIT_EMBED_FWD = 0, /* embedding forward (tile 0) */
  MT_VISIT_LAYER_FWD = 1, /* layer forward; x_i kept when i % ckpt_every == 0 */
  MT_VISIT_HEAD = 2,      /* final norm + LM head + cross-entropy, forward and backward */
  MT_VISIT_RECOMPUTE = 3, /* layer forward again inside a checkpoint block (backward pass) */
  MT_VISIT_LAYER_BWD = 4, /* layer backward (its internals recomputed from x_i in the same visit unless the
                             layer keeps them from its forward) */
  MT_VISIT_EMBED_BWD = 5  /* embedding gradient rows (no weights needed on the device) */
};
typedef struct {
  int32_t kind;      /* MT_VISIT_* */
  int32_t tile;      /* host tile whose weights the visit binds */
  int32_t layer;     /* decoder layer, -1 for the embedding and the head */
  int32_t buf;       /* device weight buffer (0 or 1), -1 for none */
  int32_t h2d;       /* 1: the tile streams into buf before the visit; 0: buf still holds it */
  int32_t buf_wait;  /* previous visit that used buf (the copy waits for its Buffer-Free event), -1 none */
  int32_t gbuf;      /* device gradient buffer (layers alternate 0 and 1; head and embedding 2), -1 none */
  int32_t gbuf_wait; /* previous visit that used gbuf (its gradients must have left first), -1 none */
} mt_visit;

/*
 * The visit order one mt_train_step runs for n_layers decoder layers,
 * checkpoint interval ckpt_every (K), keep_layers (mt_config.keep_layers) and
 * flags (MT_STORE_ACTS, MT_NO_DOUBLE_BUFFER and MT_TIE_EMBEDDINGS matter;
 * MT_RESIDENT models use the same order with every tile resident).  Host
 * only, no handle: the forward visits every layer in order, the head
 * follows, then the kept layers' backward visits (last layer first), then
 * the remaining layers' checkpoint blocks in reverse (per block [s, e):
 * layers s .. e-2 recomputed, then layers e-1 .. s backward), then the
 * embedding gradient (MegaTrain paperlayer.ai summary, §3 "Execution
 * workflow" and §A.3 "Block-wise recomputation").  A tile still held by one
 * of the two buffers is not streamed again.  Writes at most cap visits to out
 * (out may be NULL) and returns the number of visits, or MT_EINVAL for
 * n_layers < 1, ckpt_every < 1, keep_layers < 0 or cap < 0.
 */
int32_t mt_plan_schedule(int32_t n_layers, int32_t ckpt_every, int32_t keep_layers, uint32_t flags, mt_visit* out,
                         int32_t cap);

/*
 * Host-side fault injection, for tests of failure detection that fault no
 * GPU.  The next mt_train_step fails in the named host component at the
 * first visit >= `visit` that the component works on:
 *   MT_INJECT_LOADER_FAIL  the loader thread reports an error instead of
 *                          streaming that visit's tile;
 *   MT_INJECT_D2H_FAIL     the D2H thread reports an error instead of
 *                          evacuating that visit's gradients;
 *   MT_INJECT_ACCUM_FAIL   the accumulator reports an error on that visit's
 *                          first gradient slab;
 *   MT_INJECT_ADAM_FAIL    an Adam task of that visit's tile reports an error
 *                          instead of updating;
 *   MT_INJECT_LOADER_STALL the loader stops before that visit's copy without
 *                          an error, so the compute thread's bounded wait for
 *                          Weights-Ready runs out (MT_ETIMEDOUT after
 *                          timeout_ms); the loader resumes its wait for the
 *                          next step once the step has aborted.
 * The failures return MT_EINTERNAL with "injected" in mt_last_error.  As after
 * any such error, the handle then accepts only mt_get_layer_tile and
 * mt_free.  Returns MT_EINVAL for an unknown kind or a negative visit.
 */
enum {
  MT_INJECT_NONE = 0,
  MT_INJECT_LOADER_FAIL = 1,
  MT_INJECT_D2H_FAIL = 2,
  MT_INJECT_ACCUM_FAIL = 3,
  MT_INJECT_ADAM_FAIL = 4,
  MT_INJECT_LOADER_STALL = 5
};
int mt_debug_inject(mt_model* m, int32_t what, int32_t visit);

int mt_tile_count(const mt_model* m);                                /* L + 2 (L + 1 with MT_TIE_EMBEDDINGS) */
int mt_tile_info(const mt_model* m, int tile, mt_tile_desc* out);

/*
 * Copy nbytes from host memory `src` into part `part` of tile `tile`;
 * nbytes must equal the part's size (w_bytes for W and G, 2*w_bytes for M
 * and V) in the tile's internal layout (see Conventions).
 */
int mt_load_layer_tile(mt_model* m, int tile, int part, const void* src, size_t nbytes);

/*
 * One synchronous training step: forward, backward with block recompute,
 * gradient evacuation, and Adam on every tile.  tokens: host int32
 * [batch, seq+1] (n_tokens = batch*(seq+1)); or, with tokens_on_device = 1,
 * a device pointer to the same array.  On success *loss_out holds the mean
 * cross-entropy of the step (computed before the update).
 */
int mt_train_step(mt_model* m, const int32_t* tokens, size_t n_tokens, float* loss_out);
int mt_train_step_device_tokens(mt_model* m, const int32_t* tokens_dev, size_t n_tokens, float* loss_out);

/*
 * One training step over n_micro micro-batches (gradient accumulation): host
 * int32 tokens [n_micro, batch, seq+1] (n_tokens = n_micro*batch*(seq+1)).
 * Each micro-batch is a full streamed forward/backward pass; the gradient of
 * the mean loss over all n_micro*batch*seq targets accumulates in the host
 * tiles' G sections (BF16, the first pass writes, later passes add), and Adam
 * runs once, as the last pass's gradients land.  *loss_out: the mean loss.
 * n_micro = 1 is mt_train_step.  The step statistics sum over the passes.
 * Errors as mt_train_step; a non-finite loss or gradient stops the step
 * before any weight is updated.
 */
int mt_train_step_micro(mt_model* m, const int32_t* tokens, size_t n_tokens, int32_t n_micro, float* loss_out);

/*
 * Data-parallel replicas (one handle per GPU, each on its own batch) combine
 * their gradients on the host between these two calls.  The pages leave
 * several GPUs as future work (engineersofai.com breakdown, limitations;
 * author's blog, planned projects: single-machine multi-GPU training); this
 * is the host-side gradient average that needs no device collective:
 *
 * mt_train_step_grads: mt_train_step without the optimizer.  Afterwards every
 * tile's G section holds the BF16 gradient of the mean loss over this batch's
 * batch*seq targets (embedding rows of token ids the batch does not use are
 * zero); weights, moments and the step counter are unchanged.  Arguments and
 * errors as mt_train_step.
 *
 * mt_apply_adam: one Adam step of every tile from its G section as it stands
 * (left by mt_train_step_grads or replaced through mt_load_layer_tile, part
 * G), with step counter t + 1, on the host Adam workers; returns when every
 * tile is updated, then advances the counter.  The caller checks that the
 * gradients are finite.  MT_ESTATE on a handle that saw MT_ECUDA, MT_EINTERNAL
 * or MT_ETIMEDOUT; MT_ETIMEDOUT when the workers do not finish within
 * timeout_ms.
 */
int mt_train_step_grads(mt_model* m, const int32_t* tokens, size_t n_tokens, float* loss_out);
int mt_apply_adam(mt_model* m);

/*
 * Per-layer check at the workload's full shape (a debugging hook for parity
 * tests): run decoder layer `layer` (0-based; tile layer + 1) forward and
 * backward once on caller-supplied activations, with the same template,
 * kernels and launch shapes as a training step.
 *   x_in    device BF16 [batch*seq, d_model], row-major: the layer input x_j
 *   dx_out  device BF16 [batch*seq, d_model]: dL/dx_{j+1}; NULL = forward only
 *   x_out   device BF16 [batch*seq, d_model]: receives x_{j+1}; may be NULL
 *   dx_in   device BF16 [batch*seq, d_model]: receives dL/dx_j; may be NULL
 * The layer's weight gradient (BF16, tile layout) replaces the G section of
 * the host tile (read it back with mt_get_layer_tile, part G).  Adam does not
 * run and the step counter does not change.  The four buffers are owned by
 * the caller, must not overlap, and stay untouched after return.
 * Synchronous on the compute stream.  Errors: MT_EINVAL (bad layer index or
 * null x_in), MT_ESTATE (weights not loaded, or the handle is unusable),
 * MT_ETIMEDOUT (a device-side bounded wait expired), MT_ECUDA.
 */
int mt_layer_pass(mt_model* m, int layer, const void* x_in, const void* dx_out, void* x_out, void* dx_in);

/* Copy part `part` of tile `tile` into host memory `dst` (nbytes as in load). */
int mt_get_layer_tile(mt_model* m, int tile, int part, void* dst, size_t nbytes);

int mt_get_step_stats(const mt_model* m, mt_step_stats* out);

/*
 * Device timeline of the last step (MT_TIME_KERNELS; 0 intervals otherwise):
 * each visit's compute-stream span and every chunk copy on the H2D and D2H
 * streams, in milliseconds from the step's first compute-stream event (a copy
 * issued before it may start slightly earlier, i.e. at a negative time).
 * Writes at most cap intervals to out (out may be NULL) and returns the count.
 */
enum { MT_SPAN_COMPUTE = 0, MT_SPAN_H2D = 1, MT_SPAN_D2H = 2 };
typedef struct {
  int32_t kind;   /* MT_SPAN_* */
  int32_t visit;  /* the visit the span belongs to (mt_plan_schedule order) */
  double t0_ms, t1_ms;
} mt_interval;
int64_t mt_get_timeline(const mt_model* m, mt_interval* out, int64_t cap);

/*
 * Wait until every Adam update of the steps run so far has finished
 * (MT_ASYNC_ADAM; returns at once otherwise).  Returns the error of an
 * update that failed after its step had returned, else MT_OK.
 */
int mt_sync(mt_model* m);
int64_t mt_get_step(const mt_model* m);       /* Adam step counter t (0 before the first step) */
int mt_set_step(mt_model* m, int64_t step);  /* for resume */

/*
 * Replica group (mt_config.n_replicas >= 2): return once every replica of the
 * group has called mt_replica_barrier as many times as this one (bounded by
 * timeout_ms; MT_EINTERNAL at once if another replica has failed).  Used
 * between one replica's mt_load_layer_tile calls and the group's first step.
 * Returns MT_OK at once for a handle that is not in a group.
 */
int mt_replica_barrier(mt_model* m);

const char* mt_last_error(const mt_model* m);
void mt_free(mt_model* m);

/*
 * Host-only Adam on one tile-shaped range (used by the step's CPU workers;
 * exported for checking against the oracle without a GPU).
 * w, g: BF16 bit patterns (uint16); m, v: FP32; n elements; t >= 1.
 * m <- b1 m + (1-b1) g; v <- b2 v + (1-b2) g^2;
 * w <- bf16_rne(w - lr (m/(1-b1^t)) / (sqrt(v/(1-b2^t)) + eps) - lr wd w),
 * arithmetic in FP32.
 */
int mt_adam_host(uint16_t* w, const uint16_t* g, float* m, float* v, size_t n, int64_t t, float lr, float beta1,
                 float beta2, float eps, float weight_decay);

#ifdef __cplusplus
}
#endif
#endif
