/*
 * mt.h -- C ABI of libmt: the layer-streamed, host-memory-centric training step
 * of a decoder-only transformer on one GPU (GB300, sm_103a).
 *
 * The method (MegaTrain, as described on the pages cited below) keeps every
 * parameter, gradient, FP32 master weight and Adam moment in host RAM as one
 * contiguous block per layer, and treats the GPU as a transient compute
 * engine: each block's BF16 weights stream host-to-device into one of two
 * ping-pong device buffers, are bound to a weight-less layer template, run
 * forward (and later recompute + backward), and the block's BF16 gradients
 * stream device-to-host into one of K pinned slabs, where host threads apply
 * mixed-precision Adam.  Three CUDA streams (compute, weight, gradient) are
 * ordered only by three events: Weights-Ready, Backward-Done, Buffer-Free.
 *
 * Sources, cited by page and section:
 *   [Review]  dimensionstp.github.io, "MegaTrain: Full Precision Training of
 *             100B+ Parameter Large Language Models on a Single GPU Review",
 *             3-2 Module breakdown (1)-(6)
 *   [Hotdry]  blog.hotdry.top (2026-04-09), sections on the host memory layout
 *             (flat tensors, pinned staging), the three CUDA streams and double
 *             buffering, and the event-driven synchronisation protocol
 *   [Lilting] lilting.ch, "MegaTrainはシングルGPUで120BパラメータLLMをフル精度
 *             訓練する", sections on the memory breakdown, the pipelined double
 *             buffering and the stateless layer templates
 *   [Peter]   peter-blog.pages.dev, MegaTrain translation, 技術細節 (CUDA stream
 *             management, static prefetch schedule)
 *
 * Conventions for every call:
 *   - returns an mt_status; no exception crosses the ABI;
 *   - a CUDA error maps to MT_ERR_CUDA with cudaGetErrorString text available
 *     from mt_last_error(); any timeout or CUDA error latches the model into an
 *     error state in which every call except mt_last_error / mt_destroy
 *     returns MT_ERR_STATE;
 *   - one driver thread per model; the library's host workers are internal;
 *   - "device pointer" arguments are CUDA device addresses the caller owns;
 *     "stream" arguments are cudaStream_t values passed as void*.
 */
#ifndef MT_H
#define MT_H
#include <stddef.h>
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MT_OK = 0,
  MT_ERR_ARG = -1,       /* bad argument (shape, alignment, index, null)      */
  MT_ERR_STATE = -2,     /* call out of order, or model latched in error       */
  MT_ERR_HOST_OOM = -3,  /* host (pageable or pinned) allocation failed        */
  MT_ERR_CUDA = -4,      /* a CUDA runtime call or kernel launch failed        */
  MT_ERR_TIMEOUT = -5,   /* a bounded host wait (event, slab, Adam) expired    */
  MT_ERR_INTERNAL = -6,  /* a host worker failed                               */
  MT_ERR_DEVICE_OOM = -7 /* the caller's device region is too small            */
} mt_status;

#define MT_MAX_TENSORS 8

/* Opaque model handle, owned by the library (mt_destroy frees it). */
typedef struct mt_model mt_model;

/* Region of a flat block ([Hotdry] host memory layout: one contiguous block
 * per layer holding BF16 weights, BF16 gradients and FP32 Adam state). */
enum { MT_REGION_W = 0, MT_REGION_G = 1, MT_REGION_MASTER = 2, MT_REGION_M = 3, MT_REGION_V = 4 };
/* mt_read_host only, with host_grad_accum: the FP32 gradient (n_pad floats)
 * the last completed step's Adam used for the block. */
enum { MT_REGION_GACC = 5 };

/* Model, step and runtime configuration.  Plain data, copied by
 * mt_init_model.  Tokens per step T = micro_batches * batch * seq. */
typedef struct {
  int32_t n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab;
  float rope_base, rms_eps, init_std;          /* e.g. 1e4 or 1e6, 1e-6, 0.02 */
  int32_t batch, seq, micro_batches;
  int32_t ckpt_interval;   /* c in [1, n_layers]: X_s kept for s = 0, c, 2c,
                              ...; the backward recomputes each c-layer
                              segment from it ([Review] 2, block-wise
                              recomputation)                               */
  int32_t ckpt_on_host;    /* 1: layer-boundary activations in pinned host RAM
                              (device footprint independent of depth)      */
  int32_t n_grad_slabs;    /* K pinned gradient slabs ([Hotdry]: 12 in the
                              pages' system); 0 (the default): K chosen at
                              init by the static schedule (mt_get_schedule) */
  int32_t n_host_threads;  /* host worker threads; 0 = online cores         */
  float lr, beta1, beta2, adam_eps, weight_decay; /* 1e-3, .9, .999, 1e-8, 0 */
  uint64_t seed;           /* weight initialisation seed                     */
  uint32_t timeout_ms;     /* limit of every bounded host wait               */
  int32_t pin_store;       /* 0: just-in-time pack of pageable W into two
                              pinned staging buffers ([Review] 3-2 (4));
                              1: register the whole store, copy directly    */
  int32_t head_chunk;      /* tokens per LM-head chunk; 0 = automatic        */
  int32_t log_protocol;    /* 1: keep the enqueue log (mt_protocol_log)      */
  int32_t keep_host_grad;  /* 1: each slab is also unpacked into the store's
                              BF16 G region; 0: Adam reads the slab only  */
  int32_t n_buffers;       /* device weight buffers: 2 (double-buffered, the
                              pages' engine) or 1 (single-buffer ablation)  */
  int32_t host_grad_accum; /* 0: the micro-batches of a step share each
                              visit and the gradient sums on the device;
                              1: one pass over all blocks per micro-batch,
                              every pass exports its gradients, the host
                              sums them in FP32 and Adam runs on the sum
                              after the last pass ([Hotdry] gradient
                              export: accumulated into the master store) */
  int32_t n_experts;       /* 0: dense SwiGLU MLP in every decoder block;
                              E > 0 (multiple of 8, <= 128): a routed mixture
                              of E SwiGLU experts of hidden size expert_ffn,
                              top_k (<= 8) per token ([Lilting] MoE section:
                              the router picks the experts and only their
                              weights are copied to the GPU); requires
                              hidden and expert_ffn multiples of 64 and
                              host_grad_accum = 0                           */
  int32_t top_k;
  int32_t expert_ffn;
  int32_t debug_guards;    /* 1: a 4 KiB canary (0xA5) after every carved device
                              piece and every pinned host region, checked by
                              mt_sync: an overwrite latches MT_ERR_INTERNAL
                              naming the region (overflow / race detector) */
} mt_config;

typedef struct { void* base; size_t bytes; } mt_dev_region;          /* caller-owned device memory  */
typedef struct { void* compute; void* weight; void* grad; } mt_streams; /* cudaStream_t, caller-owned */

/* Bind result: a weight-less template's input slots filled with views into a
 * streamed buffer ([Review] 3-2 (5); [Lilting] Stateless Layer Templates). */
typedef struct {
  const void* w[MT_MAX_TENSORS]; /* device address of each tensor's BF16 weights   */
  void* g[MT_MAX_TENSORS];       /* device address of each tensor's BF16 gradient  */
  int32_t n_tensors, block, buf;
} mt_layer_view;

typedef struct {
  int64_t steps_done;
  int64_t h2d_bytes, d2h_bytes;       /* cumulative copies issued by the library  */
  int64_t device_bytes_used;          /* bytes of the caller's region carved      */
  double last_step_ms;                /* host wall time of the last mt_train_step */
  double adam_ms_total, pack_ms_total;/* host time in Adam workers / JIT packing  */
  int64_t host_store_bytes, pinned_bytes;
} mt_stats;

/* ------------------------------------------------------------------ model */
/* Defaults above for every runtime field; shape fields are zeroed. */
mt_status mt_default_config(mt_config* cfg);
/* Device bytes mt_init_model will carve from the caller's region: the two
 * ping-pong buffers (each the largest block's W and G regions), one layer's
 * activations for the step's tokens and fixed scratch.  It depends on the
 * widest block and the tokens per step, not on the depth ([Lilting] design
 * section: only the two buffers stay on the GPU, a fixed allocation from 7.6B
 * to 43B; [Review] 3-2 (1): device memory is bound by the layer being
 * computed and its buffers).  MT_ERR_ARG for an invalid config. */
mt_status mt_query_device_bytes(const mt_config* cfg, size_t* bytes_needed);
/* Allocates the host flat store (library-owned), fills it from the seeded
 * generator (FP32 master N(0, init_std) for matrices, 1 for RMSNorm gains,
 * W = bf16_rne(master), m = v = 0), allocates pinned staging, slabs and the
 * checkpoint store, creates the events and starts the host workers.  The
 * device region and the streams must outlive the model.
 * Sources: [Review] 3-2 (1) (host memory is the authoritative store of
 * parameters, gradients and optimizer state; the GPU starts empty) and 3-2
 * (4) (one contiguous block per layer, a few pinned staging buffers);
 * [Hotdry] host memory layout (pageable master store, two pinned staging
 * buffers sized to the largest layer, K = 12 gradient slabs); [Peter]
 * 記憶體預取策略 (the static prefetch schedule, planned here from the
 * blocks' bytes and the link bandwidth measured at init).
 * Errors: MT_ERR_ARG (invalid config, null region or stream),
 * MT_ERR_DEVICE_OOM (region smaller than mt_query_device_bytes),
 * MT_ERR_HOST_OOM (store or pinned memory), MT_ERR_CUDA. */
mt_status mt_init_model(const mt_config* cfg, mt_dev_region dev, mt_streams s, mt_model** model_out);
/* Copies the step's token ids (host, [micro][batch][seq] int32 in [0, V))
 * into pinned memory; the embedding's forward visit uploads them on the
 * compute stream.  The pages do not describe how a batch reaches the GPU;
 * the tokens are the input of the streaming forward of [Review] 3-2 (2).
 * MT_ERR_ARG for a token outside [0, V) or a null pointer. */
mt_status mt_set_tokens(mt_model* model, const int32_t* tok);

/* The pages' primitives ([Hotdry] StreamIn / Bind / gradient export; [Review]
 * 3-2 (2)-(6)).  Blocks: 0 = embedding, 1..L = decoder layers, L+1 = head
 * (final RMSNorm + LM head).  A step visits blocks 0..L+1 forward (the head
 * visit runs its forward, the loss and its backward) and then L..0 backward;
 * the calls below must follow that order (MT_ERR_STATE otherwise). */
/* Weight stream: waits Buffer-Free[buf], copies block's BF16 W (packed just in
 * time through pinned staging unless pin_store) into device buffer buf and,
 * for a decoder block's backward visit with host checkpoints, the block's
 * input activation; records Weights-Ready[buf].  Asynchronous. */
mt_status mt_stream_in(mt_model* model, int32_t block, int32_t buf);
/* Compute stream waits Weights-Ready[buf]; fills *view. */
mt_status mt_bind(mt_model* model, int32_t block, int32_t buf, mt_layer_view* view);
/* Forward visit of view->block over all micro-batches of the step (they are
 * concatenated along the token axis).  Records Buffer-Free (or, for the head,
 * Backward-Done).  Asynchronous. */
mt_status mt_step_forward(mt_model* model, const mt_layer_view* view);
/* Backward visit: recompute the block forward from its checkpointed input,
 * then the backward; weight gradients are written (BF16, round to nearest
 * even) straight into the buffer's gradient region at the flat layout
 * offsets; records Backward-Done.  Asynchronous. */
mt_status mt_step_backward(mt_model* model, const mt_layer_view* view);
/* Gradient stream: waits Backward-Done[buf], takes a free slab (the
 * lowest-numbered one; the host waits, bounded, while all K are held by
 * pending Adam jobs), copies the gradient region into it, records
 * Buffer-Free[buf] and the slab's event; *slab receives its index. */
mt_status mt_stream_out(mt_model* model, int32_t block, int32_t buf, int32_t* slab);
/* Queues block's host Adam: a worker waits (bounded) for the slab's event,
 * copies the slab into the block's G region (keep_host_grad), runs Adam
 * (t = adam_step >= 1) on master / m / v, rewrites W = bf16_rne(master) and
 * releases the slab.  Queued jobs run lowest block first: the next forward
 * needs block 0 first although its gradient arrives last. */
mt_status mt_adam_host(mt_model* model, int32_t block, int32_t slab, int32_t adam_step);
/* One whole step (0-based index `step`, which must equal the number of steps
 * done) following the static schedule; *loss (if not null) receives the step
 * loss once its value has reached the host.  Returns after enqueuing the
 * last backward visit; Adam of the last blocks may still run.
 * Sources: [Review] 3-2 (2)-(3) (streaming forward, block-wise recomputing
 * backward, three streams overlapping the next transfer, the current compute
 * and the previous gradient export); [Hotdry] event protocol; [Peter]
 * 記憶體預取策略 (prefetch timed from each layer's bytes, the link bandwidth
 * and the layer's compute time). */
mt_status mt_train_step(mt_model* model, int32_t step, float* loss);
/* Waits (bounded) for every queued copy, kernel and Adam job.  A kernel
 * whose bounded barrier wait expired (its code in the process's device error
 * word, mt_kernel_error) makes the call fail with MT_ERR_TIMEOUT and latches
 * the model: the outputs of that kernel, and the step built on them, are not
 * valid. */
mt_status mt_sync(mt_model* model);
/* Copies `bytes` of a block's region (MT_REGION_*) out of / into the host
 * store (after mt_sync).  bytes must not exceed the region (MT_ERR_ARG).
 * The store is the model's authoritative state ([Review] 3-2 (1); [Hotdry]
 * host memory layout: W, G and FP32 state of one layer in one block), so
 * these calls read and write the model itself. */
mt_status mt_read_host(mt_model* model, int32_t block, int32_t region, void* dst, size_t bytes);
mt_status mt_write_host(mt_model* model, int32_t block, int32_t region, const void* src, size_t bytes);
/* Counters since mt_init_model (bytes copied per direction, host Adam and
 * packing time, store and pinned sizes); read after mt_sync.  MT_ERR_ARG
 * for a null argument. */
mt_status mt_get_stats(const mt_model* model, mt_stats* out);
/* Save / resume.  Between steps the GPU holds no model state, so the host
 * store (every block's W, G, master, m, v) and the number of steps done are
 * the whole training state.  mt_save drains all work and writes them to a
 * file (a 64-byte header: magic, the model shape, steps done, store size;
 * then the store); mt_load reads such a file into a model of the same shape
 * and continues from its step count (the next mt_train_step takes that
 * index; tokens must be set again).  Both only between steps (MT_ERR_STATE
 * otherwise); a file of another shape or a missing file is MT_ERR_ARG; an
 * I/O failure while writing is MT_ERR_INTERNAL, while reading it latches
 * the model (its store is partly overwritten). */
mt_status mt_save(mt_model* model, const char* path);
mt_status mt_load(mt_model* model, const char* path);
/* MoE models: the per-expert token counts (n_experts int32) of block j's
 * last forward (1 <= j <= n_layers), i.e. which experts its stream-ins
 * copied; read after mt_sync.  MT_ERR_ARG for a dense model or a bad j. */
mt_status mt_expert_counts(const mt_model* model, int32_t block, int32_t* counts, int32_t n);
/* The enqueue log (lines "step stream op a b"); returns its length, or
 * -(needed) when cap is too small. */
int64_t mt_protocol_log(const mt_model* model, char* buf, int64_t cap);
/* Text of the last error ("" if none, "null model" for NULL), copied into
 * storage of the calling thread: valid until that thread calls again.
 * Error reporting has no counterpart on the pages; it belongs to this C ABI,
 * where no exception may cross the boundary. */
const char* mt_last_error(const mt_model* model);
/* Stops the host workers, waits for the work queued on the model's three
 * streams, then frees everything the library owns (host store, pinned
 * memory, events).  The caller's device region and streams are left alone.
 * Accepts NULL.  Teardown has no counterpart on the pages; the ownership it
 * releases is the one of [Hotdry] host memory layout (store and pinned
 * buffers on the host side). */
void mt_destroy(mt_model* model);

/* ------------------------------------------------------------------ host-only */
/* None of these touches a GPU. */
/* Layout of block j, in the format: [0] n_tensors [1] n_real [2] n_pad,
 * [3..7] byte offsets of the W, G, master, m, v regions, [8] block bytes,
 * [9] offset in the store, then (element offset, rows, cols) per tensor.
 * Returns the count written or -1. */
int64_t mt_layout_block(const mt_config* cfg, int32_t j, int64_t* out, int64_t cap);
/* Parameters of the model (every block's tensors, no padding), and the
 * bytes of its host flat store (16 per padded parameter, regions 4096-byte
 * aligned); -1 for an invalid config. */
int64_t mt_param_count(const mt_config* cfg);
int64_t mt_store_bytes(const mt_config* cfg);
/* The library's initialiser for block j (n_pad FP32 master values). */
mt_status mt_host_init_block(const mt_config* cfg, int32_t j, float* master);
/* The library's host Adam over n elements on n_threads threads; g_bf16 =
 * NULL applies a zero gradient (what an MoE expert no token was routed to
 * receives). */
mt_status mt_host_adam(int64_t n, const uint16_t* g_bf16, float* master, float* m, float* v,
                       uint16_t* w_bf16, int32_t adam_step, float lr, float beta1, float beta2,
                       float eps, float weight_decay, int32_t n_threads);
/* Runs the step scheduler without any device or host work and returns the
 * enqueue log of n_steps steps (as mt_protocol_log). */
int64_t mt_plan_protocol(const mt_config* cfg, int32_t n_steps, char* buf, int64_t cap);
/* The visits of one step in order, for callers driving the per-visit calls:
 * kind[v] (0 forward, 1 head: fused forward and backward, 2 recompute: a
 * forward inside the backward that rebuilds a checkpoint segment, run with
 * mt_step_forward, 3 block backward) and block[v]; the buffer of visit v is
 * v % n_buffers.  Returns the number of visits (n_layers + 3 + the recompute
 * visits), or -1 on a bad config; writes at most cap entries. */
int32_t mt_visit_plan(const mt_config* cfg, int32_t* kind, int32_t* block, int32_t cap);
/* Static prefetch schedule ([Peter] 記憶體預取策略: prefetch timing from each
 * layer's bytes, the link bandwidth and its compute time).  Per visit v of a
 * step: b[v] H2D bytes, d[v] exported gradient bytes, c[v] compute seconds,
 * a[v] Adam seconds.  stall[v] = predicted wait before visit v computes;
 * returns the slab count needed, or -1. */
int32_t mt_schedule(int32_t n_visits, const double* b, const double* d, const double* c,
                    const double* a, double bw_h2d, double bw_d2h, double* stall);
/* The static schedule as a steady-state model of the whole pipeline: the
 * pack of each visit's weights into pinned staging (on the host worker pool,
 * ahead of Adam's queued work, chunk by chunk with each chunk's copy starting
 * once it is packed), the host-to-device copy, the compute, the gradient
 * export into one of K slabs and host Adam (lowest block first among landed
 * slabs), with every dependency of the event protocol (Buffer-Free,
 * Weights-Ready, Backward-Done, a free slab, and the next step's forward of a
 * block after its Adam).  Host memory is shared: Adam runs at the smaller of
 * its idle-host rate and what host_bw leaves after the period's DMA and pack
 * traffic.  Per visit v of a step (mt_visit_plan order): kind[v], block[v],
 * b[v] host-to-device bytes, p[v] bytes packed first (0 with a pinned store),
 * d[v] exported gradient bytes, c[v] compute seconds, a[v] Adam elements of
 * the exported block.  Sources: [Peter] 記憶體預取策略 (prefetch from layer
 * bytes, link bandwidth and compute time); [Hotdry] slab pool and event
 * protocol; [Review] 3-2 (4), (6). */
typedef struct {
  int32_t n_visits;
  const int32_t *kind, *block;
  const double *b, *p, *d, *c, *a;
  int32_t n_buffers;
  double bw_h2d, bw_d2h; /* link bytes/s per direction */
  double pack_rate;      /* bytes/s the worker pool packs (0: instant) */
  double adam_rate;      /* Adam elements/s of the worker pool on an idle host (0: instant) */
  double adam_bytes;     /* host memory bytes Adam moves per element (28; 30 with the G copy) */
  double host_bw;        /* bytes/s host memory serves CPU and DMA together (0: unlimited) */
} mt_sched_in;
typedef struct {
  int32_t K;         /* slabs */
  int32_t measured;  /* mt_get_schedule: 1 if c[] was measured in the first step */
  double period_ms;  /* predicted steady-state step time */
  double stall_ms;   /* predicted compute-stream idle time per step */
  double adam_busy_ms, slab_wait_ms, pack_ms;
  double adam_gelem_s;  /* Adam's rate after DMA and the pack took their share */
  /* mt_get_schedule: the init-time measurements the plan used */
  double bw_h2d_gbs, bw_d2h_gbs, pack_gbs, adam_gelem_s_idle, host_gbs;
} mt_sched_plan;
/* Simulates the pipeline with K slabs (stall_v: n_visits entries, may be
 * null: the predicted wait before each visit computes).  MT_ERR_ARG for
 * missing arrays, n_visits < 1, K < 1 or a non-positive link bandwidth. */
mt_status mt_schedule_simulate(const mt_sched_in* in, int32_t K, mt_sched_plan* out, double* stall_v);
/* Chooses K in [1, k_max]: the shortest predicted step, then the fewest slabs
 * within 0.5 % of it. */
mt_status mt_schedule_plan(const mt_sched_in* in, int32_t k_max, mt_sched_plan* out);
/* The plan a model runs with: which = 0, made in mt_init_model from the
 * blocks' bytes, the link, pack, Adam and shared host-memory rates measured
 * there and compute times estimated from each visit's tensor FLOPs at 1.2
 * PFLOP/s (it set K when n_grad_slabs was 0); which = 1, made again once the
 * first step's per-visit compute times (CUDA events) are known (MT_ERR_STATE
 * until then). */
mt_status mt_get_schedule(const mt_model* model, int32_t which, mt_sched_plan* out);
/* Host memory bandwidth on this machine: a parallel copy of `bytes` (GB/s,
 * read + write bytes) and the library's Adam (G elements/s) on n_threads
 * threads; every pass runs 3 times and the best is reported. */
mt_status mt_host_bandwidth(size_t bytes, int32_t n_threads, double* copy_gbs, double* adam_gelem_s);
/* Per-vocabulary-row lists of token rows (CSR) used by the embedding
 * gradient: row_start[V+1], rows[T]. */
mt_status mt_token_csr(const int32_t* tok, int64_t T, int32_t V, int32_t* row_start, int32_t* rows);
/* RoPE cos/sin table [S][hd/2][2] in FP32 (angles in double). */
mt_status mt_rope_table(int32_t S, int32_t hd, double base, float* out);

/* ------------------------------------------------------------------ per-op (device) */
/* The block math as individual device calls, for tests and other callers.
 * All pointers are device addresses, row-major, 16-byte aligned; every "ld"
 * is a row stride in elements and a multiple of 8.  A call with no rows
 * (T, rows, V or n_seq * S = 0) launches nothing, writes nothing (dgamma
 * included) and returns MT_OK; pointers must still be non-null.  mt_gemm
 * needs M, N, K >= 1 (MT_ERR_ARG otherwise).  Kernels are enqueued on
 * `stream` (a cudaStream_t; NULL = the legacy default stream). */

/* D[m,n] = sum_k A(m,k) B(n,k) on tcgen05 tensor cores, FP32 accumulation.
 * A is [M][K] (a_mn = 0) or [K][M] (a_mn = 1); B is [N][K] or [K][N].
 * acc_mode 0: none; 1: Dacc = acc; 2: Dacc += acc (FP32, then used below);
 * R (optional) is added; D (optional) receives bf16_rne.  BF16 operands. */
mt_status mt_gemm(const void* A, int64_t lda, int32_t a_mn, const void* B, int64_t ldb,
                  int32_t b_mn, int32_t M, int32_t N, int32_t K, void* D, int64_t ldd,
                  const void* R, int64_t ldr, float* Dacc, int64_t ldacc, int32_t acc_mode,
                  void* stream);
/* Tiling of the dense GEMMs (mt_gemm, mt_gemm2 and those of the training
 * step) for the whole process: 0 = one CTA per 128 x 256 output tile; 1 (the
 * default), 2 and 3 = a pair of CTAs (one cluster, cta_group::2 MMAs) per
 * 256 x 256 tile, the operands split between the two SMs' shared memory.
 * Under 1 and 2 a launch whose every GEMM has K >= 8192, N >= 512 and no
 * residual uses 256 x 512 pair tiles instead.  Under 1 and 3 each pair draws its next tile
 * from a per-launch counter (the tiles in flight stay a window of consecutive
 * tiles of the raster order, so tiles that share an operand run together);
 * under 2 it takes every n-th tile of that order (n = pairs resident).  The
 * MoE grouped GEMMs always use one CTA per tile.  All modes give bitwise the
 * same results (same K order, FP32 accumulation).  Any other value changes
 * nothing; returns the mode in force before the call.  Takes effect at the
 * next launch; not synchronised with launches in flight on other threads. */
int32_t mt_gemm_mode(int32_t mode);
/* Two independent GEMMs (each as mt_gemm, arguments given as arrays of two)
 * in one persistent launch: their output tiles share one schedule. */
mt_status mt_gemm2(const void* const* A, const int64_t* lda, const int32_t* a_mn, const void* const* B,
                   const int64_t* ldb, const int32_t* b_mn, const int32_t* M, const int32_t* N,
                   const int32_t* K, void* const* D, const int64_t* ldd, void* stream);
/* RMSNorm forward: y = x * rstd * gamma, rstd = (mean(x^2)+eps)^-1/2 per row.
 * x, y: [T][H] BF16, gamma: [H] BF16, rstd: [T] FP32; H a multiple of 8 and at
 * most 24576, x, gamma and y 16-byte aligned, else MT_ERR_ARG. */
mt_status mt_rmsnorm_fwd(const void* x, const void* gamma, int64_t T, int32_t H, float eps,
                         void* y, float* rstd, void* stream);
/* RMSNorm backward: dx = d/dx + dres (dres optional), dgamma = sum over rows,
 * summed in a fixed order (the same inputs give the same bits).  H a multiple
 * of 8 and at most 12288, BF16 tensors 16-byte aligned, else MT_ERR_ARG.
 * scratch: device memory of mt_rmsnorm_bwd_scratch_bytes(T, H) bytes. */
mt_status mt_rmsnorm_bwd(const void* dy, const void* x, const void* gamma, const float* rstd,
                         const void* dres, int64_t T, int32_t H, void* dx, void* dgamma,
                         void* scratch, size_t scratch_bytes, void* stream);
/* Scratch bytes mt_rmsnorm_bwd needs for T rows of H: the dgamma partial
 * sums, min(304, ceil(T / 32)) rows of H FP32 values. */
size_t mt_rmsnorm_bwd_scratch_bytes(int64_t T, int32_t H);
/* Rotate-half RoPE of the first n_heads heads of each row of x ([T][ld]),
 * position = row mod S; cs from mt_rope_table (device copy). */
mt_status mt_rope(void* x, int64_t T, int64_t ld, int32_t n_heads, int32_t hd, int32_t S,
                  const float* cs, int32_t inverse, void* stream);
/* Causal GQA attention; qkv rows [q (nh hd) | k (nkv hd) | v (nkv hd)];
 * o [T][nh hd]; lse [nh][T] FP32 (natural log).  hd in {64, 128}. */
mt_status mt_attention_fwd(const void* qkv, int32_t n_seq, int32_t S, int32_t nh, int32_t nkv,
                           int32_t hd, void* o, float* lse, void* stream);
/* Backward into dqkv (same layout as qkv; every element written); scratch of
 * mt_attention_bwd_scratch_bytes bytes (n_seq * S * nh FP32 values: the row
 * sums delta = rowsum(dO o O)), device memory owned by the caller. */
mt_status mt_attention_bwd(const void* qkv, const void* o, const float* lse, const void* dout,
                           int32_t n_seq, int32_t S, int32_t nh, int32_t nkv, int32_t hd,
                           void* dqkv, void* scratch, size_t scratch_bytes, void* stream);
/* Scratch bytes mt_attention_bwd needs (n_seq * S * nh FP32). */
size_t mt_attention_bwd_scratch_bytes(int32_t n_seq, int32_t S, int32_t nh, int32_t hd);
/* SwiGLU: gu rows [g (F) | u (F)] BF16, h = silu(g) * u [T][F]; the
 * backward writes dgu (same layout as gu) from dh.  F a multiple of 8 and
 * 16-byte aligned tensors, else MT_ERR_ARG. */
mt_status mt_swiglu_fwd(const void* gu, int64_t T, int32_t F, void* h, void* stream);
mt_status mt_swiglu_bwd(const void* gu, const void* dh, int64_t T, int32_t F, void* dgu,
                        void* stream);
/* Embedding gather X[t] = E[tok[t]] ([T][H] from E [V][H]) and the dense
 * gradient dE (all V rows written; rows of unseen ids are zero) from the
 * token CSR of mt_token_csr (device copies of row_start[V+1], rows[T]); each
 * row sums its tokens in row order, no atomics.  H a multiple of 8 and
 * 16-byte aligned tensors, else MT_ERR_ARG. */
mt_status mt_embed_fwd(const int32_t* tok, const void* E, int64_t T, int32_t H, int32_t V,
                       void* X, void* stream);
mt_status mt_embed_bwd(const int32_t* row_start, const int32_t* rows, const void* dX, int32_t V,
                       int32_t H, void* dE, void* stream);
/* Cross-entropy rows: logits [rows][V] BF16 are overwritten with
 * (softmax - onehot(target)) * inv_norm; target < 0 marks a row with no
 * target (zero gradient, zero loss); row_loss[r] = lse - logit[target]. */
mt_status mt_cross_entropy(void* logits, const int32_t* target, int64_t rows, int32_t V,
                           float inv_norm, float* row_loss, void* stream);
/* Per-launch timing of the library's own kernels: CUDA events around each
 * launch on the compute stream.  kind 0 = GEMMs, 1 = attention forward,
 * 2 = attention backward, 3 = all other kernels.  mt_timing(model, 1) resets
 * and starts, mt_timing(model, 0) stops (after draining); read after
 * mt_sync.  flops / bytes are the algorithmic work of the timed launches. */
mt_status mt_timing(mt_model* model, int32_t enable);
mt_status mt_timing_read(mt_model* model, int32_t kind, int64_t* launches, double* ms,
                         double* flops, double* bytes);
/* Per visit of the step (the order of mt_visit_plan), the mean compute-
 * stream time of its compute part over the timed train steps (ms; from
 * after its Weights-Ready wait to the end of its kernels, so an MoE forward
 * includes its wait for the routed experts).  Writes min(cap, n) values and
 * *n_visits = n.  These are the per-block compute times the static prefetch
 * schedule (mt_schedule) takes. */
mt_status mt_timing_visits(mt_model* model, double* ms, int32_t cap, int32_t* n_visits);
/* Stream timeline.  mt_trace(model, 1) clears the timeline and starts
 * recording, without draining the work already queued (so a timeline can be
 * taken in the steady state of training): CUDA events around every weight /
 * expert / checkpoint copy on the weight stream, every visit's compute on the
 * compute stream and every gradient / checkpoint export on the gradient
 * stream enqueued from then on, and the wall time of every host Adam job that
 * ends from then on, all relative to one instant (an event on an idle private
 * stream, and the host clock right after it completed).  Calling it while
 * recording drains first.  mt_trace(model, 0) drains and stops.
 * mt_trace_json writes the timeline (after mt_sync) as Chrome trace-event
 * JSON ({"traceEvents": [...]}, times in microseconds; threads "weight
 * stream", "compute stream", "gradient stream", "host Adam"); returns its
 * length, or -(needed) when cap is too small. */
mt_status mt_trace(mt_model* model, int32_t enable);
int64_t mt_trace_json(mt_model* model, char* buf, int64_t cap);
/* RMSNorm backward that allocates nothing (same results as mt_rmsnorm_bwd).
 * The pages have no counterpart: this is for callers that cannot allocate
 * device memory -- code running during stream capture, code inside another
 * framework whose allocator owns all device memory, or callers that cannot
 * afford cudaMalloc's latency or implicit synchronisation.  The dgamma
 * partial sums go to a fixed array inside the library (9.5 MiB,
 * MT_NOALLOC_SCRATCH_FLOATS floats), which every GPU that loads the library
 * holds until exit.  Returns MT_ERR_ARG when mt_rmsnorm_bwd_scratch_bytes(T, H)
 * exceeds that array (or for the arguments mt_rmsnorm_bwd rejects).  All calls
 * share the array: calls that overlap on the GPU race.  It keeps the last
 * call's contents, and nothing in it needs to start at zero.  The first call
 * on each device looks up the array's device address; make it before any
 * stream capture. */
#define MT_NOALLOC_SCRATCH_FLOATS (304u * 8192u)
mt_status mt_rmsnorm_bwd_noalloc(const void* dy, const void* x, const void* gamma,
                                 const float* rstd, const void* dres, int64_t T, int32_t H,
                                 void* dx, void* dgamma, void* stream);
/* Routed mixture-of-experts feed-forward of one layer, forward and backward
 * in one call (the block math of an MoE decoder block after its second
 * RMSNorm; [Lilting] MoE section).  yn, x1, dout: [T][H]; Wr: [E][H];
 * We: [E][W_gu (2 Fe x H) | W_down (H x Fe)] (row e = expert e).  Writes
 * out = x1 + sum_i gate_i FFN_{e_i}(yn) ([T][H]), dyn = d/d yn ([T][H]),
 * dWr ([E][H]), dWe (same layout as We; rows of experts no token was routed
 * to are zeroed), idx / gate ([T][k], int32 / FP32: the selected experts in
 * descending logit order, ties to the lower index, and their softmax gates).
 * Router logits are FP32 sums of BF16 products.  scratch: device memory of
 * mt_moe_scratch_bytes bytes.  Synchronises `stream` once (the per-expert
 * counts size the grouped products).  E multiple of 8 and <= 128, k <= 8,
 * H and Fe multiples of 64. */
size_t mt_moe_scratch_bytes(int64_t T, int32_t H, int32_t E, int32_t k, int32_t Fe);
mt_status mt_moe_ffn(const void* yn, const void* x1, const void* Wr, const void* We, const void* dout, int64_t T,
                     int32_t H, int32_t E, int32_t k, int32_t Fe, void* out, void* dyn, void* dWr, void* dWe,
                     int32_t* idx, float* gate, void* scratch, size_t scratch_bytes, void* stream);
/* Test hook for debug_guards: overwrites one byte of guard `which` (device
 * guards first, then the pinned host ones), so that the next mt_sync must
 * report it.  MT_ERR_ARG without debug_guards or for a bad index; returns the
 * number of guards through *n_guards when not null. */
mt_status mt_debug_poke_guard(mt_model* model, int32_t which, int32_t* n_guards);
/* Host-side fault injection for failure-detection tests (process-wide):
 * kind 1 = every Adam job sleeps `value` ms before it starts (a stalled
 * worker); kind 2 = the next `value` Adam jobs throw inside a worker; kind 3 =
 * the next `value` pinned host allocations fail; kind 4 = the next `value`
 * GEMM launches issue no loads, so the kernel's bounded mbarrier waits run
 * out (about 2 s), it records code 2 in the kernel error word and returns
 * with the context intact.  value 0 clears the kind.  No kind faults, traps
 * or hangs a GPU. */
mt_status mt_fault_inject(int32_t kind, int32_t value);
/* Error word of the kernels' bounded waits (0 = none); clear != 0 resets it. */
mt_status mt_kernel_error(int32_t* code, int32_t clear);

#ifdef __cplusplus
}
#endif
#endif
