/*
 * oracle.h -- C ABI of the reference oracle (TEST INFRASTRUCTURE ONLY).
 *
 * The oracle is a plain, slow, single-threaded CPU implementation of one
 * training step of the layer-streamed method: the model arithmetic written out
 * from its definition (pre-RMSNorm SwiGLU/RoPE/GQA decoder, next-token
 * cross-entropy, bias-corrected Adam on FP32 master weights), the flat
 * layer-contiguous layout, the seeded initialisation and a simulator of the
 * three-stream event protocol.  It shares no code, header or constant table
 * with the GPU library; only tests, the smoke check and the CPU-baseline leg
 * of the benchmark may load it.
 *
 * Sources (cited by page title and section throughout):
 *   [Review]  "MegaTrain: Full Precision Training of 100B+ Parameter Large
 *             Language Models on a Single GPU Review" (dimensionstp.github.io)
 *   [Hotdry]  blog.hotdry.top, 2026-04-09 post on MegaTrain's checkpoint
 *             strategy and communication overlap
 *   [Lilting] "MegaTrainはシングルGPUで120BパラメータLLMをフル精度訓練する"
 *             (lilting.ch)
 *   [Peter]   "MegaTrain：在單一 GPU 上以全精度訓練 1000 億+參數的大型語言模型"
 *             (peter-blog.pages.dev)
 *   [Azure]   "Training 100B models on a single GPU: what MegaTrain changes and
 *             what it means for Azure" (argonsys.com)
 */
#ifndef MT_ORACLE_H
#define MT_ORACLE_H
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif

/* Model / step shape.  Plain data. */
typedef struct {
  int32_t n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab;
  int32_t batch, seq, micro;       /* tokens per step = micro*batch*seq        */
  double rope_base, rms_eps, init_std;
  /* Routed mixture of experts in place of every decoder MLP ([Lilting] MoE
   * section, GPT-OSS-style): n_experts > 0 experts of hidden size expert_ffn,
   * top_k of them per token; n_experts = 0 keeps the dense SwiGLU MLP. */
  int32_t n_experts, top_k, expert_ffn;
} or_cfg;

/* ---- layout ([Hotdry] host memory layout; [Review] 3-2 (4)) ---- */
int64_t or_n_blocks(const or_cfg* c);
/* Describes block j.  out[] receives (all int64):
 *   [0] n_tensors  [1] n_real_elems  [2] n_pad_elems
 *   [3..7] byte offsets of the W, G, master, m, v regions inside the block
 *   [8] block bytes  [9] byte offset of the block inside the store
 *   then per tensor t: [10+3t] element offset, [11+3t] rows, [12+3t] cols
 * Returns the number of int64 written, or -1 on a bad argument. */
int64_t or_layout_block(const or_cfg* c, int32_t j, int64_t* out, int64_t cap);
int64_t or_param_count(const or_cfg* c);      /* P, padding excluded */
int64_t or_store_bytes(const or_cfg* c);      /* sum of block bytes */

/* ---- seeded generator and initialisation ---- */
uint64_t or_splitmix64(uint64_t seed, uint64_t i);  /* i-th output of the stream */
double   or_normal(uint64_t key, uint64_t e);        /* Box-Muller sample e      */
/* FP32 master values of block j in layout order (n_pad floats; padding = 0). */
int32_t  or_init_block(const or_cfg* c, uint64_t seed, int32_t j, float* master);
uint16_t or_bf16_rne(float x);
float    or_bf16_to_f32(uint16_t b);

/* ---- per-op functions (fp32 "f" and fp64 "d" instances) ---- */
void or_rmsnorm_fwd_d(const double* x, const double* g, int64_t T, int64_t H, double eps,
                      double* y, double* rstd);
void or_rmsnorm_bwd_d(const double* dy, const double* x, const double* g, const double* rstd,
                      int64_t T, int64_t H, double* dx, double* dg);
void or_linear_fwd_d(const double* X, const double* W, int64_t T, int64_t N, int64_t K, double* Y);
void or_linear_dgrad_d(const double* dY, const double* W, int64_t T, int64_t N, int64_t K, double* dX);
void or_linear_wgrad_d(const double* dY, const double* X, int64_t T, int64_t N, int64_t K, double* dW);
void or_rope_d(double* x, int64_t n_seq, int64_t S, int64_t ld, int64_t n_heads, int64_t hd,
               double base, int32_t inverse);
void or_attention_fwd_d(const double* qkv, int64_t n_seq, int64_t S, int64_t nh, int64_t nkv,
                        int64_t hd, double* o, double* lse);
void or_attention_bwd_d(const double* qkv, const double* o, const double* lse, const double* dout,
                        int64_t n_seq, int64_t S, int64_t nh, int64_t nkv, int64_t hd, double* dqkv);
void or_swiglu_fwd_d(const double* gu, int64_t T, int64_t F, double* h);
void or_swiglu_bwd_d(const double* gu, const double* dh, int64_t T, int64_t F, double* dgu);
double or_cross_entropy_d(const double* logits, const int32_t* tok, int64_t n_seq, int64_t S,
                          int64_t V, double norm, double* dlogits);

/* Full forward+backward of one step (no streaming).  W[j] points at block j's
 * weights in layout order; G[j] receives block j's gradient in layout order
 * (n_pad values, padding left 0).  tok is [micro][batch][seq].  Returns the
 * step loss.  The "f" instance stores activations in fp32 (double
 * accumulators); the "d" instance is fp64 throughout. */
double or_step_fwd_bwd_f(const or_cfg* c, const float* const* W, const int32_t* tok, float* const* G);
double or_step_fwd_bwd_d(const or_cfg* c, const double* const* W, const int32_t* tok, double* const* G);
/* Forward only, returning the per-token hidden state after block j (j = 0 is
 * the embedding output, j = L the last decoder layer) in out [T, H]. */
double or_forward_hidden_f(const or_cfg* c, const float* const* W, const int32_t* tok, int32_t j,
                           float* out);

/* Smallest routing margin of the last or_step_* / or_forward_hidden_f call:
 * over every MoE layer and token, the k-th largest router logit minus the
 * (k+1)-th (+inf when no layer selects, i.e. dense or top_k = n_experts). */
double or_last_route_margin(void);
/* The MoE feed-forward of one layer on its own ("d": fp64 throughout, "f":
 * fp32 storage with double sums): given the normalised input yn [T, H], the
 * residual x1 [T, H], router weights Wr [E, H], experts We [E][W_gu (2Fe x H)
 * | W_d (H x Fe)] and the output gradient dout [T, H], writes
 * out = x1 + sum_i gate_i FFN_{e_i}(yn), dyn = d loss / d yn, dWr, dWe (every
 * expert; zero where no token was routed), the selected experts idx [T, k]
 * and their gates [T, k]; returns the smallest routing margin. */
double or_moe_layer_d(int64_t T, int64_t H, int64_t E, int64_t k, int64_t Fe, const double* yn,
                      const double* x1, const double* Wr, const double* We, const double* dout, double* out,
                      double* dyn, double* dWr, double* dWe, int32_t* idx, double* gate);
double or_moe_layer_f(int64_t T, int64_t H, int64_t E, int64_t k, int64_t Fe, const float* yn,
                      const float* x1, const float* Wr, const float* We, const float* dout, float* out,
                      float* dyn, float* dWr, float* dWe, int32_t* idx, float* gate);

/* ---- Adam ([Review] 3-2 (6); [Lilting] memory table) ---- */
/* The same with an FP32 gradient g32 (g_bf16 unused when g32 is given). */
void or_adam_f32(int64_t n, const float* g32, const uint16_t* g_bf16, float* master, float* m, float* v,
                 uint16_t* w_bf16, int32_t step, float lr, float beta1, float beta2, float eps,
                 float weight_decay);
void or_adam(int64_t n, const uint16_t* g_bf16, float* master, float* m, float* v,
             uint16_t* w_bf16, int32_t step, float lr, float beta1, float beta2, float eps,
             float weight_decay);

/* ---- event protocol simulator ([Hotdry] event-driven synchronisation) ---- */
/* Writes the ordered op list of `n_steps` training steps as text lines into
 * buf (NUL-terminated).  Returns the length, or -(needed) if cap is short.
 * ckpt_interval c in [1, n_layers]: X_s is kept for s = 0, c, 2c, ... and the
 * backward recomputes each c-layer segment from it ([Review] 2, block-wise
 * recomputation); n_buffers in {1, 2} device weight buffers; n_passes passes
 * per step (one per micro-batch with host FP32 gradient accumulation, else 1).
 * MoE layers ([Lilting] MoE section: only the experts the router selected are
 * copied in) split each forward visit: the shared weights first, the routed
 * experts after the host has read the router's choice. */
int64_t or_protocol(const or_cfg* c, int32_t n_steps, int32_t n_slabs, int32_t ckpt_on_host,
                    int32_t jit_pack, int32_t ckpt_interval, int32_t n_buffers, int32_t n_passes, char* buf,
                    int64_t cap);

/* ---- static prefetch schedule ([Peter] 記憶體預取策略) ---- */
/* Per visit v of one step (2L+3 visits): b[v] H2D bytes, d[v] gradient bytes
 * exported (0 if none), c[v] compute seconds, a[v] host Adam seconds; link
 * bandwidths in bytes/s.  Writes the predicted wait before each visit's
 * compute into stall[v] and returns the slab count the pool needs. */
int32_t or_schedule(int32_t n_visits, const double* b, const double* d, const double* c,
                    const double* a, double bw_h2d, double bw_d2h, double* stall);

#ifdef __cplusplus
}
#endif
#endif
