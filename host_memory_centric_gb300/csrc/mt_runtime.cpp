// mt_runtime.cpp -- libmt: the layer-streamed training step behind the C ABI.
//
// Host RAM is the authoritative store of every parameter, gradient and Adam
// moment; the GPU holds two ping-pong weight buffers and one layer's
// activations ([Review] 3-2 (1)-(3); [Azure] "Layer-Wise Streaming",
// "Stateless Execution").  A step visits the blocks forward (embedding,
// decoder layers, head) and then backward in reverse, and each visit is:
//   weight stream : wait Buffer-Free[b]; (pack W into pinned staging b);
//                   H2D W (+ the block's checkpointed input); Weights-Ready[b]
//   compute stream: wait Weights-Ready[b]; Bind; forward or recompute+backward;
//                   Buffer-Free[b] (forward) or Backward-Done[b] (backward)
//   gradient stream (backward visits): wait Backward-Done[b]; D2H G into a
//                   free pinned slab; Buffer-Free[b]; slab event
//   host          : an Adam worker waits for the slab event, unpacks the slab
//                   into the G region and updates master / m / v / W
// ([Hotdry] three CUDA streams and the event-driven synchronisation protocol;
// [Review] 3-2 (3)-(6)).  No host barrier sits on the path: every host wait
// is on a specific event or slab, with a deadline.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <sys/mman.h>
#include <unistd.h>

#include <chrono>
#include <cmath>
#include <cstdio>
#include <algorithm>
#include <cstring>
#include <memory>
#include <stdexcept>

#include "mt_host.h"
#include "mt_kernels.h"

using mt::bf16;
using Clock = std::chrono::steady_clock;

namespace {

// test-only host fault injection (mt_fault_inject)
std::atomic<int> g_inj_adam_delay_ms{0}, g_inj_adam_throw{0}, g_inj_pinned_fail{0};

cudaError_t pinned_alloc(void** p, size_t bytes) {
  if (g_inj_pinned_fail.load() > 0) {
    g_inj_pinned_fail--;
    *p = nullptr;
    return cudaErrorMemoryAllocation;
  }
  return cudaHostAlloc(p, bytes, cudaHostAllocDefault);
}

struct Job {
  int32_t block, slab, t, pass;  // pass < passes - 1: FP32 accumulation only
  std::vector<uint8_t> routed;   // MoE block: 1 for each expert some token was routed to
};

// Device workspace of a routed MoE layer (expert-sorted rows, R_max of them).
struct MoeWs {
  mt::MoePlan p{};
  float* logits = nullptr;  // [T][E] router logits, FP32
  bf16 *xperm = nullptr, *gu = nullptr, *h = nullptr, *y = nullptr, *dy = nullptr, *dh = nullptr,
       *dgu = nullptr, *dlog = nullptr;
};
struct MoeShape {
  int64_t T;
  int H, E, k, Fe;
};
// Host view of one layer's routing: sorted rows in use and, per routed expert,
// its segment (the K-groups of the expert weight gradients).
struct MoeRoute {
  int64_t R = 0, assigned = 0;
  std::vector<int> e, k0, klen;
};
MoeRoute route_from_counts(const int32_t* counts, int E) {
  MoeRoute r;
  int64_t row = 0;
  for (int e = 0; e < E; ++e) {
    const int64_t n = counts[e], pad = (n + 127) / 128 * 128;
    if (n > 0) {
      r.e.push_back(e);
      r.k0.push_back((int)row);
      r.klen.push_back((int)pad);
    }
    row += pad;
    r.assigned += n;
  }
  r.R = row;
  return r;
}
// Carves an MoE workspace for T tokens from base (sizes only when null).
size_t moe_carve(const MoeShape& q, uint8_t* base, MoeWs* w) {
  size_t off = 0;
  auto take = [&](int64_t bytes) -> uint8_t* {
    off = (off + 255) / 256 * 256;
    uint8_t* p = base ? base + off : nullptr;
    off += (size_t)bytes;
    return p;
  };
  const int64_t R = mt::moe_rows_max(q.T, q.E, q.k), nch = mt::moe_chunks(q.T), T = q.T;
  w->logits = (float*)take(T * q.E * 4);
  w->p.idx = (int32_t*)take(T * q.k * 4);
  w->p.gate = (float*)take(T * q.k * 4);
  w->p.slot_row = (int32_t*)take(T * q.k * 4);
  w->p.cnt = (int32_t*)take(nch * q.E * 4);
  w->p.base = (int32_t*)take(nch * q.E * 4);
  w->p.counts = (int32_t*)take(q.E * 4);
  w->p.tile_expert = (int32_t*)take(R / 128 * 4);
  w->p.perm_tok = (int32_t*)take(R * 4);
  w->xperm = (bf16*)take(R * q.H * 2);
  w->y = (bf16*)take(R * q.H * 2);
  w->dy = (bf16*)take(R * q.H * 2);
  w->gu = (bf16*)take(R * 2 * q.Fe * 2);
  w->dgu = (bf16*)take(R * 2 * q.Fe * 2);
  w->h = (bf16*)take(R * q.Fe * 2);
  w->dh = (bf16*)take(R * q.Fe * 2);
  w->dlog = (bf16*)take(T * q.E * 2);
  return (off + 255) / 256 * 256;
}

struct Dev {
  uint8_t* buf[2] = {nullptr, nullptr};
  bf16 *xslot[2] = {nullptr, nullptr}, *xck[2] = {nullptr, nullptr}, *dx[2] = {nullptr, nullptr};
  bf16 *ckdev = nullptr, *fx[2] = {nullptr, nullptr};  // device checkpoints; non-kept forward outputs
  std::vector<bf16*> seg;  // X_{s+1} .. X_{s+c-1} of the segment being recomputed
  bf16 *xn = nullptr, *x1 = nullptr, *yn = nullptr, *qkv = nullptr, *dqkv = nullptr, *attn = nullptr,
       *dattn = nullptr;
  bf16 *gu = nullptr, *dgu = nullptr, *h = nullptr, *dh = nullptr, *dyn = nullptr, *dx1 = nullptr,
       *dxn = nullptr, *logits = nullptr;
  float *rstd1 = nullptr, *rstd2 = nullptr, *lse = nullptr, *delta = nullptr,
        *row_loss = nullptr, *loss = nullptr, *rms_part = nullptr, *dwacc = nullptr, *cs = nullptr;
  int32_t *tok = nullptr, *tgt = nullptr, *csr_start = nullptr, *csr_rows = nullptr;
  MoeWs moe;  // routed MoE layers only
  // debug guards: offset (from the region base) of the 4 KiB canary after
  // each carved piece, their device copy and the first-bad-guard word
  std::vector<int64_t> guards;
  int64_t* guard_offs = nullptr;
  int* guard_bad = nullptr;
};
constexpr int64_t kGuardBytes = 4096;

// One visit of the step: 0 FWD, 1 HEAD (fused forward and backward), 2 RECOMP
// (forward rebuilding a segment's activations), 3 BWD.  seg numbers the
// backward's segments from the top; `first` marks the visit that loads the
// segment's checkpoint.
struct VisitDesc {
  int kind, j, seg;
  bool first;
};
enum { V_FWD = 0, V_HEAD = 1, V_RECOMP = 2, V_BWD = 3 };

// Block-wise recomputation with checkpoint interval c: X_s is kept for
// s = 0, c, 2c, ... < L; the decoder layers form segments [s+1, min(s+c, L)]
// handled from the top, each recomputing X_{s+1} .. X_{e-1} from X_s and then
// running the backward of layers e .. s+1.
std::vector<VisitDesc> build_plan(int L, int c) {
  std::vector<VisitDesc> p;
  for (int j = 0; j <= L; ++j) p.push_back({V_FWD, j, -1, false});
  p.push_back({V_HEAD, L + 1, -1, false});
  const int nseg = (L + c - 1) / c;
  for (int k = 0; k < nseg; ++k) {
    const int s = (nseg - 1 - k) * c, e = s + c < L ? s + c : L;
    for (int j = s + 1; j < e; ++j) p.push_back({V_RECOMP, j, k, j == s + 1});
    for (int j = e; j > s; --j) p.push_back({V_BWD, j, k, j == s + 1 && e == s + 1});
  }
  p.push_back({V_BWD, 0, -1, false});
  return p;
}

struct KStat {
  int64_t launches = 0;  // kernels launched
  double ms = 0, flops = 0, bytes = 0;
};
struct Pending {
  cudaEvent_t a, b;
  int kind, nk;  // kind < 0: the compute of visit nk (per-visit timing)
  double flops, bytes;
};

}  // namespace

struct mt_model {
  mt_config c{};
  int L = 0, H = 0, nh = 0, nkv = 0, hd = 0, F = 0, V = 0, B = 0, S = 0, M = 0, Nqkv = 0;
  bool moe = false;           // decoder blocks are routed mixtures of experts
  int E = 0, topk = 0, Fe = 0;
  int32_t* hcounts = nullptr; // pinned [L+2][E]: per-expert token counts of each MoE layer's forward
  int64_t T = 0, chunk = 0;
  std::vector<mth::BlockDesc> lay;
  std::vector<VisitDesc> plan;
  int nbuf = 2, ci = 1, nseg = 0;
  int64_t wb_max = 0;
  bool live = false;  // false: scheduler dry run (log only)
  // host memory
  uint8_t* store = nullptr;
  size_t store_bytes = 0;
  bool registered = false;
  uint8_t* staging[2] = {nullptr, nullptr};
  uint8_t* slabs = nullptr;
  uint8_t* ckpt = nullptr;
  int32_t* htok = nullptr;  // pinned: tok[T] | tgt[T] | csr_start[V+1] | csr_rows[T]
  float* hloss = nullptr;    // pinned: the loss of every pass of a step
  float* gacc = nullptr;     // host FP32 gradient accumulator (host_grad_accum)
  size_t gacc_bytes = 0;
  std::vector<int64_t> gacc_off;  // element offset of each block in gacc
  size_t pinned_bytes = 0;
  int K = 12;
  // device
  Dev d;
  uint8_t* dev_base = nullptr;
  size_t dev_bytes = 0, dev_used = 0;
  cudaStream_t sc = nullptr, sw = nullptr, sg = nullptr;
  cudaEvent_t WR[2] = {}, BD[2] = {}, BF[2] = {}, XR[2] = {}, XS[2] = {}, TOK = nullptr, LOSS = nullptr;
  cudaEvent_t RT = nullptr, ER[2] = {};  // MoE: Route-Ready (counts on the host), Experts-Ready[b]
  std::vector<cudaEvent_t> SR;
  // host workers: Adam, initialisation and the just-in-time pack share
  // `pool`; the pack's pieces go ahead of Adam's queued chunks (and the
  // driver thread copies them too), so a pack waits at most for the chunks
  // already running
  mth::Pool pool;
  // static schedule: per-visit inputs of one pass, the plans made at init
  // (compute estimated) and after the first step (compute measured)
  std::vector<int32_t> sk_kind, sk_block;
  std::vector<double> sk_b, sk_p, sk_d, sk_c, sk_a;
  mth::SimIn sim;
  mt_sched_plan plan0{}, plan1{};
  bool have_plan1 = false;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> first_ev;  // compute of each visit of the first step
  std::vector<char> first_rec;                                // ... and whether it was recorded
  std::thread adam_thr;
  std::mutex amu;
  std::condition_variable acv;
  std::deque<Job> jobs;
  bool stopping = false;
  int inflight_jobs = 0;
  std::vector<int64_t> adam_done;  // last Adam step applied per block
  std::vector<char> slab_free;
  // state
  std::atomic<bool> failed{false};
  mutable std::mutex emu;
  std::string err;
  int64_t steps_done = 0, exports = 0;
  bool used[2] = {false, false};
  int vis = 0, stage = 0;  // next visit of the current pass, and its sub-stage
  int pass = 0, npass = 1;  // micro-batch pass of the step (host_grad_accum), passes per step
  int Mp = 1;               // micro-batches one pass processes
  bool tokens_set = false;
  std::vector<std::string> log;
  // stats
  std::atomic<int64_t> h2d{0}, d2h{0};
  double last_step_ms = 0, pack_ms = 0;
  std::atomic<int64_t> adam_us{0};
  // kernel timing (events around launches on the compute stream)
  bool timing = false;
  std::vector<Pending> pend;
  std::vector<cudaEvent_t> ev_pool;
  KStat kstat[4];
  std::vector<KStat> vstat;  // per visit of the step: compute-stream time of its compute part
  // stream timeline (mt_trace): device intervals as event pairs on the stream
  // that ran them, host Adam jobs as wall-clock intervals
  struct TraceDev {
    cudaEvent_t a, b;
    char stream;
    int op, block;
    int64_t step;
  };
  struct TraceHost {
    double t0, t1;
    int block, pass;
    int64_t step;
  };
  std::vector<std::pair<uint8_t*, std::string>> hguards;  // pinned host canaries (debug_guards)
  std::atomic<bool> tracing{false};
  cudaEvent_t trace_base = nullptr;
  cudaStream_t trace_stream = nullptr;  // idle stream that timestamps the timeline's origin
  double trace_host_base = 0;
  std::vector<TraceDev> tdev;
  std::mutex tmu;  // thost is appended by the Adam dispatcher
  std::vector<TraceHost> thost;

  ~mt_model();
};

namespace {

// ---------------------------------------------------------------- errors
mt_status set_err(mt_model* m, mt_status s, const std::string& msg, bool latch = true) {
  if (m) {
    std::lock_guard<std::mutex> lk(m->emu);
    m->err = msg;
    if (latch && s != MT_ERR_ARG) m->failed = true;
  }
  return s;
}
#define CU(m, call)                                                                              \
  do {                                                                                           \
    cudaError_t e_ = (call);                                                                     \
    if (e_ != cudaSuccess)                                                                       \
      return set_err(m, MT_ERR_CUDA, std::string(#call) + ": " + cudaGetErrorString(e_));       \
  } while (0)
#define OK(x)                     \
  do {                            \
    mt_status s_ = (x);           \
    if (s_ != MT_OK) return s_;   \
  } while (0)

double now_ms() {
  return std::chrono::duration<double, std::milli>(Clock::now().time_since_epoch()).count();
}

// Bounded host wait on an event.
mt_status wait_event(mt_model* m, cudaEvent_t ev, const char* what) {
  const auto dl = Clock::now() + std::chrono::milliseconds(m->c.timeout_ms);
  for (;;) {
    const cudaError_t e = cudaEventQuery(ev);
    if (e == cudaSuccess) return MT_OK;
    if (e != cudaErrorNotReady)
      return set_err(m, MT_ERR_CUDA, std::string("event ") + what + ": " + cudaGetErrorString(e));
    if (Clock::now() > dl) return set_err(m, MT_ERR_TIMEOUT, std::string("timed out waiting for ") + what);
    if (m->failed) return MT_ERR_STATE;
    std::this_thread::sleep_for(std::chrono::microseconds(20));
  }
}

void logop(mt_model* m, const char* s, const char* op, long a, long b) {
  if (!m->c.log_protocol && m->live) return;
  char line[96];
  std::snprintf(line, sizeof line, "%lld %s %s %ld %ld", (long long)m->steps_done, s, op, a, b);
  m->log.emplace_back(line);
}

int64_t up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

int64_t head_chunk(const mt_config* c, int64_t T) {
  if (c->head_chunk > 0) return c->head_chunk < T ? c->head_chunk : T;
  const int64_t cap = (int64_t)8 << 30;
  const int64_t per = 2LL * c->vocab;
  if (T * per <= cap) return T;
  int64_t ch = cap / per / 128 * 128;
  return ch < 128 ? 128 : ch;
}

// Carves the device region; with base == nullptr only sizes it.
size_t carve(const mt_config* c, const std::vector<mth::BlockDesc>& lay, uint8_t* base, Dev* d) {
  const int64_t T = mth::tokens_per_pass(c), H = c->hidden, hd = c->head_dim, nh = c->n_heads,
                nkv = c->n_kv_heads, F = c->ffn, V = c->vocab, L = c->n_layers, S = c->seq;
  const int64_t Nqkv = (nh + 2 * nkv) * hd, chunk = head_chunk(c, T);
  int64_t wb = 0;
  for (auto& b : lay) wb = b.wbytes > wb ? b.wbytes : wb;
  size_t off = 0;
  d->guards.clear();
  auto take = [&](int64_t bytes) -> uint8_t* {
    off = (size_t)up((int64_t)off, 256);
    uint8_t* p = base ? base + off : nullptr;
    off += (size_t)bytes;
    if (c->debug_guards) {  // canary after the piece
      off = (size_t)up((int64_t)off, 256);
      d->guards.push_back((int64_t)off);
      off += (size_t)kGuardBytes;
    }
    return p;
  };
  const int64_t act = T * H * 2;
  const int64_t ci = c->ckpt_interval, nseg = (L + ci - 1) / ci;
  for (int b = 0; b < c->n_buffers; ++b) d->buf[b] = take(2 * wb);
  for (int b = 0; b < 2; ++b) d->dx[b] = (bf16*)take(act);
  if (c->ckpt_on_host) {
    for (int b = 0; b < 2; ++b) d->xslot[b] = (bf16*)take(act);
    for (int b = 0; b < 2; ++b) d->xck[b] = (bf16*)take(act);
  } else {
    d->ckdev = (bf16*)take(act * nseg);
    for (int b = 0; b < 2; ++b) d->fx[b] = (bf16*)take(act);
  }
  d->seg.assign((size_t)(ci - 1), nullptr);
  for (int64_t i = 0; i + 1 < ci; ++i) d->seg[(size_t)i] = (bf16*)take(act);
  d->xn = (bf16*)take(act);
  d->x1 = (bf16*)take(act);
  d->yn = (bf16*)take(act);
  d->dyn = (bf16*)take(act);
  d->dx1 = (bf16*)take(act);
  d->dxn = (bf16*)take(act);
  d->qkv = (bf16*)take(T * Nqkv * 2);
  d->dqkv = (bf16*)take(T * Nqkv * 2);
  d->attn = (bf16*)take(T * nh * hd * 2);
  d->dattn = (bf16*)take(T * nh * hd * 2);
  if (c->n_experts > 0) {
    const MoeShape q{T, (int)H, c->n_experts, c->top_k, c->expert_ffn};
    uint8_t* w = take((int64_t)moe_carve(q, nullptr, &d->moe));
    moe_carve(q, w, &d->moe);
  } else {
    d->gu = (bf16*)take(T * 2 * F * 2);
    d->dgu = (bf16*)take(T * 2 * F * 2);
    d->h = (bf16*)take(T * F * 2);
    d->dh = (bf16*)take(T * F * 2);
  }
  d->logits = (bf16*)take(chunk * V * 2);
  d->rstd1 = (float*)take(T * 4);
  d->rstd2 = (float*)take(T * 4);
  d->lse = (float*)take(nh * T * 4);
  d->delta = (float*)take(nh * T * 4);
  d->row_loss = (float*)take(T * 4);
  d->loss = (float*)take(256);
  d->rms_part = (float*)take(mt::rmsnorm_bwd_partial_floats(T, (int)H) * 4);
  d->dwacc = chunk < T ? (float*)take(V * H * 4) : nullptr;
  d->cs = (float*)take(S * hd * 4);
  d->tok = (int32_t*)take(T * 4);
  d->tgt = (int32_t*)take(T * 4);
  d->csr_start = (int32_t*)take((V + 1) * 4);
  d->csr_rows = (int32_t*)take(T * 4);
  if (c->debug_guards) {  // the guard table and the first-bad word, themselves unguarded
    off = (size_t)up((int64_t)off, 256);
    d->guard_offs = base ? (int64_t*)(base + off) : nullptr;
    off += d->guards.size() * sizeof(int64_t);
    off = (size_t)up((int64_t)off, 256);
    d->guard_bad = base ? (int*)(base + off) : nullptr;
    off += 256;
  }
  return (size_t)up((int64_t)off, 256);
}

// ---------------------------------------------------------------- kernel timing
cudaEvent_t take_event(mt_model* m) {
  if (!m->ev_pool.empty()) {
    cudaEvent_t e = m->ev_pool.back();
    m->ev_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}
struct Timed {
  mt_model* m;
  int kind, nk;
  double flops, bytes;
  cudaEvent_t a = nullptr;
  // nk = kernels the timed call launches
  Timed(mt_model* mm, int k, double f, double b, int n = 1) : m(mm), kind(k), nk(n), flops(f), bytes(b) {
    if (m && m->timing) {
      a = take_event(m);
      cudaEventRecord(a, m->sc);
    }
  }
  ~Timed() {
    if (a) {
      cudaEvent_t b = take_event(m);
      cudaEventRecord(b, m->sc);
      m->pend.push_back({a, b, kind, nk, flops, bytes});
    }
  }
};
void collect_timing(mt_model* m) {
  for (auto& p : m->pend) {
    float ms = 0;
    if (cudaEventElapsedTime(&ms, p.a, p.b) == cudaSuccess && p.kind < 0) {
      if (p.nk >= 0 && p.nk < (int)m->vstat.size()) {
        m->vstat[(size_t)p.nk].launches += 1;
        m->vstat[(size_t)p.nk].ms += ms;
      }
    } else if (cudaEventElapsedTime(&ms, p.a, p.b) == cudaSuccess) {
      KStat& k = m->kstat[p.kind];
      k.launches += p.nk;
      k.ms += ms;
      k.flops += p.flops;
      k.bytes += p.bytes;
    }
    m->ev_pool.push_back(p.a);
    m->ev_pool.push_back(p.b);
  }
  m->pend.clear();
}

// Timeline ops: weights (and checkpoint) in, routed experts in, a visit's
// compute (10 + visit kind), gradients out, checkpoint out.
enum { TR_H2D = 0, TR_H2D_EXP = 1, TR_D2H = 3, TR_D2H_CKPT = 4, TR_COMPUTE = 10 };
// An NVTX range over a scope (visible to profilers attached to the process;
// inert otherwise).
struct Nvtx {
  explicit Nvtx(const char* fmt, int a, int b = -1) {
    char name[48];
    std::snprintf(name, sizeof name, fmt, a, b);
    nvtxRangePushA(name);
  }
  ~Nvtx() { nvtxRangePop(); }
};

// An event pair around the work enqueued on stream s inside its scope, kept
// when the timeline is on.
struct TraceSpan {
  mt_model* m;
  cudaStream_t s;
  char stream;
  int op, block;
  cudaEvent_t a = nullptr;
  TraceSpan(mt_model* mm, cudaStream_t ss, char st, int o, int j) : m(mm), s(ss), stream(st), op(o), block(j) {
    if (m->live && m->tracing) {
      a = take_event(m);
      cudaEventRecord(a, s);
    }
  }
  ~TraceSpan() {
    if (a) {
      cudaEvent_t b = take_event(m);
      cudaEventRecord(b, s);
      m->tdev.push_back({a, b, stream, op, block, m->steps_done});
    }
  }
};

// ---------------------------------------------------------------- GEMM forms
enum { K_GEMM = 0, K_ATTN_F = 1, K_ATTN_B = 2, K_OTHER = 3 };

mt_status gemm_run(mt_model* m, const mt::GemmArgs& g) {
  Timed t(m, K_GEMM, 2.0 * g.M * g.N * g.K, 0);
  CU(m, mt::gemm(g, m->sc));
  return MT_OK;
}
// Two independent GEMMs in one persistent launch.
mt_status gemm_run2(mt_model* m, const mt::GemmArgs& a, const mt::GemmArgs& b) {
  Timed t(m, K_GEMM, 2.0 * a.M * a.N * a.K + 2.0 * b.M * b.N * b.K, 0);
  CU(m, mt::gemm_pair(a, b, m->sc));
  return MT_OK;
}
// Y[T,N] = X[T,K] W[N,K]^T (+ R)
mt::GemmArgs fprop_args(const bf16* X, const bf16* W, int64_t T, int N, int K, bf16* Y, const bf16* R) {
  return mt::GemmArgs{X, K, 0, W, K, 0, (int)T, N, K, Y, N, R, N, nullptr, 0, 0};
}
// dX[T,K] = dY[T,N] W[N,K]
mt::GemmArgs dgrad_args(const bf16* dY, const bf16* W, int64_t T, int N, int K, bf16* dX) {
  return mt::GemmArgs{dY, N, 0, W, K, 1, (int)T, K, N, dX, K, nullptr, 0, nullptr, 0, 0};
}
// dW[N,K] = dY[T,N]^T X[T,K]  (acc_mode / Dacc for chunked accumulation)
mt::GemmArgs wgrad_args(const bf16* dY, const bf16* X, int64_t T, int N, int K, bf16* dW, float* acc, int acc_mode) {
  return mt::GemmArgs{dY, N, 1, X, K, 1, N, K, (int)T, dW, K, nullptr, 0, acc, K, acc_mode};
}
mt_status fprop(mt_model* m, const bf16* X, const bf16* W, int64_t T, int N, int K, bf16* Y, const bf16* R) {
  return gemm_run(m, fprop_args(X, W, T, N, K, Y, R));
}
// The weight gradient and the input gradient of one projection share dY and
// are independent: one launch computes both.
mt_status wgrad_dgrad(mt_model* m, const bf16* dY, const bf16* X, const bf16* W, int64_t T, int N, int K, bf16* dW,
                      bf16* dX, float* acc = nullptr, int acc_mode = 0) {
  return gemm_run2(m, wgrad_args(dY, X, T, N, K, dW, acc, acc_mode), dgrad_args(dY, W, T, N, K, dX));
}

// ---------------------------------------------------------------- routed MoE block math
// [Lilting] MoE section: the router picks each token's experts; the layer is
// read as the GPT-OSS-style top-k mixture (softmax over the selected logits,
// SwiGLU experts, no router bias).  Router logits in FP32, then the routing
// plan (top-k, gates, expert-sorted rows).
mt_status moe_route(mt_model* m, const MoeShape& q, const MoeWs& w, const bf16* yn, const bf16* Wr, cudaStream_t s) {
  {
    Timed t(m, K_GEMM, 2.0 * q.T * q.E * q.H, 0);
    CU(m, mt::gemm(mt::GemmArgs{yn, q.H, 0, Wr, q.H, 0, (int)q.T, q.E, q.H, nullptr, 0, nullptr, 0, w.logits, q.E, 1},
                   s));
  }
  Timed t(m, K_OTHER, 0, 4.0 * q.T * q.E + 16.0 * q.T * q.k, 4);
  CU(m, mt::moe_plan(w.logits, q.T, q.E, q.k, w.p, s));
  return MT_OK;
}

// The routed experts over the sorted rows: gather, W_gu, SwiGLU, W_down, and
// out = x1 + gate-weighted sum (skipped when out is null: the backward's
// recompute only rebuilds what the backward reads).
mt_status moe_experts_fwd(mt_model* m, const MoeShape& q, const MoeWs& w, const MoeRoute& r, const bf16* yn,
                          const bf16* x1, const bf16* We, bf16* out, cudaStream_t s) {
  const int64_t est = 3LL * q.Fe * q.H;
  const double rows = (double)r.assigned;
  {
    Timed t(m, K_OTHER, 0, 4.0 * r.R * q.H);
    CU(m, mt::moe_gather(yn, q.H, w.p.perm_tok, r.R, w.xperm, s));
  }
  {
    Timed t(m, K_GEMM, 4.0 * rows * q.Fe * q.H, 0);
    CU(m, mt::gemm_expert_rows(mt::GemmRowsArgs{w.xperm, q.H, We, q.H, 0, est, q.E, w.p.tile_expert, (int)r.R,
                                                2 * q.Fe, q.H, w.gu, 2 * q.Fe},
                               s));
  }
  {
    Timed t(m, K_OTHER, 0, 6.0 * r.R * q.Fe);
    CU(m, mt::swiglu_fwd(w.gu, r.R, q.Fe, w.h, s));
  }
  {
    Timed t(m, K_GEMM, 2.0 * rows * q.H * q.Fe, 0);
    CU(m, mt::gemm_expert_rows(mt::GemmRowsArgs{w.h, q.Fe, We + 2LL * q.Fe * q.H, q.Fe, 0, est, q.E,
                                                w.p.tile_expert, (int)r.R, q.H, q.Fe, w.y, q.H},
                               s));
  }
  if (out) {
    Timed t(m, K_OTHER, 0, 4.0 * q.T * q.H + 2.0 * rows * q.H);
    CU(m, mt::moe_combine(x1, w.y, w.p.slot_row, w.p.gate, q.T, q.H, q.k, out, s));
  }
  return MT_OK;
}

// Backward of the MoE feed-forward from dout = dL/dx2: dyn = dL/dyn, the
// router gradient dWr and the routed experts' gradients in dWe (experts with
// no rows are not written).
mt_status moe_backward(mt_model* m, const MoeShape& q, const MoeWs& w, const MoeRoute& r, const bf16* yn,
                       const bf16* Wr, const bf16* We, const bf16* dout, bf16* dyn, bf16* dWr, bf16* dWe,
                       cudaStream_t s) {
  const int64_t est = 3LL * q.Fe * q.H;
  const double rows = (double)r.assigned;
  const int ng = (int)r.e.size();
  {
    Timed t(m, K_OTHER, 0, 4.0 * q.T * q.H + 4.0 * rows * q.H + 2.0 * q.T * q.E, 2);
    CU(m, mt::moe_combine_bwd(dout, w.y, w.p.slot_row, w.p.idx, w.p.gate, q.T, q.H, q.k, q.E, w.dy, w.dlog, s));
    CU(m, mt::moe_zero_pad(w.dy, q.H, w.p.perm_tok, r.R, s));
  }
  {  // dW_down_e = dY_e^T h_e
    Timed t(m, K_GEMM, 2.0 * rows * q.H * q.Fe, 0);
    CU(m, mt::gemm_expert_kgroups(mt::GemmKGroupArgs{w.dy, q.H, w.h, q.Fe, q.H, q.Fe, (int)r.R,
                                                     dWe + 2LL * q.Fe * q.H, q.Fe, est, ng, r.e.data(), r.k0.data(),
                                                     r.klen.data()},
                                  s));
  }
  {  // dh = dY W_down_e
    Timed t(m, K_GEMM, 2.0 * rows * q.H * q.Fe, 0);
    CU(m, mt::gemm_expert_rows(mt::GemmRowsArgs{w.dy, q.H, We + 2LL * q.Fe * q.H, q.Fe, 1, est, q.E,
                                                w.p.tile_expert, (int)r.R, q.Fe, q.H, w.dh, q.Fe},
                               s));
  }
  {
    Timed t(m, K_OTHER, 0, 10.0 * r.R * q.Fe);
    CU(m, mt::swiglu_bwd(w.gu, w.dh, r.R, q.Fe, w.dgu, s));
  }
  {  // dW_gu_e = dGU_e^T xperm_e
    Timed t(m, K_GEMM, 4.0 * rows * q.Fe * q.H, 0);
    CU(m, mt::gemm_expert_kgroups(mt::GemmKGroupArgs{w.dgu, 2 * q.Fe, w.xperm, q.H, 2 * q.Fe, q.H, (int)r.R, dWe,
                                                     q.H, est, ng, r.e.data(), r.k0.data(), r.klen.data()},
                                  s));
  }
  {  // dX = dGU W_gu_e, into dy (free by now)
    Timed t(m, K_GEMM, 4.0 * rows * q.Fe * q.H, 0);
    CU(m, mt::gemm_expert_rows(mt::GemmRowsArgs{w.dgu, 2 * q.Fe, We, q.H, 1, est, q.E, w.p.tile_expert, (int)r.R,
                                                q.H, 2 * q.Fe, w.dy, q.H},
                               s));
  }
  {
    Timed t(m, K_OTHER, 0, 2.0 * rows * q.H + 2.0 * q.T * q.H);
    CU(m, mt::moe_scatter(w.dy, w.p.slot_row, q.T, q.H, q.k, dyn, s));
  }
  {  // router: dWr = dlogits^T yn; dyn += dlogits Wr
    Timed t(m, K_GEMM, 4.0 * q.T * q.E * q.H, 0, 2);
    CU(m, mt::gemm(mt::GemmArgs{w.dlog, q.E, 1, yn, q.H, 1, q.E, q.H, (int)q.T, dWr, q.H, nullptr, 0, nullptr, 0, 0},
                   s));
    CU(m, mt::gemm(mt::GemmArgs{w.dlog, q.E, 0, Wr, q.H, 1, (int)q.T, q.H, q.E, dyn, q.H, dyn, q.H, nullptr, 0, 0},
                   s));
  }
  return MT_OK;
}

struct View {
  const bf16* w[MT_MAX_TENSORS];
  bf16* g[MT_MAX_TENSORS];
};
View make_view(mt_model* m, int j, int b) {
  View v{};
  const mth::BlockDesc& bd = m->lay[(size_t)j];
  for (int t = 0; t < bd.nt; ++t) {
    v.w[t] = reinterpret_cast<const bf16*>(m->d.buf[b] + bd.region[0]) + bd.t[t].off;
    v.g[t] = reinterpret_cast<bf16*>(m->d.buf[b] + bd.region[1]) + bd.t[t].off;
  }
  return v;
}

bf16* x_out(mt_model* m, int j) {  // where the forward writes X_j
  if (m->c.ckpt_on_host) return m->d.xslot[j % 2];
  return (j % m->ci == 0 && j < m->L) ? m->d.ckdev + (int64_t)(j / m->ci) * m->T * m->H : m->d.fx[j % 2];
}
const bf16* x_fwd_in(mt_model* m, int j) { return x_out(m, j - 1); }  // X_{j-1}
// X_{j-1} in the backward (recompute or block backward of layer j, segment
// number seg): the segment's checkpoint X_s or a recomputed X_{s+i}.
const bf16* x_seg_in(mt_model* m, int j, int seg) {
  const int s = (j - 1) / m->ci * m->ci;
  if (j - 1 == s)
    return m->c.ckpt_on_host ? m->d.xck[seg % 2] : m->d.ckdev + (int64_t)(s / m->ci) * m->T * m->H;
  return m->d.seg[(size_t)(j - s - 2)];
}
bf16* x_seg_out(mt_model* m, int j) {  // recomputed X_j, s < j < e
  const int s = (j - 1) / m->ci * m->ci;
  return m->d.seg[(size_t)(j - s - 1)];
}

// ---------------------------------------------------------------- block math
MoeShape moe_shape(const mt_model* m) { return MoeShape{m->T, m->H, m->E, m->topk, m->Fe}; }
MoeRoute moe_route_of(const mt_model* m, int j) { return route_from_counts(m->hcounts + (size_t)j * m->E, m->E); }

// Attention half of a decoder block: xn, qkv, attention, x1 = x + attn W_o^T
// and yn = RMSNorm(x1) (the MLP's or the experts' input).
mt_status attention_half(mt_model* m, const View& v, const bf16* x) {
  const int64_t T = m->T;
  const int H = m->H, nhd = m->nh * m->hd;
  cudaStream_t s = m->sc;
  Dev& d = m->d;
  {
    Timed t(m, K_OTHER, 0, 4.0 * T * H + 4.0 * T);
    CU(m, mt::rmsnorm_fwd(x, v.w[4], T, H, m->c.rms_eps, d.xn, d.rstd1, s));
  }
  OK(fprop(m, d.xn, v.w[0], T, m->Nqkv, H, d.qkv, nullptr));
  {
    Timed t(m, K_OTHER, 0, 4.0 * T * (m->nh + m->nkv) * m->hd);
    CU(m, mt::rope(d.qkv, T, m->Nqkv, m->nh + m->nkv, m->hd, m->S, d.cs, 0, s));
  }
  {
    const double fl = 4.0 * m->Mp * m->B * (double)m->nh * m->hd * (double)m->S * m->S / 2;
    Timed t(m, K_ATTN_F, fl, 0);
    CU(m, mt::attention_fwd(d.qkv, m->Mp * m->B, m->S, m->nh, m->nkv, m->hd, d.attn, d.lse, s));
  }
  OK(fprop(m, d.attn, v.w[1], T, H, nhd, d.x1, x));
  {
    Timed t(m, K_OTHER, 0, 4.0 * T * H + 4.0 * T);
    CU(m, mt::rmsnorm_fwd(d.x1, v.w[5], T, H, m->c.rms_eps, d.yn, d.rstd2, s));
  }
  return MT_OK;
}

// Decoder block forward (pre-RMSNorm, RoPE, GQA causal attention, SwiGLU MLP
// or routed experts).  With `recompute`, everything the backward reads is
// rebuilt and the final projection / combine is skipped.  An MoE block here
// has its experts resident (recompute and backward visits, which know the
// forward's routing); the forward visit itself goes through moe_forward_visit.
mt_status decoder_forward(mt_model* m, const View& v, const bf16* x, bf16* out, bool recompute, int j) {
  const int64_t T = m->T;
  const int H = m->H, F = m->F;
  cudaStream_t s = m->sc;
  Dev& d = m->d;
  OK(attention_half(m, v, x));
  if (m->moe) {
    const MoeShape q = moe_shape(m);
    OK(moe_route(m, q, d.moe, d.yn, v.w[2], s));
    return moe_experts_fwd(m, q, d.moe, moe_route_of(m, j), d.yn, d.x1, v.w[3], recompute ? nullptr : out, s);
  }
  OK(fprop(m, d.yn, v.w[2], T, 2 * F, H, d.gu, nullptr));
  {
    Timed t(m, K_OTHER, 0, 6.0 * T * F);
    CU(m, mt::swiglu_fwd(d.gu, T, F, d.h, s));
  }
  if (!recompute) OK(fprop(m, d.h, v.w[3], T, H, F, out, d.x1));
  return MT_OK;
}

// Recompute + backward of a decoder block.  dout = dL/dX_j (read), din =
// dL/dX_{j-1} (written); weight gradients land in v.g[*].
mt_status decoder_backward(mt_model* m, const View& v, const bf16* x, const bf16* dout, bf16* din, int j) {
  OK(decoder_forward(m, v, x, nullptr, true, j));
  const int64_t T = m->T;
  const int H = m->H, F = m->F, nhd = m->nh * m->hd;
  cudaStream_t s = m->sc;
  Dev& d = m->d;
  if (m->moe) {
    OK(moe_backward(m, moe_shape(m), d.moe, moe_route_of(m, j), d.yn, v.w[2], v.w[3], dout, d.dyn, v.g[2], v.g[3],
                    s));
  } else {
    OK(wgrad_dgrad(m, dout, d.h, v.w[3], T, H, F, v.g[3], d.dh));
    {
      Timed t(m, K_OTHER, 0, 10.0 * T * F);
      CU(m, mt::swiglu_bwd(d.gu, d.dh, T, F, d.dgu, s));
    }
    OK(wgrad_dgrad(m, d.dgu, d.yn, v.w[2], T, 2 * F, H, v.g[2], d.dyn));
  }
  {
    Timed t(m, K_OTHER, 0, 8.0 * T * H + 4.0 * T, 2);
    CU(m, mt::rmsnorm_bwd(d.dyn, d.x1, v.w[5], d.rstd2, dout, T, H, d.dx1, v.g[5], d.rms_part, s));
  }
  OK(wgrad_dgrad(m, d.dx1, d.attn, v.w[1], T, H, nhd, v.g[1], d.dattn));
  {
    const double fl = 10.0 * m->Mp * m->B * (double)m->nh * m->hd * (double)m->S * m->S / 2;
    Timed t(m, K_ATTN_B, fl, 0, 3);
    CU(m, mt::attention_bwd(d.qkv, d.attn, d.lse, d.dattn, m->Mp * m->B, m->S, m->nh, m->nkv, m->hd, d.dqkv,
                            d.delta, s));
  }
  {
    Timed t(m, K_OTHER, 0, 4.0 * T * (m->nh + m->nkv) * m->hd);
    CU(m, mt::rope(d.dqkv, T, m->Nqkv, m->nh + m->nkv, m->hd, m->S, d.cs, 1, s));
  }
  OK(wgrad_dgrad(m, d.dqkv, d.xn, v.w[0], T, m->Nqkv, H, v.g[0], d.dxn));
  {
    Timed t(m, K_OTHER, 0, 8.0 * T * H + 4.0 * T, 2);
    CU(m, mt::rmsnorm_bwd(d.dxn, x, v.w[4], d.rstd1, d.dx1, T, H, din, v.g[4], d.rms_part, s));
  }
  return MT_OK;
}

// Head visit: final RMSNorm, LM head, cross-entropy and their backward,
// token-chunked so the logits never exceed one chunk.
mt_status head_forward_backward(mt_model* m, const View& v, const bf16* x, bf16* din) {
  const int64_t T = m->T;
  const int H = m->H, V = m->V;
  cudaStream_t s = m->sc;
  Dev& d = m->d;
  bf16* hn = d.xn;
  bf16* dhn = d.dxn;
  float* rstd = d.rstd1;
  {
    Timed t(m, K_OTHER, 0, 4.0 * T * H);
    CU(m, mt::rmsnorm_fwd(x, v.w[0], T, H, m->c.rms_eps, hn, rstd, s));
  }
  const float inv_norm = 1.0f / (float)((double)m->M * m->B * (m->S - 1));
  for (int64_t c0 = 0; c0 < T; c0 += m->chunk) {
    const int64_t rows = (T - c0) < m->chunk ? (T - c0) : m->chunk;
    const bool first = c0 == 0, last = c0 + rows >= T;
    OK(fprop(m, hn + c0 * H, v.w[1], rows, V, H, d.logits, nullptr));
    {
      Timed t(m, K_OTHER, 0, 6.0 * rows * V);
      CU(m, mt::cross_entropy(d.logits, d.tgt + c0, rows, V, inv_norm, d.row_loss + c0, s));
    }
    if (m->chunk >= T) {
      OK(wgrad_dgrad(m, d.logits, hn, v.w[1], rows, V, H, v.g[1], dhn));
    } else {
      OK(wgrad_dgrad(m, d.logits, hn + c0 * H, v.w[1], rows, V, H, last ? v.g[1] : nullptr, dhn + c0 * H, d.dwacc,
                     first ? 1 : 2));
    }
  }
  {
    Timed t(m, K_OTHER, 0, 4.0 * T);
    CU(m, mt::reduce_sum(d.row_loss, T, inv_norm, d.loss, s));
  }
  CU(m, cudaMemcpyAsync(m->hloss + m->pass, d.loss, sizeof(float), cudaMemcpyDeviceToHost, s));
  if (m->pass + 1 == m->npass) CU(m, cudaEventRecord(m->LOSS, s));
  {
    Timed t(m, K_OTHER, 0, 8.0 * T * H, 2);
    CU(m, mt::rmsnorm_bwd(dhn, x, v.w[0], rstd, nullptr, T, H, din, v.g[0], d.rms_part, s));
  }
  return MT_OK;
}

// ---------------------------------------------------------------- Adam worker
void adam_loop(mt_model* m) {
  auto idle_since = Clock::now();
  bool idle = false;
  for (;;) {
    Job job;
    bool have = false;
    {
      // Among queued jobs whose slab has landed, take the lowest block: the
      // next step's forward consumes blocks in ascending order while the
      // backward exports them in descending order.
      std::unique_lock<std::mutex> lk(m->amu);
      m->acv.wait(lk, [m] { return m->stopping || !m->jobs.empty(); });
      if (m->jobs.empty()) return;
      // Jobs of one block run in pass order (they share its FP32 accumulator):
      // only the first queued job of each block is eligible.
      auto best = m->jobs.end();
      std::vector<int32_t> seen;
      for (auto it = m->jobs.begin(); it != m->jobs.end(); ++it) {
        if (std::find(seen.begin(), seen.end(), it->block) != seen.end()) continue;
        seen.push_back(it->block);
        const cudaError_t q = cudaEventQuery(m->SR[(size_t)it->slab]);
        if (q == cudaSuccess) {
          if (best == m->jobs.end() || it->block < best->block) best = it;
        } else if (q != cudaErrorNotReady) {
          best = it;  // let the wait below report the error
          break;
        }
      }
      if (best != m->jobs.end()) {
        job = *best;
        m->jobs.erase(best);
        have = true;
      }
    }
    if (!have) {
      if (!idle) {
        idle = true;
        idle_since = Clock::now();
      } else if (Clock::now() - idle_since > std::chrono::milliseconds(m->c.timeout_ms)) {
        set_err(m, MT_ERR_TIMEOUT, "timed out waiting for any gradient slab to land");
        std::lock_guard<std::mutex> lk(m->amu);
        m->slab_free.assign(m->slab_free.size(), 1);
        m->inflight_jobs = 0;
        m->jobs.clear();
        m->acv.notify_all();
        continue;
      }
      std::this_thread::sleep_for(std::chrono::microseconds(20));
      continue;
    }
    idle = false;
    if (const int d = g_inj_adam_delay_ms.load()) std::this_thread::sleep_for(std::chrono::milliseconds(d));
    const auto t0 = Clock::now();
    Nvtx range("ADAM block %d (slab %d)", job.block, job.slab);
    mt_status st = m->failed ? MT_ERR_STATE : wait_event(m, m->SR[(size_t)job.slab], "slab ready");
    if (st == MT_OK) {
      const mth::BlockDesc& b = m->lay[(size_t)job.block];
      uint8_t* blk = m->store + b.store_off;
      const uint16_t* slab = reinterpret_cast<const uint16_t*>(m->slabs + (size_t)job.slab * m->wb_max);
      uint16_t* G = reinterpret_cast<uint16_t*>(blk + b.region[1]);
      uint16_t* W = reinterpret_cast<uint16_t*>(blk + b.region[0]);
      float* th = reinterpret_cast<float*>(blk + b.region[2]);
      float* mm = reinterpret_cast<float*>(blk + b.region[3]);
      float* vv = reinterpret_cast<float*>(blk + b.region[4]);
      // work items: (tensor, chunk) ranges of at most 1 Mi elements; in an MoE
      // block each expert's row is its own range, and an expert no token was
      // routed to takes a zero gradient (its slab range was not exported)
      // 256 Ki-element chunks: a pack queued ahead of them waits at most for
      // the chunks already running (about 0.5 ms each)
      constexpr int64_t CH = 1 << 18;
      struct Item {
        int64_t o, n;
        bool zero;
      };
      std::vector<Item> items;
      auto add_range = [&](int64_t o, int64_t n, bool zero) {
        for (int64_t e = 0; e < n; e += CH) items.push_back({o + e, (n - e) < CH ? (n - e) : CH, zero});
      };
      for (int t = 0; t < b.nt; ++t) {
        const int64_t o = b.t[t].off, n = b.t[t].rows * b.t[t].cols;
        if (!job.routed.empty() && t == 3) {
          for (int64_t e = 0; e < b.t[t].rows; ++e) add_range(o + e * b.t[t].cols, b.t[t].cols, !job.routed[(size_t)e]);
        } else {
          add_range(o, n, false);
        }
      }
      const mt_config& c = m->c;
      bool inject_throw = false;
      if (g_inj_adam_throw.load() > 0) {
        g_inj_adam_throw--;
        inject_throw = true;
      }
      const bool last = job.pass + 1 == m->npass;
      float* acc = m->gacc ? m->gacc + m->gacc_off[(size_t)job.block] : nullptr;
      std::function<void(int64_t)> fn = [&](int64_t i) {
        if (inject_throw && i == 0) throw std::runtime_error("injected host worker fault");
        const int64_t o = items[(size_t)i].o, n = items[(size_t)i].n;
        if (!acc) {
          mth::adam(n, items[(size_t)i].zero ? nullptr : slab + o, c.keep_host_grad ? G + o : nullptr, th + o, mm + o,
                    vv + o, W + o, job.t, c.lr, c.beta1, c.beta2, c.adam_eps, c.weight_decay);
        } else if (!last) {
          mth::accumulate(n, slab + o, acc + o, job.pass == 0);
        } else {
          mth::adam_acc(n, slab + o, acc + o, c.keep_host_grad ? G + o : nullptr, th + o, mm + o, vv + o, W + o,
                        job.t, c.lr, c.beta1, c.beta2, c.adam_eps, c.weight_decay);
        }
      };
      std::string werr;
      if (!m->pool.parallel_for((int64_t)items.size(), fn, &werr))
        st = set_err(m, MT_ERR_INTERNAL, "host Adam worker: " + werr);
    }
    m->adam_us += std::chrono::duration_cast<std::chrono::microseconds>(Clock::now() - t0).count();
    if (m->tracing) {
      const double a = std::chrono::duration<double, std::milli>(t0.time_since_epoch()).count();
      const double e = now_ms();
      std::lock_guard<std::mutex> lk(m->tmu);
      m->thost.push_back({a - m->trace_host_base, e - m->trace_host_base, job.block, job.pass, (int64_t)job.t - 1});
    }
    {
      std::lock_guard<std::mutex> lk(m->amu);
      if (st == MT_OK && job.pass + 1 == m->npass) m->adam_done[(size_t)job.block] = job.t;
      m->slab_free[(size_t)job.slab] = 1;
      m->inflight_jobs--;
    }
    m->acv.notify_all();
  }
}

// Host waits (bounded) until block j has had Adam step t applied.
mt_status wait_adam(mt_model* m, int j, int64_t t) {
  std::unique_lock<std::mutex> lk(m->amu);
  const bool ok = m->acv.wait_for(lk, std::chrono::milliseconds(m->c.timeout_ms),
                                  [&] { return m->failed || m->adam_done[(size_t)j] >= t; });
  if (m->failed) return MT_ERR_STATE;
  if (!ok) return set_err(m, MT_ERR_TIMEOUT, "timed out waiting for Adam of block " + std::to_string(j));
  return MT_OK;
}

// Takes the lowest-numbered free slab, waiting (bounded) while all are held.
mt_status acquire_slab(mt_model* m, int* k) {
  std::unique_lock<std::mutex> lk(m->amu);
  auto any_free = [&] {
    for (size_t i = 0; i < m->slab_free.size(); ++i)
      if (m->slab_free[i]) return true;
    return false;
  };
  const bool ok = m->acv.wait_for(lk, std::chrono::milliseconds(m->c.timeout_ms),
                                  [&] { return m->failed || any_free(); });
  if (m->failed) return MT_ERR_STATE;
  if (!ok) return set_err(m, MT_ERR_TIMEOUT, "timed out waiting for a free gradient slab");
  for (size_t i = 0; i < m->slab_free.size(); ++i)
    if (m->slab_free[i]) {
      m->slab_free[i] = 0;
      *k = (int)i;
      return MT_OK;
    }
  return set_err(m, MT_ERR_INTERNAL, "slab bookkeeping");
}

// ---------------------------------------------------------------- visit pieces
int nvisits(const mt_model* m) { return (int)m->plan.size(); }
int visit_block(const mt_model* m, int v) { return m->plan[(size_t)v].j; }
int visit_kind(const mt_model* m, int v) { return m->plan[(size_t)v].kind; }

// The token data of pass p (from mt_set_tokens' pinned copy) to the device,
// on the compute stream ahead of the embedding forward that reads it.
mt_status upload_tokens(mt_model* m, int p) {
  const int64_t T = m->T;
  const int32_t* h = m->htok + (int64_t)p * (3 * T + m->V + 1);
  CU(m, cudaMemcpyAsync(m->d.tok, h, (size_t)T * 4, cudaMemcpyHostToDevice, m->sc));
  CU(m, cudaMemcpyAsync(m->d.tgt, h + T, (size_t)T * 4, cudaMemcpyHostToDevice, m->sc));
  CU(m, cudaMemcpyAsync(m->d.csr_start, h + 2 * T, (size_t)(m->V + 1) * 4, cudaMemcpyHostToDevice, m->sc));
  CU(m, cudaMemcpyAsync(m->d.csr_rows, h + 2 * T + m->V + 1, (size_t)T * 4, cudaMemcpyHostToDevice, m->sc));
  if (p + 1 == m->npass) CU(m, cudaEventRecord(m->TOK, m->sc));
  m->h2d += (3 * T + m->V + 1) * 4;
  return MT_OK;
}

bool moe_block(const mt_model* m, int j) { return m->moe && j >= 1 && j <= m->L; }

// Byte ranges, inside a block's W (or G) region, that a copy moves: the whole
// region, or for an MoE block the shared tensors (`trunk`: everything but
// W_experts) and/or the rows of the experts its forward routed tokens to
// (`experts`, from the counts in hcounts; adjacent rows merged).
struct Range {
  int64_t off, bytes;
};
std::vector<Range> block_ranges(const mt_model* m, int j, bool trunk, bool experts) {
  const mth::BlockDesc& bd = m->lay[(size_t)j];
  if (!moe_block(m, j)) return {{0, bd.wbytes}};
  const mth::TensorDesc& ex = bd.t[3];
  const int64_t e0 = ex.off * 2, row = ex.cols * 2, e1 = e0 + ex.rows * row;
  std::vector<Range> r;
  auto add = [&](int64_t off, int64_t bytes) {
    if (bytes <= 0) return;
    if (!r.empty() && r.back().off + r.back().bytes == off) r.back().bytes += bytes;
    else r.push_back({off, bytes});
  };
  if (trunk) add(0, e0);
  if (experts) {
    const int32_t* cnt = m->hcounts + (size_t)j * m->E;
    for (int e = 0; e < m->E; ++e)
      if (cnt[e] > 0) add(e0 + e * row, row);
  }
  if (trunk) add(e1, bd.wbytes - e1);
  return r;
}

constexpr int64_t kPackChunk = (int64_t)64 << 20;  // bytes packed before their copy is enqueued

// Host-to-device copy of the given ranges of block j's W region into device
// buffer b on the weight stream.  With the just-in-time pack (src pageable)
// each 64 MiB chunk is first copied into pinned staging b -- in 4 MiB pieces,
// enough for every worker, queued ahead of any Adam work, with the driver
// thread copying too -- and its device copy is enqueued as soon as it is
// packed, so the pack of a chunk overlaps the transfer of the previous one.
mt_status copy_ranges(mt_model* m, int b, const uint8_t* src, const std::vector<Range>& rg, bool pack) {
  constexpr int64_t PIECE = (int64_t)4 << 20;
  uint8_t* stage = m->staging[b];
  for (const Range& r : rg)
    for (int64_t c0 = 0; c0 < r.bytes;) {
      const int64_t chunk = pack ? kPackChunk : r.bytes;  // a pinned store copies each range at once
      const int64_t off = r.off + c0, len = std::min(chunk, r.bytes - c0);
      c0 += len;
      const uint8_t* from = src + off;
      if (pack) {
        const double t0 = now_ms();
        const int64_t np = (len + PIECE - 1) / PIECE;
        std::function<void(int64_t)> fn = [&](int64_t i) {
          const int64_t o = off + i * PIECE;
          std::memcpy(stage + o, src + o, (size_t)std::min(PIECE, off + len - o));
        };
        std::string werr;
        if (!m->pool.parallel_for(np, fn, &werr, true)) return set_err(m, MT_ERR_INTERNAL, "pack: " + werr);
        m->pack_ms += now_ms() - t0;
        from = stage + off;
      }
      CU(m, cudaMemcpyAsync(m->d.buf[b] + off, from, (size_t)len, cudaMemcpyHostToDevice, m->sw));
      m->h2d += len;
    }
  return MT_OK;
}

mt_status do_stream_in(mt_model* m, int j, int b) {
  const VisitDesc& vd = m->plan[(size_t)m->vis];
  const bool fwd = vd.kind <= V_HEAD;
  const bool copies = !(j == 0 && vd.kind == V_BWD);
  const mth::BlockDesc& bd = m->lay[(size_t)j];
  if (fwd && m->steps_done > 0 && m->pass == 0) {
    logop(m, "H", "WAIT_ADAM", j, -1);
    if (m->live) OK(wait_adam(m, j, m->steps_done));
  }
  const uint8_t* src = m->live ? m->store + bd.store_off + bd.region[0] : nullptr;
  // an MoE block's forward copies the shared tensors now and the routed
  // experts once the router has chosen; recompute and backward visits know
  // the forward's routing and copy both
  const std::vector<Range> rg = m->live ? block_ranges(m, j, true, !fwd) : std::vector<Range>{};
  const bool pack = copies && !m->c.pin_store;
  if (pack) {
    if (m->used[b]) {
      logop(m, "H", "WAIT_STAGE", b, -1);
      if (m->live) OK(wait_event(m, m->WR[b], "staging free"));
      if (m->live && m->moe) OK(wait_event(m, m->ER[b], "staging free (experts)"));
    }
    // the pack itself runs chunk by chunk inside the copy below (each chunk
    // packed before its device copy is enqueued)
    logop(m, "H", "PACK", j, b);
  }
  logop(m, "W", "WAIT_BF", b, -1);
  if (m->live) CU(m, cudaStreamWaitEvent(m->sw, m->BF[b], 0));
  std::unique_ptr<TraceSpan> trace_in(new TraceSpan(m, m->sw, 'W', TR_H2D, j));
  if (copies) {
    logop(m, "W", "H2D", j, b);
    if (m->live) OK(copy_ranges(m, b, src, rg, pack));
  }
  if (vd.first && m->c.ckpt_on_host) {
    // The segment's checkpoint X_s (s = j - 1) into slot seg % 2, after the
    // gradient stream finished saving it (XS of the ring slot it left from).
    const int s = j - 1, q = vd.seg % 2;
    logop(m, "W", "WAIT_XS", s % 2, -1);
    if (m->live) CU(m, cudaStreamWaitEvent(m->sw, m->XS[s % 2], 0));
    logop(m, "W", "H2D_CKPT", j, q);
    if (m->live) {
      const size_t bytes = (size_t)m->T * m->H * 2;
      CU(m, cudaMemcpyAsync(m->d.xck[q], m->ckpt + (size_t)(s / m->ci) * bytes, bytes, cudaMemcpyHostToDevice,
                            m->sw));
      m->h2d += (int64_t)bytes;
    }
  }
  trace_in.reset();  // the span ends before Weights-Ready releases the compute stream
  logop(m, "W", "REC_WR", b, -1);
  if (m->live) CU(m, cudaEventRecord(m->WR[b], m->sw));
  m->used[b] = true;
  return MT_OK;
}

mt_status do_bind(mt_model* m, int j, int b, mt_layer_view* out) {
  logop(m, "C", "WAIT_WR", b, -1);
  if (m->live) CU(m, cudaStreamWaitEvent(m->sc, m->WR[b], 0));
  if (out) {
    std::memset(out, 0, sizeof *out);
    out->block = j;
    out->buf = b;
    if (m->live) {
      const View v = make_view(m, j, b);
      out->n_tensors = m->lay[(size_t)j].nt;
      for (int t = 0; t < out->n_tensors; ++t) {
        out->w[t] = v.w[t];
        out->g[t] = v.g[t];
      }
    }
  }
  return MT_OK;
}

// Forward visit of an MoE block ([Lilting] MoE section: after the router has
// chosen, only the chosen experts' parameters go to the GPU):
//   compute: attention half, router, routing plan; the per-expert counts to
//            pinned host memory; Route-Ready;
//   host   : waits Route-Ready, reads which experts have tokens;
//   weight : copies those experts' rows into buffer b; Experts-Ready[b];
//   compute: waits Experts-Ready[b]; the experts and the combine.
mt_status moe_forward_visit(mt_model* m, int j, int b) {
  const View v = m->live ? make_view(m, j, b) : View{};
  const MoeShape q = moe_shape(m);
  if (m->live) {
    OK(attention_half(m, v, x_fwd_in(m, j)));
    OK(moe_route(m, q, m->d.moe, m->d.yn, v.w[2], m->sc));
    CU(m, cudaMemcpyAsync(m->hcounts + (size_t)j * m->E, m->d.moe.p.counts, (size_t)m->E * 4, cudaMemcpyDeviceToHost,
                          m->sc));
  }
  logop(m, "C", "REC_RT", j, -1);
  if (m->live) CU(m, cudaEventRecord(m->RT, m->sc));
  logop(m, "H", "WAIT_RT", j, -1);
  if (m->live) OK(wait_event(m, m->RT, "routing"));
  const mth::BlockDesc& bd = m->lay[(size_t)j];
  const std::vector<Range> rg = m->live ? block_ranges(m, j, false, true) : std::vector<Range>{};
  const uint8_t* src = m->live ? m->store + bd.store_off + bd.region[0] : nullptr;
  if (!m->c.pin_store) logop(m, "H", "PACK_EXP", j, b);  // packed chunk by chunk in the copy below
  logop(m, "W", "H2D_EXP", j, b);
  if (m->live) {
    TraceSpan trace_exp(m, m->sw, 'W', TR_H2D_EXP, j);
    OK(copy_ranges(m, b, src, rg, !m->c.pin_store));
  }
  logop(m, "W", "REC_ER", b, -1);
  if (m->live) CU(m, cudaEventRecord(m->ER[b], m->sw));
  logop(m, "C", "WAIT_ER", b, -1);
  if (m->live) CU(m, cudaStreamWaitEvent(m->sc, m->ER[b], 0));
  logop(m, "C", "FWD_EXP", j, b);
  if (m->live)
    OK(moe_experts_fwd(m, q, m->d.moe, moe_route_of(m, j), m->d.yn, m->d.x1, v.w[3], x_out(m, j), m->sc));
  return MT_OK;
}

mt_status do_forward(mt_model* m, int j, int b) {
  const bool head = j == m->L + 1;
  const bool writes_x = j <= m->L;
  const bool ckh = m->c.ckpt_on_host != 0;
  if (writes_x && ckh) {
    logop(m, "C", "WAIT_XS", j % 2, -1);
    if (m->live) CU(m, cudaStreamWaitEvent(m->sc, m->XS[j % 2], 0));
  }
  logop(m, "C", head ? "HEAD" : "FWD", j, b);
  std::unique_ptr<TraceSpan> trace_c(new TraceSpan(m, m->sc, 'C', TR_COMPUTE + (head ? V_HEAD : V_FWD), j));
  if (moe_block(m, j)) {
    OK(moe_forward_visit(m, j, b));
  } else if (m->live) {
    const View v = make_view(m, j, b);
    if (j == 0) {
      OK(upload_tokens(m, m->pass));
      Timed t(m, K_OTHER, 0, 4.0 * m->T * m->H);
      CU(m, mt::embed_fwd(m->d.tok, v.w[0], m->T, m->H, m->V, x_out(m, 0), m->sc));
    } else if (!head) {
      OK(decoder_forward(m, v, x_fwd_in(m, j), x_out(m, j), false, j));
    } else {
      OK(head_forward_backward(m, v, x_fwd_in(m, j), m->d.dx[m->L % 2]));
    }
  }
  trace_c.reset();  // the span ends before the events that release other streams
  const bool saves = writes_x && j < m->L && j % m->ci == 0 && ckh;
  if (saves) {
    logop(m, "C", "REC_XR", j % 2, -1);
    if (m->live) CU(m, cudaEventRecord(m->XR[j % 2], m->sc));
  }
  if (!head) {
    logop(m, "C", "REC_BF", b, -1);
    if (m->live) CU(m, cudaEventRecord(m->BF[b], m->sc));
  } else {
    logop(m, "C", "REC_BD", b, -1);
    if (m->live) CU(m, cudaEventRecord(m->BD[b], m->sc));
  }
  if (saves) {
    const int s = j % 2;
    logop(m, "G", "WAIT_XR", s, -1);
    if (m->live) CU(m, cudaStreamWaitEvent(m->sg, m->XR[s], 0));
    logop(m, "G", "D2H_CKPT", j, s);
    if (m->live) {
      TraceSpan trace_ck(m, m->sg, 'G', TR_D2H_CKPT, j);
      const size_t bytes = (size_t)m->T * m->H * 2;
      CU(m, cudaMemcpyAsync(m->ckpt + (size_t)(j / m->ci) * bytes, m->d.xslot[s], bytes, cudaMemcpyDeviceToHost,
                            m->sg));
      m->d2h += (int64_t)bytes;
    }
    logop(m, "G", "REC_XS", s, -1);
    if (m->live) CU(m, cudaEventRecord(m->XS[s], m->sg));
  }
  return MT_OK;
}

// Forward of layer j inside the backward, rebuilding X_j of its segment.
mt_status do_recompute(mt_model* m, int j, int b) {
  const int seg = m->plan[(size_t)m->vis].seg;
  logop(m, "C", "RECOMP", j, b);
  if (m->live) {
    TraceSpan trace_c(m, m->sc, 'C', TR_COMPUTE + V_RECOMP, j);
    OK(decoder_forward(m, make_view(m, j, b), x_seg_in(m, j, seg), x_seg_out(m, j), false, j));
  }
  logop(m, "C", "REC_BF", b, -1);
  if (m->live) CU(m, cudaEventRecord(m->BF[b], m->sc));
  return MT_OK;
}

mt_status do_backward(mt_model* m, int j, int b) {
  logop(m, "C", "BWD", j, b);
  if (m->live) {
    TraceSpan trace_c(m, m->sc, 'C', TR_COMPUTE + V_BWD, j);
    const View v = make_view(m, j, b);
    if (j == 0) {
      Timed t(m, K_OTHER, 0, 2.0 * m->T * m->H + 2.0 * m->V * m->H);
      CU(m, mt::embed_bwd(m->d.csr_start, m->d.csr_rows, m->d.dx[0], m->V, m->H, v.g[0], m->sc));
    } else {
      const int seg = m->plan[(size_t)m->vis].seg;
      OK(decoder_backward(m, v, x_seg_in(m, j, seg), m->d.dx[j % 2], m->d.dx[(j - 1) % 2], j));
    }
  }
  logop(m, "C", "REC_BD", b, -1);
  if (m->live) CU(m, cudaEventRecord(m->BD[b], m->sc));
  return MT_OK;
}

mt_status do_stream_out(mt_model* m, int j, int b, int* slab_out) {
  int k = 0;  // a dry run has no Adam: its slabs free at once and slab 0 is always taken
  m->exports++;
  const mth::BlockDesc& bd = m->lay[(size_t)j];
  logop(m, "G", "WAIT_BD", b, -1);
  if (m->live) CU(m, cudaStreamWaitEvent(m->sg, m->BD[b], 0));
  if (m->live) OK(acquire_slab(m, &k));
  logop(m, "H", "ACQ_SLAB", k, -1);
  logop(m, "G", "D2H", j, k);
  if (m->live) {  // an MoE block exports the shared tensors and the routed experts only
    TraceSpan trace_out(m, m->sg, 'G', TR_D2H, j);
    for (const Range& r : block_ranges(m, j, true, true)) {
      CU(m, cudaMemcpyAsync(m->slabs + (size_t)k * m->wb_max + r.off, m->d.buf[b] + bd.region[1] + r.off,
                            (size_t)r.bytes, cudaMemcpyDeviceToHost, m->sg));
      m->d2h += r.bytes;
    }
  }
  logop(m, "G", "REC_BF", b, -1);
  if (m->live) CU(m, cudaEventRecord(m->BF[b], m->sg));
  logop(m, "G", "REC_SR", k, -1);
  if (m->live) CU(m, cudaEventRecord(m->SR[(size_t)k], m->sg));
  if (slab_out) *slab_out = k;
  return MT_OK;
}

mt_status do_adam_enqueue(mt_model* m, int j, int k, int32_t t) {
  logop(m, "H", m->pass + 1 < m->npass ? "ACCUM_ENQ" : "ADAM_ENQ", j, k);
  if (m->live) {
    {
      std::lock_guard<std::mutex> lk(m->amu);
      Job job{j, k, t, m->pass, {}};
      if (moe_block(m, j)) {
        job.routed.resize((size_t)m->E);
        for (int e = 0; e < m->E; ++e) job.routed[(size_t)e] = m->hcounts[(size_t)j * m->E + e] > 0;
      }
      m->jobs.push_back(std::move(job));
      m->inflight_jobs++;
    }
    m->acv.notify_all();
  }
  return MT_OK;
}

// Sub-stages of a visit: 0 stream_in, 1 bind, 2 compute, 3 stream_out, 4 adam.
bool exports_grad(const mt_model* m, int v) {
  const int k = visit_kind(m, v);
  return k == V_BWD || k == V_HEAD;
}

void advance(mt_model* m) {
  const bool exp = exports_grad(m, m->vis);
  if ((!exp && m->stage == 2) || (exp && m->stage == 4)) {
    m->stage = 0;
    if (++m->vis == nvisits(m)) {
      m->vis = 0;
      if (++m->pass == m->npass) {
        m->pass = 0;
        m->steps_done++;
      }
    }
  } else {
    m->stage++;
  }
}

mt_status expect(mt_model* m, int stage, int block) {
  if (m->failed) return MT_ERR_STATE;
  if (m->stage != stage || visit_block(m, m->vis) != block)
    return set_err(m, MT_ERR_STATE, "call out of order: expected stage " + std::to_string(m->stage) +
                                        " of block " + std::to_string(visit_block(m, m->vis)),
                   false);
  return MT_OK;
}

mt_status run_visit(mt_model* m) {
  const int v = m->vis, j = visit_block(m, v), b = v % m->nbuf, kind = visit_kind(m, v);
  static const char* kname[] = {"FWD %d (buffer %d)", "HEAD %d (buffer %d)", "RECOMP %d (buffer %d)",
                                "BWD %d (buffer %d)"};
  Nvtx range(kname[kind], j, b);
  OK(do_stream_in(m, j, b));
  advance(m);
  OK(do_bind(m, j, b, nullptr));
  advance(m);
  cudaEvent_t ta = nullptr;
  if (m->live && m->timing) {  // per-visit compute time, after the Weights-Ready wait
    ta = take_event(m);
    CU(m, cudaEventRecord(ta, m->sc));
  }
  // the first step's per-visit compute times feed the schedule's second plan
  const bool first = m->live && m->steps_done == 0 && m->pass == 0 && (size_t)v < m->first_ev.size();
  if (first) CU(m, cudaEventRecord(m->first_ev[(size_t)v].first, m->sc));
  if (kind <= V_HEAD) OK(do_forward(m, j, b));
  else if (kind == V_RECOMP) OK(do_recompute(m, j, b));
  else OK(do_backward(m, j, b));
  if (first) {
    CU(m, cudaEventRecord(m->first_ev[(size_t)v].second, m->sc));
    m->first_rec[(size_t)v] = 1;
  }
  if (ta) {
    cudaEvent_t tb = take_event(m);
    CU(m, cudaEventRecord(tb, m->sc));
    m->pend.push_back({ta, tb, -1, v, 0.0, 0.0});
  }
  const bool exp = exports_grad(m, v);
  const int64_t t = m->steps_done + 1;
  advance(m);
  if (exp) {
    int k = 0;
    OK(do_stream_out(m, j, b, &k));
    advance(m);
    OK(do_adam_enqueue(m, j, k, (int32_t)t));
    advance(m);
  }
  return MT_OK;
}

void compute_tables(mt_model* m, std::vector<float>& cs) {
  const int half = m->hd / 2;
  cs.resize((size_t)m->S * m->hd);
  for (int p = 0; p < m->S; ++p)
    for (int i = 0; i < half; ++i) {
      const double th = std::pow((double)m->c.rope_base, -2.0 * i / (double)m->hd);
      const double a = (double)p * th;
      cs[((size_t)p * half + i) * 2] = (float)std::cos(a);
      cs[((size_t)p * half + i) * 2 + 1] = (float)std::sin(a);
    }
}

void fill_shape(mt_model* m) {
  const mt_config& c = m->c;
  m->L = c.n_layers; m->H = c.hidden; m->nh = c.n_heads; m->nkv = c.n_kv_heads; m->hd = c.head_dim;
  m->F = c.ffn; m->V = c.vocab; m->B = c.batch; m->S = c.seq; m->M = c.micro_batches;
  m->Nqkv = (m->nh + 2 * m->nkv) * m->hd;
  m->moe = c.n_experts > 0;
  m->E = c.n_experts; m->topk = c.top_k; m->Fe = c.expert_ffn;
  m->T = mth::tokens_per_pass(&c);  // device tokens of one pass
  m->npass = mth::passes_per_step(&c);
  m->Mp = c.host_grad_accum ? 1 : c.micro_batches;
  m->chunk = head_chunk(&c, m->T);
  m->lay = mth::build_layout(&c);
  m->wb_max = 0;
  for (auto& b : m->lay) m->wb_max = b.wbytes > m->wb_max ? b.wbytes : m->wb_max;
  m->K = c.n_grad_slabs > 0 ? c.n_grad_slabs : 12;  // mt_init_model plans it when 0
  m->nbuf = c.n_buffers;
  m->ci = c.ckpt_interval;
  m->nseg = (m->L + m->ci - 1) / m->ci;
  m->plan = build_plan(m->L, m->ci);
}

// ---------------------------------------------------------------- static schedule
// Tensor FLOPs of a visit's compute (forward: 2 t P_mm + causal attention
// 2 B nh hd S^2; backward: recompute without the last projection, 4 t P_mm
// and 7 B nh hd S^2 of attention; head: 6 t H V).
double visit_flops(const mt_model* m, int kind, int j) {
  const double T = (double)m->T, H = m->H, nh = m->nh, nkv = m->nkv, hd = m->hd;
  const double att = (double)m->Mp * m->B * nh * hd * (double)m->S * m->S;
  const double mlp = m->moe ? (double)m->topk * 3.0 * H * m->Fe + (double)m->E * H : 3.0 * H * m->F;
  const double last = m->moe ? (double)m->topk * H * m->Fe : H * m->F;  // down projection
  const double pmm = H * (nh + 2 * nkv) * hd + nh * hd * H + mlp;
  if (j == 0) return 0.0;
  if (j == m->L + 1) return 6.0 * T * H * m->V;
  if (kind == V_BWD) return 2.0 * T * (pmm - last) + 4.0 * T * pmm + 7.0 * att;
  return 2.0 * T * pmm + 2.0 * att;
}

// Per-visit schedule inputs of one pass; c[] estimated from FLOPs at the
// assumed rate until measured (plus a fixed 0.2 ms of launches and
// memory-bound kernels per visit).
constexpr double kAssumedFlops = 1.2e15;
void sched_inputs(mt_model* m) {
  const int n = nvisits(m);
  m->sk_kind.assign((size_t)n, 0);
  m->sk_block.assign((size_t)n, 0);
  m->sk_b.assign((size_t)n, 0.0);
  m->sk_p.assign((size_t)n, 0.0);
  m->sk_d.assign((size_t)n, 0.0);
  m->sk_c.assign((size_t)n, 0.0);
  m->sk_a.assign((size_t)n, 0.0);
  for (int v = 0; v < n; ++v) {
    const VisitDesc& vd = m->plan[(size_t)v];
    const mth::BlockDesc& bd = m->lay[(size_t)vd.j];
    const bool copies = !(vd.j == 0 && vd.kind == V_BWD);
    double b = copies ? (double)bd.wbytes : 0.0;
    if (vd.first && m->c.ckpt_on_host) b += (double)m->T * m->H * 2;
    m->sk_kind[(size_t)v] = vd.kind;
    m->sk_block[(size_t)v] = vd.j;
    m->sk_b[(size_t)v] = b;
    m->sk_p[(size_t)v] = (!m->c.pin_store && copies) ? (double)bd.wbytes : 0.0;
    const bool exp = vd.kind == V_HEAD || vd.kind == V_BWD;
    m->sk_d[(size_t)v] = exp ? (double)bd.wbytes : 0.0;
    m->sk_a[(size_t)v] = exp ? (double)bd.n_pad : 0.0;
    m->sk_c[(size_t)v] = visit_flops(m, vd.kind, vd.j) / kAssumedFlops + 2e-4;
  }
  mth::SimIn& in = m->sim;
  in.n = n;
  in.kind = m->sk_kind.data();
  in.block = m->sk_block.data();
  in.b = m->sk_b.data();
  in.p = m->sk_p.data();
  in.d = m->sk_d.data();
  in.c = m->sk_c.data();
  in.a = m->sk_a.data();
  in.nbuf = m->nbuf;
  in.chunk = (double)kPackChunk;
}

void fill_plan_out(const mth::Plan& pl, const mth::SimIn& in, int measured, mt_sched_plan* o) {
  o->K = pl.K;
  o->measured = measured;
  o->period_ms = pl.out.period * 1e3;
  o->stall_ms = pl.out.stall * 1e3;
  o->adam_busy_ms = pl.out.adam_busy * 1e3;
  o->slab_wait_ms = pl.out.slab_wait * 1e3;
  o->pack_ms = pl.out.pack * 1e3;
  o->adam_gelem_s = pl.out.adam_rate / 1e9;
  o->bw_h2d_gbs = in.bw_h2d / 1e9;
  o->bw_d2h_gbs = in.bw_d2h / 1e9;
  o->pack_gbs = in.pack_rate / 1e9;
  o->adam_gelem_s_idle = in.adam_rate / 1e9;
  o->host_gbs = in.host_bw / 1e9;
}

// Init-time measurements for the schedule: pinned copies over the link in
// each direction on the model's streams (best of three), the pool's pack rate
// (pageable store into pinned memory), host Adam on scratch arrays over the
// pool on an idle host, and the same Adam while both link directions copy,
// which gives the bytes host memory serves to CPU and DMA together.  A failed
// probe leaves its rate at 0 (the model then treats that stage as free).
void run_probes(mt_model* m) {
  mth::SimIn& in = m->sim;
  in.adam_bytes = m->c.keep_host_grad ? 30.0 : 28.0;
  const size_t bytes = (size_t)std::min<int64_t>((int64_t)64 << 20, m->wb_max);
  void* hp = nullptr;
  if (cudaHostAlloc(&hp, bytes, cudaHostAllocDefault) != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (cudaEventCreate(&e0) == cudaSuccess && cudaEventCreate(&e1) == cudaSuccess) {
    for (int dir = 0; dir < 2; ++dir) {
      cudaStream_t st = dir == 0 ? m->sw : m->sg;
      float best = 1e30f;
      for (int r = 0; r < 3; ++r) {
        cudaEventRecord(e0, st);
        if (dir == 0) cudaMemcpyAsync(m->d.buf[0], hp, bytes, cudaMemcpyHostToDevice, st);
        else cudaMemcpyAsync(hp, m->d.buf[0], bytes, cudaMemcpyDeviceToHost, st);
        cudaEventRecord(e1, st);
        float ms = 0;
        if (cudaEventSynchronize(e1) == cudaSuccess && cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess && ms > 0)
          best = std::min(best, ms);
      }
      if (best < 1e30f) (dir == 0 ? in.bw_h2d : in.bw_d2h) = (double)bytes / (best * 1e-3);
    }
  }
  // the pack: the largest block's first `bytes` of W, in 4 MiB pieces over the pool
  const mth::BlockDesc* big = &m->lay[0];
  for (auto& b : m->lay)
    if (b.wbytes > big->wbytes) big = &b;
  const int64_t pb = std::min<int64_t>((int64_t)bytes, big->wbytes), PIECE = (int64_t)4 << 20;
  const uint8_t* src = m->store + big->store_off;
  std::function<void(int64_t)> cp = [&](int64_t i) {
    const int64_t o = i * PIECE;
    std::memcpy((uint8_t*)hp + o, src + o, (size_t)std::min(PIECE, pb - o));
  };
  double best = 1e30;
  std::string err;
  for (int r = 0; r < 3; ++r) {
    const double t0 = now_ms();
    if (m->pool.parallel_for((pb + PIECE - 1) / PIECE, cp, &err, true)) best = std::min(best, now_ms() - t0);
  }
  if (best > 0 && best < 1e30) in.pack_rate = (double)pb / (best * 1e-3);
  // Adam over the pool: 16 Mi elements, on an idle host and under DMA in both directions
  const int64_t nn = (int64_t)16 << 20;
  std::vector<float> th((size_t)nn, 0.01f), mm((size_t)nn, 0.0f), vv((size_t)nn, 0.0f);
  std::vector<uint16_t> g((size_t)nn, 0x3c00), w((size_t)nn, 0), gc(m->c.keep_host_grad ? (size_t)nn : 0, 0);
  uint16_t* gcp = m->c.keep_host_grad ? gc.data() : nullptr;
  constexpr int64_t CH = 1 << 18;
  int rep = 0;
  std::function<void(int64_t)> fn = [&](int64_t i) {
    const int64_t o = i * CH, len = std::min(CH, nn - o);
    mth::adam(len, g.data() + o, gcp ? gcp + o : nullptr, th.data() + o, mm.data() + o, vv.data() + o,
              w.data() + o, rep + 1, 1e-3f, 0.9f, 0.999f, 1e-8f, 0.f);
  };
  double idle = 1e30;
  for (rep = 0; rep < 3; ++rep) {
    const double t0 = now_ms();
    if (m->pool.parallel_for((nn + CH - 1) / CH, fn, &err)) idle = std::min(idle, now_ms() - t0);
  }
  if (idle > 0 && idle < 1e30) in.adam_rate = (double)nn / (idle * 1e-3);
  // shared host memory: copies in both link directions, sized to last about
  // eight idle Adam passes, while Adam makes passes until both copy streams
  // are done; the host's total rate is the copies' bytes over their window
  // plus Adam's bytes at the rate it kept meanwhile
  cudaEvent_t f0 = nullptr, f1 = nullptr;
  if (e0 && e1 && in.adam_rate > 0 && in.bw_h2d > 0 && in.bw_d2h > 0 && cudaEventCreate(&f0) == cudaSuccess &&
      cudaEventCreate(&f1) == cudaSuccess) {
    const double t_pass = (double)nn / in.adam_rate;
    const size_t half = bytes / 2;  // H2D from the first half of the buffer, D2H into the second
    const int nc = std::max(2, (int)std::ceil(8.0 * t_pass * std::min(in.bw_h2d, in.bw_d2h) / (double)half));
    cudaEventRecord(e0, m->sw);
    cudaEventRecord(f0, m->sg);
    for (int i = 0; i < nc; ++i) {
      cudaMemcpyAsync(m->d.buf[0], hp, half, cudaMemcpyHostToDevice, m->sw);
      cudaMemcpyAsync((uint8_t*)hp + half, m->d.buf[0] + half, half, cudaMemcpyDeviceToHost, m->sg);
    }
    cudaEventRecord(e1, m->sw);
    cudaEventRecord(f1, m->sg);
    const double t0 = now_ms();
    bool ok = true;
    int passes = 0;
    for (rep = 3; ok && passes < 64; ++rep) {
      ok = m->pool.parallel_for((nn + CH - 1) / CH, fn, &err);
      ++passes;
      if (cudaEventQuery(e1) == cudaSuccess && cudaEventQuery(f1) == cudaSuccess) break;
    }
    const double ta = (now_ms() - t0) * 1e-3;
    float mw = 0, mg = 0;
    if (ok && cudaEventSynchronize(e1) == cudaSuccess && cudaEventSynchronize(f1) == cudaSuccess &&
        cudaEventElapsedTime(&mw, e0, e1) == cudaSuccess && cudaEventElapsedTime(&mg, f0, f1) == cudaSuccess) {
      const double td = std::max(mw, mg) * 1e-3;
      // Adam ran through the copies' window (it stops within one pass of its end)
      if (td > 0 && ta > 0 && passes >= 2 && ta >= 0.8 * td)
        in.host_bw = 2.0 * nc * (double)half / td + in.adam_bytes * ((double)passes * nn / ta);
    }
  }
  if (f0) cudaEventDestroy(f0);
  if (f1) cudaEventDestroy(f1);
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  cudaFreeHost(hp);
  cudaGetLastError();  // a failed probe call must not surface at a later launch
}

// The plan with the slab count the config leaves open (n_grad_slabs = 0).
mth::Plan make_plan(const mt_model* m, int k_max_budget) {
  const int k = m->c.n_grad_slabs;
  return mth::plan(m->sim, k > 0 ? k : 1, k > 0 ? k : k_max_budget);
}

// Once the first step's per-visit compute events have completed: the second
// plan, on measured compute times (K itself is allocated already).
void replan_measured(mt_model* m) {
  if (m->have_plan1 || m->first_ev.empty() || m->npass != 1) return;
  for (size_t v = 0; v < m->first_ev.size(); ++v)
    if (!m->first_rec[v]) return;  // the first step did not run through mt_train_step
  std::vector<double> c(m->first_ev.size());
  for (size_t v = 0; v < m->first_ev.size(); ++v) {
    if (cudaEventQuery(m->first_ev[v].second) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    float ms = 0;
    if (cudaEventElapsedTime(&ms, m->first_ev[v].first, m->first_ev[v].second) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    c[v] = ms * 1e-3;
  }
  m->sk_c = c;
  m->sim.c = m->sk_c.data();
  mth::Plan pl;
  pl.K = m->K;
  pl.out = mth::simulate(m->sim, m->K, 4, nullptr);
  fill_plan_out(pl, m->sim, 1, &m->plan1);
  m->have_plan1 = true;
}

}  // namespace

mt_model::~mt_model() {
  {
    std::lock_guard<std::mutex> lk(amu);
    stopping = true;
  }
  acv.notify_all();
  if (adam_thr.joinable()) adam_thr.join();
  pool.stop();
  if (live) {
    if (sc) cudaStreamSynchronize(sc);
    if (sw) cudaStreamSynchronize(sw);
    if (sg) cudaStreamSynchronize(sg);
    for (cudaEvent_t* e : {&WR[0], &WR[1], &BD[0], &BD[1], &BF[0], &BF[1], &XR[0], &XR[1], &XS[0], &XS[1], &TOK, &LOSS,
                           &RT, &ER[0], &ER[1]})
      if (*e) cudaEventDestroy(*e);
    for (auto e : SR)
      if (e) cudaEventDestroy(e);
    for (auto& e : first_ev) {
      if (e.first) cudaEventDestroy(e.first);
      if (e.second) cudaEventDestroy(e.second);
    }
    for (auto& p : pend) {
      cudaEventDestroy(p.a);
      cudaEventDestroy(p.b);
    }
    for (auto e : ev_pool) cudaEventDestroy(e);
    for (auto& t : tdev) {
      cudaEventDestroy(t.a);
      cudaEventDestroy(t.b);
    }
    if (trace_base) cudaEventDestroy(trace_base);
    if (trace_stream) cudaStreamDestroy(trace_stream);
    if (registered) cudaHostUnregister(store);
    for (int b = 0; b < 2; ++b)
      if (staging[b]) cudaFreeHost(staging[b]);
    if (slabs) cudaFreeHost(slabs);
    if (ckpt) cudaFreeHost(ckpt);
    if (htok) cudaFreeHost(htok);
    if (hloss) cudaFreeHost(hloss);
    if (hcounts) cudaFreeHost(hcounts);
  }
  if (store) munmap(store, store_bytes);
  if (gacc) munmap(gacc, gacc_bytes);
}

// ======================================================================== C ABI
extern "C" {

mt_status mt_default_config(mt_config* c) {
  if (!c) return MT_ERR_ARG;
  std::memset(c, 0, sizeof *c);
  c->rope_base = 10000.0f;
  c->rms_eps = 1e-6f;
  c->init_std = 0.02f;
  c->micro_batches = 1;
  c->ckpt_interval = 1;
  c->ckpt_on_host = 1;
  c->n_buffers = 2;
  c->n_grad_slabs = 0;  // sized by the static schedule
  c->lr = 1e-3f;
  c->beta1 = 0.9f;
  c->beta2 = 0.999f;
  c->adam_eps = 1e-8f;
  c->seed = 1;
  c->timeout_ms = 60000;
  c->keep_host_grad = 1;
  return MT_OK;
}

mt_status mt_query_device_bytes(const mt_config* c, size_t* bytes) {
  if (!bytes || !mth::config_valid(c, nullptr)) return MT_ERR_ARG;
  Dev d;
  *bytes = carve(c, mth::build_layout(c), nullptr, &d);
  return MT_OK;
}

mt_status mt_init_model(const mt_config* c, mt_dev_region dev, mt_streams s, mt_model** out) {
  if (!out) return MT_ERR_ARG;
  *out = nullptr;
  std::string why;
  if (!mth::config_valid(c, &why)) return MT_ERR_ARG;
  if (!dev.base || !s.compute || !s.weight || !s.grad) return MT_ERR_ARG;
  std::unique_ptr<mt_model> m(new mt_model());
  m->c = *c;
  m->live = true;
  fill_shape(m.get());
  m->dev_base = (uint8_t*)dev.base;
  m->dev_bytes = dev.bytes;
  m->dev_used = carve(c, m->lay, nullptr, &m->d);
  if (m->dev_used > dev.bytes) return MT_ERR_DEVICE_OOM;
  carve(c, m->lay, m->dev_base, &m->d);
  m->sc = (cudaStream_t)s.compute;
  m->sw = (cudaStream_t)s.weight;
  m->sg = (cudaStream_t)s.grad;
  mt_model* mm = m.get();

  // host flat store: pageable anonymous memory, advised for huge pages
  for (auto& b : m->lay) m->store_bytes += (size_t)b.bytes;
  void* p = mmap(nullptr, m->store_bytes, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
  if (p == MAP_FAILED) return MT_ERR_HOST_OOM;
  m->store = (uint8_t*)p;
#ifdef MADV_HUGEPAGE
  madvise(p, m->store_bytes, MADV_HUGEPAGE);
#endif
  int nth = c->n_host_threads > 0 ? c->n_host_threads : (int)std::thread::hardware_concurrency();
  if (nth < 1) nth = 1;
  m->pool.start(nth);

  // initial values, in parallel over 4 Mi-element ranges (first touch included)
  {
    struct Item { int j; int64_t e0, e1; };
    std::vector<Item> items;
    for (int j = 0; j < (int)m->lay.size(); ++j)
      for (int64_t e = 0; e < m->lay[(size_t)j].n_pad; e += (4 << 20))
        items.push_back({j, e, std::min<int64_t>(m->lay[(size_t)j].n_pad, e + (4 << 20))});
    std::function<void(int64_t)> fn = [&](int64_t i) {
      const Item& it = items[(size_t)i];
      const mth::BlockDesc& b = mm->lay[(size_t)it.j];
      uint8_t* blk = mm->store + b.store_off;
      float* th = (float*)(blk + b.region[2]);
      mth::init_block(&mm->c, b, it.j, th, it.e0, it.e1);
      uint16_t* W = (uint16_t*)(blk + b.region[0]);
      uint16_t* G = (uint16_t*)(blk + b.region[1]);
      float* m1 = (float*)(blk + b.region[3]);
      float* v1 = (float*)(blk + b.region[4]);
      for (int64_t e = it.e0; e < it.e1; ++e) {
        W[e] = mth::bf16_rne(th[e]);
        G[e] = 0;
        m1[e] = 0.f;
        v1[e] = 0.f;
      }
    };
    std::string werr;
    if (!m->pool.parallel_for((int64_t)items.size(), fn, &werr)) return MT_ERR_INTERNAL;
  }
  // The static schedule ([Peter] 記憶體預取策略): per-visit bytes from the
  // layout, link / pack / Adam rates measured here, compute estimated from
  // FLOPs; it sizes the slab pool (n_grad_slabs = 0) within a tenth of the
  // host's memory and splits the host threads between packing and Adam.
  sched_inputs(m.get());
  run_probes(m.get());
  {
    const long pages = sysconf(_SC_PHYS_PAGES), psz = sysconf(_SC_PAGESIZE);
    const double phys = pages > 0 && psz > 0 ? (double)pages * (double)psz : 64e9;
    const int kbud = (int)std::max(2.0, std::min(32.0, std::floor(0.1 * phys / (double)m->wb_max)));
    const mth::Plan pl = make_plan(m.get(), kbud);
    m->K = c->n_grad_slabs > 0 ? c->n_grad_slabs : pl.K;
    fill_plan_out(pl, m->sim, 0, &m->plan0);
  }
  if (m->npass == 1) {
    m->first_ev.assign((size_t)nvisits(m.get()), {nullptr, nullptr});
    m->first_rec.assign((size_t)nvisits(m.get()), 0);
    for (auto& e : m->first_ev) {
      CU(mm, cudaEventCreate(&e.first));
      CU(mm, cudaEventCreate(&e.second));
    }
  }
  const size_t gb = c->debug_guards ? (size_t)kGuardBytes : 0;  // canary after each pinned region
  auto guard = [&](uint8_t* p, size_t bytes, const char* name) {
    if (!gb) return;
    std::memset(p + bytes, 0xA5, gb);
    m->hguards.push_back({p + bytes, name});
  };
  if (c->pin_store) {
    if (cudaHostRegister(m->store, m->store_bytes, cudaHostRegisterDefault) != cudaSuccess) return MT_ERR_HOST_OOM;
    m->registered = true;
  } else {
    for (int b = 0; b < m->nbuf; ++b) {
      if (pinned_alloc((void**)&m->staging[b], (size_t)m->wb_max + gb) != cudaSuccess)
        return MT_ERR_HOST_OOM;
      m->pinned_bytes += (size_t)m->wb_max;
      guard(m->staging[b], (size_t)m->wb_max, b ? "pinned staging 1" : "pinned staging 0");
    }
  }
  if (pinned_alloc((void**)&m->slabs, (size_t)m->wb_max * m->K + gb) != cudaSuccess)
    return MT_ERR_HOST_OOM;
  m->pinned_bytes += (size_t)m->wb_max * m->K;
  guard(m->slabs, (size_t)m->wb_max * m->K, "gradient slabs");
  if (c->ckpt_on_host) {
    const size_t bytes = (size_t)m->nseg * m->T * m->H * 2;  // X_0, X_c, X_2c, ...
    if (pinned_alloc((void**)&m->ckpt, bytes + gb) != cudaSuccess) return MT_ERR_HOST_OOM;
    m->pinned_bytes += bytes;
    guard(m->ckpt, bytes, "host checkpoints");
  }
  const size_t tokb = (size_t)m->npass * (3 * m->T + m->V + 1) * 4;  // per pass: tok | tgt | csr start | csr rows
  if (pinned_alloc((void**)&m->htok, tokb + gb) != cudaSuccess) return MT_ERR_HOST_OOM;
  guard((uint8_t*)m->htok, tokb, "pinned tokens");
  if (pinned_alloc((void**)&m->hloss, 64 + 4 * (size_t)m->npass) != cudaSuccess) return MT_ERR_HOST_OOM;
  if (m->npass > 1) {  // host FP32 gradient accumulator, one n_pad range per block
    int64_t n = 0;
    for (auto& b : m->lay) {
      m->gacc_off.push_back(n);
      n += b.n_pad;
    }
    m->gacc_bytes = (size_t)n * 4;
    void* p = mmap(nullptr, m->gacc_bytes, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
    if (p == MAP_FAILED) return MT_ERR_HOST_OOM;
    m->gacc = (float*)p;
  }
  m->pinned_bytes += tokb + 64;
  if (m->moe) {
    const size_t cb = (size_t)(m->L + 2) * m->E * 4;
    if (pinned_alloc((void**)&m->hcounts, cb) != cudaSuccess) return MT_ERR_HOST_OOM;
    std::memset(m->hcounts, 0, cb);
    m->pinned_bytes += cb;
  }

  for (cudaEvent_t* e : {&m->WR[0], &m->WR[1], &m->BD[0], &m->BD[1], &m->BF[0], &m->BF[1], &m->XR[0], &m->XR[1],
                         &m->XS[0], &m->XS[1], &m->TOK, &m->LOSS, &m->RT, &m->ER[0], &m->ER[1]})
    CU(mm, cudaEventCreateWithFlags(e, cudaEventDisableTiming));
  m->SR.assign((size_t)m->K, nullptr);
  for (auto& e : m->SR) CU(mm, cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
  m->slab_free.assign((size_t)m->K, 1);
  m->adam_done.assign(m->lay.size(), 0);

  std::vector<float> cs;
  compute_tables(m.get(), cs);
  CU(mm, cudaMemcpyAsync(m->d.cs, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice, m->sc));
  CU(mm, cudaMemsetAsync(m->d.loss, 0, 256, m->sc));
  for (int b = 0; b < m->nbuf; ++b) CU(mm, cudaMemsetAsync(m->d.buf[b], 0, (size_t)2 * m->wb_max, m->sc));
  if (c->debug_guards) {
    for (int64_t g : m->d.guards) CU(mm, cudaMemsetAsync(m->dev_base + g, 0xA5, (size_t)kGuardBytes, m->sc));
    CU(mm, cudaMemcpyAsync(m->d.guard_offs, m->d.guards.data(), m->d.guards.size() * sizeof(int64_t),
                           cudaMemcpyHostToDevice, m->sc));
    CU(mm, cudaMemsetAsync(m->d.guard_bad, 0x7F, sizeof(int), m->sc));  // 0x7F7F7F7F: no bad guard
  }
  CU(mm, cudaStreamSynchronize(m->sc));
  m->adam_thr = std::thread(adam_loop, mm);
  *out = m.release();
  return MT_OK;
}

mt_status mt_set_tokens(mt_model* m, const int32_t* tok) {
  if (!m || !tok) return MT_ERR_ARG;
  if (m->failed) return MT_ERR_STATE;
  if (m->vis != 0 || m->stage != 0 || m->pass != 0)
    return set_err(m, MT_ERR_STATE, "mt_set_tokens: a step is in progress", false);
  const int64_t T = m->T, Tstep = T * m->npass;
  for (int64_t i = 0; i < Tstep; ++i)
    if (tok[i] < 0 || tok[i] >= m->V) return set_err(m, MT_ERR_ARG, "token id out of range", false);
  if (m->tokens_set) OK(wait_event(m, m->TOK, "previous token upload"));
  // per pass: its tokens, next-token targets (-1 at a sequence's last
  // position), and the token CSR of the embedding backward
  for (int p = 0; p < m->npass; ++p) {
    const int32_t* src = tok + (int64_t)p * T;
    int32_t* h = m->htok + (int64_t)p * (3 * T + m->V + 1);
    int32_t* tg = h + T;
    int32_t* cst = tg + T;
    int32_t* rows = cst + m->V + 1;
    std::memcpy(h, src, (size_t)T * 4);
    for (int64_t t = 0; t < T; ++t) tg[t] = (t % m->S) < m->S - 1 ? src[t + 1] : -1;
    mt_token_csr(src, T, m->V, cst, rows);
  }
  m->tokens_set = true;
  return MT_OK;
}

mt_status mt_stream_in(mt_model* m, int32_t block, int32_t buf) {
  if (!m || buf < 0 || buf >= m->nbuf) return MT_ERR_ARG;
  OK(expect(m, 0, block));
  OK(do_stream_in(m, block, buf));
  advance(m);
  return MT_OK;
}

mt_status mt_bind(mt_model* m, int32_t block, int32_t buf, mt_layer_view* view) {
  if (!m || buf < 0 || buf >= m->nbuf) return MT_ERR_ARG;
  OK(expect(m, 1, block));
  OK(do_bind(m, block, buf, view));
  advance(m);
  return MT_OK;
}

mt_status mt_step_forward(mt_model* m, const mt_layer_view* v) {
  if (!m || !v) return MT_ERR_ARG;
  if (!m->tokens_set) return set_err(m, MT_ERR_STATE, "no tokens set", false);
  if (visit_kind(m, m->vis) == V_BWD)
    return set_err(m, MT_ERR_STATE, "forward called on a block-backward visit", false);
  OK(expect(m, 2, v->block));
  if (visit_kind(m, m->vis) == V_RECOMP) OK(do_recompute(m, v->block, v->buf));
  else OK(do_forward(m, v->block, v->buf));
  advance(m);
  return MT_OK;
}

mt_status mt_step_backward(mt_model* m, const mt_layer_view* v) {
  if (!m || !v) return MT_ERR_ARG;
  if (visit_kind(m, m->vis) != V_BWD)
    return set_err(m, MT_ERR_STATE, "backward called on a forward or recompute visit", false);
  OK(expect(m, 2, v->block));
  OK(do_backward(m, v->block, v->buf));
  advance(m);
  return MT_OK;
}

mt_status mt_stream_out(mt_model* m, int32_t block, int32_t buf, int32_t* slab) {
  if (!m || buf < 0 || buf >= m->nbuf) return MT_ERR_ARG;
  OK(expect(m, 3, block));
  int k = 0;
  OK(do_stream_out(m, block, buf, &k));
  if (slab) *slab = k;
  advance(m);
  return MT_OK;
}

mt_status mt_adam_host(mt_model* m, int32_t block, int32_t slab, int32_t adam_step) {
  if (!m || slab < 0 || slab >= m->K || adam_step < 1) return MT_ERR_ARG;
  OK(expect(m, 4, block));
  OK(do_adam_enqueue(m, block, slab, adam_step));
  advance(m);
  return MT_OK;
}

mt_status mt_train_step(mt_model* m, int32_t step, float* loss) {
  if (!m) return MT_ERR_ARG;
  if (m->failed) return MT_ERR_STATE;
  if (step != m->steps_done || m->vis != 0 || m->stage != 0 || m->pass != 0)
    return set_err(m, MT_ERR_STATE, "mt_train_step: step index or visit state mismatch", false);
  if (!m->tokens_set) return set_err(m, MT_ERR_STATE, "no tokens set", false);
  if (step >= 1) replan_measured(m);
  const double t0 = now_ms();
  const int n = nvisits(m);
  for (int p = 0; p < m->npass; ++p)
    for (int v = 0; v < n; ++v) OK(run_visit(m));
  if (loss) {
    OK(wait_event(m, m->LOSS, "loss"));
    float sum = 0.f;  // the step loss is the sum of the passes' (each already divided by all micro-batches)
    for (int p = 0; p < m->npass; ++p) sum += m->hloss[p];
    *loss = sum;
  }
  m->last_step_ms = now_ms() - t0;
  return MT_OK;
}

// debug_guards: every canary still 0xA5 (all work drained)?
static mt_status check_guards(mt_model* m) {
  const int n = (int)m->d.guards.size();
  CU(m, mt::guard_check(m->dev_base, m->d.guard_offs, n, m->d.guard_bad, m->sc));
  int bad = 0;
  CU(m, cudaMemcpyAsync(&bad, m->d.guard_bad, sizeof bad, cudaMemcpyDeviceToHost, m->sc));
  CU(m, cudaStreamSynchronize(m->sc));
  if (bad >= 0 && bad < n)
    return set_err(m, MT_ERR_INTERNAL, "device guard " + std::to_string(bad) + " (after carved piece " +
                                           std::to_string(bad) + ", region offset " +
                                           std::to_string(m->d.guards[(size_t)bad]) + ") overwritten");
  for (const auto& g : m->hguards)
    for (int64_t i = 0; i < kGuardBytes; ++i)
      if (g.first[i] != 0xA5) return set_err(m, MT_ERR_INTERNAL, "host guard after " + g.second + " overwritten");
  return MT_OK;
}

mt_status mt_debug_poke_guard(mt_model* m, int32_t which, int32_t* n_guards) {
  if (!m || !m->c.debug_guards) return MT_ERR_ARG;
  const int nd = (int)m->d.guards.size(), nh = (int)m->hguards.size();
  if (n_guards) *n_guards = nd + nh;
  if (which < 0 || which >= nd + nh) return MT_ERR_ARG;
  if (which < nd) {
    CU(m, cudaMemsetAsync(m->dev_base + m->d.guards[(size_t)which], 0, 1, m->sc));
    CU(m, cudaStreamSynchronize(m->sc));
  } else {
    m->hguards[(size_t)(which - nd)].first[0] = 0;
  }
  return MT_OK;
}

mt_status mt_sync(mt_model* m) {
  if (!m) return MT_ERR_ARG;
  if (m->failed) return MT_ERR_STATE;
  for (cudaStream_t s : {m->sc, m->sw, m->sg}) {
    cudaEvent_t e;
    CU(m, cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    CU(m, cudaEventRecord(e, s));
    const mt_status st = wait_event(m, e, "stream drain");
    cudaEventDestroy(e);
    OK(st);
  }
  {
    std::unique_lock<std::mutex> lk(m->amu);
    const bool ok = m->acv.wait_for(lk, std::chrono::milliseconds(m->c.timeout_ms),
                                    [&] { return m->failed || (m->jobs.empty() && m->inflight_jobs == 0); });
    if (m->failed) return MT_ERR_STATE;
    if (!ok) return set_err(m, MT_ERR_TIMEOUT, "timed out draining Adam jobs");
  }
  if (m->timing) collect_timing(m);
  replan_measured(m);
  if (m->c.debug_guards) OK(check_guards(m));
  // a GEMM or attention kernel whose bounded wait expired has recorded a
  // code; its outputs, and the step built on them, are not valid
  int kcode = 0;
  if (mt::kernel_error_read(&kcode, 0) != cudaSuccess) cudaGetLastError();
  if (kcode != 0)
    return set_err(m, MT_ERR_TIMEOUT,
                   "a kernel's bounded wait expired (device error code " + std::to_string(kcode) + ")");
  return MT_OK;
}

mt_status mt_read_host(mt_model* m, int32_t block, int32_t region, void* dst, size_t bytes) {
  if (!m || !dst || block < 0 || block >= (int)m->lay.size() || region < 0 || region > MT_REGION_GACC)
    return MT_ERR_ARG;
  const mth::BlockDesc& b = m->lay[(size_t)block];
  if (region == MT_REGION_GACC) {
    if (!m->gacc || (int64_t)bytes > b.n_pad * 4) return MT_ERR_ARG;
    std::memcpy(dst, m->gacc + m->gacc_off[(size_t)block], bytes);
    return MT_OK;
  }
  const int64_t rb = region < 2 ? b.wbytes : b.fbytes;
  if ((int64_t)bytes > rb) return MT_ERR_ARG;
  std::memcpy(dst, m->store + b.store_off + b.region[region], bytes);
  return MT_OK;
}

mt_status mt_write_host(mt_model* m, int32_t block, int32_t region, const void* src, size_t bytes) {
  if (!m || !src || block < 0 || block >= (int)m->lay.size() || region < 0 || region > 4) return MT_ERR_ARG;
  const mth::BlockDesc& b = m->lay[(size_t)block];
  const int64_t rb = region < 2 ? b.wbytes : b.fbytes;
  if ((int64_t)bytes > rb) return MT_ERR_ARG;
  std::memcpy(m->store + b.store_off + b.region[region], src, bytes);
  return MT_OK;
}

mt_status mt_get_stats(const mt_model* m, mt_stats* o) {
  if (!m || !o) return MT_ERR_ARG;
  std::memset(o, 0, sizeof *o);
  o->steps_done = m->steps_done;
  o->h2d_bytes = m->h2d.load();
  o->d2h_bytes = m->d2h.load();
  o->device_bytes_used = (int64_t)m->dev_used;
  o->last_step_ms = m->last_step_ms;
  o->adam_ms_total = m->adam_us.load() / 1000.0;
  o->pack_ms_total = m->pack_ms;
  o->host_store_bytes = (int64_t)m->store_bytes;
  o->pinned_bytes = (int64_t)m->pinned_bytes;
  return MT_OK;
}

// ---------------------------------------------------------------- save / load
// Between steps the GPU holds no model state: the host store (W, G, master,
// m, v of every block) and the step count are the whole training state.
namespace {
constexpr char kMagic[8] = {'M', 'T', 'S', 'T', 'O', 'R', 'E', '1'};
struct FileHeader {
  char magic[8];
  int32_t shape[10];  // n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab, n_experts, top_k, expert_ffn
  int64_t steps_done, store_bytes;
};
void fill_header(const mt_model* m, FileHeader* h) {
  std::memset(h, 0, sizeof *h);
  std::memcpy(h->magic, kMagic, 8);
  const mt_config& c = m->c;
  const int32_t v[10] = {c.n_layers, c.hidden, c.n_heads, c.n_kv_heads, c.head_dim, c.ffn, c.vocab,
                         c.n_experts, c.top_k, c.expert_ffn};
  std::memcpy(h->shape, v, sizeof v);
  h->steps_done = m->steps_done;
  h->store_bytes = (int64_t)m->store_bytes;
}
mt_status between_steps(mt_model* m) {
  if (m->failed) return MT_ERR_STATE;
  if (m->vis != 0 || m->stage != 0 || m->pass != 0)
    return set_err(m, MT_ERR_STATE, "save / load only between steps", false);
  return mt_sync(m);
}
}  // namespace

mt_status mt_save(mt_model* m, const char* path) {
  if (!m || !path) return MT_ERR_ARG;
  OK(between_steps(m));
  FileHeader h;
  fill_header(m, &h);
  FILE* f = std::fopen(path, "wb");
  if (!f) return set_err(m, MT_ERR_ARG, std::string("cannot open ") + path, false);
  bool ok = std::fwrite(&h, sizeof h, 1, f) == 1;
  constexpr size_t CH = (size_t)64 << 20;
  for (size_t o = 0; ok && o < m->store_bytes; o += CH)
    ok = std::fwrite(m->store + o, 1, std::min(CH, m->store_bytes - o), f) == std::min(CH, m->store_bytes - o);
  ok = (std::fclose(f) == 0) && ok;
  if (!ok) return set_err(m, MT_ERR_INTERNAL, std::string("write failed: ") + path, false);
  return MT_OK;
}

mt_status mt_load(mt_model* m, const char* path) {
  if (!m || !path) return MT_ERR_ARG;
  OK(between_steps(m));
  FileHeader want, got;
  fill_header(m, &want);
  FILE* f = std::fopen(path, "rb");
  if (!f) return set_err(m, MT_ERR_ARG, std::string("cannot open ") + path, false);
  if (std::fread(&got, sizeof got, 1, f) != 1 || std::memcmp(got.magic, kMagic, 8) ||
      std::memcmp(got.shape, want.shape, sizeof want.shape) || got.store_bytes != want.store_bytes || got.steps_done < 0) {
    std::fclose(f);
    return set_err(m, MT_ERR_ARG, std::string("not a saved store of this model's shape: ") + path, false);
  }
  bool ok = true;
  constexpr size_t CH = (size_t)64 << 20;
  for (size_t o = 0; ok && o < m->store_bytes; o += CH)
    ok = std::fread(m->store + o, 1, std::min(CH, m->store_bytes - o), f) == std::min(CH, m->store_bytes - o);
  std::fclose(f);
  // a short read leaves a partly overwritten store: the model cannot continue
  if (!ok) return set_err(m, MT_ERR_INTERNAL, std::string("read failed: ") + path);
  m->steps_done = got.steps_done;
  {
    std::lock_guard<std::mutex> lk(m->amu);
    for (auto& d : m->adam_done) d = got.steps_done;  // Adam of every block is in the store
  }
  m->tokens_set = false;
  return MT_OK;
}

mt_status mt_expert_counts(const mt_model* m, int32_t block, int32_t* counts, int32_t n) {
  if (!m || !counts || !m->moe || block < 1 || block > m->L || n < m->E) return MT_ERR_ARG;
  std::memcpy(counts, m->hcounts + (size_t)block * m->E, (size_t)m->E * 4);
  return MT_OK;
}

int64_t mt_protocol_log(const mt_model* m, char* buf, int64_t cap) {
  if (!m) return 0;
  std::string s;
  for (auto& l : m->log) {
    s += l;
    s += '\n';
  }
  const int64_t need = (int64_t)s.size() + 1;
  if (!buf || cap < need) return -need;
  std::memcpy(buf, s.c_str(), (size_t)need);
  return need - 1;
}

const char* mt_last_error(const mt_model* m) {
  if (!m) return "null model";
  std::lock_guard<std::mutex> lk(m->emu);
  static thread_local std::string copy;
  copy = m->err;
  return copy.c_str();
}

void mt_destroy(mt_model* m) { delete m; }

// ------------------------------------------------------------------ host-only
int64_t mt_layout_block(const mt_config* c, int32_t j, int64_t* out, int64_t cap) {
  if (!mth::config_valid(c, nullptr) || !out || j < 0 || j > c->n_layers + 1) return -1;
  const auto lay = mth::build_layout(c);
  const mth::BlockDesc& b = lay[(size_t)j];
  const int64_t need = 10 + 3 * b.nt;
  if (cap < need) return -1;
  out[0] = b.nt; out[1] = b.n_real; out[2] = b.n_pad;
  for (int r = 0; r < 5; ++r) out[3 + r] = b.region[r];
  out[8] = b.bytes; out[9] = b.store_off;
  for (int t = 0; t < b.nt; ++t) {
    out[10 + 3 * t] = b.t[t].off; out[11 + 3 * t] = b.t[t].rows; out[12 + 3 * t] = b.t[t].cols;
  }
  return need;
}

int64_t mt_param_count(const mt_config* c) {
  if (!mth::config_valid(c, nullptr)) return -1;
  int64_t p = 0;
  for (auto& b : mth::build_layout(c)) p += b.n_real;
  return p;
}

int64_t mt_store_bytes(const mt_config* c) {
  if (!mth::config_valid(c, nullptr)) return -1;
  int64_t s = 0;
  for (auto& b : mth::build_layout(c)) s += b.bytes;
  return s;
}

mt_status mt_host_init_block(const mt_config* c, int32_t j, float* master) {
  if (!mth::config_valid(c, nullptr) || !master || j < 0 || j > c->n_layers + 1) return MT_ERR_ARG;
  const auto lay = mth::build_layout(c);
  const mth::BlockDesc& b = lay[(size_t)j];
  std::memset(master, 0, (size_t)b.n_pad * 4);
  mth::init_block(c, b, j, master, 0, b.n_pad);
  return MT_OK;
}

mt_status mt_host_adam(int64_t n, const uint16_t* g, float* th, float* m, float* v, uint16_t* w, int32_t t,
                       float lr, float b1, float b2, float eps, float wd, int32_t n_threads) {
  if (n < 0 || !th || !m || !v || !w || t < 1) return MT_ERR_ARG;
  mth::Pool pool;
  pool.start(n_threads > 0 ? n_threads : 1);
  constexpr int64_t CH = 1 << 18;
  std::function<void(int64_t)> fn = [&](int64_t i) {
    const int64_t o = i * CH, len = (n - o) < CH ? (n - o) : CH;
    mth::adam(len, g ? g + o : nullptr, nullptr, th + o, m + o, v + o, w + o, t, lr, b1, b2, eps, wd);
  };
  std::string err;
  const bool ok = pool.parallel_for((n + CH - 1) / CH, fn, &err);
  pool.stop();
  return ok ? MT_OK : MT_ERR_INTERNAL;
}

int64_t mt_plan_protocol(const mt_config* c, int32_t n_steps, char* buf, int64_t cap) {
  if (!mth::config_valid(c, nullptr) || n_steps < 0) return 0;
  mt_model m;
  m.c = *c;
  m.live = false;
  fill_shape(&m);
  m.tokens_set = true;
  for (int s = 0; s < n_steps; ++s)
    for (int p = 0; p < m.npass; ++p)
      for (int v = 0; v < nvisits(&m); ++v)
        if (run_visit(&m) != MT_OK) return 0;
  return mt_protocol_log(&m, buf, cap);
}

int32_t mt_visit_plan(const mt_config* c, int32_t* kind, int32_t* block, int32_t cap) {
  if (!mth::config_valid(c, nullptr)) return -1;
  const std::vector<VisitDesc> p = build_plan(c->n_layers, c->ckpt_interval);
  for (size_t v = 0; v < p.size() && (int64_t)v < cap; ++v) {
    if (kind) kind[v] = p[v].kind;
    if (block) block[v] = p[v].j;
  }
  return (int32_t)p.size();
}

int32_t mt_schedule(int32_t n, const double* b, const double* d, const double* c, const double* a, double bw_h2d,
                    double bw_d2h, double* stall) {
  if (!b || !d || !c || !a || !stall) return -1;
  return mth::schedule(n, b, d, c, a, bw_h2d, bw_d2h, stall);
}

static bool sim_in(const mt_sched_in* s, mth::SimIn* o) {
  if (!s || s->n_visits < 1 || !s->kind || !s->block || !s->b || !s->p || !s->d || !s->c || !s->a) return false;
  if (!(s->bw_h2d > 0) || !(s->bw_d2h > 0) || s->n_buffers < 1) return false;
  for (int v = 0; v < s->n_visits; ++v)
    if (s->block[v] < 0 || s->kind[v] < 0 || s->kind[v] > 3) return false;
  o->n = s->n_visits;
  o->kind = s->kind;
  o->block = s->block;
  o->b = s->b;
  o->p = s->p;
  o->d = s->d;
  o->c = s->c;
  o->a = s->a;
  o->nbuf = s->n_buffers;
  o->bw_h2d = s->bw_h2d;
  o->bw_d2h = s->bw_d2h;
  o->pack_rate = s->pack_rate;
  o->adam_rate = s->adam_rate;
  o->adam_bytes = s->adam_bytes > 0 ? s->adam_bytes : 28.0;
  o->host_bw = s->host_bw;
  o->chunk = (double)kPackChunk;
  return true;
}

mt_status mt_schedule_simulate(const mt_sched_in* in, int32_t K, mt_sched_plan* out, double* stall_v) {
  mth::SimIn si;
  if (!out || K < 1 || !sim_in(in, &si)) return MT_ERR_ARG;
  mth::Plan pl;
  pl.K = K;
  pl.out = mth::simulate(si, K, 4, stall_v);
  std::memset(out, 0, sizeof *out);
  fill_plan_out(pl, si, 0, out);
  return MT_OK;
}

mt_status mt_schedule_plan(const mt_sched_in* in, int32_t k_max, mt_sched_plan* out) {
  mth::SimIn si;
  if (!out || k_max < 1 || !sim_in(in, &si)) return MT_ERR_ARG;
  const mth::Plan pl = mth::plan(si, 1, k_max);
  std::memset(out, 0, sizeof *out);
  fill_plan_out(pl, si, 0, out);
  return MT_OK;
}

mt_status mt_get_schedule(const mt_model* m, int32_t which, mt_sched_plan* out) {
  if (!m || !out || which < 0 || which > 1) return MT_ERR_ARG;
  if (which == 1 && !m->have_plan1) return MT_ERR_STATE;
  *out = which == 0 ? m->plan0 : m->plan1;
  return MT_OK;
}

mt_status mt_host_bandwidth(size_t bytes, int32_t n_threads, double* copy_gbs, double* adam_gelem_s) {
  if (bytes < (1u << 20) || n_threads < 1) return MT_ERR_ARG;
  const int64_t n = (int64_t)(bytes / 4);
  std::vector<float> a((size_t)n, 1.0f), b((size_t)n, 0.0f);
  std::vector<uint16_t> g((size_t)n, 0x3c00), w((size_t)n, 0);
  std::vector<float> th((size_t)n, 0.01f), mv((size_t)n, 0.0f), vv((size_t)n, 0.0f);
  mth::Pool pool;
  pool.start(n_threads);
  constexpr int64_t CH = 1 << 20;
  const int64_t items = (n + CH - 1) / CH;
  std::string err;
  double best_copy = 1e30, best_adam = 1e30;
  for (int rep = 0; rep < 3; ++rep) {
    auto t0 = Clock::now();
    std::function<void(int64_t)> cp = [&](int64_t i) {
      const int64_t o = i * CH, len = (n - o) < CH ? (n - o) : CH;
      std::memcpy(b.data() + o, a.data() + o, (size_t)len * 4);
    };
    pool.parallel_for(items, cp, &err);
    best_copy = std::min(best_copy, std::chrono::duration<double>(Clock::now() - t0).count());
    t0 = Clock::now();
    std::function<void(int64_t)> ad = [&](int64_t i) {
      const int64_t o = i * CH, len = (n - o) < CH ? (n - o) : CH;
      mth::adam(len, g.data() + o, nullptr, th.data() + o, mv.data() + o, vv.data() + o, w.data() + o, rep + 1, 1e-3f,
                0.9f, 0.999f, 1e-8f, 0.0f);
    };
    pool.parallel_for(items, ad, &err);
    best_adam = std::min(best_adam, std::chrono::duration<double>(Clock::now() - t0).count());
  }
  pool.stop();
  if (copy_gbs) *copy_gbs = 2.0 * (double)n * 4 / best_copy / 1e9;
  if (adam_gelem_s) *adam_gelem_s = (double)n / best_adam / 1e9;
  return MT_OK;
}

mt_status mt_token_csr(const int32_t* tok, int64_t T, int32_t V, int32_t* row_start, int32_t* rows) {
  if (!tok || !row_start || !rows || V <= 0 || T < 0) return MT_ERR_ARG;
  std::memset(row_start, 0, (size_t)(V + 1) * 4);
  for (int64_t t = 0; t < T; ++t) {
    if (tok[t] < 0 || tok[t] >= V) return MT_ERR_ARG;
    row_start[tok[t] + 1]++;
  }
  for (int32_t v = 0; v < V; ++v) row_start[v + 1] += row_start[v];
  std::vector<int32_t> fill(row_start, row_start + V);
  for (int64_t t = 0; t < T; ++t) rows[fill[(size_t)tok[t]]++] = (int32_t)t;
  return MT_OK;
}

mt_status mt_rope_table(int32_t S, int32_t hd, double base, float* out) {
  if (S <= 0 || hd <= 0 || hd % 2 || !out) return MT_ERR_ARG;
  const int half = hd / 2;
  for (int p = 0; p < S; ++p)
    for (int i = 0; i < half; ++i) {
      const double a = (double)p * std::pow(base, -2.0 * i / (double)hd);
      out[((size_t)p * half + i) * 2] = (float)std::cos(a);
      out[((size_t)p * half + i) * 2 + 1] = (float)std::sin(a);
    }
  return MT_OK;
}

// ------------------------------------------------------------------ timing
mt_status mt_timing(mt_model* m, int32_t enable) {
  if (!m) return MT_ERR_ARG;
  if (!enable) OK(mt_sync(m));
  m->timing = enable != 0;
  for (auto& k : m->kstat) k = KStat();
  m->vstat.assign((size_t)nvisits(m), KStat());
  return MT_OK;
}

mt_status mt_trace(mt_model* m, int32_t enable) {
  if (!m) return MT_ERR_ARG;
  if (!enable || m->tracing) OK(mt_sync(m));  // the previous timeline's events complete before reuse
  if (!enable) {
    m->tracing = false;
    return MT_OK;
  }
  for (auto& t : m->tdev) {
    m->ev_pool.push_back(t.a);
    m->ev_pool.push_back(t.b);
  }
  m->tdev.clear();
  {
    std::lock_guard<std::mutex> lk(m->tmu);
    m->thost.clear();
  }
  // Device time 0: an event on a private stream with nothing queued, so it
  // completes at once; host time 0 is taken right after it has.  The model's
  // streams keep running: a timeline can start in the middle of training.
  if (!m->trace_stream) CU(m, cudaStreamCreateWithFlags(&m->trace_stream, cudaStreamNonBlocking));
  if (!m->trace_base) CU(m, cudaEventCreate(&m->trace_base));
  CU(m, cudaEventRecord(m->trace_base, m->trace_stream));
  CU(m, cudaEventSynchronize(m->trace_base));
  m->trace_host_base = now_ms();
  m->tracing = true;
  return MT_OK;
}

int64_t mt_trace_json(mt_model* m, char* buf, int64_t cap) {
  if (!m || m->failed) return 0;
  static const char* names[] = {"H2D", "H2D_EXP", "", "D2H", "D2H_CKPT"};
  static const char* kinds[] = {"FWD", "HEAD", "RECOMP", "BWD"};
  std::string js = "{\"traceEvents\":[";
  bool first = true;
  char line[256];
  auto add = [&](const char* name, const char* tid, double t0, double t1, int block, int64_t step) {
    std::snprintf(line, sizeof line,
                  "%s{\"name\":\"%s %d\",\"cat\":\"%s\",\"ph\":\"X\",\"ts\":%.3f,\"dur\":%.3f,\"pid\":0,"
                  "\"tid\":\"%s\",\"args\":{\"block\":%d,\"step\":%lld}}",
                  first ? "" : ",", name, block, tid, t0 * 1e3, (t1 - t0) * 1e3, tid, block, (long long)step);
    js += line;
    first = false;
  };
  for (const auto& t : m->tdev) {
    float a = 0, b = 0;
    if (cudaEventElapsedTime(&a, m->trace_base, t.a) != cudaSuccess ||
        cudaEventElapsedTime(&b, m->trace_base, t.b) != cudaSuccess)
      continue;  // not yet complete
    const char* name = t.op >= TR_COMPUTE ? kinds[t.op - TR_COMPUTE] : names[t.op];
    const char* tid = t.stream == 'W' ? "weight stream" : t.stream == 'C' ? "compute stream" : "gradient stream";
    add(name, tid, a, b, t.block, t.step);
  }
  {
    std::lock_guard<std::mutex> lk(m->tmu);
    for (const auto& h : m->thost) add(h.pass + 1 < m->npass ? "ACCUM" : "ADAM", "host Adam", h.t0, h.t1, h.block, h.step);
  }
  js += "]}";
  const int64_t need = (int64_t)js.size() + 1;
  if (!buf || cap < need) return -need;
  std::memcpy(buf, js.c_str(), (size_t)need);
  return need - 1;
}

mt_status mt_timing_visits(mt_model* m, double* ms, int32_t cap, int32_t* n_visits) {
  if (!m || !n_visits) return MT_ERR_ARG;
  collect_timing(m);
  *n_visits = nvisits(m);
  for (int v = 0; v < nvisits(m) && v < cap && ms; ++v) {
    const KStat& k = v < (int)m->vstat.size() ? m->vstat[(size_t)v] : KStat();
    ms[v] = k.launches ? k.ms / (double)k.launches : 0.0;
  }
  return MT_OK;
}

mt_status mt_timing_read(mt_model* m, int32_t kind, int64_t* launches, double* ms, double* flops, double* bytes) {
  if (!m || kind < 0 || kind > 3) return MT_ERR_ARG;
  collect_timing(m);
  const KStat& k = m->kstat[kind];
  if (launches) *launches = k.launches;
  if (ms) *ms = k.ms;
  if (flops) *flops = k.flops;
  if (bytes) *bytes = k.bytes;
  return MT_OK;
}

// ------------------------------------------------------------------ per-op
static mt_status cu_status(cudaError_t e) {
  if (e == cudaSuccess) return MT_OK;
  if (e == cudaErrorInvalidValue) return MT_ERR_ARG;
  return MT_ERR_CUDA;
}

mt_status mt_gemm(const void* A, int64_t lda, int32_t a_mn, const void* B, int64_t ldb, int32_t b_mn, int32_t M,
                  int32_t N, int32_t K, void* D, int64_t ldd, const void* R, int64_t ldr, float* Dacc,
                  int64_t ldacc, int32_t acc_mode, void* stream) {
  if (acc_mode < 0 || acc_mode > 2) return MT_ERR_ARG;
  mt::GemmArgs g{(const bf16*)A, lda, a_mn, (const bf16*)B, ldb, b_mn, M, N, K, (bf16*)D, ldd, (const bf16*)R,
                 ldr, Dacc, ldacc, acc_mode};
  return cu_status(mt::gemm(g, (cudaStream_t)stream));
}

int32_t mt_gemm_mode(int32_t mode) { return mt::gemm_mode(mode); }

mt_status mt_gemm2(const void* const* A, const int64_t* lda, const int32_t* a_mn, const void* const* B,
                   const int64_t* ldb, const int32_t* b_mn, const int32_t* M, const int32_t* N, const int32_t* K,
                   void* const* D, const int64_t* ldd, void* stream) {
  if (!A || !lda || !a_mn || !B || !ldb || !b_mn || !M || !N || !K || !D || !ldd) return MT_ERR_ARG;
  mt::GemmArgs g[2];
  for (int i = 0; i < 2; ++i)
    g[i] = mt::GemmArgs{(const bf16*)A[i], lda[i], a_mn[i], (const bf16*)B[i], ldb[i], b_mn[i], M[i], N[i], K[i],
                        (bf16*)D[i], ldd[i], nullptr, 0, nullptr, 0, 0};
  return cu_status(mt::gemm_pair(g[0], g[1], (cudaStream_t)stream));
}

mt_status mt_rmsnorm_fwd(const void* x, const void* gamma, int64_t T, int32_t H, float eps, void* y, float* rstd,
                         void* stream) {
  if (!x || !gamma || !y || !rstd) return MT_ERR_ARG;
  return cu_status(mt::rmsnorm_fwd((const bf16*)x, (const bf16*)gamma, T, H, eps, (bf16*)y, rstd, (cudaStream_t)stream));
}

size_t mt_rmsnorm_bwd_scratch_bytes(int64_t T, int32_t H) {
  return (size_t)mt::rmsnorm_bwd_partial_floats(T, H) * sizeof(float);
}

mt_status mt_rmsnorm_bwd(const void* dy, const void* x, const void* gamma, const float* rstd, const void* dres,
                         int64_t T, int32_t H, void* dx, void* dgamma, void* scratch, size_t scratch_bytes,
                         void* stream) {
  if (!dy || !x || !gamma || !rstd || !dx || !dgamma || !scratch) return MT_ERR_ARG;
  if (scratch_bytes < mt_rmsnorm_bwd_scratch_bytes(T, H)) return MT_ERR_ARG;
  return cu_status(mt::rmsnorm_bwd((const bf16*)dy, (const bf16*)x, (const bf16*)gamma, rstd, (const bf16*)dres, T,
                                   H, (bf16*)dx, (bf16*)dgamma, (float*)scratch, (cudaStream_t)stream));
}

mt_status mt_rope(void* x, int64_t T, int64_t ld, int32_t n_heads, int32_t hd, int32_t S, const float* cs,
                  int32_t inverse, void* stream) {
  if (!x || !cs || S <= 0) return MT_ERR_ARG;
  return cu_status(mt::rope((bf16*)x, T, ld, n_heads, hd, S, cs, inverse, (cudaStream_t)stream));
}

mt_status mt_attention_fwd(const void* qkv, int32_t n_seq, int32_t S, int32_t nh, int32_t nkv, int32_t hd, void* o,
                           float* lse, void* stream) {
  if (!qkv || !o || !lse || nkv <= 0) return MT_ERR_ARG;
  return cu_status(mt::attention_fwd((const bf16*)qkv, n_seq, S, nh, nkv, hd, (bf16*)o, lse, (cudaStream_t)stream));
}

size_t mt_attention_bwd_scratch_bytes(int32_t n_seq, int32_t S, int32_t nh, int32_t hd) {
  (void)hd;
  return (size_t)n_seq * (size_t)S * (size_t)nh * 4;  // delta [nh][T] FP32
}

mt_status mt_attention_bwd(const void* qkv, const void* o, const float* lse, const void* dout, int32_t n_seq,
                           int32_t S, int32_t nh, int32_t nkv, int32_t hd, void* dqkv, void* scratch,
                           size_t scratch_bytes, void* stream) {
  if (!qkv || !o || !lse || !dout || !dqkv || !scratch || nkv <= 0) return MT_ERR_ARG;
  if (scratch_bytes < mt_attention_bwd_scratch_bytes(n_seq, S, nh, hd)) return MT_ERR_ARG;
  return cu_status(mt::attention_bwd((const bf16*)qkv, (const bf16*)o, lse, (const bf16*)dout, n_seq, S, nh, nkv, hd,
                                     (bf16*)dqkv, (float*)scratch, (cudaStream_t)stream));
}

mt_status mt_swiglu_fwd(const void* gu, int64_t T, int32_t F, void* h, void* stream) {
  if (!gu || !h) return MT_ERR_ARG;
  return cu_status(mt::swiglu_fwd((const bf16*)gu, T, F, (bf16*)h, (cudaStream_t)stream));
}

mt_status mt_swiglu_bwd(const void* gu, const void* dh, int64_t T, int32_t F, void* dgu, void* stream) {
  if (!gu || !dh || !dgu) return MT_ERR_ARG;
  return cu_status(mt::swiglu_bwd((const bf16*)gu, (const bf16*)dh, T, F, (bf16*)dgu, (cudaStream_t)stream));
}

mt_status mt_embed_fwd(const int32_t* tok, const void* E, int64_t T, int32_t H, int32_t V, void* X, void* stream) {
  if (!tok || !E || !X) return MT_ERR_ARG;
  return cu_status(mt::embed_fwd(tok, (const bf16*)E, T, H, V, (bf16*)X, (cudaStream_t)stream));
}

mt_status mt_embed_bwd(const int32_t* row_start, const int32_t* rows, const void* dX, int32_t V, int32_t H, void* dE,
                       void* stream) {
  if (!row_start || !rows || !dX || !dE) return MT_ERR_ARG;
  return cu_status(mt::embed_bwd(row_start, rows, (const bf16*)dX, V, H, (bf16*)dE, (cudaStream_t)stream));
}

mt_status mt_cross_entropy(void* logits, const int32_t* target, int64_t rows, int32_t V, float inv_norm,
                           float* row_loss, void* stream) {
  if (!logits || !target || !row_loss) return MT_ERR_ARG;
  return cu_status(mt::cross_entropy((bf16*)logits, target, rows, V, inv_norm, row_loss, (cudaStream_t)stream));
}

size_t mt_moe_scratch_bytes(int64_t T, int32_t H, int32_t E, int32_t k, int32_t Fe) {
  if (T < 0 || H <= 0 || E <= 0 || k <= 0 || Fe <= 0) return 0;
  MoeWs w;
  return moe_carve(MoeShape{T, H, E, k, Fe}, nullptr, &w);
}

mt_status mt_moe_ffn(const void* yn, const void* x1, const void* Wr, const void* We, const void* dout, int64_t T,
                     int32_t H, int32_t E, int32_t k, int32_t Fe, void* out, void* dyn, void* dWr, void* dWe,
                     int32_t* idx, float* gate, void* scratch, size_t scratch_bytes, void* stream) {
  if (!yn || !x1 || !Wr || !We || !dout || !out || !dyn || !dWr || !dWe || !idx || !gate || !scratch)
    return MT_ERR_ARG;
  if (T < 1 || H <= 0 || H % 64 || Fe <= 0 || Fe % 64 || E < 8 || E > 128 || E % 8 || k < 1 || k > 8 || k > E)
    return MT_ERR_ARG;
  const MoeShape q{T, H, E, k, Fe};
  MoeWs w;
  if (scratch_bytes < moe_carve(q, nullptr, &w) || (reinterpret_cast<uintptr_t>(scratch) & 255)) return MT_ERR_ARG;
  moe_carve(q, (uint8_t*)scratch, &w);
  cudaStream_t s = (cudaStream_t)stream;
  const bf16 *Y = (const bf16*)yn, *X1 = (const bf16*)x1, *R = (const bf16*)Wr, *Wex = (const bf16*)We;
  OK(moe_route(nullptr, q, w, Y, R, s));
  std::vector<int32_t> counts((size_t)E);
  if (cudaMemcpyAsync(counts.data(), w.p.counts, (size_t)E * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return MT_ERR_CUDA;
  const MoeRoute r = route_from_counts(counts.data(), E);
  OK(moe_experts_fwd(nullptr, q, w, r, Y, X1, Wex, (bf16*)out, s));
  if (cudaMemsetAsync(dWe, 0, (size_t)E * 3 * Fe * H * 2, s) != cudaSuccess) return MT_ERR_CUDA;
  OK(moe_backward(nullptr, q, w, r, Y, R, Wex, (const bf16*)dout, (bf16*)dyn, (bf16*)dWr, (bf16*)dWe, s));
  if (cudaMemcpyAsync(idx, w.p.idx, (size_t)T * k * 4, cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(gate, w.p.gate, (size_t)T * k * 4, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return MT_ERR_CUDA;
  return MT_OK;
}

mt_status mt_fault_inject(int32_t kind, int32_t value) {
  if (value < 0) return MT_ERR_ARG;
  switch (kind) {
    case 1: g_inj_adam_delay_ms = value; return MT_OK;
    case 2: g_inj_adam_throw = value; return MT_OK;
    case 3: g_inj_pinned_fail = value; return MT_OK;
    case 4: mt::gemm_inject_stall(value); return MT_OK;
    default: return MT_ERR_ARG;
  }
}

mt_status mt_kernel_error(int32_t* code, int32_t clear) {
  if (!code) return MT_ERR_ARG;
  int c = 0;
  const mt_status s = cu_status(mt::kernel_error_read(&c, clear));
  *code = c;
  return s;
}

}  // extern "C"
