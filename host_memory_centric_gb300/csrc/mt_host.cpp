// mt_host.cpp -- host-side pieces of libmt that need no GPU.
#include "mt_host.h"

#include <algorithm>
#include <cmath>
#include <cstring>

namespace mth {

// ---------------------------------------------------------------- layout
bool config_valid(const mt_config* c, std::string* why) {
  auto bad = [&](const char* s) {
    if (why) *why = s;
    return false;
  };
  if (!c) return bad("null config");
  if (c->n_layers < 1 || c->hidden <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 || c->head_dim <= 0 ||
      c->ffn <= 0 || c->vocab <= 1 || c->batch <= 0 || c->seq <= 1 || c->micro_batches <= 0)
    return bad("non-positive shape field");
  if (c->n_heads % c->n_kv_heads) return bad("n_heads must be a multiple of n_kv_heads");
  if (c->hidden % 8 || c->ffn % 8 || c->head_dim % 16) return bad("hidden, ffn must be multiples of 8; head_dim of 16");
  if (c->ckpt_interval < 1 || c->ckpt_interval > c->n_layers) return bad("ckpt_interval must be in [1, n_layers]");
  if (c->n_buffers != 1 && c->n_buffers != 2) return bad("n_buffers must be 1 or 2");
  if (c->host_grad_accum != 0 && c->host_grad_accum != 1) return bad("host_grad_accum must be 0 or 1");
  if (c->n_grad_slabs < 0 || c->n_grad_slabs > 256) return bad("n_grad_slabs out of range");
  if (c->n_experts < 0) return bad("n_experts must be >= 0");
  if (c->n_experts > 0) {
    if (c->n_experts > 128 || c->n_experts % 8) return bad("n_experts must be a multiple of 8 and <= 128");
    if (c->top_k < 1 || c->top_k > 8 || c->top_k > c->n_experts) return bad("top_k must be in [1, min(8, n_experts)]");
    if (c->expert_ffn <= 0 || c->expert_ffn % 64 || c->hidden % 64)
      return bad("expert_ffn and hidden must be positive multiples of 64 with experts");
    if (c->host_grad_accum) return bad("host_grad_accum is not supported with experts");
  }
  if (c->timeout_ms == 0) return bad("timeout_ms must be positive");
  if (!(c->rms_eps > 0) || !(c->rope_base > 1)) return bad("rms_eps / rope_base");
  return true;
}

int64_t tokens_per_step(const mt_config* c) {
  return (int64_t)c->micro_batches * c->batch * c->seq;
}

static int64_t up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

std::vector<BlockDesc> build_layout(const mt_config* c) {
  const int64_t H = c->hidden, hd = c->head_dim, nh = c->n_heads, nkv = c->n_kv_heads, F = c->ffn;
  const int64_t V = c->vocab, L = c->n_layers;
  std::vector<BlockDesc> out((size_t)(L + 2));
  int64_t store = 0;
  for (int64_t j = 0; j <= L + 1; ++j) {
    BlockDesc& b = out[(size_t)j];
    int64_t shapes[MT_MAX_TENSORS][2];
    int n = 0;
    if (j == 0) {
      shapes[n][0] = V; shapes[n++][1] = H;                      // E
    } else if (j <= L && c->n_experts > 0) {
      // routed MoE block; row e of W_experts = expert e's W_gu [2Fe, H] then
      // W_down [H, Fe], so one expert is one contiguous range
      shapes[n][0] = (nh + 2 * nkv) * hd; shapes[n++][1] = H;    // W_qkv
      shapes[n][0] = H; shapes[n++][1] = nh * hd;                // W_o
      shapes[n][0] = c->n_experts; shapes[n++][1] = H;           // W_router
      shapes[n][0] = c->n_experts; shapes[n++][1] = 3 * (int64_t)c->expert_ffn * H;  // W_experts
      shapes[n][0] = H; shapes[n++][1] = 1;                      // gamma1
      shapes[n][0] = H; shapes[n++][1] = 1;                      // gamma2
    } else if (j <= L) {
      shapes[n][0] = (nh + 2 * nkv) * hd; shapes[n++][1] = H;    // W_qkv
      shapes[n][0] = H; shapes[n++][1] = nh * hd;                // W_o
      shapes[n][0] = 2 * F; shapes[n++][1] = H;                  // W_gu
      shapes[n][0] = H; shapes[n++][1] = F;                      // W_down
      shapes[n][0] = H; shapes[n++][1] = 1;                      // gamma1
      shapes[n][0] = H; shapes[n++][1] = 1;                      // gamma2
    } else {
      shapes[n][0] = H; shapes[n++][1] = 1;                      // gamma_f
      shapes[n][0] = V; shapes[n++][1] = H;                      // W_head
    }
    int64_t e = 0;
    for (int t = 0; t < n; ++t) {
      e = up(e, 128);
      b.t[t] = {e, shapes[t][0], shapes[t][1]};
      e += shapes[t][0] * shapes[t][1];
      b.n_real += shapes[t][0] * shapes[t][1];
    }
    b.nt = n;
    b.n_pad = up(e, 128);
    b.wbytes = up(2 * b.n_pad, 4096);
    b.fbytes = up(4 * b.n_pad, 4096);
    b.region[0] = 0;
    b.region[1] = b.wbytes;
    b.region[2] = 2 * b.wbytes;
    b.region[3] = 2 * b.wbytes + b.fbytes;
    b.region[4] = 2 * b.wbytes + 2 * b.fbytes;
    b.bytes = 2 * b.wbytes + 3 * b.fbytes;
    b.store_off = store;
    store += b.bytes;
  }
  return out;
}

// ---------------------------------------------------------------- numerics
uint16_t bf16_rne(float f) {
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  const bool nan = ((u >> 23) & 0xFF) == 0xFF && (u & 0x7FFFFF) != 0;
  if (nan) return (uint16_t)((u >> 16) | 0x0040);
  u = u + 0x7FFF + ((u >> 16) & 1);
  return (uint16_t)(u >> 16);
}
float bf16_val(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

// SplitMix64 (Steele, Lea, Flood 2014) evaluated at a counter: the output
// after i+1 increments of the golden gamma from `seed`.
static inline uint64_t sm64(uint64_t seed, uint64_t i) {
  uint64_t z = seed + (i + 1) * 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

void init_block(const mt_config* c, const BlockDesc& b, int j, float* master, int64_t e0, int64_t e1) {
  // element e of the padded block; padding and gains handled per range
  for (int t = 0; t < b.nt; ++t) {
    const TensorDesc& d = b.t[t];
    const int64_t n = d.rows * d.cols;
    const int64_t lo = e0 > d.off ? e0 : d.off, hi = e1 < d.off + n ? e1 : d.off + n;
    if (lo >= hi) continue;
    if (d.cols == 1) {
      for (int64_t e = lo; e < hi; ++e) master[e] = 1.0f;
      continue;
    }
    const uint64_t key = sm64(c->seed, 1 + 64ULL * (uint64_t)j + (uint64_t)t);
    for (int64_t e = lo; e < hi; ++e) {
      const uint64_t i = (uint64_t)(e - d.off);
      const uint64_t r1 = sm64(key, 2 * i), r2 = sm64(key, 2 * i + 1);
      const double u1 = (double)((r1 >> 11) + 1) * (1.0 / 9007199254740992.0);
      const double u2 = (double)(r2 >> 11) * (1.0 / 9007199254740992.0);
      const double z = std::sqrt(-2.0 * std::log(u1)) * std::cos(6.283185307179586 * u2);
      master[e] = (float)((double)c->init_std * z);
    }
  }
}

namespace {
inline float bf16f(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}
// One Adam element: gradient gi (FP32 of its BF16), moments and master in
// FP32.  step = lr / (1 - b1^t) and isb2 = 1 / sqrt(1 - b2^t) fold the bias
// corrections: m_hat / (sqrt(v_hat) + eps) = m / (1-b1^t) / (sqrt(v) isb2 + eps).
inline uint16_t adam_elem(float gi, float& th, float& m, float& v, float b1, float c1, float b2, float c2,
                          float step, float isb2, float eps, float lrwd) {
  const float mi = b1 * m + c1 * gi;
  const float vi = b2 * v + c2 * gi * gi;
  m = mi;
  v = vi;
  float x = th;
  x -= lrwd * x;
  x -= step * mi / (std::sqrt(vi) * isb2 + eps);
  th = x;
  uint32_t u;
  std::memcpy(&u, &x, 4);
  const bool nan = ((u >> 23) & 0xFF) == 0xFF && (u & 0x7FFFFF) != 0;
  const uint32_t r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16;
  return nan ? (uint16_t)((u >> 16) | 0x0040) : (uint16_t)r;
}
}  // namespace

void adam(int64_t n, const uint16_t* __restrict g, uint16_t* __restrict gcopy, float* __restrict th,
          float* __restrict m, float* __restrict v, uint16_t* __restrict w, int32_t t, float lr, float b1, float b2,
          float eps, float wd) {
  const double bc1 = 1.0 - std::pow((double)b1, (double)t);
  const double bc2 = 1.0 - std::pow((double)b2, (double)t);
  const float step = (float)((double)lr / bc1);
  const float isb2 = (float)(1.0 / std::sqrt(bc2));
  const float c1 = 1.0f - b1, c2 = 1.0f - b2, lrwd = lr * wd;
  if (!g) {  // zero gradient (an expert no token was routed to)
    for (int64_t i = 0; i < n; ++i) {
      if (gcopy) gcopy[i] = 0;
      w[i] = adam_elem(0.0f, th[i], m[i], v[i], b1, c1, b2, c2, step, isb2, eps, lrwd);
    }
  } else if (gcopy) {
    for (int64_t i = 0; i < n; ++i) {
      const uint16_t gb = g[i];
      gcopy[i] = gb;
      w[i] = adam_elem(bf16f(gb), th[i], m[i], v[i], b1, c1, b2, c2, step, isb2, eps, lrwd);
    }
  } else {
    for (int64_t i = 0; i < n; ++i)
      w[i] = adam_elem(bf16f(g[i]), th[i], m[i], v[i], b1, c1, b2, c2, step, isb2, eps, lrwd);
  }
}

// ---------------------------------------------------------------- pool
void Pool::start(int n) {
  stop_ = false;
  for (int i = 0; i < n; ++i)
    threads_.emplace_back([this] {
      for (;;) {
        Task t;
        {
          std::unique_lock<std::mutex> lk(mu_);
          cv_.wait(lk, [this] { return stop_ || !q_.empty(); });
          if (q_.empty()) return;  // stopping
          t = q_.front();
          q_.pop_front();
        }
        run(t);
      }
    });
}

void Pool::stop() {
  {
    std::lock_guard<std::mutex> lk(mu_);
    stop_ = true;
  }
  cv_.notify_all();
  for (auto& t : threads_)
    if (t.joinable()) t.join();
  threads_.clear();
}

void Pool::run(Task& t) {
  bool bad = false;
  std::string msg;
  try {
    (*t.fn)(t.i);
  } catch (const std::exception& e) {
    bad = true;
    msg = e.what();
  } catch (...) {
    bad = true;
    msg = "unknown exception in host worker";
  }
  std::lock_guard<std::mutex> lk(t.latch->mu);
  if (bad && !t.latch->bad) {
    t.latch->bad = true;
    t.latch->msg = msg;
  }
  if (--t.latch->left == 0) t.latch->cv.notify_all();
}

bool Pool::run_own(const Latch* latch) {
  Task t;
  {
    std::lock_guard<std::mutex> lk(mu_);
    auto it = std::find_if(q_.begin(), q_.end(), [&](const Task& x) { return x.latch == latch; });
    if (it == q_.end()) return false;
    t = *it;
    q_.erase(it);
  }
  run(t);
  return true;
}

bool Pool::parallel_for(int64_t n, const std::function<void(int64_t)>& fn, std::string* err, bool urgent) {
  if (n <= 0) return true;
  Latch latch;
  latch.left = n;
  {
    std::lock_guard<std::mutex> lk(mu_);
    if (urgent)
      for (int64_t i = n - 1; i >= 0; --i) q_.push_front({&fn, i, &latch});
    else
      for (int64_t i = 0; i < n; ++i) q_.push_back({&fn, i, &latch});
  }
  cv_.notify_all();
  for (;;) {
    if (run_own(&latch)) continue;  // help with this call's own queued tasks only
    std::unique_lock<std::mutex> lk(latch.mu);
    if (latch.cv.wait_for(lk, std::chrono::milliseconds(2), [&] { return latch.left == 0; })) break;
  }
  if (latch.bad) {
    if (err) *err = latch.msg;
    return false;
  }
  return true;
}

void accumulate(int64_t n, const uint16_t* __restrict g, float* __restrict acc, bool first) {
  if (first) {
    for (int64_t i = 0; i < n; ++i) acc[i] = bf16f(g[i]);
  } else {
    for (int64_t i = 0; i < n; ++i) acc[i] += bf16f(g[i]);
  }
}

void adam_acc(int64_t n, const uint16_t* __restrict g, float* __restrict acc, uint16_t* __restrict gcopy,
              float* __restrict th, float* __restrict m, float* __restrict v, uint16_t* __restrict w, int32_t t,
              float lr, float b1, float b2, float eps, float wd) {
  const double bc1 = 1.0 - std::pow((double)b1, (double)t);
  const double bc2 = 1.0 - std::pow((double)b2, (double)t);
  const float step = (float)((double)lr / bc1);
  const float isb2 = (float)(1.0 / std::sqrt(bc2));
  const float c1 = 1.0f - b1, c2 = 1.0f - b2, lrwd = lr * wd;
  for (int64_t i = 0; i < n; ++i) {
    const float gi = acc[i] + bf16f(g[i]);
    acc[i] = gi;
    if (gcopy) gcopy[i] = bf16_rne(gi);
    w[i] = adam_elem(gi, th[i], m[i], v[i], b1, c1, b2, c2, step, isb2, eps, lrwd);
  }
}

int64_t tokens_per_pass(const mt_config* c) {
  return (int64_t)(c->host_grad_accum ? 1 : c->micro_batches) * c->batch * c->seq;
}
int passes_per_step(const mt_config* c) { return c->host_grad_accum ? c->micro_batches : 1; }

// ---------------------------------------------------------------- schedule
// Two device buffers: the stream-in of visit v+1 overlaps the compute of v and
// may start once visit v-1's buffer is free, i.e. after its gradient export.
// A slab is held from the start of its export until its Adam ends.
int32_t schedule(int32_t n, const double* b, const double* d, const double* c, const double* a, double bw_h2d,
                 double bw_d2h, double* stall) {
  if (n <= 0 || !(bw_h2d > 0) || !(bw_d2h > 0)) return -1;
  stall[0] = b[0] / bw_h2d;
  for (int32_t v = 1; v < n; ++v) {
    const double export_prev = v >= 2 ? d[v - 2] / bw_d2h : 0.0;
    const double w = export_prev + b[v] / bw_h2d - c[v - 1];
    stall[v] = w > 0.0 ? w : 0.0;
  }
  int32_t need = 1;
  for (int32_t v = 0; v < n; ++v) {
    if (!(d[v] > 0)) continue;
    const double denom = c[v] > 0 ? c[v] : 1e-30;
    const int32_t k = (int32_t)std::ceil((d[v] / bw_d2h + a[v]) / denom) + 1;
    if (k > need) need = k;
  }
  return need;
}

namespace {
// Host Adam in the model: one job per export; the server takes, among the
// jobs whose slab has landed, the lowest block (the library's order).
struct SimJob {
  int32_t step, block;
  double ready, elems, end = -1;
};
struct AdamSim {
  std::vector<SimJob> jobs;
  double free_at = 0, rate = 1, busy = 0;
  size_t done = 0;
  // Decides and runs one more job; false when every job is done.
  bool next() {
    if (done == jobs.size()) return false;
    double t = free_at;
    bool any = false;
    for (const SimJob& j : jobs)
      if (j.end < 0 && j.ready <= t) any = true;
    if (!any) {  // idle until the next slab lands
      double r = 1e300;
      for (const SimJob& j : jobs)
        if (j.end < 0 && j.ready < r) r = j.ready;
      t = r;
    }
    SimJob* best = nullptr;
    for (SimJob& j : jobs)
      if (j.end < 0 && j.ready <= t && (!best || j.block < best->block)) best = &j;
    const double dur = best->elems / rate;
    best->end = t + dur;
    busy += dur;
    free_at = best->end;
    ++done;
    return true;
  }
};

SimOut simulate_at(const SimIn& in, int32_t K, int32_t steps, double* stall_v, double adam_rate) {
  SimOut out;
  const int n = in.n, nb = in.nbuf < 1 ? 1 : in.nbuf;
  AdamSim ad;
  ad.rate = adam_rate > 0 ? adam_rate : 1e30;
  const double prate = in.pack_rate > 0 ? in.pack_rate : 1e30;
  std::vector<double> h2d_end((size_t)nb, 0.0), bf((size_t)nb, 0.0), slab_release((size_t)K, 0.0);
  std::vector<int> holder((size_t)K, -1);  // job holding each slab (-1: released at slab_release)
  int nblocks = 0;
  for (int v = 0; v < n; ++v) nblocks = in.block[v] + 1 > nblocks ? in.block[v] + 1 : nblocks;
  std::vector<double> adam_done((size_t)steps * nblocks, -1.0);  // [step][block]
  double drv = 0, w_free = 0, c_free = 0, g_free = 0;
  double first_c[2] = {0, 0}, stall_sum = 0, slab_sum = 0, pack_sum = 0;
  auto release_of = [&](int k) {
    return holder[(size_t)k] < 0 ? slab_release[(size_t)k] : ad.jobs[(size_t)holder[(size_t)k]].end;
  };
  for (int s = 0; s < steps; ++s) {
    const int rec = s == steps - 1 ? 1 : (s == steps - 2 ? 0 : -1);
    for (int v = 0; v < n; ++v) {
      const int kind = in.kind[v], j = in.block[v], b = v % nb;
      double t = drv;
      if (kind <= 1 && s > 0) {  // the forward of block j waits for its previous Adam
        const size_t idx = (size_t)(s - 1) * nblocks + j;
        while (adam_done[idx] < 0 && ad.next())
          for (const SimJob& jb : ad.jobs)
            if (jb.end >= 0) adam_done[(size_t)jb.step * nblocks + jb.block] = jb.end;
        if (adam_done[idx] > t) t = adam_done[idx];
      }
      double pack_end = t, first_chunk = t;
      if (in.p[v] > 0) {
        if (h2d_end[(size_t)b] > t) t = h2d_end[(size_t)b];  // staging b free
        const double pk = in.p[v] / prate;
        if (rec == 0) pack_sum += pk;
        first_chunk = t + std::min(in.p[v], in.chunk) / prate;
        pack_end = t + pk;
      }
      // the copy starts once the first chunk is packed, the weight stream is
      // free and the buffer was released; it cannot end before the last chunk
      // is packed and copied
      double hs = first_chunk > w_free ? first_chunk : w_free;
      if (bf[(size_t)b] > hs) hs = bf[(size_t)b];
      double he = hs + in.b[v] / in.bw_h2d;
      if (in.p[v] > 0) he = std::max(he, pack_end + std::min(in.b[v], in.chunk) / in.bw_h2d);
      w_free = he;
      h2d_end[(size_t)b] = he;
      drv = pack_end;
      const double cs = c_free > he ? c_free : he;
      // the period runs from step steps-2's first compute to step steps-1's
      if ((rec == 0 && v > 0) || (rec == 1 && v == 0)) stall_sum += cs - c_free;
      if (rec >= 0 && v == 0) first_c[rec] = cs;
      if (rec == 1 && stall_v) stall_v[v] = cs - c_free;
      const double ce = cs + in.c[v];
      c_free = ce;
      if (in.d[v] > 0) {
        // a free slab: one released by the time the driver gets here, else the
        // earliest release of a held one (a held slab whose Adam is not decided
        // yet ends after every decided one)
        int k = -1;
        for (;;) {
          double best_t = 1e300;
          for (int q = 0; q < K; ++q) {
            const double r = release_of(q);
            if (r < 0) continue;
            if (r <= drv) {
              k = q;
              best_t = drv;
              break;
            }
            if (r < best_t) {
              best_t = r;
              k = q;
            }
          }
          if (k >= 0) {
            if (best_t > drv) {
              if (rec == 0) slab_sum += best_t - drv;
              drv = best_t;
            }
            break;
          }
          if (!ad.next()) break;
        }
        if (k < 0) k = 0;
        double gs = ce > g_free ? ce : g_free;
        if (drv > gs) gs = drv;
        const double ge = gs + in.d[v] / in.bw_d2h;
        g_free = ge;
        bf[(size_t)b] = ge;
        ad.jobs.push_back({s, j, ge, in.a[v]});
        holder[(size_t)k] = (int)ad.jobs.size() - 1;
      } else {
        bf[(size_t)b] = ce;
      }
    }
  }
  while (ad.next()) {
  }
  double abusy = 0;  // Adam work inside the period [first_c[0], first_c[1])
  for (const SimJob& jb : ad.jobs) {
    const double a0 = jb.end - jb.elems / ad.rate, a1 = jb.end;
    const double lo = a0 > first_c[0] ? a0 : first_c[0], hi = a1 < first_c[1] ? a1 : first_c[1];
    if (hi > lo) abusy += hi - lo;
  }
  out.period = first_c[1] - first_c[0];
  out.stall = stall_sum;
  out.adam_busy = abusy;
  out.slab_wait = slab_sum;
  out.pack = pack_sum;
  out.adam_rate = adam_rate;
  return out;
}
}  // namespace

SimOut simulate(const SimIn& in, int32_t K, int32_t steps, double* stall_v) {
  if (in.n <= 0 || K < 1 || steps < 2 || !(in.bw_h2d > 0) || !(in.bw_d2h > 0)) return SimOut{};
  double r = in.adam_rate;
  SimOut o = simulate_at(in, K, steps, nullptr, r);
  if (in.host_bw > 0 && in.adam_rate > 0) {
    // host memory is shared: Adam gets what DMA and the pack leave of host_bw
    double dma = 0, packed = 0;
    for (int v = 0; v < in.n; ++v) {
      dma += in.b[v] + in.d[v];
      packed += 2.0 * in.p[v];
    }
    for (int it = 0; it < 20 && o.period > 0; ++it) {
      const double left = in.host_bw - (dma + packed) / o.period;
      const double floor_bw = 0.25 * in.host_bw;  // DMA and the pack are never the whole period
      const double r2 = std::min(in.adam_rate, std::max(left, floor_bw) / in.adam_bytes);
      if (std::fabs(r2 - r) <= 1e-3 * r) break;
      r = r2;
      o = simulate_at(in, K, steps, nullptr, r);
    }
  }
  if (stall_v) o = simulate_at(in, K, steps, stall_v, r);
  return o;
}

Plan plan(const SimIn& in, int32_t k_min, int32_t k_max) {
  Plan best;
  if (k_min < 1) k_min = 1;
  if (k_max < k_min) k_max = k_min;
  std::vector<SimOut> all;
  double tmin = 1e300;
  for (int K = k_min; K <= k_max; ++K) {
    all.push_back(simulate(in, K, 4, nullptr));
    tmin = std::min(tmin, all.back().period);
  }
  for (int K = k_min; K <= k_max; ++K)
    if (all[(size_t)(K - k_min)].period <= tmin * 1.005) {
      best.K = K;
      best.out = all[(size_t)(K - k_min)];
      break;
    }
  return best;
}

}  // namespace mth
