// oracle.cpp -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, single-threaded CPU statement of what one step of the
// layer-streamed training method computes.  The method claims to reach the
// result of ordinary full-parameter training exactly: "no quantisation, no
// approximation, the same BF16/FP32 data copied between host and device"
// ([Lilting] section 精度の検証; [Review] 4-1).  So this file is the plain
// definition of one training step of a pre-RMSNorm decoder-only transformer
// (SwiGLU MLP, rotate-half RoPE, grouped-query causal attention, untied
// embedding and LM head, next-token cross-entropy) followed by bias-corrected
// Adam on FP32 master weights, computed layer by layer with every activation
// kept and no streaming, recomputation or fusion.
//
// Sources are cited by page title and section; see oracle.h for the list.
// Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may load
// the library built from this file.  It includes nothing from the GPU library.
#include "oracle.h"

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

namespace {

// ---------------------------------------------------------------------------
// SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
// generators", OOPSLA 2014): state advances by the golden gamma, the output is
// the variant-13 finaliser of the state.  The i-th output of a stream seeded
// with s is therefore mix(s + (i+1)*gamma), which is what we evaluate.
// ---------------------------------------------------------------------------
constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ULL;
inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}
inline uint64_t sm_out(uint64_t seed, uint64_t i) { return mix64(seed + (i + 1) * kGamma); }

// Stream key of tensor t of block j: output number 1 + 64*j + t of the seed's
// stream (a tensor index is < 64).
inline uint64_t tensor_key(uint64_t seed, int j, int t) {
  return sm_out(seed, 1 + 64ULL * (uint64_t)j + (uint64_t)t);
}

// Box-Muller (Box and Muller 1958), cosine branch, on two 53-bit uniforms:
// u1 in (0,1] so that log(u1) is finite, u2 in [0,1).
double normal_sample(uint64_t key, uint64_t e) {
  const uint64_t a = sm_out(key, 2 * e), b = sm_out(key, 2 * e + 1);
  const double u1 = (double)((a >> 11) + 1) * 0x1.0p-53;
  const double u2 = (double)(b >> 11) * 0x1.0p-53;
  return std::sqrt(-2.0 * std::log(u1)) * std::cos(2.0 * M_PI * u2);
}

// IEEE binary32 -> bfloat16, round to nearest even (NaN kept quiet).
uint16_t bf16_rne(float x) {
  uint32_t u;
  std::memcpy(&u, &x, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
  const uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}
float bf16_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// ---------------------------------------------------------------------------
// Flat layer-contiguous layout.  [Hotdry] (host memory layout, "layer-contiguous
// memory tiling") and [Review] 3-2 (4) state that one layer's BF16 weights, BF16
// gradients and FP32 optimiser state form one contiguous block so that a
// layer's stream-in is a single burst.  The pages give no finer order; the
// reading used here: regions W(bf16) | G(bf16) | master(f32) | m(f32) | v(f32),
// each starting on a 4096-byte boundary of the block; inside every region the
// same tensors sit at the same element offsets, each rounded up to 128
// elements (256 bytes of bf16).  Tensors are row-major [out, in].
//   block 0      : E [V, H]
//   block 1..L   : W_qkv [(nh+2nkv)hd, H], W_o [H, nh hd], W_gu [2F, H],
//                  W_down [H, F], gamma1 [H], gamma2 [H]
//   block L+1    : gamma_f [H], W_head [V, H]
// With n_experts = E > 0 (routed mixture of experts, [Lilting] MoE section)
// a decoder block holds W_qkv, W_o, W_router [E, H], W_experts [E, 3 Fe H],
// gamma1, gamma2, where row e of W_experts is expert e's W_gu [2Fe, H]
// followed by its W_down [H, Fe]: one expert is one contiguous range, so
// streaming only the routed experts copies whole rows of this tensor.
// ---------------------------------------------------------------------------
struct Tensor { int64_t off, rows, cols; };
struct Block {
  std::vector<Tensor> t;
  int64_t n_real = 0, n_pad = 0;
  int64_t off_W = 0, off_G = 0, off_M = 0, off_m = 0, off_v = 0, bytes = 0, store_off = 0;
};
inline int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

bool cfg_ok(const or_cfg* c) {
  return c && c->n_layers >= 0 && c->hidden > 0 && c->n_heads > 0 && c->n_kv_heads > 0 &&
         c->n_heads % c->n_kv_heads == 0 && c->head_dim > 0 && c->head_dim % 2 == 0 &&
         c->ffn > 0 && c->vocab > 0 && c->batch > 0 && c->seq > 0 && c->micro > 0 &&
         c->n_experts >= 0 &&
         (c->n_experts == 0 || (c->top_k >= 1 && c->top_k <= c->n_experts && c->expert_ffn > 0));
}

Block make_block(const or_cfg* c, int j) {
  const int64_t H = c->hidden, hd = c->head_dim, nh = c->n_heads, nkv = c->n_kv_heads;
  const int64_t F = c->ffn, V = c->vocab, L = c->n_layers;
  std::vector<std::pair<int64_t, int64_t>> shapes;
  if (j == 0) shapes = {{V, H}};
  else if (j <= L && c->n_experts > 0)
    shapes = {{(nh + 2 * nkv) * hd, H}, {H, nh * hd}, {c->n_experts, H},
              {c->n_experts, 3 * (int64_t)c->expert_ffn * H}, {H, 1}, {H, 1}};
  else if (j <= L) shapes = {{(nh + 2 * nkv) * hd, H}, {H, nh * hd}, {2 * F, H}, {H, F}, {H, 1}, {H, 1}};
  else shapes = {{H, 1}, {V, H}};
  Block b;
  int64_t cur = 0;
  for (auto& s : shapes) {
    cur = round_up(cur, 128);
    b.t.push_back({cur, s.first, s.second});
    cur += s.first * s.second;
    b.n_real += s.first * s.second;
  }
  b.n_pad = round_up(cur, 128);
  const int64_t wb = round_up(2 * b.n_pad, 4096), fb = round_up(4 * b.n_pad, 4096);
  b.off_W = 0;
  b.off_G = wb;
  b.off_M = 2 * wb;
  b.off_m = 2 * wb + fb;
  b.off_v = 2 * wb + 2 * fb;
  b.bytes = 2 * wb + 3 * fb;
  return b;
}

std::vector<Block> make_layout(const or_cfg* c) {
  std::vector<Block> v;
  int64_t off = 0;
  for (int j = 0; j < c->n_layers + 2; ++j) {
    Block b = make_block(c, j);
    b.store_off = off;
    off += b.bytes;
    v.push_back(b);
  }
  return v;
}

// ---------------------------------------------------------------------------
// Model arithmetic, templated on the storage scalar S.  Every sum is carried
// in double.  Rows are tokens ordered [sequence][position]; a step has
// n_seq = micro*batch sequences of `seq` positions.
// ---------------------------------------------------------------------------

// RMSNorm: y = x * (mean(x^2) + eps)^(-1/2) * gamma.
template <class S>
void rmsnorm_fwd(const S* x, const S* g, int64_t T, int64_t H, double eps, S* y, S* rstd) {
  for (int64_t r = 0; r < T; ++r) {
    double ss = 0;
    for (int64_t i = 0; i < H; ++i) ss += (double)x[r * H + i] * (double)x[r * H + i];
    const double rs = 1.0 / std::sqrt(ss / (double)H + eps);
    rstd[r] = (S)rs;
    for (int64_t i = 0; i < H; ++i) y[r * H + i] = (S)((double)x[r * H + i] * rs * (double)g[i]);
  }
}
// Gradient of the above: with r = rstd,
//   dx_k = r * gamma_k * dy_k - (r^3 / H) * x_k * sum_i(dy_i gamma_i x_i),
//   dgamma_i += sum_rows dy_i * x_i * r.
template <class S>
void rmsnorm_bwd(const S* dy, const S* x, const S* g, const S* rstd, int64_t T, int64_t H, S* dx,
                 S* dg) {
  std::vector<double> acc(H, 0.0);
  for (int64_t i = 0; i < H; ++i) acc[i] = (double)dg[i];
  for (int64_t r = 0; r < T; ++r) {
    const double rs = (double)rstd[r];
    double dot = 0;
    for (int64_t i = 0; i < H; ++i) dot += (double)dy[r * H + i] * (double)g[i] * (double)x[r * H + i];
    for (int64_t i = 0; i < H; ++i) {
      const double xi = (double)x[r * H + i];
      dx[r * H + i] = (S)(rs * (double)g[i] * (double)dy[r * H + i] - rs * rs * rs / (double)H * xi * dot);
      acc[i] += (double)dy[r * H + i] * xi * rs;
    }
  }
  for (int64_t i = 0; i < H; ++i) dg[i] = (S)acc[i];
}

// Linear maps with weights stored [out=N, in=K]:  Y = X W^T,  dX = dY W,
// dW = dY^T X.  Each output element is one dot product.
template <class S>
void linear_fwd(const S* X, const S* W, int64_t T, int64_t N, int64_t K, S* Y) {
  for (int64_t t = 0; t < T; ++t)
    for (int64_t n = 0; n < N; ++n) {
      const S* a = X + t * K;
      const S* b = W + n * K;
      double s = 0;
#pragma omp simd reduction(+ : s)
      for (int64_t k = 0; k < K; ++k) s += (double)a[k] * (double)b[k];
      Y[t * N + n] = (S)s;
    }
}
template <class S>
void linear_dgrad(const S* dY, const S* W, int64_t T, int64_t N, int64_t K, S* dX) {
  std::vector<double> row(K);
  for (int64_t t = 0; t < T; ++t) {
    std::fill(row.begin(), row.end(), 0.0);
    for (int64_t n = 0; n < N; ++n) {
      const double d = (double)dY[t * N + n];
      if (d == 0.0) continue;
      const S* w = W + n * K;
#pragma omp simd
      for (int64_t k = 0; k < K; ++k) row[k] += d * (double)w[k];
    }
    for (int64_t k = 0; k < K; ++k) dX[t * K + k] = (S)row[k];
  }
}
template <class S>
void linear_wgrad(const S* dY, const S* X, int64_t T, int64_t N, int64_t K, S* dW) {
  std::vector<double> acc((size_t)N * K, 0.0);
  for (int64_t t = 0; t < T; ++t)
    for (int64_t n = 0; n < N; ++n) {
      const double d = (double)dY[t * N + n];
      if (d == 0.0) continue;
      const S* x = X + t * K;
      double* a = acc.data() + n * K;
#pragma omp simd
      for (int64_t k = 0; k < K; ++k) a[k] += d * (double)x[k];
    }
  for (size_t i = 0; i < acc.size(); ++i) dW[i] = (S)acc[i];
}

// Rotate-half RoPE on n_heads heads of width hd at column 0 of each row (row
// stride ld).  Position = index inside the sequence.  theta_i = base^(-2i/hd),
// angle = pos * theta_i, both in double.  inverse != 0 applies the transpose
// (= inverse) rotation, which is the backward map.
template <class S>
void rope(S* x, int64_t n_seq, int64_t Sq, int64_t ld, int64_t n_heads, int64_t hd, double base,
          int inverse) {
  const int64_t half = hd / 2;
  for (int64_t n = 0; n < n_seq; ++n)
    for (int64_t p = 0; p < Sq; ++p) {
      S* row = x + (n * Sq + p) * ld;
      for (int64_t h = 0; h < n_heads; ++h)
        for (int64_t i = 0; i < half; ++i) {
          const double th = std::pow(base, -2.0 * (double)i / (double)hd);
          const double ang = (double)p * th;
          const double c = std::cos(ang), s = inverse ? -std::sin(ang) : std::sin(ang);
          const double a = (double)row[h * hd + i], b = (double)row[h * hd + half + i];
          row[h * hd + i] = (S)(a * c - b * s);
          row[h * hd + half + i] = (S)(b * c + a * s);
        }
    }
}

// Causal grouped-query attention.  qkv rows hold [q (nh*hd) | k (nkv*hd) |
// v (nkv*hd)]; query head h reads key/value head h / (nh/nkv).  For query
// position i: s_j = q_i.k_j / sqrt(hd) for j <= i, p = softmax(s), o_i =
// sum_j p_j v_j; lse_i = log sum_j exp(s_j) is kept for the backward.
template <class S>
void attention_fwd(const S* qkv, int64_t n_seq, int64_t Sq, int64_t nh, int64_t nkv, int64_t hd, S* o,
                   S* lse) {
  const int64_t ld = (nh + 2 * nkv) * hd, grp = nh / nkv;
  const double scale = 1.0 / std::sqrt((double)hd);
  std::vector<double> s(Sq), acc(hd);
  for (int64_t n = 0; n < n_seq; ++n)
    for (int64_t h = 0; h < nh; ++h) {
      const int64_t kh = h / grp;
      for (int64_t i = 0; i < Sq; ++i) {
        const S* q = qkv + (n * Sq + i) * ld + h * hd;
        double mx = -INFINITY;
        for (int64_t j = 0; j <= i; ++j) {
          const S* k = qkv + (n * Sq + j) * ld + nh * hd + kh * hd;
          double d = 0;
          for (int64_t e = 0; e < hd; ++e) d += (double)q[e] * (double)k[e];
          s[j] = d * scale;
          if (s[j] > mx) mx = s[j];
        }
        double den = 0;
        for (int64_t j = 0; j <= i; ++j) den += std::exp(s[j] - mx);
        std::fill(acc.begin(), acc.end(), 0.0);
        for (int64_t j = 0; j <= i; ++j) {
          const double p = std::exp(s[j] - mx) / den;
          const S* v = qkv + (n * Sq + j) * ld + (nh + nkv) * hd + kh * hd;
          for (int64_t e = 0; e < hd; ++e) acc[e] += p * (double)v[e];
        }
        for (int64_t e = 0; e < hd; ++e) o[(n * Sq + i) * nh * hd + h * hd + e] = (S)acc[e];
        lse[(n * Sq + i) * nh + h] = (S)(mx + std::log(den));
      }
    }
}
// Backward of the above (textbook softmax calculus):
//   dv_j += p_ij do_i,  dp_ij = do_i.v_j,  ds_ij = p_ij (dp_ij - sum_l p_il dp_il),
//   dq_i = scale * sum_j ds_ij k_j,  dk_j += scale * ds_ij q_i;
// key/value gradients of a shared head sum over its query heads.
template <class S>
void attention_bwd(const S* qkv, const S* o, const S* lse, const S* dout, int64_t n_seq, int64_t Sq,
                   int64_t nh, int64_t nkv, int64_t hd, S* dqkv) {
  (void)o;
  const int64_t ld = (nh + 2 * nkv) * hd, grp = nh / nkv;
  const double scale = 1.0 / std::sqrt((double)hd);
  std::vector<double> dacc((size_t)n_seq * Sq * ld, 0.0);
  std::vector<double> p(Sq), dp(Sq);
  for (int64_t n = 0; n < n_seq; ++n)
    for (int64_t h = 0; h < nh; ++h) {
      const int64_t kh = h / grp;
      for (int64_t i = 0; i < Sq; ++i) {
        const S* q = qkv + (n * Sq + i) * ld + h * hd;
        const S* dO = dout + (n * Sq + i) * nh * hd + h * hd;
        const double L = (double)lse[(n * Sq + i) * nh + h];
        double dsum = 0;
        for (int64_t j = 0; j <= i; ++j) {
          const S* k = qkv + (n * Sq + j) * ld + nh * hd + kh * hd;
          const S* v = qkv + (n * Sq + j) * ld + (nh + nkv) * hd + kh * hd;
          double d = 0, e2 = 0;
          for (int64_t e = 0; e < hd; ++e) {
            d += (double)q[e] * (double)k[e];
            e2 += (double)dO[e] * (double)v[e];
          }
          p[j] = std::exp(d * scale - L);
          dp[j] = e2;
          dsum += p[j] * dp[j];
        }
        double* dq = dacc.data() + (n * Sq + i) * ld + h * hd;
        for (int64_t j = 0; j <= i; ++j) {
          const double ds = p[j] * (dp[j] - dsum);
          const S* k = qkv + (n * Sq + j) * ld + nh * hd + kh * hd;
          double* dk = dacc.data() + (n * Sq + j) * ld + nh * hd + kh * hd;
          double* dv = dacc.data() + (n * Sq + j) * ld + (nh + nkv) * hd + kh * hd;
          for (int64_t e = 0; e < hd; ++e) {
            dq[e] += scale * ds * (double)k[e];
            dk[e] += scale * ds * (double)q[e];
            dv[e] += p[j] * (double)dO[e];
          }
        }
      }
    }
  for (size_t i = 0; i < dacc.size(); ++i) dqkv[i] = (S)dacc[i];
}

// SwiGLU: gu rows hold [g (F) | u (F)]; h = silu(g) * u, silu(z) = z / (1 + e^-z).
inline double sigmoid(double z) { return 1.0 / (1.0 + std::exp(-z)); }
template <class S>
void swiglu_fwd(const S* gu, int64_t T, int64_t F, S* h) {
  for (int64_t t = 0; t < T; ++t)
    for (int64_t i = 0; i < F; ++i) {
      const double g = (double)gu[t * 2 * F + i], u = (double)gu[t * 2 * F + F + i];
      h[t * F + i] = (S)(g * sigmoid(g) * u);
    }
}
// dg = dh * u * sigma(g) (1 + g (1 - sigma(g))),  du = dh * silu(g).
template <class S>
void swiglu_bwd(const S* gu, const S* dh, int64_t T, int64_t F, S* dgu) {
  for (int64_t t = 0; t < T; ++t)
    for (int64_t i = 0; i < F; ++i) {
      const double g = (double)gu[t * 2 * F + i], u = (double)gu[t * 2 * F + F + i];
      const double d = (double)dh[t * F + i], sg = sigmoid(g);
      dgu[t * 2 * F + i] = (S)(d * u * sg * (1.0 + g * (1.0 - sg)));
      dgu[t * 2 * F + F + i] = (S)(d * g * sg);
    }
}

// Next-token cross-entropy.  Position p of a sequence predicts token p+1; the
// last position has no target.  loss = sum over targets of
// (logsumexp(logits) - logits[target]) / norm, and dlogits = (softmax -
// onehot) / norm on rows with a target, 0 elsewhere.
template <class S>
double cross_entropy(const S* logits, const int32_t* tok, int64_t n_seq, int64_t Sq, int64_t V,
                     double norm, S* dlogits) {
  double total = 0;
  for (int64_t n = 0; n < n_seq; ++n)
    for (int64_t p = 0; p < Sq; ++p) {
      const S* z = logits + (n * Sq + p) * V;
      S* dz = dlogits + (n * Sq + p) * V;
      if (p == Sq - 1) {
        for (int64_t i = 0; i < V; ++i) dz[i] = (S)0;
        continue;
      }
      const int32_t tgt = tok[n * Sq + p + 1];
      double mx = -INFINITY;
      for (int64_t i = 0; i < V; ++i) mx = std::max(mx, (double)z[i]);
      double den = 0;
      for (int64_t i = 0; i < V; ++i) den += std::exp((double)z[i] - mx);
      const double lse = mx + std::log(den);
      total += lse - (double)z[tgt];
      for (int64_t i = 0; i < V; ++i)
        dz[i] = (S)((std::exp((double)z[i] - lse) - (i == tgt ? 1.0 : 0.0)) / norm);
    }
  return total / norm;
}

// ---------------------------------------------------------------------------
// Routed mixture-of-experts feed-forward ([Lilting] MoE section: per token the
// router picks a few of the experts; GPT-OSS-style layer).  Readings where the
// pages are silent: router logits = yn Wr^T with no bias; the selected experts
// of token t are its top_k largest logits, equal logits ordered by lower
// expert index; gates = softmax over the selected logits only; expert e is the
// same SwiGLU MLP as the dense layer with its own weights; no auxiliary
// (load-balancing) loss term:
//   x2_t = x1_t + sum_i gate_ti FFN_{e_ti}(yn_t),
//   FFN_e(y) = (silu(y Wg_e^T) * (y Wu_e^T)) Wd_e^T.
// The rows routed to expert e are processed as one matrix, in ascending
// (token, slot) order.  Backward: dgate_ti = dx2_t . FFN_e(yn_t); the
// expert's output rows get dY = gate_ti dx2_t; softmax over the selected set
// gives dlogit_{t,e_i} = gate_ti (dgate_ti - sum_l gate_tl dgate_tl) and zero
// for the others; the selection itself has no gradient.  An expert no token
// was routed to gets a zero gradient.
// ---------------------------------------------------------------------------
template <class S>
struct MoeLayer {
  int64_t T, H, E, k, Fe;
  std::vector<int32_t> idx;                 // [T][k]
  std::vector<S> gate;                      // [T][k]
  std::vector<int64_t> pos;                 // row of assignment t*k+i inside its expert's rows
  std::vector<std::vector<int64_t>> rows;   // per expert: its assignments t*k+i, ascending
  std::vector<std::vector<S>> X, GU, Hh, Y; // per expert, one row per routed assignment
  double min_margin = INFINITY;

  const S* wgu(const S* We, int64_t e) const { return We + e * 3 * Fe * H; }
  const S* wd(const S* We, int64_t e) const { return We + e * 3 * Fe * H + 2 * Fe * H; }

  void forward(const S* yn, const S* x1, const S* Wr, const S* We, S* out) {
    std::vector<S> lg((size_t)(T * E));
    linear_fwd(yn, Wr, T, E, H, lg.data());
    idx.assign((size_t)(T * k), 0);
    gate.assign((size_t)(T * k), (S)0);
    pos.assign((size_t)(T * k), 0);
    rows.assign((size_t)E, {});
    std::vector<int64_t> ord((size_t)E);
    for (int64_t t = 0; t < T; ++t) {
      const S* l = lg.data() + t * E;
      for (int64_t e = 0; e < E; ++e) ord[(size_t)e] = e;
      std::stable_sort(ord.begin(), ord.end(), [&](int64_t a, int64_t b) { return (double)l[a] > (double)l[b]; });
      if (k < E) min_margin = std::min(min_margin, (double)l[ord[(size_t)k - 1]] - (double)l[ord[(size_t)k]]);
      const double mx = (double)l[ord[0]];
      double den = 0;
      for (int64_t i = 0; i < k; ++i) den += std::exp((double)l[ord[(size_t)i]] - mx);
      for (int64_t i = 0; i < k; ++i) {
        const int64_t e = ord[(size_t)i];
        idx[(size_t)(t * k + i)] = (int32_t)e;
        gate[(size_t)(t * k + i)] = (S)(std::exp((double)l[e] - mx) / den);
        pos[(size_t)(t * k + i)] = (int64_t)rows[(size_t)e].size();
        rows[(size_t)e].push_back(t * k + i);
      }
    }
    X.assign((size_t)E, {}); GU.assign((size_t)E, {}); Hh.assign((size_t)E, {}); Y.assign((size_t)E, {});
    for (int64_t e = 0; e < E; ++e) {
      const int64_t n = (int64_t)rows[(size_t)e].size();
      if (!n) continue;
      auto& Xe = X[(size_t)e];
      Xe.resize((size_t)(n * H));
      for (int64_t r = 0; r < n; ++r) {
        const int64_t t = rows[(size_t)e][(size_t)r] / k;
        std::copy(yn + t * H, yn + (t + 1) * H, Xe.begin() + r * H);
      }
      GU[(size_t)e].resize((size_t)(n * 2 * Fe));
      Hh[(size_t)e].resize((size_t)(n * Fe));
      Y[(size_t)e].resize((size_t)(n * H));
      linear_fwd(Xe.data(), wgu(We, e), n, 2 * Fe, H, GU[(size_t)e].data());
      swiglu_fwd(GU[(size_t)e].data(), n, Fe, Hh[(size_t)e].data());
      linear_fwd(Hh[(size_t)e].data(), wd(We, e), n, H, Fe, Y[(size_t)e].data());
    }
    for (int64_t t = 0; t < T; ++t)
      for (int64_t h = 0; h < H; ++h) {
        double s = (double)x1[t * H + h];
        for (int64_t i = 0; i < k; ++i) {
          const int64_t a = t * k + i;
          s += (double)gate[(size_t)a] * (double)Y[(size_t)idx[(size_t)a]][(size_t)(pos[(size_t)a] * H + h)];
        }
        out[t * H + h] = (S)s;
      }
  }

  // dout = d loss / d x2; writes dyn (the part through this feed-forward),
  // dWr and every expert's slice of dWe (zeros for experts with no rows).
  void backward(const S* yn, const S* Wr, const S* We, const S* dout, S* dyn, S* dWr, S* dWe) const {
    std::vector<double> acc((size_t)(T * H), 0.0);
    std::vector<double> dgate((size_t)(T * k), 0.0);
    for (int64_t a = 0; a < T * k; ++a) {
      const int64_t t = a / k;
      const S* y = Y[(size_t)idx[(size_t)a]].data() + pos[(size_t)a] * H;
      double s = 0;
      for (int64_t h = 0; h < H; ++h) s += (double)dout[t * H + h] * (double)y[h];
      dgate[(size_t)a] = s;
    }
    std::fill(dWe, dWe + E * 3 * Fe * H, (S)0);
    for (int64_t e = 0; e < E; ++e) {
      const int64_t n = (int64_t)rows[(size_t)e].size();
      if (!n) continue;
      std::vector<S> dY((size_t)(n * H)), dH((size_t)(n * Fe)), dGU((size_t)(n * 2 * Fe)), dX((size_t)(n * H));
      for (int64_t r = 0; r < n; ++r) {
        const int64_t a = rows[(size_t)e][(size_t)r], t = a / k;
        for (int64_t h = 0; h < H; ++h) dY[(size_t)(r * H + h)] = (S)((double)gate[(size_t)a] * (double)dout[t * H + h]);
      }
      S* gwgu = dWe + e * 3 * Fe * H;
      S* gwd = gwgu + 2 * Fe * H;
      linear_wgrad(dY.data(), Hh[(size_t)e].data(), n, H, Fe, gwd);
      linear_dgrad(dY.data(), wd(We, e), n, H, Fe, dH.data());
      swiglu_bwd(GU[(size_t)e].data(), dH.data(), n, Fe, dGU.data());
      linear_wgrad(dGU.data(), X[(size_t)e].data(), n, 2 * Fe, H, gwgu);
      linear_dgrad(dGU.data(), wgu(We, e), n, 2 * Fe, H, dX.data());
      for (int64_t r = 0; r < n; ++r) {
        const int64_t t = rows[(size_t)e][(size_t)r] / k;
        for (int64_t h = 0; h < H; ++h) acc[(size_t)(t * H + h)] += (double)dX[(size_t)(r * H + h)];
      }
    }
    std::vector<S> dl((size_t)(T * E), (S)0), tmp((size_t)(T * H));
    for (int64_t t = 0; t < T; ++t) {
      double s = 0;
      for (int64_t i = 0; i < k; ++i) s += (double)gate[(size_t)(t * k + i)] * dgate[(size_t)(t * k + i)];
      for (int64_t i = 0; i < k; ++i) {
        const int64_t a = t * k + i;
        dl[(size_t)(t * E + idx[(size_t)a])] = (S)((double)gate[(size_t)a] * (dgate[(size_t)a] - s));
      }
    }
    linear_wgrad(dl.data(), yn, T, E, H, dWr);
    linear_dgrad(dl.data(), Wr, T, E, H, tmp.data());
    for (int64_t i = 0; i < T * H; ++i) dyn[i] = (S)(acc[(size_t)i] + (double)tmp[(size_t)i]);
  }
};

double g_last_margin = INFINITY;

template <class S>
double moe_layer(int64_t T, int64_t H, int64_t E, int64_t k, int64_t Fe, const S* yn, const S* x1, const S* Wr,
                 const S* We, const S* dout, S* out, S* dyn, S* dWr, S* dWe, int32_t* idx, S* gate) {
  if (T < 0 || H <= 0 || E <= 0 || k < 1 || k > E || Fe <= 0) return NAN;
  MoeLayer<S> m{T, H, E, k, Fe};
  m.forward(yn, x1, Wr, We, out);
  m.backward(yn, Wr, We, dout, dyn, dWr, dWe);
  std::copy(m.idx.begin(), m.idx.end(), idx);
  std::copy(m.gate.begin(), m.gate.end(), gate);
  return m.min_margin;
}

// ---------------------------------------------------------------------------
// One training step: embedding -> L decoder blocks -> final RMSNorm + LM head
// -> loss, then the backward in reverse.  Decoder block (pre-RMSNorm):
//   xn = RMSNorm(x, g1); [q|k|v] = xn Wqkv^T; RoPE(q, k); a = Attn(q, k, v)
//   x1 = x + a Wo^T;  yn = RMSNorm(x1, g2); [g|u] = yn Wgu^T; h = silu(g) u
//   x2 = x1 + h Wd^T
// Gradients of all micro-batches of the step are summed (the step loss is the
// mean over micro-batches of each micro-batch's mean token loss; every
// micro-batch has the same number of targets, so it is one mean over all).
// ---------------------------------------------------------------------------
template <class S>
struct Model {
  const or_cfg& c;
  int64_t H, nh, nkv, hd, F, V, L, T, nseq, Sq, ldq;
  std::vector<Block> lay;
  explicit Model(const or_cfg& cc) : c(cc) {
    H = c.hidden; nh = c.n_heads; nkv = c.n_kv_heads; hd = c.head_dim; F = c.ffn; V = c.vocab;
    L = c.n_layers; Sq = c.seq; nseq = (int64_t)c.micro * c.batch; T = nseq * Sq; ldq = (nh + 2 * nkv) * hd;
    lay = make_layout(&c);
  }
  const S* ten(const S* const* W, int j, int t) const { return W[j] + lay[j].t[t].off; }
  S* ten(S* const* G, int j, int t) const { return G[j] + lay[j].t[t].off; }

  struct LayerActs {
    std::vector<S> x, xn, r1, qkv, a, lse, x1, yn, r2, gu, h;
    MoeLayer<S> moe;
  };
  bool moe() const { return c.n_experts > 0; }
  double min_margin = INFINITY;

  void layer_fwd(const S* const* W, int j, const std::vector<S>& x, LayerActs& A, std::vector<S>& out) {
    A.x = x;
    A.xn.resize(T * H); A.r1.resize(T); A.qkv.resize(T * ldq); A.a.resize(T * nh * hd);
    A.lse.resize(T * nh); A.x1.resize(T * H); A.yn.resize(T * H); A.r2.resize(T);
    if (!moe()) { A.gu.resize(T * 2 * F); A.h.resize(T * F); }
    out.resize(T * H);
    rmsnorm_fwd(x.data(), ten(W, j, 4), T, H, c.rms_eps, A.xn.data(), A.r1.data());
    linear_fwd(A.xn.data(), ten(W, j, 0), T, ldq, H, A.qkv.data());
    rope(A.qkv.data(), nseq, Sq, ldq, nh + nkv, hd, c.rope_base, 0);  // q heads then k heads
    attention_fwd(A.qkv.data(), nseq, Sq, nh, nkv, hd, A.a.data(), A.lse.data());
    std::vector<S> tmp(T * H);
    linear_fwd(A.a.data(), ten(W, j, 1), T, H, nh * hd, tmp.data());
    for (int64_t i = 0; i < T * H; ++i) A.x1[i] = (S)((double)x[i] + (double)tmp[i]);
    rmsnorm_fwd(A.x1.data(), ten(W, j, 5), T, H, c.rms_eps, A.yn.data(), A.r2.data());
    if (moe()) {
      A.moe = MoeLayer<S>{T, H, (int64_t)c.n_experts, (int64_t)c.top_k, (int64_t)c.expert_ffn};
      A.moe.forward(A.yn.data(), A.x1.data(), ten(W, j, 2), ten(W, j, 3), out.data());
      min_margin = std::min(min_margin, A.moe.min_margin);
      return;
    }
    linear_fwd(A.yn.data(), ten(W, j, 2), T, 2 * F, H, A.gu.data());
    swiglu_fwd(A.gu.data(), T, F, A.h.data());
    linear_fwd(A.h.data(), ten(W, j, 3), T, H, F, tmp.data());
    for (int64_t i = 0; i < T * H; ++i) out[i] = (S)((double)A.x1[i] + (double)tmp[i]);
  }

  // dx: in = dL/dx2, out = dL/dx (the layer input).
  void layer_bwd(const S* const* W, S* const* G, int j, const LayerActs& A, std::vector<S>& dx) {
    std::vector<S> dh(moe() ? 0 : T * F), dgu(moe() ? 0 : T * 2 * F), dyn(T * H), dx1(T * H), tmp(T * H), da(T * nh * hd);
    std::vector<S> dqkv(T * ldq), dxn(T * H);
    if (moe()) {
      // x2 = x1 + sum_i gate_i FFN_{e_i}(yn)
      A.moe.backward(A.yn.data(), ten(W, j, 2), ten(W, j, 3), dx.data(), dyn.data(), ten(G, j, 2), ten(G, j, 3));
    } else {
      // x2 = x1 + h Wd^T
      linear_wgrad(dx.data(), A.h.data(), T, H, F, ten(G, j, 3));
      linear_dgrad(dx.data(), ten(W, j, 3), T, H, F, dh.data());
      swiglu_bwd(A.gu.data(), dh.data(), T, F, dgu.data());
      linear_wgrad(dgu.data(), A.yn.data(), T, 2 * F, H, ten(G, j, 2));
      linear_dgrad(dgu.data(), ten(W, j, 2), T, 2 * F, H, dyn.data());
    }
    rmsnorm_bwd(dyn.data(), A.x1.data(), ten(W, j, 5), A.r2.data(), T, H, tmp.data(), ten(G, j, 5));
    for (int64_t i = 0; i < T * H; ++i) dx1[i] = (S)((double)dx[i] + (double)tmp[i]);
    // x1 = x + a Wo^T
    linear_wgrad(dx1.data(), A.a.data(), T, H, nh * hd, ten(G, j, 1));
    linear_dgrad(dx1.data(), ten(W, j, 1), T, H, nh * hd, da.data());
    attention_bwd(A.qkv.data(), A.a.data(), A.lse.data(), da.data(), nseq, Sq, nh, nkv, hd, dqkv.data());
    rope(dqkv.data(), nseq, Sq, ldq, nh + nkv, hd, c.rope_base, 1);
    linear_wgrad(dqkv.data(), A.xn.data(), T, ldq, H, ten(G, j, 0));
    linear_dgrad(dqkv.data(), ten(W, j, 0), T, ldq, H, dxn.data());
    rmsnorm_bwd(dxn.data(), A.x.data(), ten(W, j, 4), A.r1.data(), T, H, tmp.data(), ten(G, j, 4));
    for (int64_t i = 0; i < T * H; ++i) dx[i] = (S)((double)dx1[i] + (double)tmp[i]);
  }

  void embed(const S* const* W, const int32_t* tok, std::vector<S>& x) {
    x.resize(T * H);
    const S* E = ten(W, 0, 0);
    for (int64_t t = 0; t < T; ++t)
      for (int64_t i = 0; i < H; ++i) x[t * H + i] = E[(int64_t)tok[t] * H + i];
  }

  double step(const S* const* W, const int32_t* tok, S* const* G) {
    for (int j = 0; j < L + 2; ++j) std::fill(G[j], G[j] + lay[j].n_pad, (S)0);
    std::vector<S> x;
    min_margin = INFINITY;
    embed(W, tok, x);
    std::vector<LayerActs> acts(L);
    for (int j = 1; j <= L; ++j) {
      std::vector<S> y;
      layer_fwd(W, j, x, acts[j - 1], y);
      x.swap(y);
    }
    // head: hn = RMSNorm(x, gf); logits = hn Whead^T
    const int hj = (int)L + 1;
    std::vector<S> hn(T * H), rf(T), logits(T * V), dlog(T * V), dhn(T * H), dx(T * H);
    rmsnorm_fwd(x.data(), ten(W, hj, 0), T, H, c.rms_eps, hn.data(), rf.data());
    linear_fwd(hn.data(), ten(W, hj, 1), T, V, H, logits.data());
    const double norm = (double)nseq * (double)(Sq - 1);
    const double loss = cross_entropy(logits.data(), tok, nseq, Sq, V, norm, dlog.data());
    linear_wgrad(dlog.data(), hn.data(), T, V, H, ten(G, hj, 1));
    linear_dgrad(dlog.data(), ten(W, hj, 1), T, V, H, dhn.data());
    rmsnorm_bwd(dhn.data(), x.data(), ten(W, hj, 0), rf.data(), T, H, dx.data(), ten(G, hj, 0));
    for (int j = (int)L; j >= 1; --j) layer_bwd(W, G, j, acts[j - 1], dx);
    // embedding: dE[tok[t]] += dx[t]
    S* dE = ten(G, 0, 0);
    std::vector<double> acc((size_t)V * H, 0.0);
    for (int64_t t = 0; t < T; ++t)
      for (int64_t i = 0; i < H; ++i) acc[(int64_t)tok[t] * H + i] += (double)dx[t * H + i];
    for (size_t i = 0; i < acc.size(); ++i) dE[i] = (S)acc[i];
    g_last_margin = min_margin;
    return loss;
  }

  double forward_hidden(const S* const* W, const int32_t* tok, int jstop, S* out) {
    std::vector<S> x;
    min_margin = INFINITY;
    embed(W, tok, x);
    for (int j = 1; j <= jstop && j <= L; ++j) {
      LayerActs A;
      std::vector<S> y;
      layer_fwd(W, j, x, A, y);
      x.swap(y);
    }
    std::copy(x.begin(), x.end(), out);
    g_last_margin = min_margin;
    return 0.0;
  }
};

// ---------------------------------------------------------------------------
// Event protocol of one model's life, as the op list the driver enqueues.
// [Hotdry] (three CUDA streams, double buffering, event-driven protocol):
// Weights-Ready is recorded by the weight stream after W_i lands and waited on
// by compute before Bind; Backward-Done is recorded by compute after the local
// gradient and starts the gradient export; Buffer-Free is recorded by the
// gradient stream after the export and waited on by the weight stream before
// it reuses the buffer.  K pinned slabs receive the exports; host threads wait
// on the slab, unpack and run Adam.  Readings where the pages are silent:
//   * visits per step: forward blocks 0..L+1 (the head visit runs forward,
//     loss and backward of the head), then backward blocks L..0; buffer = visit
//     index mod 2, restarting each step;
//   * in a forward visit nothing is exported, so compute records Buffer-Free;
//   * the embedding's backward reads no weights: its visit copies nothing;
//   * an export takes a free slab and the host waits while none is free; which
//     one is an allocation choice, so logs are compared modulo slab numbers and
//     this simulator numbers them round-robin (export count mod K), one valid
//     assignment;
//   * the next step's stream-in of block j waits for block j's Adam;
//   * with host-resident checkpoints, X_j (j < L) leaves on the idle gradient
//     stream during the forward and returns on the weight stream, with the
//     block's weights, for the backward; two device X slots alternate.
// ---------------------------------------------------------------------------
struct Log {
  std::string s;
  int step = 0;
  void op(const char* stream, const char* op, long a, long b) {
    char line[96];
    std::snprintf(line, sizeof line, "%d %s %s %ld %ld\n", step, stream, op, a, b);
    s += line;
  }
};

}  // namespace

// ===========================================================================
// C ABI
// ===========================================================================
extern "C" {

int64_t or_n_blocks(const or_cfg* c) { return cfg_ok(c) ? c->n_layers + 2 : -1; }

int64_t or_layout_block(const or_cfg* c, int32_t j, int64_t* out, int64_t cap) {
  if (!cfg_ok(c) || j < 0 || j > c->n_layers + 1 || !out) return -1;
  auto lay = make_layout(c);
  const Block& b = lay[j];
  const int64_t need = 10 + 3 * (int64_t)b.t.size();
  if (cap < need) return -1;
  out[0] = (int64_t)b.t.size(); out[1] = b.n_real; out[2] = b.n_pad;
  out[3] = b.off_W; out[4] = b.off_G; out[5] = b.off_M; out[6] = b.off_m; out[7] = b.off_v;
  out[8] = b.bytes; out[9] = b.store_off;
  for (size_t t = 0; t < b.t.size(); ++t) {
    out[10 + 3 * t] = b.t[t].off; out[11 + 3 * t] = b.t[t].rows; out[12 + 3 * t] = b.t[t].cols;
  }
  return need;
}

// P = L [H (nh + 2 nkv) hd + nh hd H + 3 H F + 2 H] + 2 V H + H
int64_t or_param_count(const or_cfg* c) {
  if (!cfg_ok(c)) return -1;
  int64_t p = 0;
  for (auto& b : make_layout(c)) p += b.n_real;
  return p;
}
int64_t or_store_bytes(const or_cfg* c) {
  if (!cfg_ok(c)) return -1;
  int64_t s = 0;
  for (auto& b : make_layout(c)) s += b.bytes;
  return s;
}

uint64_t or_splitmix64(uint64_t seed, uint64_t i) { return sm_out(seed, i); }
double or_normal(uint64_t key, uint64_t e) { return normal_sample(key, e); }
uint16_t or_bf16_rne(float x) { return bf16_rne(x); }
float or_bf16_to_f32(uint16_t b) { return bf16_f32(b); }

// Initial FP32 master weights: matrices N(0, init_std) from the tensor's
// stream, RMSNorm gains 1.0 (the gains' initial value is not stated on the
// pages; 1 is the usual RMSNorm initialisation), padding 0.
int32_t or_init_block(const or_cfg* c, uint64_t seed, int32_t j, float* master) {
  if (!cfg_ok(c) || j < 0 || j > c->n_layers + 1 || !master) return -1;
  const Block b = make_layout(c)[j];
  std::fill(master, master + b.n_pad, 0.0f);
  for (size_t t = 0; t < b.t.size(); ++t) {
    const Tensor& T = b.t[t];
    const bool gain = (T.cols == 1);
    const uint64_t key = tensor_key(seed, j, (int)t);
    const int64_t n = T.rows * T.cols;
    for (int64_t e = 0; e < n; ++e)
      master[T.off + e] = gain ? 1.0f : (float)(c->init_std * normal_sample(key, (uint64_t)e));
  }
  return 0;
}

void or_rmsnorm_fwd_d(const double* x, const double* g, int64_t T, int64_t H, double eps, double* y,
                      double* rstd) { rmsnorm_fwd(x, g, T, H, eps, y, rstd); }
void or_rmsnorm_bwd_d(const double* dy, const double* x, const double* g, const double* rstd, int64_t T,
                      int64_t H, double* dx, double* dg) { rmsnorm_bwd(dy, x, g, rstd, T, H, dx, dg); }
void or_linear_fwd_d(const double* X, const double* W, int64_t T, int64_t N, int64_t K, double* Y) {
  linear_fwd(X, W, T, N, K, Y);
}
void or_linear_dgrad_d(const double* dY, const double* W, int64_t T, int64_t N, int64_t K, double* dX) {
  linear_dgrad(dY, W, T, N, K, dX);
}
void or_linear_wgrad_d(const double* dY, const double* X, int64_t T, int64_t N, int64_t K, double* dW) {
  linear_wgrad(dY, X, T, N, K, dW);
}
void or_rope_d(double* x, int64_t n_seq, int64_t S, int64_t ld, int64_t n_heads, int64_t hd, double base,
               int32_t inverse) { rope(x, n_seq, S, ld, n_heads, hd, base, inverse); }
void or_attention_fwd_d(const double* qkv, int64_t n_seq, int64_t S, int64_t nh, int64_t nkv, int64_t hd,
                        double* o, double* lse) { attention_fwd(qkv, n_seq, S, nh, nkv, hd, o, lse); }
void or_attention_bwd_d(const double* qkv, const double* o, const double* lse, const double* dout,
                        int64_t n_seq, int64_t S, int64_t nh, int64_t nkv, int64_t hd, double* dqkv) {
  attention_bwd(qkv, o, lse, dout, n_seq, S, nh, nkv, hd, dqkv);
}
void or_swiglu_fwd_d(const double* gu, int64_t T, int64_t F, double* h) { swiglu_fwd(gu, T, F, h); }
void or_swiglu_bwd_d(const double* gu, const double* dh, int64_t T, int64_t F, double* dgu) {
  swiglu_bwd(gu, dh, T, F, dgu);
}
double or_cross_entropy_d(const double* logits, const int32_t* tok, int64_t n_seq, int64_t S, int64_t V,
                          double norm, double* dlogits) {
  return cross_entropy(logits, tok, n_seq, S, V, norm, dlogits);
}

double or_step_fwd_bwd_f(const or_cfg* c, const float* const* W, const int32_t* tok, float* const* G) {
  if (!cfg_ok(c)) return NAN;
  Model<float> m(*c);
  return m.step(W, tok, G);
}
double or_step_fwd_bwd_d(const or_cfg* c, const double* const* W, const int32_t* tok, double* const* G) {
  if (!cfg_ok(c)) return NAN;
  Model<double> m(*c);
  return m.step(W, tok, G);
}
double or_forward_hidden_f(const or_cfg* c, const float* const* W, const int32_t* tok, int32_t j, float* out) {
  if (!cfg_ok(c)) return NAN;
  Model<float> m(*c);
  return m.forward_hidden(W, tok, j, out);
}

double or_last_route_margin(void) { return g_last_margin; }

double or_moe_layer_d(int64_t T, int64_t H, int64_t E, int64_t k, int64_t Fe, const double* yn, const double* x1,
                      const double* Wr, const double* We, const double* dout, double* out, double* dyn, double* dWr,
                      double* dWe, int32_t* idx, double* gate) {
  return moe_layer(T, H, E, k, Fe, yn, x1, Wr, We, dout, out, dyn, dWr, dWe, idx, gate);
}
double or_moe_layer_f(int64_t T, int64_t H, int64_t E, int64_t k, int64_t Fe, const float* yn, const float* x1,
                      const float* Wr, const float* We, const float* dout, float* out, float* dyn, float* dWr,
                      float* dWe, int32_t* idx, float* gate) {
  return moe_layer(T, H, E, k, Fe, yn, x1, Wr, We, dout, out, dyn, dWr, dWe, idx, gate);
}

// Adam (Kingma and Ba 2015, Algorithm 1) on FP32 master weights with the
// gradient taken from its BF16 copy; then the BF16 working weights are
// re-derived from the master by round-to-nearest-even.  [Review] 3-2 (6) puts
// the update on the CPU; [Lilting] (memory table) fixes BF16 W/G and FP32
// master, m, v.  Decoupled weight decay (AdamW) when weight_decay != 0.
void or_adam_f32(int64_t n, const float* g32, const uint16_t* g_bf16, float* master, float* m, float* v,
                 uint16_t* w_bf16, int32_t step, float lr, float beta1, float beta2, float eps, float weight_decay);
void or_adam(int64_t n, const uint16_t* g_bf16, float* master, float* m, float* v, uint16_t* w_bf16,
             int32_t step, float lr, float beta1, float beta2, float eps, float weight_decay) {
  or_adam_f32(n, nullptr, g_bf16, master, m, v, w_bf16, step, lr, beta1, beta2, eps, weight_decay);
}
// The same update with the gradient given in FP32 (g32), as when micro-batch
// gradients are summed in FP32 on the host before the optimizer step; with
// g32 = nullptr the gradient is float(g_bf16).
void or_adam_f32(int64_t n, const float* g32, const uint16_t* g_bf16, float* master, float* m, float* v,
                 uint16_t* w_bf16, int32_t step, float lr, float beta1, float beta2, float eps, float weight_decay) {
  const float bc1 = (float)(1.0 - std::pow((double)beta1, (double)step));
  const float bc2 = (float)(1.0 - std::pow((double)beta2, (double)step));
  for (int64_t i = 0; i < n; ++i) {
    const float g = g32 ? g32[i] : bf16_f32(g_bf16[i]);
    m[i] = beta1 * m[i] + (1.0f - beta1) * g;
    v[i] = beta2 * v[i] + (1.0f - beta2) * g * g;
    const float mhat = m[i] / bc1;
    const float vhat = v[i] / bc2;
    float th = master[i];
    if (weight_decay != 0.0f) th -= lr * weight_decay * th;
    th -= lr * mhat / (std::sqrt(vhat) + eps);
    master[i] = th;
    w_bf16[i] = bf16_rne(th);
  }
}

}  // extern "C"

namespace {

// Visits of one training step.  Forward j = 0..L, then the head (L+1; its
// forward and backward are fused).  The backward runs block-wise
// recomputation ([Review] 2) streaming forward and block-wise backward: with
// checkpoint interval c only X_s, s in {0, c, 2c, ...} < L, is kept from the
// forward; the decoder layers form segments [s+1, e], e = min(s+c, L), taken
// from the top.  A segment first recomputes X_{s+1} .. X_{e-1} from X_s
// (visits of kind RECOMP, layers s+1 .. e-1 streamed in again) and then runs
// the backward of layers e .. s+1.  The embedding's backward comes last.
// With c = 1 there is no RECOMP visit.  `seg` is the segment's number from the
// top (the checkpoint-load slot is seg % 2); `first` marks the segment's first
// visit, which loads X_s.
struct Visit {
  int kind;  // 0 FWD, 1 HEAD, 2 RECOMP, 3 BWD
  long j;
  long seg;
  bool first;
};
std::vector<Visit> step_visits(long L, long c) {
  std::vector<Visit> v;
  for (long j = 0; j <= L; ++j) v.push_back({0, j, -1, false});
  v.push_back({1, L + 1, -1, false});
  const long nseg = (L + c - 1) / c;
  for (long k = 0; k < nseg; ++k) {
    const long s = (nseg - 1 - k) * c, e = std::min(s + c, L);
    for (long j = s + 1; j <= e - 1; ++j) v.push_back({2, j, k, j == s + 1});
    for (long j = e; j >= s + 1; --j) v.push_back({3, j, k, j == s + 1 && e == s + 1});
  }
  v.push_back({3, 0, -1, false});
  return v;
}

}  // namespace

extern "C" {

// Event protocol of the pages' three-stream engine ([Hotdry] event-driven
// synchronisation): per visit, the weight stream (W) waits Buffer-Free of its
// buffer, copies the block in and records Weights-Ready; compute (C) waits
// Weights-Ready, runs, and records Buffer-Free (forward, recompute: nothing to
// export) or Backward-Done; the gradient stream (G) waits Backward-Done,
// copies the gradients into a free slab, records Buffer-Free and Slab-Ready;
// the host (H) enqueues Adam on the slab.  With host gradient accumulation a
// step is n_passes passes of the whole visit list, one per micro-batch: every
// pass exports its gradients, the host adds them into an FP32 accumulator
// (ACCUM) and only the last pass's export runs Adam; the next step's first
// pass waits for Adam.  Buffers alternate per visit
// (n_buffers = 2) or one buffer serves every visit (n_buffers = 1, the pages'
// single-buffer ablation).  Host-resident checkpoints: the forward saves X_s
// from a two-slot ring (C records XR, G waits it, copies, records XS; the
// next forward write into that slot waits XS), and a segment's first visit
// loads X_s into checkpoint slot seg % 2 on W after waiting XS of the slot X_s
// was saved from.  Slabs are numbered round-robin here, one valid assignment;
// the library takes the lowest free slab and logs are compared modulo that.
int64_t or_protocol(const or_cfg* c, int32_t n_steps, int32_t n_slabs, int32_t ckpt_on_host,
                    int32_t jit_pack, int32_t ckpt_interval, int32_t n_buffers, int32_t n_passes, char* buf,
                    int64_t cap) {
  if (!cfg_ok(c) || n_slabs < 1 || n_steps < 0 || ckpt_interval < 1 || ckpt_interval > c->n_layers ||
      n_buffers < 1 || n_buffers > 2 || n_passes < 1)
    return 0;
  const long L = c->n_layers, ci = ckpt_interval;
  const std::vector<Visit> vis = step_visits(L, ci);
  Log log;
  long exports = 0;
  bool used[2] = {false, false};
  for (int st = 0; st < n_steps; ++st) {
    log.step = st;
    for (int pass = 0; pass < n_passes; ++pass)
    for (size_t vi = 0; vi < vis.size(); ++vi) {
      const Visit& V = vis[vi];
      const long j = V.j, b = (long)vi % n_buffers;
      const bool fwd = V.kind <= 1, head = V.kind == 1;
      const bool copies = !(j == 0 && V.kind == 3);
      if (fwd && st > 0 && pass == 0) log.op("H", "WAIT_ADAM", j, -1);
      if (copies && jit_pack) {
        if (used[b]) log.op("H", "WAIT_STAGE", b, -1);
        log.op("H", "PACK", j, b);
      }
      log.op("W", "WAIT_BF", b, -1);
      if (copies) log.op("W", "H2D", j, b);
      if (V.first && ckpt_on_host) {
        const long s = j - 1;  // the checkpoint X_s feeding this segment
        log.op("W", "WAIT_XS", s % 2, -1);
        log.op("W", "H2D_CKPT", j, V.seg % 2);
      }
      log.op("W", "REC_WR", b, -1);
      used[b] = true;
      log.op("C", "WAIT_WR", b, -1);
      const bool writes_x = V.kind == 0;
      if (writes_x && ckpt_on_host) log.op("C", "WAIT_XS", j % 2, -1);
      static const char* names[4] = {"FWD", "HEAD", "RECOMP", "BWD"};
      log.op("C", names[V.kind], j, b);
      if (V.kind == 0 && j >= 1 && c->n_experts > 0) {
        // MoE forward: compute records Route-Ready after the router's per-expert
        // token counts reached the host; the host reads them and queues the
        // routed experts' copy into the same buffer on W, which records
        // Experts-Ready; compute waits for it and runs the experts.  In the
        // backward (and recompute) the forward's routing is known, so the
        // experts come with the shared weights in the visit's H2D.
        log.op("C", "REC_RT", j, -1);
        log.op("H", "WAIT_RT", j, -1);
        if (jit_pack) log.op("H", "PACK_EXP", j, b);
        log.op("W", "H2D_EXP", j, b);
        log.op("W", "REC_ER", b, -1);
        log.op("C", "WAIT_ER", b, -1);
        log.op("C", "FWD_EXP", j, b);
      }
      const bool saves_x = writes_x && j < L && j % ci == 0 && ckpt_on_host;
      if (saves_x) log.op("C", "REC_XR", j % 2, -1);
      if (V.kind == 0 || V.kind == 2) {
        log.op("C", "REC_BF", b, -1);
      } else {
        log.op("C", "REC_BD", b, -1);
      }
      if (saves_x) {
        log.op("G", "WAIT_XR", j % 2, -1);
        log.op("G", "D2H_CKPT", j, j % 2);
        log.op("G", "REC_XS", j % 2, -1);
      }
      if (V.kind == 3 || head) {
        const long k = exports % n_slabs;
        ++exports;
        log.op("G", "WAIT_BD", b, -1);
        log.op("H", "ACQ_SLAB", k, -1);
        log.op("G", "D2H", j, k);
        log.op("G", "REC_BF", b, -1);
        log.op("G", "REC_SR", k, -1);
        log.op("H", pass + 1 < n_passes ? "ACCUM_ENQ" : "ADAM_ENQ", j, k);
      }
    }
  }
  const int64_t need = (int64_t)log.s.size() + 1;
  if (!buf || cap < need) return -need;
  std::memcpy(buf, log.s.c_str(), (size_t)need);
  return need - 1;
}

// Static prefetch schedule ([Peter] 記憶體預取策略: the prefetch is scheduled
// statically from each layer's parameter bytes, the link bandwidth and the
// layer's compute time).  Reading: with two buffers the stream-in of visit
// v+1 overlaps the compute of visit v and can start once visit v-1 has freed
// its buffer, i.e. after v-1's gradient export, so the predicted wait before
// v+1 computes is
//   stall[v+1] = max(0, d[v-1]/bw_d2h + b[v+1]/bw_h2d - c[v]),
// with stall[0] = b[0]/bw_h2d.  A slab is held from the start of its export to
// the end of its Adam; one export happens per visit, so the pool needs
//   K = max over exporting visits of ceil((d[v]/bw_d2h + a[v]) / c[v]) + 1.
// Arrays are per visit of one step (n_visits entries each); b = H2D bytes,
// d = gradient bytes exported (0 for visits that export nothing), c = compute
// seconds, a = Adam seconds.  The n_blocks argument is the number of visits.
int32_t or_schedule(int32_t n_visits, const double* b, const double* d, const double* cvis,
                    const double* a, double bw_h2d, double bw_d2h, double* stall) {
  if (n_visits <= 0 || bw_h2d <= 0 || bw_d2h <= 0) return -1;
  stall[0] = b[0] / bw_h2d;
  for (int v = 0; v + 1 < n_visits; ++v) {
    const double prev = v >= 1 ? d[v - 1] / bw_d2h : 0.0;
    const double w = prev + b[v + 1] / bw_h2d - cvis[v];
    stall[v + 1] = w > 0 ? w : 0.0;
  }
  int32_t k = 1;
  for (int v = 0; v < n_visits; ++v) {
    if (d[v] <= 0) continue;
    const double hold = d[v] / bw_d2h + a[v];
    const double cv = cvis[v] > 0 ? cvis[v] : 1e-30;
    const int32_t need = (int32_t)std::ceil(hold / cv) + 1;
    if (need > k) k = need;
  }
  return k;
}

}  // extern "C"
