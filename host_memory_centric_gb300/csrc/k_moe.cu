// k_moe.cu -- routed mixture-of-experts kernels (sm_103a).
//
// A routed MoE layer ([Lilting] MoE section: per token the router selects a
// few experts, and only their weights travel to the GPU) runs as:
//   router logits (FP32, a tensor-core GEMM) -> per-token top-k and gates ->
//   a deterministic counting sort of the (token, slot) assignments into
//   per-expert row segments, each padded to whole 128-row tiles -> gather of
//   the normalised input rows -> expert-grouped GEMMs (k_gemm.cu) -> combine
//   (gate-weighted sum plus the residual).  The backward mirrors it: combine
//   backward (gate gradients, router-logit gradients, gate-scaled output
//   gradients), grouped GEMMs, scatter-sum back to tokens.
// Every kernel here is HBM- or latency-bound and small next to the experts'
// GEMMs; rows move as 16-byte vectors, one warp per row.
#include "mt_kernels.h"

namespace mt {
namespace {

constexpr int MOE_CHUNK = 64;  // tokens per counting-sort chunk (one thread each)
constexpr int MOE_MAX_K = 8;

__device__ __forceinline__ float wsum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ void unpack8(const uint4& q, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 q;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&q);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return q;
}

// Per token: the k largest of its E logits in descending order, equal logits
// ordered by lower expert index (a later expert enters only when strictly
// greater), and gates = softmax over the selected logits.
__global__ void moe_topk_k(const float* __restrict__ logits, int64_t T, int E, int k, int32_t* __restrict__ idx,
                           float* __restrict__ gate) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  const float* l = logits + t * E;
  float bv[MOE_MAX_K];
  int bi[MOE_MAX_K];
  for (int i = 0; i < k; ++i) {
    bv[i] = 0.f;
    bi[i] = -1;
  }
  for (int e = 0; e < E; ++e) {
    const float v = l[e];
    if (bi[k - 1] >= 0 && !(v > bv[k - 1])) continue;
    int pos = k - 1;
    while (pos > 0 && (bi[pos - 1] < 0 || v > bv[pos - 1])) {
      bv[pos] = bv[pos - 1];
      bi[pos] = bi[pos - 1];
      --pos;
    }
    bv[pos] = v;
    bi[pos] = e;
  }
  float den = 0.f;
  for (int i = 0; i < k; ++i) den += expf(bv[i] - bv[0]);
  for (int i = 0; i < k; ++i) {
    idx[t * k + i] = bi[i];
    gate[t * k + i] = expf(bv[i] - bv[0]) / den;
  }
}

// Counting sort, pass 1: assignments per (chunk of 64 tokens, expert).
// Shared counters are laid out [expert][thread] so a warp's threads hit
// different banks.
__global__ void moe_count_k(const int32_t* __restrict__ idx, int64_t T, int k, int E, int64_t nch,
                            int32_t* __restrict__ cnt) {
  extern __shared__ int32_t sc[];
  const int tid = threadIdx.x, bd = blockDim.x;
  const int64_t c = (int64_t)blockIdx.x * bd + tid;
  if (c >= nch) return;
  for (int e = 0; e < E; ++e) sc[e * bd + tid] = 0;
  const int64_t t1 = (c + 1) * MOE_CHUNK < T ? (c + 1) * MOE_CHUNK : T;
  for (int64_t t = c * MOE_CHUNK; t < t1; ++t)
    for (int i = 0; i < k; ++i) {
      const int e = idx[t * k + i];
      if (e >= 0 && e < E) sc[e * bd + tid]++;
    }
  for (int e = 0; e < E; ++e) cnt[c * E + e] = sc[e * bd + tid];
}

// Pass 2 (one block, thread = expert): totals, segment starts (each expert's
// rows padded to a multiple of 128), the first row of every (chunk, expert),
// and the expert of every 128-row tile (-1 past the last segment).
__global__ void moe_scan_k(const int32_t* __restrict__ cnt, int64_t nch, int E, int32_t* __restrict__ base,
                           int32_t* __restrict__ counts, int32_t* __restrict__ tile_expert, int max_tiles) {
  __shared__ int32_t tot[128], seg[129];
  const int e = threadIdx.x;
  if (e < E) {
    int32_t s = 0;
    for (int64_t c = 0; c < nch; ++c) s += cnt[c * E + e];
    tot[e] = s;
    counts[e] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t r = 0;
    for (int i = 0; i < E; ++i) {
      seg[i] = r;
      r += (tot[i] + 127) / 128 * 128;
    }
    seg[E] = r;
  }
  __syncthreads();
  if (e < E) {
    int32_t r = seg[e];
    for (int64_t c = 0; c < nch; ++c) {
      base[c * E + e] = r;
      r += cnt[c * E + e];
    }
  }
  for (int tt = threadIdx.x; tt < max_tiles; tt += blockDim.x) {
    const int32_t row = tt * 128;
    int ex = -1;
    for (int i = 0; i < E && ex < 0; ++i)
      if (row >= seg[i] && row < seg[i + 1]) ex = i;
    tile_expert[tt] = ex;
  }
}

// Pass 3: every assignment (t, i) gets the next row of its expert's segment,
// chunks in token order and tokens in order inside a chunk, so rows of one
// expert are in ascending (token, slot) order.
__global__ void moe_place_k(const int32_t* __restrict__ idx, int64_t T, int k, int E, int64_t nch,
                            const int32_t* __restrict__ base, int32_t* __restrict__ perm_tok,
                            int32_t* __restrict__ slot_row) {
  extern __shared__ int32_t sc[];
  const int tid = threadIdx.x, bd = blockDim.x;
  const int64_t c = (int64_t)blockIdx.x * bd + tid;
  if (c >= nch) return;
  for (int e = 0; e < E; ++e) sc[e * bd + tid] = base[c * E + e];
  const int64_t t1 = (c + 1) * MOE_CHUNK < T ? (c + 1) * MOE_CHUNK : T;
  for (int64_t t = c * MOE_CHUNK; t < t1; ++t)
    for (int i = 0; i < k; ++i) {
      const int e = idx[t * k + i];
      if (e < 0 || e >= E) {
        slot_row[t * k + i] = -1;
        continue;
      }
      const int32_t r = sc[e * bd + tid]++;
      perm_tok[r] = (int32_t)t;
      slot_row[t * k + i] = r;
    }
}

constexpr int WARPS = 8;

// xperm[r] = yn[perm_tok[r]], zero rows where perm_tok < 0 (segment padding).
__global__ void __launch_bounds__(256) moe_gather_k(const bf16* __restrict__ yn, int H,
                                                   const int32_t* __restrict__ perm_tok, int64_t R,
                                                   bf16* __restrict__ xperm) {
  const int64_t r = (int64_t)blockIdx.x * WARPS + (threadIdx.x >> 5);
  if (r >= R) return;
  const int lane = threadIdx.x & 31;
  const int32_t t = perm_tok[r];
  uint4* dst = reinterpret_cast<uint4*>(xperm + r * H);
  const uint4* src = reinterpret_cast<const uint4*>(yn + (int64_t)(t < 0 ? 0 : t) * H);
  for (int c = lane; c < H / 8; c += 32) dst[c] = t < 0 ? make_uint4(0, 0, 0, 0) : src[c];
}

// out[t] = x1[t] + sum_i gate[t, i] * Y[slot_row[t, i]] (FP32 sum over i in
// slot order, one rounding to BF16).
__global__ void __launch_bounds__(256) moe_combine_k(const bf16* __restrict__ x1, const bf16* __restrict__ Y,
                                                    const int32_t* __restrict__ slot_row,
                                                    const float* __restrict__ gate, int64_t T, int H, int k,
                                                    bf16* __restrict__ out) {
  const int64_t t = (int64_t)blockIdx.x * WARPS + (threadIdx.x >> 5);
  if (t >= T) return;
  const int lane = threadIdx.x & 31;
  for (int c = lane * 8; c < H; c += 256) {
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int i = 0; i < k; ++i) {
      const int32_t r = slot_row[t * k + i];
      if (r < 0) continue;
      const float g = gate[t * k + i];
      float y[8];
      unpack8(*reinterpret_cast<const uint4*>(Y + (int64_t)r * H + c), y);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] += g * y[q];
    }
    float x[8];
    unpack8(*reinterpret_cast<const uint4*>(x1 + t * H + c), x);
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] += x[q];
    *reinterpret_cast<uint4*>(out + t * H + c) = pack8(acc);
  }
}

// Backward of the combine and of the gates, one warp per token:
//   dgate_i = dout_t . Y[row_i];  dY[row_i] = gate_i * dout_t;
//   dlogit[t, e_i] = gate_i (dgate_i - sum_l gate_l dgate_l), 0 for the other
//   experts (softmax over the selected logits); dlogits is BF16 [T][E].
__global__ void __launch_bounds__(256) moe_combine_bwd_k(const bf16* __restrict__ dout, const bf16* __restrict__ Y,
                                                        const int32_t* __restrict__ slot_row,
                                                        const int32_t* __restrict__ idx,
                                                        const float* __restrict__ gate, int64_t T, int H, int k,
                                                        int E, bf16* __restrict__ dY, bf16* __restrict__ dlogits) {
  const int64_t t = (int64_t)blockIdx.x * WARPS + (threadIdx.x >> 5);
  if (t >= T) return;
  const int lane = threadIdx.x & 31;
  float dg[MOE_MAX_K];
  for (int i = 0; i < k; ++i) {
    const int32_t r = slot_row[t * k + i];
    const float g = gate[t * k + i];
    float s = 0.f;
    if (r >= 0) {
      for (int c = lane * 8; c < H; c += 256) {
        float d[8], y[8], o[8];
        unpack8(*reinterpret_cast<const uint4*>(dout + t * H + c), d);
        unpack8(*reinterpret_cast<const uint4*>(Y + (int64_t)r * H + c), y);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          s += d[q] * y[q];
          o[q] = g * d[q];
        }
        *reinterpret_cast<uint4*>(dY + (int64_t)r * H + c) = pack8(o);
      }
    }
    dg[i] = wsum(s);
  }
  float sg = 0.f;
  for (int i = 0; i < k; ++i) sg += gate[t * k + i] * dg[i];
  for (int e = lane; e < E; e += 32) {
    float v = 0.f;
    for (int i = 0; i < k; ++i)
      if (idx[t * k + i] == e) v = gate[t * k + i] * (dg[i] - sg);
    dlogits[t * E + e] = __float2bfloat16_rn(v);
  }
}

// Zero the rows r < R of buf ([R][cols]) whose perm_tok[r] < 0.
__global__ void __launch_bounds__(256) moe_zero_pad_k(bf16* __restrict__ buf, int cols,
                                                     const int32_t* __restrict__ perm_tok, int64_t R) {
  const int64_t r = (int64_t)blockIdx.x * WARPS + (threadIdx.x >> 5);
  if (r >= R || perm_tok[r] >= 0) return;
  const int lane = threadIdx.x & 31;
  uint4* p = reinterpret_cast<uint4*>(buf + r * cols);
  for (int c = lane; c < cols / 8; c += 32) p[c] = make_uint4(0, 0, 0, 0);
}

// dyn[t] = sum_i dX[slot_row[t, i]] (FP32 in slot order, one BF16 rounding).
__global__ void __launch_bounds__(256) moe_scatter_k(const bf16* __restrict__ dX, const int32_t* __restrict__ slot_row,
                                                    int64_t T, int H, int k, bf16* __restrict__ dyn) {
  const int64_t t = (int64_t)blockIdx.x * WARPS + (threadIdx.x >> 5);
  if (t >= T) return;
  const int lane = threadIdx.x & 31;
  for (int c = lane * 8; c < H; c += 256) {
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int i = 0; i < k; ++i) {
      const int32_t r = slot_row[t * k + i];
      if (r < 0) continue;
      float x[8];
      unpack8(*reinterpret_cast<const uint4*>(dX + (int64_t)r * H + c), x);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] += x[q];
    }
    *reinterpret_cast<uint4*>(dyn + t * H + c) = pack8(acc);
  }
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
unsigned blocks_for(int64_t n, int per) { return (unsigned)((n + per - 1) / per); }

}  // namespace

int64_t moe_rows_max(int64_t T, int E, int k) { return (T * k + (int64_t)E * 127 + 127) / 128 * 128; }
int64_t moe_chunks(int64_t T) { return (T + MOE_CHUNK - 1) / MOE_CHUNK; }

cudaError_t moe_plan(const float* logits, int64_t T, int E, int k, const MoePlan& p, cudaStream_t s) {
  if (T < 0 || E < 1 || E > 128 || k < 1 || k > MOE_MAX_K || k > E) return cudaErrorInvalidValue;
  if (T == 0) return cudaSuccess;
  const int64_t nch = moe_chunks(T), R = moe_rows_max(T, E, k);
  constexpr int TPB = 64;
  const size_t smem = (size_t)E * TPB * sizeof(int32_t);
  moe_topk_k<<<blocks_for(T, 128), 128, 0, s>>>(logits, T, E, k, p.idx, p.gate);
  moe_count_k<<<blocks_for(nch, TPB), TPB, smem, s>>>(p.idx, T, k, E, nch, p.cnt);
  moe_scan_k<<<1, 128, 0, s>>>(p.cnt, nch, E, p.base, p.counts, p.tile_expert, (int)(R / 128));
  cudaError_t e = cudaMemsetAsync(p.perm_tok, 0xFF, (size_t)R * sizeof(int32_t), s);
  if (e != cudaSuccess) return e;
  moe_place_k<<<blocks_for(nch, TPB), TPB, smem, s>>>(p.idx, T, k, E, nch, p.base, p.perm_tok, p.slot_row);
  return cudaGetLastError();
}

cudaError_t moe_gather(const bf16* yn, int H, const int32_t* perm_tok, int64_t R, bf16* xperm, cudaStream_t s) {
  if (H % 8 || !al16(yn) || !al16(xperm)) return cudaErrorInvalidValue;
  if (R <= 0) return cudaSuccess;
  moe_gather_k<<<blocks_for(R, WARPS), 256, 0, s>>>(yn, H, perm_tok, R, xperm);
  return cudaGetLastError();
}

cudaError_t moe_combine(const bf16* x1, const bf16* Y, const int32_t* slot_row, const float* gate, int64_t T, int H,
                        int k, bf16* out, cudaStream_t s) {
  if (H % 8 || !al16(x1) || !al16(Y) || !al16(out)) return cudaErrorInvalidValue;
  if (T <= 0) return cudaSuccess;
  moe_combine_k<<<blocks_for(T, WARPS), 256, 0, s>>>(x1, Y, slot_row, gate, T, H, k, out);
  return cudaGetLastError();
}

cudaError_t moe_combine_bwd(const bf16* dout, const bf16* Y, const int32_t* slot_row, const int32_t* idx,
                            const float* gate, int64_t T, int H, int k, int E, bf16* dY, bf16* dlogits,
                            cudaStream_t s) {
  if (H % 8 || k > MOE_MAX_K || !al16(dout) || !al16(Y) || !al16(dY)) return cudaErrorInvalidValue;
  if (T <= 0) return cudaSuccess;
  moe_combine_bwd_k<<<blocks_for(T, WARPS), 256, 0, s>>>(dout, Y, slot_row, idx, gate, T, H, k, E, dY, dlogits);
  return cudaGetLastError();
}

cudaError_t moe_zero_pad(bf16* buf, int cols, const int32_t* perm_tok, int64_t R, cudaStream_t s) {
  if (cols % 8 || !al16(buf)) return cudaErrorInvalidValue;
  if (R <= 0) return cudaSuccess;
  moe_zero_pad_k<<<blocks_for(R, WARPS), 256, 0, s>>>(buf, cols, perm_tok, R);
  return cudaGetLastError();
}

cudaError_t moe_scatter(const bf16* dX, const int32_t* slot_row, int64_t T, int H, int k, bf16* dyn,
                        cudaStream_t s) {
  if (H % 8 || !al16(dX) || !al16(dyn)) return cudaErrorInvalidValue;
  if (T <= 0) return cudaSuccess;
  moe_scatter_k<<<blocks_for(T, WARPS), 256, 0, s>>>(dX, slot_row, T, H, k, dyn);
  return cudaGetLastError();
}

}  // namespace mt
