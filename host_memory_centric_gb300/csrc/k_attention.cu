// k_attention.cu -- causal grouped-query attention entry points.
//
// Tiled exact attention with an online softmax (Milakov and Gimelshein 2018;
// the FlashAttention-2 tiling of Dao 2023), so memory is O(S * hd) per head and
// sequences of any length run with the same kernels: the pages train 512K
// tokens on one GPU by bounding activation residency to one layer, which needs
// exactly this O(S) attention.  Scores live in the exp2 domain
// (s * log2(e) / sqrt(hd)); the forward keeps the natural-log LSE per row for
// the backward, which recomputes P from it.
//
// The forward and the two backward kernels run on the tcgen05 tensor cores
// (k_attention_tc.cu).  This file holds the backward's first pass,
// delta = rowsum(dO o O), and the argument checks.
#include "mt_kernels.h"

namespace mt {
namespace {

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// delta[h][t] = sum_d dO[t, h, d] * O[t, h, d].  HD / 8 lanes per (t, h),
// one 16-byte vector of each operand per lane, so a warp covers 32 * 8 / HD
// consecutive (t, h) rows with all its loads in flight at once.
template <int HD>
__global__ void __launch_bounds__(256) attn_delta_k(const bf16* __restrict__ o, const bf16* __restrict__ dout,
                                                    int64_t T, int nh, float* __restrict__ delta) {
  constexpr int LPR = HD / 8;
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t w = gid / LPR;  // (t, h) row, t-major as the tensors are laid out
  const int sub = (int)(gid % LPR);
  float s = 0.f;
  if (w < T * nh) {
    const uint4 a = reinterpret_cast<const uint4*>(o + w * HD)[sub];
    const uint4 b = reinterpret_cast<const uint4*>(dout + w * HD)[sub];
    const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 u = __bfloat1622float2(x[k]);
      const float2 v = __bfloat1622float2(y[k]);
      s += u.x * v.x + u.y * v.y;
    }
  }
#pragma unroll
  for (int off = LPR / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (sub == 0 && w < T * nh) {
    const int64_t t = w / nh;
    const int h = (int)(w % nh);
    delta[(int64_t)h * T + t] = s;
  }
}

template <int HD>
cudaError_t bwd_tc(const bf16* qkv, const bf16* o, const float* lse, const bf16* dout, int n_seq, int S, int nh,
                   int nkv, bf16* dqkv, float* delta, cudaStream_t s) {
  const int64_t T = (int64_t)n_seq * S;
  const int64_t blocks = (T * nh * (HD / 8) + 255) / 256;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  attn_delta_k<HD><<<(unsigned)blocks, 256, 0, s>>>(o, dout, T, nh, delta);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return attention_bwd_tc_core(qkv, dout, lse, delta, n_seq, S, nh, nkv, HD, dqkv, s);
}

}  // namespace

cudaError_t attention_fwd(const bf16* qkv, int n_seq, int S, int nh, int nkv, int hd, bf16* o, float* lse,
                          cudaStream_t s) {
  return attention_fwd_tc(qkv, n_seq, S, nh, nkv, hd, o, lse, s);
}

cudaError_t attention_bwd(const bf16* qkv, const bf16* o, const float* lse, const bf16* dout, int n_seq, int S,
                          int nh, int nkv, int hd, bf16* dqkv, float* delta, cudaStream_t s) {
  if (n_seq <= 0 || S <= 0) return cudaSuccess;
  if (nkv <= 0 || nh % nkv || !al16(qkv) || !al16(o) || !al16(dout) || !al16(dqkv)) return cudaErrorInvalidValue;
  if (hd == 64) return bwd_tc<64>(qkv, o, lse, dout, n_seq, S, nh, nkv, dqkv, delta, s);
  if (hd == 128) return bwd_tc<128>(qkv, o, lse, dout, n_seq, S, nh, nkv, dqkv, delta, s);
  return cudaErrorInvalidValue;
}

}  // namespace mt
