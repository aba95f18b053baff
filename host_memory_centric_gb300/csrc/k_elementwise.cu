// k_elementwise.cu -- HBM-bound kernels of the block math (sm_103a).
//
// RMSNorm forward / backward, rotate-half RoPE, SwiGLU forward / backward,
// embedding gather / dense gradient, cross-entropy with in-place dlogits, and
// small conversions.  Each kernel reads and writes its tensors once with
// 16-byte vector accesses along contiguous rows (coalesced per warp), keeps
// statistics in FP32 and reduces with warp shuffles.
#include "mt_kernels.h"

#include <type_traits>

namespace mt {
namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ void unpack8(const uint4& q, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 t = __bfloat1622float2(h[k]);
    f[2 * k] = t.x;
    f[2 * k + 1] = t.y;
  }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 q;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&q);
#pragma unroll
  for (int k = 0; k < 4; ++k) h[k] = __floats2bfloat162_rn(f[2 * k], f[2 * k + 1]);
  return q;
}

constexpr int ROW_WARPS = 8;  // rows per 256-thread block in the row kernels

// ------------------------------------------------------------------ RMSNorm
// Row kernels: one warp per row, lane l owning the 16-byte vectors l, l + 32,
// ... of the row.  NV (vectors per lane, H <= 256 NV) is a template argument
// so that every load of a row is issued before the first use and the row stays
// in registers between the statistic and the output pass; NV = 0 is the
// generic form for wider rows (loads unrolled by four, the row re-read).
// gamma is staged once per block in shared memory.
template <int NV>
__global__ void __launch_bounds__(256, 2) rmsnorm_fwd_k(const bf16* __restrict__ x, const bf16* __restrict__ g,
                                                     int64_t T, int H, float eps, bf16* __restrict__ y,
                                                     float* __restrict__ rstd) {
  extern __shared__ uint4 sg[];  // gamma, H / 8 vectors
  for (int i = threadIdx.x; i < H / 8; i += blockDim.x) sg[i] = reinterpret_cast<const uint4*>(g)[i];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * ROW_WARPS + (threadIdx.x >> 5);
  if (row >= T) return;
  const uint4* xr = reinterpret_cast<const uint4*>(x + row * H);
  uint4* yr = reinterpret_cast<uint4*>(y + row * H);
  const int nv = H / 8;
  float ss = 0.f;
  if constexpr (NV > 0) {
    uint4 xv[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) xv[j] = j * 32 + lane < nv ? xr[j * 32 + lane] : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      float f[8];
      unpack8(xv[j], f);
#pragma unroll
      for (int k = 0; k < 8; ++k) ss += f[k] * f[k];
    }
    ss = warp_sum(ss);
    const float r = rsqrtf(ss / (float)H + eps);
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int v = j * 32 + lane;
      if (v < nv) {
        float f[8], w[8];
        unpack8(xv[j], f);
        unpack8(sg[v], w);
#pragma unroll
        for (int k = 0; k < 8; ++k) f[k] = f[k] * r * w[k];
        yr[v] = pack8(f);
      }
    }
    if (lane == 0) rstd[row] = r;
  } else {
#pragma unroll 4
    for (int v = lane; v < nv; v += 32) {
      float f[8];
      unpack8(xr[v], f);
#pragma unroll
      for (int k = 0; k < 8; ++k) ss += f[k] * f[k];
    }
    ss = warp_sum(ss);
    const float r = rsqrtf(ss / (float)H + eps);
#pragma unroll 4
    for (int v = lane; v < nv; v += 32) {
      float f[8], w[8];
      unpack8(xr[v], f);
      unpack8(sg[v], w);
#pragma unroll
      for (int k = 0; k < 8; ++k) f[k] = f[k] * r * w[k];
      yr[v] = pack8(f);
    }
    if (lane == 0) rstd[row] = r;
  }
}

// RMSNorm backward.  Each block owns a contiguous run of rows and writes the
// dgamma partial sum of its rows to partial[blockIdx.x][H]; a second kernel
// adds the blocks' partials in a fixed order.  dx is computed one warp per row
// (the row's dot product needs the whole row).  No atomics: every sum runs in
// an order fixed by the row and block indices, so results are reproducible.
//
// Rows of up to 2048 (NV = H / 256 vectors per lane, a template argument):
// dy and x stay in registers between the dot product and the output, and each
// warp adds its own rows' dgamma contribution straight from those registers
// into its own FP32 accumulator row in shared memory ([8 warps][H]); the
// block then adds the eight warp rows in warp order.  Nothing is read twice
// and the warps never wait for one another inside the row loop.
template <int NV>
__global__ void __launch_bounds__(256, 2) rmsnorm_bwd_warp_k(const bf16* __restrict__ dy,
                                                             const bf16* __restrict__ x,
                                                             const bf16* __restrict__ g,
                                                             const float* __restrict__ rstd,
                                                             const bf16* __restrict__ dres, int64_t T, int H,
                                                             int64_t rows_per_block, bf16* __restrict__ dx,
                                                             float* __restrict__ partial) {
  extern __shared__ uint4 sg[];  // gamma (H / 8 vectors), then [ROW_WARPS][H] FP32 accumulators
  float* acc = reinterpret_cast<float*>(sg + H / 8);
  const int nv = H / 8;
  for (int i = threadIdx.x; i < nv; i += blockDim.x) sg[i] = reinterpret_cast<const uint4*>(g)[i];
  for (int i = threadIdx.x; i < ROW_WARPS * nv * 2; i += blockDim.x)
    reinterpret_cast<float4*>(acc)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* wacc = acc + (int64_t)warp * H;
  const int64_t r0 = (int64_t)blockIdx.x * rows_per_block;
  const int64_t r1 = min(T, r0 + rows_per_block);
  for (int64_t row = r0 + warp; row < r1; row += ROW_WARPS) {
    const uint4* dyr = reinterpret_cast<const uint4*>(dy + row * H);
    const uint4* xr = reinterpret_cast<const uint4*>(x + row * H);
    const uint4* dr = dres ? reinterpret_cast<const uint4*>(dres + row * H) : nullptr;
    uint4* dxr = reinterpret_cast<uint4*>(dx + row * H);
    const float r = rstd[row];
    uint4 av[NV], bv[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int v = j * 32 + lane;
      av[j] = v < nv ? dyr[v] : make_uint4(0, 0, 0, 0);
      bv[j] = v < nv ? xr[v] : make_uint4(0, 0, 0, 0);
    }
    float dot = 0.f;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int v = j * 32 + lane;
      if (v < nv) {
        float a[8], b[8], w[8];
        unpack8(av[j], a);
        unpack8(bv[j], b);
        unpack8(sg[v], w);
#pragma unroll
        for (int k = 0; k < 8; ++k) dot += a[k] * w[k] * b[k];
      }
    }
    dot = warp_sum(dot);
    const float c3 = r * r * r / (float)H * dot;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int v = j * 32 + lane;
      if (v < nv) {
        float a[8], b[8], w[8], o[8];
        unpack8(av[j], a);
        unpack8(bv[j], b);
        unpack8(sg[v], w);
        if (dr) {
          unpack8(dr[v], o);
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) o[k] = 0.f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) o[k] += r * w[k] * a[k] - c3 * b[k];
        dxr[v] = pack8(o);
        float4* ap = reinterpret_cast<float4*>(wacc + v * 8);
        float4 p0 = ap[0], p1 = ap[1];
        p0.x += a[0] * b[0] * r;
        p0.y += a[1] * b[1] * r;
        p0.z += a[2] * b[2] * r;
        p0.w += a[3] * b[3] * r;
        p1.x += a[4] * b[4] * r;
        p1.y += a[5] * b[5] * r;
        p1.z += a[6] * b[6] * r;
        p1.w += a[7] * b[7] * r;
        ap[0] = p0;
        ap[1] = p1;
      }
    }
  }
  __syncthreads();
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    float4 s0 = make_float4(0.f, 0.f, 0.f, 0.f), s1 = s0;
#pragma unroll
    for (int w = 0; w < ROW_WARPS; ++w) {
      const float4* ap = reinterpret_cast<const float4*>(acc + (int64_t)w * H + v * 8);
      const float4 p0 = ap[0], p1 = ap[1];
      s0.x += p0.x;
      s0.y += p0.y;
      s0.z += p0.z;
      s0.w += p0.w;
      s1.x += p1.x;
      s1.y += p1.y;
      s1.z += p1.z;
      s1.w += p1.w;
    }
    float4* p = reinterpret_cast<float4*>(partial + (int64_t)blockIdx.x * H + v * 8);
    p[0] = s0;
    p[1] = s1;
  }
}

// Wider rows: the rows go in chunks of eight.  dx one warp per row (the row
// read twice, loads unrolled by four), then the chunk's dgamma contribution
// column by column: thread t owns the 16-byte column vectors t, t + 256, ...
// and adds the chunk's rows in row order into its own FP32 accumulators in
// shared memory (the rows were just read by the block, so they come from L1).
__global__ void __launch_bounds__(256, 2) rmsnorm_bwd_k(const bf16* __restrict__ dy, const bf16* __restrict__ x,
                                                        const bf16* __restrict__ g, const float* __restrict__ rstd,
                                                        const bf16* __restrict__ dres, int64_t T, int H,
                                                        int64_t rows_per_block, bf16* __restrict__ dx,
                                                        float* __restrict__ partial) {
  extern __shared__ uint4 sg[];  // gamma (H / 8 vectors), then the FP32 accumulators (H floats)
  float* acc = reinterpret_cast<float*>(sg + H / 8);
  const int nv = H / 8;
  for (int i = threadIdx.x; i < nv; i += blockDim.x) {
    sg[i] = reinterpret_cast<const uint4*>(g)[i];
    reinterpret_cast<float4*>(acc)[2 * i] = make_float4(0.f, 0.f, 0.f, 0.f);
    reinterpret_cast<float4*>(acc)[2 * i + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t r0 = (int64_t)blockIdx.x * rows_per_block;
  const int64_t r1 = min(T, r0 + rows_per_block);
  for (int64_t c0 = r0; c0 < r1; c0 += ROW_WARPS) {  // block-uniform trip count
    const int64_t row = c0 + warp;
    if (row < r1) {
      const uint4* dyr = reinterpret_cast<const uint4*>(dy + row * H);
      const uint4* xr = reinterpret_cast<const uint4*>(x + row * H);
      const uint4* dr = dres ? reinterpret_cast<const uint4*>(dres + row * H) : nullptr;
      uint4* dxr = reinterpret_cast<uint4*>(dx + row * H);
      const float r = rstd[row];
      float dot = 0.f;
#pragma unroll 4
      for (int v = lane; v < nv; v += 32) {
        float a[8], b[8], w[8];
        unpack8(dyr[v], a);
        unpack8(xr[v], b);
        unpack8(sg[v], w);
#pragma unroll
        for (int k = 0; k < 8; ++k) dot += a[k] * w[k] * b[k];
      }
      dot = warp_sum(dot);
      const float c3 = r * r * r / (float)H * dot;
#pragma unroll 4
      for (int v = lane; v < nv; v += 32) {
        float a[8], b[8], w[8], o[8];
        unpack8(dyr[v], a);
        unpack8(xr[v], b);
        unpack8(sg[v], w);
        if (dr) {
          unpack8(dr[v], o);
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) o[k] = 0.f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) o[k] += r * w[k] * a[k] - c3 * b[k];
        dxr[v] = pack8(o);
      }
    }
    __syncthreads();  // the chunk's rows are in L1 before the column pass reads them
    const int n = (int)min((int64_t)ROW_WARPS, r1 - c0);
    float rr[ROW_WARPS];
#pragma unroll
    for (int u = 0; u < ROW_WARPS; ++u) rr[u] = u < n ? rstd[c0 + u] : 0.f;
    for (int v = threadIdx.x; v < nv; v += blockDim.x) {
      uint4 av[ROW_WARPS], bv[ROW_WARPS];
#pragma unroll
      for (int u = 0; u < ROW_WARPS; ++u) {
        av[u] = u < n ? reinterpret_cast<const uint4*>(dy + (c0 + u) * H)[v] : make_uint4(0, 0, 0, 0);
        bv[u] = u < n ? reinterpret_cast<const uint4*>(x + (c0 + u) * H)[v] : make_uint4(0, 0, 0, 0);
      }
      float4* ap = reinterpret_cast<float4*>(acc + v * 8);
      const float4 p0 = ap[0], p1 = ap[1];
      float s8[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
      for (int u = 0; u < ROW_WARPS; ++u) {
        if (u < n) {
          float a[8], b[8];
          unpack8(av[u], a);
          unpack8(bv[u], b);
#pragma unroll
          for (int k = 0; k < 8; ++k) s8[k] += a[k] * b[k] * rr[u];
        }
      }
      ap[0] = make_float4(s8[0], s8[1], s8[2], s8[3]);
      ap[1] = make_float4(s8[4], s8[5], s8[6], s8[7]);
    }
  }
  // each thread reads back only the accumulators it wrote
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    const float4* ap = reinterpret_cast<const float4*>(acc + v * 8);
    float4* p = reinterpret_cast<float4*>(partial + (int64_t)blockIdx.x * H + v * 8);
    p[0] = ap[0];
    p[1] = ap[1];
  }
}

// dgamma[c] = sum over b of partial[b][c], b ascending in eight interleaved
// slices (warp w sums b = w, w + 8, ...; four loads in flight), the slices
// then added in order: a fixed order, so the result is reproducible.  One
// block per 32 columns; lane = column.
__global__ void __launch_bounds__(256) rmsnorm_bwd_stage2_k(const float* __restrict__ partial, int nblk, int H,
                                                            bf16* __restrict__ dg) {
  __shared__ float red[ROW_WARPS][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = blockIdx.x * 32 + lane;
  float s = 0.f;
  if (c < H) {
    int b = warp;
    for (; b + 3 * ROW_WARPS < nblk; b += 4 * ROW_WARPS) {
      float t[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) t[u] = partial[(int64_t)(b + u * ROW_WARPS) * H + c];
#pragma unroll
      for (int u = 0; u < 4; ++u) s += t[u];
    }
    for (; b < nblk; b += ROW_WARPS) s += partial[(int64_t)b * H + c];
  }
  red[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && c < H) {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < ROW_WARPS; ++w) tot += red[w][lane];
    dg[c] = __float2bfloat16_rn(tot);
  }
}

// ------------------------------------------------------------------ debug guards
// One block per guard; 256 threads compare the 4096 bytes as 16-byte words.
__global__ void guard_check_k(const uint8_t* __restrict__ base, const int64_t* __restrict__ offs, int n,
                              int* __restrict__ bad) {
  const int g = blockIdx.x;
  if (g >= n) return;
  const uint4 w = reinterpret_cast<const uint4*>(base + offs[g])[threadIdx.x];
  const uint32_t k = 0xA5A5A5A5u;
  if (w.x != k || w.y != k || w.z != k || w.w != k) atomicMin(bad, g);
}

// ------------------------------------------------------------------ RoPE
// One thread rotates 8 consecutive frequency pairs of one head of one row.
__global__ void rope_k(bf16* __restrict__ x, int64_t T, int64_t ld, int n_heads, int hd, int S,
                       const float* __restrict__ cs, int inverse) {
  const int half = hd >> 1, per_head = half >> 3;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t per_row = (int64_t)n_heads * per_head;
  if (idx >= T * per_row) return;
  const int64_t row = idx / per_row;
  const int rem = (int)(idx % per_row);
  const int h = rem / per_head, i0 = (rem % per_head) * 8;
  const int pos = (int)(row % S);
  bf16* p = x + row * ld + (int64_t)h * hd;
  float a[8], b[8];
  unpack8(*reinterpret_cast<const uint4*>(p + i0), a);
  unpack8(*reinterpret_cast<const uint4*>(p + half + i0), b);
  const float4* c4 = reinterpret_cast<const float4*>(cs + ((int64_t)pos * half + i0) * 2);
  float oa[8], ob[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float4 v = c4[k];  // cos_i, sin_i, cos_{i+1}, sin_{i+1}
    const float c0 = v.x, s0 = inverse ? -v.y : v.y, c1 = v.z, s1 = inverse ? -v.w : v.w;
    oa[2 * k] = a[2 * k] * c0 - b[2 * k] * s0;
    ob[2 * k] = b[2 * k] * c0 + a[2 * k] * s0;
    oa[2 * k + 1] = a[2 * k + 1] * c1 - b[2 * k + 1] * s1;
    ob[2 * k + 1] = b[2 * k + 1] * c1 + a[2 * k + 1] * s1;
  }
  *reinterpret_cast<uint4*>(p + i0) = pack8(oa);
  *reinterpret_cast<uint4*>(p + half + i0) = pack8(ob);
}

// ------------------------------------------------------------------ SwiGLU
__device__ __forceinline__ float sigm(float z) { return 1.f / (1.f + expf(-z)); }

__global__ void swiglu_fwd_k(const bf16* __restrict__ gu, int64_t T, int F, bf16* __restrict__ h) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int per_row = F >> 3;
  if (idx >= T * per_row) return;
  const int64_t row = idx / per_row;
  const int c = (int)(idx % per_row) * 8;
  float g[8], u[8];
  unpack8(*reinterpret_cast<const uint4*>(gu + row * 2 * F + c), g);
  unpack8(*reinterpret_cast<const uint4*>(gu + row * 2 * F + F + c), u);
#pragma unroll
  for (int k = 0; k < 8; ++k) g[k] = g[k] * sigm(g[k]) * u[k];
  *reinterpret_cast<uint4*>(h + row * F + c) = pack8(g);
}

__global__ void swiglu_bwd_k(const bf16* __restrict__ gu, const bf16* __restrict__ dh, int64_t T, int F,
                             bf16* __restrict__ dgu) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int per_row = F >> 3;
  if (idx >= T * per_row) return;
  const int64_t row = idx / per_row;
  const int c = (int)(idx % per_row) * 8;
  float g[8], u[8], d[8], dg[8], du[8];
  unpack8(*reinterpret_cast<const uint4*>(gu + row * 2 * F + c), g);
  unpack8(*reinterpret_cast<const uint4*>(gu + row * 2 * F + F + c), u);
  unpack8(*reinterpret_cast<const uint4*>(dh + row * F + c), d);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float s = sigm(g[k]);
    dg[k] = d[k] * u[k] * s * (1.f + g[k] * (1.f - s));
    du[k] = d[k] * g[k] * s;
  }
  *reinterpret_cast<uint4*>(dgu + row * 2 * F + c) = pack8(dg);
  *reinterpret_cast<uint4*>(dgu + row * 2 * F + F + c) = pack8(du);
}

// ------------------------------------------------------------------ embedding
__global__ void embed_fwd_k(const int32_t* __restrict__ tok, const bf16* __restrict__ E, int64_t T, int H,
                            bf16* __restrict__ X) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int per_row = H >> 3;
  if (idx >= T * per_row) return;
  const int64_t row = idx / per_row;
  const int c = (int)(idx % per_row) * 8;
  *reinterpret_cast<uint4*>(X + row * H + c) =
      *reinterpret_cast<const uint4*>(E + (int64_t)tok[row] * H + c);
}

// One block per vocabulary row; rows no token selects are written as zeros.
__global__ void __launch_bounds__(128) embed_bwd_k(const int32_t* __restrict__ row_start,
                                                   const int32_t* __restrict__ rows, const bf16* __restrict__ dX,
                                                   int H, bf16* __restrict__ dE) {
  const int64_t v = blockIdx.x;
  const int b = row_start[v], e = row_start[v + 1];
  for (int c = threadIdx.x * 8; c < H; c += blockDim.x * 8) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int i = b; i < e; ++i) {
      float f[8];
      unpack8(*reinterpret_cast<const uint4*>(dX + (int64_t)rows[i] * H + c), f);
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] += f[k];
    }
    *reinterpret_cast<uint4*>(dE + v * H + c) = pack8(acc);
  }
}

// ------------------------------------------------------------------ cross-entropy
constexpr int CE_THREADS = 512;

__global__ void __launch_bounds__(CE_THREADS) cross_entropy_k(bf16* __restrict__ logits,
                                                              const int32_t* __restrict__ target, int V,
                                                              float inv_norm, float* __restrict__ row_loss) {
  __shared__ float sm[CE_THREADS / 32], ss[CE_THREADS / 32];
  __shared__ float zt_s, lse_s;
  const int64_t r = blockIdx.x;
  bf16* z = logits + r * (int64_t)V;
  const int tgt = target[r];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tgt < 0) {
    const uint4 zero = make_uint4(0, 0, 0, 0);
    if ((V & 7) == 0)
      for (int c = tid * 8; c < V; c += CE_THREADS * 8) *reinterpret_cast<uint4*>(z + c) = zero;
    else
      for (int c = tid; c < V; c += CE_THREADS) z[c] = __float2bfloat16_rn(0.f);
    if (tid == 0) row_loss[r] = 0.f;
    return;
  }
  if (tid == 0) zt_s = __bfloat162float(z[tgt]);
  // pass 1: per-thread running max and sum of exp, merged across the block;
  // four 16-byte loads in flight per thread
  float m = -INFINITY, s = 0.f;
  auto add = [&](float v) {
    if (v > m) {
      s = s * expf(m - v) + 1.f;
      m = v;
    } else {
      s += expf(v - m);
    }
  };
  if ((V & 7) == 0) {
#pragma unroll 4
    for (int c = tid * 8; c < V; c += CE_THREADS * 8) {
      float f[8];
      unpack8(*reinterpret_cast<const uint4*>(z + c), f);
#pragma unroll
      for (int k = 0; k < 8; ++k) add(f[k]);
    }
  } else {
    for (int c = tid; c < V; c += CE_THREADS) add(__bfloat162float(z[c]));
  }
  float wm = warp_max(m);
  float wsum = (m == -INFINITY) ? 0.f : s * expf(m - wm);
  wsum = warp_sum(wsum);
  if (lane == 0) {
    sm[warp] = wm;
    ss[warp] = wsum;
  }
  __syncthreads();
  if (warp == 0) {
    float a = lane < CE_THREADS / 32 ? sm[lane] : -INFINITY;
    float b = lane < CE_THREADS / 32 ? ss[lane] : 0.f;
    const float M = warp_max(a);
    b = (a == -INFINITY) ? 0.f : b * expf(a - M);
    b = warp_sum(b);
    if (lane == 0) {
      lse_s = M + logf(b);
      row_loss[r] = lse_s - zt_s;
    }
  }
  __syncthreads();
  const float lse = lse_s;
  // pass 2: dlogits = (softmax - onehot) * inv_norm (the row comes from L2)
  if ((V & 7) == 0) {
#pragma unroll 4
    for (int c = tid * 8; c < V; c += CE_THREADS * 8) {
      float f[8];
      unpack8(*reinterpret_cast<const uint4*>(z + c), f);
#pragma unroll
      for (int k = 0; k < 8; ++k) f[k] = (expf(f[k] - lse) - (c + k == tgt ? 1.f : 0.f)) * inv_norm;
      *reinterpret_cast<uint4*>(z + c) = pack8(f);
    }
  } else {
    for (int c = tid; c < V; c += CE_THREADS) {
      const float v = __bfloat162float(z[c]);
      z[c] = __float2bfloat16_rn((expf(v - lse) - (c == tgt ? 1.f : 0.f)) * inv_norm);
    }
  }
}

__global__ void reduce_sum_k(const float* __restrict__ x, int64_t n, float scale, float* out) {
  __shared__ double sh[32];
  double s = 0.0;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) s += (double)x[i];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += sh[w];
    out[0] = (float)(t * (double)scale);
  }
}

__global__ void f32_to_bf16_k(const float* __restrict__ x, int64_t ldx, int64_t rows, int64_t cols,
                              bf16* __restrict__ y, int64_t ldy, float scale) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows * cols) return;
  const int64_t r = idx / cols, c = idx % cols;
  y[r * ldy + c] = __float2bfloat16_rn(x[r * ldx + c] * scale);
}

__global__ void add_bf16_k(const bf16* __restrict__ a, const bf16* __restrict__ b, int64_t n8, bf16* __restrict__ y) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  float fa[8], fb[8];
  unpack8(reinterpret_cast<const uint4*>(a)[i], fa);
  unpack8(reinterpret_cast<const uint4*>(b)[i], fb);
#pragma unroll
  for (int k = 0; k < 8; ++k) fa[k] += fb[k];
  reinterpret_cast<uint4*>(y)[i] = pack8(fa);
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
inline unsigned nblocks(int64_t n, int t) { return (unsigned)((n + t - 1) / t); }

}  // namespace

// ------------------------------------------------------------------ launchers
// Vectors per lane the row kernels keep in registers for a row of H
// elements, at most MaxNV (so that two 256-thread blocks fit on an SM); 0
// selects the generic (re-reading) form.
template <int MaxNV, typename F>
cudaError_t with_nv(int H, F&& f) {
  const int per_lane = (H / 8 + 31) / 32;
  if (per_lane <= 1) return f(std::integral_constant<int, 1>());
  if (per_lane <= 2) return f(std::integral_constant<int, 2>());
  if (per_lane <= 4) return f(std::integral_constant<int, 4>());
  if constexpr (MaxNV >= 8)
    if (per_lane <= 8) return f(std::integral_constant<int, 8>());
  if constexpr (MaxNV >= 12)
    if (per_lane <= 12) return f(std::integral_constant<int, 12>());
  if constexpr (MaxNV >= 16)
    if (per_lane <= 16) return f(std::integral_constant<int, 16>());
  return f(std::integral_constant<int, 0>());
}

cudaError_t rmsnorm_fwd(const bf16* x, const bf16* gamma, int64_t T, int H, float eps, bf16* y, float* rstd,
                        cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (H % 8 || H > 24576 || !al16(x) || !al16(gamma) || !al16(y)) return cudaErrorInvalidValue;
  return with_nv<16>(H, [&](auto nv) {
    rmsnorm_fwd_k<decltype(nv)::value><<<nblocks(T, ROW_WARPS), 256, (size_t)H * 2, s>>>(x, gamma, T, H, eps, y, rstd);
    return cudaGetLastError();
  });
}

int rmsnorm_bwd_blocks(int64_t T) {
  const int64_t want = (T + ROW_WARPS * 4 - 1) / (ROW_WARPS * 4);  // >= 32 rows per block
  return (int)(want < 304 ? (want < 1 ? 1 : want) : 304);
}
int64_t rmsnorm_bwd_partial_floats(int64_t T, int H) { return (int64_t)rmsnorm_bwd_blocks(T) * H; }

cudaError_t rmsnorm_bwd_stage2(const float* partial, int nblk, int H, bf16* dgamma, cudaStream_t s) {
  rmsnorm_bwd_stage2_k<<<nblocks(H, 32), 256, 0, s>>>(partial, nblk, H, dgamma);
  return cudaGetLastError();
}

cudaError_t rmsnorm_bwd(const bf16* dy, const bf16* x, const bf16* gamma, const float* rstd, const bf16* dres,
                        int64_t T, int H, bf16* dx, bf16* dgamma, float* partial, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (H % 8 || H > 12288 || !al16(dy) || !al16(x) || !al16(gamma) || !al16(dx) || (dres && !al16(dres)))
    return cudaErrorInvalidValue;
  const int nblk = rmsnorm_bwd_blocks(T);
  const int64_t per = (T + nblk - 1) / nblk;
  if (reinterpret_cast<uintptr_t>(partial) & 15) return cudaErrorInvalidValue;
  cudaError_t e;
  if (H <= 2048) {
    // gamma + eight FP32 accumulator rows: at most 69,632 bytes
    const size_t smem = (size_t)H * 2 + (size_t)ROW_WARPS * H * 4;
    e = with_nv<8>(H, [&](auto nv) {
      constexpr int K = decltype(nv)::value;
      if constexpr (K == 0) {
        return cudaErrorInvalidValue;  // not reached: H <= 2048 has at most 8 vectors per lane
      } else {
        // the opt-in is per device, so it is set on every call (a host-side attribute write)
        const cudaError_t attr = cudaFuncSetAttribute(rmsnorm_bwd_warp_k<K>,
                                                      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (attr != cudaSuccess) return attr;
        rmsnorm_bwd_warp_k<K><<<nblk, 256, smem, s>>>(dy, x, gamma, rstd, dres, T, H, per, dx, partial);
        return cudaGetLastError();
      }
    });
  } else {
    const size_t smem = (size_t)H * 6;  // gamma + one FP32 accumulator row
    if (smem > 48 * 1024) {
      e = cudaFuncSetAttribute(rmsnorm_bwd_k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    rmsnorm_bwd_k<<<nblk, 256, smem, s>>>(dy, x, gamma, rstd, dres, T, H, per, dx, partial);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;
  return rmsnorm_bwd_stage2(partial, nblk, H, dgamma, s);
}

cudaError_t guard_check(const uint8_t* base, const int64_t* offs, int n, int* bad, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  guard_check_k<<<n, 256, 0, s>>>(base, offs, n, bad);
  return cudaGetLastError();
}

cudaError_t rope(bf16* x, int64_t T, int64_t ld, int n_heads, int hd, int S, const float* cs, int inverse,
                 cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (hd % 16 || ld % 8 || !al16(x) || !al16(cs)) return cudaErrorInvalidValue;
  const int64_t n = T * n_heads * (hd / 16);
  rope_k<<<nblocks(n, 256), 256, 0, s>>>(x, T, ld, n_heads, hd, S, cs, inverse);
  return cudaGetLastError();
}

cudaError_t swiglu_fwd(const bf16* gu, int64_t T, int F, bf16* h, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (F % 8 || !al16(gu) || !al16(h)) return cudaErrorInvalidValue;
  swiglu_fwd_k<<<nblocks(T * (F / 8), 256), 256, 0, s>>>(gu, T, F, h);
  return cudaGetLastError();
}

cudaError_t swiglu_bwd(const bf16* gu, const bf16* dh, int64_t T, int F, bf16* dgu, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (F % 8 || !al16(gu) || !al16(dh) || !al16(dgu)) return cudaErrorInvalidValue;
  swiglu_bwd_k<<<nblocks(T * (F / 8), 256), 256, 0, s>>>(gu, dh, T, F, dgu);
  return cudaGetLastError();
}

cudaError_t embed_fwd(const int32_t* tok, const bf16* E, int64_t T, int H, int V, bf16* X, cudaStream_t s) {
  (void)V;
  if (T <= 0) return cudaSuccess;
  if (H % 8 || !al16(E) || !al16(X)) return cudaErrorInvalidValue;
  embed_fwd_k<<<nblocks(T * (H / 8), 256), 256, 0, s>>>(tok, E, T, H, X);
  return cudaGetLastError();
}

cudaError_t embed_bwd(const int32_t* row_start, const int32_t* rows, const bf16* dX, int V, int H, bf16* dE,
                      cudaStream_t s) {
  if (V <= 0) return cudaSuccess;
  if (H % 8 || !al16(dX) || !al16(dE)) return cudaErrorInvalidValue;
  embed_bwd_k<<<V, 128, 0, s>>>(row_start, rows, dX, H, dE);
  return cudaGetLastError();
}

cudaError_t cross_entropy(bf16* logits, const int32_t* target, int64_t rows, int V, float inv_norm,
                          float* row_loss, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (((V & 7) == 0) && !al16(logits)) return cudaErrorInvalidValue;
  if (rows > 0x7fffffff) return cudaErrorInvalidValue;
  cross_entropy_k<<<(unsigned)rows, CE_THREADS, 0, s>>>(logits, target, V, inv_norm, row_loss);
  return cudaGetLastError();
}

cudaError_t reduce_sum(const float* x, int64_t n, float scale, float* out, cudaStream_t s) {
  reduce_sum_k<<<1, 1024, 0, s>>>(x, n, scale, out);
  return cudaGetLastError();
}

cudaError_t f32_to_bf16_2d(const float* x, int64_t ldx, int64_t rows, int64_t cols, bf16* y, int64_t ldy,
                           float scale, cudaStream_t s) {
  if (rows * cols <= 0) return cudaSuccess;
  f32_to_bf16_k<<<nblocks(rows * cols, 256), 256, 0, s>>>(x, ldx, rows, cols, y, ldy, scale);
  return cudaGetLastError();
}

cudaError_t add_bf16(const bf16* a, const bf16* b, int64_t n, bf16* y, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if (n % 8 || !al16(a) || !al16(b) || !al16(y)) return cudaErrorInvalidValue;
  add_bf16_k<<<nblocks(n / 8, 256), 256, 0, s>>>(a, b, n / 8, y);
  return cudaGetLastError();
}

}  // namespace mt
