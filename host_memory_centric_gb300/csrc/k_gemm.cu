// k_gemm.cu -- BF16 GEMM on the 5th-generation tensor cores (sm_103a).
//
// Serves the projections of every block: Y = X W^T (forward and recompute),
// dX = dY W (dgrad) and dW = dY^T X (wgrad, whose epilogue writes BF16 straight
// into the gradient region of the streamed buffer, i.e. the flat layout the
// gradient export copies out in one burst).
//
// Design (one CTA per SM, persistent over output tiles of 128 x 256):
//   warp 0      TMA producer: 128B-swizzled tiles of A and B into a 4-stage
//               shared-memory ring (mbarrier full/empty pairs);
//   warp 1      allocates 512 TMEM columns (two 128x256 FP32 accumulators)
//               and, from one thread, issues tcgen05.mma (M=128, N=256, K=16)
//               and tcgen05.commit;
//   warps 2..5  epilogue: tcgen05.ld 32x32b rows out of TMEM, optional FP32
//               accumulate / residual add, BF16 round-to-nearest-even, store;
//               the second accumulator lets the epilogue of tile i overlap the
//               main loop of tile i+1.
// Operands may be K-major or MN-major (the transpose bits of the instruction
// descriptor), so dgrad and wgrad read activations and weights in place.
// Every mbarrier wait is bounded; on expiry the kernel records an error code,
// stops issuing, drains its own copies and frees its TMEM.
//
// Dense GEMMs default to the CTA-pair form (gemm_pair_kernel): a cluster of
// two CTAs on neighbouring SMs owns a 256 x 256 output tile.  Each CTA loads
// its 128 rows of A and its 128 rows of B (the B half the peer does not hold)
// into a 6-stage ring, both CTAs' copies completing on the even CTA's full
// barrier; the even CTA's one thread issues tcgen05.mma.cta_group::2 (M=256,
// N=256), which reads both CTAs' shared memory and writes each CTA's 128
// accumulator rows into its own TMEM, and its commits arrive on both CTAs'
// barriers.  Per SM this halves the B bytes a K block moves (32 KB of operands
// for 128 x 256 x 64 instead of 48 KB), which is what limited the one-CTA
// form's tensor-pipe activity.  The K blocks are accumulated in the same
// order either way, so the two forms agree bit for bit.
//
// Tile order of the pairs: output tiles are rastered in bands of `group_m`
// 256-row tiles (chosen per launch from K, so that the operand slices of the
// tiles in flight fit in about half the L2), and each pair, after its first
// tile, draws the next from a per-launch counter.  The tiles in flight thus
// stay a window of consecutive tiles however unevenly the SMs progress, and
// tiles that share an operand slice read it from L2 rather than DRAM.  The
// even CTA's producer thread draws the tile (one tile ahead) and passes it
// through a 4-entry ring in shared memory to its MMA thread, to the odd
// CTA's producer and to both CTAs' epilogue warps.
//
// Launches whose every GEMM has K >= 8192, N >= 512 and no residual use
// 256 x 512 pair tiles: per K step two M = 256, N = 256 MMAs into one 512-column
// accumulator, each CTA loading two 128-row blocks of B per stage (4 stages
// of 48 KB).  The epilogue of a tile then cannot overlap the next tile's
// MMAs, which at these K costs a few per cent, while each tile reads its rows
// of A once for 512 output columns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "mt_kernels.h"

namespace mt {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4, UMMA_K = 16;
constexpr int A_BYTES = BM * BK * 2;           // 16 KB
constexpr int B_BYTES = BN * BK * 2;           // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int CHUNK_BYTES = 64 * BK * 2;       // one 64-wide MN chunk of an MN-major tile
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr long long kWaitCycles = 4000000000LL;  // about 2 s at 2 GHz

__device__ int g_kernel_error = 0;

struct Epi {
  bf16* D; int64_t ldd;
  const bf16* R; int64_t ldr;
  float* Dacc; int64_t ldacc; int acc_mode;
  int M, N, K;
  int tiles_m, tiles_n, group_m;
  int a_mn, b_mn;
};

constexpr int MAX_EXPERT_GROUPS = 128;

// Up to two independent GEMMs ("groups") share one persistent launch: their
// output tiles form one list, so the tail of one fills SMs the other leaves
// idle.  Two expert-grouped forms serve a routed mixture-of-experts layer
// (rows of A sorted by expert, each expert's rows padded to whole 128-row
// tiles):
//   mode 1: B is a 3-D tensor [expert][N][K] (or [expert][K][N]) and M-tile
//           tm multiplies expert tile_expert[tm] (< 0: no rows, skipped);
//   mode 2: ngrp products D_g = A_g^T B_g over row ranges of A and B (both
//           MN-major): group g covers rows [grp_k0[g], grp_k0[g] + 64 grp_nk[g])
//           and writes D + grp_e[g] * d_estride (the weight gradient of expert
//           grp_e[g]).
struct Params {
  CUtensorMap ta[2], tb[2];
  Epi e[2];
  int ngroups;
  int tile_start[3];  // tiles of group g are [tile_start[g], tile_start[g+1])
  int stall;          // test hook: the producer issues nothing, so the consumers' bounded waits run out
  const int* tile_expert;
  int* tile_ctr;      // CTA pairs: the launch's tile-ticket counter (zero on entry, reset by the last draw)
  int64_t d_estride;
  int ngrp;
  int grp_e[MAX_EXPERT_GROUPS], grp_k0[MAX_EXPERT_GROUPS], grp_nk[MAX_EXPERT_GROUPS];
};

__device__ __forceinline__ uint32_t su32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase with the given parity.  False on timeout or when
// another role has aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
  if (mbar_test(b, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_test(b, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitCycles) return false;
  }
}
__device__ __forceinline__ void tma_load(const CUtensorMap* map, uint64_t* bar, void* dst, int x,
                                         int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(su32(dst)),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(su32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load3(const CUtensorMap* map, uint64_t* bar, void* dst, int x, int y,
                                          int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(su32(dst)),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(su32(bar))
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accum));
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
      : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (all >> 4), fixed version bit 46, 128B swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ULL << 46) | (2ULL << 61);
}
// Instruction descriptor, kind::f16: D fp32, A and B bf16, transpose bits for
// MN-major operands, N >> 3, M >> 4.
__host__ __device__ constexpr uint32_t idesc(bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}


__device__ __forceinline__ void tile_mn(int tile, const Epi& e, int& tm, int& tn) {
  const int per_group = e.group_m * e.tiles_n;
  const int first = (tile / per_group) * e.group_m;
  const int gsize = min(e.tiles_m - first, e.group_m);
  const int in = tile % per_group;
  tm = first + in % gsize;
  tn = in / gsize;
}

__device__ __forceinline__ void fail(volatile int* abort_flag, int code) {
  *abort_flag = 1;
  atomicCAS(&g_kernel_error, 0, code);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Epilogue of 32 consecutive columns of one output row.
__device__ __forceinline__ void epi_store(const Epi& e, int row, int col, const uint32_t (&r)[32]) {
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
  const int nv = min(32, e.N - col);
  if (nv == 32) {
    if (e.acc_mode) {
      float4* p = reinterpret_cast<float4*>(e.Dacc + (int64_t)row * e.ldacc + col);
      if (e.acc_mode == 2) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 o = p[i];
          v[4 * i] += o.x; v[4 * i + 1] += o.y; v[4 * i + 2] += o.z; v[4 * i + 3] += o.w;
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) p[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
    if (e.R) {
      const uint4* p = reinterpret_cast<const uint4*>(e.R + (int64_t)row * e.ldr + col);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint4 q = p[i];
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = __bfloat1622float2(h[k]);
          v[8 * i + 2 * k] += f.x;
          v[8 * i + 2 * k + 1] += f.y;
        }
      }
    }
    if (e.D) {
      uint4* p = reinterpret_cast<uint4*>(e.D + (int64_t)row * e.ldd + col);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        p[i] = make_uint4(pack_bf16(v[8 * i], v[8 * i + 1]), pack_bf16(v[8 * i + 2], v[8 * i + 3]),
                          pack_bf16(v[8 * i + 4], v[8 * i + 5]), pack_bf16(v[8 * i + 6], v[8 * i + 7]));
    }
  } else {
    for (int i = 0; i < nv; ++i) {
      float x = v[i];
      if (e.acc_mode) {
        float* p = e.Dacc + (int64_t)row * e.ldacc + col + i;
        if (e.acc_mode == 2) x += *p;
        *p = x;
      }
      if (e.R) x += __bfloat162float(e.R[(int64_t)row * e.ldr + col + i]);
      if (e.D) e.D[(int64_t)row * e.ldd + col + i] = __float2bfloat16_rn(x);
    }
  }
}

// Producer side of one output tile: its K-blocks into the shared-memory ring.
// z >= 0: B is a 3-D map and z its expert coordinate; koff is added to every
// K coordinate (the first row of a K-group).
template <bool A_MN, bool B_MN>
__device__ __forceinline__ bool produce_tile(const CUtensorMap* tmA, const CUtensorMap* tmB, int tm, int tn, int nk,
                                             uint8_t* sA, uint8_t* sB, uint64_t* full, uint64_t* empty, int& stage,
                                             uint32_t& phase, volatile int* abort_flag, uint32_t& inflight_mask,
                                             uint32_t& inflight_parity, int z = -1, int koff = 0) {
  for (int kb = 0; kb < nk; ++kb) {
    if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) return false;
    mbar_expect_tx(&full[stage], STAGE_BYTES);
    uint8_t* a = sA + stage * A_BYTES;
    uint8_t* b = sB + stage * B_BYTES;
    const int k0 = koff + kb * BK;
    if (!A_MN) {
      tma_load(tmA, &full[stage], a, k0, tm * BM);
    } else {
      tma_load(tmA, &full[stage], a, tm * BM, k0);
      tma_load(tmA, &full[stage], a + CHUNK_BYTES, tm * BM + 64, k0);
    }
    if (!B_MN) {
      if (z >= 0) tma_load3(tmB, &full[stage], b, k0, tn * BN, z);
      else tma_load(tmB, &full[stage], b, k0, tn * BN);
    } else {
#pragma unroll
      for (int c = 0; c < BN / 64; ++c) {
        if (z >= 0) tma_load3(tmB, &full[stage], b + c * CHUNK_BYTES, tn * BN + 64 * c, k0, z);
        else tma_load(tmB, &full[stage], b + c * CHUNK_BYTES, tn * BN + 64 * c, k0);
      }
    }
    inflight_mask |= 1u << stage;
    inflight_parity = (inflight_parity & ~(1u << stage)) | (phase << stage);
    if (++stage == STAGES) {
      stage = 0;
      phase ^= 1;
    }
  }
  return true;
}

// MMA side of one output tile: nk K-blocks accumulated into TMEM column d.
template <bool A_MN, bool B_MN>
__device__ __forceinline__ bool mma_tile(uint32_t d, int nk, uint8_t* sA, uint8_t* sB, uint64_t* full,
                                         uint64_t* empty, int& stage, uint32_t& phase, volatile int* abort_flag) {
  constexpr uint32_t ID = idesc(A_MN, B_MN);
  for (int kb = 0; kb < nk; ++kb) {
    if (!mbar_wait(&full[stage], phase, abort_flag)) return false;
    tc_fence_after();
    const uint32_t a0 = su32(sA + stage * A_BYTES), b0 = su32(sB + stage * B_BYTES);
#pragma unroll
    for (int k = 0; k < BK / UMMA_K; ++k) {
      const uint64_t ad = A_MN ? sdesc(a0 + k * UMMA_K * 128, CHUNK_BYTES, 1024) : sdesc(a0 + k * UMMA_K * 2, 16, 1024);
      const uint64_t bd = B_MN ? sdesc(b0 + k * UMMA_K * 128, CHUNK_BYTES, 1024) : sdesc(b0 + k * UMMA_K * 2, 16, 1024);
      tc_mma(d, ad, bd, ID, (kb | k) != 0);
    }
    tc_commit(&empty[stage]);
    if (++stage == STAGES) {
      stage = 0;
      phase ^= 1;
    }
  }
  return true;
}

// Epilogue of one tile from accumulator column block acc (warp-collective loads).
__device__ __forceinline__ void epilogue_tile(const Epi& e, int local, uint32_t taddr, int row_in_tile) {
  int tm, tn;
  tile_mn(local, e, tm, tn);
  const int row = tm * BM + row_in_tile;
  for (int c = 0; c < BN / 32; ++c) {
    uint32_t r[32];
    tmem_ld32(taddr + (uint32_t)(c * 32), r);
    const int col = tn * BN + c * 32;
    if (row < e.M && col < e.N) epi_store(e, row, col, r);
  }
}

// Where output tile `tile` of an expert-grouped launch (MODE 1 or 2) lives:
// its local tile index and epilogue, the expert coordinate of B (mode 1), the
// K offset and K-block count.  False: the tile has no rows (mode 1).
template <int MODE>
__device__ __forceinline__ bool grouped_tile(const Params& p, int tile, int& local, int& z, int& koff, int& nk,
                                             Epi& e) {
  e = p.e[0];
  if (MODE == 1) {
    int tm, tn;
    tile_mn(tile, e, tm, tn);
    z = p.tile_expert[tm];
    local = tile;
    koff = 0;
    nk = (e.K + BK - 1) / BK;
    return z >= 0;
  }
  const int per = e.tiles_m * e.tiles_n;
  const int g = tile / per;
  local = tile - g * per;
  z = -1;
  koff = p.grp_k0[g];
  nk = p.grp_nk[g];
  e.D += (int64_t)p.grp_e[g] * p.d_estride;
  return true;
}

// NG groups (1 or 2) with compile-time majorness (A0, B0) and (A1, B1);
// MODE 0 plain, 1 and 2 the expert-grouped forms (NG = 1).
template <int NG, bool A0, bool B0, bool A1, bool B1, int MODE = 0>
__global__ void __launch_bounds__(THREADS, 1) gemm_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_tiles = p.tile_start[NG];
  const int split = NG > 1 ? p.tile_start[1] : num_tiles;  // first tile of group 1

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&p.ta[0]) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&p.tb[0]) : "memory");
    if (NG > 1) {
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&p.ta[1]) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&p.tb[1]) : "memory");
    }
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // stages the producer has filled and may still be in flight (for the drain)
  uint32_t inflight_mask = 0, inflight_parity = 0;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok && !p.stall; tile += gridDim.x) {
        int tm, tn;
        if (MODE != 0) {
          int local, z, koff, nk;
          Epi e;
          if (!grouped_tile<MODE>(p, tile, local, z, koff, nk, e)) continue;
          tile_mn(local, e, tm, tn);
          ok = produce_tile<A0, B0>(&p.ta[0], &p.tb[0], tm, tn, nk, sA, sB, full, empty, stage, phase, abort_flag,
                                    inflight_mask, inflight_parity, z, koff);
        } else if (NG == 1 || tile < split) {
          tile_mn(tile, p.e[0], tm, tn);
          ok = produce_tile<A0, B0>(&p.ta[0], &p.tb[0], tm, tn, (p.e[0].K + BK - 1) / BK, sA, sB, full, empty, stage,
                                    phase, abort_flag, inflight_mask, inflight_parity);
        } else {
          tile_mn(tile - split, p.e[1], tm, tn);
          ok = produce_tile<A1, B1>(&p.ta[1], &p.tb[1], tm, tn, (p.e[1].K + BK - 1) / BK, sA, sB, full, empty, stage,
                                    phase, abort_flag, inflight_mask, inflight_parity);
        }
      }
      if (!ok) fail(abort_flag, 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        int gnk = 0;
        if (MODE != 0) {
          int local, z, koff;
          Epi e;
          if (!grouped_tile<MODE>(p, tile, local, z, koff, gnk, e)) continue;
        }
        const int acc = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        ++it;
        if (!mbar_wait(&tempty[acc], aph ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * BN);
        if (MODE != 0)
          ok = mma_tile<A0, B0>(d, gnk, sA, sB, full, empty, stage, phase, abort_flag);
        else if (NG == 1 || tile < split)
          ok = mma_tile<A0, B0>(d, (p.e[0].K + BK - 1) / BK, sA, sB, full, empty, stage, phase, abort_flag);
        else
          ok = mma_tile<A1, B1>(d, (p.e[1].K + BK - 1) / BK, sA, sB, full, empty, stage, phase, abort_flag);
        if (!ok) break;
        tc_commit(&tfull[acc]);
      }
      if (!ok) fail(abort_flag, 2);
    }
  } else {
    const int q = warp & 3;  // this warp may read TMEM lanes 32q .. 32q+31
    const int row_in_tile = q * 32 + lane;
    int it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      int local = tile;
      Epi ge;
      if (MODE != 0) {
        int z, koff, nk;
        if (!grouped_tile<MODE>(p, tile, local, z, koff, nk, ge)) continue;
      }
      const int acc = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      ++it;
      // warp-uniform outcome: the TMEM loads below are warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], aph, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      if (MODE != 0) epilogue_tile(ge, local, taddr, row_in_tile);
      else if (NG == 1 || tile < split) epilogue_tile(p.e[0], tile, taddr, row_in_tile);
      else epilogue_tile(p.e[1], tile - split, taddr, row_in_tile);
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
    }
    if (!ok && lane == 0) fail(abort_flag, 3);
  }

  // On an abort, let the producer's own copies land before the CTA exits.
  if (warp == 0 && lane == 0 && *abort_flag) {
    for (int s = 0; s < STAGES; ++s)
      if (inflight_mask & (1u << s)) {
        const long long t0 = clock64();
        while (!mbar_test(&full[s], (inflight_parity >> s) & 1) && clock64() - t0 < kWaitCycles) {
        }
      }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS));
  }
}

// ---------------------------------------------------------------- CTA-pair GEMM
// Two CTAs of a cluster compute one 256 x 256 output tile with
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16): each CTA loads its own
// 128 rows of A and its own 128 rows of B (the B tile's two halves) into its
// shared memory, and the pair's even CTA issues the MMAs, which read both
// CTAs' operands; each CTA's TMEM holds its 128 rows of the accumulator.
// Per SM a 64-deep K block is 32 KB instead of 48 KB for the same MMA time,
// so six stages fit where four did.  Barriers: every copy of the pair
// completes on the even CTA's full[stage]; the MMAs' commits arrive on
// empty[stage] and on the accumulator-full barrier of both CTAs; both CTAs'
// epilogue threads arrive on the even CTA's accumulator-empty barrier.
constexpr int P_STAGES = 6;
constexpr int PA_BYTES = BM * BK * 2;         // this CTA's 128 rows of A: 16 KB
constexpr int PB_BYTES = (BN / 2) * BK * 2;   // this CTA's 128 rows of B: 16 KB
constexpr int P_STAGE_BYTES = PA_BYTES + PB_BYTES;
constexpr int P_SMEM_BYTES = P_STAGES * P_STAGE_BYTES + 1024 + 256;
// Wide tiles (NW = 2, for long-K launches): 256 x 512 per pair, one 512-column
// accumulator, each CTA holding two 128-row blocks of B per stage (48 KB), so
// 4 stages in the same shared memory.
template <int NW>
__host__ __device__ constexpr int p_stages() {
  return NW == 1 ? P_STAGES : 4;
}
static_assert(4 * (PA_BYTES + 2 * PB_BYTES) == P_STAGES * P_STAGE_BYTES, "wide and narrow rings share one layout");

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// shared::cluster address of the object at the same offset in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(su32(p)), "r"(rank));
  return a;
}
// TMA tile load into this CTA's shared memory whose completion counts on the
// pair's barrier at shared::cluster address `bar` (the even CTA's)
__device__ __forceinline__ void tma_load_pair(const CUtensorMap* map, uint32_t bar, void* dst, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(su32(dst)),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tc_mma_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accum));
}
// completion of this thread's MMAs arrives on the barrier at this offset in both CTAs of the pair
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          su32(bar)),
      "h"((uint16_t)3)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__host__ __device__ constexpr uint32_t idesc_pair(bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(BN >> 3) << 17) | ((uint32_t)((2 * BM) >> 4) << 24);
}
// 256-row tile tm and 256-column tile tn of pair tile `tile` of a group,
// rastered in bands of e.group_m row tiles
__device__ __forceinline__ void pair_tile_mn(int tile, const Epi& e, int& tm, int& tn) {
  const int tiles_m = (e.M + 2 * BM - 1) / (2 * BM);
  const int per_group = e.group_m * e.tiles_n;
  const int first = (tile / per_group) * e.group_m;
  const int gsize = min(tiles_m - first, e.group_m);
  const int in = tile % per_group;
  tm = first + in % gsize;
  tn = in / gsize;
}

// Producer side of one pair tile: this CTA's halves of A and B, K block by K
// block (B: one 128-row block per 256 columns of the tile, 256 apart).
template <bool A_MN, bool B_MN, int NW>
__device__ __forceinline__ bool produce_pair_tile(const CUtensorMap* tmA, const CUtensorMap* tmB, int arow, int brow,
                                                  int nk, uint8_t* sA, uint8_t* sB, uint64_t* full, uint64_t* empty,
                                                  bool leader, int& stage, uint32_t& phase, volatile int* abort_flag,
                                                  uint32_t& inflight_mask, uint32_t& inflight_parity) {
  for (int kb = 0; kb < nk; ++kb) {
    if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) return false;
    // the even CTA's full[stage] expects both CTAs' bytes
    if (leader) mbar_expect_tx(&full[stage], 2 * (PA_BYTES + NW * PB_BYTES));
    const uint32_t bar = cluster_addr(&full[stage], 0);
    uint8_t* a = sA + stage * PA_BYTES;
    uint8_t* b = sB + stage * (NW * PB_BYTES);
    const int k0 = kb * BK;
    if (!A_MN) {
      tma_load_pair(tmA, bar, a, k0, arow);
    } else {
      tma_load_pair(tmA, bar, a, arow, k0);
      tma_load_pair(tmA, bar, a + CHUNK_BYTES, arow + 64, k0);
    }
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      if (!B_MN) {
        tma_load_pair(tmB, bar, b + w * PB_BYTES, k0, brow + w * BN);
      } else {
        tma_load_pair(tmB, bar, b + w * PB_BYTES, brow + w * BN, k0);
        tma_load_pair(tmB, bar, b + w * PB_BYTES + CHUNK_BYTES, brow + w * BN + 64, k0);
      }
    }
    inflight_mask |= 1u << stage;
    inflight_parity = (inflight_parity & ~(1u << stage)) | (phase << stage);
    if (++stage == p_stages<NW>()) {
      stage = 0;
      phase ^= 1;
    }
  }
  return true;
}

// MMA side of one pair tile (the even CTA's issuing thread): per K step one
// M = 256, N = 256 MMA per 256 columns of the tile, into accumulator columns
// 256 w .. 256 w + 255.
template <bool A_MN, bool B_MN, int NW>
__device__ __forceinline__ bool mma_pair_tile(uint32_t d, int nk, uint8_t* sA, uint8_t* sB, uint64_t* full,
                                              uint64_t* empty, int& stage, uint32_t& phase, volatile int* abort_flag) {
  constexpr uint32_t ID = idesc_pair(A_MN, B_MN);
  for (int kb = 0; kb < nk; ++kb) {
    if (!mbar_wait(&full[stage], phase, abort_flag)) return false;
    tc_fence_after();
    const uint32_t a0 = su32(sA + stage * PA_BYTES), b0 = su32(sB + stage * (NW * PB_BYTES));
#pragma unroll
    for (int k = 0; k < BK / UMMA_K; ++k) {
      const uint64_t ad = A_MN ? sdesc(a0 + k * UMMA_K * 128, CHUNK_BYTES, 1024) : sdesc(a0 + k * UMMA_K * 2, 16, 1024);
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const uint32_t bw = b0 + w * PB_BYTES;
        const uint64_t bd = B_MN ? sdesc(bw + k * UMMA_K * 128, CHUNK_BYTES, 1024) : sdesc(bw + k * UMMA_K * 2, 16, 1024);
        tc_mma_pair(d + (uint32_t)(w * BN), ad, bd, ID, (kb | k) != 0);
      }
    }
    tc_commit_pair(&empty[stage]);  // the stage is free in both CTAs once these MMAs are done
    if (++stage == p_stages<NW>()) {
      stage = 0;
      phase ^= 1;
    }
  }
  return true;
}

constexpr int P_TRING = 4;  // tile ids in flight between the pair's producer and its consumers
// consumers that release a tile-id slot on the even CTA: its MMA thread, the odd CTA's
// producer and lane 0 of the four epilogue warps of each CTA
constexpr int P_TID_CONSUMERS = 1 + 1 + 2 * 4;

__device__ __forceinline__ bool mbar_test_cl(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// bounded wait whose acquire covers writes the peer CTA released to this barrier
__device__ __forceinline__ bool mbar_wait_cl(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
  if (mbar_test_cl(b, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_test_cl(b, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitCycles) return false;
  }
}
__device__ __forceinline__ void st_cluster_s32(uint32_t addr, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

template <int NG, bool A0, bool B0, bool A1, bool B1, int NW = 1>
__global__ void __launch_bounds__(THREADS, 1) gemm_pair_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + p_stages<NW>() * PA_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + P_STAGES * P_STAGE_BYTES);
  uint64_t* empty = full + P_STAGES;
  uint64_t* tfull = empty + P_STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* tid_full = tempty + 2;
  uint64_t* tid_empty = tid_full + P_TRING;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tid_empty + P_TRING);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* tid_ring = reinterpret_cast<volatile int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int cl = (int)(blockIdx.x >> 1), ncl = (int)(gridDim.x >> 1);
  const int num_tiles = p.tile_start[NG];
  const int split = NG > 1 ? p.tile_start[1] : num_tiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * 128);  // the epilogue threads of both CTAs (the even CTA's counts)
    }
    for (int r = 0; r < P_TRING; ++r) {
      mbar_init(&tid_full[r], 1);
      mbar_init(&tid_empty[r], P_TID_CONSUMERS);  // the even CTA's counts
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&p.ta[0]) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&p.tb[0]) : "memory");
    if (NG > 1) {
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&p.ta[1]) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&p.tb[1]) : "memory");
    }
  }
  if (warp == 1) {  // one warp of each CTA of the pair allocates, together
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before any copy or arrival reaches them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  uint32_t inflight_mask = 0, inflight_parity = 0;

  // Tile order: the pair's first tile is its cluster index; every later one is
  // a ticket drawn from the launch's counter (tile ncl + ticket), so the tiles
  // in flight are always a window of consecutive tiles of the raster order,
  // whatever the speed of each SM.  Every cluster draws until it gets a ticket
  // past the last tile; exactly ncl such tickets exist, and the cluster that
  // draws the very last one resets the counter for the launch that next uses it.
  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const int tickets = (num_tiles > ncl ? num_tiles - ncl : 0) + ncl;
      int ahead = -1;  // the ticket drawn one tile ahead (its latency hides behind the current tile's loads)
      for (int i = 0; ok && !p.stall; ++i) {
        const int slot = i % P_TRING;
        const uint32_t ph = (uint32_t)(i / P_TRING) & 1;
        int tile;
        if (leader) {
          if (!mbar_wait(&tid_empty[slot], ph ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          if (!p.tile_ctr) {  // static order: every ncl-th tile
            tile = cl + i * ncl < num_tiles ? cl + i * ncl : -1;
          } else if (i == 0 && cl < num_tiles) {
            tile = cl;
          } else {
            const int raw = ahead >= 0 ? ahead : atomicAdd(p.tile_ctr, 1);
            ahead = -1;
            if (raw >= tickets) {  // a counter left behind by an aborted launch
              ok = false;
              break;
            }
            if (raw == tickets - 1) atomicExch(p.tile_ctr, 0);
            tile = ncl + raw < num_tiles ? ncl + raw : -1;
          }
          if (tile >= 0 && p.tile_ctr) ahead = atomicAdd(p.tile_ctr, 1);
          tid_ring[slot] = tile;
          st_cluster_s32(cluster_addr((const void*)&tid_ring[slot], 1), tile);
          mbar_arrive(&tid_full[slot]);
          mbar_arrive_remote(cluster_addr(&tid_full[slot], 1));
        } else {
          if (!mbar_wait_cl(&tid_full[slot], ph, abort_flag)) {
            ok = false;
            break;
          }
          tile = tid_ring[slot];
          mbar_arrive_remote(cluster_addr(&tid_empty[slot], 0));
        }
        if (tile < 0) break;
        int tm, tn;
        if (NG == 1 || tile < split) {
          pair_tile_mn(tile, p.e[0], tm, tn);
          ok = produce_pair_tile<A0, B0, NW>(&p.ta[0], &p.tb[0], tm * 2 * BM + (int)rank * BM,
                                             tn * BN * NW + (int)rank * (BN / 2),
                                         (p.e[0].K + BK - 1) / BK, sA, sB, full, empty, leader, stage, phase,
                                         abort_flag, inflight_mask, inflight_parity);
        } else {
          pair_tile_mn(tile - split, p.e[1], tm, tn);
          ok = produce_pair_tile<A1, B1, NW>(&p.ta[1], &p.tb[1], tm * 2 * BM + (int)rank * BM,
                                             tn * BN * NW + (int)rank * (BN / 2),
                                         (p.e[1].K + BK - 1) / BK, sA, sB, full, empty, leader, stage, phase,
                                         abort_flag, inflight_mask, inflight_parity);
        }
      }
      if (!ok) fail(abort_flag, 1);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int it = 0;; ++it) {
        const int slot = it % P_TRING;
        if (!mbar_wait(&tid_full[slot], (uint32_t)(it / P_TRING) & 1, abort_flag)) {
          ok = false;
          break;
        }
        const int tile = tid_ring[slot];
        mbar_arrive(&tid_empty[slot]);
        if (tile < 0) break;
        // two 256-column accumulators, or one of 512 columns for wide tiles
        const int acc = NW == 1 ? (it & 1) : 0;
        const uint32_t aph = NW == 1 ? (uint32_t)((it >> 1) & 1) : (uint32_t)(it & 1);
        if (!mbar_wait(&tempty[acc], aph ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * BN);
        if (NG == 1 || tile < split)
          ok = mma_pair_tile<A0, B0, NW>(d, (p.e[0].K + BK - 1) / BK, sA, sB, full, empty, stage, phase, abort_flag);
        else
          ok = mma_pair_tile<A1, B1, NW>(d, (p.e[1].K + BK - 1) / BK, sA, sB, full, empty, stage, phase, abort_flag);
        if (!ok) break;
        tc_commit_pair(&tfull[acc]);  // both CTAs' epilogues may read their rows
      }
      if (!ok) fail(abort_flag, 2);
    }
  } else {
    const int q = warp & 3;  // this warp may read TMEM lanes 32q .. 32q+31
    const int row_in_tile = q * 32 + lane;
    const uint32_t tempty_lead[2] = {cluster_addr(&tempty[0], 0), cluster_addr(&tempty[1], 0)};
    bool ok = true;
    for (int it = 0;; ++it) {
      const int slot = it % P_TRING;
      // warp-uniform outcomes: the TMEM loads below are warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait_cl(&tid_full[slot], (uint32_t)(it / P_TRING) & 1, abort_flag))) {
        ok = false;
        break;
      }
      const int tile = tid_ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(cluster_addr(&tid_empty[slot], 0));
      if (tile < 0) break;
      const int acc = NW == 1 ? (it & 1) : 0;
      const uint32_t aph = NW == 1 ? (uint32_t)((it >> 1) & 1) : (uint32_t)(it & 1);
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], aph, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const Epi& e = (NG == 1 || tile < split) ? p.e[0] : p.e[1];
      int tm, tn;
      pair_tile_mn((NG == 1 || tile < split) ? tile : tile - split, e, tm, tn);
      const int row = tm * 2 * BM + (int)rank * BM + row_in_tile;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      for (int c = 0; c < BN * NW / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(taddr + (uint32_t)(c * 32), r);
        const int col = tn * BN * NW + c * 32;
        if (row < e.M && col < e.N) epi_store(e, row, col, r);
      }
      tc_fence_before();
      mbar_arrive_remote(tempty_lead[acc]);  // the even CTA counts both CTAs' epilogues
    }
    if (!ok && lane == 0) fail(abort_flag, 3);
  }

  // On an abort, let every copy in flight land before the pair exits: the
  // even CTA waits for its full barriers (which count both CTAs' bytes), the
  // odd CTA, which cannot observe its own copies, waits a fixed time.
  if (warp == 0 && lane == 0 && *abort_flag) {
    const long long t0 = clock64();
    if (leader) {
      for (int s = 0; s < P_STAGES; ++s)
        if (inflight_mask & (1u << s))
          while (!mbar_test(&full[s], (inflight_parity >> s) & 1) && clock64() - t0 < kWaitCycles) {
          }
    }
    while (clock64() - t0 < 400000) {  // about 0.2 ms
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still reach its shared memory or TMEM
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS));
  }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;
int g_num_sms = 0;
int g_pair_clusters = 0;
constexpr int kWideK = 8192;  // K from which dense pair launches use 256 x 512 tiles
constexpr int kTileCounters = 1024;  // tile-ticket counters, one per pair launch in a ring
int* g_tile_ctrs = nullptr;
std::atomic<unsigned> g_tile_ctr_next{0};
cudaError_t g_init_err = cudaSuccess;

void init_once() {
  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
    g_init_err = e != cudaSuccess ? e : cudaErrorNotSupported;
    return;
  }
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  int dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
  const void* kernels[] = {(const void*)gemm_kernel<1, false, false, false, false>,
                           (const void*)gemm_kernel<1, false, true, false, false>,
                           (const void*)gemm_kernel<1, true, false, false, false>,
                           (const void*)gemm_kernel<1, true, true, false, false>,
                           (const void*)gemm_kernel<2, true, true, false, true>,
                           (const void*)gemm_kernel<1, false, false, false, false, 1>,
                           (const void*)gemm_kernel<1, false, true, false, false, 1>,
                           (const void*)gemm_kernel<1, true, true, false, false, 2>};
  for (const void* k : kernels) {
    const cudaError_t a = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (a != cudaSuccess) g_init_err = a;
  }
  const void* pair_kernels[] = {(const void*)gemm_pair_kernel<1, false, false, false, false>,
                                (const void*)gemm_pair_kernel<1, false, true, false, false>,
                                (const void*)gemm_pair_kernel<1, true, false, false, false>,
                                (const void*)gemm_pair_kernel<1, true, true, false, false>,
                                (const void*)gemm_pair_kernel<2, true, true, false, true>,
                                (const void*)gemm_pair_kernel<1, false, false, false, false, 2>,
                                (const void*)gemm_pair_kernel<1, false, true, false, false, 2>,
                                (const void*)gemm_pair_kernel<1, true, false, false, false, 2>,
                                (const void*)gemm_pair_kernel<1, true, true, false, false, 2>,
                                (const void*)gemm_pair_kernel<2, true, true, false, true, 2>};
  for (const void* k : pair_kernels) {
    const cudaError_t a = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM_BYTES);
    if (a != cudaSuccess) g_init_err = a;
  }
  // pairs resident at once (an SM pair shares a TPC; the count can be below SMs / 2)
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(g_num_sms & ~1));
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = P_SMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int nc = 0;
  if (cudaOccupancyMaxActiveClusters(&nc, gemm_pair_kernel<1, false, false, false, false>, &cfg) != cudaSuccess ||
      nc <= 0) {
    cudaGetLastError();
    nc = g_num_sms / 2;
  }
  g_pair_clusters = nc < g_num_sms / 2 ? nc : g_num_sms / 2;
  if (cudaMalloc(&g_tile_ctrs, kTileCounters * sizeof(int)) != cudaSuccess ||
      cudaMemset(g_tile_ctrs, 0, kTileCounters * sizeof(int)) != cudaSuccess) {
    g_init_err = cudaErrorMemoryAllocation;
    g_tile_ctrs = nullptr;
  }
}

// 2-D bf16 tensor map of a row-major [rows][cols] matrix with row stride ld,
// box {64 columns, box_rows rows}, 128-byte swizzle, zero fill out of bounds.
bool make_map(CUtensorMap* m, const bf16* base, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<bf16*>(base), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D bf16 tensor map of n experts' row-major [rows][cols] matrices (row
// stride ld, expert stride estride, in elements), box {64, box_rows, 1}.
bool make_map3(CUtensorMap* m, const bf16* base, int64_t rows, int64_t cols, int64_t ld, int64_t n,
               int64_t estride, int box_rows) {
  const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)n};
  const cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)estride * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<bf16*>(base), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

std::atomic<int> g_stall_next{0};
// dense GEMMs: 0 one CTA per 128 x 256 tile; CTA pairs on 256 x 256 tiles
// (256 x 512 for long-K launches), 1 drawing tiles from a counter, 2 taking
// every ncl-th tile in raster order; 3 as 1 without the 512-wide tiles
std::atomic<int> g_gemm_mode{1};
int gemm_mode(int mode) {
  const int prev = g_gemm_mode.load();
  if (mode >= 0 && mode <= 3) g_gemm_mode = mode;
  return prev;
}
int gemm_stall_take() {
  int v = g_stall_next.load();
  while (v > 0 && !g_stall_next.compare_exchange_weak(v, v - 1)) {
  }
  return v > 0 ? 1 : 0;
}
void gemm_inject_stall(int launches) { g_stall_next = launches; }

int gemm_num_sms() {
  std::call_once(g_once, init_once);
  return g_num_sms;
}

namespace {
// pair: the B map's K-major box is one CTA's half of a 256-row tile
cudaError_t fill_group(const GemmArgs& g, CUtensorMap* ma, CUtensorMap* mb, Epi* e, bool pair) {
  if (g.M <= 0 || g.N <= 0 || g.K <= 0 || !g.A || !g.B) return cudaErrorInvalidValue;
  if (!g.D && !g.acc_mode) return cudaErrorInvalidValue;
  if ((g.lda | g.ldb) % 8 || (g.D && g.ldd % 8) || (g.R && g.ldr % 8) || (g.acc_mode && g.ldacc % 8))
    return cudaErrorInvalidValue;
  if (!al16(g.A) || !al16(g.B) || (g.D && !al16(g.D)) || (g.R && !al16(g.R)) || (g.acc_mode && !al16(g.Dacc)))
    return cudaErrorInvalidValue;
  if (g.acc_mode && !g.Dacc) return cudaErrorInvalidValue;
  // A: K-major [M][K] (box 64 x 128) or MN-major [K][M] (box 64 x 64)
  bool ok = g.a_mn ? make_map(ma, g.A, g.K, g.M, g.lda, BK) : make_map(ma, g.A, g.M, g.K, g.lda, BM);
  ok = ok && (g.b_mn ? make_map(mb, g.B, g.K, g.N, g.ldb, BK) : make_map(mb, g.B, g.N, g.K, g.ldb, pair ? BN / 2 : BN));
  if (!ok) return cudaErrorInvalidValue;
  e->D = g.D; e->ldd = g.ldd; e->R = g.R; e->ldr = g.ldr; e->Dacc = g.Dacc; e->ldacc = g.ldacc;
  e->acc_mode = g.acc_mode;
  e->M = g.M; e->N = g.N; e->K = g.K;
  e->tiles_m = (g.M + BM - 1) / BM;
  e->tiles_n = (g.N + BN - 1) / BN;
  e->group_m = 16;
  e->a_mn = g.a_mn ? 1 : 0;
  e->b_mn = g.b_mn ? 1 : 0;
  return cudaSuccess;
}

// Raster band of the CTA-pair tiles, in 256-row tiles.  The tiles in flight
// are a window of about `pairs` consecutive tiles: `band` row tiles by
// pairs / band column tiles, whose operand slices (256 rows by the whole K,
// BF16) should stay in L2 while the window passes, so that the column
// operand is read from DRAM once per band.  The tallest band whose window
// fits about half the L2 is taken (fewer bands, fewer re-reads of the column
// operand); when no band fits (long K), a square window (8 rows) keeps the
// slices the window's tiles share to a minimum.
int pair_band(int K, int pairs) {
  const double slice = 2.0 * BM * 2.0 * K;  // bytes of one 256-row operand slice
  const double budget = 64e6;
  int best = 8;
  for (int band = 16; band <= 64; band *= 2) {
    const int cols = (pairs + band - 1) / band;
    if ((band + cols + 1) * slice <= budget) best = band;
  }
  return best;
}

template <int NG, bool A0, bool B0, bool A1, bool B1, int NW = 1>
cudaError_t launch_pair_kernel(const Params& p, int tiles, cudaStream_t s) {
  const int clusters = tiles < g_pair_clusters ? tiles : g_pair_clusters;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(2 * (clusters > 0 ? clusters : 1)));
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = P_SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_pair_kernel<NG, A0, B0, A1, B1, NW>, p);
}

cudaError_t launch(const GemmArgs* gs, int n, cudaStream_t s) {
  std::call_once(g_once, init_once);
  if (g_init_err != cudaSuccess) return g_init_err;
  const int mode = g_gemm_mode.load();
  const bool pair = mode != 0 && g_pair_clusters >= 1;
  // wide pair tiles (256 x 512) when every group has a long K, at least 512
  // columns and no residual: the serial epilogue of a single accumulator is
  // then a few per cent of a tile, and each tile reads the row operand once
  // for twice the columns (with a residual to read, the longer epilogue cost
  // more than the traffic saved: 6 % on the 7.6B down projection)
  bool wide = pair && mode != 3;
  for (int i = 0; i < n; ++i) wide = wide && gs[i].K >= kWideK && gs[i].N >= 2 * BN && !gs[i].R;
  Params p;
  std::memset(&p, 0, sizeof p);
  p.ngroups = n;
  p.tile_start[0] = 0;
  for (int i = 0; i < n; ++i) {
    cudaError_t e = fill_group(gs[i], &p.ta[i], &p.tb[i], &p.e[i], pair);
    if (e != cudaSuccess) return e;
    if (pair) p.e[i].group_m = pair_band(p.e[i].K, g_pair_clusters);
    if (wide) p.e[i].tiles_n = (p.e[i].N + 2 * BN - 1) / (2 * BN);
    const int tm = pair ? (p.e[i].M + 2 * BM - 1) / (2 * BM) : p.e[i].tiles_m;
    p.tile_start[i + 1] = p.tile_start[i] + tm * p.e[i].tiles_n;
  }
  p.stall = gemm_stall_take();
  const int tiles = p.tile_start[n];
  if (pair) {
    if (mode != 2) p.tile_ctr = g_tile_ctrs + (g_tile_ctr_next.fetch_add(1) % kTileCounters);
    const Epi& e = p.e[0];
    cudaError_t r;
    if (wide) {
      if (n == 1) {
        if (!e.a_mn && !e.b_mn) r = launch_pair_kernel<1, false, false, false, false, 2>(p, tiles, s);
        else if (!e.a_mn && e.b_mn) r = launch_pair_kernel<1, false, true, false, false, 2>(p, tiles, s);
        else if (e.a_mn && !e.b_mn) r = launch_pair_kernel<1, true, false, false, false, 2>(p, tiles, s);
        else r = launch_pair_kernel<1, true, true, false, false, 2>(p, tiles, s);
      } else {
        r = launch_pair_kernel<2, true, true, false, true, 2>(p, tiles, s);
      }
      return r != cudaSuccess ? r : cudaGetLastError();
    }
    if (n == 1) {
      if (!e.a_mn && !e.b_mn) r = launch_pair_kernel<1, false, false, false, false>(p, tiles, s);
      else if (!e.a_mn && e.b_mn) r = launch_pair_kernel<1, false, true, false, false>(p, tiles, s);
      else if (e.a_mn && !e.b_mn) r = launch_pair_kernel<1, true, false, false, false>(p, tiles, s);
      else r = launch_pair_kernel<1, true, true, false, false>(p, tiles, s);
    } else {
      r = launch_pair_kernel<2, true, true, false, true>(p, tiles, s);
    }
    return r != cudaSuccess ? r : cudaGetLastError();
  }
  const int grid = tiles < g_num_sms ? tiles : g_num_sms;
  const Epi& e = p.e[0];
  if (n == 1) {
    if (!e.a_mn && !e.b_mn) gemm_kernel<1, false, false, false, false><<<grid, THREADS, SMEM_BYTES, s>>>(p);
    else if (!e.a_mn && e.b_mn) gemm_kernel<1, false, true, false, false><<<grid, THREADS, SMEM_BYTES, s>>>(p);
    else if (e.a_mn && !e.b_mn) gemm_kernel<1, true, false, false, false><<<grid, THREADS, SMEM_BYTES, s>>>(p);
    else gemm_kernel<1, true, true, false, false><<<grid, THREADS, SMEM_BYTES, s>>>(p);
  } else {
    gemm_kernel<2, true, true, false, true><<<grid, THREADS, SMEM_BYTES, s>>>(p);
  }
  return cudaGetLastError();
}
}  // namespace

cudaError_t gemm(const GemmArgs& g, cudaStream_t s) { return launch(&g, 1, s); }

namespace {
void fill_epi(Epi* e, int M, int N, int K, bf16* D, int64_t ldd) {
  std::memset(e, 0, sizeof *e);
  e->D = D; e->ldd = ldd;
  e->M = M; e->N = N; e->K = K;
  e->tiles_m = (M + BM - 1) / BM;
  e->tiles_n = (N + BN - 1) / BN;
  e->group_m = 16;
}
}  // namespace

cudaError_t gemm_expert_rows(const GemmRowsArgs& g, cudaStream_t s) {
  std::call_once(g_once, init_once);
  if (g_init_err != cudaSuccess) return g_init_err;
  if (g.M < 0 || g.M % BM || g.N <= 0 || g.K <= 0 || g.n_experts <= 0 || !g.A || !g.B || !g.D || !g.tile_expert)
    return cudaErrorInvalidValue;
  if (g.lda % 8 || g.ldb % 8 || g.ldd % 8 || g.b_estride % 8 || !al16(g.A) || !al16(g.B) || !al16(g.D))
    return cudaErrorInvalidValue;
  if (g.M == 0) return cudaSuccess;
  Params p;
  std::memset(&p, 0, sizeof p);
  bool ok = make_map(&p.ta[0], g.A, g.M, g.K, g.lda, BM);
  ok = ok && (g.b_mn ? make_map3(&p.tb[0], g.B, g.K, g.N, g.ldb, g.n_experts, g.b_estride, BK)
                     : make_map3(&p.tb[0], g.B, g.N, g.K, g.ldb, g.n_experts, g.b_estride, BN));
  if (!ok) return cudaErrorInvalidValue;
  fill_epi(&p.e[0], g.M, g.N, g.K, g.D, g.ldd);
  p.e[0].b_mn = g.b_mn ? 1 : 0;
  p.ngroups = 1;
  p.tile_start[1] = p.e[0].tiles_m * p.e[0].tiles_n;
  p.tile_expert = g.tile_expert;
  p.stall = gemm_stall_take();
  const int tiles = p.tile_start[1];
  const int grid = tiles < g_num_sms ? tiles : g_num_sms;
  if (g.b_mn) gemm_kernel<1, false, true, false, false, 1><<<grid, THREADS, SMEM_BYTES, s>>>(p);
  else gemm_kernel<1, false, false, false, false, 1><<<grid, THREADS, SMEM_BYTES, s>>>(p);
  return cudaGetLastError();
}

cudaError_t gemm_expert_kgroups(const GemmKGroupArgs& g, cudaStream_t s) {
  std::call_once(g_once, init_once);
  if (g_init_err != cudaSuccess) return g_init_err;
  if (g.M <= 0 || g.N <= 0 || g.R <= 0 || g.ngrp < 0 || g.ngrp > MAX_EXPERT_GROUPS || !g.A || !g.B || !g.D)
    return cudaErrorInvalidValue;
  if (g.lda % 8 || g.ldb % 8 || g.ldd % 8 || g.d_estride % 8 || !al16(g.A) || !al16(g.B) || !al16(g.D))
    return cudaErrorInvalidValue;
  if (g.ngrp == 0) return cudaSuccess;
  Params p;
  std::memset(&p, 0, sizeof p);
  for (int i = 0; i < g.ngrp; ++i) {
    if (g.grp_klen[i] <= 0 || g.grp_klen[i] % BK || g.grp_k0[i] < 0 || g.grp_k0[i] % BK ||
        g.grp_k0[i] + g.grp_klen[i] > g.R || g.grp_e[i] < 0)
      return cudaErrorInvalidValue;
    p.grp_e[i] = g.grp_e[i];
    p.grp_k0[i] = g.grp_k0[i];
    p.grp_nk[i] = g.grp_klen[i] / BK;
  }
  p.ngrp = g.ngrp;
  p.d_estride = g.d_estride;
  bool ok = make_map(&p.ta[0], g.A, g.R, g.M, g.lda, BK) && make_map(&p.tb[0], g.B, g.R, g.N, g.ldb, BK);
  if (!ok) return cudaErrorInvalidValue;
  fill_epi(&p.e[0], g.M, g.N, g.R, g.D, g.ldd);
  p.e[0].a_mn = 1;
  p.e[0].b_mn = 1;
  p.ngroups = 1;
  p.tile_start[1] = g.ngrp * p.e[0].tiles_m * p.e[0].tiles_n;
  p.stall = gemm_stall_take();
  const int tiles = p.tile_start[1];
  const int grid = tiles < g_num_sms ? tiles : g_num_sms;
  gemm_kernel<1, true, true, false, false, 2><<<grid, THREADS, SMEM_BYTES, s>>>(p);
  return cudaGetLastError();
}

cudaError_t gemm_pair(const GemmArgs& g0, const GemmArgs& g1, cudaStream_t s) {
  // one launch for the (wgrad, dgrad) form: A and B MN-major, then B MN-major
  if (g0.a_mn && g0.b_mn && !g1.a_mn && g1.b_mn) {
    const GemmArgs gs[2] = {g0, g1};
    return launch(gs, 2, s);
  }
  cudaError_t e = launch(&g0, 1, s);
  return e != cudaSuccess ? e : launch(&g1, 1, s);
}

cudaError_t kernel_error_read(int* code, int clear) {
  cudaError_t e = cudaMemcpyFromSymbol(code, g_kernel_error, sizeof(int));
  if (e != cudaSuccess) return e;
  if (clear) {
    const int z = 0;
    e = cudaMemcpyToSymbol(g_kernel_error, &z, sizeof(int));
    if (e != cudaSuccess) return e;
    // a GEMM that gave up may have left its tile-ticket counter mid-count
    if (*code != 0 && g_tile_ctrs) {
      e = cudaDeviceSynchronize();
      if (e == cudaSuccess) e = cudaMemset(g_tile_ctrs, 0, kTileCounters * sizeof(int));
      if (e == cudaSuccess) e = cudaDeviceSynchronize();
      if (e != cudaSuccess) return e;
    }
  }
  int a = 0;
  e = attention_error_read(&a, clear);
  if (*code == 0) *code = a;
  return e;
}

}  // namespace mt
