// k_attention_tc.cu -- causal GQA attention, forward and backward, on the
// 5th-generation tensor cores (sm_103a): tcgen05.mma with TMEM accumulators,
// TMA tiles, 320 threads per CTA (a TMA warp, an MMA warp, 8 row warps, two
// per TMEM lane quarter).
//
// Forward: a persistent CTA per SM loops over work items (128 queries, query
// head, sequence), longest rows first; the next item's Q / K loads and first
// S = Q K^T run while the softmax warps finish the previous item's epilogue:
//   warp 0      TMA producer: each item's Q tile, then K and V tiles of 128
//               keys into their rings (128-byte swizzle);
//   warp 1      allocates TMEM (S0 | S1 | O_0 | O_1) and, from one thread,
//               issues S_j = Q K_j^T (M=128, N=128) into S[j % 2] and, once the
//               softmax has written P_{j-1} over S_{j-1} (BF16, in TMEM),
//               O_0 += P V over the tile's keys 0..63 and O_1 += P V over keys
//               64..127 with P as the A operand from TMEM and V an MN-major
//               operand from shared memory;
//   warps 2..9  softmax: warp w owns the query rows of TMEM lane quarter w % 4
//               and one half of every key tile (warps 2..5 keys 0..63, 6..9
//               keys 64..127), with its own exponent base, sum and accumulator
//               O_half.  The base follows the running max lazily: it moves (and
//               O_half and the sum are rescaled) only when a tile's max exceeds
//               it by more than 8 in the exp2 domain, so P stays below 2^8 and
//               most tiles touch neither O nor the previous P V.  At the end the
//               two halves of a row merge (m = max, each side scaled by
//               2^(m_h - m)) and O / l and LSE = (m + log2 l) ln 2 go to global
//               memory.
// Splitting every row over two threads halves the per-thread softmax work per
// tile without any per-tile exchange between them.  The double-buffered S
// lets S_{j+1} run on the tensor core while the softmax works on S_j; P in
// TMEM needs no shared-memory tile, so the softmax of tile j waits for the
// previous P V only when it rescales.  tcgen05.mma operations of one thread
// run in issue order, so S_{j+2} overwrites P_j only after O += P_j V read it.
// Every mbarrier wait is bounded; an expired wait sets the kernel error word
// and the CTA stops, drains its copies and frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "mt_kernels.h"

namespace mt {
namespace {

// TMA warp, MMA warp, 8 row warps (two per TMEM lane quarter)
constexpr int ATTN_THREADS = 320;
constexpr int NFK = 3;  // forward: K tile stages
constexpr int NFV = 2;  // forward: V tile stages
constexpr long long kWaitCycles = 4000000000LL;
constexpr int CH = 16384;  // one 64-column chunk of a 128-row tile (128 rows x 128 B)

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
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
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
  if (mbar_test(b, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_test(b, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitCycles) return false;
  }
}
__device__ __forceinline__ void tma_load(const CUtensorMap* map, uint64_t* bar, void* dst, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(su32(dst)),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(su32(bar))
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accum));
}
// The same with the A operand in TMEM (K-major: lane = row of A, each 32-bit
// column two consecutive K elements, a K-step of 16 = 8 columns).
__device__ __forceinline__ void tc_mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(accum));
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
               : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// tcgen05.ld without the wait, so several loads share one tcgen05.wait::ld.
__device__ __forceinline__ void tmem_ld32_nw(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// Waits for this thread's outstanding tcgen05.ld and ties the destination
// registers to the wait, so no use of them can be scheduled before it.
__device__ __forceinline__ void tmem_wait_ld2(uint32_t (&a)[32], uint32_t (&b)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(a[i]), "+r"(b[i]));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// 2^x on the special-function unit (PTX ex2.approx.ftz.f32).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])),
      "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
      "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])),
      "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])),
      "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])),
      "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ULL << 46) | (2ULL << 61);
}
// A descriptor advanced by `bytes`: the start-address field holds addr >> 4
// and shared addresses stay below 256 KB, so the addition never carries out
// of the field.  Building descriptors once and advancing them by constants
// keeps the MMA-issuing thread's per-instruction work to one 64-bit add.
__device__ __forceinline__ uint64_t dadv(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }
__host__ __device__ constexpr uint32_t idesc(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ int g_attn_error = 0;

// Work item i of a launch over (128-query tile, head, sequence) items.
// Longest first (head_major = 0): every head's last query tile, then every
// head's second-to-last, ... (balances persistent CTAs).  Head-major
// (head_major = 1): all query tiles of one head and sequence, longest first,
// then the next head -- the CTAs running together share one KV head's keys
// and values in L2 (long sequences, one CTA per item).
struct AttnItem {
  int qb, h, n;
};
__device__ __forceinline__ AttnItem attn_item(int i, int nqb, int nh, int n_seq, int head_major) {
  if (head_major) {
    const int rest = i / nqb;
    return {nqb - 1 - i % nqb, rest % nh, rest / nh};
  }
  const int per_qb = nh * n_seq, r = i % per_qb;
  return {nqb - 1 - i / per_qb, r % nh, r / nh};
}

template <int HD, bool PERSIST>
__global__ void __launch_bounds__(ATTN_THREADS, 1)
    attn_fwd_tc_k(const __grid_constant__ CUtensorMap tm, int S, int nh, int nkv, int n_seq, bf16* __restrict__ o,
                  float* __restrict__ lse, float scale_log2, int head_major) {
  constexpr int NC = HD / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm;
  uint8_t* sK = sQ + NC * CH;        // NFK stages: K is free once S has been computed
  uint8_t* sV = sK + NFK * NC * CH;  // NFV stages: V is held until O += P V
  // the merge values of the two halves of each row [2 halves][(m, l)][128 rows]
  float* fin = reinterpret_cast<float*>(sV + NFV * NC * CH);
  uint64_t* bars = reinterpret_cast<uint64_t*>(fin + 512);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;          // [NFK]
  uint64_t* k_empty = k_full + NFK;     // [NFK]
  uint64_t* v_full = k_empty + NFK;     // [NFV]
  uint64_t* v_empty = v_full + NFV;     // [NFV]
  uint64_t* s_full = v_empty + NFV;     // [2]
  // [2]: P_g over S buffer g % 2.  One barrier per buffer: tile g + 2's P
  // needs S_{g+2}, issued only after O += P_g V, so neither barrier can
  // complete a second phase before the MMA thread has seen the first
  uint64_t* p_full = s_full + 2;
  // (the next slot is unused: O += P_g V is tracked by v_empty of P_g's V stage)
  uint64_t* fin_ready = p_full + 3;
  uint64_t* q_empty = fin_ready + 1;  // the item's last S = Q K^T has read Q
  uint64_t* o_free = q_empty + 1;     // the epilogue has read O (the next item may overwrite it)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_free + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  // Work items, longest rows first: item i is query tile nqb - 1 - i / (nh
  // n_seq) of head (i mod nh n_seq) mod nh and sequence (i mod nh n_seq) / nh.
  // Round r gives the CTA item r G + blockIdx.x for even r and r G + G - 1 -
  // blockIdx.x for odd r (G = gridDim.x): going back and forth evens out the
  // lengths, which shrink along the list.  Key tiles, P V products and items
  // are counted across items, so every barrier phase carries on.
  const int nqb = (S + 127) / 128, per_qb = nh * n_seq, n_items = nqb * per_qb;
  const int G = (int)gridDim.x;
  // PERSIST = false: one item per CTA (item blockIdx.x), compiled as
  // straight-line code without the cross-item waits
  auto item_of = [&](int rnd) {
    if constexpr (!PERSIST) return rnd == 0 ? (int)blockIdx.x : n_items;
    return rnd * G + ((rnd & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x);
  };
  const int64_t T = (int64_t)n_seq * S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < NFK; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < NFV; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 256);
    }
    mbar_init(fin_ready, 256);
    mbar_init(o_free, 256);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tm) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                 "r"(512));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM columns: S buffer b at tmem + 128 b, O of key half h at tmem + 256 + HD h
  auto tS = [tmem](int b) { return tmem + (uint32_t)(128 * b); };
  auto tO = [tmem](int h) { return tmem + 256u + (uint32_t)(HD * h); };
  uint32_t x_inflight = 0, x_par = 0;  // producer drain bookkeeping (lane 0: K stages, lane 1: V stages)
  bool q_inflight = false;
  uint32_t q_par = 0;

  if (warp == 0) {
    // lane 0 streams each item's Q and the K ring, lane 1 the V ring, each on
    // its own barriers, so a V stage still held by O += P V never delays K
    if (lane < 2) {
      const bool is_k = lane == 0;
      const int ns = is_k ? NFK : NFV;
      uint64_t* full = is_k ? k_full : v_full;
      uint64_t* empty = is_k ? k_empty : v_empty;
      uint8_t* base = is_k ? sK : sV;
      bool ok = true;
      int g = 0;  // key tiles loaded so far
      int it = 0;
      for (int i = item_of(0); i < n_items && ok; i = item_of(++it)) {
        const AttnItem w = attn_item(i, nqb, nh, n_seq, head_major);
        const int qb = w.qb, h = w.h, n = w.n;
        const int kh = h / (nh / nkv), row0 = n * S;
        const int col = (is_k ? nh + kh : nh + nkv + kh) * HD;
        if (is_k) {
          if (PERSIST && it > 0 && !mbar_wait(q_empty, (uint32_t)((it - 1) & 1), abort_flag)) {
            ok = false;
            break;
          }
          mbar_expect_tx(q_full, NC * CH);
          for (int c = 0; c < NC; ++c) tma_load(&tm, q_full, sQ + c * CH, h * HD + 64 * c, row0 + qb * 128);
          q_inflight = true;
          q_par = (uint32_t)(it & 1);
        }
        for (int j = 0; j <= qb; ++j, ++g) {
          const int s = g % ns;
          const uint32_t u = (uint32_t)(g / ns);
          if (!mbar_wait(&empty[s], (u & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&full[s], NC * CH);
          for (int c = 0; c < NC; ++c)
            tma_load(&tm, &full[s], base + (s * NC + c) * CH, col + 64 * c, row0 + 128 * j);
          x_inflight |= 1u << s;
          x_par = (x_par & ~(1u << s)) | ((u & 1) << s);
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicCAS(&g_attn_error, 0, 11);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t IS = idesc(128, 128, false, false);
      constexpr uint32_t IO = idesc(128, HD, false, true);  // A = P from TMEM, B = V MN-major
      const uint64_t dV = sdesc(su32(sV), CH, 1024);
      const uint64_t dQ = sdesc(su32(sQ), 16, 1024), dK = sdesc(su32(sK), 16, 1024);
      int it = 0;
      // O_0 += P[:, 0:64] V[0:64, :] and O_1 += P[:, 64:128] V[64:128, :] for
      // key tile g (the first of its item when `first`: O starts from zero,
      // once the previous item's epilogue has read it); P_g sits over S_g:
      // the 64 keys of half h packed in columns 64 h .. 64 h + 31
      auto issue_pv = [&](int g, bool first) -> bool {
        if (!mbar_wait(&p_full[g & 1], (uint32_t)((g >> 1) & 1), abort_flag) ||
            !mbar_wait(&v_full[g % NFV], (uint32_t)((g / NFV) & 1), abort_flag))
          return false;
        if (PERSIST && first && it > 0 && !mbar_wait(o_free, (uint32_t)((it - 1) & 1), abort_flag)) return false;
        tc_fence_after();
        const uint64_t v = dadv(dV, (g % NFV) * NC * CH);
        const uint32_t tp = tS(g & 1);
        const uint32_t acc0 = first ? 0u : 1u;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t acc = kk > 0 ? 1u : acc0;
          tc_mma_ts(tO(0), tp + (uint32_t)(kk * 8), dadv(v, kk * 16 * 128), IO, acc);
          tc_mma_ts(tO(1), tp + (uint32_t)(64 + kk * 8), dadv(v, (4 + kk) * 16 * 128), IO, acc);
        }
        // one commit serves both: the V stage is free and O_0 / O_1 hold P_g V
        tc_commit(&v_empty[g % NFV]);
        return true;
      };
      bool ok = true;
      int g = 0;  // key tiles computed so far
      for (int i = item_of(0); i < n_items && ok; i = item_of(++it)) {
        const int qb = attn_item(i, nqb, nh, n_seq, head_major).qb;
        if (!mbar_wait(q_full, (uint32_t)(it & 1), abort_flag)) {
          ok = false;
          break;
        }
        // S_g goes into the columns of S_{g-2} / P_{g-2}, whose O += P V was
        // issued before it (one thread's MMAs run in order)
        for (int j = 0; j <= qb; ++j, ++g) {
          const int s = g % NFK, b = g & 1;
          if (!mbar_wait(&k_full[s], (uint32_t)((g / NFK) & 1), abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t kd = dadv(dK, s * NC * CH);
          const uint32_t ts = tS(b);
#pragma unroll
          for (int c = 0; c < NC; ++c)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc_mma(ts, dadv(dQ, c * CH + k * 32), dadv(kd, c * CH + k * 32), IS, (c | k) != 0);
          tc_commit(&s_full[b]);
          tc_commit(&k_empty[s]);  // K_g is read by S_g only
          if (PERSIST && j == qb) tc_commit(q_empty);  // the item's last S: Q may be replaced once it is done
          if (j >= 1 && !issue_pv(g - 1, j == 1)) {
            ok = false;
            break;
          }
        }
        if (ok) ok = issue_pv(g - 1, qb == 0);
      }
      if (!ok) {
        *abort_flag = 1;
        atomicCAS(&g_attn_error, 0, 12);
      }
    }
  } else {
    // Softmax warps 2..9: for each item this thread owns query row r (TMEM lane
    // quarter warp % 4) for keys 64 half .. 64 half + 63 of every key tile,
    // with its own running max m, sum l and accumulator O_half; the two
    // halves of a row merge once at the item's end.
    const int qw = warp & 3, half = (warp - 2) >> 2;
    const int r = qw * 32 + lane;
    const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
    bool ok = true;
    int g = 0;  // key tiles seen so far
    int it = 0;
    for (int i = item_of(0); i < n_items && ok; i = item_of(++it)) {
      // only the query tile is live through the key-tile loop; the head and
      // sequence are derived again for the epilogue (register pressure: a
      // 320-thread CTA gets at most 168 registers per thread)
      const int qb = attn_item(i, nqb, nh, n_seq, head_major).qb;
      const int q0 = qb * 128;
      const int qpos = q0 + r;  // position inside the sequence
      float m_used = -INFINITY, l = 0.f;  // exponent base of this half and the sum relative to it
      for (int j = 0; j <= qb; ++j, ++g) {
        const int b = g & 1;
        const uint32_t u = (uint32_t)(g >> 1);
        // warp-uniform outcome: the TMEM loads below are warp-collective
        if (!__all_sync(0xffffffffu, mbar_wait(&s_full[b], u & 1, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[2][32];
        tmem_ld32_nw(tS(b) + lane_off + half * 64, sr[0]);
        tmem_ld32_nw(tS(b) + lane_off + half * 64 + 32, sr[1]);
        tmem_wait_ld2(sr[0], sr[1]);
        const int kbase = 128 * j + 64 * half;
        // only the diagonal tile and a tile crossing the sequence end need
        // masking; the rest of the tile's row work is instantiated twice, so
        // that the common unmasked tiles carry no per-element mask code
        auto row_tile = [&](auto masked) -> bool {
          // raw scores (masked ones -inf); the exp2-domain scale enters once, in
          // the max and in one FMA per score before ex2 (scale_log2 > 0)
          float sv[64];
          if constexpr (decltype(masked)::value) {
#pragma unroll
            for (int k = 0; k < 64; ++k) {
              const int key = kbase + k;
              sv[k] = (key > qpos || key >= S) ? -INFINITY : __uint_as_float(sr[k >> 5][k & 31]);
            }
          } else {
#pragma unroll
            for (int k = 0; k < 64; ++k) sv[k] = __uint_as_float(sr[k >> 5][k & 31]);
          }
          // eight independent chains instead of one 64-long dependency chain
          float mx8[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) mx8[k] = sv[k];
#pragma unroll
          for (int k = 8; k < 64; ++k) mx8[k & 7] = fmaxf(mx8[k & 7], sv[k]);
          const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                 fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * scale_log2;
          // lazy base: move it only when this tile's max exceeds it by more than
          // 2^8 (always on the first tile with a key); P = 2^(s - base) <= 2^8
          const bool move = mx > m_used + 8.f;
          const float alpha = move ? ex2(m_used - mx) : 1.f;  // 0 when m_used = -inf
          if (move) {
            m_used = mx;
            l *= alpha;
          }
          // O_half of rows whose base moved is rescaled once the previous P V has
          // landed in it (warp-collective TMEM traffic: the whole warp joins)
          if (j > 0 && __any_sync(0xffffffffu, move)) {
            if (!__all_sync(0xffffffffu, mbar_wait(&v_empty[(g - 1) % NFV], (uint32_t)(((g - 1) / NFV) & 1),
                                                   abort_flag)))
              return false;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < HD / 32; ++c) {
              float t[32];
              tmem_ld32(tO(half) + lane_off + c * 32, t);
#pragma unroll
              for (int k = 0; k < 32; ++k) t[k] *= alpha;
              tmem_st32(tO(half) + lane_off + c * 32, t);
            }
          }
          const float base = m_used == -INFINITY ? 0.f : m_used;
          // paired FP32 arithmetic (two lanes per instruction, each rounded as
          // the scalar form) for the exponent arguments and the sums
          const float2 sc2 = make_float2(scale_log2, scale_log2), nb2 = make_float2(-base, -base);
          float2 sum2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                            make_float2(0.f, 0.f)};
          uint32_t pw[32];
#pragma unroll
          for (int k = 0; k < 64; k += 2) {
            const float2 e = __ffma2_rn(make_float2(sv[k], sv[k + 1]), sc2, nb2);
            const float2 p = make_float2(ex2(e.x), ex2(e.y));
            sum2[(k >> 1) & 3] = __fadd2_rn(sum2[(k >> 1) & 3], p);
            pw[k >> 1] = pack2(p.x, p.y);
          }
          const float2 s01 = __fadd2_rn(sum2[0], sum2[1]), s23 = __fadd2_rn(sum2[2], sum2[3]);
          const float2 st = __fadd2_rn(s01, s23);
          l += st.x + st.y;
          // P_g (BF16 pairs) over this half's first 32 columns of S_g, which this
          // thread has already read: the A operand of the next O += P V
          tmem_st32u(tS(b) + lane_off + half * 64, pw);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&p_full[b]);
          return true;
        };
        const bool need_mask = (kbase + 63 > q0) || (kbase + 64 > S);
        if (!(need_mask ? row_tile(std::true_type{}) : row_tile(std::false_type{}))) {
          ok = false;
          break;
        }
      }
      if (!ok) break;
      const float m_old = m_used;
      // merge the two halves of the row: m = max(m_0, m_1), c_h = 2^(m_h - m),
      // l = l_0 c_0 + l_1 c_1, O = (O_0 c_0 + O_1 c_1) / l; each half writes
      // half of the hd columns, once the item's last O += P V has landed
      ok = __all_sync(0xffffffffu,
                      mbar_wait(&v_empty[(g - 1) % NFV], (uint32_t)(((g - 1) / NFV) & 1), abort_flag));
      if (ok) {
        fin[(half * 2) * 128 + r] = m_old;
        fin[(half * 2 + 1) * 128 + r] = l;
        mbar_arrive(fin_ready);
        ok = __all_sync(0xffffffffu, mbar_wait(fin_ready, (uint32_t)(it & 1), abort_flag));
      }
      if (!ok) break;
      tc_fence_after();
      const float m0 = fin[r], l0 = fin[128 + r], m1 = fin[256 + r], l1 = fin[384 + r];
      float m = fmaxf(m0, m1);
      if (m == -INFINITY) m = 0.f;  // a row past the sequence end: nothing is stored
      const float c0 = ex2(m0 - m), c1 = ex2(m1 - m);
      const float lt = l0 * c0 + l1 * c1;
      const float inv = 1.f / lt;
      const float f0 = c0 * inv, f1 = c1 * inv;
      const bool valid = qpos < S;
      const AttnItem w = attn_item(i, nqb, nh, n_seq, head_major);
      const int h = w.h, row0 = w.n * S;
      bf16* orow = o + ((int64_t)row0 + qpos) * ((int64_t)nh * HD) + (int64_t)h * HD + half * (HD / 2);
#pragma unroll
      for (int c = 0; c < HD / 64; ++c) {
        float a0[32], a1[32];
        tmem_ld32(tO(0) + lane_off + half * (HD / 2) + c * 32, a0);
        tmem_ld32(tO(1) + lane_off + half * (HD / 2) + c * 32, a1);
        if (valid) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = a0[8 * k + e] * f0 + a1[8 * k + e] * f1;
            reinterpret_cast<uint4*>(orow + c * 32)[k] =
                make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
          }
        }
      }
      // O has been read: the next item's first O += P V may overwrite it
      if (PERSIST) {
        tc_fence_before();
        mbar_arrive(o_free);
      }
      if (valid && half == 0) lse[(int64_t)h * T + row0 + qpos] = (m + log2f(lt)) * 0.6931471805599453f;
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      atomicCAS(&g_attn_error, 0, 13);
    }
  }

  if (warp == 0 && lane < 2 && *abort_flag) {
    const long long t0 = clock64();
    if (lane == 0 && q_inflight)
      while (!mbar_test(q_full, q_par) && clock64() - t0 < kWaitCycles) {
      }
    uint64_t* full = lane == 0 ? k_full : v_full;
    for (int s2 = 0; s2 < (lane == 0 ? NFK : NFV); ++s2)
      if (x_inflight & (1u << s2))
        while (!mbar_test(&full[s2], (x_par >> s2) & 1) && clock64() - t0 < kWaitCycles) {
        }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
  }
}

// ---------------------------------------------------------------------------
// Backward, as two kernels that share no accumulator (so no atomics and no
// FP32 dQ buffer).  delta[h][t] = rowsum(dO o O) is computed before them.
// Both work on 128 x 128 tiles: inside these kernels a tcgen05.mma costs
// about the same at N = 64 as at N = 128, so the wider tile halves the MMA
// count per unit of work.  TMEM holds one tile's scores (single-buffered); the
// row warps write P / dS back over the scores they have read, as BF16, and the
// accumulating MMAs read them from there as their A operand.  The MMA warp
// issues the accumulation of tile i before the scores of tile i + 1 into the
// same columns; tcgen05.mma operations of one thread run in issue order.
//
// attn_bwd_kv_k: one CTA per (128 keys, kv head, sequence), grid ordered
// longest work first; it loops over the query heads of its group and, per
// head, over 128-query tiles from the diagonal on.  Per tile:
//   MMA   S^T = K Q^T and dP^T = V dO^T (K, V resident in shared memory; Q, dO
//         tiles in a 2-stage TMA ring);
//   rows  (8 warps: key rows by TMEM lane quarter, query halves) P^T =
//         exp2(S^T scale log2e - lse log2e) with the causal mask where needed,
//         dS^T = P^T (dP^T - delta), written as BF16 over S^T / dP^T;
//   MMA   dV += P^T dO and dK += dS^T Q (dO, Q as MN-major operands).
// TMEM: S^T | dP^T | dV | dK.
//
// attn_bwd_q_k: one CTA per (128 queries, query head, sequence), longest work
// first, looping over 128-key tiles up to the diagonal.  Q and dO are written
// into TMEM once by the row warps and are the A operands of S = Q K^T and
// dP = dO V^T; the rows form P as soon as S lands (S's columns then take the
// next tile's S), then dS = P (dP - delta) written over dP; dQ += dS K reads
// dS from TMEM and K (MN-major) from shared memory; dQ scale leaves as BF16.
// TMEM: Q | dO | S | dP | dQ.  Every wait is bounded.
constexpr int CH64 = 8192;  // one 64-column chunk of a 64-row box (64 rows x 128 B)
constexpr int NQT = 2;      // Q / dO tile stages of the dK/dV kernel
constexpr int NKT = 3;      // K / V tile stages of the dQ kernel

template <int HD>
__host__ __device__ constexpr int kv_smem_bytes() {
  return (HD / 64) * CH * (2 + 2 * NQT) + 2048 + 256 + 1024;
}
template <int HD>
__host__ __device__ constexpr int q_smem_bytes() {
  return (HD / 64) * CH * 2 * NKT + 256 + 1024;
}
static_assert(kv_smem_bytes<128>() <= 232448, "dK/dV kernel shared memory");
static_assert(q_smem_bytes<128>() <= 232448, "dQ kernel shared memory");

// P / dS columns of one 16-element K-step of a 128-wide tile written back by
// the two row halves: half h's 64 values occupy columns 64 h .. 64 h + 31.
__device__ __forceinline__ uint32_t pcol(int kk) { return (uint32_t)((kk >> 2) * 64 + (kk & 3) * 8); }

template <int HD>
__global__ void __launch_bounds__(ATTN_THREADS, 1)
    attn_bwd_kv_k(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo, int S,
                  int n_seq, int nh, int nkv, const float* __restrict__ lse, const float* __restrict__ delta,
                  float scale, float scale_log2, bf16* __restrict__ dqkv) {
  constexpr int NC = HD / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = sm;                  // [128 keys][HD]: NC chunks of 128 rows
  uint8_t* sV = sK + NC * CH;
  uint8_t* sQ = sV + NC * CH;        // NQT stages of [128 q][HD]
  uint8_t* sO = sQ + NQT * NC * CH;  // dO, the same
  float* ls = reinterpret_cast<float*>(sO + NQT * NC * CH);  // [2][128] -lse log2e of the tile
  float* dls = ls + 256;                                      // [2][128] -delta of the tile
  uint64_t* bars = reinterpret_cast<uint64_t*>(dls + 256);
  uint64_t* kv_full = bars;
  uint64_t* qf = bars + 1;           // [NQT] Q / dO tile loaded
  uint64_t* qe = qf + NQT;           // [NQT] Q / dO tile consumed
  uint64_t* s1_full = qe + NQT;      // S^T in TMEM
  uint64_t* s2_full = s1_full + 1;   // dP^T in TMEM
  uint64_t* p1_full = s2_full + 1;   // P^T written back over S^T
  uint64_t* p2_full = p1_full + 1;   // dS^T written back over dP^T
  uint64_t* ld_ready = p2_full + 1;  // [2] lse / delta staged
  uint64_t* acc_full = ld_ready + 2; // dK, dV complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per_kb = nkv * n_seq;
  const int kb = (int)(blockIdx.x / per_kb);  // key tile 0 has the most query tiles
  const int g = (int)(blockIdx.x % per_kb) / n_seq, n = (int)(blockIdx.x % n_seq);
  const int grp = nh / nkv;
  const int nqb = (S + 127) / 128;
  const int per_head = nqb - kb;
  const int iters = grp * per_head;
  const int k0 = kb * 128;
  const int row0 = n * S;
  const int64_t T = (int64_t)n_seq * S;
  const int64_t ld = (int64_t)(nh + 2 * nkv) * HD;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < NQT; ++i) {
      mbar_init(&qf[i], 1);
      mbar_init(&qe[i], 1);
    }
    mbar_init(s1_full, 1);
    mbar_init(s2_full, 1);
    mbar_init(p1_full, 256);
    mbar_init(p2_full, 256);
    for (int i = 0; i < 2; ++i) mbar_init(&ld_ready[i], 256);
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tq) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tdo) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                 "r"(512));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tSt = tmem, tdPt = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + HD;
  bool kv_inflight = false;
  uint32_t q_inflight = 0, q_par = 0;

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      mbar_expect_tx(kv_full, 2 * NC * CH);
      for (int c = 0; c < NC; ++c)
        for (int hf = 0; hf < 2; ++hf) {
          tma_load(&tq, kv_full, sK + c * CH + hf * CH64, (nh + g) * HD + 64 * c, row0 + k0 + 64 * hf);
          tma_load(&tq, kv_full, sV + c * CH + hf * CH64, (nh + nkv + g) * HD + 64 * c, row0 + k0 + 64 * hf);
        }
      kv_inflight = true;
      for (int i = 0; i < iters && ok; ++i) {
        const int st = i % NQT;
        const uint32_t u = (uint32_t)(i / NQT);
        const int h = g * grp + i / per_head, q0 = (kb + i % per_head) * 128;
        if (!mbar_wait(&qe[st], (u & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        mbar_expect_tx(&qf[st], 2 * NC * CH);
        for (int c = 0; c < NC; ++c)
          for (int hf = 0; hf < 2; ++hf) {
            tma_load(&tq, &qf[st], sQ + (st * NC + c) * CH + hf * CH64, h * HD + 64 * c, row0 + q0 + 64 * hf);
            tma_load(&tdo, &qf[st], sO + (st * NC + c) * CH + hf * CH64, h * HD + 64 * c, row0 + q0 + 64 * hf);
          }
        q_inflight |= 1u << st;
        q_par = (q_par & ~(1u << st)) | ((u & 1) << st);
      }
      if (!ok) {
        *abort_flag = 1;
        atomicCAS(&g_attn_error, 0, 21);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = mbar_wait(kv_full, 0, abort_flag);
      constexpr uint32_t I_S = idesc(128, 128, false, false);  // S^T, dP^T: both operands K-major over hd
      constexpr uint32_t I_G = idesc(128, HD, false, true);    // dV, dK: A from TMEM, B = dO / Q MN-major
      const uint64_t dK = sdesc(su32(sK), 16, 1024), dV = sdesc(su32(sV), 16, 1024);
      const uint64_t dQ = sdesc(su32(sQ), 16, 1024), dO = sdesc(su32(sO), 16, 1024);
      const uint64_t dQm = sdesc(su32(sQ), CH, 1024), dOm = sdesc(su32(sO), CH, 1024);
      // Per tile i the MMAs go out as dV(i), S^T(i+1), dK(i), dP^T(i+1): dV
      // waits only for P^T, dK for dS^T, and the next tile's S^T is in flight
      // while the rows form dS^T of tile i; S^T(i+1) overwrites the P^T(i)
      // that dV(i) read before it, dP^T(i+1) the dS^T(i) dK(i) read.
      auto issue_st = [&](int i) -> bool {  // S^T = K Q^T
        const int st = i % NQT;
        if (!mbar_wait(&qf[st], (uint32_t)((i / NQT) & 1), abort_flag)) return false;
        tc_fence_after();
        const uint64_t q = dadv(dQ, st * NC * CH);
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const uint32_t off = (ks >> 2) * CH + (ks & 3) * 32;
          tc_mma(tSt, dadv(dK, off), dadv(q, off), I_S, ks != 0);
        }
        tc_commit(s1_full);
        return true;
      };
      auto issue_dpt = [&](int i) {  // dP^T = V dO^T (its Q / dO stage was waited for by issue_st)
        const uint64_t o = dadv(dO, (i % NQT) * NC * CH);
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const uint32_t off = (ks >> 2) * CH + (ks & 3) * 32;
          tc_mma(tdPt, dadv(dV, off), dadv(o, off), I_S, ks != 0);
        }
        tc_commit(s2_full);
      };
      auto issue_dv = [&](int i) -> bool {  // dV += P^T dO
        if (!mbar_wait(p1_full, (uint32_t)(i & 1), abort_flag)) return false;
        tc_fence_after();
        const uint64_t om = dadv(dOm, (i % NQT) * NC * CH);
        const uint32_t acc0 = i > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) tc_mma_ts(tdV, tSt + pcol(kk), dadv(om, kk * 2048), I_G, kk > 0 ? 1u : acc0);
        return true;
      };
      auto issue_dk = [&](int i) -> bool {  // dK += dS^T Q; the Q / dO stage is then free
        if (!mbar_wait(p2_full, (uint32_t)(i & 1), abort_flag)) return false;
        tc_fence_after();
        const int st = i % NQT;
        const uint64_t qm = dadv(dQm, st * NC * CH);
        const uint32_t acc0 = i > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) tc_mma_ts(tdK, tdPt + pcol(kk), dadv(qm, kk * 2048), I_G, kk > 0 ? 1u : acc0);
        tc_commit(&qe[st]);
        return true;
      };
      if (ok) ok = issue_st(0);
      if (ok) issue_dpt(0);
      for (int i = 0; i < iters && ok; ++i) {
        const bool more = i + 1 < iters;
        if (!issue_dv(i) || (more && !issue_st(i + 1)) || !issue_dk(i)) {
          ok = false;
          break;
        }
        if (more) issue_dpt(i + 1);
      }
      if (ok) tc_commit(acc_full);
      if (!ok) {
        *abort_flag = 1;
        atomicCAS(&g_attn_error, 0, 22);
      }
    }
  } else {
    // Row warps 2..9: warp w reads TMEM lanes 32 (w % 4) .. +31 (key rows);
    // warps 2..5 take queries 0..63 of the tile, warps 6..9 queries 64..127
    // (and at the end dK, dV respectively).
    const int qw = warp & 3, half = (warp - 2) >> 2;
    const int r = qw * 32 + lane;  // key row of S^T, dP^T, dV, dK
    const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
    const int key = k0 + r;
    const int t = threadIdx.x - 64;  // staging entry: lse (t < 128) or delta (t >= 128) of query t % 128
    float* stage = t < 128 ? ls : dls;
    auto fetch = [&](int i) -> float {
      const int h = g * grp + i / per_head, q = (kb + i % per_head) * 128 + (t & 127);
      if (q >= S) return 0.f;
      const int64_t idx = (int64_t)h * T + row0 + q;
      return t < 128 ? -(lse[idx] * 1.4426950408889634f) : -delta[idx];  // staged negated
    };
    bool ok = true;
    float nxt = fetch(0);  // one tile ahead, so the global load latency hides behind a tile
    for (int i = 0; i < iters; ++i) {
      const int b = i & 1;
      const uint32_t u = (uint32_t)(i >> 1);
      const int q0 = (kb + i % per_head) * 128;
      // Buffer b was last read in tile i-2; every thread finished that before
      // it arrived on ld_ready for tile i-1, which this thread has waited for.
      stage[b * 128 + (t & 127)] = nxt;
      mbar_arrive(&ld_ready[b]);
      if (i + 1 < iters) nxt = fetch(i + 1);
      bool w = mbar_wait(&ld_ready[b], u & 1, abort_flag);
      if (w) w = mbar_wait(s1_full, (uint32_t)(i & 1), abort_flag);
      if (!__all_sync(0xffffffffu, w)) {  // warp-uniform: the TMEM loads below are warp-collective
        ok = false;
        break;
      }
      tc_fence_after();
      const bool need_mask = (q0 < k0 + 127) || (q0 + 128 > S);
      const float4* lrow = reinterpret_cast<const float4*>(ls + b * 128 + half * 64);
      const float4* drow = reinterpret_cast<const float4*>(dls + b * 128 + half * 64);
      // phase 1: P^T from S^T, back over the first 32 S^T columns this thread read
      float p[64];
      {
        uint32_t sv[2][32];
        tmem_ld32_nw(tSt + lane_off + half * 64, sv[0]);
        tmem_ld32_nw(tSt + lane_off + half * 64 + 32, sv[1]);
        tmem_wait_ld2(sv[0], sv[1]);
        uint32_t pw[32];
        const float2 sc2 = make_float2(scale_log2, scale_log2);
        // two instantiations, so that tiles without masked entries (all but
        // the diagonal and the sequence end) carry no per-element mask code
        auto exps = [&](auto masked) {
#pragma unroll
          for (int e4 = 0; e4 < 16; ++e4) {
            const float4 l4 = lrow[e4];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {  // two paired FMAs: exponent arguments of 4 columns
              const int e = e4 * 4 + 2 * hh;
              const float2 arg = __ffma2_rn(make_float2(__uint_as_float(sv[e >> 5][e & 31]),
                                                        __uint_as_float(sv[(e + 1) >> 5][(e + 1) & 31])),
                                            sc2, hh ? make_float2(l4.z, l4.w) : make_float2(l4.x, l4.y));
              float pa = ex2(arg.x), pb = ex2(arg.y);
              if constexpr (decltype(masked)::value) {
                const int q = q0 + half * 64 + e;
                if (q < key || q >= S) pa = 0.f;
                if (q + 1 < key || q + 1 >= S) pb = 0.f;
              }
              p[e] = pa;
              p[e + 1] = pb;
            }
            pw[2 * e4] = pack2(p[4 * e4], p[4 * e4 + 1]);
            pw[2 * e4 + 1] = pack2(p[4 * e4 + 2], p[4 * e4 + 3]);
          }
        };
        if (need_mask)
          exps(std::true_type{});
        else
          exps(std::false_type{});
        tmem_st32u(tSt + lane_off + half * 64, pw);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p1_full);
      }
      // phase 2: dS^T = P^T (dP^T - delta), back over the first 32 dP^T columns
      if (!__all_sync(0xffffffffu, mbar_wait(s2_full, (uint32_t)(i & 1), abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        uint32_t dp[2][32];
        tmem_ld32_nw(tdPt + lane_off + half * 64, dp[0]);
        tmem_ld32_nw(tdPt + lane_off + half * 64 + 32, dp[1]);
        tmem_wait_ld2(dp[0], dp[1]);
        uint32_t dw[32];
#pragma unroll
        for (int e4 = 0; e4 < 16; ++e4) {
          const float4 d4 = drow[e4];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {  // dS = P (dP - delta), two columns per paired op
            const int e = e4 * 4 + 2 * hh;
            const float2 dd = __fadd2_rn(make_float2(__uint_as_float(dp[e >> 5][e & 31]),
                                                     __uint_as_float(dp[(e + 1) >> 5][(e + 1) & 31])),
                                         hh ? make_float2(d4.z, d4.w) : make_float2(d4.x, d4.y));
            const float2 v = __fmul2_rn(make_float2(p[e], p[e + 1]), dd);
            dw[2 * e4 + hh] = pack2(v.x, v.y);
          }
        }
        tmem_st32u(tdPt + lane_off + half * 64, dw);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p2_full);
      }
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, abort_flag));
    if (ok) {
      // warps 2..5: dK (scaled) of their key rows; warps 6..9: dV.  The TMEM
      // loads are warp-collective: every lane loads, only rows inside the
      // sequence store.
      tc_fence_after();
      const bool valid = key < S;
      const float f = half == 0 ? scale : 1.f;
      const uint32_t tacc = half == 0 ? tdK : tdV;
      bf16* row = dqkv + ((int64_t)row0 + (valid ? key : 0)) * ld + (int64_t)(nh + half * nkv + g) * HD;
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        float v[32];
        tmem_ld32(tacc + lane_off + c * 32, v);
        if (valid) {
#pragma unroll
          for (int i4 = 0; i4 < 4; ++i4)
            reinterpret_cast<uint4*>(row + c * 32)[i4] =
                make_uint4(pack2(v[8 * i4] * f, v[8 * i4 + 1] * f), pack2(v[8 * i4 + 2] * f, v[8 * i4 + 3] * f),
                           pack2(v[8 * i4 + 4] * f, v[8 * i4 + 5] * f), pack2(v[8 * i4 + 6] * f, v[8 * i4 + 7] * f));
        }
      }
    } else if (lane == 0) {
      *abort_flag = 1;
      atomicCAS(&g_attn_error, 0, 23);
    }
  }

  if (warp == 0 && lane == 0 && *abort_flag) {
    const long long t0 = clock64();
    if (kv_inflight)
      while (!mbar_test(kv_full, 0) && clock64() - t0 < kWaitCycles) {
      }
    for (int s2 = 0; s2 < NQT; ++s2)
      if (q_inflight & (1u << s2))
        while (!mbar_test(&qf[s2], (q_par >> s2) & 1) && clock64() - t0 < kWaitCycles) {
        }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
  }
}

template <int HD>
__global__ void __launch_bounds__(ATTN_THREADS, 1)
    attn_bwd_q_k(const __grid_constant__ CUtensorMap tq, const bf16* __restrict__ qkv, const bf16* __restrict__ dout,
                 int S, int n_seq, int nh, int nkv, const float* __restrict__ lse, const float* __restrict__ delta,
                 float scale, float scale_log2, bf16* __restrict__ dqkv) {
  constexpr int NC = HD / 64;
  constexpr int QC = HD / 2;  // TMEM columns of one BF16 row of hd values
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = sm;                  // NKT stages of [128 keys][HD]
  uint8_t* sV = sK + NKT * NC * CH;  // NKT stages of [128 keys][HD]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + NKT * NC * CH);
  uint64_t* q_ready = bars;         // Q, dO written to TMEM by the rows
  uint64_t* kvf = bars + 1;         // [NKT]
  uint64_t* kve = kvf + NKT;        // [NKT]
  uint64_t* s1_full = kve + NKT;    // S in TMEM
  uint64_t* s2_full = s1_full + 1;  // dP in TMEM
  uint64_t* ps_free = s2_full + 1;  // the rows have read S
  uint64_t* p_full = ps_free + 1;   // dS written back over dP
  uint64_t* acc_full = p_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqb = (S + 127) / 128;
  const int per_qb = nh * n_seq;
  const int qb = nqb - 1 - (int)(blockIdx.x / per_qb);  // the last query tile has the most keys
  const int h = (int)(blockIdx.x % per_qb) / n_seq, n = (int)(blockIdx.x % n_seq);
  const int kh = h / (nh / nkv);
  const int q0 = qb * 128;
  const int nkt = qb + 1;  // key tiles 0 .. qb (the last one holds the diagonal)
  const int row0 = n * S;
  const int64_t T = (int64_t)n_seq * S;
  const int64_t ld = (int64_t)(nh + 2 * nkv) * HD;

  if (threadIdx.x == 0) {
    mbar_init(q_ready, 256);
    for (int i = 0; i < NKT; ++i) {
      mbar_init(&kvf[i], 1);
      mbar_init(&kve[i], 1);
    }
    mbar_init(s1_full, 1);
    mbar_init(s2_full, 1);
    mbar_init(ps_free, 256);
    mbar_init(p_full, 256);
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tq) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                 "r"(512));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tQ = tmem, tdO = tmem + QC, tS = tmem + 2 * QC, tP = tS + 128, tdQ = tS + 256;
  uint32_t kv_inflight = 0, kv_par = 0;

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      for (int j = 0; j < nkt && ok; ++j) {
        const int st = j % NKT;
        const uint32_t u = (uint32_t)(j / NKT);
        if (!mbar_wait(&kve[st], (u & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        mbar_expect_tx(&kvf[st], 2 * NC * CH);
        for (int c = 0; c < NC; ++c)
          for (int hf = 0; hf < 2; ++hf) {
            tma_load(&tq, &kvf[st], sK + (st * NC + c) * CH + hf * CH64, (nh + kh) * HD + 64 * c,
                     row0 + 128 * j + 64 * hf);
            tma_load(&tq, &kvf[st], sV + (st * NC + c) * CH + hf * CH64, (nh + nkv + kh) * HD + 64 * c,
                     row0 + 128 * j + 64 * hf);
          }
        kv_inflight |= 1u << st;
        kv_par = (kv_par & ~(1u << st)) | ((u & 1) << st);
      }
      if (!ok) {
        *abort_flag = 1;
        atomicCAS(&g_attn_error, 0, 24);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = mbar_wait(q_ready, 0, abort_flag);
      constexpr uint32_t I_S = idesc(128, 128, false, false);  // S, dP: A (Q, dO) in TMEM, B K-major over hd
      constexpr uint32_t I_G = idesc(128, HD, false, true);    // dQ: A (dS) in TMEM, B = K as MN-major
      const uint64_t dK = sdesc(su32(sK), 16, 1024), dV = sdesc(su32(sV), 16, 1024);
      const uint64_t dKm = sdesc(su32(sK), CH, 1024);
      // Per tile j: S(j+1) as soon as the rows have read S(j); then dQ(j),
      // which reads dS(j) from the dP columns, then dP(j+1) over them.
      auto issue_s = [&](int j) -> bool {  // S = Q K^T
        const int st = j % NKT;
        if (!mbar_wait(&kvf[st], (uint32_t)((j / NKT) & 1), abort_flag)) return false;
        if (j > 0 && !mbar_wait(ps_free, (uint32_t)((j - 1) & 1), abort_flag)) return false;
        tc_fence_after();
        const uint64_t kd = dadv(dK, st * NC * CH);
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks)
          tc_mma_ts(tS, tQ + 8 * ks, dadv(kd, (ks >> 2) * CH + (ks & 3) * 32), I_S, ks != 0);
        tc_commit(s1_full);
        return true;
      };
      auto issue_dp = [&](int j) {  // dP = dO V^T (its K / V stage was waited for by issue_s)
        const uint64_t vd = dadv(dV, (j % NKT) * NC * CH);
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks)
          tc_mma_ts(tP, tdO + 8 * ks, dadv(vd, (ks >> 2) * CH + (ks & 3) * 32), I_S, ks != 0);
        tc_commit(s2_full);
      };
      auto issue_g = [&](int j) -> bool {  // dQ += dS K; the K / V stage is then free
        const int st = j % NKT;
        if (!mbar_wait(p_full, (uint32_t)(j & 1), abort_flag)) return false;
        tc_fence_after();
        const uint64_t km = dadv(dKm, st * NC * CH);
        const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_ts(tdQ, tP + pcol(kk), dadv(km, kk * 2048), I_G, kk > 0 ? 1u : acc0);
        tc_commit(&kve[st]);
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok) issue_dp(0);
      for (int j = 0; j < nkt && ok; ++j) {
        const bool more = j + 1 < nkt;
        if ((more && !issue_s(j + 1)) || !issue_g(j)) {
          ok = false;
          break;
        }
        if (more) issue_dp(j + 1);
      }
      if (ok) tc_commit(acc_full);
      if (!ok) {
        *abort_flag = 1;
        atomicCAS(&g_attn_error, 0, 25);
      }
    }
  } else {
    // Row warps 2..9: query rows by TMEM lane quarter; warps 2..5 own keys
    // 0..63 of a tile (and the first half of Q, dO, dQ's hd columns), warps
    // 6..9 keys 64..127 (and the second half).
    const int qw = warp & 3, half = (warp - 2) >> 2;
    const int r = qw * 32 + lane;  // query row
    const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
    const int q = q0 + r;
    const bool valid = q < S;
    const int64_t li = (int64_t)h * T + row0 + (valid ? q : 0);
    const float lse2 = valid ? lse[li] * 1.4426950408889634f : 0.f;
    const float dl = valid ? delta[li] : 0.f;
    // this row's half of Q and of dO into TMEM (the A operands of S and dP)
    {
      const uint4* qs = reinterpret_cast<const uint4*>(qkv + ((int64_t)row0 + (valid ? q : 0)) * ld +
                                                         (int64_t)h * HD + half * (HD / 2));
      const uint4* os = reinterpret_cast<const uint4*>(dout + ((int64_t)row0 + (valid ? q : 0)) * ((int64_t)nh * HD) +
                                                         (int64_t)h * HD + half * (HD / 2));
      uint32_t qv[QC / 2], ov[QC / 2];
#pragma unroll
      for (int i = 0; i < QC / 8; ++i) {
        const uint4 a = valid ? qs[i] : make_uint4(0, 0, 0, 0);
        const uint4 c = valid ? os[i] : make_uint4(0, 0, 0, 0);
        qv[4 * i] = a.x; qv[4 * i + 1] = a.y; qv[4 * i + 2] = a.z; qv[4 * i + 3] = a.w;
        ov[4 * i] = c.x; ov[4 * i + 1] = c.y; ov[4 * i + 2] = c.z; ov[4 * i + 3] = c.w;
      }
      if constexpr (QC / 2 == 32) {
        tmem_st32u(tQ + lane_off + half * (QC / 2), qv);
        tmem_st32u(tdO + lane_off + half * (QC / 2), ov);
      } else {
        tmem_st16(tQ + lane_off + half * (QC / 2), qv);
        tmem_st16(tdO + lane_off + half * (QC / 2), ov);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(q_ready);
    }
    bool ok = true;
    for (int j = 0; j < nkt; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait(s1_full, (uint32_t)(j & 1), abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int k0 = 128 * j + 64 * half;  // first key of this thread's 64 columns
      const bool need_mask = (k0 + 63 > q0) || (k0 + 64 > S);
      // phase 1: P from S; then S's columns are free for the next tile
      float p[64];
      {
        uint32_t sv[2][32];
        tmem_ld32_nw(tS + lane_off + half * 64, sv[0]);
        tmem_ld32_nw(tS + lane_off + half * 64 + 32, sv[1]);
        tmem_wait_ld2(sv[0], sv[1]);
        const float2 sc2 = make_float2(scale_log2, scale_log2), nl2 = make_float2(-lse2, -lse2);
        // two instantiations: tiles without masked entries carry no mask code
        auto exps = [&](auto masked) {
#pragma unroll
          for (int e = 0; e < 64; e += 2) {
            const float2 arg = __ffma2_rn(make_float2(__uint_as_float(sv[e >> 5][e & 31]),
                                                      __uint_as_float(sv[(e + 1) >> 5][(e + 1) & 31])),
                                          sc2, nl2);
            float pa = ex2(arg.x), pb = ex2(arg.y);
            if constexpr (decltype(masked)::value) {
              const int key = k0 + e;
              if (key > q || key >= S) pa = 0.f;
              if (key + 1 > q || key + 1 >= S) pb = 0.f;
            }
            p[e] = pa;
            p[e + 1] = pb;
          }
        };
        if (need_mask)
          exps(std::true_type{});
        else
          exps(std::false_type{});
        tc_fence_before();
        mbar_arrive(ps_free);
      }
      // phase 2: dS = P (dP - delta), back over the first 32 dP columns this thread read
      if (!__all_sync(0xffffffffu, mbar_wait(s2_full, (uint32_t)(j & 1), abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        uint32_t dp[2][32];
        tmem_ld32_nw(tP + lane_off + half * 64, dp[0]);
        tmem_ld32_nw(tP + lane_off + half * 64 + 32, dp[1]);
        tmem_wait_ld2(dp[0], dp[1]);
        uint32_t dw[32];
        const float2 nd2 = make_float2(-dl, -dl);
#pragma unroll
        for (int e = 0; e < 64; e += 2) {
          const float2 dd = __fadd2_rn(make_float2(__uint_as_float(dp[e >> 5][e & 31]),
                                                   __uint_as_float(dp[(e + 1) >> 5][(e + 1) & 31])),
                                       nd2);
          const float2 v = __fmul2_rn(make_float2(p[e], p[e + 1]), dd);
          dw[e / 2] = pack2(v.x, v.y);
        }
        tmem_st32u(tP + lane_off + half * 64, dw);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p_full);
      }
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, abort_flag));
    if (ok) {
      tc_fence_after();
      bf16* row = dqkv + ((int64_t)row0 + (valid ? q : 0)) * ld + (int64_t)h * HD + half * (HD / 2);
#pragma unroll
      for (int c = 0; c < HD / 64; ++c) {
        float v[32];
        tmem_ld32(tdQ + lane_off + half * (HD / 2) + c * 32, v);
        if (valid) {
#pragma unroll
          for (int i4 = 0; i4 < 4; ++i4)
            reinterpret_cast<uint4*>(row + c * 32)[i4] = make_uint4(
                pack2(v[8 * i4] * scale, v[8 * i4 + 1] * scale), pack2(v[8 * i4 + 2] * scale, v[8 * i4 + 3] * scale),
                pack2(v[8 * i4 + 4] * scale, v[8 * i4 + 5] * scale), pack2(v[8 * i4 + 6] * scale, v[8 * i4 + 7] * scale));
        }
      }
    } else if (lane == 0) {
      *abort_flag = 1;
      atomicCAS(&g_attn_error, 0, 26);
    }
  }

  if (warp == 0 && lane == 0 && *abort_flag) {
    const long long t0 = clock64();
    for (int s2 = 0; s2 < NKT; ++s2)
      if (kv_inflight & (1u << s2))
        while (!mbar_test(&kvf[s2], (kv_par >> s2) & 1) && clock64() - t0 < kWaitCycles) {
        }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
  }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;
cudaError_t g_init = cudaSuccess;

void init_once() {
  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
    g_init = e != cudaSuccess ? e : cudaErrorNotSupported;
    return;
  }
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

// Forward launches with items of at most 64 key tiles (S <= 8192) use one
// persistent CTA per SM taking items longest first, so an item's set-up
// overlaps the previous item's epilogue (S = 4096: 972 against 887 TFLOP/s
// with one CTA per item, same box); longer items amortise their set-up, and
// get one CTA per item (the one-item instantiation has no cross-item waits),
// launched head-major so the CTAs running together share one KV head's keys
// and values in L2.
constexpr int kPersistTiles = 64;

template <int HD>
constexpr int smem_bytes() {
  return (HD / 64) * 16384 * (1 + NFK + NFV) + 2048 + 1024 + 256;
}

template <int HD>
cudaError_t launch(const bf16* qkv, int n_seq, int S, int nh, int nkv, bf16* o, float* lse, cudaStream_t s) {
  const int64_t ld = (int64_t)(nh + 2 * nkv) * HD;
  const int64_t T = (int64_t)n_seq * S;
  CUtensorMap m;
  const cuuint64_t dims[2] = {(cuuint64_t)ld, (cuuint64_t)T};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estr[2] = {1, 1};
  if (g_encode(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<bf16*>(qkv), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  constexpr int SM = smem_bytes<HD>();
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_tc_k<HD, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_fwd_tc_k<HD, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SM);
  if (e != cudaSuccess) return e;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
  const int64_t n_items = (int64_t)((S + 127) / 128) * nh * n_seq;
  if (n_items > 0x7fffffff) return cudaErrorInvalidValue;
  const int nqb = (S + 127) / 128;
  if (nqb <= kPersistTiles) {
    const int sms = gemm_num_sms();
    const int grid = (int)std::min<int64_t>(n_items, sms > 0 ? sms : 148);
    attn_fwd_tc_k<HD, true><<<grid, ATTN_THREADS, SM, s>>>(m, S, nh, nkv, n_seq, o, lse, scale_log2, 0);
  } else {
    attn_fwd_tc_k<HD, false><<<(int)n_items, ATTN_THREADS, SM, s>>>(m, S, nh, nkv, n_seq, o, lse, scale_log2, 1);
  }
  return cudaGetLastError();
}

bool make_map(CUtensorMap* m, const bf16* base, int64_t ld, int64_t rows, int box_rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)ld, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<bf16*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int HD>
cudaError_t launch_bwd(const bf16* qkv, const bf16* dout, const float* lse, const float* delta, int n_seq, int S,
                       int nh, int nkv, bf16* dqkv, cudaStream_t s) {
  const int64_t T = (int64_t)n_seq * S;
  CUtensorMap mq, mo;  // 64-row boxes: sub-tiles load as one box, 128-row tiles as two
  if (!make_map(&mq, qkv, (int64_t)(nh + 2 * nkv) * HD, T, 64) || !make_map(&mo, dout, (int64_t)nh * HD, T, 64))
    return cudaErrorInvalidValue;
  constexpr int SKV = kv_smem_bytes<HD>(), SQ = q_smem_bytes<HD>();
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_kv_k<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, SKV);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_bwd_q_k<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, SQ);
  if (e != cudaSuccess) return e;
  const float scale = 1.f / sqrtf((float)HD);
  const int64_t nqb = (S + 127) / 128;
  const int64_t gkv = nqb * nkv * n_seq, gq = nqb * nh * n_seq;
  if (gkv > 0x7fffffff || gq > 0x7fffffff) return cudaErrorInvalidValue;
  attn_bwd_kv_k<HD><<<(unsigned)gkv, ATTN_THREADS, SKV, s>>>(mq, mo, S, n_seq, nh, nkv, lse, delta, scale,
                                                         scale * 1.4426950408889634f, dqkv);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_bwd_q_k<HD><<<(unsigned)gq, ATTN_THREADS, SQ, s>>>(mq, qkv, dout, S, n_seq, nh, nkv, lse, delta, scale,
                                                          scale * 1.4426950408889634f, dqkv);
  return cudaGetLastError();
}

}  // namespace

// Tensor-core attention backward core: dQ, dK and dV into dqkv (BF16, the
// layout of qkv); delta[h][t] = rowsum(dO o O) must be precomputed.
cudaError_t attention_bwd_tc_core(const bf16* qkv, const bf16* dout, const float* lse, const float* delta,
                                  int n_seq, int S, int nh, int nkv, int hd, bf16* dqkv, cudaStream_t s) {
  std::call_once(g_once, init_once);
  if (g_init != cudaSuccess) return g_init;
  if (n_seq <= 0 || S <= 0) return cudaSuccess;
  if (nh % nkv || (int64_t)n_seq * S > 0x7fffffff) return cudaErrorInvalidValue;
  if ((reinterpret_cast<uintptr_t>(qkv) | reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(dqkv)) &
      15)
    return cudaErrorInvalidValue;
  if (hd == 64) return launch_bwd<64>(qkv, dout, lse, delta, n_seq, S, nh, nkv, dqkv, s);
  if (hd == 128) return launch_bwd<128>(qkv, dout, lse, delta, n_seq, S, nh, nkv, dqkv, s);
  return cudaErrorInvalidValue;
}

// Tensor-core attention forward (see the file comment).  Same contract as
// attention_fwd; requires hd in {64, 128}, 16-byte aligned qkv and o.
cudaError_t attention_fwd_tc(const bf16* qkv, int n_seq, int S, int nh, int nkv, int hd, bf16* o, float* lse,
                             cudaStream_t s) {
  std::call_once(g_once, init_once);
  if (g_init != cudaSuccess) return g_init;
  if (n_seq <= 0 || S <= 0) return cudaSuccess;
  if (nh % nkv || n_seq > 65535 || nh > 65535 || (int64_t)n_seq * S > 0x7fffffff) return cudaErrorInvalidValue;
  if ((reinterpret_cast<uintptr_t>(qkv) | reinterpret_cast<uintptr_t>(o)) & 15) return cudaErrorInvalidValue;
  if (hd == 64) return launch<64>(qkv, n_seq, S, nh, nkv, o, lse, s);
  if (hd == 128) return launch<128>(qkv, n_seq, S, nh, nkv, o, lse, s);
  return cudaErrorInvalidValue;
}

cudaError_t attention_error_read(int* code, int clear) {
  cudaError_t e = cudaMemcpyFromSymbol(code, g_attn_error, sizeof(int));
  if (e != cudaSuccess || !clear) return e;
  const int z = 0;
  return cudaMemcpyToSymbol(g_attn_error, &z, sizeof(int));
}

}  // namespace mt
