// mt_kernels.h -- internal launchers of the sm_103a kernels (not part of the C ABI).
//
// Every launcher enqueues on the given stream and returns a cudaError_t from
// the launch; shape / alignment problems are reported as
// cudaErrorInvalidValue before anything is launched.  All tensors are
// row-major; "ld" is the row stride in elements.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mt {

typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------- GEMM
// D[m, n] = sum_k A(m, k) * B(n, k), FP32 accumulation in tensor memory.
// A is K-major ([M][K], lda) unless a_mn ([K][M], lda); B is K-major
// ([N][K], ldb) unless b_mn ([K][N], ldb).  Epilogue, in this order:
//   acc_mode 2: acc += Dacc[m, n];  acc_mode >= 1: Dacc[m, n] = acc (fp32);
//   R != null : acc += R[m, n];     D != null     : D[m, n] = bf16_rne(acc).
// Requirements: lda, ldb, ldd, ldr, ldacc multiples of 8; pointers 16-byte
// aligned; M, N, K >= 1.
struct GemmArgs {
  const bf16* A; int64_t lda; int a_mn;
  const bf16* B; int64_t ldb; int b_mn;
  int M, N, K;
  bf16* D; int64_t ldd;
  const bf16* R; int64_t ldr;
  float* Dacc; int64_t ldacc; int acc_mode;
};
cudaError_t gemm(const GemmArgs& g, cudaStream_t s);
// Two independent GEMMs in one persistent launch (their tiles share the
// schedule); same requirements as gemm() for each.
cudaError_t gemm_pair(const GemmArgs& g0, const GemmArgs& g1, cudaStream_t s);
int gemm_num_sms();
// Expert-grouped GEMMs of a routed mixture-of-experts layer, whose rows are
// sorted by expert with every expert's rows padded to whole 128-row tiles.
// Rows form: D[r, n] = sum_k A[r, k] B_e(n, k), e = tile_expert[r / 128]
// (device array; tiles with e < 0 are skipped and D's rows there untouched);
// B_e = B + e * b_estride, [N][K] (ldb) or, with b_mn, [K][N].  M = rows of A
// and D, a multiple of 128.
struct GemmRowsArgs {
  const bf16* A; int64_t lda;
  const bf16* B; int64_t ldb; int b_mn; int64_t b_estride; int n_experts;
  const int* tile_expert;
  int M, N, K;
  bf16* D; int64_t ldd;
};
cudaError_t gemm_expert_rows(const GemmRowsArgs& g, cudaStream_t s);
// K-group form (the experts' weight gradients): for group i,
// D + grp_e[i] * d_estride ([M][N], ldd) = A_i^T B_i, where A_i and B_i are
// rows [grp_k0[i], grp_k0[i] + grp_klen[i]) of A ([R][M], lda) and B ([R][N],
// ldb); k0 and klen multiples of 64; at most 128 groups (host arrays).
struct GemmKGroupArgs {
  const bf16* A; int64_t lda;
  const bf16* B; int64_t ldb;
  int M, N, R;
  bf16* D; int64_t ldd; int64_t d_estride;
  int ngrp; const int* grp_e; const int* grp_k0; const int* grp_klen;
};
cudaError_t gemm_expert_kgroups(const GemmKGroupArgs& g, cudaStream_t s);
// Test hook: the next `launches` GEMM launches issue no loads, so their bounded
// waits expire and they report through the kernel error word.
void gemm_inject_stall(int launches);
// Dense GEMM tiling (gemm and gemm_pair): 0 = one CTA per 128 x 256 output
// tile; CTA pairs (cta_group::2) per 256 x 256 tile (256 x 512 for launches
// whose every GEMM has K >= 8192 and N >= 512), 1 = tiles drawn from a
// per-launch counter, 2 = every n-th tile, 3 = as 1 without the wide tiles;
// other values only read.  Returns the previous mode.
int gemm_mode(int mode);
int gemm_stall_take();

// Device-side error word written by kernels whose bounded waits expired
// (0 = none; the GEMM's and the tensor-core attention's).  Read / cleared by
// the host.
cudaError_t kernel_error_read(int* code, int clear);
cudaError_t attention_error_read(int* code, int clear);

// ---------------------------------------------------------------- elementwise
// RMSNorm forward: y = x * rstd * gamma, rstd = (mean(x^2) + eps)^-1/2.
cudaError_t rmsnorm_fwd(const bf16* x, const bf16* gamma, int64_t T, int H, float eps, bf16* y,
                        float* rstd, cudaStream_t s);
// RMSNorm backward.  dx = r*gamma*dy - r^3/H * x * sum(dy*gamma*x) (+ dres
// if not null).  dgamma (bf16, H) = sum over rows of dy * x * r; partial is
// scratch of rmsnorm_bwd_partial_floats(T, H) floats.
cudaError_t rmsnorm_bwd(const bf16* dy, const bf16* x, const bf16* gamma, const float* rstd,
                        const bf16* dres, int64_t T, int H, bf16* dx, bf16* dgamma, float* partial,
                        cudaStream_t s);
int64_t rmsnorm_bwd_partial_floats(int64_t T, int H);
int rmsnorm_bwd_blocks(int64_t T);
// Reduces rmsnorm_bwd_blocks(T) rows of `partial` ([blocks][H] floats) into
// dgamma (bf16).
cudaError_t rmsnorm_bwd_stage2(const float* partial, int nblk, int H, bf16* dgamma, cudaStream_t s);

// Rotate-half RoPE on the first n_heads heads (width hd) of every row of
// x ([T][ld]); position = row % S; cs holds cos/sin [S][hd/2][2] in fp32.
// inverse != 0 applies the transpose rotation.
cudaError_t rope(bf16* x, int64_t T, int64_t ld, int n_heads, int hd, int S, const float* cs,
                 int inverse, cudaStream_t s);
// h = silu(g) * u with gu rows [g (F) | u (F)].
cudaError_t swiglu_fwd(const bf16* gu, int64_t T, int F, bf16* h, cudaStream_t s);
cudaError_t swiglu_bwd(const bf16* gu, const bf16* dh, int64_t T, int F, bf16* dgu, cudaStream_t s);
// X[t] = E[tok[t]].
cudaError_t embed_fwd(const int32_t* tok, const bf16* E, int64_t T, int H, int V, bf16* X,
                      cudaStream_t s);
// dE[v] = sum over t with tok[t] = v of dX[t], written densely as bf16 for all
// V rows.  row_start[V+1] / rows[T] list, per vocabulary row, the token rows
// that hold it (CSR, ascending).
cudaError_t embed_bwd(const int32_t* row_start, const int32_t* rows, const bf16* dX, int V, int H,
                      bf16* dE, cudaStream_t s);
// Cross-entropy over `rows` rows of logits ([rows][V], bf16), overwritten with
// dlogits = (softmax - onehot(target)) * inv_norm; rows with target < 0 get 0.
// row_loss[r] = lse - logit[target] (0 without target).
cudaError_t cross_entropy(bf16* logits, const int32_t* target, int64_t rows, int V, float inv_norm,
                          float* row_loss, cudaStream_t s);
// out[0] = sum(x[0..n)) * scale (single block, fixed order).
cudaError_t reduce_sum(const float* x, int64_t n, float scale, float* out, cudaStream_t s);
// y (bf16) = x (fp32) elementwise, n values; rows/ld variants for strided output.
cudaError_t f32_to_bf16_2d(const float* x, int64_t ldx, int64_t rows, int64_t cols, bf16* y,
                           int64_t ldy, float scale, cudaStream_t s);
cudaError_t add_bf16(const bf16* a, const bf16* b, int64_t n, bf16* y, cudaStream_t s);

// ---------------------------------------------------------------- debug guards
// bad[0] = the lowest index g < n whose 4096 bytes at base + offs[g] are not
// all 0xA5 (left unchanged when every guard is intact).
cudaError_t guard_check(const uint8_t* base, const int64_t* offs, int n, int* bad, cudaStream_t s);

// ---------------------------------------------------------------- routed MoE
// Device arrays of one MoE layer's routing (k_moe.cu).  T tokens, E experts
// (<= 128), k <= 8 of them per token.
struct MoePlan {
  int32_t* idx;          // [T][k] selected experts, descending logit
  float* gate;           // [T][k] softmax over the selected logits
  int32_t* slot_row;     // [T][k] row of assignment (t, i) in the expert-sorted layout
  int32_t* cnt;          // [moe_chunks(T)][E] scratch
  int32_t* base;         // [moe_chunks(T)][E] scratch
  int32_t* counts;       // [E] tokens routed to each expert
  int32_t* tile_expert;  // [moe_rows_max / 128] expert of each 128-row tile, -1 past the end
  int32_t* perm_tok;     // [moe_rows_max] token of each sorted row, -1 on padding rows
};
// Rows of the expert-sorted layout in the worst case (every expert's segment
// padded to a multiple of 128), and the counting sort's chunk count.
int64_t moe_rows_max(int64_t T, int E, int k);
int64_t moe_chunks(int64_t T);
// From FP32 router logits [T][E]: top-k (ties: lower expert index), gates,
// per-expert counts, segment layout (expert e's rows start at the sum of the
// earlier experts' counts rounded up to 128; rows of one expert in ascending
// (token, slot) order), perm_tok, slot_row and tile_expert.
cudaError_t moe_plan(const float* logits, int64_t T, int E, int k, const MoePlan& p, cudaStream_t s);
// xperm[r] = yn[perm_tok[r]] ([R][H]); padding rows zero.
cudaError_t moe_gather(const bf16* yn, int H, const int32_t* perm_tok, int64_t R, bf16* xperm, cudaStream_t s);
// out[t] = x1[t] + sum_i gate[t, i] Y[slot_row[t, i]].
cudaError_t moe_combine(const bf16* x1, const bf16* Y, const int32_t* slot_row, const float* gate, int64_t T, int H,
                        int k, bf16* out, cudaStream_t s);
// dY[slot_row[t, i]] = gate[t, i] dout[t]; dlogits [T][E] (BF16) =
// gradient of the router logits through the softmax over the selected ones.
cudaError_t moe_combine_bwd(const bf16* dout, const bf16* Y, const int32_t* slot_row, const int32_t* idx,
                            const float* gate, int64_t T, int H, int k, int E, bf16* dY, bf16* dlogits,
                            cudaStream_t s);
// Zero the padding rows (perm_tok < 0) of buf [R][cols].
cudaError_t moe_zero_pad(bf16* buf, int cols, const int32_t* perm_tok, int64_t R, cudaStream_t s);
// dyn[t] = sum_i dX[slot_row[t, i]].
cudaError_t moe_scatter(const bf16* dX, const int32_t* slot_row, int64_t T, int H, int k, bf16* dyn,
                        cudaStream_t s);

// ---------------------------------------------------------------- attention
// Causal grouped-query attention over n_seq sequences of S tokens.  qkv rows
// ([T][(nh+2nkv)hd]) hold [q | k | v]; o is [T][nh*hd]; lse is [nh][T] fp32
// (natural log).  hd in {64, 128}.
cudaError_t attention_fwd(const bf16* qkv, int n_seq, int S, int nh, int nkv, int hd, bf16* o,
                          float* lse, cudaStream_t s);
// The same forward on tcgen05 tensor cores with TMEM accumulators (used by
// attention_fwd).
cudaError_t attention_fwd_tc(const bf16* qkv, int n_seq, int S, int nh, int nkv, int hd, bf16* o, float* lse,
                             cudaStream_t s);
// Tensor-core backward core: dQ, dK, dV into dqkv (BF16); delta =
// rowsum(dO o O) precomputed.  Used by attention_bwd.
cudaError_t attention_bwd_tc_core(const bf16* qkv, const bf16* dout, const float* lse, const float* delta,
                                  int n_seq, int S, int nh, int nkv, int hd, bf16* dqkv, cudaStream_t s);
// Backward: dqkv ([T][(nh+2nkv)hd]) receives dq, dk, dv.  delta ([nh][T]
// fp32) is scratch.
cudaError_t attention_bwd(const bf16* qkv, const bf16* o, const float* lse, const bf16* dout,
                          int n_seq, int S, int nh, int nkv, int hd, bf16* dqkv, float* delta,
                          cudaStream_t s);

}  // namespace mt
