// qlora_kernels.cuh -- host-side launch interface between the C-ABI layer (api.cu) and the
// kernel translation units (quant.cu, gemm.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "qlora_common.cuh"

namespace qlora {

void count_launch();  // increments the process-wide launch counter

// ---- quantize / dequantize (quant.cu) -------------------------------------------------
cudaError_t launch_quantize(const float *W, int64_t n, uint8_t *codes, int8_t *qcode, float *c2, float *mu,
                            float *ws_absmax, double *ws_tree, int64_t p2, const NF4Tables &tab, int num_sms,
                            cudaStream_t st);
cudaError_t launch_dequantize(const uint8_t *codes, const int8_t *qcode, const float *c2, const float *mu, int64_t n,
                              uint16_t *out, const NF4Tables &tab, int num_sms, cudaStream_t st);

// ---- fused NF4-dequant GEMM with the LoRA term as extra K-steps (gemm.cu) ---------------
// Computes, per output row m (token) and feature f:
//   forward  (dx = false): Y[m, f]  = sum_k X[m, k] W^[f, k] + sum_j U[m, j] B[f, j]
//   backward (dx = true) : dX[m, f] = sum_n G[m, n] W^[n, f] + sum_j V[m, j] A[j, f]
// with W^ dequantized from the NF4 codes and the rebuilt block scales inside the main loop.
struct FusedArgs {
    int64_t N, K;          // weight matrix rows, cols
    int32_t KB;            // K / 64
    int32_t M;             // tokens
    const uint16_t *lora_src;  // forward: B [N, r]; backward: A [r, K]
    int64_t lora_ld;       // row stride of lora_src in elements (r or K)
    int32_t r;             // LoRA rank
    int32_t BN;            // token tile = MMA N (multiple of 32, <= 256)
    int32_t w_tiles;       // weight tiles: 256 rows (CTA pairs) or 128 rows (small kernel)
    int32_t m_tiles;       // units along the tokens (each mt token tiles of BN)
    int32_t splits;
    int32_t kt_main;       // k-tiles of 64 over the main contraction (K or ceil(N / 64))
    int32_t kt_lora;       // ceil(r / 64)
    uint16_t *out;         // [M, wdim] bf16 (splits == 1)
    float *partial;        // [splits, M, wdim] fp32 (splits > 1)
    int64_t wdim;          // output features: N (forward) or K (backward)
    // the NF4 tensor's own scale data, read by the small-M kernel (which rebuilds s'_b itself)
    const int8_t *scale_q;   // [N * KB] int8 block-scale codes
    const float *scale_c2;   // [ng] group constants
    const float *scale_mu;   // [1] scale offset
    NF4Tables tab;
};

struct FusedPlan {
    bool small;    // M <= 32: single-CTA small-token kernel (else CTA pairs)
    int BN;        // token tile = MMA N
    int mt;        // token tiles per unit (CTA pairs: 2 when M >= 512)
    int act_rows;  // token rows each CTA loads (BN / 2 for pairs, BN for the small kernel): the
                   // token maps' box height
    int stages, w_tiles, m_tiles, splits, kt_main, kt_lora;
    int grid;      // CTAs (even: clusters of two)
    size_t partial_bytes;
};
FusedPlan plan_fused(int64_t M, int64_t wdim, int64_t kt_main, int r64, int num_sms);
// the small-M kernel (gemm_small.cu): its plan (called by plan_fused for M <= 32) and launch
void plan_small(FusedPlan &pl, int64_t M, int64_t wdim, int64_t kt_main, int num_sms);
cudaError_t launch_small(bool dx, const CUtensorMap &map_codes, const CUtensorMap &map_act, const CUtensorMap &map_lora,
                         const FusedArgs &args, const FusedPlan &plan, cudaStream_t st);

// map_codes : codes as a 2-D byte tensor {K/2, N}; box {32, 128} (forward) or {64, 64} (backward)
// map_scales: rebuilt block scales, fp32 {N, KB} (transposed, [KB][N]); box {128, 1} or {64, 2}
// map_act   : X [M, K] (forward) or G [M, N] (backward), bf16, box {64, BN/2}, 128-byte swizzle
// map_lora  : U or V [M, ld] bf16, box {64, BN/2}, 128-byte swizzle (columns >= r read as 0)
// map_out   : the output [M, wdim] bf16, box {32, 32}, 64-byte swizzle (two-tile pair units store
//             through it, one box per epilogue warp and 32-token chunk)
cudaError_t launch_fused(bool dx, const CUtensorMap &map_codes, const CUtensorMap &map_scales,
                         const CUtensorMap &map_act, const CUtensorMap &map_lora, const CUtensorMap &map_out,
                         const FusedArgs &args, const FusedPlan &plan, cudaStream_t st);
cudaError_t launch_splitk_reduce(const float *partial, int splits, int64_t rows, int64_t cols, uint16_t *out,
                                 int num_sms, cudaStream_t st);
// out[kb * ld + n] = fmaf(q[n*KB + kb], fl32(c2 / 127), mu)   (ld = N when 0)
cudaError_t launch_dq_scales_t(const int8_t *q, const float *c2, const float *mu, int64_t N, int KB, float *out,
                               cudaStream_t st, int64_t ld = 0);

// ---- skinny LoRA products D[i, j] = sum_c P[i, c] Q[j, c], j < r64 (gemm.cu) -------------
// P: K-major ([Mp, Kc] row-major, map dims {Kc, Mp}, box {64, 128}) or
//    MN-major ([Kc, Mp] row-major, map dims {Mp, Kc}, box {64, 64}).
// Q: K-major ([r, Kc], map dims {Kc, r}, box {64, r64}) or
//    MN-major ([Kc, r], map dims {r, Kc}, box {64, 64}); rows/columns >= r read as zero.
// Split over the contraction across the CTAs of one cluster, whose fp32 partial tiles are summed
// in split order through distributed shared memory, and stored:
//   mode 0: out_h[i, j] = bf16(scale_j * D) for j < ld_h (scale_j = col_scale[j], or scale when
//           col_scale is NULL); out_h2[i, j] (nullable) for j < r
//   mode 1: out_f[j, i] = D for j < r  (transposed fp32)
//   mode 2: out_f[i, j] = D for j < r  (fp32)
struct ProjArgs {
    int Mp, r64, r, tiles, splits, ktiles;
    int mode;
    float scale;
    const float *col_scale;  // [ld_h] per-column scales (nullable)
    uint16_t *out_h;
    int ld_h;
    uint16_t *out_h2;
    float *out_f;
};
struct ProjPlan {
    int tiles, splits, ktiles;
};
ProjPlan plan_proj(int64_t Mp, int64_t Kc, int r64, int num_sms);
cudaError_t launch_proj(bool p_mn, bool q_mn, const CUtensorMap &map_p, const CUtensorMap &map_q, const ProjArgs &args,
                        cudaStream_t st);

// ---- forward for M <= 8 in one launch (gemv.cu) ------------------------------------------
// Y[m, n] = bf16(sum_b s'_b sum_{k in b} L[c_nk] X[m, k] + sum_j U[m, j] B[n, j]) and
// U = bf16(s Xa A^T) (also to U_save when given) for m < M (1..8).  map3: the codes as a 3-D byte
// tensor {128, N, floor(K/256)} (strides K/2, 128: the whole 256-column units only), box {128,
// kGemvBoxRows, kGemvBoxUnits}; map2: the codes as a 2-D byte tensor {K/2, N}, box {128,
// kGemvBoxRows}; both 128-byte swizzled.  ws: gemv_ws(N, K, r).total bytes, whose counters
// (counter_bytes at off_counters) must be zero when the kernel starts.
static constexpr int kGemvBoxRows = 32;
static constexpr int kGemvBoxUnits = 8;
bool gemv_supported(int64_t M, int64_t N, int64_t K);
struct GemvWs {
    int64_t RG;
    size_t off_u, off_partial, off_counters, counter_bytes, total;
};
GemvWs gemv_ws(int64_t N, int64_t K, int r);
cudaError_t launch_gemv(const CUtensorMap &map3, const CUtensorMap &map2, const int8_t *scale_q, const float *scale_c2,
                        const float *scale_mu, const uint16_t *X, const uint16_t *Xa, int M, int64_t N, int64_t K,
                        const uint16_t *A, const uint16_t *B, int r, float s, uint16_t *Y, uint16_t *U_save, void *ws,
                        const NF4Tables &tab, int num_sms, cudaStream_t st);

// ---- adapter merge (merge.cu): W_m = bf16(W^ + s B A) -----------------------------------
// map_codes: codes {K/2, N} u8, box {128, 128}; map_b: B [N, rb] bf16, box {64, 128}, 128-byte
// swizzle; map_a: A [r, K] bf16, box {64, 64}, 128-byte swizzle; map_out: W_m [N, K] bf16, box
// {64, 32}, 128-byte swizzle (one box per epilogue warp and 64-column group).
cudaError_t launch_merge(const CUtensorMap &map_codes, const CUtensorMap &map_b, const CUtensorMap &map_a,
                         const CUtensorMap &map_out, const int8_t *scale_q, const float *scale_c2,
                         const float *scale_mu, int64_t N, int64_t K, int r, float s, const NF4Tables &tab,
                         int num_sms, cudaStream_t st);

// ---- LoRA dropout on the adapter input (dropout.cu, merge.cu) ----------------------------
// Xd[e] = bf16(X[e] / (1 - p)) where kept, else 0 (Philox4x32-10 of (seed, offset, e)), for
// e < n (n % 64 == 0); mask_bits (nullable) [n / 32]: bit e % 32 of word e / 32 = kept.
cudaError_t launch_dropout_x(const uint16_t *X, int64_t n, uint64_t seed, uint64_t offset, float p, uint16_t *Xd,
                             uint32_t *mask_bits, int num_sms, cudaStream_t st);
// dX[m, k] = bf16(dX0[m, k] + kept(m, k) / (1 - p) * (V A)[m, k]) in place (dx0 = the dX buffer);
// map_v: V [M, rv] bf16, box {64, 128}, 128-byte swizzle; map_a: A [r, K] bf16, box {64, 64},
// 128-byte swizzle; map_dx: dX [M, K] bf16, box {64, 32}, 128-byte swizzle; r = rv.
cudaError_t launch_dropout_dx(const CUtensorMap &map_v, const CUtensorMap &map_a, const CUtensorMap &map_dx,
                              const uint16_t *dx0, const uint32_t *mask_bits, float p_drop, int64_t M, int64_t K,
                              int r, int num_sms, cudaStream_t st);

// dst[rows_dst, cols_dst] = src[rows_src, cols_src] where both indices are in range, else 0
cudaError_t launch_pad_2d(const uint16_t *src, int64_t rows_src, int64_t cols_src, uint16_t *dst, int64_t rows_dst,
                          int64_t cols_dst, int num_sms, cudaStream_t st);

}  // namespace qlora
