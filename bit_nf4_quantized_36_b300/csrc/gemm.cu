// gemm.cu -- tensor-core kernels of the QLoRA linear layer (sm_103a, tcgen05 + TMEM + TMA).
//
// 1. nf4_lora_gemm_kernel<dx, stages, mt>: the fused NF4-dequant GEMM for M > 32.  The weight
//    side is the MMA's A operand ("swap-AB": weights are the M side, tokens the N side), so that
//    each expanded weight is reused by up to mt x 256 tokens.  A cluster of two CTAs shares every
//    MMA (tcgen05.mma.cta_group::2, M = 256 weight rows): each CTA TMA-stages the packed nibbles
//    of its 128 rows and half of each token tile; eight decode warps expand the nibbles to bf16
//    through a per-block 16-entry register table (byte-permute lookups) straight into the
//    128-byte-swizzled smem layout the MMA reads; one thread of the even CTA issues the MMAs;
//    four epilogue warps per CTA drain TMEM.  The rank-r LoRA term is appended as extra K-steps
//    (weights side: zero-padded B or A rows; token side: U or V).
//      forward : A = W^ tile (K-major: rows = out features, 64 k per row)
//      backward: A = W^^T tile (MN-major: each 128-byte row holds 64 consecutive k of one
//                weight row n, the contraction index), so the same decode routine serves both.
//    Source: "QLoRA -- La base en 4 bits, LoRA encima" (paperclase, lesson 8), "Parte 4 - LoRA
//    encima": h = W^ x + (alpha/r) B A x and dL/dx = (W^ + (alpha/r) B A)^T dL/dh, with W^
//    rebuilt on every pass ("QLoRA" glossary, ultralytics: dequantized to bfloat16 right before
//    the matmul, in the forward and in backprop).
// 2. lora_proj_kernel<p_mn, q_mn>: skinny products with N = r64 <= 256 (U = X A^T, V = G B,
//    dA = V^T X, dB = G^T U), split over the contraction across the CTAs of a cluster, whose
//    fp32 partial tiles are summed in split order through distributed shared memory.
// The small-M variant of 1. is in gemm_small.cu; forwards of up to 8 tokens use the GEMV in gemv.cu.
#include <algorithm>
#include <mutex>

#include "qlora_common.cuh"
#include "qlora_kernels.cuh"

namespace qlora {

static constexpr int kProjStages = 4;                 // skinny products
static constexpr uint32_t kATileBytes = 128u * 128u;  // 128 rows x 64 bf16
static constexpr uint32_t kCodesTileBytes = 4096u;    // 128 rows x 32 B or 64 rows x 64 B
static constexpr uint32_t kScaleTileBytes = 512u;     // 128 (or 2 x 64) fp32 block scales
static constexpr uint32_t kCStageBytes = kCodesTileBytes + kScaleTileBytes;
static constexpr int kFusedThreads = 448;              // 14 warps
static constexpr int kDecodeWarp0 = 6;                 // warps 6..13 decode
static constexpr int kEpiWarp0 = 2;                    // warps 2..5 epilogue
static constexpr uint32_t kTmemCols = 512;             // two accumulators of up to 256 columns
static constexpr uint32_t kOutStageBytes = 2u * 32u * 128u * 2u;  // two [32][128] bf16 store tiles

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}

// The 16 dequantized values of one block, v[c] = bf16_rne(fl32(NF4[c] * s)), split into byte
// tables: lo[i] holds the low bytes of v[4i..4i+3], hi[i] the high bytes.
__device__ __forceinline__ void build_table(float s, const NF4Tables &tab, uint32_t (&lo)[4], uint32_t (&hi)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t p01 = bf16x2(__fmul_rn(tab.level[4 * i], s), __fmul_rn(tab.level[4 * i + 1], s));
        const uint32_t p23 = bf16x2(__fmul_rn(tab.level[4 * i + 2], s), __fmul_rn(tab.level[4 * i + 3], s));
        lo[i] = prmt(p01, p23, 0x6420u);
        hi[i] = prmt(p01, p23, 0x7531u);
    }
}

// Look up 4 codes in nibble order (c1, c0, c3, c2) (the packing puts element 2j in the high
// nibble of byte j) with selectors prepared by decode8, and return the bf16 pairs
// (e0 | e1 << 16) and (e2 | e3 << 16).  The low 3 bits of each code select within 8-entry
// halves (sel); bit 3 picks the half (sel2).
__device__ __forceinline__ void lookup4(uint32_t sel, uint32_t sel2, const uint32_t (&lo)[4], const uint32_t (&hi)[4],
                                        uint32_t &o0, uint32_t &o1) {
    const uint32_t l4 = prmt(prmt(lo[0], lo[1], sel), prmt(lo[2], lo[3], sel), sel2);
    const uint32_t h4 = prmt(prmt(hi[0], hi[1], sel), prmt(hi[2], hi[3], sel), sel2);
    o0 = prmt(l4, h4, 0x4051u);
    o1 = prmt(l4, h4, 0x6273u);
}

// 8 codes (one 32-bit word, elements 0..7) -> 4 words of bf16 pairs.  The selectors of all 8
// codes are formed at once (the byte permute reads only the low 16 bits of its selector).
__device__ __forceinline__ uint4 decode8(uint32_t x, const uint32_t (&lo)[4], const uint32_t (&hi)[4]) {
    const uint32_t sel = x & 0x77777777u;
    const uint32_t sel2 = ((x >> 1) & 0x44444444u) | 0x32103210u;
    uint4 o;
    lookup4(sel, sel2, lo, hi, o.x, o.y);
    lookup4(sel >> 16, sel2 >> 16, lo, hi, o.z, o.w);
    return o;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// 32 consecutive bf16 of one row starting at column j0, zero beyond column `jmax` (exclusive).
__device__ __forceinline__ void load_row32(const uint16_t *row, int64_t j0, int64_t jmax, bool vec_ok, uint4 (&v)[4]) {
    if (vec_ok && j0 + 32 <= jmax) {
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = __ldg(reinterpret_cast<const uint4 *>(row + j0) + i);
        return;
    }
    uint32_t w[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        const int64_t j = j0 + 2 * e;
        const uint32_t lo = (j < jmax) ? (uint32_t)__ldg(row + j) : 0u;
        const uint32_t hi = (j + 1 < jmax) ? (uint32_t)__ldg(row + j + 1) : 0u;
        w[e] = lo | (hi << 16);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}

// Warp-uniform bounded wait: lane 0 polls, the result is broadcast, and __syncwarp orders the
// other lanes' later accesses after lane 0's acquire.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile uint32_t *abort) {
    uint32_t ok = 0;
    if ((threadIdx.x & 31u) == 0) ok = mbar_wait(bar, parity, abort) ? 1u : 0u;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

struct UnitInfo {
    int w_tile, m_tile, split, kt0, kt1, nk;
};

__device__ __forceinline__ UnitInfo unit_info(const FusedArgs &p, int u) {
    UnitInfo ui;
    ui.split = u % p.splits;
    const int t = u / p.splits;
    ui.w_tile = t % p.w_tiles;
    ui.m_tile = t / p.w_tiles;
    ui.kt0 = (int)((int64_t)ui.split * p.kt_main / p.splits);
    ui.kt1 = (int)((int64_t)(ui.split + 1) * p.kt_main / p.splits);
    ui.nk = (ui.kt1 - ui.kt0) + (ui.split == p.splits - 1 ? p.kt_lora : 0);
    return ui;
}

// One unit = a 256-row weight tile (128 rows per CTA of the pair) x BN tokens x one split of
// the contraction.  The pair (a cluster of two CTAs on neighbouring SMs) shares every MMA:
//   - each CTA stages and decodes its own 128 weight rows and TMA-loads BN/2 of the tokens, every
//     copy completing on a barrier of the CTA that issued it (so each CTA can account for its
//     own copies when it unwinds after a timeout);
//   - the even CTA ("leader") issues tcgen05.mma.cta_group::2 with M = 256, N = BN, reading A
//     and B from both CTAs' shared memory and accumulating into both CTAs' TMEM;
//   - MMA completion is multicast to both CTAs' barriers; the odd CTA's decode and epilogue
//     warps report to the leader's barriers by remote arrive.
// Per SM this halves the inbound activation bytes and the MMA-issue work of a 128 x BN tile.
//
// kMT token tiles of BN per unit: with kMT = 2 every decoded weight tile feeds two MMAs (512
// tokens), halving the decode work per FLOP -- the decode (integer-pipe byte permutes) is what
// bounds a unit with one tile.  Two accumulators of 256 columns then fill the TMEM, so they are
// not double-buffered: the next unit's MMAs wait for the epilogue (kMT = 1 keeps two buffers).
template <bool kDX, int kStages, int kMT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kFusedThreads, 1)
    nf4_lora_gemm_kernel(const __grid_constant__ CUtensorMap map_codes, const __grid_constant__ CUtensorMap map_scales,
                         const __grid_constant__ CUtensorMap map_act, const __grid_constant__ CUtensorMap map_lora,
                         const __grid_constant__ CUtensorMap map_out, const FusedArgs p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // The 128-byte-swizzled tiles need 1024-byte alignment.  The dynamic shared memory of a
    // kernel without static shared memory starts aligned, and the launch requests no slack for
    // re-aligning (two-tile units use all 227 KB); should that not hold, every CTA (the layout
    // is the same in all of them) reports it and does no work.
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0) atomicOr(&g_error_word, kErrLayout);
        return;
    }
    uint8_t *smem = smem_raw;
    const uint32_t bh_rows = (uint32_t)p.BN / 2u;     // token rows this CTA loads per tile
    const uint32_t b_bytes = bh_rows * 128u;          // per token tile and stage, this CTA
    const uint32_t bs_bytes = kMT * b_bytes;          // per stage, this CTA
    constexpr int kBufs = kMT == 1 ? 2 : 1;           // accumulator buffers
    // kMT == 2: stage completion is committed every stage (the MMA thread has slack at two
    // MMAs per k16); kMT == 1: once per two stages, on empty[s | 1]
    constexpr int kPairMask = kMT == 1 ? 1 : 0;
    uint8_t *sA = smem;
    uint8_t *sB = sA + kStages * kATileBytes;
    uint8_t *sC = sB + kStages * bs_bytes;
    // kMT == 2: two [32 tokens][128 features] bf16 tiles staging the epilogue's TMA stores
    uint8_t *sOut = sC + kStages * kCStageBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sOut + (kMT == 2 ? kOutStageBytes : 0));
    uint64_t *full_c = bars;                 // codes + scales landed (or LoRA k-step announced); local
    uint64_t *full_b = bars + kStages;       // this CTA's token tiles landed (each CTA tracks its own copies)
    uint64_t *full_a = bars + 2 * kStages;   // leader: both CTAs' decoded weight tiles written
    // both: the pair MMAs reading stages s & ~1 and s | 1 finished.  Completion is committed once
    // per two stages (on empty[s | 1]) to halve the MMA thread's commit work; empty[s & ~1] is unused.
    uint64_t *empty = bars + 3 * kStages;
    uint64_t *acc_full = bars + 4 * kStages; // both [kBufs]: accumulator ready
    uint64_t *acc_empty = acc_full + 2;      // leader [kBufs]: both CTAs drained the accumulator
    uint64_t *drain = acc_empty + 2;         // leader [1]
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(drain + 1);
    volatile uint32_t *s_abort = s_tmem + 1;
    volatile uint32_t *s_epi_ok = s_tmem + 2;  // epilogue: the accumulator wait's outcome

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int pair_id = blockIdx.x >> 1;
    const int num_pairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full_c[s], 1);
            mbar_init(&full_b[s], 1);
            mbar_init(&full_a[s], 8);  // the four warps of the stage's decode group, in both CTAs
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 8);  // four epilogue warps in both CTAs
        }
        mbar_init(drain, 1);
        *s_abort = 0u;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(s_tmem, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_barrier();  // the peer's barriers are initialised before any remote arrival
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;

    const int total_units = p.w_tiles * p.m_tiles * p.splits;

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------------
        if (lane == 0) {
            tma_prefetch_desc(&map_codes);
            tma_prefetch_desc(&map_scales);
            tma_prefetch_desc(&map_act);
            tma_prefetch_desc(&map_lora);
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued_parity[kStages];
            bool issued[kStages];
            for (int i = 0; i < kStages; ++i) issued[i] = false, issued_parity[i] = 0;
            bool ok = true;
            // test hook: no codes copy (and no arrival on full_c) for the first k-step of pair 0
            bool skip_codes = leader && pair_id == 0 && (*(volatile uint32_t *)&g_inject & kInjectSkipCodes);
            for (int u = pair_id; u < total_units && ok; u += num_pairs) {
                const UnitInfo ui = unit_info(p, u);
                const int wt = ui.w_tile * 2 + (int)rank;  // this CTA's 128-row weight tile
                const int m_row = ui.m_tile * kMT * p.BN + (int)(rank * bh_rows);  // first tile's rows
                for (int j = 0; j < ui.nk; ++j) {
                    if (!mbar_wait_cl(&empty[s | kPairMask], ph ^ 1u, s_abort)) { ok = false; break; }
                    const bool lora = (ui.kt0 + j) >= ui.kt1;
                    mbar_arrive_expect_tx(&full_b[s], bs_bytes);
                    if (skip_codes && !lora) {
                        skip_codes = false;
#pragma unroll
                        for (int i = 0; i < kMT; ++i)
                            tma_load_2d(sB + s * bs_bytes + i * b_bytes, &map_act, &full_b[s], (ui.kt0 + j) * 64,
                                        m_row + i * p.BN);
                    } else if (!lora) {
                        const int kt = ui.kt0 + j;
                        uint8_t *dc = sC + s * kCStageBytes;
                        mbar_arrive_expect_tx(&full_c[s], kCStageBytes);
                        if (kDX) {
                            tma_load_2d(dc, &map_codes, &full_c[s], wt * 64, kt * 64);
                            tma_load_2d(dc + kCodesTileBytes, &map_scales, &full_c[s], kt * 64, wt * 2);
                        } else {
                            tma_load_2d(dc, &map_codes, &full_c[s], kt * 32, wt * 128);
                            tma_load_2d(dc + kCodesTileBytes, &map_scales, &full_c[s], wt * 128, kt);
                        }
#pragma unroll
                        for (int i = 0; i < kMT; ++i)
                            tma_load_2d(sB + s * bs_bytes + i * b_bytes, &map_act, &full_b[s], kt * 64, m_row + i * p.BN);
                    } else {
                        const int lt = j - (ui.kt1 - ui.kt0);
                        mbar_arrive(&full_c[s]);
#pragma unroll
                        for (int i = 0; i < kMT; ++i)
                            tma_load_2d(sB + s * bs_bytes + i * b_bytes, &map_lora, &full_b[s], lt * 64, m_row + i * p.BN);
                    }
                    issued[s] = true;
                    issued_parity[s] = ph;
                    if (++s == kStages) { s = 0; ph ^= 1u; }
                }
            }
            if (ok) {
                // every MMA commit aimed at this CTA has arrived before it may exit.  A parity
                // wait only sees a barrier's latest phase, so each stage pair is waited on once,
                // for the pass in which it was last used: that of its even stage, which every
                // pass uses first.
                for (int i = 0; i < kStages; i += 1 + kPairMask) {
                    if (issued[i] && !mbar_wait_cl(&empty[i | kPairMask], issued_parity[i], s_abort)) break;
                }
            } else {
                // let copies already in flight land before the CTA can exit.  Every copy this CTA
                // issued completes on one of its own barriers (its token tiles on full_b, its codes
                // and scales on full_c), so it can wait for all of them; the pair then meets at the
                // cluster barrier at the end, so neither CTA leaves while the other's copies land.
                for (int i = 0; i < kStages; ++i) {
                    if (!issued[i]) continue;
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(&full_b[i], issued_parity[i]) && globaltimer_ns() - t0 < 10000000ull) {}
                    while (!mbar_try_wait(&full_c[i], issued_parity[i]) && globaltimer_ns() - t0 < 20000000ull) {}
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------ MMA issuer (leader) ------------------------------
        if (lane == 0 && leader) {
            const uint32_t idesc = make_idesc_bf16((uint32_t)p.BN, kDX, false, 256u);
            const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
            int s = 0;
            uint32_t ph = 0;
            int lt = 0;
            bool ok = true;
            bool any = false;
            for (int u = pair_id; u < total_units && ok; u += num_pairs, ++lt) {
                const UnitInfo ui = unit_info(p, u);
                const int a = lt % kBufs;
                if (!mbar_wait_cl(&acc_empty[a], ((lt / kBufs) & 1) ^ 1u, s_abort)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)a * 256u;  // tile i at + i * 256
                for (int j = 0; j < ui.nk; ++j) {
                    // full_a completes only after both CTAs' decode groups have also seen their full_b
                    if (!mbar_wait_cl(&full_a[s], ph, s_abort)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = a_base + (uint32_t)s * kATileBytes;
                    const uint32_t b_addr = b_base + (uint32_t)s * bs_bytes;
#pragma unroll
                    for (int i = 0; i < kMT; ++i) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t adesc = kDX ? make_sw128_desc(a_addr + kk * 2048u, 8192u, 1024u)
                                                       : make_sw128_desc(a_addr + kk * 32u, 16u, 1024u);
                            const uint64_t bdesc = make_sw128_desc(b_addr + i * b_bytes + kk * 32u, 16u, 1024u);
                            umma_bf16_pair(d_tmem + (uint32_t)i * 256u, adesc, bdesc, idesc, (j > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    any = true;
                    if ((s & kPairMask) == kPairMask) umma_commit_pair_mc(&empty[s], 0x3);
                    if (++s == kStages) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                umma_commit_pair_mc(&acc_full[a], 0x3);
            }
            // paired commits, and the last stage used was even: release its pair too
            if (kPairMask && ok && (s & 1)) umma_commit_pair_mc(&empty[s], 0x3);
            if (!ok && any) {
                umma_commit_pair_mc(drain, 0x1);
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait_cl(drain, 0) && globaltimer_ns() - t0 < 20000000ull) {}
            }
        }
        __syncwarp();
    } else if (warp < kDecodeWarp0) {
        // ------------------------------ epilogue -----------------------------------------
        const int quarter = warp & 3;  // TMEM lanes this warp may access
        const uint32_t acc_empty_leader = mapa_shared(acc_empty, 0);
        int lt = 0;
        for (int u = pair_id; u < total_units; u += num_pairs, ++lt) {
            const UnitInfo ui = unit_info(p, u);
            const int a = lt % kBufs;
            uint32_t okw = 0;
            if (kMT == 2) {
                // one outcome for the four warps, which meet at named barriers below
                if (threadIdx.x == kEpiWarp0 * 32) *s_epi_ok = mbar_wait_cl(&acc_full[a], (lt / kBufs) & 1, s_abort) ? 1u : 0u;
                named_barrier_sync(2, 128);
                okw = *s_epi_ok;
                named_barrier_sync(2, 128);
            } else {
                if (lane == 0) okw = mbar_wait_cl(&acc_full[a], (lt / kBufs) & 1, s_abort) ? 1u : 0u;
                okw = __shfl_sync(0xffffffffu, okw, 0);
                __syncwarp();
            }
            if (!okw) break;
            tc_fence_after();
            const int64_t f = ((int64_t)ui.w_tile * 2 + rank) * 128 + quarter * 32 + lane;
            const int nchunks = kMT * p.BN / 32;
            for (int cc = 0; cc < nchunks; ++cc) {
                const int i = cc / (p.BN / 32), c = cc % (p.BN / 32);  // token tile, 32-column chunk
                const int m0 = (ui.m_tile * kMT + i) * p.BN;
                const uint32_t tcol = tmem_base + (uint32_t)a * 256u + (uint32_t)i * 256u + (uint32_t)c * 32u;
                if (kMT == 2 && p.splits == 1) {
                    // this warp's 32 features x 32 tokens as two accumulator fragments (features
                    // 16h .. 16h + 15 of the warp), written to shared memory transposed by stmatrix
                    uint32_t v[2][16];
                    tmem_ld_16x256b_x4(tcol + ((uint32_t)(quarter * 32) << 16), v[0]);
                    tmem_ld_16x256b_x4(tcol + ((uint32_t)(quarter * 32 + 16) << 16), v[1]);
                    tmem_ld_wait();
                    if (cc == nchunks - 1) {
                        // the accumulator is read out: the next unit's MMAs may start
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            if (leader) mbar_arrive(&acc_empty[a]);
                            else mbar_arrive_remote(acc_empty_leader + (uint32_t)a * 8u);
                        }
                    }
                    // each warp stages its [32 tokens][32 features] in its own double-buffered,
                    // 64-byte-swizzled 2 KB tile and stores it with one TMA store: no barrier
                    // between the epilogue warps
                    uint8_t *buf = sOut + (quarter * 2 + (cc & 1)) * (kOutStageBytes / 8);
                    if (lane == 0) bulk_wait_group_read<1>();  // this warp's store two chunks back has read buf
                    __syncwarp();
                    {
                        const int mi = lane >> 3, j = lane & 7;  // this thread addresses row j of matrix mi
                        const uint32_t buf_addr = smem_u32(buf);
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
#pragma unroll
                            for (int kk = 0; kk < 2; ++kk) {
                                // matrices: features (top, bottom 8 of 16 h .. 16 h + 15) x tokens
                                // 8 k .. 8 k + 7, k = 2 kk, 2 kk + 1
                                const int k = 2 * kk + (mi >> 1), bot = mi & 1;
                                const int tok = 8 * k + j;
                                const int ch = 2 * h + bot;  // 16-byte chunk of the token's 64-byte row
                                const uint32_t addr = buf_addr + (uint32_t)tok * 64u +
                                                      ((uint32_t)(ch ^ ((tok >> 1) & 3)) << 4);
                                const uint32_t *w = v[h] + 8 * kk;
                                stmatrix_x4_trans(addr, bf16x2(__uint_as_float(w[0]), __uint_as_float(w[1])),
                                                  bf16x2(__uint_as_float(w[2]), __uint_as_float(w[3])),
                                                  bf16x2(__uint_as_float(w[4]), __uint_as_float(w[5])),
                                                  bf16x2(__uint_as_float(w[6]), __uint_as_float(w[7])));
                            }
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&map_out, buf, (int)(((int64_t)ui.w_tile * 2 + rank) * 128) + quarter * 32,
                                     m0 + c * 32);
                        bulk_commit_group();
                    }
                    continue;
                }
                uint32_t r[32];
                tmem_ld_32x32b_x32(tcol + ((uint32_t)(quarter * 32) << 16), r);
                tmem_ld_wait();
                if (f < p.wdim) {
                    if (p.splits == 1) {
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) {
                            const int m = m0 + c * 32 + jj;
                            if (m < p.M) {
                                __nv_bfloat16 h = __float2bfloat16_rn(__uint_as_float(r[jj]));
                                if (QLORA_IN_BOUNDS((int64_t)m * p.wdim + f < (int64_t)p.M * p.wdim))
                                    p.out[(int64_t)m * p.wdim + f] = *reinterpret_cast<uint16_t *>(&h);
                            }
                        }
                    } else {
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) {
                            const int m = m0 + c * 32 + jj;
                            if (m < p.M && QLORA_IN_BOUNDS(ui.split < p.splits))
                                p.partial[((int64_t)ui.split * p.M + m) * p.wdim + f] = __uint_as_float(r[jj]);
                        }
                    }
                }
            }
            if (kMT == 2 && p.splits == 1) continue;  // released after the last TMEM read
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader) mbar_arrive(&acc_empty[a]);
                else mbar_arrive_remote(acc_empty_leader + (uint32_t)a * 8u);
            }
        }
        // the output stores have completed before the CTA exits
        if (kMT == 2 && lane == 0) bulk_wait_group_all();
    } else {
        // ------------------------------ decode warps -------------------------------------
        // Two groups of four warps take alternate pipeline stages (stage s always goes to
        // group s % 2, kStages being even).  Each thread expands one 128-byte smem row: the 64
        // weights of one NF4 block, so the block's 16-entry table is built once per 64 weights.
        const int t = (threadIdx.x - kDecodeWarp0 * 32) & 127;  // row slot 0..127
        const int group = (threadIdx.x - kDecodeWarp0 * 32) >> 7;
        const uint32_t a_base = smem_u32(sA);
        const uint32_t full_a_leader = mapa_shared(full_a, 0);
        const bool lora_vec = (p.lora_ld % 8) == 0;
        // per-thread geometry of the 128-row A tile
        uint32_t row_off, code_off, scale_off;
        int nl = 0, kbl = 0;
        if (!kDX) {
            row_off = (uint32_t)t * 128u;
            code_off = (uint32_t)t * 32u;
            scale_off = kCodesTileBytes + (uint32_t)t * 4u;
        } else {
            nl = t >> 1;
            kbl = t & 1;
            row_off = (uint32_t)kbl * 8192u + (uint32_t)nl * 128u;
            code_off = (uint32_t)nl * 64u + (uint32_t)kbl * 32u;
            scale_off = kCodesTileBytes + (uint32_t)(kbl * 64 + nl) * 4u;
        }
        const uint32_t r7 = (row_off >> 7) & 7u;  // swizzle phase of this row (tiles are 1024-aligned)
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int u = pair_id; u < total_units && ok; u += num_pairs) {
            const UnitInfo ui = unit_info(p, u);
            const int wt = ui.w_tile * 2 + (int)rank;
            const int64_t n_fwd = (int64_t)wt * 128 + t;  // forward: weight row of this thread
            const int kblock = wt * 2 + kbl;              // backward: 64-column block along K
            for (int j = 0; j < ui.nk; ++j) {
                const int my_stage = (s & 1) == group;
                if (my_stage) {
                    const bool lora = (ui.kt0 + j) >= ui.kt1;
                    const int kt = lora ? j - (ui.kt1 - ui.kt0) : ui.kt0 + j;
                    bool valid;
                    uint4 lv[8];
                    if (!kDX) {
                        valid = n_fwd < p.N;
                        if (lora && valid) {
                            const uint16_t *row = p.lora_src + n_fwd * p.lora_ld;
                            load_row32(row, (int64_t)kt * 64, p.r, lora_vec, *reinterpret_cast<uint4(*)[4]>(&lv[0]));
                            load_row32(row, (int64_t)kt * 64 + 32, p.r, lora_vec, *reinterpret_cast<uint4(*)[4]>(&lv[4]));
                        }
                    } else {
                        const int64_t n = (int64_t)kt * 64 + nl;  // contraction row (weight or LoRA row)
                        valid = kblock < p.KB && n < (lora ? (int64_t)p.r : p.N);
                        if (lora && valid) {
                            const uint4 *src = reinterpret_cast<const uint4 *>(p.lora_src + n * p.lora_ld + (int64_t)kblock * 64);
#pragma unroll
                            for (int i = 0; i < 8; ++i) lv[i] = __ldg(src + i);
                        }
                    }
                    uint32_t okw = 0;
                    if (lane == 0)
                        okw = (mbar_wait_cl(&empty[s | kPairMask], ph ^ 1u, s_abort) && mbar_wait(&full_c[s], ph, s_abort)) ? 1u : 0u;
                    okw = __shfl_sync(0xffffffffu, okw, 0);
                    __syncwarp();
                    if (!okw) { ok = false; break; }
                    const uint32_t row_addr = a_base + (uint32_t)s * kATileBytes + row_off;
                    if (!valid) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) st_shared_v4(row_addr + (((uint32_t)i ^ r7) << 4), make_uint4(0, 0, 0, 0));
                    } else if (!lora) {
                        const uint8_t *cst = sC + s * kCStageBytes;
                        const uint4 c0 = *reinterpret_cast<const uint4 *>(cst + code_off);
                        const uint4 c1 = *reinterpret_cast<const uint4 *>(cst + code_off + 16);
                        const float sc = *reinterpret_cast<const float *>(cst + scale_off);
                        uint32_t lo[4], hi[4];
                        build_table(sc, p.tab, lo, hi);
                        // 128-byte swizzle: chunk c of row r lives at chunk c ^ (r & 7)
                        st_shared_v4(row_addr + ((0u ^ r7) << 4), decode8(c0.x, lo, hi));
                        st_shared_v4(row_addr + ((1u ^ r7) << 4), decode8(c0.y, lo, hi));
                        st_shared_v4(row_addr + ((2u ^ r7) << 4), decode8(c0.z, lo, hi));
                        st_shared_v4(row_addr + ((3u ^ r7) << 4), decode8(c0.w, lo, hi));
                        st_shared_v4(row_addr + ((4u ^ r7) << 4), decode8(c1.x, lo, hi));
                        st_shared_v4(row_addr + ((5u ^ r7) << 4), decode8(c1.y, lo, hi));
                        st_shared_v4(row_addr + ((6u ^ r7) << 4), decode8(c1.z, lo, hi));
                        st_shared_v4(row_addr + ((7u ^ r7) << 4), decode8(c1.w, lo, hi));
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; ++i) st_shared_v4(row_addr + (((uint32_t)i ^ r7) << 4), lv[i]);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        // each CTA's group also waits for that CTA's token tiles, so that the
                        // leader's MMA thread has a single barrier to wait on: full_a completes
                        // when both CTAs' weight tiles are decoded and both CTAs' token tiles
                        // have landed
                        if (!mbar_wait_cl(&full_b[s], ph, s_abort)) {
                            ok = false;
                        } else if (leader) {
                            mbar_arrive(&full_a[s]);
                        } else {
                            mbar_arrive_remote(full_a_leader + (uint32_t)s * 8u);
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok ? 1u : 0u, 0) != 0;
                    if (!ok) break;
                }
                if (++s == kStages) { s = 0; ph ^= 1u; }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_barrier();  // neither CTA leaves while the pair's MMAs or remote arrivals may still touch it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------------------------------
// Skinny LoRA products D[i, j] = sum_c P[i, c] Q[j, c] (N = r64 <= 256), split over the
// contraction.  The `splits` CTAs of one 128-row tile form a thread-block cluster: each parks
// its fp32 partial tile in its own shared memory, and after a cluster barrier every CTA sums a
// slice of the rows over all partials in split order (distributed shared memory reads) --
// deterministic, with no global scratch.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void proj_store(const ProjArgs &a, int64_t i, int j, float v) {
    if (a.mode == 0) {
        if (j < a.ld_h) {
            __nv_bfloat16 h = __float2bfloat16_rn(__fmul_rn(v, a.col_scale ? a.col_scale[j] : a.scale));
            const uint16_t hb = *reinterpret_cast<uint16_t *>(&h);
            if (QLORA_IN_BOUNDS(i < a.Mp)) a.out_h[i * a.ld_h + j] = hb;
            if (a.out_h2 && j < a.r) a.out_h2[i * a.r + j] = hb;
        }
    } else if (a.mode == 1) {
        if (j < a.r) a.out_f[(int64_t)j * a.Mp + i] = v;
    } else {
        if (j < a.r) a.out_f[i * a.r + j] = v;
    }
}

__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t local_addr, uint32_t rank) {
    uint32_t ra;
    float4 v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local_addr), "r"(rank));
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(ra)
                 : "memory");
    return v;
}

template <bool kPMN, bool kQMN>
__global__ void __launch_bounds__(128, 1)
    lora_proj_kernel(const __grid_constant__ CUtensorMap map_p, const __grid_constant__ CUtensorMap map_q,
                     const ProjArgs a) {
    constexpr int kStages = kProjStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const int r64 = a.r64;
    const uint32_t q_bytes = (uint32_t)r64 * 128u;
    uint8_t *sP = smem;
    uint8_t *sQ = sP + kStages * kATileBytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(sQ + kStages * q_bytes);
    uint64_t *empty = full + kStages;
    uint64_t *done = empty + kStages;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(done + 1);
    volatile uint32_t *s_abort = s_tmem + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = (int)cluster_rank();  // the cluster spans the splits of one tile
    const int tile = blockIdx.x / a.splits;
    const int kt0 = (int)((int64_t)split * a.ktiles / a.splits);
    const int kt1 = (int)((int64_t)(split + 1) * a.ktiles / a.splits);
    const uint32_t ncols = r64 <= 64 ? 64u : (r64 <= 128 ? 128u : 256u);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
        *s_abort = 0u;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(s_tmem, ncols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;

    if (warp == 0 && lane == 0) {
        int s = 0;
        uint32_t ph = 0;
        for (int kt = kt0; kt < kt1; ++kt) {
            if (!mbar_wait(&empty[s], ph ^ 1u, s_abort)) break;
            mbar_arrive_expect_tx(&full[s], kATileBytes + q_bytes);
            uint8_t *dp = sP + s * kATileBytes;
            uint8_t *dq = sQ + s * q_bytes;
            if (kPMN) {
                tma_load_2d(dp, &map_p, &full[s], tile * 128, kt * 64);
                tma_load_2d(dp + 8192, &map_p, &full[s], tile * 128 + 64, kt * 64);
            } else {
                tma_load_2d(dp, &map_p, &full[s], kt * 64, tile * 128);
            }
            if (kQMN) {
                for (int jb = 0; jb < r64 / 64; ++jb) tma_load_2d(dq + jb * 8192, &map_q, &full[s], jb * 64, kt * 64);
            } else {
                tma_load_2d(dq, &map_q, &full[s], kt * 64, 0);
            }
            if (++s == kStages) { s = 0; ph ^= 1u; }
        }
    } else if (warp == 1 && lane == 0) {
        const uint32_t idesc = make_idesc_bf16((uint32_t)r64, kPMN, kQMN);
        const uint32_t p_base = smem_u32(sP), q_base = smem_u32(sQ);
        int s = 0;
        uint32_t ph = 0;
        for (int kt = kt0; kt < kt1; ++kt) {
            if (!mbar_wait(&full[s], ph, s_abort)) break;
            tc_fence_after();
            const uint32_t pa = p_base + (uint32_t)s * kATileBytes, qa = q_base + (uint32_t)s * q_bytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t adesc = kPMN ? make_sw128_desc(pa + kk * 2048u, 8192u, 1024u)
                                            : make_sw128_desc(pa + kk * 32u, 16u, 1024u);
                const uint64_t bdesc = kQMN ? make_sw128_desc(qa + kk * 2048u, 8192u, 1024u)
                                            : make_sw128_desc(qa + kk * 32u, 16u, 1024u);
                umma_bf16(tmem_base, adesc, bdesc, idesc, (kt > kt0 || kk > 0) ? 1u : 0u);
            }
            umma_commit(&empty[s]);
            if (++s == kStages) { s = 0; ph ^= 1u; }
        }
        umma_commit(done);  // also drains the MMAs on the error path
    }
    __syncwarp();
    // TMEM -> this CTA's fp32 partial tile in shared memory (the pipeline buffers are free once
    // `done` has completed).  Row stride r64 + 4 floats keeps the float4 stores conflict-free.
    const int pstride = r64 + 4;
    float *part = reinterpret_cast<float *>(smem);
    const int row = warp * 32 + lane;  // warp w reads TMEM lanes 32w..32w+31
    if (warp_wait(done, 0, s_abort)) {
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)(warp * 32) << 16);
        for (int c = 0; c < r64 / 32; ++c) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + (uint32_t)c * 32u, r);
            tmem_ld_wait();
            float4 *dst = reinterpret_cast<float4 *>(part + row * pstride + c * 32);
#pragma unroll
            for (int q = 0; q < 8; ++q)
                dst[q] = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                     __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
        }
    }
    tc_fence_before();
    cluster_barrier();
    // Sum over the splits in split order; this CTA owns rows [r0, r1) of the tile.
    {
        const int rows_per = (128 + a.splits - 1) / a.splits;
        const int r0 = split * rows_per, r1 = min(128, r0 + rows_per);
        const int nrow = max(0, r1 - r0), nj4 = r64 / 4;
        const uint32_t part_addr = smem_u32(part);
        for (int idx = threadIdx.x; idx < nrow * nj4; idx += blockDim.x) {
            // transposed output (mode 1): consecutive threads take consecutive rows
            const int rr = (a.mode == 1) ? r0 + idx % nrow : r0 + idx / nj4;
            const int j4 = ((a.mode == 1) ? idx / nrow : idx % nj4) * 4;
            const int64_t i = (int64_t)tile * 128 + rr;
            if (i >= a.Mp) continue;
            const uint32_t off = part_addr + (uint32_t)(rr * pstride + j4) * 4u;
            float4 acc = ld_dsmem_f4(off, 0);
            for (int sp = 1; sp < a.splits; ++sp) {
                const float4 v = ld_dsmem_f4(off, (uint32_t)sp);
                acc.x = __fadd_rn(acc.x, v.x);
                acc.y = __fadd_rn(acc.y, v.y);
                acc.z = __fadd_rn(acc.z, v.z);
                acc.w = __fadd_rn(acc.w, v.w);
            }
            proj_store(a, i, j4, acc.x);
            proj_store(a, i, j4 + 1, acc.y);
            proj_store(a, i, j4 + 2, acc.z);
            proj_store(a, i, j4 + 3, acc.w);
        }
    }
    cluster_barrier();  // peers read this CTA's shared memory until here
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, ncols);
    }
}

// ---------------------------------------------------------------------------------------
// Rebuilt block scales for the fused kernel: out[kb, n] = fmaf(q_b, fl32(c2_g / 127), mu) for
// block b = n * KB + kb (transposed, so that a weight tile's scales are one contiguous TMA
// box).  Used by the CTA-pair kernel; the small-M kernel rebuilds the scales itself.
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) dq_scales_t_kernel(const int8_t *__restrict__ q, const float *__restrict__ c2,
                                                          const float *__restrict__ mu_p, int64_t N, int KB,
                                                          float *__restrict__ out, int64_t ld) {
    __shared__ float tile[32][33];
    const float mu = *mu_p;
    const int64_t n0 = (int64_t)blockIdx.x * 32;
    const int kb0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int i = ty; i < 32; i += 8) {
        const int64_t n = n0 + i;
        const int kb = kb0 + tx;
        float v = 0.0f;
        if (n < N && kb < KB) {
            const int64_t b = n * KB + kb;
            v = __fmaf_rn((float)q[b], __fdiv_rn(c2[b >> 8], 127.0f), mu);
        }
        tile[i][tx] = v;
    }
    __syncthreads();
    for (int i = ty; i < 32; i += 8) {
        const int kb = kb0 + i;
        const int64_t n = n0 + tx;
        if (n < N && kb < KB) out[(int64_t)kb * ld + n] = tile[tx][i];
    }
}

// ---------------------------------------------------------------------------------------
// Small elementwise kernels
// ---------------------------------------------------------------------------------------
__global__ void splitk_reduce_kernel(const float *__restrict__ partial, int splits, int64_t total,
                                     uint16_t *__restrict__ out) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        float acc = partial[i];
        for (int s = 1; s < splits; ++s) acc = __fadd_rn(acc, partial[(int64_t)s * total + i]);
        __nv_bfloat16 h = __float2bfloat16_rn(acc);
        out[i] = *reinterpret_cast<uint16_t *>(&h);
    }
}

__global__ void pad_2d_kernel(const uint16_t *__restrict__ src, int64_t rows_src, int64_t cols_src,
                              uint16_t *__restrict__ dst, int64_t rows_dst, int64_t cols_dst) {
    const int64_t total = rows_dst * cols_dst;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = e / cols_dst, j = e % cols_dst;
        dst[e] = (i < rows_src && j < cols_src) ? src[i * cols_src + j] : (uint16_t)0;
    }
}

// ---------------------------------------------------------------------------------------
// Plans and launchers
// ---------------------------------------------------------------------------------------
// Pipeline depth of the fused kernel: as many stages (even, <= 8) as fit in ~220 KB, so that a
// small token tile keeps enough codes in flight to cover HBM latency.  Each CTA of the pair
// holds BN/2 token rows per stage.
static size_t fused_stage_bytes(int BN, int mt) {
    return kATileBytes + (size_t)mt * (BN / 2) * 128 + kCStageBytes;
}
static int fused_stages(int BN, int mt) {
    int st = (int)((220u * 1024u) / fused_stage_bytes(BN, mt));
    st = std::min(8, st) & ~1;
    return std::max(4, st);
}
// The fused kernel allocates all 512 TMEM columns, so it must be alone on its SM: asking for
// more than half of the SM's shared memory guarantees one resident CTA.
static size_t fused_smem_bytes(int BN, int mt, int stages) {
    const size_t need = (size_t)stages * fused_stage_bytes(BN, mt) + (mt == 2 ? kOutStageBytes : 0) + 512;
    return std::max<size_t>(need, 120 * 1024);
}
static size_t proj_smem_bytes(int r64) { return 1024 + (size_t)kProjStages * (kATileBytes + (size_t)r64 * 128) + 128; }

FusedPlan plan_fused(int64_t M, int64_t wdim, int64_t kt_main, int r64, int num_sms) {
    FusedPlan pl{};
    pl.kt_main = (int)kt_main;
    pl.kt_lora = r64 / 64;
    if (M <= 32) {
        plan_small(pl, M, wdim, kt_main, num_sms);
        return pl;
    }
    pl.small = false;
    int64_t bn = M >= 256 ? 256 : ((M + 31) / 32) * 32;
    if (bn < 32) bn = 32;
    pl.BN = (int)bn;
    pl.mt = M >= 512 ? 2 : 1;  // two 256-token tiles per decoded weight tile
    pl.act_rows = pl.BN / 2;
    pl.stages = fused_stages(pl.BN, pl.mt);
    pl.m_tiles = (int)((M + bn * pl.mt - 1) / (bn * pl.mt));
    pl.w_tiles = (int)((wdim + 255) / 256);  // 256-row tiles, one per CTA pair
    pl.splits = 1;
    const int pairs = std::max(1, num_sms / 2);
    const int64_t units = (int64_t)pl.w_tiles * pl.m_tiles;
    if (pl.m_tiles == 1 && units < 2LL * pairs) {
        // small token count: split the contraction so that the units fill whole waves
        int best = 1;
        double best_eff = 0.0;
        for (int s = 1; s <= 16 && s <= kt_main / 4; ++s) {
            const int64_t us = units * s;
            const double eff = (double)us / (double)(((us + pairs - 1) / pairs) * pairs);
            if (eff > best_eff + 1e-9) { best_eff = eff; best = s; }
            if (eff >= 0.9) break;
        }
        pl.splits = best;
    }
    const int64_t total = units * pl.splits;
    pl.grid = 2 * (int)std::min<int64_t>(total, pairs);
    pl.partial_bytes = pl.splits > 1 ? (size_t)pl.splits * (size_t)M * (size_t)wdim * 4 : 0;
    return pl;
}

// Clusters of `s` projection CTAs (shared memory for rank r64) resident at once on the current
// device; cached per (device, s, r64).  A cluster's CTAs must share a GPC, so large clusters fit
// fewer times than the SM count suggests.
static int proj_max_clusters(int s, int r64, int fallback) {
    static std::mutex mu;
    static int cache[8][9][3];  // [device < 8][s][r64 = 64, 128, 256]; zero until queried
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 8 || s < 1 || s > 8) {
        (void)cudaGetLastError();
        return fallback;
    }
    const int ri = r64 <= 64 ? 0 : (r64 <= 128 ? 1 : 2);
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev][s][ri] > 0) return cache[dev][s][ri];
    const size_t smem = proj_smem_bytes(r64);
    int n = 0;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)s, 1, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)s;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaFuncSetAttribute(lora_proj_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&n, lora_proj_kernel<false, false>, &cfg) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        return fallback;
    }
    cache[dev][s][ri] = n;
    return n;
}

ProjPlan plan_proj(int64_t Mp, int64_t Kc, int r64, int num_sms) {
    ProjPlan pl{};
    pl.tiles = (int)((Mp + 127) / 128);
    pl.ktiles = (int)((Kc + 63) / 64);
    // The splits of a tile form one cluster (at most 8, the portable size).  Cost of a choice:
    // waves of resident clusters x (k-steps per CTA + ~2 steps of set-up and reduction).
    int best = 1;
    int64_t best_cost = INT64_MAX;
    for (int s = 1; s <= std::min(8, pl.ktiles); ++s) {
        const int fit = std::max(1, proj_max_clusters(s, r64, std::max(1, num_sms / (2 * s))));
        const int64_t waves = (pl.tiles + fit - 1) / fit;
        const int64_t cost = waves * ((pl.ktiles + s - 1) / s + 2);
        if (cost < best_cost) {
            best_cost = cost;
            best = s;
        }
    }
    pl.splits = best;
    return pl;
}

// Clusters of two that can be resident at once for a given kernel and shared-memory size
// (normally one per SM pair), cached per configuration.
template <bool kDX, int kSt, int kMT>
static int max_pairs(size_t smem, int fallback) {
    static std::mutex mu;
    static size_t cached_smem = 0;
    static int cached = 0;
    static int cached_dev = -1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fallback;
    std::lock_guard<std::mutex> lock(mu);
    if (cached_smem == smem && cached_dev == dev) return cached;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2 * (unsigned)fallback, 1, 1);
    cfg.blockDim = dim3(kFusedThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, nf4_lora_gemm_kernel<kDX, kSt, kMT>, &cfg) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        return fallback;
    }
    cached_smem = smem;
    cached_dev = dev;
    cached = n;
    return n;
}

template <bool kDX, int kSt, int kMT = 1>
static cudaError_t launch_fused_t(const CUtensorMap &mc, const CUtensorMap &ms, const CUtensorMap &ma,
                                  const CUtensorMap &ml, const CUtensorMap &mo, const FusedArgs &args,
                                  const FusedPlan &plan, cudaStream_t st) {
    const size_t smem = fused_smem_bytes(plan.BN, kMT, kSt);
    cudaError_t e = cudaFuncSetAttribute(nf4_lora_gemm_kernel<kDX, kSt, kMT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // units are dealt to pairs round-robin, so any even grid is correct; more pairs than can be
    // resident would only run as a second, serial wave
    const int grid = 2 * std::max(1, std::min(plan.grid / 2, max_pairs<kDX, kSt, kMT>(smem, plan.grid / 2)));
    nf4_lora_gemm_kernel<kDX, kSt, kMT><<<grid, kFusedThreads, smem, st>>>(mc, ms, ma, ml, mo, args);
    return cudaSuccess;
}

cudaError_t launch_fused(bool dx, const CUtensorMap &map_codes, const CUtensorMap &map_scales,
                         const CUtensorMap &map_act, const CUtensorMap &map_lora, const CUtensorMap &map_out,
                         const FusedArgs &args, const FusedPlan &plan, cudaStream_t st) {
    cudaError_t e;
    const int S = plan.stages;
    if (plan.small) {
        e = launch_small(dx, map_codes, map_act, map_lora, args, plan, st);
    } else if (plan.mt == 2) {
        e = dx ? launch_fused_t<true, 4, 2>(map_codes, map_scales, map_act, map_lora, map_out, args, plan, st)
               : launch_fused_t<false, 4, 2>(map_codes, map_scales, map_act, map_lora, map_out, args, plan, st);
    } else if (dx)
        e = S == 8   ? launch_fused_t<true, 8>(map_codes, map_scales, map_act, map_lora, map_out, args, plan, st)
            : S == 6 ? launch_fused_t<true, 6>(map_codes, map_scales, map_act, map_lora, map_out, args, plan, st)
                     : launch_fused_t<true, 4>(map_codes, map_scales, map_act, map_lora, map_out, args, plan, st);
    else
        e = S == 8   ? launch_fused_t<false, 8>(map_codes, map_scales, map_act, map_lora, map_out, args, plan, st)
            : S == 6 ? launch_fused_t<false, 6>(map_codes, map_scales, map_act, map_lora, map_out, args, plan, st)
                     : launch_fused_t<false, 4>(map_codes, map_scales, map_act, map_lora, map_out, args, plan, st);
    if (e != cudaSuccess) return e;
    count_launch();
    return cudaGetLastError();
}

static int ew_grid(int64_t n, int num_sms) {
    int64_t g = (n + 255) / 256;
    return (int)std::max<int64_t>(1, std::min<int64_t>(g, (int64_t)num_sms * 8));
}

cudaError_t launch_splitk_reduce(const float *partial, int splits, int64_t rows, int64_t cols, uint16_t *out,
                                 int num_sms, cudaStream_t st) {
    const int64_t total = rows * cols;
    splitk_reduce_kernel<<<ew_grid(total, num_sms), 256, 0, st>>>(partial, splits, total, out);
    count_launch();
    return cudaGetLastError();
}

template <bool PM, bool QM>
static cudaError_t launch_proj_t(const CUtensorMap &map_p, const CUtensorMap &map_q, const ProjArgs &args,
                                 cudaStream_t st) {
    const size_t smem = proj_smem_bytes(args.r64);
    cudaError_t e =
        cudaFuncSetAttribute(lora_proj_kernel<PM, QM>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(args.tiles * args.splits));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)args.splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, lora_proj_kernel<PM, QM>, map_p, map_q, args);
}

cudaError_t launch_proj(bool p_mn, bool q_mn, const CUtensorMap &map_p, const CUtensorMap &map_q, const ProjArgs &args,
                        cudaStream_t st) {
    cudaError_t e;
    if (!p_mn && !q_mn) e = launch_proj_t<false, false>(map_p, map_q, args, st);
    else if (!p_mn && q_mn) e = launch_proj_t<false, true>(map_p, map_q, args, st);
    else if (p_mn && !q_mn) e = launch_proj_t<true, false>(map_p, map_q, args, st);
    else e = launch_proj_t<true, true>(map_p, map_q, args, st);
    if (e != cudaSuccess) return e;
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_dq_scales_t(const int8_t *q, const float *c2, const float *mu, int64_t N, int KB, float *out,
                               cudaStream_t st, int64_t ld) {
    dim3 grid((unsigned)((N + 31) / 32), (unsigned)((KB + 31) / 32));
    dq_scales_t_kernel<<<grid, 256, 0, st>>>(q, c2, mu, N, KB, out, ld > 0 ? ld : N);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_pad_2d(const uint16_t *src, int64_t rows_src, int64_t cols_src, uint16_t *dst, int64_t rows_dst,
                          int64_t cols_dst, int num_sms, cudaStream_t st) {
    pad_2d_kernel<<<ew_grid(rows_dst * cols_dst, num_sms), 256, 0, st>>>(src, rows_src, cols_src, dst, rows_dst,
                                                                         cols_dst);
    count_launch();
    return cudaGetLastError();
}

}  // namespace qlora
