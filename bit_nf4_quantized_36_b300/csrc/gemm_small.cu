// gemm_small.cu -- the fused layer for small token counts (M <= 32) on the tensor cores.
// Part of the single translation unit libqlora.cu (after gemm.cu, whose decode helpers and
// pipeline constants it uses).
#include "qlora_common.cuh"
#include "qlora_kernels.cuh"

namespace qlora {

// ---------------------------------------------------------------------------------------
// Small token counts (M <= 32, e.g. decoding).  Each weight is used by at most 32 tokens, so the
// call is bound by streaming the packed codes and by the decode arithmetic (byte permutes on the
// integer pipe), not by tensor FLOPs.  Differences from the pair kernel above:
//   - single-CTA MMAs (M = 128, N = BN in {16, 32}): a pair MMA costs about twice the issue
//     time per weight at this N;
//   - two issuer warps take alternate k-steps into separate accumulators (the per-instruction
//     issue cost, not the tensor pipe, bounds one issuer at small N); the epilogue adds them;
//   - two rings: a deep one of TMA slots (codes + token tile, 8 KB) that keeps enough bytes in
//     flight to cover HBM latency, and a short one of decoded 16 KB weight tiles, filled by
//     three decode groups (12 warps) that take alternate k-steps.  A decoded slot is reused
//     once the MMAs of the step kSmallA earlier have completed, which the commit on that
//     step's TMA slot reports;
//   - the decode threads rebuild each block scale s'_b = fmaf(q_b, fl(c2_g / 127), mu) from the
//     int8 code and the group constant themselves (bit-identical to nf4_dequantize), so the call
//     reads 1 byte of scale per 64 weights instead of a rebuilt fp32 copy written beforehand.
// ---------------------------------------------------------------------------------------
static constexpr int kSmallIssuers = 2;
static constexpr int kSmallGroups = 3;
static constexpr int kSmallC = 16;                // TMA slots
static constexpr int kSmallA = 6;                 // decoded tiles (a multiple of kSmallGroups, < kSmallC)
static constexpr int kSmallEpiWarp0 = 1 + kSmallIssuers;   // warps 3..6
static constexpr int kSmallDecodeWarp0 = kSmallEpiWarp0 + 4;  // warps 7..18
static constexpr int kSmallThreads = (kSmallDecodeWarp0 + 4 * kSmallGroups) * 32;  // 608
static constexpr uint32_t kSmallTmemCols = 128;   // 2 buffers x 2 issuers x BN (<= 32)

__device__ __forceinline__ int32_t ldg_s8_early(const int8_t *p) {
    // volatile: issued where written, so its latency overlaps the stage waits that follow
    int32_t v;
    asm volatile("ld.global.nc.s8 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

template <bool kDX, int kBN>
__global__ void __launch_bounds__(kSmallThreads, 1)
    nf4_lora_gemm_small_kernel(const __grid_constant__ CUtensorMap map_codes, const __grid_constant__ CUtensorMap map_act,
                               const __grid_constant__ CUtensorMap map_lora, const FusedArgs p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {  // see nf4_lora_gemm_kernel
        if (threadIdx.x == 0) atomicOr(&g_error_word, kErrLayout);
        return;
    }
    constexpr uint32_t b_bytes = (uint32_t)kBN * 128u;
    constexpr uint32_t c_bytes = kCodesTileBytes + b_bytes;  // TMA slot: codes, then the token tile
    uint8_t *sA = smem_raw;                                   // kSmallA x 16 KB
    uint8_t *sC = sA + kSmallA * kATileBytes;                 // kSmallC x c_bytes
    uint64_t *bars = reinterpret_cast<uint64_t *>(sC + kSmallC * c_bytes);
    uint64_t *full_c = bars;                      // [kSmallC] TMA slot landed (transaction count)
    uint64_t *empty_c = bars + kSmallC;           // [kSmallC] MMAs of the slot's step finished
    uint64_t *full_a = bars + 2 * kSmallC;        // [kSmallA] decoded tile written (4 warps)
    uint64_t *acc_full = full_a + kSmallA;        // [2], one commit per issuer
    uint64_t *acc_empty = acc_full + 2;           // [2], four epilogue warps
    uint64_t *drain = acc_empty + 2;              // [kSmallIssuers]
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(drain + kSmallIssuers);
    volatile uint32_t *s_abort = s_tmem + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSmallC; ++s) {
            mbar_init(&full_c[s], 1);
            mbar_init(&empty_c[s], 1);
        }
        for (int s = 0; s < kSmallA; ++s) mbar_init(&full_a[s], 4);
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], kSmallIssuers);
            mbar_init(&acc_empty[a], 4);
        }
        for (int i = 0; i < kSmallIssuers; ++i) mbar_init(&drain[i], 1);
        *s_abort = 0u;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(s_tmem, kSmallTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    const int total_units = p.w_tiles * p.m_tiles * p.splits;

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------------
        if (lane == 0) {
            tma_prefetch_desc(&map_codes);
            tma_prefetch_desc(&map_act);
            tma_prefetch_desc(&map_lora);
            int c = 0;
            uint32_t ph = 0;
            uint32_t issued_parity[kSmallC];
            bool issued[kSmallC];
            for (int i = 0; i < kSmallC; ++i) issued[i] = false, issued_parity[i] = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < total_units && ok; u += gridDim.x) {
                const UnitInfo ui = unit_info(p, u);
                for (int j = 0; j < ui.nk; ++j) {
                    if (!mbar_wait(&empty_c[c], ph ^ 1u, s_abort)) { ok = false; break; }
                    const bool lora = (ui.kt0 + j) >= ui.kt1;
                    uint8_t *slot = sC + c * c_bytes;
                    if (!lora) {
                        const int kt = ui.kt0 + j;
                        mbar_arrive_expect_tx(&full_c[c], c_bytes);
                        if (kDX) tma_load_2d(slot, &map_codes, &full_c[c], ui.w_tile * 64, kt * 64);
                        else tma_load_2d(slot, &map_codes, &full_c[c], kt * 32, ui.w_tile * 128);
                        tma_load_2d(slot + kCodesTileBytes, &map_act, &full_c[c], kt * 64, ui.m_tile * kBN);
                    } else {
                        const int lt = j - (ui.kt1 - ui.kt0);
                        mbar_arrive_expect_tx(&full_c[c], b_bytes);
                        tma_load_2d(slot + kCodesTileBytes, &map_lora, &full_c[c], lt * 64, ui.m_tile * kBN);
                    }
                    issued[c] = true;
                    issued_parity[c] = ph;
                    if (++c == kSmallC) { c = 0; ph ^= 1u; }
                }
            }
            if (!ok) {
                for (int i = 0; i < kSmallC; ++i) {
                    if (!issued[i]) continue;
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(&full_c[i], issued_parity[i]) && globaltimer_ns() - t0 < 20000000ull) {}
                }
            }
        }
        __syncwarp();
    } else if (warp <= kSmallIssuers) {
        // ------------------------------ MMA issuers --------------------------------------
        // Issuer i takes the k-steps g with g % kSmallIssuers == i of the CTA's step sequence
        // and accumulates into its own TMEM columns.
        const int me = warp - 1;
        if (lane == 0) {
            const uint32_t idesc = make_idesc_bf16((uint32_t)kBN, kDX, false);
            const uint32_t a_base = smem_u32(sA), c_base = smem_u32(sC);
            int g = 0;  // step counter
            int lt = 0;
            bool ok = true, any = false;
            for (int u = blockIdx.x; u < total_units && ok; u += gridDim.x, ++lt) {
                const UnitInfo ui = unit_info(p, u);
                const int a = lt & 1;
                const uint32_t d_tmem = tmem_base + (uint32_t)((a * kSmallIssuers + me) * kBN);
                bool first = true;
                for (int j = 0; j < ui.nk; ++j, ++g) {
                    if (g % kSmallIssuers != me) continue;
                    const int sa = g % kSmallA, sc = g % kSmallC;
                    if (first && !mbar_wait(&acc_empty[a], ((lt >> 1) & 1) ^ 1u, s_abort)) { ok = false; break; }
                    if (!mbar_wait(&full_a[sa], (uint32_t)(g / kSmallA) & 1u, s_abort)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = a_base + (uint32_t)sa * kATileBytes;
                    const uint32_t b_addr = c_base + (uint32_t)sc * c_bytes + kCodesTileBytes;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t adesc = kDX ? make_sw128_desc(a_addr + kk * 2048u, 8192u, 1024u)
                                                   : make_sw128_desc(a_addr + kk * 32u, 16u, 1024u);
                        const uint64_t bdesc = make_sw128_desc(b_addr + kk * 32u, 16u, 1024u);
                        umma_bf16(d_tmem, adesc, bdesc, idesc, (!first || kk > 0) ? 1u : 0u);
                    }
                    first = false;
                    any = true;
                    umma_commit(&empty_c[sc]);
                }
                if (!ok) break;
                // an issuer without a step in this unit still waits for the buffer's previous
                // use to be drained, so that its arrival lands in this unit's phase
                if (first && !mbar_wait(&acc_empty[a], ((lt >> 1) & 1) ^ 1u, s_abort)) { ok = false; break; }
                umma_commit(&acc_full[a]);  // also without a step of its own in the unit (the epilogue knows)
            }
            if (!ok && any) {
                umma_commit(&drain[me]);
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&drain[me], 0) && globaltimer_ns() - t0 < 20000000ull) {}
            }
        }
        __syncwarp();
    } else if (warp < kSmallDecodeWarp0) {
        // ------------------------------ epilogue -----------------------------------------
        const int quarter = warp & 3;
        int lt = 0, g0 = 0;
        for (int u = blockIdx.x; u < total_units; u += gridDim.x, ++lt) {
            const UnitInfo ui = unit_info(p, u);
            // a unit of one k-step leaves the other issuer's accumulator unwritten
            const bool has0 = ui.nk >= 2 || (g0 & 1) == 0, has1 = ui.nk >= 2 || (g0 & 1) == 1;
            g0 += ui.nk;
            const int a = lt & 1;
            if (!warp_wait(&acc_full[a], (lt >> 1) & 1, s_abort)) break;
            tc_fence_after();
            const int64_t f = (int64_t)ui.w_tile * 128 + quarter * 32 + lane;
            const int m0 = ui.m_tile * kBN;
            const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(a * kSmallIssuers * kBN);
            float acc[kBN];
#pragma unroll
            for (int c = 0; c < kBN / 16; ++c) {
                uint32_t r0[16], r1[16];
                tmem_ld_32x32b_x16(taddr + (uint32_t)(c * 16), r0);
                tmem_ld_32x32b_x16(taddr + (uint32_t)(kBN + c * 16), r1);
                tmem_ld_wait();
#pragma unroll
                for (int jj = 0; jj < 16; ++jj)
                    acc[c * 16 + jj] = __fadd_rn(has0 ? __uint_as_float(r0[jj]) : 0.0f, has1 ? __uint_as_float(r1[jj]) : 0.0f);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[a]);
            if (f < p.wdim) {
#pragma unroll
                for (int jj = 0; jj < kBN; ++jj) {
                    const int m = m0 + jj;
                    if (m >= p.M) break;
                    if (p.splits == 1) {
                        __nv_bfloat16 h = __float2bfloat16_rn(acc[jj]);
                        p.out[(int64_t)m * p.wdim + f] = *reinterpret_cast<uint16_t *>(&h);
                    } else {
                        p.partial[((int64_t)ui.split * p.M + m) * p.wdim + f] = acc[jj];
                    }
                }
            }
        }
    } else {
        // ------------------------------ decode warps -------------------------------------
        // Group q (4 warps, one 128-byte A row per thread) takes the k-steps g with
        // g % kSmallGroups == q; decoded tile g % kSmallA, TMA slot g % kSmallC.
        const int t = (threadIdx.x - kSmallDecodeWarp0 * 32) & 127;
        const int group = (threadIdx.x - kSmallDecodeWarp0 * 32) >> 7;
        const uint32_t a_base = smem_u32(sA);
        const bool lora_vec = (p.lora_ld % 8) == 0;
        uint32_t row_off, code_off;
        int nl = 0, kbl = 0;
        if (!kDX) {
            row_off = (uint32_t)t * 128u;
            code_off = (uint32_t)t * 32u;
        } else {
            nl = t >> 1;
            kbl = t & 1;
            row_off = (uint32_t)kbl * 8192u + (uint32_t)nl * 128u;
            code_off = (uint32_t)nl * 64u + (uint32_t)kbl * 32u;
        }
        const uint32_t r7 = (row_off >> 7) & 7u;
        int64_t g_cached = -1;
        float k_cached = 0.0f;
        const float mu = __ldg(p.scale_mu);
        int g = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < total_units && ok; u += gridDim.x) {
            const UnitInfo ui = unit_info(p, u);
            const int64_t n_fwd = (int64_t)ui.w_tile * 128 + t;
            const int kblock = ui.w_tile * 2 + kbl;
            for (int j = 0; j < ui.nk; ++j, ++g) {
                if (g % kSmallGroups != group) continue;
                const int sa = g % kSmallA, sc = g % kSmallC;
                const bool lora = (ui.kt0 + j) >= ui.kt1;
                const int kt = lora ? j - (ui.kt1 - ui.kt0) : ui.kt0 + j;
                bool valid;
                int64_t srow = 0, skb = 0;
                uint4 lv[8];
                if (!kDX) {
                    valid = n_fwd < p.N;
                    srow = n_fwd;
                    skb = kt;
                    if (lora && valid) {
                        const uint16_t *row = p.lora_src + n_fwd * p.lora_ld;
                        load_row32(row, (int64_t)kt * 64, p.r, lora_vec, *reinterpret_cast<uint4(*)[4]>(&lv[0]));
                        load_row32(row, (int64_t)kt * 64 + 32, p.r, lora_vec, *reinterpret_cast<uint4(*)[4]>(&lv[4]));
                    }
                } else {
                    const int64_t n = (int64_t)kt * 64 + nl;
                    valid = kblock < p.KB && n < (lora ? (int64_t)p.r : p.N);
                    srow = n;
                    skb = kblock;
                    if (lora && valid) {
                        const uint4 *src = reinterpret_cast<const uint4 *>(p.lora_src + n * p.lora_ld + (int64_t)kblock * 64);
#pragma unroll
                        for (int i = 0; i < 8; ++i) lv[i] = __ldg(src + i);
                    }
                }
                // block scale: the code byte is loaded before the waits, converted after them
                const bool scaled = valid && !lora;
                const int64_t b = srow * p.KB + skb;
                const int32_t q = scaled ? ldg_s8_early(p.scale_q + b) : 0;
                if (scaled && (b >> 8) != g_cached) {
                    g_cached = b >> 8;
                    k_cached = __fdiv_rn(__ldg(p.scale_c2 + g_cached), 127.0f);
                }
                // the decoded tile is free once the MMAs of step g - kSmallA completed
                uint32_t okw = 1;
                if (lane == 0) {
                    if (g >= kSmallA) {
                        const int gp = g - kSmallA;
                        okw = mbar_wait(&empty_c[gp % kSmallC], (uint32_t)(gp / kSmallC) & 1u, s_abort) ? 1u : 0u;
                    }
                    if (okw) okw = mbar_wait(&full_c[sc], (uint32_t)(g / kSmallC) & 1u, s_abort) ? 1u : 0u;
                }
                okw = __shfl_sync(0xffffffffu, okw, 0);
                __syncwarp();
                if (!okw) { ok = false; break; }
                const uint32_t row_addr = a_base + (uint32_t)sa * kATileBytes + row_off;
                if (!valid) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) st_shared_v4(row_addr + (((uint32_t)i ^ r7) << 4), make_uint4(0, 0, 0, 0));
                } else if (!lora) {
                    const uint8_t *cst = sC + sc * c_bytes;
                    const uint4 c0 = *reinterpret_cast<const uint4 *>(cst + code_off);
                    const uint4 c1 = *reinterpret_cast<const uint4 *>(cst + code_off + 16);
                    uint32_t lo[4], hi[4];
                    build_table(__fmaf_rn((float)q, k_cached, mu), p.tab, lo, hi);
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
                if (lane == 0) mbar_arrive(&full_a[sa]);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kSmallTmemCols);
    }
}

static size_t small_smem_bytes(int BN) {
    return (size_t)kSmallA * kATileBytes + (size_t)kSmallC * (kCodesTileBytes + (size_t)BN * 128) + 512;
}

// Small-M plan: 128-row tiles, all tokens in one tile, and the contraction split so that the
// units fill whole waves.  Cost per SM, in bytes streamed: waves x codes per unit, plus the fp32
// partials written and re-read by the split reduction (spread over all SMs) and a fixed charge
// for the extra launch.
void plan_small(FusedPlan &pl, int64_t M, int64_t wdim, int64_t kt_main, int num_sms) {
    pl.small = true;
    pl.mt = 1;
    pl.BN = M <= 16 ? 16 : 32;
    pl.act_rows = pl.BN;
    pl.stages = kSmallC;
    pl.m_tiles = 1;
    pl.w_tiles = (int)((wdim + 127) / 128);
    int best = 1;
    double best_cost = 0.0;
    // every split keeps at least kSmallIssuers main k-steps so that each issuer has work
    const int64_t smax = std::max<int64_t>(1, std::min<int64_t>(32, kt_main / kSmallIssuers));
    for (int64_t sp = 1; sp <= smax; ++sp) {
        const int64_t units = (int64_t)pl.w_tiles * sp;
        const int64_t waves = (units + num_sms - 1) / num_sms;
        double cost = (double)waves * (double)((kt_main + sp - 1) / sp) * (double)kCodesTileBytes;
        if (sp > 1) cost += 8.0 * (double)sp * (double)M * (double)wdim / (double)num_sms + 65536.0;
        if (sp == 1 || cost < best_cost) { best_cost = cost; best = (int)sp; }
    }
    pl.splits = best;
    pl.grid = (int)std::min<int64_t>((int64_t)pl.w_tiles * pl.splits, num_sms);
    pl.partial_bytes = pl.splits > 1 ? (size_t)pl.splits * (size_t)M * (size_t)wdim * 4 : 0;
}

template <bool kDX, int kBN>
static cudaError_t launch_small_t(const CUtensorMap &mc, const CUtensorMap &ma, const CUtensorMap &ml,
                                  const FusedArgs &args, const FusedPlan &plan, cudaStream_t st) {
    const size_t smem = small_smem_bytes(kBN);
    cudaError_t e = cudaFuncSetAttribute(nf4_lora_gemm_small_kernel<kDX, kBN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    nf4_lora_gemm_small_kernel<kDX, kBN><<<plan.grid, kSmallThreads, smem, st>>>(mc, ma, ml, args);
    return cudaSuccess;
}

cudaError_t launch_small(bool dx, const CUtensorMap &map_codes, const CUtensorMap &map_act, const CUtensorMap &map_lora,
                         const FusedArgs &args, const FusedPlan &plan, cudaStream_t st) {
    if (dx)
        return plan.BN == 16 ? launch_small_t<true, 16>(map_codes, map_act, map_lora, args, plan, st)
                             : launch_small_t<true, 32>(map_codes, map_act, map_lora, args, plan, st);
    return plan.BN == 16 ? launch_small_t<false, 16>(map_codes, map_act, map_lora, args, plan, st)
                         : launch_small_t<false, 32>(map_codes, map_act, map_lora, args, plan, st);
}

}  // namespace qlora
