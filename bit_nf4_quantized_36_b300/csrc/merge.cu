// merge.cu -- rank-r updates of a [rows, K] bf16 matrix on the tensor cores:
//   mode 0 (the adapter merge) and mode 1 (the LoRA branch of dX under dropout, below).
//
// Mode 0, the adapter merged into the dequantized base weight:
//   W_m[n, k] = bf16(W^[n, k] + s (B A)[n, k]),   s = alpha / r,
// with W^ the bf16 dequantized NF4 weight (the nf4_dequantize values) and B A accumulated in fp32.
// Source: "QLoRA" glossary (ultralytics), "Compromissos" and "QLoRA e metodos relacionados": to
// merge the adapters the base weight is first dequantized to 16 bits, and the merged model keeps
// 16-bit weights.
//
// One pass, bound by HBM (0.516 B of codes and scales read and 2 B written per weight):
//   - a unit is a 128 x 256 tile of W_m; TMA stages its packed codes and, per 64-wide chunk of the
//     rank, the B rows (K-major) and A columns (MN-major);
//   - one thread issues tcgen05.mma (M = 128, N = 256, K = 16) into a double-buffered TMEM
//     accumulator: the rank-r update costs a few MMAs per tile;
//   - eight epilogue warps (two per TMEM lane quarter, one per 128-column half) read the
//     accumulator, decode the tile's codes with the per-block table (exact bf16 W^), form
//     fma(s, acc, W^) in fp32, round to bf16, and store [128 rows][64 cols] tiles through
//     128-byte-swizzled shared memory and TMA.
//
// Mode 1, the dropout backward (dropout.cu): dX[m, k] = bf16(dX0[m, k] + D[m, k] (V A)[m, k]) in
// place, with dX0 the fused kernel's base term (dY W^), V = bf16(s dY B), and D = 1 / (1 - p) where
// the adapter input element was kept, 0 where dropped (a bit mask from the forward's generator).
// The same pipeline with V as the K-major operand; the epilogue reads dX0 from global memory and
// the mask bits instead of decoding codes.
#include "qlora_common.cuh"
#include "qlora_kernels.cuh"

namespace qlora {

static constexpr int kMrgThreads = 320;       // warp 0 TMA, warp 1 MMA, warps 2..9 epilogue
static constexpr int kMrgEpiWarp0 = 2;
static constexpr uint32_t kMrgBBytes = 128u * 128u;        // 128 rows x 64 rank (bf16), SW128
static constexpr uint32_t kMrgABytes = 4u * 64u * 128u;    // 4 MN blocks of 64 k x 64 rank, SW128
static constexpr uint32_t kMrgOpBytes = kMrgBBytes + kMrgABytes;
static constexpr uint32_t kMrgCodesBytes = 128u * 128u;    // 128 rows x 256 codes
static constexpr uint32_t kMrgOutBytes = 128u * 128u;      // staging: 128 rows x 64 bf16, SW128
static constexpr uint32_t kMrgWarpOutBytes = 32u * 128u;   // one epilogue warp's 32 rows of it
static constexpr uint32_t kMrgSmem = 2 * kMrgOpBytes + 2 * kMrgCodesBytes + 4 * kMrgOutBytes + 256;

struct MergeArgs {
    int64_t N, K;               // rows (weight rows, or tokens in mode 1), columns
    int32_t KB;                 // K / 64
    int32_t n_tiles, k_tiles;   // 128-row and 256-column tiles
    int32_t rc;                 // 64-wide chunks of the rank
    float s;                    // alpha / r
    const int8_t *scale_q;
    const float *scale_c2;
    const float *scale_mu;
    NF4Tables tab;
    const uint32_t *mask_bits;  // mode 1: [N * K / 32] kept-element bits
    float inv;                  // mode 1: 1 / (1 - p)
    const uint16_t *base;       // mode 1: dX0 [N, K] bf16 (the output, updated in place)
};

__device__ __forceinline__ uint4 ld_global_v4(const uint4 *ptr) {
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(ptr));
    return v;
}

template <int kMode>
__global__ void __launch_bounds__(kMrgThreads, 1)
    nf4_merge_kernel(const __grid_constant__ CUtensorMap map_codes, const __grid_constant__ CUtensorMap map_b,
                     const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_out,
                     const MergeArgs p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {  // the swizzled tiles need 1024-byte alignment; no slack is requested
        if (threadIdx.x == 0) atomicOr(&g_error_word, kErrLayout);
        return;
    }
    uint8_t *sOp = smem_raw;                          // [2] B chunk then A chunk
    uint8_t *sCodes = sOp + 2 * kMrgOpBytes;          // [2]
    uint8_t *sOut = sCodes + 2 * kMrgCodesBytes;      // [half][2]
    uint64_t *bars = reinterpret_cast<uint64_t *>(sOut + 4 * kMrgOutBytes);
    uint64_t *op_full = bars;           // [2] B and A chunk landed
    uint64_t *op_empty = bars + 2;      // [2] MMAs reading the chunk finished
    uint64_t *codes_full = bars + 4;    // [2]
    uint64_t *codes_empty = bars + 6;   // [2] eight epilogue warps done with the codes
    uint64_t *acc_full = bars + 8;      // [2]
    uint64_t *acc_empty = bars + 10;    // [2] eight epilogue warps done with the accumulator
    uint64_t *drain = bars + 12;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + 13);
    volatile uint32_t *s_abort = s_tmem + 1;
    volatile uint32_t *s_ok = s_tmem + 2;  // [2] per half: outcome of the unit's waits

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&op_full[i], 1);
            mbar_init(&op_empty[i], 1);
            mbar_init(&codes_full[i], 1);
            mbar_init(&codes_empty[i], 8);
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 8);
        }
        mbar_init(drain, 1);
        *s_abort = 0u;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(s_tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    const int total = p.n_tiles * p.k_tiles;

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------------
        if (lane == 0) {
            tma_prefetch_desc(&map_codes);
            tma_prefetch_desc(&map_b);
            tma_prefetch_desc(&map_a);
            int gc = 0, lt = 0;
            bool ok = true;
            bool op_issued[2] = {false, false}, codes_issued[2] = {false, false};
            uint32_t op_par[2] = {0, 0}, codes_par[2] = {0, 0};
            for (int u = blockIdx.x; u < total && ok; u += gridDim.x, ++lt) {
                const int n0 = (u / p.k_tiles) * 128, k0 = (u % p.k_tiles) * 256;
                const int cb = lt & 1;
                if (kMode == 0) {
                    if (!mbar_wait(&codes_empty[cb], ((lt >> 1) & 1) ^ 1u, s_abort)) { ok = false; break; }
                    mbar_arrive_expect_tx(&codes_full[cb], kMrgCodesBytes);
                    tma_load_2d(sCodes + cb * kMrgCodesBytes, &map_codes, &codes_full[cb], k0 / 2, n0);
                    codes_issued[cb] = true;
                    codes_par[cb] = (lt >> 1) & 1;
                }
                for (int c = 0; c < p.rc; ++c, ++gc) {
                    const int sl = gc & 1;
                    if (!mbar_wait(&op_empty[sl], ((gc >> 1) & 1) ^ 1u, s_abort)) { ok = false; break; }
                    uint8_t *op = sOp + sl * kMrgOpBytes;
                    mbar_arrive_expect_tx(&op_full[sl], kMrgOpBytes);
                    tma_load_2d(op, &map_b, &op_full[sl], c * 64, n0);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        tma_load_2d(op + kMrgBBytes + i * 8192, &map_a, &op_full[sl], k0 + 64 * i, c * 64);
                    op_issued[sl] = true;
                    op_par[sl] = (gc >> 1) & 1;
                }
            }
            if (!ok) {
                // let copies in flight land before the CTA can exit (bounded)
                const uint64_t t0 = globaltimer_ns();
                for (int i = 0; i < 2; ++i) {
                    if (op_issued[i])
                        while (!mbar_try_wait(&op_full[i], op_par[i]) && globaltimer_ns() - t0 < 20000000ull) {}
                    if (codes_issued[i])
                        while (!mbar_try_wait(&codes_full[i], codes_par[i]) && globaltimer_ns() - t0 < 20000000ull) {}
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ---------------------------------------
        if (lane == 0) {
            // A = B_lora rows (K-major), B = A_lora columns (MN-major), D = 128 x 256 fp32
            const uint32_t idesc = make_idesc_bf16(256u, false, true);
            int gc = 0, lt = 0;
            bool ok = true, any = false;
            for (int u = blockIdx.x; u < total && ok; u += gridDim.x, ++lt) {
                const int a = lt & 1;
                if (!mbar_wait(&acc_empty[a], ((lt >> 1) & 1) ^ 1u, s_abort)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)a * 256u;
                for (int c = 0; c < p.rc; ++c, ++gc) {
                    const int sl = gc & 1;
                    if (!mbar_wait(&op_full[sl], (gc >> 1) & 1, s_abort)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t b_addr = smem_u32(sOp + sl * kMrgOpBytes);
                    const uint32_t a_addr = b_addr + kMrgBBytes;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t adesc = make_sw128_desc(b_addr + kk * 32u, 16u, 1024u);
                        const uint64_t bdesc = make_sw128_desc(a_addr + kk * 2048u, 8192u, 1024u);
                        umma_bf16(d_tmem, adesc, bdesc, idesc, (c > 0 || kk > 0) ? 1u : 0u);
                    }
                    any = true;
                    umma_commit(&op_empty[sl]);
                }
                if (!ok) break;
                umma_commit(&acc_full[a]);
            }
            if (!ok && any) {
                umma_commit(drain);
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < 20000000ull) {}
            }
        }
        __syncwarp();
    } else {
        // ------------------------------ epilogue (8 warps) -------------------------------
        const int quarter = warp & 3;                 // TMEM lanes this warp may access
        const int half = (warp - kMrgEpiWarp0) >> 2;  // 128-column half of the tile
        const int row = quarter * 32 + lane;          // tile row of this thread
        const int et = threadIdx.x - (kMrgEpiWarp0 + 4 * half) * 32;  // 0..127 within the half
        const float mu = __ldg(p.scale_mu);
        const uint32_t r7 = (uint32_t)row & 7u;
        int lt = 0, store_n = 0;
        // scale code and second-level constant of this thread's two 64-blocks of unit u (zeros
        // past the matrix, or when there is no unit u)
        int32_t sq_next[2] = {0, 0};
        float c2_next[2] = {0.0f, 0.0f};
        auto load_scale_codes = [&](int u) {
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                sq_next[g] = 0;
                c2_next[g] = 0.0f;
                if (u < total) {
                    const int64_t n = (int64_t)(u / p.k_tiles) * 128 + row;
                    const int64_t kb = ((u % p.k_tiles) * 256 + half * 128 + g * 64) / 64;
                    if (n < p.N && kb < p.KB) {
                        const int64_t b = n * p.KB + kb;
                        if (QLORA_IN_BOUNDS(b < p.N * p.KB)) sq_next[g] = __ldg(p.scale_q + b);
                        c2_next[g] = __ldg(p.scale_c2 + (b >> 8));
                    }
                }
            }
        };
        if (kMode == 0) load_scale_codes(blockIdx.x);
        for (int u = blockIdx.x; u < total; u += gridDim.x, ++lt) {
            const int n0 = (u / p.k_tiles) * 128, k0 = (u % p.k_tiles) * 256;
            const int a = lt & 1;
            const int64_t n = (int64_t)n0 + row;
            // block scales of this thread's two 64-blocks: their codes were requested one unit
            // earlier (a scale-code miss costs a DRAM latency, which a whole unit's epilogue hides);
            // this unit's values are taken and the next unit's requested
            float sc[2] = {0.0f, 0.0f};
            if (kMode == 0) {
#pragma unroll
                for (int g = 0; g < 2; ++g) sc[g] = __fmaf_rn((float)sq_next[g], __fdiv_rn(c2_next[g], 127.0f), mu);
                load_scale_codes(u + (int)gridDim.x);
            }
            // one outcome per half: its four warps meet at named barriers below
            // mode 1: this thread's base values and mask words, requested before the waits
            uint4 bv[2][2][4];
            uint32_t mw[2][2];
            if (kMode == 1) {
#pragma unroll
                for (int g = 0; g < 2; ++g)
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int64_t kk = (int64_t)k0 + half * 128 + g * 64 + c * 32;
                        const bool in = n < p.N && kk < p.K;
                        const uint4 *src = reinterpret_cast<const uint4 *>(p.base + n * p.K + kk);
                        // a plain (coherent) load: this kernel rewrites these elements afterwards
#pragma unroll
                        for (int i = 0; i < 4; ++i) bv[g][c][i] = in ? ld_global_v4(src + i) : make_uint4(0, 0, 0, 0);
                        mw[g][c] = in ? __ldg(p.mask_bits + (n * p.K + kk) / 32) : 0u;
                    }
            }
            if (et == 0)
                s_ok[half] = (mbar_wait(&acc_full[a], (lt >> 1) & 1, s_abort) &&
                              (kMode == 1 || mbar_wait(&codes_full[a], (lt >> 1) & 1, s_abort))) ? 1u : 0u;
            named_barrier_sync(3 + half, 128);
            const uint32_t okw = s_ok[half];
            named_barrier_sync(3 + half, 128);
            if (!okw) break;
            tc_fence_after();
            // the codes tile is stored with the 128-byte swizzle: 16-byte chunk j of a row at j ^ (row & 7)
            const uint8_t *crow = sCodes + a * kMrgCodesBytes + row * 128;
            for (int g = 0; g < 2; ++g, ++store_n) {
                uint32_t lo[4], hi[4];
                if (kMode == 0) build_table(sc[g], p.tab, lo, hi);
                // each warp stages its own 32 rows (double-buffered) and stores them with one TMA
                // store: no barrier between the epilogue warps
                uint8_t *buf = sOut + ((warp - kMrgEpiWarp0) * 2 + (store_n & 1)) * kMrgWarpOutBytes;
                if (lane == 0) bulk_wait_group_read<1>();  // this warp's store two groups back has read buf
                __syncwarp();
                // both 32-column halves of the group's accumulator in flight before the first use
                uint32_t racc[2][32];
#pragma unroll
                for (int c = 0; c < 2; ++c)
                    tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)a * 256u +
                                           (uint32_t)(half * 128 + g * 64 + c * 32),
                                       racc[c]);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const uint32_t *r = racc[c];
                    uint32_t words[4];
                    if (kMode == 0) {  // 32 codes: chunk 4 half + 2 g + c of the row
                        const uint4 cw = *reinterpret_cast<const uint4 *>(
                            crow + ((((uint32_t)(4 * half + 2 * g + c)) ^ r7) << 4));
                        words[0] = cw.x; words[1] = cw.y; words[2] = cw.z; words[3] = cw.w;
                    }
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        // 8 bf16 base values as pairs: W^ decoded (mode 0) or dX0 (mode 1)
                        const uint4 d = kMode == 0 ? decode8(words[w], lo, hi) : bv[g][c][w];
                        const uint32_t dw[4] = {d.x, d.y, d.z, d.w};
                        uint32_t o[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float w0 = __uint_as_float(dw[e] << 16), w1 = __uint_as_float(dw[e] & 0xffff0000u);
                            float f0 = p.s, f1 = p.s;
                            if (kMode == 1) {
                                const int bit = 8 * w + 2 * e;  // element within the 32-column chunk
                                f0 = (mw[g][c] >> bit) & 1u ? p.inv : 0.0f;
                                f1 = (mw[g][c] >> (bit + 1)) & 1u ? p.inv : 0.0f;
                            }
                            const float t0 = __fmaf_rn(f0, __uint_as_float(r[8 * w + 2 * e]), w0);
                            const float t1 = __fmaf_rn(f1, __uint_as_float(r[8 * w + 2 * e + 1]), w1);
                            o[e] = bf16x2(t0, t1);
                        }
                        // 16-byte chunk (4 c + w) of this row's 128 bytes, 128-byte swizzle
                        st_shared_v4(smem_u32(buf) + (uint32_t)lane * 128u + ((((uint32_t)(4 * c + w)) ^ r7) << 4),
                                     make_uint4(o[0], o[1], o[2], o[3]));
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&map_out, buf, k0 + half * 128 + g * 64, n0 + quarter * 32);
                    bulk_commit_group();
                }
            }
            // accumulator and codes of this unit are consumed
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&acc_empty[a]);
                if (kMode == 0) mbar_arrive(&codes_empty[a]);
            }
        }
        if (lane == 0) bulk_wait_group_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

template <int kMode>
static cudaError_t launch_rank_update(const CUtensorMap &map_codes, const CUtensorMap &map_b, const CUtensorMap &map_a,
                                      const CUtensorMap &map_out, MergeArgs p, int64_t N, int64_t K, int r, int num_sms,
                                      cudaStream_t st) {
    p.N = N;
    p.K = K;
    p.KB = (int32_t)(K / 64);
    p.n_tiles = (int32_t)((N + 127) / 128);
    p.k_tiles = (int32_t)((K + 255) / 256);
    p.rc = (r + 63) / 64;
    cudaError_t e = cudaFuncSetAttribute(nf4_merge_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kMrgSmem);
    if (e != cudaSuccess) return e;
    const int64_t units = (int64_t)p.n_tiles * p.k_tiles;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(units, num_sms));
    nf4_merge_kernel<kMode><<<grid, kMrgThreads, kMrgSmem, st>>>(map_codes, map_b, map_a, map_out, p);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_merge(const CUtensorMap &map_codes, const CUtensorMap &map_b, const CUtensorMap &map_a,
                         const CUtensorMap &map_out, const int8_t *scale_q, const float *scale_c2,
                         const float *scale_mu, int64_t N, int64_t K, int r, float s, const NF4Tables &tab,
                         int num_sms, cudaStream_t st) {
    MergeArgs p{};
    p.s = s;
    p.scale_q = scale_q;
    p.scale_c2 = scale_c2;
    p.scale_mu = scale_mu;
    p.tab = tab;
    return launch_rank_update<0>(map_codes, map_b, map_a, map_out, p, N, K, r, num_sms, st);
}

cudaError_t launch_dropout_dx(const CUtensorMap &map_v, const CUtensorMap &map_a, const CUtensorMap &map_dx,
                              const uint16_t *dx0, const uint32_t *mask_bits, float p_drop, int64_t M, int64_t K,
                              int r, int num_sms, cudaStream_t st) {
    MergeArgs p{};
    p.inv = 1.0f / (1.0f - p_drop);
    p.mask_bits = mask_bits;
    p.base = dx0;
    return launch_rank_update<1>(map_v /* unused codes map */, map_v, map_a, map_dx, p, M, K, r, num_sms, st);
}

}  // namespace qlora
