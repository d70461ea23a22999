// quant.cu -- NF4 blockwise quantization, double quantization of the block scales, and
// dequantization to bf16.  CUDA-core kernels: these steps move 4.5 B (quantize) or 2.5 B
// (dequantize) per weight and do a few ALU operations per weight, so they are HBM-bound.
//
// Definitions restated ("QLoRA -- La base en 4 bits, LoRA encima", paperclase lesson 8,
// "Parte 4 - Una capa QLoRA, a mano"; "QLoRA" glossary, ultralytics, NF4 snippet):
//   s_b = max |w| over the 64-block; c = argmin_k |fl32(w / s_b) - NF4[k]|, ties to the lower k.
// Double quantization ("Parte 3 - Bits por parametro": 8-bit scales, one 32-bit constant per
// 256 blocks): a global mean offset mu and per-256-block symmetric int8 codes of s_b - mu.
#include "qlora_common.cuh"
#include "qlora_kernels.cuh"

namespace qlora {

// ---------------------------------------------------------------------------------------
// K1: per 64-block absmax, NF4 code of every weight, two codes per byte, and the fp64 sums of
// the 256-block groups' scales folded into aligned subtrees of the mean's pairwise tree.
// One CTA (256 threads, eight per SM) per run of `run` consecutive groups; 8 threads per 64-block
// (two float4 each, staged by cp.async three passes deep); the absmax is an 8-lane max reduction;
// the codes are formed two weights at a time with the packed two-lane fp32 instructions.
//
// Code rule: thr[0..14] are the exact fp32 decision thresholds of the nearest-level rule
// (thr[k] = smallest x in (L_k, L_k+1] with fl(L_k+1 - x) < fl(x - L_k)), so the code is the
// number of thresholds <= x = fl(w / s).  Identical to the argmin with fp32 distances and
// lower-index ties because no two non-adjacent levels can tie (levels are >= 0.079 apart and
// |x| <= 1).
// ---------------------------------------------------------------------------------------
// Exact: a 4-step binary search on x = fl(w / s).
__device__ __forceinline__ uint32_t nf4_code(float w, float s, const float *thr) {
    if (s == 0.0f) return kZeroCode;
    const float x = __fdiv_rn(w, s);
    uint32_t c = (x >= thr[7]) ? 8u : 0u;
    c += (x >= thr[c + 3]) ? 4u : 0u;
    c += (x >= thr[c + 1]) ? 2u : 0u;
    c += (x >= thr[c]) ? 1u : 0u;
    return c;
}

// Without a division: x0 = fl(w * fl(1/s)) is within 2^-22 of x when s is normal (|w / s| <= 1:
// two roundings of 2^-24 relative each, plus 2^-24 for x's own rounding).  The bucket index
// j = floor(16 x0 + 17) comes from one fma rounded toward -inf into [2^23, 2^24), where the ulp
// is 1, so the low bits of its bit pattern are j exactly; x0 lies in [b, b + 1/16) for
// b = -1 + (j - 1) / 16, every threshold at or below b - 2^-12 is below x, and the one after
// t = thr[c] is above x: the code is c + [t <= x].  With the table's t' (t moved by under 2^-20),
// the comparison on x0 gives [t <= x] whenever x0 is more than 2^-19 from t'; otherwise `unsure`
// asks for the exact rule.  A NaN weight makes d a NaN (unsure); the mask keeps its index in the
// table.
__device__ __forceinline__ uint32_t nf4_code_fast(float w, float rcp, const uint32_t *tab, bool &unsure) {
    const float x0 = __fmul_rn(w, rcp);
    const uint32_t e = tab[__float_as_uint(__fmaf_rd(x0, 16.0f, 8388625.0f)) & (kNF4Buckets - 1)];
    const float d = __fsub_rn(x0, __uint_as_float(e));
    unsure |= !(fabsf(d) > 0x1p-19f);
    return (e & 15u) + (d >= 0.0f ? 1u : 0u);
}

// S_g = fp64 sum of one group's scales s[0..255] (zeros past the last block) in index order, by
// one warp.  The scales are non-negative fp32 values; when the group's non-zero scales span at
// most 2^21 in binary exponent, every partial sum is an integer multiple of the smallest scale's
// ulp below 2^(24 + 21 + 8) of it, hence exact in fp64, so any summation order -- here a warp
// tree -- gives the bit pattern of the sequential sum.  Other groups (rare: scales differing by
// more than 2^21) take the sequential chain in index order.
__device__ __forceinline__ double group_sum(const float *s, uint32_t lane) {
    float v[8];
    int emin = 255, emax = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[i] = s[i * 32 + lane];
        const int e = (int)((__float_as_uint(v[i]) >> 23) & 0xFFu);
        if (v[i] != 0.0f) {
            emin = min(emin, e);
            emax = max(emax, e);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        emin = min(emin, __shfl_xor_sync(0xffffffffu, emin, o));
        emax = max(emax, __shfl_xor_sync(0xffffffffu, emax, o));
    }
    double acc = 0.0;
    if (emax - emin <= 21) {
#pragma unroll
        for (int i = 0; i < 8; ++i) acc = __dadd_rn(acc, (double)v[i]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc = __dadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
    } else if (lane == 0) {
        for (int b = 0; b < kGroup; ++b) acc = __dadd_rn(acc, (double)s[b]);
    }
    return acc;
}

static constexpr int kQuantThreads = kGroup;  // one thread per block of the group in the epilogue
static constexpr int kMeanLeaves = 1024;      // at most this many subtree sums reach the mean
// 8 threads per 64-block, two float4 each: a pass of the CTA covers 32 blocks.  Each thread
// stages its own two float4 of the next kQAhead passes in shared memory with cp.async (no
// register held while the loads are in flight), so every SM keeps eight CTAs x 256 threads x
// kQAhead x 32 B in flight at 32 registers a thread.
static constexpr int kQAhead = 3;
static constexpr int kQPassBlocks = kQuantThreads / 8;
static constexpr int kQPasses = kGroup / kQPassBlocks;  // passes per group

__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint64_t f2pack(uint32_t a, uint32_t b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ void f2unpack(uint64_t r, uint32_t &a, uint32_t &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=r"(a), "=r"(b) : "l"(r));
}

// nf4_code_fast for two weights at once, with the packed two-lane fp32 instructions (the same
// IEEE operations, lane by lane).  Returns the byte (code_a << 4) | code_b.
__device__ __forceinline__ uint32_t nf4_code_pair(float wa, float wb, uint64_t rcp2, const uint32_t *tab,
                                                  bool &unsure) {
    const uint64_t w2 = f2pack(__float_as_uint(wa), __float_as_uint(wb));
    const uint64_t k16 = 0x4180000041800000ull;   // (16, 16)
    const uint64_t kmag = 0x4B0000114B000011ull;  // (2^23 + 17, 2^23 + 17)
    uint64_t x2, y2, d2;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(x2) : "l"(w2), "l"(rcp2));
    asm("fma.rm.f32x2 %0, %1, %2, %3;" : "=l"(y2) : "l"(x2), "l"(k16), "l"(kmag));
    uint32_t ya, yb;
    f2unpack(y2, ya, yb);
    const uint32_t ea = tab[ya & (kNF4Buckets - 1)], eb = tab[yb & (kNF4Buckets - 1)];
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d2) : "l"(x2), "l"(f2pack(ea, eb)));
    uint32_t da, db;
    f2unpack(d2, da, db);
    unsure |= !(fabsf(__uint_as_float(da)) > 0x1p-19f) || !(fabsf(__uint_as_float(db)) > 0x1p-19f);
    // the code is c + [d >= 0] (d is never -0 here: x0 - t' rounds an exact zero to +0)
    const uint32_t ca = (ea & 15u) + ((da >> 31) ^ 1u), cb = (eb & 15u) + ((db >> 31) ^ 1u);
    return (ca << 4) | cb;
}

__global__ void __launch_bounds__(kQuantThreads, 8) nf4_quantize_groups_kernel(
    const float4 *__restrict__ W, int64_t nb, int64_t ng, int64_t run, uint16_t *__restrict__ codes16,
    float *__restrict__ absmax, double *__restrict__ leaves, NF4Tables tab) {
    __shared__ float4 s_in[kQAhead][2][kQuantThreads];
    __shared__ float s_thr[16];
    __shared__ float s_abs[2][kGroup];  // double-buffered over groups: one barrier per group
    __shared__ uint32_t s_tab[kNF4Buckets];
    __shared__ double s_stack[48];      // pairwise-tree stack over the run's groups
    if (threadIdx.x < 16) s_thr[threadIdx.x] = tab.thr[threadIdx.x];
    if (threadIdx.x < kNF4Buckets) s_tab[threadIdx.x] = tab.bucket[threadIdx.x];
    __syncthreads();

    // this CTA's groups [g0, g0 + run) hold blocks [B0, B1): a contiguous range of W
    const int64_t g0 = (int64_t)blockIdx.x * run;
    const int64_t B0 = min64(nb, g0 * kGroup), B1 = min64(nb, (g0 + run) * kGroup);
    const int nblk = (int)(B1 - B0);                       // < 2^31: run * 256 blocks at most
    const int ngrp = (nblk + kGroup - 1) / kGroup;         // groups of W in the run
    const uint32_t lane = threadIdx.x & 31u, l8 = threadIdx.x & 7u;
    const uint32_t gmask = 0xFFu << (lane & 24u);
    const int sub = (int)(threadIdx.x >> 3);  // block within a pass
    constexpr int kQPassStride = kQPassBlocks * 16;  // float4 (and code words) per pass
    // this thread's two float4 of a pass are W[i] and W[i + 8], and its two code words of that
    // pass codes16[i] and codes16[i + 8] (the same index): i advances by a pass each time.  `si`
    // is the index of the pass staged next, which runs kQAhead - 1 passes ahead of the one coded.
    int64_t si = (B0 + sub) * 16 + l8;
    int sblk = sub;  // block (within the run) staged next by this thread
    // staging slots: the slot read in a pass is rslot; the one staged is the slot before it
    const uint32_t slot0 = smem_u32(&s_in[0][0][threadIdx.x]);
    constexpr uint32_t kSlotBytes = 2u * kQuantThreads * 16u, kHalf = kQuantThreads * 16u;
    static_assert(kQAhead == 3, "slot rotation below");
    auto stage = [&](uint32_t wslot) {  // the next pass's two float4, or zeros past the run's blocks
        if (sblk < nblk) {
            cp_async_16(wslot, W + si);
            cp_async_16(wslot + kHalf, W + si + 8);
        } else {
            asm volatile("st.shared.v4.f32 [%0], {%1, %1, %1, %1};" ::"r"(wslot), "f"(0.0f) : "memory");
            asm volatile("st.shared.v4.f32 [%0], {%1, %1, %1, %1};" ::"r"(wslot + kHalf), "f"(0.0f) : "memory");
        }
        cp_async_commit();  // one group per pass, empty or not, keeps the wait count fixed
        si += kQPassStride;
        sblk += kQPassBlocks;
    };
    stage(slot0);
    stage(slot0 + kSlotBytes);
    uint32_t rslot = slot0;

    const int npass = ngrp * kQPasses;
    float *sa = s_abs[0] + sub;
#pragma unroll 1
    for (int p = 0; p < npass; ++p) {
        stage(rslot == slot0 ? slot0 + 2 * kSlotBytes : rslot - kSlotBytes);
        cp_async_wait<kQAhead - 1>();  // pass p has landed (only this thread reads its slots)
        float4 v, u;
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(rslot) : "memory");
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(u.x), "=f"(u.y), "=f"(u.z), "=f"(u.w) : "r"(rslot + kHalf) : "memory");
        rslot = rslot == slot0 + 2 * kSlotBytes ? slot0 : rslot + kSlotBytes;
        // |w| >= 0 orders like its bit pattern; fmaxf drops NaN (finite input is required)
        float m = fmaxf(fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))),
                        fmaxf(fmaxf(fabsf(u.x), fabsf(u.y)), fmaxf(fabsf(u.z), fabsf(u.w))));
        m = __uint_as_float(__reduce_max_sync(gmask, __float_as_uint(fmaxf(m, 0.0f))));
        // codes of the thread's 8 weights, weight i in byte i / 2 (even i in the high nibble)
        uint32_t packed = 0x77777777u;  // an all-zero block
        // the shortcut's error bound needs fl(1/m) normal: 2^-100 <= m < 2^126
        bool unsure = !(m >= 0x1p-100f && m < 0x1p126f);
        if (!unsure) {
            const uint32_t rb = __float_as_uint(__frcp_rn(m));
            const uint64_t rcp2 = f2pack(rb, rb);
            packed = nf4_code_pair(v.x, v.y, rcp2, s_tab, unsure) | (nf4_code_pair(v.z, v.w, rcp2, s_tab, unsure) << 8) |
                     (nf4_code_pair(u.x, u.y, rcp2, s_tab, unsure) << 16) |
                     (nf4_code_pair(u.z, u.w, rcp2, s_tab, unsure) << 24);
        }
        if (unsure) {  // rare: the exact rule, one weight at a time
            packed = (nf4_code(v.x, m, s_thr) << 4) | nf4_code(v.y, m, s_thr) |
                     (((nf4_code(v.z, m, s_thr) << 4) | nf4_code(v.w, m, s_thr)) << 8) |
                     (((nf4_code(u.x, m, s_thr) << 4) | nf4_code(u.y, m, s_thr)) << 16) |
                     (((nf4_code(u.z, m, s_thr) << 4) | nf4_code(u.w, m, s_thr)) << 24);
        }
        if (sblk - kQAhead * kQPassBlocks < nblk) {  // this pass's block is one of W's
            const int64_t ci = si - kQAhead * kQPassStride;  // this pass's first code word
            if (QLORA_IN_BOUNDS(ci >= 0 && ci + 8 < nb * 16)) {
                codes16[ci] = (uint16_t)packed;
                codes16[ci + 8] = (uint16_t)(packed >> 16);
            }
        }
        if (l8 == 0) *sa = m;  // 0 past the last block
        sa += kQPassBlocks;
        if ((p & (kQPasses - 1)) == kQPasses - 1) {
            // the group is closed.  One barrier: the buffer is written again two groups later,
            // after the next group's barrier, which every reader of this one has passed
            const int gi = p / kQPasses;
            const float *sg = s_abs[gi & 1];
            sa = s_abs[(gi + 1) & 1] + sub;
            __syncthreads();
            if (gi * kGroup + (int)threadIdx.x < nblk) {
                const int64_t bi = min64(nb, (int64_t)blockIdx.x * run * kGroup) + gi * kGroup + threadIdx.x;
                if (QLORA_IN_BOUNDS(bi < nb)) absmax[bi] = sg[threadIdx.x];
            }
            // the group's sum, by warp gi % 8 (the duty rotates so that no warp falls behind);
            // the push onto the shared stack follows the previous group's push, which its warp
            // made before reaching this group's barrier
            if ((int)(threadIdx.x >> 5) == (gi & 7)) {
                double sum = group_sum(sg, lane);
                if (lane == 0) {  // leaf gi of the run, paired as the tree's levels pair them
                    int lvl = 0;
                    for (int j = gi; j & 1; j >>= 1) sum = __dadd_rn(s_stack[lvl++], sum);
                    s_stack[lvl] = sum;
                }
            }
        }
    }
    cp_async_wait<0>();  // the look-ahead copies past the range are empty groups; nothing lands late
    __syncthreads();     // the last group's push
    if (threadIdx.x == 0) {
        // groups of the run past the last one of W are leaves of +0.0
        for (int64_t j = ngrp; j < run; ++j) {
            double sum = 0.0;
            int lvl = 0;
            for (int64_t k = j; k & 1; k >>= 1) sum = __dadd_rn(s_stack[lvl++], sum);
            s_stack[lvl] = sum;
        }
        leaves[blockIdx.x] = s_stack[__ffsll((long long)run) - 1];
    }
}

// K2: mu = fl32(T / nb) with an IEEE fp64 division, T the pairwise tree over the p2 group sums
// (level by level, t'[i] = t[2i] + t[2i+1]); K1 left the nl <= 1024 sums of its aligned
// subtrees, and warp 0 of every CTA pairs them the same way: each lane pairs an aligned run of
// nl / 32 of them level by level, then a butterfly of shuffles pairs the lanes' results (lane l
// adds its partner's value, and fp64 addition is commutative, so both partners hold t[2i] +
// t[2i+1]).  Then per group (one warp): c2_g = max |fl32(s_b - mu)|;
// q_b = rint(fl32(fl32(d / c2) * 127)).
static constexpr int kEncodeThreads = 1024;

__global__ void __launch_bounds__(kEncodeThreads) dq_encode_kernel(const float *__restrict__ absmax, int64_t nb,
                                                                   int64_t ng, const double *__restrict__ leaves,
                                                                   int nl, int8_t *__restrict__ qcode,
                                                                   float *__restrict__ c2_out,
                                                                   float *__restrict__ mu_out) {
    __shared__ float s_mu;
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int per = nl > 32 ? nl / 32 : 1;  // leaves per lane (a power of two, <= 32)
        const int nlanes = nl / per;            // lanes holding a subtree (a power of two)
        double t[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) t[i] = (i < per && lane < nlanes) ? leaves[lane * per + i] : 0.0;
#pragma unroll
        for (int len = 32; len > 1; len >>= 1) {
            if (len <= per) {
#pragma unroll
                for (int i = 0; i < len / 2; ++i) t[i] = __dadd_rn(t[2 * i], t[2 * i + 1]);
            }
        }
        double v = t[0];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double w = __shfl_xor_sync(0xffffffffu, v, o);
            if (o < nlanes) v = __dadd_rn(v, w);
        }
        if (lane == 0) {
            s_mu = __double2float_rn(__ddiv_rn(v, (double)nb));
            if (blockIdx.x == 0) *mu_out = s_mu;
        }
    }
    __syncthreads();
    const float mu = s_mu;
    const uint32_t lane = threadIdx.x & 31u;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t g = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; g < ng; g += warps) {
        float d[8];
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t b = g * kGroup + i * 32 + lane;
            d[i] = (b < nb) ? __fsub_rn(absmax[b], mu) : 0.0f;
            m = fmaxf(m, fabsf(d[i]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) c2_out[g] = m;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t b = g * kGroup + i * 32 + lane;
            if (b < nb) {
                float q = 0.0f;
                if (m != 0.0f) {
                    q = rintf(__fmul_rn(__fdiv_rn(d[i], m), 127.0f));
                    q = fminf(fmaxf(q, -127.0f), 127.0f);
                }
                qcode[b] = (int8_t)(int)q;
            }
        }
    }
}

// ---------------------------------------------------------------------------------------
// K3: dequantize.  One thread per 8 weights (one 32-bit word of codes -> one 16-byte store) per
// step, four steps' loads in flight before any of them is used: warp-coalesced loads and stores,
// and enough of the code stream in flight per thread.
//   s'_b = fmaf(q_b, fl32(c2_g / 127), mu);  W^ = bf16_rne(fl32(NF4[c] * s'_b))
// ---------------------------------------------------------------------------------------
static constexpr int kDqUnroll = 4;

__global__ void __launch_bounds__(256, 8) nf4_dequantize_kernel(const uint32_t *__restrict__ codes32,
                                                             const int8_t *__restrict__ qcode,
                                                             const float *__restrict__ c2,
                                                             const float *__restrict__ mu_ptr, int64_t n8,
                                                             uint4 *__restrict__ out, NF4Tables tab) {
    __shared__ float L[16];
    if (threadIdx.x < 16) L[threadIdx.x] = tab.level[threadIdx.x];
    __syncthreads();
    const float mu = *mu_ptr;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t0 < n8; t0 += kDqUnroll * stride) {
        uint32_t x[kDqUnroll];
        int32_t qb[kDqUnroll];
        float cg[kDqUnroll];
#pragma unroll
        for (int u = 0; u < kDqUnroll; ++u) {
            const int64_t t = t0 + u * stride;
            const bool in = t < n8;
            x[u] = in ? __ldcs(codes32 + t) : 0u;
            qb[u] = in ? (int32_t)qcode[t >> 3] : 0;
            cg[u] = in ? c2[t >> 11] : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < kDqUnroll; ++u) {
            const int64_t t = t0 + u * stride;
            if (t >= n8) break;
            const float s = __fmaf_rn((float)qb[u], __fdiv_rn(cg[u], 127.0f), mu);
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t byte = (x[u] >> (8 * j)) & 0xFFu;
                const float e0 = __fmul_rn(L[byte >> 4], s);   // element 2j   (high nibble)
                const float e1 = __fmul_rn(L[byte & 15u], s);  // element 2j+1 (low nibble)
                __nv_bfloat162 p = __floats2bfloat162_rn(e0, e1);
                w[j] = *reinterpret_cast<uint32_t *>(&p);
            }
            int64_t ts = t;
#ifdef QLORA_DEVICE_CHECKS
            // test hook: the first thread's first store index moved past the end of the output
            if (t == 0 && (*(volatile uint32_t *)&g_inject & kInjectBounds)) ts = n8;
#endif
            if (QLORA_IN_BOUNDS(ts < n8)) __stcs(out + ts, make_uint4(w[0], w[1], w[2], w[3]));
        }
    }
}

// ---------------------------------------------------------------------------------------
// Host-side launchers
// ---------------------------------------------------------------------------------------
static int grid_for(int64_t work_items, int per_block, int num_sms, int waves) {
    int64_t g = (work_items + per_block - 1) / per_block;
    const int64_t cap = (int64_t)num_sms * waves;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return (int)g;
}

cudaError_t launch_quantize(const float *W, int64_t n, uint8_t *codes, int8_t *qcode, float *c2, float *mu,
                            float *ws_absmax, double *ws_tree, int64_t p2, const NF4Tables &tab, int num_sms,
                            cudaStream_t st) {
    const int64_t nb = n / kBlock, ng = (nb + kGroup - 1) / kGroup;
    // runs of `run` groups (a power of two) so that at most min(1024, 8 per SM) subtree sums remain
    int64_t run = 1;
    while (p2 / run > std::min<int64_t>(kMeanLeaves, (int64_t)num_sms * 8)) run <<= 1;
    const int nl = (int)(p2 / run);
    nf4_quantize_groups_kernel<<<nl, kQuantThreads, 0, st>>>(reinterpret_cast<const float4 *>(W), nb, ng, run,
                                                             reinterpret_cast<uint16_t *>(codes), ws_absmax, ws_tree,
                                                             tab);
    count_launch();
    const int g2 = (int)std::max<int64_t>(1, std::min<int64_t>((ng + 31) / 32, (int64_t)num_sms));
    dq_encode_kernel<<<g2, kEncodeThreads, 0, st>>>(ws_absmax, nb, ng, ws_tree, nl, qcode, c2, mu);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_dequantize(const uint8_t *codes, const int8_t *qcode, const float *c2, const float *mu, int64_t n,
                              uint16_t *out, const NF4Tables &tab, int num_sms, cudaStream_t st) {
    const int64_t n8 = n / 8;
    nf4_dequantize_kernel<<<grid_for(n8, 256, num_sms, 8), 256, 0, st>>>(
        reinterpret_cast<const uint32_t *>(codes), qcode, c2, mu, n8, reinterpret_cast<uint4 *>(out), tab);
    count_launch();
    return cudaGetLastError();
}

}  // namespace qlora
