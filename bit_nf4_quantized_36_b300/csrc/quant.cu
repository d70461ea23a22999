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
// K1: per 64-block absmax, NF4 code of every weight, two codes per byte.
// 16 threads per block (float4 each); the absmax is a 16-lane shuffle reduction.
// Code rule: thr[0..14] are the exact fp32 decision thresholds of the nearest-level rule
// (thr[k] = smallest x in (L_k, L_k+1] with fl(L_k+1 - x) < fl(x - L_k)), so the code is the
// number of thresholds <= x; a 4-step binary search finds it.  Identical to the argmin with
// fp32 distances and lower-index ties because no two non-adjacent levels can tie (levels
// are >= 0.079 apart and |x| <= 1).
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t nf4_code(float w, float s, const float *thr) {
    if (s == 0.0f) return kZeroCode;
    const float x = __fdiv_rn(w, s);
    uint32_t c = (x >= thr[7]) ? 8u : 0u;
    c += (x >= thr[c + 3]) ? 4u : 0u;
    c += (x >= thr[c + 1]) ? 2u : 0u;
    c += (x >= thr[c]) ? 1u : 0u;
    return c;
}

__global__ void __launch_bounds__(256) nf4_quantize_blocks_kernel(const float4 *__restrict__ W, int64_t nb,
                                                                  uint16_t *__restrict__ codes16,
                                                                  float *__restrict__ absmax, NF4Tables tab) {
    __shared__ float s_thr[16];
    if (threadIdx.x < 16) s_thr[threadIdx.x] = tab.thr[threadIdx.x];
    __syncthreads();
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t l16 = threadIdx.x & 15u;
    const uint32_t gmask = 0xFFFFu << (lane & 16u);
    const int64_t per_cta = blockDim.x / 16;
    for (int64_t b = (int64_t)blockIdx.x * per_cta + threadIdx.x / 16; b < nb; b += (int64_t)gridDim.x * per_cta) {
        const float4 v = __ldcs(W + b * 16 + l16);
        float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
        m = fmaxf(m, __shfl_xor_sync(gmask, m, 8));
        m = fmaxf(m, __shfl_xor_sync(gmask, m, 4));
        m = fmaxf(m, __shfl_xor_sync(gmask, m, 2));
        m = fmaxf(m, __shfl_xor_sync(gmask, m, 1));
        const uint32_t c0 = nf4_code(v.x, m, s_thr), c1 = nf4_code(v.y, m, s_thr);
        const uint32_t c2 = nf4_code(v.z, m, s_thr), c3 = nf4_code(v.w, m, s_thr);
        codes16[b * 16 + l16] = (uint16_t)(((c0 << 4) | c1) | (((c2 << 4) | c3) << 8));
        if (l16 == 0) absmax[b] = m;
    }
}

// K2a: S_g = fp64 sum of the group's scales in index order; slots ng..p2-1 get +0.0.
// One warp per group.  The scales are non-negative fp32 values; when the group's non-zero scales
// span at most 2^21 in binary exponent, every partial sum is an integer multiple of the smallest
// scale's ulp below 2^(24 + 21 + 8) of it, hence exact in fp64, so any summation order -- here a
// warp tree -- gives the bit pattern of the sequential sum.  Other groups (rare: scales differing
// by more than 2^21) take the sequential chain in index order.
__global__ void __launch_bounds__(256) dq_group_sums_kernel(const float *__restrict__ absmax, int64_t nb, int64_t ng,
                                                            int64_t p2, double *__restrict__ tree) {
    const uint32_t lane = threadIdx.x & 31u;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t g = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; g < p2; g += warps) {
        if (g >= ng) {
            if (lane == 0) tree[g] = 0.0;
            continue;
        }
        float v[8];
        int emin = 255, emax = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t b = g * kGroup + i * 32 + lane;
            v[i] = (b < nb) ? absmax[b] : 0.0f;
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
            const int64_t b1 = (g * kGroup + kGroup < nb) ? g * kGroup + kGroup : nb;
            for (int64_t b = g * kGroup; b < b1; ++b) acc = __dadd_rn(acc, (double)absmax[b]);
        }
        if (lane == 0) tree[g] = acc;
    }
}

// K2b: pairwise tree over the p2 group sums (level by level: t'[i] = t[2i] + t[2i+1], ping-pong
// buffers), then mu = fl32(total / nb) with an IEEE fp64 division.  One CTA.
__global__ void __launch_bounds__(1024) dq_mean_kernel(double *__restrict__ tree, double *__restrict__ tree2,
                                                       int64_t p2, int64_t nb, float *__restrict__ mu_out) {
    double *src = tree, *dst = tree2;
    for (int64_t len = p2; len > 1; len >>= 1) {
        for (int64_t i = threadIdx.x; i < len / 2; i += blockDim.x) dst[i] = __dadd_rn(src[2 * i], src[2 * i + 1]);
        __syncthreads();
        double *t = src;
        src = dst;
        dst = t;
    }
    if (threadIdx.x == 0) *mu_out = __double2float_rn(__ddiv_rn(src[0], (double)nb));
}

// K2c: per group (one warp): c2_g = max |fl32(s_b - mu)|; q_b = rint(fl32(fl32(d / c2) * 127)).
__global__ void __launch_bounds__(256) dq_encode_kernel(const float *__restrict__ absmax, int64_t nb, int64_t ng,
                                                        const float *__restrict__ mu_ptr, int8_t *__restrict__ qcode,
                                                        float *__restrict__ c2_out) {
    const uint32_t lane = threadIdx.x & 31u;
    const float mu = *mu_ptr;
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
// K3: dequantize.  One thread per 8 weights (one 32-bit word of codes -> one 16-byte store).
//   s'_b = fmaf(q_b, fl32(c2_g / 127), mu);  W^ = bf16_rne(fl32(NF4[c] * s'_b))
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) nf4_dequantize_kernel(const uint32_t *__restrict__ codes32,
                                                             const int8_t *__restrict__ qcode,
                                                             const float *__restrict__ c2,
                                                             const float *__restrict__ mu_ptr, int64_t n8,
                                                             uint4 *__restrict__ out, NF4Tables tab) {
    __shared__ float L[16];
    if (threadIdx.x < 16) L[threadIdx.x] = tab.level[threadIdx.x];
    __syncthreads();
    const float mu = *mu_ptr;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n8; t += (int64_t)gridDim.x * blockDim.x) {
        const uint32_t x = __ldcs(codes32 + t);
        const int64_t b = t >> 3;
        const float s = __fmaf_rn((float)qcode[b], __fdiv_rn(c2[b >> 8], 127.0f), mu);
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t byte = (x >> (8 * j)) & 0xFFu;
            const float e0 = __fmul_rn(L[byte >> 4], s);   // element 2j   (high nibble)
            const float e1 = __fmul_rn(L[byte & 15u], s);  // element 2j+1 (low nibble)
            __nv_bfloat162 p = __floats2bfloat162_rn(e0, e1);
            w[j] = *reinterpret_cast<uint32_t *>(&p);
        }
        __stcs(out + t, make_uint4(w[0], w[1], w[2], w[3]));
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
    nf4_quantize_blocks_kernel<<<grid_for(nb, 16, num_sms, 8), 256, 0, st>>>(
        reinterpret_cast<const float4 *>(W), nb, reinterpret_cast<uint16_t *>(codes), ws_absmax, tab);
    count_launch();
    dq_group_sums_kernel<<<grid_for(p2, 8, num_sms, 16), 256, 0, st>>>(ws_absmax, nb, ng, p2, ws_tree);
    count_launch();
    dq_mean_kernel<<<1, 1024, 0, st>>>(ws_tree, ws_tree + p2, p2, nb, mu);
    count_launch();
    dq_encode_kernel<<<grid_for(ng, 8, num_sms, 8), 256, 0, st>>>(ws_absmax, nb, ng, mu, qcode, c2);
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
