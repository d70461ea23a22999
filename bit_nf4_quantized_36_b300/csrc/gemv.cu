// gemv.cu -- the forward layer for up to eight tokens (decoding).
//
// With M <= 8 a weight is used by at most eight tokens: the call streams the packed codes once
// and its cost is the decode arithmetic (byte-permute lookups on the integer pipe), not the
// multiply.  This path keeps everything in registers: no shared-memory staging of decoded
// tiles, no barriers between warps.
//   - One token: scalar fused multiply-adds (nf4_gemv_fma_kernel).  Two to eight tokens:
//     a warp owns 16 weight rows and one 2048-wide slice of the contraction.  Lane (g, c)
//     (g = lane / 4, c = lane % 4) decodes rows g and g + 8 of one 64-weight NF4 block per step
//     of 256 columns (block 4 j + c of the slice at step j): one 16-entry table per row and
//     block, built from the rebuilt scale s'_b, gives exactly the bf16 values nf4_dequantize
//     writes.
//   - The decoded bf16 pairs go straight into warp-level tensor-core products (mma.sync
//     m16n8k16, bf16 in, fp32 accumulate) as the A operand, with x as the B operand: lane (g, c)
//     supplies token g's x over its own block, so any permutation of the contraction within a
//     16-step is the same for A and B.  Eight token columns come at the price of one, so the
//     tensor core replaces up to eight scalar multiply-adds per decoded weight; the bf16 x bf16
//     products are exact in fp32.
//   - Each warp writes its 16 rows' slice partials to a [slices, M, N] fp32 buffer, and a
//     second kernel sums the slices in order, adds the rank-r term sum_j U[m, j] B[n, j] and
//     rounds to bf16.
// Source: "QLoRA -- La base en 4 bits, LoRA encima" (paperclase, lesson 8), "Parte 4 - LoRA
// encima": h = W^ x + (alpha/r) B A x, with W^ the bf16 dequantized weight.

namespace qlora {

static constexpr int kGemvSlice = 2048;     // contraction length per warp
static constexpr int kGemvWarps = 8;        // warps per CTA (same slice, different rows)
static constexpr int kGemvRowsPerWarp = 16;
static constexpr int kGemvRowsPerCta = kGemvWarps * kGemvRowsPerWarp;
static constexpr int kGemvMaxM = 8;

// D += A B, m16n8k16, bf16 operands, fp32 accumulators
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16 bytes of codes, read once: no L1 allocation
__device__ __forceinline__ uint4 ldg_stream_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// One token: scalar fused multiply-adds.  Lane l of a warp owns block l of the warp's 2048-wide
// slice (x in registers for all the rows the warp visits), decodes it for 8 consecutive rows in
// turn and multiplies it into fp32 with bf16 operands; a warp-shuffle tree reduces the lanes.
// With a single token the tensor-core form below wastes seven of its eight columns and loads x
// once per row group; this form measures faster there.
static constexpr int kGemvFmaRowsPerWarp = 8;
static constexpr int kGemvFmaRowsPerCta = kGemvWarps * kGemvFmaRowsPerWarp;

// a0 += lo(w) * lo(x), a1 += hi(w) * hi(x): bf16 operands, fp32 accumulators, one rounding each
__device__ __forceinline__ void fma2_bf16(uint32_t w, uint32_t x, float &a0, float &a1) {
    asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
        "mov.b32 {wl, wh}, %2;\n\t"
        "mov.b32 {xl, xh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, wl, xl, %0;\n\t"
        "fma.rn.f32.bf16 %1, wh, xh, %1;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "r"(w), "r"(x));
}

template <int kM>
__global__ void __launch_bounds__(kGemvWarps * 32)
    nf4_gemv_fma_kernel(const uint8_t *__restrict__ codes, const int8_t *__restrict__ scale_q,
                    const float *__restrict__ scale_c2, const float *__restrict__ scale_mu,
                    const uint16_t *__restrict__ X, int64_t N, int64_t K, float *__restrict__ partial,
                    const NF4Tables tab) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int slice = blockIdx.y;
    const int64_t k0 = (int64_t)slice * kGemvSlice + (int64_t)lane * 64;  // this lane's block
    const bool kvalid = k0 < K;
    const int64_t KB = K / 64;
    const float mu = __ldg(scale_mu);

    uint32_t xr[kM][32];  // x[m, k0 .. k0 + 63] as bf16 pairs
#pragma unroll
    for (int m = 0; m < kM; ++m) {
        const uint4 *xp = reinterpret_cast<const uint4 *>(X + (int64_t)m * K + k0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint4 v = kvalid ? __ldg(xp + i) : make_uint4(0, 0, 0, 0);
            xr[m][4 * i] = v.x;
            xr[m][4 * i + 1] = v.y;
            xr[m][4 * i + 2] = v.z;
            xr[m][4 * i + 3] = v.w;
        }
    }

    const int64_t row0 = (int64_t)blockIdx.x * kGemvFmaRowsPerCta + (int64_t)warp * kGemvFmaRowsPerWarp;
    int64_t g_cached = -1;
    float k_cached = 0.0f;
    // codes of the next row are requested before the current row is decoded
    uint4 c0 = make_uint4(0, 0, 0, 0), c1 = c0;
    int32_t qn = 0;
    if (kvalid && row0 < N) {
        const uint8_t *cp = codes + (row0 * K + k0) / 2;
        c0 = ldg_stream_v4(cp);
        c1 = ldg_stream_v4(cp + 16);
        qn = __ldg(scale_q + row0 * KB + k0 / 64);
    }
    for (int i = 0; i < kGemvFmaRowsPerWarp; ++i) {
        const int64_t n = row0 + i;
        if (n >= N) break;
        const uint4 a0 = c0, a1 = c1;
        const int32_t q = qn;
        if (kvalid && n + 1 < N && i + 1 < kGemvFmaRowsPerWarp) {
            const uint8_t *cp = codes + ((n + 1) * K + k0) / 2;
            c0 = ldg_stream_v4(cp);
            c1 = ldg_stream_v4(cp + 16);
            qn = __ldg(scale_q + (n + 1) * KB + k0 / 64);
        }
        float acc[kM][2];
#pragma unroll
        for (int m = 0; m < kM; ++m) acc[m][0] = acc[m][1] = 0.0f;
        if (kvalid) {
            const int64_t b = n * KB + k0 / 64;
            if ((b >> 8) != g_cached) {
                g_cached = b >> 8;
                k_cached = __fdiv_rn(__ldg(scale_c2 + g_cached), 127.0f);
            }
            uint32_t lo[4], hi[4];
            build_table(__fmaf_rn((float)q, k_cached, mu), tab, lo, hi);
            const uint32_t words[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int wi = 0; wi < 8; ++wi) {
                const uint4 d = decode8(words[wi], lo, hi);  // elements 8 wi .. 8 wi + 7
#pragma unroll
                for (int m = 0; m < kM; ++m) {
                    fma2_bf16(d.x, xr[m][4 * wi], acc[m][0], acc[m][1]);
                    fma2_bf16(d.y, xr[m][4 * wi + 1], acc[m][0], acc[m][1]);
                    fma2_bf16(d.z, xr[m][4 * wi + 2], acc[m][0], acc[m][1]);
                    fma2_bf16(d.w, xr[m][4 * wi + 3], acc[m][0], acc[m][1]);
                }
            }
        }
#pragma unroll
        for (int m = 0; m < kM; ++m) {
            float v = __fadd_rn(acc[m][0], acc[m][1]);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
            if (lane == 0) partial[((int64_t)slice * kM + m) * N + n] = v;
        }
    }
}

// Rebuilt block scale s'_b = fmaf(q_b, fl32(c2_g / 127), mu), caching the group constant.
__device__ __forceinline__ float gemv_scale(const int8_t *scale_q, const float *scale_c2, float mu, int64_t b,
                                           int64_t &g_cached, float &k_cached) {
    if ((b >> 8) != g_cached) {
        g_cached = b >> 8;
        k_cached = __fdiv_rn(__ldg(scale_c2 + g_cached), 127.0f);
    }
    return __fmaf_rn((float)__ldg(scale_q + b), k_cached, mu);
}

__global__ void __launch_bounds__(kGemvWarps * 32)
    nf4_gemv_kernel(const uint8_t *__restrict__ codes, const int8_t *__restrict__ scale_q,
                    const float *__restrict__ scale_c2, const float *__restrict__ scale_mu,
                    const uint16_t *__restrict__ X, int M, int64_t N, int64_t K, float *__restrict__ partial,
                    const NF4Tables tab) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int slice = blockIdx.y;
    const int64_t KB = K / 64;
    const float mu = __ldg(scale_mu);
    const int64_t r0 = (int64_t)blockIdx.x * kGemvRowsPerCta + (int64_t)warp * kGemvRowsPerWarp + g;  // rows r0, r0 + 8
    const bool v0 = r0 < N, v1 = r0 + 8 < N;
    const int tok = g < M ? g : 0;  // B column g: token g (columns past M are not stored)
    const int64_t kb0 = (int64_t)slice * (kGemvSlice / 64) + c;  // this lane's block at step 0
    constexpr int kSteps = kGemvSlice / 256;

    int64_t gc0 = -1, gc1 = -1;
    float kc0 = 0.0f, kc1 = 0.0f;
    float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    // codes of the next step are requested before the current one is decoded
    const uint4 kZero = make_uint4(0x77777777u, 0x77777777u, 0x77777777u, 0x77777777u);  // code 7 = 0.0
    auto load_codes = [&](int64_t kb, uint4 (&cd)[4]) {
        const bool kv = kb < KB;
        const uint8_t *p0 = codes + (r0 * K + kb * 64) / 2;
        cd[0] = (kv && v0) ? ldg_stream_v4(p0) : kZero;
        cd[1] = (kv && v0) ? ldg_stream_v4(p0 + 16) : kZero;
        cd[2] = (kv && v1) ? ldg_stream_v4(p0 + 4 * K) : kZero;
        cd[3] = (kv && v1) ? ldg_stream_v4(p0 + 4 * K + 16) : kZero;
    };
    uint4 cn[4];
    load_codes(kb0, cn);
#pragma unroll 1
    for (int j = 0; j < kSteps; ++j) {
        const int64_t kb = kb0 + 4 * j;
        const uint4 cd[4] = {cn[0], cn[1], cn[2], cn[3]};
        if (j + 1 < kSteps) load_codes(kb + 4, cn);
        // every lane takes part in every mma.sync: a block past K has zero codes (the zero level)
        // and zero x, so it adds nothing
        const bool kv = kb < KB;
        uint32_t lo0[4], hi0[4], lo1[4], hi1[4];
        build_table((kv && v0) ? gemv_scale(scale_q, scale_c2, mu, r0 * KB + kb, gc0, kc0) : 0.0f, tab, lo0, hi0);
        build_table((kv && v1) ? gemv_scale(scale_q, scale_c2, mu, (r0 + 8) * KB + kb, gc1, kc1) : 0.0f, tab, lo1, hi1);
        const uint32_t w0[8] = {cd[0].x, cd[0].y, cd[0].z, cd[0].w, cd[1].x, cd[1].y, cd[1].z, cd[1].w};
        const uint32_t w1[8] = {cd[2].x, cd[2].y, cd[2].z, cd[2].w, cd[3].x, cd[3].y, cd[3].z, cd[3].w};
        const uint4 *xp = reinterpret_cast<const uint4 *>(X + (int64_t)tok * K + kb * 64);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            // x of token `tok` over half of this block (32 columns), as bf16 pairs
            uint32_t xr[16];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 v = kv ? __ldg(xp + 4 * h + i) : make_uint4(0u, 0u, 0u, 0u);
                xr[4 * i] = v.x;
                xr[4 * i + 1] = v.y;
                xr[4 * i + 2] = v.z;
                xr[4 * i + 3] = v.w;
            }
#pragma unroll
            for (int wj = 0; wj < 4; ++wj) {
                const int wi = 4 * h + wj;
                const uint4 e0 = decode8(w0[wi], lo0, hi0);  // row r0, elements 8 wi .. 8 wi + 7
                const uint4 e1 = decode8(w1[wi], lo1, hi1);  // row r0 + 8
                mma_bf16_16816(d, e0.x, e1.x, e0.y, e1.y, xr[4 * wj], xr[4 * wj + 1]);
                mma_bf16_16816(d, e0.z, e1.z, e0.w, e1.w, xr[4 * wj + 2], xr[4 * wj + 3]);
            }
        }
    }
    // d = D[r0][2c], D[r0][2c + 1], D[r0 + 8][2c], D[r0 + 8][2c + 1] (token columns 2c, 2c + 1)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int m = 2 * c + e;
        if (m >= M) continue;
        float *dst = partial + ((int64_t)slice * M + m) * N;
        if (v0) dst[r0] = d[e];
        if (v1) dst[r0 + 8] = d[2 + e];
    }
}

// Y[m, n] = bf16(sum_s partial[s, m, n] (in slice order) + sum_j U[m, j] B[n, j])
__global__ void __launch_bounds__(256)
    gemv_finish_kernel(const float *__restrict__ partial, int slices, int M, int64_t N, const uint16_t *__restrict__ U,
                       int ldu, const uint16_t *__restrict__ B, int r, uint16_t *__restrict__ Y) {
    const int64_t total = (int64_t)M * N;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int m = (int)(i / N);
        const int64_t n = i - (int64_t)m * N;
        float acc = partial[((int64_t)0 * M + m) * N + n];
        for (int s = 1; s < slices; ++s) acc = __fadd_rn(acc, partial[((int64_t)s * M + m) * N + n]);
        float lora = 0.0f;
        for (int j = 0; j < r; ++j) {
            const float u = __uint_as_float((uint32_t)U[(int64_t)m * ldu + j] << 16);
            const float bv = __uint_as_float((uint32_t)B[n * r + j] << 16);
            lora = __fmaf_rn(u, bv, lora);
        }
        __nv_bfloat16 h = __float2bfloat16_rn(__fadd_rn(acc, lora));
        Y[i] = *reinterpret_cast<uint16_t *>(&h);
    }
}

int gemv_slices(int64_t K) { return (int)((K + kGemvSlice - 1) / kGemvSlice); }

cudaError_t launch_gemv(const uint8_t *codes, const int8_t *scale_q, const float *scale_c2, const float *scale_mu,
                        const uint16_t *X, int M, int64_t N, int64_t K, float *partial, const uint16_t *U, int ldu,
                        const uint16_t *B, int r, uint16_t *Y, const NF4Tables &tab, int num_sms, cudaStream_t st) {
    if (M < 1 || M > kGemvMaxM) return cudaErrorInvalidValue;
    if (M == 1) {
        const dim3 grid((unsigned)((N + kGemvFmaRowsPerCta - 1) / kGemvFmaRowsPerCta), (unsigned)gemv_slices(K));
        nf4_gemv_fma_kernel<1><<<grid, kGemvWarps * 32, 0, st>>>(codes, scale_q, scale_c2, scale_mu, X, N, K, partial,
                                                                tab);
    } else {
        const dim3 grid((unsigned)((N + kGemvRowsPerCta - 1) / kGemvRowsPerCta), (unsigned)gemv_slices(K));
        nf4_gemv_kernel<<<grid, kGemvWarps * 32, 0, st>>>(codes, scale_q, scale_c2, scale_mu, X, M, N, K, partial, tab);
    }
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t total = (int64_t)M * N;
    const int g = (int)std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256, (int64_t)num_sms * 8));
    gemv_finish_kernel<<<g, 256, 0, st>>>(partial, gemv_slices(K), M, N, U, ldu, B, r, Y);
    count_launch();
    return cudaGetLastError();
}

}  // namespace qlora
