// gemv.cu -- the forward layer for one or two tokens (decoding) on the CUDA cores.
//
// With M <= 2 a weight is used by at most two tokens: the call streams the packed codes once
// and its cost is the decode arithmetic, not the multiply.  This path keeps everything in
// registers: no shared-memory staging of decoded tiles, no barriers between warps, no tensor
// core issue cost.
//   - Each warp owns one 2048-wide slice of the contraction; its lanes hold that slice of x
//     (64 bf16 per lane and token) in registers for all the rows the warp visits.
//   - Per row, lane l decodes its 64-weight block (one NF4 block: one 16-entry table built
//     from the rebuilt scale s'_b, byte-permute lookups) into bf16 pairs, exactly the values
//     nf4_dequantize writes, and multiplies them into fp32 with x: bf16 x bf16 products are
//     exact in fp32 and each fused multiply-add rounds once.
//   - Warp-shuffle tree reduction over the 32 lanes; the slice partials go to a [slices, M, N]
//     fp32 buffer, and a second kernel sums the slices in order, adds the rank-r term
//     sum_j U[m, j] B[n, j] and rounds to bf16.
// Source: "QLoRA -- La base en 4 bits, LoRA encima" (paperclase, lesson 8), "Parte 4 - LoRA
// encima": h = W^ x + (alpha/r) B A x, with W^ the bf16 dequantized weight.

namespace qlora {

static constexpr int kGemvSlice = 2048;       // contraction length per warp (64 per lane)
static constexpr int kGemvWarps = 8;          // warps per CTA (same slice, different rows)
static constexpr int kGemvRowsPerWarp = 8;    // consecutive rows per warp
static constexpr int kGemvRowsPerCta = kGemvWarps * kGemvRowsPerWarp;

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

// 16 bytes of codes, read once: no L1 allocation
__device__ __forceinline__ uint4 ldg_stream_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

template <int kM>
__global__ void __launch_bounds__(kGemvWarps * 32)
    nf4_gemv_kernel(const uint8_t *__restrict__ codes, const int8_t *__restrict__ scale_q,
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

    const int64_t row0 = (int64_t)blockIdx.x * kGemvRowsPerCta + (int64_t)warp * kGemvRowsPerWarp;
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
    for (int i = 0; i < kGemvRowsPerWarp; ++i) {
        const int64_t n = row0 + i;
        if (n >= N) break;
        const uint4 a0 = c0, a1 = c1;
        const int32_t q = qn;
        if (kvalid && n + 1 < N && i + 1 < kGemvRowsPerWarp) {
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
    const dim3 grid((unsigned)((N + kGemvRowsPerCta - 1) / kGemvRowsPerCta), (unsigned)gemv_slices(K));
    if (M == 1)
        nf4_gemv_kernel<1><<<grid, kGemvWarps * 32, 0, st>>>(codes, scale_q, scale_c2, scale_mu, X, N, K, partial, tab);
    else
        nf4_gemv_kernel<2><<<grid, kGemvWarps * 32, 0, st>>>(codes, scale_q, scale_c2, scale_mu, X, N, K, partial, tab);
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
