// dropout.cu -- the LoRA dropout mask on the adapter input.
//
// The adapter branch of the layer sees x_d = x * mask / (1 - p) with mask ~ Bernoulli(1 - p)
// ("LoRA y QLoRA para un ajuste eficiente en costes" (coddykit), LoraConfig lora_dropout).  The
// mask is drawn from the counter-based generator Philox4x32-10 (Salmon, Moraes, Dror, Shaw,
// "Parallel random numbers: as easy as 1, 2, 3", SC'11), so the backward regenerates exactly the
// forward's mask from (seed, offset): element e of the row-major [M, K] input takes word e % 4 of
// the block with counter (e / 4 split into two 32-bit words, offset split likewise) and key (seed
// split likewise), and is kept when that word is >= floor(p 2^32).
namespace qlora {

// One Philox4x32-10 block.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
        k.x += 0x9E3779B9u;
        k.y += 0xBB67AE85u;
    }
    return c;
}

// x_d[e] = bf16(x[e] * inv) where kept, 0 where dropped; mask_bits (nullable): bit e % 32 of word
// e / 32 set where element e is kept.  One thread per block of 4 elements and step; the loads of
// kDropUnroll steps are issued before any is used (the stream is otherwise latency-bound).
static constexpr int kDropUnroll = 4;

__global__ void __launch_bounds__(256)
    dropout_x_kernel(const uint16_t *__restrict__ X, int64_t n, uint64_t seed, uint64_t offset, uint32_t thr,
                     float inv, uint16_t *__restrict__ Xd, uint32_t *__restrict__ mask_bits) {
    const uint2 key = make_uint2((uint32_t)seed, (uint32_t)(seed >> 32));
    const int64_t nblk = n / 4;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    // warp-uniform loop: the mask gathering below shuffles across lanes
    for (int64_t b0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b0 - (threadIdx.x & 31) < nblk;
         b0 += kDropUnroll * stride) {
        uint2 xv[kDropUnroll];
#pragma unroll
        for (int u = 0; u < kDropUnroll; ++u) {
            const int64_t b = b0 + u * stride;
            xv[u] = b < nblk ? *reinterpret_cast<const uint2 *>(X + 4 * b) : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kDropUnroll; ++u) {
            const int64_t b = b0 + u * stride;
            if (b - (threadIdx.x & 31) >= nblk) break;  // uniform over the warp
            uint32_t nib = 0;
            if (b < nblk) {
                const uint4 w = philox4x32_10(make_uint4((uint32_t)b, (uint32_t)((uint64_t)b >> 32), (uint32_t)offset,
                                                         (uint32_t)(offset >> 32)),
                                              key);
                const uint32_t words[4] = {w.x, w.y, w.z, w.w};
                const uint32_t xs[4] = {xv[u].x & 0xffffu, xv[u].x >> 16, xv[u].y & 0xffffu, xv[u].y >> 16};
                uint32_t o[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const bool keep = words[i] >= thr;
                    nib |= (keep ? 1u : 0u) << i;
                    __nv_bfloat16 h = __float2bfloat16_rn(keep ? __fmul_rn(__uint_as_float(xs[i] << 16), inv) : 0.0f);
                    o[i] = *reinterpret_cast<uint16_t *>(&h);
                }
                *reinterpret_cast<uint2 *>(Xd + 4 * b) = make_uint2(o[0] | (o[1] << 16), o[2] | (o[3] << 16));
            }
            if (mask_bits) {
                // eight lanes cover 32 consecutive elements: gather their nibbles into one word
                uint32_t word = nib << (4 * (threadIdx.x & 7));
                word |= __shfl_xor_sync(0xffffffffu, word, 1);
                word |= __shfl_xor_sync(0xffffffffu, word, 2);
                word |= __shfl_xor_sync(0xffffffffu, word, 4);
                if ((threadIdx.x & 7) == 0 && b < nblk) mask_bits[b / 8] = word;
            }
        }
    }
}

cudaError_t launch_dropout_x(const uint16_t *X, int64_t n, uint64_t seed, uint64_t offset, float p, uint16_t *Xd,
                             uint32_t *mask_bits, int num_sms, cudaStream_t st) {
    const uint32_t thr = (uint32_t)floor((double)p * 4294967296.0);
    const float inv = 1.0f / (1.0f - p);
    const int64_t nblk = n / 4;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((nblk + 255) / 256, (int64_t)num_sms * 8));
    dropout_x_kernel<<<grid, 256, 0, st>>>(X, n, seed, offset, thr, inv, Xd, mask_bits);
    count_launch();
    return cudaGetLastError();
}

}  // namespace qlora
