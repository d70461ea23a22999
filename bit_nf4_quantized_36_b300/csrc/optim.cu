// optim.cu -- the adapters' AdamW step over paged (unified-memory) optimizer states.
//
// Only the two LoRA matrices are trained ("QLoRA" glossary entry (ultralytics.com), "Como funciona
// a QLoRA"), and their optimizer states are paged: they live in NVIDIA unified memory and move to
// CPU RAM when GPU memory runs short ("Otimizadores paginados" bullet there; "Capitulo 1: Que es
// QLoRA?" (docs.skillversehub.com), "Componentes clave", "Optimizadores paginados").
//
// The states are allocated with cudaMallocManaged, so the driver may evict their pages to host
// memory under oversubscription and bring them back on the next GPU touch.  The caller moves them
// explicitly around a memory spike with qlora_paged_prefetch: to the host before the spike, back
// to the device before the next optimizer step, so that the step itself runs at HBM speed rather
// than at page-fault speed.
//
// The step is AdamW (Loshchilov and Hutter, "Decoupled weight decay regularization", ICLR 2019)
// on fp32 master weights with fp32 first and second moments, and optionally writes the bf16 copy
// of the weights that the layer kernels read.  It is a pure stream: per element it reads p, g, m,
// v (16 bytes) and writes p, m, v (+ the bf16 copy): 28 or 30 bytes, HBM-bound.
namespace qlora {

struct AdamWCoef {
    float decay;         // 1 - lr * weight_decay
    float b1, c1;        // beta1, 1 - beta1
    float b2, c2;        // beta2, 1 - beta2
    float step_size;     // lr / (1 - beta1^t)
    float bc2_sqrt;      // sqrt(1 - beta2^t)
    float eps;
};

__device__ __forceinline__ void adamw_elem(float &p, float g, float &m, float &v, const AdamWCoef &c) {
    p = __fmul_rn(p, c.decay);
    m = __fmaf_rn(c.b1, m, __fmul_rn(c.c1, g));
    v = __fmaf_rn(c.b2, v, __fmul_rn(c.c2, __fmul_rn(g, g)));
    const float denom = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), c.bc2_sqrt), c.eps);
    p = __fsub_rn(p, __fmul_rn(c.step_size, __fdiv_rn(m, denom)));
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
    __nv_bfloat16 a = __float2bfloat16_rn(lo), b = __float2bfloat16_rn(hi);
    return (uint32_t)*reinterpret_cast<uint16_t *>(&a) | ((uint32_t)*reinterpret_cast<uint16_t *>(&b) << 16);
}

// Grid-stride over groups of 4 elements (16-byte loads and stores, streaming cache hints: every
// byte is touched once); the n % 4 tail is taken by thread 0 of block 0.
__global__ void __launch_bounds__(256)
    adamw_kernel(float *__restrict__ p, const float *__restrict__ g, float *__restrict__ m, float *__restrict__ v,
                 uint16_t *__restrict__ p_bf16, int64_t n, AdamWCoef c) {
    const int64_t n4 = n / 4;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
        float4 pv = __ldcs(reinterpret_cast<const float4 *>(p) + i);
        const float4 gv = __ldcs(reinterpret_cast<const float4 *>(g) + i);
        float4 mv = __ldcs(reinterpret_cast<const float4 *>(m) + i);
        float4 vv = __ldcs(reinterpret_cast<const float4 *>(v) + i);
        adamw_elem(pv.x, gv.x, mv.x, vv.x, c);
        adamw_elem(pv.y, gv.y, mv.y, vv.y, c);
        adamw_elem(pv.z, gv.z, mv.z, vv.z, c);
        adamw_elem(pv.w, gv.w, mv.w, vv.w, c);
        __stcs(reinterpret_cast<float4 *>(p) + i, pv);
        __stcs(reinterpret_cast<float4 *>(m) + i, mv);
        __stcs(reinterpret_cast<float4 *>(v) + i, vv);
        if (p_bf16) __stcs(reinterpret_cast<uint2 *>(p_bf16) + i, make_uint2(bf16x2_bits(pv.x, pv.y), bf16x2_bits(pv.z, pv.w)));
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        for (int64_t e = 4 * n4; e < n; ++e) {
            float pe = p[e], me = m[e], ve = v[e];
            adamw_elem(pe, g[e], me, ve, c);
            p[e] = pe;
            m[e] = me;
            v[e] = ve;
            if (p_bf16) {
                __nv_bfloat16 h = __float2bfloat16_rn(pe);
                p_bf16[e] = *reinterpret_cast<uint16_t *>(&h);
            }
        }
    }
}

cudaError_t launch_adamw(float *p, const float *g, float *m, float *v, uint16_t *p_bf16, int64_t n,
                         const AdamWCoef &c, int num_sms, cudaStream_t st) {
    const int64_t n4 = n / 4;
    // 64 registers a thread: 4 resident blocks of 256 threads per SM, 64 KB of loads in flight
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((n4 + 255) / 256, (int64_t)num_sms * 4));
    adamw_kernel<<<grid, 256, 0, st>>>(p, g, m, v, p_bf16, n, c);
    count_launch();
    return cudaGetLastError();
}

static bool managed_range(const void *ptr) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeManaged;
}

}  // namespace qlora

using namespace qlora;

extern "C" {

qlora_status qlora_paged_alloc(size_t bytes, void **out) {
    if (!out) return QLORA_ERR_INVALID_ARG;
    *out = nullptr;
    if (bytes == 0) return QLORA_ERR_INVALID_ARG;
    int dev = 0, managed = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&managed, cudaDevAttrManagedMemory, dev) != cudaSuccess || !managed) {
        cudaGetLastError();
        return QLORA_ERR_CUDA;
    }
    void *p = nullptr;
    const cudaError_t e = cudaMallocManaged(&p, bytes, cudaMemAttachGlobal);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return QLORA_ERR_CUDA;
    }
    *out = p;
    return QLORA_OK;
}

qlora_status qlora_paged_free(void *ptr) {
    if (!ptr) return QLORA_OK;
    if (!managed_range(ptr)) return QLORA_ERR_INVALID_ARG;
    return cudaFree(ptr) == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}

qlora_status qlora_paged_prefetch(const void *ptr, size_t bytes, int32_t device, void *stream) {
    if (!ptr || device < QLORA_PAGE_HOST) return QLORA_ERR_INVALID_ARG;
    if (bytes == 0) return QLORA_OK;
    if (!managed_range(ptr)) return QLORA_ERR_INVALID_ARG;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess) {
        cudaGetLastError();
        return QLORA_ERR_CUDA;
    }
    if (device >= ndev) return QLORA_ERR_INVALID_ARG;
    int cur = 0, concurrent = 0;
    if (cudaGetDevice(&cur) != cudaSuccess ||
        cudaDeviceGetAttribute(&concurrent, cudaDevAttrConcurrentManagedAccess, device >= 0 ? device : cur) != cudaSuccess) {
        cudaGetLastError();
        return QLORA_ERR_CUDA;
    }
    // Without concurrent managed access the driver migrates the whole allocation at each launch
    // by itself; a prefetch is then only a hint that cannot be given.
    if (!concurrent) return QLORA_OK;
    cudaMemLocation loc{};
    loc.type = device == QLORA_PAGE_HOST ? cudaMemLocationTypeHost : cudaMemLocationTypeDevice;
    loc.id = device == QLORA_PAGE_HOST ? 0 : device;
    const cudaError_t e = cudaMemPrefetchAsync(ptr, bytes, loc, 0, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return QLORA_ERR_CUDA;
    }
    return QLORA_OK;
}

qlora_status qlora_adamw_step(const qlora_adamw *hp, int64_t t, int64_t n, float *p, const float *g, float *m, float *v,
                              uint16_t *p_bf16, void *stream) {
    if (!hp || t < 1 || n < 0) return QLORA_ERR_INVALID_ARG;
    const bool ok = std::isfinite(hp->lr) && hp->lr >= 0.0f && std::isfinite(hp->weight_decay) &&
                    hp->weight_decay >= 0.0f && hp->beta1 >= 0.0f && hp->beta1 < 1.0f && hp->beta2 >= 0.0f &&
                    hp->beta2 < 1.0f && std::isfinite(hp->eps) && hp->eps > 0.0f;
    if (!ok) return QLORA_ERR_INVALID_ARG;
    if (n == 0) return QLORA_OK;
    if (!p || !g || !m || !v) return QLORA_ERR_INVALID_ARG;
    if (!aligned16(p) || !aligned16(g) || !aligned16(m) || !aligned16(v) ||
        (reinterpret_cast<uintptr_t>(p_bf16) & 7u) != 0)
        return QLORA_ERR_MISALIGNED;
    // bias corrections in fp64 on the host, as scalars of the step
    const double bc1 = 1.0 - std::pow((double)hp->beta1, (double)t);
    const double bc2 = 1.0 - std::pow((double)hp->beta2, (double)t);
    AdamWCoef c;
    c.decay = (float)(1.0 - (double)hp->lr * (double)hp->weight_decay);
    c.b1 = hp->beta1;
    c.c1 = (float)(1.0 - (double)hp->beta1);
    c.b2 = hp->beta2;
    c.c2 = (float)(1.0 - (double)hp->beta2);
    c.step_size = (float)((double)hp->lr / bc1);
    c.bc2_sqrt = (float)std::sqrt(bc2);
    c.eps = hp->eps;
    return from_cuda(launch_adamw(p, g, m, v, p_bf16, n, c, num_sms_current(), static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
