// noalloc.cu -- nf4_quantize for callers that cannot allocate device memory.
//
// nf4_quantize needs scratch space for the per-block scales and the group sums of the scale
// mean.  Normally the caller passes it as a workspace.  Some callers cannot: a serving process or
// plugin host that reserves its whole device-memory budget up front and forbids any further
// allocation, or an embedding runtime whose own allocator must not be bypassed and that has no
// way to hand out a temporary buffer sized per matrix.  For them this file keeps one fixed
// scratch area in the library's own device module, sized for matrices of up to 2^28 weights.
namespace qlora {

// Largest matrix served: 2^28 weights (for example 16384 x 16384 or 28672 x 8192).
static constexpr int64_t kNoAllocMaxWeights = (int64_t)1 << 28;
static constexpr int64_t kNoAllocMaxBlocks = kNoAllocMaxWeights / kBlock;  // 4,194,304 block scales
static constexpr int64_t kNoAllocMaxTree = 16384;  // power of two >= max blocks / 256 (group sums)
// fp32 block scales, then two fp64 buffers of the group-sum tree: 16 MiB + 256 KiB.
static constexpr size_t kNoAllocScratchBytes =
    (size_t)kNoAllocMaxBlocks * sizeof(float) + 2 * (size_t)kNoAllocMaxTree * sizeof(double);

// Allocated with the module on every device that loads the library and held until process exit.
// In host code this name is a host-side stand-in, not a device address: the device address is
// looked up with cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch area on the current device.  Looked up on every call (a
// driver-side table read, negligible next to a quantize) so that no address outlives the module
// it belongs to, e.g. across cudaDeviceReset, which unloads and reloads the module.  A failed
// lookup is cleared from the thread's last-error state so that it cannot surface in a later call.
static cudaError_t noalloc_scratch(void **out) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return e;
    }
    *out = p;
    return cudaSuccess;
}

}  // namespace qlora

extern "C" qlora_status nf4_quantize_noalloc(const float *W, const qlora_nf4_tensor *out, void *stream) {
    using namespace qlora;
    if (!W) return QLORA_ERR_INVALID_ARG;
    qlora_status s = check_tensor(out);
    if (s != QLORA_OK) return s;
    if (!aligned16(W)) return QLORA_ERR_MISALIGNED;
    if (out->rows * out->cols > kNoAllocMaxWeights) return QLORA_ERR_UNSUPPORTED_SHAPE;
    const QuantWs w = quant_ws(out->rows, out->cols);
    if (w.total > kNoAllocScratchBytes || w.p2 > kNoAllocMaxTree) return QLORA_ERR_UNSUPPORTED_SHAPE;
    void *scratch = nullptr;
    if (noalloc_scratch(&scratch) != cudaSuccess) return QLORA_ERR_CUDA;
    // every byte the kernels read from the scratch is written earlier in the same call, so
    // nothing has to be cleared between calls
    uint8_t *base = static_cast<uint8_t *>(scratch);
    return from_cuda(launch_quantize(W, out->rows * out->cols, out->codes, out->scale_codes, out->scale_scales,
                                     out->scale_offset, reinterpret_cast<float *>(base + w.off_absmax),
                                     reinterpret_cast<double *>(base + w.off_tree), w.p2, tables(), num_sms_current(),
                                     static_cast<cudaStream_t>(stream)));
}
