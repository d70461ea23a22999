// cat.cu -- concatenated projections sharing one input: qlora_linear_fwd_cat / _bwd_cat.
//
// Modules applied to the same X (q/k/v, gate/up) run as one N-concatenated layer.  The call
// assembles, in its workspace, a concatenated view that the fused kernels already understand:
//   - the modules' packed codes end to end (one copy; for M > 32 the layer is bound by the tensor
//     cores, and the copy costs a few microseconds next to the GEMM);
//   - their rebuilt block scales side by side in one [K/64][sum N] table;
//   - A_cat = [A_0; A_1; ...] with each module's rows at offset c_i (rank padded to 8), and the
//     block-diagonal B_cat [sum N, R8] (module i's B_i at rows o_i, columns c_i);
//   - a per-column scale s_i for the pre-scaled U_cat = bf16(s (X A_cat^T)) and V_cat.
// The one fused GEMM then gives Y_cat = X W^_cat^T + U_cat B_cat^T, whose column block i is module
// i's layer output; in the backward, dX = dY_cat W^_cat + V_cat A_cat sums all modules in one fp32
// accumulation.  dA_i and dB_i come from column slices of V_cat, U_cat and dY_cat.
// For M <= 32 the layer streams the codes, so copying them would double its traffic: the call
// runs the modules one after another through the single-module path instead.
// Sources: "LoRA y QLoRA para un ajuste eficiente en costes" (coddykit), "Módulos objetivo"
// (attention projections, or all linear layers); "QLoRA -- La base en 4 bits, LoRA encima"
// (paperclase), "Parte 4 - LoRA encima" for each module's layer.

namespace qlora {

static constexpr int kCatMaxModules = 4;

struct CatScales {
    int G;
    int c[kCatMaxModules], r[kCatMaxModules];
    float s[kCatMaxModules];
};

// col_scale[j] = s_i for c_i <= j < c_i + r_i, else 0
__global__ void cat_col_scales_kernel(float *out, int R8, CatScales cs) {
    for (int j = threadIdx.x; j < R8; j += blockDim.x) {
        float v = 0.0f;
        for (int i = 0; i < cs.G; ++i)
            if (j >= cs.c[i] && j < cs.c[i] + cs.r[i]) v = cs.s[i];
        out[j] = v;
    }
}

// dst[e] = bf16(sum_g f32(src[g * stride + e])), modules summed in order
__global__ void cat_sum_bf16_kernel(const uint16_t *__restrict__ src, int G, int64_t stride, int64_t n,
                                    uint16_t *__restrict__ dst) {
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
        float acc = __uint_as_float((uint32_t)src[e] << 16);
        for (int g = 1; g < G; ++g) acc = __fadd_rn(acc, __uint_as_float((uint32_t)src[(int64_t)g * stride + e] << 16));
        __nv_bfloat16 h = __float2bfloat16_rn(acc);
        dst[e] = *reinterpret_cast<uint16_t *>(&h);
    }
}

struct CatShape {
    int G;
    int64_t M, K, KB, Ncat, Nmax;
    int R8, r8max;
    int64_t N[kCatMaxModules], o[kCatMaxModules];
    int r[kCatMaxModules], c[kCatMaxModules];
};

static bool cat_shape(const int64_t *N, const int32_t *r, int32_t G, int64_t M, int64_t K, CatShape &cs) {
    if (!N || !r || G < 1 || G > kCatMaxModules || M < 1 || M > (1LL << 31) - 1 || K < 64 || K % 64 != 0) return false;
    cs = CatShape{};
    cs.G = G;
    cs.M = M;
    cs.K = K;
    cs.KB = K / 64;
    for (int i = 0; i < G; ++i) {
        if (N[i] < 128 || N[i] % 128 != 0 || r[i] < 1 || r[i] > 256) return false;
        cs.N[i] = N[i];
        cs.o[i] = cs.Ncat;
        cs.Ncat += N[i];
        cs.Nmax = std::max(cs.Nmax, N[i]);
        cs.r[i] = r[i];
        cs.c[i] = cs.R8;
        cs.R8 += ((r[i] + 7) / 8) * 8;
        cs.r8max = std::max(cs.r8max, ((r[i] + 7) / 8) * 8);
    }
    return cs.R8 <= 256;
}

struct CatWs {
    FusedPlan fp;
    ProjPlan pu, pv;
    size_t off_codes, off_scales, off_acat, off_bcat, off_cs, off_u, off_v, off_main, total;
    // M <= 32: per-module calls
    size_t off_sub, sub_bytes, off_ytmp, off_utmp, off_dytmp, off_dxtmp;
};

static CatWs cat_ws(const CatShape &s, bool bwd, int num_sms) {
    CatWs w{};
    size_t off = 0;
    if (s.M > 32) {
        const int r64 = ((s.R8 + 63) / 64) * 64;
        w.fp = bwd ? plan_fused(s.M, s.K, (s.Ncat + 63) / 64, r64, num_sms) : plan_fused(s.M, s.Ncat, s.KB, r64, num_sms);
        w.pu = plan_proj(s.M, s.K, r64, num_sms);
        w.pv = plan_proj(s.M, s.Ncat, r64, num_sms);
        w.off_codes = off;
        off += align256((size_t)s.Ncat * (size_t)s.K / 2);
        w.off_scales = off;
        off += align256((size_t)s.KB * (size_t)s.Ncat * 4);
        w.off_acat = off;
        off += align256((size_t)s.R8 * (size_t)s.K * 2);
        w.off_bcat = off;
        off += align256((size_t)s.Ncat * (size_t)s.R8 * 2);
        w.off_cs = off;
        off += align256((size_t)s.R8 * 4);
        w.off_u = off;
        off += align256((size_t)s.M * (size_t)s.R8 * 2);
        w.off_v = off;
        if (bwd) off += align256((size_t)s.M * (size_t)s.R8 * 2);
        w.off_main = off;
        off += align256(w.fp.partial_bytes);
    } else {
        for (int i = 0; i < s.G; ++i) {
            const size_t b = bwd ? qlora_bwd_workspace_bytes(s.M, s.N[i], s.K, s.r[i])
                                 : qlora_fwd_workspace_bytes(s.M, s.N[i], s.K, s.r[i]);
            w.sub_bytes = std::max(w.sub_bytes, b);
        }
        w.off_sub = off;
        off += align256(w.sub_bytes);
        w.off_ytmp = off;  // forward: Y_i; backward: dY_i
        off += align256((size_t)s.M * (size_t)s.Nmax * 2);
        w.off_dytmp = w.off_ytmp;
        w.off_utmp = off;
        off += align256((size_t)s.M * (size_t)s.r8max * 2);
        w.off_dxtmp = off;
        if (bwd) off += align256((size_t)s.G * (size_t)s.M * (size_t)s.K * 2);
    }
    w.total = std::max<size_t>(off, 256);
    return w;
}

static qlora_status cat_check(const qlora_cat_module *mods, int32_t G, const uint16_t *X, int64_t M, CatShape &cs) {
    if (!mods || !X || G < 1 || G > kCatMaxModules) return QLORA_ERR_INVALID_ARG;
    int64_t N[kCatMaxModules];
    int32_t r[kCatMaxModules];
    int64_t K = -1;
    for (int i = 0; i < G; ++i) {
        qlora_status s = check_layer_args(mods[i].W, X, M, mods[i].A, mods[i].B, mods[i].r, mods[i].alpha);
        if (s != QLORA_OK) return s;
        if (K >= 0 && mods[i].W->cols != K) return QLORA_ERR_UNSUPPORTED_SHAPE;
        K = mods[i].W->cols;
        N[i] = mods[i].W->rows;
        r[i] = mods[i].r;
    }
    return cat_shape(N, r, G, M, K, cs) ? QLORA_OK : QLORA_ERR_UNSUPPORTED_SHAPE;
}

// The concatenated codes and rebuilt scales (read only by the fused kernel).
static cudaError_t cat_assemble_weights(const qlora_cat_module *mods, const CatShape &s, uint8_t *codes,
                                        float *scalesT, cudaStream_t st) {
    cudaError_t e;
    for (int i = 0; i < s.G; ++i) {
        const qlora_nf4_tensor *W = mods[i].W;
        if ((e = cudaMemcpyAsync(codes + s.o[i] * s.K / 2, W->codes, (size_t)s.N[i] * s.K / 2, cudaMemcpyDeviceToDevice,
                                 st)) != cudaSuccess)
            return e;
        if ((e = launch_dq_scales_t(W->scale_codes, W->scale_scales, W->scale_offset, s.N[i], (int)s.KB,
                                    scalesT + s.o[i], st, s.Ncat)) != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

// A_cat, block-diagonal B_cat and the column scales.
static cudaError_t cat_assemble_adapters(const qlora_cat_module *mods, const CatShape &s, uint16_t *Acat,
                                         uint16_t *Bcat, float *cscale, cudaStream_t st) {
    cudaError_t e;
    if ((e = cudaMemsetAsync(Acat, 0, (size_t)s.R8 * s.K * 2, st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(Bcat, 0, (size_t)s.Ncat * s.R8 * 2, st)) != cudaSuccess) return e;
    CatScales sc{};
    sc.G = s.G;
    for (int i = 0; i < s.G; ++i) {
        if ((e = cudaMemcpyAsync(Acat + (int64_t)s.c[i] * s.K, mods[i].A, (size_t)s.r[i] * s.K * 2,
                                 cudaMemcpyDeviceToDevice, st)) != cudaSuccess)
            return e;
        if ((e = cudaMemcpy2DAsync(Bcat + s.o[i] * s.R8 + s.c[i], (size_t)s.R8 * 2, mods[i].B, (size_t)s.r[i] * 2,
                                   (size_t)s.r[i] * 2, (size_t)s.N[i], cudaMemcpyDeviceToDevice, st)) != cudaSuccess)
            return e;
        sc.c[i] = s.c[i];
        sc.r[i] = s.r[i];
        sc.s[i] = mods[i].alpha / (float)mods[i].r;
    }
    cat_col_scales_kernel<<<1, 256, 0, st>>>(cscale, s.R8, sc);
    count_launch();
    return cudaGetLastError();
}

static ProjArgs cat_proj_args(const ProjPlan &pl, int64_t Mp, int r64, int r, int mode) {
    ProjArgs a{};
    a.Mp = (int)Mp;
    a.r64 = r64;
    a.r = r;
    a.tiles = pl.tiles;
    a.splits = pl.splits;
    a.ktiles = pl.ktiles;
    a.mode = mode;
    a.scale = 1.0f;
    return a;
}

static FusedArgs cat_fused_args(const CatShape &s, const FusedPlan &fp, int64_t Nrows, const uint16_t *lora_src,
                                int64_t lora_ld, uint16_t *out, float *partial, int64_t wdim) {
    FusedArgs fa{};
    fa.N = Nrows;
    fa.K = s.K;
    fa.KB = (int32_t)s.KB;
    fa.M = (int32_t)s.M;
    fa.lora_src = lora_src;
    fa.lora_ld = lora_ld;
    fa.r = s.R8;
    fa.BN = fp.BN;
    fa.w_tiles = fp.w_tiles;
    fa.m_tiles = fp.m_tiles;
    fa.splits = fp.splits;
    fa.kt_main = fp.kt_main;
    fa.kt_lora = fp.kt_lora;
    fa.out = out;
    fa.partial = partial;
    fa.wdim = wdim;
    fa.tab = tables();
    return fa;
}

// bf16 view of columns [col0, col0 + cols) of a row-major [rows, ld] matrix
static bool map_cols(CUtensorMap *m, const uint16_t *base, int64_t col0, int64_t cols, int64_t rows, int64_t ld,
                     uint32_t bi, uint32_t bo) {
    return make_map(m, base + col0, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)cols, (uint64_t)rows, (uint64_t)ld, bi,
                    bo, true);
}

}  // namespace qlora

using namespace qlora;

extern "C" {

size_t qlora_cat_fwd_workspace_bytes(const int64_t *N, const int32_t *r, int32_t G, int64_t M, int64_t K) {
    CatShape s;
    if (!cat_shape(N, r, G, M, K, s)) return (size_t)-1;
    return cat_ws(s, false, num_sms_current()).total;
}

size_t qlora_cat_bwd_workspace_bytes(const int64_t *N, const int32_t *r, int32_t G, int64_t M, int64_t K) {
    CatShape s;
    if (!cat_shape(N, r, G, M, K, s)) return (size_t)-1;
    return cat_ws(s, true, num_sms_current()).total;
}

qlora_status qlora_linear_fwd_cat(const qlora_cat_module *mods, int32_t G, const uint16_t *X, int64_t M,
                                  uint16_t *Y, uint16_t *U_save, void *ws, size_t ws_bytes, void *stream) {
    CatShape s;
    qlora_status st_ = cat_check(mods, G, X, M, s);
    if (st_ != QLORA_OK) return st_;
    if (!Y) return QLORA_ERR_INVALID_ARG;
    if (!aligned16(Y) || (U_save && !aligned16(U_save))) return QLORA_ERR_MISALIGNED;
    const int sms = num_sms_current();
    const CatWs w = cat_ws(s, false, sms);
    if (!ws || ws_bytes < w.total || !aligned16(ws)) return QLORA_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *base = static_cast<uint8_t *>(ws);
    cudaError_t e;
    if (U_save && (e = cudaMemsetAsync(U_save, 0, (size_t)M * s.R8 * 2, st)) != cudaSuccess) return from_cuda(e);

    if (M <= 32) {
        // one module at a time through the single-module path, outputs copied into their columns
        uint16_t *Yt = reinterpret_cast<uint16_t *>(base + w.off_ytmp);
        uint16_t *Ut = reinterpret_cast<uint16_t *>(base + w.off_utmp);
        for (int i = 0; i < G; ++i) {
            st_ = qlora_linear_fwd(mods[i].W, X, M, mods[i].A, mods[i].B, mods[i].r, mods[i].alpha, Yt,
                                   U_save ? Ut : nullptr, base + w.off_sub, w.sub_bytes, stream);
            if (st_ != QLORA_OK) return st_;
            if ((e = cudaMemcpy2DAsync(Y + s.o[i], (size_t)s.Ncat * 2, Yt, (size_t)s.N[i] * 2, (size_t)s.N[i] * 2,
                                       (size_t)M, cudaMemcpyDeviceToDevice, st)) != cudaSuccess)
                return from_cuda(e);
            if (U_save && (e = cudaMemcpy2DAsync(U_save + s.c[i], (size_t)s.R8 * 2, Ut, (size_t)s.r[i] * 2,
                                                 (size_t)s.r[i] * 2, (size_t)M, cudaMemcpyDeviceToDevice, st)) != cudaSuccess)
                return from_cuda(e);
        }
        return QLORA_OK;
    }

    uint8_t *codes = base + w.off_codes;
    float *scalesT = reinterpret_cast<float *>(base + w.off_scales);
    uint16_t *Acat = reinterpret_cast<uint16_t *>(base + w.off_acat);
    uint16_t *Bcat = reinterpret_cast<uint16_t *>(base + w.off_bcat);
    float *cscale = reinterpret_cast<float *>(base + w.off_cs);
    uint16_t *U = reinterpret_cast<uint16_t *>(base + w.off_u);
    float *mainp = reinterpret_cast<float *>(base + w.off_main);
    const int r64 = ((s.R8 + 63) / 64) * 64;
    // the concatenated weight on a side stream, alongside the adapter product
    Fork fk(st);
    if ((e = fk.fork()) != cudaSuccess) return from_cuda(e);
    if ((e = cat_assemble_weights(mods, s, codes, scalesT, fk.side(0))) != cudaSuccess) return from_cuda(e);
    if ((e = cat_assemble_adapters(mods, s, Acat, Bcat, cscale, st)) != cudaSuccess) return from_cuda(e);

    CUtensorMap mX_k, mA_k, mCodes, mScales, mX_act, mU_act, mY;
    if (!map_bf16(&mX_k, X, s.K, M, 64, 128) || !map_bf16(&mA_k, Acat, s.K, s.R8, 64, r64) ||
        !map_codes(&mCodes, codes, s.Ncat, s.K, false) || !map_scales(&mScales, scalesT, s.Ncat, s.KB, false) ||
        !map_bf16(&mX_act, X, s.K, M, 64, w.fp.act_rows) || !map_bf16(&mU_act, U, s.R8, M, 64, w.fp.act_rows) ||
        !map_out(&mY, Y, M, s.Ncat))
        return QLORA_ERR_CUDA;
    // U_cat = bf16(s_col (X A_cat^T))  [M, R8] (+ U_save)
    ProjArgs pu = cat_proj_args(w.pu, M, r64, s.R8, 0);
    pu.col_scale = cscale;
    pu.out_h = U;
    pu.ld_h = s.R8;
    pu.out_h2 = U_save;
    if ((e = launch_proj(false, false, mX_k, mA_k, pu, st)) != cudaSuccess) return from_cuda(e);
    if ((e = fk.join(0)) != cudaSuccess) return from_cuda(e);
    // Y_cat = X W^_cat^T + U_cat B_cat^T
    const FusedArgs fa = cat_fused_args(s, w.fp, s.Ncat, Bcat, s.R8, Y, mainp, s.Ncat);
    if ((e = timed_fused(false, mCodes, mScales, mX_act, mU_act, mY, fa, w.fp, sms, st)) != cudaSuccess)
        return from_cuda(e);
    return QLORA_OK;
}

qlora_status qlora_linear_bwd_cat(const qlora_cat_module *mods, int32_t G, const uint16_t *X, int64_t M,
                                  const uint16_t *dY, const uint16_t *U_saved, uint16_t *dX, float *const *dA,
                                  float *const *dB, void *ws, size_t ws_bytes, void *stream) {
    CatShape s;
    qlora_status st_ = cat_check(mods, G, X, M, s);
    if (st_ != QLORA_OK) return st_;
    if (!dY || !dX || !dA || !dB) return QLORA_ERR_INVALID_ARG;
    for (int i = 0; i < G; ++i)
        if (!dA[i] || !dB[i]) return QLORA_ERR_INVALID_ARG;
    if (!aligned16(dY) || !aligned16(dX) || (U_saved && !aligned16(U_saved))) return QLORA_ERR_MISALIGNED;
    for (int i = 0; i < G; ++i)
        if (!aligned16(dA[i]) || !aligned16(dB[i])) return QLORA_ERR_MISALIGNED;
    const int sms = num_sms_current();
    const CatWs w = cat_ws(s, true, sms);
    if (!ws || ws_bytes < w.total || !aligned16(ws)) return QLORA_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *base = static_cast<uint8_t *>(ws);
    cudaError_t e;

    if (M <= 32) {
        uint16_t *dYt = reinterpret_cast<uint16_t *>(base + w.off_dytmp);
        uint16_t *Ut = reinterpret_cast<uint16_t *>(base + w.off_utmp);
        uint16_t *dXt = reinterpret_cast<uint16_t *>(base + w.off_dxtmp);
        for (int i = 0; i < G; ++i) {
            if ((e = cudaMemcpy2DAsync(dYt, (size_t)s.N[i] * 2, dY + s.o[i], (size_t)s.Ncat * 2, (size_t)s.N[i] * 2,
                                       (size_t)M, cudaMemcpyDeviceToDevice, st)) != cudaSuccess)
                return from_cuda(e);
            if (U_saved && (e = cudaMemcpy2DAsync(Ut, (size_t)s.r[i] * 2, U_saved + s.c[i], (size_t)s.R8 * 2,
                                                  (size_t)s.r[i] * 2, (size_t)M, cudaMemcpyDeviceToDevice, st)) != cudaSuccess)
                return from_cuda(e);
            st_ = qlora_linear_bwd(mods[i].W, X, M, mods[i].A, mods[i].B, mods[i].r, mods[i].alpha, dYt,
                                   U_saved ? Ut : nullptr, dXt + (int64_t)i * M * s.K, dA[i], dB[i], base + w.off_sub,
                                   w.sub_bytes, stream);
            if (st_ != QLORA_OK) return st_;
        }
        const int64_t n = M * s.K;
        const int g = (int)std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, (int64_t)sms * 8));
        cat_sum_bf16_kernel<<<g, 256, 0, st>>>(dXt, G, n, n, dX);
        count_launch();
        return from_cuda(cudaGetLastError());
    }

    uint8_t *codes = base + w.off_codes;
    float *scalesT = reinterpret_cast<float *>(base + w.off_scales);
    uint16_t *Acat = reinterpret_cast<uint16_t *>(base + w.off_acat);
    uint16_t *Bcat = reinterpret_cast<uint16_t *>(base + w.off_bcat);
    float *cscale = reinterpret_cast<float *>(base + w.off_cs);
    uint16_t *U = reinterpret_cast<uint16_t *>(base + w.off_u);
    uint16_t *V = reinterpret_cast<uint16_t *>(base + w.off_v);
    float *mainp = reinterpret_cast<float *>(base + w.off_main);
    const int r64 = ((s.R8 + 63) / 64) * 64;
    Fork fk(st);
    if ((e = cat_assemble_adapters(mods, s, Acat, Bcat, cscale, st)) != cudaSuccess) return from_cuda(e);
    const uint16_t *Uq = U_saved ? U_saved : U;

    CUtensorMap mX_k, mA_k, mG_k, mB_mn, mX_mn, mCodes, mScales, mG_act, mV_act, mDX;
    if (!map_bf16(&mX_k, X, s.K, M, 64, 128) || !map_bf16(&mA_k, Acat, s.K, s.R8, 64, r64) ||
        !map_bf16(&mG_k, dY, s.Ncat, M, 64, 128) || !map_bf16(&mB_mn, Bcat, s.R8, s.Ncat, 64, 64) ||
        !map_bf16(&mX_mn, X, s.K, M, 64, 64) || !map_codes(&mCodes, codes, s.Ncat, s.K, true) ||
        !map_scales(&mScales, scalesT, s.Ncat, s.KB, true) || !map_bf16(&mG_act, dY, s.Ncat, M, 64, w.fp.act_rows) ||
        !map_bf16(&mV_act, V, s.R8, M, 64, w.fp.act_rows) || !map_out(&mDX, dX, M, s.K))
        return QLORA_ERR_CUDA;
    if (!U_saved) {
        ProjArgs pu = cat_proj_args(w.pu, M, r64, s.R8, 0);
        pu.col_scale = cscale;
        pu.out_h = U;
        pu.ld_h = s.R8;
        if ((e = launch_proj(false, false, mX_k, mA_k, pu, st)) != cudaSuccess) return from_cuda(e);
    }
    // from here: the concatenated weight and the dB_i on the side streams, V_cat here
    if ((e = fk.fork()) != cudaSuccess) return from_cuda(e);
    if ((e = cat_assemble_weights(mods, s, codes, scalesT, fk.side(0))) != cudaSuccess) return from_cuda(e);
    for (int i = 0; i < G; ++i) {  // dB_i = dY_i^T U_i (column slices)
        const int ri64 = ((s.r[i] + 63) / 64) * 64;
        CUtensorMap mG_i, mU_i;
        if (!map_cols(&mG_i, dY, s.o[i], s.N[i], M, s.Ncat, 64, 64) ||
            !map_cols(&mU_i, Uq, s.c[i], s.r[i], M, s.R8, 64, 64))
            return QLORA_ERR_CUDA;
        ProjArgs pb = cat_proj_args(plan_proj(s.N[i], M, ri64, sms), s.N[i], ri64, s.r[i], 2);
        pb.out_f = dB[i];
        if ((e = launch_proj(true, true, mG_i, mU_i, pb, fk.side(1))) != cudaSuccess) return from_cuda(e);
    }
    // V_cat = bf16(s_col (dY_cat B_cat))  [M, R8]
    ProjArgs pv = cat_proj_args(w.pv, M, r64, s.R8, 0);
    pv.col_scale = cscale;
    pv.out_h = V;
    pv.ld_h = s.R8;
    if ((e = launch_proj(false, true, mG_k, mB_mn, pv, st)) != cudaSuccess) return from_cuda(e);
    // dX on the high-priority stream; the dA_i here, in the SMs its last wave leaves idle
    cudaStream_t hp = fk.priority();
    if ((e = fk.link(st, hp)) != cudaSuccess || (e = fk.link(fk.side(0), hp)) != cudaSuccess) return from_cuda(e);
    // dX = dY_cat W^_cat + V_cat A_cat
    const FusedArgs fa = cat_fused_args(s, w.fp, s.Ncat, Acat, s.K, dX, mainp, s.K);
    if ((e = timed_fused(true, mCodes, mScales, mG_act, mV_act, mDX, fa, w.fp, sms, hp)) != cudaSuccess)
        return from_cuda(e);
    // per module: dA_i = V_i^T X (column slices of V_cat)
    for (int i = 0; i < G; ++i) {
        const int ri64 = ((s.r[i] + 63) / 64) * 64;
        CUtensorMap mV_i;
        if (!map_cols(&mV_i, V, s.c[i], s.r[i], M, s.R8, 64, 64)) return QLORA_ERR_CUDA;
        ProjArgs pa = cat_proj_args(plan_proj(s.K, M, ri64, sms), s.K, ri64, s.r[i], 1);
        pa.out_f = dA[i];
        if ((e = launch_proj(true, true, mX_mn, mV_i, pa, st)) != cudaSuccess) return from_cuda(e);
    }
    if ((e = fk.link(hp, st)) != cudaSuccess || (e = fk.join(1)) != cudaSuccess) return from_cuda(e);
    return QLORA_OK;
}

}  // extern "C"
