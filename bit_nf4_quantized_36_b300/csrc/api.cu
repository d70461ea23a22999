// api.cu -- the C ABI of libqlora (include/qlora.h): argument checks, workspace layout,
// TMA descriptor setup and the launch sequence of each call.  All arithmetic of the layer runs
// in the kernels of quant.cu and gemm.cu.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/qlora.h"
#include "qlora_common.cuh"
#include "qlora_kernels.cuh"

namespace qlora {

static std::atomic<uint64_t> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// optional event pairs around the weight-streaming step of a call (benchmark instrumentation)
static void **g_timer_events = nullptr;
static int32_t g_timer_cap = 0;
static std::atomic<int32_t> g_timer_n{0};

// Records a timer event on `st`.  Under stream capture the record becomes an event-record node
// of the graph, so that the event times every replay.
static cudaError_t timer_record(void *event, cudaStream_t st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return cudaGetLastError();
    return cudaEventRecordWithFlags(static_cast<cudaEvent_t>(event), st,
                                    cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault);
}

// Records the opening event of a timed step; returns its slot, or -1 when not timing.  A failed
// record (e.g. a NULL handle) must not be reported as the kernel's launch error.
static int32_t timer_open(cudaStream_t st) {
    void **ev = g_timer_events;
    if (!ev) return -1;
    int32_t i = g_timer_n.fetch_add(1);
    if (i >= g_timer_cap) return -1;
    if (timer_record(ev[2 * i], st) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return i;
}
static void timer_close(int32_t i, cudaStream_t st) {
    void **ev = g_timer_events;
    if (i >= 0 && ev && timer_record(ev[2 * i + 1], st) != cudaSuccess) cudaGetLastError();
}

// the fused GEMM and, when the contraction is split, the reduction of its partials
static cudaError_t timed_fused(bool dx, const CUtensorMap &mc, const CUtensorMap &ms, const CUtensorMap &ma,
                               const CUtensorMap &ml, const CUtensorMap &mo, const FusedArgs &fa, const FusedPlan &fp,
                               int num_sms, cudaStream_t st) {
    const int32_t i = timer_open(st);
    cudaError_t e = launch_fused(dx, mc, ms, ma, ml, mo, fa, fp, st);
    if (e == cudaSuccess && fp.splits > 1) e = launch_splitk_reduce(fa.partial, fp.splits, fa.M, fa.wdim, fa.out, num_sms, st);
    timer_close(i, st);
    return e;
}

// ---------------------------------------------------------------------------------------
// NF4 tables: the level constants and the exact decision thresholds of the nearest-level
// rule.  thr[k] is the smallest fp32 x in (L_k, L_k+1] with fl(L_k+1 - x) < fl(x - L_k):
// the predicate is monotone in x (fp32 subtraction is monotone), false at L_k and true at
// L_k+1, so a bisection over the ordered fp32 bit patterns finds it exactly.
// ---------------------------------------------------------------------------------------
static int64_t f32_key(float f) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return (u & 0x80000000u) ? -(int64_t)(u & 0x7FFFFFFFu) : (int64_t)u;
}
static float f32_from_key(int64_t k) {
    uint32_t u = k >= 0 ? (uint32_t)k : (0x80000000u | (uint32_t)(-k));
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}
static bool closer_to_upper(volatile float lo, volatile float hi, volatile float x) {
    volatile float du = hi - x;  // fp32, round to nearest
    volatile float dl = x - lo;
    return du < dl;
}

static const NF4Tables &tables() {
    static NF4Tables t;
    static std::once_flag once;
    std::call_once(once, [] {
        for (int i = 0; i < 16; ++i) std::memcpy(&t.level[i], &kNF4Bits[i], 4);
        for (int k = 0; k < 15; ++k) {
            const float lo = t.level[k], hi = t.level[k + 1];
            int64_t a = f32_key(lo), b = f32_key(hi);  // predicate false at a, true at b
            while (b - a > 1) {
                const int64_t m = a + (b - a) / 2;
                if (closer_to_upper(lo, hi, f32_from_key(m))) b = m; else a = m;
            }
            t.thr[k] = f32_from_key(b);
        }
        t.thr[15] = INFINITY;
        for (int j = 0; j < kNF4Buckets; ++j) {
            if (j > 33) {
                t.bucket[j] = 0x7FC00000u;
                continue;
            }
            const double start = -1.0 + (j - 1) / 16.0 - std::ldexp(1.0, -12);
            int c = 0;
            while (c < 15 && (double)t.thr[c] <= start) ++c;
            const float tc = c < 15 ? t.thr[c] : 2.0f;
            uint32_t bits;
            std::memcpy(&bits, &tc, 4);
            t.bucket[j] = (bits & ~15u) | (uint32_t)c;
        }
    });
    return t;
}

// ---------------------------------------------------------------------------------------
// Side streams.  The skinny products and the scale rebuild of one layer call are latency-bound
// (a few microseconds of set-up, pipeline fill and reduction each) and some do not depend on one
// another; those run on two side streams of the current device, forked from and joined back to
// the caller's stream with events, so that their latencies overlap.  A per-device mutex covers
// the enqueue of a call (not its execution), so concurrent host threads never mix up the events.
// If the streams cannot be created, everything runs on the caller's stream.
// ---------------------------------------------------------------------------------------
struct SideStreams {
    std::mutex mu;
    bool tried = false, ok = false;
    cudaStream_t s[2] = {nullptr, nullptr};
    cudaStream_t hp = nullptr;  // the device's highest stream priority
    cudaEvent_t ev = nullptr;   // reused: a wait takes the event's latest record at the time it is enqueued
};

static SideStreams *side_streams() {
    static SideStreams ss[16];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 16) {
        (void)cudaGetLastError();
        return nullptr;
    }
    SideStreams &x = ss[dev];
    std::lock_guard<std::mutex> lock(x.mu);
    if (!x.tried) {
        x.tried = true;
        int least = 0, greatest = 0;
        x.ok = cudaDeviceGetStreamPriorityRange(&least, &greatest) == cudaSuccess &&
               cudaStreamCreateWithFlags(&x.s[0], cudaStreamNonBlocking) == cudaSuccess &&
               cudaStreamCreateWithFlags(&x.s[1], cudaStreamNonBlocking) == cudaSuccess &&
               cudaStreamCreateWithPriority(&x.hp, cudaStreamNonBlocking, greatest) == cudaSuccess &&
               cudaEventCreateWithFlags(&x.ev, cudaEventDisableTiming) == cudaSuccess;
        if (!x.ok) (void)cudaGetLastError();
    }
    return x.ok ? &x : nullptr;
}

// One layer call's use of the side streams: fork() makes both side streams wait for what the
// caller's stream has enqueued so far; side(i) is the stream to launch independent work on and
// priority() a stream whose kernels the block scheduler serves first (both are the caller's own
// stream when side streams are unavailable); link(a, b) makes stream b wait for what stream a has
// enqueued so far; join(i) = link(side(i), caller).  Holds the device's side-stream mutex for its
// lifetime.
class Fork {
  public:
    explicit Fork(cudaStream_t caller) : st_(caller), ss_(side_streams()) {
        if (ss_) lock_ = std::unique_lock<std::mutex>(ss_->mu);
    }
    // A call that returns early (an error after some side work was enqueued) still leaves the
    // caller's stream ordered after everything it enqueued on the side streams.
    ~Fork() {
        if (!ss_) return;
        for (int i = 0; i < 3; ++i)
            if (pending_ & (1u << i)) (void)link(i < 2 ? ss_->s[i] : ss_->hp, st_);
        (void)cudaGetLastError();
    }
    cudaError_t link(cudaStream_t from, cudaStream_t to) {
        if (!ss_ || from == to) return cudaSuccess;
        cudaError_t e = cudaEventRecord(ss_->ev, from);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(to, ss_->ev, 0);
        if (e == cudaSuccess) {
            // work enqueued on a side stream after it waited is pending until it is linked back
            if (to != st_) pending_ |= bit(to);
            if (to == st_) pending_ &= ~bit(from);
        }
        return e;
    }
    cudaError_t fork() {
        cudaError_t e = link(st_, side(0));
        if (e == cudaSuccess) e = link(st_, side(1));
        return e;
    }
    cudaStream_t side(int i) const { return ss_ ? ss_->s[i] : st_; }
    cudaStream_t priority() const { return ss_ ? ss_->hp : st_; }
    cudaStream_t caller() const { return st_; }
    cudaError_t join(int i) { return link(side(i), st_); }

  private:
    uint32_t bit(cudaStream_t x) const {
        return x == ss_->s[0] ? 1u : x == ss_->s[1] ? 2u : x == ss_->hp ? 4u : 0u;
    }
    cudaStream_t st_;
    SideStreams *ss_;
    uint32_t pending_ = 0;  // side streams forked from the caller and not yet joined back
    std::unique_lock<std::mutex> lock_;
};

static int num_sms_current() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return 148; }
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 148;
    }
    return n;
}

// ---------------------------------------------------------------------------------------
// TMA descriptors
// ---------------------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// 2-D row-major tensor [outer, inner] of `esize`-byte elements with row stride `ld` elements.
static bool make_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize, uint64_t inner,
                     uint64_t outer, uint64_t ld, uint32_t box_inner, uint32_t box_outer, bool swz128,
                     CUtensorMapSwizzle swz_other = CU_TENSOR_MAP_SWIZZLE_NONE) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {ld * (uint64_t)esize};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swz128 ? CU_TENSOR_MAP_SWIZZLE_128B : swz_other, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}
static bool map_bf16(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint32_t bi, uint32_t bo) {
    return make_map(m, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, inner, outer, inner, bi, bo, true);
}
// the fused kernel's bf16 output [rows, cols], stored through TMA by each epilogue warp in
// 64-byte-swizzled [32 tokens][32 features] tiles
static bool map_out(CUtensorMap *m, const void *out, int64_t rows, int64_t cols) {
    return make_map(m, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)cols, (uint64_t)rows, (uint64_t)cols, 32u,
                    32u, false, CU_TENSOR_MAP_SWIZZLE_64B);
}
static bool map_codes(CUtensorMap *m, const void *codes, int64_t N, int64_t K, bool dx) {
    return make_map(m, codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)K / 2, (uint64_t)N, (uint64_t)K / 2,
                    dx ? 64u : 32u, dx ? 64u : 128u, false);
}
// the codes for the small-M forward: as a 3-D byte tensor {128 bytes of a row's 256-column unit,
// row, unit} over the whole units only (strides K/2 and 128 bytes; one box is kGemvBoxRows rows x
// kGemvBoxUnits units, stored unit by unit), and as the 2-D tensor {K/2, N} with boxes of one
// unit (128 bytes x kGemvBoxRows rows) for slabs that are not eight whole units; 128-byte swizzle
static bool map_codes_gemv(CUtensorMap *m3, CUtensorMap *m2, const void *codes, int64_t N, int64_t K) {
    auto fn = encode_fn();
    if (!fn) return false;
    const uint64_t whole = (uint64_t)(K / 256);
    cuuint64_t dims[3] = {128u, (uint64_t)N, whole > 0 ? whole : 1u};
    cuuint64_t strides[2] = {(uint64_t)K / 2, 128u};
    cuuint32_t box[3] = {128u, (uint32_t)kGemvBoxRows, (uint32_t)kGemvBoxUnits};
    cuuint32_t estr[3] = {1, 1, 1};
    // (with no whole unit the 3-D map is never used; it is encoded over the first row's bytes)
    if (whole == 0) {
        dims[1] = 1;
        dims[0] = (uint64_t)K / 2 >= 128 ? 128u : 16u;
    }
    CUresult r = fn(m3, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(codes), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    return make_map(m2, codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)K / 2, (uint64_t)N, (uint64_t)K / 2, 128u,
                    (uint32_t)kGemvBoxRows, true);
}
// rebuilt block scales, transposed [KB][N] fp32
static bool map_scales(CUtensorMap *m, const float *sT, int64_t N, int64_t KB, bool dx) {
    return make_map(m, sT, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (uint64_t)N, (uint64_t)KB, (uint64_t)N, dx ? 64u : 128u,
                    dx ? 2u : 1u, false);
}

// ---------------------------------------------------------------------------------------
// Workspace layouts (one function per call, used by the size query and by the call)
// ---------------------------------------------------------------------------------------
static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct QuantWs {
    int64_t nb, ng, p2;
    size_t off_absmax, off_tree, total;
};
static QuantWs quant_ws(int64_t rows, int64_t cols) {
    QuantWs w{};
    w.nb = rows * cols / kBlock;
    w.ng = (w.nb + kGroup - 1) / kGroup;
    w.p2 = 1;
    while (w.p2 < w.ng) w.p2 <<= 1;
    w.off_absmax = 0;
    w.off_tree = align256((size_t)w.nb * 4);
    w.total = w.off_tree + align256((size_t)w.p2 * 2 * sizeof(double));
    return w;
}

struct LayerWs {
    int r8, r64;
    bool gemv;  // forward with M <= 8: the one-launch small-M kernel instead of the fused kernel
    FusedPlan fp;
    ProjPlan pu, pv, pda, pdb;
    size_t off_scales, off_u, off_v, off_bpad, off_main, off_xd, off_mask, total;
};
static LayerWs layer_ws(int64_t M, int64_t N, int64_t K, int r, bool bwd, int num_sms, bool drop = false) {
    LayerWs w{};
    w.r8 = ((r + 7) / 8) * 8;
    w.r64 = ((r + 63) / 64) * 64;
    const int64_t KB = K / 64;
    w.pu = plan_proj(M, K, w.r64, num_sms);
    if (bwd) {
        w.pv = plan_proj(M, N, w.r64, num_sms);
        w.pda = plan_proj(K, M, w.r64, num_sms);
        w.pdb = plan_proj(N, M, w.r64, num_sms);
        w.fp = plan_fused(M, K, (N + 63) / 64, w.r64, num_sms);
    } else {
        w.fp = plan_fused(M, N, K / 64, w.r64, num_sms);
        w.gemv = gemv_supported(M, N, K);
    }
    size_t off = 0;
    w.off_scales = off;  // rebuilt block scales, for the CTA-pair kernel only
    if (!w.fp.small && !w.gemv) off += align256((size_t)KB * N * 4);
    w.off_u = off;
    off += align256((size_t)M * w.r8 * 2);
    w.off_v = off;
    if (bwd) off += align256((size_t)M * w.r8 * 2);
    w.off_bpad = off;
    if (bwd && r % 8 != 0) off += align256((size_t)N * w.r8 * 2);
    w.off_main = off;
    off += align256(w.gemv ? gemv_ws(N, K, r).total : w.fp.partial_bytes);
    // LoRA dropout: the masked adapter input, and (backward) its kept-element bits
    w.off_xd = off;
    if (drop) off += align256((size_t)M * K * 2);
    w.off_mask = off;
    if (drop && bwd) off += align256((size_t)M * K / 8);
    w.total = off;
    return w;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static qlora_status check_tensor(const qlora_nf4_tensor *t) {
    if (!t || !t->codes || !t->scale_codes || !t->scale_scales || !t->scale_offset) return QLORA_ERR_INVALID_ARG;
    if (t->rows < 1 || t->cols < 64 || t->cols % 64 != 0) return QLORA_ERR_UNSUPPORTED_SHAPE;
    if (t->rows > (1LL << 31) || t->cols > (1LL << 31)) return QLORA_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(t->codes)) return QLORA_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(t->scale_scales) & 3u) || (reinterpret_cast<uintptr_t>(t->scale_offset) & 3u))
        return QLORA_ERR_MISALIGNED;
    return QLORA_OK;
}

static qlora_status from_cuda(cudaError_t e) { return e == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA; }

static qlora_status check_layer_args(const qlora_nf4_tensor *W, const uint16_t *X, int64_t M, const uint16_t *A,
                                     const uint16_t *B, int32_t r, float alpha) {
    qlora_status s = check_tensor(W);
    if (s != QLORA_OK) return s;
    if (!X || !A || !B) return QLORA_ERR_INVALID_ARG;
    if (r < 1 || r > 256 || !std::isfinite(alpha)) return QLORA_ERR_INVALID_ARG;
    if (M < 1 || M > (1LL << 31) - 1) return QLORA_ERR_UNSUPPORTED_SHAPE;
    if (W->rows % 8 != 0) return QLORA_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(X) || !aligned16(A) || !aligned16(B)) return QLORA_ERR_MISALIGNED;
    return QLORA_OK;
}

}  // namespace qlora

using namespace qlora;

extern "C" {

const char *qlora_status_string(qlora_status s) {
    switch (s) {
        case QLORA_OK: return "ok";
        case QLORA_ERR_INVALID_ARG: return "invalid argument";
        case QLORA_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case QLORA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case QLORA_ERR_WORKSPACE: return "workspace missing or too small";
        case QLORA_ERR_CUDA: return "CUDA error";
        case QLORA_ERR_TIMEOUT: return "device-side wait timed out";
        case QLORA_ERR_DEVICE_CHECK: return "device-side bounds check failed";
    }
    return "unknown status";
}

uint64_t qlora_launch_count(void) { return g_launches.load(); }

void qlora_nf4_levels(float out[16]) {
    if (!out) return;
    for (int i = 0; i < 16; ++i) out[i] = tables().level[i];
}

size_t qlora_nf4_storage_bytes(int64_t rows, int64_t cols) {
    if (rows < 1 || cols < 64 || cols % 64 != 0) return 0;
    const int64_t n = rows * cols, nb = n / 64, ng = (nb + 255) / 256;
    return (size_t)(n / 2 + nb + 4 * ng + 4);
}

size_t qlora_quantize_workspace_bytes(int64_t rows, int64_t cols) {
    if (rows < 1 || cols < 64 || cols % 64 != 0) return (size_t)-1;
    return quant_ws(rows, cols).total;
}

size_t qlora_fwd_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t r) {
    if (M < 1 || N < 1 || N % 8 != 0 || K < 64 || K % 64 != 0 || r < 1 || r > 256) return (size_t)-1;
    return layer_ws(M, N, K, r, false, num_sms_current()).total;
}

size_t qlora_bwd_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t r) {
    if (M < 1 || N < 1 || N % 8 != 0 || K < 64 || K % 64 != 0 || r < 1 || r > 256) return (size_t)-1;
    return layer_ws(M, N, K, r, true, num_sms_current()).total;
}

size_t qlora_merge_workspace_bytes(int64_t N, int64_t K, int32_t r) {
    if (N < 1 || K < 64 || K % 64 != 0 || r < 1 || r > 256) return (size_t)-1;
    return (r % 8 == 0) ? 0 : align256((size_t)N * (size_t)(((r + 7) / 8) * 8) * 2);
}

qlora_status qlora_merge(const qlora_nf4_tensor *W, const uint16_t *A, const uint16_t *B, int32_t r, float alpha,
                         uint16_t *W_out, void *ws, size_t ws_bytes, void *stream) {
    qlora_status s = check_tensor(W);
    if (s != QLORA_OK) return s;
    if (!A || !B || !W_out) return QLORA_ERR_INVALID_ARG;
    if (r < 1 || r > 256 || !std::isfinite(alpha)) return QLORA_ERR_INVALID_ARG;
    const bool r_vec = (r % 8) == 0;
    if (!aligned16(A) || !aligned16(W_out) || (r_vec && !aligned16(B))) return QLORA_ERR_MISALIGNED;
    const int64_t N = W->rows, K = W->cols;
    const size_t need = qlora_merge_workspace_bytes(N, K, r);
    if (need == (size_t)-1) return QLORA_ERR_UNSUPPORTED_SHAPE;
    if (need > 0 && (!ws || ws_bytes < need || !aligned16(ws))) return QLORA_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int sms = num_sms_current();
    const int r8 = ((r + 7) / 8) * 8;
    const uint16_t *Bq = B;
    cudaError_t e;
    if (!r_vec) {
        uint16_t *Bpad = static_cast<uint16_t *>(ws);
        if ((e = launch_pad_2d(B, N, r, Bpad, N, r8, sms, st)) != cudaSuccess) return from_cuda(e);
        Bq = Bpad;
    }
    CUtensorMap mCodes, mB, mA, mOut;
    if (!make_map(&mCodes, W->codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)K / 2, (uint64_t)N, (uint64_t)K / 2,
                  128u, 128u, true) ||
        !map_bf16(&mB, Bq, r_vec ? r : r8, N, 64, 128) || !map_bf16(&mA, A, K, r, 64, 64) ||
        !map_bf16(&mOut, W_out, K, N, 64, 32))
        return QLORA_ERR_CUDA;
    return from_cuda(launch_merge(mCodes, mB, mA, mOut, W->scale_codes, W->scale_scales, W->scale_offset, N, K, r,
                                  alpha / (float)r, tables(), sms, st));
}

qlora_status nf4_quantize(const float *W, const qlora_nf4_tensor *out, void *ws, size_t ws_bytes, void *stream) {
    if (!W) return QLORA_ERR_INVALID_ARG;
    qlora_status s = check_tensor(out);
    if (s != QLORA_OK) return s;
    if (!aligned16(W)) return QLORA_ERR_MISALIGNED;
    const QuantWs w = quant_ws(out->rows, out->cols);
    if (!ws || ws_bytes < w.total || !aligned16(ws)) return QLORA_ERR_WORKSPACE;
    uint8_t *base = static_cast<uint8_t *>(ws);
    return from_cuda(launch_quantize(W, out->rows * out->cols, out->codes, out->scale_codes, out->scale_scales,
                                     out->scale_offset, reinterpret_cast<float *>(base + w.off_absmax),
                                     reinterpret_cast<double *>(base + w.off_tree), w.p2, tables(), num_sms_current(),
                                     static_cast<cudaStream_t>(stream)));
}

qlora_status nf4_dequantize(const qlora_nf4_tensor *q, uint16_t *W_out, void *stream) {
    qlora_status s = check_tensor(q);
    if (s != QLORA_OK) return s;
    if (!W_out) return QLORA_ERR_INVALID_ARG;
    if (!aligned16(W_out)) return QLORA_ERR_MISALIGNED;
    return from_cuda(launch_dequantize(q->codes, q->scale_codes, q->scale_scales, q->scale_offset, q->rows * q->cols,
                                       W_out, tables(), num_sms_current(), static_cast<cudaStream_t>(stream)));
}

static ProjArgs proj_args(const ProjPlan &pl, int64_t Mp, const LayerWs &w, int r, int mode, float scale) {
    ProjArgs a{};
    a.Mp = (int)Mp;
    a.r64 = w.r64;
    a.r = r;
    a.tiles = pl.tiles;
    a.splits = pl.splits;
    a.ktiles = pl.ktiles;
    a.mode = mode;
    a.scale = scale;
    return a;
}

static FusedArgs fused_args(const qlora_nf4_tensor *W, int64_t M, const LayerWs &w, int r, const uint16_t *lora_src,
                            int64_t lora_ld, uint16_t *out, float *partial, int64_t wdim) {
    FusedArgs fa{};
    fa.N = W->rows;
    fa.K = W->cols;
    fa.KB = (int32_t)(W->cols / 64);
    fa.M = (int32_t)M;
    fa.lora_src = lora_src;
    fa.lora_ld = lora_ld;
    fa.r = r;
    fa.BN = w.fp.BN;
    fa.w_tiles = w.fp.w_tiles;
    fa.m_tiles = w.fp.m_tiles;
    fa.splits = w.fp.splits;
    fa.kt_main = w.fp.kt_main;
    fa.kt_lora = w.fp.kt_lora;
    fa.out = out;
    fa.partial = partial;
    fa.wdim = wdim;
    fa.scale_q = W->scale_codes;
    fa.scale_c2 = W->scale_scales;
    fa.scale_mu = W->scale_offset;
    fa.tab = tables();
    return fa;
}

}  // extern "C"

namespace qlora {

static bool dropout_ok(const qlora_dropout *d) { return d && std::isfinite(d->p) && d->p >= 0.0f && d->p < 1.0f; }

// qlora_linear_fwd, with LoRA dropout on the adapter input when `d` is given
static qlora_status layer_fwd(const qlora_nf4_tensor *W, const uint16_t *X, int64_t M, const uint16_t *A,
                              const uint16_t *B, int32_t r, float alpha, const qlora_dropout *d, uint16_t *Y,
                              uint16_t *U_save, void *ws, size_t ws_bytes, void *stream) {
    qlora_status s = check_layer_args(W, X, M, A, B, r, alpha);
    if (s != QLORA_OK) return s;
    if (!Y) return QLORA_ERR_INVALID_ARG;
    if (!aligned16(Y) || (U_save && !aligned16(U_save))) return QLORA_ERR_MISALIGNED;
    const int64_t N = W->rows, K = W->cols, KB = K / 64;
    const int sms = num_sms_current();
    const LayerWs w = layer_ws(M, N, K, r, false, sms, d != nullptr);
    if (!ws || ws_bytes < w.total || !aligned16(ws)) return QLORA_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *base = static_cast<uint8_t *>(ws);
    float *scalesT = reinterpret_cast<float *>(base + w.off_scales);
    uint16_t *U = reinterpret_cast<uint16_t *>(base + w.off_u);
    float *mainp = reinterpret_cast<float *>(base + w.off_main);
    const float scale = alpha / (float)r;
    // the adapter branch's input: X, or X with the dropout mask applied
    const uint16_t *Xl = d ? reinterpret_cast<const uint16_t *>(base + w.off_xd) : X;

    cudaError_t e;
    if (w.gemv) {
        // one launch: U = bf16(s Xl A^T), Y = X W^T + U B^T; its counters are cleared first
        CUtensorMap mG3, mG2;
        if (!map_codes_gemv(&mG3, &mG2, W->codes, N, K)) return QLORA_ERR_CUDA;
        if (d && (e = launch_dropout_x(X, M * K, d->seed, d->offset, d->p, const_cast<uint16_t *>(Xl), nullptr, sms,
                                       st)) != cudaSuccess)
            return from_cuda(e);
        const GemvWs gw = gemv_ws(N, K, r);
        if ((e = cudaMemsetAsync(reinterpret_cast<uint8_t *>(mainp) + gw.off_counters, 0, gw.counter_bytes, st)) !=
            cudaSuccess)
            return from_cuda(e);
        const int32_t ti = timer_open(st);
        e = launch_gemv(mG3, mG2, W->scale_codes, W->scale_scales, W->scale_offset, X, Xl, (int)M, N, K, A, B, r, scale, Y,
                        U_save, mainp, tables(), sms, st);
        timer_close(ti, st);
        return from_cuda(e);
    }
    CUtensorMap mX_k, mA_k, mCodes, mScales, mX_act, mU_act, mY;
    std::memset(&mScales, 0, sizeof(mScales));
    if (!map_bf16(&mX_k, Xl, K, M, 64, 128) || !map_bf16(&mA_k, A, K, r, 64, w.r64) ||
        !map_codes(&mCodes, W->codes, N, K, false) ||
        (!w.fp.small && !map_scales(&mScales, scalesT, N, KB, false)) ||
        !map_bf16(&mX_act, X, K, M, 64, w.fp.act_rows) || !map_bf16(&mU_act, U, w.r8, M, 64, w.fp.act_rows) ||
        !map_out(&mY, Y, M, N))
        return QLORA_ERR_CUDA;

    Fork fk(st);
    if ((e = fk.fork()) != cudaSuccess) return from_cuda(e);
    // the fused kernel's block scales, alongside the adapter product
    if (!w.fp.small && (e = launch_dq_scales_t(W->scale_codes, W->scale_scales, W->scale_offset, N, (int)KB, scalesT,
                                               fk.side(0))) != cudaSuccess)
        return from_cuda(e);
    if (d && (e = launch_dropout_x(X, M * K, d->seed, d->offset, d->p, const_cast<uint16_t *>(Xl), nullptr, sms, st)) !=
                 cudaSuccess)
        return from_cuda(e);
    // U = bf16(s * X A^T)  [M, r8] (+ U_save [M, r]), X masked under dropout
    ProjArgs pu = proj_args(w.pu, M, w, r, 0, scale);
    pu.out_h = U;
    pu.ld_h = w.r8;
    pu.out_h2 = U_save;
    if ((e = launch_proj(false, false, mX_k, mA_k, pu, st)) != cudaSuccess) return from_cuda(e);
    if ((e = fk.join(0)) != cudaSuccess) return from_cuda(e);
    // Y = X W^T + U B^T
    const FusedArgs fa = fused_args(W, M, w, r, B, r, Y, mainp, N);
    if ((e = timed_fused(false, mCodes, mScales, mX_act, mU_act, mY, fa, w.fp, sms, st)) != cudaSuccess)
        return from_cuda(e);
    return QLORA_OK;
}

// qlora_linear_bwd, with LoRA dropout on the adapter input when `d` is given: the mask is
// regenerated from (seed, offset); dX's base term comes from the fused kernel without the adapter
// k-steps, and the masked adapter term is added by a rank-r update.
static qlora_status layer_bwd(const qlora_nf4_tensor *W, const uint16_t *X, int64_t M, const uint16_t *A,
                              const uint16_t *B, int32_t r, float alpha, const qlora_dropout *d, const uint16_t *dY,
                              const uint16_t *U_saved, uint16_t *dX, float *dA, float *dB, void *ws, size_t ws_bytes,
                              void *stream) {
    qlora_status s = check_layer_args(W, X, M, A, B, r, alpha);
    if (s != QLORA_OK) return s;
    if (!dY || !dX || !dA || !dB) return QLORA_ERR_INVALID_ARG;
    if (!aligned16(dY) || !aligned16(dX) || !aligned16(dA) || !aligned16(dB) || (U_saved && !aligned16(U_saved)))
        return QLORA_ERR_MISALIGNED;
    const int64_t N = W->rows, K = W->cols, KB = K / 64;
    const int sms = num_sms_current();
    const LayerWs w = layer_ws(M, N, K, r, true, sms, d != nullptr);
    if (!ws || ws_bytes < w.total || !aligned16(ws)) return QLORA_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *base = static_cast<uint8_t *>(ws);
    float *scalesT = reinterpret_cast<float *>(base + w.off_scales);
    uint16_t *U = reinterpret_cast<uint16_t *>(base + w.off_u);
    uint16_t *V = reinterpret_cast<uint16_t *>(base + w.off_v);
    uint16_t *Xd = reinterpret_cast<uint16_t *>(base + w.off_xd);
    uint32_t *mask = reinterpret_cast<uint32_t *>(base + w.off_mask);
    const uint16_t *Xl = d ? Xd : X;  // the adapter branch's input
    uint16_t *Bpad = reinterpret_cast<uint16_t *>(base + w.off_bpad);
    float *mainp = reinterpret_cast<float *>(base + w.off_main);
    const float scale = alpha / (float)r;
    const bool r_vec = (r % 8) == 0;
    // U as a TMA-readable [M, ru] tensor: the caller's copy when its rows are 16-byte multiples
    const uint16_t *Uq = (U_saved && r_vec) ? U_saved : U;
    const int64_t ru = (U_saved && r_vec) ? r : w.r8;
    const uint16_t *Bq = r_vec ? B : Bpad;
    const int64_t rb = r_vec ? r : w.r8;

    CUtensorMap mX_k, mA_k, mG_k, mB_mn, mX_mn, mV_mn, mG_mn, mU_mn, mCodes, mScales, mG_act, mV_act, mDX;
    CUtensorMap mV_k, mA_mn, mDX_sw;
    std::memset(&mScales, 0, sizeof(mScales));
    if (!map_bf16(&mX_k, Xl, K, M, 64, 128) || !map_bf16(&mA_k, A, K, r, 64, w.r64) ||
        !map_bf16(&mG_k, dY, N, M, 64, 128) || !map_bf16(&mB_mn, Bq, rb, N, 64, 64) ||
        !map_bf16(&mX_mn, Xl, K, M, 64, 64) || !map_bf16(&mV_mn, V, w.r8, M, 64, 64) ||
        !map_bf16(&mG_mn, dY, N, M, 64, 64) || !map_bf16(&mU_mn, Uq, ru, M, 64, 64) ||
        !map_codes(&mCodes, W->codes, N, K, true) || (!w.fp.small && !map_scales(&mScales, scalesT, N, KB, true)) ||
        !map_bf16(&mG_act, dY, N, M, 64, w.fp.act_rows) || !map_bf16(&mV_act, V, w.r8, M, 64, w.fp.act_rows) ||
        !map_out(&mDX, dX, M, K))
        return QLORA_ERR_CUDA;
    if (d && (!map_bf16(&mV_k, V, w.r8, M, 64, 128) || !map_bf16(&mA_mn, A, K, r, 64, 64) ||
              !map_bf16(&mDX_sw, dX, K, M, 64, 32)))
        return QLORA_ERR_CUDA;

    cudaError_t e;
    Fork fk(st);
    if (d && (e = launch_dropout_x(X, M * K, d->seed, d->offset, d->p, Xd, mask, sms, st)) != cudaSuccess)
        return from_cuda(e);
    if (!r_vec && (e = launch_pad_2d(B, N, r, Bpad, N, w.r8, sms, st)) != cudaSuccess) return from_cuda(e);
    // U: the forward's saved copy, or recomputed
    if (U_saved) {
        if (!r_vec && (e = launch_pad_2d(U_saved, M, r, U, M, w.r8, sms, st)) != cudaSuccess) return from_cuda(e);
    } else {
        ProjArgs pu = proj_args(w.pu, M, w, r, 0, scale);
        pu.out_h = U;
        pu.ld_h = w.r8;
        if ((e = launch_proj(false, false, mX_k, mA_k, pu, st)) != cudaSuccess) return from_cuda(e);
    }
    // from here three independent pieces: the block scales and dB on the side streams, V here
    if ((e = fk.fork()) != cudaSuccess) return from_cuda(e);
    if (!w.fp.small && (e = launch_dq_scales_t(W->scale_codes, W->scale_scales, W->scale_offset, N, (int)KB, scalesT,
                                               fk.side(0))) != cudaSuccess)
        return from_cuda(e);
    // dB = G^T U  (D[n, j] = sum_m G[m, n] U[m, j])
    ProjArgs pb = proj_args(w.pdb, N, w, r, 2, 1.0f);
    pb.out_f = dB;
    if ((e = launch_proj(true, true, mG_mn, mU_mn, pb, fk.side(1))) != cudaSuccess) return from_cuda(e);
    // V = bf16(s * G B)  [M, r8]
    ProjArgs pv = proj_args(w.pv, M, w, r, 0, scale);
    pv.out_h = V;
    pv.ld_h = w.r8;
    if ((e = launch_proj(false, true, mG_k, mB_mn, pv, st)) != cudaSuccess) return from_cuda(e);
    // dX on the high-priority stream once V and the scales are there; dA (which needs only V) here,
    // at the caller's priority: its CTAs take the SMs that the fused kernel's last wave leaves idle
    cudaStream_t hp = fk.priority();
    if ((e = fk.link(st, hp)) != cudaSuccess || (e = fk.link(fk.side(0), hp)) != cudaSuccess) return from_cuda(e);
    // dX = G W^ + V A  (under dropout: G W^, then += mask / (1 - p) * (V A))
    FusedArgs fa = fused_args(W, M, w, r, A, K, dX, mainp, K);
    if (d) fa.kt_lora = 0;
    if ((e = timed_fused(true, mCodes, mScales, mG_act, mV_act, mDX, fa, w.fp, sms, hp)) != cudaSuccess)
        return from_cuda(e);
    if (d && (e = launch_dropout_dx(mV_k, mA_mn, mDX_sw, dX, mask, d->p, M, K, w.r8, sms, hp)) != cudaSuccess)
        return from_cuda(e);
    // dA = V^T X  (D[k, j] = sum_m X[m, k] V[m, j], stored transposed)
    ProjArgs pa = proj_args(w.pda, K, w, r, 1, 1.0f);
    pa.out_f = dA;
    if ((e = launch_proj(true, true, mX_mn, mV_mn, pa, st)) != cudaSuccess) return from_cuda(e);
    if ((e = fk.link(hp, st)) != cudaSuccess || (e = fk.join(1)) != cudaSuccess) return from_cuda(e);
    return QLORA_OK;
}

}  // namespace qlora

extern "C" {

qlora_status qlora_linear_fwd(const qlora_nf4_tensor *W, const uint16_t *X, int64_t M, const uint16_t *A,
                              const uint16_t *B, int32_t r, float alpha, uint16_t *Y, uint16_t *U_save, void *ws,
                              size_t ws_bytes, void *stream) {
    return layer_fwd(W, X, M, A, B, r, alpha, nullptr, Y, U_save, ws, ws_bytes, stream);
}

qlora_status qlora_linear_bwd(const qlora_nf4_tensor *W, const uint16_t *X, int64_t M, const uint16_t *A,
                              const uint16_t *B, int32_t r, float alpha, const uint16_t *dY, const uint16_t *U_saved,
                              uint16_t *dX, float *dA, float *dB, void *ws, size_t ws_bytes, void *stream) {
    return layer_bwd(W, X, M, A, B, r, alpha, nullptr, dY, U_saved, dX, dA, dB, ws, ws_bytes, stream);
}

size_t qlora_fwd_dropout_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t r) {
    if (M < 1 || N < 1 || N % 8 != 0 || K < 64 || K % 64 != 0 || r < 1 || r > 256) return (size_t)-1;
    return layer_ws(M, N, K, r, false, num_sms_current(), true).total;
}

size_t qlora_bwd_dropout_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t r) {
    if (M < 1 || N < 1 || N % 8 != 0 || K < 64 || K % 64 != 0 || r < 1 || r > 256) return (size_t)-1;
    return layer_ws(M, N, K, r, true, num_sms_current(), true).total;
}

qlora_status qlora_linear_fwd_dropout(const qlora_nf4_tensor *W, const uint16_t *X, int64_t M, const uint16_t *A,
                                      const uint16_t *B, int32_t r, float alpha, const qlora_dropout *dropout,
                                      uint16_t *Y, uint16_t *U_save, void *ws, size_t ws_bytes, void *stream) {
    if (!dropout_ok(dropout)) return QLORA_ERR_INVALID_ARG;
    return layer_fwd(W, X, M, A, B, r, alpha, dropout, Y, U_save, ws, ws_bytes, stream);
}

qlora_status qlora_linear_bwd_dropout(const qlora_nf4_tensor *W, const uint16_t *X, int64_t M, const uint16_t *A,
                                      const uint16_t *B, int32_t r, float alpha, const qlora_dropout *dropout,
                                      const uint16_t *dY, const uint16_t *U_saved, uint16_t *dX, float *dA, float *dB,
                                      void *ws, size_t ws_bytes, void *stream) {
    if (!dropout_ok(dropout)) return QLORA_ERR_INVALID_ARG;
    return layer_bwd(W, X, M, A, B, r, alpha, dropout, dY, U_saved, dX, dA, dB, ws, ws_bytes, stream);
}

qlora_status qlora_set_kernel_timer(void **events, int32_t capacity) {
    if (capacity < 0) return QLORA_ERR_INVALID_ARG;
    for (int32_t i = 0; events && i < 2 * capacity; ++i)
        if (!events[i]) return QLORA_ERR_INVALID_ARG;
    g_timer_events = nullptr;
    g_timer_cap = events ? capacity : 0;
    g_timer_n.store(0);
    g_timer_events = events;
    return QLORA_OK;
}

int32_t qlora_kernel_timer_count(void) { return std::min(g_timer_n.load(), g_timer_cap); }

qlora_status qlora_check_device_error(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return QLORA_ERR_CUDA;
    uint32_t word = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&word, g_error_word, sizeof(word)) != cudaSuccess) return QLORA_ERR_CUDA;
    if (word && cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) != cudaSuccess) return QLORA_ERR_CUDA;
    if (word & kErrTimeout) return QLORA_ERR_TIMEOUT;
    if (word & kErrLayout) return QLORA_ERR_CUDA;
    return (word & kErrBounds) ? QLORA_ERR_DEVICE_CHECK : QLORA_OK;
}

qlora_status qlora_test_inject(uint32_t flags) {
#ifdef QLORA_DEVICE_CHECKS
    const uint32_t known = QLORA_INJECT_SKIP_CODES | QLORA_INJECT_BOUNDS;
#else
    const uint32_t known = QLORA_INJECT_SKIP_CODES;
#endif
    if (flags & ~known) return QLORA_ERR_INVALID_ARG;
    return cudaMemcpyToSymbol(g_inject, &flags, sizeof(flags)) == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}

}  // extern "C"
