// gemv.cu -- the forward layer for up to eight tokens (decoding), in one launch.
//
// With M <= 8 a weight is used by at most eight tokens: the call streams the 0.52 bytes per weight
// of packed codes and scale codes once, and everything else is small.  Two things decide the
// speed of such a kernel: how the codes are read from HBM, and the work per decoded weight.
//
// The product.  The block scale is factored out:
//     Y[m, n] = sum_b s'_b * ( sum_{k in b} L[c_nk] x_mk )  +  sum_j U[m, j] B[n, j]
// ("QLoRA -- La base en 4 bits, LoRA encima" (paperclase, lesson 8), "Parte 4 - LoRA encima":
// the layer multiplies NF4[c] * absmax by x in fp32, h = W^ x + (alpha/r) B A x.)
//   - The inner sum runs on warp-level tensor cores (mma.sync m16n8k16, bf16 in, fp32 out): the
//     A operand is the unscaled level table L[c] in bf16, the B operand is x.  A code byte holds
//     two consecutive weights, so one 32-bit load from a 256-entry table of level pairs gives
//     one A-fragment register: one byte permute (which builds the table address from the code
//     byte) and one shared load per two weights.  The table is replicated once per lane so that
//     every lane reads its own bank.
//   - Each 64-weight block gets a fresh accumulator; its four 16-wide MMA steps are scaled by
//     s'_b = fmaf(q_b, fl32(c2_g / 127), mu) (the dequantization's block scale, exactly) in fp32
//     and added to the running sums.  The weights are therefore not rounded to bf16 after the
//     scale, as in nf4_dequantize; the result differs from the product with that W^ by about
//     2^-9 relative per weight, well inside the layer tolerance.
//
// The stream.  The codes are read in stages of 32 weight rows x 1 KB of each row (2048 columns,
// one 3-D TMA box of eight 128-byte units), so that every row segment is one contiguous read:
// 128-byte pieces of many rows fetched microseconds apart ran at a quarter of the HBM bandwidth.
//   - One producer warp per CTA takes the work items from a launch-wide counter, two items ahead
//     (so an SM that gets its data late does less of the work), issues each stage's codes by TMA
//     into one of four stage slots, and rebuilds the stage's block scales
//     s'_b = fmaf(q_b, fl32(c2_g / 127), mu) (the dequantization's arithmetic) from int8 scale codes
//     it loaded a whole stage earlier, into the slot's side area (lane = weight row).
//   - Eight consumer warps each take one 256-column unit (two 16-row MMA tiles) of every stage.
//     A warp loads x of the next stage's unit while it computes the current one, and adds the
//     stages of a work item up in registers.
//   - A work item is one row group and up to four consecutive slabs; at its end each consumer
//     warp hands its sums to the CTA's finisher warp through a ring in the table's free
//     half-rows, and the finisher adds the eight warps' sums (fixed order) into the item's fp32
//     partial.
//   - The adapter's down product U = X A^T comes first: its items (the rows of A, bf16, no decode,
//     one slab each) are the first items of the first CTAs, so U is done early and by many CTAs at
//     once; the term U B^T is added by the stage of each row group's last slab (bf16 B rows as
//     the A operand, loaded at the item's first stage).
//   - The last item of a row group to be counted in (a counter per row group) finishes it: its
//     finisher adds the row group's partials in item order (so the result is deterministic) and
//     writes bf16 Y, or, for the rows of A, publishes bf16(s X A^T).
// Every wait is bounded; the counters must be zero at launch (the host clears them first).

namespace qlora {

static constexpr int kGvCW = 8;                         // consumer warps: one unit of each stage each
static constexpr int kGvProducer = kGvCW;               // warp index of the producer
static constexpr int kGvFinisher = kGvCW + 1;           // warp index of the finisher
static constexpr int kGvThreads = (kGvCW + 2) * 32;
static constexpr int kGvRows = kGemvBoxRows;            // weight rows per stage (two MMA tiles)
static_assert(kGvRows == 32, "a stage is two 16-row MMA tiles per unit");
static constexpr int kGvSub = 256;                      // contraction columns per unit
static constexpr int kGvSlab = kGvCW;                   // units per stage (slab = 2048 columns)
static_assert(kGvSlab == kGemvBoxUnits, "one TMA box per stage");
static constexpr int kGvRun = 4;                        // slabs per work item (of one row group)
static constexpr int kGvStages = 4;
static constexpr int kGvMaxM = 8;
static constexpr int kGvAcc = 8;                        // fp32 sums per lane: 2 tiles x (2 rows x 2 tokens)
static constexpr int kGvRQ = 4;                         // work items' warp sums in flight to the finisher
// Shared memory.  A stage's codes (32 rows x 8 units, 32 KB) sit in a slot of their own; its
// small parts sit in a side area per slot: the fp32 block scales s'_b [32 rows][kGvScaleLd]
// (blocks 0..31 of the slab, padded so that the rows start in different banks), and the
// descriptor {kind, rg, slab, item}, {last of item, next kind, next slab, flags}.
static constexpr uint32_t kGvBoxBytes = kGvRows * 128;           // one unit's codes
static constexpr uint32_t kGvStageBytes = kGvSlab * kGvBoxBytes;  // 32 KB
static constexpr int kGvScaleLd = 36;
static constexpr uint32_t kGvSideS = 0, kGvSideDesc = kGvRows * kGvScaleLd * 4;
static constexpr uint32_t kGvSideBytes = (kGvSideDesc + 32 + 127) & ~127u;
static_assert(kGvSideDesc + 32 <= kGvSideBytes, "side area");
// The level-pair table sits at shared-window address 0x10000, so that one byte permute forms a
// complete address (0x10000 | code byte << 8 | lane << 2).  It uses the first 128 bytes of each
// 256-byte row; the other halves hold the consumer warps' sums on their way to the finisher
// (entry (ring slot, warp, element): one half-row, one word per lane, kGvRQ slots).  Slot 0, the
// side areas and the barriers sit below the table, slots 1 .. kGvStages - 1 above it.
static constexpr uint32_t kGvTable = 0x10000u;
static constexpr uint32_t kGvTableEnd = 0x20000u;
static constexpr uint32_t kGvMaxBase = 8192u;           // largest dynamic shared memory start allowed
static constexpr uint32_t kGvTailBytes = 8 * (2 * kGvStages + 2 * kGvRQ) + 16 * kGvRQ + 16;
static constexpr uint32_t kGvBelow = kGvStageBytes + kGvStages * kGvSideBytes + kGvTailBytes;
static_assert(kGvMaxBase + kGvBelow <= kGvTable, "slot 0, side areas and barriers below the table");
static_assert(kGvRQ * kGvCW * kGvAcc <= 256, "warp sums fit the table's free half-rows");
static constexpr uint32_t kGvDynBytes = kGvTableEnd + (kGvStages - 1) * kGvStageBytes;  // with the start at 0
static_assert(kGvDynBytes <= 227u * 1024u, "shared memory budget");

enum : int { kGvKindWeight = 0, kGvKindAdapter = 1, kGvKindStop = 2 };

struct GemvArgs {
    const int8_t *scale_q;   // [N * KB] int8 block-scale codes
    const float *scale_c2;   // [ng]
    const float *scale_mu;   // [1]
    const uint16_t *X;       // [M, K] input of the base term
    const uint16_t *Xa;      // [M, K] input of the adapter term (X, or X under the dropout mask)
    const uint16_t *A;       // [r, K]
    const uint16_t *B;       // [N, r]
    uint16_t *Y;             // [M, N]
    uint16_t *U_save;        // [M, r] (nullable)
    uint16_t *Ubf;           // [8, r32]: bf16(s X_a A^T), token rows >= M zero
    float *partial;          // [n_items][kGvAcc][32]: fp32 sums of every work item
    uint32_t *counters;      // [RG + 2], zero at launch: items done per row group, adapter row
                             // groups published, work items taken
    int N, K, KB;
    int M, r, r32;
    float s;                 // alpha / r
    int S;                   // units per row: ceil(K / 256)
    int S_whole;             // units of 256 columns that are whole: floor(K / 256)
    int NS;                  // slabs per row: ceil(S / kGvSlab)
    int RU;                  // adapter row groups: r32 / 32
    int RG;                  // RU + ceil(N / 32)
    int NI;                  // work items per row group of W: ceil(NS / kGvRun)
    int n_items;             // RU * NS + (RG - RU) * NI
    float level[16];
};

// The MMAs and the table loads are not volatile: they are pure functions of their operands (the
// table is constant once built), so the compiler may interleave one block's loads with another
// block's MMAs.  The code-word loads stay volatile, ordered after the stage's barrier wait.
__device__ __forceinline__ void mma_bf16_16816(float *d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}
__device__ __forceinline__ float4 lds128f(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void sts128f(uint32_t addr, float a, float b, float c, float d) {
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// 3-D tiled TMA load (coordinates innermost first), completion counted on `bar`.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar, int32_t x, int32_t y,
                                            int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}
// Add `bytes` to the barrier's expected transaction count without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
// Global loads that are issued where they are written (volatile): the prefetches below must not be
// sunk by the compiler to the first use of their results, a stage later.
__device__ __forceinline__ uint4 ldg_pin_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_pin_u32(const void *p) {
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_pin_u16(const void *p) {
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
// Non-blocking test of a barrier phase.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Shared load ordered like the other volatile accesses (the warp sums change from stage to stage).
__device__ __forceinline__ uint32_t lds32v(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
// Level pair of code byte `kByte` of `w`: the table word at 0x10000 | byte << 8 | lane << 2
// (`lanebase` = 0x10000 | lane << 2).
template <int kByte>
__device__ __forceinline__ uint32_t pair_lookup(uint32_t w, uint32_t lanebase) {
    return lds32(prmt(w, lanebase, 0x7604u | (kByte << 4)));
}

// Work items.  The rows of A come first, one slab per item (so that U is done early, by many
// CTAs at once); then each row group of W in items of up to kGvRun consecutive slabs.  An item's
// index is also its partial-sum slot: a row group's items are consecutive, from gv_first_item.
struct GvItem {
    int rg, slab0, slab1;
};
__device__ __forceinline__ GvItem gv_item(const GemvArgs &a, int item) {
    GvItem it;
    const int nu = a.RU * a.NS;
    if (item < nu) {
        it.rg = item / a.NS;
        it.slab0 = item - it.rg * a.NS;
        it.slab1 = it.slab0 + 1;
    } else {
        const int wi = item - nu;
        const int part = wi % a.NI;
        it.rg = a.RU + wi / a.NI;
        it.slab0 = part * kGvRun;
        it.slab1 = it.slab0 + kGvRun < a.NS ? it.slab0 + kGvRun : a.NS;
    }
    return it;
}
__device__ __forceinline__ int gv_items_of(const GemvArgs &a, int rg) { return rg < a.RU ? a.NS : a.NI; }
__device__ __forceinline__ int gv_first_item(const GemvArgs &a, int rg) {
    return rg < a.RU ? rg * a.NS : a.RU * a.NS + (rg - a.RU) * a.NI;
}

__global__ void __launch_bounds__(kGvThreads, 1)
    nf4_gemv_kernel(const __grid_constant__ CUtensorMap map3, const __grid_constant__ CUtensorMap map2,
                    const __grid_constant__ GemvArgs a) {
    extern __shared__ __align__(1024) uint8_t gv_smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;

    // shared-memory layout (the table must occupy [0x10000, 0x20000) of the shared window)
    const uint32_t base = smem_u32(gv_smem);
    uint32_t dyn_bytes;
    asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn_bytes));
    const uint32_t lo_start = (base + 1023u) & ~1023u;
    if (base > kGvMaxBase || kGvDynBytes > base + dyn_bytes) {
        if (threadIdx.x == 0) atomicOr(&g_error_word, kErrLayout);
        return;
    }
    uint8_t *sm0 = gv_smem - base;  // generic pointer of shared-window address 0
    const uint32_t side_base = lo_start + kGvStageBytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(sm0 + side_base + kGvStages * kGvSideBytes);
    uint64_t *empty = full + kGvStages;
    uint64_t *rfull = empty + kGvStages;  // an item's eight warp sums are in their ring slot
    uint64_t *rempty = rfull + kGvRQ;     // the finisher has read them
    int4 *rdesc = reinterpret_cast<int4 *>(rempty + kGvRQ);  // {kind, rg, item} of the slot's item
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(rdesc + kGvRQ);
    // word of the warp sums: slot, warp, element -> half-row, lane -> word
    auto red_addr = [&](int rs, int ww, int e) -> uint32_t {
        return kGvTable + (uint32_t)((rs * kGvCW + ww) * kGvAcc + e) * 256u + 128u + ((uint32_t)lane << 2);
    };
    auto stage_addr = [&](int slot) -> uint32_t {
        return slot == 0 ? lo_start : kGvTableEnd + (uint32_t)(slot - 1) * kGvStageBytes;
    };
    auto side_addr = [&](int slot) -> uint32_t { return side_base + (uint32_t)slot * kGvSideBytes; };

    // level-pair table: word (v << 6) + l, for every lane l, holds bf16(L[v >> 4]) | bf16(L[v & 15]) << 16
    for (int idx = threadIdx.x; idx < 256 * 32; idx += kGvThreads) {
        const int v = idx >> 5, l = idx & 31;
        const __nv_bfloat16 lo = __float2bfloat16_rn(a.level[v >> 4]);
        const __nv_bfloat16 hi = __float2bfloat16_rn(a.level[v & 15]);
        const uint32_t w = (uint32_t)*reinterpret_cast<const uint16_t *>(&lo) |
                           ((uint32_t)*reinterpret_cast<const uint16_t *>(&hi) << 16);
        sts32(kGvTable + ((uint32_t)v << 8) + ((uint32_t)l << 2), w);
    }
    if (threadIdx.x < kGvStages) {
        mbar_init(&full[threadIdx.x], 1);
        mbar_init(&empty[threadIdx.x], kGvCW);
    }
    if (threadIdx.x < kGvRQ) {
        mbar_init(&rfull[threadIdx.x], kGvCW);
        mbar_init(&rempty[threadIdx.x], 1);
    }
    if (threadIdx.x == 0) {
        *abort_flag = 0u;
        tma_prefetch_desc(&map3);
        tma_prefetch_desc(&map2);
    }
    fence_mbar_init();
    __syncthreads();

    const float mu = __ldg(a.scale_mu);
    const int S = a.S, NS = a.NS;

    if (warp == kGvProducer) {
        // ---------------------------------------------------------------- producer warp --------
        // The stages in the order of the work items (taken two ahead): wait until the stage's
        // slot is free, describe it (with the stage after it, whose x the consumers load ahead),
        // issue its codes (one 3-D TMA box: 32 rows x 8 units, or a 2-D box per unit), store its
        // rebuilt block scales s'_b in the slot's side area (lane = weight row) and release it.
        // Then load the scale codes of the stage after the next one into registers.
        // This CTA's items: first its share of the adapter items (items blockIdx.x, + gridDim.x,
        // ..., so that U is computed at once by many CTAs), then items of W from the counter.
        const int nu = a.RU * a.NS;
        int u_next = blockIdx.x;
        auto fetch = [&]() -> int {  // the next item (an item of W: valid in lane 0 only)
            if (u_next < nu) {
                const int v = u_next;
                u_next += gridDim.x;
                return v;
            }
            int v = 0;
            if (lane == 0) v = nu + (int)atomicAdd(a.counters + a.RG + 1, 1u);
            return v;
        };
        int item_next = fetch();
        item_next = __shfl_sync(0xffffffffu, item_next, 0);
        int item_nn = item_next < a.n_items ? fetch() : a.n_items;
        // A cursor over the stages in item order: the item (n_items at the end), its row group,
        // the stage's slab, and the item's first and end slabs.  The producer keeps two: the
        // stage it produces and the one after it, whose scale codes are loaded a whole stage
        // before they are needed (their latency is not in any stage's path).
        struct Cur {
            int item, rg, slab, slab0, slab1;
        };
        auto advance = [&](Cur &cu) {
            if (cu.item >= 0 && cu.item < a.n_items && ++cu.slab < cu.slab1) return;
            cu.item = item_next < a.n_items ? item_next : a.n_items;
            if (cu.item >= a.n_items) return;
            const GvItem it = gv_item(a, cu.item);
            cu.rg = it.rg;
            cu.slab = cu.slab0 = it.slab0;
            cu.slab1 = it.slab1;
            item_next = __shfl_sync(0xffffffffu, item_nn, 0);
            if (item_next < a.n_items) item_nn = fetch();
        };
        // scale codes and group constants of this lane's row of a weight stage
        struct Sc {
            uint4 q0, q1;
            float c0, c1;
        };
        auto load_scales = [&](int rg, int sl, Sc &sc) {
            sc.q0 = sc.q1 = make_uint4(0u, 0u, 0u, 0u);
            sc.c0 = sc.c1 = 0.0f;
            if (rg < a.RU) return;
            const int n = (rg - a.RU) * kGvRows + lane;
            if (n >= a.N) return;
            const int kb0 = sl * 32;
            const int64_t b0 = (int64_t)n * a.KB + kb0;
            const int nb = a.KB - kb0 < 32 ? a.KB - kb0 : 32;
            if (nb == 32 && (b0 & 15) == 0) {
                sc.q0 = ldg_pin_v4(a.scale_q + b0);
                sc.q1 = ldg_pin_v4(a.scale_q + b0 + 16);
            } else {
                uint32_t wv[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                for (int jb = 0; jb < nb; ++jb)
                    wv[jb >> 2] |= (uint32_t)(uint8_t)__ldg(a.scale_q + b0 + jb) << (8 * (jb & 3));
                sc.q0 = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                sc.q1 = make_uint4(wv[4], wv[5], wv[6], wv[7]);
            }
            sc.c0 = __uint_as_float(ldg_pin_u32(a.scale_c2 + (b0 >> 8)));
            sc.c1 = __uint_as_float(ldg_pin_u32(a.scale_c2 + ((b0 + nb - 1) >> 8)));
        };
        Cur ca{-1, 0, 0, 0, 0};
        advance(ca);
        Cur cb = ca;
        advance(cb);
        Sc sc_a, sc_b;
        if (ca.item < a.n_items) load_scales(ca.rg, ca.slab, sc_a);
        if (cb.item < a.n_items) load_scales(cb.rg, cb.slab, sc_b);
        int t = 0;
        bool ok = true;
        for (;; ++t) {
            const int slot = t % kGvStages;
            uint32_t okw = 1;
            if (lane == 0 && t >= kGvStages)
                okw = mbar_wait(&empty[slot], (uint32_t)(((t / kGvStages) - 1) & 1), abort_flag) ? 1u : 0u;
            okw = __shfl_sync(0xffffffffu, okw, 0);
            __syncwarp();
            if (!okw) {
                ok = false;
                break;
            }
            const uint32_t sb = stage_addr(slot), sd = side_addr(slot);
            int4 *desc = reinterpret_cast<int4 *>(sm0 + sd + kGvSideDesc);
            if (ca.item >= a.n_items) {  // the end: a stop stage
                if (lane == 0) {
                    desc[0] = make_int4(kGvKindStop, 0, 0, 0);
                    mbar_arrive(&full[slot]);
                }
                break;
            }
            const int rg = ca.rg, slab = ca.slab;
            const int kind = rg < a.RU ? kGvKindAdapter : kGvKindWeight;
            const bool last_of_item = slab + 1 == ca.slab1;
            // the stage after this one (its x is loaded ahead by the consumers)
            int nxt_kind = kGvKindStop, nxt_slab = 0;
            if (cb.item < a.n_items) {
                nxt_kind = cb.rg < a.RU ? kGvKindAdapter : kGvKindWeight;
                nxt_slab = cb.slab;
            }
            if (lane == 0) {
                desc[0] = make_int4(kind, rg, slab, ca.item);
                // flags: bit 0 the item's first stage, bit 1 the item holds the row group's last slab
                const int flags = (slab == ca.slab0 ? 1 : 0) | (ca.slab1 == NS ? 2 : 0);
                desc[1] = make_int4(last_of_item ? 1 : 0, nxt_kind, nxt_slab, flags);
            }
            const Sc &sc_cur = sc_a;
            if (kind == kGvKindWeight) {
                // a slab of eight whole units: one 3-D box; otherwise one 2-D box per unit (the
                // 2-D map checks the columns against K / 2, the 3-D map covers whole units only)
                const int units = S - slab * kGvSlab < kGvSlab ? S - slab * kGvSlab : kGvSlab;
                const bool whole = (slab + 1) * kGvSlab <= a.S_whole;
                if (lane == 0) {
                    mbar_expect_tx(&full[slot], (uint32_t)units * kGvBoxBytes);
                    if (whole) tma_load_3d(sm0 + sb, &map3, &full[slot], 0, (rg - a.RU) * kGvRows, slab * kGvSlab);
                }
                __syncwarp();
                if (!whole && lane < units)
                    tma_load_2d(sm0 + sb + (uint32_t)lane * kGvBoxBytes, &map2, &full[slot],
                                (slab * kGvSlab + lane) * 128, (rg - a.RU) * kGvRows);
                const int n = (rg - a.RU) * kGvRows + lane;
                const int kb0 = slab * 32;
                const int b0 = n * a.KB + kb0;
                const int jsplit = 256 - (b0 & 255);
                const int jvalid = n < a.N ? (a.KB - kb0 < 32 ? a.KB - kb0 : 32) : 0;
                const float k0 = __fdiv_rn(sc_cur.c0, 127.0f);
                const uint32_t qv[8] = {sc_cur.q0.x, sc_cur.q0.y, sc_cur.q0.z, sc_cur.q0.w,
                                        sc_cur.q1.x, sc_cur.q1.y, sc_cur.q1.z, sc_cur.q1.w};
                const uint32_t srow = sd + kGvSideS + (uint32_t)lane * (kGvScaleLd * 4);
                // s'_b = fmaf(q, k, mu), the int8 code as an exact float (the byte q + 128 spliced
                // into 2^23's mantissa, minus 2^23 + 128)
                if (jvalid == 32 && jsplit >= 32) {
                    // the row's 32 blocks are all in W and in one group: two at a time, with the
                    // packed two-lane fp32 instructions (the same IEEE operations)
                    const uint64_t kk = f2pack(__float_as_uint(k0), __float_as_uint(k0));
                    const uint64_t mm = f2pack(__float_as_uint(mu), __float_as_uint(mu));
                    const uint64_t off = 0x4B0000804B000080ull;  // (2^23 + 128, 2^23 + 128)
#pragma unroll
                    for (int w4 = 0; w4 < 8; ++w4) {
                        const uint32_t qw = qv[w4] ^ 0x80808080u;
                        uint64_t p0 = f2pack(prmt(qw, 0x4B000000u, 0x7440u), prmt(qw, 0x4B000000u, 0x7441u));
                        uint64_t p1 = f2pack(prmt(qw, 0x4B000000u, 0x7442u), prmt(qw, 0x4B000000u, 0x7443u));
                        asm("sub.rn.f32x2 %0, %0, %1;" : "+l"(p0) : "l"(off));
                        asm("sub.rn.f32x2 %0, %0, %1;" : "+l"(p1) : "l"(off));
                        asm("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(p0) : "l"(kk), "l"(mm));
                        asm("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(p1) : "l"(kk), "l"(mm));
                        uint32_t v0, v1, v2, v3;
                        f2unpack(p0, v0, v1);
                        f2unpack(p1, v2, v3);
                        sts128f(srow + 16u * w4, __uint_as_float(v0), __uint_as_float(v1), __uint_as_float(v2),
                                __uint_as_float(v3));
                    }
                } else {
                    // blocks jb < jsplit use the row's first group, the rest the next one; blocks
                    // past KB and rows past N get 0
                    const float k1 = __fdiv_rn(sc_cur.c1, 127.0f);
#pragma unroll
                    for (int w4 = 0; w4 < 8; ++w4) {
                        const uint32_t qw = qv[w4] ^ 0x80808080u;
                        float v[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int jb = 4 * w4 + e;
                            const float qf = __fsub_rn(__uint_as_float(prmt(qw, 0x4B000000u, 0x7440u + (uint32_t)e)),
                                                       8388736.0f);  // 2^23 + 128
                            v[e] = jb < jvalid ? __fmaf_rn(qf, jb < jsplit ? k0 : k1, mu) : 0.0f;
                        }
                        sts128f(srow + 16u * w4, v[0], v[1], v[2], v[3]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[slot]);
            // on to the next stage; the scale codes of the one after it into registers
            ca = cb;
            sc_a = sc_b;
            if (cb.item < a.n_items) {
                advance(cb);
                if (cb.item < a.n_items) load_scales(cb.rg, cb.slab, sc_b);
            }
        }
        if (!ok && lane == 0) {
            // on a timeout, let the copies already issued land (bounded) before the CTA can exit
            for (int u = t - kGvStages + 1 > 0 ? t - kGvStages + 1 : 0; u < t; ++u) {
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&full[u % kGvStages], (uint32_t)((u / kGvStages) & 1)) &&
                       globaltimer_ns() - t0 < kWaitTimeoutNs) {
                }
            }
        }
        return;
    }

    if (warp == kGvFinisher) {
        // ---------------------------------------------------------------- finisher warp --------
        // Takes the consumer warps' sums of every work item (as many items as are ready at once)
        // and adds them in warp order.  A row group of one item is finished at once; otherwise
        // the item's sums are stored as its partial, counted in (one fence per batch, the
        // counter's result looked at one batch later, so that its round trip overlaps the next
        // batch), and the last item of a row group to arrive finishes it: the partials added in
        // item order.  Finishing writes bf16 Y for weight rows, or publishes U = bf16(s X A^T) for
        // the U B^T terms for adapter rows.
        const int gr = 2 * (g & 3) + (g >> 2);
        auto finish_vals = [&](int rg, const float *v) {
#pragma unroll
            for (int e = 0; e < kGvAcc; ++e) {
                const int row = 16 * (e >> 2) + gr + ((e & 2) ? 8 : 0);
                const int m = 2 * c + (e & 1);
                if (rg < a.RU) {
                    const int jj = rg * kGvRows + row;
                    const __nv_bfloat16 hh = __float2bfloat16_rn(__fmul_rn(a.s, v[e]));
                    const uint16_t hb = *reinterpret_cast<const uint16_t *>(&hh);
                    if (QLORA_IN_BOUNDS(m < kGvMaxM && jj < a.r32)) a.Ubf[m * a.r32 + jj] = hb;
                    if (a.U_save && m < a.M && jj < a.r) a.U_save[(int64_t)m * a.r + jj] = hb;
                } else {
                    const int nn = (rg - a.RU) * kGvRows + row;
                    if (m < a.M && nn < a.N) {
                        const __nv_bfloat16 hh = __float2bfloat16_rn(v[e]);
                        if (QLORA_IN_BOUNDS((int64_t)m * a.N + nn < (int64_t)a.M * a.N))
                            a.Y[(int64_t)m * a.N + nn] = *reinterpret_cast<const uint16_t *>(&hh);
                    }
                }
            }
            if (rg < a.RU) {
                fence_acq_rel_gpu();
                __syncwarp();
                if (lane == 0) atomicAdd(a.counters + a.RG, 1u);
            }
        };
        auto finish_partials = [&](int rg) {
            float v[kGvAcc];
#pragma unroll
            for (int e = 0; e < kGvAcc; ++e) v[e] = 0.0f;
            const float *p = a.partial + (int64_t)gv_first_item(a, rg) * (kGvAcc * 32) + lane;
            const int ni = gv_items_of(a, rg);
            int j = 0;
            for (; j + 4 <= ni; j += 4) {  // four items' loads in flight, added in item order
                float t4[4][kGvAcc];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                    for (int e = 0; e < kGvAcc; ++e) t4[jj][e] = __ldcg(p + (j + jj) * (kGvAcc * 32) + 32 * e);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                    for (int e = 0; e < kGvAcc; ++e) v[e] = __fadd_rn(v[e], t4[jj][e]);
            }
            for (; j < ni; ++j)
#pragma unroll
                for (int e = 0; e < kGvAcc; ++e) v[e] = __fadd_rn(v[e], __ldcg(p + j * (kGvAcc * 32) + 32 * e));
            finish_vals(rg, v);
        };
        // finish the row groups whose count (taken in the previous batch) came back as the last
        auto finish_counted = [&](int cnt_rg, uint32_t cnt_old) {
            uint32_t lastmask =
                __ballot_sync(0xffffffffu, cnt_rg >= 0 && cnt_old == (uint32_t)(gv_items_of(a, cnt_rg) - 1));
            if (lastmask) fence_acq_rel_gpu();
            while (lastmask) {
                const int src = __ffs(lastmask) - 1;
                lastmask &= lastmask - 1;
                finish_partials(__shfl_sync(0xffffffffu, cnt_rg, src));
            }
        };
        int cnt_rg = -1;       // lane i: the row group counted for entry i of the previous batch
        uint32_t cnt_old = 0;  // and the counter's value before that increment
        bool stop = false;
        for (int h = 0; !stop;) {
            // before blocking for more work, resolve the pending counts (one of them may complete
            // U, which the consumers may be waiting for)
            uint32_t ready = 0;
            if (lane == 0) ready = mbar_test_wait(&rfull[h % kGvRQ], (uint32_t)((h / kGvRQ) & 1)) ? 1u : 0u;
            if (!__shfl_sync(0xffffffffu, ready, 0)) {
                finish_counted(cnt_rg, cnt_old);
                cnt_rg = -1;
            }
            uint32_t okw = 1;
            if (lane == 0) okw = mbar_wait(&rfull[h % kGvRQ], (uint32_t)((h / kGvRQ) & 1), abort_flag) ? 1u : 0u;
            okw = __shfl_sync(0xffffffffu, okw, 0);
            __syncwarp();
            if (!okw) return;
            int n = 1;
            if (lane == 0)
                while (n < kGvRQ && mbar_test_wait(&rfull[(h + n) % kGvRQ], (uint32_t)(((h + n) / kGvRQ) & 1))) ++n;
            n = __shfl_sync(0xffffffffu, n, 0);
            int my_rg = -1;  // lane i < n: the row group of entry h + i, when it is to be counted
            for (int i = 0; i < n; ++i) {
                const int rs = (h + i) % kGvRQ;
                const int4 d = rdesc[rs];
                if (d.x == kGvKindStop) {
                    stop = true;
                    n = i + 1;
                    break;
                }
                float v[kGvAcc];
#pragma unroll
                for (int e = 0; e < kGvAcc; ++e) {
                    float acc = 0.0f;
#pragma unroll
                    for (int ww = 0; ww < kGvCW; ++ww) acc = __fadd_rn(acc, __uint_as_float(lds32v(red_addr(rs, ww, e))));
                    v[e] = acc;
                }
                if (gv_items_of(a, d.y) == 1) {
                    finish_vals(d.y, v);
                } else {
                    float *pp = a.partial + (int64_t)d.z * (kGvAcc * 32) + lane;
                    if (QLORA_IN_BOUNDS(d.z >= 0 && d.z < a.n_items))
#pragma unroll
                        for (int e = 0; e < kGvAcc; ++e) __stcg(pp + 32 * e, v[e]);
                    if (lane == i) my_rg = d.y;
                }
            }
            __syncwarp();
            if (lane == 0)
                for (int i = 0; i < n; ++i) mbar_arrive(&rempty[(h + i) % kGvRQ]);
            h += n;
            {
                // the previous batch's counts are back: finish what they completed
                finish_counted(cnt_rg, cnt_old);
                cnt_rg = -1;
                // this batch's partials are stored: count them in (one fence for the batch)
                if (__any_sync(0xffffffffu, my_rg >= 0)) fence_acq_rel_gpu();
                cnt_rg = my_rg;
                cnt_old = my_rg >= 0 ? atomicAdd(a.counters + my_rg, 1u) : 0u;
            }
        }
        finish_counted(cnt_rg, cnt_old);
        return;
    }

    // -------------------------------------------------------------------- consumer warps ---------
    const int w = warp;
    const uint32_t lanebase = kGvTable | ((uint32_t)lane << 2);
    // MMA row g (and g + 8) of a tile is row gr (and gr + 8) of its 16 weight rows: with this
    // order the lanes of each half-warp read distinct bank pairs of the swizzled code rows
    const int gr = 2 * (g & 3) + (g >> 2);
    float acc[kGvAcc];
#pragma unroll
    for (int e = 0; e < kGvAcc; ++e) acc[e] = 0.0f;
    // x of token g over the lane's 16 columns of each block of the warp's unit of a stage
    auto load_x = [&](int kind, int sl, uint32_t (&xf)[4][8]) {
        const uint16_t *Xs = kind == kGvKindAdapter ? a.Xa : a.X;
        const int unit = sl * kGvSlab + w;
#pragma unroll
        for (int jb = 0; jb < 4; ++jb) {
            const int k = unit * kGvSub + 64 * jb + 16 * c;
            if (kind != kGvKindStop && g < a.M && k < a.K) {
                const uint4 *px = reinterpret_cast<const uint4 *>(Xs + (int64_t)g * a.K + k);
                const uint4 v0 = ldg_pin_v4(px), v1 = ldg_pin_v4(px + 1);
                xf[jb][0] = v0.x; xf[jb][1] = v0.y; xf[jb][2] = v0.z; xf[jb][3] = v0.w;
                xf[jb][4] = v1.x; xf[jb][5] = v1.y; xf[jb][6] = v1.z; xf[jb][7] = v1.w;
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) xf[jb][i] = 0u;
            }
        }
    };
    bool u_ready = false;
    int h_items = 0;  // work items handed to the finisher
    uint32_t bfr[2][2][4] = {};  // B fragments of rank chunks w, w + 8 (two 16-row tiles)
    uint32_t ufr[2][2] = {};     // U fragments of those chunks (token g)
    // B's rank pairs are 32-bit words when r is even (then every pair starts at an even element)
    const bool b_pairs = (a.r & 1) == 0;
    // one stage: xf holds its x (loaded during the previous stage), the next stage's x goes to xn;
    // false at the end of the work (or when a wait ran out).
    auto stage = [&](int t, uint32_t (&xf)[4][8], uint32_t (&xn)[4][8]) -> bool {
        const int slot = t % kGvStages;
        uint32_t okw = 1;
        if (lane == 0) okw = mbar_wait(&full[slot], (uint32_t)((t / kGvStages) & 1), abort_flag) ? 1u : 0u;
        okw = __shfl_sync(0xffffffffu, okw, 0);
        __syncwarp();
        if (!okw) return false;
        const uint32_t sb = stage_addr(slot), sd = side_addr(slot);
        const int4 desc = *reinterpret_cast<const int4 *>(sm0 + sd + kGvSideDesc);
        if (desc.x == kGvKindStop) return false;
        const int4 desc1 = *reinterpret_cast<const int4 *>(sm0 + sd + kGvSideDesc + 16);
        const int kind = desc.x, rg = desc.y, slab = desc.z, item = desc.w;
        const bool last_of_item = desc1.x != 0;
        if (t == 0) load_x(kind, slab, xf);
        // the next stage's x, in flight while this stage is computed
        load_x(desc1.y, desc1.z, xn);
        // rows of B for the U B^T term, in flight from the first stage of the item that ends the
        // row group (lane rows as the weight rows: n0 + 16 tt (+ 8); rank pairs 16 jc + 2c (+ 8))
        if (kind == kGvKindWeight && (desc1.w & 3) == 3) {
            const int n0 = (rg - a.RU) * kGvRows + gr;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int jc = w + q * kGvCW;
#pragma unroll
                for (int tt = 0; tt < 2; ++tt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int n = n0 + 16 * tt + ((i & 1) ? 8 : 0);
                        const int j = jc * 16 + 2 * c + (i >= 2 ? 8 : 0);
                        uint32_t v = 0;
                        if (n < a.N && j < a.r) {
                            const uint16_t *row = a.B + (int64_t)n * a.r;
                            if (b_pairs)
                                v = ldg_pin_u32(row + j);
                            else
                                v = ldg_pin_u16(row + j) | (j + 1 < a.r ? ldg_pin_u16(row + j + 1) << 16 : 0u);
                        }
                        bfr[q][tt][i] = v;
                    }
            }
        }
        const int unit = slab * kGvSlab + w;
        if (unit < S) {
            if (kind == kGvKindAdapter) {
                // rows of A (bf16), no scale: lane rows j = 32 rg + 16 tt + gr (+ 8)
#pragma unroll
                for (int tt = 0; tt < 2; ++tt) {
                    const int j0 = rg * kGvRows + 16 * tt + gr, j1 = j0 + 8;
#pragma unroll
                    for (int jb = 0; jb < 4; ++jb) {
                        const int k = unit * kGvSub + 64 * jb + 16 * c;
                        uint32_t w0[8], w1[8];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int jr = e ? j1 : j0;
                            uint32_t *wv = e ? w1 : w0;
                            if (jr < a.r && k < a.K) {
                                const uint4 *p = reinterpret_cast<const uint4 *>(a.A + (int64_t)jr * a.K + k);
                                const uint4 v0 = __ldg(p), v1 = __ldg(p + 1);
                                wv[0] = v0.x; wv[1] = v0.y; wv[2] = v0.z; wv[3] = v0.w;
                                wv[4] = v1.x; wv[5] = v1.y; wv[6] = v1.z; wv[7] = v1.w;
                            } else {
#pragma unroll
                                for (int i = 0; i < 8; ++i) wv[i] = 0u;
                            }
                        }
#pragma unroll
                        for (int st = 0; st < 4; ++st)
                            mma_bf16_16816(acc + 4 * tt, w0[2 * st], w1[2 * st], w0[2 * st + 1], w1[2 * st + 1],
                                           xf[jb][2 * st], xf[jb][2 * st + 1]);
                    }
                }
            } else {
                // the warp's unit: its codes are unit w of the stage
                const uint32_t box = sb + (uint32_t)w * kGvBoxBytes;
                uint2 cw[4][4];
#pragma unroll
                for (int jb = 0; jb < 4; ++jb) {
                    const uint32_t off = (uint32_t)((((2 * jb + (c >> 1)) ^ gr) << 4) + ((c & 1) << 3));
                    const uint32_t r0 = box + (uint32_t)gr * 128u + off;
#pragma unroll
                    for (int i = 0; i < 4; ++i) cw[jb][i] = lds64(r0 + (uint32_t)(8 * i) * 128u);
                }
                // s'_b of rows gr + 8 i, blocks 4 w .. 4 w + 3
                float sc[4][4];
                const uint32_t srow = sd + kGvSideS + (uint32_t)gr * (kGvScaleLd * 4) + 16u * w;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float4 f = lds128f(srow + (uint32_t)(8 * i) * (kGvScaleLd * 4));
                    sc[i][0] = f.x;
                    sc[i][1] = f.y;
                    sc[i][2] = f.z;
                    sc[i][3] = f.w;
                }
#pragma unroll
                for (int jb = 0; jb < 4; ++jb) {
#pragma unroll
                    for (int tt = 0; tt < 2; ++tt) {
                        const uint2 cw0 = cw[jb][2 * tt], cw1 = cw[jb][2 * tt + 1];
                        float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                        mma_bf16_16816(d, pair_lookup<0>(cw0.x, lanebase), pair_lookup<0>(cw1.x, lanebase),
                                       pair_lookup<1>(cw0.x, lanebase), pair_lookup<1>(cw1.x, lanebase), xf[jb][0],
                                       xf[jb][1]);
                        mma_bf16_16816(d, pair_lookup<2>(cw0.x, lanebase), pair_lookup<2>(cw1.x, lanebase),
                                       pair_lookup<3>(cw0.x, lanebase), pair_lookup<3>(cw1.x, lanebase), xf[jb][2],
                                       xf[jb][3]);
                        mma_bf16_16816(d, pair_lookup<0>(cw0.y, lanebase), pair_lookup<0>(cw1.y, lanebase),
                                       pair_lookup<1>(cw0.y, lanebase), pair_lookup<1>(cw1.y, lanebase), xf[jb][4],
                                       xf[jb][5]);
                        mma_bf16_16816(d, pair_lookup<2>(cw0.y, lanebase), pair_lookup<2>(cw1.y, lanebase),
                                       pair_lookup<3>(cw0.y, lanebase), pair_lookup<3>(cw1.y, lanebase), xf[jb][6],
                                       xf[jb][7]);
                        acc[4 * tt + 0] = __fmaf_rn(sc[2 * tt][jb], d[0], acc[4 * tt + 0]);
                        acc[4 * tt + 1] = __fmaf_rn(sc[2 * tt][jb], d[1], acc[4 * tt + 1]);
                        acc[4 * tt + 2] = __fmaf_rn(sc[2 * tt + 1][jb], d[2], acc[4 * tt + 2]);
                        acc[4 * tt + 3] = __fmaf_rn(sc[2 * tt + 1][jb], d[3], acc[4 * tt + 3]);
                    }
                }
            }
        }
        // this warp is done with the stage's shared memory (every value read above has been used)
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);

        // U B^T, added by the stage of each weight row group's last slab: warp w takes the
        // 16-wide rank chunks w and w + 8 (A operand: bf16 rows of B, loaded at the item's first
        // stage; B operand: U, loaded once it is published)
        if (kind == kGvKindWeight && slab == NS - 1 && w * 16 < a.r32) {
            if (!u_ready) {
                uint32_t okr = 1;
                if (lane == 0 && ld_acquire_u32(a.counters + a.RG) < (uint32_t)a.RU) {
                    const uint64_t t0 = globaltimer_ns();
                    while (ld_acquire_u32(a.counters + a.RG) < (uint32_t)a.RU) {
                        if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
                            atomicOr(&g_error_word, kErrTimeout);
                            okr = 0;
                            break;
                        }
                        __nanosleep(256);
                    }
                }
                okr = __shfl_sync(0xffffffffu, okr, 0);
                __syncwarp();
                fence_acq_rel_gpu();
                u_ready = okr != 0;
                if (u_ready) {
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const int jc = w + q * kGvCW;
                        if (jc * 16 < a.r32) {
                            const uint32_t *ub = reinterpret_cast<const uint32_t *>(a.Ubf + g * a.r32 + jc * 16 + 2 * c);
                            ufr[q][0] = __ldcg(ub);
                            ufr[q][1] = __ldcg(ub + 4);
                        }
                    }
                }
            }
            if (u_ready) {
#pragma unroll
                for (int q = 0; q < 2; ++q)
                    if ((w + q * kGvCW) * 16 < a.r32)
#pragma unroll
                        for (int tt = 0; tt < 2; ++tt)
                            mma_bf16_16816(acc + 4 * tt, bfr[q][tt][0], bfr[q][tt][1], bfr[q][tt][2], bfr[q][tt][3],
                                           ufr[q][0], ufr[q][1]);
            }
        }

        // at the end of a work item, hand this warp's sums to the finisher through ring slot
        // (item count) % kGvRQ (bounded wait until the finisher has read that slot's previous item)
        if (last_of_item) {
            const int hi = h_items++;
            const int rs = hi % kGvRQ;
            uint32_t okr = 1;
            if (lane == 0 && hi >= kGvRQ)
                okr = mbar_wait(&rempty[rs], (uint32_t)(((hi / kGvRQ) - 1) & 1), abort_flag) ? 1u : 0u;
            okr = __shfl_sync(0xffffffffu, okr, 0);
            __syncwarp();
            if (!okr) return false;
#pragma unroll
            for (int e = 0; e < kGvAcc; ++e) {
                sts32(red_addr(rs, w, e), __float_as_uint(acc[e]));
                acc[e] = 0.0f;
            }
            if (w == 0 && lane == 0) rdesc[rs] = make_int4(kind, rg, item, 0);
            __syncwarp();
            if (lane == 0) mbar_arrive(&rfull[rs]);
        }
            return true;
    };
    uint32_t xa[4][8], xb[4][8];
    for (int t = 0;; ++t) {
        if (!stage(t, xa, xb)) break;
        // the next stage's x becomes the current one (a register copy: one copy of the stage body
        // keeps the code small enough for the instruction cache, which two alternating ones did not)
#pragma unroll
        for (int jb = 0; jb < 4; ++jb)
#pragma unroll
            for (int i = 0; i < 8; ++i) xa[jb][i] = xb[jb][i];
    }
    // pass the end on to the finisher (bounded wait for the ring slot)
    {
        const int hi = h_items;
        const int rs = hi % kGvRQ;
        uint32_t okr = 1;
        if (lane == 0 && hi >= kGvRQ) okr = mbar_wait(&rempty[rs], (uint32_t)(((hi / kGvRQ) - 1) & 1), abort_flag) ? 1u : 0u;
        okr = __shfl_sync(0xffffffffu, okr, 0);
        __syncwarp();
        if (okr && lane == 0) {
            if (w == 0) rdesc[rs] = make_int4(kGvKindStop, 0, 0, 0);
            mbar_arrive(&rfull[rs]);
        }
    }
}

// Workspace of the small-M forward: U (bf16, [8][r32]), the fp32 sums of every work item
// ([RU * NS + (RG - RU) * NI][kGvAcc][32]) and the counters ([RG + 2] u32, cleared before each
// launch).
GemvWs gemv_ws(int64_t N, int64_t K, int r) {
    auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
    GemvWs w{};
    const int r32 = ((r + 31) / 32) * 32;
    const int64_t S = (K + kGvSub - 1) / kGvSub;
    const int64_t ns = (S + kGvSlab - 1) / kGvSlab;
    const int64_t ni = (ns + kGvRun - 1) / kGvRun;
    w.RG = r32 / kGvRows + (N + kGvRows - 1) / kGvRows;
    w.off_u = 0;
    w.off_partial = al((size_t)kGvMaxM * r32 * 2);
    const int64_t items = (int64_t)(r32 / kGvRows) * ns + (w.RG - r32 / kGvRows) * ni;
    w.off_counters = w.off_partial + al((size_t)items * kGvAcc * 32 * 4);
    w.counter_bytes = (size_t)(w.RG + 2) * 4;
    w.total = w.off_counters + al(w.counter_bytes);
    return w;
}

// Shapes the one-launch kernel indexes with 32-bit arithmetic (block indices, units).
bool gemv_supported(int64_t M, int64_t N, int64_t K) {
    return M >= 1 && M <= kGvMaxM && N * (K / 64) < (1LL << 31) && N < (1LL << 30) && K < (1LL << 30);
}

cudaError_t launch_gemv(const CUtensorMap &map3, const CUtensorMap &map2, const int8_t *scale_q, const float *scale_c2,
                        const float *scale_mu, const uint16_t *X, const uint16_t *Xa, int M, int64_t N, int64_t K,
                        const uint16_t *A, const uint16_t *B, int r, float s, uint16_t *Y, uint16_t *U_save, void *ws,
                        const NF4Tables &tab, int num_sms, cudaStream_t st) {
    if (!gemv_supported(M, N, K)) return cudaErrorInvalidValue;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(nf4_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGvDynBytes);
    });
    if (attr_err != cudaSuccess) return attr_err;
    const GemvWs w = gemv_ws(N, K, r);
    GemvArgs a{};
    a.scale_q = scale_q;
    a.scale_c2 = scale_c2;
    a.scale_mu = scale_mu;
    a.X = X;
    a.Xa = Xa;
    a.A = A;
    a.B = B;
    a.Y = Y;
    a.U_save = U_save;
    a.N = (int)N;
    a.K = (int)K;
    a.KB = (int)(K / 64);
    a.M = M;
    a.r = r;
    a.r32 = ((r + 31) / 32) * 32;
    a.s = s;
    a.S = (int)((K + kGvSub - 1) / kGvSub);
    a.S_whole = (int)(K / kGvSub);
    a.NS = (a.S + kGvSlab - 1) / kGvSlab;
    a.RU = a.r32 / kGvRows;
    a.RG = (int)w.RG;
    a.NI = (a.NS + kGvRun - 1) / kGvRun;
    a.n_items = a.RU * a.NS + (a.RG - a.RU) * a.NI;
    for (int i = 0; i < 16; ++i) a.level[i] = tab.level[i];
    uint8_t *p = static_cast<uint8_t *>(ws);
    a.Ubf = reinterpret_cast<uint16_t *>(p + w.off_u);
    a.partial = reinterpret_cast<float *>(p + w.off_partial);
    a.counters = reinterpret_cast<uint32_t *>(p + w.off_counters);
    const unsigned grid = (unsigned)std::min<int64_t>(num_sms, a.n_items);
    nf4_gemv_kernel<<<grid, kGvThreads, kGvDynBytes, st>>>(map3, map2, a);
    count_launch();
    return cudaGetLastError();
}

}  // namespace qlora
