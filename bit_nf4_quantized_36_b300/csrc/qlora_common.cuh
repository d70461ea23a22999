// qlora_common.cuh -- shared device helpers of libqlora (sm_103a): NF4 format constants,
// the device error word, and thin inline-PTX wrappers for mbarrier, TMA and tcgen05/TMEM.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qlora {

// ---------------------------------------------------------------------------------------
// NF4 format constants.  The 16 levels of the "QLoRA" glossary's NF4 snippet (ultralytics):
// +-Phi^{-1} of evenly spaced probabilities between 0.5 and 0.9677083 (8 positive, 7
// negative, one exact zero), divided by Phi^{-1}(0.9677083), each rounded once to fp32.
// Stored as IEEE bit patterns, ascending.
// ---------------------------------------------------------------------------------------
static constexpr uint32_t kNF4Bits[16] = {
    0xbf800000u, 0xbf3239b3u, 0xbf066b30u, 0xbeca32a0u, 0xbe91a24cu, 0xbe3d353fu,
    0xbdba786bu, 0x00000000u, 0x3da2fb03u, 0x3e24cae1u, 0x3e7c04dcu, 0x3ead0338u,
    0x3ee1a4b7u, 0x3f1007aau, 0x3f3913b1u, 0x3f800000u};
static constexpr int kZeroCode = 7;
static constexpr int kBlock = 64;     // weights per absmax block
static constexpr int kGroup = 256;    // blocks per double-quantization group

// Kernel-argument copy of the tables: levels, and the 15 exact decision thresholds of the
// nearest-level rule (code = number of thresholds <= x; computed on the host).
// entries j = 0..33 for the 1/16-wide buckets j - 1 of [-1, 1]; entries 34..63 (reached only by
// a NaN) hold a NaN.  A power of two: the index is masked into the table.
static constexpr int kNF4Buckets = 64;

struct NF4Tables {
    float level[16];
    float thr[16];   // thr[0..14] used, thr[15] = +inf
    // Entry j describes the bucket starting at b = -1 + (j - 1) / 16: c = the number of thresholds
    // at or below b - 2^-12 and t = thr[c] (2.0 when c = 15), the one threshold that can fall in
    // [b - 2^-12, b + 1/16] (consecutive thresholds are at least 0.0805 apart).  Stored as t's
    // bit pattern with its low 4 mantissa bits replaced by c, which moves t by less than 2^-20.
    uint32_t bucket[kNF4Buckets];
};

// ---------------------------------------------------------------------------------------
// Device error word (latched; read and cleared by qlora_check_device_error).
// ---------------------------------------------------------------------------------------
// kErrTimeout: a bounded wait gave up; kErrLayout: a kernel found its shared memory laid out
// other than it was built for (it then does no work); kErrBounds: (device-check builds only) an
// index failed its bounds check, and the access was skipped
enum : uint32_t { kErrTimeout = 1u, kErrLayout = 2u, kErrBounds = 4u };
// Defined here: the library is one translation unit (libqlora.cu includes every .cu file).
__device__ uint32_t g_error_word = 0;
// Test hooks (qlora_test_inject): kInjectSkipCodes makes the leader CTA of the fused GEMM's first
// pair skip the codes copy of its first k-step, and with it that stage's arrival on the barrier
// its decode warps wait on, so the bounded wait runs out and the kernel unwinds without a fault.
// kInjectBounds (device-check builds only) moves one store index of nf4_dequantize past the end
// of its output, so that its bounds check fires (and skips the store).
enum : uint32_t { kInjectSkipCodes = 1u, kInjectBounds = 2u };
__device__ uint32_t g_inject = 0;

// Device-side bounds checks.  Built with QLORA_DEVICE_CHECKS (libqlora_checked.so), QLORA_IN_BOUNDS
// tests an index condition before a global-memory access: when it fails, the kernel latches
// kErrBounds in the error word and skips the access (no trap: the context stays usable and
// qlora_check_device_error reports it).  In the released library the condition is not evaluated.
#ifdef QLORA_DEVICE_CHECKS
__device__ __forceinline__ bool device_check(bool ok) {
    if (!ok) atomicOr(&g_error_word, kErrBounds);
    return ok;
}
#define QLORA_IN_BOUNDS(cond) (::qlora::device_check((cond)))
#else
#define QLORA_IN_BOUNDS(cond) (true)
#endif

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------------------
// Shared memory / mbarrier
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
// try_wait with a suspend-time hint: a waiting thread sleeps in hardware until the phase
// completes (or the hint elapses) instead of spinning and taking issue slots from the warps
// that do the work.
static constexpr uint32_t kSuspendHintNs = 200000;
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete, for at most kWaitTimeoutNs.  Every wait
// in the pipelined kernels goes through here: on a timeout (or when another thread of the CTA
// already gave up, flagged in *abort) it latches the device error word and returns false, so
// that the kernel unwinds instead of hanging.
static constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s; a stage normally takes us
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile uint32_t *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
            *abort = 1u;
            atomicOr(&g_error_word, kErrTimeout);
            return false;
        }
    }
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------------------
// TMA (tiled tensor copies global -> shared, completion counted on an mbarrier)
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar, int32_t x,
                                            int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}
// TMA store of a shared-memory tile (rows past the tensor's edges are not written), tracked by
// the thread's bulk async-group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *src, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until at most N committed bulk groups of this thread still read their shared-memory source
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// wait until all committed bulk groups of this thread have completed
__device__ __forceinline__ void bulk_wait_group_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// barrier among `count` threads (a multiple of 32) on hardware barrier `id` (1..15)
__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------------------
// tcgen05 / TMEM
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on `bar` once all tcgen05 operations issued so far by this thread have completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 32 lanes x 32 columns of 32 bit: thread i of the warp gets lane (taddr.lane + i),
// columns taddr.col .. +31.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
// 32 lanes x 16 columns of 32 bit.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
// 16 lanes x 256 bit, four repetitions along the columns: thread t (g = t / 4, c = t % 4) gets,
// for repetition k, r[4k .. 4k + 3] = (lane g, col 8k + 2c), (g, 8k + 2c + 1), (g + 8, 8k + 2c),
// (g + 8, 8k + 2c + 1), lanes and columns relative to taddr: the layout of a warp-level MMA
// accumulator fragment.
__device__ __forceinline__ void tmem_ld_16x256b_x4(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
// Four 8x8 b16 matrices from fragment registers to shared memory, each transposed: thread 8i + j
// gives the address of row j of matrix i, which receives column j of the fragment.
__device__ __forceinline__ void stmatrix_x4_trans(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(r0), "r"(r1),
                 "r"(r2), "r"(r3)
                 : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------------------
// CTA pairs (cluster of 2, cta_group::2): one MMA of M = 256 spans the tensor cores of both
// SMs; each CTA supplies 128 rows of A and half of the N columns of B from its own shared
// memory, and receives its 128 rows of D in its own TMEM.  Barrier addresses passed to the
// `_pair`/`_remote` helpers are shared::cluster addresses (see mapa_shared).
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
// Arrive on a barrier of either CTA of the cluster.  CTA-scope release: the data it publishes
// is this CTA's own shared memory (made visible to the tensor cores' async proxy by a preceding
// fence.proxy.async) or this CTA's finished TMEM reads, not global memory, and a cluster-scope
// release costs a full memory barrier (~0.5 us) on every pipeline stage.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// As mbar_try_wait / mbar_wait, with cluster-scope acquire: for barriers that the peer CTA's
// threads, TMA copies or MMA commits also arrive on.
__device__ __forceinline__ bool mbar_try_wait_cl(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cl(uint64_t *bar, uint32_t parity, volatile uint32_t *abort) {
    if (mbar_try_wait_cl(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_cl(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
            *abort = 1u;
            atomicOr(&g_error_word, kErrTimeout);
            return false;
        }
    }
}
// TMEM allocation shared by the pair: both CTAs' allocating warps execute these together.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Issued by the even CTA only: D (both CTAs' TMEM) (+)= A (both CTAs' smem) * B^T.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on the barrier at the same offset in each CTA of `cta_mask` once all pair MMAs issued
// so far by this thread have completed.
__device__ __forceinline__ void umma_commit_pair_mc(uint64_t *bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// Shared-memory matrix descriptor for tcgen05.mma, 128-byte swizzle.
//   bits  0-13: start address >> 4      bits 16-29: leading byte offset >> 4
//   bits 32-45: stride byte offset >> 4 bits 46-47: descriptor version (1)
//   bits 61-63: swizzle mode (2 = 128-byte swizzle)
// K-major operand (rows of 64 bf16 = 128 B, 8-row atoms): SBO = 1024 (next 8 rows), LBO unused.
// MN-major operand (64 MN-contiguous bf16 per 128-B row, rows along K): LBO = byte distance
// between 64-wide MN blocks, SBO = byte distance between 8-row groups along K.
__device__ __forceinline__ uint64_t make_sw128_desc(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, M = m (128, or 256 for a CTA pair),
// N = n.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format (1 = bf16),
//   bit 15 A major (1 = MN), bit 16 B major (1 = MN), 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t make_idesc_bf16(uint32_t n, bool a_mn_major, bool b_mn_major,
                                                       uint32_t m = 128u) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           ((n >> 3) << 17) | ((m >> 4) << 24);
}

// Byte offset of the 16-byte chunk `chunk` of row `row` inside a 128-byte-swizzled tile whose
// rows are 128 bytes (the layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B; the tile base is
// 1024-byte aligned).
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t chunk) {
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

}  // namespace qlora
