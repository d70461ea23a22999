/*
 * qlora.h -- C ABI of libqlora: the QLoRA frozen-base linear layer on NVIDIA B300 (sm_103a).
 *
 * The layer keeps a frozen weight matrix W [N_out, K_in] in 4-bit NormalFloat (NF4) with
 * double-quantized block scales, and trains a rank-r adapter (A [r, K], B [N, r]) on top:
 *
 *     Y = X W^T + (alpha / r) (X A^T) B^T,        W^ = dequant_bf16(W_nf4)
 *
 * Sources (page title and section):
 *   - "QLoRA -- La base en 4 bits, LoRA encima" (paperclase.com, LoRA course, lesson 8):
 *     "Parte 1" absmax per block; "Parte 2 - NormalFloat" quantile levels with an exact zero,
 *     W^ = NF4[c] * absmax; "Parte 3 - Cuanta memoria" 4 + 8/64 + 32/(64*256) bits per weight;
 *     "Parte 4 - LoRA encima" the Lineal4bit layer, h = W^ x + (alpha/r) B A x and
 *     dL/dx = (W^ + (alpha/r) B A)^T dL/dh, no gradient for W^.
 *   - "QLoRA" glossary (ultralytics.com), "Como funciona a QLoRA": NF4 levels as built in
 *     bitsandbytes, one absmax per 64 weights, scales double-quantized to 8 bits in blocks
 *     of 256, dequantized to bfloat16 right before the matmul, only the LoRA matrices updated.
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers, owned by the caller, row-major, 16-byte
 *     aligned.  bf16 tensors are passed as uint16_t bit patterns.  The library never
 *     allocates device memory; scratch space is the caller's workspace (size queries below).
 *   - Calls are asynchronous and ordered on `stream` (a cudaStream_t, NULL = legacy default
 *     stream).  The returned status covers argument checks and launch errors only.
 *     Device-side faults of the pipelined kernels (a bounded wait that ran out) are latched
 *     in a device word and reported by qlora_check_device_error().
 *   - Calls keep no state between them and may be issued from several host threads.
 *   - Shape rules: cols (K) % 64 == 0 so that no 64-weight block straddles two rows;
 *     rows (N) >= 1; tokens M >= 1; 1 <= r <= 256; alpha finite.
 */
#ifndef QLORA_H
#define QLORA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QLORA_OK = 0,
    QLORA_ERR_INVALID_ARG = 1,      /* NULL pointer, non-finite alpha, r out of range ...      */
    QLORA_ERR_UNSUPPORTED_SHAPE = 2,/* cols % 64 != 0, empty matrix, too large ...            */
    QLORA_ERR_MISALIGNED = 3,       /* a pointer is not 16-byte aligned                        */
    QLORA_ERR_WORKSPACE = 4,        /* workspace NULL or smaller than the size query returns  */
    QLORA_ERR_CUDA = 5,             /* a CUDA runtime/driver call or a kernel launch failed    */
    QLORA_ERR_TIMEOUT = 6,          /* a device-side bounded wait ran out (from the check call)*/
    QLORA_ERR_DEVICE_CHECK = 7      /* device-check build: an index failed its bounds check    */
} qlora_status;

/* One NF4 matrix with double-quantized scales.
 * Let n = rows*cols, nb = n/64 blocks (block b = flat elements [64b, 64b+64) of row-major W),
 * ng = ceil(nb/256) groups (group g = blocks [256g, 256g+256)).
 *   codes[n/2]        : byte j = (c[2j] << 4) | c[2j+1]; c = index into the NF4 table
 *   scale_codes[nb]   : int8 code q_b of the block scale, in [-127, 127]
 *   scale_scales[ng]  : fp32 c2_g, the largest |s_b - mu| in the group
 *   scale_offset[1]   : fp32 mu, the mean of all block scales of the matrix
 * The block scale is rebuilt as s'_b = fmaf(q_b, c2_g / 127, mu) and a weight as
 * bf16_rne(NF4[c] * s'_b).  All four arrays are device memory owned by the caller. */
typedef struct {
    int64_t rows;          /* N_out */
    int64_t cols;          /* K_in, a multiple of 64 */
    uint8_t *codes;
    int8_t *scale_codes;
    float *scale_scales;
    float *scale_offset;
} qlora_nf4_tensor;

/* Bytes of the four arrays of one quantized matrix: n/2 + nb + 4*ng + 4.
 * ("Parte 3 - Cuanta memoria", "Bits por parametro": 4 + 8/64 + 32/(64*256) bits per weight.)
 * Returns 0 if the shape is unsupported. */
size_t qlora_nf4_storage_bytes(int64_t rows, int64_t cols);

/* Workspace sizes (bytes, device memory) of the calls below; 0 means "no workspace needed"
 * for quantize only.  A call given less returns QLORA_ERR_WORKSPACE.  Returns (size_t)-1 if
 * the shape is unsupported. */
size_t qlora_quantize_workspace_bytes(int64_t rows, int64_t cols);
size_t qlora_fwd_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t r);
size_t qlora_bwd_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t r);
size_t qlora_merge_workspace_bytes(int64_t N, int64_t K, int32_t r);

/* NF4-quantize an fp32 matrix W [rows, cols] into `out` (its four arrays must be allocated
 * with the sizes above; out->rows/cols give the shape).
 * Definition ("Una capa QLoRA, a mano" and the glossary's NF4 snippet): per 64-block,
 * s_b = max |w|; each weight gets c = argmin_k |fl32(w / s_b) - NF4[k]| (fp32 division and
 * distances, ties to the lower k; an all-zero block gets the zero level); then the scales are
 * double-quantized ("Parte 3": 8 bits per scale, one 32-bit constant per 256 blocks):
 *   mu   = fl32(T / nb), T = pairwise fp64 tree (zero-padded to a power of two) over the
 *          group sums S_g, each S_g the fp64 sum of its scales in index order
 *   c2_g = max over the group of |fl32(s_b - mu)|
 *   q_b  = rint(fl32(fl32(fl32(s_b - mu) / c2_g) * 127)), or 0 when c2_g == 0.
 * Deterministic and bit-exact.  W must be finite.
 * ws: qlora_quantize_workspace_bytes(rows, cols) bytes of device memory (block scales and
 * group sums). */
qlora_status nf4_quantize(const float *W, const qlora_nf4_tensor *out, void *ws, size_t ws_bytes,
                          void *stream);

/* nf4_quantize without a workspace argument, for callers that cannot allocate device memory:
 * for example a serving process or plugin host that reserves its whole device-memory budget at
 * start-up and forbids later allocations, or an embedding runtime whose allocator must not be
 * bypassed.  (The source pages have no counterpart: this is an interface convenience.)
 * Same result, bit for bit, as nf4_quantize.  The scratch space lives in a fixed area inside the
 * library's device module (16 MiB + 256 KiB, held on every device that loads the library until
 * the process exits), which limits the matrix to rows * cols <= 2^28 weights; larger matrices
 * return QLORA_ERR_UNSUPPORTED_SHAPE without launching anything.  The call allocates nothing.
 * W and out must be on the current device: each call looks up the scratch area's address on the
 * current device (so no address survives a cudaDeviceReset), and the first call on a device may
 * load the library's device module there; make that first call before starting any stream
 * capture.  A failed lookup returns QLORA_ERR_CUDA.  All calls on a device share the one area,
 * so calls whose kernels may overlap on the GPU (different streams, or other host threads) race:
 * order them, e.g. on one stream.  No state carries from one call to the next. */
qlora_status nf4_quantize_noalloc(const float *W, const qlora_nf4_tensor *out, void *stream);

/* Dequantize to bf16: W_out[rows, cols] = bf16_rne(NF4[c] * s'_b) ("Cuantiles": w^ = NF4[c] *
 * absmax; glossary: dequantized to bfloat16 before the matmul).  No workspace. */
qlora_status nf4_dequantize(const qlora_nf4_tensor *q, uint16_t *W_out, void *stream);

/* ---- LoRA dropout on the adapter input ----------------------------------------------------
 * ("LoRA y QLoRA para un ajuste eficiente en costes", coddykit: LoraConfig lora_dropout=0.05.)
 * The adapter branch sees x_d = x * mask / (1 - p), mask ~ Bernoulli(1 - p) per element of X:
 *   Y = X W^T + s (X_d A^T) B^T;  dX = dY W^ + mask/(1-p) * (V A), V = bf16(s dY B);
 *   dA = V^T X_d;  dB = dY^T U,  U = bf16(s X_d A^T).
 * The mask is drawn from Philox4x32-10 (Salmon et al., SC'11): element e of the row-major [M, K]
 * X takes word e % 4 of the block with counter (e / 4 as two 32-bit words, offset as two 32-bit
 * words) and key (seed as two 32-bit words), and is kept when the word is >= floor(p 2^32).  The
 * backward call with the same (p, seed, offset) regenerates the forward's mask.  X_d is rounded
 * to bf16 (bf16(x * fl32(1 / (1 - p)))) before the adapter products.  0 <= p < 1; p = 0 keeps
 * every element (the plain layer, through the dropout code path). */
typedef struct {
    float p;
    uint64_t seed;
    uint64_t offset;
} qlora_dropout;

size_t qlora_fwd_dropout_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t r);
size_t qlora_bwd_dropout_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t r);
qlora_status qlora_linear_fwd_dropout(const qlora_nf4_tensor *W, const uint16_t *X, int64_t M, const uint16_t *A,
                                      const uint16_t *B, int32_t r, float alpha, const qlora_dropout *dropout,
                                      uint16_t *Y, uint16_t *U_save, void *ws, size_t ws_bytes, void *stream);
qlora_status qlora_linear_bwd_dropout(const qlora_nf4_tensor *W, const uint16_t *X, int64_t M, const uint16_t *A,
                                      const uint16_t *B, int32_t r, float alpha, const qlora_dropout *dropout,
                                      const uint16_t *dY, const uint16_t *U_saved, uint16_t *dX, float *dA, float *dB,
                                      void *ws, size_t ws_bytes, void *stream);

/* ---- Concatenated projections sharing one input ----------------------------------------
 * Several modules applied to the same X (q/k/v, or gate/up, with "all-linear" adapters: coddykit
 * "Módulos objetivo" and the config's target_modules) computed as one N-concatenated layer, so
 * that X is streamed once and all modules' tiles fill the GPU's waves together.
 * Module i: W_i [N_i, K] (N_i a multiple of 128, the same K for all modules), A_i [r_i, K] and
 * B_i [N_i, r_i] bf16 (16-byte aligned), 1 <= r_i <= 256, alpha_i finite.  1 <= G <= 4 modules,
 * and R8 = sum_i ceil8(r_i) <= 256.  Column offsets: o_i = N_0 + ... + N_{i-1} (outputs),
 * c_i = ceil8(r_0) + ... + ceil8(r_{i-1}) (the concatenated rank). */
typedef struct {
    const qlora_nf4_tensor *W;
    const uint16_t *A;
    const uint16_t *B;
    int32_t r;
    float alpha;
} qlora_cat_module;

/* Workspace sizes of the two calls below for modules with rows N[i] and ranks r[i]; (size_t)-1
 * for unsupported shapes. */
size_t qlora_cat_fwd_workspace_bytes(const int64_t *N, const int32_t *r, int32_t G, int64_t M, int64_t K);
size_t qlora_cat_bwd_workspace_bytes(const int64_t *N, const int32_t *r, int32_t G, int64_t M, int64_t K);

/* Y [M, sum N_i] bf16: columns o_i .. o_i + N_i - 1 hold module i's qlora_linear_fwd output.
 * U_save (nullable) [M, R8] bf16: columns c_i .. c_i + r_i - 1 hold bf16(s_i X A_i^T), the other
 * columns 0 (pass it to qlora_linear_bwd_cat). */
qlora_status qlora_linear_fwd_cat(const qlora_cat_module *mods, int32_t G, const uint16_t *X, int64_t M,
                                  uint16_t *Y, uint16_t *U_save, void *ws, size_t ws_bytes, void *stream);

/* dY [M, sum N_i] bf16 (columns as in Y); U_saved [M, R8] (nullable: recomputed).
 * dX [M, K] = sum_i (dY_i W^_i + s_i (dY_i B_i) A_i), one fp32 accumulation, bf16 out;
 * dA[i] [r_i, K] and dB[i] [N_i, r_i] fp32 as qlora_linear_bwd gives for module i. */
qlora_status qlora_linear_bwd_cat(const qlora_cat_module *mods, int32_t G, const uint16_t *X, int64_t M,
                                  const uint16_t *dY, const uint16_t *U_saved, uint16_t *dX, float *const *dA,
                                  float *const *dB, void *ws, size_t ws_bytes, void *stream);

/* Merge the adapters into the base weight ("QLoRA" glossary, "Compromissos": to merge the
 * adapters the base weight is first dequantized to 16 bits; "QLoRA e metodos relacionados": the
 * fine-tuned model is merged into 16-bit weights):
 *   W_out [N, K] (bf16) = bf16_rne(fl32(W^ + s (B A))),  s = fl32(alpha / r),
 * with W^ the nf4_dequantize values, A [r, K] and B [N, r] bf16, B A accumulated in fp32 and
 * the sum formed by one fp32 fused multiply-add (s * (B A) + W^) before the rounding.
 * Workspace: qlora_merge_workspace_bytes (B padded to a multiple of 8 columns when r % 8 != 0,
 * else none).  W_out, A and (r % 8 == 0) B must be 16-byte aligned; 1 <= r <= 256. */
qlora_status qlora_merge(const qlora_nf4_tensor *W, const uint16_t *A, const uint16_t *B, int32_t r, float alpha,
                         uint16_t *W_out, void *ws, size_t ws_bytes, void *stream);

/* Forward of the layer ("Parte 4 - LoRA encima", h = W^ x + (alpha/r) B A x):
 *   Y [M, N] (bf16) = X W^T + U B^T,   U = bf16((alpha/r) X A^T)  [M, r]
 * X [M, K] bf16, A [r, K] bf16, B [N, r] bf16; fp32 accumulation; W^ is dequantized inside the
 * GEMM main loop and never written to memory.  For M <= 8 the block scale is instead factored out
 * of each 64-weight block's dot product (the bf16 levels times x, summed in fp32, times the exact
 * block scale s'_b), so Y is the product with W^ up to the layer tolerance, not bit for bit.
 * U_save (nullable) receives U [M, r] (bf16, already multiplied by alpha/r) for the backward. */
qlora_status qlora_linear_fwd(const qlora_nf4_tensor *W, const uint16_t *X, int64_t M,
                              const uint16_t *A, const uint16_t *B, int32_t r, float alpha,
                              uint16_t *Y, uint16_t *U_save, void *ws, size_t ws_bytes, void *stream);

/* Backward of the layer ("El gradiente atraviesa la base de 4 bits": dL/dx = (W^ + (alpha/r)
 * B A)^T dL/dh; dL/dW^ is not computed; glossary: only the two LoRA matrices are updated):
 *   V  = bf16((alpha/r) dY B)                [M, r]
 *   dX = dY W^ + V A                          [M, K] bf16
 *   dA = V^T X                                [r, K] fp32   (= (alpha/r) (dY B)^T X)
 *   dB = dY^T U                               [N, r] fp32   (= (alpha/r) dY^T X A^T)
 * U_saved (nullable): the U_save of the forward; when NULL, U is recomputed from X and A.
 * dX, dA, dB are overwritten (not accumulated). */
qlora_status qlora_linear_bwd(const qlora_nf4_tensor *W, const uint16_t *X, int64_t M,
                              const uint16_t *A, const uint16_t *B, int32_t r, float alpha,
                              const uint16_t *dY, const uint16_t *U_saved, uint16_t *dX, float *dA,
                              float *dB, void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------------------
 * Paged optimizer states for the adapters ("QLoRA" glossary entry (ultralytics.com), "Como
 * funciona a QLoRA", paged-optimizers bullet; "Capitulo 1: Que es QLoRA?"
 * (docs.skillversehub.com), "Componentes clave", "Optimizadores paginados"): the states live in
 * NVIDIA unified memory and move to CPU RAM during memory spikes, so that training does not
 * fail for lack of GPU memory.
 * --------------------------------------------------------------------------------------- */

/* Location argument of qlora_paged_prefetch: host memory (any value >= 0 is a device ordinal). */
#define QLORA_PAGE_HOST (-1)

/* Allocates `bytes` of unified (managed) memory, accessible from the host and every device,
 * migrated page by page by the driver; *out receives the pointer (NULL on error).  The pages
 * are first placed on the processor that touches them first.  QLORA_ERR_INVALID_ARG for
 * bytes == 0 or out == NULL; QLORA_ERR_CUDA when the current device has no managed memory or
 * the allocation fails.  Free with qlora_paged_free. */
qlora_status qlora_paged_alloc(size_t bytes, void **out);

/* Frees memory from qlora_paged_alloc (synchronizes the device, as cudaFree does).  NULL is a
 * no-op; a pointer that is not managed memory returns QLORA_ERR_INVALID_ARG. */
qlora_status qlora_paged_free(void *ptr);

/* Moves the pages of [ptr, ptr + bytes) (inside one paged allocation) to `device` (a device
 * ordinal) or to host memory (QLORA_PAGE_HOST), asynchronously on `stream`: page the states out
 * before a memory spike and back in before the next optimizer step.  A hint: the data stays
 * valid wherever the pages are.  On a device without concurrent managed access it does nothing
 * and returns QLORA_OK.  QLORA_ERR_INVALID_ARG for a NULL or non-managed pointer or an unknown
 * device; bytes == 0 is a no-op. */
qlora_status qlora_paged_prefetch(const void *ptr, size_t bytes, int32_t device, void *stream);

/* Hyper-parameters of the adapters' AdamW step.  READING: the pages name no update rule; the
 * optimizer is AdamW (Loshchilov and Hutter, decoupled weight decay). */
typedef struct qlora_adamw {
    float lr;            /* >= 0, finite                     */
    float beta1, beta2;  /* in [0, 1)                         */
    float eps;           /* > 0, finite                      */
    float weight_decay;  /* >= 0, finite (decoupled)          */
} qlora_adamw;

/* One AdamW step, t >= 1 (the step count including this one), over n elements, in fp32:
 *   p <- p (1 - lr wd);  m <- b1 m + (1 - b1) g;  v <- b2 v + (1 - b2) g^2;
 *   p <- p - (lr / (1 - b1^t)) m / (sqrt(v) / sqrt(1 - b2^t) + eps)
 * p, m, v [n] fp32 are updated in place; g [n] fp32 is read (the dA or dB of qlora_linear_bwd).
 * Any of them may be paged memory (wherever its pages are) or device memory; all must be
 * 16-byte aligned.  p_bf16 (nullable, 8-byte aligned) receives bf16(p) after the step: the
 * adapter copy the layer calls read.  Concatenate every adapter of a model into one range to
 * update them all in one launch.  n == 0 is a no-op.  Returns QLORA_ERR_INVALID_ARG for
 * out-of-range hyper-parameters, t < 1, n < 0 or a NULL array, QLORA_ERR_MISALIGNED, or
 * QLORA_ERR_CUDA. */
qlora_status qlora_adamw_step(const qlora_adamw *hp, int64_t t, int64_t n, float *p, const float *g, float *m,
                              float *v, uint16_t *p_bf16, void *stream);

/* Synchronizes `stream`, then reads and clears the library's device error word on the current
 * device.  QLORA_OK, QLORA_ERR_TIMEOUT (a pipelined kernel gave up a bounded wait and exited
 * early; its outputs are undefined), QLORA_ERR_DEVICE_CHECK (only from libqlora_checked.so, the
 * same library built with device-side bounds checks: an index failed its check and the access
 * was skipped; the outputs are undefined) or QLORA_ERR_CUDA. */
qlora_status qlora_check_device_error(void *stream);

/* Test hook for the device-side failure path (not for normal use).  flags ==
 * QLORA_INJECT_SKIP_CODES makes every following launch of the fused NF4-dequant GEMM (layer
 * calls with more than 32 tokens, forward and backward dX) on the current device leave out one
 * copy of packed codes: the leader CTA of its first CTA pair issues no codes copy for its first
 * k-step, so that stage's barrier never completes.  The decode warps' bounded wait then runs
 * out (about 2 s), the kernel's roles drain and exit, and the next qlora_check_device_error
 * returns QLORA_ERR_TIMEOUT; the call's outputs are undefined.  flags == 0 switches it off.
 * Synchronous with respect to the host; do not change it while calls are in flight.  Returns
 * QLORA_ERR_INVALID_ARG for an unknown flag, QLORA_ERR_CUDA if the device is unusable. */
#define QLORA_INJECT_SKIP_CODES 1u
/* flags == QLORA_INJECT_BOUNDS (libqlora_checked.so only; QLORA_ERR_INVALID_ARG from the released
 * library) moves one store index of each following nf4_dequantize past the end of its output:
 * the kernel's bounds check skips that store and the next qlora_check_device_error returns
 * QLORA_ERR_DEVICE_CHECK.  Nothing is written out of bounds. */
#define QLORA_INJECT_BOUNDS 2u
qlora_status qlora_test_inject(uint32_t flags);

/* Short English description of a status code (static string). */
const char *qlora_status_string(qlora_status s);

/* Number of kernels this library has launched in this process (all devices).  Used by
 * benchmarks to count launches inside a timed region. */
uint64_t qlora_launch_count(void);

/* The 16 NF4 levels used by the library's kernels (fp32, ascending), for inspection. */
void qlora_nf4_levels(float out[16]);

/* Benchmark instrumentation (not needed for normal use).  `events` holds 2*capacity
 * cudaEvent_t handles created by the caller; from now on the library records events[2i] just
 * before and events[2i+1] just after the i-th weight-streaming step of a layer call: the
 * launch of the fused NF4-dequant GEMM kernel (forward or backward dX, with the reduction of its
 * partials when the contraction is split), or, for a forward of up to eight tokens, the
 * one-launch GEMV (which also computes the adapter terms and the finish); on the launch stream,
 * until `capacity` steps are recorded.
 * Under stream capture the records become event-record nodes of the graph, timing each replay.
 * events == NULL switches the recording off.  Process-wide; do not change it while calls are
 * in flight on other host threads.  Returns QLORA_ERR_INVALID_ARG for capacity < 0 or a NULL
 * handle among the 2*capacity events. */
qlora_status qlora_set_kernel_timer(void **events, int32_t capacity);

/* Number of weight-streaming steps recorded since the last qlora_set_kernel_timer call. */
int32_t qlora_kernel_timer_count(void);

#ifdef __cplusplus
}
#endif

#endif /* QLORA_H */
