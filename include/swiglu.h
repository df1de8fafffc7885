/*
 * swiglu.h -- C ABI of the GB300 (sm_103a) fused SwiGLU projection library.
 *
 * The operation (page "Riepilogo Tecnico: Sovrapposizione delle Attivazioni a
 * Livello di Tile per l'Inferenza Efficiente di LLM", gist.science paper
 * 2607.02521, section "Definizione del Problema"):
 *
 *     Y[M,N] = SiLU(A[M,K] x W1[K,N]) (.) (A[M,K] x W2[K,N]),
 *     SiLU(x) = x / (1 + e^-x),
 *
 * computed on tcgen05 tensor cores with FP32 accumulation; the gate and up
 * products stay on chip (tensor memory) and only Y is written, rounded once
 * to BF16 (round to nearest even).
 *
 * Conventions shared by every entry point:
 *   - All matrices are dense row-major with no padding: A is [M,K] (K
 *     contiguous), weights are [K,N] (N contiguous), Y is [M,N].
 *   - All tensor pointers are CUDA device pointers owned by the caller; the
 *     library never allocates, frees or retains them past the call.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Work is enqueued asynchronously; no entry point synchronises
 *     except swiglu_device_status().
 *   - Argument errors are reported synchronously, before anything is enqueued.
 *     CUDA launch errors are reported as SWIGLU_ERR_CUDA.  A device-side wait
 *     that exceeded its time limit (see swiglu_set_wait_timeout_ns) is recorded
 *     on the device and reported by swiglu_device_status().
 *   - Alignment rules come from the tensor-memory-accelerator copy engine:
 *     every base pointer 16-byte aligned, and every row pitch a multiple of
 *     16 bytes (K and N multiples of 8 for BF16, of 16 for FP8).
 *   - Y must not overlap any input.
 *   - M, N or K equal to 0 is valid: M = 0 or N = 0 enqueues nothing; K = 0
 *     makes every product zero, so Y is filled with zeros.
 *   - Dimensions must be below 2^31.
 *   - Threading: calls may come from several host threads; the lazily built
 *     per-device state is guarded by a lock.
 */
#ifndef SWIGLU_GB300_H
#define SWIGLU_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
typedef enum {
    SWIGLU_OK = 0,
    SWIGLU_ERR_INVALID_ARG = 1,  /* null pointer, negative size, overlap, bad variant */
    SWIGLU_ERR_MISALIGNED = 2,   /* base not 16-byte aligned or row pitch not a multiple of 16 bytes */
    SWIGLU_ERR_UNSUPPORTED = 3,  /* device is not sm_103 / sm_100 family, or size beyond limits */
    SWIGLU_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
    SWIGLU_ERR_TIMEOUT = 5       /* a device-side wait ran past its limit (see swiglu_device_status) */
} swiglu_status;

/* Kernel variants.  SWIGLU_VARIANT_AUTO lets the library choose by (M,N,K). */
typedef enum {
    SWIGLU_VARIANT_AUTO = 0,
    /* one CTA per SM, 128-row tiles, 128 output columns per tile
       (one 128x256 MMA covers the gate and up halves) */
    SWIGLU_VARIANT_1SM_N128 = 1,
    /* one CTA per SM, 128-row tiles, 64 output columns per tile (more tiles for small M) */
    SWIGLU_VARIANT_1SM_N64 = 2,
    /* CTA pair (2-CTA cluster, tcgen05 cta_group::2): 256-row tiles, 128 output
       columns, each CTA streams A rows and one weight block (large M) */
    SWIGLU_VARIANT_2SM_N128 = 3,
    /* one CTA per SM, 128-row tiles, 32 output columns per tile (small M: one
       tile per SM for N = 4864 on 152 SMs) */
    SWIGLU_VARIANT_1SM_N32 = 4,
    /* 5-8: retired numbers, kept unused; passing one returns
       SWIGLU_ERR_INVALID_ARG */
    /* split-K over a cluster of 2 CTAs (small M): each CTA multiplies half of
       the K steps of one 128-row x 64-column tile and the two partial gate/up
       accumulators are summed through distributed shared memory before the
       activation; all of a CTA's weight and A bytes fit in flight at once */
    SWIGLU_VARIANT_1SM_N64_SK2 = 9,
    /* M <= 128 only: the transposed product on CTA pairs (tcgen05
       cta_group::2 with the weights on the MMA's M side, M = 128 weight rows,
       and A's rows on its N side, half in each CTA); each pair makes 64
       output columns for all rows over all of K, so a CTA's whole K range of
       weights and A fits in flight at once and no partial sums are
       exchanged */
    SWIGLU_VARIANT_2SM_SWAP = 10,
    SWIGLU_VARIANT_COUNT_ = 11
} swiglu_variant;

/*
 * Y = SiLU(A x W1) (.) (A x W2) with BF16 A, W1, W2 and BF16 Y.
 * Page section "Metodologia", item 1 ("Kernel-1"): two weight matrices, the
 * gate and up products of one output tile computed together.
 *   A  : device, BF16 [M,K] row-major        (read)
 *   W1 : device, BF16 [K,N] row-major (gate)  (read)
 *   W2 : device, BF16 [K,N] row-major (up)    (read)
 *   Y  : device, BF16 [M,N] row-major        (written)
 */
int swiglu_fused(const void *A, const void *W1, const void *W2, void *Y,
                 int64_t M, int64_t N, int64_t K, void *stream);

/*
 * The interleaved form.  Page section "Metodologia", item 2 ("Kernel-2"):
 * one weight matrix W_fused[K,2N] whose even column 2n is gate column n and
 * whose odd column 2n+1 is up column n; one product over [M,2N,K] whose
 * adjacent accumulator columns (2n, 2n+1) give Y[m,n] = SiLU(D[m,2n]) * D[m,2n+1].
 *   A      : device, BF16 [M,K] row-major  (read)
 *   Wfused : device, BF16 [K,2N] row-major (read), as made by swiglu_pack_interleaved
 *   Y      : device, BF16 [M,N] row-major  (written)
 */
int swiglu_fused_interleaved(const void *A, const void *Wfused, void *Y,
                             int64_t M, int64_t N, int64_t K, void *stream);

/*
 * Weight packer for the interleaved form (same page, section "Metodologia",
 * item 2): Wfused[k,2n] = W1[k,n], Wfused[k,2n+1] = W2[k,n].  A one-off step at
 * model load, not part of the per-call path.
 *   W1, W2 : device, BF16 [K,N] row-major (read)
 *   Wfused : device, BF16 [K,2N] row-major (written; must not overlap W1/W2)
 */
int swiglu_pack_interleaved(const void *W1, const void *W2, void *Wfused,
                            int64_t K, int64_t N, void *stream);

/*
 * FP8 E4M3 operands with per-tensor scales (page section "Definizione del
 * Problema": quantisation to FP8 raises tensor-core density, which makes the
 * memory-bound gate/up traffic matter more).  The value of an operand element
 * is code * scale; the result is the same definition on those values,
 *     Y = SiLU(sA*sW1 * (Aq x W1q)) (.) (sA*sW2 * (Aq x W2q)),
 * with FP32 accumulation and BF16 Y.  FP8 weights are taken K-major, i.e. as
 * the [N,K] row-major transpose of the [K,N] weights of the BF16 entry points
 * (each output column's K weights contiguous), the layout quantised
 * checkpoints use.
 *   Aq       : device, E4M3 [M,K] row-major  (read)
 *   W1t, W2t : device, E4M3 [N,K] row-major  (read)
 *   sA, sW1, sW2 : device pointers to one float each (read at kernel time)
 *   Y        : device, BF16 [M,N] row-major  (written)
 * K must be a multiple of 16 and N of 8; pointers 16-byte aligned.
 */
int swiglu_fused_fp8(const void *Aq, const void *W1t, const void *W2t, const float *sA,
                     const float *sW1, const float *sW2, void *Y, int64_t M, int64_t N,
                     int64_t K, void *stream);

/* The interleaved form with FP8 operands: Wfused_t [2N,K] row-major, row 2n =
 * gate row n (scale sW1), row 2n+1 = up row n (scale sW2), as made by
 * swiglu_pack_interleaved_fp8. */
int swiglu_fused_interleaved_fp8(const void *Aq, const void *Wfused_t, const float *sA,
                                 const float *sW1, const float *sW2, void *Y, int64_t M,
                                 int64_t N, int64_t K, void *stream);

/* Packer for the FP8 interleaved form, K-major: Wfused_t[2n,:] = W1t[n,:],
 * Wfused_t[2n+1,:] = W2t[n,:] (the column interleave of the page's Kernel-2
 * in transposed storage).  W1t, W2t: E4M3 [N,K]; Wfused_t: E4M3 [2N,K]. */
int swiglu_pack_interleaved_fp8(const void *W1t, const void *W2t, void *Wfused_t, int64_t N,
                                int64_t K, void *stream);

/*
 * INT4 weights (weight-only quantisation; the page names INT4 in section
 * "Definizione del Problema" as a precision that raises tensor-core density,
 * without fixing a format).  Format: signed 4-bit two's complement codes,
 * packed two per byte along N (byte k*(N/2) + n/2 holds column n in its low
 * nibble when n is even, in its high nibble when n is odd); one BF16 scale per
 * column and per group of `group` consecutive K rows.  The weight is
 * BF16(q * s) (the product rounded once, to nearest even); the result is the
 * BF16 definition with those weights:
 *     Y = SiLU(A x W1) (.) (A x W2),  W[k,n] = BF16(q[k,n] * S[k/group, n])
 *   A        : device, BF16 [M,K] row-major      (read)
 *   W1q, W2q : device, uint8 [K, N/2] row-major  (read)
 *   S1, S2   : device, BF16 [K/group, N]         (read)
 *   Y        : device, BF16 [M,N] row-major      (written)
 * group must be a multiple of 64 dividing K; N a multiple of 32; K a multiple
 * of 8; pointers 16-byte aligned.  For M <= 128 with few columns it runs the
 * split-K cluster kernel (SWIGLU_VARIANT_1SM_N64_SK2's structure), otherwise
 * a one-CTA-per-128-column kernel over all of K (one or two 128-row blocks per
 * CTA); in both, warps decode each step's codes to BF16 in shared memory
 * before the MMA reads them: the weight stream is 4.1 bits per weight instead
 * of 16.
 */
int swiglu_fused_w4(const void *A, const void *W1q, const void *S1, const void *W2q,
                    const void *S2, void *Y, int64_t M, int64_t N, int64_t K, int64_t group,
                    void *stream);

/*
 * INT4 weights in a K-major layout, for few tokens (decode).  Same format and
 * result as swiglu_fused_w4 (page section "Definizione del Problema"), with
 * the codes rearranged once at model load by swiglu_pack_w4_kmajor:
 *   Wk : uint8 [N, K/2]: row n holds column n's K codes, eight per 32-bit
 *        little-endian word; word j holds codes k = 8j..8j+7 with code 8j+2i
 *        in nibble i and code 8j+2i+1 in nibble 4+i (i = 0..3; nibble 0 = the
 *        low four bits).
 * swiglu_pack_w4_kmajor(Wq, Wk, K, N): Wq [K, N/2] in swiglu_fused_w4's layout
 *   -> Wk; K a multiple of 8, N even, pointers 16-byte aligned, no overlap.
 * swiglu_fused_w4_kmajor: Y = SiLU(A x W1) (.) (A x W2) from A [M,K], W1k,
 *   W2k [N, K/2] (packed), S1, S2 [K/group, N] BF16 (as swiglu_fused_w4),
 *   Y [M,N]; the same size rules as swiglu_fused_w4.  Runs the transposed
 *   product (weights on the MMA's M side, tokens on its N side): one CTA per
 *   128 weight columns over all of K, the codes decoded to BF16 straight into
 *   tensor memory, the tensor core's A operand; tokens in passes of 64
 *   (M <= 64) or 128.  Built for M <= 128; larger M repeats the decode per
 *   128 tokens.
 */
int swiglu_pack_w4_kmajor(const void *Wq, void *Wk, int64_t K, int64_t N, void *stream);
int swiglu_fused_w4_kmajor(const void *A, const void *W1k, const void *S1, const void *W2k,
                           const void *S2, void *Y, int64_t M, int64_t N, int64_t K,
                           int64_t group, void *stream);

/*
 * MXFP8 and NVFP4 weights (weight-only; the formats the GEMM page names for
 * Blackwell, read per the OCP Microscaling specification and NVIDIA's NVFP4):
 *   MXFP8: C1, C2: E4M3 codes, uint8 [K,N] row-major; S1, S2: E8M0 scales,
 *          uint8 [K/32, N] (value 2^(e-127)), one per column and 32 K rows.
 *          W = BF16(E4M3(c) * 2^(e-127)).
 *   NVFP4: C1, C2: E2M1 codes, uint8 [K, N/2] (two per byte along N, column n
 *          in the low nibble when even); S1, S2: E4M3 scales, uint8 [K/16, N],
 *          one per column and 16 K rows; g1, g2: device pointers to one FP32
 *          scale per tensor.  W = E2M1(c) * E4M3(s) * g.
 * Y = SiLU(A x W1) (.) (A x W2) with BF16 A [M,K] and Y [M,N].  The codes are
 * decoded to BF16 in shared memory inside the same kernels as the INT4 form
 * (E4M3 * 2^k and E2M1 * E4M3 are exact in BF16) and multiplied on BF16 tensor
 * cores;
 * the NVFP4 tensor scales multiply the gate and up sums before the
 * activation.  K a multiple of 64, N of 32; pointers 16-byte aligned (g1, g2:
 * 4-byte).
 */
int swiglu_fused_mxfp8(const void *A, const void *C1, const void *S1, const void *C2,
                       const void *S2, void *Y, int64_t M, int64_t N, int64_t K, void *stream);
int swiglu_fused_nvfp4(const void *A, const void *C1, const void *S1, const float *g1,
                       const void *C2, const void *S2, const float *g2, void *Y, int64_t M,
                       int64_t N, int64_t K, void *stream);

/*
 * MXFP8 weights in a K-major layout, for few tokens: the same result and
 * scales as swiglu_fused_mxfp8, run by swiglu_fused_w4_kmajor's kernel.
 *   C1k, C2k: E4M3 codes, uint8 [N, K]: the byte transpose of
 *             swiglu_fused_mxfp8's [K, N] codes (row n holds column n's K
 *             codes), made once at model load.
 *   S1, S2:   E8M0 scales, uint8 [K/32, N], as swiglu_fused_mxfp8.
 * The codes are decoded to BF16 (E4M3 * 2^(e-127), exact in FP32, rounded
 * once) straight into tensor memory.  K a multiple of 64, N of 32; pointers
 * 16-byte aligned.
 */
int swiglu_fused_mxfp8_kmajor(const void *A, const void *C1k, const void *S1, const void *C2k,
                              const void *S2, void *Y, int64_t M, int64_t N, int64_t K,
                              void *stream);

/*
 * NVFP4 weights in the K-major layout, for few tokens: the same result and
 * scales as swiglu_fused_nvfp4, run by swiglu_fused_w4_kmajor's kernel.
 * E2M1 codes are four-bit codes in the same [K, N/2] byte layout as INT4, so
 * swiglu_pack_w4_kmajor turns C1, C2 into C1k, C2k ([N, K/2]) once at model
 * load.  S1, S2: E4M3 [K/16, N] as swiglu_fused_nvfp4; g1, g2: device FP32.
 * The codes are decoded exactly to BF16 (E2M1 * E4M3) straight into tensor
 * memory; g1 and g2 multiply the gate and up sums before the activation.
 * K a multiple of 64, N of 32; pointers 16-byte aligned (g1, g2: 4-byte).
 */
int swiglu_fused_nvfp4_kmajor(const void *A, const void *C1k, const void *S1, const float *g1,
                              const void *C2k, const void *S2, const float *g2, void *Y,
                              int64_t M, int64_t N, int64_t K, void *stream);

/*
 * The producer of the FP8 form's A operand: RMSNorm of each row of X followed
 * by per-tensor E4M3 quantisation (FP8 quantisation is what the page's
 * section "Definizione del Problema" names as raising tensor-core density; the
 * page defines neither step, so both follow the standard definitions):
 *     a[m,k] = x[m,k] * gamma[k] / sqrt(mean_k x[m,k]^2 + eps)
 *     *sA    = max|a| / 448          (448 = largest finite E4M3 value)
 *     Aq     = E4M3(a / *sA)         (round to nearest even, saturating)
 * A row whose mean square plus eps is zero gives zeros; *sA = 0 gives all-zero
 * codes.  Arithmetic is FP32; a code may differ from the exactly rounded one
 * only where a / *sA lies within FP32 rounding of a midpoint between codes.
 *   X     : device, BF16 [M,K] row-major (read)
 *   gamma : device, BF16 [K] (read), or NULL for all ones
 *   eps   : finite, >= 0
 *   Aq    : device, E4M3 [M,K] row-major (written), the Aq of swiglu_fused_fp8
 *   sA    : device, one float (written), the sA of swiglu_fused_fp8
 * K must be a positive multiple of 16; X, gamma and Aq 16-byte aligned.
 * Enqueues three kernels on `stream` (one that zeroes *sA, then an amax
 * pass and a quantise pass, each waiting for its predecessor through
 * programmatic dependent launch; rows longer than 25600 elements use a
 * memset and two loop kernels instead); no host sync.
 * Aq and *sA must not overlap X or gamma.  M = 0 writes *sA = 0 only.
 */
int swiglu_rmsnorm_quant_fp8(const void *X, const void *gamma, float eps, void *Aq, float *sA,
                             int64_t M, int64_t K, void *stream);

/*
 * Per-tensor E4M3 quantisation without normalisation, for weights:
 *     *s = max|x| / 448,   Xq = E4M3(x / *s)
 * with the rounding and zero rules of swiglu_rmsnorm_quant_fp8.  X: device,
 * BF16 [M,K]; Xq: device, E4M3 [M,K]; s: device float.  For the FP8 entry
 * points' K-major weights pass the [N,K] transpose of W (rows of K).  K a
 * positive multiple of 16, X and Xq 16-byte aligned.
 */
int swiglu_quant_fp8(const void *X, void *Xq, float *s, int64_t M, int64_t K, void *stream);

/*
 * The down projection that completes the MLP block the page studies (section
 * "Definizione del Problema": the gate/up materialisation is 9-37 % of MLP
 * time; the MLP ends with a product by the down-projection weight):
 *     Z[M,N] = X[M,K] x W[K,N] (+ R[M,N]),   BF16 in, FP32 accumulate, BF16 out.
 *   X : device, BF16 [M,K] row-major (read)
 *   W : device, BF16 [K,N] row-major (read)
 *   R : device, BF16 [M,N] row-major residual (read), or NULL; may equal Z
 *   Z : device, BF16 [M,N] row-major (written)
 *   workspace : device scratch of workspace_bytes (caller-owned, 16-byte
 *       aligned) used for split-K partial sums when the product has too few
 *       output tiles to occupy the GPU (small M); swiglu_linear_workspace_size()
 *       gives the bytes wanted.  NULL or too small is valid: the product then
 *       runs without splitting K (same result up to summation order).
 *       When the product's 128 x 64 output tiles, spread over clusters of 4
 *       or 8 CTAs that each take a slice of K, fit one wave of the GPU (e.g.
 *       M <= 128 with N <= 1216 on 152 SMs), the slices' partial sums are
 *       added in distributed shared memory inside each cluster and no
 *       workspace is used (the size query returns 0).
 * K and N multiples of 8; other rules as above.
 */
uint64_t swiglu_linear_workspace_size(int64_t M, int64_t N, int64_t K);
int swiglu_linear(const void *X, const void *W, const void *R, void *Z, int64_t M, int64_t N,
                  int64_t K, void *workspace, uint64_t workspace_bytes, void *stream);

/*
 * The SwiGLU MLP block built from the two entry points above:
 *     Y = BF16(SiLU(A W1) (.) (A W2)),   Z = Y W3 (+ R)
 *   A  : BF16 [M,H]; W1, W2: BF16 [H,F]; W3: BF16 [F,H]; R: BF16 [M,H] or NULL; Z: BF16 [M,H]
 *   workspace : caller-owned device scratch, at least M*F*2 bytes (Y lives in
 *       its first M*F*2 bytes, rounded up to 256), preferably
 *       swiglu_mlp_workspace_size() bytes (room for split-K partial sums).
 * Two kernels on `stream`; the second starts its set-up while the first ends
 * (programmatic dependent launch) and reads Y while it is still in L2.
 */
uint64_t swiglu_mlp_workspace_size(int64_t M, int64_t H, int64_t F);
int swiglu_mlp(const void *A, const void *W1, const void *W2, const void *W3, const void *R,
               void *Z, int64_t M, int64_t H, int64_t F, void *workspace,
               uint64_t workspace_bytes, void *stream);

/*
 * swiglu_mlp for callers that cannot allocate device memory.  The paper has no
 * counterpart to this entry point; it is a convenience of this library.
 * Some code may not call cudaMalloc or any allocating routine: a plugin that
 * is handed only the tensors it reads and writes, or a runtime whose device
 * memory is planned before it runs and that forbids allocations while it
 * executes.  This entry point takes only the inputs and the output and uses a
 * scratch area kept inside the library:
 *   - the area is a fixed 32 MiB of device memory
 *     (swiglu_mlp_noalloc_scratch_bytes()), present on every GPU the library
 *     is used on and held until the process exits;
 *   - Y (M*F BF16 values) must fit in it: M*F*2 > 32 MiB is rejected with
 *     SWIGLU_ERR_UNSUPPORTED before anything is enqueued; what is left of the
 *     area holds the down projection's split-K partial sums when they fit,
 *     and otherwise the down projection runs without splitting K;
 *   - the first call on a device looks up the area's device address, a
 *     host-side set-up step; make that first call before any stream capture
 *     that would include it.  The address is kept per device and looked up
 *     again when the device's context changes (after cudaDeviceReset);
 *   - all calls on a device share the one area, which keeps what the last call
 *     left in it; nothing in it needs to start at zero (each call writes all
 *     it later reads), but calls whose GPU work overlaps in time (unordered
 *     streams, several host threads) race on it and must be serialised by the
 *     caller.
 * Arguments, layouts and the result are those of swiglu_mlp.
 */
uint64_t swiglu_mlp_noalloc_scratch_bytes(void);
int swiglu_mlp_noalloc(const void *A, const void *W1, const void *W2, const void *W3,
                       const void *R, void *Z, int64_t M, int64_t H, int64_t F, void *stream);

/* swiglu_fused / swiglu_fused_interleaved with an explicit variant
 * (SWIGLU_VARIANT_*) instead of the library's choice; for sweeps and tests. */
int swiglu_fused_ex(const void *A, const void *W1, const void *W2, void *Y,
                    int64_t M, int64_t N, int64_t K, int32_t variant, void *stream);
int swiglu_fused_interleaved_ex(const void *A, const void *Wfused, void *Y,
                                int64_t M, int64_t N, int64_t K, int32_t variant,
                                void *stream);

/* The variant SWIGLU_VARIANT_AUTO resolves to for this shape and form
 * (interleaved = 0 or 1) on the current device.  Host-only. */
int swiglu_select_variant(int64_t M, int64_t N, int64_t K, int32_t interleaved);

/* The kernel the weight-format entry points (swiglu_fused_w4, _mxfp8, _nvfp4)
 * run for M rows and N output columns on the current device: 0 = the split-K
 * cluster kernel (M <= 128 and 2 * ceil(N/64) <= #SMs), 1 = the wide kernel
 * with one 128-row block per CTA, 2 = the wide kernel with two (M > 128 and
 * ceil(M/256) * ceil(N/128) >= 0.9 * #SMs).  -1 for negative sizes.
 * Host-only (GB300's 152 SMs when no device is visible). */
int swiglu_select_weight_kernel(int64_t M, int64_t N);

/* Forces the kernel of the weight-format entry points for later calls
 * (process-wide): 0, 1 or 2 as swiglu_select_weight_kernel numbers them, or
 * -1 (the default) for the library's choice by shape.  For sweeps and tests;
 * swiglu_select_weight_kernel reports the forced kernel while one is set.
 * Returns SWIGLU_ERR_INVALID_ARG for other values. */
int swiglu_set_weight_kernel(int32_t kernel);

/* Tile schedule of the CTA-pair kernels (process-wide) when a call has more
 * work units (output tiles, times K slices) than pairs fit on the device:
 * 1 (the default) = dynamic: the grid holds one 2-CTA cluster per unit and
 * every running pair, after its own unit, cancels clusters that have not
 * started (cluster launch control) and computes their units, so units run in
 * about launch order and tiles that share A rows and weight columns meet in
 * L2; 0 = static: one wave of pairs, pair c computing units c, c + pairs, ...
 * Results are identical.  For comparisons and tests; returns
 * SWIGLU_ERR_INVALID_ARG for other values. */
int swiglu_set_pair_schedule(int32_t dynamic);

/* Short name of a variant ("1sm_n128", ...); "?" for an unknown value. */
const char *swiglu_variant_name(int32_t variant);

/* Human-readable text of a status code. */
const char *swiglu_status_string(int32_t status);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns SWIGLU_OK, SWIGLU_ERR_TIMEOUT if a kernel gave up a wait since
 * the last call (its CTA stopped early, so that launch's Y is incomplete), or
 * SWIGLU_ERR_CUDA if the synchronisation itself failed.  If `detail` is not
 * NULL it receives a code naming the wait that gave up (0 if none).
 * While a timeout stays recorded (until this call clears it), launches of the
 * CTA-pair kernel that run more than one wave of tiles skip their work, so a
 * kernel that keeps timing out ends within about one time limit instead of
 * one per wave; read the status after any call whose result matters.
 */
int swiglu_device_status(void *stream, uint32_t *detail);

/* Time limit of every device-side wait, in nanoseconds (default 2e9, i.e. two
 * seconds; minimum 1e6).  Applies to launches enqueued after the call. */
int swiglu_set_wait_timeout_ns(uint64_t ns);

/*
 * Promise about the weights of later calls (default 0 = no promise).  With
 * on = 1 the caller guarantees that no work enqueued on a stream before a
 * call writes that call's weight matrices (true of model parameters loaded
 * once); the BF16 kernels may then start loading the weights of their first
 * K steps while the preceding kernel on the stream is still finishing
 * (programmatic dependent launch), and load A and write Y only after it has
 * completed.  With on = 0 every load waits for the preceding kernel.  A call
 * that breaks the promise may read stale weights.  Process-wide; applies to
 * calls made after it.  Returns SWIGLU_ERR_INVALID_ARG unless on is 0 or 1.
 */
int swiglu_set_weights_read_only(int32_t on);

/*
 * Failure-detection self test: enqueues one small kernel whose single wait
 * is on a barrier that nothing ever completes, with a limit of `timeout_us`
 * microseconds (1..10^6).  The kernel gives up, records SWIGLU_ERR_TIMEOUT in
 * the device error word and returns normally; the context stays usable.  Read
 * the result with swiglu_device_status().
 */
int swiglu_selftest_wait_timeout(uint32_t timeout_us, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SWIGLU_GB300_H */
