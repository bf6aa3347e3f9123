/*
 * mmq.h -- C ABI of the GB300 (sm_103a) q4_K-weight x q8_1-activation
 * quantized GEMM ("MMQ") used in LLM prefill.
 *
 * The operation (web page "20 . r15 -- f32-accumulate mma probe (dead end) +
 * rank-1 term2 rescale", section 2.1 "Where the two-term rescale comes
 * from"): activations are quantized per 32 elements to q8_1 (scale da,
 * int8 quants, integer block sum sa); weights are q4_K (256-element
 * super-blocks with fp16 d and dmin, eight 32-element sub-blocks with 6-bit
 * sc and m, 4-bit quants v).  For every 32-k chunk c,
 *     C_ij += da_ic * dsv_jc * S_ijc + dmv_jc * (da_ic * sa_ic)
 * where S_ijc = sum_k a_int[i,k] * v[j,k] exactly, dsv = d*sc and
 * dmv = -dmin*m.  The row factor dma = da*sa is formed once per token row
 * and chunk (the rank-1 fold: page "21 . r16 -- Narrow kernel gets the
 * rank-1 fold", section 2.1).
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers unless the parameter name ends in _host.
 *    All buffers are owned and allocated by the caller; the library
 *    allocates no device memory per call.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Device work
 *    is enqueued asynchronously on it; argument errors are returned
 *    synchronously before anything is enqueued.
 *  - Return value: 0 on success, a negative MMQ_ERR_* code otherwise
 *    (mmq_strerror gives the text).  Nothing is written on an error return.
 *  - Inputs must be finite; NaN/Inf activations are outside the contract.
 *  - All device pointers must be 16-byte aligned (tensor-memory-access
 *    copies require it).
 */
#ifndef MMQ_H
#define MMQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MMQ_OK 0
#define MMQ_ERR_ARG (-1)            /* null pointer, bad size or value range  */
#define MMQ_ERR_ALIGN (-2)          /* pointer not 16-byte aligned            */
#define MMQ_ERR_DEVICE (-3)         /* current device is not sm_103           */
#define MMQ_ERR_RESOURCE (-4)       /* shared/tensor memory budget exceeded:  */
                                    /* launch refused, no fallback            */
#define MMQ_ERR_CUDA (-5)           /* a CUDA runtime call or launch failed   */
#define MMQ_ERR_DEVICE_TIMEOUT (-6) /* a bounded device-side wait gave up     */

/* q8_1 activations, three planes (page r15 section 2.1: "each 32-element
 * block carrying scale da and the in-block integer sum sa"):
 *   qs  int8    [M][K]     row-major quants, q = round(x / da) in [-127, 127]
 *   da  float   [M][K/32]  per-block scale amax/127 (f32)
 *   sa  int32   [M][K/32]  per-block sum of the 32 quants                  */
typedef struct {
    int8_t* qs;
    float* da;
    int32_t* sa;
} mmq_q8_1_t;

/* Bytes of one buffer holding all three q8_1 planes for an M x K activation
 * (planes 256-byte aligned inside it).  K must be a multiple of 32.
 * Returns 0 for invalid sizes. */
size_t mmq_q8_1_bytes(int64_t M, int64_t K);

/* Carve the three planes out of a buffer of mmq_q8_1_bytes(M, K) bytes
 * (buf must be 256-byte aligned).  Host-only pointer arithmetic. */
int mmq_q8_1_view(void* buf, int64_t M, int64_t K, mmq_q8_1_t* out);

/* q8_1 quantize prepass (page r15 section 2.1; the prepass writes da and sa
 * together, so sa costs no extra pass).  Per token row i and 32-block b:
 *   amax = max |x|;  da = amax / 127 (IEEE f32 division);
 *   if da == 0: all q = 0, sa = 0;
 *   else q_k = clamp(roundf(x_k / da), -127, 127) with IEEE division and
 *        round-half-away-from-zero;  sa = sum q_k.
 * x float [M][K] row-major (device).  M >= 1, K >= 32, K % 32 == 0.
 * Output planes as in mmq_q8_1_t.  Bit-exact against the CPU reference. */
int mmq_quantize_q8_1(const float* x, int64_t M, int64_t K, mmq_q8_1_t aq,
                      void* stream);

/* Bytes of q4_K weights for an N x K matrix: N * (K/256) * 144. */
size_t mmq_q4K_bytes(int64_t N, int64_t K);

/* Host q4_K packer (page r15 section 2.1 fields; customary 144-byte
 * super-block: fp16 d, fp16 dmin, 12 bytes of 6-bit sc/m, 128 bytes of
 * nibbles).  Inputs (host, row-major):
 *   v_host    uint8  [N][K]      quants 0..15
 *   sc_host   uint8  [N][K/32]   sub-block scales 0..63
 *   m_host    uint8  [N][K/32]   sub-block mins 0..63
 *   d_host    uint16 [N][K/256]  fp16 bit patterns of d
 *   dmin_host uint16 [N][K/256]  fp16 bit patterns of dmin
 * out_host: mmq_q4K_bytes(N, K) bytes, row j's super-blocks contiguous.
 * Errors: MMQ_ERR_ARG for null pointers, N < 1, K % 256 != 0 or a field out
 * of range (nothing written). */
int mmq_pack_q4K(const uint8_t* v_host, const uint8_t* sc_host,
                 const uint8_t* m_host, const uint16_t* d_host,
                 const uint16_t* dmin_host, int64_t N, int64_t K,
                 uint8_t* out_host);

/* The GEMM: C[i][j] = sum over 32-k chunks c of
 *     da_ic * dsv_jc * S_ijc + dmv_jc * (da_ic * sa_ic)
 * (page r15 section 2.1, two-term rescale; the per-chunk integer dot S is
 * exact; the rescale is f32 with the rank-1 fold dma = da*sa per token row).
 * aq: q8_1 planes of the M x K activations; bq4k: q4_K bytes of the N x K
 * weights (row j = output feature j); C float [M][N] row-major, overwritten.
 * M >= 1 (any), N >= 1 with N % 4 == 0, K >= 256 with K % 256 == 0.
 * Picks the kernel for the shape (small-M weight-streaming kernel or the
 * large-M tensor-core kernel).  Results agree with the CPU reference within
 * |C - C_ref| <= 1e-4 * sum_k |a_k w_k| + 1e-6 and are bitwise
 * deterministic run to run on one device and build.  The grouping of the
 * f32 partial sums (K split, clusters) is chosen from the shape and the
 * device's SM count and occupancy, so the last bits of C may differ between
 * devices or builds; the tolerance is the contract across them. */
int mmq_q4K_gemm(mmq_q8_1_t aq, const uint8_t* bq4k, float* C, int64_t M,
                 int64_t N, int64_t K, void* stream);


/* Device workspace bytes for mmq_q4K_gemm_host on an M x K by N x K problem
 * (0 for shapes mmq_q4K_gemm refuses).  It holds two chunks of x, one chunk
 * of q8_1 planes and two chunks of C, a chunk being up to a quarter of the
 * rows rounded up to 128 (all rows when M <= 256). */
size_t mmq_q4K_gemm_host_workspace(int64_t M, int64_t N, int64_t K);

/* The prepass and the GEMM (page r15 section 2.1, as mmq_quantize_q8_1 then
 * mmq_q4K_gemm) with the activations and the result in HOST memory:
 * x_host float [M][K] and C_host float [M][N] row-major, weights bq4k on the
 * device.  The rows are processed in chunks.  Chunk i+1's host-to-device
 * copy, chunk i's prepass and GEMM (on `stream`) and chunk i-1's
 * device-to-host copy run concurrently, on two copy streams the library
 * keeps per device, ordered by events.  Page-locked host memory
 * (cudaHostAlloc) lets the copies overlap; pageable memory works but does
 * not overlap.  The copies start after the work already queued on `stream`,
 * and work queued on `stream` afterwards runs after the last copy, so
 * synchronizing `stream` makes C_host valid.  workspace: device memory of
 * mmq_q4K_gemm_host_workspace(M, N, K) bytes or more, 256-byte aligned,
 * caller-owned, not used by anything else until `stream` passes this call.
 * Per chunk the kernel is the one mmq_q4K_gemm picks for the chunk's rows,
 * so C equals mmq_q4K_gemm applied chunk by chunk, within the GEMM's
 * tolerance of the whole.  Errors: MMQ_ERR_ARG (null pointer, shape, small
 * workspace), MMQ_ERR_ALIGN, MMQ_ERR_DEVICE, MMQ_ERR_CUDA. */
int mmq_q4K_gemm_host(const float* x_host, const uint8_t* bq4k, float* C_host,
                      int64_t M, int64_t N, int64_t K, void* workspace,
                      size_t workspace_bytes, void* stream);

/* Size of the fixed device array behind mmq_q4K_gemm_host_noalloc: 64 MiB. */
#define MMQ_HOST_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/* mmq_q4K_gemm_host without a workspace argument.  The pages have no
 * counterpart: this entry point serves callers that hold the activations in
 * host memory but cannot hand the library device memory, for example code
 * that reaches the GPU only through this C ABI (a foreign-function caller
 * with no CUDA bindings, so no way to obtain a device pointer), or a plug-in
 * in a process whose memory pool has reserved the device's memory, where a
 * cudaMalloc of its own would fail or break that reservation (and could
 * synchronize the device on the way).
 *
 * The workspace is a file-scope device array of MMQ_HOST_NOALLOC_SCRATCH_BYTES
 * inside the library; every device on which the library's code is loaded
 * holds it until the process exits.  The call allocates no device memory
 * (no cudaMalloc or cudaFree, no allocating library routine).  The first
 * call on a device looks up the array's device address (and, as
 * mmq_q4K_gemm_host does, creates the library's two copy streams for that
 * device); make that first call before any stream capture on the device.
 *
 * Arguments, results and errors are those of mmq_q4K_gemm_host (the same
 * chunked copies and kernels, so C is what mmq_q4K_gemm_host gives),
 * except: a shape whose mmq_q4K_gemm_host_workspace(M, N, K) exceeds
 * MMQ_HOST_NOALLOC_SCRATCH_BYTES is refused with MMQ_ERR_ARG before any
 * device work (e.g. M = 2048, K = N = 4096 needs 36 MB and fits; the
 * 2048 x 11008 -> 4096 down projection needs 69 MB and does not).
 *
 * Every call uses the same array, and it keeps whatever the last call left
 * there; each call overwrites every byte it reads (nothing in it has to
 * start at zero).  Calls on one stream run one after another; calls whose
 * device work can overlap (different streams not ordered by events, or
 * several host threads) race on the array and give wrong results. */
int mmq_q4K_gemm_host_noalloc(const float* x_host, const uint8_t* bq4k,
                              float* C_host, int64_t M, int64_t N, int64_t K,
                              void* stream);

/* Kernel selection for mmq_q4K_gemm_path (testing and A/B timing).  The
 * values 4 and 5 are retired (two tensor-core variants that no shape ever
 * selected) and are refused like any unknown value. */
#define MMQ_PATH_AUTO 0
#define MMQ_PATH_MMA_S8 1   /* warp-level mma.sync s8 x s8 -> s32 kernel    */
#define MMQ_PATH_TC 2       /* tcgen05 kernel (exact integers in fp16, f32   */
                            /* accumulation in tensor memory)               */
#define MMQ_PATH_SMALL_M 3  /* weight-streaming kernels for few tokens:     */
                            /* dp4a dot products for M <= 4, mma.sync f16   */
                            /* with cluster split-K for 4 < M <= 64         */

/* ---- the tensor-core operand plane (GB300 fast path for many tokens) ----
 *
 * The pages' rescale multiplies each 32-k chunk's integer dot by its own
 * activation scale da (page r15 section 2.1), which on the tensor cores
 * means a round trip through tensor memory per chunk.  The operand plane
 * carries that scale inside the activation operand instead, so that one
 * accumulator can hold a whole 256-k super-block:
 *   per token row i and super-block b, g_ib = 2^E (E from the largest da of
 *   the block's eight chunks) and s = da * 2^-E (exact); per element
 *   hi = q * s_hi with s_hi = s rounded to 4 significant bits (an exact
 *   fp16 product) and lo = fp16(q * fp16(s - s_hi)), so hi + lo is within
 *   2^-14 of q * s; and the second term's factors dma * 2^-E (dma = da *
 *   sa, page r16 section 2.1) split into tf32 hi + lo.
 * The plane is a device-only encoding of the q8_1 values (its bytes are
 * defined by the prepass below and read only by mmq_q4K_gemm_tcop): a
 * single caller-owned buffer of mmq_q8_1_tcop_bytes(M, K) bytes, 256-byte
 * aligned. */

/* Bytes of the operand plane of M x K activations (K % 256 == 0); 0 for an
 * invalid shape. */
size_t mmq_q8_1_tcop_bytes(int64_t M, int64_t K);

/* The q8_1 prepass (exactly as mmq_quantize_q8_1: `aq` receives the same
 * bits) that also writes the operand plane `tcop` (device memory,
 * mmq_q8_1_tcop_bytes(M, K) bytes, 256-byte aligned).  K % 256 == 0.
 * MMQ_ERR_ARG / MMQ_ERR_ALIGN / MMQ_ERR_DEVICE / MMQ_ERR_CUDA as
 * mmq_quantize_q8_1. */
int mmq_quantize_q8_1_tcop(const float* x, int64_t M, int64_t K, mmq_q8_1_t aq,
                           void* tcop, void* stream);

/* C[M][N] (f32, overwritten) = the q4_K x q8_1 GEMM of the activations whose
 * operand plane `tcop` mmq_quantize_q8_1_tcop wrote, on the tcgen05 kernel
 * that accumulates whole super-blocks (128 x 256 tiles, one CTA per SM).
 * The result meets the GEMM's tolerance |C - C_ref| <= 1e-4 sum|a w| + 1e-6
 * (the plane's 2^-14 and f32 accumulation stay far inside it) but the
 * per-chunk integer dots S are never formed: mmq_q4K_block_dots covers the
 * other kernels.  Shape and alignment rules as mmq_q4K_gemm; the result
 * does not depend on the stream or on earlier calls (deterministic). */
int mmq_q4K_gemm_tcop(const void* tcop, const uint8_t* bq4k, float* C, int64_t M,
                      int64_t N, int64_t K, void* stream);

/* Number of kernels mmq_q4K_gemm_path(…, path, …) enqueues for this shape
 * on the current device: 1, or 2 when the tcgen05 kernel or the 5-64 token
 * kernel splits off its last partial round of tiles into a second, split-K
 * launch.  For counting
 * launches (e.g. in a timed region); MMQ_ERR_ARG for a shape or path the
 * GEMM refuses, MMQ_ERR_DEVICE / MMQ_ERR_CUDA as the GEMM would. */
int mmq_q4K_gemm_launches(int64_t M, int64_t N, int64_t K, int path);

/* Same as mmq_q4K_gemm with an explicit kernel.  MMQ_ERR_ARG if `path` is
 * unknown or the kernel does not accept the shape (the small-M kernel takes
 * M <= 64).  The automatic choice: M <= 64 -> small-M, else the one-CTA
 * tcgen05 kernel (which splits K over a cluster when tiles are few). */
int mmq_q4K_gemm_path(mmq_q8_1_t aq, const uint8_t* bq4k, float* C, int64_t M,
                      int64_t N, int64_t K, int path, void* stream);

/* The GEMM with its output also quantized to q8_1, so that a following GEMM
 * needs no separate prepass: `out` describes an [M][N] q8_1 buffer
 * (mmq_q8_1_bytes(M, N); N % 32 == 0) and receives exactly what
 * mmq_quantize_q8_1 would produce from the f32 result (per 32 output
 * columns: da = amax/127, q = roundf(c/da) clamped to +-127, sa = sum q).
 * Every kernel quantizes in its epilogue and C may be NULL (then no f32
 * result is stored): the tcgen05 kernel for M > 64; for M <= 64 the
 * few-token kernels, whose CTA (or cluster of CTAs, for the dot-product
 * kernel at M <= 4) covers whole 32-column output blocks.
 * Otherwise as mmq_q4K_gemm (same argument rules and error codes). */
int mmq_q4K_gemm_q8_1(mmq_q8_1_t aq, const uint8_t* bq4k, float* C, mmq_q8_1_t out,
                      int64_t M, int64_t N, int64_t K, void* stream);

/* The gate and up projections of a SwiGLU FFN block in one GEMM, with the
 * activation and the q8_1 quantization of its output in the epilogue, so
 * that the down projection gets its q8_1 input with no separate pass (the
 * fused-neighbour idea of page r12's prepass/transpose work).  bq4k_gu holds
 * the q4_K bytes of a 2F x K matrix whose rows alternate gate row f and up
 * row f (mmq_interleave_rows_q4K builds it once, at load time).  With g, u
 * the two GEMM results (the same arithmetic as mmq_q4K_gemm), the output is
 *     h = silu(g) * u = g / (1 + exp(-g)) * u           (f32, IEEE ops)
 * quantized to q8_1 exactly as mmq_quantize_q8_1 would quantize h: `out`
 * describes an [M][F] q8_1 buffer.  hf (may be NULL) receives h, f32
 * [M][F].  F % 32 == 0; other rules as mmq_q4K_gemm (N = 2F).  Runs the
 * tcgen05 kernel for M > 64 and the few-token kernels (dot-product for
 * M <= 4, mma.sync for M <= 64) below, each with the SwiGLU epilogue. */
int mmq_q4K_gemm_swiglu_q8_1(mmq_q8_1_t aq, const uint8_t* bq4k_gu, float* hf,
                             mmq_q8_1_t out, int64_t M, int64_t F, int64_t K,
                             void* stream);

/* out = the rows of gate and up (q4_K bytes, F x K each) interleaved: row 2f
 * of out is gate row f, row 2f + 1 up row f.  Any mix of host and device
 * pointers (two strided copies on `stream`); out is 2 * F * (K/256) * 144
 * bytes. */
int mmq_interleave_rows_q4K(const uint8_t* gate, const uint8_t* up, uint8_t* out,
                            int64_t F, int64_t K, void* stream);

/* Debug/test dump of the exact per-chunk integer dots (page r15 section 2.1:
 * S_ij = sum_k a_int[i,k] * v[j,k]; section 2.3: |S| <= 32*127*15) computed
 * by the same unpack and MMA (or dp4a) code as the GEMM kernel selected by
 * `path`: MMQ_PATH_MMA_S8, MMQ_PATH_TC, MMQ_PATH_SMALL_M (M <= 64: the
 * dot-product kernel for M <= 4, the mma.sync kernel above) or
 * MMQ_PATH_AUTO (the kernel mmq_q4K_gemm picks for M).  S int32
 * [M][N][K/32].  Same shape rules as the GEMM. */
int mmq_q4K_block_dots(mmq_q8_1_t aq, const uint8_t* bq4k, int32_t* S,
                       int64_t M, int64_t N, int64_t K, int path, void* stream);

/* The tcgen05 kernel (MMQ_PATH_TC) folds the 6-bit sub-block scale into its
 * weight operand, so its tensor cores form S'_ijc = sc_jc * S_ijc exactly
 * (|S'| <= 32*127*63*15 < 2^22; page r15 section 2.1 for S and sc).  This
 * dump returns S' int32 [M][N][K/32] from that kernel run on its product
 * operand, unchanged except that the epilogue writes S' instead of
 * rescaling it.  Shape rules as the GEMM. */
int mmq_q4K_scaled_block_dots(mmq_q8_1_t aq, const uint8_t* bq4k, int32_t* S,
                              int64_t M, int64_t N, int64_t K, void* stream);

/* ---- The dequantize-then-dense control path (the f16 GEMM path the pages
 * measure MMQ against: page r12, the landing note comparing MMQ with the f16
 * default GEMM path; its dequantize step a bandwidth kernel as audited on
 * page "Round 31 Track C Audit: dq_f16 (dense_mm.metal) & DW<F>
 * (mma.metal)", section 2.1).  fp16 values travel as their uint16_t bits. */

/* q4_K weights -> fp16, row-major [N][K] (caller-owned, N*K*2 bytes): element
 * k of sub-block c of a super-block is fp16(f32(d*sc_c*v_k - dmin*m_c)), the
 * difference rounded once to f32 (both products are exact in f32) and then
 * to fp16, round to nearest even both times.  N >= 1, K % 256 == 0;
 * pointers 16-byte aligned.  Bit-for-bit reproducible. */
int mmq_dequantize_q4K_f16(const uint8_t* bq4k, uint16_t* wh, int64_t N,
                           int64_t K, void* stream);

/* x float[n] -> fp16 (round to nearest even); n % 4 == 0, pointers 16-byte
 * aligned. */
int mmq_convert_f32_f16(const float* x, uint16_t* xh, int64_t n, void* stream);

/* Dense C[M][N] = A[M][K] . B[N][K]^T with fp16 A, B (row-major, K
 * contiguous) and f32 C (row-major, overwritten), on the tcgen05 tensor cores
 * with f32 accumulation.  M, N >= 1, N % 4 == 0, K % 64 == 0; pointers
 * 16-byte aligned.  Each C value is the sum of K exact products accumulated
 * in f32; results are bitwise deterministic run to run.  MMQ_ERR_RESOURCE if
 * the device's shared memory per block is too small. */
int mmq_gemm_f16(const uint16_t* A, const uint16_t* B, float* C, int64_t M,
                 int64_t N, int64_t K, void* stream);

/* ---- q6_K weights (the family the pages' MMQ line moved to next: page r15,
 * "Proof of pattern portability").  The pages print no layout; this library
 * takes the customary 210-byte super-block of 256 weights: ql[128] (low
 * nibbles), qh[64] (high bit pairs), int8 scales[16] (one per 16 weights),
 * fp16 d.  Quant q in [-32, 31] is stored as u = q + 32; element
 * 128n + 32r + l (n < 2, r < 4, l < 32) keeps the low 4 bits of u in nibble
 * r/2 of ql[64n + 32(r%2) + l] and the top 2 bits in bits 2r, 2r+1 of
 * qh[32n + l].  The weight is d * sc * q (no minimum term). */

/* Bytes of the customary layout (0 if N < 1 or K % 256 != 0). */
size_t mmq_q6K_bytes(int64_t N, int64_t K);

/* Host packer: q int8 [N][K] in [-32, 31], sc int8 [N][K/16], d fp16 bits
 * [N][K/256] -> mmq_q6K_bytes(N, K) bytes, row j's super-blocks contiguous.
 * MMQ_ERR_ARG on a quant out of range. */
int mmq_pack_q6K(const int8_t* q_host, const int8_t* sc_host, const uint16_t* d_host,
                 int64_t N, int64_t K, uint8_t* out_host);

/* Bytes of the device layout the q6_K GEMM reads: each super-block padded to
 * 224 bytes (14 zero bytes after d), so that rows are whole 16-byte pieces. */
size_t mmq_q6K_dev_bytes(int64_t N, int64_t K);

/* Customary layout (device memory, any alignment) -> device layout (dst
 * 16-byte aligned), once at load time. */
int mmq_repack_q6K(const uint8_t* src, uint8_t* dst, int64_t N, int64_t K, void* stream);

/* C = A . W^T for q8_1 activations and q6_K weights in the device layout:
 * per 16-weight sub-block s of the 32-element q8_1 block c,
 * C_ij += da_ic * d_j * sc_js * S_ijs with S the exact int32 dot.  M <= 16:
 * dp4a dot products streaming the weights; above that the tcgen05 kernel
 * (MMQ_PATH_TC below).  Shape rules and tolerance as mmq_q4K_gemm. */
int mmq_q6K_gemm(mmq_q8_1_t aq, const uint8_t* bq6k_dev, float* C, int64_t M,
                 int64_t N, int64_t K, void* stream);

/* The same with an explicit kernel family, for tests and A/B timing:
 *   MMQ_PATH_SMALL_M  the dp4a dot-product kernel (M <= 16, else MMQ_ERR_ARG);
 *   MMQ_PATH_MMA_S8   warp-level int8 mma.sync on 128 x 128 tiles, K split
 *                     over a cluster when the tiles are few;
 *   MMQ_PATH_TC       tcgen05: per 32-k chunk the exact S' = sum a * sc * q
 *                     in f32 tensor memory from fp16 operands (sc * q split
 *                     into an fp16 hi part and an exact lo part, both MMA'd),
 *                     then C += da * d * S' (page r15, "Proof of pattern
 *                     portability", for the family); persistent 128 x 128
 *                     tiles as the q4_K kernel, up to two kernels per call;
 *                     MMQ_ERR_RESOURCE if the shared-memory budget is missing;
 *   MMQ_PATH_AUTO     what mmq_q6K_gemm runs.
 * Errors as mmq_q4K_gemm_path. */
int mmq_q6K_gemm_path(mmq_q8_1_t aq, const uint8_t* bq6k_dev, float* C, int64_t M,
                      int64_t N, int64_t K, int path, void* stream);

/* The tcgen05 q6_K kernel's exact per-chunk dots from its own operands:
 * S int32 [M][N][K/32], S_ijc = sum over the chunk's two 16-weight
 * sub-blocks s of sc_js * S16_ijs (the products a * sc * q summed exactly;
 * |S| <= 32 * 127 * 4096 < 2^24).  Shape rules and errors as mmq_q6K_gemm. */
int mmq_q6K_scaled_block_dots(mmq_q8_1_t aq, const uint8_t* bq6k_dev, int32_t* S,
                              int64_t M, int64_t N, int64_t K, void* stream);

/* Kernels one mmq_q6K_gemm_path call enqueues for this shape: 1 or 2;
 * MMQ_ERR_ARG / MMQ_ERR_CUDA as mmq_q4K_gemm_launches. */
int mmq_q6K_gemm_launches(int64_t M, int64_t N, int64_t K, int path);

/* The exact per-16 dots S int32 [M][N][K/16] from the mma.sync tile kernel's
 * unpack and MMA code. */
int mmq_q6K_block_dots(mmq_q8_1_t aq, const uint8_t* bq6k_dev, int32_t* S,
                       int64_t M, int64_t N, int64_t K, void* stream);

/* ---- GGUF interop (host).  Reads and writes the tensors of GGUF files
 * (versions 2 and 3, little endian), the file format the customary q4_K /
 * q6_K super-block layouts come from.  Files are untrusted input: every
 * length and offset is checked against the file size; a file that does not
 * parse gives MMQ_ERR_ARG.  Tensor types (GGUF numbering): */
#define MMQ_GGUF_F32 0
#define MMQ_GGUF_F16 1
#define MMQ_GGUF_Q4_K 12
#define MMQ_GGUF_Q6_K 14
typedef struct mmq_gguf mmq_gguf;

/* Parse the header and tensor table of `path`; *out owns the open file
 * until mmq_gguf_close.  Tensors of other types are listed with nbytes 0. */
int mmq_gguf_open(const char* path, mmq_gguf** out);
void mmq_gguf_close(mmq_gguf* h);
int64_t mmq_gguf_tensor_count(const mmq_gguf* h);
/* Index of the tensor called `name`, or -1. */
int mmq_gguf_find(const mmq_gguf* h, const char* name);
/* Name (truncated to name_cap - 1 bytes, NUL-terminated), type, number of
 * dims and dims (dims4[0] the contiguous one; unused entries 1) and the
 * byte size of tensor i (0 if its type is not one of the four above). */
int mmq_gguf_tensor_info(const mmq_gguf* h, int64_t i, char* name, size_t name_cap,
                         uint32_t* type, uint32_t* ndim, int64_t* dims4, uint64_t* nbytes);
/* Copy tensor i's bytes into host memory (cap >= its nbytes). */
int mmq_gguf_read(mmq_gguf* h, int64_t i, void* dst_host, uint64_t cap);
/* Write n two-dimensional tensors (dims2[2i] the contiguous dim, dims2[2i+1]
 * the rows) with general.alignment = 32.  For q4_K / q6_K the bytes are the
 * customary super-blocks (mmq_pack_q4K / mmq_pack_q6K output). */
int mmq_gguf_write(const char* path, int64_t n, const char* const* names,
                   const uint32_t* types, const int64_t* dims2, const void* const* data);

/* Synchronizes `stream`, then returns and clears the current device's status
 * word: MMQ_OK, or MMQ_ERR_DEVICE_TIMEOUT if a kernel's bounded wait gave up
 * since the last call (that kernel's output is then invalid), or
 * MMQ_ERR_CUDA if the synchronization itself failed. */
int mmq_status(void* stream);

/* Static text for an MMQ_* code. */
const char* mmq_strerror(int code);

/* Programmatic dependent launch (process-wide, default off): when enabled,
 * the q8_1 prepass and the GEMM kernels (few-token and tcgen05) are launched
 * so that each may start while the previous kernel on its stream finishes.
 * A kernel so launched issues only its weight loads (or, for the tcgen05
 * kernel, only its set-up) before it waits for the previous grid to
 * complete; it reads activations and writes its outputs only after that
 * wait, so results are the same either way.  Hides most of
 * the per-kernel start cost in a decode-style sequence of small GEMMs.
 * While enabled, a GEMM's weights must not be written by the kernel
 * launched just before it on the same stream. */
void mmq_set_programmatic_launch(int enable);

/* Test hook: force the K split of the dot-product kernels (q4_K, M <= 4;
 * q6_K, M <= 16) for later calls on this host thread: ks = 1, 2 or 4 warps
 * per row group (the SwiGLU epilogue takes 1 or 2; a forced 4 makes its
 * calls fail with MMQ_ERR_CUDA), 0 restores the automatic choice.  Returns MMQ_ERR_ARG for
 * any other value.  The split changes how the row's partial sums are
 * grouped, so f32 results may differ in the last bits between splits; the
 * integer dots and the tolerance do not. */
int mmq_debug_force_gemv_split(int ks);

/* Test hook: when nonzero, the next tensor-core GEMM launch on this host
 * thread withholds one producer arrival so that its consumers' bounded
 * waits run out; the kernel then records MMQ_ERR_DEVICE_TIMEOUT and returns
 * without hanging.  Used only to test the failure path. */
void mmq_debug_inject_timeout(int enable);

#ifdef __cplusplus
}
#endif
#endif /* MMQ_H */
