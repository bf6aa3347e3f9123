// Internal declarations shared by the library's translation units (host side).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mmq.h"

namespace mmq {

// Programmatic dependent launch for the kernels that support it (the q8_1
// prepass and the few-token GEMMs): off unless mmq_set_programmatic_launch
// turned it on.
bool programmatic_launch_enabled();

// Launch configuration with the programmatic-dependent-launch attribute
// when it is enabled; attr must have room for it (numAttrs 0 or 1 on return,
// more may be appended by the caller).
inline cudaLaunchConfig_t launch_config(dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                        cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 0;
    if (programmatic_launch_enabled()) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 1;
    }
    return cfg;
}

// Per-device status word (a __device__ int defined in api.cu); kernels get
// its address as an argument and set it to an MMQ_ERR_* code on failure.
int* status_word_ptr();   // nullptr on failure (sets no error)

// Launchers (defined in the kernel translation units).  Arguments are
// already validated; they return cudaGetLastError() of the launch.
cudaError_t launch_quantize_q8_1(const float* x, int64_t M, int64_t K,
                                 mmq_q8_1_t aq, cudaStream_t s);
cudaError_t launch_gemm_mma_s8(mmq_q8_1_t aq, const uint8_t* w, float* C,
                               int32_t* S, int64_t M, int64_t N, int64_t K,
                               int* status, cudaStream_t s);
int tc_gemm_check_resources();   // MMQ_OK or MMQ_ERR_RESOURCE
// q8out.qs == nullptr: no q8_1 output; C == nullptr: no f32 output.
// swiglu: the N weight rows alternate gate / up; q8out receives the [M][N/2]
// q8_1 of silu(gate) * up and C (may be null) the same values in f32.
// S != nullptr: write the per-chunk dots instead of C (dump_scaled: S' = sc*S
// from the product's weight operand; otherwise S with sc left out).
cudaError_t launch_gemm_tc(mmq_q8_1_t aq, const uint8_t* w, float* C, mmq_q8_1_t q8out,
                           int32_t* S, int64_t M, int64_t N, int64_t K,
                           int* status, int inject_timeout, cudaStream_t s, bool swiglu = false,
                           bool dump_scaled = false);
// The tensor-core operand plane of M x K activations (written by the
// prepass's tensor-core form, read by the super-block GEMM): byte offsets of
// its three parts, each 256-byte aligned.
//   a   fp16 [M][K/32][64]  per 32-k chunk 32 values q * s_hi, then 32 values
//       fp16(q * s_lo), each in k order 0,2,1,3 per group of four (one
//       128-byte line per token row and chunk)
//   t2  f32 [M][K/256][32]  second-term factors [hi x8 | hi x8 | lo x8 | 0 x8]
//   g   f32 [M][K/256]  2^E of each token row and super-block
struct TcopLayout {
    size_t a, t2, g, bytes;
};
inline TcopLayout tcop_layout(int64_t M, int64_t K) {
    auto up = [](size_t b) { return (b + 255) & ~size_t(255); };
    TcopLayout L;
    const size_t n = size_t(M) * size_t(K), nsb = size_t(M) * size_t(K / 256);
    L.a = 0;
    L.t2 = up(4 * n);
    L.g = L.t2 + up(nsb * 128);
    L.bytes = L.g + up(nsb * 4);
    return L;
}
cudaError_t launch_quantize_q8_1_tcop(const float* x, int64_t M, int64_t K, mmq_q8_1_t aq, void* tcop,
                                      cudaStream_t s);
// The super-block-accumulating GEMM on the operand plane (gemm_sb.cu): C only.
int sb_gemm_check_resources();   // MMQ_OK or MMQ_ERR_RESOURCE
cudaError_t launch_gemm_sb(const void* tcop, const uint8_t* w, float* C, int64_t M, int64_t N, int64_t K,
                           int* status, int inject_timeout, cudaStream_t s);
// The tcgen05 kernel's launch plan for one call (gemm_tc.cu): tiles
// [0, tail_lo) in the first launch (persistent, or K split over clusters of
// first_split CTAs), tiles [tail_lo, tiles) in a second launch with K split
// over clusters of tail_split CTAs.
struct TcPlan {
    int64_t tiles = 0;
    int first_split = 1;
    int64_t tail_lo = 0;
    int tail_split = 1;
};
TcPlan tc_plan(int64_t M, int64_t N, int64_t K, int nsm, bool allow_tail);
int tc_gemm_launch_count(int64_t M, int64_t N, int64_t K);   // kernels per call, -1 on a CUDA error
// mode 0: C only; 1: also q8_1 into `out` (C may be null); 2: gate/up rows
// interleaved, q8_1 of silu(g)*u into `out` [M][N/2] and, if C is not null,
// h as f32 [M][N/2] into C; 3: the exact per-chunk dots into S [M][N][K/32]
// (C and out unused) from the same kernel the shape selects.
cudaError_t launch_gemm_small_m(mmq_q8_1_t aq, const uint8_t* w, float* C,
                                int64_t M, int64_t N, int64_t K, int* status,
                                cudaStream_t s, mmq_q8_1_t out = mmq_q8_1_t{nullptr, nullptr, nullptr},
                                int mode = 0, int32_t* S = nullptr);
constexpr int kSmallDump = 3;
// Test hook of the dot-product kernel: force its K split (0, 1, 2, 4) for the
// calling host thread; MMQ_ERR_ARG for other values.
int set_force_gemv_split(int ks);
int forced_gemv_split();   // this host thread's forced split, 0 for none
// Host-buffer pipeline (host_pipeline.cu): rows per chunk, workspace bytes,
// and the chunked copy-in / prepass + GEMM / copy-out, with `gemm` the GEMM
// to run on each chunk's q8_1 planes (MMQ_* code).
using GemmFn = int (*)(mmq_q8_1_t aq, const uint8_t* w, float* C, int64_t M, int64_t N, int64_t K,
                       cudaStream_t s);
int64_t host_chunk_rows(int64_t M);
size_t host_workspace_bytes(int64_t M, int64_t N, int64_t K);
int gemm_host(const float* x_host, const uint8_t* w, float* C_host, int64_t M, int64_t N, int64_t K, void* ws,
              cudaStream_t s, GemmFn gemm);
// Device address of the fixed workspace behind mmq_q4K_gemm_host_noalloc
// (MMQ_HOST_NOALLOC_SCRATCH_BYTES, 256-byte aligned) on the current device,
// looked up on the first call per device: MMQ_OK, MMQ_ERR_DEVICE or
// MMQ_ERR_CUDA.
int host_noalloc_scratch(void** out);
// The dp4a GEMV (M <= 4) that also writes its result as q8_1 (N % 32 == 0;
// C may be null).
cudaError_t launch_gemv_q8_1(mmq_q8_1_t aq, const uint8_t* w, float* C, mmq_q8_1_t out, int64_t M, int64_t N,
                             int64_t K, cudaStream_t s);
// The same kernel with the SwiGLU epilogue: rows interleaved gate/up (N = 2F,
// F % 32 == 0), q8_1 of silu(g)*u into out [M][F], h as f32 into hf if not null.
cudaError_t launch_gemv_swiglu_q8_1(mmq_q8_1_t aq, const uint8_t* w_gu, float* hf, mmq_q8_1_t out, int64_t M,
                                    int64_t F, int64_t K, cudaStream_t s);
// The dequantize-then-dense control path (dense.cu).
cudaError_t launch_dequantize_q4K_f16(const uint8_t* w, uint16_t* out, int64_t N, int64_t K,
                                      cudaStream_t s);
cudaError_t launch_convert_f16(const float* x, uint16_t* out, int64_t n, cudaStream_t s);
int dense_gemm_check_resources();   // MMQ_OK or MMQ_ERR_RESOURCE
cudaError_t launch_gemm_f16(const uint16_t* A, const uint16_t* B, float* C, int64_t M, int64_t N,
                            int64_t K, int* status, cudaStream_t s);
// q6_K x q8_1 (gemm_q6k.cu): S != nullptr dumps the per-16 dots instead of C.
cudaError_t launch_repack_q6K(const uint8_t* src, uint8_t* dst, int64_t N, int64_t K, cudaStream_t s);
// allow_gemv: M <= 16 (C only) takes the dp4a dot-product kernel; false forces
// the mma.sync tile kernel.
cudaError_t launch_gemm_q6k(mmq_q8_1_t aq, const uint8_t* w, float* C, int32_t* S, int64_t M,
                            int64_t N, int64_t K, cudaStream_t s, bool allow_gemv = true);
constexpr int64_t kQ6GemvMax = 16;
// q6_K on tcgen05 (gemm_q6k_tc.cu): C only, the same 128 x 128 tile plan as
// the q4_K kernel (tc_plan), one or two kernels per call.
int q6k_tc_check_resources();   // MMQ_OK or MMQ_ERR_RESOURCE
int q6k_tc_launch_count(int64_t M, int64_t N, int64_t K);
// S != nullptr: the exact per-chunk S' = sum a * sc * q (int32 [M][N][K/32])
// instead of C, from the same operands and MMAs.
cudaError_t launch_gemm_q6k_tc(mmq_q8_1_t aq, const uint8_t* w, float* C, int32_t* S, int64_t M, int64_t N,
                               int64_t K, int* status, int inject_timeout, cudaStream_t s);
int small_m_launch_count(int64_t M, int64_t N, int64_t K);   // kernels per call, -1 on a CUDA error
constexpr int64_t kSmallMMax = 64;

}  // namespace mmq
