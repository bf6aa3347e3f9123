// Instruction-rate peaks that bench.py reports fractions against and that the
// driver does not measure: the warp-level int8 tensor rate (mma.sync
// m16n8k32 s8 -> s32, the only integer tensor path on sm_103a: tcgen05.mma
// has no integer kind there), the legacy warp-level f16 tensor rate, and the
// FP32 FMA rates (scalar and packed f32x2) that bound a rescale epilogue.
//
// Every SM runs 4 CTAs of 8 warps; each warp issues long chains of
// independent instructions; one launch is timed with CUDA events after a
// warm-up launch.  Prints one JSON object.
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -o bench_peaks bench_peaks.cu && ./bench_peaks
// (python bench.py --measure-peaks does this under _build/.)
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

#define CK(x)                                                                   \
    do {                                                                        \
        cudaError_t e_ = (x);                                                   \
        if (e_ != cudaSuccess) {                                                \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));            \
            return 1;                                                           \
        }                                                                       \
    } while (0)

constexpr int kChains = 8;   // independent accumulators per warp

__global__ void imma_s8_rate(int iters, int* sink) {
    const uint32_t a0 = threadIdx.x, a1 = threadIdx.x * 3u, a2 = threadIdx.x ^ 5u, a3 = 7u;
    const uint32_t b0 = threadIdx.x * 11u, b1 = 13u;
    int c[kChains][4] = {};
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < kChains; ++i)
            asm volatile(
                "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
                "{%8,%9}, {%0,%1,%2,%3};\n"
                : "+r"(c[i][0]), "+r"(c[i][1]), "+r"(c[i][2]), "+r"(c[i][3])
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    int s = 0;
#pragma unroll
    for (int i = 0; i < kChains; ++i) s += c[i][0] ^ c[i][1] ^ c[i][2] ^ c[i][3];
    if (s == 0x12345678) sink[0] = s;   // keeps the chains alive
}

__global__ void hmma_f16_rate(int iters, int* sink) {
    const uint32_t a0 = threadIdx.x, a1 = threadIdx.x * 3u, a2 = threadIdx.x ^ 5u, a3 = 7u;
    const uint32_t b0 = threadIdx.x * 11u, b1 = 13u;
    float c[kChains][4] = {};
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < kChains; ++i)
            asm volatile(
                "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
                "{%8,%9}, {%0,%1,%2,%3};\n"
                : "+f"(c[i][0]), "+f"(c[i][1]), "+f"(c[i][2]), "+f"(c[i][3])
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kChains; ++i) s += c[i][0] + c[i][1] + c[i][2] + c[i][3];
    if (s == 1234.5f) sink[0] = 1;
}

__global__ void ffma_rate(int iters, int* sink) {
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = threadIdx.x * 0.001f + i;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = fmaf(x[i], 0.9999f, 0.0001f);
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) s += x[i];
    if (s == 1234.5f) sink[0] = 1;
}

__global__ void ffma2_rate(int iters, int* sink) {
    uint64_t x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
        x[i] = uint64_t(__float_as_uint(threadIdx.x * 0.001f + i)) | (uint64_t(__float_as_uint(i * 0.5f)) << 32);
    const uint64_t a = uint64_t(__float_as_uint(0.9999f)) | (uint64_t(__float_as_uint(0.9998f)) << 32);
    const uint64_t b = uint64_t(__float_as_uint(0.0001f)) | (uint64_t(__float_as_uint(0.0002f)) << 32);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 16; ++i) asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(x[i]) : "l"(a), "l"(b));
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) s += __uint_as_float(uint32_t(x[i])) + __uint_as_float(uint32_t(x[i] >> 32));
    if (s == 1234.5f) sink[0] = 1;
}

// Milliseconds of one launch of k after a short warm-up launch.
static int time_ms(void (*k)(int, int*), int blocks, int threads, int iters, int* sink, float* ms) {
    cudaEvent_t e0, e1;
    CK(cudaEventCreate(&e0));
    CK(cudaEventCreate(&e1));
    k<<<blocks, threads>>>(iters / 100, sink);
    CK(cudaGetLastError());
    CK(cudaDeviceSynchronize());
    CK(cudaEventRecord(e0));
    k<<<blocks, threads>>>(iters, sink);
    CK(cudaEventRecord(e1));
    CK(cudaEventSynchronize(e1));
    CK(cudaEventElapsedTime(ms, e0, e1));
    CK(cudaEventDestroy(e0));
    CK(cudaEventDestroy(e1));
    return 0;
}

int main() {
    int dev = 0, nsm = 0, clk_khz = 0;
    CK(cudaGetDevice(&dev));
    CK(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev));
    CK(cudaDeviceGetAttribute(&clk_khz, cudaDevAttrClockRate, dev));
    int* sink = nullptr;
    CK(cudaMalloc(&sink, 64));
    const int threads = 256, blocks = nsm * 4, iters = 20000;
    const double warps = double(blocks) * threads / 32, threads_all = double(blocks) * threads;
    float ms = 0.f;
    if (time_ms(imma_s8_rate, blocks, threads, iters, sink, &ms)) return 1;
    const double imma = warps * iters * kChains * (16.0 * 8 * 32) * 2 / (ms * 1e-3) / 1e12;
    if (time_ms(hmma_f16_rate, blocks, threads, iters, sink, &ms)) return 1;
    const double hmma = warps * iters * kChains * (16.0 * 8 * 16) * 2 / (ms * 1e-3) / 1e12;
    if (time_ms(ffma_rate, blocks, threads, iters, sink, &ms)) return 1;
    const double ffma = threads_all * iters * 16 * 2 / (ms * 1e-3) / 1e12;
    if (time_ms(ffma2_rate, blocks, threads, iters, sink, &ms)) return 1;
    const double ffma2 = threads_all * iters * 16 * 4 / (ms * 1e-3) / 1e12;
    CK(cudaFree(sink));
    printf("{\"int8_mma_sync_tops\": %.1f, \"f16_mma_sync_tflops\": %.1f, \"fp32_ffma_tflops\": %.1f, "
           "\"fp32_ffma2_tflops\": %.1f, \"sms\": %d, \"sm_max_mhz\": %d}\n",
           imma, hmma, ffma, ffma2, nsm, clk_khz / 1000);
    return 0;
}
