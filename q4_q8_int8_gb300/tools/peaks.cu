// Peak-rate microbenchmarks for the roofline denominators this library needs
// and the driver does not measure: the warp-level int8 tensor rate
// (mma.sync m16n8k32 s8 -> s32) and the FP32 FMA rates (scalar and f32x2)
// that bound the per-chunk rescale epilogue.  Prints one JSON line.
//
// Each kernel runs long chains of independent instructions per warp on every
// SM; timing is by CUDA events around a single launch after a warm-up.
#include <cuda_runtime.h>
#include <cstdio>
#include <cstdint>

#define CK(x) do { cudaError_t e = (x); if (e != cudaSuccess) { \
    fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e)); return 1; } } while (0)

__global__ void mma_s8_loop(int iters, int* out) {
    uint32_t a[4] = {threadIdx.x, threadIdx.x * 3u, threadIdx.x ^ 5u, 7u};
    uint32_t b0 = threadIdx.x * 11u, b1 = 13u;
    uint32_t c[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int r = 0; r < 4; ++r) c[i][r] = 0;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            asm volatile(
                "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
                "{%8,%9}, {%0,%1,%2,%3};\n"
                : "+r"(c[i][0]), "+r"(c[i][1]), "+r"(c[i][2]), "+r"(c[i][3])
                : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    int s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += c[i][0] + c[i][1] + c[i][2] + c[i][3];
    if (s == 0x12345678) out[0] = s;
}

__global__ void ffma_loop(int iters, float* out) {
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = threadIdx.x * 0.001f + i;
    const float a = 0.9999f, b = 0.0001f;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = fmaf(x[i], a, b);
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) s += x[i];
    if (s == 1234.5f) out[0] = s;
}

__global__ void ffma2_loop(int iters, float* out) {
    unsigned long long x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float2 f = make_float2(threadIdx.x * 0.001f + i, i * 0.5f);
        x[i] = *reinterpret_cast<unsigned long long*>(&f);
    }
    float2 af = make_float2(0.9999f, 0.9998f), bf = make_float2(0.0001f, 0.0002f);
    const unsigned long long a = *reinterpret_cast<unsigned long long*>(&af);
    const unsigned long long b = *reinterpret_cast<unsigned long long*>(&bf);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(x[i]) : "l"(a), "l"(b));
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float2 f = *reinterpret_cast<float2*>(&x[i]);
        s += f.x + f.y;
    }
    if (s == 1234.5f) out[0] = s;
}

int main() {
    int dev = 0, nsm = 0, clk = 0;
    CK(cudaGetDevice(&dev));
    CK(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev));
    CK(cudaDeviceGetAttribute(&clk, cudaDevAttrClockRate, dev));
    int* dout;
    CK(cudaMalloc(&dout, 64));
    cudaEvent_t e0, e1;
    CK(cudaEventCreate(&e0));
    CK(cudaEventCreate(&e1));
    const int threads = 256, blocks = nsm * 4;
    float ms;

    // mma.sync s8: 8 MMAs x iters per warp, 16*8*32 MACs each
    const int it_mma = 20000;
    mma_s8_loop<<<blocks, threads>>>(100, dout);
    CK(cudaDeviceSynchronize());
    CK(cudaEventRecord(e0));
    mma_s8_loop<<<blocks, threads>>>(it_mma, dout);
    CK(cudaEventRecord(e1));
    CK(cudaEventSynchronize(e1));
    CK(cudaEventElapsedTime(&ms, e0, e1));
    const double warps = double(blocks) * threads / 32;
    const double mma_tops = warps * it_mma * 8 * (16.0 * 8 * 32) * 2 / (ms * 1e-3) / 1e12;

    const int it_f = 20000;
    ffma_loop<<<blocks, threads>>>(100, (float*)dout);
    CK(cudaDeviceSynchronize());
    CK(cudaEventRecord(e0));
    ffma_loop<<<blocks, threads>>>(it_f, (float*)dout);
    CK(cudaEventRecord(e1));
    CK(cudaEventSynchronize(e1));
    CK(cudaEventElapsedTime(&ms, e0, e1));
    const double ffma_tflops = double(blocks) * threads * it_f * 16 * 2 / (ms * 1e-3) / 1e12;

    ffma2_loop<<<blocks, threads>>>(100, (float*)dout);
    CK(cudaDeviceSynchronize());
    CK(cudaEventRecord(e0));
    ffma2_loop<<<blocks, threads>>>(it_f, (float*)dout);
    CK(cudaEventRecord(e1));
    CK(cudaEventSynchronize(e1));
    CK(cudaEventElapsedTime(&ms, e0, e1));
    const double ffma2_tflops = double(blocks) * threads * it_f * 16 * 4 / (ms * 1e-3) / 1e12;

    printf("{\"sms\": %d, \"clock_khz_attr\": %d, \"mma_sync_s8_tops\": %.2f, "
           "\"ffma_tflops\": %.2f, \"ffma2_tflops\": %.2f}\n",
           nsm, clk, mma_tops, ffma_tflops, ffma2_tflops);
    return 0;
}
