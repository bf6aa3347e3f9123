// Peak-rate microbenchmarks for the roofline denominators this library needs
// and the driver does not measure: the warp-level int8 tensor rate
// (mma.sync m16n8k32 s8 -> s32) and the FP32 FMA rates (scalar and f32x2)
// that bound the per-chunk rescale epilogue; tensor-memory load rates; and
// the latencies of the tcgen05 GEMM's MMA-issue / mbarrier hand-off chain,
// the issue cost of one tcgen05 MMA by its N, and what an MMA-issuing
// thread's loop of waits, MMAs and commits costs per operand stage.
// Prints JSON lines.
//
// Each kernel runs long chains of independent instructions per warp on every
// SM; timing is by CUDA events around a single launch after a warm-up.
#include <cuda_runtime.h>
#include <cstdio>
#include <cstdint>

#include "../csrc/sm103_ptx.cuh"

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


// ---- tensor-memory load bandwidth: each warp reads its lane quarter of a
// 512-column allocation repeatedly (contents are whatever the allocation
// holds; only the data movement is timed).
template <int kShape, int kInflight>
__global__ void tmem_ld_loop(int iters, unsigned* out) {
    __shared__ unsigned slot;
    const int warp = threadIdx.x >> 5;
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
            (unsigned)__cvta_generic_to_shared(&slot)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    const unsigned base = slot + ((unsigned)((warp & 3) * 32) << 16);
    const unsigned col0 = (unsigned)((warp >> 2) * 64);
    unsigned acc = 0;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int f = 0; f < kInflight; ++f) {
            unsigned r[32];
            // 64-column aligned start in [0, 384]: every load stays inside the 512 columns
            const unsigned addr = base + ((col0 + (unsigned)(f * 64 + it * 64)) % 448u / 64u * 64u);
            if (kShape == 0)
                asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                    : "=r"(r[0]),"=r"(r[1]),"=r"(r[2]),"=r"(r[3]),"=r"(r[4]),"=r"(r[5]),"=r"(r[6]),"=r"(r[7]),"=r"(r[8]),"=r"(r[9]),"=r"(r[10]),"=r"(r[11]),"=r"(r[12]),"=r"(r[13]),"=r"(r[14]),"=r"(r[15]),"=r"(r[16]),"=r"(r[17]),"=r"(r[18]),"=r"(r[19]),"=r"(r[20]),"=r"(r[21]),"=r"(r[22]),"=r"(r[23]),"=r"(r[24]),"=r"(r[25]),"=r"(r[26]),"=r"(r[27]),"=r"(r[28]),"=r"(r[29]),"=r"(r[30]),"=r"(r[31]) : "r"(addr));
            else
                asm volatile("tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                    : "=r"(r[0]),"=r"(r[1]),"=r"(r[2]),"=r"(r[3]),"=r"(r[4]),"=r"(r[5]),"=r"(r[6]),"=r"(r[7]),"=r"(r[8]),"=r"(r[9]),"=r"(r[10]),"=r"(r[11]),"=r"(r[12]),"=r"(r[13]),"=r"(r[14]),"=r"(r[15]),"=r"(r[16]),"=r"(r[17]),"=r"(r[18]),"=r"(r[19]),"=r"(r[20]),"=r"(r[21]),"=r"(r[22]),"=r"(r[23]),"=r"(r[24]),"=r"(r[25]),"=r"(r[26]),"=r"(r[27]),"=r"(r[28]),"=r"(r[29]),"=r"(r[30]),"=r"(r[31]) : "r"(addr));
            asm volatile("tcgen05.wait::ld.sync.aligned;");
#pragma unroll
            for (int i = 0; i < 32; ++i) acc ^= r[i];
        }
    }
    if (acc == 0x9e3779b9u) out[0] = acc;
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        asm volatile("tcgen05.fence::after_thread_sync;");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(slot));
    }
}

// ---- legacy warp-level f16 MMA rate (mma.sync m16n8k16, f32 accumulate).
__global__ void hmma_loop(int iters, int* out) {
    uint32_t a[4] = {threadIdx.x, threadIdx.x * 3u, threadIdx.x ^ 5u, 7u};
    uint32_t b0 = threadIdx.x * 11u, b1 = 13u;
    float c[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int r = 0; r < 4; ++r) c[i][r] = 0.f;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            asm volatile(
                "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
                "{%8,%9}, {%0,%1,%2,%3};\n"
                : "+f"(c[i][0]), "+f"(c[i][1]), "+f"(c[i][2]), "+f"(c[i][3])
                : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    float s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += c[i][0] + c[i][1] + c[i][2] + c[i][3];
    if (s == 1234.5f) out[0] = 1;
}

// ---- hand-off latencies on one SM (one CTA of 512 threads): the cost of
// the tcgen05 GEMM's producer/consumer chain with no work in it.
//   test 0: one 128x128x16 f16 MMA + commit into an idle tensor pipe
//   test 1: four such MMAs + commit
//   test 2: mbarrier try_wait on an already completed phase
//   test 3/4/5: two tensor-memory slots handed between one issuing thread and
//   eight consumer warps; the issuer waits "slot empty" (8 arrivals) and then
//   signals "slot full" by a commit with no MMA (3), a plain arrive (4), or a
//   commit after four MMAs into the slot (5); consumers wait "full", arrive "empty".
// out[0] = issue cycles, out[1] = total cycles (per iteration after dividing).
__device__ __forceinline__ long long clock64_now() {
    long long c;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(c));
    return c;
}
__device__ __forceinline__ bool spin_wait(uint32_t bar, uint32_t par) {
    const long long t0 = clock64_now();
    while (!mmq::ptx::mbar_try_wait(bar, par))
        if (clock64_now() - t0 > (1ll << 30)) return false;
    return true;
}

template <int kTest>
__global__ void __launch_bounds__(512, 1) handoff_loop(int iters, long long* out) {
    using namespace mmq::ptx;
    extern __shared__ __align__(1024) uint8_t hsm[];
    uint8_t* s = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(hsm) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(s);
    uint32_t* slot = reinterpret_cast<uint32_t*>(s + 32768);
    const uint32_t done = sb + 32768 + 64, full = done + 8, empty = done + 24;   // full/empty: 2 slots each
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < 8192; i += blockDim.x) reinterpret_cast<uint32_t*>(s)[i] = 0;
    if (threadIdx.x == 0) {
        mbar_init(done, 1);
        mbar_init(full, 1);
        mbar_init(full + 8, 1);
        mbar_init(empty, 8);
        mbar_init(empty + 8, 8);
        fence_barrier_init();
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (warp == 0) {
        tmem_alloc(smem_u32(slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = *slot;
    const uint32_t idesc = idesc_f16_f32(128, 128);
    const uint64_t dA = smem_desc_sw128(sb), dB = smem_desc_sw128(sb + 16384);
    bool ok = true;
    if (kTest <= 1) {
        if (warp == 1 && lane == 0) {
            long long tiss = 0, tall = 0;
            for (int i = 0; i < iters && ok; ++i) {
                const long long t0 = clock64_now();
                for (int j = 0; j < (kTest == 0 ? 1 : 4); ++j)
                    mma_f16(tb + uint32_t((j >> 1) * 128), dA + uint64_t(2 * (j & 1)), dB + uint64_t(2 * (j & 1)),
                            idesc, uint32_t(j & 1));
                mma_commit(done);
                const long long t1 = clock64_now();
                ok = spin_wait(done, uint32_t(i & 1));
                tiss += t1 - t0;
                tall += clock64_now() - t0;
            }
            out[0] = tiss;
            out[1] = tall;
        }
    } else if (kTest == 2) {
        if (warp == 1 && lane == 0) {
            mbar_arrive(done);
            int n = 0;
            const long long t0 = clock64_now();
            for (int i = 0; i < iters; ++i) n += mbar_try_wait(done, 0u) ? 1 : 0;
            out[0] = out[1] = clock64_now() - t0;
            if (n != iters) ok = false;
        }
    } else {
        if (warp == 1 && lane == 0) {
            const long long t0 = clock64_now();
            for (int u = 0; u < iters && ok; ++u) {
                const uint32_t sl = uint32_t(u & 1) * 8u, ph = uint32_t(u >> 1) & 1u;
                ok = spin_wait(empty + sl, ph ^ 1u);
                tc_fence_after();
                if (kTest == 5)
                    for (int j = 0; j < 4; ++j)
                        mma_f16(tb + uint32_t((u & 1) * 256 + (j >> 1) * 128), dA + uint64_t(2 * (j & 1)),
                                dB + uint64_t(2 * (j & 1)), idesc, uint32_t(j & 1));
                if (kTest == 4) mbar_arrive(full + sl);
                else mma_commit(full + sl);
            }
            out[0] = out[1] = clock64_now() - t0;
            if (kTest == 5) {
                mma_commit(done);
                ok = ok && spin_wait(done, 0u);
            }
        } else if (warp >= 8) {
            for (int u = 0; u < iters && ok; ++u) {
                const uint32_t sl = uint32_t(u & 1) * 8u, ph = uint32_t(u >> 1) & 1u;
                ok = spin_wait(full + sl, ph);
                tc_fence_after();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(empty + sl);
            }
        }
    }
    if (!ok) out[2] = 1;
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tb, 512);
    }
}

// ---- tcgen05 MMA issue cost by shape: one thread issues `nmma` f16 MMAs of
// 128 x N x 16 back to back (accumulating into N columns), one commit, and
// waits for it; out[0] = issue cycles, out[1] = cycles until the commit
// arrived, summed over iterations.
template <int N>
__global__ void __launch_bounds__(128, 1) mma_burst(int iters, int nmma, long long* out) {
    using namespace mmq::ptx;
    extern __shared__ __align__(1024) uint8_t msm[];
    uint8_t* s = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(msm) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(s);
    uint32_t* slot = reinterpret_cast<uint32_t*>(s + 49152);
    const uint32_t done = sb + 49152 + 64;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < 12288; i += blockDim.x) reinterpret_cast<uint32_t*>(s)[i] = 0;
    if (threadIdx.x == 0) {
        mbar_init(done, 1);
        fence_barrier_init();
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (warp == 0) {
        tmem_alloc(smem_u32(slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = *slot;
    const uint32_t idesc = idesc_f16_f32(128, N);
    const uint64_t dA = smem_desc_sw128(sb), dB = smem_desc_sw128(sb + 16384);
    bool ok = true;
    if (warp == 1 && lane == 0) {
        long long tiss = 0, tall = 0;
        for (int i = 0; i < iters && ok; ++i) {
            const long long t0 = clock64_now();
            for (int j = 0; j < nmma; ++j)
                mma_f16(tb, dA + uint64_t(2 * (j & 3)), dB + uint64_t(2 * (j & 3)), idesc, uint32_t(j != 0));
            mma_commit(done);
            const long long t1 = clock64_now();
            ok = spin_wait(done, uint32_t(i & 1));
            tiss += t1 - t0;
            tall += clock64_now() - t0;
        }
        out[0] = tiss;
        out[1] = tall;
    }
    if (!ok) out[2] = 1;
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tb, 512);
    }
}

// ---- the MMA-issuing thread's loop shape: per "operand stage" four
// 128 x N x 16 MMAs from one of four rotating operand buffers into rotating
// tensor-memory columns, with (kMode & 1) an mbarrier try_wait (on a phase
// completed before the loop) and tcgen05.fence::after_thread_sync first,
// (kMode & 2) the same only every fourth stage, (kMode & 4) two commits
// after.  out[0] = issue cycles over all stages.  Every mbarrier here has
// an arrival count of 1.
template <int kMode, int N>
__global__ void __launch_bounds__(128, 1) mma_stage_loop(int stages, long long* out) {
    using namespace mmq::ptx;
    extern __shared__ __align__(1024) uint8_t lsm[];
    uint8_t* s = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(lsm) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(s);
    constexpr int kOp = 16384 + N * 128, kNumOp = 4;
    uint32_t* slot = reinterpret_cast<uint32_t*>(s + kNumOp * kOp);
    const uint32_t bars = sb + kNumOp * kOp + 64;   // ready, done, 4 x c, 4 x d
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < kNumOp * kOp / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(s)[i] = 0;
    if (threadIdx.x == 0) {
        for (int i = 0; i < 10; ++i) mbar_init(bars + 8 * i, 1);
        fence_barrier_init();
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) mbar_arrive(bars);   // phase 0 of "ready" completes
    if (warp == 0) {
        tmem_alloc(smem_u32(slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = *slot;
    const uint32_t idesc = idesc_f16_f32(128, N);
    bool ok = true;
    if (warp == 1 && lane == 0) {
        const long long t0 = clock64_now();
        for (int st = 0; st < stages && ok; ++st) {
            if ((kMode & 1) || ((kMode & 2) && (st & 3) == 0)) {
                ok = spin_wait(bars, 0u);
                tc_fence_after();
            }
            const uint64_t dA = smem_desc_sw128(sb + (st & 3) * kOp), dB = dA + uint64_t(16384 >> 4);
            const uint32_t d0 = tb + uint32_t((st & (256 / (2 * N) - 1)) * 2 * N);
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
                    mma_f16(d0 + uint32_t(h * N), dA + uint64_t((h * 64 + kk * 32) >> 4),
                            dB + uint64_t((h * 64 + kk * 32) >> 4), idesc, uint32_t(kk));
            if (kMode & 4) {
                mma_commit(bars + 16 + 8 * (st & 3));
                mma_commit(bars + 48 + 8 * (st & 3));
            }
        }
        mma_commit(bars + 8);
        out[0] = clock64_now() - t0;
        ok = ok && spin_wait(bars + 8, 0u);
        out[1] = clock64_now() - t0;
    }
    if (!ok) out[2] = 1;
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tb, 512);
    }
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
    // hmma f16
    hmma_loop<<<blocks, threads>>>(100, dout);
    CK(cudaDeviceSynchronize());
    CK(cudaEventRecord(e0));
    hmma_loop<<<blocks, threads>>>(it_mma, dout);
    CK(cudaEventRecord(e1));
    CK(cudaEventSynchronize(e1));
    CK(cudaEventElapsedTime(&ms, e0, e1));
    const double hmma_tflops = warps * it_mma * 8 * (16.0 * 8 * 16) * 2 / (ms * 1e-3) / 1e12;
    printf("{\"hmma_f16_f32_tflops\": %.2f}\n", hmma_tflops);

    // tensor-memory loads: bytes per SM per clock at the attribute clock
    const int it_t = 4000;
    auto run_t = [&](void (*k)(int, unsigned*), int nwarps, int inflight, const char* name) -> int {
        k<<<nsm, nwarps * 32>>>(10, (unsigned*)dout);
        if (cudaDeviceSynchronize() != cudaSuccess) return 1;
        cudaEventRecord(e0);
        k<<<nsm, nwarps * 32>>>(it_t, (unsigned*)dout);
        cudaEventRecord(e1);
        cudaEventSynchronize(e1);
        float t;
        cudaEventElapsedTime(&t, e0, e1);
        const double bytes = double(nsm) * nwarps * it_t * inflight * 32 * 32 * 4;
        const double per_sm_per_ns = bytes / nsm / (t * 1e6);
        printf("{\"tmem_ld\": \"%s\", \"warps\": %d, \"inflight\": %d, \"GBps_per_sm\": %.1f, \"bytes_per_clk_at_2070MHz\": %.1f, \"TBps_total\": %.2f}\n",
               name, nwarps, inflight, per_sm_per_ns, per_sm_per_ns / 2.07, bytes / (t * 1e-3) / 1e12);
        return 0;
    };
    if (run_t(tmem_ld_loop<0, 1>, 4, 1, "32x32b.x32") || run_t(tmem_ld_loop<0, 1>, 8, 1, "32x32b.x32") ||
        run_t(tmem_ld_loop<0, 1>, 16, 1, "32x32b.x32") || run_t(tmem_ld_loop<0, 2>, 8, 2, "32x32b.x32") ||
        run_t(tmem_ld_loop<1, 1>, 8, 1, "16x256b.x8") || run_t(tmem_ld_loop<1, 1>, 16, 1, "16x256b.x8") ||
        run_t(tmem_ld_loop<1, 2>, 8, 2, "16x256b.x8"))
        return 1;

    // hand-off latencies (cycles per iteration on one SM)
    long long* dl;
    CK(cudaMalloc(&dl, 3 * sizeof(long long)));
    auto run_h = [&](void (*k)(int, long long*), int iters, const char* name) -> int {
        const int smem = 32768 + 1024 + 128;
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 1;
        CK(cudaMemset(dl, 0, 3 * sizeof(long long)));
        k<<<1, 512, smem>>>(iters, dl);
        CK(cudaDeviceSynchronize());
        long long h[3];
        CK(cudaMemcpy(h, dl, sizeof(h), cudaMemcpyDeviceToHost));
        printf("{\"handoff\": \"%s\", \"issue_cycles\": %.1f, \"cycles\": %.1f, \"timed_out\": %lld}\n", name,
               double(h[0]) / iters, double(h[1]) / iters, h[2]);
        return 0;
    };
    if (run_h(handoff_loop<0>, 512, "1 MMA 128x128x16 + commit, idle pipe") ||
        run_h(handoff_loop<1>, 512, "4 MMAs + commit, idle pipe") ||
        run_h(handoff_loop<2>, 4096, "try_wait on a completed phase") ||
        run_h(handoff_loop<3>, 2048, "2-slot hand-off, commit without MMA, 8 consumer warps") ||
        run_h(handoff_loop<4>, 2048, "2-slot hand-off, plain arrive, 8 consumer warps") ||
        run_h(handoff_loop<5>, 2048, "2-slot hand-off, 4 MMAs + commit, 8 consumer warps"))
        return 1;

    // MMA issue cost by N (cycles per MMA on one SM)
    auto run_m = [&](void (*k)(int, int, long long*), int n, int nmma) -> int {
        const int smem = 49152 + 1024 + 128;
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 1;
        CK(cudaMemset(dl, 0, 3 * sizeof(long long)));
        const int iters = 256;
        k<<<1, 128, smem>>>(iters, nmma, dl);
        CK(cudaDeviceSynchronize());
        long long h[3];
        CK(cudaMemcpy(h, dl, sizeof(h), cudaMemcpyDeviceToHost));
        printf("{\"mma_burst\": \"128x%dx16 f16\", \"mmas\": %d, \"issue_cycles_per_mma\": %.1f, "
               "\"cycles_per_mma\": %.1f, \"timed_out\": %lld}\n",
               n, nmma, double(h[0]) / iters / nmma, double(h[1]) / iters / nmma, h[2]);
        return 0;
    };
    for (int nmma : {4, 32})
        if (run_m(mma_burst<16>, 16, nmma) || run_m(mma_burst<32>, 32, nmma) || run_m(mma_burst<64>, 64, nmma) ||
            run_m(mma_burst<128>, 128, nmma) || run_m(mma_burst<256>, 256, nmma))
            return 1;

    // the MMA thread's loop shape (cycles per operand stage of four MMAs)
    auto run_l = [&](void (*k)(int, long long*), const char* name) -> int {
        const int smem = 4 * 32768 + 1024 + 512;   // four 32 KB operand buffers + barriers
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 1;
        CK(cudaMemset(dl, 0, 3 * sizeof(long long)));
        const int stages = 64;
        k<<<1, 128, smem>>>(stages, dl);
        CK(cudaDeviceSynchronize());
        long long h[3];
        CK(cudaMemcpy(h, dl, sizeof(h), cudaMemcpyDeviceToHost));
        printf("{\"mma_stage_loop\": \"%s\", \"issue_cycles_per_stage\": %.1f, \"timed_out\": %lld}\n", name,
               double(h[0]) / stages, h[2]);
        return 0;
    };
    if (run_l(mma_stage_loop<0, 16>, "N=16: four MMAs per stage") ||
        run_l(mma_stage_loop<1, 16>, "N=16: + try_wait and fence per stage") ||
        run_l(mma_stage_loop<2, 16>, "N=16: + try_wait and fence every fourth stage") ||
        run_l(mma_stage_loop<5, 16>, "N=16: + try_wait, fence and two commits per stage") ||
        run_l(mma_stage_loop<0, 128>, "N=128: four MMAs per stage") ||
        run_l(mma_stage_loop<5, 128>, "N=128: + try_wait, fence and two commits per stage"))
        return 1;
    return 0;
}

