// q8_1 quantize prepass: float activations -> int8 quants, f32 scale and
// int32 block sum per 32 elements, in one streaming pass.
//
// Web page "20 . r15 -- f32-accumulate mma probe (dead end) + rank-1 term2
// rescale", section 2.1: each 32-element block carries its scale da and the
// in-block integer sum sa, both produced by the quantize prepass.
//
// Bandwidth kernel: x is read once (5/4 bytes written per 4 read).  A group
// of 8 lanes owns one 32-element block (one float4 per lane), so a warp
// covers four consecutive blocks = 512 contiguous bytes per load; amax and
// the sum are reduced with three xor-shuffles inside the 8-lane group.
// Each warp keeps kUnroll groups of four blocks in flight.  The quotient
// x / da is formed from the block's reciprocal with an exactness check (see
// quant1), so the bits match IEEE division followed by roundf.
#include "mmq_internal.h"
#include "q8_round.cuh"
#include "sm103_ptx.cuh"

namespace {

using namespace mmq::q8;

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__device__ __forceinline__ float4 load_stream(const float* p) {
    return __ldcs(reinterpret_cast<const float4*>(p));
}

__global__ void __launch_bounds__(kThreads)
quantize_q8_1_kernel(const float* __restrict__ x, int8_t* __restrict__ qs,
                     float* __restrict__ da, int32_t* __restrict__ sa, int64_t nblocks) {
    const int lane = threadIdx.x & 31;
    const int sub = lane >> 3;          // which of the warp's 4 blocks
    const int part = lane & 7;          // which float4 of the block
    const int64_t ngroups = (nblocks + 3) / 4;
    const int64_t warp = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * kThreads) >> 5;
    // programmatic dependent launch: x may be the previous kernel's output,
    // and the q8_1 planes may still be read by it
    mmq::ptx::griddep_launch_dependents();
    mmq::ptx::griddep_wait();

    for (int64_t g0 = warp * kUnroll; g0 < ngroups; g0 += nwarps * kUnroll) {
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t blk = (g0 + u) * 4 + sub;
            v[u] = (blk < nblocks) ? load_stream(x + blk * 32 + part * 4)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t g = g0 + u;
            const int64_t blk = g * 4 + sub;
            float amax = fmaxf(fmaxf(fabsf(v[u].x), fabsf(v[u].y)),
                               fmaxf(fabsf(v[u].z), fabsf(v[u].w)));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
            const float d = __fdiv_rn(amax, 127.0f);
            int q0 = 0, q1 = 0, q2 = 0, q3 = 0;   // a zero scale gives zero quants
            bool redo = false;
            if (d != 0.0f) {
                redo = d < 0x1p-126f;   // d below the smallest normal float: always divide
                const float r = __frcp_rn(d);
                q0 = quant_fast(v[u].x, r, redo);
                q1 = quant_fast(v[u].y, r, redo);
                q2 = quant_fast(v[u].z, r, redo);
                q3 = quant_fast(v[u].w, r, redo);
            }
            // Rare: some lane needs IEEE division.  The vote runs on all 32
            // lanes (outside the per-block branch above).
            if (__any_sync(0xffffffffu, redo)) {
                if (redo) {
                    q0 = quant_exact(v[u].x, d);
                    q1 = quant_exact(v[u].y, d);
                    q2 = quant_exact(v[u].z, d);
                    q3 = quant_exact(v[u].w, d);
                }
            }
            q0 = clamp127(q0);
            q1 = clamp127(q1);
            q2 = clamp127(q2);
            q3 = clamp127(q3);
            int s = q0 + q1 + q2 + q3;
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            s += __shfl_xor_sync(0xffffffffu, s, 4);
            const uint32_t packed = (uint32_t(q0) & 0xFFu) | ((uint32_t(q1) & 0xFFu) << 8) |
                                    ((uint32_t(q2) & 0xFFu) << 16) | ((uint32_t(q3) & 0xFFu) << 24);
            if (blk < nblocks)
                *reinterpret_cast<uint32_t*>(qs + blk * 32 + part * 4) = packed;
            // Gather the four blocks' (d, s) into lane 0 for one 16-byte store each.
            const float d1 = __shfl_sync(0xffffffffu, d, 8), d2 = __shfl_sync(0xffffffffu, d, 16),
                        d3 = __shfl_sync(0xffffffffu, d, 24);
            const int s1 = __shfl_sync(0xffffffffu, s, 8), s2 = __shfl_sync(0xffffffffu, s, 16),
                      s3 = __shfl_sync(0xffffffffu, s, 24);
            if (lane == 0 && g < ngroups) {
                if (g * 4 + 3 < nblocks) {
                    *reinterpret_cast<float4*>(da + g * 4) = make_float4(d, d1, d2, d3);
                    *reinterpret_cast<int4*>(sa + g * 4) = make_int4(s, s1, s2, s3);
                } else {
                    const float dd[4] = {d, d1, d2, d3};
                    const int ss[4] = {s, s1, s2, s3};
                    for (int t = 0; t < 4 && g * 4 + t < nblocks; ++t) {
                        da[g * 4 + t] = dd[t];
                        sa[g * 4 + t] = ss[t];
                    }
                }
            }
        }
    }
}

}  // namespace

namespace mmq {

cudaError_t launch_quantize_q8_1(const float* x, int64_t M, int64_t K, mmq_q8_1_t aq,
                                 cudaStream_t s) {
    const int64_t nblocks = M * (K / 32);
    const int64_t ngroups = (nblocks + 3) / 4;
    const int64_t warps_needed = (ngroups + kUnroll - 1) / kUnroll;
    int dev = 0, nsm = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    const int64_t max_ctas = int64_t(nsm) * (2048 / kThreads);   // one full wave
    int64_t ctas = (warps_needed + (kThreads / 32) - 1) / (kThreads / 32);
    if (ctas > max_ctas) ctas = max_ctas;
    if (ctas < 1) ctas = 1;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = launch_config(dim3(unsigned(ctas)), dim3(kThreads), 0, s, attr);
    return cudaLaunchKernelEx(&cfg, quantize_q8_1_kernel, x, aq.qs, aq.da, aq.sa, nblocks);
}

}  // namespace mmq
