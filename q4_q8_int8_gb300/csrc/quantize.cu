// q8_1 quantize prepass: float activations -> int8 quants, f32 scale and
// int32 block sum per 32 elements, in one streaming pass.
//
// Web page "20 . r15 -- f32-accumulate mma probe (dead end) + rank-1 term2
// rescale", section 2.1: each 32-element block carries its scale da and the
// in-block integer sum sa, both produced by the quantize prepass.
//
// Bandwidth kernel: x is read once (5/4 bytes written per 4 read).  A group
// of 4 lanes owns one 32-element block, each lane two float4 (elements 4p..
// 4p+3 and 16+4p..16+4p+3 for lane p of the group), so one load instruction
// of the warp covers 8 blocks in fully used 32-byte sectors; amax and the
// sum are reduced with two xor-shuffles inside the group, and the per-block
// work (the scale's division and reciprocal, the reductions, the scale and
// sum stores) is shared by 8 elements per lane.  Each warp keeps kUnroll
// groups of eight blocks in flight.  The quotient x / da is formed from the
// block's reciprocal with an exactness check (see quant_fast), so the bits
// match IEEE division followed by roundf.
//
// The tensor-core form (kTc) also writes the operand plane that the
// super-block GEMM (gemm_sb.cu) feeds straight to its tensor cores.  A warp
// instruction's eight blocks are one token row's 256-element super-block
// (K % 256 == 0), so the warp shares that super-block's exponent: with D the
// largest da of the eight blocks and e = max(biased exponent of D, 8),
// inv = 2^(134 - e) and g = 2^(e - 134); s = da * inv is exact, s_hi = s
// rounded to 4 significant bits, s_lo = fp16(s - fp16(s_hi)), and every
// quant q becomes hi = q * s_hi (an exact fp16 product, |q| <= 127) and
// lo = fp16(q * s_lo), so that hi + lo is within 2^-14 of q * s; each
// token row's chunk is one 128-byte line, 32 hi then 32 lo.  Within each
// group of four elements the plane keeps the order 0, 2, 1, 3 (the order in
// which the GEMM unpacks pairs of 4-bit weights).  Per token row
// and super-block it also writes the second term's activation factors,
// dma * inv (dma = da * sa, the rank-1 fold of web page "21 . r16 -- Narrow
// kernel gets the rank-1 fold", section 2.1) split into tf32 hi + lo, as 32
// f32 slots [hi x8 | hi x8 | lo x8 | 0 x8], and g.
#include <cuda_fp16.h>

#include "mmq_internal.h"
#include "q8_round.cuh"
#include "sm103_ptx.cuh"

namespace {

using namespace mmq::q8;

constexpr int kThreads = 256;
constexpr int kUnroll = 2;
constexpr int kBlocksPerWarp = 8;   // blocks covered by one warp instruction

__device__ __forceinline__ float4 load_stream(const float* p) {
    return __ldcs(reinterpret_cast<const float4*>(p));
}

__device__ __forceinline__ uint32_t pack4(int q0, int q1, int q2, int q3) {
    return (uint32_t(q0) & 0xFFu) | ((uint32_t(q1) & 0xFFu) << 8) | ((uint32_t(q2) & 0xFFu) << 16) |
           ((uint32_t(q3) & 0xFFu) << 24);
}

// fp16 bits of the integer q (|q| <= 127 is exact in fp16)
__device__ __forceinline__ uint32_t h2_of(int a, int b) {
    const __half2 h = __halves2half2(__int2half_rn(a), __int2half_rn(b));
    return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t hmul2u(uint32_t a, uint32_t b) {
    __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
    return *reinterpret_cast<uint32_t*>(&r);
}

struct TcPlanes {
    uint16_t* a;    // fp16 [M][K/32][64]: per chunk 32 hi then 32 lo, k order 0,2,1,3 per four
    float* t2;      // f32 [M][K/256][32]
    float* g;       // f32 [M][K/256]
};

template <bool kTc>
__global__ void __launch_bounds__(kThreads)
quantize_q8_1_kernel(const float* __restrict__ x, int8_t* __restrict__ qs,
                     float* __restrict__ da, int32_t* __restrict__ sa, int64_t nblocks, TcPlanes tc) {
    const int lane = threadIdx.x & 31;
    const int sub = lane >> 2;          // which of the warp's 8 blocks
    const int part = lane & 3;          // which pair of float4 of the block
    const int64_t ngroups = (nblocks + kBlocksPerWarp - 1) / kBlocksPerWarp;
    const int64_t warp = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * kThreads) >> 5;
    // programmatic dependent launch: x may be the previous kernel's output,
    // and the q8_1 planes may still be read by it
    mmq::ptx::griddep_launch_dependents();
    mmq::ptx::griddep_wait();
    for (int64_t g0 = warp * kUnroll; g0 < ngroups; g0 += nwarps * kUnroll) {
        float4 v[kUnroll][2];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t blk = (g0 + u) * kBlocksPerWarp + sub;
#pragma unroll
            for (int h = 0; h < 2; ++h)
                v[u][h] = (blk < nblocks) ? load_stream(x + blk * 32 + 16 * h + part * 4)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t blk = (g0 + u) * kBlocksPerWarp + sub;
            const float4 a = v[u][0], b = v[u][1];
            float amax = fmaxf(fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))),
                               fmaxf(fmaxf(fabsf(b.x), fabsf(b.y)), fmaxf(fabsf(b.z), fabsf(b.w))));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            const float d = __fdiv_rn(amax, 127.0f);
            int q[8] = {0, 0, 0, 0, 0, 0, 0, 0};   // a zero scale gives zero quants
            bool redo = false;
            if (d != 0.0f) {
                redo = d < 0x1p-126f;   // d below the smallest normal float: always divide
                const float r = __frcp_rn(d);
                q[0] = quant_fast(a.x, r, redo);
                q[1] = quant_fast(a.y, r, redo);
                q[2] = quant_fast(a.z, r, redo);
                q[3] = quant_fast(a.w, r, redo);
                q[4] = quant_fast(b.x, r, redo);
                q[5] = quant_fast(b.y, r, redo);
                q[6] = quant_fast(b.z, r, redo);
                q[7] = quant_fast(b.w, r, redo);
            }
            // Rare: some lane needs IEEE division.  The vote runs on all 32
            // lanes (outside the per-block branch above).
            if (__any_sync(0xffffffffu, redo)) {
                if (redo) {
                    q[0] = quant_exact(a.x, d);
                    q[1] = quant_exact(a.y, d);
                    q[2] = quant_exact(a.z, d);
                    q[3] = quant_exact(a.w, d);
                    q[4] = quant_exact(b.x, d);
                    q[5] = quant_exact(b.y, d);
                    q[6] = quant_exact(b.z, d);
                    q[7] = quant_exact(b.w, d);
                }
            }
            int sum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                q[i] = clamp127(q[i]);
                sum += q[i];
            }
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            if (blk < nblocks) {
                *reinterpret_cast<uint32_t*>(qs + blk * 32 + part * 4) = pack4(q[0], q[1], q[2], q[3]);
                *reinterpret_cast<uint32_t*>(qs + blk * 32 + 16 + part * 4) = pack4(q[4], q[5], q[6], q[7]);
                if (part == 0) {
                    da[blk] = d;
                    sa[blk] = sum;
                }
            }
            if (kTc) {
                // the super-block's exponent: the largest da of the warp's 8 blocks
                float D = d;
                D = fmaxf(D, __shfl_xor_sync(0xffffffffu, D, 4));
                D = fmaxf(D, __shfl_xor_sync(0xffffffffu, D, 8));
                D = fmaxf(D, __shfl_xor_sync(0xffffffffu, D, 16));
                uint32_t eb = (__float_as_uint(D) >> 23) & 0xFFu;
                eb = eb < 8u ? 8u : eb;
                const float inv = __uint_as_float((261u - eb) << 23);
                const float s = d * inv;
                const float shi = __uint_as_float((__float_as_uint(s) + 0x00080000u) & 0xFFF00000u);
                const __half hh = __float2half_rn(shi);
                const __half hl = __float2half_rn(s - __half2float(hh));
                const uint32_t sh = uint32_t(__half_as_ushort(hh)) * 0x10001u;
                const uint32_t sl = uint32_t(__half_as_ushort(hl)) * 0x10001u;
                // elements (0,2), (1,3) of each group of four as fp16 pairs
                const uint32_t p0 = h2_of(q[0], q[2]), p1 = h2_of(q[1], q[3]);
                const uint32_t p2 = h2_of(q[4], q[6]), p3 = h2_of(q[5], q[7]);
                // dma * inv for the second term; lane L of the warp writes slot L
                const float am = (d * float(sum)) * inv;
                const float amc = __shfl_sync(0xffffffffu, am, 4 * (lane & 7));
                const float ahi = __uint_as_float(__float_as_uint(amc) & 0xFFFFE000u);
                const float slot = lane < 16 ? ahi : (lane < 24 ? amc - ahi : 0.0f);
                if (blk < nblocks) {
                    uint16_t* ab = tc.a + blk * 64 + part * 4;   // hi at [0, 32), lo at [32, 64)
                    *reinterpret_cast<uint2*>(ab) = make_uint2(hmul2u(p0, sh), hmul2u(p1, sh));
                    *reinterpret_cast<uint2*>(ab + 16) = make_uint2(hmul2u(p2, sh), hmul2u(p3, sh));
                    *reinterpret_cast<uint2*>(ab + 32) = make_uint2(hmul2u(p0, sl), hmul2u(p1, sl));
                    *reinterpret_cast<uint2*>(ab + 48) = make_uint2(hmul2u(p2, sl), hmul2u(p3, sl));
                    const int64_t grp = blk >> 3;   // token row * (K/256) + super-block
                    tc.t2[grp * 32 + lane] = slot;
                    if (lane == 0) tc.g[grp] = __uint_as_float((eb - 7u) << 23);
                }
            }
        }
    }
}

}  // namespace

namespace mmq {

static cudaError_t launch_q8(const float* x, int64_t M, int64_t K, mmq_q8_1_t aq, TcPlanes tc, bool with_tc,
                             cudaStream_t s) {
    const int64_t nblocks = M * (K / 32);
    const int64_t ngroups = (nblocks + kBlocksPerWarp - 1) / kBlocksPerWarp;
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
    if (with_tc) return cudaLaunchKernelEx(&cfg, quantize_q8_1_kernel<true>, x, aq.qs, aq.da, aq.sa, nblocks, tc);
    return cudaLaunchKernelEx(&cfg, quantize_q8_1_kernel<false>, x, aq.qs, aq.da, aq.sa, nblocks, tc);
}

cudaError_t launch_quantize_q8_1(const float* x, int64_t M, int64_t K, mmq_q8_1_t aq, cudaStream_t s) {
    return launch_q8(x, M, K, aq, TcPlanes{nullptr, nullptr, nullptr}, false, s);
}

cudaError_t launch_quantize_q8_1_tcop(const float* x, int64_t M, int64_t K, mmq_q8_1_t aq, void* tcop,
                                      cudaStream_t s) {
    const TcopLayout L = tcop_layout(M, K);
    char* b = static_cast<char*>(tcop);
    TcPlanes tc{reinterpret_cast<uint16_t*>(b + L.a), reinterpret_cast<float*>(b + L.t2),
                reinterpret_cast<float*>(b + L.g)};
    return launch_q8(x, M, K, aq, tc, true, s);
}

}  // namespace mmq
