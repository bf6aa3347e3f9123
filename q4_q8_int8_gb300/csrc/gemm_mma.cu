// q4_K x q8_1 GEMM on warp-level integer MMA (mma.sync m16n8k32 s8 x s8 -> s32).
//
// This is the genuine int8 tensor path available on sm_103a (tcgen05 has no
// integer kind there).  It also serves as the control kernel for the
// tensor-memory kernel: same math, an independent data path.
//
// Math (web page "20 . r15 -- f32-accumulate mma probe (dead end) + rank-1
// term2 rescale", section 2.1): per 32-k chunk c the integer MMA produces
// S_ij exactly (|S| <= 32*127*15, section 2.3), then
//     acc_ij += (da_ic * dsv_jc) * S_ij + dma_ic * dmv_jc,
// with dsv = d*sc, dmv = -dmin*m (expanded per sub-block when a super-block
// is staged) and dma = da*sa formed once per token row and chunk (the
// rank-1 fold, page "21 . r16 -- Narrow kernel gets the rank-1 fold",
// section 2.1).
//
// Design for sm_103a (own layout, not the pages' kernels):
//  - CTA tile 128 tokens x 128 weight rows, 8 warps as 2 (tokens) x 4
//    (weights); each warp owns 64 x 32 = 4 A fragments x 4 B fragments =
//    16 independent MMA chains per chunk.
//  - One 256-k super-block per pipeline stage, 3 stages of cp.async:
//    A int8 rows padded to 272 B (conflict-free ldmatrix), the raw 144-byte
//    q4_K rows as stored (no unpack pass), and the da/sa slices.
//  - B fragments come straight from the raw nibbles: in the q4_K layout the
//    32 quants of sub-block 2p+h are nibble h of bytes 32p..32p+31, which is
//    exactly the k order of an m16n8k32 B fragment, so one 32-bit shared
//    load per fragment register serves two chunks (low / high nibble) and
//    the unpack is one shift-and-mask.  Row pitch 144 B = 36 words makes
//    the 8 rows x 4 words of a fragment load hit 32 distinct banks.
//  - The s32 accumulator is seeded with the bit pattern of 1.5 * 2^23, so
//    after the MMA its bits read as the float 1.5*2^23 + S exactly and one
//    FADD recovers S as a float (no I2F).
#include <cuda_fp16.h>

#include "mmq_internal.h"

namespace {

constexpr int BM = 128, BN = 128, kThreads = 256, kStages = 3;
constexpr int kARowBytes = 272;                        // 256 + 16 pad
constexpr int kAStage = BM * kARowBytes;               // 34816
constexpr int kWStage = BN * 144;                      // 18432
constexpr int kScaleStage = BM * 8 * 4;                // 4096 (da or sa slice)
constexpr int kStageBytes = kAStage + kWStage + 2 * kScaleStage;
constexpr int kSmemBytes = kStages * kStageBytes + 2 * (8 * 128 * 8);   // + row/col scale tables
constexpr uint32_t kBiasBits = 0x4B400000u;            // 12582912.0f
constexpr float kBias = 12582912.0f;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_s8(uint32_t (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                       uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float half_bits_to_float(uint32_t h) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

// Issue the cp.async copies of super-block `sb` into stage buffer `st`.
__device__ __forceinline__ void load_stage(uint32_t st, const mmq_q8_1_t& aq, const uint8_t* w,
                                           int64_t M, int64_t N, int64_t K, int64_t m0,
                                           int64_t n0, int64_t sb) {
    const int t = threadIdx.x;
    const int64_t nsb = K / 256, nb = K / 32;
    // A: 128 rows x 16 pieces of 16 B
#pragma unroll
    for (int i = 0; i < (BM * 16) / kThreads; ++i) {
        const int piece = t + i * kThreads;
        const int r = piece >> 4, seg = piece & 15;
        const bool ok = (m0 + r) < M;
        const int8_t* src = ok ? aq.qs + (m0 + r) * K + sb * 256 + seg * 16 : aq.qs;
        cp_async16(st + r * kARowBytes + seg * 16, src, ok);
    }
    // W: 128 rows x 9 pieces
    for (int piece = t; piece < BN * 9; piece += kThreads) {
        const int r = piece / 9, seg = piece - r * 9;
        const bool ok = (n0 + r) < N;
        const uint8_t* src = ok ? w + ((n0 + r) * nsb + sb) * 144 + seg * 16 : w;
        cp_async16(st + kAStage + r * 144 + seg * 16, src, ok);
    }
    // da, sa: 128 rows x 2 pieces each
    {
        const int r = t >> 1, seg = t & 1;
        const bool ok = (m0 + r) < M;
        const float* sd = ok ? aq.da + (m0 + r) * nb + sb * 8 + seg * 4 : aq.da;
        const int32_t* ss = ok ? aq.sa + (m0 + r) * nb + sb * 8 + seg * 4 : aq.sa;
        cp_async16(st + kAStage + kWStage + r * 32 + seg * 16, sd, ok);
        cp_async16(st + kAStage + kWStage + kScaleStage + r * 32 + seg * 16, ss, ok);
    }
}

template <bool kDump>
__global__ void __launch_bounds__(kThreads, 1)
gemm_mma_s8_kernel(mmq_q8_1_t aq, const uint8_t* __restrict__ w, float* __restrict__ C,
                   int32_t* __restrict__ S, int64_t M, int64_t N, int64_t K) {
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    float2* rowsc = reinterpret_cast<float2*>(smem + kStages * kStageBytes);   // [8][128] (da, dma)
    float2* colsc = rowsc + 8 * 128;                                          // [8][128] (dsv, dmv)

    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int wm = warp & 1, wn = warp >> 1;
    const int64_t m0 = int64_t(blockIdx.y) * BM, n0 = int64_t(blockIdx.x) * BN;
    const int64_t nsb = K / 256, nb = K / 32;

    float acc[4][4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[a][b][r] = 0.0f;

#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (s < nsb) load_stage(sbase + s * kStageBytes, aq, w, M, N, K, m0, n0, s);
        cp_async_commit();
    }

    for (int64_t sb = 0; sb < nsb; ++sb) {
        cp_async_wait<kStages - 2>();
        __syncthreads();   // stage sb visible; everyone is done with sb-1
        {
            const int64_t nx = sb + kStages - 1;
            if (nx < nsb) load_stage(sbase + (nx % kStages) * kStageBytes, aq, w, M, N, K, m0, n0, nx);
            cp_async_commit();
        }
        const int st = int(sb % kStages);
        const uint8_t* sA = smem + st * kStageBytes;
        const uint8_t* sW = sA + kAStage;
        const float* sDa = reinterpret_cast<const float*>(sW + kWStage);
        const int32_t* sSa = reinterpret_cast<const int32_t*>(sW + kWStage + kScaleStage);

        if (!kDump) {
            // Expand per-sub-block weight scales: dsv = d*sc, dmv = -dmin*m
            // (both exact in f32), and the folded row factor dma = da*sa.
            {
                const int n = t >> 1, c4 = (t & 1) * 4;
                const uint8_t* blk = sW + n * 144;
                const float d = half_bits_to_float(blk[0] | (blk[1] << 8));
                const float dmin = half_bits_to_float(blk[2] | (blk[3] << 8));
                const uint8_t* s = blk + 4;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int c = c4 + cc;
                    int sc, m;
                    if (c < 4) {
                        sc = s[c] & 63;
                        m = s[c + 4] & 63;
                    } else {
                        sc = (s[c + 4] & 15) | ((s[c - 4] >> 6) << 4);
                        m = (s[c + 4] >> 4) | ((s[c] >> 6) << 4);
                    }
                    colsc[c * 128 + n] = make_float2(d * float(sc), -(dmin * float(m)));
                }
            }
            {
                const int r = t >> 1, c4 = (t & 1) * 4;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const float da = sDa[r * 8 + c4 + cc];
                    rowsc[(c4 + cc) * 128 + r] = make_float2(da, da * float(sSa[r * 8 + c4 + cc]));
                }
            }
            __syncthreads();
        }

        const uint32_t aRowAddr = sbase + st * kStageBytes +
                                  (wm * 64 + (lane & 7) + ((lane >> 3) & 1) * 8) * kARowBytes +
                                  (lane >> 4) * 16;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            uint32_t bw[4][2];
#pragma unroll
            for (int fn = 0; fn < 4; ++fn) {
                const uint8_t* row = sW + (wn * 32 + fn * 8 + (lane >> 2)) * 144 + 16 + 32 * p + (lane & 3) * 4;
                bw[fn][0] = *reinterpret_cast<const uint32_t*>(row);
                bw[fn][1] = *reinterpret_cast<const uint32_t*>(row + 16);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int c = 2 * p + h;
                uint32_t af[4][4];
#pragma unroll
                for (int fm = 0; fm < 4; ++fm)
                    ldmatrix_x4(aRowAddr + fm * 16 * kARowBytes + c * 32, af[fm][0], af[fm][1],
                                af[fm][2], af[fm][3]);
                uint32_t ci[4][4][4];
#pragma unroll
                for (int fm = 0; fm < 4; ++fm)
#pragma unroll
                    for (int fn = 0; fn < 4; ++fn)
#pragma unroll
                        for (int r = 0; r < 4; ++r) ci[fm][fn][r] = kDump ? 0u : kBiasBits;
#pragma unroll
                for (int fn = 0; fn < 4; ++fn) {
                    const uint32_t b0 = (bw[fn][0] >> (4 * h)) & 0x0F0F0F0Fu;
                    const uint32_t b1 = (bw[fn][1] >> (4 * h)) & 0x0F0F0F0Fu;
#pragma unroll
                    for (int fm = 0; fm < 4; ++fm) mma_s8(ci[fm][fn], af[fm], b0, b1);
                }
                if (kDump) {
#pragma unroll
                    for (int fm = 0; fm < 4; ++fm)
#pragma unroll
                        for (int fn = 0; fn < 4; ++fn)
#pragma unroll
                            for (int r = 0; r < 4; ++r) {
                                const int64_t row = m0 + wm * 64 + fm * 16 + (lane >> 2) + (r >> 1) * 8;
                                const int64_t col = n0 + wn * 32 + fn * 8 + (lane & 3) * 2 + (r & 1);
                                if (row < M && col < N)
                                    S[(row * N + col) * nb + sb * 8 + c] = int32_t(ci[fm][fn][r]);
                            }
                } else {
                    float2 rs[4][2];
#pragma unroll
                    for (int fm = 0; fm < 4; ++fm)
#pragma unroll
                        for (int hr = 0; hr < 2; ++hr)
                            rs[fm][hr] = rowsc[c * 128 + wm * 64 + fm * 16 + (lane >> 2) + hr * 8];
#pragma unroll
                    for (int fn = 0; fn < 4; ++fn) {
                        const float4 cs = *reinterpret_cast<const float4*>(
                            &colsc[c * 128 + wn * 32 + fn * 8 + (lane & 3) * 2]);
#pragma unroll
                        for (int fm = 0; fm < 4; ++fm)
#pragma unroll
                            for (int r = 0; r < 4; ++r) {
                                const float2 rr = rs[fm][r >> 1];
                                const float dsv = (r & 1) ? cs.z : cs.x;
                                const float dmv = (r & 1) ? cs.w : cs.y;
                                const float s = __uint_as_float(ci[fm][fn][r]) - kBias;
                                float a = acc[fm][fn][r];
                                a = fmaf(rr.x * dsv, s, a);
                                a = fmaf(rr.y, dmv, a);
                                acc[fm][fn][r] = a;
                            }
                    }
                }
            }
        }
    }
    cp_async_wait<0>();

    if (!kDump) {
#pragma unroll
        for (int fm = 0; fm < 4; ++fm)
#pragma unroll
            for (int fn = 0; fn < 4; ++fn)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int64_t row = m0 + wm * 64 + fm * 16 + (lane >> 2) + hr * 8;
                    const int64_t col = n0 + wn * 32 + fn * 8 + (lane & 3) * 2;
                    if (row < M && col < N)
                        *reinterpret_cast<float2*>(C + row * N + col) =
                            make_float2(acc[fm][fn][2 * hr], acc[fm][fn][2 * hr + 1]);
                }
    }
}

}  // namespace

namespace mmq {

cudaError_t launch_gemm_mma_s8(mmq_q8_1_t aq, const uint8_t* w, float* C, int32_t* S,
                               int64_t M, int64_t N, int64_t K, int* status, cudaStream_t s) {
    (void)status;   // no device-side waits in this kernel
    const dim3 grid(unsigned((N + BN - 1) / BN), unsigned((M + BM - 1) / BM));
    if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
    if (S) {
        auto k = gemm_mma_s8_kernel<true>;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        k<<<grid, kThreads, kSmemBytes, s>>>(aq, w, C, S, M, N, K);
    } else {
        auto k = gemm_mma_s8_kernel<false>;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        k<<<grid, kThreads, kSmemBytes, s>>>(aq, w, C, S, M, N, K);
    }
    return cudaGetLastError();
}

}  // namespace mmq
