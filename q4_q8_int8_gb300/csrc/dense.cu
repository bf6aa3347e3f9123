// The dequantize-then-dense control path: q4_K weights expanded to fp16, the
// activations rounded to fp16, and a dense fp16 x fp16 -> f32 GEMM on the
// tcgen05 tensor cores.  This is the "f16 default path" the pages measure
// MMQ against (web page "16 . r12 -- 16-chain warp tile + ldmatrix", the
// landing note comparing MMQ with the f16 GEMM path), with its dequantize
// step a bandwidth kernel like the one audited on page "Round 31 Track C
// Audit: dq_f16 (dense_mm.metal) & DW<F> (mma.metal)", section 2.1.
//
// Dequantized weight (q4_K, 256-element super-blocks): for element k of
// sub-block c = k / 32 of a super-block with fp16 d, dmin, 6-bit sc_c, m_c
// and 4-bit v_k:
//     w_k = fp16( f32( d * sc_c * v_k - dmin * m_c ) )
// d * sc_c * v_k and dmin * m_c are exact in f32 (at most 21 and 17
// significant bits), so the f32 value is their difference rounded once
// (round to nearest even), then rounded once more to fp16.
//
// Dense GEMM: C[M][N] = A[M][K] . B[N][K]^T, A and B fp16 row-major (K
// contiguous), C f32.  One CTA per SM, persistent over 128 x 256 tiles:
//   warp 0      TMA producer: per 64-k stage a 128 x 64 A box and a 256 x 64
//               B box, 128-byte swizzled (4 stages in flight).
//   warp 1      MMA issuer (one thread): four K=16 MMAs per stage into one
//               of two 256-column tensor-memory accumulators, a commit per
//               stage to free its operand buffers, one per tile for the
//               epilogue.
//   warps 4-11  epilogue: thread = tile row (its tensor-memory lane), 128
//               columns; copies the accumulator to C while the MMA thread
//               fills the other accumulator.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "mmq_internal.h"
#include "sm103_ptx.cuh"
#include "tc_common.cuh"

namespace {

using namespace mmq::ptx;
using namespace mmq::tc;

// ------------------------------------------------------------- dequantize
// One warp per kSbPerWarp consecutive (weight row, super-block) pairs, all
// their loads issued before any store; lane = chunk c (lane / 4) x group g
// of 8 elements (lane % 4): elements 32c + 8g .. +7 are nibble c % 2 of
// bytes 32(c / 2) + 8g .. +7, and the warp's 32 16-byte stores per
// super-block are its 512 contiguous output bytes.
constexpr int kSbPerWarp = 4;

__global__ void __launch_bounds__(256) dequant_q4K_f16_kernel(const uint8_t* __restrict__ w,
                                                              __half* __restrict__ out, int64_t nsbt,
                                                              int nsb, int K) {
    const int64_t sb0 = ((int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5) * kSbPerWarp;
    if (sb0 >= nsbt) return;
    const int lane = threadIdx.x & 31, c = lane >> 2, g = lane & 3;
    uint4 hdr[kSbPerWarp];
    uint2 q[kSbPerWarp];
#pragma unroll
    for (int j = 0; j < kSbPerWarp; ++j) {
        if (sb0 + j < nsbt) {
            const uint8_t* blk = w + (sb0 + j) * 144;
            hdr[j] = *reinterpret_cast<const uint4*>(blk);
            q[j] = *reinterpret_cast<const uint2*>(blk + 16 + 32 * (c >> 1) + 8 * g);
        }
    }
#pragma unroll
    for (int j = 0; j < kSbPerWarp; ++j) {
        const int64_t sbi = sb0 + j;   // row * nsb + sb
        if (sbi >= nsbt) break;
        const int64_t row = sbi / nsb;
        const int sb = int(sbi - row * nsb);
        const float d = __half2float(__ushort_as_half(uint16_t(hdr[j].x & 0xFFFFu)));
        const float dmin = __half2float(__ushort_as_half(uint16_t(hdr[j].x >> 16)));
        const uint32_t scw = c < 4 ? sc_lo4(hdr[j].y) : sc_hi4(hdr[j].y, hdr[j].w);
        const uint32_t mw = c < 4 ? m_lo4(hdr[j].z) : m_hi4(hdr[j].z, hdr[j].w);
        const float dsc = d * float((scw >> (8 * (c & 3))) & 0xFFu);   // exact in f32
        const float dmn = dmin * float((mw >> (8 * (c & 3))) & 0xFFu);  // exact in f32
        const uint32_t sh = 4u * uint32_t(c & 1);
        uint32_t packed[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t word = i < 2 ? q[j].x : q[j].y;
            __half e[2];
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2) {
                const uint32_t v = (word >> (8 * (2 * (i & 1) + s2) + sh)) & 0xFu;
                // d * sc * v is exact in f32: one rounding for the difference
                e[s2] = __float2half_rn(__fsub_rn(dsc * float(v), dmn));
            }
            packed[i] = uint32_t(__half_as_ushort(e[0])) | (uint32_t(__half_as_ushort(e[1])) << 16);
        }
        *reinterpret_cast<uint4*>(out + row * int64_t(K) + int64_t(sb) * 256 + 32 * c + 8 * g) =
            make_uint4(packed[0], packed[1], packed[2], packed[3]);
    }
}

// f32 -> fp16 (round to nearest even), eight per thread.
__global__ void __launch_bounds__(256) convert_f16_kernel(const float4* __restrict__ x, uint4* __restrict__ y,
                                                          int64_t n8, const float* __restrict__ tail_x,
                                                          __half* __restrict__ tail_y, int tail) {
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < n8) {
        const float4 v0 = x[2 * i], v1 = x[2 * i + 1];
        const __half2 a = __floats2half2_rn(v0.x, v0.y), b = __floats2half2_rn(v0.z, v0.w);
        const __half2 c = __floats2half2_rn(v1.x, v1.y), e = __floats2half2_rn(v1.z, v1.w);
        y[i] = make_uint4(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b),
                          *reinterpret_cast<const uint32_t*>(&c), *reinterpret_cast<const uint32_t*>(&e));
    } else if (i == n8) {
        for (int t = 0; t < tail; ++t) tail_y[t] = __float2half_rn(tail_x[t]);   // n % 8 (a multiple of 4)
    }
}

// ------------------------------------------------------------- dense GEMM
constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kStages = 4;
constexpr int kEpiWarp0 = 4, kNumEpiWarps = 8;
constexpr int kThreads = (kEpiWarp0 + kNumEpiWarps) * 32;   // 384
constexpr int kTileA = BM * 128, kTileB = BN * 128;          // 64 fp16 = 128 B per row, swizzled
constexpr int kStage = kTileA + kTileB;                      // 48 KB
constexpr int kNumAcc = 2;
constexpr uint32_t kTmemCols = 512;
static_assert(kNumAcc * BN <= int(kTmemCols), "tensor memory budget");
constexpr int kOffBar = kStages * kStage;
// barriers: full / empty per stage, acc_full / acc_empty per accumulator
constexpr int kNumBars = 2 * kStages + 2 * kNumAcc;
constexpr int kOffMisc = kOffBar + kNumBars * 8;             // tmem slot, abort flag
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr uint32_t kIdesc = idesc_f16_f32(BM, BN);

struct DenseMaps {
    CUtensorMap a, b;
};

__global__ void __launch_bounds__(kThreads, 1)
gemm_f16_kernel(const __grid_constant__ DenseMaps maps, float* __restrict__ C, int M, int N, int K,
                int* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + kOffBar;
    auto full = [&](int s) { return bar0 + 8u * uint32_t(s); };
    auto empty = [&](int s) { return bar0 + 8u * uint32_t(kStages + s); };
    auto acc_full = [&](int b) { return bar0 + 8u * uint32_t(2 * kStages + b); };
    auto acc_empty = [&](int b) { return bar0 + 8u * uint32_t(2 * kStages + kNumAcc + b); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    const AbortFlag abort_flag{sbase + kOffMisc + 4};

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles_m = (M + BM - 1) / BM, tiles_n = (N + BN - 1) / BN;
    const int num_tiles = tiles_m * tiles_n;
    const int nk = K / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < kNumAcc; ++b) {
            mbar_init(acc_full(b), 1);
            mbar_init(acc_empty(b), kNumEpiWarps);
        }
        abort_flag.set(0u);
        fence_barrier_init();
        prefetch_tmap(&maps.a);
        prefetch_tmap(&maps.b);
    }
    __syncwarp();
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            Ring<kStages> rr;
            int issued[kStages] = {};
            uint32_t par[kStages] = {};
            for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
                // tiles along N fastest: the CTAs of one wave share A rows in L2
                const int m0 = (tile / tiles_n) * BM, n0 = (tile % tiles_n) * BN;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!wait_bounded(empty(rr.slot), rr.phase ^ 1u, abort_flag, status)) goto producer_done;
                    const uint32_t st = sbase + uint32_t(rr.slot * kStage);
                    mbar_arrive_expect_tx(full(rr.slot), uint32_t(kStage));
                    tma_load_2d(st, &maps.a, full(rr.slot), kb * BK, m0);
                    tma_load_2d(st + kTileA, &maps.b, full(rr.slot), kb * BK, n0);
                    issued[rr.slot] = 1;
                    par[rr.slot] = rr.phase;
                    rr.next();
                }
            }
        producer_done:
            for (int s = 0; s < kStages; ++s)
                if (issued[s]) wait_drain(full(s), par[s], status);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            Ring<kStages> rr;
            Ring<kNumAcc> ar;
            uint32_t last_bar = 0, last_par = 0;
            for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
                if (!wait_bounded(acc_empty(ar.slot), ar.phase ^ 1u, abort_flag, status)) goto mma_done;
                tc_fence_after();
                const uint32_t d = tmem_base + uint32_t(ar.slot * BN);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!wait_bounded(full(rr.slot), rr.phase, abort_flag, status)) goto mma_done;
                    tc_fence_after();
                    const uint64_t dA = smem_desc_sw128(sbase + uint32_t(rr.slot * kStage));
                    const uint64_t dB = dA + uint64_t(kTileA >> 4);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t koff = uint64_t((kk * 32) >> 4);   // 16 fp16 = 32 bytes per step
                        mma_f16(d, dA + koff, dB + koff, kIdesc, uint32_t(kb > 0 || kk > 0));
                    }
                    mma_commit(empty(rr.slot));
                    last_bar = empty(rr.slot);
                    last_par = rr.phase;
                    rr.next();
                }
                mma_commit(acc_full(ar.slot));
                ar.next();
            }
        mma_done:
            if (last_bar) wait_drain(last_bar, last_par, status);
        }
    } else if (warp >= kEpiWarp0) {
        // ---------------------------------------------------------- epilogue
        const int ew = warp - kEpiWarp0;
        const int quarter = warp & 3;
        const int colhalf = ew >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t tlane = uint32_t(quarter * 32) << 16;
        Ring<kNumAcc> ar;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            const int m0 = (tile / tiles_n) * BM, n0 = (tile % tiles_n) * BN;
            if (!wait_bounded(acc_full(ar.slot), ar.phase, abort_flag, status)) break;
            tc_fence_after();
            const uint32_t ta = tmem_base + tlane + uint32_t(ar.slot * BN + colhalf * 128);
            const int64_t gr = int64_t(m0) + row;
            float* crow = C + gr * N;
#pragma unroll 1
            for (int j = 0; j < 4; ++j) {
                uint32_t b[32];
                tmem_ld_32x32b_x32(ta + uint32_t(32 * j), b);
                tmem_wait_ld(b);
                if (gr < M) {
                    const int gc0 = n0 + colhalf * 128 + 32 * j;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int gc = gc0 + 4 * i;   // N % 4 == 0: all four columns or none
                        if (gc < N)
                            *reinterpret_cast<float4*>(crow + gc) =
                                make_float4(__uint_as_float(b[4 * i]), __uint_as_float(b[4 * i + 1]),
                                            __uint_as_float(b[4 * i + 2]), __uint_as_float(b[4 * i + 3]));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(ar.slot));
            ar.next();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace

namespace mmq {

cudaError_t launch_dequantize_q4K_f16(const uint8_t* w, uint16_t* out, int64_t N, int64_t K, cudaStream_t s) {
    const int nsb = int(K / 256);
    const int64_t nsbt = N * nsb;
    const int64_t warps = (nsbt + kSbPerWarp - 1) / kSbPerWarp;
    const int64_t blocks = (warps * 32 + 255) / 256;
    dequant_q4K_f16_kernel<<<unsigned(blocks), 256, 0, s>>>(w, reinterpret_cast<__half*>(out), nsbt, nsb, int(K));
    return cudaGetLastError();
}

cudaError_t launch_convert_f16(const float* x, uint16_t* out, int64_t n, cudaStream_t s) {
    const int64_t n8 = n / 8;
    const int tail = int(n - n8 * 8);
    const int64_t blocks = (n8 + 1 + 255) / 256;    // + one thread for the tail
    convert_f16_kernel<<<unsigned(blocks), 256, 0, s>>>(reinterpret_cast<const float4*>(x),
                                                        reinterpret_cast<uint4*>(out), n8, x + n8 * 8,
                                                        reinterpret_cast<__half*>(out) + n8 * 8, tail);
    return cudaGetLastError();
}

int dense_gemm_check_resources() {
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
        cudaGetLastError();
        return MMQ_ERR_CUDA;
    }
    return optin >= kSmemBytes ? MMQ_OK : MMQ_ERR_RESOURCE;
}

cudaError_t launch_gemm_f16(const uint16_t* A, const uint16_t* B, float* C, int64_t M, int64_t N, int64_t K,
                            int* status, cudaStream_t s) {
    DenseMaps maps;
    if (!encode_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, uint64_t(K), uint64_t(M), uint64_t(K) * 2, BK, BM,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&maps.b, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, B, uint64_t(K), uint64_t(N), uint64_t(K) * 2, BK, BN,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    int dev = 0, nsm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(gemm_f16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes)))
        return e;
    const unsigned grid = unsigned(tiles < nsm ? tiles : nsm);
    gemm_f16_kernel<<<grid, kThreads, kSmemBytes, s>>>(maps, C, int(M), int(N), int(K), status);
    return cudaGetLastError();
}

}  // namespace mmq
