// q4_K x q8_1 GEMM for few tokens (M <= 64): bound by streaming the q4_K
// weights from HBM once.
//
// Math as in the large-M kernels (web page "20 . r15 -- f32-accumulate mma
// probe (dead end) + rank-1 term2 rescale", section 2.1; fold from page
// "21 . r16 -- Narrow kernel gets the rank-1 fold", section 2.1): per 32-k
// chunk the exact integer dot S is rescaled,
//     acc += (da * dsv) * S + dma * dmv,   dsv = d*sc, dmv = -dmin*m, dma = da*sa.
//
// Design (weights are the big operand, so they go on the MMA's 16-row side
// and the tokens on its 8-column side):
//  - CTA = 4 warps = 64 weight rows (16 per warp); a cluster of S CTAs splits
//    the 256-k super-blocks of K; the S partial sums are added in rank order
//    through distributed shared memory, so the result is deterministic and
//    no global scratch is used.
//  - Per super-block one TMA stage brings the 64 raw q4_K rows (144 B each),
//    the tokens' int8 quants (two 128-byte-swizzled boxes) and their da / sa;
//    a 4-deep ring keeps up to 4 super-blocks of weights in flight per CTA.
//  - Integer dots on mma.sync m16n8k16 with fp16 operands holding exact
//    integers (nibbles as fp16 subnormals v * 2^-24, quants via the 1024
//    bit-pattern offset), f32 accumulation: S comes out exact (times 2^-24,
//    folded into dsv).  Within a chunk both operands use the same k order:
//    thread t%4 = j of a fragment covers elements 8j + 4s + {0,2} (low
//    half) and 8j + 4s + {1,3} (high half) of step s, which makes the weight
//    fragment two masks of one 32-bit word of nibbles.
//  - The rescale runs on the MMA's f32 C fragments in registers (packed
//    f32x2 arithmetic), with dsv/dmv for the warp's two rows per thread
//    expanded once per super-block.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <mutex>

#include "mmq_internal.h"
#include "sm103_ptx.cuh"

namespace {

using namespace mmq::ptx;

constexpr int kRows = 64;                 // weight rows per CTA
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 4;
constexpr int kMaxTok = 64;               // tokens per launch (M <= 64)
constexpr int kW = kRows * 144;           // 9216 B raw q4_K rows
constexpr float kDsvScale = 16777216.0f;  // 2^24: nibbles are fp16 subnormals

struct SmallMaps {
    CUtensorMap w, a, da, sa;
};

// Stage layout for a token count padded to mp (multiple of 8):
//   [0, kW)                     raw q4_K rows
//   [aoff, aoff + 2*mp*128)      token quants: two swizzled boxes of mp x 128 B
//   [doff, doff + mp*32)         da [mp][8] f32
//   [soff, soff + mp*32)         sa [mp][8] i32
struct StageLayout {
    int aoff, doff, soff, bytes;
    __host__ __device__ static StageLayout make(int mp) {
        StageLayout L;
        L.aoff = ((kW + 1023) / 1024) * 1024;                 // swizzled boxes want 1024-B alignment
        L.doff = L.aoff + 2 * mp * 128;
        L.soff = L.doff + mp * 32;
        L.bytes = ((L.soff + mp * 32 + 1023) / 1024) * 1024;
        return L;
    }
};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// four int8 -> fp16 pairs {a0, a2}, {a1, a3}, exact (1024 offset then -1152)
__device__ __forceinline__ void cvt_a4(uint32_t w, uint32_t& h02, uint32_t& h13) {
    const uint32_t u = w ^ 0x80808080u;
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    uint32_t x = prmt(u, 0x64646464u, 0x4240u), y = prmt(u, 0x64646464u, 0x4341u);
    __half2 hx = __hsub2(*reinterpret_cast<__half2*>(&x), bias);
    __half2 hy = __hsub2(*reinterpret_cast<__half2*>(&y), bias);
    h02 = *reinterpret_cast<uint32_t*>(&hx);
    h13 = *reinterpret_cast<uint32_t*>(&hy);
}

__device__ __forceinline__ void hmma(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                     uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_shared_rank(uint32_t saddr, uint32_t rank) {
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
    return d;
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

template <int NF>
__global__ void __launch_bounds__(kThreads)
gemm_small_kernel(const __grid_constant__ SmallMaps maps, float* __restrict__ C, int M, int N,
                  int K, int split, int* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    constexpr int mp = NF * 8;
    const StageLayout L = StageLayout::make(mp);
    const uint32_t bar0 = sbase + kStages * L.bytes;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kStages * L.bytes + 8 * kStages);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, j = lane & 3;
    const int rank = int(blockIdx.x % unsigned(split));
    const int n0 = int(blockIdx.x / unsigned(split)) * kRows;
    const int nsb = K / 256;
    const int sb_begin = (nsb * rank) / split, sb_end = (nsb * (rank + 1)) / split;
    const int nmine = sb_end - sb_begin;
    const uint32_t stage_tx = uint32_t(kW + 2 * mp * 128 + 2 * mp * 32);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    __syncthreads();

    auto issue = [&](int i) {   // super-block sb_begin + i into stage i % kStages
        const int s = i % kStages;
        const uint32_t st = sbase + s * L.bytes;
        const int sb = sb_begin + i;
        mbar_arrive_expect_tx(bar0 + 8 * s, stage_tx);
        tma_load_2d(st, &maps.w, bar0 + 8 * s, sb * 144, n0);
        tma_load_2d(st + L.aoff, &maps.a, bar0 + 8 * s, sb * 256, 0);
        tma_load_2d(st + L.aoff + mp * 128, &maps.a, bar0 + 8 * s, sb * 256 + 128, 0);
        tma_load_2d(st + L.doff, &maps.da, bar0 + 8 * s, sb * 8, 0);
        tma_load_2d(st + L.soff, &maps.sa, bar0 + 8 * s, sb * 8, 0);
    };
    int issued = 0;   // stages issued (thread 0's count)
    if (threadIdx.x == 0) {
        prefetch_tmap(&maps.w);
        prefetch_tmap(&maps.a);
        for (; issued < kStages && issued < nmine; ++issued) issue(issued);
    }

    uint64_t acc[NF][2];   // per token fragment: rows g (tokens 2j, 2j+1) and g + 8
#pragma unroll
    for (int f = 0; f < NF; ++f) acc[f][0] = acc[f][1] = 0ull;

    const int r0 = warp * 16 + g;   // this thread's weight rows r0 and r0 + 8 (within the CTA)
    for (int i = 0; i < nmine; ++i) {
        const int s = i % kStages;
        // A timed-out wait raises the CTA abort flag; the loop exit below is
        // decided after a barrier, so every thread leaves at the same point.
        if (wait_bounded(bar0 + 8 * s, uint32_t((i / kStages) & 1), abort_flag, status)) {
            const uint8_t* st = smem + s * L.bytes;
            // weight-row scales for the 8 chunks: dsv (times 2^24) and dmv
            float dsv[2][8], dmv[2][8];
            uint32_t wq[2][4][2];   // [row][pair][step]: nibble words, elements 8j + 4s + 0..3
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint8_t* row = st + (r0 + 8 * h) * 144;
                const uint4 hdr = *reinterpret_cast<const uint4*>(row);
                const float d = __half2float(__ushort_as_half(uint16_t(hdr.x & 0xFFFFu))) * kDsvScale;
                const float dmin = __half2float(__ushort_as_half(uint16_t(hdr.x >> 16)));
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t sc, m;
                    if (c < 4) {
                        sc = (hdr.y >> (8 * c)) & 63u;
                        m = (hdr.z >> (8 * c)) & 63u;
                    } else {
                        const int b = 8 * (c - 4);
                        sc = ((hdr.w >> b) & 15u) | (((hdr.y >> (b + 6)) & 3u) << 4);
                        m = ((hdr.w >> (b + 4)) & 15u) | (((hdr.z >> (b + 6)) & 3u) << 4);
                    }
                    dsv[h][c] = d * float(sc);
                    dmv[h][c] = -(dmin * float(m));
                }
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const uint2 v = *reinterpret_cast<const uint2*>(row + 16 + 32 * p + 8 * j);
                    wq[h][p][0] = v.x;
                    wq[h][p][1] = v.y;
                }
            }
            const float* sda = reinterpret_cast<const float*>(st + L.doff);
            const int32_t* ssa = reinterpret_cast<const int32_t*>(st + L.soff);
            const uint8_t* sa8 = st + L.aoff;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int p = c >> 1, hsh = (c & 1) * 4;   // chunk 2p: low nibbles, 2p+1: high
                uint32_t a[2][4];
#pragma unroll
                for (int sstep = 0; sstep < 2; ++sstep) {
                    a[sstep][0] = (wq[0][p][sstep] >> hsh) & 0x000F000Fu;        // row g, elements +0, +2
                    a[sstep][1] = (wq[1][p][sstep] >> hsh) & 0x000F000Fu;        // row g + 8
                    a[sstep][2] = (wq[0][p][sstep] >> (hsh + 8)) & 0x000F000Fu;  // row g, elements +1, +3
                    a[sstep][3] = (wq[1][p][sstep] >> (hsh + 8)) & 0x000F000Fu;
                }
                const uint64_t dsv0 = pack2(dsv[0][c], dsv[0][c]), dsv1 = pack2(dsv[1][c], dsv[1][c]);
                const uint64_t dmv0 = pack2(dmv[0][c], dmv[0][c]), dmv1 = pack2(dmv[1][c], dmv[1][c]);
#pragma unroll
                for (int f = 0; f < NF; ++f) {
                    // token g of fragment f: 8 bytes at chunk c, offset 8j (128-B swizzled box c / 4)
                    const int tok = 8 * f + g;
                    const uint32_t gran = uint32_t(((c & 3) * 2 + (j >> 1)) ^ (tok & 7));
                    const uint2 q = *reinterpret_cast<const uint2*>(
                        sa8 + (c >> 2) * mp * 128 + tok * 128 + (gran << 4) + (j & 1) * 8);
                    uint32_t b00, b01, b10, b11;
                    cvt_a4(q.x, b00, b01);
                    cvt_a4(q.y, b10, b11);
                    float sc4[4] = {0.f, 0.f, 0.f, 0.f};
                    hmma(sc4, a[0][0], a[0][1], a[0][2], a[0][3], b00, b01);
                    hmma(sc4, a[1][0], a[1][1], a[1][2], a[1][3], b10, b11);
                    // C fragment: (row g, tokens 8f + 2j, +1) and (row g + 8, same tokens)
                    const int t0 = 8 * f + 2 * j;
                    const float da0 = sda[t0 * 8 + c], da1 = sda[(t0 + 1) * 8 + c];
                    const uint64_t da2 = pack2(da0, da1);
                    const uint64_t dma2 =
                        pack2(da0 * float(ssa[t0 * 8 + c]), da1 * float(ssa[(t0 + 1) * 8 + c]));
                    const uint64_t s01 = pack2(sc4[0], sc4[1]), s23 = pack2(sc4[2], sc4[3]);
                    acc[f][0] = ffma2(dma2, dmv0, ffma2(fmul2(da2, dsv0), s01, acc[f][0]));
                    acc[f][1] = ffma2(dma2, dmv1, ffma2(fmul2(da2, dsv1), s23, acc[f][1]));
                }
            }
        }
        __syncthreads();   // every warp is done reading stage s
        if (*abort_flag) break;
        if (threadIdx.x == 0 && issued < nmine) {
            fence_proxy_async_smem();
            issue(issued);
            ++issued;
        }
    }
    if (threadIdx.x == 0) {
        // let every copy issued land before stage memory is reused or the CTA exits
        for (int i2 = (issued > kStages ? issued - kStages : 0); i2 < issued; ++i2)
            wait_drain(bar0 + 8 * (i2 % kStages), uint32_t((i2 / kStages) & 1), status);
    }
    __syncthreads();

    // ---- reduce the split-K partials across the cluster in rank order
    float* part = reinterpret_cast<float*>(smem);   // [NF][2][2] per thread, 16*NF B
    const uint32_t my_off = uint32_t(threadIdx.x) * (NF * 4) * 4;
    if (split > 1) {
#pragma unroll
        for (int f = 0; f < NF; ++f) {
            part[(threadIdx.x * NF + f) * 4 + 0] = lo_f(acc[f][0]);
            part[(threadIdx.x * NF + f) * 4 + 1] = hi_f(acc[f][0]);
            part[(threadIdx.x * NF + f) * 4 + 2] = lo_f(acc[f][1]);
            part[(threadIdx.x * NF + f) * 4 + 3] = hi_f(acc[f][1]);
        }
        cluster_sync();
        if (rank == 0) {
            for (int r = 1; r < split; ++r) {
                const uint32_t remote = map_shared_rank(sbase + my_off, uint32_t(r));
#pragma unroll
                for (int f = 0; f < NF; ++f) {
                    const float x0 = ld_dsmem_f32(remote + (f * 4 + 0) * 4);
                    const float x1 = ld_dsmem_f32(remote + (f * 4 + 1) * 4);
                    const float x2 = ld_dsmem_f32(remote + (f * 4 + 2) * 4);
                    const float x3 = ld_dsmem_f32(remote + (f * 4 + 3) * 4);
                    acc[f][0] = pack2(lo_f(acc[f][0]) + x0, hi_f(acc[f][0]) + x1);
                    acc[f][1] = pack2(lo_f(acc[f][1]) + x2, hi_f(acc[f][1]) + x3);
                }
            }
        }
        cluster_sync();   // remote partials stay alive until rank 0 has read them
    }
    if (rank == 0) {
#pragma unroll
        for (int f = 0; f < NF; ++f) {
            const int t0 = 8 * f + 2 * j;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = n0 + r0 + 8 * h;
                if (row < N) {
                    if (t0 < M) C[int64_t(t0) * N + row] = lo_f(acc[f][h]);
                    if (t0 + 1 < M) C[int64_t(t0 + 1) * N + row] = hi_f(acc[f][h]);
                }
            }
        }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_small() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

bool encode(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
            uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
    auto fn = get_encode_small();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NF>
cudaError_t launch_nf(const SmallMaps& maps, float* C, int64_t M, int64_t N, int64_t K, int* status,
                      cudaStream_t s) {
    const StageLayout L = StageLayout::make(NF * 8);
    const int smem = kStages * L.bytes + 8 * kStages + 16 + 1024;
    int dev = 0, nsm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    const int64_t row_tiles = (N + kRows - 1) / kRows;
    const int nsb = int(K / 256);
    // split K over a cluster so that about two CTAs land on every SM
    int split = 1;
    while (split < 8 && row_tiles * split * 2 <= 2 * int64_t(nsm) && split * 2 <= nsb) split *= 2;
    auto k = gemm_small_kernel<NF>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(row_tiles * split));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = size_t(smem);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(split);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, maps, C, int(M), int(N), int(K), split, status);
}

}  // namespace

namespace mmq {

cudaError_t launch_gemm_small_m(mmq_q8_1_t aq, const uint8_t* w, float* C, int64_t M, int64_t N,
                                int64_t K, int* status, cudaStream_t s) {
    if (M > kMaxTok) return cudaErrorInvalidValue;
    const int nf = int((M + 7) / 8);
    const uint32_t mp = uint32_t(nf * 8);
    const uint64_t nb = uint64_t(K / 32), nsb = uint64_t(K / 256);
    SmallMaps maps;
    if (!encode(&maps.w, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, nsb * 144, uint64_t(N), nsb * 144, 144,
                kRows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, aq.qs, uint64_t(K), uint64_t(M), uint64_t(K),
                128, mp, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode(&maps.da, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, aq.da, nb, uint64_t(M), nb * 4, 8, mp,
                CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode(&maps.sa, CU_TENSOR_MAP_DATA_TYPE_INT32, aq.sa, nb, uint64_t(M), nb * 4, 8, mp,
                CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    switch (nf) {
        case 1: return launch_nf<1>(maps, C, M, N, K, status, s);
        case 2: return launch_nf<2>(maps, C, M, N, K, status, s);
        case 3: return launch_nf<3>(maps, C, M, N, K, status, s);
        case 4: return launch_nf<4>(maps, C, M, N, K, status, s);
        case 5: return launch_nf<5>(maps, C, M, N, K, status, s);
        case 6: return launch_nf<6>(maps, C, M, N, K, status, s);
        case 7: return launch_nf<7>(maps, C, M, N, K, status, s);
        default: return launch_nf<8>(maps, C, M, N, K, status, s);
    }
}

}  // namespace mmq
