// q4_K x q8_1 GEMM on the 5th-generation tensor cores (tcgen05) of sm_103a.
//
// Math (web page "20 . r15 -- f32-accumulate mma probe (dead end) + rank-1
// term2 rescale", section 2.1): for every 32-k chunk c the exact integer dot
// S_ij = sum_k a_ik * v_jk (|S| <= 32*127*15, section 2.3) is rescaled into
// f32:  acc_ij += (da_ic * dsv_jc) * S_ij + dma_ic * dmv_jc, dsv = d*sc,
// dmv = -dmin*m, dma = da*sa once per token row and chunk (the rank-1 fold,
// page "21 . r16 -- Narrow kernel gets the rank-1 fold", section 2.1).
//
// sm_103a has no integer kind for tcgen05.mma, so the integers go through
// kind::f16: every quant a in [-127, 127] and nibble v in [0, 15] is an exact
// fp16 value, every product and partial sum is an integer below 2^24, so the
// f32 accumulator in tensor memory holds S exactly (checked bit for bit by the
// S dump).  The nibbles are written as fp16 subnormals v * 2^-24 (just the
// zero-extended nibble bits, no arithmetic); the 2^24 is folded into dsv.
//
// One CTA per SM, persistent over 128 (tokens) x 128 (weight rows) tiles,
// warp-specialised (16 warps; setmaxnreg moves registers to the epilogue):
//   warp 0      TMA producer: per 256-k super-block the raw int8 A tile (two
//               128-byte-swizzled boxes), the raw 144-byte q4_K rows, and the
//               da / sa slices, all zero-filled past M / N.
//   warp 1      MMA issuer (one thread): per chunk two K=16 MMAs into one of
//               four 128-column f32 tensor-memory buffers.
//   warps 2-3   scale tables per super-block: dsv/dmv per weight row and
//               chunk, (da, dma = da*sa) per token row and chunk.
//   warps 4-7   operand converters: int8 -> fp16 (exact, via the 1024-offset
//               bit pattern and one fp16 subtraction) and nibble -> fp16 into
//               the 128-byte-swizzled K-major layout, one 64-k chunk pair at a
//               time, one row per thread.
//   warps 8-15  epilogue: per chunk tcgen05.ld of the S tile (16x256b shape:
//               each thread holds 4 rows x 16 columns, so one column-scale load
//               serves four rows), the rescale with the fold in packed f32x2
//               arithmetic, the next tensor-memory load issued before the
//               current part is computed; C stored at the end of a tile.
// Within a chunk the k order of both operands is permuted identically
// (groups of four as 0,2,1,3) so that both unpacks are plain byte/nibble
// moves; a dot product does not depend on the order of its terms.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <mutex>

#include "mmq_internal.h"
#include "sm103_ptx.cuh"

namespace {

using namespace mmq::ptx;

constexpr int BM = 128, BN = 128;
constexpr int kNumRaw = 2, kNumScl = 2, kNumOp = 2, kNumTm = 4;
constexpr int kSclWarp0 = 2, kNumSclWarps = 2, kConvWarp0 = 4, kNumConvWarps = 4;
constexpr int kEpiWarp0 = 8, kNumEpiWarps = 8;
constexpr int kThreads = (kEpiWarp0 + kNumEpiWarps) * 32;   // 512
// Register split: warpgroups 0-1 (producer, MMA, scale tables, converters)
// give up registers to warpgroups 2-3 (epilogue).  Launch budget: 512 x 128.
constexpr uint32_t kRegsLow = 72, kRegsHigh = 184, kRegsLaunch = 128;
static_assert(256 * kRegsLow + 256 * kRegsHigh <= kThreads * kRegsLaunch, "register split");
constexpr uint32_t kTmemCols = 512;                          // kNumTm x BN

// Shared memory map (offsets from a 1024-byte aligned base).
constexpr int kRawASub = BM * 128;                   // 16 KB: 128 rows x 128 B, swizzled
constexpr int kRawA = 2 * kRawASub;                  // 256 k of int8
constexpr int kRawB = BN * 144;                      // raw q4_K rows
constexpr int kRawDa = BM * 8 * 4;                   // da [128][8] f32
constexpr int kRawSa = BM * 8 * 4;                   // sa [128][8] i32
constexpr int kOffRawB = kRawA, kOffRawDa = kRawA + kRawB, kOffRawSa = kOffRawDa + kRawDa;
constexpr int kRawStage = kOffRawSa + kRawSa;        // 58 KB: everything one super-block needs from HBM
constexpr int kSclCol = 8 * BN * 8;                  // [8 chunks][64 column pairs] float4
                                                     //   {dsv_2p, dsv_2p+1, dmv_2p, dmv_2p+1}
constexpr int kSclRow = 8 * BM * 8;                  // [8 chunks][128 rows] float2 {da, da*sa}
constexpr int kOffSclCol = 0;
constexpr int kOffSclRow = kOffSclCol + kSclCol;
constexpr int kSclStage = kOffSclRow + kSclRow;      // 16 KB of scale tables (no copies land here)
constexpr int kOpTile = 128 * 128;                   // 128 rows x 64 fp16 (128 B), swizzled
constexpr int kOpStage = 2 * kOpTile;                // A + B
constexpr int kOffRaw = 0;
constexpr int kOffScl = kOffRaw + kNumRaw * kRawStage;
constexpr int kOffOp = kOffScl + kNumScl * kSclStage;
constexpr int kOffBar = kOffOp + kNumOp * kOpStage;
// barriers: raw_full, raw_empty, scl_col, scl_empty, op_full, op_empty, tm_full, tm_empty
constexpr int kNumBars = 2 * kNumRaw + 2 * kNumScl + 2 * kNumOp + 2 * kNumTm;
constexpr int kOffMisc = kOffBar + kNumBars * 8;     // tmem slot, abort flag
constexpr int kSmemBytes = kOffMisc + 16 + 1024;     // + alignment slack
static_assert(kOffOp % 1024 == 0, "operand tiles need 1024-byte alignment");
static_assert(kRawStage % 1024 == 0 && kSclStage % 1024 == 0, "stage alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kRawTx = kRawStage;
constexpr uint32_t kIdesc = idesc_f16_f32(BM, BN);
constexpr float kDsvScale = 16777216.0f;             // 2^24: nibbles are fp16 subnormals

struct TmaMaps {
    CUtensorMap a, b, da, sa;
};

struct Bars {
    uint32_t base;
    __device__ uint32_t raw_full(int s) const { return base + 8 * s; }
    __device__ uint32_t raw_empty(int s) const { return base + 8 * (kNumRaw + s); }
    __device__ uint32_t scl_col(int s) const { return base + 8 * (2 * kNumRaw + s); }
    __device__ uint32_t scl_empty(int s) const { return base + 8 * (2 * kNumRaw + kNumScl + s); }
    __device__ uint32_t op_full(int s) const { return base + 8 * (2 * kNumRaw + 2 * kNumScl + s); }
    __device__ uint32_t op_empty(int s) const {
        return base + 8 * (2 * kNumRaw + 2 * kNumScl + kNumOp + s);
    }
    __device__ uint32_t tm_full(int s) const {
        return base + 8 * (2 * kNumRaw + 2 * kNumScl + 2 * kNumOp + s);
    }
    __device__ uint32_t tm_empty(int s) const {
        return base + 8 * (2 * kNumRaw + 2 * kNumScl + 2 * kNumOp + kNumTm + s);
    }
};

// Ring position: slot index and the parity of the current pass over the ring.
template <int N>
struct Ring {
    int slot = 0;
    uint32_t phase = 0;
    __device__ void next() {
        if (++slot == N) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Four int8 (a0 a1 a2 a3) -> fp16 pairs {a0, a2} and {a1, a3}, exact:
// 0x6400 | (a ^ 0x80) is the fp16 1024 + (a + 128); subtracting 1152 leaves a.
__device__ __forceinline__ void cvt_a4(uint32_t w, uint32_t& h02, uint32_t& h13) {
    const uint32_t u = w ^ 0x80808080u;
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    __half2 x = __hsub2(*reinterpret_cast<const __half2*>(&(h02 = prmt(u, 0x64646464u, 0x4240u))), bias);
    __half2 y = __hsub2(*reinterpret_cast<const __half2*>(&(h13 = prmt(u, 0x64646464u, 0x4341u))), bias);
    h02 = *reinterpret_cast<uint32_t*>(&x);
    h13 = *reinterpret_cast<uint32_t*>(&y);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_shared_rank(uint32_t saddr, uint32_t rank) {
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
    return d;
}
__device__ __forceinline__ float4 ld_dsmem_v4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Epilogue thread's 4 rows x 16 columns of the 128x128 tile (m0, n0) -> C.
__device__ __forceinline__ void store_tile(float* C, const uint64_t (&acc)[4][8], int M, int N, int m0,
                                           int n0, int quarter, int colhalf, int tq, int tr4) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int64_t gr = int64_t(m0) + quarter * 32 + tq + 8 * k;
        if (gr < M) {
            float* crow = C + gr * N;
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                const int gc = n0 + colhalf * 64 + 8 * g + 2 * tr4;
                if (gc < N)
                    *reinterpret_cast<float2*>(crow + gc) = make_float2(lo_f(acc[k][g]), hi_f(acc[k][g]));
            }
        }
    }
}

template <bool kDump>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const __grid_constant__ TmaMaps maps, float* __restrict__ C,
               int32_t* __restrict__ S, int M, int N, int K, int split, int* status, int inject_timeout) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const Bars bars{sbase + kOffBar};
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nsb = K / 256;
    const int tiles_m = (M + BM - 1) / BM, tiles_n = (N + BN - 1) / BN;
    const int num_tiles = tiles_m * tiles_n;
    // Persistent mode (split == 1): CTAs stride over all tiles and K.  Split
    // mode: a cluster of `split` CTAs shares one tile, rank r takes
    // super-blocks [nsb*r/split, nsb*(r+1)/split), and rank 0 adds the
    // partial sums in rank order.
    const int rank = split > 1 ? int(blockIdx.x % unsigned(split)) : 0;
    const int tile_first = split > 1 ? int(blockIdx.x / unsigned(split)) : int(blockIdx.x);
    const int tile_step = split > 1 ? num_tiles : int(gridDim.x);
    const int sb_lo = (nsb * rank) / split, sb_hi = (nsb * (rank + 1)) / split;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kNumRaw; ++s) {
            mbar_init(bars.raw_full(s), 1);
            mbar_init(bars.raw_empty(s), kNumConvWarps + kNumSclWarps);
        }
        for (int s = 0; s < kNumScl; ++s) {
            mbar_init(bars.scl_col(s), kNumSclWarps);
            mbar_init(bars.scl_empty(s), kNumEpiWarps);
        }
        for (int s = 0; s < kNumOp; ++s) {
            mbar_init(bars.op_full(s), kNumConvWarps);
            mbar_init(bars.op_empty(s), 1);
        }
        for (int s = 0; s < kNumTm; ++s) {
            mbar_init(bars.tm_full(s), 1);
            mbar_init(bars.tm_empty(s), kNumEpiWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
        prefetch_tmap(&maps.a);
        prefetch_tmap(&maps.b);
        prefetch_tmap(&maps.da);
        prefetch_tmap(&maps.sa);
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

    if (warp < kEpiWarp0) {
    setmaxnreg_dec<kRegsLow>();
    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            Ring<kNumRaw> rr;
            int raw_issued[kNumRaw] = {};
            uint32_t raw_par[kNumRaw] = {};
            bool first = true;
            for (int tile = tile_first; tile < num_tiles; tile += tile_step) {
                const int m0 = (tile / tiles_n) * BM, n0 = (tile % tiles_n) * BN;
                for (int sb = sb_lo; sb < sb_hi; ++sb) {
                    if (!wait_bounded(bars.raw_empty(rr.slot), rr.phase ^ 1u, abort_flag, status))
                        goto producer_done;
                    const uint32_t raw = sbase + kOffRaw + rr.slot * kRawStage;
                    if (!(first && inject_timeout)) {   // test hook: withhold this arrival
                        const uint32_t fb = bars.raw_full(rr.slot);
                        mbar_arrive_expect_tx(fb, kRawTx);
                        tma_load_2d(raw, &maps.a, fb, sb * 256, m0);
                        tma_load_2d(raw + kRawASub, &maps.a, fb, sb * 256 + 128, m0);
                        tma_load_2d(raw + kOffRawB, &maps.b, fb, sb * 144, n0);
                        tma_load_2d(raw + kOffRawDa, &maps.da, fb, sb * 8, m0);
                        tma_load_2d(raw + kOffRawSa, &maps.sa, fb, sb * 8, m0);
                        raw_issued[rr.slot] = 1;
                        raw_par[rr.slot] = rr.phase;
                    }
                    first = false;
                    rr.next();
                }
            }
        producer_done:
            // Let every copy already issued land before the CTA can exit.
            for (int s = 0; s < kNumRaw; ++s)
                if (raw_issued[s]) wait_drain(bars.raw_full(s), raw_par[s], status);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            Ring<kNumOp> orr;
            Ring<kNumTm> tr;
            int issued = 0;
            int last_slot = 0;
            uint32_t last_par = 0;
            for (int tile = tile_first; tile < num_tiles; tile += tile_step) {
                for (int sb = sb_lo; sb < sb_hi; ++sb) {
                    for (int q = 0; q < 4; ++q) {
                        if (!wait_bounded(bars.op_full(orr.slot), orr.phase, abort_flag, status))
                            goto mma_done;
                        tc_fence_after();
                        const uint32_t opA = sbase + kOffOp + orr.slot * kOpStage;
                        const uint32_t opB = opA + kOpTile;
                        for (int h = 0; h < 2; ++h) {
                            if (!wait_bounded(bars.tm_empty(tr.slot), tr.phase ^ 1u, abort_flag, status))
                                goto mma_done;
                            tc_fence_after();
                            const uint32_t d = tmem_base + uint32_t(tr.slot * BN);
#pragma unroll
                            for (int kk = 0; kk < 2; ++kk) {
                                const uint32_t koff = uint32_t(h * 64 + kk * 32);   // bytes within the 128-B row
                                mma_f16(d, smem_desc_sw128(opA + koff), smem_desc_sw128(opB + koff),
                                        kIdesc, uint32_t(kk));
                            }
                            mma_commit(bars.tm_full(tr.slot));
                            issued = 1;
                            last_slot = tr.slot;
                            last_par = tr.phase;
                            tr.next();
                        }
                        mma_commit(bars.op_empty(orr.slot));
                        orr.next();
                    }
                }
            }
        mma_done:
            if (issued) wait_drain(bars.tm_full(last_slot), last_par, status);
        }
    } else if (warp < kConvWarp0) {
        // ------------------------------------------------------ scale tables
        // Weight rows: dsv = d*sc (times 2^24 for the subnormal nibbles) and
        // dmv = -dmin*m, exact in f32, as column pairs {dsv0, dsv1, dmv0, dmv1};
        // token rows: {da, dma = da*sa}, the rank-1 fold once per row and chunk.
        const int ts = threadIdx.x - kSclWarp0 * 32;   // 0..63: rows ts and ts + 64
        Ring<kNumRaw> rr;
        Ring<kNumScl> sr;
        for (int tile = tile_first; tile < num_tiles; tile += tile_step) {
            for (int sb = sb_lo; sb < sb_hi; ++sb) {
                if (!wait_bounded(bars.raw_full(rr.slot), rr.phase, abort_flag, status)) goto scl_done;
                if (!wait_bounded(bars.scl_empty(sr.slot), sr.phase ^ 1u, abort_flag, status)) goto scl_done;
                {
                    const uint32_t rawB = sbase + kOffRaw + rr.slot * kRawStage + kOffRawB;
                    const uint32_t rawDa = sbase + kOffRaw + rr.slot * kRawStage + kOffRawDa;
                    const uint32_t rawSa = sbase + kOffRaw + rr.slot * kRawStage + kOffRawSa;
                    float* colf = reinterpret_cast<float*>(smem + kOffScl + sr.slot * kSclStage + kOffSclCol);
                    float2* row2 = reinterpret_cast<float2*>(smem + kOffScl + sr.slot * kSclStage + kOffSclRow);
#pragma unroll
                    for (int rh = 0; rh < 2; ++rh) {
                        const int t = ts + 64 * rh;
                        const uint4 hdr = ld_shared_v4(rawB + t * 144);   // d, dmin, s[0..11]
                        const float d = __half2float(__ushort_as_half(uint16_t(hdr.x & 0xFFFFu)));
                        const float dmin = __half2float(__ushort_as_half(uint16_t(hdr.x >> 16)));
                        const uint32_t s0 = hdr.y, s1 = hdr.z, s2 = hdr.w;   // s[0..3], s[4..7], s[8..11]
                        float* cp = colf + (t >> 1) * 4 + (t & 1);
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            uint32_t sc, m;
                            if (c < 4) {
                                sc = (s0 >> (8 * c)) & 63u;
                                m = (s1 >> (8 * c)) & 63u;
                            } else {
                                const int b = 8 * (c - 4);
                                sc = ((s2 >> b) & 15u) | (((s0 >> (b + 6)) & 3u) << 4);
                                m = ((s2 >> (b + 4)) & 15u) | (((s1 >> (b + 6)) & 3u) << 4);
                            }
                            cp[c * (BN * 2)] = d * float(sc) * kDsvScale;
                            cp[c * (BN * 2) + 2] = -(dmin * float(m));
                        }
                        const uint4 da0 = ld_shared_v4(rawDa + t * 32), da1 = ld_shared_v4(rawDa + t * 32 + 16);
                        const uint4 sa0 = ld_shared_v4(rawSa + t * 32);
                        const uint4 sa1 = ld_shared_v4(rawSa + t * 32 + 16);
                        const uint32_t dav[8] = {da0.x, da0.y, da0.z, da0.w, da1.x, da1.y, da1.z, da1.w};
                        const uint32_t sav[8] = {sa0.x, sa0.y, sa0.z, sa0.w, sa1.x, sa1.y, sa1.z, sa1.w};
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const float da = __uint_as_float(dav[c]);
                            row2[c * BM + t] = make_float2(da, da * float(int32_t(sav[c])));
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bars.scl_col(sr.slot));
                    mbar_arrive(bars.raw_empty(rr.slot));
                }
                sr.next();
                rr.next();
            }
        }
    scl_done:;
    } else if (warp < kEpiWarp0) {
        // -------------------------------------------------------- converters
        const int t = threadIdx.x - kConvWarp0 * 32;   // 0..127: this thread's row
        const int sw = t & 7;
        Ring<kNumRaw> rr;
        Ring<kNumOp> orr;
        for (int tile = tile_first; tile < num_tiles; tile += tile_step) {
            for (int sb = sb_lo; sb < sb_hi; ++sb) {
                if (!wait_bounded(bars.raw_full(rr.slot), rr.phase, abort_flag, status)) goto conv_done;
                const uint32_t raw = sbase + kOffRaw + rr.slot * kRawStage;
                const uint32_t rawB = raw + kOffRawB + t * 144 + 16;
                for (int q = 0; q < 4; ++q) {   // chunk pair q = chunks 2q, 2q+1
                    if (!wait_bounded(bars.op_empty(orr.slot), orr.phase ^ 1u, abort_flag, status))
                        goto conv_done;
                    const uint32_t opA = sbase + kOffOp + orr.slot * kOpStage + t * 128;
                    const uint32_t opB = opA + kOpTile;
                    uint4 wa[4], wb[2];
#pragma unroll
                    for (int g = 0; g < 4; ++g)   // A: 64 int8 of the pair, granule (q&1)*4+g of a swizzled sub-tile
                        wa[g] = ld_shared_v4(raw + (q >> 1) * kRawASub + t * 128 + ((((q & 1) * 4 + g) ^ sw) << 4));
#pragma unroll
                    for (int G = 0; G < 2; ++G)   // B: 32 bytes of nibbles, chunk 2q low / 2q+1 high
                        wb[G] = ld_shared_v4(rawB + 32 * q + 16 * G);
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        uint32_t p0, p1, p2, p3, p4, p5, p6, p7;
                        cvt_a4(wa[g].x, p0, p1);
                        cvt_a4(wa[g].y, p2, p3);
                        cvt_a4(wa[g].z, p4, p5);
                        cvt_a4(wa[g].w, p6, p7);
                        st_shared_v4(opA + (((2 * g) ^ sw) << 4), p0, p1, p2, p3);
                        st_shared_v4(opA + (((2 * g + 1) ^ sw) << 4), p4, p5, p6, p7);
                    }
#pragma unroll
                    for (int G = 0; G < 2; ++G) {
                        const uint32_t ww[4] = {wb[G].x, wb[G].y, wb[G].z, wb[G].w};
                        uint32_t lo[8], hi[8];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            lo[2 * u] = ww[u] & 0x000F000Fu;            // {e0, e2} low nibbles
                            lo[2 * u + 1] = (ww[u] >> 8) & 0x000F000Fu; // {e1, e3}
                            hi[2 * u] = (ww[u] >> 4) & 0x000F000Fu;
                            hi[2 * u + 1] = (ww[u] >> 12) & 0x000F000Fu;
                        }
                        st_shared_v4(opB + (((2 * G) ^ sw) << 4), lo[0], lo[1], lo[2], lo[3]);
                        st_shared_v4(opB + (((2 * G + 1) ^ sw) << 4), lo[4], lo[5], lo[6], lo[7]);
                        st_shared_v4(opB + (((4 + 2 * G) ^ sw) << 4), hi[0], hi[1], hi[2], hi[3]);
                        st_shared_v4(opB + (((5 + 2 * G) ^ sw) << 4), hi[4], hi[5], hi[6], hi[7]);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars.op_full(orr.slot));
                    orr.next();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.raw_empty(rr.slot));
                rr.next();
            }
        }
    conv_done:;
    }
    if (split > 1) {   // every thread of every CTA in the cluster takes both barriers
        cluster_sync_all();
        cluster_sync_all();
    }
    } else {
        setmaxnreg_inc<kRegsHigh>();
        // ---------------------------------------------------------- epilogue
        // Thread t of a warp holds, per chunk, rows quarter*32 + t/4 + 8k
        // (k = 0..3) x columns colhalf*64 + 8g + 2(t%4) + {0,1} (g = 0..7).
        // A chunk is read from tensor memory in two parts (lanes +0..15 give
        // rows k = 0,1; lanes +16..31 give k = 2,3); the load of the next part
        // is in flight while the current one is computed.
        const int ew = warp - kEpiWarp0;
        const int quarter = warp & 3;                  // tensor-memory lanes this warp may read
        const int colhalf = ew >> 2;                   // columns [64*colhalf, +64)
        const int tq = lane >> 2, tr4 = lane & 3;
        const uint32_t tlane0 = uint32_t(quarter * 32) << 16, tlane1 = uint32_t(quarter * 32 + 16) << 16;
        Ring<kNumScl> sr;
        Ring<kNumTm> tr;
        uint64_t acc[4][8];
        for (int tile = tile_first; tile < num_tiles; tile += tile_step) {
            const int m0 = (tile / tiles_n) * BM, n0 = (tile % tiles_n) * BN;
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
                for (int g = 0; g < 8; ++g) acc[k][g] = 0ull;
            uint32_t b0[32], b1[32];
            // prologue: first part of the tile's first chunk
            if (!wait_bounded(bars.scl_col(sr.slot), sr.phase, abort_flag, status)) goto epi_done;
            if (!wait_bounded(bars.tm_full(tr.slot), tr.phase, abort_flag, status)) goto epi_done;
            tc_fence_after();
            tmem_ld_16x256b_x8(tmem_base + tlane0 + uint32_t(tr.slot * BN + colhalf * 64), b0);
            tmem_wait_ld();
            for (int sb = sb_lo; sb < sb_hi; ++sb) {
                const uint8_t* scl = smem + kOffScl + sr.slot * kSclStage;
                const float4* col4 = reinterpret_cast<const float4*>(scl + kOffSclCol);
                const float2* row2 = reinterpret_cast<const float2*>(scl + kOffSclRow);
                for (int c = 0; c < 8; ++c) {
                    float4 cs[8];
#pragma unroll
                    for (int g = 0; g < 8; ++g) cs[g] = col4[c * 64 + colhalf * 32 + 4 * g + tr4];
                    float2 rr[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) rr[k] = row2[c * BM + quarter * 32 + tq + 8 * k];
                    // second part of this chunk, then compute the first part
                    tmem_ld_16x256b_x8(tmem_base + tlane1 + uint32_t(tr.slot * BN + colhalf * 64), b1);
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        if (kDump) {
                            const int64_t gr = int64_t(m0) + quarter * 32 + tq + 8 * kk;
#pragma unroll
                            for (int g = 0; g < 8; ++g)
#pragma unroll
                                for (int e = 0; e < 2; ++e) {
                                    const int64_t gc = int64_t(n0) + colhalf * 64 + 8 * g + 2 * tr4 + e;
                                    if (gr < M && gc < N)
                                        S[(gr * N + gc) * (K / 32) + sb * 8 + c] =
                                            int32_t(__uint_as_float(b0[4 * g + 2 * kk + e]) * kDsvScale);
                                }
                        } else {
                            const uint64_t da2 = pack2(rr[kk].x, rr[kk].x), dma2 = pack2(rr[kk].y, rr[kk].y);
#pragma unroll
                            for (int g = 0; g < 8; ++g) {
                                const uint64_t c1 = fmul2(da2, pack2(cs[g].x, cs[g].y));
                                const uint64_t a = ffma2(c1, pack2u(b0[4 * g + 2 * kk], b0[4 * g + 2 * kk + 1]), acc[kk][g]);
                                acc[kk][g] = ffma2(dma2, pack2(cs[g].z, cs[g].w), a);
                            }
                        }
                    }
                    tmem_wait_ld();
                    // the whole S tile of this chunk is in registers: hand the buffer back
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars.tm_empty(tr.slot));
                    tr.next();
                    const bool last_in_sb = (c == 7);
                    const bool has_next = !(last_in_sb && sb == sb_hi - 1);
                    if (last_in_sb) {   // scale tables of this super-block no longer needed
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bars.scl_empty(sr.slot));
                        sr.next();
                    }
                    if (has_next) {
                        if (last_in_sb &&
                            !wait_bounded(bars.scl_col(sr.slot), sr.phase, abort_flag, status))
                            goto epi_done;
                        if (!wait_bounded(bars.tm_full(tr.slot), tr.phase, abort_flag, status)) goto epi_done;
                        tc_fence_after();
                        tmem_ld_16x256b_x8(tmem_base + tlane0 + uint32_t(tr.slot * BN + colhalf * 64), b0);
                    }
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        const int k = 2 + kk;
                        if (kDump) {
                            const int64_t gr = int64_t(m0) + quarter * 32 + tq + 8 * k;
#pragma unroll
                            for (int g = 0; g < 8; ++g)
#pragma unroll
                                for (int e = 0; e < 2; ++e) {
                                    const int64_t gc = int64_t(n0) + colhalf * 64 + 8 * g + 2 * tr4 + e;
                                    if (gr < M && gc < N)
                                        S[(gr * N + gc) * (K / 32) + sb * 8 + c] =
                                            int32_t(__uint_as_float(b1[4 * g + 2 * kk + e]) * kDsvScale);
                                }
                        } else {
                            const uint64_t da2 = pack2(rr[k].x, rr[k].x), dma2 = pack2(rr[k].y, rr[k].y);
#pragma unroll
                            for (int g = 0; g < 8; ++g) {
                                const uint64_t c1 = fmul2(da2, pack2(cs[g].x, cs[g].y));
                                const uint64_t a = ffma2(c1, pack2u(b1[4 * g + 2 * kk], b1[4 * g + 2 * kk + 1]), acc[k][g]);
                                acc[k][g] = ffma2(dma2, pack2(cs[g].z, cs[g].w), a);
                            }
                        }
                    }
                    if (has_next) tmem_wait_ld();
                }
            }
            if (!kDump && split == 1) store_tile(C, acc, M, N, m0, n0, quarter, colhalf, tq, tr4);
        }
    epi_done:;
        if (split > 1) {
            // Each rank leaves its partial tile in its own (now idle) staging
            // memory; rank 0 pulls ranks 1..split-1 in order and stores C.
            const int e = threadIdx.x - kEpiWarp0 * 32;   // 0..255
            float4* mine = reinterpret_cast<float4*>(smem + kOffRaw) + e * 16;
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
                for (int g = 0; g < 8; g += 2)
                    mine[k * 4 + g / 2] = make_float4(lo_f(acc[k][g]), hi_f(acc[k][g]),
                                                      lo_f(acc[k][g + 1]), hi_f(acc[k][g + 1]));
            cluster_sync_all();
            if (rank == 0 && !kDump) {
                for (int r = 1; r < split; ++r) {
                    const uint32_t remote = map_shared_rank(sbase + kOffRaw + uint32_t(e) * 256u, uint32_t(r));
#pragma unroll
                    for (int k = 0; k < 4; ++k)
#pragma unroll
                        for (int g = 0; g < 8; g += 2) {
                            const float4 v = ld_dsmem_v4(remote + uint32_t(k * 4 + g / 2) * 16u);
                            acc[k][g] = pack2(lo_f(acc[k][g]) + v.x, hi_f(acc[k][g]) + v.y);
                            acc[k][g + 1] = pack2(lo_f(acc[k][g + 1]) + v.z, hi_f(acc[k][g + 1]) + v.w);
                        }
                }
                const int m0 = (tile_first / tiles_n) * BM, n0 = (tile_first % tiles_n) * BN;
                store_tile(C, acc, M, N, m0, n0, quarter, colhalf, tq, tr4);
            }
            cluster_sync_all();   // remote partials stay alive until rank 0 has read them
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

// ------------------------------------------------------------------- host
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
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

bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
               uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle sw) {
    auto fn = get_encode();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace mmq {

int tc_gemm_check_resources() {
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
        cudaGetLastError();
        return MMQ_ERR_CUDA;
    }
    return optin >= kSmemBytes ? MMQ_OK : MMQ_ERR_RESOURCE;
}

cudaError_t launch_gemm_tc(mmq_q8_1_t aq, const uint8_t* w, float* C, int32_t* S, int64_t M,
                           int64_t N, int64_t K, int* status, int inject_timeout, cudaStream_t s) {
    TmaMaps maps;
    const uint64_t nb = uint64_t(K / 32), nsb = uint64_t(K / 256);
    if (!encode_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, aq.qs, uint64_t(K), uint64_t(M),
                   uint64_t(K), 128, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&maps.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, nsb * 144, uint64_t(N), nsb * 144,
                   144, BN, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&maps.da, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, aq.da, nb, uint64_t(M), nb * 4, 8, BM,
                   CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&maps.sa, CU_TENSOR_MAP_DATA_TYPE_INT32, aq.sa, nb, uint64_t(M), nb * 4, 8, BM,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    int dev = 0, nsm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    // The register split (setmaxnreg) needs the block launched with exactly
    // kRegsLaunch registers per thread; refuse anything else.
    {
        cudaFuncAttributes fa;
        cudaError_t e = S ? cudaFuncGetAttributes(&fa, gemm_tc_kernel<true>)
                          : cudaFuncGetAttributes(&fa, gemm_tc_kernel<false>);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != int(kRegsLaunch)) return cudaErrorInvalidConfiguration;
    }
    const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    // Few tiles: split K over a cluster so that most SMs get work.
    int split = 1;
    if (tiles * 2 <= nsm)
        while (split < 8 && tiles * split * 2 <= nsm && split * 2 <= int64_t(nsb)) split *= 2;
    auto k = S ? gemm_tc_kernel<true> : gemm_tc_kernel<false>;
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes)))
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(split > 1 ? tiles * split : (tiles < nsm ? tiles : nsm)));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = size_t(kSmemBytes);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(split);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, k, maps, C, S, int(M), int(N), int(K), split, status, inject_timeout);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace mmq
