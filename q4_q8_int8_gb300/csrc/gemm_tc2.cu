// q4_K x q8_1 GEMM on the tcgen05 tensor cores of a CTA pair (.cta_group::2).
//
// Same arithmetic as the one-CTA kernel in gemm_tc.cu (web page "20 . r15 --
// f32-accumulate mma probe (dead end) + rank-1 term2 rescale", section 2.1,
// regrouped: sc inside the exact integer dot S' = sc*S, da per chunk, d per
// super-block, the second term sum_c dma*dmv per super-block as split-tf32
// MMAs; the rank-1 fold dma = da*sa of page "21 . r16 -- Narrow kernel gets
// the rank-1 fold", section 2.1, once per token row and chunk).
//
// A cluster of two CTAs on neighbouring SMs owns a 256-token x 128-weight-row
// tile. Each MMA is one M=256, N=128 instruction over both CTAs.
//   * A: CTA r supplies its own 128 token rows.
//   * B: CTA r supplies weight rows 64r..64r+63 (its half of N).
//   * D: each CTA's tensor memory receives its own 128 rows x 128 columns.
// Per SM this halves the MMA instructions and the weight-operand conversion.
// Only CTA 0 (the leader) issues MMAs. The peer's converters, table warps and
// epilogue hand their stages to the leader by arriving on the leader's
// barriers (cluster-scope release / acquire). The leader's commits multicast
// to both CTAs' barriers.
//
// Warp roles (both CTAs; 16 warps, setmaxnreg moves registers to the epilogue):
//   warp 0      TMA producer: per super-block the CTA's int8 A rows (two
//               128-byte-swizzled boxes), all 128 raw q4_K rows (the epilogue
//               needs every column's d), and the CTA's da / sa slices.
//   warp 1      leader only: MMA issuer (one thread), per operand stage four
//               M=256 K=16 f16 MMAs into one of two 256-column tensor-memory
//               slots; per super-block three K=8 tf32 MMAs of the second term.
//   warps 2-3   epilogue tables (da per token row and chunk, d * 2^24 per
//               weight row) and the split-tf32 second-term operands.
//   warps 4-7   converters: int8 -> fp16 for the CTA's 128 token rows and
//               nibble * sc -> fp16 subnormal for its 64 weight rows (two
//               threads per weight row), 128-byte-swizzled K-major.
//   warps 8-15  epilogue: thread = token row, 64 columns, as in gemm_tc.cu.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "mmq_internal.h"
#include "sm103_ptx.cuh"
#include "tc_common.cuh"

namespace {

using namespace mmq::ptx;
using namespace mmq::tc;

constexpr int BM = 128, BN = 128, BNH = 64;   // rows per CTA, columns per pair, B rows per CTA
constexpr int kNumRaw = 2, kNumScl = 3, kNumOp = 3, kNumTm = 2;
constexpr int kSclWarp0 = 2, kNumSclWarps = 2, kConvWarp0 = 4, kNumConvWarps = 4;
constexpr int kEpiWarp0 = 8, kNumEpiWarps = 8;
constexpr int kThreads = (kEpiWarp0 + kNumEpiWarps) * 32;   // 512
constexpr uint32_t kRegsLow = 80, kRegsHigh = 176, kRegsLaunch = 128;
static_assert(256 * kRegsLow + 256 * kRegsHigh <= kThreads * kRegsLaunch, "register split");
constexpr int kSlotCols = 2 * BN;
constexpr uint32_t kTmemCols = 512;
static_assert(kNumTm * kSlotCols <= int(kTmemCols), "tensor memory budget");

// Shared memory map (identical in both CTAs; offsets from a 1024-byte aligned base).
constexpr int kRawASub = BM * 128;
constexpr int kRawA = 2 * kRawASub;                  // the CTA's 128 token rows x 256 int8
constexpr int kRawB = BN * 144;                      // all 128 raw q4_K rows of the tile
constexpr int kRawDa = BM * 8 * 4;
constexpr int kRawSa = BM * 8 * 4;
constexpr int kOffRawB = kRawA, kOffRawDa = kRawA + kRawB, kOffRawSa = kOffRawDa + kRawDa;
constexpr int kRawStage = kOffRawSa + kRawSa;        // 58 KB
constexpr int kOpTileA = BM * 128;                   // 128 token rows x 64 fp16, swizzled
constexpr int kOpTileB = BNH * 128;                  // 64 weight rows x 64 fp16, swizzled
constexpr int kOpStage = kOpTileA + kOpTileB;        // 24 KB
constexpr int kMinTileA = BM * 128;                  // 128 token rows x 32 tf32 slots (24 used)
constexpr int kMinTileB = BNH * 128;                 // 64 weight rows x 32 tf32 slots
constexpr int kMinStage = kMinTileA + kMinTileB;     // 24 KB
constexpr int kSclDa = 8 * BM * 4;
constexpr int kSclD = BN * 4;
constexpr int kSclStage = kSclDa + kSclD;
constexpr int kOffRaw = 0;
constexpr int kOffOp = kOffRaw + kNumRaw * kRawStage;
constexpr int kOffMin = kOffOp + kNumOp * kOpStage;
constexpr int kOffScl = kOffMin + kMinStage;
constexpr int kOffBar = kOffScl + kNumScl * kSclStage;
constexpr int kNumBars = 2 * kNumRaw + 2 * kNumOp + 2 * kNumTm + 2 * kNumScl + 2;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
static_assert(kOffOp % 1024 == 0 && kOffMin % 1024 == 0 && kOpStage % 1024 == 0 &&
                  kOpTileA % 1024 == 0 && kMinTileA % 1024 == 0,
              "operand tiles need 1024-byte alignment");
static_assert(kRawStage % 1024 == 0 && kSclStage % 16 == 0, "stage alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kRawTx = kRawStage;
constexpr uint32_t kIdesc = idesc_f16_f32(2 * BM, BN);
constexpr uint32_t kIdescTf32 = idesc_tf32_f32(2 * BM, BN);
constexpr uint16_t kPairMask = 0x3;

struct TmaMaps {
    CUtensorMap a, b, da, sa;
};

struct Bars {
    uint32_t base;
    __device__ uint32_t at(int i) const { return base + 8 * i; }
    __device__ uint32_t raw_full(int s) const { return at(s); }
    __device__ uint32_t raw_empty(int s) const { return at(kNumRaw + s); }
    __device__ uint32_t op_full(int s) const { return at(2 * kNumRaw + s); }
    __device__ uint32_t op_empty(int s) const { return at(2 * kNumRaw + kNumOp + s); }
    __device__ uint32_t tm_full(int s) const { return at(2 * kNumRaw + 2 * kNumOp + s); }
    __device__ uint32_t tm_empty(int s) const { return at(2 * kNumRaw + 2 * kNumOp + kNumTm + s); }
    __device__ uint32_t scl_full(int s) const { return at(2 * kNumRaw + 2 * kNumOp + 2 * kNumTm + s); }
    __device__ uint32_t scl_empty(int s) const {
        return at(2 * kNumRaw + 2 * kNumOp + 2 * kNumTm + kNumScl + s);
    }
    static constexpr int kMin0 = 2 * kNumRaw + 2 * kNumOp + 2 * kNumTm + 2 * kNumScl;
    __device__ uint32_t min_full() const { return at(kMin0); }
    __device__ uint32_t min_empty() const { return at(kMin0 + 1); }
};

// Arrive on the leader CTA's copy of a barrier (the leader's own arrivals
// take the same route).
__device__ __forceinline__ void arrive_leader(uint32_t bar) { mbar_arrive_cluster(mapa_shared(bar, 0u)); }

template <bool kDump>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc2_kernel(const __grid_constant__ TmaMaps maps, float* __restrict__ C, int32_t* __restrict__ S,
                int M, int N, int K, int* status, int inject_timeout) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const Bars bars{sbase + kOffBar};
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    const AbortFlag abort_flag{sbase + kOffMisc + 4};

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t crank = cluster_ctarank();   // 0: leader, 1: peer
    const int nsb = K / 256;
    const int tiles_m = (M + 2 * BM - 1) / (2 * BM), tiles_n = (N + BN - 1) / BN;
    const int num_tiles = tiles_m * tiles_n;
    const int tile_first = int(blockIdx.x >> 1), tile_step = int(gridDim.x >> 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kNumRaw; ++s) {
            mbar_init(bars.raw_full(s), 1);
            mbar_init(bars.raw_empty(s), kNumConvWarps + kNumSclWarps);
        }
        for (int s = 0; s < kNumOp; ++s) {
            mbar_init(bars.op_full(s), 2 * kNumConvWarps);   // both CTAs' converters (leader's copy)
            mbar_init(bars.op_empty(s), 1);
        }
        for (int s = 0; s < kNumTm; ++s) {
            mbar_init(bars.tm_full(s), 1);
            mbar_init(bars.tm_empty(s), 2 * kNumEpiWarps);   // both CTAs' epilogues (leader's copy)
        }
        for (int s = 0; s < kNumScl; ++s) {
            mbar_init(bars.scl_full(s), kNumSclWarps);
            mbar_init(bars.scl_empty(s), kNumEpiWarps);
        }
        mbar_init(bars.min_full(), 2 * kNumSclWarps);   // both CTAs' table warps (leader's copy)
        mbar_init(bars.min_empty(), 1);
        abort_flag.set(0u);
        fence_barrier_init();
        fence_proxy_async_smem();
        prefetch_tmap(&maps.a);
        prefetch_tmap(&maps.b);
        prefetch_tmap(&maps.da);
        prefetch_tmap(&maps.sa);
    }
    __syncwarp();
    if (warp == 0) {
        tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();   // barrier inits and the allocation visible to both CTAs
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
                const int m0 = (tile / tiles_n) * 2 * BM + int(crank) * BM, n0 = (tile % tiles_n) * BN;
                for (int sb = 0; sb < nsb; ++sb) {
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
            for (int s = 0; s < kNumRaw; ++s)
                if (raw_issued[s]) wait_drain(bars.raw_full(s), raw_par[s], status);
        }
    } else if (warp == 1) {
        // ------------------------------------------- MMA issuer (leader only)
        if (lane == 0 && crank == 0) {
            Ring<kNumOp> orr;
            Ring<kNumTm> tr;
            Ring<1> mr;
            uint32_t last_bar = 0, last_par = 0;
            const uint32_t minA = sbase + kOffMin, minB = minA + kMinTileA;
            for (int tile = tile_first; tile < num_tiles; tile += tile_step) {
                for (int sb = 0; sb < nsb; ++sb) {
                    for (int q = 0; q < 4; ++q) {   // operand stage q: chunks 2q, 2q+1
                        if (!wait_bounded_cluster(bars.op_full(orr.slot), orr.phase, abort_flag, status))
                            goto mma_done;
                        if (!wait_bounded_cluster(bars.tm_empty(tr.slot), tr.phase ^ 1u, abort_flag, status))
                            goto mma_done;
                        tc_fence_after();
                        const uint32_t opA = sbase + kOffOp + orr.slot * kOpStage;
                        const uint32_t opB = opA + kOpTileA;
                        const uint32_t d0 = tmem_base + uint32_t(tr.slot * kSlotCols);
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int kk = 0; kk < 2; ++kk) {
                                const uint32_t koff = uint32_t(h * 64 + kk * 32);
                                mma_f16_pair(d0 + uint32_t(h * BN), smem_desc_sw128(opA + koff),
                                             smem_desc_sw128(opB + koff), kIdesc, uint32_t(kk));
                            }
                        mma_commit_pair(bars.tm_full(tr.slot), kPairMask);
                        mma_commit_pair(bars.op_empty(orr.slot), kPairMask);
                        last_bar = bars.op_empty(orr.slot);
                        last_par = orr.phase;
                        tr.next();
                        orr.next();
                    }
                    if (!kDump) {
                        if (!wait_bounded_cluster(bars.min_full(), mr.phase, abort_flag, status)) goto mma_done;
                        if (!wait_bounded_cluster(bars.tm_empty(tr.slot), tr.phase ^ 1u, abort_flag, status))
                            goto mma_done;
                        tc_fence_after();
                        const uint32_t d = tmem_base + uint32_t(tr.slot * kSlotCols);
#pragma unroll
                        for (int j = 0; j < 3; ++j)
                            mma_tf32_pair(d, smem_desc_sw128(minA + 32 * j), smem_desc_sw128(minB + 32 * j),
                                          kIdescTf32, uint32_t(j));
                        mma_commit_pair(bars.tm_full(tr.slot), kPairMask);
                        mma_commit_pair(bars.min_empty(), kPairMask);
                        last_bar = bars.min_empty();
                        last_par = mr.phase;
                        mr.next();
                        tr.next();
                    }
                }
            }
        mma_done:
            if (last_bar) wait_drain(last_bar, last_par, status);
        }
    } else if (warp < kConvWarp0) {
        // ------------------------------------------- tables and second term
        const int ts = threadIdx.x - kSclWarp0 * 32;   // 0..63
        Ring<kNumRaw> rr;
        Ring<kNumScl> sr;
        Ring<1> mr;
        for (int tile = tile_first; tile < num_tiles; tile += tile_step) {
            for (int sb = 0; sb < nsb; ++sb) {
                if (!wait_bounded(bars.raw_full(rr.slot), rr.phase, abort_flag, status)) goto scl_done;
                {
                    const uint32_t raw = sbase + kOffRaw + rr.slot * kRawStage;
                    if (!wait_bounded(bars.scl_empty(sr.slot), sr.phase ^ 1u, abort_flag, status))
                        goto scl_done;
                    const uint32_t dat = sbase + kOffScl + sr.slot * kSclStage;   // da [8][128]
                    const uint32_t dtab = dat + kSclDa;                              // d * 2^24 [128]
#pragma unroll
                    for (int rh = 0; rh < 2; ++rh) {
                        const int t = ts + 64 * rh;
                        const uint4 d0 = ld_shared_v4(raw + kOffRawDa + t * 32);
                        const uint4 d1 = ld_shared_v4(raw + kOffRawDa + t * 32 + 16);
                        const uint32_t dv[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
                        for (int c = 0; c < 8; ++c) st_shared_u32(dat + uint32_t(c * BM + t) * 4u, dv[c]);
                        const uint32_t h0 = ld_shared_v4(raw + kOffRawB + t * 144).x;
                        st_shared_u32(dtab + uint32_t(t) * 4u,
                                      __float_as_uint(__half2float(__ushort_as_half(uint16_t(h0 & 0xFFFFu))) *
                                                      kSubnormalScale));
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars.scl_full(sr.slot));
                    sr.next();
                    if (!kDump) {
                        if (!wait_bounded(bars.min_empty(), mr.phase ^ 1u, abort_flag, status)) goto scl_done;
                        const uint32_t minA = sbase + kOffMin, minB = minA + kMinTileA;
#pragma unroll
                        for (int rh = 0; rh < 2; ++rh) {
                            // token row t: dma = da * sa per chunk, split hi / lo; k slots
                            // 0-7 hi, 8-15 hi, 16-23 lo (against hi, lo, hi of dmv)
                            const int t = ts + 64 * rh;
                            const int sw = t & 7;
                            const uint32_t ra = minA + t * 128;
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const uint4 dv = ld_shared_v4(raw + kOffRawDa + t * 32 + 16 * h);
                                const uint4 sv = ld_shared_v4(raw + kOffRawSa + t * 32 + 16 * h);
                                float ah[4], al[4];
                                split_tf32(__uint_as_float(dv.x) * float(int32_t(sv.x)), ah[0], al[0]);
                                split_tf32(__uint_as_float(dv.y) * float(int32_t(sv.y)), ah[1], al[1]);
                                split_tf32(__uint_as_float(dv.z) * float(int32_t(sv.z)), ah[2], al[2]);
                                split_tf32(__uint_as_float(dv.w) * float(int32_t(sv.w)), ah[3], al[3]);
                                st_shared_v4f(ra + (((0 + h) ^ sw) << 4), ah[0], ah[1], ah[2], ah[3]);
                                st_shared_v4f(ra + (((2 + h) ^ sw) << 4), ah[0], ah[1], ah[2], ah[3]);
                                st_shared_v4f(ra + (((4 + h) ^ sw) << 4), al[0], al[1], al[2], al[3]);
                            }
                        }
                        {
                            // weight row 64*crank + ts of the tile: dmv = -dmin * m (exact), split hi / lo
                            const int sw = ts & 7;
                            const uint4 hdr = ld_shared_v4(raw + kOffRawB + (int(crank) * BNH + ts) * 144);
                            const float dmn = __half2float(__ushort_as_half(uint16_t(hdr.x >> 16)));
                            const uint32_t rb = minB + ts * 128;
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const uint32_t mw = h == 0 ? m_lo4(hdr.z) : m_hi4(hdr.z, hdr.w);
                                float bh[4], bl[4];
#pragma unroll
                                for (int i = 0; i < 4; ++i)
                                    split_tf32(-(dmn * float((mw >> (8 * i)) & 0xFFu)), bh[i], bl[i]);
                                st_shared_v4f(rb + (((0 + h) ^ sw) << 4), bh[0], bh[1], bh[2], bh[3]);
                                st_shared_v4f(rb + (((2 + h) ^ sw) << 4), bl[0], bl[1], bl[2], bl[3]);
                                st_shared_v4f(rb + (((4 + h) ^ sw) << 4), bh[0], bh[1], bh[2], bh[3]);
                            }
                        }
                        fence_proxy_async_all();
                        __syncwarp();
                        if (lane == 0) arrive_leader(bars.min_full());
                        mr.next();
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.raw_empty(rr.slot));
                rr.next();
            }
        }
    scl_done:;
    } else {
        // -------------------------------------------------------- converters
        const int t = threadIdx.x - kConvWarp0 * 32;   // 0..127: token row t
        const int sw = t & 7;
        const int bt = t & (BNH - 1), G = t >> 6;      // weight row bt (of this CTA's 64), byte half G
        const int bsw = bt & 7;
        Ring<kNumRaw> rr;
        Ring<kNumOp> orr;
        for (int tile = tile_first; tile < num_tiles; tile += tile_step) {
            for (int sb = 0; sb < nsb; ++sb) {
                if (!wait_bounded(bars.raw_full(rr.slot), rr.phase, abort_flag, status)) goto conv_done;
                const uint32_t raw = sbase + kOffRaw + rr.slot * kRawStage;
                const uint32_t hdrB = raw + kOffRawB + (int(crank) * BNH + bt) * 144;
                uint32_t scw_lo = 0x01010101u, scw_hi = 0x01010101u;   // the S dump keeps sc out
                if (!kDump) {
                    const uint4 hdr = ld_shared_v4(hdrB);
                    scw_lo = sc_lo4(hdr.y);
                    scw_hi = sc_hi4(hdr.y, hdr.w);
                }
                for (int q = 0; q < 4; ++q) {
                    if (!wait_bounded(bars.op_empty(orr.slot), orr.phase ^ 1u, abort_flag, status))
                        goto conv_done;
                    const uint32_t scw = q < 2 ? scw_lo : scw_hi;
                    const uint32_t sh = 16u * uint32_t(q & 1);
                    const uint32_t sca = (scw >> sh) & 0xFFu;
                    const uint32_t scb = (scw >> (sh + 8u)) & 0xFFu;
                    const uint32_t opA = sbase + kOffOp + orr.slot * kOpStage + t * 128;
                    const uint32_t opB = sbase + kOffOp + orr.slot * kOpStage + kOpTileA + bt * 128;
                    uint4 wa[4];
#pragma unroll
                    for (int g = 0; g < 4; ++g)
                        wa[g] = ld_shared_v4(raw + (q >> 1) * kRawASub + t * 128 + ((((q & 1) * 4 + g) ^ sw) << 4));
                    const uint4 wb = ld_shared_v4(hdrB + 16 + 32 * q + 16 * G);
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
                    {
                        const uint32_t ww[4] = {wb.x, wb.y, wb.z, wb.w};
                        uint32_t lo[8], hi[8];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            lo[2 * u] = (ww[u] & 0x000F000Fu) * sca;
                            lo[2 * u + 1] = ((ww[u] >> 8) & 0x000F000Fu) * sca;
                            hi[2 * u] = ((ww[u] >> 4) & 0x000F000Fu) * scb;
                            hi[2 * u + 1] = ((ww[u] >> 12) & 0x000F000Fu) * scb;
                        }
                        st_shared_v4(opB + (((2 * G) ^ bsw) << 4), lo[0], lo[1], lo[2], lo[3]);
                        st_shared_v4(opB + (((2 * G + 1) ^ bsw) << 4), lo[4], lo[5], lo[6], lo[7]);
                        st_shared_v4(opB + (((4 + 2 * G) ^ bsw) << 4), hi[0], hi[1], hi[2], hi[3]);
                        st_shared_v4(opB + (((5 + 2 * G) ^ bsw) << 4), hi[4], hi[5], hi[6], hi[7]);
                    }
                    fence_proxy_async_all();
                    __syncwarp();
                    if (lane == 0) arrive_leader(bars.op_full(orr.slot));
                    orr.next();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.raw_empty(rr.slot));
                rr.next();
            }
        }
    conv_done:;
    }
    } else {
        setmaxnreg_inc<kRegsHigh>();
        // ---------------------------------------------------------- epilogue
        const int ew = warp - kEpiWarp0;
        const int quarter = warp & 3;
        const int colhalf = ew >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t tlane = uint32_t(quarter * 32) << 16;
        const int nb = K / 32;
        Ring<kNumScl> sr;
        Ring<kNumTm> tr;
        uint64_t acc[32], asb[32];
        for (int tile = tile_first; tile < num_tiles; tile += tile_step) {
            const int m0 = (tile / tiles_n) * 2 * BM + int(crank) * BM, n0 = (tile % tiles_n) * BN;
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = 0ull;
            for (int sb = 0; sb < nsb; ++sb) {
                if (!wait_bounded(bars.scl_full(sr.slot), sr.phase, abort_flag, status)) goto epi_done;
                const uint32_t dat = sbase + kOffScl + sr.slot * kSclStage;
#pragma unroll
                for (int i = 0; i < 32; ++i) asb[i] = 0ull;
                for (int q = 0; q < 4; ++q) {
                    const float da0 = __uint_as_float(ld_shared_u32(dat + uint32_t(2 * q * BM + row) * 4u));
                    if (!wait_bounded(bars.tm_full(tr.slot), tr.phase, abort_flag, status)) goto epi_done;
                    tc_fence_after();
                    const uint32_t ta = tmem_base + tlane + uint32_t(tr.slot * kSlotCols + colhalf * 64);
                    if (kDump) {
                        const int64_t gr = int64_t(m0) + row;
                        const int gc = n0 + colhalf * 64;
                        uint32_t b0[16], b1[16];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int kb = sb * 8 + 2 * q + h;
                            const uint32_t th = ta + uint32_t(h * BN);
                            tmem_ld_32x32b_x16(th, b0);
                            tmem_wait_ld(b0);
                            tmem_ld_32x32b_x16(th + 16, b1);
                            dump_part(S, b0, gr, gc, M, N, nb, kb);
                            tmem_wait_ld(b1);
                            tmem_ld_32x32b_x16(th + 32, b0);
                            dump_part(S, b1, gr, gc + 16, M, N, nb, kb);
                            tmem_wait_ld(b0);
                            tmem_ld_32x32b_x16(th + 48, b1);
                            dump_part(S, b0, gr, gc + 32, M, N, nb, kb);
                            tmem_wait_ld(b1);
                            dump_part(S, b1, gr, gc + 48, M, N, nb, kb);
                        }
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) arrive_leader(bars.tm_empty(tr.slot));
                        tr.next();
                    } else {
                        const uint64_t da02 = pack2(da0, da0);
                        uint32_t b[32];
                        tmem_ld_32x32b_x32(ta, b);
                        tmem_wait_ld(b);
                        half_fma<0>(asb, b, da02);
                        tmem_ld_32x32b_x32(ta + 32, b);
                        tmem_wait_ld(b);
                        half_fma<1>(asb, b, da02);
                        const float da1 = __uint_as_float(ld_shared_u32(dat + uint32_t((2 * q + 1) * BM + row) * 4u));
                        const uint64_t da12 = pack2(da1, da1);
                        tmem_ld_32x32b_x32(ta + BN, b);
                        tmem_wait_ld(b);
                        half_fma<0>(asb, b, da12);
                        tmem_ld_32x32b_x32(ta + BN + 32, b);
                        tmem_wait_ld(b);
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) arrive_leader(bars.tm_empty(tr.slot));
                        tr.next();
                        half_fma<1>(asb, b, da12);
                    }
                }
                if (!kDump) {
                    // acc += d * 2^24 * asb for this super-block
                    const uint32_t dcol = dat + kSclDa + uint32_t(colhalf * 64) * 4u;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const uint4 dv = ld_shared_v4(dcol + 16u * i);
                        acc[2 * i] = ffma2(pack2u(dv.x, dv.y), asb[2 * i], acc[2 * i]);
                        acc[2 * i + 1] = ffma2(pack2u(dv.z, dv.w), asb[2 * i + 1], acc[2 * i + 1]);
                    }
                    // acc += the second term of this super-block
                    if (!wait_bounded(bars.tm_full(tr.slot), tr.phase, abort_flag, status)) goto epi_done;
                    tc_fence_after();
                    const uint32_t ta = tmem_base + tlane + uint32_t(tr.slot * kSlotCols + colhalf * 64);
                    const uint64_t one2 = pack2(1.0f, 1.0f);
                    uint32_t b[32];
                    tmem_ld_32x32b_x32(ta, b);
                    tmem_wait_ld(b);
                    half_fma<0>(acc, b, one2);
                    tmem_ld_32x32b_x32(ta + 32, b);
                    tmem_wait_ld(b);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) arrive_leader(bars.tm_empty(tr.slot));
                    tr.next();
                    half_fma<1>(acc, b, one2);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.scl_empty(sr.slot));
                sr.next();
            }
            if (!kDump) store_tile(C, acc, M, N, m0, n0, row, colhalf);
        }
    epi_done:;
    }

    // Neither CTA leaves (or frees tensor memory) while its peer may still
    // read its shared memory, write its tensor memory or arrive on its barriers.
    tc_fence_before();
    cluster_sync_all();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
    cluster_sync_all();
}

}  // namespace

namespace mmq {

int tc2_gemm_check_resources() {
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
        cudaGetLastError();
        return MMQ_ERR_CUDA;
    }
    return optin >= kSmemBytes ? MMQ_OK : MMQ_ERR_RESOURCE;
}

int64_t tc2_pair_tiles(int64_t M, int64_t N) { return ((M + 2 * BM - 1) / (2 * BM)) * ((N + BN - 1) / BN); }

cudaError_t launch_gemm_tc2(mmq_q8_1_t aq, const uint8_t* w, float* C, int32_t* S, int64_t M,
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
    {
        // setmaxnreg needs exactly kRegsLaunch registers per thread at launch
        cudaFuncAttributes fa;
        cudaError_t e = S ? cudaFuncGetAttributes(&fa, gemm_tc2_kernel<true>)
                          : cudaFuncGetAttributes(&fa, gemm_tc2_kernel<false>);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != int(kRegsLaunch)) return cudaErrorInvalidConfiguration;
    }
    const int64_t tiles = tc2_pair_tiles(M, N);
    const int64_t pairs = tiles < nsm / 2 ? tiles : nsm / 2;
    auto k = S ? gemm_tc2_kernel<true> : gemm_tc2_kernel<false>;
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes)))
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(2 * pairs));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = size_t(kSmemBytes);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, k, maps, C, S, int(M), int(N), int(K), status, inject_timeout);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace mmq
