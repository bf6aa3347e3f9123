// q6_K x q8_1 GEMM on the tcgen05 tensor cores.
//
// q6_K is the weight family the pages' MMQ line moved to after q4_K (web page
// "20 . r15 -- f32-accumulate mma probe (dead end) + rank-1 term2 rescale",
// section "Proof of pattern portability"): 256-element super-blocks with an
// fp16 d, a signed 8-bit scale sc per 16 consecutive weights and 6-bit quants
// q in [-32, 31]; no minimum, so the rescale has one term.  Per 32-k chunk c
// (one q8_1 block, two scale sub-blocks)
//     C_ij += da_ic * d_j * S'_ijc,   S'_ijc = sum_{k in c} a_ik * sc_j,s(k) * q_jk,
// the same sum as the per-16 form da * d * sc * S16 (the two sub-blocks'
// products added first, exactly).
//
// sm_103a has no integer kind for tcgen05.mma, so the integers go through
// kind::f16.  The activation operand is a in [-127, 127] as exact fp16 (as in
// the q4_K kernel).  The weight factor v = sc * q (|v| <= 4096) needs up to
// 13 significant bits, more than fp16 holds, so it is split into
// hi = fp16(v) (the product rounded to nearest) and lo = v - hi (|lo| <= 1,
// exact), two operand tiles that the MMA adds into the same accumulator.
// Every product is an integer below 2^19 and every partial sum is bounded by
// sum |a| (|hi| + |lo|) <= 32 * 127 * 4098 < 2^24, so the f32 tensor-memory
// accumulator holds S' exactly.
//
// One CTA per SM, persistent over 128 (tokens) x 128 (weight rows) tiles
// (or K split over a cluster when the tiles are few, with a reduce-scatter of
// the partial tiles), warp-specialised (16 warps; setmaxnreg moves registers
// to the epilogue):
//   warp 0      TMA producer: per 256-k super-block the raw int8 A tile (two
//               128-byte-swizzled boxes), the 128 weight rows' padded 224-byte
//               super-blocks, and the da slice, zero-filled past M / N.
//   warp 1      MMA issuer (one thread): per 32-k chunk four K=16 f16 MMAs
//               (hi and lo weight parts) into one of four 128-column tensor
//               memory slots, one commit per chunk.
//   warps 2-3   per super-block: da per token row and chunk, and d per weight
//               row (tables for the epilogue).
//   warps 4-7   operand converters, one row per thread, one chunk per stage:
//               int8 -> fp16 (the 1024-offset bit pattern), and the q6 unpack
//               (low nibble from ql, two high bits from qh) to q, then hi and lo
//               of sc * q with two packed fp16 operations, into the 64-byte
//               swizzled K-major layout.
//   warps 8-15  epilogue: thread = token row, 64 columns; per chunk two
//               32x32b.x32 tensor-memory loads and 32 packed f32x2 FMAs with
//               da, per super-block 32 more with d; C stored at the end of a
//               tile.
// Within a chunk the k order of both operands is 0,2,1,3 per group of four
// (the int8 unpack's pair order): a dot product does not depend on the order
// of its terms.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "mmq_internal.h"
#include "sm103_ptx.cuh"
#include "tc_common.cuh"

namespace {

using namespace mmq::ptx;
using namespace mmq::tc;

constexpr int BM = 128, BN = 128;
constexpr int kQ6DevBytes = 224;   // the device layout's padded super-block
constexpr int kNumRaw = 2, kNumScl = 3, kNumOp = 3, kNumTm = 4;
constexpr int kSclWarp0 = 2, kNumSclWarps = 2, kConvWarp0 = 4, kNumConvWarps = 4;
constexpr int kEpiWarp0 = 8, kNumEpiWarps = 8;
constexpr int kThreads = (kEpiWarp0 + kNumEpiWarps) * 32;   // 512
constexpr uint32_t kRegsLow = 80, kRegsHigh = 176, kRegsLaunch = 128;
static_assert(256 * kRegsLow + 256 * kRegsHigh <= kThreads * kRegsLaunch, "register split");
constexpr int kSlotCols = BN;   // one chunk's S' tile per slot
constexpr uint32_t kTmemCols = 512;
static_assert(kNumTm * kSlotCols <= int(kTmemCols), "tensor memory budget");

// Shared memory map (offsets from a 1024-byte aligned base).
constexpr int kRawASub = BM * 128;                   // 16 KB: 128 rows x 128 B, swizzled
constexpr int kRawA = 2 * kRawASub;                  // 256 k of int8
constexpr int kRawB = BN * kQ6DevBytes;              // 28 KB of padded q6_K rows
constexpr int kRawDa = BM * 8 * 4;                   // da [128][8] f32
constexpr int kOffRawB = kRawA, kOffRawDa = kRawA + kRawB;
constexpr int kRawStage = kOffRawDa + kRawDa;        // 64 KB: everything one super-block needs from HBM
constexpr int kOpTile = 128 * 64;                    // 128 rows x 32 fp16 (64 B), 64-byte swizzle
constexpr int kOpStage = 3 * kOpTile;                // A, weight hi, weight lo
constexpr int kSclDa = 8 * BM * 4;                   // da [8 chunks][128 rows] f32
constexpr int kSclD = BN * 4;                        // d [128 weight rows] f32
constexpr int kSclStage = kSclDa + kSclD;
constexpr int kOffRaw = 0;
constexpr int kOffOp = kOffRaw + kNumRaw * kRawStage;
constexpr int kOffScl = kOffOp + kNumOp * kOpStage;
constexpr int kOffBar = kOffScl + kNumScl * kSclStage;
constexpr int kNumBars = 2 * kNumRaw + 2 * kNumOp + 2 * kNumTm + 2 * kNumScl;
constexpr int kOffMisc = kOffBar + kNumBars * 8;     // tmem slot, abort flag
constexpr int kSmemBytes = kOffMisc + 16 + 1024;     // + alignment slack
static_assert(kOffOp % 1024 == 0 && kOpTile % 512 == 0, "operand tiles need their swizzle alignment");
static_assert(kRawStage % 1024 == 0 && kSclStage % 16 == 0, "stage alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");
// the split-K landing area [split][128 rows][BN / split] f32 reuses the raw ring
static_assert(BM * BN * 4 <= kNumRaw * kRawStage, "landing area");

constexpr uint32_t kRawTx = kRawStage;
constexpr uint32_t kIdesc = idesc_f16_f32(BM, BN);

struct TmaMaps {
    CUtensorMap a, b, da;
};

struct Bars {
    uint32_t base;
    __device__ uint32_t at(int i) const { return base + 8 * i; }
    __device__ uint32_t raw_full(int s) const { return at(s); }
    __device__ uint32_t raw_empty(int s) const { return at(kNumRaw + s); }
    static constexpr int kOp0 = 2 * kNumRaw;
    __device__ uint32_t op_full(int s) const { return at(kOp0 + s); }
    __device__ uint32_t op_empty(int s) const { return at(kOp0 + kNumOp + s); }
    static constexpr int kTm0 = kOp0 + 2 * kNumOp;
    __device__ uint32_t tm_full(int s) const { return at(kTm0 + s); }
    __device__ uint32_t tm_empty(int s) const { return at(kTm0 + kNumTm + s); }
    static constexpr int kScl0 = kTm0 + 2 * kNumTm;
    __device__ uint32_t scl_full(int s) const { return at(kScl0 + s); }
    __device__ uint32_t scl_empty(int s) const { return at(kScl0 + kNumScl + s); }
};
static_assert(Bars::kScl0 + 2 * kNumScl == kNumBars, "barrier count");

// Four 6-bit quants u = ql nibble | qh bit pair << 4 (one per byte, from one
// ql word and one qh word), made fp16 pairs {q0, q2} and {q1, q3} of
// q = u - 32 (the 1024-offset bit pattern, then one fp16 subtraction: exact).
__device__ __forceinline__ void q6_pairs(uint32_t qlw, uint32_t qhw, uint32_t nib_shift, uint32_t hb_shift,
                                         __half2& q02, __half2& q13) {
    const uint32_t u = ((qlw >> nib_shift) & 0x0F0F0F0Fu) | (((qhw >> hb_shift) & 0x03030303u) << 4);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6420), __ushort_as_half(0x6420));   // 1056
    uint32_t p02 = prmt(u, 0x64646464u, 0x4240u), p13 = prmt(u, 0x64646464u, 0x4341u);
    q02 = __hsub2(*reinterpret_cast<const __half2*>(&p02), bias);
    q13 = __hsub2(*reinterpret_cast<const __half2*>(&p13), bias);
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// 32 columns of one chunk's S' (exact integers held in f32) to S [M][N][nb].
__device__ __forceinline__ void dump_s(int32_t* S, const uint32_t (&b)[32], int64_t gr, int gc0, int M, int N,
                                       int nb, int kb) {
    if (gr >= M) return;
#pragma unroll
    for (int j = 0; j < 32; ++j)
        if (gc0 + j < N) S[(gr * N + gc0 + j) * int64_t(nb) + kb] = int32_t(__uint_as_float(b[j]));
}

// kDump: write each chunk's exact S' (int32 [M][N][K/32]) instead of C, from
// the same operands and MMAs (one launch, split == 1).
template <bool kDump>
__global__ void __launch_bounds__(kThreads, 1)
gemm_q6k_tc_kernel(const __grid_constant__ TmaMaps maps, float* __restrict__ C, int32_t* __restrict__ S, int M,
                   int N, int K, int split, int* status, int inject_timeout, int tile_lo, int num_tiles) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const Bars bars{sbase + kOffBar};
    griddep_launch_dependents();
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    const AbortFlag abort_flag{sbase + kOffMisc + 4};

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nsb = K / 256;
    const int tiles_n = (N + BN - 1) / BN;
    // As the q4_K kernel: persistent over [tile_lo, num_tiles), or a cluster
    // of `split` CTAs per tile, rank r taking super-blocks
    // [nsb*r/split, nsb*(r+1)/split).
    const int rank = split > 1 ? int(blockIdx.x % unsigned(split)) : 0;
    const int tile_first = tile_lo + (split > 1 ? int(blockIdx.x / unsigned(split)) : int(blockIdx.x));
    const int tile_step = split > 1 ? num_tiles : int(gridDim.x);
    const int sb_lo = (nsb * rank) / split, sb_hi = (nsb * (rank + 1)) / split;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kNumRaw; ++s) {
            mbar_init(bars.raw_full(s), 1);
            mbar_init(bars.raw_empty(s), kNumConvWarps + kNumSclWarps);
        }
        for (int s = 0; s < kNumOp; ++s) {
            mbar_init(bars.op_full(s), kNumConvWarps);
            mbar_init(bars.op_empty(s), 1);
        }
        for (int s = 0; s < kNumTm; ++s) {
            mbar_init(bars.tm_full(s), 1);
            mbar_init(bars.tm_empty(s), kNumEpiWarps);
        }
        for (int s = 0; s < kNumScl; ++s) {
            mbar_init(bars.scl_full(s), kNumSclWarps);
            mbar_init(bars.scl_empty(s), kNumEpiWarps);
        }
        abort_flag.set(0u);
        fence_barrier_init();
        fence_proxy_async_smem();
        prefetch_tmap(&maps.a);
        prefetch_tmap(&maps.b);
        prefetch_tmap(&maps.da);
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
            griddep_wait();   // the activations are the previous kernel's output
            Ring<kNumRaw> rr;
            uint32_t iss = 0, par = 0;   // bit s: a copy was issued into slot s / its phase
            bool first = true;
            for (int tile = tile_first; tile < num_tiles; tile += tile_step) {
                const int m0 = (tile / tiles_n) * BM, n0 = (tile % tiles_n) * BN;
                for (int sb = sb_lo; sb < sb_hi; ++sb) {
                    if (!wait_bounded(bars.raw_empty(rr.slot), rr.phase ^ 1u, abort_flag, status))
                        goto producer_done;
                    if (!(first && inject_timeout)) {   // test hook: withhold this arrival
                        const uint32_t raw = sbase + kOffRaw + rr.slot * kRawStage;
                        const uint32_t fb = bars.raw_full(rr.slot);
                        mbar_arrive_expect_tx(fb, kRawTx);
                        tma_load_2d(raw, &maps.a, fb, sb * 256, m0);
                        tma_load_2d(raw + kRawASub, &maps.a, fb, sb * 256 + 128, m0);
                        tma_load_2d(raw + kOffRawB, &maps.b, fb, sb * kQ6DevBytes, n0);
                        tma_load_2d(raw + kOffRawDa, &maps.da, fb, sb * 8, m0);
                        iss |= 1u << rr.slot;
                        par = (par & ~(1u << rr.slot)) | (rr.phase << rr.slot);
                    }
                    first = false;
                    rr.next();
                }
            }
        producer_done:
            // Let every copy already issued land before the CTA can exit.
            for (int s = 0; s < kNumRaw; ++s)
                if ((iss >> s) & 1u) wait_drain(bars.raw_full(s), (par >> s) & 1u, status);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            Ring<kNumOp> orr;
            Ring<kNumTm> tr;
            uint32_t last_bar = 0, last_par = 0;   // most recent commit, drained on exit
            for (int tile = tile_first; tile < num_tiles; tile += tile_step) {
                for (int sb = sb_lo; sb < sb_hi; ++sb) {
                    for (int c = 0; c < 8; ++c) {
                        const bool of = mbar_try_wait(bars.op_full(orr.slot), orr.phase);
                        const bool te = mbar_try_wait(bars.tm_empty(tr.slot), tr.phase ^ 1u);
                        if (!of && !wait_bounded(bars.op_full(orr.slot), orr.phase, abort_flag, status))
                            goto mma_done;
                        if (!te && !wait_bounded(bars.tm_empty(tr.slot), tr.phase ^ 1u, abort_flag, status))
                            goto mma_done;
                        tc_fence_after();
                        const uint64_t dA = smem_desc_sw64(sbase + kOffOp + orr.slot * kOpStage);
                        const uint64_t dH = dA + uint64_t(kOpTile >> 4), dL = dH + uint64_t(kOpTile >> 4);
                        const uint32_t d = tmem_base + uint32_t(tr.slot * kSlotCols);
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {   // +32 bytes per K = 16
                            mma_f16(d, dA + uint64_t(2 * kk), dH + uint64_t(2 * kk), kIdesc, uint32_t(kk));
                            mma_f16(d, dA + uint64_t(2 * kk), dL + uint64_t(2 * kk), kIdesc, 1u);
                        }
                        mma_commit(bars.tm_full(tr.slot));
                        mma_commit(bars.op_empty(orr.slot));
                        last_bar = bars.op_empty(orr.slot);
                        last_par = orr.phase;
                        tr.next();
                        orr.next();
                    }
                }
            }
        mma_done:
            if (last_bar) wait_drain(last_bar, last_par, status);
        }
    } else if (warp < kConvWarp0) {
        // ------------------------------------------------------------ tables
        const int ts = threadIdx.x - kSclWarp0 * 32;   // 0..63: rows ts and ts + 64
        Ring<kNumRaw> rr;
        Ring<kNumScl> sr;
        for (int tile = tile_first; tile < num_tiles; tile += tile_step) {
            for (int sb = sb_lo; sb < sb_hi; ++sb) {
                if (!wait_bounded(bars.raw_full(rr.slot), rr.phase, abort_flag, status)) goto scl_done;
                {
                    const uint32_t raw = sbase + kOffRaw + rr.slot * kRawStage;
                    if (!wait_bounded(bars.scl_empty(sr.slot), sr.phase ^ 1u, abort_flag, status))
                        goto scl_done;
                    const uint32_t dat = sbase + kOffScl + sr.slot * kSclStage;   // da [8][128]
                    const uint32_t dtab = dat + kSclDa;                              // d [128]
#pragma unroll
                    for (int rh = 0; rh < 2; ++rh) {
                        const int t = ts + 64 * rh;
                        const uint4 d0 = ld_shared_v4(raw + kOffRawDa + t * 32);
                        const uint4 d1 = ld_shared_v4(raw + kOffRawDa + t * 32 + 16);
                        const uint32_t dv[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
                        for (int c = 0; c < 8; ++c) st_shared_u32(dat + uint32_t(c * BM + t) * 4u, dv[c]);
                        // d: the fp16 at byte 208 of the weight row's super-block
                        const uint32_t dw = ld_shared_u32(raw + kOffRawB + t * kQ6DevBytes + 208);
                        st_shared_u32(dtab + uint32_t(t) * 4u,
                                      __float_as_uint(__half2float(__ushort_as_half(uint16_t(dw & 0xFFFFu)))));
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars.scl_full(sr.slot));
                    sr.next();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.raw_empty(rr.slot));
                rr.next();
            }
        }
    scl_done:;
    } else {
        // -------------------------------------------------------- converters
        const int t = threadIdx.x - kConvWarp0 * 32;   // 0..127: this thread's row
        const int sw128 = t & 7, sw64 = (t >> 1) & 3;
        Ring<kNumRaw> rr;
        Ring<kNumOp> orr;
        for (int tile = tile_first; tile < num_tiles; tile += tile_step) {
            for (int sb = sb_lo; sb < sb_hi; ++sb) {
                if (!wait_bounded(bars.raw_full(rr.slot), rr.phase, abort_flag, status)) goto conv_done;
                const uint32_t raw = sbase + kOffRaw + rr.slot * kRawStage;
                const uint32_t rowB = raw + kOffRawB + t * kQ6DevBytes;   // ql[128] qh[64] sc[16] d
                const uint4 scv = ld_shared_v4(rowB + 192);
                const uint32_t scw[4] = {scv.x, scv.y, scv.z, scv.w};
                for (int c = 0; c < 8; ++c) {   // chunk c = 4n + r: elements 128n + 32r + l
                    if (!wait_bounded(bars.op_empty(orr.slot), orr.phase ^ 1u, abort_flag, status))
                        goto conv_done;
                    const int n = c >> 2, r = c & 3;
                    const uint32_t opA = sbase + kOffOp + orr.slot * kOpStage + t * 64;
                    const uint32_t opH = opA + kOpTile, opL = opH + kOpTile;
                    // A: the chunk's 32 int8, granules 2(c%4), 2(c%4)+1 of sub-tile c/4
                    const uint4 wa0 = ld_shared_v4(raw + (c >> 2) * kRawASub + t * 128 +
                                                   ((uint32_t(2 * (c & 3)) ^ uint32_t(sw128)) << 4));
                    const uint4 wa1 = ld_shared_v4(raw + (c >> 2) * kRawASub + t * 128 +
                                                   ((uint32_t(2 * (c & 3) + 1) ^ uint32_t(sw128)) << 4));
                    // weights: ql bytes 64n + 32(r%2) + l (nibble r/2), qh bytes 32n + l (bits 2r)
                    const uint4 l0 = ld_shared_v4(rowB + 64 * n + 32 * (r & 1));
                    const uint4 l1 = ld_shared_v4(rowB + 64 * n + 32 * (r & 1) + 16);
                    const uint4 h0 = ld_shared_v4(rowB + 128 + 32 * n);
                    const uint4 h1 = ld_shared_v4(rowB + 128 + 32 * n + 16);
                    {
                        // granule g of the 64-byte row holds elements 8g..8g+7 (0,2,1,3 per four)
                        const uint32_t aw[8] = {wa0.x, wa0.y, wa0.z, wa0.w, wa1.x, wa1.y, wa1.z, wa1.w};
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            uint32_t p0, p1, p2, p3;
                            cvt_a4(aw[2 * g], p0, p1);
                            cvt_a4(aw[2 * g + 1], p2, p3);
                            st_shared_v4(opA + ((uint32_t(g) ^ uint32_t(sw64)) << 4), p0, p1, p2, p3);
                        }
                    }
                    {
                        const uint32_t qlw[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
                        const uint32_t qhw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
                        const uint32_t nsh = 4u * uint32_t(r >> 1), hsh = 2u * uint32_t(r);
                        // the two 16-weight sub-blocks of chunk c: scales 2c, 2c+1 (int8)
                        const uint32_t sw2 = scw[c >> 1] >> (16 * (c & 1));
                        const __half2 sa2 = __half2half2(__int2half_rn(int(int8_t(sw2 & 0xFFu))));
                        const __half2 sb2 = __half2half2(__int2half_rn(int(int8_t((sw2 >> 8) & 0xFFu))));
#pragma unroll
                        for (int g = 0; g < 4; ++g) {   // elements 8g..8g+7 of the chunk
                            const __half2 s2 = g < 2 ? sa2 : sb2;
                            uint32_t hi[4], lo[4];
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                __half2 q02, q13;
                                q6_pairs(qlw[2 * g + h], qhw[2 * g + h], nsh, hsh, q02, q13);
                                // hi = fp16(sc * q) rounded to nearest; lo = sc * q - hi, exact
                                const __half2 h02 = __hmul2(q02, s2), h13 = __hmul2(q13, s2);
                                hi[2 * h] = h2u(h02);
                                hi[2 * h + 1] = h2u(h13);
                                lo[2 * h] = h2u(__hfma2(q02, s2, __hneg2(h02)));
                                lo[2 * h + 1] = h2u(__hfma2(q13, s2, __hneg2(h13)));
                            }
                            const uint32_t o = (uint32_t(g) ^ uint32_t(sw64)) << 4;
                            st_shared_v4(opH + o, hi[0], hi[1], hi[2], hi[3]);
                            st_shared_v4(opL + o, lo[0], lo[1], lo[2], lo[3]);
                        }
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
        // Thread = token row quarter*32 + lane (the tensor-memory lane quarter
        // this warp may read) x 64 columns colhalf*64 + [0, 64).
        const int ew = warp - kEpiWarp0;
        const int quarter = warp & 3;
        const int colhalf = ew >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t tlane = uint32_t(quarter * 32) << 16;
        Ring<kNumScl> sr;
        Ring<kNumTm> tr;
        uint64_t acc[32], asb[32];
        for (int tile = tile_first; tile < num_tiles; tile += tile_step) {
            const int m0 = (tile / tiles_n) * BM, n0 = (tile % tiles_n) * BN;
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = 0ull;
            for (int sb = sb_lo; sb < sb_hi; ++sb) {
                if (!wait_bounded(bars.scl_full(sr.slot), sr.phase, abort_flag, status)) goto epi_done;
                const uint32_t dat = sbase + kOffScl + sr.slot * kSclStage;
#pragma unroll
                for (int i = 0; i < 32; ++i) asb[i] = 0ull;
                for (int c = 0; c < 8; ++c) {
                    const float da = __uint_as_float(ld_shared_u32(dat + uint32_t(c * BM + row) * 4u));
                    if (!wait_bounded(bars.tm_full(tr.slot), tr.phase, abort_flag, status)) goto epi_done;
                    tc_fence_after();
                    const uint32_t ta = tmem_base + tlane + uint32_t(tr.slot * kSlotCols + colhalf * 64);
                    const uint64_t da2 = pack2(da, da);
                    uint32_t b[32];
                    tmem_ld_32x32b_x32(ta, b);
                    tmem_wait_ld(b);
                    if constexpr (kDump) {
                        dump_s(S, b, int64_t(m0) + row, n0 + colhalf * 64, M, N, K / 32, sb * 8 + c);
                    } else {
                        half_fma<0>(asb, b, da2);
                    }
                    tmem_ld_32x32b_x32(ta + 32, b);
                    tmem_wait_ld(b);
                    // the chunk's S' tile is in registers: hand the slot back
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars.tm_empty(tr.slot));
                    tr.next();
                    if constexpr (kDump) {
                        dump_s(S, b, int64_t(m0) + row, n0 + colhalf * 64 + 32, M, N, K / 32, sb * 8 + c);
                    } else {
                        half_fma<1>(asb, b, da2);
                    }
                }
                {
                    // acc += d * asb for this super-block
                    const uint32_t dcol = dat + kSclDa + uint32_t(colhalf * 64) * 4u;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const uint4 dv = ld_shared_v4(dcol + 16u * i);
                        acc[2 * i] = ffma2(pack2u(dv.x, dv.y), asb[2 * i], acc[2 * i]);
                        acc[2 * i + 1] = ffma2(pack2u(dv.z, dv.w), asb[2 * i + 1], acc[2 * i + 1]);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.scl_empty(sr.slot));
                sr.next();
            }
            if (!kDump && split == 1) store_tile(C, acc, M, N, m0, n0, row, colhalf);
        }
    epi_done:;
        if (split > 1) {
            // Reduce-scatter over the cluster: rank r owns the tile's columns
            // [r*W, (r+1)*W), W = BN / split; every thread pushes the columns
            // it holds for other ranks into their (idle) raw ring,
            // landing[src][row][W] f32, and the owners add the partials in rank
            // order and store their columns.
            const int W = BN / split;                          // 64, 32 or 16
            const int lw = W == 64 ? 6 : (W == 32 ? 5 : 4);    // log2 W
            const int tile_m0 = (tile_first / tiles_n) * BM, tile_n0 = (tile_first % tiles_n) * BN;
            const int64_t gr = int64_t(tile_m0) + row;
            cluster_sync_all();   // every CTA of the cluster is done with its raw ring
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int c = colhalf * 64 + 4 * i;
                const int d = c >> lw;
                if (d != rank) {
                    const uint32_t off = uint32_t(((rank * BM + row) << lw) + (c - (d << lw))) * 4u;
                    st_dsmem_v4(map_shared_rank(sbase + kOffRaw + off, uint32_t(d)),
                                make_float4(lo_f(acc[2 * i]), hi_f(acc[2 * i]), lo_f(acc[2 * i + 1]),
                                            hi_f(acc[2 * i + 1])));
                }
            }
            cluster_sync_all();   // the pushed partials are visible
            if (gr < M) {
                float* crow = C + gr * N;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int c = colhalf * 64 + 4 * i;
                    const int gc = tile_n0 + c;   // N % 4 == 0: all four columns or none
                    if ((c >> lw) == rank && gc < N) {
                        const float4 own = make_float4(lo_f(acc[2 * i]), hi_f(acc[2 * i]), lo_f(acc[2 * i + 1]),
                                                       hi_f(acc[2 * i + 1]));
                        float4 sum = own;
                        for (int r = 0; r < split; ++r) {
                            const float4 p =
                                r == rank ? own
                                          : ld_shared_v4f(sbase + kOffRaw +
                                                          uint32_t(((r * BM + row) << lw) + (c - (rank << lw))) * 4u);
                            if (r == 0) {
                                sum = p;
                            } else {
                                sum.x += p.x;
                                sum.y += p.y;
                                sum.z += p.z;
                                sum.w += p.w;
                            }
                        }
                        *reinterpret_cast<float4*>(crow + gc) = sum;
                    }
                }
            }
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

int q6k_tc_check_resources() {
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
        cudaGetLastError();
        return MMQ_ERR_CUDA;
    }
    return optin >= kSmemBytes ? MMQ_OK : MMQ_ERR_RESOURCE;
}

int q6k_tc_launch_count(int64_t M, int64_t N, int64_t K) {
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    const TcPlan p = tc_plan(M, N, K, nsm, true);   // the same 128 x 128 tiles as the q4_K kernel
    return p.tail_lo < p.tiles ? 2 : 1;
}

cudaError_t launch_gemm_q6k_tc(mmq_q8_1_t aq, const uint8_t* w, float* C, int32_t* S, int64_t M, int64_t N,
                               int64_t K, int* status, int inject_timeout, cudaStream_t s) {
    TmaMaps maps;
    const uint64_t nb = uint64_t(K / 32), nsb = uint64_t(K / 256);
    if (!encode_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, aq.qs, uint64_t(K), uint64_t(M), uint64_t(K), 128, BM,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&maps.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, nsb * kQ6DevBytes, uint64_t(N), nsb * kQ6DevBytes,
                   kQ6DevBytes, BN, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&maps.da, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, aq.da, nb, uint64_t(M), nb * 4, 8, BM,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    int dev = 0, nsm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    auto k = S ? gemm_q6k_tc_kernel<true> : gemm_q6k_tc_kernel<false>;
    {
        // setmaxnreg needs exactly kRegsLaunch registers per thread at launch
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, k);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != int(kRegsLaunch)) return cudaErrorInvalidConfiguration;
    }
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes))) return e;
    auto launch = [&](int64_t lo, int64_t hi, int split, int inject) -> cudaError_t {
        const int64_t n = hi - lo;
        cudaLaunchAttribute attr[2];
        cudaLaunchConfig_t cfg = launch_config(dim3(unsigned(split > 1 ? n * split : (n < nsm ? n : nsm))),
                                               dim3(kThreads), size_t(kSmemBytes), s, attr);
        attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
        attr[cfg.numAttrs].val.clusterDim.x = unsigned(split);
        attr[cfg.numAttrs].val.clusterDim.y = 1;
        attr[cfg.numAttrs].val.clusterDim.z = 1;
        ++cfg.numAttrs;
        const cudaError_t le = cudaLaunchKernelEx(&cfg, k, maps, C, S, int(M), int(N), int(K), split, status, inject,
                                                  int(lo), int(hi));
        return le != cudaSuccess ? le : cudaGetLastError();
    };
    const TcPlan p = tc_plan(M, N, K, nsm, true);
    if (p.tiles > (int64_t(1) << 30)) return cudaErrorInvalidValue;
    if (S) return launch(0, p.tiles, 1, inject_timeout);   // the dump: every chunk written where it is formed
    if (p.tail_lo == p.tiles) return launch(0, p.tiles, p.first_split, inject_timeout);
    if ((e = launch(0, p.tail_lo, 1, inject_timeout)) != cudaSuccess) return e;
    return launch(p.tail_lo, p.tiles, p.tail_split, 0);
}

}  // namespace mmq
