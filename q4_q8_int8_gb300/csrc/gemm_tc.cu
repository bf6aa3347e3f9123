// q4_K x q8_1 GEMM on the 5th-generation tensor cores (tcgen05) of sm_103a.
//
// Math (web page "20 . r15 -- f32-accumulate mma probe (dead end) + rank-1
// term2 rescale", section 2.1): for every 32-k chunk c
//     C_ij += (da_ic * d_j * sc_jc) * S_ij + dma_ic * dmv_jc,
// S_ij = sum_k a_ik * v_jk the exact integer dot of the chunk, dmv = -dmin*m,
// dma = da*sa once per token row and chunk (the rank-1 fold, page "21 . r16 --
// Narrow kernel gets the rank-1 fold", section 2.1).  This kernel regroups the
// same sum so that the CUDA cores do one fused multiply-add per output and
// chunk:
//   * the 6-bit scale sc goes into the weight operand: the MMA computes the
//     integer S'_ij = sc_jc * S_ij (|S'| <= 32*127*63*15 < 2^22, still exact);
//   * the per-row scale is applied per chunk, the per-super-block d once per
//     super-block: acc_ij += d_j * sum_c da_ic * S'_ijc;
//   * the second term, per super-block an 8-long f32 contraction of dma with
//     dmv, runs on the tensor core in tf32 with both factors split into a
//     high and a low tf32 part (hi*hi + hi*lo + lo*hi, relative error ~2^-21)
//     and reaches the epilogue as a fifth tensor-memory hand-off per
//     super-block, added as it is.
//
// sm_103a has no integer kind for tcgen05.mma, so the integers go through
// kind::f16: every quant a in [-127, 127] is an exact fp16 value, and the
// weight factor sc*v <= 945 is written as the fp16 subnormal sc*v * 2^-24
// (just the integer in the mantissa bits); every product and partial sum is
// an integer multiple of 2^-24 below 2^-2, so the f32 accumulator holds
// S' * 2^-24 exactly.  The 2^24 is folded into d.  Two dumps write the
// accumulator per chunk instead of rescaling it: kDumpS leaves sc out of the
// weight operand and returns S itself, kDumpScaled keeps the product's
// operand and returns S' = sc * S, both bit for bit.
//
// One CTA per SM, persistent over 128 (tokens) x 128 (weight rows) tiles,
// warp-specialised (16 warps; setmaxnreg moves registers to the epilogue):
//   warp 0      TMA producer: per 256-k super-block the raw int8 A tile (two
//               128-byte-swizzled boxes), the raw 144-byte q4_K rows, and the
//               da / sa slices, all zero-filled past M / N.
//   warp 1      MMA issuer (one thread): per operand stage (two chunks) four
//               K=16 f16 MMAs into one of two 256-column f32 tensor-memory
//               slots, one hand-off per stage; per super-block three K=8 tf32
//               MMAs of the second term into the next slot.
//   warps 2-3   per super-block: the epilogue's tables (da per row and chunk,
//               d * 2^24 per weight row) and the split tf32 operands of the
//               second term (dma per token row, dmv per weight row).
//   warps 4-7   operand converters: int8 -> fp16 (exact, via the 1024-offset
//               bit pattern and one fp16 subtraction) and nibble * sc -> fp16
//               subnormal into the 128-byte-swizzled K-major layout, one 64-k
//               chunk pair at a time, one row per thread.
//   warps 8-15  epilogue: thread = token row, 64 columns; per chunk two
//               32x32b.x32 tensor-memory loads and 32 packed f32x2 FMAs, one
//               wait and one release per two chunks; per super-block 32 more
//               for d and 32 adds of the second term; C stored at the end of
//               a tile.
// Within a chunk the k order of both f16 operands is permuted identically
// (groups of four as 0,2,1,3) so that both unpacks are plain byte/nibble
// moves; a dot product does not depend on the order of its terms.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <mutex>

#include "mmq_internal.h"
#include "sm103_ptx.cuh"
#include "tc_common.cuh"

namespace {

using namespace mmq::ptx;
using namespace mmq::tc;

constexpr int BM = 128, BN = 128;
constexpr int kNumRaw = 2, kNumScl = 3, kNumOp = 2, kNumTm = 2;
constexpr int kSclWarp0 = 2, kNumSclWarps = 2, kConvWarp0 = 4, kNumConvWarps = 4;
constexpr int kEpiWarp0 = 8, kNumEpiWarps = 8;
constexpr int kThreads = (kEpiWarp0 + kNumEpiWarps) * 32;   // 512
// Register split: warpgroups 0-1 (producer, MMA, tables, converters) give up
// registers to warpgroups 2-3 (epilogue).  Launch budget: 512 x 128.
constexpr uint32_t kRegsLow = 80, kRegsHigh = 176, kRegsLaunch = 128;
static_assert(256 * kRegsLow + 256 * kRegsHigh <= kThreads * kRegsLaunch, "register split");
// Tensor memory: kNumTm slots, each two 128-column f32 buffers (the two
// chunks of one operand stage, or the second term in the first of them).
constexpr int kSlotCols = 2 * BN;
constexpr uint32_t kTmemCols = 512;
static_assert(kNumTm * kSlotCols <= int(kTmemCols), "tensor memory budget");

// Shared memory map (offsets from a 1024-byte aligned base).
constexpr int kRawASub = BM * 128;                   // 16 KB: 128 rows x 128 B, swizzled
constexpr int kRawA = 2 * kRawASub;                  // 256 k of int8
constexpr int kRawB = BN * 144;                      // raw q4_K rows
constexpr int kRawDa = BM * 8 * 4;                   // da [128][8] f32
constexpr int kRawSa = BM * 8 * 4;                   // sa [128][8] i32
constexpr int kOffRawB = kRawA, kOffRawDa = kRawA + kRawB, kOffRawSa = kOffRawDa + kRawDa;
constexpr int kRawStage = kOffRawSa + kRawSa;        // 58 KB: everything one super-block needs from HBM
constexpr int kOpTile = 128 * 128;                   // 128 rows x 64 fp16 (128 B), swizzled
constexpr int kOpStage = 2 * kOpTile;                // A + B
constexpr int kMinTile = 128 * 128;                  // 128 rows x 32 tf32 slots (24 used), swizzled
constexpr int kMinStage = 2 * kMinTile;              // dma parts + dmv parts
constexpr int kSclDa = 8 * BM * 4;                   // da [8 chunks][128 rows] f32
constexpr int kSclD = BN * 4;                        // d * 2^24 [128 weight rows] f32
constexpr int kSclStage = kSclDa + kSclD;            // 4.5 KB
constexpr int kOffRaw = 0;
constexpr int kOffOp = kOffRaw + kNumRaw * kRawStage;
constexpr int kOffMin = kOffOp + kNumOp * kOpStage;
constexpr int kOffScl = kOffMin + kMinStage;
constexpr int kOffBar = kOffScl + kNumScl * kSclStage;
// barriers: raw full/empty, op full/empty, tm full/empty, scl full/empty, min full/empty
constexpr int kNumBars = 2 * kNumRaw + 2 * kNumOp + 2 * kNumTm + 2 * kNumScl + 2;
constexpr int kOffMisc = kOffBar + kNumBars * 8;     // tmem slot, abort flag
constexpr int kSmemBytes = kOffMisc + 16 + 1024;     // + alignment slack
static_assert(kOffOp % 1024 == 0 && kOffMin % 1024 == 0, "operand tiles need 1024-byte alignment");
static_assert(kRawStage % 1024 == 0 && kSclStage % 16 == 0, "stage alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kRawTx = kRawStage;
constexpr uint32_t kIdesc = idesc_f16_f32(BM, BN);
constexpr uint32_t kIdescTf32 = idesc_tf32_f32(BM, BN);

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

// kGlu: the weight rows alternate gate / up rows; write SwiGLU(gate, up)
// quantized to q8_1 (and, if C is not null, as f32 [M][N/2] into C).
// kDump: kNoDump, or write the exact block dots instead of C (kDumpS: S with
// sc left out of the weight operand; kDumpScaled: S' = sc * S from the
// product's own operand); kQ8: also (or only, C == nullptr) write the result
// quantized to q8_1.
constexpr int kNoDump = 0, kDumpS = 1, kDumpScaled = 2;
template <int kDump, bool kQ8, bool kGlu = false>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const __grid_constant__ TmaMaps maps, float* __restrict__ C, mmq_q8_1_t q8out,
               int32_t* __restrict__ S, int M, int N, int K, int split, int* status, int inject_timeout,
               int tile_lo, int num_tiles) {
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
    // This launch covers tiles [tile_lo, num_tiles) (a launch may take only
    // the last, partial round of a larger GEMM).  Persistent mode (split ==
    // 1): CTAs stride over those tiles with all of K.  Split mode: a cluster
    // of `split` CTAs shares one tile, rank r takes super-blocks
    // [nsb*r/split, nsb*(r+1)/split), and rank 0 adds the partial sums in
    // rank order.
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
        mbar_init(bars.min_full(), kNumSclWarps);
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
            // programmatic dependent launch: everything before this point (the
            // tensor-memory allocation, barriers, tensor-map prefetch) may overlap
            // the previous kernel; its outputs (the activations) are read only
            // after it has completed.  Every later global access of this kernel
            // depends on these copies through the mbarriers.
            griddep_wait();
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
            Ring<1> mr;
            uint32_t last_bar = 0, last_par = 0;   // most recent commit, drained on exit
            const uint32_t minA = sbase + kOffMin, minB = minA + kMinTile;
            for (int tile = tile_first; tile < num_tiles; tile += tile_step) {
                for (int sb = sb_lo; sb < sb_hi; ++sb) {
                    for (int q = 0; q < 4; ++q) {   // operand stage q: chunks 2q, 2q+1
                        // probe both barriers back to back, block only on what is not ready
                        const bool of = mbar_try_wait(bars.op_full(orr.slot), orr.phase);
                        const bool te = mbar_try_wait(bars.tm_empty(tr.slot), tr.phase ^ 1u);
                        if (!of && !wait_bounded(bars.op_full(orr.slot), orr.phase, abort_flag, status))
                            goto mma_done;
                        if (!te && !wait_bounded(bars.tm_empty(tr.slot), tr.phase ^ 1u, abort_flag, status))
                            goto mma_done;
                        tc_fence_after();
                        // descriptors: the 14-bit start-address field is the only one that moves
                        const uint64_t dA = smem_desc_sw128(sbase + kOffOp + orr.slot * kOpStage);
                        const uint64_t dB = dA + uint64_t(kOpTile >> 4);
                        const uint32_t d0 = tmem_base + uint32_t(tr.slot * kSlotCols);
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int kk = 0; kk < 2; ++kk) {
                                const uint64_t koff = uint64_t((h * 64 + kk * 32) >> 4);   // 16-byte units
                                mma_f16(d0 + uint32_t(h * BN), dA + koff, dB + koff, kIdesc, uint32_t(kk));
                            }
                        mma_commit(bars.tm_full(tr.slot));
                        mma_commit(bars.op_empty(orr.slot));
                        last_bar = bars.op_empty(orr.slot);
                        last_par = orr.phase;
                        tr.next();
                        orr.next();
                    }
                    if (!kDump) {
                        // second term of this super-block: three K=8 tf32 MMAs into the
                        // next slot, handed to the epilogue like a fifth stage
                        if (!wait_bounded(bars.min_full(), mr.phase, abort_flag, status)) goto mma_done;
                        if (!wait_bounded(bars.tm_empty(tr.slot), tr.phase ^ 1u, abort_flag, status))
                            goto mma_done;
                        tc_fence_after();
                        const uint32_t d = tmem_base + uint32_t(tr.slot * kSlotCols);
#pragma unroll
                        for (int j = 0; j < 3; ++j)
                            mma_tf32(d, smem_desc_sw128(minA + 32 * j), smem_desc_sw128(minB + 32 * j),
                                     kIdescTf32, uint32_t(j));
                        mma_commit(bars.tm_full(tr.slot));
                        mma_commit(bars.min_empty());
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
        const int ts = threadIdx.x - kSclWarp0 * 32;   // 0..63: rows ts and ts + 64
        Ring<kNumRaw> rr;
        Ring<kNumScl> sr;
        Ring<1> mr;
        for (int tile = tile_first; tile < num_tiles; tile += tile_step) {
            for (int sb = sb_lo; sb < sb_hi; ++sb) {
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
                        const uint32_t minA = sbase + kOffMin, minB = minA + kMinTile;
#pragma unroll
                        for (int rh = 0; rh < 2; ++rh) {
                            const int t = ts + 64 * rh;
                            const int sw = t & 7;
                            // token row t: dma = da * sa per chunk, split hi / lo; k slots
                            // 0-7 hi, 8-15 hi, 16-23 lo (against hi, lo, hi of dmv); four
                            // chunks (one 16-byte granule) at a time
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
                            // weight row t: dmv = -dmin * m per chunk (exact in f32), split hi / lo
                            const uint4 hdr = ld_shared_v4(raw + kOffRawB + t * 144);
                            const float dmn = __half2float(__ushort_as_half(uint16_t(hdr.x >> 16)));
                            const uint32_t rb = minB + t * 128;
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
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bars.min_full());
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
        const int t = threadIdx.x - kConvWarp0 * 32;   // 0..127: this thread's row
        const int sw = t & 7;
        Ring<kNumRaw> rr;
        Ring<kNumOp> orr;
        for (int tile = tile_first; tile < num_tiles; tile += tile_step) {
            for (int sb = sb_lo; sb < sb_hi; ++sb) {
                if (!wait_bounded(bars.raw_full(rr.slot), rr.phase, abort_flag, status)) goto conv_done;
                const uint32_t raw = sbase + kOffRaw + rr.slot * kRawStage;
                const uint32_t rawB = raw + kOffRawB + t * 144 + 16;
                uint32_t scw_lo = 0x01010101u, scw_hi = 0x01010101u;   // the S dump keeps sc out
                if (kDump != kDumpS) {
                    const uint4 hdr = ld_shared_v4(raw + kOffRawB + t * 144);
                    scw_lo = sc_lo4(hdr.y);
                    scw_hi = sc_hi4(hdr.y, hdr.w);
                }
                for (int q = 0; q < 4; ++q) {   // chunk pair q = chunks 2q, 2q+1
                    if (!wait_bounded(bars.op_empty(orr.slot), orr.phase ^ 1u, abort_flag, status))
                        goto conv_done;
                    const uint32_t scw = q < 2 ? scw_lo : scw_hi;
                    const uint32_t sh = 16u * uint32_t(q & 1);
                    const uint32_t sca = (scw >> sh) & 0xFFu;          // chunk 2q: low nibbles
                    const uint32_t scb = (scw >> (sh + 8u)) & 0xFFu;   // chunk 2q+1: high nibbles
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
                            // two nibbles per 32-bit word, one per 16-bit half; times sc
                            // (<= 63 * 15 = 945, no carry into the upper half)
                            lo[2 * u] = (ww[u] & 0x000F000Fu) * sca;            // {e0, e2} low nibbles
                            lo[2 * u + 1] = ((ww[u] >> 8) & 0x000F000Fu) * sca; // {e1, e3}
                            hi[2 * u] = ((ww[u] >> 4) & 0x000F000Fu) * scb;
                            hi[2 * u + 1] = ((ww[u] >> 12) & 0x000F000Fu) * scb;
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
        // Thread = token row quarter*32 + lane (the tensor-memory lane quarter
        // this warp may read) x 64 columns colhalf*64 + [0, 64).
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
            const int m0 = (tile / tiles_n) * BM, n0 = (tile % tiles_n) * BN;
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = 0ull;
            for (int sb = sb_lo; sb < sb_hi; ++sb) {
                if (!wait_bounded(bars.scl_full(sr.slot), sr.phase, abort_flag, status)) goto epi_done;
                const uint32_t dat = sbase + kOffScl + sr.slot * kSclStage;
#pragma unroll
                for (int i = 0; i < 32; ++i) asb[i] = 0ull;
                for (int q = 0; q < 4; ++q) {   // operand stage q: chunks 2q, 2q+1 in one slot
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
                        if (lane == 0) mbar_arrive(bars.tm_empty(tr.slot));
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
                        // both S' tiles of this stage are in registers: hand the slot back
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bars.tm_empty(tr.slot));
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
                    // acc += the second term of this super-block (the fifth slot use)
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
                    if (lane == 0) mbar_arrive(bars.tm_empty(tr.slot));
                    tr.next();
                    half_fma<1>(acc, b, one2);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.scl_empty(sr.slot));
                sr.next();
            }
            if (!kDump && split == 1) {
                if (kGlu) {
                    store_tile_swiglu_q8_1(q8out, C, acc, M, N / 2, m0, n0, row, colhalf);
                } else {
                    if (!kQ8 || C) store_tile(C, acc, M, N, m0, n0, row, colhalf);
                    if (kQ8) store_tile_q8_1(q8out, acc, M, N, m0, n0, row, colhalf);
                }
            }
        }
    epi_done:;
        if (split > 1 && !kDump && !kQ8 && !kGlu) {
            // Reduce-scatter over the cluster: rank r owns the tile's columns
            // [r*W, (r+1)*W), W = BN / split.  Every thread pushes the columns
            // it holds for another rank into that rank's (idle) staging memory,
            // landing[src][row][W] f32; then each rank's owners add the split
            // partials in rank order (the same additions, in the same order,
            // as one rank pulling them all) and store their W columns.  Stores
            // to a peer need no round trip, and the ranks reduce in parallel.
            const int W = BN / split;                        // 64, 32 or 16
            const int lw = W == 64 ? 6 : (W == 32 ? 5 : 4);   // log2 W
            const int tile_m0 = (tile_first / tiles_n) * BM, tile_n0 = (tile_first % tiles_n) * BN;
            const int64_t gr = int64_t(tile_m0) + row;
            cluster_sync_all();   // every CTA of the cluster is done with its staging memory
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int c = colhalf * 64 + 4 * i;   // first of this float4's columns in the tile
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
        } else if (split > 1) {
            // Each rank leaves its partial tile in its own (now idle) staging
            // memory; rank 0 pulls ranks 1..split-1 in order and stores C.
            const int e = threadIdx.x - kEpiWarp0 * 32;   // 0..255
            float4* mine = reinterpret_cast<float4*>(smem + kOffRaw) + e * 16;
#pragma unroll
            for (int i = 0; i < 16; ++i)
                mine[i] = make_float4(lo_f(acc[2 * i]), hi_f(acc[2 * i]), lo_f(acc[2 * i + 1]),
                                      hi_f(acc[2 * i + 1]));
            cluster_sync_all();
            if (rank == 0 && !kDump) {
                for (int r = 1; r < split; ++r) {
                    const uint32_t remote = map_shared_rank(sbase + kOffRaw + uint32_t(e) * 256u, uint32_t(r));
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float4 v = ld_dsmem_v4(remote + uint32_t(i) * 16u);
                        acc[2 * i] = pack2(lo_f(acc[2 * i]) + v.x, hi_f(acc[2 * i]) + v.y);
                        acc[2 * i + 1] = pack2(lo_f(acc[2 * i + 1]) + v.z, hi_f(acc[2 * i + 1]) + v.w);
                    }
                }
                const int m0 = (tile_first / tiles_n) * BM, n0 = (tile_first % tiles_n) * BN;
                if (kGlu) {
                    store_tile_swiglu_q8_1(q8out, C, acc, M, N / 2, m0, n0, row, colhalf);
                } else {
                    if (!kQ8 || C) store_tile(C, acc, M, N, m0, n0, row, colhalf);
                    if (kQ8) store_tile_q8_1(q8out, acc, M, N, m0, n0, row, colhalf);
                }
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

// The launches of one call: [0, tail_lo) persistent (or K split over
// clusters of first_split CTAs when the tiles are few), then, if tail_lo <
// tiles, the tiles [tail_lo, tiles) of the last partial round with K split
// over clusters of tail_split CTAs.
TcPlan tc_plan(int64_t M, int64_t N, int64_t K, int nsm, bool allow_tail) {
    TcPlan p;
    const int64_t nsb = K / 256;
    p.tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    p.tail_lo = p.tiles;
    // the largest power-of-two split (<= 8, <= the super-blocks) that keeps
    // n tiles x split CTAs within one round of the SMs
    auto split_for = [&](int64_t n) {
        int sp = 1;
        while (sp < 8 && n * sp * 2 <= nsm && sp * 2 <= nsb) sp *= 2;
        return sp;
    };
    // Few tiles: split K over a cluster so that most SMs get work.
    if (p.tiles * 2 <= nsm) {
        p.first_split = split_for(p.tiles);
        return p;
    }
    // Many tiles: whole persistent rounds, then the partial last round's tiles
    // (at most half the SMs' worth) with K split, so that the idle SMs share it.
    const int64_t rem = p.tiles % nsm;
    if (allow_tail && p.tiles > nsm && rem > 0 && split_for(rem) > 1) {
        // at least 4 super-blocks per rank: a rank's fixed start-up and
        // reduction cost is not worth fewer (gate/up's 8 tail tiles: split 4)
        int sp = split_for(rem);
        while (sp > 2 && nsb / sp < 4) sp /= 2;
        p.tail_lo = p.tiles - rem;
        p.tail_split = sp;
    }
    return p;
}

int tc_gemm_launch_count(int64_t M, int64_t N, int64_t K) {
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    const TcPlan p = tc_plan(M, N, K, nsm, true);
    return p.tail_lo < p.tiles ? 2 : 1;
}

cudaError_t launch_gemm_tc(mmq_q8_1_t aq, const uint8_t* w, float* C, mmq_q8_1_t q8out, int32_t* S, int64_t M,
                           int64_t N, int64_t K, int* status, int inject_timeout, cudaStream_t s, bool swiglu,
                           bool dump_scaled) {
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
    cudaFuncAttributes fa;
    auto k = S ? (dump_scaled ? gemm_tc_kernel<kDumpScaled, false> : gemm_tc_kernel<kDumpS, false>)
               : swiglu ? gemm_tc_kernel<kNoDump, true, true>
               : (q8out.qs ? gemm_tc_kernel<kNoDump, true> : gemm_tc_kernel<kNoDump, false>);
    {
        cudaError_t e = cudaFuncGetAttributes(&fa, k);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != int(kRegsLaunch)) return cudaErrorInvalidConfiguration;
    }
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes)))
        return e;
    // One launch over tiles [lo, hi): persistent with one CTA per SM, or K
    // split over clusters of `split` CTAs, one tile per cluster.
    auto launch = [&](int64_t lo, int64_t hi, int split, int inject) -> cudaError_t {
        const int64_t n = hi - lo;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(unsigned(split > 1 ? n * split : (n < nsm ? n : nsm)));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = size_t(kSmemBytes);
        cfg.stream = s;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = unsigned(split);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (mmq::programmatic_launch_enabled()) {
            attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[1].val.programmaticStreamSerializationAllowed = 1;
            cfg.numAttrs = 2;
        }
        const cudaError_t le = cudaLaunchKernelEx(&cfg, k, maps, C, q8out, S, int(M), int(N), int(K), split, status,
                                                  inject, int(lo), int(hi));
        return le != cudaSuccess ? le : cudaGetLastError();
    };
    const TcPlan p = tc_plan(M, N, K, nsm, S == nullptr);
    // tile indices (and a tile plus the stride over tiles) stay in int
    if (p.tiles > (int64_t(1) << 30)) return cudaErrorInvalidValue;
    if (p.tail_lo == p.tiles) return launch(0, p.tiles, p.first_split, inject_timeout);
    if ((e = launch(0, p.tail_lo, 1, inject_timeout)) != cudaSuccess) return e;
    return launch(p.tail_lo, p.tiles, p.tail_split, 0);
}

}  // namespace mmq
