// q4_K x q8_1 GEMM on the tcgen05 tensor cores, accumulating a whole 256-k
// super-block in tensor memory, with the activations taken from the operand
// plane the prepass writes (quantize.cu, tensor-core form).
//
// Math (web page "20 . r15 -- f32-accumulate mma probe (dead end) + rank-1
// term2 rescale", section 2.1): for every 32-k chunk c
//     C_ij += (da_ic * d_j * sc_jc) * S_ijc + dma_ic * dmv_jc,
// S the exact integer dot of the chunk, dmv = -dmin*m, and dma = da*sa formed
// once per token row and chunk (the rank-1 fold of web page "21 . r16 --
// Narrow kernel gets the rank-1 fold", section 2.1).  This kernel regroups
// the sum per super-block b (eight chunks) so that the tensor core applies
// the per-chunk activation scale:
//     C_ij += d'_j * 2^24 * g_ib * T_ijb,
//     T_ijb = sum_c sum_k (hi_ik + lo_ik) (sc_jc v_jk 2^-24)
//           + sum_c (dma_ic / g_ib) (-m_jc (dmin_j / d'_j) 2^-24),
// where g_ib = 2^E is a power of two per token row and super-block, hi + lo
// is within 2^-14 of q_ik * da_ic / g_ib (two fp16 parts, the first an exact
// product), and d' = d, or 1 where d = 0 (then the weight operand of that
// super-block is zero, so T holds the second term alone).
//   * Activation operand: hi and lo from the prepass's plane (one 128-byte
//     line per token row and chunk, 32 hi then 32 lo), loaded by TMA straight
//     into the MMA's 128B-swizzled K-major layout; both are MMA'd against the
//     same weight operand into one accumulator.
//   * Weight operand: sc*v <= 945 written as the fp16 subnormal sc*v * 2^-24
//     (the integer in the mantissa bits), exact.
//   * The second term: per super-block an 8-long contraction, three K=8 tf32
//     MMAs on hi/lo splits of both factors (hi*hi + hi*lo + lo*hi) into the
//     same accumulator; the activation factors come split from the prepass.
// So the accumulator holds a whole super-block: the epilogue reads tensor
// memory once per super-block and does one packed multiply and one packed
// FMA per output, and no thread converts activations.
//
// One CTA per SM, persistent over 128 (tokens) x 256 (weight rows) tiles;
// every MMA is one M=128, N=256 instruction.  Warp roles (16 warps,
// setmaxnreg moves registers to the epilogue, which keeps a 128 x 256 f32
// tile):
//   warp 0      TMA producer: per super-block the 256 q4_K block headers
//               and the second term's activation factors, per pair of
//               chunks the 256 rows' 32 quant bytes, per chunk the hi|lo
//               activation tile.
//   warp 1      MMA issuer (one thread): per chunk two K=16 f16 MMAs for hi
//               and two for lo, per super-block three K=8 tf32 MMAs; one
//               accumulator slot (256 tensor-memory columns) per super-block,
//               two slots.
//   warps 2-3   per super-block: d' * 2^24 per weight row for the epilogue
//               and the split tf32 weight factors of the second term.
//   warps 4-7   weight converters, two weight rows per thread, one chunk per
//               stage: nibble * sc -> fp16 subnormal (64B swizzle).
//   warps 8-15  epilogue: thread = token row, 128 columns; per super-block
//               eight 32x32b.x16 tensor-memory loads and 64 + 64 packed
//               multiplies / FMAs; C stored at the end of a tile.
// Within a chunk the k order of both operands is 0,2,1,3 per group of four
// (the pair order of the nibble unpack; the prepass writes the activations
// in the same order): a dot product does not depend on the order of its
// terms.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "mmq_internal.h"
#include "sm103_ptx.cuh"
#include "tc_common.cuh"

namespace {

using namespace mmq::ptx;
using namespace mmq::tc;

constexpr int BM = 128;          // token rows per tile
constexpr int BN = 256;          // weight rows per tile (the MMA's N)
constexpr int kNumA = 5, kNumB = 3, kNumWH = 2, kNumWN = 4, kNumTm = 2, kNumTab = 2;
constexpr int kTabWarp0 = 2, kNumTabWarps = 2, kConvWarp0 = 4, kNumConvWarps = 4;
constexpr int kEpiWarp0 = 8, kNumEpiWarps = 8;
constexpr int kThreads = (kEpiWarp0 + kNumEpiWarps) * 32;   // 512
constexpr uint32_t kRegsLow = 72, kRegsHigh = 184, kRegsLaunch = 128;
static_assert(256 * kRegsLow + 256 * kRegsHigh <= kThreads * kRegsLaunch, "register split");
constexpr int kSlotCols = BN;
constexpr uint32_t kTmemCols = 512;
static_assert(kNumTm * kSlotCols <= int(kTmemCols), "tensor memory budget");

// Shared memory map (offsets from a 1024-byte aligned base).
constexpr int kAStage = BM * 128;      // 16 KB: 128 token rows x (32 hi | 32 lo) fp16, 128B swizzle
constexpr int kBStage = BN * 64;       // 16 KB: 256 weight rows x 32 fp16, 64B swizzle
constexpr int kWHStage = BN * 16;      // 4 KB: the 256 rows' block headers (d, dmin, 12 scale bytes)
constexpr int kWNStage = BN * 32;      // 8 KB: the 256 rows' quant bytes of one pair of chunks
constexpr int kT2A = BM * 128;         // 16 KB: 128 rows x 32 tf32 slots (24 used), 128B swizzle
constexpr int kT2B = BN * 128;         // 32 KB
constexpr int kTabStage = BN * 4;      // d' * 2^24 per weight row
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kNumA * kAStage;
constexpr int kOffWN = kOffB + kNumB * kBStage;
constexpr int kOffWH = kOffWN + kNumWN * kWNStage;
constexpr int kOffT2 = kOffWH + kNumWH * kWHStage;
constexpr int kOffTab = kOffT2 + kT2A + kT2B;
constexpr int kOffBar = kOffTab + kNumTab * kTabStage;
constexpr int kNumBars = 2 * kNumA + 2 * kNumB + 2 * kNumWH + 2 * kNumWN + 3 + 2 * kNumTm + 2 * kNumTab;
constexpr int kOffMisc = kOffBar + kNumBars * 8;   // tmem slot, abort flag, scratch word
constexpr int kSmemBytes = kOffMisc + 16 + 1024;   // + alignment slack
static_assert(kOffB % 1024 == 0 && kOffWN % 1024 == 0 && kOffT2 % 1024 == 0, "operand tiles need 1024-byte alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kIdesc = idesc_f16_f32(BM, BN);
constexpr uint32_t kIdescTf32 = idesc_tf32_f32(BM, BN);

struct TmaMaps {
    CUtensorMap a, t2, wh, wn;
};

struct Bars {
    uint32_t base;
    __device__ uint32_t at(int i) const { return base + 8u * uint32_t(i); }
    __device__ uint32_t a_full(int s) const { return at(s); }
    __device__ uint32_t a_empty(int s) const { return at(kNumA + s); }
    static constexpr int kB0 = 2 * kNumA;
    __device__ uint32_t b_full(int s) const { return at(kB0 + s); }
    __device__ uint32_t b_empty(int s) const { return at(kB0 + kNumB + s); }
    static constexpr int kWH0 = kB0 + 2 * kNumB;
    __device__ uint32_t wh_full(int s) const { return at(kWH0 + s); }
    __device__ uint32_t wh_empty(int s) const { return at(kWH0 + kNumWH + s); }
    static constexpr int kWN0 = kWH0 + 2 * kNumWH;
    __device__ uint32_t wn_full(int s) const { return at(kWN0 + s); }
    __device__ uint32_t wn_empty(int s) const { return at(kWN0 + kNumWN + s); }
    static constexpr int kT20 = kWN0 + 2 * kNumWN;
    __device__ uint32_t t2a_full() const { return at(kT20); }       // activation factors (TMA)
    __device__ uint32_t t2b_full() const { return at(kT20 + 1); }   // weight factors (table warps)
    __device__ uint32_t t2_empty() const { return at(kT20 + 2); }
    static constexpr int kTm0 = kT20 + 3;
    __device__ uint32_t tm_full(int s) const { return at(kTm0 + s); }
    __device__ uint32_t tm_empty(int s) const { return at(kTm0 + kNumTm + s); }
    static constexpr int kTab0 = kTm0 + 2 * kNumTm;
    __device__ uint32_t tab_full(int s) const { return at(kTab0 + s); }
    __device__ uint32_t tab_empty(int s) const { return at(kTab0 + kNumTab + s); }
};
static_assert(Bars::kTab0 + 2 * kNumTab == kNumBars, "barrier count");

__global__ void __launch_bounds__(kThreads, 1)
gemm_sb_kernel(const __grid_constant__ TmaMaps maps, const float* __restrict__ gplane, float* __restrict__ C,
               int M, int N, int K, int* status, int inject_timeout) {
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
    const int num_tiles = ((M + BM - 1) / BM) * tiles_n;
    const int tile_first = int(blockIdx.x), tile_step = int(gridDim.x);
    // Each tile walks its super-blocks from a start that depends on its row
    // and column tile, so that the tiles sharing a row band (or a weight
    // band) touch different super-blocks at any time: a neighbour's earlier
    // fetch is then already in L2 (the order of the sum is fixed per tile).
    auto sb_at = [=](int tile, int k) {
        const int start = (tile / tiles_n + tile % tiles_n) % nsb;
        return k + start < nsb ? k + start : k + start - nsb;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kNumA; ++s) {
            mbar_init(bars.a_full(s), 1);
            mbar_init(bars.a_empty(s), 1);
        }
        for (int s = 0; s < kNumB; ++s) {
            mbar_init(bars.b_full(s), kNumConvWarps);
            mbar_init(bars.b_empty(s), 1);
        }
        for (int s = 0; s < kNumWH; ++s) {
            mbar_init(bars.wh_full(s), 1);
            mbar_init(bars.wh_empty(s), kNumConvWarps + kNumTabWarps);
        }
        for (int s = 0; s < kNumWN; ++s) {
            mbar_init(bars.wn_full(s), 1);
            mbar_init(bars.wn_empty(s), kNumConvWarps);
        }
        mbar_init(bars.t2a_full(), 1);
        mbar_init(bars.t2b_full(), kNumTabWarps);
        mbar_init(bars.t2_empty(), 1);
        for (int s = 0; s < kNumTm; ++s) {
            mbar_init(bars.tm_full(s), 1);
            mbar_init(bars.tm_empty(s), kNumEpiWarps);
        }
        for (int s = 0; s < kNumTab; ++s) {
            mbar_init(bars.tab_full(s), kNumTabWarps);
            mbar_init(bars.tab_empty(s), kNumEpiWarps);
        }
        abort_flag.set(0u);
        fence_barrier_init();
        fence_proxy_async_smem();
        prefetch_tmap(&maps.a);
        prefetch_tmap(&maps.t2);
        prefetch_tmap(&maps.wh);
        prefetch_tmap(&maps.wn);
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
            // programmatic dependent launch: the activation plane is read only
            // after the previous kernel on the stream has completed.
            griddep_wait();
            Ring<kNumA> ar;
            Ring<kNumWH> hr;
            Ring<kNumWN> nr;
            Ring<1> t2r;
            int a_issued[kNumA] = {}, h_issued[kNumWH] = {}, n_issued[kNumWN] = {}, t2_issued = 0;
            uint32_t a_par[kNumA] = {}, h_par[kNumWH] = {}, n_par[kNumWN] = {}, t2_par = 0;
            bool first = true;
            for (int tile = tile_first; tile < num_tiles; tile += tile_step) {
                const int m0 = (tile / tiles_n) * BM, n0 = (tile % tiles_n) * BN;
                for (int kq = 0; kq < nsb; ++kq) {
                    const int sb = sb_at(tile, kq);
                    if (!wait_bounded(bars.wh_empty(hr.slot), hr.phase ^ 1u, abort_flag, status))
                        goto producer_done;
                    if (!(first && inject_timeout)) {   // test hook: withhold this arrival
                        const uint32_t fb = bars.wh_full(hr.slot);
                        mbar_arrive_expect_tx(fb, uint32_t(kWHStage));
                        tma_load_2d(sbase + kOffWH + hr.slot * kWHStage, &maps.wh, fb, sb * 144, n0);
                        h_issued[hr.slot] = 1;
                        h_par[hr.slot] = hr.phase;
                    }
                    first = false;
                    hr.next();
                    for (int c = 0; c < 8; ++c) {
                        if ((c & 1) == 0) {
                            // the quant bytes of chunks c, c+1 (nibble 0 and 1 of the same bytes)
                            if (!wait_bounded(bars.wn_empty(nr.slot), nr.phase ^ 1u, abort_flag, status))
                                goto producer_done;
                            const uint32_t fb = bars.wn_full(nr.slot);
                            mbar_arrive_expect_tx(fb, uint32_t(kWNStage));
                            tma_load_2d(sbase + kOffWN + nr.slot * kWNStage, &maps.wn, fb, sb * 144 + 16 + 16 * c, n0);
                            n_issued[nr.slot] = 1;
                            n_par[nr.slot] = nr.phase;
                            nr.next();
                        }
                        if (!wait_bounded(bars.a_empty(ar.slot), ar.phase ^ 1u, abort_flag, status))
                            goto producer_done;
                        const uint32_t fb = bars.a_full(ar.slot);
                        mbar_arrive_expect_tx(fb, uint32_t(kAStage));
                        tma_load_2d(sbase + kOffA + ar.slot * kAStage, &maps.a, fb, (sb * 8 + c) * 64, m0);
                        a_issued[ar.slot] = 1;
                        a_par[ar.slot] = ar.phase;
                        ar.next();
                    }
                    // the second term's activation factors (single buffer: after
                    // the previous super-block's tf32 MMAs have read it)
                    if (!wait_bounded(bars.t2_empty(), t2r.phase ^ 1u, abort_flag, status)) goto producer_done;
                    mbar_arrive_expect_tx(bars.t2a_full(), uint32_t(kT2A));
                    tma_load_2d(sbase + kOffT2, &maps.t2, bars.t2a_full(), sb * 32, m0);
                    t2_issued = 1;
                    t2_par = t2r.phase;
                    t2r.next();
                }
            }
        producer_done:
            // Let every copy already issued land before the CTA can exit.
            for (int s = 0; s < kNumWH; ++s)
                if (h_issued[s]) wait_drain(bars.wh_full(s), h_par[s], status);
            for (int s = 0; s < kNumWN; ++s)
                if (n_issued[s]) wait_drain(bars.wn_full(s), n_par[s], status);
            for (int s = 0; s < kNumA; ++s)
                if (a_issued[s]) wait_drain(bars.a_full(s), a_par[s], status);
            if (t2_issued) wait_drain(bars.t2a_full(), t2_par, status);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            Ring<kNumA> ar;
            Ring<kNumB> br;
            Ring<kNumTm> tr;
            Ring<1> t2r;
            uint32_t last_bar = 0, last_par = 0;   // most recent commit, drained on exit
            const uint32_t t2A = sbase + kOffT2, t2B = t2A + kT2A;
            for (int tile = tile_first; tile < num_tiles; tile += tile_step) {
                for (int kq = 0; kq < nsb; ++kq) {
                    const int sb = sb_at(tile, kq);
                    if (!wait_bounded(bars.tm_empty(tr.slot), tr.phase ^ 1u, abort_flag, status)) goto mma_done;
                    tc_fence_after();
                    const uint32_t d = tmem_base + uint32_t(tr.slot * kSlotCols);
                    for (int c = 0; c < 8; ++c) {
                        if (!wait_bounded(bars.a_full(ar.slot), ar.phase, abort_flag, status)) goto mma_done;
                        if (!wait_bounded(bars.b_full(br.slot), br.phase, abort_flag, status)) goto mma_done;
                        tc_fence_after();
                        // A: hi in bytes 0-63 and lo in bytes 64-127 of each swizzled row
                        const uint64_t dA = smem_desc_sw128(sbase + kOffA + ar.slot * kAStage);
                        const uint64_t dB = smem_desc_sw64(sbase + kOffB + br.slot * kBStage);
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            const uint64_t ko = uint64_t((kk * 32) >> 4);   // 16-byte units
                            mma_f16(d, dA + ko, dB + ko, kIdesc, uint32_t((c | kk) != 0));
                            mma_f16(d, dA + ko + 4, dB + ko, kIdesc, 1u);
                        }
                        mma_commit(bars.a_empty(ar.slot));
                        mma_commit(bars.b_empty(br.slot));
                        last_bar = bars.b_empty(br.slot);
                        last_par = br.phase;
                        ar.next();
                        br.next();
                    }
                    // the second term of this super-block into the same accumulator
                    if (!wait_bounded(bars.t2a_full(), t2r.phase, abort_flag, status)) goto mma_done;
                    if (!wait_bounded(bars.t2b_full(), t2r.phase, abort_flag, status)) goto mma_done;
                    tc_fence_after();
#pragma unroll
                    for (int j = 0; j < 3; ++j)
                        mma_tf32(d, smem_desc_sw128(t2A + 32 * j), smem_desc_sw128(t2B + 32 * j), kIdescTf32, 1u);
                    mma_commit(bars.t2_empty());
                    mma_commit(bars.tm_full(tr.slot));
                    last_bar = bars.t2_empty();
                    last_par = t2r.phase;
                    t2r.next();
                    tr.next();
                }
            }
        mma_done:
            if (last_bar) wait_drain(last_bar, last_par, status);
        }
    } else if (warp < kConvWarp0) {
        // ------------------------------------------ weight-side tables
        const int ts = threadIdx.x - kTabWarp0 * 32;   // 0..63: weight rows ts + 64 q
        Ring<kNumWH> hr;
        Ring<kNumTab> tbr;
        Ring<1> t2r;
        for (int tile = tile_first; tile < num_tiles; tile += tile_step) {
            for (int kq = 0; kq < nsb; ++kq) {
                    const int sb = sb_at(tile, kq);
                if (!wait_bounded(bars.wh_full(hr.slot), hr.phase, abort_flag, status)) goto tab_done;
                {
                    const uint32_t hb = sbase + kOffWH + hr.slot * kWHStage;
                    uint4 hdr[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) hdr[q] = ld_shared_v4(hb + uint32_t(ts + 64 * q) * 16u);
                    // d' * 2^24 per weight row for the epilogue
                    if (!wait_bounded(bars.tab_empty(tbr.slot), tbr.phase ^ 1u, abort_flag, status))
                        goto tab_done;
                    const uint32_t tab = sbase + kOffTab + tbr.slot * kTabStage;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float dd = __half2float(__ushort_as_half(uint16_t(hdr[q].x & 0xFFFFu)));
                        if (dd == 0.0f) dd = 1.0f;
                        st_shared_u32(tab + uint32_t(ts + 64 * q) * 4u, __float_as_uint(dd * kSubnormalScale));
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars.tab_full(tbr.slot));
                    tbr.next();
                    // the second term's weight factors -m * (dmin / d') * 2^-24, split
                    // hi / lo in k slots 0-7 hi, 8-15 lo, 16-23 hi (against the
                    // activation side's hi, hi, lo)
                    if (!wait_bounded(bars.t2_empty(), t2r.phase ^ 1u, abort_flag, status)) goto tab_done;
                    const uint32_t t2B = sbase + kOffT2 + kT2A;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int j = ts + 64 * q;
                        const int sw = j & 7;
                        float dd = __half2float(__ushort_as_half(uint16_t(hdr[q].x & 0xFFFFu)));
                        if (dd == 0.0f) dd = 1.0f;
                        const float dmn = __half2float(__ushort_as_half(uint16_t(hdr[q].x >> 16)));
                        const float r = __fdiv_rn(dmn, dd) * (1.0f / kSubnormalScale);
                        const uint32_t rb = t2B + uint32_t(j) * 128u;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint32_t mw = h == 0 ? m_lo4(hdr[q].z) : m_hi4(hdr[q].z, hdr[q].w);
                            float bh[4], bl[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                split_tf32(-(float((mw >> (8 * i)) & 0xFFu) * r), bh[i], bl[i]);
                            st_shared_v4f(rb + (((0 + h) ^ sw) << 4), bh[0], bh[1], bh[2], bh[3]);
                            st_shared_v4f(rb + (((2 + h) ^ sw) << 4), bl[0], bl[1], bl[2], bl[3]);
                            st_shared_v4f(rb + (((4 + h) ^ sw) << 4), bh[0], bh[1], bh[2], bh[3]);
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars.t2b_full());
                    t2r.next();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.wh_empty(hr.slot));
                hr.next();
            }
        }
    tab_done:;
    } else {
        // ------------------------------------------------ weight converters
        const int t = threadIdx.x - kConvWarp0 * 32;   // weight rows t and t + 128
        Ring<kNumWH> hr;
        Ring<kNumWN> nr;
        Ring<kNumB> br;
        for (int tile = tile_first; tile < num_tiles; tile += tile_step) {
            for (int kq = 0; kq < nsb; ++kq) {
                    const int sb = sb_at(tile, kq);
                if (!wait_bounded(bars.wh_full(hr.slot), hr.phase, abort_flag, status)) goto conv_done;
                uint32_t scl[2], sch[2];
                {
                    // d = 0: the weight operand of this super-block is zero (the
                    // tables use d' = 1 and keep the second term)
                    const uint32_t hb = sbase + kOffWH + hr.slot * kWHStage;
                    const uint4 h0 = ld_shared_v4(hb + uint32_t(t) * 16u), h1 = ld_shared_v4(hb + uint32_t(t + 128) * 16u);
                    const bool z0 = (h0.x & 0x7FFFu) == 0u, z1 = (h1.x & 0x7FFFu) == 0u;
                    scl[0] = z0 ? 0u : sc_lo4(h0.y);
                    sch[0] = z0 ? 0u : sc_hi4(h0.y, h0.w);
                    scl[1] = z1 ? 0u : sc_lo4(h1.y);
                    sch[1] = z1 ? 0u : sc_hi4(h1.y, h1.w);
                }
                loads_done(sbase + kOffMisc + 8, scl[0] ^ sch[0] ^ scl[1] ^ sch[1]);
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.wh_empty(hr.slot));
                hr.next();
                uint4 nq[2][2];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    if ((c & 1) == 0) {
                        // nibble c%2 of this pair of chunks' 32 quant bytes of each row
                        if (!wait_bounded(bars.wn_full(nr.slot), nr.phase, abort_flag, status)) goto conv_done;
                        const uint32_t nb = sbase + kOffWN + nr.slot * kWNStage;
                        nq[0][0] = ld_shared_v4(nb + uint32_t(t) * 32u);
                        nq[0][1] = ld_shared_v4(nb + uint32_t(t) * 32u + 16u);
                        nq[1][0] = ld_shared_v4(nb + uint32_t(t + 128) * 32u);
                        nq[1][1] = ld_shared_v4(nb + uint32_t(t + 128) * 32u + 16u);
                        loads_done(sbase + kOffMisc + 8,
                                   nq[0][0].x ^ nq[0][0].y ^ nq[0][0].z ^ nq[0][0].w ^ nq[0][1].x ^ nq[0][1].y ^
                                       nq[0][1].z ^ nq[0][1].w ^ nq[1][0].x ^ nq[1][0].y ^ nq[1][0].z ^ nq[1][0].w ^
                                       nq[1][1].x ^ nq[1][1].y ^ nq[1][1].z ^ nq[1][1].w);
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bars.wn_empty(nr.slot));
                        nr.next();
                    }
                    if (!wait_bounded(bars.b_empty(br.slot), br.phase ^ 1u, abort_flag, status)) goto conv_done;
                    const uint32_t bst = sbase + kOffB + br.slot * kBStage;
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int row = t + 128 * r;
                        const uint32_t osw = uint32_t((row >> 1) & 3);
                        const uint32_t sc = ((c < 4 ? scl[r] : sch[r]) >> (8 * (c & 3))) & 0xFFu;
                        const uint32_t nw[8] = {nq[r][0].x, nq[r][0].y, nq[r][0].z, nq[r][0].w,
                                                nq[r][1].x, nq[r][1].y, nq[r][1].z, nq[r][1].w};
                        const uint32_t rowb = bst + uint32_t(row) * 64u;
#pragma unroll
                        for (int G = 0; G < 4; ++G) {
                            const uint32_t x0 = nw[2 * G] >> (4 * (c & 1)), x1 = nw[2 * G + 1] >> (4 * (c & 1));
                            // two nibbles per 32-bit word, one per 16-bit half, times
                            // sc (<= 63 * 15 = 945, no carry into the upper half)
                            st_shared_v4(rowb + ((uint32_t(G) ^ osw) << 4), (x0 & 0x000F000Fu) * sc,
                                         ((x0 >> 8) & 0x000F000Fu) * sc, (x1 & 0x000F000Fu) * sc,
                                         ((x1 >> 8) & 0x000F000Fu) * sc);
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars.b_full(br.slot));
                    br.next();
                }
            }
        }
    conv_done:;
    }
    } else {
        setmaxnreg_inc<kRegsHigh>();
        // ---------------------------------------------------------- epilogue
        // Thread = token row quarter*32 + lane (the tensor-memory lane quarter
        // this warp may read) x 128 columns colhalf*128 + [0, 128).
        const int ew = warp - kEpiWarp0;
        const int quarter = warp & 3;
        const int colhalf = ew >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t tlane = uint32_t(quarter * 32) << 16;
        Ring<kNumTab> tbr;
        Ring<kNumTm> tr;
        uint64_t acc[64];
        griddep_wait();   // the 2^E plane is the previous kernel's output
        for (int tile = tile_first; tile < num_tiles; tile += tile_step) {
            const int m0 = (tile / tiles_n) * BM, n0 = (tile % tiles_n) * BN;
            const int64_t gr = int64_t(m0) + row;
#pragma unroll
            for (int i = 0; i < 64; ++i) acc[i] = 0ull;
            for (int kq = 0; kq < nsb; ++kq) {
                    const int sb = sb_at(tile, kq);
                // 2^E of this token row and super-block (0 past M: nothing stored)
                const float g = gr < M ? __ldg(gplane + gr * nsb + sb) : 0.0f;
                const uint64_t g2 = pack2(g, g);
                if (!wait_bounded(bars.tab_full(tbr.slot), tbr.phase, abort_flag, status)) goto epi_done;
                const uint32_t fcol = sbase + kOffTab + tbr.slot * kTabStage + uint32_t(colhalf * 128) * 4u;
                if (!wait_bounded(bars.tm_full(tr.slot), tr.phase, abort_flag, status)) goto epi_done;
                tc_fence_after();
                const uint32_t ta = tmem_base + tlane + uint32_t(tr.slot * kSlotCols + colhalf * 128);
#pragma unroll
                for (int p = 0; p < 8; ++p) {
                    uint32_t b[16];
                    tmem_ld_32x32b_x16(ta + uint32_t(16 * p), b);
                    tmem_wait_ld(b);
                    if (p == 7) {
                        // the whole slot is in registers: hand it back
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bars.tm_empty(tr.slot));
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint4 fv = ld_shared_v4(fcol + uint32_t(16 * p + 4 * i) * 4u);
                        acc[8 * p + 2 * i] = ffma2(fmul2(pack2u(b[4 * i], b[4 * i + 1]), g2), pack2u(fv.x, fv.y),
                                                   acc[8 * p + 2 * i]);
                        acc[8 * p + 2 * i + 1] = ffma2(fmul2(pack2u(b[4 * i + 2], b[4 * i + 3]), g2),
                                                       pack2u(fv.z, fv.w), acc[8 * p + 2 * i + 1]);
                    }
                }
                tr.next();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.tab_empty(tbr.slot));
                tbr.next();
            }
            if (gr < M) {
                float* crow = C + gr * N;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int gc = n0 + colhalf * 128 + 4 * i;   // N % 4 == 0: all four or none
                    if (gc < N)
                        *reinterpret_cast<float4*>(crow + gc) =
                            make_float4(lo_f(acc[2 * i]), hi_f(acc[2 * i]), lo_f(acc[2 * i + 1]),
                                        hi_f(acc[2 * i + 1]));
                }
            }
        }
    epi_done:;
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

int sb_gemm_check_resources() {
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
        cudaGetLastError();
        return MMQ_ERR_CUDA;
    }
    return optin >= kSmemBytes ? MMQ_OK : MMQ_ERR_RESOURCE;
}

cudaError_t launch_gemm_sb(const void* tcop, const uint8_t* w, float* C, int64_t M, int64_t N, int64_t K,
                           int* status, int inject_timeout, cudaStream_t s) {
    TmaMaps maps;
    const TcopLayout L = tcop_layout(M, K);
    const char* b = static_cast<const char*>(tcop);
    const uint64_t nsb = uint64_t(K / 256);
    if (!encode_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT16, b + L.a, uint64_t(K) * 2, uint64_t(M), uint64_t(K) * 4,
                   64, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&maps.t2, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, b + L.t2, nsb * 32, uint64_t(M), nsb * 128, 32, BM,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&maps.wh, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, nsb * 144, uint64_t(N), nsb * 144, 16, BN,
                   CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&maps.wn, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, nsb * 144, uint64_t(N), nsb * 144, 32, BN,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    int dev = 0, nsm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    {
        // setmaxnreg needs exactly kRegsLaunch registers per thread at launch
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, gemm_sb_kernel);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != int(kRegsLaunch)) return cudaErrorInvalidConfiguration;
    }
    const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    if (tiles > (int64_t(1) << 30)) return cudaErrorInvalidValue;
    const int64_t ctas = tiles < nsm ? tiles : nsm;
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(gemm_sb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes)))
        return e;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = launch_config(dim3(unsigned(ctas)), dim3(kThreads), size_t(kSmemBytes), s, attr);
    e = cudaLaunchKernelEx(&cfg, gemm_sb_kernel, maps, reinterpret_cast<const float*>(b + L.g), C, int(M), int(N),
                           int(K), status, inject_timeout);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace mmq
