// q4_K x q8_1 GEMM for few tokens on the tcgen05 tensor cores of sm_103a.
//
// Math (web page "20 . r15 -- f32-accumulate mma probe (dead end) + rank-1
// term2 rescale", section 2.1): for every 32-k chunk c
//     C_ij += (da_ic * d_j * sc_jc) * S_ij + dma_ic * dmv_jc,
// S_ij the exact integer dot of the chunk, dmv = -dmin*m, dma = da*sa once
// per token row and chunk (the rank-1 fold, page "21 . r16 -- Narrow kernel
// gets the rank-1 fold", section 2.1).
//
// With few tokens the weight stream dominates, so the roles of the operands
// are swapped against the large-M kernel: 128 weight rows are the M = 128
// side of the MMA and the tokens, padded to NP = 16, 32 or 64, the N side.
// The exact integers go through kind::f16 as in the large-M kernel (int8
// quants are exact fp16 values, sc*v <= 945 is the fp16 subnormal
// sc*v * 2^-24), so each chunk's S'_ij = sc_jc * S_ij lands exactly in its
// own NP columns of tensor memory.  A tensor-memory slot holds a whole
// super-block (NP <= 32) or half of one (NP = 64), so the MMA thread commits
// and the epilogue waits once per slot, and 2 to 4 slots are in flight.
// A tcgen05 MMA costs ~70 cycles to issue whatever its N, so with few
// tokens the MMA thread and the operand conversion, not the tensor pipe,
// set the pace; the conversion is spread over eight warps.
//
// Epilogue (thread = weight row, NP/2 token columns; da and dma come from
// per-super-block tables, dmv and d * 2^24 are the thread's own scalars):
//     asb_ij  = sum_c da_ic * S'_ijc                 (one packed FMA per pair and chunk)
//     acc_ij += dma_ic * dmv_jc                      (the second term, per chunk)
//     acc_ij += d_j * 2^24 * asb_ij                  (once per super-block)
//
// K is split over a cluster of up to 8 CTAs; every rank leaves its partial
// tile in its own shared memory and rank r adds, in rank order, the parts
// held by epilogue warps w with w % split == r, then stores them (one
// 128-byte row segment of C per warp and token).
//
// Warp roles (20 warps; setmaxnreg moves registers to the epilogue):
//   warp 0      TMA producer: per super-block the raw 144-byte q4_K rows,
//               the raw int8 token tile (two 128-byte-swizzled boxes), the
//               da / sa slices, zero-filled past N / M.
//   warp 1      MMA issuer (one thread): per operand stage (two chunks)
//               four K=16 MMAs into a 2*NP-column tensor-memory slot.
//   warps 2-3   token tables per super-block: da and dma as [chunk][token].
//   warps 4-11  converters in two groups that take alternate operand stages
//               (NP = 64: one group, warps 4-7), thread = weight row:
//               nibble * sc -> fp16 subnormal (A), int8 tokens -> fp16 (B),
//               both into the 128-byte-swizzled K-major layout; group 0 also
//               writes the row's d * 2^24 and dmv.
//   warps 12-19 epilogue.
// Within a chunk the k order of both operands is permuted identically
// (groups of four as 0,2,1,3); a dot product does not depend on it.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "mmq_internal.h"
#include "sm103_ptx.cuh"
#include "tc_common.cuh"

namespace {

using namespace mmq::ptx;
using namespace mmq::tc;

constexpr int kRowsW = 128;                          // weight rows per CTA (MMA M)
constexpr int kSclWarp0 = 2, kNumSclWarps = 2, kConvWarp0 = 4, kNumEpiWarps = 8;
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxSplit = 8;
static_assert(kMaxSplit <= kNumEpiWarps, "one reducing warp per rank at least");

template <int NP>
struct Cfg {
    static_assert(NP == 16 || NP == 32 || NP == 64, "token tile");
    static constexpr int T = NP / 2;                          // token columns per epilogue thread
    // Warp roles: NP <= 32 has eight converter warps (two groups of four);
    // NP = 64 keeps four, so that its epilogue warps can hold 2 x 32 columns
    // of accumulators in registers.
    static constexpr int kNumConvWarps = NP == 64 ? 4 : 8;
    static constexpr int kEpiWarp0 = kConvWarp0 + kNumConvWarps;
    static constexpr int kThreads = (kEpiWarp0 + kNumEpiWarps) * 32;   // 512 or 640
    // Register split per warpgroup (producer / MMA / tables; converters;
    // epilogue), within the launch budget kThreads x kRegsLaunch.
    static constexpr uint32_t kRegsLaunch = NP == 64 ? 128 : 96;
    static constexpr uint32_t kRegsCtl = NP == 64 ? 72 : 56;
    static constexpr uint32_t kRegsConv = 72;
    static constexpr uint32_t kRegsHigh = NP == 64 ? 184 : 136;
    static_assert(128 * kRegsCtl + 32 * kNumConvWarps * kRegsConv + 32 * kNumEpiWarps * kRegsHigh <=
                      uint32_t(kThreads) * kRegsLaunch,
                  "register split");
    static constexpr int kNumRaw = NP == 64 ? 3 : 4;
    static constexpr int kNumOp = NP == 64 ? 3 : 4;
    static constexpr int kNumScl = 2;
    static constexpr int kSlotChunks = NP == 64 ? 4 : 8;     // chunks per tensor-memory slot
    static constexpr int kSlotCols = kSlotChunks * NP;
    static constexpr int kNumTm = int(kTmemCols) / kSlotCols; // 4, 2, 2
    static constexpr int kStagesPerSlot = kSlotChunks / 2;
    static constexpr int kSlotsPerSb = 8 / kSlotChunks;
    // raw stage: q4_K rows | int8 tokens (two 128-k swizzled boxes) | da | sa
    static constexpr int kRawW = kRowsW * 144;                // 18 KB
    static constexpr int kRawTokSub = NP * 128;
    static constexpr int kOffRawTok = kRawW;
    static constexpr int kOffRawDa = kOffRawTok + 2 * kRawTokSub;
    static constexpr int kOffRawSa = kOffRawDa + NP * 32;
    static constexpr int kRawStage = kOffRawSa + NP * 32;
    // operand stage (64 k): A = weights 128 x 128 B | B = tokens NP x 128 B
    static constexpr int kOpA = kRowsW * 128;
    static constexpr int kOpStage = kOpA + NP * 128;
    // table stage: da [8][NP] | dma [8][NP] | dmv [8][128] | d * 2^24 [128]
    static constexpr int kOffDa = 0, kOffDma = 8 * NP * 4, kOffDmv = 16 * NP * 4;
    static constexpr int kOffDsc = kOffDmv + kRowsW * 32;
    static constexpr int kSclStage = kOffDsc + kRowsW * 4;
    static constexpr int kOffRaw = 0;
    static constexpr int kOffOp = kOffRaw + kNumRaw * kRawStage;
    static constexpr int kOffScl = kOffOp + kNumOp * kOpStage;
    static constexpr int kOffBar = kOffScl + kNumScl * kSclStage;
    static constexpr int kNumBars = 2 * kNumRaw + 2 * kNumOp + 2 * kNumTm + 2 * kNumScl;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;   // tmem slot, abort flag
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;   // + alignment slack
    static constexpr int kPartBytes = kNumEpiWarps * 32 * T * 4;
    static_assert(kRawStage % 1024 == 0 && kOpStage % 1024 == 0 && kOffOp % 1024 == 0,
                  "swizzled tiles need 1024-byte alignment");
    static_assert(kOffRawTok % 1024 == 0 && kOpA % 1024 == 0, "swizzled sub-tiles");
    static_assert(kSclStage % 16 == 0, "table alignment");
    static_assert(kPartBytes <= kNumRaw * kRawStage, "partial tile reuses the raw ring");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kNumTm * kSlotCols <= int(kTmemCols), "tensor memory budget");
    static constexpr uint32_t kIdesc = idesc_f16_f32(kRowsW, NP);
};

template <int NP>
struct Bars {
    using C = Cfg<NP>;
    uint32_t base;
    __device__ uint32_t at(int i) const { return base + 8 * i; }
    __device__ uint32_t raw_full(int s) const { return at(s); }
    __device__ uint32_t raw_empty(int s) const { return at(C::kNumRaw + s); }
    __device__ uint32_t op_full(int s) const { return at(2 * C::kNumRaw + s); }
    __device__ uint32_t op_empty(int s) const { return at(2 * C::kNumRaw + C::kNumOp + s); }
    __device__ uint32_t tm_full(int s) const { return at(2 * C::kNumRaw + 2 * C::kNumOp + s); }
    __device__ uint32_t tm_empty(int s) const { return at(2 * C::kNumRaw + 2 * C::kNumOp + C::kNumTm + s); }
    __device__ uint32_t scl_full(int s) const {
        return at(2 * C::kNumRaw + 2 * C::kNumOp + 2 * C::kNumTm + s);
    }
    __device__ uint32_t scl_empty(int s) const {
        return at(2 * C::kNumRaw + 2 * C::kNumOp + 2 * C::kNumTm + C::kNumScl + s);
    }
};

struct Maps {
    CUtensorMap w, a, da, sa;
};

template <int T>
__device__ __forceinline__ void tmem_ld_row(uint32_t taddr, uint32_t (&r)[T]) {
    if constexpr (T == 8) {
        tmem_ld_32x32b_x8(taddr, r);
    } else if constexpr (T == 16) {
        tmem_ld_32x32b_x16(taddr, r);
    } else {
        tmem_ld_32x32b_x32(taddr, r);
    }
    tmem_wait_ld(r);
}

template <int NP>
__global__ void __launch_bounds__(Cfg<NP>::kThreads, 1)
gemm_tc_small_kernel(const __grid_constant__ Maps maps, float* __restrict__ C, int M, int N, int K,
                     int split, int* status, int inject_timeout) {
    using Cf = Cfg<NP>;
    constexpr int T = Cf::T;
    constexpr int kNumConvWarps = Cf::kNumConvWarps, kEpiWarp0 = Cf::kEpiWarp0;
    constexpr int TL = T < 16 ? T : 16;   // tensor-memory columns per load in the epilogue
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const Bars<NP> bars{sbase + Cf::kOffBar};
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cf::kOffMisc);
    const AbortFlag abort_flag{sbase + Cf::kOffMisc + 4};

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nsb = K / 256;
    const int tiles_tok = (M + NP - 1) / NP;
    const int rank = int(blockIdx.x % unsigned(split));
    const int tile = int(blockIdx.x / unsigned(split));
    const int n0 = (tile / tiles_tok) * kRowsW, m0 = (tile % tiles_tok) * NP;
    const int sb_lo = (nsb * rank) / split, sb_hi = (nsb * (rank + 1)) / split;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cf::kNumRaw; ++s) {
            mbar_init(bars.raw_full(s), 1);
            mbar_init(bars.raw_empty(s), kNumConvWarps + kNumSclWarps);
        }
        for (int s = 0; s < Cf::kNumOp; ++s) {
            mbar_init(bars.op_full(s), 4);   // one converter group
            mbar_init(bars.op_empty(s), 1);
        }
        for (int s = 0; s < Cf::kNumTm; ++s) {
            mbar_init(bars.tm_full(s), 1);
            mbar_init(bars.tm_empty(s), kNumEpiWarps);
        }
        for (int s = 0; s < Cf::kNumScl; ++s) {
            mbar_init(bars.scl_full(s), 4 + kNumSclWarps);   // the row-table converter warps + tables
            mbar_init(bars.scl_empty(s), kNumEpiWarps);
        }
        abort_flag.set(0u);
        fence_barrier_init();
        fence_proxy_async_smem();
        prefetch_tmap(&maps.w);
        prefetch_tmap(&maps.a);
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
    if (warp < kConvWarp0) setmaxnreg_dec<Cf::kRegsCtl>();
    else setmaxnreg_dec<Cf::kRegsConv>();
    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            Ring<Cf::kNumRaw> rr;
            int raw_issued[Cf::kNumRaw] = {};
            uint32_t raw_par[Cf::kNumRaw] = {};
            for (int sb = sb_lo; sb < sb_hi; ++sb) {
                if (!wait_bounded(bars.raw_empty(rr.slot), rr.phase ^ 1u, abort_flag, status)) break;
                const uint32_t raw = sbase + Cf::kOffRaw + rr.slot * Cf::kRawStage;
                if (!(sb == sb_lo && inject_timeout)) {   // test hook: withhold this arrival
                    const uint32_t fb = bars.raw_full(rr.slot);
                    mbar_arrive_expect_tx(fb, uint32_t(Cf::kRawStage));
                    tma_load_2d(raw, &maps.w, fb, sb * 144, n0);
                    tma_load_2d(raw + Cf::kOffRawTok, &maps.a, fb, sb * 256, m0);
                    tma_load_2d(raw + Cf::kOffRawTok + Cf::kRawTokSub, &maps.a, fb, sb * 256 + 128, m0);
                    tma_load_2d(raw + Cf::kOffRawDa, &maps.da, fb, sb * 8, m0);
                    tma_load_2d(raw + Cf::kOffRawSa, &maps.sa, fb, sb * 8, m0);
                    raw_issued[rr.slot] = 1;
                    raw_par[rr.slot] = rr.phase;
                }
                rr.next();
            }
            // Let every copy already issued land before the CTA can exit.
            for (int s = 0; s < Cf::kNumRaw; ++s)
                if (raw_issued[s]) wait_drain(bars.raw_full(s), raw_par[s], status);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            Ring<Cf::kNumOp> orr;
            Ring<Cf::kNumTm> tr;
            uint32_t last_bar = 0, last_par = 0;   // most recent commit, drained on exit
            int in_slot = 0;                       // operand stages already in the current slot
            for (int sb = sb_lo; sb < sb_hi; ++sb) {
                for (int q = 0; q < 4; ++q) {   // operand stage q: chunks 2q, 2q+1
                    const bool of = mbar_try_wait(bars.op_full(orr.slot), orr.phase);
                    const bool te = in_slot > 0 || mbar_try_wait(bars.tm_empty(tr.slot), tr.phase ^ 1u);
                    if (!of && !wait_bounded(bars.op_full(orr.slot), orr.phase, abort_flag, status))
                        goto mma_done;
                    if (!te && !wait_bounded(bars.tm_empty(tr.slot), tr.phase ^ 1u, abort_flag, status))
                        goto mma_done;
                    tc_fence_after();
                    const uint64_t dA = smem_desc_sw128(sbase + Cf::kOffOp + orr.slot * Cf::kOpStage);
                    const uint64_t dB = dA + uint64_t(Cf::kOpA >> 4);
                    const uint32_t d0 = tmem_base + uint32_t(tr.slot * Cf::kSlotCols + in_slot * 2 * NP);
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            const uint64_t koff = uint64_t((h * 64 + kk * 32) >> 4);   // 16-byte units
                            mma_f16(d0 + uint32_t(h * NP), dA + koff, dB + koff, Cf::kIdesc, uint32_t(kk));
                        }
                    mma_commit(bars.op_empty(orr.slot));
                    last_bar = bars.op_empty(orr.slot);
                    last_par = orr.phase;
                    orr.next();
                    if (++in_slot == Cf::kStagesPerSlot) {
                        mma_commit(bars.tm_full(tr.slot));
                        tr.next();
                        in_slot = 0;
                    }
                }
            }
        mma_done:
            if (last_bar) wait_drain(last_bar, last_par, status);
        }
    } else if (warp < kConvWarp0) {
        // ----------------------------------------------------- token tables
        const int ts = threadIdx.x - kSclWarp0 * 32;   // 0..63
        Ring<Cf::kNumRaw> rr;
        Ring<Cf::kNumScl> sr;
        for (int sb = sb_lo; sb < sb_hi; ++sb) {
            if (!wait_bounded(bars.raw_full(rr.slot), rr.phase, abort_flag, status)) break;
            if (!wait_bounded(bars.scl_empty(sr.slot), sr.phase ^ 1u, abort_flag, status)) break;
            {
                const uint32_t raw = sbase + Cf::kOffRaw + rr.slot * Cf::kRawStage;
                const uint32_t tab = sbase + Cf::kOffScl + sr.slot * Cf::kSclStage;
                for (int e = ts; e < NP * 8; e += 64) {   // token e >> 3, chunk e & 7
                    const int i = e >> 3, c = e & 7;
                    const float da = __uint_as_float(ld_shared_u32(raw + Cf::kOffRawDa + uint32_t(e) * 4u));
                    const int32_t sa = int32_t(ld_shared_u32(raw + Cf::kOffRawSa + uint32_t(e) * 4u));
                    st_shared_u32(tab + Cf::kOffDa + uint32_t(c * NP + i) * 4u, __float_as_uint(da));
                    st_shared_u32(tab + Cf::kOffDma + uint32_t(c * NP + i) * 4u, __float_as_uint(da * float(sa)));
                }
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bars.scl_full(sr.slot));
                mbar_arrive(bars.raw_empty(rr.slot));
            }
            sr.next();
            rr.next();
        }
    } else {
        // -------------------------------------------------------- converters
        // Groups of four warps take whole operand stages in turn (group cg the
        // stages q = cg mod kGroups of each super-block), so that kGroups stages
        // are converted at once; thread = weight row within its group.
        constexpr int kGroups = kNumConvWarps / 4;
        const int u = threadIdx.x - kConvWarp0 * 32;
        const int cg = u >> 7, t = u & 127;
        const int sw = t & 7;
        Ring<Cf::kNumRaw> rr;
        Ring<Cf::kNumScl> sr;
        int st0 = 0;   // operand-stage index of the super-block's first stage
        for (int sb = sb_lo; sb < sb_hi; ++sb, st0 += 4) {
            if (!wait_bounded(bars.raw_full(rr.slot), rr.phase, abort_flag, status)) goto conv_done;
            {
                const uint32_t raw = sbase + Cf::kOffRaw + rr.slot * Cf::kRawStage;
                const uint32_t rawW = raw + t * 144;
                const uint4 hdr = ld_shared_v4(rawW);
                const uint32_t scw_lo = sc_lo4(hdr.y), scw_hi = sc_hi4(hdr.y, hdr.w);
                if (cg == 0) {
                    // this row's scalars for the epilogue: d * 2^24 and dmv = -dmin * m per chunk
                    if (!wait_bounded(bars.scl_empty(sr.slot), sr.phase ^ 1u, abort_flag, status)) goto conv_done;
                    const uint32_t tab = sbase + Cf::kOffScl + sr.slot * Cf::kSclStage;
                    const float d = __half2float(__ushort_as_half(uint16_t(hdr.x & 0xFFFFu)));
                    const float dmin = __half2float(__ushort_as_half(uint16_t(hdr.x >> 16)));
                    const uint32_t mlo = m_lo4(hdr.z), mhi = m_hi4(hdr.z, hdr.w);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        st_shared_u32(tab + Cf::kOffDmv + uint32_t(c * kRowsW + t) * 4u,
                                      __float_as_uint(-(dmin * float((mlo >> (8 * c)) & 0xFFu))));
                        st_shared_u32(tab + Cf::kOffDmv + uint32_t((4 + c) * kRowsW + t) * 4u,
                                      __float_as_uint(-(dmin * float((mhi >> (8 * c)) & 0xFFu))));
                    }
                    st_shared_u32(tab + Cf::kOffDsc + uint32_t(t) * 4u, __float_as_uint(d * kSubnormalScale));
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars.scl_full(sr.slot));
                    sr.next();
                }
                for (int q = cg; q < 4; q += kGroups) {   // chunk pair q = chunks 2q (low nibbles), 2q+1 (high)
                    const int ost = (st0 + q) % Cf::kNumOp;
                    const uint32_t oph = uint32_t((st0 + q) / Cf::kNumOp) & 1u;
                    if (!wait_bounded(bars.op_empty(ost), oph ^ 1u, abort_flag, status)) goto conv_done;
                    const uint32_t scw = q < 2 ? scw_lo : scw_hi;
                    const uint32_t opA = sbase + Cf::kOffOp + ost * Cf::kOpStage;
                    const uint32_t opB = opA + Cf::kOpA;
                    // A: this weight row's chunks 2q + hh as fp16 subnormals sc * v
                    const uint32_t rowA = opA + t * 128;
                    uint4 wb[2];
#pragma unroll
                    for (int G = 0; G < 2; ++G) wb[G] = ld_shared_v4(rawW + 16 + 32 * q + 16 * G);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const uint32_t nsh = 4u * uint32_t(hh);   // nibble of each byte
                        const uint32_t sc = (scw >> (16u * uint32_t(q & 1) + 8u * uint32_t(hh))) & 0xFFu;
#pragma unroll
                        for (int G = 0; G < 2; ++G) {
                            const uint32_t ww[4] = {wb[G].x, wb[G].y, wb[G].z, wb[G].w};
                            uint32_t v[8];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                // two nibbles per 32-bit word, one per 16-bit half; times sc
                                // (<= 63 * 15 = 945, no carry into the upper half)
                                v[2 * e] = ((ww[e] >> nsh) & 0x000F000Fu) * sc;
                                v[2 * e + 1] = ((ww[e] >> (nsh + 8u)) & 0x000F000Fu) * sc;
                            }
                            const int g0 = 4 * hh + 2 * G;
                            st_shared_v4(rowA + ((g0 ^ sw) << 4), v[0], v[1], v[2], v[3]);
                            st_shared_v4(rowA + (((g0 + 1) ^ sw) << 4), v[4], v[5], v[6], v[7]);
                        }
                    }
                    // B: NP token rows x 64 k of int8 -> fp16, 16 k (one raw granule) per task
                    for (int task = t; task < NP * 4; task += 128) {
                        const int i = task >> 2, g = task & 3, si = i & 7;
                        const uint4 w = ld_shared_v4(raw + Cf::kOffRawTok + (q >> 1) * Cf::kRawTokSub + i * 128 +
                                                     ((((q & 1) * 4 + g) ^ si) << 4));
                        uint32_t p0, p1, p2, p3, p4, p5, p6, p7;
                        cvt_a4(w.x, p0, p1);
                        cvt_a4(w.y, p2, p3);
                        cvt_a4(w.z, p4, p5);
                        cvt_a4(w.w, p6, p7);
                        const uint32_t rowB = opB + i * 128;
                        st_shared_v4(rowB + (((2 * g) ^ si) << 4), p0, p1, p2, p3);
                        st_shared_v4(rowB + (((2 * g + 1) ^ si) << 4), p4, p5, p6, p7);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars.op_full(ost));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.raw_empty(rr.slot));
            rr.next();
        }
    conv_done:;
    }
    if (split > 1) {   // every thread of every CTA in the cluster takes both barriers
        cluster_sync_all();
        cluster_sync_all();
    }
    } else {
        setmaxnreg_inc<Cf::kRegsHigh>();
        // ---------------------------------------------------------- epilogue
        const int ew = warp - kEpiWarp0;          // 0..7
        const int quarter = warp & 3;             // tensor-memory lanes this warp may read
        const int colhalf = ew >> 2;
        const int row = quarter * 32 + lane;      // weight row within the tile
        const int col0 = colhalf * T;             // first token column
        const uint32_t tlane = uint32_t(quarter * 32) << 16;
        Ring<Cf::kNumScl> sr;
        Ring<Cf::kNumTm> tr;
        uint64_t acc[T / 2];
#pragma unroll
        for (int k = 0; k < T / 2; ++k) acc[k] = 0ull;
        for (int sb = sb_lo; sb < sb_hi; ++sb) {
            if (!wait_bounded(bars.scl_full(sr.slot), sr.phase, abort_flag, status)) goto epi_done;
            {
                const uint32_t tab = sbase + Cf::kOffScl + sr.slot * Cf::kSclStage;
                const uint32_t dsc = ld_shared_u32(tab + Cf::kOffDsc + uint32_t(row) * 4u);
                uint64_t asb[T / 2];
#pragma unroll
                for (int k = 0; k < T / 2; ++k) asb[k] = 0ull;
                // chunk c of the super-block: its S' columns read TL at a time from
                // tensor-memory address ta
                auto chunk = [&](uint32_t ta, int c) {
                    const uint32_t dmv = ld_shared_u32(tab + Cf::kOffDmv + uint32_t(c * kRowsW + row) * 4u);
                    const uint64_t dmv2 = pack2u(dmv, dmv);
                    const uint32_t da_row = tab + Cf::kOffDa + uint32_t(c * NP + col0) * 4u;
                    const uint32_t dm_row = tab + Cf::kOffDma + uint32_t(c * NP + col0) * 4u;
#pragma unroll
                    for (int p = 0; p < T / TL; ++p) {
                        uint32_t b[TL];
                        tmem_ld_row<TL>(ta + uint32_t(p * TL), b);
#pragma unroll
                        for (int kk = 0; kk < TL / 4; ++kk) {
                            const int k = p * (TL / 4) + kk;
                            const uint4 da4 = ld_shared_v4(da_row + 16u * k);
                            const uint4 dm4 = ld_shared_v4(dm_row + 16u * k);
                            asb[2 * k] = ffma2(pack2u(b[4 * kk], b[4 * kk + 1]), pack2u(da4.x, da4.y), asb[2 * k]);
                            asb[2 * k + 1] = ffma2(pack2u(b[4 * kk + 2], b[4 * kk + 3]), pack2u(da4.z, da4.w),
                                                   asb[2 * k + 1]);
                            acc[2 * k] = ffma2(pack2u(dm4.x, dm4.y), dmv2, acc[2 * k]);
                            acc[2 * k + 1] = ffma2(pack2u(dm4.z, dm4.w), dmv2, acc[2 * k + 1]);
                        }
                    }
                };
#pragma unroll
                for (int part = 0; part < Cf::kSlotsPerSb; ++part) {
                    if (!wait_bounded(bars.tm_full(tr.slot), tr.phase, abort_flag, status)) goto epi_done;
                    tc_fence_after();
                    const uint32_t ta = tmem_base + tlane + uint32_t(tr.slot * Cf::kSlotCols + col0);
#pragma unroll
                    for (int cc = 0; cc < Cf::kSlotChunks; ++cc) chunk(ta + uint32_t(cc * NP), part * Cf::kSlotChunks + cc);
                    // every chunk of the slot has been read: hand it back
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars.tm_empty(tr.slot));
                    tr.next();
                }
                const uint64_t dsc2 = pack2u(dsc, dsc);
#pragma unroll
                for (int k = 0; k < T / 2; ++k) acc[k] = ffma2(dsc2, asb[k], acc[k]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.scl_empty(sr.slot));
            sr.next();
        }
    epi_done:;
        const int gn = n0 + row;
        if (split == 1) {
#pragma unroll
            for (int k = 0; k < T / 2; ++k) {
                const int tok = m0 + col0 + 2 * k;
                if (gn < N) {
                    if (tok < M) C[int64_t(tok) * N + gn] = lo_f(acc[k]);
                    if (tok + 1 < M) C[int64_t(tok + 1) * N + gn] = hi_f(acc[k]);
                }
            }
        } else {
            // partial tile in this CTA's (now idle) raw ring: [epilogue thread][T] f32
            const int e = ew * 32 + lane;
            const uint32_t mine = sbase + Cf::kOffRaw + uint32_t(e * T) * 4u;
#pragma unroll
            for (int k = 0; k < T / 4; ++k)
                st_shared_v4(mine + 16u * k, uint32_t(acc[2 * k]), uint32_t(acc[2 * k] >> 32),
                             uint32_t(acc[2 * k + 1]), uint32_t(acc[2 * k + 1] >> 32));
            cluster_sync_all();
            if (ew % split == rank) {
                float v[T];
#pragma unroll
                for (int i = 0; i < T; ++i) v[i] = 0.0f;
                for (int r = 0; r < split; ++r) {   // rank order: deterministic
                    const uint32_t remote = map_shared_rank(mine, uint32_t(r));
#pragma unroll
                    for (int k = 0; k < T / 4; ++k) {
                        const float4 p = ld_dsmem_v4(remote + 16u * k);
                        v[4 * k] += p.x;
                        v[4 * k + 1] += p.y;
                        v[4 * k + 2] += p.z;
                        v[4 * k + 3] += p.w;
                    }
                }
                if (gn < N) {
#pragma unroll
                    for (int i = 0; i < T; ++i) {
                        const int tok = m0 + col0 + i;
                        if (tok < M) C[int64_t(tok) * N + gn] = v[i];
                    }
                }
            }
            cluster_sync_all();   // partials stay alive until every rank has read them
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

template <int NP>
cudaError_t launch_np(const mmq_q8_1_t& aq, const uint8_t* w, float* C, int64_t M, int64_t N, int64_t K,
                      int* status, int inject_timeout, cudaStream_t s) {
    using Cf = Cfg<NP>;
    Maps maps;
    const uint64_t nb = uint64_t(K / 32), nsb = uint64_t(K / 256);
    if (!encode_2d(&maps.w, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, nsb * 144, uint64_t(N), nsb * 144, 144,
                   kRowsW, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, aq.qs, uint64_t(K), uint64_t(M), uint64_t(K),
                   128, NP, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&maps.da, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, aq.da, nb, uint64_t(M), nb * 4, 8, NP,
                   CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&maps.sa, CU_TENSOR_MAP_DATA_TYPE_INT32, aq.sa, nb, uint64_t(M), nb * 4, 8, NP,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    int dev = 0, nsm = 0, optin = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (optin < Cf::kSmemBytes) return cudaErrorInvalidConfiguration;
    auto k = gemm_tc_small_kernel<NP>;
    // The register split (setmaxnreg) needs the block launched with exactly
    // kRegsLaunch registers per thread; refuse anything else.
    {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, k);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != int(Cf::kRegsLaunch)) return cudaErrorInvalidConfiguration;
    }
    const int64_t tiles = ((N + kRowsW - 1) / kRowsW) * ((M + NP - 1) / NP);
    // split K over a cluster so that most SMs get a CTA
    int split = 1;
    while (split < kMaxSplit && tiles * split * 2 <= nsm && split * 2 <= int64_t(nsb)) split *= 2;
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::kSmemBytes)))
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(tiles * split));
    cfg.blockDim = dim3(Cf::kThreads);
    cfg.dynamicSmemBytes = size_t(Cf::kSmemBytes);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(split);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, k, maps, C, int(M), int(N), int(K), split, status, inject_timeout);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

namespace mmq {

cudaError_t launch_gemm_tc_small(mmq_q8_1_t aq, const uint8_t* w, float* C, int64_t M, int64_t N, int64_t K,
                                 int* status, int inject_timeout, cudaStream_t s) {
    if (M <= 16) return launch_np<16>(aq, w, C, M, N, K, status, inject_timeout, s);
    if (M <= 32) return launch_np<32>(aq, w, C, M, N, K, status, inject_timeout, s);
    return launch_np<64>(aq, w, C, M, N, K, status, inject_timeout, s);
}

}  // namespace mmq
