// q4_K x q8_1 GEMM for few tokens (M <= 64): bound by streaming the q4_K
// weights from HBM once.  M <= 4 uses a dp4a dot-product kernel (below);
// 4 < M <= 64 the tensor-core kernel described here.
//
// Math as in the large-M kernels (web page "20 . r15 -- f32-accumulate mma
// probe (dead end) + rank-1 term2 rescale", section 2.1; fold from page
// "21 . r16 -- Narrow kernel gets the rank-1 fold", section 2.1): per 32-k
// chunk the exact integer dot S is rescaled,
//     acc += (da * dsv) * S + dma * dmv,   dsv = d*sc, dmv = -dmin*m, dma = da*sa.
//
// Design (weights are the big operand, so they go on the MMA's 16-row side
// and the tokens on its 8-column side):
//  - CTA = G groups of 4 warps, 64 weight rows (16 per warp of a group);
//    the CTA's super-blocks are dealt round-robin to the groups, each group
//    with its own TMA stage, so the super-blocks in flight are worked on in
//    parallel; the group partials are added in group order at the end.
//  - A cluster of S CTAs splits the 256-k super-blocks of K; ranks 1..S-1
//    push their partial sums into rank 0's shared memory, which adds them in
//    rank order: deterministic, and no global scratch.
//  - Once a stage has landed, its group converts the tokens' quants into
//    ready-made fp16 MMA fragments and a (da, dma = da*sa) table in shared
//    memory, once for the group's four warps.
//  - Per super-block one TMA stage brings the 64 raw q4_K rows (144 B each),
//    the tokens' int8 quants (two 128-byte-swizzled boxes) and their da / sa.
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

#include <atomic>
#include <cstdint>
#include <mutex>
#include <type_traits>

#include "mmq_internal.h"
#include "sm103_ptx.cuh"
#include "q8_round.cuh"

namespace {

using namespace mmq::ptx;

constexpr int kRows = 64;                 // weight rows per CTA (4 row-warps x 16)
constexpr int kMaxTok = 64;               // tokens per launch (M <= 64)
constexpr int kMaxSplit = 8;              // CTAs per cluster along K
constexpr int kW = kRows * 144;           // 9216 B raw q4_K rows
constexpr float kDsvScale = 16777216.0f;  // 2^24: nibbles are fp16 subnormals

struct SmallMaps {
    CUtensorMap w, a, da, sa;
};

// Shared-memory layout for NF token fragments (mp = 8*NF tokens) and G warp
// groups.  Group q owns D TMA stages and one work area:
//   stage  [0, kW) raw q4_K rows | [aoff, +2*mp*128) token quants as two
//          128-byte-swizzled boxes | [doff, +mp*32) da [mp][8] | [soff, +mp*32) sa
//   work   [0, NF*8*32*16) fp16 token fragments [f][c][lane] (4 x u32 each) |
//          [fbytes, +8*NF*4*16) token scales [c][f][j] {da_t0, da_t1, dma_t0, dma_t1}
// With D = 2 stages a group's next super-block is in flight while it
// computes the current one.  Then come the split-K landing area (partials
// pushed by cluster ranks 1..S-1: [rank-1][128 threads][NF] float4), the
// G*D stage barriers and the abort flag.
struct Layout {
    int aoff, doff, soff, stage, fbytes, work, stages_off, work_off, red_off, bar_off, total;
    __host__ __device__ static Layout make(int nf, int groups, int depth, int split) {
        Layout L;
        const int mp = 8 * nf;
        L.aoff = ((kW + 1023) / 1024) * 1024;
        L.doff = L.aoff + 2 * mp * 128;
        L.soff = L.doff + mp * 32;
        L.stage = ((L.soff + mp * 32 + 1023) / 1024) * 1024;
        L.fbytes = nf * 8 * 32 * 16;
        L.work = L.fbytes + 8 * nf * 4 * 16;
        L.stages_off = 0;
        L.work_off = groups * depth * L.stage;
        L.red_off = L.work_off + groups * L.work;
        L.bar_off = L.red_off + (split - 1) * 128 * nf * 16;
        L.total = L.bar_off + 8 * groups * depth + 16;
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

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_shared_rank(uint32_t saddr, uint32_t rank) {
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
    return d;
}
__device__ __forceinline__ void st_dsmem_v4(uint32_t addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y),
                 "f"(v.z), "f"(v.w)
                 : "memory");
}
__device__ __forceinline__ void group_sync(int group) {   // the 4 warps (128 threads) of a group
    asm volatile("bar.sync %0, 128;" ::"r"(group + 1) : "memory");
}

// q8_1 of one 32-element block held by 8 lanes (one float4 each; the
// group's lanes xor-reduce amax and the sum): the rounding of the prepass
// (reciprocal with an exactness check, IEEE division where a quotient lies
// too close to a half-integer), so the bits equal quantize-after-store.
__device__ __forceinline__ uint32_t quantize_group8(float4 v, float& d, int& sum) {
    using namespace mmq::q8;
    float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    d = __fdiv_rn(amax, 127.0f);
    int q0 = 0, q1 = 0, q2 = 0, q3 = 0;   // a zero scale gives zero quants
    if (d != 0.0f) {
        bool redo = d < 0x1p-126f;
        const float r = __frcp_rn(d);
        q0 = quant_fast(v.x, r, redo);
        q1 = quant_fast(v.y, r, redo);
        q2 = quant_fast(v.z, r, redo);
        q3 = quant_fast(v.w, r, redo);
        if (redo) {
            q0 = quant_exact(v.x, d);
            q1 = quant_exact(v.y, d);
            q2 = quant_exact(v.z, d);
            q3 = quant_exact(v.w, d);
        }
    }
    q0 = clamp127(q0);
    q1 = clamp127(q1);
    q2 = clamp127(q2);
    q3 = clamp127(q3);
    sum = q0 + q1 + q2 + q3;
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    sum += __shfl_xor_sync(0xffffffffu, sum, 4);
    return (uint32_t(q0) & 0xFFu) | ((uint32_t(q1) & 0xFFu) << 8) | ((uint32_t(q2) & 0xFFu) << 16) |
           ((uint32_t(q3) & 0xFFu) << 24);
}

// Epilogue modes of the few-token kernels (kOut):
//  kF32    C only;
//  kQ8     the result also as q8_1 (the next GEMM's activations, with the
//          bits of a prepass over C); C may be null;
//  kSwiGLU gate and up rows interleaved (row 2f = gate f, 2f + 1 = up f):
//          h = silu(g) * u = g / (1 + exp(-g)) * u in f32, quantized to q8_1
//          ([M][N/2]); C, if not null, receives h as f32 [M][N/2];
//  kDump   no rescale: the exact per-chunk dots S go to S int32 [M][N][K/32]
//          straight from the same unpack and dot-product code.
constexpr int kF32 = 0, kQ8 = 1, kSwiGLU = 2, kDump = 3;
__host__ __device__ constexpr bool quant_out(int mode) { return mode == kQ8 || mode == kSwiGLU; }

// kOut != kF32: rank 0's first group stages the CTA's finished [tokens][64
// rows] tile in shared memory and quantizes it: two q8_1 blocks of 32 output
// columns per token (kQ8), or one block of 32 SwiGLU features (kSwiGLU).
template <int NF, int G, int D, int kOut>
__global__ void __launch_bounds__(G * 128)
gemm_small_kernel(const __grid_constant__ SmallMaps maps, float* __restrict__ C, mmq_q8_1_t out,
                  int32_t* __restrict__ S, int M, int N, int K, int split, int tile0, int* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    constexpr int mp = NF * 8;
    const Layout L = Layout::make(NF, G, D, split);
    const uint32_t bar0 = sbase + L.bar_off;
    const AbortFlag abort_flag{sbase + uint32_t(L.bar_off + 8 * G * D)};
    griddep_launch_dependents();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = warp >> 2, gt = threadIdx.x & 127;   // group, thread within the group
    const int g = lane >> 2, j = lane & 3;
    const int rank = int(blockIdx.x % unsigned(split));
    const int n0 = (tile0 + int(blockIdx.x / unsigned(split))) * kRows;
    const int nsb = K / 256;
    const int sb_begin = (nsb * rank) / split, sb_end = (nsb * (rank + 1)) / split;
    const int nmine = sb_end - sb_begin;
    const uint32_t stage_tx = uint32_t(kW + 2 * mp * 128 + 2 * mp * 32);
    // stage `slot` of this group and its barrier
    auto stage_off = [&](int slot) { return L.stages_off + (grp * D + slot) * L.stage; };
    auto stage_bar = [&](int slot) { return bar0 + 8u * uint32_t(grp * D + slot); };
    uint8_t* work = smem + L.work_off + grp * L.work;

    if (threadIdx.x == 0) {
        for (int q = 0; q < G * D; ++q) mbar_init(bar0 + 8 * q, 1);
        abort_flag.set(0u);
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    __syncthreads();

    // group leader issues the TMA of super-block sb_begin + i (the group's
    // round (i - grp) / G) into stage round % D
    int last_issued[D];   // leader only: last round issued into each stage
#pragma unroll
    for (int q = 0; q < D; ++q) last_issued[q] = -1;
    // the weight copy (which sets the stage's expected bytes) and the token
    // copies of one round, issued separately so that the first rounds'
    // weights can stream before the programmatic-launch wait
    auto issue_w = [&](int i) {
        const int round = (i - grp) / G, slot = round % D;
        const uint32_t bar = stage_bar(slot), st_s = sbase + uint32_t(stage_off(slot));
        mbar_arrive_expect_tx(bar, stage_tx);
        tma_load_2d(st_s, &maps.w, bar, (sb_begin + i) * 144, n0);
        last_issued[slot] = round;
    };
    auto issue_a = [&](int i) {
        const int sb = sb_begin + i;
        const int slot = ((i - grp) / G) % D;
        const uint32_t bar = stage_bar(slot), st_s = sbase + uint32_t(stage_off(slot));
        tma_load_2d(st_s + L.aoff, &maps.a, bar, sb * 256, 0);
        tma_load_2d(st_s + L.aoff + mp * 128, &maps.a, bar, sb * 256 + 128, 0);
        tma_load_2d(st_s + L.doff, &maps.da, bar, sb * 8, 0);
        tma_load_2d(st_s + L.soff, &maps.sa, bar, sb * 8, 0);
    };
    auto issue = [&](int i) {
        issue_w(i);
        issue_a(i);
    };
    if (gt == 0)
        for (int q = 0; q < D && grp + q * G < nmine; ++q) issue_w(grp + q * G);
    griddep_wait();   // the previous kernel's outputs (tokens) are complete
    if (gt == 0)
        for (int q = 0; q < D && grp + q * G < nmine; ++q) issue_a(grp + q * G);

    uint64_t acc[NF][2];   // per token fragment: rows g (tokens 2j, 2j+1) and g + 8
#pragma unroll
    for (int f = 0; f < NF; ++f) acc[f][0] = acc[f][1] = 0ull;

    const int r0 = (warp & 3) * 16 + g;   // this thread's weight rows r0 and r0 + 8 (within the CTA)
    int pass = 0;
    for (int i = grp; i < nmine; i += G, ++pass) {
        const int slot = pass % D;
        const uint8_t* st = smem + stage_off(slot);
        // A timed-out wait raises the CTA abort flag; the exit is decided after
        // a group barrier, so the group's threads leave together.
        const bool landed =
            wait_bounded(stage_bar(slot), uint32_t((pass / D) & 1), abort_flag, status);
        if (landed) {
            // ---- tokens: fp16 fragments and (da, dma) once for the group
            for (int e = gt; e < NF * 8 * 32; e += 128) {
                const int f = e >> 8, c = (e >> 5) & 7, ln = e & 31;
                const int tok = 8 * f + (ln >> 2), jj = ln & 3;
                const uint32_t gran = uint32_t(((c & 3) * 2 + (jj >> 1)) ^ (tok & 7));
                const uint2 q = *reinterpret_cast<const uint2*>(st + L.aoff + (c >> 2) * mp * 128 +
                                                                tok * 128 + (gran << 4) + (jj & 1) * 8);
                uint4 fr;
                cvt_a4(q.x, fr.x, fr.y);
                cvt_a4(q.y, fr.z, fr.w);
                *reinterpret_cast<uint4*>(work + e * 16) = fr;
            }
            for (int e = gt; e < 8 * NF * 4; e += 128) {
                const int c = e / (NF * 4), f = (e >> 2) % NF, jj = e & 3;
                const int t0 = 8 * f + 2 * jj;
                const float* sda = reinterpret_cast<const float*>(st + L.doff);
                const int32_t* ssa = reinterpret_cast<const int32_t*>(st + L.soff);
                const float da0 = sda[t0 * 8 + c], da1 = sda[(t0 + 1) * 8 + c];
                *reinterpret_cast<float4*>(work + L.fbytes + e * 16) =
                    make_float4(da0, da1, da0 * float(ssa[t0 * 8 + c]), da1 * float(ssa[(t0 + 1) * 8 + c]));
            }
        }
        group_sync(grp);   // fragments and token scales are ready
        if (landed) {
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
                for (int pp = 0; pp < 4; ++pp) {
                    const uint2 v = *reinterpret_cast<const uint2*>(row + 16 + 32 * pp + 8 * j);
                    wq[h][pp][0] = v.x;
                    wq[h][pp][1] = v.y;
                }
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int pp = c >> 1, hsh = (c & 1) * 4;   // chunk 2p: low nibbles, 2p+1: high
                uint32_t a[2][4];
#pragma unroll
                for (int sstep = 0; sstep < 2; ++sstep) {
                    a[sstep][0] = (wq[0][pp][sstep] >> hsh) & 0x000F000Fu;        // row g, elements +0, +2
                    a[sstep][1] = (wq[1][pp][sstep] >> hsh) & 0x000F000Fu;        // row g + 8
                    a[sstep][2] = (wq[0][pp][sstep] >> (hsh + 8)) & 0x000F000Fu;  // row g, elements +1, +3
                    a[sstep][3] = (wq[1][pp][sstep] >> (hsh + 8)) & 0x000F000Fu;
                }
                const uint64_t dsv0 = pack2(dsv[0][c], dsv[0][c]), dsv1 = pack2(dsv[1][c], dsv[1][c]);
                const uint64_t dmv0 = pack2(dmv[0][c], dmv[0][c]), dmv1 = pack2(dmv[1][c], dmv[1][c]);
#pragma unroll
                for (int f = 0; f < NF; ++f) {
                    const uint4 fr = *reinterpret_cast<const uint4*>(work + ((f * 8 + c) * 32 + lane) * 16);
                    const float4 ts = *reinterpret_cast<const float4*>(work + L.fbytes + ((c * NF + f) * 4 + j) * 16);
                    float sc4[4] = {0.f, 0.f, 0.f, 0.f};
                    hmma(sc4, a[0][0], a[0][1], a[0][2], a[0][3], fr.x, fr.y);
                    hmma(sc4, a[1][0], a[1][1], a[1][2], a[1][3], fr.z, fr.w);
                    // C fragment: (row g, tokens 8f + 2j, +1) and (row g + 8, same tokens)
                    if constexpr (kOut == kDump) {
                        // the fragment holds S * 2^-24 exactly (|S| < 2^16)
                        const int64_t kb = int64_t(sb_begin + i) * 8 + c, nb = K / 32;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int row = n0 + r0 + 8 * h;
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int t = 8 * f + 2 * j + e;
                                if (row < N && t < M)
                                    S[(int64_t(t) * N + row) * nb + kb] = int32_t(sc4[2 * h + e] * kDsvScale);
                            }
                        }
                    } else {
                        const uint64_t da2 = pack2(ts.x, ts.y), dma2 = pack2(ts.z, ts.w);
                        const uint64_t s01 = pack2(sc4[0], sc4[1]), s23 = pack2(sc4[2], sc4[3]);
                        acc[f][0] = ffma2(dma2, dmv0, ffma2(fmul2(da2, dsv0), s01, acc[f][0]));
                        acc[f][1] = ffma2(dma2, dmv1, ffma2(fmul2(da2, dsv1), s23, acc[f][1]));
                    }
                }
            }
        }
        group_sync(grp);   // the group is done reading this stage
        if (abort_flag.raised()) break;
        if (gt == 0 && i + D * G < nmine) {
            fence_proxy_async_smem();
            issue(i + D * G);
        }
    }
    if (gt == 0) {
        // the group's last copies must land before its stage memory is reused or the CTA exits
#pragma unroll
        for (int q = 0; q < D; ++q)
            if (last_issued[q] >= 0)
                wait_drain(stage_bar(q), uint32_t((last_issued[q] / D) & 1), status);
    }
    __syncthreads();
    if constexpr (kOut == kDump) return;   // S is written; nothing to add up

    // ---- add the groups' partials (super-blocks were dealt round-robin)
    float4* part = reinterpret_cast<float4*>(smem + L.stages_off);   // [G][128][NF]
    if (grp > 0) {
#pragma unroll
        for (int f = 0; f < NF; ++f)
            part[(grp * 128 + gt) * NF + f] = make_float4(lo_f(acc[f][0]), hi_f(acc[f][0]), lo_f(acc[f][1]), hi_f(acc[f][1]));
    }
    __syncthreads();
    if (grp == 0) {
        for (int q = 1; q < G; ++q)
#pragma unroll
            for (int f = 0; f < NF; ++f) {
                const float4 o = part[(q * 128 + gt) * NF + f];
                acc[f][0] = pack2(lo_f(acc[f][0]) + o.x, hi_f(acc[f][0]) + o.y);
                acc[f][1] = pack2(lo_f(acc[f][1]) + o.z, hi_f(acc[f][1]) + o.w);
            }
        // ---- split-K: ranks 1..S-1 push their partials into rank 0's landing area
        if (split > 1 && rank > 0) {
            const uint32_t dst = map_shared_rank(sbase + L.red_off, 0u) +
                                 uint32_t(((rank - 1) * 128 + gt) * NF) * 16u;
#pragma unroll
            for (int f = 0; f < NF; ++f)
                st_dsmem_v4(dst + f * 16, make_float4(lo_f(acc[f][0]), hi_f(acc[f][0]), lo_f(acc[f][1]), hi_f(acc[f][1])));
        }
    }
    if (split > 1) cluster_sync();   // pushed partials are visible in rank 0
    if (rank == 0 && grp == 0) {
        const float4* land = reinterpret_cast<const float4*>(smem + L.red_off);
        for (int r = 1; r < split; ++r)
#pragma unroll
            for (int f = 0; f < NF; ++f) {
                const float4 o = land[((r - 1) * 128 + gt) * NF + f];
                acc[f][0] = pack2(lo_f(acc[f][0]) + o.x, hi_f(acc[f][0]) + o.y);
                acc[f][1] = pack2(lo_f(acc[f][1]) + o.z, hi_f(acc[f][1]) + o.w);
            }
        if (kOut == kF32 || (kOut == kQ8 && C)) {
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
        if constexpr (quant_out(kOut)) {
            // the tile [8 NF tokens][64 rows] after the groups' partials (stage memory is idle)
            float* tile = reinterpret_cast<float*>(smem + L.stages_off + G * 128 * NF * 16);
#pragma unroll
            for (int f = 0; f < NF; ++f)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    tile[(8 * f + 2 * j) * kRows + r0 + 8 * h] = lo_f(acc[f][h]);
                    tile[(8 * f + 2 * j + 1) * kRows + r0 + 8 * h] = hi_f(acc[f][h]);
                }
            group_sync(0);
            const int part8 = gt & 7;   // 8 lanes per output block, 4 values each
            constexpr int kBlocksPerToken = kOut == kSwiGLU ? 1 : 2;
            for (int b0 = 0; b0 < M * kBlocksPerToken; b0 += 16) {   // 16 groups of 8 lanes
                const int b = b0 + (gt >> 3);
                const int t = b / kBlocksPerToken, half = b % kBlocksPerToken;
                const bool ok = b < M * kBlocksPerToken;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (ok) {
                    if constexpr (kOut == kSwiGLU) {
                        float hv[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float g = tile[t * kRows + 2 * (4 * part8 + i)];
                            const float u = tile[t * kRows + 2 * (4 * part8 + i) + 1];
                            hv[i] = __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
                        }
                        v = make_float4(hv[0], hv[1], hv[2], hv[3]);
                    } else {
                        v = *reinterpret_cast<const float4*>(&tile[t * kRows + 32 * half + 4 * part8]);
                    }
                }
                float d;
                int sum;
                const uint32_t word = quantize_group8(v, d, sum);   // all 32 lanes take part
                const int width = kOut == kSwiGLU ? N / 2 : N;       // output columns
                const int col0 = (kOut == kSwiGLU ? n0 / 2 : n0) + 32 * half;
                if (ok && col0 < width) {
                    *reinterpret_cast<uint32_t*>(out.qs + int64_t(t) * width + col0 + 4 * part8) = word;
                    if (kOut == kSwiGLU && C)
                        *reinterpret_cast<float4*>(C + int64_t(t) * width + col0 + 4 * part8) = v;
                    if (part8 == 0) {
                        out.da[int64_t(t) * (width / 32) + col0 / 32] = d;
                        out.sa[int64_t(t) * (width / 32) + col0 / 32] = sum;
                    }
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// M <= 4 tokens: a plain streaming dot product, one warp per few weight rows.
// Lane l takes each row's chunk pairs l, l+32, ...: 32 nibble bytes (chunk 2p
// in the low nibbles, 2p+1 in the high ones, both in natural k order) plus
// the super-block header.  S comes from dp4a (unsigned nibble bytes x signed
// int8 quants, exact int32), then the per-chunk rescale with the fold; the
// lanes' partial sums are added by a fixed xor-shuffle tree.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int dp4a_us(uint32_t a_u8, uint32_t b_s8, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a_u8), "r"(b_s8), "r"(c));
    return d;
}


__device__ __forceinline__ void st_dsmem_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// One warp per R consecutive weight rows: each activation load (the token's
// 64 quants of a chunk pair, its two da and sa) serves R rows, so the
// activation traffic through L1 is 1/R of one row per warp.  R rows x the
// lane's pair of weights (48 bytes each) are all requested before any is
// used.  K is split over KS warps of the CTA (pair blocks of 32 dealt
// round-robin), so that a long row takes fewer dependent load rounds per
// warp and more warps have loads in flight; the KS partial sums are added
// in slice order through shared memory.
//
// With a q8_1 output (kQ8, kSwiGLU) the kernel runs in clusters of CTAs
// covering one output block's rows (32, or 64 interleaved rows for
// SwiGLU); each row's sum goes into rank 0's shared memory and rank 0
// quantizes the block.
template <int MT, int R, int KS, int kOut>
__global__ void __launch_bounds__(128)
gemv_dp4a_kernel(mmq_q8_1_t aq, const uint8_t* __restrict__ w, float* __restrict__ C, mmq_q8_1_t out,
                 int32_t* __restrict__ S, int M, int N, int K) {
    constexpr int kGroups = 4 / KS;                        // row groups (of R rows) per CTA
    constexpr int kBlockRows = kOut == kSwiGLU ? 64 : 32;  // rows behind one q8_1 output block
    constexpr int kCluster = kBlockRows / (kGroups * R);   // CTAs per output block
    __shared__ __align__(16) float red[quant_out(kOut) ? MT : 1][kBlockRows];   // rank 0: the cluster's rows [t][row]
    __shared__ float part[KS > 1 ? 4 : 1][MT][R];          // KS > 1: each warp's partial sums
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slice = warp % KS, grp = warp / KS;
    const int row0 = (blockIdx.x * kGroups + grp) * R;   // this warp's rows row0 .. row0 + R - 1
    griddep_launch_dependents();
    if (KS == 1 && !quant_out(kOut) && row0 >= N) return;   // (with q8_1 output every row exists)
    if (quant_out(kOut)) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");   // this CTA has started
    const int nsb = K / 256, npairs = K / 64, nb = K / 32;
    float acc[MT][R];
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int r = 0; r < R; ++r) acc[t][r] = 0.0f;
    for (int base = 32 * slice; base < npairs; base += 32 * KS) {
        const int pr = base + lane;
        const int p = pr & 3;
        uint4 hdr[R], q0[R], q1[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (pr < npairs && row0 + r < N) {
                const uint8_t* blk = w + (int64_t(row0 + r) * nsb + (pr >> 2)) * 144;
                hdr[r] = __ldg(reinterpret_cast<const uint4*>(blk));
                q0[r] = __ldcs(reinterpret_cast<const uint4*>(blk + 16 + 32 * p));
                q1[r] = __ldcs(reinterpret_cast<const uint4*>(blk + 32 + 32 * p));
            } else {
                hdr[r] = q0[r] = q1[r] = make_uint4(0u, 0u, 0u, 0u);   // contributes 0
            }
        }
        // weights stream in while the previous kernel (programmatic dependent
        // launch) finishes; activations and C only after it has
        if (base == 32 * slice) griddep_wait();
        if (pr >= npairs) continue;
        float dsv[R][2], dmv[R][2];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float d = __half2float(__ushort_as_half(uint16_t(hdr[r].x & 0xFFFFu)));
            const float dmin = __half2float(__ushort_as_half(uint16_t(hdr[r].x >> 16)));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int c = 2 * p + h;   // sub-block within the super-block
                uint32_t sc, m;
                if (c < 4) {
                    sc = (hdr[r].y >> (8 * c)) & 63u;
                    m = (hdr[r].z >> (8 * c)) & 63u;
                } else {
                    const int bsh = 8 * (c - 4);
                    sc = ((hdr[r].w >> bsh) & 15u) | (((hdr[r].y >> (bsh + 6)) & 3u) << 4);
                    m = ((hdr[r].w >> (bsh + 4)) & 15u) | (((hdr[r].z >> (bsh + 6)) & 3u) << 4);
                }
                dsv[r][h] = d * float(sc);
                dmv[r][h] = -(dmin * float(m));
            }
        }
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            if (t < M) {
                const int8_t* qt = aq.qs + int64_t(t) * K + 64 * pr;
                const uint4 a0 = __ldg(reinterpret_cast<const uint4*>(qt));
                const uint4 a1 = __ldg(reinterpret_cast<const uint4*>(qt + 16));
                const uint4 a2 = __ldg(reinterpret_cast<const uint4*>(qt + 32));
                const uint4 a3 = __ldg(reinterpret_cast<const uint4*>(qt + 48));
                const float2 da = __ldg(reinterpret_cast<const float2*>(aq.da + int64_t(t) * nb + 2 * pr));
                const int2 sa = __ldg(reinterpret_cast<const int2*>(aq.sa + int64_t(t) * nb + 2 * pr));
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    // chunk 2p in the low nibbles, 2p + 1 in the high ones, natural k order
                    const uint32_t wv[8] = {q0[r].x, q0[r].y, q0[r].z, q0[r].w, q1[r].x, q1[r].y, q1[r].z, q1[r].w};
                    const uint32_t av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                    const uint32_t bv[8] = {a2.x, a2.y, a2.z, a2.w, a3.x, a3.y, a3.z, a3.w};
                    int s0 = 0, s1 = 0;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        s0 = dp4a_us(wv[e] & 0x0F0F0F0Fu, av[e], s0);
                        s1 = dp4a_us((wv[e] >> 4) & 0x0F0F0F0Fu, bv[e], s1);
                    }
                    if constexpr (kOut == kDump) {   // the exact dots of chunks 2pr, 2pr + 1
                        if (row0 + r < N) {
                            int32_t* sp = S + (int64_t(t) * N + row0 + r) * nb + 2 * pr;
                            sp[0] = s0;
                            sp[1] = s1;
                        }
                        continue;
                    }
                    float a = acc[t][r];
                    a = fmaf(da.x * dsv[r][0], float(s0), a);
                    a = fmaf(da.x * float(sa.x), dmv[r][0], a);   // rank-1 fold: dma = da*sa
                    a = fmaf(da.y * dsv[r][1], float(s1), a);
                    a = fmaf(da.y * float(sa.y), dmv[r][1], a);
                    acc[t][r] = a;
                }
            }
        }
    }
    if constexpr (kOut == kDump) return;   // S is written; nothing to add up
#pragma unroll
    for (int t = 0; t < MT; ++t) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float a = acc[t][r];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
            acc[t][r] = a;
        }
    }
    if constexpr (KS > 1) {   // add the K slices' partials in slice order (slice 0 keeps the sum)
        if (lane == 0) {
#pragma unroll
            for (int t = 0; t < MT; ++t)
#pragma unroll
                for (int r = 0; r < R; ++r) part[warp][t][r] = acc[t][r];
        }
        __syncthreads();
        if (slice == 0) {
#pragma unroll
            for (int t = 0; t < MT; ++t)
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    float a = part[warp][t][r];
#pragma unroll
                    for (int q = 1; q < KS; ++q) a += part[warp + q][t][r];
                    acc[t][r] = a;
                }
        }
    }
    if (kOut != kSwiGLU && slice == 0 && lane == 0 && C) {
#pragma unroll
        for (int t = 0; t < MT; ++t)
#pragma unroll
            for (int r = 0; r < R; ++r)
                if (t < M && row0 + r < N) C[int64_t(t) * N + row0 + r] = acc[t][r];
    }
    if constexpr (quant_out(kOut)) {
        const uint32_t rank = cluster_ctarank();
        asm volatile("barrier.cluster.wait.aligned;" ::: "memory");   // every CTA of the cluster has started
        if (slice == 0 && lane == 0) {
#pragma unroll
            for (int t = 0; t < MT; ++t)
#pragma unroll
                for (int r = 0; r < R; ++r)
                    if (t < M)
                        st_dsmem_f32(map_shared_rank(smem_u32(&red[t][(rank * kGroups + grp) * R + r]), 0),
                                     acc[t][r]);
        }
        cluster_sync();   // the block's rows are in rank 0
        if (rank == 0 && warp == 0) {
            const int t = lane >> 3, part = lane & 7;   // 8 lanes per token, 4 outputs per lane
            const int tt = t < MT ? t : 0;
            const int width = kOut == kSwiGLU ? N / 2 : N;   // output columns
            const int blk = int(blockIdx.x / kCluster);     // output columns 32 blk .. 32 blk + 31
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t < M) {
                if constexpr (kOut == kSwiGLU) {
                    float h[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float g = red[tt][2 * (part * 4 + i)], u = red[tt][2 * (part * 4 + i) + 1];
                        h[i] = __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
                    }
                    v = make_float4(h[0], h[1], h[2], h[3]);
                    if (C) *reinterpret_cast<float4*>(C + int64_t(t) * width + 32 * blk + part * 4) = v;
                } else {
                    v = *reinterpret_cast<const float4*>(&red[tt][part * 4]);
                }
            }
            float d;
            int sum;
            const uint32_t word = quantize_group8(v, d, sum);
            if (t < M) {
                *reinterpret_cast<uint32_t*>(out.qs + int64_t(t) * width + 32 * blk + part * 4) = word;
                if (part == 0) {
                    out.da[int64_t(t) * (width / 32) + blk] = d;
                    out.sa[int64_t(t) * (width / 32) + blk] = sum;
                }
            }
        }
    }
}

// Rows per warp of the dot-product kernel.  Measured on the 7B decode chain
// (224 dependent GEMMs, programmatic launch): R = 4 beats 1, 2 and (at one
// token) 8 for 1, 2 and 4 tokens.
constexpr int kGemvRows = 4;

template <int MT, int KS, int kOut>
cudaError_t launch_gemv_ks(mmq_q8_1_t aq, const uint8_t* w, float* C, mmq_q8_1_t out, int32_t* S, int64_t M,
                           int64_t N, int64_t K, cudaStream_t s) {
    constexpr int R = kGemvRows, rows = 4 / KS * R;   // rows per CTA
    constexpr int cluster = (kOut == kSwiGLU ? 64 : 32) / rows;
    static_assert(!quant_out(kOut) || (cluster >= 1 && cluster <= 8), "portable cluster size");
    cudaLaunchAttribute attr[2];
    const unsigned grid = unsigned((N + rows - 1) / rows);
    cudaLaunchConfig_t cfg = mmq::launch_config(dim3(grid), dim3(128), 0, s, attr);
    if (quant_out(kOut)) {   // grid = N / rows is a multiple of the cluster (N % 32 or N % 64 == 0)
        attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
        attr[cfg.numAttrs].val.clusterDim.x = cluster;
        attr[cfg.numAttrs].val.clusterDim.y = 1;
        attr[cfg.numAttrs].val.clusterDim.z = 1;
        ++cfg.numAttrs;
    }
    return cudaLaunchKernelEx(&cfg, gemv_dp4a_kernel<MT, R, KS, kOut>, aq, w, C, out, S, int(M), int(N), int(K));
}

// CTAs of one kernel instance that fit on a device at once (register-bound),
// found once per instance and device.
constexpr int kMaxDevices = 64;
template <int MT, int KS, int kOut>
int64_t gemv_resident_ctas() {
    static std::atomic<int64_t> cached[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        dev = -1;
    }
    int64_t v = dev >= 0 ? cached[dev].load(std::memory_order_relaxed) : 0;
    if (v == 0) {
        int nsm = 0, per_sm = 0;
        if (dev < 0 || cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            nsm = 1;
        }
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemv_dp4a_kernel<MT, kGemvRows, KS, kOut>, 128,
                                                          0) != cudaSuccess || per_sm < 1) {
            cudaGetLastError();
            per_sm = 1;
        }
        v = int64_t(per_sm) * (nsm > 0 ? nsm : 1);
        if (dev >= 0) cached[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

// Test hook: a K split forced for this host thread (0: the cost model's).
thread_local int t_force_ks = 0;

// The K split (KS warps per row group) with the lowest modelled cost:
// waves of CTAs x (dependent load rounds per warp + 1/2), the half standing
// for a wave's own start-up and drain.  More warps per row take fewer rounds
// each but make more CTAs, and a wave that is only just started costs almost
// a whole one.  Fitted to one and four tokens on the 7B shapes (4096 ->
// 4096, 11008, 12288, 22016 and 11008 -> 4096), where it picks the fastest
// of 1, 2 and 4 every time.  The SwiGLU epilogue takes KS <= 2 (its 64-row
// blocks would otherwise need clusters of 16).
template <int MT, int kOut>
cudaError_t launch_gemv(mmq_q8_1_t aq, const uint8_t* w, float* C, mmq_q8_1_t out, int32_t* S, int64_t M,
                        int64_t N, int64_t K, cudaStream_t s) {
    int ks = t_force_ks;
    if (ks == 0) {
        const int64_t npairs = K / 64;
        auto cost2 = [&](int k, int64_t resident) {   // twice the modelled cost
            const int64_t rows = 16 / k;                 // (4 / k) row groups x kGemvRows rows per CTA
            const int64_t ctas = (N + rows - 1) / rows;
            const int64_t waves = (ctas + resident - 1) / resident;
            const int64_t rounds = (npairs + 32 * k - 1) / (32 * k);
            return waves * (2 * rounds + 1);
        };
        static_assert(kGemvRows == 4, "the cost model counts 4 rows per warp");
        const int64_t c1 = cost2(1, gemv_resident_ctas<MT, 1, kOut>());
        const int64_t c2 = cost2(2, gemv_resident_ctas<MT, 2, kOut>());
        int64_t c4 = INT64_MAX;
        if constexpr (kOut != kSwiGLU) c4 = cost2(4, gemv_resident_ctas<MT, 4, kOut>());
        ks = (c1 <= c2 && c1 <= c4) ? 1 : (c4 < c2 ? 4 : 2);
    }
    if (ks == 1) return launch_gemv_ks<MT, 1, kOut>(aq, w, C, out, S, M, N, K, s);
    if (ks == 2) return launch_gemv_ks<MT, 2, kOut>(aq, w, C, out, S, M, N, K, s);
    if constexpr (kOut != kSwiGLU) {
        if (ks == 4) return launch_gemv_ks<MT, 4, kOut>(aq, w, C, out, S, M, N, K, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

namespace mmq {

cudaError_t launch_gemv_q8_1(mmq_q8_1_t aq, const uint8_t* w, float* C, mmq_q8_1_t out, int64_t M, int64_t N,
                             int64_t K, cudaStream_t s) {
    if (M < 1 || M > 4 || N % 32 != 0) return cudaErrorInvalidValue;
    switch (M) {
        case 1: return launch_gemv<1, kQ8>(aq, w, C, out, nullptr, M, N, K, s);
        case 2: return launch_gemv<2, kQ8>(aq, w, C, out, nullptr, M, N, K, s);
        default: return launch_gemv<4, kQ8>(aq, w, C, out, nullptr, M, N, K, s);
    }
}

cudaError_t launch_gemv_swiglu_q8_1(mmq_q8_1_t aq, const uint8_t* w_gu, float* hf, mmq_q8_1_t out, int64_t M,
                                    int64_t F, int64_t K, cudaStream_t s) {
    if (M < 1 || M > 4 || F % 32 != 0) return cudaErrorInvalidValue;
    switch (M) {
        case 1: return launch_gemv<1, kSwiGLU>(aq, w_gu, hf, out, nullptr, M, 2 * F, K, s);
        case 2: return launch_gemv<2, kSwiGLU>(aq, w_gu, hf, out, nullptr, M, 2 * F, K, s);
        default: return launch_gemv<4, kSwiGLU>(aq, w_gu, hf, out, nullptr, M, 2 * F, K, s);
    }
}

}  // namespace mmq

namespace {

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

// How a call's row tiles are launched: `tiles` of them in clusters of
// `split` CTAs along K, and, when those fill whole rounds of resident CTAs
// with a partial round left over, that remainder (`tail` tiles from tile
// `tiles`) as a second launch with its own larger K split, so that it takes
// a fraction of a round instead of a whole one.
struct SmallPlan {
    int64_t tiles = 0, tail = 0;
    int split = 1, tail_split = 1;
    int smem = 0, tail_smem = 0;
};

template <int NF, int G, int D, int kOut>
cudaError_t plan_nf(int64_t N, int64_t K, SmallPlan& P) {
    int dev = 0, nsm = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return cudaGetLastError();
    const int64_t row_tiles = (N + kRows - 1) / kRows;
    const int nsb = int(K / 256);
    auto fits = [&](int sp) { return Layout::make(NF, G, D, sp).total + 1024 <= optin; };
    // Split K over a cluster so that every SM gets a CTA: about two per SM
    // for one token fragment, about one for more (each CTA converts the
    // tokens of its super-blocks, so more CTAs per weight row cost more
    // conversion; measured on 4096 x 4096: M = 8 fastest at two per SM,
    // M = 16..64 at one), within the shared-memory budget of the landing area.
    const int64_t per_sm = NF == 1 ? 2 : 1;
    int split = 1;
    while (split < kMaxSplit && row_tiles * split * 2 <= per_sm * int64_t(nsm) && split * 2 <= nsb && fits(split * 2))
        split *= 2;
    P = SmallPlan{};
    P.tiles = row_tiles;
    P.split = split;
    P.smem = Layout::make(NF, G, D, split).total + 1024;   // + alignment slack
    if (P.smem > optin) return cudaErrorInvalidConfiguration;
    if (split == 1) {
        int per = 0;
        auto k = gemm_small_kernel<NF, G, D, kOut>;
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, P.smem) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, k, G * 128, size_t(P.smem)) != cudaSuccess)
            return cudaGetLastError();
        const int64_t resident = int64_t(per > 0 ? per : 1) * nsm;
        const int64_t tail = row_tiles % resident;
        if (row_tiles > resident && tail > 0) {
            int ts = 1;
            while (ts < kMaxSplit && tail * ts * 2 <= resident && ts * 2 <= nsb && fits(ts * 2)) ts *= 2;
            if (ts > 1) {
                P.tiles = row_tiles - tail;
                P.tail = tail;
                P.tail_split = ts;
                P.tail_smem = Layout::make(NF, G, D, ts).total + 1024;
            }
        }
    }
    return cudaSuccess;
}

template <int NF, int G, int D, int kOut>
cudaError_t launch_part(const SmallMaps& maps, float* C, mmq_q8_1_t out, int32_t* S, int64_t M, int64_t N,
                        int64_t K, int* status, cudaStream_t s, int64_t tile0, int64_t tiles, int split, int smem) {
    // the quantizing epilogue stages its tile behind the groups' partials in stage memory
    if (quant_out(kOut) && G * 128 * NF * 16 + 8 * NF * kRows * 4 > Layout::make(NF, G, D, split).work_off)
        return cudaErrorInvalidConfiguration;
    auto k = gemm_small_kernel<NF, G, D, kOut>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = mmq::launch_config(dim3(unsigned(tiles * split)), dim3(G * 128), size_t(smem), s, attr);
    attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
    attr[cfg.numAttrs].val.clusterDim.x = unsigned(split);
    attr[cfg.numAttrs].val.clusterDim.y = 1;
    attr[cfg.numAttrs].val.clusterDim.z = 1;
    cfg.numAttrs += 1;
    return cudaLaunchKernelEx(&cfg, k, maps, C, out, S, int(M), int(N), int(K), split, int(tile0), status);
}

template <int NF, int G, int D, int kOut>
cudaError_t launch_nf(const SmallMaps& maps, float* C, mmq_q8_1_t out, int32_t* S, int64_t M, int64_t N,
                      int64_t K, int* status, cudaStream_t s) {
    SmallPlan P;
    cudaError_t e = plan_nf<NF, G, D, kOut>(N, K, P);
    if (e != cudaSuccess) return e;
    e = launch_part<NF, G, D, kOut>(maps, C, out, S, M, N, K, status, s, 0, P.tiles, P.split, P.smem);
    if (e != cudaSuccess || P.tail == 0) return e;
    return launch_part<NF, G, D, kOut>(maps, C, out, S, M, N, K, status, s, P.tiles, P.tail, P.tail_split,
                                       P.tail_smem);
}

// The kernel instance per number of 8-token fragments: NF, warp groups G,
// TMA stages per group D.
template <typename Fn>
cudaError_t dispatch_nf(int nf, Fn&& fn) {
    using std::integral_constant;
    switch (nf) {
        case 1: return fn(integral_constant<int, 1>{}, integral_constant<int, 4>{}, integral_constant<int, 1>{});
        case 2: return fn(integral_constant<int, 2>{}, integral_constant<int, 4>{}, integral_constant<int, 2>{});
        case 3: return fn(integral_constant<int, 3>{}, integral_constant<int, 4>{}, integral_constant<int, 2>{});
        case 4: return fn(integral_constant<int, 4>{}, integral_constant<int, 4>{}, integral_constant<int, 1>{});
        case 5: return fn(integral_constant<int, 5>{}, integral_constant<int, 2>{}, integral_constant<int, 2>{});
        case 6: return fn(integral_constant<int, 6>{}, integral_constant<int, 2>{}, integral_constant<int, 2>{});
        case 7: return fn(integral_constant<int, 7>{}, integral_constant<int, 2>{}, integral_constant<int, 2>{});
        default: return fn(integral_constant<int, 8>{}, integral_constant<int, 2>{}, integral_constant<int, 2>{});
    }
}

template <int kOut>
cudaError_t launch_nf_any(int nf, const SmallMaps& maps, float* C, mmq_q8_1_t out, int32_t* S, int64_t M,
                          int64_t N, int64_t K, int* status, cudaStream_t s) {
    return dispatch_nf(nf, [&](auto F, auto G, auto D) {
        return launch_nf<decltype(F)::value, decltype(G)::value, decltype(D)::value, kOut>(maps, C, out, S, M, N, K,
                                                                                           status, s);
    });
}

}  // namespace

namespace mmq {

cudaError_t launch_gemm_small_m(mmq_q8_1_t aq, const uint8_t* w, float* C, int64_t M, int64_t N,
                                int64_t K, int* status, cudaStream_t s, mmq_q8_1_t out, int mode, int32_t* S) {
    if (M > kMaxTok || mode < kF32 || mode > kDump) return cudaErrorInvalidValue;
    if (quant_out(mode) && (out.qs == nullptr || N % (mode == kSwiGLU ? 64 : 32) != 0)) return cudaErrorInvalidValue;
    if ((mode == kDump) != (S != nullptr)) return cudaErrorInvalidValue;
    const mmq_q8_1_t none = {nullptr, nullptr, nullptr};
    if (M <= 4) {   // a few tokens: streaming dot products on dp4a
        if (mode == kQ8) return launch_gemv_q8_1(aq, w, C, out, M, N, K, s);
        if (mode == kSwiGLU) return launch_gemv_swiglu_q8_1(aq, w, C, out, M, N / 2, K, s);
        if (mode == kDump) {
            switch (M) {
                case 1: return launch_gemv<1, kDump>(aq, w, nullptr, none, S, M, N, K, s);
                case 2: return launch_gemv<2, kDump>(aq, w, nullptr, none, S, M, N, K, s);
                default: return launch_gemv<4, kDump>(aq, w, nullptr, none, S, M, N, K, s);
            }
        }
        switch (M) {
            case 1: return launch_gemv<1, kF32>(aq, w, C, none, nullptr, M, N, K, s);
            case 2: return launch_gemv<2, kF32>(aq, w, C, none, nullptr, M, N, K, s);
            default: return launch_gemv<4, kF32>(aq, w, C, none, nullptr, M, N, K, s);
        }
    }
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
    if (mode == kQ8) return launch_nf_any<kQ8>(nf, maps, C, out, nullptr, M, N, K, status, s);
    if (mode == kSwiGLU) return launch_nf_any<kSwiGLU>(nf, maps, C, out, nullptr, M, N, K, status, s);
    if (mode == kDump) return launch_nf_any<kDump>(nf, maps, nullptr, none, S, M, N, K, status, s);
    return launch_nf_any<kF32>(nf, maps, C, out, nullptr, M, N, K, status, s);
}

int small_m_launch_count(int64_t M, int64_t N, int64_t K) {
    if (M <= 4) return 1;
    SmallPlan P;
    const cudaError_t e = dispatch_nf(int((M + 7) / 8), [&](auto F, auto G, auto D) {
        return plan_nf<decltype(F)::value, decltype(G)::value, decltype(D)::value, kF32>(N, K, P);
    });
    if (e != cudaSuccess) return -1;
    return P.tail > 0 ? 2 : 1;
}

int set_force_gemv_split(int ks) {
    if (ks != 0 && ks != 1 && ks != 2 && ks != 4) return MMQ_ERR_ARG;
    t_force_ks = ks;
    return MMQ_OK;
}

int forced_gemv_split() { return t_force_ks; }

}  // namespace mmq
