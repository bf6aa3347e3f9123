// q6_K x q8_1 GEMM on warp-level integer MMA, and the load-time repack of
// q6_K weights into a 16-byte aligned device layout.
//
// q6_K is the weight family the pages' MMQ line moved to next (web page "20
// . r15 -- f32-accumulate mma probe (dead end) + rank-1 term2 rescale",
// section "Proof of pattern portability"), on warp-level mma.sync kernels.
// Weights: 256-element super-blocks with an fp16 d, an int8 scale per 16
// consecutive elements, and 6-bit quants stored as u = q + 32 (q in
// [-32, 31]); no minimum, so the rescale has one term.  Per 16-element
// sub-block s the integer MMA produces S_is exactly (|S| <= 16*127*32), then
//     acc_ij += (da_i,s/2 * d_j * sc_j,s) * S_ijs.
//
// Device layout (mmq_repack_q6K): each customary 210-byte super-block padded
// to 224 bytes (ql[128], qh[64], scales[16], d, 14 zero bytes), so that a row
// of super-blocks is a whole number of 16-byte pieces for cp.async.
//
// Design (the control kernel's shape, gemm_mma.cu): CTA tile 128 tokens x
// 128 weight rows, 8 warps as 2 x 4, 16 MMA chains per warp; one super-block
// per cp.async stage (3 in flight).  A fragments by ldmatrix from int8 rows;
// the m16n8k32 A fragment's two halves are the m16n8k16 fragments of the
// chunk's two sub-blocks.  B fragments are built from the raw bytes: for
// chunk c = 4n + r of a super-block, the four quants of a fragment register
// are nibble r/2 of one ql word and bit pair r of one qh word, and
// __vsub4(u, 32) makes them int8.  The s32 accumulators are seeded with the
// bits of 1.5 * 2^23, so one FADD recovers S as a float.
#include <cuda_fp16.h>

#include <atomic>

#include "mmq_internal.h"
#include "sm103_ptx.cuh"

namespace {

constexpr int BM = 128, BN = 128, kThreads = 256, kStages = 3;
constexpr int kQ6Bytes = 210, kQ6DevBytes = 224;
constexpr int kARowBytes = 272;                        // 256 + 16 pad
constexpr int kAStage = BM * kARowBytes;               // 34816
constexpr int kWStage = BN * kQ6DevBytes;              // 28672
constexpr int kDaStage = BM * 8 * 4;                   // 4096
constexpr int kStageBytes = kAStage + kWStage + kDaStage;
constexpr int kSmemBytes = kStages * kStageBytes + 16 * 128 * 4 + 8 * 128 * 4;   // + d*sc and da tables
constexpr uint32_t kBiasBits = 0x4B400000u;            // 12582912.0f
constexpr float kBias = 12582912.0f;
static_assert(kSmemBytes <= 232448, "shared memory budget");

// ---------------------------------------------------------------- repack
// One thread per 16-byte piece of the padded layout (14 per super-block).
__global__ void __launch_bounds__(256) repack_q6K_kernel(const uint8_t* __restrict__ src,
                                                         uint8_t* __restrict__ dst, int64_t pieces) {
    const int64_t p = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (p >= pieces) return;
    const int64_t sbi = p / 14;
    const int off = int(p - sbi * 14) * 16;
    const uint8_t* s = src + sbi * kQ6Bytes + off;
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t v = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int o = off + 4 * i + b;
            v |= uint32_t(o < kQ6Bytes ? s[4 * i + b] : 0) << (8 * b);
        }
        w[i] = v;
    }
    *reinterpret_cast<uint4*>(dst + sbi * kQ6DevBytes + off) = make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// m16n8k16 s8 x s8 -> s32, accumulate in place.
__device__ __forceinline__ void mma_s8_k16(uint32_t (&c)[4], uint32_t a0, uint32_t a1, uint32_t b) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};\n"
        : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
        : "r"(a0), "r"(a1), "r"(b));
}

__device__ __forceinline__ void load_stage(uint32_t st, const mmq_q8_1_t& aq, const uint8_t* w, int64_t M,
                                           int64_t N, int64_t K, int64_t m0, int64_t n0, int64_t sb) {
    const int t = threadIdx.x;
    const int64_t nsb = K / 256, nb = K / 32;
#pragma unroll
    for (int i = 0; i < (BM * 16) / kThreads; ++i) {   // A: 128 rows x 16 pieces
        const int piece = t + i * kThreads;
        const int r = piece >> 4, seg = piece & 15;
        const bool ok = (m0 + r) < M;
        const int8_t* src = ok ? aq.qs + (m0 + r) * K + sb * 256 + seg * 16 : aq.qs;
        cp_async16(st + r * kARowBytes + seg * 16, src, ok);
    }
    for (int piece = t; piece < BN * 14; piece += kThreads) {   // W: 128 rows x 14 pieces
        const int r = piece / 14, seg = piece - r * 14;
        const bool ok = (n0 + r) < N;
        const uint8_t* src = ok ? w + ((n0 + r) * nsb + sb) * kQ6DevBytes + seg * 16 : w;
        cp_async16(st + kAStage + r * kQ6DevBytes + seg * 16, src, ok);
    }
    {   // da: 128 rows x 2 pieces
        const int r = t >> 1, seg = t & 1;
        const bool ok = (m0 + r) < M;
        const float* sd = ok ? aq.da + (m0 + r) * nb + sb * 8 + seg * 4 : aq.da;
        cp_async16(st + kAStage + kWStage + r * 32 + seg * 16, sd, ok);
    }
}

__device__ __forceinline__ void q6_cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float4 q6_ld_peer_v4(uint32_t saddr, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(saddr), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(a)
                 : "memory");
    return v;
}

// split > 1 (few tiles): a cluster of `split` CTAs along z shares one tile,
// rank r taking super-blocks [nsb*r/split, nsb*(r+1)/split); each rank leaves
// its partial tile in its own (then idle) stage memory and rank 0 adds them
// in rank order, so the sum is the same on every run.
template <bool kDump>
__global__ void __launch_bounds__(kThreads, 1)
gemm_q6k_kernel(mmq_q8_1_t aq, const uint8_t* __restrict__ w, float* __restrict__ C, int32_t* __restrict__ S,
                int64_t M, int64_t N, int64_t K, int split) {
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    float* colsc = reinterpret_cast<float*>(smem + kStages * kStageBytes);   // d * sc [16][128]
    float* rowda = colsc + 16 * 128;                                        // da [8][128]

    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int wm = warp & 1, wn = warp >> 1;
    const int64_t m0 = int64_t(blockIdx.y) * BM, n0 = int64_t(blockIdx.x) * BN;
    const int64_t nsb = K / 256;
    const int64_t ns16 = K / 16;
    const int rank = split > 1 ? int(blockIdx.z) : 0;
    const int64_t sb_lo = nsb * rank / split, cnt = nsb * (rank + 1) / split - sb_lo;

    float acc[4][4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[a][b][r] = 0.0f;

#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (s < cnt) load_stage(sbase + s * kStageBytes, aq, w, M, N, K, m0, n0, sb_lo + s);
        cp_async_commit();
    }

    for (int64_t i = 0; i < cnt; ++i) {
        const int64_t sb = sb_lo + i;
        cp_async_wait<kStages - 2>();
        __syncthreads();   // stage i visible; everyone is done with i-1
        {
            const int64_t nx = i + kStages - 1;
            if (nx < cnt) load_stage(sbase + (nx % kStages) * kStageBytes, aq, w, M, N, K, m0, n0, sb_lo + nx);
            cp_async_commit();
        }
        const int st = int(i % kStages);
        const uint8_t* sA = smem + st * kStageBytes;
        const uint8_t* sW = sA + kAStage;
        const float* sDa = reinterpret_cast<const float*>(sW + kWStage);

        if (!kDump) {
            {   // d * sc per weight row and sub-block (exact in f32: 11 x 8 bits)
                const int n = t >> 1, s8 = (t & 1) * 8;
                const uint8_t* blk = sW + n * kQ6DevBytes;
                const float d = __half2float(__ushort_as_half(uint16_t(blk[208] | (blk[209] << 8))));
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    colsc[(s8 + k) * 128 + n] = d * float(int8_t(blk[192 + s8 + k]));
            }
            {   // da per token row and chunk
                const int r = t >> 1, c4 = (t & 1) * 4;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) rowda[(c4 + cc) * 128 + r] = sDa[r * 8 + c4 + cc];
            }
            __syncthreads();
        }

        const uint32_t aRowAddr = sbase + st * kStageBytes +
                                  (wm * 64 + (lane & 7) + ((lane >> 3) & 1) * 8) * kARowBytes + (lane >> 4) * 16;
#pragma unroll 1
        for (int n = 0; n < 2; ++n) {   // half n of the super-block: chunks 4n .. 4n + 3
#pragma unroll 1
            for (int r = 0; r < 4; ++r) {
                const int c = 4 * n + r;   // chunk within the super-block
                // this chunk's ql word (nibble r / 2) and qh word (bit pair r) per fragment and half
                uint32_t qlw[4][2], qhw[4][2];
#pragma unroll
                for (int fn = 0; fn < 4; ++fn) {
                    const uint8_t* row = sW + (wn * 32 + fn * 8 + (lane >> 2)) * kQ6DevBytes;
#pragma unroll
                    for (int kh = 0; kh < 2; ++kh) {
                        const int l = 16 * kh + (lane & 3) * 4;
                        qlw[fn][kh] = *reinterpret_cast<const uint32_t*>(row + 64 * n + 32 * (r & 1) + l);
                        qhw[fn][kh] = *reinterpret_cast<const uint32_t*>(row + 128 + 32 * n + l);
                    }
                }
                uint32_t af[4][4];
#pragma unroll
                for (int fm = 0; fm < 4; ++fm)
                    ldmatrix_x4(aRowAddr + fm * 16 * kARowBytes + c * 32, af[fm][0], af[fm][1], af[fm][2],
                                af[fm][3]);
#pragma unroll 1
                for (int kh = 0; kh < 2; ++kh) {   // sub-block 2c + kh
                    uint32_t ci[4][4][4];
#pragma unroll
                    for (int fm = 0; fm < 4; ++fm)
#pragma unroll
                        for (int fn = 0; fn < 4; ++fn)
#pragma unroll
                            for (int i = 0; i < 4; ++i) ci[fm][fn][i] = kDump ? 0u : kBiasBits;
#pragma unroll
                    for (int fn = 0; fn < 4; ++fn) {
                        // selects, not run-time indexing, keep these arrays in registers
                        const uint32_t lw = kh ? qlw[fn][1] : qlw[fn][0], hw = kh ? qhw[fn][1] : qhw[fn][0];
                        const uint32_t u = ((lw >> (4 * (r >> 1))) & 0x0F0F0F0Fu) | (((hw >> (2 * r)) & 0x03030303u) << 4);
                        const uint32_t b = __vsub4(u, 0x20202020u);   // u - 32 per byte: int8 quants
#pragma unroll
                        for (int fm = 0; fm < 4; ++fm)
                            mma_s8_k16(ci[fm][fn], kh ? af[fm][2] : af[fm][0], kh ? af[fm][3] : af[fm][1], b);
                    }
                    const int s16 = 2 * c + kh;
                    if (kDump) {
#pragma unroll
                        for (int fm = 0; fm < 4; ++fm)
#pragma unroll
                            for (int fn = 0; fn < 4; ++fn)
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const int64_t row = m0 + wm * 64 + fm * 16 + (lane >> 2) + (i >> 1) * 8;
                                    const int64_t col = n0 + wn * 32 + fn * 8 + (lane & 3) * 2 + (i & 1);
                                    if (row < M && col < N)
                                        S[(row * N + col) * ns16 + sb * 16 + s16] = int32_t(ci[fm][fn][i]);
                                }
                    } else {
                        float da[4][2];
#pragma unroll
                        for (int fm = 0; fm < 4; ++fm)
#pragma unroll
                            for (int hr = 0; hr < 2; ++hr)
                                da[fm][hr] = rowda[c * 128 + wm * 64 + fm * 16 + (lane >> 2) + hr * 8];
#pragma unroll
                        for (int fn = 0; fn < 4; ++fn) {
                            const float2 ds = *reinterpret_cast<const float2*>(
                                &colsc[s16 * 128 + wn * 32 + fn * 8 + (lane & 3) * 2]);
#pragma unroll
                            for (int fm = 0; fm < 4; ++fm)
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const float sv = __uint_as_float(ci[fm][fn][i]) - kBias;
                                    acc[fm][fn][i] = fmaf(da[fm][i >> 1] * ((i & 1) ? ds.y : ds.x), sv,
                                                          acc[fm][fn][i]);
                                }
                        }
                    }
                }
            }
        }
    }
    cp_async_wait<0>();

    if (!kDump && split > 1) {
        __syncthreads();   // every warp is done with the stages: reuse them for the partial tile
        float4* mine = reinterpret_cast<float4*>(smem) + t * 16;
#pragma unroll
        for (int fm = 0; fm < 4; ++fm)
#pragma unroll
            for (int fn = 0; fn < 4; ++fn)
                mine[fm * 4 + fn] = make_float4(acc[fm][fn][0], acc[fm][fn][1], acc[fm][fn][2], acc[fm][fn][3]);
        q6_cluster_sync();   // every rank's partial is in its shared memory
        if (rank == 0) {
            for (int r = 1; r < split; ++r)
#pragma unroll
                for (int fm = 0; fm < 4; ++fm)
#pragma unroll
                    for (int fn = 0; fn < 4; ++fn) {
                        const float4 v = q6_ld_peer_v4(sbase + uint32_t(t * 256 + (fm * 4 + fn) * 16), uint32_t(r));
                        acc[fm][fn][0] += v.x;
                        acc[fm][fn][1] += v.y;
                        acc[fm][fn][2] += v.z;
                        acc[fm][fn][3] += v.w;
                    }
        }
        q6_cluster_sync();   // the peers' memory stays alive until rank 0 has read it
        if (rank != 0) return;
    }
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

// ---------------------------------------------------------------------------
// M <= 4 tokens: a streaming dot product on dp4a, one warp per kGvR weight
// rows.  Lane l takes chunks l, l+32, ... of each row (chunk c = 4n + r of a
// super-block: its 32 quants are nibble r/2 of ql[64n + 32(r%2) + l] and
// bit pair r of qh[32n + l], l = 0..31); the 6-bit u becomes the int8 q = u -
// 32 per byte, two dp4a chains give the exact dots of the chunk's two
// 16-element sub-blocks, and acc += da * (d * sc) * S per sub-block.  Every
// activation load serves the warp's kGvR rows.  A row taking r rounds of 32
// chunks is shared by min(4, r) warps of the CTA, whose partial sums are
// added in slice order through shared memory.
// ---------------------------------------------------------------------------
constexpr int kGvR = 4;

template <int MT, int KS>
__global__ void __launch_bounds__(128)
gemv_q6k_kernel(mmq_q8_1_t aq, const uint8_t* __restrict__ w, float* __restrict__ C, int M, int N, int K) {
    constexpr int kGroups = 4 / KS;   // row groups (of kGvR rows) per CTA
    __shared__ float part[KS > 1 ? 4 : 1][MT][kGvR];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slice = warp % KS, grp = warp / KS;
    const int row0 = (blockIdx.x * kGroups + grp) * kGvR;
    mmq::ptx::griddep_launch_dependents();
    if (KS == 1 && row0 >= N) return;
    const int nsb = K / 256, nch = K / 32;
    float acc[MT][kGvR];
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int r = 0; r < kGvR; ++r) acc[t][r] = 0.0f;
    for (int base = 32 * slice; base < nch; base += 32 * KS) {
        const int ci = base + lane;   // this lane's chunk of the row
        const int c = ci & 7, n = c >> 2, rr = c & 3;
        uint4 ql[kGvR][2], qh[kGvR][2];
        uint32_t scw[kGvR], dw[kGvR];
#pragma unroll
        for (int r = 0; r < kGvR; ++r) {
            if (ci < nch && row0 + r < N) {
                const uint8_t* blk = w + (int64_t(row0 + r) * nsb + (ci >> 3)) * 224;
                ql[r][0] = __ldcs(reinterpret_cast<const uint4*>(blk + 64 * n + 32 * (rr & 1)));
                ql[r][1] = __ldcs(reinterpret_cast<const uint4*>(blk + 64 * n + 32 * (rr & 1) + 16));
                qh[r][0] = __ldcs(reinterpret_cast<const uint4*>(blk + 128 + 32 * n));
                qh[r][1] = __ldcs(reinterpret_cast<const uint4*>(blk + 128 + 32 * n + 16));
                scw[r] = __ldg(reinterpret_cast<const uint16_t*>(blk + 192 + 2 * c));
                dw[r] = __ldg(reinterpret_cast<const uint16_t*>(blk + 208));
            } else {
                ql[r][0] = ql[r][1] = qh[r][0] = qh[r][1] = make_uint4(0u, 0u, 0u, 0u);
                scw[r] = dw[r] = 0u;
            }
        }
        // weights stream in while the previous kernel (programmatic dependent
        // launch) finishes; activations and C only after it has
        if (base == 32 * slice) mmq::ptx::griddep_wait();
        if (ci >= nch) continue;
        float ds[kGvR][2];   // d * sc of the chunk's two sub-blocks (exact in f32)
        uint32_t qw[kGvR][8];   // the chunk's 32 quants as int8, once for all tokens
#pragma unroll
        for (int r = 0; r < kGvR; ++r) {
            const float d = __half2float(__ushort_as_half(uint16_t(dw[r])));
            ds[r][0] = d * float(int8_t(scw[r] & 0xFFu));
            ds[r][1] = d * float(int8_t(scw[r] >> 8));
            const uint32_t lw[8] = {ql[r][0].x, ql[r][0].y, ql[r][0].z, ql[r][0].w,
                                    ql[r][1].x, ql[r][1].y, ql[r][1].z, ql[r][1].w};
            const uint32_t hw[8] = {qh[r][0].x, qh[r][0].y, qh[r][0].z, qh[r][0].w,
                                    qh[r][1].x, qh[r][1].y, qh[r][1].z, qh[r][1].w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const uint32_t u = ((lw[e] >> (4 * (rr >> 1))) & 0x0F0F0F0Fu) | (((hw[e] >> (2 * rr)) & 0x03030303u) << 4);
                qw[r][e] = __vsub4(u, 0x20202020u);   // u - 32 per byte: int8 quants
            }
        }
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            if (t < M) {
                const int8_t* qt = aq.qs + int64_t(t) * K + 32 * ci;
                const uint4 a0 = __ldg(reinterpret_cast<const uint4*>(qt));
                const uint4 a1 = __ldg(reinterpret_cast<const uint4*>(qt + 16));
                const float da = __ldg(aq.da + int64_t(t) * nch + ci);
                const uint32_t av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                for (int r = 0; r < kGvR; ++r) {
                    int s0 = 0, s1 = 0;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        s0 = __dp4a(int(qw[r][e]), int(av[e]), s0);
                        s1 = __dp4a(int(qw[r][4 + e]), int(av[4 + e]), s1);
                    }
                    float a = acc[t][r];
                    a = fmaf(da * ds[r][0], float(s0), a);
                    a = fmaf(da * ds[r][1], float(s1), a);
                    acc[t][r] = a;
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int r = 0; r < kGvR; ++r) {
            float a = acc[t][r];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
            acc[t][r] = a;
        }
    if constexpr (KS > 1) {
        if (lane == 0) {
#pragma unroll
            for (int t = 0; t < MT; ++t)
#pragma unroll
                for (int r = 0; r < kGvR; ++r) part[warp][t][r] = acc[t][r];
        }
        __syncthreads();
        if (slice == 0) {
#pragma unroll
            for (int t = 0; t < MT; ++t)
#pragma unroll
                for (int r = 0; r < kGvR; ++r) {
                    float a = part[warp][t][r];
#pragma unroll
                    for (int q = 1; q < KS; ++q) a += part[warp + q][t][r];
                    acc[t][r] = a;
                }
        }
    }
    if (slice == 0 && lane == 0) {
#pragma unroll
        for (int t = 0; t < MT; ++t)
#pragma unroll
            for (int r = 0; r < kGvR; ++r)
                if (t < M && row0 + r < N) C[int64_t(t) * N + row0 + r] = acc[t][r];
    }
}

template <int MT, int KS>
cudaError_t launch_gemv_q6k_ks(mmq_q8_1_t aq, const uint8_t* w, float* C, int64_t M, int64_t N, int64_t K,
                               cudaStream_t s) {
    constexpr int rows = 4 / KS * kGvR;   // rows per CTA
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = mmq::launch_config(dim3(unsigned((N + rows - 1) / rows)), dim3(128), 0, s, attr);
    return cudaLaunchKernelEx(&cfg, gemv_q6k_kernel<MT, KS>, aq, w, C, int(M), int(N), int(K));
}

// CTAs of one kernel instance resident on the device at once (register
// bound), found once per instance and device.
constexpr int kMaxDevices = 64;
template <int MT, int KS>
int64_t gemv_q6k_resident() {
    static std::atomic<int64_t> cached[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        dev = -1;
    }
    int64_t v = dev >= 0 ? cached[dev].load(std::memory_order_relaxed) : 0;
    if (v == 0) {
        int nsm = 0, per = 0;
        if (dev < 0 || cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, gemv_q6k_kernel<MT, KS>, 128, 0) != cudaSuccess) {
            cudaGetLastError();
            nsm = nsm > 0 ? nsm : 1;
            per = 1;
        }
        v = int64_t(per > 0 ? per : 1) * (nsm > 0 ? nsm : 1);
        if (dev >= 0) cached[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

// The K split (KS warps per row group), from the resident CTAs of each
// instance and a cost per launch:
// * up to 4 tokens the kernel waits on memory: waves of CTAs x (dependent
//   load rounds per warp + 1/2), as for the q4_K dot-product kernel;
// * with 8 and 16 tokens it is compute-bound: waves x rounds, over splits 2
//   and 4 (ties to 4; split 1 was slowest on every measured shape).
// Measured at 16 tokens (graph replay, us, splits 1 / 2 / 4): 4096 x 4096
// 32.1 / 24.2 / 23.8, 4096 -> 11008 57.7 / 38.4 / 52.4, 11008 -> 4096
// 84.4 / 63.1 / 59.3; the rule picks the fastest of each.
template <int MT>
cudaError_t launch_gemv_q6k(mmq_q8_1_t aq, const uint8_t* w, float* C, int64_t M, int64_t N, int64_t K,
                            cudaStream_t s) {
    const int64_t nch = K / 32;
    switch (mmq::forced_gemv_split()) {   // test hook
        case 1: return launch_gemv_q6k_ks<MT, 1>(aq, w, C, M, N, K, s);
        case 2: return launch_gemv_q6k_ks<MT, 2>(aq, w, C, M, N, K, s);
        case 4: return launch_gemv_q6k_ks<MT, 4>(aq, w, C, M, N, K, s);
        default: break;
    }
    auto shape = [&](int k, int64_t resident, int64_t& waves, int64_t& rounds) {
        const int64_t rows = 4 / k * kGvR;
        const int64_t ctas = (N + rows - 1) / rows;
        waves = (ctas + resident - 1) / resident;
        rounds = (nch + 32 * k - 1) / (32 * k);
    };
    if constexpr (MT >= 8) {
        int64_t w2, r2, w4, r4;
        shape(2, gemv_q6k_resident<MT, 2>(), w2, r2);
        shape(4, gemv_q6k_resident<MT, 4>(), w4, r4);
        if (w4 * r4 <= w2 * r2) return launch_gemv_q6k_ks<MT, 4>(aq, w, C, M, N, K, s);
        return launch_gemv_q6k_ks<MT, 2>(aq, w, C, M, N, K, s);
    }
    auto cost2 = [&](int k, int64_t resident) {   // twice the modelled cost
        int64_t waves, rounds;
        shape(k, resident, waves, rounds);
        return waves * (2 * rounds + 1);
    };
    const int64_t c1 = cost2(1, gemv_q6k_resident<MT, 1>());
    const int64_t c2 = cost2(2, gemv_q6k_resident<MT, 2>());
    const int64_t c4 = cost2(4, gemv_q6k_resident<MT, 4>());
    if (c1 <= c2 && c1 <= c4) return launch_gemv_q6k_ks<MT, 1>(aq, w, C, M, N, K, s);
    if (c4 < c2) return launch_gemv_q6k_ks<MT, 4>(aq, w, C, M, N, K, s);
    return launch_gemv_q6k_ks<MT, 2>(aq, w, C, M, N, K, s);
}

}  // namespace

namespace mmq {

cudaError_t launch_repack_q6K(const uint8_t* src, uint8_t* dst, int64_t N, int64_t K, cudaStream_t s) {
    const int64_t pieces = N * (K / 256) * 14;
    const int64_t blocks = (pieces + 255) / 256;
    repack_q6K_kernel<<<unsigned(blocks), 256, 0, s>>>(src, dst, pieces);
    return cudaGetLastError();
}

cudaError_t launch_gemm_q6k(mmq_q8_1_t aq, const uint8_t* w, float* C, int32_t* S, int64_t M, int64_t N,
                            int64_t K, cudaStream_t s, bool allow_gemv) {
    if (!S && allow_gemv && M <= kQ6GemvMax) {   // a few tokens: the dot-product kernel
        if (M == 1) return launch_gemv_q6k<1>(aq, w, C, M, N, K, s);
        if (M == 2) return launch_gemv_q6k<2>(aq, w, C, M, N, K, s);
        if (M <= 4) return launch_gemv_q6k<4>(aq, w, C, M, N, K, s);
        if (M <= 8) return launch_gemv_q6k<8>(aq, w, C, M, N, K, s);
        return launch_gemv_q6k<16>(aq, w, C, M, N, K, s);
    }
    const int64_t tiles_n = (N + BN - 1) / BN, tiles_m = (M + BM - 1) / BM;
    if (tiles_m > 65535) return cudaErrorInvalidConfiguration;
    // few tiles: split K over a cluster so that more SMs stream the weights
    int dev = 0, nsm = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    const int64_t nsb = K / 256;
    int split = 1;
    while (!S && split < 8 && 2 * split <= nsb && tiles_m * tiles_n * 2 * split <= nsm) split *= 2;
    auto k = S ? gemm_q6k_kernel<true> : gemm_q6k_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(tiles_n), unsigned(tiles_m), unsigned(split));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = size_t(kSmemBytes);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = unsigned(split);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, aq, w, C, S, M, N, K, split);
}

}  // namespace mmq
