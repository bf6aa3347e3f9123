// Pieces shared by the tcgen05 GEMM kernels (one CTA and CTA-pair forms):
// operand unpack arithmetic, shared-memory and cluster accessors, the
// epilogue's packed FMA and stores, and the host-side tensor-map encoder.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <mutex>

#include "q8_round.cuh"
#include "sm103_ptx.cuh"

namespace mmq {
namespace tc {

using namespace mmq::ptx;

constexpr float kSubnormalScale = 16777216.0f;   // 2^24: weight factors are fp16 subnormals

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

// 6-bit scales / mins of a q4_K super-block (12 bytes s[0..11] as three
// words), four per word, one per byte: sub-blocks 0-3 are the low six bits
// of s[0..3] / s[4..7]; sub-blocks 4-7 take their low four bits from s[8..11]
// (low / high nibble) and their top two bits from the top of s[0..3] / s[4..7].
__device__ __forceinline__ uint32_t sc_lo4(uint32_t s0) { return s0 & 0x3F3F3F3Fu; }
__device__ __forceinline__ uint32_t sc_hi4(uint32_t s0, uint32_t s2) {
    return (s2 & 0x0F0F0F0Fu) | ((s0 >> 2) & 0x30303030u);
}
__device__ __forceinline__ uint32_t m_lo4(uint32_t s1) { return s1 & 0x3F3F3F3Fu; }
__device__ __forceinline__ uint32_t m_hi4(uint32_t s1, uint32_t s2) {
    return ((s2 >> 4) & 0x0F0F0F0Fu) | ((s1 >> 2) & 0x30303030u);
}

// x = hi + lo with hi = x truncated to tf32 (low 13 mantissa bits cleared);
// lo = x - hi is exact in f32.
__device__ __forceinline__ void split_tf32(float x, float& hi, float& lo) {
    hi = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
    lo = x - hi;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}
__device__ __forceinline__ void st_shared_v4f(uint32_t addr, float a, float b, float c, float d) {
    st_shared_v4(addr, __float_as_uint(a), __float_as_uint(b), __float_as_uint(c), __float_as_uint(d));
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
__device__ __forceinline__ float4 ld_shared_v4f(uint32_t addr) {
    const uint4 v = ld_shared_v4(addr);
    return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w));
}

// Completes this thread's shared-memory loads that produced v before what
// follows, through a store that depends on them (to a scratch word).  A
// release arrival that frees a ring slot for its next TMA copy goes after it:
// the arrival alone does not wait for a load still queued behind other
// shared-memory traffic, and the copy could land under it.
__device__ __forceinline__ void loads_done(uint32_t scratch, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(scratch), "r"(v) : "memory");
}
__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
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
// Store to a peer CTA's shared memory (an address from map_shared_rank); no
// round trip: the issuing thread does not wait for it.
__device__ __forceinline__ void st_dsmem_v4(uint32_t addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}
__device__ __forceinline__ float4 ld_dsmem_v4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// One 32-column half of a buffer: acc[16h + j] += m * D[32h + 2j, +1].
template <int H>
__device__ __forceinline__ void half_fma(uint64_t (&acc)[32], const uint32_t (&b)[32], uint64_t m2) {
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[16 * H + j] = ffma2(pack2u(b[2 * j], b[2 * j + 1]), m2, acc[16 * H + j]);
}

// S dump of one 16-column part (block dots, bit for bit).
__device__ __forceinline__ void dump_part(int32_t* S, const uint32_t (&b)[16], int64_t gr, int gc0, int M,
                                          int N, int nb, int kb) {
    if (gr >= M) return;
#pragma unroll
    for (int j = 0; j < 16; ++j)
        if (gc0 + j < N)
            S[(gr * N + gc0 + j) * int64_t(nb) + kb] = int32_t(__uint_as_float(b[j]) * kSubnormalScale);
}

// Epilogue thread's row x 64 columns of the 128x128 tile (m0, n0) -> C.
__device__ __forceinline__ void store_tile(float* C, const uint64_t (&acc)[32], int M, int N, int m0,
                                           int n0, int row, int colhalf) {
    const int64_t gr = int64_t(m0) + row;
    if (gr >= M) return;
    float* crow = C + gr * N;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int gc = n0 + colhalf * 64 + 4 * i;   // N % 4 == 0: all four columns or none
        if (gc < N)
            *reinterpret_cast<float4*>(crow + gc) =
                make_float4(lo_f(acc[2 * i]), hi_f(acc[2 * i]), lo_f(acc[2 * i + 1]), hi_f(acc[2 * i + 1]));
    }
}

// One q8_1 block from 32 f32 values: amax, da = amax / 127 (IEEE division),
// q = roundf(c / da) (the quotient of IEEE division, as in the prepass)
// clamped to +-127, sa = sum of q; da == 0 gives q = 0 and sa = 0 (web page
// "20 . r15 -- f32-accumulate mma probe (dead end) + rank-1 term2 rescale",
// section 2.1, for the format).  Writes 32 quants at qrow (16-byte aligned).
__device__ __forceinline__ void quantize_block32(const float (&v)[32], int8_t* qrow, float* da_out,
                                                 int32_t* sa_out) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const float d = __fdiv_rn(amax, 127.0f);
    int qv[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) qv[i] = 0;   // a zero scale gives zero quants
    if (d != 0.0f) {
        // the prepass's rounding: reciprocal fast path, IEEE division where
        // a quotient lies too close to a half-integer (or d is subnormal)
        bool redo = d < 0x1p-126f;
        const float r = __frcp_rn(d);
#pragma unroll
        for (int i = 0; i < 32; ++i) qv[i] = q8::quant_fast(v[i], r, redo);
        if (redo) {
#pragma unroll
            for (int i = 0; i < 32; ++i) qv[i] = q8::quant_exact(v[i], d);
        }
    }
    uint32_t w[8];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t word = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int q = q8::clamp127(qv[4 * i + e]);
            sum += q;
            word |= (uint32_t(q) & 0xFFu) << (8 * e);
        }
        w[i] = word;
    }
    *reinterpret_cast<uint4*>(qrow) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(qrow + 16) = make_uint4(w[4], w[5], w[6], w[7]);
    *da_out = d;
    *sa_out = sum;
}

// The same row x 64 columns quantized to q8_1 (two 32-column blocks of an
// [M][N] q8_1 output, N % 32 == 0): the same operation as the q8_1 prepass
// on the stored f32 values.
__device__ __forceinline__ void store_tile_q8_1(mmq_q8_1_t out, const uint64_t (&acc)[32], int M, int N,
                                                int m0, int n0, int row, int colhalf) {
    const int64_t gr = int64_t(m0) + row;
    if (gr >= M) return;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
        const int gc = n0 + colhalf * 64 + 32 * blk;
        if (gc >= N) continue;
        float v[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            v[2 * i] = lo_f(acc[16 * blk + i]);
            v[2 * i + 1] = hi_f(acc[16 * blk + i]);
        }
        const int64_t bi = gr * (N / 32) + gc / 32;
        quantize_block32(v, out.qs + gr * N + gc, out.da + bi, out.sa + bi);
    }
}

// SwiGLU of an interleaved gate / up tile, quantized to q8_1: the weight rows
// of the GEMM alternate gate_f, up_f, so each packed pair acc[i] of this
// thread's 64 columns is (g, u) of one feature, and the 32 features
// (n0 + 64 colhalf) / 2 + i form one q8_1 block of the [M][F] output
// (F % 32 == 0):  h = silu(g) * u = g / (1 + exp(-g)) * u in f32.  hf, if
// not null, receives h as f32 [M][F].
__device__ __forceinline__ void store_tile_swiglu_q8_1(mmq_q8_1_t out, float* hf, const uint64_t (&acc)[32],
                                                       int M, int F, int m0, int n0, int row, int colhalf) {
    const int64_t gr = int64_t(m0) + row;
    const int f0 = (n0 + colhalf * 64) / 2;
    if (gr >= M || f0 >= F) return;
    float h[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float g = lo_f(acc[i]), u = hi_f(acc[i]);
        h[i] = __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
    }
    if (hf) {
        float* hrow = hf + gr * F + f0;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float4*>(hrow + 4 * i) = make_float4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
    }
    const int64_t bi = gr * (F / 32) + f0 / 32;
    quantize_block32(h, out.qs + gr * F + f0, out.da + bi, out.sa + bi);
}

// ------------------------------------------------------------------- host
inline PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
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

inline bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
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

}  // namespace tc
}  // namespace mmq
