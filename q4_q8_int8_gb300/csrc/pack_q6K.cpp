// Host q6_K packer: separate fields -> customary 210-byte super-blocks.
//
// The q6_K family follows q4_K on the pages' MMQ line (web page "20 . r15 --
// f32-accumulate mma probe (dead end) + rank-1 term2 rescale", section
// "Proof of pattern portability"); the pages print no layout, and this is
// the customary one.  Per 256-weight super-block:
//   [0,128)   ql: element 128n + 32r + l (n < 2, r < 4, l < 32) keeps the
//             low 4 bits of u = q + 32 in nibble r / 2 of byte 64n + 32(r % 2) + l
//   [128,192) qh: its top 2 bits in bits 2r, 2r + 1 of byte 128 + 32n + l
//   [192,208) int8 scale of each 16 consecutive weights
//   [208,210) d, fp16 little endian
#include <cstring>

#include "../../include/mmq.h"

extern "C" size_t mmq_q6K_bytes(int64_t N, int64_t K) {
    if (N < 1 || K < 256 || (K % 256) != 0) return 0;
    return size_t(N) * size_t(K / 256) * 210;
}

extern "C" int mmq_pack_q6K(const int8_t* q_host, const int8_t* sc_host, const uint16_t* d_host,
                            int64_t N, int64_t K, uint8_t* out_host) {
    if (!q_host || !sc_host || !d_host || !out_host) return MMQ_ERR_ARG;
    if (N < 1 || K < 256 || (K % 256) != 0) return MMQ_ERR_ARG;
    for (int64_t i = 0; i < N * K; ++i)
        if (q_host[i] < -32 || q_host[i] > 31) return MMQ_ERR_ARG;
    const int64_t nsb = K / 256;
    for (int64_t j = 0; j < N; ++j) {
        for (int64_t b = 0; b < nsb; ++b) {
            uint8_t* o = out_host + (j * nsb + b) * 210;
            std::memset(o, 0, 192);
            const int8_t* q = q_host + j * K + b * 256;
            for (int n = 0; n < 2; ++n)
                for (int r = 0; r < 4; ++r)
                    for (int l = 0; l < 32; ++l) {
                        const unsigned u = unsigned(q[128 * n + 32 * r + l] + 32);   // 0..63
                        o[64 * n + 32 * (r % 2) + l] |= uint8_t((u & 15u) << (4 * (r / 2)));
                        o[128 + 32 * n + l] |= uint8_t((u >> 4) << (2 * r));
                    }
            std::memcpy(o + 192, sc_host + j * (K / 16) + b * 16, 16);
            const uint16_t d = d_host[j * nsb + b];
            o[208] = uint8_t(d & 0xFF);
            o[209] = uint8_t(d >> 8);
        }
    }
    return MMQ_OK;
}
