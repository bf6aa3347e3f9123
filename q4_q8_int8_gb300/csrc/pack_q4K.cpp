// Host q4_K packer: separate fields -> customary 144-byte super-blocks.
//
// Fields follow web page "20 . r15 -- f32-accumulate mma probe (dead end) +
// rank-1 term2 rescale", section 2.1 (fp16 d and dmin per 256-element
// super-block; 6-bit sc and m per 32-element sub-block, read back with
// get_scale_min_k4 semantics; 4-bit quants v).  Byte layout of one block:
//   [0,2)   d, fp16 little endian        [2,4)  dmin, fp16 little endian
//   [4,16)  s[12]: sub-blocks 0-3 keep sc in s[c] bits 0-5 and m in s[c+4]
//           bits 0-5; sub-blocks 4-7 keep the low nibbles of sc and m in
//           s[c+4] (sc low, m high) and their top two bits in bits 6-7 of
//           s[c-4] (sc) and s[c] (m)
//   [16,144) nibbles: element 64p + 32h + l (p < 4, h < 2, l < 32) is the
//           low (h = 0) or high (h = 1) nibble of byte 32p + l
#include <cstring>

#include "../../include/mmq.h"

extern "C" int mmq_pack_q4K(const uint8_t* v_host, const uint8_t* sc_host,
                            const uint8_t* m_host, const uint16_t* d_host,
                            const uint16_t* dmin_host, int64_t N, int64_t K,
                            uint8_t* out_host) {
    if (!v_host || !sc_host || !m_host || !d_host || !dmin_host || !out_host) return MMQ_ERR_ARG;
    if (N < 1 || K < 256 || (K % 256) != 0) return MMQ_ERR_ARG;
    const int64_t nsb = K / 256;
    for (int64_t i = 0; i < N * K; ++i)
        if (v_host[i] > 15) return MMQ_ERR_ARG;
    for (int64_t i = 0; i < N * (K / 32); ++i)
        if (sc_host[i] > 63 || m_host[i] > 63) return MMQ_ERR_ARG;

    for (int64_t j = 0; j < N; ++j) {
        for (int64_t b = 0; b < nsb; ++b) {
            uint8_t* o = out_host + (j * nsb + b) * 144;
            const uint16_t d = d_host[j * nsb + b], dm = dmin_host[j * nsb + b];
            o[0] = uint8_t(d & 0xFF);
            o[1] = uint8_t(d >> 8);
            o[2] = uint8_t(dm & 0xFF);
            o[3] = uint8_t(dm >> 8);
            const uint8_t* sc = sc_host + j * (K / 32) + b * 8;
            const uint8_t* mm = m_host + j * (K / 32) + b * 8;
            uint8_t* s = o + 4;
            for (int c = 0; c < 4; ++c) {
                s[c] = uint8_t(sc[c] | ((sc[c + 4] >> 4) << 6));
                s[c + 4] = uint8_t(mm[c] | ((mm[c + 4] >> 4) << 6));
                s[c + 8] = uint8_t((sc[c + 4] & 15) | ((mm[c + 4] & 15) << 4));
            }
            const uint8_t* v = v_host + j * K + b * 256;
            uint8_t* q = o + 16;
            for (int p = 0; p < 4; ++p)
                for (int l = 0; l < 32; ++l)
                    q[32 * p + l] = uint8_t(v[64 * p + l] | (v[64 * p + 32 + l] << 4));
        }
    }
    return MMQ_OK;
}
