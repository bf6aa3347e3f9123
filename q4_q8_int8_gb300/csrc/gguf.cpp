// GGUF interop (host): read and write the tensors of a GGUF file, so that
// q4_K / q6_K weights in the customary super-block layouts this library
// consumes can come from (or go to) the file format those layouts are used
// in.  Written from the published GGUF description (version 3, little
// endian):
//   magic "GGUF", u32 version, u64 tensor count, u64 metadata count;
//   metadata: string key, u32 value type, value (strings as u64 length +
//   bytes, arrays as u32 element type + u64 count + elements);
//   tensor infos: string name, u32 n_dims, u64 dims[n_dims] (dims[0] the
//   contiguous one), u32 tensor type, u64 offset into the data section;
//   the data section starts at the next multiple of general.alignment
//   (default 32) after the header, each tensor at its offset.
// Files are untrusted input: every length and offset is checked against the
// file size before use, and a file that does not parse is refused with
// MMQ_ERR_ARG.  Tensor types handled: F32 (0), F16 (1), Q4_K (12), Q6_K (14).
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/mmq.h"

namespace {

struct TensorInfo {
    std::string name;
    uint32_t type = 0;
    uint32_t ndim = 0;
    int64_t dims[4] = {1, 1, 1, 1};
    uint64_t offset = 0;   // absolute file offset of the data
    uint64_t nbytes = 0;
};

// bytes of a tensor of `type` with dims[0] x rest elements; 0 if unsupported
// or the row length does not fit the block size
uint64_t tensor_bytes(uint32_t type, const int64_t* dims, uint32_t ndim) {
    uint64_t rest = 1;
    for (uint32_t i = 1; i < ndim; ++i) {
        if (dims[i] < 1 || rest > (uint64_t(1) << 40) / uint64_t(dims[i])) return 0;
        rest *= uint64_t(dims[i]);
    }
    const uint64_t n0 = uint64_t(dims[0]);
    if (dims[0] < 1 || n0 > (uint64_t(1) << 40) || n0 > (uint64_t(1) << 44) / rest) return 0;   // <= 2^44 elements
    switch (type) {
        case MMQ_GGUF_F32: return n0 * rest * 4;
        case MMQ_GGUF_F16: return n0 * rest * 2;
        case MMQ_GGUF_Q4_K: return n0 % 256 ? 0 : n0 / 256 * 144 * rest;
        case MMQ_GGUF_Q6_K: return n0 % 256 ? 0 : n0 / 256 * 210 * rest;
        default: return 0;
    }
}

struct Reader {
    FILE* f = nullptr;
    uint64_t size = 0;
    uint64_t pos = 0;
    bool ok = true;
    bool read(void* dst, uint64_t n) {
        if (!ok || n > size - pos) return ok = false;
        if (n && std::fread(dst, 1, size_t(n), f) != size_t(n)) return ok = false;
        pos += n;
        return true;
    }
    bool skip(uint64_t n) {
        if (!ok || n > size - pos) return ok = false;
        if (std::fseek(f, long(pos + n), SEEK_SET) != 0) return ok = false;
        pos += n;
        return true;
    }
    template <class T>
    T get() {
        T v{};
        read(&v, sizeof(T));
        return v;
    }
    std::string str() {
        const uint64_t n = get<uint64_t>();
        if (!ok || n > (uint64_t(1) << 20) || n > size - pos) {
            ok = false;
            return {};
        }
        std::string s(size_t(n), '\0');
        read(&s[0], n);
        return s;
    }
};

// size of one metadata value of scalar type t (0 for string / array / unknown)
uint64_t scalar_size(uint32_t t) {
    switch (t) {
        case 0: case 1: case 7: return 1;   // u8, i8, bool
        case 2: case 3: return 2;           // u16, i16
        case 4: case 5: case 6: return 4;   // u32, i32, f32
        case 10: case 11: case 12: return 8;   // u64, i64, f64
        default: return 0;
    }
}

bool skip_value(Reader& r, uint32_t t, uint32_t* u32_out) {
    if (t == 8) {   // string
        r.str();
        return r.ok;
    }
    if (t == 9) {   // array
        const uint32_t et = r.get<uint32_t>();
        const uint64_t n = r.get<uint64_t>();
        if (!r.ok || n > (uint64_t(1) << 32)) return false;
        if (et == 8) {
            for (uint64_t i = 0; i < n && r.ok; ++i) r.str();
            return r.ok;
        }
        const uint64_t es = scalar_size(et);
        if (!es || n > (r.size - r.pos) / es) return false;
        return r.skip(n * es);
    }
    const uint64_t s = scalar_size(t);
    if (!s) return false;
    if (t == 4 && u32_out) return r.read(u32_out, 4);
    return r.skip(s);
}

}  // namespace

struct mmq_gguf {
    FILE* f = nullptr;
    uint32_t version = 0;
    uint32_t alignment = 32;
    std::vector<TensorInfo> tensors;
};

extern "C" {

int mmq_gguf_open(const char* path, mmq_gguf** out) {
    if (!path || !out) return MMQ_ERR_ARG;
    *out = nullptr;
    FILE* f = std::fopen(path, "rb");
    if (!f) return MMQ_ERR_ARG;
    Reader r;
    r.f = f;
    if (std::fseek(f, 0, SEEK_END) != 0) { std::fclose(f); return MMQ_ERR_ARG; }
    const long end = std::ftell(f);
    std::fseek(f, 0, SEEK_SET);
    if (end < 0) { std::fclose(f); return MMQ_ERR_ARG; }
    r.size = uint64_t(end);
    char magic[4];
    auto* h = new mmq_gguf;
    h->f = f;
    auto fail = [&]() {
        std::fclose(f);
        delete h;
        return MMQ_ERR_ARG;
    };
    if (!r.read(magic, 4) || std::memcmp(magic, "GGUF", 4) != 0) return fail();
    h->version = r.get<uint32_t>();
    if (!r.ok || (h->version != 2 && h->version != 3)) return fail();
    const uint64_t nt = r.get<uint64_t>(), nkv = r.get<uint64_t>();
    if (!r.ok || nt > (uint64_t(1) << 24) || nkv > (uint64_t(1) << 24)) return fail();
    for (uint64_t i = 0; i < nkv; ++i) {
        const std::string key = r.str();
        const uint32_t t = r.get<uint32_t>();
        if (!r.ok) return fail();
        uint32_t v = 0;
        const bool want = key == "general.alignment" && t == 4;
        if (!skip_value(r, t, want ? &v : nullptr)) return fail();
        if (want) {
            if (v == 0 || (v & (v - 1)) || v > 4096) return fail();
            h->alignment = v;
        }
    }
    h->tensors.resize(size_t(nt));
    for (auto& ti : h->tensors) {
        ti.name = r.str();
        ti.ndim = r.get<uint32_t>();
        if (!r.ok || ti.ndim < 1 || ti.ndim > 4) return fail();
        for (uint32_t d = 0; d < ti.ndim; ++d) ti.dims[d] = int64_t(r.get<uint64_t>());
        ti.type = r.get<uint32_t>();
        ti.offset = r.get<uint64_t>();
        if (!r.ok) return fail();
        ti.nbytes = tensor_bytes(ti.type, ti.dims, ti.ndim);
    }
    const uint64_t data0 = (r.pos + h->alignment - 1) / h->alignment * h->alignment;
    for (auto& ti : h->tensors) {
        if (ti.offset % h->alignment) return fail();
        if (ti.offset > r.size || data0 > r.size - ti.offset) return fail();
        ti.offset += data0;
        if (ti.nbytes && ti.nbytes > r.size - ti.offset) return fail();
    }
    *out = h;
    return MMQ_OK;
}

void mmq_gguf_close(mmq_gguf* h) {
    if (!h) return;
    if (h->f) std::fclose(h->f);
    delete h;
}

int64_t mmq_gguf_tensor_count(const mmq_gguf* h) { return h ? int64_t(h->tensors.size()) : -1; }

int mmq_gguf_find(const mmq_gguf* h, const char* name) {
    if (!h || !name) return -1;
    for (size_t i = 0; i < h->tensors.size(); ++i)
        if (h->tensors[i].name == name) return int(i);
    return -1;
}

int mmq_gguf_tensor_info(const mmq_gguf* h, int64_t i, char* name, size_t name_cap, uint32_t* type,
                         uint32_t* ndim, int64_t* dims4, uint64_t* nbytes) {
    if (!h || i < 0 || i >= int64_t(h->tensors.size())) return MMQ_ERR_ARG;
    const TensorInfo& t = h->tensors[size_t(i)];
    if (name && name_cap) {
        const size_t n = t.name.size() < name_cap - 1 ? t.name.size() : name_cap - 1;
        std::memcpy(name, t.name.data(), n);
        name[n] = '\0';
    }
    if (type) *type = t.type;
    if (ndim) *ndim = t.ndim;
    if (dims4)
        for (int d = 0; d < 4; ++d) dims4[d] = t.dims[d];
    if (nbytes) *nbytes = t.nbytes;
    return MMQ_OK;
}

int mmq_gguf_read(mmq_gguf* h, int64_t i, void* dst_host, uint64_t cap) {
    if (!h || !dst_host || i < 0 || i >= int64_t(h->tensors.size())) return MMQ_ERR_ARG;
    const TensorInfo& t = h->tensors[size_t(i)];
    if (!t.nbytes || cap < t.nbytes) return MMQ_ERR_ARG;
    if (std::fseek(h->f, long(t.offset), SEEK_SET) != 0) return MMQ_ERR_ARG;
    return std::fread(dst_host, 1, size_t(t.nbytes), h->f) == size_t(t.nbytes) ? MMQ_OK : MMQ_ERR_ARG;
}

int mmq_gguf_write(const char* path, int64_t n, const char* const* names, const uint32_t* types,
                   const int64_t* dims2, const void* const* data) {
    if (!path || n < 0 || (n && (!names || !types || !dims2 || !data))) return MMQ_ERR_ARG;
    std::vector<uint64_t> sizes(static_cast<size_t>(n));
    for (int64_t i = 0; i < n; ++i) {
        const int64_t d[2] = {dims2[2 * i], dims2[2 * i + 1]};
        sizes[size_t(i)] = tensor_bytes(types[i], d, 2);
        if (!sizes[size_t(i)] || !names[i] || !data[i]) return MMQ_ERR_ARG;
    }
    FILE* f = std::fopen(path, "wb");
    if (!f) return MMQ_ERR_ARG;
    bool ok = true;
    auto put = [&](const void* p, size_t k) { ok = ok && std::fwrite(p, 1, k, f) == k; };
    auto put_u32 = [&](uint32_t v) { put(&v, 4); };
    auto put_u64 = [&](uint64_t v) { put(&v, 8); };
    auto put_str = [&](const char* s) {
        const uint64_t k = std::strlen(s);
        put_u64(k);
        put(s, size_t(k));
    };
    const uint32_t align = 32;
    put("GGUF", 4);
    put_u32(3);
    put_u64(uint64_t(n));
    put_u64(1);                       // one metadata entry
    put_str("general.alignment");
    put_u32(4);                       // u32
    put_u32(align);
    uint64_t off = 0;
    std::vector<uint64_t> offs(static_cast<size_t>(n));
    for (int64_t i = 0; i < n; ++i) {
        put_str(names[i]);
        put_u32(2);
        put_u64(uint64_t(dims2[2 * i]));
        put_u64(uint64_t(dims2[2 * i + 1]));
        put_u32(types[i]);
        offs[size_t(i)] = off;
        put_u64(off);
        off = (off + sizes[size_t(i)] + align - 1) / align * align;
    }
    const long here = std::ftell(f);
    const uint64_t data0 = (uint64_t(here) + align - 1) / align * align;
    static const uint8_t zeros[32] = {};
    put(zeros, size_t(data0 - uint64_t(here)));
    for (int64_t i = 0; i < n; ++i) {
        put(data[i], size_t(sizes[size_t(i)]));
        const uint64_t pad = (align - sizes[size_t(i)] % align) % align;
        put(zeros, size_t(pad));
    }
    ok = (std::fclose(f) == 0) && ok;
    return ok ? MMQ_OK : MMQ_ERR_ARG;
}

}  // extern "C"
