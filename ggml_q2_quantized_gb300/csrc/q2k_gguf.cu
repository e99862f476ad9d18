// GGUF reader (host only): the tensor directory of a GGUF file and the bytes of
// its tensors, so that Q2_K (type 10) weights stored in one can be handed to the
// matmul, batched, routed, gather and dequantize calls.
//
// What it follows: mlx-native page "tests/deepseek_q2_k.rs", test
// q2_k_gguf_type_10_parses_with_exact_block_size (GgufFile::open and
// tensor_info, whose ggml_type must read Q2_K and byte_len one 84-byte block for
// a 256-element tensor), and the GGUF container layout that test writes:
//   "GGUF", version (u32), tensor count (u64), metadata count (u64),
//   metadata entries (key string, value type u32, value),
//   tensor entries (name string, n_dims u32, n_dims u64 extents with the
//   innermost first, type u32, offset u64 from the start of the data section),
//   padding to the alignment (32, or the u32 metadata value
//   "general.alignment"), then the data section.
// Strings are a u64 byte count and the bytes; everything is little-endian.
// Versions 2 and 3 share this layout (version 1 had 32-bit counts: rejected).
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <memory>
#include <string>
#include <unordered_map>
#include <vector>

#include "q2k.h"
#include "q2k_internal.h"

namespace {

q2k_status gguf_fail(q2k_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
q2k_status gguf_fail(q2k_status s, const char* fmt, ...) {
    char msg[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(msg, sizeof msg, fmt, ap);
    va_end(ap);
    q2k::set_last_error(msg);
    return s;
}

// Elements per block and bytes per block of the tensor types whose storage
// size this reader knows (the GGML type numbering a GGUF file uses); 0 = not
// known.  Only the sizes are needed: to bound each tensor's bytes.
struct TypeSize {
    uint32_t block_elems;
    uint32_t block_bytes;
};
TypeSize type_size(uint32_t t) {
    switch (t) {
        case 0: return {1, 4};      // F32
        case 1: return {1, 2};      // F16
        case 2: return {32, 18};    // Q4_0
        case 3: return {32, 20};    // Q4_1
        case 6: return {32, 22};    // Q5_0
        case 7: return {32, 24};    // Q5_1
        case 8: return {32, 34};    // Q8_0
        case 10: return {256, 84};  // Q2_K
        case 11: return {256, 110}; // Q3_K
        case 12: return {256, 144}; // Q4_K
        case 13: return {256, 176}; // Q5_K
        case 14: return {256, 210}; // Q6_K
        case 24: return {1, 1};     // I8
        case 25: return {1, 2};     // I16
        case 26: return {1, 4};     // I32
        case 27: return {1, 8};     // I64
        case 28: return {1, 8};     // F64
        case 30: return {1, 2};     // BF16
        default: return {0, 0};
    }
}

struct Tensor {
    std::string name;
    q2k_gguf_tensor info;
};

// Sequential little-endian reader over the header with bounds on every field.
class Reader {
  public:
    Reader(FILE* f, uint64_t size) : f_(f), size_(size) {}
    uint64_t pos() const { return pos_; }
    bool bytes(void* dst, uint64_t n) {
        if (n > size_ - pos_) return false;
        if (n && fread(dst, 1, n, f_) != n) return false;
        pos_ += n;
        return true;
    }
    bool skip(uint64_t n) {
        if (n > size_ - pos_) return false;
        if (fseeko(f_, static_cast<off_t>(pos_ + n), SEEK_SET) != 0) return false;
        pos_ += n;
        return true;
    }
    bool u32(uint32_t* v) {
        unsigned char b[4];
        if (!bytes(b, 4)) return false;
        *v = uint32_t(b[0]) | uint32_t(b[1]) << 8 | uint32_t(b[2]) << 16 | uint32_t(b[3]) << 24;
        return true;
    }
    bool u64(uint64_t* v) {
        uint32_t lo, hi;
        if (!u32(&lo) || !u32(&hi)) return false;
        *v = uint64_t(lo) | uint64_t(hi) << 32;
        return true;
    }
    bool str(std::string* s) {
        uint64_t n;
        if (!u64(&n) || n > size_ - pos_) return false;
        s->resize(n);
        return bytes(n ? &(*s)[0] : nullptr, n);
    }

  private:
    FILE* f_;
    uint64_t size_;
    uint64_t pos_ = 0;
};

// Bytes of one metadata value of scalar type t (0 for strings and arrays).
uint64_t scalar_bytes(uint32_t t) {
    switch (t) {
        case 0: case 1: case 7: return 1;  // u8, i8, bool
        case 2: case 3: return 2;          // u16, i16
        case 4: case 5: case 6: return 4;  // u32, i32, f32
        case 10: case 11: case 12: return 8;  // u64, i64, f64
        default: return 0;
    }
}

}  // namespace

struct q2k_gguf {
    FILE* file = nullptr;
    uint64_t file_size = 0;
    uint32_t version = 0;
    uint64_t alignment = 32;
    uint64_t data_start = 0;
    std::vector<Tensor> tensors;
    std::unordered_map<std::string, size_t> by_name;
    ~q2k_gguf() {
        if (file) fclose(file);
    }
};

namespace {

// One metadata value of type t: skipped, except general.alignment (read).
q2k_status read_value(Reader& r, q2k_gguf* g, const std::string& key, uint32_t t, int depth) {
    if (t == 8) {  // string
        std::string s;
        if (!r.str(&s)) return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "metadata '%s': truncated string", key.c_str());
        return Q2K_OK;
    }
    if (t == 9) {  // array: element type, count, elements
        uint32_t et;
        uint64_t count;
        if (depth > 0) return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "metadata '%s': nested array", key.c_str());
        if (!r.u32(&et) || !r.u64(&count))
            return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "metadata '%s': truncated array header", key.c_str());
        const uint64_t eb = scalar_bytes(et);
        if (eb) {
            if (count > UINT64_MAX / eb || !r.skip(count * eb))
                return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "metadata '%s': array runs past the file", key.c_str());
            return Q2K_OK;
        }
        if (et != 8) return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "metadata '%s': array of type %u", key.c_str(), et);
        for (uint64_t i = 0; i < count; ++i) {
            q2k_status st = read_value(r, g, key, et, depth + 1);
            if (st != Q2K_OK) return st;
        }
        return Q2K_OK;
    }
    const uint64_t nb = scalar_bytes(t);
    if (nb == 0) return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "metadata '%s': unknown value type %u", key.c_str(), t);
    if (key == "general.alignment") {
        uint32_t a;
        if (t != 4 || !r.u32(&a))
            return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "general.alignment must be a u32 value");
        if (a == 0 || (a & (a - 1)) != 0)
            return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "general.alignment %u is not a power of two", a);
        g->alignment = a;
        return Q2K_OK;
    }
    if (!r.skip(nb)) return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "metadata '%s': truncated value", key.c_str());
    return Q2K_OK;
}

q2k_status parse(q2k_gguf* g) {
    Reader r(g->file, g->file_size);
    char magic[4];
    if (!r.bytes(magic, 4) || memcmp(magic, "GGUF", 4) != 0)
        return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "not a GGUF file (magic)");
    uint64_t n_tensors, n_kv;
    if (!r.u32(&g->version)) return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "truncated header");
    if (g->version != 2 && g->version != 3)
        return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "GGUF version %u (2 and 3 are read)", g->version);
    if (!r.u64(&n_tensors) || !r.u64(&n_kv)) return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "truncated header");
    // every entry takes at least 8 bytes of the file: cheap bound on the counts
    if (n_tensors > g->file_size / 8 || n_kv > g->file_size / 8)
        return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "tensor or metadata count larger than the file");
    for (uint64_t i = 0; i < n_kv; ++i) {
        std::string key;
        uint32_t t;
        if (!r.str(&key) || !r.u32(&t))
            return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "metadata entry %llu truncated", (unsigned long long)i);
        q2k_status st = read_value(r, g, key, t, 0);
        if (st != Q2K_OK) return st;
    }
    g->tensors.resize(n_tensors);
    for (uint64_t i = 0; i < n_tensors; ++i) {
        Tensor& t = g->tensors[i];
        q2k_gguf_tensor& in = t.info;
        memset(&in, 0, sizeof in);
        if (!r.str(&t.name) || !r.u32(&in.n_dims))
            return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "tensor entry %llu truncated", (unsigned long long)i);
        if (in.n_dims < 1 || in.n_dims > 4)
            return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "tensor '%s': %u dimensions (1 to 4)", t.name.c_str(), in.n_dims);
        uint64_t n = 1;
        for (uint32_t d = 0; d < 4; ++d) in.dims[d] = 1;
        for (uint32_t d = 0; d < in.n_dims; ++d) {
            if (!r.u64(&in.dims[d]))
                return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "tensor '%s' truncated", t.name.c_str());
            if (in.dims[d] == 0 || n > UINT64_MAX / in.dims[d])
                return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "tensor '%s': bad extent", t.name.c_str());
            n *= in.dims[d];
        }
        in.n_elements = n;
        if (!r.u32(&in.ggml_type) || !r.u64(&in.offset))
            return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "tensor '%s' truncated", t.name.c_str());
        const TypeSize ts = type_size(in.ggml_type);
        if (ts.block_elems) {
            if (in.dims[0] % ts.block_elems != 0)
                return gguf_fail(Q2K_ERR_INVALID_ARGUMENT,
                                 "tensor '%s': innermost extent %llu is not a multiple of %u (type %u)",
                                 t.name.c_str(), (unsigned long long)in.dims[0], ts.block_elems, in.ggml_type);
            const uint64_t blocks = n / ts.block_elems;
            if (blocks > UINT64_MAX / ts.block_bytes)
                return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "tensor '%s': size overflows", t.name.c_str());
            in.byte_len = blocks * ts.block_bytes;
        }
        if (!g->by_name.emplace(t.name, i).second)
            return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "tensor name '%s' appears twice", t.name.c_str());
    }
    const uint64_t a = g->alignment;
    const uint64_t end = r.pos();
    g->data_start = (end + a - 1) / a * a;
    for (Tensor& t : g->tensors) {
        q2k_gguf_tensor& in = t.info;
        if (in.offset % a != 0)
            return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "tensor '%s': offset %llu is not a multiple of the alignment %llu",
                             t.name.c_str(), (unsigned long long)in.offset, (unsigned long long)a);
        if (in.offset > g->file_size || g->data_start > g->file_size - in.offset ||
            in.byte_len > g->file_size - g->data_start - in.offset)
            return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "tensor '%s': data runs past the end of the file",
                             t.name.c_str());
        in.offset += g->data_start;  // absolute from here on
    }
    return Q2K_OK;
}

}  // namespace

extern "C" {

q2k_status q2k_gguf_open(const char* path, q2k_gguf** out) {
    q2k::set_last_error("");
    if (path == nullptr || out == nullptr)
        return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "path and out must be non-NULL");
    *out = nullptr;
    std::unique_ptr<q2k_gguf> g(new q2k_gguf);
    g->file = fopen(path, "rb");
    if (g->file == nullptr) return gguf_fail(Q2K_ERR_IO, "cannot open '%s'", path);
    if (fseeko(g->file, 0, SEEK_END) != 0) return gguf_fail(Q2K_ERR_IO, "cannot seek '%s'", path);
    const off_t size = ftello(g->file);
    if (size < 0 || fseeko(g->file, 0, SEEK_SET) != 0) return gguf_fail(Q2K_ERR_IO, "cannot size '%s'", path);
    g->file_size = static_cast<uint64_t>(size);
    const q2k_status st = parse(g.get());
    if (st != Q2K_OK) return st;
    *out = g.release();
    return Q2K_OK;
}

void q2k_gguf_close(q2k_gguf* g) { delete g; }

uint64_t q2k_gguf_tensor_count(const q2k_gguf* g) { return g ? g->tensors.size() : 0; }

const char* q2k_gguf_tensor_name(const q2k_gguf* g, uint64_t index) {
    if (g == nullptr || index >= g->tensors.size()) return nullptr;
    return g->tensors[index].name.c_str();
}

q2k_status q2k_gguf_tensor_info(const q2k_gguf* g, const char* name, q2k_gguf_tensor* out) {
    q2k::set_last_error("");
    if (g == nullptr || name == nullptr || out == nullptr)
        return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "file, name and out must be non-NULL");
    auto it = g->by_name.find(name);
    if (it == g->by_name.end()) return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "no tensor named '%s'", name);
    *out = g->tensors[it->second].info;
    return Q2K_OK;
}

q2k_status q2k_gguf_read_tensor(const q2k_gguf* g, const char* name, void* dst, size_t dst_bytes) {
    q2k_gguf_tensor in;
    q2k_status st = q2k_gguf_tensor_info(g, name, &in);
    if (st != Q2K_OK) return st;
    if (in.byte_len == 0)
        return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "tensor '%s' has type %u, whose size this reader does not know",
                         name, in.ggml_type);
    if (dst == nullptr || dst_bytes != in.byte_len)
        return gguf_fail(Q2K_ERR_INVALID_ARGUMENT, "tensor '%s' has %llu bytes; dst has %zu", name,
                         (unsigned long long)in.byte_len, dst_bytes);
    if (fseeko(g->file, static_cast<off_t>(in.offset), SEEK_SET) != 0 ||
        fread(dst, 1, dst_bytes, g->file) != dst_bytes)
        return gguf_fail(Q2K_ERR_IO, "reading tensor '%s' failed", name);
    return Q2K_OK;
}

}  // extern "C"
