// gq_gguf.cu -- the GGUF reader of include/gq_gguf.h (host code only).
//
// The file is memory-mapped read-only ("Development Guide for Small AI Models (TinyLLaMA,
// etc.) Using C++", section 3.1) and parsed once at open into tables of metadata entries
// and tensor infos (section 3.2 gives the structure; the published GGUF specification the
// field widths). The parser reads through a cursor that refuses any read past the end of
// the mapping, so a truncated or malformed file ends in GQ_ERR_FORMAT and nothing reads
// outside the file. Tensor data is never copied on the host: gq_gguf_tensor_data points
// into the mapping, and gq_gguf_upload copies from there straight to the device.
#include <fcntl.h>
#include <sys/mman.h>
#include <sys/stat.h>
#include <unistd.h>

#include <climits>
#include <cstring>
#include <string>
#include <vector>

#include <cuda_runtime.h>

#include "gq_gguf.h"
#include "gq_internal.h"

namespace {

constexpr uint32_t kMagic = 0x46554747u;   // "GGUF" read as a little-endian uint32
constexpr uint64_t kDefaultAlignment = 32;
constexpr int kMaxDims = 4;
constexpr int kMaxNesting = 8;             // arrays of arrays, at most this deep

struct Kv {
    std::string key;
    uint32_t type;
    uint64_t value;   // file offset of the value (after its type)
};

struct Tensor {
    std::string name;
    uint32_t n_dims;
    uint32_t type;
    int64_t ne[kMaxDims];
    uint64_t rel;      // offset from the start of the data section
    uint64_t offset;   // offset from the start of the file
    uint64_t nbytes;   // 0 for a type of unknown size
};

// Bytes per block and elements per block of the ggml data types whose size is known here.
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
        case 9: return {32, 36};    // Q8_1
        case 10: return {256, 84};  // Q2_K
        case 11: return {256, 110}; // Q3_K
        case 12: return {256, 144}; // Q4_K
        case 13: return {256, 176}; // Q5_K
        case 14: return {256, 210}; // Q6_K
        case 15: return {256, 292}; // Q8_K
        case 24: return {1, 1};     // I8
        case 25: return {1, 2};     // I16
        case 26: return {1, 4};     // I32
        case 27: return {1, 8};     // I64
        case 28: return {1, 8};     // F64
        case 30: return {1, 2};     // BF16
        default: return {0, 0};
    }
}

// Size of a fixed-size metadata value type, 0 for string, array and unknown types.
int fixed_size(uint32_t t) {
    switch (t) {
        case GQ_GGUF_UINT8: case GQ_GGUF_INT8: case GQ_GGUF_BOOL: return 1;
        case GQ_GGUF_UINT16: case GQ_GGUF_INT16: return 2;
        case GQ_GGUF_UINT32: case GQ_GGUF_INT32: case GQ_GGUF_FLOAT32: return 4;
        case GQ_GGUF_UINT64: case GQ_GGUF_INT64: case GQ_GGUF_FLOAT64: return 8;
        default: return 0;
    }
}

// Cursor over the mapping. Invariant: pos <= size. Once a read would pass the end, ok
// turns false and every later read returns zero without moving.
struct Reader {
    const uint8_t* base;
    uint64_t size;
    uint64_t pos = 0;
    bool ok = true;

    bool need(uint64_t n) {
        if (!ok || n > size - pos) ok = false;
        return ok;
    }
    uint32_t u32() {
        uint32_t v = 0;
        if (need(4)) {
            std::memcpy(&v, base + pos, 4);
            pos += 4;
        }
        return v;
    }
    uint64_t u64() {
        uint64_t v = 0;
        if (need(8)) {
            std::memcpy(&v, base + pos, 8);
            pos += 8;
        }
        return v;
    }
    bool skip(uint64_t n) {
        if (need(n)) pos += n;
        return ok;
    }
    // A length-prefixed string: its bytes start at *off and run for *len.
    bool str(uint64_t* off, uint64_t* len) {
        const uint64_t n = u64();
        if (!need(n)) return false;
        *off = pos;
        *len = n;
        pos += n;
        return true;
    }
};

bool skip_value(Reader& r, uint32_t t, int depth) {
    const int fs = fixed_size(t);
    if (fs) return r.skip(fs);
    if (t == GQ_GGUF_STRING) {
        uint64_t off, len;
        return r.str(&off, &len);
    }
    if (t != GQ_GGUF_ARRAY || depth >= kMaxNesting) return r.ok = false;
    const uint32_t et = r.u32();
    const uint64_t n = r.u64();
    if (!r.ok) return false;
    const int efs = fixed_size(et);
    if (efs) {
        if (n > (r.size - r.pos) / static_cast<uint64_t>(efs)) return r.ok = false;
        return r.skip(n * static_cast<uint64_t>(efs));
    }
    if (et != GQ_GGUF_STRING && et != GQ_GGUF_ARRAY) return r.ok = false;
    // every element takes at least 8 bytes (a length or an array header), so the loop ends
    // within the file's size
    for (uint64_t k = 0; k < n && r.ok; ++k) skip_value(r, et, depth + 1);
    return r.ok;
}

bool mul_ok(uint64_t a, uint64_t b, uint64_t* out) {
    if (a != 0 && b > UINT64_MAX / a) return false;
    *out = a * b;
    return true;
}

}  // namespace

struct gq_gguf {
    int fd = -1;
    const uint8_t* map = nullptr;
    uint64_t size = 0;
    uint32_t version = 0;
    uint64_t alignment = kDefaultAlignment;
    uint64_t data_off = 0;
    std::vector<Kv> kv;
    std::vector<Tensor> tensors;
};

namespace {

gq_status parse(gq_gguf* f) {
    Reader r{f->map, f->size};
    if (r.u32() != kMagic || !r.ok) return GQ_ERR_FORMAT;
    f->version = r.u32();
    if (!r.ok || (f->version != 2 && f->version != 3)) return GQ_ERR_FORMAT;
    const uint64_t n_tensors = r.u64();
    const uint64_t n_kv = r.u64();
    if (!r.ok) return GQ_ERR_FORMAT;
    // every entry takes at least 12 bytes and every tensor info at least 24: bound the
    // counts by what the file could hold before reserving anything
    if (n_kv > f->size / 12 || n_tensors > f->size / 24) return GQ_ERR_FORMAT;
    f->kv.reserve(n_kv);
    for (uint64_t i = 0; i < n_kv; ++i) {
        uint64_t koff, klen;
        if (!r.str(&koff, &klen)) return GQ_ERR_FORMAT;
        Kv e;
        e.key.assign(reinterpret_cast<const char*>(f->map + koff), klen);
        e.type = r.u32();
        e.value = r.pos;
        if (!r.ok || !skip_value(r, e.type, 0)) return GQ_ERR_FORMAT;
        if (e.key == "general.alignment") {
            if (e.type != GQ_GGUF_UINT32) return GQ_ERR_FORMAT;
            uint32_t a;
            std::memcpy(&a, f->map + e.value, 4);
            if (a == 0 || (a & (a - 1)) != 0) return GQ_ERR_FORMAT;
            f->alignment = a;
        }
        f->kv.push_back(std::move(e));
    }
    f->tensors.reserve(n_tensors);
    for (uint64_t i = 0; i < n_tensors; ++i) {
        uint64_t noff, nlen;
        if (!r.str(&noff, &nlen)) return GQ_ERR_FORMAT;
        Tensor t;
        t.name.assign(reinterpret_cast<const char*>(f->map + noff), nlen);
        t.n_dims = r.u32();
        if (!r.ok || t.n_dims < 1 || t.n_dims > kMaxDims) return GQ_ERR_FORMAT;
        uint64_t nelem = 1;
        for (int d = 0; d < kMaxDims; ++d) {
            uint64_t e = 1;
            if (d < static_cast<int>(t.n_dims)) e = r.u64();
            if (!r.ok || e > static_cast<uint64_t>(INT64_MAX) || !mul_ok(nelem, e, &nelem))
                return GQ_ERR_FORMAT;
            t.ne[d] = static_cast<int64_t>(e);
        }
        if (nelem > static_cast<uint64_t>(INT64_MAX)) return GQ_ERR_FORMAT;
        t.type = r.u32();
        t.rel = r.u64();
        if (!r.ok) return GQ_ERR_FORMAT;
        const TypeSize ts = type_size(t.type);
        t.nbytes = 0;
        if (ts.block_elems) {
            if (t.ne[0] % ts.block_elems != 0) return GQ_ERR_FORMAT;   // whole blocks per row
            if (!mul_ok(nelem / ts.block_elems, ts.block_bytes, &t.nbytes)) return GQ_ERR_FORMAT;
        }
        f->tensors.push_back(std::move(t));
    }
    // The data section starts at the first multiple of the alignment after the infos.
    const uint64_t a = f->alignment;
    if (r.pos > UINT64_MAX - (a - 1)) return GQ_ERR_FORMAT;
    f->data_off = (r.pos + a - 1) / a * a;
    for (Tensor& t : f->tensors) {
        if (t.rel % a != 0) return GQ_ERR_FORMAT;
        if (f->data_off > f->size || t.rel > f->size - f->data_off) return GQ_ERR_FORMAT;
        t.offset = f->data_off + t.rel;
        if (t.nbytes > f->size - t.offset) return GQ_ERR_FORMAT;
    }
    return GQ_OK;
}

bool bad_tensor(const gq_gguf* f, int64_t i) {
    return f == nullptr || i < 0 || i >= static_cast<int64_t>(f->tensors.size());
}

bool bad_kv(const gq_gguf* f, int64_t i) {
    return f == nullptr || i < 0 || i >= static_cast<int64_t>(f->kv.size());
}

}  // namespace

extern "C" {

gq_status gq_gguf_open(const char* path, gq_gguf** out) {
    if (!path || !out) return GQ_ERR_NULL;
    *out = nullptr;
    const int fd = ::open(path, O_RDONLY | O_CLOEXEC);
    if (fd < 0) return GQ_ERR_IO;
    struct stat st;
    if (::fstat(fd, &st) != 0 || !S_ISREG(st.st_mode)) {
        ::close(fd);
        return GQ_ERR_IO;
    }
    if (st.st_size < 24) {   // smaller than the header
        ::close(fd);
        return GQ_ERR_FORMAT;
    }
    void* m = ::mmap(nullptr, static_cast<size_t>(st.st_size), PROT_READ, MAP_PRIVATE, fd, 0);
    if (m == MAP_FAILED) {
        ::close(fd);
        return GQ_ERR_IO;
    }
    gq_gguf* f = new gq_gguf;
    f->fd = fd;
    f->map = static_cast<const uint8_t*>(m);
    f->size = static_cast<uint64_t>(st.st_size);
    const gq_status s = parse(f);
    if (s != GQ_OK) {
        gq_gguf_close(f);
        return s;
    }
    *out = f;
    return GQ_OK;
}

void gq_gguf_close(gq_gguf* f) {
    if (!f) return;
    if (f->map) ::munmap(const_cast<uint8_t*>(f->map), static_cast<size_t>(f->size));
    if (f->fd >= 0) ::close(f->fd);
    delete f;
}

uint32_t gq_gguf_version(const gq_gguf* f) { return f ? f->version : 0; }

int64_t gq_gguf_tensor_count(const gq_gguf* f) {
    return f ? static_cast<int64_t>(f->tensors.size()) : 0;
}

int64_t gq_gguf_kv_count(const gq_gguf* f) { return f ? static_cast<int64_t>(f->kv.size()) : 0; }

uint64_t gq_gguf_alignment(const gq_gguf* f) { return f ? f->alignment : 0; }

gq_status gq_gguf_tensor_info(const gq_gguf* f, int64_t i, gq_gguf_tensor* out) {
    if (!f || !out) return GQ_ERR_NULL;
    if (bad_tensor(f, i)) return GQ_ERR_SHAPE;
    const Tensor& t = f->tensors[static_cast<size_t>(i)];
    out->name = t.name.c_str();
    out->n_dims = t.n_dims;
    out->type = t.type;
    for (int d = 0; d < kMaxDims; ++d) out->ne[d] = t.ne[d];
    out->offset = t.offset;
    out->nbytes = t.nbytes;
    return GQ_OK;
}

int64_t gq_gguf_find_tensor(const gq_gguf* f, const char* name) {
    if (!f || !name) return -1;
    for (size_t i = 0; i < f->tensors.size(); ++i)
        if (f->tensors[i].name == name) return static_cast<int64_t>(i);
    return -1;
}

const void* gq_gguf_tensor_data(const gq_gguf* f, int64_t i) {
    if (bad_tensor(f, i)) return nullptr;
    return f->map + f->tensors[static_cast<size_t>(i)].offset;
}

gq_status gq_gguf_tensor_matrix(const gq_gguf* f, int64_t i, gq_type* type, int64_t* M,
                                int64_t* K) {
    if (!f || !type || !M || !K) return GQ_ERR_NULL;
    if (bad_tensor(f, i)) return GQ_ERR_SHAPE;
    const Tensor& t = f->tensors[static_cast<size_t>(i)];
    const gq_type gt = static_cast<gq_type>(t.type);   // the three block ids coincide
    if (gq::block_bytes_of(gt) == 0) return GQ_ERR_TYPE;
    if (t.ne[2] != 1 || t.ne[3] != 1) return GQ_ERR_SHAPE;
    *type = gt;
    *K = t.ne[0];
    *M = t.ne[1];
    return GQ_OK;
}

gq_status gq_gguf_upload(const gq_gguf* f, int64_t i, void* dst, size_t dst_bytes,
                         void* stream) {
    if (!f || !dst) return GQ_ERR_NULL;
    if (bad_tensor(f, i)) return GQ_ERR_SHAPE;
    const Tensor& t = f->tensors[static_cast<size_t>(i)];
    if (type_size(t.type).block_elems == 0 || dst_bytes < t.nbytes) return GQ_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(dst) % 16 != 0) return GQ_ERR_ALIGN;
    if (t.nbytes == 0) return GQ_OK;
    const cudaError_t e = cudaMemcpyAsync(dst, f->map + t.offset, t.nbytes,
                                          cudaMemcpyHostToDevice,
                                          static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GQ_OK : GQ_ERR_CUDA;
}

int64_t gq_gguf_find_key(const gq_gguf* f, const char* key) {
    if (!f || !key) return -1;
    for (size_t i = 0; i < f->kv.size(); ++i)
        if (f->kv[i].key == key) return static_cast<int64_t>(i);
    return -1;
}

const char* gq_gguf_kv_key(const gq_gguf* f, int64_t i) {
    return bad_kv(f, i) ? nullptr : f->kv[static_cast<size_t>(i)].key.c_str();
}

int32_t gq_gguf_kv_type(const gq_gguf* f, int64_t i) {
    return bad_kv(f, i) ? -1 : static_cast<int32_t>(f->kv[static_cast<size_t>(i)].type);
}

gq_status gq_gguf_kv_int(const gq_gguf* f, int64_t i, int64_t* out) {
    if (!f || !out) return GQ_ERR_NULL;
    if (bad_kv(f, i)) return GQ_ERR_SHAPE;
    const Kv& e = f->kv[static_cast<size_t>(i)];
    const uint8_t* v = f->map + e.value;
    switch (e.type) {
        case GQ_GGUF_UINT8: *out = *v; return GQ_OK;
        case GQ_GGUF_INT8: *out = static_cast<int8_t>(*v); return GQ_OK;
        case GQ_GGUF_BOOL: *out = *v != 0; return GQ_OK;
        case GQ_GGUF_UINT16: { uint16_t x; std::memcpy(&x, v, 2); *out = x; return GQ_OK; }
        case GQ_GGUF_INT16: { int16_t x; std::memcpy(&x, v, 2); *out = x; return GQ_OK; }
        case GQ_GGUF_UINT32: { uint32_t x; std::memcpy(&x, v, 4); *out = x; return GQ_OK; }
        case GQ_GGUF_INT32: { int32_t x; std::memcpy(&x, v, 4); *out = x; return GQ_OK; }
        case GQ_GGUF_INT64: { int64_t x; std::memcpy(&x, v, 8); *out = x; return GQ_OK; }
        case GQ_GGUF_UINT64: {
            uint64_t x;
            std::memcpy(&x, v, 8);
            if (x > static_cast<uint64_t>(INT64_MAX)) return GQ_ERR_SHAPE;
            *out = static_cast<int64_t>(x);
            return GQ_OK;
        }
        default: return GQ_ERR_TYPE;
    }
}

gq_status gq_gguf_kv_float(const gq_gguf* f, int64_t i, double* out) {
    if (!f || !out) return GQ_ERR_NULL;
    if (bad_kv(f, i)) return GQ_ERR_SHAPE;
    const Kv& e = f->kv[static_cast<size_t>(i)];
    if (e.type == GQ_GGUF_FLOAT32) {
        float x;
        std::memcpy(&x, f->map + e.value, 4);
        *out = x;
        return GQ_OK;
    }
    if (e.type == GQ_GGUF_FLOAT64) {
        std::memcpy(out, f->map + e.value, 8);
        return GQ_OK;
    }
    return GQ_ERR_TYPE;
}

gq_status gq_gguf_kv_string(const gq_gguf* f, int64_t i, const char** data, uint64_t* len) {
    if (!f || !data || !len) return GQ_ERR_NULL;
    if (bad_kv(f, i)) return GQ_ERR_SHAPE;
    const Kv& e = f->kv[static_cast<size_t>(i)];
    if (e.type != GQ_GGUF_STRING) return GQ_ERR_TYPE;
    std::memcpy(len, f->map + e.value, 8);
    *data = reinterpret_cast<const char*>(f->map + e.value + 8);
    return GQ_OK;
}

gq_status gq_gguf_kv_array(const gq_gguf* f, int64_t i, uint32_t* elem_type, uint64_t* count,
                           const void** data) {
    if (!f || !elem_type || !count || !data) return GQ_ERR_NULL;
    if (bad_kv(f, i)) return GQ_ERR_SHAPE;
    const Kv& e = f->kv[static_cast<size_t>(i)];
    if (e.type != GQ_GGUF_ARRAY) return GQ_ERR_TYPE;
    std::memcpy(elem_type, f->map + e.value, 4);
    std::memcpy(count, f->map + e.value + 4, 8);
    *data = f->map + e.value + 12;
    return GQ_OK;
}

}  // extern "C"
