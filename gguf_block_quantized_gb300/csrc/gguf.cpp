// gguf.cpp — GGUF container: a memory-mapped reader and an in-memory writer (host code).
//
// Layout ("The GGML ecosystem, and where synapse fits", section 2, the GGUF diagram; "ggml
// Documentation", GGUF specification, "File Structure" and general.alignment; "llama.cpp
// and GGUF", "Tensor info, alignment, and mmap"), little-endian:
//   header      "GGUF", version u32 (3), n_tensors u64, n_kv u64
//   metadata    n_kv x { key: string, value type: u32, value }
//   tensor info n_tensors x { name: string, n_dims: u32, ne: u64[n_dims] (innermost first),
//               type: u32, offset: u64 }
//   padding     zeros up to a multiple of general.alignment (u32 key; 32 when absent;
//               a multiple of 8)
//   data        each tensor at data_start + offset, offset a multiple of the alignment
// A string is a u64 byte count and the bytes, without terminator; an array value is its
// element type (u32), its length (u64) and the elements, packed.  The numeric codes of the
// value types and of the tensor element types follow the public GGUF specification: the
// pages name the types but print no codes.
#include <fcntl.h>
#include <stdint.h>
#include <string.h>
#include <sys/mman.h>
#include <sys/stat.h>
#include <unistd.h>

#include <cuda_runtime.h>

#include <cstdio>
#include <set>
#include <string>
#include <vector>

#include "syn.h"

static_assert(__BYTE_ORDER__ == __ORDER_LITTLE_ENDIAN__, "fields are read with memcpy: a little-endian host");

namespace {

int64_t scalar_size(uint32_t t) {
    switch (t) {
    case SYN_GGUF_UINT8: case SYN_GGUF_INT8: case SYN_GGUF_BOOL: return 1;
    case SYN_GGUF_UINT16: case SYN_GGUF_INT16: return 2;
    case SYN_GGUF_UINT32: case SYN_GGUF_INT32: case SYN_GGUF_FLOAT32: return 4;
    case SYN_GGUF_UINT64: case SYN_GGUF_INT64: case SYN_GGUF_FLOAT64: return 8;
    default: return -1;
    }
}

// Tensor element types whose storage this reader can size: the block formats of the
// format table, F16, and the two plain float types the pages name beside them.
struct GType {
    uint32_t ggml;
    int syn;  // the library's format code; -1 where mul_mat does not take the type
    int64_t elems, bytes;
};
constexpr GType kTypes[] = {
    {SYN_GGML_F32, -1, 1, 4},
    {SYN_GGML_F16, SYN_TYPE_F16, 1, 2},
    {SYN_GGML_Q4_0, SYN_TYPE_Q4_0, 32, 18},
    {SYN_GGML_Q5_0, SYN_TYPE_Q5_0, 32, 22},
    {SYN_GGML_Q8_0, SYN_TYPE_Q8_0, 32, 34},
    {SYN_GGML_Q4_K, SYN_TYPE_Q4_K, 256, 144},
    {SYN_GGML_Q6_K, SYN_TYPE_Q6_K, 256, 210},
    {SYN_GGML_Q8_K, SYN_TYPE_Q8_K, 256, 292},
    {SYN_GGML_BF16, -1, 1, 2},
};

const GType* find_type(uint32_t ggml) {
    for (const GType& t : kTypes)
        if (t.ggml == ggml) return &t;
    return nullptr;
}

struct KV {
    std::string key;
    uint32_t type = 0;
    uint32_t arr_type = 0;
    uint64_t arr_n = 0;
    const uint8_t* val = nullptr;  // scalar bytes, string bytes, or the first array element
    uint64_t str_len = 0;
};

struct Tensor {
    std::string name;
    uint32_t n_dims = 0;
    int64_t ne[4] = {1, 1, 1, 1};
    uint32_t ggml_type = 0;
    uint64_t offset = 0;
    int64_t nbytes = -1;  // -1: an element type this reader cannot size
};

// Bounded cursor over the mapping: every read checks the remaining length first.
struct Cursor {
    const uint8_t* p;
    uint64_t n, at = 0;
    bool ok = true;
    bool take(uint64_t k) {
        if (!ok || k > n - at) ok = false;
        return ok;
    }
    uint32_t u32() {
        uint32_t v = 0;
        if (take(4)) { memcpy(&v, p + at, 4); at += 4; }
        return v;
    }
    uint64_t u64() {
        uint64_t v = 0;
        if (take(8)) { memcpy(&v, p + at, 8); at += 8; }
        return v;
    }
    // a string: its bytes (in the mapping) and length, or NULL past the end
    const uint8_t* str(uint64_t* len) {
        const uint64_t l = u64();
        if (!take(l)) return nullptr;
        const uint8_t* s = p + at;
        at += l;
        *len = l;
        return s;
    }
    bool skip(uint64_t k) {
        if (take(k)) at += k;
        return ok;
    }
};

constexpr uint64_t kMaxCount = uint64_t(1) << 32;  // entry counts and array lengths accepted

}  // namespace

struct syn_gguf {
    int fd = -1;
    const uint8_t* base = nullptr;
    uint64_t size = 0;
    uint32_t version = 0;
    uint64_t alignment = 32;
    uint64_t data_start = 0;
    std::vector<KV> kv;
    std::vector<Tensor> tensors;
};

struct syn_gguf_writer {
    std::string path;
    uint32_t alignment = 32;
    uint64_t n_kv = 0, n_tensors = 0;
    std::vector<uint8_t> kv, info, data;  // serialised metadata, tensor info, tensor data
    std::set<std::string> keys, names;
};

namespace {

int parse(syn_gguf* g) {
    Cursor c{g->base, g->size};
    if (!c.take(4) || memcmp(g->base, "GGUF", 4) != 0) return SYN_ERR_FORMAT;
    c.at = 4;
    g->version = c.u32();
    // version 2 has the field widths of version 3, which only added big-endian files
    if (!c.ok || (g->version != 2 && g->version != 3)) return SYN_ERR_FORMAT;
    const uint64_t n_tensors = c.u64(), n_kv = c.u64();
    if (!c.ok || n_tensors > kMaxCount || n_kv > kMaxCount) return SYN_ERR_FORMAT;

    std::set<std::string> seen;
    for (uint64_t i = 0; i < n_kv; i++) {
        KV e;
        uint64_t len = 0;
        const uint8_t* k = c.str(&len);
        if (!k) return SYN_ERR_FORMAT;
        e.key.assign(reinterpret_cast<const char*>(k), (size_t)len);
        e.type = c.u32();
        if (!c.ok) return SYN_ERR_FORMAT;
        if (e.type == SYN_GGUF_STRING) {
            e.val = c.str(&e.str_len);
            if (!e.val) return SYN_ERR_FORMAT;
        } else if (e.type == SYN_GGUF_ARRAY) {
            e.arr_type = c.u32();
            e.arr_n = c.u64();
            if (!c.ok || e.arr_n > kMaxCount) return SYN_ERR_FORMAT;
            e.val = g->base + c.at;
            if (e.arr_type == SYN_GGUF_STRING) {
                for (uint64_t j = 0; j < e.arr_n; j++)
                    if (!c.str(&len)) return SYN_ERR_FORMAT;
            } else {
                const int64_t sz = scalar_size(e.arr_type);  // arrays of arrays are not read
                if (sz < 0 || !c.skip(e.arr_n * (uint64_t)sz)) return SYN_ERR_FORMAT;
            }
        } else {
            const int64_t sz = scalar_size(e.type);
            if (sz < 0) return SYN_ERR_FORMAT;
            e.val = g->base + c.at;
            if (!c.skip((uint64_t)sz)) return SYN_ERR_FORMAT;
        }
        if (!seen.insert(e.key).second) return SYN_ERR_FORMAT;  // keys are unique
        if (e.key == "general.alignment") {
            if (e.type != SYN_GGUF_UINT32) return SYN_ERR_FORMAT;
            uint32_t a;
            memcpy(&a, e.val, 4);
            if (a == 0 || a % 8) return SYN_ERR_FORMAT;
            g->alignment = a;
        }
        g->kv.push_back(std::move(e));
    }

    seen.clear();
    for (uint64_t i = 0; i < n_tensors; i++) {
        Tensor t;
        uint64_t len = 0;
        const uint8_t* nm = c.str(&len);
        if (!nm) return SYN_ERR_FORMAT;
        t.name.assign(reinterpret_cast<const char*>(nm), (size_t)len);
        t.n_dims = c.u32();
        if (!c.ok || t.n_dims < 1 || t.n_dims > 4) return SYN_ERR_FORMAT;
        uint64_t count = 1;
        for (uint32_t d = 0; d < t.n_dims; d++) {
            const uint64_t v = c.u64();
            if (!c.ok || v == 0 || v > (uint64_t(1) << 40) || count > (uint64_t(1) << 50) / v) return SYN_ERR_FORMAT;
            t.ne[d] = (int64_t)v;
            count *= v;
        }
        t.ggml_type = c.u32();
        t.offset = c.u64();
        if (!c.ok) return SYN_ERR_FORMAT;
        if (const GType* gt = find_type(t.ggml_type)) {
            if (t.ne[0] % gt->elems) return SYN_ERR_FORMAT;  // rows are whole blocks
            t.nbytes = (int64_t)(count / (uint64_t)gt->elems) * gt->bytes;
        }
        if (!seen.insert(t.name).second) return SYN_ERR_FORMAT;  // names are unique
        g->tensors.push_back(std::move(t));
    }

    g->data_start = (c.at + g->alignment - 1) / g->alignment * g->alignment;
    for (const Tensor& t : g->tensors) {
        if (t.offset % g->alignment) return SYN_ERR_FORMAT;
        if (t.nbytes >= 0 && (g->data_start > g->size || t.offset > g->size - g->data_start ||
                              (uint64_t)t.nbytes > g->size - g->data_start - t.offset))
            return SYN_ERR_FORMAT;
    }
    return SYN_OK;
}

const KV* find_kv(const syn_gguf* g, const char* key) {
    for (const KV& e : g->kv)
        if (e.key == key) return &e;
    return nullptr;
}

const Tensor* tensor_at(const syn_gguf* g, int64_t i) {
    if (i < 0 || i >= (int64_t)g->tensors.size()) return nullptr;
    return &g->tensors[(size_t)i];
}

void put(std::vector<uint8_t>& v, const void* p, size_t n) {
    const uint8_t* b = static_cast<const uint8_t*>(p);
    v.insert(v.end(), b, b + n);
}
void put_u32(std::vector<uint8_t>& v, uint32_t x) { put(v, &x, 4); }
void put_u64(std::vector<uint8_t>& v, uint64_t x) { put(v, &x, 8); }
void put_str(std::vector<uint8_t>& v, const char* s, uint64_t n) {
    put_u64(v, n);
    if (n) put(v, s, (size_t)n);
}

// starts a metadata entry; rejects a NULL writer or key and a repeated key
int kv_head(syn_gguf_writer* w, const char* key, uint32_t type) {
    if (!w || !key) return SYN_ERR_NULL;
    if (!w->keys.insert(key).second) return SYN_ERR_SHAPE;
    put_str(w->kv, key, strlen(key));
    put_u32(w->kv, type);
    w->n_kv++;
    return SYN_OK;
}

}  // namespace

extern "C" {

syn_gguf* syn_gguf_open(const char* path, int* status) {
    int st = SYN_OK;
    syn_gguf* g = nullptr;
    if (!path) {
        st = SYN_ERR_NULL;
    } else {
        const int fd = open(path, O_RDONLY | O_CLOEXEC);
        struct stat sb;
        if (fd < 0) {
            st = SYN_ERR_IO;
        } else if (fstat(fd, &sb) != 0) {
            close(fd);
            st = SYN_ERR_IO;
        } else if (sb.st_size < 24) {
            close(fd);
            st = SYN_ERR_FORMAT;
        } else {
            void* m = mmap(nullptr, (size_t)sb.st_size, PROT_READ, MAP_PRIVATE, fd, 0);
            if (m == MAP_FAILED) {
                close(fd);
                st = SYN_ERR_IO;
            } else {
                g = new syn_gguf();
                g->fd = fd;
                g->base = static_cast<const uint8_t*>(m);
                g->size = (uint64_t)sb.st_size;
                st = parse(g);
                if (st != SYN_OK) {
                    syn_gguf_close(g);
                    g = nullptr;
                }
            }
        }
    }
    if (status) *status = st;
    return g;
}

void syn_gguf_close(syn_gguf* g) {
    if (!g) return;
    if (g->base) munmap(const_cast<uint8_t*>(g->base), (size_t)g->size);
    if (g->fd >= 0) close(g->fd);
    delete g;
}

int64_t syn_gguf_version(const syn_gguf* g) { return g ? (int64_t)g->version : -1; }
int64_t syn_gguf_n_tensors(const syn_gguf* g) { return g ? (int64_t)g->tensors.size() : -1; }
int64_t syn_gguf_n_kv(const syn_gguf* g) { return g ? (int64_t)g->kv.size() : -1; }
int64_t syn_gguf_alignment(const syn_gguf* g) { return g ? (int64_t)g->alignment : -1; }
int64_t syn_gguf_data_start(const syn_gguf* g) { return g ? (int64_t)g->data_start : -1; }

int64_t syn_gguf_find_tensor(const syn_gguf* g, const char* name) {
    if (!g || !name) return -1;
    for (size_t i = 0; i < g->tensors.size(); i++)
        if (g->tensors[i].name == name) return (int64_t)i;
    return -1;
}

int syn_gguf_tensor_info(const syn_gguf* g, int64_t i, const char** name, uint32_t* ggml_type, int* n_dims,
                         int64_t* ne, uint64_t* offset, const void** data, int64_t* nbytes) {
    if (!g) return SYN_ERR_NULL;
    const Tensor* t = tensor_at(g, i);
    if (!t) return SYN_ERR_NOTFOUND;
    if (name) *name = t->name.c_str();
    if (ggml_type) *ggml_type = t->ggml_type;
    if (n_dims) *n_dims = (int)t->n_dims;
    if (ne)
        for (int d = 0; d < 4; d++) ne[d] = t->ne[d];
    if (offset) *offset = t->offset;
    if (nbytes) *nbytes = t->nbytes;
    if (data) *data = t->nbytes >= 0 ? g->base + g->data_start + t->offset : nullptr;
    return SYN_OK;
}

int syn_gguf_matrix(const syn_gguf* g, const char* name, int* type, int64_t* n_out, int64_t* n_in,
                    const void** data, int64_t* nbytes) {
    if (!g || !name) return SYN_ERR_NULL;
    const int64_t i = syn_gguf_find_tensor(g, name);
    if (i < 0) return SYN_ERR_NOTFOUND;
    const Tensor& t = g->tensors[(size_t)i];
    const GType* gt = find_type(t.ggml_type);
    if (!gt || gt->syn < 0 || gt->syn == SYN_TYPE_Q8_K) return SYN_ERR_TYPE;
    if (type) *type = gt->syn;
    if (n_in) *n_in = t.ne[0];
    if (n_out) *n_out = t.ne[1] * t.ne[2] * t.ne[3];
    if (data) *data = g->base + g->data_start + t.offset;
    if (nbytes) *nbytes = t.nbytes;
    return SYN_OK;
}

int syn_gguf_upload(const syn_gguf* g, int64_t i, void* dst, int64_t dst_bytes, syn_stream_t stream) {
    if (!g || !dst) return SYN_ERR_NULL;
    const Tensor* t = tensor_at(g, i);
    if (!t) return SYN_ERR_NOTFOUND;
    if (t->nbytes < 0) return SYN_ERR_TYPE;
    if (dst_bytes < t->nbytes) return SYN_ERR_SHAPE;
    const cudaError_t e = cudaMemcpyAsync(dst, g->base + g->data_start + t->offset, (size_t)t->nbytes,
                                          cudaMemcpyHostToDevice, (cudaStream_t)stream);
    return e == cudaSuccess ? SYN_OK : SYN_ERR_CUDA;
}

int syn_gguf_kv_info(const syn_gguf* g, int64_t i, const char** key, uint32_t* value_type, uint32_t* elem_type,
                     uint64_t* n_elems) {
    if (!g) return SYN_ERR_NULL;
    if (i < 0 || i >= (int64_t)g->kv.size()) return SYN_ERR_NOTFOUND;
    const KV& e = g->kv[(size_t)i];
    if (key) *key = e.key.c_str();
    if (value_type) *value_type = e.type;
    if (elem_type) *elem_type = e.type == SYN_GGUF_ARRAY ? e.arr_type : 0;
    if (n_elems) *n_elems = e.type == SYN_GGUF_ARRAY ? e.arr_n : 0;
    return SYN_OK;
}

int syn_gguf_get_int(const syn_gguf* g, const char* key, int64_t* out) {
    if (!g || !key || !out) return SYN_ERR_NULL;
    const KV* e = find_kv(g, key);
    if (!e) return SYN_ERR_NOTFOUND;
    const uint8_t* v = e->val;
    switch (e->type) {
    case SYN_GGUF_UINT8: *out = *v; return SYN_OK;
    case SYN_GGUF_INT8: *out = (int8_t)*v; return SYN_OK;
    case SYN_GGUF_BOOL: *out = *v != 0; return SYN_OK;
    case SYN_GGUF_UINT16: { uint16_t x; memcpy(&x, v, 2); *out = x; return SYN_OK; }
    case SYN_GGUF_INT16: { int16_t x; memcpy(&x, v, 2); *out = x; return SYN_OK; }
    case SYN_GGUF_UINT32: { uint32_t x; memcpy(&x, v, 4); *out = x; return SYN_OK; }
    case SYN_GGUF_INT32: { int32_t x; memcpy(&x, v, 4); *out = x; return SYN_OK; }
    case SYN_GGUF_INT64: { int64_t x; memcpy(&x, v, 8); *out = x; return SYN_OK; }
    case SYN_GGUF_UINT64: {
        uint64_t x;
        memcpy(&x, v, 8);
        if (x > (uint64_t)INT64_MAX) return SYN_ERR_RANGE;
        *out = (int64_t)x;
        return SYN_OK;
    }
    default: return SYN_ERR_TYPE;
    }
}

int syn_gguf_get_float(const syn_gguf* g, const char* key, double* out) {
    if (!g || !key || !out) return SYN_ERR_NULL;
    const KV* e = find_kv(g, key);
    if (!e) return SYN_ERR_NOTFOUND;
    if (e->type == SYN_GGUF_FLOAT32) { float x; memcpy(&x, e->val, 4); *out = x; return SYN_OK; }
    if (e->type == SYN_GGUF_FLOAT64) { memcpy(out, e->val, 8); return SYN_OK; }
    return SYN_ERR_TYPE;
}

int syn_gguf_get_string(const syn_gguf* g, const char* key, const char** bytes, int64_t* len) {
    if (!g || !key || !bytes || !len) return SYN_ERR_NULL;
    const KV* e = find_kv(g, key);
    if (!e) return SYN_ERR_NOTFOUND;
    if (e->type != SYN_GGUF_STRING) return SYN_ERR_TYPE;
    *bytes = reinterpret_cast<const char*>(e->val);
    *len = (int64_t)e->str_len;
    return SYN_OK;
}

int syn_gguf_get_array(const syn_gguf* g, const char* key, uint32_t* elem_type, uint64_t* n, const void** data) {
    if (!g || !key || !elem_type || !n || !data) return SYN_ERR_NULL;
    const KV* e = find_kv(g, key);
    if (!e) return SYN_ERR_NOTFOUND;
    if (e->type != SYN_GGUF_ARRAY) return SYN_ERR_TYPE;
    *elem_type = e->arr_type;
    *n = e->arr_n;
    *data = e->val;
    return SYN_OK;
}

int syn_gguf_get_array_string(const syn_gguf* g, const char* key, uint64_t j, const char** bytes, int64_t* len) {
    if (!g || !key || !bytes || !len) return SYN_ERR_NULL;
    const KV* e = find_kv(g, key);
    if (!e) return SYN_ERR_NOTFOUND;
    if (e->type != SYN_GGUF_ARRAY || e->arr_type != SYN_GGUF_STRING) return SYN_ERR_TYPE;
    if (j >= e->arr_n) return SYN_ERR_NOTFOUND;
    // parse() bounds-checked every element; walk to element j
    Cursor c{e->val, g->size - (uint64_t)(e->val - g->base)};
    uint64_t l = 0;
    const uint8_t* s = nullptr;
    for (uint64_t k = 0; k <= j; k++) s = c.str(&l);
    if (!s) return SYN_ERR_FORMAT;
    *bytes = reinterpret_cast<const char*>(s);
    *len = (int64_t)l;
    return SYN_OK;
}

syn_gguf_writer* syn_gguf_writer_begin(const char* path, uint32_t alignment) {
    if (!path || alignment == 0 || alignment % 8) return nullptr;
    syn_gguf_writer* w = new syn_gguf_writer();
    w->path = path;
    w->alignment = alignment;
    if (alignment != 32) {  // a reader assumes 32 unless the file says otherwise
        kv_head(w, "general.alignment", SYN_GGUF_UINT32);
        put_u32(w->kv, alignment);
    }
    return w;
}

int syn_gguf_writer_kv_int(syn_gguf_writer* w, const char* key, uint32_t value_type, int64_t value) {
    const int64_t sz = scalar_size(value_type);
    if (sz < 0 || value_type == SYN_GGUF_FLOAT32 || value_type == SYN_GGUF_FLOAT64) return SYN_ERR_TYPE;
    if (key && strcmp(key, "general.alignment") == 0) return SYN_ERR_SHAPE;  // set by syn_gguf_writer_begin
    const int st = kv_head(w, key, value_type);
    if (st != SYN_OK) return st;
    const uint64_t u = (uint64_t)value;
    put(w->kv, &u, (size_t)sz);  // the low-order bytes
    return SYN_OK;
}

int syn_gguf_writer_kv_float(syn_gguf_writer* w, const char* key, uint32_t value_type, double value) {
    if (value_type != SYN_GGUF_FLOAT32 && value_type != SYN_GGUF_FLOAT64) return SYN_ERR_TYPE;
    const int st = kv_head(w, key, value_type);
    if (st != SYN_OK) return st;
    if (value_type == SYN_GGUF_FLOAT32) {
        const float f = (float)value;
        put(w->kv, &f, 4);
    } else {
        put(w->kv, &value, 8);
    }
    return SYN_OK;
}

int syn_gguf_writer_kv_string(syn_gguf_writer* w, const char* key, const char* bytes, int64_t len) {
    if (!bytes && len > 0) return SYN_ERR_NULL;
    if (len < 0) return SYN_ERR_SHAPE;
    const int st = kv_head(w, key, SYN_GGUF_STRING);
    if (st != SYN_OK) return st;
    put_str(w->kv, bytes, (uint64_t)len);
    return SYN_OK;
}

int syn_gguf_writer_kv_array(syn_gguf_writer* w, const char* key, uint32_t elem_type, uint64_t n, const void* data) {
    const int64_t sz = scalar_size(elem_type);
    if (sz < 0) return SYN_ERR_TYPE;
    if (!data && n > 0) return SYN_ERR_NULL;
    if (n > kMaxCount) return SYN_ERR_SHAPE;
    const int st = kv_head(w, key, SYN_GGUF_ARRAY);
    if (st != SYN_OK) return st;
    put_u32(w->kv, elem_type);
    put_u64(w->kv, n);
    if (n) put(w->kv, data, (size_t)(n * (uint64_t)sz));
    return SYN_OK;
}

int syn_gguf_writer_kv_string_array(syn_gguf_writer* w, const char* key, uint64_t n, const char* const* strs,
                                    const int64_t* lens) {
    if (n > 0 && (!strs || !lens)) return SYN_ERR_NULL;
    if (n > kMaxCount) return SYN_ERR_SHAPE;
    for (uint64_t j = 0; j < n; j++) {
        if (lens[j] < 0) return SYN_ERR_SHAPE;
        if (!strs[j] && lens[j] > 0) return SYN_ERR_NULL;
    }
    const int st = kv_head(w, key, SYN_GGUF_ARRAY);
    if (st != SYN_OK) return st;
    put_u32(w->kv, SYN_GGUF_STRING);
    put_u64(w->kv, n);
    for (uint64_t j = 0; j < n; j++) put_str(w->kv, strs[j], (uint64_t)lens[j]);
    return SYN_OK;
}

int syn_gguf_writer_add_tensor(syn_gguf_writer* w, const char* name, uint32_t ggml_type, int n_dims, const int64_t* ne,
                               const void* data, int64_t nbytes) {
    if (!w || !name || !ne || (!data && nbytes > 0)) return SYN_ERR_NULL;
    const GType* gt = find_type(ggml_type);
    if (!gt) return SYN_ERR_TYPE;
    if (n_dims < 1 || n_dims > 4) return SYN_ERR_SHAPE;
    int64_t count = 1;
    for (int d = 0; d < n_dims; d++) {
        if (ne[d] <= 0 || ne[d] > (int64_t(1) << 40) || count > (int64_t(1) << 50) / ne[d]) return SYN_ERR_SHAPE;
        count *= ne[d];
    }
    if (ne[0] % gt->elems || count / gt->elems * gt->bytes != nbytes) return SYN_ERR_SHAPE;
    if (!w->names.insert(name).second) return SYN_ERR_SHAPE;
    const uint64_t off = (w->data.size() + w->alignment - 1) / w->alignment * w->alignment;
    w->data.resize((size_t)off, 0);
    put(w->data, data, (size_t)nbytes);
    put_str(w->info, name, strlen(name));
    put_u32(w->info, (uint32_t)n_dims);
    for (int d = 0; d < n_dims; d++) put_u64(w->info, (uint64_t)ne[d]);
    put_u32(w->info, ggml_type);
    put_u64(w->info, off);
    w->n_tensors++;
    return SYN_OK;
}

int syn_gguf_writer_finish(syn_gguf_writer* w) {
    if (!w) return SYN_ERR_NULL;
    std::vector<uint8_t> head;
    put(head, "GGUF", 4);
    put_u32(head, 3);
    put_u64(head, w->n_tensors);
    put_u64(head, w->n_kv);
    const uint64_t meta_end = head.size() + w->kv.size() + w->info.size();
    const uint64_t data_start = (meta_end + w->alignment - 1) / w->alignment * w->alignment;
    const std::vector<uint8_t> pad((size_t)(data_start - meta_end), 0);
    int st = SYN_OK;
    FILE* f = fopen(w->path.c_str(), "wb");
    if (!f) {
        st = SYN_ERR_IO;
    } else {
        const std::vector<uint8_t>* parts[] = {&head, &w->kv, &w->info, &pad, &w->data};
        for (const std::vector<uint8_t>* part : parts)
            if (!part->empty() && fwrite(part->data(), 1, part->size(), f) != part->size()) st = SYN_ERR_IO;
        if (fclose(f) != 0) st = SYN_ERR_IO;
    }
    delete w;
    return st;
}

void syn_gguf_writer_abort(syn_gguf_writer* w) { delete w; }

}  // extern "C"
