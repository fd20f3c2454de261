/*
 * gq_gguf.h -- reading block-quantized weights out of GGUF files, for libgq's mul_mat.
 *
 * "Development Guide for Small AI Models (TinyLLaMA, etc.) Using C++" gives the file's
 * structure (section 3.2): magic bytes 0x46554747 ("GGUF"), a version, the tensor and
 * metadata counts, typed key-value metadata with length-prefixed keys, one info record per
 * tensor (name, dimensions, data type, offset), padding so that tensor data starts on an
 * alignment boundary (usually 32 or 64 bytes), then the aligned tensor data; and it loads
 * the file by memory mapping (section 3.1: the data is paged in from disk when first
 * touched, with no copy into a user buffer). The field widths and type codes are those of
 * the published GGUF specification (versions 2 and 3, little-endian):
 *   header      uint32 magic, uint32 version, uint64 tensor count, uint64 metadata count
 *   string      uint64 length, then that many bytes (no terminator)
 *   metadata    string key, uint32 value type, value
 *               value types: 0 uint8, 1 int8, 2 uint16, 3 int16, 4 uint32, 5 int32,
 *               6 float32, 7 bool (one byte), 8 string, 9 array (uint32 element type,
 *               uint64 count, the elements), 10 uint64, 11 int64, 12 float64
 *   tensor info string name, uint32 n_dims (1..4), uint64 ne[n_dims] (ne[0] the
 *               contiguous extent), uint32 type (ggml type id), uint64 offset (from the
 *               start of the data section, a multiple of the alignment)
 *   data        starts at the first multiple of the alignment after the last tensor
 *               info; the alignment is the uint32 metadata "general.alignment", else 32.
 * The ggml type ids of the three block formats equal gq_type: 2 Q4_0, 8 Q8_0, 12 Q4_K, and
 * a 2-D weight tensor of those types is stored exactly as gq_mul_mat reads W_blocks:
 * M = ne[1] rows of gq_row_bytes(type, K = ne[0]) bytes each. So a tensor goes from the
 * file to the GPU with one copy and no conversion.
 *
 * Every function here runs on the host. A gq_gguf handle owns the mapping and every string
 * it hands out; they stay valid until gq_gguf_close. Handles are read-only after
 * gq_gguf_open returns, so several threads may query one handle at once. Every length,
 * count and offset in the file is checked against the file's size before it is used: a
 * malformed or truncated file gives GQ_ERR_FORMAT, never a read outside the mapping.
 */
#ifndef GQ_GGUF_H_
#define GQ_GGUF_H_

#include <stddef.h>
#include <stdint.h>

#include "gq.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gq_gguf gq_gguf;   /* an open, memory-mapped GGUF file */

/* GGUF metadata value types (the published numbering). */
enum {
    GQ_GGUF_UINT8 = 0, GQ_GGUF_INT8 = 1, GQ_GGUF_UINT16 = 2, GQ_GGUF_INT16 = 3,
    GQ_GGUF_UINT32 = 4, GQ_GGUF_INT32 = 5, GQ_GGUF_FLOAT32 = 6, GQ_GGUF_BOOL = 7,
    GQ_GGUF_STRING = 8, GQ_GGUF_ARRAY = 9, GQ_GGUF_UINT64 = 10, GQ_GGUF_INT64 = 11,
    GQ_GGUF_FLOAT64 = 12
};

/* One tensor info record. */
typedef struct gq_gguf_tensor {
    const char* name;   /* NUL-terminated, owned by the handle */
    uint32_t n_dims;    /* 1..4 */
    uint32_t type;      /* ggml type id (0 F32, 1 F16, 2 Q4_0, 8 Q8_0, 12 Q4_K, 30 BF16, ...) */
    int64_t ne[4];      /* extents, ne[0] contiguous; 1 past n_dims */
    uint64_t offset;    /* byte offset of the tensor's data from the start of the FILE */
    uint64_t nbytes;    /* size of the data; 0 if this library does not know the type */
} gq_gguf_tensor;

/*
 * Opens and maps `path` read-only and parses the header, the metadata and the tensor
 * infos. On success *out is a handle for gq_gguf_close. Errors: GQ_ERR_NULL (path or out
 * NULL), GQ_ERR_IO (cannot open, stat or map), GQ_ERR_FORMAT (wrong magic, a version
 * other than 2 or 3, a length, count or offset past the end of the file, n_dims outside
 * 1..4, a negative or overflowing extent, a zero or non-power-of-two alignment, a tensor
 * offset that is not a multiple of the alignment, a quantized tensor whose ne[0] is not
 * a whole number of blocks, or data of a known type that does not fit in the file).
 * *out is left NULL on every error.
 */
gq_status gq_gguf_open(const char* path, gq_gguf** out);

/* Unmaps the file and frees the handle (NULL is a no-op). */
void gq_gguf_close(gq_gguf* f);

/* The header's version (2 or 3), tensor count, metadata count; alignment of the data. */
uint32_t gq_gguf_version(const gq_gguf* f);
int64_t gq_gguf_tensor_count(const gq_gguf* f);
int64_t gq_gguf_kv_count(const gq_gguf* f);
uint64_t gq_gguf_alignment(const gq_gguf* f);

/* Tensor info i (0 <= i < tensor count): GQ_ERR_NULL, GQ_ERR_SHAPE (i out of range). */
gq_status gq_gguf_tensor_info(const gq_gguf* f, int64_t i, gq_gguf_tensor* out);

/* Index of the tensor named `name`, or -1. */
int64_t gq_gguf_find_tensor(const gq_gguf* f, const char* name);

/* Host address of tensor i's data inside the mapping (NULL for a bad index). Reading it
 * pages the data in from the file. */
const void* gq_gguf_tensor_data(const gq_gguf* f, int64_t i);

/*
 * A 2-D tensor of a block type that gq_mul_mat takes, as gq_mul_mat's arguments:
 * *type (GQ_TYPE_Q4_0, _Q8_0 or _Q4_K), *M = ne[1], *K = ne[0]. GQ_ERR_TYPE for another
 * data type, GQ_ERR_SHAPE for a tensor with more than two non-unit dimensions or an index
 * out of range.
 */
gq_status gq_gguf_tensor_matrix(const gq_gguf* f, int64_t i, gq_type* type, int64_t* M,
                                int64_t* K);

/*
 * Copies tensor i's data from the mapping to device memory `dst` (dst_bytes available)
 * with cudaMemcpyAsync on `stream` (a cudaStream_t; NULL = the legacy default stream).
 * The mapping is pageable host memory, so the copy is staged by the CUDA driver and the
 * call returns once the source has been read. For a tensor of gq_gguf_tensor_matrix the
 * result is W_blocks for gq_mul_mat as it stands. Errors: GQ_ERR_NULL, GQ_ERR_SHAPE (bad
 * index, dst_bytes < nbytes, or a type of unknown size), GQ_ERR_ALIGN (dst not 16-byte
 * aligned), GQ_ERR_CUDA (the copy failed).
 */
gq_status gq_gguf_upload(const gq_gguf* f, int64_t i, void* dst, size_t dst_bytes,
                         void* stream);

/* Metadata. Index of key `key`, or -1; key i (NUL-terminated, owned by the handle, NULL
 * for a bad index); value type of entry i (GQ_GGUF_*, or -1 for a bad index). */
int64_t gq_gguf_find_key(const gq_gguf* f, const char* key);
const char* gq_gguf_kv_key(const gq_gguf* f, int64_t i);
int32_t gq_gguf_kv_type(const gq_gguf* f, int64_t i);

/* Value of entry i: an integer or bool type as int64 (GQ_ERR_SHAPE for a uint64 above
 * INT64_MAX), a float type as double, a string as bytes inside the mapping (not
 * NUL-terminated) and its length, an array as its element type, count and the address of
 * its first element inside the mapping (elements little-endian, one after another; string
 * and array elements keep their own length prefixes). GQ_ERR_TYPE if the entry has
 * another type, GQ_ERR_SHAPE for a bad index, GQ_ERR_NULL for a NULL output. */
gq_status gq_gguf_kv_int(const gq_gguf* f, int64_t i, int64_t* out);
gq_status gq_gguf_kv_float(const gq_gguf* f, int64_t i, double* out);
gq_status gq_gguf_kv_string(const gq_gguf* f, int64_t i, const char** data, uint64_t* len);
gq_status gq_gguf_kv_array(const gq_gguf* f, int64_t i, uint32_t* elem_type, uint64_t* count,
                           const void** data);

#ifdef __cplusplus
}
#endif

#endif /* GQ_GGUF_H_ */
