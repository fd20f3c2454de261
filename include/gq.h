/*
 * gq.h -- C ABI of libgq: block-quantized (Q4_0 / Q8_0 / Q4_K) weights times fp32
 * activations on one NVIDIA GB300 GPU (sm_103a). Reading such weights out of GGUF files:
 * gq_gguf.h.
 *
 * The operation is the `mul_mat` that "No Python! Building an AI Inference Engine
 * Exclusively in C++" (section 6) says takes over 90% of inference compute, with the
 * weight held in 32-element blocks as "Development Guide for Small AI Models (TinyLLaMA,
 * etc.) Using C++" (section 6.1) lays them out and dequantized right after the load
 * ("No Python! ...", section 9; "Development Guide ...", section 6.2).
 *
 * Conventions shared by every call below.
 *   - Shapes. W is M x K (row m holds output feature m, K contiguous); X is N x K
 *     (token n is row n, K contiguous); Y is N x M (token n is row n, M contiguous):
 *         Y[n][m] = sum_k What[m][k] * X[n][k],   i.e.  Y = X . What^T.
 *     This is the layout of the cuBLAS call in "No Python! ...", section 7.2
 *     (cublasSgemm(T, N, m, n, k, W, k, X, k, Y, m)): column-major m x n is row-major N x M.
 *   - Block layout (public, fixed). Blocks follow each other row by row, K/32 per row,
 *     with no padding between rows.
 *       Q4_0, 18 bytes: fp16 scale d (little-endian), then 16 bytes of codes; byte j holds
 *             element j in its low nibble and element j+16 in its high nibble; a code c
 *             means What = (c - 8) * d.
 *       Q8_0, 34 bytes: fp16 scale d, then 32 signed bytes c; What = c * d.
 *       Q4_K, 144-byte super-blocks of 256 weights, K/256 per row (layout at
 *             gq_quantize_q4_k).
 *   - Pointers. Every array pointer is owned by the caller; the library keeps none of them
 *     after the call returns. W_blocks and workspaces are DEVICE pointers. X, Y (and the
 *     fused forms' gamma and H) are device pointers or pointers to page-locked host memory
 *     that the device can address (cudaHostAlloc, or cudaHostRegister with
 *     cudaHostRegisterMapped; with unified addressing the host address is valid on the
 *     device). Host buffers are read and written by the kernels themselves over the host
 *     link (NVLink-C2C on GB300), with ordinary loads and stores and no separate copy; the
 *     results are the same bits as with device buffers. W_blocks must be 16-byte
 *     aligned, fp32 arrays 4-byte aligned (16-byte alignment of X is used when present).
 *     A pointer may be NULL only when its array is empty. The CUDA-core decode path
 *     (N <= 2) allocates nothing; the tensor-core paths need a workspace (see
 *     gq_mul_mat_ws).
 *   - Streams. `stream` is a cudaStream_t (NULL = the legacy default stream) passed as
 *     void* so that this header needs no CUDA include. Calls only enqueue work: they do
 *     not synchronize, and results are ready when the stream reaches them.
 *   - Overlap of consecutive calls. A decode call (N <= 64, and gq_mul_mat_q8x) is
 *     launched as a programmatic dependent of the kernel before it on the stream: its CTAs
 *     may begin loading W_blocks on SMs that the previous libgq decode call has left,
 *     before that call has completed. X and Y are touched only after it has completed, so
 *     one call's Y may be the next call's X, or the other way round. W_blocks must
 *     therefore not be memory that the immediately preceding libgq decode call on the
 *     stream writes (its Y); any other kernel in between orders the two calls as usual.
 *     A prefill call (N >= 65) begins with an ordinary launch, so it starts only after
 *     everything before it on the stream has completed.
 *   - Errors. Argument checks run on the host before anything is launched and return a
 *     negative gq_status; nothing is enqueued then. A failed CUDA launch returns
 *     GQ_ERR_CUDA. Kernels never trap: a device-side wait that runs past its limit sets a
 *     per-device status word that gq_get_last_error() returns.
 *   - Empty inputs. M == 0 or N == 0 is a valid no-op; K == 0 writes Y = 0 (empty sum).
 *   - Range. Values are finite; |w| / 7 and |w| / 127 (Q4_K: a sub-block's range / 945)
 *     must fit fp16 (|d| <= 65504). Non-finite inputs give unspecified results.
 */
#ifndef GQ_H_
#define GQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GQ_ABI_VERSION 1
/* Largest number of problems one gq_mul_mat_batched call takes. */
#define GQ_MAX_BATCH 256

typedef enum gq_type {
    GQ_TYPE_Q4_0 = 2,   /* 18-byte blocks: fp16 scale + 32 4-bit codes */
    GQ_TYPE_Q8_0 = 8,   /* 34-byte blocks: fp16 scale + 32 int8 codes */
    GQ_TYPE_Q4_K = 12   /* 144-byte super-blocks of 256 weights (layout below) */
} gq_type;

typedef enum gq_status {
    GQ_OK = 0,
    GQ_ERR_NULL = -1,     /* a required pointer is NULL */
    GQ_ERR_SHAPE = -2,    /* negative size, K not a multiple of the block (32 weights, 256
                             for Q4_K), size overflow, count */
    GQ_ERR_TYPE = -3,     /* unknown gq_type, or one the entry point does not take */
    GQ_ERR_ALIGN = -4,    /* W_blocks not 16-byte aligned, or an fp32 array not 4-byte */
    GQ_ERR_CUDA = -5,     /* a CUDA runtime call failed (launch, attribute, no device) */
    GQ_ERR_TIMEOUT = -6,  /* a device-side wait ran out (reported by gq_get_last_error) */
    GQ_ERR_FORMAT = -7,   /* gq_gguf.h: not a GGUF file, or a malformed or truncated one */
    GQ_ERR_IO = -8        /* gq_gguf.h: the file could not be opened or mapped */
} gq_status;

/* Version of this ABI (GQ_ABI_VERSION of the header the library was built with). */
int32_t gq_abi_version(void);

/* Bytes of one block: 18 (Q4_0) or 34 (Q8_0) per 32 weights, 144 (Q4_K) per 256; 0 for
 * an unknown type. */
size_t gq_block_bytes(gq_type t);

/* Bytes of one quantized row of K weights: (K / 32) * gq_block_bytes(t), or for Q4_K
 * (K / 256) * 144; 0 if K is negative or not a multiple of the block, or the type is
 * unknown. */
size_t gq_row_bytes(gq_type t, int64_t K);

/*
 * Quantize W (M x K fp32) into Q4_0 blocks, per 32-element block
 * ("A Complete Guide to llama.cpp and Customization with C++", section 2.2: w_i ~= Delta*q_i
 * with Delta = max|w_i| / 7 and q_i in [-8, 7]):
 *     amax = max_i |w_i|;  d = amax / 7 (fp32, IEEE division);  stored scale = fp16(d),
 *     round to nearest even;  code_i = clamp(roundf(w_i / d) + 8, 0, 15) with roundf
 *     rounding halves away from zero; an all-zero block stores d = 0 and codes 8.
 * Bit-for-bit reproducible. W_blocks receives M * gq_row_bytes(GQ_TYPE_Q4_0, K) bytes.
 */
gq_status gq_quantize_q4_0(const float* W, int64_t M, int64_t K, void* W_blocks,
                           void* stream);

/*
 * Quantize W into Q8_0 blocks: d = amax / 127, stored as fp16(d);
 * code_i = clamp(roundf(w_i / d), -127, 127); all-zero block -> d = 0, codes 0.
 * The pages name 8-bit quantization ("No Python! ...", section 9) without a layout; this
 * is the 4-bit rule above carried to signed 8-bit codes.
 */
gq_status gq_quantize_q8_0(const float* W, int64_t M, int64_t K, void* W_blocks,
                           void* stream);

/*
 * Q4_K super-blocks. The pages name Q4_K as the 4-bit format of a ~600 MB TinyLLaMA
 * ("Development Guide ...", section 6; "A Complete Guide to llama.cpp ...", section 2.2)
 * without a layout; this is the published GGUF Q4_K block, 256 weights in eight
 * sub-blocks of 32, 144 bytes:
 *   bytes 0-1    d (fp16), the scale of the sub-block scales
 *   bytes 2-3    dmin (fp16), the scale of the sub-block mins
 *   bytes 4-15   s[0..11]: 6-bit sub-block scales sc_j and mins m_j,
 *                j < 4:  sc_j = s[j] & 63, m_j = s[j + 4] & 63;
 *                j >= 4: sc_j = (s[j + 4] & 15) | (s[j - 4] >> 6) << 4,
 *                        m_j = (s[j + 4] >> 4) | (s[j] >> 6) << 4
 *   bytes 16-143 4-bit codes q: byte 16 + 32 g + l holds weight 64 g + l (low nibble)
 *                and weight 64 g + 32 + l (high nibble), g = 0..3, l = 0..31
 *   What = d sc_j q - dmin m_j (both products exact in fp32, rounded once).
 * gq_quantize_q4_k is this library's own quantizer (the format fixes only the
 * dequantization): per sub-block lo = min(0, min w), hi = max w, step = (hi - lo) / 15,
 * min = -lo; d = max step / 63 and dmin = max min / 63 (fp32 division, stored as fp16
 * round to nearest even); sc_j = roundf(step_j / d), m_j = roundf(min_j / dmin), clamped
 * to [0, 63] (0 where d or dmin is 0); codes roundf((w + M_j) / D_j) clamped to [0, 15]
 * with D_j = fp16(d) sc_j and M_j = fp16(dmin) m_j (0 where D_j = 0). K must be a
 * multiple of 256 (else GQ_ERR_SHAPE). Bit-for-bit reproducible.
 * The mul_mat entry points take Q4_K on the same paths as Q4_0 (CUDA-core decode for
 * N <= 2, tensor-core decode for 3..64 tokens, prefill GEMM from 65, with the same
 * workspace sizes, but for the X block sums below); the tensor-core decode with N <= 16
 * multiplies the exact codes q and applies d sc and dmin m per sub-block in fp32, and the
 * other tensor-core forms use each weight d sc q - dmin m rounded once in fp32, as
 * gq_dequantize writes it, then rounded to bf16. gq_mul_mat_rmsnorm and
 * gq_mul_mat_swiglu take it in their composite forms (norm kernel, then the product; two
 * products, then the elementwise kernel); gq_mul_mat_q8x and gq_mul_mat_q8x_batched
 * return GQ_ERR_TYPE for it (their activation blocks pair with 32-weight blocks).
 */
gq_status gq_quantize_q4_k(const float* W, int64_t M, int64_t K, void* W_blocks,
                           void* stream);

/*
 * Expand blocks back to fp32: W_out[m][k] = (c - 8) * d (Q4_0), c * d (Q8_0), or
 * d sc_j q - dmin m_j (Q4_K), exact up to Q4_K's one rounding ("Development Guide ...",
 * section 6.2, the unpack and dequantize steps). W_out receives M x K floats.
 */
gq_status gq_dequantize(const void* W_blocks, gq_type t, int64_t M, int64_t K,
                        float* W_out, void* stream);

/*
 * Y (N x M fp32) = X (N x K fp32) . What^T, What the dequantized W_blocks (M rows).
 * ("No Python! ...", sections 6 and 7.2; "A Complete Guide ...", section 2.1: N = 1 at
 * decode makes this a matrix-vector product.) The weights are dequantized inside the
 * kernel right after they are loaded and never written back.
 * N <= 2 (or K % 256 != 0): decode kernels on CUDA cores (exact integer block products
 * on a 16-bit fixed-point copy of X). 3 <= N <= 64 and K % 256 == 0: decode on tensor
 * cores; N >= 65 and K % 256 == 0: the prefill tensor-core GEMM. Both tensor-core paths
 * round X once to bf16 and accumulate in fp32. The weights enter the MMA as bf16
 * dequantized values (rounded once), except Q4_0 and Q4_K decode with N <= 16, which
 * multiply the exact codes (c - 8, or q) and apply each block's scale (and Q4_K's min,
 * against the block's sum of the bf16 X) in fp32.
 * Accuracy: |Y - Y_exact| <= 1e-3 * ||X[n]||_2 * ||What[m]||_2 per element (for the bf16
 * path, at the K >= 256 it runs on, by a wide margin for non-adversarial data). Q4_K on
 * the CUDA-core kernels forms d (sum sc S) - dmin (sum m X) per quarter super-block in
 * fp32; where the two terms cancel (super-block bytes the quantizer does not write) add
 * (K / 256 + 32) * 2^-23 * sum_k (|d sc_j q_k| + |dmin m_j|) |X[n][k]| to the bound.
 * Results are deterministic: the same inputs give the same bits on every call.
 * Y must not overlap W_blocks or X.
 */
gq_status gq_mul_mat(const void* W_blocks, gq_type t, int64_t M, int64_t K,
                     const float* X, int64_t N, float* Y, void* stream);

/*
 * Device workspace (bytes) that gq_mul_mat_ws needs for this shape: 0 on the CUDA-core
 * decode path (N <= 2); on the tensor-core decode path (3 <= N <= 64) P * K * 2 for
 * P = 16, 32 or 64 token rows of pre-arranged bf16 X (Q4_K with N <= 16: plus K / 256 * 1024
 * for the X block sums), plus 2 * 256 * 128 * P * 4 + 4096 for the partial sums (and
 * their counters) of tiles whose k range is split between CTAs;
 * N * K * 2 (a bf16 copy of X, rounded up to 256) on the prefill path (N >= 65).
 * Tensor-core paths need K a multiple of 256. 0 for invalid arguments.
 */
size_t gq_mul_mat_workspace_size(gq_type t, int64_t M, int64_t K, int64_t N);

/*
 * gq_mul_mat with caller-owned workspace: `workspace` must hold
 * gq_mul_mat_workspace_size(t, M, K, N) bytes, be 256-byte aligned and not be used by
 * other work in flight. It may be NULL when that size is 0. Nothing is allocated, so this
 * is the form to use inside CUDA graph capture. GQ_ERR_NULL if a needed workspace is NULL,
 * GQ_ERR_SHAPE if it is too small, GQ_ERR_ALIGN if misaligned.
 * gq_mul_mat itself uses a library-owned workspace for the tensor-core path: one device
 * buffer per (device, stream), allocated on first need and grown when a larger shape
 * arrives (growing synchronizes that stream and is refused, GQ_ERR_CUDA, during capture).
 */
gq_status gq_mul_mat_ws(const void* W_blocks, gq_type t, int64_t M, int64_t K,
                        const float* X, int64_t N, float* Y, void* workspace,
                        size_t workspace_bytes, void* stream);

/*
 * gq_mul_mat that never allocates device memory, for callers that cannot allocate at the
 * point where they multiply: engines that reserve all device memory up front in their own
 * arena, and real-time loops that must not stall or fail on an allocation mid-run. (The
 * pages have no counterpart: their engine allocates once from an arena; this entry point
 * exists for users of this library.)
 * Same arguments, paths, results and accuracy as gq_mul_mat. The workspace of its
 * tensor-core paths is a fixed 64 MiB device array compiled into the library:
 *   - a GPU holds that array from this module's first use on it (CUDA's default lazy
 *     module loading) or from context creation (CUDA_MODULE_LOADING=EAGER) until the
 *     process exits;
 *   - prefill (N >= 65, K % 256 == 0) keeps a bf16 copy of X there: shapes whose N * K * 2
 *     exceeds 64 MiB (N * K > 32 Mi) return GQ_ERR_SHAPE;
 *   - the tensor-core decode (3 <= N <= 64) needs at most 64 * K * 2 bytes + 16 MiB + 4 KiB
 *     there; a larger K (beyond ~390k) runs on the CUDA-core decode kernels instead;
 *   - the first call on a device looks up that array's device address (a one-time host-side
 *     set-up). The address is kept for the life of the process, so libgq must not be used
 *     again on a device the process has reset with cudaDeviceReset;
 *   - every call shares the array (each call rewrites what it reads there, and zeroes its
 *     counters, before use), so calls that overlap on the GPU -- on different streams, or
 *     from different threads -- race: serialize them.
 */
gq_status gq_mul_mat_noalloc(const void* W_blocks, gq_type t, int64_t M, int64_t K,
                             const float* X, int64_t N, float* Y, void* stream);

/* One independent problem of gq_mul_mat_batched. */
typedef struct gq_mul_mat_problem {
    const void* W_blocks;   /* M rows of gq_row_bytes(t, K) bytes, 16-byte aligned */
    const float* X;         /* N x K */
    float* Y;               /* N x M */
    int64_t M;
    int64_t K;
} gq_mul_mat_problem;

/*
 * `count` independent gq_mul_mat problems that share the block type and N, computed by
 * one launch that streams all their weights as one sequence. This is how one decode step
 * runs its many matrix-vector products without a launch per matrix. Each problem follows
 * gq_mul_mat's contract; Y buffers must not overlap each other or any input.
 * count <= GQ_MAX_BATCH. The problem array is read on the host during the call.
 */
gq_status gq_mul_mat_batched(const gq_mul_mat_problem* problems, int32_t count,
                             gq_type t, int64_t N, void* stream);

/*
 * Workspace (bytes) gq_mul_mat_batched_ws needs for these problems: the largest prefill
 * workspace among them, or the tensor-core decode workspace of the problems that take that
 * path (the partial sums once, plus every problem's X tiles), whichever is larger;
 * 0 if every problem runs on the CUDA-core decode path, and for invalid arguments.
 */
size_t gq_mul_mat_batched_workspace_size(const gq_mul_mat_problem* problems, int32_t count,
                                         gq_type t, int64_t N);

/*
 * gq_mul_mat_batched with caller-owned workspace (256-byte aligned, at least
 * gq_mul_mat_batched_workspace_size bytes, not used by other work in flight); allocates
 * nothing, so it is the form to record into a CUDA graph. gq_mul_mat_batched uses the
 * library-owned per-(device, stream) workspace instead (see gq_mul_mat_ws).
 */
gq_status gq_mul_mat_batched_ws(const gq_mul_mat_problem* problems, int32_t count,
                                gq_type t, int64_t N, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * Quantized-activation mul_mat ("A Complete Guide to llama.cpp and Customization with
 * C++", section 2.2: with x quantized like the weights, x_i ~= Delta_x q_x,i, a block's
 * dot product is Delta Delta_x sum_i q_i q_x,i and the sum is a pure integer operation):
 *   - every 32-element block of each X row is quantized exactly like a Q8_0 weight block
 *     (Delta = max |x| / 127, q_x = round(x / Delta) with halves away from zero, clamped to
 *     [-127, 127]; Delta_x is the fp16 value of Delta, held as fp32);
 *   - Y[n][m] = sum over blocks b of Delta_w[m][b] * Delta_x[n][b] * S_b, S_b = the exact
 *     integer sum of q_i * q_x,i (q_i = c - 8 for Q4_0, c for Q8_0), accumulated in fp32.
 * The result differs from gq_mul_mat by the quantization of X (an approximation the caller
 * opts into); against the definition above it is exact up to fp32 accumulation.
 * Same argument contract as gq_mul_mat, plus: K a multiple of 256 and X 16-byte aligned
 * (else GQ_ERR_SHAPE / GQ_ERR_ALIGN; GQ_ERR_SHAPE also when K is too large for the
 * activation records in shared memory). Any N: up to 4 tokens per pass over the weights.
 * Allocates nothing.
 */
gq_status gq_mul_mat_q8x(const void* W_blocks, gq_type t, int64_t M, int64_t K,
                         const float* X, int64_t N, float* Y, void* stream);

/*
 * gq_mul_mat_q8x over up to GQ_MAX_BATCH independent problems (same type and N) in one
 * launch per pass. Every problem is checked before anything is queued.
 */
gq_status gq_mul_mat_q8x_batched(const gq_mul_mat_problem* problems, int32_t count,
                                 gq_type t, int64_t N, void* stream);

/*
 * The two steps next to the product in a transformer layer, fused with it.
 *
 * gq_mul_mat_rmsnorm: Y = RMSNorm(X) . What^T, where per token n
 *     RMSNorm(x) = x / sqrt((1/K) sum_k x_k^2 + eps) (.) gamma
 * ("Development Guide for Small AI Models (TinyLLaMA, etc.) Using C++", section 4.1:
 * the norm ahead of the projections and of the LM head).
 *   - gamma: K floats (device), 4-byte aligned; eps: finite and >= 0 (else GQ_ERR_SHAPE).
 *   - K == 0 is GQ_ERR_SHAPE (the mean of nothing); other arguments as gq_mul_mat.
 *   - Decode (N <= 2, K % 256 == 0, X and gamma 16-byte aligned): one launch; the decode
 *     kernel normalizes X while it prepares it. Otherwise a per-token norm kernel writes the
 *     normalized X into library workspace and the plain product follows.
 *   - Accuracy: as gq_mul_mat, with ||RMSNorm(X)[n]||_2 in place of ||X[n]||_2.
 *
 * gq_mul_mat_swiglu: H[n][m] = Swish(G[n][m]) * U[n][m], G = X . What_gate^T,
 * U = X . What_up^T, Swish(z) = z / (1 + e^-z) (the same guide, section 4.4: the gated
 * feed-forward activation).
 *   - W_gate and W_up: M x K blocks of the same type, both 16-byte aligned; H: N x M.
 *   - K == 0 writes H = 0; other arguments as gq_mul_mat.
 *   - Decode (N <= 2, K % 256 == 0): one launch; each warp streams gate row m and up row m
 *     side by side and writes H directly. Otherwise G and U go to library workspace by two
 *     plain products and an elementwise kernel writes H.
 *   - Accuracy: |H - H_exact| <= 1.1 |U| e_G + |Swish(G)| e_U to first order, where e_G and
 *     e_U are the gq_mul_mat bounds of the two products (|Swish'| <= 1.1).
 * Both need library workspace off the decode path (like gq_mul_mat; refused while the
 * stream is being captured if it must grow). Y / H must not overlap the other arrays.
 */
gq_status gq_mul_mat_rmsnorm(const void* W_blocks, gq_type t, int64_t M, int64_t K,
                             const float* X, const float* gamma, float eps, int64_t N,
                             float* Y, void* stream);
gq_status gq_mul_mat_swiglu(const void* W_gate, const void* W_up, gq_type t, int64_t M,
                            int64_t K, const float* X, int64_t N, float* H, void* stream);

/*
 * Device-side status of the current device: synchronizes `stream`, then returns and
 * clears the status word (GQ_OK, or GQ_ERR_TIMEOUT if a kernel gave up waiting), or
 * GQ_ERR_CUDA if the stream itself reports an error.
 */
gq_status gq_get_last_error(void* stream);

/*
 * Self-test of failure detection: launches one thread that waits on a device barrier that
 * nothing ever completes, with a limit of `limit_us` microseconds (1 .. 10^7), using the
 * same bounded wait as every kernel here. The wait runs out, the kernel records it in the
 * status word and returns; the next gq_get_last_error() on this device reports
 * GQ_ERR_TIMEOUT (and clears it). No fault, no trap, no hang. GQ_ERR_SHAPE for a limit
 * out of range. (The pages' engine only asserts; this is the library's own check.)
 */
gq_status gq_selftest_wait_timeout(int64_t limit_us, void* stream);

/* Static English text for a status code. */
const char* gq_status_string(gq_status s);

#ifdef __cplusplus
}
#endif

#endif /* GQ_H_ */
