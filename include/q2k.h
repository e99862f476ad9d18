/*
 * q2k.h - C ABI of libq2k: GGML Q2_K dequantize, embedding gather and
 * weight-quantized matmul on one NVIDIA GB300 (sm_103a).
 *
 * Q2_K storage (mlx-native page "tests/deepseek_q2_k.rs", consts QK_K and
 * BLOCK_BYTES, fixture fn block, fn reference_dequant): a super-block of 256
 * weights is 84 bytes -
 *     bytes  0..15  scale byte per 16-weight group: low nibble sc, high nibble m
 *     bytes 16..79  2-bit quants q, four per byte
 *     bytes 80..81  f16 d      (little endian)
 *     bytes 82..83  f16 dmin   (little endian)
 * Weight k of a block (k = 128 half + 32 j + 16 segment + lane, shift = 2 j)
 * is  dl*q - ml  with  q = (qs[32 half + 16 segment + lane] >> shift) & 3,
 * dl = d * (sc & 15), ml = dmin * (sc >> 4) of scale byte 8 half + 2 j + segment.
 * A matrix of n rows and k columns is n rows of k/256 consecutive blocks, row
 * after row (block b of row r at byte (r * k/256 + b) * 84).
 *
 * Conventions shared by every call:
 *  - Pointers are caller-owned DEVICE memory unless stated otherwise; the
 *    library allocates no device memory in these calls and keeps no pointer
 *    after returning.
 *  - Sizes are exact: a buffer whose stated size differs from the size the
 *    geometry implies is rejected (the pages' `require` check: exact byte
 *    length, overflow-checked products).
 *  - An output may not overlap any input (the pages' `validate_disjoint`).
 *  - On any Q2K_ERR_INVALID_ARGUMENT nothing is launched; q2k_last_error()
 *    returns a message (thread-local, valid until the next call on the thread).
 *  - Work is enqueued on `stream` (NULL = the legacy default stream) and the
 *    call returns without waiting, except where stated.  Launch failures map
 *    to Q2K_ERR_CUDA.
 *  - The device is the one current on the calling thread.
 */
#ifndef Q2K_H
#define Q2K_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream, without pulling in the CUDA headers. */
typedef struct CUstream_st *q2k_stream_t;

typedef enum q2k_status {
    Q2K_OK = 0,
    Q2K_ERR_INVALID_ARGUMENT = 1, /* the pages' MlxError::InvalidArgument */
    Q2K_ERR_BAD_ID = 2,           /* an id out of range (gather, routed calls without bad_id_count) */
    Q2K_ERR_CUDA = 3,             /* a CUDA runtime call or launch failed */
    Q2K_ERR_TIMEOUT = 4,          /* a kernel gave up waiting (see q2k_device_error) */
    Q2K_ERR_NO_DEVICE = 5,        /* no sm_103 device is current */
    Q2K_ERR_IO = 6                /* a file could not be opened or read (GGUF reader) */
} q2k_status;

enum {
    Q2K_GGML_TYPE_Q2_K = 10, /* GGUF / GgmlType tag of Q2_K */
    Q2K_QK_K = 256,          /* weights per super-block */
    Q2K_BLOCK_BYTES = 84     /* bytes per super-block */
};

/* Geometry of y[m, n] = sum_k x[m, k] * W[n, k]; the pages'
 * GgmlQuantizedMatmulParams {m, n, k, ggml_type} (page "tests/deepseek_q2_k.rs",
 * fn run_dense).  16 bytes, fields in this order. */
typedef struct q2k_matmul_params {
    uint32_t m;          /* activation rows (tokens), >= 1 */
    uint32_t n;          /* weight rows = output columns, >= 1 */
    uint32_t k;          /* reduction length, a positive multiple of 256 */
    uint32_t ggml_type;  /* must be Q2K_GGML_TYPE_Q2_K */
} q2k_matmul_params;

/* The pages' EmbeddingQ2KParams {vocab_size, embed_dim, n_tokens} (page
 * "tests/deepseek_q2_k.rs", test q2_k_embedding_gather_...), plus the type tag. */
typedef struct q2k_embedding_params {
    uint32_t vocab_size; /* table rows, >= 1 */
    uint32_t embed_dim;  /* table columns, a positive multiple of 256 */
    uint32_t n_tokens;   /* ids to gather, >= 1 */
    uint32_t ggml_type;  /* must be Q2K_GGML_TYPE_Q2_K */
} q2k_embedding_params;

/* The pages' GgmlQuantizedMatmulIdParams {n_tokens, top_k, n, k, n_experts,
 * expert_stride, ggml_type} (page "tests/deepseek_q2_k.rs", fn run_expert),
 * the 32-bit fields first so the struct has no padding: 32 bytes. */
typedef struct q2k_matmul_id_params {
    uint32_t n_tokens;      /* tokens (rows of x), >= 1 */
    uint32_t top_k;         /* experts per token, >= 1 */
    uint32_t n;             /* weight rows of each expert = output columns, >= 1 */
    uint32_t k;             /* reduction length, a positive multiple of 256 */
    uint32_t n_experts;     /* experts in w, >= 1 */
    uint32_t ggml_type;     /* must be Q2K_GGML_TYPE_Q2_K */
    uint64_t expert_stride; /* bytes from one expert's matrix to the next, a multiple
                               of 4 and >= n * k/256 * 84 */
} q2k_matmul_id_params;

/* Which kernel q2k_matmul_path runs (the pages' forced-path test hooks
 * dispatch_mm_for_test / dispatch_mm_simd_for_test). */
typedef enum q2k_path {
    Q2K_PATH_AUTO = 0,   /* what q2k_matmul picks: GEMV for m <= 8, else tensor cores */
    Q2K_PATH_GEMV = 1,   /* fp32 CUDA-core streaming GEMV, any m (fastest for m <= 8) */
    Q2K_PATH_TENSOR = 2  /* bf16 tcgen05 tensor-core GEMM with fp32 accumulation */
} q2k_path;

/* q2k_dequantize - decode whole Q2_K blocks to f32.
 * Page "tests/deepseek_q2_k.rs": fn test_only_dequantize and tests
 * q2_k_host_decode_matches_all_256_canonical_values / ..._rejects_malformed_buffers.
 *   blocks      device, blocks_bytes bytes, 4-byte aligned; blocks_bytes a
 *               positive multiple of 84 (83 bytes is rejected)
 *   out         device f32, out_elems = blocks_bytes / 84 * 256 exactly
 *               (one float short is rejected); 16-byte aligned
 * Results are bit-identical to the page's f32 loop (each product rounded on
 * its own; all of them are exact in f32, so only the subtraction rounds). */
q2k_status q2k_dequantize(const void *blocks, size_t blocks_bytes,
                          float *out, size_t out_elems, q2k_stream_t stream);

/* q2k_embedding_gather - out[t, :] = decoded table row ids[t].
 * Page "tests/deepseek_q2_k.rs": fn embedding_gather_q2_k and test
 * q2_k_embedding_gather_matches_canonical_rows_and_rejects_bad_ids.
 *   table       device, table_bytes = vocab_size * embed_dim/256 * 84, 4-byte aligned
 *   ids         device u32 [n_tokens]
 *   out         device f32 [n_tokens, embed_dim], out_elems = n_tokens*embed_dim,
 *               16-byte aligned
 *   bad_id_count  device u32 or NULL.  The pages reject an id >= vocab_size.
 *               Ids live on the device here, so the check runs in the kernel:
 *               a row with a bad id is written as zeros and the bad ids are
 *               counted.
 *                 NULL: the call counts them in a word of its own, reads it
 *                 back (4 bytes) and waits for `stream` to finish, then
 *                 returns Q2K_ERR_BAD_ID if any id was out of range (the
 *                 pages' error), else Q2K_OK.  This form synchronises, so it
 *                 is refused (Q2K_ERR_INVALID_ARGUMENT) while `stream` is
 *                 being captured; at most 64 such calls may be in flight per
 *                 device at once (from concurrent host threads).
 *                 Not NULL: the count is stored there (the call zeroes it
 *                 first, stream-ordered) and the call returns without
 *                 waiting; read it after the stream completes, nonzero means
 *                 the pages' error.
 * Decoded values are bit-identical to q2k_dequantize of the same rows. */
q2k_status q2k_embedding_gather(const void *table, size_t table_bytes,
                                const uint32_t *ids, float *out, size_t out_elems,
                                const q2k_embedding_params *params,
                                uint32_t *bad_id_count, q2k_stream_t stream);

/* q2k_matmul - y[m, n] = sum_k x[m, k] * W[n, k] with W in Q2_K, the
 * dequantization fused into the product.
 * Page "tests/deepseek_q2_k.rs": fn quantized_matmul_ggml, fn run_dense.
 *   x           device f32 [m, k] row-major, x_elems = m*k, 16-byte aligned
 *   w           device, w_bytes = n * k/256 * 84, 4-byte aligned
 *   y           device f32 [m, n] row-major, y_elems = m*n, 16-byte aligned;
 *               fully overwritten
 * Path: m <= 8 runs the fp32 GEMV: each weight is formed exactly as the
 * page's f32 decode (dl*q - ml rounded once) and multiplied into fp32 sums in
 * which a product passes through at most L roundings - L = 46 for m = 1 with
 * k <= 16384, L = 71 + k/262144 otherwise - so the error is at most
 * L * 2^-24 * sum_k |x w|: within the 1e-5 tolerance for k <= 2^24, for every
 * finite x whose products x w stay in the f32 normal range.  m > 8 runs the bf16 tensor-core GEMM (x and W rounded to
 * bf16, fp32 accumulation; error within 8e-3 * sum_k |x w|), mirroring the
 * pages' switch of tolerance at rows > 8; without a workspace it uses the
 * library's scratch as described at q2k_matmul_ex.  Repeated calls on the
 * same inputs give bit-identical y (no floating-point atomics). */
q2k_status q2k_matmul(const float *x, size_t x_elems, const void *w, size_t w_bytes,
                      float *y, size_t y_elems, const q2k_matmul_params *params,
                      q2k_stream_t stream);

/* q2k_matmul_path - q2k_matmul with the kernel chosen by the caller (the
 * pages' dispatch_mm_for_test); same arguments, sizes and errors. */
q2k_status q2k_matmul_path(q2k_path path, const float *x, size_t x_elems,
                           const void *w, size_t w_bytes, float *y, size_t y_elems,
                           const q2k_matmul_params *params, q2k_stream_t stream);

/* Flags of q2k_matmul_ex. */
enum {
    /* The caller guarantees that the kernel enqueued on `stream` immediately
     * before this call does not write W (model weights that are only read).
     * The m = 1 GEMV then starts copying W before it waits for that kernel,
     * overlapping the weight stream with it.  Without the flag it only
     * prefetches W into L2 (always safe) and copies after the wait. */
    Q2K_FLAG_CONST_WEIGHTS = 1,
    /* The caller guarantees that no kernel enqueued on `stream` before this
     * call that may still be running writes x or W, or reads or writes y
     * (e.g. several projections of one activation, each with its own W and
     * y, enqueued back to back).  The m = 1 GEMV then reads x and writes y
     * without waiting for the kernel before it, so consecutive calls overlap;
     * it still waits for that kernel before it finishes, so calls complete in
     * stream order.  Implies Q2K_FLAG_CONST_WEIGHTS.
     * Both flags also apply to the tensor-core path for m <= 64 (whose GEMM
     * converts x itself): its weight copies (CONST_WEIGHTS), and its x
     * conversion and y stores (INDEPENDENT), start before the wait for the
     * kernel before.  In q2k_matmul_ex_batch, INDEPENDENT also lets a
     * tensor-path call reuse the x image of the call before it (same x, m, k
     * and workspace) and run beside it, and lets consecutive small-m calls on
     * one x share persistent grids.  The other paths ignore them. */
    Q2K_FLAG_INDEPENDENT = 2
};

/* q2k_matmul_batched_mv - `batches` independent matrix-vector products in one
 * launch: y[b, 0, :] = W_b x[b, 0, :].
 * Page "tests/deepseek_q2_k.rs": fn quantized_matmul_q2_k_batched_mv and test
 * q2_k_batched_mv_is_byte_identical_to_independent_dispatches.
 *   x   device f32 [batches, m, k], x_elems = batches*m*k, 16-byte aligned
 *   w   device, w_bytes = batches * n*k/256*84, 4-byte aligned; batch b's
 *       [n, k] matrix starts at byte b * n*k/256*84
 *   y   device f32 [batches, m, n], y_elems = batches*m*n, 16-byte aligned;
 *       fully overwritten, must not alias x or w
 *   m   must be 1 (the pages' call passes 1: matrix-vector)
 * Each batch's y is bit-identical to q2k_matmul(m = 1) of that batch's x and W
 * alone (the same kernel and arithmetic run per batch): fp32, error within
 * 1e-5 * sum_k |x w|.  batches <= 65535.
 *   scratch  not used (see q2k_x_planes_bytes). */
q2k_status q2k_matmul_batched_mv(const float *x, size_t x_elems, const void *w, size_t w_bytes,
                                 float *y, size_t y_elems, uint32_t batches, uint32_t m,
                                 uint32_t n, uint32_t k, void *scratch, size_t scratch_bytes,
                                 q2k_stream_t stream);

/* q2k_x_planes_bytes - device bytes of scratch the batched and routed calls
 * take: 0.  Their kernels bring x into the GEMV's per-slice form per thread
 * (a few instructions per CTA), which costs less than a separate launch and
 * the wait behind it.  The `scratch` arguments of those calls are accepted
 * for compatibility and not used (any value, NULL included). */
size_t q2k_x_planes_bytes(uint32_t k, uint32_t rows);

/* q2k_matmul_id - the expert-routed product of a mixture-of-experts layer:
 * y[r, :] = W_{ids[r]} x[r / top_k, :] for every route r = t*top_k + slot.
 * Page "tests/deepseek_q2_k.rs": fn quantized_matmul_id_ggml, fn run_expert and
 * tests q2_k_expert_routed_metal_matches_reference / ..._top_k_6_...
 *   x       device f32 [n_tokens, k], x_elems = n_tokens*k, 16-byte aligned
 *   w       device, the n_experts matrices [n, k], expert e at byte
 *           e * expert_stride; w_bytes >= (n_experts - 1) * expert_stride +
 *           n*k/256*84; 4-byte aligned
 *   ids     device u32 [n_tokens * top_k], token-major (route t*top_k + slot)
 *   y       device f32 [n_tokens * top_k, n], y_elems = n_tokens*top_k*n,
 *           16-byte aligned; fully overwritten, must not alias x, w or ids
 *   bad_id_count  device u32 or NULL.  Ids live on the device, so they are
 *           checked in the kernel: a route whose id is >= n_experts gets a
 *           zero row and is counted.  With NULL the call waits for its own
 *           count and returns Q2K_ERR_BAD_ID if it is nonzero (synchronising;
 *           refused during stream capture; as q2k_embedding_gather); with a
 *           device word the count is stored there (zeroed first,
 *           stream-ordered) and the call returns without waiting: nonzero
 *           after the stream completes means the pages' error.
 * Every route runs the fp32 GEMV (error within 1e-5 * sum_k |x w|; the pages
 * allow 2e-4 absolute, 1e-2 for their reduced-precision path); each route's
 * row is bit-identical to q2k_matmul(m = 1) of its token and expert.
 * n_tokens * top_k <= 65535.
 *   scratch  not used (see q2k_x_planes_bytes). */
q2k_status q2k_matmul_id(const float *x, size_t x_elems, const void *w, size_t w_bytes,
                         const uint32_t *ids, float *y, size_t y_elems,
                         const q2k_matmul_id_params *params, uint32_t *bad_id_count,
                         void *scratch, size_t scratch_bytes, q2k_stream_t stream);

/* ---- GGUF reader (host only: no device is needed or touched) -------------
 * The tensor directory of a GGUF file (versions 2 and 3) and its tensors'
 * bytes, to load Q2_K (type 10) weights into the calls above.
 * Page "tests/deepseek_q2_k.rs": test q2_k_gguf_type_10_parses_with_exact_block_size
 * (GgufFile::open, tensor_info: ggml_type Q2_K and byte_len 84 for a 256-element
 * tensor).  A malformed file (bad magic or version, truncated entries, more than
 * 4 dimensions, an innermost extent that is not a whole number of blocks, a
 * duplicate name, data past the end of the file, an offset off the alignment)
 * is Q2K_ERR_INVALID_ARGUMENT with the reason in q2k_last_error; a file that
 * cannot be opened or read is Q2K_ERR_IO.  Calls on one open file must not run
 * concurrently (they share its read position). */
typedef struct q2k_gguf q2k_gguf;  /* an open file; opaque */

typedef struct q2k_gguf_tensor {
    uint32_t ggml_type;   /* GGML type number: 10 = Q2_K (0 = F32, 1 = F16, ...) */
    uint32_t n_dims;      /* 1 to 4 */
    uint64_t dims[4];     /* extents, innermost first (a weight matrix: dims[0] = k,
                             dims[1] = n); unused ones are 1 */
    uint64_t n_elements;  /* product of the extents */
    uint64_t offset;      /* absolute byte offset of the data in the file */
    uint64_t byte_len;    /* bytes of the data (Q2_K: n_elements / 256 * 84); 0 when
                             the reader does not know the type's block size */
} q2k_gguf_tensor;   /* 64 bytes */

/* Parse the header and tensor directory of `path`; *out is the open file
 * (close it with q2k_gguf_close), NULL on error.  Tensor data is not read. */
q2k_status q2k_gguf_open(const char *path, q2k_gguf **out);
/* Close a file q2k_gguf_open returned (NULL is ignored). */
void q2k_gguf_close(q2k_gguf *file);
/* Number of tensors in the directory (0 for NULL). */
uint64_t q2k_gguf_tensor_count(const q2k_gguf *file);
/* Name of tensor `index` in directory order, valid until the file is closed;
 * NULL when index is out of range. */
const char *q2k_gguf_tensor_name(const q2k_gguf *file, uint64_t index);
/* The directory entry of tensor `name`. */
q2k_status q2k_gguf_tensor_info(const q2k_gguf *file, const char *name,
                                q2k_gguf_tensor *out);
/* Copy tensor `name`'s bytes into host memory `dst`; dst_bytes must equal its
 * byte_len (nonzero). */
q2k_status q2k_gguf_read_tensor(const q2k_gguf *file, const char *name, void *dst,
                                size_t dst_bytes);

/* q2k_matmul_id_slotted - q2k_matmul_id with one input row per route (the
 * down projection of a MoE layer, whose input is each route's own activation):
 * y[r, :] = W_{ids[r]} x[r, :], x f32 [n_tokens, top_k, k] (x_elems =
 * n_tokens*top_k*k).  Page "tests/deepseek_q2_k.rs":
 * quantized_matmul_id_ggml_pooled_slotted and test
 * q2_k_slotted_down_mm_is_byte_identical_to_flattened_rows: the result is
 * bit-identical to q2k_matmul_id with n_tokens*top_k tokens and top_k = 1.
 * Other arguments, checks and bad-id handling as q2k_matmul_id. */
q2k_status q2k_matmul_id_slotted(const float *x, size_t x_elems, const void *w, size_t w_bytes,
                                 const uint32_t *ids, float *y, size_t y_elems,
                                 const q2k_matmul_id_params *params, uint32_t *bad_id_count,
                                 void *scratch, size_t scratch_bytes, q2k_stream_t stream);

/* q2k_matmul_id_pair - two routed products sharing x and the routing (the gate
 * and up projections of a MoE layer) in one launch: y_a = routed(W_a), y_b =
 * routed(W_b), each bit-identical to its own q2k_matmul_id.  Page
 * "tests/deepseek_q2_k.rs": quantized_matmul_id_ggml_pooled_pair (fn run_expert
 * with force_mm, whose two outputs must agree bit for bit when both weight sets
 * are the same).  w_a and w_b follow q2k_matmul_id's layout with the same
 * expert_stride (w_a_bytes and w_b_bytes checked each); y_a and y_b are
 * [n_tokens*top_k, n] with y_elems each.  A bad id is counted once per product.
 * n_tokens * top_k <= 32767. */
q2k_status q2k_matmul_id_pair(const float *x, size_t x_elems, const void *w_a, size_t w_a_bytes,
                              const void *w_b, size_t w_b_bytes, const uint32_t *ids, float *y_a,
                              float *y_b, size_t y_elems, const q2k_matmul_id_params *params,
                              uint32_t *bad_id_count, void *scratch, size_t scratch_bytes,
                              q2k_stream_t stream);

/* Flag of q2k_matmul_id_ex: one x row per route (q2k_matmul_id_slotted). */
#define Q2K_ID_SLOTTED 1u

/* q2k_matmul_id_ex - q2k_matmul_id (or, with Q2K_ID_SLOTTED in `flags`,
 * q2k_matmul_id_slotted) on a chosen path.  Page "tests/deepseek_q2_k.rs":
 * fn run_expert, whose public routed product with more than 32 tokens (and the
 * forced mm_id path) is held to 1e-2 instead of 2e-4: it multiplies many routes
 * per expert as a matrix product.
 *   Q2K_PATH_GEMV    as q2k_matmul_id; workspace = its scratch (NULL allowed)
 *   Q2K_PATH_TENSOR  routes grouped per expert into 128-row tiles, each tile
 *                    multiplied on the bf16 tensor cores with fp32 accumulation
 *                    (error within 8e-3 * sum_k |x w| per element, as
 *                    q2k_matmul_path's tensor path); needs a workspace of
 *                    q2k_matmul_id_workspace_bytes(Q2K_PATH_TENSOR, ...) bytes,
 *                    16-byte aligned, aliasing no other argument, and
 *                    n_experts <= 4096.  Not a bit-for-bit match of the GEMV.
 *   Q2K_PATH_AUTO    the tensor path when n_tokens > 32 (and n_experts <=
 *                    4096), else the GEMV
 * Other arguments, checks and bad-id handling as q2k_matmul_id: a bad id's
 * route is a zero row and counted.  An unknown path or flag bit is
 * Q2K_ERR_INVALID_ARGUMENT; so is a tensor-path call without a large enough
 * workspace. */
q2k_status q2k_matmul_id_ex(q2k_path path, uint32_t flags, const float *x, size_t x_elems,
                            const void *w, size_t w_bytes, const uint32_t *ids, float *y,
                            size_t y_elems, const q2k_matmul_id_params *params,
                            uint32_t *bad_id_count, void *workspace, size_t workspace_bytes,
                            q2k_stream_t stream);

/* q2k_matmul_id_pair_ex - q2k_matmul_id_pair on a chosen path, as
 * q2k_matmul_id_ex (page fn run_expert with force_mm runs the pair on its matrix
 * path).  On the tensor path the routes are grouped and x gathered once, and one
 * GEMM per weight set reads the shared tiles: y_a and y_b each within 8e-3 *
 * sum_k |x w|, and bit-identical to two q2k_matmul_id_ex tensor calls.  The
 * tensor path's workspace is q2k_matmul_id_workspace_bytes(Q2K_PATH_TENSOR, 0,
 * params) bytes; on the GEMV path the workspace is q2k_matmul_id_pair's optional
 * scratch.  A bad id is counted once per product. */
q2k_status q2k_matmul_id_pair_ex(q2k_path path, const float *x, size_t x_elems, const void *w_a,
                                 size_t w_a_bytes, const void *w_b, size_t w_b_bytes,
                                 const uint32_t *ids, float *y_a, float *y_b, size_t y_elems,
                                 const q2k_matmul_id_params *params, uint32_t *bad_id_count,
                                 void *workspace, size_t workspace_bytes, q2k_stream_t stream);

/* q2k_matmul_id_workspace_bytes - the workspace q2k_matmul_id_ex takes on
 * `path` (AUTO resolved as there) for these params and flags: for the tensor
 * path the routes' tile table and the bf16 image of their x rows, about
 * (n_tokens*top_k + 128*min(n_experts, n_tokens*top_k)) * (2k + 4) bytes plus
 * 4 per route; for
 * the GEMV its optional scratch (q2k_x_planes_bytes).  0 for invalid params,
 * more than 65535 routes, or a tensor path with n_experts > 4096.  Geometry
 * only: no device is touched. */
size_t q2k_matmul_id_workspace_bytes(q2k_path path, uint32_t flags,
                                     const q2k_matmul_id_params *params);

/* q2k_matmul_workspace_bytes - device bytes of workspace q2k_matmul_ex can use
 * for this geometry and path (0: the path takes none).  The tensor-core path
 * stores x there as bf16 in the tile layout its shared memory uses,
 * ceil(m / 256) * 256 * k * 2 bytes; when m <= 128 and n is small (fewer than
 * 64 tiles of 128 weight rows) it splits K into P parts (P <= 8, fixed by m, n
 * and k) and adds P * m * n * 4 bytes (after 256-byte alignment) for the
 * parts' results plus one 4-byte arrival counter per 128 x 128 output tile;
 * the last part to finish a tile sums the parts in part order, so y does not
 * depend on their timing.  Returns 0 for invalid params. */
size_t q2k_matmul_workspace_bytes(const q2k_matmul_params *params, q2k_path path);

/* q2k_matmul_ex - q2k_matmul_path plus `flags` (a mask of Q2K_FLAG_*; unknown
 * bits are rejected) and an optional caller-owned workspace.
 *   workspace        device, NULL or at least q2k_matmul_workspace_bytes(params,
 *                    path) bytes, 16-byte aligned, not overlapping x, w or y.
 *                    Its contents on entry do not matter and are clobbered.
 *                    With it the tensor-core path converts x once in a prepass
 *                    and streams it into the GEMM by bulk copies.  Without it
 *                    (and in q2k_matmul / q2k_matmul_path) the library uses a
 *                    scratch of its own, 32 MiB per device, for the same
 *                    kernel when the x image fits (e.g. m <= 2048 at k = 7168,
 *                    m <= 1024 at k = 14336): same bits as with a workspace.
 *                    Such calls take turns on the GPU (each waits, through an
 *                    event, for the previous one to finish with the scratch),
 *                    so calls on different streams do not overlap there.
 *                    Inside a stream capture, or when the image does not fit,
 *                    the GEMM converts x itself instead (within the same
 *                    tolerance, not the same bits).
 *   workspace_bytes  its size (ignored when workspace is NULL).
 * Same arguments, sizes, errors and tolerances otherwise.  Calls on different
 * streams must not share a workspace while both may run. */
q2k_status q2k_matmul_ex(q2k_path path, uint32_t flags, const float *x, size_t x_elems,
                         const void *w, size_t w_bytes, float *y, size_t y_elems,
                         const q2k_matmul_params *params, void *workspace,
                         size_t workspace_bytes, q2k_stream_t stream);

/* One call of q2k_matmul_ex, for q2k_matmul_ex_batch (88 bytes). */
typedef struct q2k_matmul_call {
    const float *x;               /* as q2k_matmul_ex */
    size_t x_elems;
    const void *w;
    size_t w_bytes;
    float *y;
    size_t y_elems;
    q2k_matmul_params params;
    void *workspace;              /* NULL or as q2k_matmul_ex */
    size_t workspace_bytes;
    uint32_t path;                /* a q2k_path */
    uint32_t flags;               /* a mask of Q2K_FLAG_* */
} q2k_matmul_call;

/* q2k_matmul_ex_batch - `count` q2k_matmul_ex calls enqueued in order on one
 * stream with one crossing of the boundary (for the many projections of a
 * decode step: the host cost per call falls from a binding's argument handling
 * to the launch itself).  Every call is checked first; the first malformed
 * one returns its q2k_matmul_ex error (the message names its index) and
 * nothing is launched.  Results are those of the separate calls, bit for bit,
 * except in the runs of independent small-m calls described below (same
 * tolerance, still deterministic).  Calls may share a workspace (they run in
 * stream order).  `calls` is host memory, read during the call only.
 *   scratch  device, NULL or at least q2k_matmul_batch_scratch_bytes(calls,
 *            count) bytes, 16-byte aligned, not overlapping any call's
 *            buffers.  With it, m = 1 calls on the fp32 GEMV path (k <= 16384)
 *            that read the same x row bring x into the GEMV's per-slice form once,
 *            into the scratch, instead of once per CTA of every call (the
 *            same values: same bits).  A call of the batch that writes that
 *            row ends the sharing.  Without it (or smaller) every call
 *            converts x itself, and no run (below) is formed.
 * A tensor-path call with Q2K_FLAG_INDEPENDENT right after a tensor-path call
 * with the same x pointer, m, k and workspace (and, for both, the workspace
 * layout of one K part: m > 64 and no K split) finds x's bf16 image in that
 * workspace already: it skips the conversion and, independent of the call
 * before it by the flag's promise, may run beside that call on the SMs it
 * leaves free; it still completes after it.  Same bits as the separate call.
 * Tensor-path calls with Q2K_FLAG_INDEPENDENT and m <= 64 that follow one
 * another with the same x pointer, m and k (k a multiple of 1024, each W
 * 16-byte aligned, no call's y overlapping x) form a run when they have at
 * least 128 tiles of 128 weight rows between them and there is scratch: x is
 * converted to bf16 once, into the scratch, and the run's calls share
 * persistent grids (one per at most 32 calls) in which each CTA takes one
 * tile after another over all of k, instead of one launch per call with k
 * split into parts.  Each output is then a single fp32 accumulation over k
 * (the even and the odd 64-k stages in two sums, added in that order): within
 * the tensor path's 8e-3 * sum_k |x w| bound, and the same bits on every run,
 * though not the bits of the separate call. */
q2k_status q2k_matmul_ex_batch(const q2k_matmul_call *calls, size_t count, void *scratch,
                               size_t scratch_bytes, q2k_stream_t stream);

/* q2k_matmul_batch_scratch_bytes - device bytes of scratch q2k_matmul_ex_batch
 * uses for these calls (0: none, or malformed calls). */
size_t q2k_matmul_batch_scratch_bytes(const q2k_matmul_call *calls, size_t count);

/* q2k_matmul_static_workspace - the tensor-core matmul (as q2k_matmul_path
 * with Q2K_PATH_TENSOR and a workspace) for callers that cannot allocate
 * device memory at the point of the call: code being captured into a CUDA
 * graph, where an allocation would break or serialise the capture; hosts or
 * plugin interfaces that hand over only the input and output buffers and own
 * the device memory budget; real-time loops that must not call the allocator.
 * The pages have no counterpart of this call; it is this library's own.
 *   The x tile image normally kept in a caller workspace goes into a fixed
 *   array inside the library instead, Q2K_STATIC_WORKSPACE_BYTES (8 MiB) on
 *   every GPU that loads the library, held until the process exits.  It fits
 *   q2k_matmul_workspace_bytes(params, Q2K_PATH_TENSOR) <= 8 MiB (e.g. m = 512,
 *   k = 7168); larger geometries are rejected with Q2K_ERR_INVALID_ARGUMENT.
 *   Nothing is allocated by the call.  The first call on a device looks up the
 *   array's device address (with that device current); make that first call
 *   before any stream capture.  The address is kept once found; a lookup that
 *   fails returns Q2K_ERR_CUDA and is tried again by the next call.
 *   All calls share the one array: calls whose work may overlap on the GPU
 *   (different streams, different host threads without ordering) race on it
 *   and give wrong results; serialise them, e.g. on one stream.  Leftovers
 *   of earlier calls do not matter: each call rewrites every byte whose value
 *   reaches y (image rows past m are read but feed only dropped outputs).
 * Arguments, sizes, errors and tolerance (8e-3 * sum_k |x w|) as q2k_matmul. */
enum { Q2K_STATIC_WORKSPACE_BYTES = 8388608 };
q2k_status q2k_matmul_static_workspace(const float *x, size_t x_elems, const void *w,
                                       size_t w_bytes, float *y, size_t y_elems,
                                       const q2k_matmul_params *params, q2k_stream_t stream);

/* q2k_selftest_wait_timeout - exercise the library's bounded on-chip wait
 * (the pages have no counterpart: this library's own failure detection).
 * Enqueues on `stream` one small kernel that waits on a barrier nothing
 * completes, giving up after about limit_us microseconds (1..100000): it then
 * sets the time-out bit of the device error word and returns, without
 * faulting or hanging.  A following q2k_device_error reports that bit (and
 * clears it).  Q2K_ERR_INVALID_ARGUMENT for a limit out of range. */
q2k_status q2k_selftest_wait_timeout(uint32_t limit_us, q2k_stream_t stream);

/* q2k_device_error - read and clear the library's device error word on the
 * current device.  Kernels that wait on on-chip barriers give up after about a
 * second, set a bit here and return instead of hanging.  Synchronises
 * `stream`.  *out = 0 means no kernel gave up since the last read. */
q2k_status q2k_device_error(uint32_t *out, q2k_stream_t stream);

/* Message for the last non-OK status returned on this thread ("" if none). */
const char *q2k_last_error(void);

/* ABI version of this header (bumped on any incompatible change). */
int q2k_abi_version(void);

#define Q2K_ABI_VERSION 1

#ifdef __cplusplus
}
#endif

#endif /* Q2K_H */
