// C ABI of libq2k (declared in include/q2k.h): argument checks and dispatch.
//
// The checks follow the conventions of the mlx-native pages: exact byte
// lengths with overflow-checked products (page "src/ops/dflash2_selector.rs",
// fns product / require), outputs that may not alias inputs (fn
// validate_disjoint), and InvalidArgument before anything is launched (page
// "tests/deepseek_q2_k.rs", tests q2_k_host_decode_rejects_malformed_buffers
// and ..._rejects_bad_ids).
#include <cuda_runtime.h>

#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "q2k.h"
#include "q2k_internal.h"

static_assert(Q2K_STATIC_WORKSPACE_BYTES == q2k::kStaticWorkspaceBytes,
              "header and library disagree on the fixed scratch size");
static_assert(sizeof(q2k_matmul_id_params) == 32, "q2k_matmul_id_params layout");
static_assert(sizeof(q2k_matmul_call) == 88, "q2k_matmul_call layout");

namespace {

thread_local char g_last_error[512] = "";

q2k_status fail(q2k_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return s;
}

q2k_status cuda_fail(cudaError_t e, const char* what) {
    return fail(Q2K_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool mul_ok(size_t a, size_t b, size_t* out) {
    if (a != 0 && b > SIZE_MAX / a) return false;
    *out = a * b;
    return true;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlaps(const void* a, size_t a_bytes, const void* b, size_t b_bytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a_bytes != 0 && b_bytes != 0 && a0 < b0 + b_bytes && b0 < a0 + a_bytes;
}

struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
};

// The current device must be a compute capability 10.3 part (the library is
// built for sm_103a only).  The SM count is cached per device.
q2k_status current_device(DeviceInfo* info) {
    static int sm_cache[64];
    static int cc_cache[64];
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(Q2K_ERR_NO_DEVICE, "device ordinal %d out of range", dev);
    if (sm_cache[dev] == 0) {
        int major = 0, minor = 0, sms = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        cc_cache[dev] = major * 10 + minor;
        sm_cache[dev] = sms;
    }
    if (cc_cache[dev] != 103)
        return fail(Q2K_ERR_NO_DEVICE, "device %d has compute capability %d.%d; libq2k is built for sm_103a",
                    dev, cc_cache[dev] / 10, cc_cache[dev] % 10);
    info->device = dev;
    info->sm_count = sm_cache[dev];
    return Q2K_OK;
}

// ---- bad ids reported as a status (bad_id_count == NULL) --------------------
//
// The pages' gather and routed calls fail with an error for an id out of
// range.  Ids live on the device here, so the kernel counts them; a caller
// that passes no counter of its own gets the count in one of these words,
// read back (4 bytes) and waited for before the call returns
// Q2K_ERR_BAD_ID or Q2K_OK.  Each call in flight holds its own word.
constexpr int kStatusWords = 64;
__device__ unsigned int g_status_words[kStatusWords];

struct StatusWords {
    std::mutex mu;
    unsigned int* base[64] = {};  // device address of g_status_words, per device
    uint64_t used[64] = {};       // words held by calls in flight, per device
};

StatusWords& status_words() {
    static StatusWords s;
    return s;
}

// A free status word on `device` (current), zeroed on `stream`.
q2k_status acquire_status_word(int device, cudaStream_t stream, unsigned int** word, int* slot) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cs);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    if (cs != cudaStreamCaptureStatusNone)
        return fail(Q2K_ERR_INVALID_ARGUMENT,
                    "bad_id_count is required while the stream is being captured (without it the "
                    "call waits for its own result)");
    StatusWords& s = status_words();
    {
        std::lock_guard<std::mutex> lk(s.mu);
        if (s.base[device] == nullptr) {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_status_words);
            if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status words)");
            s.base[device] = static_cast<unsigned int*>(p);
        }
        *slot = -1;
        for (int i = 0; i < kStatusWords; ++i)
            if (((s.used[device] >> i) & 1u) == 0) {
                s.used[device] |= uint64_t(1) << i;
                *slot = i;
                break;
            }
        if (*slot < 0)
            return fail(Q2K_ERR_INVALID_ARGUMENT,
                        "more than %d calls without bad_id_count in flight on device %d",
                        kStatusWords, device);
        *word = s.base[device] + *slot;
    }
    e = cudaMemsetAsync(*word, 0, 4, stream);
    if (e != cudaSuccess) {
        std::lock_guard<std::mutex> lk(s.mu);
        s.used[device] &= ~(uint64_t(1) << *slot);
        return cuda_fail(e, "clearing the bad-id status word");
    }
    return Q2K_OK;
}

// Read the word back after the call's kernels (waits for `stream`), free it,
// and turn a nonzero count into Q2K_ERR_BAD_ID.  `launched` is the launch
// status: on failure the word is freed once the stream has drained.
q2k_status finish_status_word(int device, int slot, unsigned int* word, cudaStream_t stream,
                              cudaError_t launched, const char* what, const char* limit_name,
                              uint32_t limit) {
    unsigned int count = 0;
    cudaError_t e = launched;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&count, word, 4, cudaMemcpyDeviceToHost, stream);
    const cudaError_t sync = cudaStreamSynchronize(stream);
    if (e == cudaSuccess) e = sync;
    {
        StatusWords& s = status_words();
        std::lock_guard<std::mutex> lk(s.mu);
        s.used[device] &= ~(uint64_t(1) << slot);
    }
    if (e != cudaSuccess) return cuda_fail(e, what);
    if (count != 0)
        return fail(Q2K_ERR_BAD_ID, "%u id(s) out of range (>= %s = %u); their rows are zeros",
                    count, limit_name, limit);
    return Q2K_OK;
}

q2k_status check_matmul(const float* x, size_t x_elems, const void* w, size_t w_bytes,
                        const float* y, size_t y_elems, const q2k_matmul_params* p) {
    if (p == nullptr) return fail(Q2K_ERR_INVALID_ARGUMENT, "params is NULL");
    if (p->ggml_type != Q2K_GGML_TYPE_Q2_K)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "ggml_type %u is not Q2_K (10)", p->ggml_type);
    if (p->m == 0 || p->n == 0 || p->k == 0)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "m, n, k must be >= 1 (got %u, %u, %u)", p->m, p->n, p->k);
    if (p->k % Q2K_QK_K != 0)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "k = %u is not a multiple of 256", p->k);
    if (p->m > INT_MAX || p->n > INT_MAX || p->k > INT_MAX)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "m, n, k must fit in a signed 32-bit int");
    size_t want_x, want_w, want_y, blocks;
    if (!mul_ok(p->m, p->k, &want_x) || !mul_ok(p->n, p->k / Q2K_QK_K, &blocks) ||
        !mul_ok(blocks, Q2K_BLOCK_BYTES, &want_w) || !mul_ok(p->m, p->n, &want_y) ||
        want_x > SIZE_MAX / 4 || want_y > SIZE_MAX / 4)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "matmul shape overflows size_t");
    if (x == nullptr || w == nullptr || y == nullptr)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "x, w and y must be non-NULL");
    if (x_elems != want_x)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "x has %zu elements, expected m*k = %zu", x_elems, want_x);
    if (w_bytes != want_w)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "w has %zu bytes, expected n*k/256*84 = %zu", w_bytes, want_w);
    if (y_elems != want_y)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "y has %zu elements, expected m*n = %zu", y_elems, want_y);
    if (!aligned(x, 16) || !aligned(y, 16) || !aligned(w, 4))
        return fail(Q2K_ERR_INVALID_ARGUMENT, "x and y must be 16-byte aligned and w 4-byte aligned");
    if (overlaps(y, want_y * 4, x, want_x * 4) || overlaps(y, want_y * 4, w, want_w))
        return fail(Q2K_ERR_INVALID_ARGUMENT, "y must not alias x or w");
    return Q2K_OK;
}

// The batched and routed calls' optional scratch argument: accepted for ABI
// compatibility and not used (their kernels convert x per thread; see
// q2k_x_planes_bytes).
q2k_status check_planes_scratch(void* scratch, size_t scratch_bytes, uint32_t k, size_t rows,
                                const void* x, size_t x_bytes, const void* w, size_t w_bytes,
                                const void* y, size_t y_bytes, uint8_t** planes) {
    (void)scratch, (void)scratch_bytes, (void)k, (void)rows, (void)x, (void)x_bytes, (void)w;
    (void)w_bytes, (void)y, (void)y_bytes;
    *planes = nullptr;
    return Q2K_OK;
}

}  // namespace

void q2k::set_last_error(const char* msg) {
    snprintf(g_last_error, sizeof g_last_error, "%s", msg);
}

extern "C" {

const char* q2k_last_error(void) { return g_last_error; }

int q2k_abi_version(void) { return Q2K_ABI_VERSION; }

q2k_status q2k_dequantize(const void* blocks, size_t blocks_bytes, float* out, size_t out_elems,
                          q2k_stream_t stream) {
    g_last_error[0] = '\0';
    if (blocks == nullptr || out == nullptr)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "blocks and out must be non-NULL");
    if (blocks_bytes == 0 || blocks_bytes % Q2K_BLOCK_BYTES != 0)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "%zu bytes is not a positive whole number of 84-byte Q2_K blocks",
                    blocks_bytes);
    const size_t n_blocks = blocks_bytes / Q2K_BLOCK_BYTES;
    size_t want;
    if (!mul_ok(n_blocks, Q2K_QK_K, &want) || want > SIZE_MAX / 4)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "output size overflows size_t");
    if (out_elems != want)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "out has %zu floats, expected %zu (256 per block)", out_elems, want);
    if (!aligned(blocks, 4) || !aligned(out, 16))
        return fail(Q2K_ERR_INVALID_ARGUMENT, "blocks must be 4-byte and out 16-byte aligned");
    if (overlaps(out, want * 4, blocks, blocks_bytes))
        return fail(Q2K_ERR_INVALID_ARGUMENT, "out must not alias blocks");
    DeviceInfo dev;
    q2k_status st = current_device(&dev);
    if (st != Q2K_OK) return st;
    cudaError_t e = q2k::launch_dequant(static_cast<const uint8_t*>(blocks), out, n_blocks,
                                        dev.sm_count, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? Q2K_OK : cuda_fail(e, "q2k_dequantize launch");
}

q2k_status q2k_embedding_gather(const void* table, size_t table_bytes, const uint32_t* ids,
                                float* out, size_t out_elems, const q2k_embedding_params* p,
                                uint32_t* bad_id_count, q2k_stream_t stream) {
    g_last_error[0] = '\0';
    if (p == nullptr) return fail(Q2K_ERR_INVALID_ARGUMENT, "params is NULL");
    if (p->ggml_type != Q2K_GGML_TYPE_Q2_K)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "ggml_type %u is not Q2_K (10)", p->ggml_type);
    if (p->vocab_size == 0 || p->embed_dim == 0 || p->n_tokens == 0)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "vocab_size, embed_dim and n_tokens must be >= 1");
    if (p->embed_dim % Q2K_QK_K != 0)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "embed_dim = %u is not a multiple of 256", p->embed_dim);
    if (table == nullptr || ids == nullptr || out == nullptr)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "table, ids and out must be non-NULL");
    size_t blocks, want_table, want_out;
    if (!mul_ok(p->vocab_size, p->embed_dim / Q2K_QK_K, &blocks) ||
        !mul_ok(blocks, Q2K_BLOCK_BYTES, &want_table) || !mul_ok(p->n_tokens, p->embed_dim, &want_out) ||
        want_out > SIZE_MAX / 4)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "gather shape overflows size_t");
    if (table_bytes != want_table)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "table has %zu bytes, expected vocab*embed_dim/256*84 = %zu",
                    table_bytes, want_table);
    if (out_elems != want_out)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "out has %zu floats, expected n_tokens*embed_dim = %zu",
                    out_elems, want_out);
    if (!aligned(table, 4) || !aligned(out, 16) || !aligned(ids, 4) ||
        (bad_id_count != nullptr && !aligned(bad_id_count, 4)))
        return fail(Q2K_ERR_INVALID_ARGUMENT, "table, ids and bad_id_count must be 4-byte and out 16-byte aligned");
    const size_t out_bytes = want_out * 4;
    if (overlaps(out, out_bytes, table, want_table) || overlaps(out, out_bytes, ids, size_t(p->n_tokens) * 4) ||
        (bad_id_count != nullptr &&
         (overlaps(bad_id_count, 4, out, out_bytes) || overlaps(bad_id_count, 4, ids, size_t(p->n_tokens) * 4) ||
          overlaps(bad_id_count, 4, table, want_table))))
        return fail(Q2K_ERR_INVALID_ARGUMENT, "writable buffers must not alias inputs or each other");
    DeviceInfo dev;
    q2k_status st = current_device(&dev);
    if (st != Q2K_OK) return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned int* word = nullptr;
    int slot = -1;
    if (bad_id_count == nullptr) {
        st = acquire_status_word(dev.device, s, &word, &slot);
        if (st != Q2K_OK) return st;
    }
    cudaError_t e = q2k::launch_gather(static_cast<const uint8_t*>(table), ids, out, p->vocab_size,
                                       p->embed_dim, p->n_tokens,
                                       bad_id_count != nullptr ? bad_id_count : word, dev.sm_count, s);
    if (word != nullptr)
        return finish_status_word(dev.device, slot, word, s, e, "q2k_embedding_gather",
                                  "vocab_size", p->vocab_size);
    return e == cudaSuccess ? Q2K_OK : cuda_fail(e, "q2k_embedding_gather launch");
}

size_t q2k_matmul_workspace_bytes(const q2k_matmul_params* p, q2k_path path) {
    if (p == nullptr || p->ggml_type != Q2K_GGML_TYPE_Q2_K || p->m == 0 || p->n == 0 || p->k == 0 ||
        p->k % Q2K_QK_K != 0 || p->m > INT_MAX || p->n > INT_MAX || p->k > INT_MAX)
        return 0;
    if (path == Q2K_PATH_AUTO) path = p->m <= 8 ? Q2K_PATH_GEMV : Q2K_PATH_TENSOR;
    if (path != Q2K_PATH_TENSOR) return 0;
    const size_t m_pad = (static_cast<size_t>(p->m) + 255) / 256 * 256;
    if (m_pad > SIZE_MAX / 2 / p->k) return 0;
    return q2k::gemm_tc_workspace_bytes(int(p->m), int(p->n), int(p->k));
}

}  // extern "C"

namespace {

// q2k_matmul_ex's checks: on success *path_out is the resolved path and
// *ws_out the workspace to use (NULL when none).  Nothing is launched.
q2k_status check_matmul_ex(q2k_path path, uint32_t flags, const float* x, size_t x_elems,
                           const void* w, size_t w_bytes, const float* y, size_t y_elems,
                           const q2k_matmul_params* p, void* workspace, size_t workspace_bytes,
                           q2k_path* path_out, void** ws_out) {
    q2k_status st = check_matmul(x, x_elems, w, w_bytes, y, y_elems, p);
    if (st != Q2K_OK) return st;
    if ((flags & ~static_cast<uint32_t>(Q2K_FLAG_CONST_WEIGHTS | Q2K_FLAG_INDEPENDENT)) != 0)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "unknown flag bits 0x%x", flags);
    if (path != Q2K_PATH_AUTO && path != Q2K_PATH_GEMV && path != Q2K_PATH_TENSOR)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "unknown path %d", static_cast<int>(path));
    if (path == Q2K_PATH_AUTO) path = p->m <= 8 ? Q2K_PATH_GEMV : Q2K_PATH_TENSOR;
    void* ws = nullptr;
    if (workspace != nullptr && path == Q2K_PATH_TENSOR) {
        const size_t need = q2k::gemm_tc_workspace_bytes(int(p->m), int(p->n), int(p->k));
        if (workspace_bytes < need)
            return fail(Q2K_ERR_INVALID_ARGUMENT, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
        if (!aligned(workspace, 16))
            return fail(Q2K_ERR_INVALID_ARGUMENT, "workspace must be 16-byte aligned");
        if (overlaps(workspace, need, x, size_t(p->m) * p->k * 4) ||
            overlaps(workspace, need, w, w_bytes) || overlaps(workspace, need, y, size_t(p->m) * p->n * 4))
            return fail(Q2K_ERR_INVALID_ARGUMENT, "workspace must not alias x, w or y");
        ws = workspace;
    }
    if (path == Q2K_PATH_GEMV && (p->m + 7u) / 8u > 65535u)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "GEMV path supports m <= 524280");
    if (path == Q2K_PATH_TENSOR && (p->m + 127u) / 128u > 65535u)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "tensor-core path supports m <= 8388480");
    *path_out = path;
    *ws_out = ws;
    return Q2K_OK;
}

// Enqueue one checked call.
cudaError_t launch_matmul_ex(q2k_path path, uint32_t flags, const float* x, const void* w, float* y,
                             const q2k_matmul_params* p, void* ws, const DeviceInfo& dev,
                             cudaStream_t s, bool image_ready = false) {
    const uint8_t* wb = static_cast<const uint8_t*>(w);
    if (path == Q2K_PATH_GEMV)
        return q2k::launch_gemv(x, wb, y, int(p->m), int(p->n), int(p->k), dev.device, dev.sm_count,
                                ((flags & Q2K_FLAG_CONST_WEIGHTS) ? q2k::kGemvConstWeights : 0u) |
                                    ((flags & Q2K_FLAG_INDEPENDENT) ? q2k::kGemvIndependent : 0u),
                                s);
    const uint32_t kf = ((flags & Q2K_FLAG_CONST_WEIGHTS) ? q2k::kGemvConstWeights : 0u) |
                        ((flags & Q2K_FLAG_INDEPENDENT) ? q2k::kGemvIndependent : 0u);
    if (ws == nullptr)
        return q2k::launch_gemm_tc_plain(x, wb, y, int(p->m), int(p->n), int(p->k), dev.device,
                                         dev.sm_count, s, kf);
    return q2k::launch_gemm_tc(x, wb, y, int(p->m), int(p->n), int(p->k), dev.device, dev.sm_count, ws,
                               s, kf | (image_ready ? q2k::kImageReady : 0u));
}

}  // namespace

extern "C" {

q2k_status q2k_matmul_ex(q2k_path path, uint32_t flags, const float* x, size_t x_elems,
                         const void* w, size_t w_bytes, float* y, size_t y_elems,
                         const q2k_matmul_params* p, void* workspace, size_t workspace_bytes,
                         q2k_stream_t stream) {
    g_last_error[0] = '\0';
    q2k_path rpath;
    void* ws;
    q2k_status st = check_matmul_ex(path, flags, x, x_elems, w, w_bytes, y, y_elems, p, workspace,
                                    workspace_bytes, &rpath, &ws);
    if (st != Q2K_OK) return st;
    DeviceInfo dev;
    st = current_device(&dev);
    if (st != Q2K_OK) return st;
    cudaError_t e = launch_matmul_ex(rpath, flags, x, w, y, p, ws, dev, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? Q2K_OK : cuda_fail(e, "q2k_matmul launch");
}

}  // extern "C"

namespace {

// Which calls of a batch convert x once: m = 1 GEMV calls reading the same x
// row (same pointer and k) form a group until a call of the batch writes that
// row; groups of two or more calls get a 256-byte-aligned slot of the scratch.
struct BatchPlan {
    std::vector<q2k_path> path;
    std::vector<void*> ws;
    std::vector<int> group;          // per call: its group or -1
    std::vector<size_t> slot;        // per group: scratch offset (SIZE_MAX: alone, no slot)
    std::vector<int> run;            // per call: the length of the run it starts, else 0
    std::vector<size_t> run_slot;    // per call starting a run: its x image's scratch offset
    size_t scratch = 0;
};

// Independent tensor-path calls with m <= 64 (the small-m mode) that follow
// one another on the same x (same pointer, m and k) form a run when their
// weight tiles are enough to give every SM several: the run converts x once
// and runs as persistent grids (q2k::launch_gemm_tc_multi) instead of one
// launch per call.  A call whose output overlaps x ends the run before it.
constexpr int kMultiMinTiles = 128;

bool multi_member(const q2k_matmul_call& c, q2k_path path) {
    return path == Q2K_PATH_TENSOR && (c.flags & Q2K_FLAG_INDEPENDENT) &&
           q2k::gemm_tc_multi_eligible(int(c.params.m), int(c.params.k), c.w) &&
           !overlaps(c.y, c.y_elems * 4, c.x, size_t(c.params.m) * c.params.k * 4);
}

q2k_status plan_batch(const q2k_matmul_call* calls, size_t count, BatchPlan* bp) {
    bp->path.resize(count);
    bp->ws.resize(count);
    bp->group.assign(count, -1);
    struct Open { const float* x; uint32_t k; int id; };
    std::vector<Open> open;
    std::vector<int> uses;
    std::vector<uint32_t> ks;
    for (size_t i = 0; i < count; ++i) {
        const q2k_matmul_call& c = calls[i];
        q2k_status st = check_matmul_ex(static_cast<q2k_path>(c.path), c.flags, c.x, c.x_elems, c.w,
                                        c.w_bytes, c.y, c.y_elems, &c.params, c.workspace,
                                        c.workspace_bytes, &bp->path[i], &bp->ws[i]);
        if (st != Q2K_OK) {
            // prefix the message with the call's index (a long message loses its tail)
            char msg[sizeof g_last_error];
            const int head = snprintf(msg, sizeof msg, "call %zu: ", i);
            if (head > 0 && static_cast<size_t>(head) < sizeof msg) {
                const size_t room = sizeof msg - static_cast<size_t>(head) - 1;
                strncpy(msg + head, g_last_error, room);
                msg[sizeof msg - 1] = '\0';
                memcpy(g_last_error, msg, sizeof msg);
            }
            return st;
        }
        if (bp->path[i] == Q2K_PATH_GEMV && q2k::gemv_shares_planes(int(c.params.m), int(c.params.k))) {
            int id = -1;
            for (const Open& o : open)
                if (o.x == c.x && o.k == c.params.k) id = o.id;
            if (id < 0) {
                id = static_cast<int>(uses.size());
                uses.push_back(0);
                ks.push_back(c.params.k);
                open.push_back({c.x, c.params.k, id});
            }
            ++uses[id];
            bp->group[i] = id;
        }
        // this call's output ends every group whose x it overlaps
        const size_t y_bytes = c.y_elems * 4;
        for (size_t j = 0; j < open.size();)
            if (overlaps(c.y, y_bytes, open[j].x, size_t(open[j].k) * 4)) open.erase(open.begin() + j);
            else ++j;
    }
    bp->slot.assign(uses.size(), SIZE_MAX);
    for (size_t g = 0; g < uses.size(); ++g)
        if (uses[g] >= 2) {
            bp->slot[g] = bp->scratch;
            bp->scratch += (q2k::gemv_planes_bytes(int(ks[g])) + 255) & ~size_t(255);
        }
    bp->run.assign(count, 0);
    bp->run_slot.assign(count, SIZE_MAX);
    for (size_t i = 0; i < count;) {
        const q2k_matmul_call& c = calls[i];
        if (!multi_member(c, bp->path[i])) {
            ++i;
            continue;
        }
        size_t j = i;
        long tiles = 0;
        while (j < count && multi_member(calls[j], bp->path[j]) && calls[j].x == c.x &&
               calls[j].params.m == c.params.m && calls[j].params.k == c.params.k) {
            tiles += (calls[j].params.n + 127) / 128;
            ++j;
        }
        if (j - i >= 2 && tiles >= kMultiMinTiles) {
            bp->run[i] = static_cast<int>(j - i);
            bp->run_slot[i] = bp->scratch;
            bp->scratch += (q2k::gemm_tc_multi_scratch_bytes(int(c.params.m), int(c.params.k)) + 255) &
                           ~size_t(255);
        }
        i = j;
    }
    return Q2K_OK;
}

}  // namespace

extern "C" {

size_t q2k_matmul_batch_scratch_bytes(const q2k_matmul_call* calls, size_t count) {
    if (calls == nullptr || count == 0) return 0;
    BatchPlan bp;
    return plan_batch(calls, count, &bp) == Q2K_OK ? bp.scratch : 0;
}

q2k_status q2k_matmul_ex_batch(const q2k_matmul_call* calls, size_t count, void* scratch,
                               size_t scratch_bytes, q2k_stream_t stream) {
    g_last_error[0] = '\0';
    if (count == 0) return Q2K_OK;
    if (calls == nullptr) return fail(Q2K_ERR_INVALID_ARGUMENT, "calls is NULL");
    BatchPlan bp;
    q2k_status st = plan_batch(calls, count, &bp);
    if (st != Q2K_OK) return st;
    // without room for every slot, every call converts x itself
    const bool share = scratch != nullptr && scratch_bytes >= bp.scratch && bp.scratch > 0;
    if (share && !aligned(scratch, 16))
        return fail(Q2K_ERR_INVALID_ARGUMENT, "scratch must be 16-byte aligned");
    if (share)
        for (size_t i = 0; i < count; ++i) {
            const q2k_matmul_call& c = calls[i];
            if (overlaps(scratch, bp.scratch, c.x, c.x_elems * 4) ||
                overlaps(scratch, bp.scratch, c.w, c.w_bytes) ||
                overlaps(scratch, bp.scratch, c.y, c.y_elems * 4) ||
                (bp.ws[i] != nullptr && overlaps(scratch, bp.scratch, bp.ws[i], c.workspace_bytes)))
                return fail(Q2K_ERR_INVALID_ARGUMENT, "scratch must not alias call %zu's buffers", i);
        }
    DeviceInfo dev;
    st = current_device(&dev);
    if (st != Q2K_OK) return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    std::vector<char> prepared(bp.slot.size(), 0);
    std::vector<q2k::MultiCall> multi;
    // (without the tensor-map encoder a run's calls go one by one)
    const bool runs = share && q2k::gemm_tc_multi_available();
    for (size_t i = 0; i < count; ++i) {
        const q2k_matmul_call& c = calls[i];
        cudaError_t e = cudaSuccess;
        if (runs && bp.run[i] > 0) {
            // a run of independent small-m calls on one x: persistent grids
            const size_t len = static_cast<size_t>(bp.run[i]);
            multi.clear();
            for (size_t j = i; j < i + len; ++j)
                multi.push_back({static_cast<const uint8_t*>(calls[j].w), calls[j].y,
                                 int(calls[j].params.n)});
            e = q2k::launch_gemm_tc_multi(c.x, int(c.params.m), int(c.params.k), multi.data(),
                                          static_cast<int>(len),
                                          static_cast<uint8_t*>(scratch) + bp.run_slot[i], dev.device,
                                          dev.sm_count, s);
            if (e != cudaSuccess) {
                char what[80];
                snprintf(what, sizeof what, "q2k_matmul_ex_batch launch of calls %zu..%zu", i,
                         i + len - 1);
                return cuda_fail(e, what);
            }
            i += len - 1;
            continue;
        }
        // A tensor call right after one with the same x, m and k in the same
        // workspace finds x's image there already: when it is independent
        // (nothing still running writes its x, W or y, the call before
        // included), it skips the conversion and may run beside that call.
        bool image_ready = false;
        if (i > 0 && bp.path[i] == Q2K_PATH_TENSOR && bp.ws[i] != nullptr &&
            (c.flags & Q2K_FLAG_INDEPENDENT)) {
            const q2k_matmul_call& q = calls[i - 1];
            image_ready = bp.path[i - 1] == Q2K_PATH_TENSOR && bp.ws[i - 1] == bp.ws[i] &&
                          q.x == c.x && q.params.m == c.params.m && q.params.k == c.params.k &&
                          q2k::gemm_tc_image_reusable(int(q.params.m), int(q.params.n), int(q.params.k)) &&
                          q2k::gemm_tc_image_reusable(int(c.params.m), int(c.params.n), int(c.params.k));
        }
        const int g = bp.group[i];
        if (share && g >= 0 && bp.slot[g] != SIZE_MAX) {
            uint8_t* planes = static_cast<uint8_t*>(scratch) + bp.slot[g];
            if (!prepared[g]) {
                e = q2k::launch_prep_x_planes(c.x, int(c.params.k), planes, s);
                prepared[g] = 1;
            }
            if (e == cudaSuccess)
                e = q2k::launch_gemv(c.x, static_cast<const uint8_t*>(c.w), c.y, 1, int(c.params.n),
                                     int(c.params.k), dev.device, dev.sm_count,
                                     ((c.flags & Q2K_FLAG_CONST_WEIGHTS) ? q2k::kGemvConstWeights : 0u) |
                                         ((c.flags & Q2K_FLAG_INDEPENDENT) ? q2k::kGemvIndependent : 0u),
                                     s, planes);
        } else {
            e = launch_matmul_ex(bp.path[i], c.flags, c.x, c.w, c.y, &c.params, bp.ws[i], dev, s,
                                 image_ready);
        }
        if (e != cudaSuccess) {
            char what[64];
            snprintf(what, sizeof what, "q2k_matmul_ex_batch launch of call %zu", i);
            return cuda_fail(e, what);
        }
    }
    return Q2K_OK;
}

q2k_status q2k_matmul_path(q2k_path path, const float* x, size_t x_elems, const void* w,
                           size_t w_bytes, float* y, size_t y_elems, const q2k_matmul_params* p,
                           q2k_stream_t stream) {
    return q2k_matmul_ex(path, 0u, x, x_elems, w, w_bytes, y, y_elems, p, nullptr, 0, stream);
}

q2k_status q2k_matmul(const float* x, size_t x_elems, const void* w, size_t w_bytes, float* y,
                      size_t y_elems, const q2k_matmul_params* p, q2k_stream_t stream) {
    return q2k_matmul_path(Q2K_PATH_AUTO, x, x_elems, w, w_bytes, y, y_elems, p, stream);
}

q2k_status q2k_matmul_static_workspace(const float* x, size_t x_elems, const void* w,
                                       size_t w_bytes, float* y, size_t y_elems,
                                       const q2k_matmul_params* p, q2k_stream_t stream) {
    g_last_error[0] = '\0';
    q2k_status st = check_matmul(x, x_elems, w, w_bytes, y, y_elems, p);
    if (st != Q2K_OK) return st;
    const size_t need = q2k::gemm_tc_workspace_bytes(int(p->m), int(p->n), int(p->k));
    if (need > q2k::kStaticWorkspaceBytes)
        return fail(Q2K_ERR_INVALID_ARGUMENT,
                    "m = %u, n = %u, k = %u needs %zu bytes of scratch; the library's fixed scratch "
                    "holds %zu",
                    p->m, p->n, p->k, need, q2k::kStaticWorkspaceBytes);
    DeviceInfo dev;
    st = current_device(&dev);
    if (st != Q2K_OK) return st;
    cudaError_t e = q2k::launch_gemm_tc_static(x, static_cast<const uint8_t*>(w), y, int(p->m),
                                               int(p->n), int(p->k), dev.device, dev.sm_count,
                                               reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? Q2K_OK : cuda_fail(e, "q2k_matmul_static_workspace launch");
}

q2k_status q2k_matmul_batched_mv(const float* x, size_t x_elems, const void* w, size_t w_bytes,
                                 float* y, size_t y_elems, uint32_t batches, uint32_t m,
                                 uint32_t n, uint32_t k, void* scratch, size_t scratch_bytes,
                                 q2k_stream_t stream) {
    g_last_error[0] = '\0';
    if (m != 1) return fail(Q2K_ERR_INVALID_ARGUMENT, "batched matrix-vector takes m = 1, got %u", m);
    if (batches == 0 || batches > 65535)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "batches must be in 1..65535, got %u", batches);
    // one batch's geometry, checked as a single call would be
    const q2k_matmul_params one = {1u, n, k, Q2K_GGML_TYPE_Q2_K};
    size_t per_w = 0, want_x, want_w, want_y;
    if (k % Q2K_QK_K == 0 && !mul_ok(size_t(n), size_t(k / Q2K_QK_K) * Q2K_BLOCK_BYTES, &per_w))
        return fail(Q2K_ERR_INVALID_ARGUMENT, "matmul shape overflows size_t");
    if (!mul_ok(batches, k, &want_x) || !mul_ok(batches, per_w, &want_w) ||
        !mul_ok(batches, n, &want_y))
        return fail(Q2K_ERR_INVALID_ARGUMENT, "batched shape overflows size_t");
    if (x_elems != want_x || w_bytes != want_w || y_elems != want_y)
        return fail(Q2K_ERR_INVALID_ARGUMENT,
                    "batched sizes: x %zu (want batches*k = %zu), w %zu (want batches*n*k/256*84 = %zu), "
                    "y %zu (want batches*n = %zu)", x_elems, want_x, w_bytes, want_w, y_elems, want_y);
    q2k_status st = check_matmul(x, k, w, per_w, y, n, &one);  // shape, type, nulls, alignment
    if (st != Q2K_OK) return st;
    if (overlaps(y, want_y * 4, x, want_x * 4) || overlaps(y, want_y * 4, w, want_w))
        return fail(Q2K_ERR_INVALID_ARGUMENT, "y must not alias x or w");
    uint8_t* planes = nullptr;
    st = check_planes_scratch(scratch, scratch_bytes, k, batches, x, want_x * 4, w, want_w, y,
                              want_y * 4, &planes);
    if (st != Q2K_OK) return st;
    DeviceInfo dev;
    st = current_device(&dev);
    if (st != Q2K_OK) return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    q2k::GemvProblems pr;
    pr.x_stride = static_cast<long long>(k);
    pr.w_stride = static_cast<long long>(per_w);
    pr.y_stride = static_cast<long long>(n);
    cudaError_t e = cudaSuccess;
    if (e == cudaSuccess)
        e = q2k::launch_gemv_problems(x, static_cast<const uint8_t*>(w), y, 1, int(n), int(k),
                                      dev.device, dev.sm_count, 0u, pr, int(batches), s, planes,
                                      planes ? uint32_t(q2k::gemv_planes_stride(int(k))) : 0u);
    return e == cudaSuccess ? Q2K_OK : cuda_fail(e, "q2k_matmul_batched_mv launch");
}

}  // extern "C"

namespace {

// Checks and launch shared by the routed products: x has one row per token
// (or per route when `slotted`); wb / yb are the second weight set and output
// of a pair (NULL otherwise).  Every malformed argument is rejected before any
// device work.
// The pages' routed product takes its matrix-matrix (reduced-precision) path
// above 32 tokens; at most 32 it runs a GEMV per route.
q2k_path routed_auto_path(const q2k_matmul_id_params* p) {
    return p->n_tokens > 32 && p->n_experts <= uint32_t(q2k::kRoutedMaxExperts) ? Q2K_PATH_TENSOR
                                                                               : Q2K_PATH_GEMV;
}

q2k_status routed_call(const float* x, size_t x_elems, bool slotted, const void* wa, size_t wa_bytes,
                       const void* wb, size_t wb_bytes, const uint32_t* ids, float* ya, float* yb,
                       size_t y_elems, const q2k_matmul_id_params* p, uint32_t* bad_id_count,
                       void* scratch, size_t scratch_bytes, q2k_stream_t stream, const char* what,
                       q2k_path path = Q2K_PATH_GEMV) {
    g_last_error[0] = '\0';
    const bool pair = yb != nullptr || wb != nullptr;
    if (p == nullptr) return fail(Q2K_ERR_INVALID_ARGUMENT, "params is NULL");
    if (p->ggml_type != Q2K_GGML_TYPE_Q2_K)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "ggml_type %u is not Q2_K (10)", p->ggml_type);
    if (p->n_tokens == 0 || p->top_k == 0 || p->n == 0 || p->k == 0 || p->n_experts == 0)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "n_tokens, top_k, n, k and n_experts must be >= 1");
    if (p->k % Q2K_QK_K != 0)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "k = %u is not a multiple of 256", p->k);
    if (p->n > INT_MAX || p->k > INT_MAX)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "n and k must fit in a signed 32-bit int");
    size_t routes, expert_bytes, want_x, want_y, last;
    if (!mul_ok(p->n_tokens, p->top_k, &routes) ||
        !mul_ok(p->n, size_t(p->k / Q2K_QK_K) * Q2K_BLOCK_BYTES, &expert_bytes) ||
        !mul_ok(slotted ? routes : size_t(p->n_tokens), p->k, &want_x) ||
        !mul_ok(routes, p->n, &want_y) ||
        !mul_ok(p->n_experts - 1u, p->expert_stride, &last) || last > SIZE_MAX - expert_bytes ||
        want_x > SIZE_MAX / 4 || want_y > SIZE_MAX / 4)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "routed shape overflows size_t");
    if (routes > (pair ? 32767u : 65535u))
        return fail(Q2K_ERR_INVALID_ARGUMENT, "n_tokens * top_k must be <= %u, got %zu",
                    pair ? 32767u : 65535u, routes);
    if (p->expert_stride % 4 != 0 || p->expert_stride < expert_bytes)
        return fail(Q2K_ERR_INVALID_ARGUMENT,
                    "expert_stride %llu must be a multiple of 4 and >= n*k/256*84 = %zu",
                    static_cast<unsigned long long>(p->expert_stride), expert_bytes);
    if (x == nullptr || wa == nullptr || ids == nullptr || ya == nullptr ||
        (pair && (wb == nullptr || yb == nullptr)))
        return fail(Q2K_ERR_INVALID_ARGUMENT, "x, w, ids and y must be non-NULL");
    if (x_elems != want_x)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "x has %zu elements, expected %s*k = %zu", x_elems,
                    slotted ? "n_tokens*top_k" : "n_tokens", want_x);
    if (wa_bytes < last + expert_bytes || (pair && wb_bytes < last + expert_bytes))
        return fail(Q2K_ERR_INVALID_ARGUMENT, "w has %zu bytes, expected >= (n_experts-1)*expert_stride + "
                    "n*k/256*84 = %zu", pair && wb_bytes < wa_bytes ? wb_bytes : wa_bytes, last + expert_bytes);
    if (y_elems != want_y)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "y has %zu elements, expected n_tokens*top_k*n = %zu",
                    y_elems, want_y);
    if (!aligned(x, 16) || !aligned(ya, 16) || !aligned(wa, 4) || !aligned(ids, 4) ||
        (pair && (!aligned(yb, 16) || !aligned(wb, 4))) ||
        (bad_id_count != nullptr && !aligned(bad_id_count, 4)))
        return fail(Q2K_ERR_INVALID_ARGUMENT,
                    "x and y must be 16-byte aligned, w, ids and bad_id_count 4-byte aligned");
    const size_t y_bytes = want_y * 4, x_bytes = want_x * 4, id_bytes = routes * 4;
    const void* in[4] = {x, wa, ids, wb};
    const size_t in_bytes[4] = {x_bytes, wa_bytes, id_bytes, pair ? wb_bytes : 0};
    const void* outs[3] = {ya, yb, bad_id_count};
    const size_t out_bytes[3] = {y_bytes, pair ? y_bytes : 0, bad_id_count ? 4u : 0u};
    for (int o = 0; o < 3; ++o) {
        for (int i = 0; i < 4; ++i)
            if (overlaps(outs[o], out_bytes[o], in[i], in_bytes[i]))
                return fail(Q2K_ERR_INVALID_ARGUMENT, "writable buffers must not alias inputs or each other");
        for (int o2 = o + 1; o2 < 3; ++o2)
            if (overlaps(outs[o], out_bytes[o], outs[o2], out_bytes[o2]))
                return fail(Q2K_ERR_INVALID_ARGUMENT, "writable buffers must not alias inputs or each other");
    }
    // x rows: tokens, or routes when slotted
    const size_t x_rows = slotted ? routes : size_t(p->n_tokens);
    if (path == Q2K_PATH_AUTO) path = routed_auto_path(p);
    if (path == Q2K_PATH_TENSOR) {
        if (p->n_experts > uint32_t(q2k::kRoutedMaxExperts))
            return fail(Q2K_ERR_INVALID_ARGUMENT, "tensor-core path supports n_experts <= %d",
                        q2k::kRoutedMaxExperts);
        const size_t need = q2k::gemm_tc_routed_workspace_bytes(int(routes), int(p->n_experts), int(p->k));
        if (scratch == nullptr || scratch_bytes < need)
            return fail(Q2K_ERR_INVALID_ARGUMENT, "workspace has %zu bytes, needs %zu",
                        scratch == nullptr ? size_t(0) : scratch_bytes, need);
        if (!aligned(scratch, 16)) return fail(Q2K_ERR_INVALID_ARGUMENT, "workspace must be 16-byte aligned");
        if (overlaps(scratch, need, x, x_bytes) || overlaps(scratch, need, wa, wa_bytes) ||
            overlaps(scratch, need, ya, y_bytes) || overlaps(scratch, need, ids, id_bytes) ||
            (pair && (overlaps(scratch, need, wb, wb_bytes) || overlaps(scratch, need, yb, y_bytes))) ||
            (bad_id_count != nullptr && overlaps(scratch, need, bad_id_count, 4)))
            return fail(Q2K_ERR_INVALID_ARGUMENT, "workspace must not alias x, w, ids or y");
        DeviceInfo dev;
        q2k_status st = current_device(&dev);
        if (st != Q2K_OK) return st;
        const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        unsigned int* word = nullptr;
        int slot = -1;
        cudaError_t e = cudaSuccess;
        if (bad_id_count != nullptr) {
            e = cudaMemsetAsync(bad_id_count, 0, 4, s);
        } else {
            st = acquire_status_word(dev.device, s, &word, &slot);
            if (st != Q2K_OK) return st;
        }
        if (e == cudaSuccess)
            e = q2k::launch_gemm_tc_routed(x, static_cast<const uint8_t*>(wa),
                                           static_cast<long long>(p->expert_stride), ids, ya,
                                           int(routes), slotted ? 1 : int(p->top_k), int(p->n_experts),
                                           int(p->n), int(p->k),
                                           bad_id_count != nullptr ? bad_id_count : word, dev.device,
                                           dev.sm_count, scratch, s,
                                           pair ? static_cast<const uint8_t*>(wb) : nullptr,
                                           pair ? yb : nullptr);
        if (word != nullptr)
            return finish_status_word(dev.device, slot, word, s, e, what, "n_experts", p->n_experts);
        return e == cudaSuccess ? Q2K_OK : cuda_fail(e, what);
    }
    uint8_t* planes = nullptr;
    q2k_status st = check_planes_scratch(scratch, scratch_bytes, p->k, x_rows, x, x_bytes, wa,
                                         wa_bytes, ya, y_bytes, &planes);
    if (st == Q2K_OK && planes != nullptr && pair) {
        const size_t need = q2k::gemv_planes_stride(int(p->k)) * x_rows;
        if (overlaps(planes, need, wb, wb_bytes) || overlaps(planes, need, yb, y_bytes) ||
            overlaps(planes, need, ids, id_bytes))
            st = fail(Q2K_ERR_INVALID_ARGUMENT, "scratch must not alias x, w or y");
    }
    if (st != Q2K_OK) return st;
    DeviceInfo dev;
    st = current_device(&dev);
    if (st != Q2K_OK) return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    unsigned int* word = nullptr;
    int slot = -1;
    if (bad_id_count != nullptr) {
        e = cudaMemsetAsync(bad_id_count, 0, 4, s);
        if (e != cudaSuccess) return cuda_fail(e, "clearing bad_id_count");
    } else {
        st = acquire_status_word(dev.device, s, &word, &slot);
        if (st != Q2K_OK) return st;
    }
    q2k::GemvProblems pr;
    pr.w_stride = static_cast<long long>(p->expert_stride);
    pr.y_stride = static_cast<long long>(p->n);
    pr.ids = ids;
    pr.n_experts = p->n_experts;
    pr.top_k = slotted ? 1u : p->top_k;  // x row of route r: r / top_k, or r itself
    pr.bad_ids = bad_id_count != nullptr ? bad_id_count : word;
    if (pair) {
        pr.second_from = static_cast<int>(routes);
        pr.w2 = static_cast<const uint8_t*>(wb);
        pr.y2 = yb;
    }
    if (e == cudaSuccess)
        e = q2k::launch_gemv_problems(x, static_cast<const uint8_t*>(wa), ya, 1, int(p->n), int(p->k),
                                      dev.device, dev.sm_count, 0u, pr, int(pair ? 2 * routes : routes),
                                      s, planes, planes ? uint32_t(q2k::gemv_planes_stride(int(p->k))) : 0u);
    if (word != nullptr)
        return finish_status_word(dev.device, slot, word, s, e, what, "n_experts", p->n_experts);
    return e == cudaSuccess ? Q2K_OK : cuda_fail(e, what);
}

}  // namespace

extern "C" {

size_t q2k_x_planes_bytes(uint32_t k, uint32_t rows) {
    // The batched and routed GEMV launches bring x into their per-slice form
    // per thread (a few instructions per CTA); a separate prepare launch, and
    // the wait behind it, cost more than it saved.  They take no scratch.
    (void)k;
    (void)rows;
    return 0;
}

q2k_status q2k_matmul_id(const float* x, size_t x_elems, const void* w, size_t w_bytes,
                         const uint32_t* ids, float* y, size_t y_elems,
                         const q2k_matmul_id_params* p, uint32_t* bad_id_count, void* scratch,
                         size_t scratch_bytes, q2k_stream_t stream) {
    return routed_call(x, x_elems, false, w, w_bytes, nullptr, 0, ids, y, nullptr, y_elems, p,
                       bad_id_count, scratch, scratch_bytes, stream, "q2k_matmul_id launch");
}

q2k_status q2k_matmul_id_slotted(const float* x, size_t x_elems, const void* w, size_t w_bytes,
                                 const uint32_t* ids, float* y, size_t y_elems,
                                 const q2k_matmul_id_params* p, uint32_t* bad_id_count,
                                 void* scratch, size_t scratch_bytes, q2k_stream_t stream) {
    return routed_call(x, x_elems, true, w, w_bytes, nullptr, 0, ids, y, nullptr, y_elems, p,
                       bad_id_count, scratch, scratch_bytes, stream, "q2k_matmul_id_slotted launch");
}

size_t q2k_matmul_id_workspace_bytes(q2k_path path, uint32_t flags,
                                     const q2k_matmul_id_params* p) {
    if (p == nullptr || p->n_tokens == 0 || p->top_k == 0 || p->n == 0 || p->k == 0 ||
        p->n_experts == 0 || p->k % Q2K_QK_K != 0 || p->k > INT_MAX || (flags & ~1u) != 0)
        return 0;
    const size_t routes = size_t(p->n_tokens) * p->top_k;
    if (routes > 65535u) return 0;
    if (path == Q2K_PATH_AUTO) path = routed_auto_path(p);
    if (path == Q2K_PATH_TENSOR) {
        if (p->n_experts > uint32_t(q2k::kRoutedMaxExperts)) return 0;
        return q2k::gemm_tc_routed_workspace_bytes(int(routes), int(p->n_experts), int(p->k));
    }
    if (path != Q2K_PATH_GEMV) return 0;
    return q2k_x_planes_bytes(p->k, uint32_t((flags & Q2K_ID_SLOTTED) ? routes : p->n_tokens));
}

q2k_status q2k_matmul_id_ex(q2k_path path, uint32_t flags, const float* x, size_t x_elems,
                            const void* w, size_t w_bytes, const uint32_t* ids, float* y,
                            size_t y_elems, const q2k_matmul_id_params* p, uint32_t* bad_id_count,
                            void* workspace, size_t workspace_bytes, q2k_stream_t stream) {
    if (path != Q2K_PATH_AUTO && path != Q2K_PATH_GEMV && path != Q2K_PATH_TENSOR) {
        g_last_error[0] = '\0';
        return fail(Q2K_ERR_INVALID_ARGUMENT, "unknown path %d", static_cast<int>(path));
    }
    if ((flags & ~uint32_t(Q2K_ID_SLOTTED)) != 0) {
        g_last_error[0] = '\0';
        return fail(Q2K_ERR_INVALID_ARGUMENT, "unknown flag bits 0x%x", flags);
    }
    return routed_call(x, x_elems, (flags & Q2K_ID_SLOTTED) != 0, w, w_bytes, nullptr, 0, ids, y,
                       nullptr, y_elems, p, bad_id_count, workspace, workspace_bytes, stream,
                       "q2k_matmul_id_ex launch", path);
}

q2k_status q2k_matmul_id_pair_ex(q2k_path path, const float* x, size_t x_elems, const void* w_a,
                                 size_t w_a_bytes, const void* w_b, size_t w_b_bytes,
                                 const uint32_t* ids, float* y_a, float* y_b, size_t y_elems,
                                 const q2k_matmul_id_params* p, uint32_t* bad_id_count,
                                 void* workspace, size_t workspace_bytes, q2k_stream_t stream) {
    g_last_error[0] = '\0';
    if (path != Q2K_PATH_AUTO && path != Q2K_PATH_GEMV && path != Q2K_PATH_TENSOR)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "unknown path %d", static_cast<int>(path));
    if (y_b == nullptr || w_b == nullptr)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "x, w, ids and y must be non-NULL");
    return routed_call(x, x_elems, false, w_a, w_a_bytes, w_b, w_b_bytes, ids, y_a, y_b, y_elems, p,
                       bad_id_count, workspace, workspace_bytes, stream,
                       "q2k_matmul_id_pair_ex launch", path);
}

q2k_status q2k_matmul_id_pair(const float* x, size_t x_elems, const void* w_a, size_t w_a_bytes,
                              const void* w_b, size_t w_b_bytes, const uint32_t* ids, float* y_a,
                              float* y_b, size_t y_elems, const q2k_matmul_id_params* p,
                              uint32_t* bad_id_count, void* scratch, size_t scratch_bytes,
                              q2k_stream_t stream) {
    if (y_b == nullptr || w_b == nullptr) {
        g_last_error[0] = '\0';
        return fail(Q2K_ERR_INVALID_ARGUMENT, "x, w, ids and y must be non-NULL");
    }
    return routed_call(x, x_elems, false, w_a, w_a_bytes, w_b, w_b_bytes, ids, y_a, y_b, y_elems, p,
                       bad_id_count, scratch, scratch_bytes, stream, "q2k_matmul_id_pair launch");
}

q2k_status q2k_selftest_wait_timeout(uint32_t limit_us, q2k_stream_t stream) {
    g_last_error[0] = '\0';
    if (limit_us == 0 || limit_us > 100000)
        return fail(Q2K_ERR_INVALID_ARGUMENT, "limit_us must be in 1..100000, got %u", limit_us);
    DeviceInfo dev;
    q2k_status st = current_device(&dev);
    if (st != Q2K_OK) return st;
    cudaError_t e = q2k::launch_wait_timeout_selftest(uint64_t(limit_us) * 1000u,
                                                      reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? Q2K_OK : cuda_fail(e, "q2k_selftest_wait_timeout launch");
}

q2k_status q2k_device_error(uint32_t* out, q2k_stream_t stream) {
    g_last_error[0] = '\0';
    if (out == nullptr) return fail(Q2K_ERR_INVALID_ARGUMENT, "out is NULL");
    DeviceInfo dev;
    q2k_status st = current_device(&dev);
    if (st != Q2K_OK) return st;
    uint32_t tc = 0, gemv = 0;
    cudaError_t e = q2k::read_and_clear_tc_error(&tc, reinterpret_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = q2k::read_and_clear_gemv_error(&gemv, reinterpret_cast<cudaStream_t>(stream));
    *out = tc | gemv;
    return e == cudaSuccess ? Q2K_OK : cuda_fail(e, "q2k_device_error");
}

}  // extern "C"
