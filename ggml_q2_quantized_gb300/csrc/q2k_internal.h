// Launchers shared between the libq2k translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace q2k {

// Set the calling thread's message for q2k_last_error (the GGUF reader's
// translation unit reports through the same one).
void set_last_error(const char* msg);

cudaError_t launch_dequant(const uint8_t* blocks, float* out, size_t n_blocks, int sm_count,
                           cudaStream_t stream);

cudaError_t launch_gather(const uint8_t* table, const uint32_t* ids, float* out, uint32_t vocab,
                          uint32_t embed_dim, uint32_t n_tokens, uint32_t* bad_id_count,
                          int sm_count, cudaStream_t stream);

// fp32 GEMV path: m = 1 uses the shared-memory streaming kernel when K <= 16384
// (any 4-byte-aligned w); otherwise x rows are handled 8 at a time.
// flags (m = 1 kernel only):
//   kGemvConstWeights  the kernels that may still run do not write w: weight
//                      loads may start before the programmatic-launch wait;
//   kGemvIndependent   they touch neither x, w nor y: the kernel waits for the
//                      grid before it only at its very end (completion order).
constexpr uint32_t kGemvConstWeights = 1u;
constexpr uint32_t kGemvIndependent = 2u;
// tensor path with a workspace, one K part (gemm_tc_image_reusable): the
// workspace already holds this x's bf16 image, written for an earlier call
// that is still in the stream; the GEMM skips the prepass and its wait, may
// overlap the call before it, and completes after it
constexpr uint32_t kImageReady = 4u;
cudaError_t launch_gemv(const float* x, const uint8_t* w, float* y, int M, int N, int K,
                        int device, int sm_count, uint32_t flags, cudaStream_t stream,
                        const uint8_t* xplanes = nullptr);

// x converted once for several m = 1 calls: when gemv_shares_planes(M, K),
// launch_prep_x_planes writes gemv_planes_bytes(K) bytes (16-byte aligned
// destination) that launch_gemv(..., xplanes) calls then copy instead of
// converting x themselves (same values, so the same bits).  The prep grid
// completes before any later grid of the stream starts.
// Several x rows (rows of K floats, consecutive): planes of row r at dst + r
// gemv_planes_stride(K), for launch_gemv_problems(..., xplanes, stride) whose
// problems then find their x row's planes there.
bool gemv_shares_planes(int M, int K);
size_t gemv_planes_bytes(int K);
size_t gemv_planes_stride(int K);
cudaError_t launch_prep_x_planes(const float* x, int K, uint8_t* dst, cudaStream_t stream,
                                 int rows = 1);

// Several independent products in one launch of the GEMV kernels, each computed
// exactly as its own launch_gemv call (same kernel, same arithmetic), problem p
// being either
//   batched (ids == nullptr): x + p x_stride, w + p w_stride -> y + p y_stride;
//   routed: x row p / top_k and the weights of expert ids[p] at w + ids[p]
//           w_stride -> y + p y_stride.  An id >= n_experts gives zeros and
//           adds 1 to *bad_ids (when not null).  With second_from > 0, problems
//           p >= second_from are route p - second_from again with w2 and y2 in
//           place of w and y (two weight sets sharing the routing).
// Strides in elements (x, y) and bytes (w).  All zero: one problem.
struct GemvProblems {
    long long x_stride = 0;
    long long w_stride = 0;
    long long y_stride = 0;
    const uint32_t* ids = nullptr;
    uint32_t n_experts = 0;
    uint32_t top_k = 1;
    unsigned int* bad_ids = nullptr;
    int second_from = 0;
    const uint8_t* w2 = nullptr;
    float* y2 = nullptr;
};
cudaError_t launch_gemv_problems(const float* x, const uint8_t* w, float* y, int M, int N, int K,
                                 int device, int sm_count, uint32_t flags,
                                 const GemvProblems& pr, int n_problems, cudaStream_t stream,
                                 const uint8_t* xplanes = nullptr, uint32_t xplanes_stride = 0);

// Self-test of the bounded wait: one CTA waits for about limit_ns on a barrier
// nothing completes, then sets the GEMV error word's time-out bit.
cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, cudaStream_t stream);

// Read and clear the GEMV kernels' device error word (synchronises `stream`).
cudaError_t read_and_clear_gemv_error(uint32_t* out, cudaStream_t stream);

// Bytes of workspace the tensor-core path uses when given one: the x bf16 tile
// image, plus a buffer of per-part results when K is split (small m and n).
size_t gemm_tc_workspace_bytes(int M, int N, int K);

// bf16 tcgen05 GEMM; `device` selects per-device one-time setup.  With a
// workspace of gemm_tc_workspace_bytes(M, N, K) bytes (16-byte aligned), x is first
// converted to the bf16 tile image there and the GEMM copies A stages in bulk;
// with workspace == nullptr the GEMM converts x itself.
// flags (the small-m mode, m <= 64, only; see GemvProblems' kGemv* above):
// kGemvConstWeights lets the weight copies start before the dependency wait;
// kGemvIndependent also reads x and writes y without waiting for the grid
// before, which then only CTA (0, 0, 0) waits for, before it exits.
cudaError_t launch_gemm_tc(const float* x, const uint8_t* w, float* y, int M, int N, int K,
                           int device, int sm_count, void* workspace, cudaStream_t stream,
                           uint32_t flags = 0);
// The geometry keeps its x image in the workspace for a whole call (no small-m
// in-kernel conversion, one K part), so kImageReady may reuse it.
bool gemm_tc_image_reusable(int M, int N, int K);

// Independent products y_c = x W_c^T of one x (M <= 64 rows) in persistent
// weights-as-A grids: x converted once into `scratch`
// (gemm_tc_multi_scratch_bytes, 16-byte aligned), then one grid per at most 32
// calls, each CTA walking 128-row weight tiles of all of K (no K split).
// Each W must be 16-byte aligned and K a multiple of 1024
// (gemm_tc_multi_eligible, geometry only); the grids need the driver's
// tensor-map encoder (gemm_tc_multi_available).  No call may read or write
// another's output.
struct MultiCall {
    const uint8_t* w;
    float* y;
    int n;
};
bool gemm_tc_multi_eligible(int M, int K, const void* w);
bool gemm_tc_multi_available();
size_t gemm_tc_multi_scratch_bytes(int M, int K);
cudaError_t launch_gemm_tc_multi(const float* x, int M, int K, const MultiCall* calls, int count,
                                 void* scratch, int device, int sm_count, cudaStream_t stream);

// Routed product on tensor cores: route r = 0..routes-1 multiplies x row
// r / x_div by expert ids[r]'s weights (w + ids[r] * expert_stride, N rows)
// into y row r; ids out of range give a zero row and a count in *bad_ids (if
// not null).  With w2 and y2 (same layout) the second product reuses the
// routing and the x image: one more GEMM, and a bad id counts once per output.  The routes are grouped into 128-row x tiles per expert in a
// workspace of gemm_tc_routed_workspace_bytes bytes (16-byte aligned).
// cudaErrorInvalidValue for more than kRoutedMaxExperts experts.
constexpr int kRoutedMaxExperts = 4096;
size_t gemm_tc_routed_workspace_bytes(int routes, int n_experts, int K);
cudaError_t launch_gemm_tc_routed(const float* x, const uint8_t* w, long long expert_stride,
                                  const uint32_t* ids, float* y, int routes, int x_div,
                                  int n_experts, int N, int K, unsigned int* bad_ids, int device,
                                  int sm_count, void* workspace, cudaStream_t stream,
                                  const uint8_t* w2 = nullptr, float* y2 = nullptr);

// Size of the library's own fixed scratch for the tensor-core path (the x tile
// image), used by q2k_matmul_static_workspace.
constexpr size_t kStaticWorkspaceBytes = size_t(8) << 20;

// The tensor-core path with its x tile image in the library's fixed device
// scratch instead of a caller workspace.  cudaErrorInvalidValue when the
// image would not fit; the first call on a device looks up the scratch's
// device address (cudaGetSymbolAddress) with that device current.
cudaError_t launch_gemm_tc_static(const float* x, const uint8_t* w, float* y, int M, int N, int K,
                                  int device, int sm_count, cudaStream_t stream);

// The plain calls' scratch: the tensor-core path of a call without a
// workspace keeps its x tile image here when it fits (32 MiB: e.g. m <= 2048
// at k = 7168, m <= 1024 at k = 14336).  Such calls wait for the previous one through it
// (an event per device), so calls on different streams never share it at the
// same time; inside a stream capture, or when the image does not fit, the
// GEMM converts x itself (launch_gemm_tc without a workspace).
constexpr size_t kPlainScratchBytes = size_t(32) << 20;
cudaError_t launch_gemm_tc_plain(const float* x, const uint8_t* w, float* y, int M, int N, int K,
                                 int device, int sm_count, cudaStream_t stream, uint32_t flags = 0);

// Read and clear the tensor-core kernels' device error word (synchronises `stream`).
cudaError_t read_and_clear_tc_error(uint32_t* out, cudaStream_t stream);

}  // namespace q2k
