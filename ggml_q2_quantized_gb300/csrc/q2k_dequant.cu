// Standalone Q2_K dequantize and embedding gather (bit-exact f32 decode).
//
// mlx-native page "tests/deepseek_q2_k.rs": fn test_only_dequantize (tests
// q2_k_host_decode_*) and fn embedding_gather_q2_k (test
// q2_k_embedding_gather_matches_canonical_rows_and_rejects_bad_ids).
//
// One warp decodes one 84-byte block into 256 floats.  Lane L writes the two
// float4 runs at k = 4L and k = 128 + 4L, so a warp stores 2 x 512 contiguous
// bytes.  Every product in dl*q - ml is exact in f32 (d has an 11-bit
// significand, sc < 16, q < 4), so the result is the page's separately
// rounded f32 value whatever the evaluation order; it is still written with
// explicit round-to-nearest multiply and subtract so no contraction happens.
#include <cuda_runtime.h>

#include "q2k_device.cuh"
#include "q2k_internal.h"

namespace q2k {
namespace {

constexpr int kWarpsPerCta = 8;

__device__ __forceinline__ void decode_block_warp(const uint8_t* __restrict__ blk,
                                                  float* __restrict__ out, int lane) {
    const int j = lane >> 3;              // shift = 2 j
    const int seg = (lane >> 2) & 1;      // 16-lane segment within the 32-run
    const int l0 = (lane & 3) * 4;        // first of the 4 lanes this thread decodes
    const uint32_t dd = ld_u32(blk + 80);
    const float d = f16_bits_to_float(dd);
    const float dmin = f16_bits_to_float(dd >> 16);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const uint32_t sc = blk[8 * half + 2 * j + seg];
        const float dl = __fmul_rn(d, static_cast<float>(sc & 15u));
        const float ml = __fmul_rn(dmin, static_cast<float>(sc >> 4));
        const uint32_t qw = ld_u32(blk + 16 + 32 * half + 16 * seg + l0);
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t q = (qw >> (8 * e + 2 * j)) & 3u;
            v[e] = __fsub_rn(__fmul_rn(dl, static_cast<float>(q)), ml);
        }
        *reinterpret_cast<float4*>(out + 128 * half + 4 * lane) = make_float4(v[0], v[1], v[2], v[3]);
    }
}

__global__ void __launch_bounds__(kWarpsPerCta * 32)
dequant_kernel(const uint8_t* __restrict__ blocks, float* __restrict__ out, size_t n_blocks) {
    const int lane = threadIdx.x & 31;
    size_t wid = static_cast<size_t>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5);
    const size_t stride = static_cast<size_t>(gridDim.x) * kWarpsPerCta;
    for (; wid < n_blocks; wid += stride)
        decode_block_warp(blocks + wid * kBlockBytes, out + wid * kQK, lane);
}

__global__ void __launch_bounds__(kWarpsPerCta * 32)
gather_kernel(const uint8_t* __restrict__ table, const uint32_t* __restrict__ ids,
              float* __restrict__ out, uint32_t vocab, uint32_t blocks_per_row,
              size_t n_items, unsigned int* __restrict__ bad_id_count) {
    const int lane = threadIdx.x & 31;
    size_t item = static_cast<size_t>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5);
    const size_t stride = static_cast<size_t>(gridDim.x) * kWarpsPerCta;
    for (; item < n_items; item += stride) {
        const size_t t = item / blocks_per_row;
        const size_t b = item - t * blocks_per_row;
        const uint32_t id = ids[t];
        float* dst = out + item * kQK;
        if (id >= vocab) {
            // The pages reject such an id; with device-resident ids the kernel
            // zeroes the row and counts the token once (block 0 of the row).
            const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(dst + 4 * lane) = z;
            *reinterpret_cast<float4*>(dst + 128 + 4 * lane) = z;
            if (b == 0 && lane == 0 && bad_id_count != nullptr) atomicAdd(bad_id_count, 1u);
            continue;
        }
        const uint8_t* blk = table + (static_cast<size_t>(id) * blocks_per_row + b) * kBlockBytes;
        decode_block_warp(blk, dst, lane);
    }
}

int grid_for(size_t items, int sm_count) {
    const size_t per_cta = kWarpsPerCta;
    size_t ctas = (items + per_cta - 1) / per_cta;
    const size_t cap = static_cast<size_t>(sm_count) * 16;
    if (ctas > cap) ctas = cap;
    if (ctas < 1) ctas = 1;
    return static_cast<int>(ctas);
}

}  // namespace

cudaError_t launch_dequant(const uint8_t* blocks, float* out, size_t n_blocks, int sm_count,
                           cudaStream_t stream) {
    dequant_kernel<<<grid_for(n_blocks, sm_count), kWarpsPerCta * 32, 0, stream>>>(blocks, out,
                                                                                  n_blocks);
    return cudaGetLastError();
}

cudaError_t launch_gather(const uint8_t* table, const uint32_t* ids, float* out, uint32_t vocab,
                          uint32_t embed_dim, uint32_t n_tokens, uint32_t* bad_id_count,
                          int sm_count, cudaStream_t stream) {
    if (bad_id_count != nullptr) {
        cudaError_t e = cudaMemsetAsync(bad_id_count, 0, sizeof(uint32_t), stream);
        if (e != cudaSuccess) return e;
    }
    const uint32_t bpr = embed_dim / kQK;
    const size_t items = static_cast<size_t>(n_tokens) * bpr;
    gather_kernel<<<grid_for(items, sm_count), kWarpsPerCta * 32, 0, stream>>>(
        table, ids, out, vocab, bpr, items, reinterpret_cast<unsigned int*>(bad_id_count));
    return cudaGetLastError();
}

}  // namespace q2k
