// fp32 CUDA-core Q2_K GEMV / small-M matmul: y[m, n] = sum_k x[m, k] W[n, k].
//
// mlx-native page "tests/deepseek_q2_k.rs", fn run_dense: the decode path the
// pages test at m <= 8 with an f32 tolerance (2e-4 absolute at n = 8, k = 256).
//
// Work split: one warp per weight row n and per group of up to MT activation
// rows.  Eight lanes share one 84-byte block: lane slice s = 0..7 owns quant
// bytes [32 half + 16 seg + 8 (s & 1), +8) with half = s >> 2, seg = (s >> 1) & 1,
// i.e. 8 lanes of one segment at all four shifts = 32 weights with four scale
// bytes 8 half + 2 j + seg.  A warp covers four consecutive blocks per step,
// so a row streams as contiguous 336-byte spans.  Each weight is decoded once
// in fp32 (dl*q - ml, exact) and multiplied into MT fp32 accumulators; the
// per-lane partial sums are combined with a butterfly of warp shuffles in a
// fixed order, so repeated calls give identical bits.
#include <cuda_runtime.h>

#include "q2k_device.cuh"
#include "q2k_internal.h"

namespace q2k {
namespace {

constexpr int kGemvWarps = 8;

template <int MT>
__global__ void __launch_bounds__(kGemvWarps * 32)
gemv_kernel(const float* __restrict__ x, const uint8_t* __restrict__ w, float* __restrict__ y,
            int M, int N, int K) {
    const int lane = threadIdx.x & 31;
    const int n = blockIdx.x * kGemvWarps + (threadIdx.x >> 5);
    if (n >= N) return;  // whole warp leaves together
    const int m0 = blockIdx.y * MT;
    const int mcount = min(MT, M - m0);
    const int B = K >> 8;
    const uint8_t* row = w + static_cast<size_t>(n) * B * kBlockBytes;

    const int slice = lane & 7;
    const int half = slice >> 2;
    const int seg = (slice >> 1) & 1;
    const int l0 = (slice & 1) * 8;
    const int qoff = 16 + 32 * half + 16 * seg + l0;
    // Select scale bytes seg, seg+2, seg+4, seg+6 of the 8 bytes at 8*half.
    const uint32_t ssel = seg | ((seg + 2) << 4) | ((seg + 4) << 8) | ((seg + 6) << 12);

    float acc[MT];
#pragma unroll
    for (int mm = 0; mm < MT; ++mm) acc[mm] = 0.f;

    for (int b = lane >> 3; b < B; b += 4) {
        const uint8_t* blk = row + static_cast<size_t>(b) * kBlockBytes;
        const uint32_t q0 = ldg_stream_u32(blk + qoff);
        const uint32_t q1 = ldg_stream_u32(blk + qoff + 4);
        const uint32_t s0 = ldg_stream_u32(blk + 8 * half);
        const uint32_t s1 = ldg_stream_u32(blk + 8 * half + 4);
        const uint32_t dd = ldg_stream_u32(blk + 80);
        const uint32_t sc4 = __byte_perm(s0, s1, ssel);
        const float d = f16_bits_to_float(dd);
        const float dmin = f16_bits_to_float(dd >> 16);
        const float* xb = x + static_cast<size_t>(m0) * K + b * kQK + 128 * half + 16 * seg + l0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t sc = (sc4 >> (8 * j)) & 0xFFu;
            const float dl = __fmul_rn(d, static_cast<float>(sc & 15u));
            const float ml = __fmul_rn(dmin, static_cast<float>(sc >> 4));
            float wv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const uint32_t qw = e < 4 ? q0 : q1;
                const uint32_t q = (qw >> (8 * (e & 3) + 2 * j)) & 3u;
                wv[e] = fmaf(dl, static_cast<float>(q), -ml);  // exact: dl*q needs <= 17 bits
            }
#pragma unroll
            for (int mm = 0; mm < MT; ++mm) {
                if (mm < mcount) {
                    const float4 xa = __ldg(reinterpret_cast<const float4*>(xb + static_cast<size_t>(mm) * K + 32 * j));
                    const float4 xc = __ldg(reinterpret_cast<const float4*>(xb + static_cast<size_t>(mm) * K + 32 * j + 4));
                    float a = acc[mm];
                    a = fmaf(xa.x, wv[0], a);
                    a = fmaf(xa.y, wv[1], a);
                    a = fmaf(xa.z, wv[2], a);
                    a = fmaf(xa.w, wv[3], a);
                    a = fmaf(xc.x, wv[4], a);
                    a = fmaf(xc.y, wv[5], a);
                    a = fmaf(xc.z, wv[6], a);
                    a = fmaf(xc.w, wv[7], a);
                    acc[mm] = a;
                }
            }
        }
    }
#pragma unroll
    for (int mm = 0; mm < MT; ++mm) {
        float v = acc[mm];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
        acc[mm] = v;
    }
    if (lane == 0) {
#pragma unroll
        for (int mm = 0; mm < MT; ++mm)
            if (mm < mcount) y[static_cast<size_t>(m0 + mm) * N + n] = acc[mm];
    }
}

template <int MT>
cudaError_t launch_mt(const float* x, const uint8_t* w, float* y, int M, int N, int K,
                      cudaStream_t stream) {
    dim3 grid((N + kGemvWarps - 1) / kGemvWarps, (M + MT - 1) / MT);
    gemv_kernel<MT><<<grid, kGemvWarps * 32, 0, stream>>>(x, w, y, M, N, K);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv(const float* x, const uint8_t* w, float* y, int M, int N, int K,
                        cudaStream_t stream) {
    switch (M < 8 ? M : 8) {
        case 1: return launch_mt<1>(x, w, y, M, N, K, stream);
        case 2: return launch_mt<2>(x, w, y, M, N, K, stream);
        case 3: return launch_mt<3>(x, w, y, M, N, K, stream);
        case 4: return launch_mt<4>(x, w, y, M, N, K, stream);
        case 5: return launch_mt<5>(x, w, y, M, N, K, stream);
        case 6: return launch_mt<6>(x, w, y, M, N, K, stream);
        case 7: return launch_mt<7>(x, w, y, M, N, K, stream);
        default: return launch_mt<8>(x, w, y, M, N, K, stream);
    }
}

}  // namespace q2k
