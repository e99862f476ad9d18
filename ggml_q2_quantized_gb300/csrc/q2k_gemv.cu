// fp32 CUDA-core Q2_K GEMV / small-M matmul: y[m, n] = sum_k x[m, k] W[n, k].
//
// mlx-native page "tests/deepseek_q2_k.rs", fn run_dense: the decode path the
// pages test at m <= 8 with an f32 tolerance (2e-4 absolute at n = 8, k = 256).
//
// Two kernels:
//
// gemv_m1_kernel (m = 1, k <= 16384, 16-byte aligned W): one CTA owns a
//   contiguous chunk of weight rows.  Its bytes are prefetched into L2 before
//   the kernel waits on the previous grid (programmatic dependent launch; an L2
//   prefetch is coherent, so this is safe even if that grid wrote W), then
//   copied into shared memory by bulk asynchronous copies, four rows per
//   mbarrier so decoding starts as soon as the first rows land.  Every thread
//   owns one 64-weight slice of K - one (block, half, segment): 16 quant bytes
//   read at the four shifts - and keeps the slice of x in registers for all
//   rows of the chunk.  Per row it forms the four 16-weight sums
//   S_j = sum_l x_l q_l and adds dl_j S_j - ml_j X_j (X_j = sum_l x_l, fixed per
//   thread).  Partial sums meet in a fixed-order butterfly of warp shuffles and
//   a fixed-order sum over warps, so results are bit-reproducible.
//   kVariant selects how S_j is formed:
//     0  q to float through a byte permute into the bits of 1 + q/4, then the
//        bias removed exactly (packed f32 add) and packed f32 FMAs;
//     1  q to float by integer conversion, packed f32 FMAs;
//     2  exact integer dot products (dp4a) of q with three byte planes of x
//        scaled to 23-bit integers per slice (|x| max -> 2^21..2^22).
//
// gemv_rows_kernel (any m <= 8 per launch slice, any k): one warp per weight
//   row, eight lanes per 84-byte block, x read through the read-only cache.
#include <cuda_runtime.h>

#include "q2k_device.cuh"
#include "q2k_internal.h"

namespace q2k {

__device__ unsigned int g_gemv_error;

namespace {

#ifndef Q2K_GEMV_M1_VARIANT
#define Q2K_GEMV_M1_VARIANT 0
#endif

constexpr int kGemvWarps = 8;
constexpr int kPieceRows = 4;      // rows per bulk copy / mbarrier
constexpr int kM1MaxThreads = 256;
constexpr int kM1MaxSlices = 256;  // k <= 16384

// ------------------------------------------------------------------ m = 1

struct SliceX {
    float x[4][16];   // x at k = 256 b + 128 h + 32 j + 16 seg + l
    float X[4];       // sum_l x[j][l]
    uint32_t p0[4][4], p1[4][4], p2[4][4];  // byte planes (variant 2)
    float inv_scale;  // 2^-e (variant 2)
};

template <int kVariant>
__device__ __forceinline__ void load_slice(const float* __restrict__ xs, SliceX& s) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(xs + 32 * j + 4 * q));
            s.x[j][4 * q] = v.x;
            s.x[j][4 * q + 1] = v.y;
            s.x[j][4 * q + 2] = v.z;
            s.x[j][4 * q + 3] = v.w;
        }
        float acc = 0.f;
#pragma unroll
        for (int l = 0; l < 16; ++l) acc += s.x[j][l];
        s.X[j] = acc;
    }
    if (kVariant == 2) {
        float mx = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int l = 0; l < 16; ++l) mx = fmaxf(mx, fabsf(s.x[j][l]));
        // e such that max|x| * 2^e < 2^22: every scaled value fits 23 bits with sign
        int e = 0;
        if (mx > 0.f) e = 21 - ilogbf(mx);
        e = max(-126, min(e, 126));
        s.inv_scale = ldexpf(1.f, -e);
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t b0 = 0, b1 = 0, b2 = 0;
#pragma unroll
                for (int e4 = 0; e4 < 4; ++e4) {
                    const int v = __float2int_rn(ldexpf(s.x[j][4 * q + e4], e));
                    b0 |= (static_cast<uint32_t>(v) & 0xFFu) << (8 * e4);
                    b1 |= ((static_cast<uint32_t>(v) >> 8) & 0xFFu) << (8 * e4);
                    b2 |= ((static_cast<uint32_t>(v) >> 16) & 0xFFu) << (8 * e4);
                }
                s.p0[j][q] = b0;
                s.p1[j][q] = b1;
                s.p2[j][q] = b2;
            }
    }
}

__device__ __forceinline__ float small_uint_to_float(uint32_t byte_src, int which) {
    // byte `which` of byte_src (a value < 256) -> float, exactly, via 2^23 + v - 2^23
    const uint32_t sel = static_cast<uint32_t>(which) | (4u << 4) | (4u << 8) | (7u << 12);
    return __uint_as_float(__byte_perm(byte_src, 0x4B000000u, sel)) - 8388608.f;
}

// Partial dot product of one weight row with this thread's slice.
template <int kVariant>
__device__ __forceinline__ float slice_dot(const uint8_t* __restrict__ rp, int h, int seg,
                                           uint32_t ssel, const SliceX& s) {
    const uint8_t* qp = rp + 16 + 32 * h + 16 * seg;
    uint32_t qw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) qw[i] = ld_u32(qp + 4 * i);
    const uint32_t sc4 = __byte_perm(ld_u32(rp + 8 * h), ld_u32(rp + 8 * h + 4), ssel);
    const uint32_t dd = ld_u32(rp + 80);
    const float d = f16_bits_to_float(dd);
    const float dmin = f16_bits_to_float(dd >> 16);
    const uint32_t lo = sc4 & 0x0F0F0F0Fu;
    const uint32_t hi = (sc4 >> 4) & 0x0F0F0F0Fu;
    float p = 0.f;
    if (kVariant == 0) {
        const float d4 = 4.f * d;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float c1 = d * small_uint_to_float(lo, j);      // dl
            const float ml = dmin * small_uint_to_float(hi, j);   // ml
            (void)d4;
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t u = (j < 3) ? (qw[i] << (5 - 2 * j)) : (qw[i] >> 1);
                const uint32_t v = (u & 0x60606060u) | 0x80808080u;  // byte = 0x80 | q << 5
                float2 f01 = make_float2(__uint_as_float(__byte_perm(v, 0x3F000000u, 0x7054u)),
                                         __uint_as_float(__byte_perm(v, 0x3F000000u, 0x7154u)));
                float2 f23 = make_float2(__uint_as_float(__byte_perm(v, 0x3F000000u, 0x7254u)),
                                         __uint_as_float(__byte_perm(v, 0x3F000000u, 0x7354u)));
                // 1 + q/4 - 1 = q/4 exactly
                f01 = fadd2(f01, make_float2(-1.f, -1.f));
                f23 = fadd2(f23, make_float2(-1.f, -1.f));
                acc = ffma2(make_float2(s.x[j][4 * i], s.x[j][4 * i + 1]), f01, acc);
                acc = ffma2(make_float2(s.x[j][4 * i + 2], s.x[j][4 * i + 3]), f23, acc);
            }
            // acc = S_j / 4
            p = fmaf(4.f * c1, acc.x + acc.y, p);
            p = fmaf(-ml, s.X[j], p);
        }
    } else if (kVariant == 1) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float dl = d * static_cast<float>((lo >> (8 * j)) & 0xFFu);
            const float ml = dmin * static_cast<float>((hi >> (8 * j)) & 0xFFu);
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t t = (qw[i] >> (2 * j)) & 0x03030303u;
                const float2 f01 = make_float2(static_cast<float>(t & 0xFFu),
                                               static_cast<float>((t >> 8) & 0xFFu));
                const float2 f23 = make_float2(static_cast<float>((t >> 16) & 0xFFu),
                                               static_cast<float>(t >> 24));
                acc = ffma2(make_float2(s.x[j][4 * i], s.x[j][4 * i + 1]), f01, acc);
                acc = ffma2(make_float2(s.x[j][4 * i + 2], s.x[j][4 * i + 3]), f23, acc);
            }
            p = fmaf(dl, acc.x + acc.y, p);
            p = fmaf(-ml, s.X[j], p);
        }
    } else {
        const float dsc = d * s.inv_scale;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int a2 = 0;
            unsigned a1 = 0, a0 = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t t = (qw[i] >> (2 * j)) & 0x03030303u;
                a2 = __dp4a(static_cast<int>(s.p2[j][i]), static_cast<int>(t), a2);
                a1 = __dp4a(s.p1[j][i], t, a1);
                a0 = __dp4a(s.p0[j][i], t, a0);
            }
            const int sint = a2 * 65536 + static_cast<int>(a1 * 256u + a0);
            const float dl = dsc * static_cast<float>((lo >> (8 * j)) & 0xFFu);
            const float ml = dmin * static_cast<float>((hi >> (8 * j)) & 0xFFu);
            p = fmaf(dl, static_cast<float>(sint), p);
            p = fmaf(-ml, s.X[j], p);
        }
    }
    return p;
}

template <int kVariant>
__global__ void __launch_bounds__(kM1MaxThreads, 2)
gemv_m1_kernel(const float* __restrict__ x, const uint8_t* __restrict__ w, float* __restrict__ y,
               int N, int K, int rows_per_cta, int slices_pad, int groups) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x;
    const int B = K >> 8;
    const int S = K >> 6;
    const size_t row_bytes = static_cast<size_t>(B) * kBlockBytes;
    const int r0 = blockIdx.x * rows_per_cta;
    const int rows = min(rows_per_cta, N - r0);
    const int n_pieces = (rows + kPieceRows - 1) / kPieceRows;
    const int warps_per_group = slices_pad >> 5;
    const size_t w_smem = (static_cast<size_t>(rows_per_cta) * row_bytes + 15) & ~size_t(15);
    float* red = reinterpret_cast<float*>(smem + w_smem);
    const size_t red_bytes = (static_cast<size_t>(rows_per_cta) * warps_per_group * 4 + 7) & ~size_t(7);
    const uint32_t bars = smem_u32(smem + w_smem + red_bytes);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + w_smem + red_bytes +
                                                                8 * ((rows_per_cta + kPieceRows - 1) / kPieceRows));
    const uint8_t* gsrc = w + static_cast<size_t>(r0) * row_bytes;
    const size_t chunk = static_cast<size_t>(rows) * row_bytes;

    if (tid == 0) {
        // The weights never depend on the previous grid's results being in
        // shared memory, and an L2 prefetch is coherent with its writes.
        for (size_t off = 0; off < (chunk & ~size_t(15)); off += (size_t(1) << 20)) {
            const size_t left = (chunk & ~size_t(15)) - off;
            bulk_prefetch_l2(gsrc + off, static_cast<uint32_t>(left < (size_t(1) << 20) ? left : (size_t(1) << 20)));
        }
        for (int p = 0; p < n_pieces; ++p) mbar_init(bars + 8 * p, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    pdl_wait_prerequisites();
    pdl_allow_dependents();
    __syncthreads();

    if (tid == 0) {
        for (int p = 0; p < n_pieces; ++p) {
            const int ra = p * kPieceRows;
            const int rb = min(rows, ra + kPieceRows);
            const size_t off = static_cast<size_t>(ra) * row_bytes;
            const size_t bytes = static_cast<size_t>(rb - ra) * row_bytes;
            const size_t bulk = bytes & ~size_t(15);
            for (size_t t = bulk; t < bytes; t += 4)  // ragged end of the last piece
                *reinterpret_cast<uint32_t*>(smem + off + t) =
                    *reinterpret_cast<const uint32_t*>(gsrc + off + t);
            mbar_arrive_expect_tx(bars + 8 * p, static_cast<uint32_t>(bulk));
            bulk_copy_g2s(smem_u32(smem + off), gsrc + off, static_cast<uint32_t>(bulk), bars + 8 * p);
        }
    }

    const int g = tid / slices_pad;
    const int sl = tid - g * slices_pad;
    const bool active = sl < S;
    const int b = sl >> 2, h = (sl >> 1) & 1, seg = sl & 1;
    const uint32_t ssel = seg | ((seg + 2) << 4) | ((seg + 4) << 8) | ((seg + 6) << 12);
    SliceX s;
    if (active) {
        load_slice<kVariant>(x + 256 * b + 128 * h + 16 * seg, s);
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            s.X[j] = 0.f;
#pragma unroll
            for (int l = 0; l < 16; ++l) s.x[j][l] = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) s.p0[j][q] = s.p1[j][q] = s.p2[j][q] = 0u;
        }
        s.inv_scale = 0.f;
    }

    const int lane = tid & 31;
    const int wig = sl >> 5;  // warp index within the group
    int waited = -1;
    bool ok = true;
    for (int lr = g; lr < rows; lr += groups) {
        const int piece = lr / kPieceRows;
        if (piece != waited) {
            ok = ok && mbar_wait_bounded(bars + 8 * piece, 0, abort_flag, &g_gemv_error, kErrTimeoutGemv);
            waited = piece;
        }
        float part = 0.f;
        if (active && ok)
            part = slice_dot<kVariant>(smem + static_cast<size_t>(lr) * row_bytes + b * kBlockBytes, h, seg,
                                       ssel, s);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, off);
        if (lane == 0) red[lr * warps_per_group + wig] = part;
    }
    __syncthreads();
    for (int lr = tid; lr < rows; lr += blockDim.x) {
        float v = 0.f;
        for (int q = 0; q < warps_per_group; ++q) v += red[lr * warps_per_group + q];
        y[r0 + lr] = v;
    }
    if (tid == 0 && *abort_flag) {
        // Do not leave copies in flight into shared memory the next CTA may own.
        volatile int no_abort = 0;
        for (int p = 0; p < n_pieces; ++p)
            mbar_wait_bounded(bars + 8 * p, 0, &no_abort, &g_gemv_error, kErrTimeoutGemv);
    }
}

struct M1Plan {
    int rows_per_cta, ctas, slices_pad, groups, threads;
    size_t smem;
};

bool plan_m1(int N, int K, int sm_count, M1Plan* p) {
    const int B = K / 256;
    const int S = K / 64;
    if (S > kM1MaxSlices) return false;
    const size_t row_bytes = static_cast<size_t>(B) * kBlockBytes;
    const int slices_pad = (S + 31) / 32 * 32;
    const int groups = slices_pad >= kM1MaxThreads ? 1 : kM1MaxThreads / slices_pad;
    const size_t smem_cap = 200 * 1024;
    int rows = 0;
    for (int waves = 1;; ++waves) {
        rows = (N + sm_count * waves - 1) / (sm_count * waves);
        if (B % 4) rows = (rows + 3) / 4 * 4;  // chunk starts stay 16-byte aligned
        if (static_cast<size_t>(rows) * row_bytes <= smem_cap || rows <= kPieceRows) break;
    }
    const int wpg = slices_pad / 32;
    const int pieces = (rows + kPieceRows - 1) / kPieceRows;
    p->rows_per_cta = rows;
    p->ctas = (N + rows - 1) / rows;
    p->slices_pad = slices_pad;
    p->groups = groups;
    p->threads = slices_pad * groups;
    p->smem = ((static_cast<size_t>(rows) * row_bytes + 15) & ~size_t(15)) +
              ((static_cast<size_t>(rows) * wpg * 4 + 7) & ~size_t(7)) + 8 * pieces + 16;
    return p->smem <= 227 * 1024;
}

template <int kVariant>
cudaError_t launch_m1(const float* x, const uint8_t* w, float* y, int N, int K, const M1Plan& p,
                      int device, cudaStream_t stream) {
    static int smem_set[64] = {};
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    if (smem_set[device] < static_cast<int>(p.smem)) {
        cudaError_t e = cudaFuncSetAttribute(gemv_m1_kernel<kVariant>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             227 * 1024);
        if (e != cudaSuccess) return e;
        smem_set[device] = 227 * 1024;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.ctas);
    cfg.blockDim = dim3(p.threads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_m1_kernel<kVariant>, x, w, y, N, K, p.rows_per_cta,
                              p.slices_pad, p.groups);
}

// ------------------------------------------------------------------ general m

template <int MT>
__global__ void __launch_bounds__(kGemvWarps * 32)
gemv_rows_kernel(const float* __restrict__ x, const uint8_t* __restrict__ w, float* __restrict__ y,
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
cudaError_t launch_rows(const float* x, const uint8_t* w, float* y, int M, int N, int K,
                        cudaStream_t stream) {
    dim3 grid((N + kGemvWarps - 1) / kGemvWarps, (M + MT - 1) / MT);
    gemv_rows_kernel<MT><<<grid, kGemvWarps * 32, 0, stream>>>(x, w, y, M, N, K);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv(const float* x, const uint8_t* w, float* y, int M, int N, int K,
                        int device, int sm_count, cudaStream_t stream) {
    M1Plan plan;
    if (M == 1 && (reinterpret_cast<uintptr_t>(w) & 15u) == 0 && plan_m1(N, K, sm_count, &plan))
        return launch_m1<Q2K_GEMV_M1_VARIANT>(x, w, y, N, K, plan, device, stream);
    switch (M < 8 ? M : 8) {
        case 1: return launch_rows<1>(x, w, y, M, N, K, stream);
        case 2: return launch_rows<2>(x, w, y, M, N, K, stream);
        case 3: return launch_rows<3>(x, w, y, M, N, K, stream);
        case 4: return launch_rows<4>(x, w, y, M, N, K, stream);
        case 5: return launch_rows<5>(x, w, y, M, N, K, stream);
        case 6: return launch_rows<6>(x, w, y, M, N, K, stream);
        case 7: return launch_rows<7>(x, w, y, M, N, K, stream);
        default: return launch_rows<8>(x, w, y, M, N, K, stream);
    }
}

cudaError_t read_and_clear_gemv_error(uint32_t* out, cudaStream_t stream) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_gemv_error, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbolAsync(g_gemv_error, &zero, sizeof(unsigned int), 0,
                                cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(stream);
}

}  // namespace q2k
