// fp32 CUDA-core Q2_K GEMV / small-M matmul: y[m, n] = sum_k x[m, k] W[n, k].
//
// mlx-native page "tests/deepseek_q2_k.rs", fn run_dense: the decode path the
// pages test at m <= 8 with an f32 tolerance (2e-4 absolute at n = 8, k = 256).
//
// Two kernels:
//
// gemv_m1_kernel (m = 1, k <= 16384, 4-byte aligned W): one CTA owns a
//   contiguous chunk of weight rows.  Its bytes are prefetched into L2 before
//   the kernel waits on the previous grid (programmatic dependent launch; an L2
//   prefetch is coherent, so this is safe even if that grid wrote W), then
//   copied into shared memory by bulk asynchronous copies, eight rows per
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

constexpr int kGemvWarps = 8;
// Rows per bulk copy and mbarrier: one block of the row loop (8 rows), so a
// block waits for exactly one piece.  Piece starts are 8 rows = 672 k/256
// bytes apart, a multiple of 16, so every piece keeps the chunk's offset from
// a 16-byte boundary (as CTA chunks do, being a multiple of 4 rows apart).
constexpr int kPieceRows = 8;
constexpr int kM1MaxSlices = 256;  // k <= 16384
// Threads per CTA of the m = 1 kernel.  A dependent call runs alone once its
// predecessor completes, so it takes more threads per CTA (shorter critical
// path); independent calls overlap, so smaller CTAs let more calls share an SM
// (up to four at 116 registers a thread).
constexpr int kM1ThreadsDependent = 256;
constexpr int kM1ThreadsIndependent = 128;
// Independent calls with more than 128 slices (k > 8192): one CTA's chunk and
// x planes fill an SM's shared memory, so the CTA takes two groups of warps
// over the slices (twice the warps to hide latencies with).
inline int m1_independent_threads(int K) {
    const int slices = K / 64;
    return slices > 128 ? 2 * ((slices + 31) / 32 * 32) : kM1ThreadsIndependent;
}

// ------------------------------------------------------------------ m = 1

constexpr int kRowBatch = 4;  // rows reduced together by one transposed butterfly

// x as integers: each 16-weight run r (k = 16 r .. 16 r + 15, one (half,
// shift, segment) of a block) is scaled by 2^e_r so that its largest |x| lies
// in [2^18, 2^19), rounded to nearest (relative error <= 2^-19 of the run's
// largest |x|), and split into byte planes x_int = p2 * 65536 + p1 * 256 + p0
// (p2 signed, p1/p0 unsigned).  19 bits keep every integer product of the
// dot below 2^31 (16 * 12 * 15 * 2^19 < 2^31), so the scale multiplies stay
// in integers.  The plane words of a run are 4 consecutive weights each.
// Also kept per run: the f32 sum of its 16 x (for the -ml term) and 2^-e_r.
struct RunPlanes {
    uint32_t p0[4], p1[4], p2[4];
};

// Shared-memory home of the planes: the 4 runs of slice sl (its 48 words,
// run j's planes at 12 j) start at word kSlicePitch * sl; the odd pitch puts
// the 32 slices a warp reads at once in 32 different banks.
constexpr int kSlicePitch = 49;

__device__ __forceinline__ void convert_run(const float* __restrict__ xr, uint32_t* planes,
                                            float* run_sum, float* run_inv) {
    float v[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 t = __ldg(reinterpret_cast<const float4*>(xr + 4 * q));
        v[4 * q] = t.x;
        v[4 * q + 1] = t.y;
        v[4 * q + 2] = t.z;
        v[4 * q + 3] = t.w;
    }
    float mx = 0.f, sum = 0.f;
#pragma unroll
    for (int l = 0; l < 16; ++l) {
        mx = fmaxf(mx, fabsf(v[l]));
        sum += v[l];
    }
    // e = 18 - floor(log2 max|x|), kept within the normal range; for max|x| = 0
    // (or a subnormal max) any e gives zeros, so e = 0 then.
    const int ex = static_cast<int>((__float_as_uint(mx) >> 23) & 0xFFu);  // biased exponent
    int e = (ex == 0 || ex == 255) ? 0 : 145 - ex;                            // 18 - (ex - 127)
    e = max(-126, min(126, e));
    const float up = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);   // 2^e, exact
    RunPlanes pl;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t b0 = 0, b1 = 0, b2 = 0;
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) {
            // |x 2^e| < 2^19: adding 1.5 * 2^23 rounds it to an integer (nearest,
            // ties to even) held in the low mantissa bits.
            const float biased = fmaf(v[4 * q + e4], up, 12582912.f);
            const uint32_t xi = __float_as_uint(biased) - 0x4B400000u;  // two's complement
            b0 |= (xi & 0xFFu) << (8 * e4);
            b1 |= ((xi >> 8) & 0xFFu) << (8 * e4);
            b2 |= ((xi >> 16) & 0xFFu) << (8 * e4);
        }
        pl.p0[q] = b0;
        pl.p1[q] = b1;
        pl.p2[q] = b2;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        planes[q] = pl.p0[q];
        planes[4 + q] = pl.p1[q];
        planes[8 + q] = pl.p2[q];
    }
    *run_sum = sum;
    *run_inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e
}

struct SlicePlanes {
    RunPlanes r[4];  // shift j = 0..3
    float inv[4];    // 2^-e of the run, times 1/4 for odd j (see slice_dot)
    // The four run sums X_j as integers with one scale 2^eX for the slice
    // (largest |X_j| in [2^21, 2^22)), byte j of each word = run j's byte.
    uint32_t xq0, xq1, xq2;
    float xinv;      // 2^-eX
};

// X_j -> the slice's integer byte planes (same rounding as convert_run).
__device__ __forceinline__ void quantize_run_sums(const float (&X)[4], SlicePlanes& s) {
    float mx = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) mx = fmaxf(mx, fabsf(X[j]));
    const int ex = static_cast<int>((__float_as_uint(mx) >> 23) & 0xFFu);
    int e = (ex == 0 || ex == 255) ? 0 : 148 - ex;  // 21 - (ex - 127)
    e = max(-126, min(126, e));
    const float up = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
    uint32_t b0 = 0, b1 = 0, b2 = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t xi = __float_as_uint(fmaf(X[j], up, 12582912.f)) - 0x4B400000u;
        b0 |= (xi & 0xFFu) << (8 * j);
        b1 |= ((xi >> 8) & 0xFFu) << (8 * j);
        b2 |= ((xi >> 16) & 0xFFu) << (8 * j);
    }
    s.xq0 = b0;
    s.xq1 = b1;
    s.xq2 = b2;
    s.xinv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
}

// The 7 words of one weight row a thread needs: its 16 quant bytes, the four
// scale bytes of its segment (one per shift) and the packed f16 d, dmin.
struct RowWords {
    uint32_t q[4];
    uint32_t sc4;
    uint32_t dd;
};

__device__ __forceinline__ RowWords load_row_words(const uint8_t* __restrict__ rp, int h, int seg,
                                                   uint32_t ssel) {
    RowWords r;
    const uint8_t* qp = rp + 16 + 32 * h + 16 * seg;
#pragma unroll
    for (int i = 0; i < 4; ++i) r.q[i] = ld_u32(qp + 4 * i);
    r.sc4 = __byte_perm(ld_u32(rp + 8 * h), ld_u32(rp + 8 * h + 4), ssel);
    r.dd = ld_u32(rp + 80);
    return r;
}

// Partial dot product of one weight row with this thread's 64-weight slice:
// d sum_j sc_j 2^-e_j S_j - dmin sum_j m_j X_j with S_j = sum_l q_l x_int_l.
// The 2-bit codes of shift j sit at bits 2 j of each quant byte; the odd
// shifts are masked in place (the code times 4, no shift needed) and s.inv
// carries the compensating 1/4.  sc_j S_j is formed in integers (below 2^31,
// see convert_run) and the min term is one integer dot of the four 4-bit
// mins with the slice's quantized run sums.
__device__ __forceinline__ float slice_dot(const RowWords& r, const SlicePlanes& s) {
    const uint32_t lo = r.sc4 & 0x0F0F0F0Fu;
    const uint32_t hi = (r.sc4 >> 4) & 0x0F0F0F0Fu;
    uint32_t q4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) q4[i] = r.q[i] >> 4;
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t mask = (j & 1) ? 0x0C0C0C0Cu : 0x03030303u;
        int a2 = 0;
        unsigned a1 = 0, a0 = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t t = (j < 2 ? r.q[i] : q4[i]) & mask;
            a2 = __dp4a(static_cast<int>(s.r[j].p2[i]), static_cast<int>(t), a2);
            a1 = __dp4a(s.r[j].p1[i], t, a1);
            a0 = __dp4a(s.r[j].p0[i], t, a0);
        }
        const int sint = a2 * 65536 + static_cast<int>(a1 * 256u + a0);
        const int sc = static_cast<int>(__byte_perm(lo, 0u, static_cast<uint32_t>(j) | 0x4440u));
        acc = fmaf(static_cast<float>(sint * sc), s.inv[j], acc);
    }
    int m2 = __dp4a(static_cast<int>(s.xq2), static_cast<int>(hi), 0);
    unsigned m1 = __dp4a(s.xq1, hi, 0u), m0 = __dp4a(s.xq0, hi, 0u);
    const int mint = m2 * 65536 + static_cast<int>(m1 * 256u + m0);
    const float d = f16_bits_to_float(r.dd);
    const float dmin = f16_bits_to_float(r.dd >> 16);
    return fmaf(d, acc, -(dmin * (static_cast<float>(mint) * s.xinv)));
}

// Sum v[0..kRowBatch) over the 32 lanes; afterwards lane L holds the total of
// row (L >> 3) & (kRowBatch - 1) ... in a fixed order (deterministic).
// Returns the row index this lane's value belongs to via *row.
__device__ __forceinline__ float transpose_reduce4(float (&v)[kRowBatch], int lane, int* row) {
    // xor 16: split rows {0,1} / {2,3}
    const bool up16 = (lane & 16) != 0;
    float a0 = up16 ? v[2] : v[0], a1 = up16 ? v[3] : v[1];
    float s0 = up16 ? v[0] : v[2], s1 = up16 ? v[1] : v[3];
    a0 += __shfl_xor_sync(0xFFFFFFFFu, s0, 16);
    a1 += __shfl_xor_sync(0xFFFFFFFFu, s1, 16);
    // xor 8: split the remaining pair
    const bool up8 = (lane & 8) != 0;
    float b = up8 ? a1 : a0;
    const float t = up8 ? a0 : a1;
    b += __shfl_xor_sync(0xFFFFFFFFu, t, 8);
    b += __shfl_xor_sync(0xFFFFFFFFu, b, 4);
    b += __shfl_xor_sync(0xFFFFFFFFu, b, 2);
    b += __shfl_xor_sync(0xFFFFFFFFu, b, 1);
    *row = (up16 ? 2 : 0) + (up8 ? 1 : 0);
    return b;
}

// Bulk copies of the CTA's weight rows into shared memory, kPieceRows rows per
// mbarrier (each completes when its bytes have landed).  W needs only 4-byte
// alignment: the host plan keeps every piece start at the same offset delta
// (0, 4, 8 or 12) from a 16-byte boundary, and the chunk sits at smem_w =
// 16-byte boundary + delta, so the 16-byte-aligned middle of each piece goes by
// bulk copy and its head and ragged tail (multiples of 4 bytes below 16) by
// plain loads before the barrier's arrival.  Lane 0 of warp w issues pieces w,
// w + nwarps, ...: one thread's bulk copies complete one after another, so
// spreading them over the warps multiplies the rate at which the chunk lands.
__device__ __forceinline__ void issue_weight_copies(uint8_t* smem_w, const uint8_t* gsrc,
                                                    uint32_t bars, int rows, size_t row_bytes,
                                                    uint32_t delta, int first, int step) {
    const int n_pieces = (rows + kPieceRows - 1) / kPieceRows;
    const size_t head = (16u - delta) & 15u;
    for (int p = first; p < n_pieces; p += step) {
        const int ra = p * kPieceRows;
        const int rb = min(rows, ra + kPieceRows);
        const size_t off = static_cast<size_t>(ra) * row_bytes;
        const size_t bytes = static_cast<size_t>(rb - ra) * row_bytes;
        const size_t bulk = (bytes - head) & ~size_t(15);  // bytes >= 84 > head
        for (size_t t = 0; t < head; t += 4)
            *reinterpret_cast<uint32_t*>(smem_w + off + t) =
                *reinterpret_cast<const uint32_t*>(gsrc + off + t);
        for (size_t t = head + bulk; t < bytes; t += 4)
            *reinterpret_cast<uint32_t*>(smem_w + off + t) =
                *reinterpret_cast<const uint32_t*>(gsrc + off + t);
        mbar_arrive_expect_tx(bars + 8 * p, static_cast<uint32_t>(bulk));
        bulk_copy_g2s(smem_u32(smem_w + off + head), gsrc + off + head, static_cast<uint32_t>(bulk),
                      bars + 8 * p);
    }
}

// x (K floats) -> the run planes, run sums and run scales in shared memory,
// spread over the CTA's threads.
__device__ __forceinline__ void convert_x(const float* __restrict__ x, uint32_t* planes,
                                          float* run_sum, float* run_inv, int n_runs, int tid,
                                          int nthreads) {
    for (int r = tid; r < n_runs; r += nthreads) {
        // run r = (block, half, shift j, segment): slice 4 block + 2 half + segment
        const int slr = ((r >> 4) << 2) | (((r >> 3) & 1) << 1) | (r & 1);
        convert_run(x + 16 * r, planes + slr * kSlicePitch + 12 * ((r >> 1) & 3), &run_sum[r],
                    &run_inv[r]);
    }
}

// This thread's slice (block b, half h, segment seg) of the converted x, into
// registers: the planes of its four runs, their scales and quantized sums.
__device__ __forceinline__ void load_slice_planes(const uint32_t* planes, const float* run_sum,
                                                  const float* run_inv, int sl, bool active, int b,
                                                  int h, int seg, SlicePlanes& s) {
    float X[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        // run of (block b, half h, shift j, segment seg)
        const int run = active ? 16 * b + 8 * h + 2 * j + seg : 0;
        const uint32_t* pj = planes + (active ? sl : 0) * kSlicePitch + 12 * j;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            s.r[j].p0[q] = pj[q];
            s.r[j].p1[q] = pj[4 + q];
            s.r[j].p2[q] = pj[8 + q];
        }
        X[j] = active ? run_sum[run] : 0.f;
        s.inv[j] = active ? run_inv[run] * ((j & 1) ? 0.25f : 1.f) : 0.f;
    }
    quantize_run_sums(X, s);
}

// Rows [0, rows) of a weight chunk in shared memory (this thread's slice of
// row r at my_col + r row_bytes) against the slice planes s: group g takes the
// blocks of eight consecutive rows g, g + groups, ... (rows 8 g .. 8 g + 7,
// then 8 (g + groups) ..), and each row's total over the group's warps goes to
// red[row * warps_per_group + warp in group].  The pieces (rows 8p .. 8p + 7)
// a block reads are waited for before its rows are read, unless all pieces up
// to `waited` are known to have landed; each piece barrier completes once, so
// waiting on it again returns at once.  Returns false once a wait gave up (the
// rows after it count as zero).
__device__ __forceinline__ bool dot_rows(const uint8_t* my_col, size_t row_bytes, int rows, int g,
                                         int groups, int lane, int wig, int warps_per_group,
                                         bool active, int h, int seg, uint32_t ssel,
                                         const SlicePlanes& s, float* red, uint32_t bars,
                                         uint32_t parity, int waited, volatile int* abort_flag,
                                         bool ok) {
    constexpr int kLoad = 2 * kRowBatch;  // rows loaded and decoded together
    for (int base = g * kLoad; base < rows; base += groups * kLoad) {
        // Make sure the pieces of this block have landed, then issue all
        // shared-memory loads of the block before any arithmetic.
        const int last = min(rows - 1, base + kLoad - 1);
        for (int pw = max(waited + 1, base / kPieceRows); pw <= last / kPieceRows; ++pw)
            ok = ok && mbar_wait_backoff(bars + 8 * pw, (parity >> pw) & 1u, abort_flag,
                                         &g_gemv_error, kErrTimeoutGemv, 64);
        RowWords rw[kLoad];
#pragma unroll
        for (int u = 0; u < kLoad; ++u) {
            const int lr = min(base + u, last);
            rw[u] = load_row_words(my_col + static_cast<size_t>(lr) * row_bytes, h, seg, ssel);
        }
        float part[kLoad];
#pragma unroll
        for (int u = 0; u < kLoad; ++u) {
            const float v = slice_dot(rw[u], s);
            part[u] = (active && ok && base + u < rows) ? v : 0.f;
        }
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            float p4[kRowBatch];
#pragma unroll
            for (int u = 0; u < kRowBatch; ++u) p4[u] = part[hb * kRowBatch + u];
            int which;
            const float tot = transpose_reduce4(p4, lane, &which);
            const int lr = base + hb * kRowBatch + which;
            if ((lane & 7) == 0 && lr < rows) red[lr * warps_per_group + wig] = tot;
        }
    }
    return ok;
}

// kMaxThreads: 256 for every plan but the two-group CTAs of large k (512); the
// smaller bound leaves the compiler more registers a thread.
template <int kMaxThreads>
__global__ void __launch_bounds__(kMaxThreads, 1)
gemv_m1_kernel(const float* __restrict__ x, const uint8_t* __restrict__ w, float* __restrict__ y,
               int N, int K, int rows_per_cta, int slices_pad, int groups, uint32_t flags,
               GemvProblems pr, const uint8_t* __restrict__ xplanes, uint32_t xplanes_stride) {
    const bool independent = (flags & kGemvIndependent) != 0;
    const bool const_weights = independent || (flags & kGemvConstWeights) != 0;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x;
    const int nthreads = blockDim.x;
    const int B = K >> 8;
    const int S = K >> 6;
    const int n_runs = K >> 4;
    const size_t row_bytes = static_cast<size_t>(B) * kBlockBytes;
    const int r0 = blockIdx.x * rows_per_cta;
    const int rows = min(rows_per_cta, N - r0);
    // Problem blockIdx.y of a batch (strided x, W, y) or of a routed product
    // (x row route / top_k, the W of expert ids[route]; a pair's second set of
    // routes uses w2 and y2); one problem: all strides 0.
    const int prob = blockIdx.y;
    if (pr.ids != nullptr) {
        // the ids (and x) may come from the grid before this one
        if (!independent) pdl_wait_prerequisites();
        const bool second = pr.second_from > 0 && prob >= pr.second_from;
        const int route = second ? prob - pr.second_from : prob;
        if (second) {
            w = pr.w2;
            y = pr.y2;
        }
        y += static_cast<size_t>(route) * pr.y_stride;
        const uint32_t e = pr.ids[route];
        if (e >= pr.n_experts) {
            // no such expert: this route's outputs are zeros and the bad id is counted
            for (int lr = tid; lr < rows; lr += nthreads) y[r0 + lr] = 0.f;
            if (blockIdx.x == 0 && tid == 0 && pr.bad_ids != nullptr) atomicAdd(pr.bad_ids, 1u);
            return;
        }
        x += static_cast<size_t>(route / pr.top_k) * K;
        w += static_cast<size_t>(e) * pr.w_stride;
        if (xplanes != nullptr) xplanes += static_cast<size_t>(route / pr.top_k) * xplanes_stride;
    } else {
        x += static_cast<size_t>(prob) * pr.x_stride;
        w += static_cast<size_t>(prob) * pr.w_stride;
        y += static_cast<size_t>(prob) * pr.y_stride;
        if (xplanes != nullptr) xplanes += static_cast<size_t>(prob) * xplanes_stride;
    }
    const uint32_t delta = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(w) & 15u);
    const int n_pieces = (rows + kPieceRows - 1) / kPieceRows;
    const int max_pieces = (rows_per_cta + kPieceRows - 1) / kPieceRows;
    const int warps_per_group = slices_pad >> 5;
    // shared layout: W chunk (at offset delta) | run planes | run sums | run
    // scales | red | bars | flag
    const size_t w_smem = (static_cast<size_t>(rows_per_cta) * row_bytes + 31) & ~size_t(15);
    uint8_t* smem_w = smem + delta;
    uint32_t* planes = reinterpret_cast<uint32_t*>(smem + w_smem);
    float* run_sum = reinterpret_cast<float*>(planes + (n_runs >> 2) * kSlicePitch);
    float* run_inv = run_sum + n_runs;
    float* red = run_inv + n_runs;
    const size_t red_end = w_smem + static_cast<size_t>(n_runs >> 2) * kSlicePitch * 4 +
                           static_cast<size_t>(n_runs) * 8 +
                           static_cast<size_t>(rows_per_cta) * warps_per_group * 4;
    const size_t bar_off = (red_end + 7) & ~size_t(7);
    const uint32_t bars = smem_u32(smem + bar_off);
    const uint32_t planes_bar = bars + 8 * max_pieces;  // x planes copied in (xplanes)
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + bar_off + 8 * (max_pieces + 1));
    const uint8_t* gsrc = w + static_cast<size_t>(r0) * row_bytes;
    const size_t chunk = static_cast<size_t>(rows) * row_bytes;

    // Let the next grid in the stream start: its prologue (barrier set-up,
    // weight prefetch or copy) then overlaps this grid.  An independent call
    // lets it start at once; a dependent one once its own dependency wait has
    // returned (below), so that whatever starts after it finds the grids
    // before this one complete.
    if (independent) pdl_allow_dependents();
    const int nwarps = nthreads >> 5;
    const bool issuer = (tid & 31) == 0;
    if (tid == 0) {
        for (int p = 0; p < n_pieces; ++p) mbar_init(bars + 8 * p, 1);
        mbar_init(planes_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // x converted once for several calls (prep_x_planes_kernel, a grid that
    // completed before this one started): one bulk copy of its planes, run
    // sums and run scales, laid out as convert_x lays them out here
    const uint32_t planes_bytes = static_cast<uint32_t>(
        static_cast<size_t>(n_runs >> 2) * kSlicePitch * 4 + static_cast<size_t>(n_runs) * 8);
    if (xplanes != nullptr && tid == 0) {
        mbar_arrive_expect_tx(planes_bar, planes_bytes);
        bulk_copy_g2s(smem_u32(planes), xplanes, planes_bytes, planes_bar);
    }
    if (const_weights) {
        // The caller guarantees the grids that may still run do not write W,
        // so the weight copies may start before the dependency wait.
        if (issuer) issue_weight_copies(smem_w, gsrc, bars, rows, row_bytes, delta, tid >> 5, nwarps);
    } else if (tid == 0) {
        // An L2 prefetch is coherent with the previous grid's writes (its
        // 16-byte-aligned part; the few bytes around it come with the copies).
        const size_t head = (16u - delta) & 15u;
        const size_t pre = (chunk - head) & ~size_t(15);
        for (size_t off = 0; off < pre; off += (size_t(1) << 20)) {
            const size_t left = pre - off;
            bulk_prefetch_l2(gsrc + head + off,
                             static_cast<uint32_t>(left < (size_t(1) << 20) ? left : (size_t(1) << 20)));
        }
    }
    if (!independent) {
        pdl_wait_prerequisites();
        pdl_allow_dependents();
    }
    __syncthreads();
    if (issuer && !const_weights)
        issue_weight_copies(smem_w, gsrc, bars, rows, row_bytes, delta, tid >> 5, nwarps);
    // x -> integer planes, once per CTA, while the weights stream in
    if (xplanes == nullptr) convert_x(x, planes, run_sum, run_inv, n_runs, tid, nthreads);
    // A dependent call's copies, issued before its dependency wait, have
    // (nearly) landed by now: one thread waits for all of them, and the
    // barrier below publishes that, so the row loop needs no barrier polls of
    // its own.  An independent call's copies were issued just now: its row
    // loop waits for each piece of rows as it needs it instead, and starts on
    // the first rows while the rest are in flight.
    const bool wait_all = const_weights && !independent;
    bool all_ok = true;
    if (xplanes != nullptr && tid == 0)
        all_ok = mbar_wait_backoff(planes_bar, 0, abort_flag, &g_gemv_error, kErrTimeoutGemv, 64);
    if (wait_all && tid == 0) {
        for (int p = 0; p < n_pieces; ++p)
            all_ok = all_ok && mbar_wait_backoff(bars + 8 * p, 0, abort_flag, &g_gemv_error,
                                                 kErrTimeoutGemv, 64);
    }
    __syncthreads();

    const int g = tid / slices_pad;
    const int sl = tid - g * slices_pad;
    const bool active = sl < S;
    const int b = sl >> 2, h = (sl >> 1) & 1, seg = sl & 1;
    const uint32_t ssel = seg | ((seg + 2) << 4) | ((seg + 4) << 8) | ((seg + 6) << 12);
    SlicePlanes s;
    load_slice_planes(planes, run_sum, run_inv, sl, active, b, h, seg, s);

    const int lane = tid & 31;
    const int wig = sl >> 5;  // warp index within the group
    const uint8_t* my_col = smem_w + b * kBlockBytes;
    const int waited = wait_all ? n_pieces - 1 : -1;
    const bool ok = !(const_weights && *abort_flag);
    dot_rows(my_col, row_bytes, rows, g, groups, lane, wig, warps_per_group, active, h, seg, ssel, s,
             red, bars, 0u, waited, abort_flag, ok);
    __syncthreads();
    for (int lr = tid; lr < rows; lr += nthreads) {
        float v = 0.f;
        for (int q = 0; q < warps_per_group; ++q) v += red[lr * warps_per_group + q];
        y[r0 + lr] = v;
    }
    if (tid == 0 && *abort_flag) {
        // Do not leave copies in flight into shared memory the next CTA may own.
        volatile int no_abort = 0;
        for (int p = 0; p < n_pieces; ++p)
            mbar_wait_bounded(bars + 8 * p, 0, &no_abort, &g_gemv_error, kErrTimeoutGemv);
        if (xplanes != nullptr)
            mbar_wait_bounded(planes_bar, 0, &no_abort, &g_gemv_error, kErrTimeoutGemv);
    }
    // Independent calls finish only after the grid before them, so work
    // enqueued later on the stream sees every earlier call complete.  One CTA
    // waiting keeps the grid from completing early; the others leave and free
    // their SM for the calls after this one.
    if (independent && blockIdx.x == 0) pdl_wait_prerequisites();
}

struct M1Plan {
    int rows_per_cta, ctas, slices_pad, groups, threads;
    size_t smem;
};

size_t m1_smem(int rows, int K, int slices_pad) {
    const size_t row_bytes = static_cast<size_t>(K / 256) * kBlockBytes;
    const int n_runs = K / 16;
    const int pieces = (rows + kPieceRows - 1) / kPieceRows;
    const size_t w_smem = (static_cast<size_t>(rows) * row_bytes + 31) & ~size_t(15);
    const size_t red_end = w_smem + static_cast<size_t>(n_runs / 4) * kSlicePitch * 4 +
                           static_cast<size_t>(n_runs) * 8 + static_cast<size_t>(rows) * (slices_pad / 32) * 4;
    return ((red_end + 7) & ~size_t(7)) + 8 * (pieces + 1) + 16;
}

bool plan_m1(int N, int K, int sm_count, int threads, bool whole_batches, M1Plan* p) {
    const int B = K / 256;
    const int S = K / 64;
    if (S > kM1MaxSlices) return false;
    const int slices_pad = (S + 31) / 32 * 32;
    const int groups = slices_pad >= threads ? 1 : threads / slices_pad;
    // Rows per CTA a multiple of what one pass of the row loop covers (groups x
    // 8 rows) when asked: the loop then never decodes a row twice at the end.
    // Independent calls share the SMs, so fewer CTAs than SMs costs nothing there.
    const int quantum = whole_batches ? groups * 2 * kRowBatch : 1;
    // Independent calls overlap on the SMs: their CTAs are kept to 72 KB of
    // shared memory (three share an SM) when 32 rows still fit there, so that
    // the x conversion every CTA repeats stays a small share of its work;
    // otherwise, and for dependent calls, the largest chunk that fits is taken.
    size_t cap = size_t(200) * 1024;
    if (whole_batches && m1_smem(32, K, slices_pad) <= size_t(72) * 1024) cap = size_t(72) * 1024;
    int rows = 0;
    for (int waves = 1;; ++waves) {
        rows = (N + sm_count * waves - 1) / (sm_count * waves);
        rows = (rows + quantum - 1) / quantum * quantum;
        if (B % 4) rows = (rows + 3) / 4 * 4;  // chunk starts stay 16-byte aligned
        if (m1_smem(rows, K, slices_pad) <= cap || rows <= kPieceRows || rows <= quantum) break;
    }
    p->rows_per_cta = rows;
    p->ctas = (N + rows - 1) / rows;
    p->slices_pad = slices_pad;
    p->groups = groups;
    p->threads = slices_pad * groups;
    p->smem = m1_smem(rows, K, slices_pad);
    return p->smem <= 227 * 1024;
}

cudaError_t launch_m1(const float* x, const uint8_t* w, float* y, int N, int K, const M1Plan& p,
                      int device, uint32_t flags, const GemvProblems& pr, int n_problems,
                      const uint8_t* xplanes, uint32_t xplanes_stride, cudaStream_t stream) {
    static bool smem_set[64] = {};
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    if (!smem_set[device]) {
        cudaError_t e = cudaFuncSetAttribute(gemv_m1_kernel<256>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             227 * 1024);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gemv_m1_kernel<512>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        smem_set[device] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.ctas, n_problems);
    cfg.blockDim = dim3(p.threads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.threads > 256)
        return cudaLaunchKernelEx(&cfg, gemv_m1_kernel<512>, x, w, y, N, K, p.rows_per_cta,
                                  p.slices_pad, p.groups, flags, pr, xplanes, xplanes_stride);
    return cudaLaunchKernelEx(&cfg, gemv_m1_kernel<256>, x, w, y, N, K, p.rows_per_cta,
                              p.slices_pad, p.groups, flags, pr, xplanes, xplanes_stride);
}

// ------------------------------------------------------------------ general m

template <int MT>
__global__ void __launch_bounds__(kGemvWarps * 32)
gemv_rows_kernel(const float* __restrict__ x, const uint8_t* __restrict__ w, float* __restrict__ y,
                 int M, int N, int K, GemvProblems pr) {
    const int lane = threadIdx.x & 31;
    const int n = blockIdx.x * kGemvWarps + (threadIdx.x >> 5);
    if (n >= N) return;  // whole warp leaves together
    // problem blockIdx.z, as in gemv_m1_kernel (one x row per problem there)
    const int prob = blockIdx.z;
    if (pr.ids != nullptr) {
        const bool second = pr.second_from > 0 && prob >= pr.second_from;
        const int route = second ? prob - pr.second_from : prob;
        if (second) {
            w = pr.w2;
            y = pr.y2;
        }
        y += static_cast<size_t>(route) * pr.y_stride;
        const uint32_t e = pr.ids[route];
        if (e >= pr.n_experts) {
            if (lane == 0) y[n] = 0.f;
            if (n == 0 && lane == 0 && pr.bad_ids != nullptr) atomicAdd(pr.bad_ids, 1u);
            return;
        }
        x += static_cast<size_t>(route / pr.top_k) * K;
        w += static_cast<size_t>(e) * pr.w_stride;
    } else {
        x += static_cast<size_t>(prob) * pr.x_stride;
        w += static_cast<size_t>(prob) * pr.w_stride;
        y += static_cast<size_t>(prob) * pr.y_stride;
    }
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
                        const GemvProblems& pr, int n_problems, cudaStream_t stream) {
    dim3 grid((N + kGemvWarps - 1) / kGemvWarps, (M + MT - 1) / MT, n_problems);
    gemv_rows_kernel<MT><<<grid, kGemvWarps * 32, 0, stream>>>(x, w, y, M, N, K, pr);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv_problems(const float* x, const uint8_t* w, float* y, int M, int N, int K,
                                 int device, int sm_count, uint32_t flags,
                                 const GemvProblems& pr, int n_problems, cudaStream_t stream,
                                 const uint8_t* xplanes, uint32_t xplanes_stride) {
    M1Plan plan;
    // Several problems in one grid overlap on the SMs like independent calls
    // do, so they take the same small CTAs of whole row batches, planned per
    // problem.  (Only the K slicing decides the arithmetic of a row, so the
    // plan never changes a result bit.)
    const bool small_ctas = (flags & kGemvIndependent) != 0 || n_problems > 1;
    const int threads = small_ctas ? m1_independent_threads(K) : kM1ThreadsDependent;
    if (M == 1 && plan_m1(N, K, sm_count, threads, small_ctas, &plan))
        return launch_m1(x, w, y, N, K, plan, device, flags, pr, n_problems, xplanes,
                         xplanes_stride, stream);
    switch (M < 8 ? M : 8) {
        case 1: return launch_rows<1>(x, w, y, M, N, K, pr, n_problems, stream);
        case 2: return launch_rows<2>(x, w, y, M, N, K, pr, n_problems, stream);
        case 3: return launch_rows<3>(x, w, y, M, N, K, pr, n_problems, stream);
        case 4: return launch_rows<4>(x, w, y, M, N, K, pr, n_problems, stream);
        case 5: return launch_rows<5>(x, w, y, M, N, K, pr, n_problems, stream);
        case 6: return launch_rows<6>(x, w, y, M, N, K, pr, n_problems, stream);
        case 7: return launch_rows<7>(x, w, y, M, N, K, pr, n_problems, stream);
        default: return launch_rows<8>(x, w, y, M, N, K, pr, n_problems, stream);
    }
}

cudaError_t launch_gemv(const float* x, const uint8_t* w, float* y, int M, int N, int K,
                        int device, int sm_count, uint32_t flags, cudaStream_t stream,
                        const uint8_t* xplanes) {
    return launch_gemv_problems(x, w, y, M, N, K, device, sm_count, flags, GemvProblems{}, 1, stream,
                                xplanes, 0u);
}

bool gemv_shares_planes(int M, int K) { return M == 1 && K / 64 <= kM1MaxSlices; }

size_t gemv_planes_bytes(int K) {
    return static_cast<size_t>(K / 64) * kSlicePitch * 4 + static_cast<size_t>(K / 16) * 8;
}

size_t gemv_planes_stride(int K) { return (gemv_planes_bytes(K) + 255) & ~size_t(255); }

// x (one row) -> the integer planes, run sums and run scales in the layout the
// m = 1 kernel keeps in shared memory, for several of its calls to copy.  It
// never lets the next grid start early, so every later grid sees it complete.
__global__ void __launch_bounds__(128)
prep_x_planes_kernel(const float* __restrict__ x, int K, uint8_t* __restrict__ dst,
                     size_t stride) {
    // x row blockIdx.y -> planes at dst + blockIdx.y stride
    const int n_runs = K >> 4;
    x += static_cast<size_t>(blockIdx.y) * K;
    dst += static_cast<size_t>(blockIdx.y) * stride;
    uint32_t* planes = reinterpret_cast<uint32_t*>(dst);
    float* run_sum = reinterpret_cast<float*>(planes + (n_runs >> 2) * kSlicePitch);
    float* run_inv = run_sum + n_runs;
    convert_x(x, planes, run_sum, run_inv, n_runs, blockIdx.x * blockDim.x + threadIdx.x,
              gridDim.x * blockDim.x);
}

cudaError_t launch_prep_x_planes(const float* x, int K, uint8_t* dst, cudaStream_t stream,
                                 int rows) {
    const int n_runs = K / 16;
    prep_x_planes_kernel<<<dim3((n_runs + 127) / 128, rows), 128, 0, stream>>>(
        x, K, dst, gemv_planes_stride(K));
    return cudaGetLastError();
}

namespace {

// One CTA waits on an mbarrier that nothing ever arrives at, with the bounded
// wait every kernel of the library uses but a short limit: the wait must give
// up, record kErrTimeoutGemv and return (no hang, no fault).
__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ volatile int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0)
        mbar_wait_lean(smem_u32(&bar), 0, &abort_flag, &g_gemv_error, kErrTimeoutGemv, 256, limit_ns);
    __syncthreads();
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, cudaStream_t stream) {
    wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns);
    return cudaGetLastError();
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
