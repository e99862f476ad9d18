// fp32 CUDA-core Q2_K GEMV / small-M matmul: y[m, n] = sum_k x[m, k] W[n, k].
//
// mlx-native page "tests/deepseek_q2_k.rs", fn run_dense: the decode path the
// pages test at m <= 8 with an f32 tolerance (2e-4 absolute at n = 8, k = 256).
//
// Both kernels form every weight exactly as the page's f32 decode does
// (dl*q - ml with one rounding, the value fn reference_dequant returns) and
// multiply-accumulate it with x in fp32 along accumulation chains of bounded
// length L, so |y - sum_k x w| <= L 2^-24 sum_k |x w| (+ the f32 underflow
// range) for every finite x and W: no rounding of x, no factored dl / ml terms.
//
// gemv_m1_kernel (m = 1, k <= 16384, 4-byte aligned W): one CTA owns a
//   contiguous chunk of weight rows.  Its bytes are prefetched into L2 before
//   the kernel waits on the previous grid (programmatic dependent launch; an L2
//   prefetch is coherent, so this is safe even if that grid wrote W), then
//   copied into shared memory by bulk asynchronous copies, eight rows per
//   mbarrier so decoding starts as soon as the first rows land.  Every thread
//   owns one 64-weight slice of K - one (block, half, segment): 16 quant bytes
//   read at the four shifts - and keeps that slice of x in registers (scaled by
//   a power of two) for all rows of the chunk.  Per row and slice:
//     - the 2-bit code of (lane, shift) is masked in place out of its quant word
//       and read as the bits of a float: q 2^(s - 149), s = its bit position
//       (a subnormal, or the smallest normals, exact);
//     - one packed fp32 FMA per two weights gives w 2^-42 = fl(q 2^(s-149) *
//       dl 2^(107 - s) - ml 2^-42): the product is exact, so this is the
//       page's dl*q - ml rounded once, scaled by 2^-42 (no overflow: dl < 2^20);
//     - one packed FMA per two weights accumulates x 2^t * w 2^-42, and the
//       slice's sum is scaled back by 2^(42 - t).
//   Slice sums meet in a fixed-order butterfly of warp shuffles and a
//   fixed-order sum over warps, so results are bit-reproducible and do not
//   depend on the launch plan.
//
// gemv_rows_kernel (any m <= 8 per launch slice, any k): one warp per weight
//   row, eight lanes per 84-byte block, x read through the read-only cache;
//   per-block sums added in a fixed three-level hierarchy (bounded chains).
#include <cuda_runtime.h>

#include "q2k_device.cuh"
#include "q2k_internal.h"

// Tuning knobs (compile-time; ROWS and MINB change no bits, ACCS changes the
// order of a slice's sum and so its rounding, within the same bound):
//   Q2K_GEMV_ROWS  rows decoded together and reduced by one transposed butterfly (2 or 4)
//   Q2K_GEMV_ACCS  independent accumulator pairs per row and slice (1, 2 or 4)
//   Q2K_GEMV_MINB  CTAs per SM the 128-thread plan is compiled for (register cap)
#ifndef Q2K_GEMV_ROWS
#define Q2K_GEMV_ROWS 4
#endif
#ifndef Q2K_GEMV_ACCS
#define Q2K_GEMV_ACCS 1
#endif
#ifndef Q2K_GEMV_MINB
#define Q2K_GEMV_MINB 4
#endif
//   Q2K_GEMV_W2 / Q2K_GEMV_DOT2  form the weights / the dot with packed (1) or
//                  scalar (0) fp32 FMAs (same arithmetic, same bits)
#ifndef Q2K_GEMV_W2
#define Q2K_GEMV_W2 0
#endif
#ifndef Q2K_GEMV_DOT2
#define Q2K_GEMV_DOT2 1
#endif
//   Q2K_GEMV_PIECE_ROWS  weight rows per bulk copy and barrier (4 or 8)
#ifndef Q2K_GEMV_PIECE_ROWS
#define Q2K_GEMV_PIECE_ROWS 8
#endif
//   Q2K_GEMV_BIGK_GROUPS, Q2K_GEMV_BIGK_CAP_KB  calls with k > 8192:
//                  groups of warps per CTA (1 or 2) and the CTA's shared-memory cap
#ifndef Q2K_GEMV_BIGK_GROUPS
#define Q2K_GEMV_BIGK_GROUPS 2
#endif
#ifndef Q2K_GEMV_BIGK_CAP_KB
#define Q2K_GEMV_BIGK_CAP_KB 200
#endif

namespace q2k {

__device__ unsigned int g_gemv_error;

namespace {

constexpr int kGemvWarps = 8;
// Rows per bulk copy and mbarrier: one block of the row loop, so a block waits
// for exactly one piece.  Piece starts are 4 or 8 rows = 336 k/256 or 672 k/256
// bytes apart, multiples of 16, so every piece keeps the chunk's offset from a
// 16-byte boundary (as CTA chunks do, being a multiple of 4 rows apart).
constexpr int kPieceRows = Q2K_GEMV_PIECE_ROWS;
static_assert(kPieceRows == 4 || kPieceRows == 8, "Q2K_GEMV_PIECE_ROWS must be 4 or 8");
constexpr int kM1MaxSlices = 256;  // k <= 16384
#ifndef Q2K_GEMV_DEP_WAVES
#define Q2K_GEMV_DEP_WAVES 3
#endif
// Threads per CTA of the m = 1 kernel: 128 (small CTAs, several per SM).
// With more than 128 slices (k > 8192) one CTA's chunk fills much of an SM's
// shared memory, so the CTA takes two groups of warps over the slices (twice
// the warps to hide latencies with).
constexpr int kM1Threads = 128;
inline int m1_threads(int K) {
    const int slices = K / 64;
    return slices > 128 ? Q2K_GEMV_BIGK_GROUPS * ((slices + 31) / 32 * 32) : kM1Threads;
}

// ------------------------------------------------------------------ m = 1

constexpr int kRowBatch = Q2K_GEMV_ROWS;
static_assert(kRowBatch == 2 || kRowBatch == 4, "Q2K_GEMV_ROWS must be 2 or 4");
constexpr int kAccs = Q2K_GEMV_ACCS;
static_assert(kAccs == 1 || kAccs == 2 || kAccs == 4, "Q2K_GEMV_ACCS must be 1, 2 or 4");
constexpr int kWScaleLog2 = 42;  // the row loop forms w 2^-42

// One thread's 64-weight slice of x (block b, half h, segment seg: weights
// k = 256 b + 128 h + 32 j + 16 seg + l, l = 0..15, j = 0..3), scaled by 2^t.
// Pair P = ((i * 2 + src) * 2 + a) * 2 + jp holds lane l = 4 i + 2 src + a at
// shifts j = 2 jp and 2 jp + 1 - the order in which slice_dot reads the
// lanes out of quant word i (src 1: the word shifted down by 16).
// t = min(42, 252 - biased exponent of the slice's largest |x|): every scaled
// |x| stays below 2^126, and the products x 2^t * w 2^-42 are x w scaled by
// 2^(t - 42), exactly 1 unless some |x| of the slice is 2^84 or more.
struct SliceX {
    float2 v[32];
    float rescale;  // 2^(42 - t): back from the slice's scale to x w
};

constexpr size_t kSliceXBytes = 64 * 4;  // the 64 scaled x of a slice, in pair order

__device__ __forceinline__ void scale_slice(const float (&v)[4][16], SliceX& s) {
    float mx = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int l = 0; l < 16; ++l) mx = fmaxf(mx, fabsf(v[j][l]));
    const int eb = static_cast<int>((__float_as_uint(mx) >> 23) & 0xFFu);
    const int t = min(kWScaleLog2, 252 - eb);
    const float up = __uint_as_float(static_cast<uint32_t>(127 + t) << 23);  // 2^t, exact
    s.rescale = __uint_as_float(static_cast<uint32_t>(127 + kWScaleLog2 - t) << 23);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int src = 0; src < 2; ++src)
#pragma unroll
            for (int a = 0; a < 2; ++a)
#pragma unroll
                for (int jp = 0; jp < 2; ++jp) {
                    const int l = 4 * i + 2 * src + a;
                    s.v[((i * 2 + src) * 2 + a) * 2 + jp] =
                        make_float2(v[2 * jp][l] * up, v[2 * jp + 1][l] * up);
                }
}

// The slice of x row `x` (K floats, 16-byte aligned) for (b, h, seg).
__device__ __forceinline__ void load_slice_x(const float* __restrict__ x, int b, int h, int seg,
                                             SliceX& s) {
    const float* base = x + 256 * b + 128 * h + 16 * seg;
    float v[4][16];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 t = __ldg(reinterpret_cast<const float4*>(base + 32 * j + 4 * q));
            v[j][4 * q] = t.x;
            v[j][4 * q + 1] = t.y;
            v[j][4 * q + 2] = t.z;
            v[j][4 * q + 3] = t.w;
        }
    scale_slice(v, s);
}

// Prepared x (prep_x_kernel): slice sl's pairs at sl * 256 bytes, the rescale
// factors of all S slices after the S slices.
__device__ __forceinline__ void load_slice_prepared(const uint8_t* __restrict__ xp, int S, int sl,
                                                    SliceX& s) {
    const float4* p = reinterpret_cast<const float4*>(xp + static_cast<size_t>(sl) * kSliceXBytes);
#pragma unroll
    for (int v = 0; v < 16; ++v) {
        const float4 t = __ldg(p + v);
        s.v[2 * v] = make_float2(t.x, t.y);
        s.v[2 * v + 1] = make_float2(t.z, t.w);
    }
    s.rescale = __ldg(reinterpret_cast<const float*>(xp + static_cast<size_t>(S) * kSliceXBytes) + sl);
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

__device__ __forceinline__ float2 bits2(uint32_t a, uint32_t b) {
    return make_float2(__uint_as_float(a), __uint_as_float(b));
}

// Dot product of one weight row with this thread's slice of x.
//
// Scale byte j of the slice (sc4 byte j): sc_j = low nibble, m_j = high
// nibble.  A 4-bit field at bit position p is made an exact float by OR-ing
// it into the mantissa of 2^E and subtracting 2^E (the field times 2^(E+p-23));
// E is picked per field to give sc_j 4^-j and m_j.  Then, exactly:
//   M[a][jp] = {dl_j 2^(107 - 8a - 2j)} for j = 2 jp, 2 jp + 1 (d 2^107 or d 2^99 times sc_j 4^-j),
//   A[jp]    = {-ml_j 2^-42}.
// Quant word i holds lanes 4 i .. 4 i + 3 in its bytes; lanes 4 i + 2, 4 i + 3
// are read from the word shifted down by 16, so lane 4 i + 2 src + a has its
// code of shift j at bit s = 8 a + 2 j.  u & (3 << s), read as a float, is
// q 2^(s - 149); times M it is dl q 2^-42 exactly, and the FMA with A rounds
// dl q - ml once.
__device__ __forceinline__ float slice_dot(const RowWords& r, const SliceX& s) {
    const uint32_t sc = r.sc4;
    const uint32_t sh = sc >> 16;  // scale bytes 2, 3 in the low half
    const float2 scA = fadd2(bits2((sc & 0xFu) | 0x4B000000u, (sc & 0xF00u) | 0x46000000u),
                             make_float2(-0x1p23f, -0x1p13f));  // {sc_0, sc_1 / 4}
    const float2 scB = fadd2(bits2((sh & 0xFu) | 0x49000000u, (sh & 0xF00u) | 0x44000000u),
                             make_float2(-0x1p19f, -0x1p9f));   // {sc_2 / 16, sc_3 / 64}
    const float2 mA = fadd2(bits2((sc & 0xF0u) | 0x49000000u, (sc & 0xF000u) | 0x45000000u),
                            make_float2(-0x1p19f, -0x1p11f));   // {m_0, m_1}
    const float2 mB = fadd2(bits2((sh & 0xF0u) | 0x49000000u, (sh & 0xF000u) | 0x45000000u),
                            make_float2(-0x1p19f, -0x1p11f));   // {m_2, m_3}
    // {d 2^107, -dmin 2^-42}
    const float2 dn = fmul2(make_float2(f16_bits_to_float(r.dd), f16_bits_to_float(r.dd >> 16)),
                            make_float2(0x1p107f, -0x1p-42f));
    const float2 D0 = make_float2(dn.x, dn.x), NM = make_float2(dn.y, dn.y);
    const float2 M00 = fmul2(scA, D0), M01 = fmul2(scB, D0);
    const float2 M10 = fmul2(M00, make_float2(0x1p-8f, 0x1p-8f));  // lanes a = 1: codes 8 bits up
    const float2 M11 = fmul2(M01, make_float2(0x1p-8f, 0x1p-8f));
    const float2 A0 = fmul2(mA, NM), A1 = fmul2(mB, NM);
    float2 acc[kAccs];
#pragma unroll
    for (int c = 0; c < kAccs; ++c) acc[c] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t qw = r.q[i];
        const uint32_t qh = qw >> 16;
#pragma unroll
        for (int src = 0; src < 2; ++src) {
            const uint32_t u = src ? qh : qw;
#pragma unroll
            for (int a = 0; a < 2; ++a)
#pragma unroll
                for (int jp = 0; jp < 2; ++jp) {
                    const int s0 = 8 * a + 4 * jp;
                    const float2 g = bits2(u & (3u << s0), u & (3u << (s0 + 2)));
                    const float2 M = a ? (jp ? M11 : M10) : (jp ? M01 : M00);
                    const float2 A = jp ? A1 : A0;
#if Q2K_GEMV_W2
                    const float2 w = ffma2(g, M, A);
#else
                    const float2 w = make_float2(fmaf(g.x, M.x, A.x), fmaf(g.y, M.y, A.y));
#endif
                    const float2 xv = s.v[((i * 2 + src) * 2 + a) * 2 + jp];
#if Q2K_GEMV_DOT2
                    acc[i % kAccs] = ffma2(xv, w, acc[i % kAccs]);
#else
                    acc[i % kAccs] = make_float2(fmaf(xv.x, w.x, acc[i % kAccs].x),
                                                 fmaf(xv.y, w.y, acc[i % kAccs].y));
#endif
                }
        }
    }
#pragma unroll
    for (int c = 1; c < kAccs; ++c) acc[0] = fadd2(acc[0], acc[c]);
    return (acc[0].x + acc[0].y) * s.rescale;
}

// Sum v[0..kRowBatch) over the 32 lanes in a fixed order (deterministic);
// afterwards the lanes of row_of_lane(lane) hold that row's total.
__device__ __forceinline__ int row_of_lane(int lane) {
    return kRowBatch == 4 ? ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1) : (lane >> 4) & 1;
}

__device__ __forceinline__ float transpose_reduce(float (&v)[kRowBatch], int lane) {
    const bool up16 = (lane & 16) != 0;
    float b;
    if constexpr (kRowBatch == 4) {
        // xor 16: split rows {0,1} / {2,3}
        float a0 = up16 ? v[2] : v[0], a1 = up16 ? v[3] : v[1];
        const float s0 = up16 ? v[0] : v[2], s1 = up16 ? v[1] : v[3];
        a0 += __shfl_xor_sync(0xFFFFFFFFu, s0, 16);
        a1 += __shfl_xor_sync(0xFFFFFFFFu, s1, 16);
        // xor 8: split the remaining pair
        const bool up8 = (lane & 8) != 0;
        b = up8 ? a1 : a0;
        const float t = up8 ? a0 : a1;
        b += __shfl_xor_sync(0xFFFFFFFFu, t, 8);
    } else {
        b = up16 ? v[1] : v[0];
        const float t = up16 ? v[0] : v[1];
        b += __shfl_xor_sync(0xFFFFFFFFu, t, 16);
        b += __shfl_xor_sync(0xFFFFFFFFu, b, 8);
    }
    b += __shfl_xor_sync(0xFFFFFFFFu, b, 4);
    b += __shfl_xor_sync(0xFFFFFFFFu, b, 2);
    b += __shfl_xor_sync(0xFFFFFFFFu, b, 1);
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

// Rows [0, rows) of a weight chunk in shared memory (this thread's slice of
// row r at my_col + r row_bytes) against the slice of x: group g takes the
// blocks of eight consecutive rows g, g + groups, ... (rows 8 g .. 8 g + 7,
// then 8 (g + groups) ..), kRowBatch rows at a time, and each row's total over
// the group's warps goes to red[row * warps_per_group + warp in group].  The
// piece (rows 8p .. 8p + 7) a block reads is waited for before its rows are
// read, unless all pieces up to `waited` are known to have landed; each piece
// barrier completes once, so waiting on it again returns at once.  Rows past
// `rows` in the last block are read from the chunk's shared memory (sized for
// whole blocks of eight rows) and their sums dropped.  kB: blocks per row when
// known at compile time (the row stride then folds into the loads), else 0.
// Returns false once a wait gave up (the rows after it count as zero).
template <int kB>
__device__ __forceinline__ bool dot_rows(const uint8_t* my_col, int B, int rows, int g, int groups,
                                         int lane, int wig, int warps_per_group, bool active, int h,
                                         int seg, uint32_t ssel, const SliceX& s, float* red,
                                         uint32_t bars, int waited, volatile int* abort_flag,
                                         bool ok) {
    const int row_bytes = (kB ? kB : B) * kBlockBytes;
    for (int base = g * kPieceRows; base < rows; base += groups * kPieceRows) {
        const int piece = base / kPieceRows;
        if (piece > waited)
            ok = ok && mbar_wait_backoff(bars + 8 * piece, 0u, abort_flag, &g_gemv_error,
                                         kErrTimeoutGemv, 64);
        const bool live = active && ok;
        const uint8_t* rp = my_col + base * row_bytes;
#pragma unroll 1
        for (int rb = base; rb < min(rows, base + kPieceRows); rb += kRowBatch, rp += kRowBatch * row_bytes) {
            // issue all shared-memory loads of the rows before any arithmetic
            RowWords rw[kRowBatch];
#pragma unroll
            for (int u = 0; u < kRowBatch; ++u) rw[u] = load_row_words(rp + u * row_bytes, h, seg, ssel);
            float part[kRowBatch];
#pragma unroll
            for (int u = 0; u < kRowBatch; ++u) {
                const float v = slice_dot(rw[u], s);
                part[u] = live ? v : 0.f;
            }
            const float tot = transpose_reduce(part, lane);
            const int lr = rb + row_of_lane(lane);
            if ((lane & (32 / kRowBatch - 1)) == 0 && lr < rows) red[lr * warps_per_group + wig] = tot;
        }
    }
    return ok;
}

// kMaxThreads: 128 for k <= 8192, 256 or 512 for the one- or two-group CTAs
// of larger k; kMinBlocks caps the registers so that as many CTAs share an SM.
template <int kMaxThreads, int kMinBlocks, int kB>
__global__ void __launch_bounds__(kMaxThreads, kMinBlocks)
gemv_m1_kernel(const float* __restrict__ x, const uint8_t* __restrict__ w, float* __restrict__ y,
               int N, int K, int rows_per_cta, int slices_pad, int groups, uint32_t flags,
               GemvProblems pr, const uint8_t* __restrict__ xprep, uint32_t xprep_stride) {
    const bool independent = (flags & kGemvIndependent) != 0;
    const bool const_weights = independent || (flags & kGemvConstWeights) != 0;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x;
    const int nthreads = blockDim.x;
    const int B = kB ? kB : K >> 8;
    const int S = 4 * B;
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
        if (xprep != nullptr) xprep += static_cast<size_t>(route / pr.top_k) * xprep_stride;
    } else {
        x += static_cast<size_t>(prob) * pr.x_stride;
        w += static_cast<size_t>(prob) * pr.w_stride;
        y += static_cast<size_t>(prob) * pr.y_stride;
        if (xprep != nullptr) xprep += static_cast<size_t>(prob) * xprep_stride;
    }
    const uint32_t delta = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(w) & 15u);
    const int n_pieces = (rows + kPieceRows - 1) / kPieceRows;
    const int max_pieces = (rows_per_cta + kPieceRows - 1) / kPieceRows;
    const int warps_per_group = slices_pad >> 5;
    // shared layout: W chunk (at offset delta, room for whole blocks of eight
    // rows) | red | bars | flag
    const int rows_alloc = (rows_per_cta + kPieceRows - 1) / kPieceRows * kPieceRows;
    const size_t w_smem = (static_cast<size_t>(rows_alloc) * row_bytes + 31) & ~size_t(15);
    uint8_t* smem_w = smem + delta;
    float* red = reinterpret_cast<float*>(smem + w_smem);
    const size_t red_end = w_smem + static_cast<size_t>(rows_per_cta) * warps_per_group * 4;
    const size_t bar_off = (red_end + 7) & ~size_t(7);
    const uint32_t bars = smem_u32(smem + bar_off);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + bar_off + 8 * max_pieces);
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
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
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
    const int g = tid / slices_pad;
    const int sl = tid - g * slices_pad;
    const bool active = sl < S;
    // inactive slice lanes (S not a multiple of 32) read block 0 and discard it
    const int b = active ? sl >> 2 : 0, h = (sl >> 1) & 1, seg = sl & 1;
    SliceX sx;
    if (independent) {
        // x is not written by any grid that may still run: read it now
        if (active) {
            if (xprep != nullptr) load_slice_prepared(xprep, S, sl, sx);
            else load_slice_x(x, b, h, seg, sx);
        }
    } else {
        pdl_wait_prerequisites();
        pdl_allow_dependents();
        __syncthreads();
        if (issuer && !const_weights)
            issue_weight_copies(smem_w, gsrc, bars, rows, row_bytes, delta, tid >> 5, nwarps);
        if (active) {
            if (xprep != nullptr) load_slice_prepared(xprep, S, sl, sx);
            else load_slice_x(x, b, h, seg, sx);
        }
    }
    if (!active) {
#pragma unroll
        for (int v = 0; v < 32; ++v) sx.v[v] = make_float2(0.f, 0.f);
        sx.rescale = 0.f;
    }
    // A dependent call's copies, issued before its dependency wait, have
    // (nearly) landed by now: one thread waits for all of them, and the
    // barrier below publishes that, so the row loop needs no barrier polls of
    // its own.  Other calls' row loops wait for each piece of rows as they
    // need it instead, and start on the first rows while the rest are in flight.
    const bool wait_all = const_weights && !independent;
    bool all_ok = true;
    if (wait_all && tid == 0) {
        for (int p = 0; p < n_pieces; ++p)
            all_ok = all_ok && mbar_wait_backoff(bars + 8 * p, 0, abort_flag, &g_gemv_error,
                                                 kErrTimeoutGemv, 64);
    }
    if (wait_all) __syncthreads();

    const uint32_t ssel = seg | ((seg + 2) << 4) | ((seg + 4) << 8) | ((seg + 6) << 12);
    const int lane = tid & 31;
    const int wig = sl >> 5;  // warp index within the group
    const uint8_t* my_col = smem_w + b * kBlockBytes;
    const int waited = wait_all ? n_pieces - 1 : -1;
    const bool ok = !(wait_all && *abort_flag);
    dot_rows<kB>(my_col, B, rows, g, groups, lane, wig, warps_per_group, active, h, seg, ssel, sx,
                 red, bars, waited, abort_flag, ok);
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
    const int pieces = (rows + kPieceRows - 1) / kPieceRows;
    const size_t w_smem = (static_cast<size_t>(pieces * kPieceRows) * row_bytes + 31) & ~size_t(15);
    const size_t red_end = w_smem + static_cast<size_t>(rows) * (slices_pad / 32) * 4;
    return ((red_end + 7) & ~size_t(7)) + 8 * pieces + 16;
}

bool plan_m1(int N, int K, int sm_count, int threads, M1Plan* p, int min_waves = 1) {
    const int B = K / 256;
    const int S = K / 64;
    if (S > kM1MaxSlices) return false;
    const int slices_pad = (S + 31) / 32 * 32;
    const int groups = slices_pad >= threads ? 1 : threads / slices_pad;
    // Rows per CTA a multiple of what one pass of the row loop covers (groups x
    // 8 rows): the loop then never decodes a row twice at the end.  Calls
    // share the SMs, so fewer CTAs than SMs costs nothing.
    const int quantum = groups * kPieceRows;
    // CTAs are kept to 72 KB of shared memory (three share an SM) when 32
    // rows still fit there; otherwise to Q2K_GEMV_BIGK_CAP_KB.
    const size_t cap = m1_smem(32, K, slices_pad) <= size_t(72) * 1024
                           ? size_t(72) * 1024
                           : size_t(Q2K_GEMV_BIGK_CAP_KB) * 1024;
    int rows = 0;
    for (int waves = min_waves;; ++waves) {
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

template <int kT, int kMinB, int kB>
cudaError_t launch_m1_as(const cudaLaunchConfig_t& cfg, int device, const float* x,
                         const uint8_t* w, float* y, int N, int K, const M1Plan& p, uint32_t flags,
                         const GemvProblems& pr, const uint8_t* xprep, uint32_t xprep_stride) {
    static bool smem_set[64] = {};
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    if (!smem_set[device]) {
        const cudaError_t e = cudaFuncSetAttribute(gemv_m1_kernel<kT, kMinB, kB>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   227 * 1024);
        if (e != cudaSuccess) return e;
        smem_set[device] = true;
    }
    return cudaLaunchKernelEx(&cfg, gemv_m1_kernel<kT, kMinB, kB>, x, w, y, N, K, p.rows_per_cta,
                              p.slices_pad, p.groups, flags, pr, xprep, xprep_stride);
}

// The row stride is compiled in for the common K (2048, 4096, 7168, 14336).
template <int kT, int kMinB>
cudaError_t launch_m1_threads(const cudaLaunchConfig_t& cfg, int device, const float* x,
                              const uint8_t* w, float* y, int N, int K, const M1Plan& p,
                              uint32_t flags, const GemvProblems& pr, const uint8_t* xprep,
                              uint32_t xprep_stride) {
    switch (K / 256) {
        case 8: return launch_m1_as<kT, kMinB, 8>(cfg, device, x, w, y, N, K, p, flags, pr, xprep, xprep_stride);
        case 16: return launch_m1_as<kT, kMinB, 16>(cfg, device, x, w, y, N, K, p, flags, pr, xprep, xprep_stride);
        case 28: return launch_m1_as<kT, kMinB, 28>(cfg, device, x, w, y, N, K, p, flags, pr, xprep, xprep_stride);
        case 56: return launch_m1_as<kT, kMinB, 56>(cfg, device, x, w, y, N, K, p, flags, pr, xprep, xprep_stride);
        default: return launch_m1_as<kT, kMinB, 0>(cfg, device, x, w, y, N, K, p, flags, pr, xprep, xprep_stride);
    }
}

cudaError_t launch_m1(const float* x, const uint8_t* w, float* y, int N, int K, const M1Plan& p,
                      int device, uint32_t flags, const GemvProblems& pr, int n_problems,
                      const uint8_t* xprep, uint32_t xprep_stride, cudaStream_t stream) {
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
        return launch_m1_threads<512, 1>(cfg, device, x, w, y, N, K, p, flags, pr, xprep, xprep_stride);
    if (p.threads > 128)
        return launch_m1_threads<256, 1>(cfg, device, x, w, y, N, K, p, flags, pr, xprep, xprep_stride);
    return launch_m1_threads<128, Q2K_GEMV_MINB>(cfg, device, x, w, y, N, K, p, flags, pr, xprep,
                                                 xprep_stride);
}

// ------------------------------------------------------------------ general m

// Running sum of per-block values with a bounded accumulation chain: blocks
// are summed 16 at a time, those sums 16 at a time, and those into the total,
// so a value passes through at most 16 + 16 + ceil(nb / 256) additions for nb
// blocks, in a fixed order (counts are uniform across the lanes of a warp).
template <int MT>
struct BlockSum {
    float l0[MT], l1[MT], tot[MT];
    int c0 = 0, c1 = 0;
    __device__ __forceinline__ BlockSum() {
#pragma unroll
        for (int mm = 0; mm < MT; ++mm) l0[mm] = l1[mm] = tot[mm] = 0.f;
    }
    __device__ __forceinline__ void add(const float (&blk)[MT]) {
#pragma unroll
        for (int mm = 0; mm < MT; ++mm) l0[mm] += blk[mm];
        if (++c0 == 16) {
            c0 = 0;
#pragma unroll
            for (int mm = 0; mm < MT; ++mm) {
                l1[mm] += l0[mm];
                l0[mm] = 0.f;
            }
            if (++c1 == 16) {
                c1 = 0;
#pragma unroll
                for (int mm = 0; mm < MT; ++mm) {
                    tot[mm] += l1[mm];
                    l1[mm] = 0.f;
                }
            }
        }
    }
    __device__ __forceinline__ float total(int mm) const { return tot[mm] + (l1[mm] + l0[mm]); }
};

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

    BlockSum<MT> sum;
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
        float acc[MT];
#pragma unroll
        for (int mm = 0; mm < MT; ++mm) acc[mm] = 0.f;
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
        sum.add(acc);  // this lane's 32 weights of block b
    }
    float tot[MT];
#pragma unroll
    for (int mm = 0; mm < MT; ++mm) {
        float v = sum.total(mm);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
        tot[mm] = v;
    }
    if (lane == 0) {
#pragma unroll
        for (int mm = 0; mm < MT; ++mm)
            if (mm < mcount) y[static_cast<size_t>(m0 + mm) * N + n] = tot[mm];
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
    // Every call takes small CTAs of whole row batches (several share an SM),
    // planned per problem: independent calls and the problems of one grid
    // overlap on the SMs, and a dependent call's short critical path after
    // its wait is better served by more, smaller CTAs than by one large CTA
    // per SM.  (Only the K slicing decides the arithmetic of a row, so the
    // plan never changes a result bit.)
    // A lone dependent call has the GPU to itself: with 128-thread CTAs (k <=
    // 8192) its rows are spread over Q2K_GEMV_DEP_WAVES CTAs per SM, fewer
    // rows per thread on its critical path (a chain of 4096^2 calls 5.65 ->
    // 5.30 us per call, 14336 x 4096 14.7 against 15.7 us).  The two-group
    // CTAs of larger k measured slower that way (4096 x 14336: 18.4 against
    // 15.0 us), so they keep one wave.
    const int min_waves = (flags & kGemvIndependent) || n_problems > 1 ||
                                  m1_threads(K) != kM1Threads
                              ? 1
                              : Q2K_GEMV_DEP_WAVES;
    if (M == 1 && plan_m1(N, K, sm_count, m1_threads(K), &plan, min_waves))
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
    return static_cast<size_t>(K / 64) * (kSliceXBytes + 4);
}

size_t gemv_planes_stride(int K) { return (gemv_planes_bytes(K) + 255) & ~size_t(255); }

// x (one row per blockIdx.y) -> the m = 1 kernel's per-slice form (the scaled
// x of each 64-weight slice in the order its row loop reads them, then the
// slices' rescale factors), for several of its calls to load instead of
// converting x themselves: the same values, so the same bits.  It never lets
// the next grid start early, so every later grid sees it complete.
__global__ void __launch_bounds__(128)
prep_x_kernel(const float* __restrict__ x, int K, uint8_t* __restrict__ dst, size_t stride) {
    const int S = K >> 6;
    x += static_cast<size_t>(blockIdx.y) * K;
    dst += static_cast<size_t>(blockIdx.y) * stride;
    for (int sl = blockIdx.x * blockDim.x + threadIdx.x; sl < S; sl += gridDim.x * blockDim.x) {
        SliceX s;
        load_slice_x(x, sl >> 2, (sl >> 1) & 1, sl & 1, s);
        float4* p = reinterpret_cast<float4*>(dst + static_cast<size_t>(sl) * kSliceXBytes);
#pragma unroll
        for (int v = 0; v < 16; ++v)
            p[v] = make_float4(s.v[2 * v].x, s.v[2 * v].y, s.v[2 * v + 1].x, s.v[2 * v + 1].y);
        reinterpret_cast<float*>(dst + static_cast<size_t>(S) * kSliceXBytes)[sl] = s.rescale;
    }
}

cudaError_t launch_prep_x_planes(const float* x, int K, uint8_t* dst, cudaStream_t stream,
                                 int rows) {
    const int S = K / 64;
    prep_x_kernel<<<dim3((S + 127) / 128, rows), 128, 0, stream>>>(x, K, dst,
                                                                  gemv_planes_stride(K));
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
