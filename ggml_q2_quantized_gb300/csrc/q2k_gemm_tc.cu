// bf16 tensor-core Q2_K matmul for m > 8 (tcgen05 MMA, accumulator in TMEM).
//
// mlx-native page "tests/deepseek_q2_k.rs", fn run_dense with rows > 8 and
// the forced mm paths (dispatch_mm_for_test, dispatch_mm_simd_for_test): the
// pages run these in reduced precision (1e-2 absolute at n = 8, k = 256).
// Here both operands are rounded to bf16 (round to nearest even) and the
// products are summed in fp32 by the tensor cores.
//
// One CTA computes a 128 (x rows) x BN (weight rows) tile of y over the whole
// K, in stages of 64 K-elements held in shared memory in the 128-byte-swizzled
// K-major layout the MMA reads directly:
//   warps 0-3    convert x rows (f32 -> bf16) into the A stage, then run the
//                epilogue (TMEM -> registers -> y) for TMEM lanes 32w..32w+31;
//   BN/32 warps  decode weight rows: raw 84-byte blocks are copied from global
//                memory into a double-buffered shared slab with 4-byte
//                cp.async (coalesced across rows), then each thread decodes its
//                own row - per 16-weight segment a 4-entry bf16 table
//                {-ml, dl-ml, 2dl-ml, 3dl-ml} is built and each pair of 2-bit
//                quants picks two table entries with one byte permute;
//   1 warp       allocates TMEM and issues tcgen05.mma (one thread), each
//                stage released back to the producers by tcgen05.commit.
// Every wait is bounded (about a second); on time-out the kernel records a bit
// in the device error word, drains its MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cstring>
#include <mutex>

#include "q2k_device.cuh"
#include "q2k_internal.h"

namespace q2k {

__device__ unsigned int g_tc_error;

// Fixed scratch for callers that cannot allocate device memory: it holds the
// bf16 x tile image of the tensor-core path (ceil(m/256)*256 * k * 2 bytes).
// Every GPU that loads the library keeps these bytes until the process exits.
static __device__ __align__(256) uint8_t g_static_x_image[kStaticWorkspaceBytes];

// The plain calls' own scratch (q2k_matmul / q2k_matmul_path / q2k_matmul_ex
// without a workspace): the same x tile image, so that a caller who passes no
// workspace still gets the weights-as-A kernel.  Calls that use it are
// serialised on the GPU by an event per device (see launch_gemm_tc_plain).
static __device__ __align__(256) uint8_t g_plain_x_image[kPlainScratchBytes];

namespace {

constexpr int kBM = 128;                 // x rows per tile (MMA M)
constexpr int kKS = 64;                  // K elements per stage: one 128-byte swizzle row
constexpr int kAStage = kBM * kKS * 2;   // bytes of one A stage
constexpr int kXWarps = 4;

// Warp roles.  Without a workspace: warps 0-3 convert x into the A stages, then
// BN/32 decoder warps (one weight row per thread), then the MMA warp.  With a
// workspace (A stages arrive by bulk copy): every warp before the MMA warp
// decodes weights, two threads per row (each half a stage) when BN <= 192.
// Warps 0-3 also run the epilogue (TMEM lane quarter = warp).
template <int BN, bool kBulkA>
struct Cfg {
    static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "BN");
    static constexpr int kTPR = (kBulkA && BN <= 192) ? 2 : 1;  // decoder threads per row
    static constexpr int kDecThreads = kTPR * BN;
    static constexpr int kDecWarp0 = kBulkA ? 0 : kXWarps;
    // A (x) and B (decoded weights) have separate rings: A stages arrive by
    // copies whose latency the ring must cover, B stages are refilled by the
    // decoders a few hundred cycles ahead, so A gets the deeper ring.
    static constexpr int kAStages = (BN <= 128) ? 6 : (BN <= 192 ? 6 : 5);
    static constexpr int kBStages = (BN <= 128) ? 4 : 3;
    // raw 84-byte block slabs in flight: the decoders run kRaw - 1 blocks
    // (4 (kRaw - 1) stages) ahead of their own use to hide the weight fetch
    static constexpr int kRaw = (BN <= 128) ? 4 : (BN <= 192 ? 3 : 2);
    static constexpr int kBStage = BN * kKS * 2;
    static constexpr int kRawBytes = BN * kBlockBytes;
    static constexpr int kDecWarps = kDecThreads / 32;
    static constexpr int kMmaWarp = kDecWarp0 + kDecWarps;
    static constexpr int kThreads = (kMmaWarp + (kBulkA ? 2 : 1)) * 32;  // + A producer warp
    static constexpr int kTmemCols = BN <= 64 ? 64 : BN <= 128 ? 128 : 256;
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kAStages * kAStage;
    static constexpr int kOffRaw = kOffB + kBStages * kBStage;
    static constexpr int kOffBar = ((kOffRaw + kRaw * kRawBytes) + 7) & ~7;
    // bars: a_full[kAStages], a_empty[kAStages], b_full[kBStages], b_empty[kBStages],
    //       accum, drain, raw_full[kRaw]
    static constexpr int kNumBars = 2 * kAStages + 2 * kBStages + 2 + kRaw;
    static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack to align the base
    static_assert(kSmemBytes <= 232448, "shared memory");
};

// ---- tcgen05 / async-proxy wrappers ----------------------------------------

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), version 1 (tcgen05).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);       // start address >> 4
    d |= static_cast<uint64_t>(1u) << 16;                       // leading byte offset (unused here)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;               // stride byte offset >> 4
    d |= static_cast<uint64_t>(1u) << 46;                       // descriptor version
    d |= static_cast<uint64_t>(2u) << 61;                       // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: D f32, A and B bf16, both K-major.
__host__ __device__ constexpr uint32_t make_idesc(int m, int n) {
    return (1u << 4)                                  // D format: f32
         | (1u << 7)                                  // A format: bf16
         | (1u << 10)                                 // B format: bf16
         | (static_cast<uint32_t>(n >> 3) << 17)      // N / 8
         | (static_cast<uint32_t>(m >> 4) << 24);     // M / 16
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
          "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
          "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
          "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
          "=r"(v[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Byte offset of 16-byte chunk `c` (8 K-elements) of row `r` in a swizzled tile.
__device__ __forceinline__ uint32_t sw128_offset(int r, int c) {
    return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// Copy the raw 84-byte blocks of column `b` for the tile's BN rows into `dst`
// (row r at dst + 84 r).  Rows past N are zero-filled (d = dmin = 0 decode to 0).
template <int BN, int kThreadsDec>
__device__ __forceinline__ void issue_raw_copy(const uint8_t* __restrict__ w, uint32_t dst,
                                               int n0, int N, int blocks_per_row, int b,
                                               int td) {
    const size_t row_bytes = static_cast<size_t>(blocks_per_row) * kBlockBytes;
#pragma unroll 3
    for (int f = td; f < BN * kWordsPerBlock; f += kThreadsDec) {
        const int r = f / kWordsPerBlock;
        const int wd = f - r * kWordsPerBlock;
        const int n = n0 + r;
        const bool ok = n < N;
        const uint8_t* src = w + static_cast<size_t>(ok ? n : 0) * row_bytes +
                             static_cast<size_t>(b) * kBlockBytes + 4 * wd;
        cp_async_4(dst + r * kBlockBytes + 4 * wd, src, ok ? 4u : 0u);
    }
    cp_async_commit();
}

// Four bf16 weights of one quant word at shift 2j, picked from the table
// (lo = {v0, v1}, hi = {v2, v3}).  Returns them as two bf16x2 words.
template <int J>
__device__ __forceinline__ void decode_word(uint32_t word, uint32_t lo, uint32_t hi,
                                            uint32_t& p0, uint32_t& p1) {
    // byte i of t2 = 2 q_i for the four lanes of this word at shift 2J
    uint32_t t2;
    if constexpr (J == 0)
        t2 = (word * 2u) & 0x06060606u;
    else
        t2 = (word >> (2 * J - 1)) & 0x06060606u;
    // byte i -> nibbles (2 q_i, 2 q_i + 1); 17 * 6 + 16 < 256, so no carries.
    // Multiply-adds run on the FMA pipe and leave the integer ALU pipe (which
    // the masks and byte permutes need) less loaded.
    const uint32_t sel = t2 * 0x11u + 0x10101010u;
    p0 = __byte_perm(lo, hi, sel);
    p1 = __byte_perm(lo, hi, __umulhi(sel, 0x10000u));  // sel >> 16
}

// Stage C (0..3) of a block for one weight row, decoded into registers: for
// kJJ < 0 both 32-K halves (out[32], chunks 0..7), else half kJJ (out[16],
// chunks 4 kJJ .. 4 kJJ + 3).  Word 4 q + e of a chunk is bf16 pair e of it.
template <int C, int kJJ, int NW>
__device__ __forceinline__ void decode_stage_regs(const uint32_t (&sw)[4], float d, float dmin,
                                                  const uint32_t (&qw)[8], uint32_t (&out)[NW]) {
    constexpr int H = C >> 1;
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
        if (kJJ >= 0 && jj != kJJ) continue;
        const int j = 2 * (C & 1) + jj;
        const int base_jj = kJJ >= 0 ? 0 : jj;
#pragma unroll
        for (int seg = 0; seg < 2; ++seg) {
            const int si = 8 * H + 2 * j + seg;
            const uint32_t sc = (sw[si >> 2] >> (8 * (si & 3))) & 0xFFu;
            const float dl = __fmul_rn(d, static_cast<float>(sc & 15u));
            const float ml = __fmul_rn(dmin, static_cast<float>(sc >> 4));
            const uint32_t lo = pack_bf16x2(-ml, __fsub_rn(dl, ml));
            const uint32_t hi = pack_bf16x2(fmaf(2.f, dl, -ml), fmaf(3.f, dl, -ml));
            uint32_t* p = out + (base_jj * 2 + seg) * 8;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const uint32_t word = qw[4 * seg + t];
                if ((C & 1) == 0) {
                    if (jj == 0) decode_word<0>(word, lo, hi, p[2 * t], p[2 * t + 1]);
                    else decode_word<1>(word, lo, hi, p[2 * t], p[2 * t + 1]);
                } else {
                    if (jj == 0) decode_word<2>(word, lo, hi, p[2 * t], p[2 * t + 1]);
                    else decode_word<3>(word, lo, hi, p[2 * t], p[2 * t + 1]);
                }
            }
        }
    }
}

template <int kJJ, int NW>
__device__ __forceinline__ void decode_regs(int c, const uint32_t (&sw)[4], float d, float dmin,
                                            const uint32_t (&qw)[8], uint32_t (&out)[NW]) {
    if (c == 0) decode_stage_regs<0, kJJ>(sw, d, dmin, qw, out);
    else if (c == 1) decode_stage_regs<1, kJJ>(sw, d, dmin, qw, out);
    else if (c == 2) decode_stage_regs<2, kJJ>(sw, d, dmin, qw, out);
    else decode_stage_regs<3, kJJ>(sw, d, dmin, qw, out);
}

// Store decoded words of row r into a swizzled B stage (chunks 0..7, or the
// four chunks of half kJJ).
template <int kJJ, int NW>
__device__ __forceinline__ void store_stage(const uint32_t (&in)[NW], uint32_t b_stage, int r) {
#pragma unroll
    for (int q = 0; q < NW / 4; ++q) {
        const int chunk = (kJJ >= 0 ? 4 * kJJ : 0) + q;
        st_shared_v4(b_stage + sw128_offset(r, chunk), in[4 * q], in[4 * q + 1], in[4 * q + 2],
                     in[4 * q + 3]);
    }
}

template <int BN, bool kBulkA>
__global__ void __launch_bounds__(Cfg<BN, kBulkA>::kThreads, 1)
gemm_tc_kernel(const float* __restrict__ x, const uint8_t* __restrict__ xa,
               const uint8_t* __restrict__ w, float* __restrict__ y, int M, int N, int K) {
    using C = Cfg<BN, kBulkA>;
    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BN;
    const int m0 = blockIdx.y * kBM;
    const int n_iters = K / kKS;
    const int blocks_per_row = K / kQK;

    const uint32_t bar_afull = sbase + C::kOffBar;
    const uint32_t bar_aempty = bar_afull + 8 * C::kAStages;
    const uint32_t bar_bfull = bar_aempty + 8 * C::kAStages;
    const uint32_t bar_bempty = bar_bfull + 8 * C::kBStages;
    const uint32_t bar_accum = bar_bempty + 8 * C::kBStages;
    const uint32_t bar_drain = bar_accum + 8;
    const uint32_t bar_raw = bar_drain + 8;  // kRaw of them
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
    unsigned int* err = &g_tc_error;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kAStages; ++s) {
            // A: the producer's expect-tx arrival plus the copy's bytes, or one
            // arrival per x-producer warp without a workspace
            mbar_init(bar_afull + 8 * s, kBulkA ? 1 : kXWarps);
            mbar_init(bar_aempty + 8 * s, 1);
        }
        for (int s = 0; s < C::kBStages; ++s) {
            mbar_init(bar_bfull + 8 * s, C::kDecWarps);  // one arrival per decoder warp
            mbar_init(bar_bempty + 8 * s, 1);
        }
        mbar_init(bar_accum, 1);
        mbar_init(bar_drain, 1);
        for (int r = 0; r < C::kRaw; ++r) mbar_init(bar_raw + 8 * r, C::kDecWarps);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == C::kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(C::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_d = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

    if (!kBulkA && warp < kXWarps) {
        {
        // ---------------- x producer: f32 rows -> bf16 A stages ----------------
        const int t = threadIdx.x;
        const int c = t & 7;
        const int r0 = t >> 3;
        for (int i = 0; i < n_iters; ++i) {
            const int s = i % C::kAStages;
            if (i >= C::kAStages &&
                !__all_sync(0xFFFFFFFFu, mbar_wait_backoff(bar_aempty + 8 * s, ((i / C::kAStages) - 1) & 1,
                                                           abort_flag, err, kErrTimeoutEmpty, 128)))
                break;
            uint8_t* a_stage = smem + C::kOffA + s * kAStage;
            float4 va[8], vb[8];
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int m = m0 + r0 + 16 * it;
                if (m < M) {
                    const float4* src = reinterpret_cast<const float4*>(
                        x + static_cast<size_t>(m) * K + static_cast<size_t>(i) * kKS + 8 * c);
                    va[it] = __ldg(src);
                    vb[it] = __ldg(src + 1);
                } else {
                    va[it] = make_float4(0.f, 0.f, 0.f, 0.f);
                    vb[it] = va[it];
                }
            }
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int r = r0 + 16 * it;
                *reinterpret_cast<uint4*>(a_stage + sw128_offset(r, c)) =
                    make_uint4(pack_bf16x2(va[it].x, va[it].y), pack_bf16x2(va[it].z, va[it].w),
                               pack_bf16x2(vb[it].x, vb[it].y), pack_bf16x2(vb[it].z, vb[it].w));
            }
            fence_proxy_async_smem();  // this thread's stores -> visible to the MMA
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_afull + 8 * s);
        }
        }
    } else if (warp >= C::kDecWarp0 && warp < C::kMmaWarp) {
        // ---------------- weight decoders ----------------
        const int td = threadIdx.x - C::kDecWarp0 * 32;  // 0 .. kDecThreads - 1
        const int row = td % BN;                         // tile row
        const int half_sel = td / BN;                    // which 32-K half (two threads per row)
        const uint32_t raw0 = sbase + C::kOffRaw;
        // Start pulling this tile's weight rows into L2 now (one bulk prefetch
        // per row, all K) so the 84-byte block gathers below hit L2.
        if (td < BN && n0 + td < N) {
            const size_t row_bytes = static_cast<size_t>(blocks_per_row) * kBlockBytes;
            const uint8_t* rp = w + static_cast<size_t>(n0 + td) * row_bytes;
            const uintptr_t a = (reinterpret_cast<uintptr_t>(rp) + 15) & ~uintptr_t(15);
            const uintptr_t e = (reinterpret_cast<uintptr_t>(rp) + row_bytes) & ~uintptr_t(15);
            if (e > a) bulk_prefetch_l2(reinterpret_cast<const void*>(a), static_cast<uint32_t>(e - a));
        }
        // One cp.async group per block (an empty one past the last block), so
        // "all but the newest kRaw - 2 groups done" always means block b landed.
        for (int pb = 0; pb < C::kRaw - 1; ++pb) {
            if (pb < blocks_per_row)
                issue_raw_copy<BN, C::kDecThreads>(w, raw0 + pb * C::kRawBytes, n0, N, blocks_per_row,
                                                   pb, td);
            else
                cp_async_commit();
        }
        bool ok = true;
        for (int b = 0; b < blocks_per_row && ok; ++b) {
            const int buf = b % C::kRaw;
            cp_async_wait_group<C::kRaw - 2>();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_raw + 8 * buf);
            if (!__all_sync(0xFFFFFFFFu, mbar_wait_backoff(bar_raw + 8 * buf, (b / C::kRaw) & 1,
                                                           abort_flag, err, kErrTimeoutEmpty, 128))) {
                ok = false;
                break;
            }
            // Every thread has finished with block b - 1's slab (it arrived for
            // block b above), which is where block b + kRaw - 1 goes.
            const int nb = b + C::kRaw - 1;
            if (nb < blocks_per_row)
                issue_raw_copy<BN, C::kDecThreads>(w, raw0 + (nb % C::kRaw) * C::kRawBytes, n0, N,
                                                   blocks_per_row, nb, td);
            else
                cp_async_commit();
            const uint32_t mine = raw0 + buf * C::kRawBytes + row * kBlockBytes;
            uint32_t sw[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) sw[q] = ld_shared_u32(mine + 4 * q);
            const uint32_t dd = ld_shared_u32(mine + 80);
            const float d = f16_bits_to_float(dd);
            const float dmin = f16_bits_to_float(dd >> 16);
            uint32_t qw[8];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (c == 0 || c == 2) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) qw[q] = ld_shared_u32(mine + 16 + 32 * (c >> 1) + 4 * q);
                }
                const int i = 4 * b + c;
                const int s = i % C::kBStages;
                // Decode first (registers only), then wait for the slot: the
                // decode latency overlaps the MMAs still reading this slot.
                constexpr int NW = C::kTPR == 1 ? 32 : 16;
                uint32_t pw[NW];
                if (C::kTPR == 1) decode_regs<-1>(c, sw, d, dmin, qw, pw);
                else if (half_sel == 0) decode_regs<0>(c, sw, d, dmin, qw, pw);
                else decode_regs<1>(c, sw, d, dmin, qw, pw);
                if (i >= C::kBStages &&
                    !__all_sync(0xFFFFFFFFu,
                                mbar_wait_backoff(bar_bempty + 8 * s, ((i / C::kBStages) - 1) & 1,
                                                  abort_flag, err, kErrTimeoutEmpty, 32))) {
                    ok = false;
                    break;
                }
                const uint32_t b_stage = sbase + C::kOffB + s * C::kBStage;
                if (C::kTPR == 1) store_stage<-1>(pw, b_stage, row);
                else if (half_sel == 0) store_stage<0>(pw, b_stage, row);
                else store_stage<1>(pw, b_stage, row);
                fence_proxy_async_smem();  // this thread's stores -> visible to the MMA
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_bfull + 8 * s);
            }
        }
        cp_async_wait_all();  // no copy may land after this CTA is gone

    } else if (kBulkA && warp == C::kMmaWarp + 1) {
        // ---------------- A producer: one 16 KB bulk copy per stage ----------------
        // The prepass wrote x as bf16 in exactly this swizzled tile layout, tile
        // (m tile, K stage) at xa + (m_tile * n_iters + stage) * 16 KB.
        if (lane == 0) {
            const uint8_t* src = xa + static_cast<size_t>(blockIdx.y) * n_iters * kAStage;
            for (int i = 0; i < n_iters; ++i) {
                const int s = i % C::kAStages;
                if (i >= C::kAStages &&
                    !mbar_wait_backoff(bar_aempty + 8 * s, ((i / C::kAStages) - 1) & 1, abort_flag,
                                       err, kErrTimeoutEmpty, 32))
                    break;
                mbar_arrive_expect_tx(bar_afull + 8 * s, kAStage);
                bulk_copy_g2s(sbase + C::kOffA + s * kAStage, src + static_cast<size_t>(i) * kAStage,
                              kAStage, bar_afull + 8 * s);
            }
            if (*abort_flag) {
                // A copy may still be in flight and its barrier can no longer
                // complete: give it a bounded 50 us to land before leaving.
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 50000ull) __nanosleep(1000);
            }
        }
        __syncwarp();
    } else if (warp == C::kMmaWarp) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc(kBM, BN);
            bool ok = true;
            for (int i = 0; i < n_iters; ++i) {
                const int sa = i % C::kAStages;
                const int sb = i % C::kBStages;
                if (!mbar_wait_bounded(bar_afull + 8 * sa, (i / C::kAStages) & 1, abort_flag, err,
                                       kErrTimeoutFull) ||
                    !mbar_wait_bounded(bar_bfull + 8 * sb, (i / C::kBStages) & 1, abort_flag, err,
                                       kErrTimeoutFull)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_addr = sbase + C::kOffA + sa * kAStage;
                const uint32_t b_addr = sbase + C::kOffB + sb * C::kBStage;
#pragma unroll
                for (int kk = 0; kk < kKS / 16; ++kk)
                    mma_bf16(tmem_d, sw128_desc(a_addr + 32 * kk), sw128_desc(b_addr + 32 * kk),
                             idesc, (i | kk) != 0 ? 1u : 0u);
                // both slots are free once these MMAs have read them
                mma_commit(bar_aempty + 8 * sa);
                mma_commit(bar_bempty + 8 * sb);
            }
            if (ok) {
                mma_commit(bar_accum);
            } else {
                // Make sure no MMA is still writing TMEM before it is freed.
                mma_commit(bar_drain);
                volatile int no_abort = 0;
                mbar_wait_bounded(bar_drain, 0, &no_abort, err, kErrTimeoutDrain);
            }
        }
        __syncwarp();
    }

    if (warp < 4) {
        // ---------------- epilogue: TMEM -> y (lane quarter = warp) ----------------
        const bool ok = __all_sync(0xFFFFFFFFu,
                                   mbar_wait_backoff(bar_accum, 0, abort_flag, err, kErrTimeoutAccum, 512));
        if (ok) {
            tc_fence_after();
            const int m = m0 + warp * 32 + lane;
            const uint32_t taddr_row = tmem_d + (static_cast<uint32_t>(warp * 32) << 16);
            const bool vec_ok = (N & 3) == 0;
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(taddr_row + c0, v);
                if (m < M) {
                    float* dst = y + static_cast<size_t>(m) * N + n0 + c0;
                    const int valid = N - (n0 + c0);
                    if (vec_ok && valid >= 32) {
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            reinterpret_cast<float4*>(dst)[q] =
                                make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                            __uint_as_float(v[4 * q + 2]),
                                            __uint_as_float(v[4 * q + 3]));
                    } else {
#pragma unroll
                        for (int q = 0; q < 32; ++q)
                            if (q < valid) dst[q] = __uint_as_float(v[q]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == C::kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_d),
                     "r"(C::kTmemCols)
                     : "memory");
    }
}

// ============================================================================
// Weights-as-A variant (needs the x tile image).  The decoded weights go from
// registers straight into tensor memory (tcgen05.st) and are the MMA's A
// operand there; x stages, copied in bulk from the tile image, are the B
// operand in shared memory.  Per MMA-clock this moves far fewer shared-memory
// bytes than the variant above (no decoded-weight stores or reads), and each
// decoded weight feeds up to 256 x rows instead of 128.
//
// One CTA: 128 weight rows x up to kXRows x rows (kXRows 128 or 256).  The
// MMA is M = 128 (weight rows, TMEM lanes) x N = this tile's x rows padded to
// 16, accumulating into TMEM columns [0, N); decoded stage s (64 K) sits at
// columns kColA + 32 s, K-step t (16 weights, 8 bf16x2 columns) at + 8 t.
//   warps 0-15  decoders, then the epilogue.  Warp w stores to TMEM lanes
//               32 (w % 4) .. + 31; (w / 4) % 2 picks the 16-weight segment of
//               a 32-weight quant group and w / 8 the half of each block (its
//               two 64-K stages) the warp decodes: per block the thread reads
//               16 of its row's 32 quant bytes of that half and the half's
//               scales, and decodes all four 2-bit planes of them, two per
//               stage.  Two groups on alternate stage pairs give each warp
//               twice the time per stage (the decode is latency-bound: a scale
//               table then byte permutes, plus a barrier test per stage)
//   warp 16     TMEM allocation, MMA issue (one thread)
//   warp 17     waits for the next kPair stages to be filled and hands them to
//               the MMA warp at a named barrier both warps pass once per
//               hand-over: the MMA thread never polls an mbarrier, so nothing
//               but MMAs and commits sits between its MMAs (the MMA pipe runs
//               dry while the issuing thread is busy elsewhere)
//   warp 18     raw weight blocks: one 2-D TMA box (128 rows x 112 bytes) per
//               block (without TMA the decoders copy them with 4-byte cp.async)
//   warps 19-20 x stages, even and odd: one bulk copy each (a thread's bulk
//               copies complete one after another, so two issuers double the
//               rate a single one gets)
// ============================================================================

// Bytes per row of the raw-weight TMA box: an 84-byte block starts 0, 4, 8 or
// 12 bytes past a 16-byte boundary, so 96 would do; 112 (28 words) puts rows
// 8 banks apart instead of 24, halving the bank conflicts of the row reads.
constexpr int kTmaBoxBytes = 112;
// x tile image: super-tiles of 256 rows x 64 K (32 KB, 128-byte swizzled,
// K-major), super-tile (t, stage s) at (t * K/64 + s) * 32 KB.
constexpr int kXSuperRows = 256;
constexpr int kXSuperBytes = kXSuperRows * kKS * 2;
// most K parts one weights-as-A grid splits a row's blocks into (also the
// largest portable cluster: the parts of a small-m tile form one cluster)
constexpr int kMaxKParts = 8;
// Small m (x tiles of at most 64 rows): every K stage of the CTA's x rows is
// converted to bf16 by the kernel itself and stays in shared memory, in this
// many bytes.
constexpr int kSmallXBytes = 160 * 1024;
#ifndef Q2K_TC_SMALL_ISSUERS
#define Q2K_TC_SMALL_ISSUERS 2
#endif
#ifndef Q2K_TC_X128_ISSUERS
#define Q2K_TC_X128_ISSUERS 2
#endif
#ifndef Q2K_TC_X128_HANDOVER
#define Q2K_TC_X128_HANDOVER 4
#endif
#ifndef Q2K_TC_X256_HANDOVER
#define Q2K_TC_X256_HANDOVER 2
#endif
#ifndef Q2K_TC_X128_PAIR_RELEASE
#define Q2K_TC_X128_PAIR_RELEASE 1
#endif
#ifndef Q2K_TC_SMALL_ACC
#define Q2K_TC_SMALL_ACC (Q2K_TC_SMALL_ISSUERS)
#endif
#ifndef Q2K_TC_SMALL_STAGES
#define Q2K_TC_SMALL_STAGES 8
#endif
#ifndef Q2K_TC_SMALL_HANDOVER
#define Q2K_TC_SMALL_HANDOVER 4
#endif
#ifndef Q2K_TC_SMALL_FIRST_BOX_ALONE
#define Q2K_TC_SMALL_FIRST_BOX_ALONE 1
#endif

template <int kXRows, bool kTmaW>
struct WtCfg {
    static_assert(kXRows == 16 || kXRows == 32 || kXRows == 64 || kXRows == 128 || kXRows == 256,
                  "x rows per CTA");
    // small m: x converted in the kernel, all of the CTA's K stages resident,
    // K parts summed through the cluster's shared memory
    static constexpr bool kSmall = kXRows <= 64;
    static constexpr int kRows = 128;                       // weight rows per CTA
    static constexpr int kDecWarps = 16;                    // two groups of 8, one per block half
    static constexpr int kGroupWarps = 8;                   // decoders of one stage
    static constexpr int kDecThreads = 32 * kDecWarps;
    static constexpr int kMmaWarp = kDecWarps;
    static constexpr int kWaitWarp = kDecWarps + 1;
    static constexpr int kWWarp = kDecWarps + 2;
    static constexpr int kXWarp0 = kDecWarps + 3;
    static constexpr int kThreads = 32 * (kDecWarps + 5);
    // K stages per MMA hand-over: a hand-over (the waiter's named barrier)
    // costs about as much as one narrow MMA, so small m takes a whole block
    // (four stages) at a time
    static constexpr int kPair =
        kSmall ? Q2K_TC_SMALL_HANDOVER : (kXRows == 128 ? Q2K_TC_X128_HANDOVER : Q2K_TC_X256_HANDOVER);
    static constexpr int kXStage = kXRows * kKS * 2;        // bytes of one x stage
    static constexpr int kXStages = kSmall ? kSmallXBytes / kXStage : (kXRows == 256 ? 6 : 8);
    // x barriers: a full / empty pair per ring stage; small m has one "all of
    // x converted" barrier (one arrival per decoder warp)
    static constexpr int kXBars = kSmall ? 1 : kXStages;
    // Accumulators.  A narrow MMA (16 to 64 x rows) costs about the same
    // whatever its N, and a run of them into one accumulator issues back to
    // back; rotating over several costs more per MMA, so small m keeps one
    // unless Q2K_TC_SMALL_ACC says otherwise.
    // Threads issuing MMAs.  One thread issues narrow MMAs at about half the
    // rate the tensor core takes them, so small m (and 128-row x tiles, whose
    // accumulators leave room for a second) has two: the MMA warp the even
    // stages of a hand-over into accumulator 0, the waiter the odd ones into
    // accumulator 1.
    static constexpr int kIssuers =
        kSmall ? Q2K_TC_SMALL_ISSUERS : (kXRows == 128 ? Q2K_TC_X128_ISSUERS : 1);
    static constexpr int kAcc = kSmall ? Q2K_TC_SMALL_ACC : kIssuers;
    static_assert(kIssuers == 1 || (kIssuers == 2 && kAcc == 2 && kPair % 2 == 0), "MMA issuers");
    static constexpr uint32_t kColA = kXRows * kAcc;        // A ring after the accumulators
    static constexpr int kTmemCols = 512;
    // Decoded stages in TMEM (32 columns each).  The decoders' TMEM stores
    // and the narrow MMAs reading A from TMEM slow each other down; a ring of
    // 8 (Q2K_TC_SMALL_STAGES) keeps the decoders at most two blocks ahead and
    // measured faster than deeper rings (12, 15) or shallower ones (4, 6).
    static constexpr int kAStages =
        kSmall ? std::min(Q2K_TC_SMALL_STAGES, static_cast<int>((kTmemCols - kColA) / 32)) : 8;
    static_assert(kAStages >= 4 && kAStages % 2 == 0,
                  "a block's four stages fit in TMEM at once; small m releases stages in pairs");
    // Stages released to the producers in pairs (one commit per issuer per
    // pair) instead of one by one; with an x ring as deep as the A ring
    // (128-row tiles), one release serves both the x and the A stage.  Each
    // commit costs about as much as a narrow MMA.
    static constexpr bool kPairRelease =
        kSmall || (kXRows == 128 && Q2K_TC_X128_PAIR_RELEASE && kXStages == kAStages);
    // Raw weight slabs: the decoders take a block into registers as soon as it
    // lands, so two slabs keep the next block's copy a whole block ahead.  A
    // small-m CTA has few blocks and little else to hide their latency behind:
    // four slabs keep four blocks in flight.
    static constexpr int kRaw = kSmall ? 4 : (kTmaW ? 2 : 3);
    // Raw slab row pitch: 84 (one block per row, rows copied by cp.async), or
    // the 112-byte TMA box that holds block b at byte 4 (b % 4) (the box
    // starts at the 16-byte boundary at or below the block).
    static constexpr int kRawPitch = kTmaW ? kTmaBoxBytes : kBlockBytes;
    static constexpr int kRawBytes = kRows * kRawPitch;
    static constexpr int kOffX = 0;
    static constexpr int kOffRaw = kXStages * kXStage;
    // bars: x_full[kXBars], x_empty[kXBars], a_full[kAStages], a_empty[kAStages],
    //       raw_full[kRaw], raw_empty[kRaw], accum, drain
    static constexpr int kNumBars = 2 * kXBars + 2 * kAStages + 2 * kRaw + 2;
    static constexpr int kOffBar = ((kOffRaw + kRaw * kRawBytes) + 7) & ~7;
    static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory");
    static_assert(kColA + 32u * kAStages <= static_cast<uint32_t>(kTmemCols), "TMEM");
    static_assert(kRawBytes % 128 == 0 && kOffRaw % 1024 == 0, "TMA destination alignment");
    // the small-m epilogue reuses the x region for the 128 x kXRows f32 slice
    static_assert(!kSmall || kOffRaw >= kRows * kXRows * 4, "reduction slice");
};

// Routed mode of the weights-as-A kernel: x tile t's expert and routed rows
// (tile_info[t] = {expert or -1, rows}), the route of each of those rows
// (row_route[128 t + i], i < rows; padding rows have none), the bytes between
// experts' weights and, for the TMA view of the whole weight pool, the rows
// between them.
struct WtRouted {
    const int2* tile_info = nullptr;
    const int* row_route = nullptr;
    long long expert_stride = 0;
    int expert_rows = 0;
    // small m: kGemvConstWeights (no grid that may still run writes W: the
    // weight copies start before the dependency wait) and kGemvIndependent (it
    // touches neither x, W nor y: nothing waits for it but CTA (0, 0, 0),
    // before it exits, so calls still complete in stream order)
    uint32_t flags = 0;
};

// ---- thread-block cluster: barrier and distributed shared memory -----------

// Every thread of every CTA in the cluster arrives (release) and waits
// (acquire): shared-memory writes before it are visible to the whole cluster.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_cta_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// The address of this CTA's shared-memory word `saddr` in cluster CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map_shared(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
// Four consecutive floats of (another CTA's) shared memory in the cluster
// (16-byte aligned).
__device__ __forceinline__ float4 ld_shared_cluster_v4f(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// D[tmem_d] (+)= A[tmem_a] * B[bdesc]^T with A in tensor memory.
__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc,
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(tmem_d), "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Eight consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
        ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
          "r"(v[6]), "r"(v[7])
        : "memory");
}

// 2-D tiled TMA load of the box at (x, y) into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
          "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Stage Cp (0 or 1) of one half of a block for one thread: the two 16-weight
// K-steps of quant segment `seg` at the 2-bit planes J = 2 Cp + {0, 1}.  qh =
// the thread's four quant words of the half, sh = the half's two scale words
// shifted right by 8 seg (the segment's byte at the low byte of each 16-bit
// lane).  o0 gets K-step seg, o1 K-step 2 + seg; word 2e (2e + 1) holds the
// weights of quant byte lanes 4e, 4e + 1 (4e + 2, 4e + 3).
template <int Cp>
__device__ __forceinline__ void wt_decode_half_stage(const uint32_t* qh, const uint32_t* sh, float d,
                                                     float dmin, uint32_t (&o0)[8],
                                                     uint32_t (&o1)[8]) {
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
        constexpr int kJ0 = 2 * Cp;
        const int j = kJ0 + jj;
        // scale index 8 H + 2 j + seg -> word j / 2 of the half, byte 2 (j % 2) + seg
        const uint32_t sc = (sh[j >> 1] >> (16 * (j & 1))) & 0xFFu;
        const float dl = __fmul_rn(d, static_cast<float>(sc & 15u));
        const float ml = __fmul_rn(dmin, static_cast<float>(sc >> 4));
        const uint32_t lo = pack_bf16x2(-ml, __fsub_rn(dl, ml));
        const uint32_t hi = pack_bf16x2(fmaf(2.f, dl, -ml), fmaf(3.f, dl, -ml));
        uint32_t* o = jj == 0 ? o0 : o1;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (kJ0 + jj == 0) decode_word<0>(qh[e], lo, hi, o[2 * e], o[2 * e + 1]);
            else if (kJ0 + jj == 1) decode_word<1>(qh[e], lo, hi, o[2 * e], o[2 * e + 1]);
            else if (kJ0 + jj == 2) decode_word<2>(qh[e], lo, hi, o[2 * e], o[2 * e + 1]);
            else decode_word<3>(qh[e], lo, hi, o[2 * e], o[2 * e + 1]);
        }
    }
}

// Copy block b (84 bytes per row) of the CTA's kRows weight rows into a raw
// slab, row r at dst + 84 r; rows past N are zero-filled (they decode to 0).
template <int kRows, int kThreadsDec>
__device__ __forceinline__ void wt_issue_raw(const uint8_t* __restrict__ w, uint32_t dst, int n0,
                                             int N, size_t row_bytes, int b, int td) {
    constexpr int kWords = kRows * kWordsPerBlock;
#pragma unroll 4
    for (int f = td; f < kWords; f += kThreadsDec) {
        const int r = f / kWordsPerBlock;
        const int wd = f - r * kWordsPerBlock;
        const bool ok = n0 + r < N;
        const uint8_t* src = w + (ok ? static_cast<size_t>(n0 + r) * row_bytes +
                                           static_cast<size_t>(b) * kBlockBytes + 4 * wd
                                     : 0);
        cp_async_4(dst + r * kBlockBytes + 4 * wd, src, ok ? 4u : 0u);
    }
    cp_async_commit();
}

template <int kXRows, bool kTmaW>
__global__ void __launch_bounds__(WtCfg<kXRows, kTmaW>::kThreads, 1)
gemm_wt_kernel(const uint8_t* __restrict__ xa, const float* __restrict__ xf,
               const uint8_t* __restrict__ w, float* __restrict__ y, float* __restrict__ partial,
               unsigned int* __restrict__ tile_count, int M, int N, int K, WtRouted rt,
               const __grid_constant__ CUtensorMap tmap_w) {
    using C = WtCfg<kXRows, kTmaW>;
    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * C::kRows;
    const int m0 = blockIdx.y * kXRows;
    // Routed mode: x tile blockIdx.y holds rows of one expert (tile_info: the
    // expert, the tile's routed rows; -1: none, and the CTA leaves before any
    // set-up); its weights are that expert's, its outputs go to their routes.
    int tma_row0 = 0;  // the expert's first row in the TMA view of the weight pool
    int tile_rows = M - m0;
    if (rt.tile_info != nullptr) {
        const int2 ti = __ldg(rt.tile_info + blockIdx.y);
        if (ti.x < 0) return;
        w += static_cast<size_t>(ti.x) * rt.expert_stride;
        tma_row0 = ti.x * rt.expert_rows;
        tile_rows = ti.y;
    }
    const int nx = min(kXRows, (tile_rows + 15) & ~15);  // MMA N: the tile's x rows, padded to 16
    const int blocks_per_row = K / kQK;
    const size_t row_bytes = static_cast<size_t>(blocks_per_row) * kBlockBytes;
    // K split (gridDim.z parts): this CTA's blocks [kb0, kb0 + n_blocks) of each
    // row; loop indices below are relative to kb0 unless named otherwise
    const int kb0 = static_cast<int>(static_cast<long>(blockIdx.z) * blocks_per_row / gridDim.z);
    const int n_blocks =
        static_cast<int>(static_cast<long>(blockIdx.z + 1) * blocks_per_row / gridDim.z) - kb0;
    const int n_iters = 4 * n_blocks;  // 64-K stages
    const int n_stages_row = K / kKS;  // stages of a whole row (x image layout)

    const uint32_t bar_xfull = sbase + C::kOffBar;
    const uint32_t bar_xempty = bar_xfull + 8 * C::kXBars;
    const uint32_t bar_afull = bar_xempty + 8 * C::kXBars;
    const uint32_t bar_aempty = bar_afull + 8 * C::kAStages;
    const uint32_t bar_raw = bar_aempty + 8 * C::kAStages;
    const uint32_t bar_rawempty = bar_raw + 8 * C::kRaw;
    const uint32_t bar_accum = bar_rawempty + 8 * C::kRaw;
    const uint32_t bar_drain = bar_accum + 8;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
    unsigned int* err = &g_tc_error;

    if constexpr (C::kSmall) {
        // The grid before this one may still run (programmatic launch): set up
        // now, read x and W and write y only after waiting for it.
        pdl_allow_dependents();
    }
    if (warp == 0) {
        // the barriers are set up by the lanes of warp 0 in parallel
        for (int s = lane; s < C::kXBars; s += 32) {
            // producer's expect-tx arrival + the copy's bytes; small m: one
            // arrival per decoder warp once its share of x is converted
            mbar_init(bar_xfull + 8 * s, C::kSmall ? C::kDecWarps : 1);
            mbar_init(bar_xempty + 8 * s, 1);  // MMA commit
        }
        for (int s = lane; s < C::kAStages; s += 32) {
            mbar_init(bar_afull + 8 * s, C::kGroupWarps);  // one arrival per warp of its group
            // MMA commit(s): small m releases stages in pairs, one commit
            // from each issuer
            mbar_init(bar_aempty + 8 * s, C::kPairRelease ? C::kIssuers : 1);
        }
        for (int r = lane; r < C::kRaw; r += 32) {
            // TMA: the producer's expect-tx arrival + the box bytes; else one
            // arrival per decoder warp once its cp.async groups landed
            mbar_init(bar_raw + 8 * r, kTmaW ? 1 : C::kDecWarps);
            mbar_init(bar_rawempty + 8 * r, C::kDecWarps);  // decoders done reading (kTmaW)
        }
        if (lane == 0) {
            mbar_init(bar_accum, C::kIssuers);
            mbar_init(bar_drain, C::kIssuers);
            *abort_flag = 0;
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == C::kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(C::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

    if (warp < C::kDecWarps) {
        // ---------------- weight decoders ----------------
        const int td = threadIdx.x;
        const int quarter = warp & 3;
        const int seg = (warp >> 2) & 1;
        const int half = warp >> 3;           // block half = stages 2 half, 2 half + 1
        const int row = 32 * quarter + lane;  // weight row within the tile = TMEM lane
        const uint32_t raw0 = sbase + C::kOffRaw;
        const uint32_t t_lane = static_cast<uint32_t>(32 * quarter) << 16;
        // A columns of K-steps seg and 2 + seg, stage 0
        const uint32_t a_col0 = tmem_base + t_lane + C::kColA + 8u * seg;
        if constexpr (C::kSmall) {
            // x (and W) may be written by the grid before this one
            if (!(rt.flags & kGemvIndependent)) pdl_wait_prerequisites();
            // x rows m0 .. m0 + nx - 1 over the CTA's K stages -> bf16, stage i
            // at kOffX + i kXStage in the swizzled K-major layout the MMA reads
            // (rows past M as zeros).  One 16-byte chunk (8 K-elements) per
            // thread and pass, four passes' loads issued before any store.
            const int chunks = n_iters * nx * 8;
            const float* xk = xf + static_cast<size_t>(kb0) * kQK;
            for (int c0 = td; c0 < chunks; c0 += 4 * C::kDecThreads) {
                float4 lo[4], hi[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int c = c0 + u * C::kDecThreads;
                    const int r = (c >> 3) % nx;
                    const int i = (c >> 3) / nx;
                    lo[u] = hi[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (c < chunks && m0 + r < M) {
                        const float4* src = reinterpret_cast<const float4*>(
                            xk + static_cast<size_t>(m0 + r) * K + kKS * i + 8 * (c & 7));
                        lo[u] = __ldg(src);
                        hi[u] = __ldg(src + 1);
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int c = c0 + u * C::kDecThreads;
                    if (c < chunks) {
                        const int r = (c >> 3) % nx;
                        const int i = (c >> 3) / nx;
                        st_shared_v4(sbase + C::kOffX + i * C::kXStage + sw128_offset(r, c & 7),
                                     pack_bf16x2(lo[u].x, lo[u].y), pack_bf16x2(lo[u].z, lo[u].w),
                                     pack_bf16x2(hi[u].x, hi[u].y), pack_bf16x2(hi[u].z, hi[u].w));
                    }
                }
            }
            fence_proxy_async_smem();  // this thread's stores -> visible to the MMA
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_xfull);
        }
        if constexpr (!kTmaW) {
            // Pull the tile's weight rows into L2 now (one bulk prefetch per row).
            if (td < C::kRows && n0 + td < N) {
                const uint8_t* rp = w + static_cast<size_t>(n0 + td) * row_bytes;
                const uintptr_t a = (reinterpret_cast<uintptr_t>(rp) + 15) & ~uintptr_t(15);
                const uintptr_t e = (reinterpret_cast<uintptr_t>(rp) + row_bytes) & ~uintptr_t(15);
                if (e > a)
                    bulk_prefetch_l2(reinterpret_cast<const void*>(a), static_cast<uint32_t>(e - a));
            }
            for (int pb = 0; pb < C::kRaw - 1; ++pb) {
                if (pb < n_blocks)
                    wt_issue_raw<C::kRows, C::kDecThreads>(w, raw0 + pb * C::kRawBytes, n0, N,
                                                           row_bytes, kb0 + pb, td);
                else
                    cp_async_commit();
            }
        }
        bool ok = true;
        for (int b = 0; b < n_blocks && ok; ++b) {
            const int buf = b % C::kRaw;
            uint32_t mine;
            if constexpr (kTmaW) {
                if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(bar_raw + 8 * buf, (b / C::kRaw) & 1,
                                                               abort_flag, err, kErrTimeoutEmpty))) {
                    ok = false;
                    break;
                }
                mine = raw0 + buf * C::kRawBytes + row * C::kRawPitch + 4 * ((kb0 + b) & 3);
            } else {
                cp_async_wait_group<C::kRaw - 2>();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_raw + 8 * buf);
                if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(bar_raw + 8 * buf, (b / C::kRaw) & 1,
                                                               abort_flag, err, kErrTimeoutEmpty))) {
                    ok = false;
                    break;
                }
                // Every decoder has read block b - 1's slab (it arrived for block
                // b above): block b + kRaw - 1 goes there.
                const int nb = b + C::kRaw - 1;
                if (nb < n_blocks)
                    wt_issue_raw<C::kRows, C::kDecThreads>(w, raw0 + (nb % C::kRaw) * C::kRawBytes,
                                                           n0, N, row_bytes, kb0 + nb, td);
                else
                    cp_async_commit();
                mine = raw0 + buf * C::kRawBytes + row * kBlockBytes;
            }
            uint32_t sh[2], qh[4];
#pragma unroll
            for (int q = 0; q < 2; ++q) sh[q] = ld_shared_u32(mine + 8 * half + 4 * q) >> (8 * seg);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                qh[e] = ld_shared_u32(mine + 16 + 32 * half + 16 * seg + 4 * e);
            const uint32_t dd = ld_shared_u32(mine + 80);
            if constexpr (kTmaW) {
                // this warp has its block in registers: the slab may be refilled
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_rawempty + 8 * buf);
            }
            const float d = f16_bits_to_float(dd);
            const float dmin = f16_bits_to_float(dd >> 16);
#pragma unroll
            for (int cp = 0; cp < 2; ++cp) {
                const int i = 4 * b + 2 * half + cp;
                const int s = i % C::kAStages;
                uint32_t o0[8], o1[8];
                if (cp == 0) wt_decode_half_stage<0>(qh, sh, d, dmin, o0, o1);
                else wt_decode_half_stage<1>(qh, sh, d, dmin, o0, o1);
                // (small m releases stages in pairs: the release of stage
                // i | 1 covers stage i too)
                const int rel = (C::kPairRelease ? (i | 1) : i) % C::kAStages;
                if (i >= C::kAStages &&
                    !__all_sync(0xFFFFFFFFu,
                                mbar_wait_bounded(bar_aempty + 8 * rel, ((i / C::kAStages) - 1) & 1,
                                                  abort_flag, err, kErrTimeoutEmpty))) {
                    ok = false;
                    break;
                }
                tc_fence_after();  // the MMAs that read this stage are done
                const uint32_t a_col = a_col0 + 32u * s;
                tmem_st8(a_col, o0);
                tmem_st8(a_col + 16u, o1);
                // published as soon as its stores have landed (waiting here
                // measured faster than deferring it past the next decode)
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_afull + 8 * s);
            }
        }
        if constexpr (!kTmaW) cp_async_wait_all();  // no copy may land after this CTA is gone

        // ---------------- epilogue: TMEM -> y ----------------
        const bool acc_ok = __all_sync(
            0xFFFFFFFFu, mbar_wait_backoff(bar_accum, 0, abort_flag, err, kErrTimeoutAccum, 512));
        if (acc_ok) {
            tc_fence_after();
            const int n = n0 + row;
            const uint32_t t_row = tmem_base + t_lane;
            // 16-column groups rotate over the four warps of a lane quarter
#pragma unroll 1
            for (int c0 = 16 * (warp >> 2); c0 < nx; c0 += 64) {
                uint32_t v[16];
                tmem_ld16(t_row + c0, v);
#pragma unroll 1
                for (int a = 1; a < C::kAcc; ++a) {  // the accumulators, summed in order
                    uint32_t u[16];
                    tmem_ld16(t_row + static_cast<uint32_t>(a * kXRows) + c0, u);
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        v[q] = __float_as_uint(__uint_as_float(v[q]) + __uint_as_float(u[q]));
                }
                if (C::kSmall && gridDim.z > 1) {
                    // this part's slice, column-major (x row c, weight row
                    // `row` at word 128 c + row), in the x region the MMAs
                    // are done with; the cluster sums the parts below
                    float* red = reinterpret_cast<float*>(smem + C::kOffX);
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        if (c0 + q < nx) red[(c0 + q) * C::kRows + row] = __uint_as_float(v[q]);
                    continue;
                }
                // one K part alone goes to y; parts of a split go to their own
                // slice of the partial buffer, summed in part order below
                float* out = gridDim.z == 1 ? y : partial + static_cast<size_t>(blockIdx.z) * M * N;
                if (n < N && rt.row_route == nullptr) {
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int m = m0 + c0 + q;
                        if (m < M) out[static_cast<size_t>(m) * N + n] = __uint_as_float(v[q]);
                    }
                } else if (n < N) {
                    // routed: x row m < tile_rows is route row_route[m]
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int m = m0 + c0 + q;
                        if (c0 + q >= tile_rows) continue;
                        const int r = __ldg(rt.row_route + m);
                        if (r >= 0) out[static_cast<size_t>(r) * N + n] = __uint_as_float(v[q]);
                    }
                }
            }
        }
        if (!C::kSmall && gridDim.z > 1) {
            // K split: every part has stored its slice; the part that arrives last
            // at this tile's counter sums the slices in part order into y (no CTA
            // ever waits for another).  The counter was zeroed by the grid before.
            // The barrier orders every decoder thread's slice stores before one
            // thread's device-scope fence and count (the release); that thread
            // fences again after the count (the acquire) before the barrier that
            // lets the others read.
            volatile int* last = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
            asm volatile("bar.sync 2, %0;" ::"n"(C::kDecThreads) : "memory");
            if (td == 0) {
                __threadfence();
                pdl_wait_prerequisites();
                const unsigned prev = atomicAdd(&tile_count[blockIdx.y * gridDim.x + blockIdx.x], 1u);
                __threadfence();
                *last = prev == gridDim.z - 1 ? 1 : 0;
            }
            asm volatile("bar.sync 2, %0;" ::"n"(C::kDecThreads) : "memory");
            if (*last) {
                // all the loads of a pass are issued before any sum: one L2
                // round trip per pass instead of one per part and element
                constexpr int kMaxParts = kMaxKParts;
                constexpr int kPer = 4;
                const int parts = static_cast<int>(gridDim.z);
                const size_t mn = static_cast<size_t>(M) * N;
                const int total = C::kRows * nx;
                for (int base = td; base < total; base += kPer * C::kDecThreads) {
                    float v[kPer][kMaxParts];
                    size_t off[kPer];
                    bool ok[kPer];
#pragma unroll
                    for (int j = 0; j < kPer; ++j) {
                        const int idx = base + j * C::kDecThreads;
                        const int nn = n0 + (idx & (C::kRows - 1));
                        const int mm = m0 + idx / C::kRows;
                        ok[j] = idx < total && nn < N && mm < M;
                        off[j] = ok[j] ? static_cast<size_t>(mm) * N + nn : 0;
#pragma unroll
                        for (int p = 0; p < kMaxParts; ++p)
                            v[j][p] = ok[j] && p < parts ? __ldcg(partial + p * mn + off[j]) : 0.f;
                    }
#pragma unroll
                    for (int j = 0; j < kPer; ++j) {
                        if (!ok[j]) continue;
                        float sum = v[j][0];
#pragma unroll
                        for (int p = 1; p < kMaxParts; ++p)
                            if (p < parts) sum += v[j][p];
                        y[off[j]] = sum;
                    }
                }
            }
        }
    } else if (warp == C::kMmaWarp) {
        // ---------------- MMA issuer ----------------
        // Both this warp and the waiter pass named barrier 1 exactly
        // n_iters / kPair times, whatever happens, so neither can be left
        // waiting there; after an abort the MMAs are skipped.  Everything but
        // the MMAs is worked out per stage: x stage s starts kXStage bytes
        // (kXStage / 16 descriptor units) after stage s - 1, each K-step 32
        // bytes (2 units) after the previous one.
        const uint32_t idesc = make_idesc(kBM, nx);
        const uint64_t xdesc0 = sw128_desc(sbase + C::kOffX);
        const uint32_t a_base0 = tmem_base + C::kColA;
        for (int i0 = 0; i0 < n_iters; i0 += C::kPair) {
            asm volatile("bar.sync 1, 64;" ::: "memory");
            if (lane == 0 && !*abort_flag) {
                tc_fence_after();
#pragma unroll
                for (int u = 0; u < C::kPair; ++u) {
                    if (C::kIssuers > 1 && (u & 1)) continue;  // the waiter's stages
                    const int i = i0 + u;
                    const int sx = i % C::kXStages;
                    const int sa = i % C::kAStages;
                    const uint64_t xdesc = xdesc0 + static_cast<uint64_t>(sx * (C::kXStage >> 4));
                    const uint32_t a_s = a_base0 + 32u * sa;
#pragma unroll
                    for (int kk = 0; kk < kKS / 16; ++kk) {
                        // MMA g = 4 i + kk goes to accumulator g % kAcc (with
                        // two issuers: accumulator 0, stage i / 2 of this
                        // thread's); the first one into each starts it from zero
                        const int g = C::kIssuers > 1 ? 4 * (i >> 1) + kk : 4 * i + kk;
                        const uint32_t d =
                            tmem_base + static_cast<uint32_t>((C::kIssuers > 1 ? 0 : g % C::kAcc) * kXRows);
                        mma_bf16_tmem_a(d, a_s + 8u * kk, xdesc + 2u * kk, idesc,
                                        g >= (C::kIssuers > 1 ? 1 : C::kAcc) ? 1u : 0u);
                    }
                    // a stage is released only when the decoders refill it;
                    // small m releases them in pairs, after the second one's
                    // MMAs (a commit covers every MMA of its thread before
                    // it; with two issuers each commits its stage of the
                    // pair), since each commit costs about as much as a narrow MMA
                    if (C::kPairRelease ? ((C::kIssuers > 1 || (i & 1)) && (i & ~1) + C::kAStages < n_iters)
                                  : i + C::kAStages < n_iters)
                        mma_commit(bar_aempty + 8 * ((C::kPairRelease ? (i | 1) : i) % C::kAStages));
                    if (!C::kSmall && !C::kPairRelease) mma_commit(bar_xempty + 8 * sx);
                }
            }
            __syncwarp();
        }
        if (lane == 0) {
            if (!*abort_flag) {
                mma_commit(bar_accum);
            } else {
                // Make sure no MMA is still writing TMEM before it is freed.
                mma_commit(bar_drain);
                volatile int no_abort = 0;
                mbar_wait_bounded(bar_drain, 0, &no_abort, err, kErrTimeoutDrain);
            }
        }
        __syncwarp();
    } else if (warp == C::kWaitWarp) {
        // ---------------- stage waiter: hands filled stages to the MMA warp ----------------
        if (C::kSmall && lane == 0)  // all of x, once
            mbar_wait_bounded(bar_xfull, 0, abort_flag, err, kErrTimeoutFull);
        for (int i0 = 0; i0 < n_iters; i0 += C::kPair) {
            if (lane == 0 && !*abort_flag) {
#pragma unroll
                for (int u = 0; u < C::kPair; ++u) {
                    const int i = i0 + u;
                    if ((!C::kSmall &&
                         !mbar_wait_bounded(bar_xfull + 8 * (i % C::kXStages), (i / C::kXStages) & 1,
                                            abort_flag, err, kErrTimeoutFull)) ||
                        !mbar_wait_bounded(bar_afull + 8 * (i % C::kAStages), (i / C::kAStages) & 1,
                                           abort_flag, err, kErrTimeoutFull))
                        break;
                }
            }
            __syncwarp();
            asm volatile("bar.sync 1, 64;" ::: "memory");
            if constexpr (C::kIssuers > 1) {
                // second issuer: the odd stages of the hand-over, into
                // accumulator 1 (the epilogue adds the accumulators in order)
                if (lane == 0 && !*abort_flag) {
                    tc_fence_after();
                    const uint32_t idesc = make_idesc(kBM, nx);
                    const uint64_t xdesc0 = sw128_desc(sbase + C::kOffX);
                    const uint32_t a_base0 = tmem_base + C::kColA;
#pragma unroll
                    for (int u = 1; u < C::kPair; u += 2) {
                        const int i = i0 + u;
                        const int sx = i % C::kXStages;
                        const int sa = i % C::kAStages;
                        const uint64_t xdesc = xdesc0 + static_cast<uint64_t>(sx * (C::kXStage >> 4));
                        const uint32_t a_s = a_base0 + 32u * sa;
#pragma unroll
                        for (int kk = 0; kk < kKS / 16; ++kk)
                            mma_bf16_tmem_a(tmem_base + static_cast<uint32_t>(kXRows), a_s + 8u * kk,
                                            xdesc + 2u * kk, idesc, (i > 1 || kk > 0) ? 1u : 0u);
                        if (C::kPairRelease ? (i & ~1) + C::kAStages < n_iters : i + C::kAStages < n_iters)
                            mma_commit(bar_aempty + 8 * sa);
                        if (!C::kSmall && !C::kPairRelease) mma_commit(bar_xempty + 8 * sx);
                    }
                }
                __syncwarp();
            }
        }
        if constexpr (C::kIssuers > 1) {
            if (lane == 0) {
                if (!*abort_flag) {
                    mma_commit(bar_accum);
                } else {
                    mma_commit(bar_drain);
                    volatile int no_abort = 0;
                    mbar_wait_bounded(bar_drain, 0, &no_abort, err, kErrTimeoutDrain);
                }
            }
            __syncwarp();
        }
    } else if (warp == C::kWWarp) {
        // ---------------- raw weight blocks: one TMA box per block ----------------
        if (kTmaW && lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_w))
                         : "memory");
            if (C::kSmall && !(rt.flags & (kGemvConstWeights | kGemvIndependent)))
                pdl_wait_prerequisites();  // W may be written by it
            const uint32_t raw0 = sbase + C::kOffRaw;
            for (int b = 0; b < n_blocks; ++b) {
                const int buf = b % C::kRaw;
                if (b >= C::kRaw &&
                    !mbar_wait_bounded(bar_rawempty + 8 * buf, ((b / C::kRaw) - 1) & 1, abort_flag,
                                       err, kErrTimeoutEmpty))
                    break;
                // Small m: every CTA of the grid asks for its first block at
                // once; the rest follow when that one has landed, so the
                // first blocks are not queued behind the others in DRAM and
                // decoding starts earlier.
                if (C::kSmall && Q2K_TC_SMALL_FIRST_BOX_ALONE && b == 1 &&
                    !mbar_wait_bounded(bar_raw, 0, abort_flag, err, kErrTimeoutFull))
                    break;
                mbar_arrive_expect_tx(bar_raw + 8 * buf, C::kRawBytes);
                // x: the 16-byte boundary at or below row block kb0 + b
                // (84 (kb0 + b) - 4 ((kb0 + b) % 4))
                tma_load_2d(raw0 + buf * C::kRawBytes, &tmap_w, (kBlockBytes * (kb0 + b)) & ~15,
                            tma_row0 + n0, bar_raw + 8 * buf);
            }
            if (*abort_flag) {
                // a copy may still be in flight: give it a bounded 50 us to land
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 50000ull) __nanosleep(1000);
            }
        }
        __syncwarp();
    } else {
        // ---------------- x stages: one bulk copy each, even / odd stages ----------------
        // (small m: the decoders converted x already)
        if (!C::kSmall && lane == 0) {
            // This tile's rows of super-tile m0 / 256 (the second 128 of them when
            // the tile starts half-way into it); a whole super-tile stage when
            // kXRows is 256.  Image rows past M are never written: they feed only
            // the accumulator columns of x rows >= M, which the epilogue drops.
            const uint8_t* src = xa +
                                 (static_cast<size_t>(m0 / kXSuperRows) * n_stages_row + 4 * kb0) *
                                     kXSuperBytes +
                                 static_cast<size_t>(m0 % kXSuperRows) * (kKS * 2);
            const uint32_t bytes = kXRows == kXSuperRows ? static_cast<uint32_t>(kXSuperBytes)
                                                         : static_cast<uint32_t>(nx) * (kKS * 2);
            // The image is written by the grid before this one, unless it is
            // ready from an earlier call (kImageReady): wait for it, then let
            // the next grid start on the SMs this one leaves free (every
            // later grid of the library waits before it reads what this one
            // writes, or is independent of it).
            if (!(rt.flags & kImageReady)) pdl_wait_prerequisites();
            pdl_allow_dependents();
            for (int i = warp - C::kXWarp0; i < n_iters; i += 2) {
                const int s = i % C::kXStages;
                if (i >= C::kXStages &&
                    !mbar_wait_bounded(C::kPairRelease ? bar_aempty + 8 * ((i | 1) % C::kAStages)
                                                       : bar_xempty + 8 * s,
                                       ((i / C::kXStages) - 1) & 1, abort_flag,
                                       err, kErrTimeoutEmpty))
                    break;
                mbar_arrive_expect_tx(bar_xfull + 8 * s, bytes);
                bulk_copy_g2s(sbase + C::kOffX + s * C::kXStage,
                              src + static_cast<size_t>(i) * kXSuperBytes, bytes, bar_xfull + 8 * s);
            }
            if (*abort_flag) {
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 50000ull) __nanosleep(1000);
            }
        }
        __syncwarp();
    }

    if constexpr (C::kSmall) {
        if (gridDim.z > 1) {
            // The K parts of this tile are the CTAs of one cluster, each with
            // its slice in shared memory.  Every thread of the cluster passes
            // both barriers whatever happened before (no role returns early),
            // so neither can be left waiting.  Part r sums its share of the
            // tile's elements over the parts in part order (deterministic);
            // the second barrier keeps every slice alive until all are read.
            __syncwarp();
            cluster_sync_all();
            if (warp < C::kDecWarps) {
                const int parts = static_cast<int>(gridDim.z);
                const int rank = static_cast<int>(cluster_cta_rank());
                // part `rank` sums quads (4 consecutive elements, 16 bytes)
                // [q0, q1) of the tile's 32 nx quads
                const int quads = C::kRows * nx / 4;
                const int q0 = rank * quads / parts;
                const int q1 = (rank + 1) * quads / parts;
                const uint32_t red = sbase + C::kOffX;
                uint32_t src[kMaxKParts];
#pragma unroll
                for (int p = 0; p < kMaxKParts; ++p)
                    src[p] = cluster_map_shared(red, static_cast<uint32_t>(p < parts ? p : 0));
                // this thread's sums wait in registers until the second
                // barrier (a release arrival would otherwise wait for their
                // global stores): at most ceil(32 * 64 / 2 / 512) quads
                constexpr int kPer = (C::kRows * kXRows / 4 / 2 + C::kDecThreads - 1) / C::kDecThreads;
                float4 sums[kPer];
#pragma unroll
                for (int j = 0; j < kPer; ++j) {
                    const int q = q0 + static_cast<int>(threadIdx.x) + j * C::kDecThreads;
                    if (q >= q1) break;
                    float4 v[kMaxKParts];
#pragma unroll
                    for (int p = 0; p < kMaxKParts; ++p)
                        v[p] = p < parts ? ld_shared_cluster_v4f(src[p] + 16u * q)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                    float4 sum = v[0];
#pragma unroll
                    for (int p = 1; p < kMaxKParts; ++p) {
                        if (p < parts) {
                            sum.x += v[p].x;
                            sum.y += v[p].y;
                            sum.z += v[p].z;
                            sum.w += v[p].w;
                        }
                    }
                    sums[j] = sum;
                }
                __syncwarp();
                cluster_sync_all();
#pragma unroll
                for (int j = 0; j < kPer; ++j) {
                    const int q = q0 + static_cast<int>(threadIdx.x) + j * C::kDecThreads;
                    if (q >= q1) break;
                    // elements 4 q .. 4 q + 3: weight rows n0 + (4 q % 128) + 0..3 of x row m
                    const int nn = n0 + ((4 * q) & (C::kRows - 1));
                    const int mm = m0 + 4 * q / C::kRows;
                    if (mm >= M) continue;
                    float* out = y + static_cast<size_t>(mm) * N + nn;
                    if (nn < N) out[0] = sums[j].x;
                    if (nn + 1 < N) out[1] = sums[j].y;
                    if (nn + 2 < N) out[2] = sums[j].z;
                    if (nn + 3 < N) out[3] = sums[j].w;
                }
            } else {
                __syncwarp();
                cluster_sync_all();
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == C::kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(C::kTmemCols)
                     : "memory");
    }
    // An independent call (or one on a ready image, which never waited)
    // completes only after the grid before it, so work enqueued later on the
    // stream sees every earlier call complete.
    if (((C::kSmall && (rt.flags & kGemvIndependent)) || (!C::kSmall && (rt.flags & kImageReady))) &&
        threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
        pdl_wait_prerequisites();
}

// x (f32 [M, K]) -> bf16 in the tile image the GEMM copies into shared memory:
// super-tile (t, K stage s) is 32 KB at xa + (t * K/64 + s) * 32768 and holds
// rows 256 t .. 256 t + 255 (zeros past M) x K 64 s .. 64 s + 63 in the
// 128-byte-swizzled K-major layout (8-row groups 1024 bytes apart).  One
// thread writes one 16-byte chunk.
__device__ __forceinline__ void x_chunk_load(const float* __restrict__ x, int M, int K, size_t id,
                                             float4& lo, float4& hi) {
    const int chunks_per_row = K >> 3;
    const int m = static_cast<int>(id / chunks_per_row);
    const int j = static_cast<int>(id - static_cast<size_t>(m) * chunks_per_row);
    lo = hi = make_float4(0.f, 0.f, 0.f, 0.f);
    if (m < M) {
        const float4* src = reinterpret_cast<const float4*>(x + static_cast<size_t>(m) * K + 8 * j);
        lo = __ldg(src);
        hi = __ldg(src + 1);
    }
}
__device__ __forceinline__ void x_chunk_store(uint8_t* __restrict__ xa, int K, size_t id,
                                              const float4& lo, const float4& hi) {
    const int chunks_per_row = K >> 3;
    const int stages = K / kKS;
    const int m = static_cast<int>(id / chunks_per_row);
    const int j = static_cast<int>(id - static_cast<size_t>(m) * chunks_per_row);
    const uint4 packed = make_uint4(pack_bf16x2(lo.x, lo.y), pack_bf16x2(lo.z, lo.w),
                                    pack_bf16x2(hi.x, hi.y), pack_bf16x2(hi.z, hi.w));
    const size_t tile = static_cast<size_t>(m / kXSuperRows) * stages + (j >> 3);
    *reinterpret_cast<uint4*>(xa + tile * kXSuperBytes + sw128_offset(m % kXSuperRows, j & 7)) =
        packed;
}

// The GEMM after this kernel is launched as its programmatic dependent: it may
// start (TMEM, barriers, weight decode) as soon as every block here has begun,
// and waits for this grid to finish only before it copies the image.  Few
// blocks per SM leave room for it.  Each thread converts four chunks per
// pass, all their loads issued before any store.
__global__ void __launch_bounds__(256)
x_to_bf16_tiles_kernel(const float* __restrict__ x, uint8_t* __restrict__ xa, int M, int K,
                       size_t n_chunks, unsigned int* __restrict__ tile_count, int n_tiles) {
    pdl_allow_dependents();
    // the GEMM's per-tile arrival counters of a split K start at zero each call
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < n_tiles; t += gridDim.x * blockDim.x)
        tile_count[t] = 0u;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    constexpr int kPer = 4;
    for (size_t base = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; base < n_chunks;
         base += kPer * stride) {
        float4 lo[kPer], hi[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u)
            if (base + u * stride < n_chunks) x_chunk_load(x, M, K, base + u * stride, lo[u], hi[u]);
#pragma unroll
        for (int u = 0; u < kPer; ++u)
            if (base + u * stride < n_chunks) x_chunk_store(xa, K, base + u * stride, lo[u], hi[u]);
    }
}

template <int BN, bool kBulkA>
cudaError_t launch_bn(const float* x, const uint8_t* xa, const uint8_t* w, float* y, int M, int N,
                      int K, int device, cudaStream_t stream) {
    using C = Cfg<BN, kBulkA>;
    static bool attr_done[64] = {};
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    if (!attr_done[device]) {
        cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<BN, kBulkA>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done[device] = true;
    }
    dim3 grid((N + BN - 1) / BN, (M + kBM - 1) / kBM);
    gemm_tc_kernel<BN, kBulkA><<<grid, C::kThreads, C::kSmemBytes, stream>>>(x, xa, w, y, M, N, K);
    return cudaGetLastError();
}

template <bool kBulkA>
cudaError_t launch_width(int bn, const float* x, const uint8_t* xa, const uint8_t* w, float* y,
                         int M, int N, int K, int device, cudaStream_t stream) {
    switch (bn) {
        case 256: return launch_bn<256, kBulkA>(x, xa, w, y, M, N, K, device, stream);
        case 192: return launch_bn<192, kBulkA>(x, xa, w, y, M, N, K, device, stream);
        case 128: return launch_bn<128, kBulkA>(x, xa, w, y, M, N, K, device, stream);
        default: return launch_bn<64, kBulkA>(x, xa, w, y, M, N, K, device, stream);
    }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, []() {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// The raw weights as a 2-D byte tensor (N rows of K/256 * 84 bytes) with a
// box of kRows rows x 112 bytes.  Needs 16-byte rows (K a multiple of 1024)
// and a 16-byte aligned base; false when that or the encoder is unavailable.
bool make_weight_map(CUtensorMap* map, const uint8_t* w, int N, int K, int rows) {
    const uint64_t row_bytes = static_cast<uint64_t>(K / kQK) * kBlockBytes;
    if (row_bytes % 16 != 0 || (reinterpret_cast<uintptr_t>(w) & 15) != 0) return false;
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (encode == nullptr) return false;
    const cuuint64_t dims[2] = {row_bytes, static_cast<cuuint64_t>(N)};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kTmaBoxBytes), static_cast<cuuint32_t>(rows)};
    const cuuint32_t elem[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(w), dims, strides, box,
                  elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int kXRows, bool kTmaW>
cudaError_t launch_wt_kernel(const uint8_t* xa, const float* xf, const uint8_t* w, float* y,
                             float* partial, unsigned int* tile_count, int splits, int M, int N,
                             int K, int device, const CUtensorMap& map, cudaStream_t stream,
                             const WtRouted& rt = WtRouted{}) {
    using C = WtCfg<kXRows, kTmaW>;
    static bool attr_done[64] = {};
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    if (!attr_done[device]) {
        cudaError_t e = cudaFuncSetAttribute(gemm_wt_kernel<kXRows, kTmaW>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done[device] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((N + C::kRows - 1) / C::kRows, (M + kXRows - 1) / kXRows, splits);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (C::kSmall && splits > 1) {
        // the K parts of a tile: one cluster along z
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 1;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = static_cast<unsigned>(splits);
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, gemm_wt_kernel<kXRows, kTmaW>, xa, xf, w, y, partial,
                              tile_count, M, N, K, rt, map);
}

template <int kXRows>
cudaError_t launch_wt(const uint8_t* xa, const float* xf, const uint8_t* w, float* y,
                      float* partial, unsigned int* tile_count, int splits, int M, int N, int K,
                      int device, cudaStream_t stream, uint32_t flags = 0) {
    alignas(64) CUtensorMap map;
    WtRouted rt;
    rt.flags = flags;
    if (make_weight_map(&map, w, N, K, 128))
        return launch_wt_kernel<kXRows, true>(xa, xf, w, y, partial, tile_count, splits, M, N, K,
                                              device, map, stream, rt);
    memset(&map, 0, sizeof(map));
    return launch_wt_kernel<kXRows, false>(xa, xf, w, y, partial, tile_count, splits, M, N, K,
                                           device, map, stream, rt);
}

// K parts of the weights-as-A kernel: with fewer than 64 weight tiles (small m
// and n) the GPU would sit mostly idle, so each row's K blocks are split into
// up to 8 parts (about 128 CTAs), each part's accumulator written to its own
// slice of a partial buffer; the last part to finish on a tile sums them in
// part order, so the result does not depend on which part ends first.  Depends only on
// the geometry, so a workspace sized for it fits every device.
int wt_splits(int M, int N, int K) {
    if (M > 128) return 1;
    const long tiles = (N + 127) / 128;
    const int bpr = K / kQK;
    if (tiles >= 64 || bpr < 2) return 1;
    return static_cast<int>(std::max(1L, std::min<long>(128 / tiles, std::min(kMaxKParts, bpr))));
}

// x rows per CTA of the weights-as-A kernel: 256 (each decoded weight feeds
// twice the MMA work) once 128-row x tiles would need more than one wave of
// CTAs, else 128 (twice the CTAs).
int choose_wt_xrows(int M, int N, int sm_count) {
    const long ctas128 = static_cast<long>((N + 127) / 128) * ((M + 127) / 128);
    return ctas128 > sm_count ? 256 : 128;
}

// Tile width: the smallest estimated time with tiles spread over the SMs; a
// tile's time grows with BN (decode) plus a fixed share (x conversion, fill).
// Small m: x tile rows (16, 32 or 64; 0 = not small) and K parts.  All of a
// part's x stages (4 per block) must fit the kSmallXBytes region, so the parts
// may have to be more than wt_splits asks for; at most twice as many (and
// at most kMaxKParts), else the x-image path is used.  Geometry only.
int small_xrows(int M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 0; }

int small_splits(int M, int N, int K) {
    const int xr = small_xrows(M);
    if (xr == 0) return 0;
    const int bpr = K / kQK;
    const int max_blocks = kSmallXBytes / (xr * kKS * 2) / 4;
    const int base = wt_splits(M, N, K);
    for (int s = base; s <= kMaxKParts && s <= 2 * base && s <= bpr; ++s)
        if ((bpr + s - 1) / s <= max_blocks) return s;
    return 0;
}

int choose_bn(int M, int N, int sm_count) {
    const int cands[4] = {256, 192, 128, 64};
    int best = 128;
    long best_cost = -1;
    const long mt = (M + kBM - 1) / kBM;
    for (int bn : cands) {
        const long tiles = mt * ((N + bn - 1) / bn);
        const long waves = (tiles + sm_count - 1) / sm_count;
        const long cost = waves * (bn + 32);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = bn;
        }
    }
    return best;
}

}  // namespace

// x image (m rows padded to 256-row super-tiles) then, when K is split, the
// partial buffer (parts x m x n f32) at the next 256-byte boundary.
static size_t image_bytes(int M, int K) {
    const size_t m_pad = static_cast<size_t>((M + kXSuperRows - 1) / kXSuperRows) * kXSuperRows;
    return m_pad * static_cast<size_t>(K) * 2;
}

// With a split K: the parts' buffer, then one arrival counter per output tile.
static size_t parts_bytes(int M, int N, int splits) {
    return (static_cast<size_t>(splits) * M * N * 4 + 255) & ~size_t(255);
}

size_t gemm_tc_workspace_bytes(int M, int N, int K) {
    if (small_splits(M, N, K) > 0) return 0;  // x converted in the GEMM, parts summed on chip
    const int splits = wt_splits(M, N, K);
    if (splits == 1) return image_bytes(M, K);
    const size_t img = (image_bytes(M, K) + 255) & ~size_t(255);
    const size_t tiles = static_cast<size_t>((N + 127) / 128) * ((M + 127) / 128);
    return img + parts_bytes(M, N, splits) + tiles * 4;
}

bool gemm_tc_image_reusable(int M, int N, int K) {
    return small_splits(M, N, K) == 0 && wt_splits(M, N, K) == 1;
}

cudaError_t launch_gemm_tc(const float* x, const uint8_t* w, float* y, int M, int N, int K,
                           int device, int sm_count, void* workspace, cudaStream_t stream,
                           uint32_t flags) {
    if (const int parts = small_splits(M, N, K)) {
        switch (small_xrows(M)) {
            case 16: return launch_wt<16>(nullptr, x, w, y, nullptr, nullptr, parts, M, N, K, device, stream, flags);
            case 32: return launch_wt<32>(nullptr, x, w, y, nullptr, nullptr, parts, M, N, K, device, stream, flags);
            default: return launch_wt<64>(nullptr, x, w, y, nullptr, nullptr, parts, M, N, K, device, stream, flags);
        }
    }
    const int bn = choose_bn(M, N, sm_count);
    if (workspace == nullptr)
        return launch_width<false>(bn, x, nullptr, w, y, M, N, K, device, stream);
    uint8_t* xa = static_cast<uint8_t*>(workspace);
    const int splits = wt_splits(M, N, K);
    float* partial = nullptr;
    unsigned int* tile_count = nullptr;
    int n_tiles = 0;
    if (splits > 1) {
        uint8_t* p = xa + ((image_bytes(M, K) + 255) & ~size_t(255));
        partial = reinterpret_cast<float*>(p);
        tile_count = reinterpret_cast<unsigned int*>(p + parts_bytes(M, N, splits));
        n_tiles = ((N + 127) / 128) * ((M + 127) / 128);
    }
    // kImageReady (one K part only): the workspace already holds this x's
    // image from the call before, which is still in the stream
    const uint32_t wt_flags = splits == 1 ? (flags & kImageReady) : 0u;
    if (!wt_flags) {
        // only x's own rows: the image's padding rows are never read into a kept output
        const size_t n_chunks = static_cast<size_t>(M) * (K / 8);
        size_t blocks = (n_chunks + 255) / 256;
        const size_t cap = static_cast<size_t>(sm_count) * 4;
        if (blocks > cap) blocks = cap;
        x_to_bf16_tiles_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
            x, xa, M, K, n_chunks, tile_count, n_tiles);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (choose_wt_xrows(M, N, sm_count) == 256)
        return launch_wt<256>(xa, nullptr, w, y, partial, tile_count, splits, M, N, K, device,
                              stream, wt_flags);
    return launch_wt<128>(xa, nullptr, w, y, partial, tile_count, splits, M, N, K, device, stream,
                          wt_flags);
}

// ---- independent small-m products of one x in one persistent grid -----------
//
// Several products y_c = x W_c^T of the same x (m <= 64 rows) whose calls are
// independent of one another: one CTA per SM walks a sequence of 128-row
// weight tiles (tile t of all the calls' tiles: blockIdx.x, + gridDim.x, ...),
// each over all of K.  The decoders run on from one tile's blocks into the
// next; the two MMA issuers write tile j into accumulator pair j % 2, so the
// epilogue warps read tile j out of TMEM while tile j + 1 is multiplied.  No
// K split and no per-tile start-up: a call's tiles cost decode time only.

namespace {

#ifndef Q2K_TC_MULTI_STAGES
#define Q2K_TC_MULTI_STAGES 8
#endif
#ifndef Q2K_TC_MULTI_HANDOVER
#define Q2K_TC_MULTI_HANDOVER 4
#endif
#ifndef Q2K_TC_MULTI_RELEASE
#define Q2K_TC_MULTI_RELEASE 4
#endif
#ifndef Q2K_TC_MULTI_RAW
#define Q2K_TC_MULTI_RAW 4
#endif
#ifndef Q2K_TC_MULTI_XRES_KB
#define Q2K_TC_MULTI_XRES_KB 160
#endif
// calls per launch (the tensor maps travel in the kernel parameters)
constexpr int kMultiMaxCalls = 32;
// x stays resident for the whole grid when all its K stages fit this many
// bytes of shared memory; otherwise it cycles through a ring as deep as the
// decoded-weight ring
constexpr int kMultiXResident = Q2K_TC_MULTI_XRES_KB * 1024;

struct WtMultiCalls {
    CUtensorMap maps[kMultiMaxCalls];  // call c's weights, 128-row x 112-byte boxes
    float* y[kMultiMaxCalls];
    int n[kMultiMaxCalls];
    int tile0[kMultiMaxCalls + 1];     // call c's tiles: [tile0[c], tile0[c + 1])
    int count;
};

template <int kXRows>
struct MultiCfg {
    static constexpr int kRows = 128;
    static constexpr int kDecWarps = 16;   // as in the weights-as-A kernel
    static constexpr int kGroupWarps = 8;
    static constexpr int kDecThreads = 32 * kDecWarps;
    static constexpr int kMmaWarp = kDecWarps;
    static constexpr int kWaitWarp = kDecWarps + 1;
    static constexpr int kWWarp = kDecWarps + 2;
    static constexpr int kXWarp = kDecWarps + 3;
    static constexpr int kEpiWarp0 = kDecWarps + 4;  // four warps: lane quarters 0..3
    static constexpr int kThreads = 32 * (kDecWarps + 8);
    static_assert(kEpiWarp0 % 4 == 0, "epilogue warp w reads TMEM lane quarter w % 4");
    static constexpr int kPair = Q2K_TC_MULTI_HANDOVER;  // stages per hand-over (4: one block)
    static_assert(kPair == 2 || kPair == 4 || kPair == 8, "a whole number of hand-overs per tile");
    // stages released together (one commit from each issuer): a whole block
    // (4) measured faster than pairs (m = 16, 4096^2: 4.57 against 4.78 us
    // per call), since each commit costs an issuer about as much as an MMA
    static constexpr int kRelease = Q2K_TC_MULTI_RELEASE;
    static_assert((kRelease == 2 || kRelease == 4) && kPair % kRelease == 0, "release groups");
    static constexpr int kXStage = kXRows * kKS * 2;
    static constexpr uint32_t kColPair = 2 * kXRows;  // a tile's two accumulators
    static constexpr uint32_t kColA = 2 * kColPair;   // after both pairs
    static constexpr int kTmemCols = 512;
    // decoded-weight ring (and x ring): as deep as asked and TMEM holds, even
    // (stages are released in pairs)
    static constexpr int kStages =
        std::min(Q2K_TC_MULTI_STAGES, static_cast<int>((kTmemCols - kColA) / 32)) & ~1;
    static_assert(kStages >= 8, "two blocks of stages in flight");
    static_assert(kColA + 32u * kStages <= static_cast<uint32_t>(kTmemCols), "TMEM");
    static constexpr int kRaw = Q2K_TC_MULTI_RAW;
    static constexpr int kRawBytes = kRows * kTmaBoxBytes;
    // bars: x_full[kStages], a_full[kStages], a_empty[kStages], raw_full[kRaw],
    //       raw_empty[kRaw], acc_full[2], acc_empty[2], drain
    static constexpr int kNumBars = 3 * kStages + 2 * kRaw + 5;
    static_assert(kRawBytes % 1024 == 0 && kXStage % 1024 == 0, "TMA / swizzle alignment");
};

// x bytes of shared memory: all K stages, or the ring
template <int kXRows>
__host__ __device__ inline int multi_x_bytes(int K) {
    using C = MultiCfg<kXRows>;
    const int all = (K / kKS) * C::kXStage;
    return all <= kMultiXResident ? all : C::kStages * C::kXStage;
}
template <int kXRows>
__host__ __device__ inline int multi_smem_bytes(int K) {
    using C = MultiCfg<kXRows>;
    return multi_x_bytes<kXRows>(K) + C::kRaw * C::kRawBytes + 8 * C::kNumBars + 16 + 1024;
}

template <int kXRows>
constexpr int multi_smem_max() {
    using C = MultiCfg<kXRows>;
    return (kMultiXResident > C::kStages * C::kXStage ? kMultiXResident : C::kStages * C::kXStage) +
           C::kRaw * C::kRawBytes + 8 * C::kNumBars + 16 + 1024;
}
static_assert(multi_smem_max<16>() <= 232448 && multi_smem_max<64>() <= 232448, "shared memory");

__device__ __forceinline__ int multi_call_of(const WtMultiCalls& calls, int tile) {
    int c = 0;
    while (c + 1 < calls.count && tile >= calls.tile0[c + 1]) ++c;
    return c;
}

// MMA issuers of the persistent kernel.  The waiter (kWaiter) waits for a
// block's four stages (and, before a tile's first block, for its accumulator
// pair to be read out) and meets the MMA warp at named barrier 1; then the MMA
// warp issues the even stages into accumulator 0 of the pair, the waiter the
// odd ones into accumulator 1.  Both pass the barrier once per block of every
// tile, whatever happens, so neither can be left waiting there.  Each issuer
// is its own instantiation: the issue loop's stage arithmetic stays at
// compile time (a runtime issuer choice measured slower).
template <int kXRows, bool kWaiter>
__device__ __forceinline__ void multi_issue(int lane, uint32_t tmem_base, uint32_t sbase, int nx,
                                            int n_iters, int my_tiles, int all_iters, bool resident,
                                            uint32_t bar_xfull, uint32_t bar_afull,
                                            uint32_t bar_aempty, uint32_t bar_accfull,
                                            uint32_t bar_accempty, uint32_t bar_drain,
                                            volatile int* abort_flag, unsigned int* err) {
    using C = MultiCfg<kXRows>;
    const uint32_t idesc = make_idesc(kBM, nx);
    const uint64_t xdesc0 = sw128_desc(sbase);
    const uint32_t a_base0 = tmem_base + C::kColA;
    int G0 = 0;
    for (int j = 0; j < my_tiles; ++j) {
        const uint32_t acc = tmem_base + static_cast<uint32_t>(j & 1) * C::kColPair +
                             (kWaiter ? static_cast<uint32_t>(kXRows) : 0u);
        for (int i0 = 0; i0 < n_iters; i0 += C::kPair, G0 += C::kPair) {
            if (kWaiter && lane == 0 && !*abort_flag) {
                bool ok = true;
                if (resident && G0 == 0)
                    ok = mbar_wait_bounded(bar_xfull, 0, abort_flag, err, kErrTimeoutFull);
                if (ok && i0 == 0 && j >= 2)
                    ok = mbar_wait_bounded(bar_accempty + 8 * (j & 1), ((j >> 1) - 1) & 1,
                                           abort_flag, err, kErrTimeoutAccum);
#pragma unroll
                for (int u = 0; u < C::kPair; ++u) {
                    const int G = G0 + u;
                    const int s = G % C::kStages;
                    const uint32_t par = (G / C::kStages) & 1;
                    if (ok && !resident)
                        ok = mbar_wait_bounded(bar_xfull + 8 * s, par, abort_flag, err, kErrTimeoutFull);
                    if (ok)
                        ok = mbar_wait_bounded(bar_afull + 8 * s, par, abort_flag, err, kErrTimeoutFull);
                }
            }
            __syncwarp();
            asm volatile("bar.sync 1, 64;" ::: "memory");
            if (lane == 0 && !*abort_flag) {
                tc_fence_after();
#pragma unroll
                for (int u = kWaiter ? 1 : 0; u < C::kPair; u += 2) {
                    const int G = G0 + u;
                    const int i = i0 + u;
                    const int sx = resident ? i : G % C::kStages;
                    const uint64_t xdesc = xdesc0 + static_cast<uint64_t>(sx * (C::kXStage >> 4));
                    const uint32_t a_s = a_base0 + 32u * static_cast<uint32_t>(G % C::kStages);
#pragma unroll
                    for (int kk = 0; kk < kKS / 16; ++kk)
                        mma_bf16_tmem_a(acc, a_s + 8u * kk, xdesc + 2u * kk, idesc,
                                        (i > 1 || kk > 0) ? 1u : 0u);
                    // both issuers release a group of kRelease stages (each
                    // after its last stage of the group) once its MMAs are
                    // done, when a later stage reuses it
                    if (u % C::kRelease >= C::kRelease - 2 &&
                        (G & ~(C::kRelease - 1)) + C::kStages < all_iters)
                        mma_commit(bar_aempty + 8 * ((G | (C::kRelease - 1)) % C::kStages));
                }
                if (i0 + C::kPair == n_iters) mma_commit(bar_accfull + 8 * (j & 1));
            }
            __syncwarp();
        }
    }
    if (lane == 0 && *abort_flag) {
        // no MMA may still write TMEM when it is freed
        mma_commit(bar_drain);
        volatile int no_abort = 0;
        mbar_wait_bounded(bar_drain, 0, &no_abort, err, kErrTimeoutDrain);
    }
    __syncwarp();
}

template <int kXRows>
__global__ void __launch_bounds__(MultiCfg<kXRows>::kThreads, 1)
gemm_wt_multi_kernel(const uint8_t* __restrict__ xa, int M, int K, uint32_t flags,
                     const __grid_constant__ WtMultiCalls calls) {
    using C = MultiCfg<kXRows>;
    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nx = min(kXRows, (M + 15) & ~15);  // MMA N
    const int nb = K / kQK;                      // blocks per weight row
    const int n_iters = 4 * nb;                  // 64-K stages per tile
    const int total_tiles = calls.tile0[calls.count];
    const int my_tiles =
        static_cast<int>(blockIdx.x) < total_tiles
            ? (total_tiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
            : 0;
    const int all_iters = my_tiles * n_iters;  // this CTA's stages, all tiles
    const int x_bytes = multi_x_bytes<kXRows>(K);
    const bool resident = x_bytes == (K / kKS) * C::kXStage;
    const uint32_t off_raw = static_cast<uint32_t>(x_bytes);
    const uint32_t raw0 = sbase + off_raw;

    const uint32_t bar_xfull = raw0 + C::kRaw * C::kRawBytes;
    const uint32_t bar_afull = bar_xfull + 8 * C::kStages;
    const uint32_t bar_aempty = bar_afull + 8 * C::kStages;
    const uint32_t bar_raw = bar_aempty + 8 * C::kStages;
    const uint32_t bar_rawempty = bar_raw + 8 * C::kRaw;
    const uint32_t bar_accfull = bar_rawempty + 8 * C::kRaw;
    const uint32_t bar_accempty = bar_accfull + 16;
    const uint32_t bar_drain = bar_accempty + 16;
    uint8_t* misc = smem + off_raw + C::kRaw * C::kRawBytes + 8 * C::kNumBars;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
    unsigned int* err = &g_tc_error;

    if (warp == 0) {
        for (int s = lane; s < C::kStages; s += 32) {
            mbar_init(bar_xfull + 8 * s, 1);               // the producer's expect-tx arrival
            mbar_init(bar_afull + 8 * s, C::kGroupWarps);  // one arrival per warp of its group
            mbar_init(bar_aempty + 8 * s, 2);              // a stage pair: one commit per issuer
        }
        for (int r = lane; r < C::kRaw; r += 32) {
            mbar_init(bar_raw + 8 * r, 1);
            mbar_init(bar_rawempty + 8 * r, C::kDecWarps);
        }
        if (lane < 2) {
            mbar_init(bar_accfull + 8 * lane, 2);   // one commit per issuer
            mbar_init(bar_accempty + 8 * lane, 4);  // one arrival per epilogue warp
        }
        if (lane == 0) {
            mbar_init(bar_drain, 2);
            *abort_flag = 0;
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == C::kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(C::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

    if (warp < C::kDecWarps) {
        // ---------------- weight decoders: every block of every tile, in order ----------------
        const int quarter = warp & 3;
        const int seg = (warp >> 2) & 1;
        const int half = warp >> 3;
        const int row = 32 * quarter + lane;
        const uint32_t a_col0 =
            tmem_base + (static_cast<uint32_t>(32 * quarter) << 16) + C::kColA + 8u * seg;
        const int all_blocks = my_tiles * nb;
        for (int B = 0, b = 0; B < all_blocks; ++B, b = b + 1 == nb ? 0 : b + 1) {
            // B: block counted over all tiles; b: the same block within its row
            const int buf = B % C::kRaw;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(bar_raw + 8 * buf, (B / C::kRaw) & 1,
                                                           abort_flag, err, kErrTimeoutFull)))
                break;
            const uint32_t mine = raw0 + buf * C::kRawBytes + row * kTmaBoxBytes + 4 * (b & 3);
            uint32_t sh[2], qh[4];
#pragma unroll
            for (int q = 0; q < 2; ++q) sh[q] = ld_shared_u32(mine + 8 * half + 4 * q) >> (8 * seg);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                qh[e] = ld_shared_u32(mine + 16 + 32 * half + 16 * seg + 4 * e);
            const uint32_t dd = ld_shared_u32(mine + 80);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_rawempty + 8 * buf);
            const float d = f16_bits_to_float(dd);
            const float dmin = f16_bits_to_float(dd >> 16);
            bool ok = true;
#pragma unroll
            for (int cp = 0; cp < 2; ++cp) {
                const int G = 4 * B + 2 * half + cp;  // stage, counted over all tiles
                const int s = G % C::kStages;
                uint32_t o0[8], o1[8];
                if (cp == 0) wt_decode_half_stage<0>(qh, sh, d, dmin, o0, o1);
                else wt_decode_half_stage<1>(qh, sh, d, dmin, o0, o1);
                // the slot's last pair (stages G - 8, G - 7) released by both issuers
                if (G >= C::kStages &&
                    !__all_sync(0xFFFFFFFFu,
                                mbar_wait_bounded(bar_aempty + 8 * ((G | (C::kRelease - 1)) % C::kStages),
                                                  ((G / C::kStages) - 1) & 1, abort_flag, err,
                                                  kErrTimeoutEmpty))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_col = a_col0 + 32u * s;
                tmem_st8(a_col, o0);
                tmem_st8(a_col + 16u, o1);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_afull + 8 * s);
            }
            if (!ok) break;
        }
    } else if (warp == C::kMmaWarp) {
        multi_issue<kXRows, false>(lane, tmem_base, sbase, nx, n_iters, my_tiles, all_iters, resident,
                                   bar_xfull, bar_afull, bar_aempty, bar_accfull, bar_accempty,
                                   bar_drain, abort_flag, err);
    } else if (warp == C::kWaitWarp) {
        multi_issue<kXRows, true>(lane, tmem_base, sbase, nx, n_iters, my_tiles, all_iters, resident,
                                  bar_xfull, bar_afull, bar_aempty, bar_accfull, bar_accempty,
                                  bar_drain, abort_flag, err);
    } else if (warp == C::kWWarp) {
        // ---------------- raw weight blocks: one TMA box each ----------------
        if (lane == 0) {
            for (int c = 0; c < calls.count; ++c)
                asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&calls.maps[c]))
                             : "memory");
            // the calls are independent: no grid that may still run writes W
            int B = 0;
            bool ok = true;
            for (int j = 0; j < my_tiles && ok; ++j) {
                const int tile = static_cast<int>(blockIdx.x) + j * static_cast<int>(gridDim.x);
                const int c = multi_call_of(calls, tile);
                const int n0 = (tile - calls.tile0[c]) * C::kRows;
                for (int b = 0; b < nb; ++b, ++B) {
                    const int buf = B % C::kRaw;
                    if (B >= C::kRaw &&
                        !mbar_wait_bounded(bar_rawempty + 8 * buf, ((B / C::kRaw) - 1) & 1,
                                           abort_flag, err, kErrTimeoutEmpty)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar_raw + 8 * buf, C::kRawBytes);
                    // rows past the call's N read as zeros (they decode to 0)
                    tma_load_2d(raw0 + buf * C::kRawBytes, &calls.maps[c], (kBlockBytes * b) & ~15,
                                n0, bar_raw + 8 * buf);
                }
            }
            if (*abort_flag) {
                // a copy may still be in flight: give it a bounded 50 us to land
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 50000ull) __nanosleep(1000);
            }
        }
        __syncwarp();
    } else if (warp == C::kXWarp) {
        // ---------------- x stages from the image ----------------
        if (lane == 0) {
            // the image is written by the grid before this one, unless an
            // earlier grid of the same x already waited for it (kImageReady);
            // later grids may start once every CTA is past this point
            if (!(flags & kImageReady)) pdl_wait_prerequisites();
            pdl_allow_dependents();
            const uint32_t bytes = static_cast<uint32_t>(nx) * (kKS * 2);
            if (resident) {
                if (my_tiles > 0) {
                    mbar_arrive_expect_tx(bar_xfull, bytes * static_cast<uint32_t>(n_iters));
                    for (int i = 0; i < n_iters; ++i)
                        bulk_copy_g2s(sbase + i * C::kXStage, xa + static_cast<size_t>(i) * kXSuperBytes,
                                      bytes, bar_xfull);
                }
            } else {
                for (int G = 0, i = 0; G < all_iters; ++G, i = i + 1 == n_iters ? 0 : i + 1) {
                    const int s = G % C::kStages;
                    if (G >= C::kStages &&
                        !mbar_wait_bounded(bar_aempty + 8 * ((G | (C::kRelease - 1)) % C::kStages),
                                           ((G / C::kStages) - 1) & 1, abort_flag, err,
                                           kErrTimeoutEmpty))
                        break;
                    mbar_arrive_expect_tx(bar_xfull + 8 * s, bytes);
                    bulk_copy_g2s(sbase + s * C::kXStage,
                                  xa + static_cast<size_t>(i) * kXSuperBytes, bytes,
                                  bar_xfull + 8 * s);
                }
            }
            if (*abort_flag) {
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 50000ull) __nanosleep(1000);
            }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: accumulator pair -> y, tile by tile ----------------
        const int quarter = warp & 3;
        const int row = 32 * quarter + lane;
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(32 * quarter) << 16);
        for (int j = 0; j < my_tiles; ++j) {
            if (!__all_sync(0xFFFFFFFFu, mbar_wait_backoff(bar_accfull + 8 * (j & 1), (j >> 1) & 1,
                                                           abort_flag, err, kErrTimeoutAccum, 512)))
                break;
            tc_fence_after();
            const int tile = static_cast<int>(blockIdx.x) + j * static_cast<int>(gridDim.x);
            const int c = multi_call_of(calls, tile);
            const int N = calls.n[c];
            const int n = (tile - calls.tile0[c]) * C::kRows + row;
            float* yc = calls.y[c];
            const uint32_t t_row = t_lane + static_cast<uint32_t>(j & 1) * C::kColPair;
#pragma unroll 1
            for (int c0 = 0; c0 < nx; c0 += 16) {
                uint32_t v[16], u[16];
                tmem_ld16(t_row + c0, v);
                tmem_ld16(t_row + static_cast<uint32_t>(kXRows) + c0, u);
                if (n < N) {
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int m = c0 + q;
                        // the two accumulators added in order (even stages + odd stages)
                        if (m < M)
                            yc[static_cast<size_t>(m) * N + n] =
                                __uint_as_float(v[q]) + __uint_as_float(u[q]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_accempty + 8 * (j & 1));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == C::kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(C::kTmemCols)
                     : "memory");
    }
    // the calls complete only after the grid before them (stream order)
    if (threadIdx.x == 0 && blockIdx.x == 0) pdl_wait_prerequisites();
}

template <int kXRows>
cudaError_t launch_multi_chunk(const uint8_t* xa, int M, int K, uint32_t flags,
                               const WtMultiCalls& calls, int sm_count, int device,
                               cudaStream_t stream) {
    using C = MultiCfg<kXRows>;
    static bool attr_done[64] = {};
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    const int smem = multi_smem_bytes<kXRows>(K);
    if (!attr_done[device]) {
        cudaError_t e = cudaFuncSetAttribute(gemm_wt_multi_kernel<kXRows>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             multi_smem_max<kXRows>());
        if (e != cudaSuccess) return e;
        attr_done[device] = true;
    }
    const int tiles = calls.tile0[calls.count];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(std::min(tiles, sm_count)));
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_wt_multi_kernel<kXRows>, xa, M, K, flags, calls);
}

}  // namespace

bool gemm_tc_multi_eligible(int M, int K, const void* w) {
    return M > 0 && small_xrows(M) > 0 && K > 0 && K % (4 * kQK) == 0 &&
           (reinterpret_cast<uintptr_t>(w) & 15) == 0;
}

bool gemm_tc_multi_available() { return tensor_map_encoder() != nullptr; }

size_t gemm_tc_multi_scratch_bytes(int M, int K) { return image_bytes(M, K); }

cudaError_t launch_gemm_tc_multi(const float* x, int M, int K, const MultiCall* mc, int count,
                                 void* scratch, int device, int sm_count, cudaStream_t stream) {
    if (count <= 0) return cudaSuccess;
    uint8_t* xa = static_cast<uint8_t*>(scratch);
    {
        const size_t n_chunks = static_cast<size_t>(M) * (K / 8);
        size_t blocks = (n_chunks + 255) / 256;
        const size_t cap = static_cast<size_t>(sm_count) * 4;
        if (blocks > cap) blocks = cap;
        x_to_bf16_tiles_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
            x, xa, M, K, n_chunks, nullptr, 0);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // chunks of at most kMultiMaxCalls calls, as even as possible
    const int n_launch = (count + kMultiMaxCalls - 1) / kMultiMaxCalls;
    int first = 0;
    for (int l = 0; l < n_launch; ++l) {
        const int cnt = (count - first) / (n_launch - l);
        WtMultiCalls calls;
        memset(&calls, 0, sizeof calls);
        calls.count = cnt;
        int tiles = 0;
        for (int c = 0; c < cnt; ++c) {
            const MultiCall& q = mc[first + c];
            if (!make_weight_map(&calls.maps[c], q.w, q.n, K, 128)) return cudaErrorNotSupported;
            calls.y[c] = q.y;
            calls.n[c] = q.n;
            calls.tile0[c] = tiles;
            tiles += (q.n + 127) / 128;
        }
        calls.tile0[cnt] = tiles;
        const uint32_t flags = l > 0 ? kImageReady : 0u;
        cudaError_t e;
        switch (small_xrows(M)) {
            case 16: e = launch_multi_chunk<16>(xa, M, K, flags, calls, sm_count, device, stream); break;
            case 32: e = launch_multi_chunk<32>(xa, M, K, flags, calls, sm_count, device, stream); break;
            default: e = launch_multi_chunk<64>(xa, M, K, flags, calls, sm_count, device, stream); break;
        }
        if (e != cudaSuccess) return e;
        first += cnt;
    }
    return cudaSuccess;
}

// ---- routed products on tensor cores (mul_mat_id with many routes) -----------
//
// Route r (token r / top_k, or slot r) multiplies its x row by expert ids[r]'s
// weights.  The routes are grouped by expert into 128-row x tiles: expert e's
// routes fill ceil(count_e / 128) tiles, its last one padded; the weights-as-A
// kernel then runs one CTA per (weight tile, x tile) with the x tile's expert's
// weights and writes each row to its route.  A route's result does not depend
// on where in its tile it lands (each MMA column is a separate dot product),
// so the order the routes are placed in does not matter.

// Tiles a routed product can need: sum_e ceil(c_e / 128) <= routes / 128 + the
// number of experts that have a route.
int routed_tiles_max(int routes, int n_experts) {
    return (routes + 127) / 128 + std::min(routes, n_experts);
}

// One CTA: count the routes per expert, scan to tile starts, and write each
// x tile's {expert, rows} (-1: unused), the route of each of a tile's first
// `rows` x rows, each route's x row (-1: id out of range) and, for a route
// whose id is out of range, a zero row of y (and of y2, when not null) and a
// count (one per output).
__global__ void __launch_bounds__(1024)
route_tiles_kernel(const uint32_t* __restrict__ ids, int routes, int n_experts, int tiles_max,
                   int2* __restrict__ tile_info, int* __restrict__ row_route,
                   int* __restrict__ route_row, float* __restrict__ y, float* __restrict__ y2, int N,
                   unsigned int* __restrict__ bad_ids) {
    extern __shared__ int route_smem[];
    int* cnt = route_smem;              // per expert: routes, then the placement cursor
    int* start = route_smem + n_experts;  // per expert: first tile
    __shared__ int warp_sum[32];
    __shared__ int total_tiles;
    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    for (int e = tid; e < n_experts; e += nt) cnt[e] = 0;
    __syncthreads();
    for (int r = tid; r < routes; r += nt) {
        const uint32_t e = ids[r];
        if (e < static_cast<uint32_t>(n_experts)) {
            atomicAdd(&cnt[e], 1);
        } else {
            if (bad_ids != nullptr) atomicAdd(bad_ids, y2 != nullptr ? 2u : 1u);
            float* row = y + static_cast<size_t>(r) * N;
            for (int n = 0; n < N; ++n) row[n] = 0.0f;
            if (y2 != nullptr) {
                row = y2 + static_cast<size_t>(r) * N;
                for (int n = 0; n < N; ++n) row[n] = 0.0f;
            }
        }
    }
    __syncthreads();
    // exclusive scan of the tile counts: each thread a run of experts
    const int per = (n_experts + nt - 1) / nt;
    const int e0 = min(n_experts, tid * per), e1 = min(n_experts, e0 + per);
    int mine = 0;
    for (int e = e0; e < e1; ++e) mine += (cnt[e] + 127) >> 7;
    const int lane = tid & 31, warp = tid >> 5;
    int incl = mine;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += v;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int nw = nt >> 5;
        int v = lane < nw ? warp_sum[lane] : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int u = __shfl_up_sync(0xFFFFFFFFu, v, d);
            if (lane >= d) v += u;
        }
        if (lane < nw) warp_sum[lane] = v;  // inclusive over warps
        if (lane == nw - 1) total_tiles = v;
    }
    __syncthreads();
    int t = incl - mine + (warp > 0 ? warp_sum[warp - 1] : 0);
    for (int e = e0; e < e1; ++e) {
        start[e] = t;
        const int c = cnt[e];
        for (int j = 0; j < (c + 127) >> 7; ++j)
            tile_info[t + j] = make_int2(e, min(128, c - 128 * j));
        // (the last tile's padding rows get no route: the GEMM reads only a
        // tile's first tile_info.y rows of row_route)
        t += (c + 127) >> 7;
    }
    for (int u = total_tiles + tid; u < tiles_max; u += nt) tile_info[u] = make_int2(-1, 0);
    __syncthreads();
    for (int e = tid; e < n_experts; e += nt) cnt[e] = 0;
    __syncthreads();
    for (int r = tid; r < routes; r += nt) {
        const uint32_t e = ids[r];
        int v = -1;
        if (e < static_cast<uint32_t>(n_experts)) {
            v = 128 * start[e] + atomicAdd(&cnt[e], 1);
            row_route[v] = r;
        }
        route_row[r] = v;
    }
}

// x rows by route into the bf16 tile image of the routed rows (x tile t =
// rows 128 t .. 128 t + 127): route r's row route_row[r] gets x row r / x_div.
// Only the routes' rows are written: a tile's padding rows feed only
// accumulator columns that the GEMM's epilogue drops (each MMA column is its
// own dot product), and tiles no expert uses are never read.  One thread
// converts one 8-element chunk; consecutive threads take consecutive chunks
// of a route's row.  As x_to_bf16_tiles_kernel it lets the GEMM after it
// start early.
__global__ void __launch_bounds__(256)
gather_x_tiles_kernel(const float* __restrict__ x, uint8_t* __restrict__ xa,
                      const int* __restrict__ route_row, int x_div, int K, size_t n_chunks) {
    pdl_allow_dependents();
    const int chunks_per_row = K >> 3;
    const int stages = K / kKS;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    // four chunks per pass, all their loads issued before any conversion (a
    // pass costs one memory round trip instead of four)
    constexpr int kPer = 4;
    for (size_t base = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; base < n_chunks;
         base += kPer * stride) {
        float4 a[kPer], b[kPer];
        int v[kPer], j[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const size_t id = base + u * stride;
            v[u] = -1;
            j[u] = 0;
            a[u] = b[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (id < n_chunks) {
                const int r = static_cast<int>(id / chunks_per_row);
                j[u] = static_cast<int>(id - static_cast<size_t>(r) * chunks_per_row);
                v[u] = route_row[r];  // -1: an id out of range, no row
                if (v[u] >= 0) {
                    const float4* src = reinterpret_cast<const float4*>(
                        x + static_cast<size_t>(r / x_div) * K + 8 * j[u]);
                    a[u] = __ldg(src);
                    b[u] = __ldg(src + 1);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            if (v[u] < 0) continue;
            const uint4 packed = make_uint4(pack_bf16x2(a[u].x, a[u].y), pack_bf16x2(a[u].z, a[u].w),
                                            pack_bf16x2(b[u].x, b[u].y), pack_bf16x2(b[u].z, b[u].w));
            const size_t tile = static_cast<size_t>(v[u] / kXSuperRows) * stages + (j[u] >> 3);
            *reinterpret_cast<uint4*>(xa + tile * kXSuperBytes +
                                      sw128_offset(v[u] % kXSuperRows, j[u] & 7)) = packed;
        }
    }
}

// Workspace of a routed product: tile table, row routes, route rows, then the
// x image.
static size_t routed_info_bytes(int tiles) { return (static_cast<size_t>(tiles) * 8 + 255) & ~size_t(255); }
static size_t routed_rows_bytes(int tiles) { return static_cast<size_t>(tiles) * 128 * 4; }
static size_t routed_route_bytes(int routes) { return (static_cast<size_t>(routes) * 4 + 255) & ~size_t(255); }

size_t gemm_tc_routed_workspace_bytes(int routes, int n_experts, int K) {
    const int tiles = routed_tiles_max(routes, n_experts);
    return routed_info_bytes(tiles) + routed_rows_bytes(tiles) + routed_route_bytes(routes) +
           image_bytes(tiles * 128, K);
}

cudaError_t launch_gemm_tc_routed(const float* x, const uint8_t* w, long long expert_stride,
                                  const uint32_t* ids, float* y, int routes, int x_div,
                                  int n_experts, int N, int K, unsigned int* bad_ids, int device,
                                  int sm_count, void* workspace, cudaStream_t stream,
                                  const uint8_t* w2, float* y2) {
    if (n_experts > kRoutedMaxExperts) return cudaErrorInvalidValue;
    const int tiles = routed_tiles_max(routes, n_experts);
    const int M = tiles * 128;
    uint8_t* base = static_cast<uint8_t*>(workspace);
    int2* tile_info = reinterpret_cast<int2*>(base);
    int* row_route = reinterpret_cast<int*>(base + routed_info_bytes(tiles));
    int* route_row = reinterpret_cast<int*>(base + routed_info_bytes(tiles) + routed_rows_bytes(tiles));
    uint8_t* xa = base + routed_info_bytes(tiles) + routed_rows_bytes(tiles) + routed_route_bytes(routes);
    route_tiles_kernel<<<1, 1024, 2 * n_experts * sizeof(int), stream>>>(
        ids, routes, n_experts, tiles, tile_info, row_route, route_row, y, y2, N, bad_ids);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t n_chunks = static_cast<size_t>(routes) * (K / 8);
    size_t blocks = (n_chunks + 255) / 256;
    const size_t cap = static_cast<size_t>(sm_count) * 4;  // one wave (four blocks fit an SM)
    if (blocks > cap) blocks = cap;
    gather_x_tiles_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        x, xa, route_row, x_div, K, n_chunks);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    WtRouted rt;
    rt.tile_info = tile_info;
    rt.row_route = row_route;
    rt.expert_stride = expert_stride;
    // one GEMM per weight pool over the same tiles and x image
    for (int o = 0; o < (w2 != nullptr ? 2 : 1); ++o) {
        const uint8_t* wo = o == 0 ? w : w2;
        float* yo = o == 0 ? y : y2;
        alignas(64) CUtensorMap map;
        const long long row_bytes = static_cast<long long>(K / kQK) * kBlockBytes;
        bool tma = false;
        if (expert_stride % row_bytes == 0) {
            const long long per = expert_stride / row_bytes;
            const long long pool_rows = static_cast<long long>(n_experts - 1) * per + N;
            rt.expert_rows = static_cast<int>(per);
            tma = pool_rows <= INT_MAX && make_weight_map(&map, wo, static_cast<int>(pool_rows), K, 128);
        }
        if (tma) {
            e = launch_wt_kernel<128, true>(xa, nullptr, wo, yo, nullptr, nullptr, 1, M, N, K,
                                            device, map, stream, rt);
        } else {
            memset(&map, 0, sizeof(map));
            e = launch_wt_kernel<128, false>(xa, nullptr, wo, yo, nullptr, nullptr, 1, M, N, K,
                                             device, map, stream, rt);
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_gemm_tc_static(const float* x, const uint8_t* w, float* y, int M, int N, int K,
                                  int device, int sm_count, cudaStream_t stream) {
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    if (gemm_tc_workspace_bytes(M, N, K) > kStaticWorkspaceBytes) return cudaErrorInvalidValue;
    // In host code the array's name is only a stand-in: its device address is
    // looked up per device, with that device current (the caller's), and kept
    // once a lookup has succeeded; a failed lookup is retried by the next call.
    static std::mutex mu;
    static void* addr[64] = {};
    void* image = nullptr;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (addr[device] == nullptr) {
            void* p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, g_static_x_image);
            if (e != cudaSuccess) return e;
            if (p == nullptr) return cudaErrorInvalidSymbol;
            addr[device] = p;
        }
        image = addr[device];
    }
    return launch_gemm_tc(x, w, y, M, N, K, device, sm_count, image, stream);
}

cudaError_t launch_gemm_tc_plain(const float* x, const uint8_t* w, float* y, int M, int N, int K,
                                 int device, int sm_count, cudaStream_t stream, uint32_t flags) {
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    const size_t need = gemm_tc_workspace_bytes(M, N, K);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cs);
    if (e != cudaSuccess) return e;
    // No image needed (small m), too large, or inside a capture (where a wait
    // on another stream's event is not allowed): the GEMM converts x itself.
    if (need == 0 || need > kPlainScratchBytes || cs != cudaStreamCaptureStatusNone)
        return launch_gemm_tc(x, w, y, M, N, K, device, sm_count, nullptr, stream, flags);
    static std::mutex mu;
    static void* addr[64] = {};
    static cudaEvent_t done[64] = {};
    std::lock_guard<std::mutex> lk(mu);
    if (addr[device] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_plain_x_image);
        if (e != cudaSuccess) return e;
        if (p == nullptr) return cudaErrorInvalidSymbol;
        if (done[device] == nullptr) {
            e = cudaEventCreateWithFlags(&done[device], cudaEventDisableTiming);
            if (e != cudaSuccess) return e;
        }
        addr[device] = p;
    }
    // the previous call through this scratch (any stream) finishes first
    e = cudaStreamWaitEvent(stream, done[device], 0);
    if (e == cudaSuccess) e = launch_gemm_tc(x, w, y, M, N, K, device, sm_count, addr[device], stream, flags);
    if (e == cudaSuccess) e = cudaEventRecord(done[device], stream);
    return e;
}

cudaError_t read_and_clear_tc_error(uint32_t* out, cudaStream_t stream) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_tc_error, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbolAsync(g_tc_error, &zero, sizeof(unsigned int), 0,
                                cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(stream);
}

}  // namespace q2k
