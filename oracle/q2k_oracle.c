/*
 * CPU oracle for the GGML Q2_K dequantize, embedding gather and weight-quantized
 * matmul, as fixed by the mlx-native test page "tests/deepseek_q2_k.rs".
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or load
 * this file: only the tests, the smoke check of the entry module and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * It is deliberately plain and slow:
 *   - its own IEEE-754 binary16 decoder;
 *   - the page's canonical decode loop (fn reference_dequant: half 0..1,
 *     shift 0,2,4,6, segment 0..1, 16 lanes), in f32 exactly as the page
 *     writes it: dl = d*sc, ml = dmin*m, value = dl*q - ml, each operation
 *     rounded on its own (build with -ffp-contract=off so no FMA is formed);
 *   - the matmul as the definition y[m,n] = sum_k x[m,k]*w[n,k], every weight
 *     row fully decoded to f32 first, then a sequential f64 sum (the page's
 *     cpu_dot sums in f32; f64 is used here so the reference carries less
 *     rounding than either GPU path).  It also returns sum_k |x*w| in f64,
 *     the scale of the relative tolerances.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared -pthread.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_QK_K 256        /* weights per super-block (page const QK_K) */
#define ORACLE_BLOCK_BYTES 84  /* bytes per super-block (page const BLOCK_BYTES) */

/* IEEE-754 binary16 -> binary32, written from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.  Every binary16
 * value is exactly representable in binary32, so this is exact. */
float q2ko_f16_to_f32(uint16_t h)
{
    unsigned sign = (h >> 15) & 1u;
    unsigned expo = (h >> 10) & 31u;
    unsigned frac = h & 1023u;
    if (expo == 31u) {
        /* infinity or NaN: all-ones exponent; keep the fraction as payload */
        uint32_t bits = (sign << 31) | 0x7F800000u | ((uint32_t)frac << 13);
        float f;
        memcpy(&f, &bits, sizeof f);
        return f;
    }
    double mag;
    if (expo == 0u)
        mag = ldexp((double)frac, -24);                    /* zero or subnormal */
    else
        mag = ldexp(1024.0 + (double)frac, (int)expo - 25); /* (1 + f/1024) 2^(e-15) */
    return (float)(sign ? -mag : mag);
}

static uint16_t load_le16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* One 84-byte block -> 256 f32 values in the page's push order
 * (fn reference_dequant).  scales = bytes 0..15, qs = bytes 16..79,
 * d = f16 at 80..81, dmin = f16 at 82..83. */
void q2ko_dequant_block(const uint8_t *block, float *out)
{
    const uint8_t *scales = block;
    const uint8_t *qs = block + 16;
    const float d = q2ko_f16_to_f32(load_le16(block + 80));
    const float dmin = q2ko_f16_to_f32(load_le16(block + 82));
    int scale_index = 0;
    int pushed = 0;
    for (int half = 0; half < 2; ++half) {
        for (int shift = 0; shift <= 6; shift += 2) {
            for (int segment = 0; segment < 2; ++segment) {
                const uint8_t sc = scales[scale_index++];
                const float dl = d * (float)(sc & 0x0F);
                const float ml = dmin * (float)(sc >> 4);
                const int q_offset = half * 32 + segment * 16;
                for (int lane = 0; lane < 16; ++lane) {
                    const int q = (qs[q_offset + lane] >> shift) & 0x03;
                    const float prod = dl * (float)q;
                    out[pushed++] = prod - ml;
                }
            }
        }
    }
}

/* Host decode of a byte buffer of whole blocks (page test
 * q2_k_host_decode_rejects_malformed_buffers): the byte count must be a
 * multiple of 84 and the output must hold exactly 256 floats per block.
 * Returns 0 on success, 1 on a malformed buffer. */
int q2ko_dequantize(const uint8_t *bytes, size_t n_bytes, float *out, size_t n_out)
{
    if (n_bytes % ORACLE_BLOCK_BYTES != 0)
        return 1;
    size_t n_blocks = n_bytes / ORACLE_BLOCK_BYTES;
    if (n_out != n_blocks * ORACLE_QK_K)
        return 1;
    for (size_t b = 0; b < n_blocks; ++b)
        q2ko_dequant_block(bytes + b * ORACLE_BLOCK_BYTES, out + b * ORACLE_QK_K);
    return 0;
}

/* Embedding gather (page test q2_k_embedding_gather_matches_canonical_rows_and_
 * rejects_bad_ids): output row t is the decoded table row ids[t]; the table is
 * vocab rows of embed_dim/256 consecutive blocks.  Any id >= vocab is an
 * error (returns 2, output untouched); embed_dim not a multiple of 256
 * returns 1. */
int q2ko_gather(const uint8_t *table, uint32_t vocab, uint32_t embed_dim,
                const uint32_t *ids, uint32_t n_tokens, float *out)
{
    if (embed_dim % ORACLE_QK_K != 0)
        return 1;
    for (uint32_t t = 0; t < n_tokens; ++t)
        if (ids[t] >= vocab)
            return 2;
    const size_t blocks_per_row = embed_dim / ORACLE_QK_K;
    for (uint32_t t = 0; t < n_tokens; ++t) {
        const uint8_t *row = table + (size_t)ids[t] * blocks_per_row * ORACLE_BLOCK_BYTES;
        for (size_t b = 0; b < blocks_per_row; ++b)
            q2ko_dequant_block(row + b * ORACLE_BLOCK_BYTES,
                               out + (size_t)t * embed_dim + b * ORACLE_QK_K);
    }
    return 0;
}

/* ---- matmul: y[m,n] = sum_k x[m,k] * w[n,k] ---------------------------- */

typedef struct {
    const float *x;
    const uint8_t *w;
    double *y;
    double *s_abs;
    size_t M, N, K;
    size_t n_begin, n_end;
    float *row;  /* K floats of scratch */
} matmul_job;

static void matmul_rows(matmul_job *job)
{
    const size_t blocks_per_row = job->K / ORACLE_QK_K;
    for (size_t n = job->n_begin; n < job->n_end; ++n) {
        const uint8_t *wrow = job->w + n * blocks_per_row * ORACLE_BLOCK_BYTES;
        for (size_t b = 0; b < blocks_per_row; ++b)
            q2ko_dequant_block(wrow + b * ORACLE_BLOCK_BYTES, job->row + b * ORACLE_QK_K);
        for (size_t m = 0; m < job->M; ++m) {
            const float *xrow = job->x + m * job->K;
            double acc = 0.0, acc_abs = 0.0;
            for (size_t k = 0; k < job->K; ++k) {
                const double term = (double)xrow[k] * (double)job->row[k];
                acc += term;
                acc_abs += fabs(term);
            }
            job->y[m * job->N + n] = acc;
            if (job->s_abs)
                job->s_abs[m * job->N + n] = acc_abs;
        }
    }
}

static void *matmul_thread(void *arg)
{
    matmul_rows((matmul_job *)arg);
    return NULL;
}

/* x: f32 [M, K] row-major; w: N rows of K/256 blocks; y, s_abs: f64 [M, N].
 * scratch: n_threads * K floats.  Rows of W are split into n_threads
 * contiguous ranges, one POSIX thread each.  Returns 0, or 1 when K is not a
 * multiple of 256 or a thread could not be started. */
int q2ko_matmul(const float *x, const uint8_t *w, double *y, double *s_abs,
                size_t M, size_t N, size_t K, int n_threads, float *scratch)
{
    if (K % ORACLE_QK_K != 0 || n_threads < 1)
        return 1;
    if ((size_t)n_threads > N)
        n_threads = (int)(N ? N : 1);
    matmul_job jobs[256];
    pthread_t threads[256];
    if (n_threads > 256)
        n_threads = 256;
    for (int t = 0; t < n_threads; ++t) {
        jobs[t].x = x;
        jobs[t].w = w;
        jobs[t].y = y;
        jobs[t].s_abs = s_abs;
        jobs[t].M = M;
        jobs[t].N = N;
        jobs[t].K = K;
        jobs[t].n_begin = N * (size_t)t / (size_t)n_threads;
        jobs[t].n_end = N * (size_t)(t + 1) / (size_t)n_threads;
        jobs[t].row = scratch + (size_t)t * K;
    }
    if (n_threads == 1) {
        matmul_rows(&jobs[0]);
        return 0;
    }
    int started = 0, failed = 0;
    for (int t = 0; t < n_threads; ++t) {
        if (pthread_create(&threads[t], NULL, matmul_thread, &jobs[t]) != 0) {
            failed = 1;
            break;
        }
        ++started;
    }
    for (int t = 0; t < started; ++t)
        pthread_join(threads[t], NULL);
    return failed;
}
