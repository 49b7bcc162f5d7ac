/*
 * qmm_oracle.c -- plain, slow, obviously-correct CPU oracle for the
 * block-quantized int4 x int8 matrix product (Q4_0 weights x Q8_0
 * activations, fp32/fp64 combine).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file; only the test suite, the smoke check and the bench's
 * CPU-baseline / reference leg load it.  It shares no code, header, table or
 * constant generator with the CUDA path.
 *
 * What each function follows:
 *  - Q4_0 block format: "Guia de desarrollo de modelos de IA a pequena escala
 *    (como TinyLLaMA) con C++" (kenji.blog), section 6.1 "Arquitectura de
 *    cuantizacion por bloques": 32 values per block, one FP16 scale (2 bytes)
 *    plus 32 four-bit values (16 bytes).
 *  - Block quantization and the quantized dot: "Panduan Menggunakan llama.cpp
 *    dan Pengenalan Kustomisasi dengan C++" (kenji.blog/id), section 2.2
 *    "Dasar Matematis Kuantisasi": w_i ~ Delta*q_i with q_i in [-8,7],
 *    Delta = max|w_i| / 7, and y = sum w_i x_i ~ Delta*Delta_x*sum q_i q_x,i,
 *    the inner sum being pure integer arithmetic.
 *  - Q8_0-style int8 activations and integer kernels: Colibri page
 *    (kerneldigest.dev), "Arquitectura del Sistema".  The activation
 *    quantizer is d = max|x|/127 stored as fp16, q = round-half-away(x/d).
 *  - Plain matrix product C_ij = sum_k A_ik B_kj: "No necesitas Python!
 *    Construi un motor de inferencia de IA solo con C++" (kenji.blog),
 *    section 6, GEMM equation.
 *  - SwiGLU(x) = Swish(x W_gate) (x) (x W_up), Swish(z) = z*sigmoid(z):
 *    TinyLLaMA guide, section 4.4.
 *  - RMSNorm(x) = x / sqrt(mean(x^2) + eps) (.) gamma: TinyLLaMA guide,
 *    section 4.1 (eps is not given there; callers pass it).
 *  - Per-row-scale int4 / int2 containers: Colibri page, "Arquitectura del
 *    Sistema" (int4 container with per-row scales; int4/int2 packing); the
 *    scale rule is the llama.cpp guide's 2.2 rule applied per row, and the
 *    bit layout is this oracle's reading (the page gives none).
 *  - Q4_0 weights x fp32 activations: TinyLLaMA guide, section 6.2 (expand
 *    the 4-bit values, multiply by the scale, multiply-add with the fp32
 *    activations).
 *  - Sigmoid router selecting experts: Colibri page, "Arquitectura del
 *    Sistema" (DeepSeek-V3-style sigmoid router).  Normalisation of the
 *    selected gates over the k, tie-break to the lower expert index and
 *    absence of bias are this oracle's reading (the page is silent); the
 *    function is pinned to that reading (stable argsort of the logits, the
 *    library sigmoid, closed forms), not to anything the page fixes.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - the activation is divided by the fp32 scale d32 = amax/127 (before it is
 *    rounded to fp16 for storage); the same for weights with amax/7;
 *  - IEEE fp32 division, round-half-away-from-zero, clamp to [-127,127]
 *    (activations) and [-8,7] (weights); an all-zero block gets d = 0, q = 0;
 *  - nibble order inside the 16 bytes: byte j holds element j in its low
 *    nibble and element j+16 in its high nibble, stored as u = q + 8;
 *  - fp16 conversion is IEEE round-to-nearest-even with subnormals.
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -ffp-contract=off -pthread -lm
 * (no -ffast-math: every float operation below must be IEEE).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QK 32 /* values per block (TinyLLaMA guide 6.1) */

/* ------------------------------------------------------------------ */
/* fp16 <-> fp32, written from the IEEE 754 binary16 definition.       */
/* ------------------------------------------------------------------ */

uint16_t oq_f32_to_f16(float f)
{
    uint32_t x;
    memcpy(&x, &f, 4);
    uint32_t sign = (x >> 16) & 0x8000u;
    uint32_t ax = x & 0x7FFFFFFFu;
    uint32_t E = ax >> 23; /* biased fp32 exponent */

    if (ax > 0x7F800000u) return (uint16_t)(sign | 0x7E00u); /* NaN */
    if (ax == 0x7F800000u) return (uint16_t)(sign | 0x7C00u); /* inf */
    /* 65520 is the midpoint between 65504 (largest half) and 2^16; ties go
       to even, and 65504's last mantissa bit is odd, so >= 65520 -> inf. */
    if (ax >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u);

    if (E >= 113) { /* >= 2^-14: normal half */
        uint32_t mant = ax & 0x7FFFFFu;
        uint32_t h = ((E - 127 + 15) << 10) | (mant >> 13);
        uint32_t rem = mant & 0x1FFFu;
        if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1; /* carry may bump exponent: correct */
        return (uint16_t)(sign | h);
    }
    if (E <= 101) return (uint16_t)sign; /* below 2^-25: rounds to zero */
    {
        /* half subnormal: value = h * 2^-24; fp32 value = m * 2^(E-150) */
        uint32_t m = (ax & 0x7FFFFFu) | 0x800000u;
        uint32_t s = 126 - E; /* 14 .. 24 */
        uint32_t h = m >> s;
        uint32_t rem = m & ((1u << s) - 1u);
        uint32_t half = 1u << (s - 1);
        if (rem > half || (rem == half && (h & 1u))) h += 1;
        return (uint16_t)(sign | h);
    }
}

float oq_f16_to_f32(uint16_t h)
{
    uint32_t sign = (h >> 15) & 1u;
    uint32_t e = (h >> 10) & 0x1Fu;
    uint32_t m = h & 0x3FFu;
    double v;
    if (e == 0) v = ldexp((double)m, -24);
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexp((double)(1024 + m), (int)e - 25);
    return (float)(sign ? -v : v);
}

void oq_f32_to_f16_array(const float* in, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oq_f32_to_f16(in[i]);
}

void oq_f16_to_f32_array(const uint16_t* in, float* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oq_f16_to_f32(in[i]);
}

/* round half away from zero, exact for any finite float */
static float round_half_away(float v)
{
    double a = floor(fabs((double)v) + 0.5);
    return (float)(v < 0 ? -a : a);
}

/* ------------------------------------------------------------------ */
/* Quantizers (llama.cpp guide 2.2; Colibri "Q8_0-style" activations)  */
/* ------------------------------------------------------------------ */

/* One block: amax, d32 = amax/qmax, q = clamp(rha(v/d32), qmin, qmax). */
static void quantize_block(const float* v, float qmax, int qmin, int qmax_i, int8_t* q, uint16_t* d16)
{
    float amax = 0.0f;
    for (int i = 0; i < QK; ++i) {
        float a = fabsf(v[i]);
        if (a > amax) amax = a;
    }
    float d32 = amax / qmax; /* IEEE fp32 division */
    *d16 = oq_f32_to_f16(d32);
    for (int i = 0; i < QK; ++i) {
        int r = 0;
        if (amax != 0.0f) {
            float t = round_half_away(v[i] / d32);
            r = (int)t;
            if (r < qmin) r = qmin;
            if (r > qmax_i) r = qmax_i;
        }
        q[i] = (int8_t)r;
    }
}

/* Q8_0 activations: x [M][K] (row stride ldx) -> q [M][K], d [M][K/32]. */
void oq_quantize_q8_0(const float* x, int64_t M, int64_t K, int64_t ldx, int8_t* q, uint16_t* d)
{
    int64_t B = K / QK;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t b = 0; b < B; ++b)
            quantize_block(x + m * ldx + b * QK, 127.0f, -127, 127, q + m * K + b * QK, d + m * B + b);
}

/* Q4_0 weights: w [N][K] (row stride ldw) -> signed q [N][K] in [-8,7], d [N][K/32]. */
void oq_quantize_q4_0(const float* w, int64_t N, int64_t K, int64_t ldw, int8_t* q, uint16_t* d)
{
    int64_t B = K / QK;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < B; ++b)
            quantize_block(w + n * ldw + b * QK, 7.0f, -8, 7, q + n * K + b * QK, d + n * B + b);
}

/* Serialise Q4_0 into the page's 18-byte blocks: fp16 scale (little endian),
   then 16 bytes of nibbles, byte j = (q[j]+8) | (q[j+16]+8) << 4. */
void oq_pack_q4_0_blocks(const int8_t* q, const uint16_t* d, int64_t N, int64_t K, uint8_t* blocks)
{
    int64_t B = K / QK;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < B; ++b) {
            uint8_t* blk = blocks + (n * B + b) * 18;
            uint16_t s = d[n * B + b];
            blk[0] = (uint8_t)(s & 0xFF);
            blk[1] = (uint8_t)(s >> 8);
            const int8_t* qq = q + n * K + b * QK;
            for (int j = 0; j < 16; ++j)
                blk[2 + j] = (uint8_t)((qq[j] + 8) | ((qq[j + 16] + 8) << 4));
        }
}

/* Inverse of the above: 18-byte blocks -> signed q and scales. */
void oq_unpack_q4_0_blocks(const uint8_t* blocks, int64_t N, int64_t K, int8_t* q, uint16_t* d)
{
    int64_t B = K / QK;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < B; ++b) {
            const uint8_t* blk = blocks + (n * B + b) * 18;
            d[n * B + b] = (uint16_t)(blk[0] | (blk[1] << 8));
            int8_t* qq = q + n * K + b * QK;
            for (int j = 0; j < 16; ++j) {
                qq[j] = (int8_t)((blk[2 + j] & 0x0F) - 8);
                qq[j + 16] = (int8_t)((blk[2 + j] >> 4) - 8);
            }
        }
}

/* ------------------------------------------------------------------ */
/* Block dots and the two output paths                                 */
/* ------------------------------------------------------------------ */

/* dots[m][n][b] = sum_{i<32} qw[n][32b+i] * qx[m][32b+i]   (int32) */
void oq_block_dots(const int8_t* qw, int64_t N, int64_t K, const int8_t* qx, int64_t M, int32_t* dots)
{
    int64_t B = K / QK;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            for (int64_t b = 0; b < B; ++b) {
                int32_t s = 0;
                for (int i = 0; i < QK; ++i)
                    s += (int32_t)qw[n * K + b * QK + i] * (int32_t)qx[m * K + b * QK + i];
                dots[(m * N + n) * B + b] = s;
            }
}

/* Integer path for one (token, row): y = sum_b dw*dx*dot_b in double,
   S = sum_b |dw*dx*dot_b| (scale of the fp32 tolerance). */
static void row_int(const int8_t* qw_row, const uint16_t* dw_row, const int8_t* qx_row, const uint16_t* dx_row,
                    int64_t B, double* y, double* S)
{
    double acc = 0.0, mag = 0.0;
    for (int64_t b = 0; b < B; ++b) {
        int32_t dot = 0;
        for (int i = 0; i < QK; ++i) dot += (int32_t)qw_row[b * QK + i] * (int32_t)qx_row[b * QK + i];
        double t = (double)oq_f16_to_f32(dw_row[b]) * (double)oq_f16_to_f32(dx_row[b]) * (double)dot;
        acc += t;
        mag += fabs(t);
    }
    *y = acc;
    if (S) *S = mag;
}

typedef struct {
    const int8_t* qw;
    const uint16_t* dw;
    int64_t N, K;
    const int8_t* qx;
    const uint16_t* dx;
    int64_t M;
    const int64_t* rows; /* NULL = all rows; else list of nrows row indices */
    int64_t nrows;
    double* y; /* [M][nrows] */
    double* S; /* [M][nrows] or NULL */
    int64_t begin, end; /* slice of the output rows for this thread */
} mm_job;

static void* mm_worker(void* p)
{
    mm_job* j = (mm_job*)p;
    int64_t B = j->K / QK;
    for (int64_t r = j->begin; r < j->end; ++r) {
        int64_t n = j->rows ? j->rows[r] : r;
        for (int64_t m = 0; m < j->M; ++m)
            row_int(j->qw + n * j->K, j->dw + n * B, j->qx + m * j->K, j->dx + m * B, B,
                    &j->y[m * j->nrows + r], j->S ? &j->S[m * j->nrows + r] : NULL);
    }
    return NULL;
}

/* y[m][r] for r over `rows` (or all N rows when rows == NULL, nrows = N).
   Rows are split over `nthreads` plain threads (timing convenience only;
   every output is computed the same way whatever the thread count). */
void oq_matmul_int(const int8_t* qw, const uint16_t* dw, int64_t N, int64_t K, const int8_t* qx, const uint16_t* dx,
                   int64_t M, const int64_t* rows, int64_t nrows, double* y, double* S, int nthreads)
{
    if (!rows) nrows = N;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    mm_job jobs[256];
    int64_t per = (nrows + nthreads - 1) / nthreads;
    int used = 0;
    for (int t = 0; t < nthreads; ++t) {
        int64_t b = t * per, e = b + per;
        if (e > nrows) e = nrows;
        if (b >= e) break;
        mm_job jb = {qw, dw, N, K, qx, dx, M, rows, nrows, y, S, b, e};
        jobs[t] = jb;
        used++;
    }
    if (used <= 1) {
        if (used == 1) mm_worker(&jobs[0]);
        return;
    }
    for (int t = 0; t < used; ++t) pthread_create(&th[t], NULL, mm_worker, &jobs[t]);
    for (int t = 0; t < used; ++t) pthread_join(th[t], NULL);
}

/* Dequantize-then-multiply path in float64: y'[m][n] = sum_k (dw*qw)(dx*qx).
   Every product of two dequantized values is exact in double; only the
   summation order differs from the integer path. */
void oq_matmul_dequant(const int8_t* qw, const uint16_t* dw, int64_t N, int64_t K, const int8_t* qx,
                       const uint16_t* dx, int64_t M, double* y)
{
    int64_t B = K / QK;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double a = (double)oq_f16_to_f32(dw[n * B + k / QK]) * (double)qw[n * K + k];
                double c = (double)oq_f16_to_f32(dx[m * B + k / QK]) * (double)qx[m * K + k];
                acc += a * c;
            }
            y[m * N + n] = acc;
        }
}

/* ------------------------------------------------------------------ */
/* Per-row-scale int4 / int2 containers (Colibri page, "Arquitectura   */
/* del Sistema": an int4 container with per-row scales, int4 and int2  */
/* packing).  The page gives no layout; the readings taken:            */
/*  - delta = amax(row)/qmax in fp32, qmax = 2^(bits-1) - 1, the       */
/*    llama.cpp guide 2.2 rule applied to the whole row;               */
/*  - q = clamp(rha(w/delta), -2^(bits-1), qmax); a zero row: 0, 0;    */
/*  - codes u = q + 2^(bits-1), packed 8/bits per byte, element i of   */
/*    the row in byte i*bits/8 at bit (i mod (8/bits))*bits;           */
/*  - the scale is kept as fp32.                                       */
/* ------------------------------------------------------------------ */

void oq_quantize_rowwise(const float* w, int64_t N, int64_t K, int64_t ldw, int bits, int8_t* q, float* s)
{
    const int qmax = (1 << (bits - 1)) - 1, qmin = -(1 << (bits - 1));
    for (int64_t n = 0; n < N; ++n) {
        const float* v = w + n * ldw;
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float a = fabsf(v[k]);
            if (a > amax) amax = a;
        }
        float delta = amax / (float)qmax; /* IEEE fp32 division */
        s[n] = delta;
        for (int64_t k = 0; k < K; ++k) {
            int r = 0;
            if (amax != 0.0f) {
                r = (int)round_half_away(v[k] / delta);
                if (r < qmin) r = qmin;
                if (r > qmax) r = qmax;
            }
            q[n * K + k] = (int8_t)r;
        }
    }
}

void oq_pack_rowwise(const int8_t* q, int64_t N, int64_t K, int bits, uint8_t* packed)
{
    const int per = 8 / bits, off = 1 << (bits - 1);
    const int64_t rowb = K / per;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t j = 0; j < rowb; ++j) {
            unsigned byte = 0;
            for (int i = 0; i < per; ++i) {
                unsigned u = (unsigned)(q[n * K + j * per + i] + off);
                byte |= u << (i * bits);
            }
            packed[n * rowb + j] = (uint8_t)byte;
        }
}

void oq_unpack_rowwise(const uint8_t* packed, int64_t N, int64_t K, int bits, int8_t* q)
{
    const int per = 8 / bits, off = 1 << (bits - 1);
    const unsigned mask = (1u << bits) - 1u;
    const int64_t rowb = K / per;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t j = 0; j < rowb; ++j)
            for (int i = 0; i < per; ++i)
                q[n * K + j * per + i] = (int8_t)((int)((packed[n * rowb + j] >> (i * bits)) & mask) - off);
}

/* Per-row codes x Q8_0 activations: y[m][n] = sum_b s[n] * dx[m][b] * dot_b
   with dot_b the int32 dot over the activation's 32-value block b, combined
   in double; S[m][n] = sum_b |s[n] * dx[m][b] * dot_b|. */
void oq_matmul_rowwise_int(const int8_t* qw, const float* s, int64_t N, int64_t K, const int8_t* qx,
                           const uint16_t* dx, int64_t M, double* y, double* S)
{
    int64_t B = K / QK;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, mag = 0.0;
            for (int64_t b = 0; b < B; ++b) {
                int32_t dot = 0;
                for (int i = 0; i < QK; ++i) dot += (int32_t)qw[n * K + b * QK + i] * (int32_t)qx[m * K + b * QK + i];
                double t = (double)s[n] * (double)oq_f16_to_f32(dx[m * B + b]) * (double)dot;
                acc += t;
                mag += fabs(t);
            }
            y[m * N + n] = acc;
            S[m * N + n] = mag;
        }
}

/* Q4_0 weights x fp32 activations, the dequantize-then-FMA flow of the
   TinyLLaMA guide 6.2 (expand the 4-bit codes, multiply by the block scale,
   multiply-add with the fp32 activations): y[m][n] = sum_k (dw*qw)[n][k] *
   x[m][k] in double (each product exact); S[m][n] = sum_k |(dw*qw) x|. */
void oq_matmul_q4_0_f32(const int8_t* qw, const uint16_t* dw, int64_t N, int64_t K, const float* x, int64_t M,
                        double* y, double* S)
{
    int64_t B = K / QK;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double w = (double)oq_f16_to_f32(dw[n * B + k / QK]) * (double)qw[n * K + k];
                double t = w * (double)x[m * K + k];
                acc += t;
                mag += fabs(t);
            }
            y[m * N + n] = acc;
            S[m * N + n] = mag;
        }
}

/* ------------------------------------------------------------------ */
/* MoE pieces (Colibri page; TinyLLaMA guide 4.4)                      */
/* ------------------------------------------------------------------ */

/* Sigmoid scores, top-k by score (ties -> lower expert index), gates
   normalised over the selected k.  logits [T][E] -> ids [T][k], gates [T][k]. */
void oq_router_topk(const float* logits, int64_t T, int64_t E, int64_t k, int32_t* ids, double* gates)
{
    double* s = (double*)malloc(sizeof(double) * (size_t)E);
    char* taken = (char*)malloc((size_t)E);
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t e = 0; e < E; ++e) {
            s[e] = 1.0 / (1.0 + exp(-(double)logits[t * E + e]));
            taken[e] = 0;
        }
        double tot = 0.0;
        for (int64_t j = 0; j < k; ++j) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || s[e] > s[best])) best = e;
            taken[best] = 1;
            ids[t * k + j] = (int32_t)best;
            gates[t * k + j] = s[best];
            tot += s[best];
        }
        for (int64_t j = 0; j < k; ++j) gates[t * k + j] /= tot;
    }
    free(s);
    free(taken);
}

/* h = Swish(a) * b = a * sigmoid(a) * b in double, rounded once to fp32. */
void oq_swiglu(const double* a, const double* b, int64_t n, float* h)
{
    for (int64_t i = 0; i < n; ++i) {
        double sw = a[i] / (1.0 + exp(-a[i]));
        h[i] = (float)(sw * b[i]);
    }
}

/* RMSNorm of one vector of d values: y_i = x_i / sqrt((1/d) sum_j x_j^2 + eps)
 * * gamma_i, all in double, each y_i rounded once to fp32. */
void oq_rmsnorm(const float* x, const float* gamma, int64_t d, double eps, float* y)
{
    double ss = 0.0;
    for (int64_t j = 0; j < d; ++j) ss += (double)x[j] * (double)x[j];
    const double r = sqrt(ss / (double)d + eps);
    for (int64_t i = 0; i < d; ++i) y[i] = (float)((double)x[i] / r * (double)gamma[i]);
}

/* y[t][n] = sum_{j=0..k-1} gates[t][j] * z[t][j][n], in that order, double. */
void oq_moe_combine(const double* z, const float* gates, int64_t T, int64_t k, int64_t N, double* y)
{
    for (int64_t t = 0; t < T; ++t)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t j = 0; j < k; ++j) acc += (double)gates[t * k + j] * z[(t * k + j) * N + n];
            y[t * N + n] = acc;
        }
}
