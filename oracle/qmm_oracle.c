/*
 * qmm_oracle.c -- the plain, slow, CPU oracle for block-quantized GEMV/GEMM.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, load or call
 * this file: only the test suite, the smoke check and the benchmark's CPU
 * baseline leg do. It shares no source, header, table or helper with the CUDA
 * library; the two meet only through the bytes the seeded input generators
 * produce.
 *
 * What it computes, and from which passage:
 *
 *   oracle_f16         IEEE binary16 -> binary32, written from the format's
 *                      definition (value = m * 2^-24 for a zero exponent field,
 *                      (1024 + m) * 2^(e - 25) otherwise, Inf/NaN at e = 31).
 *                      The pages decode the same way: Vulkore
 *                      examples/llm/quant_test.cpp, `ref_fp16`, and ferrox-cuda
 *                      0.21.0 src/mul_mm.rs, `f16_to_f32`.
 *   oracle_e8m0        2^(e - 127) for every byte, e = 0 giving 2^-127 and
 *                      e = 255 giving +Inf: ferrox-cuda 0.20.0
 *                      src/mul_mm_kinds/codebook.rs, `ferrox_e8m0_to_f32` and
 *                      the test `every_e8m0_byte_is_two_to_the_e_minus_127`.
 *   oracle_elem        value of element i of one weight row, indexed by
 *                      ELEMENT (where do this element's bits live?), in fp32,
 *                      one function per block format (see each case below).
 *   oracle_dequant     every element of a rows x cols matrix.
 *   oracle_gemm        y[n*M + m] = sum_k w[m,k] * x[n,k] accumulated in fp64
 *                      (double accumulation as in Vulkore quant_test.cpp's fused
 *                      matvec check), with tol = 1e-3 * sum_k |w*x| + 1e-6.
 *   oracle_gemm_at     the same for a list of (n, m) output positions.
 *   oracle_grouped     the expert-indexed product: assignment r reads expert
 *                      expert_id[r]'s weights and activation row x_row[r].
 *
 * Formats and their page of origin:
 *   Q8_0, Q5_0, Q4_K, Q6_K    Vulkore quant_test.cpp, namespace `ref`.
 *   Q4_0                      ferrox-cuda codebook.rs, `IQ4_NL` doc comment
 *                             (Q4_0's packing: code byte j holds element j in
 *                             its low four bits and element j+16 in its high
 *                             four bits; codes carry a -8 bias).
 *   IQ4_NL, IQ4_XS, MXFP4     ferrox-cuda codebook.rs, the three kind rows and
 *                             the `KVALUES_IQ4NL` / `KVALUES_MXFP4` tables.
 *   Q4_1, Q5_1, Q8_1          named by ferrox-cuda 0.21.0 mul_mm.rs (the
 *                             `kind_by_name` test's list of kinds with no
 *                             kernel) without a layout; this file takes the
 *                             public GGUF block definitions: Q4_1 and Q5_1 are
 *                             Q4_0 and Q5_0 with unsigned codes and an f16
 *                             min after the f16 scale (w = d*q + m); Q8_1 is
 *                             Q8_0 with an f16 field after d that holds d times
 *                             the sum of the codes, which no element reads
 *                             (w = d*q). PARITY UNPINNED against the pages
 *                             for these three, as for the next three.
 *   Q5_K, Q2_K, Q3_K          named by ferrox-cuda mul_mm.rs (module docs and
 *                             `KINDS`), which also says Q5_K shares Q4_K's
 *                             6-bit scale/min unpack and that Q3_K has an
 *                             hmask-driven bias. Their byte layouts are NOT on
 *                             the pages; this file takes the public GGUF block
 *                             definitions. PARITY UNPINNED against the pages
 *                             for these three: the tests pin them only to that
 *                             reading (hand-built blocks, one-hot fields and
 *                             cross-format invariants).
 *
 * Compile with -ffp-contract=off: every product below is exact in fp32 and the
 * affine-min formats round once, at the final subtraction, exactly as written.
 *
 * Sabotage builds (-DORACLE_SABOTAGE=n) plant one plausible mistake each so
 * the tests can show that their pins fire. They are never used for parity.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_SABOTAGE
#define ORACLE_SABOTAGE 0
#endif

/* Format identifiers of the oracle (its own numbering, by name in Python). */
enum {
    OR_Q8_0 = 0, OR_Q4_0, OR_Q5_0, OR_Q4_K, OR_Q5_K, OR_Q6_K,
    OR_Q2_K, OR_Q3_K, OR_IQ4_NL, OR_IQ4_XS, OR_MXFP4,
    OR_Q4_1, OR_Q5_1, OR_Q8_1, OR_NKINDS
};

/* Bytes and elements of one block, per format. */
static const int kBlockBytes[OR_NKINDS] = {34, 18, 22, 144, 176, 210, 84, 110, 18, 136, 17, 20, 24, 36};
static const int kBlockElems[OR_NKINDS] = {32, 32, 32, 256, 256, 256, 256, 256, 32, 256, 32, 32, 32, 32};

/* IQ4_NL / IQ4_XS codebook, as printed in ferrox-cuda codebook.rs KVALUES_IQ4NL. */
static const float kIq4nl[16] = {-127.f, -104.f, -83.f, -65.f, -49.f, -35.f, -22.f, -10.f,
                                 1.f, 13.f, 25.f, 38.f, 53.f, 69.f, 89.f, 113.f};

/* E2M1 codebook, as printed in ferrox-cuda codebook.rs KVALUES_MXFP4 (code 8 is -0.0). */
static const float kE2m1[16] = {0.f, .5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f,
#if ORACLE_SABOTAGE == 7
                                0.f,
#else
                                -0.f,
#endif
                                -.5f, -1.f, -1.5f, -2.f, -3.f, -4.f, -6.f};

int oracle_block_geometry(int kind, int* block_bytes, int* block_elems) {
    if (kind < 0 || kind >= OR_NKINDS) return -1;
    *block_bytes = kBlockBytes[kind];
    *block_elems = kBlockElems[kind];
    return 0;
}

int oracle_sabotage_id(void) { return ORACLE_SABOTAGE; }

/* IEEE binary16 from its definition. */
float oracle_f16(uint16_t h) {
    const int s = (h >> 15) & 1;
    const int e = (h >> 10) & 31;
    const int m = h & 1023;
    double v;
    if (e == 31) {
        v = m ? NAN : INFINITY;
    } else if (e == 0) {
        v = ldexp((double)m, -24);
    } else {
        v = ldexp((double)(1024 + m), e - 25);
    }
    return (float)(s ? -v : v);
}

/* E8M0 scale byte: 2^(e - 127). Computed in double and narrowed: 2^-127 is an
 * fp32 subnormal (exact) and 2^128 narrows to +Inf. */
float oracle_e8m0(uint8_t e) { return (float)ldexp(1.0, (int)e - 127); }

static inline uint32_t u16le(const uint8_t* b, int o) { return (uint32_t)b[o] | ((uint32_t)b[o + 1] << 8); }
static inline uint32_t u32le(const uint8_t* b, int o) {
    return (uint32_t)b[o] | ((uint32_t)b[o + 1] << 8) | ((uint32_t)b[o + 2] << 16) | ((uint32_t)b[o + 3] << 24);
}
static inline int s8(uint8_t v) { return (v & 0x80) ? (int)v - 256 : (int)v; }

/* Low or high nibble of byte `byte`. */
static inline int nib(uint8_t byte, int high) { return high ? (byte >> 4) : (byte & 15); }

/* Q4_K / Q5_K packed 6-bit (scale, min) of sub-block j in 0..7 of the 12-byte
 * field s (Vulkore quant_test.cpp, `q4k_scale_min`; ferrox-cuda mul_mm.rs says
 * Q5_K uses the same unpack). */
static void k4_scale_min(const uint8_t* s, int j, int* sc, int* mn) {
    if (j < 4) {
        *sc = s[j] & 63;
        *mn = s[j + 4] & 63;
    } else {
        *sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        *mn = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

/* Q3_K 6-bit scale j in 0..15, before the -32 bias (GGUF reading). */
static int q3k_scale(const uint8_t* s, int j) {
    const int low4 = j < 8 ? (s[j] & 15) : (s[j - 8] >> 4);
    const int high2 = (s[8 + (j % 4)] >> (2 * (j / 4))) & 3;
    return low4 | (high2 << 4);
}

/* Element e (0 <= e < block_elems) of the block starting at b. */
static float block_elem(int kind, const uint8_t* b, int e) {
    switch (kind) {
    case OR_Q8_0: {
        /* 34 B: f16 d, 32 x int8. w = d * q. */
        return oracle_f16((uint16_t)u16le(b, 0)) * (float)s8(b[2 + e]);
    }
    case OR_Q4_0: {
        /* 18 B: f16 d, 16 B of nibbles. Byte j: low = element j, high = element j+16.
         * w = d * (q - 8). */
#if ORACLE_SABOTAGE == 4
        const int q = e < 16 ? nib(b[2 + e], 1) : nib(b[2 + e - 16], 0);
#else
        const int q = e < 16 ? nib(b[2 + e], 0) : nib(b[2 + e - 16], 1);
#endif
        return oracle_f16((uint16_t)u16le(b, 0)) * (float)(q - 8);
    }
    case OR_Q5_0: {
        /* 22 B: f16 d, u32 qh, 16 B nibbles. The fifth bit of element e is bit e
         * of qh. w = d * (q - 16). */
        const uint32_t qh = u32le(b, 2);
        const int lo = nib(b[6 + e % 16], e >= 16);
#if ORACLE_SABOTAGE == 1
        const int hb = (int)((qh >> (e >= 16 ? e - 4 : e)) & 1);
#else
        const int hb = (int)((qh >> e) & 1);
#endif
        return oracle_f16((uint16_t)u16le(b, 0)) * (float)((lo | (hb << 4)) - 16);
    }
    case OR_Q4_K:
    case OR_Q5_K: {
        /* Q4_K 144 B: f16 d, f16 dmin, 12 B scales/mins, 128 B nibbles.
         * Q5_K 176 B: the same head, then 32 B qh, then 128 B nibbles.
         * Elements come in 64-element chunks c = e/64: the first 32 are the low
         * nibbles of the chunk's 32 bytes, the next 32 the high nibbles.
         * Sub-block (32 elements) e/32 selects the (scale, min) pair.
         * w = d*sc*q - dmin*m. */
        const float d = oracle_f16((uint16_t)u16le(b, 0));
        const float dmin = oracle_f16((uint16_t)u16le(b, 2));
        int sc, mn;
        k4_scale_min(b + 4, e / 32, &sc, &mn);
        const int qs_off = kind == OR_Q4_K ? 16 : 48;
        int q = nib(b[qs_off + (e / 64) * 32 + e % 32], (e % 64) >= 32);
        if (kind == OR_Q5_K) q += 16 * ((b[16 + e % 32] >> (e / 32)) & 1);
#if ORACLE_SABOTAGE == 6
        return d * (float)sc * (float)q;
#else
        return d * (float)sc * (float)q - dmin * (float)mn;
#endif
    }
    case OR_Q6_K: {
        /* 210 B: ql[128], qh[64], int8 scales[16], f16 d at byte 208.
         * Each 128-element half h holds four interleaved 32-element quarters g:
         * low 4 bits from ql (quarters 0,1 low nibbles, 2,3 high nibbles),
         * high 2 bits from qh shifted by 2g. Scale index e/16. w = d*sc*(q-32). */
        const int h = e / 128, w = e % 128, l = w % 32, g = w / 32;
        const uint8_t byte = b[h * 64 + l + (g & 1) * 32];
        const int lo = nib(byte, g >= 2);
        const int hi = (b[128 + h * 32 + l] >> (2 * g)) & 3;
        const int q = (lo | (hi << 4)) - 32;
#if ORACLE_SABOTAGE == 5
        const int sc = s8(b[192 + e / 32]);
#else
        const int sc = s8(b[192 + e / 16]);
#endif
        return oracle_f16((uint16_t)u16le(b, 208)) * (float)sc * (float)q;
    }
    case OR_Q2_K: {
        /* GGUF reading. 84 B: scales[16] (low nibble scale, high nibble min),
         * qs[64], f16 d, f16 dmin. 2-bit code of element e sits in
         * qs[32h + l] at bit 2g, h/g/l as in Q6_K. w = d*(s&15)*q - dmin*(s>>4). */
        const int h = e / 128, w = e % 128, l = w % 32, g = w / 32;
        const int q = (b[16 + h * 32 + l] >> (2 * g)) & 3;
        const int s = b[e / 16];
        const float d = oracle_f16((uint16_t)u16le(b, 80));
        const float dmin = oracle_f16((uint16_t)u16le(b, 82));
        return d * (float)(s & 15) * (float)q - dmin * (float)(s >> 4);
    }
    case OR_Q3_K: {
        /* GGUF reading. 110 B: hmask[32], qs[64], scales[12], f16 d.
         * 2-bit code as in Q2_K (qs at byte 32); a CLEAR hmask bit e/32 of byte
         * e%32 subtracts 4. 6-bit scales (see q3k_scale) biased by -32.
         * w = d * (sc - 32) * q. */
        const int h = e / 128, w = e % 128, l = w % 32, g = w / 32;
        const int q2 = (b[32 + h * 32 + l] >> (2 * g)) & 3;
        const int hb = (b[e % 32] >> (e / 32)) & 1;
#if ORACLE_SABOTAGE == 3
        const int q = q2 - (hb ? 4 : 0);
#else
        const int q = q2 - (hb ? 0 : 4);
#endif
        const int sc = q3k_scale(b + 96, e / 16) - 32;
        return oracle_f16((uint16_t)u16le(b, 108)) * (float)sc * (float)q;
    }
    case OR_IQ4_NL: {
        /* 18 B: f16 d, 16 B of codes packed as Q4_0. w = d * KV[c]. */
        const int c = e < 16 ? nib(b[2 + e], 0) : nib(b[2 + e - 16], 1);
        return oracle_f16((uint16_t)u16le(b, 0)) * kIq4nl[c];
    }
    case OR_IQ4_XS: {
        /* 136 B: f16 d, u16 scales_h, 4 B scales_l, 128 B codes. Group ib = e/32
         * has a 6-bit scale: low 4 bits = nibble (ib & 1) of scales_l[ib/2],
         * high 2 bits = bits 2ib..2ib+1 of scales_h; biased by -32. The group's
         * 32 codes are packed as an IQ4_NL block. w = d * (ls - 32) * KV[c]. */
        const int ib = e / 32, f = e % 32;
        const int c = nib(b[8 + 16 * ib + f % 16], f >= 16);
        const uint32_t scales_h = u16le(b, 2);
#if ORACLE_SABOTAGE == 2
        const int hsh = 2 * (e / 16 % 8);
#else
        const int hsh = 2 * ib;
#endif
        const int ls = ((b[4 + ib / 2] >> (4 * (ib & 1))) & 15) | (int)(((scales_h >> hsh) & 3) << 4);
        return oracle_f16((uint16_t)u16le(b, 0)) * (float)(ls - 32) * kIq4nl[c];
    }
    case OR_MXFP4: {
        /* 17 B: E8M0 scale byte, 16 B of E2M1 codes packed as IQ4_NL.
         * w = 2^(e-127) * E2M1[c]. */
        const int c = e < 16 ? nib(b[1 + e], 0) : nib(b[1 + e - 16], 1);
        return oracle_e8m0(b[0]) * kE2m1[c];
    }
    case OR_Q4_1: {
        /* GGUF reading. 20 B: f16 d, f16 m, 16 B of nibbles packed as Q4_0.
         * Unsigned code, w = d * q + m (the product is exact; one rounding at
         * the addition). */
        const int q = e < 16 ? nib(b[4 + e], 0) : nib(b[4 + e - 16], 1);
        const float d = oracle_f16((uint16_t)u16le(b, 0));
        const float m = oracle_f16((uint16_t)u16le(b, 2));
#if ORACLE_SABOTAGE == 9
        return d * (float)q - m;
#else
        return d * (float)q + m;
#endif
    }
    case OR_Q5_1: {
        /* GGUF reading. 24 B: f16 d, f16 m, u32 qh, 16 B of nibbles; the fifth
         * bit of element e is bit e of qh, as in Q5_0. w = d * q + m. */
        const uint32_t qh = u32le(b, 4);
        const int lo = nib(b[8 + e % 16], e >= 16);
        const int q = lo | (int)(((qh >> e) & 1) << 4);
        return oracle_f16((uint16_t)u16le(b, 0)) * (float)q + oracle_f16((uint16_t)u16le(b, 2));
    }
    case OR_Q8_1: {
        /* GGUF reading. 36 B: f16 d, f16 s (= d * sum of the codes; read by
         * nothing here), 32 x int8. w = d * q. */
#if ORACLE_SABOTAGE == 10
        return oracle_f16((uint16_t)u16le(b, 0)) * (float)s8(b[2 + e]);
#else
        return oracle_f16((uint16_t)u16le(b, 0)) * (float)s8(b[4 + e]);
#endif
    }
    default:
        return NAN;
    }
}

/* Element i of the row starting at `row` (the row's blocks are contiguous). */
float oracle_elem(int kind, const uint8_t* row, int64_t i) {
    if (kind < 0 || kind >= OR_NKINDS) return NAN;
    const int bb = kBlockBytes[kind], be = kBlockElems[kind];
    return block_elem(kind, row + (size_t)(i / be) * (size_t)bb, (int)(i % be));
}

static size_t row_bytes_of(int kind, int64_t cols) {
    return (size_t)(cols / kBlockElems[kind]) * (size_t)kBlockBytes[kind];
}

int oracle_dequant(int kind, const uint8_t* w, int64_t rows, int64_t cols, float* out) {
    if (kind < 0 || kind >= OR_NKINDS || cols % kBlockElems[kind] != 0) return -1;
    const size_t rb = row_bytes_of(kind, cols);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < cols; ++k)
            out[r * cols + k] = oracle_elem(kind, w + (size_t)r * rb, k);
    return 0;
}

/* Activation element: x_dtype 0 = fp32, 1 = IEEE binary16 bits. */
static double x_at(const void* x, int x_dtype, int64_t idx) {
    if (x_dtype == 1) return (double)oracle_f16(((const uint16_t*)x)[idx]);
    return (double)((const float*)x)[idx];
}

/* One output: sum_k w[m,k] * x[xrow,k] in fp64 and its tolerance. */
static void dot_one(int kind, const uint8_t* wrow, int64_t K, const void* x, int x_dtype,
                    int64_t xrow, double* y, double* tol) {
    double acc = 0.0, mag = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        const double w = (double)oracle_elem(kind, wrow, k);
#if ORACLE_SABOTAGE == 8
        const double xv = x_at(x, x_dtype, xrow * K + (k ^ 1));
#else
        const double xv = x_at(x, x_dtype, xrow * K + k);
#endif
        acc += w * xv;
        mag += fabs(w * xv);
    }
    *y = acc;
    *tol = 1e-3 * mag + 1e-6;
}

/* Y[n*M + m] = sum_k W[m,k] X[n*K + k]; tol alike. nthreads <= 0 means one. */
int oracle_gemm(int kind, const uint8_t* w, int64_t M, int64_t K, const void* x, int x_dtype,
                int64_t N, double* y, double* tol, int nthreads) {
    if (kind < 0 || kind >= OR_NKINDS || K % kBlockElems[kind] != 0) return -1;
    const size_t rb = row_bytes_of(kind, K);
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 4) num_threads(nthreads)
#endif
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            dot_one(kind, w + (size_t)m * rb, K, x, x_dtype, n, &y[n * M + m], &tol[n * M + m]);
    (void)nthreads;
    return 0;
}

/* The same product at `count` chosen positions (n_idx[i], m_idx[i]). */
int oracle_gemm_at(int kind, const uint8_t* w, int64_t M, int64_t K, const void* x, int x_dtype,
                   int64_t count, const int64_t* n_idx, const int64_t* m_idx, double* y, double* tol) {
    if (kind < 0 || kind >= OR_NKINDS || K % kBlockElems[kind] != 0) return -1;
    const size_t rb = row_bytes_of(kind, K);
    for (int64_t i = 0; i < count; ++i) {
        if (m_idx[i] < 0 || m_idx[i] >= M) return -2;
        dot_one(kind, w + (size_t)m_idx[i] * rb, K, x, x_dtype, n_idx[i], &y[i], &tol[i]);
    }
    return 0;
}

/* Expert-indexed product: for assignment r, Y[r*M + m] = sum_k W_e[m,k] X[x_row[r]*K + k]
 * with e = expert_id[r] and W_e = W + e * expert_stride bytes. rows_sel/count
 * restrict to chosen (r, m) pairs when count >= 0; count < 0 means all. */
int oracle_grouped(int kind, const uint8_t* w, int64_t expert_stride, int n_experts,
                   const void* x, int x_dtype, const int32_t* x_row, const int32_t* expert_id,
                   int64_t n_assign, int64_t M, int64_t K,
                   int64_t count, const int64_t* r_idx, const int64_t* m_idx,
                   double* y, double* tol, int nthreads) {
    if (kind < 0 || kind >= OR_NKINDS || K % kBlockElems[kind] != 0) return -1;
    const size_t rb = row_bytes_of(kind, K);
    for (int64_t r = 0; r < n_assign; ++r)
        if (expert_id[r] < 0 || expert_id[r] >= n_experts) return -3;
    if (count >= 0) {
        for (int64_t i = 0; i < count; ++i) {
            const int64_t r = r_idx[i], m = m_idx[i];
            const uint8_t* we = w + (size_t)expert_id[r] * (size_t)expert_stride;
            dot_one(kind, we + (size_t)m * rb, K, x, x_dtype, x_row[r], &y[i], &tol[i]);
        }
        return 0;
    }
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 4) num_threads(nthreads)
#endif
    for (int64_t r = 0; r < n_assign; ++r) {
        const uint8_t* we = w + (size_t)expert_id[r] * (size_t)expert_stride;
        for (int64_t m = 0; m < M; ++m)
            dot_one(kind, we + (size_t)m * rb, K, x, x_dtype, x_row[r], &y[r * M + m], &tol[r * M + m]);
    }
    (void)nthreads;
    return 0;
}

int oracle_has_openmp(void) {
#ifdef _OPENMP
    return 1;
#else
    return 0;
#endif
}
