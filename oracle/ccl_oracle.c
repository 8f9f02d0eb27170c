/*
 * Oracle for chunk-oriented collective schedules.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no source, header, table or helper with the
 * CUDA library: the op layout below is restated here on purpose.
 *
 * What it computes (MSCCLang report, §III.1 "system design"): a program is a
 * list of chunk operations over per-rank buffers named input / output /
 * scratch; an operation is either a copy (dst := src) or a reduce
 * (dst := dst (+) src).  The compiler traces dependencies in program order, so
 * executing the operations one after another in program order is a valid
 * topological order of the traced DAG and is what this interpreter does.
 *
 * Arithmetic (reading of the pages, which never state a precision): every
 * reduce rounds its result to the buffer dtype, i.e. a partial sum travels
 * between ranks in the buffer dtype.
 *   f32  : IEEE binary32 addition, round to nearest even.
 *   bf16 : widen both operands to binary32 (exact), add in binary32, round the
 *          binary32 sum to bf16 with round-to-nearest-even.
 *   f16  : same with IEEE binary16.
 *   i32  : addition modulo 2^32.
 * Because binary32 carries at least 2p+2 bits for p = 8 (bf16) and p = 11
 * (f16), the binary32 sum rounded again to the narrow type equals the
 * correctly rounded narrow sum (double rounding is innocuous for addition
 * when the wide precision is at least 2p+2; Figueroa, 1995).
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -fPIC -shared (no vector
 * intrinsics, no -march flags: the same bits on x86-64 and aarch64).
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>

/* dtype codes */
#define OR_F32 0
#define OR_BF16 1
#define OR_F16 2
#define OR_I32 3
/* buffer kinds */
#define OR_IN 0
#define OR_OUT 1
#define OR_SCR 2
/* op codes */
#define OR_COPY 0
#define OR_REDUCE 1

/* status codes returned by oracle_run */
#define OR_OK 0
#define OR_EBADOP -1
#define OR_ERANGE -2
#define OR_EOVERLAP -3
#define OR_EDTYPE -4

/* One operation = 8 int32 words:
 *   [0] op (copy/reduce) [1] src_rank [2] src_buf [3] src_off
 *   [4] dst_rank [5] dst_buf [6] dst_off [7] count
 * Offsets and counts are in chunk units. */

/* ---------------------------------------------------------------------
 * Rounding written from the IEEE 754 definition of round-to-nearest-even:
 * keep the representable neighbour below, look at the discarded bits,
 * round up when they exceed half an ulp, or equal half an ulp and the kept
 * last bit is odd.
 * ------------------------------------------------------------------- */

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u = f32_bits(f);
    if ((u & 0x7f800000u) == 0x7f800000u) {          /* inf or NaN */
        if (u & 0x007fffffu) return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN */
        return (uint16_t)(u >> 16);
    }
    /* bf16 keeps the upper 16 bits of the binary32 pattern (same exponent
     * field); the lower 16 bits are discarded.  An increment of the kept
     * pattern carries into the exponent, which is the correct next value
     * (and reaches infinity exactly when the rounded value overflows). */
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xffffu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) kept += 1u;
    return (uint16_t)kept;
}

float oracle_bf16_to_f32(uint16_t h) { return bits_f32((uint32_t)h << 16); }

uint16_t oracle_f32_to_f16(float f)
{
    uint32_t u = f32_bits(f);
    uint32_t sign = (u >> 16) & 0x8000u;
    uint32_t e = (u >> 23) & 0xffu;
    uint32_t m = u & 0x7fffffu;
    if (e == 0xffu) return (uint16_t)(sign | 0x7c00u | (m ? 0x0200u : 0u));
    if (e == 0u) return (uint16_t)sign;   /* |x| < 2^-126, far below half of 2^-24 */
    int E = (int)e - 127;                 /* x = sig * 2^(E-23), sig in [2^23, 2^24) */
    uint32_t sig = m | 0x800000u;
    /* binary16 normal numbers (E >= -14) keep 11 significant bits; below that
     * the grid is fixed at 2^-24 and fewer bits survive. */
    int shift = (E >= -14) ? 13 : 13 + (-14 - E);
    if (shift > 25) return (uint16_t)sign; /* below a quarter of 2^-24 */
    uint32_t q = sig >> shift;
    uint32_t rem = sig & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (q & 1u))) q += 1u;
    if (E >= -14) {
        uint32_t ef = (uint32_t)(E + 15);
        if (q == 0x800u) { q = 0x400u; ef += 1u; }   /* rounded up to next binade */
        if (ef >= 31u) return (uint16_t)(sign | 0x7c00u);   /* overflow to infinity */
        return (uint16_t)(sign | (ef << 10) | (q & 0x3ffu));
    }
    /* subnormal result; q == 0x400 encodes the smallest normal number */
    return (uint16_t)(sign | q);
}

float oracle_f16_to_f32(uint16_t h)
{
    uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
    uint32_t e = ((uint32_t)h >> 10) & 0x1fu;
    uint32_t m = (uint32_t)h & 0x3ffu;
    if (e == 0x1fu) return bits_f32(sign | 0x7f800000u | (m << 13));
    if (e == 0u) {
        /* subnormal: m * 2^-24, exact in binary32 */
        float v = (float)m * 5.9604644775390625e-08f;
        return (sign ? -v : v);
    }
    return bits_f32(sign | ((e + 112u) << 23) | (m << 13));
}

/* ---------------------------------------------------------------------
 * Element reductions, one rounding per call.
 * ------------------------------------------------------------------- */

float oracle_add_f32(float a, float b) { return a + b; }

uint16_t oracle_add_bf16(uint16_t a, uint16_t b)
{
    return oracle_f32_to_bf16(oracle_bf16_to_f32(a) + oracle_bf16_to_f32(b));
}

uint16_t oracle_add_f16(uint16_t a, uint16_t b)
{
    return oracle_f32_to_f16(oracle_f16_to_f32(a) + oracle_f16_to_f32(b));
}

int32_t oracle_add_i32(int32_t a, int32_t b)
{
    return (int32_t)((uint32_t)a + (uint32_t)b);
}

/* Array forms, used by the rounding pins. */
void oracle_f32_to_bf16_array(const float* x, uint16_t* y, int64_t n)
{ for (int64_t i = 0; i < n; ++i) y[i] = oracle_f32_to_bf16(x[i]); }
void oracle_f32_to_f16_array(const float* x, uint16_t* y, int64_t n)
{ for (int64_t i = 0; i < n; ++i) y[i] = oracle_f32_to_f16(x[i]); }
void oracle_f16_to_f32_array(const uint16_t* x, float* y, int64_t n)
{ for (int64_t i = 0; i < n; ++i) y[i] = oracle_f16_to_f32(x[i]); }
void oracle_add_bf16_array(const uint16_t* a, const uint16_t* b, uint16_t* y, int64_t n)
{ for (int64_t i = 0; i < n; ++i) y[i] = oracle_add_bf16(a[i], b[i]); }
void oracle_add_f16_array(const uint16_t* a, const uint16_t* b, uint16_t* y, int64_t n)
{ for (int64_t i = 0; i < n; ++i) y[i] = oracle_add_f16(a[i], b[i]); }

static int esize_of(int dtype)
{
    switch (dtype) {
    case OR_F32: case OR_I32: return 4;
    case OR_BF16: case OR_F16: return 2;
    default: return 0;
    }
}

/* ---------------------------------------------------------------------
 * The interpreter.
 *
 * bufs[kind * nranks + r] points at rank r's buffer of that kind, laid out
 * as nchunks[kind] consecutive chunks of chunk_elems elements each.
 * Ops run one at a time in program order.  An op whose source and
 * destination ranges overlap in the same buffer is rejected (a chunk
 * operation reads its whole source before the destination is defined).
 * Returns 0, or a negative status and sets *bad_op to the failing op index.
 * ------------------------------------------------------------------- */
int oracle_run(const int32_t* ops, int nops, int nranks, const int64_t* nchunks,
               int64_t chunk_elems, int dtype, void* const* bufs, int* bad_op)
{
    int es = esize_of(dtype);
    if (bad_op) *bad_op = -1;
    if (es == 0) return OR_EDTYPE;
    for (int i = 0; i < nops; ++i) {
        const int32_t* o = ops + 8 * (int64_t)i;
        int op = o[0];
        int sr = o[1], sb = o[2], so = o[3];
        int dr = o[4], db = o[5], dof = o[6], cnt = o[7];
        if (op != OR_COPY && op != OR_REDUCE) { if (bad_op) *bad_op = i; return OR_EBADOP; }
        if (sr < 0 || sr >= nranks || dr < 0 || dr >= nranks || sb < 0 || sb > 2 || db < 0 || db > 2
            || so < 0 || dof < 0 || cnt <= 0
            || (int64_t)so + cnt > nchunks[sb] || (int64_t)dof + cnt > nchunks[db]) {
            if (bad_op) *bad_op = i;
            return OR_ERANGE;
        }
        if (sr == dr && sb == db && so < dof + cnt && dof < so + cnt) {
            if (bad_op) *bad_op = i;
            return OR_EOVERLAP;
        }
        int64_t n = (int64_t)cnt * chunk_elems;
        char* s = (char*)bufs[sb * nranks + sr] + (int64_t)so * chunk_elems * es;
        char* d = (char*)bufs[db * nranks + dr] + (int64_t)dof * chunk_elems * es;
        if (op == OR_COPY) {
            memcpy(d, s, (size_t)(n * es));
            continue;
        }
        switch (dtype) {
        case OR_F32: {
            const float* x = (const float*)s; float* y = (float*)d;
            for (int64_t k = 0; k < n; ++k) y[k] = oracle_add_f32(y[k], x[k]);
            break; }
        case OR_BF16: {
            const uint16_t* x = (const uint16_t*)s; uint16_t* y = (uint16_t*)d;
            for (int64_t k = 0; k < n; ++k) y[k] = oracle_add_bf16(y[k], x[k]);
            break; }
        case OR_F16: {
            const uint16_t* x = (const uint16_t*)s; uint16_t* y = (uint16_t*)d;
            for (int64_t k = 0; k < n; ++k) y[k] = oracle_add_f16(y[k], x[k]);
            break; }
        case OR_I32: {
            const int32_t* x = (const int32_t*)s; int32_t* y = (int32_t*)d;
            for (int64_t k = 0; k < n; ++k) y[k] = oracle_add_i32(y[k], x[k]);
            break; }
        }
    }
    return OR_OK;
}
