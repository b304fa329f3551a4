/*
 * ORACLE -- test infrastructure only. Nothing on the product path links,
 * loads or calls this file; only the tests, the smoke check and the
 * benchmark's CPU-baseline leg do.
 *
 * What it computes is the plain definition of the result, and nothing else:
 * the CPU's sequential double sum
 *
 *     double s = s0;  for (i = 0; i < n; i++) s += x[i];
 *
 * as stated in Research-1433 ("Forming the CPU's sequential double sums on a
 * GPU, bit for bit", Question), in Research-1424 section 1 ("The sum is the
 * only difference": calc_ssim() carries one double through the whole frame,
 * row after row) and in ADR-1464 (Context: iqa_ssim() adds every window's
 * term into one double per sum, left to right and top to bottom).  Each add
 * is one IEEE-754 binary64 addition, rounded to nearest with ties to even.
 *
 * The batched form is independent loops, one accumulator per sum
 * (ADR-1464, Decision: "the four are independent of one another";
 * ADR-1391, Decision item 2: six running sums per channel and scale).
 *
 * Build: this translation unit must be compiled with
 *   -O2 -fno-fast-math -ffp-contract=off -fno-tree-vectorize
 *   -fno-associative-math -fno-reciprocal-math -frounding-math
 * so that the compiler keeps every add, in order, unfused.  `volatile` on the
 * accumulator is a second guard against reassociation.
 *
 * It shares no code, header, table or helper with the CUDA path.
 */
#include <fenv.h>
#include <stdint.h>
#include <string.h>

#if defined(__FAST_MATH__)
#error "the oracle must not be built with -ffast-math"
#endif

/* One sequential sum.  x may be NULL when n == 0. */
double oracle_seqsum(const double *x, int64_t n, double s0)
{
    volatile double s = s0;
    for (int64_t i = 0; i < n; i++)
        s = s + x[i];
    return s;
}

/* nsums independent sequential sums over x[offsets[k] .. offsets[k+1]). */
void oracle_seqsum_batched(const double *x, const int64_t *offsets, int32_t nsums,
                           const double *s0s, double *outs)
{
    for (int32_t k = 0; k < nsums; k++)
        outs[k] = oracle_seqsum(x + offsets[k], offsets[k + 1] - offsets[k], s0s[k]);
}

/* stride interleaved sums, one accumulator each (ADR-1464, "float_ssim_cuda
 * sums in raster order on the host", Decision: the lcs variant's four sums
 * per window): outs[k] = s0s[k] + x[k] + x[k + stride] + ... over n terms,
 * and the frame score's epilogue means[k] = (float)(outs[k] / n). */
void oracle_seqsum_strided(const double *x, int64_t n, int32_t stride, const double *s0s, double *outs,
                           float *means)
{
    for (int32_t k = 0; k < stride; k++) {
        volatile double s = s0s[k];
        for (int64_t i = 0; i < n; i++)
            s = s + x[i * stride + k];
        outs[k] = s;
        volatile double q = s / (double)n;
        means[k] = (float)q;
    }
}

/* Trace variant: writes the running sum after every add (out[i] = s after
 * term i).  Used by tests that need the exact S at a chunk boundary. */
void oracle_seqsum_trace(const double *x, int64_t n, double s0, double *out)
{
    volatile double s = s0;
    for (int64_t i = 0; i < n; i++) {
        s = s + x[i];
        out[i] = s;
    }
}

/* Environment check: returns 0 when the host FPU is in the state the
 * definition needs, else a bit mask of what is wrong:
 *   1: rounding mode is not round-to-nearest-even
 *   2: subnormal results are flushed to zero
 *   4: subnormal inputs are treated as zero
 * The checks are functional (no inline assembly), so they run the same way on
 * x86-64 and aarch64. */
int oracle_env_check(void)
{
    int bad = 0;
    if (fegetround() != FE_TONEAREST)
        bad |= 1;
    volatile double tiny = 0x1p-1022;       /* smallest normal */
    volatile double half = 0.5;
    volatile double r = tiny * half;        /* 0x1p-1023, a subnormal */
    if (r != 0x1p-1023)
        bad |= 2;
    volatile double sub = 0x1p-1070;        /* subnormal input */
    volatile double r2 = sub + sub;         /* 0x1p-1069 */
    uint64_t bits;
    double r2v = r2;
    memcpy(&bits, &r2v, sizeof bits);
    if (bits != 0x0000000000000020ull)      /* 2^-1069 = 32 * 2^-1074 */
        bad |= 4;
    return bad;
}
