/*
 * Seeded synthetic input generator shared by the tests, the bench and the
 * oracle's callers.  It holds none of the engine's arithmetic: it only turns a
 * (seed, operand, element index) triple into an input value.
 *
 * Generator: SplitMix64 (S. Vigna's published mixer, the state-increment
 * constant is the 64-bit golden ratio), used counter-based: draw k of a stream
 * whose initial state is s0 is mix(s0 + (k + 1) * GAMMA).  Every element can
 * therefore be produced independently, in any order and in any chunk.
 *
 * Stream of operand j of a workload with seed s: s0 = s * 16 + j.
 * Uniform [0,1): the top 53 bits of a draw times 2^-53.
 * Normal: Box-Muller, one value per pair of draws (2k, 2k+1), cosine branch.
 */
#include <math.h>
#include <stdint.h>

#define DG_GAMMA 0x9E3779B97F4A7C15ULL
#define DG_RETRY 0x632BE59BD9B4E019ULL

static uint64_t dg_mix(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static uint64_t dg_draw(uint64_t s0, uint64_t k) { return dg_mix(s0 + (k + 1) * DG_GAMMA); }

static double dg_u01(uint64_t z) { return (double)(z >> 11) * (1.0 / 9007199254740992.0); }

void dg_raw_u64(uint64_t s0, int64_t offset, int64_t n, uint64_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = dg_draw(s0, (uint64_t)(offset + i));
}

/* top 32 bits of each draw: raw bit patterns for 32-bit integer inputs */
void dg_raw_u32(uint64_t s0, int64_t offset, int64_t n, uint32_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = (uint32_t)(dg_draw(s0, (uint64_t)(offset + i)) >> 32);
}

/* U(lo, hi) evaluated in double, stored as float (round to nearest) */
void dg_uniform_f32(uint64_t s0, int64_t offset, int64_t n, double lo, double hi, float *out)
{
    for (int64_t i = 0; i < n; ++i) {
        double u = dg_u01(dg_draw(s0, (uint64_t)(offset + i)));
        out[i] = (float)(lo + (hi - lo) * u);
    }
}

/* N(mu, sigma) by Box-Muller, stored as float */
void dg_normal_f32(uint64_t s0, int64_t offset, int64_t n, double mu, double sigma, float *out)
{
    const double two_pi = 6.283185307179586476925286766559;
    for (int64_t i = 0; i < n; ++i) {
        uint64_t k = (uint64_t)(offset + i);
        double u1 = dg_u01(dg_draw(s0, 2 * k));
        double u2 = dg_u01(dg_draw(s0, 2 * k + 1));
        double r = sqrt(-2.0 * log(1.0 - u1));
        out[i] = (float)(mu + sigma * r * cos(two_pi * u2));
    }
}

/* |N(0,1)| + shift, stored as float (Div divisor of the contiguous workload) */
void dg_absnormal_f32(uint64_t s0, int64_t offset, int64_t n, double shift, float *out)
{
    dg_normal_f32(s0, offset, n, 0.0, 1.0, out);
    for (int64_t i = 0; i < n; ++i) out[i] = (float)(fabs((double)out[i]) + shift);
}

/*
 * U(lo, hi) with a fraction `pzero` of exact signed zeros (sign 50/50).
 * Element k uses draws 2k (zero or not, and the zero's sign) and 2k+1 (value).
 */
void dg_uniform_zeros_f32(uint64_t s0, int64_t offset, int64_t n, double lo, double hi,
                          double pzero, float *out)
{
    for (int64_t i = 0; i < n; ++i) {
        uint64_t k = (uint64_t)(offset + i);
        uint64_t z0 = dg_draw(s0, 2 * k);
        if (dg_u01(z0) < pzero) {
            out[i] = (z0 & 1u) ? -0.0f : 0.0f;
        } else {
            double u = dg_u01(dg_draw(s0, 2 * k + 1));
            out[i] = (float)(lo + (hi - lo) * u);
        }
    }
}

/*
 * U(lo, hi) rejecting |v| < min_abs.  Attempt t of element k draws from the
 * stream s0 + t * RETRY at counter k.
 */
void dg_uniform_reject_f32(uint64_t s0, int64_t offset, int64_t n, double lo, double hi,
                           double min_abs, float *out)
{
    for (int64_t i = 0; i < n; ++i) {
        uint64_t k = (uint64_t)(offset + i);
        float v = 0.0f;
        for (uint64_t t = 0; t < 1000; ++t) {
            double u = dg_u01(dg_draw(s0 + t * DG_RETRY, k));
            v = (float)(lo + (hi - lo) * u);
            if (fabs((double)v) >= min_abs) break;
        }
        out[i] = v;
    }
}

/*
 * Integers uniform on [lo, hi]; with skip_zero, uniform on [lo, hi] \ {0}
 * (requires lo <= 0 <= hi).  Stored as int64; callers narrow.
 */
void dg_int_range(uint64_t s0, int64_t offset, int64_t n, int64_t lo, int64_t hi, int skip_zero,
                  int64_t *out)
{
    uint64_t count = (uint64_t)(hi - lo) + 1u - (skip_zero ? 1u : 0u);
    for (int64_t i = 0; i < n; ++i) {
        double u = dg_u01(dg_draw(s0, (uint64_t)(offset + i)));
        int64_t v = lo + (int64_t)(u * (double)count);
        if (v > lo + (int64_t)count - 1) v = lo + (int64_t)count - 1;
        if (skip_zero && v >= 0) v += 1;
        out[i] = v;
    }
}
