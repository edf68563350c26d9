/*
 * CPU check of the prepared exact division behind float16 and bfloat16
 * BatchNormalization and BiasPReluBN (test infrastructure; it shares no code
 * with the engine or the oracle).  Restated from the algorithm:
 *     r = RN(1/d);  q0 = RN(t r);  q1 = RN(q0 + RN(t - q0 d) r);
 *     q2 = RN(q1 + RN(t - q1 d) r)                   (remainders and updates: FMAs)
 * kept when 2^-20 <= d <= 2^20, d's significand is at most 2^24 - 5 and
 * tlow <= |t| <= RD(2^99 d) (tlow = 2^-100, or 0 where the caller's t is
 * known to be +0 or at least 2^-99 in magnitude).  pd_check counts, over
 * pairs (t, d), the quotients kept, refused, and kept but different from the
 * correctly rounded t / d.
 * `corrections` = 2 is the engine's scheme; 0 plants a scheme without them.
 * Compile with -ffp-contract=off: every operation written rounds on its own.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static uint32_t to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

void pd_check(const float *ts, const float *ds, int64_t n, int corrections, float tlow,
              int64_t *counts, int64_t *first_bad)
{
    for (int64_t i = 0; i < n; ++i) {
        float t = ts[i], d = ds[i];
        volatile float vd = d;
        float r = 1.0f / vd;
        int row_ok = d >= 0x1p-20f && d <= 0x1p20f && (to_bits(d) & 0x7FFFFFu) <= 0x7FFFFBu;
        float q = t * r;
        for (int c = 0; c < corrections; ++c) {
            float rem = fmaf(q, -d, t);
            q = fmaf(rem, r, q);
        }
        /* RD(2^99 d): 2^99 d is exact (d is a binary32 value well inside the range) */
        float thigh = d * 0x1p99f;
        if (!(row_ok && fabsf(t) >= tlow && fabsf(t) <= thigh)) { counts[1]++; continue; }
        counts[0]++;
        volatile float vt = t;
        float want = vt / vd;                     /* IEEE division, round to nearest */
        if (to_bits(q) != to_bits(want)) {
            if (counts[2] == 0) *first_bad = i;
            counts[2]++;
        }
    }
}
