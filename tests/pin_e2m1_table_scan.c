/*
 * Exhaustive pin of an E2M1 encoder against the E2M1 value table.
 *
 * For every fp32 bit pattern in [first, first + count) that is finite, the
 * expected code is found by scanning the 8 table magnitudes for the smallest
 * distance to |v| (ties go to the even code), saturating |v| > 6 to the
 * largest magnitude, with the sign bit taken from v.  The encoder under test
 * is called through a function pointer (fp64 argument, as the oracle takes
 * it).  Returns the number of disagreements; the first one is reported in
 * *first_bad.
 *
 * Table and rule: OCP Microscaling Formats (MX) v1.0, E2M1 element format,
 * conversion with roundTiesToEven and saturation (the MXFP4 elements of
 * "KroQuant ...", Sec. 4.1 "Data format").
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

typedef uint8_t (*encode_fn)(double);

static uint8_t table_scan(float f, const double mag[8])
{
    double v = (double)f;
    double a = fabs(v);
    int best = 7;
    if (!(a > mag[7])) {
        double bd = INFINITY;
        for (int k = 0; k < 8; ++k) {
            double dist = fabs(a - mag[k]);
            if (dist < bd || (dist == bd && (k & 1) == 0)) {
                bd = dist;
                best = k;
            }
        }
    }
    return (uint8_t)((signbit(v) ? 8 : 0) | best);
}

uint64_t pin_count_mismatches(uint64_t first, uint64_t count, const double *mag,
                              encode_fn enc, uint64_t *first_bad)
{
    uint64_t bad = 0, fb = UINT64_MAX;
    #pragma omp parallel for schedule(static, 1 << 16) reduction(+ : bad) reduction(min : fb)
    for (uint64_t k = 0; k < count; ++k) {
        uint32_t u = (uint32_t)(first + k);
        if (((u >> 23) & 0xFF) == 0xFF) continue;   /* inf / NaN: out of contract */
        float f;
        memcpy(&f, &u, sizeof f);
        if (enc((double)f) != table_scan(f, mag)) {
            ++bad;
            if (first + k < fb) fb = first + k;
        }
    }
    *first_bad = fb;
    return bad;
}

/* Table-scan codes for a range, packed two per byte (code of the even
 * pattern in bits 0-3): the brute-force expectation for the device encoder. */
void pin_table_scan_packed(uint64_t first, uint64_t count, const double *mag, uint8_t *out)
{
    #pragma omp parallel for schedule(static, 1 << 14)
    for (uint64_t k = 0; k < count / 2; ++k) {
        uint8_t c[2];
        for (int t = 0; t < 2; ++t) {
            uint32_t u = (uint32_t)(first + 2 * k + t);
            float f;
            memcpy(&f, &u, sizeof f);
            c[t] = table_scan(f, mag);
        }
        out[k] = (uint8_t)(c[0] | (c[1] << 4));
    }
}
