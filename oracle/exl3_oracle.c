/*
 * Float64 C decoder for the EXL3 trellis oracle.
 *
 * TEST INFRASTRUCTURE: used only through oracle/exl3_oracle.py by the tests,
 * the smoke check and the benchmark's CPU baseline.  Shares nothing with the
 * CUDA path.  Plain C, one weight at a time, bit by bit.
 *
 * Follows "EXL3 linear and grouped routed experts" (TensorFold #837), "What
 * this changes": 16x16 tiles of K-bit trellis codes, codebooks mul1 / mcg /
 * 3inst.  The bit layout, the 16-bit tail-biting bitshift state and the
 * codebook constants are the readings stated in exl3_oracle.py.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { CB_MUL1 = 0, CB_MCG = 1, CB_3INST = 2 };

/* IEEE 754 binary16 -> double, from the sign, exponent and fraction fields. */
static double half_to_double(uint32_t h)
{
    uint32_t sign = (h >> 15) & 1u, expo = (h >> 10) & 0x1Fu, frac = h & 0x3FFu;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -24);                       /* subnormal / zero */
    else if (expo == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp(1.0 + (double)frac / 1024.0, (int)expo - 15);
    return sign ? -mag : mag;
}

double oracle_codebook(uint32_t state, int cb)
{
    uint32_t x;
    if (cb == CB_MUL1) {
        x = (uint32_t)(0x83DCD12Du * state);
        double s = (double)(x & 0xFFu) + (double)((x >> 8) & 0xFFu) +
                   (double)((x >> 16) & 0xFFu) + (double)(x >> 24);
        return (s - 510.0) / sqrt(21845.0);
    }
    if (cb == CB_MCG)
        x = (uint32_t)(0xCBAC1FEDu * state);
    else
        x = (uint32_t)(89226354u * state + 64248484u);
    x = (x & 0x8FFF8FFFu) ^ 0x3B603B60u;
    return half_to_double(x & 0xFFFFu) + half_to_double(x >> 16);
}

/* State of position p: the 16 bits ending at bit (p+1)K-1 of the cyclic
 * 256K-bit string, first bit most significant. */
static uint32_t state_at(const uint32_t *words, int K, int p)
{
    int nbits = 256 * K;
    uint32_t s = 0;
    for (int i = 0; i < 16; i++) {
        int b = ((p + 1) * K - 16 + i) % nbits;
        if (b < 0)
            b += nbits;
        uint32_t bit = (words[b / 32] >> (31 - b % 32)) & 1u;
        s = (s << 1) | bit;
    }
    return s;
}

void oracle_tile_states(const uint32_t *words, int K, uint32_t *states)
{
    for (int p = 0; p < 256; p++)
        states[p] = state_at(words, K, p);
}

/* W[in][out] (row-major doubles) from T[in/16][out/16][8K]. */
int oracle_decode_projection(const uint32_t *T, int in_f, int out_f, int K, int cb,
                             double *W)
{
    if (K < 1 || K > 8 || cb < 0 || cb > 2 || in_f % 16 || out_f % 16)
        return -1;
    int ntk = in_f / 16, ntn = out_f / 16, nw = 8 * K;
#pragma omp parallel for collapse(2) schedule(static)
    for (int tk = 0; tk < ntk; tk++) {
        for (int tn = 0; tn < ntn; tn++) {
            const uint32_t *w = T + ((size_t)tk * ntn + tn) * nw;
            for (int p = 0; p < 256; p++) {
                int r = p % 16, c = p / 16;
                W[(size_t)(tk * 16 + r) * out_f + tn * 16 + c] =
                    oracle_codebook(state_at(w, K, p), cb);
            }
        }
    }
    return 0;
}

int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
