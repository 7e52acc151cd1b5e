/*
 * Fast host implementation of the synthetic-input generators of workloads/rng.py
 * (SplitMix64 counter stream, 53-bit uniforms, cosine-branch Box-Muller in double,
 * double -> float -> bfloat16 round-to-nearest-even).  Same definitions, same bits;
 * a test compares it with the numpy version.  Draws numbers only: none of the
 * decode method's arithmetic is here.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static uint64_t splitmix_at(uint64_t key, uint64_t j) /* output j of the stream */
{
    return mix64(key + (j + 1) * 0x9E3779B97F4A7C15ull);
}

static uint16_t to_bf16(double x)
{
    float f = (float)x;
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

static const double TWO_M53 = 1.0 / 9007199254740992.0;
static const double TWO_PI = 6.283185307179586;  /* 2 * numpy.pi, correctly rounded */

void fastgen_normal_bf16(uint64_t key, int64_t start, int64_t count, uint64_t spike_key, double spike_prob,
                         double spike_factor, int use_spike, uint16_t *out)
{
    for (int64_t i = 0; i < count; ++i) {
        uint64_t idx = (uint64_t)(start + i);
        uint64_t z1 = splitmix_at(key, 2 * idx), z2 = splitmix_at(key, 2 * idx + 1);
        double u1 = ((double)(z1 >> 11) + 1.0) * TWO_M53;
        double u2 = (double)(z2 >> 11) * TWO_M53;
        double n = sqrt(-2.0 * log(u1)) * cos(TWO_PI * u2);
        if (use_spike) {
            double u = (double)(splitmix_at(spike_key, idx) >> 11) * TWO_M53;
            if (u < spike_prob)
                n = n * spike_factor;
        }
        out[i] = to_bf16(n);
    }
}
