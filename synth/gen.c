/*
 * Seeded synthetic inputs shared by the tests, the benchmark and the oracle's
 * checks. This file draws random numbers and rounds them to bf16; it holds
 * none of the attention arithmetic.
 *
 * Generator (counter based, so any element can be produced independently):
 *   key(seed, tag)  = splitmix64(splitmix64(seed) ^ (tag * 0xD1B54A32D192ED03))
 *   word(key, i)    = splitmix64(key + i * 0x9E3779B97F4A7C15)
 * i.e. element i of the SplitMix64 sequence (Steele, Lea & Flood, OOPSLA 2014)
 * started from state `key`.
 *   uniform(w)      = ((w >> 11) + 1) * 2^-53                in (0, 1]
 *   normal pair i   = Box-Muller on uniform(word(2i)), uniform(word(2i+1)):
 *                     r = sqrt(-2 ln u1); z0 = r cos(2 pi u2); z1 = r sin(2 pi u2)
 * Normal number j of a stream is z_{j mod 2} of pair j/2.
 * bf16 rounding is round-to-nearest-even on the float32 bit pattern.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t splitmix64(uint64_t x) {
    x += 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return x ^ (x >> 31);
}

uint64_t synth_stream_key(uint64_t seed, uint64_t tag) {
    return splitmix64(splitmix64(seed) ^ (tag * 0xD1B54A32D192ED03ull));
}

static inline uint64_t word_at(uint64_t key, uint64_t i) {
    /* splitmix64() adds the gamma once more, so state = key + i*gamma */
    return splitmix64(key + i * 0x9E3779B97F4A7C15ull);
}

static inline double uniform_of(uint64_t w) {
    return (double)((w >> 11) + 1) * (1.0 / 9007199254740992.0);
}

static inline double normal_at(uint64_t key, uint64_t j) {
    uint64_t pair = j >> 1;
    double u1 = uniform_of(word_at(key, 2 * pair));
    double u2 = uniform_of(word_at(key, 2 * pair + 1));
    double r = sqrt(-2.0 * log(u1));
    double a = 6.283185307179586476925286766559 * u2;
    return (j & 1) ? r * sin(a) : r * cos(a);
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* Raw 64-bit words of a stream: out[i] = word(key(seed,tag), offset + i). */
void synth_words(uint64_t* out, int64_t n, uint64_t seed, uint64_t tag, uint64_t offset) {
    uint64_t key = synth_stream_key(seed, tag);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = word_at(key, offset + (uint64_t)i);
}

/* Standard normals of a stream as float64: out[i] = normal(key(seed,tag), offset + i). */
void synth_normals(double* out, int64_t n, uint64_t seed, uint64_t tag, uint64_t offset) {
    uint64_t key = synth_stream_key(seed, tag);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = normal_at(key, offset + (uint64_t)i);
}

/*
 * rows x d bf16 matrix, row r, column c:
 *   x = row_scale[r] * (centre[assign[r]*d + c] + sigma * z[r*d + c])
 * z = the normals of stream (seed, tag) from element 0; centre/assign/row_scale
 * may be NULL (centre 0, scale 1). The sum is formed in float32, then rounded.
 */
void synth_rows_bf16(uint16_t* out, int64_t rows, int d, uint64_t seed, uint64_t tag,
                     const float* centre, const int32_t* assign, float sigma,
                     const float* row_scale) {
    uint64_t key = synth_stream_key(seed, tag);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const float* cr = centre ? centre + (int64_t)assign[r] * d : 0;
        float s = row_scale ? row_scale[r] : 1.0f;
        for (int c = 0; c < d; ++c) {
            uint64_t j = (uint64_t)(r * d + c);
            float z = (float)normal_at(key, j);
            float x = (cr ? cr[c] : 0.0f) + sigma * z;
            out[r * d + c] = f32_to_bf16_rne(s * x);
        }
    }
}
