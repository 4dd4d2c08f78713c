/*
 * Seeded synthetic inputs for the shard-step workloads.
 *
 * This module is shared by the CPU oracle side and the CUDA side of the test
 * suite and by the benchmark. It holds none of the method's arithmetic: it
 * only turns (seed, step, tensor, kind, element index) into numbers.
 *
 * Generator (counter based, so any element can be drawn on its own and the
 * result does not depend on the thread count):
 *   - hash h(key, c) = splitmix64(key XOR splitmix64(c)), splitmix64 being
 *     Steele, Lea and Flood's SplitMix64 output function;
 *   - uniform u = ((h >> 11) + 0.5) * 2^-53, in (0, 1);
 *   - standard normal by Box-Muller (cosine branch only) in double;
 *   - Student-t with 3 degrees of freedom as Z0 / sqrt((Z1^2+Z2^2+Z3^2)/3).
 * Values are scaled in double, rounded to fp32 (round to nearest even), and,
 * for bf16 outputs, rounded once more from fp32 to bf16 (nearest even).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SYNTH_TWO_PI 6.283185307179586476925286766559

static inline uint64_t sm64(uint64_t x) {
    x += 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return x ^ (x >> 31);
}

static inline uint64_t hash2(uint64_t key, uint64_t c) { return sm64(key ^ sm64(c)); }

static inline double unit_open(uint64_t h) {
    return ((double)(h >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

/* j-th standard normal (j in 0..3) attached to element i of stream `key`. */
static inline double normal_at(uint64_t key, uint64_t i, uint64_t j) {
    double u1 = unit_open(hash2(key, 8 * i + 2 * j));
    double u2 = unit_open(hash2(key, 8 * i + 2 * j + 1));
    return sqrt(-2.0 * log(u1)) * cos(SYNTH_TWO_PI * u2);
}

static inline double student_t3_at(uint64_t key, uint64_t i) {
    double z0 = normal_at(key, i, 0);
    double z1 = normal_at(key, i, 1);
    double z2 = normal_at(key, i, 2);
    double z3 = normal_at(key, i, 3);
    double chi2 = z1 * z1 + z2 * z2 + z3 * z3;
    return z0 / sqrt(chi2 / 3.0);
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0;
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

uint64_t synth_key(uint64_t seed, uint64_t step, uint64_t tensor, uint64_t kind) {
    uint64_t k = sm64(seed);
    k = sm64(k ^ step);
    k = sm64(k ^ (tensor + 0x1000));
    k = sm64(k ^ (kind + 0x2000));
    return k;
}

/* kind: 0 = normal, 1 = Student-t(3). Elements [start, start+count). */
static inline double draw(int kind, uint64_t key, uint64_t i) {
    return kind == 1 ? student_t3_at(key, i) : normal_at(key, i, 0);
}

void synth_fill_f32(uint64_t key, int kind, double scale, uint64_t start, uint64_t count,
                    float* out) {
    int64_t n = (int64_t)count;
#pragma omp parallel for schedule(static, 65536)
    for (int64_t e = 0; e < n; ++e) out[e] = (float)(scale * draw(kind, key, start + (uint64_t)e));
}

void synth_fill_bf16(uint64_t key, int kind, double scale, uint64_t start, uint64_t count,
                     uint16_t* out) {
    int64_t n = (int64_t)count;
#pragma omp parallel for schedule(static, 65536)
    for (int64_t e = 0; e < n; ++e)
        out[e] = f32_to_bf16_rne((float)(scale * draw(kind, key, start + (uint64_t)e)));
}

/* Zero-fill helpers (used for the all-zero expert slices of a workload). */
void synth_zero_u16(uint16_t* out, uint64_t count) {
    int64_t n = (int64_t)count;
#pragma omp parallel for schedule(static, 65536)
    for (int64_t e = 0; e < n; ++e) out[e] = 0;
}

void synth_zero_f32(float* out, uint64_t count) {
    int64_t n = (int64_t)count;
#pragma omp parallel for schedule(static, 65536)
    for (int64_t e = 0; e < n; ++e) out[e] = 0.0f;
}

/* Pick k distinct indices out of n: the k smallest hash scores (ties by
 * index). Writes them ascending into out[0..k). Returns 0, or -1 if k > n. */
int synth_pick(uint64_t key, int32_t n, int32_t k, int32_t* out) {
    if (k > n || k < 0) return -1;
    int32_t taken = 0;
    while (taken < k) {
        int32_t best = -1;
        uint64_t best_s = 0;
        for (int32_t e = 0; e < n; ++e) {
            int used = 0;
            for (int32_t j = 0; j < taken; ++j) used |= (out[j] == e);
            if (used) continue;
            uint64_t s = hash2(key, (uint64_t)e);
            if (best < 0 || s < best_s) { best = e; best_s = s; }
        }
        out[taken++] = best;
    }
    for (int32_t a = 0; a < k; ++a)
        for (int32_t b = a + 1; b < k; ++b)
            if (out[b] < out[a]) { int32_t t = out[a]; out[a] = out[b]; out[b] = t; }
    return 0;
}

int synth_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
