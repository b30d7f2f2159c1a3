/* Exhaustive check of the residual rounding point over every ordered pair
 * (a, b) of binary16 bit patterns, 2^32 in all.
 *
 * Page "BW1000 gfx936 Pangu-Weather inference profiling", s4: the fused
 * residual add keeps the original FP16 rounding point, residual_out =
 * fp16(fp32(a) + fp32(b)).  The oracle states it as RN16 of the exact sum,
 * computed in double (where the sum of two binary16 values is exact):
 *     orc_rn16(orc_f16_to_f64(a) + orc_f16_to_f64(b)).
 * The two agree in theory (binary32 carries 24 >= 2 * 11 + 2 significand
 * bits, so rounding to it first and then to binary16 cannot differ from
 * rounding once: Figueroa, "When is double rounding innocuous?", 1995).
 * This program checks it for every pair instead of relying on the theorem.
 * The other side is computed independently of the oracle, with the C
 * compiler's binary16 type: widen both operands to float, add once in
 * float, convert the sum to _Float16 (round to nearest even).
 *
 * Results must have identical bits, except that any NaN matches any NaN.
 *
 *   residual_pairs <path to liboracle.so> <threads> [a_count]
 * prints "pairs P mismatches M" and exits 0 when M is 0.  a_count (default
 * 65536) limits the first operand to the patterns 0 .. a_count - 1.
 */
#include <dlfcn.h>
#include <pthread.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

typedef double (*decode_fn)(uint16_t);
typedef uint16_t (*round_fn)(double);

static double oracle_value[65536]; /* the oracle's exact value of each pattern */
static float widened[65536];       /* the compiler's float value of each pattern */
static round_fn oracle_rn16;

struct slice {
    uint32_t a0, a1;
    uint64_t mismatches;
    uint32_t first_a, first_b;
    uint16_t first_got, first_want;
};

static uint16_t bits_of(_Float16 h) {
    uint16_t u;
    memcpy(&u, &h, sizeof u);
    return u;
}

static int is_nan16(uint16_t u) { return (u & 0x7c00u) == 0x7c00u && (u & 0x03ffu) != 0; }

static void *run(void *arg) {
    struct slice *s = arg;
    for (uint32_t a = s->a0; a < s->a1; ++a)
        for (uint32_t b = 0; b < 65536u; ++b) {
            const float sum32 = widened[a] + widened[b];
            const uint16_t want = bits_of((_Float16)sum32);
            const uint16_t got = oracle_rn16(oracle_value[a] + oracle_value[b]);
            if (got != want && !(is_nan16(got) && is_nan16(want))) {
                if (s->mismatches == 0) {
                    s->first_a = a;
                    s->first_b = b;
                    s->first_got = got;
                    s->first_want = want;
                }
                ++s->mismatches;
            }
        }
    return NULL;
}

int main(int argc, char **argv) {
    if (argc != 3 && argc != 4) {
        fprintf(stderr, "usage: %s liboracle.so threads [a_count]\n", argv[0]);
        return 2;
    }
    long a_count = argc == 4 ? atol(argv[3]) : 65536;
    if (a_count < 1 || a_count > 65536) a_count = 65536;
    void *lib = dlopen(argv[1], RTLD_NOW);
    if (!lib) {
        fprintf(stderr, "dlopen: %s\n", dlerror());
        return 2;
    }
    decode_fn decode = (decode_fn)dlsym(lib, "orc_f16_to_f64");
    oracle_rn16 = (round_fn)dlsym(lib, "orc_rn16");
    if (!decode || !oracle_rn16) {
        fprintf(stderr, "liboracle.so lacks orc_f16_to_f64 / orc_rn16\n");
        return 2;
    }
    int threads = atoi(argv[2]);
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    for (uint32_t u = 0; u < 65536u; ++u) {
        _Float16 h;
        const uint16_t b16 = (uint16_t)u;
        memcpy(&h, &b16, sizeof h);
        widened[u] = (float)h;
        oracle_value[u] = decode((uint16_t)u);
    }
    pthread_t tid[256];
    struct slice sl[256];
    for (int t = 0; t < threads; ++t) {
        memset(&sl[t], 0, sizeof sl[t]);
        sl[t].a0 = (uint32_t)(((uint64_t)a_count * (uint64_t)t) / (uint64_t)threads);
        sl[t].a1 = (uint32_t)(((uint64_t)a_count * (uint64_t)(t + 1)) / (uint64_t)threads);
        if (pthread_create(&tid[t], NULL, run, &sl[t]) != 0) {
            fprintf(stderr, "pthread_create failed\n");
            return 2;
        }
    }
    uint64_t bad = 0;
    for (int t = 0; t < threads; ++t) {
        pthread_join(tid[t], NULL);
        if (sl[t].mismatches && !bad)
            fprintf(stderr, "first mismatch: a=0x%04x b=0x%04x oracle=0x%04x binary32 route=0x%04x\n",
                    sl[t].first_a, sl[t].first_b, sl[t].first_got, sl[t].first_want);
        bad += sl[t].mismatches;
    }
    printf("pairs %llu mismatches %llu\n", (unsigned long long)a_count * 65536ull,
           (unsigned long long)bad);
    return bad ? 1 : 0;
}
