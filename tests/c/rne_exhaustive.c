/* Exhaustive pin of the oracle's fp64 -> bf16 rounding: for every one of the
 * 2^32 binary32 bit patterns f, oracle_round_bf16((double)f) must equal the
 * result of an independent binary32 -> bf16 round-to-nearest-even written with
 * integer arithmetic (add 0x7FFF plus the lowest kept bit, then truncate; NaN
 * patterns map to the canonical 0x7FC0). Every binary32 value is exact in
 * binary64, so a single correct rounding of either kind gives the same bits.
 * Prints the number of mismatches and the first few. */
#include <pthread.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

uint16_t oracle_round_bf16(double x);

static uint16_t integer_rne(uint32_t u) {
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0x7FC0u;
    uint32_t r = u + 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(r >> 16);
}

typedef struct { uint64_t lo, hi, bad; uint32_t first[4]; } job_t;

static void *run(void *p) {
    job_t *j = (job_t *)p;
    for (uint64_t v = j->lo; v < j->hi; ++v) {
        uint32_t u = (uint32_t)v;
        float f;
        __builtin_memcpy(&f, &u, 4);
        if (oracle_round_bf16((double)f) != integer_rne(u)) {
            if (j->bad < 4) j->first[j->bad] = u;
            j->bad++;
        }
    }
    return NULL;
}

int main(int argc, char **argv) {
    int nt = argc > 1 ? atoi(argv[1]) : 8;
    if (nt < 1) nt = 1;
    if (nt > 256) nt = 256;
    pthread_t t[256];
    job_t jobs[256] = {0};
    uint64_t total = 1ull << 32;
    for (int i = 0; i < nt; ++i) {
        jobs[i].lo = total * i / nt;
        jobs[i].hi = total * (i + 1) / nt;
    }
    for (int i = 0; i < nt; ++i) pthread_create(&t[i], 0, run, &jobs[i]);
    uint64_t bad = 0;
    for (int i = 0; i < nt; ++i) {
        pthread_join(t[i], 0);
        for (uint64_t k = 0; k < jobs[i].bad && k < 4; ++k) printf("mismatch 0x%08x\n", jobs[i].first[k]);
        bad += jobs[i].bad;
    }
    printf("checked %llu mismatches %llu\n", (unsigned long long)total, (unsigned long long)bad);
    return bad != 0;
}
