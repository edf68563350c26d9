/* Host-side stress of the plan cache through the C ABI (no GPU work): T
 * threads ask for the same sequence of K new plans, released together by a
 * barrier before each one, so every key is a miss in several threads at once.
 * The cache keeps one entry per key, so all threads must receive the same
 * plan for each key.  Prints the number of keys that came back as more than
 * one plan and exits 0, or exits 2 when a call fails. */
#include <pthread.h>
#include <stdio.h>

#include "ebin.h"

#define T 8
#define K 2000

static ebin_descriptor_t desc;
static pthread_barrier_t start;
static ebin_plan_t got[T][K];
static int failed;

static void *work(void *arg) {
    const int t = (int)(long)arg;
    for (int k = 0; k < K; ++k) {
        const int64_t sa[2] = {k + 1, 32}, sb[1] = {32};
        pthread_barrier_wait(&start);
        if (ebin_plan_create(desc, sa, 2, sb, 1, &got[t][k]) != EBIN_OK) failed = 1;
    }
    return NULL;
}

int main(void) {
    if (ebin_descriptor_create(EBIN_OP_ADD, 18, NULL, EBIN_FLOAT32, EBIN_FLOAT32, &desc) != EBIN_OK)
        return 2;
    pthread_barrier_init(&start, NULL, T);
    pthread_t th[T];
    for (long t = 0; t < T; ++t) pthread_create(&th[t], NULL, work, (void *)t);
    for (int t = 0; t < T; ++t) pthread_join(th[t], NULL);
    if (failed) return 2;
    int split = 0;
    for (int k = 0; k < K; ++k) {
        for (int t = 1; t < T; ++t) {
            if (got[t][k] != got[0][k]) {
                ++split;
                break;
            }
        }
        for (int t = 0; t < T; ++t) ebin_plan_release(got[t][k]);
    }
    ebin_descriptor_destroy(desc);
    printf("%d\n", split);
    return 0;
}
