/* shard_demo.c -- the data-parallel token split from plain C99: for a (B, S)
 * token grid and `world` ranks, print each rank's tokens [t0, t1) and its
 * runs as "rank t0 t1 nruns b0 s0 nb ns ...", one line per rank, then "ok".
 * rope_partial_token_shard makes no CUDA call, so this runs without a GPU.
 *
 * Usage: shard_demo B S WORLD */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "rope_partial.h"

int main(int argc, char** argv) {
    if (argc != 4) {
        fprintf(stderr, "usage: %s B S WORLD\n", argv[0]);
        return 1;
    }
    const int64_t B = atoll(argv[1]), S = atoll(argv[2]);
    const int32_t world = (int32_t)atoi(argv[3]);
    for (int32_t rank = 0; rank < world; ++rank) {
        int64_t t0 = 0, t1 = 0;
        int32_t n = 0;
        rope_token_run_t runs[3];
        const rope_status_t st = rope_partial_token_shard(B, S, rank, world, &t0, &t1, runs, &n);
        if (st != ROPE_OK) {
            fprintf(stderr, "rank %d: %s: %s\n", (int)rank, rope_status_str(st),
                    rope_last_error_message());
            return 2;
        }
        printf("%d %lld %lld %d", (int)rank, (long long)t0, (long long)t1, (int)n);
        for (int32_t k = 0; k < n; ++k)
            printf(" %lld %lld %lld %lld", (long long)runs[k].b0, (long long)runs[k].s0,
                   (long long)runs[k].nb, (long long)runs[k].ns);
        printf("\n");
    }
    /* an invalid rank is refused */
    int64_t t0, t1;
    int32_t n;
    rope_token_run_t runs[3];
    if (rope_partial_token_shard(B, S, world, world, &t0, &t1, runs, &n) != ROPE_ERR_INVALID) return 3;
    printf("ok\n");
    return 0;
}
