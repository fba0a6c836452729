/* A plain C99 caller of the library's C ABI (include/zero3.h): the host-side
 * entry points only (planner, placement queries, accounting, status text),
 * so it runs without a GPU.  Values checked are the pages' own:
 *  - "ddp-to-zero-memory-sharding" (111qqz.com), section
 *    "ZeRO-3：参数为什么也可以分片": a layer of eight weights on four GPUs,
 *    GPU r stores weights 2r and 2r+1;
 *  - same page, sections 先把账对齐 / ZeRO-1 / ZeRO-2 / "28 GB 是怎么来的":
 *    7B parameters on 4 GPUs hold 112 / 49 / 38.5 / 28 GB of model states;
 *  - same page, communication sections: 21 GB (stages 0-2) and 31.5 GB
 *    (stage 3) sent per card for 7B on 4 GPUs with 2-byte elements.
 * Prints "ok" and exits 0 when every check holds; otherwise names the first
 * failed check and exits 1. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "zero3.h"

static int failures = 0;

static void check(int cond, const char* what) {
    if (!cond && failures++ == 0) printf("FAILED: %s\n", what);
}

static int close_to(double a, double b) { return fabs(a - b) <= 1e-9 * fabs(b); }

int main(void) {
    /* eight weights of one layer, nothing persistent, four ranks */
    const int64_t layer[1] = {8};
    zero3_plan* plan = NULL;
    check(zero3_partition(layer, NULL, 1, 4, 0, 500000000, &plan) == ZERO3_OK && plan != NULL,
          "partition of the eight-weight layer");
    if (plan) {
        zero3_plan_info info;
        memset(&info, 0, sizeof info);
        check(zero3_plan_info_get(plan, &info) == ZERO3_OK, "plan info");
        check(info.n_ranks == 4 && info.psi_p == 8 && info.psi_pad == 8 && info.shard_len == 2 &&
                  info.psi_s == 0 && info.n_partitioned == 1 && info.n_persistent == 0,
              "eight weights on four ranks: two per rank, no padding");
        zero3_tensor_info t;
        check(zero3_plan_tensor(plan, 0, &t) == ZERO3_OK && t.first_rank == 0 &&
                  t.last_rank == 3 && t.n_segments == 4 && t.persistent == 0,
              "the layer spans all four ranks");
        zero3_segment seg[4];
        int64_t n = 0;
        check(zero3_plan_segments(plan, 0, seg, 4, &n) == ZERO3_OK && n == 4, "four segments");
        for (int r = 0; r < 4 && n == 4; ++r)
            check(seg[r].rank == r && seg[r].shard_off == 0 && seg[r].tensor_off == 2 * r &&
                      seg[r].len == 2,
                  "rank r stores weights 2r and 2r+1");
        check(zero3_plan_tensor(plan, 1, &t) == ZERO3_EINVAL, "tensor index out of range");
        zero3_plan_destroy(plan);
        plan = NULL;
    }

    /* a bias below the persistence threshold stays whole on every rank */
    const int64_t mlp[3] = {1000, 10, 3000};
    check(zero3_partition(mlp, NULL, 3, 3, 100, 500000000, &plan) == ZERO3_OK, "partition mlp");
    if (plan) {
        zero3_plan_info info;
        zero3_tensor_info t;
        check(zero3_plan_info_get(plan, &info) == ZERO3_OK && info.psi_p == 4000 &&
                  info.psi_pad == 4002 && info.shard_len == 1334 && info.psi_s == 10 &&
                  info.n_persistent == 1,
              "padding to a multiple of N_d and one persistent tensor");
        check(zero3_plan_tensor(plan, 1, &t) == ZERO3_OK && t.persistent == 1 && t.offset == 0 &&
                  t.first_rank == -1,
              "the bias is persistent");
        check(zero3_plan_tensor(plan, 2, &t) == ZERO3_OK && t.persistent == 0 &&
                  t.offset == 1000 && t.first_rank == 0 && t.last_rank == 2,
              "the second weight follows the first in the flat buffer");
        zero3_plan_destroy(plan);
        plan = NULL;
    }

    /* model-state accounting, 7B on four GPUs */
    const double gb[4] = {112e9, 49e9, 38.5e9, 28e9};
    for (int stage = 0; stage < 4; ++stage) {
        double b = 0;
        check(zero3_memory_bytes(stage, 7e9, 4, &b) == ZERO3_OK && close_to(b, gb[stage]),
              "7B on four GPUs: 112 / 49 / 38.5 / 28 GB");
    }
    double e2 = 0, e3 = 0;
    check(zero3_comm_elems(2, 7e9, 4, &e2) == ZERO3_OK && close_to(2.0 * e2, 21e9),
          "stage 2 sends 21 GB per card");
    check(zero3_comm_elems(3, 7e9, 4, &e3) == ZERO3_OK && close_to(2.0 * e3, 31.5e9),
          "stage 3 sends 31.5 GB per card");

    /* argument checks and status text */
    check(zero3_partition(NULL, NULL, 1, 4, 0, 1, &plan) == ZERO3_EINVAL, "NULL numels");
    check(zero3_partition(layer, NULL, 1, 0, 0, 1, &plan) == ZERO3_EINVAL, "zero ranks");
    check(zero3_memory_bytes(4, 7e9, 4, &e2) == ZERO3_EINVAL, "stage 4 does not exist");
    const char* s = zero3_status_string(ZERO3_EINVAL);
    check(s != NULL && strlen(s) > 0, "status text");
    zero3_plan_destroy(NULL);

    if (failures == 0) printf("ok\n");
    return failures == 0 ? 0 : 1;
}
