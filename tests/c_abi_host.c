/*
 * A plain C99 caller of the library's host-only entry points: the header must
 * compile as C and the shared library must link and run without a GPU.
 * Prints "OK" and exits 0 when every check holds; otherwise prints the failed
 * check and exits 1.
 *
 * Expected values:
 *   - product counts of one NS update of a 2560 x 9728 matrix ("MuonX" page,
 *     section 3.2: 1.443 -> 1.134 TFLOPs), here as the closed forms
 *     20 m^2 n + 10 m^3 (plain) and 12 m^2 n + 22 m^3 (Gram 2+2+1);
 *   - a packed layout worked by hand: shapes 2x3, 1x5, 3x1 with owners
 *     1, 0, 1 on two ranks and 4-element alignment.  Rank 0 holds matrix 1
 *     at 0 (5 elements, 8 with alignment); rank 1 holds matrix 0 at 0
 *     (6, padded to 8) and matrix 2 at 8 (ends at 11, 12 with alignment).
 *     Segments are 12 long, so the offsets are 12 + 0, 0, 12 + 8.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "muon.h"

static int failures = 0;

#define CHECK(cond)                                                    \
    do {                                                               \
        if (!(cond)) {                                                 \
            printf("FAILED line %d: %s\n", __LINE__, #cond);           \
            ++failures;                                                \
        }                                                              \
    } while (0)

int main(void) {
    /* status strings: every code has a non-empty name */
    int codes[] = {MUON_OK, MUON_EINVAL, MUON_EDTYPE, MUON_ENOMEM, MUON_ECUDA, MUON_ENONFINITE,
                   MUON_ETIMEOUT, MUON_ENOTSUP};
    for (unsigned i = 0; i < sizeof codes / sizeof codes[0]; ++i) {
        const char* s = muon_status_str(codes[i]);
        CHECK(s != NULL && s[0] != '\0');
    }

    /* product counts */
    {
        const double m = 2560.0, n = 9728.0;
        int seg[3] = {2, 2, 1};
        double nominal = 0.0, alg = 0.0;
        CHECK(muon_ns_flops(2560, 9728, MUON_PATH_PLAIN, NULL, 0, &nominal, &alg) == MUON_OK);
        CHECK(nominal == 20.0 * m * m * n + 10.0 * m * m * m);
        CHECK(muon_ns_flops(2560, 9728, MUON_PATH_GRAM, seg, 3, &nominal, &alg) == MUON_OK);
        CHECK(nominal == 12.0 * m * m * n + 22.0 * m * m * m);
        CHECK(alg < nominal);
        /* the tall shape is oriented first: same counts */
        double nominal_t = 0.0, alg_t = 0.0;
        CHECK(muon_ns_flops(9728, 2560, MUON_PATH_GRAM, seg, 3, &nominal_t, &alg_t) == MUON_OK);
        CHECK(nominal_t == nominal && alg_t == alg);
    }

    /* owner placement: every matrix placed, loads add up, makespan is the largest */
    {
        int64_t ms[5] = {2048, 8192, 2048, 128, 1024};
        int64_t ns[5] = {2048, 2048, 8192, 512, 4096};
        int owner[5];
        double load[3], makespan = -1.0;
        int measured = -1;
        CHECK(muon_owner_plan(ms, ns, 5, MUON_BF16, 3, owner, load, &makespan, &measured) == MUON_OK);
        double sum = 0.0, mx = 0.0;
        for (int r = 0; r < 3; ++r) {
            sum += load[r];
            if (load[r] > mx) mx = load[r];
        }
        for (int i = 0; i < 5; ++i) CHECK(owner[i] >= 0 && owner[i] < 3);
        CHECK(makespan == mx);
        CHECK(sum > 0.0);
        CHECK(measured == 0 || measured == 1);
    }

    /* packed layout worked by hand */
    {
        int64_t ms[3] = {2, 1, 3};
        int64_t ns[3] = {3, 5, 1};
        int owner[3] = {1, 0, 1};
        int64_t off[3] = {-1, -1, -1}, seg = -1;
        CHECK(muon_pack_plan(ms, ns, owner, 3, 2, 4, off, &seg) == MUON_OK);
        CHECK(seg == 12);
        CHECK(off[0] == 12 && off[1] == 0 && off[2] == 20);

        /* an owner out of range is rejected with a message */
        owner[2] = 2;
        CHECK(muon_pack_plan(ms, ns, owner, 3, 2, 4, off, &seg) == MUON_EINVAL);
        const char* msg = muon_last_error_message();
        CHECK(msg != NULL && strlen(msg) > 0);
    }

    if (failures) return 1;
    printf("OK\n");
    return 0;
}
