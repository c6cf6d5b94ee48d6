/* A plain C99 caller of the library: plans the layout of a small unit on the
 * host (no GPU needed), checks the FLAT floor boundaries, and prints one line
 * per segment.  Built and run by tests/test_abi_c.py. */
#include <stdio.h>
#include <stdlib.h>

#include "fsdp_unit.h"

int main(void) {
    const int ndims[2] = {2, 1};
    const int64_t dims[3] = {64, 48, 64};   /* Linear W[64x48] + b[64] */
    int64_t P = 0, nsegs = 0;
    int rc = fsdp_plan_layout(2, ndims, dims, FSDP_LAYOUT_FLAT, 4, &P, &nsegs, NULL, 0);
    if (rc != FSDP_OK) {
        printf("error %d %s: %s\n", rc, fsdp_strerror(rc), fsdp_last_error());
        return 1;
    }
    fsdp_segment* segs = (fsdp_segment*)malloc(sizeof(fsdp_segment) * (size_t)nsegs);
    rc = fsdp_plan_layout(2, ndims, dims, FSDP_LAYOUT_FLAT, 4, &P, &nsegs, segs, nsegs);
    if (rc != FSDP_OK) return 2;
    printf("P=%lld segments=%lld\n", (long long)P, (long long)nsegs);
    for (int64_t i = 0; i < nsegs; ++i)
        printf("rank=%d global=%lld len=%lld arena=%lld\n", segs[i].rank, (long long)segs[i].global_off,
               (long long)segs[i].len, (long long)segs[i].arena_off);
    rc = fsdp_plan_layout(2, ndims, dims, FSDP_LAYOUT_FLAT, 0, &P, &nsegs, NULL, 0);
    printf("N=0 -> %s\n", fsdp_strerror(rc));
    free(segs);
    return 0;
}
