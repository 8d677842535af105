/* Plain-C client of libgdr: the header compiles as C11 and the entry points
 * link with C linkage.  Host-side calls only (no device needed): version,
 * chunk count, plan, workspace sizes, and an argument error with its message.
 * Prints "ok" and returns 0 when every check holds. */
#include <stdio.h>
#include <string.h>

#include "gdr.h"

#define CHECK(c)                                                   \
    do {                                                           \
        if (!(c)) {                                                \
            fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #c); \
            return 1;                                              \
        }                                                          \
    } while (0)

int main(void) {
    CHECK(strstr(gdr_version(), "sm_103a") != NULL);

    gdr_shape s;
    memset(&s, 0, sizeof(s));
    s.B = 1; s.T = 8192; s.Hq = 4; s.Hv = 8; s.K = 128; s.V = 128;
    CHECK(gdr_num_chunks(&s) == 128);

    gdr_opts o;
    memset(&o, 0, sizeof(o));
    gdr_plan p;
    CHECK(gdr_get_plan(&s, GDR_BF16, &o, &p) == GDR_OK);
    CHECK(p.path == GDR_PATH_TC && p.n_chunks == 128 && p.n_segments > 1);
    CHECK(gdr_get_plan(&s, GDR_F32, NULL, &p) == GDR_OK && p.path == GDR_PATH_SIMT);
    CHECK(gdr_fwd_workspace_size(&s, &o) > 0);
    CHECK(gdr_bwd_workspace_size(&s, &o) > gdr_fwd_workspace_size(&s, &o));

    /* varlen: three sequences packed along T */
    int cu[4] = {0, 100, 100, 1000};
    gdr_shape v = s;
    v.T = 1000; v.n_seqs = 3; v.cu_seqlens = cu; v.cu_seqlens_host = cu;
    CHECK(gdr_num_chunks(&v) == 2 + 0 + 15);

    /* an argument error: Hv not a multiple of Hq */
    gdr_shape bad = s;
    bad.Hq = 3;
    CHECK(gdr_get_plan(&bad, GDR_BF16, &o, &p) == GDR_ERR_SHAPE);
    CHECK(strlen(gdr_last_error()) > 0);
    CHECK(gdr_fwd_workspace_size(&bad, &o) == 0);
    printf("ok\n");
    return 0;
}
