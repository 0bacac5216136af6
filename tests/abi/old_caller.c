/* A caller compiled against the shorter, original parameter struct (the four
 * controls only). It must keep working with the current library: fields past
 * its struct_size take their defaults ("feat: prefetch streamed layers during
 * compute", Summary: the versioned struct and an executable built against the
 * previous public API). */
#include <stddef.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

typedef struct {
    uint32_t struct_size;
    uint32_t version;
    int32_t prefetch_depth;
    int32_t resident_layers;
    int64_t max_vram_bytes;
    int32_t use_pool;
} old_params;

typedef struct {
    int32_t run, step, kind, segment, slot, reserved;
    int64_t bytes;
} old_event;

typedef struct ls_ctx ls_ctx;
int32_t ls_ctx_create(const old_params* p, ls_ctx** out);
void ls_ctx_destroy(ls_ctx* c);
int32_t ls_simulate(const old_params* p, const int64_t* seg, int32_t n, const int64_t* sb, const int32_t* sid,
                    int32_t ns, int32_t runs, const int64_t* lb, old_event* ev, int64_t cap, int64_t* n_ev,
                    void* stats, int32_t* run_status);

int main(void) {
    old_params p;
    memset(&p, 0, sizeof(p));
    p.struct_size = (uint32_t)(offsetof(old_params, use_pool) + sizeof(int32_t));
    p.version = 1;
    p.prefetch_depth = 1;
    p.resident_layers = 0;
    p.max_vram_bytes = 2000;
    p.use_pool = 1;
    ls_ctx* c = 0;
    int32_t st = ls_ctx_create(&p, &c);
    if (st != 0 || !c) { printf("create %d\n", st); return 1; }
    ls_ctx_destroy(c);
    int64_t seg[4] = {1000, 1000, 1000, 1000};
    old_event ev[64];
    int64_t n = 0;
    int32_t rs[1];
    st = ls_simulate(&p, seg, 4, 0, 0, 0, 1, 0, ev, 64, &n, 0, rs);
    if (st != 0 || n != 8 || ev[0].kind != 3 || ev[0].slot != 0 || ev[1].slot != 1) {
        printf("simulate %d n=%lld\n", st, (long long)n);
        return 2;
    }
    p.struct_size = 8; /* smaller than the minimum: refused with LS_ERR_VERSION */
    st = ls_ctx_create(&p, &c);
    if (st != -2) { printf("undersized %d\n", st); return 3; }
    p.struct_size = (uint32_t)sizeof(old_params);
    p.version = 7;
    st = ls_ctx_create(&p, &c);
    if (st != -2) { printf("version %d\n", st); return 4; }
    printf("ok\n");
    return 0;
}
