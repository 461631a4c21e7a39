/*
 * c_abi_check.c -- a plain C consumer of libhalo.so (include/halo.h and
 * include/stencil.h): no Python, no PyTorch, device memory from the CUDA
 * runtime.  Built and run by tests/test_c_abi_consumer.py on a GPU.
 *
 * It builds a plan for a seeded random system (two pulses in z, one in y and
 * x), runs the coordinate exchange and the force reduction in all three modes
 * and checks what holds without an oracle:
 *   - the three modes give bit-identical coordinates and forces;
 *   - every halo coordinate equals its owner's coordinate plus 0 or one box
 *     length per component (the slot's owner from halo_local_to_global);
 *   - with integer-valued forces the total force is conserved exactly and
 *     halo_store_home returns every atom's force in input order;
 *   - the sharded data plane (4 z-slab shards, one buffer each) gives the
 *     same coordinates and forces, shard by shard;
 *   - halo_status reports no device error; bad arguments are refused;
 *   - one fused stencil iteration equals a sweep followed by an exchange.
 * Prints "c abi ok" and returns 0 on success.
 */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "halo.h"
#include "stencil.h"

#define CHECK(cond, msg)                                   \
    do {                                                   \
        if (!(cond)) {                                     \
            fprintf(stderr, "FAILED: %s (line %d)\n", msg, __LINE__); \
            return 1;                                      \
        }                                                  \
    } while (0)
#define CU(call) CHECK((call) == cudaSuccess, #call)
#define HL(call) CHECK((call) == HALO_OK, #call)

static uint64_t lcg_state = 12345u;
static double lcg01(void) {
    lcg_state = lcg_state * 6364136223846793005ull + 1442695040888963407ull;
    return (double)(lcg_state >> 11) * (1.0 / 9007199254740992.0);
}

static int run_modes(void) {
    const float box[3] = {6.2f, 6.2f, 6.2f};
    const int32_t grid[3] = {2, 4, 8};
    const float rc = 1.2f;
    const int64_t n = 24000;
    float* xyz = (float*)malloc(sizeof(float) * 3 * n);
    int32_t* dom = (int32_t*)malloc(sizeof(int32_t) * n);
    for (int64_t a = 0; a < n; a++) {
        int c[3];
        for (int d = 0; d < 3; d++) {
            float v = (float)(lcg01() * box[d]);
            if (v >= box[d]) v = 0.0f;
            xyz[3 * a + d] = v;
            c[d] = (int)floor((double)v * grid[d] / box[d]);
            if (c[d] > grid[d] - 1) c[d] = grid[d] - 1;
        }
        dom[a] = c[0] + grid[0] * (c[1] + grid[1] * c[2]);
    }
    float* d_xyz;
    int32_t* d_dom;
    CU(cudaMalloc((void**)&d_xyz, sizeof(float) * 3 * n));
    CU(cudaMalloc((void**)&d_dom, sizeof(int32_t) * n));
    CU(cudaMemcpy(d_xyz, xyz, sizeof(float) * 3 * n, cudaMemcpyHostToDevice));
    CU(cudaMemcpy(d_dom, dom, sizeof(int32_t) * n, cudaMemcpyHostToDevice));

    halo_plan* plan = NULL;
    HL(halo_setup(box, grid, rc, d_xyz, d_dom, n, NULL, &plan));
    halo_info info;
    HL(halo_query(plan, &info));
    CHECK(info.n_pulses == 4 && info.n_atoms == n, "pulse structure");
    const int64_t nl = info.n_local_total;

    /* bad arguments are refused without touching the GPU */
    CHECK(halo_exchange_x(plan, NULL, NULL) == HALO_EINVAL, "null field");
    CHECK(halo_set_mode(plan, 7, NULL) == HALO_EINVAL, "bad mode");

    float* d_loc;
    float* d_f;
    float* d_out;
    int32_t* d_gid;
    CU(cudaMalloc((void**)&d_loc, sizeof(float) * 3 * nl));
    CU(cudaMalloc((void**)&d_f, sizeof(float) * 3 * nl));
    CU(cudaMalloc((void**)&d_out, sizeof(float) * 3 * n));
    CU(cudaMalloc((void**)&d_gid, sizeof(int32_t) * nl));
    float* f0 = (float*)malloc(sizeof(float) * 3 * nl);
    for (int64_t i = 0; i < 3 * nl; i++) f0[i] = (float)((int)(lcg01() * 17.0) - 8);
    enum { NM = 4 };
    float* loc[NM];
    float* fr[NM];
    const int32_t modes[NM] = {HALO_MODE_FUSED, HALO_MODE_STEPWISE, HALO_MODE_FLAT, HALO_MODE_STAGED};
    for (int m = 0; m < NM; m++) {
        HL(halo_set_mode(plan, modes[m], NULL));
        HL(halo_load_home(plan, d_xyz, d_loc, NULL));
        HL(halo_exchange_x(plan, d_loc, NULL));
        CU(cudaMemcpy(d_f, f0, sizeof(float) * 3 * nl, cudaMemcpyHostToDevice));
        HL(halo_exchange_f(plan, d_f, NULL));
        CHECK(halo_status(plan, NULL) == HALO_OK, "device error");
        loc[m] = (float*)malloc(sizeof(float) * 3 * nl);
        fr[m] = (float*)malloc(sizeof(float) * 3 * nl);
        CU(cudaMemcpy(loc[m], d_loc, sizeof(float) * 3 * nl, cudaMemcpyDeviceToHost));
        CU(cudaMemcpy(fr[m], d_f, sizeof(float) * 3 * nl, cudaMemcpyDeviceToHost));
    }
    for (int m = 1; m < NM; m++) {
        CHECK(memcmp(loc[0], loc[m], sizeof(float) * 3 * nl) == 0, "coordinates differ between modes");
        CHECK(memcmp(fr[0], fr[m], sizeof(float) * 3 * nl) == 0, "forces differ between modes");
    }

    /* the sharded data plane: 4 shards, each its own buffer, laid out as its
       part of the dense array */
    {
        enum { NS = 4 };
        HL(halo_shard(plan, NS, NULL));
        CHECK(halo_shard(plan, 9, NULL) == HALO_EINVAL, "shard count");
        float* sx[NS];
        float* sf[NS];
        int64_t first[NS], cnt[NS], tot = 0;
        for (int k = 0; k < NS; k++) {
            int32_t fd, ndom;
            HL(halo_shard_layout(plan, k, &fd, &ndom, &first[k], &cnt[k]));
            CHECK(first[k] == tot && ndom == 16 && fd == 16 * k, "shard layout");
            tot += cnt[k];
            CU(cudaMalloc((void**)&sx[k], sizeof(float) * 3 * (cnt[k] > 0 ? cnt[k] : 1)));
            CU(cudaMalloc((void**)&sf[k], sizeof(float) * 3 * (cnt[k] > 0 ? cnt[k] : 1)));
            CU(cudaMemcpy(sf[k], f0 + 3 * first[k], sizeof(float) * 3 * cnt[k], cudaMemcpyHostToDevice));
        }
        CHECK(tot == nl, "shards tile the local layout");
        HL(halo_load_home_sharded(plan, d_xyz, sx, NULL));
        HL(halo_exchange_x_sharded(plan, sx, NULL));
        HL(halo_exchange_f_sharded(plan, sf, NULL));
        CHECK(halo_status(plan, NULL) == HALO_OK, "device error (sharded)");
        float* hx = (float*)malloc(sizeof(float) * 3 * nl);
        float* hf = (float*)malloc(sizeof(float) * 3 * nl);
        for (int k = 0; k < NS; k++) {
            CU(cudaMemcpy(hx + 3 * first[k], sx[k], sizeof(float) * 3 * cnt[k], cudaMemcpyDeviceToHost));
            CU(cudaMemcpy(hf + 3 * first[k], sf[k], sizeof(float) * 3 * cnt[k], cudaMemcpyDeviceToHost));
            CU(cudaFree(sx[k]));
            CU(cudaFree(sf[k]));
        }
        CHECK(memcmp(hx, loc[0], sizeof(float) * 3 * nl) == 0, "sharded coordinates differ");
        CHECK(memcmp(hf, fr[0], sizeof(float) * 3 * nl) == 0, "sharded forces differ");
        free(hx);
        free(hf);
    }

    /* halo coordinates = owner + 0 or L per component */
    int32_t* gid = (int32_t*)malloc(sizeof(int32_t) * nl);
    HL(halo_local_to_global(plan, d_gid, NULL));
    CU(cudaMemcpy(gid, d_gid, sizeof(int32_t) * nl, cudaMemcpyDeviceToHost));
    for (int64_t i = 0; i < nl; i++) {
        CHECK(gid[i] >= 0 && gid[i] < n, "owner id");
        for (int d = 0; d < 3; d++) {
            const float own = xyz[3 * (int64_t)gid[i] + d], got = loc[0][3 * i + d];
            CHECK(got == own || got == own + box[d], "halo coordinate is not an image of its owner");
        }
    }

    /* integer forces: per-atom totals through halo_store_home, exact */
    HL(halo_store_home(plan, d_f, d_out, NULL));
    float* out = (float*)malloc(sizeof(float) * 3 * n);
    CU(cudaMemcpy(out, d_out, sizeof(float) * 3 * n, cudaMemcpyDeviceToHost));
    double* want = (double*)calloc((size_t)3 * n, sizeof(double));
    for (int64_t i = 0; i < nl; i++)
        for (int d = 0; d < 3; d++) want[3 * (int64_t)gid[i] + d] += f0[3 * i + d];
    for (int64_t i = 0; i < 3 * n; i++) CHECK((double)out[i] == want[i], "per-atom force");

    halo_destroy(plan);
    for (int m = 0; m < NM; m++) {
        free(loc[m]);
        free(fr[m]);
    }
    free(want);
    free(out);
    free(gid);
    free(f0);
    free(xyz);
    free(dom);
    CU(cudaFree(d_xyz));
    CU(cudaFree(d_dom));
    CU(cudaFree(d_loc));
    CU(cudaFree(d_f));
    CU(cudaFree(d_out));
    CU(cudaFree(d_gid));
    return 0;
}

static int run_stencil(void) {
    stencil_plan* sp = NULL;
    CHECK(stencil_setup(2, 2, 6, &sp) == HALO_EINVAL, "n must be a multiple of 4");
    HL(stencil_setup(3, 2, 64, &sp));
    int64_t total = 0;
    HL(stencil_layout(sp, NULL, NULL, NULL, NULL, &total));
    float* h = (float*)malloc(sizeof(float) * total);
    for (int64_t i = 0; i < total; i++) h[i] = (float)lcg01();
    float *a, *b, *c;
    CU(cudaMalloc((void**)&a, sizeof(float) * total));
    CU(cudaMalloc((void**)&b, sizeof(float) * total));
    CU(cudaMalloc((void**)&c, sizeof(float) * total));
    CU(cudaMemcpy(a, h, sizeof(float) * total, cudaMemcpyHostToDevice));
    CU(cudaMemcpy(b, h, sizeof(float) * total, cudaMemcpyHostToDevice));
    CU(cudaMemcpy(c, h, sizeof(float) * total, cudaMemcpyHostToDevice));
    HL(stencil_exchange(sp, a, NULL));
    HL(stencil_sweep(sp, a, b, NULL));
    HL(stencil_exchange(sp, b, NULL));
    HL(stencil_sweep_fused(sp, a, c, NULL));
    CU(cudaDeviceSynchronize());
    float* hb = (float*)malloc(sizeof(float) * total);
    float* hc = (float*)malloc(sizeof(float) * total);
    CU(cudaMemcpy(hb, b, sizeof(float) * total, cudaMemcpyDeviceToHost));
    CU(cudaMemcpy(hc, c, sizeof(float) * total, cudaMemcpyDeviceToHost));
    CHECK(memcmp(hb, hc, sizeof(float) * total) == 0, "fused stencil step differs from sweep + exchange");
    stencil_destroy(sp);
    free(h);
    free(hb);
    free(hc);
    CU(cudaFree(a));
    CU(cudaFree(b));
    CU(cudaFree(c));
    return 0;
}

int main(void) {
    if (run_modes() != 0) return 1;
    if (run_stencil() != 0) return 1;
    printf("c abi ok\n");
    return 0;
}
