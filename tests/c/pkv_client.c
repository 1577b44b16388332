/*
 * A plain C99 client of libpagedattn: it includes only include/pagedattn.h
 * (plus the CUDA runtime for device memory in "gpu" mode) and calls the C ABI
 * directly, so the header compiles as C and the exported calls work without
 * any binding layer.
 *
 *   pkv_client host
 *       host-side calls only (no GPU needed): version, error and status
 *       strings, workspace size queries, and the argument checks of the four
 *       operations, which must return their error codes before touching a GPU.
 *
 *   pkv_client gpu DIR
 *       reads the inputs of a small decode step from DIR (raw little-endian
 *       files written by the test), runs kv_store, paged_decode and sample
 *       through the C ABI on the current GPU, and writes the updated cache,
 *       the attention output and the token ids back to DIR for the test to
 *       compare with the oracle.
 *
 * Exit status 0 on success; every failed check prints one line.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "pagedattn.h"

static int failures = 0;

#define CHECK(cond)                                                        \
    do {                                                                   \
        if (!(cond)) {                                                     \
            fprintf(stderr, "%s:%d: check failed: %s\n", __FILE__, __LINE__, #cond); \
            ++failures;                                                    \
        }                                                                  \
    } while (0)

static int host_checks(void) {
    pkv_cache_desc c = {610, 256, 8, 128};
    CHECK(pkv_version() >= 100);
    CHECK(strcmp(pkv_error_string(PKV_OK), "ok") == 0);
    CHECK(strstr(pkv_error_string(PKV_ERR_NULL_POINTER), "null") != NULL);
    CHECK(strcmp(pkv_status_string(0), "ok") == 0);
    CHECK(strstr(pkv_status_string(PKV_STATUS_SLOT_OUT_OF_RANGE), "slot") != NULL);
    CHECK(pkv_paged_decode_workspace_bytes(64, 16, 4096, c) > 0);
    CHECK(pkv_paged_decode_workspace_bytes(64, 16, 4096, c) ==
          pkv_paged_decode_workspace_bytes(64, 16, 4096, c));
    CHECK(pkv_paged_prefill_workspace_bytes(16, 16384, 32, c) > 0);
    CHECK(pkv_set_wait_poll_limit(PKV_DEFAULT_WAIT_POLLS) == PKV_OK);
    /* argument errors come back before anything is enqueued */
    CHECK(pkv_kv_store(NULL, NULL, NULL, NULL, NULL, 4, c, NULL, NULL) == PKV_ERR_NULL_POINTER);
    CHECK(pkv_kv_store(NULL, NULL, NULL, NULL, NULL, -1, c, NULL, NULL) == PKV_ERR_BAD_DIMENSION);
    CHECK(pkv_kv_store(NULL, NULL, NULL, NULL, NULL, 0, c, NULL, NULL) == PKV_OK);
    CHECK(pkv_paged_decode(NULL, NULL, NULL, NULL, 16, NULL, 4, 16, 4096, 0.1f, NULL, NULL, 0, c,
                           NULL, NULL) == PKV_ERR_NULL_POINTER);
    {
        pkv_cache_desc bad = {610, 256, 8, 96};
        CHECK(pkv_paged_decode(NULL, NULL, NULL, NULL, 16, NULL, 4, 16, 4096, 0.1f, NULL, NULL,
                               0, bad, NULL, NULL) == PKV_ERR_UNSUPPORTED_HEAD_DIM);
    }
    CHECK(pkv_paged_prefill_varlen(NULL, NULL, NULL, NULL, NULL, NULL, NULL, 2, 10, 5, 5, 16,
                                   NULL, 0, 0.1f, NULL, NULL, 0, c, NULL, NULL) ==
          PKV_ERR_NULL_POINTER);
    CHECK(pkv_sample(NULL, NULL, NULL, 2, 1000, NULL, NULL, NULL) == PKV_ERR_NULL_POINTER);
    CHECK(pkv_sample(NULL, NULL, NULL, 2, 0, NULL, NULL, NULL) == PKV_ERR_BAD_DIMENSION);
    {
        const void *kc = NULL, *vc = NULL;
        const char* pool = (const char*)0x100000;
        CHECK(pkv_layer_cache(pool, 4, 2, c, &kc, &vc) == PKV_OK);
        const size_t layer = (size_t)c.num_blocks * c.block_size * c.num_kv_heads * c.head_dim * 2;
        CHECK((const char*)kc == pool + 2 * layer);
        CHECK((const char*)vc == pool + (4 + 2) * layer);
    }
    return failures;
}

#ifdef PKV_CLIENT_GPU
#include <cuda_runtime_api.h>

static void* read_file(const char* dir, const char* name, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE* f = fopen(path, "rb");
    if (!f) {
        fprintf(stderr, "cannot open %s\n", path);
        exit(2);
    }
    void* p = malloc(bytes);
    if (fread(p, 1, bytes, f) != bytes) {
        fprintf(stderr, "short read of %s\n", path);
        exit(2);
    }
    fclose(f);
    return p;
}

static void write_file(const char* dir, const char* name, const void* p, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE* f = fopen(path, "wb");
    if (!f || fwrite(p, 1, bytes, f) != bytes) {
        fprintf(stderr, "cannot write %s\n", path);
        exit(2);
    }
    fclose(f);
}

static void* to_device(const void* h, size_t bytes) {
    void* d = NULL;
    if (cudaMalloc(&d, bytes) != cudaSuccess || cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice) != cudaSuccess) {
        fprintf(stderr, "device copy of %zu bytes failed\n", bytes);
        exit(2);
    }
    return d;
}

/* sizes.txt: NB bs Hkv D B Hq MB max_ctx vocab, then scale */
static int gpu_step(const char* dir) {
    int NB, bs, Hkv, D, B, Hq, MB, max_ctx, V;
    float scale;
    char path[4096];
    snprintf(path, sizeof path, "%s/sizes.txt", dir);
    FILE* f = fopen(path, "r");
    if (!f || fscanf(f, "%d %d %d %d %d %d %d %d %d %f", &NB, &bs, &Hkv, &D, &B, &Hq, &MB,
                     &max_ctx, &V, &scale) != 10) {
        fprintf(stderr, "bad %s\n", path);
        return 2;
    }
    fclose(f);
    pkv_cache_desc c = {NB, bs, Hkv, D};
    const size_t cache_b = (size_t)NB * bs * Hkv * D * 2, row_b = (size_t)Hkv * D * 2;
    void* kc = to_device(read_file(dir, "k_cache.bin", cache_b), cache_b);
    void* vc = to_device(read_file(dir, "v_cache.bin", cache_b), cache_b);
    void* kn = to_device(read_file(dir, "k_new.bin", B * row_b), B * row_b);
    void* vn = to_device(read_file(dir, "v_new.bin", B * row_b), B * row_b);
    void* slots = to_device(read_file(dir, "slots.bin", B * 4), B * 4);
    void* q = to_device(read_file(dir, "q.bin", (size_t)B * Hq * D * 2), (size_t)B * Hq * D * 2);
    void* bt = to_device(read_file(dir, "block_tables.bin", (size_t)B * MB * 4), (size_t)B * MB * 4);
    void* ctx = to_device(read_file(dir, "context_lens.bin", B * 4), B * 4);
    void* lg = to_device(read_file(dir, "logits.bin", (size_t)B * V * 4), (size_t)B * V * 4);
    void* tp = to_device(read_file(dir, "temperatures.bin", B * 4), B * 4);
    void* en = to_device(read_file(dir, "noise.bin", (size_t)B * V * 4), (size_t)B * V * 4);
    void *out = NULL, *ws = NULL, *ids = NULL, *status = NULL;
    const size_t ws_b = pkv_paged_decode_workspace_bytes(B, Hq, max_ctx, c);
    CHECK(cudaMalloc(&out, (size_t)B * Hq * D * 2) == cudaSuccess);
    CHECK(cudaMalloc(&ws, ws_b) == cudaSuccess);
    CHECK(cudaMalloc(&ids, B * 4) == cudaSuccess);
    CHECK(cudaMalloc(&status, 4) == cudaSuccess);
    CHECK(cudaMemset(status, 0, 4) == cudaSuccess);
    /* the step: store the new token's K/V, attend, sample (stream NULL) */
    CHECK(pkv_kv_store(kn, vn, kc, vc, (const int32_t*)slots, B, c, (uint32_t*)status, NULL) ==
          PKV_OK);
    CHECK(pkv_paged_decode(q, kc, vc, (const int32_t*)bt, MB, (const int32_t*)ctx, B, Hq,
                           max_ctx, scale, out, ws, ws_b, c, (uint32_t*)status, NULL) == PKV_OK);
    CHECK(pkv_sample((const float*)lg, (const float*)tp, (const float*)en, B, V,
                     (int32_t*)ids, (uint32_t*)status, NULL) == PKV_OK);
    CHECK(cudaDeviceSynchronize() == cudaSuccess);
    uint32_t st = 0;
    CHECK(cudaMemcpy(&st, status, 4, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(st == 0);
    void* h = malloc(cache_b);
    CHECK(cudaMemcpy(h, kc, cache_b, cudaMemcpyDeviceToHost) == cudaSuccess);
    write_file(dir, "k_cache_out.bin", h, cache_b);
    CHECK(cudaMemcpy(h, vc, cache_b, cudaMemcpyDeviceToHost) == cudaSuccess);
    write_file(dir, "v_cache_out.bin", h, cache_b);
    CHECK(cudaMemcpy(h, out, (size_t)B * Hq * D * 2, cudaMemcpyDeviceToHost) == cudaSuccess);
    write_file(dir, "out.bin", h, (size_t)B * Hq * D * 2);
    CHECK(cudaMemcpy(h, ids, B * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
    write_file(dir, "ids.bin", h, B * 4);
    free(h);
    return failures;
}
#endif

int main(int argc, char** argv) {
    if (argc >= 2 && strcmp(argv[1], "host") == 0) return host_checks() ? 1 : 0;
#ifdef PKV_CLIENT_GPU
    if (argc >= 3 && strcmp(argv[1], "gpu") == 0) return gpu_step(argv[2]) ? 1 : 0;
#endif
    fprintf(stderr, "usage: %s host | gpu DIR\n", argv[0]);
    return 2;
}
