/* A plain C user of liblazyattn: no Python, no torch. It drives the library
 * through include/lazyattn.h only, with device memory from the CUDA runtime,
 * the way a serving engine written in C or C++ would.
 *
 *   lazyattn_client host              host-only checks (entry packing, status
 *                                     strings, table size, argument validation)
 *   lazyattn_client run IN OUT        one request through the whole path:
 *                                     store documents, prefill, decode steps
 *
 * IN (little endian): int32 magic 0x4c415a59, dtype (0 fp32, 1 bf16), Hq, Hkv, D,
 * n_docs, q_len, n_steps; float64 rope_theta; int32 doc_len[n_docs]; then fp32
 * arrays: per document k, v [len][Hkv][D]; q [q_len][Hq][D]; k, v [q_len][Hkv][D];
 * per decode step q [Hq][D], k [Hkv][D], v [Hkv][D]. bf16 inputs must already be
 * bf16 values (the client keeps their top 16 bits).
 * OUT: fp32 prefill output [q_len][Hq][D], then per step the decode output [Hq][D].
 * Documents sit back to back from logical position 0, the query segment after
 * them, generated tokens after the query segment. Exit status 0 on success.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "lazyattn.h"

#define FAIL(...)                     \
    do {                              \
        fprintf(stderr, __VA_ARGS__); \
        fputc('\n', stderr);          \
        exit(1);                      \
    } while (0)
#define CHECK(call)                                                                           \
    do {                                                                                      \
        int rc_ = (call);                                                                     \
        if (rc_ != LAZYATTN_OK) FAIL("%s failed: %s", #call, lazyattn_status_string(rc_)); \
    } while (0)
#define CUDA(call)                                                                      \
    do {                                                                                \
        cudaError_t e_ = (call);                                                        \
        if (e_ != cudaSuccess) FAIL("%s failed: %s", #call, cudaGetErrorString(e_));   \
    } while (0)

static int host_checks(void) {
    /* entry packing: the documented bit layout */
    uint64_t e = lazyattn_pack_entry(123456, 5000000, 16, 1);
    if ((uint32_t)(e & 0xffffffffu) != 123456u || ((e >> 32) & ((1u << 26) - 1)) != 5000000u ||
        ((e >> 58) & 0x1f) != 16u || (e >> 63) != 1u)
        FAIL("pack_entry layout");
    if (lazyattn_pack_entry(7, 0, 0, 0) != 7u) FAIL("pack_entry of an empty entry");
    /* status strings are never NULL */
    for (int s = 1; s >= -9; --s)
        if (!lazyattn_status_string(s)) FAIL("status string %d", s);
    /* (cos, sin) rows, then the same rows paired for two-lane arithmetic */
    if (lazyattn_rope_table_bytes(128, 1000) != (size_t)2 * 1000 * 64 * 8) FAIL("rope_table_bytes");
    /* invalid descriptors are rejected before any CUDA call */
    lazyattn_pool_desc d;
    memset(&d, 0, sizeof d);
    lazyattn_pool_t pool = NULL;
    if (lazyattn_pool_create(&d, NULL, &pool) != LAZYATTN_EINVAL || pool) FAIL("zero descriptor accepted");
    if (lazyattn_pool_create(NULL, NULL, &pool) != LAZYATTN_EINVAL) FAIL("NULL descriptor accepted");
    if (lazyattn_store_doc(NULL, NULL, NULL, 1, NULL, NULL, 0, NULL) != LAZYATTN_EINVAL) FAIL("NULL pool");
    /* block-table check: two requests, the second with two tokens at each of positions 10..12 */
    uint64_t ent[4] = {lazyattn_pack_entry(0, 0, 16, 0), lazyattn_pack_entry(1, 16, 5, 1),
                       lazyattn_pack_entry(0, 0, 16, 0), lazyattn_pack_entry(2, 10, 3, 1)};
    int32_t offs[3] = {0, 2, 4}, bad = 0;
    if (lazyattn_check_batch_host(ent, offs, 1, 8, 64, &bad) != LAZYATTN_OK || bad != -1) FAIL("valid table");
    if (lazyattn_check_batch_host(ent, offs, 2, 8, 64, &bad) != LAZYATTN_EINVAL || bad != 1) FAIL("overlap");
    if (lazyattn_check_batch_host(ent, offs, 2, 2, 64, &bad) != LAZYATTN_ERANGE || bad != 1) FAIL("page range");
    printf("host checks ok\n");
    return 0;
}

static void read_exact(FILE* f, void* p, size_t n) {
    if (fread(p, 1, n, f) != n) FAIL("short input file");
}

static float* read_f32(FILE* f, size_t n) {
    float* p = (float*)malloc(n * sizeof(float) + 1);
    if (!p) FAIL("out of host memory");
    read_exact(f, p, n * sizeof(float));
    return p;
}

/* device copy of n fp32 values in the pool dtype */
static void* to_device(const float* x, size_t n, int bf16) {
    void* d = NULL;
    size_t esz = bf16 ? 2 : 4;
    CUDA(cudaMalloc(&d, n * esz));
    if (bf16) {
        uint16_t* h = (uint16_t*)malloc(n * 2 + 1);
        if (!h) FAIL("out of host memory");
        for (size_t i = 0; i < n; ++i) {
            uint32_t u;
            memcpy(&u, &x[i], 4);
            h[i] = (uint16_t)(u >> 16);
        }
        CUDA(cudaMemcpy(d, h, n * 2, cudaMemcpyHostToDevice));
        free(h);
    } else {
        CUDA(cudaMemcpy(d, x, n * 4, cudaMemcpyHostToDevice));
    }
    return d;
}

static void from_device(float* x, const void* d, size_t n, int bf16) {
    if (bf16) {
        uint16_t* h = (uint16_t*)malloc(n * 2 + 1);
        if (!h) FAIL("out of host memory");
        CUDA(cudaMemcpy(h, d, n * 2, cudaMemcpyDeviceToHost));
        for (size_t i = 0; i < n; ++i) {
            uint32_t u = (uint32_t)h[i] << 16;
            memcpy(&x[i], &u, 4);
        }
        free(h);
    } else {
        CUDA(cudaMemcpy(x, d, n * 4, cudaMemcpyDeviceToHost));
    }
}

static int run(const char* in_path, const char* out_path) {
    FILE* f = fopen(in_path, "rb");
    if (!f) FAIL("cannot open %s", in_path);
    int32_t hdr[8];
    read_exact(f, hdr, sizeof hdr);
    if (hdr[0] != 0x4c415a59) FAIL("bad magic");
    const int bf16 = hdr[1], Hq = hdr[2], Hkv = hdr[3], D = hdr[4], n_docs = hdr[5], q_len = hdr[6],
              n_steps = hdr[7];
    double theta;
    read_exact(f, &theta, sizeof theta);
    if (n_docs < 0 || n_docs > 4096 || q_len < 1 || n_steps < 0 || Hq < 1 || Hkv < 1 || D < 1 || (bf16 & ~1))
        FAIL("bad header");
    int32_t* doc_len = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_docs + 1));
    read_exact(f, doc_len, sizeof(int32_t) * (size_t)n_docs);

    /* pool sized for every document, the query segment and the generated tokens */
    int64_t ctx = 0, pages = 0;
    for (int i = 0; i < n_docs; ++i) {
        ctx += doc_len[i];
        pages += (doc_len[i] + LAZYATTN_PAGE_SIZE - 1) / LAZYATTN_PAGE_SIZE;
    }
    const int q_pages = (q_len + LAZYATTN_PAGE_SIZE - 1) / LAZYATTN_PAGE_SIZE;
    const int free_tail = q_pages * LAZYATTN_PAGE_SIZE - q_len;
    const int dec_pages = n_steps > free_tail ? (n_steps - free_tail + LAZYATTN_PAGE_SIZE - 1) / LAZYATTN_PAGE_SIZE : 0;
    pages += q_pages + dec_pages;
    const int32_t max_position = (int32_t)(ctx + q_pages * LAZYATTN_PAGE_SIZE + dec_pages * LAZYATTN_PAGE_SIZE);
    const size_t esz = bf16 ? 2 : 4;
    const size_t page_bytes = (size_t)Hkv * LAZYATTN_PAGE_SIZE * (size_t)D * esz;

    lazyattn_pool_desc d;
    memset(&d, 0, sizeof d);
    d.num_pages = (int32_t)pages;
    d.page_size = LAZYATTN_PAGE_SIZE;
    d.n_q_heads = Hq;
    d.n_kv_heads = Hkv;
    d.head_dim = D;
    d.dtype = bf16 ? LAZYATTN_BF16 : LAZYATTN_F32;
    d.rope_theta = theta;
    d.max_position = max_position;
    CUDA(cudaMalloc(&d.k_pool, (size_t)pages * page_bytes));
    CUDA(cudaMalloc(&d.v_pool, (size_t)pages * page_bytes));
    CUDA(cudaMalloc(&d.rope_table, lazyattn_rope_table_bytes(D, max_position)));
    CUDA(cudaMalloc((void**)&d.status_word, sizeof(int32_t)));
    lazyattn_pool_t pool = NULL;
    CHECK(lazyattn_pool_create(&d, NULL, &pool));

    /* block table of the one request: documents, query segment, reserved pages */
    uint64_t* entries = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)(pages + 1));
    int32_t* page_ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)(pages + 1));
    int n_ent = 0;
    int64_t start = 0;
    const size_t nq = (size_t)q_len * Hq * D;
    void* q_dev = NULL;
    for (int i = 0; i <= n_docs; ++i) {   /* i == n_docs: the query segment */
        if (i == n_docs) {                 /* q precedes the segment's k, v in the file */
            float* q = read_f32(f, nq);
            q_dev = to_device(q, nq, bf16);
            free(q);
        }
        const int n = i < n_docs ? doc_len[i] : q_len;
        float* k = read_f32(f, (size_t)n * Hkv * D);
        float* v = read_f32(f, (size_t)n * Hkv * D);
        void* dk = to_device(k, (size_t)n * Hkv * D, bf16);
        void* dv = to_device(v, (size_t)n * Hkv * D, bf16);
        int32_t np = 0;
        CHECK(lazyattn_store_doc(pool, dk, dv, n, NULL, page_ids, (int32_t)pages, &np));
        CUDA(cudaDeviceSynchronize());
        CUDA(cudaFree(dk));
        CUDA(cudaFree(dv));
        for (int j = 0; j < np; ++j) {
            const int nv = n - 16 * j < 16 ? n - 16 * j : 16;
            entries[n_ent++] = lazyattn_pack_entry(page_ids[j], (int32_t)(start + 16 * j), nv, i == n_docs);
        }
        start += n;
        free(k);
        free(v);
    }
    if (dec_pages > 0) {
        CHECK(lazyattn_alloc_pages(pool, dec_pages, page_ids));
        for (int j = 0; j < dec_pages; ++j)
            entries[n_ent++] = lazyattn_pack_entry(page_ids[j], (int32_t)(ctx + (q_pages + j) * 16), 0, 1);
    }

    int32_t offs[2] = {0, n_ent}, q_offs[2] = {0, q_len}, q_start[1] = {(int32_t)ctx};
    lazyattn_batch b;
    memset(&b, 0, sizeof b);
    b.num_requests = 1;
    b.max_entries = n_ent;
    b.max_q_len = q_len;
    b.total_q = q_len;
    CUDA(cudaMalloc((void**)&b.entries, sizeof(uint64_t) * (size_t)n_ent));
    CUDA(cudaMemcpy(b.entries, entries, sizeof(uint64_t) * (size_t)n_ent, cudaMemcpyHostToDevice));
    CUDA(cudaMalloc((void**)&b.entry_offsets, sizeof offs));
    CUDA(cudaMemcpy((void*)b.entry_offsets, offs, sizeof offs, cudaMemcpyHostToDevice));
    CUDA(cudaMalloc((void**)&b.q_offsets, sizeof q_offs));
    CUDA(cudaMemcpy((void*)b.q_offsets, q_offs, sizeof q_offs, cudaMemcpyHostToDevice));
    CUDA(cudaMalloc((void**)&b.q_start, sizeof q_start));
    CUDA(cudaMemcpy((void*)b.q_start, q_start, sizeof q_start, cudaMemcpyHostToDevice));

    FILE* o = fopen(out_path, "wb");
    if (!o) FAIL("cannot open %s", out_path);

    /* prefill */
    void* out_d = NULL;
    CUDA(cudaMalloc(&out_d, nq * esz));
    CHECK(lazyattn_prefill(pool, &b, q_dev, out_d, NULL, 0, NULL));
    float* out_h = (float*)malloc(nq * sizeof(float) + 1);
    from_device(out_h, out_d, nq, bf16);
    fwrite(out_h, sizeof(float), nq, o);

    /* decode steps */
    const size_t ws_bytes = lazyattn_workspace_size(pool, LAZYATTN_OP_DECODE, &b);
    if (ws_bytes == 0) FAIL("workspace size");
    void* ws = NULL;
    CUDA(cudaMalloc(&ws, ws_bytes));
    CUDA(cudaMemset(ws, 0, ws_bytes));
    void* dout = NULL;
    CUDA(cudaMalloc(&dout, (size_t)Hq * D * esz));
    for (int t = 0; t < n_steps; ++t) {
        float* q = read_f32(f, (size_t)Hq * D);
        float* k = read_f32(f, (size_t)Hkv * D);
        float* v = read_f32(f, (size_t)Hkv * D);
        void* dq = to_device(q, (size_t)Hq * D, bf16);
        void* dk = to_device(k, (size_t)Hkv * D, bf16);
        void* dv = to_device(v, (size_t)Hkv * D, bf16);
        CHECK(lazyattn_decode(pool, &b, dq, dk, dv, dout, ws, ws_bytes, NULL));
        from_device(out_h, dout, (size_t)Hq * D, bf16);
        fwrite(out_h, sizeof(float), (size_t)Hq * D, o);
        CUDA(cudaFree(dq));
        CUDA(cudaFree(dk));
        CUDA(cudaFree(dv));
        free(q);
        free(k);
        free(v);
    }
    int32_t status = 0;
    CHECK(lazyattn_get_device_status(pool, &status, 1, NULL));
    if (status != 0) FAIL("device status %s", lazyattn_status_string(status));
    fclose(o);
    fclose(f);

    CHECK(lazyattn_pool_destroy(pool));
    CUDA(cudaFree(q_dev));
    CUDA(cudaFree(out_d));
    CUDA(cudaFree(dout));
    CUDA(cudaFree(ws));
    CUDA(cudaFree(b.entries));
    CUDA(cudaFree((void*)b.entry_offsets));
    CUDA(cudaFree((void*)b.q_offsets));
    CUDA(cudaFree((void*)b.q_start));
    CUDA(cudaFree(d.k_pool));
    CUDA(cudaFree(d.v_pool));
    CUDA(cudaFree(d.rope_table));
    CUDA(cudaFree(d.status_word));
    free(out_h);
    free(entries);
    free(page_ids);
    free(doc_len);
    printf("run ok\n");
    return 0;
}

int main(int argc, char** argv) {
    if (argc >= 2 && strcmp(argv[1], "host") == 0) return host_checks();
    if (argc == 4 && strcmp(argv[1], "run") == 0) return run(argv[2], argv[3]);
    fprintf(stderr, "usage: %s host | run IN OUT\n", argv[0]);
    return 2;
}
