/*
 * attn_client.c -- a plain C program that uses libattn through include/attn.h
 * alone (no Python, no C++), for the tests: it shows that the header compiles
 * as C and that the library's entry points link and work from C.
 *
 *   attn_client abi
 *       No GPU needed: status strings, workspace-size queries, and calls with
 *       null pointers, which the library must reject before launching
 *       anything.  Prints "abi ok" on success.
 *   attn_client run DIR
 *       On a GPU: reads the inputs the test wrote into DIR (raw fp32 files),
 *       runs an exact and a tensor-core prefill, a decode and a kv_append +
 *       decode on cudaMalloc'd buffers, and writes the outputs back into DIR.
 *       Prints "run ok" on success.
 * Exit status 0 on success, 1 on any failed check.
 */
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "../../include/attn.h"

#define CHECK(cond, ...)                        \
    do {                                        \
        if (!(cond)) {                          \
            fprintf(stderr, __VA_ARGS__);       \
            fprintf(stderr, "\n");              \
            exit(1);                            \
        }                                       \
    } while (0)

/* Sizes shared with the test (tests/test_c_client.py). */
enum { PM = 200, PHQ = 4, PHKV = 2, PD = 64 };        /* prefill */
enum { DHQ = 8, DHKV = 2, DD = 128, DS = 1000 };       /* decode cache */

static int abi_checks(void) {
    static const attn_status_t codes[] = {ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED,
                                          ATTN_ERR_CUDA, ATTN_ERR_TIMEOUT, ATTN_ERR_RANGE};
    for (size_t i = 0; i < sizeof(codes) / sizeof(codes[0]); ++i) {
        const char* s = attn_status_string(codes[i]);
        CHECK(s != NULL && s[0] != '\0', "empty status string for %d", (int)codes[i]);
    }
    CHECK(attn_prefill_workspace_size(PM, PHQ, PHKV, PD, ATTN_PREC_FP32) == 0,
          "exact prefill must need no workspace");
    CHECK(attn_prefill_workspace_size(PM, PHQ, PHKV, PD, ATTN_PREC_FP16) > 0,
          "fp16 prefill needs its rounded K and V");
    CHECK(attn_prefill_workspace_size(PM, PHQ, PHKV, PD, ATTN_PREC_TF32) > 0,
          "TF32 prefill needs its rounded K and V");
    CHECK(attn_decode_workspace_size(DHQ, DHKV, DD, DS, 0) > 0, "decode needs partials");
    /* Null pointers: rejected before any launch. */
    CHECK(attn_prefill_causal(NULL, NULL, NULL, NULL, PM, PHQ, PHKV, PD, PHQ * PD, PHKV * PD, 0.f,
                              ATTN_PREC_FP32, NULL, 0, NULL) == ATTN_ERR_INVALID_ARG,
          "null prefill pointers must be rejected");
    CHECK(attn_decode(NULL, NULL, NULL, NULL, DHQ, DHKV, DD, DS, DS, 0, 0.f, NULL, 0, NULL) ==
              ATTN_ERR_INVALID_ARG,
          "null decode pointers must be rejected");
    CHECK(kv_append(NULL, NULL, NULL, NULL, DHKV, DD, DS, 0, NULL) == ATTN_ERR_INVALID_ARG,
          "null append pointers must be rejected");
    puts("abi ok");
    return 0;
}

static float* read_file(const char* dir, const char* name, size_t n) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE* f = fopen(path, "rb");
    CHECK(f != NULL, "cannot open %s", path);
    float* h = (float*)malloc(n * sizeof(float));
    CHECK(h != NULL && fread(h, sizeof(float), n, f) == n, "short read of %s", path);
    fclose(f);
    return h;
}

static void write_file(const char* dir, const char* name, const float* h, size_t n) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE* f = fopen(path, "wb");
    CHECK(f != NULL && fwrite(h, sizeof(float), n, f) == n, "cannot write %s", path);
    fclose(f);
}

static float* to_device(const float* h, size_t n) {
    float* d = NULL;
    CHECK(cudaMalloc((void**)&d, n * sizeof(float)) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMemcpy(d, h, n * sizeof(float), cudaMemcpyHostToDevice) == cudaSuccess, "H2D");
    return d;
}

static void from_device(float* h, const float* d, size_t n) {
    CHECK(cudaMemcpy(h, d, n * sizeof(float), cudaMemcpyDeviceToHost) == cudaSuccess, "D2H");
}

static int run(const char* dir) {
    /* ---- prefill, exact and fp16 tensor-core modes */
    const size_t nq = (size_t)PM * PHQ * PD, nkv = (size_t)PM * PHKV * PD;
    float *hq = read_file(dir, "prefill_q.bin", nq), *hk = read_file(dir, "prefill_k.bin", nkv),
          *hv = read_file(dir, "prefill_v.bin", nkv);
    float *q = to_device(hq, nq), *k = to_device(hk, nkv), *v = to_device(hv, nkv);
    float* o = NULL;
    CHECK(cudaMalloc((void**)&o, nq * sizeof(float)) == cudaSuccess, "cudaMalloc o");
    float* out_h = (float*)malloc(nq * sizeof(float));
    static const attn_precision_t precs[] = {ATTN_PREC_FP32, ATTN_PREC_FP16};
    static const char* names[] = {"prefill_o_fp32.bin", "prefill_o_fp16.bin"};
    for (int p = 0; p < 2; ++p) {
        const size_t ws_bytes = attn_prefill_workspace_size(PM, PHQ, PHKV, PD, precs[p]);
        void* ws = NULL;
        if (ws_bytes) CHECK(cudaMalloc(&ws, ws_bytes) == cudaSuccess, "cudaMalloc workspace");
        const attn_status_t st = attn_prefill_causal(q, k, v, o, PM, PHQ, PHKV, PD, PHQ * PD,
                                                     PHKV * PD, 0.f, precs[p], ws, ws_bytes, NULL);
        CHECK(st == ATTN_OK, "prefill: %s (%s)", attn_status_string(st), attn_last_error_string());
        CHECK(cudaDeviceSynchronize() == cudaSuccess, "sync");
        CHECK(attn_get_device_status() == ATTN_OK, "prefill device status");
        from_device(out_h, o, nq);
        write_file(dir, names[p], out_h, nq);
        cudaFree(ws);
    }
    cudaFree(q); cudaFree(k); cudaFree(v); cudaFree(o);
    free(hq); free(hk); free(hv); free(out_h);

    /* ---- decode over the full cache, then kv_append at the last row + decode */
    const size_t ndq = (size_t)DHQ * DD, nc = (size_t)DHKV * DS * DD, nn = (size_t)DHKV * DD;
    float *hdq = read_file(dir, "decode_q.bin", ndq), *hkc = read_file(dir, "decode_k.bin", nc),
          *hvc = read_file(dir, "decode_v.bin", nc), *hkn = read_file(dir, "decode_k_new.bin", nn),
          *hvn = read_file(dir, "decode_v_new.bin", nn);
    float *dq = to_device(hdq, ndq), *kc = to_device(hkc, nc), *vc = to_device(hvc, nc),
          *kn = to_device(hkn, nn), *vn = to_device(hvn, nn);
    float* out = NULL;
    CHECK(cudaMalloc((void**)&out, ndq * sizeof(float)) == cudaSuccess, "cudaMalloc out");
    const size_t ws_bytes = attn_decode_workspace_size(DHQ, DHKV, DD, DS, 0);
    void* ws = NULL;
    CHECK(cudaMalloc(&ws, ws_bytes) == cudaSuccess, "cudaMalloc decode workspace");
    float* hout = (float*)malloc(ndq * sizeof(float));
    attn_status_t st = attn_decode(dq, kc, vc, out, DHQ, DHKV, DD, DS, DS, 0, 0.f, ws, ws_bytes,
                                   NULL);
    CHECK(st == ATTN_OK, "decode: %s", attn_status_string(st));
    CHECK(cudaDeviceSynchronize() == cudaSuccess, "sync");
    from_device(hout, out, ndq);
    write_file(dir, "decode_out.bin", hout, ndq);
    st = kv_append(kn, vn, kc, vc, DHKV, DD, DS, DS - 1, NULL);
    CHECK(st == ATTN_OK, "kv_append: %s", attn_status_string(st));
    st = attn_decode(dq, kc, vc, out, DHQ, DHKV, DD, DS, DS, 0, 0.f, ws, ws_bytes, NULL);
    CHECK(st == ATTN_OK, "decode after append: %s", attn_status_string(st));
    CHECK(cudaDeviceSynchronize() == cudaSuccess, "sync");
    CHECK(attn_get_device_status() == ATTN_OK, "decode device status");
    from_device(hout, out, ndq);
    write_file(dir, "decode_out_appended.bin", hout, ndq);
    cudaFree(dq); cudaFree(kc); cudaFree(vc); cudaFree(kn); cudaFree(vn); cudaFree(out);
    cudaFree(ws);
    free(hdq); free(hkc); free(hvc); free(hkn); free(hvn); free(hout);
    puts("run ok");
    return 0;
}

int main(int argc, char** argv) {
    if (argc >= 2 && strcmp(argv[1], "abi") == 0) return abi_checks();
    if (argc >= 3 && strcmp(argv[1], "run") == 0) return run(argv[2]);
    fprintf(stderr, "usage: %s abi | run DIR\n", argv[0]);
    return 2;
}
