/*
 * A plain C11 client of libnrc.so, built by the tests against include/nrc.h
 * alone (no C++ and no PyTorch), so the header stays valid C and the library
 * stays usable from C.
 *
 *   nrc_client queries      host-only calls: version, workspace sizes,
 *                           status strings, argument errors (no GPU needed)
 *   nrc_client block DIR    reads DIR/dims.txt ("N C L dilation eps") and
 *                           the fp32 arrays DIR/{x,rm,rv,gamma,beta,w,bias}.bin,
 *                           runs nrc_prenorm_dilconv_residual on device copies
 *                           and writes DIR/out.bin
 *
 * Exit status 0 on success; a message on stderr otherwise.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "nrc.h"

static int fail(const char* what) {
    fprintf(stderr, "nrc_client: %s\n", what);
    return 1;
}

static int queries(void) {
    if (nrc_version() <= 0) return fail("version");
    const size_t ws = nrc_prenorm_dilconv_residual_workspace_size(256, NRC_F32);
    if (ws == 0 || ws % 256 != 0) return fail("block workspace size");
    if (nrc_prenorm_dilconv_residual_workspace_size(0, NRC_F32) != 0) return fail("C = 0");
    if (nrc_conv1d_groupnorm_workspace_size(16, 128, 256, 1024, 3, 1, 1, 1, 32) == 0)
        return fail("groupnorm workspace size");
    if (nrc_linear_bn_swish_workspace_size(1024, 8192, 8192) == 0)
        return fail("linear workspace size");
    if (strlen(nrc_status_string(NRC_ERR_TIMEOUT)) == 0) return fail("status string");
    /* null pointers are refused before any CUDA call */
    if (nrc_prenorm_dilconv_residual(NULL, NULL, NRC_F32, 1, 8, 8, 3, 1, 1, NULL, NULL, NULL,
                                     NULL, 1e-5f, NULL, NULL, NULL, 0, NULL) !=
        NRC_ERR_INVALID_ARG)
        return fail("null arguments accepted");
    printf("queries ok: version %d, block workspace %zu bytes\n", nrc_version(), ws);
    return 0;
}

static float* read_array(const char* dir, const char* name, size_t n) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s.bin", dir, name);
    FILE* f = fopen(path, "rb");
    if (!f) return NULL;
    float* a = (float*)malloc(n * sizeof(float));
    if (a && fread(a, sizeof(float), n, f) != n) {
        free(a);
        a = NULL;
    }
    fclose(f);
    return a;
}

static void* to_device(const float* h, size_t n) {
    void* d = NULL;
    if (cudaMalloc(&d, n * sizeof(float)) != cudaSuccess) return NULL;
    if (cudaMemcpy(d, h, n * sizeof(float), cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
    return d;
}

static int block(const char* dir) {
    char path[4096];
    snprintf(path, sizeof path, "%s/dims.txt", dir);
    FILE* f = fopen(path, "r");
    if (!f) return fail("dims.txt");
    int N, C, L, d;
    float eps;
    const int got = fscanf(f, "%d %d %d %d %f", &N, &C, &L, &d, &eps);
    fclose(f);
    if (got != 5) return fail("dims.txt format");
    const size_t nx = (size_t)N * C * L, nw = (size_t)C * C * 3;
    float* hx = read_array(dir, "x", nx);
    float* hrm = read_array(dir, "rm", (size_t)C);
    float* hrv = read_array(dir, "rv", (size_t)C);
    float* hg = read_array(dir, "gamma", (size_t)C);
    float* hb = read_array(dir, "beta", (size_t)C);
    float* hw = read_array(dir, "w", nw);
    float* hbias = read_array(dir, "bias", (size_t)C);
    if (!hx || !hrm || !hrv || !hg || !hb || !hw || !hbias) return fail("input arrays");
    void *x = to_device(hx, nx), *rm = to_device(hrm, C), *rv = to_device(hrv, C);
    void *g = to_device(hg, C), *b = to_device(hb, C), *w = to_device(hw, nw);
    void* bias = to_device(hbias, C);
    void *out = NULL, *ws = NULL;
    const size_t ws_bytes = nrc_prenorm_dilconv_residual_workspace_size(C, NRC_F32);
    if (!x || !rm || !rv || !g || !b || !w || !bias ||
        cudaMalloc(&out, nx * sizeof(float)) != cudaSuccess ||
        cudaMalloc(&ws, ws_bytes) != cudaSuccess)
        return fail("device buffers");
    cudaStream_t st;
    if (cudaStreamCreate(&st) != cudaSuccess) return fail("stream");
    const nrc_status s = nrc_prenorm_dilconv_residual(
        x, out, NRC_F32, N, C, L, 3, d, d, (const float*)rm, (const float*)rv, (const float*)g,
        (const float*)b, eps, w, bias, ws, ws_bytes, (void*)st);
    if (s != NRC_OK) return fail(nrc_status_string(s));
    if (nrc_query_status((void*)st) != NRC_OK) return fail("device status");
    float* hout = (float*)malloc(nx * sizeof(float));
    if (!hout || cudaMemcpy(hout, out, nx * sizeof(float), cudaMemcpyDeviceToHost) != cudaSuccess)
        return fail("copy out");
    snprintf(path, sizeof path, "%s/out.bin", dir);
    FILE* o = fopen(path, "wb");
    if (!o || fwrite(hout, sizeof(float), nx, o) != nx) return fail("out.bin");
    fclose(o);
    printf("block ok: N=%d C=%d L=%d d=%d\n", N, C, L, d);
    return 0;
}

int main(int argc, char** argv) {
    if (argc >= 2 && strcmp(argv[1], "queries") == 0) return queries();
    if (argc >= 3 && strcmp(argv[1], "block") == 0) return block(argv[2]);
    return fail("usage: nrc_client queries | nrc_client block DIR");
}
