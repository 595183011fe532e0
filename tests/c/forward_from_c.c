/*
 * A plain C caller of the library (no Python, no PyTorch): reads the
 * forward's inputs as raw 16-bit arrays from a directory, copies them into
 * cudaMalloc'd buffers, runs moe_forward on the default stream with the
 * workspace size the library reports, and writes the output back.
 *
 *   forward_from_c DIR T d_hidden d_expert E k dtype(0 = f16, 1 = bf16)
 *
 * DIR holds x.bin [T, d_hidden], wg.bin [E, d_hidden], w_gate.bin and
 * w_up.bin [E, d_expert, d_hidden], w_down.bin [E, d_hidden, d_expert]; the
 * program writes out.bin [T, d_hidden] and prints "ok" (exit 0), or an error
 * and a non-zero exit code.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "moe_routed_gate.h"

static void *read_file(const char *dir, const char *name, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "rb");
    if (!f) return NULL;
    void *buf = malloc(bytes);
    size_t got = buf ? fread(buf, 1, bytes, f) : 0;
    fclose(f);
    if (got != bytes) {
        free(buf);
        return NULL;
    }
    return buf;
}

static void *to_device(const void *host, size_t bytes) {
    void *d = NULL;
    if (cudaMalloc(&d, bytes) != cudaSuccess) return NULL;
    if (cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
    return d;
}

int main(int argc, char **argv) {
    if (argc != 8) {
        fprintf(stderr, "usage: %s DIR T d_hidden d_expert E k dtype\n", argv[0]);
        return 1;
    }
    const char *dir = argv[1];
    const int64_t T = atoll(argv[2]), d_h = atoll(argv[3]), d_e = atoll(argv[4]);
    const int64_t E = atoll(argv[5]), k = atoll(argv[6]);
    const moe_dtype_t dtype = atoi(argv[7]) == 1 ? MOE_BF16 : MOE_F16;
    const size_t es = 2;
    const size_t bx = (size_t)(T * d_h) * es, bg = (size_t)(E * d_h) * es;
    const size_t bw = (size_t)(E * d_e * d_h) * es;
    const char *names[5] = {"x.bin", "wg.bin", "w_gate.bin", "w_up.bin", "w_down.bin"};
    const size_t sizes[5] = {bx, bg, bw, bw, bw};
    void *dev[5];
    for (int i = 0; i < 5; ++i) {
        void *h = read_file(dir, names[i], sizes[i]);
        if (!h) {
            fprintf(stderr, "cannot read %s/%s (%zu bytes)\n", dir, names[i], sizes[i]);
            return 1;
        }
        dev[i] = to_device(h, sizes[i]);
        free(h);
        if (!dev[i]) {
            fprintf(stderr, "cudaMalloc / copy failed for %s\n", names[i]);
            return 1;
        }
    }
    const size_t ws_bytes = moe_forward_workspace_bytes(T, d_h, d_e, E, k, dtype);
    void *ws = NULL, *out = NULL;
    int32_t *err = NULL;
    if (ws_bytes == (size_t)-1 || cudaMalloc(&ws, ws_bytes) != cudaSuccess ||
        cudaMalloc(&out, bx) != cudaSuccess || cudaMalloc((void **)&err, sizeof(int32_t)) != cudaSuccess ||
        cudaMemset(err, 0, sizeof(int32_t)) != cudaSuccess) {
        fprintf(stderr, "workspace or output allocation failed\n");
        return 1;
    }
    /* cudaMalloc returns 256-byte aligned memory, as moe_forward requires */
    moe_status_t st = moe_forward(dev[0], dev[1], NULL, dev[2], dev[3], dev[4], T, d_h, d_e, E, k, dtype, ws,
                                  ws_bytes, out, err, NULL);
    if (st != MOE_OK) {
        fprintf(stderr, "moe_forward: %s\n", moe_status_string(st));
        return 2;
    }
    if (cudaDeviceSynchronize() != cudaSuccess) {
        fprintf(stderr, "CUDA error: %s\n", cudaGetErrorString(cudaGetLastError()));
        return 3;
    }
    int32_t herr = 0;
    void *hout = malloc(bx);
    if (!hout || cudaMemcpy(&herr, err, sizeof herr, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(hout, out, bx, cudaMemcpyDeviceToHost) != cudaSuccess) {
        fprintf(stderr, "copy back failed\n");
        return 3;
    }
    if (herr != 0) {
        fprintf(stderr, "device error word: %s\n", moe_status_string(herr));
        return 4;
    }
    char path[4096];
    snprintf(path, sizeof path, "%s/out.bin", dir);
    FILE *f = fopen(path, "wb");
    if (!f || fwrite(hout, 1, bx, f) != bx) {
        fprintf(stderr, "cannot write %s\n", path);
        return 1;
    }
    fclose(f);
    free(hout);
    for (int i = 0; i < 5; ++i) cudaFree(dev[i]);
    cudaFree(ws);
    cudaFree(out);
    cudaFree(err);
    printf("ok\n");
    return 0;
}
