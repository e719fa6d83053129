/*
 * A plain C consumer of libbq.so: no Python, no PyTorch. Reads n BF16 values (raw
 * little-endian bit patterns) from the file argv[1], runs on the current CUDA device
 *   bq_quant_i8 -> bq_dequant_i8        (block INT8 wire round trip)
 *   bq_quant_mx  (one row of n values)  (MXFP8 codes + E8M0 scales)
 * and writes to argv[2], in this order: payload int8[n], scales float[n/128], BF16
 * materialization uint16[n], E4M3 codes uint8[n], E8M0 bytes uint8[n/32].
 * It also checks that invalid calls return their status codes before any launch.
 * Exit status 0 on success; a message on stderr otherwise.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <cuda_runtime_api.h>

#include "bq.h"

#define CUDA_OK(call)                                                                    \
    do {                                                                                 \
        cudaError_t e_ = (call);                                                         \
        if (e_ != cudaSuccess) {                                                         \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));                  \
            return 2;                                                                    \
        }                                                                                \
    } while (0)

#define BQ_OK_OR_FAIL(call)                                                              \
    do {                                                                                 \
        bq_status s_ = (call);                                                           \
        if (s_ != BQ_OK) {                                                               \
            fprintf(stderr, "%s: %s\n", #call, bq_status_string(s_));                    \
            return 3;                                                                    \
        }                                                                                \
    } while (0)

int main(int argc, char **argv)
{
    if (argc != 3) {
        fprintf(stderr, "usage: %s input.bf16 output.bin\n", argv[0]);
        return 1;
    }
    if (bq_abi_version() != BQ_ABI_VERSION) {
        fprintf(stderr, "library ABI %d, header ABI %d\n", bq_abi_version(), BQ_ABI_VERSION);
        return 1;
    }
    FILE *f = fopen(argv[1], "rb");
    if (!f) return 1;
    fseek(f, 0, SEEK_END);
    const int64_t n = ftell(f) / 2;
    fseek(f, 0, SEEK_SET);
    uint16_t *hx = malloc(2 * n);
    if (!hx || fread(hx, 2, n, f) != (size_t)n) return 1;
    fclose(f);

    const int64_t wire = bq_wire_bytes(n);
    if (wire < 0) {
        fprintf(stderr, "n = %lld is not a multiple of 128\n", (long long)n);
        return 1;
    }
    void *dx, *dout;
    uint8_t *dwire, *dq, *ds;
    CUDA_OK(cudaMalloc(&dx, 2 * n));
    CUDA_OK(cudaMalloc(&dout, 2 * n));
    CUDA_OK(cudaMalloc((void **)&dwire, wire));
    CUDA_OK(cudaMalloc((void **)&dq, n));
    CUDA_OK(cudaMalloc((void **)&ds, n / 32));
    CUDA_OK(cudaMemcpy(dx, hx, 2 * n, cudaMemcpyHostToDevice));

    cudaStream_t st;
    CUDA_OK(cudaStreamCreate(&st));
    int8_t *payload = (int8_t *)dwire;
    float *scales = (float *)(dwire + n);  /* scale region at byte offset n */

    /* argument errors come back before any launch */
    if (bq_quant_i8(dx, n + 64, payload, scales, st) != BQ_ERR_SHAPE) return 4;
    if (bq_quant_i8(NULL, n, payload, scales, st) != BQ_ERR_NULL) return 4;
    if (bq_quant_i8((char *)dx + 2, n, payload, scales, st) != BQ_ERR_ALIGN) return 4;
    if (bq_quant_i8(dx, n, (int8_t *)dx, scales, st) != BQ_ERR_ALIAS) return 4;

    BQ_OK_OR_FAIL(bq_quant_i8(dx, n, payload, scales, st));
    BQ_OK_OR_FAIL(bq_dequant_i8(payload, scales, n, dout, st));
    BQ_OK_OR_FAIL(bq_quant_mx(dx, 1, n, n, dq, n, ds, n / 32, st));
    CUDA_OK(cudaStreamSynchronize(st));

    uint8_t *hwire = malloc(wire), *hq = malloc(n), *hs = malloc(n / 32);
    uint16_t *hout = malloc(2 * n);
    if (!hwire || !hq || !hs || !hout) return 1;
    CUDA_OK(cudaMemcpy(hwire, dwire, wire, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(hout, dout, 2 * n, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(hq, dq, n, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(hs, ds, n / 32, cudaMemcpyDeviceToHost));

    FILE *o = fopen(argv[2], "wb");
    if (!o) return 1;
    fwrite(hwire, 1, wire, o);   /* payload, then scales */
    fwrite(hout, 2, n, o);
    fwrite(hq, 1, n, o);
    fwrite(hs, 1, n / 32, o);
    fclose(o);

    cudaFree(dx);
    cudaFree(dout);
    cudaFree(dwire);
    cudaFree(dq);
    cudaFree(ds);
    cudaStreamDestroy(st);
    free(hx);
    free(hwire);
    free(hq);
    free(hs);
    free(hout);
    return 0;
}
