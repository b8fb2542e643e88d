/*
 * A plain C caller of libmoe_swiglu_nvfp4.so through include/moe_nvfp4.h.
 *
 *   quantize_from_c                      checks host-side argument errors
 *                                        (no device is touched) and prints
 *                                        the codes and one message
 *   quantize_from_c run IN OUT ROWS K    reads ROWS x K BF16 values (uint16
 *                                        bit patterns) from file IN,
 *                                        quantizes them on the GPU with
 *                                        moe_nvfp4_quantize and writes the
 *                                        packed bytes, then the scale bytes,
 *                                        to file OUT
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "moe_nvfp4.h"

static int check_arguments(void) {
    /* fake, suitably aligned device addresses: every call below is rejected
       on the host before anything could reach them */
    const uint16_t *x = (const uint16_t *)(uintptr_t)0x7f0000000000ull;
    uint8_t *out = (uint8_t *)(uintptr_t)0x7f0000000000ull;
    const int bad_width = moe_nvfp4_quantize(x, 4, 24, out, out, NULL);
    const int bad_rows = moe_nvfp4_quantize(x, -1, 32, out, out, NULL);
    const int null_in = moe_nvfp4_quantize(NULL, 4, 32, out, out, NULL);
    const int bad_clamp = moe_swiglu_nvfp4_quantize(x, 4, 32, 0.0f, NULL, 0, out, out, NULL);
    const int nothing = moe_nvfp4_quantize(NULL, 0, 32, NULL, NULL, NULL);
    printf("%d %d %d %d %d %d\n", bad_width, bad_rows, null_in, bad_clamp, nothing, moe_nvfp4_abi_version());
    printf("%s\n", moe_nvfp4_strerror(bad_width));
    return 0;
}

static int fail(const char *what) {
    fprintf(stderr, "quantize_from_c: %s\n", what);
    return 1;
}

static int run(const char *in_path, const char *out_path, int64_t rows, int64_t k) {
    const size_t n_in = (size_t)(rows * k), n_packed = n_in / 2, n_sf = n_in / 16;
    uint16_t *h_in = (uint16_t *)malloc(n_in * sizeof(uint16_t));
    uint8_t *h_out = (uint8_t *)malloc(n_packed + n_sf);
    if (h_in == NULL || h_out == NULL) return fail("out of host memory");
    FILE *f = fopen(in_path, "rb");
    if (f == NULL || fread(h_in, sizeof(uint16_t), n_in, f) != n_in) return fail("cannot read the input");
    fclose(f);
    void *d_in = NULL, *d_packed = NULL, *d_sf = NULL;
    if (cudaMalloc(&d_in, n_in * sizeof(uint16_t)) != cudaSuccess || cudaMalloc(&d_packed, n_packed) != cudaSuccess ||
        cudaMalloc(&d_sf, n_sf) != cudaSuccess)
        return fail("cudaMalloc failed");
    if (cudaMemcpy(d_in, h_in, n_in * sizeof(uint16_t), cudaMemcpyHostToDevice) != cudaSuccess)
        return fail("upload failed");
    const int rc = moe_nvfp4_quantize((const uint16_t *)d_in, rows, k, (uint8_t *)d_packed, (uint8_t *)d_sf, NULL);
    if (rc != 0) {
        fprintf(stderr, "quantize_from_c: %s\n", moe_nvfp4_strerror(rc));
        return 1;
    }
    if (cudaMemcpy(h_out, d_packed, n_packed, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(h_out + n_packed, d_sf, n_sf, cudaMemcpyDeviceToHost) != cudaSuccess)
        return fail("download failed");
    f = fopen(out_path, "wb");
    if (f == NULL || fwrite(h_out, 1, n_packed + n_sf, f) != n_packed + n_sf) return fail("cannot write the output");
    fclose(f);
    cudaFree(d_in);
    cudaFree(d_packed);
    cudaFree(d_sf);
    free(h_in);
    free(h_out);
    return 0;
}

int main(int argc, char **argv) {
    if (argc == 1) return check_arguments();
    if (argc == 6) return run(argv[2], argv[3], strtoll(argv[4], NULL, 10), strtoll(argv[5], NULL, 10));
    fprintf(stderr, "usage: quantize_from_c [run IN OUT ROWS K]\n");
    return 2;
}
