/* One layout -> bf16 dispatch -> combine step through the C ABI alone (no
 * Python between the caller and libep.so), for tests/test_gpu_parity.py.
 *
 * usage: c_abi_step T K E R H dir
 * reads  dir/topk_idx.bin (int64 [T, K]), dir/x.bin (bf16 bits [T, H]),
 *        dir/y.bin (bf16 bits [T*K, H]), dir/w.bin (fp32 [T, K])
 * writes dir/counts.bin (int32 [E]), dir/offsets.bin (int32 [E+1]),
 *        dir/recv.bin (bf16 bits [N, H]), dir/out.bin (bf16 bits [T, H])
 * Exit status 0 on success; otherwise the failing call is printed. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "ep.h"

static int read_file(const char* dir, const char* name, void* dst, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE* f = fopen(path, "rb");
    if (!f) return 1;
    size_t got = fread(dst, 1, bytes, f);
    fclose(f);
    return got != bytes;
}

static int write_file(const char* dir, const char* name, const void* src, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE* f = fopen(path, "wb");
    if (!f) return 1;
    size_t put = fwrite(src, 1, bytes, f);
    fclose(f);
    return put != bytes;
}

#define CK(call)                                                              \
    do {                                                                      \
        int rc_ = (int)(call);                                                \
        if (rc_ != 0) {                                                       \
            fprintf(stderr, "%s failed: %d\n", #call, rc_);                   \
            return 1;                                                         \
        }                                                                     \
    } while (0)

int main(int argc, char** argv) {
    if (argc != 7) {
        fprintf(stderr, "usage: %s T K E R H dir\n", argv[0]);
        return 2;
    }
    const int T = atoi(argv[1]), K = atoi(argv[2]), E = atoi(argv[3]), R = atoi(argv[4]), H = atoi(argv[5]);
    const char* dir = argv[6];
    const size_t slots = (size_t)T * K, rows_cap = slots;

    int64_t* h_idx = (int64_t*)malloc(slots * 8);
    uint16_t* h_x = (uint16_t*)malloc((size_t)T * H * 2);
    uint16_t* h_y = (uint16_t*)malloc(rows_cap * H * 2);
    float* h_w = (float*)malloc(slots * 4);
    if (!h_idx || !h_x || !h_y || !h_w) return 1;
    CK(read_file(dir, "topk_idx.bin", h_idx, slots * 8));
    CK(read_file(dir, "x.bin", h_x, (size_t)T * H * 2));
    CK(read_file(dir, "y.bin", h_y, rows_cap * H * 2));
    CK(read_file(dir, "w.bin", h_w, slots * 4));

    int64_t* d_idx;
    void *d_x, *d_y, *d_recv, *d_out;
    float* d_w;
    int32_t *d_cnt, *d_ntr, *d_off;
    uint8_t* d_itr;
    CK(cudaMalloc((void**)&d_idx, slots * 8));
    CK(cudaMalloc(&d_x, (size_t)T * H * 2));
    CK(cudaMalloc(&d_y, rows_cap * H * 2));
    CK(cudaMalloc((void**)&d_w, slots * 4));
    CK(cudaMalloc(&d_recv, rows_cap * H * 2));
    CK(cudaMalloc(&d_out, (size_t)T * H * 2));
    CK(cudaMalloc((void**)&d_cnt, (size_t)E * 4));
    CK(cudaMalloc((void**)&d_ntr, (size_t)R * 4));
    CK(cudaMalloc((void**)&d_itr, (size_t)T * R));
    CK(cudaMalloc((void**)&d_off, (size_t)(E + 1) * 4));
    CK(cudaMemcpy(d_idx, h_idx, slots * 8, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_x, h_x, (size_t)T * H * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_y, h_y, rows_cap * H * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_w, h_w, slots * 4, cudaMemcpyHostToDevice));

    ep_handle_t h = NULL;
    CK(ep_layout(d_idx, T, K, E, R, d_cnt, d_ntr, d_itr, d_off, NULL, NULL, &h, NULL));
    int64_t n_rows = 0;
    int32_t dev_err = 0;
    CK(ep_handle_query(h, &n_rows, &dev_err));
    CK(dev_err);
    CK(ep_dispatch(h, d_x, H, EP_DTYPE_BF16, NULL, d_recv, NULL, NULL, NULL, (int64_t)rows_cap, NULL));
    CK(ep_combine(h, d_y, (int64_t)rows_cap, H, d_w, d_out, NULL));
    CK(cudaDeviceSynchronize());

    int32_t* h_cnt = (int32_t*)malloc((size_t)E * 4);
    int32_t* h_off = (int32_t*)malloc((size_t)(E + 1) * 4);
    uint16_t* h_recv = (uint16_t*)malloc((size_t)n_rows * H * 2 + 2);
    uint16_t* h_out = (uint16_t*)malloc((size_t)T * H * 2);
    if (!h_cnt || !h_off || !h_recv || !h_out) return 1;
    CK(cudaMemcpy(h_cnt, d_cnt, (size_t)E * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(h_off, d_off, (size_t)(E + 1) * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(h_recv, d_recv, (size_t)n_rows * H * 2, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(h_out, d_out, (size_t)T * H * 2, cudaMemcpyDeviceToHost));
    CK(write_file(dir, "counts.bin", h_cnt, (size_t)E * 4));
    CK(write_file(dir, "offsets.bin", h_off, (size_t)(E + 1) * 4));
    CK(write_file(dir, "recv.bin", h_recv, (size_t)n_rows * H * 2));
    CK(write_file(dir, "out.bin", h_out, (size_t)T * H * 2));

    CK(ep_handle_destroy(h));
    cudaFree(d_idx); cudaFree(d_x); cudaFree(d_y); cudaFree(d_w); cudaFree(d_recv); cudaFree(d_out);
    cudaFree(d_cnt); cudaFree(d_ntr); cudaFree(d_itr); cudaFree(d_off);
    free(h_idx); free(h_x); free(h_y); free(h_w); free(h_cnt); free(h_off); free(h_recv); free(h_out);
    return 0;
}
