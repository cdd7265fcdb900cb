/* One decode step from plain C through the public header, with nothing but the
 * CUDA runtime for memory: append the new K/V rows (pa_reshape_and_cache),
 * then decode (pa_decode) with a workspace sized by pa_decode_workspace_size,
 * and check the device error word. fp32 caches.
 *
 * Input file (little-endian): int32 B, Hq, Hkv, D, bs, NB, max_blocks,
 * max_context_len; float32 scale; then float32 q[B][Hq][D], k_new[B][Hkv][D],
 * v_new[B][Hkv][D]; int64 slots[B]; float32 k_cache and v_cache
 * [NB][Hkv][bs][D]; int32 block_tables[B][max_blocks]; int32 lens[B].
 * Output file: float32 out[B][Hq][D]. Exit status 0 on success. C11 (the CUDA
 * runtime header uses anonymous unions). */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "pagedattn.h"

static void* load(FILE* f, size_t bytes) {
    void* p = malloc(bytes ? bytes : 1);
    if (!p || fread(p, 1, bytes, f) != bytes) exit(10);
    return p;
}

/* A device copy of `bytes` host bytes, or zeroed device memory for host NULL. */
static void* upload(const void* host, size_t bytes) {
    void* d = NULL;
    if (cudaMalloc(&d, bytes ? bytes : 16) != cudaSuccess) exit(11);
    if (host == NULL) {
        if (cudaMemset(d, 0, bytes ? bytes : 16) != cudaSuccess) exit(13);
    } else if (bytes && cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) {
        exit(12);
    }
    return d;
}

int main(int argc, char** argv) {
    if (argc != 3) return 2;
    FILE* f = fopen(argv[1], "rb");
    if (!f) return 3;
    int32_t h[8];
    float scale;
    if (fread(h, sizeof h, 1, f) != 1 || fread(&scale, sizeof scale, 1, f) != 1) return 4;
    const int B = h[0], Hq = h[1], Hkv = h[2], D = h[3], bs = h[4], NB = h[5], MB = h[6],
              mcl = h[7];
    const size_t qn = (size_t)B * Hq * D, rn = (size_t)B * Hkv * D;
    const size_t cn = (size_t)NB * Hkv * bs * D;
    void* q = load(f, qn * 4);
    void* kn = load(f, rn * 4);
    void* vn = load(f, rn * 4);
    void* slots = load(f, (size_t)B * 8);
    void* kc = load(f, cn * 4);
    void* vc = load(f, cn * 4);
    void* bt = load(f, (size_t)B * MB * 4);
    void* lens = load(f, (size_t)B * 4);
    fclose(f);

    void* dq = upload(q, qn * 4);
    void* dkn = upload(kn, rn * 4);
    void* dvn = upload(vn, rn * 4);
    void* dslots = upload(slots, (size_t)B * 8);
    void* dkc = upload(kc, cn * 4);
    void* dvc = upload(vc, cn * 4);
    void* dbt = upload(bt, (size_t)B * MB * 4);
    void* dlens = upload(lens, (size_t)B * 4);
    void* dout = upload(NULL, qn * 4);
    int32_t zero = 0;
    int32_t* derr = (int32_t*)upload(&zero, 4);
    const size_t ws_bytes = pa_decode_workspace_size(B, Hq, D, mcl);
    void* dws = upload(NULL, ws_bytes);

    pa_status st = pa_reshape_and_cache(dkn, dvn, (const int64_t*)dslots, dkc, dvc, B, Hkv, D,
                                        bs, NB, PA_DTYPE_F32, derr, NULL);
    if (st != PA_OK) return 20 + (int)st;
    st = pa_decode(dq, dkc, dvc, (const int32_t*)dbt, (const int32_t*)dlens, scale, dout, B, Hq,
                   Hkv, D, bs, NB, MB, mcl, PA_DTYPE_F32, dws, ws_bytes, derr, NULL);
    if (st != PA_OK) return 30 + (int)st;
    if (cudaDeviceSynchronize() != cudaSuccess) return 40;
    int32_t err = -1;
    if (cudaMemcpy(&err, derr, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return 41;
    if (pa_check_error_word(err) != PA_OK) return 42;
    float* out = (float*)malloc(qn * 4);
    if (!out || cudaMemcpy(out, dout, qn * 4, cudaMemcpyDeviceToHost) != cudaSuccess) return 43;
    FILE* o = fopen(argv[2], "wb");
    if (!o || fwrite(out, 4, qn, o) != qn) return 44;
    fclose(o);
    return 0;
}
