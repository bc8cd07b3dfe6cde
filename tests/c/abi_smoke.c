/* A plain C caller of libspec_verify: builds a small greedy batch whose answer
 * is fixed by construction, runs spec_verify and spec_sample through the C ABI
 * (device memory from the CUDA runtime, then the logits in mapped page-locked
 * host memory through spec_device_pointer), and checks the outputs.  Exit code 0
 * on success; the test in test_gpu_c_abi.py compiles and runs it.
 *
 * Rows: logit_j = -|j - peak| in float32, so the argmax of a row is its peak
 * (the greedy rule: accept while the draft equals the target argmax, then emit
 * the argmax of the first mismatching row, or of the bonus row). */
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "spec_verify.h"

#define B 3
#define G 4
#define V 1000

static int check(cudaError_t e, const char *what)
{
    if (e != cudaSuccess) {
        fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
        return 1;
    }
    return 0;
}

int main(void)
{
    static float target[B][G + 1][V], draft[B][G][V];
    int peaks[B][G + 1], tokens[B][G], num_draft[B] = {G, G, 2};
    float uniforms[B][G + 1], temperature[B] = {0.0f, 0.0f, 0.0f};
    for (int b = 0; b < B; ++b)
        for (int i = 0; i <= G; ++i) {
            peaks[b][i] = (37 * b + 101 * i + 5) % V;
            for (int j = 0; j < V; ++j) {
                const float d = (float)(j > peaks[b][i] ? j - peaks[b][i] : peaks[b][i] - j);
                target[b][i][j] = -d;
                if (i < G)
                    draft[b][i][j] = -d;
            }
            uniforms[b][i] = 0.5f;
        }
    /* sequence 0 drafts every peak (all accepted: bonus = peak of row G);
     * sequence 1 misses at position 2 (emits the peak of row 2);
     * sequence 2 has two drafts, both right (bonus = peak of row 2). */
    for (int b = 0; b < B; ++b)
        for (int i = 0; i < G; ++i)
            tokens[b][i] = i < num_draft[b] ? peaks[b][i] : -1;
    tokens[1][2] = (peaks[1][2] + 1) % V;
    const int want_n[B] = {G, 2, 2};
    const int want_last[B] = {peaks[0][G], peaks[1][2], peaks[2][2]};

    void *dt, *dd, *dtok, *dnum, *du, *dT, *dout, *dn, *dst;
    if (check(cudaMalloc(&dt, sizeof target), "malloc") || check(cudaMalloc(&dd, sizeof draft), "malloc") ||
        check(cudaMalloc(&dtok, sizeof tokens), "malloc") || check(cudaMalloc(&dnum, sizeof num_draft), "malloc") ||
        check(cudaMalloc(&du, sizeof uniforms), "malloc") || check(cudaMalloc(&dT, sizeof temperature), "malloc") ||
        check(cudaMalloc(&dout, sizeof(int) * B * (G + 1)), "malloc") || check(cudaMalloc(&dn, sizeof(int) * B), "malloc") ||
        check(cudaMalloc(&dst, sizeof(unsigned)), "malloc"))
        return 2;
    cudaMemcpy(dt, target, sizeof target, cudaMemcpyHostToDevice);
    cudaMemcpy(dd, draft, sizeof draft, cudaMemcpyHostToDevice);
    cudaMemcpy(dtok, tokens, sizeof tokens, cudaMemcpyHostToDevice);
    cudaMemcpy(dnum, num_draft, sizeof num_draft, cudaMemcpyHostToDevice);
    cudaMemcpy(du, uniforms, sizeof uniforms, cudaMemcpyHostToDevice);
    cudaMemcpy(dT, temperature, sizeof temperature, cudaMemcpyHostToDevice);
    cudaMemset(dst, 0, sizeof(unsigned));

    spec_status st = spec_verify(dt, dd, (const int32_t *)dtok, (const int32_t *)dnum, (const float *)du,
                                 (const float *)dT, (int32_t *)dout, (int32_t *)dn, B, G, V, SPEC_F32,
                                 (uint32_t *)dst, NULL);
    if (st != SPEC_OK) {
        fprintf(stderr, "spec_verify: %s\n", spec_status_string(st));
        return 3;
    }
    int out[B][G + 1], n[B];
    unsigned status = 0;
    if (check(cudaMemcpy(out, dout, sizeof out, cudaMemcpyDeviceToHost), "copy") ||
        check(cudaMemcpy(n, dn, sizeof n, cudaMemcpyDeviceToHost), "copy") ||
        check(cudaMemcpy(&status, dst, sizeof status, cudaMemcpyDeviceToHost), "copy"))
        return 4;
    int bad = status != 0;
    for (int b = 0; b < B; ++b) {
        bad |= n[b] != want_n[b] || out[b][n[b]] != want_last[b];
        for (int i = 0; i < n[b]; ++i)
            bad |= out[b][i] != tokens[b][i];
        for (int i = n[b] + 1; i <= G; ++i)
            bad |= out[b][i] != -1;
        printf("seq %d: accepted %d, last %d (want %d, %d)\n", b, n[b], out[b][n[b]], want_n[b], want_last[b]);
    }
    /* the sampler at T = 0 on rows t_0: the peaks of row 0 */
    void *rows;
    if (check(cudaMalloc(&rows, sizeof(float) * B * V), "malloc"))
        return 2;
    for (int b = 0; b < B; ++b)
        cudaMemcpy((float *)rows + (size_t)b * V, target[b][0], sizeof(float) * V, cudaMemcpyHostToDevice);
    st = spec_sample(rows, (const float *)du, (const float *)dT, (int32_t *)dn, B, V, SPEC_F32, NULL, NULL, NULL);
    if (st != SPEC_OK) {
        fprintf(stderr, "spec_sample: %s\n", spec_status_string(st));
        return 3;
    }
    if (check(cudaMemcpy(n, dn, sizeof n, cudaMemcpyDeviceToHost), "copy"))
        return 4;
    for (int b = 0; b < B; ++b)
        bad |= n[b] != peaks[b][0];
    /* zero copy: the logits in mapped page-locked host memory, read by the
     * early-exit kernel over the host link; same answer as from device memory */
    void *ht, *hd;
    const void *at = NULL, *ad = NULL;
    if (check(cudaHostAlloc(&ht, sizeof target, cudaHostAllocMapped), "host alloc") ||
        check(cudaHostAlloc(&hd, sizeof draft, cudaHostAllocMapped), "host alloc"))
        return 2;
    memcpy(ht, target, sizeof target);
    memcpy(hd, draft, sizeof draft);
    bad |= spec_device_pointer(ht, &at) != SPEC_OK || spec_device_pointer(hd, &ad) != SPEC_OK;
    bad |= spec_device_pointer(target, &at) != SPEC_ERR_INVALID_ARG;  /* pageable: refused, at unchanged */
    spec_verify_options opt = {0, 3, NULL, NULL};
    st = spec_verify_ex(at, ad, (const int32_t *)dtok, (const int32_t *)dnum, (const float *)du, (const float *)dT,
                        (int32_t *)dout, (int32_t *)dn, B, G, V, SPEC_F32, NULL, NULL, &opt);
    if (st != SPEC_OK) {
        fprintf(stderr, "spec_verify_ex (host rows): %s\n", spec_status_string(st));
        return 3;
    }
    int out2[B][G + 1], n2[B];
    if (check(cudaMemcpy(out2, dout, sizeof out2, cudaMemcpyDeviceToHost), "copy") ||
        check(cudaMemcpy(n2, dn, sizeof n2, cudaMemcpyDeviceToHost), "copy"))
        return 4;
    bad |= memcmp(out, out2, sizeof out) != 0 || memcmp(n2, want_n, sizeof n2) != 0;
    printf("host rows: %s\n", memcmp(out, out2, sizeof out) ? "differ" : "same tokens");
    cudaFreeHost(ht);
    cudaFreeHost(hd);
    /* a rejected argument: B < 0 */
    bad |= spec_verify(dt, dd, (const int32_t *)dtok, (const int32_t *)dnum, (const float *)du, (const float *)dT,
                       (int32_t *)dout, (int32_t *)dn, -1, G, V, SPEC_F32, NULL, NULL) != SPEC_ERR_INVALID_ARG;
    printf(bad ? "FAIL\n" : "OK\n");
    return bad ? 1 : 0;
}
