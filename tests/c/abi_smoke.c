/* The C ABI from plain C: no Python, no torch.
 *
 * One decode step on a tiny batch through include/pkv.h alone, with device
 * memory from the CUDA runtime, checked against exact properties of the
 * method: a sequence of length 1 attends only to the token it just appended,
 * so its output is that token's V bit for bit ("LLM 推理引擎内部原理" §2.3 and
 * "vLLM核心概念" §4.2.2: the new token goes into its slot, then the step
 * attends over the sequence including it); copy_blocks copies bytes; a bad
 * argument returns its status and a message without launching anything.
 * Prints "abi_smoke ok" and exits 0 on success.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "pkv.h"

#define B 3
#define HKV 2
#define G 2
#define HQ (HKV * G)
#define D 64
#define BS 16
#define NB 8

static int fails = 0;
#define CHECK(cond, what)                                   \
    do {                                                    \
        if (!(cond)) {                                      \
            fprintf(stderr, "FAIL: %s\n", what);            \
            ++fails;                                        \
        }                                                   \
    } while (0)
#define CUDA(x)                                                                 \
    do {                                                                        \
        cudaError_t e_ = (x);                                                   \
        if (e_ != cudaSuccess) {                                                \
            fprintf(stderr, "cuda error %s at %s\n", cudaGetErrorString(e_), #x); \
            return 2;                                                           \
        }                                                                       \
    } while (0)

/* exact fp16 values: +-2, +-1, +-0.5, +-0.25 */
static const uint16_t kHalves[8] = {0x4000, 0xC000, 0x3C00, 0xBC00, 0x3800, 0xB800, 0x3400, 0xB400};

static uint32_t lcg = 12345u;
static uint16_t next_half(void) {
    lcg = lcg * 1664525u + 1013904223u;
    return kHalves[(lcg >> 24) & 7u];
}

int main(void) {
    const size_t pool_elems = (size_t)NB * BS * HKV * D;
    uint16_t* hk = malloc(pool_elems * 2);
    uint16_t* hv = malloc(pool_elems * 2);
    for (size_t i = 0; i < pool_elems; ++i) {
        hk[i] = next_half();
        hv[i] = next_half();
    }
    uint16_t hq[B * HQ * D], hkn[B * HKV * D], hvn[B * HKV * D], hout[B * HQ * D];
    for (int i = 0; i < B * HQ * D; ++i) hq[i] = next_half();
    for (int i = 0; i < B * HKV * D; ++i) {
        hkn[i] = next_half();
        hvn[i] = next_half();
    }
    /* every sequence has length 1: its only position is block tables[s][0], offset 0 */
    int32_t tables[B] = {5, 2, 7};
    int32_t lens[B] = {1, 1, 1};
    int64_t slots[B] = {5 * BS, 2 * BS, 7 * BS};

    void *dk, *dv, *dq, *dkn, *dvn, *dout, *dtab, *dlen, *dslot;
    CUDA(cudaMalloc(&dk, pool_elems * 2));
    CUDA(cudaMalloc(&dv, pool_elems * 2));
    CUDA(cudaMalloc(&dq, sizeof hq));
    CUDA(cudaMalloc(&dkn, sizeof hkn));
    CUDA(cudaMalloc(&dvn, sizeof hvn));
    CUDA(cudaMalloc(&dout, sizeof hout));
    CUDA(cudaMalloc(&dtab, sizeof tables));
    CUDA(cudaMalloc(&dlen, sizeof lens));
    CUDA(cudaMalloc(&dslot, sizeof slots));
    CUDA(cudaMemcpy(dk, hk, pool_elems * 2, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(dv, hv, pool_elems * 2, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(dq, hq, sizeof hq, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(dkn, hkn, sizeof hkn, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(dvn, hvn, sizeof hvn, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(dtab, tables, sizeof tables, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(dlen, lens, sizeof lens, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(dslot, slots, sizeof slots, cudaMemcpyHostToDevice));

    CHECK(pkv_version() > 0, "pkv_version");
    CHECK(pkv_paged_kv_append(dkn, dvn, dk, dv, dslot, B, NB, BS, HKV, D, PKV_F16, NULL) == PKV_OK,
          "append status");
    const size_t ws_bytes = pkv_decode_workspace_bytes(B, HQ, HKV, D, 1, 0);
    CHECK(ws_bytes != (size_t)-1 && ws_bytes > 0, "workspace size");
    void* ws;
    CUDA(cudaMalloc(&ws, ws_bytes));
    CHECK(pkv_paged_attention_decode(dout, dq, dk, dv, dtab, 1, dlen, B, 1, HQ, HKV, D, BS, NB, 0.125f, PKV_F16, ws,
                                     ws_bytes, 0, NULL) == PKV_OK,
          "decode status");
    CUDA(cudaDeviceSynchronize());
    unsigned err_word = 0;
    CHECK(pkv_device_error(&err_word, 1) == PKV_OK && err_word == 0, "device error word");
    CUDA(cudaMemcpy(hout, dout, sizeof hout, cudaMemcpyDeviceToHost));
    /* out[s][h] = v_new[s][h / G], bit for bit */
    for (int s = 0; s < B; ++s)
        for (int h = 0; h < HQ; ++h)
            CHECK(memcmp(hout + (s * HQ + h) * D, hvn + (s * HKV + h / G) * D, D * 2) == 0, "length-1 output is V");

    /* copy_blocks: block 3 = block 5 (which now holds sequence 0's token), every layer passed */
    void* kc_list[1] = {dk};
    void* vc_list[1] = {dv};
    int64_t pairs[2] = {5, 3};
    void* dpairs;
    CUDA(cudaMalloc(&dpairs, sizeof pairs));
    CUDA(cudaMemcpy(dpairs, pairs, sizeof pairs, cudaMemcpyHostToDevice));
    CHECK(pkv_copy_blocks(kc_list, vc_list, 1, dpairs, 1, NB, BS, HKV, D, PKV_F16, NULL) == PKV_OK, "copy status");
    CUDA(cudaDeviceSynchronize());
    const size_t blk = (size_t)BS * HKV * D;
    CUDA(cudaMemcpy(hk, dk, pool_elems * 2, cudaMemcpyDeviceToHost));
    CHECK(memcmp(hk + 3 * blk, hk + 5 * blk, blk * 2) == 0, "copied block equals its source");
    CHECK(memcmp(hk + 5 * blk, hkn, HKV * D * 2) == 0, "appended row landed in slot 5*BS");

    /* host validation: head_dim 96 is not built; nothing launches */
    CHECK(pkv_paged_attention_decode(dout, dq, dk, dv, dtab, 1, dlen, B, 1, HQ, HKV, 96, BS, NB, 0.125f, PKV_F16, ws,
                                     ws_bytes, 0, NULL) == PKV_ERR_UNSUPPORTED,
          "unsupported head_dim status");
    CHECK(strlen(pkv_last_error()) > 0, "last error message");

    cudaFree(dk);
    cudaFree(dv);
    cudaFree(dq);
    cudaFree(dkn);
    cudaFree(dvn);
    cudaFree(dout);
    cudaFree(dtab);
    cudaFree(dlen);
    cudaFree(dslot);
    cudaFree(ws);
    cudaFree(dpairs);
    free(hk);
    free(hv);
    if (fails) return 1;
    printf("abi_smoke ok\n");
    return 0;
}
