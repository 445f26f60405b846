/*
 * amp_c_client.c - a plain C caller of libampfp8.so: no Python, no torch.
 *
 * Reads a binary input file, runs `steps` mixed-precision optimizer steps
 * through the C ABI (amp_unscale_check, amp_adamw_master_step with bf16
 * emission and an amax slot, fp8_quant_tensorwise_list, amp_update_scale)
 * on the legacy default stream, and writes the final state to an output file.
 *
 * Input  (little-endian): int32 n_tensors, int32 steps, then per tensor int64
 *        numel, int64 rows, int64 cols (cols == 0: no FP8 copy), then the
 *        fp32 masters, then for each step the fp16 gradient bit patterns.
 *        Hyper-parameters: lr 1e-3, betas 0.9 / 0.999, eps 1e-8, wd 0.01,
 *        S0 65536, growth 2, backoff 0.5, interval 2.
 * Output: int32 found_inf per step, float scale, int32 tracker, int32 step,
 *        then per tensor master, m, v (fp32) and bf16 bits, then per FP8
 *        tensor the e4m3fn bytes, the transposed bytes and inv_scale.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "ampfp8.h"

#define CK(x)                                                                          \
    do {                                                                               \
        int st_ = (int)(x);                                                            \
        if (st_ != 0) {                                                                \
            fprintf(stderr, "%s failed (%d): %s\n", #x, st_, amp_last_error());        \
            exit(1);                                                                   \
        }                                                                              \
    } while (0)
#define CU(x)                                                                          \
    do {                                                                               \
        cudaError_t e_ = (x);                                                          \
        if (e_ != cudaSuccess) {                                                       \
            fprintf(stderr, "%s failed: %s\n", #x, cudaGetErrorString(e_));            \
            exit(1);                                                                   \
        }                                                                              \
    } while (0)

static void *dmalloc(size_t n) {
    void *p = NULL;
    CU(cudaMalloc(&p, n ? n : 16));
    CU(cudaMemset(p, 0, n ? n : 16));
    return p;
}

static void rd(void *p, size_t n, FILE *f) {
    if (fread(p, 1, n, f) != n) { fprintf(stderr, "short input\n"); exit(1); }
}

int main(int argc, char **argv) {
    if (argc != 3) { fprintf(stderr, "usage: %s in.bin out.bin\n", argv[0]); return 2; }
    FILE *in = fopen(argv[1], "rb");
    if (!in) return 2;
    int32_t n, steps;
    rd(&n, 4, in);
    rd(&steps, 4, in);
    int64_t *numel = malloc(n * 8), *rows = malloc(n * 8), *cols = malloc(n * 8);
    for (int i = 0; i < n; ++i) { rd(&numel[i], 8, in); rd(&rows[i], 8, in); rd(&cols[i], 8, in); }

    void **p = malloc(n * sizeof(void *)), **m = malloc(n * sizeof(void *)),
         **v = malloc(n * sizeof(void *)), **g = malloc(n * sizeof(void *)),
         **b = malloc(n * sizeof(void *));
    int32_t *slots = malloc(n * 4);
    int n8 = 0;
    for (int i = 0; i < n; ++i) {
        p[i] = dmalloc(numel[i] * 4);
        m[i] = dmalloc(numel[i] * 4);
        v[i] = dmalloc(numel[i] * 4);
        g[i] = dmalloc(numel[i] * 2);
        b[i] = dmalloc(numel[i] * 2);
        slots[i] = cols[i] ? n8++ : -1;
    }
    amp_tensor_list Lp, Lm, Lv, Lg, Lb, Lx, Lq, Lqt;
    CK(amp_tensor_list_create(n, p, numel, NULL, AMP_DT_F32, NULL, &Lp));
    /* host buffers, one per tensor, fed and read back through the ABI */
    void **hp = malloc(n * sizeof(void *)), **hm = malloc(n * sizeof(void *)),
         **hv = malloc(n * sizeof(void *)), **hg = malloc(n * sizeof(void *)),
         **hb = malloc(n * sizeof(void *));
    for (int i = 0; i < n; ++i) {
        hp[i] = malloc(numel[i] * 4 + 4);
        hm[i] = malloc(numel[i] * 4 + 4);
        hv[i] = malloc(numel[i] * 4 + 4);
        hg[i] = malloc(numel[i] * 2 + 2);
        hb[i] = malloc(numel[i] * 2 + 2);
        rd(hp[i], numel[i] * 4, in);
    }
    CK(amp_tensor_list_copy_from_host(Lp, (const void *const *)hp, NULL));
    CK(amp_tensor_list_create(n, m, numel, NULL, AMP_DT_F32, NULL, &Lm));
    CK(amp_tensor_list_create(n, v, numel, NULL, AMP_DT_F32, NULL, &Lv));
    CK(amp_tensor_list_create(n, g, numel, NULL, AMP_DT_F16, NULL, &Lg));
    CK(amp_tensor_list_create(n, b, numel, NULL, AMP_DT_BF16, NULL, &Lb));
    CK(amp_tensor_list_set_amax_slots(Lb, slots, NULL));
    void **xs = malloc(n8 * sizeof(void *) + 8), **qs = malloc(n8 * sizeof(void *) + 8),
         **qts = malloc(n8 * sizeof(void *) + 8);
    int64_t *r8 = malloc(n8 * 8 + 8), *c8 = malloc(n8 * 8 + 8);
    for (int i = 0, j = 0; i < n; ++i) {
        if (!cols[i]) continue;
        xs[j] = b[i];
        qs[j] = dmalloc(numel[i]);
        qts[j] = dmalloc(numel[i]);
        r8[j] = rows[i];
        c8[j] = cols[i];
        ++j;
    }
    CK(amp_tensor_list_create(n8, xs, r8, c8, AMP_DT_BF16, NULL, &Lx));
    CK(amp_tensor_list_create(n8, qs, r8, c8, AMP_DT_E4M3FN, NULL, &Lq));
    CK(amp_tensor_list_create(n8, qts, c8, r8, AMP_DT_E4M3FN, NULL, &Lqt));

    float *scale = dmalloc(4), *amax = dmalloc(4 * (n8 + 1)), *inv = dmalloc(4 * (n8 + 1));
    int32_t *tracker = dmalloc(4), *found = dmalloc(4), *stepc = dmalloc(4);
    const float s0 = 65536.0f;
    CU(cudaMemcpy(scale, &s0, 4, cudaMemcpyHostToDevice));
    const amp_adamw_hyper hy = {1e-3, 0.9, 0.999, 1e-8, 0.01};
    int32_t *fi_log = malloc(steps * 4);
    for (int k = 0; k < steps; ++k) {
        for (int i = 0; i < n; ++i) rd(hg[i], numel[i] * 2, in);
        CK(amp_tensor_list_copy_from_host(Lg, (const void *const *)hg, NULL));
        CK(amp_unscale_check(Lg, scale, found, 0, NULL));
        CU(cudaMemcpy(&fi_log[k], found, 4, cudaMemcpyDeviceToHost));   /* for the log only */
        CK(amp_adamw_master_step(Lp, Lm, Lv, Lg, Lb, scale, found, stepc, &hy, amax, NULL));
        CK(fp8_quant_tensorwise_list(Lx, Lq, Lqt, AMP_DT_E4M3FN, 1e-12, amax, inv, found, NULL));
        CK(amp_update_scale(scale, tracker, found, 2.0f, 0.5f, 2, amax, n8, NULL));
    }
    CU(cudaDeviceSynchronize());
    fclose(in);

    FILE *out = fopen(argv[2], "wb");
    float s;
    int32_t t, st;
    CU(cudaMemcpy(&s, scale, 4, cudaMemcpyDeviceToHost));
    CU(cudaMemcpy(&t, tracker, 4, cudaMemcpyDeviceToHost));
    CU(cudaMemcpy(&st, stepc, 4, cudaMemcpyDeviceToHost));
    fwrite(fi_log, 4, steps, out);
    fwrite(&s, 4, 1, out);
    fwrite(&t, 4, 1, out);
    fwrite(&st, 4, 1, out);
    CK(amp_tensor_list_copy_to_host(Lp, hp, NULL));
    CK(amp_tensor_list_copy_to_host(Lm, hm, NULL));
    CK(amp_tensor_list_copy_to_host(Lv, hv, NULL));
    CK(amp_tensor_list_copy_to_host(Lb, hb, NULL));
    CU(cudaDeviceSynchronize());
    for (int i = 0; i < n; ++i) {
        fwrite(hp[i], 4, numel[i], out);
        fwrite(hm[i], 4, numel[i], out);
        fwrite(hv[i], 4, numel[i], out);
        fwrite(hb[i], 2, numel[i], out);
        free(hp[i]);
        free(hm[i]);
        free(hv[i]);
        free(hg[i]);
        free(hb[i]);
    }
    float *hinv = malloc(4 * (n8 + 1));
    CU(cudaMemcpy(hinv, inv, 4 * (n8 + 1), cudaMemcpyDeviceToHost));
    for (int j = 0, i = 0; i < n; ++i) {
        if (!cols[i]) continue;
        void *h = malloc(numel[i]);
        CU(cudaMemcpy(h, qs[j], numel[i], cudaMemcpyDeviceToHost));
        fwrite(h, 1, numel[i], out);
        CU(cudaMemcpy(h, qts[j], numel[i], cudaMemcpyDeviceToHost));
        fwrite(h, 1, numel[i], out);
        fwrite(&hinv[j], 4, 1, out);
        free(h);
        ++j;
    }
    fclose(out);
    amp_tensor_list all[8] = {Lp, Lm, Lv, Lg, Lb, Lx, Lq, Lqt};
    for (int i = 0; i < 8; ++i) CK(amp_tensor_list_destroy(all[i]));
    printf("ok %d steps\n", steps);
    return 0;
}
