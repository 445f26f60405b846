/*
 * amp_c_client.c - a plain C caller of libampfp8.so: no Python, no torch.
 *
 * Reads a binary input file, opens the run with the first working copies
 * (amp_emit_bf16 with the FP8 weights' amax, then fp8_quant_tensorwise_list),
 * runs `steps` mixed-precision optimizer steps through the C ABI on the legacy
 * default stream, and writes the final state to an output file.  Per step:
 *   dynamic (default)  amp_unscale_check, amp_adamw_master_step with bf16
 *                      emission and amax slots, fp8_quant_tensorwise_list,
 *                      amp_update_scale;
 *   delayed (argv[3])  amp_unscale_check, amp_adamw_master_step_fp8_delayed
 *                      over the plain tensors and the FP8 weights with an
 *                      amax history of one step (opened from the first
 *                      copy's amax), amp_update_scale_fp8_history.
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
    if (argc != 3 && argc != 4) {
        fprintf(stderr, "usage: %s in.bin out.bin [delayed]\n", argv[0]);
        return 2;
    }
    const int delayed = argc == 4;
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
    float *hist = dmalloc(4 * (n8 + 1));                        /* amax history, one step */
    int32_t *tracker = dmalloc(4), *found = dmalloc(4), *stepc = dmalloc(4);
    const float s0 = 65536.0f;
    CU(cudaMemcpy(scale, &s0, 4, cudaMemcpyHostToDevice));
    const amp_adamw_hyper hy = {1e-3, 0.9, 0.999, 1e-8, 0.01};

    /* the first working copies: bf16 = RNE(master) with the FP8 weights' amax,
     * their FP8 copies; with delayed scaling that amax opens the history */
    CK(amp_emit_bf16(Lp, Lb, amax, NULL));
    CK(fp8_quant_tensorwise_list(Lx, Lq, Lqt, AMP_DT_E4M3FN, 1e-12, amax, inv, NULL, NULL));
    if (delayed) CU(cudaMemcpy(hist, amax, 4 * (size_t)n8, cudaMemcpyDeviceToDevice));
    CU(cudaMemset(amax, 0, 4 * (size_t)(n8 + 1)));

    /* delayed scaling steps the plain tensors (1-D lists) and the FP8 weights
     * (2-D lists over the same buffers) in one call */
    amp_tensor_list Pp = NULL, Pm = NULL, Pv = NULL, Pg = NULL, Pb = NULL;
    amp_tensor_list Fp = NULL, Fm = NULL, Fv = NULL, Fg = NULL;
    if (delayed) {
        int np_ = n - n8;
        void **lp = malloc((np_ + 1) * sizeof(void *)), **lm = malloc((np_ + 1) * sizeof(void *)),
             **lv = malloc((np_ + 1) * sizeof(void *)), **lg = malloc((np_ + 1) * sizeof(void *)),
             **lb = malloc((np_ + 1) * sizeof(void *));
        void **fp = malloc((n8 + 1) * sizeof(void *)), **fm = malloc((n8 + 1) * sizeof(void *)),
             **fv = malloc((n8 + 1) * sizeof(void *)), **fg = malloc((n8 + 1) * sizeof(void *));
        int64_t *ln = malloc((np_ + 1) * 8);
        for (int i = 0, a = 0, c = 0; i < n; ++i) {
            if (cols[i]) {
                fp[c] = p[i]; fm[c] = m[i]; fv[c] = v[i]; fg[c] = g[i]; ++c;
            } else {
                lp[a] = p[i]; lm[a] = m[i]; lv[a] = v[i]; lg[a] = g[i]; lb[a] = b[i];
                ln[a] = numel[i]; ++a;
            }
        }
        CK(amp_tensor_list_create(np_, lp, ln, NULL, AMP_DT_F32, NULL, &Pp));
        CK(amp_tensor_list_create(np_, lm, ln, NULL, AMP_DT_F32, NULL, &Pm));
        CK(amp_tensor_list_create(np_, lv, ln, NULL, AMP_DT_F32, NULL, &Pv));
        CK(amp_tensor_list_create(np_, lg, ln, NULL, AMP_DT_F16, NULL, &Pg));
        CK(amp_tensor_list_create(np_, lb, ln, NULL, AMP_DT_BF16, NULL, &Pb));
        CK(amp_tensor_list_create(n8, fp, r8, c8, AMP_DT_F32, NULL, &Fp));
        CK(amp_tensor_list_create(n8, fm, r8, c8, AMP_DT_F32, NULL, &Fm));
        CK(amp_tensor_list_create(n8, fv, r8, c8, AMP_DT_F32, NULL, &Fv));
        CK(amp_tensor_list_create(n8, fg, r8, c8, AMP_DT_F16, NULL, &Fg));
        free(lp); free(lm); free(lv); free(lg); free(lb); free(ln);
        free(fp); free(fm); free(fv); free(fg);
    }

    int32_t *fi_log = malloc(steps * 4);
    for (int k = 0; k < steps; ++k) {
        for (int i = 0; i < n; ++i) rd(hg[i], numel[i] * 2, in);
        CK(amp_tensor_list_copy_from_host(Lg, (const void *const *)hg, NULL));
        CK(amp_unscale_check(Lg, scale, found, 0, NULL));
        CU(cudaMemcpy(&fi_log[k], found, 4, cudaMemcpyDeviceToHost));   /* for the log only */
        if (delayed) {
            CK(amp_adamw_master_step_fp8_delayed(Pp, Pm, Pv, Pg, Pb, Fp, Fm, Fv, Fg, Lx, Lq, Lqt,
                                                 AMP_DT_E4M3FN, 1e-12, hist, 1, amax, inv, scale,
                                                 found, stepc, &hy, NULL));
            CK(amp_update_scale_fp8_history(scale, tracker, found, 2.0f, 0.5f, 2, amax, hist, n8,
                                            1, NULL));
        } else {
            CK(amp_adamw_master_step(Lp, Lm, Lv, Lg, Lb, scale, found, stepc, &hy, amax, NULL));
            CK(fp8_quant_tensorwise_list(Lx, Lq, Lqt, AMP_DT_E4M3FN, 1e-12, amax, inv, found,
                                         NULL));
            CK(amp_update_scale(scale, tracker, found, 2.0f, 0.5f, 2, amax, n8, NULL));
        }
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
    amp_tensor_list all[17] = {Lp, Lm, Lv, Lg, Lb, Lx, Lq, Lqt, Pp, Pm, Pv, Pg, Pb, Fp, Fm, Fv, Fg};
    for (int i = 0; i < 17; ++i) CK(amp_tensor_list_destroy(all[i]));   /* NULL is accepted */
    printf("ok %d steps\n", steps);
    return 0;
}
