/* One optimizer step from plain C: device buffers from the CUDA runtime, the
 * step through the C ABI, the result checked on the host against the
 * first-step closed form of AdamW.  With m = v = 0 before step 1,
 * m_hat = g' and v_hat = g'^2, so p1 = p0 (1 - lr wd) - lr g' / (|g'| + eps)
 * with g' = c g / d.  Then the allocation-free norm of the same gradients
 * (which the step left unchanged) against the same norm and c.  Exit status
 * 0 on success. */
#include <math.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "soma_opt.h"

#define N 1000

int main(void) {
    float *hp = malloc(N * sizeof(float)), *hg = malloc(N * sizeof(float)), *out = malloc(N * sizeof(float));
    double sq = 0.0;
    for (int i = 0; i < N; ++i) {
        hp[i] = 0.01f * (float)((i % 13) - 6);
        hg[i] = 0.5f * (float)((i % 7) - 3) + 0.25f;
        sq += (double)hg[i] * hg[i];
    }
    float *p, *g, *m, *v;
    if (cudaMalloc((void **)&p, N * 4) || cudaMalloc((void **)&g, N * 4) || cudaMalloc((void **)&m, N * 4) ||
        cudaMalloc((void **)&v, N * 4)) {
        fprintf(stderr, "cudaMalloc failed\n");
        return 1;
    }
    cudaMemcpy(p, hp, N * 4, cudaMemcpyHostToDevice);
    cudaMemcpy(g, hg, N * 4, cudaMemcpyHostToDevice);
    cudaMemset(m, 0, N * 4);
    cudaMemset(v, 0, N * 4);

    const double lr = 1e-3, wd = 0.01, eps = 1e-8, d = 2.0, max_norm = 1.0;
    soma_opt_t opt = NULL;
    int32_t grp = -1;
    soma_tensor_t t = {p, g, m, v, NULL, N, 0, SOMA_DTYPE_F32, 1, 1, 0};
    double norm = 0.0, coef = 0.0;
    int32_t nonfinite = -1;
    if (soma_opt_create(&opt, 0) || soma_opt_add_group(opt, lr, 0.9, 0.999, eps, wd, &grp) ||
        soma_opt_step(opt, &t, 1, d, max_norm, NULL) || soma_opt_get_norm(opt, &norm, &coef, &nonfinite, NULL)) {
        fprintf(stderr, "library call failed: %s\n", soma_opt_last_error(opt));
        return 1;
    }
    cudaMemcpy(out, p, N * 4, cudaMemcpyDeviceToHost);

    const double ref_norm = sqrt(sq) / d;
    const double ref_c = fmin(1.0, max_norm / (ref_norm + 1e-6));
    if (nonfinite || fabs(norm - ref_norm) > 1e-5 * ref_norm || fabs(coef - ref_c) > 1e-5 * ref_c) {
        fprintf(stderr, "norm %.9g (ref %.9g), c %.9g (ref %.9g)\n", norm, ref_norm, coef, ref_c);
        return 1;
    }
    for (int i = 0; i < N; ++i) {
        const double gp = ref_c * hg[i] / d;
        const double ref = hp[i] * (1.0 - lr * wd) - lr * gp / (fabs(gp) + eps);
        if (fabs(out[i] - ref) > 2e-6 * fabs(ref) + 1e-8) {
            fprintf(stderr, "p[%d] = %.9g, closed form %.9g\n", i, out[i], ref);
            return 1;
        }
    }
    /* the norm and c again, from the entry point that allocates nothing */
    double *dnc = NULL, hnc[2] = {0.0, 0.0};
    if (cudaMalloc((void **)&dnc, sizeof hnc) || soma_clip_norm_noalloc(0, &t, 1, d, max_norm, dnc, NULL) ||
        cudaMemcpy(hnc, dnc, sizeof hnc, cudaMemcpyDeviceToHost)) {
        fprintf(stderr, "no-alloc norm failed\n");
        return 1;
    }
    if (fabs(hnc[0] - ref_norm) > 1e-5 * ref_norm || fabs(hnc[1] - ref_c) > 1e-5 * ref_c) {
        fprintf(stderr, "no-alloc norm %.9g (ref %.9g), c %.9g (ref %.9g)\n", hnc[0], ref_norm, hnc[1], ref_c);
        return 1;
    }
    cudaFree(dnc);
    soma_opt_destroy(opt);
    cudaFree(p);
    cudaFree(g);
    cudaFree(m);
    cudaFree(v);
    puts("c step ok");
    return 0;
}
