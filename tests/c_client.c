/*
 * A plain C99 client of libfa: compiles against include/fa.h alone, links
 * libfa.so, and makes the calls that need no GPU (size queries, status
 * strings, argument checks).  Prints "ok" and exits 0 when every answer is
 * the documented one.
 *
 * Built with -DFA_CLIENT_GPU (and the CUDA runtime), "c_client gpu FILE"
 * also runs the forward and the backward on a GPU with no PyTorch anywhere:
 * cudaMalloc, plain cudaMemcpy, fa_fwd then fa_bwd on a small causal GQA
 * shape, and a comparison with the float64 oracle's values in FILE
 * (tests/golden/c_client_case.txt, written by make_c_client_case.py beside
 * it).  The inputs are drawn here from SplitMix64 exactly as that script
 * draws them.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "fa.h"
#ifdef FA_CLIENT_GPU
#include <cuda_runtime_api.h>
#endif

static int failures = 0;

static void expect(int cond, const char* what) {
    if (!cond) {
        printf("FAILED: %s\n", what);
        ++failures;
    }
}

#ifdef FA_CLIENT_GPU
/* SplitMix64 (Steele, Lea and Flood, OOPSLA 2014) */
static uint64_t splitmix64(uint64_t x) {
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* element i of input tensor t as bf16 bits: a 24-bit uniform value in
   [-1, 1), exact in float32, rounded to bf16 to nearest, ties to even */
static uint16_t input_bf16(uint64_t t, uint64_t i) {
    const int64_t u = (int64_t)(splitmix64((t << 32) + i) >> 40);
    const float x = (float)(u - (1 << 23)) / (float)(1 << 23);
    uint32_t b;
    memcpy(&b, &x, 4);
    b = (b + 0x7FFFu + ((b >> 16) & 1u)) & 0xFFFF0000u;
    return (uint16_t)(b >> 16);
}

static double bf16_to_double(uint16_t h) {
    const uint32_t b = (uint32_t)h << 16;
    float f;
    memcpy(&f, &b, 4);
    return (double)f;
}

/* half the spacing of bf16 numbers at |r| (8 significant bits) */
static double bf16_half_ulp(double r) {
    const double a = fabs(r);
    return a > 0.0 ? ldexp(1.0, (int)floor(log2(a)) - 8) : 0.0;
}

#define CK(call)                                                              \
    do {                                                                      \
        cudaError_t e_ = (call);                                              \
        if (e_ != cudaSuccess) {                                              \
            printf("FAILED: %s: %s\n", #call, cudaGetErrorString(e_));        \
            return 1;                                                         \
        }                                                                     \
    } while (0)

/* The tolerances of the parity tests: max-abs 2e-2 beyond bf16 rounding for
   O, dQ, dK, dV, 1e-3 for lse; the L2 norm of each tensor within 5e-3. */
static int gpu_case(const char* path) {
    FILE* f = fopen(path, "r");
    if (f == NULL) {
        printf("FAILED: cannot open %s\n", path);
        return 1;
    }
    char line[256];
    int B = 0, H = 0, Hkv = 0, N = 0, d = 0, causal = 0;
    double scale = 0.0;
    while (fgets(line, sizeof line, f) != NULL)
        if (sscanf(line, "shape %d %d %d %d %d %d %lf", &B, &H, &Hkv, &N, &d, &causal, &scale) == 7)
            break;
    if (B <= 0 || N <= 0) {
        printf("FAILED: no shape line in %s\n", path);
        fclose(f);
        return 1;
    }
    const size_t nq = (size_t)B * N * H * d, nk = (size_t)B * N * Hkv * d, nl = (size_t)B * H * N;
    uint16_t* hin[4];
    const size_t nin[4] = {nq, nk, nk, nq};
    for (int t = 0; t < 4; ++t) {
        hin[t] = malloc(nin[t] * 2);
        if (hin[t] == NULL) return 2;
        for (size_t i = 0; i < nin[t]; ++i) hin[t][i] = input_bf16((uint64_t)t, i);
    }
    /* device buffers: q k v dout | o dq dk dv | lse | workspace */
    void *dq_in, *dk_in, *dv_in, *ddo, *dout_o, *ddq, *ddk, *ddv, *dws;
    float* dlse;
    const size_t ws = fa_bwd_workspace_size(B, H, Hkv, N, d);
    CK(cudaMalloc(&dq_in, nq * 2));
    CK(cudaMalloc(&dk_in, nk * 2));
    CK(cudaMalloc(&dv_in, nk * 2));
    CK(cudaMalloc(&ddo, nq * 2));
    CK(cudaMalloc(&dout_o, nq * 2));
    CK(cudaMalloc(&ddq, nq * 2));
    CK(cudaMalloc(&ddk, nk * 2));
    CK(cudaMalloc(&ddv, nk * 2));
    CK(cudaMalloc((void**)&dlse, nl * 4));
    CK(cudaMalloc(&dws, ws));
    CK(cudaMemcpy(dq_in, hin[0], nq * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dk_in, hin[1], nk * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dv_in, hin[2], nk * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(ddo, hin[3], nq * 2, cudaMemcpyHostToDevice));
    fa_status st = fa_fwd(dq_in, dk_in, dv_in, dout_o, dlse, B, H, Hkv, N, d, causal,
                          (float)scale, NULL);
    expect(st == FA_OK, "fa_fwd returns FA_OK");
    st = fa_bwd(dq_in, dk_in, dv_in, dout_o, ddo, dlse, ddq, ddk, ddv, dws, NULL, B, H, Hkv, N, d,
                causal, (float)scale, NULL);
    expect(st == FA_OK, "fa_bwd returns FA_OK");
    CK(cudaDeviceSynchronize());
    expect(fa_get_device_error(NULL) == FA_OK, "no device-side failure recorded");
    uint16_t* hout[4];  /* o dq dk dv */
    const size_t nout[4] = {nq, nq, nk, nk};
    void* dsrc[4] = {dout_o, ddq, ddk, ddv};
    for (int t = 0; t < 4; ++t) {
        hout[t] = malloc(nout[t] * 2);
        if (hout[t] == NULL) return 2;
        CK(cudaMemcpy(hout[t], dsrc[t], nout[t] * 2, cudaMemcpyDeviceToHost));
    }
    float* hlse = malloc(nl * 4);
    if (hlse == NULL) return 2;
    CK(cudaMemcpy(hlse, dlse, nl * 4, cudaMemcpyDeviceToHost));

    const char* names[5] = {"o", "lse", "dq", "dk", "dv"};
    int checked = 0;
    double worst[5] = {0, 0, 0, 0, 0};
    rewind(f);
    while (fgets(line, sizeof line, f) != NULL) {
        char name[16];
        double val;
        long long idx;
        int which = -1;
        if (sscanf(line, "norm %15s %lf", name, &val) == 2) {
            for (int n = 0; n < 5; ++n)
                if (strcmp(name, names[n]) == 0) which = n;
            if (which < 0) continue;
            double s2 = 0.0;
            if (which == 1) {
                for (size_t i = 0; i < nl; ++i) s2 += (double)hlse[i] * hlse[i];
            } else {
                const int t = which == 0 ? 0 : which - 1;
                for (size_t i = 0; i < nout[t]; ++i) {
                    const double g = bf16_to_double(hout[t][i]);
                    s2 += g * g;
                }
            }
            char what[64];
            snprintf(what, sizeof what, "L2 norm of %s", name);
            expect(fabs(sqrt(s2) - val) <= 5e-3 * val, what);
        } else if (sscanf(line, "%15s %lld %lf", name, &idx, &val) == 3) {
            for (int n = 0; n < 5; ++n)
                if (strcmp(name, names[n]) == 0) which = n;
            if (which < 0) continue;
            double got, err;
            if (which == 1) {
                if (idx < 0 || (size_t)idx >= nl) continue;
                got = hlse[idx];
                err = fabs(got - val);
                expect(err <= 1e-3, "lse sample within 1e-3");
            } else {
                const int t = which == 0 ? 0 : which - 1;
                if (idx < 0 || (size_t)idx >= nout[t]) continue;
                got = bf16_to_double(hout[t][idx]);
                err = fabs(got - val) - bf16_half_ulp(val);
                char what[64];
                snprintf(what, sizeof what, "%s[%lld] within 2e-2 beyond bf16 rounding", name, idx);
                expect(err <= 2e-2, what);
            }
            if (err > worst[which]) worst[which] = err;
            ++checked;
        }
    }
    fclose(f);
    printf("gpu case B=%d H=%d Hkv=%d N=%d d=%d causal=%d: %d samples; worst o %.3e lse %.3e "
           "dq %.3e dk %.3e dv %.3e\n", B, H, Hkv, N, d, causal, checked, worst[0], worst[1],
           worst[2], worst[3], worst[4]);
    expect(checked > 0, "the expected file has samples");
    cudaFree(dq_in);
    cudaFree(dk_in);
    cudaFree(dv_in);
    cudaFree(ddo);
    cudaFree(dout_o);
    cudaFree(ddq);
    cudaFree(ddk);
    cudaFree(ddv);
    cudaFree(dlse);
    cudaFree(dws);
    for (int t = 0; t < 4; ++t) {
        free(hin[t]);
        free(hout[t]);
    }
    free(hlse);
    return 0;
}
#endif

int main(int argc, char** argv) {
#ifdef FA_CLIENT_GPU
    if (argc == 3 && strcmp(argv[1], "gpu") == 0) {
        const int rc = gpu_case(argv[2]);
        if (rc != 0) return rc;
        if (failures == 0) printf("ok\n");
        return failures == 0 ? 0 : 1;
    }
#else
    (void)argc;
    (void)argv;
#endif
    /* any 256-byte-aligned, non-null address: rejected calls never touch it */
    char* raw = malloc(512);
    if (raw == NULL) return 2;
    void* p = (void*)(((uintptr_t)raw + 255u) & ~(uintptr_t)255u);

    expect(strcmp(fa_status_string(FA_OK), "FA_OK") == 0, "status string of FA_OK");
    expect(strcmp(fa_status_string(FA_ERR_INVALID_ARG), "FA_ERR_INVALID_ARG") == 0,
           "status string of FA_ERR_INVALID_ARG");

    /* workspace: 4*B*H*N for D, the fp16 copies and 512 bytes of scales, each
       part rounded up to 256 bytes */
    expect(fa_bwd_workspace_size(2, 3, 1, 5, 64) == 11008, "workspace size, small case");
    expect(fa_bwd_workspace_size(1, 1, 1, 1, 96) == 0, "workspace size, unsupported d");
    expect(fa_bwd_workspace_size(1, 6, 4, 1, 64) == 0, "workspace size, H % Hkv != 0");

    /* argument checks: returned before any device work */
    expect(fa_fwd(p, p, p, p, (float*)p, 0, 1, 1, 128, 64, 0, 0.125f, NULL) ==
               FA_ERR_INVALID_ARG, "fa_fwd with B = 0");
    expect(fa_fwd(p, p, p, p, (float*)p, 1, 6, 4, 128, 64, 0, 0.125f, NULL) ==
               FA_ERR_INVALID_ARG, "fa_fwd with H % Hkv != 0");
    expect(fa_fwd(p, p, p, p, (float*)p, 1, 1, 1, 128, 64, 0, -1.0f, NULL) ==
               FA_ERR_INVALID_ARG, "fa_fwd with a negative scale");
    expect(fa_fwd(p, p, p, p, (float*)p, 1, 1, 1, 128, 96, 0, 0.125f, NULL) ==
               FA_ERR_UNSUPPORTED, "fa_fwd with d = 96");
    expect(fa_fwd((char*)p + 8, p, p, p, (float*)p, 1, 1, 1, 128, 64, 0, 0.125f, NULL) ==
               FA_ERR_INVALID_ARG, "fa_fwd with q not 16-byte aligned");
    expect(fa_bwd(p, p, p, p, p, (float*)p, p, p, p, p, NULL, 1, 1, 1, 0, 64, 0, 0.125f, NULL) ==
               FA_ERR_INVALID_ARG, "fa_bwd with N = 0");
    expect(fa_fwd_fp8_workspace_size(1, 4, 2, 256, 64) == 0, "fp8 workspace, d = 64");
    expect(fa_fwd_splitkv_num_splits(1, 8, 2, 10, 5, 128, 1, 0) == 0,
           "split-KV plan, causal with Nq > Nk");

    free(raw);
    if (failures == 0) printf("ok\n");
    return failures == 0 ? 0 : 1;
}
