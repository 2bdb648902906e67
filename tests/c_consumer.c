/*
 * c_consumer.c -- the C ABI used from plain C99, with no Python in between.
 *
 *   c_consumer host   no GPU needed: version, status strings, the launch
 *                     planner, and the host-side argument checks through dry
 *                     runs on addresses that are never dereferenced.
 *   c_consumer gpu    a real fused call with a dynamic NVFP4 scale (N=4,
 *                     T=37, d=4096) on device buffers made with the CUDA
 *                     runtime, compared with the CPU oracle on the same
 *                     inputs: bf16 outputs within 1e-2 |ref| + 1e-3 of the
 *                     oracle's unrounded values, NVFP4 codes, scales and g
 *                     bit-exact against the oracle quantiser run on the
 *                     kernel's own out_norm.
 *
 * Test infrastructure: it links the product library and the oracle
 * (liboracle.so) side by side; neither library uses the other.
 * Exit status 0 on success; a message on stderr otherwise.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "tpar.h"

/* the oracle's C entry points (oracle/oracle.c) */
int orc_fused_rmsnorm(const uint16_t* const* partials, int n, const uint16_t* residual, const uint16_t* gamma,
                      float eps, int64_t T, int64_t d, double* h_ref, double* y_ref, uint16_t* out_res,
                      uint16_t* out_norm);
int orc_nvfp4_quantize(const uint16_t* x, int64_t T, int64_t d, int given, float g_in, uint8_t* codes,
                       uint8_t* scales, float* g_out);
double orc_bf16_to_double(uint16_t b);

static int failures = 0;
#define CHECK(cond, ...)                                  \
    do {                                                  \
        if (!(cond)) {                                    \
            fprintf(stderr, "FAIL %s:%d: ", __FILE__, __LINE__); \
            fprintf(stderr, __VA_ARGS__);                 \
            fprintf(stderr, "\n");                        \
            ++failures;                                   \
        }                                                 \
    } while (0)

/* ------------------------------------------------------------- host mode */

static int host_mode(void)
{
    CHECK(tpar_version() >= TPAR_VERSION, "version %d", tpar_version());
    for (int s = 0; s <= 6; ++s)
        CHECK(tpar_status_string((tpar_status)s) != NULL && tpar_status_string((tpar_status)s)[0] != 0,
              "status string %d", s);
    CHECK(tpar_workspace_bytes() >= 16, "workspace bytes");
    CHECK(tpar_debug_build() == 0, "release library expected");

    tpar_plan p;
    CHECK(tpar_plan_launch(8, 4096, 8, 152, 0, &p) == TPAR_OK && p.kernel == 1 && p.split == 4,
          "decode plan %d/%d", p.kernel, p.split);
    CHECK(tpar_plan_launch(4096, 8192, 8, 152, 0, &p) == TPAR_OK && p.kernel == 3 && p.grid_rows == 152,
          "prefill plan %d", p.kernel);
    CHECK(tpar_plan_launch(4096, 8192, 8, 152, TPAR_FORCE_ROW, &p) == TPAR_OK && p.kernel == 0, "row plan");
    CHECK(tpar_plan_launch(8, 4100, 8, 152, 0, &p) == TPAR_ERR_INVALID_ARG, "d %% 8");

    /* dry runs on fake, never-dereferenced addresses */
    const uintptr_t base = (uintptr_t)0x7f0000000000ull, mb = 1u << 20;
    const void* parts[4];
    for (int r = 0; r < 4; ++r)
        parts[r] = (const void*)(base + (uintptr_t)r * 4 * mb);
    void* res = (void*)(base + 64 * mb);
    void* gam = (void*)(base + 96 * mb);
    void* on = (void*)(base + 128 * mb);
    void* orr = (void*)(base + 160 * mb);
    uint8_t* codes = (uint8_t*)(base + 200 * mb);
    uint8_t* scales = (uint8_t*)(base + 240 * mb);
    float* g = (float*)(base + 250 * mb);
    CHECK(tpar_fused_rmsnorm_ex(parts, 4, res, gam, 1e-5f, 8, 4096, on, orr, codes, scales, g, TPAR_DRY_RUN, NULL,
                                NULL, NULL) == TPAR_OK,
          "valid dry run");
    CHECK(tpar_fused_rmsnorm_ex(parts, 4, res, gam, 1e-5f, 8, 4096, on, orr, codes, NULL, g, TPAR_DRY_RUN, NULL,
                                NULL, NULL) == TPAR_ERR_INVALID_ARG,
          "incomplete NVFP4 triple");
    CHECK(tpar_fused_rmsnorm_ex(parts, 4, res, gam, 1e-5f, 8, 4096, (char*)on + 8, orr, NULL, NULL, NULL,
                                TPAR_DRY_RUN, NULL, NULL, NULL) == TPAR_ERR_MISALIGNED,
          "misaligned out_norm");
    CHECK(tpar_fused_rmsnorm_ex(parts, 4, res, gam, 1e-5f, 8, 4096, (void*)parts[1], orr, NULL, NULL, NULL,
                                TPAR_DRY_RUN, NULL, NULL, NULL) == TPAR_ERR_INVALID_ARG,
          "out_norm on a partial");
    CHECK(tpar_fused_rmsnorm_ex(parts, 17, res, gam, 1e-5f, 8, 4096, on, orr, NULL, NULL, NULL, TPAR_DRY_RUN,
                                NULL, NULL, NULL) == TPAR_ERR_INVALID_ARG,
          "17 ranks");
    CHECK(tpar_fused_rmsnorm_ex(parts, 4, res, gam, 1e-5f, -1, 4096, on, orr, NULL, NULL, NULL, TPAR_DRY_RUN,
                                NULL, NULL, NULL) == TPAR_ERR_INVALID_ARG,
          "T < 0");
    CHECK(tpar_fused_rmsnorm_ex(parts, 4, res, gam, 1e-5f, 0, 4096, NULL, NULL, NULL, NULL, NULL, 0, NULL, NULL,
                                NULL) == TPAR_OK,
          "T == 0 is a no-op");
    return failures;
}

/* -------------------------------------------------------------- GPU mode */

#ifdef TPAR_C_CONSUMER_GPU
#include <cuda_runtime_api.h>

static uint16_t bf16_of(float f)  /* round to nearest even (finite inputs) */
{
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static uint32_t lcg(uint32_t* s)
{
    *s = *s * 1664525u + 1013904223u;
    return *s;
}

static float uniform_pm1(uint32_t* s) { return ((float)(lcg(s) >> 8) / 16777216.0f) * 2.0f - 1.0f; }

#define CUDA_OK(x)                                                        \
    do {                                                                  \
        cudaError_t e_ = (x);                                             \
        if (e_ != cudaSuccess) {                                          \
            fprintf(stderr, "CUDA %s at %s:%d\n", cudaGetErrorString(e_), __FILE__, __LINE__); \
            return 1;                                                     \
        }                                                                 \
    } while (0)

static int gpu_mode(void)
{
    enum { N = 4, T = 37, D = 4096 };
    const size_t td = (size_t)T * D;
    const float eps = 1e-5f;
    uint32_t seed = 12345u;
    uint16_t* hp[N];
    for (int r = 0; r < N; ++r) {
        hp[r] = (uint16_t*)malloc(td * 2);
        for (size_t i = 0; i < td; ++i)
            hp[r][i] = bf16_of(0.5f * uniform_pm1(&seed));
    }
    uint16_t* hr = (uint16_t*)malloc(td * 2);
    uint16_t* hg = (uint16_t*)malloc((size_t)D * 2);
    for (size_t i = 0; i < td; ++i)
        hr[i] = bf16_of(uniform_pm1(&seed));
    for (int i = 0; i < D; ++i)
        hg[i] = bf16_of(1.0f + 0.1f * uniform_pm1(&seed));

    CHECK(tpar_init(0) == TPAR_OK, "tpar_init");
    void *dp[N], *dr, *dg, *don, *dor, *dcodes, *dscales, *dgs;
    for (int r = 0; r < N; ++r) {
        CUDA_OK(cudaMalloc(&dp[r], td * 2));
        CUDA_OK(cudaMemcpy(dp[r], hp[r], td * 2, cudaMemcpyHostToDevice));
    }
    CUDA_OK(cudaMalloc(&dr, td * 2));
    CUDA_OK(cudaMalloc(&dg, (size_t)D * 2));
    CUDA_OK(cudaMalloc(&don, td * 2));
    CUDA_OK(cudaMalloc(&dor, td * 2));
    CUDA_OK(cudaMalloc(&dcodes, td / 2));
    CUDA_OK(cudaMalloc(&dscales, td / 16));
    CUDA_OK(cudaMalloc(&dgs, 4));
    CUDA_OK(cudaMemcpy(dr, hr, td * 2, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(dg, hg, (size_t)D * 2, cudaMemcpyHostToDevice));
    const void* cparts[N];
    for (int r = 0; r < N; ++r)
        cparts[r] = dp[r];
    CHECK(tpar_fused_rmsnorm(cparts, N, dr, dg, eps, T, D, don, dor, (uint8_t*)dcodes, (uint8_t*)dscales,
                             (float*)dgs, NULL) == TPAR_OK,
          "fused call");
    CUDA_OK(cudaDeviceSynchronize());

    uint16_t* gon = (uint16_t*)malloc(td * 2);
    uint16_t* gor = (uint16_t*)malloc(td * 2);
    uint8_t* gcodes = (uint8_t*)malloc(td / 2);
    uint8_t* gscales = (uint8_t*)malloc(td / 16);
    float gg = 0.0f;
    CUDA_OK(cudaMemcpy(gon, don, td * 2, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(gor, dor, td * 2, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(gcodes, dcodes, td / 2, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(gscales, dscales, td / 16, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(&gg, dgs, 4, cudaMemcpyDeviceToHost));

    /* the oracle on the same inputs */
    double* h = (double*)malloc(td * sizeof(double));
    double* y = (double*)malloc(td * sizeof(double));
    const uint16_t* opart[N];
    for (int r = 0; r < N; ++r)
        opart[r] = hp[r];
    CHECK(orc_fused_rmsnorm(opart, N, hr, hg, eps, T, D, h, y, NULL, NULL) == 0, "oracle");
    int bad = 0;
    for (size_t i = 0; i < td; ++i) {
        const double a = orc_bf16_to_double(gor[i]), b = orc_bf16_to_double(gon[i]);
        if (!(fabs(a - h[i]) <= 1e-2 * fabs(h[i]) + 1e-3) || !(fabs(b - y[i]) <= 1e-2 * fabs(y[i]) + 1e-3))
            ++bad;
    }
    CHECK(bad == 0, "%d elements out of tolerance", bad);
    /* NVFP4 on the kernel's own out_norm */
    uint8_t* ocodes = (uint8_t*)malloc(td / 2);
    uint8_t* oscales = (uint8_t*)malloc(td / 16);
    float og = 0.0f;
    CHECK(orc_nvfp4_quantize(gon, T, D, 0, 0.0f, ocodes, oscales, &og) == 0, "oracle quantiser");
    CHECK(memcmp(&og, &gg, 4) == 0, "global scale %g vs %g", (double)gg, (double)og);
    CHECK(memcmp(ocodes, gcodes, td / 2) == 0, "codes differ");
    CHECK(memcmp(oscales, gscales, td / 16) == 0, "scales differ");
    uint32_t code = 1;
    CHECK(tpar_device_error(0, &code) == TPAR_OK && code == 0, "device error word %u", code);

    for (int r = 0; r < N; ++r) {
        cudaFree(dp[r]);
        free(hp[r]);
    }
    cudaFree(dr); cudaFree(dg); cudaFree(don); cudaFree(dor); cudaFree(dcodes); cudaFree(dscales); cudaFree(dgs);
    free(hr); free(hg); free(gon); free(gor); free(gcodes); free(gscales); free(h); free(y); free(ocodes);
    free(oscales);
    return failures;
}
#endif

int main(int argc, char** argv)
{
    if (argc > 1 && strcmp(argv[1], "gpu") == 0) {
#ifdef TPAR_C_CONSUMER_GPU
        const int f = gpu_mode();
        if (f == 0)
            printf("c_consumer gpu: ok\n");
        return f == 0 ? 0 : 1;
#else
        fprintf(stderr, "built without TPAR_C_CONSUMER_GPU\n");
        return 2;
#endif
    }
    const int f = host_mode();
    if (f == 0)
        printf("c_consumer host: ok\n");
    return f == 0 ? 0 : 1;
}
