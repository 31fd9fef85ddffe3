/* One ZeRO-2 step through the C ABI from a C program (no Python, no torch; device memory from
 * the CUDA driver API on the primary context, which the library's runtime shares): 4 emulated
 * ranks, a
 * two-tensor model, constant gradients per rank chosen exactly representable in bf16, every
 * parameter 0.5.  The first AdamW step has a closed form (m = (1-b1) g, v = (1-b2) g^2, so
 * m / (sqrt(v) / sqrt(1-b2) + eps) = g / (|g| + eps / ...)); the 16-bit output must match it
 * within one bf16 ulp, and the step state must report t = 1.  Built and run by
 * tests/test_gpu_c_abi.py; prints "ok" on success. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda.h>

#include "zero.h"

#define ND 4
#define CHECK(x)                                                                 \
    do {                                                                         \
        int st_ = (int)(x);                                                      \
        if (st_ != 0) {                                                          \
            printf("FAIL %s -> %d: %s\n", #x, st_, zero_last_error());            \
            return 1;                                                            \
        }                                                                        \
    } while (0)
#define CUDA(x)                                                                  \
    do {                                                                         \
        CUresult e_ = (x);                                                       \
        if (e_ != CUDA_SUCCESS) {                                                \
            printf("FAIL %s: CUresult %d\n", #x, (int)e_);                        \
            return 1;                                                            \
        }                                                                        \
    } while (0)

static uint16_t bf16_of(float f) /* round to nearest even (finite values) */
{
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float float_of_bf16(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static void* dev_alloc(size_t bytes)
{
    CUdeviceptr d = 0;
    return cuMemAlloc(&d, bytes) == CUDA_SUCCESS ? (void*)(uintptr_t)d : NULL;
}

static CUdeviceptr dp(const void* p) { return (CUdeviceptr)(uintptr_t)p; }

int main(void)
{
    CUdevice dev;
    CUcontext ctx;
    CUDA(cuInit(0));
    CUDA(cuDeviceGet(&dev, 0));
    CUDA(cuDevicePrimaryCtxRetain(&ctx, dev));
    CUDA(cuCtxSetCurrent(ctx));
    const int64_t sizes[2] = {1000, 2344}; /* phi = 3344 = 4 x 836: no padding */
    zero_plan_t* plan = NULL;
    CHECK(zero_plan_create(sizes, 2, ND, 2, 0, NULL, 0, ZERO_BF16, &plan));
    zero_plan_info_t info;
    CHECK(zero_plan_info(plan, &info));
    const int64_t n = info.phi_pad;

    void* ws = dev_alloc((size_t)info.workspace_bytes);
    uint16_t* full16 = (uint16_t*)dev_alloc((size_t)n * 2);
    if (!ws || !full16) {
        printf("FAIL allocation\n");
        return 1;
    }
    float* state[ND][3][2];
    for (int r = 0; r < ND; ++r) {
        int64_t e = 0;
        CHECK(zero_rank_state_elems(plan, r, &e));
        float* ones = (float*)malloc((size_t)e * 4);
        for (int64_t i = 0; i < e; ++i) ones[i] = 0.5f;
        for (int k = 0; k < 3; ++k)
            for (int h = 0; h < 2; ++h) {
                state[r][k][h] = (float*)dev_alloc((size_t)e * 4);
                if (!state[r][k][h]) {
                    printf("FAIL allocation\n");
                    return 1;
                }
                if (k == 0 && h == 0)
                    CUDA(cuMemcpyHtoD(dp(state[r][k][h]), ones, (size_t)e * 4));
                else
                    CUDA(cuMemsetD8(dp(state[r][k][h]), 0, (size_t)e * 4));
            }
        free(ones);
        CHECK(zero_bind(plan, r, state[r][0], state[r][1], state[r][2], NULL, full16, ws));
    }
    /* rank r's gradient: (r + 1) * 2^-7 everywhere; the average is 10/4 * 2^-7 */
    void* grads[ND];
    uint16_t* host = (uint16_t*)malloc((size_t)n * 2);
    for (int r = 0; r < ND; ++r) {
        const uint16_t g = bf16_of((float)(r + 1) * 0.0078125f);
        for (int64_t i = 0; i < n; ++i) host[i] = g;
        grads[r] = dev_alloc((size_t)n * 2);
        if (!grads[r]) {
            printf("FAIL allocation\n");
            return 1;
        }
        CUDA(cuMemcpyHtoD(dp(grads[r]), host, (size_t)n * 2));
    }
    const zero_hyper_t h = {1e-3, 0.9, 0.999, 1e-8, 0.01, 0.0, 0};
    CHECK(zero_step(plan, (const void* const*)grads, ND, -1, &h, NULL));
    zero_step_result_t res;
    CHECK(zero_step_finish(plan, NULL, &res));
    if (res.t != 1 || res.skipped != 0) {
        printf("FAIL t = %lld skipped = %d\n", (long long)res.t, res.skipped);
        return 1;
    }
    CUDA(cuMemcpyDtoH(host, dp(full16), (size_t)n * 2));
    /* the first AdamW step in double: decay, then lr/(1-b1) * m / (sqrt(v)/sqrt(1-b2) + eps) */
    const double g = 2.5 * 0.0078125, b1 = 0.9, b2 = 0.999, lr = 1e-3, wd = 0.01, eps = 1e-8;
    const double m = (1 - b1) * g, v = (1 - b2) * g * g;
    double p = 0.5 - lr * wd * 0.5;
    p -= lr / (1 - b1) * (m / (sqrt(v) / sqrt(1 - b2) + eps));
    const float want = float_of_bf16(bf16_of((float)p));
    const float ulp = float_of_bf16(bf16_of((float)p) + 1) - want;
    for (int64_t i = 0; i < n; ++i) {
        const float got = float_of_bf16(host[i]);
        if (fabsf(got - want) > ulp * 1.0001f) {
            printf("FAIL element %lld: %.9g, want %.9g\n", (long long)i, got, want);
            return 1;
        }
    }
    zero_plan_destroy(plan);
    CUDA(cuDevicePrimaryCtxRelease(dev));
    printf("ok\n");
    return 0;
}
