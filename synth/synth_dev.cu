// Device side of the synthetic input generator: fills device buffers with the
// streams defined in synth_core.h (bit-identical to the host fill).  Input
// preparation only; it runs outside any timed region.
#include <cuda_runtime.h>

#include "synth_core.h"

namespace {

__global__ void __launch_bounds__(256) syn_fill_kernel(uint16_t* __restrict__ dst, int64_t n,
                                                       int64_t start, syn_stream_t s)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride)
        dst[j] = syn_value(&s, (uint64_t)(start + j));
}

}  // namespace

extern "C" {

// dst[j] = value(start + j) for j in [0, n); asynchronous on `stream`.
int syn_fill_device(void* dst, int64_t n, int64_t start, uint64_t seed, uint64_t workload,
                    uint64_t kind, uint64_t step, uint64_t rank, double sigma, int dtype,
                    int outliers, int64_t inject_index, uint32_t inject_bits, void* stream)
{
    if (n < 0 || (n > 0 && dst == nullptr)) return 1;
    if (n == 0) return 0;
    const syn_stream_t s = syn_make_stream(seed, workload, kind, step, rank, sigma, dtype,
                                           outliers, inject_index, inject_bits);
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 2;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 2;
    int64_t blocks = (n + 255) / 256;
    const int64_t cap = (int64_t)sms * 16;
    if (blocks > cap) blocks = cap;
    syn_fill_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>((uint16_t*)dst, n, start, s);
    return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

}  // extern "C"
