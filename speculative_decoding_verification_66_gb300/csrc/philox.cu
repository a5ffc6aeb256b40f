// philox.cu -- sv_philox: the device Philox4x32-10 generator evaluated for
// caller-chosen counters, so that it can be checked word for word against an
// independent implementation of its published definition (Salmon, Moraes,
// Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11). The
// verification kernels call the same device function (sv_device.cuh).
#include "spec_verify.h"
#include "sv_device.cuh"

#define SV_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

constexpr int kPhiloxThreads = 256;

__global__ void __launch_bounds__(kPhiloxThreads) philox_kernel(uint2 key, const uint4* ctr, uint4* out,
                                                                int64_t n)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
        out[i] = sv::philox4x32_10(ctr[i], key);
}

}  // namespace

SV_EXPORT int sv_philox(uint64_t seed, const uint32_t* counters, uint32_t* out, int64_t n, void* stream)
{
    if (n < 0) return SV_ERR_ARG;
    if (n >= (int64_t(1) << 40)) return SV_ERR_SIZE;
    if (n == 0) return SV_OK;
    if (counters == nullptr || out == nullptr) return SV_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(counters) | reinterpret_cast<uintptr_t>(out)) % 16 != 0)
        return SV_ERR_ALIGN;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return SV_ERR_CUDA;
    const int64_t need = (n + kPhiloxThreads - 1) / kPhiloxThreads;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    const unsigned grid = static_cast<unsigned>(need < cap ? need : cap);
    const uint2 key = make_uint2(static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
    philox_kernel<<<grid, kPhiloxThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        key, reinterpret_cast<const uint4*>(counters), reinterpret_cast<uint4*>(out), n);
    return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
