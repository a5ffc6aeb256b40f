// sv_static.cu -- spec_verify_static: the verification call for callers that
// cannot allocate device memory.
//
// Some callers cannot call cudaMalloc:
//  * code running inside a host framework that owns every device allocation
//    (a caching allocator or a fixed memory pool), where a stray cudaMalloc
//    fails once the pool holds the memory, or breaks the framework's
//    accounting;
//  * code on a latency-critical path, where cudaMalloc / cudaFree would
//    synchronise the device.
// Such callers still pass their own input and output buffers, but they have no
// workspace to give. This entry point uses a fixed scratch array that lives in
// the library's own device image instead.
//
// The scratch array is a file-scope __device__ array of kStaticScratchBytes.
// Every GPU that loads the library holds it until the process exits. Host code
// cannot use the array's name as a device address, so the address is looked up
// with cudaGetSymbolAddress, once per device, with that device current.
#include <mutex>

#include "spec_verify.h"

#define SV_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

// 8 MiB covers the headline case (B=256, K=8, V=128256) about ten times over.
constexpr size_t kStaticScratchBytes = size_t(8) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device; the first call on each
// device does the lookup. The cached address belongs to the device's primary
// context as it was at that lookup: after cudaDeviceReset (or anything else
// that destroys and recreates the primary context) the library's module is
// loaded again at a new address, so the library must be unloaded and loaded
// again before spec_verify_static is called on that device.
int scratch_address(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return SV_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return SV_OK;
}

}  // namespace

SV_EXPORT int spec_verify_static(const void* target_logits, const void* draft_logits,
                                 const int32_t* draft_tokens, int64_t B, int64_t K, int64_t V,
                                 int dtype, float temperature, uint64_t seed, int mode,
                                 int32_t* out_tokens, int32_t* num_accepted, void* stream)
{
    if (B == 0) {
        return spec_verify(target_logits, draft_logits, draft_tokens, B, K, V, dtype, temperature,
                           seed, mode, out_tokens, num_accepted, nullptr, 0, stream);
    }
    size_t need = 0;
    int rc = sv_workspace_bytes(B, K, V, dtype, mode, &need);
    if (rc != SV_OK) return rc;
    if (need > kStaticScratchBytes) return SV_ERR_SIZE;
    void* scratch = nullptr;
    rc = scratch_address(&scratch);
    if (rc != SV_OK) return rc;
    // Nothing in the scratch has to start at zero: spec_verify writes every
    // region of its workspace (pass-1 partials, sequence records, race-block
    // sums) before it reads it within the same call, and it keeps no counters
    // there.
    return spec_verify(target_logits, draft_logits, draft_tokens, B, K, V, dtype, temperature,
                       seed, mode, out_tokens, num_accepted, scratch, kStaticScratchBytes, stream);
}
