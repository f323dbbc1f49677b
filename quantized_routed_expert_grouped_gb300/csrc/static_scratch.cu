// static_scratch.cu - moe_expert_grouped_static: the expert call with its scratch (gate/up rows
// and q8_1 h rows) in a static device buffer, for callers that cannot allocate device memory.
// The buffer is declared here, its device address is looked up once per device with that device
// current, and the existing moe_expert_grouped runs on it; nothing is allocated.
#include <mutex>

#include "internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[MOE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {nullptr};

size_t round256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// Device address of this device's copy of the buffer (looked up on the first call per device).
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_E_CUDA;
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return MOE_E_CUDA;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" int moe_expert_grouped_static(const moe_expert_call* call, cudaStream_t stream) {
    if (!call) return MOE_E_NULL;
    if (call->cap_entries <= 0 || call->n_ff <= 0 || call->n_ff % 32) return call->cap_entries <= 0 ? MOE_E_CAP
                                                                                                     : MOE_E_SHAPE;
    const size_t gu_bytes = round256(static_cast<size_t>(call->cap_entries) * 2 * call->n_ff * sizeof(float));
    const size_t hq_bytes = round256(static_cast<size_t>(call->cap_entries) * (call->n_ff / 32) * sizeof(moe_q8_1));
    if (gu_bytes + hq_bytes > MOE_STATIC_SCRATCH_BYTES) return MOE_E_SCRATCH;
    void* base = nullptr;
    const int rc = scratch_address(&base);
    if (rc != MOE_OK) return rc;
    moe_expert_call c = *call;
    c.gu = static_cast<float*>(base);
    c.hq = reinterpret_cast<moe_q8_1*>(static_cast<unsigned char*>(base) + gu_bytes);
    return moe_expert_grouped(&c, stream);
}
