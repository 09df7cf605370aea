// skv_attn_fwd_static: the per-rank forward partials without a caller-supplied
// workspace.  Its scratch (the per-rank chunk lists the forward builds before
// the attention kernel runs) lives in a fixed array in device memory that
// every device holds from the moment the library loads until the process
// exits, so a call allocates nothing.
//
// Who needs it: callers that are not allowed to allocate device memory.  A
// plug-in running inside a host framework that owns the whole device memory
// pool gets only its input and output buffers; a latency-critical loop cannot
// afford cudaMalloc, which may synchronise the device and stall every other
// stream; a runtime with a fixed memory budget cannot grow it per call.
#include <mutex>

#include "skv_common.cuh"

// Capacity of the static scratch: 128 KiB (the chunk lists of a plan with 16384
// chunks over 1024 ranks plus the key bounds of 3800 query tiles fit).
constexpr size_t kStaticScratchBytes = 131072;

static __device__ __align__(256) unsigned char g_fwd_static_scratch[kStaticScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch on the current device, looked up once per
// device (host code must not use the symbol itself: it names a host-side
// stand-in, not device memory).
skv_status static_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SKV_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SKV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (!g_static_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_fwd_static_scratch) != cudaSuccess || p == nullptr) return SKV_ERR_CUDA;
        g_static_ptr[dev] = p;
    }
    *out = g_static_ptr[dev];
    return SKV_OK;
}

}  // namespace

extern "C" {

skv_status skv_attn_fwd_static(const skv_problem* prob, const void* q, const void* k, const void* v,
                               const int32_t* rank_of_chunk, float* o_part, float* lse_part, void* stream) {
    const size_t need = skv_workspace_bytes(prob, 0);
    if (need == 0) {
        // invalid problem: let the regular entry point report the precise status
        return skv_attn_fwd(prob, q, k, v, rank_of_chunk, o_part, lse_part, nullptr, 0, stream);
    }
    if (need > kStaticScratchBytes) return SKV_ERR_WORKSPACE;
    void* scratch = nullptr;
    const skv_status st = static_scratch(&scratch);
    if (st != SKV_OK) return st;
    return skv_attn_fwd(prob, q, k, v, rank_of_chunk, o_part, lse_part, scratch, kStaticScratchBytes, stream);
}

}  // extern "C"
