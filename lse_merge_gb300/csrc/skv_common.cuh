// Shared device helpers of libskv (sm_103a).  Internal; not part of the ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "skv.h"

namespace skv {

// Device status word codes (a subset of skv_status).  Kernels record the first
// error they see with atomicCAS; skv_stream_status reads and clears it.
__device__ __forceinline__ void raise_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float load(const float* p) { return *p; }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16* p) { return __bfloat162float(*p); }
};

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// Per-rank chunk lists in CSR form, built on the device from rank_of_chunk:
// rank p holds chunks list[ptr[p] .. ptr[p+1]), ascending.
struct RankCSR {
    const int32_t* ptr;    // [P+1]
    const int32_t* list;   // [n_chunks]
};

__host__ __device__ __forceinline__ int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Clamped window [s, a) of block i inside [0, S).
__device__ __forceinline__ void block_window(const int32_t* s, const int32_t* a, int i, int64_t S,
                                             int64_t& lo, int64_t& hi) {
    int64_t si = s[i], ai = a[i];
    si = si < 0 ? 0 : (si > S ? S : si);
    ai = ai < si ? si : (ai > S ? S : ai);
    lo = si;
    hi = ai;
}

}  // namespace skv

// Host-side launch helpers shared by the translation units.
namespace skv_host {

struct Ctx {
    int* status;          // device status word of the current device
    cudaStream_t stream;
    int num_sms;
    long long wait_limit; // iteration cap of bounded device waits
};

// Returns SKV_OK and fills ctx, or SKV_ERR_CUDA.
skv_status get_ctx(void* stream, Ctx& ctx);

// Counts one kernel launch of this library (skv_launch_count).
void note_launch(int n = 1);

// Optional per-kernel CUDA-event timing (skv_set_kernel_timing): slots of the
// main kernels; begin/end record events on the launching stream when enabled.
enum TimerSlot { kTimeFwd = 0, kTimeMerge = 1, kTimeBwdKV = 2, kTimeBwdQ = 3, kTimeLocalFwd = 4, kTimeLocalBwd = 5,
                 kTimeOproj = 6, kTimeSlots = 7 };
void timer_begin(int slot, cudaStream_t stream);
void timer_end(int slot, cudaStream_t stream);

// Workspace layout helpers (byte offsets, 256-byte aligned).
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace skv_host

// Checks the launch just made and counts it.
#define SKV_LAUNCHED()                                         \
    do {                                                       \
        cudaError_t _e = cudaGetLastError();                   \
        if (_e != cudaSuccess) return SKV_ERR_CUDA;            \
        skv_host::note_launch();                               \
    } while (0)

#define SKV_CUDA_CHECK(expr)                                   \
    do {                                                       \
        cudaError_t _e = (expr);                               \
        if (_e != cudaSuccess) return SKV_ERR_CUDA;            \
    } while (0)
