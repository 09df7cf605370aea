// The LSE merge with the output projection [Split-KV §4.1, Eq. 5; the MERGE_AR,
// OProj and RS_sum steps of Alg. 1's forward in "Split-KV: Efficient Context
// Parallelism for Training Diffusion Drafters"]: Y = sum_p OProj(o_bar_p) with
// o_bar_p = exp(l_p - l) o_p and OProj(x) = x W_o^T over the concatenated heads.
//
// Eq. 5 is linear in the partials, so on one device the sum is taken first: the
// merge kernel writes the merged o (bf16, the tensor the backward reads anyway)
// and a tcgen05 GEMM projects it, Y = o W_o^T.  The GEMM reads o back while it
// is still warm in L2 for most tiles; a merge inside the GEMM's operand loads
// would instead re-read the fp32 partials once per 256 output columns.
//
// GEMM tile: 128 rows x 256 output columns, K in steps of 64 through a
// four-stage TMA ring (A: 128 x 64 of o, B: 256 x 64 of W_o, 128-byte swizzle).
// Roles (192 threads): warp 0 TMA producer, warp 1 MMA issuer (one elected
// lane), warps 2-5 epilogue (TMEM -> registers -> Y, fp32).  One 256-column
// TMEM accumulator per block.
#include <cuda.h>

#include "skv_internal.h"
#include "skv_ptx.cuh"
#include "skv_tc_common.cuh"

namespace {

using namespace skv_ptx;
using namespace skv_tcc;

constexpr int kOpThreads = 192;
constexpr int kOpStages = 4;
constexpr int kOpN = 256;                          // output columns per block
constexpr int kOpK = 64;                           // K per stage (one 128-byte swizzle row)
constexpr long long kTeardownWait = 2000000000LL;  // ns

struct __align__(1024) OpSmem {
    __nv_bfloat16 a[kOpStages][BM * kOpK];        // 16 KiB a stage
    __nv_bfloat16 b[kOpStages][kOpN * kOpK];      // 32 KiB a stage (two 128-row boxes)
    uint64_t full[kOpStages], empty[kOpStages], acc_full;
    uint32_t tmem_base;
    int abort_flag;
};

__global__ void __launch_bounds__(kOpThreads, 1)
oproj_gemm_kernel(const __grid_constant__ CUtensorMap map_o, const __grid_constant__ CUtensorMap map_w, int64_t Qn,
                  int d_model, int nk, float* __restrict__ y, int* status, long long wait_limit) {
    extern __shared__ unsigned char smem_raw[];
    OpSmem& sm = *reinterpret_cast<OpSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * kOpN;
    const int64_t m0 = int64_t(blockIdx.y) * BM;
    int n_k = nk;
    if (*(volatile int*)status == SKV_ERR_TIMEOUT) n_k = 0;   // launch already void: skip the work

    if (threadIdx.x == 0) {
        for (int i = 0; i < kOpStages; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], 1);
        }
        mbar_init(&sm.acc_full, 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, kOpN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    auto abort_now = [&]() {
        atomicExch(&sm.abort_flag, 1);
        skv::raise_status(status, SKV_ERR_TIMEOUT);
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && n_k > 0) {
            prefetch_tensormap(&map_o);
            prefetch_tensormap(&map_w);
            int issued = 0;
            for (int kc = 0; kc < n_k; ++kc) {
                const int st = kc % kOpStages;
                if (kc >= kOpStages &&
                    !mbar_wait(&sm.empty[st], ((kc - kOpStages) / kOpStages) & 1, wait_limit, &sm.abort_flag)) {
                    abort_now();
                    break;
                }
                mbar_arrive_expect_tx(&sm.full[st], (BM + kOpN) * kOpK * 2);
                tma_load_2d(sm.a[st], &map_o, &sm.full[st], kc * kOpK, (int)m0);
                tma_load_2d(sm.b[st], &map_w, &sm.full[st], kc * kOpK, n0);
                tma_load_2d(sm.b[st] + 128 * kOpK, &map_w, &sm.full[st], kc * kOpK, n0 + 128);
                ++issued;
            }
            // every copy issued has landed before the block exits
            for (int st = 0; st < kOpStages && st < issued; ++st) {
                const int last = st + ((issued - 1 - st) / kOpStages) * kOpStages;
                mbar_wait(&sm.full[st], (last / kOpStages) & 1, kTeardownWait);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (n_k > 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(BM, kOpN, 0, 0);
            const uint64_t da = smem_desc(smem_u32(sm.a[0]), 16, 1024);
            const uint64_t db = smem_desc(smem_u32(sm.b[0]), 16, 1024);
            constexpr uint32_t kAst = BM * kOpK * 2 / 16, kBst = kOpN * kOpK * 2 / 16;   // stage strides (x16 B)
            bool ok = true;
            for (int kc = 0; kc < n_k; ++kc) {
                const int st = kc % kOpStages;
                if (!mbar_wait_warp(&sm.full[st], (kc / kOpStages) & 1, wait_limit, &sm.abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < kOpK / 16; ++kk)
                        mma_ss(tmem, da + (st * kAst + kk * 2), db + (st * kBst + kk * 2), idesc,
                               (kc > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&sm.empty[st]);
                }
                __syncwarp();
            }
            if (!ok && lane == 0) abort_now();
            if (elect_one()) mma_commit(&sm.acc_full);
            __syncwarp();
            // nothing of this block's may still be in flight when its TMEM is freed
            if (!mbar_wait_warp(&sm.acc_full, 0, kTeardownWait) && lane == 0)
                skv::raise_status(status, SKV_ERR_TIMEOUT);
        }
    } else {
        // ------------------------------------------------------------ epilogue warps 2-5
        const int quad = warp & 3;                        // TMEM lanes [32 quad, +32)
        const int64_t row = m0 + quad * 32 + lane;
        const uint32_t lane_base = uint32_t(quad * 32) << 16;
        if (n_k > 0 && mbar_wait_warp(&sm.acc_full, 0, wait_limit + kTeardownWait, &sm.abort_flag) &&
            !__any_sync(0xffffffffu, *(volatile int*)&sm.abort_flag != 0)) {
            tc_fence_after();
            float* yr = y + row * d_model;
#pragma unroll 1
            for (int c = 0; c < kOpN / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + c * 32, v);
                tmem_ld_wait();
                const int col0 = n0 + c * 32;
                if (row < Qn) {
                    if (col0 + 32 <= d_model) {
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            __stcs(reinterpret_cast<float4*>(yr + col0 + j),
                                   make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                               __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3])));
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            if (col0 + j < d_model)   // d_model is a multiple of 16
                                __stcs(reinterpret_cast<float4*>(yr + col0 + j),
                                       make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                                   __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3])));
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kOpN);
    }
}

}  // namespace

namespace skv_internal {

skv_status launch_oproj(const void* o, int64_t Qn, int hd, const void* w_o, int d_model, float* y,
                        const skv_host::Ctx& c) {
    if (Qn == 0) return SKV_OK;
    CUtensorMap mo, mw;
    if (!skv_tcc::make_map(&mo, o, Qn, hd) || !skv_tcc::make_map(&mw, w_o, d_model, hd)) return SKV_ERR_CUDA;
    const size_t smem = sizeof(OpSmem) + 1024;
    SKV_CUDA_CHECK(cudaFuncSetAttribute(oproj_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    const dim3 grid((unsigned)((d_model + kOpN - 1) / kOpN), (unsigned)((Qn + BM - 1) / BM));
    skv_host::timer_begin(skv_host::kTimeOproj, c.stream);
    oproj_gemm_kernel<<<grid, kOpThreads, smem, c.stream>>>(mo, mw, Qn, d_model, hd / kOpK, y, c.status,
                                                            c.wait_limit < 0 ? -c.wait_limit : c.wait_limit);
    skv_host::timer_end(skv_host::kTimeOproj, c.stream);
    SKV_LAUNCHED();
    return SKV_OK;
}

}  // namespace skv_internal
