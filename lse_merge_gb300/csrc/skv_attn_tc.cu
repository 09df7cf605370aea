// Tensor-core anchor attention of libskv for GB300 (sm_103a): tcgen05 MMA with
// TMEM accumulators, TMA-fed bf16 operands, warp-specialised roles.
//
// Forward [Split-KV §4.1 Eq. 3; Alg. 1 line 7 of "Split-KV: Efficient Context
// Parallelism for Training Diffusion Drafters"]: one thread block computes
// the partial (o_p, l_p) of one 128-row query tile, one head and one virtual
// rank p.  The key tiles it visits are the 128-key tiles of rank p's chunks
// that intersect the union of its rows' windows [s_i, a_i) (§3.1 Fig. 1);
// every other tile is never loaded.  Tiles inside every row's window are
// processed unmasked; only boundary tiles get the per-row compare.
//
// Roles (192 threads):
//   warps 0-3  softmax: thread r owns query row r; reads S from TMEM, online
//              max / exp2 / sum, writes bf16 P back to TMEM, rescales O when
//              the running max grows by more than 2^8, final o_p, l_p.
//   warp 4     MMA issuer (one thread): S = Q K^T (SS), O += P V (TS).
//   warp 5     TMA producer (one thread): Q once, K/V tiles through 2 stages.
// TMEM (512 columns): S double buffer [0,256), O [256,256+D), P double buffer
// (64 columns each, bf16 pairs) [384,512).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "skv_ptx.cuh"
#include "skv_tc.h"
#include "skv_tc_common.cuh"

namespace {

using namespace skv_ptx;
using namespace skv_tcc;

constexpr int kStages = 2;
constexpr int kFwdThreads = 192;
constexpr long long kTeardownWait = 2000000000LL;   // ns; in-flight copies / MMAs end in microseconds

template <int D>
struct __align__(1024) FwdSmem {
    __nv_bfloat16 q[D / 64][BM * 64];
    __nv_bfloat16 k[kStages][D / 64][BN * 64];
    __nv_bfloat16 v[kStages][D / 64][BN * 64];
    uint64_t q_full;
    uint64_t k_full[kStages], v_full[kStages], kv_empty[kStages];
    uint64_t s_full[2], p_full[2], o_done[2];
    uint64_t mma_fin;
    uint64_t stuck;             // never completed: target of the forced-timeout test mode
    uint32_t tmem_base;
    int abort_flag;
};

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_v, const int32_t* __restrict__ s,
                   const int32_t* __restrict__ a, int B, int64_t Qn, int H, int64_t S, int m,
                   float scale_log2, skv::RankCSR csr, float* __restrict__ o_part, float* __restrict__ lse_part,
                   int* status, long long wait_limit) {
    extern __shared__ unsigned char smem_raw[];
    FwdSmem<D>& sm = *reinterpret_cast<FwdSmem<D>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qt = blockIdx.x, h = blockIdx.y, p = blockIdx.z;
    constexpr int NP = D / 64;                       // 64-column panels per row
    constexpr uint32_t kTileBytes = BN * D * 2;      // one K or V tile (== Q tile)

    // test mode (negative limit): every block first waits on a barrier nothing
    // completes, so the timeout path runs deterministically
    const bool stuck_test = wait_limit < 0;
    if (stuck_test) wait_limit = -wait_limit;
    TileBounds tb = tile_bounds(s, a, B, Qn, S, qt);
    // once any block of the launch has timed out the result is void: the
    // remaining blocks skip their work instead of each waiting out a deadline
    if (*(volatile int*)status == SKV_ERR_TIMEOUT) tb.hi = tb.lo;

    if (tid == 0) {
        mbar_init(&sm.q_full, 1);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sm.k_full[i], 1);
            mbar_init(&sm.v_full[i], 1);
            mbar_init(&sm.kv_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.s_full[i], 1);
            mbar_init(&sm.p_full[i], 128);
            mbar_init(&sm.o_done[i], 1);
        }
        mbar_init(&sm.mma_fin, 1);
        mbar_init(&sm.stuck, 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 4) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    const uint32_t tS = tmem, tO = tmem + 256, tP = tmem + 384;

    TileIter it;
    it.init(csr, p, p + 1, m, tb.lo, tb.hi);

    if (warp == 5) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensormap(&map_q);
            prefetch_tensormap(&map_k);
            prefetch_tensormap(&map_v);
            int n = 0;
            int64_t x0;
            bool any = false;
            while (it.next(x0)) {
                if (!any) {
                    mbar_arrive_expect_tx(&sm.q_full, kTileBytes);
                    for (int c = 0; c < NP; ++c) tma_load_2d(sm.q[c], &map_q, &sm.q_full, h * D + c * 64, qt * BM);
                    any = true;
                }
                const int st = n % kStages;
                if (n >= kStages) {
                    if (!mbar_wait(&sm.kv_empty[st], ((n - kStages) / kStages) & 1, wait_limit, &sm.abort_flag)) {
                        atomicExch(&sm.abort_flag, 1);
                        skv::raise_status(status, SKV_ERR_TIMEOUT);
                        break;
                    }
                }
                if (*(volatile int*)&sm.abort_flag) break;
                mbar_arrive_expect_tx(&sm.k_full[st], kTileBytes);
                for (int c = 0; c < NP; ++c)
                    tma_load_2d(sm.k[st][c], &map_k, &sm.k_full[st], h * D + c * 64, (int)x0);
                mbar_arrive_expect_tx(&sm.v_full[st], kTileBytes);
                for (int c = 0; c < NP; ++c)
                    tma_load_2d(sm.v[st][c], &map_v, &sm.v_full[st], h * D + c * 64, (int)x0);
                ++n;
            }
            // every load this thread issued has landed before the block exits
            if (any) mbar_wait(&sm.q_full, 0, kTeardownWait);
            for (int st = 0; st < kStages && st < n; ++st) {
                const int last = st + ((n - 1 - st) / kStages) * kStages;   // last tile using stage st
                mbar_wait(&sm.k_full[st], (last / kStages) & 1, kTeardownWait);
                mbar_wait(&sm.v_full[st], (last / kStages) & 1, kTeardownWait);
            }
        }
    } else if (warp == 4) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(BM, BN, 0, 0);
            constexpr uint32_t idO = idesc_bf16_f32(BM, D, 0, 1);
            int64_t x0;
            int T = 0;
            {
                TileIter cnt = it;
                while (cnt.next(x0)) ++T;
            }
            bool ok = true;
            bool issued = false;   // any MMA in flight to wait for before TMEM is freed
            auto fail = [&]() {
                atomicExch(&sm.abort_flag, 1);
                skv::raise_status(status, SKV_ERR_TIMEOUT);
                ok = false;
            };
            if (stuck_test && !mbar_wait(&sm.stuck, 0, wait_limit, &sm.abort_flag)) fail();
            auto issue_s = [&](int n) {
                const int st = n % kStages;
                if (!mbar_wait(&sm.k_full[st], (n / kStages) & 1, wait_limit, &sm.abort_flag)) { fail(); return; }
                tc_fence_after();
                const uint32_t dS = tS + (n & 1) * BN;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk & 3) * 32;
                    const uint64_t ad = smem_desc(smem_u32(sm.q[kk >> 2]) + off, 16, 1024);
                    const uint64_t bd = smem_desc(smem_u32(sm.k[st][kk >> 2]) + off, 16, 1024);
                    mma_ss(dS, ad, bd, idS, kk > 0);
                }
                issued = true;
                mma_commit(&sm.s_full[n & 1]);
            };
            if (T > 0 && ok) {
                if (!mbar_wait(&sm.q_full, 0, wait_limit, &sm.abort_flag)) fail();
                if (ok) issue_s(0);
                for (int n = 0; n < T && ok; ++n) {
                    if (*(volatile int*)&sm.abort_flag) { ok = false; break; }
                    if (n + 1 < T) {
                        issue_s(n + 1);
                        if (!ok) break;
                    }
                    const int st = n % kStages;
                    if (!mbar_wait(&sm.p_full[n & 1], (n >> 1) & 1, wait_limit, &sm.abort_flag)) { fail(); break; }
                    if (!mbar_wait(&sm.v_full[st], (n / kStages) & 1, wait_limit, &sm.abort_flag)) { fail(); break; }
                    tc_fence_after();
                    const uint32_t aP = tP + (n & 1) * 64;
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk) {
                        const uint64_t bd = smem_desc(smem_u32(sm.v[st][0]) + kk * 2048, BN * 128, 1024);
                        mma_ts(tO, aP + kk * 8, bd, idO, (n > 0 || kk > 0) ? 1u : 0u);
                    }
                    issued = true;
                    mma_commit(&sm.o_done[n & 1]);
                    mma_commit(&sm.kv_empty[st]);
                }
            }
            // all MMAs this thread issued have completed before TMEM is freed
            // (a commit is only made when there is an MMA to track)
            if (issued) {
                mma_commit(&sm.mma_fin);
                if (!mbar_wait(&sm.mma_fin, 0, kTeardownWait)) skv::raise_status(status, SKV_ERR_TIMEOUT);
            }
        }
    } else {
        // ------------------------------------------------------------ softmax
        // tcgen05.ld/st are warp-collective: every branch around them is made
        // warp-uniform (__any_sync / __all_sync); per-row choices are data.
        constexpr unsigned kAll = 0xffffffffu;
        const int r = tid;                         // row inside the tile == TMEM lane
        const int64_t row = int64_t(qt) * BM + r;
        const bool live = row < Qn;
        int64_t rlo = 0, rhi = 0;
        if (live) skv::block_window(s, a, (int)(row / B), S, rlo, rhi);
        const uint32_t lane_base = uint32_t(warp * 32) << 16;
        float m_ref = -INFINITY, l = 0.f;
        int o_waited = 0;
        bool ok = true;
        auto uniform_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
            const bool got = mbar_wait_warp(bar, parity, wait_limit, &sm.abort_flag);
            if (!got && lane == 0) {
                atomicExch(&sm.abort_flag, 1);
                skv::raise_status(status, SKV_ERR_TIMEOUT);
            }
            return got;
        };
        auto wait_o = [&](int need) {
            while (ok && o_waited < need) {
                if (!uniform_wait(&sm.o_done[o_waited & 1], (o_waited >> 1) & 1)) {
                    ok = false;
                    break;
                }
                ++o_waited;
            }
        };
        int64_t x0;
        int n = 0;
        while (ok && it.next(x0)) {
            if (__any_sync(kAll, *(volatile int*)&sm.abort_flag != 0)) { ok = false; break; }
            if (!uniform_wait(&sm.s_full[n & 1], (n >> 1) & 1)) { ok = false; break; }
            tc_fence_after();
            float sc[BN];
            {
                uint32_t raw[BN / 32][32];               // all chunks in flight before one wait
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) tmem_ld32(tS + (n & 1) * BN + lane_base + c * 32, raw[c]);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < BN / 32; ++c)
#pragma unroll
                    for (int j = 0; j < 32; ++j) sc[c * 32 + j] = __uint_as_float(raw[c][j]);
            }
            const bool full = (x0 >= tb.flo) && (x0 + BN <= tb.fhi);
            if (!full) {
#pragma unroll
                for (int j = 0; j < BN; ++j) {
                    const int64_t x = x0 + j;
                    if (x < rlo || x >= rhi) sc[j] = -INFINITY;
                }
            }
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < BN; ++j) mx = fmaxf(mx, sc[j]);
            const float mx_s = mx * scale_log2;
            bool rescale = false;
            float alpha = 1.f;
            if (mx_s > m_ref + 8.f) {
                alpha = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - mx_s);
                rescale = (l > 0.f);
                m_ref = mx_s;
            }
            const bool warp_rescale = __any_sync(kAll, rescale);
            // P buffer n&1 was last read by PV_{n-2}; O must be final before a rescale
            wait_o(warp_rescale ? n : n - 1);
            if (!ok) break;
            if (warp_rescale) {
                const float f = rescale ? alpha : 1.f;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t rr[32];
                    tmem_ld32(tO + lane_base + c * 32, rr);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) rr[j] = __float_as_uint(__uint_as_float(rr[j]) * f);
                    tmem_st32(tO + lane_base + c * 32, rr);
                }
            }
            l *= alpha;
            float sum = 0.f;
            const float neg = (m_ref == -INFINITY) ? 0.f : -m_ref;
#pragma unroll
            for (int c = 0; c < BN / 64; ++c) {
                uint32_t pk[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float z0 = sc[c * 64 + 2 * j], z1 = sc[c * 64 + 2 * j + 1];
                    const float p0 = (z0 == -INFINITY) ? 0.f : ex2(fmaf(z0, scale_log2, neg));
                    const float p1 = (z1 == -INFINITY) ? 0.f : ex2(fmaf(z1, scale_log2, neg));
                    sum += p0 + p1;
                    pk[j] = pack_bf16(p0, p1);
                }
                tmem_st32(tP + (n & 1) * 64 + lane_base + c * 32, pk);
            }
            l += sum;
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sm.p_full[n & 1]);
            ++n;
        }
        wait_o(n);
        const bool aborted = __any_sync(kAll, *(volatile int*)&sm.abort_flag != 0);
        if (ok && !aborted) {
            const bool mine = live && l > 0.f;
            const float inv = mine ? 1.f / l : 0.f;
            float* dst = o_part + ((int64_t(p) * Qn + row) * H + h) * D;
            if (n > 0 && __any_sync(kAll, mine)) {
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t rr[32];
                    tmem_ld32(tO + lane_base + c * 32, rr);
                    tmem_ld_wait();
                    if (mine) {
#pragma unroll
                        for (int j = 0; j < 32; j += 4) {
                            float4 v4 = make_float4(__uint_as_float(rr[j]) * inv, __uint_as_float(rr[j + 1]) * inv,
                                                    __uint_as_float(rr[j + 2]) * inv,
                                                    __uint_as_float(rr[j + 3]) * inv);
                            __stcs(reinterpret_cast<float4*>(dst + c * 32 + j), v4);
                        }
                    }
                }
            }
            if (live)
                lse_part[(int64_t(p) * Qn + row) * H + h] =
                    mine ? (m_ref + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D>
skv_status launch_fwd(const skv_problem& pb, const void* q, const void* k, const void* v, skv::RankCSR csr,
                      float* o_part, float* lse_part, const skv_host::Ctx& c) {
    const int64_t Qn = int64_t(pb.n_blocks) * pb.B;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, q, Qn, int64_t(pb.n_heads) * D) || !make_map(&mk, k, pb.S, int64_t(pb.n_heads) * D) ||
        !make_map(&mv, v, pb.S, int64_t(pb.n_heads) * D))
        return SKV_ERR_CUDA;
    size_t smem = sizeof(FwdSmem<D>) + 1024;
    if (smem < 120 * 1024) smem = 120 * 1024;   // one block per SM: it owns all 512 TMEM columns
    auto kern = attn_fwd_tc_kernel<D>;
    SKV_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    const dim3 grid((unsigned)((Qn + BM - 1) / BM), (unsigned)pb.n_heads, (unsigned)pb.P);
    const float scale_log2 = pb.scale * 1.4426950408889634f;
    skv_host::timer_begin(skv_host::kTimeFwd, c.stream);
    kern<<<grid, kFwdThreads, smem, c.stream>>>(mq, mk, mv, pb.s, pb.a, pb.B, Qn, pb.n_heads, pb.S, pb.m, scale_log2,
                                                csr, o_part, lse_part, c.status, c.wait_limit);
    skv_host::timer_end(skv_host::kTimeFwd, c.stream);
    SKV_LAUNCHED();
    return SKV_OK;
}

}  // namespace

namespace skv_tc {

bool fwd_supported(const skv_problem& pb) {
    return pb.dtype == SKV_BF16 && (pb.head_dim == 64 || pb.head_dim == 128) && pb.m % BN == 0 &&
           pb.P <= 65535 && pb.n_heads <= 65535;
}
size_t fwd_scratch_bytes(const skv_problem&) { return 0; }

skv_status launch_attn_fwd_tc(const skv_problem& pb, const void* q, const void* k, const void* v, skv::RankCSR csr,
                              float* o_part, float* lse_part, void*, const skv_host::Ctx& c) {
    if (pb.head_dim == 128) return launch_fwd<128>(pb, q, k, v, csr, o_part, lse_part, c);
    return launch_fwd<64>(pb, q, k, v, csr, o_part, lse_part, c);
}

}  // namespace skv_tc
