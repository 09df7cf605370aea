// Tensor-core backward of the anchor attention (tcgen05 + TMEM + TMA), sm_103a.
//
// "Split-KV: Efficient Context Parallelism for Training Diffusion Drafters",
// Alg. 1 lines 15-17 in merged form: with the global log-sum-exp l_r and
// D_r = dO_r . o_r, every rank's score gradient is dS = P (dP - D) with
// P = exp(z - l).  Each virtual rank p owns the key tiles of its chunks, so
// its dk_p / dv_p rows are written by exactly one thread block each, and its
// dq^(p) contributions are summed into dq by fp32 reduction adds (the
// reduce-scatter of Alg. 1 line 17 made local).
//
// Key-stationary: one thread block owns a 128-key tile and one head and walks
// the 128-row query tiles whose windows meet the tile (the tile-skip list
// built by skv_kv_list_kernel; masked-out query tiles are never loaded).  Per
// query tile t (TMEM lane = key for S^T, dP^T, dV, dK; = query row for dQ):
//   S^T  = K Q_t^T          (SS)  -> TMEM A [0,128)
//   dP^T = V dO_t^T         (SS)  -> TMEM B [128,256)
//   compute warps: P^T = exp2(S^T scale log2e - l2), bf16 P^T -> TMEM A[0,64);
//                  dS^T = P^T (dP^T - D), bf16 -> shared memory (swizzled)
//   dV  += P^T dO_t         (TS)  -> TMEM [256, 256+D)
//   dK  += dS^T Q_t         (SS)  -> TMEM [384, 384+D)
//   dQ_t = dS K             (SS, dS^T read MN-major) -> TMEM B
//   compute warps: dq[rows] += scale dQ_t (red.global.add.v4.f32)
// Roles (192 threads): warps 0-3 compute, warp 4 MMA issuer, warp 5 TMA.
#include <cuda.h>
#include <math.h>

#include "skv_ptx.cuh"
#include "skv_tc.h"
#include "skv_tc_common.cuh"

namespace {

using namespace skv_ptx;
using namespace skv_tcc;

constexpr int kBwdThreads = 448;                     // WG1 warps 0-7, WG2 warps 8-11, MMA 12, TMA 13
constexpr int kMmaWarp = 12, kTmaWarp = 13;
constexpr int kSmemMax = 232448;                     // sm_100-family opt-in maximum per block
constexpr long long kTeardownWait = 2000000000LL;    // ns

template <int D>
struct BwdTiles {                                    // 1024-byte aligned (128-byte swizzle atoms)
    __nv_bfloat16 k[D / 64][BN * 64];
    __nv_bfloat16 v[D / 64][BN * 64];
    __nv_bfloat16 q[2][D / 64][BM * 64];
    __nv_bfloat16 dO[2][D / 64][BM * 64];
    __nv_bfloat16 ds[2][BN * 64];                    // dS^T [key][q], two 64-query panels
};

struct BwdMeta {                                     // per query tile, loaded with its Q/dO stage
    float lse2[BM];
    float D[BM];
    int4 bnd;                                        // the tile's key bounds (written by the producer)
    int qt;                                          // the query tile index
    int pad_[3];
};

struct BwdBars {
    uint64_t kv_full, qd_full[2], qd_empty[2], s_full, dp_full, ds_full, dq_full, dq_free, mma_fin;
    uint64_t stuck;                                  // never completed: target of the forced-timeout test mode
    uint32_t tmem_base;
    int abort_flag;
};

template <int D>
struct BwdSmem {
    BwdTiles<D> t;
    BwdMeta meta[2];
    BwdBars b;
};

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void red_add4(float* p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}


// ---------------------------------------------------------------- tile lists

// Per query tile: union (lo, hi) and full-visibility (flo, fhi) key bounds.
__global__ void qtile_bounds_kernel(const int32_t* __restrict__ s, const int32_t* __restrict__ a, int B, int64_t Qn,
                                    int64_t S, int n_qt, int4* __restrict__ out) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= n_qt) return;
    const TileBounds tb = tile_bounds(s, a, B, Qn, S, t);
    out[t] = make_int4((int)tb.lo, (int)tb.hi, (int)tb.flo, (int)tb.fhi);
}

// Tile-skip lists: for key tile k, the ascending query tiles whose union window
// meets [128k, 128k+128).  One warp per key tile; fixed capacity n_qt per list.
__global__ void kv_list_kernel(const int4* __restrict__ qtb, int n_qt, int n_kv, int32_t* __restrict__ cnt,
                               int32_t* __restrict__ list) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= n_kv) return;
    const int64_t x0 = int64_t(warp) * BN, x1 = x0 + BN;
    int n = 0;
    int32_t* dst = list + int64_t(warp) * n_qt;
    for (int base = 0; base < n_qt; base += 32) {
        const int t = base + lane;
        bool hit = false;
        if (t < n_qt) {
            const int4 b = qtb[t];
            hit = b.x < b.y && b.x < x1 && b.y > x0;
        }
        const unsigned m = __ballot_sync(0xffffffffu, hit);
        if (hit) dst[n + __popc(m & ((1u << lane) - 1u))] = t;
        n += __popc(m);
    }
    if (lane == 0) cnt[warp] = n;
}

// ------------------------------------------------------------------ kernel

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_do,
                   const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                   const float* __restrict__ lse2_hm, const float* __restrict__ D_hm, int64_t Qp,
                   const int32_t* __restrict__ s, const int32_t* __restrict__ a, int B, int64_t Qn, int H, int64_t S,
                   float scale, float scale_log2, const int4* __restrict__ qtb, const int32_t* __restrict__ kv_cnt,
                   const int32_t* __restrict__ kv_list, int n_qt, float* __restrict__ dq, float* __restrict__ dk,
                   float* __restrict__ dv, int* status, long long wait_limit) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t base_s = smem_u32(smem_raw);
    const uint32_t pad = ((base_s + 1023u) & ~1023u) - base_s;
    // the swizzled tiles must start on a 1024-byte boundary inside the allocation
    if (pad + sizeof(BwdSmem<D>) > (size_t)kSmemMax) {
        if (threadIdx.x == 0) skv::raise_status(status, SKV_ERR_UNSUPPORTED);
        return;
    }
    BwdSmem<D>& sm = *reinterpret_cast<BwdSmem<D>*>(smem_raw + pad);
    BwdTiles<D>& tl = sm.t;
    BwdBars& bb = sm.b;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kt = blockIdx.x, h = blockIdx.y;
    const int64_t x0 = int64_t(kt) * BN;
    constexpr int NP = D / 64;
    constexpr uint32_t kTile = BM * D * 2;
    // test mode (negative limit): the MMA thread first waits on a barrier nothing
    // completes, so the timeout path runs deterministically
    const bool stuck_test = wait_limit < 0;
    if (stuck_test) wait_limit = -wait_limit;
    int cnt = kv_cnt[kt];
    if (*(volatile int*)status == SKV_ERR_TIMEOUT) cnt = 0;   // launch already void: skip the work
    const int32_t* list = kv_list + int64_t(kt) * n_qt;

    if (tid == 0) {
        mbar_init(&bb.kv_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bb.qd_full[i], 1);
            mbar_init(&bb.qd_empty[i], 1);
        }
        mbar_init(&bb.s_full, 1);
        mbar_init(&bb.dp_full, 1);
        mbar_init(&bb.ds_full, 256);
        mbar_init(&bb.dq_full, 1);
        mbar_init(&bb.dq_free, 128);
        mbar_init(&bb.mma_fin, 1);
        mbar_init(&bb.stuck, 1);
        bb.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&bb.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bb.tmem_base;
    const uint32_t tA = tmem, tB = tmem + 128, tdV = tmem + 256, tdK = tmem + 384;
    auto abort_now = [&]() {
        atomicExch(&bb.abort_flag, 1);
        skv::raise_status(status, SKV_ERR_TIMEOUT);
    };

    if (warp == kTmaWarp) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && cnt > 0) {
            prefetch_tensormap(&map_q);
            prefetch_tensormap(&map_do);
            mbar_arrive_expect_tx(&bb.kv_full, 2 * kTile);
            for (int c = 0; c < NP; ++c) {
                tma_load_2d(tl.k[c], &map_k, &bb.kv_full, h * D + c * 64, (int)x0);
                tma_load_2d(tl.v[c], &map_v, &bb.kv_full, h * D + c * 64, (int)x0);
            }
            int t = 0;
            for (; t < cnt; ++t) {
                const int st = t & 1;
                if (t >= 2 && !mbar_wait(&bb.qd_empty[st], ((t - 2) >> 1) & 1, wait_limit, &bb.abort_flag)) {
                    abort_now();
                    break;
                }
                if (*(volatile int*)&bb.abort_flag) break;
                const int qt = list[t];
                const int row = qt * BM;
                sm.meta[st].qt = qt;                     // made visible by the arrive below
                sm.meta[st].bnd = qtb[qt];
                mbar_arrive_expect_tx(&bb.qd_full[st], 2 * kTile + 2 * BM * 4);
                for (int c = 0; c < NP; ++c) {
                    tma_load_2d(tl.q[st][c], &map_q, &bb.qd_full[st], h * D + c * 64, row);
                    tma_load_2d(tl.dO[st][c], &map_do, &bb.qd_full[st], h * D + c * 64, row);
                }
                bulk_load(sm.meta[st].lse2, lse2_hm + int64_t(h) * Qp + row, BM * 4, &bb.qd_full[st]);
                bulk_load(sm.meta[st].D, D_hm + int64_t(h) * Qp + row, BM * 4, &bb.qd_full[st]);
            }
            // every copy issued has landed before the block exits
            mbar_wait(&bb.kv_full, 0, kTeardownWait);
            for (int st = 0; st < 2 && st < t; ++st) {
                const int last = st + ((t - 1 - st) >> 1) * 2;
                mbar_wait(&bb.qd_full[st], (last >> 1) & 1, kTeardownWait);
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && cnt > 0) {
            constexpr uint32_t idS = idesc_bf16_f32(BN, BM, 0, 0);    // M = keys, N = queries, K = d
            constexpr uint32_t idKV = idesc_bf16_f32(BN, D, 0, 1);    // M = keys, N = d, K = queries
            constexpr uint32_t idQ = idesc_bf16_f32(BM, D, 1, 1);     // M = queries, N = d, K = keys
            bool issued = false;
            bool ok = !(stuck_test && !mbar_wait(&bb.stuck, 0, wait_limit, &bb.abort_flag));
            if (ok) ok = mbar_wait(&bb.kv_full, 0, wait_limit, &bb.abort_flag);
            auto issue_s = [&](int st) {                   // S^T = K Q^T -> A
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk & 3) * 32;
                    mma_ss(tA, smem_desc(smem_u32(tl.k[kk >> 2]) + off, 16, 1024),
                           smem_desc(smem_u32(tl.q[st][kk >> 2]) + off, 16, 1024), idS, kk > 0);
                }
                mma_commit(&bb.s_full);
            };
            auto issue_dp = [&](int st) {                  // dP^T = V dO^T -> B
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk & 3) * 32;
                    mma_ss(tB, smem_desc(smem_u32(tl.v[kk >> 2]) + off, 16, 1024),
                           smem_desc(smem_u32(tl.dO[st][kk >> 2]) + off, 16, 1024), idS, kk > 0);
                }
                mma_commit(&bb.dp_full);
            };
            if (ok) ok = mbar_wait(&bb.qd_full[0], 0, wait_limit, &bb.abort_flag);
            if (ok) {
                tc_fence_after();
                issue_s(0);
                issue_dp(0);
                issued = true;
            }
            for (int t = 0; ok && t < cnt; ++t) {
                const int st = t & 1;
                if (!mbar_wait(&bb.ds_full, t & 1, wait_limit, &bb.abort_flag)) { ok = false; break; }
                tc_fence_after();
                // dV += P^T dO.  bf16 P^T of query columns [64h, 64h+64) sits in TMEM
                // columns [64h, 64h+32) of A (each half-warpgroup writes inside its own half)
#pragma unroll
                for (int kk = 0; kk < BM / 16; ++kk)
                    mma_ts(tdV, tA + (kk >> 2) * 64 + (kk & 3) * 8,
                           smem_desc(smem_u32(tl.dO[st][0]) + kk * 2048, BM * 128, 1024), idKV,
                           (t > 0 || kk > 0) ? 1u : 0u);
                // S_{t+1} overwrites A right behind the dV MMA that reads P_t from it:
                // the MMAs of one thread execute in issue order
                const bool more = t + 1 < cnt;
                if (more) {
                    if (!mbar_wait(&bb.qd_full[(t + 1) & 1], ((t + 1) >> 1) & 1, wait_limit, &bb.abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_s((t + 1) & 1);
                }
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)      // dQ = dS K -> B
                    mma_ss(tB, smem_desc(smem_u32(tl.ds[0]) + kk * 2048, BN * 128, 1024),
                           smem_desc(smem_u32(tl.k[0]) + kk * 2048, BN * 128, 1024), idQ, kk > 0);
                mma_commit(&bb.dq_full);
#pragma unroll
                for (int kk = 0; kk < BM / 16; ++kk)      // dK += dS^T Q
                    mma_ss(tdK, smem_desc(smem_u32(tl.ds[kk >> 2]) + (kk & 3) * 32, 16, 1024),
                           smem_desc(smem_u32(tl.q[st][0]) + kk * 2048, BM * 128, 1024), idKV,
                           (t > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&bb.qd_empty[st]);
                if (more) {
                    if (!mbar_wait(&bb.dq_free, t & 1, wait_limit, &bb.abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    issue_dp((t + 1) & 1);
                }
            }
            if (!ok) abort_now();
            if (issued) {
                mma_commit(&bb.mma_fin);
                if (!mbar_wait(&bb.mma_fin, 0, kTeardownWait)) skv::raise_status(status, SKV_ERR_TIMEOUT);
            }
        }
    } else {
        constexpr unsigned kAll = 0xffffffffu;
        const int wg_warp = warp & 3;                    // TMEM lane quadrant
        const uint32_t lane_base = uint32_t(wg_warp * 32) << 16;
        const int r = wg_warp * 32 + lane;               // TMEM lane of this thread
        bool ok = true;
        auto uniform_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
            const bool got = mbar_wait_warp(bar, parity, wait_limit, &bb.abort_flag);
            if (!got && lane == 0) abort_now();
            return got;
        };
        if (warp < 8) {
            // -------------------------------------------------------- WG1: P^T and dS^T
            // warp w owns TMEM lanes (keys) of quadrant w%4 and query columns
            // [64*hf, 64*hf+64) with hf = w/4
            const int hf = warp >> 2;
            const int64_t x = x0 + r;                    // key row (S^T, dP^T, dK)
            unsigned char* ds_panel = reinterpret_cast<unsigned char*>(&tl.ds[hf][0]) + r * 128;
            for (int t = 0; t < cnt; ++t) {
                const int st = t & 1;
                if (__any_sync(kAll, *(volatile int*)&bb.abort_flag != 0)) { ok = false; break; }
                if (!uniform_wait(&bb.qd_full[st], (t >> 1) & 1)) { ok = false; break; }
                const BwdMeta& md = sm.meta[st];
                const int64_t row0 = int64_t(md.qt) * BM;
                const int4 bnd = md.bnd;
                const bool full = (x0 >= bnd.z) && (x0 + BN <= bnd.w);
                if (!uniform_wait(&bb.s_full, t & 1)) { ok = false; break; }
                tc_fence_after();
                // both 32-column chunks of S^T are loaded before one wait; P^T is kept as
                // the bf16 pairs the dV MMA consumes and dS^T is formed from those values
                uint32_t sraw[2][32];
                tmem_ld32(tA + lane_base + hf * 64, sraw[0]);
                tmem_ld32(tA + lane_base + hf * 64 + 32, sraw[1]);
                tmem_ld_wait();
                uint32_t pk[2][16];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int col0 = hf * 64 + c * 32;
                    uint32_t keep = 0xffffffffu;          // columns whose query row sees key x
                    if (!full) {                          // boundary tile: each query row's own window
                        keep = 0u;
#pragma unroll 1
                        for (int j = 0; j < 32; ++j) {
                            const int64_t qr = row0 + col0 + j;
                            int64_t lo = 0, hi = 0;
                            if (qr < Qn) skv::block_window(s, a, (int)(qr / B), S, lo, hi);
                            if (lo <= x && x < hi) keep |= 1u << j;
                        }
                    }
                    const float4* l4 = reinterpret_cast<const float4*>(md.lse2 + col0);
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const float4 l = l4[j4];
                        const float lv[4] = {l.x, l.y, l.z, l.w};
                        float pv[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int j = 4 * j4 + u;
                            pv[u] = ((keep >> j) & 1u) ? ex2(fmaf(__uint_as_float(sraw[c][j]), scale_log2, -lv[u]))
                                                       : 0.f;
                        }
                        pk[c][2 * j4] = pack_bf16(pv[0], pv[1]);
                        pk[c][2 * j4 + 1] = pack_bf16(pv[2], pv[3]);
                    }
                    // bf16 pairs of these 32 columns -> TMEM columns [64hf + 16c, +16): inside
                    // this warp's own half, over S^T columns it has read already
                    tmem_st16(tA + lane_base + hf * 64 + c * 16, pk[c]);
                }
                if (!uniform_wait(&bb.dp_full, t & 1)) { ok = false; break; }
                tc_fence_after();
                uint32_t draw[2][32];
                tmem_ld32(tB + lane_base + hf * 64, draw[0]);
                tmem_ld32(tB + lane_base + hf * 64 + 32, draw[1]);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int col0 = hf * 64 + c * 32;
                    uint32_t dk2[16];
                    const float4* d4 = reinterpret_cast<const float4*>(md.D + col0);
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const float4 dd = d4[j4];
                        const float2 p01 = unpack_bf16(pk[c][2 * j4]);
                        const float2 p23 = unpack_bf16(pk[c][2 * j4 + 1]);
                        dk2[2 * j4] = pack_bf16(p01.x * (__uint_as_float(draw[c][4 * j4]) - dd.x),
                                                p01.y * (__uint_as_float(draw[c][4 * j4 + 1]) - dd.y));
                        dk2[2 * j4 + 1] = pack_bf16(p23.x * (__uint_as_float(draw[c][4 * j4 + 2]) - dd.z),
                                                    p23.y * (__uint_as_float(draw[c][4 * j4 + 3]) - dd.w));
                    }
                    // query columns [64hf + 32c, +32) = panel hf, 16-byte chunks 4c .. 4c+3
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int chunk = c * 4 + u;
                        *reinterpret_cast<uint4*>(ds_panel + ((chunk ^ (r & 7)) << 4)) =
                            make_uint4(dk2[4 * u], dk2[4 * u + 1], dk2[4 * u + 2], dk2[4 * u + 3]);
                    }
                }
                tmem_st_wait();
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&bb.ds_full);
            }
            // dK rows of this key tile (scaled; columns split between the two halves)
            // once every MMA of the block has completed
            const bool aborted = __any_sync(kAll, *(volatile int*)&bb.abort_flag != 0);
            float* dkr = dk + (x * H + h) * D;
            constexpr int kHalf = D / 2;
            if (cnt > 0 && ok && !aborted && uniform_wait(&bb.mma_fin, 0)) {
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < kHalf / 32; ++c) {
                    const int col0 = hf * kHalf + c * 32;
                    uint32_t rk[32];
                    tmem_ld32(tdK + lane_base + col0, rk);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        __stcs(reinterpret_cast<float4*>(dkr + col0 + j),
                               make_float4(scale * __uint_as_float(rk[j]), scale * __uint_as_float(rk[j + 1]),
                                           scale * __uint_as_float(rk[j + 2]), scale * __uint_as_float(rk[j + 3])));
                }
            } else if (cnt == 0) {
#pragma unroll
                for (int j = 0; j < kHalf; j += 4)
                    __stcs(reinterpret_cast<float4*>(dkr + hf * kHalf + j), make_float4(0.f, 0.f, 0.f, 0.f));
            }
        } else {
            // -------------------------------------------------------- WG2: dQ -> dq (fp32 reductions)
            int qt_next = cnt > 0 ? list[0] : 0;
            for (int t = 0; t < cnt; ++t) {
                const int64_t qrow = int64_t(qt_next) * BM + r;   // TMEM lane = query row for dQ
                if (t + 1 < cnt) qt_next = list[t + 1];        // prefetched for the next tile
                if (__any_sync(kAll, *(volatile int*)&bb.abort_flag != 0)) { ok = false; break; }
                if (!uniform_wait(&bb.dq_full, t & 1)) { ok = false; break; }
                tc_fence_after();
                float* dst = dq + (qrow * H + h) * D;
#pragma unroll
                for (int c = 0; c < D / 32; c += 2) {         // two TMEM loads per wait
                    uint32_t rr[2][32];
                    tmem_ld32(tB + lane_base + c * 32, rr[0]);
                    tmem_ld32(tB + lane_base + c * 32 + 32, rr[1]);
                    tmem_ld_wait();
                    if (c + 2 >= D / 32) {
                        tc_fence_before();
                        mbar_arrive(&bb.dq_free);         // B may now take dP of the next tile
                    }
                    if (qrow < Qn) {
#pragma unroll
                        for (int u = 0; u < 2; ++u)
#pragma unroll
                            for (int j = 0; j < 32; j += 4)
                                red_add4(dst + (c + u) * 32 + j, scale * __uint_as_float(rr[u][j]),
                                         scale * __uint_as_float(rr[u][j + 1]), scale * __uint_as_float(rr[u][j + 2]),
                                         scale * __uint_as_float(rr[u][j + 3]));
                    }
                }
            }
            // dV rows of this key tile
            const int64_t x = x0 + r;
            float* dvr = dv + (x * H + h) * D;
            const bool aborted = __any_sync(kAll, *(volatile int*)&bb.abort_flag != 0);
            if (cnt > 0 && ok && !aborted && uniform_wait(&bb.mma_fin, 0)) {
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t rv[32];
                    tmem_ld32(tdV + lane_base + c * 32, rv);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        __stcs(reinterpret_cast<float4*>(dvr + c * 32 + j),
                               make_float4(__uint_as_float(rv[j]), __uint_as_float(rv[j + 1]),
                                           __uint_as_float(rv[j + 2]), __uint_as_float(rv[j + 3])));
                }
            } else if (cnt == 0) {
#pragma unroll
                for (int j = 0; j < D; j += 4) __stcs(reinterpret_cast<float4*>(dvr + j), make_float4(0.f, 0.f, 0.f, 0.f));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

struct BwdScratch {
    int4* qtb;
    int32_t* cnt;
    int32_t* list;
};

size_t scratch_layout(const skv_problem& pb, BwdScratch* w, char* base) {
    using skv_host::align256;
    const int64_t Qn = int64_t(pb.n_blocks) * pb.B;
    const int64_t n_qt = (Qn + BM - 1) / BM;
    const int64_t n_kv = pb.S / BN;
    size_t off = 0;
    const size_t o_qtb = off; off = align256(off + size_t(n_qt) * sizeof(int4));
    const size_t o_cnt = off; off = align256(off + size_t(n_kv) * 4);
    const size_t o_list = off; off = align256(off + size_t(n_kv) * size_t(n_qt) * 4);
    if (w) {
        w->qtb = reinterpret_cast<int4*>(base + o_qtb);
        w->cnt = reinterpret_cast<int32_t*>(base + o_cnt);
        w->list = reinterpret_cast<int32_t*>(base + o_list);
    }
    return off;
}

template <int D>
skv_status launch_bwd(const skv_problem& pb, const void* q, const void* k, const void* v, const void* dO,
                      const float* lse2_hm, const float* D_hm, float* dq, float* dk, float* dv, void* scratch,
                      const skv_host::Ctx& c) {
    const int64_t Qn = int64_t(pb.n_blocks) * pb.B;
    const int n_qt = (int)((Qn + BM - 1) / BM);
    const int64_t Qp = int64_t(n_qt) * BM;
    const int n_kv = (int)(pb.S / BN);
    BwdScratch w;
    scratch_layout(pb, &w, static_cast<char*>(scratch));
    qtile_bounds_kernel<<<(n_qt + 127) / 128, 128, 0, c.stream>>>(pb.s, pb.a, pb.B, Qn, pb.S, n_qt, w.qtb);
    SKV_LAUNCHED();
    kv_list_kernel<<<(n_kv + 7) / 8, 256, 0, c.stream>>>(w.qtb, n_qt, n_kv, w.cnt, w.list);
    SKV_LAUNCHED();
    CUtensorMap mq, mdo, mk, mv;
    const int64_t cols = int64_t(pb.n_heads) * D;
    if (!make_map(&mq, q, Qn, cols) || !make_map(&mdo, dO, Qn, cols) || !make_map(&mk, k, pb.S, cols) ||
        !make_map(&mv, v, pb.S, cols))
        return SKV_ERR_CUDA;
    SKV_CUDA_CHECK(cudaMemsetAsync(dq, 0, size_t(Qn) * cols * sizeof(float), c.stream));
    auto kern = attn_bwd_tc_kernel<D>;
    SKV_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax));
    const dim3 grid((unsigned)n_kv, (unsigned)pb.n_heads);
    kern<<<grid, kBwdThreads, kSmemMax, c.stream>>>(mq, mdo, mk, mv, lse2_hm, D_hm, Qp, pb.s, pb.a, pb.B, Qn,
                                                    pb.n_heads, pb.S, pb.scale, pb.scale * 1.4426950408889634f, w.qtb,
                                                    w.cnt, w.list, n_qt, dq, dk, dv, c.status, c.wait_limit);
    SKV_LAUNCHED();
    return SKV_OK;
}

}  // namespace

namespace skv_tc {

bool bwd_supported(const skv_problem& pb) {
    return pb.dtype == SKV_BF16 && (pb.head_dim == 64 || pb.head_dim == 128) && pb.m % BN == 0 &&
           pb.n_heads <= 65535;
}

size_t bwd_scratch_bytes(const skv_problem& pb) {
    return bwd_supported(pb) ? scratch_layout(pb, nullptr, nullptr) : 0;
}

skv_status launch_attn_bwd_tc(const skv_problem& pb, const void* q, const void* k, const void* v, const void* dO,
                              const float* lse2, const float* D, skv::RankCSR, float* dq, float* dk, float* dv,
                              void* scratch, const skv_host::Ctx& c) {
    if (pb.head_dim == 128) return launch_bwd<128>(pb, q, k, v, dO, lse2, D, dq, dk, dv, scratch, c);
    return launch_bwd<64>(pb, q, k, v, dO, lse2, D, dq, dk, dv, scratch, c);
}

}  // namespace skv_tc
