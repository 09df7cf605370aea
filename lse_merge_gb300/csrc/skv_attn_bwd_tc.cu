// Tensor-core backward of the anchor attention (tcgen05 + TMEM + TMA), sm_103a.
//
// "Split-KV: Efficient Context Parallelism for Training Diffusion Drafters",
// Alg. 1's backward in merged form: with the global log-sum-exp l_r and
// D_r = dO_r . o_r, every rank's score gradient is dS = P (dP - D) with
// P = exp(z - l).  Two kernels:
//
//  * attn_bwd_dkdv_tc_kernel -- key-stationary.  One thread block owns a
//    128-key tile and a key/value head (the tile belongs to exactly one rank, so
//    dk_p and dv_p rows are written once, no atomics) and walks, for each query
//    head of the head's group (one head without grouped queries), the query tiles
//    of its tile-skip list (built by qtile_bounds_kernel / kv_list_kernel; masked-out
//    query tiles are never loaded).  Per query tile t:
//      S^T = K Q_t^T, dP^T = V dO_t^T (SS) -> TMEM A, B
//      eight warps: P^T = exp2(S^T scale log2e - l2) as bf16 -> TMEM A over the
//                   S^T they have read; dS^T = P^T (dP^T - D) -> TMEM B likewise
//      dV += P^T dO_t (TS) as soon as P^T is in TMEM, so it overlaps the forming
//      of dS^T; then S of the next tile; dK += dS^T Q_t (TS); dP of the next tile.
//    dK and dV leave through shared memory with TMA stores.
//  * attn_bwd_dq_tc_kernel -- query-stationary.  One thread block owns a
//    128-row query tile and a head and walks the key tiles that meet the tile's
//    windows, in ascending order: dq = sum_p dq^(p) (Alg. 1's dq reduce-scatter),
//    whose ranks' chunks tile the keys exactly, is accumulated in TMEM over all of
//    them and written once.  Q and dO stay
//    in TMEM as A operands; per key tile:
//      S = Q K^T, dP = dO V^T (TS); eight warps form dS (bf16 -> TMEM over the
//      dP they read); dQ += dS K (TS).  S of the next tile is issued as soon as
//      S has been read, so it overlaps the forming of P and dS.  With grouped
//      queries the tile stacks the group's g query heads (128/g rows each), as
//      in the forward, so each K/V tile is loaded once per group.
// Recomputing S and dP in the second kernel costs two extra GEMMs per tile pair
// but removes every dq reduction from the key-stationary loop.
#include <cuda.h>
#include <math.h>

#include "skv_ptx.cuh"
#include "skv_tc.h"
#include "skv_tc_common.cuh"

namespace {

using namespace skv_ptx;
using namespace skv_tcc;

constexpr int kSmemMax = 232448;                     // sm_100-family opt-in maximum per block
constexpr long long kTeardownWait = 2000000000LL;    // ns

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// ---------------------------------------------------------------- tile lists

// Per query tile: union (lo, hi) and full-visibility (flo, fhi) key bounds.
__global__ void qtile_bounds_kernel(const int32_t* __restrict__ s, const int32_t* __restrict__ a, int B, int64_t Qn,
                                    int64_t S, int n_qt, int4* __restrict__ out, int rows) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= n_qt) return;
    const TileBounds tb = tile_bounds(s, a, B, Qn, S, t, rows);
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

// =============================================================== dK / dV

constexpr int kKvThreads = 320;                      // compute warps 0-7, MMA 8, TMA 9
constexpr int kKvMma = 8, kKvTma = 9;

constexpr int kQSt = 3;                              // Q ring depth (dO and metadata: 2)

template <int D>
struct KvTiles {                                     // 1024-byte aligned (128-byte swizzle atoms)
    __nv_bfloat16 k[D / 64][BN * 64];
    __nv_bfloat16 v[D / 64][BN * 64];
    __nv_bfloat16 q[kQSt][D / 64][BM * 64];
    __nv_bfloat16 dO[2][D / 64][BM * 64];
};

struct KvMeta {                                      // per query tile, its own two-stage ring
    float lse2[BM];
    float D[BM];
    int4 bnd;                                        // the tile's key bounds (written by the producer)
    int qt;                                          // the query tile index
    int pad_[3];
};

struct KvBars {
    uint64_t kv_full, q_full[kQSt], q_empty[kQSt], meta_full[2], meta_empty[2], do_full[2], do_empty[2];
    uint64_t s_full, p_full[2], dp_full, ds_full, mma_fin;
    uint64_t stuck;                                  // never completed: target of the forced-timeout test mode
    uint32_t tmem_base;
    int abort_flag;
};

template <int D>
struct KvSmem {
    KvTiles<D> t;
    KvMeta meta[2];
    KvBars b;
};

template <int D>
__global__ void __launch_bounds__(kKvThreads, 1)
attn_bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_do,
                        const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                        const __grid_constant__ CUtensorMap map_dk, const __grid_constant__ CUtensorMap map_dv,
                        const float* __restrict__ lse2_hm, const float* __restrict__ D_hm, int64_t Qp,
                        const int32_t* __restrict__ s, const int32_t* __restrict__ a, int B, int64_t Qn, int Hkv,
                        int gq, int64_t S, float scale, float scale_log2, const int4* __restrict__ qtb,
                        const int32_t* __restrict__ kv_cnt, const int32_t* __restrict__ kv_list, int n_qt,
                        float* __restrict__ dk, float* __restrict__ dv, int* status, long long wait_limit) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t base_s = smem_u32(smem_raw);
    const uint32_t pad = ((base_s + 1023u) & ~1023u) - base_s;
    // the swizzled tiles must start on a 1024-byte boundary inside the allocation
    if (pad + sizeof(KvSmem<D>) > (size_t)kSmemMax) {
        if (threadIdx.x == 0) skv::raise_status(status, SKV_ERR_UNSUPPORTED);
        return;
    }
    KvSmem<D>& sm = *reinterpret_cast<KvSmem<D>*>(smem_raw + pad);
    KvTiles<D>& tl = sm.t;
    KvBars& bb = sm.b;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // one key/value head kvh; its gq query heads (grouped-query layouts) are walked
    // one after the other and all accumulate into the same dK, dV
    const int kt = blockIdx.x, kvh = blockIdx.y;
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
    const int n_it = cnt * gq;                       // (query head, query tile) pairs, head-major

    if (tid == 0) {
        mbar_init(&bb.kv_full, 1);
        for (int i = 0; i < kQSt; ++i) {
            mbar_init(&bb.q_full[i], 1);
            mbar_init(&bb.q_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bb.meta_full[i], 1);
            mbar_init(&bb.meta_empty[i], 256);
            mbar_init(&bb.do_full[i], 1);
            mbar_init(&bb.do_empty[i], 1);
        }
        mbar_init(&bb.s_full, 1);
        mbar_init(&bb.p_full[0], 256);
        mbar_init(&bb.p_full[1], 256);
        mbar_init(&bb.dp_full, 1);
        mbar_init(&bb.ds_full, 256);
        mbar_init(&bb.mma_fin, 1);
        mbar_init(&bb.stuck, 1);
        bb.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kKvMma) {
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

    if (warp == kKvTma) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && cnt > 0) {
            prefetch_tensormap(&map_q);
            prefetch_tensormap(&map_do);
            mbar_arrive_expect_tx(&bb.kv_full, 2 * kTile);
            for (int c = 0; c < NP; ++c) {
                tma_load_2d(tl.k[c], &map_k, &bb.kv_full, kvh * D + c * 64, (int)x0);
                tma_load_2d(tl.v[c], &map_v, &bb.kv_full, kvh * D + c * 64, (int)x0);
            }
            // Q, the tile's metadata (l2, D, bounds) and dO have their own rings: the dK
            // MMA frees Q, the compute warps free the metadata once dS is formed and the
            // dV MMA frees dO; S of a tile needs Q first, so Q runs one stage deeper
            int nq = 0, nm = 0, nd = 0;
            for (int t = 0; t < n_it; ++t) {
                const int sq = t % kQSt, st = t & 1;
                if (t >= kQSt &&
                    !mbar_wait(&bb.q_empty[sq], ((t - kQSt) / kQSt) & 1, wait_limit, &bb.abort_flag)) {
                    abort_now();
                    break;
                }
                if (*(volatile int*)&bb.abort_flag) break;
                const int hq = kvh * gq + t / cnt;       // query head of this item
                const int qt = list[t % cnt];
                const int row = qt * BM;
                mbar_arrive_expect_tx(&bb.q_full[sq], kTile);
                for (int c = 0; c < NP; ++c) tma_load_2d(tl.q[sq][c], &map_q, &bb.q_full[sq], hq * D + c * 64, row);
                ++nq;
                if (t >= 2 && !mbar_wait(&bb.meta_empty[st], ((t - 2) >> 1) & 1, wait_limit, &bb.abort_flag)) {
                    abort_now();
                    break;
                }
                sm.meta[st].qt = qt;                     // made visible by the arrive below
                sm.meta[st].bnd = qtb[qt];
                mbar_arrive_expect_tx(&bb.meta_full[st], 2 * BM * 4);
                bulk_load(sm.meta[st].lse2, lse2_hm + int64_t(hq) * Qp + row, BM * 4, &bb.meta_full[st]);
                bulk_load(sm.meta[st].D, D_hm + int64_t(hq) * Qp + row, BM * 4, &bb.meta_full[st]);
                ++nm;
                if (t >= 2 && !mbar_wait(&bb.do_empty[st], ((t - 2) >> 1) & 1, wait_limit, &bb.abort_flag)) {
                    abort_now();
                    break;
                }
                mbar_arrive_expect_tx(&bb.do_full[st], kTile);
                for (int c = 0; c < NP; ++c) tma_load_2d(tl.dO[st][c], &map_do, &bb.do_full[st], hq * D + c * 64, row);
                ++nd;
                // no L2 prefetch here: a query tile is read by every key tile of its
                // windows, so its Q and dO are already in L2 (the hints measured slower)
            }
            // every copy issued has landed before the block exits
            mbar_wait(&bb.kv_full, 0, kTeardownWait);
            auto drain = [&](uint64_t* bars, int n, int depth) {
                for (int st = 0; st < depth && st < n; ++st) {
                    const int last = st + ((n - 1 - st) / depth) * depth;
                    mbar_wait(&bars[st], (last / depth) & 1, kTeardownWait);
                }
            };
            drain(bb.q_full, nq, kQSt);
            drain(bb.meta_full, nm, 2);
            drain(bb.do_full, nd, 2);
        }
    } else if (warp == kKvMma) {
        // ------------------------------------------------------------ MMA issuer
        // the whole warp runs the schedule (warp-uniform descriptors and counters);
        // one elected lane issues each group of MMAs and its commits
        if (cnt > 0) {
            constexpr uint32_t idS = idesc_bf16_f32(BN, BM, 0, 0);    // M = keys, N = queries, K = d
            constexpr uint32_t idKV = idesc_bf16_f32(BN, D, 0, 1);    // M = keys, N = d, K = queries
            auto wait = [&](uint64_t* bar, uint32_t parity) {
                return mbar_wait_warp(bar, parity, wait_limit, &bb.abort_flag);
            };
            bool issued = false;
            bool ok = !(stuck_test && !wait(&bb.stuck, 0));
            if (ok) ok = wait(&bb.kv_full, 0);
            // shared-memory descriptors as offsets (bytes / 16) from the first panel
            constexpr uint32_t kPanel = BN * 64 * 2 / 16, kSt = NP * kPanel;
            const uint64_t dK = smem_desc(smem_u32(tl.k[0]), 16, 1024), dV = smem_desc(smem_u32(tl.v[0]), 16, 1024);
            const uint64_t dQ = smem_desc(smem_u32(tl.q[0][0]), 16, 1024);
            const uint64_t dDO = smem_desc(smem_u32(tl.dO[0][0]), 16, 1024);
            const uint64_t dQmn = smem_desc(smem_u32(tl.q[0][0]), BM * 128, 1024);
            const uint64_t dDOmn = smem_desc(smem_u32(tl.dO[0][0]), BM * 128, 1024);
            auto issue_s = [&](int st) {                   // S^T = K Q^T -> A
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 2;
                        mma_ss(tA, dK + off, dQ + (st * kSt + off), idS, kk > 0);
                    }
                    mma_commit(&bb.s_full);
                }
                __syncwarp();
            };
            auto issue_dp = [&](int st) {                  // dP^T = V dO^T -> B
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 2;
                        mma_ss(tB, dV + off, dDO + (st * kSt + off), idS, kk > 0);
                    }
                    mma_commit(&bb.dp_full);
                }
                __syncwarp();
            };
            if (ok) ok = wait(&bb.q_full[0], 0);
            if (ok) {
                tc_fence_after();
                issue_s(0);
                issued = true;
                ok = wait(&bb.do_full[0], 0);
            }
            if (ok) {
                tc_fence_after();
                issue_dp(0);
            }
            // per query tile t (in issue order):
            //   [P_t stored]  dV += P_t^T dO_t   (P_t bf16 over the read S_t), while dS_t forms
            //   S_{t+1} -> A  right behind the dV MMAs reading P_t from A
            //   [dS_t stored] dK += dS_t^T Q_t   (dS_t bf16 over the read dP_t)
            //   dP_{t+1} -> B right behind the dK MMAs reading dS_t from B
            for (int t = 0; ok && t < n_it; ++t) {
                const int st = t & 1, sq = t % kQSt, sq1 = (t + 1) % kQSt;
                const bool more = t + 1 < n_it;
                // bf16 P^T of query columns [64h, 64h+64) sits in TMEM columns [64h, 64h+32) of
                // A; it arrives in two parts (query columns [64h, 64h+32), then [64h+32, 64h+64)
                // of both halves), and the dV MMAs of each part go as soon as it is stored
                bool got = true;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    if (!wait(&bb.p_full[c], t & 1)) { got = false; break; }
                    tc_fence_after();
                    if (elect_one()) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int kk = (i >> 1) * 4 + c * 2 + (i & 1);
                            mma_ts(tdV, tA + (kk >> 2) * 64 + (kk & 3) * 8, dDOmn + (st * kSt + kk * 128), idKV,
                                   (t > 0 || kk > 0) ? 1u : 0u);
                        }
                        if (c == 1) mma_commit(&bb.do_empty[st]);
                    }
                    __syncwarp();
                }
                if (!got) { ok = false; break; }
                if (more) {
                    if (!wait(&bb.q_full[sq1], ((t + 1) / kQSt) & 1)) { ok = false; break; }
                    tc_fence_after();
                    issue_s(sq1);
                }
                if (!wait(&bb.ds_full, t & 1)) { ok = false; break; }
                tc_fence_after();
                // bf16 dS^T of query columns [64h, 64h+64) sits in TMEM columns [64h, 64h+32) of B
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < BM / 16; ++kk)
                        mma_ts(tdK, tB + (kk >> 2) * 64 + (kk & 3) * 8, dQmn + (sq * kSt + kk * 128), idKV,
                               (t > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&bb.q_empty[sq]);
                }
                __syncwarp();
                if (more) {
                    if (!wait(&bb.do_full[(t + 1) & 1], ((t + 1) >> 1) & 1)) { ok = false; break; }
                    tc_fence_after();
                    issue_dp((t + 1) & 1);
                }
            }
            if (!ok && lane == 0) abort_now();
            if (issued) {
                if (elect_one()) mma_commit(&bb.mma_fin);
                __syncwarp();
                if (!mbar_wait_warp(&bb.mma_fin, 0, kTeardownWait) && lane == 0)
                    skv::raise_status(status, SKV_ERR_TIMEOUT);
            }
        }
    } else {
        // ------------------------------------------------------------ compute warps 0-7
        // warp w owns TMEM lanes (keys) of quadrant w%4 and query columns
        // [64*hf, 64*hf+64) with hf = w/4
        constexpr unsigned kAll = 0xffffffffu;
        const int quad = warp & 3, hf = warp >> 2;
        const uint32_t lane_base = uint32_t(quad * 32) << 16;
        const int r = quad * 32 + lane;                  // TMEM lane = key row
        const int64_t x = x0 + r;
        bool ok = true;
        auto uniform_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
            const bool got = mbar_wait_warp(bar, parity, wait_limit, &bb.abort_flag);
            if (!got && lane == 0) abort_now();
            return got;
        };
        for (int t = 0; t < n_it; ++t) {
            const int st = t & 1;
            if (__any_sync(kAll, *(volatile int*)&bb.abort_flag != 0)) { ok = false; break; }
            if (!uniform_wait(&bb.meta_full[st], (t >> 1) & 1)) { ok = false; break; }
            const KvMeta& md = sm.meta[st];
            const int64_t row0 = int64_t(md.qt) * BM;
            const int4 bnd = md.bnd;
            const bool full = (x0 >= bnd.z) && (x0 + BN <= bnd.w);
            if (!uniform_wait(&bb.s_full, t & 1)) { ok = false; break; }
            tc_fence_after();
            // both 32-column chunks of S^T are loaded before one wait.  P^T is kept as
            // the bf16 pairs the dV MMA consumes and dS^T is formed from those values.
            uint32_t sraw[2][32];
            tmem_ld32(tA + lane_base + hf * 64, sraw[0]);
            tmem_ld32(tA + lane_base + hf * 64 + 32, sraw[1]);
            tmem_ld_wait();
            uint32_t pk[2][16];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int col0 = hf * 64 + c * 32;
                uint32_t keep = 0xffffffffu;              // columns whose query row sees key x
                if (!full) {                              // boundary tile: each block's own window
                    keep = 0u;
                    const int64_t qr0 = row0 + col0;      // query rows [qr0, qr0 + 32) of this chunk
                    const int64_t qr1 = (qr0 + 32 < Qn ? qr0 + 32 : Qn);
                    if (qr0 < qr1) {
#pragma unroll 1
                        for (int64_t blk = qr0 / B; blk * B < qr1; ++blk) {
                            int64_t lo, hi;
                            skv::block_window(s, a, (int)blk, S, lo, hi);
                            if (lo <= x && x < hi) {
                                const int64_t j0 = blk * B - qr0, j1 = (blk + 1) * B - qr0;
                                const int b0 = j0 > 0 ? (int)j0 : 0, b1 = j1 < (qr1 - qr0) ? (int)j1 : (int)(qr1 - qr0);
                                keep |= (b1 >= 32 ? 0xffffffffu : ((1u << b1) - 1u)) & ~((1u << b0) - 1u);
                            }
                        }
                    }
                }
                const float4* l4 = reinterpret_cast<const float4*>(md.lse2 + col0);
                if (full) {
                    const float2 sc2 = make_float2(scale_log2, scale_log2);
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const float4 l = l4[j4];
                        const float2 z0 = __ffma2_rn(make_float2(__uint_as_float(sraw[c][4 * j4]),
                                                                 __uint_as_float(sraw[c][4 * j4 + 1])),
                                                     sc2, make_float2(-l.x, -l.y));
                        const float2 z1 = __ffma2_rn(make_float2(__uint_as_float(sraw[c][4 * j4 + 2]),
                                                                 __uint_as_float(sraw[c][4 * j4 + 3])),
                                                     sc2, make_float2(-l.z, -l.w));
                        pk[c][2 * j4] = pack_bf16(ex2(z0.x), ex2(z0.y));
                        pk[c][2 * j4 + 1] = pack_bf16(ex2(z1.x), ex2(z1.y));
                    }
                } else {
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
                }
                // bf16 P^T of columns [64hf + 32c, +32) -> TMEM A columns [64hf + 16c, +16):
                // inside this warp's half, over S^T columns it has just read
                tmem_st16(tA + lane_base + hf * 64 + c * 16, pk[c]);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bb.p_full[c]);
            }
            if (!uniform_wait(&bb.dp_full, t & 1)) { ok = false; break; }
            tc_fence_after();
            uint32_t draw[2][32];
            tmem_ld32(tB + lane_base + hf * 64, draw[0]);
            tmem_ld32(tB + lane_base + hf * 64 + 32, draw[1]);
            tmem_ld_wait();
            uint32_t d2[2][16];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int col0 = hf * 64 + c * 32;
                const float4* d4 = reinterpret_cast<const float4*>(md.D + col0);
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const float4 dd = d4[j4];
                    const float2 t01 = __fadd2_rn(
                        make_float2(__uint_as_float(draw[c][4 * j4]), __uint_as_float(draw[c][4 * j4 + 1])),
                        make_float2(-dd.x, -dd.y));
                    const float2 t23 = __fadd2_rn(
                        make_float2(__uint_as_float(draw[c][4 * j4 + 2]), __uint_as_float(draw[c][4 * j4 + 3])),
                        make_float2(-dd.z, -dd.w));
                    const float2 d01 = __fmul2_rn(unpack_bf16(pk[c][2 * j4]), t01);
                    const float2 d23 = __fmul2_rn(unpack_bf16(pk[c][2 * j4 + 1]), t23);
                    d2[c][2 * j4] = pack_bf16(d01.x, d01.y);
                    d2[c][2 * j4 + 1] = pack_bf16(d23.x, d23.y);
                }
            }
            // bf16 dS^T of columns [64hf + 32c, +32) -> TMEM B columns [64hf + 16c, +16)
            tmem_st16(tB + lane_base + hf * 64, d2[0]);
            tmem_st16(tB + lane_base + hf * 64 + 16, d2[1]);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bb.ds_full);
            mbar_arrive(&bb.meta_empty[st]);             // l2, D and the bounds of this tile are read
        }
        // dK (scaled) and dV rows of this key tile, once every MMA of the block has
        // completed; zeros if no query sees it.  Each warp stages its 32 rows x D/2
        // columns in the (now idle) Q and dO rings as 128-byte-swizzled 32x32 fp32
        // boxes and writes them with TMA stores (rows past S are dropped).
        const bool aborted = __any_sync(kAll, *(volatile int*)&bb.abort_flag != 0);
        constexpr int kHalf = D / 2;
        if (cnt > 0 && ok && !aborted && uniform_wait(&bb.mma_fin, 0)) {
            tc_fence_after();
            unsigned char* stage_k = reinterpret_cast<unsigned char*>(&tl.q[0][0][0]);
            unsigned char* stage_v = reinterpret_cast<unsigned char*>(&tl.dO[0][0][0]);
            const uint32_t row_off = uint32_t(r) * 128u;
#pragma unroll
            for (int c = 0; c < kHalf / 32; ++c) {
                uint32_t rk[32], rv[32];
                tmem_ld32(tdK + lane_base + hf * kHalf + c * 32, rk);
                tmem_ld32(tdV + lane_base + hf * kHalf + c * 32, rv);
                tmem_ld_wait();
                // panel of columns [32p, 32p+32): 128 rows x 128 bytes; 16-byte chunk j of
                // row r sits at chunk j ^ (r % 8)
                const uint32_t panel = uint32_t(hf * (kHalf / 32) + c) * (BN * 128u);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t off = panel + row_off + uint32_t((j ^ (r & 7)) * 16);
                    *reinterpret_cast<float4*>(stage_k + off) =
                        make_float4(scale * __uint_as_float(rk[4 * j]), scale * __uint_as_float(rk[4 * j + 1]),
                                    scale * __uint_as_float(rk[4 * j + 2]), scale * __uint_as_float(rk[4 * j + 3]));
                    *reinterpret_cast<float4*>(stage_v + off) =
                        make_float4(__uint_as_float(rv[4 * j]), __uint_as_float(rv[4 * j + 1]),
                                    __uint_as_float(rv[4 * j + 2]), __uint_as_float(rv[4 * j + 3]));
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
#pragma unroll
                for (int c = 0; c < kHalf / 32; ++c) {
                    const int p = hf * (kHalf / 32) + c;
                    const uint32_t off = uint32_t(p) * (BN * 128u) + uint32_t(quad * 32) * 128u;
                    tma_store_2d(&map_dk, stage_k + off, kvh * D + p * 32, (int)(x0 + quad * 32));
                    tma_store_2d(&map_dv, stage_v + off, kvh * D + p * 32, (int)(x0 + quad * 32));
                }
                bulk_commit_group();
                bulk_wait_read_all();
            }
            __syncwarp();
        } else if (cnt == 0) {
            float* dkr = dk + (x * Hkv + kvh) * D + hf * kHalf;
            float* dvr = dv + (x * Hkv + kvh) * D + hf * kHalf;
            const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int j = 0; j < kHalf; j += 4) {
                __stcs(reinterpret_cast<float4*>(dkr + j), z);
                __stcs(reinterpret_cast<float4*>(dvr + j), z);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kKvMma) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// =================================================================== dQ
//
// Q and dO of the block's query tile stay in TMEM for the whole walk (the
// compute warps copy them there once, as the bf16 pairs an A operand takes), so
// all three MMAs read only their B operand from shared memory:
//   S = Q K_n^T (TS) -> TMEM S;   dP = dO V_n^T (TS) -> TMEM dP;
//   dS = P (dP - D) as bf16 over the dP columns just read;   dQ += dS K_n (TS).
// S of the next key tile is issued as soon as S has been read; dP of the next
// tile follows the dQ MMA that reads dS from the same columns.

constexpr int kQThreads = 320;                       // compute warps 0-7, MMA 8, TMA 9
constexpr int kQMma = 8, kQTma = 9;
constexpr int kKStages = 4, kVStages = 3;

template <int D>
struct QTiles {                                      // 1024-byte aligned
    __nv_bfloat16 k[kKStages][D / 64][BN * 64];
    __nv_bfloat16 v[kVStages][D / 64][BN * 64];
};

struct QBars {
    uint64_t k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages];
    uint64_t qd_tmem, s_full, s_read, dp_full, ds_full, mma_fin, stuck;
    uint32_t tmem_base;
    int abort_flag;
};

template <int D>
struct QSmem {
    QTiles<D> t;
    QBars b;
};

template <int D>
__global__ void __launch_bounds__(kQThreads, 1)
attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                      const __nv_bfloat16* __restrict__ qg, const __nv_bfloat16* __restrict__ dOg,
                      const float* __restrict__ lse2_hm, const float* __restrict__ D_hm, int64_t Qp,
                      const int32_t* __restrict__ s, const int32_t* __restrict__ a, int B, int64_t Qn, int H,
                      int gq, int64_t S, int m, int P, float scale, float scale_log2, const int4* __restrict__ qtb,
                      int pk, skv::RankCSR csr, float* __restrict__ dq, int* status, long long wait_limit) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t base_s = smem_u32(smem_raw);
    const uint32_t pad = ((base_s + 1023u) & ~1023u) - base_s;
    if (pad + sizeof(QSmem<D>) > (size_t)kSmemMax) {
        if (threadIdx.x == 0) skv::raise_status(status, SKV_ERR_UNSUPPORTED);
        return;
    }
    QSmem<D>& sm = *reinterpret_cast<QSmem<D>*>(smem_raw + pad);
    QTiles<D>& tl = sm.t;
    QBars& bb = sm.b;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // query tiles in descending order: the last tiles of a sample see the longest
    // windows, so the longest blocks start first and the grid's tail is short ones
    // A tile holds pk query heads (the group of one key/value head when pk > 1), each
    // over R = 128/pk query rows: tile row r is query row qt*R + r % R of head
    // h0 + r / R, so the group's heads share every K/V tile.
    const int qt = gridDim.x - 1 - blockIdx.x, h0 = blockIdx.y * pk;
    const int R = BM / pk;
    const int kvh = h0 / gq;                         // key/value head of these query heads
    constexpr int NP = D / 64;
    constexpr uint32_t kTile = BM * D * 2;
    const bool stuck_test = wait_limit < 0;
    if (stuck_test) wait_limit = -wait_limit;
    int4 bnd = qtb[qt];
    if (*(volatile int*)status == SKV_ERR_TIMEOUT) bnd.y = bnd.x;   // launch already void: no tiles
    // dq = sum_p dq^(p) over every rank's chunks: on one device that is the sum over
    // every key of the tile's windows, walked in ascending order (the ranks' chunks
    // tile [0, S) exactly, so the order changes only the fp32 rounding)
    KeyRange it;
    it.init(bnd.x, bnd.y);

    if (tid == 0) {
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(&bb.k_full[i], 1);
            mbar_init(&bb.k_empty[i], 1);
        }
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(&bb.v_full[i], 1);
            mbar_init(&bb.v_empty[i], 1);
        }
        mbar_init(&bb.qd_tmem, 256);
        mbar_init(&bb.s_full, 1);
        mbar_init(&bb.s_read, 256);
        mbar_init(&bb.dp_full, 1);
        mbar_init(&bb.ds_full, 256);
        mbar_init(&bb.mma_fin, 1);
        mbar_init(&bb.stuck, 1);
        bb.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kQMma) {
        tmem_alloc(&bb.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bb.tmem_base;
    // S, dP (dS bf16 over it), dQ accumulator, Q and dO as bf16 A operands
    const uint32_t tS = tmem, tP = tmem + 128, tQ = tmem + 256, tQin = tmem + 384, tDO = tmem + 448;
    auto abort_now = [&]() {
        atomicExch(&bb.abort_flag, 1);
        skv::raise_status(status, SKV_ERR_TIMEOUT);
    };

    if (warp == kQTma) {
        // ------------------------------------------------------------ TMA producer: K and V rings
        if (lane == 0) {
            int n = 0;       // key tiles whose K load was issued
            int nv = 0;      // key tiles whose V load was issued
            int64_t x0;
            // no L2 prefetch: the query tiles of a sample walk the same key tiles
            // close together, so K and V mostly come from L2 already (hints measured slower)
            bool first = true;
            while (it.next(x0)) {
                if (first) {
                    prefetch_tensormap(&map_k);
                    prefetch_tensormap(&map_v);
                    first = false;
                }
                const int ks = n % kKStages, vs = n % kVStages;
                if (n >= kKStages &&
                    !mbar_wait(&bb.k_empty[ks], ((n - kKStages) / kKStages) & 1, wait_limit, &bb.abort_flag)) {
                    abort_now();
                    break;
                }
                if (*(volatile int*)&bb.abort_flag) break;
                mbar_arrive_expect_tx(&bb.k_full[ks], kTile);
                for (int c = 0; c < NP; ++c) tma_load_2d(tl.k[ks][c], &map_k, &bb.k_full[ks], kvh * D + c * 64, (int)x0);
                ++n;
                if (n - 1 >= kVStages &&
                    !mbar_wait(&bb.v_empty[vs], ((n - 1 - kVStages) / kVStages) & 1, wait_limit, &bb.abort_flag)) {
                    abort_now();
                    break;
                }
                mbar_arrive_expect_tx(&bb.v_full[vs], kTile);
                for (int c = 0; c < NP; ++c) tma_load_2d(tl.v[vs][c], &map_v, &bb.v_full[vs], kvh * D + c * 64, (int)x0);
                ++nv;
            }
            // every copy issued has landed before the block exits
            for (int st = 0; st < kKStages && st < n; ++st) {
                const int last = st + ((n - 1 - st) / kKStages) * kKStages;
                mbar_wait(&bb.k_full[st], (last / kKStages) & 1, kTeardownWait);
            }
            for (int st = 0; st < kVStages && st < nv; ++st) {
                const int last = st + ((nv - 1 - st) / kVStages) * kVStages;
                mbar_wait(&bb.v_full[st], (last / kVStages) & 1, kTeardownWait);
            }
        }
    } else if (warp == kQMma) {
        // ------------------------------------------------------------ MMA issuer
        // the whole warp runs the schedule (warp-uniform descriptors and counters);
        // one elected lane issues each group of MMAs and its commits
        constexpr uint32_t idS = idesc_bf16_f32(BM, BN, 0, 0);    // M = queries, N = keys, K = d
        constexpr uint32_t idQ = idesc_bf16_f32(BM, D, 0, 1);     // M = queries, N = d, K = keys
        const int T = it.count();
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            return mbar_wait_warp(bar, parity, wait_limit, &bb.abort_flag);
        };
        bool issued = false;
        bool ok = T > 0;
        if (ok && stuck_test && !wait(&bb.stuck, 0)) ok = false;
        if (ok) ok = wait(&bb.qd_tmem, 0);
        // shared-memory descriptors as offsets (bytes / 16) from the first panel
        constexpr uint32_t kPanel = BN * 64 * 2 / 16, kSt = NP * kPanel;
        const uint64_t dK = smem_desc(smem_u32(tl.k[0][0]), 16, 1024), dV = smem_desc(smem_u32(tl.v[0][0]), 16, 1024);
        const uint64_t dKmn = smem_desc(smem_u32(tl.k[0][0]), BN * 128, 1024);
        auto issue_s = [&](int n) -> bool {            // S_n = Q K_n^T -> S
            const int ks = n % kKStages;
            if (!wait(&bb.k_full[ks], (n / kKStages) & 1)) return false;
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 2;
                    mma_ts(tS, tQin + kk * 8, dK + (ks * kSt + off), idS, kk > 0);
                }
                mma_commit(&bb.s_full);
            }
            __syncwarp();
            issued = true;
            return true;
        };
        auto issue_dp = [&](int n) -> bool {           // dP_n = dO V_n^T -> dP
            const int vs = n % kVStages;
            if (!wait(&bb.v_full[vs], (n / kVStages) & 1)) return false;
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 2;
                    mma_ts(tP, tDO + kk * 8, dV + (vs * kSt + off), idS, kk > 0);
                }
                mma_commit(&bb.dp_full);
                mma_commit(&bb.v_empty[vs]);
            }
            __syncwarp();
            issued = true;
            return true;
        };
        if (ok) ok = issue_s(0) && issue_dp(0);
        for (int n = 0; ok && n < T; ++n) {
            // S_{n+1} overwrites S as soon as the compute warps have read S_n
            if (n + 1 < T) {
                if (!wait(&bb.s_read, n & 1)) { ok = false; break; }
                tc_fence_after();
                if (!issue_s(n + 1)) { ok = false; break; }
            }
            if (!wait(&bb.ds_full, n & 1)) { ok = false; break; }
            tc_fence_after();
            // dQ += dS_n K_n: bf16 dS of key columns [64h, 64h+64) sits in TMEM columns
            // [64h, 64h+32) of dP
            const int ks = n % kKStages;
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_ts(tQ, tP + (kk >> 2) * 64 + (kk & 3) * 8, dKmn + (ks * kSt + kk * 128), idQ,
                           (n > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&bb.k_empty[ks]);
            }
            __syncwarp();
            // dP_{n+1} overwrites dP right behind the dQ MMA that reads dS_n from it
            if (n + 1 < T && !issue_dp(n + 1)) { ok = false; break; }
        }
        if (!ok && T > 0 && lane == 0) abort_now();
        if (issued) {
            if (elect_one()) mma_commit(&bb.mma_fin);
            __syncwarp();
            if (!mbar_wait_warp(&bb.mma_fin, 0, kTeardownWait) && lane == 0)
                skv::raise_status(status, SKV_ERR_TIMEOUT);
        }
    } else {
        // ------------------------------------------------------------ compute warps 0-7
        // warp w owns query rows (TMEM lanes) of quadrant w%4 and key columns
        // [64*hf, 64*hf+64) with hf = w/4
        constexpr unsigned kAll = 0xffffffffu;
        const int quad = warp & 3, hf = warp >> 2;
        const uint32_t lane_base = uint32_t(quad * 32) << 16;
        const int r = quad * 32 + lane;
        const int64_t row = int64_t(qt) * R + r % R;
        const int h = h0 + r / R;                        // this row's query head
        const bool live = row < Qn;
        int64_t rlo = 0, rhi = 0;
        if (live) skv::block_window(s, a, (int)(row / B), S, rlo, rhi);
        bool ok = true;
        auto uniform_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
            const bool got = mbar_wait_warp(bar, parity, wait_limit, &bb.abort_flag);
            if (!got && lane == 0) abort_now();
            return got;
        };
        {   // this row of Q (warps of half 0) or dO (half 1) into TMEM as bf16 pairs
            const __nv_bfloat16* src = (hf == 0 ? qg : dOg) + (row * H + h) * D;
            const uint32_t dst = (hf == 0 ? tQin : tDO) + lane_base;
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t w[32];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    uint4 v4 = make_uint4(0u, 0u, 0u, 0u);
                    if (live) v4 = *reinterpret_cast<const uint4*>(src + c * 64 + u * 8);
                    w[4 * u] = v4.x;
                    w[4 * u + 1] = v4.y;
                    w[4 * u + 2] = v4.z;
                    w[4 * u + 3] = v4.w;
                }
                tmem_st32(dst + c * 32, w);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bb.qd_tmem);
        }
        const float l2 = live ? lse2_hm[int64_t(h) * Qp + row] : INFINITY;
        const float Dr = live ? D_hm[int64_t(h) * Qp + row] : 0.f;
        int64_t x0;
        int n = 0;
        while (it.next(x0)) {
            if (__any_sync(kAll, *(volatile int*)&bb.abort_flag != 0)) { ok = false; break; }
            const bool full = (x0 >= bnd.z) && (x0 + BN <= bnd.w);
            if (!uniform_wait(&bb.s_full, n & 1)) { ok = false; break; }
            tc_fence_after();
            uint32_t sraw[2][32];
            tmem_ld32(tS + lane_base + hf * 64, sraw[0]);
            tmem_ld32(tS + lane_base + hf * 64 + 32, sraw[1]);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&bb.s_read);                     // S is free for the next tile
            float pr[2][32];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t keep = 0xffffffffu;              // key columns this row sees
                if (!full) {                              // boundary tile only
                    const int64_t xc = x0 + hf * 64 + c * 32;
                    const int64_t lo = rlo - xc, hi = rhi - xc;   // window relative to the chunk
                    keep = 0u;
                    if (hi > 0 && lo < 32) {
                        const int b0 = lo > 0 ? (int)lo : 0, b1 = hi < 32 ? (int)hi : 32;
                        keep = (b1 >= 32 ? 0xffffffffu : ((1u << b1) - 1u)) & ~((1u << b0) - 1u);
                    }
                }
                if (full) {
                    const float2 sc2 = make_float2(scale_log2, scale_log2), nl2 = make_float2(-l2, -l2);
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const float2 z = __ffma2_rn(
                            make_float2(__uint_as_float(sraw[c][j]), __uint_as_float(sraw[c][j + 1])), sc2, nl2);
                        pr[c][j] = ex2(z.x);
                        pr[c][j + 1] = ex2(z.y);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        pr[c][j] = ((keep >> j) & 1u) ? ex2(fmaf(__uint_as_float(sraw[c][j]), scale_log2, -l2)) : 0.f;
                }
            }
            if (!uniform_wait(&bb.dp_full, n & 1)) { ok = false; break; }
            tc_fence_after();
            uint32_t draw[2][32];
            tmem_ld32(tP + lane_base + hf * 64, draw[0]);
            tmem_ld32(tP + lane_base + hf * 64 + 32, draw[1]);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t pk[16];
                const float2 nd2 = make_float2(-Dr, -Dr);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float2 t = __fadd2_rn(
                        make_float2(__uint_as_float(draw[c][2 * j]), __uint_as_float(draw[c][2 * j + 1])), nd2);
                    const float2 dd = __fmul2_rn(make_float2(pr[c][2 * j], pr[c][2 * j + 1]), t);
                    pk[j] = pack_bf16(dd.x, dd.y);
                }
                // bf16 dS of key columns [64hf + 32c, +32) -> TMEM columns [64hf + 16c, +16)
                // of dP: inside this warp's half, over columns read already
                tmem_st16(tP + lane_base + hf * 64 + c * 16, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bb.ds_full);
            ++n;
        }
        // dq rows (scaled), columns split between the two halves; zeros if no key
        const bool aborted = __any_sync(kAll, *(volatile int*)&bb.abort_flag != 0);
        constexpr int kHalf = D / 2;
        float* dqr = dq + (row * H + h) * D + hf * kHalf;
        if (n > 0 && ok && !aborted && uniform_wait(&bb.mma_fin, 0)) {
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < kHalf / 32; ++c) {
                uint32_t rq[32];
                tmem_ld32(tQ + lane_base + hf * kHalf + c * 32, rq);
                tmem_ld_wait();
                if (live) {
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        __stcs(reinterpret_cast<float4*>(dqr + c * 32 + j),
                               make_float4(scale * __uint_as_float(rq[j]), scale * __uint_as_float(rq[j + 1]),
                                           scale * __uint_as_float(rq[j + 2]), scale * __uint_as_float(rq[j + 3])));
                }
            }
        } else if (n == 0 && live) {
#pragma unroll
            for (int j = 0; j < kHalf; j += 4) __stcs(reinterpret_cast<float4*>(dqr + j), make_float4(0.f, 0.f, 0.f, 0.f));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kQMma) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ============================================================== host side

struct BwdScratch {
    int4* qtb;          // per 128-row query tile
    int32_t* cnt;
    int32_t* list;
    int4* gtb;          // per tile of the dQ kernel (stacked heads), or qtb
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
    // key bounds of the dQ kernel's tiles when they stack a group's query heads
    const int pk = skv_tc::pack_heads(pb);
    const int64_t n_gt = pk > 1 ? (Qn + BM / pk - 1) / (BM / pk) : 0;
    const size_t o_gtb = off; off = align256(off + size_t(n_gt) * sizeof(int4));
    if (w) {
        w->qtb = reinterpret_cast<int4*>(base + o_qtb);
        w->cnt = reinterpret_cast<int32_t*>(base + o_cnt);
        w->list = reinterpret_cast<int32_t*>(base + o_list);
        w->gtb = pk > 1 ? reinterpret_cast<int4*>(base + o_gtb) : w->qtb;
    }
    return off;
}

template <int D>
skv_status launch_bwd(const skv_problem& pb, const void* q, const void* k, const void* v, const void* dO,
                      const float* lse2_hm, const float* D_hm, skv::RankCSR csr, float* dq, float* dk, float* dv,
                      void* scratch, const skv_host::Ctx& c) {
    const int64_t Qn = int64_t(pb.n_blocks) * pb.B;
    const int n_qt = (int)((Qn + BM - 1) / BM);
    const int64_t Qp = int64_t(n_qt) * BM;
    const int n_kv = (int)(pb.S / BN);
    BwdScratch w;
    scratch_layout(pb, &w, static_cast<char*>(scratch));
    qtile_bounds_kernel<<<(n_qt + 127) / 128, 128, 0, c.stream>>>(pb.s, pb.a, pb.B, Qn, pb.S, n_qt, w.qtb, BM);
    SKV_LAUNCHED();
    kv_list_kernel<<<(n_kv + 7) / 8, 256, 0, c.stream>>>(w.qtb, n_qt, n_kv, w.cnt, w.list);
    SKV_LAUNCHED();
    const int pk = skv_tc::pack_heads(pb), R = BM / pk;
    const int n_gt = (int)((Qn + R - 1) / R);
    if (pk > 1) {
        qtile_bounds_kernel<<<(n_gt + 127) / 128, 128, 0, c.stream>>>(pb.s, pb.a, pb.B, Qn, pb.S, n_gt, w.gtb, R);
        SKV_LAUNCHED();
    }
    CUtensorMap mq, mdo, mk, mv, mdk, mdv;
    const int64_t cols = int64_t(pb.n_heads) * D, kv_cols = int64_t(pb.n_kv_heads) * D;
    const int gq = pb.n_heads / pb.n_kv_heads;
    if (!make_map(&mq, q, Qn, cols) || !make_map(&mdo, dO, Qn, cols) || !make_map(&mk, k, pb.S, kv_cols) ||
        !make_map(&mv, v, pb.S, kv_cols) || !make_map_f32(&mdk, dk, pb.S, kv_cols) ||
        !make_map_f32(&mdv, dv, pb.S, kv_cols))
        return SKV_ERR_CUDA;
    const float scale_log2 = pb.scale * 1.4426950408889634f;
    {
        auto kern = attn_bwd_dkdv_tc_kernel<D>;
        SKV_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax));
        skv_host::timer_begin(skv_host::kTimeBwdKV, c.stream);
        kern<<<dim3((unsigned)n_kv, (unsigned)pb.n_kv_heads), kKvThreads, kSmemMax, c.stream>>>(
            mq, mdo, mk, mv, mdk, mdv, lse2_hm, D_hm, Qp, pb.s, pb.a, pb.B, Qn, pb.n_kv_heads, gq, pb.S, pb.scale,
            scale_log2, w.qtb, w.cnt, w.list, n_qt, dk, dv, c.status, c.wait_limit);
        skv_host::timer_end(skv_host::kTimeBwdKV, c.stream);
        SKV_LAUNCHED();
    }
    {
        auto kern = attn_bwd_dq_tc_kernel<D>;
        SKV_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax));
        skv_host::timer_begin(skv_host::kTimeBwdQ, c.stream);
        kern<<<dim3((unsigned)n_gt, (unsigned)(pb.n_heads / pk)), kQThreads, kSmemMax, c.stream>>>(
            mk, mv, static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(dO), lse2_hm, D_hm, Qp,
            pb.s, pb.a, pb.B, Qn, pb.n_heads, gq, pb.S, pb.m, pb.P, pb.scale, scale_log2, w.gtb, pk, csr, dq,
            c.status, c.wait_limit);
        skv_host::timer_end(skv_host::kTimeBwdQ, c.stream);
        SKV_LAUNCHED();
    }
    return SKV_OK;
}

}  // namespace

namespace skv_tc {

skv_status launch_qtile_bounds(const skv_problem& pb, int4* out, const skv_host::Ctx& c, int rows) {
    const int64_t Qn = int64_t(pb.n_blocks) * pb.B;
    const int64_t n_qt = (Qn + rows - 1) / rows;
    if (n_qt == 0) return SKV_OK;
    qtile_bounds_kernel<<<(unsigned)((n_qt + 127) / 128), 128, 0, c.stream>>>(pb.s, pb.a, pb.B, Qn, pb.S, (int)n_qt, out,
                                                                            rows);
    SKV_LAUNCHED();
    return SKV_OK;
}

bool bwd_supported(const skv_problem& pb) {
    return pb.dtype == SKV_BF16 && (pb.head_dim == 64 || pb.head_dim == 128) && pb.m % BN == 0 &&
           pb.n_heads <= 65535 && pb.S <= INT32_MAX;
}

size_t bwd_scratch_bytes(const skv_problem& pb) {
    return bwd_supported(pb) ? scratch_layout(pb, nullptr, nullptr) : 0;
}

skv_status launch_attn_bwd_tc(const skv_problem& pb, const void* q, const void* k, const void* v, const void* dO,
                              const float* lse2, const float* D, skv::RankCSR csr, float* dq, float* dk, float* dv,
                              void* scratch, const skv_host::Ctx& c) {
    if (pb.head_dim == 128) return launch_bwd<128>(pb, q, k, v, dO, lse2, D, csr, dq, dk, dv, scratch, c);
    return launch_bwd<64>(pb, q, k, v, dO, lse2, D, csr, dq, dk, dv, scratch, c);
}

}  // namespace skv_tc
