// Tensor-core anchor attention forward of libskv for GB300 (sm_103a): tcgen05
// MMA with TMEM accumulators, TMA-fed bf16 operands, warp-specialised roles.
//
// Forward [Split-KV §4.1 Eq. 3; the per-rank attention of Alg. 1 in "Split-KV: Efficient Context
// Parallelism for Training Diffusion Drafters"]: one thread block computes the
// partials (o_p, l_p) of two consecutive 128-row query tiles, one head and one
// virtual rank p.  The key tiles it visits are the 128-key tiles of rank p's
// chunks that intersect the union of its rows' windows [s_i, a_i) (§3.1
// Fig. 1); every other tile is never loaded.  Tiles inside every row's window
// are processed unmasked; only boundary tiles get the per-row compare.
// Grouped-query layouts [Split-KV Table 2] stack the g query heads of one
// key/value head in a tile, 128/g rows each (row r of the tile is query row
// r % (128/g) of the tile's row range, head r / (128/g) of the group): one K/V
// tile then serves the whole group, and a tile's rows come from g times fewer
// blocks, so fewer of its key tiles are boundary tiles.  A rank whose chunks
// miss both tiles' windows only marks their rows empty.
//
// The two query tiles share every K/V tile and alternate on the tensor core,
// so one tile's exponentials overlap the other tile's MMAs.  Roles (384 threads):
//   warps 0-3, 4-7  softmax of query tile 0, 1: thread owns one row; reads S
//                   from TMEM, online max / exp2 / sum, bf16 P back to TMEM (over
//                   S), rescales O when the running max grows by more than 2^8.
//   warp 8          MMA issuer (one elected lane): S_j = Q_j K^T (SS), O_j += P_j V (TS).
//   warp 9          TMA producer (one thread): Q_0, Q_1 once, K/V through 2 stages.
//   warps 10-11     none (they complete the third warpgroup, whose registers go to
//                   the softmax warpgroups).
// TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,384), O_1 [384,512).
// bf16 P_j lies over the first 64 columns of S_j (read whole into registers first).
// The softmax warpgroups take 216 registers per thread, the issuing warpgroup 64.
// Issue order per key tile n: PV_0(n), S_0(n+1), PV_1(n), S_1(n+1); hence when
// S_j(n) has completed, PV_j(n-1) has too and O_j may be rescaled without a wait.
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
constexpr int kFwdThreads = 384;                     // warpgroups: softmax 0, softmax 1, MMA/TMA
constexpr int kMmaWarp = 8, kTmaWarp = 9;            // warps 10-11 only hand their registers over
constexpr int kRegLaunch = 168, kRegSoftmax = 216, kRegIssue = 64;   // per thread
static_assert(2 * 128 * kRegSoftmax + 128 * kRegIssue <= kFwdThreads * kRegLaunch, "register split");
constexpr long long kTeardownWait = 2000000000LL;   // ns; in-flight copies / MMAs end in microseconds
constexpr int kListCap = 64;                          // chunk indices staged in shared memory

template <int D>
struct __align__(1024) FwdSmem {
    __nv_bfloat16 q[2][D / 64][BM * 64];
    __nv_bfloat16 k[kStages][D / 64][BN * 64];
    __nv_bfloat16 v[kStages][D / 64][BN * 64];
    uint64_t q_full;
    uint64_t k_full[kStages], v_full[kStages], kv_empty[kStages];
    uint64_t s_full[2], p_full[2];
    uint64_t mma_fin;
    uint64_t stuck;             // never completed: target of the forced-timeout test mode
    int32_t clist[kListCap];    // rank p's chunk indices (when they fit)
    int list_off, list_n;
    uint32_t tmem_base;
    int abort_flag;
};

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_o,
                   const int32_t* __restrict__ s,
                   const int32_t* __restrict__ a, int B, int64_t Qn, int H, int gq, int64_t S, int m,
                   float scale_log2, skv::RankCSR csr, const int4* __restrict__ qtb, int n_qt, int pk,
                   float* __restrict__ o_part, float* __restrict__ lse_part, int* status, long long wait_limit) {
    extern __shared__ unsigned char smem_raw[];
    FwdSmem<D>& sm = *reinterpret_cast<FwdSmem<D>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // query tile pairs in descending order: the last tiles of a sample see the longest
    // windows, so the longest blocks start first and each head's tail is short ones.
    // A tile holds pk query heads (the group of one key/value head when pk > 1), each
    // over R = 128/pk query rows: tile row r is query row qt*R + r % R of head
    // h0 + r / R, so the group's heads share every K/V tile.
    const int qt0 = 2 * (gridDim.x - 1 - blockIdx.x), h0 = blockIdx.y * pk, p = blockIdx.z;
    const int R = BM / pk;
    const int kvh = h0 / gq;                         // key/value head of these query heads
    constexpr int NP = D / 64;                       // 64-column panels per row
    constexpr uint32_t kTileBytes = BN * D * 2;      // one K or V tile (== Q tile)

    // test mode (negative limit): every block first waits on a barrier nothing
    // completes, so the timeout path runs deterministically
    const bool stuck_test = wait_limit < 0;
    if (stuck_test) wait_limit = -wait_limit;
    // the tiles' key bounds (union and full-visibility range), computed by a pre-pass
    const int4 b0 = qtb[qt0];
    const int4 b1 = qt0 + 1 < n_qt ? qtb[qt0 + 1] : make_int4((int)S, 0, 0, 0);
    const TileBounds tb0{b0.x, b0.y, b0.z, b0.w}, tb1{b1.x, b1.y, b1.z, b1.w};
    int64_t lo = tb0.lo < tb1.lo ? tb0.lo : tb1.lo;
    int64_t hi = tb0.hi > tb1.hi ? tb0.hi : tb1.hi;
    // once any block of the launch has timed out the result is void: the
    // remaining blocks skip their work instead of each waiting out a deadline
    if (*(volatile int*)status == SKV_ERR_TIMEOUT) hi = lo;
    // a rank holding no key of the two tiles' windows (half of all blocks when a
    // rank keeps one chunk of each sample) only marks the tiles' rows empty:
    // lse_part = -inf, o_part unspecified; no barriers, no TMEM
    {
        TileIter probe;
        probe.init(csr, p, p + 1, m, lo, hi);
        if (probe.count() == 0) {
            if (warp < 8) {
                const int r = (warp & 3) * 32 + lane;
                const int64_t row = int64_t(qt0 + (warp >> 2)) * R + r % R;
                if (row < Qn) lse_part[(int64_t(p) * Qn + row) * H + h0 + r / R] = -INFINITY;
            }
            return;
        }
    }

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
        }
        mbar_init(&sm.mma_fin, 1);
        mbar_init(&sm.stuck, 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    if (warp == 0) {   // rank p's chunk list into shared memory, one coalesced read
        const int c0 = csr.ptr[p], nc = csr.ptr[p + 1] - c0;
        if (nc <= kListCap)
            for (int i = lane; i < nc; i += 32) sm.clist[i] = csr.list[c0 + i];
        if (lane == 0) {
            sm.list_off = c0;
            sm.list_n = nc;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    TileIter it;
    it.init_list(sm.list_n <= kListCap ? sm.clist : csr.list + sm.list_off, sm.list_n, m, lo, hi);
    auto abort_now = [&]() {
        atomicExch(&sm.abort_flag, 1);
        skv::raise_status(status, SKV_ERR_TIMEOUT);
    };

    if (warp < 8) {
        warpgroup_reg_alloc<kRegSoftmax>();
        // ------------------------------------------------------------ softmax
        // tcgen05.ld/st are warp-collective: every branch around them is made
        // warp-uniform (__any_sync / __all_sync); per-row choices are data.
        constexpr unsigned kAll = 0xffffffffu;
        const int j = warp >> 2;                       // query tile of this warpgroup
        const int quad = warp & 3;
        const int r = quad * 32 + lane;                // row inside the tile == TMEM lane
        const int64_t row = int64_t(qt0 + j) * R + r % R;
        const int h = h0 + r / R;                      // this row's query head
        const bool live = row < Qn;
        // positions fit in int32 here (anchors are int32 and S < 2^31 on this path)
        int rlo = 0, rhi = 0;
        {
            int64_t l64 = 0, h64 = 0;
            if (live) skv::block_window(s, a, (int)(row / B), S, l64, h64);
            rlo = (int)l64;
            rhi = (int)h64;
        }
        const int flo = (int)(j ? tb1.flo : tb0.flo), fhi = (int)(j ? tb1.fhi : tb0.fhi);
        const uint32_t lane_base = uint32_t(quad * 32) << 16;
        const uint32_t tS = tmem + j * 128, tO = tmem + 256 + j * 128;
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        auto uniform_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
            const bool got = mbar_wait_warp(bar, parity, wait_limit, &sm.abort_flag);
            if (!got && lane == 0) abort_now();
            return got;
        };
        int64_t x0;
        int n = 0;
        while (ok && it.next(x0)) {
            if (__any_sync(kAll, *(volatile int*)&sm.abort_flag != 0)) { ok = false; break; }
            if (!uniform_wait(&sm.s_full[j], n & 1)) { ok = false; break; }
            tc_fence_after();
            // the row's 128 scores in registers (one TMEM round), -inf outside this
            // row's window on boundary tiles
            const int xt = (int)x0;
            const bool full = (xt >= flo) && (xt + BN <= fhi);
            uint32_t sv[BN / 32][32];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) tmem_ld32(tS + lane_base + c * 32, sv[c]);
            tmem_ld_wait();
            if (!full) {
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) {
                    const int lo_c = rlo - (xt + 32 * c), hi_c = rhi - (xt + 32 * c);
                    uint32_t keep = 0u;
                    if (hi_c > 0 && lo_c < 32) {
                        const int b0 = lo_c > 0 ? lo_c : 0, b1 = hi_c < 32 ? hi_c : 32;
                        keep = (b1 >= 32 ? 0xffffffffu : ((1u << b1) - 1u)) & ~((1u << b0) - 1u);
                    }
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj)
                        if (!((keep >> jj) & 1u)) sv[c][jj] = 0xff800000u;   // -inf
                }
            }
            // row max: four independent chains of three-input maxima
            float m4[BN / 32];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
                m4[c] = -INFINITY;
#pragma unroll
                for (int jj = 0; jj < 32; jj += 2)
                    m4[c] = fmax3(m4[c], __uint_as_float(sv[c][jj]), __uint_as_float(sv[c][jj + 1]));
            }
            const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            const float mx_s = mx * scale_log2;
            bool rescale = false;
            float alpha = 1.f;
            if (mx_s > m_ref + 8.f) {
                alpha = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - mx_s);
                rescale = (l > 0.f);
                m_ref = mx_s;
            }
            l *= alpha;
            // P = 2^(z scale log2e - m) as bf16 pairs: keys [32c, 32c+32) -> columns [16c, 16c+16)
            const float neg = (m_ref == -INFINITY) ? 0.f : -m_ref;
            const float2 sc2 = make_float2(scale_log2, scale_log2), ng2 = make_float2(neg, neg);
            float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const float2 z = __ffma2_rn(
                        make_float2(__uint_as_float(sv[c][2 * jj]), __uint_as_float(sv[c][2 * jj + 1])), sc2, ng2);
                    const float2 pv = make_float2(ex2(z.x), ex2(z.y));
                    sum2[jj & 1] = __fadd2_rn(sum2[jj & 1], pv);
                    pk[jj] = pack_bf16(pv.x, pv.y);
                }
                tmem_st16(tS + lane_base + c * 16, pk);
            }
            l += (sum2[0].x + sum2[0].y) + (sum2[1].x + sum2[1].y);
            // O_j is final for tiles < n here (S_j(n) was issued after PV_j(n-1)); PV_j(n)
            // waits for p_full below
            if (__any_sync(kAll, rescale)) {
                const float f = rescale ? alpha : 1.f;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t rr[32];
                    tmem_ld32(tO + lane_base + c * 32, rr);
                    tmem_ld_wait();
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) rr[jj] = __float_as_uint(__uint_as_float(rr[jj]) * f);
                    tmem_st32(tO + lane_base + c * 32, rr);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sm.p_full[j]);
            ++n;
        }
        // every MMA (the last PV included) has completed once mma_fin fires
        const bool aborted = __any_sync(kAll, *(volatile int*)&sm.abort_flag != 0);
        if (ok && !aborted && (n == 0 || uniform_wait(&sm.mma_fin, 0))) {
            const bool mine = live && l > 0.f;
            const float inv = mine ? 1.f / l : 0.f;
            if (n > 0 && __any_sync(kAll, mine)) {
                // o_j rows leave through the (now idle) K/V ring: each warp stages its 32 rows
                // as 128-byte-swizzled 32 x 32 fp32 boxes (16-byte chunk u of row r at chunk
                // u ^ (r % 8)) and writes them with TMA stores; rows past Qn are dropped.
                // Rows that see no key are written as zeros (their lse_part is -inf).
                tc_fence_after();
                unsigned char* stage = reinterpret_cast<unsigned char*>(&sm.k[0][0][0]) + j * (D / 32) * (BM * 128);
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t rr[32];
                    tmem_ld32(tO + lane_base + c * 32, rr);
                    tmem_ld_wait();
                    unsigned char* panel = stage + c * (BM * 128) + r * 128;
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const float4 v4 = mine ? make_float4(__uint_as_float(rr[4 * u]) * inv,
                                                             __uint_as_float(rr[4 * u + 1]) * inv,
                                                             __uint_as_float(rr[4 * u + 2]) * inv,
                                                             __uint_as_float(rr[4 * u + 3]) * inv)
                                               : make_float4(0.f, 0.f, 0.f, 0.f);
                        *reinterpret_cast<float4*>(panel + ((u ^ (r & 7)) * 16)) = v4;
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    // boxes of min(R, 32) rows, each inside one head's rows
                    const int BR = R < 32 ? R : 32;
#pragma unroll
                    for (int c = 0; c < D / 32; ++c)
                        for (int rr = quad * 32; rr < quad * 32 + 32; rr += BR)
                            tma_store_3d(&map_o, stage + c * (BM * 128) + rr * 128, (h0 + rr / R) * D + c * 32,
                                         (qt0 + j) * R + rr % R, p);
                    bulk_commit_group();
                    bulk_wait_read_all();
                }
                __syncwarp();
            }
            if (live)
                lse_part[(int64_t(p) * Qn + row) * H + h] =
                    mine ? (m_ref + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        }
    } else {
        warpgroup_reg_dealloc<kRegIssue>();
        if (warp == kTmaWarp) {
            // ------------------------------------------------------------ producer
            if (lane == 0) {
                int n = 0;
                int64_t x0;
                bool any = false;
                while (it.next(x0)) {
                    if (!any) {
                        prefetch_tensormap(&map_k);
                        prefetch_tensormap(&map_v);
                        mbar_arrive_expect_tx(&sm.q_full, 2 * kTileBytes);
                        // tile j: rows [k R, k R + R) of each panel from head h0 + k
                        for (int j = 0; j < 2; ++j)
                            for (int k = 0; k < pk; ++k)
                                for (int c = 0; c < NP; ++c)
                                    tma_load_2d(&sm.q[j][c][k * R * 64], &map_q, &sm.q_full, (h0 + k) * D + c * 64,
                                                (qt0 + j) * R);
                        any = true;
                    }
                    const int st = n % kStages;
                    if (n >= kStages &&
                        !mbar_wait(&sm.kv_empty[st], ((n - kStages) / kStages) & 1, wait_limit, &sm.abort_flag)) {
                        abort_now();
                        break;
                    }
                    if (*(volatile int*)&sm.abort_flag) break;
                    mbar_arrive_expect_tx(&sm.k_full[st], kTileBytes);
                    for (int c = 0; c < NP; ++c)
                        tma_load_2d(sm.k[st][c], &map_k, &sm.k_full[st], kvh * D + c * 64, (int)x0);
                    mbar_arrive_expect_tx(&sm.v_full[st], kTileBytes);
                    for (int c = 0; c < NP; ++c)
                        tma_load_2d(sm.v[st][c], &map_v, &sm.v_full[st], kvh * D + c * 64, (int)x0);
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
        } else if (warp == kMmaWarp) {
            // ------------------------------------------------------------ MMA issuer
            // The whole warp runs the schedule, so descriptors and counters are
            // warp-uniform; one elected lane issues each group of MMAs and its commit.
            constexpr uint32_t idS = idesc_bf16_f32(BM, BN, 0, 0);
            constexpr uint32_t idO = idesc_bf16_f32(BM, D, 0, 1);
            const int T = it.count();
            auto wait = [&](uint64_t* bar, uint32_t parity) {
                return mbar_wait_warp(bar, parity, wait_limit, &sm.abort_flag);
            };
            bool ok = T > 0;
            bool issued = false;   // any MMA in flight to wait for before TMEM is freed
            if (ok && stuck_test && !wait(&sm.stuck, 0)) ok = false;
            if (ok) ok = wait(&sm.q_full, 0);
            // shared-memory descriptors: the start-address field (bytes / 16) of a panel,
            // stage or K step is an offset from the first one (every address < 256 KiB)
            constexpr uint32_t kPanel = BN * 64 * 2 / 16, kStage = NP * kPanel;
            const uint64_t dq = smem_desc(smem_u32(sm.q[0][0]), 16, 1024);
            const uint64_t dk = smem_desc(smem_u32(sm.k[0][0]), 16, 1024);
            const uint64_t dv = smem_desc(smem_u32(sm.v[0][0]), BN * 128, 1024);
            auto issue_s = [&](int j, int n) -> bool {    // S_j = Q_j K_n^T -> TMEM [128 j, 128 j + 128)
                const int st = n % kStages;
                // K_n has landed once S_0(n) could be issued
                if (j == 0 && !wait(&sm.k_full[st], (n / kStages) & 1)) return false;
                tc_fence_after();
                if (elect_one()) {
    #pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 2;
                        mma_ss(tmem + j * 128, dq + (j * kStage + off), dk + (st * kStage + off), idS, kk > 0);
                    }
                    mma_commit(&sm.s_full[j]);
                }
                __syncwarp();
                issued = true;
                return true;
            };
            auto issue_pv = [&](int j, int n) -> bool {   // O_j += P_j V_n (bf16 P_j over S_j)
                const int st = n % kStages;
                if (!wait(&sm.p_full[j], n & 1)) return false;
                // V_n has landed once PV_0(n) could be issued
                if (j == 0 && !wait(&sm.v_full[st], (n / kStages) & 1)) return false;
                tc_fence_after();
                if (elect_one()) {
    #pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        mma_ts(tmem + 256 + j * 128, tmem + j * 128 + kk * 8, dv + (st * kStage + kk * 128), idO,
                               (n > 0 || kk > 0) ? 1u : 0u);
                    if (j == 1) mma_commit(&sm.kv_empty[st]);   // both PVs of tile n have read V_n
                }
                __syncwarp();
                return true;
            };
            if (ok) ok = issue_s(0, 0) && issue_s(1, 0);
            for (int n = 0; ok && n < T; ++n) {
                // S_j(n+1) overwrites S_j right behind the PV_j(n) that reads P_j from it
                if (!issue_pv(0, n)) { ok = false; break; }
                if (n + 1 < T && !issue_s(0, n + 1)) { ok = false; break; }
                if (!issue_pv(1, n)) { ok = false; break; }
                if (n + 1 < T && !issue_s(1, n + 1)) { ok = false; break; }
            }
            if (!ok && T > 0 && lane == 0) abort_now();
            // all MMAs the warp issued have completed before TMEM is freed
            if (issued) {
                if (elect_one()) mma_commit(&sm.mma_fin);
                __syncwarp();
                if (!mbar_wait_warp(&sm.mma_fin, 0, kTeardownWait) && lane == 0)
                    skv::raise_status(status, SKV_ERR_TIMEOUT);
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

template <int D>
skv_status launch_fwd(const skv_problem& pb, const void* q, const void* k, const void* v, skv::RankCSR csr,
                      float* o_part, float* lse_part, void* scratch, const skv_host::Ctx& c) {
    const int64_t Qn = int64_t(pb.n_blocks) * pb.B;
    const int pk = skv_tc::pack_heads(pb), R = BM / pk;
    CUtensorMap mq, mk, mv, mo;
    if (!make_map(&mq, q, Qn, int64_t(pb.n_heads) * D, R) || !make_map(&mk, k, pb.S, int64_t(pb.n_kv_heads) * D) ||
        !make_map(&mv, v, pb.S, int64_t(pb.n_kv_heads) * D) ||
        !make_map_f32_3d(&mo, o_part, pb.P, Qn, int64_t(pb.n_heads) * D, R < 32 ? R : 32))
        return SKV_ERR_CUDA;
    size_t smem = sizeof(FwdSmem<D>) + 1024;
    if (smem < 120 * 1024) smem = 120 * 1024;   // one block per SM: it owns all 512 TMEM columns
    auto kern = attn_fwd_tc_kernel<D>;
    SKV_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    // the warpgroups' register split must fit the allocation the block launches with,
    // or the softmax warpgroups' setmaxnreg.inc would never be granted
    cudaFuncAttributes fa;
    SKV_CUDA_CHECK(cudaFuncGetAttributes(&fa, kern));
    if (fa.numRegs * kFwdThreads < 2 * 128 * kRegSoftmax + 128 * kRegIssue) return SKV_ERR_UNSUPPORTED;
    const int64_t n_qt = (Qn + R - 1) / R;               // tiles of R rows x pk heads
    int4* qtb = static_cast<int4*>(scratch);
    skv_status st = skv_tc::launch_qtile_bounds(pb, qtb, c, R);
    if (st != SKV_OK) return st;
    const dim3 grid((unsigned)((n_qt + 1) / 2), (unsigned)(pb.n_heads / pk), (unsigned)pb.P);
    const float scale_log2 = pb.scale * 1.4426950408889634f;
    skv_host::timer_begin(skv_host::kTimeFwd, c.stream);
    kern<<<grid, kFwdThreads, smem, c.stream>>>(mq, mk, mv, mo, pb.s, pb.a, pb.B, Qn, pb.n_heads,
                                                pb.n_heads / pb.n_kv_heads, pb.S, pb.m, scale_log2,
                                                csr, qtb, (int)n_qt, pk, o_part, lse_part, c.status, c.wait_limit);
    skv_host::timer_end(skv_host::kTimeFwd, c.stream);
    SKV_LAUNCHED();
    return SKV_OK;
}

}  // namespace

namespace skv_tc {

bool fwd_supported(const skv_problem& pb) {
    return pb.dtype == SKV_BF16 && (pb.head_dim == 64 || pb.head_dim == 128) && pb.m % BN == 0 &&
           pb.P <= 65535 && pb.n_heads <= 65535 && pb.S <= INT32_MAX &&
           int64_t(pb.n_blocks) * pb.B <= INT32_MAX;
}
size_t fwd_scratch_bytes(const skv_problem& pb) {   // per query tile key bounds (int4); none off this path
    if (!fwd_supported(pb)) return 0;
    const int64_t Qn = int64_t(pb.n_blocks) * pb.B;
    const int R = BM / pack_heads(pb);
    return size_t((Qn + R - 1) / R) * sizeof(int4);
}

skv_status launch_attn_fwd_tc(const skv_problem& pb, const void* q, const void* k, const void* v, skv::RankCSR csr,
                              float* o_part, float* lse_part, void* scratch, const skv_host::Ctx& c) {
    if (pb.head_dim == 128) return launch_fwd<128>(pb, q, k, v, csr, o_part, lse_part, scratch, c);
    return launch_fwd<64>(pb, q, k, v, csr, o_part, lse_part, scratch, c);
}

}  // namespace skv_tc
