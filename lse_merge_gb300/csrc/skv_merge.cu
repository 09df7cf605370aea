// Bandwidth-bound passes of libskv: the exact LSE merge of per-rank partials
// [Split-KV §4.1, Eq. 4; the merge step of Alg. 1], the backward pre-pass
// D_r = dO_r . o_r (Alg. 1's MERGE_BWD, merged form) and the dq sum over ranks
// (Alg. 1's dq reduce-scatter made local).  "Split-KV: Efficient Context Parallelism for
// Training Diffusion Drafters".
//
// The merge is one HBM pass: G = d/4 lanes own one row (16-byte vectors, rows
// of 64 or 128 floats are one or half a warp); the row's P log-sum-exps are
// loaded one per lane, reduced with warp shuffles, and only partials with a
// finite l_p are read -- so the bytes moved are the algorithmic ones.  Its
// backward per partial (MERGE_BWD) walks the same rows the same way.
#include <math.h>

#include "skv_common.cuh"
#include "skv_internal.h"

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void store4(float* dst, float4 v) { __stcs(reinterpret_cast<float4*>(dst), v); }
__device__ __forceinline__ void store4(__nv_bfloat16* dst, float4 v) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dst) = u;
}

// G lanes per row (G divides 32); each lane owns VPL float4 columns.
template <int G, int VPL, typename OT>
__global__ void __launch_bounds__(kThreads)
lse_merge_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part, int P,
                 int64_t rows, OT* __restrict__ o, float* __restrict__ lse_out) {
    constexpr int D4 = G * VPL;
    const int lane = threadIdx.x & 31;
    const int sub = lane % G;                  // lane inside the row group
    const int grp = lane / G;                  // row group inside the warp
    constexpr int kRowsPerWarp = 32 / G;
    constexpr unsigned kGroupBits = (G >= 32) ? 0xffffffffu : ((1u << (G & 31)) - 1u);
    const unsigned gmask = (G >= 32) ? 0xffffffffu : (kGroupBits << (grp * G));
    const int64_t warp_global = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    for (int64_t r0 = warp_global * kRowsPerWarp; r0 < rows; r0 += n_warps * kRowsPerWarp) {
        const int64_t r = r0 + grp;
        const bool live = r < rows;
        // pass 1: max and sum of exp over the row's partials (lanes stride over p)
        float mx = -INFINITY;
        for (int p = sub; p < P; p += G) {
            const float l = live ? __ldcs(lse_part + int64_t(p) * rows + r) : -INFINITY;
            mx = fmaxf(mx, l);
        }
#pragma unroll
        for (int off = G / 2; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(gmask, mx, off));
        float den = 0.f;
        if (mx != -INFINITY) {
            for (int p = sub; p < P; p += G) {
                const float l = __ldcs(lse_part + int64_t(p) * rows + r);
                den += (l == -INFINITY) ? 0.f : __expf(l - mx);
            }
        }
#pragma unroll
        for (int off = G / 2; off > 0; off >>= 1) den += __shfl_xor_sync(gmask, den, off);
        const float L = (mx == -INFINITY) ? -INFINITY : mx + __logf(den);
        // pass 2: o = sum_p exp(l_p - L) o_p over finite partials
        float4 acc[VPL];
#pragma unroll
        for (int t = 0; t < VPL; ++t) acc[t] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (live && L != -INFINITY) {
            for (int pb = 0; pb < P; pb += G) {
                const int p_me = pb + sub;
                const float l_me = p_me < P ? __ldcs(lse_part + int64_t(p_me) * rows + r) : -INFINITY;
                const float w_me = (l_me == -INFINITY) ? 0.f : __expf(l_me - L);
                unsigned fin = __ballot_sync(gmask, l_me != -INFINITY);
                if (G < 32) fin = (fin >> (grp * G)) & kGroupBits;
                // four partials in flight per lane
                while (fin) {
                    int ps[4];
                    float ws[4];
                    int cnt = 0;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        ps[u] = -1;
                        ws[u] = 0.f;
                        if (fin) {
                            const int b = __ffs(fin) - 1;
                            fin &= fin - 1;
                            ps[u] = pb + b;
                            ws[u] = __shfl_sync(gmask, w_me, grp * G + b);
                            ++cnt;
                        } else {
                            __shfl_sync(gmask, w_me, grp * G);   // keep the group converged
                        }
                    }
                    float4 val[4][VPL];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
#pragma unroll
                        for (int t = 0; t < VPL; ++t) {
                            if (ps[u] >= 0) {
                                const float4* src = reinterpret_cast<const float4*>(
                                    o_part + (int64_t(ps[u]) * rows + r) * (4 * D4));
                                val[u][t] = __ldcs(src + sub + t * G);
                            } else {
                                val[u][t] = make_float4(0.f, 0.f, 0.f, 0.f);
                            }
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u)
#pragma unroll
                        for (int t = 0; t < VPL; ++t) {
                            acc[t].x = fmaf(ws[u], val[u][t].x, acc[t].x);
                            acc[t].y = fmaf(ws[u], val[u][t].y, acc[t].y);
                            acc[t].z = fmaf(ws[u], val[u][t].z, acc[t].z);
                            acc[t].w = fmaf(ws[u], val[u][t].w, acc[t].w);
                        }
                    (void)cnt;
                }
            }
        }
        if (live) {
#pragma unroll
            for (int t = 0; t < VPL; ++t) store4(o + r * (4 * D4) + 4 * (sub + t * G), acc[t]);
            if (lse_out && sub == 0) lse_out[r] = L;
        }
    }
}

__device__ __forceinline__ float4 load4(const float* src) { return __ldcs(reinterpret_cast<const float4*>(src)); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* src) {
    const uint2 u = *reinterpret_cast<const uint2*>(src);
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}

// Backward of the merge per partial [Split-KV §4.1, Eq. 4; MERGE_BWD of
// Alg. 1's backward], for upstream gradients dO (of o) and dlse (of l):
// with w_p = exp(l_p - l) and D_p = dO . o_p,
//   do_part[p] = w_p dO,   dlse_part[p] = w_p (D_p - sum_q w_q D_q + dlse),
// where sum_q w_q D_q = dO . o is taken from the same partials (no rounded o).
// Lanes as in the merge: G lanes own a row; D_p is a group dot product, four
// partials in flight; lane 0 of the group parks D_p in dlse_part until the sum
// over partials is known, then the group's lanes finish their own partials.
template <int G, int VPL, typename GT>
__global__ void __launch_bounds__(kThreads)
lse_merge_bwd_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part, int P, int64_t rows,
                     const GT* __restrict__ dO, const float* __restrict__ dlse, float* __restrict__ do_part,
                     float* __restrict__ dlse_part) {
    constexpr int D4 = G * VPL;
    const int lane = threadIdx.x & 31;
    const int sub = lane % G;
    const int grp = lane / G;
    constexpr int kRowsPerWarp = 32 / G;
    constexpr unsigned kGroupBits = (G >= 32) ? 0xffffffffu : ((1u << (G & 31)) - 1u);
    const unsigned gmask = (G >= 32) ? 0xffffffffu : (kGroupBits << (grp * G));
    const int64_t warp_global = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    for (int64_t r0 = warp_global * kRowsPerWarp; r0 < rows; r0 += n_warps * kRowsPerWarp) {
        const int64_t r = r0 + grp;
        const bool live = r < rows;
        // the merged l, exactly as the forward merge forms it
        float mx = -INFINITY;
        for (int p = sub; p < P; p += G) {
            const float l = live ? __ldcs(lse_part + int64_t(p) * rows + r) : -INFINITY;
            mx = fmaxf(mx, l);
        }
#pragma unroll
        for (int off = G / 2; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(gmask, mx, off));
        float den = 0.f;
        if (mx != -INFINITY) {
            for (int p = sub; p < P; p += G) {
                const float l = __ldcs(lse_part + int64_t(p) * rows + r);
                den += (l == -INFINITY) ? 0.f : __expf(l - mx);
            }
        }
#pragma unroll
        for (int off = G / 2; off > 0; off >>= 1) den += __shfl_xor_sync(gmask, den, off);
        const float L = (mx == -INFINITY) ? -INFINITY : mx + __logf(den);
        const bool any = live && L != -INFINITY;
        float4 g[VPL];
#pragma unroll
        for (int t = 0; t < VPL; ++t) g[t] = any ? load4(dO + r * (4 * D4) + 4 * (sub + t * G)) : make_float4(0.f, 0.f, 0.f, 0.f);
        // D_p for every finite partial, and sum_p w_p D_p
        float dot_o = 0.f;
        if (any) {
            for (int pb = 0; pb < P; pb += G) {
                const int p_me = pb + sub;
                const float l_me = p_me < P ? __ldcs(lse_part + int64_t(p_me) * rows + r) : -INFINITY;
                const float w_me = (l_me == -INFINITY) ? 0.f : __expf(l_me - L);
                unsigned fin = __ballot_sync(gmask, l_me != -INFINITY);
                if (G < 32) fin = (fin >> (grp * G)) & kGroupBits;
                while (fin) {
                    int ps[4];
                    float ws[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        ps[u] = -1;
                        ws[u] = 0.f;
                        if (fin) {
                            const int b = __ffs(fin) - 1;
                            fin &= fin - 1;
                            ps[u] = pb + b;
                            ws[u] = __shfl_sync(gmask, w_me, grp * G + b);
                        } else {
                            __shfl_sync(gmask, w_me, grp * G);   // keep the group converged
                        }
                    }
                    float dot[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        dot[u] = 0.f;
                        if (ps[u] >= 0) {
                            const float4* src = reinterpret_cast<const float4*>(o_part + (int64_t(ps[u]) * rows + r) * (4 * D4));
#pragma unroll
                            for (int t = 0; t < VPL; ++t) {
                                const float4 x = __ldcs(src + sub + t * G);
                                dot[u] = fmaf(g[t].x, x.x, fmaf(g[t].y, x.y, fmaf(g[t].z, x.z, fmaf(g[t].w, x.w, dot[u]))));
                            }
                        }
                    }
#pragma unroll
                    for (int off = G / 2; off > 0; off >>= 1)
#pragma unroll
                        for (int u = 0; u < 4; ++u) dot[u] += __shfl_xor_sync(gmask, dot[u], off);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        dot_o = fmaf(ws[u], dot[u], dot_o);
                        if (sub == 0 && ps[u] >= 0) dlse_part[int64_t(ps[u]) * rows + r] = dot[u];
                    }
                }
            }
        }
        __syncwarp(gmask);
        const float dl = (any && dlse) ? dlse[r] : 0.f;
        if (live) {
            // lane b of the group finishes partial pb + b and hands its w_p to the
            // group for the do_part rows
            for (int pb = 0; pb < P; pb += G) {
                const int p_me = pb + sub;
                float w_me = 0.f;
                if (p_me < P) {
                    const float l = __ldcs(lse_part + int64_t(p_me) * rows + r);
                    const bool f = any && l != -INFINITY;
                    float* dst = dlse_part + int64_t(p_me) * rows + r;
                    w_me = f ? __expf(l - L) : 0.f;
                    *dst = f ? w_me * (*dst - dot_o + dl) : 0.f;
                }
                if (do_part) {
                    const int n = P - pb < G ? P - pb : G;
                    for (int b = 0; b < n; ++b) {
                        const float w = __shfl_sync(gmask, w_me, grp * G + b);
                        float* dst = do_part + (int64_t(pb + b) * rows + r) * (4 * D4);
#pragma unroll
                        for (int t = 0; t < VPL; ++t)
                            store4(dst + 4 * (sub + t * G), make_float4(w * g[t].x, w * g[t].y, w * g[t].z, w * g[t].w));
                    }
                }
            }
        }
    }
}

// CTAs of a grid-stride row kernel: as many as are resident at once on every
// SM (one wave, so no CTA waits for a second one), capped by the warps the rows
// need
template <typename K>
int one_wave(K kernel, int64_t warps_needed, const skv_host::Ctx& c) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    const int64_t need = (warps_needed + kThreads / 32 - 1) / (kThreads / 32);
    const int64_t blocks = int64_t(c.num_sms) * per_sm;
    return (int)(blocks < need ? blocks : (need > 0 ? need : 1));
}

template <typename GT>
skv_status merge_bwd_dispatch(const float* o_part, const float* lse_part, int P, int64_t rows, int d, const GT* dO,
                              const float* dlse, float* do_part, float* dlse_part, const skv_host::Ctx& c) {
#define SKV_MB(G_, V_)                                                                                  \
    {                                                                                                   \
        auto k = lse_merge_bwd_kernel<G_, V_, GT>;                                                      \
        k<<<one_wave(k, (rows + 32 / G_ - 1) / (32 / G_), c), kThreads, 0, c.stream>>>(o_part, lse_part, P, rows, dO, \
                                                                                     dlse, do_part, dlse_part); \
    }
    switch (d) {
        case 64:  SKV_MB(16, 1); break;
        case 128: SKV_MB(32, 1); break;
        case 256: SKV_MB(32, 2); break;
        case 32:  SKV_MB(8, 1); break;
        case 16:  SKV_MB(4, 1); break;
        case 8:   SKV_MB(2, 1); break;
        case 4:   SKV_MB(1, 1); break;
        default: return SKV_ERR_UNSUPPORTED;
    }
#undef SKV_MB
    SKV_LAUNCHED();
    return SKV_OK;
}

template <typename OT>
skv_status merge_dispatch(const float* o_part, const float* lse_part, int P, int64_t rows, int d, OT* o,
                          float* lse, const skv_host::Ctx& c) {
#define SKV_M(G_, V_)                                                                                       \
    {                                                                                                       \
        auto k = lse_merge_kernel<G_, V_, OT>;                                                              \
        k<<<one_wave(k, (rows + 32 / G_ - 1) / (32 / G_), c), kThreads, 0, c.stream>>>(o_part, lse_part, P, rows, o, \
                                                                                     lse);                  \
    }
    switch (d) {
        case 64:  SKV_M(16, 1); break;
        case 128: SKV_M(32, 1); break;
        case 256: SKV_M(32, 2); break;
        case 32:  SKV_M(8, 1); break;
        case 16:  SKV_M(4, 1); break;
        case 8:   SKV_M(2, 1); break;
        case 4:   SKV_M(1, 1); break;
        default: return SKV_ERR_UNSUPPORTED;
    }
#undef SKV_M
    SKV_LAUNCHED();
    return SKV_OK;
}

// D_r = sum_t dO[r,t] * o[r,t] and lse2_r = lse_r * log2(e): one warp per row.
// Input rows are (query q, head h) = q*H + h.  Output index: q*H + h
// (row-major, Qp == Qn), or h*Qp + q (head-major, Qp = Qn rounded up to the
// query tile) with pad rows q >= Qn set to lse2 = +inf, D = 0 so that they
// contribute nothing downstream.
template <typename T>
__global__ void __launch_bounds__(kThreads)
bwd_prep_kernel(const T* __restrict__ o, const T* __restrict__ dO, const float* __restrict__ lse,
                int64_t Qn, int64_t Qp, int H, int d, bool head_major, float* __restrict__ D,
                float* __restrict__ lse2) {
    const int lane = threadIdx.x & 31;
    const int64_t w = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int64_t vrows = Qp * H;
    for (int64_t vr = w; vr < vrows; vr += nw) {
        const int64_t q = vr / H, h = vr - (vr / H) * H;
        const int64_t out = head_major ? h * Qp + q : vr;
        if (q >= Qn) {
            if (lane == 0) {
                D[out] = 0.f;
                lse2[out] = INFINITY;
            }
            continue;
        }
        const int64_t r = q * H + h;
        float acc = 0.f;
        for (int t = lane; t < d; t += 32)
            acc = fmaf(skv::to_f32(o[r * d + t]), skv::to_f32(dO[r * d + t]), acc);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) {
            D[out] = acc;
            lse2[out] = lse[r] * 1.4426950408889634f;
        }
    }
}

__global__ void __launch_bounds__(kThreads)
dq_sum_kernel(const float4* __restrict__ part, int P, int64_t n4, float4* __restrict__ dq) {
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += int64_t(gridDim.x) * blockDim.x) {
        float4 acc = __ldcs(part + i);
        for (int p = 1; p < P; ++p) {
            const float4 v = __ldcs(part + int64_t(p) * n4 + i);
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        __stcs(dq + i, acc);
    }
}

}  // namespace

namespace skv_internal {

skv_status launch_merge(const float* o_part, const float* lse_part, int P, int64_t rows, int d, void* o,
                        skv_dtype o_dtype, float* lse, const skv_host::Ctx& c) {
    if (rows == 0) return SKV_OK;
    skv_host::timer_begin(skv_host::kTimeMerge, c.stream);
    const skv_status st =
        o_dtype == SKV_BF16 ? merge_dispatch(o_part, lse_part, P, rows, d, static_cast<__nv_bfloat16*>(o), lse, c)
                            : merge_dispatch(o_part, lse_part, P, rows, d, static_cast<float*>(o), lse, c);
    skv_host::timer_end(skv_host::kTimeMerge, c.stream);
    return st;
}

skv_status launch_merge_bwd(const float* o_part, const float* lse_part, int P, int64_t rows, int d, const void* dO,
                            skv_dtype do_dtype, const float* dlse, float* do_part, float* dlse_part,
                            const skv_host::Ctx& c) {
    if (rows == 0) return SKV_OK;
    return do_dtype == SKV_BF16
               ? merge_bwd_dispatch(o_part, lse_part, P, rows, d, static_cast<const __nv_bfloat16*>(dO), dlse,
                                    do_part, dlse_part, c)
               : merge_bwd_dispatch(o_part, lse_part, P, rows, d, static_cast<const float*>(dO), dlse, do_part,
                                    dlse_part, c);
}

skv_status launch_bwd_prep(const void* o, const void* dO, const float* lse, skv_dtype dt, int64_t Qn, int64_t Qp,
                           int H, int d, bool head_major, float* D, float* lse2, const skv_host::Ctx& c) {
    const int64_t vrows = Qp * H;
    if (vrows == 0) return SKV_OK;
    int64_t blocks = (vrows + (kThreads / 32) - 1) / (kThreads / 32);
    if (blocks > int64_t(c.num_sms) * 8) blocks = int64_t(c.num_sms) * 8;
    if (dt == SKV_BF16)
        bwd_prep_kernel<<<(unsigned)blocks, kThreads, 0, c.stream>>>(
            static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dO), lse, Qn, Qp, H, d,
            head_major, D, lse2);
    else
        bwd_prep_kernel<<<(unsigned)blocks, kThreads, 0, c.stream>>>(
            static_cast<const float*>(o), static_cast<const float*>(dO), lse, Qn, Qp, H, d, head_major, D, lse2);
    SKV_LAUNCHED();
    return SKV_OK;
}

skv_status launch_dq_sum(const float* dq_part, int P, int64_t rows, int d, float* dq, const skv_host::Ctx& c) {
    const int64_t n4 = rows * d / 4;
    if (n4 == 0) return SKV_OK;
    int64_t blocks = (n4 + kThreads - 1) / kThreads;
    if (blocks > int64_t(c.num_sms) * 8) blocks = int64_t(c.num_sms) * 8;
    dq_sum_kernel<<<(unsigned)blocks, kThreads, 0, c.stream>>>(reinterpret_cast<const float4*>(dq_part), P, n4,
                                                              reinterpret_cast<float4*>(dq));
    SKV_LAUNCHED();
    return SKV_OK;
}

skv_status launch_zero(float* p, int64_t n, const skv_host::Ctx& c) {
    if (n == 0) return SKV_OK;
    SKV_CUDA_CHECK(cudaMemsetAsync(p, 0, size_t(n) * sizeof(float), c.stream));
    return SKV_OK;
}

}  // namespace skv_internal
