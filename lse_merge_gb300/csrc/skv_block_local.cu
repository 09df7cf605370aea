// Block-local term of the anchor mask for libskv (sm_103a, CUDA cores).
//
// [Split-KV §3.1, Fig. 1 caption] Besides its context window, each block's B
// tokens attend bidirectionally to each other.  Those B keys/values are the
// block tokens' own projections (k_blk, v_blk [Q][Hkv][d], rows as in q); they
// form one more key set, disjoint from every context chunk, so the term is one
// more partial (o, l) of Eq. 4 and its gradients use the merged o, l like the
// context ranks do [Alg. 1 line 15 in merged form].
//
// The work is B x B x d per (block, head) -- about 1e-4 of the context term at
// the paper's sizes -- and reads/writes each row once: one 4-warp CTA per
// (block, head) forward and per (block, key/value head) backward, the block's
// rows staged in shared memory (fp32, rows padded to d+1 words so the per-key
// dot products are conflict-free), fp32 arithmetic.
#include <cuda_bf16.h>
#include <math.h>

#include "skv_internal.h"

namespace {

__device__ __forceinline__ float ld(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p, int64_t i) { return __bfloat162float(p[i]); }

constexpr unsigned kAll = 0xffffffffu;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float warp_max(float x) {
    for (int off = 16; off; off >>= 1) x = fmaxf(x, __shfl_xor_sync(kAll, x, off));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
    for (int off = 16; off; off >>= 1) x += __shfl_xor_sync(kAll, x, off);
    return x;
}

constexpr int kWarps = 4;   // warps per (block, head) CTA

// 8 consecutive elements as floats (d is a multiple of 8, rows 16-byte aligned)
__device__ __forceinline__ void ld8(const __nv_bfloat16* p, int64_t i, float (&x)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p + i);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        x[2 * e] = __uint_as_float(w[e] << 16);
        x[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    }
}
__device__ __forceinline__ void ld8(const float* p, int64_t i, float (&x)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p + i), b = *reinterpret_cast<const float4*>(p + i + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
// rows [iB, iB+B) of head h of a [Q][H][d] tensor into shared rows of stride `stride`
template <typename T>
__device__ __forceinline__ void stage_rows(const T* src, int i, int B, int H, int h, int d, float* dst, int stride) {
    const int per_row = d / 8;
    for (int e = threadIdx.x; e < B * per_row; e += blockDim.x) {
        const int r = e / per_row, t = (e - r * per_row) * 8;
        float x[8];
        ld8(src, ((int64_t(i) * B + r) * H + h) * d + t, x);
#pragma unroll
        for (int u = 0; u < 8; ++u) dst[r * stride + t + u] = x[u];
    }
}

// shared floats of one CTA
__host__ __device__ inline int fwd_floats(int B, int d) { return 2 * B * (d + 1) + B * d + B * 32; }
// (the group's dk/dv accumulators, 2 B (d + 1) more, only with grouped queries)
__host__ __device__ inline int bwd_floats(int B, int d, bool grouped) {
    return (grouped ? 6 : 4) * B * (d + 1) + 2 * B * 32 + 32;
}

// One CTA per (block i, head h).  Phase 1: warp w takes rows r = w, w + 4, ...;
// lane j < B scores key j (a d-long dot product), the row's softmax runs across
// the lanes, P goes to shared memory.  Phase 2: the same rows' outputs, lanes
// over the d columns: o_r = sum_j P_rj v_j.
template <typename T>
__global__ void __launch_bounds__(32 * kWarps)
block_local_fwd_kernel(const T* __restrict__ q, const T* __restrict__ kb, const T* __restrict__ vb, int B, int H,
                       int Hkv, int d, float scale_log2, float* __restrict__ o, float* __restrict__ lse) {
    extern __shared__ float sh[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x / H, h = blockIdx.x % H, dp = d + 1;
    const int kvh = h / (H / Hkv);                   // key/value head (grouped-query layouts)
    float* sq = sh;
    float* sk = sq + B * dp;
    float* sv = sk + B * dp;
    float* sp = sv + B * d;   // [B][32] weights of each row
    stage_rows(q, i, B, H, h, d, sq, dp);
    stage_rows(kb, i, B, Hkv, kvh, d, sk, dp);
    stage_rows(vb, i, B, Hkv, kvh, d, sv, d);
    __syncthreads();
    for (int r = warp; r < B; r += kWarps) {
        // key j on lane j (B > 16) or on lanes j and j + 16, each over half of d
        const bool two = B <= 16;
        const int j = two ? (lane & 15) : lane;
        const int t0 = two ? (lane >> 4) * (d / 2) : 0, t1 = two ? t0 + d / 2 : d;
        float acc = 0.f;
        if (j < B)
            for (int t = t0; t < t1; ++t) acc = fmaf(sq[r * dp + t], sk[j * dp + t], acc);
        if (two) acc += __shfl_xor_sync(kAll, acc, 16);
        const float z = (j < B && (!two || lane < 16)) ? acc * scale_log2 : -INFINITY;   // log2 units
        const float mx = warp_max(z);
        const float p = lane < B ? exp2f(z - mx) : 0.f;
        const float sum = warp_sum(p);
        sp[r * 32 + lane] = p / sum;
        const int64_t row = int64_t(i) * B + r;
        if (lane == 0) lse[row * H + h] = (mx + log2f(sum)) * kLn2;
        __syncwarp();
        for (int t = lane; t < d; t += 32) {
            float acc = 0.f;
            for (int j = 0; j < B; ++j) acc = fmaf(sp[r * 32 + j], sv[j * d + t], acc);
            o[(row * H + h) * d + t] = acc;
        }
    }
}

// dq += the block-local part; dk_blk, dv_blk written.  P = exp(z - l) with the
// merged l, D = dO . o with the merged o, dS = P (dP - D).  One CTA per (block,
// key/value head); the query heads of the head's group (one head without
// grouped queries) take turns, their dk, dv contributions summed in shared
// memory.  Per query head: phase 1 (rows over warps, keys over lanes) puts P and
// dS into shared memory; phase 2 (lanes over the d columns) adds the dq rows of
// this warp's rows and the dk/dv parts of this warp's keys.
template <typename T>
__global__ void __launch_bounds__(32 * kWarps)
block_local_bwd_kernel(const T* __restrict__ q, const T* __restrict__ kb, const T* __restrict__ vb,
                       const T* __restrict__ o, const float* __restrict__ lse, const T* __restrict__ dO, int B,
                       int H, int Hkv, int d, float scale, float* __restrict__ dq, float* __restrict__ dkb,
                       float* __restrict__ dvb) {
    extern __shared__ float sh[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x / Hkv, kvh = blockIdx.x % Hkv, dp = d + 1, gq = H / Hkv;
    float* sq = sh;
    float* sk = sq + B * dp;
    float* sv = sk + B * dp;
    float* sg = sv + B * dp;     // dO rows
    float* sp = sg + B * dp;     // [B][32] P
    float* ss = sp + B * 32;     // [B][32] dS
    float* sD = ss + B * 32;     // D per row
    float* sak = sD + 32;        // [B][d + 1] dk_blk rows, summed over the group
    float* sav = sak + B * dp;   // [B][d + 1] dv_blk rows
    stage_rows(kb, i, B, Hkv, kvh, d, sk, dp);
    stage_rows(vb, i, B, Hkv, kvh, d, sv, dp);
    if (gq > 1)
        for (int e = threadIdx.x; e < B * dp; e += blockDim.x) {
            sak[e] = 0.f;
            sav[e] = 0.f;
        }
    const float scale_log2 = scale * kLog2e;
    for (int h = kvh * gq; h < (kvh + 1) * gq; ++h) {
        __syncthreads();   // the previous query head is done with sq, sg, sp, ss
        stage_rows(q, i, B, H, h, d, sq, dp);
        stage_rows(dO, i, B, H, h, d, sg, dp);
        for (int r = warp; r < B; r += kWarps) {   // D_r = dO_r . o_r
            const int64_t g0 = ((int64_t(i) * B + r) * H + h) * d;
            float part = 0.f;
            for (int t = lane; t < d; t += 32) part = fmaf(ld(dO, g0 + t), ld(o, g0 + t), part);
            part = warp_sum(part);
            if (lane == 0) sD[r] = part;
        }
        __syncthreads();
        for (int r = warp; r < B; r += kWarps) {
            const float l = lse[(int64_t(i) * B + r) * H + h];
            // key j on lane j (B > 16) or on lanes j and j + 16, each over half of d
            const bool two = B <= 16;
            const int j = two ? (lane & 15) : lane;
            const int t0 = two ? (lane >> 4) * (d / 2) : 0, t1 = two ? t0 + d / 2 : d;
            float zs = 0.f, dpv = 0.f;
            if (j < B)
                for (int t = t0; t < t1; ++t) {
                    zs = fmaf(sq[r * dp + t], sk[j * dp + t], zs);
                    dpv = fmaf(sg[r * dp + t], sv[j * dp + t], dpv);
                }
            if (two) {
                zs += __shfl_xor_sync(kAll, zs, 16);
                dpv += __shfl_xor_sync(kAll, dpv, 16);
            }
            float P = 0.f, dS = 0.f;
            if (j < B && isfinite(l)) {
                P = exp2f(zs * scale_log2 - l * kLog2e);
                dS = P * (dpv - sD[r]);
            }
            if (!two || lane < 16) {
                sp[r * 32 + j] = P;
                ss[r * 32 + j] = dS;
            }
        }
        __syncthreads();
        for (int r = warp; r < B; r += kWarps) {   // dq rows
            float* dst = dq + ((int64_t(i) * B + r) * H + h) * d;
            for (int t = lane; t < d; t += 32) {
                float acc = 0.f;
                for (int j = 0; j < B; ++j) acc = fmaf(ss[r * 32 + j], sk[j * dp + t], acc);
                dst[t] = fmaf(scale, acc, dst[t]);
            }
        }
        for (int j = warp; j < B; j += kWarps) {   // dk, dv parts of the block keys (thread-owned)
            const int64_t g0 = ((int64_t(i) * B + j) * Hkv + kvh) * d;
            for (int t = lane; t < d; t += 32) {
                float ak = 0.f, av = 0.f;
                for (int r = 0; r < B; ++r) {
                    ak = fmaf(ss[r * 32 + j], sq[r * dp + t], ak);
                    av = fmaf(sp[r * 32 + j], sg[r * dp + t], av);
                }
                if (gq == 1) {                        // one query head: straight out
                    dkb[g0 + t] = scale * ak;
                    dvb[g0 + t] = av;
                } else {
                    sak[j * dp + t] = fmaf(scale, ak, sak[j * dp + t]);
                    sav[j * dp + t] += av;
                }
            }
        }
    }
    if (gq > 1)
        for (int j = warp; j < B; j += kWarps) {   // the same threads wrote these: no barrier
            const int64_t g0 = ((int64_t(i) * B + j) * Hkv + kvh) * d;
            for (int t = lane; t < d; t += 32) {
                dkb[g0 + t] = sak[j * dp + t];
                dvb[g0 + t] = sav[j * dp + t];
            }
        }
}

}  // namespace

namespace skv_internal {

bool block_local_supported(const skv_problem& pb) {
    return pb.B <= 32 && size_t(bwd_floats(pb.B, pb.head_dim, pb.n_kv_heads < pb.n_heads)) * 4 <= 200 * 1024;
}

skv_status launch_block_local_fwd(const skv_problem& pb, const void* q, const void* kb, const void* vb, float* o,
                                  float* lse, const skv_host::Ctx& c) {
    const int N = pb.n_blocks, H = pb.n_heads, Hkv = pb.n_kv_heads, d = pb.head_dim, B = pb.B;
    const int64_t items = int64_t(N) * H;
    if (items == 0) return SKV_OK;
    if (items > 0x7fffffffLL) return SKV_ERR_UNSUPPORTED;
    const int smem = fwd_floats(B, d) * 4;
    const float sl2 = pb.scale * kLog2e;
    skv_host::timer_begin(skv_host::kTimeLocalFwd, c.stream);
    if (pb.dtype == SKV_BF16) {
        using T = __nv_bfloat16;
        auto kern = block_local_fwd_kernel<T>;
        SKV_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
        kern<<<(unsigned)items, 32 * kWarps, smem, c.stream>>>(static_cast<const T*>(q), static_cast<const T*>(kb),
                                                               static_cast<const T*>(vb), B, H, Hkv, d, sl2, o, lse);
    } else {
        auto kern = block_local_fwd_kernel<float>;
        SKV_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
        kern<<<(unsigned)items, 32 * kWarps, smem, c.stream>>>(static_cast<const float*>(q),
                                                               static_cast<const float*>(kb),
                                                               static_cast<const float*>(vb), B, H, Hkv, d, sl2, o,
                                                               lse);
    }
    skv_host::timer_end(skv_host::kTimeLocalFwd, c.stream);
    SKV_LAUNCHED();
    return SKV_OK;
}

skv_status launch_block_local_bwd(const skv_problem& pb, const void* q, const void* kb, const void* vb, const void* o,
                                  const float* lse, const void* dO, float* dq, float* dkb, float* dvb,
                                  const skv_host::Ctx& c) {
    const int N = pb.n_blocks, H = pb.n_heads, Hkv = pb.n_kv_heads, d = pb.head_dim, B = pb.B;
    const int64_t items = int64_t(N) * Hkv;        // (block, key/value head)
    if (items == 0) return SKV_OK;
    if (items > 0x7fffffffLL) return SKV_ERR_UNSUPPORTED;
    const int smem = bwd_floats(B, d, Hkv < H) * 4;
    skv_host::timer_begin(skv_host::kTimeLocalBwd, c.stream);
    if (pb.dtype == SKV_BF16) {
        using T = __nv_bfloat16;
        auto kern = block_local_bwd_kernel<T>;
        SKV_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
        kern<<<(unsigned)items, 32 * kWarps, smem, c.stream>>>(
            static_cast<const T*>(q), static_cast<const T*>(kb), static_cast<const T*>(vb), static_cast<const T*>(o),
            lse, static_cast<const T*>(dO), B, H, Hkv, d, pb.scale, dq, dkb, dvb);
    } else {
        using T = float;
        auto kern = block_local_bwd_kernel<T>;
        SKV_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
        kern<<<(unsigned)items, 32 * kWarps, smem, c.stream>>>(
            static_cast<const T*>(q), static_cast<const T*>(kb), static_cast<const T*>(vb), static_cast<const T*>(o),
            lse, static_cast<const T*>(dO), B, H, Hkv, d, pb.scale, dq, dkb, dvb);
    }
    skv_host::timer_end(skv_host::kTimeLocalBwd, c.stream);
    SKV_LAUNCHED();
    return SKV_OK;
}

}  // namespace skv_internal
