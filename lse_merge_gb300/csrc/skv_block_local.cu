// Block-local term of the anchor mask for libskv (sm_103a, CUDA cores): fp32
// inputs and blocks of more than 16 rows (bf16 blocks of up to 16 rows take the
// warp-MMA kernels of skv_block_local_mma.cu).
//
// [Split-KV §3.1, Fig. 1 caption] Besides its context window, each block's B
// tokens attend bidirectionally to each other.  Those B keys/values are the
// block tokens' own projections (k_blk, v_blk [Q][Hkv][d], rows as in q); they
// form one more key set, disjoint from every context chunk, so the term is one
// more partial (o, l) of Eq. 4 and its gradients use the merged o, l like the
// context ranks do [Alg. 1's MERGE_BWD in merged form].
//
// The work is B x B x d per (block, head) -- about 1e-4 of the context term at
// the paper's sizes -- and reads/writes each row once: one 4-warp CTA per
// (block, head) forward and per (block, key/value head) backward, the block's
// rows staged in shared memory as fp32 (rows padded to d + 4 words; every
// global load of a stage in flight at once), the products register-tiled (a
// lane holds a slice of one key and streams the warp's rows past it; outputs in
// float4 columns), fp32 arithmetic.
#include <cuda_bf16.h>
#include <math.h>

#include "skv_internal.h"

namespace {

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

constexpr int kWarps = 4;        // warps per CTA
constexpr int kThreads = 32 * kWarps;

// 8 consecutive elements of a row, held as loaded (rows 16-byte aligned, d a
// multiple of 8)
template <typename T>
struct Chunk8;
template <>
struct Chunk8<__nv_bfloat16> {
    uint4 u;
    __device__ __forceinline__ void load(const __nv_bfloat16* p, int64_t i) {
        u = *reinterpret_cast<const uint4*>(p + i);
    }
    __device__ __forceinline__ void get(float (&x)[8]) const {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            x[2 * e] = __uint_as_float(w[e] << 16);
            x[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
        }
    }
};
template <>
struct Chunk8<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const float* p, int64_t i) {
        a = *reinterpret_cast<const float4*>(p + i);
        b = *reinterpret_cast<const float4*>(p + i + 4);
    }
    __device__ __forceinline__ void get(float (&x)[8]) const {
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
};

// This thread's share of rows [iB, iB + B) of head h of a [Q][Hx][D] tensor:
// chunk e = threadIdx.x + n * kThreads is row e / (D/8), columns 8 (e % (D/8)) + [0, 8).
// load() issues every global load; store() writes them as fp32 shared rows of
// stride D + 4.  The kernels take NCH = R D / 256, enough chunks for the B <= 4 R
// rows of a CTA.
template <typename T, int D, int NCH>
struct Rows {
    static constexpr int PR = D / 8;   // chunks per row
    Chunk8<T> c[NCH];
    __device__ __forceinline__ void load(const T* __restrict__ src, int i, int B, int Hx, int h) {
#pragma unroll
        for (int n = 0; n < NCH; ++n) {
            const int e = threadIdx.x + n * kThreads;
            if (e < B * PR) c[n].load(src, ((int64_t(i) * B + e / PR) * Hx + h) * D + (e % PR) * 8);
        }
    }
    __device__ __forceinline__ void store(float* dst, int B) const {
#pragma unroll
        for (int n = 0; n < NCH; ++n) {
            const int e = threadIdx.x + n * kThreads;
            if (e < B * PR) {
                float x[8];
                c[n].get(x);
                float4* out = reinterpret_cast<float4*>(dst + (e / PR) * (D + 4) + (e % PR) * 8);
                out[0] = make_float4(x[0], x[1], x[2], x[3]);
                out[1] = make_float4(x[4], x[5], x[6], x[7]);
            }
        }
    }
};

// D_r = dO_r . o_r from this thread's chunks of both, summed over the row's
// D/8 lanes (a row's chunks sit on consecutive lanes of one warp)
template <typename T, int D, int NCH>
__device__ __forceinline__ void rows_dot(const Rows<T, D, NCH>& a, const Rows<T, D, NCH>& b, int B, float* sD) {
    constexpr int PR = D / 8;
#pragma unroll
    for (int n = 0; n < NCH; ++n) {
        const int e = threadIdx.x + n * kThreads;
        float part = 0.f;
        if (e < B * PR) {
            float x[8], y[8];
            a.c[n].get(x);
            b.c[n].get(y);
#pragma unroll
            for (int u = 0; u < 8; ++u) part = fmaf(x[u], y[u], part);
        }
#pragma unroll
        for (int off = PR / 2; off; off >>= 1) part += __shfl_xor_sync(kAll, part, off);
        if (e < B * PR && e % PR == 0) sD[e / PR] = part;
    }
}

// shared floats of one CTA: q, k, v rows and the row weights (forward); q, k, v,
// dO rows, P, dS and D (backward)
__host__ __device__ inline int fwd_floats(int B, int d) { return 3 * B * (d + 4) + B * 32; }
__host__ __device__ inline int bwd_floats(int B, int d) { return 4 * B * (d + 4) + 2 * B * 32 + 32; }

// Dot products of this warp's rows r = w, w + 4, ... (R of them at most) with
// key j, register-tiled: the lane keeps KC = 16 / NP of key j's columns per
// pair in registers while the rows stream past as shared broadcasts.  R = 8
// (B <= 32): key j is lane j.  R = 4 (B <= 16): key j is lanes j and j + 16,
// each over half of the columns.  NP operand pairs: (q, k), and (dO, v) too in
// the backward.
template <int D, int R, int NP>
__device__ __forceinline__ void row_key_dots(const float* __restrict__ rows0, const float* __restrict__ keys0,
                                             const float* __restrict__ rows1, const float* __restrict__ keys1, int B,
                                             int warp, int lane, float (&acc)[NP][R]) {
    constexpr int LD = D + 4;
    constexpr bool kTwo = R == 4;
    const int j = kTwo ? (lane & 15) : lane;
    const int c0 = kTwo ? (lane >> 4) * (D / 2) : 0;
    constexpr int NCOL = kTwo ? D / 2 : D;
    const float* rows[2] = {rows0, rows1};
    const float* keys[2] = {keys0, keys1};
#pragma unroll
    for (int pp = 0; pp < NP; ++pp)
#pragma unroll
        for (int rr = 0; rr < R; ++rr) acc[pp][rr] = 0.f;
    constexpr int KC = 16 / NP, KU = KC / 4;
    if (j < B) {
#pragma unroll 1
        for (int t0 = c0; t0 < c0 + NCOL; t0 += KC) {
            float4 kr[NP][KU];
#pragma unroll
            for (int pp = 0; pp < NP; ++pp)
#pragma unroll
                for (int u = 0; u < KU; ++u) kr[pp][u] = *reinterpret_cast<const float4*>(keys[pp] + j * LD + t0 + 4 * u);
#pragma unroll
            for (int rr = 0; rr < R; ++rr) {
                const int r = warp + rr * kWarps;
                if (r < B) {
#pragma unroll
                    for (int pp = 0; pp < NP; ++pp)
#pragma unroll
                        for (int u = 0; u < KU; ++u) {
                            const float4 x = *reinterpret_cast<const float4*>(rows[pp] + r * LD + t0 + 4 * u);
                            acc[pp][rr] = fmaf(x.x, kr[pp][u].x,
                                               fmaf(x.y, kr[pp][u].y,
                                                    fmaf(x.z, kr[pp][u].z, fmaf(x.w, kr[pp][u].w, acc[pp][rr]))));
                        }
                }
            }
        }
    }
    if (kTwo)
#pragma unroll
        for (int pp = 0; pp < NP; ++pp)
#pragma unroll
            for (int rr = 0; rr < R; ++rr) acc[pp][rr] += __shfl_xor_sync(kAll, acc[pp][rr], 16);
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ float4 fma4(float a, float4 x, float4 y) {
    return make_float4(fmaf(a, x.x, y.x), fmaf(a, x.y, y.y), fmaf(a, x.z, y.z), fmaf(a, x.w, y.w));
}

// One CTA per (block i, head h).  Phase 1: the scores of warp w's rows
// r = w, w + 4, ... (row_key_dots), each row's softmax across the lanes, P to
// shared memory.  Phase 2: o_r = sum_j P_rj v_j for the same rows, lanes over
// float4 columns (d = 64: two rows per pass).
template <typename T, int D, int R>
__global__ void __launch_bounds__(kThreads)
block_local_fwd_kernel(const T* __restrict__ q, const T* __restrict__ kb, const T* __restrict__ vb, int B, int H,
                       int Hkv, float scale_log2, float* __restrict__ o, float* __restrict__ lse) {
    constexpr int LD = D + 4, NC = D / 4, SLOTS = 32 / NC, KO = R / SLOTS, NCH = R * D / 256;
    extern __shared__ float sh[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x / H, h = blockIdx.x % H;
    const int kvh = h / (H / Hkv);                   // key/value head (grouped-query layouts)
    float* sq = sh;
    float* sk = sq + B * LD;
    float* sv = sk + B * LD;
    float* sp = sv + B * LD;   // [B][32] weights of each row
    {
        Rows<T, D, NCH> a, b, c;
        a.load(q, i, B, H, h);
        b.load(kb, i, B, Hkv, kvh);
        c.load(vb, i, B, Hkv, kvh);
        a.store(sq, B);
        b.store(sk, B);
        c.store(sv, B);
    }
    __syncthreads();
    float acc[1][R];
    row_key_dots<D, R, 1>(sq, sk, nullptr, nullptr, B, warp, lane, acc);
    constexpr bool kTwo = R == 4;
    const int j = kTwo ? (lane & 15) : lane;
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        const int r = warp + rr * kWarps;
        if (r >= B) break;
        const float z = (j < B && (!kTwo || lane < 16)) ? acc[0][rr] * scale_log2 : -INFINITY;   // log2 units
        const float mx = warp_max(z);
        const float p = lane < B ? exp2f(z - mx) : 0.f;
        const float sum = warp_sum(p);
        sp[r * 32 + lane] = p / sum;
        if (lane == 0) lse[(int64_t(i) * B + r) * H + h] = (mx + log2f(sum)) * kLn2;
    }
    __syncwarp();   // a warp reads back only its own rows' weights
    const int col = lane % NC, slot = lane / NC;
    float4 ao[KO];
#pragma unroll
    for (int k = 0; k < KO; ++k) ao[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int jj = 0; jj < B; ++jj) {
        const float4 v4 = *reinterpret_cast<const float4*>(sv + jj * LD + 4 * col);
#pragma unroll
        for (int k = 0; k < KO; ++k) {
            const int r = warp + (slot + SLOTS * k) * kWarps;
            if (r < B) ao[k] = fma4(sp[r * 32 + jj], v4, ao[k]);
        }
    }
#pragma unroll
    for (int k = 0; k < KO; ++k) {
        const int r = warp + (slot + SLOTS * k) * kWarps;
        if (r < B) *reinterpret_cast<float4*>(o + ((int64_t(i) * B + r) * H + h) * D + 4 * col) = ao[k];
    }
}

// dq += the block-local part; dk_blk, dv_blk written.  P = exp(z - l) with the
// merged l, D = dO . o with the merged o, dS = P (dP - D).  One CTA per (block,
// key/value head); the query heads of the head's group (one head without
// grouped queries) take turns.  Per query head: one batch of global loads (q,
// dO, o rows and the rows' l; the dq values to add to are prefetched to L2),
// then phase 1 (row_key_dots for q . k and dO . v) puts P and dS into shared
// memory; phase 2 (lanes over float4 columns) adds the dq rows of warp w's
// rows, and each thread adds to the dk/dv columns it owns for warp w's keys
// j = w, w + 4, ..., kept in registers over the whole group.
template <typename T, int D, int R>
__global__ void __launch_bounds__(kThreads, R == 4 ? 4 : 2)   // B <= 16: four CTAs an SM (128 registers)
block_local_bwd_kernel(const T* __restrict__ q, const T* __restrict__ kb, const T* __restrict__ vb,
                       const T* __restrict__ o, const float* __restrict__ lse, const T* __restrict__ dO, int B,
                       int H, int Hkv, float scale, float* __restrict__ dq, float* __restrict__ dkb,
                       float* __restrict__ dvb) {
    constexpr int LD = D + 4, NC = D / 4, SLOTS = 32 / NC, KR = R / SLOTS, NCH = R * D / 256;
    extern __shared__ float sh[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x / Hkv, kvh = blockIdx.x % Hkv, gq = H / Hkv;
    float* sq = sh;
    float* sk = sq + B * LD;
    float* sv = sk + B * LD;
    float* sg = sv + B * LD;     // dO rows
    float* sp = sg + B * LD;     // [B][32] P
    float* ss = sp + B * 32;     // [B][32] dS
    float* sD = ss + B * 32;     // D per row
    {
        Rows<T, D, NCH> a, b;
        a.load(kb, i, B, Hkv, kvh);
        b.load(vb, i, B, Hkv, kvh);
        a.store(sk, B);
        b.store(sv, B);
    }
    const float scale_log2 = scale * kLog2e;
    constexpr bool kTwo = R == 4;
    const int j = kTwo ? (lane & 15) : lane;
    const int col = lane % NC, slot = lane / NC;
    float4 akk[KR], avv[KR];     // dk, dv columns [4 col, 4 col + 4) of keys w + 4 (slot + SLOTS k)
#pragma unroll
    for (int k = 0; k < KR; ++k) {
        akk[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        avv[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int h = kvh * gq; h < (kvh + 1) * gq; ++h) {
        __syncthreads();   // the previous query head is done with sq, sg, sp, ss, sD
        float lrow[R];
        {
            Rows<T, D, NCH> a, g, oo;
            a.load(q, i, B, H, h);
            g.load(dO, i, B, H, h);
            oo.load(o, i, B, H, h);
#pragma unroll
            for (int rr = 0; rr < R; ++rr) {
                const int r = warp + rr * kWarps;
                lrow[rr] = r < B ? lse[(int64_t(i) * B + r) * H + h] : 0.f;
            }
#pragma unroll
            for (int k = 0; k < KR; ++k) {   // the dq values this thread adds to, on their way to L2
                const int r = warp + (slot + SLOTS * k) * kWarps;
                if (r < B) prefetch_l2(dq + ((int64_t(i) * B + r) * H + h) * D + 4 * col);
            }
            a.store(sq, B);
            g.store(sg, B);
            rows_dot(g, oo, B, sD);
        }
        __syncthreads();
        float acc[2][R];
        row_key_dots<D, R, 2>(sq, sk, sg, sv, B, warp, lane, acc);
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            const int r = warp + rr * kWarps;
            if (r >= B) break;
            const float l = lrow[rr];
            float P = 0.f, dS = 0.f;
            if (j < B && isfinite(l)) {
                P = exp2f(acc[0][rr] * scale_log2 - l * kLog2e);
                dS = P * (acc[1][rr] - sD[r]);
            }
            if (!kTwo || lane < 16) {
                sp[r * 32 + j] = P;
                ss[r * 32 + j] = dS;
            }
        }
        __syncthreads();   // every row's P, dS before the key-side sums
#pragma unroll
        for (int k = 0; k < KR; ++k) {              // dq rows of this warp's rows
            const int r = warp + (slot + SLOTS * k) * kWarps;
            if (r >= B) continue;
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int jj = 0; jj < B; ++jj)
                a = fma4(ss[r * 32 + jj], *reinterpret_cast<const float4*>(sk + jj * LD + 4 * col), a);
            float4* dst = reinterpret_cast<float4*>(dq + ((int64_t(i) * B + r) * H + h) * D + 4 * col);
            *dst = fma4(scale, a, *dst);
        }
        for (int r = 0; r < B; ++r) {               // dk, dv parts of this thread's keys
            const float4 q4 = *reinterpret_cast<const float4*>(sq + r * LD + 4 * col);
            const float4 g4 = *reinterpret_cast<const float4*>(sg + r * LD + 4 * col);
#pragma unroll
            for (int k = 0; k < KR; ++k) {
                const int jk = warp + (slot + SLOTS * k) * kWarps;
                if (jk < B) {
                    akk[k] = fma4(ss[r * 32 + jk], q4, akk[k]);
                    avv[k] = fma4(sp[r * 32 + jk], g4, avv[k]);
                }
            }
        }
    }
#pragma unroll
    for (int k = 0; k < KR; ++k) {
        const int jk = warp + (slot + SLOTS * k) * kWarps;
        if (jk >= B) continue;
        const int64_t g0 = ((int64_t(i) * B + jk) * Hkv + kvh) * D + 4 * col;
        *reinterpret_cast<float4*>(dkb + g0) = make_float4(scale * akk[k].x, scale * akk[k].y, scale * akk[k].z,
                                                           scale * akk[k].w);
        *reinterpret_cast<float4*>(dvb + g0) = avv[k];
    }
}

}  // namespace

namespace skv_internal {

bool block_local_supported(const skv_problem& pb) {
    return pb.B <= 32 && (pb.head_dim == 64 || pb.head_dim == 128) &&
           size_t(bwd_floats(pb.B, pb.head_dim)) * 4 <= 200 * 1024;
}

namespace {

template <typename T, int D, int R>
skv_status fwd_launch(const skv_problem& pb, const void* q, const void* kb, const void* vb, float* o, float* lse,
                      unsigned items, const skv_host::Ctx& c) {
    const int smem = fwd_floats(pb.B, D) * 4;
    auto kern = block_local_fwd_kernel<T, D, R>;
    SKV_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    kern<<<items, kThreads, smem, c.stream>>>(static_cast<const T*>(q), static_cast<const T*>(kb),
                                              static_cast<const T*>(vb), pb.B, pb.n_heads, pb.n_kv_heads,
                                              pb.scale * kLog2e, o, lse);
    return SKV_OK;
}

template <typename T, int D, int R>
skv_status bwd_launch(const skv_problem& pb, const void* q, const void* kb, const void* vb, const void* o,
                      const float* lse, const void* dO, float* dq, float* dkb, float* dvb, unsigned items,
                      const skv_host::Ctx& c) {
    const int smem = bwd_floats(pb.B, D) * 4;
    auto kern = block_local_bwd_kernel<T, D, R>;
    SKV_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    kern<<<items, kThreads, smem, c.stream>>>(static_cast<const T*>(q), static_cast<const T*>(kb),
                                              static_cast<const T*>(vb), static_cast<const T*>(o), lse,
                                              static_cast<const T*>(dO), pb.B, pb.n_heads, pb.n_kv_heads,
                                              pb.scale, dq, dkb, dvb);
    return SKV_OK;
}

// R = rows per warp at most: 4 for B <= 16 (two lanes per key), else 8
template <typename T, int D>
skv_status fwd_rows(const skv_problem& pb, const void* q, const void* kb, const void* vb, float* o, float* lse,
                    unsigned items, const skv_host::Ctx& c) {
    return pb.B <= 16 ? fwd_launch<T, D, 4>(pb, q, kb, vb, o, lse, items, c)
                      : fwd_launch<T, D, 8>(pb, q, kb, vb, o, lse, items, c);
}

template <typename T, int D>
skv_status bwd_rows(const skv_problem& pb, const void* q, const void* kb, const void* vb, const void* o,
                    const float* lse, const void* dO, float* dq, float* dkb, float* dvb, unsigned items,
                    const skv_host::Ctx& c) {
    return pb.B <= 16 ? bwd_launch<T, D, 4>(pb, q, kb, vb, o, lse, dO, dq, dkb, dvb, items, c)
                      : bwd_launch<T, D, 8>(pb, q, kb, vb, o, lse, dO, dq, dkb, dvb, items, c);
}

}  // namespace

skv_status launch_block_local_fwd(const skv_problem& pb, const void* q, const void* kb, const void* vb, float* o,
                                  float* lse, const skv_host::Ctx& c) {
    const int64_t items = int64_t(pb.n_blocks) * pb.n_heads;
    if (items == 0) return SKV_OK;
    if (items > 0x7fffffffLL) return SKV_ERR_UNSUPPORTED;
    skv_host::timer_begin(skv_host::kTimeLocalFwd, c.stream);
    const bool bf = pb.dtype == SKV_BF16;
    const skv_status st =
        block_local_mma_supported(pb) ? launch_block_local_fwd_mma(pb, q, kb, vb, o, lse, c) :
        pb.head_dim == 128
            ? (bf ? fwd_rows<__nv_bfloat16, 128>(pb, q, kb, vb, o, lse, (unsigned)items, c)
                  : fwd_rows<float, 128>(pb, q, kb, vb, o, lse, (unsigned)items, c))
            : (bf ? fwd_rows<__nv_bfloat16, 64>(pb, q, kb, vb, o, lse, (unsigned)items, c)
                  : fwd_rows<float, 64>(pb, q, kb, vb, o, lse, (unsigned)items, c));
    skv_host::timer_end(skv_host::kTimeLocalFwd, c.stream);
    if (st != SKV_OK) return st;
    SKV_LAUNCHED();
    return SKV_OK;
}

skv_status launch_block_local_bwd(const skv_problem& pb, const void* q, const void* kb, const void* vb, const void* o,
                                  const float* lse, const void* dO, float* dq, float* dkb, float* dvb,
                                  const skv_host::Ctx& c) {
    const int64_t items = int64_t(pb.n_blocks) * pb.n_kv_heads;   // (block, key/value head)
    if (items == 0) return SKV_OK;
    if (items > 0x7fffffffLL) return SKV_ERR_UNSUPPORTED;
    skv_host::timer_begin(skv_host::kTimeLocalBwd, c.stream);
    const bool bf = pb.dtype == SKV_BF16;
    const unsigned n = (unsigned)items;
    const skv_status st =
        block_local_mma_supported(pb) ? launch_block_local_bwd_mma(pb, q, kb, vb, o, lse, dO, dq, dkb, dvb, c) :
        pb.head_dim == 128
            ? (bf ? bwd_rows<__nv_bfloat16, 128>(pb, q, kb, vb, o, lse, dO, dq, dkb, dvb, n, c)
                  : bwd_rows<float, 128>(pb, q, kb, vb, o, lse, dO, dq, dkb, dvb, n, c))
            : (bf ? bwd_rows<__nv_bfloat16, 64>(pb, q, kb, vb, o, lse, dO, dq, dkb, dvb, n, c)
                  : bwd_rows<float, 64>(pb, q, kb, vb, o, lse, dO, dq, dkb, dvb, n, c));
    skv_host::timer_end(skv_host::kTimeLocalBwd, c.stream);
    if (st != SKV_OK) return st;
    SKV_LAUNCHED();
    return SKV_OK;
}

}  // namespace skv_internal
