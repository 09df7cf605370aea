// Block-local term of the anchor mask on the tensor cores, warp-level MMA
// (libskv, sm_103a): bf16 inputs, B <= 16 rows per block, head_dim 64 or 128.
//
// [Split-KV §3.1, Fig. 1 caption] each block's B tokens also attend
// bidirectionally to the block's own B keys/values (k_blk, v_blk, rows as in q);
// the term is one more partial (o, l) of Eq. 4, and its gradients use the
// merged (o, l) of the whole mask [Alg. 1's MERGE_BWD in merged form].
//
// One warp owns one (block, head) in the forward and one (block, key/value
// head) in the backward: the block's rows are exactly one 16-row tile of the
// m16n8k16 MMA, so the scores, P V and every gradient product are a handful of
// warp MMAs with the softmax in registers; a 64- or 128-row tcgen05 tile would
// spend most of its work on the masked-out pairs of neighbouring blocks.  The
// term reads and writes each row once, so it is bound by HBM: rows are staged
// with 16-byte asynchronous copies (all of a warp's copies in flight at once)
// into padded shared rows that ldmatrix reads without bank conflicts.
#include <cuda_bf16.h>
#include <math.h>

#include "skv_internal.h"

namespace {

constexpr unsigned kAll = 0xffffffffu;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kWarpsFwd = 4, kWarpsBwd = 2;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_addr(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_addr(p)));
}

// c += a (16x16, row-major fragment) * b (16x8, column fragment); bf16 in, fp32 accumulate
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Rows [iB, iB + B) of head h of a [Q][Hx][D] bf16 tensor into 16 shared rows
// of LD elements (rows past B zero-filled), issued as 16-byte asynchronous copies.
template <int D>
__device__ __forceinline__ void stage_rows(__nv_bfloat16* dst, const __nv_bfloat16* __restrict__ src, int64_t row0,
                                           int B, int Hx, int h, int lane) {
    constexpr int LD = D + 8, PR = D / 8;
#pragma unroll
    for (int e = lane; e < 16 * PR; e += 32) {
        const int r = e / PR, c = (e % PR) * 8;
        __nv_bfloat16* d = dst + r * LD + c;
        if (r < B)
            cp_async16(d, src + ((row0 + r) * Hx + h) * D + c);
        else
            *reinterpret_cast<uint4*>(d) = make_uint4(0u, 0u, 0u, 0u);
    }
}

// S = A B^T over D columns for a 16-row tile of A and 16 rows of B (both row-major
// shared, stride LD): s[nt][] is the accumulator of key columns [8nt, 8nt + 8).
template <int D>
__device__ __forceinline__ void scores16(float (&s)[2][4], const __nv_bfloat16* a, const __nv_bfloat16* b, int lane) {
    constexpr int LD = D + 8;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int u = 0; u < 4; ++u) s[nt][u] = 0.f;
    const int ar = lane & 15, ac = (lane >> 4) * 8;                 // A: matrices (r0-7,c0), (r8-15,c0), (r0-7,c8), (r8-15,c8)
    const int br = (lane & 7) + ((lane >> 4) << 3), bc = ((lane >> 3) & 1) * 8;   // B: (k0-7,c0), (k0-7,c8), (k8-15,c0), (k8-15,c8)
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t fa[4], fb[4];
        ldsm_x4(fa, a + ar * LD + kk * 16 + ac);
        ldsm_x4(fb, b + br * LD + kk * 16 + bc);
        mma16816(s[0], fa, fb[0], fb[1]);
        mma16816(s[1], fa, fb[2], fb[3]);
    }
}

// acc[nt][] += P (16 x 16, as an A fragment) times columns [C0, C0 + 8 NT) of the
// 16 x D row-major shared matrix V (keys as K): output columns C0 + [8nt, 8nt + 8).
template <int D, int NT, int C0 = 0>
__device__ __forceinline__ void times_rows(float (&acc)[NT][4], const uint32_t (&pa)[4], const __nv_bfloat16* v,
                                           int lane) {
    constexpr int LD = D + 8;
    const int vr = (lane & 7) + ((lane >> 3) & 1) * 8, vc = (lane >> 4) * 8;   // (k0-7,n), (k8-15,n), (k0-7,n+8), (k8-15,n+8)
#pragma unroll
    for (int nt = 0; nt < NT; nt += 2) {
        uint32_t fb[4];
        ldsm_x4_t(fb, v + vr * LD + C0 + nt * 8 + vc);
        mma16816(acc[nt], pa, fb[0], fb[1]);
        mma16816(acc[nt + 1], pa, fb[2], fb[3]);
    }
}

// The accumulator fragments of a 16 x 16 product as the A fragment of the next MMA.
__device__ __forceinline__ void as_a(uint32_t (&a)[4], const float (&s)[2][4]) {
    a[0] = pack2(s[0][0], s[0][1]);
    a[1] = pack2(s[0][2], s[0][3]);
    a[2] = pack2(s[1][0], s[1][1]);
    a[3] = pack2(s[1][2], s[1][3]);
}

template <int D>
__global__ void __launch_bounds__(32 * kWarpsFwd)
block_local_fwd_mma_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kb,
                           const __nv_bfloat16* __restrict__ vb, int B, int H, int Hkv, int64_t items,
                           float scale_log2, float* __restrict__ o, float* __restrict__ lse) {
    constexpr int LD = D + 8;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t item = int64_t(blockIdx.x) * kWarpsFwd + warp;     // (block, head), head fastest
    if (item >= items) return;
    const int64_t i = item / H;
    const int h = int(item % H), kvh = h / (H / Hkv);
    __nv_bfloat16* sq = reinterpret_cast<__nv_bfloat16*>(smem_raw) + warp * 3 * 16 * LD;
    __nv_bfloat16* sk = sq + 16 * LD;
    __nv_bfloat16* sv = sk + 16 * LD;
    const int64_t row0 = i * B;
    stage_rows<D>(sq, q, row0, B, H, h, lane);
    stage_rows<D>(sk, kb, row0, B, Hkv, kvh, lane);
    stage_rows<D>(sv, vb, row0, B, Hkv, kvh, lane);
    cp_async_wait_all();
    __syncwarp();
    float s[2][4];
    scores16<D>(s, sq, sk, lane);
    // rows g and g + 8; key columns 8nt + 2c + {0, 1}
    const int g = lane >> 2, c = lane & 3;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int j = nt * 8 + 2 * c + (u & 1);
            s[nt][u] = j < B ? s[nt][u] * scale_log2 : -INFINITY;
            mx[u >> 1] = fmaxf(mx[u >> 1], s[nt][u]);
        }
    float sum[2] = {0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        mx[e] = fmaxf(mx[e], __shfl_xor_sync(kAll, mx[e], 1));
        mx[e] = fmaxf(mx[e], __shfl_xor_sync(kAll, mx[e], 2));
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            s[nt][u] = exp2f(s[nt][u] - mx[u >> 1]);
            sum[u >> 1] += s[nt][u];
        }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        sum[e] += __shfl_xor_sync(kAll, sum[e], 1);
        sum[e] += __shfl_xor_sync(kAll, sum[e], 2);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int u = 0; u < 4; ++u) s[nt][u] /= sum[u >> 1];
    uint32_t pa[4];
    as_a(pa, s);
    float acc[D / 8][4];
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
        for (int u = 0; u < 4; ++u) acc[nt][u] = 0.f;
    times_rows<D, D / 8>(acc, pa, sv, lane);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int r = g + 8 * e;
        if (r < B) {
            float* dst = o + ((row0 + r) * H + h) * D + 2 * c;
#pragma unroll
            for (int nt = 0; nt < D / 8; ++nt)
                *reinterpret_cast<float2*>(dst + nt * 8) = make_float2(acc[nt][2 * e], acc[nt][2 * e + 1]);
            if (c == 0) lse[(row0 + r) * H + h] = (mx[e] + log2f(sum[e])) * kLn2;
        }
    }
}

// dq rows g, g + 8 of head h, columns [C0, C0 + D/2): += scale dS K, the values added
// to read from their staged copy sdq (fp32 rows of D + 4)
template <int D, int C0>
__device__ __forceinline__ void dq_add(float* __restrict__ dq, const float* sdq, const uint32_t (&da)[4],
                                       const __nv_bfloat16* sk, int64_t row0, int B, int H, int h, float scale,
                                       int lane) {
    constexpr int NT = D / 16;
    const int g = lane >> 2, c = lane & 3;
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int u = 0; u < 4; ++u) acc[nt][u] = 0.f;
    times_rows<D, NT, C0>(acc, da, sk, lane);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int r = g + 8 * e;
        if (r < B) {
            float* dst = dq + ((row0 + r) * H + h) * D + C0 + 2 * c;
            const float* src = sdq + r * (D + 4) + C0 + 2 * c;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float2 old = *reinterpret_cast<const float2*>(src + nt * 8);
                *reinterpret_cast<float2*>(dst + nt * 8) =
                    make_float2(fmaf(scale, acc[nt][2 * e], old.x), fmaf(scale, acc[nt][2 * e + 1], old.y));
            }
        }
    }
}

// shared bytes of one backward warp: five bf16 row tiles (16 x (D + 8)), P and dS
// (16 x 24 bf16 each), the fp32 dq rows (16 x (D + 4)); a multiple of 16
template <int D>
constexpr int bwd_warp_bytes() {
    return (5 * 16 * (D + 8) + 2 * 16 * 24) * 2 + 16 * (D + 4) * 4;
}

// dq += the block-local part; dk_blk, dv_blk written.  One warp per (block,
// key/value head); the query heads of its group take turns, dK and dV stay in
// registers over the group.  P = exp(z - l) with the merged l, D = dO . o with
// the merged o, dS = P (dP - D).
template <int D>
__global__ void __launch_bounds__(32 * kWarpsBwd)
block_local_bwd_mma_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kb,
                           const __nv_bfloat16* __restrict__ vb, const __nv_bfloat16* __restrict__ o,
                           const float* __restrict__ lse, const __nv_bfloat16* __restrict__ dO, int B, int H,
                           int Hkv, int64_t items, float scale, float* __restrict__ dq, float* __restrict__ dkb,
                           float* __restrict__ dvb) {
    constexpr int LD = D + 8;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t item = int64_t(blockIdx.x) * kWarpsBwd + warp;     // (block, key/value head)
    if (item >= items) return;
    const int64_t i = item / Hkv;
    const int kvh = int(item % Hkv), gq = H / Hkv;
    // per warp: k, v, q, dO, o rows, the bf16 16 x 16 P and dS tiles, then the fp32 dq
    // rows the block-local part is added to
    __nv_bfloat16* sk = reinterpret_cast<__nv_bfloat16*>(smem_raw + warp * bwd_warp_bytes<D>());
    __nv_bfloat16* sv = sk + 16 * LD;
    __nv_bfloat16* sq = sv + 16 * LD;
    __nv_bfloat16* sg = sq + 16 * LD;
    __nv_bfloat16* so = sg + 16 * LD;
    __nv_bfloat16* sp = so + 16 * LD;        // P, row-major [16][24]
    __nv_bfloat16* ss = sp + 16 * 24;        // dS
    float* sdq = reinterpret_cast<float*>(ss + 16 * 24);   // [16][D + 4]
    const int64_t row0 = i * B;
    const float scale_log2 = scale * kLog2e;
    const int g = lane >> 2, c = lane & 3;
    stage_rows<D>(sk, kb, row0, B, Hkv, kvh, lane);
    stage_rows<D>(sv, vb, row0, B, Hkv, kvh, lane);
    float dk[D / 8][4], dv[D / 8][4];
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            dk[nt][u] = 0.f;
            dv[nt][u] = 0.f;
        }
    for (int h = kvh * gq; h < (kvh + 1) * gq; ++h) {
        __syncwarp();                                  // the previous head is done with sq, sg, so, sp, ss
        stage_rows<D>(sq, q, row0, B, H, h, lane);
        stage_rows<D>(sg, dO, row0, B, H, h, lane);
        stage_rows<D>(so, o, row0, B, H, h, lane);
        // the dq rows this head's part is added to, fetched with the inputs
#pragma unroll 4
        for (int e = lane; e < 16 * (D / 4); e += 32) {
            const int r = e / (D / 4), c4 = (e % (D / 4)) * 4;
            if (r < B) cp_async16(sdq + r * (D + 4) + c4, dq + ((row0 + r) * H + h) * D + c4);
        }
        float l2[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int r = g + 8 * e;
            const float l = r < B ? lse[(row0 + r) * H + h] : INFINITY;
            l2[e] = isfinite(l) ? l * kLog2e : INFINITY;   // rows with no key at all: P = 0
        }
        cp_async_wait_all();
        __syncwarp();
        // D_r = dO_r . o_r: lanes 2r, 2r + 1 take halves of row r
        float Dr;
        {
            const int r = lane >> 1, c0 = (lane & 1) * (D / 2);
            float part = 0.f;
#pragma unroll 8
            for (int t = 0; t < D / 2; t += 2) {
                const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(sg + r * LD + c0 + t);
                const __nv_bfloat162 y = *reinterpret_cast<const __nv_bfloat162*>(so + r * LD + c0 + t);
                part = fmaf(__low2float(x), __low2float(y), fmaf(__high2float(x), __high2float(y), part));
            }
            Dr = part + __shfl_xor_sync(kAll, part, 1);
        }
        const float Dg[2] = {__shfl_sync(kAll, Dr, 2 * g), __shfl_sync(kAll, Dr, 2 * (g + 8))};
        float s[2][4], dp[2][4];
        scores16<D>(s, sq, sk, lane);
        scores16<D>(dp, sg, sv, lane);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = nt * 8 + 2 * c + (u & 1), e = u >> 1;
                const float P = j < B ? exp2f(s[nt][u] * scale_log2 - l2[e]) : 0.f;
                s[nt][u] = P;
                dp[nt][u] = P * (dp[nt][u] - Dg[e]);
            }
        uint32_t pa[4], da[4];
        as_a(pa, s);
        as_a(da, dp);
        // dq rows g, g + 8 of head h: += scale dS K, in two halves of the columns
        dq_add<D, 0>(dq, sdq, da, sk, row0, B, H, h, scale, lane);
        dq_add<D, D / 2>(dq, sdq, da, sk, row0, B, H, h, scale, lane);
        // P and dS through shared memory (row-major bf16), read back transposed as
        // the A fragments of P^T and dS^T
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            *reinterpret_cast<uint32_t*>(sp + g * 24 + nt * 8 + 2 * c) = pack2(s[nt][0], s[nt][1]);
            *reinterpret_cast<uint32_t*>(sp + (g + 8) * 24 + nt * 8 + 2 * c) = pack2(s[nt][2], s[nt][3]);
            *reinterpret_cast<uint32_t*>(ss + g * 24 + nt * 8 + 2 * c) = pack2(dp[nt][0], dp[nt][1]);
            *reinterpret_cast<uint32_t*>(ss + (g + 8) * 24 + nt * 8 + 2 * c) = pack2(dp[nt][2], dp[nt][3]);
        }
        __syncwarp();
        uint32_t pt[4], dt[4];
        {
            // A fragment of X^T from row-major X: matrices (X^T rows 0-7 = X cols 0-7, ...)
            const int tr = (lane & 7) + (lane >> 4) * 8, tc = ((lane >> 3) & 1) * 8;
            ldsm_x4_t(pt, sp + tr * 24 + tc);
            ldsm_x4_t(dt, ss + tr * 24 + tc);
        }
        times_rows<D, D / 8>(dv, pt, sg, lane);        // dV += P^T dO
        times_rows<D, D / 8>(dk, dt, sq, lane);        // dK += dS^T Q
    }
    // dk_blk (scaled), dv_blk rows g, g + 8 (keys) of key/value head kvh
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int r = g + 8 * e;
        if (r < B) {
            const int64_t off = ((row0 + r) * Hkv + kvh) * D + 2 * c;
#pragma unroll
            for (int nt = 0; nt < D / 8; ++nt) {
                *reinterpret_cast<float2*>(dkb + off + nt * 8) =
                    make_float2(scale * dk[nt][2 * e], scale * dk[nt][2 * e + 1]);
                *reinterpret_cast<float2*>(dvb + off + nt * 8) = make_float2(dv[nt][2 * e], dv[nt][2 * e + 1]);
            }
        }
    }
}

template <int D>
skv_status fwd_go(const skv_problem& pb, const void* q, const void* kb, const void* vb, float* o, float* lse,
                  int64_t items, const skv_host::Ctx& c) {
    const int smem = kWarpsFwd * 3 * 16 * (D + 8) * 2;
    const int64_t grid = (items + kWarpsFwd - 1) / kWarpsFwd;
    if (grid > 0x7fffffffLL) return SKV_ERR_UNSUPPORTED;
    auto kern = block_local_fwd_mma_kernel<D>;
    SKV_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    kern<<<(unsigned)grid, 32 * kWarpsFwd, smem, c.stream>>>(
        static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(kb),
        static_cast<const __nv_bfloat16*>(vb), pb.B, pb.n_heads, pb.n_kv_heads, items, pb.scale * kLog2e, o, lse);
    return SKV_OK;
}

template <int D>
skv_status bwd_go(const skv_problem& pb, const void* q, const void* kb, const void* vb, const void* o,
                  const float* lse, const void* dO, float* dq, float* dkb, float* dvb, int64_t items,
                  const skv_host::Ctx& c) {
    const int smem = kWarpsBwd * bwd_warp_bytes<D>();
    const int64_t grid = (items + kWarpsBwd - 1) / kWarpsBwd;
    if (grid > 0x7fffffffLL) return SKV_ERR_UNSUPPORTED;
    auto kern = block_local_bwd_mma_kernel<D>;
    SKV_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    kern<<<(unsigned)grid, 32 * kWarpsBwd, smem, c.stream>>>(
        static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(kb),
        static_cast<const __nv_bfloat16*>(vb), static_cast<const __nv_bfloat16*>(o), lse,
        static_cast<const __nv_bfloat16*>(dO), pb.B, pb.n_heads, pb.n_kv_heads, items, pb.scale, dq, dkb, dvb);
    return SKV_OK;
}

}  // namespace

namespace skv_internal {

bool block_local_mma_supported(const skv_problem& pb) {
    return pb.dtype == SKV_BF16 && pb.B <= 16 && (pb.head_dim == 64 || pb.head_dim == 128);
}

skv_status launch_block_local_fwd_mma(const skv_problem& pb, const void* q, const void* kb, const void* vb, float* o,
                                      float* lse, const skv_host::Ctx& c) {
    const int64_t items = int64_t(pb.n_blocks) * pb.n_heads;
    return pb.head_dim == 128 ? fwd_go<128>(pb, q, kb, vb, o, lse, items, c)
                              : fwd_go<64>(pb, q, kb, vb, o, lse, items, c);
}

skv_status launch_block_local_bwd_mma(const skv_problem& pb, const void* q, const void* kb, const void* vb,
                                      const void* o, const float* lse, const void* dO, float* dq, float* dkb,
                                      float* dvb, const skv_host::Ctx& c) {
    const int64_t items = int64_t(pb.n_blocks) * pb.n_kv_heads;
    return pb.head_dim == 128 ? bwd_go<128>(pb, q, kb, vb, o, lse, dO, dq, dkb, dvb, items, c)
                              : bwd_go<64>(pb, q, kb, vb, o, lse, dO, dq, dkb, dvb, items, c);
}

}  // namespace skv_internal
