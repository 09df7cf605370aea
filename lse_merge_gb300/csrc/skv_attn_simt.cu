// fp32 CUDA-core anchor attention (forward partials and backward) of libskv.
//
// This is the path of fp32 problems, where tensor-core precision (bf16/tf32
// products) cannot meet fp32 accuracy.  One thread block owns up to 16 rows of
// one anchor block, one head and one virtual rank; because all B rows of a
// block share the window [s_i, a_i) [Split-KV §3.1, Fig. 1], the key range of
// a work item is the window clipped to each chunk of the rank [§4.2] and no
// element-wise mask is needed.  Key tiles of 64 rows are staged in shared
// memory as fp32.
//
// Forward: Eq. 3 of "Split-KV: Efficient Context Parallelism for Training
// Diffusion Drafters" (§4.1) with an online (running max) softmax.
// Backward: Alg. 1's backward in merged form, P = exp(z - l_global),
// dS = P (dP - D); dq^(p) is written per rank (summed by the dq-sum pass) and
// dk, dv accumulate with fp32 atomics (several blocks see the same key; with
// grouped queries, every query head of a key/value head's group too).
#include <math.h>

#include "skv_common.cuh"
#include "skv_internal.h"

namespace {

constexpr int kRows = 16;     // query rows per thread block
constexpr int kKeys = 64;     // keys per shared-memory tile
constexpr int kThreads = 128;

struct SimtSmem {
    static size_t bytes(int d, bool bwd) {
        size_t f = size_t(kRows) * d            // q
                 + size_t(kKeys) * (d + 1)      // K (padded)
                 + size_t(kKeys) * (d + 1)      // V (padded)
                 + size_t(kRows) * kKeys        // scores / P
                 + size_t(kRows) * d            // accumulator (o or dq)
                 + 4 * kRows;                   // row stats
        if (bwd) f += size_t(kRows) * d + size_t(kRows) * kKeys;   // dO, dS
        return f * sizeof(float);
    }
};

template <typename T>
__device__ __forceinline__ void load_tile(float* dst, int ld, const T* __restrict__ src, int64_t row0, int nrows,
                                          int H, int h, int d) {
    for (int e = threadIdx.x; e < kKeys * d; e += blockDim.x) {
        const int r = e / d, t = e - (e / d) * d;
        dst[r * ld + t] = r < nrows ? skv::to_f32(src[((row0 + r) * H + h) * int64_t(d) + t]) : 0.f;
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
attn_fwd_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                     const int32_t* __restrict__ s, const int32_t* __restrict__ a, int B, int n_blocks, int H,
                     int Hkv, int d, int64_t S, int m, int P, float scale, skv::RankCSR csr, float* __restrict__ o_part,
                     float* __restrict__ lse_part) {
    extern __shared__ float sm[];
    const int groups = (B + kRows - 1) / kRows;
    const int i = blockIdx.x / groups;
    const int g = blockIdx.x - i * groups;
    const int h = blockIdx.y, p = blockIdx.z;
    const int kvh = h / (H / Hkv);                   // key/value head (grouped-query layouts)
    const int r0 = i * B + g * kRows;
    const int nr = min(kRows, B - g * kRows);
    const int64_t Qn = int64_t(n_blocks) * B;
    float* sq = sm;
    float* sk = sq + kRows * d;
    float* sv = sk + kKeys * (d + 1);
    float* ss = sv + kKeys * (d + 1);
    float* acc = ss + kRows * kKeys;
    float* mrow = acc + kRows * d;
    float* lrow = mrow + kRows;
    float* alpha = lrow + kRows;
    for (int e = threadIdx.x; e < kRows * d; e += blockDim.x) {
        const int r = e / d, t = e % d;
        sq[e] = r < nr ? skv::to_f32(q[((int64_t)(r0 + r) * H + h) * d + t]) : 0.f;
        acc[e] = 0.f;
    }
    if (threadIdx.x < kRows) { mrow[threadIdx.x] = -INFINITY; lrow[threadIdx.x] = 0.f; }
    int64_t lo, hi;
    skv::block_window(s, a, i, S, lo, hi);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int ci = csr.ptr[p]; ci < csr.ptr[p + 1]; ++ci) {
        const int64_t cl = int64_t(csr.list[ci]) * m;
        const int64_t klo = lo > cl ? lo : cl;
        const int64_t khi = hi < cl + m ? hi : cl + m;
        for (int64_t kt = klo; kt < khi; kt += kKeys) {
            const int nk = (int)((khi - kt) < kKeys ? (khi - kt) : kKeys);
            load_tile(sk, d + 1, k, kt, nk, Hkv, kvh, d);
            load_tile(sv, d + 1, v, kt, nk, Hkv, kvh, d);
            __syncthreads();
            for (int e = threadIdx.x; e < kRows * kKeys; e += blockDim.x) {
                const int r = e / kKeys, c = e % kKeys;
                float z = -INFINITY;
                if (r < nr && c < nk) {
                    float dot = 0.f;
                    for (int t = 0; t < d; ++t) dot = fmaf(sq[r * d + t], sk[c * (d + 1) + t], dot);
                    z = dot * scale;
                }
                ss[e] = z;
            }
            __syncthreads();
            // online softmax: warp w owns rows w, w+4, ...; lanes own 2 columns each
            for (int r = warp; r < kRows; r += kThreads / 32) {
                const float z0 = ss[r * kKeys + lane], z1 = ss[r * kKeys + lane + 32];
                float mx = fmaxf(z0, z1);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                const float m_old = mrow[r];
                const float m_new = fmaxf(m_old, mx);
                float p0 = 0.f, p1 = 0.f, al = 1.f;
                if (m_new != -INFINITY) {
                    p0 = expf(z0 - m_new);
                    p1 = expf(z1 - m_new);
                    al = (m_old == -INFINITY) ? 0.f : expf(m_old - m_new);
                }
                ss[r * kKeys + lane] = p0;
                ss[r * kKeys + lane + 32] = p1;
                float sum = p0 + p1;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                if (lane == 0) {
                    lrow[r] = lrow[r] * al + sum;
                    mrow[r] = m_new;
                    alpha[r] = al;
                }
            }
            __syncthreads();
            for (int e = threadIdx.x; e < kRows * d; e += blockDim.x) {
                const int r = e / d, t = e % d;
                float o = acc[e] * alpha[r];
                for (int c = 0; c < nk; ++c) o = fmaf(ss[r * kKeys + c], sv[c * (d + 1) + t], o);
                acc[e] = o;
            }
            __syncthreads();
        }
    }
    for (int e = threadIdx.x; e < nr * d; e += blockDim.x) {
        const int r = e / d, t = e % d;
        const float l = lrow[r];
        o_part[((int64_t(p) * Qn + r0 + r) * H + h) * d + t] = l > 0.f ? acc[e] / l : 0.f;
    }
    if (threadIdx.x < nr) {
        const int r = threadIdx.x;
        const float l = lrow[r];
        lse_part[(int64_t(p) * Qn + r0 + r) * H + h] = l > 0.f ? mrow[r] + logf(l) : -INFINITY;
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
attn_bwd_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                     const T* __restrict__ dO, const float* __restrict__ lse, const float* __restrict__ Drow,
                     const int32_t* __restrict__ s, const int32_t* __restrict__ a, int B, int n_blocks, int H,
                     int Hkv, int d, int64_t S, int m, int P, float scale, skv::RankCSR csr,
                     float* __restrict__ dq_part, float* __restrict__ dk, float* __restrict__ dv) {
    extern __shared__ float sm[];
    const int groups = (B + kRows - 1) / kRows;
    const int i = blockIdx.x / groups;
    const int g = blockIdx.x - i * groups;
    const int h = blockIdx.y, p = blockIdx.z;
    const int kvh = h / (H / Hkv);                   // key/value head (grouped-query layouts)
    const int r0 = i * B + g * kRows;
    const int nr = min(kRows, B - g * kRows);
    const int64_t Qn = int64_t(n_blocks) * B;
    float* sq = sm;
    float* sk = sq + kRows * d;
    float* sv = sk + kKeys * (d + 1);
    float* sp = sv + kKeys * (d + 1);
    float* acc = sp + kRows * kKeys;
    float* rl = acc + kRows * d;      // lse of the rows
    float* rD = rl + kRows;           // D of the rows
    float* sdo = rD + 3 * kRows;
    float* sds = sdo + kRows * d;
    for (int e = threadIdx.x; e < kRows * d; e += blockDim.x) {
        const int r = e / d, t = e % d;
        const int64_t off = ((int64_t)(r0 + r) * H + h) * d + t;
        sq[e] = r < nr ? skv::to_f32(q[off]) : 0.f;
        sdo[e] = r < nr ? skv::to_f32(dO[off]) : 0.f;
        acc[e] = 0.f;
    }
    if (threadIdx.x < kRows) {
        const int r = threadIdx.x;
        rl[r] = r < nr ? lse[(int64_t)(r0 + r) * H + h] : -INFINITY;
        rD[r] = r < nr ? Drow[(int64_t)(r0 + r) * H + h] : 0.f;
    }
    int64_t lo, hi;
    skv::block_window(s, a, i, S, lo, hi);
    __syncthreads();
    for (int ci = csr.ptr[p]; ci < csr.ptr[p + 1]; ++ci) {
        const int64_t cl = int64_t(csr.list[ci]) * m;
        const int64_t klo = lo > cl ? lo : cl;
        const int64_t khi = hi < cl + m ? hi : cl + m;
        for (int64_t kt = klo; kt < khi; kt += kKeys) {
            const int nk = (int)((khi - kt) < kKeys ? (khi - kt) : kKeys);
            load_tile(sk, d + 1, k, kt, nk, Hkv, kvh, d);
            load_tile(sv, d + 1, v, kt, nk, Hkv, kvh, d);
            __syncthreads();
            for (int e = threadIdx.x; e < kRows * kKeys; e += blockDim.x) {
                const int r = e / kKeys, c = e % kKeys;
                float pr = 0.f, ds = 0.f;
                if (r < nr && c < nk && rl[r] != -INFINITY) {
                    float dot = 0.f, dp = 0.f;
                    for (int t = 0; t < d; ++t) {
                        dot = fmaf(sq[r * d + t], sk[c * (d + 1) + t], dot);
                        dp = fmaf(sdo[r * d + t], sv[c * (d + 1) + t], dp);
                    }
                    pr = expf(dot * scale - rl[r]);
                    ds = pr * (dp - rD[r]);
                }
                sp[e] = pr;
                sds[e] = ds;
            }
            __syncthreads();
            for (int e = threadIdx.x; e < kRows * d; e += blockDim.x) {
                const int r = e / d, t = e % d;
                float o = 0.f;
                for (int c = 0; c < nk; ++c) o = fmaf(sds[r * kKeys + c], sk[c * (d + 1) + t], o);
                acc[e] = fmaf(scale, o, acc[e]);
            }
            for (int e = threadIdx.x; e < nk * d; e += blockDim.x) {
                const int c = e / d, t = e % d;
                float gk = 0.f, gv = 0.f;
                for (int r = 0; r < nr; ++r) {
                    gk = fmaf(sds[r * kKeys + c], sq[r * d + t], gk);
                    gv = fmaf(sp[r * kKeys + c], sdo[r * d + t], gv);
                }
                const int64_t off = ((kt + c) * Hkv + kvh) * int64_t(d) + t;
                atomicAdd(dk + off, scale * gk);
                atomicAdd(dv + off, gv);
            }
            __syncthreads();
        }
    }
    for (int e = threadIdx.x; e < nr * d; e += blockDim.x) {
        const int r = e / d, t = e % d;
        dq_part[((int64_t(p) * Qn + r0 + r) * H + h) * d + t] = acc[e];
    }
}

dim3 simt_grid(const skv_problem& pb) {
    const int groups = (pb.B + kRows - 1) / kRows;
    return dim3((unsigned)(pb.n_blocks * groups), (unsigned)pb.n_heads, (unsigned)pb.P);
}

}  // namespace

namespace skv_internal {

skv_status launch_attn_fwd_simt(const skv_problem& pb, const void* q, const void* k, const void* v,
                                skv::RankCSR csr, float* o_part, float* lse_part, const skv_host::Ctx& c) {
    if (pb.n_blocks == 0) return SKV_OK;
    const size_t smem = SimtSmem::bytes(pb.head_dim, false);
    const float scale = pb.scale;
    if (pb.dtype == SKV_BF16) {
        auto kern = attn_fwd_simt_kernel<__nv_bfloat16>;
        SKV_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        kern<<<simt_grid(pb), kThreads, smem, c.stream>>>(
            static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
            static_cast<const __nv_bfloat16*>(v), pb.s, pb.a, pb.B, pb.n_blocks, pb.n_heads, pb.n_kv_heads, pb.head_dim, pb.S,
            pb.m, pb.P, scale, csr, o_part, lse_part);
    } else {
        auto kern = attn_fwd_simt_kernel<float>;
        SKV_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        kern<<<simt_grid(pb), kThreads, smem, c.stream>>>(
            static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v), pb.s, pb.a,
            pb.B, pb.n_blocks, pb.n_heads, pb.n_kv_heads, pb.head_dim, pb.S, pb.m, pb.P, scale, csr, o_part, lse_part);
    }
    SKV_LAUNCHED();
    return SKV_OK;
}

skv_status launch_attn_bwd_simt(const skv_problem& pb, const void* q, const void* k, const void* v,
                                const void* dO, const float* lse, const float* D, skv::RankCSR csr,
                                float* dq_part, float* dk, float* dv, const skv_host::Ctx& c) {
    if (pb.n_blocks == 0) return SKV_OK;
    const size_t smem = SimtSmem::bytes(pb.head_dim, true);
    if (pb.dtype == SKV_BF16) {
        auto kern = attn_bwd_simt_kernel<__nv_bfloat16>;
        SKV_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        kern<<<simt_grid(pb), kThreads, smem, c.stream>>>(
            static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
            static_cast<const __nv_bfloat16*>(v), static_cast<const __nv_bfloat16*>(dO), lse, D, pb.s, pb.a, pb.B,
            pb.n_blocks, pb.n_heads, pb.n_kv_heads, pb.head_dim, pb.S, pb.m, pb.P, pb.scale, csr, dq_part, dk, dv);
    } else {
        auto kern = attn_bwd_simt_kernel<float>;
        SKV_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        kern<<<simt_grid(pb), kThreads, smem, c.stream>>>(
            static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v),
            static_cast<const float*>(dO), lse, D, pb.s, pb.a, pb.B, pb.n_blocks, pb.n_heads, pb.n_kv_heads, pb.head_dim, pb.S, pb.m,
            pb.P, pb.scale, csr, dq_part, dk, dv);
    }
    SKV_LAUNCHED();
    return SKV_OK;
}

}  // namespace skv_internal
