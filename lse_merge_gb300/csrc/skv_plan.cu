// Planning kernels of libskv: chunk prices (Eq. 6), cost-aware LPT and the
// two baseline planners, and the per-rank chunk lists the attention kernels
// iterate.  Source: "Split-KV: Efficient Context Parallelism for Training
// Diffusion Drafters", §4.2 and Fig. 5.  All integer work, bit-exact.
#include "skv_common.cuh"
#include "skv_internal.h"

namespace {

constexpr int kCostThreads = 256;

__device__ __forceinline__ int64_t warp_sum64(int64_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// One thread block per chunk j: costs[j] = B * sum_i (min(a_i, l+m) - max(s_i, l))^+
// with l = j*m  [Split-KV §4.2, Eq. 6].  Block 0 also validates the anchors.
__global__ void __launch_bounds__(kCostThreads)
chunk_costs_kernel(const int32_t* __restrict__ s, const int32_t* __restrict__ a, int n_blocks,
                   int64_t S, int m, int B, int64_t* __restrict__ costs, int* status) {
    const int64_t lam = int64_t(blockIdx.x) * m;
    const int64_t rhs = lam + m;
    int64_t acc = 0;
    bool bad = false;
    for (int i = threadIdx.x; i < n_blocks; i += blockDim.x) {
        const int64_t si = s[i], ai = a[i];
        bad |= (si < 0) | (ai < si) | (ai > S);
        int64_t lo, hi;
        skv::block_window(s, a, i, S, lo, hi);
        const int64_t ov = (hi < rhs ? hi : rhs) - (lo > lam ? lo : lam);
        acc += ov > 0 ? ov : 0;
    }
    if (blockIdx.x == 0 && __syncthreads_or(bad) && threadIdx.x == 0)
        skv::raise_status(status, SKV_ERR_BAD_ANCHORS);
    __shared__ int64_t part[kCostThreads / 32];
    acc = warp_sum64(acc);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x < 32) {
        int64_t v = threadIdx.x < (blockDim.x >> 5) ? part[threadIdx.x] : 0;
        v = warp_sum64(v);
        if (threadIdx.x == 0) costs[blockIdx.x] = int64_t(B) * v;
    }
}

// "a is taken before b" in LPT order: cost descending, then index ascending.
__device__ __forceinline__ bool lpt_before(int64_t ca, int32_t ia, int64_t cb, int32_t ib) {
    return ca > cb || (ca == cb && ia < ib);
}

constexpr int kLptThreads = 1024;

// Cost-aware LPT [Split-KV §4.2]: one thread block.  (1) bitonic sort of
// (cost, index) in shared memory by the whole block; (2) the greedy pass by a
// single warp: the ranks' loads and chunk counts sit in shared memory, lane l
// keeps its best (load, rank) among ranks l, l+32, ... with fewer than J chunks,
// and each step is one warp-wide argmin (only the receiving lane rescans).
__global__ void __launch_bounds__(kLptThreads)
lpt_kernel(const int64_t* __restrict__ costs, int n, int P, int J,
           int32_t* __restrict__ rank_of_chunk, int32_t* __restrict__ order,
           int64_t* __restrict__ load_out) {
    extern __shared__ unsigned char smem_raw[];
    int n2 = 1;
    while (n2 < n) n2 <<= 1;
    int64_t* key = reinterpret_cast<int64_t*>(smem_raw);
    int32_t* idx = reinterpret_cast<int32_t*>(key + n2);
    for (int t = threadIdx.x; t < n2; t += blockDim.x) {
        key[t] = t < n ? costs[t] : int64_t(-1);   // padding sorts after every real chunk
        idx[t] = t < n ? t : 0x7fffffff;
    }
    __syncthreads();
    for (int kk = 2; kk <= n2; kk <<= 1) {
        for (int jj = kk >> 1; jj > 0; jj >>= 1) {
            for (int t = threadIdx.x; t < n2; t += blockDim.x) {
                const int u = t ^ jj;
                if (u > t) {
                    const bool up = (t & kk) == 0;
                    const bool t_first = lpt_before(key[t], idx[t], key[u], idx[u]);
                    if (up ? !t_first : t_first) {
                        const int64_t kt = key[t]; key[t] = key[u]; key[u] = kt;
                        const int32_t it = idx[t]; idx[t] = idx[u]; idx[u] = it;
                    }
                }
            }
            __syncthreads();
        }
    }
    // per-rank load and chunk count in shared memory, behind the sorted keys
    int64_t* rload = reinterpret_cast<int64_t*>(smem_raw + ((size_t(n2) * 12 + 7) & ~size_t(7)));
    int32_t* rheld = reinterpret_cast<int32_t*>(rload + P);
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
        rload[p] = 0;
        rheld[p] = 0;
    }
    __syncthreads();
    if (threadIdx.x >= 32) return;
    const int lane = threadIdx.x;
    constexpr int64_t kFull = 0x7fffffffffffffffLL;
    // best (load, rank) of this lane among its ranks lane, lane + 32, ... that can
    // still take a chunk; only the lane that received a chunk rescans its ranks
    int64_t best_load = kFull;
    int best_rank = 0x7fffffff;
    auto refresh = [&]() {
        best_load = kFull;
        best_rank = 0x7fffffff;
        for (int p = lane; p < P; p += 32) {
            const int64_t l = rload[p];
            if (rheld[p] < J && l < best_load) {
                best_load = l;
                best_rank = p;
            }
        }
    };
    refresh();
    for (int t = 0; t < n; ++t) {
        const int j = idx[t];
        const int64_t c = key[t];
        int64_t bl = best_load;
        int br = best_rank;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const int64_t ol = __shfl_xor_sync(0xffffffffu, bl, o);
            const int orr = __shfl_xor_sync(0xffffffffu, br, o);
            if (ol < bl || (ol == bl && orr < br)) { bl = ol; br = orr; }
        }
        if (br == 0x7fffffff) break;   // unreachable when n == P*J
        if ((br & 31) == lane) {
            order[int64_t(br) * J + rheld[br]] = j;
            rload[br] += c;
            rheld[br] += 1;
            rank_of_chunk[j] = br;
            refresh();
        }
    }
    __syncwarp();
    for (int p = lane; p < P; p += 32) load_out[p] = rload[p];
}

__global__ void contiguous_kernel(const int64_t* __restrict__ costs, int n, int P, int J,
                                  int32_t* __restrict__ rank_of_chunk, int32_t* __restrict__ order,
                                  int64_t* __restrict__ load) {
    // rank p holds chunks [pJ, (p+1)J)  [Split-KV §5.1 "No balance"]
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < n; j += gridDim.x * blockDim.x) {
        rank_of_chunk[j] = j / J;
        order[j] = j;
    }
    if (costs && load) {
        for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < P; p += gridDim.x * blockDim.x) {
            int64_t acc = 0;
            for (int t = 0; t < J; ++t) acc += costs[int64_t(p) * J + t];
            load[p] = acc;
        }
    }
}

// Zigzag loads [Split-KV §4.2 example, Fig. 5b]: block p sums, over every
// sample u and its chunks z in {p, 2P-1-p} of width L_u/(2P), the Eq. 2 load
// of those positions, computed per anchor as B * |[s_i, a_i) ∩ chunk|.
__global__ void __launch_bounds__(256)
zigzag_kernel(const int32_t* __restrict__ s, const int32_t* __restrict__ a, int n_blocks, int64_t S,
              int B, const int32_t* __restrict__ st, const int32_t* __restrict__ len, int n_samples,
              int P, int64_t* __restrict__ load, int* status) {
    const int p = blockIdx.x;
    int64_t acc = 0;
    bool bad = false;
    for (int u = 0; u < n_samples; ++u) {
        const int64_t L = len[u], s0 = st[u];
        if (L <= 0 || L % (2 * P) != 0 || s0 < 0 || s0 + L > S) { bad = true; continue; }
        const int64_t w = L / (2 * P);
        const int64_t zs[2] = {s0 + p * w, s0 + (2 * P - 1 - p) * w};
        for (int i = threadIdx.x; i < n_blocks; i += blockDim.x) {
            int64_t lo, hi;
            skv::block_window(s, a, i, S, lo, hi);
#pragma unroll
            for (int z = 0; z < 2; ++z) {
                const int64_t ov = (hi < zs[z] + w ? hi : zs[z] + w) - (lo > zs[z] ? lo : zs[z]);
                acc += ov > 0 ? ov : 0;
            }
        }
    }
    if (bad && threadIdx.x == 0) skv::raise_status(status, SKV_ERR_INVALID_ARG);
    __shared__ int64_t part[8];
    acc = warp_sum64(acc);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        int64_t v = 0;
        for (int w2 = 0; w2 < (int)(blockDim.x >> 5); ++w2) v += part[w2];
        load[p] = int64_t(B) * v;
    }
}

// Per-rank chunk lists (CSR, ascending chunk index) from rank_of_chunk: thread
// p scans the (shared-memory cached) map for its own rank.  Out-of-range ranks
// are dropped and flagged.
__global__ void __launch_bounds__(1024)
rank_csr_kernel(const int32_t* __restrict__ roc, int n, int P, int32_t* __restrict__ ptr,
                int32_t* __restrict__ list, int* status) {
    extern __shared__ int32_t sroc[];
    for (int j = threadIdx.x; j < n; j += blockDim.x) {
        const int r = roc[j];
        if (r < 0 || r >= P) skv::raise_status(status, SKV_ERR_INVALID_ARG);
        sroc[j] = r;
    }
    __syncthreads();
    // count per rank, then an exclusive scan by thread 0 in chunks of the block
    __shared__ int32_t wsum[1024];
    for (int base = 0; base < P; base += blockDim.x) {
        const int p = base + threadIdx.x;
        int cnt = 0;
        if (p < P)
            for (int j = 0; j < n; ++j) cnt += (sroc[j] == p);
        wsum[threadIdx.x] = cnt;
        __syncthreads();
        if (threadIdx.x == 0) {
            int run = base == 0 ? 0 : ptr[base];
            for (int t = 0; t < (int)blockDim.x && base + t < P; ++t) {
                ptr[base + t] = run;
                run += wsum[t];
            }
            ptr[(base + blockDim.x < (unsigned)P) ? base + blockDim.x : P] = run;
        }
        __syncthreads();
    }
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
        int pos = ptr[p];
        for (int j = 0; j < n; ++j)
            if (sroc[j] == p) list[pos++] = j;
    }
}

}  // namespace

namespace skv_internal {

skv_status launch_chunk_costs(const skv_problem& pb, int64_t* costs, const skv_host::Ctx& c) {
    const int64_t n_chunks = pb.S / pb.m;
    if (n_chunks == 0) return SKV_OK;
    chunk_costs_kernel<<<(unsigned)n_chunks, kCostThreads, 0, c.stream>>>(
        pb.s, pb.a, pb.n_blocks, pb.S, pb.m, pb.B, costs, c.status);
    SKV_LAUNCHED();
    return SKV_OK;
}

skv_status launch_lpt(const int64_t* costs, int n, int P, int J, int32_t* roc, int32_t* order,
                      int64_t* load, const skv_host::Ctx& c) {
    int n2 = 1;
    while (n2 < n) n2 <<= 1;
    // sorted (cost, index) pairs, then each rank's load and chunk count
    const size_t smem = ((size_t(n2) * (sizeof(int64_t) + sizeof(int32_t)) + 7) & ~size_t(7)) +
                        size_t(P) * (sizeof(int64_t) + sizeof(int32_t));
    SKV_CUDA_CHECK(cudaFuncSetAttribute(lpt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    lpt_kernel<<<1, kLptThreads, smem, c.stream>>>(costs, n, P, J, roc, order, load);
    SKV_LAUNCHED();
    return SKV_OK;
}

skv_status launch_contiguous(const int64_t* costs, int n, int P, int J, int32_t* roc, int32_t* order,
                             int64_t* load, const skv_host::Ctx& c) {
    const int threads = 256;
    const int grid = (int)((n > P ? n : P) + threads - 1) / threads;
    contiguous_kernel<<<grid, threads, 0, c.stream>>>(costs, n, P, J, roc, order, load);
    SKV_LAUNCHED();
    return SKV_OK;
}

skv_status launch_zigzag(const skv_problem& pb, const int32_t* st, const int32_t* len, int n_samples,
                         int64_t* load, const skv_host::Ctx& c) {
    zigzag_kernel<<<pb.P, 256, 0, c.stream>>>(pb.s, pb.a, pb.n_blocks, pb.S, pb.B, st, len, n_samples,
                                              pb.P, load, c.status);
    SKV_LAUNCHED();
    return SKV_OK;
}

skv_status launch_rank_csr(const int32_t* roc, int n, int P, int32_t* ptr, int32_t* list,
                           const skv_host::Ctx& c) {
    const size_t smem = size_t(n) * sizeof(int32_t);
    SKV_CUDA_CHECK(cudaFuncSetAttribute(rank_csr_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    rank_csr_kernel<<<1, 1024, smem, c.stream>>>(roc, n, P, ptr, list, c.status);
    SKV_LAUNCHED();
    return SKV_OK;
}

}  // namespace skv_internal
