// Helpers shared by the tensor-core attention kernels (internal).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "skv_common.cuh"

namespace skv_tcc {

constexpr int BM = 128;          // query rows per tile
constexpr int BN = 128;          // keys per tile

// Rows [qt*rows, qt*rows+rows) of the packed query (rows = 128 for a plain tile,
// 128/g when a tile stacks the g query heads of a key/value head): key bounds.
struct TileBounds {
    int64_t lo, hi;     // union of the rows' windows (empty if lo >= hi)
    int64_t flo, fhi;   // intersection: keys every live row sees
};

__device__ __forceinline__ TileBounds tile_bounds(const int32_t* s, const int32_t* a, int B, int64_t Qn, int64_t S,
                                                  int qt, int rows = BM) {
    TileBounds tb{S, 0, 0, S};
    const int64_t r0 = int64_t(qt) * rows;
    const int64_t r1 = (r0 + rows < Qn ? r0 + rows : Qn) - 1;
    bool any_empty = false;
    for (int64_t i = r0 / B; i <= r1 / B; ++i) {
        int64_t lo, hi;
        skv::block_window(s, a, (int)i, S, lo, hi);
        if (hi > lo) {
            tb.lo = lo < tb.lo ? lo : tb.lo;
            tb.hi = hi > tb.hi ? hi : tb.hi;
        } else {
            any_empty = true;
        }
        tb.flo = lo > tb.flo ? lo : tb.flo;
        tb.fhi = hi < tb.fhi ? hi : tb.fhi;
    }
    if (any_empty || r1 - r0 + 1 < rows) tb.fhi = tb.flo;   // partial or empty rows: mask every tile
    return tb;
}

// Walks the 128-key tiles of a chunk list (rank-major, ascending inside a rank)
// that intersect [lo, hi).  Every role runs its own copy and sees the same sequence.
struct TileIter {
    const int32_t* list;
    int ci, ce, m;
    int64_t x, xe, lo, hi;
    // ranks [p0, p1): the CSR list is rank-major, ascending inside a rank
    __device__ __forceinline__ void init(skv::RankCSR csr, int p0, int p1, int m_, int64_t lo_, int64_t hi_) {
        init_list(csr.list + csr.ptr[p0], csr.ptr[p1] - csr.ptr[p0], m_, lo_, hi_);
    }
    // an explicit list of n chunk indices (global or shared memory)
    __device__ __forceinline__ void init_list(const int32_t* list_, int n, int m_, int64_t lo_, int64_t hi_) {
        list = list_;
        ci = 0;
        ce = n;
        m = m_;
        lo = lo_;
        hi = hi_;
        x = 0;
        xe = 0;
    }
    // number of tiles a fresh iterator yields, chunk by chunk (no per-tile stepping)
    __device__ __forceinline__ int count() const {
        int T = 0;
        for (int i = ci; i < ce; ++i) {
            const int64_t cl = int64_t(list[i]) * m;
            const int64_t a0 = cl > lo ? cl : lo;
            const int64_t a1 = (cl + m) < hi ? (cl + m) : hi;
            if (a0 < a1) T += (int)((a1 - (a0 & ~int64_t(BN - 1)) + BN - 1) / BN);
        }
        return T;
    }
    __device__ __forceinline__ bool next(int64_t& x0) {
        while (x >= xe) {
            if (ci >= ce) return false;
            const int64_t cl = int64_t(list[ci++]) * m;
            const int64_t a0 = cl > lo ? cl : lo;
            const int64_t a1 = (cl + m) < hi ? (cl + m) : hi;
            if (a0 < a1) {
                x = a0 & ~int64_t(BN - 1);
                xe = a1;
            }
        }
        x0 = x;
        x += BN;
        return true;
    }
};

// The 128-key tiles that meet [lo, hi), ascending: the same interface as TileIter
// for a walk that does not go chunk by chunk.
struct KeyRange {
    int64_t x, xe;
    __device__ __forceinline__ void init(int64_t lo, int64_t hi) {
        x = lo & ~int64_t(BN - 1);
        xe = hi > lo ? hi : x;
    }
    __device__ __forceinline__ int count() const { return xe > x ? (int)((xe - x + BN - 1) / BN) : 0; }
    __device__ __forceinline__ bool next(int64_t& x0) {
        if (x >= xe) return false;
        x0 = x;
        x += BN;
        return true;
    }
};

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2D bf16 view [rows][cols] of a row-major tensor, 64 x box_rows boxes, 128-byte swizzle.
inline bool make_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int box_rows = 128) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D fp32 view [rows][cols] of a row-major tensor, 32x32 boxes (128-byte rows),
// 128-byte swizzle: the store side of a 32-row, 32-column register tile.
inline bool make_map_f32(CUtensorMap* map, void* ptr, int64_t rows, int64_t cols) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t es[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// 3D fp32 view [d2][d1][cols] of a row-major tensor, 32 x box_rows x 1 boxes, 128-byte
// swizzle: rows past d1 inside one d2 slice are dropped by a store.
inline bool make_map_f32_3d(CUtensorMap* map, void* ptr, int64_t d2, int64_t d1, int64_t cols, int box_rows = 32) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)d1, (cuuint64_t)d2};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 4, (cuuint64_t)(cols * d1) * 4};
    cuuint32_t box[3] = {32, (cuuint32_t)box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace skv_tcc
