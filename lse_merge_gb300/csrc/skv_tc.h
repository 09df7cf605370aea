// Tensor-core (tcgen05 / TMEM / TMA) attention kernels of libskv: interface
// used by the C-ABI layer.
#pragma once

#include "skv_common.cuh"

namespace skv_tc {

// Query heads stacked in one 128-row tile: the g = H/Hkv query heads of a key/value
// head (grouped-query layouts of Split-KV Table 2), each over 128/g rows, so one K/V
// tile serves the whole group and a tile's rows come from fewer blocks; 1 otherwise.
inline int pack_heads(const skv_problem& pb) {
    const int g = pb.n_kv_heads > 0 ? pb.n_heads / pb.n_kv_heads : 1;
    return (g > 1 && g <= 16 && 128 % g == 0) ? g : 1;
}

bool fwd_supported(const skv_problem& pb);
bool bwd_supported(const skv_problem& pb);
// Per query tile of `rows` rows: (union lo, hi, full-visibility lo, hi) of its rows' key windows.
skv_status launch_qtile_bounds(const skv_problem& pb, int4* out, const skv_host::Ctx& c, int rows = 128);
size_t fwd_scratch_bytes(const skv_problem& pb);
size_t bwd_scratch_bytes(const skv_problem& pb);

skv_status launch_attn_fwd_tc(const skv_problem& pb, const void* q, const void* k, const void* v,
                              skv::RankCSR csr, float* o_part, float* lse_part, void* scratch,
                              const skv_host::Ctx& c);
skv_status launch_attn_bwd_tc(const skv_problem& pb, const void* q, const void* k, const void* v,
                              const void* dO, const float* lse2, const float* D, skv::RankCSR csr,
                              float* dq, float* dk, float* dv, void* scratch, const skv_host::Ctx& c);

}  // namespace skv_tc
