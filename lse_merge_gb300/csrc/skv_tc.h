// Tensor-core (tcgen05 / TMEM / TMA) attention kernels of libskv: interface
// used by the C-ABI layer.
#pragma once

#include "skv_common.cuh"

namespace skv_tc {

bool fwd_supported(const skv_problem& pb);
bool bwd_supported(const skv_problem& pb);
// Per 128-row query tile: (union lo, hi, full-visibility lo, hi) of its rows' key windows.
skv_status launch_qtile_bounds(const skv_problem& pb, int4* out, const skv_host::Ctx& c);
size_t fwd_scratch_bytes(const skv_problem& pb);
size_t bwd_scratch_bytes(const skv_problem& pb);

skv_status launch_attn_fwd_tc(const skv_problem& pb, const void* q, const void* k, const void* v,
                              skv::RankCSR csr, float* o_part, float* lse_part, void* scratch,
                              const skv_host::Ctx& c);
skv_status launch_attn_bwd_tc(const skv_problem& pb, const void* q, const void* k, const void* v,
                              const void* dO, const float* lse2, const float* D, skv::RankCSR csr,
                              float* dq, float* dk, float* dv, void* scratch, const skv_host::Ctx& c);

}  // namespace skv_tc
