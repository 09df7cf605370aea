// Tensor-core anchor attention (tcgen05 + TMEM + TMA), sm_103a.
#include "skv_tc.h"

namespace skv_tc {

bool fwd_supported(const skv_problem&) { return false; }
bool bwd_supported(const skv_problem&) { return false; }
size_t fwd_scratch_bytes(const skv_problem&) { return 0; }
size_t bwd_scratch_bytes(const skv_problem&) { return 0; }

skv_status launch_attn_fwd_tc(const skv_problem&, const void*, const void*, const void*, skv::RankCSR, float*,
                              float*, void*, const skv_host::Ctx&) {
    return SKV_ERR_UNSUPPORTED;
}
skv_status launch_attn_bwd_tc(const skv_problem&, const void*, const void*, const void*, const void*,
                              const float*, const float*, skv::RankCSR, float*, float*, float*, void*,
                              const skv_host::Ctx&) {
    return SKV_ERR_UNSUPPORTED;
}

}  // namespace skv_tc
