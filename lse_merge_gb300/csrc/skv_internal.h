// Internal launcher declarations shared by the libskv translation units.
#pragma once

#include "skv_common.cuh"

namespace skv_internal {

constexpr int kLptMaxChunks = 16384;   // LPT sorts in shared memory
constexpr int kLptMaxRanks = 1024;     // LPT greedy keeps ranks in one warp's registers

skv_status launch_chunk_costs(const skv_problem& pb, int64_t* costs, const skv_host::Ctx& c);
skv_status launch_lpt(const int64_t* costs, int n, int P, int J, int32_t* roc, int32_t* order,
                      int64_t* load, const skv_host::Ctx& c);
skv_status launch_contiguous(const int64_t* costs, int n, int P, int J, int32_t* roc, int32_t* order,
                             int64_t* load, const skv_host::Ctx& c);
skv_status launch_zigzag(const skv_problem& pb, const int32_t* st, const int32_t* len, int n_samples,
                         int64_t* load, const skv_host::Ctx& c);
skv_status launch_rank_csr(const int32_t* roc, int n, int P, int32_t* ptr, int32_t* list,
                           const skv_host::Ctx& c);

skv_status launch_merge(const float* o_part, const float* lse_part, int P, int64_t rows, int d,
                        void* o, skv_dtype o_dtype, float* lse, const skv_host::Ctx& c);
skv_status launch_merge_bwd(const float* o_part, const float* lse_part, int P, int64_t rows, int d, const void* dO,
                            skv_dtype do_dtype, const float* dlse, float* do_part, float* dlse_part,
                            const skv_host::Ctx& c);
// Y = o W_o^T (tcgen05 GEMM): o bf16 [Qn][hd], w_o bf16 [d_model][hd], y fp32 [Qn][d_model]
skv_status launch_oproj(const void* o, int64_t Qn, int hd, const void* w_o, int d_model, float* y,
                        const skv_host::Ctx& c);
// D_r = dO_r . o_r and lse2_r = lse_r * log2(e) (base-2 LSE for exp2 kernels);
// row-major [Qn][H] or head-major [H][Qp] (pad rows: lse2 = +inf, D = 0)
skv_status launch_bwd_prep(const void* o, const void* dO, const float* lse, skv_dtype dt, int64_t Qn, int64_t Qp,
                           int H, int d, bool head_major, float* D, float* lse2, const skv_host::Ctx& c);
// dq[r] = sum_p dq_part[p][r]
skv_status launch_dq_sum(const float* dq_part, int P, int64_t rows, int d, float* dq,
                         const skv_host::Ctx& c);
skv_status launch_zero(float* p, int64_t n, const skv_host::Ctx& c);

// fp32 CUDA-core attention (any dtype input), one CTA per (block, head, rank)
skv_status launch_attn_fwd_simt(const skv_problem& pb, const void* q, const void* k, const void* v,
                                skv::RankCSR csr, float* o_part, float* lse_part, const skv_host::Ctx& c);
skv_status launch_attn_bwd_simt(const skv_problem& pb, const void* q, const void* k, const void* v,
                                const void* dO, const float* lse, const float* D, skv::RankCSR csr,
                                float* dq_part, float* dk, float* dv, const skv_host::Ctx& c);

// block-local term on warp-level MMA (bf16, B <= 16, head_dim 64 or 128)
bool block_local_mma_supported(const skv_problem& pb);
skv_status launch_block_local_fwd_mma(const skv_problem& pb, const void* q, const void* kb, const void* vb, float* o,
                                      float* lse, const skv_host::Ctx& c);
skv_status launch_block_local_bwd_mma(const skv_problem& pb, const void* q, const void* kb, const void* vb,
                                      const void* o, const float* lse, const void* dO, float* dq, float* dkb,
                                      float* dvb, const skv_host::Ctx& c);
// block-local term of the mask (each block over its own B keys), CUDA cores
bool block_local_supported(const skv_problem& pb);
skv_status launch_block_local_fwd(const skv_problem& pb, const void* q, const void* kb, const void* vb, float* o,
                                  float* lse, const skv_host::Ctx& c);
skv_status launch_block_local_bwd(const skv_problem& pb, const void* q, const void* kb, const void* vb, const void* o,
                                  const float* lse, const void* dO, float* dq, float* dkb, float* dvb,
                                  const skv_host::Ctx& c);

}  // namespace skv_internal
