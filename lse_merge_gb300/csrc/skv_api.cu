// C-ABI entry points of libskv: argument validation, workspace layout, the
// device status word and dispatch to the kernels.  See include/skv.h.
#include <math.h>

#include <atomic>
#include <mutex>

#include "skv_common.cuh"
#include "skv_internal.h"
#include "skv_tc.h"

// Device status word (one per device that loads the library).  Host code only
// ever uses the address returned by cudaGetSymbolAddress.
__device__ int g_skv_status;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_status_ptr[kMaxDevices] = {nullptr};
int g_num_sms[kMaxDevices] = {0};
long long g_wait_limit = 0;   // 0 = default
std::atomic<uint64_t> g_launches{0};

bool bad_ptr(const void* p, size_t align) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) % align) != 0; }

skv_status validate(const skv_problem* pb, bool attention) {
    if (!pb) return SKV_ERR_INVALID_ARG;
    if (pb->B < 1 || pb->B > 128 || pb->n_blocks < 0 || pb->n_heads < 1 || pb->S < 1 || pb->m < 1 ||
        pb->P < 1 || pb->J < 1)
        return SKV_ERR_INVALID_ARG;
    if (int64_t(pb->P) * pb->J * pb->m != pb->S) return SKV_ERR_INVALID_ARG;
    if (pb->S / pb->m > 0x7fffffffLL) return SKV_ERR_INVALID_ARG;
    if (int64_t(pb->n_blocks) * pb->B > 0x7fffffffLL) return SKV_ERR_INVALID_ARG;
    if (pb->S > 0x7fffffffLL) return SKV_ERR_INVALID_ARG;   // anchors are int32
    if (pb->n_blocks > 0 && (pb->s == nullptr || pb->a == nullptr)) return SKV_ERR_INVALID_ARG;
    if (pb->dtype != SKV_FP32 && pb->dtype != SKV_BF16) return SKV_ERR_INVALID_ARG;
    if (!(pb->scale >= 0.f) || isinf(pb->scale)) return SKV_ERR_INVALID_ARG;
    if (pb->n_kv_heads < 0 || pb->n_kv_heads > pb->n_heads ||
        (pb->n_kv_heads > 0 && pb->n_heads % pb->n_kv_heads != 0))
        return SKV_ERR_INVALID_ARG;
    if (attention) {
        if (pb->head_dim != 64 && pb->head_dim != 128) return SKV_ERR_UNSUPPORTED;
        if (pb->m % 128 != 0) return SKV_ERR_UNSUPPORTED;
        if (int64_t(pb->n_heads) * pb->head_dim > 65536) return SKV_ERR_UNSUPPORTED;
    }
    return SKV_OK;
}

skv_problem normalized(const skv_problem* pb) {
    skv_problem c = *pb;
    if (c.scale == 0.f) c.scale = 1.0f / sqrtf((float)c.head_dim);
    if (c.n_kv_heads == 0) c.n_kv_heads = c.n_heads;
    return c;
}

struct FwdWs {
    int32_t* csr_ptr;
    int32_t* csr_list;
    void* tc;             // tensor-core kernel scratch
};

struct BwdWs {
    int32_t* csr_ptr;
    int32_t* csr_list;
    float* D;
    float* lse2;
    float* dq_part;
    void* tc;
};

size_t fwd_ws_layout(const skv_problem& pb, FwdWs* w, char* base) {
    using skv_host::align256;
    const int64_t n = pb.S / pb.m;
    size_t off = 0;
    const size_t o_ptr = off; off = align256(off + size_t(pb.P + 1) * 4);
    const size_t o_list = off; off = align256(off + size_t(n) * 4);
    const size_t o_tc = off; off = align256(off + skv_tc::fwd_scratch_bytes(pb));
    if (w) {
        w->csr_ptr = reinterpret_cast<int32_t*>(base + o_ptr);
        w->csr_list = reinterpret_cast<int32_t*>(base + o_list);
        w->tc = base + o_tc;
    }
    return off;
}

size_t bwd_ws_layout(const skv_problem& pb, BwdWs* w, char* base) {
    using skv_host::align256;
    const int64_t n = pb.S / pb.m;
    const int64_t rows = int64_t(pb.n_blocks) * pb.B * pb.n_heads;
    size_t off = 0;
    const size_t o_ptr = off; off = align256(off + size_t(pb.P + 1) * 4);
    const size_t o_list = off; off = align256(off + size_t(n) * 4);
    // D and lse2: row-major [Q][H], or head-major [H][Qp] padded to whole query tiles
    const int64_t Qp = ((int64_t(pb.n_blocks) * pb.B + 127) / 128) * 128;
    const int64_t drows = Qp * pb.n_heads;
    const size_t o_D = off; off = align256(off + size_t(drows) * 4);
    const size_t o_l2 = off; off = align256(off + size_t(drows) * 4);
    const bool tc = skv_tc::bwd_supported(pb);
    const size_t o_dqp = off; off = align256(off + (tc ? 0 : size_t(pb.P) * rows * pb.head_dim * 4));
    const size_t o_tc = off; off = align256(off + skv_tc::bwd_scratch_bytes(pb));
    if (w) {
        w->csr_ptr = reinterpret_cast<int32_t*>(base + o_ptr);
        w->csr_list = reinterpret_cast<int32_t*>(base + o_list);
        w->D = reinterpret_cast<float*>(base + o_D);
        w->lse2 = reinterpret_cast<float*>(base + o_l2);
        w->dq_part = reinterpret_cast<float*>(base + o_dqp);
        w->tc = base + o_tc;
    }
    return off;
}

}  // namespace

namespace skv_host {

void note_launch(int n) { g_launches.fetch_add(uint64_t(n), std::memory_order_relaxed); }

namespace {
bool g_timing = false;
cudaEvent_t g_ev[kTimeSlots][2] = {};
bool g_ev_live[kTimeSlots] = {};
}  // namespace

void timer_begin(int slot, cudaStream_t stream) {
    if (!g_timing || slot < 0 || slot >= kTimeSlots) return;
    for (int i = 0; i < 2; ++i)
        if (!g_ev[slot][i] && cudaEventCreate(&g_ev[slot][i]) != cudaSuccess) return;
    cudaEventRecord(g_ev[slot][0], stream);
}

void timer_end(int slot, cudaStream_t stream) {
    if (!g_timing || slot < 0 || slot >= kTimeSlots || !g_ev[slot][1]) return;
    cudaEventRecord(g_ev[slot][1], stream);
    g_ev_live[slot] = true;
}

skv_status get_ctx(void* stream, Ctx& ctx) {
    int dev = 0;
    SKV_CUDA_CHECK(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return SKV_ERR_UNSUPPORTED;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_status_ptr[dev]) {
            void* p = nullptr;
            SKV_CUDA_CHECK(cudaGetSymbolAddress(&p, g_skv_status));
            int sms = 0;
            SKV_CUDA_CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
            g_status_ptr[dev] = static_cast<int*>(p);
            g_num_sms[dev] = sms;
        }
        ctx.status = g_status_ptr[dev];
        ctx.num_sms = g_num_sms[dev];
        ctx.wait_limit = g_wait_limit != 0 ? g_wait_limit : 2000000000LL;   // ns (< 0: test mode)
    }
    ctx.stream = static_cast<cudaStream_t>(stream);
    return SKV_OK;
}

}  // namespace skv_host

extern "C" {

skv_status skv_chunk_costs(const skv_problem* pb, int64_t* costs, void* stream) {
    skv_status st = validate(pb, false);
    if (st != SKV_OK) return st;
    if (bad_ptr(costs, 8)) return SKV_ERR_INVALID_ARG;
    skv_host::Ctx c;
    if ((st = skv_host::get_ctx(stream, c)) != SKV_OK) return st;
    return skv_internal::launch_chunk_costs(*pb, costs, c);
}

skv_status skv_lpt_order(const int64_t* costs, int32_t n_chunks, int32_t P, int32_t J, int32_t* rank_of_chunk,
                         int32_t* order, int64_t* load, void* stream) {
    if (P < 1 || J < 1 || int64_t(P) * J != n_chunks) return SKV_ERR_INVALID_ARG;
    if (n_chunks > skv_internal::kLptMaxChunks || P > skv_internal::kLptMaxRanks) return SKV_ERR_UNSUPPORTED;
    if (bad_ptr(costs, 8) || bad_ptr(rank_of_chunk, 4) || bad_ptr(order, 4) || bad_ptr(load, 8))
        return SKV_ERR_INVALID_ARG;
    skv_host::Ctx c;
    skv_status st = skv_host::get_ctx(stream, c);
    if (st != SKV_OK) return st;
    return skv_internal::launch_lpt(costs, n_chunks, P, J, rank_of_chunk, order, load, c);
}

skv_status skv_contiguous_order(const int64_t* costs, int32_t n_chunks, int32_t P, int32_t J,
                                int32_t* rank_of_chunk, int32_t* order, int64_t* load, void* stream) {
    if (P < 1 || J < 1 || int64_t(P) * J != n_chunks) return SKV_ERR_INVALID_ARG;
    if (bad_ptr(rank_of_chunk, 4) || bad_ptr(order, 4)) return SKV_ERR_INVALID_ARG;
    if (costs && bad_ptr(load, 8)) return SKV_ERR_INVALID_ARG;
    skv_host::Ctx c;
    skv_status st = skv_host::get_ctx(stream, c);
    if (st != SKV_OK) return st;
    return skv_internal::launch_contiguous(costs, n_chunks, P, J, rank_of_chunk, order, costs ? load : nullptr, c);
}

skv_status skv_zigzag_loads(const skv_problem* pb, const int32_t* sample_start, const int32_t* sample_len,
                            int32_t n_samples, int64_t* load, void* stream) {
    skv_status st = validate(pb, false);
    if (st != SKV_OK) return st;
    if (n_samples < 1 || bad_ptr(sample_start, 4) || bad_ptr(sample_len, 4) || bad_ptr(load, 8))
        return SKV_ERR_INVALID_ARG;
    skv_host::Ctx c;
    if ((st = skv_host::get_ctx(stream, c)) != SKV_OK) return st;
    return skv_internal::launch_zigzag(*pb, sample_start, sample_len, n_samples, load, c);
}

size_t skv_workspace_bytes(const skv_problem* pb, int which) {
    if (validate(pb, true) != SKV_OK) return 0;
    const skv_problem p = normalized(pb);
    if (which == 0) return fwd_ws_layout(p, nullptr, nullptr);
    if (which == 1) return bwd_ws_layout(p, nullptr, nullptr);
    return 0;
}

skv_status skv_attn_fwd(const skv_problem* pb_in, const void* q, const void* k, const void* v,
                        const int32_t* rank_of_chunk, float* o_part, float* lse_part, void* workspace,
                        size_t ws_bytes, void* stream) {
    skv_status st = validate(pb_in, true);
    if (st != SKV_OK) return st;
    const skv_problem pb = normalized(pb_in);
    const size_t need = fwd_ws_layout(pb, nullptr, nullptr);
    if (ws_bytes < need || bad_ptr(workspace, 256)) return SKV_ERR_WORKSPACE;
    if (pb.n_blocks > 0 && (bad_ptr(q, 16) || bad_ptr(k, 16) || bad_ptr(v, 16) || bad_ptr(o_part, 16) ||
                            bad_ptr(lse_part, 4) || bad_ptr(rank_of_chunk, 4)))
        return SKV_ERR_INVALID_ARG;
    if (pb.n_blocks == 0) return SKV_OK;
    skv_host::Ctx c;
    if ((st = skv_host::get_ctx(stream, c)) != SKV_OK) return st;
    FwdWs w;
    fwd_ws_layout(pb, &w, static_cast<char*>(workspace));
    const int n = (int)(pb.S / pb.m);
    if ((st = skv_internal::launch_rank_csr(rank_of_chunk, n, pb.P, w.csr_ptr, w.csr_list, c)) != SKV_OK) return st;
    skv::RankCSR csr{w.csr_ptr, w.csr_list};
    if (skv_tc::fwd_supported(pb))
        return skv_tc::launch_attn_fwd_tc(pb, q, k, v, csr, o_part, lse_part, w.tc, c);
    return skv_internal::launch_attn_fwd_simt(pb, q, k, v, csr, o_part, lse_part, c);
}

skv_status skv_lse_merge(const float* o_part, const float* lse_part, int32_t P, int64_t rows, int32_t head_dim,
                         void* o, skv_dtype o_dtype, float* lse, void* stream) {
    if (P < 1 || rows < 0) return SKV_ERR_INVALID_ARG;
    if (o_dtype != SKV_FP32 && o_dtype != SKV_BF16) return SKV_ERR_INVALID_ARG;
    switch (head_dim) {
        case 4: case 8: case 16: case 32: case 64: case 128: case 256: break;
        default: return SKV_ERR_UNSUPPORTED;
    }
    if (rows == 0) return SKV_OK;
    if (bad_ptr(o_part, 16) || bad_ptr(lse_part, 4) || bad_ptr(o, o_dtype == SKV_BF16 ? 8 : 16) ||
        (lse && bad_ptr(lse, 4)))
        return SKV_ERR_INVALID_ARG;
    skv_host::Ctx c;
    skv_status st = skv_host::get_ctx(stream, c);
    if (st != SKV_OK) return st;
    return skv_internal::launch_merge(o_part, lse_part, P, rows, head_dim, o, o_dtype, lse, c);
}

skv_status skv_lse_merge_oproj(const float* o_part, const float* lse_part, int32_t P, int64_t Q, int32_t n_heads,
                              int32_t head_dim, const void* w_o, int32_t d_model, void* o, float* lse, float* y,
                              void* stream) {
    if (P < 1 || Q < 0 || n_heads < 1 || d_model < 16 || d_model % 16 != 0) return SKV_ERR_INVALID_ARG;
    switch (head_dim) {
        case 64: case 128: case 256: break;
        default: return SKV_ERR_UNSUPPORTED;
    }
    const int64_t hd = int64_t(n_heads) * head_dim;
    if (hd > 65536 || d_model > 65536 || Q > 0x7fffffffLL) return SKV_ERR_UNSUPPORTED;
    if (Q == 0) return SKV_OK;
    if (bad_ptr(o_part, 16) || bad_ptr(lse_part, 4) || bad_ptr(w_o, 16) || bad_ptr(o, 16) || bad_ptr(y, 16) ||
        (lse && bad_ptr(lse, 4)))
        return SKV_ERR_INVALID_ARG;
    skv_host::Ctx c;
    skv_status st = skv_host::get_ctx(stream, c);
    if (st != SKV_OK) return st;
    // Eq. 4 over the partials into o (bf16), then Eq. 5's projection of the sum
    if ((st = skv_internal::launch_merge(o_part, lse_part, P, Q * n_heads, head_dim, o, SKV_BF16, lse, c)) != SKV_OK)
        return st;
    return skv_internal::launch_oproj(o, Q, (int)hd, w_o, d_model, y, c);
}

skv_status skv_lse_merge_bwd(const float* o_part, const float* lse_part, int32_t P, int64_t rows,
                             int32_t head_dim, const void* dO, skv_dtype do_dtype, const float* dlse, float* do_part,
                             float* dlse_part, void* stream) {
    if (P < 1 || rows < 0) return SKV_ERR_INVALID_ARG;
    if (do_dtype != SKV_FP32 && do_dtype != SKV_BF16) return SKV_ERR_INVALID_ARG;
    switch (head_dim) {
        case 4: case 8: case 16: case 32: case 64: case 128: case 256: break;
        default: return SKV_ERR_UNSUPPORTED;
    }
    if (rows == 0) return SKV_OK;
    if (bad_ptr(o_part, 16) || bad_ptr(lse_part, 4) || bad_ptr(dO, do_dtype == SKV_BF16 ? 8 : 16) ||
        bad_ptr(dlse_part, 4) || (dlse && bad_ptr(dlse, 4)) || (do_part && bad_ptr(do_part, 16)))
        return SKV_ERR_INVALID_ARG;
    skv_host::Ctx c;
    skv_status st = skv_host::get_ctx(stream, c);
    if (st != SKV_OK) return st;
    return skv_internal::launch_merge_bwd(o_part, lse_part, P, rows, head_dim, dO, do_dtype, dlse, do_part,
                                          dlse_part, c);
}

skv_status skv_attn_bwd(const skv_problem* pb_in, const void* q, const void* k, const void* v, const void* o,
                        const float* lse, const void* dO, const int32_t* rank_of_chunk, float* dq, float* dk,
                        float* dv, void* workspace, size_t ws_bytes, void* stream) {
    skv_status st = validate(pb_in, true);
    if (st != SKV_OK) return st;
    const skv_problem pb = normalized(pb_in);
    const size_t need = bwd_ws_layout(pb, nullptr, nullptr);
    if (ws_bytes < need || bad_ptr(workspace, 256)) return SKV_ERR_WORKSPACE;
    const int64_t rows = int64_t(pb.n_blocks) * pb.B * pb.n_heads;
    if (bad_ptr(k, 16) || bad_ptr(v, 16) || bad_ptr(dk, 16) || bad_ptr(dv, 16)) return SKV_ERR_INVALID_ARG;
    if (rows > 0 && (bad_ptr(q, 16) || bad_ptr(o, 16) || bad_ptr(dO, 16) || bad_ptr(lse, 4) || bad_ptr(dq, 16) ||
                     bad_ptr(rank_of_chunk, 4)))
        return SKV_ERR_INVALID_ARG;
    skv_host::Ctx c;
    if ((st = skv_host::get_ctx(stream, c)) != SKV_OK) return st;
    const int64_t kv_elems = pb.S * pb.n_kv_heads * pb.head_dim;
    const bool tc = skv_tc::bwd_supported(pb);
    if (rows == 0 || !tc) {   // the tensor-core kernel writes every dk/dv row itself
        if ((st = skv_internal::launch_zero(dk, kv_elems, c)) != SKV_OK) return st;
        if ((st = skv_internal::launch_zero(dv, kv_elems, c)) != SKV_OK) return st;
    }
    if (rows == 0) return SKV_OK;
    BwdWs w;
    bwd_ws_layout(pb, &w, static_cast<char*>(workspace));
    const int n = (int)(pb.S / pb.m);
    const int64_t Qn = int64_t(pb.n_blocks) * pb.B;
    const int64_t Qp = tc ? ((Qn + 127) / 128) * 128 : Qn;
    if ((st = skv_internal::launch_bwd_prep(o, dO, lse, pb.dtype, Qn, Qp, pb.n_heads, pb.head_dim, tc, w.D, w.lse2,
                                            c)) != SKV_OK)
        return st;
    if ((st = skv_internal::launch_rank_csr(rank_of_chunk, n, pb.P, w.csr_ptr, w.csr_list, c)) != SKV_OK) return st;
    skv::RankCSR csr{w.csr_ptr, w.csr_list};
    if (tc)   // dk_p, dv_p per key tile; dq = sum_p dq^(p) accumulated rank by rank per query tile
        return skv_tc::launch_attn_bwd_tc(pb, q, k, v, dO, w.lse2, w.D, csr, dq, dk, dv, w.tc, c);
    if ((st = skv_internal::launch_attn_bwd_simt(pb, q, k, v, dO, lse, w.D, csr, w.dq_part, dk, dv, c)) != SKV_OK)
        return st;
    return skv_internal::launch_dq_sum(w.dq_part, pb.P, rows, pb.head_dim, dq, c);
}

skv_status skv_block_local_fwd(const skv_problem* pb_in, const void* q, const void* k_blk, const void* v_blk,
                               float* o_loc, float* lse_loc, void* stream) {
    skv_status st = validate(pb_in, false);
    if (st != SKV_OK) return st;
    if (pb_in->head_dim != 64 && pb_in->head_dim != 128) return SKV_ERR_UNSUPPORTED;
    const skv_problem pb = normalized(pb_in);
    if (!skv_internal::block_local_supported(pb)) return SKV_ERR_UNSUPPORTED;
    if (pb.n_blocks == 0) return SKV_OK;
    if (bad_ptr(q, 16) || bad_ptr(k_blk, 16) || bad_ptr(v_blk, 16) || bad_ptr(o_loc, 16) || bad_ptr(lse_loc, 4))
        return SKV_ERR_INVALID_ARG;
    skv_host::Ctx c;
    if ((st = skv_host::get_ctx(stream, c)) != SKV_OK) return st;
    return skv_internal::launch_block_local_fwd(pb, q, k_blk, v_blk, o_loc, lse_loc, c);
}

skv_status skv_block_local_bwd(const skv_problem* pb_in, const void* q, const void* k_blk, const void* v_blk,
                               const void* o, const float* lse, const void* dO, float* dq, float* dk_blk,
                               float* dv_blk, void* stream) {
    skv_status st = validate(pb_in, false);
    if (st != SKV_OK) return st;
    if (pb_in->head_dim != 64 && pb_in->head_dim != 128) return SKV_ERR_UNSUPPORTED;
    const skv_problem pb = normalized(pb_in);
    if (!skv_internal::block_local_supported(pb)) return SKV_ERR_UNSUPPORTED;
    if (pb.n_blocks == 0) return SKV_OK;
    if (bad_ptr(q, 16) || bad_ptr(k_blk, 16) || bad_ptr(v_blk, 16) || bad_ptr(o, 16) || bad_ptr(lse, 4) ||
        bad_ptr(dO, 16) || bad_ptr(dq, 16) || bad_ptr(dk_blk, 16) || bad_ptr(dv_blk, 16))
        return SKV_ERR_INVALID_ARG;
    skv_host::Ctx c;
    if ((st = skv_host::get_ctx(stream, c)) != SKV_OK) return st;
    return skv_internal::launch_block_local_bwd(pb, q, k_blk, v_blk, o, lse, dO, dq, dk_blk, dv_blk, c);
}

skv_status skv_stream_status(void* stream) {
    skv_host::Ctx c;
    skv_status st = skv_host::get_ctx(stream, c);
    if (st != SKV_OK) return st;
    if (cudaStreamSynchronize(c.stream) != cudaSuccess) return SKV_ERR_CUDA;
    int h = 0;
    if (cudaMemcpy(&h, c.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SKV_ERR_CUDA;
    if (h != 0) {
        const int zero = 0;
        if (cudaMemcpy(c.status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return SKV_ERR_CUDA;
    }
    return static_cast<skv_status>(h);
}

const char* skv_status_str(skv_status s) {
    switch (s) {
        case SKV_OK: return "ok";
        case SKV_ERR_INVALID_ARG: return "invalid argument";
        case SKV_ERR_UNSUPPORTED: return "unsupported configuration";
        case SKV_ERR_CUDA: return "CUDA error";
        case SKV_ERR_TIMEOUT: return "bounded device wait timed out";
        case SKV_ERR_BAD_ANCHORS: return "anchor metadata out of range";
        case SKV_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    }
    return "unknown status";
}

uint64_t skv_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

skv_status skv_set_kernel_timing(int enable) {
    skv_host::g_timing = enable != 0;
    return SKV_OK;
}

skv_status skv_kernel_times(float* ms, int n) {
    if (!ms || n < 0) return SKV_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        ms[i] = -1.f;
        if (i >= skv_host::kTimeSlots || !skv_host::g_ev_live[i]) continue;
        if (cudaEventSynchronize(skv_host::g_ev[i][1]) != cudaSuccess) return SKV_ERR_CUDA;
        if (cudaEventElapsedTime(&ms[i], skv_host::g_ev[i][0], skv_host::g_ev[i][1]) != cudaSuccess)
            return SKV_ERR_CUDA;
        skv_host::g_ev_live[i] = false;
    }
    return SKV_OK;
}

skv_status skv_set_wait_limit(int64_t limit) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_wait_limit = limit;
    return SKV_OK;
}

}  // extern "C"
