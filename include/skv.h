/*
 * skv.h -- C ABI of libskv, the GB300 (sm_103a) Split-KV anchor-attention path.
 *
 * Method: "Split-KV: Efficient Context Parallelism for Training Diffusion
 * Drafters" (Zhang, Zhang, Xie, Fan, You), cited as [Split-KV ...].
 *
 * The path, per training step: price the context chunks (Eq. 6), balance them
 * over P virtual ranks with cost-aware LPT (§4.2), compute every rank's local
 * partial attention (o_p, l_p) (Eq. 3, Alg. 1), merge the partials
 * exactly (Eq. 4) and run the backward (Alg. 1's backward),
 * all on one GPU: the P ranks are a sweep over key/value chunks, and the
 * collectives of Alg. 1 become on-device passes.
 *
 * Conventions shared by every call
 *  - Pointers named "device" point to GPU global memory owned by the caller;
 *    the library never allocates, frees or keeps a pointer after a call
 *    returns.  Host pointers (the skv_problem struct itself) are read during
 *    the call only.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call is
 *    asynchronous on that stream; outputs are valid once the stream reaches
 *    the call.
 *  - Scalar arguments are validated on the host before any launch: a bad one
 *    returns SKV_ERR_INVALID_ARG or SKV_ERR_UNSUPPORTED and launches nothing.
 *  - Anchor metadata is checked on the device (skv_chunk_costs): violations
 *    raise SKV_ERR_BAD_ANCHORS in the per-process device status word, read by
 *    skv_stream_status.  Kernels clamp every index they derive from anchors,
 *    so bad metadata yields wrong numbers, never an out-of-bounds access.
 *  - Layouts are row-major.  Query tensors are [Q][H][d] (Q = n_blocks * B),
 *    context tensors [S][Hkv][d] (Hkv = H without grouped queries); query row r
 *    belongs to block floor(r / B).
 */
#ifndef SKV_H_
#define SKV_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SKV_API __attribute__((visibility("default")))
#else
#define SKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum skv_status {
    SKV_OK = 0,
    SKV_ERR_INVALID_ARG = 1,   /* a scalar or pointer argument is invalid */
    SKV_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. head_dim) */
    SKV_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
    SKV_ERR_TIMEOUT = 4,       /* a bounded on-device wait ran out (device status) */
    SKV_ERR_BAD_ANCHORS = 5,   /* anchor metadata violates 0 <= s_i <= a_i <= S (device status) */
    SKV_ERR_WORKSPACE = 6      /* workspace pointer NULL/misaligned or smaller than skv_workspace_bytes */
} skv_status;

typedef enum skv_dtype {
    SKV_FP32 = 0,              /* float */
    SKV_BF16 = 1               /* bfloat16 (IEEE-754 binary32 upper half) */
} skv_dtype;

/*
 * One anchor-attention problem [Split-KV §3.1, Fig. 1; §4.2].
 * Block i (rows [i*B, (i+1)*B)) attends exactly the context keys
 * s_i <= x < a_i.  The context [0, S) is cut into S/m chunks
 * [j*m, (j+1)*m); P virtual ranks hold J chunks each (P*J*m == S).
 * With grouped-query attention (the drafters of Table 2: 32 query heads over
 * 4 or 8 key/value heads) k, v, dk, dv and the block-local k_blk, v_blk,
 * dk_blk, dv_blk have Hkv heads in place of H.
 */
typedef struct skv_problem {
    int32_t B;            /* block size: query rows per anchor, 1..128        */
    int32_t n_blocks;     /* N (>= 0); Q = N*B query rows                      */
    int32_t n_heads;      /* H >= 1                                            */
    int32_t head_dim;     /* d in {64, 128}                                    */
    int64_t S;            /* packed context length >= 1                        */
    int32_t m;            /* chunk length >= 1 (attention: a multiple of 128)  */
    int32_t P;            /* virtual ranks >= 1                                */
    int32_t J;            /* chunks per rank; P*J*m must equal S               */
    const int32_t* s;     /* device [N]: sample start of block i               */
    const int32_t* a;     /* device [N]: anchor of block i, s_i <= a_i <= S    */
    skv_dtype dtype;      /* dtype of q, k, v, o (merged) and dO               */
    float scale;          /* softmax scale; 0 selects 1/sqrt(head_dim)         */
    int32_t n_kv_heads;   /* Hkv: heads of k, v (and dk, dv); 0 selects H.     */
                          /* Grouped-query layout [Table 2]: H % Hkv == 0 and  */
                          /* query head h reads key/value head h / (H / Hkv)   */
} skv_problem;

/*
 * Chunk prices, [Split-KV §4.2, Eq. 6]:
 *   costs[j] = B * sum_i (min(a_i, j*m + m) - max(s_i, j*m))^+ ,  j < S/m.
 * costs: device int64[S/m], written.  Exact integer arithmetic.  Also checks
 * 0 <= s_i <= a_i <= S for every block (SKV_ERR_BAD_ANCHORS in the device
 * status word; offending blocks are clamped into range before pricing).
 */
SKV_API skv_status skv_chunk_costs(const skv_problem* prob, int64_t* costs, void* stream);

/*
 * Cost-aware LPT [Split-KV §4.2 "Cost-aware LPT"]: chunks are taken in order of
 * (cost descending, chunk index ascending); each goes to the rank with the
 * smallest (load, rank index) among ranks holding fewer than J chunks.  The
 * final locality matching is the identity (bundle p is rank p).
 *   costs         device int64[n_chunks], read (n_chunks == P*J <= 16384,
 *                 P <= 1024; larger plans return SKV_ERR_UNSUPPORTED)
 *   rank_of_chunk device int32[n_chunks], written: rank of chunk j
 *   order         device int32[n_chunks], written: rank-major chunk lists,
 *                 order[p*J .. p*J+J) are rank p's chunks in assignment order
 *   load          device int64[P], written: C_p = sum of its chunks' costs
 * Exact integer arithmetic; one thread block.
 */
SKV_API skv_status skv_lpt_order(const int64_t* costs, int32_t n_chunks, int32_t P, int32_t J,
                         int32_t* rank_of_chunk, int32_t* order, int64_t* load, void* stream);

/*
 * "No balance" baseline [Split-KV §5.1 Baselines]: chunk j goes to rank j / J.
 * Same outputs as skv_lpt_order; costs may be NULL, in which case load may be
 * NULL too (otherwise load[p] = sum of rank p's costs).
 */
SKV_API skv_status skv_contiguous_order(const int64_t* costs, int32_t n_chunks, int32_t P, int32_t J,
                                int32_t* rank_of_chunk, int32_t* order, int64_t* load,
                                void* stream);

/*
 * Zigzag baseline [Split-KV §4.2 "A concrete example", Fig. 5b]: every sample of
 * length L is cut into 2P chunks of L/(2P) positions; rank p receives chunks p
 * and 2P-1-p of each sample.  Returns per-rank context loads C_p only (Zigzag
 * chunks are not the m-sized chunks the attention kernels consume).
 *   sample_start, sample_len  device int32[n_samples]; every sample_len must be
 *                             a multiple of 2P and the samples must lie in [0, S)
 *   load                      device int64[P], written
 */
SKV_API skv_status skv_zigzag_loads(const skv_problem* prob, const int32_t* sample_start,
                            const int32_t* sample_len, int32_t n_samples,
                            int64_t* load, void* stream);

/*
 * Workspace size in bytes of skv_attn_fwd (which = 0) or skv_attn_bwd
 * (which = 1) for this problem; 0 if the problem is invalid.  The caller
 * allocates it (256-byte aligned) and may reuse it across calls on one stream.
 */
SKV_API size_t skv_workspace_bytes(const skv_problem* prob, int which);

/*
 * Local partial attention of every virtual rank [Split-KV §4.1, Eq. 3;
 * the per-rank attention of Alg. 1]: for each rank p, each query row r and head h,
 *   z_x = scale * q_r . k_x  over the keys x in K_p with s_i <= x < a_i,
 *   lse_part[p][r][h] = log sum_x exp(z_x)          (natural log)
 *   o_part[p][r][h][:] = sum_x exp(z_x - lse) v_x
 * K_p is the union of the chunks whose rank_of_chunk equals p (any map into
 * [0, P) is accepted; entries outside it are ignored and flag
 * SKV_ERR_INVALID_ARG in the device status word).  Rows with no visible key in
 * K_p get lse_part = -inf; their o_part row is unspecified (never read by
 * skv_lse_merge).
 *   q             device [Q][H][d], dtype prob->dtype
 *   k, v          device [S][Hkv][d], dtype prob->dtype; rows 16-byte aligned
 *   rank_of_chunk device int32[S/m]
 *   o_part        device float[P][Q][H][d], written
 *   lse_part      device float[P][Q][H], written
 *   workspace     device, >= skv_workspace_bytes(prob, 0) bytes
 * bf16 problems run on the tcgen05 tensor cores (bf16 products, fp32
 * accumulation); fp32 problems run an fp32 CUDA-core kernel.
 */
SKV_API skv_status skv_attn_fwd(const skv_problem* prob, const void* q, const void* k, const void* v,
                        const int32_t* rank_of_chunk, float* o_part, float* lse_part,
                        void* workspace, size_t ws_bytes, void* stream);

/*
 * skv_attn_fwd without a workspace argument, for callers that may not
 * allocate device memory (a plug-in whose host framework owns the whole device
 * memory pool, a latency-critical loop that cannot afford a cudaMalloc that may
 * synchronise the device, a runtime held to a fixed memory budget).  The paper
 * has no counterpart to this call; it is a packaging of skv_attn_fwd.
 *
 * Same arguments, semantics and outputs as skv_attn_fwd.  The scratch the
 * forward needs (the per-rank chunk lists, 4 bytes per chunk and per rank, and
 * the key bounds of each query tile, 16 bytes each, counted only for bf16
 * problems, whose tensor-core forward uses them; a tile is 128 query rows, or
 * 128/g rows of each of the g query heads of a key/value head with grouped
 * queries) lives in a fixed 128 KiB array in device memory that every GPU
 * loading the library holds until the process exits; the call itself
 * allocates nothing.  Problems whose forward workspace
 * (skv_workspace_bytes(prob, 0)) exceeds 131072 bytes are rejected with
 * SKV_ERR_WORKSPACE before any launch -- e.g. 16384 chunks over 1024 ranks
 * with up to 3800 query tiles (Q <= 486 400 rows without grouped queries) fit.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  All calls share the one array, and each call rewrites the lists
 * before reading them (nothing in it has to start at zero), so calls that
 * overlap on the GPU (on different streams, or from different host threads
 * without ordering) race and must be serialised by the caller.  The address is
 * kept for the life of the process, like the status word's: do not use the
 * library across cudaDeviceReset of a device it has run on.
 */
SKV_API skv_status skv_attn_fwd_static(const skv_problem* prob, const void* q, const void* k, const void* v,
                                       const int32_t* rank_of_chunk, float* o_part, float* lse_part,
                                       void* stream);

/*
 * Exact LSE merge of P disjoint partials [Split-KV §4.1, Eq. 4; the merge step of Alg. 1]:
 *   lse[r] = log sum_p exp(lse_part[p][r]),
 *   o[r][:] = sum_p exp(lse_part[p][r] - lse[r]) * o_part[p][r][:].
 * Partials with lse_part = -inf are skipped (their o_part row is not read);
 * a row whose partials are all -inf gets o = 0, lse = -inf.
 *   o_part   device float[P][rows][head_dim]  (rows = Q*H for attention)
 *   lse_part device float[P][rows]
 *   o        device [rows][head_dim] of o_dtype, written (bf16: round to nearest even)
 *   lse      device float[rows], written (may be NULL)
 * head_dim must be a multiple of 4 (<= 256); o_part 16-byte aligned.
 */
SKV_API skv_status skv_lse_merge(const float* o_part, const float* lse_part, int32_t P, int64_t rows,
                         int32_t head_dim, void* o, skv_dtype o_dtype, float* lse, void* stream);

/*
 * The merge fused with the output projection [Split-KV §4.1, Eq. 5; the
 * MERGE_AR, OProj and RS_sum steps of Alg. 1's forward]: with the merge
 * weights w_p = exp(lse_part[p] - lse) of Eq. 4 and OProj(x) = x W_o^T over the
 * concatenated heads,
 *   y = sum_p OProj(w_p o_part[p]) = OProj(o),   o = sum_p w_p o_part[p].
 * The sum is linear, so it is taken before the projection: o and lse are
 * written exactly as skv_lse_merge writes them (o in bf16), then a tensor-core
 * GEMM computes y = o W_o^T from the bf16 o (fp32 accumulation).
 *   o_part   device float[P][Q][n_heads][head_dim]
 *   lse_part device float[P][Q][n_heads]
 *   w_o      device bf16 [d_model][n_heads*head_dim], row-major (the projection's
 *            weight; caller-owned)
 *   o        device bf16 [Q][n_heads][head_dim], written (the merged output,
 *            which the backward reads); 16-byte aligned
 *   lse      device float[Q][n_heads], written (may be NULL)
 *   y        device float[Q][d_model], written
 * head_dim in {64, 128, 256}; d_model a multiple of 16; w_o, o, y and o_part
 * 16-byte aligned.  Rows whose partials are all empty get o = 0 and add
 * nothing to y.  Errors: SKV_ERR_INVALID_ARG / SKV_ERR_UNSUPPORTED before any
 * launch; SKV_ERR_TIMEOUT through skv_stream_status.
 */
SKV_API skv_status skv_lse_merge_oproj(const float* o_part, const float* lse_part, int32_t P, int64_t Q,
                                       int32_t n_heads, int32_t head_dim, const void* w_o, int32_t d_model,
                                       void* o, float* lse, float* y, void* stream);

/*
 * Backward of the exact LSE merge, per partial [Split-KV §4.1, Eq. 4; the
 * MERGE_BWD step of Alg. 1's backward]: for upstream gradients dO (of o) and
 * dlse (of lse), with the merged lse and o of skv_lse_merge,
 * w_p = exp(lse_part[p][r] - lse[r]) and D_p = dO[r] . o_part[p][r]:
 *   do_part[p][r][:] = w_p * dO[r][:],
 *   dlse_part[p][r]  = w_p * (D_p - dO[r] . o[r] + dlse[r]),
 * where dO . o = sum_p w_p D_p is formed from the same partials (the merged o is
 * not an input, so a rounded copy of it plays no part) and lse is recomputed from
 * lse_part.  This is the per-rank route a multi-GPU build takes (each rank owns
 * its partial; sum_p w_p D_p is that route's all-reduce); on one GPU
 * skv_attn_bwd uses the equivalent merged form instead.  Partials with
 * lse_part = -inf get do_part = 0 and dlse_part = 0 (their o_part is not read).
 *   o_part, lse_part  as for skv_lse_merge (o_part 16-byte aligned)
 *   dO         device [rows][head_dim] of do_dtype (fp32: 16-byte, bf16: 8-byte aligned)
 *   dlse       device float[rows], or NULL for a zero gradient
 *   do_part    device float[P][rows][head_dim], written (16-byte aligned), or NULL to skip
 *   dlse_part  device float[P][rows], written
 * head_dim as for skv_lse_merge.  Errors: SKV_ERR_INVALID_ARG for P < 1,
 * rows < 0, a bad dtype or a missing/misaligned pointer; SKV_ERR_UNSUPPORTED
 * for another head_dim.  Nothing is written on an error.
 */
SKV_API skv_status skv_lse_merge_bwd(const float* o_part, const float* lse_part, int32_t P, int64_t rows,
                                     int32_t head_dim, const void* dO, skv_dtype do_dtype, const float* dlse,
                                     float* do_part, float* dlse_part, void* stream);

/*
 * Backward of the merged attention for L = sum(dO * o), lse receiving no
 * gradient [Split-KV Alg. 1's backward]: each virtual rank p produces dq^(p)
 * and the dk_p, dv_p rows of its own chunks (the keys it holds); dq is the sum
 * of the dq^(p) over ranks (Alg. 1's dq reduce-scatter, made local).  The per-rank
 * MERGE_BWD of Alg. 1 is taken in its merged form: with
 * D_r = dO_r . o_r and the global lse, the score gradient on rank p is
 * P_rx (dO_r . v_x - D_r) with P_rx = exp(z_rx - lse_r), which equals the
 * per-rank route exactly.
 *   q, dO     device [Q][H][d], dtype prob->dtype
 *   k, v      device [S][Hkv][d], dtype prob->dtype
 *   o         device [Q][H][d], dtype prob->dtype (the merged output)
 *   lse       device float[Q][H] (the merged log-sum-exp, natural log)
 *   dq        device float[Q][H][d], written
 *   dk, dv    device float[S][Hkv][d], written (keys no query sees get 0; a
 *             key/value head sums the gradients of its query heads)
 *   workspace device, >= skv_workspace_bytes(prob, 1) bytes
 */
SKV_API skv_status skv_attn_bwd(const skv_problem* prob, const void* q, const void* k, const void* v,
                        const void* o, const float* lse, const void* dO,
                        const int32_t* rank_of_chunk, float* dq, float* dk, float* dv,
                        void* workspace, size_t ws_bytes, void* stream);

/*
 * Block-local term of the anchor mask [Split-KV §3.1, Fig. 1 caption]: besides
 * its context window W_i, each block's B tokens attend bidirectionally to one
 * another.  Their keys and values (the block tokens' own projections) are
 * given laid out like q.  The term is one more key set, disjoint from every
 * context chunk, so its result is one more partial of Eq. 4: write it after
 * the P rank partials (o_loc = o_part + P*Q*H*d, lse_loc = lse_part + P*Q*H)
 * and merge P + 1 partials with skv_lse_merge to get the whole mask.
 *   q                device [Q][H][d], dtype prob->dtype (Q = n_blocks * B)
 *   k_blk, v_blk     device [Q][Hkv][d], dtype prob->dtype
 *   o_loc            device float[Q][H][d], written
 *   lse_loc          device float[Q][H], written (natural log)
 * prob->B <= 32 and head_dim 64 or 128, else SKV_ERR_UNSUPPORTED; the anchor
 * fields are not read.  Pointers 16-byte aligned (lse 4), else INVALID_ARG.
 */
SKV_API skv_status skv_block_local_fwd(const skv_problem* prob, const void* q, const void* k_blk, const void* v_blk,
                                       float* o_loc, float* lse_loc, void* stream);

/*
 * Backward of the block-local term for L = sum(dO * o) of the whole mask,
 * with o and lse the MERGED results (context ranks + this term), the same
 * merged form as skv_attn_bwd [Alg. 1's MERGE_BWD]: P = exp(z - lse), D = dO . o,
 * dS = P (dP - D).
 *   o                device [Q][H][d], dtype prob->dtype; lse device float[Q][H]
 *   dq               device float[Q][H][d], ACCUMULATED: call after
 *                    skv_attn_bwd (which writes the context part) on the same
 *                    stream, and dq holds the whole-mask gradient
 *   dk_blk, dv_blk   device float[Q][Hkv][d], written (summed over each key/value
 *                    head's query heads)
 */
SKV_API skv_status skv_block_local_bwd(const skv_problem* prob, const void* q, const void* k_blk, const void* v_blk,
                                       const void* o, const float* lse, const void* dO, float* dq, float* dk_blk,
                                       float* dv_blk, void* stream);

/*
 * Synchronises `stream`, then returns and clears the device status word of
 * the current device (SKV_ERR_BAD_ANCHORS, SKV_ERR_TIMEOUT, SKV_ERR_INVALID_ARG
 * raised by kernels), or SKV_ERR_CUDA if the stream reports a CUDA error.
 * The word is shared by all streams of the process on that device.
 */
SKV_API skv_status skv_stream_status(void* stream);

/* Static English name of a status code. */
SKV_API const char* skv_status_str(skv_status status);

/*
 * Test hook: time limit in nanoseconds (device global timer) of every bounded
 * on-device wait of the tensor-core kernels launched afterwards by this
 * process (default 2 s).  A wait that runs out sets SKV_ERR_TIMEOUT in the
 * device status word, abandons the work item and lets the kernel finish
 * cleanly.  `limit` == 0 restores the default.  `limit` < 0 is a test mode:
 * the deadline is -limit ns and every block first waits on a barrier that
 * nothing ever completes, so the timeout path runs deterministically.
 */
SKV_API skv_status skv_set_wait_limit(int64_t limit);

/*
 * Number of kernels this library has launched in the process so far (all
 * devices, all streams; host-side counter, incremented per launch).
 */
SKV_API uint64_t skv_launch_count(void);

/*
 * Measurement hook.  skv_set_kernel_timing(1) makes the library record a
 * CUDA event pair on the launching stream around each of its main kernels:
 * slot 0 the forward attention kernel, 1 the LSE merge, 2 the backward dK/dV
 * kernel, 3 the backward dQ kernel (tensor-core path), 4 and 5 the
 * block-local forward and backward, 6 the output-projection GEMM.  skv_kernel_times
 * waits for the last recorded pair of each of the first n slots and writes
 * its duration in milliseconds (-1 where nothing was recorded since the
 * previous read).  Off by default; the events are created on first use.
 */
SKV_API skv_status skv_set_kernel_timing(int enable);
SKV_API skv_status skv_kernel_times(float* ms, int n);

#ifdef __cplusplus
}
#endif
#endif /* SKV_H_ */
