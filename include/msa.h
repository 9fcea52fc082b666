/*
 * msa.h -- C ABI of the MSA (MiniMax Sparse Attention) training hot path on GB300.
 *
 * The method (MiniMax Sparse Attention summary, 7minutos.es, "¿Qué es MSA?" and
 * "Cómo funcionan las dos ramas"): an index branch -- one index-query head per GQA
 * group and one shared index-key head -- scores the causally visible keys,
 * max-pools the scores to Bk-token blocks and keeps the k best blocks per query and
 * group, the query's own block always included; a main branch runs exact softmax
 * attention of every query head of the group over the tokens of those blocks.
 * Training (same page, "Cómo se entrena MSA") adds a KL loss that pulls the index
 * distribution over the selected tokens toward the group-averaged main
 * distribution, with the teacher detached, so only the index projections get it.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are row-major and contiguous, bf16 unless stated:
 *      q, o, dO, dq      [B][N][H_q][d]
 *      k, v, dk, dv      [B][N][H_kv][d]
 *      q_idx, dq_idx     [B][N][H_kv][d_idx]
 *      k_idx, dk_idx     [B][N][d_idx]          (one index-key head for all groups)
 *      lse               [B][H_q][N]   float32, natural log of sum exp(scale q.k)
 *      lse_idx           [B][H_kv][N]  float32, natural log of sum exp(scale_idx z)
 *      block_idx         [B][H_kv][N][topk] int32, ascending block ids, -1 padded
 *    Query head h belongs to group h / (H_q / H_kv).
 *  - Every pointer is a DEVICE pointer owned by the caller, 16-byte aligned.  The
 *    library allocates nothing: each call gets a caller-owned device workspace of at
 *    least msa_workspace_size() bytes (256-byte aligned), used as scratch only
 *    during the call's kernels.
 *  - Calls are asynchronous on `stream` and return after enqueueing.  A non-zero
 *    return means nothing was enqueued (argument errors) or a launch failed.
 *    Errors found by the kernels themselves (a bounded wait that ran out) are
 *    recorded in a per-device status word, read with msa_get_device_status().
 *  - No exception, trap or abort crosses this boundary.
 *  - Supported (this build): causal = 1, Bk = 128, d in {64, 128},
 *    d_idx in {32, 64}, 1 <= topk <= 256, H_q % H_kv == 0 with G = H_q / H_kv in
 *    {1, 2, 4, 8, 16}, N <= 2^23.  N need not be a multiple of Bk.  Block selection
 *    (msa_index_topk, msa_decode) picks at most 32 blocks; topk > 32 is accepted by
 *    msa_index_topk only when topk >= nb = ceil(N / Bk) (the dense set below), and by
 *    msa_fwd / msa_bwd for any valid caller-given set.
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return / status codes. */
#define MSA_OK 0
#define MSA_ERR_ARG (-1)            /* null pointer, misaligned pointer, bad count */
#define MSA_ERR_SHAPE (-2)          /* inconsistent sizes (e.g. H_q % H_kv != 0) */
#define MSA_ERR_UNSUPPORTED (-3)    /* valid problem outside this build's kernels */
#define MSA_ERR_WORKSPACE (-4)      /* workspace NULL or smaller than required */
#define MSA_ERR_CUDA (-5)           /* a CUDA launch or runtime call failed */
#define MSA_ERR_DEVICE_TIMEOUT (-6) /* a kernel's bounded wait ran out (status word) */

/* Problem description.  scale: main softmax scale (> 0; e.g. 1/sqrt(d)).
 * scale_idx: index-logit scale sigma_I used by lse_idx, the KL and its gradients;
 * <= 0 selects 1/sqrt(d_idx).  Block selection ranks raw index dot products and
 * does not depend on scale_idx (softmax keeps the order: "El codiseño del kernel",
 * first idea).  The local block counts inside the topk budget. */
typedef struct msa_problem {
  int32_t B, N, H_q, H_kv, d, d_idx, Bk, topk;
  int32_t causal;
  float scale;
  float scale_idx;
} msa_problem_t;

/* Which call a workspace is sized for. */
#define MSA_WS_INDEX 0
#define MSA_WS_FWD 1
#define MSA_WS_BWD 2

/* Bytes of workspace the call `which` needs for problem p (0 if p is invalid). */
size_t msa_workspace_size(const msa_problem_t* p, int which);

/*
 * Index branch forward.
 *   Scores s[b,g,i,j] = q_idx[b,i,g,:] . k_idx[b,j,:] for every key j in a block
 *   wholly before query i's own block, max-pools them per Bk-token block, and keeps
 *   the topk-1 best such blocks plus the query's own block ("Cómo funcionan las dos
 *   ramas" ¶1-2; Flash-MSA article, tech.kuratif.com, ¶3 and ¶6: max-pooled
 *   128-token blocks, register top-k, local score forced to +inf).  Ranking uses
 *   the raw scores, no exp ("El codiseño del kernel", first idea).  Ties rank the
 *   lower block id first.  When fewer than topk blocks are visible all are taken
 *   and the remaining slots are -1.
 *   Dense set (indexer warm-up): with topk >= nb every visible block is taken
 *   (0 .. i/Bk, then -1) without scoring, so msa_fwd, msa_bwd and lse_idx cover the
 *   full causal context in both branches and the KL is taken over every visible
 *   token ("Cómo se entrena MSA" ¶3: the warm-up gives both branches full attention
 *   while the indexer learns from the KL alone).
 *   If lse_idx is not NULL it also writes the index log-sum-exp over the selected
 *   tokens (the cheap recompute of "Accelerating Million-Token Training", ¶4):
 *   lse_idx[b,g,i] = log sum_{j in T(b,g,i)} exp(scale_idx * s[b,g,i,j]), where
 *   T is the set of tokens j <= i of the selected blocks.
 * In:  q_idx, k_idx (bf16).  Out: block_idx (int32), lse_idx (float32, optional).
 */
int msa_index_topk(const msa_problem_t* p, const void* q_idx, const void* k_idx,
                   int32_t* block_idx, float* lse_idx, void* workspace, size_t workspace_bytes,
                   cudaStream_t stream);

/*
 * Main branch forward: exact block-sparse GQA softmax attention.
 *   For query i, head h of group g: o[b,i,h] = sum_{j in T} P_j v[b,j,g] with
 *   P = softmax_j(scale * q[b,i,h] . k[b,j,g]) over T(b,g,i) (the causally visible
 *   tokens of the group's blocks, "Cómo funcionan las dos ramas" ¶3), and
 *   lse[b,h,i] = log sum_{j in T} exp(scale q.k) kept for the backward (Flash-MSA
 *   article ¶6).  block_idx is msa_index_topk's output (or any valid set: ascending
 *   ids, own block included, -1 padding).
 * In:  q, k, v (bf16), block_idx.  Out: o (bf16), lse (float32).
 */
int msa_fwd(const msa_problem_t* p, const void* q, const void* k, const void* v,
            const int32_t* block_idx, void* o, float* lse, void* workspace,
            size_t workspace_bytes, cudaStream_t stream);

/*
 * Fused backward of the main branch and of the KL alignment loss, over the cached
 * block indices (Flash-MSA article ¶7; "Cómo se entrena MSA" ¶1-2).
 *   Main: dq, dk, dv of sum(dO * o), no KL term (the teacher is detached).
 *   KL:   p_T[j] = mean over the group's heads of P_h[j];
 *         p_I[j] = exp(scale_idx z_j - lse_idx), z_j = q_idx . k_idx[j];
 *         KL = kl_weight * sum over (b, g, i) of sum_j p_T (log p_T - log p_I);
 *         dq_idx, dk_idx are its gradients with p_T held fixed
 *         (dz_j = kl_weight (p_I - p_T)); dk_idx sums over groups.
 *   kl_weight is the per-row weight, e.g. coef / (B * H_kv * N) for a mean.
 *   o, lse: msa_fwd's outputs; lse_idx: msa_index_topk's.
 * In:  q, k, v, o, dO, q_idx, k_idx (bf16), lse, lse_idx (float32), block_idx.
 * Out: dq, dk, dv, dq_idx, dk_idx (bf16, overwritten); kl_out (one float32 on the
 *      device, overwritten with the KL value; may be NULL).
 */
int msa_bwd(const msa_problem_t* p, const void* q, const void* k, const void* v, const void* o,
            const float* lse, const void* dO, const void* q_idx, const void* k_idx,
            const int32_t* block_idx, const float* lse_idx, float kl_weight, void* dq, void* dk,
            void* dv, void* dq_idx, void* dk_idx, float* kl_out, void* workspace,
            size_t workspace_bytes, cudaStream_t stream);

/*
 * One plan per step.  msa_index_topk (for lse_idx), msa_fwd and msa_bwd each turn
 * block_idx into the same inverted lists (for every key block, the (query, slot)
 * pairs that selected it: the KV-outer query gather of "El codiseño del kernel").
 * The _plan variants build them once, into a caller-owned buffer that lives from a
 * layer's index call to its backward:
 *   msa_plan_size(p)     bytes of the plan buffer for problem p (0 if p is invalid);
 *   msa_index_topk_plan  as msa_index_topk, and writes the plan of the block_idx it
 *                        computes (also when lse_idx is NULL);
 *   msa_fwd_plan, msa_bwd_plan
 *                        as msa_fwd, msa_bwd (same workspace sizes), reading that plan
 *                        instead of building their own.
 * The plan must be the one msa_index_topk_plan wrote for the same problem and the same
 * block_idx, unchanged since.  plan must be 256-byte aligned and plan_bytes at least
 * msa_plan_size(p) (else MSA_ERR_ARG / MSA_ERR_WORKSPACE).  The plan starts with a header
 * naming its problem, written last by the build.  A reading call first checks that header
 * on the device.  If it names another problem (or no complete build), the call records
 * MSA_ERR_ARG in the device status (msa_get_device_status), empties the plan's lists, and
 * computes nothing meaningful; it never reads outside the plan's arrays.
 * Fixed-length batches only; the variable-length calls build their own plan.
 */
size_t msa_plan_size(const msa_problem_t* p);
int msa_index_topk_plan(const msa_problem_t* p, const void* q_idx, const void* k_idx,
                        int32_t* block_idx, float* lse_idx, void* plan, size_t plan_bytes,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream);
int msa_fwd_plan(const msa_problem_t* p, const void* q, const void* k, const void* v,
                 const int32_t* block_idx, void* plan, size_t plan_bytes, void* o, float* lse,
                 void* workspace, size_t workspace_bytes, cudaStream_t stream);
int msa_bwd_plan(const msa_problem_t* p, const void* q, const void* k, const void* v, const void* o,
                 const float* lse, const void* dO, const void* q_idx, const void* k_idx,
                 const int32_t* block_idx, const float* lse_idx, void* plan, size_t plan_bytes,
                 float kl_weight, void* dq, void* dk, void* dv, void* dq_idx, void* dk_idx,
                 float* kl_out, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Packed variable-length batches (the variable-length view of the sparse attention,
 * Flash-MSA article, tech.kuratif.com, ¶7).  num_seqs sequences share one token axis of
 * total_tokens tokens: sequence s holds tokens cu_seqlens[s] .. cu_seqlens[s+1]-1 of
 * every packed tensor, whose layouts are the single-sequence ones with the batch axis
 * dropped:
 *   q, o, dO, dq [T][H_q][d];  k, v, dk, dv [T][H_kv][d];  q_idx, dq_idx [T][H_kv][d_idx];
 *   k_idx, dk_idx [T][d_idx]   (T = total_tokens).
 * Each sequence is its own causal problem (its blocks start at its first token; its
 * last block may be ragged).  Per-sequence outputs are packed sequence after sequence,
 * each in the single-sequence layout:
 *   block_idx: [H_kv][L_s][topk] at element offset cu_seqlens[s] * H_kv * topk;
 *   lse_idx:   [H_kv][L_s]       at cu_seqlens[s] * H_kv;
 *   lse:       [H_q][L_s]        at cu_seqlens[s] * H_q.
 * cu_seqlens is a DEVICE array of num_seqs + 1 int32 (4-byte aligned), read by the
 * kernels only: the host never waits for it.  p->N bounds every sequence's length (the
 * batch's max_seqlen: it sizes the grids and the block space, ceil(N / 128) blocks per
 * sequence and group, at most 16384); p->B is not read.  The rules, checked on the
 * device: cu_seqlens[0] = 0, non-decreasing, cu_seqlens[num_seqs] <= total_tokens, every
 * length <= p->N.  A batch that breaks one writes no output and sets the device status to
 * MSA_ERR_ARG (msa_get_device_status).  Sequences may be empty and may start at any
 * token.  Tokens from cu_seqlens[num_seqs] to total_tokens are outside every sequence:
 * their output rows are not written (dk_idx included).
 * Each call runs a fixed number of kernels whatever num_seqs is: one small kernel
 * validates cu_seqlens and writes per-sequence spans and work tables into the head of
 * the workspace, then the single-sequence kernels run over the whole batch.
 * The workspace (256-byte aligned) is sized by msa_workspace_size_varlen for the call;
 * msa_index_topk_varlen needs one even when lse_idx is NULL.  The backward's kl_out is
 * the KL summed over every row of every sequence (weighted by kl_weight).
 */
size_t msa_workspace_size_varlen(const msa_problem_t* p, int num_seqs, int total_tokens,
                                 int which);
int msa_index_topk_varlen(const msa_problem_t* p, const int32_t* cu_seqlens, int num_seqs,
                          int total_tokens, const void* q_idx, const void* k_idx,
                          int32_t* block_idx, float* lse_idx, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream);
int msa_fwd_varlen(const msa_problem_t* p, const int32_t* cu_seqlens, int num_seqs,
                   int total_tokens, const void* q, const void* k, const void* v,
                   const int32_t* block_idx, void* o, float* lse, void* workspace,
                   size_t workspace_bytes, cudaStream_t stream);
int msa_bwd_varlen(const msa_problem_t* p, const int32_t* cu_seqlens, int num_seqs,
                   int total_tokens, const void* q, const void* k, const void* v, const void* o,
                   const float* lse, const void* dO, const void* q_idx, const void* k_idx,
                   const int32_t* block_idx, const float* lse_idx, float kl_weight, void* dq,
                   void* dk, void* dv, void* dq_idx, void* dk_idx, float* kl_out,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Decode (inference): one new query token per sequence against its KV cache.
 *   The index branch scores the new token against the cached index keys, max-pools
 *   them per Bk-token block, keeps the topk-1 best blocks wholly before its own block
 *   plus its own block ("Cómo funcionan las dos ramas" ¶1-2; the block indices are then
 *   reused by the main branch, Flash-MSA article ¶3), and the main branch attends over
 *   those blocks' causally visible tokens.  The result is row lens[b]-1 of
 *   msa_index_topk + msa_fwd run on the cache (up to rounding; near-tied blocks may be
 *   chosen either way).
 *   p->N is the cache capacity Lmax, p->B the number of sequences.
 * In:  q [B][H_q][d], q_idx [B][H_kv][d_idx] (the new token's projections, bf16);
 *      k, v [B][Lmax][H_kv][d], k_idx [B][Lmax][d_idx] (caches, bf16; the new token's
 *      own k, v, k_idx already at row lens[b]-1);
 *      lens: device int32 [B], 1 <= lens[b] <= Lmax (an invalid length is recorded as
 *      MSA_ERR_ARG in the status word and treated as 1).
 * Out: block_idx [B][H_kv][topk] (int32, ascending, -1 padded), o [B][H_q][d] (bf16),
 *      lse [B][H_q] (float32).  topk <= 32.
 * Workspace: msa_decode_workspace_size(p) bytes, 256-byte aligned.
 */
size_t msa_decode_workspace_size(const msa_problem_t* p);
int msa_decode(const msa_problem_t* p, const void* q, const void* q_idx, const void* k,
               const void* v, const void* k_idx, const int32_t* lens, int32_t* block_idx, void* o,
               float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * FP8 KV cache (E4M3).  The pages name FP8 as one of the precisions of the MSA
 * attention kernels ("El codiseño del kernel", fmha_sm100 paragraph) and give no
 * recipe; this build takes one float32 scale per (sequence, token, KV head) row:
 *   scale = amax |x| / 448 (1 for an all-zero row),
 *   code  = the E4M3 value nearest to x / scale (ties to even, |.| > 448 saturates),
 *   value seen by attention = decode(code) * scale.
 * Both divisions are IEEE round-to-nearest, so the codes are reproducible bit for bit.
 *
 * msa_quantize_kv_fp8: x [B][N][H_kv][d] bf16 (a k or v cache, p->N its capacity)
 *   -> x8 [B][N][H_kv][d] uint8 codes, scale [B][N][H_kv] float32.  Call once for k,
 *   once for v.  Only p->B, p->N, p->H_kv and p->d (64 or 128) are read.  Pointers
 *   16-byte aligned; the output buffers are overwritten.
 * msa_decode_fp8: msa_decode with the cache given as k8, v8 (codes) and k_scale,
 *   v_scale (row scales) instead of bf16 k, v; the index branch (q_idx, k_idx) stays
 *   bf16.  Same outputs, workspace (msa_decode_workspace_size) and errors.
 */
int msa_quantize_kv_fp8(const msa_problem_t* p, const void* x, uint8_t* x8, float* scale,
                        cudaStream_t stream);
int msa_decode_fp8(const msa_problem_t* p, const void* q, const void* q_idx, const uint8_t* k8,
                   const uint8_t* v8, const float* k_scale, const float* v_scale, const void* k_idx,
                   const int32_t* lens, int32_t* block_idx, void* o, float* lse, void* workspace,
                   size_t workspace_bytes, cudaStream_t stream);

/*
 * FP8 (E4M3) main-branch forward for training (d = 128): the same block-sparse
 * attention as msa_fwd with E4M3 operands on the tensor cores.  The pages list FP8
 * among the precisions of the MSA attention kernels ("El codiseño del kernel",
 * fmha_sm100 paragraph) without a recipe; this build takes:
 *   q8 [B][N][H_q][d] codes, q_scale [B][N][H_q]: one scale per (token, head) row;
 *   k8 [B][N][H_kv][d] codes, k_scale [B][H_kv][nb]: one scale per 128-key block;
 *   v8t [B][H_kv][nb][d][128] codes (v transposed within each block, keys past N
 *       zero), v_scale [B][H_kv][nb]: one scale per block;
 *   scale = amax / 448 over the row or block (1 if all zero), code = E4M3 nearest to
 *   float32(x / scale), ties to even, saturating (the KV-cache quantiser's rule);
 *   scores s_q s_k (q8 . k8) * scale, exact row max, P = exp(score - max) rounded to
 *   E4M3 for the P V product, l = sum of the unrounded P,
 *   o = s_v (P8 . v8) / l (bf16), lse = max + log l (float32).
 * msa_quantize_fwd_fp8 writes q8, q_scale, k8, k_scale, v8t, v_scale from bf16 q, k, v
 * (p->d must be 128); msa_fwd_fp8 takes them with the block sets and writes o, lse,
 * using a workspace of msa_workspace_size(p, MSA_WS_FWD) bytes.  Pointers 16-byte
 * aligned, outputs overwritten; errors as msa_fwd (MSA_ERR_UNSUPPORTED for d != 128).
 */
int msa_quantize_fwd_fp8(const msa_problem_t* p, const void* q, const void* k, const void* v,
                         uint8_t* q8, float* q_scale, uint8_t* k8, float* k_scale, uint8_t* v8t,
                         float* v_scale, cudaStream_t stream);
int msa_fwd_fp8(const msa_problem_t* p, const uint8_t* q8, const float* q_scale, const uint8_t* k8,
                const float* k_scale, const uint8_t* v8t, const float* v_scale,
                const int32_t* block_idx, void* o, float* lse, void* workspace,
                size_t workspace_bytes, cudaStream_t stream);

/* Synchronises `stream`, then reads and clears the current device's status word
 * (MSA_OK or the first MSA_ERR_* a kernel recorded since the last read). */
int msa_get_device_status(cudaStream_t stream, int* status);

/* Human-readable text for a status code (static storage). */
const char* msa_status_string(int code);

/* Test knob for the failure path, per process: the bounded device waits give up
 * after wait_limit_ns (0 restores the default of 2 s); flags bit 0
 * (MSA_DEBUG_WITHHOLD_LOAD) makes the next index-top-k launches withhold their first
 * TMA load, so the consumer's wait runs out, the kernel records
 * MSA_ERR_DEVICE_TIMEOUT and returns without hanging. */
#define MSA_DEBUG_WITHHOLD_LOAD 1
int msa_debug_set(uint64_t wait_limit_ns, int flags);

/* Profiling hook.  Kernels: MSA_KERNEL_INDEX (the index scoring + top-k kernel of
 * msa_index_topk), MSA_KERNEL_FWD (the gathered attention kernel of msa_fwd),
 * MSA_KERNEL_BWD (the fused backward kernel of msa_bwd), MSA_KERNEL_INDEX_LSE (the
 * gathered index log-sum-exp kernel of msa_index_topk when lse_idx is requested).  When start and stop are
 * both non-NULL, every later launch of that kernel records `start` on its stream
 * just before the launch and `stop` just after it; NULL clears the hook.  The
 * events are the caller's (created on the current device) and are only recorded,
 * never synchronised or destroyed by the library. */
#define MSA_KERNEL_INDEX 0
#define MSA_KERNEL_FWD 1
#define MSA_KERNEL_BWD 2
#define MSA_KERNEL_INDEX_LSE 3
int msa_set_kernel_events(int kernel, cudaEvent_t start, cudaEvent_t stop);

/* Number of kernels this library has launched in this process (all devices). */
uint64_t msa_kernel_launch_count(void);

/*
 * Index branch without a caller workspace.  Same computation and outputs as
 * msa_index_topk, for callers that cannot allocate device memory (a plug-in inside
 * a framework that owns every allocation, a service whose device footprint is fixed
 * at start-up).  The pages have no counterpart: this is an interface convenience.
 * Scratch comes from a 64 MiB array compiled into the library (every GPU that loads
 * the library holds it until exit; msa_noalloc_scratch_bytes() returns the size).
 * Problems whose index workspace (msa_workspace_size(p, MSA_WS_INDEX)) exceeds it
 * return MSA_ERR_WORKSPACE before anything is enqueued; with lse_idx == NULL no
 * scratch is used.  The first call on a device (and the first after the device's
 * context changes, e.g. after cudaDeviceReset) looks up the array's device address,
 * which may load the module: make it before any stream capture.  All calls on a
 * device share the array and it keeps the previous call's contents: each call zeroes
 * the counters it needs with a memset on `stream` (no allocation).  Calls that may
 * overlap on the GPU race and must be ordered by the caller.  `stream` must belong
 * to the current device, as for every entry point.
 */
int msa_index_topk_noalloc(const msa_problem_t* p, const void* q_idx, const void* k_idx,
                           int32_t* block_idx, float* lse_idx, cudaStream_t stream);
size_t msa_noalloc_scratch_bytes(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int msa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H_ */
