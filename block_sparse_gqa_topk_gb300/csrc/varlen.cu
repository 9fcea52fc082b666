// varlen.cu -- packed variable-length batches (cu_seqlens) over the single-sequence
// entry points.
//
// Method: the MoBA-style variable-length view of Flash-MSA (tech.kuratif.com ¶7):
// sequences of different lengths are packed along one token axis and each is its own
// causal problem, with its 128-token blocks starting at its first token.  Every call
// here validates the whole batch on the host, then runs the single-sequence entry
// point on each sequence's slice (B = 1, N = its length) in stream order, reusing one
// workspace.  The backward's per-sequence KL values land in the workspace and one
// small kernel sums them into kl_out.
#include <string.h>

#include "kernels.h"

namespace msa {
namespace {

// Sum of the per-sequence KL values (one warp, double accumulation).
__global__ void varlen_kl_sum_kernel(const float* __restrict__ part, int n, float* __restrict__ out) {
  double acc = 0.0;
  for (int i = threadIdx.x; i < n; i += 32) acc += (double)part[i];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (threadIdx.x == 0) *out = (float)acc;
}

// Validates the batch description (shapes are checked by the per-sequence calls);
// fills the per-sequence problem template.
int check_varlen(const msa_problem_t* p, const int32_t* cu, int num_seqs, msa_problem_t* one) {
  if (!p || !cu || num_seqs < 0) return MSA_ERR_ARG;
  if (cu[0] != 0) return MSA_ERR_ARG;
  for (int s = 0; s < num_seqs; ++s) {
    if (cu[s + 1] < cu[s]) return MSA_ERR_ARG;
    if ((cu[s] & 3) != 0) return MSA_ERR_ARG;  // keeps every per-sequence slice 16-byte aligned
  }
  *one = *p;
  one->B = 1;
  one->N = 0;
  return MSA_OK;
}

template <typename T>
T* at(T* base, int64_t elems, size_t elem_bytes) {
  return base ? reinterpret_cast<T*>(reinterpret_cast<uintptr_t>(base) + (uintptr_t)(elems * elem_bytes))
              : nullptr;
}
template <typename T>
const T* at(const T* base, int64_t elems, size_t elem_bytes) {
  return base ? reinterpret_cast<const T*>(reinterpret_cast<uintptr_t>(base) +
                                           (uintptr_t)(elems * elem_bytes))
              : nullptr;
}

size_t kl_tail(int num_seqs) { return align256((size_t)(num_seqs > 0 ? num_seqs : 1) * sizeof(float)); }

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" {

size_t msa_workspace_size_varlen(const msa_problem_t* p, const int32_t* cu_seqlens, int num_seqs,
                                 int which) {
  msa_problem_t one;
  if (check_varlen(p, cu_seqlens, num_seqs, &one) != MSA_OK) return 0;
  size_t need = 0;
  for (int s = 0; s < num_seqs; ++s) {
    one.N = cu_seqlens[s + 1] - cu_seqlens[s];
    if (one.N == 0) continue;
    const size_t w = msa_workspace_size(&one, which);
    if (w == 0) return 0;
    need = w > need ? w : need;
  }
  need = align256(need > 0 ? need : 256);
  if (which == MSA_WS_BWD) need += kl_tail(num_seqs);
  return need;
}

int msa_index_topk_varlen(const msa_problem_t* p, const int32_t* cu_seqlens, int num_seqs,
                          const void* q_idx, const void* k_idx, int32_t* block_idx, float* lse_idx,
                          void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  msa_problem_t one;
  int rc = check_varlen(p, cu_seqlens, num_seqs, &one);
  if (rc) return rc;
  if (lse_idx && workspace_bytes < msa_workspace_size_varlen(p, cu_seqlens, num_seqs, MSA_WS_INDEX))
    return MSA_ERR_WORKSPACE;
  for (int s = 0; s < num_seqs; ++s) {
    const int64_t c0 = cu_seqlens[s];
    one.N = cu_seqlens[s + 1] - cu_seqlens[s];
    if (one.N == 0) continue;
    rc = msa_index_topk(&one, at(q_idx, c0 * p->H_kv * p->d_idx, 2), at(k_idx, c0 * p->d_idx, 2),
                        at(block_idx, c0 * p->H_kv * p->topk, 4), at(lse_idx, c0 * p->H_kv, 4),
                        workspace, workspace_bytes, stream);
    if (rc) return rc;
  }
  return MSA_OK;
}

int msa_fwd_varlen(const msa_problem_t* p, const int32_t* cu_seqlens, int num_seqs, const void* q,
                   const void* k, const void* v, const int32_t* block_idx, void* o, float* lse,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  msa_problem_t one;
  int rc = check_varlen(p, cu_seqlens, num_seqs, &one);
  if (rc) return rc;
  if (workspace_bytes < msa_workspace_size_varlen(p, cu_seqlens, num_seqs, MSA_WS_FWD))
    return MSA_ERR_WORKSPACE;
  for (int s = 0; s < num_seqs; ++s) {
    const int64_t c0 = cu_seqlens[s];
    one.N = cu_seqlens[s + 1] - cu_seqlens[s];
    if (one.N == 0) continue;
    rc = msa_fwd(&one, at(q, c0 * p->H_q * p->d, 2), at(k, c0 * p->H_kv * p->d, 2),
                 at(v, c0 * p->H_kv * p->d, 2), at(block_idx, c0 * p->H_kv * p->topk, 4),
                 at(o, c0 * p->H_q * p->d, 2), at(lse, c0 * p->H_q, 4), workspace, workspace_bytes,
                 stream);
    if (rc) return rc;
  }
  return MSA_OK;
}

int msa_bwd_varlen(const msa_problem_t* p, const int32_t* cu_seqlens, int num_seqs, const void* q,
                   const void* k, const void* v, const void* o, const float* lse, const void* dO,
                   const void* q_idx, const void* k_idx, const int32_t* block_idx,
                   const float* lse_idx, float kl_weight, void* dq, void* dk, void* dv,
                   void* dq_idx, void* dk_idx, float* kl_out, void* workspace,
                   size_t workspace_bytes, cudaStream_t stream) {
  msa_problem_t one;
  int rc = check_varlen(p, cu_seqlens, num_seqs, &one);
  if (rc) return rc;
  const size_t need = msa_workspace_size_varlen(p, cu_seqlens, num_seqs, MSA_WS_BWD);
  if (!workspace || workspace_bytes < need) return MSA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return MSA_ERR_ARG;
  // per-sequence KL values in the workspace's tail
  const size_t body = need - kl_tail(num_seqs);
  float* kl_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + body);
  for (int s = 0; s < num_seqs; ++s) {
    const int64_t c0 = cu_seqlens[s];
    one.N = cu_seqlens[s + 1] - cu_seqlens[s];
    rc = msa_bwd(&one, at(q, c0 * p->H_q * p->d, 2), at(k, c0 * p->H_kv * p->d, 2),
                 at(v, c0 * p->H_kv * p->d, 2), at(o, c0 * p->H_q * p->d, 2),
                 at(lse, c0 * p->H_q, 4), at(dO, c0 * p->H_q * p->d, 2),
                 at(q_idx, c0 * p->H_kv * p->d_idx, 2), at(k_idx, c0 * p->d_idx, 2),
                 at(block_idx, c0 * p->H_kv * p->topk, 4), at(lse_idx, c0 * p->H_kv, 4), kl_weight,
                 at(dq, c0 * p->H_q * p->d, 2), at(dk, c0 * p->H_kv * p->d, 2),
                 at(dv, c0 * p->H_kv * p->d, 2), at(dq_idx, c0 * p->H_kv * p->d_idx, 2),
                 at(dk_idx, c0 * p->d_idx, 2), kl_part + s, workspace, body, stream);
    if (rc) return rc;
  }
  if (kl_out) {
    if (num_seqs == 0) return cudaMemsetAsync(kl_out, 0, sizeof(float), stream) == cudaSuccess
                                  ? MSA_OK : MSA_ERR_CUDA;
    varlen_kl_sum_kernel<<<1, 32, 0, stream>>>(kl_part, num_seqs, kl_out);
    note_launch();
    if (cudaGetLastError() != cudaSuccess) return MSA_ERR_CUDA;
  }
  return MSA_OK;
}

}  // extern "C"
