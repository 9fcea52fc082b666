// varlen.cu -- packed variable-length batches, with cu_seqlens on the device.
//
// Method: the variable-length view of block-sparse attention (Flash-MSA article,
// tech.kuratif.com ¶7): sequences of different lengths share one token axis and each
// is its own causal problem, its 128-token blocks starting at its first token.
//
// A packed batch runs through the same kernels as the fixed [B][N] layout, with the same
// number of launches whatever the number of sequences.  Every kernel finds a sequence's
// tokens through a (start, end) span per sequence.  The kernels whose grids are laid out
// per sequence (index scoring, the plan's count and fill, the backward preprocess) map
// their CTAs through prefix tables of their row chunks per sequence.  One small kernel,
// varlen_prepare_kernel, checks cu_seqlens on the device and writes the spans and the
// tables into the head of the call's workspace.  A batch that breaks the rules gets
// empty spans, so nothing is read or written, and MSA_ERR_ARG in the device status word.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace msa {
namespace {

constexpr int kPrepThreads = 1024;
constexpr int kPrepWarps = kPrepThreads / 32;

// Checks 0 = cu[0] <= cu[1] <= ... <= cu[n] <= T and cu[s+1] - cu[s] <= N.  Then writes
// spans[s] = (cu[s], cu[s+1]) (every span (0, 0) if a check failed) and, for each table
// k, tab[k][s] = sum over s' < s of ceil(len_s' / rows[k]), with tab[k][n] the total.
// One CTA: the scans run over the sequences 1024 at a time.
__global__ void __launch_bounds__(kPrepThreads)
    varlen_prepare_kernel(const int32_t* __restrict__ cu, int n, int64_t T, int N, int4 rows,
                          int2* __restrict__ spans, int* __restrict__ tabs, int* status) {
  __shared__ int bad;
  __shared__ int s_w[kNumVarlenTabs][kPrepWarps];
  __shared__ int carry[kNumVarlenTabs];
  if (threadIdx.x == 0) {
    bad = (__ldg(&cu[0]) != 0 || (int64_t)__ldg(&cu[n]) > T) ? 1 : 0;
    for (int k = 0; k < kNumVarlenTabs; ++k) carry[k] = 0;
  }
  __syncthreads();
  for (int s = threadIdx.x; s < n; s += kPrepThreads) {
    const int a = __ldg(&cu[s]), e = __ldg(&cu[s + 1]);
    if (e < a || e - a > N) atomicOr(&bad, 1);
  }
  __syncthreads();
  const bool ok = bad == 0;
  if (threadIdx.x == 0 && !ok) set_status(status, MSA_ERR_ARG);
  const int r[kNumVarlenTabs] = {rows.x, rows.y, rows.z, rows.w};
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int base = 0; base < n; base += kPrepThreads) {
    const int s = base + threadIdx.x;
    int a = 0, e = 0;
    if (ok && s < n) {
      a = __ldg(&cu[s]);
      e = __ldg(&cu[s + 1]);
    }
    if (s < n) spans[s] = make_int2(a, e);
    int v[kNumVarlenTabs], incl[kNumVarlenTabs];
#pragma unroll
    for (int k = 0; k < kNumVarlenTabs; ++k) {
      v[k] = (e - a + r[k] - 1) / r[k];
      incl[k] = v[k];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, incl[k], o);
        if (lane >= o) incl[k] += x;
      }
      if (lane == 31) s_w[k][warp] = incl[k];
    }
    __syncthreads();
    if (warp < kNumVarlenTabs) {  // warp k scans the warp totals of table k
      int w = s_w[warp][lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += x;
      }
      s_w[warp][lane] = w;  // inclusive over warps
    }
    __syncthreads();
    int excl[kNumVarlenTabs];
#pragma unroll
    for (int k = 0; k < kNumVarlenTabs; ++k) {
      excl[k] = carry[k] + (warp ? s_w[k][warp - 1] : 0) + incl[k] - v[k];
      if (s < n) tabs[(size_t)k * (n + 1) + s] = excl[k];
    }
    __syncthreads();
    if (threadIdx.x == kPrepThreads - 1)
#pragma unroll
      for (int k = 0; k < kNumVarlenTabs; ++k) carry[k] = excl[k] + v[k];
    __syncthreads();
  }
  if (threadIdx.x == 0)
    for (int k = 0; k < kNumVarlenTabs; ++k) tabs[(size_t)k * (n + 1) + n] = carry[k];
}

size_t header_bytes(int nseq) {
  return align256((size_t)nseq * sizeof(int2)) +
         align256((size_t)kNumVarlenTabs * (nseq + 1) * sizeof(int));
}

// The packed batch's problem: B = num_seqs sequences of at most p->N tokens on an axis of
// total_tokens.  p->B is not read.
int packed_shape(const msa_problem_t* p, int num_seqs, int total_tokens, Shape* s) {
  if (!p || num_seqs < 0 || total_tokens < 0) return MSA_ERR_ARG;
  msa_problem_t q = *p;
  q.B = num_seqs > 0 ? 1 : 0;  // the size limits below are the packed batch's own
  int rc = validate_problem(&q, s);
  if (rc) return rc;
  s->B = num_seqs;
  s->T = total_tokens;
  if (s->rows_kv() * s->topk * (int64_t)s->G >= (int64_t)1 << 31) return MSA_ERR_UNSUPPORTED;
  if (s->keys() >= (int64_t)1 << 31) return MSA_ERR_UNSUPPORTED;  // int key ids
  if (s->nb > kPlanSmemBins) return MSA_ERR_UNSUPPORTED;  // the plan's shared-memory bins
  return MSA_OK;
}

bool empty_batch(const Shape& s) { return s.B == 0 || s.T == 0 || s.N == 0; }

int check_workspace(void* ws, size_t have, size_t need) {
  if (!ws || have < need) return MSA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return MSA_ERR_ARG;
  return MSA_OK;
}

// Writes the spans and chunk tables into the workspace head and points s at them.
cudaError_t prepare(Shape* s, const int32_t* cu, void* ws, const Ctx& cx, cudaStream_t st) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  int2* spans = reinterpret_cast<int2*>(w);
  int* tabs = reinterpret_cast<int*>(w + align256((size_t)s->B * sizeof(int2)));
  const int4 rows = make_int4(varlen_chunk_rows(kTabIndexUnit, s->topk),
                              varlen_chunk_rows(kTabPlanCount, s->topk),
                              varlen_chunk_rows(kTabPlanFill, s->topk),
                              varlen_chunk_rows(kTabRows64, s->topk));
  static_assert(kNumVarlenTabs == 4, "one int4 of chunk rows");
  varlen_prepare_kernel<<<1, kPrepThreads, 0, st>>>(cu, s->B, s->T, s->N, rows, spans, tabs,
                                                    cx.status);
  note_launch();
  s->spans = spans;
  s->tabs = tabs;
  return cudaGetLastError();
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" {

size_t msa_workspace_size_varlen(const msa_problem_t* p, int num_seqs, int total_tokens,
                                 int which) {
  Shape s;
  if (packed_shape(p, num_seqs, total_tokens, &s) != MSA_OK) return 0;
  size_t body = 0;
  switch (which) {
    case MSA_WS_INDEX: body = ws_index_bytes(s); break;
    case MSA_WS_FWD: body = ws_fwd_bytes(s); break;
    case MSA_WS_BWD: body = bwd_ws_bytes(s); break;
    default: return 0;
  }
  return header_bytes(num_seqs) + body;
}

int msa_index_topk_varlen(const msa_problem_t* p, const int32_t* cu_seqlens, int num_seqs,
                          int total_tokens, const void* q_idx, const void* k_idx,
                          int32_t* block_idx, float* lse_idx, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
  Shape s;
  int rc = packed_shape(p, num_seqs, total_tokens, &s);
  if (rc) return rc;
  if (empty_batch(s)) return MSA_OK;
  if (!cu_seqlens || !aligned(cu_seqlens, 4)) return MSA_ERR_ARG;
  if ((rc = check_index_args(s, q_idx, k_idx, block_idx))) return rc;
  const size_t head = header_bytes(num_seqs);
  if ((rc = check_workspace(workspace, workspace_bytes,
                            head + (lse_idx ? ws_index_bytes(s) : 0))))
    return rc;
  Ctx cx;
  if ((rc = device_ctx(&cx))) return rc;
  cudaError_t e = prepare(&s, cu_seqlens, workspace, cx, stream);
  if (e != cudaSuccess) return finish(e);
  return finish(run_index(s, q_idx, k_idx, block_idx, lse_idx,
                          static_cast<uint8_t*>(workspace) + head, cx, stream));
}

int msa_fwd_varlen(const msa_problem_t* p, const int32_t* cu_seqlens, int num_seqs,
                   int total_tokens, const void* q, const void* k, const void* v,
                   const int32_t* block_idx, void* o, float* lse, void* workspace,
                   size_t workspace_bytes, cudaStream_t stream) {
  Shape s;
  int rc = packed_shape(p, num_seqs, total_tokens, &s);
  if (rc) return rc;
  if (empty_batch(s)) return MSA_OK;
  if (!cu_seqlens || !aligned(cu_seqlens, 4)) return MSA_ERR_ARG;
  if ((rc = check_fwd_args(q, k, v, block_idx, o, lse))) return rc;
  const size_t head = header_bytes(num_seqs);
  if ((rc = check_workspace(workspace, workspace_bytes, head + ws_fwd_bytes(s)))) return rc;
  Ctx cx;
  if ((rc = device_ctx(&cx))) return rc;
  cudaError_t e = prepare(&s, cu_seqlens, workspace, cx, stream);
  if (e != cudaSuccess) return finish(e);
  return finish(run_fwd(s, q, k, v, block_idx, o, lse, static_cast<uint8_t*>(workspace) + head,
                        cx, stream));
}

int msa_bwd_varlen(const msa_problem_t* p, const int32_t* cu_seqlens, int num_seqs,
                   int total_tokens, const void* q, const void* k, const void* v, const void* o,
                   const float* lse, const void* dO, const void* q_idx, const void* k_idx,
                   const int32_t* block_idx, const float* lse_idx, float kl_weight, void* dq,
                   void* dk, void* dv, void* dq_idx, void* dk_idx, float* kl_out,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  Shape s;
  int rc = packed_shape(p, num_seqs, total_tokens, &s);
  if (rc) return rc;
  if (!isfinite(kl_weight)) return MSA_ERR_ARG;
  if (empty_batch(s)) {
    if (kl_out) return finish(cudaMemsetAsync(kl_out, 0, sizeof(float), stream));
    return MSA_OK;
  }
  if (!cu_seqlens || !aligned(cu_seqlens, 4)) return MSA_ERR_ARG;
  const void* ins[] = {q, k, v, o, lse, dO, q_idx, k_idx, block_idx, lse_idx,
                       dq, dk, dv, dq_idx, dk_idx};
  if ((rc = check_bwd_args(ins, sizeof(ins) / sizeof(ins[0])))) return rc;
  const size_t head = header_bytes(num_seqs);
  if ((rc = check_workspace(workspace, workspace_bytes, head + bwd_ws_bytes(s)))) return rc;
  Ctx cx;
  if ((rc = device_ctx(&cx))) return rc;
  cudaError_t e = prepare(&s, cu_seqlens, workspace, cx, stream);
  if (e != cudaSuccess) return finish(e);
  return finish(run_bwd(s, q, k, v, o, lse, dO, q_idx, k_idx, block_idx, lse_idx, kl_weight, dq,
                        dk, dv, dq_idx, dk_idx, kl_out, static_cast<uint8_t*>(workspace) + head,
                        cx, stream));
}

}  // extern "C"
