// msa_api.cu -- the C ABI of libmsa.so (declared in include/msa.h).
//
// Validates every argument on the host before anything is enqueued, carves the
// caller's workspace, and sequences the kernels on the caller's stream.  The only
// library state is the per-device status word and the failure-test knob.
#include <math.h>
#include <atomic>
#include <mutex>
#include <string.h>

#include "kernels.h"

namespace msa {
namespace {

__device__ int g_status_word;  // one per device (module-scope device variable)

constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s per device-side wait
uint64_t g_wait_ns = kDefaultWaitNs;
int g_debug = 0;
std::mutex g_mu;
std::mutex g_sym_mu;

int status_ptr(int** out) {
  void* p = nullptr;
  const int rc = device_symbol_address(reinterpret_cast<const void*>(&g_status_word), &p);
  if (rc == MSA_OK) *out = static_cast<int*>(p);
  return rc;
}

int make_ctx(Ctx* cx) {
  int rc = status_ptr(&cx->status);
  if (rc) return rc;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MSA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MSA_ERR_CUDA;
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return MSA_ERR_UNSUPPORTED;  // built for sm_103a only
  {
    std::lock_guard<std::mutex> lk(g_mu);
    cx->wait_ns = g_wait_ns;
    cx->debug = g_debug;
  }
  cx->num_sms = sms;
  return MSA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Shape checks shared by every call.  Returns MSA_OK and fills s.
int check_problem(const msa_problem_t* p, Shape* s) {
  if (!p) return MSA_ERR_ARG;
  if (p->B < 0 || p->N < 0 || p->H_q <= 0 || p->H_kv <= 0 || p->d <= 0 || p->d_idx <= 0 ||
      p->Bk <= 0 || p->topk <= 0)
    return MSA_ERR_SHAPE;
  if (p->H_q % p->H_kv != 0) return MSA_ERR_SHAPE;
  if (!(p->scale > 0.f) || !isfinite(p->scale)) return MSA_ERR_ARG;
  if (!isfinite(p->scale_idx)) return MSA_ERR_ARG;
  const int G = p->H_q / p->H_kv;
  if (p->causal != 1) return MSA_ERR_UNSUPPORTED;
  if (p->Bk != 128) return MSA_ERR_UNSUPPORTED;
  if (p->d != 64 && p->d != 128) return MSA_ERR_UNSUPPORTED;
  if (p->d_idx != 32 && p->d_idx != 64) return MSA_ERR_UNSUPPORTED;
  if (p->topk > kMaxSlots) return MSA_ERR_UNSUPPORTED;
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return MSA_ERR_UNSUPPORTED;
  if (p->N > (1 << 23)) return MSA_ERR_UNSUPPORTED;  // (query << 8) | slot stays an int
  s->B = p->B;
  s->N = p->N;
  s->H_q = p->H_q;
  s->H_kv = p->H_kv;
  s->d = p->d;
  s->d_idx = p->d_idx;
  s->Bk = p->Bk;
  s->topk = p->topk;
  s->causal = p->causal;
  s->scale = p->scale;
  s->scale_idx = p->scale_idx > 0.f ? p->scale_idx : 1.0f / sqrtf((float)p->d_idx);
  s->G = G;
  s->nb = (p->N + p->Bk - 1) / p->Bk;
  s->T = (int64_t)p->B * p->N;
  s->spans = nullptr;
  s->tabs = nullptr;
  // int32 offsets index every (row, slot) entry and every partial row
  if (s->rows_kv() * s->topk * (int64_t)G >= (int64_t)1 << 31) return MSA_ERR_UNSUPPORTED;
  return MSA_OK;
}

size_t ws_index(const Shape& s) {
  return plan_bytes(s) + align256((size_t)s.rows_kv() * s.topk * 4);  // + lse partials
}
size_t ws_fwd(const Shape& s) {
  const size_t parts = (size_t)s.rows_kv() * s.topk * s.G;
  return plan_bytes(s) + align256(parts * s.d * 2) + align256(parts * 4);
}

}  // namespace

int finish(cudaError_t e) { return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA; }
size_t ws_index_bytes(const Shape& s) { return ws_index(s); }
size_t ws_fwd_bytes(const Shape& s) { return ws_fwd(s); }

int check_index_args(const Shape& s, const void* q_idx, const void* k_idx,
                     const int32_t* block_idx) {
  if (!q_idx || !k_idx || !block_idx) return MSA_ERR_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(block_idx)) return MSA_ERR_ARG;
  // selection keeps at most kMaxSelect candidates; more slots only for the dense set
  if (s.topk > kMaxSelect && s.topk < s.nb) return MSA_ERR_UNSUPPORTED;
  return MSA_OK;
}

int check_fwd_args(const void* q, const void* k, const void* v, const int32_t* block_idx,
                   const void* o, const float* lse) {
  if (!q || !k || !v || !block_idx || !o || !lse) return MSA_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(block_idx) || !aligned16(o) ||
      !aligned16(lse))
    return MSA_ERR_ARG;
  return MSA_OK;
}

int check_bwd_args(const void* const* ptrs, int n) {
  for (int i = 0; i < n; ++i)
    if (!ptrs[i] || !aligned16(ptrs[i])) return MSA_ERR_ARG;
  return MSA_OK;
}

cudaError_t run_index(const Shape& s, const void* q_idx, const void* k_idx, int32_t* block_idx,
                      float* lse_idx, void* ws, const Ctx& cx, cudaStream_t st, void* plan) {
  cudaError_t e = launch_index_topk(s, q_idx, k_idx, block_idx, cx, st);
  if (e != cudaSuccess) return e;
  Plan pl;
  if (plan) {  // the step's shared plan, built once here
    const SharedPlan sp = shared_plan_carve(s, plan);
    if ((e = launch_shared_plan(s, block_idx, sp, cx, st)) != cudaSuccess) return e;
    pl = sp.idx;
  }
  if (!lse_idx) return cudaSuccess;
  float* lse_part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + plan_bytes(s));
  if (!plan) {
    pl = plan_carve(s, ws);
    if ((e = launch_plan(s, block_idx, 128, pl, cx, st)) != cudaSuccess) return e;
  }
  return launch_index_lse(s, q_idx, k_idx, block_idx, pl, lse_part, lse_idx, cx, st);
}

cudaError_t run_fwd(const Shape& s, const void* q, const void* k, const void* v,
                    const int32_t* block_idx, void* o, float* lse, void* ws, const Ctx& cx,
                    cudaStream_t st, void* plan) {
  uint8_t* w = static_cast<uint8_t*>(ws) + plan_bytes(s);
  const size_t parts = (size_t)s.rows_kv() * s.topk * s.G;
  __nv_bfloat16* o_part = reinterpret_cast<__nv_bfloat16*>(w);
  float* lse_part = reinterpret_cast<float*>(w + align256(parts * s.d * 2));
  Plan pl;
  cudaError_t e;
  if (plan) {
    const SharedPlan sp = shared_plan_carve(s, plan);
    e = launch_shared_plan_check(s, sp, cx, st);
    pl = sp.fwd;
  } else {
    pl = plan_carve(s, ws);
    e = launch_plan(s, block_idx, 128 / s.G, pl, cx, st);
  }
  if (e != cudaSuccess) return e;
  return launch_attn_fwd(s, q, k, v, block_idx, pl, o_part, lse_part, o, lse, cx, st);
}

namespace {

std::atomic<uint64_t> g_launches{0};
cudaEvent_t g_ev[4][2] = {};

}  // namespace

void note_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

void* current_context() {
  using GetCurrent = CUresult (*)(CUcontext*);
  static GetCurrent fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<GetCurrent>(ptr);
  });
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

int device_symbol_address(const void* symbol, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MSA_ERR_CUDA;
  struct Entry {
    const void* symbol;
    void* ctx;
    void* addr;
  };
  static Entry cache[64][4] = {};
  void* ctx = current_context();
  std::lock_guard<std::mutex> lk(g_sym_mu);
  Entry* slot = nullptr;
  for (Entry& e : cache[dev]) {
    if (e.symbol == symbol) {
      slot = &e;
      break;
    }
    if (!e.symbol && !slot) slot = &e;
  }
  if (!slot) return MSA_ERR_CUDA;  // more symbols than slots: a build error, not a user's
  if (!ctx || slot->symbol != symbol || slot->ctx != ctx || !slot->addr) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, symbol) != cudaSuccess || !a) return MSA_ERR_CUDA;
    slot->symbol = symbol;
    slot->addr = a;
    slot->ctx = current_context();  // the lookup makes the primary context current
  }
  *out = slot->addr;
  return MSA_OK;
}

int validate_problem(const msa_problem_t* p, Shape* s) { return check_problem(p, s); }
int device_ctx(Ctx* cx) { return make_ctx(cx); }

void kernel_event(int kernel, bool before, cudaStream_t st) {
  cudaEvent_t ev = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (kernel >= 0 && kernel < 4 && g_ev[kernel][0] && g_ev[kernel][1])
      ev = g_ev[kernel][before ? 0 : 1];
  }
  if (ev) cudaEventRecord(ev, st);
}


}  // namespace msa

using namespace msa;

extern "C" {

int msa_version(void) { return 10000; }

int msa_set_kernel_events(int kernel, cudaEvent_t start, cudaEvent_t stop) {
  if (kernel < 0 || kernel > 3) return MSA_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  g_ev[kernel][0] = (start && stop) ? start : nullptr;
  g_ev[kernel][1] = (start && stop) ? stop : nullptr;
  return MSA_OK;
}

uint64_t msa_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* msa_status_string(int code) {
  switch (code) {
    case MSA_OK: return "ok";
    case MSA_ERR_ARG: return "invalid argument (null or misaligned pointer, bad value)";
    case MSA_ERR_SHAPE: return "inconsistent problem sizes";
    case MSA_ERR_UNSUPPORTED: return "problem outside the supported set of this build";
    case MSA_ERR_WORKSPACE: return "workspace missing or too small";
    case MSA_ERR_CUDA: return "CUDA launch or runtime error";
    case MSA_ERR_DEVICE_TIMEOUT: return "a device-side wait ran out of time";
  }
  return "unknown status";
}

size_t msa_workspace_size(const msa_problem_t* p, int which) {
  Shape s;
  if (check_problem(p, &s) != MSA_OK) return 0;
  switch (which) {
    case MSA_WS_INDEX: return ws_index(s);
    case MSA_WS_FWD: return ws_fwd(s);
    case MSA_WS_BWD: return bwd_ws_bytes(s);
  }
  return 0;
}

int msa_debug_set(uint64_t wait_limit_ns, int flags) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_wait_ns = wait_limit_ns ? wait_limit_ns : kDefaultWaitNs;
  g_debug = flags;
  return MSA_OK;
}

int msa_get_device_status(cudaStream_t stream, int* status) {
  if (!status) return MSA_ERR_ARG;
  int* dp = nullptr;
  int rc = status_ptr(&dp);
  if (rc) return rc;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MSA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, dp, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MSA_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(dp, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return MSA_ERR_CUDA;
  *status = v;
  return MSA_OK;
}

int msa_index_topk(const msa_problem_t* p, const void* q_idx, const void* k_idx,
                   int32_t* block_idx, float* lse_idx, void* workspace, size_t workspace_bytes,
                   cudaStream_t stream) {
  Shape s;
  int rc = check_problem(p, &s);
  if (rc) return rc;
  if (s.B == 0 || s.N == 0) return MSA_OK;
  if ((rc = check_index_args(s, q_idx, k_idx, block_idx))) return rc;
  if (lse_idx) {
    if (!workspace || workspace_bytes < ws_index(s)) return MSA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return MSA_ERR_ARG;
  }
  Ctx cx;
  if ((rc = make_ctx(&cx))) return rc;
  return finish(run_index(s, q_idx, k_idx, block_idx, lse_idx, workspace, cx, stream));
}

int msa_fwd(const msa_problem_t* p, const void* q, const void* k, const void* v,
            const int32_t* block_idx, void* o, float* lse, void* workspace,
            size_t workspace_bytes, cudaStream_t stream) {
  Shape s;
  int rc = check_problem(p, &s);
  if (rc) return rc;
  if (s.B == 0 || s.N == 0) return MSA_OK;
  if ((rc = check_fwd_args(q, k, v, block_idx, o, lse))) return rc;
  if (!workspace || workspace_bytes < ws_fwd(s)) return MSA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return MSA_ERR_ARG;
  Ctx cx;
  if ((rc = make_ctx(&cx))) return rc;
  return finish(run_fwd(s, q, k, v, block_idx, o, lse, workspace, cx, stream));
}

int msa_bwd(const msa_problem_t* p, const void* q, const void* k, const void* v, const void* o,
            const float* lse, const void* dO, const void* q_idx, const void* k_idx,
            const int32_t* block_idx, const float* lse_idx, float kl_weight, void* dq, void* dk,
            void* dv, void* dq_idx, void* dk_idx, float* kl_out, void* workspace,
            size_t workspace_bytes, cudaStream_t stream) {
  Shape s;
  int rc = check_problem(p, &s);
  if (rc) return rc;
  if (!isfinite(kl_weight)) return MSA_ERR_ARG;
  if (s.B == 0 || s.N == 0) {
    if (kl_out) return finish(cudaMemsetAsync(kl_out, 0, sizeof(float), stream));
    return MSA_OK;
  }
  const void* ins[] = {q, k, v, o, lse, dO, q_idx, k_idx, block_idx, lse_idx,
                       dq, dk, dv, dq_idx, dk_idx};
  if ((rc = check_bwd_args(ins, sizeof(ins) / sizeof(ins[0])))) return rc;
  if (!workspace || workspace_bytes < bwd_ws_bytes(s)) return MSA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return MSA_ERR_ARG;
  Ctx cx;
  if ((rc = make_ctx(&cx))) return rc;
  return finish(run_bwd(s, q, k, v, o, lse, dO, q_idx, k_idx, block_idx, lse_idx, kl_weight, dq,
                        dk, dv, dq_idx, dk_idx, kl_out, workspace, cx, stream));
}

size_t msa_plan_size(const msa_problem_t* p) {
  Shape s;
  if (check_problem(p, &s)) return 0;
  return shared_plan_bytes(s);
}

static int check_plan(const Shape& s, const void* plan, size_t plan_bytes) {
  if (!plan || (reinterpret_cast<uintptr_t>(plan) & 255) != 0) return MSA_ERR_ARG;
  if (plan_bytes < shared_plan_bytes(s)) return MSA_ERR_WORKSPACE;
  return MSA_OK;
}

int msa_index_topk_plan(const msa_problem_t* p, const void* q_idx, const void* k_idx,
                        int32_t* block_idx, float* lse_idx, void* plan, size_t plan_bytes,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  Shape s;
  int rc = check_problem(p, &s);
  if (rc) return rc;
  if (s.B == 0 || s.N == 0) return MSA_OK;
  if ((rc = check_index_args(s, q_idx, k_idx, block_idx))) return rc;
  if ((rc = check_plan(s, plan, plan_bytes))) return rc;
  if (lse_idx) {
    if (!workspace || workspace_bytes < ws_index(s)) return MSA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return MSA_ERR_ARG;
  }
  Ctx cx;
  if ((rc = make_ctx(&cx))) return rc;
  return finish(run_index(s, q_idx, k_idx, block_idx, lse_idx, workspace, cx, stream, plan));
}

int msa_fwd_plan(const msa_problem_t* p, const void* q, const void* k, const void* v,
                 const int32_t* block_idx, void* plan, size_t plan_bytes, void* o, float* lse,
                 void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  Shape s;
  int rc = check_problem(p, &s);
  if (rc) return rc;
  if (s.B == 0 || s.N == 0) return MSA_OK;
  if ((rc = check_fwd_args(q, k, v, block_idx, o, lse))) return rc;
  if ((rc = check_plan(s, plan, plan_bytes))) return rc;
  if (!workspace || workspace_bytes < ws_fwd(s)) return MSA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return MSA_ERR_ARG;
  Ctx cx;
  if ((rc = make_ctx(&cx))) return rc;
  return finish(run_fwd(s, q, k, v, block_idx, o, lse, workspace, cx, stream, plan));
}

int msa_bwd_plan(const msa_problem_t* p, const void* q, const void* k, const void* v, const void* o,
                 const float* lse, const void* dO, const void* q_idx, const void* k_idx,
                 const int32_t* block_idx, const float* lse_idx, void* plan, size_t plan_bytes,
                 float kl_weight, void* dq, void* dk, void* dv, void* dq_idx, void* dk_idx,
                 float* kl_out, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  Shape s;
  int rc = check_problem(p, &s);
  if (rc) return rc;
  if (!isfinite(kl_weight)) return MSA_ERR_ARG;
  if (s.B == 0 || s.N == 0) {
    if (kl_out) return finish(cudaMemsetAsync(kl_out, 0, sizeof(float), stream));
    return MSA_OK;
  }
  const void* ins[] = {q, k, v, o, lse, dO, q_idx, k_idx, block_idx, lse_idx,
                       dq, dk, dv, dq_idx, dk_idx};
  if ((rc = check_bwd_args(ins, sizeof(ins) / sizeof(ins[0])))) return rc;
  if ((rc = check_plan(s, plan, plan_bytes))) return rc;
  if (!workspace || workspace_bytes < bwd_ws_bytes(s)) return MSA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return MSA_ERR_ARG;
  Ctx cx;
  if ((rc = make_ctx(&cx))) return rc;
  return finish(run_bwd(s, q, k, v, o, lse, dO, q_idx, k_idx, block_idx, lse_idx, kl_weight, dq,
                        dk, dv, dq_idx, dk_idx, kl_out, workspace, cx, stream, plan));
}

}  // extern "C"
