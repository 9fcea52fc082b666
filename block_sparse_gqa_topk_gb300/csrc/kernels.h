// kernels.h -- host-side launchers of the MSA kernels (internal to libmsa.so).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "msa.h"

namespace msa {

// Slots per (b, g, i) row: up to kMaxSlots block ids.  Inverted-list entries pack
// (query << kSlotBits) | slot into a non-negative int (query < 2^23).  The block
// selection kernel keeps its candidates in registers and picks at most kMaxSelect
// blocks; more slots are used only by the dense set (every visible block, topk >= nb).
constexpr int kSlotBits = 8;
constexpr int kSlotMask = (1 << kSlotBits) - 1;
constexpr int kMaxSlots = 1 << kSlotBits;
constexpr int kMaxSelect = 32;
// Blocks per sequence the plan histograms in shared memory (the only plan path for
// packed variable-length batches).
constexpr int kPlanSmemBins = 16384;

// Row-chunk tables of a packed variable-length batch (written on the device by
// varlen_prepare): tab[k][b] = sum over sequences b' < b of ceil(len_b' / kVarlenChunk[k]),
// so work item w of a grid over chunks belongs to the last b with tab[k][b] <= w.
enum VarlenTable {
  kTabIndexUnit = 0,  // 256 queries: a pair of 128-query blocks of the index kernel
  kTabPlanCount = 1,  // the plan's counting CTAs
  kTabPlanFill = 2,   // the plan's fill CTAs (rows depend on topk)
  kTabRows64 = 3,     // 64 rows: the backward preprocess
  kNumVarlenTabs = 4
};

// Validated problem, with derived sizes.  A batch is either B sequences of N tokens
// (spans == nullptr; sequence b starts at token b*N) or a packed variable-length batch of
// B sequences of at most N tokens each, sequence b holding tokens spans[b].x .. spans[b].y-1
// of T (device arrays checked and written by varlen_prepare).
struct Shape {
  int B, N, H_q, H_kv, d, d_idx, Bk, topk, causal;
  float scale, scale_idx;
  int G;   // H_q / H_kv
  int nb;  // ceil(N / Bk): blocks of the longest sequence
  int64_t T = 0;                // tokens on the token axis (B*N for the fixed layout)
  const int2* spans = nullptr;  // [B] (start, end), packed batches only
  const int* tabs = nullptr;    // [kNumVarlenTabs][B + 1] row-chunk tables, packed only
  int64_t rows_kv() const { return T * H_kv; }            // (b, g, i) rows
  int64_t keys() const { return (int64_t)B * H_kv * nb; } // (b, g, block) lists
  bool packed() const { return spans != nullptr; }
  // extents of the token and batch axes of the TMA tensor maps
  uint64_t tma_tokens() const { return packed() ? (uint64_t)T : (uint64_t)N; }
  uint64_t tma_batches() const { return packed() ? 1u : (uint64_t)B; }
  const int* tab(VarlenTable k) const { return tabs ? tabs + (size_t)k * (B + 1) : nullptr; }
};

// Rows per chunk of each table (kTabPlanFill: the fill kernel's rows for this topk).
int varlen_chunk_rows(VarlenTable k, int topk);
// Work items of a grid over the chunks of table k: an upper bound the host can compute
// without reading the spans (sum of ceil(len / R) <= ceil(T / R) + B).
int64_t varlen_grid_items(const Shape& s, VarlenTable k);

// Per-call device context.
struct Ctx {
  int* status;      // device status word of the current device
  uint64_t wait_ns; // bound of every device-side wait
  int debug;        // msa_debug_set flags
  int num_sms;
};

// Inverted lists ("plan"): for every (b, g, block c), the (query, slot) pairs
// whose block set holds c, as a CSR over keys = (b*H_kv + g)*nb + c, and the
// split of every list into tiles of `qpt` queries.
struct Plan {
  int* cnt;      // [keys]      counts, reused as fill cursors
  int* off;      // [keys + 1]  CSR offsets into entries
  int* toff;     // [keys + 1]  tile offsets; toff[keys] = number of tiles
  int* entries;  // [rows_kv * topk]  (i << kSlotBits) | slot
};

size_t plan_bytes(const Shape& s);
Plan plan_carve(const Shape& s, void* ws);
cudaError_t launch_plan(const Shape& s, const int32_t* block_idx, int qpt, const Plan& pl,
                        const Ctx& cx, cudaStream_t st);

// A plan shared by the calls of one step, in a caller-owned buffer: a header naming the
// problem (written last by the build), the CSR with tiles of 128 queries (index LSE; the
// backward reads only the CSR) and a second tile split of 128 / G queries (forward).
constexpr int kPlanHeaderInts = 8;
constexpr size_t kPlanHeaderBytes = 256;
constexpr int kPlanMagic = 0x4D534150;
struct PlanHeader {
  int v[kPlanHeaderInts];
};
struct SharedPlan {
  int* hdr;
  Plan idx;  // tiles of 128 queries
  Plan fwd;  // the same CSR, tiles of 128 / G queries
};
PlanHeader plan_header(const Shape& s);
size_t shared_plan_bytes(const Shape& s);
SharedPlan shared_plan_carve(const Shape& s, void* buf);
cudaError_t launch_shared_plan(const Shape& s, const int32_t* block_idx, const SharedPlan& sp,
                               const Ctx& cx, cudaStream_t st);
cudaError_t launch_shared_plan_check(const Shape& s, const SharedPlan& sp, const Ctx& cx,
                                     cudaStream_t st);

// Index branch: tcgen05 scoring + block max-pool + register top-k -> block_idx.
cudaError_t launch_index_topk(const Shape& s, const void* q_idx, const void* k_idx,
                              int32_t* block_idx, const Ctx& cx, cudaStream_t st);

// Index LSE over the selected tokens (gathered, KV-outer) -> lse_idx.
cudaError_t launch_index_lse(const Shape& s, const void* q_idx, const void* k_idx,
                             const int32_t* block_idx, const Plan& pl, float* lse_part,
                             float* lse_idx, const Ctx& cx, cudaStream_t st);

// Main forward: gathered KV-outer partials, then the per-row combine.
cudaError_t launch_attn_fwd(const Shape& s, const void* q, const void* k, const void* v,
                            const int32_t* block_idx, const Plan& pl, __nv_bfloat16* o_part,
                            float* lse_part, void* o, float* lse, const Ctx& cx,
                            cudaStream_t st);

// Per-row merge of the forward's slot partials into o and lse.
cudaError_t launch_attn_fwd_combine(const Shape& s, const int32_t* block_idx,
                                    const __nv_bfloat16* o_part, const float* lse_part, void* o,
                                    float* lse, cudaStream_t st);

// FP8 (E4M3) forward, d = 128: per-block quantiser of k (layout kept) or v (transposed
// per block, v8t [B][H_kv][nb][d][128]) and the tcgen05 kind::f8f6f4 partials kernel.
cudaError_t launch_quantize_blocks_fp8(const Shape& s, const void* x, uint8_t* x8, float* scale,
                                       bool transpose, cudaStream_t st);
cudaError_t launch_attn_fwd_fp8_tc(const Shape& s, const uint8_t* q8, const float* q_scale,
                                   const uint8_t* k8, const float* k_scale, const uint8_t* v8t,
                                   const float* v_scale, const Plan& pl, __nv_bfloat16* o_part,
                                   float* lse_part, const Ctx& cx, cudaStream_t st);

// tcgen05 gathered forward kernel (partials only; launch_attn_fwd adds the combine).
cudaError_t launch_attn_fwd_tc(const Shape& s, const void* q, const void* k, const void* v,
                               const Plan& pl, __nv_bfloat16* o_part, float* lse_part,
                               const Ctx& cx, cudaStream_t st);

// tcgen05 fused backward tile kernel (dk, dv written; dq, dq_idx, dk_idx as partials).
cudaError_t launch_attn_bwd_tc(const Shape& s, const void* q, const void* k, const void* v,
                               const void* dO, const float* lse, const float* Dv,
                               const void* q_idx, const void* k_idx, const float* lse_idx,
                               float kl_weight, const Plan& pl, __nv_bfloat16* dq_part,
                               __nv_bfloat16* dqi_part, float* dki_part, double* kl_acc, void* dk,
                               void* dv, const Ctx& cx, cudaStream_t st);

// Backward pieces.
struct BwdBufs {
  float* D;          // [B][H_q][N]
  float* dq_acc;     // [B][N][H_q][d]
  float* dk_acc;     // [B][N][H_kv][d]
  float* dv_acc;     // [B][N][H_kv][d]
  float* dqi_acc;    // [B][N][H_kv][d_idx]
  float* dki_acc;    // [B][N][d_idx]
  double* kl_acc;    // 1
};
cudaError_t launch_attn_bwd(const Shape& s, const void* q, const void* k, const void* v,
                            const void* o, const float* lse, const void* dO, const void* q_idx,
                            const void* k_idx, const int32_t* block_idx, const float* lse_idx,
                            float kl_weight, const Plan& pl, const BwdBufs& bb, void* dq,
                            void* dk, void* dv, void* dq_idx, void* dk_idx, float* kl_out,
                            const Ctx& cx, cudaStream_t st);

// TMA descriptor encoding through the driver entry point (no libcuda link).
bool encode_tiled(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base,
                  const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                  CUtensorMapSwizzle swz);

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Shape checks shared by every entry point (msa_api.cu) and the device context of the
// current device (status word, wait limit, SM count; MSA_ERR_UNSUPPORTED off sm_103).
int validate_problem(const msa_problem_t* p, Shape* s);
int device_ctx(Ctx* cx);
int finish(cudaError_t e);  // MSA_OK or MSA_ERR_CUDA

// Argument checks and call sequences of the three training calls, shared by the fixed
// and the packed variable-length entry points (msa_api.cu, attn_bwd.cu).  ws is the
// call's workspace of ws_*_bytes(s) bytes, 256-byte aligned.
size_t ws_index_bytes(const Shape& s);
size_t ws_fwd_bytes(const Shape& s);
size_t bwd_ws_bytes(const Shape& s);
int check_index_args(const Shape& s, const void* q_idx, const void* k_idx,
                     const int32_t* block_idx);
int check_fwd_args(const void* q, const void* k, const void* v, const int32_t* block_idx,
                   const void* o, const float* lse);
int check_bwd_args(const void* const* ptrs, int n);
// With `plan` (a shared plan buffer), run_index builds it and the others read it (after
// a header check) instead of building their own in the workspace.
cudaError_t run_index(const Shape& s, const void* q_idx, const void* k_idx, int32_t* block_idx,
                      float* lse_idx, void* ws, const Ctx& cx, cudaStream_t st,
                      void* plan = nullptr);
cudaError_t run_fwd(const Shape& s, const void* q, const void* k, const void* v,
                    const int32_t* block_idx, void* o, float* lse, void* ws, const Ctx& cx,
                    cudaStream_t st, void* plan = nullptr);
cudaError_t run_bwd(const Shape& s, const void* q, const void* k, const void* v, const void* o,
                    const float* lse, const void* dO, const void* q_idx, const void* k_idx,
                    const int32_t* block_idx, const float* lse_idx, float kl_weight, void* dq,
                    void* dk, void* dv, void* dq_idx, void* dk_idx, float* kl_out, void* ws,
                    const Ctx& cx, cudaStream_t st, void* plan = nullptr);

// Launch bookkeeping (msa_api.cu): counts launches and records the profiling
// events of msa_set_kernel_events around the named kernels.
void note_launch(int n = 1);

// The calling thread's current CUDA context (the driver's cuCtxGetCurrent, reached
// through the runtime's entry-point query), or nullptr.
void* current_context();
// Device address of a module-scope __device__ variable on the current device.  The
// address is cached per (device, context) and looked up again when the context
// changes (after cudaDeviceReset the module is loaded anew and the old address is
// stale).  A first lookup may load the module: do it before any stream capture.
int device_symbol_address(const void* symbol, void** out);
void kernel_event(int kernel, bool before, cudaStream_t st);

}  // namespace msa
