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

// Validated problem, with derived sizes.
struct Shape {
  int B, N, H_q, H_kv, d, d_idx, Bk, topk, causal;
  float scale, scale_idx;
  int G;   // H_q / H_kv
  int nb;  // ceil(N / Bk)
  int64_t rows_kv() const { return (int64_t)B * H_kv * N; }  // (b, g, i) rows
  int64_t keys() const { return (int64_t)B * H_kv * nb; }    // (b, g, block) lists
};

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
