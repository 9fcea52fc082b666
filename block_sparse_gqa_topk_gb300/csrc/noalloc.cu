// noalloc.cu -- msa_index_topk_noalloc: the index branch for callers that cannot
// allocate device memory.
//
// msa_index_topk needs a caller-owned workspace when it also computes lse_idx (the
// inverted lists and the per-slot partial LSEs live there).  Some callers have no
// way to provide one: code embedded in a host framework that owns every device
// allocation and exposes no allocator to plug-ins, or a service that fixes its
// device memory footprint at start-up and forbids allocation afterwards.  This entry
// point gives them the same computation with the scratch taken from a fixed array
// compiled into the library instead.
//
// The array is a file-scope static __device__ buffer of kScratchBytes (64 MiB).
// Every GPU that loads the library holds it until the process exits.  Host code
// cannot use the array's name as a device address (on the host it names a shadow
// variable), so the first call on each device, with that device current, looks the
// address up with cudaGetSymbolAddress and caches it per (device, context); make
// that first call before any stream capture.  A new context on the device (after
// cudaDeviceReset, for instance) loads the module again, and the next call looks the
// address up again.  All calls on a device share the one array and it keeps the last
// call's contents: each call zeroes the counters it needs with a cudaMemsetAsync on
// the caller's stream (a memset into the array, not an allocation), and calls whose
// executions overlap on the GPU (different streams, no ordering) race on it and must
// not be issued.  The stream must belong to the current device, as for every other
// entry point.
#include <mutex>

#include "kernels.h"

namespace msa {
namespace {

constexpr size_t kScratchBytes = 64ull << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_scratch_mu;
struct ScratchAddr {
  void* ctx;
  void* ptr;
};
ScratchAddr g_scratch_addr[64] = {};

// Device address of the scratch array on the current device, looked up once per
// (device, context).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MSA_ERR_CUDA;
  void* ctx = current_context();
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  ScratchAddr& e = g_scratch_addr[dev];
  if (!ctx || e.ctx != ctx || !e.ptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MSA_ERR_CUDA;
    e.ptr = p;
    e.ctx = current_context();  // the lookup makes the primary context current
  }
  *out = e.ptr;
  return MSA_OK;
}

}  // namespace
}  // namespace msa

extern "C" {

size_t msa_noalloc_scratch_bytes(void) { return msa::kScratchBytes; }

int msa_index_topk_noalloc(const msa_problem_t* p, const void* q_idx, const void* k_idx,
                           int32_t* block_idx, float* lse_idx, cudaStream_t stream) {
  if (!lse_idx)  // block selection alone needs no scratch
    return msa_index_topk(p, q_idx, k_idx, block_idx, nullptr, nullptr, 0, stream);
  const size_t need = msa_workspace_size(p, MSA_WS_INDEX);
  if (need == 0)  // invalid problem: let the main entry point name the error
    return msa_index_topk(p, q_idx, k_idx, block_idx, lse_idx, nullptr, 0, stream);
  if (need > msa::kScratchBytes) return MSA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int rc = msa::scratch_address(&scratch);
  if (rc != MSA_OK) return rc;
  return msa_index_topk(p, q_idx, k_idx, block_idx, lse_idx, scratch, msa::kScratchBytes, stream);
}

}  // extern "C"
