// plan.cu -- inverted lists of the block selection.
//
// The main branch runs KV-outer: for every (batch, group, key block c) it gathers
// the queries whose block set holds c, packs them into 128-row tiles (queries x
// group heads) and runs one dense tile per 128 rows.  This is the query-gather
// reparameterisation of block-sparse attention described for both prior kernels:
// the MoBA-style varlen view of Flash-MSA (tech.kuratif.com ¶7, deephorus.pages.dev
// ¶4) and fmha_sm100's KV-outer query gather (7minutos.es, "El codiseño del
// kernel", second idea).  This file builds the lists from block_idx:
//   count  -> per-list sizes (shared-memory histograms per row chunk),
//   scan   -> CSR offsets and tile offsets (one CTA, decoupled chunks),
//   fill   -> (query << kSlotBits | slot) entries.
// HBM-bound integer work: block_idx is read twice, entries written once.
#include "common.cuh"
#include "kernels.h"

#include <algorithm>

namespace msa {
namespace {

__global__ void plan_count_kernel(const int32_t* __restrict__ block_idx, int64_t rows, int topk,
                                  int N, int nb, int* __restrict__ cnt, int* status) {
  const int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (t >= rows * topk) return;
  const int c = block_idx[t];
  if (c < 0) return;
  if (c >= nb) {  // not a block of this sequence: record it, touch nothing
    set_status(status, MSA_ERR_ARG);
    return;
  }
  const int64_t r = t / topk;  // (b*H_kv + g)*N + i
  const int64_t bg = r / N;
  atomicAdd(&cnt[bg * nb + c], 1);
}

// Exclusive scans of cnt (-> off) and of ceil(cnt / qpt) (-> toff) over all keys,
// then zeroes cnt for use as the fill cursor.  One CTA of 1024 threads.
__global__ void __launch_bounds__(1024) plan_scan_kernel(int* __restrict__ cnt,
                                                         int* __restrict__ off,
                                                         int* __restrict__ toff, int64_t keys,
                                                         int qpt) {
  __shared__ int s_a[32], s_b[32];
  __shared__ int carry_a, carry_b;
  if (threadIdx.x == 0) {
    carry_a = 0;
    carry_b = 0;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int64_t base = 0; base < keys; base += 1024) {
    const int64_t k = base + threadIdx.x;
    const int a = k < keys ? cnt[k] : 0;
    const int b = (a + qpt - 1) / qpt;
    int ia = a, ib = b;  // inclusive warp scans
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int xa = __shfl_up_sync(0xffffffffu, ia, o);
      const int xb = __shfl_up_sync(0xffffffffu, ib, o);
      if (lane >= o) {
        ia += xa;
        ib += xb;
      }
    }
    if (lane == 31) {
      s_a[warp] = ia;
      s_b[warp] = ib;
    }
    __syncthreads();
    if (warp == 0) {
      int wa = s_a[lane], wb = s_b[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int xa = __shfl_up_sync(0xffffffffu, wa, o);
        const int xb = __shfl_up_sync(0xffffffffu, wb, o);
        if (lane >= o) {
          wa += xa;
          wb += xb;
        }
      }
      s_a[lane] = wa;  // inclusive over warps
      s_b[lane] = wb;
    }
    __syncthreads();
    const int pa = carry_a + (warp ? s_a[warp - 1] : 0) + ia - a;
    const int pb = carry_b + (warp ? s_b[warp - 1] : 0) + ib - b;
    if (k < keys) {
      off[k] = pa;
      toff[k] = pb;
      cnt[k] = 0;
    }
    __syncthreads();
    if (threadIdx.x == 1023) {
      carry_a = pa + a;
      carry_b = pb + b;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    off[keys] = carry_a;
    toff[keys] = carry_b;
  }
}

__global__ void plan_fill_kernel(const int32_t* __restrict__ block_idx, int64_t rows, int topk,
                                 int N, int nb, const int* __restrict__ off,
                                 int* __restrict__ cursor, int* __restrict__ entries) {
  const int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (t >= rows * topk) return;
  const int c = block_idx[t];
  if (c < 0 || c >= nb) return;
  const int64_t r = t / topk;
  const int slot = (int)(t - r * topk);
  const int64_t bg = r / N;
  const int i = (int)(r - bg * N);
  const int64_t key = bg * nb + c;
  const int pos = off[key] + atomicAdd(&cursor[key], 1);
  entries[pos] = (i << kSlotBits) | slot;
}

// Shared-memory count: one CTA takes kRowsPerCta consecutive rows of one (b, g),
// histograms their block ids in shared memory and touches global memory once per
// non-empty bin instead of once per entry.  Used, with the sorting fill above, when
// the nb-bin histogram fits in smem.
constexpr int kRowsPerCta = 1024;
constexpr int kSmemBins = kPlanSmemBins;

__global__ void plan_count_smem_kernel(const int32_t* __restrict__ block_idx,
                                       const int2* __restrict__ spans, const int* __restrict__ tab,
                                       int B, int N, int H_kv, int topk, int nb,
                                       int* __restrict__ cnt, int* status) {
  extern __shared__ int hist[];
  // CTA -> (sequence b, group g, chunk of kRowsPerCta rows)
  const int g = blockIdx.x % H_kv;
  int b, chunk;
  if (!chunk_item(tab, B, (N + kRowsPerCta - 1) / kRowsPerCta, blockIdx.x / H_kv, &b, &chunk))
    return;
  const SeqSpan sp = seq_span(spans, b, N);
  const int64_t bg = (int64_t)b * H_kv + g;
  const int i0 = chunk * kRowsPerCta;
  const int i1 = min(sp.len, i0 + kRowsPerCta);
  for (int c = threadIdx.x; c < nb; c += blockDim.x) hist[c] = 0;
  __syncthreads();
  const int32_t* src = block_idx + (sp.t0 * H_kv + (int64_t)g * sp.len + i0) * topk;
  const int n = (i1 - i0) * topk;
  for (int e0 = threadIdx.x; e0 < n; e0 += 8 * blockDim.x) {
    int cv[8];  // eight loads in flight before the histogram updates
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = e0 + u * blockDim.x;
      cv[u] = e < n ? __ldg(&src[e]) : -1;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int c = cv[u];
      if (c < 0) continue;
      if (c >= nb) {
        set_status(status, MSA_ERR_ARG);
        continue;
      }
      atomicAdd(&hist[c], 1);
    }
  }
  __syncthreads();
  for (int c = threadIdx.x; c < nb; c += blockDim.x)
    if (hist[c]) atomicAdd(&cnt[bg * nb + c], hist[c]);
}

// Fill as a counting sort in shared memory: one CTA of kFillThreads takes `rows`
// consecutive rows of one (b, g) (rows * topk <= kFillEntries entries), loads their
// block ids into registers at once, histograms them, reserves one range of the global
// list per non-empty bin, places each entry at its bin-ordered position in shared memory
// (block id and entry index in one word), and writes the entries out in that order, so
// consecutive threads write consecutive slots of a bin's range.
constexpr int kFillThreads = 512;
constexpr int kFillEntries = 16384;  // entry index < 2^16, block id < kSmemBins <= 2^16
constexpr int kFillPer = kFillEntries / kFillThreads;

__global__ void __launch_bounds__(kFillThreads)
    plan_fill_sort_kernel(const int32_t* __restrict__ block_idx, const int2* __restrict__ spans,
                          const int* __restrict__ tab, int B, int N, int H_kv, int topk, int nb,
                          int rows, const int* __restrict__ off, int* __restrict__ cursor,
                          int* __restrict__ entries) {
  extern __shared__ int fill_smem[];
  int* hist = fill_smem;        // [nb] counts, then the bin's next position in `stage`
  int* delta = fill_smem + nb;  // [nb] global slot minus position in `stage`, per bin
  uint32_t* stage = reinterpret_cast<uint32_t*>(fill_smem + 2 * nb);  // (c << 16 | e), bin order
  __shared__ int s_warp[kFillThreads / 32];
  const int g = blockIdx.x % H_kv;
  int b, chunk;
  if (!chunk_item(tab, B, (N + rows - 1) / rows, blockIdx.x / H_kv, &b, &chunk)) return;
  const SeqSpan sp = seq_span(spans, b, N);
  const int64_t bg = (int64_t)b * H_kv + g;
  const int i0 = chunk * rows;
  const int i1 = min(sp.len, i0 + rows);
  const int32_t* src = block_idx + (sp.t0 * H_kv + (int64_t)g * sp.len + i0) * topk;
  const int n = (i1 - i0) * topk;
  int cv[kFillPer];  // block id of entry threadIdx.x + u kFillThreads, -1 if none
#pragma unroll
  for (int u = 0; u < kFillPer; ++u) {
    const int e = threadIdx.x + u * kFillThreads;
    const int c = e < n ? __ldg(&src[e]) : -1;
    cv[u] = c < nb ? c : -1;
  }
  for (int c = threadIdx.x; c < nb; c += kFillThreads) hist[c] = 0;
  __syncthreads();
#pragma unroll
  for (int u = 0; u < kFillPer; ++u)
    if (cv[u] >= 0) atomicAdd(&hist[cv[u]], 1);
  __syncthreads();
  // exclusive scan of the counts: thread t owns bins [t per, t per + per)
  const int per = (nb + kFillThreads - 1) / kFillThreads;
  const int c0 = min(nb, (int)threadIdx.x * per), c1 = min(nb, c0 + per);
  int tot = 0;
  for (int c = c0; c < c1; ++c) tot += hist[c];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int nw = kFillThreads / 32;
  int incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += x;
    }
    if (lane < nw) s_warp[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int total = s_warp[nw - 1];
  int run = (warp ? s_warp[warp - 1] : 0) + incl - tot;
  for (int c = c0; c < c1; ++c) {
    const int h = hist[c];
    delta[c] = h ? off[bg * nb + c] + atomicAdd(&cursor[bg * nb + c], h) - run : 0;
    hist[c] = run;
    run += h;
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < kFillPer; ++u)
    if (cv[u] >= 0)
      stage[atomicAdd(&hist[cv[u]], 1)] =
          ((uint32_t)cv[u] << 16) | (uint32_t)(threadIdx.x + u * kFillThreads);
  __syncthreads();
  for (int q = threadIdx.x; q < total; q += kFillThreads) {
    const uint32_t w = stage[q];
    const int c = (int)(w >> 16), e = (int)(w & 0xFFFFu);
    const int r = e / topk;
    entries[delta[c] + q] = ((i0 + r) << kSlotBits) | (e - r * topk);
  }
}

// Tile offsets of an existing CSR for a second tile size (counts from the offsets), then
// the shared plan's header, written last so that it marks a complete plan.  One block.
__global__ void __launch_bounds__(1024) plan_retile_kernel(const int* __restrict__ off,
                                                           int* __restrict__ toff, int64_t keys,
                                                           int qpt, int* __restrict__ hdr,
                                                           PlanHeader h) {
  __shared__ int s_w[32];
  __shared__ int carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int64_t base = 0; base < keys; base += 1024) {
    const int64_t k = base + threadIdx.x;
    const int n = k < keys ? __ldg(&off[k + 1]) - __ldg(&off[k]) : 0;
    int x = (n + qpt - 1) / qpt;  // inclusive warp scan of the tile counts
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_w[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = s_w[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      s_w[lane] = w;
    }
    __syncthreads();
    const int before = carry + (warp > 0 ? s_w[warp - 1] : 0);
    if (k < keys) toff[k + 1] = before + x;
    if (k == 0) toff[0] = 0;
    __syncthreads();
    if (threadIdx.x == 1023) carry = before + x;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    __threadfence();
#pragma unroll
    for (int i = 0; i < kPlanHeaderInts; ++i) hdr[i] = h.v[i];
  }
}

// A shared plan handed to a call: if its header does not name this problem, record
// MSA_ERR_ARG, clear the header (the buffer no longer holds a plan) and empty its lists
// (offsets and tile offsets all 0), so the kernels that read it do no work and never
// index past its arrays.  A block that reads the header after block 0 cleared it sees a
// mismatch too.
__global__ void plan_check_kernel(int* hdr, PlanHeader want, int* off, int* toff, int* toff2,
                                  int64_t n, int* status) {
  bool same = true;
#pragma unroll
  for (int i = 0; i < kPlanHeaderInts; ++i)
    same = same && (reinterpret_cast<volatile int*>(hdr)[i] == want.v[i]);
  if (same) return;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    set_status(status, MSA_ERR_ARG);
#pragma unroll
    for (int i = 0; i < kPlanHeaderInts; ++i) hdr[i] = 0;
  }
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    off[i] = 0;
    toff[i] = 0;
    toff2[i] = 0;
  }
}

}  // namespace

int varlen_chunk_rows(VarlenTable k, int topk) {
  switch (k) {
    case kTabIndexUnit: return 256;  // a pair of 128-query blocks
    case kTabPlanCount: return kRowsPerCta;
    case kTabRows64: return 64;
    default: return topk >= kFillEntries ? 1 : kFillEntries / topk;
  }
}

int64_t varlen_grid_items(const Shape& s, VarlenTable k) {
  const int64_t r = varlen_chunk_rows(k, s.topk);
  return (s.T + r - 1) / r + s.B;
}

size_t plan_bytes(const Shape& s) {
  const size_t keys = (size_t)s.keys();
  return align256(keys * 4) + 2 * align256((keys + 1) * 4) +
         align256((size_t)s.rows_kv() * s.topk * 4);
}

Plan plan_carve(const Shape& s, void* ws) {
  const size_t keys = (size_t)s.keys();
  uint8_t* p = static_cast<uint8_t*>(ws);
  Plan pl;
  pl.cnt = reinterpret_cast<int*>(p);
  p += align256(keys * 4);
  pl.off = reinterpret_cast<int*>(p);
  p += align256((keys + 1) * 4);
  pl.toff = reinterpret_cast<int*>(p);
  p += align256((keys + 1) * 4);
  pl.entries = reinterpret_cast<int*>(p);
  return pl;
}

PlanHeader plan_header(const Shape& s) {
  PlanHeader h;
  h.v[0] = kPlanMagic;
  h.v[1] = s.B;
  h.v[2] = s.N;
  h.v[3] = s.H_kv;
  h.v[4] = s.nb;
  h.v[5] = s.topk;
  h.v[6] = s.G;
  h.v[7] = (int)(s.T & 0x7fffffff);
  return h;
}

size_t shared_plan_bytes(const Shape& s) {
  return kPlanHeaderBytes + plan_bytes(s) + align256(((size_t)s.keys() + 1) * 4);
}

SharedPlan shared_plan_carve(const Shape& s, void* buf) {
  uint8_t* p = static_cast<uint8_t*>(buf);
  SharedPlan sp;
  sp.hdr = reinterpret_cast<int*>(p);
  sp.idx = plan_carve(s, p + kPlanHeaderBytes);
  sp.fwd = sp.idx;
  sp.fwd.toff = reinterpret_cast<int*>(p + kPlanHeaderBytes + plan_bytes(s));
  return sp;
}

cudaError_t launch_shared_plan(const Shape& s, const int32_t* block_idx, const SharedPlan& sp,
                               const Ctx& cx, cudaStream_t st) {
  // an interrupted build leaves no valid header behind
  cudaError_t e = cudaMemsetAsync(sp.hdr, 0, kPlanHeaderInts * sizeof(int), st);
  if (e != cudaSuccess) return e;
  if ((e = launch_plan(s, block_idx, 128, sp.idx, cx, st)) != cudaSuccess) return e;
  plan_retile_kernel<<<1, 1024, 0, st>>>(sp.idx.off, sp.fwd.toff, s.keys(), 128 / s.G, sp.hdr,
                                         plan_header(s));
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_shared_plan_check(const Shape& s, const SharedPlan& sp, const Ctx& cx,
                                     cudaStream_t st) {
  const int64_t n = s.keys() + 1;
  const unsigned grid = (unsigned)std::min<int64_t>((n + 255) / 256, 4 * (int64_t)cx.num_sms);
  plan_check_kernel<<<grid, 256, 0, st>>>(sp.hdr, plan_header(s), sp.idx.off, sp.idx.toff,
                                          sp.fwd.toff, n, cx.status);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_plan(const Shape& s, const int32_t* block_idx, int qpt, const Plan& pl,
                        const Ctx& cx, cudaStream_t st) {
  const int64_t keys = s.keys();
  const int64_t n = s.rows_kv() * s.topk;
  cudaError_t e = cudaMemsetAsync(pl.cnt, 0, (size_t)keys * 4, st);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)((n + 255) / 256);
  const bool smem_bins = s.nb <= kSmemBins;
  if (s.packed() && !smem_bins) return cudaErrorNotSupported;  // callers reject this first
  const int64_t chunks = (s.N + kRowsPerCta - 1) / kRowsPerCta;
  const unsigned grid_s = (unsigned)(
      s.H_kv * (s.packed() ? varlen_grid_items(s, kTabPlanCount) : (int64_t)s.B * chunks));
  const size_t hist_bytes = (size_t)s.nb * sizeof(int);
  const int fill_rows = varlen_chunk_rows(kTabPlanFill, s.topk);
  const unsigned grid_f = (unsigned)(
      s.H_kv * (s.packed() ? varlen_grid_items(s, kTabPlanFill)
                           : (int64_t)s.B * ((s.N + fill_rows - 1) / fill_rows)));
  const size_t fill_bytes = 2 * hist_bytes + (size_t)fill_rows * s.topk * sizeof(uint32_t);
  if (n > 0 && smem_bins) {
    if (hist_bytes > 48 * 1024)
      cudaFuncSetAttribute(plan_count_smem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)hist_bytes);
    if (fill_bytes > 48 * 1024)
      cudaFuncSetAttribute(plan_fill_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)fill_bytes);
    plan_count_smem_kernel<<<grid_s, 512, hist_bytes, st>>>(
        block_idx, s.spans, s.tab(kTabPlanCount), s.B, s.N, s.H_kv, s.topk, s.nb, pl.cnt,
        cx.status);
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  } else if (n > 0) {
    plan_count_kernel<<<grid, 256, 0, st>>>(block_idx, s.rows_kv(), s.topk, s.N, s.nb, pl.cnt,
                                            cx.status);
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  plan_scan_kernel<<<1, 1024, 0, st>>>(pl.cnt, pl.off, pl.toff, keys, qpt);
  note_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (n > 0 && smem_bins) {
    plan_fill_sort_kernel<<<grid_f, kFillThreads, fill_bytes, st>>>(
        block_idx, s.spans, s.tab(kTabPlanFill), s.B, s.N, s.H_kv, s.topk, s.nb, fill_rows,
        pl.off, pl.cnt, pl.entries);
    note_launch();
    e = cudaGetLastError();
  } else if (n > 0) {
    plan_fill_kernel<<<grid, 256, 0, st>>>(block_idx, s.rows_kv(), s.topk, s.N, s.nb, pl.off,
                                           pl.cnt, pl.entries);
    note_launch();
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace msa
