// index_lse.cu -- log-sum-exp of the index branch over each query's selected tokens,
// on the 5th-generation tensor cores.
//
// Method: the index distribution of a query row is the softmax of its scaled
// index scores over the tokens of its k selected blocks, the student side of the
// KL alignment loss (MSA summary, 7minutos.es, "Cómo se entrena MSA" ¶1-2).  The
// top-k never computes it (the selection is exp-free, "El codiseño del kernel");
// its normaliser is recomputed afterwards over the selected blocks only
// ("Accelerating Million-Token Training", deephorus.pages.dev, ¶4): this file.
//
// Work unit: a tile is one key block c of one (batch, group) and up to 128 of the
// queries whose block set holds c (the inverted lists of plan.cu with 128 queries
// per tile).  Per CTA (persistent, a contiguous range of tiles):
//   warps 12-15 loaders: gather the tile's 128 q_idx rows with cp.async into a
//               4-stage ring in the swizzled K-major layout tcgen05 reads; one
//               thread TMA-loads the block's k_idx tile into a 2-deep buffer;
//   warp 16     TMEM owner + one MMA thread: S = Q_idx K_idx^T (128 x 128, K = d_idx)
//               into a 4-slot TMEM ring;
//   warps 0-11  three warpgroups taking every third tile (thread = row = TMEM lane):
//               tcgen05.ld the row's 128 scores, causal mask, max, exp2 sum, and the
//               partial lse of (row, slot).
// Loaders and softmax warps fetch a tile's key and entries one tile ahead of its use.
// A second kernel merges the k partials of every row.  The exp2 throughput of the
// SM bounds the first kernel: 128 x 128 exponentials per tile.
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace msa {
namespace {

constexpr int kSoftWG = 3;      // softmax warpgroups, taking every third tile
constexpr int kLoadWarp0 = 4 * kSoftWG;      // 4 loader warps
constexpr int kMmaWarp = kLoadWarp0 + 4;     // MMA + TMEM owner
constexpr int kThreads = 32 * (kMmaWarp + 1);
constexpr int kLoadThreads = 128;
constexpr int kQStages = 4;
constexpr int kSlots = 4;      // TMEM score slots of 128 fp32 columns
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

template <int DI>
struct LseLayout {
  static constexpr int kRowB = DI * 2;                // 64 or 128 bytes per row
  static constexpr int kTile = 128 * kRowB;           // one 128-row operand
  static constexpr int kK = 0;                        // 2 k_idx buffers
  static constexpr int kQ = 2 * kTile;                // kQStages q_idx tiles
  static constexpr int kBar = kQ + kQStages * kTile;
  // kfull[2], kempty[2], qfull[kQStages], qempty[kQStages], sfull[kSlots],
  // tfree[kSlots], mmadone
  static constexpr int kNumBars = 4 + 2 * kQStages + 2 * kSlots + 1;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  // >= 116 KB so that one CTA (and its 512-column TMEM allocation) owns an SM
  static constexpr int kAlloc = (kBytes + 1024 > 118 * 1024) ? kBytes + 1024 : 118 * 1024;
};

struct LseParams {
  const __nv_bfloat16* q_idx;  // [T][H_kv][DI]
  const int2* spans;           // packed batches: (start, end) per sequence
  const int* off;
  const int* toff;
  const int* entries;
  float* lse_part;             // [(t0*H_kv + g*len + i)*topk + slot]
  int64_t keys;
  int N, H_kv, nb, topk;
  float scale_log2;            // scale_idx * log2(e)
  uint64_t wait_ns;
  int* status;
};

__device__ __forceinline__ int lse_find_key(const int* __restrict__ toff, int64_t keys, int t) {
  int64_t lo = 0, hi = keys - 1;
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) >> 1;
    if (__ldg(&toff[mid]) <= t) lo = mid; else hi = mid - 1;
  }
  return (int)lo;
}

// Key of tile t, given that the tiles of a CTA are visited in increasing order.
struct Cursor {
  int key = -1;
  __device__ __forceinline__ int at(const int* __restrict__ toff, int64_t keys, int t) {
    if (key < 0) {
      key = lse_find_key(toff, keys, t);
    } else {
      while (key + 1 < keys && __ldg(&toff[key + 1]) <= t) ++key;
    }
    return key;
  }
};

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <int DI>
__global__ void __launch_bounds__(kThreads, 1)
    index_lse_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const LseParams p) {
  using L = LseLayout<DI>;
  constexpr int RB = L::kRowB;
  constexpr int CH = DI / 8;  // 16-byte chunks per row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sK = smem + L::kK;
  uint8_t* sQ = smem + L::kQ;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* kfull = bars;                 // [2] k_idx tile landed
  uint64_t* kempty = bars + 2;            // [2] last MMA of the block retired
  uint64_t* qfull = bars + 4;             // [kQStages] q rows gathered
  uint64_t* qempty = qfull + kQStages;    // [kQStages] MMA done reading
  uint64_t* sfull = qempty + kQStages;    // [kSlots] scores in TMEM
  uint64_t* tfree = sfull + kSlots;       // [kSlots] scores read out
  uint64_t* mmadone = tfree + kSlots;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = __ldg(&p.toff[p.keys]);
  const int per = (total + gridDim.x - 1) / gridDim.x;
  const int t_begin = blockIdx.x * per;
  const int t_end = min(total, t_begin + per);
  const int n_tiles = max(0, t_end - t_begin);

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 1);
    }
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&qfull[s], kLoadThreads);
      mbar_init(&qempty[s], 1);
    }
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&sfull[s], 1);
      mbar_init(&tfree[s], 4);  // one arrive per warp of the reading warpgroup
    }
    mbar_init(mmadone, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (n_tiles > 0) {
    if (warp >= kLoadWarp0 && warp < kMmaWarp) {
      // ================================ loaders =================================
      // Per tile: (new block) TMA its k_idx tile -> gather q(u), whose stage completes
      // through cp.async arrivals as the rows land.  The k_idx wait is on the block two
      // keys back: its last tile is at most u-2, whose rows were issued in an earlier
      // iteration, and the MMA thread releases the buffer right after that tile's MMA.
      const int lt = threadIdx.x - 32 * kLoadWarp0;
      Cursor kc;
      int prev_key = -1, k_loads = 0, k_issued = 0;
      // Thread lt copies the 16-byte column chf of rows r0, r0 + RS, ...  A tile's key and
      // the entries of these rows are fetched one tile ahead, so the entry loads of tile
      // u+1 are in flight while the rows of tile u are copied.
      constexpr int RS = kLoadThreads / CH;  // rows per pass
      constexpr int NR = 128 / RS;           // rows per thread
      const int r0 = lt / CH, chf = lt % CH;
      int cur_key = 0, nxt_key = 0;
      int cur_ent[NR], nxt_ent[NR];
      auto fetch = [&](int u, int& key, int (&ent)[NR]) {
        const int t = t_begin + u;
        key = kc.at(p.toff, p.keys, t);
        const int e0 = __ldg(&p.off[key]) + (t - __ldg(&p.toff[key])) * 128;
        const int ne = min(128, __ldg(&p.off[key + 1]) - e0);
#pragma unroll
        for (int k = 0; k < NR; ++k) {
          const int r = r0 + RS * k;
          ent[k] = r < ne ? __ldg(&p.entries[e0 + r]) : -1;
        }
      };
      if (n_tiles > 0) fetch(0, cur_key, cur_ent);
      for (int u = 0; u < n_tiles && !*abort_flag; ++u) {
        const int st = u % kQStages;
        const int key = cur_key;
        if (u + 1 < n_tiles) fetch(u + 1, nxt_key, nxt_ent);
        const int bg = key / p.nb, c = key - bg * p.nb;
        const int b = bg / p.H_kv, g = bg - b * p.H_kv;
        const SeqSpan sp = seq_span(p.spans, b, p.N);
        if (key != prev_key) {
          if (lt == 0) {
            const int kb = k_loads & 1;
            if (k_loads >= 2 &&
                !mbar_wait(&kempty[kb], ((k_loads >> 1) - 1) & 1, p.wait_ns, abort_flag))
              *abort_flag = 1;
            if (!*abort_flag) {
              mbar_arrive_expect_tx(&kfull[kb], L::kTile);
              tma_load_3d(sK + kb * L::kTile, &tm_k, &kfull[kb], 0, sp.tn + c * 128, sp.tb);
              k_issued = k_loads + 1;
            }
          }
          ++k_loads;
          prev_key = key;
        }
        if (!mbar_wait(&qempty[st], ((u / kQStages) & 1) ^ 1, p.wait_ns, abort_flag)) {
          *abort_flag = 1;
          break;
        }
        uint8_t* dq = sQ + st * L::kTile;
        const __nv_bfloat16* qg = p.q_idx + (sp.t0 * p.H_kv + g) * DI + chf * 8;
#pragma unroll
        for (int k = 0; k < NR; ++k) {
          const int r = r0 + RS * k;
          const bool ok = cur_ent[k] >= 0;
          const int i = ok ? (cur_ent[k] >> kSlotBits) : 0;
          cp_async_16(dq + swz<RB>(r, chf), qg + (int64_t)i * p.H_kv * DI, ok);
        }
        cp_async_commit();
        // this thread's copies count toward the tile's stage as soon as they land (the
        // MMA thread orders them before the tensor core's reads with a proxy fence)
        cp_async_mbar_arrive(&qfull[st]);
        cur_key = nxt_key;
#pragma unroll
        for (int k = 0; k < NR; ++k) cur_ent[k] = nxt_ent[k];
      }
      cp_async_wait<0>();  // nothing may still be landing when the CTA exits
      // teardown: every k_idx TMA issued must have landed before the CTA exits
      if (lt == 0)
        for (int n = max(0, k_issued - 2); n < k_issued; ++n)
          mbar_wait(&kfull[n & 1], (n >> 1) & 1, 1000000000ull);
    } else if (warp == kMmaWarp) {
      // ============================== MMA issuer ================================
      if (lane == 0) {
        constexpr uint32_t idesc = umma_idesc_bf16_f32(128, 128);
        Cursor kc;
        int cur_key = -1, k_uses = 0;
        bool issued = false, ok = true;
        for (int u = 0; u < n_tiles; ++u) {
          const int key = kc.at(p.toff, p.keys, t_begin + u);
          if (key != cur_key) {
            if (!mbar_wait(&kfull[k_uses & 1], (k_uses >> 1) & 1, p.wait_ns, abort_flag)) {
              ok = false;
              break;
            }
            ++k_uses;
            cur_key = key;
          }
          const int st = u % kQStages, sl = u % kSlots;
          if (!mbar_wait(&qfull[st], (u / kQStages) & 1, p.wait_ns, abort_flag) ||
              !mbar_wait(&tfree[sl], ((u / kSlots) & 1) ^ 1, p.wait_ns, abort_flag)) {
            ok = false;
            break;
          }
          fence_proxy_async_smem();  // the q_idx rows came by cp.async (generic proxy)
          tc_fence_after();
          const uint64_t qd = umma_desc_kmajor<RB>(smem_u32(sQ + st * L::kTile));
          const uint64_t kd = umma_desc_kmajor<RB>(smem_u32(sK + ((k_uses - 1) & 1) * L::kTile));
#pragma unroll
          for (int kk = 0; kk < DI / 16; ++kk)  // +32 bytes per K=16 step
            tc_mma_bf16(tmem + 128 * sl, qd + 2 * kk, kd + 2 * kk, idesc, kk > 0 ? 1u : 0u);
          tc_commit(&qempty[st]);
          tc_commit(&sfull[sl]);
          issued = true;
          // after the block's last tile its k_idx buffer may be refilled
          Cursor peek = kc;
          if (u + 1 < n_tiles && peek.at(p.toff, p.keys, t_begin + u + 1) != key)
            tc_commit(&kempty[(k_uses - 1) & 1]);
        }
        if (!ok) *abort_flag = 1;
        if (issued) {
          tc_commit(mmadone);
          mbar_wait(mmadone, 0, 1000000000ull);
        }
      }
    } else {
      // ====================== row log-sum-exp: warps 0-11 =======================
      const int wg = warp >> 2;
      const int row = (warp & 3) * 32 + lane;  // TMEM lane
      const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
      const float sl2 = p.scale_log2;
      Cursor kc;
      // the key and this row's entry of the warpgroup's next tile are fetched while the
      // current tile is processed
      auto fetch = [&](int u, int& key, int& ent) {
        const int t = t_begin + u;
        key = kc.at(p.toff, p.keys, t);
        const int e0 = __ldg(&p.off[key]) + (t - __ldg(&p.toff[key])) * 128;
        const int ne = min(128, __ldg(&p.off[key + 1]) - e0);
        ent = row < ne ? __ldg(&p.entries[e0 + row]) : -1;
      };
      int nxt_key = 0, nxt_ent = -1;
      if (wg < n_tiles) fetch(wg, nxt_key, nxt_ent);
      for (int u = wg; u < n_tiles; u += kSoftWG) {
        const int sl = u % kSlots;
        const int key = nxt_key, ent = nxt_ent;
        if (u + kSoftWG < n_tiles) fetch(u + kSoftWG, nxt_key, nxt_ent);
        const int bg = key / p.nb, c = key - bg * p.nb;
        const int b = bg / p.H_kv, g = bg - b * p.H_kv;
        const SeqSpan sp = seq_span(p.spans, b, p.N);
        const int i = ent >> kSlotBits;
        const bool ok =
            __all_sync(0xffffffffu, mbar_wait(&sfull[sl], (u / kSlots) & 1, p.wait_ns, abort_flag));
        if (!ok) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const int jlim = ent >= 0 ? min(i, sp.len - 1) - c * 128 : -1;  // last valid column
        const bool full = __all_sync(0xffffffffu, jlim >= 127);
        // One pass over the row: the exp2 offset is the max of its first 32 columns
        // (column 0, the block's first key, is visible to every real row).  The lse is
        // exact for any offset; only overflow matters, so a row sum above 2^64 (a later
        // score far above the offset) takes the exact row max and a second pass.  The
        // TMEM slot is handed back after that check.
        const uint32_t srow = tmem + lane_base + 128 * sl;
        auto exp_sum = [&](const uint32_t (&r)[64], int c0, float ms, float2& acc) {
          if (full) {  // packed pairs: one FFMA2 and one FADD2 per two scores
            const float2 scl = make_float2(sl2, sl2), off = make_float2(-ms, -ms);
#pragma unroll
            for (int x = 0; x < 64; x += 2) {
              const float2 a =
                  ffma2(make_float2(__uint_as_float(r[x]), __uint_as_float(r[x + 1])), scl, off);
              acc = fadd2(acc, make_float2(ex2_fast(a.x), ex2_fast(a.y)));
            }
          } else {
#pragma unroll
            for (int x = 0; x < 64; x += 2) {
              acc.x += c0 + x <= jlim ? ex2_fast(__uint_as_float(r[x]) * sl2 - ms) : 0.f;
              acc.y += c0 + x + 1 <= jlim ? ex2_fast(__uint_as_float(r[x + 1]) * sl2 - ms) : 0.f;
            }
          }
        };
        auto load64 = [&](uint32_t (&r)[64], int c0) {
          tmem_ld_32x32b_x32(srow + c0, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
          tmem_ld_32x32b_x32(srow + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
          tmem_wait_ld();
        };
        float ms;
        float2 acc = make_float2(0.f, 0.f);
        {
          uint32_t r[64];
          float m0;
          // a full tile takes the offset from the first load's own max reduction
          tmem_ld_max_32x32b_x32(srow, *reinterpret_cast<uint32_t(*)[32]>(&r[0]), m0);
          tmem_ld_32x32b_x32(srow + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
          tmem_wait_ld();
          if (!full) {
            m0 = -INFINITY;
#pragma unroll
            for (int x = 0; x < 32; x += 2)
              m0 = fmax3(m0, x <= jlim ? __uint_as_float(r[x]) : -INFINITY,
                         x + 1 <= jlim ? __uint_as_float(r[x + 1]) : -INFINITY);
          }
          ms = m0 == -INFINITY ? 0.f : m0 * sl2;
          exp_sum(r, 0, ms, acc);
          load64(r, 64);
          exp_sum(r, 64, ms, acc);
        }
        float l = acc.x + acc.y;
        if (__any_sync(0xffffffffu, l > 0x1p64f)) {  // rare: exact max, second pass
          float m = -INFINITY;
#pragma unroll 1
          for (int h = 0; h < 4; ++h) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(srow + 32 * h, r);
            tmem_wait_ld();
#pragma unroll
            for (int x = 0; x < 32; ++x)
              m = fmaxf(m, 32 * h + x <= jlim ? __uint_as_float(r[x]) : -INFINITY);
          }
          ms = m == -INFINITY ? 0.f : m * sl2;
          acc = make_float2(0.f, 0.f);
#pragma unroll 1
          for (int c0 = 0; c0 < 128; c0 += 64) {
            uint32_t r[64];
            load64(r, c0);
            exp_sum(r, c0, ms, acc);
          }
          l = acc.x + acc.y;
        }
        // the scores are in registers: hand the slot back to the MMA
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tfree[sl]);
        if (ent >= 0) {
          p.lse_part[(sp.t0 * p.H_kv + (int64_t)g * sp.len + i) * p.topk + (ent & kSlotMask)] =
              l > 0.f ? (ms + log2f(l)) * kLn2 : -INFINITY;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) set_status(p.status, MSA_ERR_DEVICE_TIMEOUT);
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// lse_idx[b,g,i] = log-sum-exp over the row's valid slots of the partial lse.  A row's
// slots are read by W consecutive lanes (W = topk rounded up to a power of two, at most
// 32; 32 / W rows per warp), each lane keeping a running (max, sum) over its slots; the
// pairs are merged across the row's lanes by shuffles.
__device__ __forceinline__ void lse_merge(float& m, float& l, float m2, float l2) {
  const float mm = fmaxf(m, m2);
  l = mm == -INFINITY ? 0.f : l * __expf(m - mm) + l2 * __expf(m2 - mm);
  m = mm;
}

template <int V>
__global__ void lse_combine_kernel(const float* __restrict__ lse_part,
                                   const int32_t* __restrict__ block_idx,
                                   float* __restrict__ lse_idx, const int2* __restrict__ spans,
                                   int B, int N, int H_kv, int64_t rows, int topk, int nb, int W) {
  // W lanes per row, V consecutive slots per lane and load (V = 4: 16-byte loads of the
  // row's block ids and partials, so that enough bytes are in flight to stream them)
  const int lane = threadIdx.x & 31;
  const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t r = warp * (32 / W) + lane / W;
  const int sl = lane % W;
  bool live = r < rows;
  if (live && spans) {
    RowPos rp;
    live = row_pos(spans, B, N, H_kv, r, &rp);  // tokens outside every sequence
  }
  float m = -INFINITY, l = 0.f;
  if (live) {
    for (int s = V * sl; s < topk; s += V * W) {
      int c[V];
      float v[V];
      if constexpr (V == 4) {
        const int4 c4 = __ldg(reinterpret_cast<const int4*>(block_idx + r * topk + s));
        const float4 v4 = __ldg(reinterpret_cast<const float4*>(lse_part + r * topk + s));
        c[0] = c4.x, c[1] = c4.y, c[2] = c4.z, c[3] = c4.w;
        v[0] = v4.x, v[1] = v4.y, v[2] = v4.z, v[3] = v4.w;
      } else {
        c[0] = __ldg(&block_idx[r * topk + s]);
        v[0] = __ldg(&lse_part[r * topk + s]);
      }
#pragma unroll
      for (int e = 0; e < V; ++e)
        if (c[e] >= 0 && c[e] < nb) lse_merge(m, l, v[e], 1.f);
    }
  }
  for (int o = W / 2; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
    lse_merge(m, l, m2, l2);
  }
  if (live && sl == 0) lse_idx[r] = m + logf(l);
}

template <int DI>
cudaError_t launch_lse_tc(const CUtensorMap& tk, const LseParams& prm, const Ctx& cx,
                          cudaStream_t st) {
  using L = LseLayout<DI>;
  auto kern = index_lse_tc_kernel<DI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  kernel_event(MSA_KERNEL_INDEX_LSE, true, st);
  kern<<<cx.num_sms, kThreads, L::kAlloc, st>>>(tk, prm);
  kernel_event(MSA_KERNEL_INDEX_LSE, false, st);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_index_lse(const Shape& s, const void* q_idx, const void* k_idx,
                             const int32_t* block_idx, const Plan& pl, float* lse_part,
                             float* lse_idx, const Ctx& cx, cudaStream_t st) {
  const int DI = s.d_idx;
  CUtensorMap tk;
  const uint64_t dims[3] = {(uint64_t)DI, s.tma_tokens(), s.tma_batches()};
  const uint64_t strides[2] = {(uint64_t)DI * 2, s.tma_tokens() * DI * 2};
  const uint32_t box[3] = {(uint32_t)DI, 128, 1};
  if (!encode_tiled(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, k_idx, dims, strides, box,
                    DI == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  LseParams prm;
  prm.q_idx = static_cast<const __nv_bfloat16*>(q_idx);
  prm.spans = s.spans;
  prm.off = pl.off;
  prm.toff = pl.toff;
  prm.entries = pl.entries;
  prm.lse_part = lse_part;
  prm.keys = s.keys();
  prm.N = s.N;
  prm.H_kv = s.H_kv;
  prm.nb = s.nb;
  prm.topk = s.topk;
  prm.scale_log2 = s.scale_idx * kLog2e;
  prm.wait_ns = cx.wait_ns;
  prm.status = cx.status;
  cudaError_t e = DI == 64 ? launch_lse_tc<64>(tk, prm, cx, st) : launch_lse_tc<32>(tk, prm, cx, st);
  if (e != cudaSuccess) return e;
  const int64_t rows = s.rows_kv();
  // rows of whole 16-byte groups of slots, both arrays 16-byte aligned: 4 slots a load
  const bool vec = (s.topk & 3) == 0 && (reinterpret_cast<uintptr_t>(block_idx) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(lse_part) & 15) == 0;
  const int per_lane = vec ? 4 : 1;
  int W = 1;
  while (W * per_lane < s.topk && W < 32) W <<= 1;
  const int64_t warps = (rows + (32 / W) - 1) / (32 / W);
  if (vec)
    lse_combine_kernel<4><<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(
        lse_part, block_idx, lse_idx, s.spans, s.B, s.N, s.H_kv, rows, s.topk, s.nb, W);
  else
    lse_combine_kernel<1><<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(
        lse_part, block_idx, lse_idx, s.spans, s.B, s.N, s.H_kv, rows, s.topk, s.nb, W);
  note_launch();
  return cudaGetLastError();
}

}  // namespace msa
