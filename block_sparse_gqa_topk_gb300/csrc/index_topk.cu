// index_topk.cu -- MSA index branch: causal index scoring, 128-token block
// max-pooling and exp-free top-k with the forced local block, in one kernel.
//
// Method: MiniMax Sparse Attention summary (7minutos.es), "Cómo funcionan las dos
// ramas" ¶1-2 (one index-query head per GQA group, one shared index-key head,
// max-pool to blocks, top-k per query and group, own block always kept) and "El
// codiseño del kernel" (rank raw scores, no max/exp/sum); Flash-MSA article
// (tech.kuratif.com) ¶6 (top-k kept per query row in registers while keys stream,
// local score forced to +inf).
//
// GB300 design.  One CTA owns a pair of GQA groups and a pair of query blocks
// (qb, nb-1-qb), so every CTA scores exactly nb-1 key blocks under the causal
// mask.  Per key block:
//   - a TMA producer warp streams the 128 x d_idx k_idx tile into a smem ring
//     (SWIZZLE_128B / 64B, the layout tcgen05 reads directly);
//   - one thread issues tcgen05.mma: S_g = Q_idx,g (128 x d_idx) . K^T for both
//     groups into a 2-slot TMEM ring (2 slots x 2 groups x 128 fp32 columns);
//   - 8 epilogue warps (one thread per query row and group) read the row's 128
//     scores with max-reducing TMEM loads (tcgen05.ld.red, four of 32 columns), so
//     the block score needs no max chain, and update a sorted top-(k-1) list in
//     registers.
// The local (diagonal) block is never scored: it is always selected.  Nothing but
// block_idx is written: the pooled scores never leave the SM.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace msa {
namespace {

constexpr int kStages = 6;
constexpr int kThreads = 320;  // warps 0-7 epilogue, 8 TMA producer, 9 MMA + TMEM owner
constexpr int kTmemCols = 512;

template <int DI>
struct IdxLayout {
  static constexpr int kRowBytes = DI * 2;
  static constexpr int kTile = 128 * kRowBytes;  // one 128-row operand tile
  static constexpr int kQOff = 0;                // 2 tiles (group pair)
  static constexpr int kKOff = 2 * kTile;        // kStages tiles
  static constexpr int kBarOff = kKOff + kStages * kTile;
  static constexpr int kNumBars = 2 * kStages + 2 + 4 + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  // >= 116 KB so that a single CTA (and its 512-column TMEM allocation) owns an SM
  static constexpr int kAlloc = (kBytes + 1024 > 118 * 1024) ? kBytes + 1024 : 118 * 1024;
};

struct IdxParams {
  int32_t* block_idx;
  const int2* spans;  // packed batches: (start, end) per sequence; nullptr: fixed [B][N]
  const int* units;   // packed batches: prefix counts of ceil(len / 256) per sequence
  int B, N, H_kv, nb, topk;
  int n_units;  // fixed layout: ceil(nb / 2) query-block pairs per sequence
  // fixed layout: units from split_from on (the last wave's) are split in two CTAs, one
  // group of the pair each, so that the last wave's CTAs are shorter
  int split_from;
  int n_gp;     // ceil(H_kv / 2) group pairs
  uint64_t wait_ns;
  int debug;
  int* status;
};

// Writes the final set of one row: the sorted non-local ids (up to M, -1 = none)
// followed by the own block, padded with -1.
template <int KM>
__device__ __forceinline__ void store_row(int32_t* dst, const int (&id)[KM], int M, int own,
                                          int topk) {
  constexpr int KS = KM + 1;
  int v[KS];
#pragma unroll
  for (int s = 0; s < KM; ++s) v[s] = (s < M && id[s] >= 0) ? id[s] : 0x7fffffff;
  v[KM] = own;
  // every non-local id is below the own block (causal), -1 slots sort last
  // odd-even transposition sort, KS passes
#pragma unroll
  for (int pass = 0; pass < KS; ++pass)
#pragma unroll
    for (int b = (pass & 1); b + 1 < KS; b += 2) {
      const int lo = min(v[b], v[b + 1]), hi = max(v[b], v[b + 1]);
      v[b] = lo;
      v[b + 1] = hi;
    }
  if ((topk & 3) == 0 && (KS & 3) == 0) {
#pragma unroll
    for (int s = 0; s < KS; s += 4) {
      if (s < topk) {
        int4 w;
        w.x = v[s] == 0x7fffffff ? -1 : v[s];
        w.y = v[s + 1] == 0x7fffffff ? -1 : v[s + 1];
        w.z = v[s + 2] == 0x7fffffff ? -1 : v[s + 2];
        w.w = v[s + 3] == 0x7fffffff ? -1 : v[s + 3];
        *reinterpret_cast<int4*>(dst + s) = w;
      }
    }
  } else {
#pragma unroll
    for (int s = 0; s < KS; ++s)
      if (s < topk) dst[s] = v[s] == 0x7fffffff ? -1 : v[s];
  }
}

template <int DI, int KM>
__global__ void __launch_bounds__(kThreads, 1)
    index_topk_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k, const IdxParams p) {
  using L = IdxLayout<DI>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem + L::kQOff;
  uint8_t* sK = smem + L::kKOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* full = bars;                    // [kStages] k tile landed
  uint64_t* empty = bars + kStages;         // [kStages] k tile consumed by the MMAs
  uint64_t* qfull = bars + 2 * kStages;     // q tiles landed
  uint64_t* qempty = qfull + 1;             // q tiles no longer read
  uint64_t* accfull = qfull + 2;            // [2] TMEM slot holds finished scores
  uint64_t* accempty = qfull + 4;           // [2] TMEM slot drained by the epilogue
  uint64_t* mmadone = qfull + 6;            // all MMAs retired (teardown)
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA -> (sequence, group pair, query-block pair); the pair (u, nbs-1-u) of a
  // sequence of nbs blocks
  int b, u, gp, half = -1;  // half >= 0: this CTA takes group 2 gp + half of a split unit
  if (!p.units) {
    int x = blockIdx.x;
    if (x >= p.split_from) {
      half = (x - p.split_from) & 1;
      x = p.split_from + (x - p.split_from) / 2;
    }
    u = x % p.n_units;
    gp = (x / p.n_units) % p.n_gp;
    b = x / (p.n_units * p.n_gp);
  } else {
    gp = blockIdx.x % p.n_gp;
    if (!chunk_item(p.units, p.B, 0, blockIdx.x / p.n_gp, &b, &u)) return;  // whole CTA
  }
  const SeqSpan sp = seq_span(p.spans, b, p.N);
  const int g0 = 2 * gp + (half > 0 ? 1 : 0);
  const int ng = half >= 0 ? 1 : min(2, p.H_kv - g0);
  const int qa = (sp.len + 127) / 128 - 1 - u;  // heavy block first
  const int nq = (u < qa) ? 2 : 1;
  const int M = p.topk - 1;     // non-local slots

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(qfull, 1);
    mbar_init(qempty, 1);
    mbar_init(&accfull[0], 1);
    mbar_init(&accfull[1], 1);
    mbar_init(&accempty[0], 4 * ng);
    mbar_init(&accempty[1], 4 * ng);
    mbar_init(mmadone, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 8) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0 && !(p.debug & MSA_DEBUG_WITHHOLD_LOAD)) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      int kt = 0, qloads = 0;
      for (int n = 0; n < nq && !*abort_flag; ++n) {
        const int qb = n == 0 ? qa : u;
        const int nt = qb;  // key blocks 0 .. qb-1
        if (nt == 0) continue;
        if (qloads > 0 && !mbar_wait(qempty, (qloads - 1) & 1, p.wait_ns, abort_flag)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(qfull, ng * L::kTile);
        for (int gi = 0; gi < ng; ++gi)
          tma_load_4d(sQ + gi * L::kTile, &tm_q, qfull, 0, g0 + gi, sp.tn + qb * 128, sp.tb);
        ++qloads;
        for (int t = 0; t < nt; ++t, ++kt) {
          const int s = kt % kStages, use = kt / kStages;
          if (!mbar_wait(&empty[s], (use & 1) ^ 1, p.wait_ns, abort_flag)) {
            *abort_flag = 1;
            break;
          }
          mbar_arrive_expect_tx(&full[s], L::kTile);
          tma_load_3d(sK + s * L::kTile, &tm_k, &full[s], 0, sp.tn + t * 128, sp.tb);
        }
      }
      // teardown: every load issued must have landed before the CTA exits
      for (int s = 0; s < kStages && kt > 0; ++s) {
        const int last = (s < kt) ? (kt - 1 - ((kt - 1 - s) % kStages)) : -1;
        if (last >= 0) mbar_wait(&full[s], (last / kStages) & 1, 1000000000ull);
      }
      if (qloads > 0) mbar_wait(qfull, (qloads - 1) & 1, 1000000000ull);
    }
  } else if (warp == 9) {
    // ------------------------------ MMA issuer --------------------------------
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16_f32(128, 128);
      int kt = 0, at = 0, qloads = 0;
      bool issued = false;
      for (int n = 0; n < nq && !*abort_flag; ++n) {
        const int qb = n == 0 ? qa : u;
        const int nt = qb;
        if (nt == 0) continue;
        if (!mbar_wait(qfull, qloads & 1, p.wait_ns, abort_flag)) {
          *abort_flag = 1;
          break;
        }
        ++qloads;
        tc_fence_after();
        const uint64_t qdesc0 = umma_desc_kmajor<L::kRowBytes>(smem_u32(sQ));
        const uint64_t qdesc1 = umma_desc_kmajor<L::kRowBytes>(smem_u32(sQ + L::kTile));
        for (int t = 0; t < nt; ++t, ++kt, ++at) {
          const int s = kt % kStages, use = kt / kStages;
          const int a = at & 1, ause = at >> 1;
          if (!mbar_wait(&full[s], use & 1, p.wait_ns, abort_flag) ||
              !mbar_wait(&accempty[a], (ause & 1) ^ 1, p.wait_ns, abort_flag)) {
            *abort_flag = 1;
            break;
          }
          tc_fence_after();
          const uint64_t kdesc = umma_desc_kmajor<L::kRowBytes>(smem_u32(sK + s * L::kTile));
#pragma unroll
          for (int gi = 0; gi < 2; ++gi) {
            if (gi < ng) {
              const uint32_t d_tmem = tmem + a * 256 + gi * 128;
              const uint64_t qd = gi == 0 ? qdesc0 : qdesc1;
#pragma unroll
              for (int kk = 0; kk < DI / 16; ++kk)  // +32 bytes per K=16 step
                tc_mma_bf16(d_tmem, qd + 2 * kk, kdesc + 2 * kk, idesc, kk > 0 ? 1u : 0u);
            }
          }
          issued = true;
          tc_commit(&empty[s]);
          tc_commit(&accfull[a]);
        }
        if (*abort_flag) break;
        tc_commit(qempty);
      }
      // teardown: wait until every issued MMA has retired before TMEM is freed
      if (issued) {
        tc_commit(mmadone);
        mbar_wait(mmadone, 0, 1000000000ull);
      }
    }
  } else {
    // ------------------------------ epilogue ----------------------------------
    const int gi = warp >> 2;  // group of the pair
    const int quad = warp & 3; // TMEM lanes 32*quad .. 32*quad+31
    const int row = quad * 32 + lane;
    if (gi < ng) {
      const int g = g0 + gi;
      int at = 0;
      for (int n = 0; n < nq; ++n) {
        const int qb = n == 0 ? qa : u;
        const int nt = qb;
        float val[KM];
        int id[KM];
        // Slots >= M (only when topk-1 is below the instantiated KM) hold +inf and
        // never move, so the first M slots behave as a top-M list.
#pragma unroll
        for (int s = 0; s < KM; ++s) {
          val[s] = s < M ? -INFINITY : INFINITY;
          id[s] = -1;
        }
        const bool exact = (M == KM);
        bool ok = true;
        for (int t = 0; t < nt; ++t, ++at) {
          const int a = at & 1, ause = at >> 1;
          // warp-uniform decision: every lane must take part in the tcgen05.ld below
          ok = __all_sync(0xffffffffu, mbar_wait(&accfull[a], ause & 1, p.wait_ns, abort_flag));
          if (!ok) {
            *abort_flag = 1;
            break;
          }
          tc_fence_after();
          const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + a * 256 + gi * 128;
          // the block score: each 32-column load returns its own max (the reducing
          // TMEM load of sm_103a), so no max chain runs over the loaded registers
          float m = -INFINITY;
#pragma unroll 1
          for (int h = 0; h < 4; ++h) {
            uint32_t r[32];
            float mh;
            tmem_ld_max_32x32b_x32(taddr + h * 32, r, mh);
            tmem_wait_ld();
            m = fmaxf(m, mh);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&accempty[a]);
          // sorted insert of (m, t).  The first M slots stay ordered by (score
          // descending, block ascending): m lands in the first slot whose score it
          // beats strictly (after every equal score, which came from a lower block)
          // and the slots after it shift down by one.  When the list overflows, the
          // entry dropped has the lowest score and, among equal scores, the highest
          // block, as the selection rule wants.  Each slot's new value depends on the
          // old list only, so there is no carry from slot to slot.
          if (!exact || m > val[KM - 1]) {
            bool gt[KM];
#pragma unroll
            for (int s = 0; s < KM; ++s) gt[s] = m > val[s];
#pragma unroll
            for (int s = KM - 1; s > 0; --s) {
              val[s] = gt[s] ? (gt[s - 1] ? val[s - 1] : m) : val[s];
              id[s] = gt[s] ? (gt[s - 1] ? id[s - 1] : t) : id[s];
            }
            val[0] = gt[0] ? m : val[0];
            id[0] = gt[0] ? t : id[0];
          }
        }
        if (__any_sync(0xffffffffu, !ok || *abort_flag)) break;  // warp-uniform exit
        const int i = qb * 128 + row;
        if (i < sp.len) {
          int32_t* dst = p.block_idx + (sp.t0 * p.H_kv + (int64_t)g * sp.len + i) * p.topk;
          store_row<KM>(dst, id, M, qb, p.topk);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) set_status(p.status, MSA_ERR_DEVICE_TIMEOUT);
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Sets that need no scoring.  topk == 1: every row gets only its own block.
// topk >= nb: every visible block is selected (blocks 0..i/128 ascending, then -1) --
// the dense set of the indexer warm-up, where both branches see the full causal
// context ("Cómo se entrena MSA" ¶3: warm-up with full attention in both branches).
__global__ void forced_set_kernel(int32_t* __restrict__ block_idx, const int2* __restrict__ spans,
                                  int B, int N, int H_kv, int64_t rows, int topk, int all) {
  const int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (t >= rows * topk) return;
  const int64_t r = t / topk;
  const int s = (int)(t % topk);
  RowPos rp;
  if (!row_pos(spans, B, N, H_kv, r, &rp)) return;  // tokens outside every sequence
  const int c = rp.i / 128;
  block_idx[t] = all ? (s <= c ? s : -1) : (s == 0 ? c : -1);
}

template <int DI, int KM>
cudaError_t launch_tc(const Shape& s, const CUtensorMap& tq, const CUtensorMap& tk,
                      const IdxParams& p, int grid, cudaStream_t st) {
  using L = IdxLayout<DI>;
  auto kern = index_topk_tc_kernel<DI, KM>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  kernel_event(MSA_KERNEL_INDEX, true, st);
  kern<<<grid, kThreads, L::kAlloc, st>>>(tq, tk, p);
  kernel_event(MSA_KERNEL_INDEX, false, st);
  note_launch();
  return cudaGetLastError();
}

template <int DI>
cudaError_t launch_di(const Shape& s, const CUtensorMap& tq, const CUtensorMap& tk,
                      const IdxParams& p, int grid, cudaStream_t st) {
  const int M = s.topk - 1;
  if (M <= 3) return launch_tc<DI, 3>(s, tq, tk, p, grid, st);
  if (M <= 7) return launch_tc<DI, 7>(s, tq, tk, p, grid, st);
  if (M <= 15) return launch_tc<DI, 15>(s, tq, tk, p, grid, st);
  return launch_tc<DI, 31>(s, tq, tk, p, grid, st);
}

}  // namespace

cudaError_t launch_index_topk(const Shape& s, const void* q_idx, const void* k_idx,
                              int32_t* block_idx, const Ctx& cx, cudaStream_t st) {
  if (s.B == 0 || s.N == 0 || s.T == 0 || s.H_kv == 0) return cudaSuccess;
  if (s.topk == 1 || s.topk >= s.nb) {
    const int64_t n = s.rows_kv() * s.topk;
    forced_set_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(
        block_idx, s.spans, s.B, s.N, s.H_kv, s.rows_kv(), s.topk, s.topk >= s.nb);
    note_launch();
    return cudaGetLastError();
  }
  if (s.topk > kMaxSelect) return cudaErrorNotSupported;  // callers reject this case first
  const int DI = s.d_idx;
  const CUtensorMapSwizzle swz = DI == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUtensorMap tq, tk;
  {
    const uint64_t dims[4] = {(uint64_t)DI, (uint64_t)s.H_kv, s.tma_tokens(), s.tma_batches()};
    const uint64_t strides[3] = {(uint64_t)DI * 2, (uint64_t)s.H_kv * DI * 2,
                                 s.tma_tokens() * s.H_kv * DI * 2};
    const uint32_t box[4] = {(uint32_t)DI, 1, 128, 1};
    if (!encode_tiled(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, q_idx, dims, strides, box, swz))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)DI, s.tma_tokens(), s.tma_batches()};
    const uint64_t strides[2] = {(uint64_t)DI * 2, s.tma_tokens() * DI * 2};
    const uint32_t box[3] = {(uint32_t)DI, 128, 1};
    if (!encode_tiled(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, k_idx, dims, strides, box, swz))
      return cudaErrorInvalidValue;
  }
  IdxParams p;
  p.block_idx = block_idx;
  p.spans = s.spans;
  p.units = s.tab(kTabIndexUnit);
  p.B = s.B;
  p.N = s.N;
  p.H_kv = s.H_kv;
  p.nb = s.nb;
  p.topk = s.topk;
  p.n_units = (s.nb + 1) / 2;
  p.n_gp = (s.H_kv + 1) / 2;
  p.wait_ns = cx.wait_ns;
  p.debug = cx.debug;
  p.status = cx.status;
  int64_t grid = (int64_t)p.n_gp * (s.packed() ? varlen_grid_items(s, kTabIndexUnit)
                                                : (int64_t)s.B * p.n_units);
  // One CTA per SM.  Every unit of the fixed layout scores the same number of key tiles,
  // so a last wave of at most half the SMs would leave the rest idle: its units go to two
  // CTAs each, one group apiece (only when every pair holds two groups).
  p.split_from = 0x7fffffff;
  const int64_t rem = grid % cx.num_sms;
  if (!s.packed() && s.H_kv % 2 == 0 && grid > cx.num_sms && rem > 0 && 2 * rem <= cx.num_sms) {
    p.split_from = (int)(grid - rem);
    grid += rem;
  }
  if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
  if (DI == 64) return launch_di<64>(s, tq, tk, p, (int)grid, st);
  return launch_di<32>(s, tq, tk, p, (int)grid, st);
}

bool encode_tiled(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base,
                  const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                  CUtensorMapSwizzle swz) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !ptr)
      return false;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = fn(m, dt, (cuuint32_t)rank, const_cast<void*>(base),
                        reinterpret_cast<const cuuint64_t*>(dims),
                        reinterpret_cast<const cuuint64_t*>(strides_bytes),
                        reinterpret_cast<const cuuint32_t*>(box), estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace msa
