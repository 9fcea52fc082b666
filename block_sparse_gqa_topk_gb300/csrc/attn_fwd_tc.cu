// attn_fwd_tc.cu -- main-branch block-sparse forward on the 5th-generation tensor
// cores (tcgen05 + TMEM), over the gathered tiles of plan.cu.
//
// Method: MSA summary (7minutos.es), "Cómo funcionan las dos ramas" ¶3 (exact
// softmax attention of every head of a group over the causally visible tokens of
// the group's blocks) and "El codiseño del kernel" (KV-outer query gather packing
// queries x heads into one 128x128 score MMA, split + combine across CTAs);
// Flash-MSA article (tech.kuratif.com) ¶6 (the LSE is kept for the backward).
//
// A tile is one key block c of one (batch, group) and 128 rows = 128/G gathered
// queries x G heads.  Per CTA (persistent, a contiguous range of tiles):
//   warps 8-10 loaders: gather the tile's q rows with cp.async into a 3-stage ring
//              in the 128-byte-swizzled K-major layout tcgen05 reads (a stage completes
//              through cp.async arrivals as its rows land); one thread TMA-loads K and V
//              of the block when the key changes;
//   warp 11    TMEM owner + one MMA thread: S = Q K^T (M=N=128, K=d) into a 2-deep
//              TMEM ring, then O = P V with V as an MN-major operand;
//   warps 0-7  two softmax warpgroups taking alternate tiles (thread = row = TMEM
//              lane): one pass over S with the max of the first 32 columns as the
//              exp2 offset (exact two-pass fallback when a row sum would overflow),
//              P (bf16) into smem for the PV MMA, S released at once; then O from
//              TMEM, normalised, stored as bf16 partials with their lse.
// S and O have separate release barriers, so the next S MMA of a warpgroup overlaps
// its O epilogue.  Every wait is bounded; on expiry the CTA unwinds and records
// MSA_ERR_DEVICE_TIMEOUT.
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace msa {
namespace {

constexpr int kTcThreads = 384;  // 12 warps: 8 softmax, 3 loaders, 1 MMA
constexpr int kLoadThreads = 96;
constexpr int kQStages = 3;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct FwdTcParams {
  const __nv_bfloat16* q;
  const int2* spans;      // packed batches: (start, end) per sequence
  const int* off;
  const int* toff;
  const int* entries;
  __nv_bfloat16* o_part;  // [(rkv*topk + slot)*G + h][D]
  float* lse_part;        // [(rkv*topk + slot)*G + h]
  int64_t keys;
  int N, H_kv, nb, topk;
  float scale_log2;
  uint64_t wait_ns;
  int* status;
};

template <int D>
struct TcLayout {
  static constexpr int kHalves = D / 64;        // 64-element (128-byte) column blocks
  static constexpr int kHalf = 128 * 128;       // one [128 rows][64] bf16 block
  static constexpr int kTile = kHalves * kHalf; // 128 x D bf16
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTile;
  static constexpr int kQ = kV + kTile;                  // kQStages tiles
  static constexpr int kP = kQ + kQStages * kTile;       // [2][128 rows][128 keys] bf16
  static constexpr int kBar = kP + 2 * 2 * kHalf;
  // barriers: kvfull, kvempty, qfull[3], qempty[3], sfull[2], ofull[2], sfree[2],
  //           ofree[2], pfull[2], pempty[2], mmadone
  static constexpr int kNumBars = 2 + 2 * kQStages + 8 + 5;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;
};

// K-major tile split in 64-column blocks: element (r, k) of a [128][D] tile.
template <int D>
__device__ __forceinline__ uint32_t kmaj_off(int r, int chunk) {  // chunk = k / 8
  return (uint32_t)((chunk >> 3) * (128 * 128) + r * 128 + (((chunk & 7) ^ (r & 7)) << 4));
}

// Descriptor of an MN-major operand (contiguous along N) stored as [K rows][64-wide
// column blocks] with the 128-byte swizzle: SBO = 1024 (8 K-rows), LBO = the stride
// between 64-wide column blocks.
__device__ __forceinline__ uint64_t umma_desc_mnmajor_sw128(uint32_t smem_addr, uint32_t lbo) {
  return (uint64_t)((smem_addr & 0x3FFFF) >> 4) | ((uint64_t)(lbo >> 4) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ int tc_find_key(const int* __restrict__ toff, int64_t keys, int t) {
  int64_t lo = 0, hi = keys - 1;
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) >> 1;
    if (__ldg(&toff[mid]) <= t) lo = mid; else hi = mid - 1;
  }
  return (int)lo;
}

// Key of tile t given the key of an earlier tile of the same CTA (tiles are visited
// in increasing order, so keys only move forward; empty keys are skipped).
struct KeyCursor {
  int key = -1;
  __device__ __forceinline__ int at(const int* __restrict__ toff, int64_t keys, int t) {
    if (key < 0) {
      key = tc_find_key(toff, keys, t);
    } else {
      while (key + 1 < keys && __ldg(&toff[key + 1]) <= t) ++key;
    }
    return key;
  }
};

// Byte offset of 16-byte chunk `chunk` of row r in rows of 128 bytes, swizzled.
__device__ __forceinline__ uint32_t sw128_row(int r, int chunk) {
  return (uint32_t)(r * 128 + (((chunk & 7) ^ (r & 7)) << 4));
}

// The value of x, opaque to the optimiser: addresses derived from it are recomputed
// inside a loop instead of being hoisted and held in registers across it.
__device__ __forceinline__ int opaque(int x) {
  asm volatile("" : "+r"(x));
  return x;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <int D, int G>
__global__ void __launch_bounds__(kTcThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const FwdTcParams p) {
  using L = TcLayout<D>;
  constexpr int QPT = 128 / G;
  constexpr int CH = D / 8;  // 16-byte chunks per q row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sK = smem + L::kK;
  uint8_t* sV = smem + L::kV;
  uint8_t* sQ = smem + L::kQ;
  uint8_t* sP = smem + L::kP;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* kvfull = bars;
  uint64_t* kvempty = bars + 1;
  uint64_t* qfull = bars + 2;
  uint64_t* qempty = qfull + kQStages;
  uint64_t* sfull = qempty + kQStages;
  uint64_t* ofull = sfull + 2;
  uint64_t* sfree = ofull + 2;   // [2] softmax done reading S[b]
  uint64_t* ofree = sfree + 2;   // [2] epilogue done reading O[b]
  uint64_t* pfull = ofree + 2;   // [2]
  uint64_t* pempty = pfull + 2;  // [2]
  uint64_t* mmadone = pempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = __ldg(&p.toff[p.keys]);
  const int per = (total + gridDim.x - 1) / gridDim.x;
  const int t_begin = blockIdx.x * per;
  const int t_end = min(total, t_begin + per);
  const int n_tiles = max(0, t_end - t_begin);

  if (threadIdx.x == 0) {
    mbar_init(kvfull, 1);
    mbar_init(kvempty, 1);
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&qfull[s], kLoadThreads);  // every loader thread
      mbar_init(&qempty[s], 1);   // tcgen05.commit after the S MMA
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sfull[b], 1);
      mbar_init(&ofull[b], 1);
      mbar_init(&sfree[b], 4);  // one arrive per softmax warp
      mbar_init(&ofree[b], 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&pfull[b], 4);
      mbar_init(&pempty[b], 1);
    }
    mbar_init(mmadone, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 11) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // TMEM columns: S[b] at 128*b, O[b] at 256 + 128*b

  if (n_tiles > 0) {
    if (warp >= 8 && warp < 11) {
      // ================================ loaders =================================
      // Order per tile: gather q(u), whose stage completes through cp.async arrivals as
      // the rows land -> (new block) swap K/V once the previous block's last PV MMA is
      // done.
      const int lt = threadIdx.x - 256;  // 0 .. kLoadThreads-1
      KeyCursor kc;
      int prev_key = -1, kv_loads = 0, kv_issued = 0;
      // A tile's key and entries (once per warp: lane l holds query slots l + 32 m) are
      // fetched one tile ahead, so the entry loads of tile u+1 are in flight while the
      // rows of tile u are copied.
      constexpr int NE = (QPT + 31) / 32;
      int cur_key = 0, nxt_key = 0;
      int my_ent[NE], nxt_ent[NE];
      auto fetch = [&](int u, int& key, int (&ent)[NE]) {
        const int t = t_begin + u;
        key = kc.at(p.toff, p.keys, t);
        const int e0 = __ldg(&p.off[key]) + (t - __ldg(&p.toff[key])) * QPT;
        const int ne = min(QPT, __ldg(&p.off[key + 1]) - e0);
#pragma unroll
        for (int m = 0; m < NE; ++m) {
          const int qs = lane + 32 * m;
          ent[m] = qs < ne ? __ldg(&p.entries[e0 + qs]) : -1;
        }
      };
      if (n_tiles > 0) fetch(0, cur_key, my_ent);
      for (int u = 0; u < n_tiles && !*abort_flag; ++u) {
        const int st = u % kQStages;
        const int key = cur_key;
        if (u + 1 < n_tiles) fetch(u + 1, nxt_key, nxt_ent);
        const int bg = key / p.nb, c = key - bg * p.nb;
        const int b = bg / p.H_kv, g = bg - b * p.H_kv;
        const SeqSpan sp = seq_span(p.spans, b, p.N);
        if (!mbar_wait(&qempty[st], ((u / kQStages) & 1) ^ 1, p.wait_ns, abort_flag)) {
          *abort_flag = 1;
          break;
        }
        uint8_t* dq = sQ + st * L::kTile;
        // Each thread copies one fixed 16-byte column (chf) of the G head rows of the
        // queries q0, q0 + QS, ...: one shuffle for the query's entry and one source
        // address per query, then G copies at a fixed stride.
        static_assert(kLoadThreads % CH == 0, "loader threads cover whole rows");
        constexpr int QS = kLoadThreads / CH;          // queries per pass
        constexpr int NPASS = (QPT + QS - 1) / QS;     // passes (the same for every lane)
        const int chf = lt % CH;
        const __nv_bfloat16* qg = p.q + (sp.t0 * p.H_kv * G + (int64_t)g * G) * D + chf * 8;
        const int64_t qrow = (int64_t)p.H_kv * G * D;  // elements between consecutive queries
        uint8_t* dcol = dq + (chf >> 3) * L::kHalf;
#pragma unroll 2
        for (int pass = 0; pass < NPASS; ++pass) {
          const int qi = lt / CH + QS * pass;
          int ent = -1;
#pragma unroll
          for (int m = 0; m < NE; ++m) {
            const int v = __shfl_sync(0xffffffffu, my_ent[m], qi & 31);
            if ((qi >> 5) == m) ent = v;
          }
          if (qi < QPT) {
            const bool ok = ent >= 0;
            const __nv_bfloat16* src = qg + (ok ? (int64_t)(ent >> kSlotBits) * qrow : 0);
#pragma unroll
            for (int h = 0; h < G; ++h) {
              const int r = qi * G + h;
              cp_async_16(dcol + r * 128 + (((chf & 7) ^ (r & 7)) << 4), src + h * D, ok);
            }
          }
        }
        cp_async_commit();
        // this thread's copies count toward the tile's stage as soon as they land (the
        // MMA thread makes them visible to the tensor core with a proxy fence)
        cp_async_mbar_arrive(&qfull[st]);
        if (key != prev_key) {
          if (lt == 0) {
            // the previous block's MMAs must be done with K/V before they are replaced
            if (kv_loads > 0 && !mbar_wait(kvempty, (kv_loads - 1) & 1, p.wait_ns, abort_flag))
              *abort_flag = 1;
            if (!*abort_flag) {
              mbar_arrive_expect_tx(kvfull, 2 * L::kTile);
#pragma unroll
              for (int h = 0; h < L::kHalves; ++h) {
                tma_load_4d(sK + h * L::kHalf, &tm_k, kvfull, h * 64, g, sp.tn + c * 128, sp.tb);
                tma_load_4d(sV + h * L::kHalf, &tm_v, kvfull, h * 64, g, sp.tn + c * 128, sp.tb);
              }
              kv_issued = kv_loads + 1;
            }
          }
          ++kv_loads;
          prev_key = key;
        }
        cur_key = nxt_key;
#pragma unroll
        for (int m = 0; m < NE; ++m) my_ent[m] = nxt_ent[m];
      }
      cp_async_wait<0>();  // nothing may still be landing when the CTA exits
      // teardown: the last K/V TMA issued must have landed
      if (lt == 0 && kv_issued > 0) mbar_wait(kvfull, (kv_issued - 1) & 1, 1000000000ull);
    } else if (warp == 11) {
      // ============================== MMA issuer ================================
      if (lane == 0) {
        constexpr uint32_t idesc_s = umma_idesc_bf16_f32(128, 128);
        constexpr uint32_t idesc_o = umma_idesc_bf16_f32(128, D) | (1u << 16);  // B MN-major
        const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aP = smem_u32(sP);
        int kv_uses = 0;
        int cur_key = -1;
        bool issued = false;
        KeyCursor kc;
        auto issue_s = [&](int u) -> bool {
          const int st = u % kQStages, b = u & 1;
          if (!mbar_wait(&qfull[st], (u / kQStages) & 1, p.wait_ns, abort_flag)) return false;
          // the gathered rows were written by cp.async (generic proxy): order them before
          // the tensor core's reads
          fence_proxy_async_smem();
          if (!mbar_wait(&sfree[b], ((u >> 1) & 1) ^ 1, p.wait_ns, abort_flag)) return false;
          tc_fence_after();
          const uint32_t aQ = smem_u32(sQ + st * L::kTile);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * L::kHalf + (kk & 3) * 32;
            tc_mma_bf16(tmem + 128 * b, umma_desc_kmajor<128>(aQ + off),
                        umma_desc_kmajor<128>(aK + off), idesc_s, kk > 0 ? 1u : 0u);
          }
          tc_commit(&qempty[st]);
          tc_commit(&sfull[b]);
          issued = true;
          return true;
        };
        auto wait_kv = [&](int u) -> bool {
          const int key = kc.at(p.toff, p.keys, t_begin + u);
          if (key != cur_key) {
            if (!mbar_wait(kvfull, kv_uses & 1, p.wait_ns, abort_flag)) return false;
            ++kv_uses;
            cur_key = key;
          }
          return true;
        };
        bool ok = wait_kv(0) && issue_s(0);
        for (int u = 0; u < n_tiles && ok; ++u) {
          const int b = u & 1;
          const bool has_next = u + 1 < n_tiles;
          KeyCursor peek = kc;
          const bool next_same = has_next && peek.at(p.toff, p.keys, t_begin + u + 1) == cur_key;
          if (next_same) ok = issue_s(u + 1);
          if (!ok) break;
          if (!mbar_wait(&pfull[b], (u >> 1) & 1, p.wait_ns, abort_flag) ||
              !mbar_wait(&ofree[b], ((u >> 1) & 1) ^ 1, p.wait_ns, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {  // 16 keys per step
            const uint32_t pa = aP + b * 2 * L::kHalf + (kk >> 2) * L::kHalf + (kk & 3) * 32;
            const uint32_t vb = aV + kk * 2048;  // 16 K-rows = 2 swizzle atoms
            tc_mma_bf16(tmem + 256 + 128 * b, umma_desc_kmajor<128>(pa),
                        umma_desc_mnmajor_sw128(vb, L::kHalf), idesc_o, kk > 0 ? 1u : 0u);
          }
          tc_commit(&pempty[b]);
          tc_commit(&ofull[b]);
          if (has_next && !next_same) {
            tc_commit(kvempty);  // this block's K/V may be replaced
            ok = wait_kv(u + 1) && issue_s(u + 1);
          }
        }
        if (!ok) *abort_flag = 1;
        if (issued) {
          tc_commit(mmadone);
          mbar_wait(mmadone, 0, 1000000000ull);
        }
      }
    } else {
      // ====================== softmax + epilogue: warps 0-7 =======================
      // Warpgroup wg handles the tiles u with u % 2 == wg, i.e. TMEM buffer wg and
      // P tile wg, so the two groups' softmax and epilogues overlap.
      const int wg = warp >> 2;
      const int row = (warp & 3) * 32 + lane;  // TMEM lane
      uint8_t* sPw = sP + wg * 2 * L::kHalf;
      KeyCursor kc;
      const int qi = row / G;
      // the key and this row's entry of the warpgroup's next tile are fetched while the
      // current tile is processed
      auto fetch = [&](int u, int& key, int& ent) {
        const int t = t_begin + u;
        key = kc.at(p.toff, p.keys, t);
        const int e0 = __ldg(&p.off[key]) + (t - __ldg(&p.toff[key])) * QPT;
        const int ne = min(QPT, __ldg(&p.off[key + 1]) - e0);
        ent = qi < ne ? __ldg(&p.entries[e0 + qi]) : -1;
      };
      int nxt_key = 0, nxt_ent = -1;
      if (wg < n_tiles) fetch(wg, nxt_key, nxt_ent);
      for (int u = wg; u < n_tiles; u += 2) {
        const int b = wg;
        const int key = nxt_key, ent = nxt_ent;
        if (u + 2 < n_tiles) fetch(u + 2, nxt_key, nxt_ent);
        const int bg = key / p.nb, c = key - bg * p.nb;
        const int i = ent >> kSlotBits;
        const int rowv = opaque(row), lanev = opaque(lane);
        bool ok = __all_sync(0xffffffffu, mbar_wait(&sfull[b], (u >> 1) & 1, p.wait_ns, abort_flag));
        if (!ok) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        // causal mask j <= i (and j < N), scaled to log2 units
        const int bb = bg / p.H_kv, gg = bg - bb * p.H_kv;
        const SeqSpan sp = seq_span(p.spans, bb, p.N);
        const int jlim = ent >= 0 ? min(i, sp.len - 1) - c * 128 : -1;  // last valid column
        // blocks wholly before every query of the warp need no mask (the usual case)
        const bool full = __all_sync(0xffffffffu, jlim >= 127);
        // P (bf16) into this group's K-major smem operand, once its previous PV is done
        ok = __all_sync(0xffffffffu, mbar_wait(&pempty[b], ((u >> 1) & 1) ^ 1, p.wait_ns, abort_flag));
        if (!ok) {
          *abort_flag = 1;
          break;
        }
        const uint32_t srow = tmem + ((uint32_t)(rowv & ~31) << 16) + 128 * b;
        // exp2 of 64 scores (columns 64 hp ..) minus the offset ms -> P, row sum
        auto exp_pack = [&](const uint32_t (&r)[64], int hp, float ms, float& l) {
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {  // 8 columns -> one 16-byte P chunk
            float e[8];
#pragma unroll
            for (int x = 0; x < 8; ++x) {
              const float v = __uint_as_float(r[8 * ch + x]) * p.scale_log2 - ms;
              e[x] = (full || 64 * hp + 8 * ch + x <= jlim) ? ex2_fast(v) : 0.f;
              l += e[x];
            }
            uint4 w;
            w.x = pack_bf16(e[0], e[1]);
            w.y = pack_bf16(e[2], e[3]);
            w.z = pack_bf16(e[4], e[5]);
            w.w = pack_bf16(e[6], e[7]);
            *reinterpret_cast<uint4*>(sPw + kmaj_off<128>(rowv, 8 * hp + ch)) = w;
          }
        };
        auto load64 = [&](uint32_t (&r)[64], int hp) {
          tmem_ld_32x32b_x32(srow + 64 * hp, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
          tmem_ld_32x32b_x32(srow + 64 * hp + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
          tmem_wait_ld();
        };
        // One pass: the offset is the max of the first 32 columns (column 0, the block's
        // first key, is visible to every real row).  The partial lse ms + log2(l) is exact
        // for any offset; only overflow matters, so a row sum above 2^64 falls back to
        // the exact row max and a second pass.
        float ms, l = 0.f;
        {
          uint32_t r[64];
          load64(r, 0);
          float m0 = -INFINITY;
          if (full) {
#pragma unroll
            for (int x = 0; x < 32; x += 2) m0 = fmax3(m0, __uint_as_float(r[x]), __uint_as_float(r[x + 1]));
          } else {
#pragma unroll
            for (int x = 0; x < 32; x += 2)
              m0 = fmax3(m0, x <= jlim ? __uint_as_float(r[x]) : -INFINITY,
                         x + 1 <= jlim ? __uint_as_float(r[x + 1]) : -INFINITY);
          }
          ms = m0 == -INFINITY ? 0.f : m0 * p.scale_log2;
          exp_pack(r, 0, ms, l);
          load64(r, 1);
          exp_pack(r, 1, ms, l);
        }
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
          ms = m == -INFINITY ? 0.f : m * p.scale_log2;
          l = 0.f;
#pragma unroll 1
          for (int hp = 0; hp < 2; ++hp) {
            uint32_t r[64];
            load64(r, hp);
            exp_pack(r, hp, ms, l);
          }
        }
        // S[b] has been read: the next S MMA into it may start
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfree[b]);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pfull[b]);
        // ---- epilogue: O row / l -> bf16 partial, lse partial ----
        ok = __all_sync(0xffffffffu, mbar_wait(&ofull[b], (u >> 1) & 1, p.wait_ns, abort_flag));
        if (!ok) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        int prow = -1;
        if (ent >= 0) {
          prow = (int)(((sp.t0 * p.H_kv + (int64_t)gg * sp.len + i) * p.topk + (ent & kSlotMask)) * G +
                       row % G);
          p.lse_part[prow] = l > 0.f ? (ms + log2f(l)) * kLn2 : -INFINITY;
        }
        // Stage 64 columns at a time in this warp's own (now free) P rows, swizzled,
        // then store whole 128-byte partial-row segments (4 rows per instruction).
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          uint8_t* stg = sPw + h * L::kHalf + (warp & 3) * 32 * 128;
          uint32_t r2[2][32];
          const uint32_t orow = tmem + ((uint32_t)(rowv & ~31) << 16) + 256 + 128 * b + 64 * h;
          tmem_ld_32x32b_x32(orow, r2[0]);
          tmem_ld_32x32b_x32(orow + 32, r2[1]);
          tmem_wait_ld();
          if (h == D / 64 - 1) {  // O[b] has been read: the next PV into it may start
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ofree[b]);
          }
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const uint32_t (&r)[32] = r2[hh];
#pragma unroll
            for (int x = 0; x < 32; x += 8) {
              const float2 iv = make_float2(inv, inv);
              uint32_t wv[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 y = fmul2(
                    make_float2(__uint_as_float(r[x + 2 * e]), __uint_as_float(r[x + 2 * e + 1])), iv);
                wv[e] = pack_bf16(y.x, y.y);
              }
              *reinterpret_cast<uint4*>(stg + sw128_row(lanev, 4 * hh + x / 8)) =
                  make_uint4(wv[0], wv[1], wv[2], wv[3]);
            }
          }
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int x = lanev + 32 * k;
            const int rr = x >> 3, cc = x & 7;
            const int pr = __shfl_sync(0xffffffffu, prow, rr);
            const uint4 v = *reinterpret_cast<const uint4*>(stg + sw128_row(rr, cc));
            if (pr >= 0) *reinterpret_cast<uint4*>(p.o_part + (int64_t)pr * D + 64 * h + 8 * cc) = v;
          }
          __syncwarp();
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) set_status(p.status, MSA_ERR_DEVICE_TIMEOUT);
  if (warp == 11) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int G>
cudaError_t launch_fwd_tc_dg(const FwdTcParams& prm, const CUtensorMap& tk, const CUtensorMap& tv,
                             const Ctx& cx, cudaStream_t st) {
  using L = TcLayout<D>;
  auto kern = fwd_tc_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  kernel_event(MSA_KERNEL_FWD, true, st);
  kern<<<cx.num_sms, kTcThreads, L::kAlloc, st>>>(tk, tv, prm);
  kernel_event(MSA_KERNEL_FWD, false, st);
  note_launch();
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_fwd_tc_d(int G, const FwdTcParams& prm, const CUtensorMap& tk,
                            const CUtensorMap& tv, const Ctx& cx, cudaStream_t st) {
  switch (G) {
    case 1: return launch_fwd_tc_dg<D, 1>(prm, tk, tv, cx, st);
    case 2: return launch_fwd_tc_dg<D, 2>(prm, tk, tv, cx, st);
    case 4: return launch_fwd_tc_dg<D, 4>(prm, tk, tv, cx, st);
    case 8: return launch_fwd_tc_dg<D, 8>(prm, tk, tv, cx, st);
    case 16: return launch_fwd_tc_dg<D, 16>(prm, tk, tv, cx, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_attn_fwd_tc(const Shape& s, const void* q, const void* k, const void* v,
                               const Plan& pl, __nv_bfloat16* o_part, float* lse_part,
                               const Ctx& cx, cudaStream_t st) {
  CUtensorMap tk, tv;
  const uint64_t dims[4] = {(uint64_t)s.d, (uint64_t)s.H_kv, s.tma_tokens(), s.tma_batches()};
  const uint64_t strides[3] = {(uint64_t)s.d * 2, (uint64_t)s.H_kv * s.d * 2,
                               s.tma_tokens() * s.H_kv * s.d * 2};
  const uint32_t box[4] = {64, 1, 128, 1};
  if (!encode_tiled(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, k, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tiled(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, v, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  FwdTcParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.spans = s.spans;
  prm.off = pl.off;
  prm.toff = pl.toff;
  prm.entries = pl.entries;
  prm.o_part = o_part;
  prm.lse_part = lse_part;
  prm.keys = s.keys();
  prm.N = s.N;
  prm.H_kv = s.H_kv;
  prm.nb = s.nb;
  prm.topk = s.topk;
  prm.scale_log2 = s.scale * kLog2e;
  prm.wait_ns = cx.wait_ns;
  prm.status = cx.status;
  if (s.d == 128) return launch_fwd_tc_d<128>(s.G, prm, tk, tv, cx, st);
  return launch_fwd_tc_d<64>(s.G, prm, tk, tv, cx, st);
}

}  // namespace msa
