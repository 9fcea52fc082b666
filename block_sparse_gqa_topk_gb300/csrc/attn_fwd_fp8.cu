// attn_fwd_fp8.cu -- main-branch block-sparse forward with FP8 (E4M3) operands on the
// 5th-generation tensor cores (tcgen05.mma kind::f8f6f4), and the quantisers that
// prepare those operands from the bf16 q, k, v of a training step.
//
// Method: MSA summary (7minutos.es), "Cómo funcionan las dos ramas" ¶3 (exact softmax
// attention of every head of a group over the causally visible tokens of the group's
// blocks) and "El codiseño del kernel" (FP8 among the precisions of the MSA attention
// kernels; KV-outer query gather with split partials and a combine).
//
// FP8 reading (the pages give no recipe):
//   q:  one float32 scale per (token, head) row, s_q = amax / 448 (1 for a zero row);
//   k, v: one float32 scale per (batch, group, 128-key block), s = amax / 448 over the
//       block's real keys and all d values (1 for a zero block);
//   code = E4M3 nearest to float32(x / s), ties to even, saturating at 448;
//   scores  S = s_q s_k (q8 . k8) (fp32 accumulate), softmax with the exact row max;
//   P = exp(S - max) in (0, 1] rounded to E4M3 (no scale), l = sum of the unrounded P;
//   O = s_v (P8 . v8) / l, lse = max + log l (natural log), both from the fp32 P.
// v is stored transposed per block, v8t[b][g][c][d][128 keys], so that it is the
// K-major B operand of the P V product, like every other operand here.
//
// A tile is one key block c of one (batch, group) and 128 rows = 128/G gathered queries
// x G heads (the inverted lists of plan.cu, as the bf16 forward).  Per CTA:
//   warps 8-10 loaders: cp.async gathers of the tile's q8 rows (128 B each) into a
//              4-stage ring, 128-byte swizzled K-major; one thread TMA-loads K8 and V8t
//              when the key block changes;
//   warp 11    TMEM owner and MMA thread: S = Q8 K8^T (M=N=128, K=d, 4 x K=32) into a
//              2-deep TMEM ring, then O = P8 V8 (K = 128 keys);
//   warps 0-7  two softmax warpgroups taking alternate tiles (thread = row = TMEM lane):
//              the row max over S, P = exp2((S - max) c) with c = log2(e) scale s_q s_k,
//              P8 to shared memory, the row sum; then O from TMEM times s_v / l -> bf16
//              partial and the partial lse.  The per-row merge is the bf16 forward's.
#include <cudaTypedefs.h>
#include <cuda_fp8.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace msa {
namespace {

constexpr int kThreads8 = 384;  // 12 warps: 8 softmax, 3 loaders, 1 MMA
constexpr int kLoad8 = 96;
constexpr int kStages8 = 4;
constexpr int kD8 = 128;        // head dim of the FP8 forward
constexpr float kLog2e8 = 1.4426950408889634f;
constexpr float kLn2_8 = 0.6931471805599453f;

struct Fwd8Params {
  const uint8_t* q8;      // [B][N][H_q][d] E4M3
  const float* q_scale;   // [B][N][H_q]
  const float* k_scale;   // [B][H_kv][nb]
  const float* v_scale;   // [B][H_kv][nb]
  const int* off;
  const int* toff;
  const int* entries;
  __nv_bfloat16* o_part;  // [(rkv*topk + slot)*G + h][d]
  float* lse_part;        // [(rkv*topk + slot)*G + h]
  int64_t keys;
  int N, H_kv, nb, topk;
  float scale_log2;
  uint64_t wait_ns;
  int* status;
};

struct L8 {
  static constexpr int kTile = 128 * 128;  // [128 rows][128 bytes], 128-byte swizzle
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTile;
  static constexpr int kQ = kV + kTile;                 // kStages8 tiles
  static constexpr int kP = kQ + kStages8 * kTile;      // [2][128 rows][128 keys] E4M3
  static constexpr int kBar = kP + 2 * kTile;
  // barriers: kvfull, kvempty, qfull[4], qempty[4], sfull[2], ofull[2], sfree[2],
  //           ofree[2], pfull[2], pempty[2], mmadone
  static constexpr int kNumBars = 2 + 2 * kStages8 + 12 + 1;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;
};

// Instruction descriptor, kind::f8f6f4: E4M3 A and B (format 0), fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// D[tmem] (+)= A[smem] x B[smem]^T with 8-bit operands (K = 32 per instruction).
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ uint32_t sw_row(int r, int chunk) {  // 128-byte rows, swizzled
  return (uint32_t)(r * 128 + (((chunk & 7) ^ (r & 7)) << 4));
}
__device__ __forceinline__ void fence_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Two floats -> two E4M3 bytes (lo in the low byte), round to nearest even, saturating.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3) & 0xFFFFu;
}

__device__ __forceinline__ int find_key8(const int* __restrict__ toff, int64_t keys, int t) {
  int64_t lo = 0, hi = keys - 1;
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) >> 1;
    if (__ldg(&toff[mid]) <= t) lo = mid; else hi = mid - 1;
  }
  return (int)lo;
}
// Key of tile t given the key of an earlier tile of the same CTA (tiles are visited in
// increasing order, so keys only move forward; empty keys are skipped).
struct Cursor8 {
  int key = -1;
  __device__ __forceinline__ int at(const int* __restrict__ toff, int64_t keys, int t) {
    if (key < 0) {
      key = find_key8(toff, keys, t);
    } else {
      while (key + 1 < keys && __ldg(&toff[key + 1]) <= t) ++key;
    }
    return key;
  }
};

template <int G>
__global__ void __launch_bounds__(kThreads8, 1)
    fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const Fwd8Params p) {
  using L = L8;
  constexpr int QPT = 128 / G;
  constexpr int CH = kD8 / 16;  // 16-byte chunks per q8 row
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
  uint64_t* qempty = qfull + kStages8;
  uint64_t* sfull = qempty + kStages8;
  uint64_t* ofull = sfull + 2;
  uint64_t* sfree = ofull + 2;
  uint64_t* ofree = sfree + 2;
  uint64_t* pfull = ofree + 2;
  uint64_t* pempty = pfull + 2;
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
    for (int s = 0; s < kStages8; ++s) {
      mbar_init(&qfull[s], kLoad8);
      mbar_init(&qempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sfull[b], 1);
      mbar_init(&ofull[b], 1);
      mbar_init(&sfree[b], 4);
      mbar_init(&ofree[b], 4);
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
      const int lt = threadIdx.x - 256;
      static_assert(kLoad8 % CH == 0, "loader threads cover whole rows");
      constexpr int RS = kLoad8 / CH;  // queries per pass
      const int chf = lt % CH;
      Cursor8 kc;
      int prev_key = -1, kv_loads = 0, kv_issued = 0;
      // a tile's key and entries (lane l holds query slots l + 32 m), fetched one tile
      // ahead so the entry loads of tile u+1 overlap the copies of tile u
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
        const int st = u % kStages8;
        const int key = cur_key;
        if (u + 1 < n_tiles) fetch(u + 1, nxt_key, nxt_ent);
        const int bg = key / p.nb, c = key - bg * p.nb;
        const int b = bg / p.H_kv, g = bg - b * p.H_kv;
        if (!mbar_wait(&qempty[st], ((u / kStages8) & 1) ^ 1, p.wait_ns, abort_flag)) {
          *abort_flag = 1;
          break;
        }
        uint8_t* dq = sQ + st * L::kTile;
        const uint8_t* qg = p.q8 + ((int64_t)b * p.N * p.H_kv * G + (int64_t)g * G) * kD8 + chf * 16;
        const int64_t qrow = (int64_t)p.H_kv * G * kD8;  // bytes between consecutive queries
        // whole queries per thread: one shuffle and one source address per query, then
        // its G head rows at a fixed stride (RS queries per pass, the same passes for
        // every lane)
        constexpr int NPASS = (QPT + RS - 1) / RS;
#pragma unroll 2
        for (int pass = 0; pass < NPASS; ++pass) {
          const int qi = lt / CH + RS * pass;
          int ent = -1;
#pragma unroll
          for (int m = 0; m < NE; ++m) {
            const int v = __shfl_sync(0xffffffffu, my_ent[m], qi & 31);
            if ((qi >> 5) == m) ent = v;
          }
          if (qi < QPT) {
            const bool ok = ent >= 0;
            const uint8_t* src = qg + (ok ? (int64_t)(ent >> kSlotBits) * qrow : 0);
#pragma unroll
            for (int h = 0; h < G; ++h) cp_async_16(dq + sw_row(qi * G + h, chf), src + h * kD8, ok);
          }
        }
        cp_async_commit();
        // this thread's copies count toward the tile's stage as soon as they land (the
        // MMA thread orders them before the tensor core's reads with a proxy fence)
        cp_async_mbar_arrive(&qfull[st]);
        if (key != prev_key) {
          if (lt == 0) {
            if (kv_loads > 0 && !mbar_wait(kvempty, (kv_loads - 1) & 1, p.wait_ns, abort_flag))
              *abort_flag = 1;
            if (!*abort_flag) {
              mbar_arrive_expect_tx(kvfull, 2 * L::kTile);
              tma_load_4d(sK, &tm_k, kvfull, 0, g, c * 128, b);
              tma_load_3d(sV, &tm_v, kvfull, 0, c * 128, b * p.H_kv + g);
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
      if (lt == 0 && kv_issued > 0) mbar_wait(kvfull, (kv_issued - 1) & 1, 1000000000ull);
    } else if (warp == 11) {
      // ============================== MMA issuer ================================
      if (lane == 0) {
        constexpr uint32_t idesc = idesc_e4m3_f32(128, 128);
        const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aP = smem_u32(sP);
        int kv_uses = 0, cur_key = -1;
        bool issued = false;
        Cursor8 kc;
        auto issue_s = [&](int u) -> bool {
          const int st = u % kStages8, b = u & 1;
          if (!mbar_wait(&qfull[st], (u / kStages8) & 1, p.wait_ns, abort_flag)) return false;
          fence_async();  // the q rows came by cp.async (generic proxy)
          if (!mbar_wait(&sfree[b], ((u >> 1) & 1) ^ 1, p.wait_ns, abort_flag)) return false;
          tc_fence_after();
          const uint32_t aQ = smem_u32(sQ + st * L::kTile);
#pragma unroll
          for (int kk = 0; kk < kD8 / 32; ++kk)
            tc_mma_f8(tmem + 128 * b, umma_desc_kmajor<128>(aQ + 32 * kk),
                      umma_desc_kmajor<128>(aK + 32 * kk), idesc, kk > 0 ? 1u : 0u);
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
          Cursor8 peek = kc;
          const bool next_same = has_next && peek.at(p.toff, p.keys, t_begin + u + 1) == cur_key;
          if (next_same) ok = issue_s(u + 1);
          if (!ok) break;
          if (!mbar_wait(&pfull[b], (u >> 1) & 1, p.wait_ns, abort_flag) ||
              !mbar_wait(&ofree[b], ((u >> 1) & 1) ^ 1, p.wait_ns, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // O = P8 V8: A = P8 [rows][keys], B = V8t [d][keys], both K-major (K = keys)
#pragma unroll
          for (int kk = 0; kk < 128 / 32; ++kk)
            tc_mma_f8(tmem + 256 + 128 * b, umma_desc_kmajor<128>(aP + b * L::kTile + 32 * kk),
                      umma_desc_kmajor<128>(aV + 32 * kk), idesc, kk > 0 ? 1u : 0u);
          tc_commit(&pempty[b]);
          tc_commit(&ofull[b]);
          if (has_next && !next_same) {
            tc_commit(kvempty);
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
      const int wg = warp >> 2;
      const int row = (warp & 3) * 32 + lane;  // TMEM lane
      uint8_t* sPw = sP + wg * L::kTile;
      Cursor8 kc;
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
        const int bb = bg / p.H_kv, g = bg - bb * p.H_kv;
        // per-row score factor: log2(e) * scale * s_q(row) * s_k(block)
        const float sq = ent >= 0 ? __ldg(&p.q_scale[((int64_t)bb * p.N + i) * p.H_kv * G + g * G + row % G])
                                  : 0.f;
        const float cf = p.scale_log2 * sq * __ldg(&p.k_scale[key]);
        const float sv = __ldg(&p.v_scale[key]);
        bool ok = __all_sync(0xffffffffu, mbar_wait(&sfull[b], (u >> 1) & 1, p.wait_ns, abort_flag));
        if (!ok) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const int jlim = ent >= 0 ? min(i, p.N - 1) - c * 128 : -1;  // last valid column
        const bool full = __all_sync(0xffffffffu, jlim >= 127);
        const uint32_t srow = tmem + ((uint32_t)(row & ~31) << 16) + 128 * b;
        // pass 1: the row max over the valid columns
        float m = -INFINITY;
#pragma unroll 1
        for (int h = 0; h < 4; ++h) {
          uint32_t r[32];
          float mh;
          tmem_ld_max_32x32b_x32(srow + 32 * h, r, mh);  // mh: max of the 32 columns
          tmem_wait_ld();
          if (full) {
            m = fmaxf(m, mh);
          } else {
#pragma unroll
            for (int x = 0; x < 32; ++x) m = fmaxf(m, 32 * h + x <= jlim ? __uint_as_float(r[x]) : -INFINITY);
          }
        }
        // P8 into this group's smem operand, once its previous P V product is done
        ok = __all_sync(0xffffffffu, mbar_wait(&pempty[b], ((u >> 1) & 1) ^ 1, p.wait_ns, abort_flag));
        if (!ok) {
          *abort_flag = 1;
          break;
        }
        const float mc = m == -INFINITY ? 0.f : m * cf;
        float l = 0.f;
        // pass 2: P = exp2(S cf - max cf) in (0, 1] -> E4M3, row sum of the fp32 P
#pragma unroll 1
        for (int h = 0; h < 4; ++h) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(srow + 32 * h, r);
          tmem_wait_ld();
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {  // 16 columns -> one 16-byte P8 chunk
            float e[16];
#pragma unroll
            for (int x = 0; x < 16; ++x) {
              const int col = 32 * h + 16 * ch + x;
              e[x] = (full || col <= jlim) ? ex2_fast(__uint_as_float(r[16 * ch + x]) * cf - mc) : 0.f;
              l += e[x];
            }
            uint4 w;
            w.x = e4m3x2(e[0], e[1]) | (e4m3x2(e[2], e[3]) << 16);
            w.y = e4m3x2(e[4], e[5]) | (e4m3x2(e[6], e[7]) << 16);
            w.z = e4m3x2(e[8], e[9]) | (e4m3x2(e[10], e[11]) << 16);
            w.w = e4m3x2(e[12], e[13]) | (e4m3x2(e[14], e[15]) << 16);
            *reinterpret_cast<uint4*>(sPw + sw_row(row, 2 * h + ch)) = w;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfree[b]);
        fence_async();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pfull[b]);
        // ---- epilogue: O row * s_v / l -> bf16 partial, lse partial ----
        ok = __all_sync(0xffffffffu, mbar_wait(&ofull[b], (u >> 1) & 1, p.wait_ns, abort_flag));
        if (!ok) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const float inv = l > 0.f ? sv / l : 0.f;
        int prow = -1;
        if (ent >= 0) {
          prow = (int)((((int64_t)bg * p.N + i) * p.topk + (ent & kSlotMask)) * G + row % G);
          p.lse_part[prow] = l > 0.f ? (mc + log2f(l)) * kLn2_8 : -INFINITY;
        }
        const uint32_t orow = tmem + ((uint32_t)(row & ~31) << 16) + 256 + 128 * b;
        // Stage 64 columns at a time (32 rows x 128 bytes) in this warp's own P rows,
        // free since the P V product is done, then store whole 128-byte segments of the
        // partial rows (4 rows per instruction).
        uint8_t* stg = sPw + (warp & 3) * 32 * 128;
#pragma unroll
        for (int hp = 0; hp < 2; ++hp) {
          uint32_t r2[2][32];
          tmem_ld_32x32b_x32(orow + 64 * hp, r2[0]);
          tmem_ld_32x32b_x32(orow + 64 * hp + 32, r2[1]);
          tmem_wait_ld();
          if (hp == 1) {  // O[b] has been read: the next P V product into it may start
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ofree[b]);
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int x = 0; x < 32; x += 8) {
              const float2 iv = make_float2(inv, inv);
              uint32_t wv[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {  // packed pairs: one FMUL2 per two values
                const float2 y = fmul2(
                    make_float2(__uint_as_float(r2[h][x + 2 * e]), __uint_as_float(r2[h][x + 2 * e + 1])),
                    iv);
                wv[e] = pack_bf16(y.x, y.y);
              }
              *reinterpret_cast<uint4*>(stg + sw_row(lane, 4 * h + x / 8)) =
                  make_uint4(wv[0], wv[1], wv[2], wv[3]);
            }
          }
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int x = lane + 32 * k;
            const int rr = x >> 3, cc = x & 7;
            const int pr = __shfl_sync(0xffffffffu, prow, rr);
            const uint4 v = *reinterpret_cast<const uint4*>(stg + sw_row(rr, cc));
            if (pr >= 0) *reinterpret_cast<uint4*>(p.o_part + (int64_t)pr * kD8 + 64 * hp + 8 * cc) = v;
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

// ---------------------------------------------------------------------------
// Quantisers
// ---------------------------------------------------------------------------
// One CTA per (b, g, block c) of k or v [B][N][H_kv][128]: the block's amax over its real
// keys, s = amax / 448 (1 for a zero block), codes of x / s.  k keeps its layout
// (x8 [B][N][H_kv][d]); v is written transposed per block (x8 = v8t [B][H_kv][nb][d][128],
// keys past N as 0).
template <bool kTranspose>
__global__ void __launch_bounds__(256) quantize_block_fp8_kernel(
    const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ x8, float* __restrict__ scale,
    int N, int H_kv, int nb) {
  __shared__ float red[8];
  __shared__ uint8_t tile[kTranspose ? 128 * 129 : 1];  // [d][keys], padded rows
  const int64_t blk = blockIdx.x;  // (b * H_kv + g) * nb + c
  const int c = (int)(blk % nb);
  const int64_t bg = blk / nb;
  const int g = (int)(bg % H_kv);
  const int64_t b = bg / H_kv;
  const int tid = threadIdx.x;
  // thread tid handles key r = tid / 2, d values [64 (tid % 2), +64)
  const int r = tid >> 1, d0 = (tid & 1) * 64;
  const int j = c * 128 + r;
  const bool in = j < N;
  float v[64];
  const __nv_bfloat16* src = x + ((b * N + (in ? j : 0)) * H_kv + g) * kD8 + d0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint4 w = in ? __ldg(reinterpret_cast<const uint4*>(src) + q) : make_uint4(0u, 0u, 0u, 0u);
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[8 * q + 2 * e] = __low2float(h2[e]);
      v[8 * q + 2 * e + 1] = __high2float(h2[e]);
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < 64; ++e) amax = fmaxf(amax, fabsf(v[e]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[w]);
  const float sc = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  if (tid == 0) scale[blk] = sc;
  uint32_t codes[16];  // 64 codes, 4 per word
#pragma unroll
  for (int e = 0; e < 64; e += 4) {
    const uint32_t lo = (uint32_t)__nv_cvt_float2_to_fp8x2(
                            make_float2(__fdiv_rn(v[e], sc), __fdiv_rn(v[e + 1], sc)), __NV_SATFINITE,
                            __NV_E4M3) & 0xFFFFu;
    const uint32_t hi = (uint32_t)__nv_cvt_float2_to_fp8x2(
                            make_float2(__fdiv_rn(v[e + 2], sc), __fdiv_rn(v[e + 3], sc)), __NV_SATFINITE,
                            __NV_E4M3) & 0xFFFFu;
    codes[e / 4] = in ? (lo | (hi << 16)) : 0u;
  }
  if constexpr (!kTranspose) {
    if (in) {
      uint4* dst = reinterpret_cast<uint4*>(x8 + ((b * N + j) * H_kv + g) * kD8 + d0);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        dst[q] = make_uint4(codes[4 * q], codes[4 * q + 1], codes[4 * q + 2], codes[4 * q + 3]);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 64; ++e) tile[(d0 + e) * 129 + r] = (uint8_t)(codes[e / 4] >> (8 * (e % 4)));
    __syncthreads();
    // row dd of the block's [d][128 keys] tile: 128 bytes, written as 8 x 16 bytes
    uint8_t* out = x8 + blk * (int64_t)(kD8 * 128);
    for (int q = tid; q < kD8 * 8; q += 256) {
      const int dd = q >> 3, k0 = (q & 7) * 16;
      uint32_t w[4];
#pragma unroll
      for (int z = 0; z < 4; ++z)
        w[z] = (uint32_t)tile[dd * 129 + k0 + 4 * z] | ((uint32_t)tile[dd * 129 + k0 + 4 * z + 1] << 8) |
               ((uint32_t)tile[dd * 129 + k0 + 4 * z + 2] << 16) |
               ((uint32_t)tile[dd * 129 + k0 + 4 * z + 3] << 24);
      *reinterpret_cast<uint4*>(out + dd * 128 + k0) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

template <int G>
cudaError_t launch_fp8_g(const Fwd8Params& prm, const CUtensorMap& tk, const CUtensorMap& tv,
                         const Ctx& cx, cudaStream_t st) {
  auto kern = fwd_fp8_kernel<G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L8::kAlloc);
  if (e != cudaSuccess) return e;
  kernel_event(MSA_KERNEL_FWD, true, st);
  kern<<<cx.num_sms, kThreads8, L8::kAlloc, st>>>(tk, tv, prm);
  kernel_event(MSA_KERNEL_FWD, false, st);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize_blocks_fp8(const Shape& s, const void* x, uint8_t* x8, float* scale,
                                       bool transpose, cudaStream_t st) {
  const int64_t blocks = (int64_t)s.B * s.H_kv * s.nb;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  if (transpose)
    quantize_block_fp8_kernel<true><<<(unsigned)blocks, 256, 0, st>>>(xb, x8, scale, s.N, s.H_kv, s.nb);
  else
    quantize_block_fp8_kernel<false><<<(unsigned)blocks, 256, 0, st>>>(xb, x8, scale, s.N, s.H_kv, s.nb);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_attn_fwd_fp8_tc(const Shape& s, const uint8_t* q8, const float* q_scale,
                                   const uint8_t* k8, const float* k_scale, const uint8_t* v8t,
                                   const float* v_scale, const Plan& pl, __nv_bfloat16* o_part,
                                   float* lse_part, const Ctx& cx, cudaStream_t st) {
  if (s.d != kD8) return cudaErrorNotSupported;
  CUtensorMap tk, tv;
  {
    const uint64_t dims[4] = {(uint64_t)kD8, (uint64_t)s.H_kv, (uint64_t)s.N, (uint64_t)s.B};
    const uint64_t strides[3] = {(uint64_t)kD8, (uint64_t)s.H_kv * kD8,
                                 (uint64_t)s.N * s.H_kv * kD8};
    const uint32_t box[4] = {128, 1, 128, 1};
    if (!encode_tiled(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, k8, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    // v8t [B*H_kv][nb*d][128 keys]: the block's [d][128] tile at row c*d
    const uint64_t dims[3] = {128, (uint64_t)s.nb * kD8, (uint64_t)s.B * s.H_kv};
    const uint64_t strides[2] = {128, (uint64_t)s.nb * kD8 * 128};
    const uint32_t box[3] = {128, 128, 1};
    if (!encode_tiled(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, v8t, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  Fwd8Params prm;
  prm.q8 = q8;
  prm.q_scale = q_scale;
  prm.k_scale = k_scale;
  prm.v_scale = v_scale;
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
  prm.scale_log2 = s.scale * kLog2e8;
  prm.wait_ns = cx.wait_ns;
  prm.status = cx.status;
  switch (s.G) {
    case 1: return launch_fp8_g<1>(prm, tk, tv, cx, st);
    case 2: return launch_fp8_g<2>(prm, tk, tv, cx, st);
    case 4: return launch_fp8_g<4>(prm, tk, tv, cx, st);
    case 8: return launch_fp8_g<8>(prm, tk, tv, cx, st);
    default: return launch_fp8_g<16>(prm, tk, tv, cx, st);
  }
}

}  // namespace msa

using namespace msa;

extern "C" {

int msa_quantize_fwd_fp8(const msa_problem_t* p, const void* q, const void* k, const void* v,
                         uint8_t* q8, float* q_scale, uint8_t* k8, float* k_scale, uint8_t* v8t,
                         float* v_scale, cudaStream_t stream) {
  Shape s;
  int rc = validate_problem(p, &s);
  if (rc) return rc;
  if (s.d != kD8) return MSA_ERR_UNSUPPORTED;
  if (s.B == 0 || s.N == 0) return MSA_OK;
  const void* ptrs[] = {q, k, v, q8, q_scale, k8, k_scale, v8t, v_scale};
  for (const void* t : ptrs)
    if (!t || (reinterpret_cast<uintptr_t>(t) & 15) != 0) return MSA_ERR_ARG;
  // q: one scale per (token, head) row -- the per-row quantiser over H_q heads
  msa_problem_t pq = *p;
  pq.H_kv = p->H_q;
  if ((rc = msa_quantize_kv_fp8(&pq, q, q8, q_scale, stream))) return rc;
  if (launch_quantize_blocks_fp8(s, k, k8, k_scale, false, stream) != cudaSuccess ||
      launch_quantize_blocks_fp8(s, v, v8t, v_scale, true, stream) != cudaSuccess)
    return MSA_ERR_CUDA;
  return MSA_OK;
}

int msa_fwd_fp8(const msa_problem_t* p, const uint8_t* q8, const float* q_scale, const uint8_t* k8,
                const float* k_scale, const uint8_t* v8t, const float* v_scale,
                const int32_t* block_idx, void* o, float* lse, void* workspace,
                size_t workspace_bytes, cudaStream_t stream) {
  Shape s;
  int rc = validate_problem(p, &s);
  if (rc) return rc;
  if (s.d != kD8) return MSA_ERR_UNSUPPORTED;
  if (s.B == 0 || s.N == 0) return MSA_OK;
  const void* ptrs[] = {q8, q_scale, k8, k_scale, v8t, v_scale, block_idx, o, lse};
  for (const void* t : ptrs)
    if (!t || (reinterpret_cast<uintptr_t>(t) & 15) != 0) return MSA_ERR_ARG;
  if (!workspace || workspace_bytes < msa_workspace_size(p, MSA_WS_FWD)) return MSA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return MSA_ERR_ARG;
  Ctx cx;
  if ((rc = device_ctx(&cx))) return rc;
  Plan pl = plan_carve(s, workspace);
  uint8_t* w = static_cast<uint8_t*>(workspace) + plan_bytes(s);
  const size_t parts = (size_t)s.rows_kv() * s.topk * s.G;
  __nv_bfloat16* o_part = reinterpret_cast<__nv_bfloat16*>(w);
  float* lse_part = reinterpret_cast<float*>(w + align256(parts * s.d * 2));
  cudaError_t e = launch_plan(s, block_idx, 128 / s.G, pl, cx, stream);
  if (e == cudaSuccess)
    e = launch_attn_fwd_fp8_tc(s, q8, q_scale, k8, k_scale, v8t, v_scale, pl, o_part, lse_part,
                               cx, stream);
  if (e == cudaSuccess) e = launch_attn_fwd_combine(s, block_idx, o_part, lse_part, o, lse, stream);
  return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

}  // extern "C"
