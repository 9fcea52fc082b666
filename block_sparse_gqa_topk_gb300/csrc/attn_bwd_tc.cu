// attn_bwd_tc.cu -- fused backward of the MSA main branch and of the KL alignment loss
// on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Method: Flash-MSA article (tech.kuratif.com) ¶7 -- proxy and main gradients in one
// pass over the cached block indices (the proxy's signal needs both branches'
// probabilities); MSA summary (7minutos.es), "Cómo se entrena MSA" ¶1-2 -- KL from
// the group-averaged main distribution (teacher, detached) to the index
// distribution over the selected tokens; only the index projections receive it.
//
// Work: one CTA owns one key block (b, g, c) at a time (static round-robin over keys
// in block-major order, heaviest blocks first) and walks the block's inverted list in
// chunks of R rows (R/G gathered queries x G heads; R = 64 for G >= 4, 16 G for G = 1, 2,
// so a chunk holds at most the 16 query slots of the z and dk_idx products).
//   tcgen05 (one MMA thread, accumulators in TMEM, every M = 128):
//     (1) S^T  = K Q^T          M=128 keys, N=R rows, K=d
//     (2) dP^T = V dO^T         M=128 keys, N=R rows, K=d
//     (z) z^T  = k_idx q_idx^T  M=128 keys, N=16 slots, K=d_idx   (into the dQ^T columns)
//     (3) dV  += P^T dO         M=128 keys, N=d,  K=R rows    (dO as MN-major B)
//     (4) dK  += dS^T Q         M=128 keys, N=d,  K=R rows    (Q as MN-major B)
//     (5) dQ^T = K^T dS^T       M=d, N=R rows, K=128 keys     (both MN-major)
//     (6) dk_idx += dz^T q_idx  M=128 keys, N=d_idx, K=16 slots
//   epilogue warps 0-7 (two warpgroups, each owning R/2 of the R row columns; thread =
//   key):
//     E1  P^T = exp(scale S^T - lse), dS^T = P^T (dP^T - D) -> smem; the teacher p_T
//         (group mean of P) stays in registers; with z^T from TMEM: p_I, the KL and
//         dz = w (p_I - p_T) for the warpgroup's slots -> dz^T in smem
//     dq_idx (mma.sync, per warpgroup, while (3)-(6) run): dq_idx^T = k_idx^T dz^T
//     E2  dQ^T from TMEM (thread = d) -> bf16 per-slot partials
// Chunk u+1's (1)(2) overlap chunk u's E2.  After the block's last chunk dK, dV and
// dk_idx (TMEM) are written once: no atomics on dk/dv/dk_idx.
// Warp 8: loader (TMA boxes for q, G head rows per query, q_idx rows, K, V and k_idx;
// cp.async for the per-row scalars).  Warp 9: cp.async gather of the chunk's dO rows.
// Warp 10: TMEM owner and MMA issuer.
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace msa {
namespace {

constexpr int kThreads = 352;  // 11 warps
constexpr int kEpiWarps = 8;
constexpr int kLoadArrivals = 96;  // per chunk: warp 8 (plain stores + cp.async), warp 9 (cp.async)
// rows per chunk: 64 (64/G queries) for G >= 4; 16 G (16 queries) for G = 1, 2, so a
// chunk never holds more than the 16 query slots of the z and dk_idx MMAs
__host__ __device__ constexpr int rows_per_chunk(int G) { return G >= 4 ? 64 : 16 * G; }
constexpr int kQS = 16;    // query slots per chunk
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct BwdTcParams {
  const __nv_bfloat16 *q, *dO, *q_idx, *k_idx;
  const int2* spans;  // packed batches: (start, end) per sequence
  const float *lse, *Dv, *lse_idx;
  const int* off;
  const int* entries;
  __nv_bfloat16 *dk, *dv, *dq_part, *dqi_part;
  float* dki_part;
  double* kl_acc;
  int64_t keys;
  int B, N, T, H_kv, nb, topk, DI;
  float scale, scale_log2, sidx, sidx_log2, w;
  uint64_t wait_ns;
  int* status;
};

template <int D, int R>
struct BL {
  static constexpr int kKH = 128 * 128;             // [128][64] bf16 block
  static constexpr int kK = 0;
  static constexpr int kV = kK + (D / 64) * kKH;
  static constexpr int kKi = kV + (D / 64) * kKH;   // k_idx [128][64], zero-padded
  static constexpr int kQH = R * 128;               // [R][64] bf16 block
  // big stage (2 slots): q and dO rows of a chunk, released by the MMAs (3)-(5)
  static constexpr int kSQ = 0;
  static constexpr int kSdO = kSQ + (D / 64) * kQH;
  static constexpr int kBig = kSdO + (D / 64) * kQH;
  // small stage (3 slots): q_idx rows and per-row scalars, released by the epilogue
  // and the dk_idx MMA
  static constexpr int kSQi = 0;                      // [16][64] bf16 (SW128)
  static constexpr int kSLse = kSQi + 16 * 128;       // float[64] lse (natural log)
  static constexpr int kSD = kSLse + 64 * 4;          // float[64] D
  static constexpr int kSRi = kSD + 64 * 4;           // int[64] query index of the row, -1 pad
  static constexpr int kSRp = kSRi + 64 * 4;          // int[64] dq partial row, -1 pad
  static constexpr int kSQiq = kSRp + 64 * 4;         // int[16] query index of the slot, -1 pad
  static constexpr int kSQp = kSQiq + 16 * 4;         // int[16] dq_idx partial row, -1 pad
  static constexpr int kSLi = kSQp + 16 * 4;          // float[16] lse_idx (natural log)
  static constexpr int kSmall = ((kSLi + 16 * 4) + 1023) & ~1023;
  static constexpr int kBig0 = kKi + kKH;
  static constexpr int kSmall0 = kBig0 + 2 * kBig;
  static constexpr int kPT = kSmall0 + 3 * kSmall;    // P^T [128][64] bf16 (SW128)
  static constexpr int kdST = kPT + 128 * 128;        // dS^T [128][64]
  // dz^T bf16 [128 keys][16 slots]: 32-byte rows in the 32-byte swizzle, the K-major A
  // operand of the dk_idx MMA
  static constexpr int kDZ = kdST + 128 * 128;
  // dQ staging, one [32 rows][32 d] bf16 block (64-byte rows) per epilogue warp
  static constexpr int kStg = kDZ + 128 * 32;
  static constexpr int kBar = kStg + 8 * 32 * 64;
  static constexpr int kNumBars = 18;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;
};

__device__ __forceinline__ uint32_t sw128(int r, int chunk) {  // within a [rows][64] block
  return (uint32_t)(r * 128 + (((chunk & 7) ^ (r & 7)) << 4));
}
__device__ __forceinline__ uint32_t swz32(int row, int chunk) {  // 32-byte rows
  return (uint32_t)(row * 32 + ((chunk ^ ((row >> 2) & 1)) << 4));
}
__device__ __forceinline__ uint64_t desc_k(uint32_t a) { return umma_desc_kmajor<128>(a); }
__device__ __forceinline__ uint64_t desc_mn(uint32_t a, uint32_t lbo) {
  return (uint64_t)((a & 0x3FFFF) >> 4) | ((uint64_t)(lbo >> 4) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
// K-major operand with 32-byte rows in the 32-byte swizzle: SBO = 8 rows x 32 B.
__device__ __forceinline__ uint64_t desc_sw32(uint32_t a) {
  return (uint64_t)((a & 0x3FFFF) >> 4) | ((uint64_t)(256 >> 4) << 32) | (1ull << 46) | (6ull << 61);
}
__host__ __device__ constexpr uint32_t idesc(int M, int N, int a_mn, int b_mn) {
  return umma_idesc_bf16_f32(M, N) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16);
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// TMEM columns
// z^T (16 columns) lives in the dQ^T columns between E2 of one chunk and (5) of the next.
constexpr uint32_t cDK = 0, cDV = 128, cST = 256, cDPT = 320, cDQT = 384, cDKI = 448, cZ = cDQT;

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_qi, const __grid_constant__ CUtensorMap tm_ki,
                  const BwdTcParams p) {
  constexpr int R = rows_per_chunk(G);  // rows per chunk
  constexpr int RW = R / 2;             // rows per warpgroup
  constexpr int RB = RW < 16 ? RW : 16; // rows per TMEM load step in E1
  using L = BL<D, R>;
  constexpr int QC = R / G;   // real queries per chunk
  constexpr int QH = RW / G;  // queries per warpgroup half
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::kBar);
  uint64_t* kvfull = bar + 0;
  uint64_t* kvempty = bar + 1;  // MMA commit + 8 epilogue warps (k_idx reads)
  uint64_t* qfull = bar + 2;    // [2] chunk gathered (both stage parts)
  uint64_t* bempty = bar + 4;   // [2] big stage free: MMA commit after (3)-(5)
  uint64_t* sempty = bar + 6;   // [3] small stage free: dk_idx MMA commit + 8 epilogue warps
  uint64_t* b_s = bar + 9;      // (1)(2) done
  uint64_t* b_p = bar + 10;     // E1 done (P^T, dS^T in smem)
  uint64_t* b_q = bar + 11;     // (3)(4)(5) done
  uint64_t* b_e = bar + 12;     // E2 has read dQ^T into registers
  uint64_t* b_key = bar + 13;   // block's MMAs done
  uint64_t* b_kfree = bar + 14; // block's accumulators read out
  uint64_t* mmadone = bar + 15;
  uint64_t* b_z = bar + 16;      // z^T = k_idx q_idx^T in the dQ^T columns
  uint64_t* e_wg = bar + 17;     // [2] a warpgroup's four warps have written their dz
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BG = p.B * p.H_kv;

  if (threadIdx.x == 0) {
    mbar_init(kvfull, 1);
    mbar_init(kvempty, 1 + kEpiWarps);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&qfull[s], kLoadArrivals);
      mbar_init(&bempty[s], 1);
    }
    for (int s = 0; s < 3; ++s) mbar_init(&sempty[s], 1 + kEpiWarps);
    mbar_init(b_s, 1);
    mbar_init(b_p, kEpiWarps);
    mbar_init(b_q, 1);
    mbar_init(b_e, kEpiWarps);
    mbar_init(b_key, 1);
    mbar_init(b_kfree, kEpiWarps);
    mbar_init(mmadone, 1);
    mbar_init(b_z, 1);
    mbar_init(&e_wg[0], 4);
    mbar_init(&e_wg[1], 4);
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int x = threadIdx.x; x < 128 * 32 / 16; x += blockDim.x)
    reinterpret_cast<uint4*>(sm + L::kDZ)[x] = make_uint4(0u, 0u, 0u, 0u);
  if (warp == 10) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 8) {
    // ================================== loader ==================================
    // One warp, lane q = query slot q of the chunk.  The rows of a query are its G
    // heads, consecutive in q and dO, so each is one TMA box per 64-column half,
    // written straight into the swizzled K-major operand layout (the 128-byte swizzle
    // follows the shared-memory address, so a box of G rows may start at any row).
    // Padding slots read past the token axis and land as zeros.  The per-row scalars
    // are 4-byte cp.async copies; the stage is published when the TMA bytes, every
    // lane's copies (cp.async arrive) and every lane's plain stores (arrive) are in.
    int u = 0, nkeys = 0, kv_issued = 0;  // nkeys: blocks with at least one chunk
    int next_ent = -1;
    bool ok = true;
    for (int64_t kk = blockIdx.x; kk < p.keys && ok && !*abort_flag; kk += gridDim.x) {
      const int c = (int)(kk / BG), bg = (int)(kk % BG);
      const int b = bg / p.H_kv, g = bg - b * p.H_kv;
      const SeqSpan sp = seq_span(p.spans, b, p.N);
      const int key = bg * p.nb + c;
      const int e_begin = __ldg(&p.off[key]), e_end = __ldg(&p.off[key + 1]);
      const int nch = (e_end - e_begin + QC - 1) / QC;
      for (int ch = 0; ch < nch; ++ch, ++u) {
        const int s = u & 1, s3 = u % 3;
        if (ch == 0) {
          // new block: once the previous block is done with K, V and k_idx, load them
          bool okk = true;
          if (lane == 0) {
            okk = nkeys == 0 || mbar_wait(kvempty, (nkeys - 1) & 1, p.wait_ns, abort_flag);
            if (okk) {
              mbar_arrive_expect_tx(kvfull, 2 * (D / 64) * L::kKH + L::kKH);
#pragma unroll
              for (int h = 0; h < D / 64; ++h) {
                tma_load_4d(sm + L::kK + h * L::kKH, &tm_k, kvfull, h * 64, g, sp.tn + c * 128, sp.tb);
                tma_load_4d(sm + L::kV + h * L::kKH, &tm_v, kvfull, h * 64, g, sp.tn + c * 128, sp.tb);
              }
              tma_load_3d(sm + L::kKi, &tm_ki, kvfull, 0, sp.tn + c * 128, sp.tb);
              kv_issued = nkeys + 1;
            }
          }
          if (!(ok = __shfl_sync(0xffffffffu, okk, 0))) break;
        }
        ok = __all_sync(0xffffffffu, mbar_wait(&bempty[s], ((u >> 1) & 1) ^ 1, p.wait_ns, abort_flag) &&
                                         mbar_wait(&sempty[s3], ((u / 3) & 1) ^ 1, p.wait_ns, abort_flag));
        if (!ok) break;
        uint8_t* st = sm + L::kBig0 + s * L::kBig;       // q, dO
        uint8_t* ss = sm + L::kSmall0 + s3 * L::kSmall;  // q_idx, scalars
        const int q0 = e_begin + ch * QC;
        const int nq = min(QC, e_end - q0);
        // this chunk's entries (prefetched one chunk ahead), lane q = query slot q
        const int my_ent = ch == 0 ? (lane < nq ? __ldg(&p.entries[q0 + lane]) : -1) : next_ent;
        {
          const int q1 = q0 + QC;
          const int nq1 = min(QC, e_end - q1);
          next_ent = (ch + 1 < nch && lane < nq1) ? __ldg(&p.entries[q1 + lane]) : -1;
        }
        if (lane == 0) mbar_expect_tx(&qfull[s], R * D * 2 + kQS * 128);
        __syncwarp();
        const bool okq = my_ent >= 0;
        const int iq = okq ? (my_ent >> kSlotBits) : 0;
        const int zq = okq ? (int)(sp.t0 + iq) : p.T;  // past the token axis: zeros
        if (lane < QC) {
#pragma unroll
          for (int h = 0; h < D / 64; ++h) {
            const uint32_t o = h * L::kQH + lane * G * 128;
            tma_load_3d(st + L::kSQ + o, &tm_q, &qfull[s], h * 64, g * G, zq);
          }
        }
        if (lane < kQS) tma_load_3d(ss + L::kSQi + lane * 128, &tm_qi, &qfull[s], 0, g, zq);
#pragma unroll
        for (int k = 0; k < 2; ++k) {  // rows lane, lane + 32 of the 64-row scalar arrays
          const int r = lane + 32 * k, qi = (r / G) & 31, h = r % G;
          const int ent0 = __shfl_sync(0xffffffffu, my_ent, qi);
          const int ent = r < R ? ent0 : -1;  // rows past the chunk: padding
          const bool okr = ent >= 0;
          const int ri = okr ? (ent >> kSlotBits) : -1;
          const int64_t x = sp.t0 * p.H_kv * G + (int64_t)(g * G + h) * sp.len + (okr ? ri : 0);
          cp_async_4(ss + L::kSLse + 4 * r, p.lse + x, okr);
          cp_async_4(ss + L::kSD + 4 * r, p.Dv + x, okr);
          reinterpret_cast<int*>(ss + L::kSRi)[r] = ri;
          reinterpret_cast<int*>(ss + L::kSRp)[r] =
              okr ? (int)(((sp.t0 * p.H_kv + (int64_t)g * sp.len + ri) * p.topk + (ent & kSlotMask)) * G + h)
                  : -1;
        }
        if (lane < kQS) {
          reinterpret_cast<int*>(ss + L::kSQiq)[lane] = okq ? iq : -1;
          reinterpret_cast<int*>(ss + L::kSQp)[lane] =
              okq ? (int)((sp.t0 * p.H_kv + (int64_t)g * sp.len + iq) * p.topk + (my_ent & kSlotMask)) : -1;
          cp_async_4(ss + L::kSLi + 4 * lane, p.lse_idx + sp.t0 * p.H_kv + (int64_t)g * sp.len + iq, okq);
        }
        mbar_arrive(&qfull[s]);           // this lane's plain stores
        cp_async_mbar_arrive(&qfull[s]);  // this lane's cp.async copies, once landed
      }
      if (nch > 0) ++nkeys;
    }
    if (!ok) *abort_flag = 1;
    // nothing may still be landing in shared memory when the CTA exits
    cp_async_wait<0>();
    if (lane == 0) {
      for (int v = max(0, u - 2); v < u; ++v) mbar_wait(&qfull[v & 1], (v >> 1) & 1, 1000000000ull);
      if (kv_issued > 0) mbar_wait(kvfull, (kv_issued - 1) & 1, 1000000000ull);
    }
    __syncwarp();
  } else if (warp == 9) {
    // ================================ dO gather =================================
    // The chunk's dO rows (G heads of each gathered query) by cp.async into the same
    // swizzled layout, in parallel with warp 8's TMA boxes for q: the copy engines
    // and the load/store path share the chunk's bytes.
    int u = 0;
    int next_ent = -1;
    bool ok = true;
    for (int64_t kk = blockIdx.x; kk < p.keys && ok && !*abort_flag; kk += gridDim.x) {
      const int c = (int)(kk / BG), bg = (int)(kk % BG);
      const int b = bg / p.H_kv, g = bg - b * p.H_kv;
      const SeqSpan sp = seq_span(p.spans, b, p.N);
      const int key = bg * p.nb + c;
      const int e_begin = __ldg(&p.off[key]), e_end = __ldg(&p.off[key + 1]);
      const int nch = (e_end - e_begin + QC - 1) / QC;
      for (int ch = 0; ch < nch; ++ch, ++u) {
        const int s = u & 1;
        if (!(ok = __all_sync(0xffffffffu,
                              mbar_wait(&bempty[s], ((u >> 1) & 1) ^ 1, p.wait_ns, abort_flag))))
          break;
        const int q0 = e_begin + ch * QC;
        const int nq = min(QC, e_end - q0);
        const int my_ent = ch == 0 ? (lane < nq ? __ldg(&p.entries[q0 + lane]) : -1) : next_ent;
        {
          const int q1 = q0 + QC;
          const int nq1 = min(QC, e_end - q1);
          next_ent = (ch + 1 < nch && lane < nq1) ? __ldg(&p.entries[q1 + lane]) : -1;
        }
        uint8_t* st = sm + L::kBig0 + s * L::kBig + L::kSdO;
        static_assert((R * (D / 8)) % 32 == 0, "whole passes of the warp");
#pragma unroll 4
        for (int x = lane; x < R * (D / 8); x += 32) {
          const int r = x / (D / 8), cc = x % (D / 8);
          const int qi = r / G, h = r % G;
          const int ent = __shfl_sync(0xffffffffu, my_ent, qi);
          const bool okr = ent >= 0;
          const int i = okr ? (ent >> kSlotBits) : 0;
          const int64_t src = ((sp.t0 + i) * p.H_kv * G + g * G + h) * D + cc * 8;
          cp_async_16(st + (cc >> 3) * L::kQH + sw128(r, cc), p.dO + src, okr);
        }
        cp_async_mbar_arrive(&qfull[s]);
      }
    }
    if (!ok) *abort_flag = 1;
    cp_async_wait<0>();
  } else if (warp == 10) {
    // ================================ MMA issuer =================================
    if (lane == 0) {
      const uint32_t aK = smem_u32(sm + L::kK), aV = smem_u32(sm + L::kV);
      const uint32_t aPT = smem_u32(sm + L::kPT), adST = smem_u32(sm + L::kdST);
      constexpr uint32_t i12 = idesc(128, R, 0, 0), i34 = idesc(128, D, 0, 1);
      constexpr uint32_t i5 = idesc(128, R, 1, 1);
      constexpr uint32_t iki = idesc(128, 64, 0, 1);  // dk_idx += dz^T q_idx (K = 16 slots)
      constexpr uint32_t iz = idesc(128, 16, 0, 0);   // z^T = k_idx q_idx^T (K = d_idx)
      const uint32_t aDZ = smem_u32(sm + L::kDZ), aKi = smem_u32(sm + L::kKi);
      int u = 0, nkeys = 0;
      bool ok = true, issued = false;
      for (int64_t kk = blockIdx.x; kk < p.keys && ok; kk += gridDim.x) {
        const int c = (int)(kk / BG), bg = (int)(kk % BG);
        const int key = bg * p.nb + c;
        const int e_begin = __ldg(&p.off[key]), e_end = __ldg(&p.off[key + 1]);
        const int nch = (e_end - e_begin + QC - 1) / QC;
        if (nch == 0) continue;
        for (int ch = 0; ch < nch && ok; ++ch, ++u) {
          const int s = u & 1;
          const uint32_t st = smem_u32(sm + L::kBig0 + s * L::kBig);
          const uint32_t aQ = st + L::kSQ, adO = st + L::kSdO;
          const uint32_t aQi = smem_u32(sm + L::kSmall0 + (u % 3) * L::kSmall + L::kSQi);
          ok = mbar_wait(&qfull[s], (u >> 1) & 1, p.wait_ns, abort_flag);
          if (ok && ch == 0) ok = mbar_wait(kvfull, nkeys & 1, p.wait_ns, abort_flag);
          if (ok && ch == 0 && nkeys > 0)
            ok = mbar_wait(b_kfree, (nkeys - 1) & 1, p.wait_ns, abort_flag);
          if (!ok) break;
          tc_fence_after();
          // (1) S^T = K Q^T, (2) dP^T = V dO^T      (K = d)
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t ko = (k >> 2) * L::kKH + (k & 3) * 32;
            const uint32_t qo = (k >> 2) * L::kQH + (k & 3) * 32;
            tc_mma_bf16(tmem + cST, desc_k(aK + ko), desc_k(aQ + qo), i12, k > 0);
            tc_mma_bf16(tmem + cDPT, desc_k(aV + ko), desc_k(adO + qo), i12, k > 0);
          }
          tc_commit(b_s);
          issued = true;
          // z^T = k_idx q_idx^T (K = d_idx, zero-padded to 64) into the dQ^T columns once
          // E2 of the previous chunk has read them; this commit also covers the previous
          // chunk's dk_idx MMA, so E1 may then overwrite dz
          if (u > 0 && !(ok = mbar_wait(b_e, (u - 1) & 1, p.wait_ns, abort_flag))) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 4; ++k)  // K = d_idx (the columns past it are zeros)
            if (16 * k < p.DI) tc_mma_bf16(tmem + cZ, desc_k(aKi + k * 32), desc_k(aQi + k * 32), iz, k > 0);
          tc_commit(b_z);
          if (!(ok = mbar_wait(b_p, u & 1, p.wait_ns, abort_flag))) break;
          tc_fence_after();
          // (3) dV += P^T dO, (4) dK += dS^T Q     (K = R rows)
#pragma unroll
          for (int k = 0; k < R / 16; ++k) {
            const uint32_t acc = (ch > 0 || k > 0) ? 1u : 0u;
            tc_mma_bf16(tmem + cDV, desc_k(aPT + k * 32), desc_mn(adO + k * 2048, L::kQH), i34, acc);
            tc_mma_bf16(tmem + cDK, desc_k(adST + k * 32), desc_mn(aQ + k * 2048, L::kQH), i34, acc);
          }
          // (5) dQ^T = K^T dS^T                     (K = 128 keys)
#pragma unroll
          for (int k = 0; k < 8; ++k)
            tc_mma_bf16(tmem + cDQT, desc_mn(aK + k * 2048, L::kKH), desc_mn(adST + k * 2048, L::kKH),
                        i5, k > 0);
          // (6) dk_idx += dz^T q_idx                 (K = 16 query slots)
          tc_mma_bf16(tmem + cDKI, desc_sw32(aDZ), desc_mn(aQi, L::kQH), iki, ch > 0 ? 1u : 0u);
          tc_commit(b_q);
          tc_commit(&bempty[s]);
          tc_commit(&sempty[u % 3]);
          if (ch == nch - 1) {
            tc_commit(kvempty);
            tc_commit(b_key);
          }
        }
        if (ok) ++nkeys;
      }
      if (!ok) *abort_flag = 1;
      if (issued) {
        tc_commit(mmadone);
        mbar_wait(mmadone, 0, 1000000000ull);
      }
    }
  } else if (warp < 8) {
    // ============================= epilogue warps 0-7 =============================
    const int wg = warp >> 2;              // which 32 of the 64 row columns
    const int tl = (warp & 3) * 32 + lane; // TMEM lane: key (E1, block end), d (E2)
    const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;
    const int q4 = warp & 3;               // this warp's 32 keys (E1, KL) / 32 d (E2)
    const uint8_t* sKi = sm + L::kKi;
    uint8_t* sDZ = sm + L::kDZ;
    double kl = 0.0;
    int u = 0, nkeys = 0;
    bool ok = true;
    for (int64_t kk = blockIdx.x; kk < p.keys && ok; kk += gridDim.x) {
      const int c = (int)(kk / BG), bg = (int)(kk % BG);
      const int b = bg / p.H_kv, g = bg - b * p.H_kv;
      const SeqSpan sp = seq_span(p.spans, b, p.N);
      const int key = bg * p.nb + c;
      const int e_begin = __ldg(&p.off[key]), e_end = __ldg(&p.off[key + 1]);
      const int nch = (e_end - e_begin + QC - 1) / QC;
      const int j = c * 128 + tl;  // key of this thread's TMEM lane
      for (int ch = 0; ch < nch; ++ch, ++u) {
        const int s = u & 1;
        const uint8_t* ss = sm + L::kSmall0 + (u % 3) * L::kSmall;
        const float* s_lse = reinterpret_cast<const float*>(ss + L::kSLse);
        const float* s_D = reinterpret_cast<const float*>(ss + L::kSD);
        const int* s_ri = reinterpret_cast<const int*>(ss + L::kSRi);
        const int* s_rp = reinterpret_cast<const int*>(ss + L::kSRp);
        const int* s_qi = reinterpret_cast<const int*>(ss + L::kSQiq);
        const int* s_qp = reinterpret_cast<const int*>(ss + L::kSQp);
        const float* s_li = reinterpret_cast<const float*>(ss + L::kSLi);
        const uint8_t* sQi = ss + L::kSQi;
        ok = __all_sync(0xffffffffu, mbar_wait(&qfull[s], (u >> 1) & 1, p.wait_ns, abort_flag) &&
                                         (ch > 0 || mbar_wait(kvfull, nkeys & 1, p.wait_ns, abort_flag)) &&
                                         mbar_wait(b_s, u & 1, p.wait_ns, abort_flag) &&
                                         mbar_wait(b_z, u & 1, p.wait_ns, abort_flag));
        if (!ok) break;
        tc_fence_after();
        // ---- E1: this warpgroup's 32 rows of key tl: P^T, dS^T, teacher ----
        {
          float pt[QH];
#pragma unroll
          for (int q = 0; q < QH; ++q) pt[q] = 0.f;
#pragma unroll
          for (int hh = 0; hh < RW / RB; ++hh) {  // RB rows at a time
            uint32_t a[RB], d2[RB];
            if constexpr (RB == 32) {
              tmem_ld_32x32b_x32(tmem + lb + cST + RW * wg + RB * hh, a);
              tmem_ld_32x32b_x32(tmem + lb + cDPT + RW * wg + RB * hh, d2);
            } else if constexpr (RB == 16) {
              tmem_ld_32x32b_x16(tmem + lb + cST + RW * wg + RB * hh, a);
              tmem_ld_32x32b_x16(tmem + lb + cDPT + RW * wg + RB * hh, d2);
            } else {
              tmem_ld_32x32b_x8(tmem + lb + cST + RW * wg + RB * hh, a);
              tmem_ld_32x32b_x8(tmem + lb + cDPT + RW * wg + RB * hh, d2);
            }
            tmem_wait_ld();
            uint32_t pk[RB / 2], dk2[RB / 2];  // bf16 pairs
#pragma unroll
            for (int x4 = 0; x4 < RB; x4 += 4) {
              const int r0 = RW * wg + RB * hh + x4;
              const int4 ri4 = *reinterpret_cast<const int4*>(s_ri + r0);
              const float4 ls4 = *reinterpret_cast<const float4*>(s_lse + r0);
              const float4 dd4 = *reinterpret_cast<const float4*>(s_D + r0);
              const int ri[4] = {ri4.x, ri4.y, ri4.z, ri4.w};  // -1 for padding rows
              const float ls[4] = {ls4.x * kLog2e, ls4.y * kLog2e, ls4.z * kLog2e, ls4.w * kLog2e};
              const float dd[4] = {dd4.x, dd4.y, dd4.z, dd4.w};
              float pv[4], dv2[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int x = x4 + e;
                const float v =
                    j <= ri[e] ? ex2_fast(__uint_as_float(a[x]) * p.scale_log2 - ls[e]) : 0.f;
                pv[e] = v;
                dv2[e] = v * (__uint_as_float(d2[x]) - dd[e]);
                pt[(RB * hh + x) / G] += v;
              }
              pk[x4 / 2] = pack_bf16(pv[0], pv[1]);
              pk[x4 / 2 + 1] = pack_bf16(pv[2], pv[3]);
              dk2[x4 / 2] = pack_bf16(dv2[0], dv2[1]);
              dk2[x4 / 2 + 1] = pack_bf16(dv2[2], dv2[3]);
            }
#pragma unroll
            for (int cc = 0; cc < RB / 8; ++cc) {
              const uint32_t o = sw128(tl, (RW * wg + RB * hh) / 8 + cc);
              *reinterpret_cast<uint4*>(sm + L::kPT + o) =
                  make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
              *reinterpret_cast<uint4*>(sm + L::kdST + o) =
                  make_uint4(dk2[4 * cc], dk2[4 * cc + 1], dk2[4 * cc + 2], dk2[4 * cc + 3]);
            }
          }
          // ---- KL for key tl and this warpgroup's QH query slots (teacher in registers) ----
          uint32_t zr[QH];
          if constexpr (QH == 8) {
            tmem_ld_32x32b_x8(tmem + lb + cZ + QH * wg, zr);
          } else if constexpr (QH == 4) {
            tmem_ld_32x32b_x4(tmem + lb + cZ + QH * wg, zr);
          } else {
            tmem_ld_32x32b_x2(tmem + lb + cZ + QH * wg, zr);
          }
          tmem_wait_ld();
          float klc = 0.f;
          uint32_t dzp[QH / 2];
#pragma unroll
          for (int q2 = 0; q2 < QH; q2 += 2) {
            float dz[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int q = q2 + e, sl = QH * wg + q;
              const bool valid = j <= s_qi[sl];  // s_qi = -1 for padding slots
              const float zl2 = __uint_as_float(zr[q]) * p.sidx_log2 - s_li[sl] * kLog2e;  // log2 p_I
              const float pI = valid ? ex2_fast(zl2) : 0.f;
              const float pT = pt[q] * (1.f / G);  // group-averaged main probability
              if (valid && pT > 0.f) klc += pT * (__log2f(pT) - zl2);
              dz[e] = valid ? p.w * (pI - pT) : 0.f;
            }
            dzp[q2 / 2] = pack_bf16(dz[0], dz[1]);
          }
          kl += (double)(klc * kLn2);
          if constexpr (QH == 8) {  // slots 8 wg .. 8 wg + 7: one 16-byte chunk of the dz row
            *reinterpret_cast<uint4*>(sDZ + swz32(tl, wg)) = make_uint4(dzp[0], dzp[1], dzp[2], dzp[3]);
          } else if constexpr (QH == 4) {  // slots 4 wg .. 4 wg + 3: half of chunk 0
            *reinterpret_cast<uint2*>(sDZ + swz32(tl, 0) + 8 * wg) = make_uint2(dzp[0], dzp[1]);
          } else {                         // slots 2 wg, 2 wg + 1: a quarter of chunk 0
            *reinterpret_cast<uint32_t*>(sDZ + swz32(tl, 0) + 4 * wg) = dzp[0];
          }
        }
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_p);
        // dz of this warpgroup's slots complete for every key (dq_idx below reads all keys)
        __syncwarp();
        if (lane == 0) mbar_arrive(&e_wg[wg]);
        ok = __all_sync(0xffffffffu, mbar_wait(&e_wg[wg], u & 1, p.wait_ns, abort_flag));
        if (!ok) break;
        // this warpgroup's slots are n8 tile nt of dz (8 slots each, G <= 4); with G = 8
        // or 16 both warpgroups share tile 0 and each keeps its own QH slots
        constexpr int NT = (QH == 8) ? 1 : 0;
        const int nt = NT ? wg : 0;
        if (16 * q4 < p.DI) {
          // dq_idx^T (16 d x 8 slots of this warpgroup) = k_idx^T dz^T   (k = 128 keys)
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int ks2 = 0; ks2 < 4; ++ks2) {  // two 16-key steps per x4 dz load
            uint32_t bz[4];
            ldmatrix_x4_trans(bz, sDZ + swz32(32 * ks2 + (lane & 7) + (((lane >> 3) & 1) << 3) +
                                                  ((lane >> 4) << 4), nt));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t a[4];
              ldmatrix_x4_trans(a, sKi + sw128(32 * ks2 + 16 * h + (lane & 7) + ((lane >> 4) << 3),
                                               2 * q4 + ((lane >> 3) & 1)));
              mma_bf16_16816(acc, a, bz[2 * h], bz[2 * h + 1]);
            }
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int qs = 8 * nt + (lane & 3) * 2 + (e & 1);
            const int dd = 16 * q4 + (lane >> 2) + ((e >> 1) << 3);
            const int qp = s_qp[qs];
            if ((NT || qs / QH == wg) && qp >= 0)
              p.dqi_part[(int64_t)qp * p.DI + dd] = __float2bfloat16(acc[e] * p.sidx);
          }
        }
        // ---- E2: dQ^T columns of this warpgroup's rows (thread = d) ----
        ok = __all_sync(0xffffffffu, mbar_wait(b_q, u & 1, p.wait_ns, abort_flag));
        if (!ok) break;
        tc_fence_after();
        if (tl < D) {  // warp-uniform
          uint32_t a[RW];
          if constexpr (RW == 32) {
            tmem_ld_32x32b_x32(tmem + lb + cDQT + RW * wg, a);
          } else if constexpr (RW == 16) {
            tmem_ld_32x32b_x16(tmem + lb + cDQT + RW * wg, a);
          } else {
            tmem_ld_32x32b_x8(tmem + lb + cDQT + RW * wg, a);
          }
          tmem_wait_ld();
          // dQ^T is in registers: the z^T MMA of the next chunk may take its columns
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(b_e);
          // stage this warp's [RW rows][32 d] block so the global stores below write
          // 64-byte row segments; lanes (2m, 2m+1) swap one value so each stores a pair
          uint8_t* stg = sm + L::kStg + warp * (32 * 64);
          const bool odd = lane & 1;
#pragma unroll
          for (int x = 0; x < RW; x += 2) {
            const float v0 = __uint_as_float(a[x]) * p.scale;
            const float v1 = __uint_as_float(a[x + 1]) * p.scale;
            const float mine = odd ? v1 : v0;
            const float give = odd ? v0 : v1;
            const float got = __shfl_xor_sync(0xffffffffu, give, 1);
            *reinterpret_cast<uint32_t*>(stg + (x + (odd ? 1 : 0)) * 64 + (lane & ~1) * 2) =
                odd ? pack_bf16(got, mine) : pack_bf16(mine, got);
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < RW / 8; ++i) {
            const int k = lane + 32 * i;
            const int r = k >> 2, cc = k & 3;
            const int rp = s_rp[RW * wg + r];
            const uint4 v = *reinterpret_cast<const uint4*>(stg + r * 64 + cc * 16);
            if (rp >= 0) *reinterpret_cast<uint4*>(p.dq_part + (int64_t)rp * D + 32 * q4 + cc * 8) = v;
          }
          __syncwarp();
        } else {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(b_e);
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sempty[u % 3]);
          if (ch == nch - 1) mbar_arrive(kvempty);
        }
      }
      if (!ok) break;
      // ---- block end: dK (x scale), dV and the dk_idx share from TMEM ----
      const bool in = j < sp.len;
      __nv_bfloat16* dk_row = p.dk + ((sp.t0 + j) * p.H_kv + g) * D;
      __nv_bfloat16* dv_row = p.dv + ((sp.t0 + j) * p.H_kv + g) * D;
      if (nch == 0) {
        if (in) {
          for (int x = wg * (D / 2); x < (wg + 1) * (D / 2); ++x) {
            dk_row[x] = __float2bfloat16(0.f);
            dv_row[x] = __float2bfloat16(0.f);
          }
          if (32 * wg < p.DI) {
            float4* dst = reinterpret_cast<float4*>(
                p.dki_part + ((sp.t0 + j) * p.H_kv + g) * p.DI + 32 * wg);
#pragma unroll
            for (int x = 0; x < 8; ++x) dst[x] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
      } else {
        ok = __all_sync(0xffffffffu, mbar_wait(b_key, nkeys & 1, p.wait_ns, abort_flag));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          const int col = wg * (D / 2) + 32 * h;
          uint32_t a[32], d2[32];
          tmem_ld_32x32b_x32(tmem + lb + cDK + col, a);
          tmem_ld_32x32b_x32(tmem + lb + cDV + col, d2);
          tmem_wait_ld();
          if (in) {
#pragma unroll
            for (int x = 0; x < 32; x += 8) {
              uint4 wk, wv;
              wk.x = pack_bf16(__uint_as_float(a[x]) * p.scale, __uint_as_float(a[x + 1]) * p.scale);
              wk.y = pack_bf16(__uint_as_float(a[x + 2]) * p.scale, __uint_as_float(a[x + 3]) * p.scale);
              wk.z = pack_bf16(__uint_as_float(a[x + 4]) * p.scale, __uint_as_float(a[x + 5]) * p.scale);
              wk.w = pack_bf16(__uint_as_float(a[x + 6]) * p.scale, __uint_as_float(a[x + 7]) * p.scale);
              wv.x = pack_bf16(__uint_as_float(d2[x]), __uint_as_float(d2[x + 1]));
              wv.y = pack_bf16(__uint_as_float(d2[x + 2]), __uint_as_float(d2[x + 3]));
              wv.z = pack_bf16(__uint_as_float(d2[x + 4]), __uint_as_float(d2[x + 5]));
              wv.w = pack_bf16(__uint_as_float(d2[x + 6]), __uint_as_float(d2[x + 7]));
              *reinterpret_cast<uint4*>(dk_row + col + x) = wk;
              *reinterpret_cast<uint4*>(dv_row + col + x) = wv;
            }
          }
        }
        // dk_idx share of group g: warpgroup wg holds d_idx columns 32 wg .. 32 wg + 31
        if (32 * wg < p.DI) {
          uint32_t a[32];
          tmem_ld_32x32b_x32(tmem + lb + cDKI + 32 * wg, a);
          tmem_wait_ld();
          if (in) {
            float4* dst = reinterpret_cast<float4*>(
                p.dki_part + ((sp.t0 + j) * p.H_kv + g) * p.DI + 32 * wg);
#pragma unroll
            for (int x = 0; x < 8; ++x)
              dst[x] = make_float4(__uint_as_float(a[4 * x]) * p.sidx, __uint_as_float(a[4 * x + 1]) * p.sidx,
                                   __uint_as_float(a[4 * x + 2]) * p.sidx, __uint_as_float(a[4 * x + 3]) * p.sidx);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_kfree);
        ++nkeys;
      }
    }
    if (!ok) *abort_flag = 1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) kl += __shfl_xor_sync(0xffffffffu, kl, o);
    if (lane == 0 && kl != 0.0) atomicAdd(p.kl_acc, kl * (double)p.w);
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) set_status(p.status, MSA_ERR_DEVICE_TIMEOUT);
  if (warp == 10) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

struct BwdMaps {
  CUtensorMap k, v, q, qi, ki;
};

template <int D, int G>
cudaError_t launch_dg(const BwdTcParams& prm, const BwdMaps& m, const Ctx& cx, cudaStream_t st) {
  using L = BL<D, rows_per_chunk(G)>;
  auto kern = bwd_tc_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  kernel_event(MSA_KERNEL_BWD, true, st);
  kern<<<cx.num_sms, kThreads, L::kAlloc, st>>>(m.k, m.v, m.q, m.qi, m.ki, prm);
  kernel_event(MSA_KERNEL_BWD, false, st);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd_tc(const Shape& s, const void* q, const void* k, const void* v,
                               const void* dO, const float* lse, const float* Dv,
                               const void* q_idx, const void* k_idx, const float* lse_idx,
                               float kl_weight, const Plan& pl, __nv_bfloat16* dq_part,
                               __nv_bfloat16* dqi_part, float* dki_part, double* kl_acc, void* dk,
                               void* dv, const Ctx& cx, cudaStream_t st) {
  // K, V: [tokens][H_kv][d] per batch, one (64-column, 128-key) box per half.
  // q: [T][H_q][d], one (64-column, G-head) box per query and half (dO is gathered by
  // cp.async).
  // q_idx: [T][H_kv][d_idx], one row box per query slot; k_idx: [tokens][d_idx] per
  // batch, one 128-key box.  All 128-byte swizzled; the q_idx and k_idx boxes are 64
  // columns wide whatever d_idx is, so with d_idx = 32 the upper half lands as zeros.
  if (s.T >= 0x7fffffff) return cudaErrorInvalidValue;  // token coordinates are int32
  BwdMaps m;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
  const uint64_t H_q = (uint64_t)s.H_kv * s.G, T = (uint64_t)s.T, DI = (uint64_t)s.d_idx;
  const uint64_t dkv[4] = {(uint64_t)s.d, (uint64_t)s.H_kv, s.tma_tokens(), s.tma_batches()};
  const uint64_t skv[3] = {(uint64_t)s.d * 2, (uint64_t)s.H_kv * s.d * 2,
                           s.tma_tokens() * s.H_kv * s.d * 2};
  const uint32_t bkv[4] = {64, 1, 128, 1};
  const uint64_t dq[3] = {(uint64_t)s.d, H_q, T};
  const uint64_t sq[2] = {(uint64_t)s.d * 2, H_q * s.d * 2};
  const uint32_t bq[3] = {64, (uint32_t)s.G, 1};
  const uint64_t dqi[3] = {DI, (uint64_t)s.H_kv, T};
  const uint64_t sqi[2] = {DI * 2, (uint64_t)s.H_kv * DI * 2};
  const uint32_t bqi[3] = {64, 1, 1};
  const uint64_t dki[3] = {DI, s.tma_tokens(), s.tma_batches()};
  const uint64_t ski[2] = {DI * 2, s.tma_tokens() * DI * 2};
  const uint32_t bki[3] = {64, 128, 1};
  if (!encode_tiled(&m.k, bf, 4, k, dkv, skv, bkv, sw) || !encode_tiled(&m.v, bf, 4, v, dkv, skv, bkv, sw) ||
      !encode_tiled(&m.q, bf, 3, q, dq, sq, bq, sw) ||
      !encode_tiled(&m.qi, bf, 3, q_idx, dqi, sqi, bqi, sw) ||
      !encode_tiled(&m.ki, bf, 3, k_idx, dki, ski, bki, sw))
    return cudaErrorInvalidValue;
  BwdTcParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.dO = static_cast<const __nv_bfloat16*>(dO);
  p.q_idx = static_cast<const __nv_bfloat16*>(q_idx);
  p.k_idx = static_cast<const __nv_bfloat16*>(k_idx);
  p.spans = s.spans;
  p.lse = lse;
  p.Dv = Dv;
  p.lse_idx = lse_idx;
  p.off = pl.off;
  p.entries = pl.entries;
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.dq_part = dq_part;
  p.dqi_part = dqi_part;
  p.dki_part = dki_part;
  p.kl_acc = kl_acc;
  p.keys = s.keys();
  p.B = s.B;
  p.N = s.N;
  p.T = (int)s.T;
  p.H_kv = s.H_kv;
  p.nb = s.nb;
  p.topk = s.topk;
  p.DI = s.d_idx;
  p.scale = s.scale;
  p.scale_log2 = s.scale * kLog2e;
  p.sidx = s.scale_idx;
  p.sidx_log2 = s.scale_idx * kLog2e;
  p.w = kl_weight;
  p.wait_ns = cx.wait_ns;
  p.status = cx.status;
#define MSA_BWD_G(DD)                                                  \
  switch (s.G) {                                                       \
    case 1: return launch_dg<DD, 1>(p, m, cx, st);                \
    case 2: return launch_dg<DD, 2>(p, m, cx, st);                \
    case 4: return launch_dg<DD, 4>(p, m, cx, st);                \
    case 8: return launch_dg<DD, 8>(p, m, cx, st);                \
    default: return launch_dg<DD, 16>(p, m, cx, st);              \
  }
  if (s.d == 128) MSA_BWD_G(128)
  MSA_BWD_G(64)
#undef MSA_BWD_G
}

}  // namespace msa
