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
// chunks of 64 rows (64/G gathered queries x G heads; 16 query slots).
//   tcgen05 (one MMA thread, accumulators in TMEM, every M = 128):
//     (1) S^T  = K Q^T     M=128 keys, N=64 rows, K=d
//     (2) dP^T = V dO^T    M=128 keys, N=64 rows, K=d
//     (3) dV  += P^T dO    M=128 keys, N=d,  K=64 rows   (dO as MN-major B)
//     (4) dK  += dS^T Q    M=128 keys, N=d,  K=64 rows   (Q as MN-major B)
//     (5) dQ^T = K^T dS^T  M=d, N=64 rows, K=128 keys    (both MN-major)
//   epilogue warps 0-7 (two warpgroups, each owning 32 of the 64 row columns):
//     E1  P^T = exp(scale S^T - lse), dS^T = P^T (dP^T - D) -> smem; p_T (teacher)
//     KL  (mma.sync, while (3)-(5) run) z = k_idx q_idx^T, p_I, dz = w (p_I - p_T),
//         dk_idx += dz^T q_idx (registers), dq_idx = dz k_idx -> per-slot partials
//     E2  dQ^T columns -> bf16 per-slot partials
// Chunk u+1's (1)(2) overlap chunk u's E2.  After the block's last chunk dK, dV
// (TMEM) and dk_idx (registers) are written once: no atomics on dk/dv/dk_idx.
// Warps 8-9: loaders (cp.async gathers of q, dO, q_idx rows and k_idx; TMA for K, V).
// Warp 10: TMEM owner and MMA issuer.
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace msa {
namespace {

constexpr int kThreads = 352;  // 11 warps
constexpr int kEpiWarps = 8;
constexpr int kLoadThreads = 64;
constexpr int kRows = 64;  // rows per chunk
constexpr int kQS = 16;    // query slots per chunk
constexpr int kTS = 17;    // teacher row stride (floats): conflict-free column access
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct BwdTcParams {
  const __nv_bfloat16 *q, *dO, *q_idx, *k_idx;
  const float *lse, *Dv, *lse_idx;
  const int* off;
  const int* entries;
  __nv_bfloat16 *dk, *dv, *dq_part, *dqi_part;
  float* dki_part;
  double* kl_acc;
  int64_t keys;
  int B, N, H_kv, nb, topk, DI;
  float scale, scale_log2, sidx, sidx_log2, w;
  uint64_t wait_ns;
  int* status;
};

template <int D>
struct BL {
  static constexpr int kKH = 128 * 128;             // [128][64] bf16 block
  static constexpr int kK = 0;
  static constexpr int kV = kK + (D / 64) * kKH;
  static constexpr int kKi = kV + (D / 64) * kKH;   // k_idx [128][64], zero-padded
  static constexpr int kQH = 64 * 128;              // [64][64] bf16 block
  static constexpr int kSQ = 0;
  static constexpr int kSdO = kSQ + (D / 64) * kQH;
  static constexpr int kSQi = kSdO + (D / 64) * kQH;  // [16][64]
  static constexpr int kSLse = kSQi + 16 * 128;       // float[64] lse (natural log)
  static constexpr int kSD = kSLse + 64 * 4;          // float[64] D
  static constexpr int kSRi = kSD + 64 * 4;           // int[64] query index of the row, -1 pad
  static constexpr int kSRp = kSRi + 64 * 4;          // int[64] dq partial row, -1 pad
  static constexpr int kSQiq = kSRp + 64 * 4;         // int[16] query index of the slot, -1 pad
  static constexpr int kSQp = kSQiq + 16 * 4;         // int[16] dq_idx partial row, -1 pad
  static constexpr int kSLi = kSQp + 16 * 4;          // float[16] lse_idx (natural log)
  static constexpr int kStage = ((kSLi + 16 * 4) + 1023) & ~1023;
  static constexpr int kStages0 = kKi + kKH;
  static constexpr int kPT = kStages0 + 2 * kStage;   // P^T [128][64] bf16 (SW128)
  static constexpr int kdST = kPT + 128 * 128;        // dS^T [128][64]
  static constexpr int kTeach = kdST + 128 * 128;     // p_T float [128][17] (padded rows)
  static constexpr int kDZ = kTeach + 128 * 17 * 4;   // dz bf16 [128][16] (32-byte rows)
  static constexpr int kStg = kDZ + 128 * 32;        // dQ staging [2][32 rows][272 B]
  static constexpr int kStgRow = 2 * D + 16;
  static constexpr int kBar = kStg + 2 * 32 * kStgRow;
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
__host__ __device__ constexpr uint32_t idesc(int M, int N, int a_mn, int b_mn) {
  return umma_idesc_bf16_f32(M, N) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16);
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// TMEM columns
constexpr uint32_t cDK = 0, cDV = 128, cST = 256, cDPT = 320, cDQT = 384;

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const BwdTcParams p) {
  using L = BL<D>;
  constexpr int QC = kRows / G;  // real queries per chunk
  constexpr int QH = 32 / G;     // queries per warpgroup half (32 rows)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::kBar);
  uint64_t* kvfull = bar + 0;
  uint64_t* kvempty = bar + 1;  // MMA commit + 8 epilogue warps (k_idx reads)
  uint64_t* qfull = bar + 2;    // [2]
  uint64_t* qempty = bar + 4;   // [2] MMA commit + 8 epilogue warps
  uint64_t* b_s = bar + 6;      // (1)(2) done
  uint64_t* b_p = bar + 7;      // E1 done (P^T, dS^T in smem)
  uint64_t* b_q = bar + 8;      // (3)(4)(5) done
  uint64_t* b_e = bar + 9;      // E2 done (dQ^T columns read)
  uint64_t* b_key = bar + 10;   // block's MMAs done
  uint64_t* b_kfree = bar + 11; // block's accumulators read out
  uint64_t* mmadone = bar + 12;
  uint64_t* e_sync1 = bar + 13;  // every epilogue warp has written its teacher rows
  uint64_t* e_sync2 = bar + 14;  // every epilogue warp has written its dz rows
  uint64_t* e_stg = bar + 15;    // [2] a warpgroup's dQ rows are staged (bars 15, 16)
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BG = p.B * p.H_kv;

  if (threadIdx.x == 0) {
    mbar_init(kvfull, 1);
    mbar_init(kvempty, 1 + kEpiWarps);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&qfull[s], kLoadThreads);
      mbar_init(&qempty[s], 1 + kEpiWarps);
    }
    mbar_init(b_s, 1);
    mbar_init(b_p, kEpiWarps);
    mbar_init(b_q, 1);
    mbar_init(b_e, kEpiWarps);
    mbar_init(b_key, 1);
    mbar_init(b_kfree, kEpiWarps);
    mbar_init(mmadone, 1);
    mbar_init(e_sync1, kEpiWarps);
    mbar_init(e_sync2, kEpiWarps);
    mbar_init(&e_stg[0], 4);
    mbar_init(&e_stg[1], 4);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 10) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 8 || warp == 9) {
    // ================================= loaders ==================================
    const int lt = threadIdx.x - 256;  // 0..63
    int u = 0, nkeys = 0, kv_issued = 0;  // nkeys: blocks with at least one chunk
    int next_ent = -1;
    for (int64_t kk = blockIdx.x; kk < p.keys && !*abort_flag; kk += gridDim.x) {
      const int c = (int)(kk / BG), bg = (int)(kk % BG);
      const int b = bg / p.H_kv, g = bg - b * p.H_kv;
      const int key = bg * p.nb + c;
      const int e_begin = __ldg(&p.off[key]), e_end = __ldg(&p.off[key + 1]);
      const int nch = (e_end - e_begin + QC - 1) / QC;
      for (int ch = 0; ch < nch && !*abort_flag; ++ch, ++u) {
        const int s = u & 1;
        // publish the previous chunk first: it is needed as soon as the chunk before
        // it finishes, which may be before this chunk's stage is free
        if (u >= 1) {
          cp_async_wait<0>();
          fence_async_smem();
          mbar_arrive(&qfull[(u - 1) & 1]);
        }
        if (ch == 0) {
          // new block: wait until the previous block is done with K, V and k_idx
          if (nkeys > 0 && !mbar_wait(kvempty, (nkeys - 1) & 1, p.wait_ns, abort_flag)) {
            *abort_flag = 1;
            break;
          }
          if (lt == 0) {
            mbar_arrive_expect_tx(kvfull, 2 * (D / 64) * L::kKH);
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
              tma_load_4d(sm + L::kK + h * L::kKH, &tm_k, kvfull, h * 64, g, c * 128, b);
              tma_load_4d(sm + L::kV + h * L::kKH, &tm_v, kvfull, h * 64, g, c * 128, b);
            }
            kv_issued = nkeys + 1;
          }
          for (int x = lt; x < 128 * 8; x += kLoadThreads) {  // k_idx rows, zero-padded
            const int r = x / 8, cc = x % 8;
            const int j = c * 128 + r;
            const bool ok = j < p.N && cc * 8 < p.DI;
            const int64_t src = ((int64_t)b * p.N + (ok ? j : 0)) * p.DI + (ok ? cc * 8 : 0);
            cp_async_16(sm + L::kKi + sw128(r, cc), p.k_idx + src, ok);
          }
        }
        if (!mbar_wait(&qempty[s], ((u >> 1) & 1) ^ 1, p.wait_ns, abort_flag)) {
          *abort_flag = 1;
          break;
        }
        uint8_t* st = sm + L::kStages0 + s * L::kStage;
        const int q0 = e_begin + ch * QC;
        const int nq = min(QC, e_end - q0);
        // this chunk's entries (prefetched one chunk ahead), lane q = query slot q
        const int my_ent = ch == 0 ? (lane < nq ? __ldg(&p.entries[q0 + lane]) : -1) : next_ent;
        {
          const int q1 = q0 + QC;
          const int nq1 = min(QC, e_end - q1);
          next_ent = (ch + 1 < nch && lane < nq1) ? __ldg(&p.entries[q1 + lane]) : -1;
        }
        for (int x = lt; x < kRows * (D / 8); x += kLoadThreads) {
          const int r = x / (D / 8), cc = x % (D / 8);
          const int qi = r / G, h = r % G;
          const int ent = __shfl_sync(0xffffffffu, my_ent, qi);
          const bool ok = ent >= 0;
          const int i = ok ? (ent >> 5) : 0;
          const int64_t src = (((int64_t)b * p.N + i) * p.H_kv * G + g * G + h) * D + cc * 8;
          const uint32_t o = (cc >> 3) * L::kQH + sw128(r, cc);
          cp_async_16(st + L::kSQ + o, p.q + src, ok);
          cp_async_16(st + L::kSdO + o, p.dO + src, ok);
        }
        for (int x = lt; x < kQS * 8; x += kLoadThreads) {
          const int qi = x / 8, cc = x % 8;
          const int ent = __shfl_sync(0xffffffffu, my_ent, qi);
          const bool ok = ent >= 0 && cc * 8 < p.DI;
          const int i = ok ? (ent >> 5) : 0;
          const int64_t src = (((int64_t)b * p.N + i) * p.H_kv + g) * p.DI + (ok ? cc * 8 : 0);
          cp_async_16(st + L::kSQi + sw128(qi, cc), p.q_idx + src, ok);
        }
        {
          const int r = lt, qi = r / G, h = r % G;  // one row per loader thread
          const int ent = __shfl_sync(0xffffffffu, my_ent, qi);
          const bool ok = ent >= 0;
          const int ri = ok ? (ent >> 5) : -1;
          const int64_t x = ((int64_t)b * p.H_kv * G + g * G + h) * p.N + (ok ? ri : 0);
          cp_async_4(st + L::kSLse + 4 * r, p.lse + x, ok);
          cp_async_4(st + L::kSD + 4 * r, p.Dv + x, ok);
          reinterpret_cast<int*>(st + L::kSRi)[r] = ri;
          reinterpret_cast<int*>(st + L::kSRp)[r] =
              ok ? (int)((((int64_t)bg * p.N + ri) * p.topk + (ent & 31)) * G + h) : -1;
          if (lt < kQS) {
            const bool okq = my_ent >= 0;
            const int iq = okq ? (my_ent >> 5) : 0;
            reinterpret_cast<int*>(st + L::kSQiq)[lt] = okq ? iq : -1;
            reinterpret_cast<int*>(st + L::kSQp)[lt] =
                okq ? (int)(((int64_t)bg * p.N + iq) * p.topk + (my_ent & 31)) : -1;
            cp_async_4(st + L::kSLi + 4 * lt, p.lse_idx + (int64_t)bg * p.N + iq, okq);
          }
        }
        cp_async_commit();
      }
      if (nch > 0) ++nkeys;
    }
    cp_async_wait<0>();
    fence_async_smem();
    if (u > 0 && !*abort_flag) mbar_arrive(&qfull[(u - 1) & 1]);
    if (lt == 0 && kv_issued > 0) mbar_wait(kvfull, (kv_issued - 1) & 1, 1000000000ull);
  } else if (warp == 10) {
    // ================================ MMA issuer =================================
    if (lane == 0) {
      const uint32_t aK = smem_u32(sm + L::kK), aV = smem_u32(sm + L::kV);
      const uint32_t aPT = smem_u32(sm + L::kPT), adST = smem_u32(sm + L::kdST);
      constexpr uint32_t i12 = idesc(128, 64, 0, 0), i34 = idesc(128, D, 0, 1);
      constexpr uint32_t i5 = idesc(128, 64, 1, 1);
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
          const uint32_t st = smem_u32(sm + L::kStages0 + s * L::kStage);
          const uint32_t aQ = st + L::kSQ, adO = st + L::kSdO;
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
          if (!(ok = mbar_wait(b_p, u & 1, p.wait_ns, abort_flag))) break;
          if (u > 0 && !(ok = mbar_wait(b_e, (u - 1) & 1, p.wait_ns, abort_flag))) break;
          tc_fence_after();
          // (3) dV += P^T dO, (4) dK += dS^T Q     (K = 64 rows)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t acc = (ch > 0 || k > 0) ? 1u : 0u;
            tc_mma_bf16(tmem + cDV, desc_k(aPT + k * 32), desc_mn(adO + k * 2048, L::kQH), i34, acc);
            tc_mma_bf16(tmem + cDK, desc_k(adST + k * 32), desc_mn(aQ + k * 2048, L::kQH), i34, acc);
          }
          // (5) dQ^T = K^T dS^T                     (K = 128 keys)
#pragma unroll
          for (int k = 0; k < 8; ++k)
            tc_mma_bf16(tmem + cDQT, desc_mn(aK + k * 2048, L::kKH), desc_mn(adST + k * 2048, L::kKH),
                        i5, k > 0);
          tc_commit(b_q);
          tc_commit(&qempty[s]);
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
  } else {
    // ============================= epilogue warps 0-7 =============================
    const int wg = warp >> 2;              // which 32 of the 64 row columns
    const int tl = (warp & 3) * 32 + lane; // TMEM lane: key (E1, block end), d (E2)
    const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;
    const int kw = warp * 16;              // mma.sync: this warp's 16 keys
    const uint8_t* sKi = sm + L::kKi;
    float* sTeach = reinterpret_cast<float*>(sm + L::kTeach);
    uint8_t* sDZ = sm + L::kDZ;
    float dki[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) dki[n][0] = dki[n][1] = dki[n][2] = dki[n][3] = 0.f;
    double kl = 0.0;
    int u = 0, nkeys = 0;
    bool ok = true;
    for (int64_t kk = blockIdx.x; kk < p.keys && ok; kk += gridDim.x) {
      const int c = (int)(kk / BG), bg = (int)(kk % BG);
      const int b = bg / p.H_kv, g = bg - b * p.H_kv;
      const int key = bg * p.nb + c;
      const int e_begin = __ldg(&p.off[key]), e_end = __ldg(&p.off[key + 1]);
      const int nch = (e_end - e_begin + QC - 1) / QC;
      const int j = c * 128 + tl;  // key of this thread's TMEM lane
      for (int ch = 0; ch < nch; ++ch, ++u) {
        const int s = u & 1;
        const uint8_t* st = sm + L::kStages0 + s * L::kStage;
        const float* s_lse = reinterpret_cast<const float*>(st + L::kSLse);
        const float* s_D = reinterpret_cast<const float*>(st + L::kSD);
        const int* s_ri = reinterpret_cast<const int*>(st + L::kSRi);
        const int* s_rp = reinterpret_cast<const int*>(st + L::kSRp);
        const int* s_qi = reinterpret_cast<const int*>(st + L::kSQiq);
        const int* s_qp = reinterpret_cast<const int*>(st + L::kSQp);
        const float* s_li = reinterpret_cast<const float*>(st + L::kSLi);
        const uint8_t* sQi = st + L::kSQi;
        ok = __all_sync(0xffffffffu, mbar_wait(&qfull[s], (u >> 1) & 1, p.wait_ns, abort_flag) &&
                                         mbar_wait(b_s, u & 1, p.wait_ns, abort_flag));
        if (!ok) break;
        tc_fence_after();
        // ---- E1: this warpgroup's 32 rows of key tl: P^T, dS^T, teacher ----
        {
          uint32_t a[32], d2[32];
          tmem_ld_32x32b_x32(tmem + lb + cST + 32 * wg, a);
          tmem_ld_32x32b_x32(tmem + lb + cDPT + 32 * wg, d2);
          tmem_wait_ld();
          uint32_t pk[16], dk2[16];  // bf16 pairs
          float pt[QH];
#pragma unroll
          for (int q = 0; q < QH; ++q) pt[q] = 0.f;
#pragma unroll
          for (int x = 0; x < 32; x += 2) {
            float pv[2], dv2[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int r = 32 * wg + x + e;
              const bool valid = j <= s_ri[r];  // s_ri = -1 for padding rows
              const float v =
                  valid ? ex2_fast(__uint_as_float(a[x + e]) * p.scale_log2 - s_lse[r] * kLog2e) : 0.f;
              pv[e] = v;
              dv2[e] = v * (__uint_as_float(d2[x + e]) - s_D[r]);
              pt[(x + e) / G] += v;
            }
            pk[x / 2] = pack_bf16(pv[0], pv[1]);
            dk2[x / 2] = pack_bf16(dv2[0], dv2[1]);
          }
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            *reinterpret_cast<uint4*>(sm + L::kPT + sw128(tl, 4 * wg + cc)) =
                make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
            *reinterpret_cast<uint4*>(sm + L::kdST + sw128(tl, 4 * wg + cc)) =
                make_uint4(dk2[4 * cc], dk2[4 * cc + 1], dk2[4 * cc + 2], dk2[4 * cc + 3]);
          }
#pragma unroll
          for (int q = 0; q < QH; ++q) sTeach[tl * kTS + wg * QH + q] = pt[q] * (1.f / G);
          if (QC < kQS && wg == 1) {  // padded query slots of the teacher
#pragma unroll
            for (int q = QC; q < kQS; ++q) sTeach[tl * kTS + q] = 0.f;
          }
        }
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_p);
        // teacher complete for every key (bounded mbarrier, not bar.sync: a warp
        // that gives up must not leave the others waiting forever)
        __syncwarp();
        if (lane == 0) mbar_arrive(e_sync1);
        ok = __all_sync(0xffffffffu, mbar_wait(e_sync1, u & 1, p.wait_ns, abort_flag));
        if (!ok) break;
        // ---- KL on mma.sync (overlaps the MMAs (3)-(5)) ----
        {
          float zt[2][4];
#pragma unroll
          for (int n = 0; n < 2; ++n) zt[n][0] = zt[n][1] = zt[n][2] = zt[n][3] = 0.f;
#pragma unroll
          for (int kc = 0; kc < 4; ++kc) {  // d_idx (zero-padded to 64)
            uint32_t a[4], bq[4];
            ldmatrix_x4(a, sKi + sw128(kw + (lane & 15), kc * 2 + (lane >> 4)));
            ldmatrix_x4(bq, sQi + sw128((lane & 7) + ((lane >> 4) << 3), kc * 2 + ((lane >> 3) & 1)));
            mma_bf16_16816(zt[0], a, bq[0], bq[1]);
            mma_bf16_16816(zt[1], a, bq[2], bq[3]);
          }
          const int kl0 = kw + (lane >> 2);
          float klc = 0.f;
#pragma unroll
          for (int n = 0; n < 2; ++n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int qs = n * 8 + (lane & 3) * 2 + (e & 1);
              const int kloc = kl0 + ((e >> 1) << 3);
              const bool valid = c * 128 + kloc <= s_qi[qs];  // s_qi = -1 for padding
              const float zl2 = zt[n][e] * p.sidx_log2 - s_li[qs] * kLog2e;  // log2 p_I
              const float pI = valid ? ex2_fast(zl2) : 0.f;
              const float pT = sTeach[kloc * kTS + qs];
              if (valid && pT > 0.f) klc += pT * (__log2f(pT) - zl2);
              zt[n][e] = valid ? p.w * (pI - pT) : 0.f;  // dz
            }
            *reinterpret_cast<uint32_t*>(sDZ + swz32(kl0, n) + (lane & 3) * 4) =
                pack_bf16(zt[n][0], zt[n][1]);
            *reinterpret_cast<uint32_t*>(sDZ + swz32(kl0 + 8, n) + (lane & 3) * 4) =
                pack_bf16(zt[n][2], zt[n][3]);
          }
          kl += (double)(klc * kLn2);
          // dk_idx(16 keys x 64) += dz^T q_idx   (k = 16 query slots)
          uint32_t az[4];
          az[0] = pack_bf16(zt[0][0], zt[0][1]);
          az[1] = pack_bf16(zt[0][2], zt[0][3]);
          az[2] = pack_bf16(zt[1][0], zt[1][1]);
          az[3] = pack_bf16(zt[1][2], zt[1][3]);
          const int qrow = (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
          for (int n2 = 0; n2 < 4; ++n2) {
            uint32_t bq[4];
            ldmatrix_x4_trans(bq, sQi + sw128(qrow, n2 * 2 + (lane >> 4)));
            mma_bf16_16816(dki[2 * n2], az, bq[0], bq[1]);
            mma_bf16_16816(dki[2 * n2 + 1], az, bq[2], bq[3]);
          }
        }
        __syncwarp();  // dz complete for every key
        if (lane == 0) mbar_arrive(e_sync2);
        ok = __all_sync(0xffffffffu, mbar_wait(e_sync2, u & 1, p.wait_ns, abort_flag));
        if (!ok) break;
        if (warp * 16 < p.DI) {
          // dq_idx(16 slots x 16 d_idx) = dz k_idx   (k = 128 keys)
          float acc[2][4];
#pragma unroll
          for (int n = 0; n < 2; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            uint32_t a[4], bk[4];
            ldmatrix_x4_trans(a, sDZ + swz32(ks * 16 + (lane & 7) + ((lane >> 4) << 3), (lane >> 3) & 1));
            ldmatrix_x4_trans(bk, sKi + sw128(ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3),
                                              warp * 2 + (lane >> 4)));
            mma_bf16_16816(acc[0], a, bk[0], bk[1]);
            mma_bf16_16816(acc[1], a, bk[2], bk[3]);
          }
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int qs = (lane >> 2) + hh * 8;
            const int qp = s_qp[qs];
            if (qp >= 0) {
              __nv_bfloat16* dst = p.dqi_part + (int64_t)qp * p.DI + warp * 16;
#pragma unroll
              for (int n = 0; n < 2; ++n)
                *reinterpret_cast<uint32_t*>(dst + n * 8 + (lane & 3) * 2) =
                    pack_bf16(acc[n][2 * hh] * p.sidx, acc[n][2 * hh + 1] * p.sidx);
            }
          }
        }
        // ---- E2: dQ^T columns of this warpgroup (thread = d) ----
        ok = __all_sync(0xffffffffu, mbar_wait(b_q, u & 1, p.wait_ns, abort_flag));
        if (!ok) break;
        tc_fence_after();
        if (tl < D) {  // warp-uniform
          uint32_t a[32];
          tmem_ld_32x32b_x32(tmem + lb + cDQT + 32 * wg, a);
          tmem_wait_ld();
          // stage the warpgroup's 32 rows (row-major, padded) so the global stores
          // below write whole 256-byte partial rows; lanes (2m, 2m+1) swap one value
          // so each stores a bf16 pair
          uint8_t* stg = sm + L::kStg + wg * 32 * L::kStgRow;
          const bool odd = lane & 1;
          const int dcol = tl & ~1;
#pragma unroll
          for (int x = 0; x < 32; x += 2) {
            const float v0 = __uint_as_float(a[x]) * p.scale;
            const float v1 = __uint_as_float(a[x + 1]) * p.scale;
            const float mine = odd ? v1 : v0;
            const float give = odd ? v0 : v1;
            const float got = __shfl_xor_sync(0xffffffffu, give, 1);
            *reinterpret_cast<uint32_t*>(stg + (x + (odd ? 1 : 0)) * L::kStgRow + dcol * 2) =
                odd ? pack_bf16(got, mine) : pack_bf16(mine, got);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&e_stg[wg]);
        ok = __all_sync(0xffffffffu, mbar_wait(&e_stg[wg], u & 1, p.wait_ns, abort_flag));
        if (!ok) break;
        {
          const uint8_t* stg = sm + L::kStg + wg * 32 * L::kStgRow;
          const int wt = (warp & 3) * 32 + lane;  // 0..127 within the warpgroup
          constexpr int CPR = D / 8;              // 16-byte chunks per row
#pragma unroll
          for (int x = wt; x < 32 * CPR; x += 128) {
            const int r = x / CPR, cc = x % CPR;
            const int rp = s_rp[32 * wg + r];
            const uint4 v = *reinterpret_cast<const uint4*>(stg + r * L::kStgRow + cc * 16);
            if (rp >= 0) *reinterpret_cast<uint4*>(p.dq_part + (int64_t)rp * D + cc * 8) = v;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(b_e);
          mbar_arrive(&qempty[s]);
          if (ch == nch - 1) mbar_arrive(kvempty);
        }
      }
      if (!ok) break;
      // ---- block end: dK (x scale), dV from TMEM; dk_idx share from registers ----
      const bool in = j < p.N;
      __nv_bfloat16* dk_row = p.dk + (((int64_t)b * p.N + j) * p.H_kv + g) * D;
      __nv_bfloat16* dv_row = p.dv + (((int64_t)b * p.N + j) * p.H_kv + g) * D;
      if (nch == 0) {
        if (in) {
          for (int x = wg * (D / 2); x < (wg + 1) * (D / 2); ++x) {
            dk_row[x] = __float2bfloat16(0.f);
            dv_row[x] = __float2bfloat16(0.f);
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
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_kfree);
        ++nkeys;
      }
      // dk_idx share of group g for this warp's 16 keys (C-fragment layout)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int jj = c * 128 + kw + (lane >> 2) + hh * 8;
        if (jj < p.N) {
          float* dst = p.dki_part + (((int64_t)b * p.H_kv + g) * p.N + jj) * p.DI;
#pragma unroll
          for (int n = 0; n < 8; ++n) {
            const int col = n * 8 + (lane & 3) * 2;
            if (col < p.DI) {
              dst[col] = dki[n][2 * hh] * p.sidx;
              dst[col + 1] = dki[n][2 * hh + 1] * p.sidx;
            }
          }
        }
      }
#pragma unroll
      for (int n = 0; n < 8; ++n) dki[n][0] = dki[n][1] = dki[n][2] = dki[n][3] = 0.f;
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

template <int D, int G>
cudaError_t launch_dg(const BwdTcParams& prm, const CUtensorMap& tk, const CUtensorMap& tv,
                      const Ctx& cx, cudaStream_t st) {
  using L = BL<D>;
  auto kern = bwd_tc_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  kernel_event(MSA_KERNEL_BWD, true, st);
  kern<<<cx.num_sms, kThreads, L::kAlloc, st>>>(tk, tv, prm);
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
  CUtensorMap tk, tv;
  const uint64_t dims[4] = {(uint64_t)s.d, (uint64_t)s.H_kv, (uint64_t)s.N, (uint64_t)s.B};
  const uint64_t strides[3] = {(uint64_t)s.d * 2, (uint64_t)s.H_kv * s.d * 2,
                               (uint64_t)s.N * s.H_kv * s.d * 2};
  const uint32_t box[4] = {64, 1, 128, 1};
  if (!encode_tiled(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, k, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tiled(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, v, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  BwdTcParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.dO = static_cast<const __nv_bfloat16*>(dO);
  p.q_idx = static_cast<const __nv_bfloat16*>(q_idx);
  p.k_idx = static_cast<const __nv_bfloat16*>(k_idx);
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
  if (s.d == 128) return s.G == 4 ? launch_dg<128, 4>(p, tk, tv, cx, st) : launch_dg<128, 8>(p, tk, tv, cx, st);
  return s.G == 4 ? launch_dg<64, 4>(p, tk, tv, cx, st) : launch_dg<64, 8>(p, tk, tv, cx, st);
}

}  // namespace msa
