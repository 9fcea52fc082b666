// attn_bwd.cu -- fused backward of the MSA main branch and of the KL alignment loss.
//
// Method: Flash-MSA article (tech.kuratif.com) ¶7 -- proxy and main gradients are
// computed together because the proxy's training signal needs both branches'
// probabilities, over the cached block indices, so the backward is linear in N;
// MSA summary (7minutos.es), "Cómo se entrena MSA" ¶1-2 -- the KL pulls the index
// distribution over the selected tokens toward the main distribution averaged over
// the group's heads; the teacher is detached and only the index projections get
// the KL gradient.
//
// Per row (query i, head h of group g) over its token set T:
//   P_h = exp(scale q.k - lse_h),  dS_h = P_h (dO_h . v - D_h),  D_h = dO_h . o_h
//   dq_h = scale sum dS_h k,  dk += scale dS_h q_h,  dv += P_h dO_h
//   p_T = mean_h P_h,  p_I = exp(scale_idx q_idx.k_idx - lse_idx),
//   dz = w (p_I - p_T),  dq_idx = scale_idx sum dz k_idx,  dk_idx += scale_idx dz q_idx,
//   KL += w sum p_T (log p_T - log p_I).
//
// GB300 layout of the work.  KV-outer over the inverted lists of plan.cu: one CTA
// owns one key block (b, g, c) at a time, pulled heavy-first (early blocks are
// selected by the most queries) from a device counter.  The block's K, V, k_idx
// stay in shared memory; dK and dV accumulate in registers (8 warps x 16 keys) over
// every gathered chunk of 64 rows (query x head) and are written once, so dk/dv need
// no atomics; dk_idx accumulates in shared memory and is summed over groups by a
// reduce kernel; dq and dq_idx are written as per-(query, slot) partials and summed
// by reduce kernels.  Chunks are double-buffered with cp.async; contractions are
// mma.sync m16n8k16 (bf16 in, fp32 accumulate).
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace msa {
namespace {

constexpr int kBwdThreads = 256;
constexpr int kRows = 64;  // rows (query x head) per chunk
constexpr int kQCP = 16;   // query slots per chunk, padded to one MMA tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct BwdParams {
  const __nv_bfloat16 *q, *k, *v, *dO, *q_idx, *k_idx;
  const float *lse, *Dv, *lse_idx;
  const int *off, *entries;
  __nv_bfloat16 *dk, *dv;
  __nv_bfloat16* dq_part;   // [(rkv*topk + slot)*G + h][D]
  __nv_bfloat16* dqi_part;  // [(rkv*topk + slot)][DI]
  float* dki_part;          // [B][H_kv][N][DI]
  double* kl_acc;
  int* key_counter;
  int64_t keys;
  int B, N, H_kv, nb, topk;
  float scale, scale_log2, sidx, sidx_log2, w;
};

// 32-byte rows (16 bf16): 2 chunks, swapped every 4 rows so 8-row ldmatrix phases
// hit distinct banks.
__device__ __forceinline__ uint32_t swz32(int row, int chunk) {
  return (uint32_t)(row * 32 + ((chunk ^ ((row >> 2) & 1)) << 4));
}

template <int D, int DI>
struct BwdSmem {
  static constexpr int kRB = 2 * D, kRBI = 2 * DI;
  static constexpr int kK = 0;
  static constexpr int kV = kK + 128 * kRB;
  static constexpr int kKi = kV + 128 * kRB;
  // one chunk buffer: Q, dO, q_idx rows and per-row / per-query scalars
  static constexpr int kBQ = 0;
  static constexpr int kBdO = kBQ + kRows * kRB;
  static constexpr int kBQi = kBdO + kRows * kRB;
  static constexpr int kBLse = kBQi + kQCP * kRBI;  // float[64] lse * log2(e)
  static constexpr int kBD = kBLse + kRows * 4;     // float[64] D
  static constexpr int kBEnt = kBD + kRows * 4;     // int[16] query entries
  static constexpr int kBLi = kBEnt + kQCP * 4;     // float[16] lse_idx * log2(e)
  static constexpr int kBuf = kBLi + kQCP * 4;
  static constexpr int kBuf0 = kKi + 128 * kRBI;
  static constexpr int kdS = kBuf0 + 2 * kBuf;        // bf16 [128 keys][64 rows]
  static constexpr int kPT = kdS + 128 * 128;         // float [128][16]
  static constexpr int kdZ = kPT + 128 * kQCP * 4;    // bf16 [128][16]
  static constexpr int kKiAcc = kdZ + 128 * 32;       // float [128][DI + 4]
  static constexpr int kMisc = kKiAcc + 128 * (DI + 4) * 4;
  static constexpr int kBytes = kMisc + 16;
};

template <int D, int DI, int G>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_kernel(const BwdParams p) {
  using L = BwdSmem<D, DI>;
  constexpr int RB = L::kRB, RBI = L::kRBI;
  constexpr int QC = kRows / G;  // queries per chunk
  static_assert(QC <= kQCP, "chunk queries");
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sK = smem + L::kK;
  uint8_t* sV = smem + L::kV;
  uint8_t* sKi = smem + L::kKi;
  uint8_t* sdS = smem + L::kdS;
  float* sPT = reinterpret_cast<float*>(smem + L::kPT);
  uint8_t* sdZ = smem + L::kdZ;
  float* sKiAcc = reinterpret_cast<float*>(smem + L::kKiAcc);
  int* s_key = reinterpret_cast<int*>(smem + L::kMisc);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BG = p.B * p.H_kv;
  const int kw0 = warp * 16;  // this warp's 16 keys of the block
  double kl_loc = 0.0;

  for (;;) {
    if (threadIdx.x == 0) *s_key = atomicAdd(p.key_counter, 1);
    __syncthreads();
    const int kk = *s_key;
    __syncthreads();
    if (kk >= p.keys) break;
    const int c = kk / BG, bg = kk - c * BG;  // heavy-first: block-major order
    const int b = bg / p.H_kv, g = bg - b * p.H_kv;
    const int key = bg * p.nb + c;
    const int e_begin = __ldg(&p.off[key]), e_end = __ldg(&p.off[key + 1]);
    const int nch = (e_end - e_begin + QC - 1) / QC;

    // ---- block operands: K, V (group g), k_idx (shared head) ----
    for (int x = threadIdx.x; x < 128 * (D / 8); x += kBwdThreads) {
      const int r = x / (D / 8), ch = x % (D / 8);
      const int j = c * 128 + r;
      const bool ok = j < p.N;
      const int64_t src = (((int64_t)b * p.N + (ok ? j : 0)) * p.H_kv + g) * D + ch * 8;
      cp_async_16(sK + swz<RB>(r, ch), p.k + src, ok);
      cp_async_16(sV + swz<RB>(r, ch), p.v + src, ok);
    }
    for (int x = threadIdx.x; x < 128 * (DI / 8); x += kBwdThreads) {
      const int r = x / (DI / 8), ch = x % (DI / 8);
      const int j = c * 128 + r;
      const bool ok = j < p.N;
      const int64_t src = ((int64_t)b * p.N + (ok ? j : 0)) * DI + ch * 8;
      cp_async_16(sKi + swz<RBI>(r, ch), p.k_idx + src, ok);
    }
    for (int x = threadIdx.x; x < 128 * (DI + 4); x += kBwdThreads) sKiAcc[x] = 0.f;

    auto load_chunk = [&](int ch, int sl) {
      uint8_t* buf = smem + L::kBuf0 + sl * L::kBuf;
      const int q0 = e_begin + ch * QC;
      const int nq = min(QC, e_end - q0);
      for (int x = threadIdx.x; x < kRows * (D / 8); x += kBwdThreads) {
        const int r = x / (D / 8), cc = x % (D / 8);
        const int qi = r / G, h = r % G;
        const bool ok = qi < nq;
        const int i = ok ? (__ldg(&p.entries[q0 + qi]) >> 5) : 0;
        const int64_t src = (((int64_t)b * p.N + i) * p.H_kv * G + g * G + h) * D + cc * 8;
        cp_async_16(buf + L::kBQ + swz<RB>(r, cc), p.q + src, ok);
        cp_async_16(buf + L::kBdO + swz<RB>(r, cc), p.dO + src, ok);
      }
      for (int x = threadIdx.x; x < kQCP * (DI / 8); x += kBwdThreads) {
        const int qi = x / (DI / 8), cc = x % (DI / 8);
        const bool ok = qi < nq;
        const int i = ok ? (__ldg(&p.entries[q0 + qi]) >> 5) : 0;
        const int64_t src = (((int64_t)b * p.N + i) * p.H_kv + g) * DI + cc * 8;
        cp_async_16(buf + L::kBQi + swz<RBI>(qi, cc), p.q_idx + src, ok);
      }
      float* s_lse = reinterpret_cast<float*>(buf + L::kBLse);
      float* s_D = reinterpret_cast<float*>(buf + L::kBD);
      int* s_ent = reinterpret_cast<int*>(buf + L::kBEnt);
      float* s_li = reinterpret_cast<float*>(buf + L::kBLi);
      if (threadIdx.x < kRows) {
        const int r = threadIdx.x, qi = r / G, h = r % G;
        if (qi < nq) {
          const int i = __ldg(&p.entries[q0 + qi]) >> 5;
          const int64_t x = ((int64_t)b * p.H_kv * G + g * G + h) * p.N + i;
          s_lse[r] = __ldg(&p.lse[x]) * kLog2e;
          s_D[r] = __ldg(&p.Dv[x]);
        } else {
          s_lse[r] = 0.f;
          s_D[r] = 0.f;
        }
      } else if (threadIdx.x < kRows + kQCP) {
        const int qi = threadIdx.x - kRows;
        if (qi < nq) {
          const int e = __ldg(&p.entries[q0 + qi]);
          s_ent[qi] = e;
          s_li[qi] = __ldg(&p.lse_idx[((int64_t)bg) * p.N + (e >> 5)]) * kLog2e;
        } else {
          s_ent[qi] = -1;
          s_li[qi] = 0.f;
        }
      }
    };

    if (nch > 0) load_chunk(0, 0);
    cp_async_commit();

    float dk[D / 8][4], dv[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) dk[n][e] = dv[n][e] = 0.f;

    for (int ch = 0; ch < nch; ++ch) {
      const int sl = ch & 1;
      if (ch + 1 < nch) {
        load_chunk(ch + 1, sl ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      __syncthreads();
      const uint8_t* buf = smem + L::kBuf0 + sl * L::kBuf;
      const uint8_t* sQ = buf + L::kBQ;
      const uint8_t* sdO = buf + L::kBdO;
      const uint8_t* sQi = buf + L::kBQi;
      const float* s_lse = reinterpret_cast<const float*>(buf + L::kBLse);
      const float* s_D = reinterpret_cast<const float*>(buf + L::kBD);
      const int* s_ent = reinterpret_cast<const int*>(buf + L::kBEnt);
      const float* s_li = reinterpret_cast<const float*>(buf + L::kBLi);

      // ================= phase 1: P^T, dS^T for this warp's keys ==================
      const int jr0 = c * 128 + kw0 + (lane >> 2);  // key of fragment rows 0..7 (+8)
#pragma unroll
      for (int sc = 0; sc < 2; ++sc) {
        const int rs = sc * 32;
        float st[4][4], dp[4][4];
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) st[n][e] = dp[n][e] = 0.f;
#pragma unroll
        for (int kc = 0; kc < D / 16; ++kc) {
          uint32_t ak[4], av[4];
          ldmatrix_x4(ak, sK + swz<RB>(kw0 + (lane & 15), kc * 2 + (lane >> 4)));
          ldmatrix_x4(av, sV + swz<RB>(kw0 + (lane & 15), kc * 2 + (lane >> 4)));
#pragma unroll
          for (int n2 = 0; n2 < 2; ++n2) {
            const int row = rs + n2 * 16 + (lane & 7) + ((lane >> 4) << 3);
            uint32_t bq[4], bo[4];
            ldmatrix_x4(bq, sQ + swz<RB>(row, kc * 2 + ((lane >> 3) & 1)));
            ldmatrix_x4(bo, sdO + swz<RB>(row, kc * 2 + ((lane >> 3) & 1)));
            mma_bf16_16816(st[2 * n2], ak, bq[0], bq[1]);
            mma_bf16_16816(st[2 * n2 + 1], ak, bq[2], bq[3]);
            mma_bf16_16816(dp[2 * n2], av, bo[0], bo[1]);
            mma_bf16_16816(dp[2 * n2 + 1], av, bo[2], bo[3]);
          }
        }
        // P^T and dS^T (st <- P, dp <- dS)
#pragma unroll
        for (int n = 0; n < 4; ++n) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int r = rs + n * 8 + (lane & 3) * 2 + (e & 1);
            const int j = jr0 + ((e >> 1) << 3);
            const int ent = s_ent[r / G];
            const int i = ent >> 5;
            const bool valid = ent >= 0 && j < p.N && j <= i;
            const float P = valid ? exp2f(st[n][e] * p.scale_log2 - s_lse[r]) : 0.f;
            st[n][e] = P;
            dp[n][e] = P * (dp[n][e] - s_D[r]);
          }
        }
        // dV += P^T dO, dK += dS^T Q  (k = rows)
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          uint32_t ap[4], as[4];
          ap[0] = pack_bf16(st[2 * ks][0], st[2 * ks][1]);
          ap[1] = pack_bf16(st[2 * ks][2], st[2 * ks][3]);
          ap[2] = pack_bf16(st[2 * ks + 1][0], st[2 * ks + 1][1]);
          ap[3] = pack_bf16(st[2 * ks + 1][2], st[2 * ks + 1][3]);
          as[0] = pack_bf16(dp[2 * ks][0], dp[2 * ks][1]);
          as[1] = pack_bf16(dp[2 * ks][2], dp[2 * ks][3]);
          as[2] = pack_bf16(dp[2 * ks + 1][0], dp[2 * ks + 1][1]);
          as[3] = pack_bf16(dp[2 * ks + 1][2], dp[2 * ks + 1][3]);
          const int row = rs + ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
          for (int n2 = 0; n2 < D / 16; ++n2) {
            uint32_t bo[4], bq[4];
            ldmatrix_x4_trans(bo, sdO + swz<RB>(row, n2 * 2 + (lane >> 4)));
            ldmatrix_x4_trans(bq, sQ + swz<RB>(row, n2 * 2 + (lane >> 4)));
            mma_bf16_16816(dv[2 * n2], ap, bo[0], bo[1]);
            mma_bf16_16816(dv[2 * n2 + 1], ap, bo[2], bo[3]);
            mma_bf16_16816(dk[2 * n2], as, bq[0], bq[1]);
            mma_bf16_16816(dk[2 * n2 + 1], as, bq[2], bq[3]);
          }
        }
        // dS^T -> smem [key][row] for dQ; teacher p_T -> smem [key][query]
#pragma unroll
        for (int n = 0; n < 4; ++n) {
          const int rr = rs + n * 8;
          const int kl = kw0 + (lane >> 2);
          *reinterpret_cast<uint32_t*>(sdS + swz<128>(kl, rr >> 3) + (lane & 3) * 4) =
              pack_bf16(dp[n][0], dp[n][1]);
          *reinterpret_cast<uint32_t*>(sdS + swz<128>(kl + 8, rr >> 3) + (lane & 3) * 4) =
              pack_bf16(dp[n][2], dp[n][3]);
          float pa = st[n][0] + st[n][1], pb = st[n][2] + st[n][3];
          if constexpr (G >= 4) {
            pa += __shfl_xor_sync(0xffffffffu, pa, 1);
            pb += __shfl_xor_sync(0xffffffffu, pb, 1);
          }
          if constexpr (G >= 8) {
            pa += __shfl_xor_sync(0xffffffffu, pa, 2);
            pb += __shfl_xor_sync(0xffffffffu, pb, 2);
          }
          const int col = rr + (lane & 3) * 2;  // first row of this thread's pair
          if (col % G == 0) {
            const int qloc = col / G;
            sPT[kl * kQCP + qloc] = pa * (1.f / G);
            sPT[(kl + 8) * kQCP + qloc] = pb * (1.f / G);
          }
        }
      }
      // padded query slots of the teacher are zero
      if constexpr (QC < kQCP) {
        constexpr int PAD = kQCP - QC;
        for (int x = threadIdx.x; x < 128 * PAD; x += kBwdThreads)
          sPT[(x / PAD) * kQCP + QC + x % PAD] = 0.f;
      }
      __syncthreads();

      // ================= phase 2: dQ rows; KL terms; dK_idx =======================
      {
        const int mr = 16 * (warp & 3), dh = warp >> 2;
        constexpr int NT = D / 16;  // 8-column tiles in this warp's half of D
        float dq[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) dq[n][0] = dq[n][1] = dq[n][2] = dq[n][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          uint32_t a[4];
          ldmatrix_x4_trans(a, sdS + swz<128>(ks * 16 + (lane & 7) + ((lane >> 4) << 3),
                                              (mr >> 3) + ((lane >> 3) & 1)));
          const int krow = ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
          for (int n2 = 0; n2 < NT / 2; ++n2) {
            uint32_t bk[4];
            ldmatrix_x4_trans(bk, sK + swz<RB>(krow, dh * (D / 16) + n2 * 2 + (lane >> 4)));
            mma_bf16_16816(dq[2 * n2], a, bk[0], bk[1]);
            mma_bf16_16816(dq[2 * n2 + 1], a, bk[2], bk[3]);
          }
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int r = mr + (lane >> 2) + hh * 8;
          const int ent = s_ent[r / G];
          if (ent >= 0) {
            const int64_t rkv = (int64_t)bg * p.N + (ent >> 5);
            __nv_bfloat16* dst =
                p.dq_part + ((rkv * p.topk + (ent & 31)) * G + r % G) * D + dh * (D / 2);
#pragma unroll
            for (int n = 0; n < NT; ++n)
              *reinterpret_cast<uint32_t*>(dst + n * 8 + (lane & 3) * 2) =
                  pack_bf16(dq[n][2 * hh] * p.scale, dq[n][2 * hh + 1] * p.scale);
          }
        }
      }
      {
        // z^T = k_idx q_idx^T for this warp's 16 keys x 16 query slots
        float zt[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n) zt[n][0] = zt[n][1] = zt[n][2] = zt[n][3] = 0.f;
#pragma unroll
        for (int kc = 0; kc < DI / 16; ++kc) {
          uint32_t a[4], bq[4];
          ldmatrix_x4(a, sKi + swz<RBI>(kw0 + (lane & 15), kc * 2 + (lane >> 4)));
          ldmatrix_x4(bq, sQi + swz<RBI>((lane & 7) + ((lane >> 4) << 3), kc * 2 + ((lane >> 3) & 1)));
          mma_bf16_16816(zt[0], a, bq[0], bq[1]);
          mma_bf16_16816(zt[1], a, bq[2], bq[3]);
        }
        const int kl = kw0 + (lane >> 2);
        const int jr = c * 128 + kl;
#pragma unroll
        for (int n = 0; n < 2; ++n) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int qs = n * 8 + (lane & 3) * 2 + (e & 1);
            const int key_l = kl + ((e >> 1) << 3);
            const int j = jr + ((e >> 1) << 3);
            const int ent = s_ent[qs];
            const bool valid = ent >= 0 && j < p.N && j <= (ent >> 5);
            const float zl2 = zt[n][e] * p.sidx_log2 - s_li[qs];  // log2 p_I
            const float pI = valid ? exp2f(zl2) : 0.f;
            const float pT = sPT[key_l * kQCP + qs];
            if (valid && pT > 0.f) kl_loc += (double)pT * (double)((log2f(pT) - zl2) * kLn2);
            zt[n][e] = valid ? p.w * (pI - pT) : 0.f;  // dz
          }
          *reinterpret_cast<uint32_t*>(sdZ + swz32(kl, n) + (lane & 3) * 4) =
              pack_bf16(zt[n][0], zt[n][1]);
          *reinterpret_cast<uint32_t*>(sdZ + swz32(kl + 8, n) + (lane & 3) * 4) =
              pack_bf16(zt[n][2], zt[n][3]);
        }
        // dK_idx(16 keys x DI) += dZ^T q_idx (k = 16 query slots)
        uint32_t az[4];
        az[0] = pack_bf16(zt[0][0], zt[0][1]);
        az[1] = pack_bf16(zt[0][2], zt[0][3]);
        az[2] = pack_bf16(zt[1][0], zt[1][1]);
        az[3] = pack_bf16(zt[1][2], zt[1][3]);
        const int qrow = (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
        for (int n2 = 0; n2 < DI / 16; ++n2) {
          uint32_t bq[4];
          ldmatrix_x4_trans(bq, sQi + swz<RBI>(qrow, n2 * 2 + (lane >> 4)));
          float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
          mma_bf16_16816(acc0, az, bq[0], bq[1]);
          mma_bf16_16816(acc1, az, bq[2], bq[3]);
          float* r0 = sKiAcc + kl * (DI + 4) + n2 * 16 + (lane & 3) * 2;
          float* r1 = r0 + 8 * (DI + 4);
          r0[0] += acc0[0];
          r0[1] += acc0[1];
          r1[0] += acc0[2];
          r1[1] += acc0[3];
          r0[8] += acc1[0];
          r0[9] += acc1[1];
          r1[8] += acc1[2];
          r1[9] += acc1[3];
        }
      }
      __syncthreads();

      // ================= phase 3: dq_idx = scale_idx dZ k_idx ======================
      if (warp < DI / 16) {
        float acc[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          uint32_t a[4], bk[4];
          ldmatrix_x4_trans(a, sdZ + swz32(ks * 16 + (lane & 7) + ((lane >> 4) << 3),
                                          (lane >> 3) & 1));
          ldmatrix_x4_trans(bk, sKi + swz<RBI>(ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3),
                                               warp * 2 + (lane >> 4)));
          mma_bf16_16816(acc[0], a, bk[0], bk[1]);
          mma_bf16_16816(acc[1], a, bk[2], bk[3]);
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int qs = (lane >> 2) + hh * 8;
          const int ent = s_ent[qs];
          if (ent >= 0) {
            const int64_t rkv = (int64_t)bg * p.N + (ent >> 5);
            __nv_bfloat16* dst = p.dqi_part + (rkv * p.topk + (ent & 31)) * DI + warp * 16;
#pragma unroll
            for (int n = 0; n < 2; ++n)
              *reinterpret_cast<uint32_t*>(dst + n * 8 + (lane & 3) * 2) =
                  pack_bf16(acc[n][2 * hh] * p.sidx, acc[n][2 * hh + 1] * p.sidx);
          }
        }
      }
      __syncthreads();
    }
    cp_async_wait<0>();
    __syncthreads();

    // ---- write dK (x scale), dV of this block and its dk_idx share ----
    {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int j = c * 128 + kw0 + (lane >> 2) + hh * 8;
        if (j < p.N) {
          const int64_t base = (((int64_t)b * p.N + j) * p.H_kv + g) * D;
#pragma unroll
          for (int n = 0; n < D / 8; ++n) {
            const int d0 = n * 8 + (lane & 3) * 2;
            *reinterpret_cast<uint32_t*>(p.dk + base + d0) =
                pack_bf16(dk[n][2 * hh] * p.scale, dk[n][2 * hh + 1] * p.scale);
            *reinterpret_cast<uint32_t*>(p.dv + base + d0) = pack_bf16(dv[n][2 * hh], dv[n][2 * hh + 1]);
          }
        }
      }
      for (int x = threadIdx.x; x < 128 * DI; x += kBwdThreads) {
        const int r = x / DI, col = x % DI;
        const int j = c * 128 + r;
        if (j < p.N)
          p.dki_part[(((int64_t)b * p.H_kv + g) * p.N + j) * DI + col] =
              sKiAcc[r * (DI + 4) + col] * p.sidx;
      }
    }
    __syncthreads();
  }

  // ---- KL: warp reduce, one double atomic per warp ----
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) kl_loc += __shfl_xor_sync(0xffffffffu, kl_loc, o);
  if (lane == 0 && kl_loc != 0.0) atomicAdd(p.kl_acc, kl_loc * (double)p.w);
}

// D[b,h,i] = dO[b,i,h,:] . o[b,i,h,:]; one warp per (b, i, h).
template <int D>
__global__ void bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                               const __nv_bfloat16* __restrict__ dO, float* __restrict__ Dv,
                               int64_t rows, int N, int H_q) {
  const int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= rows) return;  // rows = B*N*H_q, w = (b*N + i)*H_q + h
  constexpr int E = D / 32;
  const __nv_bfloat16* a = o + w * D + lane * E;
  const __nv_bfloat16* bb = dO + w * D + lane * E;
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(a + e);
    const __nv_bfloat162 y = *reinterpret_cast<const __nv_bfloat162*>(bb + e);
    s += __low2float(x) * __low2float(y) + __high2float(x) * __high2float(y);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) {
    const int h = (int)(w % H_q);
    const int64_t bi = w / H_q;
    const int i = (int)(bi % N);
    const int64_t b = bi / N;
    Dv[(b * H_q + h) * N + i] = s;
  }
}

// Sum of the per-slot partials of one (b, g, i) row: dq (the G heads of the group, G*W
// contiguous bf16 per slot) or dq_idx (G = 1, W = d_idx).  Lanes read 16-byte chunks;
// when a row has fewer than 32 chunks a warp serves several rows.
template <int W, int G>
__global__ void __launch_bounds__(256) slot_reduce_kernel(
    const __nv_bfloat16* __restrict__ part, const int32_t* __restrict__ block_idx,
    __nv_bfloat16* __restrict__ out, int64_t rows_kv, int N, int H_kv, int topk, int nb) {
  constexpr int TC = G * W / 8;               // 16-byte chunks per row and slot
  constexpr int RPW = TC >= 32 ? 1 : 32 / TC; // rows per warp
  constexpr int CPL = TC >= 32 ? TC / 32 : 1; // chunks per lane
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t rkv = warp * RPW + (TC >= 32 ? 0 : lane / TC);
  const int l = TC >= 32 ? lane : lane % TC;
  if (rkv >= rows_kv) return;
  const int i = (int)(rkv % N);
  const int64_t bg = rkv / N;
  const int g = (int)(bg % H_kv);
  const int64_t b = bg / H_kv;
  float acc[CPL][8];
#pragma unroll
  for (int x = 0; x < CPL; ++x)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[x][e] = 0.f;
  const int32_t* sel = block_idx + rkv * topk;
  for (int s = 0; s < topk; ++s) {
    const int c = __ldg(&sel[s]);
    if (c < 0 || c >= nb) continue;
    const uint4* src = reinterpret_cast<const uint4*>(part + (rkv * topk + s) * G * W);
#pragma unroll
    for (int x = 0; x < CPL; ++x) {
      const uint4 raw = __ldg(&src[l + 32 * x]);
      const __nv_bfloat162* pr = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc[x][2 * e] += __low2float(pr[e]);
        acc[x][2 * e + 1] += __high2float(pr[e]);
      }
    }
  }
  // out row: dq [b][i][g*G .. g*G+G-1][W]  or  dq_idx [b][i][g][W]
  uint4* dst = reinterpret_cast<uint4*>(out + ((b * N + i) * H_kv + g) * (int64_t)G * W);
#pragma unroll
  for (int x = 0; x < CPL; ++x) {
    uint4 o;
    uint32_t* pw = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int e = 0; e < 4; ++e) pw[e] = pack_bf16(acc[x][2 * e], acc[x][2 * e + 1]);
    dst[l + 32 * x] = o;
  }
}

// dk_idx[b,j,:] = sum over groups of the per-group shares.
__global__ void dki_reduce_kernel(const float* __restrict__ part, __nv_bfloat16* __restrict__ out,
                                  int B, int N, int H_kv, int DI) {
  const int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const int64_t per_b = (int64_t)N * DI;
  if (t >= (int64_t)B * per_b) return;
  const int64_t b = t / per_b, r = t - b * per_b;
  float s = 0.f;
  for (int g = 0; g < H_kv; ++g) s += part[(b * H_kv + g) * per_b + r];
  out[t] = __float2bfloat16(s);
}

__global__ void kl_out_kernel(const double* __restrict__ acc, float* __restrict__ out) {
  *out = (float)*acc;
}

template <int D, int DI, int G>
cudaError_t launch_bwd_kernel(const BwdParams& p, const Ctx& cx, cudaStream_t st) {
  using L = BwdSmem<D, DI>;
  auto kern = bwd_kernel<D, DI, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
  if (e != cudaSuccess) return e;
  kernel_event(MSA_KERNEL_BWD, true, st);
  kern<<<cx.num_sms, kBwdThreads, L::kBytes, st>>>(p);
  kernel_event(MSA_KERNEL_BWD, false, st);
  note_launch();
  return cudaGetLastError();
}

template <int D, int DI>
cudaError_t dispatch_bwd_g(int G, const BwdParams& p, const Ctx& cx, cudaStream_t st) {
  if (G == 4) return launch_bwd_kernel<D, DI, 4>(p, cx, st);
  if (G == 8) return launch_bwd_kernel<D, DI, 8>(p, cx, st);
  return cudaErrorInvalidValue;
}

struct BwdWs {
  Plan pl;
  int* counter;
  float* Dv;
  __nv_bfloat16* dq_part;
  __nv_bfloat16* dqi_part;
  float* dki_part;
  double* kl_acc;
};

size_t carve(const Shape& s, void* ws, BwdWs* out) {
  uint8_t* base = static_cast<uint8_t*>(ws);
  size_t off = plan_bytes(s);
  const size_t parts = (size_t)s.rows_kv() * s.topk;
  BwdWs w;
  if (base) w.pl = plan_carve(s, base);
  w.counter = reinterpret_cast<int*>(base + off);
  w.kl_acc = reinterpret_cast<double*>(base + off + 128);
  off += 256;
  w.Dv = reinterpret_cast<float*>(base + off);
  off += align256((size_t)s.B * s.H_q * s.N * 4);
  w.dq_part = reinterpret_cast<__nv_bfloat16*>(base + off);
  off += align256(parts * s.G * s.d * 2);
  w.dqi_part = reinterpret_cast<__nv_bfloat16*>(base + off);
  off += align256(parts * s.d_idx * 2);
  w.dki_part = reinterpret_cast<float*>(base + off);
  off += align256((size_t)s.B * s.H_kv * s.N * s.d_idx * 4);
  if (out) *out = w;
  return off;
}

}  // namespace

size_t bwd_ws_bytes(const Shape& s) { return carve(s, nullptr, nullptr); }

cudaError_t run_bwd(const Shape& s, const void* q, const void* k, const void* v, const void* o,
                    const float* lse, const void* dO, const void* q_idx, const void* k_idx,
                    const int32_t* block_idx, const float* lse_idx, float kl_weight, void* dq,
                    void* dk, void* dv, void* dq_idx, void* dk_idx, float* kl_out, void* ws,
                    const Ctx& cx, cudaStream_t st) {
  BwdWs w;
  carve(s, ws, &w);
  cudaError_t e = launch_plan(s, block_idx, kRows / s.G, w.pl, cx, st);
  if (e != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(w.counter, 0, 256, st)) != cudaSuccess) return e;  // counter + KL
  {
    const int64_t rows = (int64_t)s.B * s.N * s.H_q;
    const unsigned grid = (unsigned)((rows * 32 + 255) / 256);
    if (s.d == 128)
      bwd_pre_kernel<128><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(o),
                                                static_cast<const __nv_bfloat16*>(dO), w.Dv, rows,
                                                s.N, s.H_q);
    else
      bwd_pre_kernel<64><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(o),
                                               static_cast<const __nv_bfloat16*>(dO), w.Dv, rows,
                                               s.N, s.H_q);
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  BwdParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.dO = static_cast<const __nv_bfloat16*>(dO);
  p.q_idx = static_cast<const __nv_bfloat16*>(q_idx);
  p.k_idx = static_cast<const __nv_bfloat16*>(k_idx);
  p.lse = lse;
  p.Dv = w.Dv;
  p.lse_idx = lse_idx;
  p.off = w.pl.off;
  p.entries = w.pl.entries;
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.dq_part = w.dq_part;
  p.dqi_part = w.dqi_part;
  p.dki_part = w.dki_part;
  p.kl_acc = w.kl_acc;
  p.key_counter = w.counter;
  p.keys = s.keys();
  p.B = s.B;
  p.N = s.N;
  p.H_kv = s.H_kv;
  p.nb = s.nb;
  p.topk = s.topk;
  p.scale = s.scale;
  p.scale_log2 = s.scale * kLog2e;
  p.sidx = s.scale_idx;
  p.sidx_log2 = s.scale_idx * kLog2e;
  p.w = kl_weight;
  if (s.d == 128 && s.d_idx == 64) e = dispatch_bwd_g<128, 64>(s.G, p, cx, st);
  else if (s.d == 128) e = dispatch_bwd_g<128, 32>(s.G, p, cx, st);
  else if (s.d_idx == 64) e = dispatch_bwd_g<64, 64>(s.G, p, cx, st);
  else e = dispatch_bwd_g<64, 32>(s.G, p, cx, st);
  if (e != cudaSuccess) return e;
  {
    __nv_bfloat16* dqb = static_cast<__nv_bfloat16*>(dq);
    __nv_bfloat16* dqib = static_cast<__nv_bfloat16*>(dq_idx);
    const int64_t R = s.rows_kv();
    auto grid_for = [&](int tc) {
      const int64_t rpw = tc >= 32 ? 1 : 32 / tc;
      const int64_t warps = (R + rpw - 1) / rpw;
      return (unsigned)((warps + 7) / 8);
    };
    if (s.d == 128 && s.G == 4)
      slot_reduce_kernel<128, 4><<<grid_for(64), 256, 0, st>>>(w.dq_part, block_idx, dqb, R, s.N,
                                                              s.H_kv, s.topk, s.nb);
    else if (s.d == 128)
      slot_reduce_kernel<128, 8><<<grid_for(128), 256, 0, st>>>(w.dq_part, block_idx, dqb, R, s.N,
                                                               s.H_kv, s.topk, s.nb);
    else if (s.G == 4)
      slot_reduce_kernel<64, 4><<<grid_for(32), 256, 0, st>>>(w.dq_part, block_idx, dqb, R, s.N,
                                                             s.H_kv, s.topk, s.nb);
    else
      slot_reduce_kernel<64, 8><<<grid_for(64), 256, 0, st>>>(w.dq_part, block_idx, dqb, R, s.N,
                                                             s.H_kv, s.topk, s.nb);
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (s.d_idx == 64)
      slot_reduce_kernel<64, 1><<<grid_for(8), 256, 0, st>>>(w.dqi_part, block_idx, dqib, R, s.N,
                                                            s.H_kv, s.topk, s.nb);
    else
      slot_reduce_kernel<32, 1><<<grid_for(4), 256, 0, st>>>(w.dqi_part, block_idx, dqib, R, s.N,
                                                            s.H_kv, s.topk, s.nb);
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t n = (int64_t)s.B * s.N * s.d_idx;
    dki_reduce_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(
        w.dki_part, static_cast<__nv_bfloat16*>(dk_idx), s.B, s.N, s.H_kv, s.d_idx);
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (kl_out) {
    kl_out_kernel<<<1, 1, 0, st>>>(w.kl_acc, kl_out);
    note_launch();
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace msa
