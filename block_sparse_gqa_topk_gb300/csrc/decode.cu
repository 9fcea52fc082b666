// decode.cu -- MSA decode: one new query token per sequence against its KV cache.
//
// Method: at inference the index branch scores the new token against the cached
// index keys, max-pools them per 128-token block and keeps the query's own block plus
// the k-1 best earlier blocks (MSA summary, 7minutos.es, "Cómo funcionan las dos ramas"
// ¶1-2; the block indices are then reused by the main branch, Flash-MSA article,
// tech.kuratif.com, ¶3); the main branch is exact softmax attention of the group's heads
// over those blocks, split across blocks and combined.  For a cache of length L the
// result equals row L-1 of the training path (msa_index_topk + msa_fwd) on the cache.
//
// Decode moves the cache from HBM once and does little arithmetic per byte; the small
// products run on mma.sync so that the loads, not shared-memory traffic, set the pace:
//   decode_pool_kernel    one warp per earlier key block: pooled scores of up to 16
//                         groups (mma.sync, k_idx fragments straight from HBM);
//   decode_select_kernel  one CTA per (sequence, group): exact top-(k-1) (ties -> lower
//                         block) by per-lane lists, warp rounds and a counting rank;
//   decode_attn_kernel    one CTA per (sequence, group, slot): the block's K/V in smem,
//                         scores and P V on mma.sync, softmax partial (lse); the
//                         group's last CTA merges its k partials into o and lse.
#include <cuda_fp8.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace msa {
namespace {

struct DecodeParams {
  const __nv_bfloat16* q;      // [B][H_q][d]
  const __nv_bfloat16* q_idx;  // [B][H_kv][d_idx]
  const __nv_bfloat16* k;      // [B][Lmax][H_kv][d]
  const __nv_bfloat16* v;      // [B][Lmax][H_kv][d]
  const __nv_bfloat16* k_idx;  // [B][Lmax][d_idx]
  const uint8_t* k8;           // [B][Lmax][H_kv][d] E4M3 codes (FP8 cache; else null)
  const uint8_t* v8;
  const float* k_scale;        // [B][Lmax][H_kv] per-row scales of k8, v8
  const float* v_scale;
  const int32_t* lens;         // [B], 1 <= lens[b] <= Lmax
  int32_t* block_idx;          // [B][H_kv][topk]
  float* pooled;               // [B][H_kv][nbm]
  float* o_part;               // [B][H_kv][topk][G][d]
  float* lse_part;             // [B][H_kv][topk][G]
  int* arrive;                 // [B][H_kv] finished attention CTAs
  __nv_bfloat16* o;            // [B][H_q][d]
  float* lse;                  // [B][H_q]
  int B, Lmax, H_kv, G, d, d_idx, topk, nbm;
  float scale;
  int* status;
};

__device__ __forceinline__ int seq_len(const DecodeParams& p, int b, int* status) {
  int L = __ldg(&p.lens[b]);
  if (L < 1 || L > p.Lmax) {  // invalid length: recorded, treated as a one-token cache
    if (threadIdx.x == 0) atomicCAS(status, 0, MSA_ERR_ARG);
    L = 1;
  }
  return L;
}

// pooled[b][g][c] = max over the 128 keys j of block c of q_idx[b,g] . k_idx[b,j], for
// every block wholly before the query's block.  The scores of a block are a small
// contraction (128 keys x H_kv groups x d_idx) done with mma.sync m16n8k16: A = the
// block's k_idx rows straight from global memory, B = the query index vectors (held in
// registers for the whole warp).  Grid (ceil(nbm / 8), B, ceil(H_kv / (8 NT))), 8 warps,
// one key block per warp, 8 NT groups per CTA.
//
// Each lane reads 16 contiguous bytes of a key row per load.  The fragment slots of a
// 16-wide k step are filled from those bytes in a fixed order (a0: elements 0-1, a2:
// 2-3 of the first k step, 4-7 for the second), and the query fragments are read with
// the same order, so every product pairs matching d; the dot product is order-free.
template <int DI, int NT>
__global__ void __launch_bounds__(256) decode_pool_kernel(const DecodeParams p) {
  griddep_launch_dependents();  // the selection may be scheduled while the pool drains
  const int b = blockIdx.y;
  const int L = seq_len(p, b, p.status);
  const int c_own = (L - 1) / 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * 8 + warp;
  if (c >= c_own) return;
  const int gq = lane >> 2, tq = lane & 3;  // fragment row / column group
  constexpr int NP = DI / 32;                // 32-wide d chunks: two k steps each
  // query fragments: group n = gq of each n tile, d = 32 j + 8 tq + 0..7
  uint4 bq[NT][NP];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int grp = blockIdx.z * 8 * NT + nt * 8 + gq;
    const uint4* qrow = reinterpret_cast<const uint4*>(p.q_idx + ((int64_t)b * p.H_kv + grp) * DI);
#pragma unroll
    for (int j = 0; j < NP; ++j) bq[nt][j] = grp < p.H_kv ? __ldg(&qrow[j * 4 + tq]) : make_uint4(0, 0, 0, 0);
  }
  float mx[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) mx[nt][0] = mx[nt][1] = -INFINITY;
  const uint4* kb = reinterpret_cast<const uint4*>(p.k_idx + ((int64_t)b * p.Lmax + c * 128) * DI);
#pragma unroll 2
  for (int mt = 0; mt < 8; ++mt) {  // 16 keys per tile: rows gq and gq + 8
    uint4 w0[NP], w1[NP];
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      w0[j] = __ldg(&kb[(mt * 16 + gq) * (DI / 8) + j * 4 + tq]);
      w1[j] = __ldg(&kb[(mt * 16 + gq + 8) * (DI / 8) + j * 4 + tq]);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < NP; ++j) {
        const uint32_t a0[4] = {w0[j].x, w1[j].x, w0[j].y, w1[j].y};
        const uint32_t a1[4] = {w0[j].z, w1[j].z, w0[j].w, w1[j].w};
        mma_bf16_16816(acc, a0, bq[nt][j].x, bq[nt][j].y);
        mma_bf16_16816(acc, a1, bq[nt][j].z, bq[nt][j].w);
      }
      mx[nt][0] = fmax3(mx[nt][0], acc[0], acc[2]);  // group 2 tq, keys gq and gq + 8
      mx[nt][1] = fmax3(mx[nt][1], acc[1], acc[3]);  // group 2 tq + 1
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float m = mx[nt][e];
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
      const int grp = blockIdx.z * 8 * NT + nt * 8 + 2 * tq + e;
      if (gq == 0 && grp < p.H_kv) p.pooled[((int64_t)b * p.H_kv + grp) * p.nbm + c] = m;
    }
}

// Block scores as sortable 64-bit keys: larger key = larger score, equal scores -> the
// lower block id first.  Keys of distinct blocks are distinct.
__device__ __forceinline__ uint64_t rank_key(float v, int id) {
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // order-preserving map to unsigned
  return ((uint64_t)u << 32) | (uint32_t)(0x7fffffff - id);
}
__device__ __forceinline__ int key_id(uint64_t key) { return 0x7fffffff - (int)(uint32_t)key; }

// block_idx[b][g][:] = the k-1 best earlier blocks (pooled descending, lower id first on
// ties) and the own block, ascending, -1 padded.  One CTA of 8 warps per (b, g):
//   1. every lane keeps a sorted list of its own best KM candidates (registers);
//   2. each warp takes its best M = min(k-1, c_own) in M rounds of a warp-wide max over
//      the lanes' list heads, into shared memory;
//   3. each of the 8 M survivors counts the survivors above it: rank < M is selected,
//      and the selected ids are placed in ascending order by a second count.
template <int KM>
__global__ void __launch_bounds__(256) decode_select_kernel(const DecodeParams p) {
  __shared__ uint64_t s_top[8 * KM];  // warp w's best M at [w M, w M + M)
  __shared__ int s_sel[KM];
  griddep_launch_dependents();  // the attention may be scheduled while this runs
  const int b = blockIdx.y, g = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = seq_len(p, b, p.status);
  const int c_own = (L - 1) / 128;
  const float* src = p.pooled + ((int64_t)b * p.H_kv + g) * p.nbm;
  const int M = min(p.topk - 1, c_own);
  uint64_t top[KM];
#pragma unroll
  for (int s = 0; s < KM; ++s) top[s] = 0;  // below every real key
  griddep_wait();  // the pooled scores (the length above is an input)
  for (int c0 = warp * 32 + lane; c0 < c_own; c0 += 4 * 256) {
    float v4[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v4[u] = c0 + 256 * u < c_own ? __ldg(&src[c0 + 256 * u]) : 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (c0 + 256 * u >= c_own) break;
      uint64_t x = rank_key(v4[u], c0 + 256 * u);
      if (x <= top[KM - 1]) continue;
#pragma unroll
      for (int s = 0; s < KM; ++s) {  // sorted insert, descending
        const uint64_t hi = x > top[s] ? x : top[s];
        x = x > top[s] ? top[s] : x;
        top[s] = hi;
      }
    }
  }
  // warp's best M: each round takes the largest list head, as a warp max of the key's
  // high word and then of the low word among the lanes holding that high word
  for (int r = 0; r < M; ++r) {
    const uint32_t hi = (uint32_t)(top[0] >> 32), lo = (uint32_t)top[0];
    const uint32_t mhi = __reduce_max_sync(0xffffffffu, hi);
    const uint32_t mlo = __reduce_max_sync(0xffffffffu, hi == mhi ? lo : 0u);
    const uint64_t best = ((uint64_t)mhi << 32) | mlo;
    if (lane == 0) s_top[warp * M + r] = best;  // 0 when the warp had fewer than M candidates
    if (best != 0 && top[0] == best) {
#pragma unroll
      for (int s = 0; s + 1 < KM; ++s) top[s] = top[s + 1];
      top[KM - 1] = 0;
    }
  }
  __syncthreads();
  // selection among the 8 M survivors, then ascending order of the selected ids
  const int n = 8 * M;
  const int t = threadIdx.x;
  uint64_t mine = 0;
  int above = n;
  if (t < n) {
    mine = s_top[t];
    above = 0;
    for (int u = 0; u < n; ++u) above += s_top[u] > mine ? 1 : 0;
  }
  const bool sel = mine != 0 && above < M;
  if (sel) s_sel[above] = key_id(mine);
  __syncthreads();
  int32_t* dst = p.block_idx + ((int64_t)b * p.H_kv + g) * p.topk;
  if (t < M) {
    const int id = s_sel[t];
    int pos = 0;
    for (int u = 0; u < M; ++u) pos += s_sel[u] < id ? 1 : 0;
    dst[pos] = id;
  }
  if (t == 0) {
    dst[M] = c_own;  // every selected block lies before the own block
    p.arrive[(int64_t)b * p.H_kv + g] = 0;  // arrival count of the attention CTAs
  }
  for (int s = M + 1 + t; s < p.topk; s += blockDim.x) dst[s] = -1;
}

// Softmax partial of every head of group g over block c (slot `part`); writes lse_part
// and the normalised o_part of the slot.  Both products are mma.sync m16n8k16
// contractions with the group's heads as the 8-wide n dimension:
//   S^T[key][h] = K[key][:] . q_h              (warp w: keys 16w..16w+15)
//   O^T[dd][h]  = sum_key V[key][dd] P[h][key] (warp w: dd = 16w..16w+15)
// K is read straight from global memory into A fragments: each lane loads 16 contiguous
// bytes of a key row (8 for an FP8 row) per 32-wide d chunk, and the fragment slots of
// the chunk's two k steps take them in a fixed order that the query fragments repeat,
// so every product pairs matching d.  V rows are staged in shared memory (cp.async, or
// 16-byte loads widened from E4M3) for ldmatrix.trans.  Rows past the visible end of
// the block are zero.  The scores go through shared memory for the per-head softmax; P
// is rounded to bf16 for the second product (with an FP8 cache the V row scale is
// folded into it), its row sum l stays fp32.
template <int D, int NT, bool F8>
__device__ __forceinline__ void block_partial(const DecodeParams& p, uint8_t* dsm, int64_t part,
                                              int c, int b, int g, int L, float* s_l, float* s_sv) {
  constexpr int KS = D + 8;    // padded V row (bf16): conflict-free ldmatrix phases
  constexpr int PS = 128 + 8;  // padded P row (bf16)
  constexpr int NP = D / 32;   // 32-wide d chunks (two k steps each)
  __nv_bfloat16* sV = reinterpret_cast<__nv_bfloat16*>(dsm);
  float* sS = reinterpret_cast<float*>(dsm + 128 * KS * 2);        // [8 NT][128]
  __nv_bfloat16* sP = reinterpret_cast<__nv_bfloat16*>(sS + 8 * NT * 128);  // [8 NT][PS]
  const int G = p.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int jmax = min(L - 1, c * 128 + 127) - c * 128;  // last visible row of the block
  const int64_t row0 = ((int64_t)b * p.Lmax + c * 128) * p.H_kv + g;  // (b, c 128, g)
  // ---- V rows into shared memory ----
  constexpr int CH = F8 ? D / 16 : D / 8;  // 16-byte chunks per V row
  constexpr int PER = 128 * CH / 256;      // chunks per thread
  uint4 vw[F8 ? PER : 1];
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int x = threadIdx.x + u * 256;
    const int r = x / CH, ch = x % CH;
    const bool ok = r <= jmax;  // row c 128 + r < L <= Lmax
    const int64_t row = row0 + (int64_t)r * p.H_kv;
    if constexpr (F8) {
      vw[u] = ok ? __ldg(reinterpret_cast<const uint4*>(p.v8 + row * D + ch * 16))
                 : make_uint4(0, 0, 0, 0);
    } else {
      cp_async_16(sV + r * KS + ch * 8, p.v + (ok ? row * D + ch * 8 : 0), ok);
    }
  }
  if constexpr (!F8) cp_async_commit();
  // ---- K fragments (rows 16 warp + gq and + 8) and the query fragments ----
  const int ka = warp * 16 + gq, kb = ka + 8;
  uint4 wa[NP], wb[NP];
#pragma unroll
  for (int j = 0; j < NP; ++j) {
    if constexpr (F8) {
      const uint2 ca = ka <= jmax ? __ldg(reinterpret_cast<const uint2*>(p.k8 + (row0 + (int64_t)ka * p.H_kv) * D + 32 * j + 8 * tq))
                                  : make_uint2(0, 0);
      const uint2 cb = kb <= jmax ? __ldg(reinterpret_cast<const uint2*>(p.k8 + (row0 + (int64_t)kb * p.H_kv) * D + 32 * j + 8 * tq))
                                  : make_uint2(0, 0);
      uint32_t ta[4], tb[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {  // fp8 pairs (2e, 2e+1) -> bf16 pairs
        const __nv_fp8x2_storage_t a2 = (__nv_fp8x2_storage_t)((e < 2 ? ca.x : ca.y) >> (16 * (e & 1)));
        const __nv_fp8x2_storage_t b2 = (__nv_fp8x2_storage_t)((e < 2 ? cb.x : cb.y) >> (16 * (e & 1)));
        const float2 fa = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(a2, __NV_E4M3)));
        const float2 fb = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(b2, __NV_E4M3)));
        ta[e] = pack_bf16(fa.x, fa.y);
        tb[e] = pack_bf16(fb.x, fb.y);
      }
      wa[j] = make_uint4(ta[0], ta[1], ta[2], ta[3]);
      wb[j] = make_uint4(tb[0], tb[1], tb[2], tb[3]);
    } else {
      wa[j] = ka <= jmax ? __ldg(reinterpret_cast<const uint4*>(p.k + (row0 + (int64_t)ka * p.H_kv) * D) + 4 * j + tq)
                         : make_uint4(0, 0, 0, 0);
      wb[j] = kb <= jmax ? __ldg(reinterpret_cast<const uint4*>(p.k + (row0 + (int64_t)kb * p.H_kv) * D) + 4 * j + tq)
                         : make_uint4(0, 0, 0, 0);
    }
  }
  float ska = 1.f, skb = 1.f;  // K row scales (FP8)
  if constexpr (F8) {
    ska = ka <= jmax ? __ldg(&p.k_scale[row0 + (int64_t)ka * p.H_kv]) : 0.f;
    skb = kb <= jmax ? __ldg(&p.k_scale[row0 + (int64_t)kb * p.H_kv]) : 0.f;
  }
  // query fragments: head nt 8 + gq, d = 32 j + 8 tq + 0..7 (zero for heads >= G)
  uint4 bq[NT][NP];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int h = nt * 8 + gq;
    const uint4* qrow =
        reinterpret_cast<const uint4*>(p.q + ((int64_t)b * p.H_kv * G + (int64_t)g * G + h) * D);
#pragma unroll
    for (int j = 0; j < NP; ++j) bq[nt][j] = h < G ? __ldg(&qrow[4 * j + tq]) : make_uint4(0, 0, 0, 0);
  }
  if constexpr (F8) {  // widen the staged V rows and keep their scales
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int x = threadIdx.x + u * 256;
      const int r = x / CH, ch = x % CH;
      const uint32_t vv[4] = {vw[u].x, vw[u].y, vw[u].z, vw[u].w};
      uint32_t vo[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const __nv_fp8x2_storage_t v2 = (__nv_fp8x2_storage_t)(vv[e >> 1] >> (16 * (e & 1)));
        const float2 vf = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(v2, __NV_E4M3)));
        vo[e] = pack_bf16(vf.x, vf.y);
      }
      uint4* vd = reinterpret_cast<uint4*>(sV + r * KS + ch * 16);
      vd[0] = make_uint4(vo[0], vo[1], vo[2], vo[3]);
      vd[1] = make_uint4(vo[4], vo[5], vo[6], vo[7]);
    }
    for (int r = threadIdx.x; r < 128; r += blockDim.x)
      s_sv[r] = r <= jmax ? __ldg(&p.v_scale[row0 + (int64_t)r * p.H_kv]) : 0.f;
  }
  // ---- scores ----
  float sc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      const uint32_t a0[4] = {wa[j].x, wb[j].x, wa[j].y, wb[j].y};
      const uint32_t a1[4] = {wa[j].z, wb[j].z, wa[j].w, wb[j].w};
      mma_bf16_16816(sc[nt], a0, bq[nt][j].x, bq[nt][j].y);
      mma_bf16_16816(sc[nt], a1, bq[nt][j].z, bq[nt][j].w);
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int h = nt * 8 + 2 * tq + (e & 1), r = (e >> 1) ? kb : ka;
      const float raw = F8 ? sc[nt][e] * ((e >> 1) ? skb : ska) : sc[nt][e];
      sS[h * 128 + r] = r <= jmax ? raw * p.scale : -INFINITY;
    }
  if constexpr (!F8) cp_async_wait<0>();  // V landed
  __syncthreads();
  // per head: max, exp, sum (one warp per head); padding heads get P = 0
  for (int h = warp; h < 8 * NT; h += 8) {
    if (h >= G) {
      for (int r = lane; r < PS; r += 32) sP[h * PS + r] = __float2bfloat16(0.f);
      continue;
    }
    float v[4], m = -INFINITY;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[i] = sS[h * 128 + lane + 32 * i];
      m = fmaxf(m, v[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float l = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float e = expf(v[i] - m);  // masked: exp(-inf) = 0
      // FP8 cache: the V row scale folds into P (o = sum_j e_j s_j v8_j / l)
      sP[h * PS + lane + 32 * i] = __float2bfloat16(F8 ? e * s_sv[lane + 32 * i] : e);
      l += e;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) {
      s_l[h] = l;
      p.lse_part[part + h] = m + logf(l);
    }
  }
  __syncthreads();
  if (warp < D / 16) {
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    const int mi = lane >> 3, ri = lane & 7;
    // ldmatrix.trans of V rows (keys) gives the A fragment of V^T: matrix mi covers
    // keys (mi >> 1) * 8 + 0..7 and columns dd = 16 warp + (mi & 1) * 8 + 0..7
    const __nv_bfloat16* vrow = sV + ((mi >> 1) * 8 + ri) * KS + warp * 16 + (mi & 1) * 8;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t a[4];
      ldmatrix_x4_trans(a, vrow + ks * 16 * KS);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const __nv_bfloat16* prow = sP + (nt * 8 + gq) * PS + ks * 16 + 2 * tq;
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(prow);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(prow + 8);
        mma_bf16_16816(acc[nt], a, b0, b1);
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int h = nt * 8 + 2 * tq + (e & 1), dd = warp * 16 + gq + (e >> 1) * 8;
        if (h < G) p.o_part[(part + h) * D + dd] = acc[nt][e] / s_l[h];
      }
  }
}

// o[b][g G + h] and lse[b][g G + h] for every head of group g from the group's k
// partials (log-sum-exp merge).  The filled slots come first (block ids ascending, then
// -1 padding with lse = -inf).  Run by one CTA after all partials are written; reads
// them through L2, every slot's load of an output element issued together.
__device__ __forceinline__ void combine_group(const DecodeParams& p, int b, int g, float* s_w) {
  const int G = p.G, K = p.topk;
  const int64_t base = ((int64_t)b * p.H_kv + g) * K;
  const int64_t head0 = (int64_t)b * p.H_kv * G + (int64_t)g * G;
  __shared__ int s_n;
  for (int i = threadIdx.x; i < K * G; i += blockDim.x) s_w[i] = __ldcg(&p.lse_part[base * G + i]);
  __syncthreads();
  for (int h = threadIdx.x; h < G; h += blockDim.x) {
    int n = 0;
    float m = -INFINITY;
    for (int s = 0; s < K; ++s) {
      const float ls = s_w[s * G + h];
      if (ls != -INFINITY) n = s + 1;
      m = fmaxf(m, ls);
    }
    float l = 0.f;
    for (int s = 0; s < n; ++s) l += expf(s_w[s * G + h] - m);
    for (int s = 0; s < n; ++s) s_w[s * G + h] = expf(s_w[s * G + h] - m) / l;
    p.lse[head0 + h] = m + logf(l);
    if (h == 0) s_n = n;
  }
  __syncthreads();
  const int n = s_n;  // the same for every head: the group's filled slots
  const float* op = p.o_part + base * G * p.d;
  for (int x = threadIdx.x; x < G * p.d; x += blockDim.x) {
    const int h = x / p.d;
    float acc = 0.f;
#pragma unroll 8
    for (int s = 0; s < n; ++s) acc = fmaf(s_w[s * G + h], __ldcg(&op[(int64_t)s * G * p.d + x]), acc);
    p.o[head0 * p.d + x] = __float2bfloat16(acc);
  }
}

// Grid (topk, H_kv, B), 256 threads: CTA (s, g, b) computes the partial of slot s of
// group g; the last of the group's topk CTAs to finish (an arrival count that the
// selection kernel zeroed) merges the group's partials into o and lse.
template <int D, int NT, bool F8>
__global__ void __launch_bounds__(256) decode_attn_kernel(const DecodeParams p) {
  extern __shared__ __align__(16) uint8_t dsm[];
  __shared__ float s_l[8 * NT];
  __shared__ float s_sv[F8 ? 128 : 1];  // FP8 V row scales
  __shared__ float s_w[32 * 16];  // [topk][G] merge weights
  __shared__ int s_last;
  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int L = seq_len(p, b, p.status);  // an input: read while the selection finishes
  griddep_wait();  // the selection and its zeroed arrival counts
  const int64_t part = (((int64_t)b * p.H_kv + g) * p.topk + s) * p.G;
  const int c = __ldg(&p.block_idx[((int64_t)b * p.H_kv + g) * p.topk + s]);
  if (c < 0) {
    for (int h = threadIdx.x; h < p.G; h += blockDim.x) p.lse_part[part + h] = -INFINITY;
  } else {
    block_partial<D, NT, F8>(p, dsm, part, c, b, g, L, s_l, s_sv);
  }
  __threadfence();  // this CTA's partial is visible before its arrival
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&p.arrive[(int64_t)b * p.H_kv + g], 1) == p.topk - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  combine_group(p, b, g, s_w);
}

size_t decode_ws_parts(const Shape& s, size_t* off_pooled, size_t* off_o, size_t* off_lse,
                       size_t* off_arrive) {
  const int nbm = s.nb;
  size_t off = 0;
  *off_pooled = off;
  off += align256((size_t)s.B * s.H_kv * (nbm > 0 ? nbm : 1) * 4);
  *off_o = off;
  off += align256((size_t)s.B * s.H_kv * s.topk * s.G * s.d * 4);
  *off_lse = off;
  off += align256((size_t)s.B * s.H_kv * s.topk * s.G * 4);
  *off_arrive = off;
  off += align256((size_t)s.B * s.H_kv * 4);
  return off;
}

// E4M3 codes and per-row scales of a [rows][D] bf16 tensor (the FP8 KV cache): one
// warp per row; scale = amax / 448 (1 for an all-zero row), code = nearest E4M3 value
// of x / scale with ties to even and saturation at 448.  Both divisions are IEEE
// round-to-nearest so the codes are reproducible bit for bit.
template <int D>
__global__ void __launch_bounds__(256) quantize_fp8_kernel(const __nv_bfloat16* __restrict__ x,
                                                            uint8_t* __restrict__ x8,
                                                            float* __restrict__ scale,
                                                            int64_t rows) {
  constexpr int E = D / 32;  // values per lane
  const int lane = threadIdx.x & 31;
  const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (row >= rows) return;
  float v[E];
  const __nv_bfloat16* src = x + row * D + lane * E;
  if constexpr (E == 4) {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(src));
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&w.x);
    const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&w.y);
    v[0] = __low2float(a); v[1] = __high2float(a); v[2] = __low2float(c); v[3] = __high2float(c);
  } else {
    const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(src));
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&w);
    v[0] = __low2float(a); v[1] = __high2float(a);
  }
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(v[e]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float sc = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  uint32_t packed = 0;
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    const float2 f = make_float2(__fdiv_rn(v[e], sc), __fdiv_rn(v[e + 1], sc));
    const uint32_t two = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
    packed |= (two & 0xFFFFu) << (8 * e);
  }
  uint8_t* dst = x8 + row * D + lane * E;
  if constexpr (E == 4) *reinterpret_cast<uint32_t*>(dst) = packed;
  else *reinterpret_cast<uint16_t*>(dst) = (uint16_t)packed;
  if (lane == 0) scale[row] = sc;
}

// The cache a decode call reads: bf16 k, v, or E4M3 codes with their row scales.
struct DecodeCache {
  const void* k;
  const void* v;
  const uint8_t* k8;
  const uint8_t* v8;
  const float* k_scale;
  const float* v_scale;
};

// Shared driver of msa_decode and msa_decode_fp8: index pooling and selection
// (bf16 index branch), then the split attention over the selected blocks.
// Launches a kernel of this file with programmatic stream serialization: it may be
// scheduled while the previous kernel in the stream drains, and waits for that kernel
// (griddep_wait) before reading what it wrote.
template <typename Kern>
cudaError_t launch_after(Kern kern, dim3 grid, size_t smem, cudaStream_t stream,
                         const DecodeParams& dp) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, dp);
}

int run_decode(const msa_problem_t* p, const void* q, const void* q_idx, const DecodeCache& kv,
               const void* k_idx, const int32_t* lens, int32_t* block_idx, void* o, float* lse,
               void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  Shape s;
  int rc = validate_problem(p, &s);
  if (rc) return rc;
  if (s.B == 0) return MSA_OK;
  if (s.N == 0) return MSA_ERR_SHAPE;  // N is the cache capacity Lmax
  if (s.topk > kMaxSelect) return MSA_ERR_UNSUPPORTED;
  const bool f8 = kv.k8 != nullptr;
  const void* ptrs[] = {q, q_idx, f8 ? (const void*)kv.k8 : kv.k, f8 ? (const void*)kv.v8 : kv.v,
                        k_idx, lens, block_idx, o, lse};
  for (const void* x : ptrs)
    if (!x || (reinterpret_cast<uintptr_t>(x) & 15) != 0) return MSA_ERR_ARG;
  if (f8 && ((reinterpret_cast<uintptr_t>(kv.k_scale) & 3) || (reinterpret_cast<uintptr_t>(kv.v_scale) & 3)))
    return MSA_ERR_ARG;
  size_t off_pooled, off_o, off_lse, off_arrive;
  const size_t need = decode_ws_parts(s, &off_pooled, &off_o, &off_lse, &off_arrive);
  if (!workspace || workspace_bytes < need) return MSA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return MSA_ERR_ARG;
  Ctx cx;
  if ((rc = device_ctx(&cx))) return rc;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  DecodeParams dp;
  dp.q = static_cast<const __nv_bfloat16*>(q);
  dp.q_idx = static_cast<const __nv_bfloat16*>(q_idx);
  dp.k = static_cast<const __nv_bfloat16*>(kv.k);
  dp.v = static_cast<const __nv_bfloat16*>(kv.v);
  dp.k8 = kv.k8;
  dp.v8 = kv.v8;
  dp.k_scale = kv.k_scale;
  dp.v_scale = kv.v_scale;
  dp.k_idx = static_cast<const __nv_bfloat16*>(k_idx);
  dp.lens = lens;
  dp.block_idx = block_idx;
  dp.pooled = reinterpret_cast<float*>(w + off_pooled);
  dp.o_part = reinterpret_cast<float*>(w + off_o);
  dp.lse_part = reinterpret_cast<float*>(w + off_lse);
  dp.arrive = reinterpret_cast<int*>(w + off_arrive);
  dp.o = static_cast<__nv_bfloat16*>(o);
  dp.lse = lse;
  dp.B = s.B;
  dp.Lmax = s.N;
  dp.H_kv = s.H_kv;
  dp.G = s.G;
  dp.d = s.d;
  dp.d_idx = s.d_idx;
  dp.topk = s.topk;
  dp.nbm = s.nb;
  dp.scale = s.scale;
  dp.status = cx.status;
  const int pool_nt = s.H_kv > 8 ? 2 : 1;
  const dim3 gpool((unsigned)((s.nb + 7) / 8), (unsigned)s.B,
                   (unsigned)((s.H_kv + 8 * pool_nt - 1) / (8 * pool_nt)));
#define MSA_POOL(DI, NT) decode_pool_kernel<DI, NT><<<gpool, 256, 0, stream>>>(dp)
  if (s.d_idx == 64) {
    if (pool_nt == 1) MSA_POOL(64, 1); else MSA_POOL(64, 2);
  } else {
    if (pool_nt == 1) MSA_POOL(32, 1); else MSA_POOL(32, 2);
  }
#undef MSA_POOL
  note_launch();
  const dim3 gsel((unsigned)s.H_kv, (unsigned)s.B);
  cudaError_t e = s.topk - 1 <= 15 ? launch_after(decode_select_kernel<15>, gsel, 0, stream, dp)
                                   : launch_after(decode_select_kernel<31>, gsel, 0, stream, dp);
  if (e != cudaSuccess) return MSA_ERR_CUDA;
  note_launch();
  const int attn_nt = s.G <= 8 ? 1 : 2;
  const size_t attn_smem = (size_t)128 * (s.d + 8) * 2 + (size_t)8 * attn_nt * 128 * 4 +
                           (size_t)8 * attn_nt * (128 + 8) * 2;
  const dim3 gattn((unsigned)s.topk, (unsigned)s.H_kv, (unsigned)s.B);
#define MSA_ATTN(D, NT, F8)                                                                   \
  do {                                                                                        \
    e = cudaFuncSetAttribute(decode_attn_kernel<D, NT, F8>,                                   \
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)attn_smem);    \
    if (e == cudaSuccess)                                                                     \
      e = launch_after(decode_attn_kernel<D, NT, F8>, gattn, attn_smem, stream, dp);          \
  } while (0)
  if (f8) {
    if (s.d == 128) {
      if (s.G <= 8) MSA_ATTN(128, 1, true); else MSA_ATTN(128, 2, true);
    } else {
      if (s.G <= 8) MSA_ATTN(64, 1, true); else MSA_ATTN(64, 2, true);
    }
  } else {
    if (s.d == 128) {
      if (s.G <= 8) MSA_ATTN(128, 1, false); else MSA_ATTN(128, 2, false);
    } else {
      if (s.G <= 8) MSA_ATTN(64, 1, false); else MSA_ATTN(64, 2, false);
    }
  }
#undef MSA_ATTN
  if (e != cudaSuccess) return MSA_ERR_CUDA;
  note_launch();
  return cudaGetLastError() == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" {

size_t msa_decode_workspace_size(const msa_problem_t* p) {
  Shape s;
  if (validate_problem(p, &s) != MSA_OK) return 0;
  size_t a, b, c, d;
  return decode_ws_parts(s, &a, &b, &c, &d);
}

int msa_decode(const msa_problem_t* p, const void* q, const void* q_idx, const void* k,
               const void* v, const void* k_idx, const int32_t* lens, int32_t* block_idx, void* o,
               float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  DecodeCache kv = {k, v, nullptr, nullptr, nullptr, nullptr};
  return run_decode(p, q, q_idx, kv, k_idx, lens, block_idx, o, lse, workspace, workspace_bytes,
                    stream);
}

int msa_decode_fp8(const msa_problem_t* p, const void* q, const void* q_idx, const uint8_t* k8,
                   const uint8_t* v8, const float* k_scale, const float* v_scale, const void* k_idx,
                   const int32_t* lens, int32_t* block_idx, void* o, float* lse, void* workspace,
                   size_t workspace_bytes, cudaStream_t stream) {
  if (!k8 || !v8 || !k_scale || !v_scale) return MSA_ERR_ARG;
  DecodeCache kv = {nullptr, nullptr, k8, v8, k_scale, v_scale};
  return run_decode(p, q, q_idx, kv, k_idx, lens, block_idx, o, lse, workspace, workspace_bytes,
                    stream);
}

int msa_quantize_kv_fp8(const msa_problem_t* p, const void* x, uint8_t* x8, float* scale,
                        cudaStream_t stream) {
  // only the cache's sizes matter here: B, N (capacity), H_kv, d
  if (!p) return MSA_ERR_ARG;
  if (p->B < 0 || p->N < 0 || p->H_kv <= 0) return MSA_ERR_SHAPE;
  if (p->d != 64 && p->d != 128) return MSA_ERR_UNSUPPORTED;
  const int64_t rows = (int64_t)p->B * p->N * p->H_kv;
  if (rows == 0) return MSA_OK;
  if (rows > ((int64_t)1 << 40)) return MSA_ERR_UNSUPPORTED;
  const void* ptrs[] = {x, x8, scale};
  for (const void* t : ptrs)
    if (!t || (reinterpret_cast<uintptr_t>(t) & 15) != 0) return MSA_ERR_ARG;
  const int64_t blocks = (rows + 7) / 8;
  if (blocks > 0x7fffffffLL) return MSA_ERR_UNSUPPORTED;
  const unsigned grid = (unsigned)blocks;
  if (p->d == 128)
    quantize_fp8_kernel<128><<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(x), x8,
                                                        scale, rows);
  else
    quantize_fp8_kernel<64><<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(x), x8,
                                                       scale, rows);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

}  // extern "C"
