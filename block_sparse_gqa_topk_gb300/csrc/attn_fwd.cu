// attn_fwd.cu -- main-branch block-sparse forward and the index-LSE recompute.
//
// Both are the same gathered, KV-outer computation over the inverted lists built by
// plan.cu: a tile is one key block c of one (batch, group) and up to 128 rows, a
// row being a (query, head) pair of the queries whose set holds c.
//   main (MSA summary, 7minutos.es, "Cómo funcionan las dos ramas" ¶3): rows are
//     the G query heads of up to 128/G queries; S = scale Q K_c^T over the block's
//     causally visible tokens, the tile's softmax partial (normalised o, lse) is
//     written per (query, slot, head) and a combine kernel merges the k partials
//     of each row into o and the saved lse (Flash-MSA article, tech.kuratif.com,
//     ¶6); the two-phase split/combine is fmha_sm100's ("El codiseño del kernel").
//   index LSE (deephorus.pages.dev ¶4: recomputed cheaply, not fused with the
//     top-k): rows are single queries of the group's index head, S = scale_idx
//     q_idx k_idx^T, only the partial lse is written, then combined.
// Tiles are contiguous per CTA so that consecutive tiles of the same key block
// reuse the K/V tile; loads are cp.async into XOR-swizzled smem, double-buffered
// across tiles; the contractions use mma.sync m16n8k16 (bf16 in, fp32 accumulate).
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace msa {
namespace {

constexpr int kFwdThreads = 256;  // 8 warps x 16 rows

struct GatherParams {
  const __nv_bfloat16* q;  // row source: q (main) or q_idx (index)
  const __nv_bfloat16* k;  // k (main) or k_idx (index)
  const __nv_bfloat16* v;  // main only
  const int* off;
  const int* toff;
  const int* entries;
  __nv_bfloat16* o_part;  // main only: [(row_kv*topk + slot)*G + h][D]
  float* lse_part;        // [(row_kv*topk + slot)*G + h]
  int64_t keys;
  int N, H_kv, nb, topk, causal;
  int q_tok_stride;  // elements between consecutive tokens of the row source
  int k_tok_stride;  // elements between consecutive tokens of k (and v)
  int k_shared;      // 1: one k head for all groups (index branch)
  float scale_log2;  // softmax scale * log2(e)
};

__device__ __forceinline__ int find_key(const int* __restrict__ toff, int64_t keys, int t) {
  // largest key with toff[key] <= t (toff is non-decreasing, toff[keys] > t)
  int64_t lo = 0, hi = keys - 1;
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) >> 1;
    if (__ldg(&toff[mid]) <= t) lo = mid; else hi = mid - 1;
  }
  return (int)lo;
}

template <int D, int G, bool MAIN>
struct FwdSmem {
  static constexpr int kRowB = D * 2;
  static constexpr int kTileB = 128 * kRowB;
  static constexpr int kBuf = (MAIN ? 3 : 2) * kTileB;  // K, (V), Q
  static constexpr int kBytes = 2 * kBuf + 2 * 128 * 4;  // + per-row entry cache
};

template <int D, int G, bool MAIN>
__global__ void __launch_bounds__(kFwdThreads, 1) gather_fwd_kernel(const GatherParams p) {
  using L = FwdSmem<D, G, MAIN>;
  constexpr int QPT = 128 / G;
  constexpr int RB = L::kRowB;
  constexpr int CH = D / 8;  // 16-byte chunks per row
  extern __shared__ __align__(128) uint8_t smem[];
  int* s_ent = reinterpret_cast<int*>(smem + 2 * L::kBuf);  // [2][128] packed entries / -1

  const int total = __ldg(&p.toff[p.keys]);
  const int per = (total + gridDim.x - 1) / gridDim.x;
  const int t_begin = blockIdx.x * per;
  const int t_end = min(total, t_begin + per);
  if (t_begin >= t_end) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int key_in[2] = {-1, -1};

  // issue the loads of tile t into buffer slot `sl`
  auto load_tile = [&](int t, int sl) {
    uint8_t* buf = smem + sl * L::kBuf;
    uint8_t* sK = buf;
    uint8_t* sV = buf + L::kTileB;
    uint8_t* sQ = buf + (MAIN ? 2 : 1) * L::kTileB;
    const int key = find_key(p.toff, p.keys, t);
    const int bg = key / p.nb, c = key - bg * p.nb;
    const int b = bg / p.H_kv, g = bg - b * p.H_kv;
    const int e0 = __ldg(&p.off[key]) + (t - __ldg(&p.toff[key])) * QPT;
    const int ne = min(QPT, __ldg(&p.off[key + 1]) - e0);
    if (key_in[sl] != key) {
      key_in[sl] = key;
      const int koff = p.k_shared ? 0 : g * D;
      for (int x = threadIdx.x; x < 128 * CH; x += kFwdThreads) {
        const int r = x / CH, ch = x % CH;
        const int j = c * 128 + r;
        const bool ok = j < p.N;
        const int64_t src = ((int64_t)b * p.N + (ok ? j : 0)) * p.k_tok_stride + koff + ch * 8;
        cp_async_16(sK + swz<RB>(r, ch), p.k + src, ok);
        if (MAIN) cp_async_16(sV + swz<RB>(r, ch), p.v + src, ok);
      }
    }
    int* ent = s_ent + sl * 128;
    for (int x = threadIdx.x; x < 128 * CH; x += kFwdThreads) {
      const int r = x / CH, ch = x % CH;
      const int qi = r / G, h = r % G;
      const bool ok = qi < ne;
      int i = 0;
      if (ok) i = __ldg(&p.entries[e0 + qi]) >> 5;
      const int64_t src = ((int64_t)b * p.N + i) * p.q_tok_stride + (int64_t)(g * G + h) * D + ch * 8;
      cp_async_16(sQ + swz<RB>(r, ch), p.q + src, ok);
    }
    if (threadIdx.x < 128) {
      const int qi = threadIdx.x / G;
      ent[threadIdx.x] = qi < ne ? __ldg(&p.entries[e0 + qi]) : -1;
    }
    cp_async_commit();
    return key;
  };

  int cur_key = load_tile(t_begin, 0);
  for (int t = t_begin; t < t_end; ++t) {
    const int sl = (t - t_begin) & 1;
    int nxt_key = -1;
    if (t + 1 < t_end) {
      // the other slot was last read by tile t-1; all threads passed the barrier
      nxt_key = load_tile(t + 1, sl ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();

    const uint8_t* buf = smem + sl * L::kBuf;
    const uint8_t* sK = buf;
    const uint8_t* sV = buf + L::kTileB;
    const uint8_t* sQ = buf + (MAIN ? 2 : 1) * L::kTileB;
    const int* ent = s_ent + sl * 128;
    const int key = cur_key;
    const int bg = key / p.nb, c = key - bg * p.nb;

    // ---- S = Q K^T for this warp's 16 rows ----
    float acc[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    const int r0 = warp * 16;
#pragma unroll
    for (int kc = 0; kc < D / 16; ++kc) {
      uint32_t a[4];
      ldmatrix_x4(a, sQ + swz<RB>(r0 + (lane & 15), kc * 2 + (lane >> 4)));
#pragma unroll
      for (int n2 = 0; n2 < 8; ++n2) {  // pairs of 8-key tiles
        uint32_t bf[4];
        const int krow = n2 * 16 + (lane & 7) + ((lane >> 4) << 3);
        ldmatrix_x4(bf, sK + swz<RB>(krow, kc * 2 + ((lane >> 3) & 1)));
        mma_bf16_16816(acc[2 * n2], a, bf[0], bf[1]);
        mma_bf16_16816(acc[2 * n2 + 1], a, bf[2], bf[3]);
      }
    }

    // ---- masked softmax of the two rows this thread holds ----
    const int ra = r0 + (lane >> 2), rb = ra + 8;
    const int enta = ent[ra], entb = ent[rb];
    const int ia = enta >= 0 ? (enta >> 5) : -1;
    const int ib = entb >= 0 ? (entb >> 5) : -1;
    const int jbase = c * 128 + (lane & 3) * 2;
    float ma = -INFINITY, mb = -INFINITY;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int j = jbase + n * 8 + e;
        const bool va = ia >= 0 && j < p.N && (!p.causal || j <= ia);
        const bool vb = ib >= 0 && j < p.N && (!p.causal || j <= ib);
        acc[n][e] = va ? acc[n][e] * p.scale_log2 : -INFINITY;
        acc[n][2 + e] = vb ? acc[n][2 + e] * p.scale_log2 : -INFINITY;
        ma = fmaxf(ma, acc[n][e]);
        mb = fmaxf(mb, acc[n][2 + e]);
      }
    }
    ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 1));
    ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 2));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
    const float msa_ = ma == -INFINITY ? 0.f : ma;  // empty rows stay all-zero
    const float msb_ = mb == -INFINITY ? 0.f : mb;
    float la = 0.f, lb = 0.f;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        acc[n][e] = exp2f(acc[n][e] - msa_);
        acc[n][2 + e] = exp2f(acc[n][2 + e] - msb_);
        la += acc[n][e];
        lb += acc[n][2 + e];
      }
    }
    la += __shfl_xor_sync(0xffffffffu, la, 1);
    la += __shfl_xor_sync(0xffffffffu, la, 2);
    lb += __shfl_xor_sync(0xffffffffu, lb, 1);
    lb += __shfl_xor_sync(0xffffffffu, lb, 2);
    constexpr float kLn2 = 0.6931471805599453f;
    const int64_t slot_a = enta >= 0 ? (((int64_t)bg * p.N + ia) * p.topk + (enta & 31)) : -1;
    const int64_t slot_b = entb >= 0 ? (((int64_t)bg * p.N + ib) * p.topk + (entb & 31)) : -1;
    const int ha = ra % G, hb = rb % G;

    if (MAIN) {
      // ---- O = P V, normalised by l ----
      float o[D / 8][4];
#pragma unroll
      for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
#pragma unroll
      for (int kc = 0; kc < 8; ++kc) {  // 16 keys per step
        uint32_t a[4];
        a[0] = pack_bf16(acc[2 * kc][0], acc[2 * kc][1]);
        a[1] = pack_bf16(acc[2 * kc][2], acc[2 * kc][3]);
        a[2] = pack_bf16(acc[2 * kc + 1][0], acc[2 * kc + 1][1]);
        a[3] = pack_bf16(acc[2 * kc + 1][2], acc[2 * kc + 1][3]);
#pragma unroll
        for (int n2 = 0; n2 < D / 16; ++n2) {
          uint32_t bf[4];
          const int vrow = kc * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
          ldmatrix_x4_trans(bf, sV + swz<RB>(vrow, n2 * 2 + (lane >> 4)));
          mma_bf16_16816(o[2 * n2], a, bf[0], bf[1]);
          mma_bf16_16816(o[2 * n2 + 1], a, bf[2], bf[3]);
        }
      }
      const float inva = la > 0.f ? 1.f / la : 0.f;
      const float invb = lb > 0.f ? 1.f / lb : 0.f;
      __nv_bfloat16* pa = slot_a >= 0 ? p.o_part + (slot_a * G + ha) * D : nullptr;
      __nv_bfloat16* pb = slot_b >= 0 ? p.o_part + (slot_b * G + hb) * D : nullptr;
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        const int d0 = n * 8 + (lane & 3) * 2;
        if (pa) *reinterpret_cast<uint32_t*>(pa + d0) = pack_bf16(o[n][0] * inva, o[n][1] * inva);
        if (pb) *reinterpret_cast<uint32_t*>(pb + d0) = pack_bf16(o[n][2] * invb, o[n][3] * invb);
      }
    }
    if ((lane & 3) == 0) {
      if (slot_a >= 0) p.lse_part[slot_a * G + ha] = la > 0.f ? (msa_ + log2f(la)) * kLn2 : -INFINITY;
      if (slot_b >= 0) p.lse_part[slot_b * G + hb] = lb > 0.f ? (msb_ + log2f(lb)) * kLn2 : -INFINITY;
    }
    __syncthreads();  // slot sl is free for tile t+2
    cur_key = nxt_key;
  }
}

// o[b,i,h] and lse[b,h,i] from the k partials of each (b, g, i) row.  One warp per
// row: the partials of one slot are G*D contiguous bf16 (all heads of the group), read
// as 16-byte chunks; the per-(slot, head) weights exp(lse_s - lse) come from shared
// memory, computed by G lanes.
template <int D, int G>
__global__ void __launch_bounds__(256) fwd_combine_kernel(
    const __nv_bfloat16* __restrict__ o_part, const float* __restrict__ lse_part,
    const int32_t* __restrict__ block_idx, __nv_bfloat16* __restrict__ o,
    float* __restrict__ lse, int64_t rows, int N, int H_kv, int topk, int nb) {
  constexpr int TC = G * D / 8;              // 16-byte chunks per slot
  constexpr int CPL = (TC + 31) / 32;        // chunks per lane
  __shared__ float wts[8][32 * G];
  const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rkv = (int64_t)blockIdx.x * 8 + wib;  // (b*H_kv + g)*N + i
  if (rkv >= rows) return;
  const int i = (int)(rkv % N);
  const int64_t bg = rkv / N;
  const int g = (int)(bg % H_kv);
  const int64_t b = bg / H_kv;
  const int32_t* sel = block_idx + rkv * topk;
  float* w = wts[wib];
  if (lane < G) {
    const int h = lane;
    float m = -INFINITY;
    for (int s = 0; s < topk; ++s) {
      const int c = __ldg(&sel[s]);
      if (c >= 0 && c < nb) m = fmaxf(m, __ldg(&lse_part[(rkv * topk + s) * G + h]));
    }
    float l = 0.f;
    for (int s = 0; s < topk; ++s) {
      const int c = __ldg(&sel[s]);
      const float ls = (c >= 0 && c < nb) ? __ldg(&lse_part[(rkv * topk + s) * G + h]) : -INFINITY;
      const float e = ls == -INFINITY ? 0.f : __expf(ls - m);
      w[s * G + h] = e;
      l += e;
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    for (int s = 0; s < topk; ++s) w[s * G + h] *= inv;
    lse[(b * H_kv * G + g * G + h) * N + i] = m + logf(l);
  }
  __syncwarp();
  float acc[CPL][8];
#pragma unroll
  for (int x = 0; x < CPL; ++x)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[x][e] = 0.f;
  for (int s = 0; s < topk; ++s) {
    const int c = __ldg(&sel[s]);
    if (c < 0 || c >= nb) continue;  // same for every lane
    const uint4* src = reinterpret_cast<const uint4*>(o_part + (rkv * topk + s) * G * D);
#pragma unroll
    for (int x = 0; x < CPL; ++x) {
      const int ch = lane + 32 * x;
      if (ch < TC) {
        const float wt = w[s * G + (ch * 8) / D];
        const uint4 raw = __ldg(&src[ch]);
        const __nv_bfloat162* pr = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[x][2 * e] += wt * __low2float(pr[e]);
          acc[x][2 * e + 1] += wt * __high2float(pr[e]);
        }
      }
    }
  }
  uint4* dst = reinterpret_cast<uint4*>(o + ((b * N + i) * H_kv * G + (int64_t)g * G) * D);
#pragma unroll
  for (int x = 0; x < CPL; ++x) {
    const int ch = lane + 32 * x;
    if (ch < TC) {
      uint4 out;
      uint32_t* pw = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
      for (int e = 0; e < 4; ++e) pw[e] = pack_bf16(acc[x][2 * e], acc[x][2 * e + 1]);
      dst[ch] = out;
    }
  }
}

// lse_idx[b,g,i] = logsumexp over the row's valid slots of the partial lse.
__global__ void lse_combine_kernel(const float* __restrict__ lse_part,
                                   const int32_t* __restrict__ block_idx,
                                   float* __restrict__ lse_idx, int64_t rows, int topk, int nb) {
  const int64_t r = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (r >= rows) return;
  const int32_t* sel = block_idx + r * topk;
  float m = -INFINITY;
  for (int s = 0; s < topk; ++s)
    if (sel[s] >= 0 && sel[s] < nb) m = fmaxf(m, lse_part[r * topk + s]);
  float l = 0.f;
  for (int s = 0; s < topk; ++s)
    if (sel[s] >= 0 && sel[s] < nb) l += __expf(lse_part[r * topk + s] - m);
  lse_idx[r] = m + logf(l);
}

template <int D, int G, bool MAIN>
cudaError_t launch_gather(const GatherParams& p, const Ctx& cx, cudaStream_t st) {
  using L = FwdSmem<D, G, MAIN>;
  auto kern = gather_fwd_kernel<D, G, MAIN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
  if (e != cudaSuccess) return e;
  kern<<<cx.num_sms, kFwdThreads, L::kBytes, st>>>(p);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_index_lse(const Shape& s, const void* q_idx, const void* k_idx,
                             const int32_t* block_idx, const Plan& pl, float* lse_part,
                             float* lse_idx, const Ctx& cx, cudaStream_t st) {
  GatherParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q_idx);
  p.k = static_cast<const __nv_bfloat16*>(k_idx);
  p.v = nullptr;
  p.off = pl.off;
  p.toff = pl.toff;
  p.entries = pl.entries;
  p.o_part = nullptr;
  p.lse_part = lse_part;
  p.keys = s.keys();
  p.N = s.N;
  p.H_kv = s.H_kv;
  p.nb = s.nb;
  p.topk = s.topk;
  p.causal = s.causal;
  p.q_tok_stride = s.H_kv * s.d_idx;
  p.k_tok_stride = s.d_idx;
  p.k_shared = 1;
  p.scale_log2 = s.scale_idx * 1.4426950408889634f;
  cudaError_t e = s.d_idx == 64 ? launch_gather<64, 1, false>(p, cx, st)
                                : launch_gather<32, 1, false>(p, cx, st);
  if (e != cudaSuccess) return e;
  const int64_t rows = s.rows_kv();
  lse_combine_kernel<<<(unsigned)((rows + 255) / 256), 256, 0, st>>>(lse_part, block_idx, lse_idx,
                                                                     rows, s.topk, s.nb);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_attn_fwd(const Shape& s, const void* q, const void* k, const void* v,
                            const int32_t* block_idx, const Plan& pl, __nv_bfloat16* o_part,
                            float* lse_part, void* o, float* lse, const Ctx& cx,
                            cudaStream_t st) {
  cudaError_t e = launch_attn_fwd_tc(s, q, k, v, pl, o_part, lse_part, cx, st);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)((s.rows_kv() + 7) / 8);
  __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(o);
#define MSA_COMBINE(DD, GG)                                                                 \
  fwd_combine_kernel<DD, GG><<<grid, 256, 0, st>>>(o_part, lse_part, block_idx, ob, lse,     \
                                                   s.rows_kv(), s.N, s.H_kv, s.topk, s.nb)
  if (s.d == 128) {
    switch (s.G) {
      case 1: MSA_COMBINE(128, 1); break;
      case 2: MSA_COMBINE(128, 2); break;
      case 4: MSA_COMBINE(128, 4); break;
      case 8: MSA_COMBINE(128, 8); break;
      default: MSA_COMBINE(128, 16); break;
    }
  } else {
    switch (s.G) {
      case 1: MSA_COMBINE(64, 1); break;
      case 2: MSA_COMBINE(64, 2); break;
      case 4: MSA_COMBINE(64, 4); break;
      case 8: MSA_COMBINE(64, 8); break;
      default: MSA_COMBINE(64, 16); break;
    }
  }
#undef MSA_COMBINE
  note_launch();
  return cudaGetLastError();
}

}  // namespace msa
