// attn_fwd.cu -- main-branch forward entry: the tcgen05 partial kernel
// (attn_fwd_tc.cu) followed by the combine of the k per-slot partials of every row.
//
// Method: MSA summary (7minutos.es), "Cómo funcionan las dos ramas" ¶3 (exact
// softmax attention over the selected blocks) and "El codiseño del kernel" (the
// two-phase split/combine); Flash-MSA article (tech.kuratif.com) ¶6 (the lse is
// kept for the backward).  Every slot of a row holds a normalised partial o_s and
// its lse_s; the row's output is sum_s exp(lse_s - lse) o_s with
// lse = log sum_s exp(lse_s).
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace msa {
namespace {

// o[b,i,h] and lse[b,h,i] from the k partials of each (b, g, i) row.  One warp per
// row.  The (slot, head) lse partials of the row are contiguous: lane l reads pairs
// l, l + 32, ... at once (head l % G, since G divides 32), and shuffles across the lanes
// of one head give its max and sum; the weights exp(lse_s - lse) go to shared memory.
// The partials of one slot are G*D contiguous bf16 (all heads of the group), read as
// 16-byte chunks, eight loads a lane in flight at a time.  Up to 32 slots.
template <int D, int G>
__global__ void __launch_bounds__(256) fwd_combine_kernel(
    const __nv_bfloat16* __restrict__ o_part, const float* __restrict__ lse_part,
    const int32_t* __restrict__ block_idx, __nv_bfloat16* __restrict__ o,
    float* __restrict__ lse, const int2* __restrict__ spans, int B, int64_t rows, int N, int H_kv,
    int topk, int nb) {
  constexpr int TC = G * D / 8;              // 16-byte chunks per slot
  constexpr int CPL = (TC + 31) / 32;        // chunks per lane
  constexpr int NP = (32 * G + 31) / 32;     // (slot, head) pairs per lane, 32 slots at most
  constexpr int SB = CPL >= 8 ? 1 : 8 / CPL;  // slots in flight: 8 loads per lane
  __shared__ float wts[8][32 * G];
  const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rkv = (int64_t)blockIdx.x * 8 + wib;  // t0*H_kv + g*len + i
  if (rkv >= rows) return;
  RowPos rp;
  if (!row_pos(spans, B, N, H_kv, rkv, &rp)) return;  // tokens outside every sequence
  const int i = rp.i, g = rp.h;
  const SeqSpan sp = rp.sp;
  const int32_t* sel = block_idx + rkv * topk;
  float* w = wts[wib];
  const int npair = topk * G;
  float ls[NP];
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < NP; ++j) {
    const int pr = lane + 32 * j;
    ls[j] = -INFINITY;
    if (pr < npair) {
      const int c = __ldg(&sel[pr / G]);
      if (c >= 0 && c < nb) ls[j] = __ldg(&lse_part[rkv * npair + pr]);
    }
    m = fmaxf(m, ls[j]);
  }
#pragma unroll
  for (int o = G; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float l = 0.f;
#pragma unroll
  for (int j = 0; j < NP; ++j) {
    ls[j] = ls[j] == -INFINITY ? 0.f : __expf(ls[j] - m);
    l += ls[j];
  }
#pragma unroll
  for (int o = G; o < 32; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int j = 0; j < NP; ++j) {
    const int pr = lane + 32 * j;
    if (pr < npair) w[pr] = ls[j] * inv;
  }
  if (lane < G) lse[sp.t0 * H_kv * G + (int64_t)(g * G + lane) * sp.len + i] = m + logf(l);
  __syncwarp();
  float acc[CPL][8];
#pragma unroll
  for (int x = 0; x < CPL; ++x)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[x][e] = 0.f;
  const uint4* src = reinterpret_cast<const uint4*>(o_part + rkv * topk * G * D);
  for (int s0 = 0; s0 < topk; s0 += SB) {
    uint4 raw[SB][CPL];
#pragma unroll
    for (int j = 0; j < SB; ++j) {
      const int s = s0 + j;
      const int c = s < topk ? __ldg(&sel[s]) : -1;
      const bool valid = c >= 0 && c < nb;  // partials of unused slots were never written
#pragma unroll
      for (int x = 0; x < CPL; ++x) {
        const int ch = lane + 32 * x;
        raw[j][x] = (valid && ch < TC) ? __ldg(&src[s * TC + ch]) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int j = 0; j < SB; ++j) {
      const int s = s0 + j;
      if (s >= topk) break;
#pragma unroll
      for (int x = 0; x < CPL; ++x) {
        const int ch = lane + 32 * x;
        if (ch < TC) {
          const float wt = w[s * G + (ch * 8) / D];
          const __nv_bfloat162* pr = reinterpret_cast<const __nv_bfloat162*>(&raw[j][x]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc[x][2 * e] += wt * __low2float(pr[e]);
            acc[x][2 * e + 1] += wt * __high2float(pr[e]);
          }
        }
      }
    }
  }
  uint4* dst = reinterpret_cast<uint4*>(o + ((sp.t0 + i) * H_kv * G + (int64_t)g * G) * D);
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

// The same merge for rows of more than 32 slots (the dense set of the indexer
// warm-up): G lanes find each head's max m and sum l over the slots and lay the
// weights exp(lse_s - m) / l out in shared memory 32 slots at a time (the first 32
// from the sum pass, later ones recomputed).
template <int D, int G>
__global__ void __launch_bounds__(256) fwd_combine_wide_kernel(
    const __nv_bfloat16* __restrict__ o_part, const float* __restrict__ lse_part,
    const int32_t* __restrict__ block_idx, __nv_bfloat16* __restrict__ o,
    float* __restrict__ lse, const int2* __restrict__ spans, int B, int64_t rows, int N, int H_kv,
    int topk, int nb) {
  constexpr int TC = G * D / 8;              // 16-byte chunks per slot
  constexpr int CPL = (TC + 31) / 32;        // chunks per lane
  __shared__ float wts[8][32 * G];
  const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rkv = (int64_t)blockIdx.x * 8 + wib;  // t0*H_kv + g*len + i
  if (rkv >= rows) return;
  RowPos rp;
  if (!row_pos(spans, B, N, H_kv, rkv, &rp)) return;  // tokens outside every sequence
  const int i = rp.i, g = rp.h;
  const SeqSpan sp = rp.sp;
  const int32_t* sel = block_idx + rkv * topk;
  float* w = wts[wib];
  float m = -INFINITY, inv = 0.f;
  if (lane < G) {
    const int h = lane;
    for (int s = 0; s < topk; ++s) {
      const int c = __ldg(&sel[s]);
      if (c >= 0 && c < nb) m = fmaxf(m, __ldg(&lse_part[(rkv * topk + s) * G + h]));
    }
    float l = 0.f;
    for (int s = 0; s < topk; ++s) {
      const int c = __ldg(&sel[s]);
      const float ls = (c >= 0 && c < nb) ? __ldg(&lse_part[(rkv * topk + s) * G + h]) : -INFINITY;
      const float e = ls == -INFINITY ? 0.f : __expf(ls - m);
      if (s < 32) w[s * G + h] = e;  // the first chunk's weights, scaled below
      l += e;
    }
    inv = l > 0.f ? 1.f / l : 0.f;
    for (int s = 0; s < min(32, topk); ++s) w[s * G + h] *= inv;
    lse[sp.t0 * H_kv * G + (int64_t)(g * G + h) * sp.len + i] = m + logf(l);
  }
  float acc[CPL][8];
#pragma unroll
  for (int x = 0; x < CPL; ++x)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[x][e] = 0.f;
  for (int s0 = 0; s0 < topk; s0 += 32) {
    const int ns = min(32, topk - s0);
    __syncwarp();  // the previous chunk's weights are consumed
    if (s0 > 0 && lane < G) {  // slots beyond the first 32 (the dense set only)
      const int h = lane;
      for (int t = 0; t < ns; ++t) {
        const int c = __ldg(&sel[s0 + t]);
        const float ls =
            (c >= 0 && c < nb) ? __ldg(&lse_part[(rkv * topk + s0 + t) * G + h]) : -INFINITY;
        w[t * G + h] = ls == -INFINITY ? 0.f : __expf(ls - m) * inv;
      }
    }
    __syncwarp();
    for (int t = 0; t < ns; ++t) {
      const int s = s0 + t;
      const int c = __ldg(&sel[s]);
      if (c < 0 || c >= nb) continue;  // same for every lane
      const uint4* src = reinterpret_cast<const uint4*>(o_part + (rkv * topk + s) * G * D);
#pragma unroll
      for (int x = 0; x < CPL; ++x) {
        const int ch = lane + 32 * x;
        if (ch < TC) {
          const float wt = w[t * G + (ch * 8) / D];
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
  }
  uint4* dst = reinterpret_cast<uint4*>(o + ((sp.t0 + i) * H_kv * G + (int64_t)g * G) * D);
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

}  // namespace

cudaError_t launch_attn_fwd(const Shape& s, const void* q, const void* k, const void* v,
                            const int32_t* block_idx, const Plan& pl, __nv_bfloat16* o_part,
                            float* lse_part, void* o, float* lse, const Ctx& cx,
                            cudaStream_t st) {
  cudaError_t e = launch_attn_fwd_tc(s, q, k, v, pl, o_part, lse_part, cx, st);
  if (e != cudaSuccess) return e;
  return launch_attn_fwd_combine(s, block_idx, o_part, lse_part, o, lse, st);
}

cudaError_t launch_attn_fwd_combine(const Shape& s, const int32_t* block_idx,
                                    const __nv_bfloat16* o_part, const float* lse_part, void* o,
                                    float* lse, cudaStream_t st) {
  const unsigned grid = (unsigned)((s.rows_kv() + 7) / 8);
  __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(o);
#define MSA_COMBINE(DD, GG)                                                                   \
  do {                                                                                         \
    if (s.topk <= 32)                                                                          \
      fwd_combine_kernel<DD, GG><<<grid, 256, 0, st>>>(o_part, lse_part, block_idx, ob, lse,   \
                                                       s.spans, s.B, s.rows_kv(), s.N, s.H_kv, \
                                                       s.topk, s.nb);                          \
    else                                                                                       \
      fwd_combine_wide_kernel<DD, GG><<<grid, 256, 0, st>>>(o_part, lse_part, block_idx, ob,   \
                                                            lse, s.spans, s.B, s.rows_kv(),    \
                                                            s.N, s.H_kv, s.topk, s.nb);        \
  } while (0)
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
