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
// The tile work is the tcgen05 kernel of attn_bwd_tc.cu; this file holds the
// preprocess (D = rowsum(dO o)), the reductions of the per-slot dq / dq_idx
// partials and of the per-group dk_idx shares, and the call sequence.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace msa {
namespace {

// D[b,h,i] = dO[b,i,h,:] . o[b,i,h,:] (layout of lse: t0*H_q + h*len + i).  One CTA per
// 64 consecutive queries i of one (b, h): TPR = D / 8 threads per row (16-byte loads),
// every pass's loads issued before the sums, and D written along i.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ dO,
                                                      float* __restrict__ Dv,
                                                      const int2* __restrict__ spans,
                                                      const int* __restrict__ tab, int B, int N,
                                                      int H_q) {
  constexpr int TPR = D / 8;      // threads per row
  constexpr int RPP = 256 / TPR;  // rows per pass
  constexpr int NP = 64 / RPP;    // passes
  const int h = blockIdx.x % H_q;
  int b, chunk;
  if (!chunk_item(tab, B, (N + 63) / 64, blockIdx.x / H_q, &b, &chunk)) return;
  const SeqSpan sp = seq_span(spans, b, N);
  const int i0 = chunk * 64;
  const int t = threadIdx.x % TPR, rr = threadIdx.x / TPR;
  uint4 xa[NP], xb[NP];
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    const int i = i0 + q * RPP + rr;
    if (i < sp.len) {
      const int64_t off = ((sp.t0 + i) * H_q + h) * D + t * 8;
      xa[q] = __ldg(reinterpret_cast<const uint4*>(o + off));
      xb[q] = __ldg(reinterpret_cast<const uint4*>(dO + off));
    } else {
      xa[q] = make_uint4(0u, 0u, 0u, 0u);
      xb[q] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&xa[q]);
    const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&xb[q]);
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      s += __low2float(x[e]) * __low2float(y[e]) + __high2float(x[e]) * __high2float(y[e]);
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    const int i = i0 + q * RPP + rr;
    if (t == 0 && i < sp.len) Dv[sp.t0 * H_q + (int64_t)h * sp.len + i] = s;
  }
}

// Sum of the per-slot partials of one (b, g, i) row: dq (the G heads of the group, G*W
// contiguous bf16 per slot) or dq_idx (G = 1, W = d_idx).  Lanes read 16-byte chunks;
// when a row has fewer than 32 chunks a warp serves several rows.
template <int W, int G>
__global__ void __launch_bounds__(256) slot_reduce_kernel(
    const __nv_bfloat16* __restrict__ part, const int32_t* __restrict__ block_idx,
    __nv_bfloat16* __restrict__ out, const int2* __restrict__ spans, int B, int64_t rows_kv,
    int N, int H_kv, int topk, int nb) {
  constexpr int TC = G * W / 8;               // 16-byte chunks per row and slot
  constexpr int RPW = TC >= 32 ? 1 : 32 / TC; // rows per warp
  constexpr int CPL = TC >= 32 ? TC / 32 : 1; // chunks per lane
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t rkv = warp * RPW + (TC >= 32 ? 0 : lane / TC);
  const int l = TC >= 32 ? lane : lane % TC;
  if (rkv >= rows_kv) return;
  RowPos rp;
  const bool valid = row_pos(spans, B, N, H_kv, rkv, &rp);  // tokens outside every sequence
  if (!valid) return;
  const int i = rp.i, g = rp.h;
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
  // out row: dq [t0 + i][g*G .. g*G+G-1][W]  or  dq_idx [t0 + i][g][W]
  uint4* dst = reinterpret_cast<uint4*>(out + ((rp.sp.t0 + i) * H_kv + g) * (int64_t)G * W);
#pragma unroll
  for (int x = 0; x < CPL; ++x) {
    uint4 o;
    uint32_t* pw = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int e = 0; e < 4; ++e) pw[e] = pack_bf16(acc[x][2 * e], acc[x][2 * e + 1]);
    dst[l + 32 * x] = o;
  }
}

// dk_idx[j,:] = sum over groups of the per-group shares (part [T][H_kv][DI], every token
// of every sequence written by the tile kernel; tokens outside every sequence hold 0).
__global__ void dki_reduce_kernel(const float* __restrict__ part, __nv_bfloat16* __restrict__ out,
                                  const int2* __restrict__ spans, int B, int64_t T, int H_kv,
                                  int DI) {
  const int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (t >= T * DI) return;
  const int64_t j = t / DI, r = t - j * DI;
  if (spans && j >= __ldg(&spans[B - 1].y)) return;  // past the last sequence
  float s = 0.f;
  for (int g = 0; g < H_kv; ++g) s += part[(j * H_kv + g) * DI + r];
  out[t] = __float2bfloat16(s);
}

__global__ void kl_out_kernel(const double* __restrict__ acc, float* __restrict__ out) {
  *out = (float)*acc;
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
  off += align256((size_t)s.T * s.H_q * 4);
  w.dq_part = reinterpret_cast<__nv_bfloat16*>(base + off);
  off += align256(parts * s.G * s.d * 2);
  w.dqi_part = reinterpret_cast<__nv_bfloat16*>(base + off);
  off += align256(parts * s.d_idx * 2);
  w.dki_part = reinterpret_cast<float*>(base + off);
  off += align256((size_t)s.T * s.H_kv * s.d_idx * 4);
  if (out) *out = w;
  return off;
}

}  // namespace

size_t bwd_ws_bytes(const Shape& s) { return carve(s, nullptr, nullptr); }

cudaError_t run_bwd(const Shape& s, const void* q, const void* k, const void* v, const void* o,
                    const float* lse, const void* dO, const void* q_idx, const void* k_idx,
                    const int32_t* block_idx, const float* lse_idx, float kl_weight, void* dq,
                    void* dk, void* dv, void* dq_idx, void* dk_idx, float* kl_out, void* ws,
                    const Ctx& cx, cudaStream_t st, void* plan) {
  BwdWs w;
  carve(s, ws, &w);
  cudaError_t e;
  if (plan) {  // the step's shared plan (the backward reads its CSR only)
    const SharedPlan sp = shared_plan_carve(s, plan);
    e = launch_shared_plan_check(s, sp, cx, st);
    w.pl = sp.idx;
  } else {
    e = launch_plan(s, block_idx, 64 / s.G, w.pl, cx, st);
  }
  if (e != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(w.counter, 0, 256, st)) != cudaSuccess) return e;  // counter + KL
  {
    const int64_t blocks = (int64_t)s.H_q * (s.packed() ? varlen_grid_items(s, kTabRows64)
                                                        : (int64_t)s.B * ((s.N + 63) / 64));
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    const unsigned grid = (unsigned)blocks;
    if (s.d == 128)
      bwd_pre_kernel<128><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(o),
                                                static_cast<const __nv_bfloat16*>(dO), w.Dv,
                                                s.spans, s.tab(kTabRows64), s.B, s.N, s.H_q);
    else
      bwd_pre_kernel<64><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(o),
                                               static_cast<const __nv_bfloat16*>(dO), w.Dv,
                                               s.spans, s.tab(kTabRows64), s.B, s.N, s.H_q);
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  e = launch_attn_bwd_tc(s, q, k, v, dO, lse, w.Dv, q_idx, k_idx, lse_idx, kl_weight, w.pl,
                         w.dq_part, w.dqi_part, w.dki_part, w.kl_acc, dk, dv, cx, st);
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
#define MSA_SLOT_REDUCE(W, GG)                                                                \
  slot_reduce_kernel<W, GG><<<grid_for(GG * W / 8), 256, 0, st>>>(                             \
      w.dq_part, block_idx, dqb, s.spans, s.B, R, s.N, s.H_kv, s.topk, s.nb)
    if (s.d == 128) {
      switch (s.G) {
        case 1: MSA_SLOT_REDUCE(128, 1); break;
        case 2: MSA_SLOT_REDUCE(128, 2); break;
        case 4: MSA_SLOT_REDUCE(128, 4); break;
        case 8: MSA_SLOT_REDUCE(128, 8); break;
        default: MSA_SLOT_REDUCE(128, 16); break;
      }
    } else {
      switch (s.G) {
        case 1: MSA_SLOT_REDUCE(64, 1); break;
        case 2: MSA_SLOT_REDUCE(64, 2); break;
        case 4: MSA_SLOT_REDUCE(64, 4); break;
        case 8: MSA_SLOT_REDUCE(64, 8); break;
        default: MSA_SLOT_REDUCE(64, 16); break;
      }
    }
#undef MSA_SLOT_REDUCE
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (s.d_idx == 64)
      slot_reduce_kernel<64, 1><<<grid_for(8), 256, 0, st>>>(w.dqi_part, block_idx, dqib, s.spans,
                                                            s.B, R, s.N, s.H_kv, s.topk, s.nb);
    else
      slot_reduce_kernel<32, 1><<<grid_for(4), 256, 0, st>>>(w.dqi_part, block_idx, dqib, s.spans,
                                                            s.B, R, s.N, s.H_kv, s.topk, s.nb);
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t n = s.T * s.d_idx;
    dki_reduce_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(
        w.dki_part, static_cast<__nv_bfloat16*>(dk_idx), s.spans, s.B, s.T, s.H_kv, s.d_idx);
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
