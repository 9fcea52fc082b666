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
// Decode moves the cache from HBM once and does little arithmetic per byte, so these
// kernels run on the CUDA cores with coalesced 16-byte loads:
//   decode_pool_kernel    one warp per earlier key block, all groups: pooled scores;
//   decode_select_kernel  one CTA per (sequence, group): exact top-(k-1) by repeated
//                         block-wide argmax (ties -> lower block), plus the own block;
//   decode_attn_kernel    one CTA per (sequence, group, slot): the block's K/V in smem,
//                         scores, softmax partial (lse) and P V for every head;
//   decode_combine_kernel one CTA per (sequence, head): merges the k partials.
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
  const int32_t* lens;         // [B], 1 <= lens[b] <= Lmax
  int32_t* block_idx;          // [B][H_kv][topk]
  float* pooled;               // [B][H_kv][nbm]
  float* o_part;               // [B][H_kv][topk][G][d]
  float* lse_part;             // [B][H_kv][topk][G]
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
// every block wholly before the query's block.  Grid (ceil(nbm / 8), B), 8 warps.
template <int DI>
__global__ void __launch_bounds__(256) decode_pool_kernel(const DecodeParams p) {
  extern __shared__ float sq[];  // [H_kv][DI] query index vectors
  const int b = blockIdx.y;
  for (int x = threadIdx.x; x < p.H_kv * DI; x += blockDim.x)
    sq[x] = __bfloat162float(p.q_idx[(int64_t)b * p.H_kv * DI + x]);
  __syncthreads();
  const int L = seq_len(p, b, p.status);
  const int c_own = (L - 1) / 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * 8 + warp;
  if (c >= c_own) return;
  // the lane's keys c*128 + lane + 32 i (i < 4); groups outer, one key row in registers
  // at a time (the re-reads for later groups hit L1)
  for (int g = 0; g < p.H_kv; ++g) {
    const float* qg = sq + g * DI;
    float m = -INFINITY;
#pragma unroll 1
    for (int i = 0; i < 4; ++i) {
      const uint4* src = reinterpret_cast<const uint4*>(
          p.k_idx + ((int64_t)b * p.Lmax + c * 128 + lane + 32 * i) * DI);
      float sacc = 0.f;
#pragma unroll
      for (int x = 0; x < DI / 8; ++x) {
        const uint4 w = __ldg(&src[x]);
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          sacc = fmaf(qg[8 * x + 2 * e], __low2float(h2[e]), sacc);
          sacc = fmaf(qg[8 * x + 2 * e + 1], __high2float(h2[e]), sacc);
        }
      }
      m = fmaxf(m, sacc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) p.pooled[((int64_t)b * p.H_kv + g) * p.nbm + c] = m;
  }
}

// block_idx[b][g][:] = the k-1 best earlier blocks (pooled descending, lower id first on
// ties) and the own block, ascending, -1 padded.  One CTA (256 threads) per (b, g).
__global__ void __launch_bounds__(256) decode_select_kernel(const DecodeParams p) {
  extern __shared__ float sp[];  // [nbm] candidate scores; selected ones set to -inf
  __shared__ float rv[8];
  __shared__ int ri[8];
  __shared__ int chosen[32];
  const int b = blockIdx.y, g = blockIdx.x;
  const int L = seq_len(p, b, p.status);
  const int c_own = (L - 1) / 128;
  const float* src = p.pooled + ((int64_t)b * p.H_kv + g) * p.nbm;
  for (int c = threadIdx.x; c < c_own; c += blockDim.x) sp[c] = src[c];
  __syncthreads();
  const int M = min(p.topk - 1, c_own);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = 0; r < M; ++r) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int c = threadIdx.x; c < c_own; c += blockDim.x) {
      const float v = sp[c];
      if (v > bv || (v == bv && c < bi)) {
        bv = v;
        bi = c;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == 0) {
      rv[warp] = bv;
      ri[warp] = bi;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      float v = rv[0];
      int id = ri[0];
      for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
        if (rv[w] > v || (rv[w] == v && ri[w] < id)) {
          v = rv[w];
          id = ri[w];
        }
      if (id < 0 || id >= c_own) id = 0;  // only when every candidate is -inf/NaN
      chosen[r] = id;
      sp[id] = -INFINITY;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    int v[32];
    for (int s = 0; s < M; ++s) v[s] = chosen[s];
    v[M] = c_own;
    for (int a = 1; a <= M; ++a)  // insertion sort, at most 32 entries
      for (int s = a; s > 0 && v[s - 1] > v[s]; --s) {
        const int t = v[s - 1];
        v[s - 1] = v[s];
        v[s] = t;
      }
    int32_t* dst = p.block_idx + ((int64_t)b * p.H_kv + g) * p.topk;
    for (int s = 0; s < p.topk; ++s) dst[s] = s <= M ? v[s] : -1;
  }
}

// Softmax partial of every head of group g over the selected block in slot s.
// Grid (topk, H_kv, B), 256 threads.
template <int D>
__global__ void __launch_bounds__(256) decode_attn_kernel(const DecodeParams p) {
  constexpr int KS = D + 8;  // padded K/V row (bf16): conflict-free row-wise 16-byte reads
  extern __shared__ __align__(16) uint8_t dsm[];
  __nv_bfloat16* sK = reinterpret_cast<__nv_bfloat16*>(dsm);
  __nv_bfloat16* sV = sK + 128 * KS;
  float* sQ = reinterpret_cast<float*>(sV + 128 * KS);  // [G][D]
  float* sP = sQ + p.G * D;                               // [G][128]
  float* sM = sP + p.G * 128;                             // [G] max, [G] sum
  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int G = p.G;
  const int64_t part = (((int64_t)b * p.H_kv + g) * p.topk + s) * G;
  const int c = __ldg(&p.block_idx[((int64_t)b * p.H_kv + g) * p.topk + s]);
  if (c < 0) {
    for (int h = threadIdx.x; h < G; h += blockDim.x) p.lse_part[part + h] = -INFINITY;
    return;
  }
  const int L = seq_len(p, b, p.status);
  const int jmax = min(L - 1, c * 128 + 127) - c * 128;  // last visible row of the block
  // K, V rows of the block and the group's query heads
  for (int x = threadIdx.x; x < 128 * (D / 8); x += blockDim.x) {
    const int r = x / (D / 8), ch = x % (D / 8);
    const int j = c * 128 + r;
    uint4 kw = make_uint4(0u, 0u, 0u, 0u), vw = kw;
    if (j < p.Lmax && r <= jmax) {
      const int64_t off = (((int64_t)b * p.Lmax + j) * p.H_kv + g) * D + ch * 8;
      kw = __ldg(reinterpret_cast<const uint4*>(p.k + off));
      vw = __ldg(reinterpret_cast<const uint4*>(p.v + off));
    }
    *reinterpret_cast<uint4*>(sK + r * KS + ch * 8) = kw;
    *reinterpret_cast<uint4*>(sV + r * KS + ch * 8) = vw;
  }
  for (int x = threadIdx.x; x < G * D; x += blockDim.x)
    sQ[x] = __bfloat162float(p.q[((int64_t)b * p.H_kv * G + g * G) * D + x]);
  __syncthreads();
  // scores: thread -> (key r, heads h = hs, hs + 2, ...)
  {
    const int r = threadIdx.x & 127;
    for (int h = threadIdx.x >> 7; h < G; h += 2) {
      float acc = 0.f;
      const float* qh = sQ + h * D;
#pragma unroll 4
      for (int x = 0; x < D; x += 8) {
        const uint4 w = *reinterpret_cast<const uint4*>(sK + r * KS + x);
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc = fmaf(qh[x + 2 * e], __low2float(h2[e]), acc);
          acc = fmaf(qh[x + 2 * e + 1], __high2float(h2[e]), acc);
        }
      }
      sP[h * 128 + r] = r <= jmax ? acc * p.scale : -INFINITY;
    }
  }
  __syncthreads();
  // per head: max, exp, sum (one warp per head)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int h = warp; h < G; h += (int)(blockDim.x >> 5)) {
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < 4; ++i) m = fmaxf(m, sP[h * 128 + lane + 32 * i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float l = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float e = expf(sP[h * 128 + lane + 32 * i] - m);  // masked: exp(-inf) = 0
      sP[h * 128 + lane + 32 * i] = e;
      l += e;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) {
      sM[h] = m;
      sM[G + h] = l;
      p.lse_part[part + h] = m + logf(l);
    }
  }
  __syncthreads();
  // O partial (normalised): thread -> (head, d)
  for (int x = threadIdx.x; x < G * D; x += blockDim.x) {
    const int h = x / D, dd = x % D;
    float acc = 0.f;
    const float* ph = sP + h * 128;
    for (int r = 0; r <= jmax; ++r) acc = fmaf(ph[r], __bfloat162float(sV[r * KS + dd]), acc);
    p.o_part[(part + h) * D + dd] = acc / sM[G + h];
  }
}

// o[b][h] and lse[b][h] from the k partials of head h.  One CTA (D threads) per (b, h).
__global__ void decode_combine_kernel(const DecodeParams p) {
  const int bh = blockIdx.x;
  const int b = bh / (p.H_kv * p.G), h = bh % (p.H_kv * p.G);
  const int g = h / p.G, hh = h % p.G;
  const int64_t base = ((int64_t)b * p.H_kv + g) * p.topk;
  float m = -INFINITY;
  for (int s = 0; s < p.topk; ++s) m = fmaxf(m, p.lse_part[(base + s) * p.G + hh]);
  float l = 0.f, acc = 0.f;
  for (int s = 0; s < p.topk; ++s) {
    const float ls = p.lse_part[(base + s) * p.G + hh];
    if (ls == -INFINITY) continue;
    const float w = expf(ls - m);
    l += w;
    acc = fmaf(w, p.o_part[((base + s) * p.G + hh) * p.d + threadIdx.x], acc);
  }
  p.o[((int64_t)b * p.H_kv * p.G + h) * p.d + threadIdx.x] = __float2bfloat16(l > 0.f ? acc / l : 0.f);
  if (threadIdx.x == 0) p.lse[(int64_t)b * p.H_kv * p.G + h] = m + logf(l);
}

size_t decode_ws_parts(const Shape& s, size_t* off_pooled, size_t* off_o, size_t* off_lse) {
  const int nbm = s.nb;
  size_t off = 0;
  *off_pooled = off;
  off += align256((size_t)s.B * s.H_kv * (nbm > 0 ? nbm : 1) * 4);
  *off_o = off;
  off += align256((size_t)s.B * s.H_kv * s.topk * s.G * s.d * 4);
  *off_lse = off;
  off += align256((size_t)s.B * s.H_kv * s.topk * s.G * 4);
  return off;
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" {

size_t msa_decode_workspace_size(const msa_problem_t* p) {
  Shape s;
  if (validate_problem(p, &s) != MSA_OK) return 0;
  size_t a, b, c;
  return decode_ws_parts(s, &a, &b, &c);
}

int msa_decode(const msa_problem_t* p, const void* q, const void* q_idx, const void* k,
               const void* v, const void* k_idx, const int32_t* lens, int32_t* block_idx, void* o,
               float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  Shape s;
  int rc = validate_problem(p, &s);
  if (rc) return rc;
  if (s.B == 0) return MSA_OK;
  if (s.N == 0) return MSA_ERR_SHAPE;  // N is the cache capacity Lmax
  const void* ptrs[] = {q, q_idx, k, v, k_idx, lens, block_idx, o, lse};
  for (const void* x : ptrs)
    if (!x || (reinterpret_cast<uintptr_t>(x) & 15) != 0) return MSA_ERR_ARG;
  size_t off_pooled, off_o, off_lse;
  const size_t need = decode_ws_parts(s, &off_pooled, &off_o, &off_lse);
  if (!workspace || workspace_bytes < need) return MSA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return MSA_ERR_ARG;
  Ctx cx;
  if ((rc = device_ctx(&cx))) return rc;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  DecodeParams dp;
  dp.q = static_cast<const __nv_bfloat16*>(q);
  dp.q_idx = static_cast<const __nv_bfloat16*>(q_idx);
  dp.k = static_cast<const __nv_bfloat16*>(k);
  dp.v = static_cast<const __nv_bfloat16*>(v);
  dp.k_idx = static_cast<const __nv_bfloat16*>(k_idx);
  dp.lens = lens;
  dp.block_idx = block_idx;
  dp.pooled = reinterpret_cast<float*>(w + off_pooled);
  dp.o_part = reinterpret_cast<float*>(w + off_o);
  dp.lse_part = reinterpret_cast<float*>(w + off_lse);
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
  const size_t pool_smem = (size_t)s.H_kv * s.d_idx * sizeof(float);
  if (pool_smem > 48 * 1024) return MSA_ERR_UNSUPPORTED;
  const dim3 gpool((unsigned)((s.nb + 7) / 8), (unsigned)s.B);
  if (s.d_idx == 64) decode_pool_kernel<64><<<gpool, 256, pool_smem, stream>>>(dp);
  else decode_pool_kernel<32><<<gpool, 256, pool_smem, stream>>>(dp);
  note_launch();
  const size_t sel_smem = (size_t)s.nb * sizeof(float);
  if (sel_smem > 48 * 1024) {
    if (cudaFuncSetAttribute(decode_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sel_smem) != cudaSuccess)
      return MSA_ERR_CUDA;
  }
  decode_select_kernel<<<dim3((unsigned)s.H_kv, (unsigned)s.B), 256, sel_smem, stream>>>(dp);
  note_launch();
  const size_t attn_smem = (size_t)2 * 128 * (s.d + 8) * 2 + (size_t)s.G * (s.d + 128 + 2) * 4;
  const dim3 gattn((unsigned)s.topk, (unsigned)s.H_kv, (unsigned)s.B);
  cudaError_t e;
  if (s.d == 128) {
    e = cudaFuncSetAttribute(decode_attn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)attn_smem);
    if (e == cudaSuccess) decode_attn_kernel<128><<<gattn, 256, attn_smem, stream>>>(dp);
  } else {
    e = cudaFuncSetAttribute(decode_attn_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)attn_smem);
    if (e == cudaSuccess) decode_attn_kernel<64><<<gattn, 256, attn_smem, stream>>>(dp);
  }
  if (e != cudaSuccess) return MSA_ERR_CUDA;
  note_launch();
  decode_combine_kernel<<<(unsigned)(s.B * s.H_q), (unsigned)s.d, 0, stream>>>(dp);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

}  // extern "C"
