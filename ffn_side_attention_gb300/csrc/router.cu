// router.cu -- R1: router logits, top-k and softmax over the selected logits.
//
// "MoE 大规模分布式推理工程实战", section 4.1 (the balanced top-k router's
// forward): logits of a bias-free linear gate, plus an optional per-expert
// bias, top-k on the logits, softmax over the k selected logits.
//
// Bit-reproducible logits.  The selected expert set depends on every bit of
// the logits, so they are computed in one fixed fp32 order (the same order a
// CPU implementation can follow):
//   channels are taken in chunks of 8; chunk c belongs to lane c % 32 of a
//   warp; each lane runs p = fma(x[h], w[h], p) from +0 over its chunks in
//   ascending order (channels ascending inside a chunk); the 32 lane sums are
//   folded with xor-butterflies 16, 8, 4, 2, 1 (lane 0's value is the sum);
//   the bias, when present, is added last in one fp32 addition.
// Selection: expert a ranks before b iff l_a > l_b, or l_a == l_b and a < b;
// slot j holds the j-th ranked expert.  Weights w_j = exp(l_j - l_0) / sum over
// the selected (fp32, expf), so they sum to 1.
//
// Work split: CTA (x, y) computes logits of tokens [16x, 16x+16) against
// experts [32y, 32y+32); warp w covers 4 tokens x 16 experts (64 fp32
// accumulators per lane).  The last CTA to finish a token tile (counted with
// an atomic ticket) runs the top-k for those 16 tokens from the complete
// logit rows and resets the ticket for the next forward.
#include "afd_internal.cuh"

namespace afd {
namespace {

constexpr int kTokPerWarp = 4;
constexpr int kExpPerWarp = 16;
constexpr int kMaxK = 16;

struct Chunk8 {
  float v[8];
};

template <typename TA>
__device__ __forceinline__ void load8(const TA* p, Chunk8& c);

template <>
__device__ __forceinline__ void load8<uint16_t>(const uint16_t* p, Chunk8& c) {
  uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  c.v[0] = bf16_lo(u.x); c.v[1] = bf16_hi(u.x);
  c.v[2] = bf16_lo(u.y); c.v[3] = bf16_hi(u.y);
  c.v[4] = bf16_lo(u.z); c.v[5] = bf16_hi(u.z);
  c.v[6] = bf16_lo(u.w); c.v[7] = bf16_hi(u.w);
}

template <>
__device__ __forceinline__ void load8<float>(const float* p, Chunk8& c) {
  float4 a = __ldg(reinterpret_cast<const float4*>(p));
  float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  c.v[0] = a.x; c.v[1] = a.y; c.v[2] = a.z; c.v[3] = a.w;
  c.v[4] = b.x; c.v[5] = b.y; c.v[6] = b.z; c.v[7] = b.w;
}

// (value, index) ordering of the selection: larger value first, then lower id.
__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

template <typename TA>
__global__ void __launch_bounds__(256) router_kernel(SrcTable st, const TA* __restrict__ wrT,
                                                     const float* __restrict__ bias, int H, int E, int k,
                                                     float* __restrict__ logits, int32_t* __restrict__ topk_idx,
                                                     float* __restrict__ topk_w, int32_t* __restrict__ ticket) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = st.T;
  const int t_base = blockIdx.x * kRouterTokTile + (warp >> 1) * kTokPerWarp;
  const int e_base = blockIdx.y * kRouterExpTile + (warp & 1) * kExpPerWarp;

  // rows of this warp's tokens (nullptr past the batch)
  const TA* xrow[kTokPerWarp];
#pragma unroll
  for (int i = 0; i < kTokPerWarp; ++i) {
    int t = t_base + i;
    if (t < T) {
      int m = src_of_token(st, t);
      xrow[i] = reinterpret_cast<const TA*>(st.src[m]) + (size_t)(t - st.row0[m]) * H;
    } else {
      xrow[i] = nullptr;
    }
  }

  float acc[kTokPerWarp][kExpPerWarp];
#pragma unroll
  for (int i = 0; i < kTokPerWarp; ++i)
#pragma unroll
    for (int j = 0; j < kExpPerWarp; ++j) acc[i][j] = 0.0f;

  const int nchunk = H >> 3;
  for (int c = lane; c < nchunk; c += kWarp) {
    Chunk8 xc[kTokPerWarp];
#pragma unroll
    for (int i = 0; i < kTokPerWarp; ++i) {
      if (xrow[i]) load8<TA>(xrow[i] + 8 * c, xc[i]);
      else {
#pragma unroll
        for (int q = 0; q < 8; ++q) xc[i].v[q] = 0.0f;
      }
    }
#pragma unroll
    for (int j = 0; j < kExpPerWarp; ++j) {
      int e = e_base + j;
      if (e >= E) continue;
      Chunk8 wc;
      load8<TA>(wrT + (size_t)e * H + 8 * c, wc);
#pragma unroll
      for (int i = 0; i < kTokPerWarp; ++i)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[i][j] = fmaf(xc[i].v[q], wc.v[q], acc[i][j]);
    }
  }

  // fold the 32 lane partial sums: xor 16, 8, 4, 2, 1
#pragma unroll
  for (int i = 0; i < kTokPerWarp; ++i)
#pragma unroll
    for (int j = 0; j < kExpPerWarp; ++j) {
      float v = acc[i][j];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) v = v + __shfl_xor_sync(0xffffffffu, v, o);
      acc[i][j] = v;
    }

  // every lane now holds every sum; lane (p % 32) writes pair p
#pragma unroll
  for (int i = 0; i < kTokPerWarp; ++i)
#pragma unroll
    for (int j = 0; j < kExpPerWarp; ++j) {
      int p = i * kExpPerWarp + j;
      int t = t_base + i, e = e_base + j;
      if ((p & 31) == lane && t < T && e < E) {
        float v = acc[i][j];
        if (bias) v = __fadd_rn(v, __ldg(bias + e));
        logits[(size_t)t * E + e] = v;
      }
    }

  // ---- the last CTA of this token tile selects the top-k
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    int prev = atomicAdd(ticket + blockIdx.x, 1);
    s_last = (prev == (int)gridDim.y - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  constexpr int kMaxPerLane = (kMaxExperts + 31) / 32;  // E <= 256 -> 8 per lane
  for (int tt = warp; tt < kRouterTokTile; tt += 8) {
    int t = blockIdx.x * kRouterTokTile + tt;
    if (t >= T) break;
    float v[kMaxPerLane];
    bool taken[kMaxPerLane];
#pragma unroll
    for (int q = 0; q < kMaxPerLane; ++q) {
      int e = lane + 32 * q;
      v[q] = (e < E) ? __ldcg(logits + (size_t)t * E + e) : 0.0f;
      taken[q] = (e >= E);
    }
    float sel_v[kMaxK];
    int sel_i[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j >= k) break;
      // best untaken entry of this lane
      float bv = 0.0f;
      int bi = 0x7fffffff;
#pragma unroll
      for (int q = 0; q < kMaxPerLane; ++q) {
        int e = lane + 32 * q;
        if (!taken[q] && (bi == 0x7fffffff || ranks_before(v[q], e, bv, bi))) {
          bv = v[q];
          bi = e;
        }
      }
      // warp arg-best
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (oi != 0x7fffffff && (bi == 0x7fffffff || ranks_before(ov, oi, bv, bi))) {
          bv = ov;
          bi = oi;
        }
      }
      sel_v[j] = bv;
      sel_i[j] = bi;
#pragma unroll
      for (int q = 0; q < kMaxPerLane; ++q)
        if (lane + 32 * q == bi) taken[q] = true;
    }
    if (lane == 0) {
      float den = 0.0f;
      float ex[kMaxK];
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j >= k) break;
        ex[j] = expf(sel_v[j] - sel_v[0]);
        den += ex[j];
      }
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j >= k) break;
        topk_idx[(size_t)t * k + j] = sel_i[j];
        topk_w[(size_t)t * k + j] = ex[j] / den;
      }
    }
  }
  if (threadIdx.x == 0) ticket[blockIdx.x] = 0;
}

}  // namespace

cudaError_t launch_router(const SrcTable& st, const void* wrT, const float* bias, const LayerDims& d,
                          Workspace& ws, cudaStream_t s) {
  if (st.T == 0) return cudaSuccess;
  dim3 grid((st.T + kRouterTokTile - 1) / kRouterTokTile, (d.E + kRouterExpTile - 1) / kRouterExpTile);
  if (d.dtype == AFD_FP32)
    router_kernel<float><<<grid, 256, 0, s>>>(st, static_cast<const float*>(wrT), bias, d.H, d.E, d.k,
                                              ws.logits, ws.topk_idx, ws.topk_w, ws.tile_counter);
  else
    router_kernel<uint16_t><<<grid, 256, 0, s>>>(st, static_cast<const uint16_t*>(wrT), bias, d.H, d.E,
                                                 d.k, ws.logits, ws.topk_idx, ws.topk_w, ws.tile_counter);
  return cudaGetLastError();
}

}  // namespace afd
