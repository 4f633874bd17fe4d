// routing.cu -- R2: per-expert histogram, exclusive prefix sum and the stable
// expert-contiguous order of the routed (token, slot) pairs.
//
// "MoE 大规模分布式推理工程实战", section 2.2 (custom all-to-all): count the
// items per destination, turn the counts into offsets with a prefix sum, and
// pack items destination-contiguously; here the destination is an expert.
// "MoE系统与AFD架构概述", section 3.3: routing results are pre-sorted so the
// expert kernels read contiguous rows.
//
// Definitions (entry i = t*k + j is token t's slot j, expert idx[i]):
//   counts[e]  = number of entries with expert e
//   offsets[e] = sum of counts[e'] for e' < e   (offsets[E] = T*k)
//   the packed rows of expert e are offsets[e] .. offsets[e+1]-1 and hold its
//   tokens in ascending order; perm[row] = token, pos[i] = row.
// A shared expert (S = 1) is group E with all T tokens in token order: rows
// T*k .. T*k+T-1.  tile_base[g] = sum over g' < g of ceil(counts[g'] / BN), the
// GEMM work list (BN = tokens per GEMM tile).
//
// One CTA of 32 warps.  Entries are split into 32 contiguous segments, one
// per warp, so segment order is entry order.  Pass 1: each warp counts its
// segment per expert (match.any groups equal experts of a 32-entry step; the
// group's lowest lane adds the group size).  A column scan over warps turns
// the counts into per-warp bases, a scan over experts gives the offsets.
// Pass 2 repeats the walk and gives each entry
//   row = offsets[e] + base[warp][e] + (equal experts in earlier lanes),
// which is exactly the stable (by token) counting-sort position.
#include "afd_internal.cuh"

namespace afd {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBatch = 16;  // 32-entry steps whose ids are loaded together

// inclusive scan of one value per lane
__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

__global__ void __launch_bounds__(kThreads, 1)
    routing_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int S, int BN,
                   int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ tile_base,
                   int32_t* __restrict__ perm, int32_t* __restrict__ pos, int* err) {
  extern __shared__ int smem[];
  const int G = E + S;                 // groups (routed + shared)
  int* hist = smem;                    // [kWarps][E]
  int* s_off = smem + kWarps * E;      // [G + 1]
  int* s_tb = s_off + G + 1;           // [G + 1]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = T * k;
  const int seg = ((N + kWarps * 32 - 1) / (kWarps * 32)) * 32;
  const int beg = warp * seg, end = min(N, beg + seg);

  for (int i = threadIdx.x; i < kWarps * E; i += kThreads) hist[i] = 0;
  __syncthreads();

  // pass 1: per-warp counts.  The expert ids of kBatch steps are loaded up
  // front (independent loads in flight), then walked in order.
  int* my = hist + warp * E;
  for (int b0 = beg; b0 < end; b0 += 32 * kBatch) {
    int ev[kBatch];
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int i = b0 + 32 * q + lane;
      ev[q] = (i < end) ? __ldg(idx + i) : -1;
    }
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      if (b0 + 32 * q >= end) break;
      int e = ev[q];
      if (e >= E || e < -1) {
        atomicOr(err, kErrRange);
        e = -1;
      }
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();

  // per-expert column scan over warps -> per-warp bases; totals -> counts
  __shared__ int s_cnt[kMaxExperts + 1];
  for (int e = threadIdx.x; e < E; e += kThreads) {
    int run = 0;
    for (int w = 0; w < kWarps; ++w) {
      int c = hist[w * E + e];
      hist[w * E + e] = run;
      run += c;
    }
    s_cnt[e] = run;
  }
  if (threadIdx.x == 0 && S) s_cnt[E] = T;
  __syncthreads();

  // exclusive scans over the groups: offsets and GEMM tile bases (warp 0)
  if (warp == 0) {
    int carry_o = 0, carry_t = 0;
    for (int g0 = 0; g0 < G; g0 += 32) {
      int g = g0 + lane;
      int c = (g < G) ? s_cnt[g] : 0;
      int nt = (c + BN - 1) / BN;
      int io = warp_incl_scan(c, lane);
      int it = warp_incl_scan(nt, lane);
      if (g < G) {
        s_off[g] = carry_o + io - c;
        s_tb[g] = carry_t + it - nt;
      }
      carry_o += __shfl_sync(0xffffffffu, io, 31);
      carry_t += __shfl_sync(0xffffffffu, it, 31);
    }
    if (lane == 0) {
      s_off[G] = carry_o;
      s_tb[G] = carry_t;
    }
  }
  __syncthreads();
  for (int g = threadIdx.x; g <= G; g += kThreads) {
    offsets[g] = s_off[g];
    tile_base[g] = s_tb[g];
    if (g < G) counts[g] = s_cnt[g];
  }

  // pass 2: positions
  for (int b0 = beg; b0 < end; b0 += 32 * kBatch) {
    int ev[kBatch];
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int i = b0 + 32 * q + lane;
      ev[q] = (i < end) ? __ldg(idx + i) : -1;
    }
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      if (b0 + 32 * q >= end) break;
      const int i = b0 + 32 * q + lane;
      int e = ev[q];
      if (e >= E || e < -1) e = -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      if (e >= 0) {
        const int rank = my[e] + __popc(peers & ((1u << lane) - 1u));
        const int row = s_off[e] + rank;
        perm[row] = i / k;
        pos[i] = row;
      }
      __syncwarp();
      if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
      __syncwarp();
    }
  }
  // shared expert rows: token order
  if (S)
    for (int t = threadIdx.x; t < T; t += kThreads) perm[N + t] = t;
}

}  // namespace

cudaError_t launch_routing(const LayerDims& d, int T, Workspace& ws, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int G = d.E + d.S;
  size_t smem = sizeof(int) * ((size_t)kWarps * d.E + 2 * (G + 1));
  const int bn = d.dtype == AFD_FP8_E4M3 ? kGemmBNFp8 : bf16_tile_tokens(d, T);  // tokens per GEMM tile
  routing_kernel<<<1, kThreads, smem, s>>>(ws.topk_idx, T, d.k, d.E, d.S, bn, ws.counts, ws.offsets,
                                           ws.tile_base, ws.perm, ws.pos, ws.err);
  return cudaGetLastError();
}

}  // namespace afd
