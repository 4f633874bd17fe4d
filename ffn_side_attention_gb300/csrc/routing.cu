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
// Batches of at most 32 tokens: one launch of one warp, routing_warp_kernel (lane =
// token; per-expert bit words in shared memory give counts and ranks).  It took ~0.4 us
// less than the 256-thread block at T = 6 (qwen3 shapes).
// Batches of at most 256 tokens (one block): one launch, routing_one_block_kernel.
// The block ranks its tokens' entries (below), keeps the per-expert counts in shared
// memory, scans them and writes pos / perm, with no global synchronisation.
//
// 257..2048 tokens: one launch, routing_fused_kernel (below).
// Larger batches: two launches, both one thread per token in blocks of 256 tokens:
//   block_rank: per block, the per-expert counts (to a [blocks][E] array) and
//     each entry's rank among the block's entries of the same expert, in
//     token order.  A token's k experts are distinct, so that rank is the
//     number of earlier tokens of the block that chose the expert: each warp
//     sets bit `lane` of a per-expert word for every expert its token chose;
//     the rank is the popcount of the lower lanes' bits plus the popcounts of
//     the earlier warps' words.
//   place: every block re-adds the block counts (totals, its own base per
//     expert), scans them into offsets and tile bases, and writes
//     pos = offsets[e] + base + rank and perm[pos] = token.
// A single launch with a device-wide barrier between the two steps (a ticket,
// then a generation flag, bounded waits) was built and measured slower than the
// two launches with programmatic dependent launch: the second launch's blocks are
// resident and released by the hardware as soon as the first grid completes,
// while the barrier's atomics and polling cost more.
#include "afd_internal.cuh"

namespace afd {
namespace {

constexpr int kTok = 256;                  // tokens per block (one per thread)
constexpr int kWarpsPerBlock = kTok / 32;  // 8
constexpr int kRouteMaxK = 16;             // slots per token (the layer's limit on k)

__global__ void __launch_bounds__(kTok) block_rank_kernel(const int32_t* __restrict__ idx, int T, int k, int E,
                                                          int32_t* __restrict__ block_hist,
                                                          int32_t* __restrict__ rank, int* err) {
  pdl_begin();
  extern __shared__ uint32_t bits[];  // [kWarpsPerBlock][E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kTok + threadIdx.x;
  for (int i = threadIdx.x; i < kWarpsPerBlock * E; i += kTok) bits[i] = 0;
  __syncthreads();
  uint32_t* my = bits + warp * E;
  // this token's experts, all loaded before any use (a load per slot in a loop over k
  // serialised the round trips: T = 3160 routing 16.7 -> 15.4 us with this and the batched
  // loads of place_kernel)
  int ex[kRouteMaxK];
#pragma unroll
  for (int j = 0; j < kRouteMaxK; ++j) ex[j] = (j < k && t < T) ? __ldg(idx + (size_t)t * k + j) : -1;
#pragma unroll
  for (int j = 0; j < kRouteMaxK; ++j) {
    if (j >= k || t >= T) break;
    if (ex[j] < 0 || ex[j] >= E) {
      atomicOr(err, kErrRange);
      ex[j] = -1;
    } else {
      atomicOr(my + ex[j], 1u << lane);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kTok) {
    int total = 0;
    for (int w = 0; w < kWarpsPerBlock; ++w) total += __popc(bits[w * E + e]);
    block_hist[(size_t)blockIdx.x * E + e] = total;
  }
  if (t < T) {
    const uint32_t lower = (1u << lane) - 1u;
#pragma unroll
    for (int j = 0; j < kRouteMaxK; ++j)
      if (ex[j] >= 0) {
        int r = __popc(my[ex[j]] & lower);
        for (int w = 0; w < warp; ++w) r += __popc(bits[w * E + ex[j]]);
        rank[(size_t)t * k + j] = r;
      }
  }
}

// inclusive scan of one value per lane
__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// Exclusive scans of the group counts into row offsets and GEMM tile bases (BN tokens
// per tile), by a whole block of kTok threads: one group per thread, warp scans, then
// the warp totals (integer sums, so the order does not matter).  A group past the
// block's threads (G = 257) is added last by the last thread.  Ends with a barrier.
__device__ __forceinline__ void scan_groups(const int* s_cnt, int G, int BN, int* s_off, int* s_tb) {
  __shared__ int s_wo[kWarpsPerBlock], s_wt[kWarpsPerBlock];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = threadIdx.x;
  const int c = (g < G) ? s_cnt[g] : 0;
  const int nt = (c + BN - 1) / BN;
  const int io = warp_incl_scan(c, lane);
  const int it = warp_incl_scan(nt, lane);
  if (lane == 31) {
    s_wo[warp] = io;
    s_wt[warp] = it;
  }
  __syncthreads();
  int po = 0, pt = 0;
  for (int w = 0; w < warp; ++w) {
    po += s_wo[w];
    pt += s_wt[w];
  }
  if (g < G) {
    s_off[g] = po + io - c;
    s_tb[g] = pt + it - nt;
  }
  if (threadIdx.x == kTok - 1) {
    int to = po + io, tt = pt + it;
    for (int x = kTok; x < G; ++x) {
      s_off[x] = to;
      s_tb[x] = tt;
      to += s_cnt[x];
      tt += (s_cnt[x] + BN - 1) / BN;
    }
    s_off[G] = to;
    s_tb[G] = tt;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kTok)
    place_kernel(const int32_t* __restrict__ idx, const int32_t* __restrict__ block_hist, int nblocks, int T, int k,
                 int E, int S, int BN, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                 int32_t* __restrict__ tile_base, int32_t* __restrict__ perm, int32_t* __restrict__ pos,
                 int32_t* __restrict__ gu_done) {
  pdl_begin();
  __shared__ int s_cnt[kMaxExperts + 1], s_base[kMaxExperts], s_off[kMaxExperts + 1], s_tb[kMaxExperts + 1];
  const int G = E + S;
  for (int e = threadIdx.x; e < E; e += kTok) {
    int before = 0, total = 0;
    for (int b0 = 0; b0 < nblocks; b0 += 16) {  // sixteen blocks' counts in flight at once
      int c[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) c[u] = b0 + u < nblocks ? __ldg(block_hist + (size_t)(b0 + u) * E + e) : 0;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        if (b0 + u < (int)blockIdx.x) before += c[u];
        total += c[u];
      }
    }
    s_cnt[e] = total;
    s_base[e] = before;
  }
  if (threadIdx.x == 0 && S) s_cnt[E] = T;
  __syncthreads();
  scan_groups(s_cnt, G, BN, s_off, s_tb);
  if (blockIdx.x == 0)
    for (int g = threadIdx.x; g <= G; g += kTok) {
      offsets[g] = s_off[g];
      tile_base[g] = s_tb[g];
      if (g < G) {
        counts[g] = s_cnt[g];
        gu_done[g] = 0;  // this forward's gate/up GEMM counts its finished items here
      }
    }
  const int t = blockIdx.x * kTok + threadIdx.x;
  if (t < T) {
    int ex[kRouteMaxK], rk[kRouteMaxK];  // experts and in-block ranks, all loaded before any use
#pragma unroll
    for (int j = 0; j < kRouteMaxK; ++j) {
      ex[j] = j < k ? __ldg(idx + (size_t)t * k + j) : -1;
      rk[j] = j < k ? pos[(size_t)t * k + j] : 0;  // pos holds the in-block rank
    }
#pragma unroll
    for (int j = 0; j < kRouteMaxK; ++j) {
      const int e = ex[j];
      if (j >= k || e < 0 || e >= E) continue;
      const int row = s_off[e] + s_base[e] + rk[j];
      pos[(size_t)t * k + j] = row;
      perm[row] = t;
    }
    if (S) perm[(size_t)T * k + t] = t;
  }
}

// Whole routing of a batch of at most kTok tokens in one block: ranks (as in
// block_rank_kernel), counts kept in shared memory, exclusive scans, placement.
__global__ void __launch_bounds__(kTok)
    routing_one_block_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int S, int BN,
                             int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                             int32_t* __restrict__ tile_base, int32_t* __restrict__ perm, int32_t* __restrict__ pos,
                             int32_t* __restrict__ gu_done, int* err) {
  pdl_begin();
  extern __shared__ uint32_t bits[];  // [kWarpsPerBlock][E]
  __shared__ int s_cnt[kMaxExperts + 1], s_off[kMaxExperts + 1], s_tb[kMaxExperts + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = threadIdx.x;
  const int G = E + S;
  for (int i = threadIdx.x; i < kWarpsPerBlock * E; i += kTok) bits[i] = 0;
  __syncthreads();
  uint32_t* my = bits + warp * E;
  int ex[kRouteMaxK];
#pragma unroll
  for (int j = 0; j < kRouteMaxK; ++j) {
    ex[j] = -1;
    if (j < k && t < T) {
      const int e = __ldg(idx + (size_t)t * k + j);
      if (e < 0 || e >= E) {
        atomicOr(err, kErrRange);
      } else {
        ex[j] = e;
        atomicOr(my + e, 1u << lane);
      }
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kTok) {
    int total = 0;
    for (int w = 0; w < kWarpsPerBlock; ++w) total += __popc(bits[w * E + e]);
    s_cnt[e] = total;
  }
  if (threadIdx.x == 0 && S) s_cnt[E] = T;
  __syncthreads();
  scan_groups(s_cnt, G, BN, s_off, s_tb);
  for (int g = threadIdx.x; g <= G; g += kTok) {
    offsets[g] = s_off[g];
    tile_base[g] = s_tb[g];
    if (g < G) {
      counts[g] = s_cnt[g];
      gu_done[g] = 0;  // this forward's gate/up GEMM counts its finished items here
    }
  }
  if (t < T) {
    const uint32_t lower = (1u << lane) - 1u;
#pragma unroll
    for (int j = 0; j < kRouteMaxK; ++j)
      if (ex[j] >= 0) {
        const int e = ex[j];
        int r = __popc(my[e] & lower);
        for (int w = 0; w < warp; ++w) r += __popc(bits[w * E + e]);
        const int row = s_off[e] + r;
        pos[(size_t)t * k + j] = row;
        perm[row] = t;
      }
    if (S) perm[(size_t)T * k + t] = t;
  }
}


// Batches of at most 32 tokens: the routing tables built by one warp (lane = token).
__global__ void __launch_bounds__(32)
    routing_warp_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int S, int BN,
                        int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ tile_base,
                        int32_t* __restrict__ perm, int32_t* __restrict__ pos, int32_t* __restrict__ gu_done, int* err) {
  pdl_begin();
  __shared__ uint32_t s_bits[kMaxExperts];  // per expert: bit t set if token t chose it
  __shared__ int s_goff[kMaxExperts + 1];
  const int lane = threadIdx.x;
  const int G = E + S;
  for (int e = lane; e < E; e += 32) s_bits[e] = 0u;
  __syncwarp();
  int ex[kRouteMaxK];
#pragma unroll
  for (int j = 0; j < kRouteMaxK; ++j) {
    ex[j] = -1;
    if (j < k && lane < T) {
      const int e = __ldg(idx + (size_t)lane * k + j);
      if (e < 0 || e >= E) {
        atomicOr(err, kErrRange);
      } else {
        ex[j] = e;
        atomicOr(&s_bits[e], 1u << lane);
      }
    }
  }
  __syncwarp();
  // lane l scans groups [l c, l c + c): local sums, then a warp scan of the sums
  const int c = (G + 31) / 32;
  int lo_rows = 0, lo_tiles = 0;
  for (int i = 0; i < c; ++i) {
    const int g = lane * c + i;
    if (g < G) {
      const int n = g < E ? __popc(s_bits[g]) : T;
      lo_rows += n;
      lo_tiles += (n + BN - 1) / BN;
    }
  }
  const int ir = warp_incl_scan(lo_rows, lane), it = warp_incl_scan(lo_tiles, lane);
  int row = ir - lo_rows, tile = it - lo_tiles;
  for (int i = 0; i < c; ++i) {
    const int g = lane * c + i;
    if (g < G) {
      const int n = g < E ? __popc(s_bits[g]) : T;
      s_goff[g] = row;
      offsets[g] = row;
      tile_base[g] = tile;
      counts[g] = n;
      gu_done[g] = 0;  // this forward's gate/up GEMM counts its finished items here
      row += n;
      tile += (n + BN - 1) / BN;
    }
  }
  if (lane == 31) {
    offsets[G] = row;
    tile_base[G] = tile;
  }
  __syncwarp();
  if (lane < T) {
    const uint32_t lower = (1u << lane) - 1u;
#pragma unroll
    for (int j = 0; j < kRouteMaxK; ++j)
      if (ex[j] >= 0) {
        const int r = s_goff[ex[j]] + __popc(s_bits[ex[j]] & lower);
        pos[(size_t)lane * k + j] = r;
        perm[r] = lane;
      }
    if (S) perm[(size_t)T * k + lane] = lane;
  }
}


// Batches of 257..kFusedMaxTok tokens in one launch, no global synchronisation: block b
// ranks its own 256 tokens' entries (as block_rank_kernel) and counts every token's
// entries itself (per-warp histograms in shared memory), which gives both the totals
// and its base (entries of the tokens before its own) without a second launch.
__global__ void __launch_bounds__(kTok)
    routing_fused_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int S, int BN,
                         int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ tile_base,
                         int32_t* __restrict__ perm, int32_t* __restrict__ pos, int32_t* __restrict__ gu_done,
                         int* err) {
  pdl_begin();
  extern __shared__ uint32_t bits[];  // [kWarpsPerBlock][E] rank words, then [kWarpsPerBlock][2][E] counts
  int* whist = reinterpret_cast<int*>(bits + kWarpsPerBlock * E);  // per warp: [0][E] before, [1][E] total
  __shared__ int s_cnt[kMaxExperts + 1], s_base[kMaxExperts], s_off[kMaxExperts + 1], s_tb[kMaxExperts + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = E + S;
  const int t = blockIdx.x * kTok + threadIdx.x;
  for (int i = threadIdx.x; i < kWarpsPerBlock * E * 3; i += kTok) bits[i] = 0;
  __syncthreads();
  uint32_t* my = bits + warp * E;
  int ex[kRouteMaxK];
#pragma unroll
  for (int j = 0; j < kRouteMaxK; ++j) ex[j] = (j < k && t < T) ? __ldg(idx + (size_t)t * k + j) : -1;
#pragma unroll
  for (int j = 0; j < kRouteMaxK; ++j) {
    if (j >= k || t >= T) break;
    if (ex[j] < 0 || ex[j] >= E) {
      atomicOr(err, kErrRange);
      ex[j] = -1;
    } else {
      atomicOr(my + ex[j], 1u << lane);
    }
  }
  // every entry of the batch: per-warp counts (total, and before this block's tokens)
  int* hb = whist + warp * 2 * E;
  const int n = T * k, n_before = (int)blockIdx.x * kTok * k;
  for (int i0 = threadIdx.x; i0 < n; i0 += kTok * 8) {
    int e8[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) e8[u] = i0 + u * kTok < n ? __ldg(idx + i0 + u * kTok) : -1;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = e8[u];
      if (e < 0 || e >= E) continue;
      atomicAdd(hb + E + e, 1);
      if (i0 + u * kTok < n_before) atomicAdd(hb + e, 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kTok) {
    int before = 0, total = 0;
    for (int w = 0; w < kWarpsPerBlock; ++w) {
      before += whist[w * 2 * E + e];
      total += whist[w * 2 * E + E + e];
    }
    s_cnt[e] = total;
    s_base[e] = before;
  }
  if (threadIdx.x == 0 && S) s_cnt[E] = T;
  __syncthreads();
  scan_groups(s_cnt, G, BN, s_off, s_tb);
  if (blockIdx.x == 0)
    for (int g = threadIdx.x; g <= G; g += kTok) {
      offsets[g] = s_off[g];
      tile_base[g] = s_tb[g];
      if (g < G) {
        counts[g] = s_cnt[g];
        gu_done[g] = 0;  // this forward's gate/up GEMM counts its finished items here
      }
    }
  if (t < T) {
    const uint32_t lower = (1u << lane) - 1u;
#pragma unroll
    for (int j = 0; j < kRouteMaxK; ++j)
      if (ex[j] >= 0) {
        const int e = ex[j];
        int r = __popc(my[e] & lower);
        for (int w = 0; w < warp; ++w) r += __popc(bits[w * E + e]);
        const int row = s_off[e] + s_base[e] + r;
        pos[(size_t)t * k + j] = row;
        perm[row] = t;
      }
    if (S) perm[(size_t)T * k + t] = t;
  }
}

}  // namespace

__global__ void wait_probe_kernel(int* err, long long limit) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  mbar_wait(&bar, 0, &abort, err, limit);  // phase 0 never completes
}

// One launch up to this many tokens.  Every block of the single launch reads all T*k
// entries, so its cost grows with T times the blocks: up to 2048 tokens it beat the two
// launches (qwen3 shapes: T = 395 step -2.9 us, T = 1580 -1.2 us; DeepSeek-V3 T = 512
// -3.8 us, T = 2048 -4 us); at T = 3160 and 4096 it was slower (+6 us at 4096).
constexpr int kFusedMaxTok = 2048;

int routing_launches(int T) { return T <= kFusedMaxTok ? 1 : 2; }

cudaError_t launch_routing(const LayerDims& d, int T, Workspace& ws, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int nblocks = (T + kTok - 1) / kTok;
  const int bn = d.dtype == AFD_FP8_E4M3 ? kGemmBNFp8 : bf16_tile_tokens(d, T);  // tokens per GEMM tile
  if (T <= 32) {
    const cudaError_t e_ = launch_k(routing_warp_kernel, dim3(1), dim3(32), 0, s, ws.topk_idx, T, d.k, d.E, d.S, bn,
                                    ws.counts, ws.offsets, ws.tile_base, ws.perm, ws.pos, ws.gu_done, ws.err);
    if (e_ != cudaSuccess) return e_;
    return cudaGetLastError();
  }
  if (nblocks == 1) {
    const cudaError_t e_ = launch_k(routing_one_block_kernel, dim3(1), dim3(kTok),
                                    sizeof(uint32_t) * kWarpsPerBlock * d.E, s, ws.topk_idx, T, d.k, d.E, d.S, bn,
                                    ws.counts, ws.offsets, ws.tile_base, ws.perm, ws.pos, ws.gu_done, ws.err);
    if (e_ != cudaSuccess) return e_;
    return cudaGetLastError();
  }
  if (T <= kFusedMaxTok) {
    const cudaError_t e_ = launch_k(routing_fused_kernel, dim3(nblocks), dim3(kTok),
                                    sizeof(uint32_t) * kWarpsPerBlock * d.E * 3, s, ws.topk_idx, T, d.k, d.E, d.S, bn,
                                    ws.counts, ws.offsets, ws.tile_base, ws.perm, ws.pos, ws.gu_done, ws.err);
    if (e_ != cudaSuccess) return e_;
    return cudaGetLastError();
  }
  {
    const cudaError_t e_ = launch_k(block_rank_kernel, dim3(nblocks), dim3(kTok),
                                    sizeof(uint32_t) * kWarpsPerBlock * d.E, s, ws.topk_idx, T, d.k, d.E,
                                    ws.block_hist, ws.pos, ws.err);
    if (e_ != cudaSuccess) return e_;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  {
    const cudaError_t e_ = launch_k(place_kernel, dim3(nblocks), dim3(kTok), 0, s, ws.topk_idx, ws.block_hist,
                                    nblocks, T, d.k, d.E, d.S, bn, ws.counts, ws.offsets, ws.tile_base, ws.perm,
                                    ws.pos, ws.gu_done);
    if (e_ != cudaSuccess) return e_;
  }
  return cudaGetLastError();
}

}  // namespace afd
