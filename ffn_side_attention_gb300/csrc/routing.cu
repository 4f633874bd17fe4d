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
// One launch, in chunks of 256 tokens (one thread per token), a persistent grid of
// at most one block per SM walking the chunks:
//   1. rank: per chunk, the per-expert counts (to a [chunks][E] array) and each
//      entry's rank among the chunk's entries of the same expert, in token
//      order (kept in pos).  A token's k experts are distinct, so that rank is
//      the number of earlier tokens of the chunk that chose the expert: each
//      warp sets bit `lane` of a per-expert word for every expert its token
//      chose; the rank is the popcount of the lower lanes' bits plus the
//      popcounts of the earlier warps' words.
//   2. barrier: each block reads the barrier's generation, then, once its chunks'
//      counts are out, takes a ticket; the last block resets the ticket and
//      advances the generation (release); the others wait for it to change
//      (acquire), with the same bounded wait as every other cross-block wait: on
//      expiry they set the device error word and return.  The state lives on the
//      device, so a forward captured in a CUDA graph and replayed synchronises
//      the same way.  Every waiting block already holds its ticket and the grid
//      is no larger than the SM count, so a waiting block never keeps the last
//      one from running;
//   3. every block then reads the chunk counts (independent loads, one running
//      prefix per expert), keeps the bases of its own chunks, scans the totals
//      into offsets (block 0 also writes counts, offsets, GEMM tile bases and
//      zeroes the gate/up progress counters) and writes
//      pos = offsets[e] + chunk base + rank and perm[pos] = token.
// The earlier two-launch form (rank, then place with every block re-adding
// the counts) cost one more kernel boundary per forward.
#include <mutex>

#include "afd_internal.cuh"

namespace afd {
namespace {

constexpr int kTok = 256;                  // tokens per chunk (one per thread)
constexpr int kWarpsPerBlock = kTok / 32;  // 8
constexpr size_t kRoutingMaxSmem = 200 * 1024;  // dynamic shared memory of the routing kernel (opt-in)
constexpr int kRouteMaxK = 16;                  // slots per token (the layer's limit on k)

// inclusive scan of one value per lane
__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

__device__ __forceinline__ void st_release_gpu(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Wait until *p != v (acquire), bounded like the other cross-block waits; on expiry the
// kErrTimeout bit of the error word is set and false returned.
__device__ __forceinline__ bool wait_change(const int* p, int v, int* err) {
  if (ld_acquire_gpu(p) != v) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(32);
    if (ld_acquire_gpu(p) != v) return true;
    if ((it & 63u) == 0 && clock64() - t0 > 4000000000ll) {
      atomicOr(err, kErrTimeout);
      return false;
    }
  }
}

struct RoutingArgs {
  const int32_t* idx;
  int T, k, E, S, BN, nchunks;
  int nmine;            // chunks per block at most: ceil(nchunks / grid)
  int32_t* chunk_hist;  // [nchunks][E] per-chunk counts
  int32_t* counts;
  int32_t* offsets;
  int32_t* tile_base;
  int32_t* perm;
  int32_t* pos;  // in-chunk ranks, then packed rows
  int32_t* gu_done;
  int32_t* ticket;  // zero between launches
  int32_t* flag;    // barrier generation, advanced once per launch by its last block
  int* err;
};

__global__ void __launch_bounds__(kTok) routing_kernel(const RoutingArgs a) {
  pdl_begin();
  extern __shared__ uint32_t dyn[];  // bits [kWarpsPerBlock][E], then bases [nmine][E]
  uint32_t* bits = dyn;
  int32_t* s_base = reinterpret_cast<int32_t*>(dyn + kWarpsPerBlock * a.E);
  __shared__ int s_ok;
  __shared__ int s_cnt[kMaxExperts + 1], s_off[kMaxExperts + 1], s_tb[kMaxExperts + 1];
  const int E = a.E, k = a.k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // 1. ranks within each chunk, chunk counts.  The thread's expert ids and ranks of the
  // block's last chunk stay in registers for step 3 (earlier chunks go through pos).
  int ex[kRouteMaxK], rk[kRouteMaxK];
  int last_c = -1;
  for (int c = blockIdx.x; c < a.nchunks; c += gridDim.x) {
    const int t = c * kTok + threadIdx.x;
    for (int i = threadIdx.x; i < kWarpsPerBlock * E; i += kTok) bits[i] = 0;
    __syncthreads();
    uint32_t* my = bits + warp * E;
#pragma unroll
    for (int j = 0; j < kRouteMaxK; ++j) {
      ex[j] = -1;
      if (j < k && t < a.T) {
        const int e = __ldg(a.idx + (size_t)t * k + j);
        if (e < 0 || e >= E) {
          atomicOr(a.err, kErrRange);
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
      a.chunk_hist[(size_t)c * E + e] = total;
    }
    const uint32_t lower = (1u << lane) - 1u;
#pragma unroll
    for (int j = 0; j < kRouteMaxK; ++j) {
      rk[j] = 0;
      if (ex[j] >= 0) {
        const int e = ex[j];
        int r = __popc(my[e] & lower);
        for (int w = 0; w < warp; ++w) r += __popc(bits[w * E + e]);
        rk[j] = r;
        if (c + (int)gridDim.x < a.nchunks) a.pos[(size_t)t * k + j] = r;  // not the last chunk
      }
    }
    last_c = c;
    __syncthreads();  // bits are reused by the next chunk
  }
  // 2. grid barrier: the last block to take a ticket releases the others by advancing the
  // generation every block read before taking its ticket (no host-side state, so a
  // forward captured in a CUDA graph and replayed synchronises the same way)
  if (threadIdx.x == 0) {
    const int gen = ld_acquire_gpu(a.flag);  // read before this block's ticket
    __threadfence();  // this block's chunk counts are visible before its ticket
    if (atomicAdd(a.ticket, 1) == (int)gridDim.x - 1) {
      *a.ticket = 0;  // every block has taken its ticket: reset for the next launch
      __threadfence();
      st_release_gpu(a.flag, gen + 1);
      s_ok = 1;
    } else {
      s_ok = wait_change(a.flag, gen, a.err) ? 1 : 0;
    }
  }
  __syncthreads();
  if (!s_ok) return;
  // 3. per expert: the running prefix over chunks (the loads are independent), the bases
  // of this block's chunks and the total
  const int G = E + a.S;
  for (int e = threadIdx.x; e < E; e += kTok) {
    int run = 0;
#pragma unroll 8
    for (int c = 0; c < a.nchunks; ++c) {
      if (c % (int)gridDim.x == (int)blockIdx.x) s_base[(c / (int)gridDim.x) * E + e] = run;
      run += __ldcg(a.chunk_hist + (size_t)c * E + e);
    }
    s_cnt[e] = run;
  }
  if (threadIdx.x == 0 && a.S) s_cnt[E] = a.T;
  __syncthreads();
  if (warp == 0) {  // exclusive scans over the groups: offsets and GEMM tile bases
    int carry_o = 0, carry_t = 0;
    for (int g0 = 0; g0 < G; g0 += 32) {
      const int g = g0 + lane;
      const int cg = (g < G) ? s_cnt[g] : 0;
      const int nt = (cg + a.BN - 1) / a.BN;
      const int io = warp_incl_scan(cg, lane);
      const int it = warp_incl_scan(nt, lane);
      if (g < G) {
        s_off[g] = carry_o + io - cg;
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
  if (blockIdx.x == 0)
    for (int g = threadIdx.x; g <= G; g += kTok) {
      a.offsets[g] = s_off[g];
      a.tile_base[g] = s_tb[g];
      if (g < G) {
        a.counts[g] = s_cnt[g];
        a.gu_done[g] = 0;  // this forward's gate/up GEMM counts its finished items here
      }
    }
  // packed rows
  for (int c = blockIdx.x, i = 0; c < a.nchunks; c += gridDim.x, ++i) {
    const int t = c * kTok + threadIdx.x;
    if (t >= a.T) continue;
    if (c == last_c) {
#pragma unroll
      for (int j = 0; j < kRouteMaxK; ++j)
        if (ex[j] >= 0) {
          const int row = s_off[ex[j]] + s_base[i * E + ex[j]] + rk[j];
          a.pos[(size_t)t * k + j] = row;
          a.perm[row] = t;
        }
    } else {
      for (int j = 0; j < k; ++j) {
        const size_t q = (size_t)t * k + j;
        const int e = __ldg(a.idx + q);
        if (e < 0 || e >= E) continue;
        const int row = s_off[e] + s_base[i * E + e] + a.pos[q];
        a.pos[q] = row;
        a.perm[row] = t;
      }
    }
    if (a.S) a.perm[(size_t)a.T * k + t] = t;
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

cudaError_t launch_routing(const LayerDims& d, int T, Workspace& ws, int num_sms, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int nchunks = (T + kTok - 1) / kTok;
  RoutingArgs a{};
  a.idx = ws.topk_idx;
  a.T = T;
  a.k = d.k;
  a.E = d.E;
  a.S = d.S;
  a.BN = d.dtype == AFD_FP8_E4M3 ? kGemmBNFp8 : bf16_tile_tokens(d, T);  // tokens per GEMM tile
  a.nchunks = nchunks;
  a.chunk_hist = ws.block_hist;
  a.counts = ws.counts;
  a.offsets = ws.offsets;
  a.tile_base = ws.tile_base;
  a.perm = ws.perm;
  a.pos = ws.pos;
  a.gu_done = ws.gu_done;
  a.ticket = ws.route_sync;
  a.flag = ws.route_sync + 1;
  a.err = ws.err;
  const int grid = nchunks < num_sms ? nchunks : num_sms;
  a.nmine = (nchunks + grid - 1) / grid;
  const size_t smem = sizeof(uint32_t) * (size_t)(kWarpsPerBlock + a.nmine) * d.E;
  if (smem > kRoutingMaxSmem) return cudaErrorInvalidValue;  // ~25M tokens: beyond any workspace here
  if (smem > 48 * 1024) {
    static std::once_flag once;
    static cudaError_t set_e = cudaSuccess;
    std::call_once(once, [] {
      set_e = cudaFuncSetAttribute(routing_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRoutingMaxSmem);
    });
    if (set_e != cudaSuccess) return set_e;
  }
  {
    const cudaError_t e_ = launch_k(routing_kernel, dim3(grid), dim3(kTok), smem, s, a);
    if (e_ != cudaSuccess) return e_;
  }
  return cudaGetLastError();
}

}  // namespace afd
