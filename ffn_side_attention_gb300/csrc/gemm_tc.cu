// gemm_tc.cu -- R4/R5: grouped expert GEMMs on the 5th-generation tensor
// cores (tcgen05.mma, accumulators in TMEM, operands staged by TMA).
//
// The expert FFN of the layer is SwiGLU (gate/up projections, SiLU-gated
// product, down projection).  "MoE系统与AFD架构概述", section 2.1, counts
// its work as 6*B*H*I FLOPs per expert pass; section 3.3 fuses the activation
// into the expert kernel.  Both GEMMs are grouped over experts: the rows of
// expert e are the packed rows offsets[e] .. offsets[e+1]-1.
//
// Swap-AB: decode batches give an expert few tokens (1..~250), so the weight
// matrix is the MMA's M side (128 weight rows per MMA) and the expert's tokens
// are the N side (16..128, padded to 16).  At create time the weights are
// re-laid as contiguous 16 KB tiles (128 output rows x 128 bytes of K, K
// blocks of one row block consecutive), so each TMA box is one sequential
// DRAM read and both operands are K-major.
//   gate/up:  D0 = Wg^T[e][i0:i0+128, :] * P[rows]^T, D1 = Wu^T[...] * P^T;
//             h[row, i] = silu(D0) * D1 -> bf16   (one CTA item = 128 channels)
//   down:     D0 = Wd^T[e][o0:o0+128, :] * h^T,   D1 = rows o0+128..o0+256
//             Y[row, o] = D -> bf16                (one CTA item = 256 columns)
// Two accumulators of up to 128 fp32 columns, double buffered (the epilogue of
// one item overlaps the MMAs of the next), fill the 512 TMEM columns.
//
// Work list: item = (group g, m tile, token tile) in that order, enumerated on
// the device from tile_base (no host sync); items of one (g, m tile) are
// adjacent so concurrently running CTAs share the weight tile in L2.  The
// kernel is persistent: grid = SM count, CTA c takes items c, c+grid, ...
// (launches of at most four rounds spread them evenly over fewer CTAs).
//
// The down launch starts before the gate/up launch ends: the gate/up epilogue
// warps count each expert's finished items (after a fence on their h stores)
// and the down token producer loads an expert's h rows once its count is
// complete, so experts whose gate/up is done proceed during the gate/up tail.
//
// Warp roles (608 threads): warp 0 lane 0 streams weight tiles into their
// own ring (L2 evict-first); warp 18 lane 0 streams the token tiles into a
// second, shallower ring (evict-last); warp 1 owns TMEM and lane 0 issues
// tcgen05.mma; warps 2-17 are the epilogue (warp w reads TMEM lanes
// 32*(w%4) .. +31; the four warps of a lane quarter take every fourth 32-token
// chunk).  With one accumulator buffer (256-token tiles) the next item's
// MMAs wait for the epilogue, so it runs on four warps per SM sub-partition
// and uses the fast exponential and division for SiLU (their error is far
// below bf16 rounding).  Separate rings keep more weight bytes in flight than a
// ring of (weights + tokens) stages would in the same shared memory: the
// weights come from HBM, the tokens from L2.  Every mbarrier wait is bounded:
// on a timeout the CTA raises its abort flag and the device error word, every
// role stops, issued copies and MMAs are drained, TMEM is freed and the kernel
// returns.
//
// Direct form (gate/up of a batch of at most kDirectMaxTok = 8 tokens): no pack
// runs.  The token producer's lanes copy the tile's rows (one lane per row) from
// the tokens' own source buffers, one 128-byte row of K per copy through
// one-row tensor maps whose 128-byte swizzle follows the shared-memory
// address, so the rows land as a 32-row box would place them.  The kernel
// builds its work list from the router's top-k itself (a bit per token per
// group), so the weight stream starts while the routing kernel still runs; it
// lets the down launch start only after that kernel has completed.
#include <cuda_bf16.h>

#include <type_traits>

#include "afd_internal.cuh"

namespace afd {
namespace {

constexpr int kRowBytes = 128;               // one 128-byte swizzle row of K
constexpr int kATile = kGemmBM * kRowBytes;  // 16 KB
constexpr int kBBoxRows = 32;                // rows per TMA box of B
constexpr int kEpiWarps = 16;
constexpr int kTokWarp = 2 + kEpiWarps;       // token producer
constexpr int kThreads = 32 * (kTokWarp + 1);  // 608
constexpr int kWTileBytes = 2 * kATile;      // one weight stage: two 128-row tiles
constexpr int kEvenRounds = 4;  // launches of at most this many item rounds share them out evenly
constexpr int kPfSteps = 4;                  // weight K blocks prefetched into L2 ahead of the loads

// Tile shape per token-tile width BN: 128 -> 5 weight + 3 token stages and
// two TMEM accumulator buffers (epilogue overlaps the next item); 256 -> 3 + 3
// stages and one accumulator buffer (an expert's <= 256 tokens share one pass
// over its weights).
template <int BN>
struct TileCfg {
  static constexpr int kWStages = BN == 256 ? 3 : 5;
  static constexpr int kXStages = 3;
  static constexpr int kBTile = BN * kRowBytes;
  static constexpr int kDynSmem = kWStages * kWTileBytes + kXStages * kBTile + 1024;
  static constexpr int kAbuf = 512 / (2 * BN);  // TMEM accumulator buffers
};
constexpr uint32_t kTmemCols = 512;
constexpr long long kDrainCycles = 400000000ll;  // ~0.2 s

struct TcArgs {
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* tile_base;
  int G;                 // groups: routed experts + shared
  int num_kb;            // K / 64
  int MT;                // m tiles per group
  int a_rows_per_group;  // A rows per group (I for gate/up, H for down)
  int a_mt_stride;       // A rows per m tile (128 gate/up, 256 down)
  int a1_offset;         // A1 rows relative to A0 (0: other map; 128: same map)
  uint16_t* out;         // bf16 [rows, ld_out]
  int ld_out;
  int mode;              // 0: SwiGLU(D0, D1) ; 1: D0 | D1 as two column blocks
  int* err;
  // Per-group progress of the gate/up launch: mode 0 adds one per epilogue warp per item
  // once that warp's h stores are visible; mode 1 (down) loads a group's h rows once the
  // count reaches kEpiWarps * done_mt * (its token tiles), instead of waiting for the
  // whole gate/up grid.  Null: mode 1 waits for the previous grid.
  int32_t* done;
  int done_mt;           // gate/up items per token tile (I / 128)
};

// Kernel parameter of the direct form (sources' one-row maps) or an empty stand-in.
struct NoSrc {};
template <bool DIRECT>
using SrcParam = typename std::conditional<DIRECT, DirectSrc, NoSrc>::type;

struct Item {
  int g, mt, row0, nrows;
};

template <int BN>
__device__ __forceinline__ Item decode_item(int item, int MT, int G, const int* tb, const int* off,
                                            const int* cnt) {
  int lo = 0, hi = G - 1;  // last g with MT * tb[g] <= item
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (MT * tb[mid] <= item) lo = mid; else hi = mid - 1;
  }
  Item it;
  it.g = lo;
  const int nt_g = tb[lo + 1] - tb[lo];
  const int local = item - MT * tb[lo];
  it.mt = local / nt_g;
  const int nt = local - it.mt * nt_g;
  it.row0 = off[lo] + nt * BN;
  it.nrows = min(BN, cnt[lo] - nt * BN);
  return it;
}


// SwiGLU's sigmoid with one special-function op per value.  The gate/up epilogue of a
// 256-token tile does not overlap the MMA (one TMEM accumulator), and two such ops per
// value (exponential and reciprocal) made it bound by that unit: qwen3 shapes, T = 3160,
// gate/up 584 -> 573 us with the reciprocal below.
__device__ __forceinline__ float ex2_f32(float x) {  // 2^x
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// 1/d for d in [1, 2] by Newton-Raphson division: the linear initial estimate
// 24/17 - 8/17 d (relative error at most 1/17 on [1, 2]) and three steps
// y += y (1 - d y), each squaring the relative error: (1/17)^8 < 2^-32.
__device__ __forceinline__ float2 rcp_newton_1_2(float2 d) {
  const float2 c0 = make_float2(24.0f / 17.0f, 24.0f / 17.0f), c1 = make_float2(-8.0f / 17.0f, -8.0f / 17.0f);
  const float2 one = make_float2(1.0f, 1.0f), nd = make_float2(-d.x, -d.y);
  float2 y = __ffma2_rn(c1, d, c0);
#pragma unroll
  for (int i = 0; i < 3; ++i) y = __ffma2_rn(y, __ffma2_rn(nd, y, one), y);
  return y;
}

__device__ __forceinline__ uint16_t f2bf(float v) {
  __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t*>(&b);
}

template <int BN, bool DIRECT>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                     const __grid_constant__ CUtensorMap tmB, const TcArgs args,
                     const __grid_constant__ SrcParam<DIRECT> ds) {
  // Dependent launch: this kernel starts only after the previous one (the pack,
  // or the gate/up GEMM) has passed its own wait, so the routing tables are final
  // and the weights are constant: the weight producer streams at once, and only
  // the token producer waits for the previous kernel's output (P or h).  The
  // epilogue writes (h, Y) are read by nothing that can still be running.
  // Direct form (no pack): the previous kernel is the routing kernel, which started
  // once the router had completed; this kernel reads only the router's top-k and the
  // sources before its wait on that kernel (below).
  if constexpr (!DIRECT) pdl_trigger();
  constexpr int kWS = TileCfg<BN>::kWStages, kXS = TileCfg<BN>::kXStages, kBTile = TileCfg<BN>::kBTile;
  constexpr uint32_t kAbuf = TileCfg<BN>::kAbuf;
  extern __shared__ uint8_t dyn_smem[];
  uint8_t* smem = dyn_smem + ((1024u - (smem_u32(dyn_smem) & 1023u)) & 1023u);
  uint8_t* wsm = smem;                     // [kWS][2 x 16 KB]
  uint8_t* xsm = smem + kWS * kWTileBytes;  // [kXS][BN x 128 B]

  __shared__ __align__(8) uint64_t bars[2 * kWS + 2 * kXS + 5];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_tb[kMaxExperts + 1], s_off[kMaxExperts + 1], s_cnt[kMaxExperts];
  __shared__ uint32_t s_mask[DIRECT ? kMaxExperts : 1];  // direct form: each group's tokens
  uint64_t* wfull = bars;
  uint64_t* wempty = bars + kWS;
  uint64_t* xfull = bars + 2 * kWS;
  uint64_t* xempty = xfull + kXS;
  uint64_t* tfull = xempty + kXS;        // [2] accumulator buffer ready for the epilogue
  uint64_t* tempty = tfull + 2;          // [2] accumulator buffer drained by the epilogue
  uint64_t* drain = tfull + 4;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = args.G;
  if constexpr (DIRECT) {
    // The routing tables of this batch, built from the router's top-k (complete: the
    // routing kernel that launched this grid waited for it), as the routing kernel builds
    // them: per group a bit per token, counts, offsets and tile bases by a warp scan.
    for (int g = threadIdx.x; g < G; g += kThreads) s_mask[g] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < ds.T * ds.k; i += kThreads) {
      const int e = ds.topk_idx[i];
      if (e >= 0 && e < ds.E) atomicOr(&s_mask[e], 1u << (i / ds.k));
    }
    if (ds.S && threadIdx.x == 0) s_mask[ds.E] = ds.T >= 32 ? ~0u : (1u << ds.T) - 1u;
    __syncthreads();
    if (warp == 0) {
      const int c = (G + 31) / 32;
      int rows = 0, tiles = 0;
      for (int i = 0; i < c; ++i) {
        const int g = lane * c + i;
        if (g < G) {
          const int n = __popc(s_mask[g]);
          rows += n;
          tiles += (n + BN - 1) / BN;
        }
      }
      int ir = rows, it = tiles;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, ir, o), b = __shfl_up_sync(0xffffffffu, it, o);
        if (lane >= o) {
          ir += a;
          it += b;
        }
      }
      int row = ir - rows, tile = it - tiles;
      for (int i = 0; i < c; ++i) {
        const int g = lane * c + i;
        if (g < G) {
          const int n = __popc(s_mask[g]);
          s_off[g] = row;
          s_tb[g] = tile;
          s_cnt[g] = n;
          row += n;
          tile += (n + BN - 1) / BN;
        }
      }
      if (lane == 31) {
        s_off[G] = row;
        s_tb[G] = tile;
      }
    }
  } else {
    for (int g = threadIdx.x; g <= G; g += kThreads) {
      s_tb[g] = args.tile_base[g];
      s_off[g] = args.offsets[g];
      if (g < G) s_cnt[g] = args.counts[g];
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kWS; ++s) {
      mbar_init(&wfull[s], 1);
      mbar_init(&wempty[s], 1);
    }
    for (int s = 0; s < kXS; ++s) {
      mbar_init(&xfull[s], 1);
      mbar_init(&xempty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kEpiWarps);
    }
    mbar_init(drain, 1);
    s_abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA0);
    tma_prefetch_desc(&tmA1);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int total = args.MT * s_tb[G];
  // Equal rounds for short launches: with R = ceil(total / grid) <= kEvenRounds rounds, only
  // ceil(total / R) CTAs take items, R (or R - 1) each, instead of a last round where a few
  // SMs stream one more item each at the rate one SM reaches alone.  With more rounds that
  // tail is a small share and the SMs left idle would cost more than it.
  const int rounds = total > 0 ? (total + (int)gridDim.x - 1) / (int)gridDim.x : 1;
  const int nact = rounds <= kEvenRounds ? (total + rounds - 1) / rounds : (int)gridDim.x;
  const int first = (int)blockIdx.x < nact ? (int)blockIdx.x : total;  // idle CTAs take none
  volatile int* abort = &s_abort;
  // Direct form: the down launch reads the routing kernel's tables as it starts, so this
  // grid lets it launch only once that kernel has completed: every thread waits for it and
  // then triggers; the two producers do so once their first stages are issued.
  if constexpr (DIRECT)
    if (!(warp == 0 && lane == 0) && warp != kTokWarp) {
      pdl_wait();
      pdl_trigger();
    }

  if (DIRECT && warp == kTokWarp) {
    if constexpr (DIRECT) {
      // ---------------- token producer, direct form: lane r copies row r of the item's
      // tile from its token's source, one 128-byte row of K per copy (a group holds at
      // most kDirectMaxTok rows, and the warp takes up to 32).  Rows past nrows keep stale
      // contents: they feed only accumulator columns that no epilogue thread stores.
      const uint64_t pol = l2_policy_evict_last();
      int s = 0, issued = 0;
      uint32_t ph = 0, filled = 0, fill_ph = 0;
      bool ok = true;
      for (int item = first; ok && item < total; item += nact) {
        const Item it = decode_item<BN>(item, args.MT, G, s_tb, s_off, s_cnt);
        if (it.nrows > 32) {  // not reachable from a batch of at most kDirectMaxTok tokens
          if (lane == 0) {
            *abort = 1;
            atomicOr(args.err, kErrRange);
          }
          ok = false;
          break;
        }
        const CUtensorMap* map = nullptr;
        int row = 0;
        if (lane < it.nrows) {
          uint32_t m = s_mask[it.g];  // the group's rows are its tokens in ascending order
          for (int j = it.row0 - s_off[it.g] + lane; j > 0; --j) m &= m - 1u;
          const int t = __ffs(m) - 1;
          int lo = 0, hi = ds.M - 1;  // last source m with row0[m] <= t
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (ds.row0[mid] <= t) lo = mid; else hi = mid - 1;
          }
          map = &ds.maps.m[lo];
          row = t - ds.row0[lo];
        }
        for (int kb = 0; kb < args.num_kb; ++kb) {
          int go = 1;
          if (lane == 0) {
            go = mbar_wait(&xempty[s], ph ^ 1u, abort, args.err);
            if (go) mbar_arrive_expect_tx(&xfull[s], (uint32_t)(it.nrows * kRowBytes));
          }
          if (!__shfl_sync(0xffffffffu, go, 0)) {
            ok = false;
            break;
          }
          if (lane < it.nrows)
            tma_load_2d_hint(xsm + s * kBTile + lane * kRowBytes, map, &xfull[s], kb * 64, row, pol);
          filled |= 1u << s;
          fill_ph = (fill_ph & ~(1u << s)) | (ph << s);
          if (++s == kXS) {
            s = 0;
            ph ^= 1u;
          }
          if (++issued == kXS) {
            pdl_wait();
            pdl_trigger();
          }
        }
      }
      if (issued < kXS) {
        pdl_wait();
        pdl_trigger();
      }
      if (!ok && lane == 0)  // let the copies already issued land before the CTA exits
        for (int q = 0; q < kXS; ++q)
          if ((filled >> q) & 1u) mbar_wait_cycles(&xfull[q], (fill_ph >> q) & 1u, kDrainCycles);
    }
  } else if (warp == 0 || warp == kTokWarp) {
    if (lane == 0) {
      // ---------------- TMA producers: warp 0 weights, warp kTokWarp tokens
      const bool wprod = warp == 0;
      const int nst = wprod ? kWS : kXS;
      uint64_t* fb = wprod ? wfull : xfull;
      uint64_t* eb = wprod ? wempty : xempty;
      const uint64_t pol = wprod ? l2_policy_evict_first() : l2_policy_evict_last();
      // the token operand is the previous kernel's output: the whole grid (gate/up, after the
      // pack) or, for down with progress counters, each group's gate/up items (below)
      const bool per_group = args.mode == 1 && args.done != nullptr;
      if (!wprod && !per_group) pdl_wait();
      int ready_g = -1;
      int s = 0;
      uint32_t ph = 0, filled = 0, fill_ph = 0;
      bool ok = true;
      // tiled weights: tile (row block rb, K block kb) starts at tile row (rb * num_kb + kb) * 128
      auto row_blocks = [&](const Item& it, int& rb0, int& rb1) {
        rb0 = it.g * (args.a_rows_per_group / 128) + it.mt * (args.a_mt_stride / 128);
        rb1 = rb0 + args.a1_offset / 128;
      };
      // L2 prefetch cursor (weights only): runs kPfSteps K blocks ahead of the loads
      int pf_item = first, pf_kb = 0, pf_rb0 = 0, pf_rb1 = 0;
      long pf_n = 0, ld_n = 0;
      if (wprod && pf_item < total) row_blocks(decode_item<BN>(pf_item, args.MT, G, s_tb, s_off, s_cnt), pf_rb0, pf_rb1);
      for (int item = first; ok && item < total; item += nact) {
        const Item it = decode_item<BN>(item, args.MT, G, s_tb, s_off, s_cnt);
        int rb0, rb1;
        row_blocks(it, rb0, rb1);
        const int nbox = (it.nrows + kBBoxRows - 1) / kBBoxRows;
        const uint32_t bytes = wprod ? (uint32_t)kWTileBytes : (uint32_t)(nbox * kBBoxRows * kRowBytes);
        if (!wprod && per_group && it.g != ready_g) {
          const int target = kEpiWarps * args.done_mt * (s_tb[it.g + 1] - s_tb[it.g]);
          if (!wait_count(args.done + it.g, target, abort, args.err)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();  // the TMA reads below see the h rows the count covers
          ready_g = it.g;
        }
        for (int kb = 0; kb < args.num_kb; ++kb, ++ld_n) {
          if (wprod)
            for (; pf_n <= ld_n + kPfSteps && pf_item < total; ++pf_n) {
              tma_prefetch_l2_2d(&tmA0, 0, (pf_rb0 * args.num_kb + pf_kb) * 128);
              tma_prefetch_l2_2d(&tmA1, 0, (pf_rb1 * args.num_kb + pf_kb) * 128);
              if (++pf_kb == args.num_kb) {
                pf_kb = 0;
                pf_item += nact;
                if (pf_item < total)
                  row_blocks(decode_item<BN>(pf_item, args.MT, G, s_tb, s_off, s_cnt), pf_rb0, pf_rb1);
              }
            }
          if (!mbar_wait(&eb[s], ph ^ 1u, abort, args.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&fb[s], bytes);
          if (DIRECT && wprod && ld_n + 1 == kWS) {
            pdl_wait();
            pdl_trigger();
          }
          if (wprod) {
            uint8_t* st = wsm + s * kWTileBytes;
            tma_load_2d_hint(st, &tmA0, &fb[s], 0, (rb0 * args.num_kb + kb) * 128, pol);
            tma_load_2d_hint(st + kATile, &tmA1, &fb[s], 0, (rb1 * args.num_kb + kb) * 128, pol);
          } else {
            uint8_t* st = xsm + s * kBTile;
            for (int b = 0; b < nbox; ++b)
              tma_load_2d_hint(st + b * kBBoxRows * kRowBytes, &tmB, &fb[s], kb * 64, it.row0 + b * kBBoxRows, pol);
          }
          filled |= 1u << s;
          fill_ph = (fill_ph & ~(1u << s)) | (ph << s);
          if (++s == nst) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (DIRECT && wprod && ld_n < kWS) {  // fewer loads than the first ring: wait now
        pdl_wait();
        pdl_trigger();
      }
      if (!ok)  // let the copies already issued land before the CTA exits
        for (int q = 0; q < nst; ++q)
          if ((filled >> q) & 1u) mbar_wait_cycles(&fb[q], (fill_ph >> q) & 1u, kDrainCycles);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      int ws_ = 0, xs = 0;
      uint32_t wph = 0, xph = 0, ic = 0;
      bool ok = true;
      for (int item = first; ok && item < total; item += nact, ++ic) {
        const Item it = decode_item<BN>(item, args.MT, G, s_tb, s_off, s_cnt);
        const int N = (it.nrows + 15) & ~15;
        const uint32_t idesc = mma_idesc(1u, kGemmBM, N);
        const uint32_t a = ic % kAbuf;  // accumulator buffer of this item
        if (!mbar_wait(&tempty[a], ((ic / kAbuf) & 1u) ^ 1u, abort, args.err)) break;
        tc_fence_after();
        const uint32_t d0 = tmem + a * (2u * BN), d1 = d0 + BN;
        for (int kb = 0; kb < args.num_kb; ++kb) {
          if (!mbar_wait(&wfull[ws_], wph, abort, args.err) || !mbar_wait(&xfull[xs], xph, abort, args.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint8_t* st = wsm + ws_ * kWTileBytes;
          const uint64_t da0 = sw128_desc(st);
          const uint64_t da1 = sw128_desc(st + kATile);
          const uint64_t db = sw128_desc(xsm + xs * kBTile);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // 4 x K=16 per 128-byte row
            const uint32_t acc = (kb | kk) ? 1u : 0u;
            mma_f16(d0, da0 + 2 * kk, db + 2 * kk, idesc, acc);
            mma_f16(d1, da1 + 2 * kk, db + 2 * kk, idesc, acc);
          }
          tc_commit(&wempty[ws_]);
          tc_commit(&xempty[xs]);
          if (++ws_ == kWS) {
            ws_ = 0;
            wph ^= 1u;
          }
          if (++xs == kXS) {
            xs = 0;
            xph ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&tfull[a]);
      }
      tc_commit(drain);  // all MMAs issued above complete before TMEM is freed
      mbar_wait_cycles(drain, 0, kDrainCycles);
    }
  } else if (warp >= 2 && warp < 2 + kEpiWarps) {
    // ---------------- epilogue: warps 2..17
    const int quad = warp & 3, part = (warp - 2) >> 2;  // lane quarter; which of every 4 chunks
    const int r = quad * 32 + lane;  // row of the 128-row MMA tile
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    uint32_t ic = 0;
    for (int item = first; item < total; item += nact, ++ic) {
      const Item it = decode_item<BN>(item, args.MT, G, s_tb, s_off, s_cnt);
      const uint32_t a = ic % kAbuf;
      if (!mbar_wait(&tfull[a], (ic / kAbuf) & 1u, abort, args.err)) break;
      tc_fence_after();
      const uint32_t t_buf = t_lane + a * (2u * BN);
      for (int c = 32 * part; c < it.nrows; c += 32 * (kEpiWarps / 4)) {
        float d0[32], d1[32];
        tmem_ld_32x32b_x32(t_buf + (uint32_t)c, d0);
        tmem_ld_32x32b_x32(t_buf + (uint32_t)(BN + c), d1);
        tmem_ld_wait();
        const int nn = min(32, it.nrows - c);
        // one output row per token: this thread writes column (m tile, r) of rows row0+c .. +nn-1
        uint16_t* o = args.out + (size_t)(it.row0 + c) * args.ld_out +
                      (args.mode == 0 ? it.mt * kGemmBM : it.mt * 2 * kGemmBM) + r;
        if (args.mode == 0) {
          constexpr float kLog2e = 1.4426950408889634f;
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            // sigmoid(g) = 1 / (1 + e) for g >= 0 and e / (1 + e) otherwise, e = e^-|g| in (0, 1]:
            // one special-function op per value (the exponential), the reciprocal on the FMA pipe
            const float2 g = make_float2(d0[j], d0[j + 1]);
            const float2 e = make_float2(ex2_f32(-fabsf(g.x) * kLog2e), ex2_f32(-fabsf(g.y) * kLog2e));
            const float2 r = rcp_newton_1_2(make_float2(1.0f + e.x, 1.0f + e.y));
            const float s0 = g.x >= 0.0f ? r.x : e.x * r.x, s1 = g.y >= 0.0f ? r.y : e.y * r.y;
            if (j < nn) *o = f2bf(g.x * s0 * d1[j]);
            o += args.ld_out;
            if (j + 1 < nn) *o = f2bf(g.y * s1 * d1[j + 1]);
            o += args.ld_out;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (j < nn) {
              o[0] = f2bf(d0[j]);
              o[kGemmBM] = f2bf(d1[j]);
            }
            o += args.ld_out;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[a]);
      if (args.mode == 0 && args.done != nullptr) {  // this warp's h stores of the item are out
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(args.done + it.g, 1);
      }
    }
  }

  // The per-group down launch reads h through the progress counters and never waits for
  // the gate/up grid as a whole.  When it completes normally every gate/up increment has
  // been made (each group's count reached its total), so nothing of that grid can touch
  // the counters after the next forward's routing zeroes them.  A CTA that gave up (a
  // bounded wait ran out) waits for the previous grid before it exits, so "this kernel
  // complete implies every earlier kernel complete" holds on that path too.  (An exit
  // wait in every thread on every path cost 2.7% of the step at T=3160.)
  __syncthreads();
  if (threadIdx.x == 0 && *abort) pdl_wait();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t gemm_tc_setup() {
  cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel<128, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       TileCfg<128>::kDynSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_bf16_kernel<128, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             TileCfg<128>::kDynSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(gemm_bf16_kernel<256, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              TileCfg<256>::kDynSmem);
}

template <int BN>
static cudaError_t launch_bn(const LayerDims& d, int T, const TcWeights& w, Workspace& ws, int num_sms,
                             cudaStream_t s, int which, const DirectSrc* direct) {
  const int G = d.E + d.S;
  const long rows = (long)T * (d.k + d.S);
  const long tiles_ub = rows / BN + G + 1;
  TcArgs a{};
  a.counts = ws.counts;
  a.offsets = ws.offsets;
  a.tile_base = ws.tile_base;
  a.G = G;
  a.err = ws.err;
  const CUtensorMap *m0, *m1, *mb;
  if (which == 0) {  // gate/up + SwiGLU: K = H, items of 128 intermediate channels
    a.num_kb = d.H / 64;
    a.MT = d.I / kGemmBM;
    a.a_rows_per_group = d.I;
    a.a_mt_stride = kGemmBM;
    a.a1_offset = 0;
    a.out = static_cast<uint16_t*>(ws.Hb);
    a.ld_out = d.I;
    a.mode = 0;
    a.done = ws.gu_done;
    m0 = w.tm_wg;
    m1 = w.tm_wu;
    mb = &ws.tm_P;
  } else {  // down: K = I, items of 256 output columns (two 128-row MMAs)
    a.num_kb = d.I / 64;
    a.MT = d.H / (2 * kGemmBM);
    a.a_rows_per_group = d.H;
    a.a_mt_stride = 2 * kGemmBM;
    a.a1_offset = kGemmBM;
    a.out = static_cast<uint16_t*>(ws.Y);
    a.ld_out = d.H;
    a.mode = 1;
    a.done = ws.gu_done;
    a.done_mt = d.I / kGemmBM;
    m0 = w.tm_wd;
    m1 = w.tm_wd;
    mb = &ws.tm_H;
  }
  const long items_ub = tiles_ub * a.MT;
  const int grid = (int)(items_ub < num_sms ? items_ub : num_sms);
  cudaError_t e_;
  if constexpr (BN == 128) {
    if (direct)
      e_ = launch_k(gemm_bf16_kernel<128, true>, dim3(grid), dim3(kThreads), TileCfg<128>::kDynSmem, s, *m0, *m1,
                    *mb, a, *direct);
    else
      e_ = launch_k(gemm_bf16_kernel<128, false>, dim3(grid), dim3(kThreads), TileCfg<128>::kDynSmem, s, *m0,
                    *m1, *mb, a, NoSrc{});
  } else {
    if (direct) return cudaErrorInvalidValue;
    e_ = launch_k(gemm_bf16_kernel<BN, false>, dim3(grid), dim3(kThreads), TileCfg<BN>::kDynSmem, s, *m0, *m1, *mb,
                  a, NoSrc{});
  }
  if (e_ != cudaSuccess) return e_;
  return cudaGetLastError();
}

int bf16_tile_tokens(const LayerDims& d, int T) {
  // one pass over an expert's weights for its tokens when they are many
  return (long)T * d.k > 112L * d.E ? 256 : 128;
}

cudaError_t launch_gemm_tc(const LayerDims& d, int T, const TcWeights& w, Workspace& ws, int num_sms,
                           cudaStream_t s, int which, const DirectSrc* direct) {
  if (T == 0) return cudaSuccess;
  if (d.dtype != AFD_BF16) return cudaErrorNotSupported;
  if (direct && (which != 0 || T > kDirectMaxTok)) return cudaErrorInvalidValue;
  return bf16_tile_tokens(d, T) == 256 ? launch_bn<256>(d, T, w, ws, num_sms, s, which, direct)
                                       : launch_bn<128>(d, T, w, ws, num_sms, s, which, direct);
}

}  // namespace afd
