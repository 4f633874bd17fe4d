// gemm_fp8.cu -- R4/R5 for the fp8 layer: grouped expert GEMMs on e4m3
// operands (tcgen05.mma kind::f8f6f4) with fp32 block scales.
//
// FP8 experts ("大模型推理的内存与计算解耦：AFD 架构解析与性能验证", section 1:
// the MoE FFN runs as an fp8 grouped GEMM; "MoE系统与AFD架构概述", section
// 3.3: FP8 activations).  Weights carry one fp32 scale per 128x128 block,
// activations one per token per 128 channels, so the product of one 128-wide
// K block is
//     sW[m-block, kb] * sA[token, kb] * sum_{k in kb} qW[m, k] * qA[token, k]
// and the result is the sum of those over kb.  The tensor core computes the
// inner sums; the scales are applied in fp32 ("promotion"):
//   * one pipeline stage = one K block (128 bytes of e4m3 per row);
//   * the MMA writes each block's partial into one of two TMEM buffers
//     (ping-pong), accumulating only inside the block;
//   * eight epilogue warps read the partial, multiply by sW * sA[token] and
//     add it to fp32 accumulators held in registers (warp w covers TMEM lanes
//     32*(w%4) .. +31 and half of the 128 token columns); the producer
//     warpgroup gives registers up (setmaxnreg) so the 128 accumulators of an
//     epilogue thread stay in registers;
//   * after the last block: gate/up -> h = silu(G) * U, re-quantised per token
//     per 128 channels of I (scale = amax/448, e4m3 RNE, saturating); down ->
//     Y in bf16.
// Tiles: 128 weight rows per MMA (two accumulators: gate+up, or two halves of
// 256 down rows), up to 128 tokens per tile; TMEM = 2 buffers x 2 accumulators
// x 128 columns.  TMA ring of 4 stages x 48 KB.  Same device-side work list,
// persistent CTAs and bounded waits as the bf16 kernel.
#include <cuda_bf16.h>

#include "afd_internal.cuh"

namespace afd {
namespace {

constexpr int kBN = kGemmBNFp8;                   // 128 tokens per tile
constexpr int kStages = 4;
constexpr int kRowBytes = 128;                    // one K block of e4m3
constexpr int kATile = kGemmBM * kRowBytes;       // 16 KB
constexpr int kBTile = kBN * kRowBytes;           // 16 KB
constexpr int kBBoxRows = 32;
constexpr int kStageBytes = 2 * kATile + kBTile;  // 48 KB
constexpr int kDynSmem = kStages * kStageBytes + 1024;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 128 + 32 * kEpiWarps;  // 384: warpgroup 0 = producer, MMA, 2 idle; 1-2 = epilogue
constexpr int kRegsLow = 56;                    // setmaxnreg of warpgroup 0
constexpr int kRegsHigh = 224;                  // setmaxnreg of the epilogue warpgroups
// The split must fit in what the block is launched with:
// 128 * kRegsLow + 256 * kRegsHigh <= 384 * (registers per thread at launch).
constexpr int kRegsNeeded = (128 * kRegsLow + 256 * kRegsHigh + kThreads - 1) / kThreads;  // 168
constexpr uint32_t kTmemCols = 512;
constexpr long long kDrainCycles = 400000000ll;  // ~0.2 s
constexpr int kMaxKb = 56;                        // K blocks per GEMM (K <= 7168)

struct Fp8Args {
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* tile_base;
  int G;
  int num_kb;            // K / 128
  int MT;                // m tiles per group
  int a_rows_per_group;
  int a_mt_stride;
  int a1_offset;
  const float* sA0;      // weight block scales of A0: [G][a_rows_per_group/128][num_kb]
  const float* sA1;
  int sa1_block_offset;  // A1's 128-row block relative to A0's (0: own scale array; 1: next block)
  const float* sB;       // activation scales [rows][num_kb]
  void* out;             // mode 0: e4m3 codes [rows][ld_out]; mode 1: bf16 [rows][ld_out]
  float* out_scale;      // mode 0: [rows][ld_out/128]
  int ld_out;
  int mode;
  int* err;
};

struct Item {
  int g, mt, row0, nrows;
};

__device__ __forceinline__ Item decode_item(int item, int MT, int G, const int* tb, const int* off, const int* cnt) {
  int lo = 0, hi = G - 1;  // last g with MT * tb[g] <= item
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (MT * tb[mid] <= item) lo = mid; else hi = mid - 1;
  }
  Item it;
  it.g = lo;
  const int nt_g = tb[lo + 1] - tb[lo];
  const int local = item - MT * tb[lo];
  it.mt = local / nt_g;
  const int nt = local - it.mt * nt_g;
  it.row0 = off[lo] + nt * kBN;
  it.nrows = min(kBN, cnt[lo] - nt * kBN);
  return it;
}

__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ uint8_t cvt_e4m3(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return (uint8_t)(r & 0xff);
}

__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow)); }
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh)); }

// Barrier of the eight epilogue warps on an mbarrier (count 8, one arrival
// per warp), with the same bounded wait as every other wait of the kernel.
__device__ __forceinline__ bool epi_sync(uint64_t* bar, uint32_t& phase, int lane, volatile int* abort, int* err) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
  const bool ok = mbar_wait(bar, phase, abort, err);
  phase ^= 1u;
  __syncwarp();
  return ok;
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                    const __grid_constant__ CUtensorMap tmB, const Fp8Args args) {
  extern __shared__ uint8_t dyn_smem[];
  uint8_t* smem = dyn_smem + ((1024u - (smem_u32(dyn_smem) & 1023u)) & 1023u);

  __shared__ __align__(8) uint64_t bars[2 * kStages + 6];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_tb[kMaxExperts + 1], s_off[kMaxExperts + 1], s_cnt[kMaxExperts];
  __shared__ float s_red[2][4][64];  // per column half, quadrant, column: |h| maxima
  __shared__ __align__(16) float s_sc[kMaxKb][kBN];  // this item's activation scales, [kb][token column]
  __shared__ float s_w[2][kMaxKb];                   // this item's weight block scales (A0, A1)
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* pfull = bars + 2 * kStages;       // [2] MMA -> epilogue
  uint64_t* pempty = bars + 2 * kStages + 2;  // [2] epilogue -> MMA
  uint64_t* drain = bars + 2 * kStages + 4;
  uint64_t* ebar = bars + 2 * kStages + 5;    // epilogue warps' own barrier

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = args.G;
  for (int g = threadIdx.x; g <= G; g += kThreads) {
    s_tb[g] = args.tile_base[g];
    s_off[g] = args.offsets[g];
    if (g < G) s_cnt[g] = args.counts[g];
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&pfull[b], 1);
      mbar_init(&pempty[b], kEpiWarps);
    }
    mbar_init(drain, 1);
    mbar_init(ebar, kEpiWarps);
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
  volatile int* abort = &s_abort;

  if (warp < 4) {
    regs_dec();
    if (warp == 0 && lane == 0) {
      // ---------------- TMA producer
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_b = l2_policy_evict_last();
      int s = 0;
      uint32_t ph = 0, filled = 0, fill_ph = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
        const Item it = decode_item(item, args.MT, G, s_tb, s_off, s_cnt);
        // tiled weights: tile (row block rb, K block kb) starts at tile row (rb * num_kb + kb) * 128
        const int rb0 = it.g * (args.a_rows_per_group / 128) + it.mt * (args.a_mt_stride / 128);
        const int rb1 = rb0 + args.a1_offset / 128;
        const int nbox = (it.nrows + kBBoxRows - 1) / kBBoxRows;
        const uint32_t bytes = 2 * kATile + nbox * kBBoxRows * kRowBytes;
        for (int kb = 0; kb < args.num_kb; ++kb) {
          if (!mbar_wait(&empty[s], ph ^ 1u, abort, args.err)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + s * kStageBytes;
          mbar_arrive_expect_tx(&full[s], bytes);
          tma_load_2d_hint(st, &tmA0, &full[s], 0, (rb0 * args.num_kb + kb) * 128, pol_w);
          tma_load_2d_hint(st + kATile, &tmA1, &full[s], 0, (rb1 * args.num_kb + kb) * 128, pol_w);
          for (int b = 0; b < nbox; ++b)
            tma_load_2d_hint(st + 2 * kATile + b * kBBoxRows * kRowBytes, &tmB, &full[s], kb * 128,
                             it.row0 + b * kBBoxRows, pol_b);
          filled |= 1u << s;
          fill_ph = (fill_ph & ~(1u << s)) | (ph << s);
          if (++s == kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok)  // let the copies already issued land before the CTA exits
        for (int q = 0; q < kStages; ++q)
          if ((filled >> q) & 1u) mbar_wait_cycles(&full[q], (fill_ph >> q) & 1u, kDrainCycles);
    } else if (warp == 1 && lane == 0) {
      // ---------------- MMA issuer: one fresh partial per K block
      int s = 0;
      uint32_t ph = 0, gstep = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
        const Item it = decode_item(item, args.MT, G, s_tb, s_off, s_cnt);
        const int N = (it.nrows + 15) & ~15;
        const uint32_t idesc = mma_idesc(0u, kGemmBM, N);  // e4m3 x e4m3 -> f32
        for (int kb = 0; kb < args.num_kb; ++kb, ++gstep) {
          const uint32_t b = gstep & 1u, use = gstep >> 1;
          if (!mbar_wait(&pempty[b], (use & 1u) ^ 1u, abort, args.err) ||
              !mbar_wait(&full[s], ph, abort, args.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint8_t* st = smem + s * kStageBytes;
          const uint64_t da0 = sw128_desc(st), da1 = sw128_desc(st + kATile), db = sw128_desc(st + 2 * kATile);
          const uint32_t d0 = tmem + b * 256u, d1 = d0 + 128u;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // 4 x K=32 per 128-byte block
            mma_f8(d0, da0 + 2 * kk, db + 2 * kk, idesc, kk ? 1u : 0u);
            mma_f8(d1, da1 + 2 * kk, db + 2 * kk, idesc, kk ? 1u : 0u);
          }
          tc_commit(&empty[s]);
          tc_commit(&pfull[b]);
          if (++s == kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      tc_commit(drain);  // all MMAs issued above complete before TMEM is freed
      mbar_wait_cycles(drain, 0, kDrainCycles);
    }
  } else {
    regs_inc();
    // ---------------- epilogue: warps 4..11
    const int ew = warp - 4;
    const int quad = warp & 3, half = ew >> 2;
    const int r = quad * 32 + lane;  // row of the 128-row tile
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    uint32_t gstep = 0, ephase = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
      const Item it = decode_item(item, args.MT, G, s_tb, s_off, s_cnt);
      const int c0 = half * 64;
      const int nc = max(0, min(64, it.nrows - c0));  // this warp's columns
      const int nkb = args.num_kb;
      // stage the item's scales in shared memory (the previous item is done with them)
      if (!epi_sync(ebar, ephase, lane, abort, args.err)) break;
      {
        const size_t blk0 = (size_t)it.g * (args.a_rows_per_group / 128) + it.mt * (args.a_mt_stride / 128);
        const float* sB = args.sB + (size_t)it.row0 * nkb;  // rows row0 .. row0+nrows-1 are contiguous
        for (int q = ew * 32 + lane; q < it.nrows * nkb; q += 32 * kEpiWarps) {
          const int col = q / nkb, kb = q - col * nkb;
          s_sc[kb][col] = __ldg(sB + q);
        }
        for (int q = ew * 32 + lane; q < 2 * nkb; q += 32 * kEpiWarps) {
          const int which = q / nkb, kb = q - which * nkb;
          s_w[which][kb] = __ldg((which ? args.sA1 + (blk0 + args.sa1_block_offset) * nkb : args.sA0 + blk0 * nkb) + kb);
        }
      }
      if (!epi_sync(ebar, ephase, lane, abort, args.err)) break;
      float acc0[64], acc1[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) acc0[j] = acc1[j] = 0.0f;
      for (int kb = 0; kb < nkb; ++kb, ++gstep) {
        const uint32_t b = gstep & 1u, use = gstep >> 1;
        if (!mbar_wait(&pfull[b], use & 1u, abort, args.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float w0 = s_w[0][kb], w1 = s_w[1][kb];
#pragma unroll
        for (int cc = 0; cc < 64; cc += 32) {
          if (cc < nc) {
            float p0[32], p1[32];
            const uint32_t col = t_lane + b * 256u + (uint32_t)(c0 + cc);
            tmem_ld_x16(col, p0);
            tmem_ld_x16(col + 16u, p0 + 16);
            tmem_ld_x16(col + 128u, p1);
            tmem_ld_x16(col + 144u, p1 + 16);
            tmem_ld_wait();
            const float4* sc4 = reinterpret_cast<const float4*>(&s_sc[kb][c0 + cc]);
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
              const float4 sa = sc4[j4];
              const float sv[4] = {sa.x, sa.y, sa.z, sa.w};
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int j = 4 * j4 + u;
                acc0[cc + j] = fmaf(w0 * sv[u], p0[j], acc0[cc + j]);
                acc1[cc + j] = fmaf(w1 * sv[u], p1[j], acc1[cc + j]);
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pempty[b]);
      }
      if (!ok) break;
      // ---- item epilogue
      if (args.mode == 0) {
        // h = silu(G) * U, then e4m3 per token per 128 channels (this tile's rows)
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const float g = acc0[j];
          acc0[j] = g / (1.0f + expf(-g)) * acc1[j];
        }
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          float a = fabsf(acc0[j]);
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
          if (lane == 0) s_red[half][quad][j] = a;
        }
        if (!epi_sync(ebar, ephase, lane, abort, args.err)) break;
        uint8_t* outq = static_cast<uint8_t*>(args.out);
        const int nblk = args.ld_out / 128;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          if (j < nc) {
            const float amax = fmaxf(fmaxf(s_red[half][0][j], s_red[half][1][j]),
                                     fmaxf(s_red[half][2][j], s_red[half][3][j]));
            const float sc = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
            const size_t row = (size_t)(it.row0 + c0 + j);
            outq[row * args.ld_out + it.mt * 128 + r] =
                amax == 0.0f ? (uint8_t)0 : cvt_e4m3(__fdiv_rn(acc0[j], sc));
            if (r == 0) args.out_scale[row * nblk + it.mt] = sc;
          }
        }
        // s_red is reused by the next item: the sync at the next item's start orders it
      } else {
        uint16_t* outy = static_cast<uint16_t*>(args.out);
        const int col = it.mt * 2 * kGemmBM + r;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          if (j < nc) {
            const size_t row = (size_t)(it.row0 + c0 + j);
            __nv_bfloat16 y0 = __float2bfloat16_rn(acc0[j]), y1 = __float2bfloat16_rn(acc1[j]);
            outy[row * args.ld_out + col] = *reinterpret_cast<uint16_t*>(&y0);
            outy[row * args.ld_out + col + kGemmBM] = *reinterpret_cast<uint16_t*>(&y1);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t gemm_fp8_setup() {
  cudaFuncAttributes fa{};
  cudaError_t e = cudaFuncGetAttributes(&fa, gemm_fp8_kernel);
  if (e != cudaSuccess) return e;
  // setmaxnreg.inc waits until registers are free: refuse a build whose launch
  // register count cannot cover the split rather than risk a wait that never ends.
  if (fa.numRegs < kRegsNeeded) return cudaErrorInvalidConfiguration;
  return cudaFuncSetAttribute(gemm_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem);
}

cudaError_t launch_gemm_fp8(const LayerDims& d, int T, const TcWeights& w, Workspace& ws, int num_sms,
                            cudaStream_t s, int which) {
  if (T == 0) return cudaSuccess;
  const int G = d.E + d.S;
  const long rows = (long)T * (d.k + d.S);
  const long tiles_ub = rows / kBN + G + 1;
  Fp8Args a{};
  a.counts = ws.counts;
  a.offsets = ws.offsets;
  a.tile_base = ws.tile_base;
  a.G = G;
  a.err = ws.err;
  if (which == 0) {  // gate/up + SwiGLU + e4m3 h: K = H
    a.num_kb = d.H / 128;
    a.MT = d.I / kGemmBM;
    a.a_rows_per_group = d.I;
    a.a_mt_stride = kGemmBM;
    a.a1_offset = 0;
    a.sA0 = w.sg;
    a.sA1 = w.su;
    a.sa1_block_offset = 0;
    a.sB = ws.P_scale;
    a.out = ws.Hb;
    a.out_scale = ws.H_scale;
    a.ld_out = d.I;
    a.mode = 0;
    const long items_ub = tiles_ub * a.MT;
    const int grid = (int)(items_ub < num_sms ? items_ub : num_sms);
    gemm_fp8_kernel<<<grid, kThreads, kDynSmem, s>>>(*w.tm_wg, *w.tm_wu, ws.tm_P, a);
    return cudaGetLastError();
  }
  // down: K = I, items of 256 output columns
  a.num_kb = d.I / 128;
  a.MT = d.H / (2 * kGemmBM);
  a.a_rows_per_group = d.H;
  a.a_mt_stride = 2 * kGemmBM;
  a.a1_offset = kGemmBM;
  a.sA0 = w.sd;
  a.sA1 = w.sd;
  a.sa1_block_offset = 1;
  a.sB = ws.H_scale;
  a.out = ws.Y;
  a.out_scale = nullptr;
  a.ld_out = d.H;
  a.mode = 1;
  const long items_ub = tiles_ub * a.MT;
  const int grid = (int)(items_ub < num_sms ? items_ub : num_sms);
  gemm_fp8_kernel<<<grid, kThreads, kDynSmem, s>>>(*w.tm_wd, *w.tm_wd, ws.tm_H, a);
  return cudaGetLastError();
}

}  // namespace afd
