// pack_combine.cu -- R3 pack and R6 combine.
//
// Pack: "MoE 大规模分布式推理工程实战", section 2.2 (the pack kernel gathers
// each item's token row into a destination-contiguous buffer using the
// prefix-sum offsets); here rows are gathered straight from the M
// attention-instance buffers into expert-contiguous order.  For the fp8 layer
// the pack also quantises ("MoE系统与AFD架构概述", section 3.3, FP8
// activations): per row, per 128 channels, scale = amax / 448 (IEEE fp32
// division), code = e4m3(x / scale) rounded to nearest even with saturation;
// an all-zero block gets scale 1.
//
// Combine: same page, section 1.1 (combine brings the k processed copies of a
// token back).  out[t] = sum_j w[t,j] * Y[pos[t,j]] in slot order (+ the
// shared expert's row), accumulated in fp32 and rounded once; written to the
// token's own output buffer.  No atomics: the result is run-to-run identical.
//
// Both are HBM-bound row moves: one warp per token, 16-byte vector accesses.
#include "afd_internal.cuh"

namespace afd {
namespace {

__device__ __forceinline__ uint8_t* out_row(const SrcTable& st, int t, size_t row_bytes) {
  int m = src_of_token(st, t);
  return reinterpret_cast<uint8_t*>(st.out[m]) + (size_t)(t - st.row0[m]) * row_bytes;
}

__device__ __forceinline__ uint32_t cvt_e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Packed rows of token t: its k routed copies (pos[t*k + j]) and, with a
// shared expert, row T*k + t.  One warp per token: each source row is read
// once (and quantised once) and stored to all of its packed rows.
constexpr int kMaxCopies = 17;  // k <= 16, plus the shared expert

__device__ __forceinline__ int packed_rows(const int32_t* __restrict__ pos, int t, int T, int k, int S, int* rows) {
  int n = 0;
  for (int j = 0; j < k; ++j) rows[n++] = __ldg(pos + (size_t)t * k + j);
  if (S) rows[n++] = T * k + t;
  return n;
}

// Work unit = (token, G consecutive 512-byte chunks of its row): one warp, 16
// bytes per lane per chunk; the unit's G loads are all issued before its stores,
// and units spread over the grid keep many rows' copies in flight.  G was
// measured: 8 for the plain copy, 4 where the unit also quantises (8 made the
// DeepSeek-V3 fp8 pack slower).
constexpr int kPackGCopy = 8;
constexpr int kPackGFp8 = 4;
constexpr int kPackSmallChunks = 1024;  // up to this many 512-byte chunks: one chunk per unit

// bf16 / fp32 layers: row copy.  G chunks per unit; warps per block from the launch.
template <int G>
__global__ void __launch_bounds__(256) pack_copy_kernel(SrcTable st, const int32_t* __restrict__ pos, int T, int k,
                                                        int S, int row_bytes, uint8_t* __restrict__ P) {
  pdl_begin();
  const int lane = threadIdx.x & 31, wpb = blockDim.x >> 5;
  const int nchunk = (row_bytes + 511) >> 9;  // 512 bytes per warp step
  const int ngroup = (nchunk + G - 1) / G;
  const int nvec = row_bytes >> 4;
  const long units = (long)T * ngroup;
  for (long u = (long)blockIdx.x * wpb + (threadIdx.x >> 5); u < units; u += (long)gridDim.x * wpb) {
    const int t = (int)(u / ngroup), c0 = (int)(u - (long)t * ngroup) * G;
    int rows[kMaxCopies];
    const int n = packed_rows(pos, t, T, k, S, rows);
    const uint4* src = reinterpret_cast<const uint4*>(src_row(st, t, row_bytes));
    uint4 x[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int v = (c0 + g) * 32 + lane;
      if (v < nvec) x[g] = __ldg(src + v);
    }
    for (int q = 0; q < n; ++q) {
      uint4* dst = reinterpret_cast<uint4*>(P + (size_t)rows[q] * row_bytes);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const int v = (c0 + g) * 32 + lane;
        if (v < nvec) dst[v] = x[g];
      }
    }
  }
}

// fp8 layer: e4m3 codes + one fp32 scale per 128 channels, computed once per
// token.  A 256-channel warp step holds two 128-channel blocks of 16 lanes.
// Scales are stored K-block major (P_scale[block * scale_ld + row]), so the
// GEMM reads one block's scales of consecutive rows as one coalesced load.
__global__ void __launch_bounds__(256) pack_fp8_kernel(SrcTable st, const int32_t* __restrict__ pos, int T, int k,
                                                       int S, int H, uint8_t* __restrict__ P,
                                                       float* __restrict__ P_scale, int scale_ld) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int nchunk = H >> 8;  // H % 256 == 0: whole warp active
  const int ngroup = (nchunk + kPackGFp8 - 1) / kPackGFp8;
  const long units = (long)T * ngroup;
  for (long u = (long)blockIdx.x * 8 + (threadIdx.x >> 5); u < units; u += (long)gridDim.x * 8) {
    const int t = (int)(u / ngroup), c0 = (int)(u - (long)t * ngroup) * kPackGFp8;
    int rows[kMaxCopies];
    const int n = packed_rows(pos, t, T, k, S, rows);
    const uint4* src = reinterpret_cast<const uint4*>(src_row(st, t, (size_t)H * 2));
    uint4 x8[kPackGFp8];
#pragma unroll
    for (int g = 0; g < kPackGFp8; ++g)
      if (c0 + g < nchunk) x8[g] = __ldg(src + (c0 + g) * 32 + lane);
#pragma unroll
    for (int g = 0; g < kPackGFp8; ++g) {
      if (c0 + g >= nchunk) break;
      const int v = (c0 + g) * 32 + lane;
      const float x[8] = {bf16_lo(x8[g].x), bf16_hi(x8[g].x), bf16_lo(x8[g].y), bf16_hi(x8[g].y),
                          bf16_lo(x8[g].z), bf16_hi(x8[g].z), bf16_lo(x8[g].w), bf16_hi(x8[g].w)};
      float amax = 0.0f;
#pragma unroll
      for (int q = 0; q < 8; ++q) amax = fmaxf(amax, fabsf(x[q]));
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const float scale = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
      uint2 q = make_uint2(0u, 0u);
      if (amax != 0.0f) {
        const uint32_t q01 = cvt_e4m3x2(__fdiv_rn(x[1], scale), __fdiv_rn(x[0], scale));
        const uint32_t q23 = cvt_e4m3x2(__fdiv_rn(x[3], scale), __fdiv_rn(x[2], scale));
        const uint32_t q45 = cvt_e4m3x2(__fdiv_rn(x[5], scale), __fdiv_rn(x[4], scale));
        const uint32_t q67 = cvt_e4m3x2(__fdiv_rn(x[7], scale), __fdiv_rn(x[6], scale));
        q = make_uint2(q01 | (q23 << 16), q45 | (q67 << 16));
      }
      for (int r = 0; r < n; ++r) {
        reinterpret_cast<uint2*>(P + (size_t)rows[r] * H)[v] = q;
        if ((lane & 15) == 0) P_scale[(size_t)(v >> 4) * scale_ld + rows[r]] = scale;
      }
    }
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}

// bf16 Y (bf16 / fp8 layers): work unit = (token, 256-column chunk), one warp,
// 8 channels per lane.  KC = k at compile time (0: runtime k) so the k row
// loads of a unit are all in flight together.
template <int KC>
__global__ void __launch_bounds__(256) combine_bf16_kernel(SrcTable st, const int32_t* __restrict__ pos,
                                                           const float* __restrict__ topk_w,
                                                           const uint16_t* __restrict__ Y, int T, int k_rt, int S,
                                                           int H, int early) {
  // The next kernel of the stream (the next forward's first) may launch early only when
  // this grid fits one wave of resident blocks: otherwise its blocks, resident and waiting,
  // would take thread slots from this memory-bound grid's later waves (measured: T=3160
  // and qwen3 fp8 steps 0.3-0.5% faster with the late trigger, T=6 unchanged).
  pdl_wait();
  if (early) pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int k = KC ? KC : k_rt;
  const int nchunk = H >> 8;
  const long units = (long)T * nchunk;
  // Y rows are read once: loaded evict-first, so the rows the down GEMM left in L2 stay
  // there until their own reader comes (measured: T=3160 combine 44 -> 37.6 us)
  const uint64_t pol = l2_policy_evict_first();
  const int wpb = blockDim.x >> 5;
  for (long u = (long)blockIdx.x * wpb + (threadIdx.x >> 5); u < units; u += (long)gridDim.x * wpb) {
    const int t = (int)(u / nchunk), c = (int)(u - (long)t * nchunk);
    const int v = c * 32 + lane;
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
#pragma unroll 8
    for (int j = 0; j < k; ++j) {
      const int r = __ldg(pos + (size_t)t * k + j);
      const float w = __ldg(topk_w + (size_t)t * k + j);
      const uint4 y = ld_nc_hint_v4(reinterpret_cast<const uint4*>(Y + (size_t)r * H) + v, pol);
      acc[0] = fmaf(w, bf16_lo(y.x), acc[0]); acc[1] = fmaf(w, bf16_hi(y.x), acc[1]);
      acc[2] = fmaf(w, bf16_lo(y.y), acc[2]); acc[3] = fmaf(w, bf16_hi(y.y), acc[3]);
      acc[4] = fmaf(w, bf16_lo(y.z), acc[4]); acc[5] = fmaf(w, bf16_hi(y.z), acc[5]);
      acc[6] = fmaf(w, bf16_lo(y.w), acc[6]); acc[7] = fmaf(w, bf16_hi(y.w), acc[7]);
    }
    if (S) {
      const uint4 y = ld_nc_hint_v4(reinterpret_cast<const uint4*>(Y + (size_t)(T * k + t) * H) + v, pol);
      acc[0] += bf16_lo(y.x); acc[1] += bf16_hi(y.x); acc[2] += bf16_lo(y.y); acc[3] += bf16_hi(y.y);
      acc[4] += bf16_lo(y.z); acc[5] += bf16_hi(y.z); acc[6] += bf16_lo(y.w); acc[7] += bf16_hi(y.w);
    }
    reinterpret_cast<uint4*>(out_row(st, t, (size_t)H * 2))[v] =
        make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                   pack_bf16x2(acc[6], acc[7]));
  }
}

// fp32 layer: 4 channels per lane step.
__global__ void __launch_bounds__(256) combine_f32_kernel(SrcTable st, const int32_t* __restrict__ pos,
                                                          const float* __restrict__ topk_w,
                                                          const float* __restrict__ Y, int T, int k, int S, int H) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  for (int t = blockIdx.x * 8 + (threadIdx.x >> 5); t < T; t += gridDim.x * 8) {
    float4* o = reinterpret_cast<float4*>(out_row(st, t, (size_t)H * 4));
    for (int v = lane; v < (H >> 2); v += 32) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j = 0; j < k; ++j) {
        int r = __ldg(pos + (size_t)t * k + j);
        float w = __ldg(topk_w + (size_t)t * k + j);
        float4 y = __ldg(reinterpret_cast<const float4*>(Y + (size_t)r * H) + v);
        acc.x = fmaf(w, y.x, acc.x); acc.y = fmaf(w, y.y, acc.y);
        acc.z = fmaf(w, y.z, acc.z); acc.w = fmaf(w, y.w, acc.w);
      }
      if (S) {
        float4 y = __ldg(reinterpret_cast<const float4*>(Y + (size_t)(T * k + t) * H) + v);
        acc.x += y.x; acc.y += y.y; acc.z += y.z; acc.w += y.w;
      }
      o[v] = acc;
    }
  }
}

inline int grid_for(int rows_per_block_units, int units, int num_sms) {
  int want = (units + rows_per_block_units - 1) / rows_per_block_units;
  int cap = num_sms * 16;
  return want < cap ? (want > 0 ? want : 1) : cap;
}

}  // namespace

cudaError_t launch_pack(const SrcTable& st, const LayerDims& d, int T, Workspace& ws, int num_sms,
                        cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int row_bytes = d.H * (d.dtype == AFD_FP32 ? 4 : 2);
  const int G = d.dtype == AFD_FP8_E4M3 ? kPackGFp8 : kPackGCopy;
  const int grid = grid_for(8, T * (((row_bytes + 511) / 512 + G - 1) / G), num_sms);
  if (d.dtype == AFD_FP8_E4M3)
    {
      const cudaError_t e_ = launch_k(pack_fp8_kernel, dim3(grid), dim3(256), 0, s, st, ws.pos, T, d.k, d.S, d.H,
                                      static_cast<uint8_t*>(ws.P), ws.P_scale, ws.scale_ld);
      if (e_ != cudaSuccess) return e_;
    }
  else if (T * ((row_bytes + 511) / 512) <= kPackSmallChunks)
    {
      // few tokens: one 512-byte chunk per unit and two warps per block, so the stores
      // of the copies spread over many SMs instead of draining from a few (qwen3 shapes,
      // 6 and 48 tokens: pack 10.2 -> 6.1 us; at 395 tokens and above this form was
      // slower than 8-chunk units)
      const int units = T * ((row_bytes + 511) / 512);
      const cudaError_t e_ = launch_k(pack_copy_kernel<1>, dim3((units + 1) / 2), dim3(64), 0, s, st, ws.pos, T, d.k,
                                      d.S, row_bytes, static_cast<uint8_t*>(ws.P));
      if (e_ != cudaSuccess) return e_;
    }
  else
    {
      const cudaError_t e_ = launch_k(pack_copy_kernel<kPackGCopy>, dim3(grid), dim3(256), 0, s, st, ws.pos, T, d.k,
                                      d.S, row_bytes, static_cast<uint8_t*>(ws.P));
      if (e_ != cudaSuccess) return e_;
    }
  return cudaGetLastError();
}

cudaError_t launch_combine(const SrcTable& st, const LayerDims& d, int T, Workspace& ws, int num_sms,
                           cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int units = d.dtype == AFD_FP32 ? T : T * (d.H / 256);
  // few tokens: two warps per block, so the k row reads of the units spread over more SMs
  // (qwen3 shapes: T = 6 step 0.2361 -> 0.2352 ms, T = 24 0.5495 -> 0.5465 ms)
  const bool small = d.dtype != AFD_FP32 && units <= kPackSmallChunks;
  const int grid = small ? (units + 1) / 2 : grid_for(8, units, num_sms);
  const dim3 blk(small ? 64 : 256);
  const uint16_t* Y = static_cast<const uint16_t*>(ws.Y);
  const int early = small || grid <= num_sms * 8;  // one wave of 8 resident blocks per SM
  if (d.dtype == AFD_FP32)
    return launch_k(combine_f32_kernel, dim3(grid), dim3(256), 0, s, st, ws.pos, ws.topk_w,
                    static_cast<const float*>(ws.Y), T, d.k, d.S, d.H);
  switch (d.k) {  // k known at compile time keeps a unit's k row loads in flight together
    case 1:
      return launch_k(combine_bf16_kernel<1>, dim3(grid), blk, 0, s, st, ws.pos, ws.topk_w, Y, T, d.k, d.S, d.H, early);
    case 2:
      return launch_k(combine_bf16_kernel<2>, dim3(grid), blk, 0, s, st, ws.pos, ws.topk_w, Y, T, d.k, d.S, d.H, early);
    case 3:
      return launch_k(combine_bf16_kernel<3>, dim3(grid), blk, 0, s, st, ws.pos, ws.topk_w, Y, T, d.k, d.S, d.H, early);
    case 4:
      return launch_k(combine_bf16_kernel<4>, dim3(grid), blk, 0, s, st, ws.pos, ws.topk_w, Y, T, d.k, d.S, d.H, early);
    case 6:
      return launch_k(combine_bf16_kernel<6>, dim3(grid), blk, 0, s, st, ws.pos, ws.topk_w, Y, T, d.k, d.S, d.H, early);
    case 8:
      return launch_k(combine_bf16_kernel<8>, dim3(grid), blk, 0, s, st, ws.pos, ws.topk_w, Y, T, d.k, d.S, d.H, early);
    default:
      return launch_k(combine_bf16_kernel<0>, dim3(grid), blk, 0, s, st, ws.pos, ws.topk_w, Y, T, d.k, d.S, d.H, early);
  }
}

}  // namespace afd
