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
// Work split: CTA (x, y) computes the logits of tokens [32x, 32x+32) against
// experts [ET y, ET y + ET) (ET = 32 for bf16, 16 for fp32).  Channels are
// consumed in slabs of 256 (32 chunks, so lane l always owns chunk l of a
// slab, which keeps the order above); each slab of the token rows and expert
// rows is staged in shared memory with cp.async (3 stages for bf16).  Warp w
// owns 8 tokens x 8 experts (64 fp32 accumulators per lane).  For bf16 the
// products use the mixed-precision fma.rn.f32.bf16 (bf16 x bf16 + f32, one
// rounding): bf16 products are exact in fp32, so it equals fma on the
// widened values and needs no conversion instructions.  The last CTA to
// finish a token tile (atomic ticket) selects the top-k for its 32 tokens and
// resets the ticket.
#include "afd_internal.cuh"

namespace afd {
namespace {

constexpr int kTT = kRouterTokTile;  // 32 tokens per CTA
constexpr int kWT = 8;               // tokens per warp
constexpr int kWE = 8;               // experts per warp
constexpr int kSlab = 256;           // channels per slab
constexpr int kMaxK = 16;

// per activation type: experts per CTA, threads, cp.async stages
template <typename TA>
struct Cfg;
template <>
struct Cfg<uint16_t> {
  static constexpr int ET = 32, kThreads = 512, kStages = 3;
};
template <>
struct Cfg<float> {
  static constexpr int ET = 16, kThreads = 256, kStages = 2;
};

template <typename TA>
constexpr int slab_bytes() {
  return (kTT + Cfg<TA>::ET) * kSlab * (int)sizeof(TA);
}
template <typename TA>
constexpr int router_smem_bytes() {
  return Cfg<TA>::kStages * slab_bytes<TA>();
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// c + a * b for the low / high bf16 halves of two packed words (one rounding)
__device__ __forceinline__ float fma_bf16_lo(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, al, bl, %3;\n\t}"
      : "=f"(d)
      : "r"(a), "r"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fma_bf16_hi(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, ah, bh, %3;\n\t}"
      : "=f"(d)
      : "r"(a), "r"(b), "f"(c));
  return d;
}

__device__ __forceinline__ void lds8(const float* p, float* v) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *(reinterpret_cast<const float4*>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// (value, index) ordering of the selection: larger value first, then lower id.
__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Stage slab s (channels [256 s, 256 s + 256)) of the CTA's token rows and
// expert rows into shared memory.  Rows past T or E are left untouched: their
// accumulators are never written out.
template <typename TA>
__device__ __forceinline__ void stage_slab(TA* sx, TA* sw, const TA* const* xrow, const TA* __restrict__ wrT,
                                           int e0, int E, int H, int s) {
  constexpr int kET = Cfg<TA>::ET, kThreads = Cfg<TA>::kThreads;
  constexpr int kUnits = (int)sizeof(TA) * 8 / 16;  // 16-byte pieces per 8-channel chunk
  const int nch = min(32, (H >> 3) - 32 * s);       // chunks in this slab
  const int per_row = nch * kUnits;
  for (int u = threadIdx.x; u < (kTT + kET) * per_row; u += kThreads) {
    const int r = u / per_row, q = u - r * per_row;
    const TA* src;
    TA* dst;
    if (r < kTT) {
      if (!xrow[r]) continue;
      src = xrow[r];
      dst = sx + r * kSlab;
    } else {
      const int e = e0 + (r - kTT);
      if (e >= E) continue;
      src = wrT + (size_t)e * H;
      dst = sw + (r - kTT) * kSlab;
    }
    const int off = q * (16 / (int)sizeof(TA));  // element offset inside the slab
    cp_async16(dst + off, src + (size_t)s * kSlab + off);
  }
}

// One 8-channel chunk of the warp's 8 x 8 block: acc[i][j] += x_i . w_j over
// the chunk's channels in ascending order.
__device__ __forceinline__ void chunk_fma(const uint16_t* sx, const uint16_t* sw, int lane,
                                          float (&acc)[kWT][kWE]) {
  uint4 xr[kWT];
#pragma unroll
  for (int i = 0; i < kWT; ++i) xr[i] = *reinterpret_cast<const uint4*>(sx + i * kSlab + 8 * lane);
#pragma unroll
  for (int j = 0; j < kWE; ++j) {
    const uint4 wr = *reinterpret_cast<const uint4*>(sw + j * kSlab + 8 * lane);
#pragma unroll
    for (int i = 0; i < kWT; ++i) {
      float a = acc[i][j];
      a = fma_bf16_lo(xr[i].x, wr.x, a); a = fma_bf16_hi(xr[i].x, wr.x, a);
      a = fma_bf16_lo(xr[i].y, wr.y, a); a = fma_bf16_hi(xr[i].y, wr.y, a);
      a = fma_bf16_lo(xr[i].z, wr.z, a); a = fma_bf16_hi(xr[i].z, wr.z, a);
      a = fma_bf16_lo(xr[i].w, wr.w, a); a = fma_bf16_hi(xr[i].w, wr.w, a);
      acc[i][j] = a;
    }
  }
}
__device__ __forceinline__ void chunk_fma(const float* sx, const float* sw, int lane, float (&acc)[kWT][kWE]) {
  float xf[kWT][8];
#pragma unroll
  for (int i = 0; i < kWT; ++i) lds8(sx + i * kSlab + 8 * lane, xf[i]);
#pragma unroll
  for (int j = 0; j < kWE; ++j) {
    float wf[8];
    lds8(sw + j * kSlab + 8 * lane, wf);
#pragma unroll
    for (int i = 0; i < kWT; ++i)
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[i][j] = fmaf(xf[i][q], wf[q], acc[i][j]);
  }
}

template <typename TA>
__global__ void __launch_bounds__(Cfg<TA>::kThreads, 1)
    router_kernel(SrcTable st, const TA* __restrict__ wrT, const float* __restrict__ bias, int H, int E, int k,
                  float* __restrict__ logits, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                  int32_t* __restrict__ ticket) {
  pdl_begin();
  constexpr int kET = Cfg<TA>::ET, kThreads = Cfg<TA>::kThreads, kStages = Cfg<TA>::kStages;
  constexpr int kEG = kET / kWE;  // expert groups of warps
  extern __shared__ __align__(16) uint8_t router_smem[];
  __shared__ const TA* xrow[kTT];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = st.T;
  const int t0 = blockIdx.x * kTT, e0 = blockIdx.y * kET;
  for (int r = threadIdx.x; r < kTT; r += kThreads) {
    const int t = t0 + r;
    if (t < T) {
      const int m = src_of_token(st, t);
      xrow[r] = reinterpret_cast<const TA*>(st.src[m]) + (size_t)(t - st.row0[m]) * H;
    } else {
      xrow[r] = nullptr;
    }
  }
  __syncthreads();

  auto buf = [&](int b) { return reinterpret_cast<TA*>(router_smem + b * slab_bytes<TA>()); };
  const int nslab = (H + kSlab - 1) / kSlab;
  const int wt = (warp / kEG) * kWT;  // warp's first token (in the CTA tile)
  const int we = (warp % kEG) * kWE;  // warp's first expert (in the CTA tile)

  float acc[kWT][kWE];
#pragma unroll
  for (int i = 0; i < kWT; ++i)
#pragma unroll
    for (int j = 0; j < kWE; ++j) acc[i][j] = 0.0f;

#pragma unroll
  for (int p = 0; p < kStages - 1; ++p) {
    if (p < nslab) stage_slab<TA>(buf(p), buf(p) + kTT * kSlab, xrow, wrT, e0, E, H, p);
    cp_async_commit();
  }
  for (int s = 0; s < nslab; ++s) {
    cp_async_wait<kStages - 2>();
    __syncthreads();
    if (s + kStages - 1 < nslab) {
      TA* nb = buf((s + kStages - 1) % kStages);
      stage_slab<TA>(nb, nb + kTT * kSlab, xrow, wrT, e0, E, H, s + kStages - 1);
    }
    cp_async_commit();
    const TA* sx = buf(s % kStages);
    if (32 * s + lane < (H >> 3))  // lane owns chunk 32 s + lane
      chunk_fma(sx + wt * kSlab, sx + (kTT + we) * kSlab, lane, acc);
  }

  // fold the 32 lane partial sums: xor 16, 8, 4, 2, 1
#pragma unroll
  for (int i = 0; i < kWT; ++i)
#pragma unroll
    for (int j = 0; j < kWE; ++j) {
      float v = acc[i][j];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) v = v + __shfl_xor_sync(0xffffffffu, v, o);
      acc[i][j] = v;
    }
  // every lane holds every sum; lane (p % 32) writes pair p
#pragma unroll
  for (int i = 0; i < kWT; ++i)
#pragma unroll
    for (int j = 0; j < kWE; ++j) {
      const int p = i * kWE + j;
      const int t = t0 + wt + i, e = e0 + we + j;
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
  if (threadIdx.x == 0) s_last = (atomicAdd(ticket + blockIdx.x, 1) == (int)gridDim.y - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  constexpr int kMaxPerLane = (kMaxExperts + 31) / 32;  // E <= 256 -> 8 per lane
  for (int tt = warp; tt < kTT; tt += kThreads / 32) {
    const int t = t0 + tt;
    if (t >= T) break;
    float v[kMaxPerLane];
    bool taken[kMaxPerLane];
#pragma unroll
    for (int q = 0; q < kMaxPerLane; ++q) {
      const int e = lane + 32 * q;
      v[q] = (e < E) ? __ldcg(logits + (size_t)t * E + e) : 0.0f;
      taken[q] = (e >= E);
    }
    float sel_v[kMaxK];
    int sel_i[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j >= k) break;
      float bv = 0.0f;
      int bi = 0x7fffffff;
#pragma unroll
      for (int q = 0; q < kMaxPerLane; ++q) {
        const int e = lane + 32 * q;
        if (!taken[q] && (bi == 0x7fffffff || ranks_before(v[q], e, bv, bi))) {
          bv = v[q];
          bi = e;
        }
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
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
      float den = 0.0f, ex[kMaxK];
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

cudaError_t router_setup() {
  cudaError_t e = cudaFuncSetAttribute(router_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       router_smem_bytes<float>());
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(router_kernel<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              router_smem_bytes<uint16_t>());
}

cudaError_t launch_router(const SrcTable& st, const void* wrT, const float* bias, const LayerDims& d,
                          Workspace& ws, cudaStream_t s) {
  if (st.T == 0) return cudaSuccess;
  if (d.dtype == AFD_FP32) {
    dim3 grid((st.T + kTT - 1) / kTT, (d.E + Cfg<float>::ET - 1) / Cfg<float>::ET);
    {
      const cudaError_t e_ = launch_k(router_kernel<float>, dim3(grid), dim3(Cfg<float>::kThreads),
                                      router_smem_bytes<float>(), s, st, static_cast<const float*>(wrT), bias,
                                      d.H, d.E, d.k, ws.logits, ws.topk_idx, ws.topk_w, ws.tile_counter);
      if (e_ != cudaSuccess) return e_;
    }
  } else {
    dim3 grid((st.T + kTT - 1) / kTT, (d.E + Cfg<uint16_t>::ET - 1) / Cfg<uint16_t>::ET);
    {
      const cudaError_t e_ = launch_k(router_kernel<uint16_t>, dim3(grid), dim3(Cfg<uint16_t>::kThreads),
                                      router_smem_bytes<uint16_t>(), s, st, static_cast<const uint16_t*>(wrT),
                                      bias, d.H, d.E, d.k, ws.logits, ws.topk_idx, ws.topk_w, ws.tile_counter);
      if (e_ != cudaSuccess) return e_;
    }
  }
  return cudaGetLastError();
}

}  // namespace afd
