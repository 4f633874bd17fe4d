// router_noalloc.cu -- the layer's router (logits, top-k, softmax over the
// selected logits) for callers that cannot allocate device memory.
//
// Who cannot allocate: a caller that hands all of the GPU's memory to its own
// pool up front (an attention-side serving process reserving HBM for its KV
// cache, for instance) has nothing left for cudaMalloc, and a caller inside a
// latency-critical decode loop must not make an allocation call, which can
// block or synchronise the device.  Such a caller still wants routing
// decisions identical to the full layer's.
//
// This entry point computes exactly what the full layer's router computes
// (same fp32 summation order, same selection order, same weights), reading
// the router weights in the caller's [H, E] layout, with no allocation: its
// only scratch (the logits and one completion ticket per 16-token tile) is the
// file-scope array g_router_scratch below, which every GPU that loads this
// library holds until the process exits.
//
// Set-up: the first call on a device (with that device current) looks up the
// array's device address with cudaGetSymbolAddress and caches it for that
// device for the life of the process; make that first call before any stream
// capture begins.  A device reset invalidates the cached address, so a caller
// that resets the device must restart the process before calling again.  Every call
// shares the one array: calls whose kernels overlap on the GPU (two streams,
// two host threads) race on it and must be serialised by the caller.  Each
// call clears the tickets (they must start at zero) with cudaMemsetAsync on
// its stream; the logits are fully written before they are read.
#include <mutex>

#include "afd_internal.cuh"

namespace afd {
namespace {

constexpr int kNaMaxTokens = 4096;   // tokens per call
constexpr int kNaMaxExperts = 256;   // experts
constexpr int kNaTokTile = 16;       // tokens per CTA
constexpr int kNaExpTile = 32;       // experts per CTA (two warps of 16)
constexpr int kNaTokPerWarp = 4;
constexpr int kNaExpPerWarp = 16;
constexpr int kNaMaxK = 16;
constexpr size_t kNaLogitBytes = (size_t)kNaMaxTokens * kNaMaxExperts * sizeof(float);
constexpr size_t kNaTickets = kNaMaxTokens / kNaTokTile;

// logits [T, E] fp32 (T*E <= 4096*256), then the per-tile tickets: 4 MiB + 1 KiB
static __device__ __align__(256) unsigned char g_router_scratch[kNaLogitBytes + kNaTickets * sizeof(int32_t)];

std::mutex g_na_mutex;
constexpr int kNaMaxDevices = 64;
void* g_na_addr[kNaMaxDevices] = {};

// Device address of g_router_scratch on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kNaMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_na_mutex);
  if (!g_na_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_router_scratch);
    if (e != cudaSuccess) return e;
    if (!p) return cudaErrorInvalidSymbol;
    g_na_addr[dev] = p;
  }
  *out = g_na_addr[dev];
  return cudaSuccess;
}

struct Row8 {
  float v[8];
};

__device__ __forceinline__ void na_load8(const uint16_t* p, Row8& c) {
  uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  c.v[0] = bf16_lo(u.x); c.v[1] = bf16_hi(u.x); c.v[2] = bf16_lo(u.y); c.v[3] = bf16_hi(u.y);
  c.v[4] = bf16_lo(u.z); c.v[5] = bf16_hi(u.z); c.v[6] = bf16_lo(u.w); c.v[7] = bf16_hi(u.w);
}
__device__ __forceinline__ void na_load8(const float* p, Row8& c) {
  float4 a = __ldg(reinterpret_cast<const float4*>(p));
  float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  c.v[0] = a.x; c.v[1] = a.y; c.v[2] = a.z; c.v[3] = a.w; c.v[4] = b.x; c.v[5] = b.y; c.v[6] = b.z; c.v[7] = b.w;
}

__device__ __forceinline__ bool na_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Same arithmetic as the layer's router kernel; the weights are read as
// W[h, e] (row h holds all experts) instead of the layer's [e, h] copy.  For
// channel h = 8c + q the warp's 16 experts are 8-expert groups of one row.
template <typename TA>
__global__ void __launch_bounds__(256) router_noalloc_kernel(SrcTable st, const TA* __restrict__ w_he,
                                                             const float* __restrict__ bias, int H, int E, int k,
                                                             float* __restrict__ logits, int32_t* __restrict__ ticket,
                                                             int32_t* __restrict__ topk_idx,
                                                             float* __restrict__ topk_w) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = st.T;
  const int t_base = blockIdx.x * kNaTokTile + (warp >> 1) * kNaTokPerWarp;
  const int e_base = blockIdx.y * kNaExpTile + (warp & 1) * kNaExpPerWarp;
  const bool lo_ok = e_base < E, hi_ok = e_base + 8 < E;  // E % 8 == 0

  const TA* xrow[kNaTokPerWarp];
#pragma unroll
  for (int i = 0; i < kNaTokPerWarp; ++i) {
    int t = t_base + i;
    if (t < T) {
      int m = src_of_token(st, t);
      xrow[i] = reinterpret_cast<const TA*>(st.src[m]) + (size_t)(t - st.row0[m]) * H;
    } else {
      xrow[i] = nullptr;
    }
  }
  float acc[kNaTokPerWarp][kNaExpPerWarp];
#pragma unroll
  for (int i = 0; i < kNaTokPerWarp; ++i)
#pragma unroll
    for (int j = 0; j < kNaExpPerWarp; ++j) acc[i][j] = 0.0f;

  for (int c = lane; c < (H >> 3); c += kWarp) {
    Row8 xc[kNaTokPerWarp];
#pragma unroll
    for (int i = 0; i < kNaTokPerWarp; ++i) {
      if (xrow[i]) na_load8(xrow[i] + 8 * c, xc[i]);
      else {
#pragma unroll
        for (int q = 0; q < 8; ++q) xc[i].v[q] = 0.0f;
      }
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const TA* wrow = w_he + (size_t)(8 * c + q) * E + e_base;
      Row8 w0, w1;
      if (lo_ok) na_load8(wrow, w0);
      if (hi_ok) na_load8(wrow + 8, w1);
#pragma unroll
      for (int i = 0; i < kNaTokPerWarp; ++i) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (lo_ok) acc[i][j] = fmaf(xc[i].v[q], w0.v[j], acc[i][j]);
          if (hi_ok) acc[i][8 + j] = fmaf(xc[i].v[q], w1.v[j], acc[i][8 + j]);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kNaTokPerWarp; ++i)
#pragma unroll
    for (int j = 0; j < kNaExpPerWarp; ++j) {
      float v = acc[i][j];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) v = v + __shfl_xor_sync(0xffffffffu, v, o);
      acc[i][j] = v;
    }
#pragma unroll
  for (int i = 0; i < kNaTokPerWarp; ++i)
#pragma unroll
    for (int j = 0; j < kNaExpPerWarp; ++j) {
      int p = i * kNaExpPerWarp + j;
      int t = t_base + i, e = e_base + j;
      if ((p & 31) == lane && t < T && e < E) {
        float v = acc[i][j];
        if (bias) v = __fadd_rn(v, __ldg(bias + e));
        logits[(size_t)t * E + e] = v;
      }
    }

  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(ticket + blockIdx.x, 1) == (int)gridDim.y - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  constexpr int kPerLane = kNaMaxExperts / 32;
  for (int tt = warp; tt < kNaTokTile; tt += 8) {
    const int t = blockIdx.x * kNaTokTile + tt;
    if (t >= T) break;
    float v[kPerLane];
    bool taken[kPerLane];
#pragma unroll
    for (int q = 0; q < kPerLane; ++q) {
      int e = lane + 32 * q;
      v[q] = (e < E) ? __ldcg(logits + (size_t)t * E + e) : 0.0f;
      taken[q] = (e >= E);
    }
    float sel_v[kNaMaxK];
    int sel_i[kNaMaxK];
#pragma unroll
    for (int j = 0; j < kNaMaxK; ++j) {
      if (j >= k) break;
      float bv = 0.0f;
      int bi = 0x7fffffff;
#pragma unroll
      for (int q = 0; q < kPerLane; ++q) {
        int e = lane + 32 * q;
        if (!taken[q] && (bi == 0x7fffffff || na_before(v[q], e, bv, bi))) {
          bv = v[q];
          bi = e;
        }
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (oi != 0x7fffffff && (bi == 0x7fffffff || na_before(ov, oi, bv, bi))) {
          bv = ov;
          bi = oi;
        }
      }
      sel_v[j] = bv;
      sel_i[j] = bi;
#pragma unroll
      for (int q = 0; q < kPerLane; ++q)
        if (lane + 32 * q == bi) taken[q] = true;
    }
    if (lane == 0) {
      float den = 0.0f, ex[kNaMaxK];
#pragma unroll
      for (int j = 0; j < kNaMaxK; ++j) {
        if (j >= k) break;
        ex[j] = expf(sel_v[j] - sel_v[0]);
        den += ex[j];
      }
#pragma unroll
      for (int j = 0; j < kNaMaxK; ++j) {
        if (j >= k) break;
        topk_idx[(size_t)t * k + j] = sel_i[j];
        topk_w[(size_t)t * k + j] = ex[j] / den;
      }
    }
  }
  if (threadIdx.x == 0) ticket[blockIdx.x] = 0;
}

}  // namespace
}  // namespace afd

extern "C" int afd_ffn_router_noalloc(void* stream, const void* const* src_ptrs_dev, const int* src_counts_host,
                                      int M, int H, int E, int k, afd_dtype dtype, const void* w_router_dev,
                                      const float* router_bias_dev, int* topk_idx_dev, float* topk_w_dev) {
  using namespace afd;
  if (dtype != AFD_FP32 && dtype != AFD_BF16 && dtype != AFD_FP8_E4M3) return AFD_EINVAL;
  if (H <= 0 || H % 8 || E <= 0 || E % 8 || k <= 0 || k > E || M < 0) return AFD_EINVAL;
  if (E > kNaMaxExperts || k > kNaMaxK || M > AFD_MAX_SOURCES) return AFD_ECAPACITY;
  if (M > 0 && (!src_ptrs_dev || !src_counts_host)) return AFD_EINVAL;
  SrcTable st{};
  st.M = M;
  long long T = 0;
  for (int m = 0; m < M; ++m) {
    if (src_counts_host[m] < 0) return AFD_EINVAL;
    if (src_counts_host[m] > 0 && (!src_ptrs_dev[m] || (reinterpret_cast<uintptr_t>(src_ptrs_dev[m]) & 15)))
      return AFD_EINVAL;
    st.src[m] = src_ptrs_dev[m];
    st.row0[m] = (int)T;
    T += src_counts_host[m];
    if (T > kNaMaxTokens) return AFD_ECAPACITY;
  }
  st.row0[M] = (int)T;
  st.T = (int)T;
  if (T == 0) return AFD_OK;
  if (!w_router_dev || !topk_idx_dev || !topk_w_dev || (reinterpret_cast<uintptr_t>(w_router_dev) & 15))
    return AFD_EINVAL;

  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return AFD_ECUDA;
  float* logits = static_cast<float*>(scratch);
  int32_t* tickets = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(scratch) + kNaLogitBytes);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int tiles = (int)((T + kNaTokTile - 1) / kNaTokTile);
  if (cudaMemsetAsync(tickets, 0, tiles * sizeof(int32_t), s) != cudaSuccess) return AFD_ECUDA;
  dim3 grid(tiles, (E + kNaExpTile - 1) / kNaExpTile);
  if (dtype == AFD_FP32)
    router_noalloc_kernel<float><<<grid, 256, 0, s>>>(st, static_cast<const float*>(w_router_dev), router_bias_dev, H,
                                                      E, k, logits, tickets, topk_idx_dev, topk_w_dev);
  else
    router_noalloc_kernel<uint16_t><<<grid, 256, 0, s>>>(st, static_cast<const uint16_t*>(w_router_dev),
                                                         router_bias_dev, H, E, k, logits, tickets, topk_idx_dev,
                                                         topk_w_dev);
  return cudaGetLastError() == cudaSuccess ? AFD_OK : AFD_ECUDA;
}
