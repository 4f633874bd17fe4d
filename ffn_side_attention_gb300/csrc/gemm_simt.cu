// gemm_simt.cu -- grouped SwiGLU expert GEMMs for the fp32 layer (CUDA cores,
// fp32 FMA, no TF32), and the transpose kernels used to re-lay weights at
// create time.
//
// The fp32 layer is the small end-to-end check of the method; its GEMMs are
// far too small to feed tensor cores and fp32 accuracy is required, so they
// run as plain FMA loops: thread = one output column of one packed row.
//   gate/up: h[r, i] = silu(sum_h P[r,h] Wg[e,h,i]) * (sum_h P[r,h] Wu[e,h,i])
//   down:    Y[r, o] = sum_i h[r,i] Wd[e,i,o]
// with e the expert (or shared group) owning packed row r.
#include "afd_internal.cuh"

namespace afd {
namespace {

__device__ __forceinline__ int group_of_row(const int32_t* offsets, int G, int r) {
  int lo = 0, hi = G - 1;  // last g with offsets[g] <= r
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(offsets + mid) <= r) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(128) simt_gateup_kernel(const float* __restrict__ P, const int32_t* __restrict__ offsets,
                                                          int G, int H, int I, const float* __restrict__ wg,
                                                          const float* __restrict__ wu, float* __restrict__ Hb) {
  pdl_begin();
  const int r = blockIdx.x;
  const int i = blockIdx.y * 128 + threadIdx.x;
  const int e = group_of_row(offsets, G, r);
  if (i >= I) return;
  const float* p = P + (size_t)r * H;
  const float* g = wg + (size_t)e * H * I + i;
  const float* u = wu + (size_t)e * H * I + i;
  float ag = 0.f, au = 0.f;
  for (int h = 0; h < H; ++h) {
    float x = __ldg(p + h);
    ag = fmaf(x, __ldg(g + (size_t)h * I), ag);
    au = fmaf(x, __ldg(u + (size_t)h * I), au);
  }
  float silu = ag / (1.0f + expf(-ag));
  Hb[(size_t)r * I + i] = silu * au;
}

__global__ void __launch_bounds__(128) simt_down_kernel(const float* __restrict__ Hb, const int32_t* __restrict__ offsets,
                                                        int G, int H, int I, const float* __restrict__ wd,
                                                        float* __restrict__ Y) {
  pdl_begin();
  const int r = blockIdx.x;
  const int o = blockIdx.y * 128 + threadIdx.x;
  const int e = group_of_row(offsets, G, r);
  if (o >= H) return;
  const float* hh = Hb + (size_t)r * I;
  const float* d = wd + (size_t)e * I * H + o;
  float acc = 0.f;
  for (int i = 0; i < I; ++i) acc = fmaf(__ldg(hh + i), __ldg(d + (size_t)i * H), acc);
  Y[(size_t)r * H + o] = acc;
}

// batched transpose [batch][rows][cols] -> [batch][cols][rows], element of E bytes
template <typename Elem>
__global__ void transpose_kernel(const Elem* __restrict__ src, Elem* __restrict__ dst, int rows, int cols) {
  __shared__ Elem tile[32][33];
  const size_t base = (size_t)blockIdx.z * rows * cols;
  int c = blockIdx.x * 32 + threadIdx.x;
  for (int y = threadIdx.y; y < 32; y += 8) {
    int r = blockIdx.y * 32 + y;
    if (r < rows && c < cols) tile[y][threadIdx.x] = src[base + (size_t)r * cols + c];
  }
  __syncthreads();
  int r = blockIdx.y * 32 + threadIdx.x;
  for (int y = threadIdx.y; y < 32; y += 8) {
    int cc = blockIdx.x * 32 + y;
    if (r < rows && cc < cols) dst[base + (size_t)cc * rows + r] = tile[threadIdx.x][y];
  }
}

// Weight tiling for the tensor-core GEMMs.  src holds `batch` matrices
// [K][R] (the caller's [in][out] layout); dst holds, per matrix, tiles of 128
// output rows x 128 bytes of K, ordered (row block, K block): tile (rb, kb) is
// one contiguous 16 KB block holding rows rb*128 .. +127 of the transposed
// matrix, K elements kb*KW .. +KW-1, so every TMA box of the GEMM reads one
// contiguous block and an item's K blocks follow each other in memory.
template <typename Elem>
__global__ void __launch_bounds__(256) tile_weights_kernel(const Elem* __restrict__ src, Elem* __restrict__ dst,
                                                           int K, int R) {
  constexpr int KW = 128 / (int)sizeof(Elem);
  __shared__ Elem tile[KW][128 + 4];
  const int rb = blockIdx.x, kb = blockIdx.y;
  const size_t base = (size_t)blockIdx.z * K * R;
  const Elem* s = src + base + (size_t)kb * KW * R + (size_t)rb * 128;
  for (int i = threadIdx.x; i < KW * 128; i += 256) tile[i >> 7][i & 127] = s[(size_t)(i >> 7) * R + (i & 127)];
  __syncthreads();
  Elem* d = dst + base + ((size_t)rb * (K / KW) + kb) * 128 * KW;
  for (int i = threadIdx.x; i < KW * 128; i += 256) d[i] = tile[i % KW][i / KW];
}

}  // namespace

cudaError_t launch_tile_weights(const void* src, void* dst, int batch, int K, int R, int elem_bytes,
                                cudaStream_t s) {
  if ((size_t)batch * K * R == 0) return cudaSuccess;
  const int kw = 128 / elem_bytes;
  if (R % 128 || K % kw) return cudaErrorInvalidValue;
  dim3 grid(R / 128, K / kw, batch);
  if (elem_bytes == 1)
    tile_weights_kernel<uint8_t><<<grid, 256, 0, s>>>(static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst),
                                                      K, R);
  else if (elem_bytes == 2)
    tile_weights_kernel<uint16_t><<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(src),
                                                       static_cast<uint16_t*>(dst), K, R);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_gemm_simt(const LayerDims& d, int T, const float* wg, const float* wu, const float* wd,
                             Workspace& ws, cudaStream_t s, int which) {
  const int rows = T * (d.k + d.S);
  if (rows == 0) return cudaSuccess;
  const int G = d.E + d.S;
  if (which == 0) {
    {
      const cudaError_t e_ = launch_k(simt_gateup_kernel, dim3(dim3(rows, (d.I + 127) / 128)), dim3(128), 0, s,
                                      static_cast<const float*>(ws.P), ws.offsets, G, d.H, d.I, wg, wu,
                                      static_cast<float*>(ws.Hb));
      if (e_ != cudaSuccess) return e_;
    }
    return cudaGetLastError();
  }
  {
    const cudaError_t e_ = launch_k(simt_down_kernel, dim3(dim3(rows, (d.H + 127) / 128)), dim3(128), 0, s,
                                    static_cast<const float*>(ws.Hb), ws.offsets, G, d.H, d.I, wd,
                                    static_cast<float*>(ws.Y));
    if (e_ != cudaSuccess) return e_;
  }
  return cudaGetLastError();
}

cudaError_t launch_transpose(const void* src, void* dst, int batch, int rows, int cols, int elem_bytes,
                             cudaStream_t s) {
  if ((size_t)batch * rows * cols == 0) return cudaSuccess;
  dim3 grid((cols + 31) / 32, (rows + 31) / 32, batch), block(32, 8);
  switch (elem_bytes) {
    case 1:
      transpose_kernel<uint8_t><<<grid, block, 0, s>>>(static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst),
                                                       rows, cols);
      break;
    case 2:
      transpose_kernel<uint16_t><<<grid, block, 0, s>>>(static_cast<const uint16_t*>(src),
                                                        static_cast<uint16_t*>(dst), rows, cols);
      break;
    case 4:
      transpose_kernel<uint32_t><<<grid, block, 0, s>>>(static_cast<const uint32_t*>(src),
                                                        static_cast<uint32_t*>(dst), rows, cols);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_transpose_f32(const float* src, float* dst, int batch, int rows, int cols, cudaStream_t s) {
  return launch_transpose(src, dst, batch, rows, cols, 4, s);
}

}  // namespace afd
