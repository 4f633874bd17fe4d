// afd_internal.cuh -- internal structures, launch declarations and inline-PTX
// helpers (mbarrier, TMA, tcgen05/TMEM) shared by the kernels of libafd_ffn.
#pragma once

#include <cuda.h>
#include <utility>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/afd_ffn.h"

namespace afd {

// ---------------------------------------------------------------- constants
constexpr int kWarp = 32;
constexpr int kRouterTokTile = 32;  // tokens per router CTA
constexpr int kGemmBN = 256;        // largest token tile of the bf16 GEMMs (MMA N)
constexpr int kGemmBM = 128;        // weight rows per MMA (MMA M)
constexpr int kGemmBNFp8 = 128;     // max tokens per fp8 GEMM tile
constexpr int kMaxExperts = 257;    // routed + shared
constexpr int kRouterMaxSplits = 8; // K splits of the tensor-core router logits

// device error word bits
constexpr int kErrTimeout = 1;
constexpr int kErrRange = 2;

// ---------------------------------------------------------------- batch table
// The M source/output buffers of one forward, passed by value to kernels.
// Token t lives in buffer m with row0[m] <= t < row0[m+1], row t - row0[m].
struct SrcTable {
  const void* src[AFD_MAX_SOURCES];
  void* out[AFD_MAX_SOURCES];
  int row0[AFD_MAX_SOURCES + 1];
  int M;
  int T;
};

__device__ __forceinline__ int src_of_token(const SrcTable& s, int t) {
  int lo = 0, hi = s.M - 1;  // last m with row0[m] <= t
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (s.row0[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// token t's row in its source buffer
__device__ __forceinline__ const uint8_t* src_row(const SrcTable& st, int t, size_t row_bytes) {
  const int m = src_of_token(st, t);
  return reinterpret_cast<const uint8_t*>(st.src[m]) + (size_t)(t - st.row0[m]) * row_bytes;
}

// ---------------------------------------------------------------- workspace
struct Workspace {
  int32_t* topk_idx = nullptr;  // [maxT*k]
  float* topk_w = nullptr;      // [maxT*k]
  float* logits = nullptr;      // [maxT*E]
  int32_t* tile_counter = nullptr;  // [ceil(maxT/kRouterTokTile)]
  int32_t* tok_ticket = nullptr;    // [maxT] per-token completion tickets of the small-batch router
  int32_t* counts = nullptr;    // [E+S]
  int32_t* offsets = nullptr;   // [E+S+1]
  int32_t* tile_base = nullptr; // [E+S+1], prefix of ceil(counts / GEMM tile tokens)
  int32_t* gu_done = nullptr;   // [E+S] gate/up items finished per group (bf16 GEMMs; zeroed by the routing)
  int32_t* block_hist = nullptr; // [ceil(maxT/256)][E] per-block expert counts of the routing kernels
  int32_t* perm = nullptr;      // [max_rows] token of each packed row
  int32_t* pos = nullptr;       // [maxT*k]  packed row of each (t, j)
  float* row_w = nullptr;       // [max_rows] routing weight of each packed row
  void* P = nullptr;            // [max_rows, H] packed activations
  float* P_scale = nullptr;     // [H/128][scale_ld] (fp8), K-block major: one block's scales are contiguous by row
  void* Hb = nullptr;           // [max_rows, I] SwiGLU output
  float* H_scale = nullptr;     // [I/128][scale_ld] (fp8), same layout
  int scale_ld = 0;             // row stride of P_scale / H_scale (= max_rows)
  void* Y = nullptr;            // [max_rows, H] weighted expert outputs
  int* err = nullptr;           // device error word
  void* stage = nullptr;        // forward_host staging: [maxT, H] in + [maxT, H] out
  float* rpart = nullptr;       // [kRouterMaxSplits][maxT][E] router logit partials
  int last_T = 0;
  bool direct = false;          // the last forward's gate/up read its tokens from the sources (P unwritten)
  CUtensorMap tm_P, tm_H;       // B operands of the two GEMMs
  bool ready = false;
};

// ---------------------------------------------------------------- launches
// Programmatic dependent launch.  Every kernel of a forward starts with
// pdl_begin(): griddepcontrol.wait returns once the previous kernel of the
// stream has completed and its writes are visible (a no-op for a normal
// launch), so nothing upstream is read early; launch_dependents then lets the
// next kernel's CTAs be scheduled while this one runs, which hides the next
// launch's latency behind this kernel's tail.  Completion order is unchanged:
// each kernel waits for its predecessor, hence for every earlier one -- with one
// exception: the bf16 down GEMM reads h through per-expert progress counters and
// does not wait for the gate/up grid as a whole, except on its abort path.  It
// completes only after every gate/up increment, so the gate/up grid writes
// nothing the next forward depends on after the down grid has completed.
__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// The two halves, for kernels that start work that does not depend on the
// previous kernel (constant weights, routing tables built two kernels back)
// before waiting.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Order this thread's earlier generic-proxy accesses (an acquire that saw another CTA's
// data) before its later async-proxy ones (TMA reads of that data).
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                            Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Tensor maps of the M source buffers (bf16 [rows, H], 128-row boxes, 128-byte swizzle):
// the tensor-core router reads its token tiles straight from the sources.  Passed by
// value as a kernel parameter (8 KB at the source limit).
struct SrcMaps {
  CUtensorMap m[AFD_MAX_SOURCES];
};

// bf16 layers, batches of at most kDirectMaxTok tokens: no pack runs, and the gate/up GEMM
// loads each packed row's token straight from its source through one-row tensor maps
// (every group then holds at most kDirectMaxTok rows; the token producer takes up to 32,
// one per lane), with a work list it builds from the router's top-k.  The limit is where
// the two forms cross (qwen3 shapes, ms per step, pack then direct: 6 tokens 0.2333 /
// 0.2322, 8 tokens 0.3004 / 0.2968, 12 tokens 0.3896 / 0.3913, 32 tokens 0.5770 /
// 0.6218): one copy per row and K block, against one 32-row box from P, costs more as
// the groups grow.
constexpr int kDirectMaxTok = 8;
struct DirectSrc {
  SrcMaps maps;                    // one-row boxes: 64 columns x 1 row, 128-byte swizzle
  int row0[AFD_MAX_SOURCES + 1];  // as SrcTable::row0
  int M;
  const int32_t* topk_idx;         // [T][k] the router's picks: the GEMM builds the tables from them
  int T, k, E, S;
};

// ---------------------------------------------------------------- launchers
struct LayerDims {
  int H, I, E, k, S, dtype;  // dtype: afd_dtype
};

cudaError_t launch_router(const SrcTable& st, const void* wrT, const float* bias, const LayerDims& d,
                          Workspace& ws, cudaStream_t s);
cudaError_t router_setup();  // opt-in shared memory sizes (once per process)
cudaError_t router_tc_setup();
int router_tc_launches(const LayerDims& d, int T, int num_sms);  // kernels launch_router_tc enqueues
cudaError_t launch_router_wnorm(const void* wrT, int H, int E, float* wnorm, cudaStream_t s);
// maps: the sources' tensor maps, read when router_tc_launches(d, T, num_sms) > 1
cudaError_t launch_router_tc(const SrcTable& st, const SrcMaps& maps, const void* wrT, const float* bias,
                             const float* wnorm, const CUtensorMap* tm_wr, const LayerDims& d, Workspace& ws,
                             int num_sms, cudaStream_t s);
cudaError_t launch_routing(const LayerDims& d, int T, Workspace& ws, cudaStream_t s);
int routing_launches(int T);  // 1 for at most 2048 tokens, else 2
cudaError_t launch_pack(const SrcTable& st, const LayerDims& d, int T, Workspace& ws, int num_sms,
                        cudaStream_t s);
cudaError_t launch_combine(const SrcTable& st, const LayerDims& d, int T, Workspace& ws, int num_sms,
                           cudaStream_t s);
cudaError_t launch_gemm_simt(const LayerDims& d, int T, const float* wg, const float* wu, const float* wd,
                             Workspace& ws, cudaStream_t s, int which);  // which: 0 gate/up, 1 down

struct TcWeights {
  const CUtensorMap* tm_wg;  // gate, tiled: per group (I/128) x (H/KW) tiles of 128 rows x 128 bytes
  const CUtensorMap* tm_wu;  // up, same
  const CUtensorMap* tm_wd;  // down, tiled: per group (H/128) x (I/KW) tiles
  const float* sg;           // fp8: [(E+S), I/128, H/128]  (m-block major)
  const float* su;
  const float* sd;           // fp8: [(E+S), H/128, I/128]
};
// which: 0 gate/up + SwiGLU, 1 down.  direct (gate/up of a batch of at most kDirectMaxTok
// tokens only): the token rows come from the sources instead of P.
cudaError_t launch_gemm_tc(const LayerDims& d, int T, const TcWeights& w, Workspace& ws, int num_sms,
                           cudaStream_t s, int which, const DirectSrc* direct = nullptr);
cudaError_t gemm_tc_setup();  // opt-in shared memory sizes (once per process)
int bf16_tile_tokens(const LayerDims& d, int T);  // token-tile width of the bf16 GEMMs for a batch of T
cudaError_t launch_gemm_fp8(const LayerDims& d, int T, const TcWeights& w, Workspace& ws, int num_sms,
                            cudaStream_t s, int which);  // fp8 layer: 0 gate/up + SwiGLU + e4m3 h, 1 down
cudaError_t gemm_fp8_setup();

cudaError_t launch_transpose(const void* src, void* dst, int batch, int rows, int cols, int elem_bytes,
                             cudaStream_t s);
// batch x [K][R] -> per matrix 16 KB tiles (128 rows of R x 128 bytes of K), (row block, K block) order
cudaError_t launch_tile_weights(const void* src, void* dst, int batch, int K, int R, int elem_bytes,
                                cudaStream_t s);
cudaError_t launch_transpose_f32(const float* src, float* dst, int batch, int rows, int cols,
                                 cudaStream_t s);

// ---------------------------------------------------------------- device helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// --- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar`, giving up after about `limit_cycles` SM
// clocks (~2 s at GB300 clocks) or as soon as another thread of the CTA raised
// `*abort`.  The clock and the abort flag are read once every 256 failed
// polls, so a wait that succeeds quickly costs nothing extra.  On a timeout
// the CTA abort flag and the kErrTimeout bit of the device error word are set.
// Returns false when the caller must abandon its work.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int* err,
                                          long long limit_cycles = 4000000000ll) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*abort) return false;
      if (clock64() - t0 > limit_cycles) {
        *abort = 1;
        atomicOr(err, kErrTimeout);
        return false;
      }
    }
  }
}

// A block that waits on a barrier nothing arrives on, through mbar_wait with a
// limit of `limit` cycles: the fault-path test of the bounded waits (sets the
// kErrTimeout bit and returns).
__global__ void wait_probe_kernel(int* err, long long limit);

// Wait until *p >= target (acquire), with the same bound and abort flag as mbar_wait.
__device__ __forceinline__ bool wait_count(const int* p, int target, volatile int* abort, int* err) {
  if (ld_acquire_gpu(p) >= target) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(64);
    if (ld_acquire_gpu(p) >= target) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (clock64() - t0 > 4000000000ll) {
        *abort = 1;
        atomicOr(err, kErrTimeout);
        return false;
      }
    }
  }
}

// Bounded wait without the abort flag (drains in-flight copies and MMAs).
__device__ __forceinline__ bool mbar_wait_cycles(uint64_t* bar, uint32_t parity, long long limit_cycles) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > limit_cycles) return false;
  return true;
}

// --- TMA (tiled, 2D) global -> shared, completion on an mbarrier
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
// Contiguous bulk copy global -> shared (both 16-byte aligned, bytes a
// multiple of 16), completing on `bar` with `bytes` of transaction count.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
// Prefetch one tile of a tensor map into L2 only (no shared memory, no
// barrier): lets HBM requests run further ahead than the shared-memory ring.
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// 16-byte read-only load with an L2 cache-policy hint
__device__ __forceinline__ uint4 ld_nc_hint_v4(const void* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.b32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

// --- tcgen05 / TMEM
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive once on `bar` when all tcgen05.mma issued so far by this thread complete.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16 (bf16 inputs, fp32 accumulate)
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Same for e4m3 x e4m3 (kind::f8f6f4), fp32 accumulate.
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 lanes x 32 consecutive fp32 columns: thread i of the warp gets row
// (lane base + i), columns [col, col+32).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
// The tile must start on a 1024-byte boundary.
__device__ __forceinline__ uint64_t sw128_desc(const void* tile) {
  uint64_t a = smem_u32(tile);
  uint64_t d = 0;
  d |= (a >> 4) & 0x3fffull;          // start address (16-byte units)
  d |= 1ull << 16;                    // leading byte offset (unused when swizzled)
  d |= (uint64_t)(1024 >> 4) << 32;   // stride byte offset: next 8-row group
  d |= 1ull << 46;                    // descriptor version
  d |= 2ull << 61;                    // 128-byte swizzle
  return d;
}

// Instruction descriptor: fp32 accumulate, both operands K-major, M x N.
// ab_fmt: kind::f16 -> 1 = bf16; kind::f8f6f4 -> 0 = e4m3.
__device__ __forceinline__ uint32_t mma_idesc(uint32_t ab_fmt, int M, int N) {
  return (1u << 4) | (ab_fmt << 7) | (ab_fmt << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

}  // namespace afd
