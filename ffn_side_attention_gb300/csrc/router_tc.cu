// router_tc.cu -- R1 for bf16/fp8 layers: the same top-k as the canonical
// fp32 router (router.cu), with the bulk of the logits on the tensor cores.
//
// "MoE 大规模分布式推理工程实战", section 4.1: logits of a bias-free linear
// gate (+ optional bias), top-k on the logits, softmax over the selected.
//
// The selection is defined by the canonical fp32 logits L (router.cu's order).
// Computing all T*E of them on CUDA cores is most of the router's cost, but
// only the experts near a token's k-th largest logit can change the answer:
//   1. logits: Lt = X . Wr on tcgen05 (bf16 in, fp32 accumulate), the token
//      tiles read by TMA straight from the source buffers (a tile never spans two
//      sources), K split over CTAs into fp32 partials added in a fixed order;
//   2. select (one warp per token): ||x_t||_2 from the token row (rounded up), then
//      with b_e a bound on |Lt_e - L_e|, the
//      canonical top-k is contained in C = {e : Lt_e + b_e >= m}, m = k-th
//      largest of Lt - b (k experts have L >= m, and any e outside C has
//      L_e <= Lt_e + b_e < m).  The canonical L is then computed for the
//      candidates only (same order as router.cu), and the top-k and weights
//      are taken from those exact values.  Over 64 candidates -> all experts.
// Small batches (a grid of at most kSmallRouterWaves waves of (8 tokens x 8
// experts) blocks) skip the estimate: one kernel computes every canonical
// logit and the top-k (latency, not work, bounds them there).
// Bound: |Lt - exact| + |L - exact| <= (g_tc + g_c) * sum_h |x_h w_h|, and
// sum |x w| <= ||x|| ||w_e|| (Cauchy-Schwarz, both norms rounded up).
// g_c = n u / (1 - n u), n = H/32 + 6, u = 2^-24 (the fp32 fma chain and fold);
// g_tc = (H/8 + splits + 2) * 2^-21: the tensor core multiplies bf16 values
// exactly and adds them to its fp32 accumulator in groups (16 products per
// K=16 instruction); it is taken to lose at most 2^-21 of sum |x w| per group
// of 8 products (fp32 accumulation with truncation loses at most 2^-23 per
// rounding: a factor 4 of margin, and a rounding counted every 8 products
// rather than every 16), plus one step per split partial and two more.  The
// GPU test of this band measures, on every shape the layer runs this path on,
// the estimate's error against the canonical logits.  Each side's bias
// addition adds 2^-24 |Lt| rounding, covered by an extra
// 2^-22 (|Lt_e| + |bias_e|) + 2^-100.
#include <cuda_bf16.h>

#include "afd_internal.cuh"

namespace afd {
namespace {

constexpr int kMaxCand = 64;
// small-batch path while its grid is at most this many waves (with 128 experts: up to 152
// tokens; at 192 and 197 tokens the estimate path took 23.5 us against 33.6 us for this one)
constexpr int kSmallRouterWaves = 2;

// ---------------------------------------------------------------- 1. logits
constexpr int kRBM = 128;                     // experts per MMA tile
constexpr int kRBN = 128;                     // tokens per tile
constexpr int kRStages = 4;
constexpr int kRTile = 128 * 128;             // 16 KB: 128 rows x 64 bf16
constexpr int kRStageBytes = 2 * kRTile;
constexpr int kRDynSmem = kRStages * kRStageBytes + 1024;
constexpr long long kRDrainCycles = 400000000ll;

struct LogitArgs {
  int T, E, num_kb, kb_per_split;
  float* part;  // [splits][T][E]
  int* err;
  int nsrc;                          // sources
  int tile0[AFD_MAX_SOURCES + 1];    // first token tile of each source (prefix of ceil(rows / 128))
  int row0[AFD_MAX_SOURCES + 1];     // first token of each source
};

// CTA (n, m, s): token tile n (tile j of source src: its tokens [128 j, +128)),
// experts [128 m, +128), K blocks of split s.  Rows past the source's end are read
// as zeros and not stored.
__global__ void __launch_bounds__(192, 1)
    router_logits_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ SrcMaps maps,
                            const LogitArgs args) {
  pdl_begin();
  extern __shared__ uint8_t dyn_smem[];
  uint8_t* smem = dyn_smem + ((1024u - (smem_u32(dyn_smem) & 1023u)) & 1023u);
  __shared__ __align__(8) uint64_t bars[2 * kRStages + 2];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  uint64_t* full = bars;
  uint64_t* empty = bars + kRStages;
  uint64_t* tfull = bars + 2 * kRStages;
  uint64_t* drain = tfull + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int lo = 0, hi = args.nsrc - 1;  // last source whose first tile is at most this one
  while (lo < hi) {                // (an empty source shares its first tile with the next)
    const int mid = (lo + hi + 1) >> 1;
    if (args.tile0[mid] <= (int)blockIdx.x) lo = mid; else hi = mid - 1;
  }
  const int src = lo;
  const int jt = (int)blockIdx.x - args.tile0[src];
  const int n0 = args.row0[src] + jt * kRBN, m0 = blockIdx.y * kRBM;
  const int nrows = min(kRBN, args.row0[src + 1] - n0);
  const CUtensorMap* tmX = &maps.m[src];
  const int kb0 = blockIdx.z * args.kb_per_split;
  const int nkb = min(args.kb_per_split, args.num_kb - kb0);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(drain, 1);
    s_abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(tmX);
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort = &s_abort;
  if (warp == 0 && lane == 0) {
    int s = 0;
    uint32_t ph = 0, filled = 0, fill_ph = 0;
    bool ok = true;
    for (int kb = 0; kb < nkb; ++kb) {
      if (!mbar_wait(&empty[s], ph ^ 1u, abort, args.err)) {
        ok = false;
        break;
      }
      uint8_t* st = smem + s * kRStageBytes;
      mbar_arrive_expect_tx(&full[s], 2 * kRTile);
      tma_load_2d(st, &tmW, &full[s], (kb0 + kb) * 64, m0);
      tma_load_2d(st + kRTile, tmX, &full[s], (kb0 + kb) * 64, jt * kRBN);
      filled |= 1u << s;
      fill_ph = (fill_ph & ~(1u << s)) | (ph << s);
      if (++s == kRStages) {
        s = 0;
        ph ^= 1u;
      }
    }
    if (!ok)
      for (int q = 0; q < kRStages; ++q)
        if ((filled >> q) & 1u) mbar_wait_cycles(&full[q], (fill_ph >> q) & 1u, kRDrainCycles);
  } else if (warp == 1 && lane == 0) {
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    const uint32_t idesc = mma_idesc(1u, kRBM, kRBN);
    for (int kb = 0; kb < nkb; ++kb) {
      if (!mbar_wait(&full[s], ph, abort, args.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint8_t* st = smem + s * kRStageBytes;
      const uint64_t da = sw128_desc(st), db = sw128_desc(st + kRTile);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) mma_f16(tmem, da + 2 * kk, db + 2 * kk, idesc, (kb | kk) ? 1u : 0u);
      tc_commit(&empty[s]);
      if (++s == kRStages) {
        s = 0;
        ph ^= 1u;
      }
    }
    if (ok) tc_commit(tfull);
    tc_commit(drain);
    mbar_wait_cycles(drain, 0, kRDrainCycles);
  } else if (warp >= 2) {
    const int quad = warp & 3;
    const int e = m0 + quad * 32 + lane;
    if (nkb > 0 && mbar_wait(tfull, 0, abort, args.err)) {
      tc_fence_after();
      const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
      float* out = args.part + (size_t)blockIdx.z * args.T * args.E;
      for (int c = 0; c < nrows; c += 32) {
        float d[32];
        tmem_ld_32x32b_x32(t_lane + (uint32_t)c, d);
        tmem_ld_wait();
        if (e < args.E) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c + j < nrows) out[(size_t)(n0 + c + j) * args.E + e] = d[j];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// ---------------------------------------------------------------- 2. select
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

// Canonical dot (router.cu's order): lane l runs the fma chain over chunks
// l, l+32, ... of 8 channels, then the xor fold.  All lanes return the sum.
// Loads are issued D chunks ahead of the chain; the chain's order is
// unchanged.
template <int D>
__device__ __forceinline__ float canonical_dot_warp(const uint16_t* __restrict__ x, const uint16_t* __restrict__ w,
                                                    int H, int lane) {
  const int nc = H >> 3;
  const uint4* xa = reinterpret_cast<const uint4*>(x);
  const uint4* wa = reinterpret_cast<const uint4*>(w);
  float p = 0.0f;
  for (int c0 = lane; c0 < nc; c0 += 32 * D) {
    uint4 a[D], b[D];
#pragma unroll
    for (int i = 0; i < D; ++i)
      if (c0 + 32 * i < nc) {
        a[i] = __ldg(xa + c0 + 32 * i);
        b[i] = __ldg(wa + c0 + 32 * i);
      }
#pragma unroll
    for (int i = 0; i < D; ++i)
      if (c0 + 32 * i < nc) {
        p = fma_bf16_lo(a[i].x, b[i].x, p); p = fma_bf16_hi(a[i].x, b[i].x, p);
        p = fma_bf16_lo(a[i].y, b[i].y, p); p = fma_bf16_hi(a[i].y, b[i].y, p);
        p = fma_bf16_lo(a[i].z, b[i].z, p); p = fma_bf16_hi(a[i].z, b[i].z, p);
        p = fma_bf16_lo(a[i].w, b[i].w, p); p = fma_bf16_hi(a[i].w, b[i].w, p);
      }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) p = p + __shfl_xor_sync(0xffffffffu, p, o);
  return p;
}

// Two canonical dots of one token row against two expert rows: one pass over
// the chunks loads x once and advances both chains (each in the order above).
__device__ __forceinline__ float chain8(const uint4& a, const uint4& b, float p) {
  p = fma_bf16_lo(a.x, b.x, p); p = fma_bf16_hi(a.x, b.x, p);
  p = fma_bf16_lo(a.y, b.y, p); p = fma_bf16_hi(a.y, b.y, p);
  p = fma_bf16_lo(a.z, b.z, p); p = fma_bf16_hi(a.z, b.z, p);
  p = fma_bf16_lo(a.w, b.w, p); p = fma_bf16_hi(a.w, b.w, p);
  return p;
}
__device__ __forceinline__ void canonical_dot2_warp(const uint16_t* __restrict__ x, const uint16_t* __restrict__ w1,
                                                    const uint16_t* __restrict__ w2, int H, int lane, float& v1,
                                                    float& v2) {
  const int nc = H >> 3;
  const uint4* xa = reinterpret_cast<const uint4*>(x);
  const uint4* wa = reinterpret_cast<const uint4*>(w1);
  const uint4* wb = reinterpret_cast<const uint4*>(w2);
  float p1 = 0.0f, p2 = 0.0f;
  for (int c = lane; c < nc; c += 32) {
    const uint4 a = __ldg(xa + c), b = __ldg(wa + c), d = __ldg(wb + c);
    p1 = chain8(a, b, p1);
    p2 = chain8(a, d, p2);
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    p1 = p1 + __shfl_xor_sync(0xffffffffu, p1, o);
    p2 = p2 + __shfl_xor_sync(0xffffffffu, p2, o);
  }
  v1 = p1;
  v2 = p2;
}

// Four canonical dots in one pass (x read once for four expert rows).
__device__ __forceinline__ void canonical_dot4_warp(const uint16_t* __restrict__ x, const uint16_t* const (&w)[4],
                                                    int H, int lane, float (&v)[4]) {
  const int nc = H >> 3;
  const uint4* xa = reinterpret_cast<const uint4*>(x);
  float p[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int c = lane; c < nc; c += 32) {
    const uint4 a = __ldg(xa + c);
    uint4 b[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) b[i] = __ldg(reinterpret_cast<const uint4*>(w[i]) + c);
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = chain8(a, b[i], p[i]);
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = p[i] + __shfl_xor_sync(0xffffffffu, p[i], o);
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = p[i];
}

// The same two dots with the token row in shared memory (xs: this warp's copy).
__device__ __forceinline__ void canonical_dot2_xs(const uint4* xs, const uint16_t* __restrict__ w1,
                                                  const uint16_t* __restrict__ w2, int H, int lane, float& v1,
                                                  float& v2) {
  const int nc = H >> 3;
  const uint4* wa = reinterpret_cast<const uint4*>(w1);
  const uint4* wb = reinterpret_cast<const uint4*>(w2);
  float p1 = 0.0f, p2 = 0.0f;
  // unrolled so that several chunks' router-row loads are in flight ahead of the
  // chains; each lane's chain still runs over its chunks in ascending order
#pragma unroll 8
  for (int c = lane; c < nc; c += 32) {
    const uint4 a = xs[c], b = __ldg(wa + c), d = __ldg(wb + c);
    p1 = chain8(a, b, p1);
    p2 = chain8(a, d, p2);
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    p1 = p1 + __shfl_xor_sync(0xffffffffu, p1, o);
    p2 = p2 + __shfl_xor_sync(0xffffffffu, p2, o);
  }
  v1 = p1;
  v2 = p2;
}
__device__ __forceinline__ float canonical_dot_xs(const uint4* xs, const uint16_t* __restrict__ w, int H, int lane) {
  const int nc = H >> 3;
  const uint4* wa = reinterpret_cast<const uint4*>(w);
  float p = 0.0f;
#pragma unroll 8
  for (int c = lane; c < nc; c += 32) p = chain8(xs[c], __ldg(wa + c), p);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) p = p + __shfl_xor_sync(0xffffffffu, p, o);
  return p;
}

// Order-preserving key of a float: larger value, larger key; +0 and -0 share one
// key, as they compare equal.  Key 0 is below every value's key (that of -inf is
// 0x007fffff) and marks an entry that is taken or absent.
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t b = __float_as_uint(__fadd_rn(v, 0.0f));  // -0 + 0 = +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Warp-wide best entry (value desc, id asc; entry q of lane l is id l + 32 q) among
// the keys not yet 0: one max-reduction over the warp, then the lowest id holding
// that key.  The entry's key is set to 0 (taken); returns its id.
template <int PER>
__device__ __forceinline__ int warp_take_best(uint32_t (&key)[PER], int lane) {
  uint32_t best = 0;
#pragma unroll
  for (int q = 0; q < PER; ++q) best = max(best, key[q]);
  const uint32_t w = __reduce_max_sync(0xffffffffu, best);
  int bi = 0;
#pragma unroll
  for (int q = PER - 1; q >= 0; --q) {
    const unsigned m = __ballot_sync(0xffffffffu, key[q] == w);
    if (m) bi = 32 * q + __ffs(m) - 1;
  }
#pragma unroll
  for (int q = 0; q < PER; ++q)
    if (lane + 32 * q == bi) key[q] = 0u;
  return bi;
}

// value of entry e (warp-uniform) to every lane
template <int PER>
__device__ __forceinline__ float warp_value(const float (&v)[PER], int e) {
  float x = v[0];
#pragma unroll
  for (int q = 1; q < PER; ++q)
    if (q == (e >> 5)) x = v[q];
  return __shfl_sync(0xffffffffu, x, e & 31);
}

// Top-k (value desc, id asc) among the entries not marked in tk, then the
// softmax over the selected: lane j writes slot j.  The exponentials are those
// of one thread's loop over the slots and their sum runs in slot order.
template <int PER>
__device__ __forceinline__ void write_topk(const float (&lc)[PER], const bool (&tk)[PER], int k, int lane,
                                           int32_t* __restrict__ idx, float* __restrict__ wout) {
  uint32_t key[PER];
#pragma unroll
  for (int q = 0; q < PER; ++q) key[q] = tk[q] ? 0u : order_key(lc[q]);
  float my_v = 0.0f;  // lane j: the j-th selected value and expert
  int my_i = 0;
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    const int bi = warp_take_best<PER>(key, lane);
    const float bv = warp_value<PER>(lc, bi);
    if (lane == j) {
      my_v = bv;
      my_i = bi;
    }
  }
  const float v0 = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = expf(my_v - v0);
  float den = 0.0f;
#pragma unroll 1
  for (int j = 0; j < k; ++j) den += __shfl_sync(0xffffffffu, ex, j);
  if (lane < k) {
    idx[lane] = my_i;
    wout[lane] = ex / den;
  }
}

// Token rows of one select block in shared memory: used up to H = 4096.  At H = 7168
// (112 KB per block) the router was slower (DeepSeek-V3 T=4096: 150 -> 199 us).
constexpr int kSelXsMaxBytes = 8 * 4096 * 2;
constexpr int kSelXsThreeBytes = 220 * 1024;  // three such blocks per SM

struct SelectArgs {
  SrcTable st;          // token rows, read in place from the source buffers
  const uint16_t* wrT;  // [E][H]
  const float* wnorm;   // [E], rounded up
  const float* bias;
  const float* part;    // [splits][T][E]
  int splits, T, H, E, k;
  float g;              // g_tc + g_c
  float* logits;
  int32_t* topk_idx;
  float* topk_w;
};

// One warp per token (8 tokens per block): for many tokens, every warp runs
// its token from the bounds to the weights without waiting for the others.
// MINB = blocks per SM the register budget is sized for: 2 gives each warp
// registers for two dot chains at once, 3 fits 50% more tokens per wave (the
// launcher takes 3 only when that turns a second wave into none).  XS: each
// warp first copies its token row into shared memory, so the candidate dots
// read only the expert rows from L2 (the row is reused by every candidate).
// PER = entries per lane (E <= 32 PER): the selection rounds and the candidate
// bookkeeping cost instructions per entry, and with a whole wave of warps on the
// SMs the kernel is bound by instruction issue (T=3160: 58 -> 50 us with PER = 4
// instead of 8 for 128 experts, and the split partials loaded four splits at a time).
template <int MINB, bool XS, int PER>
__global__ void __launch_bounds__(256, MINB) router_select_warp_kernel(const SelectArgs a) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= a.T) return;
  extern __shared__ uint4 sel_xs[];  // XS: [8 warps][H / 8]
  uint4* xs = sel_xs + (size_t)(threadIdx.x >> 5) * (a.H >> 3);
  const uint16_t* x = reinterpret_cast<const uint16_t*>(src_row(a.st, t, (size_t)a.H * 2));
  float xn;  // ||x_t||_2 rounded up (lane chains over its chunks, then a butterfly), and with
  {          // XS the row into shared memory on the same pass
    const uint4* xg = reinterpret_cast<const uint4*>(x);
    float ss = 0.0f;
    for (int c = lane; c < (a.H >> 3); c += 32) {
      const uint4 u = __ldg(xg + c);
      if (XS) xs[c] = u;
      const float f[8] = {bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y),
                          bf16_lo(u.z), bf16_hi(u.z), bf16_lo(u.w), bf16_hi(u.w)};
#pragma unroll
      for (int q = 0; q < 8; ++q) ss = fmaf(f[q], f[q], ss);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    xn = sqrtf(ss) * (1.0f + 1.0f / 1024.0f);
    if (XS) __syncwarp();
  }
  const int E = a.E, k = a.k;
  float* lrow = a.logits + (size_t)t * E;
  float lo[PER], hi[PER];  // bounds of the estimate (the estimate itself goes to the logits row now)
  bool taken[PER];
  float est[PER], wn[PER], bs[PER];
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    const int e = lane + 32 * q;
    taken[q] = e >= E;
    est[q] = 0.0f;
    wn[q] = taken[q] ? 0.0f : __ldg(a.wnorm + e);
    bs[q] = (taken[q] || !a.bias) ? 0.0f : __ldg(a.bias + e);
  }
  // the split partials, four splits of every group in flight at once; each sum in split order
  for (int sp0 = 0; sp0 < a.splits; sp0 += 4) {
    float pv[4][PER];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int q = 0; q < PER; ++q)
        pv[u][q] = (sp0 + u < a.splits && !taken[q])
                       ? __ldcg(a.part + ((size_t)(sp0 + u) * a.T + t) * E + lane + 32 * q)
                       : 0.0f;
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int q = 0; q < PER; ++q)
        if (sp0 + u < a.splits) est[q] += pv[u][q];
  }
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    const int e = lane + 32 * q;
    lo[q] = hi[q] = 0.0f;
    if (e < E) {
      float s = est[q];
      if (a.bias) s = __fadd_rn(s, bs[q]);
      const float b = a.g * xn * wn[q] + 0x1p-22f * (fabsf(s) + fabsf(bs[q])) + 0x1p-100f;
      lrow[e] = s;  // replaced by the canonical value below if e is a candidate
      lo[q] = s - b;
      hi[q] = s + b;
    }
  }
  // m = k-th largest lower end
  float m = 0.0f;
  {
    uint32_t key[PER];
#pragma unroll
    for (int q = 0; q < PER; ++q) key[q] = taken[q] ? 0u : order_key(lo[q]);
    int bi = 0;
#pragma unroll 1
    for (int j = 0; j < k; ++j) bi = warp_take_best<PER>(key, lane);
    m = warp_value<PER>(lo, bi);
  }
  // candidates: upper end >= m
  unsigned cmask[PER];
  int ncand = 0;
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    cmask[q] = __ballot_sync(0xffffffffu, !taken[q] && hi[q] >= m);
    ncand += __popc(cmask[q]);
  }
  const bool all = ncand > kMaxCand;
  // canonical logits of the candidates (all experts when too many)
  float lc[PER];
  if (XS) {  // token row in shared memory: two candidates of a group of 32 per pass
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      lc[q] = -INFINITY;
      unsigned msk = all ? __ballot_sync(0xffffffffu, !taken[q]) : cmask[q];
      while (msk) {
        const int s1 = __ffs(msk) - 1;
        msk &= msk - 1;
        const int e1 = s1 + 32 * q;
        float v1, v2 = 0.0f;
        int s2 = -1;
        if (msk) {
          s2 = __ffs(msk) - 1;
          msk &= msk - 1;
          canonical_dot2_xs(xs, a.wrT + (size_t)e1 * a.H, a.wrT + (size_t)(s2 + 32 * q) * a.H, a.H, lane, v1, v2);
        } else {
          v1 = canonical_dot_xs(xs, a.wrT + (size_t)e1 * a.H, a.H, lane);
        }
        if (a.bias) v1 = __fadd_rn(v1, __ldg(a.bias + e1));
        if (lane == s1) lc[q] = v1;
        if (s2 >= 0) {
          if (a.bias) v2 = __fadd_rn(v2, __ldg(a.bias + s2 + 32 * q));
          if (lane == s2) lc[q] = v2;
        }
      }
    }
  } else {  // token row from L2: up to four candidates (from any group) per pass over it
    unsigned cm[PER];  // candidates still to compute, per group of 32 experts (warp-uniform)
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      lc[q] = -INFINITY;
      cm[q] = all ? __ballot_sync(0xffffffffu, !taken[q]) : cmask[q];
    }
    // the value of expert e goes to lane e % 32 of group e / 32
    auto put = [&](int e, float v) {
      if (a.bias) v = __fadd_rn(v, __ldg(a.bias + e));
#pragma unroll
      for (int q = 0; q < PER; ++q)
        if (q == (e >> 5) && lane == (e & 31)) lc[q] = v;
    };
    auto next = [&]() {  // lowest remaining candidate
      int e = -1;
#pragma unroll
      for (int q = PER - 1; q >= 0; --q)
        if (cm[q]) e = 32 * q + __ffs(cm[q]) - 1;
#pragma unroll
      for (int q = 0; q < PER; ++q)
        if (q == (e >> 5)) cm[q] &= cm[q] - 1;
      return e;
    };
    int left = 0;
#pragma unroll
    for (int q = 0; q < PER; ++q) left += __popc(cm[q]);
    for (; left >= 4; left -= 4) {
      int e4[4];
      const uint16_t* w4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        e4[i] = next();
        w4[i] = a.wrT + (size_t)e4[i] * a.H;
      }
      float v4[4];
      canonical_dot4_warp(x, w4, a.H, lane, v4);
#pragma unroll
      for (int i = 0; i < 4; ++i) put(e4[i], v4[i]);
    }
    if (left >= 2) {
      const int e1 = next(), e2 = next();
      float v1, v2;
      canonical_dot2_warp(x, a.wrT + (size_t)e1 * a.H, a.wrT + (size_t)e2 * a.H, a.H, lane, v1, v2);
      put(e1, v1);
      put(e2, v2);
      left -= 2;
    }
    if (left) {
      const int e1 = next();
      put(e1, canonical_dot_warp<1>(x, a.wrT + (size_t)e1 * a.H, a.H, lane));
    }
  }
  // logits row for inspection: canonical where computed (the estimate stays elsewhere)
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    const int e = lane + 32 * q;
    if (e < E && (all || ((cmask[q] >> lane) & 1u))) lrow[e] = lc[q];
  }
  // top-k among the exact values (non-candidates are -inf and never win)
  bool tk[PER];
#pragma unroll
  for (int q = 0; q < PER; ++q) tk[q] = taken[q] || !(all || ((cmask[q] >> lane) & 1u));
  write_topk<PER>(lc, tk, k, lane, a.topk_idx + (size_t)t * k, a.topk_w + (size_t)t * k);
}

// ---------------------------------------------------------------- small batches
// Few tokens: every logit in the canonical order, straight from the source
// buffers, in one launch (no staging, no estimate).  Block = 8 warps = 8
// tokens x kOct experts (2, 4 or 8): thread 0 copies the block's kOct router
// rows (contiguous in W_r) and its token rows into shared memory, bulk copies
// on one barrier; lane l then runs the canonical chain over chunks l, l+32, ...
// for the kOct experts at once (kOct independent chains).  The chunk loop
// stays rolled: fully unrolled over a token row held in registers, the kernel
// was slower (qwen3 shapes, 6 tokens: 20.5 -> 17.3 us per router launch with
// this form).
// The last warp to finish a token (atomic ticket per token) selects its top-k
// from the stored logits and resets the ticket.
constexpr int kSelWarps = 8;
constexpr int kOctMax = 8;            // experts per block: 2, 4 or 8
constexpr int kSmallMaxChunks = 28;   // H <= 7168: chunks of 8 channels per lane
constexpr int kSmallMaxH = 32 * 8 * kSmallMaxChunks;
constexpr int kSmallDynSmem = (kOctMax + kSelWarps) * kSmallMaxH * 2;  // 224 KB

template <int kOct, int PER>
__global__ void __launch_bounds__(32 * kSelWarps, 1)
    router_small_kernel(const SrcTable st, const uint16_t* __restrict__ wrT, const float* __restrict__ bias, int H,
                        int E, int k, float* __restrict__ logits, int32_t* __restrict__ topk_idx,
                        float* __restrict__ topk_w, int32_t* __restrict__ ticket, int* err) {
  extern __shared__ __align__(16) uint4 s_w[];  // [kOct][H/8] router rows, then [8][H/8] token rows
  __shared__ __align__(8) uint64_t bar;
  __shared__ int s_abort;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int noct = (E + kOct - 1) / kOct;
  const int oct = blockIdx.x % noct;
  const int e0 = oct * kOct, ne = min(kOct, E - e0);
  const int nc = H >> 3;
  // the router rows are weights: their copy starts before the wait on the previous kernel,
  // the token rows' after it (a caller may feed one layer's outputs back as the sources)
  if (threadIdx.x == 0) {
    s_abort = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
    const int tok0 = (blockIdx.x / noct) * kSelWarps, ntok = min(kSelWarps, st.T - tok0);
    mbar_arrive_expect_tx(&bar, (uint32_t)((ne + ntok) * nc * 16));
    bulk_load(s_w, reinterpret_cast<const uint4*>(wrT) + (size_t)e0 * nc, (uint32_t)(ne * nc * 16), &bar);
  }
  pdl_begin();
  if (threadIdx.x == 0) {
    const int tok0 = (blockIdx.x / noct) * kSelWarps, ntok = min(kSelWarps, st.T - tok0);
    for (int w = 0; w < ntok; ++w) {
      const int tw = tok0 + w, m = src_of_token(st, tw);
      bulk_load(s_w + (size_t)(kOct + w) * nc, reinterpret_cast<const uint4*>(st.src[m]) + (size_t)(tw - st.row0[m]) * nc,
                (uint32_t)(nc * 16), &bar);
    }
  }
  const int tok0 = (blockIdx.x / noct) * kSelWarps;
  const int t = tok0 + warp;
  const bool valid = t < st.T;
  float p[kOct];
#pragma unroll
  for (int i = 0; i < kOct; ++i) p[i] = 0.0f;
  __syncthreads();  // barrier initialised before anyone waits on it
  const bool ok = mbar_wait(&bar, 0, &s_abort, err);  // every thread: the copies land before the block exits
  if (!valid || !ok) return;
  const uint4* xs = s_w + (size_t)(kOct + warp) * nc;
#pragma unroll 2
  for (int c = lane; c < nc; c += 32) {
    const uint4 a = xs[c];
#pragma unroll
    for (int i = 0; i < kOct; ++i)
      if (i < ne) {
        const uint4 b = s_w[i * nc + c];
        p[i] = fma_bf16_lo(a.x, b.x, p[i]); p[i] = fma_bf16_hi(a.x, b.x, p[i]);
        p[i] = fma_bf16_lo(a.y, b.y, p[i]); p[i] = fma_bf16_hi(a.y, b.y, p[i]);
        p[i] = fma_bf16_lo(a.z, b.z, p[i]); p[i] = fma_bf16_hi(a.z, b.z, p[i]);
        p[i] = fma_bf16_lo(a.w, b.w, p[i]); p[i] = fma_bf16_hi(a.w, b.w, p[i]);
      }
  }
  float v = 0.0f;
#pragma unroll
  for (int i = 0; i < kOct; ++i) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) p[i] = p[i] + __shfl_xor_sync(0xffffffffu, p[i], o);
    if (lane == i) v = p[i];
  }
  if (lane < ne) {
    if (bias) v = __fadd_rn(v, __ldg(bias + e0 + lane));
    logits[(size_t)t * E + e0 + lane] = v;
  }
  __threadfence();
  int last = 0;
  if (lane == 0) last = atomicAdd(ticket + t, 1) == noct - 1;
  if (!__shfl_sync(0xffffffffu, last, 0)) return;
  __threadfence();
  float lc[PER];
  bool tk[PER];
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    const int e = lane + 32 * q;
    tk[q] = e >= E;
    lc[q] = e < E ? __ldcg(logits + (size_t)t * E + e) : -INFINITY;
  }
  write_topk<PER>(lc, tk, k, lane, topk_idx + (size_t)t * k, topk_w + (size_t)t * k);
  if (lane == 0) ticket[t] = 0;
}

__global__ void wnorm_kernel(const uint16_t* __restrict__ wrT, int H, int E, float* __restrict__ wnorm) {
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (e >= E) return;
  double ss = 0.0;
  for (int h = lane; h < H; h += 32) {
    const double v = (double)__uint_as_float((uint32_t)wrT[(size_t)e * H + h] << 16);
    ss += v * v;
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) wnorm[e] = (float)(sqrt(ss) * (1.0 + 1.0 / 1024.0));
}

}  // namespace

cudaError_t router_tc_setup() {
  cudaError_t e = cudaFuncSetAttribute(router_logits_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRDynSmem);
  if (e != cudaSuccess) return e;
  for (auto f : {router_select_warp_kernel<2, true, 2>, router_select_warp_kernel<3, true, 2>,
                 router_select_warp_kernel<2, true, 4>, router_select_warp_kernel<3, true, 4>,
                 router_select_warp_kernel<2, true, 8>, router_select_warp_kernel<3, true, 8>}) {
    e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kSelXsMaxBytes);
    if (e != cudaSuccess) return e;
  }
  for (auto f : {router_small_kernel<2, 2>, router_small_kernel<4, 2>, router_small_kernel<8, 2>,
                 router_small_kernel<2, 4>, router_small_kernel<4, 4>, router_small_kernel<8, 4>,
                 router_small_kernel<2, 8>, router_small_kernel<4, 8>, router_small_kernel<8, 8>}) {
    e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmallDynSmem);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// entries per lane of the selection: E <= 32 * PER
static int router_per(int E) { return E <= 64 ? 2 : (E <= 128 ? 4 : 8); }

template <int PER>
static void (*select_kernel(bool three, bool xs))(const SelectArgs) {
  return three ? (xs ? router_select_warp_kernel<3, true, PER> : router_select_warp_kernel<3, false, PER>)
               : (xs ? router_select_warp_kernel<2, true, PER> : router_select_warp_kernel<2, false, PER>);
}

template <int kOct>
static auto small_kernel(int per) {
  return per == 2 ? router_small_kernel<kOct, 2> : (per == 4 ? router_small_kernel<kOct, 4> : router_small_kernel<kOct, 8>);
}

cudaError_t launch_router_wnorm(const void* wrT, int H, int E, float* wnorm, cudaStream_t s) {
  wnorm_kernel<<<(E + 7) / 8, 256, 0, s>>>(static_cast<const uint16_t*>(wrT), H, E, wnorm);
  return cudaGetLastError();
}

int router_tc_splits(const LayerDims& d, int token_tiles, int num_sms) {
  const int tiles = token_tiles * ((d.E + kRBM - 1) / kRBM);
  const int num_kb = d.H / 64;
  int splits = num_sms / tiles;  // whole waves: tiles * splits <= SM count
  splits = splits < 1 ? 1 : splits;
  const int max_splits = num_kb / 4 > 0 ? num_kb / 4 : 1;
  if (splits > max_splits) splits = max_splits;
  if (splits > kRouterMaxSplits) splits = kRouterMaxSplits;
  return splits;
}

// Experts per small-router block: the fewest that keep the grid within one wave.  Each
// warp's chains get shorter with fewer experts, and more SMs share the router rows
// (qwen3 shapes, 6 tokens: 2 experts per block, router 17.4 -> 13.9 us).
static int small_oct(const LayerDims& d, int T, int num_sms) {
  const int tg = (T + kSelWarps - 1) / kSelWarps;
  for (int o = 2; o < kOctMax; o *= 2)
    if ((long)((d.E + o - 1) / o) * tg <= num_sms) return o;
  return kOctMax;
}

static bool router_small_path(const LayerDims& d, int T, int num_sms) {
  const int noct = (d.E + kOctMax - 1) / kOctMax;
  return (long)noct * ((T + kSelWarps - 1) / kSelWarps) <= (long)kSmallRouterWaves * num_sms && d.H <= kSmallMaxH;
}

int router_tc_launches(const LayerDims& d, int T, int num_sms) { return router_small_path(d, T, num_sms) ? 1 : 2; }

cudaError_t launch_router_tc(const SrcTable& st, const SrcMaps& maps, const void* wrT, const float* bias,
                             const float* wnorm, const CUtensorMap* tm_wr, const LayerDims& d, Workspace& ws,
                             int num_sms, cudaStream_t s) {
  const int T = st.T;
  if (T == 0) return cudaSuccess;
  if (router_small_path(d, T, num_sms)) {
    const int oct = small_oct(d, T, num_sms);
    const int noct = (d.E + oct - 1) / oct;
    const int per = router_per(d.E);
    auto kern = oct == 2 ? small_kernel<2>(per) : (oct == 4 ? small_kernel<4>(per) : small_kernel<8>(per));
    {
      const cudaError_t e_ = launch_k(kern, dim3(noct * ((T + kSelWarps - 1) / kSelWarps)),
                                      dim3(32 * kSelWarps), (size_t)(oct + kSelWarps) * d.H * 2, s, st,
                                      static_cast<const uint16_t*>(wrT), bias, d.H, d.E, d.k, ws.logits,
                                      ws.topk_idx, ws.topk_w, ws.tok_ticket, ws.err);
      if (e_ != cudaSuccess) return e_;
    }
    return cudaGetLastError();
  }
  const int num_kb = d.H / 64;
  LogitArgs la{};
  la.T = T;
  la.E = d.E;
  la.num_kb = num_kb;
  la.part = ws.rpart;
  la.err = ws.err;
  la.nsrc = st.M;
  la.tile0[0] = 0;
  for (int m = 0; m < st.M; ++m) {
    la.row0[m] = st.row0[m];
    la.tile0[m + 1] = la.tile0[m] + (st.row0[m + 1] - st.row0[m] + kRBN - 1) / kRBN;
  }
  la.row0[st.M] = st.row0[st.M];
  const int ntiles = la.tile0[st.M];
  const int splits = router_tc_splits(d, ntiles, num_sms);
  la.kb_per_split = (num_kb + splits - 1) / splits;
  const int nsplit = (num_kb + la.kb_per_split - 1) / la.kb_per_split;
  dim3 grid(ntiles, (d.E + kRBM - 1) / kRBM, nsplit);
  {
    const cudaError_t e_ = launch_k(router_logits_tc_kernel, dim3(grid), dim3(192), kRDynSmem, s, *tm_wr, maps, la);
    if (e_ != cudaSuccess) return e_;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  SelectArgs sa{};
  sa.st = st;
  sa.wrT = static_cast<const uint16_t*>(wrT);
  sa.wnorm = wnorm;
  sa.bias = bias;
  sa.part = ws.rpart;
  sa.splits = nsplit;
  sa.T = T;
  sa.H = d.H;
  sa.E = d.E;
  sa.k = d.k;
  const double u = 1.0 / 16777216.0;  // 2^-24
  const double n = d.H / 32.0 + 6.0;
  const double g_c = n * u / (1.0 - n * u);
  const double g_tc = (d.H / 8.0 + nsplit + 2.0) * (1.0 / 2097152.0);  // 2^-21 per 8 products
  sa.g = (float)((g_c + g_tc) * 1.0001);
  sa.logits = ws.logits;
  sa.topk_idx = ws.topk_idx;
  sa.topk_w = ws.topk_w;
  const int blocks = (T + kSelWarps - 1) / kSelWarps;
  // token rows in shared memory when 8 of them fit the opt-in size; 3 blocks per SM
  // only if their rows fit the SM's shared memory too
  const size_t xs_bytes = (size_t)kSelWarps * d.H * 2;
  const bool xs = xs_bytes <= (size_t)kSelXsMaxBytes;
  const bool three = blocks > 2 * num_sms && blocks <= 3 * num_sms && (!xs || 3 * xs_bytes <= kSelXsThreeBytes);
  const int per = router_per(d.E);
  void (*kern)(const SelectArgs) =
      per == 2 ? select_kernel<2>(three, xs) : (per == 4 ? select_kernel<4>(three, xs) : select_kernel<8>(three, xs));
  {
    const cudaError_t e_ = launch_k(kern, dim3(blocks), dim3(32 * kSelWarps), xs ? xs_bytes : 0, s, sa);
    if (e_ != cudaSuccess) return e_;
  }
  return cudaGetLastError();
}

}  // namespace afd
