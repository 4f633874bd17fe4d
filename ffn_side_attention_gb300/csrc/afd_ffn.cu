// afd_ffn.cu -- the C ABI of libafd_ffn.so (declared in include/afd_ffn.h).
//
// Host side only: argument validation, weight re-layout at create time,
// workspace ownership, TMA descriptor set-up and the launch sequence of one
// forward (router -> routing tables -> pack -> gate/up GEMM -> down GEMM ->
// combine; no pack for bf16 batches of at most 8 tokens), all enqueued on the
// caller's stream with no host synchronisation.
// The batch shape (src_counts) is the control-plane metadata of the FastAFD
// blog's transport (section 3); the M device pointers are its data plane.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "afd_internal.cuh"

using afd::LayerDims;
using afd::SrcTable;
using afd::Workspace;

struct afd_ffn {
  afd_ffn_config cfg{};
  LayerDims dims{};
  int device = 0;
  int num_sms = 0;
  size_t max_rows = 0;
  size_t bytes = 0;
  // weights in kernel layout
  void* wrT = nullptr;      // [E, H] router, K-major
  float* bias = nullptr;    // [E] or null
  float* wnorm = nullptr;   // [E] ||w_e||_2 rounded up (bf16/fp8 router bound)
  CUtensorMap tm_wr{};      // router weights for the tensor-core logits
  void* wgT = nullptr;      // gate, per group [I/128][H/KW][128][KW] (KW = 128 bytes of K)
  void* wuT = nullptr;      // up, same
  void* wdT = nullptr;      // down, per group [H/128][I/KW][128][KW]
  float* sgT = nullptr;     // fp8: [(E+S), I/128, H/128]
  float* suT = nullptr;
  float* sdT = nullptr;     // fp8: [(E+S), H/128, I/128]
  float* wg32 = nullptr;    // fp32 layer: [(E+S), H, I]
  float* wu32 = nullptr;
  float* wd32 = nullptr;    // fp32 layer: [(E+S), I, H]
  CUtensorMap tm_wg{}, tm_wu{}, tm_wd{};
  Workspace ws[AFD_MAX_MICRO];
  // tensor maps of each workspace's last sources (the tensor-core router reads its token
  // tiles through them); re-encoded when a source pointer or row count changes
  afd::SrcMaps src_maps[AFD_MAX_MICRO];
  const void* map_src[AFD_MAX_MICRO][AFD_MAX_SOURCES] = {};
  int map_rows[AFD_MAX_MICRO][AFD_MAX_SOURCES] = {};
  // the same with one-row boxes, for the gate/up GEMM's direct form (bf16 batches of at
  // most kDirectMaxTok tokens), with the sources' first rows
  afd::DirectSrc direct_src[AFD_MAX_MICRO];
  const void* map1_src[AFD_MAX_MICRO][AFD_MAX_SOURCES] = {};
  int map1_rows[AFD_MAX_MICRO][AFD_MAX_SOURCES] = {};
  cudaStream_t mstream[AFD_MAX_MICRO] = {};
  cudaEvent_t ev_fork = nullptr;
  cudaEvent_t ev_join[AFD_MAX_MICRO] = {};
  // afd_ffn_forward_host_async: copy-in and copy-out streams, one compute stream per
  // staging slot (sources + outputs), and per slot the events that order reuse
  cudaStream_t astream[4] = {};  // copy-in, compute slot 0, copy-out, compute slot 1
  void* astage[2] = {};
  cudaEvent_t ev_in[2] = {}, ev_done[2] = {}, ev_out[2] = {};
  unsigned long long async_calls = 0;
  int async_last_micro = 1;  // n_micro of the previous asynchronous call
  int route_ws = 0;          // workspace holding the last forward's routing
  int async_rc = 0;  // first error of an enqueued call, reported by afd_ffn_host_wait
  // per-kernel timing: AFD_NUM_KERNELS + 1 events per recorded forward
  bool prof_on = false;
  std::vector<cudaEvent_t> prof_events;
  size_t prof_used = 0;
  std::string err;
};

namespace {

thread_local std::string g_create_err;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int fail(afd_ffn* h, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (h) h->err = buf; else g_create_err = buf;
  return code;
}

#define CUDA_TRY(h, call)                                                                       \
  do {                                                                                          \
    cudaError_t e_ = (call);                                                                    \
    if (e_ != cudaSuccess) return fail((h), AFD_ECUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

bool get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 2D K-major operand: [outer rows][inner K], box = 128 bytes of K x box_rows,
// 128-byte swizzle (matches the tcgen05 shared-memory descriptor).
bool make_map(CUtensorMap* m, void* base, bool fp8, uint64_t inner, uint64_t outer, uint32_t box_rows) {
  const int esz = fp8 ? 1 : 2;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * esz};
  cuuint32_t box[2] = {(cuuint32_t)(128 / esz), box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int dmalloc(afd_ffn* h, void** p, size_t n) {
  *p = nullptr;
  if (n == 0) return AFD_OK;
  cudaError_t e = cudaMalloc(p, n);
  if (e != cudaSuccess) return fail(h, AFD_ECUDA, "cudaMalloc(%zu): %s", n, cudaGetErrorString(e));
  h->bytes += n;
  return AFD_OK;
}

template <typename T>
int dmalloc_t(afd_ffn* h, T** p, size_t count) {
  return dmalloc(h, reinterpret_cast<void**>(p), count * sizeof(T));
}

size_t act_bytes(const afd_ffn_config& c) { return c.dtype == AFD_FP32 ? 4 : 2; }
size_t wt_bytes(const afd_ffn_config& c) { return c.dtype == AFD_FP32 ? 4 : (c.dtype == AFD_BF16 ? 2 : 1); }

int alloc_workspace(afd_ffn* h, Workspace& ws) {
  if (ws.ready) return AFD_OK;
  const afd_ffn_config& c = h->cfg;
  const size_t T = c.max_tokens, k = c.k, E = c.E, G = (size_t)c.E + c.n_shared, R = h->max_rows;
  const size_t ab = c.dtype == AFD_FP8_E4M3 ? 1 : act_bytes(c);  // packed activation element
  const size_t yb = act_bytes(c);
  int rc;
  if ((rc = dmalloc_t(h, &ws.topk_idx, T * k)) || (rc = dmalloc_t(h, &ws.topk_w, T * k)) ||
      (rc = dmalloc_t(h, &ws.logits, T * E)) ||
      (rc = dmalloc_t(h, &ws.tile_counter, (T + afd::kRouterTokTile - 1) / afd::kRouterTokTile)) ||
      (rc = dmalloc_t(h, &ws.tok_ticket, T)) ||
      (rc = dmalloc_t(h, &ws.counts, G)) || (rc = dmalloc_t(h, &ws.offsets, G + 1)) ||
      (rc = dmalloc_t(h, &ws.tile_base, G + 1)) || (rc = dmalloc_t(h, &ws.gu_done, G)) || (rc = dmalloc_t(h, &ws.block_hist, ((T + 255) / 256) * E)) ||
      (rc = dmalloc_t(h, &ws.perm, R)) ||
      (rc = dmalloc_t(h, &ws.pos, T * k)) || (rc = dmalloc(h, &ws.P, R * c.H * ab)) ||
      (rc = dmalloc(h, &ws.Hb, R * c.I * (c.dtype == AFD_FP8_E4M3 ? 1 : act_bytes(c)))) ||
      (rc = dmalloc(h, &ws.Y, R * c.H * yb)) || (rc = dmalloc_t(h, &ws.err, 1)))
    return rc;
  if (c.dtype == AFD_FP8_E4M3) {
    if ((rc = dmalloc_t(h, &ws.P_scale, R * (c.H / 128))) || (rc = dmalloc_t(h, &ws.H_scale, R * (c.I / 128))))
      return rc;
    ws.scale_ld = (int)R;
  }
  if (c.dtype != AFD_FP32)
    if ((rc = dmalloc_t(h, &ws.rpart, (size_t)afd::kRouterMaxSplits * T * E))) return rc;
  CUDA_TRY(h, cudaMemset(ws.tile_counter, 0, sizeof(int32_t) * ((T + afd::kRouterTokTile - 1) / afd::kRouterTokTile)));
  CUDA_TRY(h, cudaMemset(ws.err, 0, sizeof(int)));
  CUDA_TRY(h, cudaMemset(ws.tok_ticket, 0, sizeof(int32_t) * T));
  CUDA_TRY(h, cudaMemset(ws.P, 0, R * c.H * ab));
  CUDA_TRY(h, cudaMemset(ws.Hb, 0, R * c.I * (c.dtype == AFD_FP8_E4M3 ? 1 : act_bytes(c))));
  if (c.dtype != AFD_FP32) {
    const bool fp8 = c.dtype == AFD_FP8_E4M3;
    if (!make_map(&ws.tm_P, ws.P, fp8, c.H, R, 32) || !make_map(&ws.tm_H, ws.Hb, fp8, c.I, R, 32))
      return fail(h, AFD_ECUDA, "cuTensorMapEncodeTiled failed for a workspace operand");
  }
  ws.ready = true;
  return AFD_OK;
}

void free_workspace(Workspace& ws) {
  void* ptrs[] = {ws.topk_idx, ws.topk_w, ws.logits, ws.tile_counter, ws.tok_ticket, ws.counts, ws.offsets, ws.tile_base,
                  ws.block_hist, ws.perm, ws.pos, ws.P, ws.P_scale, ws.Hb, ws.H_scale, ws.Y, ws.err,
                  ws.stage, ws.rpart};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  ws = Workspace{};
}

int validate_config(const afd_ffn_config* c) {
  if (!c) return fail(nullptr, AFD_EINVAL, "config is NULL");
  if (c->dtype != AFD_FP32 && c->dtype != AFD_BF16 && c->dtype != AFD_FP8_E4M3)
    return fail(nullptr, AFD_EINVAL, "unknown dtype %d", (int)c->dtype);
  if (c->H <= 0 || c->I <= 0 || c->E <= 0 || c->k <= 0)
    return fail(nullptr, AFD_EINVAL, "H, I, E, k must be positive");
  if (c->E > 256) return fail(nullptr, AFD_EINVAL, "E=%d exceeds 256 experts", c->E);
  if (c->k > c->E) return fail(nullptr, AFD_EINVAL, "k=%d exceeds E=%d", c->k, c->E);
  if (c->k > 16) return fail(nullptr, AFD_EUNSUPPORTED, "k=%d exceeds the router's 16 slots", c->k);
  if (c->n_shared != 0 && c->n_shared != 1) return fail(nullptr, AFD_EINVAL, "n_shared must be 0 or 1");
  if (c->max_sources < 1 || c->max_sources > AFD_MAX_SOURCES)
    return fail(nullptr, AFD_EINVAL, "max_sources must be in [1, %d]", AFD_MAX_SOURCES);
  if (c->max_tokens < 1) return fail(nullptr, AFD_EINVAL, "max_tokens must be positive");
  if ((long long)c->max_tokens * (c->k + c->n_shared) * (c->H > c->I ? c->H : c->I) >= (1LL << 40))
    return fail(nullptr, AFD_EINVAL, "max_tokens too large");
  if (c->dtype == AFD_FP32) {
    if (c->H % 8) return fail(nullptr, AFD_EINVAL, "fp32 layer needs H %% 8 == 0 (H=%d)", c->H);
  } else {
    if (c->H % 256) return fail(nullptr, AFD_EINVAL, "bf16/fp8 layer needs H %% 256 == 0 (H=%d)", c->H);
    if (c->I % 128) return fail(nullptr, AFD_EINVAL, "bf16/fp8 layer needs I %% 128 == 0 (I=%d)", c->I);
  }
  return AFD_OK;
}

int validate_batch(afd_ffn* h, const void* const* src, const int* counts, int M, void* const* out, int* T_out) {
  if (!h) return AFD_EINVAL;
  if (M < 0 || M > h->cfg.max_sources)
    return fail(h, AFD_ECAPACITY, "M=%d outside [0, max_sources=%d]", M, h->cfg.max_sources);
  if (M > 0 && (!src || !counts || !out)) return fail(h, AFD_EINVAL, "src_ptrs, src_counts, out_ptrs must be non-NULL");
  long long T = 0;
  for (int m = 0; m < M; ++m) {
    if (counts[m] < 0) return fail(h, AFD_EINVAL, "src_counts[%d]=%d is negative", m, counts[m]);
    T += counts[m];
    if (counts[m] == 0) continue;
    if (!src[m] || !out[m]) return fail(h, AFD_EINVAL, "buffer %d has rows but a NULL pointer", m);
    if ((reinterpret_cast<uintptr_t>(src[m]) | reinterpret_cast<uintptr_t>(out[m])) & 15)
      return fail(h, AFD_EINVAL, "buffer %d is not 16-byte aligned", m);
  }
  if (T > h->cfg.max_tokens)
    return fail(h, AFD_ECAPACITY, "T=%lld exceeds max_tokens=%d", T, h->cfg.max_tokens);
  *T_out = (int)T;
  return AFD_OK;
}

SrcTable make_table(const void* const* src, const int* counts, int M, void* const* out) {
  SrcTable st{};
  st.M = M;
  st.row0[0] = 0;
  for (int m = 0; m < M; ++m) {
    st.src[m] = src[m];
    st.out[m] = out[m];
    st.row0[m + 1] = st.row0[m] + counts[m];
  }
  st.T = st.row0[M];
  return st;
}

// Profiling: record the i-th event of the current forward (i = 0 before the
// first kernel, i = n after kernel n).
int prof_mark(afd_ffn* h, int i, cudaStream_t s) {
  if (!h->prof_on) return AFD_OK;
  if (i == 0 && h->prof_used + AFD_NUM_KERNELS + 1 > h->prof_events.size()) {
    for (int q = 0; q <= AFD_NUM_KERNELS; ++q) {
      cudaEvent_t e;
      CUDA_TRY(h, cudaEventCreate(&e));
      h->prof_events.push_back(e);
    }
  }
  CUDA_TRY(h, cudaEventRecord(h->prof_events[h->prof_used + i], s));
  if (i == AFD_NUM_KERNELS) h->prof_used += AFD_NUM_KERNELS + 1;
  return AFD_OK;
}

// The launch sequence of one forward on one workspace.
// NVTX range around the enqueue of one stage (a trace tool maps it onto the stage's
// kernels; without a tool attached the calls return at once)
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Tensor maps of the sources of st (bf16 [rows, H], box_rows-row boxes), encoded again
// only where a pointer or row count changed since the last forward on that cache.
int update_src_maps(afd_ffn* h, const SrcTable& st, afd::SrcMaps& maps, const void** cached_src, int* cached_rows,
                    uint32_t box_rows) {
  for (int m = 0; m < st.M; ++m) {
    const int rows = st.row0[m + 1] - st.row0[m];
    if (rows == 0 || (cached_src[m] == st.src[m] && cached_rows[m] == rows)) continue;
    if (!make_map(&maps.m[m], const_cast<void*>(st.src[m]), false, h->cfg.H, rows, box_rows))
      return fail(h, AFD_ECUDA, "cuTensorMapEncodeTiled failed for source %d", m);
    cached_src[m] = st.src[m];
    cached_rows[m] = rows;
  }
  return AFD_OK;
}

bool direct_form(const afd::LayerDims& d, int T) { return d.dtype == AFD_BF16 && T <= afd::kDirectMaxTok; }

int run_layer(afd_ffn* h, const SrcTable& st, Workspace& ws, cudaStream_t s) {
  const LayerDims& d = h->dims;
  const int T = st.T;
  ws.last_T = T;
  if (T == 0) return AFD_OK;
  NvtxRange range_layer("afd.forward");
  int rc;
  afd::TcWeights w{&h->tm_wg, &h->tm_wu, &h->tm_wd, h->sgT, h->suT, h->sdT};
  const int wi = (int)(&ws - h->ws);
  const bool direct = direct_form(d, T);
  ws.direct = direct;
  afd::DirectSrc* ds = direct ? &h->direct_src[wi] : nullptr;
  if (direct) {
    if ((rc = update_src_maps(h, st, ds->maps, h->map1_src[wi], h->map1_rows[wi], 1))) return rc;
    for (int m = 0; m <= st.M; ++m) ds->row0[m] = st.row0[m];
    ds->M = st.M;
    ds->topk_idx = ws.topk_idx;
    ds->T = T;
    ds->k = d.k;
    ds->E = d.E;
    ds->S = d.S;
  }
  if ((rc = prof_mark(h, 0, s))) return rc;
  {
    NvtxRange r("afd.router");
    if (d.dtype == AFD_FP32)
      CUDA_TRY(h, afd::launch_router(st, h->wrT, h->bias, d, ws, s));
    else
    {
      if (afd::router_tc_launches(d, T, h->num_sms) > 1 &&
          (rc = update_src_maps(h, st, h->src_maps[wi], h->map_src[wi], h->map_rows[wi], 128)))
        return rc;
      CUDA_TRY(h, afd::launch_router_tc(st, h->src_maps[wi], h->wrT, h->bias, h->wnorm, &h->tm_wr, d, ws,
                                        h->num_sms, s));
    }
  }
  if ((rc = prof_mark(h, 1, s))) return rc;
  {
    NvtxRange r("afd.routing");
    CUDA_TRY(h, afd::launch_routing(d, T, ws, s));
  }
  if ((rc = prof_mark(h, 2, s))) return rc;
  if (!direct) {  // the direct form's gate/up reads the sources itself
    NvtxRange r("afd.pack");
    CUDA_TRY(h, afd::launch_pack(st, d, T, ws, h->num_sms, s));
  }
  if ((rc = prof_mark(h, 3, s))) return rc;
  for (int which = 0; which < 2; ++which) {
    NvtxRange r(which ? "afd.gemm_down" : "afd.gemm_gateup");
    if (d.dtype == AFD_FP32)
      CUDA_TRY(h, afd::launch_gemm_simt(d, T, h->wg32, h->wu32, h->wd32, ws, s, which));
    else if (d.dtype == AFD_FP8_E4M3)
      CUDA_TRY(h, afd::launch_gemm_fp8(d, T, w, ws, h->num_sms, s, which));
    else
      CUDA_TRY(h, afd::launch_gemm_tc(d, T, w, ws, h->num_sms, s, which, which == 0 ? ds : nullptr));
    if ((rc = prof_mark(h, 4 + which, s))) return rc;
  }
  {
    NvtxRange r("afd.combine");
    CUDA_TRY(h, afd::launch_combine(st, d, T, ws, h->num_sms, s));
  }
  return prof_mark(h, 6, s);
}

int create_impl(const afd_ffn_config* cfg, const afd_ffn_weights* w, afd_ffn* h) {
  const afd_ffn_config& c = *cfg;
  h->cfg = c;
  h->dims = LayerDims{c.H, c.I, c.E, c.k, c.n_shared, (int)c.dtype};
  h->max_rows = (size_t)c.max_tokens * (c.k + c.n_shared);
  CUDA_TRY(h, cudaGetDevice(&h->device));
  CUDA_TRY(h, cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device));
  CUDA_TRY(h, afd::router_setup());
  if (c.dtype != AFD_FP32) {
    int major = 0, minor = 0;
    CUDA_TRY(h, cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, h->device));
    CUDA_TRY(h, cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, h->device));
    if (major != 10 || minor != 3)
      return fail(h, AFD_EUNSUPPORTED, "tensor-core path is built for sm_103a; device is sm_%d%d", major, minor);
    if (!get_encoder()) return fail(h, AFD_ECUDA, "cuTensorMapEncodeTiled entry point unavailable");
    CUDA_TRY(h, afd::gemm_tc_setup());
    CUDA_TRY(h, afd::gemm_fp8_setup());
    CUDA_TRY(h, afd::router_tc_setup());
  }

  const size_t H = c.H, I = c.I, E = c.E, S = c.n_shared, G = E + S;
  const size_t ab = act_bytes(c), wb = wt_bytes(c);
  int rc;
  cudaStream_t s = nullptr;

  // router: [H, E] -> [E, H]
  if ((rc = dmalloc(h, &h->wrT, E * H * ab))) return rc;
  CUDA_TRY(h, afd::launch_transpose(w->w_router, h->wrT, 1, (int)H, (int)E, (int)ab, s));
  if (c.dtype != AFD_FP32) {
    if ((rc = dmalloc_t(h, &h->wnorm, E))) return rc;
    CUDA_TRY(h, afd::launch_router_wnorm(h->wrT, (int)H, (int)E, h->wnorm, s));
    if (!make_map(&h->tm_wr, h->wrT, false, H, E, 128))
      return fail(h, AFD_ECUDA, "cuTensorMapEncodeTiled failed for the router weights");
  }
  if (w->router_bias) {
    if ((rc = dmalloc_t(h, &h->bias, E))) return rc;
    CUDA_TRY(h, cudaMemcpy(h->bias, w->router_bias, E * sizeof(float), cudaMemcpyDeviceToDevice));
  }

  if (c.dtype == AFD_FP32) {
    if ((rc = dmalloc_t(h, &h->wg32, G * H * I)) || (rc = dmalloc_t(h, &h->wu32, G * H * I)) ||
        (rc = dmalloc_t(h, &h->wd32, G * I * H)))
      return rc;
    CUDA_TRY(h, cudaMemcpy(h->wg32, w->w_gate, E * H * I * 4, cudaMemcpyDeviceToDevice));
    CUDA_TRY(h, cudaMemcpy(h->wu32, w->w_up, E * H * I * 4, cudaMemcpyDeviceToDevice));
    CUDA_TRY(h, cudaMemcpy(h->wd32, w->w_down, E * I * H * 4, cudaMemcpyDeviceToDevice));
    if (S) {
      CUDA_TRY(h, cudaMemcpy(h->wg32 + E * H * I, w->sh_gate, H * I * 4, cudaMemcpyDeviceToDevice));
      CUDA_TRY(h, cudaMemcpy(h->wu32 + E * H * I, w->sh_up, H * I * 4, cudaMemcpyDeviceToDevice));
      CUDA_TRY(h, cudaMemcpy(h->wd32 + E * I * H, w->sh_down, I * H * 4, cudaMemcpyDeviceToDevice));
    }
  } else {
    if ((rc = dmalloc(h, &h->wgT, G * I * H * wb)) || (rc = dmalloc(h, &h->wuT, G * I * H * wb)) ||
        (rc = dmalloc(h, &h->wdT, G * H * I * wb)))
      return rc;
    uint8_t* g8 = static_cast<uint8_t*>(h->wgT);
    uint8_t* u8 = static_cast<uint8_t*>(h->wuT);
    uint8_t* d8 = static_cast<uint8_t*>(h->wdT);
    CUDA_TRY(h, afd::launch_tile_weights(w->w_gate, g8, (int)E, (int)H, (int)I, (int)wb, s));
    CUDA_TRY(h, afd::launch_tile_weights(w->w_up, u8, (int)E, (int)H, (int)I, (int)wb, s));
    CUDA_TRY(h, afd::launch_tile_weights(w->w_down, d8, (int)E, (int)I, (int)H, (int)wb, s));
    if (S) {
      CUDA_TRY(h, afd::launch_tile_weights(w->sh_gate, g8 + E * I * H * wb, 1, (int)H, (int)I, (int)wb, s));
      CUDA_TRY(h, afd::launch_tile_weights(w->sh_up, u8 + E * I * H * wb, 1, (int)H, (int)I, (int)wb, s));
      CUDA_TRY(h, afd::launch_tile_weights(w->sh_down, d8 + E * H * I * wb, 1, (int)I, (int)H, (int)wb, s));
    }
    const bool fp8 = c.dtype == AFD_FP8_E4M3;
    if (fp8) {
      // block scales, m-block major: gate/up [(E+S)][I/128][H/128], down [(E+S)][H/128][I/128]
      const size_t hb = H / 128, ib = I / 128;
      if ((rc = dmalloc_t(h, &h->sgT, G * ib * hb)) || (rc = dmalloc_t(h, &h->suT, G * ib * hb)) ||
          (rc = dmalloc_t(h, &h->sdT, G * hb * ib)))
        return rc;
      CUDA_TRY(h, afd::launch_transpose_f32(w->s_gate, h->sgT, (int)E, (int)hb, (int)ib, s));
      CUDA_TRY(h, afd::launch_transpose_f32(w->s_up, h->suT, (int)E, (int)hb, (int)ib, s));
      CUDA_TRY(h, afd::launch_transpose_f32(w->s_down, h->sdT, (int)E, (int)ib, (int)hb, s));
      if (S) {
        CUDA_TRY(h, afd::launch_transpose_f32(w->sh_s_gate, h->sgT + E * ib * hb, 1, (int)hb, (int)ib, s));
        CUDA_TRY(h, afd::launch_transpose_f32(w->sh_s_up, h->suT + E * ib * hb, 1, (int)hb, (int)ib, s));
        CUDA_TRY(h, afd::launch_transpose_f32(w->sh_s_down, h->sdT + E * hb * ib, 1, (int)ib, (int)hb, s));
      }
    }
    // tiled weights: rows of 128 bytes (one K block of one output row), 128-row boxes
    const uint64_t kw = 128 / wb, tile_rows = G * H * I / kw;
    if (!make_map(&h->tm_wg, h->wgT, fp8, kw, tile_rows, 128) ||
        !make_map(&h->tm_wu, h->wuT, fp8, kw, tile_rows, 128) || !make_map(&h->tm_wd, h->wdT, fp8, kw, tile_rows, 128))
      return fail(h, AFD_ECUDA, "cuTensorMapEncodeTiled failed for a weight operand");
  }
  if ((rc = alloc_workspace(h, h->ws[0]))) return rc;
  CUDA_TRY(h, cudaDeviceSynchronize());
  CUDA_TRY(h, cudaGetLastError());
  return AFD_OK;
}

}  // namespace

extern "C" {

const char* afd_ffn_create_error(void) { return g_create_err.c_str(); }

int afd_ffn_create(const afd_ffn_config* cfg, const afd_ffn_weights* w, afd_ffn_t* out) {
  g_create_err.clear();
  if (!out) return fail(nullptr, AFD_EINVAL, "out is NULL");
  *out = nullptr;
  int rc = validate_config(cfg);
  if (rc) return rc;
  if (!w || !w->w_router || !w->w_gate || !w->w_up || !w->w_down)
    return fail(nullptr, AFD_EINVAL, "router and expert weight pointers must be non-NULL");
  if (cfg->dtype == AFD_FP8_E4M3 && (!w->s_gate || !w->s_up || !w->s_down))
    return fail(nullptr, AFD_EINVAL, "fp8 layer needs s_gate, s_up, s_down");
  if (cfg->n_shared) {
    if (!w->sh_gate || !w->sh_up || !w->sh_down)
      return fail(nullptr, AFD_EINVAL, "n_shared=1 needs sh_gate, sh_up, sh_down");
    if (cfg->dtype == AFD_FP8_E4M3 && (!w->sh_s_gate || !w->sh_s_up || !w->sh_s_down))
      return fail(nullptr, AFD_EINVAL, "fp8 shared expert needs sh_s_gate, sh_s_up, sh_s_down");
  }
  afd_ffn* h = new afd_ffn();
  rc = create_impl(cfg, w, h);
  if (rc) {
    g_create_err = h->err;
    afd_ffn_destroy(h);
    return rc;
  }
  *out = h;
  return AFD_OK;
}

int afd_ffn_forward(afd_ffn_t h, void* stream, const void* const* src_ptrs_dev, const int* src_counts_host, int M,
                    void* const* out_ptrs_dev) {
  int T = 0;
  int rc = validate_batch(h, src_ptrs_dev, src_counts_host, M, out_ptrs_dev, &T);
  if (rc) return rc;
  SrcTable st = make_table(src_ptrs_dev, src_counts_host, M, out_ptrs_dev);
  h->route_ws = 0;
  return run_layer(h, st, h->ws[0], static_cast<cudaStream_t>(stream));
}

int afd_ffn_forward_pipelined(afd_ffn_t h, void* stream, int n_micro, const void* const* src_ptrs_dev,
                              const int* src_counts_host, int M, void* const* out_ptrs_dev) {
  int T = 0;
  int rc = validate_batch(h, src_ptrs_dev, src_counts_host, M, out_ptrs_dev, &T);
  if (rc) return rc;
  if (n_micro < 1 || n_micro > AFD_MAX_MICRO)
    return fail(h, AFD_EINVAL, "n_micro=%d outside [1, %d]", n_micro, AFD_MAX_MICRO);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  h->route_ws = 0;
  if (!h->ev_fork) CUDA_TRY(h, cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming));
  for (int i = 0; i < n_micro; ++i) {
    if (!h->mstream[i]) CUDA_TRY(h, cudaStreamCreateWithFlags(&h->mstream[i], cudaStreamNonBlocking));
    if (!h->ev_join[i]) CUDA_TRY(h, cudaEventCreateWithFlags(&h->ev_join[i], cudaEventDisableTiming));
    if ((rc = alloc_workspace(h, h->ws[i]))) return rc;
  }
  CUDA_TRY(h, cudaEventRecord(h->ev_fork, s));
  // contiguous token ranges: the first T % n get one extra token
  const int q = T / n_micro, rem = T % n_micro;
  int t0 = 0;
  for (int i = 0; i < n_micro; ++i) {
    const int len = q + (i < rem ? 1 : 0);
    const int t1 = t0 + len;
    const void* sub_src[AFD_MAX_SOURCES];
    void* sub_out[AFD_MAX_SOURCES];
    int sub_cnt[AFD_MAX_SOURCES];
    int sm = 0, row0 = 0;
    for (int m = 0; m < M; ++m) {
      const int a = row0 > t0 ? row0 : t0;
      const int b = row0 + src_counts_host[m] < t1 ? row0 + src_counts_host[m] : t1;
      if (b > a) {
        const size_t off = (size_t)(a - row0) * h->cfg.H * act_bytes(h->cfg);
        sub_src[sm] = static_cast<const uint8_t*>(src_ptrs_dev[m]) + off;
        sub_out[sm] = static_cast<uint8_t*>(out_ptrs_dev[m]) + off;
        sub_cnt[sm] = b - a;
        ++sm;
      }
      row0 += src_counts_host[m];
    }
    SrcTable st = make_table(sub_src, sub_cnt, sm, sub_out);
    CUDA_TRY(h, cudaStreamWaitEvent(h->mstream[i], h->ev_fork, 0));
    if ((rc = run_layer(h, st, h->ws[i], h->mstream[i]))) return rc;
    CUDA_TRY(h, cudaEventRecord(h->ev_join[i], h->mstream[i]));
    CUDA_TRY(h, cudaStreamWaitEvent(s, h->ev_join[i], 0));
    t0 = t1;
  }
  return AFD_OK;
}

int afd_ffn_forward_host(afd_ffn_t h, void* stream, int n_micro, const void* const* src_ptrs_host,
                         const int* src_counts_host, int M, void* const* out_ptrs_host) {
  int T = 0;
  int rc = validate_batch(h, src_ptrs_host, src_counts_host, M, out_ptrs_host, &T);
  if (rc) return rc;
  if (n_micro < 1 || n_micro > AFD_MAX_MICRO)
    return fail(h, AFD_EINVAL, "n_micro=%d outside [1, %d]", n_micro, AFD_MAX_MICRO);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Workspace& ws = h->ws[0];
  const size_t rowb = (size_t)h->cfg.H * act_bytes(h->cfg);
  if (!ws.stage && (rc = dmalloc(h, &ws.stage, 2 * (size_t)h->cfg.max_tokens * rowb))) return rc;
  uint8_t* in = static_cast<uint8_t*>(ws.stage);
  uint8_t* outb = in + (size_t)h->cfg.max_tokens * rowb;
  const void* dsrc[AFD_MAX_SOURCES];
  void* dout[AFD_MAX_SOURCES];
  size_t r = 0;
  for (int m = 0; m < M; ++m) {
    dsrc[m] = in + r * rowb;
    dout[m] = outb + r * rowb;
    if (src_counts_host[m] > 0)
      CUDA_TRY(h, cudaMemcpyAsync(in + r * rowb, src_ptrs_host[m], src_counts_host[m] * rowb,
                                  cudaMemcpyHostToDevice, s));
    r += src_counts_host[m];
  }
  if (n_micro > 1) {
    if ((rc = afd_ffn_forward_pipelined(h, stream, n_micro, dsrc, src_counts_host, M, dout))) return rc;
  } else {
    SrcTable st = make_table(dsrc, src_counts_host, M, dout);
    h->route_ws = 0;
    if ((rc = run_layer(h, st, ws, s))) return rc;
  }
  r = 0;
  for (int m = 0; m < M; ++m) {
    if (src_counts_host[m] > 0)
      CUDA_TRY(h, cudaMemcpyAsync(out_ptrs_host[m], outb + r * rowb, src_counts_host[m] * rowb,
                                  cudaMemcpyDeviceToHost, s));
    r += src_counts_host[m];
  }
  CUDA_TRY(h, cudaStreamSynchronize(s));
  return AFD_OK;
}

int afd_ffn_forward_host_async(afd_ffn_t h, int n_micro, const void* const* src_ptrs_host,
                               const int* src_counts_host, int M, void* const* out_ptrs_host) {
  int T = 0;
  int rc = validate_batch(h, src_ptrs_host, src_counts_host, M, out_ptrs_host, &T);
  if (rc) return rc;
  if (n_micro < 1 || n_micro > AFD_MAX_MICRO)
    return fail(h, AFD_EINVAL, "n_micro=%d outside [1, %d]", n_micro, AFD_MAX_MICRO);
  const size_t rowb = (size_t)h->cfg.H * act_bytes(h->cfg);
  const size_t slot_bytes = 2 * (size_t)h->cfg.max_tokens * rowb;
  for (int i = 0; i < 4; ++i)
    if (!h->astream[i]) CUDA_TRY(h, cudaStreamCreateWithFlags(&h->astream[i], cudaStreamNonBlocking));
  for (int q = 0; q < 2; ++q) {
    if (!h->astage[q] && (rc = dmalloc(h, &h->astage[q], slot_bytes))) return rc;
    for (cudaEvent_t* e : {&h->ev_in[q], &h->ev_done[q], &h->ev_out[q]})
      if (!*e) CUDA_TRY(h, cudaEventCreateWithFlags(e, cudaEventDisableTiming));
  }
  const int q = (int)(h->async_calls & 1u);
  // Single-pass calls alternate between two compute streams and workspaces, so one
  // batch's router and pack can run while the previous batch's last kernels finish.
  // A micro-batched call uses workspaces 0..n_micro-1 and follows the other slot's call.
  cudaStream_t cin = h->astream[0], comp = h->astream[q ? 3 : 1], cout = h->astream[2];
  Workspace& wsq = h->ws[q];
  if (n_micro == 1 && (rc = alloc_workspace(h, wsq))) return rc;
  ++h->async_calls;
  uint8_t* in = static_cast<uint8_t*>(h->astage[q]);
  uint8_t* outb = in + (size_t)h->cfg.max_tokens * rowb;
  const void* dsrc[AFD_MAX_SOURCES];
  void* dout[AFD_MAX_SOURCES];
  // copy-in: the slot's sources are free once the layer two calls back has finished
  CUDA_TRY(h, cudaStreamWaitEvent(cin, h->ev_done[q], 0));
  size_t r = 0;
  for (int m = 0; m < M; ++m) {
    dsrc[m] = in + r * rowb;
    dout[m] = outb + r * rowb;
    if (src_counts_host[m] > 0)
      CUDA_TRY(h, cudaMemcpyAsync(in + r * rowb, src_ptrs_host[m], src_counts_host[m] * rowb,
                                  cudaMemcpyHostToDevice, cin));
    r += src_counts_host[m];
  }
  CUDA_TRY(h, cudaEventRecord(h->ev_in[q], cin));
  // compute: after this call's copy-in and after the slot's outputs two calls back went out
  CUDA_TRY(h, cudaStreamWaitEvent(comp, h->ev_in[q], 0));
  CUDA_TRY(h, cudaStreamWaitEvent(comp, h->ev_out[q], 0));
  if (n_micro > 1 || h->async_last_micro > 1)  // workspaces shared with the other slot's call
    CUDA_TRY(h, cudaStreamWaitEvent(comp, h->ev_done[q ^ 1], 0));
  h->async_last_micro = n_micro;
  if (n_micro > 1) {
    rc = afd_ffn_forward_pipelined(h, comp, n_micro, dsrc, src_counts_host, M, dout);
  } else {
    SrcTable st = make_table(dsrc, src_counts_host, M, dout);
    rc = run_layer(h, st, wsq, comp);
    h->route_ws = q;
  }
  if (rc) {
    if (!h->async_rc) h->async_rc = rc;
    // part of the layer may have been enqueued: mark the slot busy until it has run, so
    // the next call on this slot does not overwrite sources those kernels still read
    cudaEventRecord(h->ev_done[q], comp);
    cudaEventRecord(h->ev_out[q], comp);
    return rc;
  }
  CUDA_TRY(h, cudaEventRecord(h->ev_done[q], comp));
  // copy-out
  CUDA_TRY(h, cudaStreamWaitEvent(cout, h->ev_done[q], 0));
  r = 0;
  for (int m = 0; m < M; ++m) {
    if (src_counts_host[m] > 0)
      CUDA_TRY(h, cudaMemcpyAsync(out_ptrs_host[m], outb + r * rowb, src_counts_host[m] * rowb,
                                  cudaMemcpyDeviceToHost, cout));
    r += src_counts_host[m];
  }
  CUDA_TRY(h, cudaEventRecord(h->ev_out[q], cout));
  return AFD_OK;
}

int afd_ffn_host_wait(afd_ffn_t h) {
  if (!h) return AFD_EINVAL;
  for (cudaStream_t s : h->astream)
    if (s) CUDA_TRY(h, cudaStreamSynchronize(s));
  const int rc = h->async_rc;
  h->async_rc = 0;
  return rc;
}

int afd_ffn_debug_routing(afd_ffn_t h, void* stream, int* topk_idx, float* topk_w, int* counts, int* offsets,
                          int* perm_token, int* pos, float* logits) {
  if (!h) return AFD_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Workspace& ws = h->ws[h->route_ws];
  const size_t T = ws.last_T, k = h->cfg.k, E = h->cfg.E;
  auto cp = [&](void* dst, const void* src, size_t n) -> cudaError_t {
    if (!dst || n == 0) return cudaSuccess;
    return cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToDevice, s);
  };
  CUDA_TRY(h, cp(topk_idx, ws.topk_idx, T * k * 4));
  CUDA_TRY(h, cp(topk_w, ws.topk_w, T * k * 4));
  CUDA_TRY(h, cp(logits, ws.logits, T * E * 4));
  if (T == 0) {
    if (counts) CUDA_TRY(h, cudaMemsetAsync(counts, 0, E * 4, s));
    if (offsets) CUDA_TRY(h, cudaMemsetAsync(offsets, 0, (E + 1) * 4, s));
    return AFD_OK;
  }
  CUDA_TRY(h, cp(counts, ws.counts, E * 4));
  CUDA_TRY(h, cp(offsets, ws.offsets, (E + 1) * 4));
  CUDA_TRY(h, cp(perm_token, ws.perm, T * k * 4));
  CUDA_TRY(h, cp(pos, ws.pos, T * k * 4));
  return AFD_OK;
}

int afd_ffn_debug_operands(afd_ffn_t h, void* stream, void* P, float* P_scale, void* Hmid, float* H_scale) {
  if (!h) return AFD_EINVAL;
  const bool fp8 = h->cfg.dtype == AFD_FP8_E4M3;
  if (!fp8 && (P_scale || H_scale)) return fail(h, AFD_EINVAL, "operand scales exist only for the fp8 layer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Workspace& ws = h->ws[h->route_ws];
  if (!ws.ready) return fail(h, AFD_EINVAL, "no forward has run on this handle");
  const size_t R = (size_t)ws.last_T * (h->cfg.k + h->cfg.n_shared);
  if (R == 0) return AFD_OK;
  const size_t H = h->cfg.H, I = h->cfg.I, eb = fp8 ? 1 : act_bytes(h->cfg);
  if (P && ws.direct)
    return fail(h, AFD_EINVAL, "P is not written for bf16 batches of at most %d tokens", afd::kDirectMaxTok);
  if (P) CUDA_TRY(h, cudaMemcpyAsync(P, ws.P, R * H * eb, cudaMemcpyDeviceToDevice, s));
  if (Hmid) CUDA_TRY(h, cudaMemcpyAsync(Hmid, ws.Hb, R * I * eb, cudaMemcpyDeviceToDevice, s));
  // scales are stored K-block major with row stride scale_ld: copy the first R of each block
  const size_t ld = (size_t)ws.scale_ld * sizeof(float), w = R * sizeof(float);
  if (P_scale)
    CUDA_TRY(h, cudaMemcpy2DAsync(P_scale, w, ws.P_scale, ld, w, H / 128, cudaMemcpyDeviceToDevice, s));
  if (H_scale)
    CUDA_TRY(h, cudaMemcpy2DAsync(H_scale, w, ws.H_scale, ld, w, I / 128, cudaMemcpyDeviceToDevice, s));
  return AFD_OK;
}

int afd_ffn_debug_inject(afd_ffn_t h, void* stream, int kind, long long arg) {
  if (!h) return AFD_EINVAL;
  if (kind != AFD_INJECT_TIMEOUT && kind != AFD_INJECT_RANGE)
    return fail(h, AFD_EINVAL, "unknown injection kind %d", kind);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Workspace& ws = h->ws[0];
  int rc = alloc_workspace(h, ws);
  if (rc) return rc;
  if (kind == AFD_INJECT_TIMEOUT) {
    const long long limit = arg < 1000 ? 1000 : (arg > 4000000000ll ? 4000000000ll : arg);
    afd::wait_probe_kernel<<<1, 32, 0, s>>>(ws.err, limit);
    CUDA_TRY(h, cudaGetLastError());
    return AFD_OK;
  }
  // one token whose first expert id is E; the others valid
  std::vector<int32_t> idx(h->cfg.k);
  for (int j = 0; j < h->cfg.k; ++j) idx[j] = j == 0 ? h->cfg.E : j - 1;
  CUDA_TRY(h, cudaMemcpyAsync(ws.topk_idx, idx.data(), idx.size() * sizeof(int32_t), cudaMemcpyHostToDevice, s));
  CUDA_TRY(h, cudaStreamSynchronize(s));  // idx is a host temporary
  CUDA_TRY(h, afd::launch_routing(h->dims, 1, ws, s));
  return AFD_OK;
}

int afd_ffn_check(afd_ffn_t h, void* stream) {
  if (!h) return AFD_EINVAL;
  CUDA_TRY(h, cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  int word = 0;
  for (auto& ws : h->ws) {
    if (!ws.ready) continue;
    for (auto ms : h->mstream)
      if (ms) CUDA_TRY(h, cudaStreamSynchronize(ms));
    int v = 0;
    CUDA_TRY(h, cudaMemcpy(&v, ws.err, sizeof(int), cudaMemcpyDeviceToHost));
    CUDA_TRY(h, cudaMemset(ws.err, 0, sizeof(int)));
    word |= v;
  }
  if (word)
    return fail(h, AFD_EDEVICE, "device error word 0x%x:%s%s", word,
                (word & afd::kErrTimeout) ? " a bounded wait timed out;" : "",
                (word & afd::kErrRange) ? " a routing value was out of range;" : "");
  return AFD_OK;
}

int afd_ffn_profile_begin(afd_ffn_t h) {
  if (!h) return AFD_EINVAL;
  h->prof_on = true;
  h->prof_used = 0;
  return AFD_OK;
}

int afd_ffn_profile_end(afd_ffn_t h, double* ms_per_kernel, int* n_forwards) {
  if (!h || !ms_per_kernel) return AFD_EINVAL;
  CUDA_TRY(h, cudaDeviceSynchronize());
  for (int q = 0; q < AFD_NUM_KERNELS; ++q) ms_per_kernel[q] = 0.0;
  const size_t nf = h->prof_used / (AFD_NUM_KERNELS + 1);
  for (size_t f = 0; f < nf; ++f)
    for (int q = 0; q < AFD_NUM_KERNELS; ++q) {
      float ms = 0.f;
      CUDA_TRY(h, cudaEventElapsedTime(&ms, h->prof_events[f * (AFD_NUM_KERNELS + 1) + q],
                                       h->prof_events[f * (AFD_NUM_KERNELS + 1) + q + 1]));
      ms_per_kernel[q] += ms;
    }
  if (n_forwards) *n_forwards = (int)nf;
  h->prof_on = false;
  h->prof_used = 0;
  return AFD_OK;
}

// router (one kernel for fp32 and small bf16/fp8 batches; tensor-core logits and
// select otherwise), the routing tables (one launch up to 2048 tokens, two above),
// pack (none for bf16 batches of at most kDirectMaxTok = 8 tokens), two GEMMs, combine
int afd_ffn_launches_per_forward(afd_ffn_t h, int T) {
  if (!h || T < 1) return AFD_EINVAL;
  const afd::LayerDims& d = h->dims;
  const int router = d.dtype == AFD_FP32 ? 1 : afd::router_tc_launches(d, T, h->num_sms);
  const int pack = direct_form(d, T) ? 0 : 1;
  return router + afd::routing_launches(T) + pack + 2 /* GEMMs */ + 1 /* combine */;
}

const char* afd_ffn_last_error(afd_ffn_t h) { return h ? h->err.c_str() : "handle is NULL"; }

size_t afd_ffn_device_bytes(afd_ffn_t h) { return h ? h->bytes : 0; }

void afd_ffn_destroy(afd_ffn_t h) {
  if (!h) return;
  cudaDeviceSynchronize();
  for (auto& ws : h->ws) free_workspace(ws);
  void* ptrs[] = {h->wrT, h->bias, h->wnorm, h->wgT, h->wuT, h->wdT, h->sgT, h->suT, h->sdT, h->wg32, h->wu32, h->wd32};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  for (auto s : h->mstream)
    if (s) cudaStreamDestroy(s);
  for (auto s : h->astream)
    if (s) cudaStreamDestroy(s);
  for (int q = 0; q < 2; ++q) {
    if (h->astage[q]) cudaFree(h->astage[q]);
    for (cudaEvent_t e : {h->ev_in[q], h->ev_done[q], h->ev_out[q]})
      if (e) cudaEventDestroy(e);
  }
  for (auto e : h->ev_join)
    if (e) cudaEventDestroy(e);
  if (h->ev_fork) cudaEventDestroy(h->ev_fork);
  for (auto e : h->prof_events) cudaEventDestroy(e);
  delete h;
}

}  // extern "C"
