// api.cu -- the extern "C" entry points of libmtgr.so (declared in mtgr.h):
// argument checks, workspace carving, tensor-map encoding and kernel dispatch.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "gemm.cuh"
#include "plan.cuh"

namespace mtgr {

// ---- launchers defined in the other translation units ----
// n_norm: per-user n_u of the 1/n_u factor, q_begin: per-user first query row
// the forward computes (device arrays; NULL = the segment length / 0)
cudaError_t launch_user_info(const int32_t*, int32_t, const uint8_t*, int64_t, UserInfo*, int32_t*, cudaStream_t,
                             const int32_t* n_norm = nullptr, const int32_t* q_begin = nullptr);
cudaError_t launch_plan(const int32_t*, int32_t, const uint8_t*, int64_t, int32_t, int32_t*, int32_t*, cudaStream_t,
                        const int32_t* n_norm = nullptr, const int32_t* q_begin = nullptr, int64_t ds_cap = 0);
cudaError_t launch_visible_counts(const int32_t*, int32_t, const uint8_t*, const int64_t*, int64_t, int32_t*,
                                  int64_t*, cudaStream_t);
cudaError_t launch_expand_rows(const void*, const int32_t*, int64_t, void*, int64_t, int64_t, cudaStream_t);
cudaError_t launch_wait_timeout(int32_t*, cudaStream_t);
template <typename T, typename TY>
cudaError_t launch_gln_fwd(const T*, TY*, float*, float*, const uint8_t*, const float*, const float*, int64_t, int,
                           float, cudaStream_t);
template <typename TD, typename T>
cudaError_t launch_gln_bwd(const TD*, const T*, const float*, const float*, const uint8_t*, const float*, const T*,
                           T*, float*, float*, float*, int64_t, int, const float*, cudaStream_t);
cudaError_t launch_grad_to_f16(const __nv_bfloat16*, __half*, int64_t, unsigned*, float*, cudaStream_t);
int gln_bwd_blocks(int64_t rows);
template <typename TOi, typename TU, typename TY>
cudaError_t launch_ln_gate_fwd(const TOi*, const TU*, int64_t, TY*, float*, float*, int64_t, int, float,
                               cudaStream_t);
template <typename TD, typename TG, typename TOi, typename TU, typename TO>
cudaError_t launch_ln_gate_bwd(const TD*, const TOi*, const TU*, int64_t, const float*, const float*, TO*, TG*,
                               int64_t, const TG*, int64_t, int, cudaStream_t);
cudaError_t launch_bf16_to_f16(const __nv_bfloat16*, int64_t, __half*, int64_t, int64_t, int, cudaStream_t);
cudaError_t launch_attn_f32_fwd(const float*, const float*, const float*, int64_t, const UserInfo*, int,
                                const int64_t*, int64_t, int, int, float*, cudaStream_t);
cudaError_t launch_attn_f32_bwd(const float*, const float*, const float*, int64_t, const float*, const UserInfo*,
                                int, const int64_t*, int64_t, int, int, float*, float*, float*, int64_t,
                                const float*, const float*, const float*, cudaStream_t);
cudaError_t launch_attn_fwd_f16(const __half*, const __half*, const __half*, int64_t, int64_t, int, int,
                                const int32_t*, int32_t, const int64_t*, __half*, int32_t*, cudaStream_t, float*);
template <typename TU, typename TY>
cudaError_t launch_ln_gate_fwd_parts(const float*, int64_t, __half*, const TU*, int64_t, TY*, float*, float*, int64_t,
                                     int, float, cudaStream_t);
cudaError_t launch_attn_bwd_f16(const __half* q, const __half* k, const __half* v, int64_t ld, const __half* dO,
                                int64_t T, int H, int d, const int32_t* plan, int32_t B, const int64_t* ts, void* dq,
                                void* dk, void* dv, int64_t ldg, const void* mq, const void* mk, const void* mv,
                                bool g_f16, int32_t* status, cudaStream_t s, uint8_t* ds_store, int64_t ds_cap);

// ---- kernel tracing ----
namespace {
struct TraceRec {
  const char* name;
  cudaEvent_t a, b;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
std::vector<TraceRec> g_trace;
std::vector<cudaEvent_t> g_pool;
size_t g_pool_used = 0;
int g_open = -1;

cudaEvent_t pool_event() {
  if (g_pool_used == g_pool.size()) {
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    g_pool.push_back(e);
  }
  return g_pool[g_pool_used++];
}
}  // namespace

void trace_begin(const char* name, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (!g_trace_on || g_open >= 0) return;
  cudaEvent_t a = pool_event(), b = pool_event();
  if (!a || !b) return;
  cudaEventRecord(a, s);
  g_trace.push_back({name, a, b});
  g_open = (int)g_trace.size() - 1;
}

void trace_end(cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (g_open < 0) return;
  cudaEventRecord(g_trace[g_open].b, s);
  g_open = -1;
}

// ---- error state ----
static thread_local char g_err[512] = "";

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

mtgr_status cuda_status(cudaError_t e, const char* where) {
  set_error("%s: %s", where, cudaGetErrorString(e));
  return MTGR_ERR_CUDA;
}

// SM count of the current device, cached per device (host threads may race to
// fill an entry; they all store the same value)
int num_sms() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, looked up once (the initialisation
// of a function-local static is thread-safe)
static EncodeTiledFn encode_fn() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(ptr);
    return nullptr;
  }();
  return fn;
}

static bool make_tmap_16bit_2d(CUtensorMapDataType dt, CUtensorMap* m, const void* base, uint64_t rows,
                               uint64_t cols, uint64_t ld, uint32_t box_cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows == 0 || cols == 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
bool make_tmap_bf16_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                       uint32_t box_cols, uint32_t box_rows) {
  return make_tmap_16bit_2d(CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, m, base, rows, cols, ld, box_cols, box_rows);
}
bool make_tmap_f16_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                      uint32_t box_cols, uint32_t box_rows) {
  return make_tmap_16bit_2d(CU_TENSOR_MAP_DATA_TYPE_FLOAT16, m, base, rows, cols, ld, box_cols, box_rows);
}
bool make_tmap_out(CUtensorMap* m, OutType t, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                   uint64_t slices, uint32_t box_cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows == 0 || cols == 0) return false;
  const CUtensorMapDataType dt = t == OUT_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : t == OUT_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t es = t == OUT_F32 ? 4 : 2;
  const uint64_t inner = box_cols * es;
  if (inner != 64 && inner != 128) return false;
  const CUtensorMapSwizzle sw = inner == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  cuuint64_t dims[3] = {cols, rows, slices > 0 ? slices : 1};
  cuuint64_t strides[2] = {ld * es, rows * ld * es};
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, dt, slices > 0 ? 3 : 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// Workspace carving
// ---------------------------------------------------------------------------
static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
static size_t esize(mtgr_dtype dt) { return dt == MTGR_F32 ? 4 : 2; }

// Attention workspace: status word, jagged tile plan, dO; in the bf16 path the
// tensor-core operands are f16: q, k, v are converted once (exactly) into f16
// copies, and dO, P, dS are produced in f16 (11 significand bits instead of 8).
struct AttnWs {
  size_t status, plan, dO, qkv16, opart, total;
  bool key_split;
};
// Key split of the forward: when even twice the per-query-tile items of the
// batch (at most (T/128 + B)·H) fit in one wave, each item's key tiles are
// shared by two CTAs (a ranking request of one user: 72 items for 148 SMs).
static bool attn_key_split(int32_t B, int64_t T, int32_t H) {
  return 2 * ((T / 128 + B) * (int64_t)H) <= num_sms();
}
static AttnWs attn_ws(int32_t B, int64_t T, int32_t H, int32_t d, mtgr_dtype dt, bool convert_qkv = true) {
  AttnWs w;
  const size_t THD = (size_t)T * H * d;
  size_t o = 0;
  w.status = o;
  o += 256;
  w.plan = o;
  o += align256(sizeof(int32_t) * (size_t)plan_layout(B, T, H).total);
  w.dO = o;
  o += align256(THD * esize(dt));
  w.qkv16 = o;
  if (dt == MTGR_BF16 && convert_qkv) o += 3 * align256(THD * 2);
  w.key_split = dt != MTGR_F32 && T > 0 && attn_key_split(B, T, H);
  w.opart = o;
  if (w.key_split) o += align256(2 * THD * sizeof(float));  // two [T, H*d] fp32 halves, T*H*d apart
  w.total = o;
  return w;
}

// Layer workspace.  In the MTGR_BF16 path the layer keeps its activations and
// gradients in f16 between steps (11 significand bits): w16 holds f16 copies
// of W_uqkv and W_o, dxo16 the upstream gradient scaled by a power of two
// (gscale: its max-magnitude word, then the scale s and 1/s).
struct LayerWs {
  AttnWs attn;
  size_t attn_base, dY, dZ, dxn, gln_part, wpart, w16, dxo16, gscale, total;
  int splits_uqkv, splits_o;
  int splits_out;  // forward output projection: split over K when its tiles leave most SMs idle
};
// Split-K count for a weight-gradient GEMM (M x N output, K = tokens): the
// persistent kernel runs tiles x splits work units over the SMs, and each
// slice costs one fp32 M x N partial in the reduction, so take the fewest
// splits (at most 16) whose waves are within 2% as full as the fullest.
static int choose_splits(int64_t M, int64_t N, int64_t K) {
  const int64_t tiles = ((M + 127) / 128) * ((N + 255) / 256);
  const int64_t sms = num_sms();
  auto fill = [&](int s) {
    const int64_t units = tiles * s;
    return (double)units / (double)(((units + sms - 1) / sms) * sms);
  };
  double best = 0.0;
  for (int req = 1; req <= 16; ++req) best = fmax(best, fill(gemm_splits(K, req)));
  for (int req = 1; req <= 16; ++req) {
    const int s = gemm_splits(K, req);  // the count the GEMM actually runs
    if (fill(s) >= best - 0.02) return s;
  }
  return 1;
}
static LayerWs layer_ws(int32_t B, int64_t T, int32_t D, int32_t H, int32_t d, mtgr_dtype dt) {
  LayerWs w;
  const int64_t HD = (int64_t)H * d;
  w.attn = attn_ws(B, T, H, d, dt, /*convert_qkv=*/false);
  size_t o = 0;
  w.attn_base = o;
  o += w.attn.total;
  w.dY = o;
  o += align256((size_t)T * HD * esize(dt));
  w.dZ = o;
  o += align256((size_t)T * 4 * HD * esize(dt));
  w.dxn = o;
  o += align256((size_t)T * D * esize(dt));
  w.gln_part = o;
  o += align256((size_t)gln_bwd_blocks(T) * 8 * D * sizeof(float));
  w.splits_uqkv = dt == MTGR_BF16 ? choose_splits(D, 4 * HD, T) : 1;  // weight gradients: bf16 path only
  w.splits_o = dt == MTGR_BF16 ? choose_splits(HD, D, T) : 1;
  // x' = x + y·W_o has ceil(T/128)·ceil(D/256) output tiles: a short batch
  // (one ranking request) leaves most SMs without one, so it runs split over
  // K = H·d_h into fp32 slices that one pass adds to the residual.  Every
  // slice costs T·D fp32 written and read again, so take as many as fit in one
  // wave, at most 4.
  const int64_t out_tiles = ((T + 127) / 128) * ((D + 255) / 256);
  const int64_t fit = out_tiles > 0 ? num_sms() / out_tiles : 1;
  w.splits_out = (dt != MTGR_F32 && T > 0 && fit >= 2) ? gemm_splits(HD, (int)(fit < 4 ? fit : 4)) : 1;
  const size_t p1 = (size_t)w.splits_uqkv * D * 4 * HD, p2 = (size_t)w.splits_o * HD * D;
  const size_t p3 = w.splits_out > 1 ? (size_t)w.splits_out * T * D : 0;
  const size_t pm = p1 > p2 ? (p1 > p3 ? p1 : p3) : (p2 > p3 ? p2 : p3);
  w.wpart = o;
  o += align256(pm * sizeof(float));
  w.w16 = o;
  if (dt == MTGR_BF16) o += align256((size_t)D * 4 * HD * 2) + align256((size_t)HD * D * 2);
  w.dxo16 = o;
  if (dt == MTGR_BF16) o += align256((size_t)T * D * 2);
  w.gscale = o;
  o += 256;
  w.total = o;
  return w;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define REQUIRE(cond, code, ...)   \
  do {                             \
    if (!(cond)) {                 \
      set_error(__VA_ARGS__);      \
      return code;                 \
    }                              \
  } while (0)

static mtgr_status check_meta(const int32_t* offsets, int32_t B, const uint8_t* gid, int64_t T) {
  REQUIRE(B >= 0 && T >= 0, MTGR_ERR_INVALID_ARG, "B and T must be non-negative");
  REQUIRE(T < (int64_t(1) << 31) - 256, MTGR_ERR_UNSUPPORTED, "T must be below 2^31");
  REQUIRE(offsets != nullptr, MTGR_ERR_INVALID_ARG, "offsets is NULL");
  REQUIRE(T == 0 || gid != nullptr, MTGR_ERR_INVALID_ARG, "gid is NULL");
  return MTGR_OK;
}

// The backward's dS tile store: the bytes of the caller's workspace beyond
// the `used` bytes the call needs, from the next 1024-byte boundary, as whole
// dS tiles (plan.cuh); no slots when nothing is left over.
struct DsStore {
  uint8_t* base = nullptr;
  int64_t slots = 0;
};
static DsStore ds_store_region(uint8_t* ws, size_t ws_bytes, size_t used) {
  DsStore r;
  const uintptr_t a = reinterpret_cast<uintptr_t>(ws), end = a + ws_bytes;
  const uintptr_t start = (a + used + 1023) & ~uintptr_t(1023);
  if (ws_bytes > used && end > start && (end - start) >= (uintptr_t)kDsTileBytes) {
    r.base = reinterpret_cast<uint8_t*>(start);
    r.slots = (int64_t)((end - start) / kDsTileBytes);
  }
  return r;
}

// ---------------------------------------------------------------------------
// bf16-path attention on f16 tensor-core operands (shared by the attention
// entry points and the layer).  u is bf16 or f16 (u_f16); y, dq/dk/dv/du bf16.
// ---------------------------------------------------------------------------
static mtgr_status attn_fwd_bf16_core(const __half* q16, const __half* k16, const __half* v16, int64_t ld16,
                                      const void* u, bool u_f16, int64_t ldu, const int32_t* offsets, int32_t B,
                                      const uint8_t* gid, const int64_t* ts, int64_t T, int H, int d, float eps,
                                      void* y, __half* o, float* mean, float* rstd, uint8_t* ws,
                                      const AttnWs& w, cudaStream_t s, bool plan_ready = false,
                                      bool y_f16 = false, const int32_t* n_norm = nullptr,
                                      const int32_t* q_begin = nullptr, bool do_gate = true) {
  // plan_ready: an earlier call on the same batch left its status word and work
  // lists in this workspace (the layers of a stack share them)
  int32_t* status = reinterpret_cast<int32_t*>(ws + w.status);
  int32_t* plan = reinterpret_cast<int32_t*>(ws + w.plan);
  if (!plan_ready) MTGR_CUDA_TRY(cudaMemsetAsync(status, 0, sizeof(int32_t), s), "attn_fwd status");
  if (T == 0 || B == 0) return MTGR_OK;
  if (!plan_ready)
    MTGR_CUDA_TRY(launch_plan(offsets, B, gid, T, H, plan, status, s, n_norm, q_begin), "attn_fwd plan");
  // the key split needs the gate (which adds the halves) and every query row
  const bool split = w.key_split && do_gate && q_begin == nullptr;
  float* opart = split ? reinterpret_cast<float*>(ws + w.opart) : nullptr;
  MTGR_CUDA_TRY(launch_attn_fwd_f16(q16, k16, v16, ld16, T, H, d, plan, B, ts, o, status, s, opart),
                "attn_fwd tcgen05");
  if (!do_gate) return MTGR_OK;
  const int HD = H * d;
  const int64_t ps = T * HD;  // the halves' distance (the forward kernel's pstride)
  cudaError_t e =
      split ? (y_f16   ? launch_ln_gate_fwd_parts(opart, ps, o, static_cast<const __half*>(u), ldu,
                                                  static_cast<__half*>(y), mean, rstd, T, HD, eps, s)
               : u_f16 ? launch_ln_gate_fwd_parts(opart, ps, o, static_cast<const __half*>(u), ldu,
                                                  static_cast<__nv_bfloat16*>(y), mean, rstd, T, HD, eps, s)
                       : launch_ln_gate_fwd_parts(opart, ps, o, static_cast<const __nv_bfloat16*>(u), ldu,
                                                  static_cast<__nv_bfloat16*>(y), mean, rstd, T, HD, eps, s))
      :
      y_f16   ? launch_ln_gate_fwd(o, static_cast<const __half*>(u), ldu, static_cast<__half*>(y), mean, rstd, T, HD,
                                   eps, s)
      : u_f16 ? launch_ln_gate_fwd(o, static_cast<const __half*>(u), ldu, static_cast<__nv_bfloat16*>(y), mean, rstd,
                                   T, HD, eps, s)
              : launch_ln_gate_fwd(o, static_cast<const __nv_bfloat16*>(u), ldu, static_cast<__nv_bfloat16*>(y), mean,
                                   rstd, T, HD, eps, s);
  if (e != cudaSuccess) return cuda_status(e, "attn_fwd gate");
  return MTGR_OK;
}

// layer16 (the layer's own call): dy, u, the gradients dq/dk/dv/du and the
// multiplier dsilu are f16; otherwise (the attention entry point) all bf16.
static mtgr_status attn_bwd_bf16_core(const void* dy, const __half* q16, const __half* k16,
                                      const __half* v16, int64_t ld16, const void* u, bool layer16, int64_t ldu,
                                      const __half* o, const float* mean, const float* rstd, const int32_t* offsets,
                                      int32_t B, const uint8_t* gid, const int64_t* ts, int64_t T, int H, int d,
                                      void* dq, void* dk, void* dv, void* du, int64_t ldg, const void* dsilu,
                                      uint8_t* ws, const AttnWs& w, cudaStream_t s, const DsStore& ds) {
  int32_t* status = reinterpret_cast<int32_t*>(ws + w.status);
  int32_t* plan = reinterpret_cast<int32_t*>(ws + w.plan);
  MTGR_CUDA_TRY(cudaMemsetAsync(status, 0, sizeof(int32_t), s), "attn_bwd status");
  if (T == 0 || B == 0) return MTGR_OK;
  MTGR_CUDA_TRY(launch_plan(offsets, B, gid, T, H, plan, status, s, nullptr, nullptr, ds.slots), "attn_bwd plan");
  const int64_t HD = (int64_t)H * d;
  __half* dO = reinterpret_cast<__half*>(ws + w.dO);
  cudaError_t e =
      layer16 ? launch_ln_gate_bwd(static_cast<const __half*>(dy), o, static_cast<const __half*>(u), ldu, mean, rstd,
                                   dO, static_cast<__half*>(du), ldg, static_cast<const __half*>(dsilu), T, (int)HD, s)
              : launch_ln_gate_bwd(static_cast<const __nv_bfloat16*>(dy), o, static_cast<const __nv_bfloat16*>(u),
                                   ldu, mean, rstd, dO, static_cast<__nv_bfloat16*>(du), ldg,
                                   static_cast<const __nv_bfloat16*>(dsilu), T, (int)HD, s);
  if (e != cudaSuccess) return cuda_status(e, "attn_bwd gate");
  const uint16_t* m16 = static_cast<const uint16_t*>(dsilu);
  MTGR_CUDA_TRY(launch_attn_bwd_f16(q16, k16, v16, ld16, dO, T, H, d, plan, B, ts, dq, dk, dv, ldg,
                                    m16 ? m16 + HD : nullptr, m16 ? m16 + 2 * HD : nullptr,
                                    m16 ? m16 + 3 * HD : nullptr, layer16, status, s, ds.base, ds.slots),
                "attn_bwd tcgen05");
  return MTGR_OK;
}

}  // namespace mtgr

using namespace mtgr;

// ===========================================================================
extern "C" {

const char* mtgr_last_error(void) { return g_err; }

void mtgr_trace_enable(int on) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace_on = on != 0;
}

void mtgr_trace_reset(void) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace.clear();
  g_pool_used = 0;
  g_open = -1;
}

int mtgr_trace_report(int max_entries, char* names, int name_len, double* total_ms, int32_t* launches) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  std::vector<std::string> keys;
  std::vector<double> ms;
  std::vector<int32_t> cnt;
  for (const TraceRec& r : g_trace) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) return -1;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) return -1;
    size_t k = 0;
    while (k < keys.size() && keys[k] != r.name) ++k;
    if (k == keys.size()) {
      keys.push_back(r.name);
      ms.push_back(0.0);
      cnt.push_back(0);
    }
    ms[k] += t;
    cnt[k] += 1;
  }
  const int n = (int)keys.size();
  for (int k = 0; k < n && k < max_entries; ++k) {
    if (names && name_len > 0) {
      strncpy(names + (size_t)k * name_len, keys[k].c_str(), name_len - 1);
      names[(size_t)k * name_len + name_len - 1] = 0;
    }
    if (total_ms) total_ms[k] = ms[k];
    if (launches) launches[k] = cnt[k];
  }
  return n;
}
int mtgr_version(void) { return 100; }

mtgr_status mtgr_validate_batch(const int32_t* offsets, int32_t B, const uint8_t* gid, int64_t T,
                                int32_t* status_word, mtgr_stream_t stream) {
  mtgr_status st = check_meta(offsets, B, gid, T);
  if (st != MTGR_OK) return st;
  REQUIRE(status_word != nullptr, MTGR_ERR_INVALID_ARG, "status_word is NULL");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  MTGR_CUDA_TRY(cudaMemsetAsync(status_word, 0, sizeof(int32_t), s), "validate_batch memset");
  MTGR_CUDA_TRY(launch_user_info(offsets, B, gid, T, nullptr, status_word, s), "validate_batch");
  return MTGR_OK;
}

mtgr_status mtgr_debug_visible_counts(const int32_t* offsets, int32_t B, const uint8_t* gid, const int64_t* ts,
                                      int64_t T, int32_t* cnt, int64_t* total_pairs, mtgr_stream_t stream) {
  mtgr_status st = check_meta(offsets, B, gid, T);
  if (st != MTGR_OK) return st;
  REQUIRE(total_pairs != nullptr && (T == 0 || (cnt && ts)), MTGR_ERR_INVALID_ARG, "NULL output / ts");
  MTGR_CUDA_TRY(launch_visible_counts(offsets, B, gid, ts, T, cnt, total_pairs,
                                      reinterpret_cast<cudaStream_t>(stream)),
                "visible_counts");
  return MTGR_OK;
}

mtgr_status mtgr_debug_plan_counts(const void* workspace, int32_t B, int32_t* counts_host, mtgr_stream_t stream) {
  REQUIRE(workspace != nullptr && counts_host != nullptr && B >= 0, MTGR_ERR_INVALID_ARG,
          "NULL workspace / counts_host or B < 0");
  // the attention workspace (first in a layer workspace): status word, then the plan
  const int32_t* plan = reinterpret_cast<const int32_t*>(static_cast<const uint8_t*>(workspace) + 256);
  const int32_t* counts = plan + plan_layout(B, 0, 1).counts;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  MTGR_CUDA_TRY(cudaMemcpyAsync(counts_host, counts, 4 * sizeof(int32_t), cudaMemcpyDeviceToHost, s), "plan counts");
  MTGR_CUDA_TRY(cudaStreamSynchronize(s), "plan counts");
  return MTGR_OK;
}

mtgr_status mtgr_debug_wait_timeout(int32_t* status_word, mtgr_stream_t stream) {
  REQUIRE(status_word != nullptr, MTGR_ERR_INVALID_ARG, "status_word is NULL");
  MTGR_CUDA_TRY(launch_wait_timeout(status_word, reinterpret_cast<cudaStream_t>(stream)), "wait_timeout");
  return MTGR_OK;
}

mtgr_status mtgr_expand_rows(const void* src, const int32_t* rows, int64_t n, void* dst, int64_t T, int32_t D,
                             mtgr_dtype dtype, mtgr_stream_t stream) {
  REQUIRE(n >= 0 && T >= 0 && D > 0, MTGR_ERR_INVALID_ARG, "n, T must be >= 0 and D > 0");
  REQUIRE(dtype == MTGR_BF16 || dtype == MTGR_F32, MTGR_ERR_UNSUPPORTED, "dtype");
  const int64_t row_bytes = (int64_t)D * (dtype == MTGR_BF16 ? 2 : 4);
  REQUIRE(row_bytes % 16 == 0, MTGR_ERR_INVALID_ARG, "a row must be a multiple of 16 bytes (D %% 8 == 0 for bf16)");
  REQUIRE(T == 0 || dst != nullptr, MTGR_ERR_INVALID_ARG, "dst is NULL");
  REQUIRE(n == 0 || (src != nullptr && rows != nullptr), MTGR_ERR_INVALID_ARG, "src / rows is NULL");
  REQUIRE(aligned16(src) && aligned16(dst), MTGR_ERR_INVALID_ARG, "src and dst must be 16-byte aligned");
  if (T == 0) return MTGR_OK;
  MTGR_CUDA_TRY(launch_expand_rows(src, rows, n, dst, T, row_bytes, reinterpret_cast<cudaStream_t>(stream)),
                "expand_rows");
  return MTGR_OK;
}

mtgr_status mtgr_group_layernorm_fwd(const void* x, void* y, float* mean, float* rstd, const uint8_t* gid,
                                     const float* gamma, const float* beta, int64_t T, int32_t D, float eps,
                                     mtgr_dtype dtype, mtgr_stream_t stream) {
  REQUIRE(T >= 0 && D > 0 && D % 8 == 0 && D <= 4096, MTGR_ERR_UNSUPPORTED, "D must be a multiple of 8 in [8, 4096]");
  REQUIRE(dtype == MTGR_F32 || dtype == MTGR_BF16 || dtype == MTGR_F16, MTGR_ERR_INVALID_ARG, "bad dtype");
  if (T == 0) return MTGR_OK;
  REQUIRE(x && y && gid && gamma && beta, MTGR_ERR_INVALID_ARG, "NULL pointer");
  REQUIRE(aligned16(x) && aligned16(y) && aligned16(gamma) && aligned16(beta), MTGR_ERR_INVALID_ARG,
          "tensors must be 16-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e =
      dtype == MTGR_BF16 ? launch_gln_fwd(static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y),
                                          mean, rstd, gid, gamma, beta, T, D, eps, s)
      : dtype == MTGR_F16 ? launch_gln_fwd(static_cast<const __half*>(x), static_cast<__half*>(y), mean, rstd, gid,
                                           gamma, beta, T, D, eps, s)
                          : launch_gln_fwd(static_cast<const float*>(x), static_cast<float*>(y), mean, rstd, gid,
                                           gamma, beta, T, D, eps, s);
  if (e != cudaSuccess) return cuda_status(e, "group_layernorm_fwd");
  return MTGR_OK;
}

size_t mtgr_group_layernorm_bwd_workspace_size(int64_t T, int32_t D) {
  return align256((size_t)gln_bwd_blocks(T) * 8 * (size_t)D * sizeof(float));
}

mtgr_status mtgr_group_layernorm_bwd(const void* dy, const void* x, const float* mean, const float* rstd,
                                     const uint8_t* gid, const float* gamma, const void* dx_residual, void* dx,
                                     float* dgamma, float* dbeta, int64_t T, int32_t D, mtgr_dtype dtype,
                                     void* workspace, size_t workspace_bytes, mtgr_stream_t stream) {
  REQUIRE(T >= 0 && D > 0 && D % 8 == 0 && D <= 4096, MTGR_ERR_UNSUPPORTED, "D must be a multiple of 8 in [8, 4096]");
  REQUIRE(dtype != MTGR_F16, MTGR_ERR_UNSUPPORTED, "MTGR_F16 is supported by the forward entry points only");
  REQUIRE(dtype == MTGR_F32 || dtype == MTGR_BF16, MTGR_ERR_INVALID_ARG, "bad dtype");
  REQUIRE(dgamma && dbeta, MTGR_ERR_INVALID_ARG, "NULL dgamma/dbeta");
  REQUIRE(workspace && workspace_bytes >= mtgr_group_layernorm_bwd_workspace_size(T, D), MTGR_ERR_WORKSPACE,
          "workspace too small");
  REQUIRE(T == 0 || (dy && x && mean && rstd && gid && gamma && dx), MTGR_ERR_INVALID_ARG, "NULL pointer");
  REQUIRE(aligned16(dy) && aligned16(x) && aligned16(dx) && aligned16(gamma) && aligned16(dx_residual),
          MTGR_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e =
      dtype == MTGR_BF16
          ? launch_gln_bwd(static_cast<const __nv_bfloat16*>(dy), static_cast<const __nv_bfloat16*>(x), mean, rstd,
                           gid, gamma, static_cast<const __nv_bfloat16*>(dx_residual), static_cast<__nv_bfloat16*>(dx),
                           dgamma, dbeta, static_cast<float*>(workspace), T, D, nullptr, s)
          : launch_gln_bwd(static_cast<const float*>(dy), static_cast<const float*>(x), mean, rstd, gid, gamma,
                           static_cast<const float*>(dx_residual), static_cast<float*>(dx), dgamma, dbeta,
                           static_cast<float*>(workspace), T, D, nullptr, s);
  if (e != cudaSuccess) return cuda_status(e, "group_layernorm_bwd");
  return MTGR_OK;
}

size_t mtgr_attn_workspace_size(int32_t B, int64_t T, int32_t n_heads, int32_t d_h, mtgr_dtype dtype) {
  if (B < 0 || T < 0 || n_heads <= 0 || d_h <= 0) return 0;
  return attn_ws(B, T, n_heads, d_h, dtype).total;
}

size_t mtgr_attn_ds_store_size(const int32_t* offsets_host, int32_t B, int32_t n_heads, int32_t d_h,
                               mtgr_dtype dtype) {
  if (offsets_host == nullptr || B <= 0 || n_heads <= 0) return 0;
  if (dtype != MTGR_BF16 || (d_h != 64 && d_h != 128)) return 0;
  int64_t tiles = 0;
  for (int32_t b = 0; b < B; ++b) {
    const int64_t n = (int64_t)offsets_host[b + 1] - offsets_host[b];
    if (n < 0) return 0;
    const int64_t nt = (n + kTile - 1) / kTile;
    tiles += nt * nt;
  }
  if (tiles == 0) return 0;
  return (size_t)tiles * n_heads * kDsTileBytes + 1024;  // + the 1024-byte alignment of the store
}

static mtgr_status check_attn(const void* q, const void* k, const void* v, const void* u, int64_t ld_in,
                              const int32_t* offsets, int32_t B, const uint8_t* gid, const int64_t* ts, int64_t T,
                              int32_t H, int32_t d, mtgr_dtype dtype, void* ws, size_t ws_bytes) {
  mtgr_status st = check_meta(offsets, B, gid, T);
  if (st != MTGR_OK) return st;
  REQUIRE(H >= 1 && d >= 1, MTGR_ERR_INVALID_ARG, "n_heads and d_h must be positive");
  if (dtype == MTGR_BF16) {
    REQUIRE(d == 64 || d == 128, MTGR_ERR_UNSUPPORTED, "bf16 path supports d_h in {64, 128}");
    REQUIRE(ld_in % 8 == 0, MTGR_ERR_INVALID_ARG, "ld_in must be a multiple of 8");
  } else if (dtype == MTGR_F32) {
    REQUIRE(d <= 128 && d % 4 == 0, MTGR_ERR_UNSUPPORTED, "fp32 path supports d_h <= 128, d_h % 4 == 0");
    REQUIRE(ld_in % 4 == 0, MTGR_ERR_INVALID_ARG, "ld_in must be a multiple of 4");
  } else {
    REQUIRE(dtype != MTGR_F16, MTGR_ERR_UNSUPPORTED, "MTGR_F16 is supported by the layer and stack forward only");
    REQUIRE(false, MTGR_ERR_INVALID_ARG, "bad dtype");
  }
  REQUIRE((int64_t)H * d % 8 == 0 && H * d <= 4096, MTGR_ERR_UNSUPPORTED, "H*d_h must be a multiple of 8, <= 4096");
  REQUIRE(ld_in >= (int64_t)H * d, MTGR_ERR_INVALID_ARG, "ld_in < H*d_h");
  REQUIRE(T == 0 || (q && k && v && u && ts), MTGR_ERR_INVALID_ARG, "NULL q/k/v/u/ts");
  REQUIRE(aligned16(q) && aligned16(k) && aligned16(v) && aligned16(u), MTGR_ERR_INVALID_ARG,
          "q/k/v/u must be 16-byte aligned");
  REQUIRE(ws && ws_bytes >= attn_ws(B, T, H, d, dtype).total && aligned16(ws), MTGR_ERR_WORKSPACE,
          "workspace missing or smaller than mtgr_attn_workspace_size()");
  return MTGR_OK;
}

mtgr_status mtgr_hstu_attn_fwd(const void* q, const void* k, const void* v, const void* u, int64_t ld_in,
                               const int32_t* offsets, int32_t B, const uint8_t* gid, const int64_t* ts,
                               int64_t T, int32_t n_heads, int32_t d_h, float eps, void* y, void* o_saved,
                               float* ln_mean, float* ln_rstd, mtgr_dtype dtype, void* workspace,
                               size_t workspace_bytes, mtgr_stream_t stream) {
  mtgr_status st = check_attn(q, k, v, u, ld_in, offsets, B, gid, ts, T, n_heads, d_h, dtype, workspace,
                              workspace_bytes);
  if (st != MTGR_OK) return st;
  REQUIRE(T == 0 || (y && o_saved && ln_mean && ln_rstd), MTGR_ERR_INVALID_ARG, "NULL output");
  REQUIRE(aligned16(y) && aligned16(o_saved), MTGR_ERR_INVALID_ARG, "outputs must be 16-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const AttnWs w = attn_ws(B, T, n_heads, d_h, dtype);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int64_t HD = (int64_t)n_heads * d_h;
  if (dtype == MTGR_BF16) {
    __half* q16 = reinterpret_cast<__half*>(ws + w.qkv16);
    __half* k16 = q16 + align256(T * HD * 2) / 2;
    __half* v16 = k16 + align256(T * HD * 2) / 2;
    using bf = __nv_bfloat16;
    MTGR_CUDA_TRY(launch_bf16_to_f16(static_cast<const bf*>(q), ld_in, q16, HD, T, (int)HD, s), "attn_fwd f16 q");
    MTGR_CUDA_TRY(launch_bf16_to_f16(static_cast<const bf*>(k), ld_in, k16, HD, T, (int)HD, s), "attn_fwd f16 k");
    MTGR_CUDA_TRY(launch_bf16_to_f16(static_cast<const bf*>(v), ld_in, v16, HD, T, (int)HD, s), "attn_fwd f16 v");
    return attn_fwd_bf16_core(q16, k16, v16, HD, u, false, ld_in, offsets, B, gid, ts, T, n_heads, d_h, eps,
                              static_cast<bf*>(y), static_cast<__half*>(o_saved), ln_mean, ln_rstd, ws, w, s);
  }
  int32_t* status = reinterpret_cast<int32_t*>(ws + w.status);
  int32_t* plan = reinterpret_cast<int32_t*>(ws + w.plan);
  MTGR_CUDA_TRY(cudaMemsetAsync(status, 0, sizeof(int32_t), s), "attn_fwd status");
  if (T == 0 || B == 0) return MTGR_OK;
  MTGR_CUDA_TRY(launch_plan(offsets, B, gid, T, n_heads, plan, status, s), "attn_fwd plan");
  const PlanLayout L = plan_layout(B, T, n_heads);
  MTGR_CUDA_TRY(launch_attn_f32_fwd(static_cast<const float*>(q), static_cast<const float*>(k),
                                    static_cast<const float*>(v), ld_in,
                                    reinterpret_cast<const UserInfo*>(plan + L.users), B, ts, T, n_heads, d_h,
                                    static_cast<float*>(o_saved), s),
                "attn_fwd fp32");
  MTGR_CUDA_TRY(launch_ln_gate_fwd(static_cast<const float*>(o_saved), static_cast<const float*>(u), ld_in,
                                   static_cast<float*>(y), ln_mean, ln_rstd, T, (int)HD, eps, s),
                "attn_fwd gate");
  return MTGR_OK;
}

mtgr_status mtgr_hstu_attn_bwd(const void* dy, const void* q, const void* k, const void* v, const void* u,
                               int64_t ld_in, const void* o_saved, const float* ln_mean, const float* ln_rstd,
                               const int32_t* offsets, int32_t B, const uint8_t* gid, const int64_t* ts,
                               int64_t T, int32_t n_heads, int32_t d_h, void* dq, void* dk, void* dv, void* du,
                               int64_t ld_grad, const void* dsilu_uqkv, mtgr_dtype dtype, void* workspace,
                               size_t workspace_bytes, mtgr_stream_t stream) {
  mtgr_status st = check_attn(q, k, v, u, ld_in, offsets, B, gid, ts, T, n_heads, d_h, dtype, workspace,
                              workspace_bytes);
  if (st != MTGR_OK) return st;
  const int64_t HD = (int64_t)n_heads * d_h;
  REQUIRE(T == 0 || (dy && o_saved && ln_mean && ln_rstd && dq && dk && dv && du), MTGR_ERR_INVALID_ARG,
          "NULL pointer");
  REQUIRE(ld_grad >= HD && ld_grad % 8 == 0, MTGR_ERR_INVALID_ARG, "ld_grad must be >= H*d_h and a multiple of 8");
  REQUIRE(aligned16(dy) && aligned16(o_saved) && aligned16(dq) && aligned16(dk) && aligned16(dv) &&
              aligned16(du) && aligned16(dsilu_uqkv),
          MTGR_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  REQUIRE(dsilu_uqkv == nullptr || ld_grad == 4 * HD, MTGR_ERR_INVALID_ARG,
          "with dsilu_uqkv, ld_grad must be 4*H*d_h");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const AttnWs w = attn_ws(B, T, n_heads, d_h, dtype);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (dtype == MTGR_BF16) {
    using bf = __nv_bfloat16;
    __half* q16 = reinterpret_cast<__half*>(ws + w.qkv16);
    __half* k16 = q16 + align256(T * HD * 2) / 2;
    __half* v16 = k16 + align256(T * HD * 2) / 2;
    MTGR_CUDA_TRY(launch_bf16_to_f16(static_cast<const bf*>(q), ld_in, q16, HD, T, (int)HD, s), "attn_bwd f16 q");
    MTGR_CUDA_TRY(launch_bf16_to_f16(static_cast<const bf*>(k), ld_in, k16, HD, T, (int)HD, s), "attn_bwd f16 k");
    MTGR_CUDA_TRY(launch_bf16_to_f16(static_cast<const bf*>(v), ld_in, v16, HD, T, (int)HD, s), "attn_bwd f16 v");
    return attn_bwd_bf16_core(static_cast<const bf*>(dy), q16, k16, v16, HD, u, false, ld_in,
                              static_cast<const __half*>(o_saved), ln_mean, ln_rstd, offsets, B, gid, ts, T, n_heads,
                              d_h, static_cast<bf*>(dq), static_cast<bf*>(dk), static_cast<bf*>(dv),
                              static_cast<bf*>(du), ld_grad, static_cast<const bf*>(dsilu_uqkv), ws, w, s,
                              ds_store_region(ws, workspace_bytes, w.total));
  }
  int32_t* status = reinterpret_cast<int32_t*>(ws + w.status);
  int32_t* plan = reinterpret_cast<int32_t*>(ws + w.plan);
  MTGR_CUDA_TRY(cudaMemsetAsync(status, 0, sizeof(int32_t), s), "attn_bwd status");
  if (T == 0 || B == 0) return MTGR_OK;
  MTGR_CUDA_TRY(launch_plan(offsets, B, gid, T, n_heads, plan, status, s), "attn_bwd plan");
  const PlanLayout L = plan_layout(B, T, n_heads);
  const float* m = static_cast<const float*>(dsilu_uqkv);
  float* dO = reinterpret_cast<float*>(ws + w.dO);
  MTGR_CUDA_TRY(launch_ln_gate_bwd(static_cast<const float*>(dy), static_cast<const float*>(o_saved),
                                   static_cast<const float*>(u), ld_in, ln_mean, ln_rstd, dO,
                                   static_cast<float*>(du), ld_grad, m, T, (int)HD, s),
                "attn_bwd gate");
  MTGR_CUDA_TRY(launch_attn_f32_bwd(static_cast<const float*>(q), static_cast<const float*>(k),
                                    static_cast<const float*>(v), ld_in, dO,
                                    reinterpret_cast<const UserInfo*>(plan + L.users), B, ts, T, n_heads, d_h,
                                    static_cast<float*>(dq), static_cast<float*>(dk), static_cast<float*>(dv),
                                    ld_grad, m ? m + HD : nullptr, m ? m + 2 * HD : nullptr,
                                    m ? m + 3 * HD : nullptr, s),
                "attn_bwd fp32");
  return MTGR_OK;
}

// ---------------------------------------------------------------------------
// Layer
// ---------------------------------------------------------------------------
size_t mtgr_layer_workspace_size(int32_t B, int64_t T, int32_t d_model, int32_t n_heads, int32_t d_h,
                                 mtgr_dtype dtype) {
  if (B < 0 || T < 0 || d_model <= 0 || n_heads <= 0 || d_h <= 0) return 0;
  return layer_ws(B, T, d_model, n_heads, d_h, dtype).total;
}

static mtgr_status check_layer(const mtgr_layer_weights* w, const int32_t* offsets, int32_t B, const uint8_t* gid,
                               int64_t T, mtgr_dtype dtype, void* ws, size_t ws_bytes) {
  REQUIRE(w != nullptr, MTGR_ERR_INVALID_ARG, "weights is NULL");
  mtgr_status st = check_meta(offsets, B, gid, T);
  if (st != MTGR_OK) return st;
  const int D = w->d_model, H = w->n_heads, d = w->d_h;
  REQUIRE(D > 0 && H > 0 && d > 0, MTGR_ERR_INVALID_ARG, "bad layer dims");
  REQUIRE(D % 64 == 0 && D <= 4096 && (H * d) % 64 == 0, MTGR_ERR_UNSUPPORTED,
          "d_model and H*d_h must be multiples of 64 (d_model <= 4096)");
  REQUIRE(dtype == MTGR_F32 || dtype == MTGR_BF16 || dtype == MTGR_F16, MTGR_ERR_INVALID_ARG, "bad dtype");
  if (dtype != MTGR_F32)
    REQUIRE(d == 64 || d == 128, MTGR_ERR_UNSUPPORTED, "the tensor-core path supports d_h in {64, 128}");
  REQUIRE(w->w_uqkv && w->w_o && w->gamma && w->beta, MTGR_ERR_INVALID_ARG, "NULL weight");
  REQUIRE(aligned16(w->w_uqkv) && aligned16(w->w_o) && aligned16(w->gamma) && aligned16(w->beta),
          MTGR_ERR_INVALID_ARG, "weights must be 16-byte aligned");
  REQUIRE((w->w_uqkv_f16 == nullptr) == (w->w_o_f16 == nullptr), MTGR_ERR_INVALID_ARG,
          "set both f16 weight copies or neither");
  REQUIRE(aligned16(w->w_uqkv_f16) && aligned16(w->w_o_f16), MTGR_ERR_INVALID_ARG,
          "f16 weight copies must be 16-byte aligned");
  REQUIRE(ws && aligned16(ws) && ws_bytes >= layer_ws(B, T, D, H, d, dtype).total, MTGR_ERR_WORKSPACE,
          "workspace missing or smaller than mtgr_layer_workspace_size()");
  return MTGR_OK;
}

// f16 operands of a MTGR_BF16 layer's two weight matrices: the caller's copies
// when given, else conversions into the workspace at c.
static cudaError_t layer_weights_f16(const mtgr_layer_weights* w, __half* c, const __half** wu16,
                                     const __half** wo16, cudaStream_t s) {
  const int D = w->d_model;
  const int64_t HD = (int64_t)w->n_heads * w->d_h, N4 = 4 * HD;
  if (w->w_uqkv_f16) {
    *wu16 = static_cast<const __half*>(w->w_uqkv_f16);
    *wo16 = static_cast<const __half*>(w->w_o_f16);
    return cudaSuccess;
  }
  __half* co = c + align256((size_t)D * N4 * 2) / 2;
  cudaError_t e = launch_bf16_to_f16(static_cast<const __nv_bfloat16*>(w->w_uqkv), N4, c, N4, D, (int)N4, s);
  if (e == cudaSuccess) e = launch_bf16_to_f16(static_cast<const __nv_bfloat16*>(w->w_o), D, co, D, HD, D, s);
  *wu16 = c;
  *wo16 = co;
  return e;
}

static mtgr_status layer_fwd_impl(const mtgr_layer_weights* w, const void* x, void* x_out,
                                  const mtgr_layer_saved* sv, const int32_t* offsets, int32_t B, const uint8_t* gid,
                                  const int64_t* ts, int64_t T, mtgr_dtype dtype, void* workspace,
                                  size_t workspace_bytes, mtgr_stream_t stream, bool plan_ready,
                                  const int32_t* n_norm = nullptr, bool keep_dsilu = true) {
  // keep_dsilu = false: a forward for inference, which writes no silu'(z)
  mtgr_status st = check_layer(w, offsets, B, gid, T, dtype, workspace, workspace_bytes);
  if (st != MTGR_OK) return st;
  REQUIRE(sv != nullptr, MTGR_ERR_INVALID_ARG, "saved is NULL");
  REQUIRE(T == 0 || (x && x_out && sv->xn && (sv->dsilu || !keep_dsilu) && sv->uqkv && sv->o && sv->y && sv->gln_mean &&
                     sv->gln_rstd && sv->ln_mean && sv->ln_rstd && ts),
          MTGR_ERR_INVALID_ARG, "NULL tensor");
  REQUIRE(aligned16(x) && aligned16(x_out) && aligned16(sv->xn) && aligned16(sv->dsilu) && aligned16(sv->uqkv) &&
              aligned16(sv->o) && aligned16(sv->y),
          MTGR_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  const int D = w->d_model, H = w->n_heads, d = w->d_h;
  const int64_t HD = (int64_t)H * d, N4 = 4 * HD;
  const LayerWs L = layer_ws(B, T, D, H, d, dtype);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t* status = reinterpret_cast<int32_t*>(ws + L.attn_base + L.attn.status);
  if (T == 0) return MTGR_OK;
  mtgr_status r;
  // 16-bit tensor-core path: every operand f16 (MTGR_F16; MTGR_BF16 with f16
  // copies of its weights and f16 activations between the steps)
  const bool bf_io = dtype == MTGR_BF16;
  const __half* wu16 = static_cast<const __half*>(w->w_uqkv);
  const __half* wo16 = static_cast<const __half*>(w->w_o);
  if (bf_io) {
    MTGR_CUDA_TRY(layer_weights_f16(w, reinterpret_cast<__half*>(ws + L.w16), &wu16, &wo16, s), "layer_fwd W f16");
    // xn = GLN(x) in f16
    cudaError_t e = launch_gln_fwd(static_cast<const __nv_bfloat16*>(x), static_cast<__half*>(sv->xn), sv->gln_mean,
                                   sv->gln_rstd, gid, w->gamma, w->beta, T, D, w->eps_gln, s);
    if (e != cudaSuccess) return cuda_status(e, "layer_fwd gln");
  } else {
    r = mtgr_group_layernorm_fwd(x, sv->xn, sv->gln_mean, sv->gln_rstd, gid, w->gamma, w->beta, T, D, w->eps_gln,
                                 dtype, stream);
    if (r != MTGR_OK) return r;
  }
  if (dtype != MTGR_F32) {
    using bf = __nv_bfloat16;
    GemmArgs g{};
    g.M = T; g.N = N4; g.K = D;
    g.A = static_cast<const bf*>(sv->xn); g.lda = D; g.a_mn_major = false;
    g.B = reinterpret_cast<const bf*>(wu16); g.ldb = N4; g.b_mn_major = true;
    g.ab_f16 = true;
    // [U|Q|K|V] = silu(z) and silu'(z), both f16
    g.epi = EPI_SILU; g.C = sv->uqkv; g.c_f16 = true; g.ldc = N4;
    g.Z = keep_dsilu ? static_cast<bf*>(sv->dsilu) : nullptr; g.ldz = N4;
    g.z_f16 = true;
    g.splits = 1; g.status = status; g.name = "gemm_uqkv";
    MTGR_CUDA_TRY(launch_gemm_bf16(g, s), "layer_fwd uqkv gemm");
  } else {
    MTGR_CUDA_TRY(launch_gemm_f32(EPI_SILU, T, N4, D, static_cast<const float*>(sv->xn), D, 1,
                                  static_cast<const float*>(w->w_uqkv), N4, 1, static_cast<float*>(sv->uqkv), N4,
                                  nullptr, 0, static_cast<float*>(sv->dsilu), N4, s),
                  "layer_fwd uqkv gemm");
  }
  if (dtype != MTGR_F32) {
    const __half* a = static_cast<const __half*>(sv->uqkv);
    r = attn_fwd_bf16_core(a + HD, a + 2 * HD, a + 3 * HD, N4, a, true, N4, offsets, B, gid, ts, T, H, d, w->eps_ln,
                           sv->y, static_cast<__half*>(sv->o), sv->ln_mean, sv->ln_rstd, ws + L.attn_base, L.attn, s,
                           plan_ready, /*y_f16=*/true, n_norm);
  } else {
    const float* a = static_cast<const float*>(sv->uqkv);
    r = mtgr_hstu_attn_fwd(a + HD, a + 2 * HD, a + 3 * HD, a, N4, offsets, B, gid, ts, T, H, d, w->eps_ln, sv->y,
                           sv->o, sv->ln_mean, sv->ln_rstd, dtype, ws + L.attn_base, L.attn.total, stream);
  }
  if (r != MTGR_OK) return r;
  if (dtype != MTGR_F32) {
    using bf = __nv_bfloat16;
    GemmArgs g{};
    g.M = T; g.N = D; g.K = HD;
    g.A = static_cast<const bf*>(sv->y); g.lda = HD; g.a_mn_major = false;
    g.B = reinterpret_cast<const bf*>(wo16); g.ldb = D; g.b_mn_major = true;
    g.ab_f16 = true;
    g.status = status; g.name = "gemm_out";
    if (L.splits_out > 1) {
      // x' = x + Σ_k slices of y·W_o, the slices in fp32
      float* parts = reinterpret_cast<float*>(ws + L.wpart);
      g.epi = EPI_F32; g.C = parts; g.ldc = D; g.splits = L.splits_out;
      MTGR_CUDA_TRY(launch_gemm_bf16(g, s), "layer_fwd out gemm");
      MTGR_CUDA_TRY(launch_split_reduce_residual(parts, gemm_splits(HD, L.splits_out), T * D, T * D, x, x_out, !bf_io,
                                                 s),
                    "layer_fwd out reduce");
    } else {
      // x' = x + y·W_o in the layer's dtype
      g.epi = EPI_RESIDUAL; g.C = x_out; g.c_f16 = !bf_io; g.ldc = D; g.R = static_cast<const bf*>(x); g.ldr = D;
      g.r_f16 = !bf_io;
      g.splits = 1;
      MTGR_CUDA_TRY(launch_gemm_bf16(g, s), "layer_fwd out gemm");
    }
  } else {
    MTGR_CUDA_TRY(launch_gemm_f32(EPI_RESIDUAL, T, D, HD, static_cast<const float*>(sv->y), HD, 1,
                                  static_cast<const float*>(w->w_o), D, 1, static_cast<float*>(x_out), D,
                                  static_cast<const float*>(x), D, nullptr, 0, s),
                  "layer_fwd out gemm");
  }
  return MTGR_OK;
}

mtgr_status mtgr_layer_weights_to_f16(const mtgr_layer_weights* w, void* w_uqkv_f16, void* w_o_f16,
                                      mtgr_stream_t stream) {
  REQUIRE(w != nullptr && w->w_uqkv && w->w_o && w_uqkv_f16 && w_o_f16, MTGR_ERR_INVALID_ARG, "NULL pointer");
  const int D = w->d_model;
  const int64_t HD = (int64_t)w->n_heads * w->d_h, N4 = 4 * HD;
  REQUIRE(D > 0 && HD > 0 && D % 8 == 0 && HD % 8 == 0, MTGR_ERR_INVALID_ARG, "bad layer dims");
  REQUIRE(aligned16(w->w_uqkv) && aligned16(w->w_o) && aligned16(w_uqkv_f16) && aligned16(w_o_f16),
          MTGR_ERR_INVALID_ARG, "weights must be 16-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  MTGR_CUDA_TRY(launch_bf16_to_f16(static_cast<const __nv_bfloat16*>(w->w_uqkv), N4, static_cast<__half*>(w_uqkv_f16),
                                   N4, D, (int)N4, s),
                "weights_to_f16 W_uqkv");
  MTGR_CUDA_TRY(launch_bf16_to_f16(static_cast<const __nv_bfloat16*>(w->w_o), D, static_cast<__half*>(w_o_f16), D, HD,
                                   D, s),
                "weights_to_f16 W_o");
  return MTGR_OK;
}

mtgr_status mtgr_hstu_layer_fwd(const mtgr_layer_weights* w, const void* x, void* x_out,
                                const mtgr_layer_saved* sv, const int32_t* offsets, int32_t B, const uint8_t* gid,
                                const int64_t* ts, int64_t T, mtgr_dtype dtype, void* workspace,
                                size_t workspace_bytes, mtgr_stream_t stream) {
  return layer_fwd_impl(w, x, x_out, sv, offsets, B, gid, ts, T, dtype, workspace, workspace_bytes, stream, false);
}

mtgr_status mtgr_hstu_stack_fwd(const mtgr_layer_weights* w, int32_t n_layers, const void* x, void* x_out, void* act,
                                const mtgr_layer_saved* sv, const int32_t* offsets, int32_t B, const uint8_t* gid,
                                const int64_t* ts, int64_t T, mtgr_dtype dtype, void* workspace,
                                size_t workspace_bytes, mtgr_stream_t stream) {
  REQUIRE(w != nullptr && n_layers >= 1, MTGR_ERR_INVALID_ARG, "weights is NULL or n_layers < 1");
  for (int32_t l = 1; l < n_layers; ++l)
    REQUIRE(w[l].d_model == w[0].d_model && w[l].n_heads == w[0].n_heads && w[l].d_h == w[0].d_h,
            MTGR_ERR_INVALID_ARG, "every layer of a stack must have the same d_model, n_heads and d_h");
  REQUIRE(T == 0 || n_layers == 1 || (act != nullptr && act != x && act != x_out), MTGR_ERR_INVALID_ARG,
          "act must be a separate [T, d_model] buffer when n_layers > 1");
  REQUIRE(T == 0 || x != x_out, MTGR_ERR_INVALID_ARG, "x and x_out may not alias");
  const void* in = x;
  for (int32_t l = 0; l < n_layers; ++l) {
    void* out = ((n_layers - 1 - l) & 1) ? act : x_out;  // the last layer writes x_out
    // one work-list build serves every layer: they share the batch and the workspace
    const mtgr_status r = layer_fwd_impl(w + l, in, out, sv, offsets, B, gid, ts, T, dtype, workspace,
                                         workspace_bytes, stream, l > 0, nullptr, /*keep_dsilu=*/false);
    if (r != MTGR_OK) return r;
    in = out;
  }
  return MTGR_OK;
}

mtgr_status mtgr_hstu_layer_bwd(const mtgr_layer_weights* w, const void* x, const mtgr_layer_saved* sv,
                                const void* dx_out, void* dx, const mtgr_layer_grads* gr, const int32_t* offsets,
                                int32_t B, const uint8_t* gid, const int64_t* ts, int64_t T, mtgr_dtype dtype,
                                void* workspace, size_t workspace_bytes, mtgr_stream_t stream) {
  REQUIRE(dtype != MTGR_F16, MTGR_ERR_UNSUPPORTED, "MTGR_F16 is supported by the forward entry points only");
  mtgr_status st = check_layer(w, offsets, B, gid, T, dtype, workspace, workspace_bytes);
  if (st != MTGR_OK) return st;
  REQUIRE(sv && gr && gr->dw_uqkv && gr->dw_o && gr->dgamma && gr->dbeta, MTGR_ERR_INVALID_ARG,
          "NULL saved / grads");
  REQUIRE(T == 0 || (x && dx_out && dx && sv->xn && sv->dsilu && sv->uqkv && sv->o && sv->y && sv->gln_mean &&
                     sv->gln_rstd && sv->ln_mean && sv->ln_rstd && ts),
          MTGR_ERR_INVALID_ARG, "NULL tensor");
  REQUIRE(aligned16(x) && aligned16(dx_out) && aligned16(dx), MTGR_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  const int D = w->d_model, H = w->n_heads, d = w->d_h;
  const int64_t HD = (int64_t)H * d, N4 = 4 * HD;
  const LayerWs L = layer_ws(B, T, D, H, d, dtype);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t* status = reinterpret_cast<int32_t*>(ws + L.attn_base + L.attn.status);
  void* dY = ws + L.dY;
  void* dZ = ws + L.dZ;
  void* dxn = ws + L.dxn;
  float* wpart = reinterpret_cast<float*>(ws + L.wpart);
  if (T == 0) {
    MTGR_CUDA_TRY(cudaMemsetAsync(gr->dw_uqkv, 0, sizeof(float) * D * N4, s), "layer_bwd zero");
    MTGR_CUDA_TRY(cudaMemsetAsync(gr->dw_o, 0, sizeof(float) * HD * D, s), "layer_bwd zero");
    MTGR_CUDA_TRY(cudaMemsetAsync(gr->dgamma, 0, sizeof(float) * 4 * D, s), "layer_bwd zero");
    MTGR_CUDA_TRY(cudaMemsetAsync(gr->dbeta, 0, sizeof(float) * 4 * D, s), "layer_bwd zero");
    return MTGR_OK;
  }
  using bf = __nv_bfloat16;
  // MTGR_BF16: gradients are carried in f16 (11 significand bits) scaled by a
  // power of two s (from max|dx'|, so that f16's range holds them whatever the
  // loss scale); the weight gradients, dγ, dβ and dx leave multiplied by 1/s.
  // Weights are used as exact f16 copies.
  const __half* wu16 = nullptr;
  const __half* wo16 = nullptr;
  const __half* dxo16 = nullptr;
  const float* inv_scale = nullptr;
  if (dtype == MTGR_BF16) {
    MTGR_CUDA_TRY(layer_weights_f16(w, reinterpret_cast<__half*>(ws + L.w16), &wu16, &wo16, s), "layer_bwd W f16");
    float* gs = reinterpret_cast<float*>(ws + L.gscale + 16);
    MTGR_CUDA_TRY(launch_grad_to_f16(static_cast<const bf*>(dx_out), reinterpret_cast<__half*>(ws + L.dxo16), T * D,
                                     reinterpret_cast<unsigned*>(ws + L.gscale), gs, s),
                  "layer_bwd dx' f16");
    dxo16 = reinterpret_cast<const __half*>(ws + L.dxo16);
    inv_scale = gs + 1;
  }
  // 1. dY = dx' · W_oᵀ
  if (dtype == MTGR_BF16) {
    GemmArgs g{};
    g.M = T; g.N = HD; g.K = D;
    g.A = reinterpret_cast<const bf*>(dxo16); g.lda = D; g.a_mn_major = false;
    g.B = reinterpret_cast<const bf*>(wo16); g.ldb = D; g.b_mn_major = false;
    g.ab_f16 = true;
    g.epi = EPI_PLAIN; g.C = dY; g.c_f16 = true; g.ldc = HD; g.splits = 1; g.status = status; g.name = "gemm_dY";
    MTGR_CUDA_TRY(launch_gemm_bf16(g, s), "layer_bwd dY gemm");
  } else {
    MTGR_CUDA_TRY(launch_gemm_f32(EPI_PLAIN, T, HD, D, static_cast<const float*>(dx_out), D, 1,
                                  static_cast<const float*>(w->w_o), 1, D, static_cast<float*>(dY), HD, nullptr, 0,
                                  nullptr, 0, s),
                  "layer_bwd dY gemm");
  }
  // 2. dW_o = Yᵀ · dx'
  if (dtype == MTGR_BF16) {
    GemmArgs g{};
    g.M = HD; g.N = D; g.K = T;
    g.A = static_cast<const bf*>(sv->y); g.lda = HD; g.a_mn_major = true;
    g.B = reinterpret_cast<const bf*>(dxo16); g.ldb = D; g.b_mn_major = true;
    g.ab_f16 = true;
    g.epi = EPI_F32; g.C = L.splits_o > 1 ? (void*)wpart : (void*)gr->dw_o; g.ldc = D; g.out_scale = inv_scale;
    g.splits = L.splits_o; g.status = status; g.name = "gemm_dWo";
    MTGR_CUDA_TRY(launch_gemm_bf16(g, s), "layer_bwd dW_o gemm");
    if (L.splits_o > 1)
      MTGR_CUDA_TRY(launch_split_reduce(wpart, L.splits_o, HD * D, HD * D, gr->dw_o, s), "layer_bwd dW_o reduce");
  } else {
    MTGR_CUDA_TRY(launch_gemm_f32(EPI_PLAIN, HD, D, T, static_cast<const float*>(sv->y), 1, HD,
                                  static_cast<const float*>(dx_out), D, 1, gr->dw_o, D, nullptr, 0, nullptr, 0, s),
                  "layer_bwd dW_o gemm");
  }
  // 3. attention backward with the SiLU backward of the projection fused: dZ = [dU|dQ|dK|dV] ⊙ silu'(z)
  mtgr_status r;
  if (dtype == MTGR_BF16) {
    const __half* a = static_cast<const __half*>(sv->uqkv);
    __half* dz = static_cast<__half*>(dZ);
    r = attn_bwd_bf16_core(dY, a + HD, a + 2 * HD, a + 3 * HD, N4, a, true, N4, static_cast<const __half*>(sv->o),
                           sv->ln_mean, sv->ln_rstd, offsets, B, gid, ts, T, H, d, dz + HD, dz + 2 * HD, dz + 3 * HD,
                           dz, N4, sv->dsilu, ws + L.attn_base, L.attn, s,
                           ds_store_region(ws, workspace_bytes, L.total));
  } else {
    const float* a = static_cast<const float*>(sv->uqkv);
    float* dz = static_cast<float*>(dZ);
    r = mtgr_hstu_attn_bwd(dY, a + HD, a + 2 * HD, a + 3 * HD, a, N4, sv->o, sv->ln_mean, sv->ln_rstd, offsets, B,
                           gid, ts, T, H, d, dz + HD, dz + 2 * HD, dz + 3 * HD, dz, N4, sv->dsilu, dtype,
                           ws + L.attn_base, L.attn.total, stream);
  }
  if (r != MTGR_OK) return r;
  // 4. dW_uqkv = xnᵀ · dZ ;  5. dxn = dZ · W_uqkvᵀ
  if (dtype == MTGR_BF16) {
    GemmArgs g{};
    g.M = D; g.N = N4; g.K = T;
    g.A = static_cast<const bf*>(sv->xn); g.lda = D; g.a_mn_major = true;
    g.B = static_cast<const bf*>(dZ); g.ldb = N4; g.b_mn_major = true;
    g.ab_f16 = true;
    g.epi = EPI_F32; g.C = L.splits_uqkv > 1 ? (void*)wpart : (void*)gr->dw_uqkv; g.ldc = N4;
    g.out_scale = inv_scale;
    g.splits = L.splits_uqkv; g.status = status; g.name = "gemm_dWuqkv";
    MTGR_CUDA_TRY(launch_gemm_bf16(g, s), "layer_bwd dW_uqkv gemm");
    if (L.splits_uqkv > 1)
      MTGR_CUDA_TRY(launch_split_reduce(wpart, L.splits_uqkv, (int64_t)D * N4, (int64_t)D * N4, gr->dw_uqkv, s),
                    "layer_bwd dW_uqkv reduce");
    GemmArgs h{};
    h.M = T; h.N = D; h.K = N4;
    h.A = static_cast<const bf*>(dZ); h.lda = N4; h.a_mn_major = false;
    h.B = reinterpret_cast<const bf*>(wu16); h.ldb = N4; h.b_mn_major = false;
    h.ab_f16 = true;
    h.epi = EPI_PLAIN; h.C = dxn; h.c_f16 = true; h.ldc = D; h.splits = 1; h.status = status; h.name = "gemm_dxn";
    MTGR_CUDA_TRY(launch_gemm_bf16(h, s), "layer_bwd dxn gemm");
    // 6. GLN backward (dxn f16, scaled by s) + residual path
    cudaError_t e = launch_gln_bwd(static_cast<const __half*>(dxn), static_cast<const bf*>(x), sv->gln_mean,
                                   sv->gln_rstd, gid, w->gamma, static_cast<const bf*>(dx_out), static_cast<bf*>(dx),
                                   gr->dgamma, gr->dbeta, reinterpret_cast<float*>(ws + L.gln_part), T, D, inv_scale,
                                   s);
    if (e != cudaSuccess) return cuda_status(e, "layer_bwd gln");
    return MTGR_OK;
  }
  MTGR_CUDA_TRY(launch_gemm_f32(EPI_PLAIN, D, N4, T, static_cast<const float*>(sv->xn), 1, D,
                                static_cast<const float*>(dZ), N4, 1, gr->dw_uqkv, N4, nullptr, 0, nullptr, 0, s),
                "layer_bwd dW_uqkv gemm");
  MTGR_CUDA_TRY(launch_gemm_f32(EPI_PLAIN, T, D, N4, static_cast<const float*>(dZ), N4, 1,
                                static_cast<const float*>(w->w_uqkv), 1, N4, static_cast<float*>(dxn), D, nullptr, 0,
                                nullptr, 0, s),
                "layer_bwd dxn gemm");
  // 6. GLN backward + residual path
  return mtgr_group_layernorm_bwd(dxn, x, sv->gln_mean, sv->gln_rstd, gid, w->gamma, dx_out, dx, gr->dgamma,
                                  gr->dbeta, T, D, dtype, ws + L.gln_part,
                                  mtgr_group_layernorm_bwd_workspace_size(T, D), stream);
}


}  // extern "C"

// ---------------------------------------------------------------------------
// Chunked candidate scoring of one request, the history encoded once
// ---------------------------------------------------------------------------
namespace mtgr {
namespace {
// meta[0..1] = offsets {0, T}, meta[2] = n_u, meta[3] = first query row; the
// segment's group ids and stamps: history rows 0 .. n_hist-1, then candidates
// c0 .. c0+c-1 of the request (rows n_hist + c0 .. of gid / ts).
__global__ void chunk_meta_kernel(int32_t* meta, uint8_t* gid_out, int64_t* ts_out, const uint8_t* gid,
                                  const int64_t* ts, int32_t n_hist, int32_t c0, int32_t c, int32_t n_total,
                                  int32_t q0) {
  const int T = n_hist + c;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i == 0) {
    meta[0] = 0;
    meta[1] = T;
    meta[2] = n_total;
    meta[3] = q0;
  }
  if (gid_out && i < T) {
    const int src = i < n_hist ? i : n_hist + c0 + (i - n_hist);
    gid_out[i] = gid[src];
    ts_out[i] = ts[src];
  }
}

struct ChunkWs {
  size_t meta, gid, ts, layer, xn, dsilu, o, y, gstat, lstat, total;
};
// rows_a: rows of the attention segment; rows_c: rows of the projections
static ChunkWs chunk_ws(int64_t rows_a, int64_t rows_c, int D, int H, int d, mtgr_dtype dt) {
  ChunkWs w;
  const int64_t HD = (int64_t)H * d;
  size_t o = 0;
  w.meta = o;
  o += 256;
  w.gid = o;
  o += align256((size_t)rows_a);
  w.ts = o;
  o += align256((size_t)rows_a * 8);
  w.layer = o;
  o += layer_ws(1, rows_a, D, H, d, dt).total;
  w.xn = o;
  o += align256((size_t)rows_c * D * 2);
  w.dsilu = o;
  o += align256((size_t)rows_c * 4 * HD * 2);
  w.o = o;
  o += align256((size_t)rows_a * HD * 2);
  w.y = o;
  o += align256((size_t)rows_c * HD * 2);
  w.gstat = o;
  o += align256((size_t)rows_c * 8);
  w.lstat = o;
  o += align256((size_t)rows_a * 8);
  w.total = o;
  return w;
}

// Cache layout: every layer's [U|Q|K|V] rows (history, then one chunk), then
// every layer's f16 copies of W_uqkv and W_o (used by the MTGR_BF16 path, made
// once by the history call instead of once per chunk).
static size_t cache_rows_bytes(int32_t n_layers, int32_t n_hist, int32_t chunk, int32_t H, int32_t d) {
  return align256((size_t)n_layers * ((size_t)n_hist + chunk) * 4 * (size_t)H * d * 2);
}
static size_t cache_w16_bytes(int32_t D, int32_t H, int32_t d) {
  const size_t N4 = 4 * (size_t)H * d;
  return align256((size_t)D * N4 * 2) + align256((size_t)H * d * D * 2);
}

static mtgr_status check_chunked(const mtgr_layer_weights* w, int32_t n_layers, int32_t chunk, int32_t n_hist,
                                 int32_t n_cand, mtgr_dtype dtype) {
  REQUIRE(w != nullptr && n_layers >= 1, MTGR_ERR_INVALID_ARG, "weights is NULL or n_layers < 1");
  REQUIRE(dtype == MTGR_BF16 || dtype == MTGR_F16, MTGR_ERR_UNSUPPORTED,
          "chunked candidate scoring runs on the 16-bit tensor-core path (MTGR_BF16 or MTGR_F16)");
  REQUIRE(n_hist >= 0 && n_cand >= 0 && chunk >= 1, MTGR_ERR_INVALID_ARG, "n_hist, n_cand >= 0 and chunk >= 1");
  REQUIRE((int64_t)n_hist + chunk < (int64_t(1) << 30), MTGR_ERR_UNSUPPORTED, "request too long");
  for (int32_t l = 1; l < n_layers; ++l)
    REQUIRE(w[l].d_model == w[0].d_model && w[l].n_heads == w[0].n_heads && w[l].d_h == w[0].d_h,
            MTGR_ERR_INVALID_ARG, "every layer must have the same d_model, n_heads and d_h");
  return MTGR_OK;
}
}  // namespace
}  // namespace mtgr

extern "C" {

size_t mtgr_stack_cache_size(int32_t n_layers, int32_t n_hist, int32_t chunk, int32_t d_model, int32_t n_heads,
                             int32_t d_h) {
  if (n_layers < 1 || n_hist < 0 || chunk < 1 || d_model <= 0 || n_heads <= 0 || d_h <= 0) return 0;
  return cache_rows_bytes(n_layers, n_hist, chunk, n_heads, d_h) +
         (size_t)n_layers * cache_w16_bytes(d_model, n_heads, d_h);
}

size_t mtgr_stack_chunk_workspace_size(int32_t n_hist, int32_t chunk, int32_t d_model, int32_t n_heads, int32_t d_h,
                                       mtgr_dtype dtype) {
  if (n_hist < 0 || chunk < 1 || d_model <= 0 || n_heads <= 0 || d_h <= 0) return 0;
  const size_t a = chunk_ws(n_hist, n_hist, d_model, n_heads, d_h, dtype).total;
  const size_t b = chunk_ws((int64_t)n_hist + chunk, chunk, d_model, n_heads, d_h, dtype).total;
  return a > b ? a : b;
}

mtgr_status mtgr_hstu_stack_hist_fwd(const mtgr_layer_weights* w, int32_t n_layers, const void* x_hist, void* act,
                                     void* cache, int32_t chunk, const uint8_t* gid, const int64_t* ts, int32_t n_hist,
                                     int32_t n_cand, mtgr_dtype dtype, void* workspace, size_t workspace_bytes,
                                     mtgr_stream_t stream) {
  mtgr_status st = check_chunked(w, n_layers, chunk, n_hist, n_cand, dtype);
  if (st != MTGR_OK) return st;
  const int D = w->d_model, H = w->n_heads, d = w->d_h;
  const int64_t HD = (int64_t)H * d, N4 = 4 * HD;
  const ChunkWs C = chunk_ws(n_hist, n_hist, D, H, d, dtype);
  REQUIRE(workspace && aligned16(workspace) &&
              workspace_bytes >= mtgr_stack_chunk_workspace_size(n_hist, chunk, D, H, d, dtype),
          MTGR_ERR_WORKSPACE, "workspace missing or smaller than mtgr_stack_chunk_workspace_size()");
  REQUIRE(cache && aligned16(cache), MTGR_ERR_INVALID_ARG, "cache is NULL or not 16-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == MTGR_BF16) {  // the chunk calls use these f16 copies of the weights
    uint8_t* wc = static_cast<uint8_t*>(cache) + cache_rows_bytes(n_layers, n_hist, chunk, H, d);
    for (int32_t l = 0; l < n_layers; ++l) {
      __half* cw = reinterpret_cast<__half*>(wc + (size_t)l * cache_w16_bytes(D, H, d));
      MTGR_CUDA_TRY(launch_bf16_to_f16(static_cast<const __nv_bfloat16*>(w[l].w_uqkv), N4, cw, N4, D, (int)N4, s),
                    "stack_hist W_uqkv f16");
      MTGR_CUDA_TRY(launch_bf16_to_f16(static_cast<const __nv_bfloat16*>(w[l].w_o), D,
                                       cw + align256((size_t)D * N4 * 2) / 2, D, HD, D, s),
                    "stack_hist W_o f16");
    }
  }
  if (n_hist == 0) return MTGR_OK;
  REQUIRE(x_hist && act && gid && ts, MTGR_ERR_INVALID_ARG, "NULL pointer");
  REQUIRE(aligned16(x_hist) && aligned16(act), MTGR_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* meta = reinterpret_cast<int32_t*>(ws + C.meta);
  chunk_meta_kernel<<<1, 32, 0, s>>>(meta, nullptr, nullptr, gid, ts, n_hist, 0, 0, n_hist + n_cand, 0);
  MTGR_CUDA_TRY(cudaGetLastError(), "stack_hist meta");
  mtgr_layer_saved sv{};
  sv.xn = ws + C.xn;
  sv.dsilu = ws + C.dsilu;
  sv.o = ws + C.o;
  sv.y = ws + C.y;
  sv.gln_mean = reinterpret_cast<float*>(ws + C.gstat);
  sv.gln_rstd = sv.gln_mean + n_hist;
  sv.ln_mean = reinterpret_cast<float*>(ws + C.lstat);
  sv.ln_rstd = sv.ln_mean + n_hist;
  const size_t act_half = align256((size_t)n_hist * D * 2);
  const void* in = x_hist;
  for (int32_t l = 0; l < n_layers; ++l) {
    void* out = static_cast<uint8_t*>(act) + (l & 1) * act_half;
    sv.uqkv = static_cast<uint8_t*>(cache) + (size_t)l * ((size_t)n_hist + chunk) * N4 * 2;
    // history rows see history rows only: their activations are those of the whole request, with its n_u
    st = layer_fwd_impl(w + l, in, out, &sv, meta, 1, gid, ts, n_hist, dtype, ws + C.layer,
                        layer_ws(1, n_hist, D, H, d, dtype).total, stream, l > 0, meta + 2, /*keep_dsilu=*/false);
    if (st != MTGR_OK) return st;
    in = out;
  }
  return MTGR_OK;
}

mtgr_status mtgr_hstu_stack_cand_fwd(const mtgr_layer_weights* w, int32_t n_layers, const void* x_cand, void* x_out,
                                     void* act, void* cache, int32_t chunk, const uint8_t* gid, const int64_t* ts,
                                     int32_t n_hist, int32_t n_cand, int32_t c0, int32_t c, mtgr_dtype dtype,
                                     void* workspace, size_t workspace_bytes, mtgr_stream_t stream) {
  mtgr_status st = check_chunked(w, n_layers, chunk, n_hist, n_cand, dtype);
  if (st != MTGR_OK) return st;
  REQUIRE(c >= 0 && c <= chunk && c0 >= 0 && (int64_t)c0 + c <= n_cand, MTGR_ERR_INVALID_ARG,
          "the chunk must satisfy 0 <= c <= chunk and c0 + c <= n_cand");
  const int D = w->d_model, H = w->n_heads, d = w->d_h;
  const int64_t HD = (int64_t)H * d, N4 = 4 * HD;
  const int64_t Tc = (int64_t)n_hist + c;
  const ChunkWs C = chunk_ws(Tc, c, D, H, d, dtype);
  REQUIRE(workspace && aligned16(workspace) &&
              workspace_bytes >= mtgr_stack_chunk_workspace_size(n_hist, chunk, D, H, d, dtype),
          MTGR_ERR_WORKSPACE, "workspace missing or smaller than mtgr_stack_chunk_workspace_size()");
  if (c == 0) return MTGR_OK;
  REQUIRE(x_cand && x_out && cache && gid && ts && (n_layers == 1 || act), MTGR_ERR_INVALID_ARG, "NULL pointer");
  REQUIRE(x_cand != x_out && (n_layers == 1 || (act != x_cand && act != x_out)), MTGR_ERR_INVALID_ARG,
          "x_cand, x_out and act must be distinct");
  REQUIRE(aligned16(x_cand) && aligned16(x_out) && aligned16(act) && aligned16(cache), MTGR_ERR_INVALID_ARG,
          "tensors must be 16-byte aligned");
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t* meta = reinterpret_cast<int32_t*>(ws + C.meta);
  uint8_t* gid_c = ws + C.gid;
  int64_t* ts_c = reinterpret_cast<int64_t*>(ws + C.ts);
  chunk_meta_kernel<<<(unsigned)((Tc + 255) / 256), 256, 0, s>>>(meta, gid_c, ts_c, gid, ts, n_hist, c0, c,
                                                                  n_hist + n_cand, n_hist);
  MTGR_CUDA_TRY(cudaGetLastError(), "stack_cand meta");
  const LayerWs L = layer_ws(1, Tc, D, H, d, dtype);
  uint8_t* lws = ws + C.layer;
  int32_t* status = reinterpret_cast<int32_t*>(lws + L.attn_base + L.attn.status);
  __half* xn = reinterpret_cast<__half*>(ws + C.xn);
  __half* o = reinterpret_cast<__half*>(ws + C.o);
  __half* y = reinterpret_cast<__half*>(ws + C.y);
  float* gmean = reinterpret_cast<float*>(ws + C.gstat);
  float* lmean = reinterpret_cast<float*>(ws + C.lstat);
  using bf = __nv_bfloat16;
  const bool bf_io = dtype == MTGR_BF16;
  const void* in = x_cand;
  for (int32_t l = 0; l < n_layers; ++l) {
    const mtgr_layer_weights& W = w[l];
    void* out = ((n_layers - 1 - l) & 1) ? act : x_out;  // the last layer writes x_out
    __half* a = reinterpret_cast<__half*>(static_cast<uint8_t*>(cache) + (size_t)l * ((size_t)n_hist + chunk) * N4 * 2);
    const __half* wu16 = static_cast<const __half*>(W.w_uqkv);
    const __half* wo16 = static_cast<const __half*>(W.w_o);
    if (bf_io) {  // f16 copies made by the history call
      const __half* cw = reinterpret_cast<const __half*>(static_cast<const uint8_t*>(cache) +
                                                         cache_rows_bytes(n_layers, n_hist, chunk, H, d) +
                                                         (size_t)l * cache_w16_bytes(D, H, d));
      wu16 = cw;
      wo16 = cw + align256((size_t)D * N4 * 2) / 2;
    }
    // 1. GLN of the candidate rows (group ids from the segment's candidate part)
    cudaError_t e = bf_io ? launch_gln_fwd(static_cast<const bf*>(in), xn, gmean, gmean + c, gid_c + n_hist, W.gamma,
                                           W.beta, c, D, W.eps_gln, s)
                          : launch_gln_fwd(static_cast<const __half*>(in), xn, gmean, gmean + c, gid_c + n_hist,
                                           W.gamma, W.beta, c, D, W.eps_gln, s);
    if (e != cudaSuccess) return cuda_status(e, "cand gln");
    // 2. [U|Q|K|V] of the candidates, appended to the cached history rows
    {
      GemmArgs g{};
      g.M = c; g.N = N4; g.K = D;
      g.A = reinterpret_cast<const bf*>(xn); g.lda = D; g.a_mn_major = false;
      g.B = reinterpret_cast<const bf*>(wu16); g.ldb = N4; g.b_mn_major = true;
      g.ab_f16 = true;
      g.epi = EPI_SILU; g.C = a + (size_t)n_hist * N4; g.c_f16 = true; g.ldc = N4;
      g.Z = nullptr; g.ldz = N4; g.z_f16 = true;  // inference: no silu'(z)
      g.splits = 1; g.status = status; g.name = "gemm_uqkv";
      MTGR_CUDA_TRY(launch_gemm_bf16(g, s), "cand uqkv gemm");
    }
    // 3. attention of the candidate query tiles over [history | chunk], n_u of the whole request
    st = attn_fwd_bf16_core(a + HD, a + 2 * HD, a + 3 * HD, N4, a, true, N4, meta, 1, gid_c, ts_c, Tc, H, d, W.eps_ln,
                            nullptr, o, nullptr, nullptr, lws + L.attn_base, L.attn, s, l > 0, true, meta + 2,
                            meta + 3, /*do_gate=*/false);
    if (st != MTGR_OK) return st;
    // 4. LN(O) ⊙ U of the candidate rows
    e = launch_ln_gate_fwd(o + (size_t)n_hist * HD, a + (size_t)n_hist * N4, N4, y, lmean, lmean + c, c, (int)HD,
                           W.eps_ln, s);
    if (e != cudaSuccess) return cuda_status(e, "cand gate");
    // 5. x' = x + y·W_o
    {
      GemmArgs g{};
      g.M = c; g.N = D; g.K = HD;
      g.A = reinterpret_cast<const bf*>(y); g.lda = HD; g.a_mn_major = false;
      g.B = reinterpret_cast<const bf*>(wo16); g.ldb = D; g.b_mn_major = true;
      g.ab_f16 = true;
      g.epi = EPI_RESIDUAL; g.C = out; g.c_f16 = !bf_io; g.ldc = D; g.R = static_cast<const bf*>(in); g.ldr = D;
      g.r_f16 = !bf_io;
      g.splits = 1; g.status = status; g.name = "gemm_out";
      MTGR_CUDA_TRY(launch_gemm_bf16(g, s), "cand out gemm");
    }
    in = out;
  }
  return MTGR_OK;
}

}  // extern "C"
