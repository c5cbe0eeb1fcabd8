// api.cu -- C ABI of libi8q: error reporting, device helpers and the
// dynamic quantized inner-product context (Simd
// "SynetDynamicQuantizedInnerProduct16b": Init, Enable, InternalBufferSize,
// ExternalBufferSize, Info, SetParams, Forward, Clear).
#include <map>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "common.cuh"

namespace i8q {

static thread_local std::string g_last_error;

void set_error(const std::string& msg) { g_last_error = msg; }

int fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return I8Q_ERR_CUDA;
}

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
int g_sm_count[kMaxDevices] = {0};
uint32_t* g_status[kMaxDevices] = {nullptr};
}  // namespace

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_sm_count[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

int once_per_device(const void* key, int (*init)(void*), void* arg) {
  int dev = 0;
  I8Q_CUDA_TRY(cudaGetDevice(&dev));
  static std::recursive_mutex mu;
  static std::map<std::pair<const void*, int>, int> done;
  std::lock_guard<std::recursive_mutex> lk(mu);
  const auto k = std::make_pair(key, dev);
  auto it = done.find(k);
  if (it != done.end()) return it->second;
  const int rc = init(arg);
  done[k] = rc;
  return rc;
}

int smem_attr(const void* func, int bytes) {
  struct A {
    const void* f;
    int b;
  } a{func, bytes};
  return once_per_device(func, [](void* p) -> int {
    const A* x = static_cast<const A*>(p);
    I8Q_CUDA_TRY(cudaFuncSetAttribute(x->f, cudaFuncAttributeMaxDynamicSharedMemorySize, x->b));
    return I8Q_OK;
  }, &a);
}

uint32_t* device_status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_status[dev]) {
    uint32_t* p = nullptr;
    if (cudaMalloc(&p, 256) != cudaSuccess) return nullptr;
    if (cudaMemset(p, 0, 256) != cudaSuccess) {
      cudaFree(p);
      return nullptr;
    }
    g_status[dev] = p;
  }
  return g_status[dev];
}

// ---- kernel timing ----------------------------------------------------------
namespace {
struct ProfEvent {
  std::string name;
  cudaEvent_t begin = nullptr, end = nullptr;
};
struct ProfTotal {
  std::string name;
  long long launches = 0;
  double ms = 0.0;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfEvent> g_prof_events;
std::vector<ProfEvent> g_prof_open;  // begun, not yet ended (per name, LIFO)
std::vector<ProfTotal> g_prof_totals;

void prof_destroy_events(std::vector<ProfEvent>& v) {
  for (auto& e : v) {
    if (e.begin) cudaEventDestroy(e.begin);
    if (e.end) cudaEventDestroy(e.end);
  }
  v.clear();
}
}  // namespace

bool profiling_enabled() { return g_prof_on; }

void profile_record(const char* name, cudaStream_t s, bool begin) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (begin) {
    ProfEvent e;
    e.name = name;
    if (cudaEventCreate(&e.begin) != cudaSuccess || cudaEventRecord(e.begin, s) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    g_prof_open.push_back(e);
    return;
  }
  for (size_t i = g_prof_open.size(); i-- > 0;) {
    if (g_prof_open[i].name == name) {
      ProfEvent e = g_prof_open[i];
      g_prof_open.erase(g_prof_open.begin() + (long)i);
      if (cudaEventCreate(&e.end) != cudaSuccess || cudaEventRecord(e.end, s) != cudaSuccess) {
        cudaGetLastError();
        cudaEventDestroy(e.begin);
        return;
      }
      g_prof_events.push_back(e);
      return;
    }
  }
}

}  // namespace i8q

using namespace i8q;

extern "C" int i8q_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  prof_destroy_events(g_prof_events);
  prof_destroy_events(g_prof_open);
  g_prof_totals.clear();
  g_prof_on = on != 0;
  return I8Q_OK;
}

extern "C" int i8q_profile_collect(void) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  I8Q_CUDA_TRY(cudaDeviceSynchronize());
  for (auto& e : g_prof_events) {
    float ms = 0.0f;
    I8Q_CUDA_TRY(cudaEventElapsedTime(&ms, e.begin, e.end));
    ProfTotal* t = nullptr;
    for (auto& x : g_prof_totals)
      if (x.name == e.name) t = &x;
    if (!t) {
      g_prof_totals.push_back(ProfTotal{e.name, 0, 0.0});
      t = &g_prof_totals.back();
    }
    t->launches += 1;
    t->ms += ms;
  }
  prof_destroy_events(g_prof_events);
  return (int)g_prof_totals.size();
}

extern "C" int i8q_profile_entry(int i, const char** name, long long* launches, double* total_ms) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (i < 0 || i >= (int)g_prof_totals.size()) return fail(I8Q_ERR_INVALID_ARG, "profile_entry: index out of range");
  if (name) *name = g_prof_totals[i].name.c_str();
  if (launches) *launches = g_prof_totals[i].launches;
  if (total_ms) *total_ms = g_prof_totals[i].ms;
  return I8Q_OK;
}

extern "C" const char* i8q_last_error(void) { return g_last_error.c_str(); }

extern "C" const char* i8q_version(void) { return "i8q 0.1 sm_103a"; }

extern "C" int i8q_sync_status(void* stream) {
  I8Q_CUDA_TRY(cudaStreamSynchronize(as_stream(stream)));
  I8Q_CUDA_TRY(cudaGetLastError());
  uint32_t* w = device_status_word();
  if (!w) return fail(I8Q_ERR_CUDA, "sync_status: no status word");
  uint32_t h = 0;
  I8Q_CUDA_TRY(cudaMemcpy(&h, w, sizeof(h), cudaMemcpyDeviceToHost));
  if (h) {
    I8Q_CUDA_TRY(cudaMemset(w, 0, sizeof(uint32_t)));
    return fail(I8Q_ERR_DEVICE_TIMEOUT, "a device-side bounded wait gave up (status " + std::to_string(h) + ")");
  }
  return I8Q_OK;
}

// ===========================================================================
// dynamic quantized inner-product context
// ===========================================================================

struct i8q_qgemm_ctx {
  int device = 0;
  size_t M = 0, N = 0, K = 0;
  int typeA = 0, typeB = 0, typeC = 0, constB = 0, bias = 0, act = 0, avoid = 0;
  int64_t Kp = 0;
  bool params_set = false;
  int core = 0;           // CORE_* below
  bool use_tc = false;    // core == CORE_TC: bf16 operand copies are kept
  // internal storage
  int8_t* iBt = nullptr;
  __nv_bfloat16* iBt_bf16 = nullptr;
  float* scaleB = nullptr;
  int32_t* colsum = nullptr;
  float* biasv = nullptr;
  void* fallback = nullptr;
  size_t internal_bytes = 0;
  // host staging of forward_host, and its upload / compute / download
  // streams with per-chunk events (created on first use)
  void* stage = nullptr;
  size_t stage_bytes = 0;
  cudaStream_t pipe[3] = {nullptr, nullptr, nullptr};
  cudaEvent_t ev_in[16] = {}, ev_out[16] = {}, ev_start = nullptr;
  std::string info;
};

namespace {

size_t a256(size_t v) { return (v + 255) & ~size_t(255); }

struct BufLayout {
  size_t uA, uA_bf16, scaleA, zeroA, iBt, iBt_bf16, scaleB, colsum, colmax, total;
};

BufLayout buf_layout(const i8q_qgemm_ctx* c) {
  BufLayout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = a256(o + bytes);
    return at;
  };
  L.uA = take(c->M * (size_t)c->Kp);
  L.uA_bf16 = c->use_tc ? take(c->M * (size_t)c->Kp * 2) : 0;
  L.scaleA = take(c->M * 4);
  L.zeroA = take(c->M * 4);
  if (!c->constB) {
    L.iBt = take(c->N * (size_t)c->Kp);
    L.iBt_bf16 = c->use_tc ? take(c->N * (size_t)c->Kp * 2) : 0;
    L.scaleB = take(c->N * 4);
    L.colsum = take(c->N * 4);
    L.colmax = take(c->N * 4);
  }
  L.total = o;
  return L;
}

void free_ctx_buffers(i8q_qgemm_ctx* c) {
  cudaFree(c->iBt);
  cudaFree(c->iBt_bf16);
  cudaFree(c->scaleB);
  cudaFree(c->colsum);
  cudaFree(c->biasv);
  cudaFree(c->fallback);
  cudaFree(c->stage);
  for (auto& st : c->pipe)
    if (st) cudaStreamDestroy(st), st = nullptr;
  for (auto& e : c->ev_in)
    if (e) cudaEventDestroy(e), e = nullptr;
  for (auto& e : c->ev_out)
    if (e) cudaEventDestroy(e), e = nullptr;
  if (c->ev_start) cudaEventDestroy(c->ev_start), c->ev_start = nullptr;
  c->iBt = nullptr;
  c->iBt_bf16 = nullptr;
  c->scaleB = nullptr;
  c->colsum = nullptr;
  c->biasv = nullptr;
  c->fallback = nullptr;
  c->stage = nullptr;
}

bool same_config(const i8q_qgemm_ctx* c, size_t M, size_t N, size_t K, int tA, int tB, int tC, int constB, int bias,
                 int act, int avoid) {
  return c->M == M && c->N == N && c->K == K && c->typeA == tA && c->typeB == tB && c->typeC == tC &&
         c->constB == constB && c->bias == bias && c->act == act && c->avoid == avoid;
}

template <typename T>
int dmalloc(T** p, size_t bytes, size_t* total) {
  if (cudaMalloc(reinterpret_cast<void**>(p), bytes ? bytes : 1) != cudaSuccess) {
    cudaGetLastError();
    return fail(I8Q_ERR_ALLOC, "cudaMalloc of " + std::to_string(bytes) + " bytes failed");
  }
  *total += bytes;
  return I8Q_OK;
}

// Core selection.  Products with enough work run on the tensor-core path
// (exact integers on the bf16 pipe, 128 x 256 tiles); small ones run in one
// fused launch on dp4a (row quantization and sums together), whose fixed
// cost is a few microseconds.  The int8 mma.sync core is kept for the
// override and as the path for very long K outside both.
// I8Q_FORCE_CORE=imma|tc|small overrides the choice (tests run every core
// on the same shapes); tc1 / tc2 also pin the tensor-core path to its
// single-CTA or CTA-pair kernel.
enum Core : int { CORE_IMMA = 0, CORE_TC = 1, CORE_SMALL = 2 };

int choose_core(size_t M, size_t N, int64_t Kp) {
  const char* f = getenv("I8Q_FORCE_CORE");
  const bool small_ok = Kp <= small_max_kp();
  if (f && std::string(f) == "imma") return CORE_IMMA;
  if (f && (std::string(f) == "tc" || std::string(f) == "tc1" || std::string(f) == "tc2")) return CORE_TC;
  if (f && std::string(f) == "small") return small_ok ? CORE_SMALL : CORE_IMMA;
  const double macs = (double)M * (double)N * (double)Kp;
  if (small_ok && macs <= (double)(1 << 27)) return CORE_SMALL;
  return CORE_TC;
}

}  // namespace

extern "C" int i8q_qgemm_dyn_init(i8q_qgemm_ctx** ctx, size_t M, size_t N, size_t K, int typeA, int typeB, int typeC,
                                  int constB, int bias, int activation, int avoidOverflow) {
  if (!ctx) return fail(I8Q_ERR_INVALID_ARG, "qgemm_dyn_init: ctx is NULL");
  constB = constB ? 1 : 0;
  bias = bias ? 1 : 0;
  avoidOverflow = avoidOverflow ? 1 : 0;
  if (M == 0 || N == 0 || K == 0) return fail(I8Q_ERR_INVALID_ARG, "qgemm_dyn_init: M, N, K must be >= 1");
  if (K > 65536) return fail(I8Q_ERR_UNSUPPORTED, "qgemm_dyn_init: K > 65536 (int32 sums could overflow)");
  if (typeA != I8Q_F32 && typeA != I8Q_BF16) return fail(I8Q_ERR_INVALID_ARG, "qgemm_dyn_init: typeA must be F32 or BF16");
  if (typeC != I8Q_F32 && typeC != I8Q_BF16) return fail(I8Q_ERR_INVALID_ARG, "qgemm_dyn_init: typeC must be F32 or BF16");
  if (constB) {
    if (typeB != I8Q_F32 && typeB != I8Q_S8)
      return fail(I8Q_ERR_INVALID_ARG, "qgemm_dyn_init: constant B must be F32 or S8");
  } else {
    if (typeB != I8Q_F32 && typeB != I8Q_BF16)
      return fail(I8Q_ERR_INVALID_ARG, "qgemm_dyn_init: non-constant B must be F32 or BF16 (S8 only when constant)");
  }
  if (activation < I8Q_ACT_IDENTITY || activation > I8Q_ACT_GELU)
    return fail(I8Q_ERR_UNSUPPORTED, "qgemm_dyn_init: unknown activation");
  if (*ctx && same_config(*ctx, M, N, K, typeA, typeB, typeC, constB, bias, activation, avoidOverflow)) return I8Q_OK;

  i8q_qgemm_ctx* c = new (std::nothrow) i8q_qgemm_ctx();
  if (!c) return fail(I8Q_ERR_ALLOC, "qgemm_dyn_init: host allocation failed");
  I8Q_CUDA_TRY(cudaGetDevice(&c->device));
  c->M = M;
  c->N = N;
  c->K = K;
  c->typeA = typeA;
  c->typeB = typeB;
  c->typeC = typeC;
  c->constB = constB;
  c->bias = bias;
  c->act = activation;
  c->avoid = avoidOverflow;
  c->Kp = round_up((int64_t)K, 64);
  c->core = choose_core(M, N, c->Kp);
  c->use_tc = c->core == CORE_TC;
  int rc = I8Q_OK;
  size_t total = 0;
  if (constB) {
    rc = dmalloc(&c->iBt, N * (size_t)c->Kp, &total);
    if (!rc && c->use_tc) rc = dmalloc(&c->iBt_bf16, N * (size_t)c->Kp * 2, &total);
    if (!rc) rc = dmalloc(&c->scaleB, N * 4, &total);
    if (!rc) rc = dmalloc(&c->colsum, N * 4, &total);
  }
  if (!rc) rc = dmalloc(&c->biasv, N * 4, &total);
  if (!rc) rc = dmalloc(&c->fallback, buf_layout(c).total, &total);
  if (!rc && cudaMemset(c->biasv, 0, N * 4) != cudaSuccess) rc = cuda_fail(cudaGetLastError(), "cudaMemset(bias)");
  if (rc) {
    free_ctx_buffers(c);
    delete c;
    return rc;
  }
  c->internal_bytes = total;
  c->params_set = !constB;
  if (*ctx) i8q_qgemm_dyn_clear(ctx);
  *ctx = c;
  return I8Q_OK;
}

extern "C" int i8q_qgemm_dyn_enabled(const i8q_qgemm_ctx* ctx) { return ctx && ctx->params_set ? 1 : 0; }

extern "C" size_t i8q_qgemm_dyn_internal_buffer_size(const i8q_qgemm_ctx* ctx) {
  return ctx ? ctx->internal_bytes + ctx->stage_bytes : 0;
}

extern "C" size_t i8q_qgemm_dyn_external_buffer_size(const i8q_qgemm_ctx* ctx) {
  return ctx ? buf_layout(ctx).total : 0;
}

extern "C" const char* i8q_qgemm_dyn_info(i8q_qgemm_ctx* ctx) {
  if (!ctx) return nullptr;
  ctx->info = std::string("sm_103a ") +
              (ctx->core == CORE_TC      ? "tcgen05.kind::f16 exact-int (bf16 operands, fp32 chunks drained to int32)"
               : ctx->core == CORE_SMALL ? "fused row quantization + dp4a.u32.s32 int32, 4 rows x 32 columns per CTA"
                                         : "mma.sync.m16n8k32.u8.s8 int32 128x128x64 4-stage") +
              "; A per-row uint8, B per-column int8" + (ctx->avoid && ctx->typeB != I8Q_S8 ? " [-64,63]" : "");
  return ctx->info.c_str();
}

extern "C" int i8q_qgemm_dyn_set_params(i8q_qgemm_ctx* ctx, const void* weight, const float* scale, const float* bias,
                                        const float* params, void* stream) {
  (void)params;
  if (!ctx) return fail(I8Q_ERR_NOT_INITIALIZED, "qgemm_dyn_set_params: no context");
  cudaStream_t s = as_stream(stream);
  const size_t N = ctx->N, K = ctx->K;
  if (ctx->constB) {
    if (!weight) return fail(I8Q_ERR_INVALID_ARG, "qgemm_dyn_set_params: weight is required for constant B");
    if (ctx->typeB == I8Q_S8 && !scale)
      return fail(I8Q_ERR_INVALID_ARG, "qgemm_dyn_set_params: scale is required for int8 B");
    const size_t wbytes = K * N * (ctx->typeB == I8Q_S8 ? 1 : 4);
    void* tmp = nullptr;
    // staging copy of the weight, then N words of column-max scratch
    if (cudaMalloc(&tmp, a256(wbytes) + N * 4) != cudaSuccess) {
      cudaGetLastError();
      return fail(I8Q_ERR_ALLOC, "qgemm_dyn_set_params: staging allocation failed");
    }
    int rc = I8Q_OK;
    if (cudaMemcpyAsync(tmp, weight, wbytes, cudaMemcpyDefault, s) != cudaSuccess)
      rc = cuda_fail(cudaGetLastError(), "cudaMemcpyAsync(weight)");
    if (!rc) {
      if (ctx->typeB == I8Q_S8) {
        rc = launch_repack_cols_s8((const int8_t*)tmp, (int64_t)K, (int64_t)N, (int64_t)N, ctx->iBt, ctx->iBt_bf16,
                                   ctx->Kp, ctx->colsum, s);
        if (!rc && cudaMemcpyAsync(ctx->scaleB, scale, N * 4, cudaMemcpyDefault, s) != cudaSuccess)
          rc = cuda_fail(cudaGetLastError(), "cudaMemcpyAsync(scale)");
      } else {
        rc = launch_quantize_cols(tmp, I8Q_F32, (int64_t)K, (int64_t)N, ctx->avoid, ctx->iBt, ctx->iBt_bf16, ctx->Kp,
                                  ctx->scaleB, ctx->colsum,
                                  reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(tmp) + a256(wbytes)), s);
      }
    }
    cudaError_t e = cudaStreamSynchronize(s);
    cudaFree(tmp);
    if (rc) return rc;
    if (e != cudaSuccess) return cuda_fail(e, "qgemm_dyn_set_params: weight preparation");
  }
  if (ctx->bias) {
    if (bias) I8Q_CUDA_TRY(cudaMemcpyAsync(ctx->biasv, bias, N * 4, cudaMemcpyDefault, s));
    else I8Q_CUDA_TRY(cudaMemsetAsync(ctx->biasv, 0, N * 4, s));
    I8Q_CUDA_TRY(cudaStreamSynchronize(s));
  }
  ctx->params_set = true;
  return I8Q_OK;
}

namespace {

// Forward of rows row0 .. row0 + rows - 1 (all rows by default): A and C
// point at the first of them; their row quantization goes to the same rows
// of buf.
int forward_impl(i8q_qgemm_ctx* ctx, const void* A, const void* B, void* buf, void* C, int out_mode, cudaStream_t s,
                 int64_t row0 = 0, int64_t rows = -1) {
  if (!ctx) return fail(I8Q_ERR_NOT_INITIALIZED, "qgemm_dyn_forward: no context");
  if (!ctx->params_set) return fail(I8Q_ERR_NOT_INITIALIZED, "qgemm_dyn_forward: SetParams was not called");
  if (!A || !C) return fail(I8Q_ERR_INVALID_ARG, "qgemm_dyn_forward: A and C are required");
  if (!ctx->constB && !B) return fail(I8Q_ERR_INVALID_ARG, "qgemm_dyn_forward: B is required (B is not constant)");
  uint8_t* base = static_cast<uint8_t*>(buf ? buf : ctx->fallback);
  if (reinterpret_cast<uintptr_t>(base) & 255) return fail(I8Q_ERR_INVALID_ARG, "qgemm_dyn_forward: buf must be 256-byte aligned");
  const BufLayout L = buf_layout(ctx);
  uint8_t* uA = base + L.uA + row0 * ctx->Kp;
  __nv_bfloat16* uA_bf16 = ctx->use_tc ? reinterpret_cast<__nv_bfloat16*>(base + L.uA_bf16) + row0 * ctx->Kp : nullptr;
  float* scaleA = reinterpret_cast<float*>(base + L.scaleA) + row0;
  int32_t* zeroA = reinterpret_cast<int32_t*>(base + L.zeroA) + row0;
  const int64_t M = rows < 0 ? (int64_t)ctx->M : rows, N = (int64_t)ctx->N, K = (int64_t)ctx->K;
  const bool small = ctx->core == CORE_SMALL;
  int rc = I8Q_OK;
  if (!small) {
    rc = launch_quantize_rows(A, ctx->typeA, M, K, K, uA, uA_bf16, ctx->Kp, scaleA, zeroA, s);
    if (rc) return rc;
  }
  const int8_t* iBt = ctx->iBt;
  const __nv_bfloat16* iBt_bf16 = ctx->iBt_bf16;
  const float* scaleB = ctx->scaleB;
  const int32_t* colsum = ctx->colsum;
  if (!ctx->constB) {
    int8_t* q = reinterpret_cast<int8_t*>(base + L.iBt);
    __nv_bfloat16* qb = ctx->use_tc ? reinterpret_cast<__nv_bfloat16*>(base + L.iBt_bf16) : nullptr;
    float* sb = reinterpret_cast<float*>(base + L.scaleB);
    int32_t* cs = reinterpret_cast<int32_t*>(base + L.colsum);
    // the tensor-core product reads only the bf16 codes
    rc = launch_quantize_cols(B, ctx->typeB, K, N, ctx->avoid, ctx->use_tc ? nullptr : q, qb, ctx->Kp, sb, cs,
                              reinterpret_cast<uint32_t*>(base + L.colmax), s);
    if (rc) return rc;
    iBt = q;
    iBt_bf16 = qb;
    scaleB = sb;
    colsum = cs;
  }
  GemmEpilogue ep{zeroA, scaleA, colsum, scaleB, ctx->bias ? ctx->biasv : nullptr, ctx->act, out_mode, C, N};
  if (small) return launch_gemm_small(A, ctx->typeA, M, K, ctx->Kp, iBt, N, uA, scaleA, zeroA, ep, s);
  if (ctx->use_tc) {
    // |uA - 128| <= 2^7; |iB| <= 2^7, or 2^6 in the narrowed range
    const int qb = (ctx->typeB == I8Q_S8 || !ctx->avoid) ? 7 : 6;
    rc = launch_gemm_tc(uA_bf16, iBt_bf16, M, N, ctx->Kp, 7 + qb, ep, s);
    if (rc != I8Q_ERR_UNSUPPORTED) return rc;
    if (!ctx->constB) {
      // the int8 codes were not written for the tensor-core product
      rc = launch_quantize_cols(B, ctx->typeB, K, N, ctx->avoid, const_cast<int8_t*>(iBt), nullptr, ctx->Kp,
                                const_cast<float*>(scaleB), const_cast<int32_t*>(colsum),
                                reinterpret_cast<uint32_t*>(base + L.colmax), s);
      if (rc) return rc;
    }
  }
  return launch_gemm_imma(uA, iBt, M, N, ctx->Kp, ep, s);
}

}  // namespace

extern "C" int i8q_qgemm_dyn_forward(i8q_qgemm_ctx* ctx, const void* A, const void* B, void* buf, void* C,
                                     void* stream) {
  if (ctx && !C) return fail(I8Q_ERR_INVALID_ARG, "qgemm_dyn_forward: C is NULL");
  return forward_impl(ctx, A, B, buf, C, ctx && ctx->typeC == I8Q_BF16 ? OUT_BF16 : OUT_F32, as_stream(stream));
}

extern "C" int i8q_qgemm_dyn_forward_s32(i8q_qgemm_ctx* ctx, const void* A, const void* B, void* buf, int32_t* acc,
                                         void* stream) {
  return forward_impl(ctx, A, B, buf, acc, OUT_S32, as_stream(stream));
}

extern "C" int i8q_qgemm_dyn_forward_host(i8q_qgemm_ctx* ctx, const void* A_host, void* C_host, void* stream) {
  if (!ctx) return fail(I8Q_ERR_NOT_INITIALIZED, "qgemm_dyn_forward_host: no context");
  if (!A_host || !C_host) return fail(I8Q_ERR_INVALID_ARG, "qgemm_dyn_forward_host: A and C are required");
  if (!ctx->constB) return fail(I8Q_ERR_INVALID_ARG, "qgemm_dyn_forward_host: needs a constant-B context");
  const size_t a_bytes = ctx->M * ctx->K * (ctx->typeA == I8Q_F32 ? 4 : 2);
  const size_t c_bytes = ctx->M * ctx->N * (ctx->typeC == I8Q_F32 ? 4 : 2);
  const size_t need = a256(a_bytes) + a256(c_bytes);
  if (ctx->stage_bytes < need) {
    cudaFree(ctx->stage);
    ctx->stage = nullptr;
    ctx->stage_bytes = 0;
    if (cudaMalloc(&ctx->stage, need) != cudaSuccess) {
      cudaGetLastError();
      return fail(I8Q_ERR_ALLOC, "qgemm_dyn_forward_host: staging allocation failed");
    }
    ctx->stage_bytes = need;
  }
  cudaStream_t s = as_stream(stream);
  uint8_t* dA = static_cast<uint8_t*>(ctx->stage);
  uint8_t* dC = dA + a256(a_bytes);
  // Rows are independent (A is quantized per row, B is constant), so the
  // call runs as a pipeline over row chunks: chunk i computes while chunk
  // i + 1 is uploaded and chunk i - 1 downloaded, on three streams of the
  // context ordered by events; it still returns only when C_host is filled.
  const int64_t M = (int64_t)ctx->M;
  const int nch = (int)std::max<int64_t>(1, std::min<int64_t>(8, M / 1024));
  if (nch == 1) {
    I8Q_CUDA_TRY(cudaMemcpyAsync(dA, A_host, a_bytes, cudaMemcpyHostToDevice, s));
    int rc = i8q_qgemm_dyn_forward(ctx, dA, nullptr, nullptr, dC, stream);
    if (rc) return rc;
    I8Q_CUDA_TRY(cudaMemcpyAsync(C_host, dC, c_bytes, cudaMemcpyDeviceToHost, s));
    I8Q_CUDA_TRY(cudaStreamSynchronize(s));
    return I8Q_OK;
  }
  for (auto& st : ctx->pipe)
    if (!st) I8Q_CUDA_TRY(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));
  for (int i = 0; i < nch; ++i) {
    if (!ctx->ev_in[i]) I8Q_CUDA_TRY(cudaEventCreateWithFlags(&ctx->ev_in[i], cudaEventDisableTiming));
    if (!ctx->ev_out[i]) I8Q_CUDA_TRY(cudaEventCreateWithFlags(&ctx->ev_out[i], cudaEventDisableTiming));
  }
  if (!ctx->ev_start) I8Q_CUDA_TRY(cudaEventCreateWithFlags(&ctx->ev_start, cudaEventDisableTiming));
  // work already queued on the caller's stream comes first
  I8Q_CUDA_TRY(cudaEventRecord(ctx->ev_start, s));
  for (auto st : ctx->pipe) I8Q_CUDA_TRY(cudaStreamWaitEvent(st, ctx->ev_start, 0));
  const size_t a_row = a_bytes / M, c_row = c_bytes / M;
  const int out_mode = ctx->typeC == I8Q_BF16 ? OUT_BF16 : OUT_F32;
  const int64_t per = (M + nch - 1) / nch;
  for (int i = 0; i < nch; ++i) {
    const int64_t r0 = i * per, rows = std::min<int64_t>(per, M - r0);
    if (rows <= 0) break;
    I8Q_CUDA_TRY(cudaMemcpyAsync(dA + r0 * a_row, static_cast<const uint8_t*>(A_host) + r0 * a_row, rows * a_row,
                                 cudaMemcpyHostToDevice, ctx->pipe[0]));
    I8Q_CUDA_TRY(cudaEventRecord(ctx->ev_in[i], ctx->pipe[0]));
    I8Q_CUDA_TRY(cudaStreamWaitEvent(ctx->pipe[1], ctx->ev_in[i], 0));
    int rc = forward_impl(ctx, dA + r0 * a_row, nullptr, nullptr, dC + r0 * c_row, out_mode, ctx->pipe[1], r0, rows);
    if (rc) {
      cudaStreamSynchronize(ctx->pipe[0]);
      cudaStreamSynchronize(ctx->pipe[1]);
      cudaStreamSynchronize(ctx->pipe[2]);
      return rc;
    }
    I8Q_CUDA_TRY(cudaEventRecord(ctx->ev_out[i], ctx->pipe[1]));
    I8Q_CUDA_TRY(cudaStreamWaitEvent(ctx->pipe[2], ctx->ev_out[i], 0));
    I8Q_CUDA_TRY(cudaMemcpyAsync(static_cast<uint8_t*>(C_host) + r0 * c_row, dC + r0 * c_row, rows * c_row,
                                 cudaMemcpyDeviceToHost, ctx->pipe[2]));
  }
  I8Q_CUDA_TRY(cudaStreamSynchronize(ctx->pipe[0]));
  I8Q_CUDA_TRY(cudaStreamSynchronize(ctx->pipe[1]));
  I8Q_CUDA_TRY(cudaStreamSynchronize(ctx->pipe[2]));
  return I8Q_OK;
}

extern "C" int i8q_qgemm_dyn_buf_views(i8q_qgemm_ctx* ctx, void* buf, uint8_t** uA, size_t* lda, float** scaleA,
                                       int32_t** zeroA) {
  if (!ctx) return fail(I8Q_ERR_NOT_INITIALIZED, "qgemm_dyn_buf_views: no context");
  uint8_t* base = static_cast<uint8_t*>(buf ? buf : ctx->fallback);
  const BufLayout L = buf_layout(ctx);
  if (uA) *uA = base + L.uA;
  if (lda) *lda = (size_t)ctx->Kp;
  if (scaleA) *scaleA = reinterpret_cast<float*>(base + L.scaleA);
  if (zeroA) *zeroA = reinterpret_cast<int32_t*>(base + L.zeroA);
  return I8Q_OK;
}

extern "C" int i8q_qgemm_dyn_weight_views(i8q_qgemm_ctx* ctx, void* buf, int8_t** iBt, void** iBt_bf16, size_t* ldb,
                                          float** scaleB, int32_t** colsum) {
  if (!ctx) return fail(I8Q_ERR_NOT_INITIALIZED, "qgemm_dyn_weight_views: no context");
  if (ldb) *ldb = (size_t)ctx->Kp;
  if (ctx->constB) {
    if (iBt) *iBt = ctx->iBt;
    if (iBt_bf16) *iBt_bf16 = ctx->iBt_bf16;
    if (scaleB) *scaleB = ctx->scaleB;
    if (colsum) *colsum = ctx->colsum;
    return I8Q_OK;
  }
  // B quantized by the last Forward into buf: the tensor-core product
  // writes only the bf16 codes, the other cores only the int8 ones
  uint8_t* base = static_cast<uint8_t*>(buf ? buf : ctx->fallback);
  if (!base) return fail(I8Q_ERR_INVALID_ARG, "qgemm_dyn_weight_views: no buffer");
  const BufLayout L = buf_layout(ctx);
  if (iBt) *iBt = ctx->use_tc ? nullptr : reinterpret_cast<int8_t*>(base + L.iBt);
  if (iBt_bf16) *iBt_bf16 = ctx->use_tc ? base + L.iBt_bf16 : nullptr;
  if (scaleB) *scaleB = reinterpret_cast<float*>(base + L.scaleB);
  if (colsum) *colsum = reinterpret_cast<int32_t*>(base + L.colsum);
  return I8Q_OK;
}

extern "C" void i8q_qgemm_dyn_clear(i8q_qgemm_ctx** ctx) {
  if (!ctx || !*ctx) return;
  i8q_qgemm_ctx* c = *ctx;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(c->device);
  cudaDeviceSynchronize();
  free_ctx_buffers(c);
  cudaSetDevice(prev);
  delete c;
  *ctx = nullptr;
}
