// C entry points of libcsa_b300: argument validation, then kernel launches on
// the caller's stream.  Nothing here computes; every step runs in a kernel.
#include <stdarg.h>
#include <stdio.h>

#include <atomic>
#include <mutex>

#include "common.cuh"

using namespace csa;

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  g_err[0] = '\0';
  return CSA_OK;
}

int cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return ok();
  return fail(CSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define REQUIRE(cond, code, ...) \
  do {                           \
    if (!(cond)) return fail(code, __VA_ARGS__); \
  } while (0)

int check_ptr(const void* p, const char* name) {
  if (!p) return fail(CSA_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned16(p)) return fail(CSA_ERR_ALIGNMENT, "%s is not 16-byte aligned", name);
  return CSA_OK;
}

#define CHECK_PTR(p)                          \
  do {                                        \
    int _r = check_ptr((p), #p);              \
    if (_r != CSA_OK) return _r;              \
  } while (0)

int check_rows(const csa_rows* r, const char* name, int width, int64_t min_rows, bool allow_e4m3,
               int e4m3_nope, bool allow_e2m1) {
  if (!r) return fail(CSA_ERR_INVALID_ARG, "%s is NULL", name);
  if (r->dtype != CSA_F32 && r->dtype != CSA_BF16 && r->dtype != CSA_E4M3 &&
      r->dtype != CSA_E2M1)
    return fail(CSA_ERR_UNSUPPORTED, "%s: unknown dtype %d", name, (int)r->dtype);
  if (r->dtype == CSA_E4M3 && !allow_e4m3)
    return fail(CSA_ERR_UNSUPPORTED, "%s: e4m3 rows are not accepted here", name);
  if (r->dtype == CSA_E2M1) {
    if (!allow_e2m1) return fail(CSA_ERR_UNSUPPORTED, "%s: e2m1 rows are not accepted here", name);
    if (r->width % 2 != 0 || r->nope != r->width)
      return fail(CSA_ERR_INVALID_ARG, "%s: e2m1 rows need an even width and nope == width", name);
    if (!r->scale) return fail(CSA_ERR_INVALID_ARG, "%s.scale is NULL", name);
    if (!aligned16(r->scale)) return fail(CSA_ERR_ALIGNMENT, "%s.scale is not 16-byte aligned", name);
  }
  if (r->width != width)
    return fail(CSA_ERR_INVALID_ARG, "%s: width %d, expected %d", name, r->width, width);
  if (r->n_rows < min_rows)
    return fail(CSA_ERR_INVALID_ARG, "%s: n_rows %lld < %lld needed", name, (long long)r->n_rows,
                (long long)min_rows);
  if (!r->data) return fail(CSA_ERR_INVALID_ARG, "%s.data is NULL", name);
  if (!aligned16(r->data)) return fail(CSA_ERR_ALIGNMENT, "%s.data is not 16-byte aligned", name);
  if (r->dtype == CSA_E4M3) {
    if (e4m3_nope >= 0 && r->nope != e4m3_nope)
      return fail(CSA_ERR_UNSUPPORTED, "%s: e4m3 nope %d, expected %d", name, r->nope, e4m3_nope);
    if (r->nope < 1 || r->nope > r->width)
      return fail(CSA_ERR_INVALID_ARG, "%s: nope %d out of range", name, r->nope);
    if (!r->scale) return fail(CSA_ERR_INVALID_ARG, "%s.scale is NULL", name);
    if (!aligned16(r->scale)) return fail(CSA_ERR_ALIGNMENT, "%s.scale is not 16-byte aligned", name);
    if (r->nope < r->width) {
      if (!r->rope) return fail(CSA_ERR_INVALID_ARG, "%s.rope is NULL", name);
      if (!aligned16(r->rope)) return fail(CSA_ERR_ALIGNMENT, "%s.rope is not 16-byte aligned", name);
    }
  }
  return CSA_OK;
}

#define CHECK(expr)              \
  do {                           \
    int _r = (expr);             \
    if (_r != CSA_OK) return _r; \
  } while (0)

int check_params(const csa_params* p, bool need_index, bool need_topk) {
  if (!p) return fail(CSA_ERR_INVALID_ARG, "params is NULL");
  REQUIRE(p->B >= 1, CSA_ERR_INVALID_ARG, "B = %d < 1", p->B);
  REQUIRE(p->m >= 1, CSA_ERR_INVALID_ARG, "m = %d < 1", p->m);
  REQUIRE(p->window >= 0, CSA_ERR_INVALID_ARG, "window = %d < 0", p->window);
  if (need_index) {
    REQUIRE(p->H_I >= 1 && p->d_I >= 1, CSA_ERR_INVALID_ARG, "H_I = %d, d_I = %d", p->H_I, p->d_I);
    REQUIRE((int64_t)p->H_I * p->d_I <= 32768, CSA_ERR_UNSUPPORTED, "H_I * d_I = %d > 32768",
            p->H_I * p->d_I);
  }
  if (need_topk) REQUIRE(p->k >= 1, CSA_ERR_INVALID_ARG, "k = %d < 1", p->k);
  return CSA_OK;
}

int check_attn_params(const csa_params* p) {
  REQUIRE(p->H >= 1, CSA_ERR_INVALID_ARG, "H = %d < 1", p->H);
  REQUIRE(p->D_qk >= 1 && p->D_qk <= 1024, CSA_ERR_UNSUPPORTED, "D_qk = %d not in [1, 1024]",
          p->D_qk);
  REQUIRE(p->D_v >= 1 && p->D_v <= p->D_qk && p->D_v <= 512, CSA_ERR_UNSUPPORTED,
          "D_v = %d not in [1, min(D_qk, 512)]", p->D_v);
  return CSA_OK;
}

int check_positions(int64_t q_pos0, int Q, int64_t N, int m) {
  REQUIRE(Q >= 0, CSA_ERR_INVALID_ARG, "Q = %d < 0", Q);
  REQUIRE(q_pos0 >= 0, CSA_ERR_INVALID_ARG, "q_pos0 = %lld < 0", (long long)q_pos0);
  REQUIRE(N >= 0, CSA_ERR_INVALID_ARG, "N = %lld < 0", (long long)N);
  (void)m;
  return CSA_OK;
}

int check_window(const csa_params* p, const csa_rows* raw, int64_t raw_pos0, int64_t q_pos0,
                 int Q) {
  if (Q == 0) return CSA_OK;
  int64_t first = q_pos0 - p->window + 1;
  if (first < 0) first = 0;
  const int64_t last = q_pos0 + Q - 1;
  if (p->window == 0) return CSA_OK;
  REQUIRE(first >= raw_pos0 && last < raw_pos0 + raw->n_rows, CSA_ERR_INVALID_ARG,
          "raw rows hold positions [%lld, %lld) but the windows need [%lld, %lld]",
          (long long)raw_pos0, (long long)(raw_pos0 + raw->n_rows), (long long)first,
          (long long)last);
  return CSA_OK;
}

std::atomic<int> g_stall_next{0};

}  // namespace

namespace csa {
bool take_debug_stall(int kernel) {
  int want = kernel;
  return g_stall_next.compare_exchange_strong(want, 0);
}
}  // namespace csa

extern "C" {

const char* csa_last_error(void) { return g_err; }

int csa_debug_stall_next(int kernel) {
  REQUIRE(kernel == 0 || kernel == CSA_STALL_INDEX || kernel == CSA_STALL_ATTEND,
          CSA_ERR_INVALID_ARG, "unknown kernel %d", kernel);
  g_stall_next.store(kernel);
  return ok();
}

int csa_device_status(csa_stream_t stream) {
  int code = 0, code2 = 0;
  cudaError_t e = index_tc_status(&code, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_status(e, "csa_device_status");
  e = attend_tc_status(&code2, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_status(e, "csa_device_status");
  if (code == 0) code = code2;
  e = gproj_status(&code2, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_status(e, "csa_device_status");
  if (code == 0) code = code2;
  if (code != 0)
    return fail(CSA_ERR_TIMEOUT, "a bounded device-side wait gave up (site %d); the outputs of the "
                                 "calls since the last check are not valid", code);
  return ok();
}

int csa_compress(const void* x, const void* gate, csa_dtype in_dtype, const float* bias, int B,
                 int64_t x_pos0, int64_t T, int m, int C, int64_t s_begin, int64_t s_end,
                 const csa_rows* out, csa_stream_t stream) {
  REQUIRE(in_dtype == CSA_F32 || in_dtype == CSA_BF16, CSA_ERR_UNSUPPORTED,
          "in_dtype must be F32 or BF16");
  REQUIRE(B >= 1 && m >= 1 && C >= 1 && T >= 0, CSA_ERR_INVALID_ARG,
          "bad sizes B=%d m=%d C=%d T=%lld", B, m, C, (long long)T);
  REQUIRE(s_begin >= 0 && s_end >= s_begin, CSA_ERR_INVALID_ARG, "bad entry range [%lld, %lld)",
          (long long)s_begin, (long long)s_end);
  REQUIRE(x_pos0 >= 0, CSA_ERR_INVALID_ARG, "x_pos0 < 0");
  CHECK(check_rows(out, "out", C, s_end, true, -1, true));
  if (s_end > s_begin) {
    CHECK_PTR(x);
    CHECK_PTR(gate);
    CHECK_PTR(bias);
    REQUIRE(s_begin * m >= x_pos0 && s_end * m <= x_pos0 + T, CSA_ERR_INVALID_ARG,
            "entries [%lld, %lld) pool tokens outside the rows given [%lld, %lld)",
            (long long)s_begin, (long long)s_end, (long long)x_pos0, (long long)(x_pos0 + T));
  }
  return cuda_status(launch_compress(x, gate, in_dtype, bias, B, x_pos0, T, m, C, s_begin, s_end,
                                     *out, (cudaStream_t)stream),
                     "csa_compress");
}

int csa_index(const csa_params* p, const void* q_idx, csa_dtype q_dtype, const float* q_scale,
              const float* w, const csa_rows* keys, int64_t q_pos0, int Q, int64_t N,
              float* scores, csa_stream_t stream) {
  return csa_index_ex(p, q_idx, q_dtype, q_scale, w, keys, q_pos0, Q, N, scores, CSA_F32, stream);
}

int csa_index_ex(const csa_params* p, const void* q_idx, csa_dtype q_dtype, const float* q_scale,
                 const float* w, const csa_rows* keys, int64_t q_pos0, int Q, int64_t N,
                 void* scores, csa_dtype scores_dtype, csa_stream_t stream) {
  REQUIRE(scores_dtype == CSA_F32 || scores_dtype == CSA_BF16, CSA_ERR_UNSUPPORTED,
          "scores must be F32 or BF16");
  CHECK(check_params(p, true, false));
  CHECK(check_positions(q_pos0, Q, N, p->m));
  CHECK(check_rows(keys, "keys", p->d_I, N, true, p->d_I, true));
  REQUIRE(q_dtype == CSA_F32 || q_dtype == CSA_BF16 || q_dtype == CSA_E4M3, CSA_ERR_UNSUPPORTED,
          "unknown q_dtype");
  REQUIRE((q_dtype == CSA_E4M3) == (keys->dtype == CSA_E4M3 || keys->dtype == CSA_E2M1),
          CSA_ERR_UNSUPPORTED, "q_idx must be e4m3 exactly when the keys are e4m3 or e2m1");
  if (Q == 0 || N == 0) return ok();
  CHECK_PTR(q_idx);
  CHECK_PTR(w);
  CHECK_PTR(scores);
  if (q_dtype == CSA_E4M3) CHECK_PTR(q_scale);
  return cuda_status(launch_index(*p, q_idx, q_dtype, q_scale, w, *keys, q_pos0, Q, N, scores,
                                  scores_dtype == CSA_BF16, (cudaStream_t)stream),
                     "csa_index");
}

int csa_topk(const csa_params* p, const float* scores, int64_t q_pos0, int Q, int64_t N,
             int32_t* idx, void* ws, size_t ws_bytes, csa_stream_t stream) {
  return csa_topk_ex(p, scores, CSA_F32, q_pos0, Q, N, idx, ws, ws_bytes, stream);
}

int csa_topk_ex(const csa_params* p, const void* scores, csa_dtype scores_dtype, int64_t q_pos0,
                int Q, int64_t N, int32_t* idx, void* ws, size_t ws_bytes, csa_stream_t stream) {
  REQUIRE(scores_dtype == CSA_F32 || scores_dtype == CSA_BF16, CSA_ERR_UNSUPPORTED,
          "scores must be F32 or BF16");
  CHECK(check_params(p, false, true));
  CHECK(check_positions(q_pos0, Q, N, p->m));
  if (Q == 0) return ok();
  CHECK_PTR(idx);
  if (N > 0) CHECK_PTR(scores);
  REQUIRE(N <= 0x7fffffffLL, CSA_ERR_UNSUPPORTED, "N too large for int32 indices");
  const size_t need = topk_workspace(*p, Q, N);
  if (need) {
    REQUIRE(ws && ws_bytes >= need, CSA_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, need);
    REQUIRE(aligned16(ws), CSA_ERR_ALIGNMENT, "workspace is not 16-byte aligned");
  }
  return cuda_status(launch_topk(*p, scores, scores_dtype == CSA_BF16, q_pos0, Q, N, idx, ws,
                                 (cudaStream_t)stream),
                     "csa_topk");
}

// ---------------------------------------------------------------------------
// csa_topk_noalloc: csa_topk with its scratch in a fixed buffer of this
// library instead of a caller workspace.  It is meant for callers that cannot
// obtain device memory at the point of the call: code embedded in a host
// framework that owns every device allocation, or paths that must not call
// cudaMalloc because it can synchronise the device.  The buffer is a
// file-scope device array, so every GPU that loads the library holds it
// until the process exits.  Host code only sees a host-side stand-in for
// the array's name, so its device address is looked up once per device, with
// that device current, and handed to the kernels.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_topk_noalloc_scratch[CSA_TOPK_NOALLOC_MAX_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up on
// the first call per device).
int noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e, "csa_topk_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return fail(CSA_ERR_UNSUPPORTED, "csa_topk_noalloc: device %d beyond %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_topk_noalloc_scratch);
    if (e != cudaSuccess) return cuda_status(e, "csa_topk_noalloc: cudaGetSymbolAddress");
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return CSA_OK;
}

}  // namespace

extern "C" int csa_topk_noalloc(const csa_params* p, const float* scores, int64_t q_pos0, int Q,
                                int64_t N, int32_t* idx, csa_stream_t stream) {
  CHECK(check_params(p, false, true));
  CHECK(check_positions(q_pos0, Q, N, p->m));
  if (Q == 0) return ok();
  CHECK_PTR(idx);
  if (N > 0) CHECK_PTR(scores);
  REQUIRE(N <= 0x7fffffffLL, CSA_ERR_UNSUPPORTED, "N too large for int32 indices");
  const size_t need = topk_workspace(*p, Q, N);
  REQUIRE(need <= (size_t)CSA_TOPK_NOALLOC_MAX_BYTES, CSA_ERR_WORKSPACE,
          "csa_topk_noalloc: these sizes need %zu bytes of scratch, the static buffer holds %zu "
          "(use csa_topk with a workspace)",
          need, (size_t)CSA_TOPK_NOALLOC_MAX_BYTES);
  void* ws = nullptr;
  if (need) CHECK(noalloc_scratch(&ws));
  return cuda_status(launch_topk(*p, scores, false, q_pos0, Q, N, idx, ws, (cudaStream_t)stream),
                     "csa_topk_noalloc");
}

// The raw rows of the raw-token variant must hold every token a selected
// block can cover (positions 0 .. m*N-1) besides the windows.
static int check_raw_blocks(const csa_params* p, const csa_rows* raw, int64_t raw_pos0, int64_t N) {
  REQUIRE(raw_pos0 == 0, CSA_ERR_INVALID_ARG,
          "raw-token attention: raw rows must start at position 0 (raw_pos0 = %lld)",
          (long long)raw_pos0);
  REQUIRE(raw->n_rows >= N * p->m, CSA_ERR_INVALID_ARG,
          "raw-token attention: %lld raw rows cannot hold the tokens of %lld blocks of %d",
          (long long)raw->n_rows, (long long)N, p->m);
  return CSA_OK;
}

static int attend_common(const csa_params* p, const void* q, csa_dtype q_dtype, const csa_rows* kv,
                         const csa_rows* raw, int64_t raw_pos0, const int32_t* idx, int mode,
                         int64_t q_pos0, int Q, int64_t N, void* out, csa_dtype out_dtype, void* ws,
                         size_t ws_bytes, cudaStream_t st, const char* name) {
  CHECK(check_params(p, false, mode != kAttendDense));
  CHECK(check_attn_params(p));
  CHECK(check_positions(q_pos0, Q, N, p->m));
  REQUIRE(q_dtype == CSA_F32 || q_dtype == CSA_BF16, CSA_ERR_UNSUPPORTED, "q must be F32 or BF16");
  REQUIRE(out_dtype == CSA_F32 || out_dtype == CSA_BF16, CSA_ERR_UNSUPPORTED,
          "out must be F32 or BF16");
  if (mode != kAttendRawBlocks) CHECK(check_rows(kv, "kv", p->D_qk, N, true, p->D_v, false));
  if (p->window > 0 || mode == kAttendRawBlocks) {
    CHECK(check_rows(raw, "raw", p->D_qk, 0, false, -1, false));
    REQUIRE(raw_pos0 >= 0, CSA_ERR_INVALID_ARG, "raw_pos0 < 0");
    CHECK(check_window(p, raw, raw_pos0, q_pos0, Q));
  }
  if (mode == kAttendRawBlocks) CHECK(check_raw_blocks(p, raw, raw_pos0, N));
  if (Q == 0) return ok();
  CHECK_PTR(q);
  CHECK_PTR(out);
  if (mode != kAttendDense) CHECK_PTR(idx);
  const size_t need = attend_workspace(*p, Q, N, mode);
  if (need) {
    REQUIRE(ws && ws_bytes >= need, CSA_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, need);
    REQUIRE(aligned16(ws), CSA_ERR_ALIGNMENT, "workspace is not 16-byte aligned");
  }
  // the kernels take two row blocks: without raw rows they get the entry cache
  // twice, without an entry cache (raw-token variant) the raw rows twice
  const csa_rows& kv_or_raw = mode == kAttendRawBlocks ? *raw : *kv;
  const csa_rows& raw_or_kv = (raw && (p->window > 0 || mode == kAttendRawBlocks)) ? *raw : *kv;
  return cuda_status(launch_attend(*p, q, q_dtype, kv_or_raw, raw_or_kv, raw_pos0, idx, mode, q_pos0,
                                   Q, N, out, out_dtype, ws, st),
                     name);
}

int csa_attend(const csa_params* p, const void* q, csa_dtype q_dtype, const csa_rows* kv,
               const csa_rows* raw, int64_t raw_pos0, const int32_t* idx, int64_t q_pos0, int Q,
               int64_t N, void* out, csa_dtype out_dtype, void* ws, size_t ws_bytes,
               csa_stream_t stream) {
  return attend_common(p, q, q_dtype, kv, raw, raw_pos0, idx, kAttendEntries, q_pos0, Q, N, out,
                       out_dtype, ws, ws_bytes, (cudaStream_t)stream, "csa_attend");
}

int csa_attend_raw(const csa_params* p, const void* q, csa_dtype q_dtype, const csa_rows* raw,
                   int64_t raw_pos0, const int32_t* idx, int64_t q_pos0, int Q, int64_t N,
                   void* out, csa_dtype out_dtype, void* ws, size_t ws_bytes,
                   csa_stream_t stream) {
  return attend_common(p, q, q_dtype, nullptr, raw, raw_pos0, idx, kAttendRawBlocks, q_pos0, Q, N,
                       out, out_dtype, ws, ws_bytes, (cudaStream_t)stream, "csa_attend_raw");
}

int hca_attend(const csa_params* p, const void* q, csa_dtype q_dtype, const csa_rows* kv,
               const csa_rows* raw, int64_t raw_pos0, int64_t q_pos0, int Q, int64_t N, void* out,
               csa_dtype out_dtype, void* ws, size_t ws_bytes, csa_stream_t stream) {
  return attend_common(p, q, q_dtype, kv, raw, raw_pos0, nullptr, kAttendDense, q_pos0, Q, N, out,
                       out_dtype, ws, ws_bytes, (cudaStream_t)stream, "hca_attend");
}

// Workspace layout of csa_forward: [scores B*Q*N fp32][idx B*Q*k int32][max(topk, attend)]
static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t csa_workspace_size(const csa_params* p, int which, int Q, int64_t N) {
  if (!p || Q < 0 || N < 0 || p->B < 1) return 0;
  switch (which) {
    case CSA_WS_TOPK: return topk_workspace(*p, Q, N);
    case CSA_WS_ATTEND: return attend_workspace(*p, Q, N, kAttendEntries);
    case CSA_WS_HCA: return attend_workspace(*p, Q, N, kAttendDense);
    case CSA_WS_ATTEND_RAW: return attend_workspace(*p, Q, N, kAttendRawBlocks);
    case CSA_WS_FORWARD: {
      // either attention of csa_forward (entries, or the raw tokens of the blocks)
      size_t s = align256((size_t)p->B * Q * N * sizeof(float));
      s += align256((size_t)p->B * Q * (size_t)(p->k > 0 ? p->k : 0) * sizeof(int32_t));
      size_t a = topk_workspace(*p, Q, N), b = attend_workspace(*p, Q, N, kAttendEntries);
      const size_t c = attend_workspace(*p, Q, N, kAttendRawBlocks);
      if (c > b) b = c;
      return s + align256(a > b ? a : b);
    }
    default: return 0;
  }
}

int csa_forward(const csa_params* p, const csa_forward_args* a, void* ws, size_t ws_bytes,
                csa_stream_t stream) {
  CHECK(check_params(p, true, true));
  CHECK(check_attn_params(p));
  REQUIRE(a != nullptr, CSA_ERR_INVALID_ARG, "args is NULL");
  CHECK(check_positions(a->q_pos0, a->Q, 0, p->m));
  if (a->Q == 0) return ok();
  const int64_t N = n_vis(a->q_pos0 + a->Q - 1, p->m);
  REQUIRE(a->n_cached >= 0 && a->n_cached <= N, CSA_ERR_INVALID_ARG, "n_cached %lld not in [0, %lld]",
          (long long)a->n_cached, (long long)N);
  REQUIRE(a->raw_dtype == CSA_F32 || a->raw_dtype == CSA_BF16, CSA_ERR_UNSUPPORTED,
          "raw rows must be F32 or BF16");
  csa_rows raw;
  raw.dtype = a->raw_dtype;
  raw.data = const_cast<void*>(a->x);
  raw.rope = nullptr;
  raw.scale = nullptr;
  raw.n_rows = a->R;
  raw.width = p->D_qk;
  raw.nope = p->D_qk;
  const size_t need = csa_workspace_size(p, CSA_WS_FORWARD, a->Q, N);
  REQUIRE(ws && ws_bytes >= need, CSA_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, need);
  REQUIRE(aligned16(ws), CSA_ERR_ALIGNMENT, "workspace is not 16-byte aligned");
  // validate every step before launching the first one
  CHECK(check_rows(&a->kv, "kv", p->D_qk, N, true, p->D_v, false));
  CHECK(check_rows(&a->keys, "keys", p->d_I, N, true, p->d_I, true));
  CHECK(check_rows(&raw, "raw", p->D_qk, 0, false, -1, false));
  // raw-token variant: the attention reads every raw row from raw_all
  csa_rows raw_all = raw;
  const int mode = a->raw_all ? kAttendRawBlocks : kAttendEntries;
  if (a->raw_all) {
    raw_all.data = const_cast<void*>(a->raw_all);
    raw_all.n_rows = a->raw_all_rows;
    CHECK(check_rows(&raw_all, "raw_all", p->D_qk, 0, false, -1, false));
    REQUIRE(raw_all.dtype == CSA_BF16 || raw_all.dtype == CSA_F32, CSA_ERR_UNSUPPORTED,
            "raw_all must be F32 or BF16");
    CHECK(check_window(p, &raw_all, 0, a->q_pos0, a->Q));
    CHECK(check_raw_blocks(p, &raw_all, 0, N));
  } else {
    CHECK(check_window(p, &raw, a->raw_pos0, a->q_pos0, a->Q));
  }
  if (N > a->n_cached) {
    REQUIRE(a->n_cached * p->m >= a->raw_pos0 && N * p->m <= a->raw_pos0 + a->R, CSA_ERR_INVALID_ARG,
            "entries [%lld, %lld) pool tokens outside the raw rows [%lld, %lld)",
            (long long)a->n_cached, (long long)N, (long long)a->raw_pos0,
            (long long)(a->raw_pos0 + a->R));
    CHECK_PTR(a->x);
    CHECK_PTR(a->gate);
    CHECK_PTR(a->bias);
    CHECK_PTR(a->xi);
    CHECK_PTR(a->gate_i);
    CHECK_PTR(a->bias_i);
  }
  CHECK_PTR(a->q);
  CHECK_PTR(a->q_idx);
  CHECK_PTR(a->w);
  CHECK_PTR(a->out);
  REQUIRE(a->q_dtype == CSA_F32 || a->q_dtype == CSA_BF16, CSA_ERR_UNSUPPORTED,
          "q must be F32 or BF16");
  REQUIRE(a->out_dtype == CSA_F32 || a->out_dtype == CSA_BF16, CSA_ERR_UNSUPPORTED,
          "out must be F32 or BF16");
  REQUIRE((a->q_idx_dtype == CSA_E4M3) ==
              (a->keys.dtype == CSA_E4M3 || a->keys.dtype == CSA_E2M1),
          CSA_ERR_UNSUPPORTED, "q_idx must be e4m3 exactly when the keys are e4m3 or e2m1");
  if (a->q_idx_dtype == CSA_E4M3) CHECK_PTR(a->q_idx_scale);
  REQUIRE(a->score_dtype == CSA_F32 || a->score_dtype == CSA_BF16, CSA_ERR_UNSUPPORTED,
          "score_dtype must be F32 or BF16");
  const bool bf16_scores = a->score_dtype == CSA_BF16;

  cudaStream_t st = (cudaStream_t)stream;
  char* w8 = reinterpret_cast<char*>(ws);
  void* scores = w8;  // fp32 or bf16; the region is sized for fp32
  w8 += align256((size_t)p->B * a->Q * N * sizeof(float));
  int32_t* idx = reinterpret_cast<int32_t*>(w8);
  w8 += align256((size_t)p->B * a->Q * (size_t)p->k * sizeof(int32_t));
  void* rest = w8;

  cudaError_t e;
  if (N > a->n_cached) {
    e = launch_compress_pair(a->x, a->gate, a->bias, p->D_qk, a->kv, a->xi, a->gate_i, a->bias_i,
                             p->d_I, a->keys, a->raw_dtype, p->B, a->raw_pos0, a->R, p->m,
                             a->n_cached, N, st);
    if (e != cudaSuccess) return cuda_status(e, "csa_forward/compress");
  }
  e = launch_index(*p, a->q_idx, a->q_idx_dtype, a->q_idx_scale, a->w, a->keys, a->q_pos0, a->Q, N,
                   scores, bf16_scores, st, /*fill_invisible=*/false);
  if (e != cudaSuccess) return cuda_status(e, "csa_forward/index");
  e = launch_topk(*p, scores, bf16_scores, a->q_pos0, a->Q, N, idx, rest, st);
  if (e != cudaSuccess) return cuda_status(e, "csa_forward/topk");
  if (mode == kAttendRawBlocks)
    e = launch_attend(*p, a->q, a->q_dtype, raw_all, raw_all, 0, idx, mode, a->q_pos0, a->Q, N,
                      a->out, a->out_dtype, rest, st);
  else
    e = launch_attend(*p, a->q, a->q_dtype, a->kv, raw, a->raw_pos0, idx, mode, a->q_pos0, a->Q, N,
                      a->out, a->out_dtype, rest, st);
  return cuda_status(e, "csa_forward/attend");
}

}  // extern "C"

extern "C" int csa_group_proj(const void* o, int64_t T, int H, int D_v, const void* w, int G,
                              int d_g, void* y, csa_dtype y_dtype, csa_stream_t stream) {
  REQUIRE(T >= 0 && H >= 1 && D_v >= 1 && G >= 1 && d_g >= 1, CSA_ERR_INVALID_ARG,
          "bad sizes T=%lld H=%d D_v=%d G=%d d_g=%d", (long long)T, H, D_v, G, d_g);
  REQUIRE(H % G == 0, CSA_ERR_INVALID_ARG, "H = %d is not a multiple of G = %d", H, G);
  REQUIRE(y_dtype == CSA_F32 || y_dtype == CSA_BF16, CSA_ERR_UNSUPPORTED, "y must be F32 or BF16");
  const int64_t K = (int64_t)(H / G) * D_v;
  REQUIRE(K % 64 == 0 && K <= (1 << 30), CSA_ERR_UNSUPPORTED,
          "group width (H/G)*D_v = %lld is not a multiple of 64", (long long)K);
  REQUIRE(d_g % 256 == 0, CSA_ERR_UNSUPPORTED, "d_g = %d is not a multiple of 256", d_g);
  REQUIRE(T < (1ll << 31) && (int64_t)G * d_g < (1ll << 31), CSA_ERR_UNSUPPORTED, "sizes too large");
  if (T == 0) return ok();
  CHECK_PTR(o);
  CHECK_PTR(w);
  CHECK_PTR(y);
  REQUIRE(aligned16(o) && aligned16(w) && aligned16(y), CSA_ERR_ALIGNMENT,
          "o, w and y must be 16-byte aligned");
  return cuda_status(launch_group_proj(o, T, H, D_v, w, G, d_g, y, y_dtype == CSA_F32,
                                       (cudaStream_t)stream),
                     "csa_group_proj");
}
