/*
 * csa.h -- C ABI of libcsa_b300.so: the forward pass of Compressed Sparse
 * Attention (CSA) and Heavily Compressed Attention (HCA) on one B300 (sm_103a).
 *
 * Sources (page title, section):
 *   [csdn]   "一文搞懂 DeepSeek：从 V3 的 KV 压缩与 MoE，到 V4 的百万 token 上下文",
 *            section "V4 改进一：CSA 与 HCA" (the whole pipeline); section
 *            "V3 看家本领一：MLA" (latent + decoupled RoPE key row layout).
 *   [yudong] "DeepSeek-V4 详解", section 2.2 Steps 1-4 (CSA) and section 2.3
 *            Steps 1-2 (HCA).
 *   [jaylab] "DeepSeek-V4 — 百万 Token 上下文的高效 MoE 模型", section
 *            "其他技术细节" (the bullet on the mixed BF16 / FP8 KV cache).
 *
 * Conventions shared by every call
 * --------------------------------
 * Memory.   Every tensor argument is a DEVICE pointer owned by the caller.
 *           The library never allocates, frees or synchronises; scratch
 *           memory is a caller-provided workspace sized by
 *           csa_workspace_size().  Tensors are dense, row-major, with the
 *           shapes given below (batch outermost).
 * Streams.  All work is enqueued on `stream` (0 = legacy default stream).
 * Positions. Query i of every sequence sits at absolute token position
 *           q_pos0 + i.  Entry s (s >= 0) pools tokens s*m .. s*m+m-1 and is
 *           visible to the query at position t iff (s+1)*m - 1 <= t, i.e.
 *           s < n_vis(t) = (t+1)/m (integer division).  The raw window of t
 *           is tokens max(0, t-W+1) .. t, t included.
 * Status.   Every call returns CSA_OK (0) or a negative csa_status; on error
 *           nothing is launched and no output is touched, and
 *           csa_last_error() returns a message for the calling thread.
 *           Device-side faults are not caught here; they surface as CUDA
 *           errors on the stream.
 * Alignment. Every device pointer must be 16-byte aligned
 *           (CSA_ERR_ALIGNMENT otherwise).
 * Reentrancy. Calls keep no state between invocations (apart from the
 *           thread-local error message) and may be issued from several host
 *           threads; two calls that write the same buffer race.
 * Determinism. For fixed inputs every output is bitwise reproducible and
 *           independent of the batch size and of the slot a sequence takes
 *           in the batch ([csdn] section "V4 的其他升级", the bullet on
 *           deterministic kernels).
 */
#ifndef CSA_B300_H
#define CSA_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* csa_stream_t; /* == cudaStream_t */

typedef enum {
  CSA_F32 = 0,  /* IEEE binary32 */
  CSA_BF16 = 1, /* bfloat16 */
  CSA_E4M3 = 2, /* OCP FP8 E4M3 ("fn": no inf, NaN = 0x7f/0xff) with fp32 row scales */
  CSA_E2M1 = 3  /* OCP FP4 E2M1 (values 0, 0.5, 1, 1.5, 2, 3, 4, 6 and negatives), two codes per
                   byte, with fp32 row scales: indexer keys only */
} csa_dtype;

typedef enum {
  CSA_OK = 0,
  CSA_ERR_INVALID_ARG = -1, /* null pointer, bad shape, inconsistent positions */
  CSA_ERR_UNSUPPORTED = -2, /* dtype / shape combination without a kernel */
  CSA_ERR_ALIGNMENT = -3,   /* a pointer is not 16-byte aligned */
  CSA_ERR_WORKSPACE = -4,   /* workspace missing or smaller than required */
  CSA_ERR_CUDA = -5,        /* a launch failed (message holds the CUDA error) */
  CSA_ERR_TIMEOUT = -6      /* a bounded device-side wait gave up */
} csa_status;

/*
 * A block of rows (compressed entries, raw tokens or indexer keys), one
 * sequence after the other: row r of sequence b is element [b, r].
 *   dtype F32 / BF16: `data` is [B, n_rows, width]; rope, scale unused (NULL).
 *   dtype E4M3 (mixed layout, [jaylab] "其他技术细节"): the first `nope`
 *       channels of each row are e4m3 codes in `data` [B, n_rows, nope] with
 *       one fp32 scale per row in `scale` [B, n_rows] (value = code * scale);
 *       the remaining width - nope channels (the RoPE dims) are bfloat16 in
 *       `rope` [B, n_rows, width - nope] (NULL when nope == width).
 *   dtype E2M1 (FP4 indexer keys, [csdn] section "V4 的其他升级": the
 *       indexer's QK path in FP4, turned into FP8 without loss): `data` is
 *       [B, n_rows, width / 2] bytes, channel 2i in the low and channel 2i + 1
 *       in the high four bits of byte i; one fp32 scale per row in `scale`
 *       (value = code * scale); width even, nope == width, rope NULL.  Accepted
 *       as the key cache of csa_index / csa_index_ex / csa_forward (with E4M3
 *       q_idx) and as the output of csa_compress.
 */
typedef struct {
  csa_dtype dtype;
  void* data;
  void* rope;
  float* scale;
  int64_t n_rows; /* rows per sequence (the batch stride) */
  int width;      /* channels per row */
  int nope;       /* E4M3 only: channels stored as e4m3 (<= width) */
} csa_rows;

/* Model constants of one CSA / HCA layer. */
typedef struct {
  int B;      /* sequences in the batch */
  int m;      /* block size: 4 for CSA, 128 for HCA ([yudong] 2.2 / 2.3 Step 1) */
  int H;      /* query heads sharing one KV (MQA), e.g. 128 */
  int D_qk;   /* key / query width: latent + rope, e.g. 512 + 64 = 576 */
  int D_v;    /* value width: the leading D_v channels of a key row, e.g. 512 */
  int H_I;    /* indexer heads, e.g. 64 */
  int d_I;    /* indexer width, e.g. 128 */
  int k;      /* entries kept per query (top-k), e.g. 1024 */
  int window; /* raw window W, e.g. 128 */
  float scale;/* softmax scale applied to q.k, e.g. 1/sqrt(576) */
} csa_params;

/*
 * csa_compress -- pool every m adjacent raw rows into one entry
 * ([csdn] section "V4 改进一：CSA 与 HCA", first CSA step; [yudong] 2.2
 * Step 1, 2.3 Step 1):
 *   E[b,s,c] = sum_{i<m} softmax_i(gate[b,sm+i,c] + bias[i,c]) * x[b,sm+i,c]
 * (softmax over the m positions, separately for every channel c).
 *
 *   x, gate   [B, T, C] raw rows and gate logits, dtype `in_dtype` (F32 or
 *             BF16), row j holding token position x_pos0 + j.
 *   bias      [m, C] fp32 learned position bias.
 *   s_begin, s_end  entries to produce, per sequence; every token they pool
 *             must lie in [x_pos0, x_pos0 + T).
 *   out       entry rows, width C, n_rows >= s_end; entry s goes to row s.
 *             F32 out: fp32 arithmetic.  BF16 out: the bfloat16 value nearest
 *             to the exact result (fp32 arithmetic with a float64 recompute of
 *             the elements whose fp32 result lies too close to a rounding
 *             boundary to decide it).  E4M3 out: mixed layout, computed in
 *             float64; scale = fp32(amax over the nope channels / 448) (1 for
 *             an all-zero row); code = e4m3 round-to-nearest-even (saturating)
 *             of value / scale; rope channels rounded to bfloat16.
 * Errors: INVALID_ARG (null pointer, m < 1, C < 1, s_end > out->n_rows,
 * tokens outside x), UNSUPPORTED (in_dtype not F32/BF16), ALIGNMENT.
 */
int csa_compress(const void* x, const void* gate, csa_dtype in_dtype, const float* bias,
                 int B, int64_t x_pos0, int64_t T, int m, int C, int64_t s_begin,
                 int64_t s_end, const csa_rows* out, csa_stream_t stream);

/*
 * csa_index -- lightning indexer scores ([csdn] section "V4 改进一：CSA 与
 * HCA", second CSA step; [yudong] 2.2 Step 2):
 *   I[b,i,s] = sum_{j<H_I} w[b,i,j] * max(0, q_idx[b,i,j,:] . keys[b,s,:])
 * for s < min(N, n_vis(q_pos0+i)); -inf for every other s < N.
 *
 *   q_idx     [B, Q, H_I, d_I], dtype `q_dtype` (F32, BF16 or E4M3); for
 *             E4M3 `q_scale` [B, Q, H_I] fp32 row scales, else NULL.
 *   w         [B, Q, H_I] fp32 per-head weights.
 *   keys      indexer-key rows, width d_I (F32, BF16, or E4M3 with nope ==
 *             d_I and a row scale); n_rows >= N.
 *   scores    [B, Q, N] fp32 output.
 * The products are accumulated in fp32 (tensor cores for BF16 / E4M3 with
 * d_I a multiple of 64 and H_I a multiple of 16 up to 256, CUDA cores
 * otherwise); e4m3 scales multiply the fp32 dot products.
 * Errors: INVALID_ARG, UNSUPPORTED (q_dtype != keys dtype class), ALIGNMENT.
 */
int csa_index(const csa_params* p, const void* q_idx, csa_dtype q_dtype, const float* q_scale,
              const float* w, const csa_rows* keys, int64_t q_pos0, int Q, int64_t N,
              float* scores, csa_stream_t stream);

/*
 * csa_index_ex -- csa_index with the scores stored in `scores_dtype`:
 * CSA_F32 (as csa_index) or CSA_BF16 ([csdn] section "V4 的其他升级": the
 * index scores drop to BF16, which doubles the speed of the top-k).  BF16
 * scores are the fp32 scores rounded to the nearest bf16 (ties to even);
 * invisible entries hold -inf.  `scores` is [B, Q, N] of that dtype.
 * Errors: as csa_index; CSA_ERR_UNSUPPORTED for another scores_dtype.
 */
int csa_index_ex(const csa_params* p, const void* q_idx, csa_dtype q_dtype, const float* q_scale,
                 const float* w, const csa_rows* keys, int64_t q_pos0, int Q, int64_t N,
                 void* scores, csa_dtype scores_dtype, csa_stream_t stream);

/*
 * csa_topk -- keep the best entries per query ([csdn] section "V4 改进一：CSA
 * 与 HCA", second CSA step; [yudong] 2.2 Step 3):
 *   idx[b,i,:] = the min(k, n_vis) indices s < n_vis = min(N, n_vis(q_pos0+i))
 *   with the largest scores[b,i,s], ascending, then -1 up to k.
 * Ties go to the lower index; -0.0 and +0.0 are equal.  Scores must not be
 * NaN.  The selection is exact: no score is rounded.
 *   scores    [B, Q, N] fp32 (as written by csa_index).
 *   idx       [B, Q, k] int32 output.
 *   ws        workspace of at least csa_workspace_size(p, CSA_WS_TOPK, Q, N)
 *             bytes (may be NULL when that size is 0).
 */
int csa_topk(const csa_params* p, const float* scores, int64_t q_pos0, int Q, int64_t N,
             int32_t* idx, void* ws, size_t ws_bytes, csa_stream_t stream);

/*
 * csa_topk_ex -- csa_topk over scores of dtype `scores_dtype` (CSA_F32 or
 * CSA_BF16, as written by csa_index_ex).  BF16 scores tie far more often;
 * ties still go to the lower index.  Same workspace as csa_topk.
 * Errors: as csa_topk; CSA_ERR_UNSUPPORTED for another scores_dtype.
 */
int csa_topk_ex(const csa_params* p, const void* scores, csa_dtype scores_dtype, int64_t q_pos0,
                int Q, int64_t N, int32_t* idx, void* ws, size_t ws_bytes, csa_stream_t stream);

/*
 * csa_topk_noalloc -- csa_topk for callers that cannot allocate device memory
 * at the point of the call (for instance code inside a host framework that
 * owns every device allocation, or a path that must not call cudaMalloc
 * because it can synchronise the device).  The pages have no counterpart of
 * this call: it is a convenience of this library.
 *
 * Same arguments, results and errors as csa_topk, without the workspace: the
 * scratch lives in one static device array of CSA_TOPK_NOALLOC_MAX_BYTES
 * inside the library, which every GPU that loads the library holds until the
 * process exits.  The call allocates and frees nothing.
 *   - Sizes whose scratch (csa_workspace_size(p, CSA_WS_TOPK, Q, N)) exceeds
 *     CSA_TOPK_NOALLOC_MAX_BYTES are rejected with CSA_ERR_WORKSPACE.
 *   - The first call on a device looks up the array's device address on that
 *     device (it must be the current device) and keeps it for the life of
 *     the process; make that first call before any stream capture.  The
 *     kept address assumes the device's primary context: after
 *     cudaDeviceReset, or with another driver-API context made current, the
 *     library's module may sit at another address, and this call must not
 *     be used.
 *   - All calls share the one array.  Each call writes every scratch byte it
 *     later reads before reading it, so nothing carries over from an earlier
 *     call; but calls that overlap on the GPU (other streams, other host
 *     threads) race on the array: serialise them.
 */
#define CSA_TOPK_NOALLOC_MAX_BYTES (16u << 20)

int csa_topk_noalloc(const csa_params* p, const float* scores, int64_t q_pos0, int Q, int64_t N,
                     int32_t* idx, csa_stream_t stream);

/*
 * csa_attend -- shared-KV (MQA) attention of every query head over the
 * selected entries plus the raw window ([csdn] section "V4 改进一：CSA 与
 * HCA": recent raw KV in a sliding window, one KV shared by all heads;
 * [yudong] 2.2 Step 4):
 *   keys K = { kv[b,s] : s in idx[b,i,:], s >= 0 } ++ { raw token u in window(t) }
 *   out[b,i,h,:] = sum_j softmax_j(scale * q[b,i,h,:] . K_j) * K_j[0:D_v]
 * (the value is the leading D_v channels of the key row: the latent of
 * [csdn] MLA; the RoPE channels only enter the score).  A window token is a
 * key of its own even when a selected entry covers it.  No keys -> zeros.
 *
 *   q         [B, Q, H, D_qk], dtype `q_dtype` (F32 or BF16).
 *   kv        entry rows, width D_qk (F32, BF16, or E4M3 with nope == D_v).
 *   raw       raw-token rows, width D_qk, row j = position raw_pos0 + j, F32 or
 *             BF16; must hold the window of every query.
 *   idx       [B, Q, k] int32 as written by csa_topk (indices < N or -1).
 *   out       [B, Q, H, D_v], dtype `out_dtype` (F32 or BF16; fp32 accumulate,
 *             one rounding at the end).
 *   ws        at least csa_workspace_size(p, CSA_WS_ATTEND, Q, N) bytes.
 */
int csa_attend(const csa_params* p, const void* q, csa_dtype q_dtype, const csa_rows* kv,
               const csa_rows* raw, int64_t raw_pos0, const int32_t* idx, int64_t q_pos0, int Q,
               int64_t N, void* out, csa_dtype out_dtype, void* ws, size_t ws_bytes,
               csa_stream_t stream);

/*
 * csa_attend_raw -- the raw-token variant of the CSA attention ([yudong] 2.2
 * Steps 3-4: each selected block stands for its m original tokens and the
 * attention runs over those tokens; hongke120.com page, section 2.2, item 3):
 *   keys K = { raw token s*m + r : s in idx[b,i,:], s >= 0, r < m }, block by
 *            block in list order, ++ { raw token u in window(t) }
 *   out[b,i,h,:] = sum_j softmax_j(scale * q[b,i,h,:] . K_j) * K_j[0:D_v]
 * A window token is a key of its own even when a selected block holds it.
 *
 *   q, idx, out, ws  as for csa_attend; ws of at least
 *             csa_workspace_size(p, CSA_WS_ATTEND_RAW, Q, N) bytes.
 *   raw       raw-token rows, width D_qk (F32 or BF16), row j = position
 *             raw_pos0 + j; raw_pos0 must be 0 and the rows must hold every
 *             token of the N blocks (n_rows >= m*N) and every window.
 * Errors: as csa_attend, and INVALID_ARG when the raw rows do not start at
 * position 0 or cannot hold the blocks' tokens.
 */
int csa_attend_raw(const csa_params* p, const void* q, csa_dtype q_dtype, const csa_rows* raw,
                   int64_t raw_pos0, const int32_t* idx, int64_t q_pos0, int Q, int64_t N,
                   void* out, csa_dtype out_dtype, void* ws, size_t ws_bytes,
                   csa_stream_t stream);

/*
 * hca_attend -- HCA dense attention ([csdn] section "V4 改进一：CSA 与 HCA",
 * the HCA paragraph; [yudong] 2.3 Step 2): as csa_attend with the key set every visible entry
 * s < min(N, n_vis(t)) (p->m is the HCA block size, e.g. 128; p->k and the
 * indexer fields are ignored) followed by the raw window.
 */
int hca_attend(const csa_params* p, const void* q, csa_dtype q_dtype, const csa_rows* kv,
               const csa_rows* raw, int64_t raw_pos0, int64_t q_pos0, int Q, int64_t N,
               void* out, csa_dtype out_dtype, void* ws, size_t ws_bytes, csa_stream_t stream);

/*
 * Inputs of the fused CSA forward pass.  Raw rows cover token positions
 * raw_pos0 .. raw_pos0 + R - 1 of every sequence.
 */
typedef struct {
  const void* x;       /* [B, R, D_qk] raw KV rows (also the window keys) */
  const void* gate;    /* [B, R, D_qk] gate logits */
  const float* bias;   /* [m, D_qk] */
  const void* xi;      /* [B, R, d_I] raw indexer-key rows */
  const void* gate_i;  /* [B, R, d_I] */
  const float* bias_i; /* [m, d_I] */
  csa_dtype raw_dtype; /* dtype of x, gate, xi, gate_i (F32 or BF16) */
  int64_t R;
  int64_t raw_pos0;
  const void* q;       /* [B, Q, H, D_qk] */
  csa_dtype q_dtype;
  const void* q_idx;   /* [B, Q, H_I, d_I] */
  csa_dtype q_idx_dtype;
  const float* q_idx_scale; /* [B, Q, H_I] for E4M3, else NULL */
  const float* w;      /* [B, Q, H_I] */
  int64_t q_pos0;
  int Q;
  csa_rows kv;         /* entry cache (in/out): rows n_cached .. N-1 are written */
  csa_rows keys;       /* indexer-key cache (in/out), same rows */
  int64_t n_cached;    /* entries already in both caches */
  void* out;           /* [B, Q, H, D_v] */
  csa_dtype out_dtype;
  /* Raw-token variant (csa_attend_raw): the raw KV rows of positions
   * 0 .. raw_all_rows-1 of every sequence, [B, raw_all_rows, D_qk] in
   * raw_dtype, holding every token of the visible blocks and the windows;
   * the attention then runs over the raw tokens of the selected blocks and
   * reads its window from here.  NULL: the attention runs over the selected
   * entries (csa_attend). */
  const void* raw_all;
  int64_t raw_all_rows;
  /* Dtype of the indexer scores in the workspace: CSA_F32 (0, the default of
   * a zero-initialised struct) or CSA_BF16 (csa_index_ex). */
  csa_dtype score_dtype;
} csa_forward_args;

/*
 * csa_forward -- the whole CSA step ([csdn] V4 改进一; [yudong] 2.2 Steps 1-4):
 *   1. compress entries n_cached .. N-1 (N = n_vis(q_pos0 + Q - 1)) of both
 *      caches from the raw rows (csa_compress);
 *   2. score every visible entry (csa_index);
 *   3. keep the top-k (csa_topk);
 *   4. attend over them plus the window (csa_attend; csa_attend_raw over the
 *      raw tokens of the selected blocks when raw_all is given).
 * The scores and index lists live in the workspace:
 *   ws_bytes >= csa_workspace_size(p, CSA_WS_FORWARD, Q, N).
 */
int csa_forward(const csa_params* p, const csa_forward_args* a, void* ws, size_t ws_bytes,
                csa_stream_t stream);

enum { CSA_WS_TOPK = 0, CSA_WS_ATTEND = 1, CSA_WS_HCA = 2, CSA_WS_FORWARD = 3,
       CSA_WS_ATTEND_RAW = 4 };

/* Workspace bytes needed by the call `which` (CSA_WS_*) for Q queries per
 * sequence over N entries; 0 on invalid arguments. */
size_t csa_workspace_size(const csa_params* p, int which, int Q, int64_t N);

/*
 * csa_device_status -- synchronise `stream` and report whether a bounded
 * device-side wait in a kernel launched since the previous check gave up
 * (CSA_ERR_TIMEOUT; the outputs of those calls are then not valid).  The
 * tensor-core kernels wait on mbarriers for their own TMA copies and MMAs;
 * each wait gives up after 2 s instead of hanging, records the site and lets
 * the kernel exit.  Clears the recorded state.  CSA_OK otherwise.
 */
int csa_device_status(csa_stream_t stream);

/*
 * csa_debug_stall_next -- test aid for the failure path of the bounded
 * device-side waits.  Arms a one-shot: the next launch of the named
 * tensor-core kernel (CSA_STALL_INDEX: the indexer of csa_index /
 * csa_forward; CSA_STALL_ATTEND: the attention of csa_attend / hca_attend /
 * csa_forward) makes its first CTA's MMA issuer wait, while that CTA's first
 * loads are in flight, on a device flag that nothing sets.  The wait gives up
 * after 0.1 s through the same path as any wait that runs out: it records
 * its site, every other wait of the launch gives up, each CTA lets its own
 * copies and MMAs in flight land and exits.  The next csa_device_status then
 * returns CSA_ERR_TIMEOUT; the outputs of that launch are not valid, and the
 * following calls run normally.  Process-wide; 0 disarms.  Not for use in
 * production: it exists so that tests can observe the timeout report.
 * Errors: INVALID_ARG (unknown kernel).
 */
enum { CSA_STALL_INDEX = 1, CSA_STALL_ATTEND = 2 };
int csa_debug_stall_next(int kernel);

/*
 * csa_group_proj -- grouped output projection after the attention ([csdn]
 * section "V4 改进一：CSA 与 HCA", the CSA paragraph's last sentence: the
 * output is projected in groups to save compute).  The H heads form G
 * consecutive groups of H/G heads; group g's head outputs, side by side in a
 * row of o, are projected by that group's own matrix:
 *   y[t, g*d_g + n] = sum_{j < K} o[t, g*K + j] * w[g, n, j],   K = (H/G)*D_v
 *
 *   o   [T, H, D_v] BF16 (the attention output, e.g. csa_attend's `out` with
 *       T = B*Q), row-major, caller-owned device memory.
 *   w   [G, d_g, K] BF16: row n of group g holds column n of the group's
 *       [K, d_g] matrix (both operands K-contiguous).
 *   y   [T, G*d_g], dtype y_dtype (F32 or BF16; fp32 accumulation, one
 *       rounding at the end), written completely.
 * Runs on the tensor cores; needs K a multiple of 64 and d_g a multiple of
 * 256 (else CSA_ERR_UNSUPPORTED), H a multiple of G (CSA_ERR_INVALID_ARG),
 * o / w / y 16-byte aligned (CSA_ERR_ALIGNMENT).  T = 0 does nothing.  Its
 * bounded device waits report through csa_device_status.
 */
int csa_group_proj(const void* o, int64_t T, int H, int D_v, const void* w, int G, int d_g,
                   void* y, csa_dtype y_dtype, csa_stream_t stream);

/* Message describing the last error returned on the calling thread ("" if none). */
const char* csa_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* CSA_B300_H */
