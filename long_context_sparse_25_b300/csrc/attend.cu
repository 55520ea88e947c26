// Step 4 of CSA (and HCA's dense attention): shared-KV MQA over a key list of
// compressed entries followed by the raw window, with an online softmax.
//
//   o[b,i,h,:] = sum_j softmax_j(scale * q[b,i,h,:] . K_j) * K_j[0:D_v]
//
// Sources: "一文搞懂 DeepSeek：从 V3 的 KV 压缩与 MoE，到 V4 的百万 token 上下文",
// section "V4 改进一：CSA 与 HCA" (sliding window of raw KV; MQA with one shared
// KV; HCA attends densely) and section "V3 看家本领一：MLA" (values come from
// the latent, the decoupled RoPE key only enters the score);
// "DeepSeek-V4 详解" section 2.2 Step 4 and 2.3 Step 2.
//
// This is the CUDA-core path (fp32 arithmetic): the fp32 workloads, whose
// 1e-4 bound rules out bf16 operands, and shapes the tensor-core path
// (attend_tc.cu) does not take.  A CTA
// takes 16 heads of one query and one split of its key list; keys are staged
// in shared memory in tiles of 32 rows converted to fp32.  Splits of the key
// list are fixed by the key-list length alone (never by the batch), and their
// partial (max, sum, o) are merged in split order by a combine kernel, so the
// result does not depend on the batch a sequence runs in.
#include "common.cuh"

namespace csa {

bool attend_tc_supported(const csa_params& p, csa_dtype q_dtype, const csa_rows& kv,
                         const csa_rows& raw, int Q, int64_t N, csa_dtype out_dtype, int mode);
size_t attend_tc_workspace(const csa_params& p, int Q, int64_t N, int mode, int64_t q_pos0);
cudaError_t launch_attend_tc(const csa_params& p, const void* q, const csa_rows& kv,
                             const csa_rows& raw, int64_t raw_pos0, const int32_t* idx, int mode,
                             int64_t q_pos0, int Q, int64_t N, void* out, csa_dtype out_dtype,
                             void* ws, cudaStream_t st);

namespace {

constexpr int kHG = 16;       // heads per CTA
constexpr int kKT = 32;       // keys per tile
constexpr int kThreads = 256;
constexpr int kMaxDvPerThread = 32;  // D_v <= 512

// Row of the virtual key list: entry index (>= 0), or raw token (a window
// token or a token of a selected block, encoded as -(pos + 2)), or -1 for an
// empty slot.
struct KeyList {
  const int32_t* idx;  // [k] selected entries of this query, or nullptr (dense)
  int k;               // length of the first part (entries, or raw tokens of the blocks)
  int m;               // raw-token blocks: tokens per block; 0 otherwise
  int64_t N;           // entries in the cache
  int64_t lo;          // first window position
  int64_t len;         // first part + window
  __device__ __forceinline__ int64_t at(int64_t j) const {
    if (j < k) {
      if (!idx) return j;
      if (m == 0) return (int64_t)idx[j];
      const int64_t s = idx[j / m];
      return (s >= 0 && s < N) ? -((s * m + j % m) + 2) : -1;
    }
    return -((lo + (j - k)) + 2);
  }
};

__global__ void __launch_bounds__(kThreads) attend_simt_kernel(
    const void* __restrict__ q, csa_dtype q_dtype, RowView kv, RowView raw, int64_t raw_pos0,
    const int32_t* __restrict__ idx, int mode, int64_t q_pos0, int Q, int64_t N, int H,
    int D_qk, int D_v, int k, int W, int m, float scale, int splits, int64_t split_len,
    void* __restrict__ out, csa_dtype out_dtype, float* __restrict__ ws) {
  extern __shared__ float sm[];
  const int ldk = D_qk + 1;
  float* Qs = sm;                           // [kHG][D_qk]
  float* Ks = Qs + kHG * D_qk;              // [kKT][ldk]
  float* P = Ks + kKT * ldk;                // [kHG][kKT]
  float* alpha_s = P + kHG * kKT;           // [kHG]
  __shared__ int64_t rows[kKT];

  const int split = blockIdx.z;
  const int hg = blockIdx.y;
  const int64_t qrow = blockIdx.x;  // b * Q + i
  const int i = (int)(qrow % Q);
  const int b = (int)(qrow / Q);
  const int64_t t = q_pos0 + i;
  const int tid = threadIdx.x;

  KeyList kl;
  kl.lo = t - W + 1 > 0 ? t - W + 1 : 0;
  kl.N = N;
  kl.m = 0;
  if (mode == kAttendDense) {
    int64_t nv = n_vis(t, m);
    kl.k = (int)(nv < N ? nv : N);
    kl.idx = nullptr;
  } else {
    kl.k = mode == kAttendRawBlocks ? k * m : k;
    kl.m = mode == kAttendRawBlocks ? m : 0;
    kl.idx = idx + qrow * (int64_t)k;
  }
  kl.len = kl.k + (t - kl.lo + 1);
  const int64_t j0 = (int64_t)split * split_len;
  int64_t j1 = j0 + split_len;
  if (j1 > kl.len) j1 = kl.len;

  for (int e = tid; e < kHG * D_qk; e += kThreads) {
    int hh = e / D_qk, c = e % D_qk;
    int h = hg * kHG + hh;
    Qs[e] = h < H ? load_elem(q, q_dtype, (qrow * H + h) * (int64_t)D_qk + c) * scale : 0.f;
  }

  const int my_h = tid / 16;        // head (within group) for S / O work
  const int lane16 = tid % 16;
  const int ndv = (D_v + 15) / 16;  // output columns per thread
  float o[kMaxDvPerThread];
#pragma unroll
  for (int c = 0; c < kMaxDvPerThread; ++c) o[c] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;  // valid in the softmax warps (per head)

  for (int64_t jt = j0; jt < j1; jt += kKT) {
    __syncthreads();
    if (tid < kKT) rows[tid] = (jt + tid < j1) ? kl.at(jt + tid) : -1;
    __syncthreads();
    for (int e = tid; e < kKT * D_qk; e += kThreads) {
      int jj = e / D_qk, c = e % D_qk;
      int64_t r = rows[jj];
      float v = 0.f;
      if (r >= 0) v = kv.get(b, r, c);
      else if (r <= -2) v = raw.get(b, (-r - 2) - raw_pos0, c);
      Ks[jj * ldk + c] = v;
    }
    __syncthreads();
    // scores: thread -> (head my_h, keys lane16 and lane16 + 16)
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      int jj = lane16 + 16 * half;
      const float* qh = Qs + my_h * D_qk;
      const float* kr = Ks + jj * ldk;
      float acc = 0.f;
      for (int c = 0; c < D_qk; ++c) acc = fmaf(qh[c], kr[c], acc);
      P[my_h * kKT + jj] = rows[jj] == -1 ? -INFINITY : acc;
    }
    __syncthreads();
    // online softmax: warp w handles heads 2w, 2w+1 (lanes 0-15 / 16-31 hold
    // keys j and j+16 of each)
    {
      const int w = tid >> 5, lane = tid & 31;
#pragma unroll
      for (int hh2 = 0; hh2 < 2; ++hh2) {
        const int hh = 2 * w + hh2;
        float s = P[hh * kKT + lane];
        float mx = s;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        // m_run / l_run of head hh live in lane hh2 of warp w
        float m_old = __shfl_sync(0xffffffffu, m_run, hh2);
        float l_old = __shfl_sync(0xffffffffu, l_run, hh2);
        float m_new = fmaxf(m_old, mx);
        float p = (m_new == -INFINITY) ? 0.f : __expf(s - m_new);
        float a = (m_new == -INFINITY) ? 1.f : __expf(m_old - m_new);
        float sum = p;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        P[hh * kKT + lane] = p;
        if (lane == hh2) { m_run = m_new; l_run = l_old * a + sum; }
        if (lane == 0) alpha_s[hh] = a;
      }
    }
    __syncthreads();
    {
      const float a = alpha_s[my_h];
      const float* ph = P + my_h * kKT;
#pragma unroll
      for (int c = 0; c < kMaxDvPerThread; ++c) {
        if (c < ndv) {
          int d = lane16 + 16 * c;
          float acc = o[c] * a;
          if (d < D_v) {
#pragma unroll 8
            for (int jj = 0; jj < kKT; ++jj) acc = fmaf(ph[jj], Ks[jj * ldk + d], acc);
          }
          o[c] = acc;
        }
      }
    }
  }
  __syncthreads();
  // publish (m, l) of every head through shared memory
  {
    const int w = tid >> 5, lane = tid & 31;
    if (lane < 2) {
      P[(2 * w + lane) * kKT + 0] = m_run;
      P[(2 * w + lane) * kKT + 1] = l_run;
    }
  }
  __syncthreads();
  const int h = hg * kHG + my_h;
  if (h >= H) return;
  const float mh = P[my_h * kKT + 0], lh = P[my_h * kKT + 1];
  if (splits == 1) {
    const float inv = lh > 0.f ? 1.f / lh : 0.f;
    const int64_t obase = (qrow * H + h) * (int64_t)D_v;
    for (int c = 0; c < ndv; ++c) {
      int d = lane16 + 16 * c;
      if (d >= D_v) break;
      float v = o[c] * inv;
      if (out_dtype == CSA_F32) reinterpret_cast<float*>(out)[obase + d] = v;
      else reinterpret_cast<uint16_t*>(out)[obase + d] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
    }
  } else {
    // partials: [rows*H][splits][D_v + 2]
    float* pw = ws + ((qrow * H + h) * (int64_t)splits + split) * (int64_t)(D_v + 2);
    for (int c = 0; c < ndv; ++c) {
      int d = lane16 + 16 * c;
      if (d >= D_v) break;
      pw[d] = o[c];
    }
    if (lane16 == 0) { pw[D_v] = mh; pw[D_v + 1] = lh; }
  }
}

__global__ void combine_kernel(const float* __restrict__ ws, int splits, int D_v, int64_t n_heads,
                               void* __restrict__ out, csa_dtype out_dtype) {
  const int64_t qh = blockIdx.x;
  if (qh >= n_heads) return;
  const float* base = ws + qh * (int64_t)splits * (D_v + 2);
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, base[s * (D_v + 2) + D_v]);
  float L = 0.f;
  for (int s = 0; s < splits; ++s) {
    float ms = base[s * (D_v + 2) + D_v];
    if (ms != -INFINITY) L += base[s * (D_v + 2) + D_v + 1] * __expf(ms - M);
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  for (int d = threadIdx.x; d < D_v; d += blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < splits; ++s) {
      float ms = base[s * (D_v + 2) + D_v];
      if (ms != -INFINITY) acc += base[s * (D_v + 2) + d] * __expf(ms - M);
    }
    float v = acc * inv;
    if (out_dtype == CSA_F32) reinterpret_cast<float*>(out)[qh * D_v + d] = v;
    else reinterpret_cast<uint16_t*>(out)[qh * D_v + d] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
}

// Split rule: a fixed number of keys per split, chosen from the key-list
// length only.  Prefill-sized launches (many queries) use one split.
void split_plan(const csa_params& p, int Q, int64_t N, int mode, int* splits, int64_t* split_len) {
  int64_t max_len;
  if (mode == kAttendDense) {
    max_len = N + p.window;
  } else if (mode == kAttendRawBlocks) {
    max_len = (int64_t)p.k * p.m + p.window;
  } else {
    max_len = (int64_t)p.k + p.window;
  }
  if (max_len < 1) max_len = 1;
  const int64_t rows = (int64_t)p.B * Q;
  if (rows >= 1024) {
    *splits = 1;
    *split_len = max_len;
    return;
  }
  const int64_t len = 128;  // keys per split
  *split_len = len;
  *splits = (int)ceil_div(max_len, len);
}

}  // namespace

// Scratch of either path (the dtypes that pick the path are not known here):
// the larger of the CUDA-core split partials and the tensor-core ones.  The
// tensor-core plan is largest for the latest query, which sees the most
// entries, so that position bounds it for every q_pos0.
size_t attend_workspace(const csa_params& p, int Q, int64_t N, int mode) {
  int splits;
  int64_t split_len;
  split_plan(p, Q, N, mode, &splits, &split_len);
  size_t simt = 0;
  if (splits > 1) simt = (size_t)p.B * Q * p.H * splits * (p.D_v + 2) * sizeof(float);
  const size_t tc = attend_tc_workspace(p, Q, N, mode, (int64_t)1 << 62);
  return simt > tc ? simt : tc;
}

cudaError_t launch_attend(const csa_params& p, const void* q, csa_dtype q_dtype, const csa_rows& kv,
                          const csa_rows& raw, int64_t raw_pos0, const int32_t* idx, int mode,
                          int64_t q_pos0, int Q, int64_t N, void* out, csa_dtype out_dtype,
                          void* ws, cudaStream_t st) {
  const int64_t rows = (int64_t)p.B * Q;
  if (rows <= 0) return cudaSuccess;
  if (attend_tc_supported(p, q_dtype, kv, raw, Q, N, out_dtype, mode))
    return launch_attend_tc(p, q, kv, raw, raw_pos0, idx, mode, q_pos0, Q, N, out, out_dtype, ws,
                            st);
  int splits;
  int64_t split_len;
  split_plan(p, Q, N, mode, &splits, &split_len);
  const int D_qk = p.D_qk;
  size_t smem = ((size_t)kHG * D_qk + (size_t)kKT * (D_qk + 1) + kHG * kKT + kHG) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(attend_simt_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)rows, (unsigned)ceil_div(p.H, kHG), (unsigned)splits);
  attend_simt_kernel<<<grid, kThreads, smem, st>>>(
      q, q_dtype, make_view(kv), make_view(raw), raw_pos0, idx, mode, q_pos0, Q, N, p.H,
      D_qk, p.D_v, p.k, p.window, p.m, p.scale, splits, split_len, out, out_dtype,
      reinterpret_cast<float*>(ws));
  e = cudaGetLastError();
  if (e != cudaSuccess || splits == 1) return e;
  combine_kernel<<<(unsigned)(rows * p.H), 128, 0, st>>>(reinterpret_cast<const float*>(ws), splits,
                                                         p.D_v, rows * p.H, out, out_dtype);
  return cudaGetLastError();
}

}  // namespace csa
