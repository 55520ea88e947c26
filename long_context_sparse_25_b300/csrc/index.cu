// Step 2 of CSA: the lightning indexer.
//
//   I[b,i,s] = sum_j w[b,i,j] * max(0, q_idx[b,i,j,:] . keys[b,s,:])   (s visible)
//
// Sources: "一文搞懂 DeepSeek：从 V3 的 KV 压缩与 MoE，到 V4 的百万 token 上下文",
// section "V4 改进一：CSA 与 HCA" (a light indexer scores every compressed entry
// against the query); "DeepSeek-V4 详解" section 2.2 Step 2 (DSA-style
// lightning indexer, FP8).
//
// This file holds the CUDA-core path, used for fp32 inputs and for shapes the
// tensor-core path (index_tc.cu) does not take.  One CTA scores 128 keys of
// one query: the query's H_I x d_I rows (scales folded in) sit in shared
// memory, each thread owns one key and accumulates in fp32.
#include "common.cuh"

namespace csa {

bool index_tc_supported(const csa_params& p, csa_dtype q_dtype, const csa_rows& keys, int Q);
cudaError_t launch_index_tc(const csa_params& p, const void* q_idx, csa_dtype q_dtype,
                            const float* q_scale, const float* w, const csa_rows& keys,
                            int64_t q_pos0, int Q, int64_t N, void* scores, bool scores_bf16,
                            cudaStream_t st, bool fill_invisible);

namespace {

constexpr int kKeysPerCta = 128;

__global__ void __launch_bounds__(kKeysPerCta) index_simt_kernel(
    const void* __restrict__ q_idx, csa_dtype q_dtype, const float* __restrict__ q_scale,
    const float* __restrict__ w, RowView keys, int H_I, int d_I, int m, int64_t q_pos0, int Q,
    int64_t N, void* __restrict__ scores, int scores_bf16) {
  extern __shared__ float sm[];
  float* qs = sm;                      // [H_I][d_I]
  float* ws = sm + (size_t)H_I * d_I;  // [H_I]
  const int64_t n_chunks = (N + kKeysPerCta - 1) / kKeysPerCta;
  const int64_t chunk = blockIdx.x % n_chunks;
  const int64_t qrow = blockIdx.x / n_chunks;  // b * Q + i
  const int i = (int)(qrow % Q);
  const int b = (int)(qrow / Q);
  for (int e = threadIdx.x; e < H_I * d_I; e += blockDim.x) {
    const int j = e / d_I;
    float v;
    if (q_dtype == CSA_E4M3)
      v = e4m3_to_f32(reinterpret_cast<const uint8_t*>(q_idx)[qrow * H_I * d_I + e]) *
          q_scale[qrow * H_I + j];
    else
      v = load_elem(q_idx, q_dtype, qrow * H_I * d_I + e);
    qs[e] = v;
  }
  for (int j = threadIdx.x; j < H_I; j += blockDim.x) ws[j] = w[qrow * H_I + j];
  __syncthreads();

  const int64_t s = chunk * kKeysPerCta + threadIdx.x;
  if (s >= N) return;
  const int64_t nv = n_vis(q_pos0 + i, m);
  float out = -INFINITY;
  if (s < nv) {
    float acc = 0.f;
    for (int j = 0; j < H_I; ++j) {
      const float* qj = qs + (size_t)j * d_I;
      float dot = 0.f;
      for (int d = 0; d < d_I; ++d) dot = fmaf(qj[d], keys.get(b, s, d), dot);
      acc = fmaf(ws[j], fmaxf(dot, 0.f), acc);
    }
    out = acc;
  }
  if (scores_bf16)
    reinterpret_cast<uint16_t*>(scores)[qrow * N + s] = __bfloat16_as_ushort(__float2bfloat16_rn(out));
  else
    reinterpret_cast<float*>(scores)[qrow * N + s] = out;
}

}  // namespace

cudaError_t launch_index(const csa_params& p, const void* q_idx, csa_dtype q_dtype,
                         const float* q_scale, const float* w, const csa_rows& keys,
                         int64_t q_pos0, int Q, int64_t N, void* scores, bool scores_bf16,
                         cudaStream_t st, bool fill_invisible) {
  if (N <= 0 || Q <= 0 || p.B <= 0) return cudaSuccess;
  if (index_tc_supported(p, q_dtype, keys, Q))
    return launch_index_tc(p, q_idx, q_dtype, q_scale, w, keys, q_pos0, Q, N, scores, scores_bf16,
                           st, fill_invisible);
  const int64_t blocks = ceil_div(N, kKeysPerCta) * Q * p.B;
  if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
  dim3 grid((unsigned)blocks);
  size_t smem = ((size_t)p.H_I * p.d_I + p.H_I) * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(index_simt_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  index_simt_kernel<<<grid, kKeysPerCta, smem, st>>>(q_idx, q_dtype, q_scale, w, make_view(keys),
                                                     p.H_I, p.d_I, p.m, q_pos0, Q, N, scores,
                                                     scores_bf16 ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace csa
