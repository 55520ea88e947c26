// Step 1 of CSA / HCA: softmax-gated block pooling with a learned position bias.
//
//   E[b,s,c] = sum_{i<m} softmax_i(gate[b,sm+i,c] + bias[i,c]) * x[b,sm+i,c]
//
// Sources: "一文搞懂 DeepSeek：从 V3 的 KV 压缩与 MoE，到 V4 的百万 token 上下文",
// section "V4 改进一：CSA 与 HCA" (m adjacent tokens pooled by softmax weights
// with a position bias); "DeepSeek-V4 详解" section 2.2 Step 1 (m = 4) and 2.3
// Step 1 (m' = 128).
//
// The work is a pure stream over x and the gates (HBM bound): one thread owns
// VEC adjacent channels of one entry and reads them with 16-byte loads, so a
// warp reads whole 512-byte stretches of a row.  The softmax is taken in two
// passes over the m rows (max, then exp / sums); the second pass re-reads
// rows the same thread has just read (L1 hits).
#include "common.cuh"

namespace csa {
namespace {

template <typename T, int VEC>
struct Vec;
template <>
struct Vec<float, 4> {
  __device__ static void load(const void* p, int64_t i, float* o) {
    float4 v = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p) + i);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
};
template <>
struct Vec<uint16_t, 8> {
  __device__ static void load(const void* p, int64_t i, float* o) {
    uint4 v = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p) + i);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      o[2 * j] = __uint_as_float(w[j] << 16);
      o[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
  }
};
template <typename T>
struct Vec<T, 1> {
  __device__ static void load(const void* p, int64_t i, float* o) {
    if constexpr (sizeof(T) == 4) o[0] = reinterpret_cast<const float*>(p)[i];
    else o[0] = bf16_to_f32(reinterpret_cast<const uint16_t*>(p)[i]);
  }
};

// float64 recompute of one channel; used when the fp32 result lies too close
// to a bfloat16 rounding boundary to decide the rounding.
template <typename T>
__device__ double pool_f64(const void* x, const void* g, const float* bias, int64_t row0, int C,
                           int m, int c) {
  double mx = -INFINITY;
  for (int i = 0; i < m; ++i) {
    float gv;
    Vec<T, 1>::load(g, (row0 + i) * C + c, &gv);
    mx = fmax(mx, (double)gv + (double)bias[i * C + c]);
  }
  double S = 0.0, A = 0.0;
  for (int i = 0; i < m; ++i) {
    float gv, xv;
    Vec<T, 1>::load(g, (row0 + i) * C + c, &gv);
    Vec<T, 1>::load(x, (row0 + i) * C + c, &xv);
    double e = exp((double)gv + (double)bias[i * C + c] - mx);
    S += e;
    A += e * (double)xv;
  }
  return A / S;
}

// out_mode: 0 = fp32 rows, 1 = bf16 rounded from the fp32 result,
//           2 = bf16 nearest to the exact result (guard band + fp64 recompute).
template <typename T, int VEC>
__global__ void __launch_bounds__(256) compress_kernel(const void* __restrict__ x,
                                                       const void* __restrict__ g,
                                                       const float* __restrict__ bias, int B,
                                                       int64_t T_rows, int64_t row_off, int m,
                                                       int C, int64_t s_begin, int64_t n_s,
                                                       void* __restrict__ out, int64_t out_rows,
                                                       int out_mode) {
  const int CV = C / VEC;
  const int64_t total = (int64_t)B * n_s * CV;
  for (int64_t item = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; item < total;
       item += (int64_t)gridDim.x * blockDim.x) {
    const int cv = (int)(item % CV);
    const int64_t bs = item / CV;
    const int64_t s = s_begin + bs % n_s;
    const int b = (int)(bs / n_s);
    const int c0 = cv * VEC;
    // first raw row of the block, relative to the rows held in x / g
    const int64_t row0 = (int64_t)b * T_rows + s * m - row_off;

    float mx[VEC], zabs[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) { mx[v] = -INFINITY; zabs[v] = 0.f; }
    for (int i = 0; i < m; ++i) {
      float gv[VEC];
      Vec<T, VEC>::load(g, (row0 + i) * C + c0, gv);
#pragma unroll
      for (int v = 0; v < VEC; ++v) {
        float z = gv[v] + bias[i * C + c0 + v];
        mx[v] = fmaxf(mx[v], z);
        zabs[v] = fmaxf(zabs[v], fabsf(z));
      }
    }
    float S[VEC], A[VEC], Aabs[VEC], dmax[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) { S[v] = 0.f; A[v] = 0.f; Aabs[v] = 0.f; dmax[v] = 0.f; }
    for (int i = 0; i < m; ++i) {
      float gv[VEC], xv[VEC];
      Vec<T, VEC>::load(g, (row0 + i) * C + c0, gv);
      Vec<T, VEC>::load(x, (row0 + i) * C + c0, xv);
#pragma unroll
      for (int v = 0; v < VEC; ++v) {
        float d = (gv[v] + bias[i * C + c0 + v]) - mx[v];
        float e = expf(d);
        dmax[v] = fmaxf(dmax[v], fabsf(d));
        S[v] += e;
        A[v] = fmaf(e, xv[v], A[v]);
        Aabs[v] = fmaf(e, fabsf(xv[v]), Aabs[v]);
      }
    }
    const int64_t orow = (int64_t)b * out_rows + s;
    if (out_mode == 0) {
      float* o = reinterpret_cast<float*>(out) + orow * C + c0;
#pragma unroll
      for (int v = 0; v < VEC; ++v) o[v] = A[v] / S[v];
    } else {
      uint16_t* o = reinterpret_cast<uint16_t*>(out) + orow * C + c0;
#pragma unroll
      for (int v = 0; v < VEC; ++v) {
        float r = A[v] / S[v];
        __nv_bfloat16 h = __float2bfloat16_rn(r);
        if (out_mode == 2) {
          // Error bound of the fp32 evaluation (unit roundoff u = 2^-24):
          // expf within 2 ulp, its argument off by u(|z| + |d|), m-term sums
          // off by m*u relative to sum e|x|; doubled for safety.
          float bound = Aabs[v] / S[v];
          float guard = (2.f * m + 8.f + 2.f * zabs[v] + 2.f * dmax[v]) * 2.f * 5.9604645e-8f * bound +
                        1e-38f;
          __nv_bfloat16 lo = __float2bfloat16_rn(r - guard);
          __nv_bfloat16 hi = __float2bfloat16_rn(r + guard);
          if (__bfloat16_as_ushort(lo) != __bfloat16_as_ushort(hi))
            h = __double2bfloat16(pool_f64<T>(x, g, bias, row0, C, m, c0 + v));
        }
        o[v] = __bfloat16_as_ushort(h);
      }
    }
  }
}

// Mixed e4m3 + bf16 output: one block per entry, float64 arithmetic.
template <typename T>
__global__ void __launch_bounds__(256) compress_e4m3_kernel(
    const void* __restrict__ x, const void* __restrict__ g, const float* __restrict__ bias,
    int64_t T_rows, int64_t row_off, int m, int C, int nope, int64_t s_begin, int64_t n_s,
    uint8_t* __restrict__ codes, uint16_t* __restrict__ rope, float* __restrict__ scale,
    int64_t out_rows) {
  extern __shared__ double vals[];  // [C]
  __shared__ double red[32];
  const int64_t s = s_begin + blockIdx.x % n_s;
  const int b = (int)(blockIdx.x / n_s);
  const int64_t row0 = (int64_t)b * T_rows + s * m - row_off;
  double amax = 0.0;
  for (int c = threadIdx.x; c < C; c += blockDim.x) {
    double v = pool_f64<T>(x, g, bias, row0, C, m, c);
    vals[c] = v;
    if (c < nope) amax = fmax(amax, fabs(v));
  }
  for (int o = 16; o > 0; o >>= 1) amax = fmax(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    double a = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0;
    for (int o = 16; o > 0; o >>= 1) a = fmax(a, __shfl_xor_sync(0xffffffffu, a, o));
    if (threadIdx.x == 0) red[0] = a;
  }
  __syncthreads();
  amax = red[0];
  const float sc = amax > 0.0 ? __double2float_rn(amax / 448.0) : 1.0f;
  const int64_t orow = (int64_t)b * out_rows + s;
  if (threadIdx.x == 0) scale[orow] = sc;
  for (int c = threadIdx.x; c < C; c += blockDim.x) {
    if (c < nope) {
      codes[orow * nope + c] =
          (uint8_t)__nv_cvt_double_to_fp8(vals[c] / (double)sc, __NV_SATFINITE, __NV_E4M3);
    } else {
      rope[orow * (C - nope) + (c - nope)] = __bfloat16_as_ushort(__double2bfloat16(vals[c]));
    }
  }
}

}  // namespace

cudaError_t launch_compress(const void* x, const void* gate, csa_dtype in_dtype, const float* bias,
                            int B, int64_t x_pos0, int64_t T, int m, int C, int64_t s_begin,
                            int64_t s_end, const csa_rows& out, cudaStream_t st) {
  const int64_t n_s = s_end - s_begin;
  if (n_s <= 0 || B <= 0) return cudaSuccess;
  if (out.dtype == CSA_E4M3) {
    const int64_t blocks = (int64_t)B * n_s;
    const size_t smem = (size_t)C * sizeof(double);
    if (in_dtype == CSA_F32)
      compress_e4m3_kernel<float><<<(unsigned)blocks, 256, smem, st>>>(
          x, gate, bias, T, x_pos0, m, C, out.nope, s_begin, n_s, (uint8_t*)out.data,
          (uint16_t*)out.rope, out.scale, out.n_rows);
    else
      compress_e4m3_kernel<uint16_t><<<(unsigned)blocks, 256, smem, st>>>(
          x, gate, bias, T, x_pos0, m, C, out.nope, s_begin, n_s, (uint8_t*)out.data,
          (uint16_t*)out.rope, out.scale, out.n_rows);
    return cudaGetLastError();
  }
  const int out_mode = out.dtype == CSA_F32 ? 0 : (m <= 16 ? 2 : 1);
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  auto grid_for = [&](int vec) {
    int64_t items = (int64_t)B * n_s * (C / vec);
    int64_t blocks = ceil_div(items, 256);
    int64_t cap = (int64_t)sms * 16;
    return (unsigned)(blocks < cap ? blocks : cap);
  };
  if (in_dtype == CSA_F32) {
    if (C % 4 == 0)
      compress_kernel<float, 4><<<grid_for(4), 256, 0, st>>>(x, gate, bias, B, T, x_pos0, m, C,
                                                             s_begin, n_s, out.data, out.n_rows,
                                                             out_mode);
    else
      compress_kernel<float, 1><<<grid_for(1), 256, 0, st>>>(x, gate, bias, B, T, x_pos0, m, C,
                                                             s_begin, n_s, out.data, out.n_rows,
                                                             out_mode);
  } else {
    if (C % 8 == 0)
      compress_kernel<uint16_t, 8><<<grid_for(8), 256, 0, st>>>(x, gate, bias, B, T, x_pos0, m,
                                                                C, s_begin, n_s, out.data,
                                                                out.n_rows, out_mode);
    else
      compress_kernel<uint16_t, 1><<<grid_for(1), 256, 0, st>>>(x, gate, bias, B, T, x_pos0, m,
                                                                C, s_begin, n_s, out.data,
                                                                out.n_rows, out_mode);
  }
  return cudaGetLastError();
}

}  // namespace csa
