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
// warp reads whole 512-byte stretches of a row.  For m <= 16 the softmax is
// taken in two passes over the m rows (max, then exp / sums; the second pass
// re-reads rows the same thread has just read, L1 hits); blocks of more rows
// (m' = 128) are read once with a running maximum.  One launch can pool the
// same blocks into two caches (the KV entries and the indexer keys of a
// decode step), each cache a contiguous range of CTAs.
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
// Packed form of VEC elements (kept packed while loads are in flight).
template <typename T, int VEC>
struct Packed;
template <>
struct Packed<float, 4> {
  using type = float4;
  __device__ static type load(const void* p, int64_t i) {
    return *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p) + i);
  }
  __device__ static void unpack(const type& v, float* o) {
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
};
template <>
struct Packed<uint16_t, 8> {
  using type = uint4;
  __device__ static type load(const void* p, int64_t i) {
    return *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p) + i);
  }
  __device__ static void unpack(const type& v, float* o) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      o[2 * j] = __uint_as_float(w[j] << 16);
      o[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
  }
};
template <typename T>
struct Packed<T, 1> {
  using type = float;
  __device__ static type load(const void* p, int64_t i) {
    float o;
    if constexpr (sizeof(T) == 4) o = reinterpret_cast<const float*>(p)[i];
    else o = bf16_to_f32(reinterpret_cast<const uint16_t*>(p)[i]);
    return o;
  }
  __device__ static void unpack(const type& v, float* o) { o[0] = v; }
};

template <typename T>
struct Vec<T, 1> {
  __device__ static void load(const void* p, int64_t i, float* o) {
    if constexpr (sizeof(T) == 4) o[0] = reinterpret_cast<const float*>(p)[i];
    else o[0] = bf16_to_f32(reinterpret_cast<const uint16_t*>(p)[i]);
  }
};

// float64 recompute of one channel: the last resort for a result that even
// the double-float evaluation below cannot place on one side of a bfloat16
// rounding boundary (float64 is slow on this part, so it must stay rare).
template <typename T>
__device__ __noinline__ double pool_f64(const void* x, const void* g, const float* bias, int64_t row0, int C,
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

// ---- double-float arithmetic: a value is the unevaluated sum hi + lo of two
// floats (about 48 significant bits), built on the error-free transformations
// TwoSum (Knuth) and TwoProduct (Dekker, here with a fused multiply-add).
struct ff {
  float hi, lo;
};
__device__ __forceinline__ ff ff_two_sum(float a, float b) {
  const float s = a + b;
  const float bb = s - a;
  return {s, (a - (s - bb)) + (b - bb)};
}
__device__ __forceinline__ ff ff_fast_two_sum(float a, float b) {  // |a| >= |b|
  const float s = a + b;
  return {s, b - (s - a)};
}
__device__ __forceinline__ ff ff_add(ff a, ff b) {
  ff s = ff_two_sum(a.hi, b.hi);
  const ff t = ff_two_sum(a.lo, b.lo);
  s.lo += t.hi;
  s = ff_fast_two_sum(s.hi, s.lo);
  s.lo += t.lo;
  return ff_fast_two_sum(s.hi, s.lo);
}
__device__ __forceinline__ ff ff_mul_f(ff a, float b) {
  const float p = a.hi * b;
  float e = fmaf(a.hi, b, -p);
  e = fmaf(a.lo, b, e);
  return ff_fast_two_sum(p, e);
}
__device__ __forceinline__ ff ff_mul(ff a, ff b) {
  const float p = a.hi * b.hi;
  float e = fmaf(a.hi, b.hi, -p);
  e = fmaf(a.hi, b.lo, e);
  e = fmaf(a.lo, b.hi, e);
  return ff_fast_two_sum(p, e);
}
// a / b by two Newton corrections of the float quotient.
__device__ __forceinline__ ff ff_div(ff a, ff b) {
  const float q1 = a.hi / b.hi;
  ff r = ff_add(a, ff_mul_f(b, -q1));
  const float q2 = r.hi / b.hi;
  r = ff_add(r, ff_mul_f(b, -q2));
  const float q3 = r.hi / b.hi;
  return ff_add(ff_fast_two_sum(q1, q2), ff{q3, 0.f});
}
__device__ __forceinline__ bool ff_gt(ff a, ff b) { return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo); }

// 1/n! for n = 0..13 as double-floats (high part: the float nearest 1/n!;
// low part: the float nearest the rest).
__constant__ float c_inv_fact[14][2] = {
    {1.0f, 0.0f},
    {1.0f, 0.0f},
    {0.5f, 0.0f},
    {0.1666666716337204f, -4.967053879312289e-09f},
    {0.0416666679084301f, -1.2417634698280722e-09f},
    {0.008333333767950535f, -4.34617203337595e-10f},
    {0.0013888889225199819f, -3.3631094437103215e-11f},
    {0.00019841270113829523f, -2.725596874933456e-12f},
    {2.4801587642286904e-05f, -3.40699609366682e-13f},
    {2.7557318844628753e-06f, 3.793571224297229e-14f},
    {2.755731998149713e-07f, -7.575112209051195e-15f},
    {2.5052107943679403e-08f, 4.4176230446483665e-16f},
    {2.0876755879584152e-09f, 1.1082839147459852e-16f},
    {1.6059044372074283e-10f, -5.352526511562726e-18f},
};

// e^d for four d <= 0 at once in double-float: for each, Cody-Waite
// reduction d = k ln2 + r (|r| <= ln2/2, ln2 held as a double-float) and the
// Taylor series of e^r to degree 13 (|r|^14/14! < 2^-50) in Horner form; the
// four Horner chains are interleaved so that their latencies overlap.  Below
// d = -120 (e^d < 2^-173, nothing next to the e^0 term) the result is 0.
__device__ void ff_exp4_nonpos(const ff (&d)[4], ff (&e)[4]) {
  const float ln2_hi = 0.693147182464599609375f;
  const float ln2_lo = -1.904654323148236017e-09f;
  ff r[4], s[4];
  int ki[4];
  bool zero[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    zero[j] = d[j].hi < -120.f;
    const ff dj = zero[j] ? ff{0.f, 0.f} : d[j];
    const float k = rintf(dj.hi * 1.44269504088896340736f);
    const float p = k * ln2_hi;
    const ff kl = ff_fast_two_sum(p, fmaf(k, ln2_hi, -p) + k * ln2_lo);
    r[j] = ff_add(dj, ff{-kl.hi, -kl.lo});
    s[j] = ff{c_inv_fact[13][0], c_inv_fact[13][1]};
    ki[j] = (int)k;
  }
#pragma unroll 1
  for (int n = 12; n >= 0; --n) {
    const ff cn{c_inv_fact[n][0], c_inv_fact[n][1]};
#pragma unroll
    for (int j = 0; j < 4; ++j) s[j] = ff_add(ff_mul(s[j], r[j]), cn);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j)
    e[j] = zero[j] ? ff{0.f, 0.f} : ff{ldexpf(s[j].hi, ki[j]), ldexpf(s[j].lo, ki[j])};
}

// Pooled value of one channel in double-float; *mag (if given) receives
// sum_i w_i |x_i|, the scale its error is relative to (about 2^-44 of it).
template <typename T>
__device__ ff pool_ff(const void* x, const void* g, const float* bias, int64_t row0, int C, int m,
                      int c, float* mag = nullptr) {
  ff mx{-INFINITY, 0.f};
  for (int i = 0; i < m; ++i) {
    float gv;
    Vec<T, 1>::load(g, (row0 + i) * C + c, &gv);
    const ff z = ff_two_sum(gv, bias[i * C + c]);  // exact
    if (i == 0 || ff_gt(z, mx)) mx = z;
  }
  ff S{0.f, 0.f}, A{0.f, 0.f};
  for (int i0 = 0; i0 < m; i0 += 4) {  // four rows' exponentials at a time
    ff d[4], e[4];
    float xv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = i0 + j;
      xv[j] = 0.f;
      d[j] = ff{-1000.f, 0.f};  // past the last row: e = 0, not summed
      if (i < m) {
        float gv;
        Vec<T, 1>::load(g, (row0 + i) * C + c, &gv);
        Vec<T, 1>::load(x, (row0 + i) * C + c, &xv[j]);
        d[j] = ff_add(ff_two_sum(gv, bias[i * C + c]), ff{-mx.hi, -mx.lo});
      }
    }
    ff_exp4_nonpos(d, e);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (i0 + j < m) {
        S = ff_add(S, e[j]);
        A = ff_add(A, ff_mul_f(e[j], xv[j]));
        if (mag) *mag += e[j].hi * fabsf(xv[j]);
      }
    }
  }
  if (mag) *mag /= S.hi;
  return ff_div(A, S);
}

// The bfloat16 nearest to the exact pooled value.  hi + lo is within about
// 2^-44 * sum w|x| of it.  Unless the sum cancels by more than 2^14 (then
// float64 decides), that is far below half a float ulp of hi, so hi + lo
// rounds the same way as the exact value unless hi is itself a rounding
// midpoint (every other float is a full float ulp away from the nearest
// midpoint); then the sign of lo decides, and a lo too small to trust sends
// the channel to float64.
//
// Compiled once (not inlined, its loops rolled): a few lanes of a warp take
// this path, and an inlined copy per unrolled channel left them waiting on
// instruction fetches through long stretches of cold code.
template <typename T>
__device__ __noinline__ uint16_t pool_bf16_exact(const void* x, const void* g, const float* bias, int64_t row0,
                                    int C, int m, int c) {
  float mag = 0.f;
  const ff v = pool_ff<T>(x, g, bias, row0, C, m, c, &mag);
  const uint32_t hb = __float_as_uint(v.hi);
  const bool cancels = mag > ldexpf(fabsf(v.hi), 14);
  const bool midpoint = (hb & 0xffffu) == 0x8000u;
  if (cancels || (midpoint && fabsf(v.lo) <= ldexpf(fabsf(v.hi), -28)))
    return __bfloat16_as_ushort(__double2bfloat16(pool_f64<T>(x, g, bias, row0, C, m, c)));
  if (!midpoint) return __bfloat16_as_ushort(__float2bfloat16_rn(v.hi));
  const uint16_t t = (uint16_t)(hb >> 16);  // truncated: the midpoint's smaller magnitude side
  return ((v.lo > 0.f) == (v.hi > 0.f)) ? (uint16_t)(t + 1) : t;
}

// One pooling job: a set of rows (x, gates, position bias) of C channels
// and the cache its entries go to.
// out_mode: 0 = fp32 rows, 1 = bf16 rounded from the fp32 result,
//           2 = bf16 nearest to the exact result (guard band + double-float
//               recompute of the channels too close to a rounding boundary).
struct CJob {
  const void* x;
  const void* g;
  const float* bias;
  int C;
  void* out;
  int64_t out_rows;
  int out_mode;
};

// The items of one job, from `first`, every `stride`-th.
template <typename T, int VEC>
__device__ __forceinline__ void pool_job(const CJob& J, int64_t first, int64_t stride, int B,
                                         int64_t T_rows, int64_t row_off, int m, int64_t s_begin,
                                         int64_t n_s) {
  const void* __restrict__ x = J.x;
  const void* __restrict__ g = J.g;
  const float* __restrict__ bias = J.bias;
  const int C = J.C;
  void* __restrict__ out = J.out;
  const int64_t out_rows = J.out_rows;
  const int out_mode = J.out_mode;
  const int CV = C / VEC;
  const int64_t total = (int64_t)B * n_s * CV;
  for (int64_t item = first; item < total; item += stride) {
    const int cv = (int)(item % CV);
    const int64_t bs = item / CV;
    const int64_t s = s_begin + bs % n_s;
    const int b = (int)(bs / n_s);
    const int c0 = cv * VEC;
    // first raw row of the block, relative to the rows held in x / g
    const int64_t row0 = (int64_t)b * T_rows + s * m - row_off;

    if (out_mode != 2 && m > 16) {
      // one pass with a running maximum (large blocks: m' = 128 rows are read
      // once, eight rows' loads in flight at a time); the result is rounded
      // once, so no error bound is needed
      float mx[VEC], S[VEC], A[VEC];
#pragma unroll
      for (int v = 0; v < VEC; ++v) { mx[v] = -INFINITY; S[v] = 0.f; A[v] = 0.f; }
      using P = Packed<T, VEC>;
      for (int i0 = 0; i0 < m; i0 += 8) {
        typename P::type gp[8], xp[8];
#pragma unroll
        for (int ii = 0; ii < 8; ++ii) {
          if (i0 + ii < m) {
            gp[ii] = P::load(g, (row0 + i0 + ii) * C + c0);
            xp[ii] = P::load(x, (row0 + i0 + ii) * C + c0);
          }
        }
#pragma unroll
        for (int ii = 0; ii < 8; ++ii) {
          if (i0 + ii < m) {
            float gv[VEC], xv[VEC];
            P::unpack(gp[ii], gv);
            P::unpack(xp[ii], xv);
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
              const float z = gv[v] + bias[(i0 + ii) * C + c0 + v];
              if (z > mx[v]) {  // rescale what has been summed so far
                const float r = __expf(mx[v] - z);  // 0 for the first row
                S[v] *= r;
                A[v] *= r;
                mx[v] = z;
              }
              const float e = __expf(z - mx[v]);
              S[v] += e;
              A[v] = fmaf(e, xv[v], A[v]);
            }
          }
        }
      }
      const int64_t orow1 = (int64_t)b * out_rows + s;
      if (out_mode == 0) {
        float* o = reinterpret_cast<float*>(out) + orow1 * C + c0;
#pragma unroll
        for (int v = 0; v < VEC; ++v) o[v] = A[v] / S[v];
      } else {
        uint16_t* o = reinterpret_cast<uint16_t*>(out) + orow1 * C + c0;
#pragma unroll
        for (int v = 0; v < VEC; ++v) o[v] = __bfloat16_as_ushort(__float2bfloat16_rn(A[v] / S[v]));
      }
      continue;
    }
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
            h = __ushort_as_bfloat16(pool_bf16_exact<T>(x, g, bias, row0, C, m, c0 + v));
        }
        o[v] = __bfloat16_as_ushort(h);
      }
    }
  }
}

// One launch for one or two jobs (a decode step pools its new entry for the
// KV cache and for the indexer-key cache together): blocks [0, blocks0) take
// job 0, the rest job 1, so a block's job is uniform.
template <typename T, int VEC>
__global__ void __launch_bounds__(256) compress_kernel(const CJob j0, const CJob j1,
                                                       unsigned blocks0, int B, int64_t T_rows,
                                                       int64_t row_off, int m, int64_t s_begin,
                                                       int64_t n_s) {
  if (blockIdx.x < blocks0)
    pool_job<T, VEC>(j0, (int64_t)blockIdx.x * blockDim.x + threadIdx.x,
                     (int64_t)blocks0 * blockDim.x, B, T_rows, row_off, m, s_begin, n_s);
  else
    pool_job<T, VEC>(j1, (int64_t)(blockIdx.x - blocks0) * blockDim.x + threadIdx.x,
                     (int64_t)(gridDim.x - blocks0) * blockDim.x, B, T_rows, row_off, m, s_begin,
                     n_s);
}

// Mixed e4m3 + bf16 output: one block per entry, one thread per channel (the
// double-float pool of a channel is a long dependent chain: a thread that
// took three of them made a decode step's compress three chains long); the
// pooled values in double-float (exact in float64), then the row scale and
// the codes in float64.
template <typename T>
__global__ void __launch_bounds__(1024) compress_e4m3_kernel(
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
    const ff pv = pool_ff<T>(x, g, bias, row0, C, m, c);
    const double v = (double)pv.hi + (double)pv.lo;
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

// FP4 E2M1 code of x (round to nearest, ties to the even mantissa bit,
// saturating at +-6): the grid is 0.5 below 2, 1 in [2, 4), 2 in [4, 6].
__device__ __forceinline__ uint32_t e2m1_code(double x) {
  const double ax = fmin(fabs(x), 6.0);
  const double q = ax < 2.0 ? 0.5 : (ax < 4.0 ? 1.0 : 2.0);
  const double r = fmin(rint(ax / q) * q, 6.0);  // rint: half to even on the grid
  // magnitude -> code: 0, .5, 1, 1.5 -> 0..3; 2, 3 -> 4, 5; 4, 6 -> 6, 7
  const uint32_t mag = r < 2.0 ? (uint32_t)(r * 2.0) : (r < 4.0 ? (uint32_t)r + 2u : (uint32_t)(r * 0.5) + 4u);
  return mag | (signbit(x) ? 8u : 0u);
}

// FP4 output (indexer keys): one block per entry, one thread per channel; the
// pooled values in double-float (exact in float64), the row scale amax / 6
// rounded to fp32, the codes decided in float64, two per byte.
template <typename T>
__global__ void __launch_bounds__(1024) compress_e2m1_kernel(
    const void* __restrict__ x, const void* __restrict__ g, const float* __restrict__ bias,
    int64_t T_rows, int64_t row_off, int m, int C, int64_t s_begin, int64_t n_s,
    uint8_t* __restrict__ codes, float* __restrict__ scale, int64_t out_rows) {
  extern __shared__ double vals[];  // [C]
  __shared__ double red[32];
  const int64_t s = s_begin + blockIdx.x % n_s;
  const int b = (int)(blockIdx.x / n_s);
  const int64_t row0 = (int64_t)b * T_rows + s * m - row_off;
  double amax = 0.0;
  for (int c = threadIdx.x; c < C; c += blockDim.x) {
    const ff pv = pool_ff<T>(x, g, bias, row0, C, m, c);
    const double v = (double)pv.hi + (double)pv.lo;
    vals[c] = v;
    amax = fmax(amax, fabs(v));
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
  const float sc = amax > 0.0 ? __double2float_rn(amax / 6.0) : 1.0f;
  const int64_t orow = (int64_t)b * out_rows + s;
  if (threadIdx.x == 0) scale[orow] = sc;
  for (int c2 = threadIdx.x; c2 < C / 2; c2 += blockDim.x) {
    const uint32_t lo = e2m1_code(vals[2 * c2] / (double)sc);
    const uint32_t hi = e2m1_code(vals[2 * c2 + 1] / (double)sc);
    codes[orow * (C / 2) + c2] = (uint8_t)(lo | (hi << 4));
  }
}

}  // namespace

// Threads of a one-block-per-entry kernel: one per channel, whole warps, at
// most 1024 (wider rows loop).
static int entry_threads(int C) {
  const int t = (C + 31) / 32 * 32;
  return t > 1024 ? 1024 : (t < 32 ? 32 : t);
}

// Channels per thread: 4 fp32 / 8 bf16 (16-byte loads) unless the step has
// few entries (a decode step): then one channel per thread, so that the rare
// channels needing the exact-rounding recompute sit in different threads (a
// warp runs its lanes' recomputes one after another) and the grid is wider.
static int pool_vec(csa_dtype in_dtype, int C, int B, int64_t n_s, int m) {
  const bool few = (int64_t)B * n_s * m < 4096;
  if (few) return 1;
  if (in_dtype == CSA_F32) return C % 4 == 0 ? 4 : 1;
  return C % 8 == 0 ? 8 : 1;
}

static cudaError_t launch_pool(const CJob& j0, const CJob& j1, csa_dtype in_dtype, int B,
                               int64_t x_pos0, int64_t T, int m, int64_t s_begin, int64_t n_s,
                               cudaStream_t st) {
  const int vec = pool_vec(in_dtype, j0.C, B, n_s, m);
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // blocks of each job: one item per thread, at most 16 blocks per SM in all
  const int64_t items0 = (int64_t)B * n_s * (j0.C / vec), items1 = (int64_t)B * n_s * (j1.C / vec);
  const int64_t cap = (int64_t)sms * 16;
  int64_t b0 = ceil_div(items0, 256), b1 = ceil_div(items1, 256);
  if (b0 + b1 > cap) {
    const int64_t c0 = cap * items0 / (items0 + items1);
    b0 = b0 < c0 ? b0 : (c0 < 1 ? 1 : c0);
    b1 = b1 < cap - b0 ? b1 : cap - b0;
  }
  if (b0 < 1) b0 = 1;
  const unsigned blocks0 = (unsigned)b0, grid = (unsigned)(b0 + b1);
  if (in_dtype == CSA_F32) {
    if (vec == 4)
      compress_kernel<float, 4><<<grid, 256, 0, st>>>(j0, j1, blocks0, B, T, x_pos0, m, s_begin, n_s);
    else
      compress_kernel<float, 1><<<grid, 256, 0, st>>>(j0, j1, blocks0, B, T, x_pos0, m, s_begin, n_s);
  } else {
    if (vec == 8)
      compress_kernel<uint16_t, 8><<<grid, 256, 0, st>>>(j0, j1, blocks0, B, T, x_pos0, m,
                                                         s_begin, n_s);
    else
      compress_kernel<uint16_t, 1><<<grid, 256, 0, st>>>(j0, j1, blocks0, B, T, x_pos0, m,
                                                         s_begin, n_s);
  }
  return cudaGetLastError();
}

cudaError_t launch_compress(const void* x, const void* gate, csa_dtype in_dtype, const float* bias,
                            int B, int64_t x_pos0, int64_t T, int m, int C, int64_t s_begin,
                            int64_t s_end, const csa_rows& out, cudaStream_t st) {
  const int64_t n_s = s_end - s_begin;
  if (n_s <= 0 || B <= 0) return cudaSuccess;
  if (out.dtype == CSA_E2M1) {
    const int64_t blocks = (int64_t)B * n_s;
    const size_t smem = (size_t)C * sizeof(double);
    if (in_dtype == CSA_F32)
      compress_e2m1_kernel<float><<<(unsigned)blocks, entry_threads(C), smem, st>>>(
          x, gate, bias, T, x_pos0, m, C, s_begin, n_s, (uint8_t*)out.data, out.scale, out.n_rows);
    else
      compress_e2m1_kernel<uint16_t><<<(unsigned)blocks, entry_threads(C), smem, st>>>(
          x, gate, bias, T, x_pos0, m, C, s_begin, n_s, (uint8_t*)out.data, out.scale, out.n_rows);
    return cudaGetLastError();
  }
  if (out.dtype == CSA_E4M3) {
    const int64_t blocks = (int64_t)B * n_s;
    const size_t smem = (size_t)C * sizeof(double);
    if (in_dtype == CSA_F32)
      compress_e4m3_kernel<float><<<(unsigned)blocks, entry_threads(C), smem, st>>>(
          x, gate, bias, T, x_pos0, m, C, out.nope, s_begin, n_s, (uint8_t*)out.data,
          (uint16_t*)out.rope, out.scale, out.n_rows);
    else
      compress_e4m3_kernel<uint16_t><<<(unsigned)blocks, entry_threads(C), smem, st>>>(
          x, gate, bias, T, x_pos0, m, C, out.nope, s_begin, n_s, (uint8_t*)out.data,
          (uint16_t*)out.rope, out.scale, out.n_rows);
    return cudaGetLastError();
  }
  CJob j0{x, gate, bias, C, out.data, out.n_rows, out.dtype == CSA_F32 ? 0 : (m <= 16 ? 2 : 1)};
  CJob j1{nullptr, nullptr, nullptr, 0, nullptr, 0, 0};
  return launch_pool(j0, j1, in_dtype, B, x_pos0, T, m, s_begin, n_s, st);
}

cudaError_t launch_compress_pair(const void* x0, const void* g0, const float* bias0, int C0,
                                 const csa_rows& out0, const void* x1, const void* g1,
                                 const float* bias1, int C1, const csa_rows& out1,
                                 csa_dtype in_dtype, int B, int64_t x_pos0, int64_t T, int m,
                                 int64_t s_begin, int64_t s_end, cudaStream_t st) {
  const int64_t n_s = s_end - s_begin;
  const bool pair = out0.dtype != CSA_E4M3 && out1.dtype != CSA_E4M3 &&
                    out0.dtype != CSA_E2M1 && out1.dtype != CSA_E2M1 &&
                    pool_vec(in_dtype, C0, B, n_s, m) == pool_vec(in_dtype, C1, B, n_s, m);
  if (n_s <= 0 || B <= 0) return cudaSuccess;
  if (!pair) {
    cudaError_t e = launch_compress(x0, g0, in_dtype, bias0, B, x_pos0, T, m, C0, s_begin, s_end,
                                    out0, st);
    if (e != cudaSuccess) return e;
    return launch_compress(x1, g1, in_dtype, bias1, B, x_pos0, T, m, C1, s_begin, s_end, out1, st);
  }
  const int mode_bf16 = m <= 16 ? 2 : 1;
  CJob j0{x0, g0, bias0, C0, out0.data, out0.n_rows, out0.dtype == CSA_F32 ? 0 : mode_bf16};
  CJob j1{x1, g1, bias1, C1, out1.data, out1.n_rows, out1.dtype == CSA_F32 ? 0 : mode_bf16};
  return launch_pool(j0, j1, in_dtype, B, x_pos0, T, m, s_begin, n_s, st);
}

}  // namespace csa
