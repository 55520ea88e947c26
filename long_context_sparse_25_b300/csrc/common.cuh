// Internal helpers shared by the kernels of libcsa_b300 (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/csa.h"

namespace csa {

// ---------------------------------------------------------------- scalars
__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
  return __uint_as_float(((uint32_t)h) << 16);
}
__device__ __forceinline__ float e4m3_to_f32(uint8_t c) {
  __nv_fp8_e4m3 v;
  v.__x = c;
  return (float)v;
}

// FP4 E2M1 code (low four bits) -> fp32: s ee m, bias 1; the magnitudes
// 0, 0.5, 1, 1.5, 2, 3, 4, 6.
__device__ __forceinline__ float e2m1_to_f32(uint8_t c) {
  const int e = (c >> 1) & 3, m = c & 1;
  const float mag = e == 0 ? 0.5f * (float)m : (1.f + 0.5f * (float)m) * (float)(1 << (e - 1));
  return (c & 8) ? -mag : mag;
}

// Load element `i` of a row stored as fp32 / bf16 (e4m3 rows go through
// RowView below, which also applies the row scale).
__device__ __forceinline__ float load_elem(const void* base, csa_dtype dt, int64_t i) {
  if (dt == CSA_F32) return reinterpret_cast<const float*>(base)[i];
  return bf16_to_f32(reinterpret_cast<const uint16_t*>(base)[i]);
}

// Order-preserving map of an fp32 score to uint32: larger float -> larger key.
// -0.0 is mapped like +0.0 so that signed zeros tie.
__device__ __forceinline__ uint32_t score_key(float x) {
  uint32_t b = __float_as_uint(x);
  if ((b << 1) == 0) b = 0;  // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// A device view of one csa_rows block (passed by value into kernels).
struct RowView {
  csa_dtype dtype;
  const void* data;
  const uint16_t* rope;
  const float* scale;
  int64_t n_rows;
  int width;
  int nope;

  __device__ __forceinline__ int64_t row_index(int b, int64_t r) const {
    return (int64_t)b * n_rows + r;
  }
  // Channel c of row (b, r) as fp32 (e4m3 / e2m1 codes multiplied by the row scale).
  __device__ __forceinline__ float get(int b, int64_t r, int c) const {
    int64_t ri = row_index(b, r);
    if (dtype == CSA_E2M1) {
      const uint8_t byte = reinterpret_cast<const uint8_t*>(data)[ri * (width / 2) + c / 2];
      return e2m1_to_f32((uint8_t)((byte >> ((c & 1) * 4)) & 0xF)) * scale[ri];
    }
    if (dtype == CSA_E4M3) {
      if (c < nope)
        return e4m3_to_f32(reinterpret_cast<const uint8_t*>(data)[ri * nope + c]) * scale[ri];
      return bf16_to_f32(rope[ri * (width - nope) + (c - nope)]);
    }
    return load_elem(data, dtype, ri * width + c);
  }
};

inline RowView make_view(const csa_rows& r) {
  RowView v;
  v.dtype = r.dtype;
  v.data = r.data;
  v.rope = reinterpret_cast<const uint16_t*>(r.rope);
  v.scale = r.scale;
  v.n_rows = r.n_rows;
  v.width = r.width;
  v.nope = r.dtype == CSA_E4M3 ? r.nope : r.width;
  return v;
}

__host__ __device__ inline int64_t n_vis(int64_t t, int m) { return (t + 1) / m; }

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ------------------------------------------------- launchers (internal ABI)
// Each returns cudaGetLastError() of its launches.
cudaError_t launch_compress(const void* x, const void* gate, csa_dtype in_dtype, const float* bias,
                            int B, int64_t x_pos0, int64_t T, int m, int C, int64_t s_begin,
                            int64_t s_end, const csa_rows& out, cudaStream_t st);
// The same blocks pooled into two caches (KV entries and indexer keys) in one
// launch when both take the same kernel; otherwise two launches.
cudaError_t launch_compress_pair(const void* x0, const void* g0, const float* bias0, int C0,
                                 const csa_rows& out0, const void* x1, const void* g1,
                                 const float* bias1, int C1, const csa_rows& out1,
                                 csa_dtype in_dtype, int B, int64_t x_pos0, int64_t T, int m,
                                 int64_t s_begin, int64_t s_end, cudaStream_t st);

// fill_invisible: write -inf for entries beyond each query's visibility (the
// fused forward skips it: top-k never reads them).
// scores_bf16: the scores are stored as bf16 (round to nearest even; -inf
// stays -inf) instead of fp32.
cudaError_t launch_index(const csa_params& p, const void* q_idx, csa_dtype q_dtype,
                         const float* q_scale, const float* w, const csa_rows& keys,
                         int64_t q_pos0, int Q, int64_t N, void* scores, bool scores_bf16,
                         cudaStream_t st, bool fill_invisible = true);

// Test aid (csa_debug_stall_next): true once, for the first launch of the
// named kernel after the aid was armed, which then clears it.
enum { kStallIndex = 1, kStallAttend = 2 };
bool take_debug_stall(int kernel);

// Read and clear the device error words of the bounded waits (0 = none).
cudaError_t index_tc_status(int* code, cudaStream_t st);
cudaError_t attend_tc_status(int* code, cudaStream_t st);
cudaError_t gproj_status(int* code, cudaStream_t st);

// Grouped output projection (gproj_tc.cu): y [T, G*d_g] = per group g,
// o[:, g*K .. (g+1)*K) . w[g]^T with K = (H/G)*D_v.
cudaError_t launch_group_proj(const void* o, int64_t T, int H, int D_v, const void* w, int G,
                              int d_g, void* y, bool y_f32, cudaStream_t st);

size_t topk_workspace(const csa_params& p, int Q, int64_t N);
int topk_launches(const csa_params& p, int Q, int64_t N);
// bf16: the scores are bf16 bit patterns (16-bit keys) instead of fp32.
cudaError_t launch_topk(const csa_params& p, const void* scores, bool bf16, int64_t q_pos0, int Q,
                        int64_t N, int32_t* idx, void* ws, cudaStream_t st);

// Key list of the attention: the selected entries (CSA), every visible
// entry (HCA), or the m raw tokens of every selected entry's block (the
// raw-token variant of CSA); the raw window follows in every case.
enum AttendMode { kAttendEntries = 0, kAttendDense = 1, kAttendRawBlocks = 2 };

size_t attend_workspace(const csa_params& p, int Q, int64_t N, int mode);
cudaError_t launch_attend(const csa_params& p, const void* q, csa_dtype q_dtype, const csa_rows& kv,
                          const csa_rows& raw, int64_t raw_pos0, const int32_t* idx, int mode,
                          int64_t q_pos0, int Q, int64_t N, void* out, csa_dtype out_dtype,
                          void* ws, cudaStream_t st);

}  // namespace csa
