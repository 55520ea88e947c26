// Step 3 of CSA: per-query top-k of the indexer scores.
//
// Sources: "一文搞懂 DeepSeek：从 V3 的 KV 压缩与 MoE，到 V4 的百万 token 上下文",
// section "V4 改进一：CSA 与 HCA" (keep the top-k highest-scoring entries);
// "DeepSeek-V4 详解" section 2.2 Step 3 (Top-1024).
//
// Exact radix select on order-preserving 32-bit keys of the fp32 scores
// (-0 folded onto +0): four 8-bit digit passes from the most significant end
// find the key T of the kk-th largest score and how many of the entries equal
// to T are still needed; a final pass over the row in index order keeps every
// key > T and the lowest-index keys == T, compacting with block-wide prefix
// sums, so the output comes out ascending with no sort.
//
// Rows up to kSmemRow entries are staged once in shared memory; longer rows
// (decode over 10^5..10^6 entries) are re-read from global memory / L2 in
// each pass by one CTA, or split over several CTAs by the multi-CTA path.
#include "common.cuh"

namespace csa {
namespace {

constexpr int kThreads = 1024;
constexpr int kSmemRow = 16384;

struct BlockScan {
  // exclusive prefix sum of v over the block; *total gets the block sum
  __device__ static int run(int v, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[wid] = x;
    __syncthreads();
    if (wid == 0) {
      int nw = blockDim.x >> 5;
      int ws = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, ws, o);
        if (lane >= o) ws += y;
      }
      warp_sums[lane] = ws;  // inclusive
    }
    __syncthreads();
    int before = wid > 0 ? warp_sums[wid - 1] : 0;
    *total = warp_sums[(blockDim.x >> 5) - 1];
    __syncthreads();
    return before + x - v;
  }
};

template <bool kSmem>
__global__ void __launch_bounds__(kThreads) topk_row_kernel(const float* __restrict__ scores,
                                                            int64_t q_pos0, int Q, int64_t N,
                                                            int m, int k,
                                                            int32_t* __restrict__ idx) {
  __shared__ int hist[256];
  __shared__ int warp_sums[32];
  __shared__ uint32_t sh_prefix;
  __shared__ int sh_need;
  extern __shared__ uint32_t row_keys[];  // kSmem: [n]

  const int64_t row = blockIdx.x;  // b * Q + i
  const int i = (int)(row % Q);
  const int64_t nvv = n_vis(q_pos0 + i, m);
  const int64_t n = nvv < N ? nvv : N;
  const int kk = (int)(n < k ? n : k);
  const float* srow = scores + row * N;
  int32_t* orow = idx + row * (int64_t)k;

  for (int j = kk + threadIdx.x; j < k; j += blockDim.x) orow[j] = -1;
  if (kk == n) {  // everything visible is kept
    for (int j = threadIdx.x; j < kk; j += blockDim.x) orow[j] = j;
    return;
  }
  if (kSmem) {
    for (int64_t s = threadIdx.x; s < n; s += blockDim.x) row_keys[s] = score_key(srow[s]);
  }
  auto key_at = [&](int64_t s) -> uint32_t {
    return kSmem ? row_keys[s] : score_key(__ldg(srow + s));
  };

  uint32_t prefix = 0, mask = 0;
  int need = kk;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int j = threadIdx.x; j < 256; j += blockDim.x) hist[j] = 0;
    __syncthreads();
    for (int64_t s = threadIdx.x; s < n; s += blockDim.x) {
      uint32_t kx = key_at(s);
      if ((kx & mask) == prefix) atomicAdd(&hist[(kx >> shift) & 255], 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // digits 255..0 in 8 chunks of 32: find the digit where the count of
      // larger-or-equal keys first reaches `need`
      const int lane = threadIdx.x;
      int above = 0;  // keys with a larger digit
      int found = -1, found_above = 0;
      for (int chunk = 7; chunk >= 0 && found < 0; --chunk) {
        int d = chunk * 32 + (31 - lane);  // lane 0 holds the largest digit
        int c = hist[d];
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        unsigned hit = __ballot_sync(0xffffffffu, above + incl >= need);
        if (hit) {
          int l = __ffs(hit) - 1;
          int excl = __shfl_sync(0xffffffffu, incl - c, l);
          found = chunk * 32 + (31 - l);
          found_above = above + excl;
        } else {
          above += __shfl_sync(0xffffffffu, incl, 31);
        }
      }
      if (lane == 0) {
        sh_prefix = prefix | ((uint32_t)found << shift);
        sh_need = need - found_above;
      }
    }
    __syncthreads();
    prefix = sh_prefix;
    need = sh_need;
    mask |= 255u << shift;
    __syncthreads();
  }
  // prefix == key of the kk-th largest score; keep keys > prefix and the
  // first `need` keys == prefix in index order.
  int taken = 0, eq_seen = 0;
  for (int64_t base = 0; base < n; base += blockDim.x) {
    const int64_t s = base + threadIdx.x;
    uint32_t kx = s < n ? key_at(s) : 0;
    int gt = (s < n && kx > prefix) ? 1 : 0;
    int eq = (s < n && kx == prefix) ? 1 : 0;
    int eq_tot;
    int eq_rank = eq_seen + BlockScan::run(eq, warp_sums, &eq_tot);
    int take = gt | (eq & (eq_rank < need ? 1 : 0));
    int take_tot;
    int pos = taken + BlockScan::run(take, warp_sums, &take_tot);
    if (take) orow[pos] = (int32_t)s;
    taken += take_tot;
    eq_seen += eq_tot;
  }
}

}  // namespace

size_t topk_workspace(const csa_params& p, int Q, int64_t N) {
  (void)p; (void)Q; (void)N;
  return 0;
}

cudaError_t launch_topk(const csa_params& p, const float* scores, int64_t q_pos0, int Q,
                        int64_t N, int32_t* idx, void* ws, cudaStream_t st) {
  (void)ws;
  const int64_t rows = (int64_t)p.B * Q;
  if (rows <= 0) return cudaSuccess;
  if (N <= kSmemRow) {
    size_t smem = (size_t)N * sizeof(uint32_t);
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(topk_row_kernel<true>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    topk_row_kernel<true><<<(unsigned)rows, kThreads, smem, st>>>(scores, q_pos0, Q, N, p.m, p.k,
                                                                  idx);
  } else {
    topk_row_kernel<false><<<(unsigned)rows, kThreads, 0, st>>>(scores, q_pos0, Q, N, p.m, p.k,
                                                                idx);
  }
  return cudaGetLastError();
}

}  // namespace csa
