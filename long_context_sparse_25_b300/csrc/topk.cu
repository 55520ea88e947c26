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


// ------------------------------------------------------------------------
// Long rows with few rows (decode: B rows of 10^5..10^6 entries) are split
// over many CTAs in three kernels:
//   A  hist:   each CTA histograms the top kDigitBits bits of its slice's keys
//              into the row's global histogram;
//   B  filter: each CTA finds the boundary digit (the one holding the kk-th
//              largest key), appends every index with a larger digit to the
//              row's "selected" list and every (key, index) with the boundary
//              digit to the row's candidate list;
//   C  final:  one CTA per row picks the still-needed candidates exactly, by
//              a radix select on the 64-bit composite (key << 32 | ~index),
//              whose values are all distinct and order ties by lower index;
//              then sorts the kk indices ascending (bitonic, shared memory).
// The lists are filled in whatever order the atomics give, but the final
// set is unique and sorted, so the output is deterministic.
constexpr int kDigitBits = 12;
constexpr int kBins = 1 << kDigitBits;
constexpr int kMaxK = 4096;         // bitonic sort capacity of kernel C
constexpr int kCandSmem = 3840;     // candidates kept in shared memory by kernel C (static smem < 48 KB)

struct LongRows {
  int* hist;          // [rows][kBins]
  int* counts;        // [rows][2]: selected, candidates
  int32_t* selected;  // [rows][k]
  unsigned long long* cand;  // [rows][N]
};

__device__ __forceinline__ int64_t row_visible(int64_t row, int Q, int64_t q_pos0, int m, int64_t N) {
  const int i = (int)(row % Q);
  const int64_t nv = n_vis(q_pos0 + i, m);
  return nv < N ? nv : N;
}

__global__ void __launch_bounds__(512) topk_hist_kernel(const float* __restrict__ scores,
                                                        int64_t q_pos0, int Q, int64_t N, int m,
                                                        int k, LongRows lr) {
  __shared__ int h[kBins];
  const int64_t row = blockIdx.y;
  const int64_t n = row_visible(row, Q, q_pos0, m, N);
  if (n <= k) return;  // everything kept: kernel C handles it directly
  for (int j = threadIdx.x; j < kBins; j += blockDim.x) h[j] = 0;
  __syncthreads();
  const int64_t per = (n + gridDim.x - 1) / gridDim.x;
  const int64_t s0 = blockIdx.x * per, s1 = s0 + per < n ? s0 + per : n;
  const float* srow = scores + row * N;
  for (int64_t s = s0 + threadIdx.x; s < s1; s += blockDim.x)
    atomicAdd(&h[score_key(__ldg(srow + s)) >> (32 - kDigitBits)], 1);
  __syncthreads();
  int* gh = lr.hist + row * kBins;
  for (int j = threadIdx.x; j < kBins; j += blockDim.x)
    if (h[j]) atomicAdd(&gh[j], h[j]);
}

// boundary digit of a row from its histogram (block-wide), with the count of
// keys in larger digits
__device__ void find_boundary(const int* gh, int kk, int* sh, int* out_digit, int* out_above) {
  // sh: kBins ints of shared memory; suffix sums from the top digit down
  for (int j = threadIdx.x; j < kBins; j += blockDim.x) sh[j] = gh[j];
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int above = 0;
    for (int base = kBins - 32; base >= 0; base -= 32) {
      const int d = base + 31 - lane;  // lane 0: largest digit of the chunk
      const int c = sh[d];
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      unsigned hit = __ballot_sync(0xffffffffu, above + incl >= kk);
      if (hit) {
        const int l = __ffs(hit) - 1;
        const int excl = __shfl_sync(0xffffffffu, incl - c, l);
        if (lane == 0) {
          *out_digit = base + 31 - l;
          *out_above = above + excl;
        }
        break;
      }
      above += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(512) topk_filter_kernel(const float* __restrict__ scores,
                                                          int64_t q_pos0, int Q, int64_t N, int m,
                                                          int k, LongRows lr) {
  __shared__ int sh[kBins];
  __shared__ int digit, above;
  const int64_t row = blockIdx.y;
  const int64_t n = row_visible(row, Q, q_pos0, m, N);
  if (n <= k) return;
  find_boundary(lr.hist + row * kBins, k, sh, &digit, &above);
  const uint32_t dstar = (uint32_t)digit;
  const int64_t per = (n + gridDim.x - 1) / gridDim.x;
  const int64_t s0 = blockIdx.x * per, s1 = s0 + per < n ? s0 + per : n;
  const float* srow = scores + row * N;
  int* cnt = lr.counts + row * 2;
  int32_t* sel = lr.selected + row * (int64_t)k;
  unsigned long long* cand = lr.cand + row * N;
  const int lane = threadIdx.x & 31;
  for (int64_t base = s0; base < s1; base += blockDim.x) {
    const int64_t s = base + threadIdx.x;
    uint32_t key = 0, d = 0;
    if (s < s1) {
      key = score_key(__ldg(srow + s));
      d = key >> (32 - kDigitBits);
    }
    const bool up = s < s1 && d > dstar;
    const bool eq = s < s1 && d == dstar;
    unsigned mu = __ballot_sync(0xffffffffu, up);
    unsigned me = __ballot_sync(0xffffffffu, eq);
    int bu = 0, be = 0;
    if (lane == 0) {
      if (mu) bu = atomicAdd(&cnt[0], __popc(mu));
      if (me) be = atomicAdd(&cnt[1], __popc(me));
    }
    bu = __shfl_sync(0xffffffffu, bu, 0);
    be = __shfl_sync(0xffffffffu, be, 0);
    const unsigned lower = (1u << lane) - 1u;
    if (up) sel[bu + __popc(mu & lower)] = (int32_t)s;
    if (eq)
      cand[be + __popc(me & lower)] =
          ((unsigned long long)key << 32) | (unsigned long long)(~(uint32_t)s);
  }
}

// radix select over 64-bit composites: the `need`-th largest (all distinct)
template <bool kSmem>
__device__ unsigned long long select_composite(const unsigned long long* v, int64_t n, int need,
                                               int* hist, unsigned long long* sh_prefix,
                                               int* sh_need) {
  unsigned long long prefix = 0, mask = 0;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int j = threadIdx.x; j < 256; j += blockDim.x) hist[j] = 0;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
      unsigned long long x = v[i];
      if ((x & mask) == prefix) atomicAdd(&hist[(int)((x >> shift) & 255)], 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      int acc_above = 0;
      for (int chunk = 7; chunk >= 0; --chunk) {
        const int d = chunk * 32 + (31 - lane);
        const int c = hist[d];
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        unsigned hit = __ballot_sync(0xffffffffu, acc_above + incl >= need);
        if (hit) {
          const int l = __ffs(hit) - 1;
          const int excl = __shfl_sync(0xffffffffu, incl - c, l);
          if (lane == 0) {
            *sh_prefix = prefix | ((unsigned long long)(chunk * 32 + 31 - l) << shift);
            *sh_need = need - (acc_above + excl);
          }
          break;
        }
        acc_above += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    __syncthreads();
    prefix = *sh_prefix;
    need = *sh_need;
    mask |= 255ull << shift;
    __syncthreads();
  }
  return prefix;
}

__global__ void __launch_bounds__(1024) topk_final_kernel(int64_t q_pos0, int Q, int64_t N, int m,
                                                          int k, LongRows lr,
                                                          int32_t* __restrict__ idx) {
  __shared__ int hist[256];
  __shared__ unsigned long long sh_prefix;
  __shared__ int sh_need;
  __shared__ int sort_buf[kMaxK];
  __shared__ unsigned long long cbuf[kCandSmem];
  __shared__ int sh_taken;
  const int64_t row = blockIdx.x;
  const int64_t n = row_visible(row, Q, q_pos0, m, N);
  int32_t* orow = idx + row * (int64_t)k;
  const int kk = (int)(n < k ? n : k);
  for (int j = kk + threadIdx.x; j < k; j += blockDim.x) orow[j] = -1;
  if (n <= k) {
    for (int j = threadIdx.x; j < kk; j += blockDim.x) orow[j] = j;
    return;
  }
  const int n_up = lr.counts[row * 2 + 0];
  const int n_cand = lr.counts[row * 2 + 1];
  const int need = kk - n_up;  // >= 1 by construction of the boundary digit
  const unsigned long long* cand = lr.cand + row * N;
  unsigned long long thr;
  const bool in_smem = n_cand <= kCandSmem;
  if (in_smem) {
    for (int j = threadIdx.x; j < n_cand; j += blockDim.x) cbuf[j] = cand[j];
    __syncthreads();
    thr = select_composite<true>(cbuf, n_cand, need, hist, &sh_prefix, &sh_need);
  } else {
    thr = select_composite<false>(cand, n_cand, need, hist, &sh_prefix, &sh_need);
  }
  // gather the kk indices
  const int32_t* sel = lr.selected + row * (int64_t)k;
  for (int j = threadIdx.x; j < n_up; j += blockDim.x) sort_buf[j] = sel[j];
  if (threadIdx.x == 0) sh_taken = n_up;
  __syncthreads();
  for (int j = threadIdx.x; j < n_cand; j += blockDim.x) {
    const unsigned long long x = in_smem ? cbuf[j] : cand[j];
    if (x >= thr) {
      const int pos = atomicAdd(&sh_taken, 1);
      sort_buf[pos] = (int)(~(uint32_t)(x & 0xffffffffull));
    }
  }
  __syncthreads();
  int P = 1;
  while (P < kk) P <<= 1;
  for (int j = kk + threadIdx.x; j < P; j += blockDim.x) sort_buf[j] = 0x7fffffff;
  __syncthreads();
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = threadIdx.x; t < P / 2; t += blockDim.x) {
        const int i = 2 * t - (t & (stride - 1));
        const int j = i + stride;
        const bool asc = (i & size) == 0;
        const int a = sort_buf[i], b = sort_buf[j];
        if ((a > b) == asc) {
          sort_buf[i] = b;
          sort_buf[j] = a;
        }
      }
      __syncthreads();
    }
  }
  for (int j = threadIdx.x; j < kk; j += blockDim.x) orow[j] = sort_buf[j];
}

bool use_long_rows(const csa_params& p, int Q, int64_t N) {
  const int64_t rows = (int64_t)p.B * Q;
  return N > kSmemRow && p.k <= kMaxK && rows < 256;
}

size_t long_rows_bytes(const csa_params& p, int Q, int64_t N, size_t* off) {
  const int64_t rows = (int64_t)p.B * Q;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t r = o;
    o += (bytes + 255) & ~(size_t)255;
    return r;
  };
  off[0] = take((size_t)rows * kBins * sizeof(int));
  off[1] = take((size_t)rows * 2 * sizeof(int));
  off[2] = take((size_t)rows * p.k * sizeof(int32_t));
  off[3] = take((size_t)rows * N * sizeof(unsigned long long));
  return o;
}

}  // namespace

size_t topk_workspace(const csa_params& p, int Q, int64_t N) {
  if (!use_long_rows(p, Q, N)) return 0;
  size_t off[4];
  return long_rows_bytes(p, Q, N, off);
}

int topk_launches(const csa_params& p, int Q, int64_t N) { return use_long_rows(p, Q, N) ? 3 : 1; }

cudaError_t launch_topk(const csa_params& p, const float* scores, int64_t q_pos0, int Q,
                        int64_t N, int32_t* idx, void* ws, cudaStream_t st) {
  const int64_t rows = (int64_t)p.B * Q;
  if (rows <= 0) return cudaSuccess;
  if (use_long_rows(p, Q, N)) {
    size_t off[4];
    const size_t bytes = long_rows_bytes(p, Q, N, off);
    char* w = reinterpret_cast<char*>(ws);
    LongRows lr{reinterpret_cast<int*>(w + off[0]), reinterpret_cast<int*>(w + off[1]),
                reinterpret_cast<int32_t*>(w + off[2]),
                reinterpret_cast<unsigned long long*>(w + off[3])};
    (void)bytes;
    cudaError_t e = cudaMemsetAsync(w, 0, off[2], st);  // histograms and counters
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int slices = (int)ceil_div(4 * sms, rows);
    const int64_t max_slices = ceil_div(N, 2048);
    if (slices > max_slices) slices = (int)max_slices;
    if (slices < 1) slices = 1;
    dim3 g((unsigned)slices, (unsigned)rows);
    topk_hist_kernel<<<g, 512, 0, st>>>(scores, q_pos0, Q, N, p.m, p.k, lr);
    topk_filter_kernel<<<g, 512, 0, st>>>(scores, q_pos0, Q, N, p.m, p.k, lr);
    topk_final_kernel<<<(unsigned)rows, 1024, 0, st>>>(q_pos0, Q, N, p.m, p.k, lr, idx);
    return cudaGetLastError();
  }
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
