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
//
// Scores stored in bf16 ("一文搞懂 DeepSeek" section "V4 的其他升级": bf16
// index scores make the top-k selection twice as fast) take 16-bit keys,
// the upper half of the fp32 key of the same value: two digit passes, and
// half the bytes read per pass.
#include "common.cuh"

namespace csa {
namespace {

// Order-preserving key of score i of a row: fp32 scores give 32-bit keys,
// bf16 scores (bit patterns) 16-bit keys.
template <typename ST>
struct ScoreKey;
template <>
struct ScoreKey<float> {
  static constexpr int kBits = 32;
  __device__ static __forceinline__ uint32_t at(const float* p, int64_t i) {
    return score_key(__ldg(p + i));
  }
};
template <>
struct ScoreKey<uint16_t> {
  static constexpr int kBits = 16;
  __device__ static __forceinline__ uint32_t at(const uint16_t* p, int64_t i) {
    return score_key(__uint_as_float((uint32_t)__ldg(p + i) << 16)) >> 16;
  }
};

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

template <bool kSmem, typename ST>
__global__ void __launch_bounds__(kThreads) topk_row_kernel(const ST* __restrict__ scores,
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
  const ST* srow = scores + row * N;
  int32_t* orow = idx + row * (int64_t)k;

  for (int j = kk + threadIdx.x; j < k; j += blockDim.x) orow[j] = -1;
  if (kk == n) {  // everything visible is kept
    for (int j = threadIdx.x; j < kk; j += blockDim.x) orow[j] = j;
    return;
  }
  if (kSmem) {
    for (int64_t s = threadIdx.x; s < n; s += blockDim.x) row_keys[s] = ScoreKey<ST>::at(srow, s);
  }
  auto key_at = [&](int64_t s) -> uint32_t {
    return kSmem ? row_keys[s] : ScoreKey<ST>::at(srow, s);
  };

  uint32_t prefix = 0, mask = 0;
  int need = kk;
  for (int shift = ScoreKey<ST>::kBits - 8; shift >= 0; shift -= 8) {
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
// Long rows with few rows (decode: B rows of 10^5..10^6 entries), in three
// kernels over the order-preserving 32-bit keys:
//   A  sample: one CTA per row radix-selects, from 4096 evenly spaced keys of
//              the row, the key tau of rank r = 4 k ns / n: about 4k keys of
//              the row are >= tau;
//   B  filter: S CTAs per row; each warp compacts its contiguous part of the
//              row, in index order (ballots), into a list of the (key, index)
//              composites of its keys >= tau;
//   C  final:  one CTA per row; if at least kk keys reached tau the kk largest
//              of the row are all among them: a radix select on their keys
//              gives the key T of the kk-th largest and how many keys equal to
//              T are needed, and one pass over the candidates (already in
//              index order) keeps every key > T and the lowest-index keys == T.
//              If fewer reached tau (a sample far from the row, never seen on
//              these workloads), the CTA selects over the whole row.
// A histogram of the raw key bits would do the same in one pass, but scores
// often share a few binades, so its atomics pile up on a handful of bins.
constexpr int kMaxK = 4096;         // largest k of this path
constexpr int kSample = 4096;       // keys sampled per row
constexpr int kCandSmem = 8192;     // candidates kernel C keeps in shared memory
constexpr int kWarpsB = 16;         // warps of kernel B (512 threads)
constexpr int kMaxSlices = 256;     // slices x kWarpsB lists fit kernel C's shared memory
constexpr int kMaxLists = kMaxSlices * kWarpsB;
constexpr int kTargetCtas = 592;    // slices of all rows together: one wave of 4 x 148 CTAs

struct LongRows {
  int S;                     // slices per row
  uint32_t* tau;             // [rows]
  int* cnt;                  // [rows][S * kWarpsB]
  unsigned long long* cand;  // [rows][N]: each warp's candidates from its part's start
};

__device__ __forceinline__ int64_t row_visible(int64_t row, int Q, int64_t q_pos0, int m, int64_t N) {
  const int i = (int)(row % Q);
  const int64_t nv = n_vis(q_pos0 + i, m);
  return nv < N ? nv : N;
}

// part `part` of `parts` equal parts of [0, n)
__device__ __forceinline__ void part_range(int64_t n, int parts, int part, int64_t* p0, int64_t* p1) {
  *p0 = n * part / parts;
  *p1 = n * (part + 1) / parts;
}

// The need-th largest of get(i), i < n, by 8-bit radix passes from the top
// (block-wide; values with bits above `bits` ignored).  Key type U.
template <typename U, int kBits, typename Get>
__device__ U radix_select(Get get, int64_t n, int need, int* hist, U* sh_prefix, int* sh_need) {
  U prefix = 0, mask = 0;
  for (int shift = kBits - 8; shift >= 0; shift -= 8) {
    for (int j = threadIdx.x; j < 256; j += blockDim.x) hist[j] = 0;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
      const U x = get(i);
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
        const unsigned hit = __ballot_sync(0xffffffffu, acc_above + incl >= need);
        if (hit) {
          const int l = __ffs(hit) - 1;
          const int excl = __shfl_sync(0xffffffffu, incl - c, l);
          if (lane == 0) {
            *sh_prefix = prefix | ((U)(chunk * 32 + 31 - l) << shift);
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
    mask |= (U)255 << shift;
    __syncthreads();
  }
  return prefix;
}

template <typename ST>
__global__ void __launch_bounds__(1024) topk_sample_kernel(const ST* __restrict__ scores,
                                                           int64_t q_pos0, int Q, int64_t N, int m,
                                                           int k, LongRows lr) {
  __shared__ uint32_t keys[kSample];
  __shared__ int hist[256];
  __shared__ uint32_t sh_prefix;
  __shared__ int sh_need;
  const int64_t row = blockIdx.x;
  const int64_t n = row_visible(row, Q, q_pos0, m, N);
  if (n <= k) return;
  const int ns = n < kSample ? (int)n : kSample;
  const ST* srow = scores + row * N;
  for (int j = threadIdx.x; j < ns; j += blockDim.x)
    keys[j] = ScoreKey<ST>::at(srow, (int64_t)j * n / ns);
  __syncthreads();
  int64_t r = (4 * (int64_t)k * ns + n - 1) / n;
  if (r > ns) r = ns;
  if (r < 1) r = 1;
  const uint32_t tau = radix_select<uint32_t, ScoreKey<ST>::kBits>(
      [&](int64_t i) { return keys[i]; }, ns, (int)r, hist, &sh_prefix, &sh_need);
  if (threadIdx.x == 0) lr.tau[row] = tau;
}

template <typename ST>
__global__ void __launch_bounds__(512, 4) topk_filter_kernel(const ST* __restrict__ scores,
                                                          int64_t q_pos0, int Q, int64_t N, int m,
                                                          int k, LongRows lr) {
  const int64_t row = blockIdx.y;
  const int s = blockIdx.x;
  const int64_t n = row_visible(row, Q, q_pos0, m, N);
  if (n <= k) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t tau = __ldcg(lr.tau + row);
  int64_t s0, s1, w0, w1;
  part_range(n, lr.S, s, &s0, &s1);
  part_range(s1 - s0, kWarpsB, warp, &w0, &w1);
  w0 += s0;
  w1 += s0;
  // positions within the row fit 32 bits (rows are < 2^31 entries)
  const ST* wrow = scores + row * N + w0;
  unsigned long long* cand = lr.cand + row * N + w0;
  const int len = (int)(w1 - w0), pos0 = (int)w0;
  const unsigned lt_mask = (1u << lane) - 1u;
  int nc = 0;
  for (int base = 0; base < len; base += 8 * 32) {
    uint32_t key[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int t = base + j * 32 + lane;
      key[j] = t < len ? ScoreKey<ST>::at(wrow, t) : 0u;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int t = base + j * 32 + lane;
      const unsigned b = __ballot_sync(0xffffffffu, t < len && key[j] >= tau);
      if ((b >> lane) & 1u)
        cand[nc + __popc(b & lt_mask)] =
            ((unsigned long long)key[j] << 32) | (unsigned long long)(~(uint32_t)(pos0 + t));
      nc += __popc(b);
    }
  }
  if (lane == 0) lr.cnt[row * lr.S * kWarpsB + s * kWarpsB + warp] = nc;
}

// List holding flat position f of lists that start at off[0..L) (ascending).
__device__ __forceinline__ int find_list(const int* off, int L, int f) {
  int lo = 0, hi = L - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= f) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Exclusive prefix of cnt[0..L) into off[0..L) (shared), L <= kMaxLists, by a
// 1024-thread block; returns the total.
__device__ int list_offsets(const int* cnt, int L, int* off, int* warp_sums) {
  constexpr int kPer = kMaxLists / 1024;
  const int l0 = threadIdx.x * kPer;
  int v[kPer], local = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    v[j] = l0 + j < L ? __ldcg(cnt + l0 + j) : 0;
    local += v[j];
  }
  int total;
  int acc = BlockScan::run(local, warp_sums, &total);
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    if (l0 + j < L) off[l0 + j] = acc;
    acc += v[j];
  }
  return total;
}

template <typename ST>
__global__ void __launch_bounds__(1024) topk_final_kernel(const ST* __restrict__ scores,
                                                          int64_t q_pos0, int Q, int64_t N, int m,
                                                          int k, LongRows lr,
                                                          int32_t* __restrict__ idx) {
  extern __shared__ unsigned long long dsm[];
  unsigned long long* cbuf = dsm;                          // [kCandSmem]
  int* off = reinterpret_cast<int*>(cbuf + kCandSmem);     // [kMaxLists]
  __shared__ int hist[256];
  __shared__ int warp_sums[32];
  __shared__ unsigned long long sh_prefix64;
  __shared__ uint32_t sh_prefix32;
  __shared__ int sh_need, sh_nc;
  const int64_t row = blockIdx.x;
  const int64_t n = row_visible(row, Q, q_pos0, m, N);
  int32_t* orow = idx + row * (int64_t)k;
  const int kk = (int)(n < k ? n : k);
  for (int j = kk + threadIdx.x; j < k; j += blockDim.x) orow[j] = -1;
  if (n <= k) {
    for (int j = threadIdx.x; j < kk; j += blockDim.x) orow[j] = j;
    return;
  }
  const int S = lr.S, L = S * kWarpsB;
  {
    const int c = list_offsets(lr.cnt + row * L, L, off, warp_sums);
    if (threadIdx.x == 0) sh_nc = c;
  }
  __syncthreads();
  const int nc = sh_nc;
  const ST* srow = scores + row * N;
  if (nc < kk) {
    // fewer than kk keys reached tau: exact select over the whole row (the
    // kk-th largest key, then every larger key and the lowest-index equal
    // ones, in index order)
    const uint32_t T = radix_select<uint32_t, ScoreKey<ST>::kBits>(
        [&](int64_t i) { return ScoreKey<ST>::at(srow, i); }, n, kk, hist, &sh_prefix32, &sh_need);
    const int need_eq = sh_need;  // keys equal to T still needed
    int taken = 0, eq_seen = 0;
    for (int64_t base = 0; base < n; base += blockDim.x) {
      const int64_t t = base + threadIdx.x;
      const uint32_t kx = t < n ? ScoreKey<ST>::at(srow, t) : 0u;
      const int gt = (t < n && kx > T) ? 1 : 0;
      const int eq = (t < n && kx == T) ? 1 : 0;
      int eq_tot, take_tot;
      const int eq_rank = eq_seen + BlockScan::run(eq, warp_sums, &eq_tot);
      const int take = gt | (eq & (eq_rank < need_eq ? 1 : 0));
      const int pos = taken + BlockScan::run(take, warp_sums, &take_tot);
      if (take) orow[pos] = (int32_t)t;
      taken += take_tot;
      eq_seen += eq_tot;
    }
    return;
  }
  // list l covers [list_start(l), ...) of the row: slice l / kWarpsB, warp part l % kWarpsB
  auto list_start = [&](int l) -> int64_t {
    int64_t s0, s1, w0, w1;
    part_range(n, S, l / kWarpsB, &s0, &s1);
    part_range(s1 - s0, kWarpsB, l % kWarpsB, &w0, &w1);
    return s0 + w0;
  };
  auto cand_at = [&](int64_t f) -> unsigned long long {
    const int l = find_list(off, L, (int)f);
    return __ldcg(lr.cand + row * N + list_start(l) + (f - off[l]));
  };
  const bool in_smem = nc <= kCandSmem;
  if (in_smem)
    for (int f = threadIdx.x; f < nc; f += blockDim.x) cbuf[f] = cand_at(f);
  __syncthreads();
  // the key of the kk-th largest candidate, and how many keys equal to it
  // are needed: the lowest-index ones (candidates are in index order)
  const uint32_t T = radix_select<uint32_t, ScoreKey<ST>::kBits>(
      [&](int64_t i) { return (uint32_t)((in_smem ? cbuf[i] : cand_at(i)) >> 32); }, nc, kk, hist,
      &sh_prefix32, &sh_need);
  const int need_eq = sh_need;
  int taken = 0, eq_seen = 0;
  for (int base = 0; base < nc; base += blockDim.x) {
    const int f = base + threadIdx.x;
    unsigned long long x = 0;
    if (f < nc) x = in_smem ? cbuf[f] : cand_at(f);
    const uint32_t kx = (uint32_t)(x >> 32);
    const int gt = (f < nc && kx > T) ? 1 : 0;
    const int eq = (f < nc && kx == T) ? 1 : 0;
    int eq_tot, take_tot;
    const int eq_rank = eq_seen + BlockScan::run(eq, warp_sums, &eq_tot);
    const int take = gt | (eq & (eq_rank < need_eq ? 1 : 0));
    const int pos = taken + BlockScan::run(take, warp_sums, &take_tot);
    if (take) orow[pos] = (int32_t)(~(uint32_t)(x & 0xffffffffull));
    taken += take_tot;
    eq_seen += eq_tot;
  }
}

bool use_long_rows(const csa_params& p, int Q, int64_t N) {
  const int64_t rows = (int64_t)p.B * Q;
  return N > kSmemRow && p.k <= kMaxK && rows < 256;
}

int long_rows_slices(const csa_params& p, int Q, int64_t N) {
  const int64_t rows = (int64_t)p.B * Q;
  int64_t S = kTargetCtas / rows;  // no second, partial wave
  const int64_t cap = ceil_div(N, 2048);
  if (S > cap) S = cap;
  if (S > kMaxSlices) S = kMaxSlices;
  return S < 1 ? 1 : (int)S;
}

// Workspace layout; off[0..2] receive the offsets of the fields of LongRows.
size_t long_rows_bytes(const csa_params& p, int Q, int64_t N, size_t* off) {
  const int64_t rows = (int64_t)p.B * Q;
  const int S = long_rows_slices(p, Q, N);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t r = o;
    o += (bytes + 255) & ~(size_t)255;
    return r;
  };
  off[0] = take((size_t)rows * sizeof(uint32_t));                 // tau
  off[1] = take((size_t)rows * S * kWarpsB * sizeof(int));        // cnt
  off[2] = take((size_t)rows * N * sizeof(unsigned long long));   // cand
  return o;
}

}  // namespace

size_t topk_workspace(const csa_params& p, int Q, int64_t N) {
  if (!use_long_rows(p, Q, N)) return 0;
  size_t off[3];
  return long_rows_bytes(p, Q, N, off);
}

int topk_launches(const csa_params& p, int Q, int64_t N) { return use_long_rows(p, Q, N) ? 3 : 1; }

namespace {

template <typename ST>
cudaError_t launch_topk_t(const csa_params& p, const ST* scores, int64_t q_pos0, int Q, int64_t N,
                          int32_t* idx, void* ws, cudaStream_t st) {
  const int64_t rows = (int64_t)p.B * Q;
  if (rows <= 0) return cudaSuccess;
  if (use_long_rows(p, Q, N)) {
    size_t off[3];
    long_rows_bytes(p, Q, N, off);
    char* w = reinterpret_cast<char*>(ws);
    LongRows lr;
    lr.S = long_rows_slices(p, Q, N);
    lr.tau = reinterpret_cast<uint32_t*>(w + off[0]);
    lr.cnt = reinterpret_cast<int*>(w + off[1]);
    lr.cand = reinterpret_cast<unsigned long long*>(w + off[2]);
    topk_sample_kernel<ST><<<(unsigned)rows, 1024, 0, st>>>(scores, q_pos0, Q, N, p.m, p.k, lr);
    dim3 g((unsigned)lr.S, (unsigned)rows);
    topk_filter_kernel<ST><<<g, 32 * kWarpsB, 0, st>>>(scores, q_pos0, Q, N, p.m, p.k, lr);
    const size_t smem = kCandSmem * sizeof(unsigned long long) + kMaxLists * sizeof(int);
    cudaError_t e = cudaFuncSetAttribute(topk_final_kernel<ST>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    topk_final_kernel<ST><<<(unsigned)rows, 1024, smem, st>>>(scores, q_pos0, Q, N, p.m, p.k, lr,
                                                             idx);
    return cudaGetLastError();
  }
  if (N <= kSmemRow) {
    size_t smem = (size_t)N * sizeof(uint32_t);
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(topk_row_kernel<true, ST>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    topk_row_kernel<true, ST><<<(unsigned)rows, kThreads, smem, st>>>(scores, q_pos0, Q, N, p.m,
                                                                     p.k, idx);
  } else {
    topk_row_kernel<false, ST><<<(unsigned)rows, kThreads, 0, st>>>(scores, q_pos0, Q, N, p.m, p.k,
                                                                   idx);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_topk(const csa_params& p, const void* scores, bool bf16, int64_t q_pos0, int Q,
                        int64_t N, int32_t* idx, void* ws, cudaStream_t st) {
  if (bf16)
    return launch_topk_t(p, reinterpret_cast<const uint16_t*>(scores), q_pos0, Q, N, idx, ws, st);
  return launch_topk_t(p, reinterpret_cast<const float*>(scores), q_pos0, Q, N, idx, ws, st);
}

}  // namespace csa
