// Step 3 of CSA: per-query top-k of the indexer scores.
//
// Sources: "一文搞懂 DeepSeek：从 V3 的 KV 压缩与 MoE，到 V4 的百万 token 上下文",
// section "V4 改进一：CSA 与 HCA" (keep the top-k highest-scoring entries);
// "DeepSeek-V4 详解" section 2.2 Step 3 (Top-1024).
//
// Exact radix select on order-preserving 32-bit keys of the fp32 scores
// (-0 folded onto +0): digit passes of 12, 12 and 8 bits from the most
// significant end (shared-memory histograms of 4096 bins, scanned by the whole
// block) find the key T of the kk-th largest score and how many of the entries equal
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
// the upper half of the fp32 key of the same value: two digit passes (12 and
// 4 bits), and half the bytes read per pass.
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

constexpr int kDigit = 12;  // digit width of the block-wide selects
constexpr int kBins = 1 << kDigit;

// The need-th largest of get(i), i < n, by a 1024-thread block, in digit
// passes from the top of 12 bits (the last one narrower), at most `passes`
// of them: returns the prefix found (the low bits not examined clear) and
// leaves in *sh_need how many keys with that prefix are still needed.  hist
// holds kBins counts; thread t scans bins from the top, kPer at a time
// (kPer * blockDim.x == kBins).
template <int kBits, int kPer = 4, typename Get>
__device__ uint32_t select12(Get get, int n, int need, int passes, int* hist, int* warp_sums,
                             uint32_t* sh_prefix, int* sh_need) {
  uint32_t prefix = 0, mask = 0;
  int hi = kBits;
  for (int pass = 0; pass < passes && hi > 0; ++pass) {
    const int w = hi >= kDigit ? kDigit : hi;
    const int shift = hi - w;
    const int nb = 1 << w;
    for (int j = threadIdx.x; j < nb; j += blockDim.x) hist[j] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const uint32_t x = get(i);
      if ((x & mask) == prefix) atomicAdd(&hist[(x >> shift) & (uint32_t)(nb - 1)], 1);
    }
    __syncthreads();
    int c[kPer], local = 0;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int b = nb - 1 - kPer * (int)threadIdx.x - q;
      c[q] = b >= 0 ? hist[b] : 0;
      local += c[q];
    }
    int total;
    const int above = BlockScan::run(local, warp_sums, &total);  // keys in higher bins
    if (above < need && above + local >= need) {
      int acc = above;
#pragma unroll
      for (int q = 0; q < kPer; ++q) {
        if (acc + c[q] >= need) {
          *sh_prefix = prefix | ((uint32_t)(nb - 1 - kPer * (int)threadIdx.x - q) << shift);
          *sh_need = need - acc;
          break;
        }
        acc += c[q];
      }
    }
    __syncthreads();
    prefix = *sh_prefix;
    need = *sh_need;
    mask |= (uint32_t)(nb - 1) << shift;
    hi = shift;
    __syncthreads();
  }
  return prefix;
}

// Keeps, in index order, every i < n with key(i) > T and the first need_eq
// with key(i) == T, calling put(pos, i) for the pos-th one kept (a 1024-thread
// block).  The 32 warps take contiguous segments: each counts its keys > T
// and == T by ballots, warp 0 turns the counts into output offsets, and each
// warp walks its segment again, writing at those offsets.
template <typename Key, typename Put>
__device__ void take_in_order(Key key, int n, uint32_t T, int need_eq, int* wcnt, Put put) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned lt = (1u << lane) - 1u;
  const int seg = (n + 31) / 32;
  const int s0 = min(n, warp * seg), s1 = min(n, s0 + seg);
  int gt = 0, eq = 0;
  for (int b = s0; b < s1; b += 32) {
    const int i = b + lane;
    const uint32_t x = i < s1 ? key(i) : 0u;
    gt += __popc(__ballot_sync(0xffffffffu, i < s1 && x > T));
    eq += __popc(__ballot_sync(0xffffffffu, i < s1 && x == T));
  }
  if (lane == 0) {
    wcnt[warp] = gt;
    wcnt[32 + warp] = eq;
  }
  __syncthreads();
  if (warp == 0) {
    const int g = wcnt[lane], e = wcnt[32 + lane];
    int e_incl = e;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, e_incl, o);
      if (lane >= o) e_incl += y;
    }
    const int e_before = e_incl - e;
    const int take = g + min(max(need_eq - e_before, 0), e);
    int t_incl = take;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t_incl, o);
      if (lane >= o) t_incl += y;
    }
    wcnt[lane] = t_incl - take;
    wcnt[32 + lane] = e_before;
  }
  __syncthreads();
  int pos = wcnt[warp], eq_seen = wcnt[32 + warp];
  for (int b = s0; b < s1; b += 32) {
    const int i = b + lane;
    const uint32_t x = i < s1 ? key(i) : 0u;
    const bool g = i < s1 && x > T, e = i < s1 && x == T;
    const unsigned be = __ballot_sync(0xffffffffu, e);
    const bool take = g || (e && eq_seen + __popc(be & lt) < need_eq);
    const unsigned bt = __ballot_sync(0xffffffffu, take);
    if (take) put(pos + __popc(bt & lt), i);
    pos += __popc(bt);
    eq_seen += __popc(be);
  }
}

template <bool kSmem, typename ST>
__global__ void __launch_bounds__(kThreads) topk_row_kernel(const ST* __restrict__ scores,
                                                            int64_t q_pos0, int Q, int64_t N,
                                                            int m, int k,
                                                            int32_t* __restrict__ idx) {
  __shared__ int hist[kBins];
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

  const uint32_t prefix = select12<ScoreKey<ST>::kBits>(
      [&](int s) { return key_at(s); }, (int)n, kk, 3, hist, warp_sums, &sh_prefix, &sh_need);
  const int need = sh_need;
  // prefix == key of the kk-th largest score; keep keys > prefix and the
  // first `need` keys == prefix in index order.
  take_in_order([&](int s) { return key_at(s); }, (int)n, prefix, need, hist,
                [&](int pos, int s) { orow[pos] = (int32_t)s; });
}


// ------------------------------------------------------------------------
// Long rows with few rows (decode: B rows of 10^5..10^6 entries), in three
// kernels over the order-preserving 32-bit keys:
//   A  sample: one CTA per row finds, from 4096 evenly spaced keys of the
//              row, the top 24 bits of the key of rank r = 4 k ns / n (two
//              12-bit digit passes); tau is that prefix with the low bits
//              clear, so at least r sampled keys are >= tau, and about 4k
//              keys of the row (one CTA per row: in every filter CTA of the
//              row the same select cost more than this launch);
//   B  filter: S CTAs per row; each warp compacts its contiguous part of the
//              row, in index order (ballots), into a list of the (key, index)
//              composites of its keys >= tau;
//   C  final:  one CTA per row; if at least kk keys reached tau the kk largest
//              of the row are all among them: the lists are copied into
//              shared memory, a radix select on their keys (12-bit digits)
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
constexpr int kFilterKeys = 16;     // keys in flight per lane in kernel B
constexpr int kMaxSlices = 256;     // slices x kWarpsB lists fit kernel C's shared memory
constexpr int kMaxLists = kMaxSlices * kWarpsB;
constexpr int kTargetCtas = 296;    // slices of all rows together: one wave of 2 x 148 CTAs

struct LongRows {
  int S;                     // slices per row (a power of two)
  int logL;                  // log2 of the lists per row, S * kWarpsB
  uint32_t* tau;             // [rows]
  int* cnt;                  // [rows][S * kWarpsB]
  unsigned long long* cand;  // [rows][N]: each warp's candidates from its part's start
};

__device__ __forceinline__ int64_t row_visible(int64_t row, int Q, int64_t q_pos0, int m, int64_t N) {
  const int i = (int)(row % Q);
  const int64_t nv = n_vis(q_pos0 + i, m);
  return nv < N ? nv : N;
}

// Start of list l of the 2^logL lists that split [0, n) (list 2^logL: n):
// nearly equal parts, each starting at a multiple of 4.
__device__ __forceinline__ int64_t list_begin(int64_t n, int logL, int l) {
  return l >= (1 << logL) ? n : (((n * l) >> logL) & ~(int64_t)3);
}

// The smallest fp32 value whose key is >= key (score_key is monotonic, so
// score_key(x) >= key exactly when x >= key_floor(key)).
__device__ __forceinline__ float key_floor(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// Four consecutive scores (index a multiple of 4) as fp32.
__device__ __forceinline__ float4 load4(const float* p, int64_t i) {
  return __ldg(reinterpret_cast<const float4*>(p + i));
}
__device__ __forceinline__ float4 load4(const uint16_t* p, int64_t i) {
  const uint2 w = __ldg(reinterpret_cast<const uint2*>(p + i));
  return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                     __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
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
  __shared__ int hist[kBins];
  __shared__ int warp_sums[32];
  __shared__ uint32_t sh_prefix;
  __shared__ int sh_need;
  const int64_t row = blockIdx.x;
  const int64_t n = row_visible(row, Q, q_pos0, m, N);
  if (n <= k) return;
  const int ns = n < kSample ? (int)n : kSample;
  const ST* srow = scores + row * N;
  // key j of the sample: entry floor(j n / ns) (ns = 4096 a power of two)
  for (int j = threadIdx.x; j < ns; j += blockDim.x)
    keys[j] = ScoreKey<ST>::at(srow, ns == kSample ? ((int64_t)j * n) >> 12 : (int64_t)j);
  __syncthreads();
  int64_t r = (4 * (int64_t)k * ns + n - 1) / n;
  if (r > ns) r = ns;
  if (r < 1) r = 1;
  const uint32_t tau = select12<ScoreKey<ST>::kBits>([&](int i) { return keys[i]; }, ns, (int)r, 2,
                                                     hist, warp_sums, &sh_prefix, &sh_need);
  if (threadIdx.x == 0) lr.tau[row] = tau;
}

// kVec: the row length is a multiple of 4 and the scores 16-byte aligned,
// so a lane loads four consecutive scores at once; the comparison with tau
// is made on the fp32 values (x >= key_floor(tau) exactly when its key is
// >= tau), the key computed for the candidates only.
template <typename ST, bool kVec>
__global__ void __launch_bounds__(512, 2) topk_filter_kernel(const ST* __restrict__ scores,
                                                          int64_t q_pos0, int Q, int64_t N, int m,
                                                          int k, LongRows lr) {
  const int64_t row = blockIdx.y;
  const int s = blockIdx.x;
  const int64_t n = row_visible(row, Q, q_pos0, m, N);
  if (n <= k) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int l = s * kWarpsB + warp;
  const int64_t w0 = list_begin(n, lr.logL, l), w1 = list_begin(n, lr.logL, l + 1);
  const ST* srow = scores + row * N;
  unsigned long long* cand = lr.cand + row * N + w0;
  constexpr int kU = kFilterKeys / 4;  // float4 loads in flight per lane
  const uint32_t tau = __ldcg(lr.tau + row);
  const float tf = key_floor(ScoreKey<ST>::kBits == 32 ? tau : tau << 16);
  const unsigned lt_mask = (1u << lane) - 1u;
  // candidate: key above, complemented index below (positions fit 32 bits)
  int nc = 0;
  if (kVec) {
    // lane L holds the 16 scores base + 16 L .. base + 16 L + 15 (kU float4
    // loads); its mask of those >= tau, popcounts scanned over the warp, give
    // each lane's place in the list; a candidate's key is re-read (an L1 hit)
    for (int64_t base = w0; base < w1; base += 32 * kFilterKeys) {
      const int64_t i0 = base + kFilterKeys * lane;
      const bool full = base + 32 * kFilterKeys <= w1;  // warp-uniform
      float4 v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u)
        v[u] = (full || i0 + 4 * u < w1) ? load4(srow, i0 + 4 * u) : make_float4(0.f, 0.f, 0.f, 0.f);
      uint32_t bits = 0;
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        bits |= (v[u].x >= tf ? 1u : 0u) << (4 * u);
        bits |= (v[u].y >= tf ? 1u : 0u) << (4 * u + 1);
        bits |= (v[u].z >= tf ? 1u : 0u) << (4 * u + 2);
        bits |= (v[u].w >= tf ? 1u : 0u) << (4 * u + 3);
      }
      if (!full) {
        const int64_t left = w1 - i0;
        bits &= left >= kFilterKeys ? 0xffffffffu : (left > 0 ? (1u << left) - 1u : 0u);
      }
      const int c = __popc(bits);
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      int pos = nc + incl - c;
      while (bits) {
        const int e = __ffs(bits) - 1;
        bits &= bits - 1u;
        const int64_t i = i0 + e;
        cand[pos++] = ((unsigned long long)ScoreKey<ST>::at(srow, i) << 32) |
                      (unsigned long long)(~(uint32_t)i);
      }
      nc += __shfl_sync(0xffffffffu, incl, 31);
    }
  } else {
    for (int64_t base = w0; base < w1; base += kFilterKeys * 32) {
      uint32_t key[kFilterKeys];
#pragma unroll
      for (int j = 0; j < kFilterKeys; ++j) {
        const int64_t t = base + j * 32 + lane;
        key[j] = t < w1 ? ScoreKey<ST>::at(srow, t) : 0u;
      }
#pragma unroll
      for (int j = 0; j < kFilterKeys; ++j) {
        const int64_t t = base + j * 32 + lane;
        const unsigned b = __ballot_sync(0xffffffffu, t < w1 && key[j] >= tau);
        if ((b >> lane) & 1u)
          cand[nc + __popc(b & lt_mask)] =
              ((unsigned long long)key[j] << 32) | (unsigned long long)(~(uint32_t)t);
        nc += __popc(b);
      }
    }
  }
  if (lane == 0) lr.cnt[row * lr.S * kWarpsB + l] = nc;
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
  int* off = reinterpret_cast<int*>(cbuf + kCandSmem);     // [kMaxLists + 1]
  int* hist = off + kMaxLists + 1;                         // [kBins]
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
    if (threadIdx.x == 0) {
      sh_nc = c;
      off[L] = c;
    }
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
    take_in_order([&](int t) { return ScoreKey<ST>::at(srow, t); }, (int)n, T, need_eq, hist,
                  [&](int pos, int t) { orow[pos] = (int32_t)t; });
    return;
  }
  // list l (slice l / kWarpsB, warp l % kWarpsB of kernel B) covers
  // [list_begin(l), list_begin(l + 1)) of the row
  auto list_start = [&](int l) -> int64_t { return list_begin(n, lr.logL, l); };
  auto cand_at = [&](int64_t f) -> unsigned long long {
    const int l = find_list(off, L, (int)f);
    return __ldcg(lr.cand + row * N + list_start(l) + (f - off[l]));
  };
  const bool in_smem = nc <= kCandSmem;
  if (in_smem) {
    // the lists (each contiguous in cand) copied by cp.async, all of them in
    // flight at once: a warp per list when they are long, a thread per list
    // when they are short (few rows split into many slices: up to 4096 lists
    // of a few candidates each)
    auto copy = [&](int l, int e0, int step) {
      const int o = off[l], c = off[l + 1] - o;
      const unsigned long long* src = lr.cand + row * N + list_start(l);
      for (int e = e0; e < c; e += step) {
        const uint32_t dst = (uint32_t)__cvta_generic_to_shared(cbuf + o + e);
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src + e) : "memory");
      }
    };
    if (nc >= 16 * L) {
      for (int l = threadIdx.x >> 5; l < L; l += 32) copy(l, threadIdx.x & 31, 32);
    } else {
      for (int l = threadIdx.x; l < L; l += blockDim.x) copy(l, 0, 1);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  }
  __syncthreads();
  // the key of the kk-th largest candidate, and how many keys equal to it
  // are needed: the lowest-index ones (candidates are in index order)
  const uint32_t T =
      in_smem ? select12<ScoreKey<ST>::kBits>([&](int i) { return (uint32_t)(cbuf[i] >> 32); }, nc,
                                              kk, 3, hist, warp_sums, &sh_prefix32, &sh_need)
              : radix_select<uint32_t, ScoreKey<ST>::kBits>(
                    [&](int64_t i) { return (uint32_t)(cand_at(i) >> 32); }, nc, kk, hist,
                    &sh_prefix32, &sh_need);
  const int need_eq = sh_need;
  auto cand = [&](int f) { return in_smem ? cbuf[f] : cand_at(f); };
  take_in_order([&](int f) { return (uint32_t)(cand(f) >> 32); }, nc, T, need_eq, hist,
                [&](int pos, int f) { orow[pos] = (int32_t)(~(uint32_t)(cand(f) & 0xffffffffull)); });
}

bool use_long_rows(const csa_params& p, int Q, int64_t N) {
  const int64_t rows = (int64_t)p.B * Q;
  return N > kSmemRow && p.k <= kMaxK && rows < 256;
}

// A power of two: no second, partial wave of kernel B
int long_rows_slices(const csa_params& p, int Q, int64_t N) {
  const int64_t rows = (int64_t)p.B * Q;
  int64_t lim = kTargetCtas / rows;
  const int64_t cap = ceil_div(N, 2048);
  if (lim > cap) lim = cap;
  if (lim > kMaxSlices) lim = kMaxSlices;
  int S = 1;
  while (2 * S <= lim) S *= 2;
  return S;
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
    lr.logL = 0;
    while ((1 << lr.logL) < lr.S * kWarpsB) ++lr.logL;
    lr.tau = reinterpret_cast<uint32_t*>(w + off[0]);
    lr.cnt = reinterpret_cast<int*>(w + off[1]);
    lr.cand = reinterpret_cast<unsigned long long*>(w + off[2]);
    topk_sample_kernel<ST><<<(unsigned)rows, 1024, 0, st>>>(scores, q_pos0, Q, N, p.m, p.k, lr);
    dim3 g((unsigned)lr.S, (unsigned)rows);
    if (N % 4 == 0 && reinterpret_cast<uintptr_t>(scores) % 16 == 0)
      topk_filter_kernel<ST, true><<<g, 32 * kWarpsB, 0, st>>>(scores, q_pos0, Q, N, p.m, p.k, lr);
    else
      topk_filter_kernel<ST, false><<<g, 32 * kWarpsB, 0, st>>>(scores, q_pos0, Q, N, p.m, p.k, lr);
    const size_t smem = kCandSmem * sizeof(unsigned long long) + (kMaxLists + 1 + kBins) * sizeof(int);
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
