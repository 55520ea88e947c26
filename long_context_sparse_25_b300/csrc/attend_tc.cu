// Tensor-core path of steps 4 / 5 (CSA sparse MQA, HCA dense MQA, and the
// raw-token variant of CSA): tcgen05 MMAs with TMEM accumulators, key rows
// gathered (per-lane cp.async, or TMA boxes for runs of consecutive rows)
// into a ring of 128-byte-swizzled shared-memory chunks.
//
//   o[b,i,h,:] = sum_j softmax_j(scale * q[b,i,h,:] . K_j) * K_j[0:D_v]
//
// Sources: "一文搞懂 DeepSeek：从 V3 的 KV 压缩与 MoE，到 V4 的百万 token 上下文",
// section "V4 改进一：CSA 与 HCA" (selected entries plus a sliding window of
// raw KV, one KV shared by all heads: MQA; HCA attends densely) and section
// "V3 看家本领一：MLA" (the value is the latent, the decoupled RoPE key only
// enters the score); "DeepSeek-V4 详解" section 2.2 Steps 3-4 (bf16, 128
// heads; the selected blocks stand for their original tokens) and section 2.3
// Step 2.
//
// Key lists.  Entries: the selected entries, then the raw window.  Dense
// (HCA): every visible entry, then the window.  Raw blocks: the m raw tokens
// of every selected entry's block, then the window.
//
// Mapping.  The 128 heads of one query are the MMA's M side, so one shared
// key row feeds every head.  A 128 x 512 fp32 output accumulator alone fills
// all 512 TMEM columns, so a work item owns one half of the value dims (256
// columns) and computes the 128 x 128 score tile S = Q K^T itself.  TMEM: two
// S buffers (columns 0-255) and O (columns 256-511).  After the softmax reads
// S it writes P (bf16 pairs) over the score columns it has read, and P . V
// takes A from TMEM.
//
// Persistent CTAs.  A launch enumerates work items (query row, value half,
// split of the key list); each CTA takes a contiguous range of them and runs
// them back to back through one pipeline: the next item's score tiles are
// computed while the softmax warps drain the previous item's O, and Q (the
// query's 128 x D_qk rows, loaded by TMA, a barrier per 16 KB chunk) is
// loaded once for all the items of a query that follow one another (both
// value halves, every split).  Split boundaries depend on the key-list length
// only, never on the batch, so results are batch-invariant.
//
// Gathers.  Three producer warps fill the ring: each lane gathers 16-byte
// units of its rows with cp.async, which arrive on the chunk's barrier by
// themselves once they land.  A tile of 128 consecutive valid entries (HCA)
// or of window rows is one TMA box per chunk instead, issued by one thread
// that accounts for every producer's arrival.  For every tile the producers issue
// the D_qk/64 key chunks of that tile, then the D_v/128 value chunks of the
// previous tile (the ring is too small to keep them from the score pass).
//
// Mixed-precision caches (e4m3 nope dims with a row scale c_j, bf16 RoPE
// dims): QK^T runs on the codes themselves, which are exact in bf16, and on
// the RoPE dims divided by the row scale (split exactly into a bf16 high and
// low part, two ring slots that meet the same Q chunk), so the tile holds
// S'_j = q_nope . code_j + q_rope . (rope_j / c_j) and the softmax takes
// S_j = c_j S'_j.  P . V runs on the codes with c_j folded into P, split
// exactly into a bf16 high and low part (two MMAs per K step).
//
// Softmax: one thread per head row, log2 domain, running maximum raised only
// when a tile's maximum exceeds it by more than 2^8 (then O and the running
// sum are rescaled); P = 2^(x - m) <= 2^8 fits bf16 and fp32 comfortably.
//
// Roles: warps 0-2 producers, warp 3 TMEM allocator + MMA issuer (one
// thread; descriptors advanced by constant offsets), warps 4-7 softmax and
// output.  Every mbarrier wait is bounded; a timeout is recorded in a device
// error word, every other wait then gives up, each CTA lets its own copies
// and MMAs in flight land, and the kernel returns.
#include <cudaTypedefs.h>

#include <cstring>
#include <type_traits>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace csa {

namespace {

__device__ int g_attend_tc_error = 0;
__device__ int g_attend_never_set = 0;  // the test aid's flag: nothing sets it

constexpr int kT = 128;              // keys per tile
constexpr int kRing = 5;             // key chunk slots
constexpr uint32_t kChunk = 16384;   // 128 rows x 128 bytes
constexpr int kMaxQChunks = 9;       // D_qk <= 576
constexpr float kRescaleLog2 = 8.f;  // rescale when the maximum grows by more than 2^8
constexpr int kProdWarps = 3;        // warps 0-2: key-chunk producers
constexpr int kProd = kProdWarps * 32;
constexpr int kUnits = (kChunk / 16 + kProd - 1) / kProd;  // 16-byte units per producer thread
constexpr int kHalfUnits = (kUnits + 1) / 2;                  // mixed caches: loads in flight at once
constexpr int kMmaWarp = 3;          // warp 3: TMEM allocator + MMA issuer
constexpr int kThreads = 256;        // + warps 4-7: softmax / output

enum KeyMode { kEntries = kAttendEntries, kDense = kAttendDense, kRawBlocks = kAttendRawBlocks };

struct AttArgs {
  int B, Q, H, D_qk, D_v, k, W, m;
  int nc;    // D_qk / 64: Q chunks
  int nsc;   // key chunk loads per tile for QK^T (mixed: nope/64 codes + 2 per RoPE chunk)
  int nvc;   // D_v / 128: value chunks per half
  int mode;  // KeyMode
  int e4m3;
  int splits, tps;  // splits per (query, half); tiles per split
  int stall;        // test aid: CTA 0's MMA issuer first waits on a flag that nothing sets
  int64_t n_items;  // B * Q * 2 * splits
  int64_t N, kv_rows, raw_rows, raw_pos0, q_pos0;
  float c_log2;  // scale * log2(e)
  const int32_t* idx;
  const uint16_t* kv16;  // bf16 entries: [B, kv_rows, D_qk]
  const uint8_t* codes;  // e4m3 entries: [B, kv_rows, nope]
  const uint16_t* rope;  // [B, kv_rows, D_qk - nope]
  const float* kscale;   // [B, kv_rows]
  int nope;
  const uint16_t* raw16;  // raw rows [B, raw_rows, D_qk]
  void* out;
  int out_f32;
  float* part;  // splits > 1: [rows*H][splits][D_v] unnormalised O
  float* ml;    // splits > 1: [rows*H][splits][2] (max, sum), log2 domain
};

struct KeyList {
  int64_t t, lo;
  int kd;     // slots of the first part with meaning (k, k*m, or the visible entries)
  int k_ent;  // first part rounded up to a multiple of 4 (gather groups never straddle)
  int w_len;  // window tokens
  int len;    // k_ent + w_len
};

__device__ __forceinline__ KeyList key_list(const AttArgs& a, int i) {
  KeyList kl;
  kl.t = a.q_pos0 + i;
  kl.lo = kl.t - a.W + 1 > 0 ? kl.t - a.W + 1 : 0;
  kl.w_len = a.W > 0 ? (int)(kl.t - kl.lo + 1) : 0;
  if (a.mode == kDense) {
    int64_t nv = n_vis(kl.t, a.m);
    kl.kd = (int)(nv < a.N ? nv : a.N);
  } else if (a.mode == kRawBlocks) {
    kl.kd = a.k * a.m;
  } else {
    kl.kd = a.k;
  }
  kl.k_ent = (kl.kd + 3) & ~3;
  kl.len = kl.k_ent + kl.w_len;
  return kl;
}

// One work item: (query row, value half, split) and its run of tiles.
struct Item {
  int64_t qrow;  // b * Q + i
  int b, i, half, split;
  KeyList kl;
  int tile0, n;  // first tile of the split, tiles in it (0: no key)
};

__device__ __forceinline__ Item make_item(const AttArgs& a, int64_t id) {
  Item it;
  it.split = (int)(id % a.splits);
  it.half = (int)((id / a.splits) & 1);
  it.qrow = id / ((int64_t)a.splits * 2);
  it.i = (int)(it.qrow % a.Q);
  it.b = (int)(it.qrow / a.Q);
  it.kl = key_list(a, it.i);
  const int n_all = (it.kl.len + kT - 1) / kT;
  it.tile0 = it.split * a.tps;
  int n = n_all - it.tile0;
  if (n > a.tps) n = a.tps;
  if (n < 0) n = 0;
  it.n = n;
  return it;
}

// Source row of key slot j of a query's list: an entry row (entry cache) or a
// raw row (window, or a raw-token block).  Empty slots point at a valid row
// of the same kind (row 0) and are masked in the softmax.
struct SlotSrc {
  int64_t row;  // row index into the entry cache or into the raw rows
  bool raw;
  bool valid;
};

// The index-list word of key slot j (only selected slots read the list; the
// others return 0 and are resolved by slot_src from the slot number).
__device__ __forceinline__ int32_t slot_word(const AttArgs& a, const KeyList& kl, int64_t qrow,
                                             int j) {
  if (a.mode == kDense || j >= kl.kd) return 0;
  if (j >= kl.k_ent && a.W > 0) return 0;
  const int e = a.mode == kRawBlocks ? j / a.m : j;
  return a.idx[qrow * (int64_t)a.k + e];
}

// `word`: slot_word of the same slot (fetched ahead of use).
__device__ __forceinline__ SlotSrc slot_src(const AttArgs& a, const KeyList& kl, int b, int j,
                                            int32_t word) {
  SlotSrc r;
  if (j < kl.k_ent || a.W == 0) {
    int64_t e = 0;
    bool v = false;
    if (j < kl.kd) {
      if (a.mode == kDense) {
        e = j;
        v = true;
      } else {
        e = word;
        v = e >= 0 && e < a.N;  // -1 (and anything out of range) is an empty slot
        if (!v) e = 0;
      }
    }
    if (a.mode == kRawBlocks) {
      const int64_t pos = e * a.m + (v ? j % a.m : 0);
      r.row = (int64_t)b * a.raw_rows + (v ? pos - a.raw_pos0 : 0);
      r.raw = true;
    } else {
      r.row = (int64_t)b * a.kv_rows + e;
      r.raw = false;
    }
    r.valid = v;
  } else {
    const int w = j - kl.k_ent;
    r.valid = w < kl.w_len;
    const int64_t pos = kl.lo + (r.valid ? w : 0);
    r.row = (int64_t)b * a.raw_rows + (pos - a.raw_pos0);
    r.raw = true;
  }
  return r;
}

// 16 bytes of a 128-byte swizzled row: unit u of row r of a chunk.
__device__ __forceinline__ uint32_t swz(int r, int u) {
  return (uint32_t)(r * 128 + ((u ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return l | (h << 16);
}

// Mixed-precision cache: the raw bits of one 16-byte unit of a chunk (8 dims
// from dim c*64 + uc*8 of one key row) and what the conversion needs, loaded
// first so that a producer thread has all its loads of a chunk in flight at
// once.
struct RawUnit {
  uint4 v;
  float inv;  // RoPE units of an entry row: 1 / row scale
  int kind;   // 0: bf16 values as they are, 1: e4m3 codes in v.x / v.y, 2: bf16 RoPE / scale
};

__device__ __forceinline__ RawUnit mixed_load(const AttArgs& a, int64_t row, bool raw, int d0) {
  RawUnit r;
  r.inv = 1.f;
  if (raw) {
    r.kind = 0;
    r.v = __ldg(reinterpret_cast<const uint4*>(a.raw16 + row * a.D_qk + d0));
  } else if (d0 >= a.nope) {
    r.kind = 2;
    const int rw = a.D_qk - a.nope;
    r.v = __ldg(reinterpret_cast<const uint4*>(a.rope + row * rw + (d0 - a.nope)));
    r.inv = 1.f / __ldg(a.kscale + row);
  } else {
    r.kind = 1;
    const uint2 cv = __ldg(reinterpret_cast<const uint2*>(a.codes + row * a.nope + d0));
    r.v = make_uint4(cv.x, cv.y, 0u, 0u);
  }
  return r;
}

// e4m3 codes -> bf16 (exact: every e4m3 value is a bf16 value).
__device__ __forceinline__ uint4 codes_to_bf16(const uint4& v) {
  const uint32_t w2[2] = {v.x, v.y};
  uint32_t o[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const uint32_t word = w2[e / 2];
    const int sh = (e & 1) * 16;
    o[e] = pack_bf16(e4m3_to_f32((uint8_t)(word >> sh)), e4m3_to_f32((uint8_t)(word >> (sh + 8))));
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// A unit as the bf16 operand of the score pass: `lo` selects the low part of
// the RoPE-over-scale split (zero for every other kind).
__device__ __forceinline__ void mixed_convert(const RawUnit& r, uint4& hi, uint4& lo) {
  if (r.kind == 1) {
    hi = codes_to_bf16(r.v);
    lo = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  if (r.kind == 0) {
    hi = r.v;
    lo = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const uint32_t w[4] = {r.v.x, r.v.y, r.v.z, r.v.w};
  uint32_t h[4], l[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float f0 = bf16_to_f32((uint16_t)(w[e] & 0xffffu)) * r.inv;
    const float f1 = bf16_to_f32((uint16_t)(w[e] >> 16)) * r.inv;
    h[e] = pack_bf16(f0, f1);
    l[e] = pack_bf16(f0 - __bfloat162float(__float2bfloat16_rn(f0)),
                     f1 - __bfloat162float(__float2bfloat16_rn(f1)));
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// Arrive on `bar` (without raising its expected count) once every cp.async
// this thread has issued so far has landed.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(tc::smem_u32(bar))
               : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// `count` arrivals on `bar` at once (the producers that do not take part in a
// chunk loaded by TMA).
__device__ __forceinline__ void mbar_arrive_n(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(tc::smem_u32(bar)), "r"(count)
               : "memory");
}

template <bool kE4M3>
__global__ void __launch_bounds__(kThreads, 1)
    attend_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_kv,
                     const __grid_constant__ CUtensorMap tm_raw, const AttArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  uint8_t* sQ = smem;
  uint8_t* sRing = sQ + (size_t)a.nc * kChunk;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sRing + (size_t)kRing * kChunk);
  uint64_t* ring_full = bars;
  uint64_t* ring_empty = bars + kRing;
  uint64_t* q_full = bars + 2 * kRing;       // [kMaxQChunks]: one per Q chunk, once per Q load
  uint64_t* q_empty = q_full + kMaxQChunks;  // once per Q load: its last score MMA done
  uint64_t* s_full = q_empty + 1;            // [2]
  uint64_t* p_full = s_full + 2;             // [2]
  uint64_t* mask_full = p_full + 2;          // [2]
  uint64_t* mask_empty = mask_full + 2;      // [2]
  // PV(g) completes o_done[g & 1]: with two barriers no waiter can fall two
  // phases behind (a parity wait cannot tell phase j from phase j + 2)
  uint64_t* o_done = mask_empty + 2;  // [2]
  uint64_t* o_free = o_done + 2;      // once per item: its O has been read out
  uint64_t* mma_done = o_free + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  uint32_t* smask = tmem_slot + 4;                       // [2][4] ballot words of a tile's valid slots
  float* svscale = reinterpret_cast<float*>(smask + 8);  // mixed: [2][128] row scales of a tile

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* err = &g_attend_tc_error;
  // this CTA's work items: a contiguous range (consecutive items share Q)
  const int64_t it_begin = a.n_items * blockIdx.x / gridDim.x;
  const int64_t it_end = a.n_items * (blockIdx.x + 1) / gridDim.x;
  const int ncode = kE4M3 ? a.nope / 64 : a.nc;  // key chunks that meet one Q chunk each

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRing; ++s) {
      tc::mbar_init(&ring_full[s], kProd);  // every producer thread arrives
      tc::mbar_init(&ring_empty[s], 1);
    }
    for (int c = 0; c < kMaxQChunks; ++c) tc::mbar_init(&q_full[c], 1);
    tc::mbar_init(q_empty, 1);
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&s_full[s], 1);
      tc::mbar_init(&p_full[s], 4);
      tc::mbar_init(&mask_full[s], kProdWarps);
      tc::mbar_init(&mask_empty[s], 4);
      tc::mbar_init(&o_done[s], 1);
    }
    tc::mbar_init(o_free, 4);
    tc::mbar_init(mma_done, 1);
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tm_q);
    if (!kE4M3) {
      if (a.mode == kDense) tc::prefetch_tmap(&tm_kv);
      if (a.W > 0) tc::prefetch_tmap(&tm_raw);
    }
  }
  if (warp == kMmaWarp) tc::tmem_alloc(tmem_slot, 512);
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < kProdWarps) {
    // ------------------------------------------------------------ producers
    // Thread pt copies the 16-byte units pt + kProd*i of every gathered chunk
    // (unit u: row u/8, bytes 16*(u%8) of the row) with cp.async, each lane
    // with its own row address; each thread's copies of a chunk arrive on the
    // chunk's barrier by themselves when they land, so a producer never waits
    // for its own copies and runs ahead as far as the ring lets it.  A chunk
    // loaded by TMA is issued by warp 0 (lane 0 arrives for all 96 producers,
    // with the byte count); warps 1-2 only wait for its slot.
    const int pt = threadIdx.x;
    uint32_t pslot = 0, pph = 0;  // ring slot and the parity of its release
    bool ok = true;
    uint32_t tma_mask = 0, tma_par = 0;  // pt 0: slots whose last fill was TMA, and its parity
    uint32_t q_loads = 0;
    int64_t last_q = -1;
    int64_t g = 0;  // tiles so far (mask barrier phases)
    const uint8_t* kvb = reinterpret_cast<const uint8_t*>(a.kv16);
    const uint8_t* rawb = reinterpret_cast<const uint8_t*>(a.raw16);
    const int64_t rowb = (int64_t)a.D_qk * 2;
    // swizzled destination of each of this thread's units within a chunk;
    // only the last unit can fall outside the chunk (threads pt >= 64)
    uint32_t dso[kUnits];
#pragma unroll
    for (int i = 0; i < kUnits; ++i) {
      const int unit = pt + kProd * i;
      dso[i] = swz(unit >> 3, unit & 7);
    }
    const bool last_unit = pt + kProd * (kUnits - 1) < (int)(kChunk / 16);
    // rows of tile u's units (bf16 caches: the byte address of the unit in
    // chunk 0; mixed caches: the row and whether it is a raw row), the two
    // mask slots of each thread, and how the tile loads
    struct TileRows {
      // bf16 caches: the byte address of the unit in chunk 0; mixed caches:
      // the row (whether it is a raw row: bit i of wb; rows of the batch stay
      // below 2^31)
      typename std::conditional<kE4M3, int32_t, int64_t>::type rr[kUnits];
      uint32_t wb;
      SlotSrc s0, s1;
      int tma;    // bf16: 1 = 128 consecutive entry rows, 2 = 128 consecutive raw rows
      int tma_y;  //   (one box per chunk from tma_y); 0 = gathered
    };
    auto wait_slot = [&](uint32_t s, uint32_t par) -> bool {
      int okw = 1;
      if (lane == 0) okw = tc::mbar_wait(&ring_empty[s], par ^ 1, err, 11);
      return __shfl_sync(0xffffffffu, okw, 0) != 0;
    };
    auto advance = [&]() {
      if (++pslot == kRing) {
        pslot = 0;
        pph ^= 1;
      }
    };
    // key chunk c of a tile (bf16 caches: the Q chunk it meets is c; mixed:
    // a chunk of codes, or of a value half) into the next ring slot
    auto issue_chunk = [&](int c, const TileRows& t) -> bool {
      if (!kE4M3 && t.tma) {
        // every warp waits for the slot, also those that do not fill it: a
        // parity wait cannot tell a release from the one two fills later, so
        // no warp may run more than one fill of a slot ahead of the consumer
        if (!wait_slot(pslot, pph)) return false;
        if (warp == 0) {
          uint8_t* dst = sRing + pslot * kChunk;
          if (lane == 0) {
            tc::mbar_expect_tx(&ring_full[pslot], kChunk);
            mbar_arrive_n(&ring_full[pslot], kProd - 1);
            tma_mask |= 1u << pslot;
            tma_par = (tma_par & ~(1u << pslot)) | (pph << pslot);
          }
          if (lane == 0)
            tc::tma_load_2d(dst, t.tma == 1 ? &tm_kv : &tm_raw, &ring_full[pslot], c * 64, t.tma_y);
        }
        advance();
        return true;
      }
      if (!wait_slot(pslot, pph)) return false;
      if (pt == 0) tma_mask &= ~(1u << pslot);
      const uint32_t dst = tc::smem_u32(sRing + pslot * kChunk);
      if (kE4M3) {
        // the loads of half a chunk in flight at once, then their conversions
#pragma unroll
        for (int i0 = 0; i0 < kUnits; i0 += kHalfUnits) {
          RawUnit raw[kHalfUnits];
#pragma unroll
          for (int ii = 0; ii < kHalfUnits; ++ii) {
            const int i = i0 + ii, unit = pt + kProd * i;
            if (i < kUnits - 1 || (i == kUnits - 1 && last_unit))
              raw[ii] = mixed_load(a, t.rr[i], (t.wb >> i) & 1, c * 64 + (unit & 7) * 8);
          }
#pragma unroll
          for (int ii = 0; ii < kHalfUnits; ++ii) {
            const int i = i0 + ii;
            if (i < kUnits - 1 || (i == kUnits - 1 && last_unit)) {
              uint4 hi, lo;
              mixed_convert(raw[ii], hi, lo);
              *reinterpret_cast<uint4*>(sRing + pslot * kChunk + dso[i]) = hi;
            }
          }
        }
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&ring_full[pslot]);
      } else {
        const int coff = c * 128;
#pragma unroll
        for (int i = 0; i < kUnits; ++i)
          if (i < kUnits - 1 || last_unit)
            cp_async16(dst + dso[i], reinterpret_cast<const uint8_t*>(t.rr[i]) + coff);
        cp_async_arrive_noinc(&ring_full[pslot]);
      }
      advance();
      return true;
    };
    // Mixed caches: the high and the low part of RoPE chunk c (RoPE dims
    // over the row scale) into two consecutive slots from one load.
    auto issue_pair = [&](int c, const TileRows& t) -> bool {
      const uint32_t s0 = pslot, p0 = pph;
      const uint32_t s1 = pslot + 1 == kRing ? 0 : pslot + 1;
      const uint32_t p1 = s1 == 0 ? pph ^ 1 : pph;
      if (!wait_slot(s0, p0) || !wait_slot(s1, p1)) return false;
      if (pt == 0) tma_mask &= ~((1u << s0) | (1u << s1));
#pragma unroll
      for (int i0 = 0; i0 < kUnits; i0 += kHalfUnits) {
        RawUnit raw[kHalfUnits];
#pragma unroll
        for (int ii = 0; ii < kHalfUnits; ++ii) {
          const int i = i0 + ii, unit = pt + kProd * i;
          if (i < kUnits - 1 || (i == kUnits - 1 && last_unit))
            raw[ii] = mixed_load(a, t.rr[i], (t.wb >> i) & 1, c * 64 + (unit & 7) * 8);
        }
#pragma unroll
        for (int ii = 0; ii < kHalfUnits; ++ii) {
          const int i = i0 + ii;
          if (i < kUnits - 1 || (i == kUnits - 1 && last_unit)) {
            uint4 hi, lo;
            mixed_convert(raw[ii], hi, lo);
            *reinterpret_cast<uint4*>(sRing + s0 * kChunk + dso[i]) = hi;
            *reinterpret_cast<uint4*>(sRing + s1 * kChunk + dso[i]) = lo;
          }
        }
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&ring_full[s0]);
      tc::mbar_arrive(&ring_full[s1]);
      advance();
      advance();
      return true;
    };
    // A warp's units of a chunk cover 44 key rows (unit i of lane L is row
    // 4 warp + 12 i + L/8, shared by 8 lanes): lane L looks up rows q = L
    // and q = L + 32 of that list and the lanes exchange them by shuffles.
    // Key-list words are fetched a tile ahead: those two rows and the two
    // mask slots pt and pt + 96.
    struct TileWords {
      int32_t w[4];
    };
    const bool has1 = pt + kProd < kT;
    auto unit_row = [&](int q) -> int { return 4 * warp + 12 * (q >> 2) + (q & 3); };
    const int q1 = lane, q2 = lane + 32;
    const bool has_q2 = q2 < 4 * kUnits;
    auto tile_words = [&](const Item& it, int u, TileWords& t) {
      const KeyList& kl = it.kl;
      const int jt = (it.tile0 + u) * kT;
      const int r1 = unit_row(q1), r2 = unit_row(q2);
      t.w[0] = r1 < kT ? slot_word(a, kl, it.qrow, jt + r1) : 0;
      t.w[1] = (has_q2 && r2 < kT) ? slot_word(a, kl, it.qrow, jt + r2) : 0;
      t.w[2] = slot_word(a, kl, it.qrow, jt + pt);
      t.w[3] = slot_word(a, kl, it.qrow, jt + (has1 ? pt + kProd : pt));
    };
    auto tile_rows = [&](const Item& it, int u, const TileWords& tw, TileRows& t) {
      const KeyList& kl = it.kl;
      const int b = it.b;
      const int jt = (it.tile0 + u) * kT;
      // (row | raw << 63) of this lane's two rows of the warp's list
      auto packed = [&](int r, int32_t word) -> unsigned long long {
        const SlotSrc ss = slot_src(a, kl, b, jt + (r < kT ? r : 0), word);
        return (unsigned long long)ss.row | ((unsigned long long)(ss.raw ? 1 : 0) << 63);
      };
      const unsigned long long v1 = packed(unit_row(q1), tw.w[0]);
      const unsigned long long v2 = has_q2 ? packed(unit_row(q2), tw.w[1]) : 0ull;
      t.wb = 0;
#pragma unroll
      for (int i = 0; i < kUnits; ++i) {
        const int src = 4 * i + (lane >> 3);
        const unsigned long long a1 = __shfl_sync(0xffffffffu, v1, src & 31);
        const unsigned long long a2 = __shfl_sync(0xffffffffu, v2, src & 31);
        const unsigned long long v = src < 32 ? a1 : a2;
        const int64_t row = (int64_t)(v & ~(1ull << 63));
        const bool raw = (v >> 63) != 0;
        if (kE4M3) {
          t.rr[i] = (int32_t)row;
          t.wb |= (raw ? 1u : 0u) << i;
        } else {
          t.rr[i] = reinterpret_cast<int64_t>((raw ? rawb : kvb) + row * rowb + (lane & 7) * 16);
        }
      }
      t.tma = 0;
      t.tma_y = 0;
      if (!kE4M3) {
        if (a.mode == kDense && jt + kT <= kl.kd) {
          // every slot a valid entry, entry j in row j (a tile with masked
          // slots is gathered: rows past the valid entries may hold anything,
          // and a masked slot's row still meets a zero weight in P . V)
          t.tma = 1;
          t.tma_y = (int)((int64_t)b * a.kv_rows + jt);
        } else if (a.W > 0 && jt >= kl.k_ent) {
          // every slot a window slot: raw rows lo + (j - k_ent) (past the
          // window: masked; past the rows: zero-filled)
          t.tma = 2;
          t.tma_y = (int)((int64_t)b * a.raw_rows + (kl.lo - a.raw_pos0) + (jt - kl.k_ent));
        }
      }
      t.s0 = slot_src(a, kl, b, jt + pt, tw.w[2]);
      t.s1 = slot_src(a, kl, b, jt + (has1 ? pt + kProd : pt), tw.w[3]);
    };
    // the value chunks of a tile (after the key chunks of the next one)
    auto issue_values = [&](const TileRows& t, int half) -> bool {
      for (int c = 0; c < a.nvc; ++c)
        if (!issue_chunk(half * a.nvc + c, t)) return false;
      return true;
    };
    TileRows cur, prev;
    TileWords wnext;
    int prev_half = 0;
    bool have_prev = false;
    for (int64_t id = it_begin; id < it_end && ok; ++id) {
      const Item it = make_item(a, id);
      if (it.n == 0) continue;
      if (it.qrow != last_q) {
        // Q of a new query: once the previous query's last score MMA is done
        if (warp == 0) {
          int okw = 1;
          if (lane == 0) {
            if (q_loads > 0) okw = tc::mbar_wait(q_empty, (q_loads - 1) & 1, err, 13);
            if (okw) {
              // a barrier per chunk: the first tile's QK^T starts as its chunks land
              for (int c = 0; c < a.nc; ++c) {
                tc::mbar_expect_tx(&q_full[c], kChunk);
                tc::tma_load_2d(sQ + c * kChunk, &tm_q, &q_full[c], c * 64, (int)(it.qrow * a.H));
              }
            }
          }
          ok = __shfl_sync(0xffffffffu, okw, 0) != 0;
          if (!ok) break;
        }
        ++q_loads;
        last_q = it.qrow;
      }
      tile_words(it, 0, wnext);
      tile_rows(it, 0, wnext, cur);
      for (int u = 0; u < it.n && ok; ++u) {
        if (u + 1 < it.n) tile_words(it, u + 1, wnext);  // in flight during this tile's issues
        // validity of slots pt and pt + 96 (and, for mixed caches, the scale
        // of their rows) for the softmax: ballot word w covers slots 32w .. 32w+31
        const uint32_t sb = (uint32_t)(g & 1);
        int okw = 1;
        if (lane == 0) okw = tc::mbar_wait(&mask_empty[sb], (uint32_t)((g >> 1) & 1) ^ 1, err, 12);
        if (!__shfl_sync(0xffffffffu, okw, 0)) {
          ok = false;
          break;
        }
        const uint32_t bal0 = __ballot_sync(0xffffffffu, cur.s0.valid);
        const uint32_t bal1 = __ballot_sync(0xffffffffu, has1 && cur.s1.valid);
        if (lane == 0) {
          smask[sb * 4 + warp] = bal0;
          if (warp == 0) smask[sb * 4 + 3] = bal1;
        }
        if (kE4M3) {
          svscale[sb * 128 + pt] =
              (cur.s0.valid && !cur.s0.raw) ? __ldg(a.kscale + cur.s0.row) : 1.f;
          if (has1)
            svscale[sb * 128 + pt + kProd] =
                (cur.s1.valid && !cur.s1.raw) ? __ldg(a.kscale + cur.s1.row) : 1.f;
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&mask_full[sb]);
        // QK^T chunks: mixed caches the code chunks, then (high, low) pairs of
        // the RoPE chunks; bf16 caches the nc chunks in order
        for (int c = 0; c < ncode && ok; ++c) ok = issue_chunk(c, cur);
        if (kE4M3)
          for (int c = ncode; c < a.nc && ok; ++c) ok = issue_pair(c, cur);
        if (ok && have_prev) ok = issue_values(prev, prev_half);
        prev = cur;
        prev_half = it.half;
        have_prev = true;
        ++g;
        if (u + 1 < it.n) tile_rows(it, u + 1, wnext, cur);
      }
    }
    if (ok && have_prev) ok = issue_values(prev, prev_half);
    // every copy must land before the CTA can exit: this thread's cp.async,
    // and (pt 0) the last Q load and the TMA loads of the ring not yet known
    // to have landed (only after an error: otherwise the MMA issuer waited for
    // all of them)
    cp_async_wait<0>();
    if (pt == 0) {
      if (q_loads > 0)
        for (int c = 0; c < a.nc; ++c) tc::mbar_drain(&q_full[c], (q_loads - 1) & 1);
      for (int s = 0; s < kRing; ++s)
        if ((tma_mask >> s) & 1u) tc::mbar_drain(&ring_full[s], (tma_par >> s) & 1u);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_s = tc::idesc(128, kT, 1, 1);
      const uint32_t id_pv = tc::idesc(128, 64, 1, 1, 0, 1);
      bool ok = true;
      // test aid: the producers' first loads are in flight while this waits
      if (a.stall && blockIdx.x == 0) ok = tc::flag_wait(&g_attend_never_set, tc::kStallNs, err, 28);
      // descriptors of Q chunk 0 and ring slot 0 (K-major for S, MN-major
      // for PV); other chunks / slots / K steps are constant offsets in the
      // start-address field, so each MMA costs the issuing thread a couple of
      // integer adds
      const uint64_t qd0 = tc::sdesc_sw128(tc::smem_u32(sQ));
      const uint64_t rd0 = tc::sdesc_sw128(tc::smem_u32(sRing));
      const uint64_t vd0 = tc::sdesc_sw128_mn(tc::smem_u32(sRing));
      constexpr uint32_t kChunk16 = kChunk >> 4;
      uint32_t slot = 0, ph = 0;  // ring slot and the parity of its fill
      auto next_slot = [&]() {
        if (++slot == kRing) {
          slot = 0;
          ph ^= 1;
        }
      };
      uint32_t q_loads = 0, q_seen = 0;  // Q loads so far; chunks of the current one seen landed
      int64_t last_q = -1;
      uint32_t used = 0;  // items with keys so far (o_free phases)
      // PV(gp) of the previous tile is issued after S of the next one, so the
      // softmax of a tile overlaps the next tile's QK^T
      auto issue_pv = [&](int64_t gp, bool first, uint32_t item_no) -> bool {
        const uint32_t sb = (uint32_t)(gp & 1);
        // the item's first PV overwrites O: the previous item's O must be read out
        if (first && item_no > 0 && !tc::mbar_wait(o_free, (item_no - 1) & 1, err, 25)) return false;
        if (!tc::mbar_wait(&p_full[sb], (uint32_t)((gp >> 1) & 1), err, 22)) return false;
        tc::tc_fence_after();
        const uint32_t p_tmem = tmem + sb * 128;
        for (int c = 0; c < a.nvc; ++c) {
          if (!tc::mbar_wait(&ring_full[slot], ph, err, 23)) return false;
          tc::fence_proxy_async_smem();  // gathered rows -> tensor cores
          tc::tc_fence_after();
          const uint64_t vd = vd0 + slot * kChunk16;
          const uint32_t o_tmem = tmem + 256 + 64 * c;
#pragma unroll
          for (int ks = 0; ks < kT / 16; ++ks) {
            // 16 keys per K step: 16 rows of 128 bytes; their P (bf16 pairs)
            // in 8 columns at 32 (ks/2) + 8 (ks%2), the low part 16 further
            const uint64_t bd = vd + (uint64_t)(ks * (2048 >> 4));
            const uint32_t pa = p_tmem + 32 * (ks >> 1) + 8 * (ks & 1);
            tc::mma_bf16_ts(o_tmem, pa, bd, id_pv, (!first || ks > 0) ? 1u : 0u);
            if (kE4M3) tc::mma_bf16_ts(o_tmem, pa + 16, bd, id_pv, 1u);
          }
          tc::mma_commit(&ring_empty[slot]);
          next_slot();
        }
        tc::mma_commit(&o_done[sb]);
        return true;
      };
      int64_t g = 0, pv_g = -1;
      bool pv_first = false;
      uint32_t pv_item = 0;
      for (int64_t id = it_begin; id < it_end && ok; ++id) {
        const Item it = make_item(a, id);
        if (it.n == 0) continue;
        if (it.qrow != last_q) {
          // the previous Q's last score MMA has been issued: release it once done
          if (q_loads > 0) tc::mma_commit(q_empty);
          ++q_loads;
          last_q = it.qrow;
          q_seen = 0;
        }
        for (int u = 0; u < it.n && ok; ++u) {
          const uint32_t sb = (uint32_t)(g & 1);
          const uint32_t s_tmem = tmem + sb * 128;
          for (int cc = 0; cc < a.nsc && ok; ++cc) {
            // the Q chunk this key chunk meets (mixed caches: the code chunks,
            // then a (high, low) pair per RoPE chunk)
            const int c = cc < ncode ? cc : ncode + ((cc - ncode) >> 1);
            if (!((q_seen >> c) & 1u)) {
              if (!tc::mbar_wait(&q_full[c], (q_loads - 1) & 1, err, 21)) {
                ok = false;
                break;
              }
              q_seen |= 1u << c;
            }
            if (!tc::mbar_wait(&ring_full[slot], ph, err, 24)) {
              ok = false;
              break;
            }
            tc::fence_proxy_async_smem();  // gathered rows -> tensor cores
            tc::tc_fence_after();
            const uint64_t qd = qd0 + (uint32_t)c * kChunk16;
            const uint64_t rd = rd0 + slot * kChunk16;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)  // 16 bf16 (32 bytes) per K step
              tc::mma_bf16(s_tmem, qd + (uint64_t)(ks * 2), rd + (uint64_t)(ks * 2), id_s,
                           (cc > 0 || ks > 0) ? 1u : 0u);
            tc::mma_commit(&ring_empty[slot]);
            next_slot();
          }
          if (!ok) break;
          tc::mma_commit(&s_full[sb]);
          if (pv_g >= 0) ok = issue_pv(pv_g, pv_first, pv_item);
          pv_g = g;
          pv_first = u == 0;
          pv_item = used;
          ++g;
        }
        ++used;
      }
      if (ok && pv_g >= 0) issue_pv(pv_g, pv_first, pv_item);
      // every MMA issued must have completed before TMEM is released
      tc::mma_commit(mma_done);
      tc::mbar_drain(mma_done, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax (warps 4-7)
    const int quarter = warp & 3;
    const int h = quarter * 32 + lane;  // head row == TMEM lane
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const int hv = a.D_v / 2;
    bool ok = true;
    int64_t g = 0;
    auto wait1 = [&](uint64_t* bar, uint32_t par, int code) -> bool {
      int okw = lane == 0 ? (int)tc::mbar_wait(bar, par, err, code) : 0;
      okw = __shfl_sync(0xffffffffu, okw, 0);
      __syncwarp();
      return okw != 0;
    };
    for (int64_t id = it_begin; id < it_end && ok; ++id) {
      const Item it = make_item(a, id);
      const int64_t orow = it.qrow * a.H + h;
      float m_ref = -INFINITY, l_run = 0.f;
      for (int u = 0; u < it.n && ok; ++u) {
        const uint32_t sb = (uint32_t)(g & 1), par = (uint32_t)((g >> 1) & 1);
        // every lane acquires the producers' ballot words itself
        const bool mk = tc::mbar_wait(&mask_full[sb], par, err, 31);
        if (!__all_sync(0xffffffffu, mk)) {
          ok = false;
          break;
        }
        uint32_t bal[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) bal[q] = *reinterpret_cast<volatile uint32_t*>(&smask[sb * 4 + q]);
        __syncwarp();
        if (!kE4M3 && lane == 0) tc::mbar_arrive(&mask_empty[sb]);
        if (!wait1(&s_full[sb], par, 32)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        // Two passes over the tile's scores, 32 columns at a time (few live
        // registers): the row maximum, then P.  P of keys 32q .. 32q+31 goes,
        // as bf16 pairs, over the 32 score columns just read: the high part
        // to columns 32q .. 32q+15, the low part (mixed caches) to 32q+16 ..
        // 32q+31.
        const uint32_t s_col = tmem + lane_base + sb * 128;
        float m_tile = -INFINITY;
#pragma unroll 1
        for (int gq = 0; gq < kT / 32; ++gq) {
          uint32_t r[32];
          tc::tmem_ld32(s_col + gq * 32, r);
          tc::tmem_wait_ld();
          const uint32_t bw = bal[gq];
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int j = gq * 32 + jj;
            const float cs = kE4M3 ? svscale[sb * 128 + j] * a.c_log2 : a.c_log2;
            const float xv = ((bw >> jj) & 1u) ? __uint_as_float(r[jj]) * cs : -INFINITY;
            m_tile = fmaxf(m_tile, xv);
          }
        }
        const bool grow = m_tile > m_ref + kRescaleLog2;
        const bool rescale = grow && m_ref != -INFINITY;
        const float alpha = grow ? exp2f(m_ref - m_tile) : 1.f;
        if (__any_sync(0xffffffffu, rescale)) {
          // O holds the tiles before u of this item: wait for PV(g-1), then scale the rows
          if (!wait1(&o_done[(g - 1) & 1], (uint32_t)(((g - 1) >> 1) & 1), 33)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const float f = rescale ? alpha : 1.f;
          for (int gq = 0; gq < 256 / 32; ++gq) {
            uint32_t r[32];
            tc::tmem_ld32(tmem + lane_base + 256 + gq * 32, r);
            tc::tmem_wait_ld();
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) r[jj] = __float_as_uint(__uint_as_float(r[jj]) * f);
            tc::tmem_st32(tmem + lane_base + 256 + gq * 32, r);
          }
          tc::tmem_wait_st();
        }
        if (grow) {
          l_run *= alpha;
          m_ref = m_tile;
        }
        // P = 2^(x - m_ref) (mixed caches: times the value row's scale,
        // split exactly into bf16 high + low parts: outlier rows carry values
        // up to ~20x unit scale, too large for one rounding of P)
#pragma unroll 1
        for (int gq = 0; gq < kT / 32; ++gq) {
          uint32_t r[32];
          tc::tmem_ld32(s_col + gq * 32, r);
          tc::tmem_wait_ld();
          const uint32_t bw = bal[gq];
          uint32_t pk[16], pl[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            float pp[2], lo[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int jj = 2 * c + e, j = gq * 32 + jj;
              const float sv = kE4M3 ? svscale[sb * 128 + j] : 1.f;
              const float xv = ((bw >> jj) & 1u) ? __uint_as_float(r[jj]) * (sv * a.c_log2)
                                                 : -INFINITY;
              const float pj = m_ref == -INFINITY ? 0.f : exp2f(xv - m_ref);
              l_run += pj;
              pp[e] = kE4M3 ? pj * sv : pj;
              lo[e] = kE4M3 ? pp[e] - __bfloat162float(__float2bfloat16_rn(pp[e])) : 0.f;
            }
            pk[c] = pack_bf16(pp[0], pp[1]);
            pl[c] = pack_bf16(lo[0], lo[1]);
          }
          tc::tmem_st16(s_col + gq * 32, pk);
          if (kE4M3) tc::tmem_st16(s_col + gq * 32 + 16, pl);
        }
        tc::tmem_wait_st();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (kE4M3) tc::mbar_arrive(&mask_empty[sb]);
          tc::mbar_arrive(&p_full[sb]);
        }
        ++g;
      }
      if (!ok) break;
      // ---------------------------------------------------------- output of the item
      const bool have_o = it.n > 0;
      if (have_o) {
        // PV of the item's last tile completes o_done[(g-1) & 1]; that barrier
        // cannot be further ahead (the next item's first PV waits for o_free)
        if (!wait1(&o_done[(g - 1) & 1], (uint32_t)(((g - 1) >> 1) & 1), 35)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
      }
      if (a.splits == 1) {
        const float inv = (have_o && l_run > 0.f) ? 1.f / l_run : 0.f;
        for (int gq = 0; gq < hv / 32; ++gq) {
          uint32_t r[32];
          if (have_o) {
            tc::tmem_ld32(tmem + lane_base + 256 + gq * 32, r);
            tc::tmem_wait_ld();
          }
          const int64_t o0 = orow * a.D_v + it.half * hv + gq * 32;
          if (a.out_f32) {
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + o0);
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              float4 o;
              o.x = have_o ? __uint_as_float(r[4 * v + 0]) * inv : 0.f;
              o.y = have_o ? __uint_as_float(r[4 * v + 1]) * inv : 0.f;
              o.z = have_o ? __uint_as_float(r[4 * v + 2]) * inv : 0.f;
              o.w = have_o ? __uint_as_float(r[4 * v + 3]) * inv : 0.f;
              dst[v] = o;
            }
          } else {
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.out) + o0);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float f0 = have_o ? __uint_as_float(r[8 * v + 2 * e]) * inv : 0.f;
                const float f1 = have_o ? __uint_as_float(r[8 * v + 2 * e + 1]) * inv : 0.f;
                w[e] = pack_bf16(f0, f1);
              }
              dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      } else {
        const int64_t prow = orow * a.splits + it.split;
        float4* dst = reinterpret_cast<float4*>(a.part + prow * a.D_v + it.half * hv);
        for (int gq = 0; gq < hv / 32; ++gq) {
          uint32_t r[32];
          if (have_o) {
            tc::tmem_ld32(tmem + lane_base + 256 + gq * 32, r);
            tc::tmem_wait_ld();
          }
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            float4 o;
            o.x = have_o ? __uint_as_float(r[4 * v + 0]) : 0.f;
            o.y = have_o ? __uint_as_float(r[4 * v + 1]) : 0.f;
            o.z = have_o ? __uint_as_float(r[4 * v + 2]) : 0.f;
            o.w = have_o ? __uint_as_float(r[4 * v + 3]) : 0.f;
            dst[gq * 8 + v] = o;
          }
        }
        if (it.half == 0) {
          a.ml[prow * 2 + 0] = have_o ? m_ref : -INFINITY;
          a.ml[prow * 2 + 1] = have_o ? l_run : 0.f;
        }
      }
      if (have_o) {
        // O has been read: the next item's first PV may overwrite it
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(o_free);
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

// Merge the splits of one (query, head) in split order (log2 domain).
__global__ void __launch_bounds__(128) attend_tc_combine_kernel(const float* __restrict__ part,
                                                                const float* __restrict__ ml,
                                                                int splits, int D_v,
                                                                void* __restrict__ out,
                                                                int out_f32) {
  const int64_t qh = blockIdx.x;
  const float* mlr = ml + qh * splits * 2;
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, mlr[2 * s]);
  float L = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float ms = mlr[2 * s];
    if (ms != -INFINITY) L += mlr[2 * s + 1] * exp2f(ms - M);
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  for (int d4 = threadIdx.x; d4 < D_v / 4; d4 += blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < splits; ++s) {
      const float ms = mlr[2 * s];
      if (ms == -INFINITY) continue;
      const float f = exp2f(ms - M);
      const float4 p = reinterpret_cast<const float4*>(part + (qh * splits + s) * D_v)[d4];
      acc.x = fmaf(p.x, f, acc.x);
      acc.y = fmaf(p.y, f, acc.y);
      acc.z = fmaf(p.z, f, acc.z);
      acc.w = fmaf(p.w, f, acc.w);
    }
    if (out_f32) {
      reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + qh * D_v)[d4] =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    } else {
      uint2 w;
      w.x = pack_bf16(acc.x * inv, acc.y * inv);
      w.y = pack_bf16(acc.z * inv, acc.w * inv);
      reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(out) + qh * D_v)[d4] = w;
    }
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D map over a row-major [rows, cols] bf16 matrix: box of 64 columns
// (128 bytes) x box_rows, 128-byte swizzle.
bool make_map_bf16(CUtensorMap* map, const void* base, int64_t rows, int cols, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Slots of the first part of the longest key list of the launch.
int64_t first_part(const csa_params& p, int Q, int64_t N, int mode, int64_t q_pos0) {
  if (mode == kDense) {
    int64_t kd = n_vis(q_pos0 + Q - 1, p.m);
    return kd > N ? N : kd;
  }
  return mode == kRawBlocks ? (int64_t)p.k * p.m : (int64_t)p.k;
}

// Longest key list of the launch, in tiles.
int max_tiles(const csa_params& p, int Q, int64_t N, int mode, int64_t q_pos0) {
  const int64_t len = ((first_part(p, Q, N, mode, q_pos0) + 3) & ~3ll) + p.window;
  return (int)ceil_div(len, kT);
}

int num_sms() {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 148;
}

}  // namespace

// Split plan of the tensor-core path: one split per (query, half) for
// multi-query launches; decode (one query per sequence) cuts the key list
// into runs of kDecodeTiles tiles (more when that would exceed 16 runs), so
// that the few queries of a decode step spread over the GPU.  Depends on Q
// and the key-list length only, never on the batch.
constexpr int kDecodeTiles = 5;

void attend_tc_plan(const csa_params& p, int Q, int64_t N, int mode, int64_t q_pos0, int* splits,
                    int* tps) {
  const int nt = max_tiles(p, Q, N, mode, q_pos0);
  if (Q > 1 || nt <= kDecodeTiles) {
    *splits = 1;
    *tps = nt > 0 ? nt : 1;
    return;
  }
  int t = (int)ceil_div(nt, 16);
  if (t < kDecodeTiles) t = kDecodeTiles;
  *tps = t;
  *splits = (int)ceil_div(nt, t);
}

// Scratch for the split partials.  A shorter key list can take more splits
// (17 tiles: 9 splits of 2; 16 tiles: 16 splits of 1), so the bound is
// min(16, tiles of the longest list).
size_t attend_tc_workspace(const csa_params& p, int Q, int64_t N, int mode, int64_t q_pos0) {
  int splits, tps;
  attend_tc_plan(p, Q, N, mode, q_pos0, &splits, &tps);
  if (splits <= 1) return 0;
  const int nt = max_tiles(p, Q, N, mode, q_pos0);
  splits = nt < 16 ? nt : 16;
  const size_t rows = (size_t)p.B * Q * p.H * splits;
  const size_t part = (rows * p.D_v * sizeof(float) + 255) & ~(size_t)255;
  return part + rows * 2 * sizeof(float);
}

bool attend_tc_supported(const csa_params& p, csa_dtype q_dtype, const csa_rows& kv,
                         const csa_rows& raw, int Q, int64_t N, csa_dtype out_dtype, int mode) {
  if (q_dtype != CSA_BF16) return false;
  if (out_dtype != CSA_BF16 && out_dtype != CSA_F32) return false;
  if (p.H != 128) return false;
  if (p.D_qk % 64 != 0 || p.D_qk / 64 > kMaxQChunks) return false;
  if (p.D_v % 128 != 0 || p.D_v > 512 || p.D_v > p.D_qk) return false;
  if (N < 1) return false;
  if (mode == kRawBlocks) {
    if (raw.dtype != CSA_BF16) return false;
  } else if (kv.dtype == CSA_E4M3) {
    if (kv.nope != p.D_v || kv.nope % 64 != 0) return false;
  } else if (kv.dtype != CSA_BF16) {
    return false;
  }
  if ((p.window > 0 || mode == kRawBlocks) && raw.dtype != CSA_BF16) return false;
  if ((int64_t)p.B * kv.n_rows >= (1ll << 31)) return false;
  if ((p.window > 0 || mode == kRawBlocks) && (int64_t)p.B * raw.n_rows >= (1ll << 31)) return false;
  if ((int64_t)p.B * Q * p.H >= (1ll << 31)) return false;
  return encode_fn() != nullptr;
}

cudaError_t attend_tc_status(int* code, cudaStream_t st) {
  int h = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&h, g_attend_tc_error, sizeof(int), 0,
                                            cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return e;
  *code = h;
  if (h != 0) {
    int zero = 0;
    e = cudaMemcpyToSymbol(g_attend_tc_error, &zero, sizeof(int));
  }
  return e;
}

cudaError_t launch_attend_tc(const csa_params& p, const void* q, const csa_rows& kv,
                             const csa_rows& raw, int64_t raw_pos0, const int32_t* idx, int mode,
                             int64_t q_pos0, int Q, int64_t N, void* out, csa_dtype out_dtype,
                             void* ws, cudaStream_t st) {
  AttArgs a{};
  const bool e4m3 = kv.dtype == CSA_E4M3 && mode != kRawBlocks;
  const bool uses_raw = p.window > 0 || mode == kRawBlocks;
  a.B = p.B;
  a.Q = Q;
  a.H = p.H;
  a.D_qk = p.D_qk;
  a.D_v = p.D_v;
  a.k = p.k;
  a.W = p.window;
  a.m = p.m;
  a.nc = p.D_qk / 64;
  a.nope = e4m3 ? kv.nope : p.D_qk;
  a.nsc = e4m3 ? a.nope / 64 + 2 * (a.nc - a.nope / 64) : a.nc;
  a.nvc = p.D_v / 128;
  a.mode = mode;
  a.e4m3 = e4m3 ? 1 : 0;
  a.N = N;
  a.kv_rows = kv.n_rows;
  a.raw_rows = uses_raw ? raw.n_rows : 0;
  a.raw_pos0 = raw_pos0;
  a.q_pos0 = q_pos0;
  a.c_log2 = p.scale * 1.4426950408889634f;
  a.idx = idx;
  a.kv16 = reinterpret_cast<const uint16_t*>(kv.data);
  a.codes = reinterpret_cast<const uint8_t*>(kv.data);
  a.rope = reinterpret_cast<const uint16_t*>(kv.rope);
  a.kscale = kv.scale;
  a.raw16 = reinterpret_cast<const uint16_t*>(raw.data);
  a.out = out;
  a.out_f32 = out_dtype == CSA_F32 ? 1 : 0;
  a.stall = take_debug_stall(kStallAttend) ? 1 : 0;
  attend_tc_plan(p, Q, N, mode, q_pos0, &a.splits, &a.tps);
  a.n_items = (int64_t)p.B * Q * 2 * a.splits;
  // partials at the front of the workspace, (max, sum) pairs after them
  const size_t rows = (size_t)p.B * Q * p.H * a.splits;
  a.part = reinterpret_cast<float*>(ws);
  a.ml = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) +
                                  ((rows * p.D_v * sizeof(float) + 255) & ~(size_t)255));

  CUtensorMap tm_q, tm_kv, tm_raw;
  memset(&tm_kv, 0, sizeof(tm_kv));
  memset(&tm_raw, 0, sizeof(tm_raw));
  if (!make_map_bf16(&tm_q, q, (int64_t)p.B * Q * p.H, p.D_qk, 128)) return cudaErrorInvalidValue;
  if (!e4m3) {
    // dense runs of entry rows and window rows load as 128-row boxes
    if (mode == kDense &&
        !make_map_bf16(&tm_kv, kv.data, (int64_t)p.B * kv.n_rows, p.D_qk, 128))
      return cudaErrorInvalidValue;
    if (p.window > 0 &&
        !make_map_bf16(&tm_raw, raw.data, (int64_t)p.B * raw.n_rows, p.D_qk, 128))
      return cudaErrorInvalidValue;
  }
  int64_t grid = num_sms();
  if (a.n_items < grid) grid = a.n_items;
  if (grid < 1) return cudaSuccess;
  const size_t smem = 1024 + (size_t)a.nc * kChunk + (size_t)kRing * kChunk +
                      (2 * kRing + kMaxQChunks + 14) * sizeof(uint64_t) + 16 + 32 +
                      2 * 128 * sizeof(float);
  cudaError_t e;
  if (e4m3) {
    e = cudaFuncSetAttribute(attend_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    attend_tc_kernel<true><<<(unsigned)grid, kThreads, smem, st>>>(tm_q, tm_kv, tm_raw, a);
  } else {
    e = cudaFuncSetAttribute(attend_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    attend_tc_kernel<false><<<(unsigned)grid, kThreads, smem, st>>>(tm_q, tm_kv, tm_raw, a);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess || a.splits == 1) return e;
  attend_tc_combine_kernel<<<(unsigned)((int64_t)p.B * Q * p.H), 128, 0, st>>>(
      a.part, a.ml, a.splits, p.D_v, out, a.out_f32);
  return cudaGetLastError();
}

}  // namespace csa
