// Tensor-core path of steps 4 / 5 (CSA sparse MQA, HCA dense MQA): tcgen05
// MMAs with TMEM accumulators, key rows gathered (cp.async, or one TMA box per
// chunk for runs of consecutive rows) into a ring of 128-byte-swizzled
// shared-memory chunks.
//
//   o[b,i,h,:] = sum_j softmax_j(scale * q[b,i,h,:] . K_j) * K_j[0:D_v]
//
// Sources: "一文搞懂 DeepSeek：从 V3 的 KV 压缩与 MoE，到 V4 的百万 token 上下文",
// section "V4 改进一：CSA 与 HCA" (selected entries plus a sliding window of
// raw KV, one KV shared by all heads: MQA; HCA attends densely) and section
// "V3 看家本领一：MLA" (the value is the latent, the decoupled RoPE key only
// enters the score); "DeepSeek-V4 详解" section 2.2 Step 4 (bf16, 128 heads)
// and section 2.3 Step 2.
//
// Mapping.  The 128 heads of one query are the MMA's M side, so one shared
// key row feeds every head.  A 128 x 512 fp32 output accumulator alone fills
// all 512 TMEM columns, so each CTA owns one half of the value dims (256
// columns) and computes the 128 x 128 score tile S = Q K^T itself (both halves
// of a query compute the same S; the extra QK^T work buys an accumulator that
// fits).  TMEM: two S buffers (columns 0-255) and O (columns 256-511).  After
// the softmax reads S it writes P (bf16 pairs) over the first 64 columns of
// the same buffer, and P . V runs with A taken from TMEM.
//
// Shared memory: Q of the query (D_qk/64 chunks of 128 x 64 bf16, loaded once
// by TMA, a barrier per chunk, and resident) and a ring of kRing chunks of 128
// keys x 64 dims.  For
// every tile of 128 keys three producer warps gather the D_qk/64 chunks of the
// keys and then, one tile later, the D_v/128 chunks of the value half, with
// 16-byte cp.async copies.  The tile's 128 rows go through a table in shared
// memory: each producer thread resolves two slots of the key list and writes
// their rows, then reads the rows of its own units; each lane computes its
// own gathered addresses and swizzled destinations (TMA gathers take their
// operands from warp-uniform registers, so 32 lanes with 32 different rows
// serialise).  Each thread's
// copies of a chunk arrive on the chunk's barrier by themselves once they
// have landed (cp.async.mbarrier.arrive), so the producers run ahead as far
// as the ring allows; the MMA issuer, after its wait, issues the proxy fence
// that makes the rows visible to the tensor cores.  A tile whose 128 slots
// are all valid consecutive entries (HCA) or all window slots is one TMA box
// per chunk instead.  Mixed-precision caches (e4m3 codes with a row scale
// c_j, RoPE dims in bf16) run in f16: the codes are exact in f16, so a code
// chunk is the codes themselves (one conversion instruction per two codes),
// and the row scale moves out of the keys: the tile holds S'_j = q_nope .
// code_j + q_rope . (rope_j / c_j), the RoPE dims over the row scale split
// exactly into an f16 high and low part (two ring slots that meet the same Q
// chunk), and the softmax takes S_j = c_j S'_j.  These chunks pass through
// the producers' registers: a thread issues the 8-byte code loads of two
// chunks before it waits for their ring slots, and every value and scale
// load of the RoPE chunk before its two slots.  P . V runs on the codes with
// c_j folded into P, rounded once to f16.  Q is converted to f16 in shared
// memory once per CTA.  The MMA order is S(0), S(1), PV(0), S(2), PV(1), ...
// so the softmax of tile u overlaps S(u+1).  A key row doubles as its value
// row: the same 128-byte swizzled chunk is K-major for QK^T and MN-major for
// PV.
//
// Softmax: one thread per head row, log2 domain, running maximum updated only
// when a tile's maximum exceeds it by more than 2^8 (then O and the running
// sum are rescaled); P = 2^(x - m) <= 2^8 fits bf16 and fp32 comfortably.
//
// Raw-token variant ("DeepSeek-V4 详解" section 2.2 Steps 3-4): the key list
// is the m raw tokens of every selected block, block by block in list order,
// then the window; slot j < k*m reads raw row idx[j/m]*m + j%m of the raw
// rows (which then hold every position from 0), gathered like the entries.
//
// Decode (one query per sequence) splits the key list into fixed runs of
// tiles (chosen from the key-list length only, never from the batch) and
// merges the splits in order in attend_tc_combine_kernel.
//
// Roles: warps 0-2 producers, warp 3 TMEM allocator + MMA issuer (one
// thread; descriptors advanced by constant offsets), warps 4-7 softmax /
// rescale / epilogue.  Every mbarrier wait is bounded; a timeout is recorded
// in a device error word and the kernel returns.
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstring>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace csa {

namespace {

__device__ int g_attend_tc_error = 0;
__device__ int g_attend_never_set = 0;  // test aid: a flag that nothing sets

constexpr int kT = 128;              // keys per tile
constexpr int kRing = 5;             // key chunk slots
constexpr uint32_t kChunk = 16384;   // 128 rows x 128 bytes
constexpr int kMaxQChunks = 9;       // D_qk <= 576
constexpr float kRescaleLog2 = 8.f;  // rescale when the maximum grows by more than 2^8
constexpr int kProdWarps = 3;        // warps 0-2: key-chunk producers (cp.async)
constexpr int kProd = kProdWarps * 32;
constexpr int kUnits = (kChunk / 16 + kProd - 1) / kProd;  // 16-byte units per producer thread
constexpr int kMmaWarp = 3;          // warp 3: TMEM allocator + MMA issuer
constexpr int kThreads = 256;        // + warps 4-7: softmax / epilogue

struct AttArgs {
  int B, Q, H, D_qk, D_v, k, W, m;
  int nc;   // D_qk / 64
  int nsc;  // key chunk slots per tile for QK^T (nc; e4m3: the RoPE chunks take two each)
  int nvc;  // D_v / 128: value chunks per half
  int dense;    // every visible entry (HCA)
  int rawblk;   // the raw tokens of the selected blocks (raw-token variant)
  int e4m3;
  int stall;    // test aid: CTA 0's MMA issuer first waits on a flag that nothing sets
  int splits, tps;  // splits per (query, half); tiles per split
  int64_t N, kv_rows, raw_rows, raw_pos0, q_pos0;
  float c_log2;  // scale * log2(e)
  const int32_t* idx;
  const uint16_t* kv16;  // bf16 entries: [B, kv_rows, D_qk]
  const uint8_t* codes;  // e4m3 entries: [B, kv_rows, nope]
  const uint16_t* rope;  // [B, kv_rows, D_qk - nope]
  const float* kscale;   // [B, kv_rows]
  int nope;
  const uint16_t* raw16;  // raw rows (e4m3 path reads the window itself)
  void* out;
  int out_f32;
  float* part;  // splits > 1: [rows*H][splits][D_v] unnormalised O
  float* ml;    // splits > 1: [rows*H][splits][2] (max, sum), log2 domain
};

struct KeyList {
  int64_t t, lo;
  int kd;     // slots of the first part with meaning (k, k*m raw tokens, or the visible entries)
  int k_ent;  // entry part rounded up to a multiple of 4 (gather groups never straddle)
  int w_len;  // window tokens
  int len;    // k_ent + w_len
};

__device__ __forceinline__ KeyList key_list(const AttArgs& a, int i) {
  KeyList kl;
  kl.t = a.q_pos0 + i;
  kl.lo = kl.t - a.W + 1 > 0 ? kl.t - a.W + 1 : 0;
  kl.w_len = a.W > 0 ? (int)(kl.t - kl.lo + 1) : 0;
  if (a.dense) {
    int64_t nv = n_vis(kl.t, a.m);
    kl.kd = (int)(nv < a.N ? nv : a.N);
  } else {
    kl.kd = a.rawblk ? a.k * a.m : a.k;
  }
  kl.k_ent = (kl.kd + 3) & ~3;
  kl.len = kl.k_ent + kl.w_len;
  return kl;
}

// Source row of key slot j of a query's list: an entry row (entry cache) or
// a raw row (window, or a raw-token block).  Empty slots point at a valid
// row of the same kind and are masked in the softmax.
struct SlotSrc {
  int64_t row;  // row index into the entry cache or into the raw rows
  bool win;     // a raw row
  bool valid;
};

// The index-list word of key slot j (only selected-entry slots read the list;
// the others return 0 and are resolved by slot_src from the slot number).
__device__ __forceinline__ int32_t slot_word(const AttArgs& a, const KeyList& kl, int64_t qrow,
                                             int j) {
  if ((j < kl.k_ent || a.W == 0) && j < kl.kd && !a.dense)
    return a.idx[qrow * (int64_t)a.k + (a.rawblk ? j / a.m : j)];
  return 0;
}

// `word`: slot_word of the same slot (fetched ahead of use).
__device__ __forceinline__ SlotSrc slot_src(const AttArgs& a, const KeyList& kl, int b, int j,
                                            int32_t word) {
  SlotSrc r;
  if (j < kl.k_ent || a.W == 0) {
    int64_t e = 0;
    bool v = false;
    if (j < kl.kd) {
      if (a.dense) {
        e = j;
        v = true;
      } else {
        e = word;
        v = e >= 0 && e < a.N;  // -1 (and anything out of range) is an empty slot
        if (!v) e = 0;
      }
    }
    if (a.rawblk) {
      // token j % m of block e (empty slots: the sequence's first raw row)
      r.row = (int64_t)b * a.raw_rows + (v ? e * a.m + j % a.m - a.raw_pos0 : 0);
      r.win = true;
    } else {
      r.row = (int64_t)b * a.kv_rows + e;
      r.win = false;
    }
    r.valid = v;
  } else {
    const int w = j - kl.k_ent;
    r.valid = w < kl.w_len;
    const int64_t pos = kl.lo + (r.valid ? w : 0);
    r.row = (int64_t)b * a.raw_rows + (pos - a.raw_pos0);
    r.win = true;
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

// Mixed-precision cache: the 16 bytes (8 dims, from dim c*64 + uc*8) of one
// key row that a producer thread writes into a chunk, as f16.  The raw unit
// is loaded first (all of a chunk's loads in flight), converted after.
struct MixUnit {
  uint4 v;    // kind 0: 8 bf16 values; kind 1: 8 e4m3 codes in v.x, v.y
  float inv;  // RoPE dims of an entry: 1 / row scale; else 1
  int kind;
};

// A code chunk unit of row pointer sp (the unit's bytes in chunk 0: codes of
// an entry, or bf16 values of a window row) for chunk c.
__device__ __forceinline__ MixUnit mix_load_code(const uint8_t* sp, bool win, int c) {
  MixUnit r;
  r.inv = 1.f;
  r.kind = win ? 0 : 1;
  if (win) {
    r.v = __ldg(reinterpret_cast<const uint4*>(sp + c * 128));
  } else {
    const uint2 cv = __ldg(reinterpret_cast<const uint2*>(sp + c * 64));
    r.v = make_uint4(cv.x, cv.y, 0u, 0u);
  }
  return r;
}

// Eight e4m3 codes (byte i = code i) as eight f16 values, exactly (every
// e4m3 value is an f16 value).
__device__ __forceinline__ uint4 e4m3x8_to_f16x8(uint2 w) {
  uint4 o;
  asm("{\n\t.reg .b16 a0, a1, a2, a3;\n\t"
      "mov.b32 {a0, a1}, %4;\n\t"
      "mov.b32 {a2, a3}, %5;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a0;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, a1;\n\t"
      "cvt.rn.f16x2.e4m3x2 %2, a2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %3, a3;\n\t}"
      : "=r"(o.x), "=r"(o.y), "=r"(o.z), "=r"(o.w)
      : "r"(w.x), "r"(w.y));
  return o;
}

__device__ __forceinline__ uint32_t f16x2_bits(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// A code chunk or a value chunk: the codes exactly; bf16 values (window rows)
// rounded to f16.
__device__ __forceinline__ uint4 mix_f16(const MixUnit& r) {
  uint32_t o[4];
  if (r.kind == 1) {
    return e4m3x8_to_f16x8(make_uint2(r.v.x, r.v.y));
  } else {
    const uint32_t w4[4] = {r.v.x, r.v.y, r.v.z, r.v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = f16x2_bits(bf16_lo(w4[e]), bf16_hi(w4[e]));
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// A RoPE chunk: value * inv split into an f16 high part and an f16 low part
// (the rest, rounded): together within about 2^-22 of value * inv.
__device__ __forceinline__ void mix_f16_pair(const MixUnit& r, uint4& hi, uint4& lo) {
  const uint32_t w4[4] = {r.v.x, r.v.y, r.v.z, r.v.w};
  uint32_t h[4], l[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float x0 = bf16_lo(w4[e]) * r.inv, x1 = bf16_hi(w4[e]) * r.inv;
    const __half2 hh = __floats2half2_rn(x0, x1);
    const float2 hf = __half22float2(hh);
    h[e] = *reinterpret_cast<const uint32_t*>(&hh);
    l[e] = f16x2_bits(x0 - hf.x, x1 - hf.y);
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
  uint64_t* q_full = bars + 2 * kRing;  // [kMaxQChunks]: one per Q chunk
  uint64_t* s_full = q_full + kMaxQChunks;  // [2]
  uint64_t* p_full = s_full + 2;      // [2]
  uint64_t* mask_full = p_full + 2;   // [2]
  uint64_t* mask_empty = mask_full + 2;  // [2]
  // PV(u) completes o_done[u & 1]: with two barriers no waiter can fall two
  // phases behind (a parity wait cannot tell phase j from phase j + 2)
  uint64_t* o_done = mask_empty + 2;  // [2]
  uint64_t* mma_done = o_done + 2;
  uint64_t* q_conv = mma_done + 1;  // e4m3: Q converted to f16 by every producer
  uint64_t* row_full = q_conv + 1;   // the tile's row table written
  uint64_t* row_empty = row_full + 1;  // ... and read by every producer warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(row_empty + 1);
  uint32_t* smask = tmem_slot + 4;  // [2][4] ballot words of the tile's valid slots
  float* svscale = reinterpret_cast<float*>(smask + 8);  // e4m3: [2][128] row scales of the tile
  uint32_t* srow = reinterpret_cast<uint32_t*>(svscale + 256);  // [128] row | window << 31

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* err = &g_attend_tc_error;

  // work item: (query row, value half, split)
  const int split = (int)(blockIdx.x % a.splits);
  const int half = (int)((blockIdx.x / a.splits) & 1);
  const int64_t qrow = blockIdx.x / ((int64_t)a.splits * 2);  // b * Q + i
  const int i = (int)(qrow % a.Q);
  const int b = (int)(qrow / a.Q);
  const KeyList kl = key_list(a, i);
  const int n_tiles_all = (kl.len + kT - 1) / kT;
  const int tile0 = split * a.tps;
  int n = n_tiles_all - tile0;
  if (n > a.tps) n = a.tps;
  if (n < 0) n = 0;
  const int vc0 = half * a.nvc;  // first key chunk that is a value chunk of this half

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRing; ++s) {
      tc::mbar_init(&ring_full[s], kProdWarps * 32);  // every producer thread arrives
      tc::mbar_init(&ring_empty[s], 1);
    }
    for (int c = 0; c < kMaxQChunks; ++c) tc::mbar_init(&q_full[c], 1);
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&s_full[s], 1);
      tc::mbar_init(&p_full[s], 4);
      tc::mbar_init(&mask_full[s], kProdWarps);
      tc::mbar_init(&mask_empty[s], 4);
    }
    tc::mbar_init(&o_done[0], 1);
    tc::mbar_init(&o_done[1], 1);
    tc::mbar_init(mma_done, 1);
    tc::mbar_init(q_conv, kProd);
    tc::mbar_init(row_full, kProdWarps);
    tc::mbar_init(row_empty, kProdWarps);
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tm_q);
    if (!kE4M3) {
      tc::prefetch_tmap(&tm_kv);
      if (a.W > 0) tc::prefetch_tmap(&tm_raw);
    }

  }
  if (warp == kMmaWarp) tc::tmem_alloc(tmem_slot, 512);
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < kProdWarps) {
    // ------------------------------------------------------------ producers
    // Thread pt copies the 16-byte units pt + kProd*i of every chunk (unit u:
    // row u/8, bytes 16*(u%8) of the row) with cp.async, each lane with its
    // own gathered address.  Each thread's copies of a chunk arrive on the
    // chunk's barrier by themselves when they land (cp.async.mbarrier.arrive),
    // so a producer never waits for its own copies: it runs ahead as far as
    // the ring lets it, and the MMA issuer makes the landed rows visible to
    // the tensor cores (proxy fence) after its wait.  The key-list words of
    // the next tile are fetched a whole tile ahead.
    const int pt = threadIdx.x;
    if (n > 0) {
      if (pt == 0) {
        // a barrier per chunk: the first tile's QK^T starts as its Q chunks land
        for (int c = 0; c < a.nc; ++c) {
          tc::mbar_expect_tx(&q_full[c], kChunk);
          tc::tma_load_2d(sQ + c * kChunk, &tm_q, &q_full[c], c * 64, (int)(qrow * a.H));
        }
      }
      const uint8_t* kvb = reinterpret_cast<const uint8_t*>(a.kv16);
      const uint8_t* rawb = reinterpret_cast<const uint8_t*>(a.raw16);
      const int64_t rowb = (int64_t)a.D_qk * 2;
      uint32_t pslot = 0, pph = 0;  // ring slot and the parity of its release
      bool ok = true;
      if (kE4M3) {
        // Q to f16 in place (elementwise, so the swizzle does not matter),
        // then one arrival per producer thread on q_conv
        for (int c = 0; c < a.nc && ok; ++c) ok = tc::mbar_wait(&q_full[c], 0, err, 13);
        if (ok) {
          for (int u = pt; u < a.nc * (int)(kChunk / 16); u += kProd) {
            uint4* q4 = reinterpret_cast<uint4*>(sQ) + u;
            const uint4 v = *q4;
            *q4 = make_uint4(f16x2_bits(bf16_lo(v.x), bf16_hi(v.x)),
                             f16x2_bits(bf16_lo(v.y), bf16_hi(v.y)),
                             f16x2_bits(bf16_lo(v.z), bf16_hi(v.z)),
                             f16x2_bits(bf16_lo(v.w), bf16_hi(v.w)));
          }
          tc::fence_proxy_async_smem();
          tc::mbar_arrive(q_conv);
        }
      }
      uint32_t tma_mask = 0, tma_par = 0;  // pt 0: slots whose last fill was TMA, and its parity
      // swizzled destination of each of this thread's units within a chunk;
      // only the last unit can fall outside the chunk (threads pt >= 64)
      uint32_t dso[kUnits];
#pragma unroll
      for (int i = 0; i < kUnits; ++i) {
        const int unit = pt + kProd * i;
        dso[i] = swz(unit >> 3, unit & 7);
      }
      const bool last_unit = pt + kProd * (kUnits - 1) < (int)(kChunk / 16);
      // gathered rows of tile u's units (bf16 caches: the byte address of the
      // unit in chunk 0; mixed caches: the row and its kind), and the two mask
      // slots of each thread
      struct TileRows {
        uint32_t rr[kUnits];  // the rows (fewer than 2^31 in all)
        const uint8_t* sp[kUnits];
        uint32_t wb;
        SlotSrc s0, s1;
        int tma;    // bf16 caches: 1 = 128 consecutive entry rows, 2 = 128 consecutive
        int tma_y;  //   raw rows (from tma_y), loaded by one TMA box per chunk; 0 = gathered
        bool code_only;  // mixed caches: no window row among the warp's units
      };
      auto issue_chunk = [&](int c, const TileRows& t) -> bool {
        int okw = 1;
        if (lane == 0) okw = tc::mbar_wait(&ring_empty[pslot], pph ^ 1, err, 11);
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (!okw) return false;
        const uint32_t dst = tc::smem_u32(sRing + pslot * kChunk);
        if (!kE4M3 && t.tma) {
          // one TMA box: the chunk's barrier completes on its bytes and on
          // every producer's own arrival (thread 0's carries the byte count).
          // Each producer arrives itself, after its warp saw the slot
          // released: a warp that skipped the chunks of a run of boxes could
          // fall two fills behind the ring, where a parity wait takes the
          // release it waits for to be still pending.
          if (pt == 0) {
            tc::mbar_expect_tx(&ring_full[pslot], kChunk);
            tma_mask |= 1u << pslot;
            tma_par = (tma_par & ~(1u << pslot)) | (pph << pslot);
            tc::tma_load_2d(sRing + pslot * kChunk, t.tma == 1 ? &tm_kv : &tm_raw,
                            &ring_full[pslot], c * 64, t.tma_y);
          } else {
            tc::mbar_arrive(&ring_full[pslot]);
          }
        } else if (kE4M3) {
          // every load of the chunk in flight first, then the conversions
          MixUnit raw[kUnits];
#pragma unroll
          for (int i = 0; i < kUnits; ++i) {
            const int unit = pt + kProd * i;
            if (unit < (int)(kChunk / 16))
              raw[i] = mix_load_code(t.sp[i], (t.wb >> i) & 1, c);
          }
#pragma unroll
          for (int i = 0; i < kUnits; ++i) {
            const int unit = pt + kProd * i;
            if (unit < (int)(kChunk / 16))
              *reinterpret_cast<uint4*>(sRing + pslot * kChunk + dso[i]) = mix_f16(raw[i]);
          }
          tc::fence_proxy_async_smem();
          tc::mbar_arrive(&ring_full[pslot]);
        } else {
          const int coff = c * 128;
#pragma unroll
          for (int i = 0; i < kUnits; ++i)
            if (i < kUnits - 1 || last_unit) cp_async16(dst + dso[i], t.sp[i] + coff);
          cp_async_arrive_noinc(&ring_full[pslot]);
          if (pt == 0) tma_mask &= ~(1u << pslot);
        }
        if (++pslot == kRing) {
          pslot = 0;
          pph ^= 1;
        }
        return true;
      };
      // Mixed caches: two code chunks per round (c0 of rows t0, c1 of rows t1)
      // into the next two slots.  A producer thread's loads of a chunk wait
      // one memory latency, so it keeps two chunks' loads in flight, issued
      // before the slots are known to be free.
      auto issue_code2 = [&](int c0, const TileRows& t0, int c1, const TileRows& t1) -> bool {
        const uint32_t s0 = pslot, p0 = pph;
        const uint32_t s1 = pslot + 1 == kRing ? 0 : pslot + 1;
        const uint32_t p1 = s1 == 0 ? pph ^ 1 : pph;
        auto wait_slots = [&]() -> bool {
          int okw = 1;
          if (lane == 0)
            okw = tc::mbar_wait(&ring_empty[s0], p0 ^ 1, err, 11) &&
                  tc::mbar_wait(&ring_empty[s1], p1 ^ 1, err, 11);
          return __shfl_sync(0xffffffffu, okw, 0) != 0;
        };
        if (t0.code_only && t1.code_only) {
          // codes only (warp-uniform): 8 bytes per unit, widened in registers
          uint2 v0[kUnits], v1[kUnits];
#pragma unroll
          for (int i = 0; i < kUnits; ++i)
            if (i < kUnits - 1 || last_unit) {
              v0[i] = __ldg(reinterpret_cast<const uint2*>(t0.sp[i] + c0 * 64));
              v1[i] = __ldg(reinterpret_cast<const uint2*>(t1.sp[i] + c1 * 64));
            }
          if (!wait_slots()) return false;
#pragma unroll
          for (int i = 0; i < kUnits; ++i)
            if (i < kUnits - 1 || last_unit) {
              *reinterpret_cast<uint4*>(sRing + s0 * kChunk + dso[i]) = e4m3x8_to_f16x8(v0[i]);
              *reinterpret_cast<uint4*>(sRing + s1 * kChunk + dso[i]) = e4m3x8_to_f16x8(v1[i]);
            }
        } else {
          MixUnit raw0[kUnits], raw1[kUnits];
#pragma unroll
          for (int i = 0; i < kUnits; ++i)
            if (i < kUnits - 1 || last_unit) {
              raw0[i] = mix_load_code(t0.sp[i], (t0.wb >> i) & 1, c0);
              raw1[i] = mix_load_code(t1.sp[i], (t1.wb >> i) & 1, c1);
            }
          if (!wait_slots()) return false;
#pragma unroll
          for (int i = 0; i < kUnits; ++i)
            if (i < kUnits - 1 || last_unit) {
              *reinterpret_cast<uint4*>(sRing + s0 * kChunk + dso[i]) = mix_f16(raw0[i]);
              *reinterpret_cast<uint4*>(sRing + s1 * kChunk + dso[i]) = mix_f16(raw1[i]);
            }
        }
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&ring_full[s0]);
        tc::mbar_arrive(&ring_full[s1]);
        pslot = s1 + 1 == kRing ? 0 : s1 + 1;
        pph = pslot == 0 ? p1 ^ 1 : p1;
        return true;
      };
      // Mixed caches: the high and the low part of RoPE chunk c (over the row
      // scale) go to two consecutive slots from one load.  Every unit's value
      // and scale loads are issued first, without branches (a window row
      // reads scale 0 and takes 1), so that no load waits for the division
      // of an earlier unit; then the slots are waited for.
      auto issue_pair = [&](int c, const TileRows& t) -> bool {
        const uint32_t s0 = pslot, p0 = pph;
        const uint32_t s1 = pslot + 1 == kRing ? 0 : pslot + 1;
        const uint32_t p1 = s1 == 0 ? pph ^ 1 : pph;
        const int d0 = c * 64 + (lane & 7) * 8;  // unit & 7 == lane & 7
        const int rw = a.D_qk - a.nope;
        uint4 rv[kUnits];
        float ks[kUnits];
#pragma unroll
        for (int i = 0; i < kUnits; ++i)
          if (i < kUnits - 1 || last_unit) {
            const bool win = (t.wb >> i) & 1;
            const int64_t row = t.rr[i];
            const uint16_t* src = win ? a.raw16 + row * a.D_qk + d0 : a.rope + row * rw + (d0 - a.nope);
            rv[i] = __ldg(reinterpret_cast<const uint4*>(src));
            ks[i] = __ldg(a.kscale + (win ? 0 : row));
          }
        int okw = 1;
        if (lane == 0)
          okw = tc::mbar_wait(&ring_empty[s0], p0 ^ 1, err, 11) &&
                tc::mbar_wait(&ring_empty[s1], p1 ^ 1, err, 11);
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (!okw) return false;
#pragma unroll
        for (int i = 0; i < kUnits; ++i) {
          if (i < kUnits - 1 || last_unit) {
            MixUnit r;
            r.v = rv[i];
            r.kind = 0;
            r.inv = ((t.wb >> i) & 1) ? 1.f : 1.f / ks[i];
            uint4 hi, lo;
            mix_f16_pair(r, hi, lo);
            *reinterpret_cast<uint4*>(sRing + s0 * kChunk + dso[i]) = hi;
            *reinterpret_cast<uint4*>(sRing + s1 * kChunk + dso[i]) = lo;
          }
        }
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&ring_full[s0]);
        tc::mbar_arrive(&ring_full[s1]);
        pslot = s1 + 1 == kRing ? 0 : s1 + 1;
        pph = pslot == 0 ? p1 ^ 1 : p1;
        return true;
      };
      // The tile's 128 key rows go through a table in shared memory: thread
      // pt resolves slots pt and pt + 96 (which it needs for the softmax's
      // masks anyway) and writes them; after every producer has, it reads the
      // rows of its own units (unit i: row pt/8 + 12 i).  row_full / row_empty
      // (one arrival per producer warp) order the writes of a table against
      // the reads of the one before it.  Key-list words are fetched a tile
      // ahead.
      struct TileWords {
        int32_t w[2];
      };
      const bool has1 = pt + kProd < kT;
      auto tile_words = [&](int u, TileWords& t) {
        const int jt = (tile0 + u) * kT;
        t.w[0] = slot_word(a, kl, qrow, jt + pt);
        t.w[1] = slot_word(a, kl, qrow, jt + (has1 ? pt + kProd : pt));
      };
      int tbl = 0;  // tables written so far
      auto tile_rows = [&](int u, const TileWords& tw, TileRows& t) -> bool {
        const int jt = (tile0 + u) * kT;
        t.s0 = slot_src(a, kl, b, jt + pt, tw.w[0]);
        t.s1 = slot_src(a, kl, b, jt + (has1 ? pt + kProd : pt), tw.w[1]);
        // every warp has read the previous table
        if (tbl > 0 && !tc::mbar_wait(row_empty, (tbl - 1) & 1, err, 14)) return false;
        srow[pt] = (uint32_t)t.s0.row | (t.s0.win ? 0x80000000u : 0u);
        if (has1) srow[pt + kProd] = (uint32_t)t.s1.row | (t.s1.win ? 0x80000000u : 0u);
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(row_full);
        if (!tc::mbar_wait(row_full, tbl & 1, err, 15)) return false;
        t.wb = 0;
#pragma unroll
        for (int i = 0; i < kUnits; ++i) {
          const int r = (i < kUnits - 1 || last_unit) ? (pt >> 3) + (kProd / 8) * i : 0;
          const uint32_t v = srow[r];
          const int64_t row = (int64_t)(v & 0x7fffffffu);
          const bool win = (v >> 31) != 0;
          t.rr[i] = (uint32_t)row;
          t.wb |= (win ? 1u : 0u) << i;
          t.sp[i] = win ? rawb + row * rowb + (lane & 7) * 16
                  : (kE4M3 ? a.codes + row * a.nope + (lane & 7) * 8
                           : kvb + row * rowb + (lane & 7) * 16);
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(row_empty);
        ++tbl;
        t.code_only = kE4M3 && __all_sync(0xffffffffu, t.wb == 0);
        t.tma = 0;
        t.tma_y = 0;
        if (!kE4M3) {
          if (a.dense && jt + kT <= kl.kd) {
            // every slot a valid entry, entry j in row j (a tile with masked
            // slots is gathered: rows past the valid entries may hold anything,
            // and a masked slot's row still meets a zero weight in P . V)
            t.tma = 1;
            t.tma_y = (int)((int64_t)b * a.kv_rows + jt);
          } else if (a.W > 0 && jt >= kl.k_ent) {
            // every slot a window slot: raw rows lo + (j - k_ent) (past the
            // window: masked; past the cache: zero-filled)
            t.tma = 2;
            t.tma_y = (int)((int64_t)b * a.raw_rows + (kl.lo - a.raw_pos0) + (jt - kl.k_ent));
          }
        }
        return true;
      };
      TileRows cur, prev;
      TileWords wnext;
      tile_words(0, wnext);
      ok = ok && tile_rows(0, wnext, cur);
      for (int u = 0; u <= n && ok; ++u) {
        if (u + 1 < n) tile_words(u + 1, wnext);  // in flight during this tile's issues
        if (u < n) {
          // validity of slots pt and pt + 96 (and, for mixed caches, the scale
          // of their value rows) for the softmax: ballot word w covers slots
          // 32w .. 32w+31
          int okw = 1;
          if (lane == 0) okw = tc::mbar_wait(&mask_empty[u & 1], ((u >> 1) & 1) ^ 1, err, 12);
          okw = __shfl_sync(0xffffffffu, okw, 0);
          if (!okw) break;
          const uint32_t bal0 = __ballot_sync(0xffffffffu, cur.s0.valid);
          const uint32_t bal1 = __ballot_sync(0xffffffffu, has1 && cur.s1.valid);
          if (lane == 0) {
            smask[(u & 1) * 4 + warp] = bal0;
            if (warp == 0) smask[(u & 1) * 4 + 3] = bal1;
          }
          // mixed caches: the value rows' scales load while the QK^T chunks
          // are issued; the words are published after them (the softmax
          // needs them only once S is complete)
          float ksv0 = 1.f, ksv1 = 1.f;
          if (kE4M3) {
            if (cur.s0.valid && !cur.s0.win) ksv0 = __ldg(a.kscale + cur.s0.row);
            if (has1 && cur.s1.valid && !cur.s1.win) ksv1 = __ldg(a.kscale + cur.s1.row);
          } else {
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&mask_full[u & 1]);
          }
          // QK^T chunks: the nc chunks in order; mixed caches' RoPE chunks as
          // (high, low) pairs
          const int ncode = kE4M3 ? a.nope / 64 : a.nc;
          if (kE4M3) {
            int c = 0;
            for (; c + 1 < ncode && ok; c += 2) ok = issue_code2(c, cur, c + 1, cur);
            if (c < ncode && ok) ok = issue_chunk(c, cur);
          } else {
            for (int c = 0; c < ncode && ok; ++c) ok = issue_chunk(c, cur);
          }
          if (kE4M3) {
            for (int c = ncode; c < a.nc && ok; ++c) ok = issue_pair(c, cur);
            svscale[(u & 1) * 128 + pt] = ksv0;
            if (has1) svscale[(u & 1) * 128 + pt + kProd] = ksv1;
            __syncwarp();
            if (lane == 0 && ok) tc::mbar_arrive(&mask_full[u & 1]);
          }
        }
        if (u >= 1)
          if (kE4M3) {
            int c = 0;
            for (; c + 1 < a.nvc && ok; c += 2) ok = issue_code2(vc0 + c, prev, vc0 + c + 1, prev);
            if (c < a.nvc && ok) ok = issue_chunk(vc0 + c, prev);
          } else {
            for (int c = 0; c < a.nvc && ok; ++c) ok = issue_chunk(vc0 + c, prev);
          }
        prev = cur;
        if (u + 1 < n && ok) ok = tile_rows(u + 1, wnext, cur);
      }
      // every copy must land before the CTA can exit: this thread's cp.async
      // (their arrivals on the ring barriers happen by themselves), and (pt 0)
      // the Q load and the ring's TMA boxes not yet known to have landed
      // (only after an error: otherwise the MMA issuer waited for all of them;
      // a box whose barrier also misses the arrival of a producer that gave up
      // is waited for up to the bounded-wait limit, long after it landed)
      cp_async_wait<0>();
      if (pt == 0) {
        for (int c = 0; c < a.nc; ++c) tc::mbar_drain(&q_full[c], 0);
        for (int s = 0; s < kRing; ++s)
          if ((tma_mask >> s) & 1u) tc::mbar_drain(&ring_full[s], (tma_par >> s) & 1u);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      // bf16 operands, or f16 for mixed caches (format 1 / 0 of kind::f16)
      const uint32_t fmt = kE4M3 ? 0u : 1u;
      const uint32_t id_s = tc::idesc(128, kT, fmt, fmt);
      const uint32_t id_pv = tc::idesc(128, 64, fmt, fmt, 0, 1);
      bool ok = true;
      // test aid: the producers' first loads are in flight while this waits
      if (a.stall && blockIdx.x == 0) ok = tc::flag_wait(&g_attend_never_set, tc::kStallNs, err, 28);
      uint32_t q_seen = 0;  // Q chunks known to have landed
      // descriptors of Q chunk 0 and ring slot 0 (K-major for S, MN-major
      // for PV); other chunks / slots / K steps are constant offsets in the
      // start-address field, so each MMA costs the issuing thread a couple of
      // integer adds (building descriptors per MMA made this loop, not the
      // tensor core, the limit)
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
      auto issue_pv = [&](int u) -> bool {
        const uint32_t sb = u & 1;
        if (!tc::mbar_wait(&p_full[sb], (u >> 1) & 1, err, 22)) return false;
        tc::tc_fence_after();
        const uint32_t p_tmem = tmem + sb * 128;
        for (int c = 0; c < a.nvc; ++c) {
          if (!tc::mbar_wait(&ring_full[slot], ph, err, 23)) return false;
          if (!kE4M3) tc::fence_proxy_async_smem();  // cp.async rows -> tensor cores
          tc::tc_fence_after();
          const uint64_t vd = vd0 + slot * kChunk16;
          const uint32_t o_tmem = tmem + 256 + 64 * c;
#pragma unroll
          for (int ks = 0; ks < kT / 16; ++ks) {
            // 16 keys per K step: 16 rows of 128 bytes
            const uint64_t bd = vd + (uint64_t)(ks * (2048 >> 4));
            tc::mma_bf16_ts(o_tmem, p_tmem + 8 * ks, bd, id_pv, (u > 0 || ks > 0) ? 1u : 0u);
          }
          tc::mma_commit(&ring_empty[slot]);
          next_slot();
        }
        tc::mma_commit(&o_done[u & 1]);
        return true;
      };
      for (int u = 0; u < n && ok; ++u) {
        const uint32_t sb = u & 1;
        const uint32_t s_tmem = tmem + sb * 128;
        for (int cc = 0; cc < a.nsc && ok; ++cc) {
          // the Q chunk this key chunk meets (the producers' order: the code
          // chunks, then mixed caches' (high, low) pairs of the RoPE chunks)
          const int ncode = kE4M3 ? a.nope / 64 : a.nc;
          const int c = cc < ncode ? cc : ncode + ((cc - ncode) >> 1);
          if (kE4M3) {
            if (!q_seen && !tc::mbar_wait(q_conv, 0, err, 21)) { ok = false; break; }
            q_seen = 1;
          } else if (!((q_seen >> c) & 1u)) {
            if (!tc::mbar_wait(&q_full[c], 0, err, 21)) { ok = false; break; }
            q_seen |= 1u << c;
          }
          if (!tc::mbar_wait(&ring_full[slot], ph, err, 24)) { ok = false; break; }
          if (!kE4M3) tc::fence_proxy_async_smem();  // cp.async rows -> tensor cores
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
        if (u >= 1) ok = issue_pv(u - 1);
      }
      if (ok) issue_pv(n - 1);
      // every MMA issued must have completed before TMEM is released
      tc::mma_commit(mma_done);
      tc::mbar_drain(mma_done, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax (warps 4-7)
    const int quarter = warp & 3;
    const int h = quarter * 32 + lane;  // head row == TMEM lane
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    float m_ref = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int u = 0; u < n && ok; ++u) {
      const uint32_t sb = u & 1;
      // every lane acquires the producer's ballot words itself
      const bool mk = tc::mbar_wait(&mask_full[sb], (u >> 1) & 1, err, 31);
      if (!__all_sync(0xffffffffu, mk)) { ok = false; break; }
      uint32_t bal[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        bal[q] = *reinterpret_cast<volatile uint32_t*>(&smask[sb * 4 + q]);
      __syncwarp();
      if (!kE4M3 && lane == 0) tc::mbar_arrive(&mask_empty[sb]);
      int okw = lane == 0 ? (int)tc::mbar_wait(&s_full[sb], (u >> 1) & 1, err, 32) : 0;
      okw = __shfl_sync(0xffffffffu, okw, 0);
      __syncwarp();
      if (!okw) { ok = false; break; }
      tc::tc_fence_after();
      float x[kT];
#pragma unroll
      for (int g = 0; g < kT / 32; ++g) {
        uint32_t r[32];
        tc::tmem_ld32(tmem + lane_base + sb * 128 + g * 32, r);
        tc::tmem_wait_ld();
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) x[g * 32 + jj] = __uint_as_float(r[jj]);
      }
      float m_tile = -INFINITY;
#pragma unroll
      for (int j = 0; j < kT; ++j) {
        const bool v = (bal[j >> 5] >> (j & 31)) & 1u;
        // mixed caches: the tile holds S' = S / c_j
        x[j] = v ? x[j] * (kE4M3 ? a.c_log2 * svscale[sb * 128 + j] : a.c_log2) : -INFINITY;
        m_tile = fmaxf(m_tile, x[j]);
      }
      const bool grow = m_tile > m_ref + kRescaleLog2;
      const bool rescale = grow && m_ref != -INFINITY;
      const float alpha = grow ? exp2f(m_ref - m_tile) : 1.f;
      if (__any_sync(0xffffffffu, rescale)) {
        // O holds the tiles before u: wait for PV(u-1), then scale the rows
        okw = lane == 0 ? (int)tc::mbar_wait(&o_done[(u - 1) & 1], ((u - 1) >> 1) & 1, err, 33) : 0;
        okw = __shfl_sync(0xffffffffu, okw, 0);
        __syncwarp();
        if (!okw) { ok = false; break; }
        tc::tc_fence_after();
        const float f = rescale ? alpha : 1.f;
        for (int g = 0; g < 256 / 32; ++g) {
          uint32_t r[32];
          tc::tmem_ld32(tmem + lane_base + 256 + g * 32, r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) r[jj] = __float_as_uint(__uint_as_float(r[jj]) * f);
          tc::tmem_st32(tmem + lane_base + 256 + g * 32, r);
        }
        tc::tmem_wait_st();
      }
      if (grow) {
        l_run *= alpha;
        m_ref = m_tile;
      }
      // P = 2^(x - m_ref) as bf16 pairs over the first 64 columns of the buffer
      // (mixed caches: P times the value row's scale, as f16 pairs)
#pragma unroll
      for (int j = 0; j < kT; ++j) {
        const float pj = m_ref == -INFINITY ? 0.f : exp2f(x[j] - m_ref);
        l_run += pj;
        x[j] = kE4M3 ? pj * svscale[sb * 128 + j] : pj;
      }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c)
          pk[c] = kE4M3 ? f16x2_bits(x[hh * 64 + 2 * c], x[hh * 64 + 2 * c + 1])
                        : pack_bf16(x[hh * 64 + 2 * c], x[hh * 64 + 2 * c + 1]);
        tc::tmem_st32(tmem + lane_base + sb * 128 + hh * 32, pk);
      }
      tc::tmem_wait_st();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (kE4M3) tc::mbar_arrive(&mask_empty[sb]);
        tc::mbar_arrive(&p_full[sb]);
      }
    }
    // ------------------------------------------------------------ epilogue
    bool have_o = ok && n > 0;
    if (have_o) {
      // PV(n-1) is the ((n-1)/2)-th completion of o_done[(n-1) & 1]; that
      // barrier cannot be further ahead (no PV(n+1))
      int okw = 1;
      if (lane == 0) okw = tc::mbar_wait(&o_done[(n - 1) & 1], ((n - 1) >> 1) & 1, err, 35);
      okw = __shfl_sync(0xffffffffu, okw, 0);
      __syncwarp();
      have_o = okw != 0;
      tc::tc_fence_after();
    }
    if (ok) {
      const int hv = a.D_v / 2;
      const int64_t orow = qrow * a.H + h;
      if (a.splits == 1) {
        const float inv = (have_o && l_run > 0.f) ? 1.f / l_run : 0.f;
        for (int g = 0; g < hv / 32; ++g) {
          uint32_t r[32];
          if (have_o) {
            tc::tmem_ld32(tmem + lane_base + 256 + g * 32, r);
            tc::tmem_wait_ld();
          }
          const int64_t o0 = orow * a.D_v + half * hv + g * 32;
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
        const int64_t prow = orow * a.splits + split;
        float4* dst = reinterpret_cast<float4*>(a.part + prow * a.D_v + half * hv);
        for (int g = 0; g < hv / 32; ++g) {
          uint32_t r[32];
          if (have_o) {
            tc::tmem_ld32(tmem + lane_base + 256 + g * 32, r);
            tc::tmem_wait_ld();
          }
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            float4 o;
            o.x = have_o ? __uint_as_float(r[4 * v + 0]) : 0.f;
            o.y = have_o ? __uint_as_float(r[4 * v + 1]) : 0.f;
            o.z = have_o ? __uint_as_float(r[4 * v + 2]) : 0.f;
            o.w = have_o ? __uint_as_float(r[4 * v + 3]) : 0.f;
            dst[g * 8 + v] = o;
          }
        }
        if (half == 0) {
          a.ml[prow * 2 + 0] = have_o ? m_ref : -INFINITY;
          a.ml[prow * 2 + 1] = have_o ? l_run : 0.f;
        }
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

// Longest key list of the launch, in tiles.
int max_tiles(const csa_params& p, int Q, int64_t N, int mode, int64_t q_pos0) {
  const bool dense = mode == kAttendDense;
  int64_t kd;
  if (dense) {
    kd = n_vis(q_pos0 + Q - 1, p.m);
    if (kd > N) kd = N;
  } else {
    kd = mode == kAttendRawBlocks ? (int64_t)p.k * p.m : (int64_t)p.k;
  }
  const int64_t len = ((kd + 3) & ~3ll) + p.window;
  return (int)ceil_div(len, kT);
}

}  // namespace

// Split plan of the tensor-core path: one split per (query, half) for
// multi-query launches; decode (one query per sequence) cuts the key list
// into runs of tiles (more per run when that would exceed 16 runs), so a CTA
// pipelines several tiles and writes one partial for them.  Runs are 5 tiles
// for lists up to 16 tiles (a CSA list of 1,152 keys: 5 + 4), 8 for longer
// ones (raw-token and HCA lists: fewer, longer CTAs measured faster), and
// mixed caches, whose CTAs spend longer per tile, split no list of up to 12
// tiles.  Depends on Q, the key-list length and the cache format only, never
// on the batch.
constexpr int kDecodeTiles = 5;
constexpr int kDecodeTilesLong = 8;
constexpr int kDecodeTilesMixed = 12;

void attend_tc_plan(const csa_params& p, int Q, int64_t N, int mode, int64_t q_pos0, bool mixed,
                    int* splits, int* tps) {
  const int nt = max_tiles(p, Q, N, mode, q_pos0);
  const int run = mixed ? kDecodeTilesMixed : (nt > 16 ? kDecodeTilesLong : kDecodeTiles);
  if (Q > 1 || nt <= run) {
    *splits = 1;
    *tps = nt > 0 ? nt : 1;
    return;
  }
  int t = (int)ceil_div(nt, 16);
  if (t < run) t = run;
  *tps = t;
  *splits = (int)ceil_div(nt, t);
}

// Scratch for the split partials.  A shorter key list can take more splits
// (17 tiles: 9 splits of 2; 16 tiles: 16 splits of 1), so the bound is
// min(16, tiles of the longest list).
size_t attend_tc_workspace(const csa_params& p, int Q, int64_t N, int mode, int64_t q_pos0) {
  int splits, tps;
  attend_tc_plan(p, Q, N, mode, q_pos0, false, &splits, &tps);  // the most splits of either format
  if (splits <= 1) return 0;
  const int nt = max_tiles(p, Q, N, mode, q_pos0);
  splits = nt < 16 ? nt : 16;
  const size_t rows = (size_t)p.B * Q * p.H * splits;
  const size_t part = (rows * p.D_v * sizeof(float) + 255) & ~(size_t)255;
  return part + rows * 2 * sizeof(float);
}

bool attend_tc_supported(const csa_params& p, csa_dtype q_dtype, const csa_rows& kv,
                         const csa_rows& raw, int Q, int64_t N, csa_dtype out_dtype, int mode) {
  const bool rawblk = mode == kAttendRawBlocks;
  if (q_dtype != CSA_BF16) return false;
  if (out_dtype != CSA_BF16 && out_dtype != CSA_F32) return false;
  if (p.H != 128) return false;
  if (p.D_qk % 64 != 0 || p.D_qk / 64 > kMaxQChunks) return false;
  if (p.D_v % 128 != 0 || p.D_v > 512 || p.D_v > p.D_qk) return false;
  if (N < 1) return false;
  if (rawblk) {
    if (raw.dtype != CSA_BF16) return false;
  } else if (kv.dtype == CSA_E4M3) {
    if (kv.nope != p.D_v || kv.nope % 64 != 0) return false;
  } else if (kv.dtype != CSA_BF16) {
    return false;
  }
  if ((p.window > 0 || rawblk) && raw.dtype != CSA_BF16) return false;
  if ((int64_t)p.B * kv.n_rows >= (1ll << 31)) return false;
  if ((p.window > 0 || rawblk) && (int64_t)p.B * raw.n_rows >= (1ll << 31)) return false;
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
  a.B = p.B;
  a.Q = Q;
  a.H = p.H;
  a.D_qk = p.D_qk;
  a.D_v = p.D_v;
  a.k = p.k;
  a.W = p.window;
  a.m = p.m;
  a.nc = p.D_qk / 64;
  // mixed caches: each RoPE chunk takes two slots (high and low part)
  a.nsc = a.nc + (kv.dtype == CSA_E4M3 && mode != kAttendRawBlocks ? a.nc - kv.nope / 64 : 0);
  a.nvc = p.D_v / 128;
  a.dense = mode == kAttendDense ? 1 : 0;
  a.rawblk = mode == kAttendRawBlocks ? 1 : 0;
  a.e4m3 = kv.dtype == CSA_E4M3 && !a.rawblk ? 1 : 0;
  a.stall = take_debug_stall(kStallAttend) ? 1 : 0;
  a.N = N;
  a.kv_rows = kv.n_rows;
  a.raw_rows = (p.window > 0 || a.rawblk) ? raw.n_rows : 0;
  a.raw_pos0 = raw_pos0;
  a.q_pos0 = q_pos0;
  a.c_log2 = p.scale * 1.4426950408889634f;
  a.idx = idx;
  a.kv16 = reinterpret_cast<const uint16_t*>(kv.data);
  a.codes = reinterpret_cast<const uint8_t*>(kv.data);
  a.rope = reinterpret_cast<const uint16_t*>(kv.rope);
  a.kscale = kv.scale;
  a.nope = kv.dtype == CSA_E4M3 ? kv.nope : p.D_qk;
  a.raw16 = reinterpret_cast<const uint16_t*>(raw.data);
  a.out = out;
  a.out_f32 = out_dtype == CSA_F32 ? 1 : 0;
  attend_tc_plan(p, Q, N, mode, q_pos0, a.e4m3 != 0, &a.splits, &a.tps);
  // partials at the front of the workspace, (max, sum) pairs after them
  const size_t rows = (size_t)p.B * Q * p.H * a.splits;
  a.part = reinterpret_cast<float*>(ws);
  a.ml = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) +
                                  ((rows * p.D_v * sizeof(float) + 255) & ~(size_t)255));

  CUtensorMap tm_q, tm_kv, tm_raw;
  memset(&tm_kv, 0, sizeof(tm_kv));
  memset(&tm_raw, 0, sizeof(tm_raw));
  if (!make_map_bf16(&tm_q, q, (int64_t)p.B * Q * p.H, p.D_qk, 128)) return cudaErrorInvalidValue;
  // bf16 caches: dense runs of entry rows and window rows load as 128-row boxes
  // the producers pass rows around as 31-bit indices
  if ((int64_t)p.B * kv.n_rows > 0x7fffffff || (int64_t)p.B * raw.n_rows > 0x7fffffff)
    return cudaErrorInvalidValue;
  if (!a.e4m3) {
    if (!make_map_bf16(&tm_kv, kv.data, (int64_t)p.B * kv.n_rows, p.D_qk, 128))
      return cudaErrorInvalidValue;
    if (p.window > 0 &&
        !make_map_bf16(&tm_raw, raw.data, (int64_t)p.B * raw.n_rows, p.D_qk, 128))
      return cudaErrorInvalidValue;
  }
  const int64_t grid = (int64_t)p.B * Q * 2 * a.splits;
  if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
  const size_t smem = 1024 + (size_t)a.nc * kChunk + (size_t)kRing * kChunk +
                      (2 * kRing + 14 + kMaxQChunks) * sizeof(uint64_t) + 16 + 32 + 2 * 128 * sizeof(float) +
                      128 * sizeof(uint32_t);
  cudaError_t e;
  if (a.e4m3) {
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
