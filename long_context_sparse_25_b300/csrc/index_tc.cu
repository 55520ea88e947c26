// Tensor-core path of the lightning indexer (tcgen05 MMA, TMEM accumulators,
// TMA-fed shared-memory ring).
//
//   I[b,i,s] = sum_j w[b,i,j] * max(0, q_idx[b,i,j,:] . keys[b,s,:])
//
// Sources: "一文搞懂 DeepSeek：从 V3 的 KV 压缩与 MoE，到 V4 的百万 token 上下文",
// section "V4 改进一：CSA 与 HCA" (the lightning indexer scores every compressed
// entry); "DeepSeek-V4 详解" section 2.2 Step 2 (DSA-style indexer in FP8).
//
// Mapping.  One MMA tile is D[128 keys x NQ*H_I] = K_tile[128 x d_I] .
// Qblk[NQ*H_I x d_I]^T: the keys are the M side, so that each TMEM lane (one
// thread of the epilogue) holds every head of its key and the head reduction
// sum_j w_j ReLU(.) stays inside one thread.  Decode (one query per sequence)
// uses N = 64 and streams the key cache from HBM; prefill packs NQ = 4 queries
// (N = 256) so that each key tile read from L2 feeds 4x more MMA work.
//
// Roles (warp-specialised, one CTA per SM, persistent):
//   warp 0      TMA producer: key tiles into a ring of stages (128 KB of
//               32 KB bf16 tiles, 192 KB of 16 KB e4m3 tiles in flight),
//               query blocks into one or two B buffers;
//   warp 1      TMEM allocator and MMA issuer (one thread; descriptors are
//               advanced by constant offsets in an unrolled K loop, and the
//               next stage's and accumulator's barriers are probed ahead);
//   warps 2-9   two epilogue warpgroups: tcgen05.ld of the accumulator, ReLU,
//               weighted head sum, e4m3 row scales, coalesced fp32 stores of
//               the scores.  They take alternate tiles (decode) or split the
//               queries of an N = 256 tile (prefill).
// Up to eight accumulators live in TMEM, so the MMA of a tile never waits for
// the epilogue of an earlier one.
//
// FP4 keys ("一文搞懂 DeepSeek" section "V4 的其他升级": the indexer's QK path
// in FP4, dequantised to FP8 without loss): the producer's TMA brings a tile
// of packed E2M1 codes (half the bytes) into a staging buffer, two converter
// warps turn every code into its E4M3 code (each E2M1 value is an E4M3 value)
// in the 128-byte swizzled layout of the e4m3 stage, and the MMA and the
// epilogue run as for e4m3 keys (the row scale is applied to the score).  Every mbarrier wait is bounded; a timeout
// is recorded in a device error word (read by csa_device_status) and the
// kernel returns.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace csa {

namespace {

__device__ int g_index_tc_error = 0;
__device__ int g_index_never_set = 0;  // the test aid's flag: nothing sets it

constexpr int kTileKeys = 128;
constexpr int kMaxAcc = 8;  // accumulator buffers in TMEM (up to 512 columns)

struct TcArgs {
  int B, Q, H_I, d_I, m, NQ, nQB, tps;  // tps: key tiles per sequence (all N)
  int64_t N, n_rows, q_pos0;
  int mode;                             // 0: every query block sees all tiles; 1: causal units
  int64_t total;                        // mode 0: B*nQB*tps tiles; mode 1: B*nQB units
  int stages, nb, nacc;  // nacc: TMEM accumulator buffers, a power of two
  int alt;               // 1: the two epilogue warpgroups take alternate tiles (all queries)
  uint32_t a_bytes, b_bytes, a_chunk_bytes, b_chunk_bytes;
  int chunk_elems, n_chunks, ksteps;
  uint32_t tmem_cols;
  int stall;  // test aid: CTA 0's MMA issuer first waits on a flag that nothing sets
  uint32_t stg_bytes;  // FP4 keys: bytes of a staged tile of codes
  const float* w;
  const float* q_scale;  // e4m3 only
  const float* k_scale;  // e4m3 only
  void* scores;      // [B, Q, N] fp32, or bf16 bit patterns (scores_bf16)
  int scores_bf16;
};

__device__ __forceinline__ int tiles_visible(const TcArgs& a, int qb) {
  int last = (qb + 1) * a.NQ;
  if (last > a.Q) last = a.Q;
  int64_t nv = n_vis(a.q_pos0 + last - 1, a.m);
  if (nv > a.N) nv = a.N;
  return (int)((nv + kTileKeys - 1) / kTileKeys);
}

// The (b, qb, kt) tiles of one CTA, in the same order for every role.  The
// sizes it walks by are copied into the struct (registers): read through a
// pointer to the kernel's parameters they were generic loads of parameter
// space on every tile, a few hundred cycles of the MMA issuer's loop.
struct Sched {
  int mode, tps, nQB, B, c, G;
  int64_t total;
  int64_t t, t_end;  // mode 0
  int64_t r;         // mode 1: round
  int b, qb, kt, kt_end;

  __device__ void init(const TcArgs& args, int cta, int grid) {
    mode = args.mode;
    tps = args.tps;
    nQB = args.nQB;
    B = args.B;
    total = args.total;
    c = cta;
    G = grid;
    if (mode == 0) {
      t = total * cta / grid;
      t_end = total * (cta + 1) / grid;
      // position of tile t, then walked forward without divisions
      const int64_t per_b = (int64_t)nQB * tps;
      b = (int)(t / per_b);
      qb = (int)((t / tps) % nQB);
      kt = (int)(t % tps);
    } else {
      r = 0;
      kt = 0;
      kt_end = 0;
    }
  }

  __device__ bool next(const TcArgs& args, int& ob, int& oqb, int& okt) {
    if (mode == 0) {
      if (t >= t_end) return false;
      ob = b;
      oqb = qb;
      okt = kt;
      ++t;
      if (++kt == tps) {
        kt = 0;
        if (++qb == nQB) {
          qb = 0;
          ++b;
        }
      }
      return true;
    }
    while (kt >= kt_end) {
      // zig-zag over units ordered from the heaviest (latest queries) down
      int64_t p = r * G + ((r & 1) ? (G - 1 - c) : c);
      ++r;
      if (p >= total) return false;
      int64_t u = total - 1 - p;
      qb = (int)(u / B);
      b = (int)(u % B);
      kt = 0;
      kt_end = tiles_visible(args, qb);
    }
    ob = b;
    oqb = qb;
    okt = kt++;
    return true;
  }
};

// The MMAs of one key tile: K steps of 32 bytes (16 bf16 or 32 e4m3), four
// per 128-byte swizzled chunk.  A descriptor is advanced by adding the byte
// offset / 16 to its start-address field, so the unrolled loop spends a couple
// of integer adds per MMA: the single issuing thread would otherwise take
// longer to build descriptors than the tensor core takes for an N = 64 MMA.
template <int KSTEPS, bool kFP8>
__device__ __forceinline__ void issue_tile(uint32_t d, uint64_t ad, uint64_t bd, uint32_t b_chunk16,
                                           uint32_t id) {
#pragma unroll
  for (int kk = 0; kk < KSTEPS; ++kk) {
    const uint64_t a_k = ad + (uint64_t)((kk >> 2) * ((kTileKeys * 128) >> 4) + (kk & 3) * 2);
    const uint64_t b_k = bd + (uint64_t)((kk >> 2) * b_chunk16 + (kk & 3) * 2);
    if (kFP8) tc::mma_e4m3(d, a_k, b_k, id, kk > 0 ? 1u : 0u);
    else tc::mma_bf16(d, a_k, b_k, id, kk > 0 ? 1u : 0u);
  }
}

// Four E2M1 codes (the low four bits of each nibble of `nib4`, channel order
// from the lowest nibble) -> four E4M3 codes, one per byte.  A byte permute
// looks up the magnitude (0, 0.5, 1, 1.5 | 2, 3, 4, 6 as E4M3 bytes); the
// sign bit moves to bit 7.
__device__ __forceinline__ uint32_t e2m1x4_to_e4m3x4(uint32_t nib4) {
  const uint32_t mag = __byte_perm(0x3C383000u, 0x4C484440u, nib4 & 0x7777u);
  const uint32_t sgn = ((nib4 & 0x8u) << 4) | ((nib4 & 0x80u) << 8) | ((nib4 & 0x800u) << 12) |
                       ((nib4 & 0x8000u) << 16);
  return mag | sgn;
}

constexpr int kConvWarps = 2;  // FP4 keys: warps converting staged codes to E4M3

template <bool kFP8, int kEpiWG, bool kFP4>
__global__ void __launch_bounds__(64 + 128 * kEpiWG + (kFP4 ? 32 * kConvWarps : 0), 1)
    index_tc_kernel(const __grid_constant__ CUtensorMap tm_keys,
                    const __grid_constant__ CUtensorMap tm_q, const TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = sA + (size_t)a.stages * a.a_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + (size_t)a.nb * a.b_bytes);
  uint64_t* a_full = bars;
  uint64_t* a_empty = bars + a.stages;
  uint64_t* b_full = bars + 2 * a.stages;
  uint64_t* b_empty = b_full + 2;
  uint64_t* acc_full = b_empty + 2;
  uint64_t* acc_empty = acc_full + kMaxAcc;
  uint64_t* mma_done = acc_empty + kMaxAcc;
  uint64_t* stg_full = mma_done + 1;  // FP4 keys: [stages] staged tile of codes landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(stg_full + (kFP4 ? a.stages : 0));
  uint8_t* sS = sB + (size_t)a.nb * a.b_bytes;  // FP4 keys: staging, moved past the barriers below
  if (kFP4) {
    sS = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(tmem_slot + 4) + 1023) & ~(uintptr_t)1023);
  }
  // [epilogue warps][QPW * H_I], read as float4: 16-byte aligned
  float* a_w_smem = reinterpret_cast<float*>(
      (reinterpret_cast<uintptr_t>(kFP4 ? sS + (size_t)a.stages * a.stg_bytes
                                        : reinterpret_cast<uint8_t*>(tmem_slot + 4)) + 15) &
      ~(uintptr_t)15);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NM = a.NQ * a.H_I;  // MMA N
  int* err = &g_index_tc_error;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      // FP4 keys: a stage is full once every converter warp has written it
      tc::mbar_init(&a_full[s], kFP4 ? kConvWarps : 1);
      tc::mbar_init(&a_empty[s], 1);
      if (kFP4) tc::mbar_init(&stg_full[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&b_full[s], 1);
      tc::mbar_init(&b_empty[s], 1);
    }
    for (int s = 0; s < a.nacc; ++s) {
      tc::mbar_init(&acc_full[s], 1);
      tc::mbar_init(&acc_empty[s], a.alt ? 4 : 4 * kEpiWG);
    }
    tc::mbar_init(mma_done, 1);
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tm_keys);
    tc::prefetch_tmap(&tm_q);
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, a.tmem_cols);
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  Sched sch;
  sch.init(a, blockIdx.x, gridDim.x);
  int b, qb, kt;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      uint32_t it = 0, qcount = 0;
      int pb = -1, pqb = -1;
      while (sch.next(a, b, qb, kt)) {
        if (b != pb || qb != pqb) {
          const uint32_t bi = qcount % a.nb;
          if (!tc::mbar_wait(&b_empty[bi], ((qcount / a.nb) & 1) ^ 1, err, 1)) break;
          tc::mbar_expect_tx(&b_full[bi], a.b_bytes);
          const int y = (b * a.Q + qb * a.NQ) * a.H_I;
          for (int ch = 0; ch < a.n_chunks; ++ch)
            tc::tma_load_2d(sB + bi * a.b_bytes + ch * a.b_chunk_bytes, &tm_q, &b_full[bi],
                            ch * a.chunk_elems, y);
          ++qcount;
          pb = b;
          pqb = qb;
        }
        const uint32_t s = it % a.stages;
        if (!tc::mbar_wait(&a_empty[s], ((it / a.stages) & 1) ^ 1, err, 2)) break;
        const int y = (int)((int64_t)b * a.n_rows + (int64_t)kt * kTileKeys);
        if (kFP4) {
          // the stage's MMA is done, so the converters are done with its staging too
          tc::mbar_expect_tx(&stg_full[s], a.stg_bytes);
          tc::tma_load_2d(sS + (size_t)s * a.stg_bytes, &tm_keys, &stg_full[s], 0, y);
        } else {
          tc::mbar_expect_tx(&a_full[s], a.a_bytes);
          for (int ch = 0; ch < a.n_chunks; ++ch)
            tc::tma_load_2d(sA + s * a.a_bytes + ch * a.a_chunk_bytes, &tm_keys, &a_full[s],
                            ch * a.chunk_elems, y);
        }
        ++it;
      }
      // let the loads this CTA issued land before it can exit (only matters
      // when a wait above gave up; otherwise the MMA issuer consumed them all)
      for (uint32_t j = it > (uint32_t)a.stages ? it - a.stages : 0; j < it; ++j)
        tc::mbar_drain(kFP4 ? &stg_full[j % a.stages] : &a_full[j % a.stages], (j / a.stages) & 1);
      for (uint32_t j = qcount > (uint32_t)a.nb ? qcount - a.nb : 0; j < qcount; ++j)
        tc::mbar_drain(&b_full[j % a.nb], (j / a.nb) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t id = kFP8 ? tc::idesc(kTileKeys, NM, 0, 0) : tc::idesc(kTileKeys, NM, 1, 1);
      // descriptors of stage 0 / query buffer 0; the others are whole-buffer
      // offsets in the start-address field (shared memory stays below 256 KB)
      const uint64_t ad0 = tc::sdesc_sw128(tc::smem_u32(sA));
      const uint64_t bd0 = tc::sdesc_sw128(tc::smem_u32(sB));
      const uint32_t a_stage16 = a.a_bytes >> 4, b_buf16 = a.b_bytes >> 4;
      const uint32_t b_chunk16 = a.b_chunk_bytes >> 4;
      uint32_t s = 0, s_ph = 0;      // ring stage and the parity of its fill
      uint32_t acc = 0, acc_ph = 0;  // accumulator buffer and its parity
      bool a_ready = false, acc_ready = false;  // already seen by an early probe
      uint32_t qcount = 0, bi = 0;
      int pb = -1, pqb = -1;
      bool ok = true;
      // test aid: the producer's first loads are in flight while this waits
      if (a.stall && blockIdx.x == 0) ok = tc::flag_wait(&g_index_never_set, tc::kStallNs, err, 7);
      while (ok && sch.next(a, b, qb, kt)) {
        if (b != pb || qb != pqb) {
          if (qcount > 0) tc::mma_commit(&b_empty[(qcount - 1) % a.nb]);
          bi = qcount % a.nb;
          if (!tc::mbar_wait(&b_full[bi], (qcount / a.nb) & 1, err, 3)) { ok = false; break; }
          ++qcount;
          pb = b;
          pqb = qb;
        }
        if (!a_ready && !tc::mbar_wait(&a_full[s], s_ph, err, 4)) { ok = false; break; }
        if (!acc_ready && !tc::mbar_wait(&acc_empty[acc], acc_ph ^ 1, err, 5)) { ok = false; break; }
        // probe the next stage's fill and the next accumulator's release now
        // (non-blocking): each answer is needed only at the next tile, so the
        // latency of the probes overlaps this tile's MMA issue
        {
          const uint32_t ns = s + 1 == (uint32_t)a.stages ? 0 : s + 1;
          const uint32_t na = acc + 1 == (uint32_t)a.nacc ? 0 : acc + 1;
          a_ready = tc::mbar_test_wait(&a_full[ns], ns == 0 ? s_ph ^ 1 : s_ph);
          acc_ready = tc::mbar_test_wait(&acc_empty[na], (na == 0 ? acc_ph ^ 1 : acc_ph) ^ 1);
        }
        tc::tc_fence_after();
        const uint32_t d = tmem_base + acc * NM;
        const uint64_t ad = ad0 + s * a_stage16, bd = bd0 + bi * b_buf16;
        switch (a.ksteps) {
          case 4: issue_tile<4, kFP8>(d, ad, bd, b_chunk16, id); break;
          case 8: issue_tile<8, kFP8>(d, ad, bd, b_chunk16, id); break;
          case 12: issue_tile<12, kFP8>(d, ad, bd, b_chunk16, id); break;
          default: issue_tile<16, kFP8>(d, ad, bd, b_chunk16, id); break;
        }
        tc::mma_commit(&a_empty[s]);
        tc::mma_commit(&acc_full[acc]);
        if (++s == (uint32_t)a.stages) { s = 0; s_ph ^= 1; }
        if (++acc == (uint32_t)a.nacc) { acc = 0; acc_ph ^= 1; }
      }
      // every MMA issued must have completed before TMEM is released
      tc::mma_commit(mma_done);
      tc::mbar_drain(mma_done, 0);
    }
  } else if (kFP4 && warp >= 2 + 4 * kEpiWG) {
    // ------------------------------------------------------------ converters
    // Tile it: wait for its staged codes, write their E4M3 codes into the
    // stage (each 16 bytes of codes -- 32 channels of one row -- become two
    // 16-byte units of the row), make the writes visible to the tensor
    // cores, then one arrival per warp on the stage's barrier.
    const int ct = threadIdx.x - (64 + 128 * kEpiWG);
    const int upr = a.d_I / 32;  // 16-byte units of codes per row
    const int units = kTileKeys * upr;
    uint32_t it = 0;
    bool ok = true;
    while (ok && sch.next(a, b, qb, kt)) {
      const uint32_t s = it % a.stages;
      if (!tc::mbar_wait(&stg_full[s], (it / a.stages) & 1, err, 8)) { ok = false; break; }
      const uint8_t* src = sS + (size_t)s * a.stg_bytes;
      uint8_t* dst = sA + (size_t)s * a.a_bytes;
      for (int u = ct; u < units; u += 32 * kConvWarps) {
        const int r = u / upr, p = u - r * upr;
        const uint4 v = *reinterpret_cast<const uint4*>(src + (size_t)u * 16);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          o[2 * e] = e2m1x4_to_e4m3x4(w[e] & 0xffffu);
          o[2 * e + 1] = e2m1x4_to_e4m3x4(w[e] >> 16);
        }
        // channels 32p .. 32p+31: chunk p / 4 of the row, units 2 (p % 4) and +1
        uint8_t* crow = dst + (size_t)(p >> 2) * a.a_chunk_bytes + (size_t)r * 128;
        const int u0 = (p & 3) * 2;
        *reinterpret_cast<uint4*>(crow + (((u0) ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(crow + (((u0 + 1) ^ (r & 7)) << 4)) =
            make_uint4(o[4], o[5], o[6], o[7]);
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&a_full[s]);
      ++it;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int wg = ew >> 2;
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int row = quarter * 32 + lane;
    // queries per warpgroup and the first of them: the warpgroups split the
    // queries of every tile, or (alt) take alternate tiles with all queries
    const int QPW = a.alt ? a.NQ : a.NQ / kEpiWG;
    const int qoff = a.alt ? 0 : wg * QPW;
    // this warp's copy of the head weights of its QPW queries (per-warp, so
    // no barrier across warps is needed)
    float* sw = a_w_smem + (size_t)ew * QPW * a.H_I;
    uint32_t acc_it = 0;
    int cur_b = -1, cur_qb = -1;
    int64_t nv_q[4] = {0, 0, 0, 0};  // visible entries of this warpgroup's queries
    uint32_t tile_i = 0;
    while (sch.next(a, b, qb, kt)) {
      if (a.alt && (int)(tile_i++ & 1) != wg) {  // the other warpgroup's tile
        ++acc_it;
        continue;
      }
      const int64_t s = (int64_t)kt * kTileKeys + row;
      // the e4m3 key scale is fetched before the accumulator wait (its
      // latency would otherwise sit on the epilogue's critical path)
      float ks = 1.f;
      if (kFP8 && s < a.N) ks = __ldg(a.k_scale + (int64_t)b * a.n_rows + s);
      if (b != cur_b || qb != cur_qb) {
        // stage w (times the e4m3 query-row scale) once per query block
        __syncwarp();
        for (int e = lane; e < QPW * a.H_I; e += 32) {
          const int ql = e / a.H_I, j = e - ql * a.H_I;
          int i = qb * a.NQ + qoff + ql;
          if (i >= a.Q) i = a.Q - 1;
          const int64_t wi = ((int64_t)b * a.Q + i) * a.H_I + j;
          float wj = __ldg(a.w + wi);
          if (kFP8) wj *= __ldg(a.q_scale + wi);
          sw[e] = wj;
        }
        __syncwarp();
        for (int ql = 0; ql < QPW; ++ql) {
          const int i = qb * a.NQ + qoff + ql;
          const int64_t nv = i < a.Q ? n_vis(a.q_pos0 + i, a.m) : 0;
          nv_q[ql] = nv > a.N ? a.N : nv;
        }
        cur_b = b;
        cur_qb = qb;
      }
      const uint32_t acc = acc_it & (a.nacc - 1);
      // one lane waits, the warp follows converged (tcgen05.ld is .sync.aligned)
      int okw = lane == 0 ? (int)tc::mbar_wait(&acc_full[acc], (acc_it / a.nacc) & 1, err, 6) : 0;
      okw = __shfl_sync(0xffffffffu, okw, 0);
      __syncwarp();
      if (!okw) break;
      tc::tc_fence_after();
      float sc[4];
      for (int ql = 0; ql < QPW; ++ql) {
        const int qi = qoff + ql;
        const uint32_t col = acc * NM + qi * a.H_I;
        const float4* wq = reinterpret_cast<const float4*>(sw + ql * a.H_I);
        float part[4] = {0.f, 0.f, 0.f, 0.f};
        for (int j0 = 0; j0 < a.H_I; j0 += 64) {
          uint32_t r0[32], r1[32];
          const bool two = j0 + 32 < a.H_I;
          tc::tmem_ld32(tmem_base + ((uint32_t)(quarter * 32) << 16) + col + j0, r0);
          if (two) tc::tmem_ld32(tmem_base + ((uint32_t)(quarter * 32) << 16) + col + j0 + 32, r1);
          tc::tmem_wait_ld();
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const float4 w4 = wq[j0 / 4 + v];
            part[0] = fmaf(w4.x, fmaxf(__uint_as_float(r0[4 * v + 0]), 0.f), part[0]);
            part[1] = fmaf(w4.y, fmaxf(__uint_as_float(r0[4 * v + 1]), 0.f), part[1]);
            part[2] = fmaf(w4.z, fmaxf(__uint_as_float(r0[4 * v + 2]), 0.f), part[2]);
            part[3] = fmaf(w4.w, fmaxf(__uint_as_float(r0[4 * v + 3]), 0.f), part[3]);
          }
          if (two) {
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              const float4 w4 = wq[j0 / 4 + 8 + v];
              part[0] = fmaf(w4.x, fmaxf(__uint_as_float(r1[4 * v + 0]), 0.f), part[0]);
              part[1] = fmaf(w4.y, fmaxf(__uint_as_float(r1[4 * v + 1]), 0.f), part[1]);
              part[2] = fmaf(w4.z, fmaxf(__uint_as_float(r1[4 * v + 2]), 0.f), part[2]);
              part[3] = fmaf(w4.w, fmaxf(__uint_as_float(r1[4 * v + 3]), 0.f), part[3]);
            }
          }
        }
        sc[ql] = (part[0] + part[1]) + (part[2] + part[3]);
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&acc_empty[acc]);
      if (s < a.N) {
        for (int ql = 0; ql < QPW; ++ql) {
          const int i = qb * a.NQ + qoff + ql;
          if (i >= a.Q) break;
          const float v = s < nv_q[ql] ? sc[ql] * ks : -INFINITY;
          const int64_t o = ((int64_t)b * a.Q + i) * a.N + s;
          if (a.scores_bf16)
            reinterpret_cast<uint16_t*>(a.scores)[o] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
          else
            reinterpret_cast<float*>(a.scores)[o] = v;
        }
      }
      ++acc_it;
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base, a.tmem_cols);
  }
}

// -inf for entries beyond each query's visibility (the causal part of a
// prefill score matrix that the tensor-core kernel never touches).
__global__ void fill_invisible_kernel(void* __restrict__ scores, int bf16, int Q, int64_t N, int m,
                                      int64_t q_pos0) {
  const int64_t row = blockIdx.x;  // b * Q + i
  const int i = (int)(row % Q);
  const int64_t nv = n_vis(q_pos0 + i, m);
  for (int64_t s = nv + threadIdx.x; s < N; s += blockDim.x) {
    if (bf16) reinterpret_cast<uint16_t*>(scores)[row * N + s] = 0xFF80u;  // bf16 -inf
    else reinterpret_cast<float*>(scores)[row * N + s] = -INFINITY;
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

// 2-D map over a row-major [rows, cols] matrix of 1- or 2-byte elements with a
// box of 128 bytes x box_rows and the 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, bool fp8, int64_t rows, int cols, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  const int esz = fp8 ? 1 : 2;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * esz};
  cuuint32_t box[2] = {(cuuint32_t)(128 / esz), (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D map over the packed FP4 key codes, [rows, bytes] uint8: a box of the
// whole row (bytes <= 256, a multiple of 16) x box_rows, unswizzled.
bool make_map_fp4(CUtensorMap* map, const void* base, int64_t rows, int bytes, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)bytes, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)bytes};
  cuuint32_t box[2] = {(cuuint32_t)bytes, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int pow2_at_least(int x) {
  int p = 32;
  while (p < x) p <<= 1;
  return p;
}

}  // namespace

bool index_tc_supported(const csa_params& p, csa_dtype q_dtype, const csa_rows& keys, int Q) {
  (void)Q;
  const bool fp8 = keys.dtype == CSA_E4M3 || keys.dtype == CSA_E2M1;
  if (fp8 != (q_dtype == CSA_E4M3)) return false;
  if (!fp8 && !(keys.dtype == CSA_BF16 && q_dtype == CSA_BF16)) return false;
  if (fp8 && keys.nope != keys.width) return false;
  const int esz = fp8 ? 1 : 2;
  if ((p.d_I * esz) % 128 != 0 || p.d_I * esz > 512) return false;
  if (p.H_I % 32 != 0 || p.H_I > 256) return false;
  if ((int64_t)p.B * keys.n_rows >= (1ll << 31)) return false;
  return encode_fn() != nullptr;
}

cudaError_t index_tc_status(int* code, cudaStream_t st) {
  int h = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&h, g_index_tc_error, sizeof(int), 0,
                                            cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return e;
  *code = h;
  if (h != 0) {
    int zero = 0;
    e = cudaMemcpyToSymbol(g_index_tc_error, &zero, sizeof(int));
  }
  return e;
}

cudaError_t launch_index_tc(const csa_params& p, const void* q_idx, csa_dtype q_dtype,
                            const float* q_scale, const float* w, const csa_rows& keys,
                            int64_t q_pos0, int Q, int64_t N, void* scores, bool scores_bf16,
                            cudaStream_t st, bool fill_invisible) {
  const bool fp4 = keys.dtype == CSA_E2M1;         // staged, converted to E4M3
  const bool fp8 = keys.dtype == CSA_E4M3 || fp4;  // e4m3 MMA
  (void)q_dtype;
  TcArgs a{};
  a.B = p.B;
  a.Q = Q;
  a.H_I = p.H_I;
  a.d_I = p.d_I;
  a.m = p.m;
  a.N = N;
  a.n_rows = keys.n_rows;
  a.q_pos0 = q_pos0;
  a.NQ = (Q >= 4 && p.H_I <= 64) ? 256 / p.H_I : (Q >= 2 && p.H_I <= 128 ? 256 / p.H_I : 1);
  if (a.NQ > 4) a.NQ = 4;
  if (a.NQ > Q) a.NQ = 1;
  a.nQB = (Q + a.NQ - 1) / a.NQ;
  a.tps = (int)ceil_div(N, kTileKeys);
  const int NM = a.NQ * p.H_I;
  // Two epilogue warpgroups: they split the queries of an N = 256 tile, or
  // otherwise take alternate tiles (one warpgroup reducing a tile's heads is
  // latency-bound and could not keep up with the key stream)
  const int epi_wg = 2;
  a.alt = (NM == 256 && a.NQ >= 2) ? 0 : 1;
  const int esz = fp8 ? 1 : 2;
  a.chunk_elems = 128 / esz;
  a.n_chunks = p.d_I * esz / 128;
  a.ksteps = p.d_I * esz / 32;
  a.a_chunk_bytes = kTileKeys * 128;
  a.b_chunk_bytes = NM * 128;
  a.a_bytes = a.a_chunk_bytes * a.n_chunks;
  a.b_bytes = a.b_chunk_bytes * a.n_chunks;
  // The key stream is latency-bound (a key tile takes ~4 us from TMA issue to
  // arrival under full load), so the ring takes all the shared memory that is
  // left: 227 KB less the alignment pad, the barriers, the staged head
  // weights and the query buffers (two when that still leaves 4 key stages).
  const size_t wbytes =
      (size_t)4 * epi_wg * (a.alt ? a.NQ : a.NQ / epi_wg) * p.H_I * sizeof(float);
  a.stg_bytes = fp4 ? (uint32_t)(kTileKeys * p.d_I / 2) : 0u;
  const size_t fixed = 1024 + (5 + 2 * kMaxAcc) * sizeof(uint64_t) + 16 + 16 + wbytes +
                       (fp4 ? 1024 : 0);
  const size_t per_stage = a.a_bytes + 2 * sizeof(uint64_t) +
                           (fp4 ? a.stg_bytes + sizeof(uint64_t) : 0);
  const size_t limit = 227 * 1024;
  auto stages_for = [&](int nb) {
    const size_t used = fixed + (size_t)nb * a.b_bytes;
    return used >= limit ? 0 : (int)((limit - used) / per_stage);
  };
  a.nb = stages_for(2) >= 4 ? 2 : 1;
  int stages = stages_for(a.nb);
  // about 128 KB of key tiles in flight per SM keeps HBM busiest with 32 KB
  // bf16 tiles (more only queues up); the 16 KB e4m3 tiles take 192 KB
  const int cap = (int)(((fp8 ? 192 : 128) * 1024) / a.a_bytes);
  if (stages > (cap > 4 ? cap : 4)) stages = cap > 4 ? cap : 4;
  if (stages < 2) return cudaErrorNotSupported;
  a.stages = stages;
  // as many accumulator buffers as TMEM holds (at least two): the MMA of a
  // key tile then never waits for the epilogue of an earlier one, so each
  // ring stage is released as soon as its MMA has read it
  a.nacc = 2;
  while (a.nacc < kMaxAcc && 2 * a.nacc * NM <= 512) a.nacc *= 2;
  a.tmem_cols = (uint32_t)pow2_at_least(a.nacc * NM);
  if (a.tmem_cols > 512) return cudaErrorNotSupported;
  const bool all_visible = n_vis(q_pos0, p.m) >= N;
  a.mode = all_visible ? 0 : 1;
  a.total = all_visible ? (int64_t)p.B * a.nQB * a.tps : (int64_t)p.B * a.nQB;
  a.w = w;
  a.q_scale = q_scale;
  a.k_scale = keys.scale;
  a.scores = scores;
  a.scores_bf16 = scores_bf16 ? 1 : 0;
  a.stall = take_debug_stall(kStallIndex) ? 1 : 0;

  CUtensorMap tm_keys, tm_q;
  if (fp4) {
    if (!make_map_fp4(&tm_keys, keys.data, (int64_t)p.B * keys.n_rows, p.d_I / 2, kTileKeys))
      return cudaErrorInvalidValue;
  } else if (!make_map(&tm_keys, keys.data, fp8, (int64_t)p.B * keys.n_rows, p.d_I, kTileKeys)) {
    return cudaErrorInvalidValue;
  }
  if (!make_map(&tm_q, q_idx, fp8, (int64_t)p.B * Q * p.H_I, p.d_I, NM)) return cudaErrorInvalidValue;

  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t grid = sms;
  if (a.total < grid) grid = a.total;
  if (grid < 1) grid = 1;
  const size_t smem = 1024 + (size_t)a.stages * a.a_bytes + (size_t)a.nb * a.b_bytes +
                      (2 * a.stages + 5 + 2 * kMaxAcc + (fp4 ? a.stages : 0)) * sizeof(uint64_t) +
                      16 + 16 + wbytes + (fp4 ? 1024 + (size_t)a.stages * a.stg_bytes : 0);
  const int threads = 64 + 128 * epi_wg + (fp4 ? 32 * kConvWarps : 0);
  cudaError_t e;
#define CSA_LAUNCH_TC(FP8, EW, FP4)                                                             \
  do {                                                                                          \
    e = cudaFuncSetAttribute(index_tc_kernel<FP8, EW, FP4>,                                     \
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);           \
    if (e != cudaSuccess) return e;                                                             \
    index_tc_kernel<FP8, EW, FP4><<<(unsigned)grid, threads, smem, st>>>(tm_keys, tm_q, a);     \
  } while (0)
  if (fp4) {
    CSA_LAUNCH_TC(true, 2, true);
  } else if (fp8) {
    if (epi_wg == 2) CSA_LAUNCH_TC(true, 2, false); else CSA_LAUNCH_TC(true, 1, false);
  } else {
    if (epi_wg == 2) CSA_LAUNCH_TC(false, 2, false); else CSA_LAUNCH_TC(false, 1, false);
  }
#undef CSA_LAUNCH_TC
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (fill_invisible && !all_visible) {
    fill_invisible_kernel<<<(unsigned)((int64_t)p.B * Q), 256, 0, st>>>(scores, scores_bf16 ? 1 : 0,
                                                                        Q, N, p.m, q_pos0);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace csa
