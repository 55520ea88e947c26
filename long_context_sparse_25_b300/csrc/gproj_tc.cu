// Grouped output projection after the shared-KV attention, on the tensor
// cores (tcgen05 MMA, TMEM accumulators, TMA-fed shared-memory ring).
//
//   y[t, g*d_g + n] = sum_{j < K} o[t, g*K + j] * w[g, n, j],   K = (H/G) * D_v
//
// Source: "一文搞懂 DeepSeek：从 V3 的 KV 压缩与 MoE，到 V4 的百万 token 上下文",
// section "V4 改进一：CSA 与 HCA" (the CSA paragraph's last sentence: the
// attention output is projected in groups to save compute).  Group g takes
// heads g*H/G .. (g+1)*H/G - 1 of o [T, H, D_v], whose outputs sit next to
// each other in o's row (K contiguous elements from column g*K), and projects
// them with its own matrix, stored transposed as w [G, d_g, K] so that both
// operands are K-major.
//
// Tiles: 128 tokens x 256 features per tile (one M = 128, N = 256 MMA per
// 16-element K step), 64-element K blocks (one 128-byte swizzle atom) per ring
// stage: 16 KB of o and 32 KB of w, loaded by two TMA boxes.  When those tiles
// would leave most SMs idle (a decode step: one block of tokens), the tiles
// are 128 x 64 with eight 24 KB stages, so the weight stream spreads over
// every SM.  Persistent CTAs
// (one per SM) take tiles in (group, token block, feature block) order with
// the feature block fastest, so the CTAs working at the same time share each
// token block's rows of o in L2, and a group's 16 MB of weights stay in L2
// while every token block passes.
//
// Roles: warp 0 TMA producer (one thread), warp 1 TMEM allocator and MMA
// issuer (one thread; descriptors advanced by constant offsets), warps 2-5
// epilogue (tcgen05.ld of the accumulator, bf16 / fp32 conversion, stores).
// Two accumulators (of 256 or 64 columns) in TMEM, so the MMAs of a tile run
// while the epilogue drains the previous one.  Every mbarrier wait
// is bounded; a timeout is recorded in a device error word (read by
// csa_device_status) and the kernel returns after its copies and MMAs in
// flight have landed.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace csa {

namespace {

__device__ int g_gproj_error = 0;

constexpr int kBM = 128;                       // tokens per tile
constexpr int kBK = 64;                        // K elements per stage (128 bytes)
constexpr uint32_t kABytes = kBM * 128;        // 16 KB
constexpr int kThreads = 192;

// Features per tile: 256 (a prefill: many token blocks) or 64 (a decode step:
// one token block, so narrow tiles spread the weight stream over every SM),
// with the stage count that keeps about 192 KB of operands in flight.
template <int BN>
struct Tile {
  static constexpr int kBN = BN;
  static constexpr uint32_t kBBytes = BN * 128;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = BN == 256 ? 4 : 8;
};

struct GpArgs {
  int64_t T;
  int G, d_g, K, nkb;   // nkb = K / 64
  int n_mb, n_nb;       // token blocks, feature blocks per group
  int64_t n_tiles;      // G * n_mb * n_nb
  int64_t y_ld;         // G * d_g
  int out_f32;
  void* y;
};

__device__ __forceinline__ void tile_coords(const GpArgs& a, int64_t tile, int& g, int& mb,
                                            int& nb) {
  nb = (int)(tile % a.n_nb);
  const int64_t r = tile / a.n_nb;
  mb = (int)(r % a.n_mb);
  g = (int)(r / a.n_mb);
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gproj_tc_kernel(const __grid_constant__ CUtensorMap tm_o,
                    const __grid_constant__ CUtensorMap tm_w, const GpArgs a) {
  constexpr int kBN = Tile<BN>::kBN;
  constexpr uint32_t kStageBytes = Tile<BN>::kStageBytes;
  constexpr int kStages = Tile<BN>::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)kStages * kStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* acc_full = bars + 2 * kStages;  // [2]
  uint64_t* acc_empty = acc_full + 2;       // [2]
  uint64_t* mma_done = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* err = &g_gproj_error;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&acc_full[s], 1);
      tc::mbar_init(&acc_empty[s], 4);  // one arrival per epilogue warp
    }
    tc::mbar_init(mma_done, 1);
    tc::fence_mbar_init();
    tc::prefetch_tmap(&tm_o);
    tc::prefetch_tmap(&tm_w);
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, 2 * kBN < 32 ? 32 : 2 * kBN);
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      uint32_t it = 0;
      bool ok = true;
      for (int64_t tile = blockIdx.x; tile < a.n_tiles && ok; tile += gridDim.x) {
        int g, mb, nb;
        tile_coords(a, tile, g, mb, nb);
        const int ya = mb * kBM, yw = g * a.d_g + nb * kBN;
        for (int kb = 0; kb < a.nkb; ++kb, ++it) {
          const uint32_t s = it % kStages;
          if (!tc::mbar_wait(&empty[s], ((it / kStages) & 1) ^ 1, err, 41)) { ok = false; break; }
          uint8_t* st = smem + (size_t)s * kStageBytes;
          tc::mbar_expect_tx(&full[s], kStageBytes);
          tc::tma_load_2d(st, &tm_o, &full[s], g * a.K + kb * kBK, ya);
          tc::tma_load_2d(st + kABytes, &tm_w, &full[s], kb * kBK, yw);
        }
      }
      // the loads this CTA issued land before it can exit (matters only when
      // a wait gave up; otherwise the MMA issuer consumed them all)
      for (uint32_t j = it > (uint32_t)kStages ? it - kStages : 0; j < it; ++j)
        tc::mbar_drain(&full[j % kStages], (j / kStages) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t id = tc::idesc(kBM, kBN, 1, 1);
      const uint64_t ad0 = tc::sdesc_sw128(tc::smem_u32(smem));
      const uint64_t bd0 = tc::sdesc_sw128(tc::smem_u32(smem + kABytes));
      constexpr uint32_t kStage16 = kStageBytes >> 4;
      uint32_t it = 0, j = 0;
      bool ok = true;
      for (int64_t tile = blockIdx.x; tile < a.n_tiles && ok; tile += gridDim.x, ++j) {
        const uint32_t acc = j & 1;
        if (!tc::mbar_wait(&acc_empty[acc], ((j >> 1) & 1) ^ 1, err, 42)) { ok = false; break; }
        tc::tc_fence_after();
        const uint32_t d = tmem_base + acc * kBN;
        for (int kb = 0; kb < a.nkb; ++kb, ++it) {
          const uint32_t s = it % kStages;
          if (!tc::mbar_wait(&full[s], (it / kStages) & 1, err, 43)) { ok = false; break; }
          tc::tc_fence_after();
          const uint64_t ad = ad0 + s * kStage16, bd = bd0 + s * kStage16;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)  // 32 bytes per K step
            tc::mma_bf16(d, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), id,
                         (kb > 0 || kk > 0) ? 1u : 0u);
          tc::mma_commit(&empty[s]);
        }
        if (!ok) break;
        tc::mma_commit(&acc_full[acc]);
      }
      // every MMA issued must have completed before TMEM is released
      tc::mma_commit(mma_done);
      tc::mbar_drain(mma_done, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // the TMEM lanes this warp may access
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    uint32_t j = 0;
    for (int64_t tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x, ++j) {
      int g, mb, nb;
      tile_coords(a, tile, g, mb, nb);
      const uint32_t acc = j & 1;
      int okw = lane == 0 ? (int)tc::mbar_wait(&acc_full[acc], (j >> 1) & 1, err, 44) : 0;
      okw = __shfl_sync(0xffffffffu, okw, 0);
      __syncwarp();
      if (!okw) break;
      tc::tc_fence_after();
      const int64_t row = (int64_t)mb * kBM + quarter * 32 + lane;
      const int64_t col0 = (int64_t)g * a.d_g + (int64_t)nb * kBN;
#pragma unroll 1
      for (int c = 0; c < kBN; c += 32) {
        uint32_t r[32];
        tc::tmem_ld32(tmem_base + lane_base + acc * kBN + c, r);
        tc::tmem_wait_ld();
        if (row < a.T) {
          if (a.out_f32) {
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<float*>(a.y) + row * a.y_ld +
                                                  col0 + c);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[v] = make_uint4(r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
          } else {
            uint32_t pk[16];
#pragma unroll
            for (int v = 0; v < 16; ++v) {
              const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r[2 * v])));
              const uint32_t hi =
                  __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r[2 * v + 1])));
              pk[v] = lo | (hi << 16);
            }
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.y) + row * a.y_ld +
                                                  col0 + c);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&acc_empty[acc]);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base, 2 * kBN < 32 ? 32 : 2 * kBN);
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

// 2-D map over a row-major [rows, cols] bf16 matrix with row stride ld
// elements: box of 64 columns (128 bytes) x box_rows, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld,
              int box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      n = 148;
  }
  return n;
}

}  // namespace

cudaError_t gproj_status(int* code, cudaStream_t st) {
  int h = 0;
  cudaError_t e =
      cudaMemcpyFromSymbolAsync(&h, g_gproj_error, sizeof(int), 0, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return e;
  *code = h;
  if (h != 0) {
    int zero = 0;
    e = cudaMemcpyToSymbol(g_gproj_error, &zero, sizeof(int));
  }
  return e;
}

cudaError_t launch_group_proj(const void* o, int64_t T, int H, int D_v, const void* w, int G,
                              int d_g, void* y, bool y_f32, cudaStream_t st) {
  GpArgs a{};
  a.T = T;
  a.G = G;
  a.d_g = d_g;
  a.K = (H / G) * D_v;
  a.nkb = a.K / kBK;
  a.n_mb = (int)((T + kBM - 1) / kBM);
  // narrow tiles when the wide ones would leave most SMs idle
  const int64_t wide_tiles = (int64_t)G * a.n_mb * (d_g / 256);
  const bool narrow = wide_tiles < num_sms() / 2;
  const int BN = narrow ? 64 : 256;
  a.n_nb = d_g / BN;
  a.n_tiles = (int64_t)G * a.n_mb * a.n_nb;
  a.y_ld = (int64_t)G * d_g;
  a.out_f32 = y_f32 ? 1 : 0;
  a.y = y;
  if (a.n_tiles == 0) return cudaSuccess;
  CUtensorMap tm_o, tm_w;
  if (!make_map(&tm_o, o, T, (int64_t)H * D_v, (int64_t)H * D_v, kBM)) return cudaErrorInvalidValue;
  if (!make_map(&tm_w, w, (int64_t)G * d_g, a.K, a.K, BN)) return cudaErrorInvalidValue;
  int64_t grid = num_sms();
  if (a.n_tiles < grid) grid = a.n_tiles;
  auto launch = [&](auto tile) -> cudaError_t {
    using T = decltype(tile);
    const size_t smem =
        1024 + (size_t)T::kStages * T::kStageBytes + (2 * T::kStages + 5) * sizeof(uint64_t) + 16;
    cudaError_t e = cudaFuncSetAttribute(gproj_tc_kernel<T::kBN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    gproj_tc_kernel<T::kBN><<<(unsigned)grid, kThreads, smem, st>>>(tm_o, tm_w, a);
    return cudaGetLastError();
  };
  return narrow ? launch(Tile<64>{}) : launch(Tile<256>{});
}

}  // namespace csa
