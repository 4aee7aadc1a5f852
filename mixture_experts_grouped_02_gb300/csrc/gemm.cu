// gemm.cu -- the two grouped GEMMs of the MoE expert FFN on sm_103a.
//
// One persistent, warp-specialised kernel template serves both:
//
//  * gate/up (GEMM1): A = 128 token rows gathered by index from x by four
//    producer warps (16-byte cp.async per lane, eight lanes per 128-byte row,
//    written straight into the 128-byte swizzled layout, then a proxy fence
//    and an mbarrier arrive once the copies of two later stages are issued), B = 128 gate rows and the 128 matching up rows of w13[e]
//    stacked into one 256-row operand, so a single M=128 x N=256 MMA puts
//    gate in accumulator columns 0..127 and up in 128..255 of the same TMEM
//    lane.  The epilogue forms SiLU(gate) * up per lane and stores h.
//    Sources: "MOE Bmm1 Fused Gather", load_activations (gathered token
//    rows, padded rows masked), mma_partition and epilogue_partition
//    (activation in the GEMM epilogue); "factor_moe_fused_gemm.cu",
//    fused_silu_gate_kernel (gate = first half of w13's rows).
//  * down (GEMM2): A = 128 consecutive rows of h (a plain TMA tile, since
//    the sorted rows are contiguous), B = 256 rows of w2[e]; the epilogue
//    multiplies by the routing weight and stores fp32 y.  Source: "moe
//    triton kernel use tma", review comment on TOKEN_INPUT_USE_TMA /
//    MUL_ROUTED_WEIGHT.
//
// Roles: the first P warps load (P = 4 for gate/up: the gather plus the TMA of
// the weight tiles; P = 1 for down: TMA only), warp P issues tcgen05.mma from
// one thread and owns the TMEM allocation, warps P+1 .. P+4 run the epilogue
// (warp w reads TMEM lanes 32*(w%4) .. +31).  A 4-stage shared-memory ring of
// 48 KB stages (16 KB A + 32 KB B, 128-byte swizzled K-major rows) is handed
// over with full/empty mbarriers; two 256-column fp32 accumulators in TMEM
// let the epilogue of one tile overlap the MMAs of the next.  Tiles are
// walked in bands of N tiles so that the CTAs resident at one time share
// weight tiles and token tiles in L2 (the banded raster of the Gluon
// example's banded_row_major).
//
// Every wait is bounded (kWaitTimeoutNs): on expiry the kernel records
// MOE_ERR_TIMEOUT, lets its copies and MMAs in flight drain (again bounded),
// frees TMEM and returns.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "sched.cuh"

namespace moe {
namespace {

enum Kind { kGateUp = 0, kDown = 1 };

template <typename T>
struct Elem;
template <>
struct Elem<__nv_bfloat16> {
  static constexpr uint32_t kFmt = 1;  // bf16 in kind::f16
};
template <>
struct Elem<float> {
  static constexpr uint32_t kFmt = 2;  // tf32 in kind::tf32
};

template <int KIND, typename T>
struct Cfg {
  static constexpr int kBM = kBlockM;                     // tokens per tile (MMA M)
  static constexpr int kBN = 256;                         // MMA N
  static constexpr int kRowBytes = 128;                   // one swizzle atom row
  static constexpr int kBK = kRowBytes / sizeof(T);       // elements per k-tile
  static constexpr int kUmmaK = 32 / sizeof(T);           // K of one MMA (32 bytes)
  static constexpr int kStages = 4;
  static constexpr int kABytes = kBM * kRowBytes;         // 16 KB
  static constexpr int kBBytes = kBN * kRowBytes;         // 32 KB
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kAccCols = kBN;                    // fp32 columns per accumulator
  static constexpr int kTmemCols = 2 * kAccCols;          // two accumulators
  static constexpr uint32_t kIdesc = make_idesc(Elem<T>::kFmt, kBM, kBN);
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024;
  static constexpr int kProducerWarps = KIND == kGateUp ? 4 : 1;
  static constexpr int kMmaWarp = kProducerWarps;
  static constexpr int kThreads = (kProducerWarps + 1 + 4) * 32;
  // gate/up: each producer thread marks a stage full only once its cp.async
  // group for that stage has landed, kGatherLag stages after issuing it.  The
  // lag leaves one stage of slack: stage n is published while the tensor core
  // still works on n - 1 (a lag of kStages - 1 would publish n only after n - 1
  // is freed and the next copies are issued, idling the tensor core each stage)
  static constexpr int kGatherLag = kStages - 2;
  static constexpr uint32_t kFullArrivals = KIND == kGateUp ? kProducerWarps * 32 + 1 : 1;
  static constexpr uint32_t kTxBytes = KIND == kGateUp ? kBBytes : kStageBytes;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  return g / (1.0f + __expf(-g)) * u;
}

template <int KIND, typename T>
__global__ void __launch_bounds__(Cfg<KIND, T>::kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ GemmArgs a, const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB) {
  using C = Cfg<KIND, T>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[C::kStages];
  __shared__ __align__(8) uint64_t empty_bar[C::kStages];
  __shared__ __align__(8) uint64_t accf_bar[2];
  __shared__ __align__(8) uint64_t acce_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_skip;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t smemA = smem_base;
  const uint32_t smemB = smem_base + C::kStages * C::kABytes;

  if (threadIdx.x == 0) {
    s_skip = (a.status != nullptr && *reinterpret_cast<volatile int32_t*>(a.status) != 0);
    s_abort = 0;
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(smem_u32(&full_bar[i]), C::kFullArrivals);
      mbar_init(smem_u32(&empty_bar[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&accf_bar[i]), 1);
      mbar_init(smem_u32(&acce_bar[i]), 128);
    }
    mbar_init(smem_u32(&drain_bar), 1);
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  __syncthreads();
  if (s_skip) return;
  if (warp == C::kMmaWarp) tmem_alloc(smem_u32(&s_tmem_base), C::kTmemCols);
  if (warp == 0 && lane == 0) {
    if constexpr (KIND == kDown) tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = s_tmem_base;

  const int num_blocks = *a.num_blocks;
  const int total = num_blocks * a.n_tiles * a.splits;
  const uint64_t to = a.timeout_ns;

  if (warp < C::kProducerWarps) {
    if constexpr (KIND == kGateUp) {
      // -------------------------------------------------- gather producer
      // thread pt copies 16-byte chunk (pt % 8) of rows pt/8 + 16 j, j < 8,
      // into the swizzled A tile: chunk c of row r sits at chunk c ^ (r % 8)
      const int pt = threadIdx.x;
      const int chunk = pt & 7;
      const int row0 = pt >> 3;
      constexpr int kElemsPerChunk = 16 / sizeof(T);
      const T* x = static_cast<const T*>(a.x);
      uint32_t stage = 0, phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const Tile t = decode_tile(tile, num_blocks, a);
        const int4 bi = reinterpret_cast<const int4*>(a.block_info)[t.mb];
        const int e = bi.x, r0 = bi.z, valid = bi.w;
        int kb, ke;
        split_range(a, t.split, kb, ke);
        const T* src[8];
        uint32_t dst_off[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int r = row0 + 16 * j;
          // padding slots read token 0; their products are never stored
          const int tok = r < valid ? a.sorted_ids[r0 + r] / a.K : 0;
          src[j] = x + static_cast<long long>(tok) * a.H + chunk * kElemsPerChunk;
          dst_off[j] = r * C::kRowBytes + ((chunk ^ (r & 7)) << 4);
        }
        for (int kt = kb; kt < ke; ++kt) {
          if (!mbar_wait_bounded(smem_u32(&empty_bar[stage]), phase ^ 1, &s_abort, to)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&full_bar[stage]);
          if (pt == 0) {
            mbar_arrive_expect_tx(fb, C::kTxBytes);
            const uint32_t b_dst = smemB + stage * C::kBBytes;
            const int grow = e * 2 * a.I + t.nt * 128;
            tma_load_2d(b_dst, &tmB, fb, kt * C::kBK, grow);
            tma_load_2d(b_dst + 128 * C::kRowBytes, &tmB, fb, kt * C::kBK, grow + a.I);
          }
          const uint32_t a_dst = smemA + stage * C::kABytes;
#pragma unroll
          for (int j = 0; j < 8; ++j) cp_async_16(a_dst + dst_off[j], src[j] + kt * C::kBK);
          cp_async_commit();
          ++issued;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
          if (issued > C::kGatherLag) {
            // the group issued kGatherLag stages ago has landed: publish it to
            // the tensor core (async proxy) and mark it full
            cp_async_wait<C::kGatherLag>();
            fence_proxy_async_smem();
            const long long n = issued - 1 - C::kGatherLag;
            mbar_arrive(smem_u32(&full_bar[n % C::kStages]));
          }
        }
      }
      cp_async_wait<0>();
      fence_proxy_async_smem();
      for (long long n = issued > C::kGatherLag ? issued - C::kGatherLag : 0; n < issued; ++n)
        mbar_arrive(smem_u32(&full_bar[n % C::kStages]));
      if (!ok && pt == 0) {
        // let the weight copies already issued land before the CTA exits
        const long long first = issued > C::kStages ? issued - C::kStages : 0;
        for (long long n = first; n < issued; ++n)
          drain_wait(smem_u32(&full_bar[n % C::kStages]),
                     static_cast<uint32_t>((n / C::kStages) & 1), to / 4);
      }
    } else {
    // ---------------------------------------------------------- TMA producer
    uint32_t stage = 0, phase = 0;
    long long issued = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const Tile t = decode_tile(tile, num_blocks, a);
      const int4 bi = reinterpret_cast<const int4*>(a.block_info)[t.mb];
      const int e = bi.x, r0 = bi.z;
      int kb, ke;
      split_range(a, t.split, kb, ke);
      for (int kt = kb; kt < ke; ++kt) {
        int good = 1;
        if (lane == 0) good = mbar_wait_bounded(smem_u32(&empty_bar[stage]), phase ^ 1, &s_abort, to);
        good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t fb = smem_u32(&full_bar[stage]);
          mbar_arrive_expect_tx(fb, C::kTxBytes);
          tma_load_2d(smemA + stage * C::kABytes, &tmA, fb, kt * C::kBK, r0);
          tma_load_2d(smemB + stage * C::kBBytes, &tmB, fb, kt * C::kBK, e * a.H + t.nt * C::kBN);
        }
        ++issued;
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (!ok && lane == 0) {
      // let the copies already issued land before the CTA's memory goes away
      const long long first = issued > C::kStages ? issued - C::kStages : 0;
      for (long long n = first; n < issued; ++n)
        drain_wait(smem_u32(&full_bar[n % C::kStages]),
                   static_cast<uint32_t>((n / C::kStages) & 1), to / 4);
    }
    }
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const Tile t = decode_tile(tile, num_blocks, a);
        int kb, ke;
        split_range(a, t.split, kb, ke);
        if (!mbar_wait_bounded(smem_u32(&acce_bar[acc]), acc_phase ^ 1, &s_abort, to)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * C::kAccCols;
        for (int kt = kb; kt < ke; ++kt) {
          if (!mbar_wait_bounded(smem_u32(&full_bar[stage]), phase, &s_abort, to)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a_base = smemA + stage * C::kABytes;
          const uint32_t b_base = smemB + stage * C::kBBytes;
#pragma unroll
          for (int k = 0; k < C::kBK / C::kUmmaK; ++k) {
            const uint64_t ad = sw128_kmajor_desc(a_base + k * 32);
            const uint64_t bd = sw128_kmajor_desc(b_base + k * 32);
            const uint32_t accum = (kt > kb || k > 0) ? 1u : 0u;
            if constexpr (Elem<T>::kFmt == 1)
              umma_bf16(d_tmem, ad, bd, C::kIdesc, accum);
            else
              umma_tf32(d_tmem, ad, bd, C::kIdesc, accum);
          }
          umma_commit(smem_u32(&empty_bar[stage]));
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(&accf_bar[acc]));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (!ok) {
        // wait for the MMAs already issued before TMEM is released
        umma_commit(smem_u32(&drain_bar));
        drain_wait(smem_u32(&drain_bar), 0, to / 4);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;          // TMEM lane quarter this warp may read
    const int r = q * 32 + lane;     // row of the tile = TMEM lane
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const Tile t = decode_tile(tile, num_blocks, a);
      const int4 bi = reinterpret_cast<const int4*>(a.block_info)[t.mb];
      const int r0 = bi.z, valid = bi.w;
      const bool row_ok = r < valid;
      float wrow = 0.0f;
      if constexpr (KIND == kDown) {
        if (row_ok) wrow = a.topk_weights[a.sorted_ids[r0 + r]];
      }
      int good = 1;
      if (lane == 0) good = mbar_wait_bounded(smem_u32(&accf_bar[acc]), acc_phase, &s_abort, to);
      good = __shfl_sync(0xffffffffu, good, 0);
      if (!good) break;
      tc_fence_after_sync();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * C::kAccCols;
      if constexpr (KIND == kGateUp) {
        T* h = reinterpret_cast<T*>(a.out) + static_cast<long long>(r0 + r) * a.I;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32(taddr + c * 32, g);
          tmem_ld32(taddr + 128 + c * 32, u);
          tmem_wait_ld();
          const int j0 = t.nt * 128 + c * 32;
          if (row_ok && j0 < a.I) {
            if constexpr (Elem<T>::kFmt == 1) {
              uint4* dst = reinterpret_cast<uint4*>(h + j0);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint4 pk;
                pk.x = pack_bf16x2(silu_mul(__uint_as_float(g[8 * v + 0]), __uint_as_float(u[8 * v + 0])),
                                   silu_mul(__uint_as_float(g[8 * v + 1]), __uint_as_float(u[8 * v + 1])));
                pk.y = pack_bf16x2(silu_mul(__uint_as_float(g[8 * v + 2]), __uint_as_float(u[8 * v + 2])),
                                   silu_mul(__uint_as_float(g[8 * v + 3]), __uint_as_float(u[8 * v + 3])));
                pk.z = pack_bf16x2(silu_mul(__uint_as_float(g[8 * v + 4]), __uint_as_float(u[8 * v + 4])),
                                   silu_mul(__uint_as_float(g[8 * v + 5]), __uint_as_float(u[8 * v + 5])));
                pk.w = pack_bf16x2(silu_mul(__uint_as_float(g[8 * v + 6]), __uint_as_float(u[8 * v + 6])),
                                   silu_mul(__uint_as_float(g[8 * v + 7]), __uint_as_float(u[8 * v + 7])));
                dst[v] = pk;
              }
            } else {
              float4* dst = reinterpret_cast<float4*>(h + j0);
#pragma unroll
              for (int v = 0; v < 8; ++v) {
                float4 o;
                o.x = silu_mul(__uint_as_float(g[4 * v + 0]), __uint_as_float(u[4 * v + 0]));
                o.y = silu_mul(__uint_as_float(g[4 * v + 1]), __uint_as_float(u[4 * v + 1]));
                o.z = silu_mul(__uint_as_float(g[4 * v + 2]), __uint_as_float(u[4 * v + 2]));
                o.w = silu_mul(__uint_as_float(g[4 * v + 3]), __uint_as_float(u[4 * v + 3]));
                dst[v] = o;
              }
            }
          }
        }
      } else {
        float* y = reinterpret_cast<float*>(a.out) +
                   (static_cast<long long>(t.split) * a.cap + r0 + r) * a.H;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t v[32];
          tmem_ld32(taddr + c * 32, v);
          tmem_wait_ld();
          const int col0 = t.nt * C::kBN + c * 32;
          if (row_ok && col0 < a.H) {
            float4* dst = reinterpret_cast<float4*>(y + col0);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              float4 o;
              o.x = wrow * __uint_as_float(v[4 * i + 0]);
              o.y = wrow * __uint_as_float(v[4 * i + 1]);
              o.z = wrow * __uint_as_float(v[4 * i + 2]);
              o.w = wrow * __uint_as_float(v[4 * i + 3]);
              dst[i] = o;
            }
          }
        }
      }
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&acce_bar[acc]));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && s_abort) report_error(a.status, MOE_ERR_TIMEOUT);
  if (warp == C::kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

template <int KIND, typename T>
cudaError_t launch(const GemmArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmB, int grid,
                   cudaStream_t s) {
  using C = Cfg<KIND, T>;
  auto kern = grouped_gemm_kernel<KIND, T>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (err != cudaSuccess) return err;
  kern<<<grid, C::kThreads, C::kSmemBytes, s>>>(a, tmA, tmB);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_gate_up(int dtype, const GemmArgs& a, const CUtensorMap& tmA,
                                const CUtensorMap& tmB, int grid, cudaStream_t s) {
  if (dtype == MOE_BF16) return launch<kGateUp, __nv_bfloat16>(a, tmA, tmB, grid, s);
  return launch<kGateUp, float>(a, tmA, tmB, grid, s);
}

cudaError_t launch_gemm_down(int dtype, const GemmArgs& a, const CUtensorMap& tmA,
                             const CUtensorMap& tmB, int grid, cudaStream_t s) {
  if (dtype == MOE_BF16) return launch<kDown, __nv_bfloat16>(a, tmA, tmB, grid, s);
  return launch<kDown, float>(a, tmA, tmB, grid, s);
}

}  // namespace moe
