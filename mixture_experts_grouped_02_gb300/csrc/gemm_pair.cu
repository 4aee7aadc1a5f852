// gemm_pair.cu -- the two grouped GEMMs on CTA pairs (tcgen05 cta_group::2),
// for workloads with many tokens per expert.
//
// Same operation, operands and epilogues as gemm.cu (gate/up: gathered token
// rows x [gate; up] rows of w13[e], SiLU*up; down: contiguous h rows x w2[e],
// routing weight).  The difference is the tile: one 256-row align block per
// pair of CTAs in a cluster of two, M = 256 x N = 256 per MMA instruction.
// Each CTA holds 128 of the block's rows (A) and 128 of the 256 weight rows
// (B: the leader the gate rows, the follower the matching up rows; or the two
// halves of 256 w2 rows), so a CTA moves 32 KB per 64-wide K step for as many
// MMA FLOPs as a single-CTA 128 x 256 tile moves 48 KB for.  With 32 KB
// stages, six of them fit in shared memory.  This follows the pages'
// two-CTA mode of the "MOE Bmm1 Fused Gather" example (num_ctas = 2, the
// weight operand split across the pair), without TMA multicast: every CTA
// loads only its own halves.
//
// Protocol:
//  * A arrives in sorted order (gate/up: the token rows were written to their
//    sorted slots by the gather step; down: h), so one producer thread per CTA
//    loads its 128 A rows and its half of the weight rows by TMA; the leader
//    declares the bytes of both CTAs on its full barrier and the follower's
//    copies (cta_group::2) complete there directly -- no thread of the
//    follower has to signal the leader per stage.  (A gather by cp.async here
//    would need a cluster-scoped release per stage, and such a release waits
//    for every earlier memory operation of the releasing thread.)
//  * the leader's MMA thread issues tcgen05.mma.cta_group::2 (A and B read
//    from the same shared-memory addresses in both CTAs, D rows 0-127 into the
//    leader's TMEM, 128-255 into the follower's) and commits to the empty and
//    accumulator-full barriers of both CTAs at once (multicast commit);
//  * each CTA's epilogue reads its own 128 TMEM lanes exactly as gemm.cu; the
//    follower's epilogue threads arrive on a barrier of their own CTA and one
//    otherwise idle lane relays the release of each accumulator to the leader;
//  * both CTAs allocate TMEM as a pair, and meet at a cluster barrier before
//    releasing it.
// All waits are bounded (kWaitTimeoutNs) as in gemm.cu.
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
  static constexpr uint32_t kFmt = 1;
};
template <>
struct Elem<float> {
  static constexpr uint32_t kFmt = 2;
};

template <int KIND, typename T>
struct PairCfg {
  static constexpr int kRowsPerCta = 128;                // rows of the 256-row block
  static constexpr int kBN = 256;                        // MMA N for the pair
  static constexpr int kBHalf = kBN / 2;                 // weight rows per CTA
  static constexpr int kRowBytes = 128;
  static constexpr int kBK = kRowBytes / sizeof(T);
  static constexpr int kUmmaK = 32 / sizeof(T);
  static constexpr int kStages = 6;
  static constexpr int kABytes = kRowsPerCta * kRowBytes;  // 16 KB
  static constexpr int kBBytes = kBHalf * kRowBytes;       // 16 KB
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kAccCols = kBN;
  static constexpr int kTmemCols = 2 * kAccCols;
  static constexpr int kProducerWarps = 1;
  static constexpr int kMmaWarp = kProducerWarps;
  static constexpr int kThreads = (kProducerWarps + 1 + 4) * 32;
  // bytes both CTAs' copies deliver to the leader's full barrier per stage
  static constexpr uint32_t kTxBytes = 2 * kStageBytes;
  static constexpr uint32_t kIdesc = make_idesc(Elem<T>::kFmt, 256, kBN);
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  return g / (1.0f + __expf(-g)) * u;
}

// Give copies this CTA issued time to land before its shared memory goes
// away (used only when a wait has run out).
__device__ __forceinline__ void settle(uint64_t ns) {
  const uint64_t t0 = global_timer_ns();
  while (global_timer_ns() - t0 < ns) {
  }
}

template <int KIND, typename T>
__global__ void __launch_bounds__(PairCfg<KIND, T>::kThreads, 1)
    pair_gemm_kernel(const __grid_constant__ GemmArgs a, const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB) {
  using C = PairCfg<KIND, T>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[C::kStages];
  __shared__ __align__(8) uint64_t empty_bar[C::kStages];
  __shared__ __align__(8) uint64_t accf_bar[2];
  __shared__ __align__(8) uint64_t acce_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ __align__(8) uint64_t relay_acce[2];           // follower: epilogue done
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_skip;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();      // 0 = leader, 1 = follower
  const bool leader = rank == 0;
  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t smemA = smem_base;
  const uint32_t smemB = smem_base + C::kStages * C::kABytes;

  if (threadIdx.x == 0) {
    s_skip = (a.status != nullptr && *reinterpret_cast<volatile int32_t*>(a.status) != 0);
    s_abort = 0;
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(smem_u32(&full_bar[i]), 1);
      mbar_init(smem_u32(&empty_bar[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&accf_bar[i]), 1);
      mbar_init(smem_u32(&acce_bar[i]), 128 + 1);
      mbar_init(smem_u32(&relay_acce[i]), 128);
    }
    mbar_init(smem_u32(&drain_bar), 1);
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  cluster_sync();  // barriers of both CTAs initialised before any remote arrive
  // the pair allocates TMEM together, so both CTAs take the leader's decision
  __shared__ int s_skip_pair;
  if (threadIdx.x == 0)
    s_skip_pair = leader ? s_skip
                         : static_cast<int>(ld_shared_cluster_u32(mapa_shared(smem_u32(&s_skip), 0)));
  __syncthreads();
  const bool skip = s_skip_pair != 0;
  if (!skip && warp == C::kMmaWarp) tmem_alloc_pair(smem_u32(&s_tmem_base), C::kTmemCols);
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = s_tmem_base;

  const int num_blocks = skip ? 0 : *a.num_blocks;
  const int total = num_blocks * a.n_tiles * a.splits;
  const int cluster = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;
  const uint64_t to = a.timeout_ns;

  if (warp < C::kProducerWarps) {
    // ------------------------------------------------------------ producer
    const uint32_t full0 = mapa_shared(smem_u32(&full_bar[0]), 0);  // leader's barriers
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    for (int tile = cluster; tile < total && ok; tile += nclusters) {
      const Tile t = decode_tile(tile, num_blocks, a);
      const int4 bi = reinterpret_cast<const int4*>(a.block_info)[t.mb];
      const int e = bi.x;
      const int r0 = bi.z + static_cast<int>(rank) * C::kRowsPerCta;
      // this CTA's half of the weight rows: gate rows (leader) and the matching
      // up rows (follower), or the two halves of 256 w2 rows
      const int brow = KIND == kGateUp
                           ? e * 2 * a.I + static_cast<int>(rank) * a.I + t.nt * C::kBHalf
                           : e * a.H + t.nt * C::kBN + static_cast<int>(rank) * C::kBHalf;
      int kb, ke;
      split_range(a, t.split, kb, ke);
      for (int kt = kb; kt < ke; ++kt) {
        int good = 1;
        if (lane == 0)
          good = mbar_wait_bounded(smem_u32(&empty_bar[stage]), phase ^ 1, &s_abort, to);
        good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t fb = full0 + stage * 8u;
          if (leader) mbar_arrive_expect_tx(smem_u32(&full_bar[stage]), C::kTxBytes);
          tma_load_2d_pair(smemA + stage * C::kABytes, &tmA, fb, kt * C::kBK, r0);
          tma_load_2d_pair(smemB + stage * C::kBBytes, &tmB, fb, kt * C::kBK, brow);
        }
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (!ok) settle(to / 8);
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (leader && lane == 0) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = cluster; tile < total && ok; tile += nclusters) {
        const Tile t = decode_tile(tile, num_blocks, a);
        int kb, ke;
        split_range(a, t.split, kb, ke);
        if (!mbar_wait_bounded_cluster(smem_u32(&acce_bar[acc]), acc_phase ^ 1, &s_abort, to)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * C::kAccCols;
        for (int kt = kb; kt < ke; ++kt) {
          if (!mbar_wait_bounded_cluster(smem_u32(&full_bar[stage]), phase, &s_abort, to)) {
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
              umma_bf16_pair(d_tmem, ad, bd, C::kIdesc, accum);
            else
              umma_tf32_pair(d_tmem, ad, bd, C::kIdesc, accum);
          }
          umma_commit_pair(smem_u32(&empty_bar[stage]), 0x3);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit_pair(smem_u32(&accf_bar[acc]), 0x3);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (!ok) {
        umma_commit_pair(smem_u32(&drain_bar), 0x1);
        drain_wait(smem_u32(&drain_bar), 0, to / 4);
      }
    } else if (!leader && lane == 1) {
      // relay: each accumulator the follower's epilogue released -> leader
      const uint32_t acce0 = mapa_shared(smem_u32(&acce_bar[0]), 0);
      uint32_t acc = 0, acc_phase = 0;
      for (int tile = cluster; tile < total; tile += nclusters) {
        if (!mbar_wait_bounded(smem_u32(&relay_acce[acc]), acc_phase, &s_abort, to)) break;
        mbar_arrive_cluster(acce0 + acc * 8u);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int r = q * 32 + lane;
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = cluster; tile < total; tile += nclusters) {
      const Tile t = decode_tile(tile, num_blocks, a);
      const int4 bi = reinterpret_cast<const int4*>(a.block_info)[t.mb];
      const int r0 = bi.z + static_cast<int>(rank) * C::kRowsPerCta;
      const int valid = bi.w - static_cast<int>(rank) * C::kRowsPerCta;
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
      mbar_arrive(leader ? smem_u32(&acce_bar[acc]) : smem_u32(&relay_acce[acc]));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();  // neither CTA releases TMEM or exits while its peer may use it
  if (threadIdx.x == 0 && s_abort) report_error(a.status, MOE_ERR_TIMEOUT);
  if (!skip && warp == C::kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, C::kTmemCols);
  }
}

template <int KIND, typename T>
cudaLaunchConfig_t pair_config(int grid, cudaStream_t s, cudaLaunchAttribute* attr) {
  using C = PairCfg<KIND, T>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// How many CTA pairs of this kernel the device holds at once (the persistent
// grid must not exceed it, or the extra pairs would run as a second wave).
template <int KIND, typename T>
int max_pairs() {
  using C = PairCfg<KIND, T>;
  auto kern = pair_gemm_kernel<KIND, T>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pair_config<KIND, T>(2, nullptr, attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <int KIND, typename T>
cudaError_t launch(const GemmArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmB, int grid,
                   cudaStream_t s) {
  using C = PairCfg<KIND, T>;
  auto kern = pair_gemm_kernel<KIND, T>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pair_config<KIND, T>(grid, s, attr);
  return cudaLaunchKernelEx(&cfg, kern, a, tmA, tmB);
}

}  // namespace

int pair_max_active(int kind, int dtype) {
  if (kind == 0)
    return dtype == MOE_BF16 ? max_pairs<kGateUp, __nv_bfloat16>() : max_pairs<kGateUp, float>();
  return dtype == MOE_BF16 ? max_pairs<kDown, __nv_bfloat16>() : max_pairs<kDown, float>();
}

cudaError_t launch_pair_gate_up(int dtype, const GemmArgs& a, const CUtensorMap& tmA,
                                const CUtensorMap& tmB, int grid, cudaStream_t s) {
  if (dtype == MOE_BF16) return launch<kGateUp, __nv_bfloat16>(a, tmA, tmB, grid, s);
  return launch<kGateUp, float>(a, tmA, tmB, grid, s);
}

cudaError_t launch_pair_down(int dtype, const GemmArgs& a, const CUtensorMap& tmA,
                             const CUtensorMap& tmB, int grid, cudaStream_t s) {
  if (dtype == MOE_BF16) return launch<kDown, __nv_bfloat16>(a, tmA, tmB, grid, s);
  return launch<kDown, float>(a, tmA, tmB, grid, s);
}

}  // namespace moe
