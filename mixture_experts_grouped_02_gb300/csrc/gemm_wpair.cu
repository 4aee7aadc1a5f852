// gemm_wpair.cu -- the two bf16/fp32 grouped GEMMs of the expert FFN:
//   gate/up: h[s, j] = SiLU(w13[e, j, :] . x_s) * (w13[e, I + j, :] . x_s)
//   down:    y[q, s, c] = w_s * sum_{j in split q} w2[e, c, j] * h[s, j]
// for every valid slot s of an align block of expert e (x_s: the token row
// of slot s, in sorted order as moe_gather_rows writes it; w_s its routing
// weight).  Sources: "factor_moe_fused_gemm.cu", fused_silu_gate_kernel
// (gate = first half of the w13 rows, SiLU(g) = g / (1 + e^-g)); "moe triton
// kernel use tma", the review comment on TOKEN_INPUT_USE_TMA /
// MUL_ROUTED_WEIGHT (token rows contiguous in sorted order, routing weight
// in the down projection's epilogue); "MOE Bmm1 Fused Gather" (weights as
// the MMA's A operand, the gathered tokens as B, two-CTA mode).
//
// Tile.  One tcgen05.mma.cta_group::2 covers 256 weight rows (128 per CTA of
// a cluster of two) and N tokens of one align block, N = the block's valid
// row count rounded up to 16 (at most 256).  A block of an expert that
// received 5 tokens runs N = 16 instead of a full 128- or 256-row tile, so
// padding costs next to no tensor-core time and a sparsely used expert's
// tiles are pure weight streaming.  Per CTA and 64-wide K step: 128 weight
// rows (16 KB) and N/2 token rows, loaded as a 16-row box when N <= 32
// (decode) and as a 128-row box otherwise.  A stage carries two K steps
// (three 64 KB stages): the pipeline pays a fixed cost per stage, besides its
// bytes and MMAs, and two K steps per stage took the Mixtral-shaped prefill
// GEMMs from 1.21 / 0.64 ms to 1.13 / 0.60 ms against six stages of one.
// Decode-like launches use the DUAL instantiation (WCfg): six stages of one
// K step for large tiles, and for tiles of at most 32 tokens two K steps of
// weights in the W and X slots with their 16-row token boxes in a T slot.
// Gather mode (GemmArgs::gather, gate/up only): the token rows come straight
// from x, four rows per tile::gather4 copy by the x row of each slot, in
// place of the box of sorted rows; the shared-memory layout is the same.
//  * gate/up: a CTA's 128 weight rows are 64 gate rows and the 64 up rows
//    with the same indices j, so TMEM lanes 0-63 hold gate and 64-127 up of
//    the same j for every token column.  The epilogue warp of lanes
//    32q..32q+31 (q < 2) and the one of lanes 64+32q.. exchange half of each
//    32-column chunk through shared memory and each forms SiLU(g)*u for 16
//    tokens; the 32 lanes of a warp store 32 consecutive h values of a row;
//  * down: TMEM lane = output column, so the 32 lanes of a warp store 32
//    consecutive fp32 of one y row (128 bytes) per token.
//
// Pair protocol.  One producer thread per CTA issues its TMA copies with the
// .cta_group::2 form, which completes them on the LEADER's full barrier; the
// leader alone declares both CTAs' bytes there, so no follower thread signals
// the leader per stage (a cluster-scope release would wait for all of the
// releasing thread's earlier memory operations).  The leader's MMA thread
// issues the pair MMAs (A and B read from the same shared-memory offsets in
// both CTAs; each CTA's TMEM receives its 128 rows of D) and commits with a
// multicast to both CTAs' empty and accumulator-full barriers.  The
// follower's epilogue threads arrive on a barrier of their own CTA and one
// idle lane relays each accumulator release to the leader.  Both CTAs
// allocate TMEM as a pair and meet at a cluster barrier before freeing it.
//
// Schedule.  Persistent: one cluster per SM pair, tiles (block, weight tile,
// K split) walked in bands of weight tiles so that co-resident pairs share
// weight and token tiles in L2; two TMEM accumulators, so the epilogue of one
// tile overlaps the MMAs of the next.
//
// Every mbarrier wait is bounded (GemmArgs::timeout_ns of wall clock): a
// thread that gives up raises the CTA's abort flag, which every other wait
// polls, lets issued copies and MMAs drain, and the kernel records
// MOE_ERR_TIMEOUT in the status word and frees its TMEM.  A test launch
// (GemmArgs::starve) issues no copies, so that this path runs with nothing
// in flight.
#include <cuda_bf16.h>

#include "bounds.cuh"
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

// DUAL: the launch is made of small tiles (decode-like): each stage of a
// tile of at most 32 tokens carries two K steps of weights (W and X slots)
// and their two 16-row token boxes (T slot), twice the weight bytes in
// flight per pair.  Mixed with large tiles this measured slower, so it is a
// separate instantiation, chosen by the host (GemmArgs::dual_small).
template <int KIND, typename T, bool DUAL = false>
struct WCfg {
  static constexpr int kWRows = 128;          // weight rows per CTA (MMA M = 256 per pair)
  static constexpr int kNMax = 256;           // tokens per tile at most
  static constexpr int kRowBytes = 128;
  static constexpr int kBK = kRowBytes / sizeof(T);
  static constexpr int kUmmaK = 32 / sizeof(T);
  static constexpr int kSub = DUAL ? 1 : 2;   // K steps per stage (large tiles)
  static constexpr int kStages = DUAL ? 6 : 3;
  static constexpr int kStepWBytes = kWRows * kRowBytes;        // one K step of weights: 16 KB
  static constexpr int kABytes = kSub * kStepWBytes;            // W slot
  static constexpr int kBigRows = kNMax / 2;                    // token box rows
  static constexpr int kSmallRows = 16;
  static constexpr int kStepXBytes = kBigRows * kRowBytes;      // one K step of tokens: 16 KB
  static constexpr int kBBytes = kSub * kStepXBytes;            // X slot
  static constexpr int kSmallBytes = kSmallRows * kRowBytes;    // one 16-row token box
  static constexpr int kTBytes = DUAL ? 2 * kSmallBytes : 0;    // T slot (DUAL)
  static constexpr int kStageBytes = kABytes + kBBytes + kTBytes;
  static constexpr int kAccCols = kNMax;
  static constexpr int kTmemCols = 2 * kAccCols;
  static constexpr int kProducerWarp = 0;
  static constexpr int kMmaWarp = 1;
  static constexpr int kThreads = (2 + 4) * 32;
  // gate/up exchange: 2 warp pairs x 2 directions x 16 columns x 32 lanes
  static constexpr int kXchgBytes = KIND == kGateUp ? 2 * 2 * 16 * 32 * 4 : 0;
  static constexpr int kSmemBytes = kStages * kStageBytes + kXchgBytes + 1024;
};

// The activation of the first GEMM: SiLU(g) * u, or the clamped SwiGLU of
// GPT-OSS ("MOE Bmm1 Fused Gather", _swiglu_step1/2): the gate clamped from
// above at `limit`, the linear branch to [-limit, limit], then
// g * sigmoid(alpha g) * (u + 1).
__device__ __forceinline__ float activate(const Epilogue& ep, float g, float u) {
  if (ep.act == MOE_ACT_SWIGLU_CLAMP) {
    g = fminf(g, ep.limit);
    u = fmaxf(fminf(u, ep.limit), -ep.limit);
    return __fdividef(g, 1.0f + __expf(-ep.alpha * g)) * (u + 1.0f);
  }
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

__device__ __forceinline__ void settle(uint64_t ns) {
  const uint64_t t0 = global_timer_ns();
  while (global_timer_ns() - t0 < ns) {
  }
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Barrier `id` over `threads` threads that also ANDs `pred` across them.
__device__ __forceinline__ int named_bar_and(int id, int threads, int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred), "r"(id), "r"(threads)
      : "memory");
  return r;
}

// Tokens the MMA of a block with `valid` rows covers: a multiple of 16.
__device__ __forceinline__ int tile_n(int valid) {
  return min(256, max(16, (valid + 15) & ~15));
}

template <typename T>
__device__ __forceinline__ void store_h(T* p, float v);
template <>
__device__ __forceinline__ void store_h<float>(float* p, float v) {
  *p = v;
}

template <int KIND, typename T, bool DUAL>
__global__ void __launch_bounds__(WCfg<KIND, T, DUAL>::kThreads, 1)
    wpair_gemm_kernel(const __grid_constant__ GemmArgs a, const __grid_constant__ CUtensorMap tmTok,
                      const __grid_constant__ CUtensorMap tmTokS,
                      const __grid_constant__ CUtensorMap tmW,
                      const __grid_constant__ CUtensorMap tmWu,
                      const __grid_constant__ CUtensorMap tmX) {
  using C = WCfg<KIND, T, DUAL>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[C::kStages];
  __shared__ __align__(8) uint64_t empty_bar[C::kStages];
  __shared__ __align__(8) uint64_t accf_bar[2];
  __shared__ __align__(8) uint64_t acce_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ __align__(8) uint64_t relay_acce[2];
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_skip;
  __shared__ int s_skip_pair;
  __shared__ volatile int s_abort;
  // gather mode: x rows of this CTA's tokens of the current tile (producer)
  __shared__ int s_rows[WCfg<KIND, T, DUAL>::kNMax / 2];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t smemA = smem_base;                               // W slots
  const uint32_t smemB = smem_base + C::kStages * C::kABytes;     // X slots
  const uint32_t smemT = smemB + C::kStages * C::kBBytes;         // T slots (DUAL)
  float* xchg = reinterpret_cast<float*>(smem_raw + (smem_base - smem_u32(smem_raw)) +
                                         C::kStages * C::kStageBytes);

  // the earlier kernels of the stream (align, gather or the gate/up GEMM)
  // have finished before anything they wrote is read
  pdl_wait();
  pdl_launch_dependents();
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
  cluster_sync();
  if (threadIdx.x == 0)
    s_skip_pair = leader ? s_skip
                         : static_cast<int>(ld_shared_cluster_u32(mapa_shared(smem_u32(&s_skip), 0)));
  __syncthreads();
  const bool skip = s_skip_pair != 0;
  if (!skip && warp == C::kMmaWarp) tmem_alloc_pair(smem_u32(&s_tmem_base), C::kTmemCols);
  if (warp == C::kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmTok);
    tma_prefetch_desc(&tmTokS);
    tma_prefetch_desc(&tmW);
    if (KIND == kGateUp) tma_prefetch_desc(&tmWu);
    if (a.gather) tma_prefetch_desc(&tmX);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = s_tmem_base;

  const int num_blocks = skip ? 0 : checked_num_blocks(*a.num_blocks, a.max_blocks, a.status);
  const int total = num_blocks * a.n_tiles * a.splits;
  const int cluster = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;
  const uint64_t to = a.timeout_ns;

  if (warp == C::kProducerWarp) {
    // ------------------------------------------------------------ producer
    // (a.starve, the failure-path test: no copies at all, so that the
    // pipeline's first wait runs out with nothing in flight)
    if (lane == 0 && !a.starve) {
      const uint32_t full0 = mapa_shared(smem_u32(&full_bar[0]), 0);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int tile = cluster; tile < total && ok; tile += nclusters) {
        const Tile t = decode_tile(tile, num_blocks, a);
        const int4 bi = reinterpret_cast<const int4*>(a.block_info)[t.mb];
        const int e = bi.x;
        const int n = tile_n(bi.w);
        const int half = n >> 1;
        const bool small = half <= C::kSmallRows;
        const int tok_row = bi.z + static_cast<int>(rank) * half;
        // token rows per K step: a 16- or 128-row box of the sorted rows, or
        // (gather mode) this CTA's `half` rows gathered from x, four at a
        // time, by the x row of each slot (padding slots read row 0; their
        // accumulator columns are not stored)
        const int tok_rows = a.gather ? half : (small ? C::kSmallRows : C::kBigRows);
        if (a.gather) {
          for (int i = 0; i < half; ++i) {
            const long long slot = static_cast<long long>(tok_row) + i;
            int x_row = 0;
            if (slot < a.cap) {
              const int sid = a.sorted_ids[slot];
              if (sid >= 0 && sid < a.T * a.K) x_row = sid / a.K;
            }
            s_rows[i] = x_row;
          }
        }
        auto load_tokens = [&](uint32_t dst, uint32_t fb, int kcoord) {
          if (a.gather) {
            for (int g = 0; g < half; g += 4)
              tma_gather4_pair(dst + g * C::kRowBytes, &tmX, fb, kcoord, s_rows[g], s_rows[g + 1],
                               s_rows[g + 2], s_rows[g + 3]);
          } else {
            tma_load_2d_pair(dst, small ? &tmTokS : &tmTok, fb, kcoord, tok_row);
          }
        };
        // bytes of one K step of both CTAs
        const uint32_t tx = 2u * static_cast<uint32_t>(C::kStepWBytes + tok_rows * C::kRowBytes);
        // this CTA's weight rows: 64 gate rows j and the 64 up rows j (at
        // the same row of the up map, shifted by up_row_offset), or 128 rows
        // of w2
        const int wrow = KIND == kGateUp
                             ? e * a.w_rows_per_expert + t.nt * 128 + static_cast<int>(rank) * 64
                             : e * a.H + t.nt * 256 + static_cast<int>(rank) * 128;
        int kb, ke;
        split_range(a, t.split, kb, ke);
        if (DUAL && small) {
          // two K steps per stage: weights in the W and X slots, token boxes
          // in the two halves of the T slot
          for (int kt = kb; kt < ke; kt += 2) {
            if (!mbar_wait_bounded(smem_u32(&empty_bar[stage]), phase ^ 1, &s_abort, to)) {
              ok = false;
              break;
            }
            const uint32_t fb = full0 + stage * 8u;
            const int nk = min(2, ke - kt);
            const uint32_t st = smemT + stage * C::kTBytes;
            if (leader) mbar_arrive_expect_tx(smem_u32(&full_bar[stage]), tx * nk);
            for (int u = 0; u < nk; ++u) {
              const uint32_t sw = u == 0 ? smemA + stage * C::kABytes : smemB + stage * C::kBBytes;
              if constexpr (KIND == kGateUp) {
                tma_load_2d_pair(sw, &tmW, fb, (kt + u) * C::kBK, wrow);
                tma_load_2d_pair(sw + C::kABytes / 2, &tmWu, fb, (kt + u) * C::kBK,
                                 wrow + a.up_row_offset);
              } else {
                tma_load_2d_pair(sw, &tmW, fb, (kt + u) * C::kBK, wrow);
              }
              load_tokens(st + u * C::kSmallBytes, fb, (kt + u) * C::kBK);
            }
            if (++stage == C::kStages) {
              stage = 0;
              phase ^= 1;
            }
          }
          continue;
        }
        for (int kt = kb; kt < ke; kt += C::kSub) {
          if (!mbar_wait_bounded(smem_u32(&empty_bar[stage]), phase ^ 1, &s_abort, to)) {
            ok = false;
            break;
          }
          const uint32_t fb = full0 + stage * 8u;
          const int nk = min(C::kSub, ke - kt);
          if (leader) mbar_arrive_expect_tx(smem_u32(&full_bar[stage]), tx * nk);
          for (int u = 0; u < nk; ++u) {
            const uint32_t sa = smemA + stage * C::kABytes + u * C::kStepWBytes;
            if constexpr (KIND == kGateUp) {
              tma_load_2d_pair(sa, &tmW, fb, (kt + u) * C::kBK, wrow);
              tma_load_2d_pair(sa + C::kStepWBytes / 2, &tmWu, fb, (kt + u) * C::kBK,
                               wrow + a.up_row_offset);
            } else {
              tma_load_2d_pair(sa, &tmW, fb, (kt + u) * C::kBK, wrow);
            }
            load_tokens(smemB + stage * C::kBBytes + u * C::kStepXBytes, fb, (kt + u) * C::kBK);
          }
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) settle(to / 8);
    }
    __syncwarp();
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (leader && lane == 0) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = cluster; tile < total && ok; tile += nclusters) {
        const Tile t = decode_tile(tile, num_blocks, a);
        const int4 bi = reinterpret_cast<const int4*>(a.block_info)[t.mb];
        const uint32_t idesc = make_idesc(Elem<T>::kFmt, 256, tile_n(bi.w));
        int kb, ke;
        split_range(a, t.split, kb, ke);
        if (!mbar_wait_bounded_cluster(smem_u32(&acce_bar[acc]), acc_phase ^ 1, &s_abort, to)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * C::kAccCols;
        if (DUAL && (tile_n(bi.w) >> 1) <= C::kSmallRows) {  // as the producer decides
          for (int kt = kb; kt < ke; kt += 2) {
            if (!mbar_wait_bounded_cluster(smem_u32(&full_bar[stage]), phase, &s_abort, to)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const int nk = min(2, ke - kt);
            for (int u = 0; u < nk; ++u) {
              const uint32_t a_base =
                  u == 0 ? smemA + stage * C::kABytes : smemB + stage * C::kBBytes;
              const uint32_t b_base = smemT + stage * C::kTBytes + u * C::kSmallBytes;
#pragma unroll
              for (int k = 0; k < C::kBK / C::kUmmaK; ++k) {
                const uint64_t ad = sw128_kmajor_desc(a_base + k * 32);
                const uint64_t bd = sw128_kmajor_desc(b_base + k * 32);
                const uint32_t accum = (kt > kb || u > 0 || k > 0) ? 1u : 0u;
                if constexpr (Elem<T>::kFmt == 1)
                  umma_bf16_pair(d_tmem, ad, bd, idesc, accum);
                else
                  umma_tf32_pair(d_tmem, ad, bd, idesc, accum);
              }
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
          continue;
        }
        for (int kt = kb; kt < ke; kt += C::kSub) {
          if (!mbar_wait_bounded_cluster(smem_u32(&full_bar[stage]), phase, &s_abort, to)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const int nk = min(C::kSub, ke - kt);
          for (int u = 0; u < nk; ++u) {
            const uint32_t a_base = smemA + stage * C::kABytes + u * C::kStepWBytes;
            const uint32_t b_base = smemB + stage * C::kBBytes + u * C::kStepXBytes;
#pragma unroll
            for (int k = 0; k < C::kBK / C::kUmmaK; ++k) {
              const uint64_t ad = sw128_kmajor_desc(a_base + k * 32);
              const uint64_t bd = sw128_kmajor_desc(b_base + k * 32);
              const uint32_t accum = (kt > kb || u > 0 || k > 0) ? 1u : 0u;
              if constexpr (Elem<T>::kFmt == 1)
                umma_bf16_pair(d_tmem, ad, bd, idesc, accum);
              else
                umma_tf32_pair(d_tmem, ad, bd, idesc, accum);
            }
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
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = cluster; tile < total; tile += nclusters) {
      const Tile t = decode_tile(tile, num_blocks, a);
      const int4 bi = reinterpret_cast<const int4*>(a.block_info)[t.mb];
      // checked build: a block outside the held experts or the capacity
      // stores and loads nothing (valid = 0)
      const bool bi_ok = block_in_bounds(bi, a.n_held, a.cap, C::kNMax, a.status);
      const int valid = bi_ok ? bi.w : 0;
      const int n = tile_n(bi.w);
      // down: the routing weight and token row of slot 32j + lane, and this
      // lane's w2 bias, loaded before the accumulator is ready so that
      // their latency hides behind the MMAs (short-K tiles are otherwise
      // bound by these dependent loads)
      constexpr int kChunks = C::kNMax / 32;
      float w_r[kChunks];
      int tok_r[kChunks];
      float bias2 = 0.0f;
      if constexpr (KIND == kDown) {
        int sid[kChunks];
#pragma unroll
        for (int j = 0; j < kChunks; ++j) {
          const int my = 32 * j + lane;
          sid[j] = my < valid ? a.sorted_ids[bi.z + my] : -1;
          if (sid[j] >= 0 && !in_bounds(sid[j] < a.T * a.K, a.status)) sid[j] = -1;
        }
#pragma unroll
        for (int j = 0; j < kChunks; ++j) {
          w_r[j] = sid[j] >= 0 ? a.topk_weights[sid[j]] : 0.0f;
          tok_r[j] = sid[j] >= 0 ? sid[j] / a.K : 0;
        }
        // the w2 bias joins once, in the first K split
        const int c = t.nt * 256 + static_cast<int>(rank) * 128 + q * 32 + lane;
        if (a.ep.b2 != nullptr && t.split == 0 && c < a.H && bi_ok)
          bias2 = a.ep.b2[static_cast<long long>(bi.x) * a.H + c];
      }
      int good = 1;
      if (lane == 0) good = mbar_wait_bounded(smem_u32(&accf_bar[acc]), acc_phase, &s_abort, to);
      good = __shfl_sync(0xffffffffu, good, 0);
      // the two warps of an exchange pair leave together or not at all
      if constexpr (KIND == kGateUp) good = named_bar_and(1 + (q & 1), 64, good);
      if (!good) break;
      tc_fence_after_sync();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * C::kAccCols;
      if constexpr (KIND == kGateUp) {
        const bool gate_warp = q < 2;
        const int pq = q & 1;
        const int j = t.nt * 128 + static_cast<int>(rank) * 64 + pq * 32 + lane;
        float* x_g = xchg + (pq * 2 + 0) * 16 * 32;  // gate, columns 16..31 of a chunk
        float* x_u = xchg + (pq * 2 + 1) * 16 * 32;  // up, columns 0..15
        T* hcol = reinterpret_cast<T*>(a.out) + j;
        // this lane's bias: of gate j (lanes 0-63) or of up j (64-127)
        float bias = 0.0f;
        if (a.ep.b13 != nullptr && j < a.I && bi_ok)
          bias = a.ep.b13[gate_warp ? gate_bias_index(a.ep, a.I, bi.x, j)
                                    : up_bias_index(a.ep, a.I, bi.x, j)];
        for (int c0 = 0; c0 < n; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(taddr + c0, v);
          tmem_wait_ld();
          if (gate_warp) {
#pragma unroll
            for (int i = 0; i < 16; ++i) x_g[i * 32 + lane] = __uint_as_float(v[16 + i]) + bias;
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) x_u[i * 32 + lane] = __uint_as_float(v[i]) + bias;
          }
          named_bar_sync(1 + pq, 64);
          // gate warp: tokens c0..c0+15; up warp: tokens c0+16..c0+31
          const int nb = gate_warp ? c0 : c0 + 16;
          float hv[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float g = gate_warp ? __uint_as_float(v[i]) + bias : x_g[i * 32 + lane];
            const float u = gate_warp ? x_u[i * 32 + lane] : __uint_as_float(v[16 + i]) + bias;
            hv[i] = activate(a.ep, g, u);
          }
          if constexpr (sizeof(T) == 2) {
            // lanes 2m and 2m+1 hold columns j and j+1: per pair of rows the
            // even lane stores row i and the odd lane row i+1, each as one
            // bf16x2 word, after one exchange (j < I is the same for the
            // whole warp, as I is a multiple of 64)
            const bool odd = lane & 1;
            __nv_bfloat16* hpair = reinterpret_cast<__nv_bfloat16*>(a.out) + (j & ~1);
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              const float recv = __shfl_xor_sync(0xffffffffu, odd ? hv[i] : hv[i + 1], 1);
              const int r = odd ? i + 1 : i;
              const __nv_bfloat162 pk =
                  odd ? __floats2bfloat162_rn(recv, hv[i + 1]) : __floats2bfloat162_rn(hv[i], recv);
              if (j < a.I && nb + r < valid)
                *reinterpret_cast<__nv_bfloat162*>(
                    hpair + static_cast<long long>(bi.z + nb + r) * a.I) = pk;
            }
          } else if (j < a.I) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (nb + i < valid) store_h<T>(hcol + static_cast<long long>(bi.z + nb + i) * a.I, hv[i]);
          }
          named_bar_sync(1 + pq, 64);  // the exchange slots are free again
        }
      } else {
        const int c = t.nt * 256 + static_cast<int>(rank) * 128 + q * 32 + lane;
        float* ycol = reinterpret_cast<float*>(a.out) +
                      static_cast<long long>(t.split) * a.cap * a.H + c;
        const float bias = bias2;
#pragma unroll
        for (int jc = 0; jc < kChunks; ++jc) {
          const int c0 = 32 * jc;
          if (c0 >= n) break;
          uint32_t v[32];
          tmem_ld32(taddr + c0, v);
          // routing weight (and, for a fused combine, the token row) of slot
          // c0 + lane, broadcast below
          const float w_l = w_r[jc];
          const int tok_l = tok_r[jc];
          tmem_wait_ld();
          if (a.fused) {
            // the scatter-add: 32 lanes add 128 contiguous bytes of one row
            float* acc_c = reinterpret_cast<float*>(a.out) + c;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float w = __shfl_sync(0xffffffffu, w_l, i);
              const int tok = __shfl_sync(0xffffffffu, tok_l, i);
              if (c0 + i < valid && c < a.H)
                atomicAdd(acc_c + static_cast<long long>(tok) * a.H, w * (__uint_as_float(v[i]) + bias));
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float w = __shfl_sync(0xffffffffu, w_l, i);
              if (c0 + i < valid && c < a.H)
                ycol[static_cast<long long>(bi.z + c0 + i) * a.H] = w * (__uint_as_float(v[i]) + bias);
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
  cluster_sync();
  if (threadIdx.x == 0 && s_abort) report_error(a.status, MOE_ERR_TIMEOUT);
  if (!skip && warp == C::kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, C::kTmemCols);
  }
}

template <int KIND, typename T, bool DUAL>
cudaLaunchConfig_t wpair_config(int grid, cudaStream_t s, cudaLaunchAttribute* attr) {
  using C = WCfg<KIND, T, DUAL>;
  return pdl_config(dim3(grid), dim3(C::kThreads), C::kSmemBytes, s, attr, 2);
}

// Pairs held at once (both instantiations keep one CTA per SM).
template <int KIND, typename T, bool DUAL = false>
int max_pairs() {
  using C = WCfg<KIND, T, DUAL>;
  auto kern = wpair_gemm_kernel<KIND, T, DUAL>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = wpair_config<KIND, T, DUAL>(2, nullptr, attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <int KIND, typename T, bool DUAL>
cudaError_t launch_as(const GemmArgs& a, const CUtensorMap& tmTok, const CUtensorMap& tmTokS,
                      const CUtensorMap& tmW, const CUtensorMap& tmWu, const CUtensorMap& tmX,
                      int grid, cudaStream_t s) {
  using C = WCfg<KIND, T, DUAL>;
  auto kern = wpair_gemm_kernel<KIND, T, DUAL>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = wpair_config<KIND, T, DUAL>(grid, s, attr);
  return cudaLaunchKernelEx(&cfg, kern, a, tmTok, tmTokS, tmW, tmWu, tmX);
}

template <int KIND, typename T>
cudaError_t launch(const GemmArgs& a, const CUtensorMap& tmTok, const CUtensorMap& tmTokS,
                   const CUtensorMap& tmW, const CUtensorMap& tmWu, const CUtensorMap& tmX,
                   int grid, cudaStream_t s) {
  if (a.dual_small) return launch_as<KIND, T, true>(a, tmTok, tmTokS, tmW, tmWu, tmX, grid, s);
  return launch_as<KIND, T, false>(a, tmTok, tmTokS, tmW, tmWu, tmX, grid, s);
}

}  // namespace

int wpair_max_active(int kind, int dtype) {
  if (kind == 0)
    return dtype == MOE_BF16 ? max_pairs<kGateUp, __nv_bfloat16>() : max_pairs<kGateUp, float>();
  return dtype == MOE_BF16 ? max_pairs<kDown, __nv_bfloat16>() : max_pairs<kDown, float>();
}

cudaError_t launch_wpair_gate_up(int dtype, const GemmArgs& a, const CUtensorMap& tmTok,
                                 const CUtensorMap& tmTokS, const CUtensorMap& tmW,
                                 const CUtensorMap& tmWu, const CUtensorMap& tmX, int grid,
                                 cudaStream_t s) {
  if (dtype == MOE_BF16)
    return launch<kGateUp, __nv_bfloat16>(a, tmTok, tmTokS, tmW, tmWu, tmX, grid, s);
  return launch<kGateUp, float>(a, tmTok, tmTokS, tmW, tmWu, tmX, grid, s);
}

cudaError_t launch_wpair_down(int dtype, const GemmArgs& a, const CUtensorMap& tmTok,
                              const CUtensorMap& tmTokS, const CUtensorMap& tmW, int grid,
                              cudaStream_t s) {
  if (dtype == MOE_BF16)
    return launch<kDown, __nv_bfloat16>(a, tmTok, tmTokS, tmW, tmW, tmTok, grid, s);
  return launch<kDown, float>(a, tmTok, tmTokS, tmW, tmW, tmTok, grid, s);
}

}  // namespace moe
