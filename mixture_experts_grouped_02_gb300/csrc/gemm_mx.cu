// gemm_mx.cu -- the two grouped GEMMs of the low-precision MoE expert FFN:
// fp8 (e4m3) activations times mxfp4 weights (e2m1 values, one e8m0 scale per
// 32 K elements), tcgen05 block-scaled MMAs (kind::mxf8f6f4) on sm_103a.
//
// Sources: "MOE Bmm1 Fused Gather" -- load_weights brings a weight tile and
// its scale tile in by TMA, mma_partition copies the scales into tensor
// memory (tcgen05_copy) and issues block-scaled MMAs of e2m1 weights against
// e4m3 activations, and ws_matmul_kernel fills the activation scale tensor
// with the e8m0 code 127 (unit scales; here the per-row fp8 scale of x is
// applied in the epilogue instead); the weights arrive pre-arranged for the
// kernel (its MX4 value and scale layouts); pack_e4m3x2 (fp32 -> e4m3, round
// to nearest even, saturating) for the hidden activation.  The epilogues form
// SiLU(g)*u per row (gate/up) and multiply the routing weight (down), as the
// bf16 GEMMs do.
//
// Layout per CTA (one per SM, persistent, tiles walked in bands of N tiles
// so that co-resident CTAs share weight tiles in L2):
//  * tile = 128 sorted rows x 192 weight rows, one MMA of N = 192 per
//    32-element K block: gate/up: 96 gate rows and the matching 96 up rows
//    of w13[e]; down: 192 rows of w2[e];
//  * 5 shared-memory stages of 128 K elements: A = 128 rows of e4m3 (128 B,
//    128-byte swizzled K-major), B = 192 rows of e2m1 expanded by the TMA
//    unit into the 16-byte slots the block-scaled MMA reads 4-bit operands
//    from (16 values in the first 8 bytes), swizzled the same way, and the
//    tile's 1 KB scale image (two 128-row parts of 512 bytes);
//  * the weights are packed tile-major (moe_pack_mx_weights): the 192 weight
//    rows x 128 K elements of one stage are 12 KB of consecutive bytes,
//    loaded by one TMA box (a stage issues three copies: A, weights, scales;
//    the weights as two 96-row boxes measured 3-7 % slower);
//  * one producer thread fills a stage with TMA: A as a plain tile of sorted
//    rows (gate/up: the fp8 step has already written each token's codes to
//    the slots it occupies, so the gather happened there; down: hq; the end
//    of K past the tensor reads as zeros; a block of at most 64 valid rows
//    loads a 64-row box, half the bytes), the weight tile and the two scale
//    images (bulk copies), all completing one mbarrier;
//  * the MMA thread copies each stage's scale image into tensor memory (two
//    tcgen05.cp of 32 x 128 bits replicated into the four lane quarters, at
//    columns 0 and 4 of the stage's block: column c of lane l holds the 4
//    K-block scales of tile row 32c + l) and issues the MMAs, choosing the
//    scale byte of each 32-element K block by the instruction descriptor's
//    scale ids.  One N = 192 MMA per K block instead of two of N = 96 halves
//    the MMA instructions and the reads of the A tile: measured, the MMA
//    instructions of this kernel, not their arithmetic, had set its pace;
//  * tensor memory: two 192-column fp32 accumulators, 4 columns of unit A
//    scales at column 384, and a 16-column block of B scales per stage from
//    column 400 (6 columns used; every copy and MMA operand starts on a
//    multiple of 4 columns).
//
// Every mbarrier wait is bounded (MxArgs::timeout_ns of wall clock); a thread
// that gives up raises the CTA's abort flag, which every other wait polls,
// and the kernel records MOE_ERR_TIMEOUT, drains and frees its TMEM.  A test
// launch (MxArgs::starve) issues no copies, so that this path runs with
// nothing in flight.
#include <cuda_bf16.h>

#include "bounds.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "sched.cuh"

namespace moe {
namespace {

enum MxKind { kMxGateUp = 0, kMxDown = 1 };

template <int KIND>
struct MxCfg {
  static constexpr int kBM = kBlockM;                 // 128 sorted rows
  static constexpr int kHalf = 96;                    // weight rows per MMA
  static constexpr int kBN = 2 * kHalf;               // weight rows per tile
  static constexpr int kRowBytes = 128;
  static constexpr int kBK = 128;                     // K elements per stage
  static constexpr int kUmmaK = 32;                   // K per MMA (one scale block)
  static constexpr int kStages = 5;
  static constexpr int kABytes = kBM * kRowBytes;     // 16 KB
  static constexpr int kAHalfRows = kBM / 2;          // the short A box (blocks of <= 64 rows)
  static constexpr int kAHalfBytes = kAHalfRows * kRowBytes;
  static constexpr int kBBytes = kBN * kRowBytes;     // 24 KB in shared memory
  static constexpr int kBDataBytes = kBN * kBK / 2;   // 12 KB of packed values
  static constexpr int kSfImage = 512;                // 128 tile rows x 4 K blocks of scales
  static constexpr int kSfBytes = 2 * kSfImage;       // the tile's 192 rows (and filler)
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kAccCols = kBN;                // 192 fp32 columns
  static constexpr int kSfaCol = 2 * kAccCols;        // 384: unit A scales (4 columns)
  static constexpr int kSfbCol0 = kSfaCol + 16;       // 400: B scales, 16 columns per stage
  static constexpr int kSfbStride = 16;
  static constexpr int kTmemCols = 512;
  static constexpr int kProducerWarps = 1;
  static constexpr int kMmaWarp = kProducerWarps;
  static constexpr int kThreads = (kProducerWarps + 1 + 4) * 32;
  // bytes the TMA unit and the bulk copies deliver per stage
  static constexpr uint32_t kTxBytes = kABytes + kBDataBytes + kSfBytes;
  static constexpr int kSmemBytes = kStages * (kStageBytes + kSfBytes) + 1024;
  static constexpr uint32_t kIdesc = make_idesc_mx_e4m3_e2m1(kBM, kBN);
};
static_assert(MxCfg<0>::kSfbCol0 + MxCfg<0>::kStages * MxCfg<0>::kSfbStride <=
                  MxCfg<0>::kTmemCols,
              "TMEM budget");

// First TMEM column of a stage's B scales (a multiple of 16).
template <int KIND>
__device__ __forceinline__ uint32_t sfb_col(int stage) {
  return MxCfg<KIND>::kSfbCol0 + stage * MxCfg<KIND>::kSfbStride;
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// Barrier over the 128 epilogue threads (named barrier 1) that also ANDs
// `pred` across them.
__device__ __forceinline__ int epilogue_bar_and(int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred)
      : "memory");
  return r;
}

// The activation: SiLU(g) * u, or GPT-OSS's clamped SwiGLU ("MOE Bmm1 Fused
// Gather", _swiglu_step1/2): gate clamped from above at `limit`, linear
// branch to [-limit, limit], g * sigmoid(alpha g) * (u + 1).
__device__ __forceinline__ float activate(const Epilogue& ep, float g, float u) {
  if (ep.act == MOE_ACT_SWIGLU_CLAMP) {
    g = fminf(g, ep.limit);
    u = fmaxf(fminf(u, ep.limit), -ep.limit);
    return __fdividef(g, 1.0f + __expf(-ep.alpha * g)) * (u + 1.0f);
  }
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// Outer coordinate of the first of the 192 rows of weight tile nt of expert
// e over K tile kt in the tile-major value map (rows of 128 K elements; the
// host checks that it fits in 32 bits).
__device__ __forceinline__ int value_row(const MxArgs& a, int e, int nt, int kt) {
  return static_cast<int>(
      ((static_cast<long long>(e) * a.n_tiles + nt) * a.kp_tiles + kt) * 192);
}
// The 1 KB scale image of weight tile nt of expert e over K tile kt.
__device__ __forceinline__ const uint8_t* sf_image(const MxArgs& a, int e, int nt, int kt) {
  return a.w_scale + ((static_cast<long long>(e) * a.n_tiles + nt) * a.kp_tiles + kt) * 1024;
}

template <int KIND>
__global__ void __launch_bounds__(MxCfg<KIND>::kThreads, 1)
    mx_gemm_kernel(const __grid_constant__ MxArgs a, const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmA64,
                   const __grid_constant__ CUtensorMap tmW) {
  using C = MxCfg<KIND>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[C::kStages];
  __shared__ __align__(8) uint64_t empty_bar[C::kStages];
  __shared__ __align__(8) uint64_t accf_bar[2];
  __shared__ __align__(8) uint64_t acce_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_skip;
  __shared__ volatile int s_abort;
  // biases of the tile's 192 weight rows (gate/up: 96 gate then 96 up;
  // down: 192 columns of the w2 bias), one set per accumulator
  __shared__ float s_bias[2][C::kBN];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t smemA = smem_base;
  const uint32_t smemB = smemA + C::kStages * C::kABytes;
  const uint32_t smemS = smemB + C::kStages * C::kBBytes;

  // the earlier kernels of the stream have finished before their output is read
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
      mbar_init(smem_u32(&acce_bar[i]), 128);
    }
    mbar_init(smem_u32(&drain_bar), 1);
    fence_barrier_init();
  }
  // the TMA unit writes only the first 8 bytes of each 16-byte slot of B;
  // the other 8 stay zero
  {
    uint4* b = reinterpret_cast<uint4*>(smem_raw + (smemB - smem_u32(smem_raw)));
    for (int i = threadIdx.x; i < C::kStages * C::kBBytes / 16; i += blockDim.x)
      b[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  fence_proxy_async_smem();
  __syncthreads();
  if (s_skip) return;
  if (warp == C::kMmaWarp) tmem_alloc(smem_u32(&s_tmem_base), C::kTmemCols);
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmA64);
    tma_prefetch_desc(&tmW);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = s_tmem_base;
  if (warp > C::kMmaWarp) {  // unit activation scales, one lane quarter per epilogue warp
    tmem_st4(tmem_base + (static_cast<uint32_t>((warp & 3) * 32) << 16) + C::kSfaCol,
             0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
    tmem_wait_st();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();

  const int num_blocks = checked_num_blocks(*a.num_blocks, a.max_blocks, a.status);
  const int total = num_blocks * a.n_tiles * a.splits;
  const uint64_t to = a.timeout_ns;

  // A tile, weight tile and scale images of one stage; thread-0 work.  A
  // block of at most 64 valid rows loads only its first 64 A rows: rows 64-127
  // of the stage keep whatever an earlier stage left there, which reaches
  // only accumulator rows 64-127 (each accumulator row reads its own A row),
  // and the epilogue stores none of those.
  auto load_stage = [&](const Tile& t, int e, int r0, bool short_a, int kt, uint32_t stage,
                        bool bi_ok) {
    const uint32_t fb = smem_u32(&full_bar[stage]);
    const uint32_t b_dst = smemB + stage * C::kBBytes;
    const uint32_t s_dst = smemS + stage * C::kSfBytes;
    mbar_arrive_expect_tx(fb, C::kTxBytes - (short_a ? C::kABytes - C::kAHalfBytes : 0));
    tma_load_2d(smemA + stage * C::kABytes, short_a ? &tmA64 : &tmA, fb, kt * C::kBK, r0);
    // the tile's 192 weight rows (gate/up: 96 gate rows, then the 96 up rows
    // of the same indices)
    tma_load_2d(b_dst, &tmW, fb, 0, value_row(a, e, t.nt, kt));
    bulk_load(s_dst, bi_ok ? sf_image(a, e, t.nt, kt) : a.w_scale, C::kSfBytes, fb);
  };

  if (warp < C::kProducerWarps) {
      // ------------------------------------------------------- TMA producer
      // (a.starve, the failure-path test: no copies at all, so that the
      // pipeline's first wait runs out with nothing in flight)
      uint32_t stage = 0, phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok && !a.starve; tile += gridDim.x) {
        const Tile t = decode_tile(tile, num_blocks, a);
        const int4 bi = reinterpret_cast<const int4*>(a.block_info)[t.mb];
        const int e = bi.x, r0 = bi.z;
        const bool bi_ok = block_in_bounds(bi, a.n_held, a.cap, C::kBM, nullptr);
        const bool short_a = bi.w <= C::kAHalfRows;
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
          if (lane == 0) load_stage(t, e, r0, short_a, kt, stage, bi_ok);
          ++issued;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok && lane == 0) {
        const long long first = issued > C::kStages ? issued - C::kStages : 0;
        for (long long n = first; n < issued; ++n)
          drain_wait(smem_u32(&full_bar[n % C::kStages]),
                     static_cast<uint32_t>((n / C::kStages) & 1), to / 4);
      }
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      const uint32_t sfa = tmem_base + C::kSfaCol;
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
          const uint32_t s_base = smemS + stage * C::kSfBytes;
          // tile rows 0-127 to columns 0-3, rows 128-191 (and filler) to 4-7
          const uint32_t sfb = tmem_base + sfb_col<KIND>(stage);
          tmem_cp_32x128b_x4(sfb, rows16_desc(s_base));
          tmem_cp_32x128b_x4(sfb + 4, rows16_desc(s_base + C::kSfImage));
#pragma unroll
          for (int k = 0; k < C::kBK / C::kUmmaK; ++k) {
            const uint64_t ad = sw128_kmajor_desc(a_base + k * 32);
            const uint64_t bd = sw128_kmajor_desc(b_base + k * 32);
            const uint32_t idesc = idesc_with_sf_ids(C::kIdesc, k, k);
            const uint32_t accum = (kt > kb || k > 0) ? 1u : 0u;
            umma_mxf8f6f4(d_tmem, ad, bd, idesc, sfa, sfb, accum);
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
        umma_commit(smem_u32(&drain_bar));
        drain_wait(smem_u32(&drain_bar), 0, to / 4);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int et = threadIdx.x - (C::kMmaWarp + 1) * 32;  // 0..127 over the epilogue warps
    const bool has_bias = KIND == kMxGateUp ? a.ep.b13 != nullptr : a.ep.b2 != nullptr;
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const Tile t = decode_tile(tile, num_blocks, a);
      const int4 bi = reinterpret_cast<const int4*>(a.block_info)[t.mb];
      // checked build: a block outside the held experts or the capacity
      // loads and stores nothing (valid = 0)
      const bool bi_ok = block_in_bounds(bi, a.n_held, a.cap, C::kBM, a.status);
      const int r0 = bi.z, valid = bi_ok ? bi.w : 0;
      if (has_bias && bi_ok) {
        // this tile's biases, read once; the slot of this accumulator was
        // last read two tiles ago, before the barrier of the previous tile
        for (int i = et; i < C::kBN; i += 128) {
          float b = 0.0f;
          if constexpr (KIND == kMxGateUp) {
            const int j = t.nt * C::kHalf + (i % C::kHalf);
            if (j < a.I)
              b = a.ep.b13[i < C::kHalf ? gate_bias_index(a.ep, a.I, bi.x, j)
                                        : up_bias_index(a.ep, a.I, bi.x, j)];
          } else {
            const int c = t.nt * C::kBN + i;
            if (c < a.H && t.split == 0) b = a.ep.b2[static_cast<long long>(bi.x) * a.H + c];
          }
          s_bias[acc][i] = b;
        }
      }
      const bool row_ok = r < valid;
      float rs = 0.0f, wt = 0.0f;
      int tok = 0;  // down, fused combine: the accumulator row
      if (row_ok) {
        int i = a.sorted_ids[r0 + r];
        if (!in_bounds(i >= 0 && i < a.T * a.K, a.status)) i = 0;
        if constexpr (KIND == kMxGateUp) {
          rs = a.x_row_scale[i / a.K];
        } else {
          wt = a.topk_weights[i];
          rs = wt * a.h_scale;
          tok = i / a.K;
        }
      }
      int good = 1;
      if (lane == 0) good = mbar_wait_bounded(smem_u32(&accf_bar[acc]), acc_phase, &s_abort, to);
      good = __shfl_sync(0xffffffffu, good, 0);
      // the four epilogue warps agree on going on (and see the biases)
      good = epilogue_bar_and(good);
      if (!good) break;
      tc_fence_after_sync();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * C::kAccCols;
      const float* sb = s_bias[acc];
      if constexpr (KIND == kMxGateUp) {
        // a / h_scale as a product with the fp32 reciprocal (1.4 % faster
        // than the IEEE division; the two differ by at most an ulp of fp32
        // before the e4m3 rounding, and not at all for a power-of-two scale)
        const float inv_hs = 1.0f / a.h_scale;
        uint8_t* hq = static_cast<uint8_t*>(a.out) + static_cast<long long>(r0 + r) * a.I;
#pragma unroll 1
        for (int c = 0; c < 3; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32(taddr + c * 32, g);
          tmem_ld32(taddr + C::kHalf + c * 32, u);
          tmem_wait_ld();
          const int j0 = t.nt * C::kHalf + c * 32;
          if (row_ok && j0 < a.I) {
            uint32_t pk[8];
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              float o[4];
#pragma unroll
              for (int w = 0; w < 4; ++w) {
                float gg = rs * __uint_as_float(g[4 * v + w]);
                float uu = rs * __uint_as_float(u[4 * v + w]);
                if (has_bias) {
                  gg += sb[c * 32 + 4 * v + w];
                  uu += sb[C::kHalf + c * 32 + 4 * v + w];
                }
                o[w] = activate(a.ep, gg, uu) * inv_hs;
              }
              pk[v] = e4m3x4(o[0], o[1], o[2], o[3]);
            }
            uint4* dst = reinterpret_cast<uint4*>(hq + j0);
            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      } else {
        // the row of y, or (fused combine) the token's accumulator row
        float* y = static_cast<float*>(a.out) +
                   (a.fused ? static_cast<long long>(tok)
                            : static_cast<long long>(t.split) * a.cap + r0 + r) * a.H;
#pragma unroll 1
        for (int c = 0; c < 6; ++c) {
          uint32_t v[32];
          tmem_ld32(taddr + c * 32, v);
          tmem_wait_ld();
          const int col0 = t.nt * C::kBN + c * 32;
          if (row_ok && col0 < a.H) {
            float4* dst = reinterpret_cast<float4*>(y + col0);
            // the w2 bias (zero past the first K split) times the weight
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              float o[4];
#pragma unroll
              for (int w = 0; w < 4; ++w)
                o[w] = rs * __uint_as_float(v[4 * i + w]) +
                       (has_bias ? wt * sb[c * 32 + 4 * i + w] : 0.0f);
              if (a.fused)
                atomicAdd(dst + i, make_float4(o[0], o[1], o[2], o[3]));
              else
                dst[i] = make_float4(o[0], o[1], o[2], o[3]);
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

template <int KIND>
cudaError_t launch(const MxArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmA64,
                   const CUtensorMap& tmW, int grid, cudaStream_t s) {
  using C = MxCfg<KIND>;
  auto kern = mx_gemm_kernel<KIND>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = pdl_config(dim3(grid), dim3(C::kThreads), C::kSmemBytes, s, attr);
  return cudaLaunchKernelEx(&cfg, kern, a, tmA, tmA64, tmW);
}

// ------------------------------------------------------------------ packing

// Row of the natural (E, R, K) tensor that lands at packed row `row` (of
// expert e = row / R): the same row, or with two interleaved sections
// (rows 2j, 2j+1 = section 0 and 1 of index j) the row that section layout
// puts there.
__device__ __forceinline__ long long natural_row(long long row, int R, int interleaved) {
  if (!interleaved) return row;
  const long long e = row / R;
  const int r = static_cast<int>(row - e * R);
  const int half = R / 2;
  return e * R + (r < half ? 2 * r : 2 * (r - half) + 1);
}

// Packed values, tile-major: byte 64 r + b of tile (e, weight tile nt, K
// tile kt) holds natural bytes 64 kt + b (K elements 128 kt + 2b and 2b + 1)
// of tile row r: for two sections (w13) gate row 96 nt + r (r < 96) or up
// row 96 nt + r - 96, for one section (w2) row 192 nt + r; zero past the
// section's rows or past K; interleaved gate/up rows are put in halves.  One
// tile is 192 x 64 bytes.
__global__ void pack_values_kernel(const uint8_t* __restrict__ w, int E, int R, int K,
                                   int sections, int n_tiles, int kp_tiles, int interleaved,
                                   uint8_t* __restrict__ out) {
  const int in_pitch = K / 2;
  const int rows_per_sec = R / sections;
  const int span = 192 / sections;  // rows of one section in a tile
  const long long n = static_cast<long long>(E) * n_tiles * kp_tiles * 192 * 64;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int b = static_cast<int>(i & 63);
    long long t = i >> 6;
    const int r = static_cast<int>(t % 192);
    t /= 192;
    const int kt = static_cast<int>(t % kp_tiles);
    t /= kp_tiles;
    const int nt = static_cast<int>(t % n_tiles);
    const int e = static_cast<int>(t / n_tiles);
    const int sec = r / span;
    const int srow = span * nt + r % span;
    const int col = 64 * kt + b;
    uint8_t v = 0;
    if (srow < rows_per_sec && col < in_pitch) {
      const long long row = natural_row(static_cast<long long>(e) * R + sec * rows_per_sec + srow,
                                        R, interleaved);
      v = w[row * in_pitch + col];
    }
    out[i] = v;
  }
}

// Scale images, one of 1 KB per (expert, weight tile, K tile): byte
// 512 p + 16 l + 4 c + b is the scale of tile row 128 p + 32 c + l, K block
// 4 kt + b, else 127.  Tile row r of weight tile t is, for two sections
// (w13), row 96 t + r of the gate rows (r < 96) or row 96 t + r - 96 of the
// up rows, and for one section (w2) row 192 t + r; rows past the section's
// end and tile rows 192-255 are unit scales.
__global__ void pack_scales_kernel(const uint8_t* __restrict__ sc, int E, int R, int K,
                                   int sections, int n_tiles, int kp_tiles, int interleaved,
                                   uint8_t* __restrict__ out) {
  const int nblk = K / 32;
  const int rows_per_sec = R / sections;
  const int span = 192 / sections;  // rows of one section in a tile
  const long long n = static_cast<long long>(E) * n_tiles * kp_tiles * 1024;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int byte = static_cast<int>(i & 1023);
    long long img = i >> 10;
    const int kt = static_cast<int>(img % kp_tiles);
    img /= kp_tiles;
    const int t = static_cast<int>(img % n_tiles);
    const int e = static_cast<int>(img / n_tiles);
    const int p = byte >> 9, l = (byte >> 4) & 31, c = (byte >> 2) & 3, b = byte & 3;
    const int tr = 128 * p + 32 * c + l;
    const int sec = tr / span;
    const int srow = span * t + tr % span;
    const int blk = 4 * kt + b;
    uint8_t v = 127;
    if (tr < 192 && srow < rows_per_sec && blk < nblk) {
      const long long row = natural_row(static_cast<long long>(e) * R + sec * rows_per_sec + srow,
                                        R, interleaved);
      v = sc[row * nblk + blk];
    }
    out[i] = v;
  }
}

}  // namespace

cudaError_t launch_mx_gate_up(const MxArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmA64,
                              const CUtensorMap& tmW, int grid, cudaStream_t s) {
  return launch<kMxGateUp>(a, tmA, tmA64, tmW, grid, s);
}

cudaError_t launch_mx_down(const MxArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmA64,
                           const CUtensorMap& tmW, int grid, cudaStream_t s) {
  return launch<kMxDown>(a, tmA, tmA64, tmW, grid, s);
}

cudaError_t launch_pack_mx(const uint8_t* w, const uint8_t* w_scale, int E, int R, int K,
                           int sections, int interleaved, uint8_t* w_packed, uint8_t* s_packed,
                           cudaStream_t s) {
  const int Kp = (K + 127) / 128 * 128;
  pack_values_kernel<<<1184, 256, 0, s>>>(w, E, R, K, sections, mx_weight_tiles(R, sections),
                                          Kp / 128, interleaved, w_packed);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  pack_scales_kernel<<<1184, 256, 0, s>>>(w_scale, E, R, K, sections,
                                          mx_weight_tiles(R, sections), Kp / 128, interleaved,
                                          s_packed);
  return cudaGetLastError();
}

}  // namespace moe
