// gemm_mx.cu -- the two grouped GEMMs of the low-precision MoE expert FFN:
// fp8 (e4m3) activations times mxfp4 weights (e2m1 values, one e8m0 scale per
// 32 K elements), tcgen05 block-scaled MMAs (kind::mxf8f6f4) on sm_103a.
//
// Sources: "MOE Bmm1 Fused Gather" -- mma_partition issues block-scaled MMAs
// of e2m1 weights against e4m3 activations with the weight scales copied into
// tensor memory before each MMA, and ws_matmul_kernel fills the activation
// scale tensor with the e8m0 code 127 (unit scales; here the per-row fp8 scale
// of x is applied in the epilogue instead); pack_e4m3x2 (fp32 -> e4m3, round
// to nearest even, saturating) for the hidden activation.  The SiLU*up and
// routing-weight epilogues are those of gemm.cu.
//
// Layout per CTA (one per SM, persistent, bands of N tiles as in gemm.cu):
//  * tile = 128 sorted rows x 192 weight rows, as two MMAs of N = 96:
//    gate/up: 96 gate rows and the matching 96 up rows of w13[e];
//    down: 192 rows of w2[e];
//  * 5 shared-memory stages of 40 KB, 128 K elements each: A = 128 rows of
//    e4m3 (128 B, 128-byte swizzled K-major), B = 192 rows of e2m1 in the
//    padded form the block-scaled MMA reads 4-bit operands in (16 values =
//    8 packed bytes at the start of each 16-byte slot, the other 8 bytes
//    zero), swizzled the same way;
//  * producer warps 0-3 fill a stage with cp.async (16-byte chunks of A --
//    gathered token rows for gate/up, contiguous h rows for down -- and
//    8-byte packed chunks of B straight from the weights' natural packed
//    layout; the ragged end of K is zero-filled), and write the stage's B
//    scale factors (fetched one stage ahead) into tensor memory with
//    tcgen05.st; they publish the stage (proxy fence, tcgen05 fence, mbarrier
//    arrive) once the copies of kStages - 2 later stages are issued;
//  * warp 4 issues the MMAs from one thread; warps 5-8 run the epilogue;
//  * tensor memory: two 192-column fp32 accumulators, 4 columns of unit A
//    scales, and per stage and MMA half 4 columns of B scales.
//
// Scale factors in tensor memory: one 32-bit word per lane and column holds
// the scales of 4 consecutive 32-element K blocks of one row (byte j = block
// j, chosen per MMA by the instruction descriptor's scale ids); the rows of a
// 128-row scale matrix are spread over 4 columns, column c of lane l holding
// row 32c + l, and the same words are written into each of the 4 lane
// quarters so that every quarter of the tensor core reads all of them.
//
// All waits are bounded as in gemm.cu.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "sched.cuh"

namespace moe {
namespace {

enum MxKind { kMxGateUp = 0, kMxDown = 1 };

struct MxCfg {
  static constexpr int kBM = kBlockM;                 // 128 sorted rows
  static constexpr int kHalf = 96;                    // weight rows per MMA
  static constexpr int kBN = 2 * kHalf;               // weight rows per tile
  static constexpr int kRowBytes = 128;
  static constexpr int kBK = 128;                     // K elements per stage
  static constexpr int kUmmaK = 32;                   // K per MMA (one scale block)
  static constexpr int kStages = 5;
  static constexpr int kABytes = kBM * kRowBytes;     // 16 KB
  static constexpr int kBBytes = kBN * kRowBytes;     // 24 KB
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kAccCols = kBN;                // 192 fp32 columns
  static constexpr int kSfaCol = 2 * kAccCols;        // 384: unit A scales (4 columns)
  static constexpr int kSfbCol0 = kSfaCol + 4;        // 388: B scales, 4 columns per stage/half
  static constexpr int kTmemCols = 512;
  static constexpr int kProducerWarps = 4;
  static constexpr int kMmaWarp = kProducerWarps;
  static constexpr int kThreads = (kProducerWarps + 1 + 4) * 32;
  // a producer thread publishes stage n once stage n + kLag is issued; the lag
  // leaves one stage of slack so that n is published while the tensor core
  // still works on n - 1
  static constexpr int kLag = kStages - 2;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024;
  static constexpr uint32_t kIdesc = make_idesc_mx_e4m3_e2m1(kBM, kHalf);
};
static_assert(MxCfg::kSfbCol0 + MxCfg::kStages * 2 * 4 <= MxCfg::kTmemCols, "TMEM budget");
static_assert(MxCfg::kLag < MxCfg::kStages, "publication lag must stay inside the ring");

__device__ __forceinline__ uint32_t sfb_col(int stage, int half) {
  return MxCfg::kSfbCol0 + (stage * 2 + half) * 4;
}

// Scales of K blocks 4*kt .. 4*kt+3 of one weight row, one byte each
// (blocks past the row's end read as 127, a unit scale; their values are 0).
// Rows of an even number of blocks are read as two 16-bit words.
__device__ __forceinline__ uint32_t scale_word(const uint8_t* srow, int kt, int nblocks) {
  const int b0 = kt * 4;
  if ((nblocks & 1) == 0 && b0 + 4 <= nblocks) {
    const uint16_t* p = reinterpret_cast<const uint16_t*>(srow + b0);
    return static_cast<uint32_t>(__ldg(p)) | (static_cast<uint32_t>(__ldg(p + 1)) << 16);
  }
  uint32_t w = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const int blk = b0 + b;
    const uint32_t v = blk < nblocks ? static_cast<uint32_t>(__ldg(srow + blk)) : 127u;
    w |= v << (8 * b);
  }
  return w;
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  return g / (1.0f + __expf(-g)) * u;
}

template <int KIND>
__global__ void __launch_bounds__(MxCfg::kThreads, 1) mx_gemm_kernel(const __grid_constant__ MxArgs a) {
  using C = MxCfg;
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
      mbar_init(smem_u32(&full_bar[i]), C::kProducerWarps * 32);
      mbar_init(smem_u32(&empty_bar[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&accf_bar[i]), 1);
      mbar_init(smem_u32(&acce_bar[i]), 128);
    }
    mbar_init(smem_u32(&drain_bar), 1);
    fence_barrier_init();
  }
  // the padding half of every 16-byte slot of the B stages stays zero: the
  // copies below only ever write the first 8 bytes of a slot
  {
    uint4* b = reinterpret_cast<uint4*>(smem_raw + (smemB - smem_u32(smem_raw)));
    for (int i = threadIdx.x; i < C::kStages * C::kBBytes / 16; i += blockDim.x)
      b[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  fence_proxy_async_smem();
  __syncthreads();
  if (s_skip) return;
  if (warp == C::kMmaWarp) tmem_alloc(smem_u32(&s_tmem_base), C::kTmemCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = s_tmem_base;
  if (warp < C::kProducerWarps) {  // unit activation scales, every lane quarter
    tmem_st4(tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + C::kSfaCol, 0x7F7F7F7Fu,
             0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
    tmem_wait_st();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();

  const int num_blocks = *a.num_blocks;
  const int total = num_blocks * a.n_tiles * a.splits;
  const uint64_t to = a.timeout_ns;
  const int nblocks_k = a.Kdim / 32;  // scale blocks per weight row
  const long long wpitch = a.Kdim / 2;

  if (warp < C::kProducerWarps) {
    // ------------------------------------------------------------ producer
    const int pt = threadIdx.x;      // 0..127
    const int ch = pt & 7;           // chunk of the 128-element k-tile (16 elements)
    const int rb = pt >> 3;          // rows rb + 16 j
    const uint32_t sf_lane = static_cast<uint32_t>(warp * 32) << 16;
    uint32_t stage = 0, phase = 0;
    long long issued = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const Tile t = decode_tile(tile, num_blocks, a);
      const int4 bi = reinterpret_cast<const int4*>(a.block_info)[t.mb];
      const int e = bi.x, r0 = bi.z, valid = bi.w;
      int kb, ke;
      split_range(a, t.split, kb, ke);
      const uint8_t* arow[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int r = rb + 16 * j;
        if constexpr (KIND == kMxGateUp) {
          const int tok = r < valid ? a.sorted_ids[r0 + r] / a.K : 0;
          arow[j] = a.a + static_cast<long long>(tok) * a.H;
        } else {
          arow[j] = a.a + static_cast<long long>(r0 + r) * a.I;
        }
      }
      // weight row of tile row n (0..191); rows past the expert's end are
      // clamped to its last row (their products are never stored)
      auto wrow_of = [&](int n) -> long long {
        if constexpr (KIND == kMxGateUp) {
          const int h = n >= C::kHalf ? 1 : 0;
          const int jj = min(t.nt * C::kHalf + (n - h * C::kHalf), a.I - 1);
          return static_cast<long long>(e) * 2 * a.I + h * a.I + jj;
        } else {
          return static_cast<long long>(e) * a.H + min(t.nt * C::kBN + n, a.H - 1);
        }
      };
      const uint8_t* brow[12];
#pragma unroll
      for (int j = 0; j < 12; ++j) brow[j] = a.w + wrow_of(rb + 16 * j) * wpitch;
      const uint8_t* srow[2][3];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int c = 0; c < 3; ++c)
          srow[h][c] = a.w_scale + wrow_of(h * C::kHalf + 32 * c + lane) * nblocks_k;

      // scale words of the next stage are fetched one stage ahead
      uint32_t sw[2][3];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int c = 0; c < 3; ++c) sw[h][c] = kb < ke ? scale_word(srow[h][c], kb, nblocks_k) : 0u;

      for (int kt = kb; kt < ke; ++kt) {
        if (!mbar_wait_bounded(smem_u32(&empty_bar[stage]), phase ^ 1, &s_abort, to)) {
          ok = false;
          break;
        }
        const uint32_t a_dst = smemA + stage * C::kABytes;
        const uint32_t b_dst = smemB + stage * C::kBBytes;
        const int ka = kt * C::kBK + ch * 16;
        const bool in_k = ka < a.Kdim;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int r = rb + 16 * j;
          cp_async_16_zfill(a_dst + r * C::kRowBytes + ((ch ^ (r & 7)) << 4),
                            in_k ? arow[j] + ka : arow[j], in_k ? 16u : 0u);
        }
#pragma unroll
        for (int j = 0; j < 12; ++j) {
          const int n = rb + 16 * j;
          cp_async_8_zfill(b_dst + n * C::kRowBytes + ((ch ^ (n & 7)) << 4),
                           in_k ? brow[j] + ka / 2 : brow[j], in_k ? 8u : 0u);
        }
        cp_async_commit();
#pragma unroll
        for (int h = 0; h < 2; ++h)
          tmem_st4(tmem_base + sf_lane + sfb_col(stage, h), sw[h][0], sw[h][1], sw[h][2],
                   0x7F7F7F7Fu);
        tmem_wait_st();
        if (kt + 1 < ke) {
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int c = 0; c < 3; ++c) sw[h][c] = scale_word(srow[h][c], kt + 1, nblocks_k);
        }
        ++issued;
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1;
        }
        if (issued > C::kLag) {
          cp_async_wait<C::kLag>();
          fence_proxy_async_smem();
          tc_fence_before_sync();
          const long long n = issued - 1 - C::kLag;
          mbar_arrive(smem_u32(&full_bar[n % C::kStages]));
        }
      }
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    tc_fence_before_sync();
    for (long long n = issued > C::kLag ? issued - C::kLag : 0; n < issued; ++n)
      mbar_arrive(smem_u32(&full_bar[n % C::kStages]));
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
#pragma unroll
          for (int k = 0; k < C::kBK / C::kUmmaK; ++k) {
            const uint64_t ad = sw128_kmajor_desc(a_base + k * 32);
            const uint32_t idesc = idesc_with_sf_ids(C::kIdesc, k, k);
            const uint32_t accum = (kt > kb || k > 0) ? 1u : 0u;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint64_t bd =
                  sw128_kmajor_desc(b_base + h * C::kHalf * C::kRowBytes + k * 32);
              umma_mxf8f6f4(d_tmem + h * C::kHalf, ad, bd, idesc, sfa,
                            tmem_base + sfb_col(stage, h), accum);
            }
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
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const Tile t = decode_tile(tile, num_blocks, a);
      const int4 bi = reinterpret_cast<const int4*>(a.block_info)[t.mb];
      const int r0 = bi.z, valid = bi.w;
      const bool row_ok = r < valid;
      float rs = 0.0f;
      if (row_ok) {
        const int i = a.sorted_ids[r0 + r];
        if constexpr (KIND == kMxGateUp)
          rs = a.x_row_scale[i / a.K];
        else
          rs = a.topk_weights[i] * a.h_scale;
      }
      int good = 1;
      if (lane == 0) good = mbar_wait_bounded(smem_u32(&accf_bar[acc]), acc_phase, &s_abort, to);
      good = __shfl_sync(0xffffffffu, good, 0);
      if (!good) break;
      tc_fence_after_sync();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * C::kAccCols;
      if constexpr (KIND == kMxGateUp) {
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
                const float gg = rs * __uint_as_float(g[4 * v + w]);
                const float uu = rs * __uint_as_float(u[4 * v + w]);
                o[w] = __fdiv_rn(silu_mul(gg, uu), a.h_scale);
              }
              pk[v] = e4m3x4(o[0], o[1], o[2], o[3]);
            }
            uint4* dst = reinterpret_cast<uint4*>(hq + j0);
            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      } else {
        float* y = static_cast<float*>(a.out) +
                   (static_cast<long long>(t.split) * a.cap + r0 + r) * a.H;
#pragma unroll 1
        for (int c = 0; c < 6; ++c) {
          uint32_t v[32];
          tmem_ld32(taddr + c * 32, v);
          tmem_wait_ld();
          const int col0 = t.nt * C::kBN + c * 32;
          if (row_ok && col0 < a.H) {
            float4* dst = reinterpret_cast<float4*>(y + col0);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(rs * __uint_as_float(v[4 * i + 0]), rs * __uint_as_float(v[4 * i + 1]),
                                   rs * __uint_as_float(v[4 * i + 2]), rs * __uint_as_float(v[4 * i + 3]));
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
cudaError_t launch(const MxArgs& a, int grid, cudaStream_t s) {
  auto kern = mx_gemm_kernel<KIND>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         MxCfg::kSmemBytes);
  if (err != cudaSuccess) return err;
  kern<<<grid, MxCfg::kThreads, MxCfg::kSmemBytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mx_gate_up(const MxArgs& a, int grid, cudaStream_t s) {
  return launch<kMxGateUp>(a, grid, s);
}

cudaError_t launch_mx_down(const MxArgs& a, int grid, cudaStream_t s) {
  return launch<kMxDown>(a, grid, s);
}

}  // namespace moe
