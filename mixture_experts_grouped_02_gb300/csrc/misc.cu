// misc.cu -- the bandwidth-bound stages: the deterministic per-token combine
// and the per-row fp8 (e4m3) activation step.
#include <cuda_bf16.h>

#include <algorithm>

#include "bounds.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

// out[t, :] = sum_k sum_q y[q, inv_perm[t*K + k], :], fp32 in k order, then
// one rounding to the output type.  A negative slot (an assignment to an
// expert another shard holds) adds nothing.  Source: the index_add of the "Current
// PyTorch path" in "factor_moe_fused_gemm.cu" and its
// weighted_scatter_add_kernel, made deterministic: each token owns its row,
// so no atomics and a fixed summation order.  CTA (x, y) handles groups of
// TPC token rows x*TPC, (x + gridDim.x)*TPC, ... and the y-th run of 1024
// columns of them, so that a handful of tokens still spreads over many SMs;
// 16-byte loads of y.  With one split, a thread issues the loads of all
// TPC*K <= 8 assignments of its group before it sums any (TPC = 4 tokens for
// top-2, 2 for top-3/4, 1 above), which keeps enough bytes in flight when K
// is small.
constexpr int kCombineBatch = 8;

template <typename OutT>
__device__ __forceinline__ void store_out4(OutT* row, int c, float4 acc) {
  if constexpr (sizeof(OutT) == 2) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&lo);
    pk.y = *reinterpret_cast<uint32_t*>(&hi);
    reinterpret_cast<uint2*>(row)[c] = pk;
  } else {
    reinterpret_cast<float4*>(row)[c] = acc;
  }
}

__device__ __forceinline__ void add4(float4& acc, const float4 v) {
  acc.x += v.x;
  acc.y += v.y;
  acc.z += v.z;
  acc.w += v.w;
}

// One split, K <= kCombineBatch / TPC: the loads of the group's TPC tokens
// all in flight, then each token's sum in k order.
template <typename OutT, int TPC>
__device__ __forceinline__ void combine_group(const float* __restrict__ y,
                                              const int32_t* __restrict__ inv_perm, int T, int K,
                                              int H, int t0, int c, OutT* __restrict__ out,
                                              long long cap, const int32_t* status) {
  constexpr int KM = kCombineBatch / TPC;
  float4 v[TPC][KM];
  unsigned live = 0;  // bit u*KM + k: assignment k of token t0 + u has a slot here
#pragma unroll
  for (int u = 0; u < TPC; ++u)
#pragma unroll
    for (int k = 0; k < KM; ++k)
      if (k < K && t0 + u < T) {
        const int sl = inv_perm[static_cast<long long>(t0 + u) * K + k];
        if (sl >= 0 && in_bounds(sl < cap, status)) {
          v[u][k] = __ldg(reinterpret_cast<const float4*>(y + static_cast<long long>(sl) * H) + c);
          live |= 1u << (u * KM + k);
        }
      }
#pragma unroll
  for (int u = 0; u < TPC; ++u) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < KM; ++k)
      if ((live >> (u * KM + k)) & 1u) add4(acc, v[u][k]);
    if (t0 + u < T) store_out4(out + static_cast<long long>(t0 + u) * H, c, acc);
  }
}

// TPC > 1 is launched only with one split and K <= kCombineBatch / TPC.
template <typename OutT, int TPC>
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y, int splits,
                                                      long long cap,
                                                      const int32_t* __restrict__ inv_perm, int T,
                                                      int K, int H, OutT* __restrict__ out,
                                                      const int32_t* status) {
  pdl_wait();
  pdl_launch_dependents();
  if (status != nullptr && *status != 0) return;
  const int h4 = H >> 2;
  const int c_end = min(h4, static_cast<int>(blockIdx.y + 1) * 256);
  for (int t0 = blockIdx.x * TPC; t0 < T; t0 += gridDim.x * TPC) {
    for (int c = blockIdx.y * 256 + threadIdx.x; c < c_end; c += blockDim.x) {
      if constexpr (TPC > 1) {
        combine_group<OutT, TPC>(y, inv_perm, T, K, H, t0, c, out, cap, status);
      } else if (splits == 1 && K <= kCombineBatch) {
        combine_group<OutT, 1>(y, inv_perm, T, K, H, t0, c, out, cap, status);
      } else {
        // the splits of each assignment four loads at a time, added in
        // split order (the decode shapes run up to 19 splits)
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k = 0; k < K; ++k) {
          const long long row = inv_perm[static_cast<long long>(t0) * K + k];
          if (row < 0 || !in_bounds(row < cap, status)) continue;
          const float4* col = reinterpret_cast<const float4*>(y + row * H) + c;
          const long long plane = cap * (H >> 2);  // float4s between splits
          for (int q = 0; q < splits; q += 4) {
            float4 v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (q + j < splits) v[j] = __ldg(col + (q + j) * plane);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (q + j < splits) add4(acc, v[j]);
          }
        }
        store_out4(out + static_cast<long long>(t0) * H, c, acc);
      }
    }
  }
}

__device__ __forceinline__ float load_act(const void* x, int bf16, long long idx) {
  if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(x)[idx]);
  return reinterpret_cast<const float*>(x)[idx];
}

// Per-row e4m3 quantisation: s_t = amax_t / 448 (1 for an all-zero row),
// xq = cvt.rn.satfinite.e4m3(x / s_t), both in fp32 with IEEE rounding.
// Source: "MOE Bmm1 Fused Gather", pack_e4m3x2 (the same conversion
// instruction); one scale per row is this workload's reading.
__global__ void __launch_bounds__(256) quantize_x_kernel(const void* __restrict__ x, int bf16,
                                                         int T, int H, uint8_t* __restrict__ xq,
                                                         float* __restrict__ row_scale) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float s_red[8];
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    const long long base = static_cast<long long>(t) * H;
    float amax = 0.0f;
    for (int c = threadIdx.x; c < H; c += blockDim.x) amax = fmaxf(amax, fabsf(load_act(x, bf16, base + c)));
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = s_red[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) amax = fmaxf(amax, s_red[w]);
    const float s = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    if (threadIdx.x == 0) row_scale[t] = s;
    for (int c = 2 * threadIdx.x; c < H; c += 2 * blockDim.x) {
      const float v0 = __fdiv_rn(load_act(x, bf16, base + c), s);
      const float v1 = __fdiv_rn(load_act(x, bf16, base + c + 1), s);
      uint16_t pk;
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pk) : "f"(v1), "f"(v0));
      *reinterpret_cast<uint16_t*>(xq + base + c) = pk;
    }
    __syncthreads();
  }
}

// The same quantisation, with each token's codes written to every slot of the
// expert-sorted list the token occupies (xq_sorted[inv_perm[t*K + k]]), so that
// the block-scaled gate/up GEMM reads contiguous rows: the token gather is
// fused into this pass, which reads every row of x anyway.  Negative slots
// (another shard's experts) are skipped.
__global__ void __launch_bounds__(256) quantize_gather_x_kernel(
    const void* __restrict__ x, int bf16, int T, int H, int K, const int32_t* __restrict__ inv_perm,
    uint8_t* __restrict__ xq_sorted, float* __restrict__ row_scale, float4* __restrict__ acc_zero,
    const int32_t* status, long long cap) {
  pdl_wait();
  pdl_launch_dependents();
  if (status != nullptr && *status != 0) return;
  __shared__ float s_red[8];
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    const long long base = static_cast<long long>(t) * H;
    if (acc_zero != nullptr)  // the fused combine's accumulator row of this token
      for (int c = threadIdx.x; c < (H >> 2); c += blockDim.x)
        acc_zero[(base >> 2) + c] = make_float4(0.f, 0.f, 0.f, 0.f);
    float amax = 0.0f;
    for (int c = threadIdx.x; c < H; c += blockDim.x) amax = fmaxf(amax, fabsf(load_act(x, bf16, base + c)));
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = s_red[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) amax = fmaxf(amax, s_red[w]);
    const float s = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    if (threadIdx.x == 0) row_scale[t] = s;
    for (int c = 2 * threadIdx.x; c < H; c += 2 * blockDim.x) {
      const float v0 = __fdiv_rn(load_act(x, bf16, base + c), s);
      const float v1 = __fdiv_rn(load_act(x, bf16, base + c + 1), s);
      uint16_t pk;
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pk) : "f"(v1), "f"(v0));
      for (int k = 0; k < K; ++k) {
        const long long slot = inv_perm[static_cast<long long>(t) * K + k];
        if (slot >= 0 && in_bounds(slot < cap, status))
          *reinterpret_cast<uint16_t*>(xq_sorted + slot * H + c) = pk;
      }
    }
    __syncthreads();
  }
}

// 16 consecutive activations of a row as fp32 (two or four 16-byte loads).
template <bool BF16>
__device__ __forceinline__ void load16(const void* x, long long idx, float (&v)[16]) {
  if constexpr (BF16) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(x) + idx);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 q = p[h];
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[8 * h + 2 * i] = __uint_as_float(w[i] << 16);
        v[8 * h + 2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
      }
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(x) + idx);
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const float4 q = p[h];
      v[4 * h] = q.x;
      v[4 * h + 1] = q.y;
      v[4 * h + 2] = q.z;
      v[4 * h + 3] = q.w;
    }
  }
}

// quantize_gather_x_kernel for rows of a multiple of 16 elements with x and
// xq_sorted 16-byte aligned: a thread takes runs of 16 elements (16-byte
// loads) and writes their 16 codes with one 16-byte store per slot of the
// token.  Every code is computed exactly as in the general kernel.
template <bool BF16>
__global__ void __launch_bounds__(256) quantize_gather_x16_kernel(
    const void* __restrict__ x, int T, int H, int K, const int32_t* __restrict__ inv_perm,
    uint8_t* __restrict__ xq_sorted, float* __restrict__ row_scale, float4* __restrict__ acc_zero,
    const int32_t* status, long long cap) {
  pdl_wait();
  pdl_launch_dependents();
  if (status != nullptr && *status != 0) return;
  __shared__ float s_red[8];
  const int runs = H >> 4;
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    const long long base = static_cast<long long>(t) * H;
    if (acc_zero != nullptr)  // the fused combine's accumulator row of this token
      for (int c = threadIdx.x; c < (H >> 2); c += blockDim.x)
        acc_zero[(base >> 2) + c] = make_float4(0.f, 0.f, 0.f, 0.f);
    float amax = 0.0f;
    for (int r = threadIdx.x; r < runs; r += blockDim.x) {
      float v[16];
      load16<BF16>(x, base + 16 * r, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = s_red[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) amax = fmaxf(amax, s_red[w]);
    const float s = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    if (threadIdx.x == 0) row_scale[t] = s;
    for (int r = threadIdx.x; r < runs; r += blockDim.x) {
      float v[16];
      load16<BF16>(x, base + 16 * r, v);
      uint32_t pk[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint16_t h;
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
            : "=h"(h)
            : "f"(__fdiv_rn(v[2 * i + 1], s)), "f"(__fdiv_rn(v[2 * i], s)));
        pk[i] = h;
      }
      const uint4 q = make_uint4(pk[0] | (pk[1] << 16), pk[2] | (pk[3] << 16),
                                 pk[4] | (pk[5] << 16), pk[6] | (pk[7] << 16));
      for (int k = 0; k < K; ++k) {
        const long long slot = inv_perm[static_cast<long long>(t) * K + k];
        if (slot >= 0 && in_bounds(slot < cap, status))
          *reinterpret_cast<uint4*>(xq_sorted + slot * H + 16 * r) = q;
      }
    }
    __syncthreads();
  }
}

// Token rows to sorted slots: xs[inv_perm[t*K + k], :] = x[t, :] for every
// choice k of token t (rows of padding slots untouched).  The gather of the
// gate/up GEMM done as its own pass, for the CTA-pair GEMMs whose A operand
// then arrives by plain TMA tiles.  16-byte copies; a CTA per token row;
// negative slots (another shard's experts) are skipped.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x,
                                                          int T, int row_vec, int K,
                                                          const int32_t* __restrict__ inv_perm,
                                                          uint4* __restrict__ xs,
                                                          float4* __restrict__ acc_zero,
                                                          int acc_vec, const int32_t* status,
                                                          long long cap) {
  pdl_wait();
  pdl_launch_dependents();
  if (status != nullptr && *status != 0) return;
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    if (acc_zero != nullptr)  // the fused combine's accumulator row of this token
      for (int c = threadIdx.x; c < acc_vec; c += blockDim.x)
        acc_zero[static_cast<long long>(t) * acc_vec + c] = make_float4(0.f, 0.f, 0.f, 0.f);
    const uint4* src = x + static_cast<long long>(t) * row_vec;
    for (int c = threadIdx.x; c < row_vec; c += blockDim.x) {
      const uint4 v = __ldg(src + c);
      for (int k = 0; k < K; ++k) {
        const long long slot = inv_perm[static_cast<long long>(t) * K + k];
        if (slot >= 0 && in_bounds(slot < cap, status)) xs[slot * row_vec + c] = v;
      }
    }
  }
}

// out = acc rounded once to the output type, 4 columns per thread.  Source:
// the final cast of the scatter-add path of "factor_moe_fused_gemm.cu"
// (fp32 accumulation, then the model dtype).
template <typename OutT>
__global__ void __launch_bounds__(256) combine_finish_kernel(const float4* __restrict__ acc,
                                                             long long n4, OutT* __restrict__ out,
                                                             const int32_t* status) {
  pdl_wait();
  pdl_launch_dependents();
  if (status != nullptr && *status != 0) return;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    store_out4(out + 4 * i, 0, __ldg(acc + i));
}

}  // namespace

cudaError_t launch_gather_rows(const void* x, int T, int row_bytes, int K, const int32_t* inv_perm,
                               void* xs, float* acc_zero, int H, const int32_t* status,
                               cudaStream_t s, long long cap) {
  const int grid = T < 65535 ? T : 65535;
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = pdl_config(dim3(grid), dim3(256), 0, s, attr);
  return cudaLaunchKernelEx(&cfg, gather_rows_kernel, static_cast<const uint4*>(x), T,
                            row_bytes / 16, K, inv_perm, static_cast<uint4*>(xs),
                            reinterpret_cast<float4*>(acc_zero), H / 4, status, cap);
}

cudaError_t launch_quantize_gather_x(const void* x, int x_dtype, int T, int H, int K,
                                     const int32_t* inv_perm, uint8_t* xq_sorted,
                                     float* row_scale, float* acc_zero, const int32_t* status,
                                     cudaStream_t s, long long cap) {
  const int grid = T < 65535 ? T : 65535;
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = pdl_config(dim3(grid), dim3(256), 0, s, attr);
  float4* acc4 = reinterpret_cast<float4*>(acc_zero);
  const bool vec = H % 16 == 0 && (reinterpret_cast<uintptr_t>(x) & 15u) == 0 &&
                   (reinterpret_cast<uintptr_t>(xq_sorted) & 15u) == 0;
  if (vec && x_dtype == MOE_BF16)
    return cudaLaunchKernelEx(&cfg, quantize_gather_x16_kernel<true>, x, T, H, K, inv_perm,
                              xq_sorted, row_scale, acc4, status, cap);
  if (vec)
    return cudaLaunchKernelEx(&cfg, quantize_gather_x16_kernel<false>, x, T, H, K, inv_perm,
                              xq_sorted, row_scale, acc4, status, cap);
  return cudaLaunchKernelEx(&cfg, quantize_gather_x_kernel, x, x_dtype == MOE_BF16 ? 1 : 0, T, H,
                            K, inv_perm, xq_sorted, row_scale, acc4, status, cap);
}

cudaError_t launch_combine_finish(const float* acc, int T, int H, int out_dtype, void* out,
                                  const int32_t* status, cudaStream_t s) {
  const long long n4 = static_cast<long long>(T) * (H / 4);
  const int grid = static_cast<int>(std::min<long long>((n4 + 255) / 256, 152ll * 16));
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = pdl_config(dim3(grid), dim3(256), 0, s, attr);
  const float4* a4 = reinterpret_cast<const float4*>(acc);
  if (out_dtype == MOE_BF16)
    return cudaLaunchKernelEx(&cfg, combine_finish_kernel<__nv_bfloat16>, a4, n4,
                              static_cast<__nv_bfloat16*>(out), status);
  return cudaLaunchKernelEx(&cfg, combine_finish_kernel<float>, a4, n4, static_cast<float*>(out),
                            status);
}

cudaError_t launch_combine(const float* y, int splits, long long cap, const int32_t* inv_perm,
                           int T, int K, int H, int out_dtype, void* out, int32_t* status,
                           cudaStream_t s) {
  // tokens per group: all loads of a group in flight at once (one split)
  const int tpc = splits != 1 ? 1 : K <= 1 ? 8 : K <= 2 ? 4 : K <= 4 ? 2 : 1;
  const int groups = (T + tpc - 1) / tpc;
  const dim3 grid(groups < 65535 ? groups : 65535, (H / 4 + 255) / 256);
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = pdl_config(grid, dim3(256), 0, s, attr);
  const int32_t* st = static_cast<const int32_t*>(status);
  if (out_dtype == MOE_BF16) {
    using bf16 = __nv_bfloat16;
    bf16* o = reinterpret_cast<bf16*>(out);
    switch (tpc) {
      case 8: return cudaLaunchKernelEx(&cfg, combine_kernel<bf16, 8>, y, splits, cap, inv_perm, T, K, H, o, st);
      case 4: return cudaLaunchKernelEx(&cfg, combine_kernel<bf16, 4>, y, splits, cap, inv_perm, T, K, H, o, st);
      case 2: return cudaLaunchKernelEx(&cfg, combine_kernel<bf16, 2>, y, splits, cap, inv_perm, T, K, H, o, st);
      default: return cudaLaunchKernelEx(&cfg, combine_kernel<bf16, 1>, y, splits, cap, inv_perm, T, K, H, o, st);
    }
  }
  float* o = reinterpret_cast<float*>(out);
  switch (tpc) {
    case 8: return cudaLaunchKernelEx(&cfg, combine_kernel<float, 8>, y, splits, cap, inv_perm, T, K, H, o, st);
    case 4: return cudaLaunchKernelEx(&cfg, combine_kernel<float, 4>, y, splits, cap, inv_perm, T, K, H, o, st);
    case 2: return cudaLaunchKernelEx(&cfg, combine_kernel<float, 2>, y, splits, cap, inv_perm, T, K, H, o, st);
    default: return cudaLaunchKernelEx(&cfg, combine_kernel<float, 1>, y, splits, cap, inv_perm, T, K, H, o, st);
  }
}

cudaError_t launch_quantize_x(const void* x, int x_dtype, int T, int H, uint8_t* xq,
                              float* row_scale, cudaStream_t s) {
  const int grid = T < 65535 ? T : 65535;
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = pdl_config(dim3(grid), dim3(256), 0, s, attr);
  return cudaLaunchKernelEx(&cfg, quantize_x_kernel, x, x_dtype == MOE_BF16 ? 1 : 0, T, H, xq,
                            row_scale);
}

}  // namespace moe
