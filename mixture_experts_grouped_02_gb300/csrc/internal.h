// internal.h -- declarations shared by the library's translation units
// (kernel launchers and the C ABI in moe_abi.cu).  Not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/moe.h"

namespace moe {

// The argument checks moe_forward makes on a problem before any launch
// (shapes, dtypes, shard, epilogue, GEMM shape support): MOE_OK or the
// status moe_forward returns for it.
int validate_forward_problem(const moe_problem_t* p);

// Default wall-clock limit of any single pipeline wait inside a kernel.
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;

// Align blocks of the block-scaled GEMMs (their M tile), and the smaller of
// the two automatic block sizes of the bf16/fp32 GEMMs.
constexpr int kBlockM = 128;

// Launch configuration with programmatic stream serialisation: the kernel
// may be launched while the previous kernel of the stream is still running
// and waits for it in pdl_wait() (every kernel of the path does so before it
// reads anything an earlier kernel wrote).  cluster_x > 1 adds a cluster
// dimension.  `attr` must hold two entries and outlive the launch call.
inline cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                     cudaLaunchAttribute* attr, unsigned cluster_x = 1) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cfg;
}

// Activation and biases of the expert FFN (moe_problem_t).
struct Epilogue {
  int act;             // MOE_ACT_SILU / MOE_ACT_SWIGLU_CLAMP
  float alpha, limit;  // MOE_ACT_SWIGLU_CLAMP
  int interleaved;     // w13 rows and w13_bias entries: gate 2j, up 2j+1
  const float* b13;    // (L, 2I) or null
  const float* b2;     // (L, H) or null
};

// Row of gate j / up j of expert e in w13_bias.
__host__ __device__ inline long long gate_bias_index(const Epilogue& ep, int I, int e, int j) {
  return static_cast<long long>(e) * 2 * I + (ep.interleaved ? 2 * j : j);
}
__host__ __device__ inline long long up_bias_index(const Epilogue& ep, int I, int e, int j) {
  return static_cast<long long>(e) * 2 * I + (ep.interleaved ? 2 * j + 1 : I + j);
}

// Router logits of the routing step folded into align (moe_route_align).
struct RouteArgs {
  const void* logits;  // (T, E) fp32 or bf16, or null: the ids are given
  int bf16;            // logits are bf16
  int T, E, K;
  int32_t* ids;        // (T, K) out
  float* weights;      // (T, K) out
  int32_t* status;
};

struct AlignArgs {
  RouteArgs route;     // route.logits != null: route first, into `ids`
  const int32_t* ids;
  int n_assign;  // T*K
  int E;         // ids lie in [0, E)
  int e_base;    // first expert of this shard
  int e_local;   // experts of this shard (E when unsharded)
  int block_m;
  long long cap;
  int32_t* counts;
  int32_t* offsets;
  int32_t* padded_offsets;
  int32_t* sorted_ids;
  int32_t* inv_perm;
  int32_t* block_info;
  int32_t* num_blocks;
  int32_t* status;
};

// Arguments of one grouped-GEMM launch (both GEMMs).
struct GemmArgs {
  int T, H, I, E, K;
  int n_tiles;   // tiles along the output (N) dimension
  int k_tiles;   // 128-byte k-tiles over the whole reduction
  int splits;    // reduction splits (down projection); 1 for gate/up
  int band;      // N tiles per raster band
  long long cap; // rows of the padded sorted list
  const void* x;               // gate/up: token rows in sorted order (cap, H)
  const int32_t* sorted_ids;
  const int32_t* block_info;
  const int32_t* num_blocks;
  const float* topk_weights;  // down projection: routing weight per flat index
  void* out;                  // gate/up: h (cap, I); down: y (splits, cap, H) fp32, or
                              // the (T, H) fp32 accumulator when `fused`
  int fused;                  // down: add rows into the accumulator (atomics)
  int dual_small;             // tiles of at most 32 tokens load two K steps per stage
  int32_t* status;
  unsigned long long timeout_ns;
  int starve;                 // failure-path test: the producers issue no copies
  int n_held;                 // experts whose weights the call holds
  int max_blocks;             // entries of block_info (cap / block_m)
  Epilogue ep;
  int w_rows_per_expert;      // gate/up: rows of one expert in the gate weight map
  int up_row_offset;          // gate/up: up row j = gate row j + this (in the up map)
  int gather;                 // gate/up: token rows gathered from x (T rows) by sorted_ids
};

// Arguments of one block-scaled (fp8 activations x mxfp4 weights) grouped
// GEMM launch.  The reduction dimension is Kdim = H (gate/up) or I (down).
struct MxArgs {
  int T, H, I, E, K;
  int Kdim;
  int n_tiles, k_tiles, splits, band;
  long long cap;
  const uint8_t* a;            // gate/up: xq in sorted order (cap, H); down: hq (cap, I)
  const float* x_row_scale;    // gate/up: per-token fp32 scale of xq
  const uint8_t* w_scale;      // scale images (E, n_tiles, kp_tiles, 1 KB)
  int sections;                // 2 for w13 (gate rows, up rows), 1 for w2
  int kp_tiles;                // 128-element K tiles per padded weight row
  const int32_t* sorted_ids;
  const int32_t* block_info;
  const int32_t* num_blocks;
  const float* topk_weights;   // down: routing weight per flat index
  void* out;                   // gate/up: hq (cap, I) e4m3; down: y (splits, cap, H) fp32,
                               // or the (T, H) fp32 accumulator when `fused`
  int fused;                   // down: add rows into the accumulator (atomics)
  float h_scale;               // hq = e4m3(a / h_scale)
  int32_t* status;
  unsigned long long timeout_ns;
  int starve;                  // failure-path test: the producer issues no copies
  int n_held;                  // experts whose weights the call holds
  int max_blocks;              // entries of block_info (cap / 128)
  Epilogue ep;
};

// tmW: packed e2m1 values of w13 / w2, tile-major (E, weight tiles, K tiles)
// x 192 rows of 128 elements (64 bytes), box 128 x 192, expanded to 16-byte
// slots in shared memory.  tmA: the e4m3 A rows in sorted order, xq (cap x H bytes) for
// gate/up, hq (cap x I bytes) for down, box 128 x 128; tmA64: the same rows with
// a box of 128 x 64, loaded for blocks of at most 64 valid rows.
cudaError_t launch_mx_gate_up(const MxArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmA64,
                              const CUtensorMap& tmW, int grid, cudaStream_t s);
cudaError_t launch_mx_down(const MxArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmA64,
                           const CUtensorMap& tmW, int grid, cudaStream_t s);
cudaError_t launch_pack_mx(const uint8_t* w, const uint8_t* w_scale, int E, int R, int K,
                           int sections, int interleaved, uint8_t* w_packed, uint8_t* s_packed,
                           cudaStream_t s);

// 192-row weight tiles of an expert's R rows: 96 rows of each of two
// sections (w13: gate and up), or 192 rows of one (w2).  One scale image
// per tile and K tile.
inline int mx_weight_tiles(int R, int sections) {
  return sections == 2 ? (R / 2 + 95) / 96 : (R + 191) / 192;
}
inline int mx_padded_k(int K) { return (K + 127) / 128 * 128; }

cudaError_t launch_align(const AlignArgs& a, cudaStream_t s);
// The many-CTA align of large batches: CTAs of 8 warps, each warp counting a
// chunk of align_multi_chunk(n) ids; int32 scratch of per-warp counts
// whist[warps][e_local] and per-CTA totals ctot[ctas][e_local], then one
// scan CTA over the CTA totals, then the scatter.  Same outputs as
// launch_align (num_blocks is cleared with a memset first).
constexpr long long kAlignMultiMin = 16384;
int align_multi_chunk(long long n_assign);
int align_multi_warps(long long n_assign);
size_t align_multi_scratch_ints(long long n_assign, int e_local);
cudaError_t launch_align_multi(const AlignArgs& a, int32_t* scratch, cudaStream_t s);
// The routing step alone, a warp per token over many CTAs (large batches).
cudaError_t launch_route(const RouteArgs& r, cudaStream_t s);
// Largest batch whose routing the single-CTA align kernel does itself.
constexpr int kRouteInAlignMaxTokens = 1024;
cudaError_t launch_combine(const float* y, int splits, long long cap, const int32_t* inv_perm,
                           int T, int K, int H, int out_dtype, void* out, int32_t* status,
                           cudaStream_t s);
cudaError_t launch_quantize_x(const void* x, int x_dtype, int T, int H, uint8_t* xq,
                              float* row_scale, cudaStream_t s);
// acc_zero (nullable): rows of H fp32 of a fused combine's accumulator,
// set to zero for every token by the same CTAs.
// cap: rows of the sorted buffer (the checked build tests slots against it;
// kUnknownCap when the caller did not say).
constexpr long long kUnknownCap = 1ll << 62;
cudaError_t launch_gather_rows(const void* x, int T, int row_bytes, int K, const int32_t* inv_perm,
                               void* xs, float* acc_zero, int H, const int32_t* status,
                               cudaStream_t s, long long cap = kUnknownCap);
cudaError_t launch_quantize_gather_x(const void* x, int x_dtype, int T, int H, int K,
                                     const int32_t* inv_perm, uint8_t* xq_sorted,
                                     float* row_scale, float* acc_zero, const int32_t* status,
                                     cudaStream_t s, long long cap = kUnknownCap);
cudaError_t launch_combine_finish(const float* acc, int T, int H, int out_dtype, void* out,
                                  const int32_t* status, cudaStream_t s);

// Align blocks of 256 rows: the largest token tile of the bf16/fp32 GEMMs.
constexpr int kPairBlockM = 256;

// The bf16/fp32 grouped GEMMs on CTA pairs with the weights on the MMA's M
// side (gemm_wpair.cu); grid = 2 x clusters.  tmTok / tmTokS: token rows in sorted order (x for gate/up, h for down),
// boxes of 128 and 16 rows; tmW: w13 (box 64 rows) or w2 (box 128 rows).
int wpair_max_active(int kind, int dtype);
// tmWu: the map of the up rows (gate/up; the same map as tmW when w13 is in
// halves); unused by down.  tmX (gate/up with GemmArgs::gather): x as T rows
// of H elements, box 64 x 1 (bf16; 32 x 1 fp32), read by tile::gather4.
cudaError_t launch_wpair_gate_up(int dtype, const GemmArgs& a, const CUtensorMap& tmTok,
                                 const CUtensorMap& tmTokS, const CUtensorMap& tmW,
                                 const CUtensorMap& tmWu, const CUtensorMap& tmX, int grid,
                                 cudaStream_t s);
cudaError_t launch_wpair_down(int dtype, const GemmArgs& a, const CUtensorMap& tmTok,
                              const CUtensorMap& tmTokS, const CUtensorMap& tmW, int grid,
                              cudaStream_t s);

}  // namespace moe
