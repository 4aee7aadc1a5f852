// moe_abi.cu -- the C ABI declared in include/moe.h: argument checks,
// workspace layout, TMA descriptor encoding and stage launches.  Allocates
// nothing; every launch goes on the caller's stream.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "sched.cuh"

namespace moe {
size_t align_smem_bytes(int E);
}

using namespace moe;

namespace {

constexpr int kAbiVersion = 3;
constexpr size_t kWsAlign = 1024;
constexpr int kMaxExperts = 1024;
constexpr int kMaxDevices = 64;

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool valid_dtype_pair(int act, int weight) {
  if (act != MOE_F32 && act != MOE_BF16) return false;
  if (weight == act) return true;
  return weight == MOE_E2M1_MX && act == MOE_BF16;
}

// Experts held by this call: the shard's, or all E.
int local_experts(const moe_problem_t* p) {
  return p->local_experts > 0 ? p->local_experts : p->E;
}

int check_problem(const moe_problem_t* p) {
  if (p == nullptr) return MOE_ERR_INVALID_ARG;
  if (p->T < 0 || p->H <= 0 || p->I <= 0 || p->E <= 0 || p->K <= 0) return MOE_ERR_INVALID_ARG;
  if (!valid_dtype_pair(p->act, p->weight)) return MOE_ERR_INVALID_ARG;
  if (p->block_m != 0 && p->block_m != 16 && p->block_m != 32 && p->block_m != 64 &&
      p->block_m != 128 && p->block_m != 256)
    return MOE_ERR_INVALID_ARG;
  if (p->expert_base < 0 || p->local_experts < 0 ||
      static_cast<long long>(p->expert_base) + p->local_experts > p->E ||
      (p->local_experts == 0 && p->expert_base != 0))
    return MOE_ERR_INVALID_ARG;
  if (local_experts(p) > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  if (p->activation != MOE_ACT_SILU && p->activation != MOE_ACT_SWIGLU_CLAMP)
    return MOE_ERR_INVALID_ARG;
  if (p->activation == MOE_ACT_SWIGLU_CLAMP &&
      !(p->swiglu_limit > 0.0f && p->swiglu_limit < 3.0e38f && p->swiglu_alpha > -3.0e38f &&
        p->swiglu_alpha < 3.0e38f))
    return MOE_ERR_INVALID_ARG;
  if (p->gate_up_interleaved != 0 && p->gate_up_interleaved != 1) return MOE_ERR_INVALID_ARG;
  if (p->fused_combine != 0 && p->fused_combine != 1) return MOE_ERR_INVALID_ARG;
  const long long na = static_cast<long long>(p->T) * p->K;
  if (na >= (1ll << 30)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// Rows per align block.  The bf16/fp32 GEMMs take a block's tokens as the
// MMA's N (up to 256, rounded up to 16 from the block's valid rows), so the
// block size bounds the tile and costs no MMA work on padding: 256-row
// blocks once experts receive 256 rows on average (larger tiles move fewer
// bytes into the SMs per MMA), 128 otherwise (a smaller padded workspace).
// The block-scaled GEMMs tile 128 rows.
int block_m_of(const moe_problem_t* p) {
  if (p->block_m != 0) return p->block_m;
  if (p->weight == MOE_E2M1_MX) return kBlockM;
  const long long na = static_cast<long long>(p->T) * p->K;
  return na >= 256ll * p->E ? kPairBlockM : kBlockM;
}

bool is_mx(const moe_problem_t* p) { return p->weight == MOE_E2M1_MX; }

// The bf16/fp32 GEMMs read 128-byte k-tiles (64 bf16 / 32 fp32); any align
// block of at most 256 rows is one tile.  The block-scaled GEMMs need 128-row
// blocks and whole 32-element scale blocks along K (the end of K inside a
// 128-element tile is zero-filled).
int check_gemm_shapes(const moe_problem_t* p) {
  const int bm = block_m_of(p);
  if (is_mx(p) && bm != kBlockM) return MOE_ERR_UNSUPPORTED;
  if (is_mx(p)) {
    if (p->H % 32 != 0 || p->I % 32 != 0) return MOE_ERR_UNSUPPORTED;
    // TMA row coordinates of the tile-major packed values are 32-bit
    const long long L = p->local_experts > 0 ? p->local_experts : p->E;
    const long long tiles13 = L * mx_weight_tiles(2 * p->I, 2) * (mx_padded_k(p->H) / 128);
    const long long tiles2 = L * mx_weight_tiles(p->H, 1) * (mx_padded_k(p->I) / 128);
    if (std::max(tiles13, tiles2) * 192 >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
    if (!(p->h_scale >= 0.0f) || p->h_scale > 3.0e38f) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
  }
  const int bk = p->act == MOE_BF16 ? 64 : 32;
  if (p->H % bk != 0 || p->I % bk != 0) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

float h_scale_of(const moe_problem_t* p) { return p->h_scale > 0.0f ? p->h_scale : 1.0f; }

// Down-projection tiling: N columns per tile and K elements per k-tile.
int down_tile_n(const moe_problem_t* p) { return is_mx(p) ? 192 : 256; }
int down_tile_k(const moe_problem_t* p) { return is_mx(p) ? 128 : (p->act == MOE_BF16 ? 64 : 32); }

size_t act_bytes(int dtype) { return dtype == MOE_BF16 ? 2 : 4; }

// Launch geometry of each device, looked up once per device (the current
// device at the time of the call).
struct DeviceInfo {
  int sms = 0;
  int pairs[2][2] = {{-1, -1}, {-1, -1}};  // [kind][bf16]: CTA pairs held at once
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return -1;
  }
  return dev;
}

int sm_count() {
  const int dev = current_device();
  if (dev < 0) return 152;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_dev[dev].sms == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = 152;
    }
    g_dev[dev].sms = n;
  }
  return g_dev[dev].sms;
}

long long capacity(long long T, long long K, long long E, long long bm) {
  const long long na = T * K;
  return na + std::min(E, na) * (bm - 1);
}

int pairs_held(int kind, int dtype);

// K splits of the down projection.  Only batches too small to give every
// worker (CTA pair, or SM for the block-scaled GEMM) several tiles split: the
// count makes the number of (tile, split) units fill whole waves of
// workers as closely as possible, each split keeping at least 4 k-tiles.
// The block count is estimated on the host (at most one partly filled block
// per active expert).
int default_splits(const moe_problem_t* p) {
  const int bm = block_m_of(p);
  const long long na = static_cast<long long>(p->T) * p->K;
  if (na == 0) return 1;
  const long long L = local_experts(p);
  const long long cap = capacity(p->T, p->K, L, bm);
  const long long est_blocks =
      std::max(1ll, std::min({cap / bm, na, (na + bm - 1) / bm + std::min(L, na) - 1}));
  const long long n_tiles = (p->H + down_tile_n(p) - 1) / down_tile_n(p);
  const long long k_tiles = std::max(1, (p->I + down_tile_k(p) - 1) / down_tile_k(p));
  const long long units = std::max(1ll, est_blocks * n_tiles);
  const long long workers = is_mx(p) ? sm_count() : pairs_held(1, p->act);
  if (units >= 4 * workers) return 1;
  const long long s_max = std::min(32ll, std::max(1ll, k_tiles / 4));
  long long best = 1;
  double best_eff = 0.0;
  for (long long sp = 1; sp <= s_max; ++sp) {
    const long long u = units * sp;
    const long long waves = (u + workers - 1) / workers;
    const double eff = static_cast<double>(u) / static_cast<double>(waves * workers);
    if (eff > best_eff + 0.02) {
      best_eff = eff;
      best = sp;
    }
  }
  return static_cast<int>(best);
}

struct Layout {
  size_t off[MOE_WS_NUM];
  size_t size[MOE_WS_NUM];
  size_t total;
};

void layout_of(const moe_problem_t* p, Layout* L) {
  const int bm = block_m_of(p);
  const long long na = static_cast<long long>(p->T) * p->K;
  const long long cap = capacity(p->T, p->K, local_experts(p), bm);
  const bool mx = p->weight == MOE_E2M1_MX;
  const int splits = default_splits(p);
  size_t sz[MOE_WS_NUM] = {};
  sz[MOE_WS_STATUS] = 256;
  sz[MOE_WS_COUNTS] = 4ull * local_experts(p);
  sz[MOE_WS_OFFSETS] = 4ull * (local_experts(p) + 1);
  sz[MOE_WS_PADDED_OFFSETS] = 4ull * (local_experts(p) + 1);
  sz[MOE_WS_SORTED_IDS] = 4ull * cap;
  sz[MOE_WS_INV_PERM] = 4ull * na;
  sz[MOE_WS_BLOCK_INFO] = 16ull * (cap / bm);
  sz[MOE_WS_NUM_BLOCKS] = 4;
  // A rows in sorted order: e4m3 codes (MX), activation rows (CTA pairs)
  sz[MOE_WS_XQ] = static_cast<size_t>(cap) * p->H * (mx ? 1 : act_bytes(p->act));
  sz[MOE_WS_X_SCALE] = mx ? 4ull * p->T : 0;
  sz[MOE_WS_H] = static_cast<size_t>(cap) * p->I * (mx ? 1 : act_bytes(p->act));
  // y rows in sorted order per split, or the fused combine's accumulator
  sz[MOE_WS_Y] = p->fused_combine ? 4ull * p->T * p->H
                                  : 4ull * splits * static_cast<size_t>(cap) * p->H;
  sz[MOE_WS_ALIGN] = na >= kAlignMultiMin ? 4 * align_multi_scratch_ints(na, local_experts(p)) : 0;
  size_t off = 0;
  for (int i = 0; i < MOE_WS_NUM; ++i) {
    L->off[i] = off;
    L->size[i] = sz[i];
    off = round_up(off + sz[i], kWsAlign);
  }
  L->total = off;
}

// ---------------------------------------------------------------- TMA maps

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    else
      cudaGetLastError();
  });
  return g_encode;
}

// 2-D row-major tensor of `outer` rows of `inner` elements, `row_bytes`
// apart, read in 128-byte swizzled boxes of box_inner x box_outer elements.
int make_map_typed(CUtensorMap* tm, CUtensorMapDataType dt, const void* base, long long inner,
                   long long outer, long long row_bytes, int box_inner, int box_outer) {
  auto enc = encoder();
  if (enc == nullptr) return MOE_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(base) & 31u) != 0) return MOE_ERR_INVALID_ARG;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner),
                             static_cast<cuuint32_t>(box_outer)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(tm, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_INVALID_ARG;
}

// bf16 / fp32 row-major tensor (outer rows of `inner` elements).
int make_map(CUtensorMap* tm, int dtype, const void* base, long long inner, long long outer,
             int box_inner, int box_outer) {
  auto enc = encoder();
  if (enc == nullptr) return MOE_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0) return MOE_ERR_INVALID_ARG;
  const CUtensorMapDataType dt =
      dtype == MOE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * act_bytes(dtype)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner),
                             static_cast<cuuint32_t>(box_outer)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(tm, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_INVALID_ARG;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

int run_align(const int32_t* ids, int T, int K, int E, int e_base, int e_local, int bm,
              int32_t* counts, int32_t* offsets, int32_t* padded_offsets, int32_t* sorted_ids,
              int32_t* inv_perm, int32_t* block_info, int32_t* num_blocks, int32_t* status,
              cudaStream_t s, const RouteArgs* route = nullptr) {
  AlignArgs a;
  std::memset(&a.route, 0, sizeof(a.route));
  if (route != nullptr) a.route = *route;
  a.ids = ids;
  a.n_assign = T * K;
  a.E = E;
  a.e_base = e_base;
  a.e_local = e_local;
  a.block_m = bm;
  a.cap = capacity(T, K, e_local, bm);
  a.counts = counts;
  a.offsets = offsets;
  a.padded_offsets = padded_offsets;
  a.sorted_ids = sorted_ids;
  a.inv_perm = inv_perm;
  a.block_info = block_info;
  a.num_blocks = num_blocks;
  a.status = status;
  return cuda_status(launch_align(a, s));
}

Epilogue epilogue_of(const moe_problem_t* p) {
  Epilogue ep;
  ep.act = p->activation;
  ep.alpha = p->swiglu_alpha;
  ep.limit = p->swiglu_limit;
  ep.interleaved = p->gate_up_interleaved;
  ep.b13 = p->w13_bias;
  ep.b2 = p->w2_bias;
  return ep;
}

// The failure-path test (moe_test_gemm_wait_timeout): while set on this
// thread, the GEMM launches it makes starve their pipelines and give up
// after `timeout_ns`.
struct WaitTest {
  unsigned long long timeout_ns;
};
thread_local const WaitTest* t_wait_test = nullptr;

template <class Args>
void apply_wait_test(Args& a) {
  if (t_wait_test != nullptr) {
    a.timeout_ns = t_wait_test->timeout_ns;
    a.starve = 1;
  }
}

// Decode-like problems: at most 32 tokens in all, or at most 32 rows per
// expert on average, so that most align blocks hold at most 32 tokens.
bool decode_like(const moe_problem_t* p) {
  return p->T <= 32 || static_cast<long long>(p->T) * p->K <= 32ll * local_experts(p);
}

GemmArgs base_args(const moe_problem_t* p) {
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.T = p->T;
  a.H = p->H;
  a.I = p->I;
  a.E = p->E;
  a.K = p->K;
  a.cap = capacity(p->T, p->K, local_experts(p), block_m_of(p));
  a.n_held = local_experts(p);
  a.max_blocks = static_cast<int>(a.cap / block_m_of(p));
  a.timeout_ns = kWaitTimeoutNs;
  a.ep = epilogue_of(p);
  // decode-like launches, where most align blocks hold at most 32 tokens:
  // at most 32 tokens in all, or at most 32 rows per expert on average.
  // Their tiles stream weights, and two K steps per stage double the bytes
  // in flight; in prefill launches (hundreds of rows per expert) the same
  // stages measured slower.
  a.dual_small = decode_like(p);
  apply_wait_test(a);
  return a;
}

// Persistent grid of CTA pairs: no more pairs than the device holds at once
// (cluster placement can leave SMs without a partner), so that every pair
// is resident from the start, and no more than there are tiles.
int pair_limit(int kind, int dtype) {
  const int dev = current_device();
  if (dev < 0) return 0;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  int& v = g_dev[dev].pairs[kind][dtype == MOE_BF16 ? 1 : 0];
  if (v < 0) v = wpair_max_active(kind, dtype);
  return v;
}

int pairs_held(int kind, int dtype) {
  long long limit = sm_count() / 2;
  const int held = pair_limit(kind, dtype);
  if (held > 0) limit = std::min<long long>(limit, held);
  return static_cast<int>(std::max(1ll, limit));
}

int pair_grid(long long tiles, int kind, int dtype) {
  const long long clusters = std::max(1ll, std::min<long long>(pairs_held(kind, dtype), tiles));
  return static_cast<int>(2 * clusters);
}

// Gate/up: token rows x w13, on CTA pairs with 256 weight rows (128 gate +
// 128 up indices j) per tile.  rows: x in sorted order (cap rows, as
// moe_gather_rows writes it), or with `gather` x itself (T rows), which the
// producer gathers by sorted_ids.
int run_gemm1(const moe_problem_t* p, const void* rows, const void* w13,
              const int32_t* sorted_ids, const int32_t* block_info, const int32_t* num_blocks,
              void* h, int32_t* status, cudaStream_t s, bool gather = false) {
  GemmArgs a = base_args(p);
  const int bk = p->act == MOE_BF16 ? 64 : 32;
  a.n_tiles = (p->I + 127) / 128;
  a.k_tiles = p->H / bk;
  a.splits = 1;
  a.band = gate_up_band(a.n_tiles);
  a.sorted_ids = sorted_ids;
  a.block_info = block_info;
  a.num_blocks = num_blocks;
  a.out = h;
  a.status = status;
  a.x = rows;
  a.gather = gather ? 1 : 0;
  CUtensorMap tmTok, tmTokS, tmW, tmWu, tmX;
  int rc;
  if (p->gate_up_interleaved) {
    // gate rows 2j and up rows 2j+1: two maps of I rows per expert, each row
    // two w13 rows apart
    const CUtensorMapDataType dt =
        p->act == MOE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const long long row_bytes = 2ll * p->H * act_bytes(p->act);
    const long long rows = 1ll * p->I * local_experts(p);
    rc = make_map_typed(&tmW, dt, w13, p->H, rows, row_bytes, bk, 64);
    if (rc == MOE_OK)
      rc = make_map_typed(&tmWu, dt, static_cast<const char*>(w13) + p->H * act_bytes(p->act),
                          p->H, rows, row_bytes, bk, 64);
    a.w_rows_per_expert = p->I;
    a.up_row_offset = 0;
  } else {
    rc = make_map(&tmW, p->act, w13, p->H, 2ll * p->I * local_experts(p), bk, 64);
    tmWu = tmW;
    a.w_rows_per_expert = 2 * p->I;
    a.up_row_offset = p->I;
  }
  if (gather) {
    if (rc == MOE_OK) rc = make_map(&tmX, p->act, rows, p->H, p->T, bk, 1);
    tmTok = tmTokS = tmX;  // not read
  } else {
    if (rc == MOE_OK) rc = make_map(&tmTok, p->act, rows, p->H, a.cap, bk, 128);
    if (rc == MOE_OK) rc = make_map(&tmTokS, p->act, rows, p->H, a.cap, bk, 16);
    tmX = tmTok;  // not read
  }
  if (rc != MOE_OK) return rc;
  const long long max_tiles = (a.cap / block_m_of(p)) * a.n_tiles;
  return cuda_status(launch_wpair_gate_up(p->act, a, tmTok, tmTokS, tmW, tmWu, tmX,
                                          pair_grid(max_tiles, 0, p->act), s));
}

// Down: h rows x w2 x routing weight, on CTA pairs with 256 w2 rows per tile.
int run_gemm2(const moe_problem_t* p, const void* h, const void* w2, const float* topk_weights,
              const int32_t* sorted_ids, const int32_t* block_info, const int32_t* num_blocks,
              float* y, int splits, int32_t* status, cudaStream_t s) {
  GemmArgs a = base_args(p);
  const int bk = p->act == MOE_BF16 ? 64 : 32;
  a.n_tiles = (p->H + 255) / 256;
  a.k_tiles = p->I / bk;
  a.splits = splits;
  a.band = down_band(a.n_tiles);
  a.sorted_ids = sorted_ids;
  a.block_info = block_info;
  a.num_blocks = num_blocks;
  a.topk_weights = topk_weights;
  a.out = y;
  a.fused = p->fused_combine;
  a.status = status;
  CUtensorMap tmTok, tmTokS, tmW;
  int rc = make_map(&tmW, p->act, w2, p->I, 1ll * p->H * local_experts(p), bk, 128);
  if (rc == MOE_OK) rc = make_map(&tmTok, p->act, h, p->I, a.cap, bk, 128);
  if (rc == MOE_OK) rc = make_map(&tmTokS, p->act, h, p->I, a.cap, bk, 16);
  if (rc != MOE_OK) return rc;
  const long long max_tiles = (a.cap / block_m_of(p)) * a.n_tiles * splits;
  return cuda_status(launch_wpair_down(p->act, a, tmTok, tmTokS, tmW,
                                       pair_grid(max_tiles, 1, p->act), s));
}

// Rows of 128 K elements in the tile-major packed values of an (E, R, K)
// weight tensor with `sections` sections: E * weight tiles * K tiles tiles
// of 192 rows each.
long long mx_value_rows(long long E, int R, int K, int sections) {
  return E * mx_weight_tiles(R, sections) * (mx_padded_k(K) / 128) * 192ll;
}

MxArgs mx_args(const moe_problem_t* p) {
  MxArgs a;
  std::memset(&a, 0, sizeof(a));
  a.T = p->T;
  a.H = p->H;
  a.I = p->I;
  a.E = p->E;
  a.K = p->K;
  a.cap = capacity(p->T, p->K, local_experts(p), kBlockM);
  a.n_held = local_experts(p);
  a.max_blocks = static_cast<int>(a.cap / kBlockM);
  a.h_scale = h_scale_of(p);
  a.timeout_ns = kWaitTimeoutNs;
  a.ep = epilogue_of(p);
  apply_wait_test(a);
  return a;
}

bool aligned(const void* ptr, uintptr_t n) { return (reinterpret_cast<uintptr_t>(ptr) % n) == 0; }

int run_gemm1_mx(const moe_problem_t* p, const void* xq, const float* x_row_scale, const void* w13,
                 const uint8_t* w13_scale, const int32_t* sorted_ids, const int32_t* block_info,
                 const int32_t* num_blocks, void* hq, int32_t* status, cudaStream_t s) {
  if (!aligned(xq, 32) || !aligned(hq, 16) || !aligned(w13, 32) || !aligned(w13_scale, 16))
    return MOE_ERR_INVALID_ARG;
  MxArgs a = mx_args(p);
  const int Hp = mx_padded_k(p->H);
  a.Kdim = p->H;
  a.n_tiles = (p->I + 95) / 96;
  a.k_tiles = Hp / 128;
  a.splits = 1;
  // every weight tile of a block in one band: the co-resident CTAs then
  // share the block's A rows in L2 across all its weight tiles (measured
  // 2 % faster than bands of 8 on the low-precision workload)
  a.band = a.n_tiles;
  a.a = static_cast<const uint8_t*>(xq);
  a.x_row_scale = x_row_scale;
  a.w_scale = w13_scale;
  a.sections = 2;
  a.kp_tiles = Hp / 128;
  CUtensorMap tmA, tmA64, tmW;
  int rc = make_map_typed(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, p->H, a.cap, p->H, 128, 128);
  if (rc == MOE_OK)
    rc = make_map_typed(&tmA64, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, p->H, a.cap, p->H, 128, 64);
  if (rc != MOE_OK) return rc;
  rc = make_map_typed(&tmW, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, w13, 128,
                      mx_value_rows(local_experts(p), 2 * p->I, p->H, 2), 64, 128, 192);
  if (rc != MOE_OK) return rc;
  a.sorted_ids = sorted_ids;
  a.block_info = block_info;
  a.num_blocks = num_blocks;
  a.out = hq;
  a.status = status;
  const long long max_tiles = (a.cap / kBlockM) * a.n_tiles;
  const int grid = static_cast<int>(std::max(1ll, std::min<long long>(sm_count(), max_tiles)));
  return cuda_status(launch_mx_gate_up(a, tmA, tmA64, tmW, grid, s));
}

int run_gemm2_mx(const moe_problem_t* p, const void* hq, const void* w2, const uint8_t* w2_scale,
                 const float* topk_weights, const int32_t* sorted_ids, const int32_t* block_info,
                 const int32_t* num_blocks, float* y, int splits, int32_t* status,
                 cudaStream_t s) {
  if (!aligned(hq, 32) || !aligned(w2, 32) || !aligned(w2_scale, 16) || !aligned(y, 16))
    return MOE_ERR_INVALID_ARG;
  MxArgs a = mx_args(p);
  const int Ip = mx_padded_k(p->I);
  a.Kdim = p->I;
  a.n_tiles = (p->H + 191) / 192;
  a.k_tiles = Ip / 128;
  a.splits = splits;
  a.band = a.n_tiles;  // as for gate/up
  a.a = static_cast<const uint8_t*>(hq);
  a.w_scale = w2_scale;
  a.sections = 1;
  a.kp_tiles = Ip / 128;
  a.fused = p->fused_combine;
  CUtensorMap tmA, tmA64, tmW;
  int rc = make_map_typed(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, hq, p->I, a.cap, p->I, 128, 128);
  if (rc == MOE_OK)
    rc = make_map_typed(&tmA64, CU_TENSOR_MAP_DATA_TYPE_UINT8, hq, p->I, a.cap, p->I, 128, 64);
  if (rc != MOE_OK) return rc;
  rc = make_map_typed(&tmW, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, w2, 128,
                      mx_value_rows(local_experts(p), p->H, p->I, 1), 64, 128, 192);
  if (rc != MOE_OK) return rc;
  a.sorted_ids = sorted_ids;
  a.block_info = block_info;
  a.num_blocks = num_blocks;
  a.topk_weights = topk_weights;
  a.out = y;
  a.status = status;
  const long long max_tiles = (a.cap / kBlockM) * a.n_tiles * splits;
  const int grid = static_cast<int>(std::max(1ll, std::min<long long>(sm_count(), max_tiles)));
  return cuda_status(launch_mx_down(a, tmA, tmA64, tmW, grid, s));
}

}  // namespace

int moe::validate_forward_problem(const moe_problem_t* p) {
  const int rc = check_problem(p);
  return rc != MOE_OK ? rc : check_gemm_shapes(p);
}

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case MOE_ERR_WORKSPACE: return "workspace too small or misaligned";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_BAD_ID: return "expert id outside [0, E)";
    case MOE_ERR_TIMEOUT: return "pipeline wait timed out";
    case MOE_ERR_BOUNDS: return "index outside its buffer (checked build)";
    default: return "unknown status";
  }
}

int moe_abi_version(void) { return kAbiVersion; }

int moe_resolve_block_m(const moe_problem_t* p) {
  if (check_problem(p) != MOE_OK) return -1;
  return block_m_of(p);
}

size_t moe_align_capacity(int T, int K, int E, int block_m) {
  if (T < 0 || K <= 0 || E <= 0 || block_m <= 0) return 0;
  return static_cast<size_t>(capacity(T, K, E, block_m));
}

int moe_gemm2_default_splits(const moe_problem_t* p) {
  if (check_problem(p) != MOE_OK) return -1;
  return default_splits(p);
}

size_t moe_workspace_size(const moe_problem_t* p) {
  if (check_problem(p) != MOE_OK) return 0;
  Layout L;
  layout_of(p, &L);
  return L.total;
}

int moe_workspace_offsets(const moe_problem_t* p, size_t offsets[MOE_WS_NUM],
                          size_t sizes[MOE_WS_NUM]) {
  const int rc = check_problem(p);
  if (rc != MOE_OK) return rc;
  if (offsets == nullptr) return MOE_ERR_INVALID_ARG;
  Layout L;
  layout_of(p, &L);
  for (int i = 0; i < MOE_WS_NUM; ++i) {
    offsets[i] = L.off[i];
    if (sizes != nullptr) sizes[i] = L.size[i];
  }
  return MOE_OK;
}

int moe_align(const int32_t* topk_ids, int T, int K, int E, int block_m, int32_t* counts,
              int32_t* offsets, int32_t* padded_offsets, int32_t* sorted_ids, int32_t* inv_perm,
              int32_t* block_info, int32_t* num_blocks, int32_t* dev_status, void* stream) {
  return moe_align_local(topk_ids, T, K, E, 0, E, block_m, counts, offsets, padded_offsets,
                         sorted_ids, inv_perm, block_info, num_blocks, nullptr, 0, dev_status,
                         stream);
}

size_t moe_align_scratch_bytes(int T, int K, int local_experts) {
  if (T < 0 || K <= 0 || local_experts <= 0) return 0;
  const long long na = static_cast<long long>(T) * K;
  if (na < kAlignMultiMin) return 0;
  return 4 * align_multi_scratch_ints(na, local_experts);
}

int moe_align_local(const int32_t* topk_ids, int T, int K, int E, int expert_base,
                    int local_experts, int block_m, int32_t* counts, int32_t* offsets,
                    int32_t* padded_offsets, int32_t* sorted_ids, int32_t* inv_perm,
                    int32_t* block_info, int32_t* num_blocks, void* scratch,
                    size_t scratch_bytes, int32_t* dev_status, void* stream) {
  if (T < 0 || K <= 0 || E <= 0) return MOE_ERR_INVALID_ARG;
  if (block_m != 16 && block_m != 32 && block_m != 64 && block_m != 128 && block_m != 256)
    return MOE_ERR_INVALID_ARG;
  if (expert_base < 0 || local_experts <= 0 ||
      static_cast<long long>(expert_base) + local_experts > E)
    return MOE_ERR_INVALID_ARG;
  if (local_experts > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(T) * K >= (1ll << 30)) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!topk_ids || !counts || !offsets || !padded_offsets || !sorted_ids || !inv_perm ||
      !block_info || !num_blocks)
    return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(block_info) & 15u) != 0) return MOE_ERR_INVALID_ARG;
  const size_t need = moe_align_scratch_bytes(T, K, local_experts);
  if (need > 0 && scratch != nullptr) {
    if (scratch_bytes < need || (reinterpret_cast<uintptr_t>(scratch) & 15u) != 0)
      return MOE_ERR_WORKSPACE;
    AlignArgs al;
    std::memset(&al, 0, sizeof(al));
    al.ids = topk_ids;
    al.n_assign = T * K;
    al.E = E;
    al.e_base = expert_base;
    al.e_local = local_experts;
    al.block_m = block_m;
    al.cap = capacity(T, K, local_experts, block_m);
    al.counts = counts;
    al.offsets = offsets;
    al.padded_offsets = padded_offsets;
    al.sorted_ids = sorted_ids;
    al.inv_perm = inv_perm;
    al.block_info = block_info;
    al.num_blocks = num_blocks;
    al.status = dev_status;
    return cuda_status(launch_align_multi(al, static_cast<int32_t*>(scratch),
                                          static_cast<cudaStream_t>(stream)));
  }
  return run_align(topk_ids, T, K, E, expert_base, local_experts, block_m, counts, offsets,
                   padded_offsets, sorted_ids, inv_perm, block_info, num_blocks, dev_status,
                   static_cast<cudaStream_t>(stream));
}

int moe_route_align(const void* logits, int logit_dtype, int T, int E, int K, int expert_base,
                    int local_experts, int block_m, int32_t* topk_ids, float* topk_weights,
                    int32_t* counts, int32_t* offsets, int32_t* padded_offsets,
                    int32_t* sorted_ids, int32_t* inv_perm, int32_t* block_info,
                    int32_t* num_blocks, int32_t* dev_status, void* stream) {
  if (T < 0 || E <= 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (logit_dtype != MOE_BF16 && logit_dtype != MOE_F32) return MOE_ERR_INVALID_ARG;
  if (K > E) return MOE_ERR_INVALID_ARG;
  if (K > 32 || E > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  if (block_m != 16 && block_m != 32 && block_m != 64 && block_m != 128 && block_m != 256)
    return MOE_ERR_INVALID_ARG;
  if (expert_base < 0 || local_experts <= 0 ||
      static_cast<long long>(expert_base) + local_experts > E)
    return MOE_ERR_INVALID_ARG;
  if (static_cast<long long>(T) * K >= (1ll << 30)) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!logits || !topk_ids || !topk_weights || !counts || !offsets || !padded_offsets ||
      !sorted_ids || !inv_perm || !block_info || !num_blocks)
    return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(block_info) & 15u) != 0) return MOE_ERR_INVALID_ARG;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  RouteArgs r;
  r.logits = logits;
  r.bf16 = logit_dtype == MOE_BF16;
  r.T = T;
  r.E = E;
  r.K = K;
  r.ids = topk_ids;
  r.weights = topk_weights;
  r.status = dev_status;
  const bool in_align = T <= kRouteInAlignMaxTokens;
  if (!in_align && launch_route(r, s) != cudaSuccess) return MOE_ERR_CUDA;
  return run_align(topk_ids, T, K, E, expert_base, local_experts, block_m, counts, offsets,
                   padded_offsets, sorted_ids, inv_perm, block_info, num_blocks, dev_status, s,
                   in_align ? &r : nullptr);
}

int moe_quantize_x_fp8(const void* x, int x_dtype, int T, int H, uint8_t* xq, float* row_scale,
                       void* stream) {
  if (T < 0 || H <= 0 || (H & 1) != 0) return MOE_ERR_INVALID_ARG;
  if (x_dtype != MOE_BF16 && x_dtype != MOE_F32) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !xq || !row_scale) return MOE_ERR_INVALID_ARG;
  return cuda_status(
      launch_quantize_x(x, x_dtype, T, H, xq, row_scale, static_cast<cudaStream_t>(stream)));
}

int moe_gather_rows(const void* x, int dtype, int T, int H, int K, const int32_t* inv_perm,
                    void* x_sorted, float* acc_zero, int32_t* dev_status, void* stream) {
  if (T < 0 || H <= 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_BF16 && dtype != MOE_F32) return MOE_ERR_INVALID_ARG;
  const long long row_bytes = static_cast<long long>(H) * act_bytes(dtype);
  if (row_bytes % 16 != 0) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!x || !inv_perm || !x_sorted) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(x_sorted) & 15u) ||
      (reinterpret_cast<uintptr_t>(acc_zero) & 15u))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_gather_rows(x, T, static_cast<int>(row_bytes), K, inv_perm, x_sorted,
                                        acc_zero, H, dev_status,
                                        static_cast<cudaStream_t>(stream)));
}

int moe_quantize_gather_x_fp8(const void* x, int x_dtype, int T, int H, int K,
                              const int32_t* inv_perm, uint8_t* xq_sorted, float* row_scale,
                              float* acc_zero, int32_t* dev_status, void* stream) {
  if (T < 0 || H <= 0 || (H & 1) != 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (x_dtype != MOE_BF16 && x_dtype != MOE_F32) return MOE_ERR_INVALID_ARG;
  if (acc_zero != nullptr && H % 4 != 0) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!x || !inv_perm || !xq_sorted || !row_scale) return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(acc_zero) & 15u) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_quantize_gather_x(x, x_dtype, T, H, K, inv_perm, xq_sorted, row_scale,
                                              acc_zero, dev_status,
                                              static_cast<cudaStream_t>(stream)));
}

int moe_combine_finish(const float* acc, int T, int H, int out_dtype, void* out,
                       int32_t* dev_status, void* stream) {
  if (T < 0 || H <= 0) return MOE_ERR_INVALID_ARG;
  if (out_dtype != MOE_BF16 && out_dtype != MOE_F32) return MOE_ERR_INVALID_ARG;
  if (H % 4 != 0) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!acc || !out) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(acc) & 15u) ||
      (reinterpret_cast<uintptr_t>(out) & (out_dtype == MOE_BF16 ? 7u : 15u)))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine_finish(acc, T, H, out_dtype, out, dev_status,
                                           static_cast<cudaStream_t>(stream)));
}

int moe_gemm1_silu(const moe_problem_t* p, const void* x, const float* x_row_scale,
                   const void* w13, const uint8_t* w13_scale, const int32_t* sorted_ids,
                   const int32_t* block_info, const int32_t* num_blocks, void* h,
                   int32_t* dev_status, void* stream) {
  int rc = check_problem(p);
  if (rc != MOE_OK) return rc;
  rc = check_gemm_shapes(p);
  if (rc != MOE_OK) return rc;
  if (p->T == 0) return MOE_OK;
  if (!x || !w13 || !sorted_ids || !block_info || !num_blocks || !h) return MOE_ERR_INVALID_ARG;
  if (is_mx(p)) {
    if (!x_row_scale || !w13_scale) return MOE_ERR_INVALID_ARG;
    return run_gemm1_mx(p, x, x_row_scale, w13, w13_scale, sorted_ids, block_info, num_blocks, h,
                        dev_status, static_cast<cudaStream_t>(stream));
  }
  return run_gemm1(p, x, w13, sorted_ids, block_info, num_blocks, h, dev_status,
                   static_cast<cudaStream_t>(stream));
}

int moe_gemm1_silu_gather(const moe_problem_t* p, const void* x, const void* w13,
                          const int32_t* sorted_ids, const int32_t* block_info,
                          const int32_t* num_blocks, void* h, int32_t* dev_status, void* stream) {
  int rc = check_problem(p);
  if (rc != MOE_OK) return rc;
  rc = check_gemm_shapes(p);
  if (rc != MOE_OK) return rc;
  if (is_mx(p)) return MOE_ERR_UNSUPPORTED;
  if (p->T == 0) return MOE_OK;
  if (!x || !w13 || !sorted_ids || !block_info || !num_blocks || !h) return MOE_ERR_INVALID_ARG;
  return run_gemm1(p, x, w13, sorted_ids, block_info, num_blocks, h, dev_status,
                   static_cast<cudaStream_t>(stream), true);
}

int moe_gemm2_weighted(const moe_problem_t* p, const void* h, const void* w2,
                       const uint8_t* w2_scale, const float* topk_weights,
                       const int32_t* sorted_ids, const int32_t* block_info,
                       const int32_t* num_blocks, float* y, int k_splits, int32_t* dev_status,
                       void* stream) {
  int rc = check_problem(p);
  if (rc != MOE_OK) return rc;
  rc = check_gemm_shapes(p);
  if (rc != MOE_OK) return rc;
  const int k_tiles = (p->I + down_tile_k(p) - 1) / down_tile_k(p);
  if (k_splits < 1 || k_splits > k_tiles) return MOE_ERR_INVALID_ARG;
  if (p->T == 0) return MOE_OK;
  if (!h || !w2 || !topk_weights || !sorted_ids || !block_info || !num_blocks || !y)
    return MOE_ERR_INVALID_ARG;
  if (is_mx(p)) {
    if (!w2_scale) return MOE_ERR_INVALID_ARG;
    return run_gemm2_mx(p, h, w2, w2_scale, topk_weights, sorted_ids, block_info, num_blocks, y,
                        k_splits, dev_status, static_cast<cudaStream_t>(stream));
  }
  return run_gemm2(p, h, w2, topk_weights, sorted_ids, block_info, num_blocks, y, k_splits,
                   dev_status, static_cast<cudaStream_t>(stream));
}

int moe_test_gemm_wait_timeout(const moe_problem_t* p, int gemm, const void* a_rows,
                               const float* x_row_scale, const void* w, const uint8_t* w_scale,
                               const float* topk_weights, const int32_t* sorted_ids,
                               const int32_t* block_info, const int32_t* num_blocks, void* out,
                               int k_splits, unsigned long long wait_limit_ns,
                               int32_t* dev_status, void* stream) {
  if (gemm != 1 && gemm != 2) return MOE_ERR_INVALID_ARG;
  if (wait_limit_ns < 1000000ull || wait_limit_ns > kWaitTimeoutNs) return MOE_ERR_INVALID_ARG;
  const WaitTest test{wait_limit_ns};
  t_wait_test = &test;
  const int rc = gemm == 1 ? moe_gemm1_silu(p, a_rows, x_row_scale, w, w_scale, sorted_ids,
                                            block_info, num_blocks, out, dev_status, stream)
                           : moe_gemm2_weighted(p, a_rows, w, w_scale, topk_weights, sorted_ids,
                                                block_info, num_blocks,
                                                static_cast<float*>(out), k_splits, dev_status,
                                                stream);
  t_wait_test = nullptr;
  return rc;
}

int moe_combine(const float* y, int k_splits, size_t cap, const int32_t* inv_perm, int T, int K,
                int H, int out_dtype, void* out, int32_t* dev_status, void* stream) {
  if (T < 0 || K <= 0 || H <= 0 || k_splits < 1) return MOE_ERR_INVALID_ARG;
  if (out_dtype != MOE_BF16 && out_dtype != MOE_F32) return MOE_ERR_INVALID_ARG;
  if (H % 4 != 0) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!y || !inv_perm || !out) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(y, k_splits, static_cast<long long>(cap), inv_perm, T, K, H,
                                    out_dtype, out, dev_status,
                                    static_cast<cudaStream_t>(stream)));
}

int moe_forward(const moe_problem_t* p, const void* x, const int32_t* topk_ids,
                const float* topk_weights, const void* w13, const uint8_t* w13_scale,
                const void* w2, const uint8_t* w2_scale, void* out, void* workspace,
                size_t workspace_bytes, void* stream) {
  int rc = validate_forward_problem(p);
  if (rc != MOE_OK) return rc;
  if (p->T == 0) return MOE_OK;
  if (!x || !topk_ids || !topk_weights || !w13 || !w2 || !out || !workspace)
    return MOE_ERR_INVALID_ARG;
  if (is_mx(p) && (!w13_scale || !w2_scale)) return MOE_ERR_INVALID_ARG;
  Layout L;
  layout_of(p, &L);
  if (workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto part = [&](int i) { return ws + L.off[i]; };
  int32_t* status = reinterpret_cast<int32_t*>(part(MOE_WS_STATUS));
  int32_t* sorted_ids = reinterpret_cast<int32_t*>(part(MOE_WS_SORTED_IDS));
  int32_t* block_info = reinterpret_cast<int32_t*>(part(MOE_WS_BLOCK_INFO));
  int32_t* num_blocks = reinterpret_cast<int32_t*>(part(MOE_WS_NUM_BLOCKS));
  int32_t* inv_perm = reinterpret_cast<int32_t*>(part(MOE_WS_INV_PERM));
  float* y = reinterpret_cast<float*>(part(MOE_WS_Y));
  float* acc_zero = p->fused_combine ? y : nullptr;  // zeroed by the gather step
  void* h = part(MOE_WS_H);
  const int splits = default_splits(p);
  const int bm = block_m_of(p);

  if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
  rc = moe_align_local(topk_ids, p->T, p->K, p->E, p->expert_base, local_experts(p), bm,
                       reinterpret_cast<int32_t*>(part(MOE_WS_COUNTS)),
                       reinterpret_cast<int32_t*>(part(MOE_WS_OFFSETS)),
                       reinterpret_cast<int32_t*>(part(MOE_WS_PADDED_OFFSETS)), sorted_ids,
                       inv_perm, block_info, num_blocks, part(MOE_WS_ALIGN),
                       L.size[MOE_WS_ALIGN], status, stream);
  if (rc != MOE_OK) return rc;
  if (is_mx(p)) {
    uint8_t* xq = part(MOE_WS_XQ);
    float* xs = reinterpret_cast<float*>(part(MOE_WS_X_SCALE));
    if (launch_quantize_gather_x(x, p->act, p->T, p->H, p->K, inv_perm, xq, xs, acc_zero, status,
                                 s, capacity(p->T, p->K, local_experts(p), bm)) != cudaSuccess)
      return MOE_ERR_CUDA;
    rc = run_gemm1_mx(p, xq, xs, w13, w13_scale, sorted_ids, block_info, num_blocks, h, status, s);
    if (rc != MOE_OK) return rc;
    rc = run_gemm2_mx(p, h, w2, w2_scale, topk_weights, sorted_ids, block_info, num_blocks, y,
                      splits, status, s);
    if (rc != MOE_OK) return rc;
  } else {
    void* xs = part(MOE_WS_XQ);  // token rows in sorted order
    if (launch_gather_rows(x, p->T, static_cast<int>(p->H * act_bytes(p->act)), p->K, inv_perm,
                           xs, acc_zero, p->H, status, s,
                           capacity(p->T, p->K, local_experts(p), bm)) != cudaSuccess)
      return MOE_ERR_CUDA;
    rc = run_gemm1(p, xs, w13, sorted_ids, block_info, num_blocks, h, status, s);
    if (rc != MOE_OK) return rc;
    rc = run_gemm2(p, h, w2, topk_weights, sorted_ids, block_info, num_blocks, y, splits, status,
                   s);
    if (rc != MOE_OK) return rc;
  }
  if (p->fused_combine)
    return cuda_status(launch_combine_finish(y, p->T, p->H, p->act, out, status, s));
  return cuda_status(launch_combine(y, splits, capacity(p->T, p->K, local_experts(p), bm),
                                    inv_perm, p->T, p->K, p->H, p->act, out, status, s));
}

size_t moe_mx_packed_bytes(int E, int R, int K, int sections, size_t* value_bytes,
                           size_t* scale_bytes) {
  if (E <= 0 || R <= 0 || K <= 0 || K % 32 != 0 || (sections != 1 && sections != 2) ||
      R % sections != 0)
    return 0;
  const size_t Kp = static_cast<size_t>(mx_padded_k(K));
  const size_t vb = static_cast<size_t>(mx_value_rows(E, R, K, sections)) * 64;
  const size_t sb = static_cast<size_t>(E) * mx_weight_tiles(R, sections) * (Kp / 128) * 1024;
  if (value_bytes) *value_bytes = vb;
  if (scale_bytes) *scale_bytes = sb;
  return vb + sb;
}

int moe_pack_mx_weights(const uint8_t* w, const uint8_t* w_scale, int E, int R, int K,
                        int sections, int interleaved, uint8_t* w_packed, uint8_t* scale_packed,
                        void* stream) {
  if (moe_mx_packed_bytes(E, R, K, sections, nullptr, nullptr) == 0) return MOE_ERR_INVALID_ARG;
  if (interleaved != 0 && (interleaved != 1 || sections != 2)) return MOE_ERR_INVALID_ARG;
  if (!w || !w_scale || !w_packed || !scale_packed) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_pack_mx(w, w_scale, E, R, K, sections, interleaved, w_packed,
                                    scale_packed, static_cast<cudaStream_t>(stream)));
}

int moe_device_info(int* sm_count_out, int* pair_clusters_out) {
  if (sm_count_out) *sm_count_out = sm_count();
  if (pair_clusters_out) *pair_clusters_out = pairs_held(0, MOE_BF16);
  return MOE_OK;
}

int moe_get_device_status(const int32_t* dev_status, void* stream) {
  if (dev_status == nullptr) return MOE_ERR_INVALID_ARG;
  int32_t v = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&v, dev_status, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  return v == 0 ? MOE_OK : v;
}

}  // extern "C"
