// align.cu -- routing alignment: expert histogram, padded prefix sums,
// stable scatter into the expert-sorted padded list, inverse permutation
// and per-block work descriptors.
//
// Sources: "factor_moe_fused_gemm.cu", build_expert_map_kernel (expert
// counts, CSR offsets and the token permutation; its atomics leave the order
// within an expert undefined, here the order is the ascending flat index);
// "moe triton kernel use tma", mblocks_to_tuple_info (one (expert, M-index,
// token start) tuple per M-block); "MOE Bmm1 Fused Gather",
// load_activations (padding slots of a block are masked).
//
// One CTA of 32 warps does the whole job for small batches; the work is a
// few passes over T*K int32 ids.  Large batches (from kAlignMultiMin ids,
// given a scratch) spread the passes over many CTAs (align_hist_kernel,
// align_scan_kernel, align_scatter_kernel below), same result.  Warp w owns
// a contiguous chunk of the flat index range and a private histogram row in
// shared memory:
//   1. histogram: per 32-id batch, ballots over the bits of the id group
//      equal ids and the group's lowest lane adds the group size to the
//      warp's row;
//   2. per expert, an exclusive scan over the warps' rows gives each warp its
//      start inside the expert; a block-wide scan over experts gives the CSR
//      and padded offsets;
//   3. scatter: the warps walk their chunks again in the same order; an id's
//      slot is padded_offset[e] + warp start + running count + rank among the
//      equal ids of lower lanes.  Chunks are in index order, batches in index
//      order, lanes in index order, so the result is the stable order.
//   4. padding slots, the tail up to the capacity, and block descriptors.
// Expert-parallel shard: only the experts [e_base, e_base + e_local) get
// lists (all per-expert outputs are indexed by e - e_base); an assignment to
// another expert is left out and its inverse-permutation entry is -1.  The
// shard of all E experts is the plain align.  Source for the shard: the
// "MOE Bmm1 Fused Gather" example's init_routing_data, which keeps the
// histogram of the local experts of one expert shard.
#include <cuda_bf16.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kAlignWarps = 32;
constexpr int kAlignThreads = kAlignWarps * 32;
// Batches of 32 ids a warp loads at once before it works through them in
// order: keeps several loads in flight instead of one round trip per batch.
constexpr int kAlignUnroll = 8;

// ids [base + 32u + lane] for u < kAlignUnroll, -1 at or past `hi`.  Plain
// loads: the ids may have been written by this kernel's routing step.
__device__ __forceinline__ void load_ids(const int* ids, int base, int hi, int lane,
                                         int (&e)[kAlignUnroll]) {
#pragma unroll
  for (int u = 0; u < kAlignUnroll; ++u) {
    const int i = base + 32 * u + lane;
    e[u] = i < hi ? ids[i] : -1;
  }
}

// ---------------------------------------------------------------- routing
// Top-K routing of one token by one warp, from its E router logits: the
// experts of the K largest logits in descending order (an equal logit goes
// to the lower expert id) and the softmax over the experts renormalised
// over the K chosen, which is the softmax over the chosen logits alone.
// Source: "MOE Bmm1 Fused Gather", init_routing_data (topk with
// apply_softmax feeding the expert histogram).  Lane l owns experts
// l, l + 32, ... (E <= 1024); each of the K rounds takes every lane's best
// untaken expert and a warp arg-max.  A token whose remaining logits all
// compare false (NaN) records MOE_ERR_DEVICE_BAD_ID.
__device__ __forceinline__ float logit_at(const RouteArgs& r, long long idx) {
  if (r.bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(r.logits)[idx]);
  return reinterpret_cast<const float*>(r.logits)[idx];
}

__device__ __forceinline__ void route_token(const RouteArgs& r, int t, int lane) {
  const long long row = static_cast<long long>(t) * r.E;
  unsigned taken = 0;  // bit i: expert lane + 32 i chosen
  float my_v = 0.0f;   // lane k keeps the k-th choice
  int my_id = 0;
  for (int k = 0; k < r.K; ++k) {
    float bv = -INFINITY;
    int bid = 0x7fffffff;
    for (int i = 0, e = lane; e < r.E; ++i, e += 32) {
      if ((taken >> i) & 1u) continue;
      const float l = logit_at(r, row + e);
      if (bid == 0x7fffffff || l > bv) {  // ids ascend per lane: ties keep the lower
        if (!(l != l)) {
          bv = l;
          bid = e;
        }
      }
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, d);
      const int oid = __shfl_xor_sync(0xffffffffu, bid, d);
      if (ov > bv || (ov == bv && oid < bid)) {
        bv = ov;
        bid = oid;
      }
    }
    if (bid == 0x7fffffff) {  // nothing left that compares
      if (lane == 0) report_error(r.status, MOE_ERR_DEVICE_BAD_ID);
      bid = 0;
    } else if ((bid & 31) == lane) {
      taken |= 1u << (bid >> 5);
    }
    if (lane == k) {
      my_v = bv;
      my_id = bid;
    }
  }
  const float v0 = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = lane < r.K ? expf(my_v - v0) : 0.0f;
  float sum = ex;
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, d);
  if (lane < r.K) {
    r.ids[static_cast<long long>(t) * r.K + lane] = my_id;
    r.weights[static_cast<long long>(t) * r.K + lane] = ex / sum;
  }
}

__global__ void __launch_bounds__(256) route_kernel(const RouteArgs r) {
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  for (int t = w; t < r.T; t += nw) route_token(r, t, lane);
}

// Lanes of the warp whose `key` equals this lane's, keys in [0, 2^nbits):
// one ballot per key bit (a warp-level multi-split), the same set
// __match_any_sync gives, at a cost set by the key width.
__device__ __forceinline__ unsigned peers_of(int key, int nbits) {
  unsigned m = 0xffffffffu;
  for (int b = 0; b < nbits; ++b) {
    const int bit = (key >> b) & 1;
    const unsigned bal = __ballot_sync(0xffffffffu, bit);
    m &= bit ? bal : ~bal;
  }
  return m;
}

// Block-wide exclusive scan of two int values per thread (1024 threads).
__device__ __forceinline__ void block_exclusive_scan2(int& a, int& b, int* s_tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int ia = a, ib = b;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int na = __shfl_up_sync(0xffffffffu, ia, d);
    const int nb = __shfl_up_sync(0xffffffffu, ib, d);
    if (lane >= d) {
      ia += na;
      ib += nb;
    }
  }
  if (lane == 31) {
    s_tmp[warp] = ia;
    s_tmp[32 + warp] = ib;
  }
  __syncthreads();
  if (warp == 0) {
    int wa = s_tmp[lane], wb = s_tmp[32 + lane];
    int xa = wa, xb = wb;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int na = __shfl_up_sync(0xffffffffu, xa, d);
      const int nb = __shfl_up_sync(0xffffffffu, xb, d);
      if (lane >= d) {
        xa += na;
        xb += nb;
      }
    }
    s_tmp[lane] = xa - wa;  // exclusive warp prefix
    s_tmp[32 + lane] = xb - wb;
  }
  __syncthreads();
  a = ia - a + s_tmp[warp];
  b = ib - b + s_tmp[32 + warp];
  __syncthreads();
}

// ---------------------------------------------------------------- passes
// The passes of the align, shared by the single-CTA kernel and the kernels
// of the many-CTA path.  A warp owns the flat index range [lo, hi) and a
// histogram row `my_hist` of L counters in shared memory.

// 1. Count the warp's ids per local expert: per 32-id batch, ballots over
// the bits of the id group equal ids and the group's lowest lane adds the
// group size.  Returns whether an id outside [0, E) was seen.
__device__ __forceinline__ bool hist_pass(const AlignArgs& p, int lo, int hi, int lane,
                                          int key_bits, int* my_hist) {
  const int E = p.E, L = p.e_local;
  bool bad = false;
  for (int base0 = lo; base0 < hi; base0 += 32 * kAlignUnroll) {
    int ev[kAlignUnroll];
    load_ids(p.ids, base0, hi, lane, ev);
#pragma unroll
    for (int u = 0; u < kAlignUnroll; ++u) {
      int e = ev[u];
      if (base0 + 32 * u + lane < hi && (e < 0 || e >= E)) {
        bad = true;
        e = -1;
      } else if (e >= 0) {
        e -= p.e_base;  // local expert; another shard's expert is left out
        if (e < 0 || e >= L) e = -1;
      }
      const unsigned peers = peers_of(e + 1, key_bits);
      if (e >= 0 && lane == __ffs(peers) - 1) my_hist[e] += __popc(peers);
      __syncwarp();
    }
  }
  return __any_sync(0xffffffffu, bad);
}

// 3. Stable scatter of the warp's ids: slot = padded_offset[e] + the warp's
// start inside the expert (my_hist on entry) + rank among the equal ids of
// lower lanes; the range and the batches are walked in index order.
__device__ __forceinline__ void scatter_pass(const AlignArgs& p, int lo, int hi, int lane,
                                             int key_bits, const int* s_pad, int* my_hist) {
  const int L = p.e_local;
  for (int base0 = lo; base0 < hi; base0 += 32 * kAlignUnroll) {
    int ev[kAlignUnroll];
    load_ids(p.ids, base0, hi, lane, ev);
#pragma unroll
    for (int u = 0; u < kAlignUnroll; ++u) {
      const int i = base0 + 32 * u + lane;
      int e = ev[u] - p.e_base;
      if (i >= hi || e < 0 || e >= L) {
        if (i < hi) p.inv_perm[i] = -1;  // routed to an expert of another shard
        e = -1;
      }
      const unsigned peers = peers_of(e + 1, key_bits);
      if (e >= 0) {
        const unsigned lower = peers & ((1u << lane) - 1u);
        const int slot = s_pad[e] + my_hist[e] + __popc(lower);
        p.sorted_ids[slot] = i;
        p.inv_perm[i] = slot;
      }
      __syncwarp();
      if (e >= 0 && lane == __ffs(peers) - 1) my_hist[e] += __popc(peers);
      __syncwarp();
    }
  }
}

// 2b. From the expert counts s_cnt: CSR and padded offsets (block scans over
// experts in runs of 1024) into the outputs and s_pad[0..L].  All threads of
// a 1024-thread CTA.
__device__ __forceinline__ void offsets_pass(const AlignArgs& p, const int* s_cnt, int* s_pad,
                                             int* s_tmp, int* s_carry) {
  const int L = p.e_local, bm = p.block_m, tid = threadIdx.x;
  if (tid == 0) {
    s_carry[0] = 0;
    s_carry[1] = 0;
  }
  __syncthreads();
  for (int e0 = 0; e0 < L; e0 += kAlignThreads) {
    const int e = e0 + tid;
    const int c = e < L ? s_cnt[e] : 0;
    int a = c;
    int b = (c + bm - 1) / bm * bm;
    const int carry_a = s_carry[0], carry_b = s_carry[1];
    const int pa = b;  // padded count, kept for the carry update
    block_exclusive_scan2(a, b, s_tmp);
    a += carry_a;
    b += carry_b;
    if (e < L) {
      p.offsets[e] = a;
      p.padded_offsets[e] = b;
      s_pad[e] = b;
    }
    if (e == min(L, e0 + kAlignThreads) - 1) {  // last expert of this chunk
      s_carry[0] = a + c;
      s_carry[1] = b + pa;
    }
    __syncthreads();
  }
  if (tid == 0) {
    p.offsets[L] = s_carry[0];
    p.padded_offsets[L] = s_carry[1];
    s_pad[L] = s_carry[1];
  }
  __syncthreads();
}

// 4. Padding slots of each expert and the tail [padded_offsets[L], cap) get
// the sentinel; block descriptors {expert, m, first slot, valid rows}, and
// {-1, 0, 0, 0} past num_blocks.  All threads of a 1024-thread CTA.
__device__ __forceinline__ void finish_pass(const AlignArgs& p, const int* s_cnt,
                                            const int* s_pad) {
  const int L = p.e_local, bm = p.block_m, na = p.n_assign, tid = threadIdx.x;
  // a warp per expert, its lanes on consecutive padding slots (coalesced)
  for (int e = tid >> 5; e < L; e += kAlignWarps)
    for (int s = s_pad[e] + s_cnt[e] + (tid & 31); s < s_pad[e + 1]; s += 32)
      p.sorted_ids[s] = na;
  for (long long s = s_pad[L] + tid; s < p.cap; s += kAlignThreads) p.sorted_ids[s] = na;
  const int nb = s_pad[L] / bm;
  const long long max_blocks = p.cap / bm;
  int4* bi = reinterpret_cast<int4*>(p.block_info);
  for (long long b = tid; b < max_blocks; b += kAlignThreads) {
    int4 v = make_int4(-1, 0, 0, 0);
    if (b < nb) {
      const int row = static_cast<int>(b) * bm;
      // the expert whose padded range holds `row`: the smallest e with
      // s_pad[e + 1] > row
      int l = 0, h = L;
      while (l < h) {
        const int mid = (l + h) >> 1;
        if (s_pad[mid + 1] > row)
          h = mid;
        else
          l = mid + 1;
      }
      const int m = (row - s_pad[l]) / bm;
      v = make_int4(l, m, row, min(bm, s_cnt[l] - m * bm));
    }
    bi[b] = v;
  }
  if (tid == 0) p.num_blocks[0] = nb;
}

// Batches of at most 32 assignments (decode steps): one warp reads the ids,
// counts them per local expert and ranks each among the lower lanes with
// the same expert (the stable order), then the whole CTA writes the offsets,
// padding and descriptors with the passes above.  A few barriers instead of
// the per-warp histograms' chain of passes: this CTA's time is its barriers
// and memory round trips, not its arithmetic (measured 9.3 us for two ids).
__device__ __forceinline__ void align_small(const AlignArgs& p, int key_bits, int* s_cnt,
                                            int* s_pad, int* s_tmp, int* s_carry, int* s_bad) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int L = p.e_local, na = p.n_assign;
  for (int x = tid; x < L; x += kAlignThreads) s_cnt[x] = 0;
  __syncthreads();
  int e = -1, rank = 0;
  if (tid < 32) {
    const int id = lane < na ? p.ids[lane] : -1;
    const bool bad = lane < na && (id < 0 || id >= p.E);
    if (__any_sync(0xffffffffu, bad) && lane == 0) *s_bad = 1;
    if (lane < na && !bad) e = id - p.e_base;  // local expert
    if (e < 0 || e >= L) e = -1;               // another shard's expert: not listed here
    const unsigned peers = peers_of(e + 1, key_bits);
    rank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && lane == __ffs(peers) - 1) s_cnt[e] = __popc(peers);
  }
  __syncthreads();
  if (*s_bad) {
    if (tid == 0) {
      report_error(p.status, MOE_ERR_DEVICE_BAD_ID);
      p.num_blocks[0] = 0;
    }
    return;
  }
  for (int x = tid; x < L; x += kAlignThreads) p.counts[x] = s_cnt[x];
  offsets_pass(p, s_cnt, s_pad, s_tmp, s_carry);
  if (tid < na) {
    if (e >= 0) {
      const int slot = s_pad[e] + rank;
      p.sorted_ids[slot] = tid;
      p.inv_perm[tid] = slot;
    } else {
      p.inv_perm[tid] = -1;
    }
  }
  finish_pass(p, s_cnt, s_pad);
}

// ---------------------------------------------------------------- kernels

// The whole align in one CTA of 32 warps (batches up to a few ten thousand
// ids, and the routing of batches up to 1024 tokens).
__global__ void __launch_bounds__(kAlignThreads, 1) align_kernel(const AlignArgs p) {
  extern __shared__ int sm[];
  const int L = p.e_local;  // experts of this shard: [e_base, e_base + L)
  const int key_bits = 32 - __clz(L);  // keys e + 1 in [0, L], 0 = not counted here
  int* hist = sm;                        // [kAlignWarps][L]
  int* s_pad = hist + kAlignWarps * L;   // [L + 1] padded offsets
  int* s_cnt = s_pad + L + 1;            // [L]
  __shared__ int s_tmp[64];
  __shared__ int s_bad;
  __shared__ int s_carry[2];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int na = p.n_assign;

  pdl_wait();  // ids written by the routing kernel, when it ran first
  pdl_launch_dependents();
  if (tid == 0) s_bad = 0;
  if (na > 32)
    for (int i = tid; i < kAlignWarps * L; i += kAlignThreads) hist[i] = 0;
  // 0. routing of small batches, in this CTA: a warp per token; the ids it
  //    writes are read back below after the barrier
  if (p.route.logits != nullptr)
    for (int t = warp; t < p.route.T; t += kAlignWarps) route_token(p.route, t, lane);
  __syncthreads();
  if (na <= 32) {
    align_small(p, key_bits, s_cnt, s_pad, s_tmp, s_carry, &s_bad);
    return;
  }

  // chunk of warp w: [w*chunk, min(na, (w+1)*chunk)), chunk a multiple of 32
  const int chunk = ((na + kAlignWarps - 1) / kAlignWarps + 31) & ~31;
  const int lo = warp * chunk;
  const int hi = min(na, lo + chunk);
  int* my_hist = hist + warp * L;

  if (hist_pass(p, lo, hi, lane, key_bits, my_hist) && lane == 0) s_bad = 1;
  __syncthreads();
  if (s_bad) {
    if (tid == 0) {
      report_error(p.status, MOE_ERR_DEVICE_BAD_ID);
      p.num_blocks[0] = 0;
    }
    return;
  }

  // 2. per-expert scan over warps: each warp's start inside the expert
  for (int e = tid; e < L; e += kAlignThreads) {
    int run = 0;
    for (int w = 0; w < kAlignWarps; ++w) {
      const int c = hist[w * L + e];
      hist[w * L + e] = run;
      run += c;
    }
    s_cnt[e] = run;
    p.counts[e] = run;
  }
  offsets_pass(p, s_cnt, s_pad, s_tmp, s_carry);
  scatter_pass(p, lo, hi, lane, key_bits, s_pad, my_hist);
  finish_pass(p, s_cnt, s_pad);
}

// Many-CTA path for large batches, CTAs of 8 warps: (A) per-warp histograms
// of fixed-size chunks into the scratch rows whist[w][0..L), and each CTA's
// totals into ctot[c][0..L); (B) one CTA turns the CTA totals into
// exclusive per-expert bases (a scan over CTAs), and writes the counts,
// offsets, padding and block descriptors; (C) each warp starts from its
// CTA's base plus the counts of the lower warps of its CTA and scatters its
// chunk.  A bad id: A sets num_blocks = -1 (the host cleared it first), B
// reports it, writes num_blocks = 0 and padded_offsets[0] = -1, and C then
// writes nothing.
constexpr int kMultiWarps = 8;

__global__ void __launch_bounds__(kMultiWarps * 32) align_hist_kernel(const AlignArgs p,
                                                                     int32_t* whist,
                                                                     int32_t* ctot, int chunk) {
  extern __shared__ int sm[];
  const int L = p.e_local, key_bits = 32 - __clz(L);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gw = blockIdx.x * kMultiWarps + warp;
  pdl_wait();
  pdl_launch_dependents();
  int* my_hist = sm + warp * L;
  for (int i = lane; i < L; i += 32) my_hist[i] = 0;
  __syncwarp();
  const long long lo = static_cast<long long>(gw) * chunk;
  const int hi = static_cast<int>(min(static_cast<long long>(p.n_assign), lo + chunk));
  const bool bad = lo < hi ? hist_pass(p, static_cast<int>(lo), hi, lane, key_bits, my_hist)
                           : false;
  if (bad && lane == 0) p.num_blocks[0] = -1;
  __syncwarp();
  for (int i = lane; i < L; i += 32) whist[static_cast<long long>(gw) * L + i] = my_hist[i];
  __syncthreads();
  for (int e = threadIdx.x; e < L; e += blockDim.x) {
    int sum = 0;
#pragma unroll
    for (int w = 0; w < kMultiWarps; ++w) sum += sm[w * L + e];
    ctot[static_cast<long long>(blockIdx.x) * L + e] = sum;
  }
}

__global__ void __launch_bounds__(kAlignThreads, 1) align_scan_kernel(const AlignArgs p,
                                                                     int32_t* ctot, int nctas) {
  extern __shared__ int sm[];
  const int L = p.e_local, tid = threadIdx.x;
  int* s_pad = sm;             // [L + 1]
  int* s_cnt = s_pad + L + 1;  // [L]
  __shared__ int s_tmp[64];
  __shared__ int s_carry[2];
  pdl_wait();
  pdl_launch_dependents();
  if (*reinterpret_cast<volatile int32_t*>(p.num_blocks) < 0) {
    if (tid == 0) {
      report_error(p.status, MOE_ERR_DEVICE_BAD_ID);
      p.num_blocks[0] = 0;
      p.padded_offsets[0] = -1;
    }
    return;
  }
  // 2. per expert, the exclusive scan of the CTAs' totals in CTA order
  for (int e = tid; e < L; e += kAlignThreads) {
    int run = 0;
    int c = 0;
    for (; c + 8 <= nctas; c += 8) {
      int v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = ctot[static_cast<long long>(c + u) * L + e];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        ctot[static_cast<long long>(c + u) * L + e] = run;
        run += v[u];
      }
    }
    for (; c < nctas; ++c) {
      const int v = ctot[static_cast<long long>(c) * L + e];
      ctot[static_cast<long long>(c) * L + e] = run;
      run += v;
    }
    s_cnt[e] = run;
    p.counts[e] = run;
  }
  offsets_pass(p, s_cnt, s_pad, s_tmp, s_carry);
  finish_pass(p, s_cnt, s_pad);
}

__global__ void __launch_bounds__(kMultiWarps * 32) align_scatter_kernel(
    const AlignArgs p, const int32_t* whist, const int32_t* ctot, int chunk) {
  extern __shared__ int sm[];
  const int L = p.e_local, key_bits = 32 - __clz(L);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gw = blockIdx.x * kMultiWarps + warp;
  int* s_pad = sm;                          // [L + 1]
  int* my_hist = sm + (L + 1) + warp * L;   // this warp's starts
  pdl_wait();
  pdl_launch_dependents();
  if (p.padded_offsets[0] != 0) return;  // bad ids: nothing to scatter
  for (int i = threadIdx.x; i <= L; i += blockDim.x) s_pad[i] = p.padded_offsets[i];
  const long long lo = static_cast<long long>(gw) * chunk;
  const int hi = static_cast<int>(min(static_cast<long long>(p.n_assign), lo + chunk));
  // start of this warp inside expert e: the CTA's base plus the counts of
  // the CTA's lower warps
  const int32_t* wrow = whist + static_cast<long long>(blockIdx.x) * kMultiWarps * L;
  for (int e = lane; e < L; e += 32) {
    int start = 0;
    if (lo < hi) {
      start = ctot[static_cast<long long>(blockIdx.x) * L + e];
      for (int w = 0; w < warp; ++w) start += wrow[w * L + e];
    }
    my_hist[e] = start;
  }
  __syncthreads();
  if (lo < hi) scatter_pass(p, static_cast<int>(lo), hi, lane, key_bits, s_pad, my_hist);
}

}  // namespace

size_t align_smem_bytes(int L) {
  return sizeof(int) * (static_cast<size_t>(kAlignWarps) * L + (L + 1) + L);
}

cudaError_t launch_route(const RouteArgs& r, cudaStream_t s) {
  const int blocks = static_cast<int>(std::min<long long>((r.T + 7) / 8, 152ll * 8));
  route_kernel<<<blocks, 256, 0, s>>>(r);
  return cudaGetLastError();
}

// Ids per warp: 256, or more once the batch would need over 32 CTAs per SM
// (the scratch stays below 4864 warps' rows).
int align_multi_chunk(long long n_assign) {
  constexpr long long kMaxWarps = 152ll * 32;
  const long long c = (n_assign + kMaxWarps - 1) / kMaxWarps;
  return static_cast<int>(std::max(256ll, (c + 31) / 32 * 32));
}

int align_multi_warps(long long n_assign) {
  const long long chunk = align_multi_chunk(n_assign);
  return static_cast<int>((n_assign + chunk - 1) / chunk);
}

size_t align_multi_scratch_ints(long long n_assign, int e_local) {
  const int nwarps = align_multi_warps(n_assign);
  const int nctas = (nwarps + kMultiWarps - 1) / kMultiWarps;
  // whist rows for every warp of every CTA, then the CTA totals
  return static_cast<size_t>(nctas) * (kMultiWarps + 1) * static_cast<size_t>(e_local);
}

cudaError_t launch_align_multi(const AlignArgs& a, int32_t* scratch, cudaStream_t s) {
  const int chunk = align_multi_chunk(a.n_assign);
  const int nwarps = align_multi_warps(a.n_assign);
  const int nctas = (nwarps + kMultiWarps - 1) / kMultiWarps;
  const int L = a.e_local;
  int32_t* whist = scratch;
  int32_t* ctot = scratch + static_cast<size_t>(nctas) * kMultiWarps * L;
  cudaError_t err = cudaMemsetAsync(a.num_blocks, 0, sizeof(int32_t), s);
  if (err != cudaSuccess) return err;
  const size_t smem_a = sizeof(int) * kMultiWarps * static_cast<size_t>(L);
  const size_t smem_b = sizeof(int) * (2 * static_cast<size_t>(L) + 1);
  const size_t smem_c = sizeof(int) * (kMultiWarps * static_cast<size_t>(L) + L + 1);
  if ((err = cudaFuncSetAttribute(align_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(smem_a))) != cudaSuccess ||
      (err = cudaFuncSetAttribute(align_scatter_kernel,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(smem_c))) != cudaSuccess)
    return err;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pdl_config(dim3(nctas), dim3(kMultiWarps * 32), smem_a, s, attr);
  if ((err = cudaLaunchKernelEx(&cfg, align_hist_kernel, a, whist, ctot, chunk)) != cudaSuccess)
    return err;
  cfg = pdl_config(dim3(1), dim3(kAlignThreads), smem_b, s, attr);
  if ((err = cudaLaunchKernelEx(&cfg, align_scan_kernel, a, ctot, nctas)) != cudaSuccess)
    return err;
  cfg = pdl_config(dim3(nctas), dim3(kMultiWarps * 32), smem_c, s, attr);
  return cudaLaunchKernelEx(&cfg, align_scatter_kernel, a, static_cast<const int32_t*>(whist),
                            static_cast<const int32_t*>(ctot), chunk);
}

cudaError_t launch_align(const AlignArgs& a, cudaStream_t s) {
  const size_t smem = align_smem_bytes(a.e_local);
  cudaError_t err = cudaFuncSetAttribute(align_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = pdl_config(dim3(1), dim3(kAlignThreads), smem, s, attr);
  return cudaLaunchKernelEx(&cfg, align_kernel, a);
}

}  // namespace moe
