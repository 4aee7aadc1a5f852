// sched.cuh -- the persistent tile schedule shared by the grouped GEMMs:
// the band width of the pair GEMMs, tile index -> (M block, N tile, K split)
// in bands of N tiles, the K range of a split, and a bounded drain wait used
// when a kernel gives up.
#pragma once

#include "internal.h"
#include "ptx.cuh"

namespace moe {

// Weight tiles per band of the pair GEMMs' tile order (host side; blocks x
// the band's weight tiles, block-major).  A block's token rows are read once
// per band, and the blocks of one expert reuse a weight tile only while they
// run in the same round of the persistent grid, which a wide band spreads
// out.  Gate/up: with many weight tiles (Mixtral-shaped: 112) a band of 16
// reads the token rows 7 times instead of 14 (DRAM traffic 1.43x -> 1.26-1.32x
// of the algorithmic bytes over three captures, 1 % faster); with few (DeepSeek-V3-shaped: 16) a
// band of 8 measured faster.  Down: a band of 16 measured 1-3 % faster on
// every shape.
inline int gate_up_band(int n_tiles) {
  const int band = n_tiles >= 64 ? 16 : 8;
  return n_tiles < band ? n_tiles : band;
}
inline int down_band(int n_tiles) { return n_tiles < 16 ? n_tiles : 16; }

struct Tile {
  int mb, nt, split;
};

template <class Args>
__device__ __forceinline__ Tile decode_tile(int tile, int num_blocks, const Args& a) {
  Tile t;
  const int per_split = num_blocks * a.n_tiles;
  t.split = tile / per_split;
  const int rem = tile - t.split * per_split;
  const int band = a.band;
  const int full_bands = a.n_tiles / band;
  const int band_tiles = num_blocks * band;
  const int b = rem / band_tiles;
  if (b < full_bands) {
    const int w = rem - b * band_tiles;
    t.mb = w / band;
    t.nt = b * band + w % band;
  } else {
    const int tail = a.n_tiles - full_bands * band;
    const int w = rem - full_bands * band_tiles;
    t.mb = w / tail;
    t.nt = full_bands * band + w % tail;
  }
  return t;
}

template <class Args>
__device__ __forceinline__ void split_range(const Args& a, int split, int& kb, int& ke) {
  kb = static_cast<int>((static_cast<long long>(a.k_tiles) * split) / a.splits);
  ke = static_cast<int>((static_cast<long long>(a.k_tiles) * (split + 1)) / a.splits);
}

// Wait without looking at the abort flag (used only while draining).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > timeout_ns) return;
  }
}

}  // namespace moe
