// sched.cuh -- the persistent tile schedule shared by the grouped GEMMs:
// tile index -> (M block, N tile, K split) in bands of N tiles, the K range
// of a split, and a bounded drain wait used when a kernel gives up.
#pragma once

#include "internal.h"
#include "ptx.cuh"

namespace moe {

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
