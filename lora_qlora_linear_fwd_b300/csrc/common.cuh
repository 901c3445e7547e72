// Shared pieces of the kernels: tile geometry, parameter blocks, schedule.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace lora {

constexpr int kBM = 128;       // rows of an output tile (tensor-core M)
constexpr int kBK = 64;        // K elements per pipeline stage (one 128-B swizzle row)
constexpr int kMaxGroups = 2;  // projections sharing one x in a single launch

// Dynamic shared memory available to one CTA on sm_100-class parts.
constexpr int kSmemLimit = 232448;

// Persistent schedule over the output tiles (m-block, n-tile).  Worker w
// takes tiles t = w, w + W, w + 2W, ... of a grouped raster order: the
// order sweeps `group_m` m-blocks for one n-tile, then the same m-blocks for
// the next n-tile, and moves on to the next group of m-blocks when every
// n-tile is done.  The W tiles in flight at any moment then cover about
// group_m m-blocks and W / group_m n-tiles, whose x rows and W rows stay in
// L2 while the neighbouring workers reuse them.  Tiles are independent (the
// rank-r term arrives as extra K-blocks), so any order is valid.
struct Schedule {
  int m_blocks, n_tiles;
  int group_m;
  int workers;
};

// Tile iterator shared by every role of a persistent CTA (or CTA pair).
struct TileIter {
  int t, total, step, n_tiles, m_blocks, group_m;
  int m_, nt_;
  __device__ void decode() {
    const int span = group_m * n_tiles;
    const int g = t / span;
    const int first = g * group_m;
    const int gsize = min(group_m, m_blocks - first);
    const int rr = t - g * span;
    m_ = first + rr % gsize;
    nt_ = rr / gsize;
  }
  __device__ void init(const Schedule &s, int worker) {
    n_tiles = s.n_tiles;
    m_blocks = s.m_blocks;
    group_m = s.group_m;
    total = m_blocks * n_tiles;
    step = s.workers;
    t = worker;
    if (t < total) decode();
  }
  __device__ bool valid() const { return t < total; }
  __device__ int m() const { return m_; }
  __device__ int nt() const { return nt_; }
  __device__ void next() {
    t += step;
    if (t < total) decode();
  }
};

}  // namespace lora
