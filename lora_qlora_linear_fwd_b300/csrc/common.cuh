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
// n-tile is done; odd groups sweep the n-tiles backwards, so the wave that
// crosses into a new group meets the W rows the last one left in L2.  The W
// tiles in flight at any moment then cover about group_m m-blocks and
// W / group_m n-tiles, whose x rows and W rows stay in L2 while the
// neighbouring workers reuse them.  Tiles are independent (the rank-r term
// arrives as extra K-blocks), so any order is valid.
//
// Contiguous form (`contiguous` set): the tiles are ordered m-block by
// m-block (all n-tiles of an m-block in a row) and worker w takes the range
// [total·w/W, total·(w+1)/W) of that order, so it meets each of its m-blocks
// in one run of consecutive tiles (a segment).  The forward with the
// down-projection in the GEMM forms x·Aᵀ once per segment, on its first tile.
struct Schedule {
  int m_blocks, n_tiles;
  int group_m;
  int workers;
  int contiguous;
};

// Tile iterator shared by every role of a persistent CTA (or CTA pair).
struct TileIter {
  int t, total, step, end, n_tiles, m_blocks, group_m;
  int m_, nt_;
  bool contig, first;
  __device__ void decode() {
    if (contig) {
      m_ = t / n_tiles;
      nt_ = t - m_ * n_tiles;
      return;
    }
    const int span = group_m * n_tiles;
    const int g = t / span;
    const int first_m = g * group_m;
    const int gsize = min(group_m, m_blocks - first_m);
    const int rr = t - g * span;
    m_ = first_m + rr % gsize;
    nt_ = (g & 1) ? n_tiles - 1 - rr / gsize : rr / gsize;
  }
  __device__ void init(const Schedule &s, int worker) {
    n_tiles = s.n_tiles;
    m_blocks = s.m_blocks;
    group_m = s.group_m;
    total = m_blocks * n_tiles;
    contig = s.contiguous != 0;
    first = true;
    if (contig) {
      t = (int)((long long)total * worker / s.workers);
      end = (int)((long long)total * (worker + 1) / s.workers);
      step = 1;
    } else {
      t = worker;
      end = total;
      step = s.workers;
    }
    if (t < end) decode();
  }
  __device__ bool valid() const { return t < end; }
  __device__ int m() const { return m_; }
  __device__ int nt() const { return nt_; }
  // first tile of a run of tiles of one m-block (contiguous form only)
  __device__ bool seg_start() const { return contig && (first || nt_ == 0); }
  // last tile of such a run
  __device__ bool seg_last() const { return contig && (t + 1 >= end || nt_ + 1 == n_tiles); }
  __device__ void next() {
    t += step;
    first = false;
    if (t < end) decode();
  }
};

}  // namespace lora
