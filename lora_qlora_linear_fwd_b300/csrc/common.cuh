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

// Persistent schedules over the output tiles (m-block, n-tile):
//  * grid (contiguous == 0): worker c owns m-blocks m = cm + gm*i and
//    n-tiles nt = cn + gn*j (cm = c % gm, cn = c / gm).  All workers run on a
//    compact gm x gn block of tiles at any time (operands stay in L2).
//  * contiguous (contiguous == 1): worker c owns the tiles
//    [c*T/W, (c+1)*T/W) of the m-major order (T tiles, W workers), which
//    balances the tile count to within one per worker.
// Either way a worker walks n-tiles of one m-block in a row, so the rank-r
// down-projection is formed once per m-block (and projection) and reused.
struct Schedule {
  int gm, gn;
  int m_blocks, n_tiles;
  int contiguous;
  int workers;
};

// Tile iterator shared by every role of a persistent CTA (or CTA pair).
struct TileIter {
  int cm, cn, gm, gn, m_blocks, n_tiles;
  int mi, nj;         // grid: current (i, j)
  int t, t_begin, t_end;
  int contiguous;
  __device__ void init(const Schedule &s, int worker) {
    gm = s.gm;
    gn = s.gn;
    m_blocks = s.m_blocks;
    n_tiles = s.n_tiles;
    contiguous = s.contiguous;
    cm = worker % gm;
    cn = worker / gm;
    mi = 0;
    nj = 0;
    const long long total = (long long)m_blocks * n_tiles;
    t_begin = (int)(total * worker / s.workers);
    t_end = (int)(total * (worker + 1) / s.workers);
    t = t_begin;
  }
  __device__ bool valid() const {
    return contiguous ? t < t_end : (cm + gm * mi < m_blocks && cn < n_tiles);
  }
  __device__ int m() const { return contiguous ? t / n_tiles : cm + gm * mi; }
  __device__ int nt() const { return contiguous ? t % n_tiles : cn + gn * nj; }
  __device__ bool first_of_m() const {
    return contiguous ? (t == t_begin || t % n_tiles == 0) : nj == 0;
  }
  __device__ void next() {
    if (contiguous) {
      ++t;
      return;
    }
    ++nj;
    if (cn + gn * nj >= n_tiles) {
      nj = 0;
      ++mi;
    }
  }
};

}  // namespace lora
