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

// Persistent schedule: CTA c owns m-blocks  m = cm + gm*i  and n-tiles
// nt = cn + gn*j  (cm = c % gm, cn = c / gm).  All concurrently running CTAs
// work on a compact gm x gn block of output tiles (operands stay in L2) and a
// CTA keeps its m-block for all its n-tiles, so the rank-r down-projection
// x·Aᵀ is computed once per m-block and reused.
struct Schedule {
  int gm, gn;
  int m_blocks, n_tiles;
};

// Tile iterator shared by every role of a persistent CTA.
struct TileIter {
  int cm, cn, gm, gn, m_blocks, n_tiles;
  int mi, nj;  // current (i, j)
  __device__ void init(const Schedule &s, int cta) {
    gm = s.gm;
    gn = s.gn;
    m_blocks = s.m_blocks;
    n_tiles = s.n_tiles;
    cm = cta % gm;
    cn = cta / gm;
    mi = 0;
    nj = 0;
  }
  // Returns false when the CTA has no more tiles.
  __device__ bool valid() const { return cm + gm * mi < m_blocks && cn < n_tiles; }
  __device__ int m() const { return cm + gm * mi; }
  __device__ int nt() const { return cn + gn * nj; }
  __device__ bool first_of_m() const { return nj == 0; }
  __device__ void next() {
    ++nj;
    if (cn + gn * nj >= n_tiles) {
      nj = 0;
      ++mi;
    }
  }
};

}  // namespace lora
