// Work units of the forward kernels (bf16 and e4m3): one CTA owns 256 query rows of one
// (batch, head), i.e. two 128-row tiles, and walks the key blocks that either tile needs.
// Key blocks wholly above the causal diagonal, past the sequence's key length, or zero in
// the 128 x 128 block mask are skipped (course week 13, step 2; reading guide, "Extension:
// block-sparse FlashAttention").
#pragma once

#include "fa_internal.cuh"

namespace fa {
namespace units {

constexpr int kBlk = 128;  // rows of a Q tile / keys of a K,V tile

struct Unit {
  int bh, q0, L, nb;
};

// Does query tile t (rows q0 + 128t ...) of this unit need key block j?
__device__ __forceinline__ bool need(const Problem& p, const Unit& u, int t, int j) {
  const int r0 = u.q0 + t * kBlk;
  if (r0 >= p.N) return false;
  if (j * kBlk >= u.L) return false;
  if (p.causal && j * kBlk > r0 + kBlk - 1) return false;
  if (p.blockmask && !p.blockmask[(r0 / kBlk) * u.nb + j]) return false;
  return true;
}

__device__ __forceinline__ int key_blocks(const Problem& p, const Unit& u) {
  int jend = (u.L + kBlk - 1) / kBlk;
  if (p.causal) {
    const int last_row = min(u.q0 + 2 * kBlk, p.N) - 1;
    jend = min(jend, last_row / kBlk + 1);
  }
  return jend;
}

__device__ __forceinline__ int next_any(const Problem& p, const Unit& u, int j, int jend) {
  for (++j; j < jend; ++j)
    if (need(p, u, 0, j) || need(p, u, 1, j)) return j;
  return -1;
}

// The unit of CTA blockIdx.x: heavy (late, causal) query blocks first.
__device__ __forceinline__ Unit make_unit(const Problem& p) {
  const int nqb = (p.N + 2 * kBlk - 1) / (2 * kBlk);
  const int bhs = p.B * p.H;
  Unit u;
  u.bh = blockIdx.x % bhs;
  u.q0 = (nqb - 1 - static_cast<int>(blockIdx.x / bhs)) * 2 * kBlk;
  int L = p.N;
  if (p.kv_len) {
    L = p.kv_len[u.bh / p.H];
    L = L < 0 ? 0 : (L > p.N ? p.N : L);
  }
  u.L = L;
  u.nb = (p.N + kBlk - 1) / kBlk;
  return u;
}

}  // namespace units
}  // namespace fa
