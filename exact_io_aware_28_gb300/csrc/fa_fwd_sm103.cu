// Forward attention on sm_103a tensor cores (tcgen05 + TMA), bf16 in, fp32 accumulate.
//
// What it computes is the tiled forward with a running (max, sum) state: for each block
// of 128 query rows and each block j of 128 keys, S_ij = Q_i K_j^T, the running row
// maximum and row sum are updated and O_i is rescaled and accumulated with P_ij V_j
// (FlashAttention reading guide, arXiv 2205.14135, "Method", steps 1-4; answer page
// "How FlashAttention works for training", section 2.1).  O is kept unnormalised and
// divided by the row sum once at the end (course week 13, step 2 keeps the unnormalised
// accumulator and multiplies it by e^{m_old - m_new} on a new maximum); the only other
// output is the per-row logsumexp.  Key blocks wholly above the causal diagonal and zero
// blocks of the 128 x 128 block mask are never loaded or multiplied (course week 13,
// step 2; reading guide, "Extension: block-sparse FlashAttention").
//
// GB300 mapping (one CTA = 256 query rows of one (batch, head) = two 128-row tiles):
//   warp 0        TMA producer: Q0, Q1 once, then K_j, V_j through a ring of stages;
//   warp 1        MMA issuer (one thread): S_t = Q_t K_j^T into TMEM, O_t += P_t V_j with P
//                 read from TMEM; issue order PV0(j), S0(j+1), PV1(j), S1(j+1) keeps the
//                 tensor pipe busy while each softmax warpgroup works on its own tile;
//   warp 2        tensor-memory allocation;
//   warps 4-11    softmax: all eight warps work on each tile in turn (tile 0, then tile 1,
//                 for every key block), a thread holding two rows of 32 keys through the
//                 16-lane TMEM shapes; scores read with tcgen05.ld, exp2 with scale*log2(e)
//                 folded in, P written back as bf16 over the first 64 columns of the tile's S
//                 region, O rescaled in TMEM only when the running maximum grows by more than
//                 2^8 (exact: the final division uses the same reference maximum);
//   epilogue      the softmax warps read O from TMEM, divide by the row sum and store bf16.
// Tensor memory (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+d), O1 [384,384+d).
// Every mbarrier wait is bounded; on expiry the CTA records FA_ERR_TIMEOUT and exits cleanly.
#include <atomic>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "fa_fwd_units.cuh"
#include "fa_internal.cuh"
#include "fa_philox.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

using namespace ptx;
using namespace units;

constexpr int kSub = 128 * 128;         // bytes of a [128 rows][64 bf16] 128B-swizzled subtile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only past a 256x growth
constexpr int kThreads = 384;

template <int D>
struct Cfg {
  static constexpr int NSUB = D / 64;
  static constexpr int TILE = NSUB * kSub;
  static constexpr int NSTAGE = D == 128 ? 4 : 8;
  static constexpr int SMEM = 1024 + 2 * TILE + NSTAGE * TILE + 256;
};

struct Bars {
  uint64_t q_full;
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
  uint64_t o_staged[2];  // a tile of O is in shared memory, ready for the TMA store
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int never;  // stays 0: waits that must not be cut short by an abort
};
static_assert(sizeof(Bars) <= 256, "barrier block");

// DROP: dropout on P (the generator bytes of fa_philox.cuh); the row sums keep every term.
template <int D, bool DROP>
__global__ void __launch_bounds__(kThreads, 1)
fwd_sm103_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                 const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mo,
                 float* __restrict__ lse, Problem p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = base;                       // [2][TILE]
  uint8_t* sKV = base + 2 * C::TILE;        // [NSTAGE][TILE]
  Bars* bars = reinterpret_cast<Bars*>(sKV + C::NSTAGE * C::TILE);
  volatile int* abort_flag = &bars->abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // Work unit: groups of G heads, G as large as keeps a group's K and V (4 N d bytes per
  // head) within 64 MiB of L2, so that co-resident CTAs read each K, V tile from DRAM about
  // once; in each group heavy (late, causal) query blocks first, the group's heads fastest.
  // The dropout instance keeps all heads in one group, which measured faster for it.
  const int nqb = (p.N + 2 * kBlk - 1) / (2 * kBlk);
  const int bhs = p.B * p.H;
  Unit u;
  {
    const long long per_head = 4ll * p.N * D;
    const int G = DROP ? bhs
                       : static_cast<int>(max(1ll, min(static_cast<long long>(bhs),
                                                       (64ll << 20) / per_head)));
    const int b = blockIdx.x, g = b / (G * nqb), r = b - g * G * nqb;
    const int Gg = min(G, bhs - g * G);
    u.bh = g * G + r % Gg;
    u.q0 = (nqb - 1 - r / Gg) * 2 * kBlk;
  }
  u.nb = (p.N + kBlk - 1) / kBlk;

  if (tid == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < C::NSTAGE; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 2);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 2 * kBlk);
      mbar_init(&bars->o_done[t], 1);
      mbar_init(&bars->o_staged[t], 2 * kBlk);
    }
    mbar_init(&bars->drain, 2);
    bars->abort = 0;
    bars->never = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = bars->tmem_base;
  // Set-up done; global memory (the key lengths included) only after the previous kernel in
  // the stream has completed.
  griddep_wait();
  griddep_launch_dependents();
  {
    int L = p.N;
    if (p.kv_len) {
      const int b = u.bh / p.H;
      L = p.kv_len[b];
      L = L < 0 ? 0 : (L > p.N ? p.N : L);
    }
    u.L = L;
  }
  const int jend = key_blocks(p, u);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mk);
      tma_prefetch_desc(&mv);
      mbar_arrive_expect_tx(&bars->q_full, 2 * C::TILE);
      for (int t = 0; t < 2; ++t)
        for (int s = 0; s < C::NSUB; ++s)
          tma_load_3d(sQ + t * C::TILE + s * kSub, &mq, &bars->q_full, 64 * s, u.q0 + t * kBlk,
                      u.bh);
      int stage = 0, round = 0;
      bool ok = true;
      for (int j = next_any(p, u, -1, jend); ok && j >= 0; j = next_any(p, u, j, jend)) {
        for (int which = 0; which < 2 && ok; ++which) {
          ok = mbar_wait(&bars->kv_empty[stage], (round & 1) ^ 1, abort_flag, p.err, p.wait_ns);
          if (!ok) break;
          mbar_arrive_expect_tx(&bars->kv_full[stage], C::TILE);
          const CUtensorMap* m = which == 0 ? &mk : &mv;
          for (int s = 0; s < C::NSUB; ++s)
            tma_load_3d(sKV + stage * C::TILE + s * kSub, m, &bars->kv_full[stage], 64 * s,
                        j * kBlk, u.bh);
          if (++stage == C::NSTAGE) {
            stage = 0;
            ++round;
          }
        }
      }
    }
  } else if (warp == 1 || warp == 3) {
    // ------------------------------------------------------------ MMA issuers
    // One thread per query tile: warp 1 issues tile 0's MMAs, warp 3 tile 1's.
    // tcgen05.mma returns only once the tensor pipe takes the instruction, so a single
    // issuer runs in step with the pipe and every wait it makes between two groups is a
    // bubble; with one issuer per tile the pipe takes the other tile's MMAs meanwhile.
    // Each issuer walks the whole K/V ring (both tiles release every slot, so kv_empty
    // counts two arrivals) and, per key block j, issues O_t += P_t V_j after its softmax
    // handshake, then S_t = Q_t K_{j+1}^T.  In-order execution of one thread's MMAs keeps
    // S_t(j+1) from overwriting P_t(j) before the P V product has read it.  Descriptors
    // are built once and advanced by adding (offset >> 4) to the start-address field.
    if (lane == 0) {
      const int t = warp == 1 ? 0 : 1;
      constexpr uint32_t idS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idO = idesc_bf16(128, D, false, true);
      constexpr uint64_t kTileD = C::TILE >> 4;
      const uint64_t dQ = sw128_desc(smem_u32(sQ + t * C::TILE), 16, 1024);  // K-major Q_t
      const uint64_t dK = sw128_desc(smem_u32(sKV), 16, 1024);     // K-major K stages
      const uint64_t dV = sw128_desc(smem_u32(sKV), kSub, 1024);   // MN-major V stages
      const uint32_t tS = tb + t * 128, tO = tb + 256 + t * 128;
      int last = -1;
      for (int j = jend - 1; j >= 0 && last < 0; --j)
        if (need(p, u, t, j)) last = j;
      int cs = 0;
      uint32_t cr = 0;  // ring slot and the parity of its current fill
      int npv = 0;
      bool ok = mbar_wait(&bars->q_full, 0, abort_flag, p.err, p.wait_ns);
      tc_fence_after();
      // S_t = Q_t K^T of ring slot `slot`: groups of four MMAs, each group's descriptors
      // built before its first MMA issues, so the four go out back to back.
      auto issue_s = [&](int slot) {
        const uint64_t dKs = dK + static_cast<uint64_t>(slot) * kTileD;
#pragma unroll
        for (int g = 0; g < D / 64; ++g) {
          uint64_t da[4], db[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int kk = 4 * g + k;
            const uint64_t off = static_cast<uint64_t>(((kk >> 2) * kSub + (kk & 3) * 32) >> 4);
            da[k] = dQ + off;
            db[k] = dKs + off;
          }
          mma_ss_x4(tS, da, db, idS, g > 0 ? 1u : 0u);
        }
        mma_commit(&bars->s_full[t]);
      };
      int j = next_any(p, u, -1, jend);
      if (ok && j >= 0) {
        const int ks = cs;
        ok = mbar_wait(&bars->kv_full[ks], cr & 1, abort_flag, p.err, p.wait_ns);
        if (++cs == C::NSTAGE) { cs = 0; ++cr; }
        tc_fence_after();
        if (ok) {
          if (need(p, u, t, j)) issue_s(ks);
          mma_commit(&bars->kv_empty[ks]);
        }
      }
      while (ok && j >= 0) {
        const int jn = next_any(p, u, j, jend);
        // V_j, then K of the next key block: the producer loads them in this order.
        const int vs = cs;
        ok = mbar_wait(&bars->kv_full[vs], cr & 1, abort_flag, p.err, p.wait_ns);
        if (++cs == C::NSTAGE) { cs = 0; ++cr; }
        int ks = -1;
        if (ok && jn >= 0) {
          ks = cs;
          ok = mbar_wait(&bars->kv_full[ks], cr & 1, abort_flag, p.err, p.wait_ns);
          if (++cs == C::NSTAGE) { cs = 0; ++cr; }
        }
        if (!ok) break;
        tc_fence_after();
        if (need(p, u, t, j)) {
          ok = mbar_wait(&bars->p_full[t], npv & 1, abort_flag, p.err, p.wait_ns);
          tc_fence_after();
          if (!ok) break;
          const uint64_t dVs = dV + static_cast<uint64_t>(vs) * kTileD;
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            uint32_t ta[4];
            uint64_t db[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              ta[k] = tS + 8 * (4 * g + k);
              db[k] = dVs + static_cast<uint64_t>((2048 * (4 * g + k)) >> 4);
            }
            mma_ts_x4(tO, ta, db, idO, (npv > 0 || g > 0) ? 1u : 0u);
          }
          ++npv;
          if (j == last) mma_commit(&bars->o_done[t]);
        }
        mma_commit(&bars->kv_empty[vs]);
        if (jn >= 0) {
          if (need(p, u, t, jn)) issue_s(ks);
          mma_commit(&bars->kv_empty[ks]);
        }
        j = jn;
      }
      // Drain: every MMA issued by either thread has completed before tensor memory is
      // released (the barrier counts one arrival per issuer).
      mma_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, &bars->never, nullptr, p.wait_ns);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax warps
    // All eight warps work on each tile in turn (tile 0 then tile 1 for every key block),
    // so a tile's softmax runs on two warps per SM sub-partition.  Warp 4 + q + 4h owns
    // rows 32q + 16h + [0, 16) of both tiles through the 16-lane TMEM shapes: thread t holds
    // rows A = 32q + 16h + t/4 and B = A + 8, keys 8c + 2(t%4) + {0, 1} for c = 0..15.  The
    // four threads of a row combine their row maxima with two shuffles; row sums stay
    // partial per thread until the epilogue.
    const int q4 = warp & 3, h = (warp - 4) >> 2, t4 = lane & 3;
    const int rA = 32 * q4 + 16 * h + (lane >> 2), rB = rA + 8;   // rows within a tile
    const uint32_t lane_base = tb + (static_cast<uint32_t>(32 * q4 + 16 * h) << 16);
    const float c = p.scale * kLog2e;
    const uint64_t c2 = f2_pack(c, c);
    float m_run[2][2] = {{-INFINITY, -INFINITY}, {-INFINITY, -INFINITY}};  // [tile][A/B]
    float l_part[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    int n_t[2] = {0, 0};
    // Dropout: the generator's counter word x1 (this thread's row pair) is fixed per tile.
    philox::PrefixX0 pfx[2] = {};
    if constexpr (DROP) {
#pragma unroll
      for (int t = 0; t < 2; ++t)
        pfx[t] = philox::prefix_x0(philox::row_pair(u.q0 + t * kBlk + rA),
                                   static_cast<uint32_t>(u.bh), p.drop_offset, p.drop_seed_lo,
                                   p.drop_seed_hi);
    }
    bool ok = true;
    for (int j = 0; j < jend && ok; ++j) {
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (!ok || !need(p, u, t, j)) continue;
        ok = mbar_wait_warp(&bars->s_full[t], n_t[t] & 1, abort_flag, p.err, p.wait_ns);
        if (!ok) break;
        tc_fence_after();
        uint32_t v[64];
        tmem_ld_16x256b_x16_wait(lane_base + t * 128, v);
        float sv[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) sv[i] = __uint_as_float(v[i]);
        const int k0 = j * kBlk;
        const int row0 = u.q0 + t * kBlk;
        const bool edge = (p.causal && k0 + kBlk - 1 > row0) || (k0 + kBlk > u.L);
        if (edge) {
          const int lim_len = u.L - 1 - k0;
          const int limA = min(p.causal ? row0 + rA - k0 : kBlk - 1, lim_len);
          const int limB = min(p.causal ? row0 + rB - k0 : kBlk - 1, lim_len);
#pragma unroll
          for (int cc = 0; cc < 16; ++cc) {
            const int key = 8 * cc + 2 * t4;
            if (key > limA) sv[4 * cc] = -INFINITY;
            if (key + 1 > limA) sv[4 * cc + 1] = -INFINITY;
            if (key > limB) sv[4 * cc + 2] = -INFINITY;
            if (key + 1 > limB) sv[4 * cc + 3] = -INFINITY;
          }
        }
        float ma0 = fmaxf(sv[0], sv[1]), ma1 = fmaxf(sv[4], sv[5]);
        float mb0 = fmaxf(sv[2], sv[3]), mb1 = fmaxf(sv[6], sv[7]);
#pragma unroll
        for (int cc = 2; cc < 16; cc += 2) {
          ma0 = fmax3(ma0, sv[4 * cc], sv[4 * cc + 1]);
          mb0 = fmax3(mb0, sv[4 * cc + 2], sv[4 * cc + 3]);
          ma1 = fmax3(ma1, sv[4 * cc + 4], sv[4 * cc + 5]);
          mb1 = fmax3(mb1, sv[4 * cc + 6], sv[4 * cc + 7]);
        }
        float mA = fmaxf(ma0, ma1), mB = fmaxf(mb0, mb1);
        mA = fmaxf(mA, __shfl_xor_sync(0xffffffffu, mA, 1));
        mB = fmaxf(mB, __shfl_xor_sync(0xffffffffu, mB, 1));
        mA = fmaxf(mA, __shfl_xor_sync(0xffffffffu, mA, 2));
        mB = fmaxf(mB, __shfl_xor_sync(0xffffffffu, mB, 2));
        mA *= c;
        mB *= c;
        const float oldA = m_run[t][0], oldB = m_run[t][1];
        const float newA = mA > oldA + kRescaleThreshold ? mA : oldA;
        const float newB = mB > oldB + kRescaleThreshold ? mB : oldB;
        const bool chA = newA != oldA, chB = newB != oldB;
        const float alphaA = chA ? ex2(oldA - newA) : 1.f;  // old = -inf gives 0
        const float alphaB = chB ? ex2(oldB - newB) : 1.f;
        const float useA = newA == -INFINITY ? 0.f : newA;
        const float useB = newB == -INFINITY ? 0.f : newB;
        const uint64_t nA = f2_pack(-useA, -useA), nB = f2_pack(-useB, -useB);
        uint64_t accA = f2_pack(0.f, 0.f), accB = accA;
        uint32_t pk[32];
        philox::Words keep{};
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) {
          if constexpr (DROP) {
            // One generator call per four key chunks: word cc % 4 holds the bytes of keys
            // 8cc + 2(t % 4) + {0, 1} of rows A and B, in that order.
            if ((cc & 3) == 0) {
              keep = philox::run_x0(pfx[t], static_cast<uint32_t>(4 * (4 * j + (cc >> 2)) + t4));
#pragma unroll
              for (int k = 0; k < 4; ++k)
                keep.w[k] = philox::keep_bytes(keep.w[k], 0x01010101u * p.drop_threshold);
            }
          }
          const float2 xa = f2_unpack(ffma2(f2_pack(sv[4 * cc], sv[4 * cc + 1]), c2, nA));
          const float2 xb = f2_unpack(ffma2(f2_pack(sv[4 * cc + 2], sv[4 * cc + 3]), c2, nB));
          const float pa0 = ex2(xa.x), pa1 = ex2(xa.y);
          const float pb0 = ex2(xb.x), pb1 = ex2(xb.y);
          accA = fadd2(accA, f2_pack(pa0, pa1));
          accB = fadd2(accB, f2_pack(pb0, pb1));
          pk[2 * cc] = pack_bf16x2(pa0, pa1);
          pk[2 * cc + 1] = pack_bf16x2(pb0, pb1);
          if constexpr (DROP) {  // dropped probabilities leave P V but not the row sums
            pk[2 * cc] &= __byte_perm(keep.w[cc & 3], 0u, 0x1100);
            pk[2 * cc + 1] &= __byte_perm(keep.w[cc & 3], 0u, 0x3322);
          }
        }
        // P (bf16 pairs) overwrites the first 64 columns of this tile's S region in this
        // warp's 16 lanes, which no other warp reads; the load above has completed.
        tmem_st_16x128b_x16(lane_base + t * 128, pk);
        const float2 sa = f2_unpack(accA), sb = f2_unpack(accB);
        l_part[t][0] = l_part[t][0] * alphaA + (sa.x + sa.y);
        l_part[t][1] = l_part[t][1] * alphaB + (sb.x + sb.y);
        m_run[t][0] = newA;
        m_run[t][1] = newB;
        // Rescale the running O (the P V products issued before the S just read are done).
        if (n_t[t] > 0 && __any_sync(0xffffffffu, chA || chB)) {
#pragma unroll
          for (int half = 0; half < D / 64; ++half) {
            uint32_t o[32];
            const uint32_t oaddr = lane_base + 256 + t * 128 + 64 * half;
            tmem_ld_16x256b_x8_wait(oaddr, o);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              o[i] = __float_as_uint(__uint_as_float(o[i]) * ((i & 2) ? alphaB : alphaA));
            tmem_st_16x256b_x8(oaddr, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_full[t]);
        ++n_t[t];
      }
    }
    // ------------------------------------------------------------ epilogue
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      if (ok && n_t[t] > 0) {
        ok = mbar_wait_warp(&bars->o_done[t], 0, abort_flag, p.err, p.wait_ns);
        tc_fence_after();
      }
      if (!ok) break;
      float lA = l_part[t][0], lB = l_part[t][1];
      lA += __shfl_xor_sync(0xffffffffu, lA, 1);
      lB += __shfl_xor_sync(0xffffffffu, lB, 1);
      lA += __shfl_xor_sync(0xffffffffu, lA, 2);
      lB += __shfl_xor_sync(0xffffffffu, lB, 2);
      float invA = lA > 0.f ? 1.f / lA : 0.f, invB = lB > 0.f ? 1.f / lB : 0.f;
      if constexpr (DROP) {
        invA *= p.drop_scale;
        invB *= p.drop_scale;
      }
      const int rowA = u.q0 + t * kBlk + rA, rowB = rowA + 8;
      // O / l as bf16 into this tile's Q buffer (every S MMA that read it has completed: they
      // precede the last P V product of this tile), in the 128-byte-swizzled layout of the
      // TMA box; one thread then stores the tile with the TMA (rows past N are clipped).
      uint8_t* stage = sQ + t * C::TILE;
#pragma unroll
      for (int half = 0; half < D / 64; ++half) {
        uint32_t ov[32];
        if (n_t[t] > 0) {
          tmem_ld_16x256b_x8_wait(lane_base + 256 + t * 128 + 64 * half, ov);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = 0u;
        }
        uint8_t* sub = stage + half * kSub;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          const uint32_t byte = static_cast<uint32_t>(4 * t4);   // column 8cc + 2t4, bf16
          *reinterpret_cast<uint32_t*>(sub + rA * 128 + ((cc ^ (rA & 7)) << 4) + byte) =
              pack_bf16x2(__uint_as_float(ov[4 * cc]) * invA, __uint_as_float(ov[4 * cc + 1]) * invA);
          *reinterpret_cast<uint32_t*>(sub + rB * 128 + ((cc ^ (rB & 7)) << 4) + byte) =
              pack_bf16x2(__uint_as_float(ov[4 * cc + 2]) * invB, __uint_as_float(ov[4 * cc + 3]) * invB);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars->o_staged[t]);
      if (warp == 4 && lane == 0 && u.q0 + t * kBlk < p.N) {
        if (mbar_wait(&bars->o_staged[t], 0, abort_flag, p.err, p.wait_ns)) {
#pragma unroll
          for (int half = 0; half < D / 64; ++half)
            tma_store_3d(&mo, stage + half * kSub, 64 * half, u.q0 + t * kBlk, u.bh);
          bulk_commit_group();
        }
      }
      if (t4 == 0) {
        float* lrow = lse + static_cast<size_t>(u.bh) * p.N;
        if (rowA < p.N) lrow[rowA] = lA > 0.f ? (m_run[t][0] + __log2f(lA)) * kLn2 : -INFINITY;
        if (rowB < p.N) lrow[rowB] = lB > 0.f ? (m_run[t][1] + __log2f(lB)) * kLn2 : -INFINITY;
      }
    }
  }

  if (warp == 4 && lane == 0) bulk_wait_group_all();
  tc_fence_before();
  __syncthreads();
  if (bars->abort && tid == 0) {
    // Let any bulk copy still in flight land before the CTA's shared memory is released.
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 1000000ull) {
    }
  }
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  // Looked up once (a function-local static is thread-safe); null if the driver lacks it.
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

}  // namespace

// [B*H, N, d] bf16 viewed as a 3-D tensor (d innermost); 64-column boxes of `box_rows` rows,
// 128B swizzle, rows beyond N read as zero.
bool make_head_map_rows(CUtensorMap* map, const void* ptr, int BH, int N, int d, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [BH, rows, inner] bytes (inner contiguous) with 128 x 128 boxes and 128-byte swizzle;
// elements outside the tensor read as zero.
bool make_u8_map(CUtensorMap* map, const void* ptr, int BH, int rows, int inner) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner),
                           static_cast<cuuint64_t>(rows) * static_cast<cuuint64_t>(inner)};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_head_map(CUtensorMap* map, const void* ptr, int BH, int N, int d) {
  return make_head_map_rows(map, ptr, BH, N, d, 128);
}

// [B*H, N, d] fp32 accumulator as a 3-D tensor with 32 x 32 boxes (128-byte rows, 128-byte
// swizzle); rows beyond N are outside the map, so a box that overhangs the sequence end is
// clipped.
bool make_acc_map(CUtensorMap* map, const void* ptr, int BH, int N, int d) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(N) * d * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool DROP>
static cudaError_t fwd_launch(const Problem& p, const void* q, const void* k, const void* v,
                              void* o, float* lse, cudaStream_t s) {
  CUtensorMap mq, mk, mv, mo;
  const int BH = p.B * p.H;
  if (!make_head_map(&mq, q, BH, p.N, D) || !make_head_map(&mk, k, BH, p.N, D) ||
      !make_head_map(&mv, v, BH, p.N, D) || !make_head_map(&mo, o, BH, p.N, D))
    return cudaErrorInvalidValue;
  static std::atomic<bool> attr_set[64];  // per device; a race repeats the same call
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev].load()) {
    cudaError_t e = cudaFuncSetAttribute(fwd_sm103_kernel<D, DROP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true);
  }
  const int nqb = (p.N + 255) / 256;
  dim3 grid(static_cast<unsigned>(BH) * nqb);
  return launch_dependent(fwd_sm103_kernel<D, DROP>, grid, dim3(kThreads), Cfg<D>::SMEM, s, mq,
                          mk, mv, mo, lse, p);
}

cudaError_t launch_fwd_sm103(const Problem& p, const void* q, const void* k, const void* v,
                             void* o, float* lse, cudaStream_t s) {
  if (p.drop_threshold > 0)
    return p.d == 64 ? fwd_launch<64, true>(p, q, k, v, o, lse, s)
                     : fwd_launch<128, true>(p, q, k, v, o, lse, s);
  return p.d == 64 ? fwd_launch<64, false>(p, q, k, v, o, lse, s)
                   : fwd_launch<128, false>(p, q, k, v, o, lse, s);
}

}  // namespace fa
