// Backward attention on sm_103a tensor cores (tcgen05 + TMA), key-outer.
//
// The backward recomputes the scores and probabilities block by block from Q, K and the
// saved logsumexp instead of reading a stored P (answer page "How FlashAttention works
// for training", sections 3 and 3.1; course week 13, step 2), and forms the gradients
// by the chain rule (the answer page's printed formulas for dQ and dK are garbled; these
// are the standard ones):
//   P_ij  = exp(scale q_i.k_j - lse_i)          dV_j += sum_i P_ij dO_i
//   dP_ij = dO_i . v_j                           dS_ij = P_ij (dP_ij - D_i)
//   dK_j += scale sum_i dS_ij q_i                dQ_i += scale sum_j dS_ij k_j
// with D_i = rowsum(dO_i o O_i) precomputed by the preprocess kernel.  The scale of dQ is
// applied by the dQ-convert kernel.
//
// GB300 mapping: one CTA owns a block of 128 keys of one (batch, head) and keeps K_j, V_j
// in shared memory; it walks the 128-row query blocks i that see those keys (i >= j under
// the causal mask, mask[i][j] = 1 under a block mask), accumulating dK_j, dV_j in tensor
// memory and adding each dQ_i partial to an fp32 accumulator in global memory.
// Per query block the tensor pipe runs five MMAs (all M = 128, bf16 in, fp32 out):
//   S^T  = K_j Q_i^T   (A: K_j K-major smem,    B: Q_i K-major smem)    -> TMEM Ra
//   dP^T = V_j dO_i^T  (A: V_j K-major smem,    B: dO_i K-major smem)   -> TMEM Rb
//   dV  += P^T dO_i    (A: P^T bf16 in TMEM,    B: dO_i MN-major smem)  -> TMEM [256,256+d)
//   dK  += dS^T Q_i    (A: dS^T bf16 in TMEM,   B: Q_i MN-major smem)   -> TMEM dK columns
//   dQ_i = dS K_j      (A: dS^T MN-major smem,  B: K_j MN-major smem)   -> TMEM dQ columns
// with R0 = [0,128) and R1 = [128,256).  P^T is written over already-read S^T columns and
// dS^T over already-read dP^T columns.  With d = 128 the two regions swap roles every block:
// block n has Ra = R[n % 2], Rb the other, and its dQ partial (TMEM lane = query row) goes
// into Ra once dV has read P^T there (dK at [384,512)).  With d = 64, Ra = R0, Rb = R1 and
// the dQ partial has columns of its own, [320,384) (dK at [384,448)).
// Warps (16): 0-3 the dQ drain, 4-7 and 8-11 two warpgroups that each take 64 of the 128
// query columns of every key row (phase A: P^T from S^T; phase B: dS^T from dP^T), 12 TMA
// producer (K_j, V_j once; Q_i and dO_i through two-stage rings) and tensor-memory
// allocation, 13 MMA issuer, 14-15 idle.  The drain copies each dQ_i partial out of TMEM
// into 128-byte-swizzled [32 rows][32 columns] fp32 boxes in shared memory and adds them to
// the fp32 accumulator in global memory with TMA bulk reduce-adds.
// MMA issue order per block n, d = 128: dV(n), dQ(n), dK(n), S^T(n+1), dP^T(n+1).  The dQ
// drain and the bulk reduce-adds behind it decide when the next phase B may reuse the dS
// tile, so dQ(n) goes first once phase B(n) is done.  S^T(n+1) goes into Rb(n) as soon as
// dK(n) (issued before it) has read dS^T(n) there, without waiting for the drain; dP^T(n+1)
// goes into Ra(n) once the drain has copied the partial out of it in one load.
// d = 64: dV(n), S^T(n+1), then (after phase B(n)) dQ(n), dK(n), dP^T(n+1): with dQ in columns
// of its own nothing waits for the drain, and S^T(n+1) goes into R0 as soon as dV(n) (issued
// before it; one thread's MMAs run in issue order) has read P^T(n), so it is ready when the
// softmax warps finish phase B(n).
// Every mbarrier wait is bounded; on expiry the CTA records FA_ERR_TIMEOUT and exits.
#include <atomic>

#include <cuda.h>
#include <math.h>

#include "fa_internal.cuh"
#include "fa_philox.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

constexpr int kBlk = 128;
constexpr int kSub = 128 * 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kProducerWarp = 12;  // also allocates tensor memory
constexpr int kMmaWarp = 13;       // warps 14-15 idle
constexpr int kThreads = 512;
// Registers per thread after reallocation (d = 128; launched with 128): the MMA issuer takes
// the TMEM region of each block as a runtime address and needs more than 56.
constexpr int kRegsDrain = 168;    // warps 0-3
constexpr int kRegsSoftmax = 136;  // warps 4-11
constexpr int kRegsControl = 72;   // warps 12-15
constexpr int kRegsLaunch = 128;   // 65536 / kThreads
static_assert(4 * 32 * (kRegsDrain + 2 * kRegsSoftmax + kRegsControl) == kThreads * kRegsLaunch,
              "register split must equal the launch allocation");
// setmaxnreg.inc may only raise a warp's count and .dec only lower it.
static_assert(kRegsDrain >= kRegsLaunch && kRegsSoftmax >= kRegsLaunch &&
                  kRegsControl <= kRegsLaunch,
              "drain and softmax warps take registers, control warps release them");

template <int D>
struct Cfg {
  static constexpr int NSUB = D / 64;
  static constexpr int TILE = NSUB * kSub;         // one 128 x d bf16 tile
  static constexpr int NSTAGE = 2;                 // Q_i / dO_i ring
  static constexpr int DS = 2 * kSub;              // dS^T, 128 x 128 bf16
  static constexpr int SMEM = 1024 + 2 * TILE + NSTAGE * 2 * TILE + DS + 1024 + 256;
  // TMEM columns of the dQ partial: R0 (after dV has read P^T) with d = 128, columns of
  // its own with d = 64; and of the dK accumulator.
  static constexpr bool SEP_DQ = D == 64;
  static constexpr uint32_t COL_DQ = SEP_DQ ? 320u : 0u;
  static constexpr uint32_t COL_DK = 384u;
};

struct Bars {
  uint64_t kv_full;
  uint64_t q_full[2];
  uint64_t q_empty[2];
  uint64_t do_full[2];
  uint64_t do_empty[2];
  uint64_t s_full;
  uint64_t dp_full;
  uint64_t p_ready;
  uint64_t ds_ready;
  uint64_t dq_full;
  uint64_t dq_free;
  uint64_t stats_full;
  uint64_t sds_free;
  uint64_t acc_done;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int never;  // stays 0: waits that must not be cut short by an abort
};
static_assert(sizeof(Bars) <= 256, "barrier block");

struct Unit {
  int bh, j, L, nb, nq;
};

__device__ __forceinline__ bool need(const Problem& p, const Unit& u, int i) {
  if (u.j * kBlk >= u.L) return false;
  if (p.causal && i < u.j) return false;
  if (p.blockmask && !p.blockmask[i * u.nb + u.j]) return false;
  return true;
}

__device__ __forceinline__ int next_q(const Problem& p, const Unit& u, int i) {
  for (++i; i < u.nq; ++i)
    if (need(p, u, i)) return i;
  return -1;
}

// Byte offset of bf16 element (row, col) in a [rows][128] tile stored as two 128B-swizzled
// [rows][64] subtiles (16-byte chunk c of row r lands in chunk c ^ (r % 8)).
__device__ __forceinline__ uint32_t sw128_offset(int row, int col) {
  const int sub = col >> 6, chunk = (col & 63) >> 3;
  return sub * kSub + (row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4) +
         ((col & 7) << 1);
}

// DROP: dropout on P, its mask regenerated from the generator of fa_philox.cuh: dV takes
// P o Z (scaled by 1 / (1 - p) in the epilogue), dS = P o (Z o dP / (1 - p) - D).
template <int D, bool DROP>
__global__ void __launch_bounds__(kThreads, 1)
bwd_sm103_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                 const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
                 const __grid_constant__ CUtensorMap mdq, const float* __restrict__ lse, const float* __restrict__ Dsum,
                 float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dk,
                 __nv_bfloat16* __restrict__ dv, Problem p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sK = base;
  uint8_t* sV = sK + C::TILE;
  uint8_t* sQ = sV + C::TILE;                  // [NSTAGE][Q tile, dO tile]
  uint8_t* sDS = sQ + C::NSTAGE * 2 * C::TILE;
  float* sL = reinterpret_cast<float*>(sDS + C::DS);   // [128] -lse * log2(e) (or -inf)
  float* sD = sL + kBlk;                               // [128] -D
  Bars* bars = reinterpret_cast<Bars*>(sD + kBlk);
  volatile int* abort_flag = &bars->abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  Unit u;
  u.nb = (p.N + kBlk - 1) / kBlk;
  u.nq = u.nb;
  const int bhs = p.B * p.H;
  {
    // Grid order: groups of G heads, G as large as keeps a group's Q and dO (bf16) and its dQ
    // accumulator (fp32), 8 N d bytes per head, within 64 MiB of L2; in each group key block
    // j ascending (small j first: the most query blocks under causal), the group's heads
    // fastest.  The co-resident CTAs then read each Q and dO tile from DRAM about once and
    // reduce into accumulators that stay in L2.  The dropout instance keeps all heads in one
    // group (heads fastest), which measured faster for it.
    if constexpr (DROP) {
      u.bh = blockIdx.x % bhs;
      u.j = blockIdx.x / bhs;
    } else {
      const long long per_head = 8ll * p.N * D;
      const int G = static_cast<int>(
          max(1ll, min(static_cast<long long>(bhs), (64ll << 20) / per_head)));
      const int b = blockIdx.x, g = b / (G * u.nb), r = b - g * G * u.nb;
      const int Gg = min(G, bhs - g * G);
      u.j = r / Gg;
      u.bh = g * G + r % Gg;
    }
  }

  if (tid == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], 1);
      mbar_init(&bars->do_full[s], 1);
      // Released by the MMA commit and by the two dQ-drain warps that stage their partial
      // in the dO stage once its MMAs are done.
      mbar_init(&bars->do_empty[s], 3);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_ready, 2 * kBlk);
    mbar_init(&bars->ds_ready, 2 * kBlk);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_free, kBlk);
    mbar_init(&bars->stats_full, 2 * kBlk);
    mbar_init(&bars->sds_free, 2);
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    bars->never = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = bars->tmem_base;
  // d = 128: the two 128-column regions swap roles every block -- S^T, P^T and then the dQ
  // partial of block n in R[n % 2], dP^T and dS^T in the other -- so that S^T of the next
  // block need not wait for the drain; d = 64 keeps S^T in R0 and dP^T in R1.
  auto s_reg = [](int n) { return C::SEP_DQ ? 0u : static_cast<uint32_t>(n & 1) * 128u; };
  auto d_reg = [&](int n) { return 128u - s_reg(n); };
  // Set-up done; global memory (the key lengths and the block mask included) only after the
  // previous kernel in the stream has completed.
  griddep_wait();
  griddep_launch_dependents();
  {
    int L = p.N;
    if (p.kv_len) {
      L = p.kv_len[u.bh / p.H];
      L = L < 0 ? 0 : (L > p.N ? p.N : L);
    }
    u.L = L;
  }
  const int first = next_q(p, u, -1);
  // Registers (d = 128): launched with 128 per thread (512 threads).  The producer / MMA
  // warpgroup (warps 12-15) gives 56 of them back; the dQ drain warpgroup (warps 0-3) takes
  // 40, so a drain warp can hold a whole 128-column dQ row slice, and each softmax
  // warpgroup 8, so phase A can load all 64 of its S^T columns at once:
  // 4 x 32 x (168 + 136 + 136 + 72) = 512 x 128.  With d = 64 everything fits as launched.
  static_assert(kThreads == 512 && kRegsDrain + 2 * kRegsSoftmax + kRegsControl == 4 * 128, "register split");

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    if constexpr (D == 128) regs_release_to<kRegsControl>();
    if (lane == 0 && first >= 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mdo);
      mbar_arrive_expect_tx(&bars->kv_full, 2 * C::TILE);
      for (int s = 0; s < C::NSUB; ++s) {
        tma_load_3d(sK + s * kSub, &mk, &bars->kv_full, 64 * s, u.j * kBlk, u.bh);
        tma_load_3d(sV + s * kSub, &mv, &bars->kv_full, 64 * s, u.j * kBlk, u.bh);
      }
      int stage = 0, round = 0;
      for (int i = first; i >= 0; i = next_q(p, u, i)) {
        uint8_t* dst = sQ + stage * 2 * C::TILE;
        if (!mbar_wait(&bars->q_empty[stage], (round & 1) ^ 1, abort_flag, p.err, p.wait_ns))
          break;
        mbar_arrive_expect_tx(&bars->q_full[stage], C::TILE);
        for (int s = 0; s < C::NSUB; ++s)
          tma_load_3d(dst + s * kSub, &mq, &bars->q_full[stage], 64 * s, i * kBlk, u.bh);
        if (!mbar_wait(&bars->do_empty[stage], (round & 1) ^ 1, abort_flag, p.err, p.wait_ns))
          break;
        mbar_arrive_expect_tx(&bars->do_full[stage], C::TILE);
        for (int s = 0; s < C::NSUB; ++s)
          tma_load_3d(dst + C::TILE + s * kSub, &mdo, &bars->do_full[stage], 64 * s, i * kBlk,
                      u.bh);
        if (++stage == C::NSTAGE) {
          stage = 0;
          ++round;
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if constexpr (D == 128) regs_release_to<kRegsControl>();
    if (lane == 0 && first >= 0) {
      constexpr uint32_t idSS = idesc_bf16(128, 128, false, false);  // S^T, dP^T
      constexpr uint32_t idKN = idesc_bf16(128, D, false, true);     // dV, dK (B MN-major)
      constexpr uint32_t idMN = idesc_bf16(128, D, true, true);      // dQ (A, B MN-major)
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aDS = smem_u32(sDS);
      const uint32_t aQ0 = smem_u32(sQ);
      auto q_addr = [&](int n) { return aQ0 + (n & 1) * 2 * C::TILE; };
      // TMEM column of the bf16 A operand (P^T at 0, dS^T at 128) for k-step kk: query
      // columns 0-63 sit in the first 32 columns of the region, 64-127 in columns 64-95.
      auto a_col = [](uint32_t region, int kk) {
        return region + (kk < 4 ? 8 * kk : 64 + 8 * (kk - 4));
      };
      // Groups of four MMAs from one asm statement, descriptors built first (advanced from
      // their k = 0 form by the byte offset >> 4), so that the four go out back to back.
      auto issue_ss_k = [&](uint32_t tdst, uint32_t aA, uint32_t aB) {   // K-major A and B
        const uint64_t dA = sw128_desc(aA, 16, 1024), dB = sw128_desc(aB, 16, 1024);
        const uint32_t a_lo = static_cast<uint32_t>(dA), b_lo = static_cast<uint32_t>(dB);
#pragma unroll
        for (int g = 0; g < D / 64; ++g) {
          uint32_t da[4], db[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t off = static_cast<uint32_t>((g * kSub + k * 32) >> 4);
            da[k] = a_lo + off;
            db[k] = b_lo + off;
          }
          mma_ss_x4_lo(tdst, da, static_cast<uint32_t>(dA >> 32), db,
                       static_cast<uint32_t>(dB >> 32), idSS, g > 0 ? 1u : 0u);
        }
      };
      auto issue_s = [&](int n, uint32_t tdst) {
        issue_ss_k(tdst, aK, q_addr(n));
        mma_commit(&bars->s_full);
      };
      auto issue_dp = [&](int n, uint32_t tdst) {
        issue_ss_k(tdst, aV, q_addr(n) + C::TILE);
        mma_commit(&bars->dp_full);
      };
      bool ok = mbar_wait(&bars->kv_full, 0, abort_flag, p.err, p.wait_ns);
      ok = ok && mbar_wait(&bars->q_full[0], 0, abort_flag, p.err, p.wait_ns);
      tc_fence_after();
      if (ok) issue_s(0, tb);
      ok = ok && mbar_wait(&bars->do_full[0], 0, abort_flag, p.err, p.wait_ns);
      tc_fence_after();
      if (ok) issue_dp(0, tb + 128);
      // tds: TMEM address of the region holding dS^T (bf16 pairs as the A operand).
      // A from TMEM (bf16 pairs at ta), B MN-major: dV += P^T dO, dK += dS^T Q.
      auto issue_ts = [&](uint32_t tdst, uint32_t ta, uint32_t aB, bool acc) {
        const uint64_t dB = sw128_desc(aB, kSub, 1024);
        const uint32_t b_lo = static_cast<uint32_t>(dB);
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          uint32_t a4[4], db[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int kk = 4 * g + k;
            a4[k] = ta + a_col(0, kk);
            db[k] = b_lo + 128u * kk;
          }
          mma_ts_x4_lo(tdst, a4, db, static_cast<uint32_t>(dB >> 32), idKN,
                       (acc || g > 0) ? 1u : 0u);
        }
      };
      auto issue_dk = [&](uint32_t aQ, int n, uint32_t tds) {
        issue_ts(tb + C::COL_DK, tds, aQ, n > 0);
      };
      auto issue_dq = [&](uint32_t tdst) {
        const uint64_t dA = sw128_desc(aDS, kSub, 1024), dB = sw128_desc(aK, kSub, 1024);
        const uint32_t a_lo = static_cast<uint32_t>(dA), b_lo = static_cast<uint32_t>(dB);
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          uint32_t da[4], db[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            da[k] = a_lo + 128u * (4 * g + k);
            db[k] = b_lo + 128u * (4 * g + k);
          }
          mma_ss_x4_lo(tdst, da, static_cast<uint32_t>(dA >> 32), db,
                       static_cast<uint32_t>(dB >> 32), idMN, g > 0 ? 1u : 0u);
        }
        mma_commit(&bars->dq_full);
      };
      int n = 0;
      for (int i = first; ok && i >= 0; ++n) {
        const int in = next_q(p, u, i);
        const uint32_t aQ = q_addr(n), aDO = aQ + C::TILE;
        const uint32_t par = s_reg(n);   // this block's S^T region (0 or 128)
        const uint32_t tP = tb + par;     // ... where P^T is
        // dV += P^T dO_i  (dO_i was waited for before dP^T(n))
        ok = mbar_wait(&bars->p_ready, n & 1, abort_flag, p.err, p.wait_ns);
        tc_fence_after();
        if (!ok) break;
        issue_ts(tb + 256, tP, aDO, n > 0);
        if constexpr (C::SEP_DQ) {
          if (in >= 0) {
            // S^T of the next block over P^T(n), which dV(n) (issued before it) reads first;
            // the softmax warps find it ready when they finish phase B(n).
            ok = mbar_wait(&bars->q_full[(n + 1) & 1], ((n + 1) >> 1) & 1, abort_flag, p.err,
                           p.wait_ns);
            tc_fence_after();
            if (!ok) break;
            issue_s(n + 1, tb);
          }
          ok = mbar_wait(&bars->ds_ready, n & 1, abort_flag, p.err, p.wait_ns);
          // dQ_i = dS K_j into its own columns (the drain has long copied out dQ(n-1)).
          if (ok && n > 0) ok = mbar_wait(&bars->dq_free, (n - 1) & 1, abort_flag, p.err, p.wait_ns);
          tc_fence_after();
          if (!ok) break;
          issue_dq(tb + C::COL_DQ);
          issue_dk(aQ, n, tb + 128u);
          mma_commit(&bars->q_empty[n & 1]);
          mma_commit(&bars->do_empty[n & 1]);
          if (in >= 0) {
            ok = mbar_wait(&bars->do_full[(n + 1) & 1], ((n + 1) >> 1) & 1, abort_flag, p.err,
                           p.wait_ns);
            tc_fence_after();
            if (!ok) break;
            issue_dp(n + 1, tb + 128);
          }
        } else {
          // dQ_i = dS K_j first, into this block's S^T region (dV has read P^T there): its drain
          // and the TMA reduce-adds behind it gate the next phase B.  dK reads dS^T from the
          // other region, and S^T of the next block goes over it at once (one thread's MMAs run
          // in issue order); dP^T of the next block takes this block's region once the drain
          // has copied dQ_i out of it.
          ok = mbar_wait(&bars->ds_ready, n & 1, abort_flag, p.err, p.wait_ns);
          tc_fence_after();
          if (!ok) break;
          issue_dq(tP);
          issue_dk(aQ, n, tb + 128u - par);
          mma_commit(&bars->q_empty[n & 1]);
          mma_commit(&bars->do_empty[n & 1]);
          if (in >= 0) {
            ok = mbar_wait(&bars->q_full[(n + 1) & 1], ((n + 1) >> 1) & 1, abort_flag, p.err,
                           p.wait_ns);
            tc_fence_after();
            if (!ok) break;
            issue_s(n + 1, tb + 128u - par);
            ok = mbar_wait(&bars->dq_free, n & 1, abort_flag, p.err, p.wait_ns);
            ok = ok && mbar_wait(&bars->do_full[(n + 1) & 1], ((n + 1) >> 1) & 1, abort_flag,
                                 p.err, p.wait_ns);
            tc_fence_after();
            if (!ok) break;
            issue_dp(n + 1, tb + par);
          }
        }
        i = in;
      }
      mma_commit(&bars->acc_done);
      mma_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, &bars->never, nullptr, p.wait_ns);
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ P^T and dS^T (key rows)
    if constexpr (D == 128) regs_grow_to<kRegsSoftmax>();
    const int w = (warp - 4) >> 2;              // query columns [64w, 64w + 64)
    const int r = ((warp & 3) << 5) + lane;     // key row within the block = TMEM lane
    const int key = u.j * kBlk + r;
    const bool key_live = key < u.L;
    const uint32_t lane_base = tb + (static_cast<uint32_t>((warp & 3) << 5) << 16);
    const float c = p.scale * kLog2e;
    const size_t row_off = static_cast<size_t>(u.bh) * p.N;
    // Raw lse and D of one column of the next block, loaded a block ahead; they are only
    // transformed when written to shared memory, so the loads never stall this block.
    float st_lse = -INFINITY, st_dd = 0.f;
    auto load_stats = [&](int iq) {
      const int qrow = iq * kBlk + 64 * w + r;
      const bool in = iq >= 0 && qrow < p.N;
      st_lse = in ? lse[row_off + qrow] : -INFINITY;
      st_dd = in ? Dsum[row_off + qrow] : 0.f;
    };
    if (r < 64) load_stats(first);
    bool ok = true;
    int n = 0;
    for (int i = first; ok && i >= 0; i = next_q(p, u, i), ++n) {
      // Every thread of both warpgroups has finished phase B of the previous block (and so
      // with the statistics buffer) once ds_ready of that block has completed.
      if (n > 0) {
        ok = mbar_wait_warp(&bars->ds_ready, (n - 1) & 1, abort_flag, p.err, p.wait_ns);
        if (!ok) break;
      }
      // Column statistics of this query block, negated for packed fma/add: -lse * log2(e)
      // (-inf where the row is outside the sequence or sees no key, so that P = 0 there)
      // and -D.  They were loaded
      // into registers during the previous block; the next block's are requested now.
      if (r < 64) {
        sL[64 * w + r] = st_lse == -INFINITY ? -INFINITY : -st_lse * kLog2e;
        sD[64 * w + r] = -st_dd;
        load_stats(next_q(p, u, i));
      }
      mbar_arrive(&bars->stats_full);
      ok = mbar_wait_warp(&bars->stats_full, n & 1, abort_flag, p.err, p.wait_ns);
      if (!ok) break;
      const bool diag = p.causal && i == u.j;
      const int lim = diag ? r : 0;   // diagonal block: query column q sees key r iff q >= r
      // Dropout: bit x of zbits keeps element (query 128 i + 64 w + x, this key row).  Rows x
      // and x + 8 (x % 16 < 8) share a generator call, x2 = 8 (x >> 4) + (x & 7) numbering
      // the 32 calls of this warpgroup's columns (counter word rho = 64 i + 32 w + x2); this
      // key's two bytes sit in word (key >> 3) & 3 at bytes (key & 1) and 2 + (key & 1).
      // The eight lanes g = (lane & 1) + 2 ((lane >> 3) & 3) of one key octet need the same
      // 32 calls: lane g makes calls 4g .. 4g + 3 and packs, for every partner g', the keep
      // bits of g' (bit k + 4 s for call 4g + k, row x + 8 s) into byte g' of a 64-bit word;
      // an 8 x 8 byte transpose over xor-shuffles hands every lane its 64 bits.
      uint64_t zbits = 0;
      if constexpr (DROP) {
        const uint32_t octet = philox::key_octet(key);
        const uint32_t thr4 = 0x01010101u * static_cast<uint32_t>(p.drop_threshold);
        const int g = (lane & 1) | (((lane >> 3) & 3) << 1);
        uint64_t M = 0;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const philox::Words cw4 = philox::philox4x32_10(
              octet, static_cast<uint32_t>(64 * i + 32 * w + 4 * g + kk),
              static_cast<uint32_t>(u.bh), p.drop_offset, p.drop_seed_lo, p.drop_seed_hi);
#pragma unroll
          for (int cw = 0; cw < 4; ++cw) {
            // bytes of word cw: (g' = 2cw, row x), (2cw + 1, x), (2cw, x + 8), (2cw + 1, x + 8)
            const uint32_t t = philox::keep_bytes(cw4.w[cw], thr4) & (0x01010101u << kk);
            const uint32_t chunk = (t & 0xFFFFu) | ((t >> 12) & 0xFFF0u);
            M |= static_cast<uint64_t>(chunk) << (16 * cw);
          }
        }
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) {
          const int src = g ^ rr;   // the partner whose calls this round's byte comes from
          uint32_t b = static_cast<uint32_t>(M >> (8 * src)) & 0xFFu;
          if (rr) b = __shfl_xor_sync(0xffffffffu, b, (rr & 1) | ((rr >> 1) << 3));
          const int base = 16 * (src >> 1) + 4 * (src & 1);   // x of call 4 src, row x
          zbits |= (static_cast<uint64_t>(b & 0xFu) << base) |
                   (static_cast<uint64_t>(b >> 4) << (base + 8));
        }
      }
      // ---- phase A: P^T = exp2(S^T * c - lse * log2 e) for this warpgroup's 64 columns
      ok = mbar_wait_warp(&bars->s_full, n & 1, abort_flag, p.err, p.wait_ns);
      if (!ok) break;
      tc_fence_after();
      uint32_t pp[32];
      const uint64_t c2 = f2_pack(c, c);
      // Off the diagonal, every query column of a live key row is visible: no masks.
      const bool masked = diag || !key_live;
      // Both halves of this warpgroup's S^T columns in one round trip.
      uint32_t sva[64];
      const uint32_t sR = s_reg(n), dR = d_reg(n);
      tmem_ld64_wait(lane_base + sR + 64 * w, lane_base + sR + 64 * w + 32, sva);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t* sv = sva + 32 * h;
        const float* L = sL + 64 * w + 32 * h;
        const float2* L2 = reinterpret_cast<const float2*>(L);
        if (!masked) {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 l = L2[e / 2];
            const float2 x = f2_unpack(ffma2(f2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])),
                                             c2, f2_pack(l.x, l.y)));
            pp[16 * h + e / 2] = pack_bf16x2(ex2(x.x), ex2(x.y));
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int q0 = 64 * w + 32 * h + e;
            float pa = ex2(fmaf(__uint_as_float(sv[e]), c, L[e]));
            float pb = ex2(fmaf(__uint_as_float(sv[e + 1]), c, L[e + 1]));
            if (!key_live || q0 < lim) pa = 0.f;
            if (!key_live || q0 + 1 < lim) pb = 0.f;
            pp[16 * h + e / 2] = pack_bf16x2(pa, pb);
          }
        }
      }
      // P^T over this warpgroup's own, already-read S^T columns [64w, 64w + 32).
      if constexpr (DROP) {
        // dV takes P o Z; phase B still needs P itself.
        uint32_t pz[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const uint32_t b = static_cast<uint32_t>(zbits >> (2 * e)) & 3u;
          pz[e] = pp[e] & ((b & 1u ? 0x0000FFFFu : 0u) | (b & 2u ? 0xFFFF0000u : 0u));
        }
        tmem_st32(lane_base + sR + 64 * w, pz);
      } else {
        tmem_st32(lane_base + sR + 64 * w, pp);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_ready);
      // ---- phase B: dS^T = P^T o (dP^T - D)
      // -D of the first half's columns, read while dP^T is still being computed.
      const float4* D4 = reinterpret_cast<const float4*>(sD + 64 * w);
      float4 dvals[8];
#pragma unroll
      for (int e4 = 0; e4 < 8; ++e4) dvals[e4] = D4[e4];
      ok = mbar_wait_warp(&bars->dp_full, n & 1, abort_flag, p.err, p.wait_ns);
      // d = 128: two drain warps staged the previous dQ partial in the dS^T tile; with d = 64
      // the wait is taken just before the first store into the tile (below).
      if (D == 128 && ok && n > 0)
        ok = mbar_wait_warp(&bars->sds_free, (n - 1) & 1, abort_flag, p.err, p.wait_ns);
      if (!ok) break;
      tc_fence_after();
      const uint64_t ks2 = f2_pack(p.drop_scale, p.drop_scale);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t dpv[32], dsp[16];
        if (h == 1) {  // the second half's -D, in flight during the TMEM load
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) dvals[e4] = D4[8 + e4];
        }
        tmem_ld32_wait(lane_base + dR + 64 * w + 32 * h, dpv);
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 nd = dvals[e4];   // -D
          const float2 p01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pp[16 * h + 2 * e4]));
          const float2 p23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pp[16 * h + 2 * e4 + 1]));
          float2 d01, d23;
          if constexpr (DROP) {
            // dS = P o (Z o dP / (1 - p) - D): dropped dP entries are cleared with a bit mask,
            // the kept ones scaled by the packed keep scale.
            const uint32_t zh = static_cast<uint32_t>(zbits >> (32 * h)) >> (4 * e4);
            const uint32_t dp0 = dpv[4 * e4 + 0] & (0u - (zh & 1u));
            const uint32_t dp1 = dpv[4 * e4 + 1] & (0u - ((zh >> 1) & 1u));
            const uint32_t dp2 = dpv[4 * e4 + 2] & (0u - ((zh >> 2) & 1u));
            const uint32_t dp3 = dpv[4 * e4 + 3] & (0u - ((zh >> 3) & 1u));
            d01 = f2_unpack(fmul2(f2_pack(p01.x, p01.y),
                ffma2(f2_pack(__uint_as_float(dp0), __uint_as_float(dp1)), ks2,
                      f2_pack(nd.x, nd.y))));
            d23 = f2_unpack(fmul2(f2_pack(p23.x, p23.y),
                ffma2(f2_pack(__uint_as_float(dp2), __uint_as_float(dp3)), ks2,
                      f2_pack(nd.z, nd.w))));
          } else {
            d01 = f2_unpack(fmul2(f2_pack(p01.x, p01.y),
                fadd2(f2_pack(__uint_as_float(dpv[4 * e4 + 0]), __uint_as_float(dpv[4 * e4 + 1])), f2_pack(nd.x, nd.y))));
            d23 = f2_unpack(fmul2(f2_pack(p23.x, p23.y),
                fadd2(f2_pack(__uint_as_float(dpv[4 * e4 + 2]), __uint_as_float(dpv[4 * e4 + 3])), f2_pack(nd.z, nd.w))));
          }
          dsp[2 * e4] = pack_bf16x2(d01.x, d01.y);
          dsp[2 * e4 + 1] = pack_bf16x2(d23.x, d23.y);
        }
        // dS^T over this warpgroup's already-read dP^T columns, and into the swizzled
        // shared tile (row r, query columns 64w + 32h ...).
        tmem_st16(lane_base + dR + 64 * w + 16 * h, dsp);
        // d = 64: two drain warps staged the previous dQ partial in the dS^T tile: wait for
        // their bulk reduce-adds to have read it before the first store into the tile.
        if (D == 64 && h == 0 && n > 0)
          ok = mbar_wait_warp(&bars->sds_free, (n - 1) & 1, abort_flag, p.err, p.wait_ns);
        if (ok) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint4 v4 = make_uint4(dsp[4 * g], dsp[4 * g + 1], dsp[4 * g + 2], dsp[4 * g + 3]);
            *reinterpret_cast<uint4*>(sDS + sw128_offset(r, 64 * w + 32 * h + 8 * g)) = v4;
          }
        }
      }
      tmem_wait_st();
      if (!ok) break;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->ds_ready);
    }
    // ------------------------------------------------------------ dK (w = 0), dV (w = 1)
    if (ok && n > 0) {
      ok = mbar_wait_warp(&bars->acc_done, 0, abort_flag, p.err, p.wait_ns);
      tc_fence_after();
    }
    // TMEM loads are warp-collective: every lane loads, only rows inside the sequence store.
    if (ok) {
      const bool store = key < p.N;
      const float mul = w == 0 ? p.scale : (DROP ? p.drop_scale : 1.f);
      __nv_bfloat16* dst = (w == 0 ? dk : dv) + (row_off + key) * D;
      const uint32_t col0 = w == 0 ? C::COL_DK : 256u;
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t a[32];
        if (n > 0) {
          tmem_ld32_wait(lane_base + col0 + cc * 32, a);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) a[e] = 0u;
        }
        if (!store) continue;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint4 wv;
          wv.x = pack_bf16x2(__uint_as_float(a[8 * g]) * mul, __uint_as_float(a[8 * g + 1]) * mul);
          wv.y = pack_bf16x2(__uint_as_float(a[8 * g + 2]) * mul, __uint_as_float(a[8 * g + 3]) * mul);
          wv.z = pack_bf16x2(__uint_as_float(a[8 * g + 4]) * mul, __uint_as_float(a[8 * g + 5]) * mul);
          wv.w = pack_bf16x2(__uint_as_float(a[8 * g + 6]) * mul, __uint_as_float(a[8 * g + 7]) * mul);
          *reinterpret_cast<uint4*>(dst + cc * 32 + 8 * g) = wv;
        }
      }
    }
  } else if (warp >= 14) {
    if constexpr (D == 128) regs_release_to<kRegsControl>();  // idle control warps
  } else if (warp < 4) {
    // ------------------------------------------------------------ dQ partials
    if constexpr (D == 128) regs_grow_to<kRegsDrain>();
    const uint32_t lane_base = tb + (static_cast<uint32_t>((warp & 3) << 5) << 16);
    bool ok = true;
    int n = 0;
    const int wq = warp & 3;
    for (int i = first; ok && i >= 0; i = next_q(p, u, i)) {
      ok = mbar_wait_warp(&bars->dq_full, n & 1, abort_flag, p.err, p.wait_ns);
      if (!ok) break;
      tc_fence_after();
      {
        // Lane = query row.  Each warp copies its 32 rows x d columns of the partial out of
        // TMEM into [32 q][32 d] fp32 boxes with the 128-byte swizzle (16-byte stores, no
        // bank conflicts), releases the TMEM columns at once, and hands the boxes to the TMA
        // unit as bulk reduce-adds into the accumulator.  Warps 0-1 stage in this block's dO
        // stage (its MMAs are done with it; the next dO load into it waits for these reads),
        // warps 2-3 in the dS^T tile (the next phase B waits for these reads).
        const int q0 = i * kBlk + 32 * wq;
        uint8_t* st = wq < 2 ? sQ + (n & 1) * 2 * C::TILE + C::TILE + wq * (D / 32) * 4096
                             : sDS + (wq - 2) * (D / 32) * 4096;
        {
          uint32_t v[D];
          if constexpr (D == 128) {
            tmem_ld128_wait(lane_base + s_reg(n), v);
          } else {
            tmem_ld64_wait(lane_base + C::COL_DQ, lane_base + C::COL_DQ + 32, v);
          }
          tc_fence_before();
          mbar_arrive(&bars->dq_free);
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint8_t* row = st + cc * 4096 + lane * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<uint4*>(row + ((j ^ (lane & 7)) << 4)) =
                  make_uint4(v[32 * cc + 4 * j], v[32 * cc + 4 * j + 1],
                             v[32 * cc + 4 * j + 2], v[32 * cc + 4 * j + 3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          // The boxes in the dS^T tile go to the TMA first: the next phase B waits for them,
          // while the dO stage is only needed again two blocks later.
          bool go = true;
          if (wq < 2) go = mbar_wait(&bars->sds_free, n & 1, abort_flag, p.err, p.wait_ns);
          if (go && q0 < p.N) {
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc)
              tma_reduce_add_3d(&mdq, st + cc * 4096, 32 * cc, q0, u.bh);
            bulk_commit_group();
            bulk_wait_group_read<0>();
          }
          mbar_arrive(wq < 2 ? &bars->do_empty[n & 1] : &bars->sds_free);
        }
        __syncwarp();
      }
      ++n;
    }
  }

  if (warp < 4 && lane == 0) bulk_wait_group_all();
  tc_fence_before();
  __syncthreads();
  if (bars->abort && tid == 0) {
    // Let any bulk copy still in flight land before the CTA's shared memory is released.
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 1000000ull) {
    }
  }
  __syncthreads();
  if (warp == kProducerWarp) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
}

template <int D, bool DROP>
cudaError_t bwd_launch(const Problem& p, const void* q, const void* k, const void* v,
                       const float* lse, const void* dO, const float* Dsum, float* dq_acc,
                       void* dk, void* dv, cudaStream_t s) {
  CUtensorMap mq, mk, mv, mdo, mdq;
  const int BH = p.B * p.H;
  if (!make_head_map(&mq, q, BH, p.N, D) || !make_head_map(&mk, k, BH, p.N, D) ||
      !make_head_map(&mv, v, BH, p.N, D) || !make_head_map(&mdo, dO, BH, p.N, D) ||
      !make_acc_map(&mdq, dq_acc, BH, p.N, D))
    return cudaErrorInvalidValue;
  static std::atomic<bool> attr_set[64];  // per device; a race repeats the same call
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev].load()) {
    cudaError_t e = cudaFuncSetAttribute(bwd_sm103_kernel<D, DROP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    if constexpr (D == 128) {
      // The in-kernel register split (drain, softmax, control) adds up to exactly 128 per
      // thread at launch: a kernel built with another count would wait forever in
      // setmaxnreg, so it is refused here.
      cudaFuncAttributes fattr;
      e = cudaFuncGetAttributes(&fattr, bwd_sm103_kernel<D, DROP>);
      if (e != cudaSuccess) return e;
      if (fattr.numRegs != kRegsLaunch) return cudaErrorInvalidConfiguration;
    }
    attr_set[dev].store(true);
  }
  const int nkb = (p.N + kBlk - 1) / kBlk;
  dim3 grid(static_cast<unsigned>(BH) * nkb);
  return launch_dependent(bwd_sm103_kernel<D, DROP>, grid, dim3(kThreads), Cfg<D>::SMEM, s, mq,
                          mk, mv, mdo, mdq, lse, Dsum, dq_acc, static_cast<__nv_bfloat16*>(dk),
                          static_cast<__nv_bfloat16*>(dv), p);
}

}  // namespace

cudaError_t launch_bwd_sm103(const Problem& p, const void* q, const void* k, const void* v,
                             const float* lse, const void* dO, const float* Dsum, float* dq_acc,
                             void* dk, void* dv, cudaStream_t s) {
  if (p.drop_threshold > 0)
    return p.d == 64 ? bwd_launch<64, true>(p, q, k, v, lse, dO, Dsum, dq_acc, dk, dv, s)
                     : bwd_launch<128, true>(p, q, k, v, lse, dO, Dsum, dq_acc, dk, dv, s);
  return p.d == 64 ? bwd_launch<64, false>(p, q, k, v, lse, dO, Dsum, dq_acc, dk, dv, s)
                   : bwd_launch<128, false>(p, q, k, v, lse, dO, Dsum, dq_acc, dk, dv, s);
}

}  // namespace fa
