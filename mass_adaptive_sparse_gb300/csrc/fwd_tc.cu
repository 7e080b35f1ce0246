// MALA forward on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// "MassAlloc Attention: Let Attention Allocate Its Own Compute", Algorithm 1
// and §2.2 Eq. (3): for each 128-row query block, the legal 128-key blocks
// are visited from the diagonal toward earlier keys.  Every tile's scores
// S = Q K^T are formed; the tile is skipped iff, for every valid row,
// rowmax(S) - m - log l < log(tau / L_q) (l = 0 keeps).  A skipped tile issues
// no V load and no P V product and leaves (m, l, O) unchanged (App. A.1).
//
// One CTA = two adjacent query blocks (slots 0 and 1) of one head; both walk
// the same key blocks, so each K tile is loaded once for the pair.  384 threads;
// warps 0-3 hold the control roles:
//   warps 0, 3  sequencers, one thread per slot: O_s += P_s V, then at once the
//              slot's next S_s = Q_s K^T.  The tensor pipe takes new MMAs only
//              as it drains, so each sequencer gathers everything its turn
//              needs (vote, P, V, K) first, then takes the turn from the other
//              by a token barrier.  The slots thus alternate on the pipe in a
//              fixed order, one slot's softmax overlapping the other slot's
//              MMAs, and only the hand-off separates two MMA groups.  A K or V
//              stage is released by one commit per slot.  Warp 3 also owns TMEM.
//   warp 1     V loader (one thread): follows the votes in step order and loads
//              the V tile of a key block once a slot keeps it.  The 2-stage V
//              ring takes one phase per step; a step that no slot keeps
//              completes its phase with a plain arrival.  A sequencer ends
//              each step only once the loader has seen all of its votes, and
//              votes and keep flags alternate between two barriers / words by
//              step parity, so no wait can meet a phase from two steps later.
//   warp 2     TMA producer: both Q tiles once, then a 3-stage K ring.
//   warps 4-7  softmax of slot 0, warps 8-11 softmax of slot 1: thread r owns
//              query row r of its slot (TMEM lane r) and all 128 columns, so
//              the row max, the Eq. 3 test and the row sums need no exchange;
//              the slot's 128 rows vote on the tile with one barrier reduction.
// TMEM: S_0 (columns 0-127), S_1 (128-255), O_0 (256-383), O_1 (384-511).
// P (bf16, two keys per 32-bit column) is written over the slot's consumed S:
// keys 0-63 into its columns 0-31 and keys 64-127 into columns 64-95; the next
// Q K^T of that slot is issued after its P V on the same tensor pipe, which
// executes them in order.  The running max is only moved when it grows by more
// than 2^8 (log2 units); P and l are kept relative to the max in use, which
// leaves m + log l = log Z unchanged, so the test is unaffected.
#include <cuda_bf16.h>

#include "mala_internal.h"
#include "tc_common.cuh"

namespace mala {
namespace {

using namespace tc;

constexpr int kD = 128;                 // head dim
constexpr int kBlk = 128;               // B_q = B_k
constexpr int kTile = kBlk * kD * 2;    // 32 KiB: one 128 x 128 bf16 tile
constexpr int kHalf = kTile / 2;        // one 64-column TMA box
constexpr int kNK = 3;                  // K stages
constexpr int kNV = 2;                  // V stages
constexpr int kThreads = 384;
constexpr int kSmem = kTile * (2 + kNK + kNV) + 1024;
constexpr uint32_t kColO = 256;
constexpr float kRescale = 8.0f;        // move the running max only past 2^8 growth

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kNK], k_empty[kNK];
  uint64_t v_full[kNV], v_empty[kNV];
  uint64_t s_full[2];     // Q K^T of the slot complete (so is its previous P V)
  uint64_t dec[2][2];     // [slot][step parity]: the slot's rows voted (keep_flag written), S read out
  uint64_t p_ready[2];    // P of a kept tile is in TMEM (one arrival per warp)
  uint64_t o_done[2];     // every MMA of the slot complete
  uint64_t vl_done[2];    // [step parity]: the V loader has seen every vote of the step
  uint64_t tok[2];        // [slot]: the other slot's sequencer has taken its turn
  uint64_t fin[2];        // every MMA of a sequencer complete (its own wait before exit)
};

// Four consecutive output values to global memory (8 bytes of bf16, 16 of fp32).
template <typename Tout>
__device__ __forceinline__ void store_out4(Tout* dst, float4 x);

template <>
__device__ __forceinline__ void store_out4<__nv_bfloat16>(__nv_bfloat16* dst, float4 x) {
  *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16(x.x, x.y), pack_bf16(x.z, x.w));
}

template <>
__device__ __forceinline__ void store_out4<float>(float* dst, float4 x) {
  *reinterpret_cast<float4*>(dst) = x;
}

// Scores of the columns past `last` (the last legal one) become -inf.
__device__ __forceinline__ void mask_cols(uint32_t* sr, int last) {
#pragma unroll
  for (int c = 0; c < 64; ++c)
    if (c > last) sr[c] = 0xff800000u;
}

// 64 raw scores -> 32 packed bf16 pairs of P = exp2(S * scale - m) in sr[0..31];
// acc sums P exactly (two lanes per register), r0 / r1 sum the even / odd
// columns' P as rounded to bf16.
__device__ __forceinline__ void exp_pack(uint32_t* sr, uint64_t nsc2, uint64_t nm2, uint64_t& acc, float& r0,
                                         float& r1) {
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    float e0, e1;
    f2_split(fma2(f2(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), nsc2, nm2), e0, e1);
    const float p0 = ex2(e0), p1 = ex2(e1);
    const uint32_t w = pack_bf16(p0, p1);
    acc = add2(acc, f2(p0, p1));
    add_bf16x2(r0, r1, w);
    sr[c] = w;
  }
}

// Epilogue of a softmax warp: its 32 query rows of O / l (128 columns) leave
// TMEM 32 columns at a time through a padded shared-memory tile (rows 36 floats
// apart: the row-wise float4 writes and the four-rows-at-a-time float4 reads
// both take the minimum four wavefronts), so that each global store
// instruction writes four whole row segments rather than 32 scattered pieces.
// `stage` is the slot's Q buffer, free once the slot's products are done.  Not
// inlined: that keeps the main loop's code as it was (0.4 ms faster at 128K
// than the inlined form).  o_out: [lb, seqlen_q, heads_q, 128] of Tout; rows at
// or past Lq are not written.
template <typename Tout>
__device__ __noinline__ void write_o(uint8_t* smem_raw, uint32_t stage, int warp, int lane, int qb, int Lq, int row0,
                                     int bc, int h, int lb, int seqlen_q, int heads_q, void* o_out, uint32_t o_taddr,
                                     float inv, int* status) {
  fence_proxy_async_smem();
  float* tp = reinterpret_cast<float*>(smem_raw + (stage - smem_u32(smem_raw))) + (warp & 3) * (32 * 36);
  const int rr0 = lane >> 3, cc = 4 * (lane & 7);
  const size_t o_elems = static_cast<size_t>(lb) * seqlen_q * heads_q * kD;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float o[32];
    tmem_ld32_sync(o_taddr + c * 32, reinterpret_cast<uint32_t*>(o));
    float4* w4 = reinterpret_cast<float4*>(tp + lane * 36);
#pragma unroll
    for (int u = 0; u < 8; ++u)
      w4[u] = make_float4(o[4 * u] * inv, o[4 * u + 1] * inv, o[4 * u + 2] * inv, o[4 * u + 3] * inv);
    __syncwarp();
#pragma unroll
    for (int k4 = 0; k4 < 8; ++k4) {
      const int rr = 4 * k4 + rr0;
      const int qr = qb * kBlk + 32 * (warp & 3) + rr;
      const float4 x = *reinterpret_cast<const float4*>(tp + rr * 36 + cc);
      const size_t off = ((static_cast<size_t>(bc) * seqlen_q + row0 + qr) * heads_q + h) * kD + 32 * c + cc;
      if (qr < Lq && dbg_idx(off + 3, o_elems, status)) store_out4<Tout>(static_cast<Tout*>(o_out) + off, x);
    }
    __syncwarp();
  }
}

template <typename Tout>
__global__ void __launch_bounds__(kThreads, 1)
fwd_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
              const __grid_constant__ CUtensorMap mv, const FwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) Bars bars;
  __shared__ uint32_t tmem_sh;
  __shared__ int keep_flag[2][2];     // [slot][step parity]
  __shared__ int abort_flag;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = base;                       // slot s at sQ + s * kTile
  const uint32_t sK = base + 2 * kTile;
  const uint32_t sV = base + kTile * (2 + kNK);

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  // CTA order (CTAs start in index order): sequence, KV head, query-block pair
  // (heaviest first), then the query heads of the KV head.  The CTAs running at
  // once then walk the key blocks of one KV head side by side, so each K and V
  // tile comes from DRAM about once per launch (1.12 GB of DRAM traffic at
  // 128K x 8 heads, against 7.9 GB with heads fastest) and from L2 after that.
  const int G = a.Hq / a.Hkv;
  const int npairs = (((a.cu ? a.Lmax : a.Lq) + kBlk - 1) / kBlk + 1) / 2;
  const int cta = static_cast<int>(blockIdx.x);
  const int gi = cta % G, py = (cta / G) % npairs, bhk = cta / G / npairs;
  const int h = (bhk % a.Hkv) * G + gi, b = bhk / a.Hkv;
  // this CTA's sequence: its lengths, first row and batch coordinate in the layout
  const SeqSpan sq = seq_span(a, b);
  const int Lq = sq.Lq, Lk = sq.Lk, row0 = sq.row0, bc = sq.bc;
  const int Tr = (Lq + kBlk - 1) / kBlk, Tc = (Lk + kBlk - 1) / kBlk;
  // tile rows / columns of mask and counts (a packed batch pads each sequence to Lmax)
  const int mTr = a.cu ? (a.Lmax + kBlk - 1) / kBlk : Tr, mTc = a.cu ? mTr : Tc;
  const int lb = a.cu ? 1 : a.B;         // batch extent of the layout (a packed batch is one run of rows)
  const int pair = (Tr + 1) / 2 - 1 - py;   // heaviest pairs first
  if (pair < 0) return;                  // past the sequence's query blocks (packed batches)
  const int nslots = (2 * pair + 1 < Tr) ? 2 : 1;
  const int hk = h / (a.Hq / a.Hkv);
  // top key block of each slot; the pair walks from the higher one down to 0
  int jtop_s[2];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int qb = 2 * pair + s;
    jtop_s[s] = a.causal ? min(Tc - 1, (min(Lq, qb * kBlk + kBlk) - 1) / kBlk) : Tc - 1;
  }
  if (nslots == 1) jtop_s[1] = -1;
  const int jtop = max(jtop_s[0], jtop_s[1]);
  const int ntiles = jtop + 1;
  // slot s takes part in steps t >= first[s] (key block jtop - t); its local
  // step is u = t - first[s].  The two slots' first steps differ by at most one.
  const int first0 = jtop - jtop_s[0];
  const int first1 = nslots == 2 ? jtop - jtop_s[1] : ntiles;

  if (warp == 3) tmem_alloc<512>(smem_u32(&tmem_sh));
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bars.q_full), 1);
    // a K or V stage is released by one arrival per slot
    for (int i = 0; i < kNK; ++i) { mbar_init(smem_u32(&bars.k_full[i]), 1); mbar_init(smem_u32(&bars.k_empty[i]), nslots); }
    for (int i = 0; i < kNV; ++i) { mbar_init(smem_u32(&bars.v_full[i]), 1); mbar_init(smem_u32(&bars.v_empty[i]), nslots); }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bars.s_full[s]), 1);
      mbar_init(smem_u32(&bars.dec[s][0]), 1);
      mbar_init(smem_u32(&bars.dec[s][1]), 1);
      mbar_init(smem_u32(&bars.p_ready[s]), 4);   // one arrival per warp of the slot
      mbar_init(smem_u32(&bars.o_done[s]), 1);
    }
    mbar_init(smem_u32(&bars.vl_done[0]), 1);
    mbar_init(smem_u32(&bars.vl_done[1]), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars.tok[i]), 1);
      mbar_init(smem_u32(&bars.fin[i]), 1);
    }
    fence_barrier_init();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_sh;
  volatile int* abortp = &abort_flag;

  if (warp == 2) {
    // ---------------- TMA producer: Q tiles once, then the K ring ----------------
    if (lane == 0) {
      prefetch_tensormap(&mq);
      prefetch_tensormap(&mk);
      const uint32_t qf = smem_u32(&bars.q_full);
      mbar_expect_tx(qf, kTile * nslots);
      for (int s = 0; s < nslots; ++s) {
        const int row = row0 + (2 * pair + s) * kBlk;
        if (dbg_box(64, h, row, bc, kD, a.Hq, row0, row0 + Lq, a.Lq, lb, a.status)) {
          tma_load_4d(sQ + s * kTile, &mq, qf, 0, h, row, bc);
          tma_load_4d(sQ + s * kTile + kHalf, &mq, qf, 64, h, row, bc);
        }
      }
      // test hook (failure detection): CTA (0, 0) leaves its first K tile
      // unloaded, so the waits for it expire and the CTA gives up
      const bool drop = a.inject != 0 && cta == 0;
      int issued = 0;                     // steps reached (loads issued, or the one dropped)
      for (int t = 0; t < ntiles; ++t) {
        const int st = t % kNK, n = t / kNK;
        if (n > 0 && !mbar_wait(smem_u32(&bars.k_empty[st]), (n - 1) & 1, abortp, a.status)) break;
        if (!(drop && t == 0)) {
          const uint32_t kf = smem_u32(&bars.k_full[st]);
          const int row = row0 + (jtop - t) * kBlk;
          mbar_expect_tx(kf, kTile);
          if (dbg_box(64, hk, row, bc, kD, a.Hkv, row0, row0 + Lk, a.Lk, lb, a.status)) {
            tma_load_4d(sK + st * kTile, &mk, kf, 0, hk, row, bc);
            tma_load_4d(sK + st * kTile + kHalf, &mk, kf, 64, hk, row, bc);
          }
        }
        ++issued;
      }
      // every issued load lands before the CTA can finish
      mbar_drain(smem_u32(&bars.q_full), 0, a.status);
      for (int t = max(0, issued - kNK); t < issued; ++t)
        if (!(drop && t == 0)) mbar_drain(smem_u32(&bars.k_full[t % kNK]), (t / kNK) & 1, a.status);
    }
  } else if (warp == 1) {
    // ---------------- V loader ----------------
    if (lane == 0) {
      prefetch_tensormap(&mv);
      const int first[2] = {first0, first1};
      int armed = -1;              // last step whose V phase this thread armed
      for (int t = 0; t < ntiles; ++t) {
        const int vs = t % kNV;
        bool load = false, ok = true;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          if (!ok || t < first[s]) continue;
          const int u = t - first[s];
          ok = mbar_wait(smem_u32(&bars.dec[s][u & 1]), (u >> 1) & 1, abortp, a.status);
          if (ok && !load && keep_flag[s][u & 1]) {
            // the stage's previous step (t - 2) is done with it
            if (t >= kNV) ok = mbar_wait(smem_u32(&bars.v_empty[vs]), (t / kNV - 1) & 1, abortp, a.status);
            if (ok) {
              const uint32_t vf = smem_u32(&bars.v_full[vs]);
              mbar_expect_tx(vf, kTile);
              const int row = row0 + (jtop - t) * kBlk;
              if (dbg_box(64, hk, row, bc, kD, a.Hkv, row0, row0 + Lk, a.Lk, lb, a.status)) {
                tma_load_4d(sV + vs * kTile, &mv, vf, 0, hk, row, bc);
                tma_load_4d(sV + vs * kTile + kHalf, &mv, vf, 64, hk, row, bc);
              }
              load = true;
              armed = t;
            }
          }
        }
        if (!ok) break;
        if (!load) {
          // no slot keeps this key block: complete the step's phase without a load
          if (t >= kNV && !mbar_wait(smem_u32(&bars.v_empty[vs]), (t / kNV - 1) & 1, abortp, a.status)) break;
          mbar_arrive(smem_u32(&bars.v_full[vs]));
          armed = t;
        }
        mbar_arrive(smem_u32(&bars.vl_done[t & 1]));
      }
      // loads of the last armed steps land before the CTA can finish
      for (int t = max(0, armed - 1); t <= armed; ++t)
        mbar_drain(smem_u32(&bars.v_full[t % kNV]), (t / kNV) & 1, a.status);
    }
  } else if (warp == 0 || warp == 3) {
    // ---------------- sequencers: one thread per slot, turns passed by token ----------------
    const int s = warp == 0 ? 0 : 1;
    if (lane == 0 && s < nslots) {
      constexpr uint32_t idesc_qk = idesc_f16(1, 0, 0, kBlk, kBlk);
      constexpr uint32_t idesc_pv = idesc_f16(1, 0, 1, kBlk, kD);
      const int first = s == 0 ? first0 : first1;
      const bool solo = nslots == 1;
      // the slot whose first step comes first takes the first turn
      const bool leads = solo || (s == 0 ? first0 <= first1 : first1 < first0);
      const uint64_t dq = desc_kmajor_sw128(sQ + s * kTile);
      const uint32_t d_s = tmem + s * 128, d_o = tmem + kColO + s * 128;
      int turn = 0;                // turns taken
      // wait for the other slot's last turn (its MMAs are then queued ahead)
      auto take_turn = [&]() -> bool {
        const int k = leads ? turn - 1 : turn;
        return solo || k < 0 || mbar_wait(smem_u32(&bars.tok[s]), k & 1, abortp, a.status);
      };
      auto pass_turn = [&]() {
        if (!solo) mbar_arrive(smem_u32(&bars.tok[1 - s]));
        ++turn;
      };
      int kwaited = first - 1;     // K stages waited for, in step order
      auto wait_k = [&](int t) -> bool {
        while (kwaited < t) {
          ++kwaited;
          if (!mbar_wait(smem_u32(&bars.k_full[kwaited % kNK]), (kwaited / kNK) & 1, abortp, a.status))
            return false;
        }
        return true;
      };
      // S_s = Q_s K(t)^T, reported at once
      auto issue_qk = [&](int t) {
        const uint64_t dk = desc_kmajor_sw128(sK + (t % kNK) * kTile);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = ((k / 4) * kHalf + (k % 4) * 32) >> 4;
          mma_ss(d_s, dq + off, dk + off, idesc_qk, k > 0);
        }
        mma_commit(smem_u32(&bars.s_full[s]));
      };
      bool ok = mbar_wait(smem_u32(&bars.q_full), 0, abortp, a.status);
      // steps before this slot's first one: it reads neither their K nor their V
      for (int t = 0; t < first; ++t) {
        mbar_arrive(smem_u32(&bars.k_empty[t % kNK]));
        mbar_arrive(smem_u32(&bars.v_empty[t % kNV]));
      }
      // turn 0: the slot's first product
      ok = ok && wait_k(first) && take_turn();
      if (ok) {
        fence_after_sync();
        issue_qk(first);
        pass_turn();
        mma_commit(smem_u32(&bars.k_empty[first % kNK]));
      }
      int nkeep = 0;
      for (int t = first; ok && t < ntiles; ++t) {
        const int vs = t % kNV, u = t - first;
        const bool more = t + 1 < ntiles;
        // everything this turn needs, gathered before taking it, in the order
        // it becomes ready (P last but the turn)
        ok = mbar_wait(smem_u32(&bars.dec[s][u & 1]), (u >> 1) & 1, abortp, a.status);
        const bool keep = ok && keep_flag[s][u & 1];
        if (ok && more) ok = wait_k(t + 1);
        if (keep) ok = ok && mbar_wait(smem_u32(&bars.v_full[vs]), (t / kNV) & 1, abortp, a.status);
        if (keep) ok = ok && mbar_wait(smem_u32(&bars.p_ready[s]), nkeep & 1, abortp, a.status);
        ok = ok && take_turn();
        if (!ok) break;
        fence_after_sync();
        if (keep) {
          // O_s += P_s V: P of keys 0-63 in columns 0-31 of S_s, keys 64-127 in 64-95
          const uint64_t dv = desc_mnmajor_sw128(sV + vs * kTile, kHalf, 1024);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ts(d_o, d_s + (k / 4) * 64 + (k % 4) * 8, dv + ((k * 2048) >> 4), idesc_pv,
                   (nkeep > 0 || k > 0) ? 1u : 0u);
          ++nkeep;
        }
        if (more) {
          issue_qk(t + 1);
        } else {
          mma_commit(smem_u32(&bars.o_done[s]));
        }
        pass_turn();
        if (more) mma_commit(smem_u32(&bars.k_empty[(t + 1) % kNK]));
        // The V loader has seen every vote of this step (and waited for the
        // stage's previous phase) before this slot releases the stage or
        // takes its next turn, so no barrier completes a phase ahead of its waiter.
        ok = mbar_wait(smem_u32(&bars.vl_done[t & 1]), (t >> 1) & 1, abortp, a.status);
        if (ok) mma_commit(smem_u32(&bars.v_empty[vs]));
      }
      // all MMAs of this thread complete before TMEM is released
      mma_commit(smem_u32(&bars.fin[s]));
      mbar_drain(smem_u32(&bars.fin[s]), 0, a.status);
    }
  } else if (warp >= 4) {
    // ---------------- softmax: thread r of slot s owns query row r ----------------
    const int s = (warp >> 2) - 1, r = tid & 127;
    if (s < nslots) {
      const int qb = 2 * pair + s;
      const int qrow = qb * kBlk + r;
      const bool valid = qrow < Lq;
      const int lim = a.causal ? min(qrow, Lk - 1) : Lk - 1;       // last legal key of this row
      const float thr = a.log2_tau - log2f(a.causal ? static_cast<float>(qrow + 1) : static_cast<float>(Lk));
      const bool test = a.tau > 0.f;
      const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
      const uint32_t colS = s * 128, colO = kColO + s * 128;
      // row state: l is the exact fp32 sum of P (Eq. 3 test and lse); lr sums
      // the bf16-rounded P that enters the P V product (normalises O)
      float m_used = -INFINITY, l = 0.f, lr = 0.f;
      int nret = 0, it = 0;
      bool ok = true;
      uint8_t* mask_row = a.mask ? a.mask + ((static_cast<size_t>(b) * a.Hq + h) * mTr + qb) * mTc : nullptr;
      const int t0 = jtop - jtop_s[s];

      // After a timed-out wait the loop runs on without breaking (waits then
      // fail at once), so the slot's barrier reductions always stay matched.
      for (int t = t0; t < ntiles; ++t) {
        const int j = jtop - t;
        ok = mbar_wait(smem_u32(&bars.s_full[s]), it & 1, abortp, a.status) && ok;
        ++it;
        fence_after_sync();
        // S is streamed in two 64-column halves (64 live scores per thread):
        // the max pass reads both, the exponent pass reuses the second half
        // still in registers and reloads the first.
        // Interior tiles (not diagonal, no ragged edge) need no masking.
        const bool interior = (a.causal ? j < qb : (j + 1) * kBlk <= Lk) && (qb + 1) * kBlk <= Lq;
        const int cmax = valid ? lim - j * kBlk : -1;   // last legal column of this row in the tile
        uint32_t sr[64];                        // raw scores Q.K of one half, later packed P
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          tmem_ld64_sync(lane_addr + colS + 64 * hf, sr);
          if (!interior) mask_cols(sr, cmax - 64 * hf);
          // row max over legal keys (raw dot products; the scale is positive)
#pragma unroll
          for (int c = 0; c < 64; c += 2)
            mx[(c >> 1) & 7] = max3(mx[(c >> 1) & 7], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
        }
        const float mraw = max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
        const float mt = mraw * a.scale_log2;
        const bool has = valid && lim >= j * kBlk;
        const int keep_row = has && (!test || l == 0.f || !(mt - m_used - lg2(l) < thr));
        fence_before_sync();                    // the S read-out precedes the hand-back
        const int keep = named_vote_or(1 + s, 128, keep_row);
        const int u = it - 1;                   // local step of this slot
        if (r == 0) {
          keep_flag[s][u & 1] = keep;
          if (mask_row && dbg_idx(((static_cast<size_t>(b) * a.Hq + h) * mTr + qb) * mTc + j,
                                  static_cast<size_t>(a.B) * a.Hq * mTr * mTc, a.status))
            mask_row[j] = static_cast<uint8_t>(keep);
          mbar_arrive(smem_u32(&bars.dec[s][u & 1]));
        }
        if (!keep) continue;
        ++nret;
        // online update (Algorithm 1), with a lazily moved reference max
        float alpha = 1.f;
        if (has && mt > m_used + kRescale) {
          alpha = (m_used == -INFINITY) ? 0.f : ex2(m_used - mt);
          m_used = mt;
        }
        const float mref = (m_used == -INFINITY) ? 0.f : m_used;
        const uint64_t nsc2 = f2(a.scale_log2, a.scale_log2), nm2 = f2(-mref, -mref);
        uint64_t acc = f2(0.f, 0.f);
        float r0 = 0.f, r1 = 0.f;
        // P = exp2(S * scale - m_ref) as bf16 pairs; P of keys 64-127 goes over
        // the (consumed) scores of keys 64-95, P of keys 0-63 over keys 0-31
        exp_pack(sr, nsc2, nm2, acc, r0, r1);
        tmem_st32(lane_addr + colS + 64, sr);
        tmem_ld64_sync(lane_addr + colS, sr);
        if (!interior) mask_cols(sr, cmax);
        exp_pack(sr, nsc2, nm2, acc, r0, r1);
        float rowsum, rowsum_r;
        {
          float x0, x1;
          f2_split(acc, x0, x1);
          rowsum = x0 + x1;
          rowsum_r = r0 + r1;
        }
        // O rescale when the reference max moved.  The slot's previous P V is
        // complete: it was issued before the Q K^T whose completion s_full reported.
        if (nret > 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32_sync(lane_addr + colO + c * 32, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(lane_addr + colO + c * 32, o);
          }
        }
        tmem_st32(lane_addr + colS, sr);
        tmem_st_wait();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars.p_ready[s]));   // P is in TMEM
        l = l * alpha + rowsum;
        lr = lr * alpha + rowsum_r;
      }

      // epilogue: every MMA of the slot complete, then O / l and lse = m + log l
      ok = mbar_wait(smem_u32(&bars.o_done[s]), 0, abortp, a.status) && ok;
      fence_after_sync();
      if (__all_sync(0xffffffffu, ok && !*abortp)) {
        const bool store = valid && dbg_idx((static_cast<size_t>(bc) * a.Hq + h) * a.Lq + row0 + qrow,
                                            static_cast<size_t>(lb) * a.Hq * a.Lq, a.status);
        const float inv = 1.f / lr;
        write_o<Tout>(smem_raw, sQ + s * kTile, warp, lane, qb, Lq, row0, bc, h, lb, a.Lq, a.Hq, a.o, lane_addr + colO, inv,
                      a.status);
        if (store) a.lse[(static_cast<size_t>(bc) * a.Hq + h) * a.Lq + row0 + qrow] = (m_used + log2f(l)) * kLn2;
        if (a.counts != nullptr && r == 0 &&
            dbg_idx((static_cast<size_t>(b) * a.Hq + h) * mTr + qb, static_cast<size_t>(a.B) * a.Hq * mTr, a.status))
          a.counts[(static_cast<size_t>(b) * a.Hq + h) * mTr + qb] = nret;
      }
      fence_before_sync();
    }
  }

  __syncthreads();
  if (warp == 3) {
    fence_after_sync();
    tmem_dealloc<512>(tmem);
  }
}

}  // namespace

bool fwd_tc_supported(const FwdArgs& a) {
  return a.in_dt == kBF16 && a.D == kD && a.blk == kBlk;
}

cudaError_t launch_fwd_tc(const FwdArgs& a, cudaStream_t s, int* launches) {
  CUtensorMap mq, mk, mv;
  const int lb = a.cu ? 1 : a.B;           // a packed batch is one run of Lq rows
  if (!encode_bshd_map(&mq, a.q, lb, a.Lq, a.Hq, kD, kBlk) ||
      !encode_bshd_map(&mk, a.k, lb, a.Lk, a.Hkv, kD, kBlk) ||
      !encode_bshd_map(&mv, a.v, lb, a.Lk, a.Hkv, kD, kBlk))
    return cudaErrorInvalidValue;
  const int tr = ((a.cu ? a.Lmax : a.Lq) + kBlk - 1) / kBlk;
  const dim3 grid(static_cast<unsigned>(a.Hq) * a.B * ((tr + 1) / 2));
  ++*launches;
  cudaError_t e;
  if (a.out_dt == kBF16) {
    auto kern = fwd_tc_kernel<__nv_bfloat16>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, kSmem, s>>>(mq, mk, mv, a);
  } else {
    auto kern = fwd_tc_kernel<float>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, kSmem, s>>>(mq, mk, mv, a);
  }
  return cudaGetLastError();
}

}  // namespace mala
