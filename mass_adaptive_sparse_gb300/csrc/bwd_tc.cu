// MALA backward on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// "MassAlloc Attention: Let Attention Allocate Its Own Compute", Algorithm 2
// and §2.2 Eq. (4), key-major (App. A.1): one CTA owns a 128-key block of one
// KV head and visits, for each query head of the group, the query blocks with
// a legal entry in ascending order.  Each tile's transposed scores
// S^T = K Q^T are recomputed; the tile is skipped iff S - lse < log(tau / L_q)
// on every valid causal entry.  A skipped tile loads no dO and runs no
// post-score work.  A retained tile runs
//   P^T = exp(S^T - lse), dP^T = V dO^T, dS^T = P^T o (dP^T - D),
//   dV += P^T dO, dK += dS^T Q, dQ += dS K  (formed as dQ^T = K^T dS^T and
//   added to an fp32 accumulator by bulk tensor reduce-adds).
//
// All post-score products run on fp16 operands (exact fp16 copies of Q, K, V,
// dO made by the preprocess kernel); P and dS are rounded to fp16, which keeps
// the gradients within 2e-4 mean relative error where bf16 would not.
//
// 320 threads: warps 0-7 = two "math" warpgroups; thread (c, r) of group c
// owns key row r = TMEM lane r and the 64 query columns [64c, 64c + 64) of
// S^T, P^T, dP^T and dS (and, for the dQ^T read-out, head dim r of those 64
// queries); warp 8 = TMA producer (K, V once; Q ring); warp 9 =
// MMA issuer.  dS is stored pre-multiplied by the softmax scale, so dQ and dK
// come out of the products already scaled.
// TMEM columns: two 128-column regions, tile t in region t & 1, each holding
// in turn S^T, P^T (fp16: queries 0-63 in its columns [0,32), 64-127 in
// [64,96)), dP^T (after dV has read P^T) and dQ^T (after the math warps have
// read dP^T); then [256,384) dV and [384,512) dK.  The next tile's scores go
// into the other region as soon as the dQ^T left there has been read out, so
// neither dP^T nor the scores wait for the dQ hand-off of the tile before.
// dS is written to shared memory once, in the 128-byte-swizzled layout that
// is K-major for dK = dS^T Q (A = dS^T) and MN-major for dQ = dS K (A = dS).
//
// Hand-offs to the MMA warp are made as early as each can be: thread 0
// publishes a tile's decision right after the vote (its mask and counter
// bookkeeping come after), each math warp signals its part of P^T once its
// own TMEM stores have landed, and a skipped tile's Q slot goes back to the
// producer at the decision.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "mala_internal.h"
#include "tc_common.cuh"

namespace mala {
namespace {

using namespace tc;

constexpr int kD = 128;
constexpr int kBlk = 128;
constexpr int kTile = kBlk * kD * 2;    // 32 KiB of fp16
constexpr int kHalf = kTile / 2;
constexpr int kThreads = 320;
constexpr int kMath = 256;            // two math warpgroups
// shared memory: K, V, Q[2], dO, dS (doubles as dQ staging for queries 0-63),
// dQ staging for queries 64-127
constexpr int kOffK = 0, kOffV = kTile, kOffQ = 2 * kTile, kOffDO = 4 * kTile, kOffDS = 5 * kTile,
              kOffST = 6 * kTile;
constexpr int kSmem = 7 * kTile + 1024;
constexpr uint32_t kColDV = 256, kColDK = 384;
// TMEM region (S^T, P^T, dP^T, dQ^T) of tile t
__device__ __forceinline__ uint32_t region(int t) { return static_cast<uint32_t>(t & 1) * 128u; }

struct Bars {
  uint64_t kv_full;
  uint64_t q_full[2], q_empty[2];
  uint64_t do_full;
  uint64_t s_full, dec, p_ready, dp_full, ds_ready, dq_full, dq_free;
  uint64_t fin;
};



__device__ __forceinline__ float f16_lo(uint32_t w) { return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu))); }
__device__ __forceinline__ float f16_hi(uint32_t w) { return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16))); }
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }



__device__ __forceinline__ uint32_t pack_f16_2(uint64_t v) {
  float lo, hi;
  f2_split(v, lo, hi);
  return pack_f16(lo, hi);
}

// Four consecutive gradient values to global memory (16 bytes of fp32, 8 of bf16).
template <typename Tg>
__device__ __forceinline__ void store_grad4(Tg* dst, float4 x);

template <>
__device__ __forceinline__ void store_grad4<float>(float* dst, float4 x) {
  *reinterpret_cast<float4*>(dst) = x;
}

template <>
__device__ __forceinline__ void store_grad4<__nv_bfloat16>(__nv_bfloat16* dst, float4 x) {
  *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16(x.x, x.y), pack_bf16(x.z, x.w));
}

// Epilogue of a math warp: its 32 key rows x 64 columns (group cg) of dV and
// dK leave TMEM through a padded shared-memory tile (rows 36 floats apart: the
// row-wise float4 writes and the four-rows-at-a-time float4 reads both take the
// minimum four wavefronts), so that each global store instruction writes four
// whole 128-byte row segments rather than 32 scattered 16-byte pieces.  The
// tile sits in the K / V area, free once every product is done.  Not inlined:
// inlined, it changed the main loop's code and cost 0.5 ms at 128K.
// dv, dk: [lb, seqlen_k, heads_kv, 128] of Tg; key rows at or past Lk are not written.
template <typename Tg>
__device__ __noinline__ void write_dkdv(uint8_t* smem_raw, uint32_t sK, int warp, int lane, int cg, int nret, int kb,
                                        int Lk, int row0, int bc, int hk, int lb, int seqlen_k, int heads_kv, void* dv,
                                        void* dk, uint32_t lane_addr, int* status) {
  fence_proxy_async_smem();
  float* tp = reinterpret_cast<float*>(smem_raw + (sK - smem_u32(smem_raw))) + warp * (32 * 36);
  const int rr0 = lane >> 3, cc = 4 * (lane & 7);
  const size_t tensor_elems = static_cast<size_t>(lb) * seqlen_k * heads_kv * kD;
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    Tg* dst = static_cast<Tg*>(m == 0 ? dv : dk);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      uint32_t v[32];
      if (nret > 0) {
        tmem_ld32_sync(lane_addr + (m == 0 ? kColDV : kColDK) + 64 * cg + c * 32, v);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = 0u;
      }
      float4* w4 = reinterpret_cast<float4*>(tp + lane * 36);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        w4[u] = make_float4(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]),
                            __uint_as_float(v[4 * u + 2]), __uint_as_float(v[4 * u + 3]));
      __syncwarp();
#pragma unroll
      for (int k4 = 0; k4 < 8; ++k4) {
        const int rr = 4 * k4 + rr0;                          // row of this warp's tile
        const int kr = kb * kBlk + 32 * (warp & 3) + rr;       // key
        const float4 x = *reinterpret_cast<const float4*>(tp + rr * 36 + cc);
        const size_t off = ((static_cast<size_t>(bc) * seqlen_k + row0 + kr) * heads_kv + hk) * kD + 64 * cg + 32 * c + cc;
        if (kr < Lk && dbg_idx(off + 3, tensor_elems, status)) store_grad4<Tg>(dst + off, x);
      }
      __syncwarp();
    }
  }
}

template <typename Tg>
__global__ void __launch_bounds__(kThreads, 1)
bwd_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
              const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
              const __grid_constant__ CUtensorMap mdq, const BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) Bars bars;
  __shared__ uint32_t tmem_sh;
  __shared__ int flag;
  __shared__ int abort_flag;
  __shared__ __align__(16) float vec_lse[kBlk], vec_d[kBlk], vec_c[kBlk];

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sK = base + kOffK, sV = base + kOffV, sQ = base + kOffQ, sDO = base + kOffDO, sDS = base + kOffDS,
                 sST = base + kOffST;

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  // CTA order (CTAs start in index order): sequence, KV head, then key block,
  // small key blocks (most work) first.  Concurrent CTAs thus cover many key
  // blocks of few heads: they read the same Q and dO tiles and add into the
  // same dQ tiles at nearly the same time, in L2 rather than DRAM (6.3 GB of
  // DRAM traffic at 128K x 8 heads, 1.5 ms faster than with heads fastest).
  const int ntc = ((a.cu ? a.Lmax : a.Lk) + kBlk - 1) / kBlk;
  const int bh = static_cast<int>(blockIdx.x) / ntc;
  const int hk = bh % a.Hkv, b = bh / a.Hkv;
  const int kb = static_cast<int>(blockIdx.x) % ntc;
  // this CTA's sequence: its lengths, first row and batch coordinate in the layout
  const SeqSpan sq = seq_span(a, b);
  const int Lq = sq.Lq, Lk = sq.Lk, row0 = sq.row0, bc = sq.bc;
  const int G = a.Hq / a.Hkv;
  const int Tr = (Lq + kBlk - 1) / kBlk, Tc = (Lk + kBlk - 1) / kBlk;
  if (kb >= Tc) return;                  // past the sequence's key blocks (packed batches)
  // tile rows / columns of mask and counts (a packed batch pads each sequence to Lmax)
  const int mTr = a.cu ? (a.Lmax + kBlk - 1) / kBlk : Tr, mTc = a.cu ? mTr : Tc;
  const int lb = a.cu ? 1 : a.B;         // batch extent of the layout (a packed batch is one run of rows)
  const int ibot = a.causal ? kb : 0;
  const int ni = Tr - ibot;
  const int ntiles = G * ni;

  if (warp == 0) tmem_alloc<512>(smem_u32(&tmem_sh));
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bars.kv_full), 1);
    for (int i = 0; i < 2; ++i) { mbar_init(smem_u32(&bars.q_full[i]), 1); mbar_init(smem_u32(&bars.q_empty[i]), 1); }
    mbar_init(smem_u32(&bars.do_full), 1);
    mbar_init(smem_u32(&bars.s_full), 1);
    mbar_init(smem_u32(&bars.dec), 1);
    mbar_init(smem_u32(&bars.p_ready), kMath / 32);   // one arrival per math warp
    mbar_init(smem_u32(&bars.dp_full), 1);
    mbar_init(smem_u32(&bars.ds_ready), 1);
    mbar_init(smem_u32(&bars.dq_full), 1);
    mbar_init(smem_u32(&bars.dq_free), 1);
    mbar_init(smem_u32(&bars.fin), 1);
    fence_barrier_init();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_sh;
  volatile int* abortp = &abort_flag;

  if (warp == 8) {
    // ---------------- TMA producer: K, V once; Q ring of 2 ----------------
    if (lane == 0) {
      prefetch_tensormap(&mq);
      prefetch_tensormap(&mk);
      prefetch_tensormap(&mv);
      prefetch_tensormap(&mdo);
      const uint32_t kvf = smem_u32(&bars.kv_full);
      mbar_expect_tx(kvf, 2 * kTile);
      if (dbg_box(64, hk, row0 + kb * kBlk, bc, kD, a.Hkv, row0, row0 + Lk, a.Lk, lb, a.status)) {
        tma_load_4d(sK, &mk, kvf, 0, hk, row0 + kb * kBlk, bc);
        tma_load_4d(sK + kHalf, &mk, kvf, 64, hk, row0 + kb * kBlk, bc);
        tma_load_4d(sV, &mv, kvf, 0, hk, row0 + kb * kBlk, bc);
        tma_load_4d(sV + kHalf, &mv, kvf, 64, hk, row0 + kb * kBlk, bc);
      }
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int s = t & 1, n = t >> 1;
        if (n > 0 && !mbar_wait(smem_u32(&bars.q_empty[s]), (n - 1) & 1, abortp, a.status)) break;
        const int h = hk * G + t / ni, i = ibot + t % ni;
        const uint32_t qf = smem_u32(&bars.q_full[s]);
        mbar_expect_tx(qf, kTile);
        if (dbg_box(64, h, row0 + i * kBlk, bc, kD, a.Hq, row0, row0 + Lq, a.Lq, lb, a.status)) {
          tma_load_4d(sQ + s * kTile, &mq, qf, 0, h, row0 + i * kBlk, bc);
          tma_load_4d(sQ + s * kTile + kHalf, &mq, qf, 64, h, row0 + i * kBlk, bc);
        }
        ++issued;
      }
      // every issued load lands before the CTA can finish, abort or not
      mbar_drain(kvf, 0, a.status);
      for (int t = max(0, issued - 2); t < issued; ++t)
        mbar_drain(smem_u32(&bars.q_full[t & 1]), (t >> 1) & 1, a.status);
    }
  } else if (warp == 9) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t id_kk = idesc_f16(0, 0, 0, kBlk, kBlk);    // A, B K-major (fp16)
      constexpr uint32_t id_kmn = idesc_f16(0, 0, 1, kBlk, kD);     // A K-major (or TMEM), B MN-major
      constexpr uint32_t id_mnmn = idesc_f16(0, 1, 1, kBlk, kD);    // A, B MN-major
      bool ok = mbar_wait(smem_u32(&bars.kv_full), 0, abortp, a.status);
      auto issue_qk = [&](int t) -> bool {
        const int s = t & 1;
        if (!mbar_wait(smem_u32(&bars.q_full[s]), (t >> 1) & 1, abortp, a.status)) return false;
        fence_after_sync();
        const uint32_t qb = sQ + s * kTile;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = (k / 4) * kHalf + (k % 4) * 32;
          mma_ss(tmem + region(t), desc_kmajor_sw128(sK + off), desc_kmajor_sw128(qb + off), id_kk, k > 0);
        }
        mma_commit(smem_u32(&bars.s_full));
        return true;
      };
      if (ok) ok = issue_qk(0);
      int nret = 0;
      int pend = -1, pend_region = 0;       // retained tile whose dQ^T awaits read-out, and its region
      for (int t = 0; ok && t < ntiles; ++t) {
        // the tile's decision comes at the vote; a kept tile's dO (requested
        // then) is waited for while P is formed, and P, the last to be ready, last
        if (!mbar_wait(smem_u32(&bars.dec), t & 1, abortp, a.status)) break;
        const int ret = flag;
        const uint32_t qb = sQ + (t & 1) * kTile;
        const uint32_t rg = tmem + region(t);
        // a skipped tile's Q slot is free at once: its scores are complete (the
        // vote came after them), and the producer can start the next load now
        if (!ret) mbar_arrive(smem_u32(&bars.q_empty[t & 1]));
        if (ret) {
          if (!mbar_wait(smem_u32(&bars.do_full), nret & 1, abortp, a.status) ||
              !mbar_wait(smem_u32(&bars.p_ready), nret & 1, abortp, a.status))
            break;
          fence_after_sync();
          // dV += P^T dO   (A = P^T from TMEM: queries 0-63 packed in the region's
          // columns 0-31, queries 64-127 in columns 64-95, each written by its math group)
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ts(tmem + kColDV, rg + (k / 4) * 64 + (k % 4) * 8,
                   desc_mnmajor_sw128(sDO + k * 2048, kHalf, 1024), id_kmn, (nret > 0 || k > 0) ? 1u : 0u);
          // dP^T = V dO^T over P^T (read by dV above: MMAs execute in issue order)
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t off = (k / 4) * kHalf + (k % 4) * 32;
            mma_ss(rg, desc_kmajor_sw128(sV + off), desc_kmajor_sw128(sDO + off), id_kk, k > 0);
          }
          mma_commit(smem_u32(&bars.dp_full));
        }
        // the next scores into the other region, once the dQ^T left there has been read out
        if (t + 1 < ntiles) {
          if (pend >= 0 && pend_region == ((t + 1) & 1)) {
            if (!mbar_wait(smem_u32(&bars.dq_free), pend & 1, abortp, a.status)) break;
            pend = -1;
          }
          if (!issue_qk(t + 1)) break;
        }
        if (!ret) continue;
        if (!mbar_wait(smem_u32(&bars.ds_ready), nret & 1, abortp, a.status)) break;
        fence_after_sync();
        // dK += dS^T Q   (A = dS^T: K-major view of the dS tile)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ss(tmem + kColDK, desc_kmajor_sw128(sDS + (k / 4) * kHalf + (k % 4) * 32),
                 desc_mnmajor_sw128(qb + k * 2048, kHalf, 1024), id_kmn, (nret > 0 || k > 0) ? 1u : 0u);
        mma_commit(smem_u32(&bars.q_empty[t & 1]));
        // dQ^T = K^T dS^T  (A = K tile read MN-major, B = the same dS tile read
        // MN-major) over dP^T, which the math warps have read: TMEM lane = head
        // dim, column = query, so the read-out adds whole 128-byte rows of dQ
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ss(rg, desc_mnmajor_sw128(sK + k * 2048, kHalf, 1024),
                 desc_mnmajor_sw128(sDS + k * 2048, kHalf, 1024), id_mnmn, k > 0);
        mma_commit(smem_u32(&bars.dq_full));
        pend = nret;
        pend_region = t & 1;
        ++nret;
      }
      mma_commit(smem_u32(&bars.fin));
      mbar_drain(smem_u32(&bars.fin), 0, a.status);
    }
  } else {
    // ---------------- math warpgroups ----------------
    const int r = tid & 127;                    // key row = TMEM lane
    const int cg = tid >> 7;                    // column group: queries / head dims [64cg, 64cg + 64)
    const int key = kb * kBlk + r;
    const bool key_ok = key < Lk;
    const bool keys_full = kb * kBlk + kBlk <= Lk;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const bool test = a.tau > 0.f;
    const float sl2 = a.scale_log2;
    const float inv_sl2 = 1.f / sl2;
    int nret = 0, do_issued = 0, head_kept = 0;
    bool ok = true;
    // query block, head and TMEM region of the last retained tile (for its dQ
    // read-out, one iteration later), and how many dQ tiles have been read out
    int prev_q0 = 0, prev_h = 0;
    uint32_t prev_rg = 0;
    int flushed = 0;

    // per-query vectors of tile t (fetched by group 0 one tile ahead): lse and
    // D as loaded, and the decision threshold log2(tau / L_q).  The arithmetic
    // on the loaded values waits until the vectors are written, a tile later,
    // so the loads' latency is not paid where they are issued.
    float n_lse = 0.f, n_d = 0.f, n_thr = INFINITY;
    auto fetch = [&](int h, int i) {
      const int q = i * kBlk + r;
      if (q < Lq) {
        const size_t off = (static_cast<size_t>(bc) * a.Hq + h) * a.Lq + row0 + q;
        const bool in = dbg_idx(off, static_cast<size_t>(lb) * a.Hq * a.Lq, a.status);
        n_lse = in ? a.lse[off] : 0.f;
        n_d = in ? a.delta[off] : 0.f;
        n_thr = test ? a.log2_tau - lg2(a.causal ? static_cast<float>(q + 1) : static_cast<float>(Lk))
                     : -INFINITY;
      } else {
        n_lse = 0.f; n_d = 0.f; n_thr = INFINITY;     // out of range: never kept
      }
    };
    if (ntiles > 0 && cg == 0) fetch(hk * G, ibot);

    // Move the finished dQ^T tile (lane = head dim r, columns = queries) out of
    // TMEM, release its region, and add it into the fp32 accumulator with
    // two bulk reduce-adds of 64 query rows: group 0 stages its rows in the dS
    // buffer (free: dK and dQ have consumed it), group 1 in the staging buffer.
    // Thread 0 owns the bulk groups.  Returns false on abort.
    auto flush_dq = [&](int which, bool release) -> bool {
      ok = ok && mbar_wait(smem_u32(&bars.dq_full), which & 1, abortp, a.status);
      // the staging buffer of group 1 was last read by the previous flush's second reduce-add
      if (tid == 0) bulk_wait_read0();
      named_sync(1, kMath);
      fence_after_sync();
      float* stage = reinterpret_cast<float*>(smem_raw + ((cg == 0 ? sDS : sST) - smem_u32(smem_raw)));
      if (__all_sync(0xffffffffu, ok)) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t v[32];
          tmem_ld32_sync(lane_addr + prev_rg + 64 * cg + c * 32, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) stage[(c * 32 + e) * kD + r] = __uint_as_float(v[e]);
        }
      }
      fence_before_sync();
      fence_proxy_async_smem();
      if (named_vote_or(1, kMath, !ok || *abortp)) return false;
      if (tid == 0) {
        if (release) mbar_arrive(smem_u32(&bars.dq_free));
        // two bulk groups: the first (staged in the dS buffer) is waited for alone before dS is written
        // rows past the sequence add exact zeros (their dS columns are 0)
        if (prev_q0 < Lq &&
            dbg_box(64, prev_h, row0 + prev_q0, bc, kD, a.Hq, row0, row0 + Lq, a.Lq, lb, a.status))
          tma_reduce_add_4d(&mdq, sDS, 0, prev_h, row0 + prev_q0, bc);
        bulk_commit();
        if (prev_q0 + 64 < Lq &&
            dbg_box(64, prev_h, row0 + prev_q0 + 64, bc, kD, a.Hq, row0, row0 + Lq, a.Lq, lb, a.status))
          tma_reduce_add_4d(&mdq, sST, 0, prev_h, row0 + prev_q0 + 64, bc);
        bulk_commit();
      }
      return true;
    };

    // tile t = (head h, query block i), heads in turn, query blocks ascending;
    // carried along rather than divided out of t, which the next vote waits for
    int h = hk * G, i = ibot;
    for (int t = 0; t < ntiles; ++t, i = (i + 1 < Tr) ? i + 1 : ibot, h += (i == ibot) ? 1 : 0) {
      const int q0 = i * kBlk;
      if (cg == 0) {
        // lse in log2 units; scale * D (dS = P (scale dP - scale D)); the
        // threshold on the raw dot product (keep iff raw S >= c)
        const float l2 = n_lse * kLog2e;
        vec_lse[r] = -l2;                     // negated: P = exp2(S * scale_log2 + vec_lse)
        vec_d[r] = -n_d * a.scale;            // negated: dS = P (scale dP + vec_d)
        vec_c[r] = n_thr == INFINITY ? INFINITY : (l2 + n_thr) * inv_sl2;
      }
      named_sync(1, kMath);
      if (cg == 0 && t + 1 < ntiles) {
        const int i1 = (i + 1 < Tr) ? i + 1 : ibot;
        fetch(i1 == ibot ? h + 1 : h, i1);
      }

      ok = mbar_wait(smem_u32(&bars.s_full), t & 1, abortp, a.status);
      fence_after_sync();
      // Eq. (4): keep iff some valid entry has S - lse >= log(tau / L_q)
      const bool diag = a.causal && q0 == kb * kBlk;
      const int qlim = Lq - q0;                   // query columns at or beyond this are out of range
      const int qmin = diag ? r : 0;              // causal: query >= key inside the diagonal tile
      const bool interior = !diag && qlim >= kBlk && keys_full;
      const float4* c4 = reinterpret_cast<const float4*>(&vec_c[64 * cg]);
      int keep_row = 0;
      if (__all_sync(0xffffffffu, ok)) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t sr[32];
          tmem_ld32_sync(lane_addr + region(t) + 64 * cg + c * 32, sr);
          float gap = -INFINITY;
          if (interior) {
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const float4 cc = c4[(c * 32 + e) / 4];
              gap = fmaxf(gap, fmaxf(fmaxf(__uint_as_float(sr[e]) - cc.x, __uint_as_float(sr[e + 1]) - cc.y),
                                     fmaxf(__uint_as_float(sr[e + 2]) - cc.z, __uint_as_float(sr[e + 3]) - cc.w)));
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int q = 64 * cg + c * 32 + e;
              if (key_ok && q < qlim && q >= qmin) gap = fmaxf(gap, __uint_as_float(sr[e]) - vec_c[q]);
            }
          }
          keep_row |= gap >= 0.f ? 1 : 0;
        }
      }
      fence_before_sync();
      // an abort is caught at the vote after P^T is stored, or (skipped tiles)
      // by the next tile's waits, which return at once once the flag is up
      const int keep = named_vote_or(1, kMath, keep_row && ok);
      // the decision goes to the MMA warp first: a skipped tile's successor waits on it
      if (tid == 0) {
        flag = keep;
        mbar_arrive(smem_u32(&bars.dec));
      }
      const size_t mrow_i = ((static_cast<size_t>(b) * a.Hq + h) * mTr + i) * mTc + kb;
      uint8_t* mrow = a.mask && dbg_idx(mrow_i, static_cast<size_t>(a.B) * a.Hq * mTr * mTc, a.status)
                          ? a.mask + mrow_i : nullptr;
      if (tid == 0) {
        head_kept += keep;
        if (i == Tr - 1) {                        // last query block of this head
          if (a.counts != nullptr &&
              dbg_idx((static_cast<size_t>(b) * a.Hq + h) * mTc + kb, static_cast<size_t>(a.B) * a.Hq * mTc, a.status))
            a.counts[(static_cast<size_t>(b) * a.Hq + h) * mTc + kb] = head_kept;
          head_kept = 0;
        }
      }
      if (!keep) {
        if (tid == 0 && mrow) *mrow = 0;
        // the previous retained tile's dQ is read out here too: the MMA warp
        // waits for it before the scores of tile t + 1 go into its region
        if (nret > flushed) {
          if (!flush_dq(nret - 1, true)) break;
          flushed = nret;
        }
        continue;
      }
      if (tid == 0) {
        if (mrow) *mrow = 1;
        // dO of this tile, loaded only now that the tile is retained.  The
        // buffer is free: the previous kept tile's dV and dP^T read it, and
        // every math thread has already seen that dP^T complete (dV runs first).
        if (ok) {
          const uint32_t df = smem_u32(&bars.do_full);
          mbar_expect_tx(df, kTile);
          if (dbg_box(64, h, row0 + q0, bc, kD, a.Hq, row0, row0 + Lq, a.Lq, lb, a.status)) {
            tma_load_4d(sDO, &mdo, df, 0, h, row0 + q0, bc);
            tma_load_4d(sDO + kHalf, &mdo, df, 64, h, row0 + q0, bc);
          }
          ++do_issued;
        }
      }
      // P^T = exp2(S * scale_log2 - lse) in fp16, written over this group's S columns
      const float4* l4 = reinterpret_cast<const float4*>(&vec_lse[64 * cg]);
      const uint64_t sl2x2 = f2(sl2, sl2);
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t sr[32];
        tmem_ld32_sync(lane_addr + region(t) + 64 * cg + c * 32, sr);
        if (interior) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 ll = l4[(c * 32 + e) / 4];
            float x0, x1, x2, x3;
            f2_split(fma2(f2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), sl2x2, f2(ll.x, ll.y)), x0, x1);
            f2_split(fma2(f2(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])), sl2x2, f2(ll.z, ll.w)), x2, x3);
            pk[c * 16 + e / 2] = pack_f16(ex2(x0), ex2(x1));
            pk[c * 16 + e / 2 + 1] = pack_f16(ex2(x2), ex2(x3));
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int q = 64 * cg + c * 32 + e;
            const bool l0 = key_ok && q < qlim && q >= qmin;
            const bool l1 = key_ok && q + 1 < qlim && q + 1 >= qmin;
            const float p0 = l0 ? ex2(fmaf(__uint_as_float(sr[e]), sl2, vec_lse[q])) : 0.f;
            const float p1 = l1 ? ex2(fmaf(__uint_as_float(sr[e + 1]), sl2, vec_lse[q + 1])) : 0.f;
            pk[c * 16 + e / 2] = pack_f16(p0, p1);
          }
        }
      }
      tmem_st32(lane_addr + region(t) + 64 * cg, pk);   // inside this group's own S columns
      tmem_st_wait();
      fence_before_sync();
      // each warp hands its P^T over as soon as its own stores have landed; an
      // abort is caught at the dS vote, and the waits before it return at once
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars.p_ready));
      // the previous retained tile's dQ is read out while dV and dP^T run; the
      // MMA warp waits for it only before the next scores go into its region
      if (nret > flushed) {
        if (!flush_dq(nret - 1, true)) break;
        flushed = nret;
      }
      ok = mbar_wait(smem_u32(&bars.dp_full), nret & 1, abortp, a.status);
      fence_after_sync();
      // dS^T = scale * P^T o (dP^T - D), fp16, computed into registers first so
      // that the bulk reduce-adds have time to finish reading the dS buffer
      uint32_t w[32];
      if (__all_sync(0xffffffffu, ok)) {
        const float4* d4 = reinterpret_cast<const float4*>(&vec_d[64 * cg]);
        const uint64_t sc2 = f2(a.scale, a.scale);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t dp[32];
          tmem_ld32_sync(lane_addr + region(t) + 64 * cg + c * 32, dp);
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            const float4 dd = d4[(c * 32 + 2 * e) / 4];
            const uint32_t pw0 = pk[c * 16 + e], pw1 = pk[c * 16 + e + 1];
            const uint64_t t0 = fma2(f2(__uint_as_float(dp[2 * e]), __uint_as_float(dp[2 * e + 1])), sc2,
                                     f2(dd.x, dd.y));
            const uint64_t t1 = fma2(f2(__uint_as_float(dp[2 * e + 2]), __uint_as_float(dp[2 * e + 3])), sc2,
                                     f2(dd.z, dd.w));
            w[c * 16 + e] = pack_f16_2(mul2(f2(f16_lo(pw0), f16_hi(pw0)), t0));
            w[c * 16 + e + 1] = pack_f16_2(mul2(f2(f16_lo(pw1), f16_hi(pw1)), t1));
          }
        }
      }
      // the dS buffer is free again once the first bulk reduce-add has read it
      if (nret > 0) {
        if (tid == 0) bulk_wait_read1();
        named_sync(1, kMath);
      }
      // into half cg of the swizzled dS tile (row = key r): 8 chunks of 8 queries
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t addr = sDS + cg * kHalf + r * 128 + ((u ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                     :: "r"(addr), "r"(w[4 * u]), "r"(w[4 * u + 1]), "r"(w[4 * u + 2]), "r"(w[4 * u + 3])
                     : "memory");
      }
      fence_proxy_async_smem();
      fence_before_sync();
      if (named_vote_or(1, kMath, !ok || *abortp)) break;
      if (tid == 0) mbar_arrive(smem_u32(&bars.ds_ready));
      prev_q0 = q0;
      prev_h = h;
      prev_rg = region(t);
      ++nret;
    }

    // last dQ tile, then dK, dV out of TMEM (loads are warp-collective; stores per key)
    if (nret > flushed && !*abortp) flush_dq(nret - 1, false);
    if (tid == 0) bulk_wait0();        // every reduce-add has landed before the CTA exits
    fence_after_sync();
    if (__all_sync(0xffffffffu, ok && !*abortp)) {
      write_dkdv<Tg>(smem_raw, sK, warp, lane, cg, nret, kb, Lk, row0, bc, hk, lb, a.Lk, a.Hkv, a.dv, a.dk, lane_addr,
                     a.status);
    }
    // a dO load issued for an abandoned tile must land before the CTA exits
    if (tid == 0 && *abortp && do_issued > 0)
      mbar_drain(smem_u32(&bars.do_full), (do_issued - 1) & 1, a.status);
    fence_before_sync();
  }

  __syncthreads();
  if (warp == 0) {
    fence_after_sync();
    tmem_dealloc<512>(tmem);
  }
}

// True if one of the four bf16 values of v is finite and beyond fp16's range
// (|x| > 65504), where the fp16 copy would become +-inf.
__device__ __forceinline__ bool beyond_fp16(uint2 v) {
  const float m = fmaxf(fmaxf(fabsf(bf16_lo(v.x)), fabsf(bf16_hi(v.x))), fmaxf(fabsf(bf16_lo(v.y)), fabsf(bf16_hi(v.y))));
  return m > 65504.f && m <= 3.4e38f;
}

// Exact fp16 copies of q, k, v, dO (bf16 in; exact for |x| in the fp16
// normal range), D = rowsum(O * dO), and a zeroed fp32 dQ accumulator.  One
// warp per row; each lane converts 4 of the 128 elements.  A finite input
// beyond fp16's range sets kStatusFp16Range (its copy would be +-inf).
__global__ void bwd_tc_prep_kernel(const BwdArgs a, uint32_t* q16, uint32_t* k16, uint32_t* v16, uint32_t* do16) {
  const size_t lb = a.cu ? 1 : a.B;       // a packed batch is one run of Lq rows
  const size_t qrows = lb * a.Lq * a.Hq;
  const size_t krows = lb * a.Lk * a.Hkv;
  const size_t row = (static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  if (row < qrows) {
    const uint2 qv = reinterpret_cast<const uint2*>(a.q)[row * 32 + lane];
    const uint2 dv = reinterpret_cast<const uint2*>(a.dout)[row * 32 + lane];
    const uint2 ov = reinterpret_cast<const uint2*>(a.o)[row * 32 + lane];
    reinterpret_cast<uint2*>(q16)[row * 32 + lane] =
        make_uint2(pack_f16(bf16_lo(qv.x), bf16_hi(qv.x)), pack_f16(bf16_lo(qv.y), bf16_hi(qv.y)));
    reinterpret_cast<uint2*>(do16)[row * 32 + lane] =
        make_uint2(pack_f16(bf16_lo(dv.x), bf16_hi(dv.x)), pack_f16(bf16_lo(dv.y), bf16_hi(dv.y)));
    if (__any_sync(0xffffffffu, beyond_fp16(qv) || beyond_fp16(dv)) && lane == 0)
      atomicOr(a.status, kStatusFp16Range);
    float s = bf16_lo(ov.x) * bf16_lo(dv.x) + bf16_hi(ov.x) * bf16_hi(dv.x) +
              bf16_lo(ov.y) * bf16_lo(dv.y) + bf16_hi(ov.y) * bf16_hi(dv.y);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    reinterpret_cast<float4*>(a.dq_acc + row * kD)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lane == 0) {
      const int h = static_cast<int>(row % a.Hq);
      const size_t bq = row / a.Hq;
      const int q = static_cast<int>(bq % a.Lq);
      const size_t bb = bq / a.Lq;
      a.delta[(bb * a.Hq + h) * a.Lq + q] = s;
    }
  }
  if (row < krows) {
    const uint2 kv = reinterpret_cast<const uint2*>(a.k)[row * 32 + lane];
    const uint2 vv = reinterpret_cast<const uint2*>(a.v)[row * 32 + lane];
    reinterpret_cast<uint2*>(k16)[row * 32 + lane] =
        make_uint2(pack_f16(bf16_lo(kv.x), bf16_hi(kv.x)), pack_f16(bf16_lo(kv.y), bf16_hi(kv.y)));
    reinterpret_cast<uint2*>(v16)[row * 32 + lane] =
        make_uint2(pack_f16(bf16_lo(vv.x), bf16_hi(vv.x)), pack_f16(bf16_lo(vv.y), bf16_hi(vv.y)));
    if (__any_sync(0xffffffffu, beyond_fp16(kv) || beyond_fp16(vv)) && lane == 0)
      atomicOr(a.status, kStatusFp16Range);
  }
}

}  // namespace

bool bwd_tc_supported(const BwdArgs& a) {
  return a.in_dt == kBF16 && a.D == kD && a.blk == kBlk;
}

size_t bwd_tc_scratch_bytes(int B, int Lq, int Lk, int Hq, int Hkv, int D) {
  return 2 * (static_cast<size_t>(B) * Lq * Hq * D + static_cast<size_t>(B) * Lk * Hkv * D) * sizeof(__half);
}

cudaError_t launch_bwd_tc(const BwdArgs& a, cudaStream_t s, int* launches) {
  // fp16 copies: q, dO [B, Lq, Hq, D] then k, v [B, Lk, Hkv, D] (two halves per 32-bit word)
  const int lb = a.cu ? 1 : a.B;           // a packed batch is one run of Lq rows
  uint32_t* q16 = static_cast<uint32_t*>(a.scratch);
  uint32_t* do16 = q16 + static_cast<size_t>(lb) * a.Lq * a.Hq * kD / 2;
  uint32_t* k16 = do16 + static_cast<size_t>(lb) * a.Lq * a.Hq * kD / 2;
  uint32_t* v16 = k16 + static_cast<size_t>(lb) * a.Lk * a.Hkv * kD / 2;
  const size_t rows = std::max(static_cast<size_t>(lb) * a.Lq * a.Hq, static_cast<size_t>(lb) * a.Lk * a.Hkv);
  bwd_tc_prep_kernel<<<static_cast<unsigned>((rows * 32 + 255) / 256), 256, 0, s>>>(a, q16, k16, v16, do16);
  ++*launches;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap mq, mk, mv, mdo;
  if (!encode_bshd_map(&mq, q16, lb, a.Lq, a.Hq, kD, kBlk, true) ||
      !encode_bshd_map(&mdo, do16, lb, a.Lq, a.Hq, kD, kBlk, true) ||
      !encode_bshd_map(&mk, k16, lb, a.Lk, a.Hkv, kD, kBlk, true) ||
      !encode_bshd_map(&mv, v16, lb, a.Lk, a.Hkv, kD, kBlk, true))
    return cudaErrorInvalidValue;
  CUtensorMap mdq;
  if (!encode_bshd_f32_map(&mdq, a.dq_acc, lb, a.Lq, a.Hq, kD, 64)) return cudaErrorInvalidValue;
  const int tc = ((a.cu ? a.Lmax : a.Lk) + kBlk - 1) / kBlk;
  const dim3 grid(static_cast<unsigned>(a.Hkv) * a.B * tc);
  ++*launches;
  if (a.grad_dt == kBF16) {
    auto kern = bwd_tc_kernel<__nv_bfloat16>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, kSmem, s>>>(mq, mk, mv, mdo, mdq, a);
  } else {
    auto kern = bwd_tc_kernel<float>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, kSmem, s>>>(mq, mk, mv, mdo, mdq, a);
  }
  return cudaGetLastError();
}

}  // namespace mala
