// MALA forward on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// "MassAlloc Attention: Let Attention Allocate Its Own Compute", Algorithm 1
// and §2.2 Eq. (3): for each 128-row query block, the legal 128-key blocks
// are visited from the diagonal toward earlier keys.  Every tile's scores
// S = Q K^T are formed; the tile is skipped iff, for every valid row,
// rowmax(S) - m - log l < log(tau / L_q) (l = 0 keeps).  A skipped tile issues
// no V load and no P V product and leaves (m, l, O) unchanged (App. A.1).
//
// One CTA = one query block of one head, 320 threads:
//   warps 0-7  softmax, two warpgroups: thread (c, r) owns columns [64c, 64c+64)
//              of query row r = TMEM lane r.  The groups combine the row max
//              and row sums through shared memory (each keeps a copy of the
//              row state), vote on the tile, and for retained tiles thread 0
//              issues the V load; P = exp2(S - m) goes as bf16 into TMEM
//              inside each group's own S columns.
//   warp 8     TMA producer for Q and K (2-stage K ring).
//   warp 9     MMA issuer: S = Q K^T (SS, K-major operands) and
//              O += P V (A = P from TMEM, B = V MN-major), accumulate in TMEM.
// TMEM: three S buffers (columns 0, 128, 256) and O (columns 384..511), so
// scores run two tiles ahead of the softmax while a retained tile waits for
// its V.  The running max is only moved when it grows by more than 2^8
// (log2 units); P and l are kept relative to the max in use, which leaves
// m + log l = log Z unchanged, so the test is unaffected.
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
constexpr int kNK = 2;                  // K stages
constexpr int kNV = 3;                  // V stages
constexpr int kNS = 3;                  // S buffers in TMEM
constexpr int kThreads = 320;
constexpr int kSoft = 256;              // two softmax warpgroups
constexpr int kSmem = kTile * (1 + kNK + kNV) + 1024;
constexpr uint32_t kColO = 384;
constexpr float kRescale = 8.0f;        // move the running max only past 2^8 growth

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kNK], k_empty[kNK];
  uint64_t v_full[kNV], v_empty[kNV];
  uint64_t s_full[kNS], sm_done[kNS];
  uint64_t pv_done[2];
  uint64_t fin;
};


template <typename Tout>
__device__ __forceinline__ void store_row(Tout* dst, const float* v, float scale);

template <>
__device__ __forceinline__ void store_row<__nv_bfloat16>(__nv_bfloat16* dst, const float* v, float scale) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 w;
    w.x = pack_bf16(v[8 * i + 0] * scale, v[8 * i + 1] * scale);
    w.y = pack_bf16(v[8 * i + 2] * scale, v[8 * i + 3] * scale);
    w.z = pack_bf16(v[8 * i + 4] * scale, v[8 * i + 5] * scale);
    w.w = pack_bf16(v[8 * i + 6] * scale, v[8 * i + 7] * scale);
    d4[i] = w;
  }
}

template <>
__device__ __forceinline__ void store_row<float>(float* dst, const float* v, float scale) {
  float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    d4[i] = make_float4(v[4 * i] * scale, v[4 * i + 1] * scale, v[4 * i + 2] * scale, v[4 * i + 3] * scale);
}

template <typename Tout>
__global__ void __launch_bounds__(kThreads, 1)
fwd_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
              const __grid_constant__ CUtensorMap mv, const FwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) Bars bars;
  __shared__ uint32_t tmem_sh;
  __shared__ int flag[kNS];
  __shared__ int abort_flag;
  __shared__ float xmax[2][kBlk], xsum[2][kBlk], xsumr[2][kBlk];   // per-group row partials

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = base;
  const uint32_t sK = base + kTile;
  const uint32_t sV = base + kTile * (1 + kNK);

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int bh = blockIdx.x;
  const int h = bh % a.Hq, b = bh / a.Hq;
  const int Tr = (a.Lq + kBlk - 1) / kBlk, Tc = (a.Lk + kBlk - 1) / kBlk;
  const int qb = Tr - 1 - static_cast<int>(blockIdx.y);          // heaviest query blocks first
  const int hk = h / (a.Hq / a.Hkv);
  const int jtop = a.causal ? min(Tc - 1, (min(a.Lq, qb * kBlk + kBlk) - 1) / kBlk) : Tc - 1;
  const int ntiles = jtop + 1;

  if (warp == 0) tmem_alloc<512>(smem_u32(&tmem_sh));
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bars.q_full), 1);
    for (int i = 0; i < kNK; ++i) { mbar_init(smem_u32(&bars.k_full[i]), 1); mbar_init(smem_u32(&bars.k_empty[i]), 1); }
    for (int i = 0; i < kNV; ++i) { mbar_init(smem_u32(&bars.v_full[i]), 1); mbar_init(smem_u32(&bars.v_empty[i]), 1); }
    for (int i = 0; i < kNS; ++i) {
      mbar_init(smem_u32(&bars.s_full[i]), 1);
      mbar_init(smem_u32(&bars.sm_done[i]), kSoft / 32);     // one arrival per softmax warp
    }
    mbar_init(smem_u32(&bars.pv_done[0]), 1);
    mbar_init(smem_u32(&bars.pv_done[1]), 1);
    mbar_init(smem_u32(&bars.fin), 1);
    fence_barrier_init();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_sh;
  volatile int* abortp = &abort_flag;

  if (warp == 8) {
    // ---------------- TMA producer: Q once, then the K ring ----------------
    if (lane == 0) {
      prefetch_tensormap(&mq);
      prefetch_tensormap(&mk);
      prefetch_tensormap(&mv);
      const uint32_t qf = smem_u32(&bars.q_full);
      mbar_expect_tx(qf, kTile);
      tma_load_4d(sQ, &mq, qf, 0, h, qb * kBlk, b);
      tma_load_4d(sQ + kHalf, &mq, qf, 64, h, qb * kBlk, b);
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % kNK, n = t / kNK;
        if (n > 0 && !mbar_wait(smem_u32(&bars.k_empty[s]), (n - 1) & 1, abortp, a.status)) break;
        const uint32_t kf = smem_u32(&bars.k_full[s]);
        const int row = (jtop - t) * kBlk;
        mbar_expect_tx(kf, kTile);
        tma_load_4d(sK + s * kTile, &mk, kf, 0, hk, row, b);
        tma_load_4d(sK + s * kTile + kHalf, &mk, kf, 64, hk, row, b);
        ++issued;
      }
      // drain: every issued load has landed before the CTA can finish
      for (int t = max(0, issued - kNK); t < issued; ++t)
        mbar_wait(smem_u32(&bars.k_full[t % kNK]), (t / kNK) & 1, abortp, a.status);
    }
  } else if (warp == 9) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_f16(1, 0, 0, kBlk, kBlk);
      constexpr uint32_t idesc_pv = idesc_f16(1, 0, 1, kBlk, kD);
      bool ok = mbar_wait(smem_u32(&bars.q_full), 0, abortp, a.status);
      auto issue_qk = [&](int t) -> bool {
        const int s = t % kNK, n = t / kNK;
        if (!mbar_wait(smem_u32(&bars.k_full[s]), n & 1, abortp, a.status)) return false;
        fence_after_sync();
        const uint32_t d = tmem + (t % kNS) * 128;
        const uint32_t kbase = sK + s * kTile;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = (k / 4) * kHalf + (k % 4) * 32;
          mma_ss(d, desc_kmajor_sw128(sQ + off), desc_kmajor_sw128(kbase + off), idesc_qk, k > 0);
        }
        mma_commit(smem_u32(&bars.k_empty[s]));
        mma_commit(smem_u32(&bars.s_full[t % kNS]));
        return true;
      };
      if (ok) ok = issue_qk(0);
      if (ok && ntiles > 1) ok = issue_qk(1);
      int npv = 0;
      for (int t = 0; ok && t < ntiles; ++t) {
        const int sb = t % kNS;
        if (!mbar_wait(smem_u32(&bars.sm_done[sb]), (t / kNS) & 1, abortp, a.status)) break;
        fence_after_sync();
        if (t + 2 < ntiles && !issue_qk(t + 2)) break;
        if (flag[sb]) {
          const int vs = npv % kNV;
          if (!mbar_wait(smem_u32(&bars.v_full[vs]), (npv / kNV) & 1, abortp, a.status)) break;
          fence_after_sync();
          const uint32_t vbase = sV + vs * kTile;
          // P: keys 0-63 packed in columns 0-31 of the S buffer, keys 64-127 in 64-95
          const uint32_t p_tmem = tmem + sb * 128;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ts(tmem + kColO, p_tmem + (k / 4) * 64 + (k % 4) * 8, desc_mnmajor_sw128(vbase + k * 2048, kHalf, 1024),
                   idesc_pv, (npv > 0 || k > 0) ? 1u : 0u);
          mma_commit(smem_u32(&bars.v_empty[vs]));
          mma_commit(smem_u32(&bars.pv_done[npv & 1]));
          ++npv;
        }
      }
      // all MMAs of this thread complete before TMEM is released
      mma_commit(smem_u32(&bars.fin));
      mbar_wait(smem_u32(&bars.fin), 0, abortp, a.status);
    }
  } else {
    // ---------------- softmax: thread (cg, r) = columns [64cg, 64cg+64) of row r ----------------
    const int r = tid & 127, cg = tid >> 7;
    const int qrow = qb * kBlk + r;
    const bool valid = qrow < a.Lq;
    const int lim = a.causal ? min(qrow, a.Lk - 1) : a.Lk - 1;   // last legal key of this row
    const float thr = a.log2_tau - log2f(a.causal ? static_cast<float>(qrow + 1) : static_cast<float>(a.Lk));
    const bool test = a.tau > 0.f;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    // row state, identical in both groups: l is the exact fp32 sum of P (Eq. 3
    // test and lse); lr sums the bf16-rounded P that enters the P V product
    float m_used = -INFINITY, l = 0.f, lr = 0.f;
    // the other group's row sums of a retained tile are read a tile later,
    // after the next row-max barrier has published them
    float alpha_pend = 1.f;
    bool sum_pend = false;
    int nret = 0, vissued = 0;
    bool ok = true;
    uint8_t* mask_row = a.mask ? a.mask + ((static_cast<size_t>(b) * a.Hq + h) * Tr + qb) * Tc : nullptr;

    for (int t = 0; t < ntiles; ++t) {
      const int j = jtop - t, sb = t % kNS;
      ok = mbar_wait(smem_u32(&bars.s_full[sb]), (t / kNS) & 1, abortp, a.status);
      fence_after_sync();
      uint32_t sr[64];                        // raw scores Q.K of this group's columns, later packed P
      if (__all_sync(0xffffffffu, ok)) tmem_ld64_sync(lane_addr + sb * 128 + 64 * cg, sr);
      // row max over legal keys (raw dot products; the scale is positive).
      // Interior tiles (not diagonal, no ragged edge) need no masking.
      const int cmax = valid ? lim - j * kBlk - 64 * cg : -1;
      const bool interior = (a.causal ? j < qb : (j + 1) * kBlk <= a.Lk) && (qb + 1) * kBlk <= a.Lq;
      float mraw = -INFINITY;
      if (interior) {
#pragma unroll
        for (int c = 0; c < 64; c += 2)
          mraw = fmaxf(mraw, fmaxf(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])));
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float x = (c <= cmax) ? __uint_as_float(sr[c]) : -INFINITY;
          sr[c] = __float_as_uint(x);
          mraw = fmaxf(mraw, x);
        }
      }
      xmax[cg][r] = mraw;
      fence_before_sync();
      if (named_vote_or(1, kSoft, !ok || *abortp)) break;   // also the barrier for xmax, xsum
      if (sum_pend) {
        l = l * alpha_pend + (xsum[0][r] + xsum[1][r]);
        lr = lr * alpha_pend + (xsumr[0][r] + xsumr[1][r]);
        sum_pend = false;
      }
      const float mt = fmaxf(xmax[0][r], xmax[1][r]) * a.scale_log2;
      const bool has = valid && lim >= j * kBlk;
      const int keep_row = has && (!test || l == 0.f || !(mt - m_used - lg2(l) < thr));
      // both groups hold every row's full maximum, so each votes alone (same result)
      const int keep = named_vote_or(2 + cg, 128, keep_row);
      if (!keep) {
        if (tid == 0) {
          flag[sb] = 0;
          if (mask_row) mask_row[j] = 0;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars.sm_done[sb]));
        continue;
      }
      if (tid == 0) {
        // V of this tile: loaded only now that the tile is retained
        const int vs = vissued % kNV, n = vissued / kNV;
        if (n > 0) ok = mbar_wait(smem_u32(&bars.v_empty[vs]), (n - 1) & 1, abortp, a.status);
        if (ok) {
          const uint32_t vf = smem_u32(&bars.v_full[vs]);
          mbar_expect_tx(vf, kTile);
          tma_load_4d(sV + vs * kTile, &mv, vf, 0, hk, j * kBlk, b);
          tma_load_4d(sV + vs * kTile + kHalf, &mv, vf, 64, hk, j * kBlk, b);
          ++vissued;
        }
        if (mask_row) mask_row[j] = 1;
      }
      // online update (Algorithm 1), with a lazily moved reference max
      float alpha = 1.f;
      if (has && mt > m_used + kRescale) {
        alpha = (m_used == -INFINITY) ? 0.f : ex2(m_used - mt);
        m_used = mt;
      }
      const float mref = (m_used == -INFINITY) ? 0.f : m_used;
      const float nscale = a.scale_log2;
      const uint64_t nsc2 = f2(nscale, nscale), nm2 = f2(-mref, -mref);
      uint64_t acc = f2(0.f, 0.f), accr = f2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        float e0, e1;
        f2_split(fma2(f2(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), nsc2, nm2), e0, e1);
        const float p0 = ex2(e0), p1 = ex2(e1);
        const uint32_t w = pack_bf16(p0, p1);
        acc = add2(acc, f2(p0, p1));
        accr = add2(accr, f2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u)));
        sr[c] = w;                            // P packed over the consumed scores
      }
      float rowsum, rowsum_r;
      {
        float x0, x1;
        f2_split(acc, x0, x1);
        rowsum = x0 + x1;
        f2_split(accr, x0, x1);
        rowsum_r = x0 + x1;
      }
      xsum[cg][r] = rowsum;
      xsumr[cg][r] = rowsum_r;
      // O must be rescaled when the reference max moved: wait for the last P V
      if (nret > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        const int prev = nret - 1;
        if (ok) ok = mbar_wait(smem_u32(&bars.pv_done[prev & 1]), (prev >> 1) & 1, abortp, a.status);
        fence_after_sync();
        if (__all_sync(0xffffffffu, ok)) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t o[32];
            tmem_ld32_sync(lane_addr + kColO + 64 * cg + c * 32, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(lane_addr + kColO + 64 * cg + c * 32, o);
          }
        }
      }
      tmem_st32(lane_addr + sb * 128 + 64 * cg, sr);   // inside this group's own S columns
      tmem_st_wait();
      fence_before_sync();
      // each warp hands its P over once its TMEM stores are complete (an abort
      // is caught by the next tile's first vote)
      if (tid == 0) flag[sb] = 1;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars.sm_done[sb]));
      alpha_pend = alpha;
      sum_pend = true;
      ++nret;
    }
    named_sync(1, kSoft);                     // publishes the last tile's row sums
    if (sum_pend) {
      l = l * alpha_pend + (xsum[0][r] + xsum[1][r]);
      lr = lr * alpha_pend + (xsumr[0][r] + xsumr[1][r]);
    }

    // epilogue: wait for the last P V, then O / l and lse = m + log l
    if (ok && !*abortp && nret > 0) {
      const int last = nret - 1;
      ok = mbar_wait(smem_u32(&bars.pv_done[last & 1]), (last >> 1) & 1, abortp, a.status);
    }
    fence_after_sync();
    if (__all_sync(0xffffffffu, ok && !*abortp)) {
      Tout* orow = static_cast<Tout*>(a.o) + ((static_cast<size_t>(b) * a.Lq + (valid ? qrow : 0)) * a.Hq + h) * kD;
      const float inv = 1.f / lr;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float o[32];
        tmem_ld32_sync(lane_addr + kColO + 64 * cg + c * 32, reinterpret_cast<uint32_t*>(o));
        if (valid) store_row<Tout>(orow + 64 * cg + c * 32, o, inv);
      }
      if (valid && cg == 0) a.lse[(static_cast<size_t>(b) * a.Hq + h) * a.Lq + qrow] = (m_used + log2f(l)) * kLn2;
      if (a.counts != nullptr && tid == 0) a.counts[(static_cast<size_t>(b) * a.Hq + h) * Tr + qb] = nret;
    }
    // V loads issued but never consumed (abort path) must land before exit
    if (tid == 0) {
      for (int n = max(0, vissued - kNV); n < vissued; ++n)
        mbar_wait(smem_u32(&bars.v_full[n % kNV]), (n / kNV) & 1, abortp, a.status);
    }
    fence_before_sync();
  }

  __syncthreads();
  if (warp == 0) {
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
  if (!encode_bshd_map(&mq, a.q, a.B, a.Lq, a.Hq, kD, kBlk) ||
      !encode_bshd_map(&mk, a.k, a.B, a.Lk, a.Hkv, kD, kBlk) ||
      !encode_bshd_map(&mv, a.v, a.B, a.Lk, a.Hkv, kD, kBlk))
    return cudaErrorInvalidValue;
  const int tr = (a.Lq + kBlk - 1) / kBlk;
  dim3 grid(a.Hq * a.B, tr);
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
