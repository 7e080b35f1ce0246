// MALA split-KV decode, bandwidth-oriented (bf16, head_dim 128, 128-key tiles).
//
// "MassAlloc Attention: Let Attention Allocate Its Own Compute", App. A.1
// ("Fused decoding execution") and §2.4: one query per sequence against its
// KV cache; every tile is scored, and V is loaded and P V run only for tiles
// the test of Eq. (3) keeps.  Each split starts from its own empty (m, l),
// visits its tiles newest to oldest and tests against L = N (the full
// context).  The G query heads sharing a KV head form the query block: a tile
// is kept if any of them keeps it.  In the per-head variant each query head
// decides for itself: V is loaded if any head keeps the tile, and a head that
// skips it takes P = 0 and keeps its (m, l).  The split writes
// (m, l, l_rounded, u) for the exact merge of "Why exact attention does not
// need a quadratic matrix".
//
// One CTA of 288 threads per (KV head, split, sequence):
//   warp 8     TMA producer: K tiles, 3-stage ring, running ahead.
//   warps 0-3  score warps: S^T = K q^T with mma.sync m16n8k16 (keys as M, the
//              G <= 8 heads as N), one barrier per tile that exchanges each
//              warp's tile maxima and running partial sums, the test (lane g
//              decides head g, a ballot combines the heads), and for kept
//              tiles the V load and P (bf16) into one of three slots.
//   warps 4-7  P V warps: O^T += V^T P^T for each published slot (warp w owns
//              head dims 32(w-4)..32(w-4)+31), off the score warps' path.
// The reference max m is moved lazily (only past 2^8 growth); every P slot
// carries the m it was computed with, and O is rescaled to it before its P V.
#include <cuda_bf16.h>

#include "mala_internal.h"
#include "tc_common.cuh"

namespace mala {
namespace {

using namespace tc;

constexpr int kD = 128;
constexpr int kBK = 128;
constexpr int kTile = kBK * kD * 2;
constexpr int kHalf = kTile / 2;
constexpr int kNK = 3;          // K ring
constexpr int kNV = 3;          // V ring = P slots
constexpr int kThreads = 288;
constexpr int kSmem = kTile * (kNK + kNV) + 1024;
constexpr float kRescale = 8.0f;

struct Bars {
  uint64_t k_full[kNK], k_empty[kNK];
  uint64_t v_full[kNV], p_full[kNV], slot_empty[kNV];
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// smem byte address of 16-byte chunk `chunk` (8 bf16 along d) of row `row` in a
// [128 rows x 128 d] tile stored as two 128-byte-swizzled 64-column halves.
__device__ __forceinline__ uint32_t sw_addr(uint32_t base, int row, int dchunk) {
  return base + (dchunk >> 3) * kHalf + row * 128 + (((dchunk & 7) ^ (row & 7)) << 4);
}

__device__ __forceinline__ float* split_record(const DecArgs& a, int sp, int b, int h) {
  return a.partial + ((static_cast<size_t>(sp) * a.B + b) * a.Hq + h) * (kD + 4);
}

__global__ void __launch_bounds__(kThreads, 1)
decode_mma_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv, const DecArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) Bars bars;
  __shared__ int abort_flag;
  __shared__ int pv_done;                                   // P V products finished (for the exit path)
  // per score warp: tile max and running partial sums (exact, rounded) per head; by tile parity
  // (index 2 of xl: the final sums, written while a slower warp may still read index 0 or 1)
  __shared__ float xmax[2][4][8], xl[3][4][8], xlr[4][8];
  __shared__ __align__(16) uint16_t pslot[kNV][8][kBK];    // P (bf16) of kept tiles, [head][key]
  __shared__ float pslot_m[kNV][8];                         // reference max each P was taken against
  __shared__ int pslot_end[kNV];                            // 1: no more tiles

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sK = base, sV = base + kNK * kTile;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int hk = blockIdx.x, sp = blockIdx.y, b = blockIdx.z;
  const int G = a.Hq / a.Hkv;
  const int n_b = decode_seq_len(a, b);                // this sequence's cache length
  const int T = (n_b + kBK - 1) / kBK;
  const int Tmax = (a.N + kBK - 1) / kBK;              // row length of the tile mask
  const int per = (T + a.splits - 1) / a.splits;
  const int t0 = sp * per, t1 = min(T, t0 + per);
  const int ntiles = max(0, t1 - t0);

  if (tid == 0) {
    abort_flag = 0;
    pv_done = 0;
    for (int i = 0; i < kNK; ++i) { mbar_init(smem_u32(&bars.k_full[i]), 1); mbar_init(smem_u32(&bars.k_empty[i]), 1); }
    for (int i = 0; i < kNV; ++i) {
      mbar_init(smem_u32(&bars.v_full[i]), 1);
      mbar_init(smem_u32(&bars.p_full[i]), 128);
      mbar_init(smem_u32(&bars.slot_empty[i]), 128);
    }
    fence_barrier_init();
  }
  __syncthreads();
  volatile int* abortp = &abort_flag;

  if (warp == 8) {
    if (lane == 0 && ntiles > 0) {
      prefetch_tensormap(&mk);
      prefetch_tensormap(&mv);
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % kNK, n = t / kNK;
        if (n > 0 && !mbar_wait(smem_u32(&bars.k_empty[s]), (n - 1) & 1, abortp, a.status)) break;
        const int row = (t1 - 1 - t) * kBK;                 // newest tile first
        const uint32_t kf = smem_u32(&bars.k_full[s]);
        mbar_expect_tx(kf, kTile);
        if (dbg_box(64, hk, row, b, kD, a.Hkv, 0, n_b, a.N, a.B, a.status)) {
          tma_load_4d(sK + s * kTile, &mk, kf, 0, hk, row, b);
          tma_load_4d(sK + s * kTile + kHalf, &mk, kf, 64, hk, row, b);
        }
        ++issued;
      }
      int never = 0;      // in-flight K loads must land before exit, abort or not
      for (int t = max(0, issued - kNK); t < issued; ++t)
        mbar_wait(smem_u32(&bars.k_full[t % kNK]), (t / kNK) & 1, &never, a.status);
    }
    return;
  }

  const int gq = lane >> 2, cq = lane & 3;       // fragment row group / column pair

  if (warp >= 4) {
    // ---------------- P V warps ----------------
    const int pw = warp - 4;
    float m_o0 = -INFINITY, m_o1 = -INFINITY;   // reference max of this thread's O columns (heads 2cq, 2cq+1)
    float o[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[i][e] = 0.f;
    bool ok = true;
    int n = 0;
    for (;; ++n) {
      const int vs = n % kNV;
      ok = ok && mbar_wait(smem_u32(&bars.p_full[vs]), (n / kNV) & 1, abortp, a.status);
      if (!__all_sync(0xffffffffu, ok) || pslot_end[vs]) break;
      ok = ok && mbar_wait(smem_u32(&bars.v_full[vs]), (n / kNV) & 1, abortp, a.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      // rescale O to the reference max this P was taken against
      const float mn0 = pslot_m[vs][2 * cq], mn1 = pslot_m[vs][2 * cq + 1];
      const float f0 = (m_o0 == -INFINITY) ? 0.f : ex2(m_o0 - mn0);
      const float f1 = (m_o1 == -INFINITY) ? 0.f : ex2(m_o1 - mn1);
      if (mn0 != -INFINITY) { o[0][0] *= f0; o[0][2] *= f0; o[1][0] *= f0; o[1][2] *= f0; m_o0 = mn0; }
      if (mn1 != -INFINITY) { o[0][1] *= f1; o[0][3] *= f1; o[1][1] *= f1; o[1][3] *= f1; m_o1 = mn1; }
      const uint32_t vbase = sV + vs * kTile;
      const uint32_t* prow = reinterpret_cast<const uint32_t*>(&pslot[vs][gq][0]);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t b0 = prow[(16 * k + 2 * cq) / 2];
        const uint32_t b1 = prow[(16 * k + 8 + 2 * cq) / 2];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          // A = V^T (16 d x 16 keys): four 8x8 transposed loads
          const int key = 16 * k + (lane & 7) + 8 * (lane >> 4);
          const int dchunk = (32 * pw + 16 * mt) / 8 + ((lane >> 3) & 1);
          uint32_t a0, a1, a2, a3;
          ldsm_x4_t(sw_addr(vbase, key, dchunk), a0, a1, a2, a3);
          mma_bf16(o[mt], a0, a1, a2, a3, b0, b1);
        }
      }
      mbar_arrive(smem_u32(&bars.slot_empty[vs]));
    }
    if (tid == 128) pv_done = n;
    if (__all_sync(0xffffffffu, ok) && !*abortp) {
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hrow = 0; hrow < 2; ++hrow) {
          const int d = 32 * pw + 16 * mt + gq + 8 * hrow;
#pragma unroll
          for (int e = 0; e < 2; ++e)
            if (2 * cq + e < G &&
                dbg_idx(((static_cast<size_t>(sp) * a.B + b) * a.Hq + hk * G + 2 * cq + e) * (kD + 4) + 4 + d,
                        static_cast<size_t>(a.splits) * a.B * a.Hq * (kD + 4), a.status))
              split_record(a, sp, b, hk * G + 2 * cq + e)[4 + d] = o[mt][2 * hrow + e];
        }
    }
    named_sync(2, 256);
    return;
  }

  // ---------------- score warps ----------------
  const bool test = a.tau > 0.f;
  const float thr = a.log2_tau - log2f(static_cast<float>(n_b));
  const float sl2 = a.scale_log2;
  const int g = lane & 7;                        // the head this lane decides

  // q^T as the B operand (K = d, N = heads): b0b1 = q[head gq][16k + 2cq ..], b2b3 = q[gq][16k + 8 + 2cq ..]
  uint32_t qb[8][2];
  {
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(a.q) +
                                                             (static_cast<size_t>(b) * a.Hq + hk * G + gq) * kD);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      qb[k][0] = gq < G ? qrow[(16 * k + 2 * cq) / 2] : 0u;
      qb[k][1] = gq < G ? qrow[(16 * k + 8 + 2 * cq) / 2] : 0u;
    }
  }
  float m_g = -INFINITY;                 // reference max of head g
  float lw0 = 0.f, lw1 = 0.f;            // this warp's partial sums for heads 2cq, 2cq+1 (exact)
  float lr0 = 0.f, lr1 = 0.f;            // the same sums of P as rounded to bf16
  int nret = 0, kept = 0, kept_g = 0;    // tiles kept by the group / by head g (lane g)
  bool ok = true;

  for (int t = 0; t < ntiles; ++t) {
    const int j = t1 - 1 - t;
    const int s = t % kNK;
    ok = ok && mbar_wait(smem_u32(&bars.k_full[s]), (t / kNK) & 1, abortp, a.status);
    // S^T for this warp's 32 keys: acc[mt] = rows (keys) 32w + 16mt + {gq, gq+8}, cols (heads) {2cq, 2cq+1}
    float acc[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][e] = 0.f;
    if (__all_sync(0xffffffffu, ok)) {
      const uint32_t kbase = sK + s * kTile;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          const int key = 32 * warp + 16 * mt + (lane & 7) + 8 * ((lane >> 3) & 1);
          const int dchunk = 2 * k + (lane >> 4);
          uint32_t a0, a1, a2, a3;
          ldsm_x4(sw_addr(kbase, key, dchunk), a0, a1, a2, a3);
          mma_bf16(acc[mt], a0, a1, a2, a3, qb[k][0], qb[k][1]);
        }
      }
    }
    // mask keys beyond the cache, row max per head
    const int kbase_idx = j * kBK + 32 * warp;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
      for (int hrow = 0; hrow < 2; ++hrow) {
        const bool valid = kbase_idx + 16 * mt + gq + 8 * hrow < n_b;
        acc[mt][2 * hrow] = valid ? acc[mt][2 * hrow] * sl2 : -INFINITY;
        acc[mt][2 * hrow + 1] = valid ? acc[mt][2 * hrow + 1] * sl2 : -INFINITY;
        mx0 = fmaxf(mx0, acc[mt][2 * hrow]);
        mx1 = fmaxf(mx1, acc[mt][2 * hrow + 1]);
      }
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    // publish this tile's maxima and the partial sums after the previous tile
    if (gq == 0) {
      xmax[t & 1][warp][2 * cq] = mx0; xmax[t & 1][warp][2 * cq + 1] = mx1;
      xl[t & 1][warp][2 * cq] = lw0; xl[t & 1][warp][2 * cq + 1] = lw1;
    }
    if (named_vote_or(1, 128, !ok || *abortp)) break;      // also the barrier for the exchange / K reads
    if (tid == 0) mbar_arrive(smem_u32(&bars.k_empty[s]));
    // Eq. (3) for head g: tile max - (m + log2 l) < log2(tau / N), l = 0 keeps
    const float tm = fmaxf(fmaxf(xmax[t & 1][0][g], xmax[t & 1][1][g]), fmaxf(xmax[t & 1][2][g], xmax[t & 1][3][g]));
    const float lt = (xl[t & 1][0][g] + xl[t & 1][1][g]) + (xl[t & 1][2][g] + xl[t & 1][3][g]);
    const bool keep_g = g < G && (lt == 0.f || !(tm - m_g - lg2(lt) < thr));
    const bool keep = !test || __any_sync(0xffffffffu, keep_g);
    // head g's own decision: in the group variant every head follows the group
    const bool own_g = a.per_head ? (!test || keep_g) : keep;
    if (a.mask != nullptr) {
      if (!a.per_head && tid == 0 &&
          dbg_idx((static_cast<size_t>(b) * a.Hkv + hk) * Tmax + j, static_cast<size_t>(a.B) * a.Hkv * Tmax, a.status))
        a.mask[(static_cast<size_t>(b) * a.Hkv + hk) * Tmax + j] = keep ? 1 : 0;
      if (a.per_head && tid < G &&
          dbg_idx((static_cast<size_t>(b) * a.Hq + hk * G + tid) * Tmax + j, static_cast<size_t>(a.B) * a.Hq * Tmax,
                  a.status))
        a.mask[(static_cast<size_t>(b) * a.Hq + hk * G + tid) * Tmax + j] = own_g ? 1 : 0;
    }
    if (!keep) continue;
    ++kept;
    kept_g += own_g ? 1 : 0;
    const int vs = nret % kNV;
    // the slot (P and V) is free once the P V of kept tile nret - kNV is done
    if (nret >= kNV) ok = ok && mbar_wait(smem_u32(&bars.slot_empty[vs]), ((nret / kNV) - 1) & 1, abortp, a.status);
    if (!__all_sync(0xffffffffu, ok)) continue;        // the next tile's vote ends every score warp's loop
    if (tid == 96) {
      const uint32_t vf = smem_u32(&bars.v_full[vs]);
      mbar_expect_tx(vf, kTile);
      if (dbg_box(64, hk, j * kBK, b, kD, a.Hkv, 0, n_b, a.N, a.B, a.status)) {
        tma_load_4d(sV + vs * kTile, &mv, vf, 0, hk, j * kBK, b);
        tma_load_4d(sV + vs * kTile + kHalf, &mv, vf, 64, hk, j * kBK, b);
      }
    }
    // lazily moved reference max (lane g), broadcast for this thread's heads 2cq, 2cq+1
    float alpha_g = 1.f;
    if (own_g && tm > m_g + kRescale) {
      alpha_g = (m_g == -INFINITY) ? 0.f : ex2(m_g - tm);
      m_g = tm;
    }
    const float m0 = __shfl_sync(0xffffffffu, m_g, 2 * cq), m1 = __shfl_sync(0xffffffffu, m_g, 2 * cq + 1);
    const float al0 = __shfl_sync(0xffffffffu, alpha_g, 2 * cq), al1 = __shfl_sync(0xffffffffu, alpha_g, 2 * cq + 1);
    const float mr0 = m0 == -INFINITY ? 0.f : m0;
    const float mr1 = m1 == -INFINITY ? 0.f : m1;
    // a head that skips this tile contributes P = 0 (its (m, l) stay as they are)
    const bool k0 = __shfl_sync(0xffffffffu, own_g, 2 * cq), k1 = __shfl_sync(0xffffffffu, own_g, 2 * cq + 1);
    float se0 = 0.f, se1 = 0.f, sr0 = 0.f, sr1 = 0.f;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
      for (int hrow = 0; hrow < 2; ++hrow) {
        const int key = 32 * warp + 16 * mt + gq + 8 * hrow;
        const float p0 = k0 ? ex2(acc[mt][2 * hrow] - mr0) : 0.f;
        const float p1 = k1 ? ex2(acc[mt][2 * hrow + 1] - mr1) : 0.f;
        const uint32_t w = pack_bf16(p0, p1);
        se0 += p0; se1 += p1;
        sr0 += __uint_as_float(w << 16);
        sr1 += __uint_as_float(w & 0xffff0000u);
        pslot[vs][2 * cq][key] = static_cast<uint16_t>(w & 0xffffu);
        pslot[vs][2 * cq + 1][key] = static_cast<uint16_t>(w >> 16);
      }
    }
    if (warp == 0 && lane < 8) pslot_m[vs][lane] = m_g;
    if (tid == 0) pslot_end[vs] = 0;
    mbar_arrive(smem_u32(&bars.p_full[vs]));
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      se0 += __shfl_xor_sync(0xffffffffu, se0, off);
      se1 += __shfl_xor_sync(0xffffffffu, se1, off);
      sr0 += __shfl_xor_sync(0xffffffffu, sr0, off);
      sr1 += __shfl_xor_sync(0xffffffffu, sr1, off);
    }
    lw0 = lw0 * al0 + se0; lw1 = lw1 * al1 + se1;
    lr0 = lr0 * al0 + sr0; lr1 = lr1 * al1 + sr1;
    ++nret;
  }
  // end of tiles for the P V warps (their slot must be free first)
  const int es = nret % kNV;
  if (nret >= kNV) ok = ok && mbar_wait(smem_u32(&bars.slot_empty[es]), ((nret / kNV) - 1) & 1, abortp, a.status);
  if (ok) {
    if (tid == 0) pslot_end[es] = 1;
    mbar_arrive(smem_u32(&bars.p_full[es]));
  }

  // split record: (m, l, l_rounded, 0) per query head, m in log2 units
  if (gq == 0) {
    xl[2][warp][2 * cq] = lw0; xl[2][warp][2 * cq + 1] = lw1;
    xlr[warp][2 * cq] = lr0; xlr[warp][2 * cq + 1] = lr1;
  }
  named_sync(1, 128);
  if (warp == 0 && lane < G && !*abortp &&
      dbg_idx(((static_cast<size_t>(sp) * a.B + b) * a.Hq + hk * G + lane) * (kD + 4) + 3,
              static_cast<size_t>(a.splits) * a.B * a.Hq * (kD + 4), a.status)) {
    float* rec = split_record(a, sp, b, hk * G + lane);
    rec[0] = m_g;
    rec[1] = (xl[2][0][lane] + xl[2][1][lane]) + (xl[2][2][lane] + xl[2][3][lane]);
    rec[2] = (xlr[0][lane] + xlr[1][lane]) + (xlr[2][lane] + xlr[3][lane]);
    rec[3] = 0.f;
  }
  if (a.counts != nullptr && !*abortp) {
    if (!a.per_head && tid == 0 &&
        dbg_idx((static_cast<size_t>(b) * a.Hkv + hk) * a.splits + sp, static_cast<size_t>(a.B) * a.Hkv * a.splits,
                a.status))
      a.counts[(static_cast<size_t>(b) * a.Hkv + hk) * a.splits + sp] = kept;
    if (a.per_head && tid < G &&
        dbg_idx((static_cast<size_t>(b) * a.Hq + hk * G + tid) * a.splits + sp, static_cast<size_t>(a.B) * a.Hq * a.splits,
                a.status))
      a.counts[(static_cast<size_t>(b) * a.Hq + hk * G + tid) * a.splits + sp] = kept_g;
  }
  named_sync(2, 256);
  // V loads issued but never consumed (abort path) must land before exit; these
  // waits ignore the abort flag (they are still bounded in time)
  if (tid == 0) {
    int never = 0;
    for (int n = pv_done; n < nret; ++n) mbar_wait(smem_u32(&bars.v_full[n % kNV]), (n / kNV) & 1, &never, a.status);
  }
}

}  // namespace

bool decode_mma_supported(const DecArgs& a) {
  return a.in_dt == kBF16 && a.D == kD && a.blk == kBK && a.Hq / a.Hkv <= 8;
}

cudaError_t launch_decode_mma(const DecArgs& a, cudaStream_t s, int* launches) {
  CUtensorMap mk, mv;
  if (!encode_bshd_map(&mk, a.k, a.B, a.N, a.Hkv, kD, kBK) || !encode_bshd_map(&mv, a.v, a.B, a.N, a.Hkv, kD, kBK))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.Hkv, a.splits, a.B);
  ++*launches;
  decode_mma_kernel<<<grid, kThreads, kSmem, s>>>(mk, mv, a);
  return cudaGetLastError();
}

}  // namespace mala
