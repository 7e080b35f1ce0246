// CUDA-core MALA kernels with fp32 arithmetic throughout.
//
// These serve the fp32 workloads (where a tensor-core path would round the
// operands) and any shape the tensor-core kernels do not cover.  They follow
// the same tile schedule and decision rule as the tensor-core kernels:
//   "MassAlloc Attention: Let Attention Allocate Its Own Compute",
//   Algorithm 1 / Eq. (3) (forward), Algorithm 2 / Eq. (4) (backward),
//   App. A.1 (split-KV decoding); split merge from "Why exact attention does
//   not need a quadratic matrix", Method/Mechanism.
//
// Scores are kept in log2 units (s2 = s * log2 e), so every test
// "x < log(tau / L)" becomes "x2 < log2(tau) - log2(L)" and exp becomes exp2.
//
// Thread layout of the prefill kernels: TPR = D / 32 threads own one row of
// the block (a query row in forward, a key row in backward); thread `part` of
// a row owns the 32 head dimensions {c * TPR + part}.  Dot products are
// reduced across the TPR adjacent lanes with xor shuffles.

#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>

#include "mala_internal.h"

namespace mala {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float ld(const float* p) { return *p; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st(float* p, float x) { *p = x; }
template <typename T> __device__ __forceinline__ T zero();
template <> __device__ __forceinline__ float zero<float>() { return 0.f; }
template <> __device__ __forceinline__ __nv_bfloat16 zero<__nv_bfloat16>() { return __float2bfloat16_rn(0.f); }
__device__ __forceinline__ void st(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

template <int TPR>
__device__ __forceinline__ float row_sum(float x) {
#pragma unroll
  for (int off = 1; off < TPR; off <<= 1) x += __shfl_xor_sync(kFull, x, off);
  return x;
}

// ---------------------------------------------------------------------------
// Forward: one CTA per (query block, query head, batch).
// ---------------------------------------------------------------------------
template <typename Tin, typename Tout, int D, int BLK>
__global__ void __launch_bounds__(BLK * (D / 32))
fwd_simt_kernel(const FwdArgs a) {
  constexpr int TPR = D / 32;
  constexpr int NT = BLK * TPR;
  constexpr int SS = BLK + 1;                 // padded row stride of the score tile
  extern __shared__ float smem[];
  float* Ks = smem;                           // [BLK][D]
  float* Vs = Ks + BLK * D;                   // [BLK][D]
  float* Ss = Vs + BLK * D;                   // [BLK][SS] scores, log2 units

  const int qb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  // this CTA's sequence: its lengths, first row and batch coordinate in the layout
  const SeqSpan sq = seq_span(a, b);
  const int Lq = sq.Lq, Lk = sq.Lk, row0 = sq.row0, bc = sq.bc;
  const int Tr = (Lq + BLK - 1) / BLK;
  const int Tc = (Lk + BLK - 1) / BLK;
  if (qb >= Tr) return;                   // past the sequence's query blocks (packed batches)
  // tile rows / columns of mask and counts (a packed batch pads each sequence to Lmax)
  const int mTr = a.cu ? (a.Lmax + BLK - 1) / BLK : Tr, mTc = a.cu ? mTr : Tc;
  const int hk = h / (a.Hq / a.Hkv);
  const int tid = threadIdx.x, r = tid / TPR, part = tid % TPR;
  const int qrow = qb * BLK + r;
  const bool row_valid = qrow < Lq;
  const Tin* qg = static_cast<const Tin*>(a.q);
  const Tin* kg = static_cast<const Tin*>(a.k);
  const Tin* vg = static_cast<const Tin*>(a.v);

  float qv[32], acc[32];
  {
    const Tin* qp = qg + ((static_cast<size_t>(bc) * a.Lq + row0 + (row_valid ? qrow : 0)) * a.Hq + h) * D;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      qv[c] = row_valid ? ld(qp + c * TPR + part) * a.scale_log2 : 0.f;
      acc[c] = 0.f;
    }
  }
  float m = -INFINITY, l = 0.f;
  const float lvis = a.causal ? static_cast<float>(qrow + 1) : static_cast<float>(Lk);
  const float thr = a.log2_tau - log2f(lvis);
  const bool test = a.tau > 0.f;
  const int jtop = a.causal ? min(Tc - 1, (min(Lq, qb * BLK + BLK) - 1) / BLK) : Tc - 1;
  int kept = 0;

  for (int j = jtop; j >= 0; --j) {
    const int k0 = j * BLK;
    __syncthreads();
    for (int idx = tid; idx < BLK * D; idx += NT) {
      const int kr = idx / D, c = idx % D, key = k0 + kr;
      Ks[idx] = key < Lk ? ld(kg + ((static_cast<size_t>(bc) * a.Lk + row0 + key) * a.Hkv + hk) * D + c) : 0.f;
    }
    __syncthreads();
    float mt = -INFINITY;
    for (int kr = 0; kr < BLK; ++kr) {
      float s = 0.f;
#pragma unroll
      for (int c = 0; c < 32; ++c) s = fmaf(qv[c], Ks[kr * D + c * TPR + part], s);
      s = row_sum<TPR>(s);
      const int key = k0 + kr;
      const bool legal = row_valid && key < Lk && (!a.causal || key <= qrow);
      s = legal ? s : -INFINITY;
      mt = fmaxf(mt, s);
      if (part == 0) Ss[r * SS + kr] = s;
    }
    // Eq. (3): the row keeps the tile unless rowmax - m - log l < log(tau / L_q);
    // l = 0 keeps it; rows with no legal key here do not vote.
    bool keep_row = false;
    if (row_valid && mt > -INFINITY)
      keep_row = !test || l == 0.f || !(mt - m - log2f(l) < thr);
    int keep = __syncthreads_or(keep_row);
    // forced decisions: the given tile set, with no test (matched-work controls)
    if (a.force != nullptr) keep = a.force[((static_cast<size_t>(b) * a.Hq + h) * mTr + qb) * mTc + j] != 0;
    if (a.mask != nullptr && tid == 0)
      a.mask[((static_cast<size_t>(b) * a.Hq + h) * mTr + qb) * mTc + j] = keep ? 1 : 0;
    if (!keep) continue;
    ++kept;
    for (int idx = tid; idx < BLK * D; idx += NT) {
      const int kr = idx / D, c = idx % D, key = k0 + kr;
      Vs[idx] = key < Lk ? ld(vg + ((static_cast<size_t>(bc) * a.Lk + row0 + key) * a.Hkv + hk) * D + c) : 0.f;
    }
    __syncthreads();
    if (mt > -INFINITY) {
      const float m_new = fmaxf(m, mt);
      const float alpha = l > 0.f ? exp2f(m - m_new) : 1.f;
      l *= alpha;
#pragma unroll
      for (int c = 0; c < 32; ++c) acc[c] *= alpha;
      for (int kr = 0; kr < BLK; ++kr) {
        const float p = exp2f(Ss[r * SS + kr] - m_new);
        l += p;
#pragma unroll
        for (int c = 0; c < 32; ++c) acc[c] = fmaf(p, Vs[kr * D + c * TPR + part], acc[c]);
      }
      m = m_new;
    }
  }
  if (row_valid) {
    Tout* op = static_cast<Tout*>(a.o) + ((static_cast<size_t>(bc) * a.Lq + row0 + qrow) * a.Hq + h) * D;
    // l = 0 only when forced decisions keep none of the row's keys: o = 0, lse = -inf
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int c = 0; c < 32; ++c) st(op + c * TPR + part, acc[c] * inv);
    if (part == 0)
      a.lse[(static_cast<size_t>(bc) * a.Hq + h) * a.Lq + row0 + qrow] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
  }
  if (a.counts != nullptr && tid == 0) a.counts[(static_cast<size_t>(b) * a.Hq + h) * mTr + qb] = kept;
}

// ---------------------------------------------------------------------------
// Reference region mass (the matched-work study of the MALA paper, App. C.2):
// for query block qb and key tile j, the sum over the block's valid rows and
// the tile's legal keys of exp(s - lse), lse being the row's final
// log-normaliser.  One CTA per (query block, query head, batch), one tile at a
// time from the diagonal down; illegal tiles get 0.
// ---------------------------------------------------------------------------
template <typename Tin, int D, int BLK>
__global__ void __launch_bounds__(BLK * (D / 32))
region_mass_kernel(const FwdArgs a) {
  constexpr int TPR = D / 32;
  constexpr int NT = BLK * TPR;
  extern __shared__ float smem[];
  float* Ks = smem;                           // [BLK][D]
  __shared__ float tile_sum;

  const int qb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int Lq = a.Lq, Lk = a.Lk;
  const int Tr = (Lq + BLK - 1) / BLK, Tc = (Lk + BLK - 1) / BLK;
  if (qb >= Tr) return;
  const int hk = h / (a.Hq / a.Hkv);
  const int tid = threadIdx.x, r = tid / TPR, part = tid % TPR;
  const int qrow = qb * BLK + r;
  const bool row_valid = qrow < Lq;
  const Tin* qg = static_cast<const Tin*>(a.q);
  const Tin* kg = static_cast<const Tin*>(a.k);

  float qv[32];
  {
    const Tin* qp = qg + ((static_cast<size_t>(b) * Lq + (row_valid ? qrow : 0)) * a.Hq + h) * D;
#pragma unroll
    for (int c = 0; c < 32; ++c) qv[c] = row_valid ? ld(qp + c * TPR + part) * a.scale_log2 : 0.f;
  }
  const float lse2 = row_valid ? a.lse[(static_cast<size_t>(b) * a.Hq + h) * Lq + qrow] * kLog2e : 0.f;
  const int jtop = a.causal ? min(Tc - 1, (min(Lq, qb * BLK + BLK) - 1) / BLK) : Tc - 1;
  float* out = a.region_mass + ((static_cast<size_t>(b) * a.Hq + h) * Tr + qb) * Tc;
  for (int j = jtop + 1 + tid; j < Tc; j += NT) out[j] = 0.f;

  for (int j = jtop; j >= 0; --j) {
    const int k0 = j * BLK;
    __syncthreads();
    for (int idx = tid; idx < BLK * D; idx += NT) {
      const int kr = idx / D, c = idx % D, key = k0 + kr;
      Ks[idx] = key < Lk ? ld(kg + ((static_cast<size_t>(b) * Lk + key) * a.Hkv + hk) * D + c) : 0.f;
    }
    if (tid == 0) tile_sum = 0.f;
    __syncthreads();
    float ps = 0.f;
    for (int kr = 0; kr < BLK; ++kr) {
      float s = 0.f;
#pragma unroll
      for (int c = 0; c < 32; ++c) s = fmaf(qv[c], Ks[kr * D + c * TPR + part], s);
      s = row_sum<TPR>(s);
      const int key = k0 + kr;
      const bool legal = row_valid && key < Lk && (!a.causal || key <= qrow);
      if (legal && part == 0) ps += exp2f(s - lse2);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(kFull, ps, off);
    if ((tid & 31) == 0) atomicAdd(&tile_sum, ps);
    __syncthreads();
    if (tid == 0) out[j] = tile_sum;
  }
}

// ---------------------------------------------------------------------------
// Backward preprocess: D = rowsum(O * dO) per (b, h, q), and zero the fp32
// dQ accumulator.  One warp per row.
// ---------------------------------------------------------------------------
template <typename Tin>
__global__ void bwd_preprocess_kernel(const BwdArgs a) {
  const size_t rows = static_cast<size_t>(a.cu ? 1 : a.B) * a.Lq * a.Hq;   // a packed batch: one run
  const size_t row = (static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  if (row >= rows) return;
  const Tin* op = static_cast<const Tin*>(a.o) + row * a.D;
  const Tin* dp = static_cast<const Tin*>(a.dout) + row * a.D;
  float s = 0.f;
  for (int c = lane; c < a.D; c += 32) {
    s = fmaf(ld(op + c), ld(dp + c), s);
    a.dq_acc[row * a.D + c] = 0.f;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(kFull, s, off);
  if (lane == 0) {
    // row = (b * Lq + q) * Hq + h  ->  delta[(b * Hq + h) * Lq + q]
    const int h = static_cast<int>(row % a.Hq);
    const size_t bq = row / a.Hq;
    const int q = static_cast<int>(bq % a.Lq);
    const size_t b = bq / a.Lq;
    a.delta[(b * a.Hq + h) * a.Lq + q] = s;
  }
}

template <typename Tg>
__global__ void dq_convert_kernel(const BwdArgs a) {
  const size_t n = static_cast<size_t>(a.cu ? 1 : a.B) * a.Lq * a.Hq * a.D;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    st(static_cast<Tg*>(a.dq) + i, a.dq_acc[i]);
}

// ---------------------------------------------------------------------------
// Backward: one CTA per (key block, KV head, batch); it loops over the query
// heads of the KV group and, for each, over the query blocks in ascending
// order from the diagonal.  dK, dV stay in registers; dQ is added to the
// fp32 accumulator with atomics.
// ---------------------------------------------------------------------------
template <typename Tin, typename Tg, int D, int BLK>
__global__ void __launch_bounds__(BLK * (D / 32))
bwd_simt_kernel(const BwdArgs a) {
  constexpr int TPR = D / 32;
  constexpr int NT = BLK * TPR;
  constexpr int KS = D + TPR;                  // padded row stride of K, V tiles
  constexpr int SS = BLK + 1;
  extern __shared__ float smem[];
  Tin* Ks = reinterpret_cast<Tin*>(smem);      // [BLK][KS]  (own key block)
  Tin* Vs = Ks + BLK * KS;                     // [BLK][KS]
  Tin* Qs = Vs + BLK * KS;                     // [BLK][D]
  Tin* dOs = Qs + BLK * D;                     // [BLK][D]
  float* Ss = reinterpret_cast<float*>(dOs + BLK * D);   // [BLK keys][SS]: S^T, then dS^T
  float* lse2 = Ss + BLK * SS;                 // [BLK]
  float* dlt = lse2 + BLK;                     // [BLK]
  float* thr = dlt + BLK;                      // [BLK]

  const int kb = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  // this CTA's sequence: its lengths, first row and batch coordinate in the layout
  const SeqSpan sq = seq_span(a, b);
  const int Lq = sq.Lq, Lk = sq.Lk, row0 = sq.row0, bc = sq.bc;
  const int Tr = (Lq + BLK - 1) / BLK;
  const int Tc = (Lk + BLK - 1) / BLK;
  if (kb >= Tc) return;                   // past the sequence's key blocks (packed batches)
  // tile rows / columns of mask and counts (a packed batch pads each sequence to Lmax)
  const int mTr = a.cu ? (a.Lmax + BLK - 1) / BLK : Tr, mTc = a.cu ? mTr : Tc;
  const int G = a.Hq / a.Hkv;
  const int tid = threadIdx.x, kr = tid / TPR, part = tid % TPR;
  const int key = kb * BLK + kr;
  const Tin* qg = static_cast<const Tin*>(a.q);
  const Tin* kg = static_cast<const Tin*>(a.k);
  const Tin* vg = static_cast<const Tin*>(a.v);
  const Tin* dog = static_cast<const Tin*>(a.dout);
  const bool test = a.tau > 0.f;

  for (int idx = tid; idx < BLK * D; idx += NT) {
    const int rr = idx / D, c = idx % D, kk = kb * BLK + rr;
    const size_t off = ((static_cast<size_t>(bc) * a.Lk + row0 + (kk < Lk ? kk : 0)) * a.Hkv + hk) * D + c;
    Ks[rr * KS + c] = kk < Lk ? kg[off] : zero<Tin>();
    Vs[rr * KS + c] = kk < Lk ? vg[off] : zero<Tin>();
  }
  float dk[32], dv[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) dk[c] = dv[c] = 0.f;
  const int ibot = a.causal ? (kb * BLK) / BLK : 0;

  for (int hh = 0; hh < G; ++hh) {
    const int h = hk * G + hh;
    int kept = 0;
    for (int i = ibot; i < Tr; ++i) {
      const int q0 = i * BLK;
      __syncthreads();
      for (int idx = tid; idx < BLK * D; idx += NT) {
        const int rr = idx / D, c = idx % D, qq = q0 + rr;
        const size_t off = ((static_cast<size_t>(bc) * a.Lq + row0 + (qq < Lq ? qq : 0)) * a.Hq + h) * D + c;
        Qs[idx] = qq < Lq ? qg[off] : zero<Tin>();
        dOs[idx] = qq < Lq ? dog[off] : zero<Tin>();
      }
      for (int rr = tid; rr < BLK; rr += NT) {
        const int qq = q0 + rr;
        const size_t off = (static_cast<size_t>(bc) * a.Hq + h) * a.Lq + row0 + (qq < Lq ? qq : 0);
        lse2[rr] = qq < Lq ? a.lse[off] * kLog2e : 0.f;
        dlt[rr] = qq < Lq ? a.delta[off] : 0.f;
        thr[rr] = a.log2_tau - log2f(a.causal ? static_cast<float>(qq + 1) : static_cast<float>(Lk));
      }
      __syncthreads();
      // Scores S^T of this tile; Eq. (4): keep iff some valid entry has
      // S - lse >= log(tau / L_q).
      bool keep_local = false;
      for (int qq = 0; qq < BLK; ++qq) {
        float s = 0.f;
#pragma unroll
        for (int c = 0; c < 32; ++c)
          s = fmaf(ld(Ks + kr * KS + c * TPR + part), ld(Qs + qq * D + c * TPR + part), s);
        s = row_sum<TPR>(s) * a.scale_log2;
        const int qrow = q0 + qq;
        const bool valid = key < Lk && qrow < Lq && (!a.causal || key <= qrow);
        s = valid ? s : -INFINITY;
        if (valid && (!test || !(s - lse2[qq] < thr[qq]))) keep_local = true;
        if (part == 0) Ss[kr * SS + qq] = s;
      }
      const int keep = __syncthreads_or(keep_local);
      if (a.mask != nullptr && tid == 0)
        a.mask[((static_cast<size_t>(b) * a.Hq + h) * mTr + i) * mTc + kb] = keep ? 1 : 0;
      if (!keep) continue;
      ++kept;
      for (int qq = 0; qq < BLK; ++qq) {
        const float p = exp2f(Ss[kr * SS + qq] - lse2[qq]);
        float dp = 0.f;
#pragma unroll
        for (int c = 0; c < 32; ++c)
          dp = fmaf(ld(Vs + kr * KS + c * TPR + part), ld(dOs + qq * D + c * TPR + part), dp);
        dp = row_sum<TPR>(dp);
        const float ds = p * (dp - dlt[qq]);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          dv[c] = fmaf(p, ld(dOs + qq * D + c * TPR + part), dv[c]);
          dk[c] = fmaf(ds, ld(Qs + qq * D + c * TPR + part), dk[c]);
        }
        __syncwarp();
        if (part == 0) Ss[kr * SS + qq] = ds;
      }
      __syncthreads();
      // dQ_i += scale * dS^T K_j : thread (row qq = tid / TPR, part) sums over keys.
      {
        const int qq = tid / TPR;
        const int qrow = q0 + qq;
        if (qrow < Lq) {
          float* dqp = a.dq_acc + ((static_cast<size_t>(bc) * a.Lq + row0 + qrow) * a.Hq + h) * D;
          for (int c = 0; c < 32; ++c) {
            float sum = 0.f;
            for (int k2 = 0; k2 < BLK; ++k2)
              sum = fmaf(Ss[k2 * SS + qq], ld(Ks + k2 * KS + c * TPR + part), sum);
            atomicAdd(dqp + c * TPR + part, sum * a.scale);
          }
        }
      }
    }
    if (a.counts != nullptr && tid == 0) a.counts[(static_cast<size_t>(b) * a.Hq + h) * mTc + kb] = kept;
  }
  if (key < Lk) {
    const size_t off = ((static_cast<size_t>(bc) * a.Lk + row0 + key) * a.Hkv + hk) * D;
    Tg* dkp = static_cast<Tg*>(a.dk) + off;
    Tg* dvp = static_cast<Tg*>(a.dv) + off;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      st(dkp + c * TPR + part, dk[c] * a.scale);
      st(dvp + c * TPR + part, dv[c]);
    }
  }
}

// ---------------------------------------------------------------------------
// Split-KV decode: one CTA of 128 threads per (split, KV head, batch); the G
// query heads of the group form the query block (or, per head, each query head
// decides alone: a head that skips a kept tile takes P = 0 and keeps its
// (m, l)).  Writes (m, l, u) per head.
// ---------------------------------------------------------------------------
template <typename Tin, int D, int G, int BK>
__global__ void __launch_bounds__(128)
decode_split_simt_kernel(const DecArgs a) {
  constexpr int NT = 128, NW = NT / 32;
  extern __shared__ float smem[];
  float (*qs)[D] = reinterpret_cast<float (*)[D]>(smem);                 // [G][D]
  float (*Ks)[D + 1] = reinterpret_cast<float (*)[D + 1]>(smem + G * D);  // [BK][D+1]
  float (*Vs)[D] = reinterpret_cast<float (*)[D]>(smem + G * D + BK * (D + 1));   // [BK][D]
  float (*Ps)[BK] = reinterpret_cast<float (*)[BK]>(smem + G * D + BK * (2 * D + 1));  // [G][BK]
  float (*red)[NW] = reinterpret_cast<float (*)[NW]>(smem + G * D + BK * (2 * D + 1) + G * BK);

  const int sp = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const Tin* qg = static_cast<const Tin*>(a.q);
  const Tin* kg = static_cast<const Tin*>(a.k);
  const Tin* vg = static_cast<const Tin*>(a.v);
  const int n_b = decode_seq_len(a, b);                // this sequence's cache length
  const int T = (n_b + BK - 1) / BK;
  const int Tmax = (a.N + BK - 1) / BK;                // row length of the tile mask
  const int per = (T + a.splits - 1) / a.splits;
  const int t0 = sp * per, t1 = min(T, t0 + per);
  const bool test = a.tau > 0.f;
  const float thr = a.log2_tau - log2f(static_cast<float>(n_b));

  for (int idx = tid; idx < G * D; idx += NT) {
    const int g = idx / D, c = idx % D;
    qs[g][c] = ld(qg + (static_cast<size_t>(b) * a.Hq + hk * G + g) * D + c) * a.scale_log2;
  }
  float m[G], l[G], u[G];
#pragma unroll
  for (int g = 0; g < G; ++g) { m[g] = -INFINITY; l[g] = 0.f; u[g] = 0.f; }
  int kept = 0;
  __shared__ int kept_h[G];             // tiles kept by each head (per-head variant)
  if (tid < G) kept_h[tid] = 0;

  for (int j = t1 - 1; j >= t0; --j) {
    const int k0 = j * BK;
    __syncthreads();
    for (int idx = tid; idx < BK * D; idx += NT) {
      const int kr = idx / D, c = idx % D, key = k0 + kr;
      Ks[kr][c] = key < n_b ? ld(kg + ((static_cast<size_t>(b) * a.N + key) * a.Hkv + hk) * D + c) : 0.f;
    }
    __syncthreads();
    float mloc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) mloc[g] = -INFINITY;
    for (int kr = tid; kr < BK; kr += NT) {
      const bool valid = k0 + kr < n_b;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float s = 0.f;
        for (int c = 0; c < D; ++c) s = fmaf(qs[g][c], Ks[kr][c], s);
        s = valid ? s : -INFINITY;
        Ps[g][kr] = s;
        mloc[g] = fmaxf(mloc[g], s);
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float x = mloc[g];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(kFull, x, off));
      if (lane == 0) red[g][warp] = x;
    }
    __syncthreads();
    float mt[G];
    uint32_t own = 0;                     // bit g: head g keeps the tile
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float x = red[g][0];
#pragma unroll
      for (int w = 1; w < NW; ++w) x = fmaxf(x, red[g][w]);
      mt[g] = x;
      if (!test || l[g] == 0.f || !(x - m[g] - log2f(l[g]) < thr)) own |= 1u << g;
    }
    const bool keep = own != 0;
    if (!a.per_head && keep) own = (1u << G) - 1u;   // group: every head follows the group
    if (a.mask != nullptr && tid == 0) {
      if (a.per_head) {
#pragma unroll
        for (int g = 0; g < G; ++g)
          a.mask[(static_cast<size_t>(b) * a.Hq + hk * G + g) * Tmax + j] = (own >> g) & 1u;
      } else {
        a.mask[(static_cast<size_t>(b) * a.Hkv + hk) * Tmax + j] = keep ? 1 : 0;
      }
    }
    if (!keep) continue;
    ++kept;
    if (tid < G) kept_h[tid] += (own >> tid) & 1u;
    for (int idx = tid; idx < BK * D; idx += NT) {
      const int kr = idx / D, c = idx % D, key = k0 + kr;
      Vs[kr][c] = key < n_b ? ld(vg + ((static_cast<size_t>(b) * a.N + key) * a.Hkv + hk) * D + c) : 0.f;
    }
    float mnew[G], alpha[G], psum[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const bool og = (own >> g) & 1u;
      mnew[g] = og ? fmaxf(m[g], mt[g]) : m[g];
      alpha[g] = (og && l[g] > 0.f) ? exp2f(m[g] - mnew[g]) : 1.f;
      psum[g] = 0.f;
    }
    __syncthreads();   // red[] reads above and Ps writes below; Vs complete
    for (int kr = tid; kr < BK; kr += NT) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float p = ((own >> g) & 1u) ? exp2f(Ps[g][kr] - mnew[g]) : 0.f;
        Ps[g][kr] = p;
        psum[g] += p;
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float x = psum[g];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(kFull, x, off);
      if (lane == 0) red[g][warp] = x;
    }
    __syncthreads();
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float x = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) x += red[g][w];
      l[g] = alpha[g] * l[g] + x;
      m[g] = mnew[g];
    }
    for (int c = tid; c < D; c += NT) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float s = alpha[g] * u[g];
        for (int kr = 0; kr < BK; ++kr) s = fmaf(Ps[g][kr], Vs[kr][c], s);
        u[g] = s;
      }
    }
  }
  for (int c = tid; c < D; c += NT) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float* pp = a.partial + ((static_cast<size_t>(sp) * a.B + b) * a.Hq + hk * G + g) * (D + 4);
      if (c == 0) { pp[0] = m[g]; pp[1] = l[g]; pp[2] = l[g]; pp[3] = 0.f; }   // P is not rounded here
      pp[4 + c] = u[g];
    }
  }
  if (a.counts != nullptr && tid == 0) {
    if (a.per_head) {
#pragma unroll
      for (int g = 0; g < G; ++g) a.counts[(static_cast<size_t>(b) * a.Hq + hk * G + g) * a.splits + sp] = kept_h[g];
    } else {
      a.counts[(static_cast<size_t>(b) * a.Hkv + hk) * a.splits + sp] = kept;
    }
  }
}

// Exact merge of the splits' (m, l, u): one CTA per (query head, batch).
// o = sum_s e^(m_s - M) u_s / sum_s e^(m_s - M) l_rounded_s (the sums of the P
// values that entered the P V products); lse = M + log sum_s e^(m_s - M) l_s.
template <typename Tout>
__global__ void decode_merge_kernel(const DecArgs a) {
  const int h = blockIdx.x, b = blockIdx.y;
  const int D = a.D;
  const size_t stride = static_cast<size_t>(a.B) * a.Hq * (D + 4);
  const float* base = a.partial + (static_cast<size_t>(b) * a.Hq + h) * (D + 4);
  float mmax = -INFINITY;
  for (int s = 0; s < a.splits; ++s)
    if (base[s * stride + 1] > 0.f) mmax = fmaxf(mmax, base[s * stride]);
  float lsum = 0.f, lrsum = 0.f;
  for (int s = 0; s < a.splits; ++s) {
    const float ls = base[s * stride + 1];
    if (ls > 0.f) {
      const float w = exp2f(base[s * stride] - mmax);
      lsum += w * ls;
      lrsum += w * base[s * stride + 2];
    }
  }
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float u = 0.f;
    for (int s = 0; s < a.splits; ++s) {
      const float ls = base[s * stride + 1];
      if (ls > 0.f) u += exp2f(base[s * stride] - mmax) * base[s * stride + 4 + c];
    }
    // a sequence with no keys (a rejected length) has lsum = 0: NaN output
    st(static_cast<Tout*>(a.o) + (static_cast<size_t>(b) * a.Hq + h) * D + c, lsum > 0.f ? u / lrsum : NAN);
  }
  if (threadIdx.x == 0) a.lse[static_cast<size_t>(b) * a.Hq + h] = lsum > 0.f ? (mmax + log2f(lsum)) * kLn2 : NAN;
}

// ---------------------------------------------------------------------------
// Dispatch.
// ---------------------------------------------------------------------------
template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

template <typename Tin, typename Tout, int D, int BLK>
cudaError_t fwd_go(const FwdArgs& a, cudaStream_t s) {
  const size_t smem = fwd_simt_smem(a.in_dt, D, BLK);
  auto kern = fwd_simt_kernel<Tin, Tout, D, BLK>;
  cudaError_t e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(((a.cu ? a.Lmax : a.Lq) + BLK - 1) / BLK, a.Hq, a.B);
  kern<<<grid, BLK * (D / 32), smem, s>>>(a);
  return cudaGetLastError();
}

template <typename Tin, typename Tout>
cudaError_t fwd_pick(const FwdArgs& a, cudaStream_t s) {
  if (a.D == 64 && a.blk == 64) return fwd_go<Tin, Tout, 64, 64>(a, s);
  if (a.D == 64 && a.blk == 128) return fwd_go<Tin, Tout, 64, 128>(a, s);
  if (a.D == 128 && a.blk == 64) return fwd_go<Tin, Tout, 128, 64>(a, s);
  return fwd_go<Tin, Tout, 128, 128>(a, s);
}

template <typename Tin, int D, int BLK>
cudaError_t mass_go(const FwdArgs& a, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(BLK) * D * sizeof(float);
  auto kern = region_mass_kernel<Tin, D, BLK>;
  cudaError_t e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((a.Lq + BLK - 1) / BLK, a.Hq, a.B);
  kern<<<grid, BLK * (D / 32), smem, s>>>(a);
  return cudaGetLastError();
}

template <typename Tin, typename Tg, int D, int BLK>
cudaError_t bwd_go(const BwdArgs& a, cudaStream_t s) {
  const size_t smem = bwd_simt_smem(a.in_dt, D, BLK);
  auto kern = bwd_simt_kernel<Tin, Tg, D, BLK>;
  cudaError_t e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(((a.cu ? a.Lmax : a.Lk) + BLK - 1) / BLK, a.Hkv, a.B);
  kern<<<grid, BLK * (D / 32), smem, s>>>(a);
  return cudaGetLastError();
}

template <typename Tin, typename Tg>
cudaError_t bwd_pick(const BwdArgs& a, cudaStream_t s) {
  if (a.D == 64 && a.blk == 64) return bwd_go<Tin, Tg, 64, 64>(a, s);
  if (a.D == 64 && a.blk == 128) return bwd_go<Tin, Tg, 64, 128>(a, s);
  if (a.D == 128 && a.blk == 64) return bwd_go<Tin, Tg, 128, 64>(a, s);
  return bwd_go<Tin, Tg, 128, 128>(a, s);
}

template <typename Tin, int D, int G, int BK>
cudaError_t dec_go_gb(const DecArgs& a, cudaStream_t s) {
  const size_t smem = (static_cast<size_t>(G) * D + BK * (2 * D + 1) + G * BK + G * 4) * sizeof(float);
  auto kern = decode_split_simt_kernel<Tin, D, G, BK>;
  cudaError_t e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.splits, a.Hkv, a.B);
  kern<<<grid, 128, smem, s>>>(a);
  return cudaGetLastError();
}

template <typename Tin, int D, int G>
cudaError_t dec_go_g(const DecArgs& a, cudaStream_t s) {
  return a.blk == 64 ? dec_go_gb<Tin, D, G, 64>(a, s) : dec_go_gb<Tin, D, G, 128>(a, s);
}

template <typename Tin, int D>
cudaError_t dec_go(const DecArgs& a, cudaStream_t s) {
  switch (a.Hq / a.Hkv) {
    case 1: return dec_go_g<Tin, D, 1>(a, s);
    case 2: return dec_go_g<Tin, D, 2>(a, s);
    case 4: return dec_go_g<Tin, D, 4>(a, s);
    default: return dec_go_g<Tin, D, 8>(a, s);
  }
}

}  // namespace

size_t fwd_simt_smem(int /*in_dt*/, int D, int blk) {
  return (2u * blk * D + static_cast<size_t>(blk) * (blk + 1)) * sizeof(float);
}

size_t bwd_simt_smem(int in_dt, int D, int blk) {
  const size_t es = in_dt == kBF16 ? 2 : 4;
  const int tpr = D / 32;
  size_t bytes = 2 * static_cast<size_t>(blk) * (D + tpr) * es + 2 * static_cast<size_t>(blk) * D * es;
  bytes = (bytes + 15) / 16 * 16;
  bytes += (static_cast<size_t>(blk) * (blk + 1) + 3 * blk) * sizeof(float);
  return bytes;
}

cudaError_t launch_region_mass(const FwdArgs& a, cudaStream_t s, int* launches) {
  ++*launches;
  if (a.in_dt == kBF16) {
    if (a.D == 64) return a.blk == 64 ? mass_go<__nv_bfloat16, 64, 64>(a, s) : mass_go<__nv_bfloat16, 64, 128>(a, s);
    return a.blk == 64 ? mass_go<__nv_bfloat16, 128, 64>(a, s) : mass_go<__nv_bfloat16, 128, 128>(a, s);
  }
  if (a.D == 64) return a.blk == 64 ? mass_go<float, 64, 64>(a, s) : mass_go<float, 64, 128>(a, s);
  return a.blk == 64 ? mass_go<float, 128, 64>(a, s) : mass_go<float, 128, 128>(a, s);
}

cudaError_t launch_fwd_simt(const FwdArgs& a, cudaStream_t s, int* launches) {
  ++*launches;
  if (a.in_dt == kBF16)
    return a.out_dt == kBF16 ? fwd_pick<__nv_bfloat16, __nv_bfloat16>(a, s) : fwd_pick<__nv_bfloat16, float>(a, s);
  return a.out_dt == kBF16 ? fwd_pick<float, __nv_bfloat16>(a, s) : fwd_pick<float, float>(a, s);
}

cudaError_t launch_bwd_preprocess(const BwdArgs& a, cudaStream_t s, int* launches) {
  ++*launches;
  const size_t rows = static_cast<size_t>(a.cu ? 1 : a.B) * a.Lq * a.Hq;   // a packed batch: one run
  const unsigned blocks = static_cast<unsigned>((rows * 32 + 255) / 256);
  if (a.in_dt == kBF16) bwd_preprocess_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(a);
  else bwd_preprocess_kernel<float><<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_simt(const BwdArgs& a, cudaStream_t s, int* launches) {
  ++*launches;
  if (a.in_dt == kBF16)
    return a.grad_dt == kBF16 ? bwd_pick<__nv_bfloat16, __nv_bfloat16>(a, s) : bwd_pick<__nv_bfloat16, float>(a, s);
  return a.grad_dt == kBF16 ? bwd_pick<float, __nv_bfloat16>(a, s) : bwd_pick<float, float>(a, s);
}

cudaError_t launch_dq_convert(const BwdArgs& a, cudaStream_t s, int* launches) {
  ++*launches;
  const size_t n = static_cast<size_t>(a.cu ? 1 : a.B) * a.Lq * a.Hq * a.D;
  const unsigned blocks = static_cast<unsigned>(std::min<size_t>((n + 255) / 256, 152u * 16u));
  if (a.grad_dt == kBF16) dq_convert_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(a);
  else dq_convert_kernel<float><<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode_simt(const DecArgs& a, cudaStream_t s, int* launches) {
  ++*launches;
  if (a.in_dt == kBF16) return a.D == 64 ? dec_go<__nv_bfloat16, 64>(a, s) : dec_go<__nv_bfloat16, 128>(a, s);
  return a.D == 64 ? dec_go<float, 64>(a, s) : dec_go<float, 128>(a, s);
}

cudaError_t launch_decode_merge(const DecArgs& a, cudaStream_t s, int* launches) {
  ++*launches;
  dim3 grid(a.Hq, a.B);
  if (a.out_dt == kBF16) decode_merge_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(a);
  else decode_merge_kernel<float><<<grid, 128, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace mala
