// Internal declarations shared by the translation units of libmala.so.
// Host-side argument blocks and the launch functions of every kernel family.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mala {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Element types of the ABI (values match mala_dtype).
enum Dtype : int { kBF16 = 0, kFP32 = 1 };

// Device status word codes (bitwise OR of events).
enum StatusCode : int {
  kStatusWaitTimeout = 1,   // an mbarrier wait ran past its time limit
  kStatusBadLength = 2,     // a variable-length sequence (decode cache length or packed prefill bounds) was invalid
  kStatusFp16Range = 4,     // a finite bf16 input of the tensor-core backward lies beyond fp16's range (|x| > 65504)
  kStatusDebugBounds = 8    // bounds-checked build only: a TMA coordinate or global index out of range (skipped)
};

// Bounds checks of the bounds-checked build (-DMALA_DEBUG): every TMA box
// origin and global index is checked against the extents the host validated;
// a violation sets kStatusDebugBounds and the caller skips the access (a
// skipped load ends in an expired, bounded wait, never a fault).  In the
// release build the checks are constant true and compile away.
#ifdef __CUDACC__
#ifdef MALA_DEBUG
__device__ __forceinline__ bool dbg_ok(bool ok, int* status) {
  if (!ok) atomicOr(status, kStatusDebugBounds);
  return ok;
}
#else
__device__ __forceinline__ bool dbg_ok(bool, int*) { return true; }
#endif
// index < n (a flat global index against its buffer's element count)
__device__ __forceinline__ bool dbg_idx(size_t index, size_t n, int* status) { return dbg_ok(index < n, status); }
// Origin (x, h, row, b) of a TMA box over a [B, rows, H, D] tensor whose
// current sequence spans rows [lo, hi): x a multiple of 8 elements (16 bytes
// of 16-bit data) inside D, h and b in range, row inside [lo, hi) and hi <= rows.
__device__ __forceinline__ bool dbg_box(int x, int h, int row, int b, int D, int H, int lo, int hi, int rows, int B,
                                        int* status) {
  return dbg_ok(x >= 0 && x % 8 == 0 && x < D && h >= 0 && h < H && b >= 0 && b < B && row >= lo && row < hi &&
                hi <= rows, status);
}
#endif

// Prefill calls take either B sequences of Lq query / Lk key rows ([B, L, H, D]
// tensors, cu == null), or B sequences of different lengths packed along one
// token axis of Lq = Lk = total rows ([total, H, D] tensors, lse [Hq, total]),
// sequence b holding rows cu[b] .. cu[b + 1] - 1 and none longer than Lmax.
struct FwdArgs {
  const void* q; const void* k; const void* v; void* o; float* lse;
  int B, Lq, Lk, Hq, Hkv, D;
  const int32_t* cu;    // [B + 1] sequence starts (device) of a packed batch, or null
  int Lmax;             // longest sequence: tile rows of mask / counts and the grid
  int in_dt, out_dt, causal, blk;
  float tau;            // >= 0; 0 = dense
  float log2_tau;       // log2(tau), used only when tau > 0
  float scale_log2;     // softmax_scale * log2(e): scores kept in log2 units
  int32_t* counts;      // [B, Hq, Tr] or null
  uint8_t* mask;        // [B, Hq, Tr, Tc] or null
  int* status;          // device status word
  int inject;           // test hook: CTA (0, 0) drops its first K load (tensor-core kernel)
  const uint8_t* force; // [B, Hq, Tr, Tc] tile decisions to follow instead of the test, or null
                        // (CUDA-core forward only)
  float* region_mass;   // [B, Hq, Tr, Tc] output of the region-mass kernel (lse is then an input)
};

struct BwdArgs {
  const void* q; const void* k; const void* v; const void* o; const void* dout;
  const float* lse; void* dq; void* dk; void* dv;
  int B, Lq, Lk, Hq, Hkv, D;
  const int32_t* cu;    // as FwdArgs
  int Lmax;
  int in_dt, grad_dt, causal, blk;
  float tau, log2_tau, scale_log2, scale;
  float* delta;         // workspace: D_i = rowsum(O * dO)   [B, Hq, Lq]
  float* dq_acc;        // workspace (or dq itself when fp32): fp32 [B, Lq, Hq, D]
  void* scratch;        // workspace: kernel-specific staging (may be null)
  int32_t* counts;      // [B, Hq, Tc] or null
  uint8_t* mask;        // [B, Hq, Tr, Tc] or null
  int* status;
};

struct DecArgs {
  const void* q; const void* k; const void* v; void* o; float* lse;
  int B, N, Hq, Hkv, D;     // N: cache length (the padded length when `lens` is set)
  const int32_t* lens;      // per-sequence cache lengths [B] (device), or null: all N
  int in_dt, out_dt, blk, splits;
  float tau, log2_tau, scale_log2;
  float* partial;       // workspace: [splits, B, Hq, D + 4] = (m, l, l_rounded, 0, u[D]), m in log2 units;
                        // l sums P exactly, l_rounded sums P as rounded for the P V product
  int per_head;         // 0: the KV head's query heads decide together; 1: each query head alone
  int32_t* counts;      // [B, Hkv, splits] ([B, Hq, splits] per head) or null
  uint8_t* mask;        // [B, Hkv, T] ([B, Hq, T] per head) or null
  int* status;
};

#ifdef __CUDACC__
// Sequence b of a prefill call: its query / key lengths, the row of its first
// token and its batch coordinate in the tensors' layout (0 for a packed batch).
// A packed sequence whose bounds are not 0 <= cu[b] <= cu[b + 1] <= total with
// at most Lmax rows raises kStatusBadLength and comes back empty.
struct SeqSpan {
  int Lq, Lk, row0, bc;
};

template <typename Args>
__device__ __forceinline__ SeqSpan seq_span(const Args& a, int b) {
  if (a.cu == nullptr) return {a.Lq, a.Lk, 0, b};
  const int s0 = a.cu[b], s1 = a.cu[b + 1];
  if (s0 < 0 || s1 < s0 || s1 > a.Lq || s1 - s0 > a.Lmax) {
    if (threadIdx.x == 0) atomicOr(a.status, kStatusBadLength);
    return {0, 0, 0, 0};
  }
  return {s1 - s0, s1 - s0, s0, 0};
}

// Cache length of sequence b: N, or lens[b] for a variable-length decode.  A
// length outside [1, N] raises kStatusBadLength and gives 0 (no keys: the
// sequence's output and lse come out NaN).
__device__ __forceinline__ int decode_seq_len(const DecArgs& a, int b) {
  if (a.lens == nullptr) return a.N;
  const int n = a.lens[b];
  if (n < 1 || n > a.N) {
    atomicOr(a.status, kStatusBadLength);
    return 0;
  }
  return n;
}
#endif

// Each launcher returns the first CUDA error and adds its launches to *launches.
cudaError_t launch_fwd_simt(const FwdArgs& a, cudaStream_t s, int* launches);
cudaError_t launch_bwd_simt(const BwdArgs& a, cudaStream_t s, int* launches);
cudaError_t launch_decode_simt(const DecArgs& a, cudaStream_t s, int* launches);
cudaError_t launch_bwd_preprocess(const BwdArgs& a, cudaStream_t s, int* launches);
cudaError_t launch_dq_convert(const BwdArgs& a, cudaStream_t s, int* launches);
cudaError_t launch_decode_merge(const DecArgs& a, cudaStream_t s, int* launches);
// Reference mass of every (query block, key tile) region from the final lse.
cudaError_t launch_region_mass(const FwdArgs& a, cudaStream_t s, int* launches);

// Tensor-core (tcgen05) kernels: bf16 inputs, head_dim 128, 128 x 128 tiles.
bool fwd_tc_supported(const FwdArgs& a);
cudaError_t launch_fwd_tc(const FwdArgs& a, cudaStream_t s, int* launches);
bool bwd_tc_supported(const BwdArgs& a);
// Workspace bytes of the fp16 operand copies the tensor-core backward makes.
size_t bwd_tc_scratch_bytes(int B, int Lq, int Lk, int Hq, int Hkv, int D);
// Preprocess (fp16 copies, D, zeroed dQ accumulator) + main kernel.
cudaError_t launch_bwd_tc(const BwdArgs& a, cudaStream_t s, int* launches);
bool decode_mma_supported(const DecArgs& a);
cudaError_t launch_decode_mma(const DecArgs& a, cudaStream_t s, int* launches);

// Shared-memory bytes the SIMT kernels need (0 = shape not supported).
size_t fwd_simt_smem(int in_dt, int D, int blk);
size_t bwd_simt_smem(int in_dt, int D, int blk);

}  // namespace mala
