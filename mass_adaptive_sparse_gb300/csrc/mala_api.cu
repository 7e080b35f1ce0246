// C ABI of libmala.so (declarations and contracts in include/mala.h):
// argument validation, workspace layout, kernel selection, device status word.

#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>

#include "../../include/mala.h"
#include "mala_internal.h"

namespace {

using namespace mala;

// Set by kernels whose bounded waits expire; read and cleared by mala_device_status.
__device__ int g_device_status = 0;

std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_inject_next{0};         // one-shot failure-detection test hook
thread_local int g_last_cuda_error = 0;   // cudaError_t of this thread's last MALA_ERR_CUDA

constexpr int kMaxDevices = 64;

// Device address of a __device__ symbol on the current device, looked up once
// per device and cached (the host-side name is only a stand-in).  Concurrent
// first calls from several host threads store the same address; the slots
// are atomic, so that is well defined.
template <typename T, typename Sym>
T* symbol_address(std::atomic<T*> (&cache)[kMaxDevices], const Sym& sym) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  T* p = cache[dev].load(std::memory_order_relaxed);
  if (p == nullptr) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, sym) != cudaSuccess) return nullptr;
    p = static_cast<T*>(addr);
    cache[dev].store(p, std::memory_order_relaxed);
  }
  return p;
}

int* status_word() {
  static std::atomic<int*> cache[kMaxDevices] = {};
  return symbol_address(cache, g_device_status);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool ok_dtype(int d) { return d == MALA_BF16 || d == MALA_FP32; }
size_t round256(size_t x) { return (x + 255) / 256 * 256; }

mala_status finish(cudaError_t e, int launches) {
  g_launches.fetch_add(static_cast<uint64_t>(launches), std::memory_order_relaxed);
  if (e != cudaSuccess) g_last_cuda_error = static_cast<int>(e);
  return e == cudaSuccess ? MALA_OK : MALA_ERR_CUDA;
}

// Common shape checks of the prefill calls.
mala_status check_prefill(int batch, int seqlen_q, int seqlen_k, int heads_q, int heads_kv,
                          int head_dim, int in_dt, int out_dt, int causal, int block_q,
                          int block_k, float tau, float scale) {
  if (batch < 1 || seqlen_q < 1 || seqlen_k < 1 || heads_q < 1 || heads_kv < 1) return MALA_ERR_INVALID_ARG;
  if (batch > 65535 || heads_q > 65535 || heads_q % heads_kv != 0) return MALA_ERR_INVALID_ARG;
  if (!ok_dtype(in_dt) || !ok_dtype(out_dt)) return MALA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return MALA_ERR_INVALID_ARG;
  if (causal == 1 && seqlen_q != seqlen_k) return MALA_ERR_INVALID_ARG;
  if (!(tau >= 0.f) || !std::isfinite(tau)) return MALA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return MALA_ERR_INVALID_ARG;
  if (block_q < 1 || block_k < 1) return MALA_ERR_INVALID_ARG;
  if (head_dim < 1) return MALA_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return MALA_ERR_UNSUPPORTED;
  if (block_q != block_k || (block_q != 64 && block_q != 128)) return MALA_ERR_UNSUPPORTED;
  // the kernels number their CTAs (batch x heads x tile rows or columns) with 32-bit ints
  const int64_t tiles = (static_cast<int64_t>(seqlen_q > seqlen_k ? seqlen_q : seqlen_k) + block_q - 1) / block_q;
  if (static_cast<int64_t>(batch) * heads_q * tiles > INT32_MAX) return MALA_ERR_UNSUPPORTED;
  return MALA_OK;
}

struct BwdLayout {
  size_t delta = 0, dq_acc = 0, scratch = 0, total = 0;
};

// Scratch of mala_decode_noalloc: the per-split (m, l, u) records, at most
// kNoAllocDecodeFloats floats (4 MiB).  Every device that loads the library
// holds one copy until the process exits.
constexpr size_t kNoAllocDecodeFloats = size_t(1) << 20;
__device__ __align__(256) float g_decode_scratch[kNoAllocDecodeFloats];

// Device address of g_decode_scratch on the current device, looked up once per
// device (the host-side name is only a stand-in, not a device address).
float* decode_scratch() {
  static std::atomic<float*> cache[kMaxDevices] = {};
  return symbol_address(cache, g_decode_scratch);
}

// Workspace: D [B, Hq, Lq] fp32 | dQ accumulator fp32 (bf16 gradients only) |
// fp16 operand copies (tensor-core path: bf16 inputs, head_dim 128).
BwdLayout bwd_layout(int batch, int seqlen_q, int seqlen_k, int heads_q, int heads_kv, int head_dim,
                     int in_dt, int grad_dt) {
  BwdLayout w;
  const size_t rows = static_cast<size_t>(batch) * seqlen_q * heads_q;
  w.delta = 0;
  size_t off = round256(rows * sizeof(float));
  w.dq_acc = off;
  if (grad_dt == MALA_BF16) off += round256(rows * head_dim * sizeof(float));
  w.scratch = off;
  if (in_dt == MALA_BF16 && head_dim == 128)
    off += round256(bwd_tc_scratch_bytes(batch, seqlen_q, seqlen_k, heads_q, heads_kv, head_dim));
  w.total = off;
  return w;
}

// Argument checks shared by the decode entry points (workspace excepted).
mala_status check_decode(const void* q, const void* k_cache, const void* v_cache, const void* o,
                         const float* lse, int batch, int cache_len, int heads_q, int heads_kv,
                         int head_dim, int in_dtype, int out_dtype, int block_k, int num_splits,
                         float tau, float softmax_scale) {
  const void* ptrs[] = {q, k_cache, v_cache, o, lse};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return MALA_ERR_INVALID_ARG;
  if (batch < 1 || cache_len < 1 || heads_q < 1 || heads_kv < 1 || heads_q % heads_kv != 0)
    return MALA_ERR_INVALID_ARG;
  if (batch > 65535 || heads_kv > 65535) return MALA_ERR_INVALID_ARG;
  if (!ok_dtype(in_dtype) || !ok_dtype(out_dtype)) return MALA_ERR_INVALID_ARG;
  if (!(tau >= 0.f) || !std::isfinite(tau)) return MALA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return MALA_ERR_INVALID_ARG;
  if (num_splits < 1 || num_splits > 256 || block_k < 1 || head_dim < 1) return MALA_ERR_INVALID_ARG;
  const int g = heads_q / heads_kv;
  if (g != 1 && g != 2 && g != 4 && g != 8) return MALA_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return MALA_ERR_UNSUPPORTED;
  if (block_k != 64 && block_k != 128) return MALA_ERR_UNSUPPORTED;
  return MALA_OK;
}

// Split kernel (tensor-core or CUDA-core) then the exact merge.
mala_status run_decode(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                       const int32_t* cache_lens, int batch, int cache_len, int heads_q, int heads_kv,
                       int head_dim, int in_dtype, int out_dtype, int block_k, int num_splits, float tau,
                       float softmax_scale, float* partial, int32_t* retained_counts, uint8_t* tile_mask,
                       int* status, void* stream, int per_head = 0) {
  DecArgs a{};
  a.q = q; a.k = k_cache; a.v = v_cache; a.o = o; a.lse = lse;
  a.B = batch; a.N = cache_len; a.Hq = heads_q; a.Hkv = heads_kv; a.D = head_dim;
  a.lens = cache_lens;
  a.in_dt = in_dtype; a.out_dt = out_dtype; a.blk = block_k; a.splits = num_splits;
  a.tau = tau; a.log2_tau = tau > 0.f ? std::log2(tau) : 0.f;
  a.scale_log2 = softmax_scale * kLog2e;
  a.partial = partial;
  a.per_head = per_head;
  a.counts = retained_counts; a.mask = tile_mask; a.status = status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int launches = 0;
  cudaError_t e = decode_mma_supported(a) ? launch_decode_mma(a, s, &launches) : launch_decode_simt(a, s, &launches);
  if (e == cudaSuccess) e = launch_decode_merge(a, s, &launches);
  return finish(e, launches);
}

bool workspace_ok(const void* workspace, size_t workspace_bytes, size_t need) {
  return workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0 && workspace_bytes >= need;
}

// Forward of B sequences of Lq / Lk rows (cu == null) or of a packed batch
// (cu != null, Lq = Lk = total rows, each sequence at most Lmax long).
mala_status run_fwd(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* cu,
                    int batch, int seqlen_q, int seqlen_k, int lmax, int heads_q, int heads_kv, int head_dim,
                    int in_dtype, int out_dtype, int causal, int block_q, int block_k, float tau,
                    float softmax_scale, int32_t* retained_counts, uint8_t* tile_mask, void* stream,
                    const uint8_t* force = nullptr) {
  if (!q || !k || !v || !o || !lse) return MALA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return MALA_ERR_INVALID_ARG;
  mala_status st = check_prefill(batch, seqlen_q, seqlen_k, heads_q, heads_kv, head_dim, in_dtype,
                                 out_dtype, causal, block_q, block_k, tau, softmax_scale);
  if (st != MALA_OK) return st;
  int* status = status_word();
  if (!status) return MALA_ERR_CUDA;
  FwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse;
  a.B = batch; a.Lq = seqlen_q; a.Lk = seqlen_k; a.Hq = heads_q; a.Hkv = heads_kv; a.D = head_dim;
  a.cu = cu; a.Lmax = lmax;
  a.in_dt = in_dtype; a.out_dt = out_dtype; a.causal = causal; a.blk = block_q;
  a.tau = tau; a.log2_tau = tau > 0.f ? std::log2(tau) : 0.f;
  a.scale_log2 = softmax_scale * kLog2e;
  a.counts = retained_counts; a.mask = tile_mask; a.status = status;
  a.force = force;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int launches = 0;
  // forced decisions run on the CUDA-core kernel (an evaluation path)
  const bool tc = force == nullptr && fwd_tc_supported(a);
  if (tc) a.inject = g_inject_next.exchange(0);
  cudaError_t e = tc ? launch_fwd_tc(a, s, &launches) : launch_fwd_simt(a, s, &launches);
  return finish(e, launches);
}

// Host-side checks of a packed batch (the bounds themselves are checked on the device).
bool check_packed(const int32_t* cu, int batch, int total, int lmax) {
  return cu && (reinterpret_cast<uintptr_t>(cu) & 3u) == 0 && batch >= 1 && total >= 1 && lmax >= 1 &&
         lmax <= total;
}

// Backward of B sequences of Lq / Lk rows (cu == null) or of a packed batch
// (cu != null, Lq = Lk = total rows, each sequence at most Lmax long).
mala_status run_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                    void* dq, void* dk, void* dv, const int32_t* cu, int batch, int seqlen_q, int seqlen_k,
                    int lmax, int heads_q, int heads_kv, int head_dim, int in_dtype, int grad_dtype, int causal,
                    int block_q, int block_k, float tau, float softmax_scale, void* workspace,
                    size_t workspace_bytes, int32_t* retained_counts, uint8_t* tile_mask, void* stream) {
  const void* ptrs[] = {q, k, v, o, dout, lse, dq, dk, dv};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return MALA_ERR_INVALID_ARG;
  mala_status st = check_prefill(batch, seqlen_q, seqlen_k, heads_q, heads_kv, head_dim, in_dtype,
                                 grad_dtype, causal, block_q, block_k, tau, softmax_scale);
  if (st != MALA_OK) return st;
  // a packed batch is laid out as one run of seqlen_q = seqlen_k = total rows
  const BwdLayout w = bwd_layout(cu ? 1 : batch, seqlen_q, seqlen_k, heads_q, heads_kv, head_dim, in_dtype,
                                 grad_dtype);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < w.total)
    return MALA_ERR_WORKSPACE;
  int* status = status_word();
  if (!status) return MALA_ERR_CUDA;
  char* ws = static_cast<char*>(workspace);
  BwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.o = o; a.dout = dout; a.lse = lse; a.dq = dq; a.dk = dk; a.dv = dv;
  a.B = batch; a.Lq = seqlen_q; a.Lk = seqlen_k; a.Hq = heads_q; a.Hkv = heads_kv; a.D = head_dim;
  a.cu = cu; a.Lmax = lmax;
  a.in_dt = in_dtype; a.grad_dt = grad_dtype; a.causal = causal; a.blk = block_q;
  a.tau = tau; a.log2_tau = tau > 0.f ? std::log2(tau) : 0.f;
  a.scale_log2 = softmax_scale * kLog2e; a.scale = softmax_scale;
  a.delta = reinterpret_cast<float*>(ws + w.delta);
  a.dq_acc = grad_dtype == MALA_FP32 ? static_cast<float*>(dq) : reinterpret_cast<float*>(ws + w.dq_acc);
  a.scratch = ws + w.scratch;
  a.counts = retained_counts; a.mask = tile_mask; a.status = status;
  const bool tc = bwd_tc_supported(a);
  if (!tc && bwd_simt_smem(in_dtype, head_dim, block_q) > 227u * 1024u) return MALA_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int launches = 0;
  cudaError_t e = cudaSuccess;
  if (tc) {
    e = launch_bwd_tc(a, s, &launches);
  } else {
    e = launch_bwd_preprocess(a, s, &launches);
    if (e == cudaSuccess) e = launch_bwd_simt(a, s, &launches);
  }
  if (e == cudaSuccess && grad_dtype == MALA_BF16) e = launch_dq_convert(a, s, &launches);
  return finish(e, launches);
}

}  // namespace

extern "C" {

const char* mala_status_string(mala_status status) {
  switch (status) {
    case MALA_OK: return "MALA_OK";
    case MALA_ERR_INVALID_ARG: return "MALA_ERR_INVALID_ARG";
    case MALA_ERR_UNSUPPORTED: return "MALA_ERR_UNSUPPORTED";
    case MALA_ERR_WORKSPACE: return "MALA_ERR_WORKSPACE";
    case MALA_ERR_CUDA: return "MALA_ERR_CUDA";
    case MALA_ERR_TIMEOUT: return "MALA_ERR_TIMEOUT";
  }
  return "MALA_ERR_UNKNOWN";
}

mala_status mala_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                     int batch, int seqlen_q, int seqlen_k, int heads_q, int heads_kv,
                     int head_dim, mala_dtype in_dtype, mala_dtype out_dtype, int causal,
                     int block_q, int block_k, float tau, float softmax_scale,
                     int32_t* retained_counts, uint8_t* tile_mask, void* stream) {
  return run_fwd(q, k, v, o, lse, nullptr, batch, seqlen_q, seqlen_k, seqlen_q, heads_q, heads_kv, head_dim,
                 in_dtype, out_dtype, causal, block_q, block_k, tau, softmax_scale, retained_counts, tile_mask,
                 stream);
}

mala_status mala_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int32_t* cu_seqlens, int batch, int total_tokens, int max_seqlen,
                            int heads_q, int heads_kv, int head_dim, mala_dtype in_dtype,
                            mala_dtype out_dtype, int causal, int block_q, int block_k, float tau,
                            float softmax_scale, int32_t* retained_counts, uint8_t* tile_mask,
                            void* stream) {
  if (!check_packed(cu_seqlens, batch, total_tokens, max_seqlen)) return MALA_ERR_INVALID_ARG;
  return run_fwd(q, k, v, o, lse, cu_seqlens, batch, total_tokens, total_tokens, max_seqlen, heads_q, heads_kv,
                 head_dim, in_dtype, out_dtype, causal, block_q, block_k, tau, softmax_scale, retained_counts,
                 tile_mask, stream);
}

mala_status mala_fwd_forced(const void* q, const void* k, const void* v, void* o, float* lse,
                            int batch, int seqlen_q, int seqlen_k, int heads_q, int heads_kv,
                            int head_dim, mala_dtype in_dtype, mala_dtype out_dtype, int causal,
                            int block_q, int block_k, float softmax_scale, const uint8_t* tile_keep,
                            int32_t* retained_counts, uint8_t* tile_mask, void* stream) {
  if (!tile_keep) return MALA_ERR_INVALID_ARG;
  return run_fwd(q, k, v, o, lse, nullptr, batch, seqlen_q, seqlen_k, seqlen_q, heads_q, heads_kv, head_dim,
                 in_dtype, out_dtype, causal, block_q, block_k, 0.f, softmax_scale, retained_counts, tile_mask,
                 stream, tile_keep);
}

mala_status mala_region_mass(const void* q, const void* k, const float* lse, float* region_mass,
                             int batch, int seqlen_q, int seqlen_k, int heads_q, int heads_kv,
                             int head_dim, mala_dtype in_dtype, int causal, int block_q, int block_k,
                             float softmax_scale, void* stream) {
  if (!q || !k || !lse || !region_mass) return MALA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(region_mass) & 3u))
    return MALA_ERR_INVALID_ARG;
  mala_status st = check_prefill(batch, seqlen_q, seqlen_k, heads_q, heads_kv, head_dim, in_dtype, in_dtype,
                                 causal, block_q, block_k, 0.f, softmax_scale);
  if (st != MALA_OK) return st;
  FwdArgs a{};
  a.q = q; a.k = k; a.lse = const_cast<float*>(lse); a.region_mass = region_mass;
  a.B = batch; a.Lq = seqlen_q; a.Lk = seqlen_k; a.Hq = heads_q; a.Hkv = heads_kv; a.D = head_dim;
  a.Lmax = seqlen_q;
  a.in_dt = in_dtype; a.out_dt = in_dtype; a.causal = causal; a.blk = block_q;
  a.scale_log2 = softmax_scale * kLog2e;
  int launches = 0;
  cudaError_t e = launch_region_mass(a, static_cast<cudaStream_t>(stream), &launches);
  return finish(e, launches);
}

size_t mala_bwd_workspace_size(int batch, int seqlen_q, int seqlen_k, int heads_q, int heads_kv,
                               int head_dim, mala_dtype in_dtype, mala_dtype grad_dtype) {
  if (batch < 1 || seqlen_q < 1 || seqlen_k < 1 || heads_q < 1 || heads_kv < 1 || head_dim < 1) return 0;
  return bwd_layout(batch, seqlen_q, seqlen_k, heads_q, heads_kv, head_dim, in_dtype, grad_dtype).total;
}

mala_status mala_bwd(const void* q, const void* k, const void* v, const void* o,
                     const void* dout, const float* lse, void* dq, void* dk, void* dv,
                     int batch, int seqlen_q, int seqlen_k, int heads_q, int heads_kv,
                     int head_dim, mala_dtype in_dtype, mala_dtype grad_dtype, int causal,
                     int block_q, int block_k, float tau, float softmax_scale,
                     void* workspace, size_t workspace_bytes,
                     int32_t* retained_counts, uint8_t* tile_mask, void* stream) {
  return run_bwd(q, k, v, o, dout, lse, dq, dk, dv, nullptr, batch, seqlen_q, seqlen_k, seqlen_q, heads_q,
                 heads_kv, head_dim, in_dtype, grad_dtype, causal, block_q, block_k, tau, softmax_scale,
                 workspace, workspace_bytes, retained_counts, tile_mask, stream);
}

size_t mala_bwd_varlen_workspace_size(int total_tokens, int heads_q, int heads_kv, int head_dim,
                                      mala_dtype in_dtype, mala_dtype grad_dtype) {
  return mala_bwd_workspace_size(1, total_tokens, total_tokens, heads_q, heads_kv, head_dim, in_dtype, grad_dtype);
}

mala_status mala_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                            const void* dout, const float* lse, void* dq, void* dk, void* dv,
                            const int32_t* cu_seqlens, int batch, int total_tokens, int max_seqlen,
                            int heads_q, int heads_kv, int head_dim, mala_dtype in_dtype,
                            mala_dtype grad_dtype, int causal, int block_q, int block_k, float tau,
                            float softmax_scale, void* workspace, size_t workspace_bytes,
                            int32_t* retained_counts, uint8_t* tile_mask, void* stream) {
  if (!check_packed(cu_seqlens, batch, total_tokens, max_seqlen)) return MALA_ERR_INVALID_ARG;
  return run_bwd(q, k, v, o, dout, lse, dq, dk, dv, cu_seqlens, batch, total_tokens, total_tokens, max_seqlen,
                 heads_q, heads_kv, head_dim, in_dtype, grad_dtype, causal, block_q, block_k, tau, softmax_scale,
                 workspace, workspace_bytes, retained_counts, tile_mask, stream);
}

size_t mala_decode_workspace_size(int batch, int heads_q, int head_dim, int num_splits) {
  if (batch < 1 || heads_q < 1 || head_dim < 1 || num_splits < 1) return 0;
  return round256(static_cast<size_t>(num_splits) * batch * heads_q * (head_dim + 4) * sizeof(float));
}

mala_status mala_decode(const void* q, const void* k_cache, const void* v_cache, void* o,
                        float* lse, int batch, int cache_len, int heads_q, int heads_kv,
                        int head_dim, mala_dtype in_dtype, mala_dtype out_dtype, int block_k,
                        int num_splits, float tau, float softmax_scale,
                        void* workspace, size_t workspace_bytes,
                        int32_t* retained_counts, uint8_t* tile_mask, void* stream) {
  const mala_status c = check_decode(q, k_cache, v_cache, o, lse, batch, cache_len, heads_q, heads_kv, head_dim,
                                     in_dtype, out_dtype, block_k, num_splits, tau, softmax_scale);
  if (c != MALA_OK) return c;
  if (!workspace_ok(workspace, workspace_bytes, mala_decode_workspace_size(batch, heads_q, head_dim, num_splits)))
    return MALA_ERR_WORKSPACE;
  int* status = status_word();
  if (!status) return MALA_ERR_CUDA;
  return run_decode(q, k_cache, v_cache, o, lse, nullptr, batch, cache_len, heads_q, heads_kv, head_dim, in_dtype,
                    out_dtype, block_k, num_splits, tau, softmax_scale, static_cast<float*>(workspace),
                    retained_counts, tile_mask, status, stream);
}

mala_status mala_decode_per_head(const void* q, const void* k_cache, const void* v_cache, void* o,
                                 float* lse, int batch, int cache_len, int heads_q, int heads_kv,
                                 int head_dim, mala_dtype in_dtype, mala_dtype out_dtype, int block_k,
                                 int num_splits, float tau, float softmax_scale,
                                 void* workspace, size_t workspace_bytes,
                                 int32_t* retained_counts, uint8_t* tile_mask, void* stream) {
  const mala_status c = check_decode(q, k_cache, v_cache, o, lse, batch, cache_len, heads_q, heads_kv, head_dim,
                                     in_dtype, out_dtype, block_k, num_splits, tau, softmax_scale);
  if (c != MALA_OK) return c;
  if (!workspace_ok(workspace, workspace_bytes, mala_decode_workspace_size(batch, heads_q, head_dim, num_splits)))
    return MALA_ERR_WORKSPACE;
  int* status = status_word();
  if (!status) return MALA_ERR_CUDA;
  return run_decode(q, k_cache, v_cache, o, lse, nullptr, batch, cache_len, heads_q, heads_kv, head_dim, in_dtype,
                    out_dtype, block_k, num_splits, tau, softmax_scale, static_cast<float*>(workspace),
                    retained_counts, tile_mask, status, stream, /*per_head=*/1);
}

mala_status mala_decode_varlen(const void* q, const void* k_cache, const void* v_cache, void* o,
                               float* lse, const int32_t* cache_lens, int batch, int max_cache_len,
                               int heads_q, int heads_kv, int head_dim, mala_dtype in_dtype,
                               mala_dtype out_dtype, int block_k, int num_splits, float tau,
                               float softmax_scale, void* workspace, size_t workspace_bytes,
                               int32_t* retained_counts, uint8_t* tile_mask, void* stream) {
  if (!cache_lens || (reinterpret_cast<uintptr_t>(cache_lens) & 3u) != 0) return MALA_ERR_INVALID_ARG;
  const mala_status c = check_decode(q, k_cache, v_cache, o, lse, batch, max_cache_len, heads_q, heads_kv,
                                     head_dim, in_dtype, out_dtype, block_k, num_splits, tau, softmax_scale);
  if (c != MALA_OK) return c;
  if (!workspace_ok(workspace, workspace_bytes, mala_decode_workspace_size(batch, heads_q, head_dim, num_splits)))
    return MALA_ERR_WORKSPACE;
  int* status = status_word();
  if (!status) return MALA_ERR_CUDA;
  return run_decode(q, k_cache, v_cache, o, lse, cache_lens, batch, max_cache_len, heads_q, heads_kv, head_dim,
                    in_dtype, out_dtype, block_k, num_splits, tau, softmax_scale, static_cast<float*>(workspace),
                    retained_counts, tile_mask, status, stream);
}

mala_status mala_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, void* o,
                                float* lse, int batch, int cache_len, int heads_q, int heads_kv,
                                int head_dim, mala_dtype in_dtype, mala_dtype out_dtype, int block_k,
                                int num_splits, float tau, float softmax_scale,
                                int32_t* retained_counts, uint8_t* tile_mask, void* stream) {
  const mala_status c = check_decode(q, k_cache, v_cache, o, lse, batch, cache_len, heads_q, heads_kv, head_dim,
                                     in_dtype, out_dtype, block_k, num_splits, tau, softmax_scale);
  if (c != MALA_OK) return c;
  const size_t need = static_cast<size_t>(num_splits) * batch * heads_q * (head_dim + 4);
  if (need > kNoAllocDecodeFloats) return MALA_ERR_WORKSPACE;
  float* scratch = decode_scratch();
  int* status = status_word();
  if (!scratch || !status) return MALA_ERR_CUDA;
  return run_decode(q, k_cache, v_cache, o, lse, nullptr, batch, cache_len, heads_q, heads_kv, head_dim, in_dtype,
                    out_dtype, block_k, num_splits, tau, softmax_scale, scratch, retained_counts, tile_mask,
                    status, stream);
}

size_t mala_decode_noalloc_max_floats(void) { return kNoAllocDecodeFloats; }

mala_status mala_device_status(void* stream, int* device_code) {
  if (!device_code) return MALA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MALA_ERR_CUDA;
  int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_device_status, sizeof(int)) != cudaSuccess) return MALA_ERR_CUDA;
  const int zero = 0;
  if (word != 0 && cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess) return MALA_ERR_CUDA;
  *device_code = word;
  if (word & kStatusWaitTimeout) return MALA_ERR_TIMEOUT;
  return word == 0 ? MALA_OK : MALA_ERR_INVALID_ARG;
}

uint64_t mala_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

void mala_test_drop_next_load(void) { g_inject_next.store(1); }

int mala_last_cuda_error(void) { return g_last_cuda_error; }

const char* mala_cuda_error_string(int code) { return cudaGetErrorString(static_cast<cudaError_t>(code)); }

}  // extern "C"
