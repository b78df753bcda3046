// Block attention backward that allocates nothing: a variant of
// cp_attn_block_bwd whose scratch (the fp32 dQ/dK/dV accumulators and the
// per-row Delta) lives in a fixed array compiled into the library, for callers
// that cannot allocate device memory and cannot hand over a workspace.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it (kScratchBytes) until the process exits.  Host code never
// uses the array's name as an address: the device address is obtained once
// per device with cudaGetSymbolAddress, with that device current, and passed
// to the kernels.  All calls share the array: calls whose work overlaps on the
// GPU (different streams, or different host threads on one device) race on
// it, and the array keeps the last call's contents, so each call clears the
// accumulators that must start at zero before using them.
#include <math.h>
#include <string.h>

#include <mutex>
#include <string>

#include "common.cuh"

namespace cpa {
namespace {

constexpr size_t kScratchBytes = 32ull << 20;  // 32 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {nullptr};

// Device address of the scratch array on the current device (set up on first use).
cp_status scratch_address(void** out) {
  int dev = 0;
  cp_status st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != CP_OK) return st;
  if (dev < 0 || dev >= 64) {
    set_last_error("device index out of range for the built-in scratch table");
    return CP_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    st = cuda_check(cudaGetSymbolAddress(&p, g_noalloc_scratch),
                    "cudaGetSymbolAddress(built-in scratch)");
    if (st != CP_OK) return st;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return CP_OK;
}

size_t al256(size_t x) { return (x + 255) / 256 * 256; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cp_status bad(cp_status code, const std::string& msg) {
  set_last_error(msg);
  return code;
}

}  // namespace
}  // namespace cpa

using namespace cpa;

extern "C" cp_status cp_attn_block_bwd_noalloc(const void* q, const void* k, const void* v,
                                               const void* out, const void* dout, const float* lse,
                                               int64_t Sq, int64_t Sk, int32_t Hq, int32_t Hkv,
                                               int32_t D, int32_t dtype, const cp_mask* mask,
                                               float scale, void* dq, void* dk, void* dv,
                                               void* stream) {
  if (dtype != CP_F32 && dtype != CP_BF16) return bad(CP_ERR_DTYPE, "dtype must be CP_F32 or CP_BF16");
  if (Hq < 1 || Hkv < 1) return bad(CP_ERR_INVALID_ARG, "head counts must be >= 1");
  if (Hq % Hkv != 0) return bad(CP_ERR_SHAPE, "Hq must be a multiple of Hkv");
  if (dtype == CP_F32 && !(D == 16 || D == 32 || D == 64 || D == 128))
    return bad(CP_ERR_SHAPE, "D must be one of 16, 32, 64, 128");
  if (dtype == CP_BF16 && !(D == 64 || D == 128))
    return bad(CP_ERR_DTYPE, "bf16 attention supports D = 64 or 128");
  if (Sq < 0 || Sk < 0) return bad(CP_ERR_INVALID_ARG, "Sq and Sk must be >= 0");
  cp_mask m = {1, 0, 0, 1, 1, nullptr, 0, 0};
  if (mask) m = *mask;
  if (m.q_stride < 1 || m.k_stride < 1) return bad(CP_ERR_INVALID_ARG, "mask strides must be >= 1");
  if (m.window < 0) return bad(CP_ERR_INVALID_ARG, "mask window must be >= 0");
  if (m.window > 0 && !m.causal) return bad(CP_ERR_UNSUPPORTED, "a sliding window needs the causal rule");
  const int64_t qmax = m.q_offset + m.q_stride * (Sq > 0 ? Sq - 1 : 0);
  const int64_t kmax = m.k_offset + m.k_stride * (Sk > 0 ? Sk - 1 : 0);
  if (llabs(m.q_offset) > INT32_MAX || llabs(m.k_offset) > INT32_MAX || llabs(qmax) > INT32_MAX ||
      llabs(kmax) > INT32_MAX)
    return bad(CP_ERR_UNSUPPORTED, "positions must fit in int32");
  if (m.cu_seqlens && m.n_docs < 1) return bad(CP_ERR_INVALID_ARG, "n_docs must be >= 1 with cu_seqlens");
  // Scratch layout: Delta [Hq, Sq] | dQ [Sq, Hq, D] | dK [Sk, Hkv, D] | dV [Sk, Hkv, D], fp32.
  const size_t off_delta = 0;
  const size_t off_dq = off_delta + al256((size_t)Sq * Hq * 4);
  const size_t off_dk = off_dq + al256((size_t)Sq * Hq * D * 4);
  const size_t off_dv = off_dk + al256((size_t)Sk * Hkv * D * 4);
  const size_t need = off_dv + al256((size_t)Sk * Hkv * D * 4);
  if (need > kScratchBytes)
    return bad(CP_ERR_UNSUPPORTED,
               "cp_attn_block_bwd_noalloc needs " + std::to_string(need) +
                   " bytes of scratch for these sizes; the built-in scratch holds " +
                   std::to_string(kScratchBytes) + " bytes (use cp_attn_block_bwd with a workspace)");
  if (Sq == 0 && Sk == 0) return CP_OK;
  const void* must_q[] = {q, out, dout, lse, dq};
  const void* must_k[] = {k, v, dk, dv};
  for (const void* p : must_q)
    if (Sq > 0 && (!p || !aligned16(p))) return bad(p ? CP_ERR_ALIGN : CP_ERR_INVALID_ARG,
                                                    "query-side tensors must be non-NULL and 16-byte aligned");
  for (const void* p : must_k)
    if (Sk > 0 && (!p || !aligned16(p))) return bad(p ? CP_ERR_ALIGN : CP_ERR_INVALID_ARG,
                                                    "key-side tensors must be non-NULL and 16-byte aligned");
  if (scale == 0.f) scale = 1.0f / sqrtf((float)D);

  void* base = nullptr;
  cp_status st = scratch_address(&base);
  if (st != CP_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  char* b = static_cast<char*>(base);
  float* delta = reinterpret_cast<float*>(b + off_delta);
  float* dq_acc = reinterpret_cast<float*>(b + off_dq);
  float* dk_acc = reinterpret_cast<float*>(b + off_dk);
  float* dv_acc = reinterpret_cast<float*>(b + off_dv);
  const int is_bf16 = dtype == CP_BF16;

  // The tensor-core kernels write every gradient row once, in bf16 (no accumulators);
  // otherwise the array keeps the previous call's values: clear the accumulators first.
  const size_t qb = (size_t)Sq * Hq * D * 2, kb = (size_t)Sk * Hkv * D * 2;  // bf16 when direct
  const void* outs[3] = {dq, dk, dv};
  const size_t ob[3] = {qb, kb, kb};
  const void* ins[5] = {q, k, v, dout, lse};
  const size_t ib[5] = {qb, kb, kb, qb, (size_t)Sq * Hq * 4};
  const bool direct = bwd_writes_bf16(dtype, D) && Sq > 0 && Sk > 0 && grads_apart(outs, ob, 3, ins, ib, 5);
  if (!direct) {
    if ((st = launch_zero(dq_acc, (size_t)Sq * Hq * D * 4, s)) != CP_OK) return st;
    if ((st = launch_zero(dk_acc, (size_t)Sk * Hkv * D * 4, s)) != CP_OK) return st;
    if ((st = launch_zero(dv_acc, (size_t)Sk * Hkv * D * 4, s)) != CP_OK) return st;
  }
  if ((st = launch_bwd_preprocess(out, dout, delta, Sq, Hq, D, (int32_t)Sq, is_bf16, s)) != CP_OK)
    return st;

  Schedule sched;  // host stack; the kernels receive it by value
  memset(&sched, 0, sizeof(sched));
  sched.n_groups = 1;
  sched.g[0].q_row0 = 0;  // key-major: the group is the key block
  sched.g[0].nq = (int32_t)Sk;
  sched.g[0].pos_off = (int32_t)m.k_offset;
  sched.g[0].pos_stride = (int32_t)m.k_stride;
  sched.g[0].seg_begin = 0;
  sched.g[0].seg_count = Sq > 0 ? 1 : 0;
  sched.n_segs = sched.g[0].seg_count;
  sched.s[0].k_row0 = 0;  // the segment is the query block
  sched.s[0].nk = (int32_t)Sq;
  sched.s[0].pos_off = (int32_t)m.q_offset;
  sched.s[0].pos_stride = (int32_t)m.q_stride;

  BwdArgs a;
  memset(&a, 0, sizeof(a));
  a.q = q; a.k = k; a.v = v; a.dout = dout; a.lse = lse; a.delta = delta;
  a.dq_acc = dq_acc; a.dk_acc = dk_acc; a.dv_acc = dv_acc;
  a.q_ld = (int64_t)Hq * D; a.k_ld = (int64_t)Hkv * D;
  a.Hq = Hq; a.Hkv = Hkv; a.D = D; a.lse_ld = (int32_t)Sq;
  a.scale = scale; a.scale_log2 = scale * 1.4426950408889634f;
  a.causal = m.causal; a.cu_seqlens = m.cu_seqlens; a.n_docs = m.cu_seqlens ? m.n_docs : 0;
  a.window = m.window;
  a.err = device_error_word();
  if (direct) {
    a.dq_out = dq; a.dk_out = dk; a.dv_out = dv;
  }
  st = bwd_writes_bf16(dtype, D) ? launch_attn_bwd_tc(a, sched, Sq, Sk, s)
                                 : launch_attn_bwd_simt(a, sched, is_bf16, s);
  if (st != CP_OK || direct) return st;
  if ((st = launch_cast_out(dq_acc, dq, Sq * Hq * D, is_bf16, s)) != CP_OK) return st;
  if ((st = launch_cast_out(dk_acc, dk, Sk * Hkv * D, is_bf16, s)) != CP_OK) return st;
  return launch_cast_out(dv_acc, dv, Sk * Hkv * D, is_bf16, s);
}
