// Block attention backward that allocates no device memory: a variant of
// cp_attn_block_bwd_typed whose scratch (the fp32 dQ/dK/dV accumulators and the
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
  // The rules of the workspace form come first (S*H < 2^31 bounds every size below,
  // so the scratch layout cannot wrap around).
  cp_mask m;
  cp_status st = check_block_args(Sq, Sk, Hq, Hkv, D, dtype, mask, &m);
  if (st != CP_OK) return st;
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
                   std::to_string(kScratchBytes) + " bytes (use cp_attn_block_bwd_typed with a workspace)");
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
  st = scratch_address(&base);
  if (st != CP_OK) return st;
  char* b = static_cast<char*>(base);
  // The typed form: the scratch's fp32 accumulators are cleared (or unused) by the run
  // itself, so nothing a previous call left in the array reaches this call's result.
  BlockBwdOut o;
  o.typed = true;
  o.dq = dq;
  o.dk = dk;
  o.dv = dv;
  o.dq_acc = reinterpret_cast<float*>(b + off_dq);
  o.dk_acc = reinterpret_cast<float*>(b + off_dk);
  o.dv_acc = reinterpret_cast<float*>(b + off_dv);
  o.accumulate = 0;
  return block_bwd_run(q, k, v, out, dout, lse, Sq, Sk, Hq, Hkv, D, dtype, m, scale, o,
                       reinterpret_cast<float*>(b + off_delta), (cudaStream_t)stream);
}
