// Log-sum-exp merge of two partial attentions over disjoint key sets.
//
// Handbook chapter "Context parallelism: Ring Attention and Ulysses", section
// "Ring Attention: passing the KV once around a ring": two blocks' results
// combine as lse = log(e^lse1 + e^lse2) and o = o1 e^(lse1-lse) + o2 e^(lse2-lse).
// Here lse is formed as max + log1p(e^(min-max)), which is the same value
// without overflow; a row where both parts are empty (-inf) stays empty.
//
// HBM-bound: per row and head, 3*D elements of o move (two reads, one write)
// and 3 lse floats.  One block takes a tile of kRows consecutive rows and every
// head: its threads first read the tile's lse values (kRows consecutive floats
// per head, whole 32-byte sectors), form the weights into shared memory and
// write the merged lse; then they stream the tile's o rows, which are one
// contiguous range of kRows*H*D elements, four 16-byte vectors in flight per
// thread (the first four issued before the weights are formed).  Each lse value and each o vector is read and written by the same
// thread, so an in-place merge (o = o1, lse = lse1) is safe.
#include "common.cuh"

namespace cpa {
namespace {

constexpr int kRows = 8;       // rows per block
constexpr int kThreads = 256;
constexpr int kUnroll = 4;     // o vectors in flight per thread

struct MergeParams {
  const void* o1;
  const float* lse1;
  const void* o2;
  const float* lse2;
  void* o;
  float* lse;
  uint32_t Sq, H, D;
  uint32_t vph;  // 16-byte vectors per (row, head): D / elements per vector
};

__device__ __forceinline__ void merge_weights(float l1, float l2, float* w1, float* w2,
                                              float* lnew) {
  float mx = fmaxf(l1, l2), mn = fminf(l1, l2);
  if (mx == -INFINITY) {
    *w1 = 0.f;
    *w2 = 0.f;
    *lnew = -INFINITY;
    return;
  }
  float L = mx + log1pf(expf(mn - mx));
  *w1 = expf(l1 - L);
  *w2 = expf(l2 - L);
  *lnew = L;
}

template <bool kF32>
__device__ __forceinline__ uint4 merge_vec(uint4 a, uint4 b, float2 w) {
  uint4 r;
  if (kF32) {
    r.x = __float_as_uint(__uint_as_float(a.x) * w.x + __uint_as_float(b.x) * w.y);
    r.y = __float_as_uint(__uint_as_float(a.y) * w.x + __uint_as_float(b.y) * w.y);
    r.z = __float_as_uint(__uint_as_float(a.z) * w.x + __uint_as_float(b.z) * w.y);
    r.w = __float_as_uint(__uint_as_float(a.w) * w.x + __uint_as_float(b.w) * w.y);
  } else {
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
    __nv_bfloat162* r2 = reinterpret_cast<__nv_bfloat162*>(&r);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float2 fa = __bfloat1622float2(a2[k]);
      float2 fb = __bfloat1622float2(b2[k]);
      r2[k] = __floats2bfloat162_rn(fa.x * w.x + fb.x * w.y, fa.y * w.x + fb.y * w.y);
    }
  }
  return r;
}

template <bool kF32>
__global__ void __launch_bounds__(kThreads) lse_merge_kernel(MergeParams p) {
  extern __shared__ float2 w_sm[];  // [kRows][H] (w1, w2)
  const uint32_t i0 = blockIdx.x * kRows;
  const uint32_t rows = min((uint32_t)kRows, p.Sq - i0);
  // the tile's o rows: one contiguous range of vectors
  const uint64_t base = (uint64_t)i0 * p.H * p.vph;
  const uint32_t n = rows * p.H * p.vph;
  const uint4* a = reinterpret_cast<const uint4*>(p.o1) + base;
  const uint4* b = reinterpret_cast<const uint4*>(p.o2) + base;
  uint4* o = reinterpret_cast<uint4*>(p.o) + base;
  uint4 va[kUnroll], vb[kUnroll];
  auto load = [&](uint32_t v0) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t v = v0 + u * kThreads;
      if (v < n) {
        va[u] = __ldcs(a + v);
        vb[u] = __ldcs(b + v);
      }
    }
  };
  load(threadIdx.x);  // the first vectors are in flight while the weights are formed
  // weights and merged lse of the tile: thread t takes (head t / kRows, row t % kRows)
  for (uint32_t t = threadIdx.x; t < (uint32_t)kRows * p.H; t += kThreads) {
    const uint32_t h = t / kRows, r = t - h * kRows;
    if (r < rows) {
      const uint64_t li = (uint64_t)h * p.Sq + i0 + r;
      float w1, w2, lnew;
      merge_weights(p.lse1[li], p.lse2[li], &w1, &w2, &lnew);
      w_sm[r * p.H + h] = make_float2(w1, w2);
      p.lse[li] = lnew;
    }
  }
  __syncthreads();
  for (uint32_t v0 = threadIdx.x; v0 < n; v0 += kThreads * kUnroll) {
    if (v0 != threadIdx.x) load(v0);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t v = v0 + u * kThreads;
      if (v < n) __stcs(o + v, merge_vec<kF32>(va[u], vb[u], w_sm[v / p.vph]));
    }
  }
}

}  // namespace

cp_status launch_lse_merge(const void* o1, const float* lse1, const void* o2, const float* lse2,
                           void* o, float* lse, int64_t Sq, int32_t H, int32_t D, int32_t o_f32,
                           cudaStream_t st) {
  if (Sq == 0 || H == 0) return CP_OK;
  MergeParams p;
  p.o1 = o1;
  p.lse1 = lse1;
  p.o2 = o2;
  p.lse2 = lse2;
  p.o = o;
  p.lse = lse;
  p.Sq = (uint32_t)Sq;
  p.H = (uint32_t)H;
  p.D = (uint32_t)D;
  p.vph = (uint32_t)D / (o_f32 ? 4u : 8u);  // a row of one head is a whole number of vectors
  if ((uint64_t)kRows * H * p.vph > 0xffffffffull || (uint64_t)Sq > 0xffffffffull) {
    set_last_error("lse merge: too many rows or heads for one launch");
    return CP_ERR_UNSUPPORTED;
  }
  const size_t smem = (size_t)kRows * H * sizeof(float2);
  if (smem > 48 * 1024) {
    set_last_error("lse merge: too many heads for one block's weight table");
    return CP_ERR_UNSUPPORTED;
  }
  const uint64_t blocks = ((uint64_t)Sq + kRows - 1) / kRows;
  if (blocks > 0x7fffffffull) {
    set_last_error("lse merge: too many rows for one launch");
    return CP_ERR_UNSUPPORTED;
  }
  if (o_f32)
    lse_merge_kernel<true><<<(unsigned)blocks, kThreads, smem, st>>>(p);
  else
    lse_merge_kernel<false><<<(unsigned)blocks, kThreads, smem, st>>>(p);
  return cuda_check(cudaGetLastError(), "lse_merge_kernel launch");
}

}  // namespace cpa
