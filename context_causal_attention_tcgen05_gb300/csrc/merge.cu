// Log-sum-exp merge of two partial attentions over disjoint key sets.
//
// Handbook chapter "Context parallelism: Ring Attention and Ulysses", section
// "Ring Attention: passing the KV once around a ring": two blocks' results
// combine as lse = log(e^lse1 + e^lse2) and o = o1 e^(lse1-lse) + o2 e^(lse2-lse).
// Here lse is formed as max + log1p(e^(min-max)), which is the same value
// without overflow; a row where both parts are empty (-inf) stays empty.
//
// HBM-bound: per row and head, 3*D elements of o move (two reads, one write)
// and 3 lse floats.  One thread handles one 16-byte vector of o (4 fp32 or 8
// bf16 elements); the D/elements-per-vector threads of one (row, head) are
// lanes of one warp, so the lse of that row is read by all of them before any
// of them writes it (in-place merge is allowed).
#include "common.cuh"

namespace cpa {
namespace {

struct MergeParams {
  const void* o1;
  const float* lse1;
  const void* o2;
  const float* lse2;
  void* o;
  float* lse;
  uint64_t total_vec;
  uint32_t Sq, H, D;
  uint32_t vec_per_row;  // D / elements per vector
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
__global__ void __launch_bounds__(256) lse_merge_kernel(MergeParams p) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  // Every lane of a warp runs the same number of iterations, so __syncwarp is safe.
  const uint64_t warp_base = ((uint64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31u));
  const uint32_t lane = threadIdx.x & 31u;
  for (uint64_t wb = warp_base; wb < p.total_vec; wb += stride) {
    uint64_t v = wb + lane;
    bool active = v < p.total_vec;
    float w1 = 0.f, w2 = 0.f, lnew = -INFINITY;
    uint32_t i = 0, h = 0;
    bool head_lane = false;
    if (active) {
      uint64_t rh = v / p.vec_per_row;  // row*H + head
      head_lane = (v - rh * p.vec_per_row) == 0;
      i = (uint32_t)(rh / p.H);
      h = (uint32_t)(rh - (uint64_t)i * p.H);
      uint64_t li = (uint64_t)h * p.Sq + i;
      merge_weights(p.lse1[li], p.lse2[li], &w1, &w2, &lnew);
    }
    __syncwarp();
    if (active) {
      if (kF32) {
        float4 a = reinterpret_cast<const float4*>(p.o1)[v];
        float4 b = reinterpret_cast<const float4*>(p.o2)[v];
        float4 r;
        r.x = a.x * w1 + b.x * w2;
        r.y = a.y * w1 + b.y * w2;
        r.z = a.z * w1 + b.z * w2;
        r.w = a.w * w1 + b.w * w2;
        reinterpret_cast<float4*>(p.o)[v] = r;
      } else {
        uint4 a = reinterpret_cast<const uint4*>(p.o1)[v];
        uint4 b = reinterpret_cast<const uint4*>(p.o2)[v];
        const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
        uint4 r;
        __nv_bfloat162* r2 = reinterpret_cast<__nv_bfloat162*>(&r);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float2 fa = __bfloat1622float2(a2[k]);
          float2 fb = __bfloat1622float2(b2[k]);
          r2[k] = __floats2bfloat162_rn(fa.x * w1 + fb.x * w2, fa.y * w1 + fb.y * w2);
        }
        reinterpret_cast<uint4*>(p.o)[v] = r;
      }
      if (head_lane) p.lse[(uint64_t)h * p.Sq + i] = lnew;
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
  uint32_t epv = o_f32 ? 4 : 8;
  p.vec_per_row = (uint32_t)D / epv;
  p.total_vec = (uint64_t)Sq * H * p.vec_per_row;
  uint64_t want = (p.total_vec + 255) / 256;
  uint32_t blocks = (uint32_t)(want < 152ull * 32 ? want : 152ull * 32);
  if (o_f32)
    lse_merge_kernel<true><<<blocks, 256, 0, st>>>(p);
  else
    lse_merge_kernel<false><<<blocks, 256, 0, st>>>(p);
  return cuda_check(cudaGetLastError(), "lse_merge_kernel launch");
}

}  // namespace cpa
