// FFMA (non-tensor-core) block attention, forward and backward.
//
// This is the exact-fp32 path (fp32 inputs are not rounded to a narrower
// tensor-core type) and the backward used for fp32.  It computes the
// handbook's attention(q, k, v, causal, q_offset, k_offset) -> (out, lse)
// ("Context parallelism: Ring Attention and Ulysses", section "Which
// operations partition directly") blockwise with an online softmax, over a
// schedule of query groups and key/value segments (see common.cuh).
//
// Forward: one CTA = 4 warps = one tile of 16 query rows of one head.  Key
// and value tiles of 32 rows are staged in shared memory as fp32; lane j of a
// warp scores key j of the tile for one query row, the row's running max and
// sum are warp reductions, and lane d accumulates output columns d, d+32, ...
//
// Backward (exact derivative of the definition; the pages give no backward):
// one CTA = one tile of 32 keys of one key/value head, looping over the G
// query heads that read it and every query row of every query segment that
// sees it.  dK and dV of the tile accumulate in shared memory and are stored
// once (or added to the fp32 outputs in the accumulating form); dQ accumulates
// in an fp32 buffer with atomic adds (zeroed by the caller unless accumulating).
#include <math.h>

#include "common.cuh"
#include "ptx.cuh"

namespace cpa {
namespace {

constexpr int kFwdRows = 16;
constexpr int kKT = 32;  // key tile
constexpr int kMaxD = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <typename T>
__global__ void __launch_bounds__(128) attn_fwd_simt_kernel(AttnArgs a, Schedule s) {
  extern __shared__ float smem[];
  const int D = a.D;
  const int Dp = D + 1;
  float* qs = smem;                  // [16][D]
  float* ks = qs + kFwdRows * D;     // [32][D+1]
  float* vs = ks + kKT * Dp;         // [32][D+1]

  int g, tile, h;
  decode_unit(s, kFwdRows, a.Hq, blockIdx.x, &g, &tile, &h);
  const QGroup grp = s.g[g];
  const int hk = h / (a.Hq / a.Hkv);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  const int i0 = tile * kFwdRows;

  for (int e = threadIdx.x; e < kFwdRows * D; e += 128) {
    int r = e / D, d = e - r * D;
    int i = i0 + r;
    qs[e] = (i < grp.nq && CP_DCHECK((int64_t)grp.q_row0 + i < a.q_rows, a.err))
                ? load_as_f32(q + (int64_t)(grp.q_row0 + i) * a.q_ld + (int64_t)h * D + d)
                : 0.f;
  }

  // Per row state (4 rows per warp).
  float m[4], l[4], acc[4][4];
  int64_t pq[4], dst[4], den[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
    int i = i0 + warp + 4 * r;
    pq[r] = (int64_t)grp.pos_off + (int64_t)grp.pos_stride * i;
    dst[r] = 0;
    den[r] = 0;
    if (a.cu_seqlens && i < grp.nq) doc_bounds(a.cu_seqlens, a.n_docs, pq[r], &dst[r], &den[r]);
  }

  for (int si = 0; si < grp.seg_count; ++si) {
    const KSeg seg = s.s[grp.seg_begin + si];
    for (int j0 = 0; j0 < seg.nk; j0 += kKT) {
      __syncthreads();
      for (int e = threadIdx.x; e < kKT * D; e += 128) {
        int r = e / D, d = e - r * D;
        int j = j0 + r;
        float kv = 0.f, vv = 0.f;
        if (j < seg.nk && CP_DCHECK((int64_t)seg.k_row0 + j < a.k_rows, a.err)) {
          int64_t off = (int64_t)(seg.k_row0 + j) * a.k_ld + (int64_t)hk * D + d;
          kv = load_as_f32(k + off);
          vv = load_as_f32(v + off);
        }
        ks[r * Dp + d] = kv;
        vs[r * Dp + d] = vv;
      }
      __syncthreads();
      const int j = j0 + lane;
      const int64_t pk = (int64_t)seg.pos_off + (int64_t)seg.pos_stride * j;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int row = warp + 4 * r;
        if (i0 + row >= grp.nq) continue;  // warp-uniform
        bool vis = j < seg.nk;
        if (a.causal) vis = vis && (pk <= pq[r]);
        if (a.window > 0) vis = vis && (pq[r] - pk < a.window);
        if (a.cu_seqlens) vis = vis && (pk >= dst[r]) && (pk < den[r]);
        float sc = -INFINITY;
        if (vis) {
          float dot = 0.f;
          for (int d = 0; d < D; ++d) dot = fmaf(qs[row * D + d], ks[lane * Dp + d], dot);
          sc = dot * a.scale_log2;
        }
        float mt = warp_max(sc);
        float mn = fmaxf(m[r], mt);
        if (mn == -INFINITY) continue;  // nothing visible yet for this row
        float alpha = exp2f(m[r] - mn);  // m = -inf -> 0
        float p = vis ? exp2f(sc - mn) : 0.f;
        l[r] = l[r] * alpha + warp_sum(p);
        m[r] = mn;
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] *= alpha;
        for (int jj = 0; jj < kKT; ++jj) {
          float pj = __shfl_sync(0xffffffffu, p, jj);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            int d = lane + 32 * c;
            if (d < D) acc[r][c] = fmaf(pj, vs[jj * Dp + d], acc[r][c]);
          }
        }
      }
    }
  }

  T* o = static_cast<T*>(a.o);
  float* of = static_cast<float*>(a.o);
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    int i = i0 + warp + 4 * r;
    if (i >= grp.nq) continue;
    if (!CP_DCHECK((int64_t)grp.o_row0 + i < a.q_rows, a.err)) continue;
    float inv = l[r] > 0.f ? 1.f / l[r] : 0.f;
    int64_t orow = (int64_t)(grp.o_row0 + i) * a.o_ld + (int64_t)(grp.o_head0 + h) * D;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      int d = lane + 32 * c;
      if (d < D) {
        if (a.o_f32)
          of[orow + d] = acc[r][c] * inv;
        else
          store_from_f32(o + orow + d, acc[r][c] * inv);
      }
    }
    const int64_t li = (int64_t)(grp.lse_head0 + h) * a.lse_ld + grp.lse_col0 + i;
    if (lane == 0 && CP_DCHECK(li < a.lse_size, a.err)) {
      float L = l[r] > 0.f ? (m[r] + log2f(l[r])) * kLn2 : -INFINITY;
      a.lse[li] = L;
    }
  }
}

// Backward: schedule groups are KEY chunks, segments are the query runs that see them.
template <typename T>
__global__ void __launch_bounds__(128) attn_bwd_simt_kernel(BwdArgs a, Schedule s) {
  extern __shared__ float smem[];
  const int D = a.D;
  const int Dp = D + 1;
  float* ks = smem;            // [32][D+1]
  float* vs = ks + kKT * Dp;   // [32][D+1]
  float* dks = vs + kKT * Dp;  // [32][D+1]
  float* dvs = dks + kKT * Dp; // [32][D+1]
  float* qrow = dvs + kKT * Dp;  // [4][D]
  float* dorow = qrow + 4 * D;   // [4][D]

  int g, tile, hk;
  decode_unit(s, kKT, a.Hkv, blockIdx.x, &g, &tile, &hk);
  const QGroup kg = s.g[g];  // key chunk: q_row0/nq/pos_* describe KEY rows here
  const int G = a.Hq / a.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  const T* dout = static_cast<const T*>(a.dout);
  const int j0 = tile * kKT;

  for (int e = threadIdx.x; e < kKT * D; e += 128) {
    int r = e / D, d = e - r * D;
    int j = j0 + r;
    float kv = 0.f, vv = 0.f;
    if (j < kg.nq && CP_DCHECK((int64_t)kg.q_row0 + j < a.k_rows, a.err)) {
      int64_t off = (int64_t)(kg.q_row0 + j) * a.k_ld + (int64_t)hk * D + d;
      kv = load_as_f32(k + off);
      vv = load_as_f32(v + off);
    }
    ks[r * Dp + d] = kv;
    vs[r * Dp + d] = vv;
    dks[r * Dp + d] = 0.f;
    dvs[r * Dp + d] = 0.f;
  }
  __syncthreads();

  const int j = j0 + lane;
  const int64_t pk = (int64_t)kg.pos_off + (int64_t)kg.pos_stride * j;
  float* myq = qrow + warp * D;
  float* mydo = dorow + warp * D;

  for (int hh = 0; hh < G; ++hh) {
    const int h = hk * G + hh;
    for (int si = 0; si < kg.seg_count; ++si) {
      const KSeg qs = s.s[kg.seg_begin + si];  // query run
      for (int i = warp; i < qs.nk; i += 4) {
        const int64_t qrow_idx = (int64_t)(qs.k_row0 + i);
        if (!CP_DCHECK(qrow_idx < a.q_rows && (int64_t)h * a.lse_ld + qrow_idx < a.lse_size, a.err))
          continue;  // warp-uniform
        const int64_t pq = (int64_t)qs.pos_off + (int64_t)qs.pos_stride * i;
        __syncwarp();
        for (int d = lane; d < D; d += 32) {
          myq[d] = load_as_f32(q + qrow_idx * a.q_ld + (int64_t)h * D + d);
          mydo[d] = load_as_f32(dout + qrow_idx * a.q_ld + (int64_t)h * D + d);
        }
        __syncwarp();
        int64_t dst = 0, den = 0;
        if (a.cu_seqlens) doc_bounds(a.cu_seqlens, a.n_docs, pq, &dst, &den);
        bool vis = j < kg.nq;
        if (a.causal) vis = vis && (pk <= pq);
        if (a.window > 0) vis = vis && (pq - pk < a.window);
        if (a.cu_seqlens) vis = vis && (pk >= dst) && (pk < den);
        const float lse = a.lse[(int64_t)h * a.lse_ld + qrow_idx];
        const float delta = a.delta[(int64_t)h * a.lse_ld + qrow_idx];
        float p = 0.f, ds = 0.f;
        if (vis && lse != -INFINITY) {
          float dot = 0.f, dpv = 0.f;
          for (int d = 0; d < D; ++d) {
            dot = fmaf(myq[d], ks[lane * Dp + d], dot);
            dpv = fmaf(mydo[d], vs[lane * Dp + d], dpv);
          }
          p = exp2f(dot * a.scale_log2 - lse * kLog2e);
          ds = p * (dpv - delta);
        }
        if (__any_sync(0xffffffffu, p != 0.f || ds != 0.f)) {
          float dqc[4] = {0.f, 0.f, 0.f, 0.f};
          for (int jj = 0; jj < kKT; ++jj) {
            float pj = __shfl_sync(0xffffffffu, p, jj);
            float dsj = __shfl_sync(0xffffffffu, ds, jj) * a.scale;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              int d = lane + 32 * c;
              if (d < D) {
                dqc[c] = fmaf(dsj, ks[jj * Dp + d], dqc[c]);
                atomicAdd(&dks[jj * Dp + d], dsj * myq[d]);
                atomicAdd(&dvs[jj * Dp + d], pj * mydo[d]);
              }
            }
          }
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            int d = lane + 32 * c;
            if (d < D) atomicAdd(a.dq_acc + qrow_idx * a.q_ld + (int64_t)h * D + d, dqc[c]);
          }
        }
      }
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < kKT * D; e += 128) {
    int r = e / D, d = e - r * D;
    int jj = j0 + r;
    if (jj < kg.nq && CP_DCHECK((int64_t)kg.q_row0 + jj < a.k_rows, a.err)) {
      int64_t off = (int64_t)(kg.q_row0 + jj) * a.k_ld + (int64_t)hk * D + d;
      a.dk_acc[off] = dks[r * Dp + d] + (a.accumulate ? a.dk_acc[off] : 0.f);
      a.dv_acc[off] = dvs[r * Dp + d] + (a.accumulate ? a.dv_acc[off] : 0.f);
    }
  }
}

// delta[h][row] = sum_d dout[row,h,d] * out[row,h,d]  (one warp per (row, head)).
template <typename T>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const T* out, const T* dout,
                                                             float* delta, int64_t rows, int H,
                                                             int D, int lse_ld) {
  int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int lane = threadIdx.x & 31;
  int64_t total = rows * H;
  for (; w < total; w += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    int64_t row = w / H;
    int h = (int)(w - row * H);
    const T* o = out + (row * H + h) * D;
    const T* g = dout + (row * H + h) * D;
    float acc = 0.f;
    for (int d = lane; d < D; d += 32) acc = fmaf(load_as_f32(o + d), load_as_f32(g + d), acc);
    acc = warp_sum(acc);
    if (lane == 0) delta[(int64_t)h * lse_ld + row] = acc;
  }
}

template <typename T>
__global__ void __launch_bounds__(256) cast_kernel(const float* src, T* dst, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    store_from_f32(dst + i, src[i]);
}

__global__ void __launch_bounds__(256) zero_kernel(int4* p, int64_t n16) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
       i += (int64_t)gridDim.x * blockDim.x)
    p[i] = make_int4(0, 0, 0, 0);
}

// One thread waits on a barrier that nothing arrives on, with a limit.
__global__ void bounded_wait_probe_kernel(int32_t* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
    (void)ptx::mbar_wait_bounded(&bar, 0, &abort_flag, err, limit_ns);
  }
}

}  // namespace

cp_status launch_attn_fwd_simt(const AttnArgs& a, Schedule& s, int is_bf16, cudaStream_t st) {
  int64_t units = schedule_units(s, kFwdRows, a.Hq);
  if (units == 0) return CP_OK;
  size_t smem = (size_t)(kFwdRows * a.D + 2 * kKT * (a.D + 1)) * sizeof(float);
  if (is_bf16) {
    cudaFuncSetAttribute(attn_fwd_simt_kernel<__nv_bfloat16>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    attn_fwd_simt_kernel<__nv_bfloat16><<<(unsigned)units, 128, smem, st>>>(a, s);
  } else {
    cudaFuncSetAttribute(attn_fwd_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    attn_fwd_simt_kernel<float><<<(unsigned)units, 128, smem, st>>>(a, s);
  }
  return cuda_check(cudaGetLastError(), "attn_fwd_simt_kernel launch");
}

cp_status launch_attn_bwd_simt(const BwdArgs& a, Schedule& s, int is_bf16, cudaStream_t st) {
  int64_t units = schedule_units(s, kKT, a.Hkv);
  if (units == 0) return CP_OK;
  size_t smem = (size_t)(4 * kKT * (a.D + 1) + 8 * a.D) * sizeof(float);
  if (is_bf16) {
    cudaFuncSetAttribute(attn_bwd_simt_kernel<__nv_bfloat16>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    attn_bwd_simt_kernel<__nv_bfloat16><<<(unsigned)units, 128, smem, st>>>(a, s);
  } else {
    cudaFuncSetAttribute(attn_bwd_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    attn_bwd_simt_kernel<float><<<(unsigned)units, 128, smem, st>>>(a, s);
  }
  return cuda_check(cudaGetLastError(), "attn_bwd_simt_kernel launch");
}

cp_status launch_bwd_preprocess(const void* out, const void* dout, float* delta, int64_t rows,
                                int32_t H, int32_t D, int32_t lse_ld, int is_bf16,
                                cudaStream_t st) {
  if (rows == 0) return CP_OK;
  int64_t warps = rows * H;
  int64_t blocks = (warps * 32 + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  if (is_bf16)
    bwd_preprocess_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout), delta,
        rows, H, D, lse_ld);
  else
    bwd_preprocess_kernel<float><<<(unsigned)blocks, 256, 0, st>>>(
        static_cast<const float*>(out), static_cast<const float*>(dout), delta, rows, H, D,
        lse_ld);
  return cuda_check(cudaGetLastError(), "bwd_preprocess_kernel launch");
}

cp_status launch_cast_out(const float* src, void* dst, int64_t n, int is_bf16, cudaStream_t st) {
  if (n == 0) return CP_OK;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 32) blocks = 152 * 32;
  if (is_bf16)
    cast_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, st>>>(
        src, static_cast<__nv_bfloat16*>(dst), n);
  else
    cast_kernel<float><<<(unsigned)blocks, 256, 0, st>>>(src, static_cast<float*>(dst), n);
  return cuda_check(cudaGetLastError(), "cast_kernel launch");
}

cp_status launch_zero(void* p, size_t bytes, cudaStream_t st) {
  if (bytes == 0) return CP_OK;
  int64_t n16 = (int64_t)(bytes / 16);
  int64_t blocks = (n16 + 255) / 256;
  if (blocks > 152 * 32) blocks = 152 * 32;
  zero_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<int4*>(p), n16);
  return cuda_check(cudaGetLastError(), "zero_kernel launch");
}

cp_status launch_bounded_wait_probe(int32_t timeout_us, int32_t* err, cudaStream_t st) {
  bounded_wait_probe_kernel<<<1, 32, 0, st>>>(err, (uint64_t)timeout_us * 1000ull);
  return cuda_check(cudaGetLastError(), "bounded_wait_probe_kernel launch");
}

}  // namespace cpa
