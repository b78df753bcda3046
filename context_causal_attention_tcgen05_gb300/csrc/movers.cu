// Data-movement kernels of the hot path: the zigzag (DUAL_CHUNK_SWAP) and
// striped reorders and their inverses, and the Ulysses sequence<->head
// exchange, which on one GPU is a layout permute rather than an all-to-all.
//
// Sources: handbook chapter "Context parallelism: Ring Attention and Ulysses",
// sections "Ulysses: transposing between the sequence and the heads"
// (seq_to_head / head_to_seq) and "The zigzag partition" (rank r holds blocks
// r and 2P-1-r of 2P); MaxText pull request "Add Packing Support for Context
// Parallelism (Ring Attention) #2906" (ReorderStrategy STRIPED, read as
// token-granular round robin: rank r holds positions r, r+P, ...).
//
// Every one of these is a gather of contiguous byte runs: output run u comes
// from input run map(u).  Runs are multiples of 16 bytes, so each thread moves
// 16-byte vectors; consecutive threads cover consecutive output vectors, so
// stores are fully coalesced and loads are coalesced within a run (runs are
// >= 512 bytes at the model shapes).  Loads and stores bypass L1 and are
// marked streaming: every byte is touched exactly once.
#include <string.h>

#include <algorithm>
#include <string>

#include "common.cuh"

namespace cpa {
namespace {

struct GatherParams {
  const int4* x;
  int4* y;
  uint32_t total_vec;  // output vectors
  uint32_t run_vec;    // vectors per run
  uint32_t P;
  uint32_t a;          // kind-specific: zigzag -> P; striped -> S/P; ulysses -> S
  uint32_t b;          // replicated seq2head: Hkv
  int kind;
  uint32_t in_vec;     // input vectors (index checks of debug builds)
  int32_t* err;        // device error word
};

// Several gathers in one launch: blocks [block0[i], block0[i+1]) serve gather i.
struct GatherBatch {
  GatherParams t[kMaxGatherBatch];
  uint32_t block0[kMaxGatherBatch + 1];
  int32_t n;
};

__device__ __forceinline__ uint32_t zigzag_slot_source(uint32_t u, uint32_t P) {
  uint32_t r = u >> 1, j = u & 1;  // slot u = (rank r, half j) <- chunk j ? 2P-1-r : r
  return j ? (2 * P - 1 - r) : r;
}
__device__ __forceinline__ uint32_t zigzag_chunk_source(uint32_t c, uint32_t P) {
  return c < P ? 2 * c : 2 * (2 * P - 1 - c) + 1;  // chunk c <- its (rank, half) slot
}

__device__ __forceinline__ uint32_t source_run(const GatherParams& p, uint32_t u) {
  switch (p.kind) {
    case kZigzagReorder:  // out run u = (rank r = u/2, half j = u%2) <- chunk j ? 2P-1-r : r
      return zigzag_slot_source(u, p.P);
    case kZigzagRestore:  // out run = chunk c <- (rank, half) slot
      return zigzag_chunk_source(u, p.P);
    case kZigzagReorderCols:  // lse [H, S]: run u = (head h, slot) of 2P per head row
    case kZigzagRestoreCols: {
      uint32_t h = u / (2 * p.P), c = u - h * 2 * p.P;
      return h * 2 * p.P +
             (p.kind == kZigzagReorderCols ? zigzag_slot_source(c, p.P) : zigzag_chunk_source(c, p.P));
    }
    case kStripedReorder: {  // out row u = r*(S/P) + i <- in row i*P + r
      uint32_t r = u / p.a, i = u - r * p.a;
      return i * p.P + r;
    }
    case kStripedRestore: {  // out row u = i*P + r <- in row r*(S/P) + i
      uint32_t i = u / p.P, r = u - i * p.P;
      return r * p.a + i;
    }
    case kSeq2Head: {  // out run u = rank p*S + s <- in run s*P + p  (run = H/P heads)
      uint32_t rank = u / p.a, s = u - rank * p.a;
      return s * p.P + rank;
    }
    case kSeq2HeadRep: {  // out run u = rank p*S + s <- in run s*Hkv + p/(P/Hkv)  (run = one head)
      uint32_t rank = u / p.a, s = u - rank * p.a;
      return s * p.b + rank / (p.P / p.b);
    }
    default: {  // kHead2Seq: out run u = s*P + p <- in run p*S + s
      uint32_t s = u / p.P, rank = u - s * p.P;
      return rank * p.a + s;
    }
  }
}

constexpr int kThreads = 256;
constexpr int kVecPerThread = 4;

__global__ void __launch_bounds__(kThreads) row_gather_kernel(const __grid_constant__ GatherBatch bt) {
  int ti = 0;
  while (ti + 1 < bt.n && blockIdx.x >= bt.block0[ti + 1]) ++ti;
  const GatherParams& p = bt.t[ti];
  uint32_t base = (blockIdx.x - bt.block0[ti]) * (kThreads * kVecPerThread) + threadIdx.x;
  int4 buf[kVecPerThread];
  uint32_t dst[kVecPerThread];
#pragma unroll
  for (int k = 0; k < kVecPerThread; ++k) {
    uint32_t i = base + k * kThreads;
    dst[k] = i;
    if (i < p.total_vec) {
      uint32_t u = i / p.run_vec;
      uint32_t w = i - u * p.run_vec;
      uint64_t src = (uint64_t)source_run(p, u) * p.run_vec + w;
      if (CP_DCHECK(src < p.in_vec, p.err))
        buf[k] = __ldcs(p.x + src);
      else
        dst[k] = 0xffffffffu;  // debug builds: out-of-range source, nothing stored
    }
  }
#pragma unroll
  for (int k = 0; k < kVecPerThread; ++k)
    if (dst[k] < p.total_vec) __stcs(p.y + dst[k], buf[k]);
}

// lse [H, S] column permute with the row maps above (runs of one column).
struct LsePermParams {
  const float* x;
  float* y;
  uint32_t S, P, H, C;
  int kind;
  int32_t* err;  // device error word (index checks of debug builds)
};

__device__ __forceinline__ uint32_t lse_source_col(const LsePermParams& p, uint32_t col) {
  switch (p.kind) {
    case kZigzagReorder: {  // col = r*2C + j*C + c
      uint32_t r = col / (2 * p.C), rem = col - r * 2 * p.C, j = rem / p.C, c = rem - j * p.C;
      uint32_t chunk = j ? (2 * p.P - 1 - r) : r;
      return chunk * p.C + c;
    }
    case kZigzagRestore: {  // col = chunk*C + c
      uint32_t chunk = col / p.C, c = col - chunk * p.C;
      uint32_t slot = chunk < p.P ? 2 * chunk : 2 * (2 * p.P - 1 - chunk) + 1;
      return slot * p.C + c;
    }
    case kStripedReorder: {  // col = r*(S/P) + i <- i*P + r
      uint32_t n = p.S / p.P, r = col / n, i = col - r * n;
      return i * p.P + r;
    }
    default: {  // kStripedRestore: col = i*P + r <- r*(S/P) + i
      uint32_t n = p.S / p.P, i = col / p.P, r = col - i * p.P;
      return r * n + i;
    }
  }
}

__global__ void __launch_bounds__(256) lse_permute_kernel(LsePermParams p) {
  uint64_t total = (uint64_t)p.S * p.H;
  for (uint64_t t = blockIdx.x * 256ull + threadIdx.x; t < total; t += (uint64_t)gridDim.x * 256) {
    uint32_t h = (uint32_t)(t / p.S), col = (uint32_t)(t - (uint64_t)h * p.S);
    const uint32_t sc = lse_source_col(p, col);
    if (CP_DCHECK(sc < p.S, p.err)) p.y[t] = p.x[(uint64_t)h * p.S + sc];
  }
}

// lse-shaped [H, S] fp32 -> the Ulysses head-major order [H/P][P*S]: rank p's
// heads h' = 0..H/P-1 become heads of one P*S-row problem (row p*S + s).
__global__ void __launch_bounds__(256) lse_heads_kernel(const float* x, float* y, uint32_t S, uint32_t P,
                                                        uint32_t Hp, uint64_t total, int32_t* err) {
  for (uint64_t t = blockIdx.x * 256ull + threadIdx.x; t < total; t += (uint64_t)gridDim.x * 256) {
    const uint64_t PS = (uint64_t)P * S;
    const uint32_t hp = (uint32_t)(t / PS);
    const uint64_t rem = t - (uint64_t)hp * PS;
    const uint32_t rank = (uint32_t)(rem / S), s = (uint32_t)(rem - (uint64_t)rank * S);
    const uint64_t src = ((uint64_t)rank * Hp + hp) * S + s;
    if (CP_DCHECK(src < total, err)) y[t] = x[src];
  }
}

// fp32 gradients in the Ulysses layout [P][S][Hp][D] -> [S][Hd][D] in the output
// dtype, summing the R = P*Hp/Hd consecutive copies of each destination head
// (R = 1 without replication).  One thread per 16-byte output vector.
template <bool kBf16>
__global__ void __launch_bounds__(256) heads_to_seq_sum_kernel(const float* src, void* dst, uint32_t S,
                                                               uint32_t Hd, uint32_t R, uint32_t Hp,
                                                               uint32_t D, uint64_t total_vec, uint64_t src_elems,
                                                               int32_t* err) {
  constexpr uint32_t kEpv = kBf16 ? 8 : 4;  // elements per 16-byte output vector
  const uint32_t vpr = D / kEpv;            // vectors per head row
  for (uint64_t t = blockIdx.x * 256ull + threadIdx.x; t < total_vec; t += (uint64_t)gridDim.x * 256) {
    const uint64_t row = t / vpr;  // s * Hd + hd
    const uint32_t dv = (uint32_t)(t - row * vpr);
    const uint32_t s = (uint32_t)(row / Hd), hd = (uint32_t)(row - (uint64_t)s * Hd);
    float acc[kEpv];
#pragma unroll
    for (uint32_t e = 0; e < kEpv; ++e) acc[e] = 0.f;
    for (uint32_t r = 0; r < R; ++r) {
      const uint32_t g = hd * R + r, rank = g / Hp, hp = g - rank * Hp;
      const uint64_t off = (((uint64_t)rank * S + s) * Hp + hp) * D + (uint64_t)dv * kEpv;
      if (!CP_DCHECK(off + kEpv <= src_elems, err)) continue;
      const float4* sp = reinterpret_cast<const float4*>(src + off);
#pragma unroll
      for (uint32_t e = 0; e < kEpv / 4; ++e) {
        const float4 f = __ldcs(sp + e);
        acc[4 * e] += f.x;
        acc[4 * e + 1] += f.y;
        acc[4 * e + 2] += f.z;
        acc[4 * e + 3] += f.w;
      }
    }
    if (kBf16) {
      uint4 o;
      __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
      for (int e = 0; e < 4; ++e) o2[e] = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
      __stcs(reinterpret_cast<uint4*>(dst) + t, o);
    } else {
      __stcs(reinterpret_cast<float4*>(dst) + t, make_float4(acc[0], acc[1], acc[2], acc[3]));
    }
  }
}

// One launch for n gathers (n <= kMaxGatherBatch), blocks split by output size.
cp_status launch_gathers(const GatherParams* ps, int n, cudaStream_t st, const char* what) {
  GatherBatch bt;
  memset(&bt, 0, sizeof(bt));
  const uint32_t per_block = kThreads * kVecPerThread;
  uint64_t blocks = 0;
  int m = 0;
  for (int i = 0; i < n; ++i) {
    if (ps[i].total_vec == 0) continue;
    bt.t[m] = ps[i];
    bt.block0[m] = (uint32_t)blocks;
    blocks += (ps[i].total_vec + per_block - 1) / per_block;
    ++m;
  }
  if (m == 0) return CP_OK;
  if (blocks >= (1ull << 31)) {
    set_last_error("permute launch too large");
    return CP_ERR_UNSUPPORTED;
  }
  bt.block0[m] = (uint32_t)blocks;
  bt.n = m;
  row_gather_kernel<<<(uint32_t)blocks, kThreads, 0, st>>>(bt);
  return cuda_check(cudaGetLastError(), what);
}

// Gather parameters of one job (row maps as in source_run).
cp_status fill_gather(const GatherJob& j, GatherParams& p) {
  p.x = static_cast<const int4*>(j.x);
  p.y = static_cast<int4*>(j.y);
  p.P = (uint32_t)j.P;
  p.b = 0;
  p.kind = j.kind;
  p.err = device_error_word();
  uint64_t total_bytes = (uint64_t)j.S * (uint64_t)j.row_bytes;
  uint64_t total_vec = total_bytes / 16;
  if (total_vec >= (1ull << 32)) {
    set_last_error("tensor larger than 64 GiB is not supported by the permute kernels");
    return CP_ERR_UNSUPPORTED;
  }
  p.total_vec = (uint32_t)total_vec;
  p.in_vec = (uint32_t)total_vec;  // the maps are permutations
  switch (j.kind) {
    case kZigzagReorder:
    case kZigzagRestore:
      p.run_vec = (uint32_t)(total_vec / (2 * (uint64_t)j.P));
      p.a = (uint32_t)j.P;
      break;
    case kZigzagReorderCols:  // S = heads, row_bytes = one lse row; 2P runs per row
    case kZigzagRestoreCols:
      p.run_vec = (uint32_t)(j.row_bytes / (2 * j.P) / 16);
      p.a = (uint32_t)j.P;
      break;
    case kStripedReorder:
    case kStripedRestore:
      p.run_vec = (uint32_t)(j.row_bytes / 16);
      p.a = (uint32_t)(j.S / j.P);
      break;
    default:  // Ulysses: runs of H/P heads
      p.run_vec = (uint32_t)(j.row_bytes / j.P / 16);  // (H/P)*D elements
      p.a = (uint32_t)j.S;
      break;
  }
  return CP_OK;
}

}  // namespace

cp_status launch_row_gather_batch(const GatherJob* jobs, int n, cudaStream_t st) {
  if (n < 1 || n > kMaxGatherBatch) {
    set_last_error("a permute batch holds 1 to " + std::to_string(kMaxGatherBatch) + " tensors");
    return CP_ERR_INVALID_ARG;
  }
  GatherParams ps[kMaxGatherBatch];
  for (int i = 0; i < n; ++i) {
    if (jobs[i].S == 0) {
      ps[i].total_vec = 0;
      continue;
    }
    cp_status r = fill_gather(jobs[i], ps[i]);
    if (r != CP_OK) return r;
  }
  return launch_gathers(ps, n, st, "row_gather_kernel launch");
}

cp_status launch_kv_replicate(const void* x, void* y, int64_t S, int32_t Hkv, int64_t head_bytes,
                              int32_t P, cudaStream_t st) {
  if (S == 0) return CP_OK;
  GatherParams p;
  p.x = static_cast<const int4*>(x);
  p.y = static_cast<int4*>(y);
  p.P = (uint32_t)P;
  p.a = (uint32_t)S;
  p.b = (uint32_t)Hkv;
  p.kind = kSeq2HeadRep;
  p.err = device_error_word();
  p.run_vec = (uint32_t)(head_bytes / 16);
  p.in_vec = (uint32_t)((uint64_t)S * Hkv * p.run_vec);  // each head of the input once
  const uint64_t total_vec = (uint64_t)P * S * p.run_vec;  // every rank's copy
  if (total_vec >= (1ull << 32)) {
    set_last_error("tensor larger than 64 GiB is not supported by the permute kernels");
    return CP_ERR_UNSUPPORTED;
  }
  p.total_vec = (uint32_t)total_vec;
  return launch_gathers(&p, 1, st, "row_gather_kernel launch (replicated seq2head)");
}

cp_status launch_lse_to_heads(const float* x, float* y, int64_t S, int32_t H, int32_t P,
                              cudaStream_t st) {
  if (S == 0 || H == 0) return CP_OK;
  const uint64_t total = (uint64_t)S * H;
  const uint32_t blocks = (uint32_t)std::min<uint64_t>((total + 255) / 256, 152ull * 16);
  lse_heads_kernel<<<blocks, 256, 0, st>>>(x, y, (uint32_t)S, (uint32_t)P, (uint32_t)(H / P), total,
                                           device_error_word());
  return cuda_check(cudaGetLastError(), "lse_heads_kernel launch");
}

cp_status launch_heads_to_seq_sum(const float* src, void* dst, int64_t S, int32_t Hd, int32_t R,
                                  int32_t P, int32_t Hp, int32_t D, int is_bf16, cudaStream_t st) {
  if (S == 0) return CP_OK;
  const uint64_t total_vec = (uint64_t)S * Hd * (D / (is_bf16 ? 8 : 4));
  const uint32_t blocks = (uint32_t)std::min<uint64_t>((total_vec + 255) / 256, 152ull * 32);
  const uint64_t src_elems = (uint64_t)P * S * Hp * D;
  int32_t* err = device_error_word();
  if (is_bf16)
    heads_to_seq_sum_kernel<true><<<blocks, 256, 0, st>>>(src, dst, (uint32_t)S, (uint32_t)Hd, (uint32_t)R,
                                                          (uint32_t)Hp, (uint32_t)D, total_vec, src_elems, err);
  else
    heads_to_seq_sum_kernel<false><<<blocks, 256, 0, st>>>(src, dst, (uint32_t)S, (uint32_t)Hd, (uint32_t)R,
                                                           (uint32_t)Hp, (uint32_t)D, total_vec, src_elems, err);
  return cuda_check(cudaGetLastError(), "heads_to_seq_sum_kernel launch");
}

cp_status launch_row_gather(int kind, const void* x, void* y, int64_t S, int64_t row_bytes,
                            int32_t P, int32_t H_for_ulysses, cudaStream_t st) {
  (void)H_for_ulysses;
  GatherJob j{kind, x, y, S, row_bytes, P};
  return launch_row_gather_batch(&j, 1, st);
}

cp_status launch_lse_permute(int kind, const float* x, float* y, int64_t S, int32_t H, int32_t P,
                             cudaStream_t st) {
  if (S == 0 || H == 0) return CP_OK;
  LsePermParams p;
  p.x = x;
  p.y = y;
  p.S = (uint32_t)S;
  p.P = (uint32_t)P;
  p.H = (uint32_t)H;
  p.C = (kind == kZigzagReorder || kind == kZigzagRestore) ? (uint32_t)(S / (2 * P)) : 0;
  p.kind = kind;
  p.err = device_error_word();
  uint64_t total = (uint64_t)S * H;
  uint32_t blocks = (uint32_t)std::min<uint64_t>((total + 255) / 256, 152ull * 16);
  lse_permute_kernel<<<blocks, 256, 0, st>>>(p);
  return cuda_check(cudaGetLastError(), "lse_permute_kernel launch");
}

}  // namespace cpa
