// tcgen05 block attention backward for bf16 (fp32 accumulation), D = 64 or 128.
//
// The exact derivative of the handbook's attention ("Context parallelism:
// Ring Attention and Ulysses", section "Which operations partition
// directly"; the pages give no backward), given the FINAL out and lse of
// every query row (for a ring: the merged ones):
//   P = exp(scale*S - lse),  dV = P^T dO,  dP = dO V^T,
//   dS = P o (dP - Delta),   Delta = rowsum(dO o O),
//   dQ = scale * dS K,       dK = scale * dS^T Q.
//
// Two kernels, neither uses atomics (gradients are deterministic).  Every
// product is M=128 x N=128 per instruction: a tcgen05.mma costs about the same
// time for N = 64 as for N = 128, so 64-wide tiles would halve the rate.
//
// attn_bwd_dkdv_kernel: one CTA = one 128-key tile of one key/value head
//   (K, V in shared memory), looping over the G query heads that read it and
//   every 128-row query tile that can see the keys (a key-major schedule:
//   group = key run, segments = query runs).  Per query tile j:
//     S^T = K Q^T (TMEM 0..127), dP^T = V dO^T (TMEM 128..255)
//     softmax warps (thread = key row, each warpgroup 64 of the query
//       columns): phase 1 P^T from S^T as soon as S^T lands (written back
//       over S^T, two bf16 per column); phase 2 dS^T once dP^T lands
//     dV += P^T dO (TMEM 256..383), dK += dS^T Q (TMEM 384..511), P^T and dS^T
//       as the TMEM A operand
//   MMA issue order dV_j, S^T_{j+1}, dK_j, dP^T_{j+1}: the tensor pipe always
//   has the next tile's scores queued while the softmax works.  lse and Delta
//   of each query tile are staged with cp.async alongside the Q/dO tiles.
//
// attn_bwd_dq_kernel: one CTA = one 128-row query tile of one query head.  Q and
//   dO are loaded once into shared memory; the CTA walks every 128-key tile it
//   sees (a query-major schedule, as in the forward), K in a 3-stage and V in a
//   2-stage ring:
//     S = Q K^T (TMEM 0..127), dP = dO V^T (TMEM 128..255 for even tiles,
//     384..511 for odd ones)
//     softmax warps (thread = query row, each warpgroup 64 of the key columns):
//       phase 1 P from S (S is released as soon as it is in registers), phase 2
//       dS once dP lands, written over dP in the same buffer
//     dQ += dS K (TMEM 256..383)
//   MMA issue order S_{j+1}, dP_{j+1}, dQ_j: with two dP / dS buffers dP_{j+1}
//   does not wait for dQ_j, so the softmax's second phase of tile j+1 finds its
//   dP ready.
// This recomputes S and dP once more than a single fused kernel (7 instead of
// 5 matrix products) in exchange for no fp32 atomic traffic on dQ.
// Warps: 0..7 softmax (two warpgroups), 8 TMA producer, 9 MMA issuer (one
// thread), 10..11 spare (the third warpgroup gives registers to the softmax
// ones with setmaxnreg).  Every mbarrier wait is bounded (as in the forward).
// Both kernels launch their units heaviest first (the schedule's launch order:
// units that see the most tiles start first, the lightest fill the last wave),
// and take the sliding window as a template flag.
#include <cuda.h>

#include <vector>

#include "common.cuh"
#include "ptx.cuh"

namespace cpa {
namespace {

constexpr int kThreads = 384;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kSoftmaxThreads = 256;

// 32 fp32 accumulator columns (raw TMEM words) times mul, rounded to bf16, as
// four 16-byte stores (dst 16-byte aligned).
__device__ __forceinline__ void store_row_bf16(__nv_bfloat16* dst, const uint32_t (&rr)[32], float mul) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int v4 = 0; v4 < 4; ++v4)
    d4[v4] = make_uint4(ptx::pack_bf16x2(__uint_as_float(rr[8 * v4 + 0]) * mul, __uint_as_float(rr[8 * v4 + 1]) * mul),
                        ptx::pack_bf16x2(__uint_as_float(rr[8 * v4 + 2]) * mul, __uint_as_float(rr[8 * v4 + 3]) * mul),
                        ptx::pack_bf16x2(__uint_as_float(rr[8 * v4 + 4]) * mul, __uint_as_float(rr[8 * v4 + 5]) * mul),
                        ptx::pack_bf16x2(__uint_as_float(rr[8 * v4 + 6]) * mul, __uint_as_float(rr[8 * v4 + 7]) * mul));
}
// 32 fp32 accumulator columns times mul into 32 fp32 values (dst 16-byte aligned):
// overwritten, or added to what dst holds when `add` (the accumulating form).
__device__ __forceinline__ void store_row_f32(float* dst, const uint32_t (&rr)[32], float mul, int add) {
  float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int v4 = 0; v4 < 8; ++v4) {
    float4 x = make_float4(__uint_as_float(rr[4 * v4]) * mul, __uint_as_float(rr[4 * v4 + 1]) * mul,
                           __uint_as_float(rr[4 * v4 + 2]) * mul, __uint_as_float(rr[4 * v4 + 3]) * mul);
    if (add) {
      const float4 o = d4[v4];
      x.x += o.x;
      x.y += o.y;
      x.z += o.z;
      x.w += o.w;
    }
    d4[v4] = x;
  }
}
// Register split (launch: 384 x 168 = 64512): the TMA/MMA warpgroup drops to 72, the
// two softmax warpgroups rise to 216: 128*72 + 256*216 = 64512 (no spills in either).
constexpr int kRegsLow = 72;
constexpr int kRegsHigh = 216;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint64_t kDrainNs = 200000000ull;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kTileRows = 128;
// One [128 rows][HD] bf16 tile: HD/64 regions of 64 columns (16 KB each, 128-byte swizzle).
template <int HD>
constexpr int tile_bytes() { return kTileRows * HD * 2; }
constexpr int kSegCap = 128;                   // segments per group kept in shared memory

// Operand descriptors as a tile's base descriptor plus a compile-time step per K
// slice (the start-address field counts 16-byte units in its low 14 bits, and
// shared memory ends below 2^18 bytes, so the step never carries out of it).
// K-major, 128B swizzle: K step of 16 bf16 = 32 bytes inside a 64-column (16 KB) region.
__device__ __forceinline__ uint64_t desc_k_base(uint32_t base) { return ptx::smem_desc_sw128(base, 16, 1024); }
__device__ __forceinline__ constexpr uint64_t desc_k_step(int kk) {
  return (uint64_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
}
// MN-major, 128B swizzle: K step of 16 rows of 128 bytes; next 64 N columns at +16 KB.
__device__ __forceinline__ uint64_t desc_mn_base(uint32_t base) { return ptx::smem_desc_sw128(base, 16384, 1024); }
__device__ __forceinline__ constexpr uint64_t desc_mn_step(int kk) { return (uint64_t)((kk * (16 * 128)) >> 4); }
// TMEM A operand of K = 128 packed over two 64-column halves written by the two
// warpgroups: K step kk (16 values = 8 columns) of half kk / 4.
__device__ __forceinline__ uint32_t a_split(uint32_t base, int kk) {
  return base + (kk >> 2) * 64 + (kk & 3) * 8;
}

__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t par, volatile int* abort_flag,
                                         int32_t* err) {
  bool ok = ptx::mbar_wait_bounded(bar, par, abort_flag, err, kWaitNs);
  return __all_sync(0xffffffffu, ok);
}

// ====================================================================== dK / dV

constexpr int A_QST = 2;  // Q/dO stages

template <int HD>
struct ALayout {
  static constexpr int kTileBytes = tile_bytes<HD>();
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kQ = kV + kTileBytes;            // A_QST stages
  static constexpr int kDO = kQ + A_QST * kTileBytes;   // A_QST stages
  static constexpr int kLse = kDO + A_QST * kTileBytes;  // A_QST x (128 lse, 128 Delta) fp32
  static constexpr int kBar = kLse + A_QST * 2 * kTileRows * 4;
  static constexpr int kSeg = kBar + 256;  // the group's query runs (up to kSegCap)
  static constexpr int kBytes = kSeg + kSegCap * (int)sizeof(KSeg);
  static constexpr int kSmemRequest = kBytes + 1024;
};

struct ABars {
  uint64_t kv_full;
  uint64_t q_full[A_QST], q_empty[A_QST];
  uint64_t s_full, dp_full;  // S^T / dP^T of the current tile in TMEM
  uint64_t p_full, ds_full;  // P^T / dS^T written back by the softmax
  uint64_t done;             // every MMA of the CTA has completed
  uint32_t tmem_base;
  int abort_flag;
};

struct QTile {
  int32_t q_row;
  int32_t nq;
  int64_t pq_lo;
  int32_t qstride;
  int32_t h;
  int32_t full;
};

struct KeyCtx {
  int64_t pk_lo, pk_hi;
  int64_t en_lo;   // end of the document holding pk_lo
  int64_t win_hi;  // pk_hi + window - 1 (last query position any key sees), INT64_MAX without
  int causal, docs, window;
  int G, hk;
};

// Walks the query tiles that see some key of the CTA's key tile: the G query heads
// of the key/value head, each over the query runs in order.  Identical in every role.
struct QIter {
  const KSeg* segs;
  int nseg, hh, si, i, hi;
};

__device__ __forceinline__ void qiter_init(QIter& it, const KSeg* segs, int nseg, const KeyCtx& c) {
  it.segs = segs;
  it.nseg = nseg;
  it.hh = 0;
  it.si = 0;
  it.i = it.hi = 0;
  if (nseg > 0) query_tile_range(segs[0], kTileRows, c.pk_lo, c.causal, c.win_hi, it.i, it.hi);
}

__device__ __forceinline__ bool qiter_next(QIter& it, const KeyCtx& c, QTile& t) {
  while (it.hh < c.G) {
    if (it.si < it.nseg && it.i < it.hi) {
      const KSeg sg = it.segs[it.si];
      const int i0 = it.i * kTileRows;
      const int nq = min(kTileRows, sg.nk - i0);
      const int64_t pq_lo = (int64_t)sg.pos_off + (int64_t)sg.pos_stride * i0;
      const int64_t pq_hi = pq_lo + (int64_t)sg.pos_stride * (nq - 1);
      t.q_row = sg.k_row0 + i0;
      t.nq = nq;
      t.pq_lo = pq_lo;
      t.qstride = sg.pos_stride;
      t.h = c.hk * c.G + it.hh;
      t.full = (nq == kTileRows) && (c.causal ? pq_lo >= c.pk_hi : 1) && !c.docs;
      if (c.docs && c.causal) t.full = (nq == kTileRows) && pq_lo >= c.pk_hi && c.en_lo > pq_hi;
      if (c.window > 0) t.full = t.full && pq_hi - c.pk_lo < c.window;
      ++it.i;
      return true;
    }
    if (it.si < it.nseg && ++it.si < it.nseg) {
      query_tile_range(it.segs[it.si], kTileRows, c.pk_lo, c.causal, c.win_hi, it.i, it.hi);
      continue;
    }
    if (++it.hh < c.G) {
      it.si = 0;
      it.i = it.hi = 0;
      if (it.nseg > 0) query_tile_range(it.segs[0], kTileRows, c.pk_lo, c.causal, c.win_hi, it.i, it.hi);
    }
  }
  return false;
}

__device__ __forceinline__ int count_qtiles(const KSeg* segs, int nseg, const KeyCtx& c) {
  int n = 0;
  for (int si = 0; si < nseg; ++si) {
    int lo, hi;
    query_tile_range(segs[si], kTileRows, c.pk_lo, c.causal, c.win_hi, lo, hi);
    n += hi - lo;
  }
  return n * c.G;
}

// kWin: the sliding window is applied (a.window > 0); without it the window
// terms fold away at compile time.  Same flag on the dQ kernel.
template <int HD, bool kWin>
__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_dkdv_kernel(const __grid_constant__ BwdArgs a, const __grid_constant__ Schedule s,
                     const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  using L = ALayout<HD>;
  constexpr int D = HD;
  constexpr int kTileBytes = L::kTileBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  ABars* bars = reinterpret_cast<ABars*>(smem + L::kBar);
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* lse_all = reinterpret_cast<float*>(smem + L::kLse);

  int g, tile, hk;
  decode_unit_blocked(s, kTileRows, a.kv_head_block, a.kv_pairs, blockIdx.x, &g, &tile, &hk);
  const int32_t k_row0 = s.g[g].q_row0 + tile * kTileRows;  // key-major schedule: group = key run
  const int nk_tile = min(kTileRows, s.g[g].nq - tile * kTileRows);
  const int seg_begin = s.g[g].seg_begin, seg_end = seg_begin + s.g[g].seg_count;

  KeyCtx c;
  c.causal = a.causal;
  c.docs = a.cu_seqlens != nullptr;
  c.G = a.Hq / a.Hkv;
  c.hk = hk;
  c.pk_lo = (int64_t)s.g[g].pos_off + (int64_t)s.g[g].pos_stride * (tile * kTileRows);
  c.pk_hi = c.pk_lo + (int64_t)s.g[g].pos_stride * (nk_tile - 1);
  c.en_lo = INT64_MAX;
  if (c.docs) {
    int64_t st;
    doc_bounds(a.cu_seqlens, a.n_docs, c.pk_lo, &st, &c.en_lo);
  }
  c.window = kWin ? a.window : 0;
  c.win_hi = c.window > 0 ? c.pk_hi + c.window - 1 : INT64_MAX;

  // The group's query runs, read at every tile by every role: shared memory when they fit.
  const int nseg = seg_end - seg_begin;
  KSeg* seg_sm = reinterpret_cast<KSeg*>(smem + L::kSeg);
  const KSeg* segs = nseg <= kSegCap ? seg_sm : &s.s[seg_begin];
  if (nseg <= kSegCap)
    for (int i = threadIdx.x; i < nseg; i += kThreads) seg_sm[i] = s.s[seg_begin + i];
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bars->kv_full, 1);
    for (int i = 0; i < A_QST; ++i) {
      ptx::mbar_init(&bars->q_full[i], 1 + 32);  // TMA (expect_tx) + each producer lane's cp.async
      ptx::mbar_init(&bars->q_empty[i], 1);
    }
    ptx::mbar_init(&bars->s_full, 1);
    ptx::mbar_init(&bars->dp_full, 1);
    ptx::mbar_init(&bars->p_full, kSoftmaxThreads);
    ptx::mbar_init(&bars->ds_full, kSoftmaxThreads);
    ptx::mbar_init(&bars->done, 1);
    bars->abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(&bars->tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    ptx::prefetch_tensormap(&tm_q);
    ptx::prefetch_tensormap(&tm_do);
    ptx::prefetch_tensormap(&tm_k);
    ptx::prefetch_tensormap(&tm_v);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort_flag;

  if (warp >= 8) {
    ptx::setmaxnreg_dec<kRegsLow>();
    if (warp == kProducerWarp) {
      // ---------------------------------------------------------- producer (whole warp)
      if (lane == 0) {
        (void)CP_DCHECK(k_row0 < a.k_rows, a.err);  // TMA clips; the check reports
        ptx::mbar_arrive_expect_tx(&bars->kv_full, 2 * kTileBytes);
        for (int r = 0; r < D / 64; ++r) {
          ptx::tma_load_2d(smem + L::kK + r * 16384, &tm_k, &bars->kv_full, hk * D + r * 64, k_row0);
          ptx::tma_load_2d(smem + L::kV + r * 16384, &tm_v, &bars->kv_full, hk * D + r * 64, k_row0);
        }
      }
      QIter it;
      qiter_init(it, segs, nseg, c);
      int j = 0;
      QTile t;
      int issued[A_QST] = {0, 0};
      while (__all_sync(0xffffffffu, *abort_flag == 0) && qiter_next(it, c, t)) {
        const int st = j % A_QST;
        if (j >= A_QST && !wait_all(&bars->q_empty[st], ((j / A_QST) - 1) & 1, abort_flag, a.err)) break;
        if (lane == 0) {
          (void)CP_DCHECK(t.q_row >= 0 && t.q_row < a.q_rows, a.err);
          ptx::mbar_arrive_expect_tx(&bars->q_full[st], 2 * kTileBytes);
          for (int r = 0; r < D / 64; ++r) {
            ptx::tma_load_2d(smem + L::kQ + st * kTileBytes + r * 16384, &tm_q, &bars->q_full[st],
                             t.h * D + r * 64, t.q_row);
            ptx::tma_load_2d(smem + L::kDO + st * kTileBytes + r * 16384, &tm_do, &bars->q_full[st],
                             t.h * D + r * 64, t.q_row);
          }
        }
        // lse and Delta of the tile's rows (columns past the run are masked and never read)
        float* lse_st = lse_all + st * 2 * kTileRows;
        for (int cidx = lane; cidx < t.nq; cidx += 32) {
          const int64_t off = (int64_t)t.h * a.lse_ld + t.q_row + cidx;
          if (!CP_DCHECK(off < a.lse_size, a.err)) continue;
          ptx::cp_async4(lse_st + cidx, a.lse + off);
          ptx::cp_async4(lse_st + kTileRows + cidx, a.delta + off);
        }
        ptx::cp_async_arrive(&bars->q_full[st]);
        issued[st] = j + 1;
        ++j;
      }
      if (lane == 0 && *abort_flag) {
        (void)ptx::mbar_wait_bounded(&bars->kv_full, 0, nullptr, nullptr, kDrainNs);
        for (int st = 0; st < A_QST; ++st)
          if (issued[st] > 0)
            (void)ptx::mbar_wait_bounded(&bars->q_full[st], ((issued[st] - 1) / A_QST) & 1, nullptr,
                                         nullptr, kDrainNs);
      }
      __syncwarp();
    } else if (warp == kMmaWarp) {
      // ---------------------------------------------------------- MMA issuer
      if (lane == 0) {
        constexpr uint32_t id_s = ptx::idesc_bf16_f32(128, 128, 0, 0);   // K Q^T, V dO^T
        constexpr uint32_t id_kv = ptx::idesc_bf16_f32(128, D, 0, 1);    // P^T dO, dS^T Q (TMEM A)
        const uint32_t k_addr = sbase + L::kK, v_addr = sbase + L::kV;
        bool issued = false;
        auto wait = [&](uint64_t* bar, uint32_t par) {
          return ptx::mbar_wait_bounded(bar, par, abort_flag, a.err, kWaitNs);
        };
        auto scores = [&](uint32_t d, uint32_t a_addr, uint32_t b_addr) {
          const uint64_t ad = desc_k_base(a_addr), bd = desc_k_base(b_addr);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            ptx::mma_bf16_ss(tmem + d, ad + desc_k_step(kk), bd + desc_k_step(kk), id_s, kk > 0);
        };
        auto grads = [&](uint32_t d, uint32_t a_tmem, uint32_t b_addr, bool acc) {
          const uint64_t bd = desc_mn_base(b_addr);
#pragma unroll
          for (int kk = 0; kk < kTileRows / 16; ++kk)
            ptx::mma_bf16_ts(tmem + d, a_split(tmem + a_tmem, kk), bd + desc_mn_step(kk), id_kv,
                             (acc || kk > 0) ? 1u : 0u);
        };
        const int n = count_qtiles(segs, nseg, c);  // no schedule walking between products
        if (wait(&bars->kv_full, 0)) {
          int j = 0;
          bool have = n > 0;
          if (have) {
            if (!wait(&bars->q_full[0], 0)) have = false;
            if (have) {
              ptx::tc_fence_after();
              scores(0, k_addr, sbase + L::kQ);
              ptx::tc_commit(&bars->s_full);
              scores(128, v_addr, sbase + L::kDO);
              ptx::tc_commit(&bars->dp_full);
              issued = true;
            }
          }
          while (have) {
            const bool more = j + 1 < n;
            const int st = j % A_QST, st1 = (j + 1) % A_QST;
            // dV += P^T dO once P^T is written back
            if (!wait(&bars->p_full, j & 1)) break;
            ptx::tc_fence_after();
            grads(256, 0, sbase + L::kDO + st * kTileBytes, j > 0);
            // next tile's S^T (reuses the S^T columns after dV has read P^T)
            if (more) {
              if (!wait(&bars->q_full[st1], ((j + 1) / A_QST) & 1)) break;
              ptx::tc_fence_after();
              scores(0, k_addr, sbase + L::kQ + st1 * kTileBytes);
              ptx::tc_commit(&bars->s_full);
            }
            // dK += dS^T Q once dS^T is written back
            if (!wait(&bars->ds_full, j & 1)) break;
            ptx::tc_fence_after();
            grads(384, 128, sbase + L::kQ + st * kTileBytes, j > 0);
            ptx::tc_commit(&bars->q_empty[st]);
            if (more) {
              scores(128, v_addr, sbase + L::kDO + st1 * kTileBytes);
              ptx::tc_commit(&bars->dp_full);
            }
            ++j;
            have = more;
          }
        }
        if (issued) {
          ptx::tc_commit(&bars->done);
          (void)ptx::mbar_wait_bounded(&bars->done, 0, nullptr, a.err, kWaitNs);
        } else {
          ptx::mbar_arrive(&bars->done);
        }
      }
      __syncwarp();
    }
  } else {
    ptx::setmaxnreg_inc<kRegsHigh>();
    // ------------------------------------------------------------ softmax warpgroups (thread = key row)
    const int quad = warp & 3;
    const int wg = warp >> 2;
    const int cb = wg * 64;  // this warpgroup's 64 query columns of the 128
    const int r = quad * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
    const int64_t pk = c.pk_lo + (int64_t)s.g[g].pos_stride * r;
    int64_t st_k = 0, en_k = INT64_MAX;
    if (c.docs && r < nk_tile) doc_bounds(a.cu_seqlens, a.n_docs, pk, &st_k, &en_k);
    const float sl2 = a.scale_log2;
    const uint64_t sl2x2 = ptx::f2_pack(sl2, sl2), nlog2e2 = ptx::f2_pack(-kLog2e, -kLog2e);
    const uint64_t neg1x2 = ptx::f2_pack(-1.f, -1.f);
    QIter it;
    qiter_init(it, segs, nseg, c);
    int j = 0;
    QTile t;
    bool ok = true;
    while (__all_sync(0xffffffffu, *abort_flag == 0) && qiter_next(it, c, t)) {
      const int st = j % A_QST;
      int64_t hi = t.nq - 1, lo = 0;  // visible query columns of this key row: [lo, hi]
      if (r >= nk_tile) {
        hi = -1;
      } else if (!t.full) {
        if (c.causal) {
          const int64_t d0 = pk - t.pq_lo;  // need pq >= pk
          lo = max(lo, d0 <= 0 ? (int64_t)0 : udiv_pos(d0 + t.qstride - 1, t.qstride));
        }
        if (c.docs) {
          const int64_t d1 = en_k - 1 - t.pq_lo;  // need pq < end of the key's document
          hi = min(hi, d1 < 0 ? (int64_t)-1 : udiv_pos(d1, t.qstride));
          if (!c.causal) {  // and pq >= start of the key's document
            const int64_t d2 = st_k - t.pq_lo;
            lo = max(lo, d2 <= 0 ? (int64_t)0 : udiv_pos(d2 + t.qstride - 1, t.qstride));
          }
        }
        if (c.window > 0) {  // need pq <= pk + window - 1
          const int64_t d3 = pk + c.window - 1 - t.pq_lo;
          hi = min(hi, d3 < 0 ? (int64_t)-1 : udiv_pos(d3, t.qstride));
        }
      }
      const int ilo = (int)min(lo, (int64_t)kTileRows), ihi = (int)max(hi, (int64_t)-1);
      if (!wait_all(&bars->q_full[st], (j / A_QST) & 1, abort_flag, a.err)) { ok = false; break; }
      const float* lse_st = lse_all + st * 2 * kTileRows + cb;
      const float* del_st = lse_st + kTileRows;
      // phase 1: P^T = 2^(S^T*scale*log2e - lse*log2e)
      if (!wait_all(&bars->s_full, j & 1, abort_flag, a.err)) { ok = false; break; }
      ptx::tc_fence_after();
      float p[64];
      uint32_t sr2[2][32];  // both halves in flight before one wait
      ptx::tmem_ld32(lane_addr + cb, sr2[0]);
      ptx::tmem_ld32(lane_addr + cb + 32, sr2[1]);
      ptx::tmem_wait_ld_regs(sr2[0]);
      ptx::tmem_wait_ld_regs(sr2[1]);
#pragma unroll
      for (int hc = 0; hc < 64; hc += 32) {
        const uint32_t* sr = sr2[hc / 32];
        if (t.full) {  // every pair visible: no per-column mask
#pragma unroll
          for (int cc = 0; cc < 32; cc += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(lse_st + hc + cc);
            const uint64_t nl01 = ptx::fmul2(ptx::f2_pack(l4.x, l4.y), nlog2e2);
            const uint64_t nl23 = ptx::fmul2(ptx::f2_pack(l4.z, l4.w), nlog2e2);
            float a0, a1, a2, a3;
            ptx::f2_unpack(ptx::ffma2(ptx::f2_pack(__uint_as_float(sr[cc]), __uint_as_float(sr[cc + 1])),
                                      sl2x2, nl01), a0, a1);
            ptx::f2_unpack(ptx::ffma2(ptx::f2_pack(__uint_as_float(sr[cc + 2]), __uint_as_float(sr[cc + 3])),
                                      sl2x2, nl23), a2, a3);
            p[hc + cc] = ptx::ex2_approx(a0);
            p[hc + cc + 1] = ptx::ex2_approx(a1);
            p[hc + cc + 2] = ptx::ex2_approx(a2);
            p[hc + cc + 3] = ptx::ex2_approx(a3);
          }
        } else {
#pragma unroll
          for (int cc = 0; cc < 32; ++cc) {
            const int col = cb + hc + cc;
            const bool vis = col >= ilo && col <= ihi;  // masked columns read nothing staged
            p[hc + cc] = vis ? ptx::ex2_approx(fmaf(__uint_as_float(sr[cc]), sl2, -lse_st[hc + cc] * kLog2e))
                             : 0.f;
          }
        }
      }
      {
        uint32_t pk32[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) pk32[i] = ptx::pack_bf16x2(p[2 * i], p[2 * i + 1]);
        ptx::tmem_st32(lane_addr + cb, pk32);  // P^T over the first 32 of this warpgroup's columns
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&bars->p_full);
      }
      // phase 2: dS^T = P^T o (dP^T - Delta), 32 columns at a time, packed over the dP^T columns
      // already read (half h of the packed values lands on columns of half 0)
      if (!wait_all(&bars->dp_full, j & 1, abort_flag, a.err)) { ok = false; break; }
      ptx::tc_fence_after();
#pragma unroll
      for (int hc = 0; hc < 64; hc += 32) {
        uint32_t dr[32];
        ptx::tmem_ld32(lane_addr + 128 + cb + hc, dr);
        ptx::tmem_wait_ld_regs(dr);
        uint32_t dd[16];
        if (t.full) {
#pragma unroll
          for (int cc = 0; cc < 32; cc += 2) {
            const float2 d2 = *reinterpret_cast<const float2*>(del_st + hc + cc);
            // dP - Delta as an exact fma with -1, then P * (dP - Delta)
            const uint64_t tt = ptx::ffma2(ptx::f2_pack(d2.x, d2.y), neg1x2,
                                           ptx::f2_pack(__uint_as_float(dr[cc]), __uint_as_float(dr[cc + 1])));
            float ds0, ds1;
            ptx::f2_unpack(ptx::fmul2(ptx::f2_pack(p[hc + cc], p[hc + cc + 1]), tt), ds0, ds1);
            dd[cc / 2] = ptx::pack_bf16x2(ds0, ds1);
          }
        } else {
#pragma unroll
          for (int cc = 0; cc < 32; cc += 2) {
            const int col = cb + hc + cc;
            const bool v0 = col >= ilo && col <= ihi, v1 = col + 1 >= ilo && col + 1 <= ihi;
            const float ds0 = v0 ? p[hc + cc] * (__uint_as_float(dr[cc]) - del_st[hc + cc]) : 0.f;
            const float ds1 = v1 ? p[hc + cc + 1] * (__uint_as_float(dr[cc + 1]) - del_st[hc + cc + 1]) : 0.f;
            dd[cc / 2] = ptx::pack_bf16x2(ds0, ds1);
          }
        }
        ptx::tmem_st16(lane_addr + 128 + cb + hc / 2, dd);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&bars->ds_full);
      ++j;
    }
    // ------------------------------------------------------------ dK / dV epilogue
    ok = ok && __all_sync(0xffffffffu, *abort_flag == 0);
    if (ok) ok = wait_all(&bars->done, 0, abort_flag, a.err);
    if (ok) {
      ptx::tc_fence_after();
      const bool valid = r < nk_tile && CP_DCHECK((int64_t)k_row0 + r < a.k_rows, a.err);
      const int64_t krow = (int64_t)(k_row0 + r) * a.k_ld + (int64_t)hk * D;
      float* dst = (wg == 0 ? a.dv_acc : a.dk_acc) + krow;  // warpgroup 0: dV, 1: dK
      void* out_bf = wg == 0 ? a.dv_out : a.dk_out;
      __nv_bfloat16* dst_bf = out_bf ? static_cast<__nv_bfloat16*>(out_bf) + krow : nullptr;
      const float mul = wg == 0 ? 1.f : a.scale;
      const uint32_t col0 = wg == 0 ? 256 : 384;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t rr[32];
        if (j > 0) {
          ptx::tmem_ld32(lane_addr + col0 + ch * 32, rr);
          ptx::tmem_wait_ld_regs(rr);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) rr[i] = 0u;
        }
        if (valid && dst_bf) {
          store_row_bf16(dst_bf + ch * 32, rr, mul);
        } else if (valid) {
          store_row_f32(dst + ch * 32, rr, mul, a.accumulate);
        }
      }
    }
    ptx::tc_fence_before();
  }

  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ====================================================================== dQ

constexpr int B_KST = 3;      // K stages (K_j is last read by dQ_j, the last product of tile j)
constexpr int B_VST = 2;      // V stages (V_j is last read by dP_j, two products earlier)
constexpr int kSegCapB = 96;  // key runs kept in shared memory (the tiles take the rest)

template <int HD>
struct BLayout {
  static constexpr int kTileBytes = tile_bytes<HD>();
  static constexpr int kQ = 0;                        // the CTA's query tile
  static constexpr int kDO = kQ + kTileBytes;         // its dO tile
  static constexpr int kK = kDO + kTileBytes;         // B_KST stages
  static constexpr int kV = kK + B_KST * kTileBytes;  // B_VST stages
  static constexpr int kBar = kV + B_VST * kTileBytes;
  static constexpr int kSeg = kBar + 256;  // the group's key runs (up to kSegCapB)
  static constexpr int kBytes = kSeg + kSegCapB * (int)sizeof(KSeg);
  static constexpr int kSmemRequest = kBytes + 1024;
};
static_assert(BLayout<128>::kSmemRequest <= 227 * 1024, "dQ kernel: shared memory per CTA");

struct BBars {
  uint64_t q_full;                         // Q and dO tiles landed
  uint64_t k_full[B_KST], k_empty[B_KST];  // K tile of a stage landed / released (after dQ_j)
  uint64_t v_full[B_VST], v_empty[B_VST];  // V tile of a stage landed / released (after dP_j)
  uint64_t s_full;      // S of the current tile in TMEM
  uint64_t s_free;      // the softmax has read S
  uint64_t dp_full[2];  // dP of tile j in buffer j % 2
  uint64_t ds_full[2];  // dS of tile j written back over buffer j % 2
  uint64_t done;        // every MMA of the CTA has completed
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(BBars) <= 256, "dQ kernel barriers");

struct TileCtx {
  int64_t pq_lo, pq_hi;
  int64_t st_lo, st_hi, en_lo, en_hi;
  int64_t win_lo;  // pq_lo - window + 1 (first key position any query sees), INT64_MIN without
  int causal, docs, window;
};

struct KvTile {
  int32_t k_row;
  int32_t nk;
  int64_t pk_lo;
  int32_t kstride;
  int32_t full;
};

// Walks the key/value tiles (128 keys) of the query group with any visible pair.
// Identical in every role.
struct KIter {
  const KSeg* segs;
  int nseg, si, i, hi;
};

__device__ __forceinline__ void kiter_range(KIter& it, const TileCtx& c) {
  key_tile_range(it.segs[it.si], kTileRows, c.pq_hi, c.st_lo, c.en_hi, c.causal, c.docs, c.win_lo, it.i,
                 it.hi);
}

__device__ __forceinline__ void kiter_init(KIter& it, const KSeg* segs, int nseg, const TileCtx& c) {
  it.segs = segs;
  it.nseg = nseg;
  it.si = 0;
  it.i = it.hi = 0;
  if (nseg > 0) kiter_range(it, c);
}

__device__ __forceinline__ bool kiter_next(KIter& it, const TileCtx& c, KvTile& t) {
  while (it.si < it.nseg) {
    if (it.i < it.hi) {
      const KSeg sg = it.segs[it.si];
      const int j0 = it.i * kTileRows;
      const int nk = min(kTileRows, sg.nk - j0);
      const int64_t pk_lo = (int64_t)sg.pos_off + (int64_t)sg.pos_stride * j0;
      const int64_t pk_hi = pk_lo + (int64_t)sg.pos_stride * (nk - 1);
      t.k_row = sg.k_row0 + j0;
      t.nk = nk;
      t.pk_lo = pk_lo;
      t.kstride = sg.pos_stride;
      t.full = (nk == kTileRows) && (!c.causal || pk_hi <= c.pq_lo) &&
               (!c.docs || (pk_lo >= c.st_hi && pk_hi < c.en_lo)) &&
               (c.window == 0 || c.pq_hi - pk_lo < c.window);
      ++it.i;
      return true;
    }
    if (++it.si < it.nseg) kiter_range(it, c);
  }
  return false;
}

__device__ __forceinline__ int count_ktiles(const KSeg* segs, int nseg, const TileCtx& c) {
  int n = 0;
  for (int si = 0; si < nseg; ++si) {
    int lo, hi;
    key_tile_range(segs[si], kTileRows, c.pq_hi, c.st_lo, c.en_hi, c.causal, c.docs, c.win_lo, lo, hi);
    n += hi - lo;
  }
  return n;
}

template <int HD, bool kWin>
__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_dq_kernel(const __grid_constant__ BwdArgs a, const __grid_constant__ Schedule s,
                   const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  using L = BLayout<HD>;
  constexpr int D = HD;
  constexpr int kTileBytes = L::kTileBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  BBars* bars = reinterpret_cast<BBars*>(smem + L::kBar);
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  int g, tile, h;
  decode_unit_blocked(s, kTileRows, a.q_head_block, a.q_pairs, blockIdx.x, &g, &tile, &h);
  const int hk = h / (a.Hq / a.Hkv);
  const int32_t q_row0 = s.g[g].q_row0, nq = s.g[g].nq;
  const int32_t qpos_off = s.g[g].pos_off, qpos_st = s.g[g].pos_stride;
  const int seg_begin = s.g[g].seg_begin, seg_end = seg_begin + s.g[g].seg_count;
  const int i0 = tile * kTileRows;
  const int nq_tile = min(kTileRows, nq - i0);

  TileCtx c;
  c.causal = a.causal;
  c.docs = a.cu_seqlens != nullptr;
  c.pq_lo = (int64_t)qpos_off + (int64_t)qpos_st * i0;
  c.pq_hi = c.pq_lo + (int64_t)qpos_st * (nq_tile - 1);
  c.st_lo = c.st_hi = c.en_lo = c.en_hi = 0;
  if (c.docs) {
    doc_bounds(a.cu_seqlens, a.n_docs, c.pq_lo, &c.st_lo, &c.en_lo);
    doc_bounds(a.cu_seqlens, a.n_docs, c.pq_hi, &c.st_hi, &c.en_hi);
  }
  c.window = kWin ? a.window : 0;
  c.win_lo = c.window > 0 ? c.pq_lo - c.window + 1 : INT64_MIN;

  // The group's key runs, read at every tile by every role: shared memory when they fit.
  const int nseg = seg_end - seg_begin;
  KSeg* seg_sm = reinterpret_cast<KSeg*>(smem + L::kSeg);
  const KSeg* segs = nseg <= kSegCapB ? seg_sm : &s.s[seg_begin];
  if (nseg <= kSegCapB)
    for (int i = threadIdx.x; i < nseg; i += kThreads) seg_sm[i] = s.s[seg_begin + i];
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bars->q_full, 1);
    for (int i = 0; i < B_KST; ++i) {
      ptx::mbar_init(&bars->k_full[i], 1);
      ptx::mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < B_VST; ++i) {
      ptx::mbar_init(&bars->v_full[i], 1);
      ptx::mbar_init(&bars->v_empty[i], 1);
    }
    ptx::mbar_init(&bars->s_full, 1);
    ptx::mbar_init(&bars->s_free, kSoftmaxThreads);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&bars->dp_full[i], 1);
      ptx::mbar_init(&bars->ds_full[i], kSoftmaxThreads);
    }
    ptx::mbar_init(&bars->done, 1);
    bars->abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(&bars->tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    ptx::prefetch_tensormap(&tm_q);
    ptx::prefetch_tensormap(&tm_do);
    ptx::prefetch_tensormap(&tm_k);
    ptx::prefetch_tensormap(&tm_v);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort_flag;

  if (warp >= 8) {
    ptx::setmaxnreg_dec<kRegsLow>();
    if (warp == kProducerWarp) {
      // ---------------------------------------------------------- TMA producer
      if (lane == 0) {
        (void)CP_DCHECK((int64_t)q_row0 + i0 < a.q_rows, a.err);  // TMA clips; the check reports
        ptx::mbar_arrive_expect_tx(&bars->q_full, 2 * kTileBytes);
        for (int r = 0; r < D / 64; ++r) {
          ptx::tma_load_2d(smem + L::kQ + r * 16384, &tm_q, &bars->q_full, h * D + r * 64, q_row0 + i0);
          ptx::tma_load_2d(smem + L::kDO + r * 16384, &tm_do, &bars->q_full, h * D + r * 64, q_row0 + i0);
        }
        KIter it;
        kiter_init(it, segs, nseg, c);
        int j = 0;
        KvTile t;
        int issued_k[B_KST] = {0, 0, 0}, issued_v[B_VST] = {0, 0};
        while (!*abort_flag && kiter_next(it, c, t)) {
          const int sk = j % B_KST, sv = j % B_VST;
          (void)CP_DCHECK(t.k_row >= 0 && t.k_row < a.k_rows, a.err);
          if (j >= B_KST && !ptx::mbar_wait_bounded(&bars->k_empty[sk], ((j / B_KST) - 1) & 1, abort_flag,
                                                     a.err, kWaitNs))
            break;
          ptx::mbar_arrive_expect_tx(&bars->k_full[sk], kTileBytes);
          for (int r = 0; r < D / 64; ++r)
            ptx::tma_load_2d(smem + L::kK + sk * kTileBytes + r * 16384, &tm_k, &bars->k_full[sk],
                             hk * D + r * 64, t.k_row);
          issued_k[sk] = j + 1;
          if (j >= B_VST && !ptx::mbar_wait_bounded(&bars->v_empty[sv], ((j / B_VST) - 1) & 1, abort_flag,
                                                     a.err, kWaitNs))
            break;
          ptx::mbar_arrive_expect_tx(&bars->v_full[sv], kTileBytes);
          for (int r = 0; r < D / 64; ++r)
            ptx::tma_load_2d(smem + L::kV + sv * kTileBytes + r * 16384, &tm_v, &bars->v_full[sv],
                             hk * D + r * 64, t.k_row);
          issued_v[sv] = j + 1;
          ++j;
        }
        if (*abort_flag) {
          (void)ptx::mbar_wait_bounded(&bars->q_full, 0, nullptr, nullptr, kDrainNs);
          for (int st = 0; st < B_KST; ++st)
            if (issued_k[st] > 0)
              (void)ptx::mbar_wait_bounded(&bars->k_full[st], ((issued_k[st] - 1) / B_KST) & 1, nullptr,
                                           nullptr, kDrainNs);
          for (int st = 0; st < B_VST; ++st)
            if (issued_v[st] > 0)
              (void)ptx::mbar_wait_bounded(&bars->v_full[st], ((issued_v[st] - 1) / B_VST) & 1, nullptr,
                                           nullptr, kDrainNs);
        }
      }
      __syncwarp();
    } else if (warp == kMmaWarp) {
      // ---------------------------------------------------------- MMA issuer
      if (lane == 0) {
        constexpr uint32_t id_s = ptx::idesc_bf16_f32(128, 128, 0, 0);  // Q K^T, dO V^T (shared memory)
        constexpr uint32_t id_q = ptx::idesc_bf16_f32(128, D, 0, 1);    // dS K (TMEM A)
        bool any = false;
        auto wait = [&](uint64_t* bar, uint32_t par) {
          return ptx::mbar_wait_bounded(bar, par, abort_flag, a.err, kWaitNs);
        };
        auto scores = [&](uint32_t d, uint32_t a_addr, uint32_t b_addr) {
          const uint64_t ad = desc_k_base(a_addr), bd = desc_k_base(b_addr);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            ptx::mma_bf16_ss(tmem + d, ad + desc_k_step(kk), bd + desc_k_step(kk), id_s, kk > 0);
        };
        // dP / dS of tile j live in TMEM columns 128.. (j even) or 384.. (j odd), so
        // dP_{j+1} is issued as soon as the softmax has read S_j, before dS_j exists.
        // Issue order per tile: S_{j+1}, dP_{j+1}, dQ_j; each gap between two
        // products holds one barrier wait (the loads' are normally complete: their
        // test is the cheap path) and no schedule walking.
        const int n = count_ktiles(segs, nseg, c);
        bool ok = n > 0 && wait(&bars->q_full, 0) && wait(&bars->k_full[0], 0);
        if (ok) {
          ptx::tc_fence_after();
          scores(0, sbase + L::kQ, sbase + L::kK);
          ptx::tc_commit(&bars->s_full);
          any = true;
          ok = wait(&bars->v_full[0], 0);
          if (ok) {
            ptx::tc_fence_after();
            scores(128, sbase + L::kDO, sbase + L::kV);
            ptx::tc_commit(&bars->dp_full[0]);
            ptx::tc_commit(&bars->v_empty[0]);
          }
        }
        for (int j = 0; ok && j < n; ++j) {
          if (j + 1 < n) {
            const int j1 = j + 1, sk1 = j1 % B_KST, sv1 = j1 % B_VST;
            // S_{j+1} once the softmax has read S_j
            if (!(ok = wait(&bars->s_free, j & 1))) break;
            if (!(ok = wait(&bars->k_full[sk1], (j1 / B_KST) & 1))) break;
            ptx::tc_fence_after();
            scores(0, sbase + L::kQ, sbase + L::kK + sk1 * kTileBytes);
            ptx::tc_commit(&bars->s_full);
            // dP_{j+1} into the other buffer (dQ_{j-1}, which read it, is ahead in the pipe)
            if (!(ok = wait(&bars->v_full[sv1], (j1 / B_VST) & 1))) break;
            ptx::tc_fence_after();
            scores(j1 & 1 ? 384 : 128, sbase + L::kDO, sbase + L::kV + sv1 * kTileBytes);
            ptx::tc_commit(&bars->dp_full[j1 & 1]);
            ptx::tc_commit(&bars->v_empty[sv1]);
          }
          // dQ += dS_j K_j once dS_j is written back (two warpgroup halves of 64 keys)
          if (!(ok = wait(&bars->ds_full[j & 1], (j >> 1) & 1))) break;
          ptx::tc_fence_after();
          {
            const uint64_t kd = desc_mn_base(sbase + L::kK + (j % B_KST) * kTileBytes);
            const uint32_t ds = j & 1 ? 384 : 128;
#pragma unroll
            for (int kk = 0; kk < kTileRows / 16; ++kk)
              ptx::mma_bf16_ts(tmem + 256, a_split(tmem + ds, kk), kd + desc_mn_step(kk), id_q,
                               (j > 0 || kk > 0) ? 1u : 0u);
          }
          ptx::tc_commit(&bars->k_empty[j % B_KST]);
        }
        if (any) {
          ptx::tc_commit(&bars->done);
          (void)ptx::mbar_wait_bounded(&bars->done, 0, nullptr, a.err, kWaitNs);
        } else {
          ptx::mbar_arrive(&bars->done);
        }
      }
      __syncwarp();
    }
  } else {
    ptx::setmaxnreg_inc<kRegsHigh>();
    // ------------------------------------------------------------ softmax warpgroups (thread = query row)
    const int quad = warp & 3;
    const int w = warp >> 2;
    const int cb = w * 64;  // this warpgroup's 64 key columns of the 128
    const int r = quad * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
    const bool row_valid = r < nq_tile;
    const int64_t pq = c.pq_lo + (int64_t)qpos_st * r;
    int64_t st_r = 0, en_r = 0;
    if (c.docs && row_valid) doc_bounds(a.cu_seqlens, a.n_docs, pq, &st_r, &en_r);
    float nlse2 = 0.f, delta = 0.f;  // -lse*log2(e); rows without a visible key are fully masked
    if (row_valid) {
      const int64_t col = (int64_t)h * a.lse_ld + q_row0 + i0 + r;
      if (CP_DCHECK(col < a.lse_size, a.err)) {
        nlse2 = -a.lse[col] * kLog2e;
        delta = a.delta[col];
      }
    }
    const float sl2 = a.scale_log2;
    const uint64_t sl2x2 = ptx::f2_pack(sl2, sl2), nl2x2 = ptx::f2_pack(nlse2, nlse2);
    const uint64_t nd2x2 = ptx::f2_pack(-delta, -delta);
    KIter it;
    kiter_init(it, segs, nseg, c);
    int j = 0;
    KvTile t;
    bool ok = true;
    while (__all_sync(0xffffffffu, *abort_flag == 0) && kiter_next(it, c, t)) {
      int64_t hi = t.nk - 1, lo = 0;
      if (!row_valid) {
        hi = -1;
      } else if (!t.full) {
        if (c.causal) {
          const int64_t d = pq - t.pk_lo;
          hi = min(hi, d < 0 ? (int64_t)-1 : udiv_pos(d, t.kstride));
        }
        if (c.docs) {
          const int64_t da = st_r - t.pk_lo;
          lo = max(lo, da <= 0 ? (int64_t)0 : udiv_pos(da + t.kstride - 1, t.kstride));
          const int64_t db = en_r - 1 - t.pk_lo;
          hi = min(hi, db < 0 ? (int64_t)-1 : udiv_pos(db, t.kstride));
        }
        if (c.window > 0) {  // need pk >= pq - window + 1
          const int64_t dw = pq - c.window + 1 - t.pk_lo;
          lo = max(lo, dw <= 0 ? (int64_t)0 : udiv_pos(dw + t.kstride - 1, t.kstride));
        }
      }
      const int ilo = (int)min(lo, (int64_t)kTileRows), ihi = (int)max(hi, (int64_t)-1);
      // phase 1: P from S, then release S for the next tile
      if (!wait_all(&bars->s_full, j & 1, abort_flag, a.err)) { ok = false; break; }
      ptx::tc_fence_after();
      float p[64];
      const bool fast = t.full && nq_tile == kTileRows;  // every pair visible: no per-column mask
      uint32_t sr2[2][32];  // both halves in flight before one wait
      ptx::tmem_ld32(lane_addr + cb, sr2[0]);
      ptx::tmem_ld32(lane_addr + cb + 32, sr2[1]);
      ptx::tmem_wait_ld_regs(sr2[0]);
      ptx::tmem_wait_ld_regs(sr2[1]);
      ptx::tc_fence_before();
      ptx::mbar_arrive(&bars->s_free);  // S is in registers: the next S may overwrite it
#pragma unroll
      for (int hc = 0; hc < 64; hc += 32) {
        const uint32_t* sr = sr2[hc / 32];
        if (fast) {
#pragma unroll
          for (int cc = 0; cc < 32; cc += 2) {
            float a0, a1;
            ptx::f2_unpack(ptx::ffma2(ptx::f2_pack(__uint_as_float(sr[cc]), __uint_as_float(sr[cc + 1])),
                                      sl2x2, nl2x2), a0, a1);
            p[hc + cc] = ptx::ex2_approx(a0);
            p[hc + cc + 1] = ptx::ex2_approx(a1);
          }
        } else {
#pragma unroll
          for (int cc = 0; cc < 32; ++cc) {
            const int col = cb + hc + cc;
            const bool vis = col >= ilo && col <= ihi;
            p[hc + cc] = vis ? ptx::ex2_approx(fmaf(__uint_as_float(sr[cc]), sl2, nlse2)) : 0.f;
          }
        }
      }
      // phase 2: dS = P o (dP - Delta), 32 columns at a time, packed over the dP columns
      // already read, in this tile's buffer
      const uint32_t buf = j & 1 ? 384 : 128;
      if (!wait_all(&bars->dp_full[j & 1], (j >> 1) & 1, abort_flag, a.err)) { ok = false; break; }
      ptx::tc_fence_after();
#pragma unroll
      for (int hc = 0; hc < 64; hc += 32) {
        uint32_t dr[32];
        ptx::tmem_ld32(lane_addr + buf + cb + hc, dr);
        ptx::tmem_wait_ld_regs(dr);
        uint32_t dd[16];
        if (fast) {
#pragma unroll
          for (int cc = 0; cc < 32; cc += 2) {
            const uint64_t tt = ptx::fadd2(ptx::f2_pack(__uint_as_float(dr[cc]), __uint_as_float(dr[cc + 1])),
                                           nd2x2);
            float ds0, ds1;
            ptx::f2_unpack(ptx::fmul2(ptx::f2_pack(p[hc + cc], p[hc + cc + 1]), tt), ds0, ds1);
            dd[cc / 2] = ptx::pack_bf16x2(ds0, ds1);
          }
        } else {
#pragma unroll
          for (int cc = 0; cc < 32; cc += 2) {
            const int col = cb + hc + cc;
            const bool v0 = col >= ilo && col <= ihi, v1 = col + 1 >= ilo && col + 1 <= ihi;
            const float ds0 = v0 ? p[hc + cc] * (__uint_as_float(dr[cc]) - delta) : 0.f;
            const float ds1 = v1 ? p[hc + cc + 1] * (__uint_as_float(dr[cc + 1]) - delta) : 0.f;
            dd[cc / 2] = ptx::pack_bf16x2(ds0, ds1);
          }
        }
        ptx::tmem_st16(lane_addr + buf + cb + hc / 2, dd);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&bars->ds_full[j & 1]);
      ++j;
    }
    // ------------------------------------------------------------ dQ epilogue
    ok = ok && __all_sync(0xffffffffu, *abort_flag == 0);
    if (ok) ok = wait_all(&bars->done, 0, abort_flag, a.err);
    if (ok) {
      ptx::tc_fence_after();
      const int64_t qrow = (int64_t)(q_row0 + i0 + r) * a.q_ld + (int64_t)h * D;
      float* dst = a.dq_acc + qrow;
      __nv_bfloat16* dst_bf = a.dq_out ? static_cast<__nv_bfloat16*>(a.dq_out) + qrow : nullptr;
#pragma unroll
      for (int ch = w * (D / 64); ch < (w + 1) * (D / 64); ++ch) {  // D/2 columns per warpgroup
        uint32_t rr[32];
        if (j > 0) {
          ptx::tmem_ld32(lane_addr + 256 + ch * 32, rr);
          ptx::tmem_wait_ld_regs(rr);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) rr[i] = 0u;
        }
        if (!CP_DCHECK(!row_valid || (int64_t)q_row0 + i0 + r < a.q_rows, a.err)) {
          // out of the q rows: skipped (debug builds)
        } else if (row_valid && dst_bf) {
          store_row_bf16(dst_bf + ch * 32, rr, a.scale);
        } else if (row_valid) {
          store_row_f32(dst + ch * 32, rr, a.scale, a.accumulate);
        }
      }
    }
    ptx::tc_fence_before();
  }

  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ====================================================================== host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D map over a [rows, H*D] bf16 buffer; box 64 columns x 128 rows, 128-byte swizzle.
cp_status make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) {
    set_last_error("cuTensorMapEncodeTiled unavailable from the driver");
    return CP_ERR_CUDA;
  }
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kTileRows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_last_error("cuTensorMapEncodeTiled failed (code " + std::to_string((int)r) + ")");
    return CP_ERR_CUDA;
  }
  return CP_OK;
}

// Turns a key-major schedule (group = key run, segments = query runs) into the
// query-major one (group = query run, segments = key runs) with the same pairs.
bool invert_schedule(const Schedule& km, Schedule& qm) {
  struct Run {
    int32_t row0, n, pos_off, pos_stride;
    bool operator==(const Run& o) const {
      return row0 == o.row0 && n == o.n && pos_off == o.pos_off && pos_stride == o.pos_stride;
    }
  };
  std::vector<Run> qruns;
  std::vector<std::vector<Run>> keys_of;
  for (int gi = 0; gi < km.n_groups; ++gi) {
    const QGroup& kg = km.g[gi];
    Run kr{kg.q_row0, kg.nq, kg.pos_off, kg.pos_stride};
    for (int si = 0; si < kg.seg_count; ++si) {
      const KSeg& qs = km.s[kg.seg_begin + si];
      Run qr{qs.k_row0, qs.nk, qs.pos_off, qs.pos_stride};
      size_t idx = 0;
      while (idx < qruns.size() && !(qruns[idx] == qr)) ++idx;
      if (idx == qruns.size()) {
        qruns.push_back(qr);
        keys_of.emplace_back();
      }
      keys_of[idx].push_back(kr);
    }
  }
  if ((int)qruns.size() > kMaxGroups) return false;
  qm.n_groups = 0;
  qm.n_segs = 0;
  for (size_t i = 0; i < qruns.size(); ++i) {
    QGroup& g = qm.g[qm.n_groups++];
    memset(&g, 0, sizeof(g));
    g.q_row0 = qruns[i].row0;
    g.nq = qruns[i].n;
    g.pos_off = qruns[i].pos_off;
    g.pos_stride = qruns[i].pos_stride;
    g.seg_begin = qm.n_segs;
    for (const Run& kr : keys_of[i]) {
      if (qm.n_segs >= kMaxSegs) return false;
      KSeg& sg = qm.s[qm.n_segs++];
      sg.k_row0 = kr.row0;
      sg.nk = kr.n;
      sg.pos_off = kr.pos_off;
      sg.pos_stride = kr.pos_stride;
      g.seg_count++;
    }
  }
  return true;
}

// Key/value heads per block of a backward launch order (decode_unit_blocked): the
// most whole key/value heads, a divisor of Hkv, whose shared operand bytes (the
// other side's rows a unit reads: Q and dO of the head's query heads for dK/dV, K
// and V for dQ) fit kL2SharedBytes together.  Every head fastest (one block) when
// the groups read disjoint rows of the other side (Ulysses' ranks) or with packed
// documents, as in the forward.
#ifndef CP_DEBUG
constexpr int64_t kL2SharedBytes = 128ll << 20;
#else
constexpr int64_t kL2SharedBytes = 1;  // debug build: one key/value head per block at any size
#endif
int kv_heads_per_block(const Schedule& s, const BwdArgs& a, int64_t other_rows, int64_t bytes_per_kv_head) {
  int64_t other_max = 0;
  for (int i = 0; i < s.n_groups; ++i) {
    int64_t n = 0;
    for (int j = s.g[i].seg_begin; j < s.g[i].seg_begin + s.g[i].seg_count; ++j) n += s.s[j].nk;
    other_max = std::max(other_max, n);
  }
  if (a.cu_seqlens || 2 * other_max < other_rows) return a.Hkv;
  int kb = (int)std::min<int64_t>(a.Hkv, std::max<int64_t>(1, kL2SharedBytes / std::max<int64_t>(1, bytes_per_kv_head)));
  while (a.Hkv % kb) --kb;
  return kb;
}

template <int HD>
cp_status launch_typed(const BwdArgs& a, Schedule& s, int64_t q_rows, int64_t k_rows, cudaStream_t st) {
  // setmaxnreg.inc waits until the registers it asks for are free in the block's launch
  // budget, so launch only if each kernel's compiled register count covers the split.
  const bool win = a.window > 0;
  auto dkdv_kernel = win ? attn_bwd_dkdv_kernel<HD, true> : attn_bwd_dkdv_kernel<HD, false>;
  auto dq_kernel = win ? attn_bwd_dq_kernel<HD, true> : attn_bwd_dq_kernel<HD, false>;
  for (const void* kfn : {(const void*)dkdv_kernel, (const void*)dq_kernel}) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kfn);
    if (e != cudaSuccess) return cuda_check(e, "cudaFuncGetAttributes(attn_bwd)");
    if ((int64_t)fa.numRegs * kThreads < 128 * kRegsLow + 256 * kRegsHigh) {
      set_last_error("attention backward compiled with " + std::to_string(fa.numRegs) +
                     " registers per thread, too few for its warpgroup register split");
      return CP_ERR_UNSUPPORTED;
    }
  }
  CUtensorMap mq, mdo, mk, mv;
  cp_status r;
  if ((r = make_map(&mq, a.q, q_rows, (int64_t)a.Hq * HD)) != CP_OK) return r;
  if ((r = make_map(&mdo, a.dout, q_rows, (int64_t)a.Hq * HD)) != CP_OK) return r;
  if ((r = make_map(&mk, a.k, k_rows, (int64_t)a.Hkv * HD)) != CP_OK) return r;
  if ((r = make_map(&mv, a.v, k_rows, (int64_t)a.Hkv * HD)) != CP_OK) return r;

  // dK / dV over the key-major schedule
  BwdArgs ab = a;
  int64_t units = schedule_units(s, kTileRows, a.Hkv);
  schedule_order(s, kTileRows, kTileRows, true, a.causal, a.window, a.cu_seqlens != nullptr);
  ab.kv_pairs = (int32_t)(units / a.Hkv);
  ab.kv_head_block = kv_heads_per_block(s, a, q_rows, (int64_t)(a.Hq / a.Hkv) * HD * 2 * 2 * q_rows);
  if (units > 0) {
    cudaError_t e = cudaFuncSetAttribute(dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         ALayout<HD>::kSmemRequest);
    if (e != cudaSuccess) return cuda_check(e, "cudaFuncSetAttribute(attn_bwd_dkdv)");
    dkdv_kernel<<<(unsigned)units, kThreads, ALayout<HD>::kSmemRequest, st>>>(ab, s, mq, mdo, mk, mv);
    if ((r = cuda_check(cudaGetLastError(), "attn_bwd_dkdv_kernel launch")) != CP_OK) return r;
  }
  // dQ over the query-major schedule (same pairs)
  Schedule* qm = new Schedule;
  if (!invert_schedule(s, *qm)) {
    delete qm;
    set_last_error("backward schedule too large to invert");
    return CP_ERR_UNSUPPORTED;
  }
  units = schedule_units(*qm, kTileRows, a.Hq);
  schedule_order(*qm, kTileRows, kTileRows, false, a.causal, a.window, a.cu_seqlens != nullptr);
  ab.q_pairs = (int32_t)(units / a.Hq);
  ab.q_head_block = (a.Hq / a.Hkv) * kv_heads_per_block(*qm, a, k_rows, (int64_t)HD * 2 * 2 * k_rows);
  if (units > 0) {
    cudaError_t e = cudaFuncSetAttribute(dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         BLayout<HD>::kSmemRequest);
    if (e != cudaSuccess) {
      delete qm;
      return cuda_check(e, "cudaFuncSetAttribute(attn_bwd_dq)");
    }
    dq_kernel<<<(unsigned)units, kThreads, BLayout<HD>::kSmemRequest, st>>>(ab, *qm, mq, mdo, mk, mv);
    r = cuda_check(cudaGetLastError(), "attn_bwd_dq_kernel launch");
  }
  delete qm;
  return r;
}

}  // namespace

cp_status launch_attn_bwd_tc(const BwdArgs& a, Schedule& s, int64_t q_rows, int64_t k_rows,
                             cudaStream_t st) {
  if (a.D == 128) return launch_typed<128>(a, s, q_rows, k_rows, st);
  if (a.D == 64) return launch_typed<64>(a, s, q_rows, k_rows, st);
  set_last_error("tcgen05 attention backward supports D = 64 or 128");
  return CP_ERR_UNSUPPORTED;
}

}  // namespace cpa
