// tcgen05 block attention backward for bf16 (fp32 accumulation), D = 128.
//
// The exact derivative of the handbook's attention ("Context parallelism:
// Ring Attention and Ulysses", section "Which operations partition
// directly"; the pages give no backward), given the FINAL out and lse of
// every query row (for a ring: the merged ones):
//   P = exp(scale*S - lse),  dV = P^T dO,  dP = dO V^T,
//   dS = P o (dP - Delta),   Delta = rowsum(dO o O),
//   dQ = scale * dS K,       dK = scale * dS^T Q.
//
// Two kernels, neither uses atomics (gradients are deterministic):
//
// attn_bwd_dkdv_kernel: one CTA = one 128-key tile of one key/value head,
//   looping over the G query heads that read it and every 64-row query tile
//   that can see the keys (a key-major schedule: group = key run, segments =
//   query runs).  Per query tile:
//     S^T  = K Q^T, dP^T = V dO^T  -> TMEM, double-buffered (cols 0..255)
//     softmax warps (thread = key row): P^T and dS^T (bf16) written back over
//       the S^T / dP^T columns they came from
//     dV += P^T dO, dK += dS^T Q   -> TMEM accumulators (cols 256..511), with
//       P^T and dS^T as the TMEM A operand; issued after the NEXT tile's S^T so
//       the softmax of one tile overlaps the products of its neighbours
//   dK and dV are stored once at the end.  lse and Delta of each query tile
//   are staged in shared memory by the producer warp with the Q/dO tiles.
//
// attn_bwd_dq_kernel: one CTA = one 128-row query tile of one query head,
//   walking every 64-key tile it sees (a query-major schedule, as in the
//   forward).  Per key tile:
//     S = Q K^T, dP = dO V^T       -> TMEM, double-buffered (cols 0..255)
//     softmax warps (thread = query row): dS (bf16) written over the dP columns
//     dQ += dS K                   -> TMEM accumulator (cols 256..383), dS as
//       the TMEM A operand
//   dQ is stored once at the end.
//
// This recomputes S and dP once more than a single fused kernel (7 instead of
// 5 matrix products) in exchange for no fp32 atomic traffic on dQ.
// Warps: 0..3 and 4..7 are two softmax warpgroups that take alternate tiles
// (two independent MMA -> softmax -> MMA chains per CTA, so each hides the
// other's hand-off latency), each with its own TMEM S/dP buffer; 8 TMA
// producer, 9 MMA issuer (one thread); the third warpgroup gives registers to
// the softmax ones (setmaxnreg).
// Every mbarrier wait is bounded (as in the forward kernel).
#include <cuda.h>

#include <vector>

#include "common.cuh"
#include "ptx.cuh"

namespace cpa {
namespace {

constexpr int D = 128;
constexpr int kThreads = 384;       // warps 0..7 softmax (two warpgroups), 8 TMA, 9 MMA, 10..11 spare
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kWgThreads = 128;
// Register split (launch: 384 x 168 = 64512): the TMA/MMA warpgroup drops to 88, the
// two softmax warpgroups rise to 208: 128*88 + 256*208 = 64512.
constexpr int kRegsLow = 88;
constexpr int kRegsHigh = 208;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint64_t kDrainNs = 200000000ull;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint64_t desc_k(uint32_t base, int kk, uint32_t region_bytes) {
  // K-major, 128B swizzle: K step of 16 bf16 = 32 bytes inside a 64-column region.
  return ptx::smem_desc_sw128(base + (kk >> 2) * region_bytes + (kk & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t desc_mn(uint32_t base, int kk, uint32_t lbo) {
  // MN-major, 128B swizzle: K step of 16 rows of 128 bytes; next 64 MN columns at +lbo.
  return ptx::smem_desc_sw128(base + kk * (16 * 128), lbo, 1024);
}

__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t par, volatile int* abort_flag,
                                         int32_t* err) {
  bool ok = ptx::mbar_wait_bounded(bar, par, abort_flag, err, kWaitNs);
  return __all_sync(0xffffffffu, ok);
}

// ====================================================================== dK / dV

constexpr int A_BK = 128;  // keys per CTA
constexpr int A_BQ = 64;   // queries per tile
constexpr int A_QST = 3;   // Q/dO stages

struct ALayout {
  static constexpr int kKV = A_BK * D * 2;       // 32 KB
  static constexpr int kQT = A_BQ * D * 2;       // 16 KB
  static constexpr int kK = 0;
  static constexpr int kV = kK + kKV;
  static constexpr int kQ = kV + kKV;            // A_QST stages
  static constexpr int kDO = kQ + A_QST * kQT;   // A_QST stages
  static constexpr int kLse = kDO + A_QST * kQT;  // A_QST x (64 lse*log2e, 64 Delta)
  static constexpr int kBar = kLse + A_QST * 2 * A_BQ * 4;
  static constexpr int kBytes = kBar + 256;
  static constexpr int kSmemRequest = kBytes + 1024;
};

struct ABars {
  uint64_t kv_full;
  uint64_t q_full[A_QST], q_empty[A_QST];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t done;  // every MMA of the CTA has completed
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
  int64_t en_lo;  // end of the document holding pk_lo
  int causal, docs;
  int G, hk;
};

// Next query tile (over the G query heads, then the query runs) that sees some key of the tile.
__device__ __forceinline__ bool next_qtile(const Schedule& s, const KeyCtx& c, int seg_begin,
                                           int seg_end, int& hh, int& seg, int& i0, QTile& t) {
  while (hh < c.G) {
    if (seg >= seg_end) {
      ++hh;
      seg = seg_begin;
      i0 = 0;
      continue;
    }
    const int32_t q_row0 = s.s[seg].k_row0, nq_seg = s.s[seg].nk;
    const int32_t poff = s.s[seg].pos_off, pst = s.s[seg].pos_stride;
    if (i0 >= nq_seg) {
      ++seg;
      i0 = 0;
      continue;
    }
    const int nq = min(A_BQ, nq_seg - i0);
    const int64_t pq_lo = (int64_t)poff + (int64_t)pst * i0;
    const int64_t pq_hi = pq_lo + (int64_t)pst * (nq - 1);
    const int icur = i0;
    i0 += A_BQ;
    if (c.causal && pq_hi < c.pk_lo) continue;  // every query before every key
    t.q_row = q_row0 + icur;
    t.nq = nq;
    t.pq_lo = pq_lo;
    t.qstride = pst;
    t.h = c.hk * c.G + hh;
    t.full = (nq == A_BQ) && (c.causal ? pq_lo >= c.pk_hi : 1) && !c.docs;
    if (c.docs && c.causal) t.full = (nq == A_BQ) && pq_lo >= c.pk_hi && c.en_lo > pq_hi;
    return true;
  }
  return false;
}

__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_dkdv_kernel(const __grid_constant__ BwdArgs a, const __grid_constant__ Schedule s,
                     const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  using L = ALayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  ABars* bars = reinterpret_cast<ABars*>(smem + L::kBar);
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* lse_all = reinterpret_cast<float*>(smem + L::kLse);

  int g, tile, hk;
  decode_unit(s, A_BK, a.Hkv, blockIdx.x, &g, &tile, &hk);
  const int32_t k_row0 = s.g[g].q_row0 + tile * A_BK;  // key-major schedule: group = key run
  const int nk_tile = min(A_BK, s.g[g].nq - tile * A_BK);
  const int seg_begin = s.g[g].seg_begin, seg_end = seg_begin + s.g[g].seg_count;

  KeyCtx c;
  c.causal = a.causal;
  c.docs = a.cu_seqlens != nullptr;
  c.G = a.Hq / a.Hkv;
  c.hk = hk;
  c.pk_lo = (int64_t)s.g[g].pos_off + (int64_t)s.g[g].pos_stride * (tile * A_BK);
  c.pk_hi = c.pk_lo + (int64_t)s.g[g].pos_stride * (nk_tile - 1);
  c.en_lo = INT64_MAX;
  if (c.docs) {
    int64_t st;
    doc_bounds(a.cu_seqlens, a.n_docs, c.pk_lo, &st, &c.en_lo);
  }

  if (threadIdx.x == 0) {
    ptx::mbar_init(&bars->kv_full, 1);
    for (int i = 0; i < A_QST; ++i) {
      ptx::mbar_init(&bars->q_full[i], 2);  // TMA (expect_tx) + the warp's lse/Delta stores
      ptx::mbar_init(&bars->q_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&bars->s_full[i], 1);
      ptx::mbar_init(&bars->p_full[i], kWgThreads);
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
    // ------------------------------------------------------------ producer (whole warp)
    if (lane == 0) {
      ptx::mbar_arrive_expect_tx(&bars->kv_full, 2 * L::kKV);
      for (int r = 0; r < D / 64; ++r) {
        ptx::tma_load_2d(smem + L::kK + r * 16384, &tm_k, &bars->kv_full, hk * D + r * 64, k_row0);
        ptx::tma_load_2d(smem + L::kV + r * 16384, &tm_v, &bars->kv_full, hk * D + r * 64, k_row0);
      }
    }
    int hh = 0, seg = seg_begin, i0 = 0, j = 0;
    QTile t;
    int issued[A_QST] = {0, 0, 0};
    while (__all_sync(0xffffffffu, *abort_flag == 0) &&
           next_qtile(s, c, seg_begin, seg_end, hh, seg, i0, t)) {
      const int st = j % A_QST;
      if (j >= A_QST && !wait_all(&bars->q_empty[st], ((j / A_QST) - 1) & 1, abort_flag, a.err)) break;
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(&bars->q_full[st], 2 * L::kQT);
        for (int r = 0; r < D / 64; ++r) {
          ptx::tma_load_2d(smem + L::kQ + st * L::kQT + r * 8192, &tm_q, &bars->q_full[st],
                           t.h * D + r * 64, t.q_row);
          ptx::tma_load_2d(smem + L::kDO + st * L::kQT + r * 8192, &tm_do, &bars->q_full[st],
                           t.h * D + r * 64, t.q_row);
        }
      }
      float* lse_st = lse_all + st * 2 * A_BQ;
      for (int cidx = lane; cidx < A_BQ; cidx += 32) {
        float lv = INFINITY, dv = 0.f;  // +inf: rows past the run (or seeing nothing) get P = 0
        if (cidx < t.nq) {
          const float Lr = a.lse[(int64_t)t.h * a.lse_ld + t.q_row + cidx];
          lv = (Lr == -INFINITY) ? INFINITY : Lr * kLog2e;
          dv = a.delta[(int64_t)t.h * a.lse_ld + t.q_row + cidx];
        }
        lse_st[cidx] = lv;
        lse_st[A_BQ + cidx] = dv;
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bars->q_full[st]);
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
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = ptx::idesc_bf16_f32(128, A_BQ, 0, 0);  // K Q^T, V dO^T
      constexpr uint32_t id_kv = ptx::idesc_bf16_f32(128, D, 0, 1);    // P^T dO, dS^T Q (TMEM A)
      const uint32_t k_addr = sbase + L::kK, v_addr = sbase + L::kV;
      bool issued = false;
      // S^T and dP^T of query tile jj into TMEM buffer jj & 1
      auto issue_s = [&](int jj) -> bool {
        const int st = jj % A_QST, b = jj & 1;
        if (!ptx::mbar_wait_bounded(&bars->q_full[st], (jj / A_QST) & 1, abort_flag, a.err, kWaitNs))
          return false;
        ptx::tc_fence_after();
        const uint32_t q_addr = sbase + L::kQ + st * L::kQT;
        const uint32_t do_addr = sbase + L::kDO + st * L::kQT;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_bf16_ss(tmem + b * 128, desc_k(k_addr, kk, 16384), desc_k(q_addr, kk, 8192), id_s,
                           kk > 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_bf16_ss(tmem + b * 128 + 64, desc_k(v_addr, kk, 16384), desc_k(do_addr, kk, 8192),
                           id_s, kk > 0);
        ptx::tc_commit(&bars->s_full[b]);
        issued = true;
        return true;
      };
      if (ptx::mbar_wait_bounded(&bars->kv_full, 0, abort_flag, a.err, kWaitNs)) {
        int hh = 0, seg = seg_begin, i0 = 0;
        QTile t;
        int found = 0;  // query tiles the iterator has produced so far
        bool exhausted = false;
        auto advance = [&]() {
          if (!exhausted) {
            if (next_qtile(s, c, seg_begin, seg_end, hh, seg, i0, t)) ++found;
            else exhausted = true;
          }
        };
        bool fail = false;
        advance();
        if (found > 0 && !issue_s(0)) fail = true;
        advance();
        if (!fail && found > 1 && !issue_s(1)) fail = true;
        for (int j = 0; !fail && j < found; ++j) {
          const int b = j & 1, st = j % A_QST;
          if (!ptx::mbar_wait_bounded(&bars->p_full[b], (j >> 1) & 1, abort_flag, a.err, kWaitNs)) break;
          ptx::tc_fence_after();
          const uint32_t q_addr = sbase + L::kQ + st * L::kQT;
          const uint32_t do_addr = sbase + L::kDO + st * L::kQT;
          // P^T / dS^T: 64 queries packed two per column (K step kk = 8 columns)
#pragma unroll
          for (int kk = 0; kk < A_BQ / 16; ++kk)
            ptx::mma_bf16_ts(tmem + 256, tmem + b * 128 + kk * 8, desc_mn(do_addr, kk, 8192), id_kv,
                             (j > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < A_BQ / 16; ++kk)
            ptx::mma_bf16_ts(tmem + 384, tmem + b * 128 + 64 + kk * 8, desc_mn(q_addr, kk, 8192), id_kv,
                             (j > 0 || kk > 0) ? 1u : 0u);
          ptx::tc_commit(&bars->q_empty[st]);
          advance();
          if (found > j + 2 && !issue_s(j + 2)) break;  // reuses buffer b after these products
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
    const int w = warp >> 2;  // this warpgroup takes the query tiles j with j % 2 == w
    const int r = quad * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
    const int64_t pk = c.pk_lo + (int64_t)s.g[g].pos_stride * r;
    int64_t st_k = 0, en_k = INT64_MAX;
    if (c.docs && r < nk_tile) doc_bounds(a.cu_seqlens, a.n_docs, pk, &st_k, &en_k);
    const float sl2 = a.scale_log2;
    int hh = 0, seg = seg_begin, i0 = 0, j = 0;
    QTile t;
    bool ok = true;
    while (__all_sync(0xffffffffu, *abort_flag == 0) &&
           next_qtile(s, c, seg_begin, seg_end, hh, seg, i0, t)) {
      if ((j & 1) != w) {
        ++j;
        continue;
      }
      const int st = j % A_QST, b = w;
      int64_t hi = t.nq - 1, lo = 0;  // visible query columns of this key row: [lo, hi]
      if (r >= nk_tile) {
        hi = -1;
      } else if (!t.full) {
        if (c.causal) {
          const int64_t d0 = pk - t.pq_lo;  // need pq >= pk
          lo = max(lo, d0 <= 0 ? (int64_t)0 : (d0 + t.qstride - 1) / t.qstride);
        }
        if (c.docs) {
          const int64_t d1 = en_k - 1 - t.pq_lo;  // need pq < end of the key's document
          hi = min(hi, d1 < 0 ? (int64_t)-1 : d1 / t.qstride);
          if (!c.causal) {  // and pq >= start of the key's document
            const int64_t d2 = st_k - t.pq_lo;
            lo = max(lo, d2 <= 0 ? (int64_t)0 : (d2 + t.qstride - 1) / t.qstride);
          }
        }
      }
      const int ilo = (int)lo, ihi = (int)max(hi, (int64_t)-1);
      // lse/Delta of this tile were stored by the producer before q_full completed
      if (!wait_all(&bars->q_full[st], (j / A_QST) & 1, abort_flag, a.err)) { ok = false; break; }
      if (!wait_all(&bars->s_full[b], (j >> 1) & 1, abort_flag, a.err)) { ok = false; break; }
      ptx::tc_fence_after();
      uint32_t sr[2][32], dr[2][32];
      ptx::tmem_ld32(lane_addr + b * 128 + 0, sr[0]);
      ptx::tmem_ld32(lane_addr + b * 128 + 32, sr[1]);
      ptx::tmem_ld32(lane_addr + b * 128 + 64, dr[0]);
      ptx::tmem_ld32(lane_addr + b * 128 + 96, dr[1]);
      ptx::tmem_wait_ld_regs(sr[0]);
      ptx::tmem_wait_ld_regs(sr[1]);
      ptx::tmem_wait_ld_regs(dr[0]);
      ptx::tmem_wait_ld_regs(dr[1]);
      const float* lse_st = lse_all + st * 2 * A_BQ;
      uint32_t pp[32], dd[32];
#pragma unroll
      for (int cc = 0; cc < A_BQ; cc += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(lse_st + cc);
        const float4 d4 = *reinterpret_cast<const float4*>(lse_st + A_BQ + cc);
        const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
        const float dl[4] = {d4.x, d4.y, d4.z, d4.w};
        float p[4], ds[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int col = cc + u;
          const float sv = __uint_as_float(sr[col >> 5][col & 31]);
          const float dp = __uint_as_float(dr[col >> 5][col & 31]);
          p[u] = (col >= ilo && col <= ihi) ? ptx::ex2_approx(fmaf(sv, sl2, -lv[u])) : 0.f;
          ds[u] = p[u] * (dp - dl[u]);
        }
        pp[cc / 2] = ptx::pack_bf16x2(p[0], p[1]);
        pp[cc / 2 + 1] = ptx::pack_bf16x2(p[2], p[3]);
        dd[cc / 2] = ptx::pack_bf16x2(ds[0], ds[1]);
        dd[cc / 2 + 1] = ptx::pack_bf16x2(ds[2], ds[3]);
      }
      // P^T and dS^T (two bf16 per column) over the S^T / dP^T columns just read
      ptx::tmem_st32(lane_addr + b * 128, pp);
      ptx::tmem_st32(lane_addr + b * 128 + 64, dd);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&bars->p_full[b]);
      ++j;
    }
    // ------------------------------------------------------------ dK / dV epilogue
    ok = ok && __all_sync(0xffffffffu, *abort_flag == 0);
    if (ok) ok = wait_all(&bars->done, 0, abort_flag, a.err);
    if (ok) {
      ptx::tc_fence_after();
      const bool valid = r < nk_tile;
      const int64_t krow = (int64_t)(k_row0 + r) * a.k_ld + (int64_t)hk * D;
      {
        const int which = warp >> 2;  // warpgroup 0 stores dV, warpgroup 1 stores dK
        float* dst = (which == 0 ? a.dv_acc : a.dk_acc) + krow;
        const float mul = which == 0 ? 1.f : a.scale;
        const uint32_t col0 = which == 0 ? 256 : 384;
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
          if (valid) {
            float4* d4 = reinterpret_cast<float4*>(dst + ch * 32);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              d4[v4] = make_float4(__uint_as_float(rr[4 * v4]) * mul, __uint_as_float(rr[4 * v4 + 1]) * mul,
                                   __uint_as_float(rr[4 * v4 + 2]) * mul, __uint_as_float(rr[4 * v4 + 3]) * mul);
          }
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

constexpr int B_BQ = 128;  // query rows per CTA
constexpr int B_BN = 64;   // keys per tile
constexpr int B_KST = 3;   // K/V stages

struct BLayout {
  static constexpr int kQT = B_BQ * D * 2;   // 32 KB
  static constexpr int kKT = B_BN * D * 2;   // 16 KB
  static constexpr int kQ = 0;
  static constexpr int kDO = kQ + kQT;
  static constexpr int kK = kDO + kQT;       // B_KST stages
  static constexpr int kV = kK + B_KST * kKT;
  static constexpr int kBar = kV + B_KST * kKT;
  static constexpr int kBytes = kBar + 256;
  static constexpr int kSmemRequest = kBytes + 1024;
};

struct BBars {
  uint64_t q_full;
  uint64_t k_full[B_KST], v_full[B_KST], kv_empty[B_KST];
  uint64_t s_full[2];
  uint64_t ds_full[2];
  uint64_t done;  // every MMA of the CTA has completed
  uint32_t tmem_base;
  int abort_flag;
};

struct TileCtx {
  int64_t pq_lo, pq_hi;
  int64_t st_lo, st_hi, en_lo, en_hi;
  int causal, docs;
};

struct KvTile {
  int32_t k_row;
  int32_t nk;
  int64_t pk_lo;
  int32_t kstride;
  int32_t full;
};

// Next key/value tile (64 keys) of the query group with any visible pair.
__device__ __forceinline__ bool next_ktile(const Schedule& s, const TileCtx& c, int seg_end, int& seg,
                                           int& j0, KvTile& t) {
  while (seg < seg_end) {
    const int32_t k_row0 = s.s[seg].k_row0, nk_seg = s.s[seg].nk;
    const int32_t poff = s.s[seg].pos_off, pst = s.s[seg].pos_stride;
    if (j0 >= nk_seg) {
      ++seg;
      j0 = 0;
      continue;
    }
    const int nk = min(B_BN, nk_seg - j0);
    const int64_t pk_lo = (int64_t)poff + (int64_t)pst * j0;
    const int64_t pk_hi = pk_lo + (int64_t)pst * (nk - 1);
    const int jcur = j0;
    j0 += B_BN;
    if ((c.causal && pk_lo > c.pq_hi) || (c.docs && pk_lo >= c.en_hi)) {
      ++seg;
      j0 = 0;
      continue;
    }
    if (c.docs && pk_hi < c.st_lo) continue;
    t.k_row = k_row0 + jcur;
    t.nk = nk;
    t.pk_lo = pk_lo;
    t.kstride = pst;
    t.full = (nk == B_BN) && (!c.causal || pk_hi <= c.pq_lo) &&
             (!c.docs || (pk_lo >= c.st_hi && pk_hi < c.en_lo));
    return true;
  }
  return false;
}

__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_dq_kernel(const __grid_constant__ BwdArgs a, const __grid_constant__ Schedule s,
                   const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  using L = BLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  BBars* bars = reinterpret_cast<BBars*>(smem + L::kBar);
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  int g, tile, h;
  decode_unit(s, B_BQ, a.Hq, blockIdx.x, &g, &tile, &h);
  const int hk = h / (a.Hq / a.Hkv);
  const int32_t q_row0 = s.g[g].q_row0, nq = s.g[g].nq;
  const int32_t qpos_off = s.g[g].pos_off, qpos_st = s.g[g].pos_stride;
  const int seg_begin = s.g[g].seg_begin, seg_end = seg_begin + s.g[g].seg_count;
  const int i0 = tile * B_BQ;
  const int nq_tile = min(B_BQ, nq - i0);

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

  if (threadIdx.x == 0) {
    ptx::mbar_init(&bars->q_full, 1);
    for (int i = 0; i < B_KST; ++i) {
      ptx::mbar_init(&bars->k_full[i], 1);
      ptx::mbar_init(&bars->v_full[i], 1);
      ptx::mbar_init(&bars->kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&bars->s_full[i], 1);
      ptx::mbar_init(&bars->ds_full[i], kWgThreads);
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
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      ptx::mbar_arrive_expect_tx(&bars->q_full, 2 * L::kQT);
      for (int r = 0; r < D / 64; ++r) {
        ptx::tma_load_2d(smem + L::kQ + r * 16384, &tm_q, &bars->q_full, h * D + r * 64, q_row0 + i0);
        ptx::tma_load_2d(smem + L::kDO + r * 16384, &tm_do, &bars->q_full, h * D + r * 64, q_row0 + i0);
      }
      int seg = seg_begin, j0 = 0, j = 0;
      KvTile t;
      int issued[B_KST] = {0, 0, 0};
      while (!*abort_flag && next_ktile(s, c, seg_end, seg, j0, t)) {
        const int st = j % B_KST;
        if (j >= B_KST && !ptx::mbar_wait_bounded(&bars->kv_empty[st], ((j / B_KST) - 1) & 1, abort_flag,
                                                   a.err, kWaitNs))
          break;
        ptx::mbar_arrive_expect_tx(&bars->k_full[st], L::kKT);
        for (int r = 0; r < D / 64; ++r)
          ptx::tma_load_2d(smem + L::kK + st * L::kKT + r * 8192, &tm_k, &bars->k_full[st],
                           hk * D + r * 64, t.k_row);
        ptx::mbar_arrive_expect_tx(&bars->v_full[st], L::kKT);
        for (int r = 0; r < D / 64; ++r)
          ptx::tma_load_2d(smem + L::kV + st * L::kKT + r * 8192, &tm_v, &bars->v_full[st],
                           hk * D + r * 64, t.k_row);
        issued[st] = j + 1;
        ++j;
      }
      if (*abort_flag) {
        (void)ptx::mbar_wait_bounded(&bars->q_full, 0, nullptr, nullptr, kDrainNs);
        for (int st = 0; st < B_KST; ++st)
          if (issued[st] > 0) {
            const uint32_t par = ((issued[st] - 1) / B_KST) & 1;
            (void)ptx::mbar_wait_bounded(&bars->k_full[st], par, nullptr, nullptr, kDrainNs);
            (void)ptx::mbar_wait_bounded(&bars->v_full[st], par, nullptr, nullptr, kDrainNs);
          }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = ptx::idesc_bf16_f32(B_BQ, B_BN, 0, 0);  // Q K^T, dO V^T
      constexpr uint32_t id_q = ptx::idesc_bf16_f32(B_BQ, D, 0, 1);     // dS K
      const uint32_t q_addr = sbase + L::kQ, do_addr = sbase + L::kDO;
      bool any = false;
      if (ptx::mbar_wait_bounded(&bars->q_full, 0, abort_flag, a.err, kWaitNs)) {
        int seg = seg_begin, j0 = 0, j = 0;
        KvTile t;
        bool more = next_ktile(s, c, seg_end, seg, j0, t);
        while (true) {
          if (more) {
            const int st = j % B_KST, b = j & 1;
            if (!ptx::mbar_wait_bounded(&bars->k_full[st], (j / B_KST) & 1, abort_flag, a.err, kWaitNs))
              break;
            if (!ptx::mbar_wait_bounded(&bars->v_full[st], (j / B_KST) & 1, abort_flag, a.err, kWaitNs))
              break;
            ptx::tc_fence_after();
            const uint32_t k_addr = sbase + L::kK + st * L::kKT;
            const uint32_t v_addr = sbase + L::kV + st * L::kKT;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              ptx::mma_bf16_ss(tmem + b * 128, desc_k(q_addr, kk, 16384), desc_k(k_addr, kk, 8192), id_s,
                               kk > 0);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              ptx::mma_bf16_ss(tmem + b * 128 + 64, desc_k(do_addr, kk, 16384), desc_k(v_addr, kk, 8192),
                               id_s, kk > 0);
            ptx::tc_commit(&bars->s_full[b]);
            any = true;
          }
          if (j >= 1) {
            const int jp = j - 1, stp = jp % B_KST, bp = jp & 1;
            if (!ptx::mbar_wait_bounded(&bars->ds_full[bp], (jp >> 1) & 1, abort_flag, a.err, kWaitNs))
              break;
            ptx::tc_fence_after();
            const uint32_t k_addr = sbase + L::kK + stp * L::kKT;
            // dS: 64 keys packed two per column over the dP columns (K step kk = 8 columns)
#pragma unroll
            for (int kk = 0; kk < B_BN / 16; ++kk)
              ptx::mma_bf16_ts(tmem + 256, tmem + bp * 128 + 64 + kk * 8, desc_mn(k_addr, kk, 8192), id_q,
                               (jp > 0 || kk > 0) ? 1u : 0u);
            ptx::tc_commit(&bars->kv_empty[stp]);
          }
          if (!more) break;
          ++j;
          more = next_ktile(s, c, seg_end, seg, j0, t);
        }
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
    const int w = warp >> 2;  // this warpgroup takes the key tiles j with j % 2 == w
    const int r = quad * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
    const int64_t pq = c.pq_lo + (int64_t)qpos_st * r;
    const bool row_valid = r < nq_tile;
    int64_t st_r = 0, en_r = 0;
    if (c.docs && row_valid) doc_bounds(a.cu_seqlens, a.n_docs, pq, &st_r, &en_r);
    float lse2 = INFINITY, delta = 0.f;
    if (row_valid) {
      const int64_t col = (int64_t)h * a.lse_ld + q_row0 + i0 + r;
      const float Lr = a.lse[col];
      lse2 = (Lr == -INFINITY) ? INFINITY : Lr * kLog2e;
      delta = a.delta[col];
    }
    const float sl2 = a.scale_log2;
    int seg = seg_begin, j0 = 0, j = 0;
    KvTile t;
    bool ok = true;
    while (__all_sync(0xffffffffu, *abort_flag == 0) && next_ktile(s, c, seg_end, seg, j0, t)) {
      if ((j & 1) != w) {
        ++j;
        continue;
      }
      const int b = w;
      int64_t hi = t.nk - 1, lo = 0;
      if (!t.full) {
        if (c.causal) {
          const int64_t d = pq - t.pk_lo;
          hi = min(hi, d < 0 ? (int64_t)-1 : d / t.kstride);
        }
        if (c.docs) {
          const int64_t da = st_r - t.pk_lo;
          lo = max(lo, da <= 0 ? (int64_t)0 : (da + t.kstride - 1) / t.kstride);
          const int64_t db = en_r - 1 - t.pk_lo;
          hi = min(hi, db < 0 ? (int64_t)-1 : db / t.kstride);
        }
      }
      const int ilo = (int)lo, ihi = (int)max(hi, (int64_t)-1);
      if (!wait_all(&bars->s_full[b], (j >> 1) & 1, abort_flag, a.err)) { ok = false; break; }
      ptx::tc_fence_after();
      uint32_t sr[2][32], dr[2][32];
      ptx::tmem_ld32(lane_addr + b * 128 + 0, sr[0]);
      ptx::tmem_ld32(lane_addr + b * 128 + 32, sr[1]);
      ptx::tmem_ld32(lane_addr + b * 128 + 64, dr[0]);
      ptx::tmem_ld32(lane_addr + b * 128 + 96, dr[1]);
      ptx::tmem_wait_ld_regs(sr[0]);
      ptx::tmem_wait_ld_regs(sr[1]);
      ptx::tmem_wait_ld_regs(dr[0]);
      ptx::tmem_wait_ld_regs(dr[1]);
      uint32_t dd[32];
#pragma unroll
      for (int cc = 0; cc < B_BN; cc += 2) {
        float ds[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int col = cc + u;
          const float sv = __uint_as_float(sr[col >> 5][col & 31]);
          const float dp = __uint_as_float(dr[col >> 5][col & 31]);
          const float p = (col >= ilo && col <= ihi) ? ptx::ex2_approx(fmaf(sv, sl2, -lse2)) : 0.f;
          ds[u] = p * (dp - delta);
        }
        dd[cc / 2] = ptx::pack_bf16x2(ds[0], ds[1]);
      }
      // dS (two bf16 per column) over the dP columns just read
      ptx::tmem_st32(lane_addr + b * 128 + 64, dd);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&bars->ds_full[b]);
      ++j;
    }
    // ------------------------------------------------------------ dQ epilogue
    ok = ok && __all_sync(0xffffffffu, *abort_flag == 0);
    if (ok) ok = wait_all(&bars->done, 0, abort_flag, a.err);
    if (ok) {
      ptx::tc_fence_after();
      float* dst = a.dq_acc + (int64_t)(q_row0 + i0 + r) * a.q_ld + (int64_t)h * D;
#pragma unroll
      for (int ch = (warp >> 2) * 2; ch < (warp >> 2) * 2 + 2; ++ch) {  // 64 columns per warpgroup
        uint32_t rr[32];
        if (j > 0) {
          ptx::tmem_ld32(lane_addr + 256 + ch * 32, rr);
          ptx::tmem_wait_ld_regs(rr);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) rr[i] = 0u;
        }
        if (row_valid) {
          float4* d4 = reinterpret_cast<float4*>(dst + ch * 32);
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4)
            d4[v4] = make_float4(__uint_as_float(rr[4 * v4]) * a.scale, __uint_as_float(rr[4 * v4 + 1]) * a.scale,
                                 __uint_as_float(rr[4 * v4 + 2]) * a.scale, __uint_as_float(rr[4 * v4 + 3]) * a.scale);
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

cp_status make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, uint32_t box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) {
    set_last_error("cuTensorMapEncodeTiled unavailable from the driver");
    return CP_ERR_CUDA;
  }
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, box_rows};
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

}  // namespace

cp_status launch_attn_bwd_tc(const BwdArgs& a, Schedule& s, int64_t q_rows, int64_t k_rows,
                             cudaStream_t st) {
  if (a.D != D) {
    set_last_error("tcgen05 attention backward supports D = 128");
    return CP_ERR_UNSUPPORTED;
  }
  CUtensorMap mq64, mdo64, mk128, mv128, mq128, mdo128, mk64, mv64;
  cp_status r;
  if ((r = make_map(&mq64, a.q, q_rows, (int64_t)a.Hq * D, A_BQ)) != CP_OK) return r;
  if ((r = make_map(&mdo64, a.dout, q_rows, (int64_t)a.Hq * D, A_BQ)) != CP_OK) return r;
  if ((r = make_map(&mk128, a.k, k_rows, (int64_t)a.Hkv * D, A_BK)) != CP_OK) return r;
  if ((r = make_map(&mv128, a.v, k_rows, (int64_t)a.Hkv * D, A_BK)) != CP_OK) return r;
  if ((r = make_map(&mq128, a.q, q_rows, (int64_t)a.Hq * D, B_BQ)) != CP_OK) return r;
  if ((r = make_map(&mdo128, a.dout, q_rows, (int64_t)a.Hq * D, B_BQ)) != CP_OK) return r;
  if ((r = make_map(&mk64, a.k, k_rows, (int64_t)a.Hkv * D, B_BN)) != CP_OK) return r;
  if ((r = make_map(&mv64, a.v, k_rows, (int64_t)a.Hkv * D, B_BN)) != CP_OK) return r;

  // setmaxnreg.inc waits until the registers it asks for are free in the block's launch
  // budget, so launch only if each kernel's compiled register count covers the split.
  for (const void* kfn : {(const void*)attn_bwd_dkdv_kernel, (const void*)attn_bwd_dq_kernel}) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kfn);
    if (e != cudaSuccess) return cuda_check(e, "cudaFuncGetAttributes(attn_bwd)");
    if ((int64_t)fa.numRegs * kThreads < 128 * kRegsLow + 256 * kRegsHigh) {
      set_last_error("attention backward compiled with " + std::to_string(fa.numRegs) +
                     " registers per thread, too few for its warpgroup register split");
      return CP_ERR_UNSUPPORTED;
    }
  }
  // dK / dV over the key-major schedule
  int64_t units = schedule_units(s, A_BK, a.Hkv);
  if (units > 0) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         ALayout::kSmemRequest);
    if (e != cudaSuccess) return cuda_check(e, "cudaFuncSetAttribute(attn_bwd_dkdv)");
    attn_bwd_dkdv_kernel<<<(unsigned)units, kThreads, ALayout::kSmemRequest, st>>>(a, s, mq64, mdo64,
                                                                                    mk128, mv128);
    if ((r = cuda_check(cudaGetLastError(), "attn_bwd_dkdv_kernel launch")) != CP_OK) return r;
  }
  // dQ over the query-major schedule (same pairs)
  Schedule* qm = new Schedule;
  if (!invert_schedule(s, *qm)) {
    delete qm;
    set_last_error("backward schedule too large to invert");
    return CP_ERR_UNSUPPORTED;
  }
  units = schedule_units(*qm, B_BQ, a.Hq);
  if (units > 0) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         BLayout::kSmemRequest);
    if (e != cudaSuccess) {
      delete qm;
      return cuda_check(e, "cudaFuncSetAttribute(attn_bwd_dq)");
    }
    attn_bwd_dq_kernel<<<(unsigned)units, kThreads, BLayout::kSmemRequest, st>>>(a, *qm, mq128, mdo128,
                                                                                  mk64, mv64);
    r = cuda_check(cudaGetLastError(), "attn_bwd_dq_kernel launch");
  }
  delete qm;
  return r;
}

}  // namespace cpa
