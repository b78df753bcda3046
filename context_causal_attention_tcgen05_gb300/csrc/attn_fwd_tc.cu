// tcgen05 block attention forward for bf16 (fp32 accumulation), sm_103a.
//
// Computes the handbook's attention(q, k, v, causal, q_offset, k_offset) ->
// (out, lse) ("Context parallelism: Ring Attention and Ulysses", section
// "Which operations partition directly") for every query group of a schedule
// (common.cuh), walking each group's key/value segments in order with an
// online softmax.  For the ring, the segments are the key/value blocks the
// ranks hold at steps 0..P-1, so the online-softmax rescaling IS the ring's
// log-sum-exp merge (section "Ring Attention: passing the KV once around a
// ring": lse = log(e^lse1 + e^lse2), o = o1 e^(lse1-lse) + o2 e^(lse2-lse)).
//
// One CTA = two 128-row query tiles (Q0, Q1) of one head, 12 warps:
//   warps 0..3  softmax of Q0, warps 4..7 softmax of Q1: thread t owns query
//               row t of its tile (its TMEM lane).  It reads its S row with
//               tcgen05.ld, masks boundary tiles only, keeps the running max
//               in the log2 domain, and writes P (bf16) back into the first 64
//               columns of its S buffer with tcgen05.st.  O is rescaled in
//               TMEM only when the max grew by more than 2^8 (otherwise the
//               stale max is kept; the final normalisation absorbs it).
//   warp 8      TMA producer: Q0/Q1 once, K and V tiles (128 keys) in a 2-stage
//               ring of 128B-swizzled shared-memory buffers, one barrier per
//               stage.  (Warps 8..11 form the third warpgroup, which gives
//               registers to the softmax ones.)
//   warp 9      MMA issuer (one thread), ping-pong order per key tile j:
//                 S0 = Q0 K_j^T | O1 += P1 V_{j-1} | S1 = Q1 K_j^T | O0 += P0 V_j
//               so each softmax overlaps the other tile's two products.  The
//               pipe queues about one MMA, so the issuer does no schedule
//               walking in the loop and at most one barrier wait between products.
//               P is the A operand straight from TMEM (M=128 lanes, two bf16 per
//               column); V is the B operand from shared memory (MN-major).
// TMEM: S0/P0 cols 0..127, O0 128..255, S1/P1 256..383, O1 384..511.
// Epilogue: each softmax warp normalises its 32 rows of O and, for bf16 output,
// stages them in its query tile's Q buffer (free once every product completed)
// in the 128-byte swizzled layout, then one lane writes them with TMA stores
// (32-row boxes); fp32 output and warps holding rows past the group's end store
// each row directly.  The sliding window is a template flag, so the unwindowed
// kernel carries none of its terms.
// Key/value tiles entirely masked for both query tiles are never loaded;
// fully visible tiles skip the mask.  Every mbarrier wait is bounded; on
// expiry the CTA records CP_ERR_DEVICE_TIMEOUT in the device error word,
// drains its own copies and MMAs, frees its TMEM and returns.
#include <cuda.h>
#include <string.h>

#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"

namespace cpa {
namespace {

constexpr int BM = 128;          // rows per query tile
constexpr int kRowsPerCta = 2 * BM;
constexpr int BN = 128;          // keys per key/value tile
constexpr int kThreads = 384;        // 3 warpgroups
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;         // warps 10, 11 only rebalance registers
// Register split (launch: 384 x 168 = 64512): the producer/MMA warpgroup drops to
// 64, the two softmax warpgroups rise to 216: 128*64 + 256*216 = 63488 <= 64512.
constexpr int kRegsLow = 64;
constexpr int kRegsHigh = 216;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s per wait
constexpr uint64_t kDrainNs = 200000000ull;   // 0.2 s when draining after an abort
constexpr float kRescaleThreshold = 8.0f;     // log2 units: rescale when the max grows by > 2^8
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kSegCap = 128;                  // segments per group kept in shared memory
#ifndef CP_DEBUG
constexpr int64_t kL2KvBytes = 32ll << 20;    // K/V bytes the launch order keeps in flight
#else
constexpr int64_t kL2KvBytes = 1;             // debug build: one key/value head per block at any size
#endif

template <int D>
struct Layout {
  static constexpr int kTile = 128 * D * 2;  // one 128-row tile of bf16 [rows][D]
  static constexpr int kQ = 0;               // Q0, Q1
  static constexpr int kK = kQ + 2 * kTile;  // 2 stages
  static constexpr int kV = kK + 2 * kTile;  // 2 stages
  static constexpr int kBar = kV + 2 * kTile;
  static constexpr int kSeg = kBar + 256;  // the group's key/value segments (up to kSegCap)
  static constexpr int kBytes = kSeg + kSegCap * (int)sizeof(KSeg);
  // One CTA per SM: TMEM (512 columns) is allocated whole.
  static constexpr int kSmemRequest = kBytes + 1024 > 120 * 1024 ? kBytes + 1024 : 120 * 1024;
};

struct Bars {
  uint64_t q_full;
  uint64_t kv_full[2];   // K and V tile of a stage landed
  uint64_t kv_empty[2];  // every product reading the stage completed
  uint64_t s_full[2];  // per query tile
  uint64_t p_full[2];  // per query tile
  uint64_t o_done;
  uint32_t tmem_base;
  int abort_flag;
};

// Visibility bounds of a span of query rows (for tile classification).
struct SpanCtx {
  int64_t pq_lo, pq_hi;                // positions of the first / last valid query rows
  int64_t st_lo, st_hi, en_lo, en_hi;  // document [start, end) of pq_lo and pq_hi
  int64_t win_lo;   // pq_lo - window + 1: first position any row's window reaches (INT64_MIN: none)
  int64_t full_lo;  // first key position every row of the span sees (document and window starts)
};

struct KvTile {
  int32_t k_row;
  int32_t nk;
  int64_t pk_lo, pk_hi;
  int32_t kstride;
};

__device__ __forceinline__ void span_init(SpanCtx& c, const AttnArgs& a, int32_t window, int64_t pq_lo,
                                          int64_t pq_hi) {
  c.pq_lo = pq_lo;
  c.pq_hi = pq_hi;
  c.st_lo = c.st_hi = c.en_lo = c.en_hi = 0;
  c.win_lo = window > 0 ? pq_lo - window + 1 : INT64_MIN;
  c.full_lo = window > 0 ? pq_hi - window + 1 : INT64_MIN;
  if (a.cu_seqlens) {
    doc_bounds(a.cu_seqlens, a.n_docs, pq_lo, &c.st_lo, &c.en_lo);
    doc_bounds(a.cu_seqlens, a.n_docs, pq_hi, &c.st_hi, &c.en_hi);
    c.full_lo = max(c.full_lo, c.st_hi);
  }
}

// Visible key/value tiles [lo, hi) of one segment for the CTA's query span.
__device__ __forceinline__ void seg_range(const KSeg& sg, const SpanCtx& c, int causal, int docs,
                                          int& lo, int& hi) {
  key_tile_range(sg, BN, c.pq_hi, c.st_lo, c.en_hi, causal, docs, c.win_lo, lo, hi);
}

// Walks the visible key/value tiles of the CTA's segments in order.  Identical in every role.
struct TileIter {
  const KSeg* segs;
  int nseg, si, i, hi;
};

__device__ __forceinline__ void iter_init(TileIter& it, const KSeg* segs, int nseg, const SpanCtx& c,
                                          int causal, int docs) {
  it.segs = segs;
  it.nseg = nseg;
  it.si = 0;
  it.i = it.hi = 0;
  if (nseg > 0) seg_range(segs[0], c, causal, docs, it.i, it.hi);
}

__device__ __forceinline__ bool iter_next(TileIter& it, const SpanCtx& c, int causal, int docs, KvTile& t) {
  while (it.si < it.nseg) {
    if (it.i < it.hi) {
      const KSeg sg = it.segs[it.si];
      const int j0 = it.i * BN;
      t.k_row = sg.k_row0 + j0;
      t.nk = min(BN, sg.nk - j0);
      t.pk_lo = (int64_t)sg.pos_off + (int64_t)sg.pos_stride * j0;
      t.pk_hi = t.pk_lo + (int64_t)sg.pos_stride * (t.nk - 1);
      t.kstride = sg.pos_stride;
      ++it.i;
      return true;
    }
    if (++it.si < it.nseg) seg_range(it.segs[it.si], c, causal, docs, it.i, it.hi);
  }
  return false;
}

// Every (row, key) pair of the tile visible for this query span (no mask needed)?
__device__ __forceinline__ bool tile_full(const SpanCtx& c, const KvTile& t, int causal, int docs) {
  return (t.nk == BN) && (!causal || t.pk_hi <= c.pq_lo) && t.pk_lo >= c.full_lo &&
         (!docs || t.pk_hi < c.en_lo);
}

template <int D>
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile_base, int kk) {
  // K step of 16 bf16 = 32 bytes inside a 64-column (128-byte) swizzle region.
  return ptx::smem_desc_sw128(tile_base + (kk >> 2) * (128 * 128) + (kk & 3) * 32, 16, 1024);
}

template <int D>
__device__ __forceinline__ uint64_t desc_v_mnmajor(uint32_t tile_base, int kk) {
  // 16 key rows per K step (16 * 128 bytes); next 64 d-columns at +16 KB (LBO); next 8 keys at +1 KB (SBO).
  return ptx::smem_desc_sw128(tile_base + kk * (16 * 128), 128 * 128, 1024);
}

// kWin: the sliding window is applied (a.window > 0); without it the window
// terms fold away at compile time.  kP > 0: position-tiled striped buffers of kP
// ranks (AttnArgs::perm_p): the schedule's rows are positions, every tile is
// loaded as one 3-D TMA box of 128/kP rows of each rank (128 consecutive
// positions), and shared-memory row r of a tile holds position
// start + (r % (128/kP)) * kP + r / (128/kP).
template <int D, bool kOutF32, bool kWin, int kP>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_tc_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ Schedule s,
                   const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_o) {
  using L = Layout<D>;
  constexpr int kM = kP > 0 ? BM / kP : 1;  // rows of each rank in a tile (position-tiled)
  static_assert(kP == 0 || (BM % kP == 0 && kP >= 4 && kP <= 16), "position tiles: 4 <= kP <= 16");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kBar);
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Launch order: blocks of head_block heads (whole key/value heads); within a block
  // every (group, tile) pair in the schedule's order, the block's heads fastest, so
  // the CTAs resident together read the key/value tiles of a few heads through L2.
  int g, tile, h;
  decode_unit_blocked(s, kRowsPerCta, a.head_block, a.total_units / a.Hq, blockIdx.x, &g, &tile, &h);
  const int hk = h / (a.Hq / a.Hkv);
  const int32_t window = kWin ? a.window : 0;
  const int32_t q_row0 = s.g[g].q_row0, nq = s.g[g].nq;
  const int32_t qpos_off = s.g[g].pos_off, qpos_st = s.g[g].pos_stride;
  const int seg_begin = s.g[g].seg_begin, seg_end = seg_begin + s.g[g].seg_count;
  const int i0 = tile * kRowsPerCta;
  const int nq0 = min(BM, nq - i0);
  const int nq1 = max(0, min(BM, nq - i0 - BM));
  const bool has1 = nq1 > 0;
  const int causal = a.causal, docs = a.cu_seqlens != nullptr;

  SpanCtx cta;  // both query tiles together
  {
    const int64_t lo = (int64_t)qpos_off + (int64_t)qpos_st * i0;
    span_init(cta, a, window, lo, lo + (int64_t)qpos_st * (nq0 + nq1 - 1));
  }

  // The group's segments, read at every tile by every role: shared memory when they fit.
  const int nseg = seg_end - seg_begin;
  KSeg* seg_sm = reinterpret_cast<KSeg*>(smem + L::kSeg);
  const KSeg* segs = nseg <= kSegCap ? seg_sm : &s.s[seg_begin];
  if (nseg <= kSegCap)
    for (int i = threadIdx.x; i < nseg; i += kThreads) seg_sm[i] = s.s[seg_begin + i];
  int pj = 0;
  int issued[2] = {0, 0};
  auto issue_kv = [&](const KvTile& t) {
    const int st = pj & 1;
    (void)CP_DCHECK(t.k_row >= 0 && t.k_row < a.k_rows, a.err);
    ptx::mbar_arrive_expect_tx(&bars->kv_full[st], 2 * L::kTile);
#pragma unroll
    for (int r = 0; r < D / 64; ++r) {
      if constexpr (kP > 0) {  // 128 consecutive positions: kM rows of every rank
        ptx::tma_load_3d(smem + L::kK + st * L::kTile + r * 16384, &tm_k, &bars->kv_full[st],
                         hk * D + r * 64, t.k_row / kP, 0);
        ptx::tma_load_3d(smem + L::kV + st * L::kTile + r * 16384, &tm_v, &bars->kv_full[st],
                         hk * D + r * 64, t.k_row / kP, 0);
      } else {
        ptx::tma_load_2d(smem + L::kK + st * L::kTile + r * 16384, &tm_k, &bars->kv_full[st],
                         hk * D + r * 64, t.k_row);
        ptx::tma_load_2d(smem + L::kV + st * L::kTile + r * 16384, &tm_v, &bars->kv_full[st],
                         hk * D + r * 64, t.k_row);
      }
    }
    issued[st] = pj + 1;
    ++pj;
  };
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bars->q_full, 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&bars->kv_full[i], 1);
      ptx::mbar_init(&bars->kv_empty[i], 1);
      ptx::mbar_init(&bars->s_full[i], 1);
      ptx::mbar_init(&bars->p_full[i], 128);
    }
    ptx::mbar_init(&bars->o_done, 1);
    bars->abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    ptx::prefetch_tensormap(&tm_q);
    ptx::prefetch_tensormap(&tm_k);
    ptx::prefetch_tensormap(&tm_v);
    if (!kOutF32 && a.o_tma) ptx::prefetch_tensormap(&tm_o);
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(&bars->tmem_base, kTmemCols);
    ptx::tmem_relinquish();
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
      (void)CP_DCHECK((int64_t)q_row0 + i0 < a.q_rows, a.err);  // TMA clips; the check reports
      ptx::mbar_arrive_expect_tx(&bars->q_full, (has1 ? 2 : 1) * L::kTile);
      for (int w = 0; w < (has1 ? 2 : 1); ++w)
#pragma unroll
        for (int r = 0; r < D / 64; ++r) {
          if constexpr (kP > 0)
            ptx::tma_load_3d(smem + L::kQ + w * L::kTile + r * 16384, &tm_q, &bars->q_full,
                             h * D + r * 64, (q_row0 + i0 + w * BM) / kP, 0);
          else
            ptx::tma_load_2d(smem + L::kQ + w * L::kTile + r * 16384, &tm_q, &bars->q_full,
                             h * D + r * 64, q_row0 + i0 + w * BM);
        }
      TileIter pit;
      iter_init(pit, segs, nseg, cta, causal, docs);
      KvTile t;
      while (!*abort_flag && iter_next(pit, cta, causal, docs, t)) {
        if (pj >= 2 && !ptx::mbar_wait_bounded(&bars->kv_empty[pj & 1], ((pj >> 1) - 1) & 1, abort_flag,
                                               a.err, kWaitNs))
          break;
        issue_kv(t);
      }
      if (*abort_flag) {
        // drain: wait (bounded) for this CTA's own copies still in flight
        (void)ptx::mbar_wait_bounded(&bars->q_full, 0, nullptr, nullptr, kDrainNs);
        for (int st = 0; st < 2; ++st)
          if (issued[st] > 0)
            (void)ptx::mbar_wait_bounded(&bars->kv_full[st], ((issued[st] - 1) >> 1) & 1, nullptr,
                                         nullptr, kDrainNs);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The tile count up front, one segment per lane.
    int n_tiles = 0;
    for (int si = lane; si < nseg; si += 32) {
      int lo, hi;
      seg_range(segs[si], cta, causal, docs, lo, hi);
      n_tiles += hi - lo;
    }
    n_tiles = __reduce_add_sync(0xffffffffu, n_tiles);
    if (lane == 0) {
      constexpr uint32_t idesc_qk = ptx::idesc_bf16_f32(BM, BN, 0, 0);
      constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(BM, D, 0, 1);  // V is MN-major
      auto qk = [&](int w, int st) {
        const uint32_t q_addr = sbase + L::kQ + w * L::kTile;
        const uint32_t k_addr = sbase + L::kK + st * L::kTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_bf16_ss(tmem + w * 256, desc_kmajor<D>(q_addr, kk), desc_kmajor<D>(k_addr, kk),
                           idesc_qk, kk > 0);
      };
      auto pv = [&](int w, int st, bool acc) {
        const uint32_t v_addr = sbase + L::kV + st * L::kTile;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)  // P: 16 keys = 8 TMEM columns per step
          ptx::mma_bf16_ts(tmem + w * 256 + 128, tmem + w * 256 + kk * 8,
                           desc_v_mnmajor<D>(v_addr, kk), idesc_pv, (acc || kk > 0) ? 1u : 0u);
      };
      auto wait = [&](uint64_t* bar, uint32_t par) {
        return ptx::mbar_wait_bounded(bar, par, abort_flag, a.err, kWaitNs);
      };
      // The issuing thread stalls at each tcgen05.mma until the pipe accepts it, so
      // every gap between two products holds at most one barrier wait and no
      // schedule walking (the tile count is known up front).
      const int n = n_tiles;
      bool ok = wait(&bars->q_full, 0);
      bool any = false;
      if (ok && n > 0) {
        ok = wait(&bars->kv_full[0], 0);
        if (ok) {  // S0 = Q0 K_0^T
          ptx::tc_fence_after();
          qk(0, 0);
          ptx::tc_commit(&bars->s_full[0]);
          any = true;
        }
        for (int j = 0; ok && j < n; ++j) {
          const int st = j & 1;
          if (has1 && j >= 1) {  // O1 += P1 V_{j-1}
            const int stp = (j - 1) & 1;
            if (!(ok = wait(&bars->p_full[1], (j - 1) & 1))) break;
            ptx::tc_fence_after();
            pv(1, stp, j - 1 > 0);
            ptx::tc_commit(&bars->kv_empty[stp]);
          }
          if (has1) {  // S1 = Q1 K_j^T
            qk(1, st);
            ptx::tc_commit(&bars->s_full[1]);
          }
          // O0 += P0 V_j
          if (!(ok = wait(&bars->p_full[0], j & 1))) break;
          ptx::tc_fence_after();
          pv(0, st, j > 0);
          if (!has1) ptx::tc_commit(&bars->kv_empty[st]);
          if (j + 1 < n) {  // S0 = Q0 K_{j+1}^T
            const int st1 = (j + 1) & 1;
            if (!(ok = wait(&bars->kv_full[st1], ((j + 1) >> 1) & 1))) break;
            ptx::tc_fence_after();
            qk(0, st1);
            ptx::tc_commit(&bars->s_full[0]);
          }
        }
        if (ok && has1) {  // O1 += P1 V_{n-1}
          const int jp = n - 1, stp = jp & 1;
          if (wait(&bars->p_full[1], jp & 1)) {
            ptx::tc_fence_after();
            pv(1, stp, jp > 0);
            ptx::tc_commit(&bars->kv_empty[stp]);
          }
        }
      }
      // o_done: every MMA of this CTA has completed (also the TMEM release condition)
      if (any) {
        ptx::tc_commit(&bars->o_done);
        (void)ptx::mbar_wait_bounded(&bars->o_done, 0, nullptr, a.err, kWaitNs);
      } else {
        ptx::mbar_arrive(&bars->o_done);
      }
    }
    __syncwarp();
  }
  } else {
    ptx::setmaxnreg_inc<kRegsHigh>();
    // ------------------------------------------------------------ softmax warpgroups
    const int w = warp >> 2;               // query tile of this warpgroup
    const int quad = warp & 3;             // TMEM lane quadrant of this warp
    const int r = quad * 32 + lane;        // query row within the tile
    const int nq_w = w == 0 ? nq0 : nq1;
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16) + w * 256;
    if (w == 0 || has1) {
      SpanCtx mine;
      const int64_t pq_lo_w = cta.pq_lo + (int64_t)qpos_st * (w * BM);
      span_init(mine, a, window, pq_lo_w, pq_lo_w + (int64_t)qpos_st * (nq_w - 1));
      // position of this thread's row (its offset in the tile's position window)
      const int r_off = kP > 0 ? (r % kM) * kP + r / kM : r;
      const int64_t pq = pq_lo_w + (int64_t)qpos_st * r_off;
      int64_t st_r = 0, en_r = 0;
      if (docs && r_off < nq_w) doc_bounds(a.cu_seqlens, a.n_docs, pq, &st_r, &en_r);
      // first key position the row sees: its document's start and its window's start
      const int64_t first_r = max(docs ? st_r : INT64_MIN, window > 0 ? pq - window + 1 : INT64_MIN);
      const float sl2 = a.scale_log2;
      const uint64_t sl2x2 = ptx::f2_pack(sl2, sl2);
      float m = -INFINITY, l = 0.f;
      TileIter it;
      iter_init(it, segs, nseg, cta, causal, docs);
      int j = 0;
      KvTile t;
      auto wwait = [&](uint64_t* bar, uint32_t par) {
        bool ok = ptx::mbar_wait_bounded(bar, par, abort_flag, a.err, kWaitNs);
        return __all_sync(0xffffffffu, ok);
      };
      while (__all_sync(0xffffffffu, *abort_flag == 0) && iter_next(it, cta, causal, docs, t)) {
        const bool full = tile_full(mine, t, causal, docs);
        int ilo = 0, ihi = BN - 1;
        if (!full) {
          int64_t hi = t.nk - 1, lo = 0;
          if (causal) {
            const int64_t d = pq - t.pk_lo;
            hi = min(hi, d < 0 ? (int64_t)-1 : udiv_pos(d, t.kstride));
          }
          if (docs) {
            const int64_t db = en_r - 1 - t.pk_lo;
            hi = min(hi, db < 0 ? (int64_t)-1 : udiv_pos(db, t.kstride));
          }
          if (first_r > t.pk_lo)  // keys before first_r are hidden
            lo = udiv_pos(first_r - t.pk_lo + t.kstride - 1, t.kstride);
          ilo = (int)min(lo, (int64_t)BN);
          ihi = (int)max(hi, (int64_t)-1);
        }
        if (!wwait(&bars->s_full[w], j & 1)) break;
        ptx::tc_fence_after();
        float sv[BN];
        {
          uint32_t rr[BN / 32][32];
#pragma unroll
          for (int ch = 0; ch < BN / 32; ++ch) ptx::tmem_ld32(lane_addr + ch * 32, rr[ch]);
#pragma unroll
          for (int ch = 0; ch < BN / 32; ++ch) {
            ptx::tmem_wait_ld_regs(rr[ch]);
#pragma unroll
            for (int i = 0; i < 32; ++i) sv[ch * 32 + i] = __uint_as_float(rr[ch][i]);
          }
        }
        if (!full) {  // [ilo, ihi]: visible offsets in the key tile's position window
#pragma unroll
          for (int i = 0; i < BN; ++i) {
            const int oi = kP > 0 ? (i % kM) * kP + i / kM : i;  // compile-time per column
            sv[i] = (oi >= ilo && oi <= ihi) ? sv[i] : -INFINITY;
          }
        }
        float mx[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
        for (int i = 4; i < BN; i += 8) {
          mx[0] = ptx::fmax3(mx[0], sv[i], sv[i + 1]);
          mx[1] = ptx::fmax3(mx[1], sv[i + 2], sv[i + 3]);
          if (i + 7 < BN) {
            mx[2] = ptx::fmax3(mx[2], sv[i + 4], sv[i + 5]);
            mx[3] = ptx::fmax3(mx[3], sv[i + 6], sv[i + 7]);
          }
        }
        const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2;
        const float m_new = fmaxf(m, mt);
        const bool need = m_new > m + kRescaleThreshold;
        const bool warp_need = __any_sync(0xffffffffu, need);
        if (warp_need) {
          const float alpha = (m == -INFINITY) ? 0.f : ptx::ex2_approx(m - m_new);
          if (m_new != -INFINITY) m = m_new;
          l *= alpha;
          if (j > 0) {
            // the previous P V of this tile completed before this tile's S (commit order)
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
              uint32_t rr[32];
              ptx::tmem_ld32(lane_addr + 128 + ch * 32, rr);
              ptx::tmem_wait_ld_regs(rr);
#pragma unroll
              for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
              ptx::tmem_st32(lane_addr + 128 + ch * 32, rr);
            }
          }
        }
        const float neg_m = (m == -INFINITY) ? 0.f : -m;
        const uint64_t nm2 = ptx::f2_pack(neg_m, neg_m);
        uint64_t lsum[4] = {ptx::f2_pack(0.f, 0.f), ptx::f2_pack(0.f, 0.f), ptx::f2_pack(0.f, 0.f),
                            ptx::f2_pack(0.f, 0.f)};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int c = half * 64 + 2 * i;
            float x0, x1;
            ptx::f2_unpack(ptx::ffma2(ptx::f2_pack(sv[c], sv[c + 1]), sl2x2, nm2), x0, x1);
            const float p0 = ptx::ex2_approx(x0), p1 = ptx::ex2_approx(x1);
            lsum[i & 3] = ptx::fadd2(lsum[i & 3], ptx::f2_pack(p0, p1));
            pk[i] = ptx::pack_bf16x2(p0, p1);
          }
          ptx::tmem_st32(lane_addr + half * 32, pk);  // P over the first 64 columns of S
        }
        const uint64_t lsum2 = ptx::fadd2(ptx::fadd2(lsum[0], lsum[1]), ptx::fadd2(lsum[2], lsum[3]));
        float ls0, ls1;
        ptx::f2_unpack(lsum2, ls0, ls1);
        l += ls0 + ls1;
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&bars->p_full[w]);
        ++j;
      }
      // ------------------------------------------------------------ epilogue
      bool ok = __all_sync(0xffffffffu, *abort_flag == 0);
      if (ok) ok = wwait(&bars->o_done, 0);
      if (ok) {
        ptx::tc_fence_after();
        const bool valid = r_off < nq_w;
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        // the buffer row of a tile row: rank r / kM, row tile_i0 + r % kM of that rank
        // (position-tiled), else the schedule's row
        const int32_t tile_i0 = kP > 0 ? (i0 + w * BM) / kP : 0;
        auto buf_row = [&](int rr_) -> int64_t {
          if constexpr (kP > 0) return (int64_t)(rr_ / kM) * a.perm_n + tile_i0 + rr_ % kM;
          return (int64_t)s.g[g].o_row0 + i0 + w * BM + rr_;
        };
        const int32_t oh = s.g[g].o_head0 + h;  // output head column block
        const int64_t orow = buf_row(r) * a.o_ld + (int64_t)oh * D;
        // bf16 output of a warp whose 32 rows are all valid: staged in this query tile's
        // Q buffer (free once o_done fired) in the 128-byte swizzled layout of the O
        // tensor map, then written by one TMA store per 64 columns.
        const bool staged = !kOutF32 && a.o_tma && (kP > 0 ? nq_w == BM : quad * 32 + 32 <= nq_w) &&
                            CP_DCHECK(kP > 0 || buf_row(quad * 32 + 31) < a.q_rows, a.err);
        if (staged) {
          uint8_t* stg = smem + L::kQ + w * L::kTile + quad * (32 * D * 2);
#pragma unroll
          for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t rr[32];
            if (j > 0) {
              ptx::tmem_ld32(lane_addr + 128 + ch * 32, rr);
              ptx::tmem_wait_ld_regs(rr);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) rr[i] = 0u;
            }
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              const int c = ch * 4 + v4;  // 16-byte chunk of the row (8 columns)
              uint4* dst = reinterpret_cast<uint4*>(stg + (c >> 3) * 4096 + lane * 128 +
                                                    (((c & 7) ^ (lane & 7)) << 4));
              *dst = make_uint4(ptx::pack_bf16x2(__uint_as_float(rr[8 * v4 + 0]) * inv_l,
                                                 __uint_as_float(rr[8 * v4 + 1]) * inv_l),
                                ptx::pack_bf16x2(__uint_as_float(rr[8 * v4 + 2]) * inv_l,
                                                 __uint_as_float(rr[8 * v4 + 3]) * inv_l),
                                ptx::pack_bf16x2(__uint_as_float(rr[8 * v4 + 4]) * inv_l,
                                                 __uint_as_float(rr[8 * v4 + 5]) * inv_l),
                                ptx::pack_bf16x2(__uint_as_float(rr[8 * v4 + 6]) * inv_l,
                                                 __uint_as_float(rr[8 * v4 + 7]) * inv_l));
            }
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if constexpr (kP > 0) {  // the warp's 32 rows: 32/kM ranks of kM rows, or 32 rows of one rank
              const int32_t y0 = tile_i0 + (kM >= 32 ? (quad * 32) % kM : 0);
              const int32_t z0 = (quad * 32) / kM;
#pragma unroll
              for (int hf = 0; hf < D / 64; ++hf)
                ptx::tma_store_3d(&tm_o, stg + hf * 4096, oh * D + hf * 64, y0, z0);
            } else {
              const int32_t y0 = s.g[g].o_row0 + i0 + w * BM + quad * 32;
#pragma unroll
              for (int hf = 0; hf < D / 64; ++hf) ptx::tma_store_2d(&tm_o, stg + hf * 4096, oh * D + hf * 64, y0);
            }
            ptx::bulk_commit_group();
          }
        }
#pragma unroll
        for (int ch = 0; ch < D / 32 && !staged; ++ch) {
          uint32_t rr[32];
          if (j > 0) {
            ptx::tmem_ld32(lane_addr + 128 + ch * 32, rr);
            ptx::tmem_wait_ld_regs(rr);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) rr[i] = 0u;
          }
          if (valid && CP_DCHECK(buf_row(r) < a.q_rows, a.err)) {
            if (kOutF32) {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.o) + orow + ch * 32);
#pragma unroll
              for (int v4 = 0; v4 < 8; ++v4)
                dst[v4] = make_float4(__uint_as_float(rr[4 * v4]) * inv_l,
                                      __uint_as_float(rr[4 * v4 + 1]) * inv_l,
                                      __uint_as_float(rr[4 * v4 + 2]) * inv_l,
                                      __uint_as_float(rr[4 * v4 + 3]) * inv_l);
            } else {
              uint4* dst =
                  reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.o) + orow + ch * 32);
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4)
                dst[v4] = make_uint4(
                    ptx::pack_bf16x2(__uint_as_float(rr[8 * v4 + 0]) * inv_l,
                                     __uint_as_float(rr[8 * v4 + 1]) * inv_l),
                    ptx::pack_bf16x2(__uint_as_float(rr[8 * v4 + 2]) * inv_l,
                                     __uint_as_float(rr[8 * v4 + 3]) * inv_l),
                    ptx::pack_bf16x2(__uint_as_float(rr[8 * v4 + 4]) * inv_l,
                                     __uint_as_float(rr[8 * v4 + 5]) * inv_l),
                    ptx::pack_bf16x2(__uint_as_float(rr[8 * v4 + 6]) * inv_l,
                                     __uint_as_float(rr[8 * v4 + 7]) * inv_l));
            }
          }
        }
        const int64_t li = (int64_t)(s.g[g].lse_head0 + h) * a.lse_ld +
                           (kP > 0 ? buf_row(r) : (int64_t)s.g[g].lse_col0 + i0 + w * BM + r);
        if (valid && CP_DCHECK(li < a.lse_size, a.err)) {
          const float Lr = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
          a.lse[li] = Lr;
        }
        if (staged && lane == 0) ptx::bulk_wait_group_read0();  // the CTA's smem outlives the reads
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

// ---------------------------------------------------------------- host side

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
cp_status make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows = 128,
                   bool report = true) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) {
    if (report) set_last_error("cuTensorMapEncodeTiled unavailable from the driver");
    return CP_ERR_CUDA;
  }
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (report) set_last_error("cuTensorMapEncodeTiled failed (code " + std::to_string((int)r) + ")");
    return CP_ERR_CUDA;
  }
  return CP_OK;
}

// 3-D map over a striped buffer [P][n][cols] bf16 (rank-major): box 64 columns x
// box_rows rows x box_ranks ranks, 128-byte swizzle.  A box of 128/P rows of all P
// ranks holds 128 consecutive positions.
cp_status make_map_striped(CUtensorMap* m, const void* base, int64_t n, int64_t P, int64_t cols, int box_rows,
                           int box_ranks) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) {
    set_last_error("cuTensorMapEncodeTiled unavailable from the driver");
    return CP_ERR_CUDA;
  }
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)(n > 0 ? n : 1), (cuuint64_t)P};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)cols * 2 * (cuuint64_t)n};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_ranks};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_last_error("cuTensorMapEncodeTiled (striped) failed (code " + std::to_string((int)r) + ")");
    return CP_ERR_CUDA;
  }
  return CP_OK;
}

template <int D, bool kOutF32, bool kWin, int kP = 0>
cp_status launch_typed(const AttnArgs& a, Schedule& s, const CUtensorMap& mq, const CUtensorMap& mk,
                       const CUtensorMap& mv, const CUtensorMap& mo, int64_t units, cudaStream_t st) {
  using L = Layout<D>;
  auto kern = attn_fwd_tc_kernel<D, kOutF32, kWin, kP>;
  // setmaxnreg.inc waits until the registers it asks for are free in the block's
  // launch budget, so launch only if the split fits that budget.
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return cuda_check(e, "cudaFuncGetAttributes(attn_fwd_tc)");
  if ((int64_t)fa.numRegs * kThreads < 128 * kRegsLow + 256 * kRegsHigh) {
    set_last_error("attn_fwd_tc compiled with " + std::to_string(fa.numRegs) +
                   " registers per thread, too few for its warpgroup register split");
    return CP_ERR_UNSUPPORTED;
  }
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemRequest);
  if (e != cudaSuccess) return cuda_check(e, "cudaFuncSetAttribute(attn_fwd_tc)");
  kern<<<(unsigned)units, kThreads, L::kSmemRequest, st>>>(a, s, mq, mk, mv, mo);
  return cuda_check(cudaGetLastError(), "attn_fwd_tc_kernel launch");
}

}  // namespace

cp_status launch_attn_fwd_tc(const AttnArgs& a, Schedule& s, int64_t q_rows, int64_t k_rows,
                             cudaStream_t st) {
  int64_t units = schedule_units(s, kRowsPerCta, a.Hq);
  if (units == 0) return CP_OK;
  if (units > 0x7fffffff) {
    set_last_error("too many query tiles for one launch");
    return CP_ERR_UNSUPPORTED;
  }
  // Inside each block of heads, the (group, tile) pairs that see the most key tiles
  // start first (when the causal rule or a window sets the weights).
  schedule_order(s, kRowsPerCta, BN, false, a.causal, a.window, a.cu_seqlens != nullptr);
  // Heads per block of the launch order: the most whole key/value heads (a divisor
  // of Hkv, at least one) whose K and V fit kL2KvBytes together.  This pays when
  // every group reads most of the key rows (the ring, one block pair).  When groups
  // read disjoint rows (Ulysses' ranks), or with packed documents (a unit reads
  // only its documents' keys), one block (every head fastest) measured faster.
  AttnArgs ab = a;
  {
    int64_t keys_max = 0;
    for (int i = 0; i < s.n_groups; ++i) {
      int64_t n = 0;
      for (int j = s.g[i].seg_begin; j < s.g[i].seg_begin + s.g[i].seg_count; ++j) n += s.s[j].nk;
      keys_max = std::max(keys_max, n);
    }
    const int64_t kv_bytes = std::max<int64_t>(1, k_rows * (int64_t)a.D * 2 * 2);
    int kb = (int)std::min<int64_t>(a.Hkv, std::max<int64_t>(1, kL2KvBytes / kv_bytes));
    if (a.cu_seqlens || 2 * keys_max < k_rows) kb = a.Hkv;
    while (a.Hkv % kb) --kb;
    ab.head_block = kb * (a.Hq / a.Hkv);
    ab.total_units = (int32_t)units;
  }
  CUtensorMap mq, mk, mv;
  cp_status r;
  if (a.perm_p > 0) {
    // position-tiled striped buffers (bf16 output, D = 128, no window): every map is
    // 3-D over [P][n][H*D]; the O map's box is one warp's 32 rows
    const int P = a.perm_p, M = BM / P;
    if (!(a.D == 128 && !a.o_f32 && a.window == 0 && (P == 4 || P == 8 || P == 16))) {
      set_last_error("position-tiled striped forward: D = 128, bf16 output, P in {4, 8, 16}");
      return CP_ERR_UNSUPPORTED;
    }
    CUtensorMap mo;
    if ((r = make_map_striped(&mq, a.q, a.perm_n, P, (int64_t)a.Hq * a.D, M, P)) != CP_OK) return r;
    if ((r = make_map_striped(&mk, a.k, a.perm_n, P, (int64_t)a.Hkv * a.D, M, P)) != CP_OK) return r;
    if ((r = make_map_striped(&mv, a.v, a.perm_n, P, (int64_t)a.Hkv * a.D, M, P)) != CP_OK) return r;
    if ((r = make_map_striped(&mo, a.o, a.perm_n, P, a.o_ld, M >= 32 ? 32 : M, M >= 32 ? 1 : 32 / M)) != CP_OK)
      return r;
    AttnArgs ao = ab;
    ao.o_tma = 1;
    if (P == 4) return launch_typed<128, false, false, 4>(ao, s, mq, mk, mv, mo, units, st);
    if (P == 8) return launch_typed<128, false, false, 8>(ao, s, mq, mk, mv, mo, units, st);
    return launch_typed<128, false, false, 16>(ao, s, mq, mk, mv, mo, units, st);
  }
  if ((r = make_map(&mq, a.q, q_rows, (int64_t)a.Hq * a.D)) != CP_OK) return r;
  if ((r = make_map(&mk, a.k, k_rows, (int64_t)a.Hkv * a.D)) != CP_OK) return r;
  if ((r = make_map(&mv, a.v, k_rows, (int64_t)a.Hkv * a.D)) != CP_OK) return r;
  // O map (32-row boxes) over the output rows the schedule writes; without one
  // (fp32 output, or a base the tensor map cannot take) rows are stored directly.
  CUtensorMap mo;
  memset(&mo, 0, sizeof(mo));
  AttnArgs ao = ab;
  ao.o_tma = 0;
  if (!a.o_f32) {
    int64_t o_rows = 0;
    for (int i = 0; i < s.n_groups; ++i) o_rows = std::max<int64_t>(o_rows, (int64_t)s.g[i].o_row0 + s.g[i].nq);
    ao.o_tma = make_map(&mo, a.o, o_rows, a.o_ld, 32, false) == CP_OK ? 1 : 0;
  }
  const bool win = a.window > 0;
  if (a.D == 128) {
    if (win)
      return a.o_f32 ? launch_typed<128, true, true>(ao, s, mq, mk, mv, mo, units, st)
                     : launch_typed<128, false, true>(ao, s, mq, mk, mv, mo, units, st);
    return a.o_f32 ? launch_typed<128, true, false>(ao, s, mq, mk, mv, mo, units, st)
                   : launch_typed<128, false, false>(ao, s, mq, mk, mv, mo, units, st);
  }
  if (a.D == 64) {
    if (win)
      return a.o_f32 ? launch_typed<64, true, true>(ao, s, mq, mk, mv, mo, units, st)
                     : launch_typed<64, false, true>(ao, s, mq, mk, mv, mo, units, st);
    return a.o_f32 ? launch_typed<64, true, false>(ao, s, mq, mk, mv, mo, units, st)
                   : launch_typed<64, false, false>(ao, s, mq, mk, mv, mo, units, st);
  }
  set_last_error("tcgen05 attention supports D = 64 or 128");
  return CP_ERR_UNSUPPORTED;
}

}  // namespace cpa
