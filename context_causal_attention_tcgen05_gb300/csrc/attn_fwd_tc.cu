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
// One CTA = one 128-row query tile of one head; 6 warps:
//   warp 0      TMA producer: Q once, then K and V tiles (128 keys) into a
//               2-stage ring of 128B-swizzled shared-memory buffers.
//   warp 1      MMA issuer (one thread): S = Q K^T into one of two TMEM
//               buffers (M=128, N=128, K=D), then O += P V into TMEM
//               (M=128, N=D, K=128) once the softmax has written P.
//               Issue order QK(j), PV(j-1) lets QK(j) overlap softmax(j-1).
//   warps 2..5  softmax: thread t owns query row t (its TMEM lane): reads its
//               S row with tcgen05.ld, applies the causal / document mask on
//               boundary tiles only, keeps the running max in the log2
//               domain, writes P (bf16) to shared memory in the MMA's K-major
//               128B-swizzled layout, and rescales its O row in TMEM only when
//               the max grew by more than 2^8 (otherwise the stale max is kept
//               and the final normalisation absorbs it).
// Key/value tiles entirely masked (after every query of the tile, or outside
// the tile's documents) are never loaded; fully visible tiles skip the mask.
// Every mbarrier wait is bounded; on expiry the CTA records
// CP_ERR_DEVICE_TIMEOUT in the device error word, drains its own copies and
// MMAs, frees its TMEM and returns.
#include <cuda.h>

#include "common.cuh"
#include "ptx.cuh"

namespace cpa {
namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s per wait
constexpr uint64_t kDrainNs = 200000000ull;   // 0.2 s when draining after an abort
constexpr float kRescaleThreshold = 8.0f;     // log2 units: rescale when the max grows by > 2^8
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct Layout {
  static constexpr int kTile = 128 * D * 2;  // one 128-row tile of bf16 [rows][D]
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTile;      // 2 stages
  static constexpr int kV = kK + 2 * kTile;  // 2 stages
  static constexpr int kP = kV + 2 * kTile;  // [128][BN] bf16
  static constexpr int kPBytes = 128 * BN * 2;
  static constexpr int kBar = kP + kPBytes;
  static constexpr int kBytes = kBar + 256;
  // One CTA per SM: TMEM (512 columns) is allocated whole.
  static constexpr int kSmemRequest = kBytes + 1024 > 120 * 1024 ? kBytes + 1024 : 120 * 1024;
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[2], v_full[2];
  uint64_t k_empty[2], v_empty[2];
  uint64_t s_full[2];
  uint64_t p_full;
  uint64_t o_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

struct TileCtx {
  int64_t pq_lo, pq_hi;             // positions of the first / last valid query rows
  int64_t st_lo, st_hi, en_lo, en_hi;  // document [start, end) of pq_lo and pq_hi
  int causal, docs;
};

struct KvTile {
  int32_t k_row;
  int32_t nk;
  int64_t pk_lo;
  int32_t kstride;
  int32_t full;
};

// Next key/value tile of the group with any visible pair.  Identical in every role.
__device__ __forceinline__ bool next_tile(const Schedule& s, const TileCtx& c, int seg_end,
                                          int& seg, int& j0, KvTile& t) {
  while (seg < seg_end) {
    const int32_t k_row0 = s.s[seg].k_row0, nk_seg = s.s[seg].nk;
    const int32_t poff = s.s[seg].pos_off, pst = s.s[seg].pos_stride;
    if (j0 >= nk_seg) {
      ++seg;
      j0 = 0;
      continue;
    }
    const int nk = min(BN, nk_seg - j0);
    const int64_t pk_lo = (int64_t)poff + (int64_t)pst * j0;
    const int64_t pk_hi = pk_lo + (int64_t)pst * (nk - 1);
    const int jcur = j0;
    j0 += BN;
    if ((c.causal && pk_lo > c.pq_hi) || (c.docs && pk_lo >= c.en_hi)) {
      ++seg;  // this and every later tile of the segment lie after the queries
      j0 = 0;
      continue;
    }
    if (c.docs && pk_hi < c.st_lo) continue;  // before the first query's document
    t.k_row = k_row0 + jcur;
    t.nk = nk;
    t.pk_lo = pk_lo;
    t.kstride = pst;
    t.full = (nk == BN) && (!c.causal || pk_hi <= c.pq_lo) &&
             (!c.docs || (pk_lo >= c.st_hi && pk_hi < c.en_lo));
    return true;
  }
  return false;
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

template <int D, bool kOutF32>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_tc_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ Schedule s,
                   const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kBar);
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  int g, tile, h;
  decode_unit(s, BM, a.Hq, blockIdx.x, &g, &tile, &h);
  const int hk = h / (a.Hq / a.Hkv);
  const int32_t q_row0 = s.g[g].q_row0, nq = s.g[g].nq;
  const int32_t qpos_off = s.g[g].pos_off, qpos_st = s.g[g].pos_stride;
  const int seg_begin = s.g[g].seg_begin, seg_end = seg_begin + s.g[g].seg_count;
  const int i0 = tile * BM;
  const int nq_tile = min(BM, nq - i0);

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
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&bars->k_full[i], 1);
      ptx::mbar_init(&bars->v_full[i], 1);
      ptx::mbar_init(&bars->k_empty[i], 1);
      ptx::mbar_init(&bars->v_empty[i], 1);
      ptx::mbar_init(&bars->s_full[i], 1);
    }
    ptx::mbar_init(&bars->p_full, 128);
    ptx::mbar_init(&bars->o_full, 1);
    ptx::mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&bars->tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tensormap(&tm_q);
    ptx::prefetch_tensormap(&tm_k);
    ptx::prefetch_tensormap(&tm_v);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      ptx::mbar_arrive_expect_tx(&bars->q_full, L::kTile);
#pragma unroll
      for (int r = 0; r < D / 64; ++r)
        ptx::tma_load_2d(smem + L::kQ + r * 16384, &tm_q, &bars->q_full, h * D + r * 64,
                         q_row0 + i0);
      int seg = seg_begin, j0 = 0, j = 0;
      KvTile t;
      int issued[2] = {0, 0};
      while (!*abort_flag && next_tile(s, c, seg_end, seg, j0, t)) {
        const int st = j & 1;
        if (j >= 2 && !ptx::mbar_wait_bounded(&bars->k_empty[st], ((j >> 1) - 1) & 1, abort_flag,
                                              a.err, kWaitNs))
          break;
        ptx::mbar_arrive_expect_tx(&bars->k_full[st], L::kTile);
#pragma unroll
        for (int r = 0; r < D / 64; ++r)
          ptx::tma_load_2d(smem + L::kK + st * L::kTile + r * 16384, &tm_k, &bars->k_full[st],
                           hk * D + r * 64, t.k_row);
        if (j >= 2 && !ptx::mbar_wait_bounded(&bars->v_empty[st], ((j >> 1) - 1) & 1, abort_flag,
                                              a.err, kWaitNs)) {
          issued[st] = j + 1;
          break;
        }
        ptx::mbar_arrive_expect_tx(&bars->v_full[st], L::kTile);
#pragma unroll
        for (int r = 0; r < D / 64; ++r)
          ptx::tma_load_2d(smem + L::kV + st * L::kTile + r * 16384, &tm_v, &bars->v_full[st],
                           hk * D + r * 64, t.k_row);
        issued[st] = j + 1;
        ++j;
      }
      if (*abort_flag) {
        // drain: wait (bounded) for this CTA's own copies still in flight
        (void)ptx::mbar_wait_bounded(&bars->q_full, 0, nullptr, nullptr, kDrainNs);
        for (int st = 0; st < 2; ++st)
          if (issued[st] > 0) {
            const uint32_t par = ((issued[st] - 1) >> 1) & 1;
            (void)ptx::mbar_wait_bounded(&bars->k_full[st], par, nullptr, nullptr, kDrainNs);
            (void)ptx::mbar_wait_bounded(&bars->v_full[st], par, nullptr, nullptr, kDrainNs);
          }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = ptx::idesc_bf16_f32(BM, BN, 0, 0);
      constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(BM, D, 0, 1);
      const uint32_t q_addr = sbase + L::kQ, p_addr = sbase + L::kP;
      const uint32_t o_tmem = tmem + 256;
      bool any = false;
      if (ptx::mbar_wait_bounded(&bars->q_full, 0, abort_flag, a.err, kWaitNs)) {
        int seg = seg_begin, j0 = 0, j = 0;
        KvTile t;
        bool more = next_tile(s, c, seg_end, seg, j0, t);
        while (true) {
          if (more) {  // S(j) = Q K(j)^T
            const int st = j & 1;
            if (!ptx::mbar_wait_bounded(&bars->k_full[st], (j >> 1) & 1, abort_flag, a.err, kWaitNs))
              break;
            ptx::tc_fence_after();
            const uint32_t k_addr = sbase + L::kK + st * L::kTile;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              ptx::mma_bf16_ss(tmem + st * 128, desc_kmajor<D>(q_addr, kk), desc_kmajor<D>(k_addr, kk),
                               idesc_qk, kk > 0);
            ptx::tc_commit(&bars->s_full[st]);
            ptx::tc_commit(&bars->k_empty[st]);
            any = true;
          }
          if (j >= 1) {  // O += P(j-1) V(j-1)
            const int jp = j - 1, st = jp & 1;
            if (!ptx::mbar_wait_bounded(&bars->p_full, jp & 1, abort_flag, a.err, kWaitNs)) break;
            if (!ptx::mbar_wait_bounded(&bars->v_full[st], (jp >> 1) & 1, abort_flag, a.err, kWaitNs))
              break;
            ptx::tc_fence_after();
            const uint32_t v_addr = sbase + L::kV + st * L::kTile;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              ptx::mma_bf16_ss(o_tmem, desc_kmajor<D>(p_addr, kk), desc_v_mnmajor<D>(v_addr, kk),
                               idesc_pv, (jp > 0 || kk > 0) ? 1u : 0u);
            ptx::tc_commit(&bars->o_full);
            ptx::tc_commit(&bars->v_empty[st]);
          }
          if (!more) break;
          ++j;
          more = next_tile(s, c, seg_end, seg, j0, t);
        }
      }
      if (any) {  // all MMAs of this CTA complete before TMEM is released
        ptx::tc_commit(&bars->drain);
        (void)ptx::mbar_wait_bounded(&bars->drain, 0, nullptr, a.err, kWaitNs);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warpgroup
    const int quad = warp & 3;             // TMEM lane quadrant of this warp
    const int r = quad * 32 + lane;        // query row within the tile
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
    const int64_t pq = c.pq_lo + (int64_t)qpos_st * r;
    int64_t st_r = 0, en_r = 0;
    if (c.docs && r < nq_tile) doc_bounds(a.cu_seqlens, a.n_docs, pq, &st_r, &en_r);
    const float sl2 = a.scale_log2;
    float m = -INFINITY, l = 0.f;
    int seg = seg_begin, j0 = 0, j = 0;
    KvTile t;
    uint8_t* prow = smem + L::kP + r * 128;
    // Waits are made warp-uniform so the warp-collective tcgen05.ld/st and
    // votes below always run converged.
    auto wwait = [&](uint64_t* bar, uint32_t par) {
      bool ok = ptx::mbar_wait_bounded(bar, par, abort_flag, a.err, kWaitNs);
      return __all_sync(0xffffffffu, ok);
    };
    while (__all_sync(0xffffffffu, *abort_flag == 0) && next_tile(s, c, seg_end, seg, j0, t)) {
      const int st = j & 1;
      if (!wwait(&bars->s_full[st], (j >> 1) & 1)) break;
      ptx::tc_fence_after();
      float sv[BN];
      {
        uint32_t rr[BN / 32][32];
#pragma unroll
        for (int ch = 0; ch < BN / 32; ++ch) ptx::tmem_ld32(lane_addr + st * 128 + ch * 32, rr[ch]);
#pragma unroll
        for (int ch = 0; ch < BN / 32; ++ch) {
          ptx::tmem_wait_ld_regs(rr[ch]);
#pragma unroll
          for (int i = 0; i < 32; ++i) sv[ch * 32 + i] = __uint_as_float(rr[ch][i]);
        }
      }
      if (!t.full) {
        int64_t hi = t.nk - 1, lo = 0;
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
        const int ilo = (int)lo, ihi = (int)max(hi, (int64_t)-1);
#pragma unroll
        for (int i = 0; i < BN; ++i) sv[i] = (i >= ilo && i <= ihi) ? sv[i] : -INFINITY;
      }
      float mx0 = sv[0], mx1 = sv[1], mx2 = sv[2], mx3 = sv[3];
#pragma unroll
      for (int i = 4; i < BN; i += 4) {
        mx0 = fmaxf(mx0, sv[i]);
        mx1 = fmaxf(mx1, sv[i + 1]);
        mx2 = fmaxf(mx2, sv[i + 2]);
        mx3 = fmaxf(mx3, sv[i + 3]);
      }
      const float mt = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
      const float m_new = fmaxf(m, mt);
      const bool need = m_new > m + kRescaleThreshold;
      const bool warp_need = __any_sync(0xffffffffu, need);
      float alpha = 1.f;
      if (warp_need) {
        alpha = (m == -INFINITY) ? 0.f : ptx::ex2_approx(m - m_new);
        if (m_new != -INFINITY) m = m_new;
        l *= alpha;
      }
      const float neg_m = (m == -INFINITY) ? 0.f : -m;
      float l0 = 0.f, l1 = 0.f;
      uint32_t pk[BN / 2];
#pragma unroll
      for (int i = 0; i < BN; i += 2) {
        const float p0 = ptx::ex2_approx(fmaf(sv[i], sl2, neg_m));
        const float p1 = ptx::ex2_approx(fmaf(sv[i + 1], sl2, neg_m));
        l0 += p0;
        l1 += p1;
        pk[i / 2] = ptx::pack_bf16x2(p0, p1);
      }
      l += l0 + l1;
      // P and O are free once the previous P V has completed.
      if (j > 0) {
        if (!wwait(&bars->o_full, (j - 1) & 1)) break;
        ptx::tc_fence_after();
        if (warp_need) {
#pragma unroll
          for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t rr[32];
            ptx::tmem_ld32(lane_addr + 256 + ch * 32, rr);
            ptx::tmem_wait_ld_regs(rr);
#pragma unroll
            for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
            ptx::tmem_st32(lane_addr + 256 + ch * 32, rr);
          }
          ptx::tmem_wait_st();
        }
      }
#pragma unroll
      for (int cc = 0; cc < BN / 8; ++cc) {
        uint8_t* dst = prow + (cc >> 3) * 16384 + (((cc & 7) ^ (r & 7)) << 4);
        *reinterpret_cast<uint4*>(dst) =
            make_uint4(pk[cc * 4 + 0], pk[cc * 4 + 1], pk[cc * 4 + 2], pk[cc * 4 + 3]);
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&bars->p_full);
      ++j;
    }
    // ------------------------------------------------------------ epilogue
    bool ok = __all_sync(0xffffffffu, *abort_flag == 0);
    if (ok && j > 0) {
      ok = wwait(&bars->o_full, (j - 1) & 1);
      ptx::tc_fence_after();
    }
    if (ok) {
      const bool valid = r < nq_tile;
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const int64_t orow = (int64_t)(s.g[g].o_row0 + i0 + r) * a.o_ld + (int64_t)h * D;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t rr[32];
        if (j > 0) {
          ptx::tmem_ld32(lane_addr + 256 + ch * 32, rr);
          ptx::tmem_wait_ld_regs(rr);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) rr[i] = 0u;
        }
        if (valid) {
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
      if (valid) {
        const float L = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
        a.lse[(int64_t)(s.g[g].lse_head0 + h) * a.lse_ld + s.g[g].lse_col0 + i0 + r] = L;
      }
    }
    ptx::tc_fence_before();
  }

  __syncthreads();
  if (warp == 1) {
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
cp_status make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) {
    set_last_error("cuTensorMapEncodeTiled unavailable from the driver");
    return CP_ERR_CUDA;
  }
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, 128};
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

template <int D, bool kOutF32>
cp_status launch_typed(const AttnArgs& a, Schedule& s, const CUtensorMap& mq, const CUtensorMap& mk,
                       const CUtensorMap& mv, int64_t units, cudaStream_t st) {
  using L = Layout<D>;
  auto kern = attn_fwd_tc_kernel<D, kOutF32>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       L::kSmemRequest);
  if (e != cudaSuccess) return cuda_check(e, "cudaFuncSetAttribute(attn_fwd_tc)");
  kern<<<(unsigned)units, kThreads, L::kSmemRequest, st>>>(a, s, mq, mk, mv);
  return cuda_check(cudaGetLastError(), "attn_fwd_tc_kernel launch");
}

}  // namespace

cp_status launch_attn_fwd_tc(const AttnArgs& a, Schedule& s, int64_t q_rows, int64_t k_rows,
                             cudaStream_t st) {
  int64_t units = schedule_units(s, BM, a.Hq);
  if (units == 0) return CP_OK;
  if (units > 0x7fffffff) {
    set_last_error("too many query tiles for one launch");
    return CP_ERR_UNSUPPORTED;
  }
  CUtensorMap mq, mk, mv;
  cp_status r;
  if ((r = make_map(&mq, a.q, q_rows, (int64_t)a.Hq * a.D)) != CP_OK) return r;
  if ((r = make_map(&mk, a.k, k_rows, (int64_t)a.Hkv * a.D)) != CP_OK) return r;
  if ((r = make_map(&mv, a.v, k_rows, (int64_t)a.Hkv * a.D)) != CP_OK) return r;
  if (a.D == 128)
    return a.o_f32 ? launch_typed<128, true>(a, s, mq, mk, mv, units, st)
                   : launch_typed<128, false>(a, s, mq, mk, mv, units, st);
  if (a.D == 64)
    return a.o_f32 ? launch_typed<64, true>(a, s, mq, mk, mv, units, st)
                   : launch_typed<64, false>(a, s, mq, mk, mv, units, st);
  set_last_error("tcgen05 attention supports D = 64 or 128");
  return CP_ERR_UNSUPPORTED;
}

}  // namespace cpa
