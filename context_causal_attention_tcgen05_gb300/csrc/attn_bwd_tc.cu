// tcgen05 block attention backward for bf16 (fp32 accumulation), D = 128.
//
// The exact derivative of the handbook's attention ("Context parallelism:
// Ring Attention and Ulysses", section "Which operations partition
// directly"; the pages give no backward), given the FINAL out and lse of
// every query row (for a ring: the merged ones):
//   P = exp(scale*S - lse),  dV = P^T dO,  dP = dO V^T,
//   dS = P o (dP - Delta),   Delta = rowsum(dO o O),
//   dQ = scale * dS K,       dK = scale * dS^T Q.
// The schedule is key-major (common.cuh): a group is a run of key rows, its
// segments are the query runs that may see it.
//
// One CTA = one 128-key tile of one key/value head; it loops over the G query
// heads of that key/value head and every 64-row query tile that can see the
// keys, so dK and dV accumulate in TMEM and are stored once (no atomics).
// Per query tile (all MMAs M=128, bf16 in, fp32 out, operands in 128B-swizzled
// shared memory):
//   S^T  = K Q^T      [keys x q]   TMEM cols   0..63
//   dP^T = V dO^T     [keys x q]   TMEM cols  64..127
//   softmax warps (thread = key row): P^T, dS^T -> shared memory (bf16)
//   dV  += P^T dO     [keys x D]   TMEM cols 128..255
//   dK  += dS^T Q     [keys x D]   TMEM cols 256..383
//   dQ^T = K^T dS^T   [D x q]      TMEM cols 384..447
//   softmax warps (thread = d): dQ^T column c -> fp32 atomic add into dQ
//   (32 consecutive d per warp: coalesced reductions).
// Warps: 0 TMA producer (K, V once; Q, dO per tile, 2 stages), 1 MMA issuer,
// 2..5 softmax / epilogue.  Every wait is bounded (as in the forward).
#include <cuda.h>

#include "common.cuh"
#include "ptx.cuh"

namespace cpa {
namespace {

constexpr int D = 128;
constexpr int BK = 128;  // keys per CTA
constexpr int BQ = 64;   // queries per tile
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint64_t kDrainNs = 200000000ull;
constexpr float kLog2e = 1.4426950408889634f;

struct BLayout {
  static constexpr int kKV = 128 * D * 2;        // 32 KB: [128 keys][D]
  static constexpr int kQT = BQ * D * 2;         // 16 KB: [64 q][D]
  static constexpr int kK = 0;
  static constexpr int kV = kK + kKV;
  static constexpr int kQ = kV + kKV;            // 2 stages
  static constexpr int kDO = kQ + 2 * kQT;       // 2 stages
  static constexpr int kPT = kDO + 2 * kQT;      // [128 keys][64 q] bf16
  static constexpr int kDST = kPT + BK * BQ * 2;
  static constexpr int kLse = kDST + BK * BQ * 2;  // 64 floats lse*log2e, 64 floats Delta
  static constexpr int kBar = kLse + 2 * BQ * 4;
  static constexpr int kBytes = kBar + 256;
  static constexpr int kSmemRequest = kBytes + 1024;
};

struct BBars {
  uint64_t kv_full;
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full;
  uint64_t p_full;
  uint64_t mma_done;
  uint64_t drain;
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
  int64_t st_hi;  // start of the document holding pk_hi
  int causal, docs;
  int G, hk;
};

// Next query tile (over the G query heads, then the segments) that sees some key of the tile.
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
    const int nq = min(BQ, nq_seg - i0);
    const int64_t pq_lo = (int64_t)poff + (int64_t)pst * i0;
    const int64_t pq_hi = pq_lo + (int64_t)pst * (nq - 1);
    const int icur = i0;
    i0 += BQ;
    if (c.causal && pq_hi < c.pk_lo) continue;          // every query before every key
    if (c.docs && pq_lo >= c.en_lo && c.en_lo > c.pk_hi) {
      // every query after the end of the keys' (single) document
      ++seg;
      i0 = 0;
      continue;
    }
    if (c.docs && pq_hi < c.st_hi && pq_hi < c.pk_lo) continue;
    t.q_row = q_row0 + icur;
    t.nq = nq;
    t.pq_lo = pq_lo;
    t.qstride = pst;
    t.h = c.hk * c.G + hh;
    t.full = (nq == BQ) && c.causal && (pq_lo >= c.pk_hi) && (!c.docs || c.en_lo > pq_hi);
    if (!c.causal) t.full = (nq == BQ) && !c.docs;
    return true;
  }
  return false;
}

__device__ __forceinline__ uint64_t desc_k(uint32_t base, int kk, uint32_t region_bytes) {
  return ptx::smem_desc_sw128(base + (kk >> 2) * region_bytes + (kk & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t desc_mn(uint32_t base, int kk, uint32_t lbo) {
  return ptx::smem_desc_sw128(base + kk * (16 * 128), lbo, 1024);
}

__device__ __forceinline__ void red_add_f32(float* addr, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_tc_kernel(const __grid_constant__ BwdArgs a, const __grid_constant__ Schedule s,
                   const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  using L = BLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  BBars* bars = reinterpret_cast<BBars*>(smem + L::kBar);
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  int g, tile, hk;
  decode_unit(s, BK, a.Hkv, blockIdx.x, &g, &tile, &hk);
  const int32_t k_row0 = s.g[g].q_row0 + tile * BK;  // key-major schedule: group = key run
  const int nk_tile = min(BK, s.g[g].nq - tile * BK);
  const int seg_begin = s.g[g].seg_begin, seg_end = seg_begin + s.g[g].seg_count;

  KeyCtx c;
  c.causal = a.causal;
  c.docs = a.cu_seqlens != nullptr;
  c.G = a.Hq / a.Hkv;
  c.hk = hk;
  c.pk_lo = (int64_t)s.g[g].pos_off + (int64_t)s.g[g].pos_stride * (tile * BK);
  c.pk_hi = c.pk_lo + (int64_t)s.g[g].pos_stride * (nk_tile - 1);
  c.en_lo = INT64_MAX;
  c.st_hi = 0;
  if (c.docs) {
    int64_t st, en;
    doc_bounds(a.cu_seqlens, a.n_docs, c.pk_lo, &st, &en);
    c.en_lo = en;
    doc_bounds(a.cu_seqlens, a.n_docs, c.pk_hi, &st, &en);
    c.st_hi = st;
  }

  if (threadIdx.x == 0) {
    ptx::mbar_init(&bars->kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&bars->q_full[i], 1);
      ptx::mbar_init(&bars->q_empty[i], 1);
    }
    ptx::mbar_init(&bars->s_full, 1);
    ptx::mbar_init(&bars->p_full, 128);
    ptx::mbar_init(&bars->mma_done, 1);
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
    ptx::prefetch_tensormap(&tm_do);
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
      ptx::mbar_arrive_expect_tx(&bars->kv_full, 2 * L::kKV);
      for (int r = 0; r < D / 64; ++r) {
        ptx::tma_load_2d(smem + L::kK + r * 16384, &tm_k, &bars->kv_full, hk * D + r * 64, k_row0);
        ptx::tma_load_2d(smem + L::kV + r * 16384, &tm_v, &bars->kv_full, hk * D + r * 64, k_row0);
      }
      int hh = 0, seg = seg_begin, i0 = 0, j = 0;
      QTile t;
      int issued[2] = {0, 0};
      while (!*abort_flag && next_qtile(s, c, seg_begin, seg_end, hh, seg, i0, t)) {
        const int st = j & 1;
        if (j >= 2 && !ptx::mbar_wait_bounded(&bars->q_empty[st], ((j >> 1) - 1) & 1, abort_flag,
                                              a.err, kWaitNs))
          break;
        ptx::mbar_arrive_expect_tx(&bars->q_full[st], 2 * L::kQT);
        for (int r = 0; r < D / 64; ++r) {
          ptx::tma_load_2d(smem + L::kQ + st * L::kQT + r * 8192, &tm_q, &bars->q_full[st],
                           t.h * D + r * 64, t.q_row);
          ptx::tma_load_2d(smem + L::kDO + st * L::kQT + r * 8192, &tm_do, &bars->q_full[st],
                           t.h * D + r * 64, t.q_row);
        }
        issued[st] = j + 1;
        ++j;
      }
      if (*abort_flag) {
        (void)ptx::mbar_wait_bounded(&bars->kv_full, 0, nullptr, nullptr, kDrainNs);
        for (int st = 0; st < 2; ++st)
          if (issued[st] > 0)
            (void)ptx::mbar_wait_bounded(&bars->q_full[st], ((issued[st] - 1) >> 1) & 1, nullptr,
                                         nullptr, kDrainNs);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = ptx::idesc_bf16_f32(128, BQ, 0, 0);   // K Q^T, V dO^T
      constexpr uint32_t id_kv = ptx::idesc_bf16_f32(128, D, 0, 1);   // P^T dO, dS^T Q
      constexpr uint32_t id_dq = ptx::idesc_bf16_f32(128, BQ, 1, 1);  // K^T dS^T
      const uint32_t k_addr = sbase + L::kK, v_addr = sbase + L::kV;
      const uint32_t pt_addr = sbase + L::kPT, dst_addr = sbase + L::kDST;
      bool any = false;
      if (ptx::mbar_wait_bounded(&bars->kv_full, 0, abort_flag, a.err, kWaitNs)) {
        int hh = 0, seg = seg_begin, i0 = 0, j = 0;
        QTile t;
        while (!*abort_flag && next_qtile(s, c, seg_begin, seg_end, hh, seg, i0, t)) {
          const int st = j & 1;
          if (!ptx::mbar_wait_bounded(&bars->q_full[st], (j >> 1) & 1, abort_flag, a.err, kWaitNs))
            break;
          ptx::tc_fence_after();
          const uint32_t q_addr = sbase + L::kQ + st * L::kQT;
          const uint32_t do_addr = sbase + L::kDO + st * L::kQT;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            ptx::mma_bf16_ss(tmem + 0, desc_k(k_addr, kk, 16384), desc_k(q_addr, kk, 8192), id_s, kk > 0);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            ptx::mma_bf16_ss(tmem + 64, desc_k(v_addr, kk, 16384), desc_k(do_addr, kk, 8192), id_s, kk > 0);
          ptx::tc_commit(&bars->s_full);
          any = true;
          if (!ptx::mbar_wait_bounded(&bars->p_full, j & 1, abort_flag, a.err, kWaitNs)) break;
          ptx::tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BQ / 16; ++kk)
            ptx::mma_bf16_ss(tmem + 128, desc_k(pt_addr, kk, 16384), desc_mn(do_addr, kk, 8192), id_kv,
                             (j > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < BQ / 16; ++kk)
            ptx::mma_bf16_ss(tmem + 256, desc_k(dst_addr, kk, 16384), desc_mn(q_addr, kk, 8192), id_kv,
                             (j > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            ptx::mma_bf16_ss(tmem + 384, desc_mn(k_addr, kk, 16384), desc_mn(dst_addr, kk, 0), id_dq,
                             kk > 0);
          ptx::tc_commit(&bars->mma_done);
          ptx::tc_commit(&bars->q_empty[st]);
          ++j;
        }
      }
      if (any) {
        ptx::tc_commit(&bars->drain);
        (void)ptx::mbar_wait_bounded(&bars->drain, 0, nullptr, a.err, kWaitNs);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax / dS / dQ warpgroup
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // key row (and d for the dQ^T read-out)
    const int tid = threadIdx.x - 64;
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
    float* lse_s = reinterpret_cast<float*>(smem + L::kLse);
    float* del_s = lse_s + BQ;
    const int64_t pk = c.pk_lo + (int64_t)s.g[g].pos_stride * r;
    int64_t en_k = INT64_MAX;
    if (c.docs && r < nk_tile) {
      int64_t st;
      doc_bounds(a.cu_seqlens, a.n_docs, pk, &st, &en_k);
    }
    const float sl2 = a.scale_log2;
    auto wwait = [&](uint64_t* bar, uint32_t par) {
      bool ok = ptx::mbar_wait_bounded(bar, par, abort_flag, a.err, kWaitNs);
      return __all_sync(0xffffffffu, ok);
    };
    auto group_sync = [&]() { asm volatile("bar.sync 1, 128;" ::: "memory"); };
    int hh = 0, seg = seg_begin, i0 = 0, j = 0;
    QTile t;
    bool ok = true;
    while (__all_sync(0xffffffffu, *abort_flag == 0) && next_qtile(s, c, seg_begin, seg_end, hh, seg, i0, t)) {
      // lse (log2 domain; +inf for rows that see nothing or lie past the run) and Delta
      group_sync();  // previous tile's readers are done with lse_s / del_s
      if (tid < BQ) {
        float v = INFINITY;
        if (tid < t.nq) {
          const float L = a.lse[(int64_t)t.h * a.lse_ld + t.q_row + tid];
          v = (L == -INFINITY) ? INFINITY : L * kLog2e;
        }
        lse_s[tid] = v;
      } else {
        const int cidx = tid - BQ;
        del_s[cidx] = cidx < t.nq ? a.delta[(int64_t)t.h * a.lse_ld + t.q_row + cidx] : 0.f;
      }
      group_sync();
      // visible query columns of this key row: [c_lo, c_hi]
      int64_t hi = t.nq - 1, lo = 0;
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
        }
      }
      const int ilo = (int)lo, ihi = (int)max(hi, (int64_t)-1);
      if (!wwait(&bars->s_full, j & 1)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      uint32_t sr[2][32], dr[2][32];
      ptx::tmem_ld32(lane_addr + 0, sr[0]);
      ptx::tmem_ld32(lane_addr + 32, sr[1]);
      ptx::tmem_ld32(lane_addr + 64, dr[0]);
      ptx::tmem_ld32(lane_addr + 96, dr[1]);
      ptx::tmem_wait_ld_regs(sr[0]);
      ptx::tmem_wait_ld_regs(sr[1]);
      ptx::tmem_wait_ld_regs(dr[0]);
      ptx::tmem_wait_ld_regs(dr[1]);
      // previous tile's dV/dK/dQ MMAs read P^T / dS^T: wait for them before overwriting
      if (j > 0) {
        if (!wwait(&bars->mma_done, (j - 1) & 1)) {
          ok = false;
          break;
        }
      }
      uint32_t pp[BQ / 2], dd[BQ / 2];
#pragma unroll
      for (int cc = 0; cc < BQ; cc += 2) {
        float p0 = 0.f, p1 = 0.f;
        const float s0 = __uint_as_float(sr[cc >> 5][cc & 31]);
        const float s1 = __uint_as_float(sr[(cc + 1) >> 5][(cc + 1) & 31]);
        if (cc >= ilo && cc <= ihi) p0 = ptx::ex2_approx(fmaf(s0, sl2, -lse_s[cc]));
        if (cc + 1 >= ilo && cc + 1 <= ihi) p1 = ptx::ex2_approx(fmaf(s1, sl2, -lse_s[cc + 1]));
        const float dp0 = __uint_as_float(dr[cc >> 5][cc & 31]);
        const float dp1 = __uint_as_float(dr[(cc + 1) >> 5][(cc + 1) & 31]);
        pp[cc / 2] = ptx::pack_bf16x2(p0, p1);
        dd[cc / 2] = ptx::pack_bf16x2(p0 * (dp0 - del_s[cc]), p1 * (dp1 - del_s[cc + 1]));
      }
      uint8_t* prow = smem + L::kPT + r * 128;
      uint8_t* drow = smem + L::kDST + r * 128;
#pragma unroll
      for (int ch = 0; ch < BQ / 8; ++ch) {
        const int off = ((ch ^ (r & 7)) << 4);
        *reinterpret_cast<uint4*>(prow + off) = make_uint4(pp[4 * ch], pp[4 * ch + 1], pp[4 * ch + 2], pp[4 * ch + 3]);
        *reinterpret_cast<uint4*>(drow + off) = make_uint4(dd[4 * ch], dd[4 * ch + 1], dd[4 * ch + 2], dd[4 * ch + 3]);
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&bars->p_full);
      // dQ^T of this tile: thread = d, columns = query rows
      if (!wwait(&bars->mma_done, j & 1)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      uint32_t qr[2][32];
      ptx::tmem_ld32(lane_addr + 384, qr[0]);
      ptx::tmem_ld32(lane_addr + 416, qr[1]);
      ptx::tmem_wait_ld_regs(qr[0]);
      ptx::tmem_wait_ld_regs(qr[1]);
      float* dq_col = a.dq_acc + (int64_t)t.q_row * a.q_ld + (int64_t)t.h * D + r;
#pragma unroll
      for (int cc = 0; cc < BQ; ++cc)
        if (cc < t.nq) red_add_f32(dq_col + (int64_t)cc * a.q_ld, __uint_as_float(qr[cc >> 5][cc & 31]) * a.scale);
      ptx::tc_fence_before();
      ++j;
      // mma_done(j-1) was consumed above; the next tile waits on it again only as "previous"
    }
    // ------------------------------------------------------------ dK / dV epilogue
    ok = ok && __all_sync(0xffffffffu, *abort_flag == 0);
    if (ok) {
      ptx::tc_fence_after();
      const bool valid = r < nk_tile;
      const int64_t krow = (int64_t)(k_row0 + r) * a.k_ld + (int64_t)hk * D;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        float* dst = (which == 0 ? a.dv_acc : a.dk_acc) + krow;
        const float mul = which == 0 ? 1.f : a.scale;
        const uint32_t col0 = which == 0 ? 128 : 256;
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
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

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

}  // namespace

cp_status launch_attn_bwd_tc(const BwdArgs& a, Schedule& s, int64_t q_rows, int64_t k_rows,
                             cudaStream_t st) {
  if (a.D != D) {
    set_last_error("tcgen05 attention backward supports D = 128");
    return CP_ERR_UNSUPPORTED;
  }
  int64_t units = schedule_units(s, BK, a.Hkv);
  if (units == 0) return CP_OK;
  CUtensorMap mq, mdo, mk, mv;
  cp_status r;
  if ((r = make_map(&mq, a.q, q_rows, (int64_t)a.Hq * D, BQ)) != CP_OK) return r;
  if ((r = make_map(&mdo, a.dout, q_rows, (int64_t)a.Hq * D, BQ)) != CP_OK) return r;
  if ((r = make_map(&mk, a.k, k_rows, (int64_t)a.Hkv * D, BK)) != CP_OK) return r;
  if ((r = make_map(&mv, a.v, k_rows, (int64_t)a.Hkv * D, BK)) != CP_OK) return r;
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       BLayout::kSmemRequest);
  if (e != cudaSuccess) return cuda_check(e, "cudaFuncSetAttribute(attn_bwd_tc)");
  attn_bwd_tc_kernel<<<(unsigned)units, kThreads, BLayout::kSmemRequest, st>>>(a, s, mq, mdo, mk, mv);
  return cuda_check(cudaGetLastError(), "attn_bwd_tc_kernel launch");
}

}  // namespace cpa
