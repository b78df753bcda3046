// C ABI (include/cp_attn.h): argument validation, workspace layout, and the
// ring / Ulysses drivers over P virtual ranks held in one GPU's memory.
//
// Sources: handbook chapter "Context parallelism: Ring Attention and Ulysses"
// (sections "Ulysses: transposing between the sequence and the heads", "Ring
// Attention: passing the KV once around a ring", "The zigzag partition") and
// the MaxText pull request "Add Packing Support for Context Parallelism (Ring
// Attention) #2906" (reorder strategies; packing accepted only with a
// load-balanced ring).
//
// On one GPU the ring's point-to-point KV pass is an index: at step s virtual
// rank r reads the key/value rows of rank (r - s) mod P from the reordered
// buffer.  The Ulysses all-to-all is the seq2head / head2seq permute kernel.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"

namespace cpa {

static thread_local std::string g_last_error;

void set_last_error(const std::string& msg) { g_last_error = msg; }

cp_status cuda_check(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return CP_OK;
  set_last_error(std::string(what) + ": " + cudaGetErrorString(e));
  return CP_ERR_CUDA;
}

// The device error word: a kernel that gives up on a bounded wait records a
// code here; cp_check_device_status reads and clears it.
__device__ int32_t g_device_error = 0;

static std::mutex g_err_mu;
static int32_t* g_err_ptr[64] = {nullptr};

int32_t* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<int32_t*>(p);
  }
  return g_err_ptr[dev];
}

int64_t schedule_units(Schedule& s, int tile_rows, int heads) {
  int64_t tiles = 0;
  for (int i = 0; i < s.n_groups; ++i) {
    s.g[i].tile0 = (int32_t)tiles;
    tiles += (s.g[i].nq + tile_rows - 1) / tile_rows;
  }
  s.n_order = 0;
  return tiles * heads;
}

// Tiles of segment sg (tiles of `tile` rows) that a tile of the group spanning
// positions [p_lo, p_hi] works on: query-major, key tiles not after p_hi and not
// wholly before the window start; key-major, query tiles not wholly before p_lo
// and starting within p_hi + window - 1.
static int64_t tiles_seen(const KSeg& sg, int tile, int64_t p_lo, int64_t p_hi, bool key_major,
                          int causal, int window) {
  const int64_t n = (sg.nk + tile - 1) / tile;
  const int64_t step = (int64_t)sg.pos_stride * tile;
  int64_t lo = 0, hi = n;
  auto clamp = [&](int64_t x) { return x < 0 ? (int64_t)0 : (x > n ? n : x); };
  if (!key_major) {
    if (causal) hi = clamp(p_hi < sg.pos_off ? 0 : (p_hi - sg.pos_off) / step + 1);
    if (window > 0) {  // last key of tile i >= p_lo - window + 1
      const int64_t first = p_lo - window + 1 - sg.pos_off;
      if (first > 0) lo = clamp((first / sg.pos_stride - (tile - 1)) / tile);
    }
  } else {
    if (causal) {  // last query of tile i >= p_lo
      const int64_t d = p_lo - sg.pos_off;
      if (d > 0) lo = clamp((d / sg.pos_stride - (tile - 1)) / tile);
    }
    if (window > 0) {  // first query of tile i <= p_hi + window - 1
      const int64_t last = p_hi + window - 1 - sg.pos_off;
      hi = clamp(last < 0 ? 0 : last / step + 1);
    }
  }
  return hi > lo ? hi - lo : 0;
}

void schedule_order(Schedule& s, int tile_rows, int other_tile, bool key_major, int causal, int window,
                    bool docs) {
  s.n_order = 0;
  if (docs || (!causal && window <= 0)) return;
  std::vector<std::pair<int64_t, int32_t>> w;  // (weight, entry) in the default order
  for (int gi = 0; gi < s.n_groups; ++gi) {
    const QGroup& g = s.g[gi];
    const int ntiles = (g.nq + tile_rows - 1) / tile_rows;
    if (ntiles >= (1 << 20)) return;
    for (int local = 0; local < ntiles; ++local) {
      const int t = ntiles - 1 - local;
      const int64_t r0 = (int64_t)t * tile_rows, r1 = std::min<int64_t>(r0 + tile_rows, g.nq) - 1;
      const int64_t p_lo = g.pos_off + (int64_t)g.pos_stride * r0;
      const int64_t p_hi = g.pos_off + (int64_t)g.pos_stride * r1;
      int64_t seen = 0;
      for (int si = g.seg_begin; si < g.seg_begin + g.seg_count; ++si)
        seen += tiles_seen(s.s[si], other_tile, p_lo, p_hi, key_major, causal, window);
      w.emplace_back(seen, (int32_t)((gi << 20) | t));
      if ((int)w.size() > kMaxOrder) return;
    }
  }
  std::stable_sort(w.begin(), w.end(),
                   [](const std::pair<int64_t, int32_t>& x, const std::pair<int64_t, int32_t>& y) {
                     return x.first > y.first;
                   });
  for (size_t i = 0; i < w.size(); ++i) s.order[i] = w[i].second;
  s.n_order = (int32_t)w.size();
}

}  // namespace cpa

using namespace cpa;

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

size_t dtype_size(int32_t dt) { return dt == CP_F32 ? 4 : 2; }

#define CP_REQUIRE(cond, code, msg)   \
  do {                                \
    if (!(cond)) {                    \
      set_last_error(msg);            \
      return code;                    \
    }                                 \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cp_status check_tensor(const void* p, const char* name, bool may_be_null_if_empty, bool empty) {
  if (p == nullptr) {
    if (may_be_null_if_empty && empty) return CP_OK;
    set_last_error(std::string(name) + " is NULL");
    return CP_ERR_INVALID_ARG;
  }
  if (!aligned16(p)) {
    set_last_error(std::string(name) + " is not 16-byte aligned");
    return CP_ERR_ALIGN;
  }
  return CP_OK;
}

#define CP_CHECK_T(p, name, empty)                                    \
  do {                                                                \
    cp_status _st = check_tensor((p), (name), true, (empty));         \
    if (_st != CP_OK) return _st;                                     \
  } while (0)

#define CP_TRY(expr)               \
  do {                             \
    cp_status _st = (expr);        \
    if (_st != CP_OK) return _st;  \
  } while (0)

cp_status check_common(int32_t Hq, int32_t Hkv, int32_t D, int32_t dtype) {
  CP_REQUIRE(dtype == CP_F32 || dtype == CP_BF16, CP_ERR_DTYPE, "dtype must be CP_F32 or CP_BF16");
  CP_REQUIRE(Hq >= 1 && Hkv >= 1, CP_ERR_INVALID_ARG, "head counts must be >= 1");
  CP_REQUIRE(Hq % Hkv == 0, CP_ERR_SHAPE, "Hq must be a multiple of Hkv (grouped-query attention)");
  if (dtype == CP_F32) {
    CP_REQUIRE(D == 16 || D == 32 || D == 64 || D == 128, CP_ERR_SHAPE,
               "D must be one of 16, 32, 64, 128");
  } else {
    CP_REQUIRE(D == 64 || D == 128, CP_ERR_DTYPE,
               "bf16 attention (tcgen05 kernel) supports D = 64 or 128");
  }
  return CP_OK;
}

bool fits_i32(int64_t x) { return x >= -(int64_t)INT32_MAX && x <= (int64_t)INT32_MAX; }

// One rank's run of rows in a reordered buffer with an affine position map.
struct Piece {
  int32_t row0, n, pos_off, pos_stride;
};

// Rank holdings for a ring layout, rows in the reordered buffer (rank-major).
std::vector<std::vector<Piece>> rank_pieces(int64_t S, int32_t P, int32_t layout) {
  std::vector<std::vector<Piece>> out(P);
  if (layout == CP_REORDER_CONTIGUOUS) {
    int32_t C = (int32_t)(S / P);
    for (int r = 0; r < P; ++r) out[r].push_back({r * C, C, r * C, 1});
  } else if (layout == CP_REORDER_DUAL_CHUNK_SWAP) {
    int32_t C = (int32_t)(S / (2 * P));
    for (int r = 0; r < P; ++r) {
      out[r].push_back({2 * r * C, C, r * C, 1});
      out[r].push_back({2 * r * C + C, C, (2 * P - 1 - r) * C, 1});
    }
  } else {  // striped
    int32_t n = (int32_t)(S / P);
    for (int r = 0; r < P; ++r) out[r].push_back({r * n, n, r, P});
  }
  return out;
}

int64_t piece_pos_max(const Piece& p) { return (int64_t)p.pos_off + (int64_t)p.pos_stride * (p.n - 1); }

// Could any key of `k` be visible to any query of `q` under the causal rule?
bool maybe_visible(const Piece& q, const Piece& k, int causal) {
  if (q.n == 0 || k.n == 0) return false;
  if (!causal) return true;
  return k.pos_off <= piece_pos_max(q);
}

void add_group(Schedule& s, const Piece& q) {
  QGroup& g = s.g[s.n_groups++];
  memset(&g, 0, sizeof(g));
  g.q_row0 = q.row0;
  g.nq = q.n;
  g.pos_off = q.pos_off;
  g.pos_stride = q.pos_stride;
  g.seg_begin = s.n_segs;
  g.seg_count = 0;
  g.lse_col0 = q.row0;
  g.lse_head0 = 0;
  g.o_row0 = q.row0;
}

void add_seg(Schedule& s, const Piece& k) {
  KSeg& sg = s.s[s.n_segs++];
  sg.k_row0 = k.row0;
  sg.nk = k.n;
  sg.pos_off = k.pos_off;
  sg.pos_stride = k.pos_stride;
  s.g[s.n_groups - 1].seg_count++;
}

// Heaviest group first (more key rows to visit), so long query tiles start early.
void sort_groups_by_work(Schedule& s) {
  std::vector<int> idx(s.n_groups);
  std::vector<int64_t> w(s.n_groups, 0);
  for (int i = 0; i < s.n_groups; ++i) {
    idx[i] = i;
    for (int k = 0; k < s.g[i].seg_count; ++k) w[i] += s.s[s.g[i].seg_begin + k].nk;
    w[i] *= (int64_t)s.g[i].nq > 0 ? 1 : 0;
  }
  std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) { return w[a] > w[b]; });
  QGroup tmp[kMaxGroups];
  for (int i = 0; i < s.n_groups; ++i) tmp[i] = s.g[idx[i]];
  for (int i = 0; i < s.n_groups; ++i) s.g[i] = tmp[i];
}

// Ring schedule.  step < 0: every step (fused); else only that step.  seq_out:
// out rows and lse columns go to the pieces' sequence positions instead of their
// rows in the ranks' layout (pieces of consecutive positions only), i.e. the
// restore is done by the attention's own output writes.
void build_ring_schedule(Schedule& s, int64_t S, int32_t P, int32_t layout, int step, int causal,
                         bool seq_out = false) {
  auto pieces = rank_pieces(S, P, layout);
  s.n_groups = 0;
  s.n_segs = 0;
  for (int r = 0; r < P; ++r) {
    for (const Piece& q : pieces[r]) {
      add_group(s, q);
      if (seq_out) {
        s.g[s.n_groups - 1].o_row0 = q.pos_off;
        s.g[s.n_groups - 1].lse_col0 = q.pos_off;
      }
      for (int st = 0; st < P; ++st) {
        if (step >= 0 && st != step) continue;
        int src = ((r - st) % P + P) % P;
        for (const Piece& k : pieces[src])
          if (maybe_visible(q, k, causal)) add_seg(s, k);
      }
    }
  }
  sort_groups_by_work(s);
}

// Key-major schedule for the backward: one group per key piece, segments =
// the query pieces that may see it.
void build_ring_bwd_schedule(Schedule& s, int64_t S, int32_t P, int32_t layout, int causal) {
  auto pieces = rank_pieces(S, P, layout);
  s.n_groups = 0;
  s.n_segs = 0;
  for (int r = 0; r < P; ++r)
    for (const Piece& k : pieces[r]) {
      add_group(s, k);
      for (int r2 = 0; r2 < P; ++r2)
        for (const Piece& q : pieces[r2])
          if (maybe_visible(q, k, causal)) add_seg(s, q);
    }
  sort_groups_by_work(s);
}

int32_t resolve_layout(int32_t reorder, const int32_t* cu) {
  if (reorder == CP_REORDER_AUTO) return cu ? CP_REORDER_STRIPED : CP_REORDER_DUAL_CHUNK_SWAP;
  return reorder;
}

cp_status launch_fwd(const AttnArgs& a0, Schedule& s, int32_t dtype, int64_t q_rows,
                     int64_t k_rows, cudaStream_t st) {
  // buffer extents for the debug build's index checks: q and o share their rows; the
  // lse array holds the heads the schedule's groups reach
  AttnArgs a = a0;
  a.q_rows = q_rows;
  a.k_rows = k_rows;
  int64_t heads = 0;
  for (int i = 0; i < s.n_groups; ++i) heads = std::max<int64_t>(heads, (int64_t)s.g[i].lse_head0 + a.Hq);
  a.lse_size = heads * a.lse_ld;
  if (dtype == CP_BF16) return launch_attn_fwd_tc(a, s, q_rows, k_rows, st);
  return launch_attn_fwd_simt(a, s, 0, st);
}

}  // namespace
bool cpa::bwd_writes_bf16(int32_t dtype, int32_t D) { return dtype == CP_BF16 && (D == 64 || D == 128); }

bool cpa::grads_apart(const void* const* outs, const size_t* out_bytes, int n_out, const void* const* ins,
                      const size_t* in_bytes, int n_in) {
  for (int i = 0; i < n_out; ++i)
    for (int j = 0; j < n_in; ++j) {
      const char* o = static_cast<const char*>(outs[i]);
      const char* x = static_cast<const char*>(ins[j]);
      if (o && x && !(o + out_bytes[i] <= x || x + in_bytes[j] <= o)) return false;
    }
  return true;
}
namespace {

cp_status launch_bwd(const BwdArgs& a0, Schedule& s, int32_t dtype, int64_t q_rows,
                     int64_t k_rows, cudaStream_t st) {
  BwdArgs a = a0;  // buffer extents for the debug build's index checks
  a.q_rows = q_rows;
  a.k_rows = k_rows;
  a.lse_size = (int64_t)a.Hq * a.lse_ld;
  // bf16 runs on the tensor-core kernels (D = 64 or 128); fp32 on the exact FFMA kernel.
  if (bwd_writes_bf16(dtype, a.D)) return launch_attn_bwd_tc(a, s, q_rows, k_rows, st);
  return launch_attn_bwd_simt(a, s, dtype == CP_BF16, st);
}

AttnArgs make_fwd_args(const void* q, const void* k, const void* v, void* o, float* lse,
                       int32_t Hq, int32_t Hkv, int32_t D, int64_t lse_ld, int32_t causal,
                       const int32_t* cu, int32_t n_docs, float scale, int o_f32) {
  AttnArgs a;
  memset(&a, 0, sizeof(a));
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.q_ld = (int64_t)Hq * D;
  a.k_ld = (int64_t)Hkv * D;
  a.o_ld = (int64_t)Hq * D;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.lse_ld = (int32_t)lse_ld;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.causal = causal;
  a.cu_seqlens = cu;
  a.n_docs = cu ? n_docs : 0;
  a.err = device_error_word();
  a.o_f32 = o_f32;
  return a;
}

// ---------------------------------------------------------------- workspace layouts
// Partial results of the STEPWISE ring (fp32), relative to their own base.
struct RingPartialsWs {
  size_t o_acc, lse_acc, o_step, lse_step, total;
};
RingPartialsWs ring_partials_ws(int64_t S, int32_t Hq, int32_t D, int32_t mode) {
  RingPartialsWs w;
  size_t off = 0;
  w.o_acc = w.lse_acc = w.o_step = w.lse_step = 0;
  if (mode == CP_RING_STEPWISE) {
    w.o_acc = off; off += align_up((size_t)S * Hq * D * 4);
    w.lse_acc = off; off += align_up((size_t)S * Hq * 4);
    w.o_step = off; off += align_up((size_t)S * Hq * D * 4);
    w.lse_step = off; off += align_up((size_t)S * Hq * 4);
  }
  w.total = off;
  return w;
}

struct RingFwdWs {
  size_t q, k, v, o, lse, partials, total;
  RingPartialsWs pw;
};
RingFwdWs ring_fwd_ws(int64_t S, int32_t Hq, int32_t Hkv, int32_t D, int32_t dtype, int32_t mode) {
  RingFwdWs w;
  size_t es = dtype_size(dtype);
  size_t off = 0;
  w.q = off; off += align_up((size_t)S * Hq * D * es);
  w.k = off; off += align_up((size_t)S * Hkv * D * es);
  w.v = off; off += align_up((size_t)S * Hkv * D * es);
  w.o = off; off += align_up((size_t)S * Hq * D * es);
  w.lse = off; off += align_up((size_t)S * Hq * 4);
  w.pw = ring_partials_ws(S, Hq, D, mode);
  w.partials = off; off += w.pw.total;
  w.total = off;
  return w;
}

struct RingBwdWs {
  size_t q, k, v, o, dout, lse, delta, dq, dk, dv, total;
};
RingBwdWs ring_bwd_ws(int64_t S, int32_t Hq, int32_t Hkv, int32_t D, int32_t dtype) {
  RingBwdWs w;
  size_t es = dtype_size(dtype);
  size_t off = 0;
  w.q = off; off += align_up((size_t)S * Hq * D * es);
  w.k = off; off += align_up((size_t)S * Hkv * D * es);
  w.v = off; off += align_up((size_t)S * Hkv * D * es);
  w.o = off; off += align_up((size_t)S * Hq * D * es);
  w.dout = off; off += align_up((size_t)S * Hq * D * es);
  w.lse = off; off += align_up((size_t)S * Hq * 4);
  w.delta = off; off += align_up((size_t)S * Hq * 4);
  w.dq = off; off += align_up((size_t)S * Hq * D * 4);
  w.dk = off; off += align_up((size_t)S * Hkv * D * 4);
  w.dv = off; off += align_up((size_t)S * Hkv * D * 4);
  w.total = off;
  return w;
}

struct BlockBwdWs {
  size_t delta, dq, dk, dv, total;
};
BlockBwdWs block_bwd_ws(int64_t Sq, int64_t Sk, int32_t Hq, int32_t Hkv, int32_t D) {
  BlockBwdWs w;
  size_t off = 0;
  w.delta = off; off += align_up((size_t)Sq * Hq * 4);
  w.dq = off; off += align_up((size_t)Sq * Hq * D * 4);
  w.dk = off; off += align_up((size_t)Sk * Hkv * D * 4);
  w.dv = off; off += align_up((size_t)Sk * Hkv * D * 4);
  w.total = off;
  return w;
}

// Copies of each key/value head in the Ulysses exchange ("Ulysses: transposing
// between the sequence and the heads": the exchange hands every rank H/P heads;
// with fewer key/value heads than ranks they are replicated by group first).
// R = 1 when Hkv % P == 0; R = P / Hkv when P % Hkv == 0; 0 (unsupported) otherwise.
int32_t ulysses_kv_replicas(int32_t Hkv, int32_t P) {
  if (Hkv % P == 0) return 1;
  if (P % Hkv == 0) return P / Hkv;
  return 0;
}

struct UlyssesWs {
  size_t q, k, v, o, total;
};
UlyssesWs ulysses_ws(int64_t S, int32_t Hq, int32_t Hkv, int32_t D, int32_t dtype, int32_t P) {
  UlyssesWs w;
  size_t es = dtype_size(dtype);
  const int32_t R = ulysses_kv_replicas(Hkv, P) > 0 ? ulysses_kv_replicas(Hkv, P) : 1;
  size_t off = 0;
  w.q = off; off += align_up((size_t)S * Hq * D * es);
  w.k = off; off += align_up((size_t)S * Hkv * R * D * es);
  w.v = off; off += align_up((size_t)S * Hkv * R * D * es);
  w.o = off; off += align_up((size_t)S * Hq * D * es);
  w.total = off;
  return w;
}

// Ulysses inside groups x ring across groups: the ring-ordered q, k, v, their
// head-major copies (the ring-ordered buffers then hold the head-major output
// and the head-major q copy the ring-ordered output), and lse in ring order.
struct UspWs {
  size_t q_re, k_re, v_re, qh, kh, vh, lse, total;
};
UspWs usp_ws(int64_t S, int32_t Hq, int32_t Hkv, int32_t D, int32_t dtype) {
  UspWs w;
  size_t es = dtype_size(dtype);
  const size_t nq = (size_t)S * Hq * D * es, nkv = (size_t)S * Hkv * D * es;
  size_t off = 0;
  w.q_re = off; off += align_up(nq);
  w.k_re = off; off += align_up(nkv);
  w.v_re = off; off += align_up(nkv);
  w.qh = off; off += align_up(nq);
  w.kh = off; off += align_up(nkv);
  w.vh = off; off += align_up(nkv);
  w.lse = off; off += align_up((size_t)S * Hq * 4);
  w.total = off;
  return w;
}

// Ulysses backward: q, k, v, dout in the head-major layout, lse and Delta in the
// head-major row order, fp32 gradient accumulators in the head-major layout.
struct UlyssesBwdWs {
  size_t q, k, v, dout, delta, lse_h, delta_h, dq, dk, dv, total;
};
UlyssesBwdWs ulysses_bwd_ws(int64_t S, int32_t Hq, int32_t Hkv, int32_t D, int32_t dtype, int32_t P) {
  UlyssesBwdWs w;
  size_t es = dtype_size(dtype);
  const int32_t R = ulysses_kv_replicas(Hkv, P) > 0 ? ulysses_kv_replicas(Hkv, P) : 1;
  const size_t nq = (size_t)S * Hq * D, nkv = (size_t)S * Hkv * R * D;
  size_t off = 0;
  w.q = off; off += align_up(nq * es);
  w.k = off; off += align_up(nkv * es);
  w.v = off; off += align_up(nkv * es);
  w.dout = off; off += align_up(nq * es);
  w.delta = off; off += align_up((size_t)S * Hq * 4);
  w.lse_h = off; off += align_up((size_t)S * Hq * 4);
  w.delta_h = off; off += align_up((size_t)S * Hq * 4);
  w.dq = off; off += align_up(nq * 4);
  w.dk = off; off += align_up(nkv * 4);
  w.dv = off; off += align_up(nkv * 4);
  w.total = off;
  return w;
}

char* ws_at(void* base, size_t off) { return static_cast<char*>(base) + off; }

// The ring over P virtual ranks on buffers already in the ranks' layout:
// q/k/v rows in rank order; o rows and lse columns in rank order, or in sequence
// order when seq_out (FUSED mode, zigzag or contiguous layout: every piece is a
// run of consecutive positions, so the attention writes each row where the
// restore would have put it).
cp_status ring_core(const void* q_re, const void* k_re, const void* v_re, void* o_re, float* lse_re,
                    int64_t S, int32_t Hq, int32_t Hkv, int32_t D, int32_t dtype, int32_t P,
                    int32_t layout, int32_t mode, const int32_t* cu_seqlens, int32_t n_docs,
                    void* partials, const RingPartialsWs& w, cudaStream_t st, bool seq_out = false) {
  const float scale = 1.0f / sqrtf((float)D);
  Schedule* s = new Schedule;
  cp_status result = CP_OK;
  if (mode == CP_RING_FUSED && layout == CP_REORDER_STRIPED && dtype == CP_BF16 && D == 128 &&
      (P == 4 || P == 8 || P == 16)) {
    // Striped, position-tiled: every rank's rows are in this GPU's memory, so the
    // kernel tiles by position (a tile = 128/P rows of each rank, 128 consecutive
    // positions) instead of by rank; the online softmax still merges every key
    // block a query row sees, and the result is the ring's.  Each query tile then
    // meets one causal diagonal instead of one per source rank.
    s->n_groups = 0;
    s->n_segs = 0;
    add_group(*s, Piece{0, (int32_t)S, 0, 1});
    add_seg(*s, Piece{0, (int32_t)S, 0, 1});
    AttnArgs a = make_fwd_args(q_re, k_re, v_re, o_re, lse_re, Hq, Hkv, D, S, 1, cu_seqlens,
                               n_docs, scale, 0);
    a.perm_p = P;
    a.perm_n = (int32_t)(S / P);
    result = launch_fwd(a, *s, dtype, S, S, st);
  } else if (mode == CP_RING_FUSED) {
    build_ring_schedule(*s, S, P, layout, -1, 1, seq_out);
    AttnArgs a = make_fwd_args(q_re, k_re, v_re, o_re, lse_re, Hq, Hkv, D, S, 1, cu_seqlens,
                               n_docs, scale, 0);
    result = launch_fwd(a, *s, dtype, S, S, st);
  } else {
    float* o_acc = reinterpret_cast<float*>(ws_at(partials, w.o_acc));
    float* lse_acc = reinterpret_cast<float*>(ws_at(partials, w.lse_acc));
    float* o_step = reinterpret_cast<float*>(ws_at(partials, w.o_step));
    float* lse_step = reinterpret_cast<float*>(ws_at(partials, w.lse_step));
    for (int step = 0; step < P && result == CP_OK; ++step) {
      build_ring_schedule(*s, S, P, layout, step, 1);
      float* o_dst = step == 0 ? o_acc : o_step;
      float* l_dst = step == 0 ? lse_acc : lse_step;
      AttnArgs a = make_fwd_args(q_re, k_re, v_re, o_dst, l_dst, Hq, Hkv, D, S, 1, cu_seqlens,
                                 n_docs, scale, 1);
      result = launch_fwd(a, *s, dtype, S, S, st);
      if (result == CP_OK && step > 0)
        result = launch_lse_merge(o_acc, lse_acc, o_step, lse_step, o_acc, lse_acc, S, Hq, D, 1, st);
    }
    if (result == CP_OK) result = launch_cast_out(o_acc, o_re, S * Hq * D, dtype == CP_BF16, st);
    if (result == CP_OK)
      result = cuda_check(cudaMemcpyAsync(lse_re, lse_acc, (size_t)S * Hq * 4,
                                          cudaMemcpyDeviceToDevice, st), "lse copy");
  }
  delete s;
  return result;
}

cp_status check_ring_args(int64_t S, int32_t Hq, int32_t Hkv, int32_t D, int32_t dtype, int32_t P,
                          int32_t layout, const int32_t* cu, int32_t n_docs) {
  CP_TRY(check_common(Hq, Hkv, D, dtype));
  CP_REQUIRE(P >= 1 && P <= 32, CP_ERR_INVALID_ARG, "P must be in [1, 32]");
  CP_REQUIRE(S >= 0, CP_ERR_INVALID_ARG, "S must be >= 0");
  CP_REQUIRE(layout >= CP_REORDER_CONTIGUOUS && layout <= CP_REORDER_STRIPED, CP_ERR_INVALID_ARG,
             "reorder must be a cp_reorder value");
  if (layout == CP_REORDER_DUAL_CHUNK_SWAP) {
    CP_REQUIRE(S % (2 * P) == 0, CP_ERR_SHAPE, "DUAL_CHUNK_SWAP needs S % (2P) == 0");
    CP_REQUIRE(P <= 16, CP_ERR_UNSUPPORTED, "DUAL_CHUNK_SWAP supports P <= 16");
  } else {
    CP_REQUIRE(S % P == 0, CP_ERR_SHAPE, "ring needs S % P == 0");
  }
  CP_REQUIRE(S * (int64_t)Hq < (int64_t)INT32_MAX, CP_ERR_UNSUPPORTED, "S*Hq must be < 2^31");
  if (cu) {
    CP_REQUIRE(layout != CP_REORDER_CONTIGUOUS, CP_ERR_UNSUPPORTED,
               "packed documents are supported only with a load-balanced ring "
               "(DUAL_CHUNK_SWAP, STRIPED or AUTO)");
    CP_REQUIRE(n_docs >= 1, CP_ERR_INVALID_ARG, "n_docs must be >= 1 with cu_seqlens");
  }
  return CP_OK;
}

}  // namespace

cp_status cpa::check_block_args(int64_t Sq, int64_t Sk, int32_t Hq, int32_t Hkv, int32_t D, int32_t dtype,
                                const cp_mask* mask, cp_mask* m) {
  CP_TRY(check_common(Hq, Hkv, D, dtype));
  CP_REQUIRE(Sq >= 0 && Sk >= 0, CP_ERR_INVALID_ARG, "Sq and Sk must be >= 0");
  CP_REQUIRE(Sq * (int64_t)Hq < (int64_t)INT32_MAX && Sk * (int64_t)Hkv < (int64_t)INT32_MAX,
             CP_ERR_UNSUPPORTED, "S*H must be < 2^31");
  *m = cp_mask{1, 0, 0, 1, 1, nullptr, 0, 0};
  if (mask) *m = *mask;
  CP_REQUIRE(m->q_stride >= 1 && m->k_stride >= 1, CP_ERR_INVALID_ARG, "mask strides must be >= 1");
  CP_REQUIRE(m->window >= 0, CP_ERR_INVALID_ARG, "mask window must be >= 0");
  CP_REQUIRE(m->window == 0 || m->causal, CP_ERR_UNSUPPORTED, "a sliding window needs the causal rule");
  // Offsets and strides are bounded before any product is formed, so the
  // position arithmetic below cannot overflow int64.
  CP_REQUIRE(fits_i32(m->q_offset) && fits_i32(m->k_offset) && m->q_stride <= INT32_MAX &&
                 m->k_stride <= INT32_MAX,
             CP_ERR_UNSUPPORTED, "positions must fit in int32");
  CP_REQUIRE(fits_i32(m->q_offset + m->q_stride * (Sq > 0 ? Sq - 1 : 0)) &&
                 fits_i32(m->k_offset + m->k_stride * (Sk > 0 ? Sk - 1 : 0)),
             CP_ERR_UNSUPPORTED, "positions must fit in int32");
  CP_REQUIRE(!m->cu_seqlens || m->n_docs >= 1, CP_ERR_INVALID_ARG, "n_docs must be >= 1 with cu_seqlens");
  return CP_OK;
}

cp_status cpa::block_bwd_run(const void* q, const void* k, const void* v, const void* out, const void* dout,
                             const float* lse, int64_t Sq, int64_t Sk, int32_t Hq, int32_t Hkv, int32_t D,
                             int32_t dtype, const cp_mask& m, float scale, const BlockBwdOut& o, float* delta,
                             cudaStream_t st) {
  const int is_bf16 = dtype == CP_BF16;
  const bool tc = bwd_writes_bf16(dtype, D);
  bool direct = false;  // typed bf16 gradients written by the tensor-core kernels themselves
  if (o.typed) {
    // Every gradient row is written once, in bf16, with no zeroing or cast pass, but
    // only into outputs that share no bytes with what the kernels still read.
    const size_t qb = (size_t)Sq * Hq * D * dtype_size(dtype), kb = (size_t)Sk * Hkv * D * dtype_size(dtype);
    const void* outs[3] = {o.dq, o.dk, o.dv};
    const size_t ob[3] = {qb, kb, kb};
    const void* ins[5] = {q, k, v, dout, lse};
    const size_t ib[5] = {qb, kb, kb, qb, (size_t)Sq * Hq * 4};
    direct = tc && Sq > 0 && Sk > 0 && grads_apart(outs, ob, 3, ins, ib, 5);
    if (!direct) {
      CP_TRY(launch_zero(o.dq_acc, (size_t)Sq * Hq * D * 4, st));
      CP_TRY(launch_zero(o.dk_acc, (size_t)Sk * Hkv * D * 4, st));
      CP_TRY(launch_zero(o.dv_acc, (size_t)Sk * Hkv * D * 4, st));
    }
  } else if (!tc && !o.accumulate) {
    // the FFMA kernel adds dQ atomically (dK/dV rows are stored once): start it at zero
    CP_TRY(launch_zero(o.dq_acc, (size_t)Sq * Hq * D * 4, st));
  }
  CP_TRY(launch_bwd_preprocess(out, dout, delta, Sq, Hq, D, (int32_t)Sq, is_bf16, st));
  Schedule* s = new Schedule;
  s->n_groups = 0;
  s->n_segs = 0;
  add_group(*s, Piece{0, (int32_t)Sk, (int32_t)m.k_offset, (int32_t)m.k_stride});
  if (Sq > 0) add_seg(*s, Piece{0, (int32_t)Sq, (int32_t)m.q_offset, (int32_t)m.q_stride});
  BwdArgs a;
  memset(&a, 0, sizeof(a));
  a.q = q; a.k = k; a.v = v; a.dout = dout; a.lse = lse; a.delta = delta;
  a.dq_acc = o.dq_acc; a.dk_acc = o.dk_acc; a.dv_acc = o.dv_acc;
  a.q_ld = (int64_t)Hq * D; a.k_ld = (int64_t)Hkv * D;
  a.Hq = Hq; a.Hkv = Hkv; a.D = D; a.lse_ld = (int32_t)Sq;
  a.scale = scale; a.scale_log2 = scale * 1.4426950408889634f;
  a.causal = m.causal; a.cu_seqlens = m.cu_seqlens; a.n_docs = m.cu_seqlens ? m.n_docs : 0;
  a.window = m.window;
  a.accumulate = o.typed ? 0 : o.accumulate;
  a.err = device_error_word();
  if (direct) {
    a.dq_out = o.dq; a.dk_out = o.dk; a.dv_out = o.dv;
  }
  cp_status stt = launch_bwd(a, *s, dtype, Sq, Sk, st);
  delete s;
  CP_TRY(stt);
  if (o.typed && !direct) {
    CP_TRY(launch_cast_out(o.dq_acc, o.dq, Sq * Hq * D, is_bf16, st));
    CP_TRY(launch_cast_out(o.dk_acc, o.dk, Sk * Hkv * D, is_bf16, st));
    CP_TRY(launch_cast_out(o.dv_acc, o.dv, Sk * Hkv * D, is_bf16, st));
  }
  return CP_OK;
}

// ====================================================================== C ABI
extern "C" {

const char* cp_version(void) { return "0.1.0"; }

const char* cp_last_error(void) { return g_last_error.c_str(); }

const char* cp_status_string(int32_t st) {
  switch (st) {
    case CP_OK: return "CP_OK";
    case CP_ERR_INVALID_ARG: return "CP_ERR_INVALID_ARG";
    case CP_ERR_SHAPE: return "CP_ERR_SHAPE";
    case CP_ERR_DTYPE: return "CP_ERR_DTYPE";
    case CP_ERR_ALIGN: return "CP_ERR_ALIGN";
    case CP_ERR_UNSUPPORTED: return "CP_ERR_UNSUPPORTED";
    case CP_ERR_WORKSPACE: return "CP_ERR_WORKSPACE";
    case CP_ERR_CUDA: return "CP_ERR_CUDA";
    case CP_ERR_DEVICE_TIMEOUT: return "CP_ERR_DEVICE_TIMEOUT";
    case CP_ERR_DEVICE_INDEX: return "CP_ERR_DEVICE_INDEX";
    default: return "CP_ERR_UNKNOWN";
  }
}

cp_status cp_attn_block_fwd(const void* q, const void* k, const void* v, int64_t Sq, int64_t Sk,
                            int32_t Hq, int32_t Hkv, int32_t D, int32_t dtype, const cp_mask* mask,
                            float scale, void* out, float* lse, void* stream) {
  cp_mask m;
  CP_TRY(check_block_args(Sq, Sk, Hq, Hkv, D, dtype, mask, &m));
  if (Sq == 0) return CP_OK;
  CP_CHECK_T(q, "q", false);
  CP_CHECK_T(k, "k", Sk == 0);
  CP_CHECK_T(v, "v", Sk == 0);
  CP_CHECK_T(out, "out", false);
  CP_CHECK_T(lse, "lse", false);
  if (scale == 0.f) scale = 1.0f / sqrtf((float)D);
  Schedule* s = new Schedule;
  s->n_groups = 0;
  s->n_segs = 0;
  add_group(*s, Piece{0, (int32_t)Sq, (int32_t)m.q_offset, (int32_t)m.q_stride});
  s->g[0].lse_col0 = 0;
  if (Sk > 0) add_seg(*s, Piece{0, (int32_t)Sk, (int32_t)m.k_offset, (int32_t)m.k_stride});
  AttnArgs a = make_fwd_args(q, k, v, out, lse, Hq, Hkv, D, Sq, m.causal, m.cu_seqlens, m.n_docs,
                             scale, 0);
  a.window = m.window;
  cp_status st = launch_fwd(a, *s, dtype, Sq, Sk, (cudaStream_t)stream);
  delete s;
  return st;
}

// Pointer checks shared by both block backward forms (q side when Sq > 0, k side when Sk > 0).
static cp_status check_block_bwd_ptrs(const void* q, const void* k, const void* v, const void* out,
                                      const void* dout, const float* lse, const void* dq, const void* dk,
                                      const void* dv, int64_t Sq, int64_t Sk) {
  CP_CHECK_T(q, "q", Sq == 0);
  CP_CHECK_T(out, "out", Sq == 0);
  CP_CHECK_T(dout, "dout", Sq == 0);
  CP_CHECK_T(lse, "lse", Sq == 0);
  CP_CHECK_T(dq, "dq", Sq == 0);
  CP_CHECK_T(k, "k", Sk == 0);
  CP_CHECK_T(v, "v", Sk == 0);
  CP_CHECK_T(dk, "dk", Sk == 0);
  CP_CHECK_T(dv, "dv", Sk == 0);
  return CP_OK;
}

cp_status cp_attn_block_bwd(const void* q, const void* k, const void* v, const void* out,
                            const void* dout, const float* lse, int64_t Sq, int64_t Sk, int32_t Hq,
                            int32_t Hkv, int32_t D, int32_t dtype, const cp_mask* mask, float scale,
                            float* dq_acc, float* dk_acc, float* dv_acc, int32_t accumulate,
                            void* workspace, size_t ws_bytes, void* stream) {
  cp_mask m;
  CP_TRY(check_block_args(Sq, Sk, Hq, Hkv, D, dtype, mask, &m));
  CP_REQUIRE(accumulate == 0 || accumulate == 1, CP_ERR_INVALID_ARG, "accumulate must be 0 or 1");
  if (Sq == 0 && Sk == 0) return CP_OK;
  const size_t delta_bytes = align_up((size_t)Sq * Hq * 4);
  CP_REQUIRE(Sq == 0 || (workspace && ws_bytes >= delta_bytes), CP_ERR_WORKSPACE,
             "workspace too small for the block backward (4*Hq*Sq bytes of Delta)");
  if (Sq > 0) CP_CHECK_T(workspace, "workspace", false);
  CP_TRY(check_block_bwd_ptrs(q, k, v, out, dout, lse, dq_acc, dk_acc, dv_acc, Sq, Sk));
  // The fp32 outputs are read back when accumulating and written while the kernels
  // still read the inputs: they may overlap neither an input nor each other.
  const size_t es = dtype_size(dtype);
  const size_t qb = (size_t)Sq * Hq * D * es, kb = (size_t)Sk * Hkv * D * es;
  const size_t qa = (size_t)Sq * Hq * D * 4, ka = (size_t)Sk * Hkv * D * 4;
  const void* outs[3] = {dq_acc, dk_acc, dv_acc};
  const size_t ob[3] = {qa, ka, ka};
  const void* ins[7] = {q, k, v, out, dout, lse, Sq > 0 ? workspace : nullptr};
  const size_t ib[7] = {qb, kb, kb, qb, qb, (size_t)Sq * Hq * 4, delta_bytes};
  CP_REQUIRE(grads_apart(outs, ob, 3, ins, ib, 7) && grads_apart(outs, ob, 1, outs + 1, ob + 1, 2) &&
                 grads_apart(outs + 1, ob + 1, 1, outs + 2, ob + 2, 1),
             CP_ERR_INVALID_ARG,
             "dq_acc, dk_acc and dv_acc must not overlap an input, the workspace or each other");
  if (scale == 0.f) scale = 1.0f / sqrtf((float)D);
  BlockBwdOut o;
  memset(&o, 0, sizeof(o));
  o.typed = false;
  o.dq_acc = dq_acc;
  o.dk_acc = dk_acc;
  o.dv_acc = dv_acc;
  o.accumulate = accumulate;
  return block_bwd_run(q, k, v, out, dout, lse, Sq, Sk, Hq, Hkv, D, dtype, m, scale, o,
                       static_cast<float*>(workspace), (cudaStream_t)stream);
}

cp_status cp_attn_block_bwd_typed(const void* q, const void* k, const void* v, const void* out,
                                  const void* dout, const float* lse, int64_t Sq, int64_t Sk, int32_t Hq,
                                  int32_t Hkv, int32_t D, int32_t dtype, const cp_mask* mask, float scale,
                                  void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                                  void* stream) {
  cp_mask m;
  CP_TRY(check_block_args(Sq, Sk, Hq, Hkv, D, dtype, mask, &m));
  if (Sq == 0 && Sk == 0) return CP_OK;
  BlockBwdWs w = block_bwd_ws(Sq, Sk, Hq, Hkv, D);
  CP_REQUIRE(workspace && ws_bytes >= w.total, CP_ERR_WORKSPACE, "workspace too small for block bwd");
  CP_CHECK_T(workspace, "workspace", false);
  CP_TRY(check_block_bwd_ptrs(q, k, v, out, dout, lse, dq, dk, dv, Sq, Sk));
  if (scale == 0.f) scale = 1.0f / sqrtf((float)D);
  BlockBwdOut o;
  o.typed = true;
  o.dq = dq;
  o.dk = dk;
  o.dv = dv;
  o.dq_acc = reinterpret_cast<float*>(ws_at(workspace, w.dq));
  o.dk_acc = reinterpret_cast<float*>(ws_at(workspace, w.dk));
  o.dv_acc = reinterpret_cast<float*>(ws_at(workspace, w.dv));
  o.accumulate = 0;
  return block_bwd_run(q, k, v, out, dout, lse, Sq, Sk, Hq, Hkv, D, dtype, m, scale, o,
                       reinterpret_cast<float*>(ws_at(workspace, w.delta)), (cudaStream_t)stream);
}

cp_status cp_lse_merge(const void* o1, const float* lse1, const void* o2, const float* lse2,
                       void* o, float* lse, int64_t Sq, int32_t H, int32_t D, int32_t o_dtype,
                       void* stream) {
  CP_REQUIRE(o_dtype == CP_F32 || o_dtype == CP_BF16, CP_ERR_DTYPE, "o_dtype must be CP_F32 or CP_BF16");
  CP_REQUIRE(Sq >= 0 && H >= 1 && D >= 1, CP_ERR_INVALID_ARG, "Sq >= 0, H >= 1, D >= 1 required");
  CP_REQUIRE(((size_t)D * dtype_size(o_dtype)) % 16 == 0, CP_ERR_ALIGN,
             "D * sizeof(o_dtype) must be a multiple of 16 bytes");
  CP_REQUIRE((size_t)D * dtype_size(o_dtype) <= 512, CP_ERR_UNSUPPORTED,
             "D * sizeof(o_dtype) must be <= 512 bytes");
  if (Sq == 0) return CP_OK;
  CP_CHECK_T(o1, "o1", false);
  CP_CHECK_T(o2, "o2", false);
  CP_CHECK_T(o, "o", false);
  CP_REQUIRE(lse1 && lse2 && lse, CP_ERR_INVALID_ARG, "lse pointers must not be NULL");
  return launch_lse_merge(o1, lse1, o2, lse2, o, lse, Sq, H, D, o_dtype == CP_F32,
                          (cudaStream_t)stream);
}

static cp_status permute_common(int kind, const void* x, void* y, int64_t S, int32_t H, int32_t D,
                                int32_t P, int32_t dtype, void* stream) {
  CP_REQUIRE(dtype == CP_F32 || dtype == CP_BF16, CP_ERR_DTYPE, "dtype must be CP_F32 or CP_BF16");
  CP_REQUIRE(S >= 0 && H >= 1 && D >= 1, CP_ERR_INVALID_ARG, "S >= 0, H >= 1, D >= 1 required");
  CP_REQUIRE(P >= 1 && P <= 1024, CP_ERR_INVALID_ARG, "P must be in [1, 1024]");
  size_t row_bytes = (size_t)H * D * dtype_size(dtype);
  if (kind == kSeq2Head || kind == kHead2Seq) {
    CP_REQUIRE(S % P == 0, CP_ERR_SHAPE, "Ulysses needs S % P == 0");
    CP_REQUIRE(H % P == 0, CP_ERR_SHAPE, "Ulysses needs H % P == 0 (degree limited by heads)");
    CP_REQUIRE((row_bytes / P) % 16 == 0, CP_ERR_ALIGN,
               "(H/P)*D*sizeof(dtype) must be a multiple of 16 bytes");
    CP_REQUIRE((uint64_t)S * P < (1ull << 32), CP_ERR_UNSUPPORTED, "S*P must be < 2^32");
  } else if (kind == kZigzagReorder || kind == kZigzagRestore) {
    CP_REQUIRE(S % (2 * P) == 0, CP_ERR_SHAPE, "zigzag needs S % (2P) == 0");
    CP_REQUIRE(row_bytes % 16 == 0, CP_ERR_ALIGN, "H*D*sizeof(dtype) must be a multiple of 16 bytes");
  } else {
    CP_REQUIRE(S % P == 0, CP_ERR_SHAPE, "striped needs S % P == 0");
    CP_REQUIRE(row_bytes % 16 == 0, CP_ERR_ALIGN, "H*D*sizeof(dtype) must be a multiple of 16 bytes");
  }
  if (S == 0) return CP_OK;
  CP_CHECK_T(x, "x", false);
  CP_CHECK_T(y, "y", false);
  const char* xb = static_cast<const char*>(x);
  const char* yb = static_cast<const char*>(y);
  size_t nbytes = (size_t)S * row_bytes;
  CP_REQUIRE(xb + nbytes <= yb || yb + nbytes <= xb, CP_ERR_INVALID_ARG, "x and y must not overlap");
  return launch_row_gather(kind, x, y, S, (int64_t)row_bytes, P, H, (cudaStream_t)stream);
}

cp_status cp_ulysses_seq2head(const void* x, void* y, int64_t S, int32_t H, int32_t D, int32_t P,
                              int32_t dtype, void* stream) {
  return permute_common(kSeq2Head, x, y, S, H, D, P, dtype, stream);
}
cp_status cp_ulysses_head2seq(const void* y, void* x, int64_t S, int32_t H, int32_t D, int32_t P,
                              int32_t dtype, void* stream) {
  return permute_common(kHead2Seq, y, x, S, H, D, P, dtype, stream);
}
cp_status cp_zigzag_reorder(const void* x, void* y, int64_t S, int32_t H, int32_t D, int32_t P,
                            int32_t dtype, void* stream) {
  return permute_common(kZigzagReorder, x, y, S, H, D, P, dtype, stream);
}
cp_status cp_zigzag_restore(const void* y, void* x, int64_t S, int32_t H, int32_t D, int32_t P,
                            int32_t dtype, void* stream) {
  return permute_common(kZigzagRestore, y, x, S, H, D, P, dtype, stream);
}
cp_status cp_striped_reorder(const void* x, void* y, int64_t S, int32_t H, int32_t D, int32_t P,
                             int32_t dtype, void* stream) {
  return permute_common(kStripedReorder, x, y, S, H, D, P, dtype, stream);
}
cp_status cp_striped_restore(const void* y, void* x, int64_t S, int32_t H, int32_t D, int32_t P,
                             int32_t dtype, void* stream) {
  return permute_common(kStripedRestore, y, x, S, H, D, P, dtype, stream);
}

// The lse [H, S] column map of a zigzag reorder or restore as one gather job, when
// every chunk is a whole number of 16-byte runs and both arrays are 16-byte aligned
// (otherwise the column kernel, which moves single floats, does it).
static bool lse_cols_job(int row_kind, const float* x, float* y, int64_t S, int32_t H, int32_t P,
                         GatherJob& j) {
  if (row_kind != kZigzagReorder && row_kind != kZigzagRestore) return false;
  if ((S / (2 * P)) % 4 != 0 || !aligned16(x) || !aligned16(y)) return false;
  j = GatherJob{row_kind == kZigzagReorder ? kZigzagReorderCols : kZigzagRestoreCols, x, y, (int64_t)H,
                S * 4, P};
  return true;
}

static bool disjoint(const void* a, const void* b, size_t nbytes) {
  const char* x = static_cast<const char*>(a);
  const char* y = static_cast<const char*>(b);
  return x + nbytes <= y || y + nbytes <= x;
}

// Checks shared by the batched ring permutes; returns the row map kind.
static cp_status ring_permute_check(int64_t S, int32_t D, int32_t dtype, int32_t P, int32_t reorder,
                                    int inverse, int* kind) {
  CP_REQUIRE(reorder == CP_REORDER_DUAL_CHUNK_SWAP || reorder == CP_REORDER_STRIPED, CP_ERR_INVALID_ARG,
             "reorder must be DUAL_CHUNK_SWAP or STRIPED");
  CP_REQUIRE(dtype == CP_F32 || dtype == CP_BF16, CP_ERR_DTYPE, "dtype must be CP_F32 or CP_BF16");
  CP_REQUIRE(S >= 0 && D >= 1 && P >= 1 && P <= 1024, CP_ERR_INVALID_ARG, "bad sizes");
  const bool zz = reorder == CP_REORDER_DUAL_CHUNK_SWAP;
  CP_REQUIRE(S % (zz ? 2 * P : P) == 0, CP_ERR_SHAPE, "S must divide into the layout's chunks");
  *kind = zz ? (inverse ? kZigzagRestore : kZigzagReorder) : (inverse ? kStripedRestore : kStripedReorder);
  return CP_OK;
}

cp_status cp_ring_reorder_qkv(const void* q, const void* k, const void* v, void* q_re, void* k_re,
                              void* v_re, int64_t S, int32_t Hq, int32_t Hkv, int32_t D, int32_t dtype,
                              int32_t P, int32_t reorder, void* stream) {
  int kind = 0;
  CP_TRY(ring_permute_check(S, D, dtype, P, reorder, 0, &kind));
  CP_REQUIRE(Hq >= 1 && Hkv >= 1, CP_ERR_INVALID_ARG, "Hq >= 1 and Hkv >= 1 required");
  const size_t qb = (size_t)Hq * D * dtype_size(dtype), kb = (size_t)Hkv * D * dtype_size(dtype);
  CP_REQUIRE(qb % 16 == 0 && kb % 16 == 0, CP_ERR_ALIGN, "H*D*sizeof(dtype) must be a multiple of 16 bytes");
  if (S == 0) return CP_OK;
  CP_CHECK_T(q, "q", false);
  CP_CHECK_T(k, "k", false);
  CP_CHECK_T(v, "v", false);
  CP_CHECK_T(q_re, "q_re", false);
  CP_CHECK_T(k_re, "k_re", false);
  CP_CHECK_T(v_re, "v_re", false);
  CP_REQUIRE(disjoint(q, q_re, S * qb) && disjoint(k, k_re, S * kb) && disjoint(v, v_re, S * kb),
             CP_ERR_INVALID_ARG, "each input and its reordered copy must not overlap");
  GatherJob jobs[3] = {{kind, q, q_re, S, (int64_t)qb, P}, {kind, k, k_re, S, (int64_t)kb, P},
                       {kind, v, v_re, S, (int64_t)kb, P}};
  return launch_row_gather_batch(jobs, 3, (cudaStream_t)stream);
}

cp_status cp_ring_restore(const void* o_re, const float* lse_re, void* out, float* lse, int64_t S,
                          int32_t Hq, int32_t D, int32_t dtype, int32_t P, int32_t reorder, void* stream) {
  int kind = 0;
  CP_TRY(ring_permute_check(S, D, dtype, P, reorder, 1, &kind));
  CP_REQUIRE(Hq >= 1, CP_ERR_INVALID_ARG, "Hq >= 1 required");
  CP_REQUIRE((uint64_t)S * Hq < (1ull << 32), CP_ERR_UNSUPPORTED, "S*Hq must be < 2^32");
  const size_t ob = (size_t)Hq * D * dtype_size(dtype);
  CP_REQUIRE(ob % 16 == 0, CP_ERR_ALIGN, "Hq*D*sizeof(dtype) must be a multiple of 16 bytes");
  CP_REQUIRE((lse_re == nullptr) == (lse == nullptr), CP_ERR_INVALID_ARG,
             "lse_re and lse must both be given or both be NULL");
  if (S == 0) return CP_OK;
  CP_CHECK_T(o_re, "o_re", false);
  CP_CHECK_T(out, "out", false);
  CP_REQUIRE(disjoint(o_re, out, S * ob), CP_ERR_INVALID_ARG, "o_re and out must not overlap");
  if (lse)
    CP_REQUIRE(disjoint(lse_re, lse, (size_t)S * Hq * 4), CP_ERR_INVALID_ARG, "lse_re and lse must not overlap");
  cudaStream_t st = (cudaStream_t)stream;
  GatherJob jobs[2] = {{kind, o_re, out, S, (int64_t)ob, P}, {}};
  int n = 1;
  if (lse && lse_cols_job(kind, lse_re, lse, S, Hq, P, jobs[1])) n = 2;
  CP_TRY(launch_row_gather_batch(jobs, n, st));
  if (lse && n == 1) CP_TRY(launch_lse_permute(kind, lse_re, lse, S, Hq, P, st));
  return CP_OK;
}

cp_status cp_lse_reorder(const float* x, float* y, int64_t S, int32_t H, int32_t P,
                         int32_t reorder, int32_t inverse, void* stream) {
  CP_REQUIRE(reorder == CP_REORDER_DUAL_CHUNK_SWAP || reorder == CP_REORDER_STRIPED,
             CP_ERR_INVALID_ARG, "reorder must be DUAL_CHUNK_SWAP or STRIPED");
  CP_REQUIRE(S >= 0 && H >= 1 && P >= 1 && P <= 1024, CP_ERR_INVALID_ARG, "bad sizes");
  CP_REQUIRE(S % (reorder == CP_REORDER_DUAL_CHUNK_SWAP ? 2 * P : P) == 0, CP_ERR_SHAPE,
             "S must divide into the layout's chunks");
  CP_REQUIRE((uint64_t)S * H < (1ull << 32), CP_ERR_UNSUPPORTED, "S*H must be < 2^32");
  if (S == 0) return CP_OK;
  CP_REQUIRE(x && y, CP_ERR_INVALID_ARG, "x and y must not be NULL");
  CP_REQUIRE(x + (size_t)S * H <= y || y + (size_t)S * H <= x, CP_ERR_INVALID_ARG,
             "x and y must not overlap");
  int kind = reorder == CP_REORDER_DUAL_CHUNK_SWAP ? (inverse ? kZigzagRestore : kZigzagReorder)
                                                   : (inverse ? kStripedRestore : kStripedReorder);
  return launch_lse_permute(kind, x, y, S, H, P, (cudaStream_t)stream);
}

cp_status cp_workspace_size(int32_t op, int64_t S, int32_t Hq, int32_t Hkv, int32_t D,
                            int32_t dtype, int32_t P, int32_t mode, size_t* bytes) {
  CP_REQUIRE(bytes != nullptr, CP_ERR_INVALID_ARG, "bytes must not be NULL");
  CP_REQUIRE(S >= 0 && Hq >= 1 && Hkv >= 1 && D >= 1 && P >= 1, CP_ERR_INVALID_ARG,
             "sizes must be positive");
  CP_REQUIRE(dtype == CP_F32 || dtype == CP_BF16, CP_ERR_DTYPE, "dtype must be CP_F32 or CP_BF16");
  switch (op) {
    case CP_OP_RING_FWD:
      CP_REQUIRE(mode == CP_RING_FUSED || mode == CP_RING_STEPWISE, CP_ERR_INVALID_ARG,
                 "mode must be a cp_ring_mode value");
      *bytes = ring_fwd_ws(S, Hq, Hkv, D, dtype, mode).total;
      return CP_OK;
    case CP_OP_RING_BWD:
      *bytes = ring_bwd_ws(S, Hq, Hkv, D, dtype).total;
      return CP_OK;
    case CP_OP_ULYSSES_FWD:
      *bytes = ulysses_ws(S, Hq, Hkv, D, dtype, P).total;
      return CP_OK;
    case CP_OP_ULYSSES_BWD:
      *bytes = ulysses_bwd_ws(S, Hq, Hkv, D, dtype, P).total;
      return CP_OK;
    case CP_OP_USP_FWD:  // independent of the degrees
      *bytes = usp_ws(S, Hq, Hkv, D, dtype).total;
      return CP_OK;
    case CP_OP_BLOCK_BWD:  // S is max(Sq, Sk) here
      *bytes = block_bwd_ws(S, S, Hq, Hkv, D).total;
      return CP_OK;
    case CP_OP_RING_FWD_REORDERED:
      CP_REQUIRE(mode == CP_RING_FUSED || mode == CP_RING_STEPWISE, CP_ERR_INVALID_ARG,
                 "mode must be a cp_ring_mode value");
      *bytes = ring_partials_ws(S, Hq, D, mode).total;
      return CP_OK;
    default:
      set_last_error("op must be a cp_op value");
      return CP_ERR_INVALID_ARG;
  }
}

cp_status cp_ring_attention(const void* q, const void* k, const void* v, int64_t S, int32_t Hq,
                            int32_t Hkv, int32_t D, int32_t dtype, int32_t P, int32_t reorder,
                            int32_t mode, const int32_t* cu_seqlens, int32_t n_docs, void* out,
                            float* lse, void* workspace, size_t ws_bytes, void* stream) {
  CP_REQUIRE(reorder >= CP_REORDER_CONTIGUOUS && reorder <= CP_REORDER_AUTO, CP_ERR_INVALID_ARG,
             "reorder must be a cp_reorder value");
  CP_REQUIRE(mode == CP_RING_FUSED || mode == CP_RING_STEPWISE, CP_ERR_INVALID_ARG,
             "mode must be a cp_ring_mode value");
  int32_t layout = resolve_layout(reorder, cu_seqlens);
  CP_TRY(check_ring_args(S, Hq, Hkv, D, dtype, P, layout, cu_seqlens, n_docs));
  if (S == 0) return CP_OK;
  RingFwdWs w = ring_fwd_ws(S, Hq, Hkv, D, dtype, mode);
  CP_REQUIRE(workspace && ws_bytes >= w.total, CP_ERR_WORKSPACE, "workspace too small for ring fwd");
  CP_CHECK_T(workspace, "workspace", false);
  CP_CHECK_T(q, "q", false);
  CP_CHECK_T(k, "k", false);
  CP_CHECK_T(v, "v", false);
  CP_CHECK_T(out, "out", false);
  CP_CHECK_T(lse, "lse", false);
  cudaStream_t st = (cudaStream_t)stream;
  const size_t es = dtype_size(dtype);
  void* q_re = ws_at(workspace, w.q);
  void* k_re = ws_at(workspace, w.k);
  void* v_re = ws_at(workspace, w.v);
  void* o_re = ws_at(workspace, w.o);
  float* lse_re = reinterpret_cast<float*>(ws_at(workspace, w.lse));
  const int fwd_kind = layout == CP_REORDER_DUAL_CHUNK_SWAP ? kZigzagReorder : kStripedReorder;
  const int back_kind = layout == CP_REORDER_DUAL_CHUNK_SWAP ? kZigzagRestore : kStripedRestore;
  // Contiguous layout: rank r already holds rows [rC, (r+1)C) in place.
  const bool moved = layout != CP_REORDER_CONTIGUOUS;
  // Zigzag with the fused ring: the attention writes out and lse in sequence order
  // (each rank's chunks are runs of consecutive positions), so no restore pass.
  const bool fused_restore = layout == CP_REORDER_DUAL_CHUNK_SWAP && mode == CP_RING_FUSED;
  if (fused_restore) {
    o_re = out;
    lse_re = lse;
  }
  if (moved) {
    GatherJob jobs[3] = {{fwd_kind, q, q_re, S, (int64_t)Hq * D * (int64_t)es, P},
                         {fwd_kind, k, k_re, S, (int64_t)Hkv * D * (int64_t)es, P},
                         {fwd_kind, v, v_re, S, (int64_t)Hkv * D * (int64_t)es, P}};
    CP_TRY(launch_row_gather_batch(jobs, 3, st));
  } else {
    q_re = const_cast<void*>(q);
    k_re = const_cast<void*>(k);
    v_re = const_cast<void*>(v);
    o_re = out;
    lse_re = lse;
  }
  CP_TRY(ring_core(q_re, k_re, v_re, o_re, lse_re, S, Hq, Hkv, D, dtype, P, layout, mode,
                   cu_seqlens, n_docs, ws_at(workspace, w.partials), w.pw, st, fused_restore));
  if (moved && !fused_restore) {
    GatherJob jobs[2] = {{back_kind, o_re, out, S, (int64_t)Hq * D * (int64_t)es, P}, {}};
    const int n = lse_cols_job(back_kind, lse_re, lse, S, Hq, P, jobs[1]) ? 2 : 1;
    CP_TRY(launch_row_gather_batch(jobs, n, st));
    if (n == 1) CP_TRY(launch_lse_permute(back_kind, lse_re, lse, S, Hq, P, st));
  }
  return CP_OK;
}

cp_status cp_ring_attention_reordered(const void* q, const void* k, const void* v, int64_t S,
                                      int32_t Hq, int32_t Hkv, int32_t D, int32_t dtype, int32_t P,
                                      int32_t reorder, int32_t mode, const int32_t* cu_seqlens,
                                      int32_t n_docs, void* out, float* lse, void* workspace,
                                      size_t ws_bytes, void* stream) {
  CP_REQUIRE(reorder >= CP_REORDER_CONTIGUOUS && reorder <= CP_REORDER_AUTO, CP_ERR_INVALID_ARG,
             "reorder must be a cp_reorder value");
  CP_REQUIRE(mode == CP_RING_FUSED || mode == CP_RING_STEPWISE, CP_ERR_INVALID_ARG,
             "mode must be a cp_ring_mode value");
  int32_t layout = resolve_layout(reorder, cu_seqlens);
  CP_TRY(check_ring_args(S, Hq, Hkv, D, dtype, P, layout, cu_seqlens, n_docs));
  if (S == 0) return CP_OK;
  RingPartialsWs w = ring_partials_ws(S, Hq, D, mode);
  if (w.total > 0) {
    CP_REQUIRE(workspace && ws_bytes >= w.total, CP_ERR_WORKSPACE,
               "workspace too small for the stepwise ring");
    CP_CHECK_T(workspace, "workspace", false);
  }
  CP_CHECK_T(q, "q", false);
  CP_CHECK_T(k, "k", false);
  CP_CHECK_T(v, "v", false);
  CP_CHECK_T(out, "out", false);
  CP_CHECK_T(lse, "lse", false);
  return ring_core(q, k, v, out, lse, S, Hq, Hkv, D, dtype, P, layout, mode, cu_seqlens, n_docs,
                   workspace, w, (cudaStream_t)stream);
}

cp_status cp_ring_attention_reordered_to_seq(const void* q, const void* k, const void* v, int64_t S,
                                             int32_t Hq, int32_t Hkv, int32_t D, int32_t dtype,
                                             int32_t P, int32_t reorder, const int32_t* cu_seqlens,
                                             int32_t n_docs, void* out, float* lse, void* stream) {
  CP_REQUIRE(reorder >= CP_REORDER_CONTIGUOUS && reorder <= CP_REORDER_AUTO, CP_ERR_INVALID_ARG,
             "reorder must be a cp_reorder value");
  int32_t layout = resolve_layout(reorder, cu_seqlens);
  CP_REQUIRE(layout != CP_REORDER_STRIPED, CP_ERR_UNSUPPORTED,
             "sequence-order output needs runs of consecutive positions (zigzag or contiguous)");
  CP_TRY(check_ring_args(S, Hq, Hkv, D, dtype, P, layout, cu_seqlens, n_docs));
  if (S == 0) return CP_OK;
  CP_CHECK_T(q, "q", false);
  CP_CHECK_T(k, "k", false);
  CP_CHECK_T(v, "v", false);
  CP_CHECK_T(out, "out", false);
  CP_CHECK_T(lse, "lse", false);
  RingPartialsWs w = ring_partials_ws(S, Hq, D, CP_RING_FUSED);
  return ring_core(q, k, v, out, lse, S, Hq, Hkv, D, dtype, P, layout, CP_RING_FUSED, cu_seqlens, n_docs,
                   nullptr, w, (cudaStream_t)stream, true);
}

cp_status cp_ring_attention_bwd(const void* q, const void* k, const void* v, const void* out,
                                const float* lse, const void* dout, int64_t S, int32_t Hq,
                                int32_t Hkv, int32_t D, int32_t dtype, int32_t P, int32_t reorder,
                                const int32_t* cu_seqlens, int32_t n_docs, void* dq, void* dk,
                                void* dv, void* workspace, size_t ws_bytes, void* stream) {
  CP_REQUIRE(reorder >= CP_REORDER_CONTIGUOUS && reorder <= CP_REORDER_AUTO, CP_ERR_INVALID_ARG,
             "reorder must be a cp_reorder value");
  int32_t layout = resolve_layout(reorder, cu_seqlens);
  CP_TRY(check_ring_args(S, Hq, Hkv, D, dtype, P, layout, cu_seqlens, n_docs));
  if (S == 0) return CP_OK;
  RingBwdWs w = ring_bwd_ws(S, Hq, Hkv, D, dtype);
  CP_REQUIRE(workspace && ws_bytes >= w.total, CP_ERR_WORKSPACE, "workspace too small for ring bwd");
  CP_CHECK_T(workspace, "workspace", false);
  CP_CHECK_T(q, "q", false);
  CP_CHECK_T(k, "k", false);
  CP_CHECK_T(v, "v", false);
  CP_CHECK_T(out, "out", false);
  CP_CHECK_T(dout, "dout", false);
  CP_CHECK_T(dq, "dq", false);
  CP_CHECK_T(dk, "dk", false);
  CP_CHECK_T(dv, "dv", false);
  CP_REQUIRE(lse != nullptr, CP_ERR_INVALID_ARG, "lse must not be NULL");
  cudaStream_t st = (cudaStream_t)stream;
  const size_t es = dtype_size(dtype);
  const int is_bf16 = dtype == CP_BF16;
  const bool moved = layout != CP_REORDER_CONTIGUOUS;
  const int fwd_kind = layout == CP_REORDER_DUAL_CHUNK_SWAP ? kZigzagReorder : kStripedReorder;
  const int back_kind = layout == CP_REORDER_DUAL_CHUNK_SWAP ? kZigzagRestore : kStripedRestore;
  const void *q_re = q, *k_re = k, *v_re = v, *o_re = out, *do_re = dout;
  const float* lse_re = lse;
  if (moved) {
    void* qw = ws_at(workspace, w.q);
    void* kw = ws_at(workspace, w.k);
    void* vw = ws_at(workspace, w.v);
    void* ow = ws_at(workspace, w.o);
    void* dw = ws_at(workspace, w.dout);
    float* lw = reinterpret_cast<float*>(ws_at(workspace, w.lse));
    const int64_t qb = (int64_t)Hq * D * (int64_t)es, kb = (int64_t)Hkv * D * (int64_t)es;
    GatherJob jobs[6] = {{fwd_kind, q, qw, S, qb, P},   {fwd_kind, k, kw, S, kb, P},
                         {fwd_kind, v, vw, S, kb, P},   {fwd_kind, out, ow, S, qb, P},
                         {fwd_kind, dout, dw, S, qb, P}, {}};
    const int n = lse_cols_job(fwd_kind, lse, lw, S, Hq, P, jobs[5]) ? 6 : 5;
    CP_TRY(launch_row_gather_batch(jobs, n, st));
    if (n == 5) CP_TRY(launch_lse_permute(fwd_kind, lse, lw, S, Hq, P, st));
    q_re = qw; k_re = kw; v_re = vw; o_re = ow; do_re = dw; lse_re = lw;
  }
  float* delta = reinterpret_cast<float*>(ws_at(workspace, w.delta));
  float* dq_acc = reinterpret_cast<float*>(ws_at(workspace, w.dq));
  float* dk_acc = reinterpret_cast<float*>(ws_at(workspace, w.dk));
  float* dv_acc = reinterpret_cast<float*>(ws_at(workspace, w.dv));
  // The tensor-core kernels write every gradient row once, in bf16: no zeroing, no cast.
  // Reordered: into the (then unused) fp32 accumulator space, since the dQ kernel still
  // reads the staged k/v after the dK/dV kernel is done.  In place: into the outputs,
  // if they share no bytes with what the kernels read.
  const size_t qbytes = (size_t)S * Hq * D * es, kbytes = (size_t)S * Hkv * D * es;
  const void* outs[3] = {dq, dk, dv};
  const size_t ob[3] = {qbytes, kbytes, kbytes};
  const void* ins[5] = {q, k, v, dout, lse};
  const size_t ib[5] = {qbytes, kbytes, kbytes, qbytes, (size_t)S * Hq * 4};
  const bool direct = bwd_writes_bf16(dtype, D) && (moved || grads_apart(outs, ob, 3, ins, ib, 5));
  if (!direct) CP_TRY(launch_zero(dq_acc, (size_t)S * Hq * D * 4, st));
  CP_TRY(launch_bwd_preprocess(o_re, do_re, delta, S, Hq, D, (int32_t)S, is_bf16, st));
  // where the gradients land in rank order (then restored when the layout moved)
  void* dq_c = !moved ? dq : direct ? static_cast<void*>(dq_acc) : ws_at(workspace, w.q);
  void* dk_c = !moved ? dk : direct ? static_cast<void*>(dk_acc) : ws_at(workspace, w.k);
  void* dv_c = !moved ? dv : direct ? static_cast<void*>(dv_acc) : ws_at(workspace, w.v);
  Schedule* s = new Schedule;
  build_ring_bwd_schedule(*s, S, P, layout, 1);
  BwdArgs a;
  memset(&a, 0, sizeof(a));
  a.q = q_re; a.k = k_re; a.v = v_re; a.dout = do_re; a.lse = lse_re; a.delta = delta;
  a.dq_acc = dq_acc; a.dk_acc = dk_acc; a.dv_acc = dv_acc;
  a.q_ld = (int64_t)Hq * D; a.k_ld = (int64_t)Hkv * D;
  a.Hq = Hq; a.Hkv = Hkv; a.D = D; a.lse_ld = (int32_t)S;
  a.scale = 1.0f / sqrtf((float)D);
  a.scale_log2 = a.scale * 1.4426950408889634f;
  a.causal = 1; a.cu_seqlens = cu_seqlens; a.n_docs = cu_seqlens ? n_docs : 0;
  a.err = device_error_word();
  if (direct) {
    a.dq_out = dq_c; a.dk_out = dk_c; a.dv_out = dv_c;
  }
  cp_status stt = launch_bwd(a, *s, dtype, S, S, st);
  delete s;
  CP_TRY(stt);
  if (!direct) {
    CP_TRY(launch_cast_out(dq_acc, dq_c, S * Hq * D, is_bf16, st));
    CP_TRY(launch_cast_out(dk_acc, dk_c, S * Hkv * D, is_bf16, st));
    CP_TRY(launch_cast_out(dv_acc, dv_c, S * Hkv * D, is_bf16, st));
  }
  if (moved) {  // back to sequence order
    GatherJob jobs[3] = {{back_kind, dq_c, dq, S, (int64_t)Hq * D * (int64_t)es, P},
                         {back_kind, dk_c, dk, S, (int64_t)Hkv * D * (int64_t)es, P},
                         {back_kind, dv_c, dv, S, (int64_t)Hkv * D * (int64_t)es, P}};
    CP_TRY(launch_row_gather_batch(jobs, 3, st));
  }
  return CP_OK;
}

cp_status cp_ulysses_attention(const void* q, const void* k, const void* v, int64_t S, int32_t Hq,
                               int32_t Hkv, int32_t D, int32_t dtype, int32_t P,
                               const int32_t* cu_seqlens, int32_t n_docs, int32_t window, void* out,
                               float* lse, void* workspace, size_t ws_bytes, void* stream) {
  CP_REQUIRE(window >= 0, CP_ERR_INVALID_ARG, "window must be >= 0");
  CP_TRY(check_common(Hq, Hkv, D, dtype));
  CP_REQUIRE(P >= 1 && P <= 64, CP_ERR_INVALID_ARG, "P must be in [1, 64]");
  CP_REQUIRE(S >= 0, CP_ERR_INVALID_ARG, "S must be >= 0");
  CP_REQUIRE(Hq % P == 0, CP_ERR_SHAPE, "Ulysses needs Hq % P == 0");
  CP_REQUIRE(ulysses_kv_replicas(Hkv, P) > 0, CP_ERR_SHAPE,
             "Ulysses needs Hkv % P == 0, or P % Hkv == 0 (key/value heads replicated P/Hkv times)");
  CP_REQUIRE(S % P == 0, CP_ERR_SHAPE, "Ulysses needs S % P == 0");
  CP_REQUIRE(S * (int64_t)Hq < (int64_t)INT32_MAX && S * (int64_t)P < (int64_t)INT32_MAX,
             CP_ERR_UNSUPPORTED, "S*Hq and S*P must be < 2^31");
  CP_REQUIRE(!cu_seqlens || n_docs >= 1, CP_ERR_INVALID_ARG, "n_docs must be >= 1 with cu_seqlens");
  const size_t es = dtype_size(dtype);
  const int32_t R = ulysses_kv_replicas(Hkv, P);
  CP_REQUIRE(((size_t)(Hkv * R / P) * D * es) % 16 == 0, CP_ERR_ALIGN,
             "(Hkv/P)*D*sizeof(dtype) must be a multiple of 16 bytes");
  if (S == 0) return CP_OK;
  UlyssesWs w = ulysses_ws(S, Hq, Hkv, D, dtype, P);
  CP_REQUIRE(workspace && ws_bytes >= w.total, CP_ERR_WORKSPACE, "workspace too small for Ulysses");
  CP_CHECK_T(workspace, "workspace", false);
  CP_CHECK_T(q, "q", false);
  CP_CHECK_T(k, "k", false);
  CP_CHECK_T(v, "v", false);
  CP_CHECK_T(out, "out", false);
  CP_CHECK_T(lse, "lse", false);
  cudaStream_t st = (cudaStream_t)stream;
  void* qh = ws_at(workspace, w.q);
  void* kh = ws_at(workspace, w.k);
  void* vh = ws_at(workspace, w.v);
  void* oh = ws_at(workspace, w.o);
  if (R == 1) {
    GatherJob jobs[3] = {{kSeq2Head, q, qh, S, (int64_t)Hq * D * (int64_t)es, P},
                         {kSeq2Head, k, kh, S, (int64_t)Hkv * D * (int64_t)es, P},
                         {kSeq2Head, v, vh, S, (int64_t)Hkv * D * (int64_t)es, P}};
    CP_TRY(launch_row_gather_batch(jobs, 3, st));
  } else {  // rank p gets a copy of key/value head p / R
    CP_TRY(launch_row_gather(kSeq2Head, q, qh, S, (int64_t)Hq * D * es, P, Hq, st));
    CP_TRY(launch_kv_replicate(k, kh, S, Hkv, (int64_t)D * es, P, st));
    CP_TRY(launch_kv_replicate(v, vh, S, Hkv, (int64_t)D * es, P, st));
  }
  const int32_t Hqp = Hq / P, Hkvp = Hkv * R / P;
  Schedule* s = new Schedule;
  s->n_groups = 0;
  s->n_segs = 0;
  // Rank p's attention writes its query heads straight into out's sequence layout
  // (rows = positions, head columns p*Hqp ..): the head2seq of out is done by the
  // attention's own output writes, as lse's is.
  for (int p = 0; p < P; ++p) {
    add_group(*s, Piece{(int32_t)(p * S), (int32_t)S, 0, 1});
    s->g[p].lse_col0 = 0;
    s->g[p].lse_head0 = p * Hqp;
    s->g[p].o_row0 = 0;
    s->g[p].o_head0 = p * Hqp;
    add_seg(*s, Piece{(int32_t)(p * S), (int32_t)S, 0, 1});
  }
  (void)oh;
  AttnArgs a = make_fwd_args(qh, kh, vh, out, lse, Hqp, Hkvp, D, S, 1, cu_seqlens, n_docs,
                             1.0f / sqrtf((float)D), 0);
  a.o_ld = (int64_t)Hq * D;
  a.window = window;
  cp_status stt = launch_fwd(a, *s, dtype, (int64_t)P * S, (int64_t)P * S, st);
  delete s;
  return stt;
}

cp_status cp_usp_attention(const void* q, const void* k, const void* v, int64_t S, int32_t Hq,
                           int32_t Hkv, int32_t D, int32_t dtype, int32_t P_ulysses, int32_t P_ring,
                           int32_t reorder, const int32_t* cu_seqlens, int32_t n_docs, void* out,
                           float* lse, void* workspace, size_t ws_bytes, void* stream) {
  CP_REQUIRE(reorder >= CP_REORDER_CONTIGUOUS && reorder <= CP_REORDER_AUTO, CP_ERR_INVALID_ARG,
             "reorder must be a cp_reorder value");
  CP_REQUIRE(P_ulysses >= 1 && P_ring >= 1 && P_ulysses * P_ring <= 64, CP_ERR_INVALID_ARG,
             "P_ulysses, P_ring >= 1 and P_ulysses * P_ring <= 64 required");
  const int32_t layout = resolve_layout(reorder, cu_seqlens);
  CP_TRY(check_ring_args(S, Hq, Hkv, D, dtype, P_ring, layout, cu_seqlens, n_docs));
  CP_REQUIRE(Hq % P_ulysses == 0 && Hkv % P_ulysses == 0, CP_ERR_SHAPE,
             "USP needs Hq % P_ulysses == 0 and Hkv % P_ulysses == 0");
  CP_REQUIRE((S / P_ring) % P_ulysses == 0, CP_ERR_SHAPE,
             "USP needs each ring group's tokens (S / P_ring) to split evenly over P_ulysses ranks");
  const size_t es = dtype_size(dtype);
  const int32_t Hqp = Hq / P_ulysses, Hkvp = Hkv / P_ulysses;
  CP_REQUIRE(((size_t)Hkvp * D * es) % 16 == 0, CP_ERR_ALIGN,
             "(Hkv/P_ulysses)*D*sizeof(dtype) must be a multiple of 16 bytes");
  if (S == 0) return CP_OK;
  UspWs w = usp_ws(S, Hq, Hkv, D, dtype);
  CP_REQUIRE(workspace && ws_bytes >= w.total, CP_ERR_WORKSPACE, "workspace too small for USP");
  CP_CHECK_T(workspace, "workspace", false);
  CP_CHECK_T(q, "q", false);
  CP_CHECK_T(k, "k", false);
  CP_CHECK_T(v, "v", false);
  CP_CHECK_T(out, "out", false);
  CP_CHECK_T(lse, "lse", false);
  cudaStream_t st = (cudaStream_t)stream;
  const bool moved = layout != CP_REORDER_CONTIGUOUS;
  const int fwd_kind = layout == CP_REORDER_DUAL_CHUNK_SWAP ? kZigzagReorder : kStripedReorder;
  const int back_kind = layout == CP_REORDER_DUAL_CHUNK_SWAP ? kZigzagRestore : kStripedRestore;
  const void *q_re = q, *k_re = k, *v_re = v;
  if (moved) {  // the ring's partition across groups
    GatherJob jobs[3] = {{fwd_kind, q, ws_at(workspace, w.q_re), S, (int64_t)Hq * D * (int64_t)es, P_ring},
                         {fwd_kind, k, ws_at(workspace, w.k_re), S, (int64_t)Hkv * D * (int64_t)es, P_ring},
                         {fwd_kind, v, ws_at(workspace, w.v_re), S, (int64_t)Hkv * D * (int64_t)es, P_ring}};
    CP_TRY(launch_row_gather_batch(jobs, 3, st));
    q_re = ws_at(workspace, w.q_re);
    k_re = ws_at(workspace, w.k_re);
    v_re = ws_at(workspace, w.v_re);
  }
  // the exchange inside each group: head share u of every token (the ring order is kept)
  void* qh = ws_at(workspace, w.qh);
  void* kh = ws_at(workspace, w.kh);
  void* vh = ws_at(workspace, w.vh);
  {
    GatherJob jobs[3] = {{kSeq2Head, q_re, qh, S, (int64_t)Hq * D * (int64_t)es, P_ulysses},
                         {kSeq2Head, k_re, kh, S, (int64_t)Hkv * D * (int64_t)es, P_ulysses},
                         {kSeq2Head, v_re, vh, S, (int64_t)Hkv * D * (int64_t)es, P_ulysses}};
    CP_TRY(launch_row_gather_batch(jobs, 3, st));
  }
  // the fused ring across groups, once per head share, in one launch
  Schedule* ring = new Schedule;
  Schedule* s = new Schedule;
  // Zigzag and contiguous ring pieces are runs of consecutive positions: the attention
  // then writes out and lse at their final places (sequence rows, head share u's
  // columns), so neither the head2seq nor the restore runs afterwards.
  const bool direct = layout != CP_REORDER_STRIPED;
  build_ring_schedule(*ring, S, P_ring, layout, -1, 1, direct);
  if ((int64_t)ring->n_groups * P_ulysses > kMaxGroups || (int64_t)ring->n_segs * P_ulysses > kMaxSegs) {
    delete ring;
    delete s;
    set_last_error("USP schedule too large (ring groups x P_ulysses exceeds the schedule capacity)");
    return CP_ERR_UNSUPPORTED;
  }
  s->n_groups = 0;
  s->n_segs = 0;
  for (int u = 0; u < P_ulysses; ++u)
    for (int gi = 0; gi < ring->n_groups; ++gi) {
      const QGroup& rg = ring->g[gi];
      QGroup& g = s->g[s->n_groups++];
      g = rg;
      g.q_row0 = rg.q_row0 + u * (int32_t)S;
      g.o_row0 = direct ? rg.o_row0 : rg.o_row0 + u * (int32_t)S;
      g.o_head0 = direct ? u * Hqp : 0;
      g.lse_head0 = rg.lse_head0 + u * Hqp;  // lse columns: sequence order when direct, else ring order
      g.seg_begin = s->n_segs;
      for (int si = 0; si < rg.seg_count; ++si) {
        KSeg sg = ring->s[rg.seg_begin + si];
        sg.k_row0 += u * (int32_t)S;
        s->s[s->n_segs++] = sg;
      }
    }
  sort_groups_by_work(*s);
  delete ring;
  // outputs: head-major into the ring-ordered q buffer (free after seq2head, or never used
  // when the layout is contiguous), lse in ring order
  void* oh = ws_at(workspace, w.q_re);
  float* lse_re = (moved && !direct) ? reinterpret_cast<float*>(ws_at(workspace, w.lse)) : lse;
  AttnArgs a = make_fwd_args(qh, kh, vh, direct ? out : oh, lse_re, Hqp, Hkvp, D, S, 1, cu_seqlens, n_docs,
                             1.0f / sqrtf((float)D), 0);
  if (direct) a.o_ld = (int64_t)Hq * D;
  cp_status stt = launch_fwd(a, *s, dtype, (int64_t)P_ulysses * S, (int64_t)P_ulysses * S, st);
  delete s;
  CP_TRY(stt);
  if (direct) return CP_OK;
  if (moved) {
    void* o_re = ws_at(workspace, w.qh);  // free after the attention
    CP_TRY(launch_row_gather(kHead2Seq, oh, o_re, S, (int64_t)Hq * D * es, P_ulysses, Hq, st));
    CP_TRY(launch_row_gather(back_kind, o_re, out, S, (int64_t)Hq * D * es, P_ring, Hq, st));
    CP_TRY(launch_lse_permute(back_kind, lse_re, lse, S, Hq, P_ring, st));
  } else {
    CP_TRY(launch_row_gather(kHead2Seq, oh, out, S, (int64_t)Hq * D * es, P_ulysses, Hq, st));
  }
  return CP_OK;
}

cp_status cp_ulysses_attention_bwd(const void* q, const void* k, const void* v, const void* out,
                                   const float* lse, const void* dout, int64_t S, int32_t Hq,
                                   int32_t Hkv, int32_t D, int32_t dtype, int32_t P,
                                   const int32_t* cu_seqlens, int32_t n_docs, int32_t window, void* dq,
                                   void* dk, void* dv, void* workspace, size_t ws_bytes, void* stream) {
  CP_TRY(check_common(Hq, Hkv, D, dtype));
  CP_REQUIRE(window >= 0, CP_ERR_INVALID_ARG, "window must be >= 0");
  CP_REQUIRE(P >= 1 && P <= 64, CP_ERR_INVALID_ARG, "P must be in [1, 64]");
  CP_REQUIRE(S >= 0, CP_ERR_INVALID_ARG, "S must be >= 0");
  CP_REQUIRE(Hq % P == 0, CP_ERR_SHAPE, "Ulysses needs Hq % P == 0");
  CP_REQUIRE(ulysses_kv_replicas(Hkv, P) > 0, CP_ERR_SHAPE,
             "Ulysses needs Hkv % P == 0, or P % Hkv == 0 (key/value heads replicated P/Hkv times)");
  CP_REQUIRE(S % P == 0, CP_ERR_SHAPE, "Ulysses needs S % P == 0");
  CP_REQUIRE(S * (int64_t)Hq < (int64_t)INT32_MAX && S * (int64_t)P < (int64_t)INT32_MAX,
             CP_ERR_UNSUPPORTED, "S*Hq and S*P must be < 2^31");
  CP_REQUIRE(!cu_seqlens || n_docs >= 1, CP_ERR_INVALID_ARG, "n_docs must be >= 1 with cu_seqlens");
  const size_t es = dtype_size(dtype);
  const int32_t R = ulysses_kv_replicas(Hkv, P);
  const int32_t Hqp = Hq / P, Hkvp = Hkv * R / P;
  CP_REQUIRE(((size_t)Hkvp * D * es) % 16 == 0, CP_ERR_ALIGN,
             "(Hkv/P)*D*sizeof(dtype) must be a multiple of 16 bytes");
  if (S == 0) return CP_OK;
  UlyssesBwdWs w = ulysses_bwd_ws(S, Hq, Hkv, D, dtype, P);
  CP_REQUIRE(workspace && ws_bytes >= w.total, CP_ERR_WORKSPACE, "workspace too small for Ulysses bwd");
  CP_CHECK_T(workspace, "workspace", false);
  CP_CHECK_T(q, "q", false);
  CP_CHECK_T(k, "k", false);
  CP_CHECK_T(v, "v", false);
  CP_CHECK_T(out, "out", false);
  CP_CHECK_T(dout, "dout", false);
  CP_CHECK_T(dq, "dq", false);
  CP_CHECK_T(dk, "dk", false);
  CP_CHECK_T(dv, "dv", false);
  CP_REQUIRE(lse != nullptr, CP_ERR_INVALID_ARG, "lse must not be NULL");
  cudaStream_t st = (cudaStream_t)stream;
  const int is_bf16 = dtype == CP_BF16;
  void* qh = ws_at(workspace, w.q);
  void* kh = ws_at(workspace, w.k);
  void* vh = ws_at(workspace, w.v);
  void* doh = ws_at(workspace, w.dout);
  float* delta = reinterpret_cast<float*>(ws_at(workspace, w.delta));
  float* lse_h = reinterpret_cast<float*>(ws_at(workspace, w.lse_h));
  float* delta_h = reinterpret_cast<float*>(ws_at(workspace, w.delta_h));
  float* dq_acc = reinterpret_cast<float*>(ws_at(workspace, w.dq));
  float* dk_acc = reinterpret_cast<float*>(ws_at(workspace, w.dk));
  float* dv_acc = reinterpret_cast<float*>(ws_at(workspace, w.dv));
  // head_to_seq is the backward of seq_to_head: the gradients take the same
  // exchange as the outputs.  Delta = rowsum(dO o O) on the sequence layout
  // (same [Hq, S] order as lse), then both go to the head-major row order.
  {
    GatherJob jobs[4] = {{kSeq2Head, q, qh, S, (int64_t)Hq * D * (int64_t)es, P},
                         {kSeq2Head, dout, doh, S, (int64_t)Hq * D * (int64_t)es, P},
                         {kSeq2Head, k, kh, S, (int64_t)Hkv * D * (int64_t)es, P},
                         {kSeq2Head, v, vh, S, (int64_t)Hkv * D * (int64_t)es, P}};
    CP_TRY(launch_row_gather_batch(jobs, R == 1 ? 4 : 2, st));
  }
  if (R > 1) {
    CP_TRY(launch_kv_replicate(k, kh, S, Hkv, (int64_t)D * es, P, st));
    CP_TRY(launch_kv_replicate(v, vh, S, Hkv, (int64_t)D * es, P, st));
  }
  CP_TRY(launch_bwd_preprocess(out, dout, delta, S, Hq, D, (int32_t)S, is_bf16, st));
  CP_TRY(launch_lse_to_heads(lse, lse_h, S, Hq, P, st));
  CP_TRY(launch_lse_to_heads(delta, delta_h, S, Hq, P, st));
  CP_TRY(launch_zero(dq_acc, (size_t)S * Hq * D * 4, st));
  // P independent full-sequence problems: key-major schedule, rank p's keys see its queries
  Schedule* s = new Schedule;
  s->n_groups = 0;
  s->n_segs = 0;
  for (int p = 0; p < P; ++p) {
    add_group(*s, Piece{(int32_t)(p * S), (int32_t)S, 0, 1});
    add_seg(*s, Piece{(int32_t)(p * S), (int32_t)S, 0, 1});
  }
  BwdArgs a;
  memset(&a, 0, sizeof(a));
  a.q = qh; a.k = kh; a.v = vh; a.dout = doh; a.lse = lse_h; a.delta = delta_h;
  a.dq_acc = dq_acc; a.dk_acc = dk_acc; a.dv_acc = dv_acc;
  a.q_ld = (int64_t)Hqp * D; a.k_ld = (int64_t)Hkvp * D;
  a.Hq = Hqp; a.Hkv = Hkvp; a.D = D; a.lse_ld = (int32_t)(P * S);
  a.scale = 1.0f / sqrtf((float)D);
  a.scale_log2 = a.scale * 1.4426950408889634f;
  a.causal = 1; a.cu_seqlens = cu_seqlens; a.n_docs = cu_seqlens ? n_docs : 0;
  a.window = window;
  a.err = device_error_word();
  cp_status stt = launch_bwd(a, *s, dtype, (int64_t)P * S, (int64_t)P * S, st);
  delete s;
  CP_TRY(stt);
  // back to [S, H, D] in the input dtype; replicated key/value heads sum their copies
  CP_TRY(launch_heads_to_seq_sum(dq_acc, dq, S, Hq, 1, P, Hqp, D, is_bf16, st));
  CP_TRY(launch_heads_to_seq_sum(dk_acc, dk, S, Hkv, R, P, Hkvp, D, is_bf16, st));
  CP_TRY(launch_heads_to_seq_sum(dv_acc, dv, S, Hkv, R, P, Hkvp, D, is_bf16, st));
  return CP_OK;
}

cp_status cp_check_device_status(void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  cp_status s = cuda_check(cudaStreamSynchronize(st), "cudaStreamSynchronize");
  if (s != CP_OK) return s;
  int32_t* ew = device_error_word();
  if (!ew) {
    set_last_error("device error word unavailable");
    return CP_ERR_CUDA;
  }
  int32_t code = 0;
  s = cuda_check(cudaMemcpy(&code, ew, sizeof(code), cudaMemcpyDeviceToHost), "read error word");
  if (s != CP_OK) return s;
  if (code != 0) {
    int32_t zero = 0;
    (void)cudaMemcpy(ew, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (code == kDevIndex) {
      set_last_error("a kernel's index check failed and skipped the access (debug build)");
      return CP_ERR_DEVICE_INDEX;
    }
    set_last_error("a kernel gave up on a bounded wait (device error code " +
                   std::to_string(code) + ")");
    return CP_ERR_DEVICE_TIMEOUT;
  }
  return CP_OK;
}

cp_status cp_debug_bounded_wait(int32_t timeout_us, void* stream) {
  CP_REQUIRE(timeout_us >= 1 && timeout_us <= 1000000, CP_ERR_INVALID_ARG,
             "timeout_us must be in [1, 1000000]");
  int32_t* ew = device_error_word();
  CP_REQUIRE(ew != nullptr, CP_ERR_CUDA, "device error word unavailable");
  return launch_bounded_wait_probe(timeout_us, ew, (cudaStream_t)stream);
}

}  // extern "C"
