// Internal declarations shared by the library's translation units.
//
// The attention kernels consume a "schedule": a list of query groups, each
// with the list of key/value segments it attends to, in the order the ring
// visits them.  One schedule describes every use of block attention in the
// library: a single block pair (one group, one segment), the P virtual ranks
// of the ring (a group per query chunk, segments in ring order), and the P
// virtual ranks of Ulysses (a group per rank over the permuted buffer).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "cp_attn.h"

namespace cpa {

constexpr int kMaxGroups = 64;
constexpr int kMaxSegs = 1024;
constexpr int kMaxOrder = 2048;  // (group, tile) pairs a launch order table can hold

// A run of query rows that share one affine position map.
struct QGroup {
  int32_t q_row0;      // first row in the q (and o) buffer
  int32_t nq;          // number of rows
  int32_t pos_off;     // global position of row 0
  int32_t pos_stride;  // position step between rows (>= 1)
  int32_t seg_begin;   // first segment index in Schedule::s
  int32_t seg_count;   // number of segments
  int32_t tile0;       // running count of query tiles before this group (set by the launcher)
  int32_t lse_col0;    // lse column of row 0
  int32_t lse_head0;   // lse head (row of the [H, cols] lse) of head 0
  int32_t o_row0;      // first output row
  int32_t o_head0;     // output head offset: head h of the group goes to out column (o_head0 + h) * D
  int32_t pad1;
};

// A run of key/value rows with one affine position map.
struct KSeg {
  int32_t k_row0;
  int32_t nk;
  int32_t pos_off;
  int32_t pos_stride;
};

struct Schedule {
  int32_t n_groups;
  int32_t n_segs;
  QGroup g[kMaxGroups];
  KSeg s[kMaxSegs];
  // Launch order of the (group, tile) pairs, heaviest first: entry = group << 20 | tile.
  // n_order = 0: groups in order, each group's tiles last to first.
  int32_t n_order;
  int32_t order[kMaxOrder];
};

// Everything else an attention launch needs (pointers, strides, mask).
struct AttnArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int64_t q_ld;  // elements between consecutive rows of q (Hq*D)
  int64_t k_ld;  // elements between consecutive rows of k and v (Hkv*D)
  int64_t o_ld;  // elements between consecutive rows of o
  int32_t Hq, Hkv, D;
  int32_t lse_ld;     // columns per lse head row
  float scale_log2;   // softmax scale * log2(e)
  float scale;        // softmax scale
  int32_t causal;
  const int32_t* cu_seqlens;  // device, n_docs+1, or nullptr
  int32_t n_docs;
  int32_t* err;       // device error word
  int32_t total_units;
  int32_t o_f32;      // output dtype: 1 fp32, 0 same as input
  int32_t o_tma;      // bf16 output written by TMA stores through the launch's O tensor map
  int32_t window;     // sliding window (causal only): pos_q - pos_k < window; 0 = none
  // Buffer extents, for the index checks of debug builds: rows of q (and o) and of
  // k / v, and floats in the lse array.
  int64_t q_rows, k_rows, lse_size;
  // Position-tiled striped buffers (perm_p > 0): q, k, v, o are [perm_p][perm_n][H*D]
  // (rank r's row i holds position i*perm_p + r) and the schedule's rows are
  // positions; a tile of 128 positions is 128/perm_p rows of every rank.
  int32_t perm_p, perm_n;
  // Forward launch order: units in blocks of head_block heads (whole key/value
  // heads), each block's heads fastest; total_units = (group, tile) pairs x Hq.
  int32_t head_block;
};

// Backward extras.
struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* dout;
  const float* lse;    // [Hq, lse_ld], natural log
  const float* delta;  // [Hq, lse_ld], rowsum(dout*out)
  float* dq_acc;       // [rows_q, Hq, D] fp32
  float* dk_acc;       // [rows_k, Hkv, D] fp32
  float* dv_acc;       // [rows_k, Hkv, D] fp32
  // bf16 outputs written directly by the tensor-core kernels (same layout as the
  // accumulators; every row is written once, so no zeroing or cast pass); NULL:
  // the fp32 accumulators above are written instead.
  void* dq_out;
  void* dk_out;
  void* dv_out;
  int64_t q_ld, k_ld;
  int32_t Hq, Hkv, D;
  int32_t lse_ld;
  float scale_log2, scale;
  int32_t causal;
  const int32_t* cu_seqlens;
  int32_t n_docs;
  int32_t* err;
  int32_t total_units;
  int32_t window;      // sliding window (causal only): pos_q - pos_k < window; 0 = none
  int32_t accumulate;  // fp32 outputs: add into the values already there (each row is still
                       // written by one CTA, so no atomics); 0 = overwrite
  // Buffer extents, for the index checks of debug builds: rows of q / dout / dq and
  // of k / v / dk / dv, and floats in the lse (and Delta) array.
  int64_t q_rows, k_rows, lse_size;
  // Launch orders (decode_unit_blocked): (group, tile) pairs of the key-major and the
  // query-major schedule, and heads per block of each launch.
  int32_t kv_pairs, q_pairs, kv_head_block, q_head_block;
};

// Device error codes written into the error word (first writer wins).
enum DeviceError : int32_t {
  kDevOk = 0,
  kDevTimeout = 1,
  kDevIndex = 2,  // debug builds: an index check failed (the access was skipped)
};

// ---------------------------------------------------------------- host side helpers (api.cu)
void set_last_error(const std::string& msg);
int32_t* device_error_word();  // device address of the error word for the current device
cp_status cuda_check(cudaError_t e, const char* what);

// Validates the sizes, dtype and mask of one (query block, key block) pair: the
// rules every block call shares (Hq % Hkv, D for the dtype, S*H < 2^31, strides,
// window, positions in int32, n_docs).  On success *m holds the mask to apply
// (the default causal mask when `mask` is NULL).
cp_status check_block_args(int64_t Sq, int64_t Sk, int32_t Hq, int32_t Hkv, int32_t D, int32_t dtype,
                           const cp_mask* mask, cp_mask* m);

// Gradient destinations of one block backward.  Typed form: dq/dk/dv in the input
// dtype are overwritten and dq_acc/dk_acc/dv_acc are fp32 scratch.  Accumulating
// form (typed == false): dq_acc/dk_acc/dv_acc are the caller's fp32 outputs,
// overwritten (accumulate == 0) or added to (accumulate != 0).
struct BlockBwdOut {
  bool typed;
  void* dq;
  void* dk;
  void* dv;
  float* dq_acc;
  float* dk_acc;
  float* dv_acc;
  int32_t accumulate;
};
// Runs the block backward of a validated call: Delta into `delta` ([Hq, Sq] fp32),
// the attention backward kernels, and the zero / cast passes the typed form needs.
cp_status block_bwd_run(const void* q, const void* k, const void* v, const void* out, const void* dout,
                        const float* lse, int64_t Sq, int64_t Sk, int32_t Hq, int32_t Hkv, int32_t D,
                        int32_t dtype, const cp_mask& m, float scale, const BlockBwdOut& o, float* delta,
                        cudaStream_t st);

// ---------------------------------------------------------------- launchers (one per .cu)
// movers.cu
cp_status launch_row_gather(int kind, const void* x, void* y, int64_t S, int64_t row_bytes,
                            int32_t P, int32_t H_for_ulysses, cudaStream_t st);

// One gather of a batch: S rows of row_bytes from x to y with the row map of `kind`
// (a GatherKind) over P ranks.  For the *Cols kinds S counts lse heads and
// row_bytes is one lse row (sequence length x 4).
struct GatherJob {
  int kind;
  const void* x;
  void* y;
  int64_t S;
  int64_t row_bytes;
  int32_t P;
};
constexpr int kMaxGatherBatch = 6;
// Runs 1..kMaxGatherBatch gathers in one launch.
cp_status launch_row_gather_batch(const GatherJob* jobs, int n, cudaStream_t st);
cp_status launch_lse_permute(int kind, const float* x, float* y, int64_t S, int32_t H, int32_t P,
                             cudaStream_t st);
// merge.cu
cp_status launch_lse_merge(const void* o1, const float* lse1, const void* o2, const float* lse2,
                           void* o, float* lse, int64_t Sq, int32_t H, int32_t D, int32_t o_f32,
                           cudaStream_t st);
// attn_simt.cu
cp_status launch_attn_fwd_simt(const AttnArgs& a, Schedule& s, int is_bf16, cudaStream_t st);
cp_status launch_attn_bwd_simt(const BwdArgs& a, Schedule& s, int is_bf16, cudaStream_t st);
cp_status launch_bwd_preprocess(const void* out, const void* dout, float* delta, int64_t rows,
                                int32_t H, int32_t D, int32_t lse_ld, int is_bf16, cudaStream_t st);
cp_status launch_cast_out(const float* src, void* dst, int64_t n, int is_bf16, cudaStream_t st);
cp_status launch_zero(void* p, size_t bytes, cudaStream_t st);
// movers.cu (Ulysses with replicated key/value heads, and the Ulysses backward)
cp_status launch_kv_replicate(const void* x, void* y, int64_t S, int32_t Hkv, int64_t head_bytes,
                              int32_t P, cudaStream_t st);
cp_status launch_lse_to_heads(const float* x, float* y, int64_t S, int32_t H, int32_t P,
                              cudaStream_t st);
cp_status launch_heads_to_seq_sum(const float* src, void* dst, int64_t S, int32_t Hd, int32_t R,
                                  int32_t P, int32_t Hp, int32_t D, int is_bf16, cudaStream_t st);
cp_status launch_bounded_wait_probe(int32_t timeout_us, int32_t* err, cudaStream_t st);
// attn_fwd_tc.cu
cp_status launch_attn_fwd_tc(const AttnArgs& a, Schedule& s, int64_t q_rows, int64_t k_rows,
                             cudaStream_t st);
// attn_bwd_tc.cu
cp_status launch_attn_bwd_tc(const BwdArgs& a, Schedule& s, int64_t q_rows, int64_t k_rows,
                             cudaStream_t st);

// Row-gather kinds.
enum GatherKind : int {
  kZigzagReorder = 0,
  kZigzagRestore = 1,
  kStripedReorder = 2,
  kStripedRestore = 3,
  kSeq2Head = 4,
  kHead2Seq = 5,
  kSeq2HeadRep = 6,  // Ulysses seq2head of key/value heads replicated P/Hkv times
  kZigzagReorderCols = 7,  // the zigzag maps on the columns of an lse [H, S] fp32 array,
  kZigzagRestoreCols = 8,  // as 16-byte runs (needs S/(2P) % 4 == 0)
};

// True when the backward runs on the tensor-core kernels (bf16, D = 64 or 128), which
// write bf16 gradients directly (BwdArgs::dq_out etc.).
bool bwd_writes_bf16(int32_t dtype, int32_t D);
// True when none of the n_out output ranges overlaps any of the n_in input ranges
// (NULL entries are skipped).
bool grads_apart(const void* const* outs, const size_t* out_bytes, int n_out, const void* const* ins,
                 const size_t* in_bytes, int n_in);

// Fills group tile prefix sums for a query tile height; returns total units (tiles x heads).
// Clears the launch order table.
int64_t schedule_units(Schedule& s, int tile_rows, int heads);

// Fills the launch order table (after schedule_units with the same tile_rows) so that
// the CTAs with the most visible tiles of the other side start first and the lightest
// fill the last wave (the backward kernels use it; the forward's own order measured as
// fast).  The weight counts tiles from positions alone (causal rule and
// sliding window); with documents, without the causal rule, or when the pairs do not
// fit the table, the order is left as schedule_units set it.  key_major: groups are
// key runs and segments query runs (the key-stationary backward).
void schedule_order(Schedule& s, int tile_rows, int other_tile, bool key_major, int causal,
                    int window, bool docs);

}  // namespace cpa

// ---------------------------------------------------------------- device helpers
namespace cpa {

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void record_device_error(int32_t* err, int32_t code) {
  if (err) atomicCAS(err, 0, code);
}

// Index checks of debug builds (compiled with -DCP_DEBUG): CP_DCHECK(cond, err) is
// true when cond holds; otherwise it records kDevIndex in the error word and is
// false, and the caller skips the access.  Release builds compile it to true.
__device__ __forceinline__ bool debug_check(bool ok, int32_t* err) {
  if (!ok) record_device_error(err, kDevIndex);
  return ok;
}
#ifdef CP_DEBUG
#define CP_DCHECK(cond, err) (::cpa::debug_check((cond), (err)))
#else
#define CP_DCHECK(cond, err) (true)
#endif

__device__ __forceinline__ float bf16_to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ float load_as_f32(const T* p);
template <>
__device__ __forceinline__ float load_as_f32<float>(const float* p) {
  return *p;
}
template <>
__device__ __forceinline__ float load_as_f32<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

template <typename T>
__device__ __forceinline__ void store_from_f32(T* p, float x);
template <>
__device__ __forceinline__ void store_from_f32<float>(float* p, float x) {
  *p = x;
}
template <>
__device__ __forceinline__ void store_from_f32<__nv_bfloat16>(__nv_bfloat16* p, float x) {
  *p = __float2bfloat16_rn(x);
}

// floor(a / b) for b > 0.
__device__ __forceinline__ int64_t floor_div(int64_t a, int64_t b) {
  int64_t q = a / b;
  if ((a % b != 0) && (a < 0)) --q;
  return q;
}

// Start and end (exclusive) of the packed document holding position p.
__device__ __forceinline__ void doc_bounds(const int32_t* cu, int32_t n_docs, int64_t p,
                                           int64_t* start, int64_t* end) {
  int lo = 0, hi = n_docs - 1;
  while (lo < hi) {  // largest d with cu[d] <= p
    int mid = (lo + hi + 1) >> 1;
    if ((int64_t)__ldg(cu + mid) <= p) lo = mid; else hi = mid - 1;
  }
  *start = __ldg(cu + lo);
  *end = __ldg(cu + lo + 1);
}

// a / b for a >= 0, b > 0: one 32-bit division when both fit (positions and
// strides of any buffer one GPU holds do), 64-bit otherwise.
__device__ __forceinline__ int64_t udiv_pos(int64_t a, int64_t b) {
  return ((uint64_t)a | (uint64_t)b) < 0x80000000ull ? (int64_t)((uint32_t)a / (uint32_t)b) : a / b;
}

// Tiles of `tile` rows over one schedule segment.  Positions grow with the row
// index (pos_stride >= 1), so each visibility test below holds for a prefix or a
// suffix of the segment's tiles and a range is found without walking them.

// Key tiles [lo, hi) of segment sg holding a key that some query of a span can
// see: not after the span's last query pq_hi (causal), not at or after the end
// en_hi of that query's document, not wholly before the start st_lo of the first
// query's document (documents only), not wholly before win_lo = (first query) -
// window + 1 (sliding window; INT64_MIN without one).
__device__ __forceinline__ void key_tile_range(const KSeg& sg, int tile, int64_t pq_hi, int64_t st_lo,
                                               int64_t en_hi, int causal, int docs, int64_t win_lo,
                                               int& lo, int& hi) {
  const int64_t step = (int64_t)sg.pos_stride * tile;  // position advance per tile
  hi = (sg.nk + tile - 1) / tile;
  if (causal) {  // first key of the tile <= pq_hi
    const int64_t d = pq_hi - sg.pos_off;
    hi = d < 0 ? 0 : (int)min((int64_t)hi, udiv_pos(d, step) + 1);
  }
  if (docs) {  // first key of the tile < en_hi
    const int64_t d = en_hi - 1 - sg.pos_off;
    hi = d < 0 ? 0 : (int)min((int64_t)hi, udiv_pos(d, step) + 1);
  }
  lo = 0;
  const int64_t first = max(docs ? st_lo : INT64_MIN, win_lo);  // first position any query sees
  if (first != INT64_MIN && hi > 0) {  // last key of the tile >= first: a lower bound, then step forward
    const int64_t d = first - sg.pos_off;
    if (d > 0) lo = (int)min((int64_t)hi, max((int64_t)0, (udiv_pos(d, sg.pos_stride) - (tile - 1)) / tile));
    while (lo < hi) {
      const int n = min(tile, sg.nk - lo * tile);
      if ((int64_t)sg.pos_off + (int64_t)sg.pos_stride * (lo * tile + n - 1) >= first) break;
      ++lo;
    }
  }
  if (lo > hi) lo = hi;
}

// Query tiles [lo, hi) of segment sg holding a query at or after key position
// pk_lo (causal; every tile otherwise) and starting no later than win_hi =
// (last key) + window - 1 (sliding window; INT64_MAX without one).
__device__ __forceinline__ void query_tile_range(const KSeg& sg, int tile, int64_t pk_lo, int causal,
                                                 int64_t win_hi, int& lo, int& hi) {
  hi = (sg.nk + tile - 1) / tile;
  if (win_hi != INT64_MAX) {  // first query of the tile <= win_hi
    const int64_t d = win_hi - sg.pos_off;
    hi = d < 0 ? 0 : (int)min((int64_t)hi, udiv_pos(d, (int64_t)sg.pos_stride * tile) + 1);
  }
  lo = 0;
  if (causal) {  // last query of the tile >= pk_lo: a lower bound, then step forward
    const int64_t d = pk_lo - sg.pos_off;
    if (d > 0) lo = (int)min((int64_t)hi, max((int64_t)0, (udiv_pos(d, sg.pos_stride) - (tile - 1)) / tile));
    while (lo < hi) {
      const int n = min(tile, sg.nk - lo * tile);
      if ((int64_t)sg.pos_off + (int64_t)sg.pos_stride * (lo * tile + n - 1) >= pk_lo) break;
      ++lo;
    }
  }
  if (lo > hi) lo = hi;
}

// Locates unit u in a schedule: query group, query tile index, head.
__device__ __forceinline__ void decode_unit(const Schedule& s, int tile_rows, int heads, int u,
                                            int* g_out, int* tile_out, int* h_out) {
  int h = u % heads;
  int rest = u / heads;
  if (s.n_order > 0) {
    const int e = s.order[rest];
    *g_out = e >> 20;
    *tile_out = e & 0xfffff;
    *h_out = h;
    return;
  }
  int g = 0;
  for (int i = 1; i < s.n_groups; ++i)
    if (s.g[i].tile0 <= rest) g = i;
  int ntiles = (s.g[g].nq + tile_rows - 1) / tile_rows;
  int local = rest - s.g[g].tile0;
  *g_out = g;
  *tile_out = ntiles - 1 - local;  // heaviest (last) tiles of a group first
  *h_out = h;
}

// Unit u of a launch ordered in blocks of head_block heads: the block is
// u / (head_block * pairs); inside it the (group, tile) pairs come in the launch
// order table's (else the default) order with the block's heads fastest, so the
// CTAs resident together share the other side's rows of a few heads in L2.
// head_block = heads gives the plain order (every head fastest).
__device__ __forceinline__ void decode_unit_blocked(const Schedule& s, int tile_rows, int head_block,
                                                    int pairs, int u, int* g_out, int* tile_out,
                                                    int* h_out) {
  const int per_block = head_block * pairs;
  const int b = u / per_block, rem = u - b * per_block, pair = rem / head_block;
  int h0;
  decode_unit(s, tile_rows, 1, pair, g_out, tile_out, &h0);
  *h_out = b * head_block + (rem - pair * head_block);
}

}  // namespace cpa
