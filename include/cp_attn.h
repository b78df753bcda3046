/*
 * cp_attn.h -- C ABI of the GB300 (sm_103a) causal context-parallel attention library.
 *
 * The sequence of a causal softmax attention is split into P "virtual ranks"
 * that all live in one GPU's HBM.  The calls below follow the statement of the
 * problem in the handbook chapter "Context parallelism: Ring Attention and
 * Ulysses" (sections "Which operations partition directly", "Ulysses:
 * transposing between the sequence and the heads", "Ring Attention: passing
 * the KV once around a ring", "The zigzag partition") and the reorder
 * strategies of the MaxText pull request "Add Packing Support for Context
 * Parallelism (Ring Attention) #2906" (ReorderStrategy DUAL_CHUNK_SWAP /
 * STRIPED / AUTO).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Tensors are row-major [S, H, D] (D fastest) as in the handbook's
 *    attention(q, k, v): q is [Sq, Hq, D], k and v are [Sk, Hkv, D].
 *    Grouped-query attention: query head h reads key/value head h / (Hq/Hkv).
 *  - lse (log-sum-exp of the scaled scores, natural log) is fp32 [H, Sq].
 *  - Every tensor pointer is a DEVICE pointer, 16-byte aligned, owned by the
 *    caller.  The library allocates no device memory: scratch space comes from
 *    a caller workspace whose size cp_workspace_size() reports.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Calls only enqueue work and return; they do not synchronise,
 *    except cp_check_device_status().
 *  - Arguments are validated before any launch; a refused call launches
 *    nothing and returns a negative cp_status; cp_last_error() then holds a
 *    thread-local message naming the offending argument.
 *  - dtype is CP_F32 or CP_BF16 for the q/k/v/out tensors; accumulation and
 *    softmax are fp32 in both cases.  bf16 outputs are rounded to nearest even.
 *  - A row that sees no key (all masked) has lse = -inf and out = 0.
 */
#ifndef CP_ATTN_H
#define CP_ATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CP_API __attribute__((visibility("default")))
#else
#define CP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CP_OK = 0,
  CP_ERR_INVALID_ARG = -1,    /* null pointer, bad enum, negative size */
  CP_ERR_SHAPE = -2,          /* sizes that do not divide (S % P, H % P, Hq % Hkv, ...) */
  CP_ERR_DTYPE = -3,          /* dtype not CP_F32 / CP_BF16, or not supported for this D */
  CP_ERR_ALIGN = -4,          /* pointer not 16-byte aligned, row bytes not a multiple of 16 */
  CP_ERR_UNSUPPORTED = -5,    /* valid in principle but not provided (e.g. packing with contiguous ring) */
  CP_ERR_WORKSPACE = -6,      /* workspace NULL or smaller than cp_workspace_size() */
  CP_ERR_CUDA = -7,           /* a CUDA runtime call failed (launch error, ...) */
  CP_ERR_DEVICE_TIMEOUT = -8, /* a kernel's bounded wait expired (reported by cp_check_device_status) */
  CP_ERR_DEVICE_INDEX = -9    /* library built with CP_DEBUG: a kernel's index check failed and the
                                 access was skipped (reported by cp_check_device_status) */
} cp_status;

typedef enum { CP_F32 = 0, CP_BF16 = 1 } cp_dtype;

/* Load-balancing layout of the ring (ReorderStrategy of the MaxText packing PR).
 * CONTIGUOUS: rank r holds positions [r*S/P, (r+1)*S/P).
 * DUAL_CHUNK_SWAP (zigzag): 2P chunks of C = S/(2P); rank r holds chunk r then chunk 2P-1-r.
 * STRIPED: rank r holds positions r, r+P, r+2P, ... (token-granular round robin).
 * AUTO: STRIPED when documents are packed (cu_seqlens != NULL), else DUAL_CHUNK_SWAP. */
typedef enum {
  CP_REORDER_CONTIGUOUS = 0,
  CP_REORDER_DUAL_CHUNK_SWAP = 1,
  CP_REORDER_STRIPED = 2,
  CP_REORDER_AUTO = 3
} cp_reorder;

/* How the ring's P steps are executed on one GPU.
 * FUSED: one launch; each query tile walks the ring's key/value blocks in ring
 *   order (src = r, r-1, ... mod P) and merges them in the kernel's online
 *   softmax, which is the same log-sum-exp merge.
 * STEPWISE: one attention launch per ring step writing a partial (o, lse) in
 *   fp32, followed by cp_lse_merge into the running result, as in the ring
 *   section's loop. */
typedef enum { CP_RING_FUSED = 0, CP_RING_STEPWISE = 1 } cp_ring_mode;

/* Which operation a workspace is sized for (cp_workspace_size). */
typedef enum {
  CP_OP_RING_FWD = 0,
  CP_OP_RING_BWD = 1,
  CP_OP_ULYSSES_FWD = 2,
  CP_OP_BLOCK_BWD = 3,
  CP_OP_RING_FWD_REORDERED = 4,
  CP_OP_ULYSSES_BWD = 5,
  CP_OP_USP_FWD = 6
} cp_op;

/* Visibility rule of one (query block, key block) pair.
 * Query row i sits at global position q_offset + q_stride*i, key row j at
 * k_offset + k_stride*j (strides >= 1; 1 = contiguous block, P = striped).
 * causal != 0: key j is visible to query i only if pos_k(j) <= pos_q(i)
 *   (the handbook's masked_fill(ki > qi) with offsets).
 * cu_seqlens (DEVICE pointer, n_docs+1 int32 ascending from 0, or NULL):
 *   packed documents; a key is visible only if it lies in the query's
 *   document.  Positions must lie in [0, cu_seqlens[n_docs]). */
typedef struct {
  int32_t causal;
  int64_t q_offset, k_offset;
  int64_t q_stride, k_stride;
  const int32_t* cu_seqlens;
  int32_t n_docs;
  int32_t window;  /* sliding window: with causal, key visible iff pos_q - pos_k < window; 0 = none */
} cp_mask;

/* ---------------------------------------------------------------- block attention */

/* Forward attention of one block pair, returning out and the per-row lse
 * ("Which operations partition directly": attention(q, k, v, causal,
 * q_offset, k_offset) -> (out, lse)).
 *   q [Sq,Hq,D], k/v [Sk,Hkv,D] in `dtype`; out [Sq,Hq,D] in `dtype`; lse [Hq,Sq] fp32.
 *   mask: host pointer; NULL means causal with zero offsets, unit strides, one document.
 *   scale: softmax scale; 0 means 1/sqrt(D).
 * Supported: D in {16,32,64,128} for CP_F32 (FFMA kernel); D in {64,128} for
 * CP_BF16 (tcgen05 kernel); Sq, Sk >= 0 (Sq = 0 is a no-op); Hq % Hkv == 0. */
CP_API cp_status cp_attn_block_fwd(const void* q, const void* k, const void* v, int64_t Sq, int64_t Sk,
                            int32_t Hq, int32_t Hkv, int32_t D, int32_t dtype, const cp_mask* mask,
                            float scale, void* out, float* lse, void* stream);

/* Backward of cp_attn_block_fwd for the same block pair, accumulating into fp32
 * gradients, so that a caller can walk the ring of "Ring Attention: passing
 * the KV once around a ring" one (rank, source) block pair at a time and sum
 * the pairs' contributions.  The pages give no backward: this is the exact
 * gradient of sum(dout * out) of the section "Which operations partition
 * directly"'s attention, given the FINAL out and lse of the query rows (for a
 * ring, the merged ones, not this pair's partial ones), i.e.
 * P = exp(scale*s - lse), dS = P (dP - rowsum(dout*out)),
 * dq = scale * dS k, dk = scale * dS^T q, dv = P^T dout.
 *   q, out, dout [Sq,Hq,D] and k, v [Sk,Hkv,D] in `dtype`; lse [Hq,Sq] fp32.
 *   dq_acc [Sq,Hq,D], dk_acc and dv_acc [Sk,Hkv,D]: fp32 device buffers owned
 *   by the caller.  accumulate = 0 overwrites them with this pair's gradients;
 *   accumulate = 1 adds this pair's gradients to what they hold.  dk/dv of a
 *   key/value head are summed over its Hq/Hkv query heads.  They may overlap
 *   neither an input, the workspace, nor each other (CP_ERR_INVALID_ARG).
 *   workspace: >= 4*Hq*Sq bytes (Delta = rowsum(dout*out)); the size
 *   cp_workspace_size(CP_OP_BLOCK_BWD, ...) reports covers it.  Calls on one
 *   stream that add into the same buffers are ordered by the stream.
 *   mask, scale and the supported sizes as cp_attn_block_fwd; accumulate other
 *   than 0 or 1: CP_ERR_INVALID_ARG.  Asynchronous on `stream`. */
CP_API cp_status cp_attn_block_bwd(const void* q, const void* k, const void* v, const void* out,
                            const void* dout, const float* lse, int64_t Sq, int64_t Sk, int32_t Hq,
                            int32_t Hkv, int32_t D, int32_t dtype, const cp_mask* mask, float scale,
                            float* dq_acc, float* dk_acc, float* dv_acc, int32_t accumulate,
                            void* workspace, size_t ws_bytes, void* stream);

/* The same backward with gradients in the input dtype, overwritten (no
 * accumulation): dq [Sq,Hq,D], dk/dv [Sk,Hkv,D] in `dtype`.  For bf16 (D = 64
 * or 128) the tensor-core kernels write them directly; gradients that share
 * storage with an input are still correct (then fp32 accumulators in the
 * workspace are cast after the kernels, as on the FFMA path).
 *   workspace: >= cp_workspace_size(CP_OP_BLOCK_BWD, ...) bytes (Delta and fp32
 *   accumulators).  Other arguments as cp_attn_block_bwd. */
CP_API cp_status cp_attn_block_bwd_typed(const void* q, const void* k, const void* v, const void* out,
                                         const void* dout, const float* lse, int64_t Sq, int64_t Sk,
                                         int32_t Hq, int32_t Hkv, int32_t D, int32_t dtype,
                                         const cp_mask* mask, float scale, void* dq, void* dk, void* dv,
                                         void* workspace, size_t ws_bytes, void* stream);

/* cp_attn_block_bwd_typed without a workspace, allocating no device memory
 * (the pages have no counterpart: this is a library facility).  For callers
 * that may not allocate device memory and have no workspace to hand over:
 * code running behind a plugin or custom-operator interface that passes only
 * input and output buffers, runtimes that plan all device memory ahead of time
 * and forbid allocation afterwards, or processes whose allocator belongs to
 * another runtime.  Arguments, layouts and results are those of
 * cp_attn_block_bwd_typed minus the workspace.
 *   Scratch: a 32 MiB array built into the library (every GPU that loads the
 *   library keeps it until the process exits).  Sizes whose scratch
 *   (4*Hq*Sq + 4*D*(Hq*Sq + 2*Hkv*Sk) bytes, each part rounded up to 256) does
 *   not fit return CP_ERR_UNSUPPORTED with a message; nothing is launched.
 *   The first call on a device looks up the array's device address (with that
 *   device current); make that first call before any stream capture.
 *   All calls share the array and it keeps the last call's contents (each call
 *   clears what must start at zero): calls that overlap on the GPU race, so
 *   serialise them (one stream per device).  Host-side bookkeeping (argument
 *   checks, the launch schedule) may use the host heap. */
CP_API cp_status cp_attn_block_bwd_noalloc(const void* q, const void* k, const void* v,
                                           const void* out, const void* dout, const float* lse,
                                           int64_t Sq, int64_t Sk, int32_t Hq, int32_t Hkv,
                                           int32_t D, int32_t dtype, const cp_mask* mask,
                                           float scale, void* dq, void* dk, void* dv,
                                           void* stream);

/* ---------------------------------------------------------------- ring merge */

/* Merge two partial attentions over disjoint key sets ("Ring Attention":
 * lse = log(e^lse1 + e^lse2), o = o1 e^(lse1-lse) + o2 e^(lse2-lse)).
 *   o1, o2, o [Sq,H,D] in `o_dtype` (CP_F32 or CP_BF16); lse1, lse2, lse [H,Sq] fp32.
 *   o may alias o1 and lse may alias lse1 (in-place accumulation).
 *   A row with both parts empty (-inf) stays empty (lse = -inf, o = 0). */
CP_API cp_status cp_lse_merge(const void* o1, const float* lse1, const void* o2, const float* lse2,
                       void* o, float* lse, int64_t Sq, int32_t H, int32_t D, int32_t o_dtype,
                       void* stream);

/* ---------------------------------------------------------------- Ulysses exchange */

/* Sequence -> head exchange of P virtual ranks ("Ulysses": seq_to_head, one
 * all-to-all, here an in-HBM permute).
 *   x [S,H,D] (= rank r's slice [S/P,H,D] at rows r*S/P) -> y [P][S][H/P][D],
 *   y[p][s][h'][:] = x[s][p*H/P + h'][:].  Requires S % P == 0, H % P == 0,
 *   (H/P)*D*sizeof(dtype) % 16 == 0.  Bit-exact; x and y must not overlap. */
CP_API cp_status cp_ulysses_seq2head(const void* x, void* y, int64_t S, int32_t H, int32_t D, int32_t P,
                              int32_t dtype, void* stream);
/* Inverse (head_to_seq): y [P][S][H/P][D] -> x [S,H,D]. */
CP_API cp_status cp_ulysses_head2seq(const void* y, void* x, int64_t S, int32_t H, int32_t D, int32_t P,
                              int32_t dtype, void* stream);

/* ---------------------------------------------------------------- load-balancing reorders */

/* Zigzag / DUAL_CHUNK_SWAP ("The zigzag partition"): y = the ranks' holdings
 * concatenated in rank order: rank r's rows [r*2C, (r+1)*2C) are chunk r then
 * chunk 2P-1-r of x, C = S/(2P).  Requires S % (2P) == 0.  Rows are H*D
 * elements (H may be any head count).  Bit-exact; x and y must not overlap. */
CP_API cp_status cp_zigzag_reorder(const void* x, void* y, int64_t S, int32_t H, int32_t D, int32_t P,
                            int32_t dtype, void* stream);
CP_API cp_status cp_zigzag_restore(const void* y, void* x, int64_t S, int32_t H, int32_t D, int32_t P,
                            int32_t dtype, void* stream);

/* Striped: y[r*(S/P) + i] = x[i*P + r] (rank r holds positions r, r+P, ...).
 * Requires S % P == 0.  Bit-exact; x and y must not overlap. */
CP_API cp_status cp_striped_reorder(const void* x, void* y, int64_t S, int32_t H, int32_t D, int32_t P,
                             int32_t dtype, void* stream);
CP_API cp_status cp_striped_restore(const void* y, void* x, int64_t S, int32_t H, int32_t D, int32_t P,
                             int32_t dtype, void* stream);

/* The same row maps applied to the columns of an lse [H,S] fp32 array:
 * inverse = 0 takes sequence order to the ranks' order, inverse = 1 back.
 * reorder is CP_REORDER_DUAL_CHUNK_SWAP or CP_REORDER_STRIPED. */
CP_API cp_status cp_lse_reorder(const float* x, float* y, int64_t S, int32_t H, int32_t P,
                                int32_t reorder, int32_t inverse, void* stream);

/* The ring's input and output permutes of one pass in one launch each (the
 * handbook's "The zigzag partition" and the MaxText packing PR's STRIPED
 * strategy; reorder is CP_REORDER_DUAL_CHUNK_SWAP or CP_REORDER_STRIPED).
 * cp_ring_reorder_qkv: q [S,Hq,D] -> q_re, k/v [S,Hkv,D] -> k_re/v_re in the
 * ranks' order, the row map of cp_zigzag_reorder / cp_striped_reorder.
 * cp_ring_restore: o_re [S,Hq,D] -> out and lse_re [Hq,S] -> lse back in
 * sequence order (lse_re and lse may both be NULL: out only).  Device
 * pointers, caller-owned; a source and its destination must not overlap.
 * Bit-exact copies; results equal the single-tensor calls.  Errors:
 * CP_ERR_INVALID_ARG (layout, NULL, overlap), CP_ERR_SHAPE (S not a multiple
 * of 2P / P), CP_ERR_ALIGN (H*D*sizeof(dtype) not a multiple of 16 bytes). */
CP_API cp_status cp_ring_reorder_qkv(const void* q, const void* k, const void* v, void* q_re, void* k_re,
                                     void* v_re, int64_t S, int32_t Hq, int32_t Hkv, int32_t D,
                                     int32_t dtype, int32_t P, int32_t reorder, void* stream);
CP_API cp_status cp_ring_restore(const void* o_re, const float* lse_re, void* out, float* lse, int64_t S,
                                 int32_t Hq, int32_t D, int32_t dtype, int32_t P, int32_t reorder,
                                 void* stream);

/* ---------------------------------------------------------------- drivers */

/* Causal ring attention over P virtual ranks ("Ring Attention" with the
 * layout of `reorder`).  q [S,Hq,D], k/v [S,Hkv,D], out [S,Hq,D] and lse [Hq,S]
 * are in ORIGINAL sequence order; the driver reorders q/k/v into the
 * workspace, runs the ring (skipping key blocks with no visible pair), and
 * restores out (for DUAL_CHUNK_SWAP with FUSED, the ring writes out and lse
 * in sequence order directly, as cp_ring_attention_reordered_to_seq).  cu_seqlens (device, n_docs+1) packs documents; packing is
 * accepted only with a load-balanced layout (DUAL_CHUNK_SWAP, STRIPED or AUTO),
 * as in the MaxText packing PR.  Requires S % P == 0 (S % 2P for
 * DUAL_CHUNK_SWAP), 1 <= P <= 32.  workspace >= cp_workspace_size(CP_OP_RING_FWD). */
CP_API cp_status cp_ring_attention(const void* q, const void* k, const void* v, int64_t S, int32_t Hq,
                            int32_t Hkv, int32_t D, int32_t dtype, int32_t P, int32_t reorder,
                            int32_t mode, const int32_t* cu_seqlens, int32_t n_docs, void* out,
                            float* lse, void* workspace, size_t ws_bytes, void* stream);

/* The ring of cp_ring_attention on buffers ALREADY in the ranks' layout (the
 * output of cp_zigzag_reorder / cp_striped_reorder, or sequence order for
 * CONTIGUOUS), as a data loader that shards by rank would deliver them:
 * q/k/v/out rows and lse [Hq,S] columns are in rank order; cu_seqlens is in
 * sequence positions.  No reorder or restore is done.  FUSED needs no
 * workspace (may be NULL); STEPWISE needs cp_workspace_size(CP_OP_RING_FWD_REORDERED)
 * bytes for its fp32 partial results. */
CP_API cp_status cp_ring_attention_reordered(const void* q, const void* k, const void* v, int64_t S,
                                             int32_t Hq, int32_t Hkv, int32_t D, int32_t dtype,
                                             int32_t P, int32_t reorder, int32_t mode,
                                             const int32_t* cu_seqlens, int32_t n_docs, void* out,
                                             float* lse, void* workspace, size_t ws_bytes,
                                             void* stream);

/* cp_ring_attention_reordered in FUSED mode, with out [S,Hq,D] and lse [Hq,S]
 * written in SEQUENCE order: the restore of cp_ring_attention is done by the
 * attention's own output writes (each rank's pieces of the DUAL_CHUNK_SWAP and
 * CONTIGUOUS layouts are runs of consecutive positions, so every output row is
 * written once, at its sequence position).  q/k/v are in the ranks' layout as
 * for cp_ring_attention_reordered; cu_seqlens is in sequence positions.  STRIPED
 * (and AUTO with documents) returns CP_ERR_UNSUPPORTED.  No workspace. */
CP_API cp_status cp_ring_attention_reordered_to_seq(const void* q, const void* k, const void* v, int64_t S,
                                                    int32_t Hq, int32_t Hkv, int32_t D, int32_t dtype,
                                                    int32_t P, int32_t reorder, const int32_t* cu_seqlens,
                                                    int32_t n_docs, void* out, float* lse, void* stream);

/* Backward of cp_ring_attention: dq [S,Hq,D], dk/dv [S,Hkv,D] (original
 * order) from the forward's out and lse and the upstream gradient dout.
 * Every (query block, key block) pair the ring visits is differentiated with
 * the final merged lse; dK/dV of a key/value head are summed over its query
 * heads.  workspace >= cp_workspace_size(CP_OP_RING_BWD). */
CP_API cp_status cp_ring_attention_bwd(const void* q, const void* k, const void* v, const void* out,
                                const float* lse, const void* dout, int64_t S, int32_t Hq,
                                int32_t Hkv, int32_t D, int32_t dtype, int32_t P, int32_t reorder,
                                const int32_t* cu_seqlens, int32_t n_docs, void* dq, void* dk,
                                void* dv, void* workspace, size_t ws_bytes, void* stream);

/* Ulysses attention over P virtual ranks ("Ulysses"): seq2head of q, k, v;
 * full-sequence causal attention of each rank's Hq/P query heads (Hkv/P
 * key/value heads); head2seq of out.  Requires Hq % P == 0, S % P == 0, and
 * Hkv % P == 0 or P % Hkv == 0: with fewer key/value heads than ranks each
 * key/value head is replicated P/Hkv times (the chapter's note on grouped
 * heads under Ulysses), so rank p reads head p / (P/Hkv), the head of its
 * query heads under the consecutive grouping.  Otherwise CP_ERR_SHAPE.
 * `window` > 0 adds the sliding-window rule of cp_mask (the transformers pull
 * request tests Ulysses with it); 0 = plain causal.  Negative: CP_ERR_INVALID_ARG.
 * out [S,Hq,D], lse [Hq,S].  workspace >= cp_workspace_size(CP_OP_ULYSSES_FWD). */
CP_API cp_status cp_ulysses_attention(const void* q, const void* k, const void* v, int64_t S, int32_t Hq,
                               int32_t Hkv, int32_t D, int32_t dtype, int32_t P,
                               const int32_t* cu_seqlens, int32_t n_docs, int32_t window, void* out,
                               float* lse, void* workspace, size_t ws_bytes, void* stream);

/* Ulysses inside groups of P_ulysses ranks, the ring across P_ring groups (the
 * chapter's note that the two schemes compose: "Ulysses" splits the heads
 * inside a group, "Ring Attention" passes the key/value blocks between
 * groups).  Ring rank g's positions (reorder over P_ring, as in
 * cp_ring_attention) form group g; inside it the exchange gives each of the
 * P_ulysses ranks all of the group's tokens for Hq/P_ulysses heads; the FUSED
 * ring then runs across groups for every head share (one launch for all).
 *   q [S,Hq,D], k/v [S,Hkv,D] in sequence order; out [S,Hq,D], lse [Hq,S].
 *   Ring rules as cp_ring_attention with P = P_ring; Hq % P_ulysses == 0,
 *   Hkv % P_ulysses == 0, (S / P_ring) % P_ulysses == 0 (CP_ERR_SHAPE), and
 *   P_ulysses * P_ring <= 64.  workspace >= cp_workspace_size(CP_OP_USP_FWD)
 *   (independent of the degrees).  Caller-owned device pointers, 16-byte
 *   aligned; asynchronous on `stream`. */
CP_API cp_status cp_usp_attention(const void* q, const void* k, const void* v, int64_t S, int32_t Hq,
                                  int32_t Hkv, int32_t D, int32_t dtype, int32_t P_ulysses, int32_t P_ring,
                                  int32_t reorder, const int32_t* cu_seqlens, int32_t n_docs, void* out,
                                  float* lse, void* workspace, size_t ws_bytes, void* stream);

/* Backward of cp_ulysses_attention ("Ulysses: transposing between the sequence
 * and the heads"; the pages give no backward: this is the exact gradient of
 * the definition with the FINAL lse, as for the ring).  head_to_seq is the
 * backward of seq_to_head, so q, k, v and dout take the forward's exchange,
 * every rank differentiates its full-sequence attention over its heads, and
 * dq, dk, dv come back through head_to_seq; replicated key/value heads sum
 * their copies' gradients.
 *   q, out, dout: [S,Hq,D]; k, v: [S,Hkv,D]; lse: [Hq,S] fp32 from the forward.
 *   dq [S,Hq,D], dk/dv [S,Hkv,D]: written (not accumulated), input dtype.
 *   Same shape rules as cp_ulysses_attention; all device pointers 16-byte
 *   aligned, caller-owned; workspace >= cp_workspace_size(CP_OP_ULYSSES_BWD)
 *   (fp32 accumulators and the exchanged tensors).  Asynchronous on `stream`. */
CP_API cp_status cp_ulysses_attention_bwd(const void* q, const void* k, const void* v, const void* out,
                                          const float* lse, const void* dout, int64_t S, int32_t Hq,
                                          int32_t Hkv, int32_t D, int32_t dtype, int32_t P,
                                          const int32_t* cu_seqlens, int32_t n_docs, int32_t window,
                                          void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                                          void* stream);

/* Workspace bytes needed by `op` (a cp_op) for these sizes; `mode` is the
 * cp_ring_mode for CP_OP_RING_FWD and ignored otherwise.  For CP_OP_BLOCK_BWD
 * pass S = max(Sq, Sk) (P is ignored): the size serves both cp_attn_block_bwd
 * and cp_attn_block_bwd_typed.  Returns CP_OK and writes *bytes, or an error
 * for invalid sizes. */
CP_API cp_status cp_workspace_size(int32_t op, int64_t S, int32_t Hq, int32_t Hkv, int32_t D,
                            int32_t dtype, int32_t P, int32_t mode, size_t* bytes);

/* ---------------------------------------------------------------- status */

/* Synchronises `stream`, then reports (and clears) the library's device error
 * word: CP_ERR_DEVICE_TIMEOUT if a kernel gave up on a bounded wait since the
 * last check, CP_ERR_DEVICE_INDEX if a debug build's index check failed,
 * CP_ERR_CUDA if the stream holds a CUDA error, else CP_OK. */
CP_API cp_status cp_check_device_status(void* stream);

/* Test hook for the bounded-wait path: launches one block that waits on a
 * barrier nothing arrives on, with a limit of `timeout_us` microseconds
 * (1..1000000).  The wait gives up, records CP_ERR_DEVICE_TIMEOUT in the device
 * error word and the kernel returns; nothing faults or hangs. */
CP_API cp_status cp_debug_bounded_wait(int32_t timeout_us, void* stream);

CP_API const char* cp_status_string(int32_t status);
/* Thread-local message describing the last refused or failed call on this thread. */
CP_API const char* cp_last_error(void);
/* Library version, "major.minor.patch". */
CP_API const char* cp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CP_ATTN_H */
