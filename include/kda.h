/*
 * kda.h -- C ABI of libkda, the GB300 (sm_103a) library for the Kimi Delta
 * Attention (KDA) recurrent-state hot path of a serving engine.
 *
 * The method.  Every attention head keeps a d_k x d_v state S (128 x 128)
 * updated per token as
 *     alpha_t = exp(g_t),  g_t = -softplus(raw gate_t)      (per key channel)
 *     beta_t  = sigmoid(raw beta_t)                         (per token and head)
 *     u_t = beta_t (v_t - (Diag(alpha_t) S_{t-1})^T k_t)
 *     S_t = Diag(alpha_t) S_{t-1} + k_t u_t^T,      o_t = S_t^T (scale q_t).
 * The serving pages that motivate each call:
 *   - "State semantics" page (rollback, fork, replay, TP): rollback is an
 *     exact block copy (section 2), a fork copies the whole state per
 *     candidate (section 3), decode and verify activate gates inside the
 *     kernel (section 4).
 *   - SGLang PR 34820 page: chunk prefill writes the fp32 accumulator at a
 *     per-sequence chunk index as the prefix-cache snapshot (implementation
 *     breakdown, items 1-2, and the Helion kernel listing).
 *   - vLLM PR 51855 page (RecoverSSM): verify keeps one checkpoint per request
 *     and records fp32 u and activation-dtype key / raw gate (implementation
 *     breakdown, items 1 and 3); commit rebuilds the state at the accepted
 *     length in closed form after sampling (item 4).
 *
 * Conventions shared by every entry point
 *   - All pointers are DEVICE pointers unless stated otherwise; the caller
 *     owns all memory.  The library allocates nothing.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) and never synchronises with the host.
 *   - Activations are packed [rows, H, 128] with the channel contiguous, raw
 *     beta is [rows, H].  `in_dtype` gives their element type (bf16 or fp32).
 *     Outputs are [rows, H, d_v] of `out_dtype`; bf16 outputs are rounded to
 *     nearest-even from the fp32 result.
 *   - States are stored transposed: pool[slot][h][v][k] = S[k][v] (d_v rows
 *     of d_k contiguous elements): fp32 (64 KiB per head) unless flags hold
 *     KDA_STATE_BF16 or KDA_STATE_F16 (32 KiB per head); see below.
 *   - d_k = d_v = 128 and chunk = 64 are the supported shapes; others return
 *     KDA_ERR_UNSUPPORTED.  Every device pointer must be 16-byte aligned.
 *   - Host-checkable errors (null pointer, bad size, misalignment) return a
 *     kda_status and launch nothing.  Data-dependent errors found on the GPU
 *     (a bad slot, track index, accepted length or cu_seqlens entry, an
 *     overlap in a copy set) are OR-ed into *dev_status (device int32, may be
 *     NULL) and the offending unit is skipped; kernels never trap.
 *   - flags: KDA_GATE_LOG = the gate input already holds g (log decay);
 *     KDA_BETA_ACT = the beta input already holds beta.  Default: both raw.
 *     KDA_STATE_BF16 / KDA_STATE_F16 = the state type (default fp32).
 *     KDA_QK_L2NORM = q and k normalised per (row, head) inside the kernels.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1, /* null pointer, negative size, misalignment   */
    KDA_ERR_UNSUPPORTED = 2, /* shape or dtype outside the supported set    */
    KDA_ERR_CUDA = 3         /* a CUDA launch or runtime call failed         */
} kda_status;

typedef enum { KDA_BF16 = 0, KDA_F32 = 1 } kda_dtype;

#define KDA_GATE_LOG 1u
#define KDA_BETA_ACT 2u
/* kda_chunk_prefill only: evaluate token by token (the recurrent form) instead
 * of chunk by chunk on the tensor cores; used to measure the chunk-vs-recurrent
 * numerical gap ("state semantics" page, section 4 and its open item). */
#define KDA_PREFILL_RECURRENT 4u
/* Element type of every state the call reads or writes (pool slots, and the
 * prefill's snapshots): fp32 by default, bf16 or fp16 with one of these bits
 * (both set: KDA_ERR_UNSUPPORTED).  Computation stays fp32; loads widen
 * exactly and each store rounds the fp32 result once, to nearest even, into
 * the slot's type (SGLang PR 34820 page, key files: the fp32 snapshot is
 * converted exactly once into the pool dtype, and an fp16 pool is never
 * rounded through bf16 on the way).  A 16-bit state slot is 32 KiB per head;
 * the pool layout is otherwise unchanged. */
#define KDA_STATE_BF16 8u
#define KDA_STATE_F16 16u
/* q and k are L2-normalised per (row, head) inside the kernels before any use,
 * in fp32: x / sqrt(sum_i x_i^2 + 1e-6) (the serving configurations normalise
 * q and k per head; this does it in the path instead of in a separate pass).
 * kda_spec_verify's key record still holds k as given; kda_spec_commit and
 * kda_spec_accept_commit with the same flag normalise the recorded key the
 * same way.  kda_chunk_prefill honours it on every path (two-phase,
 * single-pass and token-serial). */
#define KDA_QK_L2NORM 32u

/* bits OR-ed into *dev_status by the kernels */
#define KDA_DEV_BAD_SLOT 1     /* slot index >= pool size (or required and < 0) */
#define KDA_DEV_BAD_TRACK 2    /* track_chunk_idx outside [-1, n_chunks-1]      */
#define KDA_DEV_BAD_ACCEPT 4   /* accepted length outside [0, q_len], bad q_len */
#define KDA_DEV_BAD_SEQLEN 8   /* cu_seqlens not monotone or past T_tot         */
#define KDA_DEV_OVERLAP 16     /* slot-copy sets not disjoint                    */
#define KDA_DEV_TIMEOUT 32     /* a bounded wait inside a kernel gave up         */

#define KDA_MAX_POOLS 16

/*
 * kda_chunk_prefill -- chunked prefill over variable-length packed sequences
 * (SGLang PR 34820 page, the fp32 track-state snapshot in chunk prefill).
 *
 *   q, k, gate_raw : [T_tot, H, d_k] in_dtype;  v : [T_tot, H, d_v] in_dtype
 *   beta_raw       : [T_tot, H] in_dtype
 *   cu_seqlens     : [N+1] int32 (device), cu_seqlens[0] = 0, non-decreasing,
 *                    cu_seqlens[N] <= T_tot.  Sequence n is rows
 *                    [cu_seqlens[n], cu_seqlens[n+1]); chunks restart at each
 *                    sequence start and the last chunk may be partial.
 *   state_pool     : [P, H, d_v, d_k] states.  init_slot[n] >= 0 reads the
 *                    initial state from that slot (< 0: zero state);
 *                    final_slot[n] >= 0 receives the state after the whole
 *                    sequence (< 0: not written).  init and final may be the
 *                    same slot (in-place continuation).  init_slot / final_slot
 *                    may be NULL (= all -1).
 *   track_chunk_idx: [N, M] int32 (device) or NULL when M = 0.  Entry j >= 0
 *                    asks for the fp32 state after exactly j*chunk tokens of the
 *                    sequence (j = 0 is the initial state), j in
 *                    [0, n_chunks-1]; -1 = unused.
 *   track_state    : [N, M, H, d_v, d_k] snapshots in the state type (written
 *                    only for valid entries; the fp32 accumulator itself, or
 *                    with a 16-bit state type that accumulator rounded once).
 *   out            : [T_tot, H, d_v] out_dtype.
 *   workspace      : optional device scratch of ws_bytes bytes.
 *                    ws_bytes >= kda_chunk_prefill_workspace_size(...) (about
 *                    2 KiB per token-head: every (chunk, head)'s prepared
 *                    operands, plus 64 KiB per (sequence, head), plus 3 MiB
 *                    per (sequence, head) when N <= 8 and the rows hold at
 *                    least 256 chunks per sequence) runs the two-phase path:
 *                    all chunks' state-independent work in parallel on every
 *                    SM, then one sequential pass per (sequence, head).  Up
 *                    to 8 long sequences with few (sequence, head) pairs run
 *                    that pass in chunk segments, all at once (each middle
 *                    segment's linear state map and offset, the segment
 *                    start states chained from them on the GPU, then every
 *                    segment swept from its start: within fp32 rounding of
 *                    the unsegmented pass, deterministic), when a cost model
 *                    expects it to pay; one sequence otherwise, with up to a
 *                    quarter as many heads as SMs, runs its segments one
 *                    after another, each beside the preparation of the next
 *                    (the same results bit for bit).  A smaller
 *                    workspace (>= 16 * ceil(N / 4) bytes) runs the single-pass
 *                    kernel with the longest sequences first; NULL runs it in
 *                    input order.  The paths agree within the stated
 *                    tolerances; the single-pass results do not depend on the
 *                    order (bit-identical).
 * The chunk algorithm runs on the tensor cores: two-phase (bf16 or fp32
 * activations, N <= 4096, M <= 512, a workspace of the size above), else
 * single-pass (bf16 activations).  fp32 activations without that workspace,
 * and any call with KDA_PREFILL_RECURRENT, run the token-serial kernel.
 * Units of work are (sequence, head); sequences must not share a final slot.
 */
kda_status kda_chunk_prefill(const void* q, const void* k, const void* v, const void* beta_raw,
                             const void* gate_raw, kda_dtype in_dtype, const int32_t* cu_seqlens,
                             int32_t N, int32_t T_tot, int32_t H, int32_t dk, int32_t dv,
                             int32_t chunk, float scale, uint32_t flags, void* state_pool,
                             int64_t P, const int32_t* init_slot, const int32_t* final_slot,
                             const int32_t* track_chunk_idx, int32_t M, void* track_state,
                             void* out, kda_dtype out_dtype, void* workspace, size_t ws_bytes,
                             int32_t* dev_status, void* stream);

size_t kda_chunk_prefill_workspace_size(int32_t T_tot, int32_t N, int32_t H, int32_t dk,
                                        int32_t dv, int32_t chunk);

/*
 * kda_recurrent_decode -- one token per request, state updated in place in a
 * slot-indexed state pool ("state semantics" page, section 4: decode applies
 * the gate activation inside the kernel).
 *
 *   q, k, gate_raw : [R, H, d_k];  v : [R, H, d_v];  beta_raw : [R, H]
 *   slot           : [R] int32.  slot < 0: padding request, skipped, its
 *                    output row is written as zeros.  slot >= P: skipped,
 *                    zero output, KDA_DEV_BAD_SLOT.  Slots of one call must be
 *                    distinct: this is not checked, and a slot listed twice
 *                    leaves its state undefined (two blocks update it at once)
 *                    with no dev_status bit set.
 *   out            : [R, H, d_v] out_dtype.
 */
kda_status kda_recurrent_decode(const void* q, const void* k, const void* v, const void* beta_raw,
                                const void* gate_raw, kda_dtype in_dtype, int32_t R, int32_t H,
                                int32_t dk, int32_t dv, float scale, uint32_t flags,
                                void* state_pool, int64_t P, const int32_t* slot, void* out,
                                kda_dtype out_dtype, int32_t* dev_status, void* stream);

/*
 * kda_spec_verify -- speculative verify from one checkpoint per request
 * (vLLM PR 51855 page, implementation breakdown item 3: read the checkpoint
 * only, compute the output at every speculative position, record u and the
 * key / raw gate).
 *
 *   q, k, gate_raw : [R*K, H, d_k];  v : [R*K, H, d_v];  beta_raw : [R*K, H]
 *                    (request r's position t is row r*K + t).
 *   q_len          : [R] int32 in [0, K] or NULL (= K for all).
 *   ckpt_slot      : [R] int32: the checkpoint read from state_pool (never
 *                    written).  < 0: request skipped; >= P: skipped +
 *                    KDA_DEV_BAD_SLOT.
 *   rec_u          : [R, H, K, d_v] fp32, u_t as computed here.
 *   rec_kg         : [R, H, K, 2*d_k] of in_dtype: k_t followed by the raw
 *                    gate exactly as given.
 *   out            : [R*K, H, d_v] out_dtype.
 * Positions t >= q_len and skipped requests get zero outputs and records.
 * K <= 16 (else KDA_ERR_UNSUPPORTED); K = 0 or R = 0 launches nothing.
 */
kda_status kda_spec_verify(const void* q, const void* k, const void* v, const void* beta_raw,
                           const void* gate_raw, kda_dtype in_dtype, int32_t R, int32_t K,
                           const int32_t* q_len, int32_t H, int32_t dk, int32_t dv, float scale,
                           uint32_t flags, const void* state_pool, int64_t P,
                           const int32_t* ckpt_slot, float* rec_u, void* rec_kg, void* out,
                           kda_dtype out_dtype, int32_t* dev_status, void* stream);

/* One short-convolution state tensor (HOST descriptor): slot s starts at
 * base + s*slot_stride_bytes and holds n_rows rows of row_bytes bytes (row j
 * at + j*row_bytes; a row is one position, its channels contiguous). */
typedef struct {
    void* base;                /* device, 16-byte aligned                       */
    int64_t slot_stride_bytes; /* multiple of 16, >= n_rows * row_bytes          */
    int64_t row_bytes;         /* channels * element size, multiple of 16        */
    int32_t n_rows;            /* keep history rows + room for the step's inputs */
    int32_t num_slots;
} kda_conv_desc;

/*
 * kda_spec_accept -- the accepted length of every speculative request, on the
 * device (vLLM PR 51855 page, implementation breakdown item 4: the commit plan
 * computes the runtime accepted lengths on the GPU, and num_accepted_tokens is
 * written straight back to GPU buffers).  Its output feeds kda_spec_commit on
 * the same stream with no host synchronisation.
 *
 *   tokens       : [R, K] int32, the verify step's input ids; tokens[r][0] is
 *                  the last committed token, tokens[r][1..q_len_r-1] the drafts.
 *   sampled      : [R, K] int32, the target's sampled ids; sampled[r][i] is the
 *                  token for the position after i.
 *   q_len        : [R] or NULL (= K).  Ids at or past q_len_r are never read.
 *   num_accepted : [R] int32 out.  a_r = 1 + the number of leading drafts with
 *                  tokens[r][i+1] == sampled[r][i]; 1 <= a_r <= q_len_r.
 *                  q_len_r = 0 gives 0; q_len_r outside [0, K] gives -1 and
 *                  KDA_DEV_BAD_ACCEPT (kda_spec_commit then skips the request).
 *   next_token   : [R] int32 out or NULL: sampled[r][a_r - 1], the next input
 *                  (the first rejected draft's replacement, or the bonus
 *                  token when every draft is kept); -1 when a_r <= 0.
 * 1 <= K <= 32 (else KDA_ERR_UNSUPPORTED).  Integer work: results are exact.
 */
kda_status kda_spec_accept(const int32_t* tokens, const int32_t* sampled, const int32_t* q_len,
                           int32_t R, int32_t K, int32_t* num_accepted, int32_t* next_token,
                           int32_t* dev_status, void* stream);

/*
 * kda_spec_commit -- rebuild the state at the accepted length a_r in closed
 * form (vLLM PR 51855 page, implementation breakdown item 4: the commit plan
 * computes accepted lengths on the GPU, the commit kernel rebuilds the state
 * in reverse order in one shot, without re-running the recursion):
 *     S_a = Diag(exp sum_{t<=a} g_t) S_0 + sum_{t<=a} Diag(exp sum_{t<s<=a} g_s) k_t u_t^T
 * with g_t recomputed from the recorded raw gate.
 *
 *   ckpt_slot    : [R] checkpoint slot (S_0).   dst_slot: [R] or NULL (= ckpt,
 *                  in place).  num_accepted: [R] in [0, q_len_r].
 *   q_len        : [R] or NULL (= K).   rec_u, rec_kg: as written by verify;
 *                  rec_dtype is rec_kg's element type.
 *   plan_out     : [R, 3] int32 (a, src, dst) or NULL; a = -1 marks a request
 *                  that was skipped (bad slot or bad accepted length, with the
 *                  matching dev_status bit).
 * a = 0 writes nothing when dst == src and copies S_0 otherwise.  Destinations
 * must be distinct and must not be another request's checkpoint: this is not
 * checked, and a violation leaves the states involved undefined with no
 * dev_status bit set.  K <= 32 (else KDA_ERR_UNSUPPORTED).
 */
kda_status kda_spec_commit(void* state_pool, int64_t P, const int32_t* ckpt_slot,
                           const int32_t* dst_slot, const int32_t* num_accepted,
                           const int32_t* q_len, int32_t R, int32_t K, int32_t H, int32_t dk,
                           int32_t dv, uint32_t flags, const float* rec_u, const void* rec_kg,
                           kda_dtype rec_dtype, int32_t* plan_out, int32_t* dev_status,
                           void* stream);

/* Optional work of kda_spec_accept_commit, done in the same launch (HOST
 * struct; NULL, or n_convs = 0 and seq_len0 = NULL, asks for none).
 *   Short-convolution windows: convs (HOST array of n_convs descriptors),
 *     conv_slot ([R] device), conv_keep -- moved exactly as kda_conv_compact
 *     with the accepted lengths would.
 *   Align mode (vLLM PR 51855 page, implementation breakdown item 4: the plan
 *   computes the align boundaries and the running block index): seq_len0
 *     ([R] device, tokens before the step) and block_size.  When the accepted
 *     span seq_len0+1 .. seq_len0+a holds a multiple b of block_size, the
 *     state after a_b = b - seq_len0 accepted positions (the state at the
 *     boundary) is rebuilt from the same records into block_slot[r] (device
 *     [R], < 0: not written; >= P: KDA_DEV_BAD_SLOT); block_idx_out[r]
 *     (device [R] or NULL) receives floor((seq_len0 + a) / block_size), -1
 *     for a skipped request.  block_size < K returns KDA_ERR_UNSUPPORTED:
 *     with smaller blocks one step can cross two boundaries (the gap the
 *     RecoverSSM page records for mamba_block_size < num_speculative_tokens
 *     + 1).  Block slots must be distinct from every other slot of the call.
 */
typedef struct {
    const kda_conv_desc* convs;
    const int32_t* conv_slot;
    const int32_t* seq_len0;
    const int32_t* block_slot;
    int32_t* block_idx_out;
    int32_t n_convs;
    int32_t conv_keep;
    int32_t block_size;
    int32_t reserved; /* 0 */
} kda_commit_extras;

/*
 * kda_spec_accept_commit -- kda_spec_accept and kda_spec_commit in one launch:
 * every commit block derives its request's accepted length from the token ids
 * itself (same rule as kda_spec_accept), so the plan and the rebuild of the
 * vLLM PR 51855 page (implementation breakdown item 4) cost one launch on the
 * step's critical path.
 *
 *   tokens, sampled : [R, K] int32, as for kda_spec_accept (1 <= K <= 32).
 *   num_accepted    : [R] int32 out or NULL: the accepted lengths (-1 for a
 *                     q_len outside [0, K]).
 *   next_token      : [R] int32 out or NULL, as for kda_spec_accept.
 *   extras          : HOST struct or NULL: optional work of the same launch
 *                     (see kda_commit_extras).
 *   Every other argument is as for kda_spec_commit; the plan rows, the pool
 *   and dev_status come out exactly as kda_spec_accept followed by
 *   kda_spec_commit (and kda_conv_compact) would leave them.
 */
kda_status kda_spec_accept_commit(void* state_pool, int64_t P, const int32_t* ckpt_slot,
                                  const int32_t* dst_slot, const int32_t* tokens,
                                  const int32_t* sampled, const int32_t* q_len, int32_t R,
                                  int32_t K, int32_t H, int32_t dk, int32_t dv, uint32_t flags,
                                  const float* rec_u, const void* rec_kg, kda_dtype rec_dtype,
                                  int32_t* num_accepted, int32_t* next_token, int32_t* plan_out,
                                  const kda_commit_extras* extras, int32_t* dev_status,
                                  void* stream);

/*
 * kda_conv_compact -- the short-convolution window after a speculative step,
 * on up to KDA_MAX_POOLS conv tensors in one launch (vLLM PR 51855 page,
 * implementation breakdown item 4: the commit compacts the convolution
 * history; the conv state is a sliding window moved by an offset copy).
 *
 *   convs        : HOST array of n_convs descriptors.
 *   slot         : [R] int32 (device): the request's slot in every tensor;
 *                  < 0 skips it, >= num_slots skips it with KDA_DEV_BAD_SLOT.
 *   num_accepted : [R] int32 (device), e.g. from kda_spec_accept(_commit).
 *   keep         : history rows (the conv width minus one), >= 1.
 * Rows keep.. of a slot hold the step's inputs (position t at row keep+t).
 * After a accepted positions, rows a .. a+keep-1 move to rows 0 .. keep-1
 * (memmove semantics; rows past keep are left as they were); a = 0 changes
 * nothing; a < 0 or a + keep > n_rows skips the request with
 * KDA_DEV_BAD_ACCEPT.  Byte copy: any element type, results exact.
 */
kda_status kda_conv_compact(const kda_conv_desc* convs, int32_t n_convs, const int32_t* slot,
                            const int32_t* num_accepted, int32_t R, int32_t keep,
                            int32_t* dev_status, void* stream);

/*
 * kda_slot_copy -- one fused launch that clears, copies and fans out state
 * slots across several pools ("state semantics" page, section 2: rollback is
 * an exact block copy, replayed on every pool in one launch; section 3: a
 * fork copies the parent state to each candidate).
 *
 *   pools       : HOST array of n_pools (<= KDA_MAX_POOLS) descriptors; slot s
 *                 of pool i is slot_bytes bytes at base + s*slot_stride_bytes.
 *                 base, slot_stride_bytes and slot_bytes must be multiples of 16.
 *   clear_slots : [n_clear] slots zeroed in every pool.
 *   src_slots   : [n_src]; dst_offsets: [n_src+1] (CSR, dst_offsets[0] = 0,
 *                 dst_offsets[n_src] = n_dst); dst_slots: [n_dst].  Source i
 *                 is copied byte for byte to dst_slots[dst_offsets[i] ..
 *                 dst_offsets[i+1]-1] in every pool.
 *   workspace   : >= kda_slot_copy_workspace_size(smallest num_slots over the
 *                 pools) bytes of device scratch (the disjointness check's
 *                 bitmap over the slot ids, which are all below that size).
 * Precondition, checked on the GPU: destinations pairwise distinct and
 * disjoint from sources and clears; clears distinct and disjoint from sources;
 * every slot < num_slots of every pool.  On a violation nothing is copied and
 * KDA_DEV_OVERLAP / KDA_DEV_BAD_SLOT is set.  Under the precondition the
 * result is exact and independent of ordering.
 */
typedef struct {
    void* base;
    int64_t slot_stride_bytes;
    int64_t slot_bytes;
    int64_t num_slots;
} kda_pool_desc;

kda_status kda_slot_copy(const kda_pool_desc* pools, int32_t n_pools, const int32_t* clear_slots,
                         int32_t n_clear, const int32_t* src_slots, const int32_t* dst_offsets,
                         const int32_t* dst_slots, int32_t n_src, int32_t n_dst, void* workspace,
                         size_t ws_bytes, int32_t* dev_status, void* stream);

size_t kda_slot_copy_workspace_size(int64_t num_slots);

/*
 * kda_slot_copy_noalloc -- kda_slot_copy without a caller-provided workspace.
 * The serving pages have no counterpart; this entry point exists for callers
 * that cannot allocate device memory on demand (an engine whose allocator owns
 * all device memory after start-up, or a path where a cudaMalloc and the
 * device synchronisation it may cause are not acceptable).
 *
 * The disjointness check uses a fixed scratch array inside the library's own
 * device memory, sized for KDA_SLOT_COPY_NOALLOC_MAX_SLOTS slots (about
 * 128 KiB, held on every GPU that loads the library until the process exits).
 *   - Arguments and results are those of kda_slot_copy minus the workspace.
 *   - Returns KDA_ERR_UNSUPPORTED when the smallest pool has more than
 *     KDA_SLOT_COPY_NOALLOC_MAX_SLOTS slots; nothing is launched then.
 *   - Allocates nothing: no cudaMalloc / cudaFree and no allocating library
 *     call.  The array's device address belongs to a CUDA context: the first
 *     call in each context looks it up (cudaGetSymbolAddress, with that
 *     context current) and caches it under the context's unique id, so a
 *     context made later (after cudaDeviceReset, or another context the
 *     caller makes current) gets its own lookup and never a stale address.
 *     Make the first call in a context before any stream capture.
 *   - All calls share the one array; the kernel clears the part it uses on
 *     every call, but calls that may overlap on the GPU (different streams
 *     without ordering between them) race on it and must be serialised.
 */
#define KDA_SLOT_COPY_NOALLOC_MAX_SLOTS (1 << 20)

kda_status kda_slot_copy_noalloc(const kda_pool_desc* pools, int32_t n_pools,
                                 const int32_t* clear_slots, int32_t n_clear,
                                 const int32_t* src_slots, const int32_t* dst_offsets,
                                 const int32_t* dst_slots, int32_t n_src, int32_t n_dst,
                                 int32_t* dev_status, void* stream);

/*
 * kda_selftest_bounded_wait -- diagnostic: runs the kernels' bounded mbarrier
 * wait on a barrier nothing arrives on, for `polls` polls, and ORs
 * KDA_DEV_TIMEOUT into *dev_status when the wait gives up (it always does).
 * *cycles (device, may be NULL) receives the SM cycles the wait took.  The
 * kernels use 2^18 polls (a poll of a pending barrier suspends the thread for
 * some microseconds, so about a second); a wait that gives up there reports
 * the same bit and the call returns normally, with the context still usable.
 */
kda_status kda_selftest_bounded_wait(uint32_t polls, int32_t* dev_status,
                                     unsigned long long* cycles, void* stream);

const char* kda_status_string(kda_status s);

/* Version of the library ABI (major * 100 + minor). */
int32_t kda_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
