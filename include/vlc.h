/*
 * vlc.h -- C ABI of the varlen block-diagonal causal attention library for
 * isolated sequence packing (NVIDIA GB300, sm_103a).
 *
 * The problem (sources are cited by page title and section):
 *
 *  - Packed THD layout.  Several independent samples are concatenated into one
 *    token buffer with no batch dimension; q, k, v are [total, H, d]
 *    ("Long-context training: remove padding", vllbc, section on cu_seqlens and
 *    the THD format).
 *  - cu_seqlens.  int32 prefix sums [0, L_1, L_1+L_2, ..., total]; segment r is
 *    the half-open range [cu_r, cu_{r+1}).  Valid only if cu[0] == 0, the
 *    entries strictly increase, cu[nseg] == total and max_seqlen equals the
 *    largest difference ("Sequence packing and variable-length attention",
 *    charlestar, section "Nine tokens together keep three sample identities").
 *  - Isolation.  Token i attends to token j iff both lie in the same segment
 *    and p_j <= p_i; the mask is applied before the softmax normalisation:
 *    O = softmax(Q K^T / sqrt(d) + M) V with M in {0, -inf} (same page, section
 *    "EOS is content; isolation happens before softmax").  No work is issued
 *    for key tiles of another segment or wholly above the diagonal.
 *  - Positions.  p_i = i - cu_r (per-segment reset); RoPE rotates q and k by
 *    R(p_i) with fixed frequencies theta^(-2j/d), rotate-half pairing
 *    (x_j, x_{j+d/2}) (same page, "Positions are reset per segment"; "Packing
 *    document boundary", operatorworld, pitfall 2).
 *  - Labels.  Pre-shifted next-token labels, -100 at each segment's last token
 *    ("Length grouping, de-padding and packing", ai-infra-kb M020, section 06).
 *
 * Conventions for every call:
 *  - All data pointers are DEVICE pointers owned by the caller.  The library
 *    allocates no device memory; scratch lives in the caller's workspace
 *    (size from vlc_workspace_bytes).
 *  - Work is enqueued asynchronously on the caller's stream (a cudaStream_t,
 *    passed as void*; NULL is the legacy default stream).
 *  - A non-zero return is a host-side error detected before anything was
 *    enqueued (bad argument, unsupported shape, workspace too small, CUDA launch
 *    failure).  Content errors in cu_seqlens are found on the device: they set
 *    bits in the workspace's device error word, every later kernel of that call
 *    becomes a no-op, and vlc_get_error() reports them.  Nothing traps.
 *  - bf16 tensors are contiguous [total, H, d] row-major (last dim stride 1),
 *    d in {64, 128}, H >= 1.  lse is fp32 [H, total], natural log.
 */
#ifndef VLC_H
#define VLC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    VLC_OK = 0,
    VLC_ERR_ARG = 1,           /* null pointer, non-positive size, bad enum */
    VLC_ERR_CU_SEQLENS = 2,    /* device found cu_seqlens / max_seqlen invalid */
    VLC_ERR_UNSUPPORTED = 3,   /* head_dim not 64/128, sizes beyond the limits below */
    VLC_ERR_WORKSPACE = 4,     /* workspace pointer null / too small / misaligned */
    VLC_ERR_CUDA = 5,          /* a CUDA runtime call failed */
    VLC_ERR_TIMEOUT = 6,       /* a bounded device-side wait gave up */
    VLC_ERR_LABEL = 7          /* device found a label outside [0, vocab) other than -100 */
} vlc_status;

/* Device error word bits (vlc_get_error folds them into a vlc_status). */
#define VLC_DEVERR_CU_FIRST 0x1    /* cu[0] != 0 */
#define VLC_DEVERR_CU_ORDER 0x2    /* some cu[r+1] <= cu[r] */
#define VLC_DEVERR_CU_TOTAL 0x4    /* cu[nseg] != total */
#define VLC_DEVERR_MAXLEN 0x8      /* max_seqlen != largest segment length */
#define VLC_DEVERR_LABEL 0x10      /* a label outside [0, vocab) and not -100 */
#define VLC_DEVERR_CU_PADDED 0x20  /* cu_padded[0] != 0, a slot shorter than its segment,
                                      or cu_padded[nseg] != total */
#define VLC_DEVERR_QKV 0x40        /* a segment with fewer keys than queries (cu_kv) */
#define VLC_DEVERR_POS 0x80        /* a position outside [0, max_pos] (vlc_rope_pos) */
#define VLC_DEVERR_TIMEOUT 0x100   /* a bounded mbarrier wait expired */

/* Limits checked on the host. */
#define VLC_MAX_SEQLEN (1 << 20)   /* longest segment */
#define VLC_WORKLIST_FWD 0
#define VLC_WORKLIST_BWD 1

/* Human-readable name of a vlc_status value. */
const char* vlc_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int vlc_version(void);

/* Limit, in microseconds, of each bounded wait inside the attention kernels
 * launched after this call, for the whole process (0 restores the default of
 * 2 s).  A wait that expires raises VLC_DEVERR_TIMEOUT: the kernel drains its
 * own copies and MMAs, frees its tensor memory and returns, later kernels of the
 * call do nothing, and vlc_get_error reports VLC_ERR_TIMEOUT; the context stays
 * usable.  A limit below the default also makes the waits poll instead of
 * sleeping, so a very short limit makes the first wait that is not already
 * complete expire.  This exists to exercise that failure path (the pages have no
 * counterpart); a production caller leaves the default. */
void vlc_set_wait_limit_us(uint32_t us);

/* Bytes of workspace needed by vlc_attn_fwd (is_bwd = 0) or vlc_attn_bwd
 * (is_bwd = 1) for these sizes.  Returns 0 for invalid sizes.  The workspace
 * must be 256-byte aligned; its contents need no initialisation. */
size_t vlc_workspace_bytes(int32_t nseg, int32_t total, int32_t H, int32_t d,
                           int32_t max_seqlen, int is_bwd);

/* Capacity (in items) that vlc_build_worklist may write for these sizes:
 * an upper bound of sum_r ceil(L_r / tile) = nseg + total / tile. */
int64_t vlc_worklist_capacity(int32_t nseg, int32_t total, int32_t tile);

/* Local positions and pre-shifted labels (one kernel, HBM-bound).
 *   cu         int32 [nseg+1]   segment boundaries (see above)
 *   tokens     int64 [total]    token ids
 *   seg_ignore uint8 [nseg] or NULL; segments with a non-zero byte (padding
 *              tails) get labels -100 everywhere ("Sequence Packing",
 *              llm-compass, implementation notes)
 *   pos_out    int32 [total]    p_i = i - cu_r
 *   labels_out int64 [total]    tokens[i+1] if i+1 < cu_{r+1} and r is not
 *              ignored, else -100
 *   err_out    int32 [1] or NULL; if given, cu validity bits (VLC_DEVERR_*
 *              except MAXLEN) are OR-ed into it.  With invalid cu the outputs
 *              are unspecified but every access stays in bounds. */
int vlc_build_positions_labels(const int32_t* cu, int32_t nseg, const int64_t* tokens,
                               int32_t total, const uint8_t* seg_ignore, int32_t* pos_out,
                               int64_t* labels_out, int32_t* err_out, void* stream);

/* Work list (the first kernel of both attention calls, exposed for checking).
 * Validates cu against total/max_seqlen, then writes
 *   kind == VLC_WORKLIST_FWD: items {seg, q_tile, kv_lo, kv_hi}, one per q tile
 *       of BM rows; key tiles [kv_lo, kv_hi) = [0, ceil(min(L, (q_tile+1)BM)/BN));
 *       segments by descending q-tile count (ties by index), q tiles last to first.
 *   kind == VLC_WORKLIST_BWD: items {seg, kv_tile, q_lo, q_hi}, one per key tile
 *       of BN rows; q tiles [floor(kv_tile*BN/BM), ceil(L/BM)); segments by
 *       descending key-tile count (ties by index), key tiles first to last.
 * No item refers to another segment's rows and no tile lies wholly above the
 * diagonal ("Packing document boundary", operatorworld, pitfall 1: the varlen
 * kernel does not spend FLOPs on cross-document blocks).
 *   items_out     int32 [capacity][4], 16-byte aligned
 *   seg_order_out int32 [2*nseg+1]: the sorted segment order, then the item
 *                 offset of each sorted segment (prefix sums, last = count)
 *   count_out     int32 [1]: number of items (0 on error)
 *   err_out       int32 [1]: VLC_DEVERR_* bits are OR-ed in (caller zeroes it)
 *   capacity must be >= vlc_worklist_capacity(nseg, total, tile) where tile is
 *   BM (forward) or BN (backward); BM, BN powers of two in [16, 256];
 *   ceil(max_seqlen / tile) must stay below 16384. */
int vlc_build_worklist(const int32_t* cu, int32_t nseg, int32_t total, int32_t max_seqlen,
                       int32_t BM, int32_t BN, int kind, int32_t* items_out, int64_t capacity,
                       int32_t* seg_order_out, int32_t* count_out, int32_t* err_out,
                       void* stream);

/* Forward varlen attention with per-segment RoPE reset.
 *   q, k, v   bf16 [total, H, d]
 *   softmax_scale <= 0 selects 1/sqrt(d)
 *   rope_theta == 0 disables RoPE; otherwise q and k are rotated by R(p_i)
 *              inside the kernel (the rotated values are rounded to bf16 before
 *              the tensor-core contraction)
 *   o         bf16 [total, H, d]  (written for every token)
 *   lse       fp32 [H, total]     ln sum_j exp(s_ij) over the allowed keys
 *   ws        workspace of at least vlc_workspace_bytes(..., 0) bytes. */
int vlc_attn_fwd(const void* q, const void* k, const void* v, const int32_t* cu, int32_t nseg,
                 int32_t total, int32_t H, int32_t d, int32_t max_seqlen, float softmax_scale,
                 float rope_theta, void* o, float* lse, void* ws, size_t ws_bytes, void* stream);

/* Backward of vlc_attn_fwd: gradients of sum(O * dO) with respect to q, k, v
 * (through the RoPE rotation).  o and lse are the forward outputs.
 *   dout, q, k, v, o  bf16 [total, H, d];  lse fp32 [H, total]
 *   dq, dk, dv        bf16 [total, H, d]
 *   ws                workspace of at least vlc_workspace_bytes(..., 1) bytes. */
int vlc_attn_bwd(const void* dout, const void* q, const void* k, const void* v, const void* o,
                 const float* lse, const int32_t* cu, int32_t nseg, int32_t total, int32_t H,
                 int32_t d, int32_t max_seqlen, float softmax_scale, float rope_theta, void* dq,
                 void* dk, void* dv, void* ws, size_t ws_bytes, void* stream);

/* Grouped key/value heads (an extension of the pages' equal-head setting, which
 * they list next to the varlen interface): k, v, dk, dv are [total, H_kv, d] with
 * H_kv dividing H, and query head h attends with key/value head h / (H / H_kv);
 * dk and dv sum the contributions of the H / H_kv query heads of their group.
 * Everything else is as in vlc_attn_fwd / vlc_attn_bwd, which are these calls
 * with H_kv = H.  Workspace sizes come from vlc_workspace_bytes_gqa (the
 * backward's rotated-k copy has H_kv heads). */
size_t vlc_workspace_bytes_gqa(int32_t nseg, int32_t total, int32_t H, int32_t H_kv, int32_t d,
                               int32_t max_seqlen, int is_bwd);
int vlc_attn_fwd_gqa(const void* q, const void* k, const void* v, const int32_t* cu, int32_t nseg,
                     int32_t total, int32_t H, int32_t H_kv, int32_t d, int32_t max_seqlen,
                     float softmax_scale, float rope_theta, void* o, float* lse, void* ws,
                     size_t ws_bytes, void* stream);
int vlc_attn_bwd_gqa(const void* dout, const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const int32_t* cu, int32_t nseg, int32_t total, int32_t H,
                     int32_t H_kv, int32_t d, int32_t max_seqlen, float softmax_scale,
                     float rope_theta, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                     void* stream);

/* Option bits of vlc_attn_fwd_ex / vlc_attn_bwd_ex. */
#define VLC_ROPE_INTERLEAVED 0x1u  /* RoPE pairs (x_{2j}, x_{2j+1}) instead of (x_j, x_{j+d/2}) */
#define VLC_QK_ROTATED 0x2u        /* q and k hold R(p) q, R(p) k (from vlc_rope_qk or
                                      vlc_rope_pos): the forward rotates nothing; the backward
                                      rotates nothing and takes dq, dk back through R(p)^T
                                      (rope_theta and the pairing bit as for the rotation); the
                                      backward takes it for self-attention only */
#define VLC_KEYS_ALL_VISIBLE 0x4u  /* the _qkv calls only: every key of a query's key segment is
                                      visible (a block of keys that all precede the block of
                                      queries, as in a context-parallel ring).  The forward
                                      needs VLC_QK_ROTATED (or rope_theta == 0); the backward
                                      needs rope_theta == 0 and returns the gradients with
                                      respect to the operands as given */

/* vlc_attn_fwd_gqa / vlc_attn_bwd_gqa with a padded layout and an option word;
 * cu_padded == NULL and flags == 0 is exactly those calls.
 *
 * cu_padded (device int32 [nseg+1] or NULL): padding between segments, the
 * padded q/kv offsets of Megatron's PackedSeqParams and TE's pad_between_seqs
 * that "Sequence packing and variable-length attention" (charlestar, the
 * Megatron/TE data path) describes.  Segment r still has L_r = cu[r+1] - cu[r]
 * tokens, now at rows cu_padded[r] .. cu_padded[r] + L_r - 1; the rest of its
 * slot, up to cu_padded[r+1], is padding.  total counts all rows (cu_padded[nseg]).
 * Positions restart at 0 at each slot start.  Padding rows are not tokens: no
 * query attends to them and they attend to nothing.  Outputs at padding rows:
 * o = 0 and lse = -inf (the log of an empty sum); dq, dk, dv = 0.  Inputs at
 * padding rows (q, k, v, dout, o) must be finite: they never reach a result,
 * but the tensor cores multiply them by zero weights.  Validity (cu_padded[0]
 * == 0, every slot at least its segment's length, cu_padded[nseg] == total) is
 * checked on the device and reported as VLC_DEVERR_CU_PADDED; cu must then
 * still start at 0, increase, and have max_seqlen as its largest step.
 *
 * flags: VLC_ROPE_INTERLEAVED rotates the adjacent pairs (x_{2j}, x_{2j+1}) of
 * q and k by p_i * theta^(-2j/d), the complex-number form of RoFormer's
 * rotation that the same page ("Positions are reset per segment") cites next
 * to the rotate-half form of HF Llama; the per-segment reset and the
 * frequencies are unchanged, and the backward un-rotates dq and dk with the
 * same pairing.  The bit has no effect when rope_theta == 0.  Unknown bits
 * return VLC_ERR_ARG.
 *
 * Workspace sizes are those of vlc_workspace_bytes_gqa with total = all rows. */
int vlc_attn_fwd_ex(const void* q, const void* k, const void* v, const int32_t* cu,
                    const int32_t* cu_padded, int32_t nseg, int32_t total, int32_t H, int32_t H_kv,
                    int32_t d, int32_t max_seqlen, float softmax_scale, float rope_theta,
                    uint32_t flags, void* o, float* lse, void* ws, size_t ws_bytes, void* stream);
int vlc_attn_bwd_ex(const void* dout, const void* q, const void* k, const void* v, const void* o,
                    const float* lse, const int32_t* cu, const int32_t* cu_padded, int32_t nseg,
                    int32_t total, int32_t H, int32_t H_kv, int32_t d, int32_t max_seqlen,
                    float softmax_scale, float rope_theta, uint32_t flags, void* dq, void* dk,
                    void* dv, void* ws, size_t ws_bytes, void* stream);

/* Queries and keys/values with segments of their own (cu_seqlens_q != cu_seqlens_kv),
 * the non-square case that "Sequence packing and variable-length attention"
 * (charlestar, section "The varlen interface makes each logical segment the
 * compute range") says follows a convention of its own rather than the square
 * lower-triangle rule.  The convention taken is
 * bottom-right alignment (the one FlashAttention's varlen interface uses since
 * 2.1): segment r has L_r = cu_q[r+1] - cu_q[r] queries and Lk_r = cu_kv[r+1] -
 * cu_kv[r] >= L_r keys; its queries are the last L_r positions, so query p sits
 * at position p + Lk_r - L_r, attends keys j <= p + Lk_r - L_r of its own
 * segment, and RoPE rotates it by that position (keys by j).  L_r == Lk_r is the
 * self-attention of vlc_attn_fwd_ex.
 *   q, dout, o, dq  bf16 [total_q, H, d];  k, v, dk, dv  bf16 [total_kv, H_kv, d]
 *   lse             fp32 [H, total_q]
 *   cu_q, cu_kv     device int32 [nseg+1] each; both start at 0 and increase,
 *                   cu_q[nseg] == total_q, cu_kv[nseg] == total_kv, every
 *                   Lk_r >= L_r (else VLC_DEVERR_QKV), max_seqlen_q / _kv the
 *                   largest L_r / Lk_r (checked on the device like cu_seqlens)
 *   flags           as in vlc_attn_fwd_ex
 * Workspace: vlc_workspace_bytes_qkv.  No padded layout on this path. */
size_t vlc_workspace_bytes_qkv(int32_t nseg, int32_t total_q, int32_t total_kv, int32_t H, int32_t H_kv,
                               int32_t d, int32_t max_seqlen_q, int32_t max_seqlen_kv, int is_bwd);
int vlc_attn_fwd_qkv(const void* q, const void* k, const void* v, const int32_t* cu_q,
                     const int32_t* cu_kv, int32_t nseg, int32_t total_q, int32_t total_kv, int32_t H,
                     int32_t H_kv, int32_t d, int32_t max_seqlen_q, int32_t max_seqlen_kv,
                     float softmax_scale, float rope_theta, uint32_t flags, void* o, float* lse, void* ws,
                     size_t ws_bytes, void* stream);
int vlc_attn_bwd_qkv(const void* dout, const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const int32_t* cu_q, const int32_t* cu_kv, int32_t nseg,
                     int32_t total_q, int32_t total_kv, int32_t H, int32_t H_kv, int32_t d,
                     int32_t max_seqlen_q, int32_t max_seqlen_kv, float softmax_scale, float rope_theta,
                     uint32_t flags, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- context-parallel split
 * A long segment costs O(L^2) whatever the packing ("Sequence packing and
 * variable-length attention", charlestar, section on the two ledgers); spreading
 * it over a context-parallel group needs shards and communication that follow
 * the global segment boundaries, and a length that is a multiple of 2 * cp
 * ("Long-context training: remove padding", vllbc, failure-modes section).
 *
 * vlc_cp_partition (host): every segment of length L (a multiple of 2 * cp, else
 * VLC_ERR_ARG with *bad_seg = the first offending segment) is cut into 2 * cp
 * chunks of m = L / (2 cp); rank `rank` holds chunk `rank` (its low half) and
 * chunk 2 cp - 1 - rank (its high half) of every segment, so every rank has the
 * same causal work, (2 cp - 1) m^2 + m (m + 1) per segment.  Outputs (caller-
 * owned host arrays, total / cp rows):
 *   rows      int64 [total / cp]: the pack row of each local row: the low chunks
 *             of all segments in segment order, then the high chunks
 *   pos       int32 [total / cp]: its position inside its segment (for RoPE)
 *   cu_chunk  int32 [nseg + 1]: prefix sums of the chunk lengths m_r: each half
 *             of the local buffer is a packed buffer whose segments are the chunks
 * vlc_cp_block_mode: what the queries of (q_rank, q_half) see in the keys of
 * (kv_rank, kv_half) of the same segments: VLC_CP_BLOCK_ALL (the key chunk comes
 * first: vlc_attn_fwd_qkv with VLC_KEYS_ALL_VISIBLE), VLC_CP_BLOCK_CAUSAL (the
 * same chunk: the causal square block, L == Lk), VLC_CP_BLOCK_NONE (nothing to
 * compute); -1 for invalid arguments.  A ring step hands every rank another
 * rank's two key/value halves; the partial results (O, LSE) of a query half over
 * the blocks it sees are combined with vlc_lse_merge.  The backward of a block is
 * vlc_attn_bwd_qkv with the merged O and LSE of the query half, rope_theta == 0
 * (gradients with respect to the rotated operands) and VLC_KEYS_ALL_VISIBLE where
 * the forward had it; a query half's dq' and a key half's dk', dv are the sums
 * (vlc_sum_parts) over the blocks they took part in, and vlc_rope_pos with
 * VLC_ROPE_TRANSPOSE takes dq', dk' back to dq, dk. */
#define VLC_CP_BLOCK_NONE 0
#define VLC_CP_BLOCK_CAUSAL 1
#define VLC_CP_BLOCK_ALL 2
int vlc_cp_partition(const int32_t* cu, int32_t nseg, int32_t cp, int32_t rank, int64_t* rows, int32_t* pos,
                     int32_t* cu_chunk, int32_t* bad_seg);
int vlc_cp_block_mode(int32_t cp, int32_t q_rank, int32_t q_half, int32_t kv_rank, int32_t kv_half);

/* RoPE by explicit positions: out[i] = R(pos[i]) x[i] for every head of row i
 * ("Sequence packing and variable-length attention", charlestar, section
 * "Positions are reset per segment": the rotation of vlc_rope_qk, here with the
 * positions given, e.g. those of vlc_cp_partition or vlc_build_positions_labels),
 * rounded once to bf16.
 *   x, out    bf16 [rows, H, d] (d = 64 or 128), 16-byte aligned, not overlapping
 *   pos       device int32 [rows], 0 <= pos[i] <= max_pos; a position outside
 *             sets VLC_DEVERR_POS in the workspace word and that row's out = 0
 *   flags     VLC_ROPE_INTERLEAVED selects the pairing; VLC_ROPE_TRANSPOSE applies
 *             R(pos[i])^T instead (takes gradients with respect to rotated
 *             operands back to the unrotated ones); rope_theta > 0
 *   ws        vlc_rope_pos_workspace_bytes(max_pos, d) bytes, 256-byte aligned
 *             (error word and cos/sin table); vlc_get_error reads it */
#define VLC_ROPE_TRANSPOSE 0x8u
size_t vlc_rope_pos_workspace_bytes(int32_t max_pos, int32_t d);
int vlc_rope_pos(const void* x, const int32_t* pos, int32_t rows, int32_t H, int32_t d, int32_t max_pos,
                 float rope_theta, uint32_t flags, void* out, void* ws, size_t ws_bytes, void* stream);

/* Combine attention results over disjoint key sets into the result over their
 * union: LSE = ln sum_k e^{LSE_k}, O = sum_k e^{LSE_k - LSE} O_k, in fp32 (a
 * part with LSE_k = -inf, no visible key, weighs nothing; rows with no part
 * above -inf get O = 0, LSE = -inf).  The parts of a context-parallel ring
 * (vlc_cp_block_mode) merge into the rows' full attention.
 *   o_parts    host array of nparts device pointers, bf16 [rows, H, d] each
 *   lse_parts  host array of nparts device pointers, fp32 [H, rows] each
 *   1 <= nparts <= VLC_LSE_MERGE_MAX; o bf16 [rows, H, d], lse fp32 [H, rows],
 *   not overlapping the parts.  d = 64 or 128; o and the O parts 16-byte aligned. */
#define VLC_LSE_MERGE_MAX 16
int vlc_lse_merge(const void* const* o_parts, const float* const* lse_parts, int32_t nparts, int32_t rows,
                  int32_t H, int32_t d, void* o, float* lse, void* stream);

/* out = sum of nparts bf16 arrays of `elems` elements (a multiple of 8), accumulated
 * in fp32 and rounded once: the partial gradients of a context-parallel ring's
 * blocks.  parts: host array of device pointers, 16-byte aligned; out must not
 * overlap them; 1 <= nparts <= VLC_LSE_MERGE_MAX. */
int vlc_sum_parts(const void* const* parts, int32_t nparts, int64_t elems, void* out, void* stream);

/* ---------------------------------------------------------------- host packing
 * The data step in front of the path; plain host functions (no device, no
 * stream), deterministic (ties go to the smaller index).
 *
 * vlc_pack: windows of `capacity` tokens from samples of lengths[i] >= 1 tokens,
 * each occupying lengths[i] + extra (the BOS/EOS reserve that "Packing document
 * boundary" (operatorworld, practical checklist) asks first-fit decreasing to
 * keep).  mode ("Sequence Packing", llm-compass, section on binning):
 *   VLC_PACK_FFD        sort by size, largest first, then first fit
 *   VLC_PACK_FIRST_FIT  first fit in the given order (Megatron's dp_balanced
 *                       order, as "Long-context training: remove padding"
 *                       describes it)
 *   VLC_PACK_NEXT_FIT   streaming: the current window, else a new one
 * A sample larger than a window is not cut (the same page: over-long samples
 * are reported, not truncated): it gets a window of its own and is counted in
 * *oversize_out.  Outputs (caller-owned host arrays):
 *   bin_of     int32 [n]    window of sample i (windows numbered as opened)
 *   order      int64 [n]    samples grouped by window, each window's samples in
 *                           placement order (its cu_seqlens are their prefix sums)
 *   bin_start  int64 [n+1]  window w holds order[bin_start[w] .. bin_start[w+1])
 *   *nbins_out, *oversize_out (oversize_out may be NULL)
 * The window count over capacity gives the nominal tokens; sum(lengths) /
 * (nbins * capacity) is eta, the effective share the checklist monitors.
 * Returns VLC_ERR_ARG for a null pointer, n < 1, capacity < 1, extra < 0, a
 * length < 1 or an unknown mode. */
#define VLC_PACK_FFD 0
#define VLC_PACK_FIRST_FIT 1
#define VLC_PACK_NEXT_FIT 2
int vlc_pack(const int32_t* lengths, int64_t n, int32_t capacity, int32_t extra, int mode, int32_t* bin_of,
             int64_t* order, int64_t* bin_start, int64_t* nbins_out, int64_t* oversize_out);

/* vlc_shard_packs: windows to `ranks` data-parallel ranks by their attention
 * work ("Sequence packing and variable-length attention", charlestar: equal
 * token counts can hide unequal sum(L_r^2); balance that).  A window's cost is
 * the sum of its samples' lengths (VLC_COST_TOKENS) or of their squares
 * (VLC_COST_SUMSQ); windows by cost, largest first, each to the rank with the
 * least load so far (longest-processing-time greedy).  order / bin_start as
 * written by vlc_pack.  Outputs: rank_of_bin int32 [nbins], rank_load int64
 * [ranks].  Every rank that runs it on the same inputs gets the same answer, so
 * the ranks split the packs without exchanging anything.  VLC_ERR_UNSUPPORTED
 * if a load overflows int64. */
#define VLC_COST_TOKENS 0
#define VLC_COST_SUMSQ 1
int vlc_shard_packs(const int32_t* lengths, const int64_t* order, const int64_t* bin_start, int64_t nbins,
                    int32_t ranks, int cost_kind, int32_t* rank_of_bin, int64_t* rank_load);

/* q' = R(p_i) q and k' = R(p_i) k for every row (per-segment positions, the
 * rotation of vlc_attn_fwd, rounded once to bf16), written to caller buffers of
 * the same layouts (qrot [total, H, d], krot [total, H_kv, d]); rows past a
 * segment's length in a padded layout become zeros.  A training step can rotate
 * once and then call vlc_attn_fwd_ex / vlc_attn_bwd_ex with VLC_QK_ROTATED on q',
 * k': the forward then carries no in-kernel rotation and the backward's prep pass
 * computes rowsum(dO * O) alone, instead of each pass rotating again.  cu and
 * cu_padded are validated as in vlc_attn_fwd_ex (errors through the workspace
 * word); flags: VLC_ROPE_INTERLEAVED.  rope_theta > 0.  Workspace: the forward's
 * (vlc_workspace_bytes_gqa(..., 0)). */
int vlc_rope_qk(const void* q, const void* k, const int32_t* cu, const int32_t* cu_padded, int32_t nseg,
                int32_t total, int32_t H, int32_t H_kv, int32_t d, int32_t max_seqlen, float rope_theta,
                uint32_t flags, void* qrot, void* krot, void* ws, size_t ws_bytes, void* stream);

/* The forward with RoPE in the kernel ("Sequence packing and variable-length
 * attention", charlestar, sections "EOS is content; isolation happens before
 * softmax" and "Positions are reset per segment") that also returns the rotated
 * operands it attended with: qrot = R(p_i) q ([total, H, d]) and krot = R(p_i) k
 * ([total, H_kv, d]), bf16, per-segment positions.  A training step then runs
 * vlc_attn_bwd_ex with VLC_QK_ROTATED on qrot, krot (its prep pass computes
 * rowsum(dO * O) alone) and needs no separate rotation pass: k is rotated by the
 * pass that prepares it for the kernel (written to krot), and the kernel writes
 * each q tile's rows as it rotates them.  o, lse, the other arguments and the
 * device error word as in vlc_attn_fwd_gqa; flags: VLC_ROPE_INTERLEAVED.
 * Self-attention, no padded layout; rope_theta > 0 (else VLC_ERR_ARG); qrot and
 * krot device pointers, 16-byte aligned, owned by the caller.  Workspace:
 * vlc_workspace_bytes_gqa(..., 0) (its optional rotated-k region is not used). */
int vlc_attn_fwd_rot(const void* q, const void* k, const void* v, const int32_t* cu, int32_t nseg,
                     int32_t total, int32_t H, int32_t H_kv, int32_t d, int32_t max_seqlen,
                     float softmax_scale, float rope_theta, uint32_t flags, void* o, float* lse,
                     void* qrot, void* krot, void* ws, size_t ws_bytes, void* stream);

/* Forward attention for callers that cannot allocate device memory.  No
 * counterpart on the pages: it exists for callers that may not obtain memory
 * per call, such as code running inside another runtime's execution hook (a
 * plugin's enqueue function, a host callback) where allocating is forbidden,
 * or services whose device-memory budget is fixed at start-up, and so cannot
 * supply the workspace vlc_attn_fwd takes.
 * Same arguments and result as vlc_attn_fwd, without ws/ws_bytes; the scratch
 * lives in one file-scope device array of VLC_NOALLOC_SCRATCH_BYTES per GPU,
 * held until the process exits.
 *   err_out  int32 [1] device word or NULL: overwritten, in stream order, with
 *            this call's VLC_DEVERR_* bits (0 when the call found no error).
 * Returns VLC_ERR_WORKSPACE, before enqueuing anything, when the forward
 * workspace without its optional rotated-k region exceeds the array; when the
 * whole workspace (vlc_workspace_bytes(..., 0)) fits, k is rotated once into it
 * as in vlc_attn_fwd.  Invalid or unsupported arguments give the
 * status vlc_attn_fwd gives for them.
 * The first call on a device looks up the array's address (do it before any
 * stream capture begins).  All calls share the array: calls whose GPU work can
 * overlap race on it, so order them on one stream or with events.  Calls no
 * cudaMalloc, cudaFree or other allocating routine. */
#define VLC_NOALLOC_SCRATCH_BYTES (8u << 20)
int vlc_attn_fwd_noalloc(const void* q, const void* k, const void* v, const int32_t* cu,
                         int32_t nseg, int32_t total, int32_t H, int32_t d, int32_t max_seqlen,
                         float softmax_scale, float rope_theta, void* o, float* lse,
                         int32_t* err_out, void* stream);

/* Shifted next-token cross-entropy statistics of a packed buffer
 * ("Sequence packing and variable-length attention", charlestar, sections
 * "After isolation one cross-boundary prediction pair remains" and "Packing
 * should not decide how much a long sample weighs").  With pre-shifted labels
 * (vlc_build_positions_labels), logit row i contributes
 *   CE_i = ln sum_c exp(logits[i][c]) - logits[i][labels[i]]   if labels[i] != -100.
 *   logits        bf16 [total, vocab] row-major (vocab >= 1; rows with a -100
 *                 label are not read)
 *   labels        int64 [total]
 *   cu            int32 [nseg + 1] segment offsets, or NULL for one segment
 *                 covering the buffer (nseg is then ignored and taken as 1)
 *   loss_sum      float [1]: sum of CE_i over the pack (fp32; accumulated in fp64)
 *   target_count  int64 [1]: number of rows with a label other than -100
 *   seg_loss      float [nseg] or NULL: per-segment sums S_r
 *   seg_count     int32 [nseg] or NULL: per-segment target counts n_r
 *   ws, ws_bytes  workspace of at least vlc_ce_workspace_bytes(total, nseg) bytes,
 *                 256-byte aligned; its error word (vlc_get_error) receives
 *                 VLC_DEVERR_LABEL for an out-of-range label (that row counts
 *                 nothing) and the VLC_DEVERR_CU_* bits for an invalid cu.
 * All reductions have a fixed order: results are bitwise reproducible. */
size_t vlc_ce_workspace_bytes(int32_t total, int32_t nseg);
int vlc_shifted_ce(const void* logits, int32_t vocab, int32_t total, const int64_t* labels,
                   const int32_t* cu, int32_t nseg, float* loss_sum, int64_t* target_count,
                   float* seg_loss, int32_t* seg_count, void* ws, size_t ws_bytes, void* stream);

/* Synchronise `stream` and read the workspace's device error word.
 * Returns VLC_OK, VLC_ERR_CU_SEQLENS, VLC_ERR_LABEL, VLC_ERR_TIMEOUT or (a
 * position out of range in vlc_rope_pos) VLC_ERR_ARG;
 * *bits_out (if not NULL) receives the raw VLC_DEVERR_* bits. */
int vlc_get_error(const void* ws, int32_t* bits_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* VLC_H */
