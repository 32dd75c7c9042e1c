/*
 * spd.h -- C ABI of the GB300 (sm_103a) sample-packing and document-masked
 * attention library (libspd.so).
 *
 * Three operations, one per step of the packed-training hot path:
 *
 *   spd_pack_tokens      token lists -> packed rows: input_ids, labels,
 *                        indexes, cu_seqlens, max_seqlen
 *                        (InternEvo page "Data loading and flow", sections
 *                        "Dataloader loading data" and "Fetching data from the
 *                        Dataloader").
 *   spd_varlen_attn_fwd  causal attention over packed rows with the
 *                        block-diagonal (per-document causal) mask given by
 *                        cu_seqlens (page "Sample Packing: attention problems of
 *                        long-sequence LLM training", sections 3 "Attention
 *                        Mask" and 5.1 "FlashAttention", the varlen split into
 *                        one causal attention per document).
 *   spd_varlen_attn_bwd  its exact gradient (dQ, dK, dV).
 *
 * and the data steps that follow packing (page "Data loading and flow",
 * section "Processing data"): spd_unpack_data and
 * spd_split_sequence_parallel, and the sequence-parallel padding before the
 * split (spd_pad_for_sequence_parallel); the steps next to attention: rotary
 * position embedding with per-document positions (spd_rope, and fused into
 * the forward's prologue: spd_varlen_attn_fwd_rope) and the masked token loss
 * over the packed labels (spd_masked_token_loss).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers are DEVICE pointers unless the argument says "host". The caller
 *   owns and allocates all memory (inputs, outputs and workspace); the library
 *   allocates nothing and keeps no global state beyond a per-device cache of
 *   the SM count. Entry points are thread-safe.
 * - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *   stream). The return value reports what the host can check before launch.
 *   Errors the GPU finds (bad cu_seqlens, bad document lengths, a bounded
 *   wait that ran out) are written to a status word at the start of the
 *   workspace; spd_read_status() synchronises the stream and returns it. Each
 *   call clears the status word first, so it reports the most recent call
 *   that used that workspace. No kernel traps; on a device error the kernels
 *   finish early and the outputs are unspecified.
 * - Workspaces must be at least the size the matching *_workspace_size()
 *   returns and 256-byte aligned. Calls that share a workspace must not
 *   overlap on the GPU (use one stream, or one workspace per stream).
 * - All integer outputs are int32 (the page prints torch tensors; values are
 *   identical). Pad id is 0 and the ignore label is -100.
 */
#ifndef SPD_H
#define SPD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *spd_stream_t; /* same type as cudaStream_t */

enum {
    SPD_OK = 0,
    SPD_ERR_INVALID_ARG = -1,    /* host: null/misaligned pointer, bad size or shape */
    SPD_ERR_UNSUPPORTED = -2,    /* host: head_dim or GPU not supported */
    SPD_ERR_CUDA = -3,           /* host: a CUDA runtime/driver call failed */
    SPD_ERR_BAD_SEQLENS = -4,    /* device: cu_seqlens not 0 = c0 < c1 < ... = total */
    SPD_ERR_DEVICE_TIMEOUT = -5, /* device: a bounded wait ran out */
    SPD_ERR_WORKSPACE = -6,      /* host: workspace too small or misaligned */
    SPD_ERR_BAD_DOCS = -7,       /* device: a document length <= 0 or sum != num_tokens */
    SPD_ERR_TOO_LARGE = -8       /* host: problem exceeds the fixed scratch of a no-allocation entry point */
};

/* Text for a status code (static storage). */
const char *spd_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int spd_version(void);

/*
 * Measurement hook. For the calling host thread, make the launcher of one
 * kernel record `begin_event` / `end_event` (cudaEvent_t handles created by
 * the caller) on the launch stream immediately before and after that kernel,
 * so its duration can be read with cudaEventElapsedTime. kernel:
 * SPD_PROFILE_NONE (off), SPD_PROFILE_PACK_STREAM (the token-stream kernel of
 * spd_pack_tokens: its one kernel with at most 1024 documents, and in
 * build_pack mode at most 512 rows; else the second of its two kernels),
 * SPD_PROFILE_ATTN_FWD / SPD_PROFILE_ATTN_BWD (the main
 * attention kernel of each call, without the scheduling and pre/post-pass
 * kernels). Null events turn it off. Returns SPD_OK or SPD_ERR_INVALID_ARG.
 */
enum {
    SPD_PROFILE_NONE = 0,
    SPD_PROFILE_PACK_STREAM = 1,
    SPD_PROFILE_ATTN_FWD = 2,
    SPD_PROFILE_ATTN_BWD = 3,
    SPD_PROFILE_UNPACK = 4,   /* the kernel of spd_unpack_data */
    SPD_PROFILE_SPLIT = 5,    /* the kernel of spd_split_sequence_parallel */
    SPD_PROFILE_ROPE = 6,     /* the kernel of spd_rope */
    SPD_PROFILE_LOSS = 7,     /* the row kernel of spd_masked_token_loss */
    SPD_PROFILE_PAD = 8       /* the kernel of spd_pad_for_sequence_parallel */
};
int spd_set_profile_events(void *begin_event, void *end_event, int kernel);

/*
 * Failure-detection test hook. For the calling host thread, make the next
 * spd_varlen_attn_fwd (which = SPD_DEBUG_SKIP_FWD_Q) or spd_varlen_attn_bwd
 * (which = SPD_DEBUG_SKIP_BWD_KV) leave one producer arrive out: the TMA
 * producer of each CTA does not load its first unit's Q tile pair (forward) or
 * K / V tile (backward), so the consumer's bounded wait (2 s) runs out. The
 * kernel then stops every role at its next bounded wait, lets its own copies
 * land, frees its tensor memory and writes SPD_ERR_DEVICE_TIMEOUT into the
 * status word; outputs are undefined, the CUDA context stays usable. The hook
 * is consumed by that one call. SPD_DEBUG_SKIP_NONE clears it. Returns SPD_OK
 * or SPD_ERR_INVALID_ARG. Not for production use; the pages have no
 * counterpart.
 */
enum {
    SPD_DEBUG_SKIP_NONE = 0,
    SPD_DEBUG_SKIP_FWD_Q = 1,
    SPD_DEBUG_SKIP_BWD_KV = 2
};
int spd_debug_skip_arrive(int which);

/*
 * Synchronise `stream` and return the device status word of the last call
 * that used workspace `ws` (SPD_OK or a negative SPD_ERR_* code) in
 * *device_status (host). Returns SPD_OK or SPD_ERR_CUDA.
 */
int spd_read_status(const void *ws, spd_stream_t stream, int *device_status);

/*
 * Inspection hook: synchronise `stream`, then copy to the host the tile
 * schedule that the last spd_varlen_attn_fwd or spd_varlen_attn_bwd call built
 * in workspace `ws` (the work list every head's CTAs take units from, sorted by
 * cost, largest first; page "Sample Packing ...", section 5.1: only tiles with unmasked
 * entries are visited). *num_units (host) receives the number of work units per
 * head; units (host int32 [capacity][4]; may be NULL if capacity is 0) the first
 * min(capacity, *num_units) of them, each {segment start, segment end, tile,
 * cost}, with n = ceil((segment end - segment start) / 128) tiles of 128
 * tokens in the segment:
 *   forward:  q tiles `tile` and `tile` + 1 (if < n); q tile i reads kv tiles
 *             0 .. i; cost = the number of (q tile, kv tile) blocks read;
 *   backward: if bit 30 of `tile` is set, the one kv tile t = `tile` with
 *             that bit cleared, cost = n - t; else the pair of kv tiles `tile`
 *             and n - 1 - `tile`, cost = n + 1 (a segment's pairs sit in
 *             consecutive entries, in order). Kv tile t reads q tiles t .. n - 1
 *             of every q head of its kv head.
 * Only the diagonal blocks (q tile == kv tile) hold masked entries. Returns
 * SPD_OK, SPD_ERR_INVALID_ARG or SPD_ERR_CUDA. Not needed for normal use.
 */
int spd_attn_read_schedule(const void *ws, spd_stream_t stream, int32_t *num_units, int32_t *units,
                           int64_t capacity);

/* ------------------------------------------------------------------------- */
/* Packing                                                                   */
/* ------------------------------------------------------------------------- */

/*
 * Output sizes of spd_pack_tokens (all host arguments and results).
 *   use_packed_dataset != 0 (build_pack): rows = ceil(num_tokens / plen),
 *   use_packed_dataset == 0 (build_unpack): rows = ceil(num_docs / micro_bsz),
 *   with plen = micro_bsz * seq_len. *max_segs bounds num_segs: size
 *   cu_seqlens with max_segs + 1 entries. Returns SPD_ERR_INVALID_ARG if a
 *   size is <= 0 (num_docs / num_tokens may be 0) or rows * plen exceeds
 *   2^31 - 65537 (positions are 32-bit in the kernels, which step up to one
 *   chunk past the last position before their bounds checks).
 */
int spd_pack_rows(int64_t num_docs, int64_t num_tokens, int micro_bsz, int seq_len,
                  int use_packed_dataset, int64_t *rows, int64_t *max_segs);

/*
 * Host only (no GPU work): the exact number of segments spd_pack_tokens will
 * write to num_segs for these document lengths (doc_lens: HOST int32
 * [num_docs], each >= 1), so a caller can size and launch the attention calls
 * without reading num_segs back from the device. Packed mode: one segment per
 * row a document spans, plus the padding tail of the last row if it is not
 * full; unpack mode: each row's documents (cut to seq_len) plus the row's
 * padding tail if any. SPD_ERR_INVALID_ARG for bad arguments.
 */
int spd_pack_num_segs(const int32_t *doc_lens, int64_t num_docs, int micro_bsz, int seq_len,
                      int use_packed_dataset, int64_t *num_segs);

/* Workspace bytes spd_pack_tokens needs for num_docs documents. */
size_t spd_pack_workspace_size(int64_t num_docs);

/*
 * Pack documents into rows of plen = micro_bsz * seq_len tokens.
 *
 * Follows the InternEvo page "Data loading and flow", section "Dataloader
 * loading data":
 *   use_packed_dataset != 0 (build_pack): the documents are laid end to end
 *     and cut every plen tokens; a document that does not fit continues at the
 *     start of the next row; the last row is padded with 0. Each document's
 *     labels are its tokens from the second on followed by -100, taken before
 *     the cut (so a row's last label may be the next row's first token);
 *     padding labels are -100.
 *   use_packed_dataset == 0 (build_unpack): at most micro_bsz documents per
 *     row; each is cut to seq_len tokens and the excess dropped; labels come
 *     from the cut document; rows are padded with 0 / -100.
 * and section "Fetching data from the Dataloader" for the segment fields:
 *   segments of a row are the runs of one document's tokens, then the padding
 *   tail as its own segment; indexes[p] is p's position inside its segment
 *   (restarting at 0 at every segment start, padding included); max_seqlen[r]
 *   is the longest segment of row r.
 *
 * Inputs (device): tokens int32 [num_tokens] (the documents concatenated),
 *   doc_lens int32 [num_docs], each >= 1, summing to num_tokens (checked on
 *   the GPU: SPD_ERR_BAD_DOCS).
 * Outputs (device), with rows from spd_pack_rows:
 *   input_ids, labels, indexes  int32 [rows * plen], row-major;
 *   cu_seqlens   int32 [num_segs + 1], GLOBAL token offsets: row r's
 *                boundaries plus r * plen, each shared row end once, so
 *                cu_seqlens is directly the attention calls' argument;
 *   row_seg_ptr  int32 [rows + 1]: row r's segments are
 *                cu_seqlens[row_seg_ptr[r] .. row_seg_ptr[r+1]];
 *   max_seqlen   int32 [rows];
 *   num_segs     int32 [1].
 * Any output pointer may be unaligned; 16-byte aligned outputs take the
 * vectorised store path. Returns SPD_ERR_INVALID_ARG / SPD_ERR_WORKSPACE /
 * SPD_ERR_CUDA from the host; device errors go to the status word.
 */
int spd_pack_tokens(const int32_t *tokens, const int32_t *doc_lens, int64_t num_docs,
                    int64_t num_tokens, int micro_bsz, int seq_len, int use_packed_dataset,
                    int32_t *input_ids, int32_t *labels, int32_t *indexes, int32_t *cu_seqlens,
                    int32_t *row_seg_ptr, int32_t *max_seqlen, int32_t *num_segs, void *ws,
                    size_t ws_bytes, spd_stream_t stream);

/*
 * unpack_data (page "Data loading and flow", section "Processing data", the
 * use_packed_dataset=False path): every packed row holds at most micro_bsz
 * documents as segments; segment m of row r becomes output row (r, m) of
 * seq_len positions, its first min(length, seq_len) tokens copied from
 * input_ids / labels and the rest 0 / -100. Output rows without a segment are
 * all 0 / -100; segments beyond the first micro_bsz of a row (none in rows that
 * spd_pack_tokens built with use_packed_dataset == 0) are dropped. cu_seqlens
 * and indexes have no unpacked form (the page drops them).
 *
 * Inputs (device), as spd_pack_tokens writes them: input_ids, labels int32
 *   [rows * micro_bsz * seq_len]; cu_seqlens int32 (global offsets);
 *   row_seg_ptr int32 [rows + 1].
 * Outputs (device): out_ids, out_labels int32 [rows][micro_bsz][seq_len].
 * rows == 0 is a no-op. Returns SPD_ERR_INVALID_ARG (micro_bsz or seq_len < 1,
 * rows < 0, rows * micro_bsz * seq_len > 2^31 - 65537, a null or unaligned
 * pointer), SPD_ERR_UNSUPPORTED (not an sm_103 GPU) or SPD_ERR_CUDA. No
 * workspace: the segment offsets are trusted as spd_pack_tokens produced them.
 */
int spd_unpack_data(const int32_t *input_ids, const int32_t *labels, const int32_t *cu_seqlens,
                    const int32_t *row_seg_ptr, int64_t rows, int micro_bsz, int seq_len, int32_t *out_ids,
                    int32_t *out_labels, spd_stream_t stream);

/*
 * pad_for_sequence_parallel (XTuner page "Sequence parallel training of
 * extremely long sequences", section "Sequence parallel API", data pad and
 * split): pad every row of an int32 tensor [rows][len] to padded = the
 * smallest multiple of sp_size >= len, so the row splits evenly over the
 * sequence-parallel ranks: dst int32 [rows][padded], dst[r][j] = src[r][j]
 * for j < len; the added positions hold pad_value, or, with count_positions
 * != 0, count 0, 1, 2, ... (position ids). The page names the tensors
 * (input_ids, labels, position_ids, attention_mask) but not the values; the
 * binding pads input_ids with 0 (the pad id), labels with -100 (the ignore
 * index), position_ids by counting (the padding tail is its own segment, as
 * in the packing rules) and attention_mask with 0. Returns
 * SPD_ERR_INVALID_ARG for sp_size < 1, rows < 0, len < 0,
 * rows * padded > 2^31 - 65537, or a null / unaligned pointer with work to do;
 * SPD_ERR_UNSUPPORTED or SPD_ERR_CUDA as above.
 */
int spd_pad_for_sequence_parallel(const int32_t *src, int32_t *dst, int64_t rows, int64_t len, int sp_size,
                                  int32_t pad_value, int count_positions, spd_stream_t stream);

/*
 * split_data_sequence_parallel (page "Data loading and flow", section
 * "Processing data", isp with tp size > 1): rank `rank` of sp_size keeps the
 * contiguous chunk [rank * len / sp_size, (rank + 1) * len / sp_size) of the
 * sequence dimension of every row. Up to three int32 tensors of one shape
 * [rows][len] per call (the page splits input_ids, indexes and labels; an
 * unpacked batch has no indexes): src_i -> dst_i int32 [rows][len / sp_size];
 * unused slots are NULL (src_i and dst_i together). Returns
 * SPD_ERR_INVALID_ARG if len % sp_size != 0 (the sequence must be padded
 * first), sp_size < 1, rank outside [0, sp_size), rows < 0, len < 0,
 * rows * len > 2^31 - 65537, or a pointer is unaligned / unpaired;
 * SPD_ERR_UNSUPPORTED or SPD_ERR_CUDA as above.
 */
int spd_split_sequence_parallel(const int32_t *src0, const int32_t *src1, const int32_t *src2, int64_t rows,
                                int64_t len, int sp_size, int rank, int32_t *dst0, int32_t *dst1, int32_t *dst2,
                                spd_stream_t stream);

/*
 * Rotary position embedding with per-document positions, in place (the
 * attention-layer pseudo code under Figure 1 of the XTuner page "序列并行"
 * applies it to q and k before attention; positions are the pack's `indexes`,
 * restarting at every document: page "Sample Packing ...", section 4.1,
 * reset_position_id). Rotate-half form: channel j < d/2 of every head is
 * paired with channel j + d/2 and turned by p * theta_j, theta_j =
 * rope_theta^(-2j/d) (rope_theta <= 0: 10000); inverse != 0 turns by
 * -p * theta_j, which maps dq / dk of the rotated tensors back to the inputs.
 *
 * q bf16 [T, Hq, head_dim], k bf16 [T, Hkv, head_dim], rotated in place; either
 * may be NULL. positions int32 [T], each >= 0 (indexes of spd_pack_tokens).
 * head_dim 64 or 128. The angle is exact to ~1e-9 rad for any int32 position.
 * Returns SPD_ERR_INVALID_ARG (bad sizes, q / k not 16-byte aligned, positions
 * NULL while T > 0), SPD_ERR_UNSUPPORTED or SPD_ERR_CUDA.
 */
int spd_rope(uint16_t *q, uint16_t *k, const int32_t *positions, int64_t total_tokens, int Hq, int Hkv,
             int head_dim, float rope_theta, int inverse, spd_stream_t stream);

/*
 * Masked token loss over packed labels (XTuner page "序列并行", section
 * "Reduce Loss": the rank's loss is the mean token cross-entropy over labels
 * that are not -100; num_tokens = (labels != -100).sum() weighs it in
 * reduce_sequence_parallel_loss). For token t with a counted label:
 * token_loss[t] = logsumexp(logits[t]) - logits[t][label] (natural log, fp32);
 * ignored tokens (label -100) get 0. *loss_sum (fp64) is the sum over tokens in
 * a fixed order (reproducible), *num_tokens the count of counted tokens; the
 * caller forms the mean loss_sum / num_tokens, or the token-weighted mean over
 * sequence-parallel ranks. If dlogits is not NULL it receives
 * (softmax(logits[t]) - onehot(label)) * grad_scale (bf16), zero rows for
 * ignored tokens (grad_scale = 1 / total counted tokens for the mean).
 *
 * logits bf16 [T, V], labels int32 [T] (the pack's labels), token_loss fp32
 * [T], loss_sum double [1], num_tokens int32 [1], dlogits bf16 [T, V] or NULL,
 * device_status int32 [1] or NULL: receives SPD_ERR_INVALID_ARG if a label is
 * outside [0, V) and not -100 (that token then counts for nothing; the caller
 * clears the word before the call). Returns SPD_ERR_INVALID_ARG (bad sizes,
 * null or unaligned pointers), SPD_ERR_UNSUPPORTED or SPD_ERR_CUDA.
 */
int spd_masked_token_loss(const uint16_t *logits, const int32_t *labels, int64_t T, int64_t V, float *token_loss,
                          double *loss_sum, int32_t *num_tokens, uint16_t *dlogits, float grad_scale,
                          int32_t *device_status, spd_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Attention                                                                 */
/* ------------------------------------------------------------------------- */

/*
 * Workspace bytes for spd_varlen_attn_fwd (bwd == 0) or spd_varlen_attn_bwd
 * (bwd != 0). The backward workspace holds an fp32 dQ accumulator of
 * Hq * total_tokens * head_dim floats plus the row terms D = rowsum(dO * O).
 * Returns 0 for unsupported arguments.
 */
size_t spd_attn_workspace_size(int64_t total_tokens, int32_t num_segs, int Hq, int Hkv,
                               int head_dim, int bwd);

/*
 * Forward attention over packed rows.
 *
 * For every segment s = [a, b) of cu_seqlens, q head h and token i in s, with
 * kv head g = h / (Hq / Hkv) (GQA: consecutive q heads share a kv head, the
 * InternEvo page "Data loading and flow", section "Computing attention"):
 *   S_ij = softmax_scale * q[i,h,:] . k[j,g,:]   for a <= j <= i
 *   out[i,h,:] = sum_j softmax_j(S_i.) v[j,g,:],  lse[h,i] = log sum_j exp(S_ij)
 * Segments never interact: a packed row gives the same result as its documents
 * attended separately (page "Sample Packing ...", section 3 "Attention Mask").
 * Only the tiles of each document's own causal triangle are visited (section
 * 5.1 "FlashAttention"); the varlen split makes every document its own
 * causal attention.
 *
 * Inputs (device, contiguous, bf16 as uint16 bit patterns, 16-byte aligned):
 *   q [total_tokens, Hq, head_dim], k, v [total_tokens, Hkv, head_dim];
 *   cu_seqlens int32 [num_segs + 1], 0 = c0 < c1 < ... < c_num_segs =
 *   total_tokens (checked on the GPU: SPD_ERR_BAD_SEQLENS);
 *   max_seqlen (host) bounds the longest segment (a hint; <= 0 = unknown).
 * head_dim is 64 or 128; Hq % Hkv == 0; total_tokens and Hq * total_tokens
 * at most 2^31 - 65537; softmax_scale <= 0 means 1 / sqrt(head_dim).
 * Outputs (device): out bf16 [total_tokens, Hq, head_dim]; lse fp32
 *   [Hq, total_tokens] (natural log).
 */
int spd_varlen_attn_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                        const int32_t *cu_seqlens, int32_t num_segs, int64_t total_tokens,
                        int32_t max_seqlen, int Hq, int Hkv, int head_dim, float softmax_scale,
                        uint16_t *out, float *lse, void *ws, size_t ws_bytes,
                        spd_stream_t stream);

/*
 * spd_varlen_attn_fwd with rotary position embedding fused into its prologue:
 * the attention of RoPE(q), RoPE(k) and v, where every q and k row is rotated
 * by its position inside its segment, p = i - cu_seqlens[s] for token i of
 * segment s (positions restart at every document, page "Sample Packing ...",
 * section 4.1, reset_position_id; for the cu_seqlens of spd_pack_tokens these
 * positions are exactly its `indexes`). The rotation is the one spd_rope applies
 * (rotate-half: channel j < head_dim/2 with channel j + head_dim/2, angle
 * p * rope_theta^(-2j/head_dim); rope_theta <= 0 means 10000), done on each Q and
 * K tile in shared memory after its copy lands and before the tensor cores read
 * it; the rotated tiles are rounded to bf16 like spd_rope's output, and never
 * written to HBM (the XTuner page "序列并行", Figure 1 pseudo code, applies
 * apply_rotary_pos_emb to q and k right before the attention call). q and k are
 * read, not modified. Arguments, layouts, workspace and errors as for
 * spd_varlen_attn_fwd. The backward of this forward is spd_varlen_attn_bwd on
 * spd_rope-rotated copies of q and k (same positions, e.g. the pack's indexes),
 * followed by spd_rope(..., inverse = 1) on dq and dk.
 */
int spd_varlen_attn_fwd_rope(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                             const int32_t *cu_seqlens, int32_t num_segs, int64_t total_tokens,
                             int32_t max_seqlen, int Hq, int Hkv, int head_dim, float softmax_scale,
                             float rope_theta, uint16_t *out, float *lse, void *ws, size_t ws_bytes,
                             spd_stream_t stream);

/*
 * Backward of spd_varlen_attn_fwd: with P_ij = exp(S_ij - lse_i),
 * D_i = dout_i . out_i and dS_ij = P_ij (dout_i . v_j - D_i):
 *   dq_i = scale sum_j dS_ij k_j,
 *   dk_j = scale sum_{h in g} sum_i dS_ij q_i,
 *   dv_j = sum_{h in g} sum_i P_ij dout_i.
 * Inputs as for the forward plus out (bf16), dout (bf16) [total_tokens, Hq,
 * head_dim] and the forward's lse. grad_dtype 0 writes dq / dk / dv as bf16
 * (uint16 bit patterns), 1 as fp32; shapes [total_tokens, Hq | Hkv, head_dim].
 */
int spd_varlen_attn_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                        const uint16_t *out, const uint16_t *dout, const float *lse,
                        const int32_t *cu_seqlens, int32_t num_segs, int64_t total_tokens,
                        int32_t max_seqlen, int Hq, int Hkv, int head_dim, float softmax_scale,
                        int grad_dtype, void *dq, void *dk, void *dv, void *ws,
                        size_t ws_bytes, spd_stream_t stream);

/*
 * Forward attention without any workspace, for callers that cannot allocate
 * device memory: code that runs inside a host framework which owns all device
 * memory and hands out only the tensors of the operation, or a latency-critical
 * path that must not call cudaMalloc / cudaFree (which can synchronise the
 * whole device) and keeps no buffers of its own.
 *
 * The pages this library follows have no counterpart to this entry point; it
 * computes exactly what spd_varlen_attn_fwd computes, with the same argument
 * meaning, layouts and host checks, minus ws / ws_bytes, and allocates nothing.
 * Its scratch (status word and tile work list) is one fixed array of
 * SPD_NOALLOC_SCRATCH_BYTES (4 MiB) in the library's device image: every GPU
 * that loads the library holds it until the process exits. The rule is exact:
 * a problem fits while spd_attn_workspace_size(total_tokens, num_segs, Hq,
 * Hkv, head_dim, 0) <= SPD_NOALLOC_SCRATCH_BYTES, i.e. 16 bytes per work tile
 * (ceil(total_tokens / 128) + num_segs tiles) plus 4 bytes per segment and a
 * 256-byte header stay within 4 MiB: up to about 262,000 tiles, e.g. 33
 * million tokens in a few thousand documents, but not 16.9 million tokens in
 * 131,072 documents. A problem that does not fit returns SPD_ERR_TOO_LARGE
 * before anything is launched; shape and pointer errors are reported first
 * (SPD_ERR_INVALID_ARG / SPD_ERR_UNSUPPORTED, as for spd_varlen_attn_fwd).
 *
 * The first call on each device looks up the array's device address with that
 * device current (a runtime symbol query, no allocation); make that first call
 * before any stream capture. All calls share the one array and the array keeps
 * the last call's contents (each call rewrites what it reads), so calls that
 * overlap on the GPU -- on different streams, or from different threads --
 * race: serialise them.
 *
 * device_status (device pointer to one int32, may be NULL) receives the call's
 * device status word (SPD_OK or SPD_ERR_BAD_SEQLENS / SPD_ERR_DEVICE_TIMEOUT),
 * written on `stream` after the kernels. It is written only when the call
 * returns SPD_OK: after any other return code it holds whatever it held
 * before.
 */
#define SPD_NOALLOC_SCRATCH_BYTES (4u << 20)
int spd_varlen_attn_fwd_noalloc(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                const int32_t *cu_seqlens, int32_t num_segs, int64_t total_tokens,
                                int32_t max_seqlen, int Hq, int Hkv, int head_dim, float softmax_scale,
                                uint16_t *out, float *lse, int32_t *device_status, spd_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPD_H */
