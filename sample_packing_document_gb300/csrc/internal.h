// Launch functions shared between the C-ABI front end (api.cu) and the kernel
// translation units. Host-side only; every function launches on `stream` and
// returns a cudaError_t.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace spd {

// Measurement hook (spd_set_profile_events): when `which` names a kernel,
// its launcher records `begin` / `end` on the launch stream around that one
// kernel. Per host thread.
enum { kProfNone = 0, kProfPackStream = 1, kProfAttnFwd = 2, kProfAttnBwd = 3, kProfUnpack = 4, kProfSplit = 5, kProfRope = 6, kProfLoss = 7, kProfPad = 8 };
struct ProfileHook {
    cudaEvent_t begin = nullptr, end = nullptr;
    int which = kProfNone;
};
ProfileHook &profile_hook();

// Test hook of spd_debug_skip_arrive for the calling host thread: 1 if it is
// armed for `which` (and then clears it), else 0.
int &debug_skip_slot();
int take_debug_skip(int which);

inline void prof_begin(int which, cudaStream_t s)
{
    ProfileHook &h = profile_hook();
    if (h.which == which && h.begin) cudaEventRecord(h.begin, s);
}
inline void prof_end(int which, cudaStream_t s)
{
    ProfileHook &h = profile_hook();
    if (h.which == which && h.end) cudaEventRecord(h.end, s);
}

// Workspace header: [0] status word, [1] tile count; the rest per operation.
// Workspace header (int32 words): [0] status, [1] work units per head, [2] work
// counter of the persistent kernels, [3] long units per head (see unit_of).
constexpr size_t kWsHeader = 256;
// Largest number of positions (rows x row length) a packing or data-step call
// accepts: the kernels keep positions in 32 bits and read or write up to one
// chunk (<= 4096 positions) past the last one before their bounds checks, so
// the sums must stay below 2^31.
constexpr long long kMaxPositions = 0x7fffffffLL - 65536;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------- packing
struct PackArgs {
    const int32_t *tokens;
    const int32_t *doc_lens;
    int32_t num_docs;
    int32_t num_tokens;
    int32_t micro_bsz;
    int32_t seq_len;
    int32_t plen;
    int32_t rows;
    int32_t packed;
    int32_t *input_ids;
    int32_t *labels;
    int32_t *indexes;
    int32_t *cu_seqlens;
    int32_t *row_seg_ptr;
    int32_t *max_seqlen;
    int32_t *num_segs;
    int *status;
    // workspace arrays, num_docs + 1 entries each
    int32_t *doc_out;   // first output position of each document (+ sentinel)
    int32_t *doc_in;    // first input position of each document
    int32_t *doc_keep;  // tokens kept of each document
    int32_t *aligned;   // build_pack: documents d' in [1, d) that start on a row start (+ total at [num_docs])
    unsigned *ticket;            // build_pack prefix kernel: CTA order counter
    unsigned long long *look;    // build_pack prefix kernel: 2 x CTAs look-back descriptors
    int vec_out;        // 1: output pointers are 16-byte aligned
    int vec_in;         // 1: tokens is 16-byte aligned
};

size_t pack_ws_bytes(int64_t num_docs);
cudaError_t launch_pack(const PackArgs &a, int num_sms, cudaStream_t stream);

// ---------------------------------------------------------------- data steps after packing
struct UnpackArgs {
    const int32_t *input_ids, *labels;     // packed rows [rows * micro_bsz * seq_len]
    const int32_t *cu_seqlens, *row_seg_ptr;
    int32_t rows, micro_bsz, seq_len;
    int32_t *out_ids, *out_labels;         // [rows][micro_bsz][seq_len]
    int vec_out;                           // 1: outputs 16-byte aligned
};
cudaError_t launch_unpack(const UnpackArgs &a, int num_sms, cudaStream_t stream);

struct SplitArgs {
    const int32_t *src[3];
    int32_t *dst[3];
    int n_tensors;
    int32_t rows, len, sp_size, rank;
    int vec;                               // 1: 16-byte copies (aligned pointers, chunk % 4 == 0)
};
cudaError_t launch_split(const SplitArgs &a, int num_sms, cudaStream_t stream);

// ---------------------------------------------------------------- sequence-parallel padding
struct PadArgs {
    const int32_t *src;                    // [rows][len]
    int32_t *dst;                          // [rows][padded]
    int32_t rows, len, padded;
    int32_t value;                         // fill of the added positions ...
    int count;                             // ... or 1: they count 0, 1, 2, ...
    int vec;                               // 1: 16-byte stores (aligned dst)
    int vec_src;                           // 1: src is 16-byte aligned
};
cudaError_t launch_pad(const PadArgs &a, int num_sms, cudaStream_t stream);

// ---------------------------------------------------------------- rotary position embedding
struct RopeArgs {
    uint16_t *q, *k;                 // bf16 [T, Hq, d] / [T, Hkv, d], in place (either may be null)
    const int32_t *pos;              // [T] positions (>= 0)
    int32_t T, Hq, Hkv, d;
    int inverse;                     // 1: rotate by -angle
    unsigned long long freq[64];     // turns per position of pair j as 64-bit fixed point (j < d/2)
};
cudaError_t launch_rope(const RopeArgs &a, int num_sms, cudaStream_t stream);

// ---------------------------------------------------------------- masked token loss
struct LossArgs {
    const uint16_t *logits;          // bf16 [T, V]
    const int32_t *labels;           // [T], -100 = not counted
    int32_t T, V;
    float *token_loss;               // [T]
    double *loss_sum;                // [1]
    int32_t *num_tokens;             // [1]
    uint16_t *dlogits;               // bf16 [T, V] or null
    float grad_scale;
    int32_t *status;                 // [1] or null: SPD_ERR_INVALID_ARG on a label outside [0, V)
    int vec;                         // 1: rows in 16-byte chunks (V % 8 == 0, aligned pointers)
};
cudaError_t launch_loss(const LossArgs &a, int num_sms, cudaStream_t stream);

// ---------------------------------------------------------------- tile schedule
// One work unit of the tile schedule: tiles of one segment (see
// launch_schedule for the forward and backward meaning of `t`); `cost` is the
// number of (q tile, kv tile) blocks the unit computes.
struct Tile {
    int32_t seg_start;
    int32_t seg_end;
    int32_t t;      // block index inside the segment
    int32_t cost;
};

constexpr int kTile = 128;
constexpr int kSingleTile = 1 << 30;   // backward schedule: Tile.t names one kv tile, not a pair

// Upper bound of the tile count for total_tokens tokens in num_segs segments.
inline int64_t max_tiles(int64_t total_tokens, int64_t num_segs)
{
    return (total_tokens + kTile - 1) / kTile + num_segs;
}

// Builds the work list into the workspace (after the header): validates
// cu_seqlens (status SPD_ERR_BAD_SEQLENS on failure) and writes the unit count
// to ws[1]. Units are sorted by cost, largest first. order 0 (forward): unit =
// tiles per work unit (2 = a pair of consecutive q tiles), Tile.t the unit's
// first q tile. order 1 (backward): Tile.t with kSingleTile set is the single
// kv tile t & ~kSingleTile (cost n - t); otherwise the pair of kv tiles Tile.t
// and n - 1 - Tile.t of a segment of n tiles (cost n + 1), the pairs of a
// segment in consecutive slots; heads = kv heads of the launch; seg_order
// (num_segs + 1 int32 of scratch) is required.
// Work unit w of `heads` x n_tiles, the tile list of every head sorted by cost
// (largest first): the first n_long tiles of every head (the units much longer
// than a head's share of one SM) come first, interleaved across heads so the
// longest start first; then the rest, head-major (the CTAs on one head run
// together, so the tiles they share stay in L2).
__device__ __forceinline__ void unit_of(int w, int n_tiles, int n_long, int heads, int &head, int &idx)
{
    const int lead = n_long * heads;
    if (w < lead) {
        head = w % heads;
        idx = w / heads;
    } else {
        const int r = w - lead, per = n_tiles - n_long;
        head = r / per;
        idx = n_long + r % per;
    }
}

cudaError_t launch_schedule(const int32_t *cu_seqlens, int32_t num_segs, int64_t total_tokens,
                            int order, int unit, int num_sms, int heads, void *ws, int32_t *seg_order,
                            cudaStream_t stream);
size_t schedule_ws_bytes(int64_t total_tokens, int32_t num_segs);

// ---------------------------------------------------------------- attention
struct AttnFwdArgs {
    CUtensorMap tm_q, tm_k, tm_v;
    CUtensorMap tm_o;  // out as (d, Hq, T), boxes of 64 d x 32 rows
    uint16_t *out;
    float *lse;
    const Tile *tiles;
    const int32_t *tile_count;
    int32_t *work_counter;  // next work unit (zeroed by the scheduler kernel)
    const int32_t *long_count;  // long units per head (see unit_of)
    int *status;
    int32_t total_tokens;
    int32_t Hq, Hkv;
    int32_t grid_tiles;  // tile slots per head in the grid (blockIdx = head * grid_tiles + tile)
    float scale_log2;    // softmax_scale * log2(e)
    float scale;
    int debug_skip;      // test hook: the producer leaves its first Q load out
    int rope;            // 1: rotate Q and K in shared memory by their in-segment positions (RoPE)
    unsigned long long freq[64];  // RoPE turns per position of pair j as 64-bit fixed point (j < d/2)
};

cudaError_t launch_attn_fwd(const AttnFwdArgs &a, int head_dim, int64_t grid_tiles,
                            cudaStream_t stream);

struct AttnBwdArgs {
    CUtensorMap tm_q, tm_k, tm_v, tm_do;
    CUtensorMap tm_dqacc;  // fp32 dQ accumulator as [Hq * d / 32][T][32]
    CUtensorMap tm_dk, tm_dv;  // bf16 dK / dV, boxes of 64 d x 32 rows (used when store_tma)
    const uint16_t *out;
    const uint16_t *dout;
    const float *lse;
    float *dq_acc;   // fp32 [Hq][head_dim / 32][total_tokens][32] (d-blocked)
    float *delta;    // [Hq, total_tokens] fp32
    void *dq, *dk, *dv;
    int grad_fp32;
    int store_tma;   // dK / dV rows leave through TMA stores (bf16 grads, d = 128)
    const Tile *tiles;
    const int32_t *tile_count;
    int32_t *work_counter;  // next work unit (zeroed by the scheduler kernel)
    const int32_t *long_count;  // long units per head (see unit_of)
    int *status;
    int32_t total_tokens;
    int32_t Hq, Hkv;
    float scale_log2;
    float scale;
    int debug_skip;      // test hook: the producer leaves its first K / V load out
};

cudaError_t launch_attn_bwd(const AttnBwdArgs &a, int head_dim, int64_t max_units,
                            cudaStream_t stream);

}  // namespace spd
