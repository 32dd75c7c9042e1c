// C-ABI front end (include/spd.h): argument checks, workspace carving, TMA
// tensor maps, kernel launches. No allocation, no synchronisation except in
// spd_read_status.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/spd.h"
#include "internal.h"

namespace spd {
namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];
std::atomic<int> g_cc[kMaxDevices];

// SM count and compute capability (major * 10 + minor) of the current device.
int device_info(int *sms, int *cc)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SPD_ERR_CUDA;
    if (dev >= 0 && dev < kMaxDevices && g_sms[dev].load() > 0) {
        *sms = g_sms[dev].load();
        *cc = g_cc[dev].load();
        return SPD_OK;
    }
    int n = 0, ma = 0, mi = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&ma, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&mi, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return SPD_ERR_CUDA;
    if (dev >= 0 && dev < kMaxDevices) {
        g_cc[dev].store(ma * 10 + mi);
        g_sms[dev].store(n);
    }
    *sms = n;
    *cc = ma * 10 + mi;
    return SPD_OK;
}

int require_sm103(int *sms)
{
    int cc = 0;
    int rc = device_info(sms, &cc);
    if (rc != SPD_OK) return rc;
    return cc == 103 ? SPD_OK : SPD_ERR_UNSUPPORTED;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn()
{
    static std::atomic<EncodeTiled> fn{nullptr};
    EncodeTiled f = fn.load();
    if (f) return f;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
        return nullptr;
    f = reinterpret_cast<EncodeTiled>(p);
    fn.store(f);
    return f;
}

// Tensor map over a [T, H, D] bf16 array: dims (D, H, T), box (64, 1, 128),
// 128-byte swizzle; rows past T read as zero.
int make_map(CUtensorMap *m, const void *base, int64_t T, int H, int D, int box_rows = kTile)
{
    EncodeTiled f = encode_fn();
    if (!f) return SPD_ERR_CUDA;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2};
    cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SPD_OK : SPD_ERR_CUDA;
}

// Tensor map over the fp32 dQ accumulator laid out [Hq * D / 32][T][32]:
// dims (32, T, Hq * D / 32), box (32, 32, 1), 128-byte swizzle. Rows past T
// are clipped by the reduce.
int make_dqacc_map(CUtensorMap *m, float *base, int64_t T, int Hq, int D)
{
    EncodeTiled f = encode_fn();
    if (!f) return SPD_ERR_CUDA;
    cuuint64_t dims[3] = {32, static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(Hq) * (D / 32)};
    cuuint64_t strides[2] = {32 * 4, static_cast<cuuint64_t>(T) * 32 * 4};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = f(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SPD_OK : SPD_ERR_CUDA;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? SPD_OK : SPD_ERR_CUDA; }

int check_attn_shape(int64_t T, int32_t num_segs, int Hq, int Hkv, int D)
{
    if (D != 64 && D != 128) return SPD_ERR_UNSUPPORTED;
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return SPD_ERR_INVALID_ARG;
    if (T < 0 || T > kMaxPositions || num_segs < 0 || num_segs > T) return SPD_ERR_INVALID_ARG;
    if ((T > 0) != (num_segs > 0)) return SPD_ERR_INVALID_ARG;
    if (static_cast<int64_t>(Hq) * T > kMaxPositions) return SPD_ERR_INVALID_ARG;
    return SPD_OK;
}

// backward workspace: schedule, the scheduler's segment order, D, dQ accumulator
size_t bwd_order_off(int64_t T, int32_t num_segs) { return align_up(schedule_ws_bytes(T, num_segs), 256); }
size_t bwd_delta_off(int64_t T, int32_t num_segs)
{
    return bwd_order_off(T, num_segs) + align_up(sizeof(int32_t) * static_cast<size_t>(num_segs + 1), 256);
}
size_t bwd_acc_off(int64_t T, int32_t num_segs, int Hq)
{
    return bwd_delta_off(T, num_segs) + align_up(sizeof(float) * static_cast<size_t>(Hq) * T, 256);
}

int clear_status(void *ws, cudaStream_t stream)
{
    return cuda_rc(cudaMemsetAsync(ws, 0, sizeof(int), stream));
}

}  // namespace

ProfileHook &profile_hook()
{
    static thread_local ProfileHook hook;
    return hook;
}

// The test hook of spd_debug_skip_arrive, per host thread.
int &debug_skip_slot()
{
    static thread_local int which = SPD_DEBUG_SKIP_NONE;
    return which;
}

int take_debug_skip(int which)
{
    int &s = debug_skip_slot();
    if (s != which) return 0;
    s = SPD_DEBUG_SKIP_NONE;
    return 1;
}

}  // namespace spd

using namespace spd;

// The forward call with or without the in-kernel RoPE rotation of q and k.
static int attn_fwd_impl(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int32_t *cu_seqlens,
                         int32_t num_segs, int64_t total_tokens, int Hq, int Hkv, int head_dim,
                         float softmax_scale, int rope, float rope_theta, uint16_t *out, float *lse, void *ws,
                         size_t ws_bytes, spd_stream_t stream)
{
    int rc = check_attn_shape(total_tokens, num_segs, Hq, Hkv, head_dim);
    if (rc != SPD_OK) return rc;
    if (!ws || !aligned(ws, 256)) return SPD_ERR_WORKSPACE;
    if (ws_bytes < spd_attn_workspace_size(total_tokens, num_segs, Hq, Hkv, head_dim, 0)) return SPD_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (total_tokens == 0) return clear_status(ws, s);
    if (!q || !k || !v || !out || !lse || !cu_seqlens) return SPD_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(lse, 4) ||
        !aligned(cu_seqlens, 4))
        return SPD_ERR_INVALID_ARG;
    int sms = 0;
    rc = require_sm103(&sms);
    if (rc != SPD_OK) return rc;
    if (!(softmax_scale > 0.f)) softmax_scale = 1.0f / std::sqrt(static_cast<float>(head_dim));

    rc = cuda_rc(launch_schedule(cu_seqlens, num_segs, total_tokens, 0, 2, sms, Hkv, ws, nullptr, s));
    if (rc != SPD_OK) return rc;
    AttnFwdArgs a = {};
    if ((rc = make_map(&a.tm_q, q, total_tokens, Hq, head_dim)) != SPD_OK) return rc;
    if ((rc = make_map(&a.tm_k, k, total_tokens, Hkv, head_dim)) != SPD_OK) return rc;
    if ((rc = make_map(&a.tm_o, out, total_tokens, Hq, head_dim, 32)) != SPD_OK) return rc;
    if ((rc = make_map(&a.tm_v, v, total_tokens, Hkv, head_dim)) != SPD_OK) return rc;
    char *base = static_cast<char *>(ws);
    a.out = out;
    a.lse = lse;
    a.tiles = reinterpret_cast<const Tile *>(base + kWsHeader);
    a.tile_count = reinterpret_cast<const int32_t *>(base) + 1;
    a.work_counter = reinterpret_cast<int32_t *>(base) + 2;
    a.long_count = reinterpret_cast<const int32_t *>(base) + 3;
    a.status = reinterpret_cast<int *>(base);
    a.total_tokens = static_cast<int32_t>(total_tokens);
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.scale = softmax_scale;
    a.scale_log2 = softmax_scale * 1.4426950408889634f;
    a.debug_skip = take_debug_skip(SPD_DEBUG_SKIP_FWD_Q);
    a.rope = rope;
    if (rope) {
        const double theta = rope_theta > 0.f ? static_cast<double>(rope_theta) : 10000.0;
        for (int j = 0; j < head_dim / 2; ++j) {
            // turns per position, theta_j / (2 pi) < 1/6, as 64-bit fixed point
            const double turns = std::pow(theta, -2.0 * j / head_dim) / (2.0 * 3.141592653589793238462643);
            a.freq[j] = static_cast<unsigned long long>(std::ldexp(turns, 64));
        }
    }
    return cuda_rc(launch_attn_fwd(a, head_dim, (total_tokens + 2 * kTile - 1) / (2 * kTile) + num_segs, s));
}

extern "C" {

const char *spd_status_string(int s)
{
    switch (s) {
    case SPD_OK: return "ok";
    case SPD_ERR_INVALID_ARG: return "invalid argument";
    case SPD_ERR_UNSUPPORTED: return "unsupported (head_dim or GPU)";
    case SPD_ERR_CUDA: return "CUDA error";
    case SPD_ERR_BAD_SEQLENS: return "cu_seqlens is not 0 = c0 < c1 < ... = total_tokens";
    case SPD_ERR_DEVICE_TIMEOUT: return "a bounded device wait ran out";
    case SPD_ERR_WORKSPACE: return "workspace too small or misaligned";
    case SPD_ERR_BAD_DOCS: return "a document length <= 0 or lengths do not sum to num_tokens";
    case SPD_ERR_TOO_LARGE: return "problem exceeds the fixed scratch of the no-allocation entry point";
    default: return "unknown status";
    }
}

int spd_version(void) { return 100; }

int spd_debug_skip_arrive(int which)
{
    if (which < SPD_DEBUG_SKIP_NONE || which > SPD_DEBUG_SKIP_BWD_KV) return SPD_ERR_INVALID_ARG;
    spd::debug_skip_slot() = which;
    return SPD_OK;
}

int spd_set_profile_events(void *begin_event, void *end_event, int kernel)
{
    if (kernel < SPD_PROFILE_NONE || kernel > SPD_PROFILE_PAD) return SPD_ERR_INVALID_ARG;
    ProfileHook &h = profile_hook();
    h.begin = static_cast<cudaEvent_t>(begin_event);
    h.end = static_cast<cudaEvent_t>(end_event);
    h.which = (begin_event && end_event) ? kernel : kProfNone;
    return SPD_OK;
}

int spd_read_status(const void *ws, spd_stream_t stream, int *device_status)
{
    if (!ws || !device_status) return SPD_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return SPD_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SPD_ERR_CUDA;
    *device_status = v;
    return SPD_OK;
}

int spd_attn_read_schedule(const void *ws, spd_stream_t stream, int32_t *num_units, int32_t *units,
                           int64_t capacity)
{
    if (!ws || !num_units || capacity < 0 || (capacity > 0 && !units)) return SPD_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int32_t n = 0;
    if (cudaMemcpyAsync(&n, static_cast<const int32_t *>(ws) + 1, sizeof(int32_t), cudaMemcpyDeviceToHost, s) !=
        cudaSuccess)
        return SPD_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SPD_ERR_CUDA;
    *num_units = n;
    const int64_t m = n < capacity ? n : capacity;
    if (m > 0) {
        static_assert(sizeof(Tile) == 4 * sizeof(int32_t), "Tile is four int32 words");
        if (cudaMemcpyAsync(units, static_cast<const char *>(ws) + kWsHeader, sizeof(Tile) * static_cast<size_t>(m),
                            cudaMemcpyDeviceToHost, s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return SPD_ERR_CUDA;
    }
    return SPD_OK;
}

int spd_pack_rows(int64_t num_docs, int64_t num_tokens, int micro_bsz, int seq_len, int use_packed_dataset,
                  int64_t *rows, int64_t *max_segs)
{
    if (!rows || !max_segs) return SPD_ERR_INVALID_ARG;
    if (micro_bsz <= 0 || seq_len <= 0 || num_docs < 0 || num_tokens < 0) return SPD_ERR_INVALID_ARG;
    if (num_docs > 0x7fffffffLL || num_tokens > 0x7fffffffLL) return SPD_ERR_INVALID_ARG;
    if ((num_docs == 0) != (num_tokens == 0)) return SPD_ERR_INVALID_ARG;
    const int64_t plen = static_cast<int64_t>(micro_bsz) * seq_len;
    const int64_t r = use_packed_dataset ? (num_tokens + plen - 1) / plen : (num_docs + micro_bsz - 1) / micro_bsz;
    if (r * plen > kMaxPositions) return SPD_ERR_INVALID_ARG;
    *rows = r;
    *max_segs = num_docs + 2 * r;
    if (*max_segs > 0x7fffffffLL) return SPD_ERR_INVALID_ARG;
    return SPD_OK;
}

int spd_pack_num_segs(const int32_t *doc_lens, int64_t num_docs, int micro_bsz, int seq_len, int use_packed_dataset,
                      int64_t *num_segs)
{
    if (!num_segs || (num_docs > 0 && !doc_lens)) return SPD_ERR_INVALID_ARG;
    if (micro_bsz <= 0 || seq_len <= 0 || num_docs < 0 || num_docs > 0x7fffffffLL) return SPD_ERR_INVALID_ARG;
    const int64_t plen = static_cast<int64_t>(micro_bsz) * seq_len;
    int64_t segs = 0;
    if (use_packed_dataset) {
        // one segment per row a document spans, then the padding tail of the last row
        int64_t start = 0;
        for (int64_t d = 0; d < num_docs; ++d) {
            if (doc_lens[d] <= 0) return SPD_ERR_INVALID_ARG;
            segs += (start + doc_lens[d] - 1) / plen - start / plen + 1;
            start += doc_lens[d];
        }
        if (start % plen != 0) ++segs;
    } else {
        // each row: its (at most micro_bsz) documents cut to seq_len, then the padding tail
        for (int64_t first = 0; first < num_docs; first += micro_bsz) {
            int64_t kept = 0;
            for (int64_t d = first; d < num_docs && d < first + micro_bsz; ++d) {
                if (doc_lens[d] <= 0) return SPD_ERR_INVALID_ARG;
                kept += doc_lens[d] < seq_len ? doc_lens[d] : seq_len;
                ++segs;
            }
            if (kept < plen) ++segs;
        }
    }
    *num_segs = segs;
    return SPD_OK;
}

size_t spd_pack_workspace_size(int64_t num_docs)
{
    if (num_docs < 0) return 0;
    return pack_ws_bytes(num_docs);
}

int spd_pack_tokens(const int32_t *tokens, const int32_t *doc_lens, int64_t num_docs, int64_t num_tokens,
                    int micro_bsz, int seq_len, int use_packed_dataset, int32_t *input_ids, int32_t *labels,
                    int32_t *indexes, int32_t *cu_seqlens, int32_t *row_seg_ptr, int32_t *max_seqlen,
                    int32_t *num_segs, void *ws, size_t ws_bytes, spd_stream_t stream)
{
    int64_t rows = 0, max_segs = 0;
    int rc = spd_pack_rows(num_docs, num_tokens, micro_bsz, seq_len, use_packed_dataset, &rows, &max_segs);
    if (rc != SPD_OK) return rc;
    if (!ws || !aligned(ws, 256)) return SPD_ERR_WORKSPACE;
    if (ws_bytes < spd_pack_workspace_size(num_docs)) return SPD_ERR_WORKSPACE;
    if (!cu_seqlens || !row_seg_ptr || !num_segs) return SPD_ERR_INVALID_ARG;
    if (rows > 0 && (!input_ids || !labels || !indexes || !max_seqlen)) return SPD_ERR_INVALID_ARG;
    if (num_docs > 0 && (!tokens || !doc_lens)) return SPD_ERR_INVALID_ARG;
    const void *ptrs[] = {tokens, doc_lens, input_ids, labels, indexes, cu_seqlens, row_seg_ptr, max_seqlen, num_segs};
    for (const void *p : ptrs)
        if (p && !aligned(p, 4)) return SPD_ERR_INVALID_ARG;
    int sms = 0;
    rc = require_sm103(&sms);
    if (rc != SPD_OK) return rc;

    PackArgs a = {};
    a.tokens = tokens;
    a.doc_lens = doc_lens;
    a.num_docs = static_cast<int32_t>(num_docs);
    a.num_tokens = static_cast<int32_t>(num_tokens);
    a.micro_bsz = micro_bsz;
    a.seq_len = seq_len;
    a.plen = micro_bsz * seq_len;
    a.rows = static_cast<int32_t>(rows);
    a.packed = use_packed_dataset ? 1 : 0;
    a.input_ids = input_ids;
    a.labels = labels;
    a.indexes = indexes;
    a.cu_seqlens = cu_seqlens;
    a.row_seg_ptr = row_seg_ptr;
    a.max_seqlen = max_seqlen;
    a.num_segs = num_segs;
    a.status = static_cast<int *>(ws);
    a.vec_out = aligned(input_ids, 16) && aligned(labels, 16) && aligned(indexes, 16);
    a.vec_in = aligned(tokens, 16);
    return cuda_rc(launch_pack(a, sms, reinterpret_cast<cudaStream_t>(stream)));
}

int spd_unpack_data(const int32_t *input_ids, const int32_t *labels, const int32_t *cu_seqlens,
                    const int32_t *row_seg_ptr, int64_t rows, int micro_bsz, int seq_len, int32_t *out_ids,
                    int32_t *out_labels, spd_stream_t stream)
{
    if (micro_bsz < 1 || seq_len < 1 || rows < 0) return SPD_ERR_INVALID_ARG;
    const int64_t total = rows * static_cast<int64_t>(micro_bsz) * seq_len;
    if (total > kMaxPositions) return SPD_ERR_INVALID_ARG;
    if (rows == 0) return SPD_OK;
    const void *ptrs[] = {input_ids, labels, cu_seqlens, row_seg_ptr, out_ids, out_labels};
    for (const void *p : ptrs)
        if (!p || !aligned(p, 4)) return SPD_ERR_INVALID_ARG;
    int sms = 0;
    int rc = require_sm103(&sms);
    if (rc != SPD_OK) return rc;
    UnpackArgs a = {};
    a.input_ids = input_ids;
    a.labels = labels;
    a.cu_seqlens = cu_seqlens;
    a.row_seg_ptr = row_seg_ptr;
    a.rows = static_cast<int32_t>(rows);
    a.micro_bsz = micro_bsz;
    a.seq_len = seq_len;
    a.out_ids = out_ids;
    a.out_labels = out_labels;
    a.vec_out = aligned(out_ids, 16) && aligned(out_labels, 16);
    return cuda_rc(launch_unpack(a, sms, reinterpret_cast<cudaStream_t>(stream)));
}

int spd_pad_for_sequence_parallel(const int32_t *src, int32_t *dst, int64_t rows, int64_t len, int sp_size,
                                  int32_t pad_value, int count_positions, spd_stream_t stream)
{
    if (sp_size < 1 || rows < 0 || len < 0 || len > 0x7fffffffLL) return SPD_ERR_INVALID_ARG;
    const int64_t padded = (len + sp_size - 1) / sp_size * sp_size;
    if (rows * padded > kMaxPositions) return SPD_ERR_INVALID_ARG;
    if (rows == 0 || padded == 0) return SPD_OK;
    if (!dst || !aligned(dst, 4) || (len > 0 && (!src || !aligned(src, 4)))) return SPD_ERR_INVALID_ARG;
    int sms = 0;
    int rc = require_sm103(&sms);
    if (rc != SPD_OK) return rc;
    PadArgs a = {};
    a.src = src;
    a.dst = dst;
    a.rows = static_cast<int32_t>(rows);
    a.len = static_cast<int32_t>(len);
    a.padded = static_cast<int32_t>(padded);
    a.value = pad_value;
    a.count = count_positions ? 1 : 0;
    a.vec = aligned(dst, 16) ? 1 : 0;
    a.vec_src = aligned(src, 16) ? 1 : 0;
    return cuda_rc(launch_pad(a, sms, reinterpret_cast<cudaStream_t>(stream)));
}

int spd_split_sequence_parallel(const int32_t *src0, const int32_t *src1, const int32_t *src2, int64_t rows,
                                int64_t len, int sp_size, int rank, int32_t *dst0, int32_t *dst1, int32_t *dst2,
                                spd_stream_t stream)
{
    if (sp_size < 1 || rank < 0 || rank >= sp_size || rows < 0 || len < 0) return SPD_ERR_INVALID_ARG;
    if (len % sp_size != 0 || rows * len > kMaxPositions) return SPD_ERR_INVALID_ARG;
    const int32_t *src[3] = {src0, src1, src2};
    int32_t *dst[3] = {dst0, dst1, dst2};
    SplitArgs a = {};
    bool vec = (len / sp_size) % 4 == 0;
    for (int i = 0; i < 3; ++i) {
        if ((src[i] == nullptr) != (dst[i] == nullptr)) return SPD_ERR_INVALID_ARG;
        if (!src[i]) continue;
        if (!aligned(src[i], 4) || !aligned(dst[i], 4)) return SPD_ERR_INVALID_ARG;
        vec = vec && aligned(src[i], 16) && aligned(dst[i], 16);
        a.src[a.n_tensors] = src[i];
        a.dst[a.n_tensors] = dst[i];
        ++a.n_tensors;
    }
    if (rows == 0 || len == 0 || a.n_tensors == 0) return SPD_OK;
    int sms = 0;
    int rc = require_sm103(&sms);
    if (rc != SPD_OK) return rc;
    a.rows = static_cast<int32_t>(rows);
    a.len = static_cast<int32_t>(len);
    a.sp_size = sp_size;
    a.rank = rank;
    a.vec = vec ? 1 : 0;
    return cuda_rc(launch_split(a, sms, reinterpret_cast<cudaStream_t>(stream)));
}

int spd_rope(uint16_t *q, uint16_t *k, const int32_t *positions, int64_t total_tokens, int Hq, int Hkv,
             int head_dim, float rope_theta, int inverse, spd_stream_t stream)
{
    if (head_dim != 64 && head_dim != 128) return SPD_ERR_UNSUPPORTED;
    if (total_tokens < 0 || total_tokens > kMaxPositions || Hq < 0 || Hkv < 0) return SPD_ERR_INVALID_ARG;
    if ((q && Hq == 0) || (k && Hkv == 0)) return SPD_ERR_INVALID_ARG;
    if (static_cast<int64_t>(Hq > Hkv ? Hq : Hkv) * total_tokens * head_dim > (1LL << 40)) return SPD_ERR_INVALID_ARG;
    if ((q && !aligned(q, 16)) || (k && !aligned(k, 16))) return SPD_ERR_INVALID_ARG;
    if (total_tokens == 0 || (!q && !k)) return SPD_OK;
    if (!positions || !aligned(positions, 4)) return SPD_ERR_INVALID_ARG;
    int sms = 0;
    int rc = require_sm103(&sms);
    if (rc != SPD_OK) return rc;
    RopeArgs a = {};
    a.q = q;
    a.k = k;
    a.pos = positions;
    a.T = static_cast<int32_t>(total_tokens);
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.d = head_dim;
    a.inverse = inverse ? 1 : 0;
    const double base = rope_theta > 0.f ? static_cast<double>(rope_theta) : 10000.0;
    for (int j = 0; j < head_dim / 2; ++j) {
        // turns per position, theta_j / (2 pi) < 1/6, as 64-bit fixed point
        const double turns = std::pow(base, -2.0 * j / head_dim) / (2.0 * 3.141592653589793238462643);
        a.freq[j] = static_cast<unsigned long long>(std::ldexp(turns, 64));
    }
    return cuda_rc(launch_rope(a, sms, reinterpret_cast<cudaStream_t>(stream)));
}

int spd_masked_token_loss(const uint16_t *logits, const int32_t *labels, int64_t T, int64_t V, float *token_loss,
                          double *loss_sum, int32_t *num_tokens, uint16_t *dlogits, float grad_scale,
                          int32_t *device_status, spd_stream_t stream)
{
    if (T < 0 || T > 0x7fffffffLL || V < 1 || V > 0x7fffffffLL) return SPD_ERR_INVALID_ARG;
    if (!loss_sum || !num_tokens || !aligned(loss_sum, 8) || !aligned(num_tokens, 4)) return SPD_ERR_INVALID_ARG;
    if (T > 0 && (!logits || !labels || !token_loss)) return SPD_ERR_INVALID_ARG;
    const void *p4[] = {labels, token_loss, device_status};
    for (const void *p : p4)
        if (p && !aligned(p, 4)) return SPD_ERR_INVALID_ARG;
    if ((logits && !aligned(logits, 2)) || (dlogits && !aligned(dlogits, 2))) return SPD_ERR_INVALID_ARG;
    int sms = 0;
    int rc = require_sm103(&sms);
    if (rc != SPD_OK) return rc;
    LossArgs a = {};
    a.logits = logits;
    a.labels = labels;
    a.T = static_cast<int32_t>(T);
    a.V = static_cast<int32_t>(V);
    a.token_loss = token_loss;
    a.loss_sum = loss_sum;
    a.num_tokens = num_tokens;
    a.dlogits = dlogits;
    a.grad_scale = grad_scale;
    a.status = device_status;
    a.vec = V % 8 == 0 && aligned(logits, 16) && (!dlogits || aligned(dlogits, 16));
    return cuda_rc(launch_loss(a, sms, reinterpret_cast<cudaStream_t>(stream)));
}

size_t spd_attn_workspace_size(int64_t total_tokens, int32_t num_segs, int Hq, int Hkv, int head_dim, int bwd)
{
    if (check_attn_shape(total_tokens, num_segs, Hq, Hkv, head_dim) != SPD_OK) return 0;
    if (!bwd) return schedule_ws_bytes(total_tokens, num_segs);
    return bwd_acc_off(total_tokens, num_segs, Hq) +
           align_up(sizeof(float) * static_cast<size_t>(Hq) * total_tokens * head_dim, 256);
}

int spd_varlen_attn_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int32_t *cu_seqlens,
                        int32_t num_segs, int64_t total_tokens, int32_t max_seqlen, int Hq, int Hkv, int head_dim,
                        float softmax_scale, uint16_t *out, float *lse, void *ws, size_t ws_bytes,
                        spd_stream_t stream)
{
    (void)max_seqlen;
    return attn_fwd_impl(q, k, v, cu_seqlens, num_segs, total_tokens, Hq, Hkv, head_dim, softmax_scale, 0, 0.f,
                         out, lse, ws, ws_bytes, stream);
}

int spd_varlen_attn_fwd_rope(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int32_t *cu_seqlens,
                             int32_t num_segs, int64_t total_tokens, int32_t max_seqlen, int Hq, int Hkv,
                             int head_dim, float softmax_scale, float rope_theta, uint16_t *out, float *lse,
                             void *ws, size_t ws_bytes, spd_stream_t stream)
{
    (void)max_seqlen;
    return attn_fwd_impl(q, k, v, cu_seqlens, num_segs, total_tokens, Hq, Hkv, head_dim, softmax_scale, 1,
                         rope_theta, out, lse, ws, ws_bytes, stream);
}

int spd_varlen_attn_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *out,
                        const uint16_t *dout, const float *lse, const int32_t *cu_seqlens, int32_t num_segs,
                        int64_t total_tokens, int32_t max_seqlen, int Hq, int Hkv, int head_dim,
                        float softmax_scale, int grad_dtype, void *dq, void *dk, void *dv, void *ws,
                        size_t ws_bytes, spd_stream_t stream)
{
    (void)max_seqlen;
    int rc = check_attn_shape(total_tokens, num_segs, Hq, Hkv, head_dim);
    if (rc != SPD_OK) return rc;
    if (grad_dtype != 0 && grad_dtype != 1) return SPD_ERR_INVALID_ARG;
    if (!ws || !aligned(ws, 256)) return SPD_ERR_WORKSPACE;
    if (ws_bytes < spd_attn_workspace_size(total_tokens, num_segs, Hq, Hkv, head_dim, 1)) return SPD_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (total_tokens == 0) return clear_status(ws, s);
    if (!q || !k || !v || !out || !dout || !lse || !cu_seqlens || !dq || !dk || !dv) return SPD_ERR_INVALID_ARG;
    const void *p16[] = {q, k, v, out, dout, dq, dk, dv};
    for (const void *p : p16)
        if (!aligned(p, 16)) return SPD_ERR_INVALID_ARG;
    if (!aligned(lse, 4) || !aligned(cu_seqlens, 4)) return SPD_ERR_INVALID_ARG;
    int sms = 0;
    rc = require_sm103(&sms);
    if (rc != SPD_OK) return rc;
    if (!(softmax_scale > 0.f)) softmax_scale = 1.0f / std::sqrt(static_cast<float>(head_dim));

    rc = cuda_rc(launch_schedule(cu_seqlens, num_segs, total_tokens, 1, 1, sms, Hkv, ws,
                                 reinterpret_cast<int32_t *>(static_cast<char *>(ws) +
                                                             bwd_order_off(total_tokens, num_segs)),
                                 s));
    if (rc != SPD_OK) return rc;
    AttnBwdArgs a = {};
    if ((rc = make_map(&a.tm_q, q, total_tokens, Hq, head_dim)) != SPD_OK) return rc;
    if ((rc = make_map(&a.tm_k, k, total_tokens, Hkv, head_dim)) != SPD_OK) return rc;
    if ((rc = make_map(&a.tm_v, v, total_tokens, Hkv, head_dim)) != SPD_OK) return rc;
    if ((rc = make_map(&a.tm_do, dout, total_tokens, Hq, head_dim)) != SPD_OK) return rc;
    char *base = static_cast<char *>(ws);
    a.out = out;
    a.dout = dout;
    a.lse = lse;
    a.delta = reinterpret_cast<float *>(base + bwd_delta_off(total_tokens, num_segs));
    a.dq_acc = reinterpret_cast<float *>(base + bwd_acc_off(total_tokens, num_segs, Hq));
    if ((rc = make_dqacc_map(&a.tm_dqacc, a.dq_acc, total_tokens, Hq, head_dim)) != SPD_OK) return rc;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.grad_fp32 = grad_dtype;
    a.store_tma = grad_dtype == 0 && head_dim == 128;
    if (a.store_tma) {
        if ((rc = make_map(&a.tm_dk, dk, total_tokens, Hkv, head_dim, 32)) != SPD_OK) return rc;
        if ((rc = make_map(&a.tm_dv, dv, total_tokens, Hkv, head_dim, 32)) != SPD_OK) return rc;
    }
    a.tiles = reinterpret_cast<const Tile *>(base + kWsHeader);
    a.tile_count = reinterpret_cast<const int32_t *>(base) + 1;
    a.work_counter = reinterpret_cast<int32_t *>(base) + 2;
    a.long_count = reinterpret_cast<const int32_t *>(base) + 3;
    a.status = reinterpret_cast<int *>(base);
    a.total_tokens = static_cast<int32_t>(total_tokens);
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.scale = softmax_scale;
    a.scale_log2 = softmax_scale * 1.4426950408889634f;
    a.debug_skip = take_debug_skip(SPD_DEBUG_SKIP_BWD_KV);
    return cuda_rc(launch_attn_bwd(a, head_dim, max_tiles(total_tokens, num_segs), s));
}

}  // extern "C"
