// Packing kernels: documents -> packed rows (input_ids, labels, indexes) and
// the segment fields (cu_seqlens, row_seg_ptr, max_seqlen, num_segs).
//
// Rules: InternEvo page "Data loading and flow", section "Dataloader loading
// data" (build_pack with use_packed_dataset = True, build_unpack with False;
// pad id 0, label = next token of the same document, -100 at a document's last
// token and on padding) and section "Fetching data from the Dataloader"
// (cu_seqlens: segment boundaries of a row, the padding tail being its own
// segment; indexes: position inside the current segment).
//
// build_pack with at most 1024 documents and 512 rows runs as one fused
// launch (pack_fused_kernel), build_unpack with at most 1024 documents as
// another (unpack_fused_kernel). Otherwise, two launches on one stream:
//   build_pack:
//     pack_prefix_kernel  prefix sums of the document lengths (document starts)
//                         and of the "starts on a row start" flags, 4096
//                         documents per CTA, CTAs chained by a decoupled
//                         look-back; num_segs, the last row's end; zeroes
//                         max_seqlen. Work ~ num_docs.
//     pack_packed_stream_kernel  all SMs: the token stream (input_ids, labels,
//                         indexes in 16-byte stores) and the segment fields of
//                         the boundaries inside each CTA's chunk (cu_seqlens,
//                         row_seg_ptr, max_seqlen). Work ~ output positions.
//   build_unpack:
//     pack_scan_kernel    one CTA: prefix sums, the document -> output position
//                         map and every segment field.
//     unpack_stream_kernel  all SMs: the token stream.
// The stream kernels are programmatic dependent launches: in build_pack mode
// the stream kernel loads its tokens and stores input_ids (which needs no
// document boundaries) while the prefix kernel runs, then waits for its
// results before labels, indexes and the segment fields.
#include "internal.h"
#include "ptx.cuh"

namespace spd {
namespace {

constexpr int kScanThreads = 1024;
constexpr int kScanItems = 4;  // documents per thread per pass
constexpr int kStreamThreads = 256;
constexpr int kStreamIters = 4;
constexpr int kChunk = kStreamThreads * 4 * kStreamIters;  // positions per CTA

// Exclusive scan of one value per thread over a 1024-thread block.
// Returns the exclusive prefix; *total gets the block sum. `sh` holds 33 slots.
__device__ long long block_excl_scan(long long v, long long *total, long long *sh)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[warp] = x;
    __syncthreads();
    if (warp == 0) {
        long long w = sh[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            long long y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        sh[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    long long warp_excl = warp ? sh[warp - 1] : 0;
    *total = sh[31];
    __syncthreads();  // sh is reused by the next call
    return warp_excl + x - v;
}

// ---------------------------------------------------------------- build_pack prefix
constexpr int kPrefixDocs = kScanThreads * kScanItems;   // documents per prefix CTA

// Decoupled look-back over the prefix CTAs, by one warp of each: publish this
// CTA's aggregate, then read the predecessors' published words 32 at a time
// (lane l reads CTA bid - 1 - l - 32 k), adding up aggregates back to the
// nearest inclusive prefix; publish the inclusive prefix. A CTA only waits on
// CTAs that took their order ticket earlier, which are running, so the chain
// ends; the wait is bounded all the same (status SPD_ERR_DEVICE_TIMEOUT).
// Values are clamped below 2^40 (valid inputs stay below 2^31). Returns the
// exclusive prefix in every lane.
__device__ long long lookback_excl(unsigned long long *look, int bid, long long agg, int *status)
{
    constexpr unsigned long long kAgg = 1ull << 62, kInc = 2ull << 62, kVal = (1ull << 62) - 1;
    constexpr long long kCap = 1LL << 40;
    const int lane = threadIdx.x & 31;
    const unsigned long long v = static_cast<unsigned long long>(agg < kCap ? agg : kCap);
    if (bid == 0) {
        if (lane == 0) st_release_u64(look, kInc | v);
        return 0;
    }
    if (lane == 0) st_release_u64(look + bid, kAgg | v);
    long long excl = 0;
    int base = bid - 1;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        const int j = base - lane;
        // before CTA 0 nothing is added: read as an inclusive zero
        const unsigned long long w = j >= 0 ? ld_acquire_u64(look + j) : kInc;
        const unsigned long long state = w >> 62;
        const unsigned inc = __ballot_sync(0xffffffffu, state == 2);
        const unsigned empty = __ballot_sync(0xffffffffu, state == 0);
        const int first = inc ? __ffs(inc) - 1 : 32;   // nearest inclusive prefix in the window
        const unsigned needed = first == 32 ? 0xffffffffu : (first == 31 ? 0xffffffffu : (2u << first) - 1u);
        if (empty & needed) {                          // a predecessor has not published yet
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                if (lane == 0) set_status(status, kErrTimeout);
                break;
            }
            continue;
        }
        long long x = lane <= first ? static_cast<long long>(w & kVal) : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        excl += x;
        if (first < 32) break;
        base -= 32;
    }
    const long long incl = excl + static_cast<long long>(v);
    if (lane == 0) st_release_u64(look + bid, kInc | static_cast<unsigned long long>(incl < kCap ? incl : kCap));
    return excl;
}

__global__ void __launch_bounds__(kScanThreads) pack_prefix_kernel(PackArgs a, int nb)
{
    // Launched as a programmatic dependent of whatever precedes it on the
    // stream: it waits for that grid (and its memory) first, then lets the
    // stream kernel start, which may load its tokens and store input_ids
    // meanwhile.
    pdl_wait();
    pdl_launch_dependents();
    __shared__ long long sh[33];
    __shared__ long long s_excl[2];   // this CTA's exclusive prefix: document starts, aligned starts
    __shared__ int s_bid, bad_s;
    const int tid = threadIdx.x;
    const int nd = a.num_docs, rows = a.rows;
    const long long plen = a.plen, total = a.num_tokens;
    if (tid == 0) {
        if (nb == 1) *a.status = 0;   // several CTAs: the host cleared it
        s_bid = nb > 1 ? static_cast<int>(atomicAdd(a.ticket, 1u)) : 0;
        bad_s = 0;
    }
    __syncthreads();
    const int bid = s_bid;
    for (long long r = static_cast<long long>(bid) * kScanThreads + tid; r < rows;
         r += static_cast<long long>(nb) * kScanThreads)
        a.max_seqlen[r] = 0;

    // document starts
    const int d0 = bid * kPrefixDocs + tid * kScanItems;
    int len[kScanItems];
    long long sum = 0;
    bool bad = false;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        const int d = d0 + k;
        len[k] = d < nd ? a.doc_lens[d] : 0;
        if (d < nd && len[k] <= 0) bad = true;
        if (len[k] < 0) len[k] = 0;
        sum += len[k];
    }
    long long agg;
    const long long e = block_excl_scan(sum, &agg, sh);
    if (nb > 1) {   // one CTA: nothing to chain
        if (tid < 32) {
            const long long x = lookback_excl(a.look, bid, agg, a.status);
            if (tid == 0) s_excl[0] = x;
        }
    } else if (tid == 0) {
        s_excl[0] = 0;
    }
    __syncthreads();
    long long start[kScanItems];
    long long run = s_excl[0] + e;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        start[k] = run;
        run += len[k];
    }
    // documents (other than the first) that start on a row start: the same
    // boundary as the row start, counted so the boundary ranks stay exact
    int flag[kScanItems], fsum = 0;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        const int d = d0 + k;
        // valid starts are below 2^31 (larger ones fail the length check below)
        flag[k] = (d >= 1 && d < nd && static_cast<unsigned>(start[k]) % static_cast<unsigned>(plen) == 0) ? 1 : 0;
        fsum += flag[k];
    }
    long long fagg;
    const long long fe = block_excl_scan(fsum, &fagg, sh);
    if (nb > 1) {
        if (tid < 32) {
            const long long x = lookback_excl(a.look + nb, bid, fagg, a.status);
            if (tid == 0) s_excl[1] = x;
        }
    } else if (tid == 0) {
        s_excl[1] = 0;
    }
    __syncthreads();
    long long frun = s_excl[1] + fe;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        const int d = d0 + k;
        if (d < nd) {
            a.doc_out[d] = static_cast<int32_t>(start[k]);
            a.aligned[d] = static_cast<int32_t>(frun);
        }
        frun += flag[k];
    }
    if (bad) atomicOr(&bad_s, 1);
    __syncthreads();
    if (tid == 0) {
        bool fail = bad_s != 0;
        if (bid == nb - 1) {
            // The CTA holding the last document knows the totals: the end of the
            // last document, the segment count (rows, plus one per document start
            // not on a row start, plus the padding tail), the last row's end.
            const long long tot_len = s_excl[0] + agg, tot_al = s_excl[1] + fagg;
            if (tot_len != total) fail = true;
            if (!fail) {
                const long long pad = total % plen != 0;
                // no documents: no rows and no segments (cu_seqlens = {0})
                const long long num_segs = rows == 0 ? 0 : rows + nd - 1 - tot_al + pad;
                a.doc_out[nd] = static_cast<int32_t>(total);
                a.aligned[nd] = static_cast<int32_t>(tot_al);
                *a.num_segs = static_cast<int32_t>(num_segs);
                a.row_seg_ptr[rows] = static_cast<int32_t>(num_segs);
                a.cu_seqlens[num_segs] = static_cast<int32_t>(rows * plen);
            }
        }
        if (fail) {
            set_status(a.status, kErrBadDocs);
            *a.num_segs = 0;
        }
    }
}

// First index d in [lo, hi) with a[d] >= x (hi if none); a strictly increasing.
__device__ __forceinline__ int lower_bound(const int32_t *a, int lo, int hi, long long x)
{
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (a[mid] < x) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// Largest d in [lo, hi) with a[d] <= x; assumes a[lo] <= x.
__device__ __forceinline__ int last_le(const int32_t *a, int lo, int hi, long long x)
{
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (a[mid] <= x) lo = mid;
        else hi = mid;
    }
    return lo;
}

__global__ void __launch_bounds__(kScanThreads) pack_scan_kernel(PackArgs a, int32_t *aux)
{
    pdl_launch_dependents();
    __shared__ long long sh[33];
    __shared__ int bad_s;
    const int tid = threadIdx.x;
    const int nd = a.num_docs;
    const long long plen = a.plen;
    if (tid == 0) {
        *a.status = 0;
        bad_s = 0;
    }
    for (int r = tid; r < a.rows; r += kScanThreads) a.max_seqlen[r] = 0;

    // Pass 1: exclusive prefix sums of the raw lengths (input offsets) and of
    // the kept lengths (output offsets before the row split).
    long long carry_raw = 0, carry_keep = 0;
    bool bad = false;
    for (int base = 0; base < nd; base += kScanThreads * kScanItems) {
        int len[kScanItems], keep[kScanItems];
        long long sraw = 0, skeep = 0;
#pragma unroll
        for (int k = 0; k < kScanItems; ++k) {
            int d = base + tid * kScanItems + k;
            len[k] = d < nd ? a.doc_lens[d] : 0;
            if (d < nd && len[k] <= 0) bad = true;
            if (len[k] < 0) len[k] = 0;
            keep[k] = a.packed ? len[k] : min(len[k], a.seq_len);
            sraw += len[k];
            skeep += keep[k];
        }
        long long traw, tkeep;
        long long eraw = block_excl_scan(sraw, &traw, sh) + carry_raw;
        long long ekeep = block_excl_scan(skeep, &tkeep, sh) + carry_keep;
#pragma unroll
        for (int k = 0; k < kScanItems; ++k) {
            int d = base + tid * kScanItems + k;
            if (d < nd) {
                a.doc_in[d] = static_cast<int32_t>(eraw);
                a.doc_keep[d] = keep[k];
                aux[d] = static_cast<int32_t>(ekeep);  // unpack: global kept prefix
            }
            eraw += len[k];
            ekeep += keep[k];
        }
        carry_raw += traw;
        carry_keep += tkeep;
        if (carry_raw > 0x7fffffffLL) bad = true;
    }
    if (bad) atomicOr(&bad_s, 1);
    __syncthreads();
    if (bad_s || carry_raw != a.num_tokens) {
        if (tid == 0) {
            set_status(a.status, kErrBadDocs);
            *a.num_segs = 0;
        }
        return;
    }
    if (tid == 0) {
        a.doc_in[nd] = static_cast<int32_t>(carry_raw);
        aux[nd] = static_cast<int32_t>(carry_keep);
    }
    __syncthreads();

    // build_unpack (build_pack runs pack_prefix_kernel instead)
    int num_segs;
    // One segment per kept document, plus a padding segment in every row
    // that the kept documents do not fill.
    const int mb = a.micro_bsz;
    long long carry_pad = 0;
    for (int base = 0; base < a.rows; base += kScanThreads) {
        int r = base + tid;
        int flag = 0;
        if (r < a.rows) {
            int d0 = r * mb, d1 = min(nd, d0 + mb);
            long long fill = static_cast<long long>(aux[d1]) - aux[d0];
            flag = fill < plen ? 1 : 0;
        }
        long long tot;
        long long e = block_excl_scan(flag, &tot, sh) + carry_pad;
        if (r < a.rows) a.row_seg_ptr[r] = static_cast<int32_t>(static_cast<long long>(r) * mb + e);
        carry_pad += tot;
    }
    num_segs = static_cast<int>(nd + carry_pad);
    if (tid == 0) a.row_seg_ptr[a.rows] = num_segs;
    __syncthreads();
    for (int d = tid; d < nd; d += kScanThreads) {
        int r = d / mb;
        long long out = r * plen + aux[d] - aux[r * mb];
        a.doc_out[d] = static_cast<int32_t>(out);
        a.cu_seqlens[a.row_seg_ptr[r] + (d - r * mb)] = static_cast<int32_t>(out);
    }
    for (int r = tid; r < a.rows; r += kScanThreads) {
        int d0 = r * mb, d1 = min(nd, d0 + mb);
        long long fill = static_cast<long long>(aux[d1]) - aux[d0];
        if (fill < plen)
            a.cu_seqlens[a.row_seg_ptr[r] + (d1 - d0)] = static_cast<int32_t>(r * plen + fill);
    }
    if (tid == 0) a.cu_seqlens[num_segs] = static_cast<int32_t>(a.rows * plen);
    if (tid == 0) *a.num_segs = num_segs;
    __syncthreads();
    for (int i = tid; i < num_segs; i += kScanThreads) {
        int s = a.cu_seqlens[i];
        atomicMax(&a.max_seqlen[s / plen], a.cu_seqlens[i + 1] - s);
    }
}

// build_unpack token stream: row r holds documents r * micro_bsz .. +micro_bsz - 1,
// each truncated to SEQ_LEN and placed one after the other, then padding.
// kChunk consecutive output positions per CTA, four per thread per iteration.
// A thread keeps its row and its current document (output start, kept length,
// input start) in registers: a division where a group of four starts past the
// row, a search among the row's documents where it starts past the document,
// and a step to the next document (which starts where the kept part ends)
// inside a group.
__global__ void __launch_bounds__(kStreamThreads) unpack_stream_kernel(PackArgs a)
{
    const int plen = a.plen, mb = a.micro_bsz, nd = a.num_docs;
    const int npos = a.rows * plen;   // rows * plen <= 2^31 - 65537 is checked on the host
    const int P0 = static_cast<int>(blockIdx.x) * kChunk;
    const int P1 = min(npos, P0 + kChunk);
    pdl_wait();
    if (*reinterpret_cast<volatile int *>(a.status) != 0) return;
    int row_end = 0, d_end = 0;        // the current row's end and its documents' end index
    int dd = 0, start = 0, keep = 0, src = 0;
    auto load_doc = [&](int d) {
        dd = d;
        start = a.doc_out[d];
        keep = a.doc_keep[d];
        src = a.doc_in[d];
    };
#pragma unroll
    for (int it = 0; it < kStreamIters; ++it) {
        const int p = P0 + (it * kStreamThreads + threadIdx.x) * 4;
        if (p >= P1) break;
        int32_t id[4], lab[4], idx[4];
        if (p >= row_end) {                                  // a new row: its documents d0 .. d_end - 1
            const int r = p / plen;
            row_end = (r + 1) * plen;
            const int d0 = r * mb;
            d_end = min(nd, d0 + mb);
            load_doc(last_le(a.doc_out, d0, d_end, p));      // doc_out[d0] = r * plen <= p
        } else if (p - start >= keep && dd + 1 < d_end) {    // past the document: a later one of the row
            load_doc(last_le(a.doc_out, dd + 1, d_end, p));  // doc_out[dd + 1] = start + keep <= p
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int q = p + k;
            if (q >= P1) {
                id[k] = lab[k] = idx[k] = 0;
                continue;
            }
            if (q >= row_end) {                              // one position further: the next row's first
                row_end += plen;
                const int d0 = d_end;                        // the next row's first document
                d_end = min(nd, d0 + mb);
                load_doc(d0);
            }
            int t = q - start;
            if (t >= keep && dd + 1 < d_end) {               // the next document starts where this one's kept part ends
                load_doc(dd + 1);
                t = q - start;
            }
            if (t < keep) {
                id[k] = a.tokens[src + t];
                lab[k] = (t + 1 < keep) ? a.tokens[src + t + 1] : -100;
                idx[k] = t;
            } else {                                         // the row's padding tail
                id[k] = 0;
                lab[k] = -100;
                idx[k] = t - keep;
            }
        }
        if (a.vec_out && p + 4 <= P1) {
            *reinterpret_cast<int4 *>(a.input_ids + p) = make_int4(id[0], id[1], id[2], id[3]);
            *reinterpret_cast<int4 *>(a.labels + p) = make_int4(lab[0], lab[1], lab[2], lab[3]);
            *reinterpret_cast<int4 *>(a.indexes + p) = make_int4(idx[0], idx[1], idx[2], idx[3]);
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (p + k < P1) {
                    a.input_ids[p + k] = id[k];
                    a.labels[p + k] = lab[k];
                    a.indexes[p + k] = idx[k];
                }
            }
        }
    }
}

// ---------------------------------------------------------------- fused path
// build_pack with few documents and rows (the common case): one launch. Every
// CTA scans the document lengths itself into shared memory (they are a few KB
// and stay in L2); CTA 0 then writes the segment fields and the status word,
// every other CTA 1024 output positions. Same rules and outputs as the
// two-kernel path.
constexpr int kFusedThreads = 256;
constexpr int kFusedDocs = 1024;   // documents the fused path accepts
constexpr int kFusedRows = 512;    // rows the fused path accepts
constexpr int kFusedIters = 1;
constexpr int kFusedChunk = kFusedThreads * 4 * kFusedIters;

__device__ int block_excl_scan256(int v, int *total, int *sh)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < kFusedThreads / 32 ? sh[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kFusedThreads / 32) sh[lane] = w;
    }
    __syncthreads();
    const int r = (warp ? sh[warp - 1] : 0) + x - v;
    *total = sh[kFusedThreads / 32 - 1];
    __syncthreads();
    return r;
}

// Largest d in [0, n) with a[d] <= x; assumes a[0] <= x.
__device__ __forceinline__ int last_le_smem(const int32_t *a, int n, int x)
{
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (a[mid] <= x) lo = mid;
        else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ int32_t int4_at(const int4 &v, int k)
{
    return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
}

// build_pack token stream (more documents or rows than the fused path takes):
// kChunk consecutive output positions per CTA, four per thread per iteration.
// The chunk's tokens are loaded once into registers and input_ids (which needs
// no document boundaries) is stored while the scan kernel may still run. After
// the scan, the CTA finds the document holding its first position with a
// block-wide search (256 sampled starts per round, one barrier each) and
// stages the starts of the documents its chunk overlaps in shared memory;
// labels and indexes then need no global lookups. At most 40 registers per
// thread (6 resident CTAs per SM).
constexpr int kWin = 1024;   // document starts staged per CTA

__global__ void __launch_bounds__(kStreamThreads, 6) pack_packed_stream_kernel(PackArgs a)
{
    __shared__ int32_t s_doc[kWin];
    __shared__ int32_t s_max[kWin];   // per-row maxima of this chunk's segments
    const int tid = threadIdx.x, lane = tid & 31;
    const int total = a.num_tokens, nd = a.num_docs, plen = a.plen;
    const int npos = a.rows * plen;   // rows * plen <= 2^31 - 1 is checked on the host
    const int P0 = static_cast<int>(blockIdx.x) * kChunk;
    const int P1 = min(npos, P0 + kChunk);

    int4 tk[kStreamIters];
    int32_t nx[kStreamIters];   // the token after each group of four (its last label)
#pragma unroll
    for (int it = 0; it < kStreamIters; ++it) {
        const int p = P0 + (it * kStreamThreads + tid) * 4;
        if (a.vec_in && p + 4 <= total) {
            tk[it] = __ldg(reinterpret_cast<const int4 *>(a.tokens + p));
        } else {
            tk[it].x = p < total ? __ldg(a.tokens + p) : 0;
            tk[it].y = p + 1 < total ? __ldg(a.tokens + p + 1) : 0;
            tk[it].z = p + 2 < total ? __ldg(a.tokens + p + 2) : 0;
            tk[it].w = p + 3 < total ? __ldg(a.tokens + p + 3) : 0;
        }
    }
#pragma unroll
    for (int it = 0; it < kStreamIters; ++it) {
        const int p = P0 + (it * kStreamThreads + tid) * 4;
        int32_t v = __shfl_down_sync(0xffffffffu, tk[it].x, 1);
        if (lane == 31) v = p + 4 < total ? __ldg(a.tokens + p + 4) : 0;
        nx[it] = v;
        if (p >= P1) continue;
        if (a.vec_out && p + 4 <= P1) {
            *reinterpret_cast<int4 *>(a.input_ids + p) = tk[it];
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (p + k < P1) a.input_ids[p + k] = int4_at(tk[it], k);
        }
    }
    pdl_wait();
    if (*reinterpret_cast<volatile int *>(a.status) != 0) return;

    // The document holding position P0 (chunks wholly in the padding need none):
    // doc_out[lo] <= P0 < doc_out[hi] throughout, the range shrinking 256-fold
    // per round.
    __shared__ int s_cnt;
    int d_lo = 0, W = 0, Wn = 0;
    bool staged = false;
    if (tid == 0) s_cnt = 0;
    if (P0 < total) {
        int lo = 0, hi = nd;
        while (hi - lo > 1) {
            const int step = (hi - lo + kStreamThreads - 1) / kStreamThreads;
            const int idx = lo + tid * step;
            const bool le = idx < hi && a.doc_out[idx] <= P0;
            const int cnt = __syncthreads_count(le);   // >= 1: doc_out[lo] <= P0
            lo += (cnt - 1) * step;
            hi = min(hi, lo + step);
        }
        d_lo = lo;
        W = min(kWin, nd + 1 - d_lo);   // doc_out[nd] = num_tokens ends the last document
        for (int i = tid; i < W; i += kStreamThreads) s_doc[i] = a.doc_out[d_lo + i];
        __syncthreads();
        // staged when the window reaches past the chunk's last token; the
        // searches then stay inside its first Wn entries (the starts below the
        // chunk's end and the one after them)
        const int lim = min(P1, total);
        staged = s_doc[W - 1] > lim - 1;
        int c = 0;
        for (int i = tid; i < W; i += kStreamThreads) c += s_doc[i] < lim;
        if (c) atomicAdd(&s_cnt, c);
        __syncthreads();
        Wn = min(W, s_cnt + 1);
    }

    // The current document's bounds and row are kept across positions: a
    // search only where a group of four starts past the document, a division
    // only where it starts past the row.
    auto doc = [&](int i) -> int { return staged ? s_doc[i] : a.doc_out[d_lo + i]; };
    int d = 0, start = 0, end = 0, row_start = 0, row_end = 0;
#pragma unroll
    for (int it = 0; it < kStreamIters; ++it) {
        const int p = P0 + (it * kStreamThreads + tid) * 4;
        if (p >= P1) break;
        int32_t lab[4], idx[4];
        if (p < total && p >= end) {
            d = staged ? last_le_smem(s_doc, Wn, p) : last_le(a.doc_out, d_lo, nd, p) - d_lo;
            start = doc(d);
            end = doc(d + 1);
        }
        if (p >= row_end) {
            row_start = p - p % plen;
            row_end = row_start + plen;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int q = p + k;
            if (q >= total) {   // the padding segment starts at num_tokens
                lab[k] = -100;
                idx[k] = q - total;
                continue;
            }
            if (q >= end) {     // q < doc_out[nd] = total
                do ++d;
                while (doc(d + 1) <= q);
                start = doc(d);
                end = doc(d + 1);
            }
            if (q >= row_end) {   // q grows by one: at most one row further
                row_start = row_end;
                row_end += plen;
            }
            const int next = k < 3 ? int4_at(tk[it], k + 1) : nx[it];
            lab[k] = q + 1 < end ? next : -100;
            idx[k] = q - (start > row_start ? start : row_start);
        }
        if (a.vec_out && p + 4 <= P1) {
            *reinterpret_cast<int4 *>(a.labels + p) = make_int4(lab[0], lab[1], lab[2], lab[3]);
            *reinterpret_cast<int4 *>(a.indexes + p) = make_int4(idx[0], idx[1], idx[2], idx[3]);
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (p + k < P1) {
                    a.labels[p + k] = lab[k];
                    a.indexes[p + k] = idx[k];
                }
            }
        }
    }

    // Segment fields of the boundaries inside this chunk: document starts not on
    // a row start, row starts and the padding start. A boundary's place in
    // cu_seqlens follows from the counts the prefix kernel wrote: before a
    // document start s (document d) lie the row starts up to s and the
    // documents 1 .. d - 1 that do not start on a row start; before a row start
    // r * plen, r row starts and the documents 1 .. ds - 1 (ds the first
    // document starting at or after it) less the ones on a row start. Each
    // segment's length goes to its row's max_seqlen (zeroed by the prefix kernel).
    const int rows = a.rows;
    auto doc_start = [&](int d) -> int {
        const int i = d - d_lo;
        return (i >= 0 && i < W) ? s_doc[i] : a.doc_out[d];
    };
    // Per-row maxima of this chunk's segments are first combined in shared
    // memory (a chunk of very short documents holds hundreds of segments of
    // one row; one global atomic each would queue on one address), then added
    // with one global atomic per row. Chunks spanning more rows than the
    // staging holds use global atomics directly.
    const int row0 = P0 / plen;
    const int nrow = (P1 - 1) / plen - row0 + 1;
    const bool smem_max = nrow <= kWin;
    for (int i = tid; i < nrow && smem_max; i += kStreamThreads) s_max[i] = 0;
    __syncthreads();
    auto seg_max = [&](int row, int len) {
        if (smem_max) atomicMax(&s_max[row - row0], len);
        else atomicMax(&a.max_seqlen[row], len);
    };
    if (P0 < total) {
        for (int d = d_lo + tid; d < nd; d += kStreamThreads) {
            const int st = doc_start(d);
            if (st >= P1) break;
            if (st < P0 || st % plen == 0) continue;   // on a row start: the row's boundary below
            const int row = st / plen;
            const int end = min(doc_start(d + 1), (row + 1) * plen);
            a.cu_seqlens[(st - 1) / plen + d - a.aligned[d]] = st;
            seg_max(row, end - st);
        }
    }
    const int r_first = row0 + (P0 != row0 * plen);   // the first row starting at or after P0
    for (int r = r_first + tid; r < rows; r += kStreamThreads) {
        const int x = r * plen;   // < rows * plen <= 2^31 - 65537
        if (x >= P1) break;
        // the first document starting at or after x (inside the staged window
        // when x is a token of this chunk)
        const int ds = (staged && x < total) ? d_lo + lower_bound(s_doc, 0, Wn, x) : lower_bound(a.doc_out, 0, nd, x);
        const int rank = r == 0 ? 0 : r + ds - 1 - a.aligned[ds];
        a.cu_seqlens[rank] = x;
        a.row_seg_ptr[r] = rank;
        // the segment from x ends at the next document start, the row end or num_tokens
        int next = x + plen;
        if (ds < nd) {
            const int sd = a.doc_out[ds];
            next = min(next, sd == x ? a.doc_out[ds + 1] : sd);
        } else {
            next = min(next, total);
        }
        seg_max(r, next - x);
    }
    if (tid == 0 && total % plen != 0 && P0 <= total && total < P1) {   // the padding tail of the last row
        a.cu_seqlens[*a.num_segs - 1] = total;
        seg_max(total / plen, rows * plen - total);
    }
    if (smem_max) {
        __syncthreads();
        for (int i = tid; i < nrow; i += kStreamThreads)
            if (s_max[i] > 0) atomicMax(&a.max_seqlen[row0 + i], s_max[i]);
    }
}

// At most 32 registers per thread (8 resident CTAs per SM): the 1025 CTAs of a
// million-token row then run as one wave. Launched as a programmatic dependent
// of whatever precedes it on the stream: it lets the next launch be scheduled
// at once and waits for the previous grid (and its memory) before its first
// global access, so back-to-back packs overlap launch latency only.
__global__ void __launch_bounds__(kFusedThreads, 8) pack_fused_kernel(PackArgs a)
{
    pdl_launch_dependents();
    pdl_wait();
    __shared__ int32_t s_start[kFusedDocs + 1];
    __shared__ int sh[32];
    __shared__ int bad_s;
    const int tid = threadIdx.x;
    const int nd = a.num_docs;
    // all positions fit in int32 (rows * plen <= 2^31 - 1 is checked on the host)
    const int plen = a.plen, total = a.num_tokens;
    const int npos = a.rows * plen;
    if (tid == 0) bad_s = 0;

    // The token loads need no document boundaries: issue them first so their
    // latency overlaps the scan. tk[k] = tokens[p + k], k = 0..4 (k = 4 feeds
    // the label of position p + 3).
    const int p = static_cast<int>(blockIdx.x - 1) * kFusedChunk + tid * 4;
    int32_t tk[5];
#pragma unroll
    for (int k = 0; k < 5; ++k)
        tk[k] = (blockIdx.x > 0 && p + k < total) ? __ldg(a.tokens + p + k) : 0;

    // document starts: exclusive scan of the lengths, 4 per thread
    {
        int len[4];
        long long sum64 = 0;
        bool bad = false;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int d = tid * 4 + k;
            len[k] = d < nd ? a.doc_lens[d] : 0;
            if (d < nd && len[k] <= 0) bad = true;
            if (len[k] < 0) len[k] = 0;
            sum64 += len[k];
        }
        // valid lengths sum to num_tokens <= 2^31 - 1, so any partial sum above it is bad
        if (sum64 > a.num_tokens) bad = true;
        const int sum = bad ? 0 : static_cast<int>(sum64);
        if (bad) atomicOr(&bad_s, 1);
        int tot;
        int e = block_excl_scan256(sum, &tot, sh);
        long long run = e;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int d = tid * 4 + k;
            if (d < nd) s_start[d] = static_cast<int32_t>(run);
            run += len[k];
        }
        if (tid == 0) {
            s_start[nd] = tot;
            if (tot != a.num_tokens) bad_s = 1;
        }
    }
    __syncthreads();
    if (bad_s) {
        if (blockIdx.x == 0 && tid == 0) {
            *a.status = kErrBadDocs;   // CTA 0 alone owns the status word in this launch
            *a.num_segs = 0;
        }
        return;
    }

    // CTA 0 writes the segment fields; CTAs 1.. write 1024 output positions each,
    // four consecutive positions per thread
    if (blockIdx.x > 0 && p < npos) {
        int32_t id[4], lab[4], idx[4];
        int d = p < total ? last_le_smem(s_start, nd, p) : 0;
        int start = s_start[d], end = s_start[d + 1];   // document d (s_start[nd] = total)
        int row_start = p - p % plen;                    // one division per thread
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int q = p + k;
            if (q >= npos) { id[k] = lab[k] = idx[k] = 0; continue; }
            if (q >= total) {
                id[k] = 0;
                lab[k] = -100;
                idx[k] = q - total;
                continue;
            }
            if (q >= end) {                              // the next document(s)
                do ++d;
                while (s_start[d + 1] <= q);
                start = s_start[d];
                end = s_start[d + 1];
            }
            while (q >= row_start + plen) row_start += plen;
            id[k] = tk[k];
            lab[k] = (q + 1 < end) ? tk[k + 1] : -100;
            idx[k] = q - (start > row_start ? start : row_start);
        }
        if (a.vec_out && p + 4 <= npos) {
            *reinterpret_cast<int4 *>(a.input_ids + p) = make_int4(id[0], id[1], id[2], id[3]);
            *reinterpret_cast<int4 *>(a.labels + p) = make_int4(lab[0], lab[1], lab[2], lab[3]);
            *reinterpret_cast<int4 *>(a.indexes + p) = make_int4(idx[0], idx[1], idx[2], idx[3]);
        } else {
            for (int k = 0; k < 4 && p + k < npos; ++k) {
                a.input_ids[p + k] = id[k];
                a.labels[p + k] = lab[k];
                a.indexes[p + k] = idx[k];
            }
        }
    }
    if (blockIdx.x != 0) return;

    // CTA 0: segment boundaries are the union of document starts, row starts and
    // the padding start; a document start on a row start is the same boundary
    // (counted by the "aligned" scan so ranks stay exact).
    __shared__ int32_t s_aligned[kFusedDocs + 1];   // aligned starts before document d
    __shared__ int32_t s_cu[kFusedDocs + 2 * kFusedRows + 1];
    __shared__ int32_t s_max[kFusedRows];
    {
        int f[4], sum = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int d = tid * 4 + k;
            f[k] = (d >= 1 && d < nd && (s_start[d] % plen) == 0) ? 1 : 0;
            sum += f[k];
        }
        int tot;
        int run = block_excl_scan256(sum, &tot, sh);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int d = tid * 4 + k;
            if (d <= nd) s_aligned[d] = run;
            run += f[k];
        }
        if (tid == 0) s_aligned[nd] = tot;
    }
    for (int r = tid; r < a.rows; r += kFusedThreads) s_max[r] = 0;
    __syncthreads();
    const int pad = (total % plen) != 0;
    const int num_segs = a.rows == 0 ? 0 : static_cast<int>(a.rows + nd - 1 - s_aligned[nd] + pad);
    for (int d = tid; d < nd; d += kFusedThreads) {
        const int st = s_start[d];
        if (d >= 1 && (st % plen) != 0) s_cu[(st - 1) / plen + d - s_aligned[d]] = st;
    }
    for (int r = tid; r <= a.rows; r += kFusedThreads) {
        int rank = 0;
        if (r > 0) {
            // first document starting at or after r * plen
            const int x = r * plen;
            int lo = 0, hi = nd;
            while (lo < hi) {
                int mid = (lo + hi) >> 1;
                if (s_start[mid] < x) lo = mid + 1;
                else hi = mid;
            }
            rank = r + lo - 1 - s_aligned[lo] + ((r == a.rows && pad) ? 1 : 0);
        }
        s_cu[rank] = r * plen;
        a.row_seg_ptr[r] = rank;
    }
    if (tid == 0 && pad) s_cu[num_segs - 1] = total;
    __syncthreads();
    for (int i = tid; i <= num_segs; i += kFusedThreads) a.cu_seqlens[i] = s_cu[i];
    for (int i = tid; i < num_segs; i += kFusedThreads)
        atomicMax(&s_max[s_cu[i] / plen], s_cu[i + 1] - s_cu[i]);
    __syncthreads();
    for (int r = tid; r < a.rows; r += kFusedThreads) a.max_seqlen[r] = s_max[r];
    if (tid == 0) {
        *a.num_segs = num_segs;
        *a.status = 0;
    }
}

// build_unpack with at most 1024 documents (so at most 1024 rows): one launch.
// Every CTA scans the document lengths into shared memory (the raw lengths'
// prefix gives a document's input start, the kept lengths' prefix its place
// in its row); CTA 0 then writes the segment fields and the status word,
// every other CTA 1024 output positions. Same rules and outputs as
// pack_scan_kernel + unpack_stream_kernel.
__global__ void __launch_bounds__(kFusedThreads, 8) unpack_fused_kernel(PackArgs a)
{
    pdl_launch_dependents();
    pdl_wait();
    __shared__ int32_t s_in[kFusedDocs + 1];   // input start of each document (+ num_tokens)
    __shared__ int32_t s_k[kFusedDocs + 1];    // kept tokens before each document (+ all kept)
    __shared__ int sh[32];
    __shared__ int bad_s;
    const int tid = threadIdx.x;
    const int nd = a.num_docs, mb = a.micro_bsz, plen = a.plen;
    const int npos = a.rows * plen;   // rows * plen <= 2^31 - 65537 is checked on the host
    if (tid == 0) bad_s = 0;
    {
        int len[4], kp[4];
        long long sraw = 0;
        bool bad = false;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int d = tid * 4 + k;
            len[k] = d < nd ? a.doc_lens[d] : 0;
            if (d < nd && len[k] <= 0) bad = true;
            if (len[k] < 0) len[k] = 0;
            kp[k] = min(len[k], a.seq_len);
            sraw += len[k];
        }
        // valid lengths sum to num_tokens <= 2^31 - 1, so any partial sum above it is bad
        if (sraw > a.num_tokens) bad = true;
        if (bad) atomicOr(&bad_s, 1);
        int tot_raw, tot_keep;
        long long eraw = block_excl_scan256(bad ? 0 : static_cast<int>(sraw), &tot_raw, sh);
        long long ekeep = block_excl_scan256(bad ? 0 : kp[0] + kp[1] + kp[2] + kp[3], &tot_keep, sh);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int d = tid * 4 + k;
            if (d < nd) {
                s_in[d] = static_cast<int32_t>(eraw);
                s_k[d] = static_cast<int32_t>(ekeep);
            }
            eraw += len[k];
            ekeep += kp[k];
        }
        if (tid == 0) {
            s_in[nd] = tot_raw;
            s_k[nd] = tot_keep;
            if (tot_raw != a.num_tokens) bad_s = 1;
        }
    }
    __syncthreads();
    if (bad_s) {
        if (blockIdx.x == 0 && tid == 0) {
            *a.status = kErrBadDocs;   // CTA 0 alone owns the status word in this launch
            *a.num_segs = 0;
        }
        return;
    }

    if (blockIdx.x > 0) {
        const int p = static_cast<int>(blockIdx.x - 1) * kFusedChunk + tid * 4;
        if (p >= npos) return;
        // row r holds documents d0 .. d_end - 1 one after the other, then padding;
        // the row's documents start at r * plen + s_k[d] - s_k[d0]
        const int r = p / plen;
        int row_start = r * plen;
        int d0 = r * mb, d_end = min(nd, d0 + mb);
        int base = row_start - s_k[d0];
        int dd = d0 + last_le_smem(s_k + d0, d_end - d0, p - base);
        int start = base + s_k[dd], keep = s_k[dd + 1] - s_k[dd];
        int32_t id[4], lab[4], idx[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int q = p + k;
            if (q >= npos) {
                id[k] = lab[k] = idx[k] = 0;
                continue;
            }
            if (q >= row_start + plen) {   // one position further: the next row's first
                row_start += plen;
                d0 = d_end;
                d_end = min(nd, d0 + mb);
                base = row_start - s_k[d0];
                dd = d0;
                start = row_start;
                keep = s_k[dd + 1] - s_k[dd];
            }
            int t = q - start;
            if (t >= keep && dd + 1 < d_end) {   // the next document starts where this one's kept part ends
                ++dd;
                start += keep;
                keep = s_k[dd + 1] - s_k[dd];
                t = q - start;
            }
            if (t < keep) {
                const int src = s_in[dd] + t;
                id[k] = __ldg(a.tokens + src);
                lab[k] = (t + 1 < keep) ? __ldg(a.tokens + src + 1) : -100;
                idx[k] = t;
            } else {                             // the row's padding tail
                id[k] = 0;
                lab[k] = -100;
                idx[k] = t - keep;
            }
        }
        if (a.vec_out && p + 4 <= npos) {
            *reinterpret_cast<int4 *>(a.input_ids + p) = make_int4(id[0], id[1], id[2], id[3]);
            *reinterpret_cast<int4 *>(a.labels + p) = make_int4(lab[0], lab[1], lab[2], lab[3]);
            *reinterpret_cast<int4 *>(a.indexes + p) = make_int4(idx[0], idx[1], idx[2], idx[3]);
        } else {
            for (int k = 0; k < 4 && p + k < npos; ++k) {
                a.input_ids[p + k] = id[k];
                a.labels[p + k] = lab[k];
                a.indexes[p + k] = idx[k];
            }
        }
        return;
    }

    // CTA 0: one segment per document, plus the padding tail of every row its
    // documents do not fill; a row's first segment comes after the documents
    // and padding tails of the rows before it (all full rows of micro_bsz
    // documents). max_seqlen per row from shared-memory maxima.
    __shared__ int32_t s_rsp[kFusedDocs];
    __shared__ int32_t s_rmax[kFusedDocs];
    const int rows = a.rows;
    int f[4], fsum = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int r = tid * 4 + k;
        f[k] = 0;
        if (r < rows) {
            const int d0 = r * mb, d1 = min(nd, d0 + mb);
            const int fill = s_k[d1] - s_k[d0];
            f[k] = fill < plen ? 1 : 0;
            s_rmax[r] = f[k] ? plen - fill : 0;
        }
        fsum += f[k];
    }
    int npad;
    int run = block_excl_scan256(fsum, &npad, sh);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int r = tid * 4 + k;
        if (r < rows) s_rsp[r] = r * mb + run;
        run += f[k];
    }
    __syncthreads();
    const int num_segs = nd + npad;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int d = tid * 4 + k;
        if (d < nd) {
            const int r = d / mb, d0 = r * mb;
            a.cu_seqlens[s_rsp[r] + d - d0] = r * plen + s_k[d] - s_k[d0];
            atomicMax(&s_rmax[r], s_k[d + 1] - s_k[d]);
        }
        const int r = tid * 4 + k;
        if (r < rows && f[k]) {
            const int d0 = r * mb, d1 = min(nd, d0 + mb);
            a.cu_seqlens[s_rsp[r] + d1 - d0] = r * plen + s_k[d1] - s_k[d0];
        }
    }
    __syncthreads();
    for (int r = tid; r < rows; r += kFusedThreads) {
        a.max_seqlen[r] = s_rmax[r];
        a.row_seg_ptr[r] = s_rsp[r];
    }
    if (tid == 0) {
        a.row_seg_ptr[rows] = num_segs;
        a.cu_seqlens[num_segs] = npos;
        *a.num_segs = num_segs;
        *a.status = 0;
    }
}

}  // namespace

size_t pack_ws_bytes(int64_t num_docs)
{
    // status header + 4 arrays of num_docs + 1 int32 + the prefix kernel's CTA
    // ticket and look-back descriptors (two per CTA)
    const size_t nb = static_cast<size_t>((num_docs + kPrefixDocs - 1) / kPrefixDocs);
    return kWsHeader + 4 * align_up(sizeof(int32_t) * static_cast<size_t>(num_docs + 1), 256) +
           align_up(8 + 16 * (nb > 0 ? nb : 1), 256);
}

cudaError_t launch_pack(const PackArgs &a_in, int num_sms, cudaStream_t stream)
{
    (void)num_sms;
    PackArgs a = a_in;
    const size_t arr = align_up(sizeof(int32_t) * static_cast<size_t>(a.num_docs + 1), 256);
    char *ws = reinterpret_cast<char *>(a.status);
    a.doc_out = reinterpret_cast<int32_t *>(ws + kWsHeader);
    a.doc_in = reinterpret_cast<int32_t *>(ws + kWsHeader + arr);
    a.doc_keep = reinterpret_cast<int32_t *>(ws + kWsHeader + 2 * arr);
    int32_t *aux = reinterpret_cast<int32_t *>(ws + kWsHeader + 3 * arr);
    a.aligned = aux;
    a.ticket = reinterpret_cast<unsigned *>(ws + kWsHeader + 4 * arr);
    a.look = reinterpret_cast<unsigned long long *>(ws + kWsHeader + 4 * arr + 8);

    const long long npos = static_cast<long long>(a.rows) * a.plen;
    if (a.packed && a.num_docs >= 1 && a.num_docs <= kFusedDocs && a.rows <= kFusedRows) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(1 + (npos + kFusedChunk - 1) / kFusedChunk));
        cfg.blockDim = dim3(kFusedThreads);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        prof_begin(kProfPackStream, stream);
        cudaError_t e0 = cudaLaunchKernelEx(&cfg, pack_fused_kernel, a);
        prof_end(kProfPackStream, stream);
        return e0;
    }
    if (!a.packed && a.num_docs >= 1 && a.num_docs <= kFusedDocs) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(1 + (npos + kFusedChunk - 1) / kFusedChunk));
        cfg.blockDim = dim3(kFusedThreads);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        prof_begin(kProfPackStream, stream);
        cudaError_t e0 = cudaLaunchKernelEx(&cfg, unpack_fused_kernel, a);
        prof_end(kProfPackStream, stream);
        return e0;
    }
    cudaError_t e;
    if (a.packed) {
        const int nb = static_cast<int>((static_cast<long long>(a.num_docs) + kPrefixDocs - 1) / kPrefixDocs);
        if (nb > 1) {
            // several CTAs chain their prefixes: clear the status word, the ticket
            // and the look-back descriptors first
            if ((e = cudaMemsetAsync(a.status, 0, sizeof(int), stream)) != cudaSuccess) return e;
            if ((e = cudaMemsetAsync(a.ticket, 0, 8 + 16 * static_cast<size_t>(nb), stream)) != cudaSuccess)
                return e;
        }
        cudaLaunchConfig_t pcfg = {};
        pcfg.gridDim = dim3(static_cast<unsigned>(nb > 0 ? nb : 1));
        pcfg.blockDim = dim3(kScanThreads);
        pcfg.stream = stream;
        cudaLaunchAttribute pattr[1];
        pattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        pattr[0].val.programmaticStreamSerializationAllowed = 1;
        pcfg.attrs = pattr;
        pcfg.numAttrs = 1;
        if ((e = cudaLaunchKernelEx(&pcfg, pack_prefix_kernel, a, nb > 0 ? nb : 1)) != cudaSuccess) return e;
    } else {
        pack_scan_kernel<<<1, kScanThreads, 0, stream>>>(a, aux);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (npos == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((npos + kChunk - 1) / kChunk));
    cfg.blockDim = dim3(kStreamThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    prof_begin(kProfPackStream, stream);
    e = a.packed ? cudaLaunchKernelEx(&cfg, pack_packed_stream_kernel, a)
                 : cudaLaunchKernelEx(&cfg, unpack_stream_kernel, a);
    prof_end(kProfPackStream, stream);
    return e;
}

}  // namespace spd
