// Data steps after packing (InternEvo page "Data loading and flow", section
// "Processing data"):
//   unpack_data                   packed rows -> [rows][micro_bsz][seq_len], one
//                                 segment (document) per output row, cut to
//                                 seq_len, padded with 0 / -100;
//   split_data_sequence_parallel  the rank's contiguous 1/sp_size chunk of the
//                                 sequence dimension of each row;
// and pad_for_sequence_parallel (XTuner page "Sequence parallel training of
// extremely long sequences", sequence parallel API): each row padded at its
// end to a multiple of sp_size.
// All are pure data movement (HBM-bound): every thread takes groups of four
// consecutive output positions, grid-stride, with 16-byte stores where the
// output row layout allows (and, for the padding, 16-byte loads realigned
// across the warp where a row's source start is not).
#include "internal.h"
#include "ptx.cuh"

namespace spd {
namespace {

constexpr int kThreads = 256;
constexpr int32_t kPad = 0, kIgnore = -100;

__global__ void __launch_bounds__(kThreads) unpack_kernel(UnpackArgs a)
{
    const int32_t plen = a.micro_bsz * a.seq_len;
    const int32_t total = a.rows * plen;
    const bool vec = a.vec_out && (a.seq_len & 3) == 0;   // a group of 4 never crosses an output row
    // 64-bit loop index: the step past the last group must not wrap (total < 2^31)
    for (int64_t xl = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) * 4; xl < total;
         xl += static_cast<int64_t>(gridDim.x) * kThreads * 4) {
        const int32_t x = static_cast<int32_t>(xl);
        int32_t id[4], lab[4];
        int32_t cur_key = -1, a0 = 0, n = 0;   // segment of the last output row looked up
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            id[k] = kPad;
            lab[k] = kIgnore;
            const int32_t p = x + k;
            if (p >= total) continue;
            const int32_t r = p / plen, rem = p - r * plen;
            const int32_t m = rem / a.seq_len, j = rem - m * a.seq_len;
            const int32_t key = r * a.micro_bsz + m;
            if (key != cur_key) {          // output row (r, m) <- segment row_seg_ptr[r] + m of row r
                cur_key = key;
                const int32_t s = a.row_seg_ptr[r] + m;
                if (s < a.row_seg_ptr[r + 1]) {
                    a0 = a.cu_seqlens[s];
                    n = min(a.cu_seqlens[s + 1] - a0, a.seq_len);
                } else {
                    a0 = 0;
                    n = 0;
                }
            }
            if (j < n) {
                id[k] = a.input_ids[a0 + j];
                lab[k] = a.labels[a0 + j];
            }
        }
        if (vec) {
            *reinterpret_cast<int4 *>(a.out_ids + x) = make_int4(id[0], id[1], id[2], id[3]);
            *reinterpret_cast<int4 *>(a.out_labels + x) = make_int4(lab[0], lab[1], lab[2], lab[3]);
        } else {
            for (int k = 0; k < 4 && x + k < total; ++k) {
                a.out_ids[x + k] = id[k];
                a.out_labels[x + k] = lab[k];
            }
        }
    }
}

__global__ void __launch_bounds__(kThreads) split_kernel(SplitArgs a)
{
    const int32_t chunk = a.len / a.sp_size;
    const int32_t total = a.rows * chunk;
    const int32_t off = a.rank * chunk;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads * 4;
    // Two groups of four positions per thread and iteration, every load issued
    // before the first store (up to six 16-byte loads in flight per thread).
    // 64-bit loop index: the step past the last group must not wrap (total < 2^31).
    for (int64_t xl = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) * 4; xl < total;
         xl += 2 * stride) {
        int32_t x[2], src[2];
        bool full[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t xu = xl + u * stride;
            x[u] = xu < total ? static_cast<int32_t>(xu) : total;
            const int32_t r = x[u] / chunk, j = x[u] - r * chunk;
            src[u] = r * a.len + off + j;
            full[u] = a.vec && x[u] + 4 <= total;   // chunk % 4 == 0: the group stays in one row
        }
        int4 v[2][3];
        // unrolled over the (at most three) tensors so that the pointer arrays are
        // indexed with constants and stay in the parameter space
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int t = 0; t < 3; ++t)
                if (t < a.n_tensors && full[u]) v[u][t] = *reinterpret_cast<const int4 *>(a.src[t] + src[u]);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            if (x[u] >= total) continue;
#pragma unroll
            for (int t = 0; t < 3; ++t) {
                if (t >= a.n_tensors) break;
                if (full[u]) {
                    *reinterpret_cast<int4 *>(a.dst[t] + x[u]) = v[u][t];
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        if (x[u] + k >= total) break;
                        const int32_t rr = (x[u] + k) / chunk, jj = (x[u] + k) - rr * chunk;
                        a.dst[t][x[u] + k] = a.src[t][rr * a.len + off + jj];
                    }
                }
            }
        }
    }
}

// dst[r][j] = src[r][j] (j < len), else the fill; four consecutive outputs per
// thread (one 16-byte store when aligned: dst rows need not be, the group may
// straddle two rows).
__global__ void __launch_bounds__(kThreads) pad_kernel(PadArgs a)
{
    const int32_t total = a.rows * a.padded;
    const int lane = threadIdx.x & 31;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads * 4;
    // Two groups of four output positions per thread and iteration, all eight
    // loads issued before the stores. 64-bit loop index: the step past the last
    // group must not wrap (total < 2^31).
    for (int64_t xl = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) * 4; xl < total;
         xl += 2 * stride) {
        int32_t v[2][4];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t xu = xl + u * stride;
            // A warp's 128 consecutive outputs [X, X + 128) inside one row and
            // before its padding tail come from 128 consecutive source values:
            // one aligned 16-byte load per lane (plus the next vector for lane
            // 31) realigned by the warp-uniform shift with a shuffle. Every input
            // below is the same on all lanes, and X + 128 <= total keeps all of
            // them in this iteration, so the shuffles see the whole warp.
            const int64_t X = xu - 4 * lane;
            bool fast = a.vec && a.vec_src && X + 128 <= total;
            int32_t r0 = 0, j0 = 0;
            if (fast) {
                r0 = static_cast<int32_t>(X / a.padded);
                j0 = static_cast<int32_t>(X - static_cast<int64_t>(r0) * a.padded);
                fast = j0 + 128 <= a.len;
            }
            const int64_t S = static_cast<int64_t>(r0) * a.len + j0;   // source of output X
            const int64_t B = S & ~3ll;
            const int sh = static_cast<int>(S & 3);
            if (fast && sh && B + 132 > static_cast<int64_t>(a.rows) * a.len) fast = false;
            if (fast) {
                const int4 mine = *reinterpret_cast<const int4 *>(a.src + B + 4 * lane);
                int4 nxt;
                nxt.x = __shfl_down_sync(0xffffffffu, mine.x, 1);
                nxt.y = __shfl_down_sync(0xffffffffu, mine.y, 1);
                nxt.z = __shfl_down_sync(0xffffffffu, mine.z, 1);
                if (lane == 31 && sh) nxt = *reinterpret_cast<const int4 *>(a.src + B + 128);
                if (sh == 0) {
                    v[u][0] = mine.x; v[u][1] = mine.y; v[u][2] = mine.z; v[u][3] = mine.w;
                } else if (sh == 1) {
                    v[u][0] = mine.y; v[u][1] = mine.z; v[u][2] = mine.w; v[u][3] = nxt.x;
                } else if (sh == 2) {
                    v[u][0] = mine.z; v[u][1] = mine.w; v[u][2] = nxt.x; v[u][3] = nxt.y;
                } else {
                    v[u][0] = mine.w; v[u][1] = nxt.x; v[u][2] = nxt.y; v[u][3] = nxt.z;
                }
                continue;
            }
            // the row of the group's first position; a group crosses at most into the next row
            const int32_t x = xu < total ? static_cast<int32_t>(xu) : total;
            int32_t r = x / a.padded, j = x - r * a.padded;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int32_t q = x + k;
                if (k > 0 && ++j == a.padded) {
                    j = 0;
                    ++r;
                }
                if (q >= total) {
                    v[u][k] = 0;
                    continue;
                }
                v[u][k] = j < a.len ? a.src[static_cast<int64_t>(r) * a.len + j] : (a.count ? j - a.len : a.value);
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t xu = xl + u * stride;
            if (xu >= total) continue;
            const int32_t x = static_cast<int32_t>(xu);
            if (a.vec && x + 4 <= total) {
                *reinterpret_cast<int4 *>(a.dst + x) = make_int4(v[u][0], v[u][1], v[u][2], v[u][3]);
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (x + k < total) a.dst[x + k] = v[u][k];
            }
        }
    }
}

unsigned grid_for(int64_t groups, int num_sms)
{
    long long blocks = (groups + kThreads - 1) / kThreads;
    const long long cap = static_cast<long long>(num_sms > 0 ? num_sms : 1) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return static_cast<unsigned>(blocks);
}

}  // namespace

cudaError_t launch_unpack(const UnpackArgs &a, int num_sms, cudaStream_t stream)
{
    const int64_t total = static_cast<int64_t>(a.rows) * a.micro_bsz * a.seq_len;
    if (total == 0) return cudaSuccess;
    prof_begin(kProfUnpack, stream);
    unpack_kernel<<<grid_for((total + 3) / 4, num_sms), kThreads, 0, stream>>>(a);
    prof_end(kProfUnpack, stream);
    return cudaGetLastError();
}

cudaError_t launch_pad(const PadArgs &a, int num_sms, cudaStream_t stream)
{
    const int64_t total = static_cast<int64_t>(a.rows) * a.padded;
    if (total == 0) return cudaSuccess;
    prof_begin(kProfPad, stream);
    pad_kernel<<<grid_for((total + 3) / 4, num_sms), kThreads, 0, stream>>>(a);
    prof_end(kProfPad, stream);
    return cudaGetLastError();
}

cudaError_t launch_split(const SplitArgs &a, int num_sms, cudaStream_t stream)
{
    const int64_t total = static_cast<int64_t>(a.rows) * (a.len / a.sp_size);
    if (total == 0 || a.n_tensors == 0) return cudaSuccess;
    prof_begin(kProfSplit, stream);
    split_kernel<<<grid_for((total + 3) / 4, num_sms), kThreads, 0, stream>>>(a);
    prof_end(kProfSplit, stream);
    return cudaGetLastError();
}

}  // namespace spd
