// Tile scheduler: cu_seqlens -> a work list of 128-token tiles, longest first.
//
// Varlen attention splits the block-diagonal causal mask into one causal
// attention per document (page "Sample Packing: attention problems of
// long-sequence LLM training", section 5.1 "FlashAttention"), so a tile never
// spans two segments and only the tiles of each document's own causal
// triangle are ever visited. Listing work by decreasing cost
// (longest-processing-time first) lets the many short units fill in behind the
// few long ones when documents are very uneven.
//
// Forward (order 0): a unit is two consecutive q tiles t, t + 1 of a segment
// that one CTA computes together; q tile i reads kv tiles 0 .. i, so the cost is
// (t + 1) + (t + 2). Units are counting-sorted by cost over all units.
//
// Backward (order 1): kv tile t reads q tiles t .. n - 1 (cost n - t). In a
// long segment that is still short against one SM's share of the launch, the
// kv tiles p and n - 1 - p form one unit (cost n + 1, the same for every pair of the
// segment): the CTAs that take a document's pairs together also finish
// together and walk nearby q tiles meanwhile (the first tile of a pair upward
// from its diagonal, the second downward to its diagonal), so the Q / dO tiles
// and dQ rows they share stay in L2. Longer segments keep one unit per kv tile,
// so that the longest-first list can still balance them.
//
// One CTA: validates cu_seqlens, counts work per segment, sorts, writes the
// list; the sort and the list are built in parallel by all threads.
#include "internal.h"
#include "ptx.cuh"

namespace spd {
namespace {

constexpr int kThreads = 1024;
constexpr int kCostCap = 4 * kThreads - 1;  // costs above this share one bin (order among them is free)
constexpr int kPairMin = 16;                // backward: segments of at least this many tiles may be paired

__device__ long long block_scan_excl(long long v, long long *total, long long *sh)
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
        sh[lane] = w;
    }
    __syncthreads();
    long long r = (warp ? sh[warp - 1] : 0) + x - v;
    *total = sh[31];
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kThreads) schedule_kernel(const int32_t *cu, int32_t nsegs,
                                                            int64_t T, int order, int unit, int num_sms,
                                                            int *status, int32_t *count, Tile *tiles,
                                                            int32_t *tile_off, int32_t *seg_order, int heads)
{
    // The backward's preprocessing kernel depends on nothing computed here: let
    // it start at once (programmatic dependent launch; it waits for this grid
    // before it completes). No effect on kernels launched without the attribute.
    pdl_launch_dependents();
    __shared__ int bins[kCostCap + 1];
    __shared__ long long sh[33];
    __shared__ int bad_s;
    __shared__ unsigned long long total_cost;
    const int tid = threadIdx.x;
    if (tid == 0) {
        *status = 0;
        count[1] = 0;   // work counter of the persistent kernels
        count[2] = 0;   // long units per head
        bad_s = 0;
        total_cost = 0;
    }
    for (int c = tid; c <= kCostCap; c += kThreads) bins[c] = 0;
    __syncthreads();

    // Validate and count tiles per segment.
    bool bad = (tid == 0) && (cu[0] != 0 || static_cast<int64_t>(cu[nsegs]) != T);
    long long carry = 0;
    for (int base = 0; base < nsegs; base += kThreads) {
        int s = base + tid;
        long long n = 0;
        if (s < nsegs) {
            int a = cu[s], b = cu[s + 1];
            if (b <= a) bad = true;
            else n = ((b - a + kTile - 1) / kTile + unit - 1) / unit;
        }
        long long tot;
        long long e = block_scan_excl(n, &tot, sh) + carry;
        if (s < nsegs) tile_off[s] = static_cast<int32_t>(e);
        carry += tot;
    }
    if (bad) atomicOr(&bad_s, 1);
    if (tid == 0) tile_off[nsegs] = static_cast<int32_t>(carry);
    __syncthreads();
    if (bad_s) {
        if (tid == 0) {
            set_status(status, kErrBadSeqlens);
            *count = 0;
        }
        return;
    }
    if (order) {
        // ---------------------------------------------------- backward
        // A segment of n kv tiles is "paired" when it is long (n >= kPairMin:
        // its q tiles and dQ rows do not all stay in L2 while its kv tiles are
        // worked through) but its pair cost n + 1 is at most a quarter of one
        // SM's share of the whole launch: its kv tiles p and n - 1 - p form one
        // unit (the middle tile of an odd n stays single), and its pairs take
        // consecutive slots of their cost bin, in order. Other segments keep one
        // unit per kv tile (cost n - t): short ones gain nothing from pairing,
        // and very long ones need the finer grain for the longest-first list to
        // balance them. Units are counting-sorted by cost over everything.
        unsigned long long my_cost = 0;
        for (int sg = tid; sg < nsegs; sg += kThreads) {
            const long long n = (cu[sg + 1] - cu[sg] + kTile - 1) / kTile;
            my_cost += static_cast<unsigned long long>(n * (n + 1) / 2);
        }
        atomicAdd(&total_cost, my_cost);
        __syncthreads();
        const long long c_pair =
            max(2LL, static_cast<long long>(total_cost) * heads / (4LL * num_sms));
        auto paired = [&](long long n) { return n >= kPairMin && n + 1 <= c_pair; };
        // counts: one per single tile, floor(n / 2) per paired segment in bin n + 1
        for (int sg = tid; sg < nsegs; sg += kThreads) {
            const long long n = (cu[sg + 1] - cu[sg] + kTile - 1) / kTile;
            if (paired(n)) atomicAdd(&bins[static_cast<int>(min(n + 1, static_cast<long long>(kCostCap)))],
                                     static_cast<int>(n / 2));
        }
        for (int i = tid; i < static_cast<int>(carry); i += kThreads) {
            int lo = 0, hi = nsegs;  // largest segment with tile_off[s] <= i
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (tile_off[mid] <= i) lo = mid;
                else hi = mid;
            }
            const int n = (cu[lo + 1] - cu[lo] + kTile - 1) / kTile, t = i - tile_off[lo];
            if (!paired(n) || (n & 1 && 2 * t + 1 == n)) atomicAdd(&bins[min(n - t, kCostCap)], 1);
        }
        __syncthreads();
        {
            const long long c_long = max(4LL, (2LL * static_cast<long long>(total_cost) + num_sms - 1) / num_sms);
            int n_long = 0;
            if (c_long <= kCostCap)
                for (int c = static_cast<int>(c_long) + tid; c <= kCostCap; c += kThreads) n_long += bins[c];
            if (n_long) atomicAdd(&count[2], n_long);
            int v[4], sum = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                v[k] = bins[kCostCap - (4 * tid + k)];
                sum += v[k];
            }
            long long tot;
            long long run = block_scan_excl(sum, &tot, sh);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                bins[kCostCap - (4 * tid + k)] = static_cast<int>(run);
                run += v[k];
            }
            if (tid == 0) *count = static_cast<int32_t>(tot);
        }
        __syncthreads();
        // slots: a paired segment reserves floor(n / 2) consecutive ones
        for (int sg = tid; sg < nsegs; sg += kThreads) {
            const long long n = (cu[sg + 1] - cu[sg] + kTile - 1) / kTile;
            if (paired(n))
                seg_order[sg] = atomicAdd(&bins[static_cast<int>(min(n + 1, static_cast<long long>(kCostCap)))],
                                          static_cast<int>(n / 2));
        }
        __syncthreads();
        for (int i = tid; i < static_cast<int>(carry); i += kThreads) {
            int lo = 0, hi = nsegs;
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (tile_off[mid] <= i) lo = mid;
                else hi = mid;
            }
            const int n = (cu[lo + 1] - cu[lo] + kTile - 1) / kTile, t = i - tile_off[lo];
            Tile w;
            w.seg_start = cu[lo];
            w.seg_end = cu[lo + 1];
            if (paired(n) && 2 * t + 1 < n) {          // first tile of pair t
                w.t = t;
                w.cost = n + 1;
                tiles[seg_order[lo] + t] = w;
            } else if (!paired(n) || 2 * t + 1 == n) {  // a single tile
                w.t = t | kSingleTile;
                w.cost = n - t;
                tiles[atomicAdd(&bins[min(n - t, kCostCap)], 1)] = w;
            }
        }
        return;
    }

    const int ntiles = static_cast<int>(carry);

    auto locate = [&](int i, int &s, int &t, int &n, int &cost) {
        int lo = 0, hi = nsegs;  // largest s with tile_off[s] <= i
        while (hi - lo > 1) {
            int mid = (lo + hi) >> 1;
            if (tile_off[mid] <= i) lo = mid;
            else hi = mid;
        }
        s = lo;
        t = (i - tile_off[s]) * unit;                       // first tile of the unit
        n = (cu[s + 1] - cu[s] + kTile - 1) / kTile;        // tiles of the segment
        cost = (t + 1) + (unit > 1 && t + 1 < n ? t + 2 : 0);  // kv tiles of each q tile
    };

    unsigned long long my_cost = 0;
    for (int i = tid; i < ntiles; i += kThreads) {
        int s, t, n, cost;
        locate(i, s, t, n, cost);
        atomicAdd(&bins[min(cost, kCostCap)], 1);
        my_cost += static_cast<unsigned long long>(cost);
    }
    atomicAdd(&total_cost, my_cost);
    __syncthreads();
    // Long units: cost at least twice one SM's share of a head's total. They are
    // taken first, across heads (see unit_of), so none starts late in the list.
    // (Costs above kCostCap share a bin and are not told apart: then none is long.)
    {
        const long long c_long = max(4LL, (2LL * static_cast<long long>(total_cost) + num_sms - 1) / num_sms);
        int n_long = 0;
        if (c_long <= kCostCap)
            for (int c = static_cast<int>(c_long) + tid; c <= kCostCap; c += kThreads) n_long += bins[c];
        if (n_long) atomicAdd(&count[2], n_long);
    }
    // Descending exclusive scan: bins[c] <- number of tiles with a larger cost.
    // Thread tid owns costs kCostCap - 4 tid .. kCostCap - 4 tid - 3.
    {
        int v[4], sum = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[k] = bins[kCostCap - (4 * tid + k)];
            sum += v[k];
        }
        long long tot;
        long long run = block_scan_excl(sum, &tot, sh);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            bins[kCostCap - (4 * tid + k)] = static_cast<int>(run);
            run += v[k];
        }
    }
    __syncthreads();
    for (int i = tid; i < ntiles; i += kThreads) {
        int s, t, n, cost;
        locate(i, s, t, n, cost);
        int pos = atomicAdd(&bins[min(cost, kCostCap)], 1);
        Tile w;
        w.seg_start = cu[s];
        w.seg_end = cu[s + 1];
        w.t = t;
        w.cost = cost;
        tiles[pos] = w;
    }
    if (tid == 0) *count = ntiles;
}

}  // namespace

size_t schedule_ws_bytes(int64_t total_tokens, int32_t num_segs)
{
    return kWsHeader + align_up(sizeof(Tile) * static_cast<size_t>(max_tiles(total_tokens, num_segs)), 256) +
           align_up(sizeof(int32_t) * static_cast<size_t>(num_segs + 1), 256);
}

cudaError_t launch_schedule(const int32_t *cu_seqlens, int32_t num_segs, int64_t total_tokens,
                            int order, int unit, int num_sms, int heads, void *ws, int32_t *seg_order,
                            cudaStream_t stream)
{
    if (order && !seg_order) return cudaErrorInvalidValue;
    char *base = reinterpret_cast<char *>(ws);
    int *status = reinterpret_cast<int *>(base);
    int32_t *count = reinterpret_cast<int32_t *>(base) + 1;
    Tile *tiles = reinterpret_cast<Tile *>(base + kWsHeader);
    int32_t *tile_off = reinterpret_cast<int32_t *>(
        base + kWsHeader + align_up(sizeof(Tile) * static_cast<size_t>(max_tiles(total_tokens, num_segs)), 256));
    schedule_kernel<<<1, kThreads, 0, stream>>>(cu_seqlens, num_segs, total_tokens, order, unit,
                                                num_sms > 0 ? num_sms : 1, status, count, tiles, tile_off,
                                                seg_order, heads > 0 ? heads : 1);
    return cudaGetLastError();
}

}  // namespace spd
