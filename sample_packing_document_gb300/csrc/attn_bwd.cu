// Backward of the document-masked causal attention.
//
// With P_ij = exp(S_ij - LSE_i), D_i = dO_i . O_i and dS_ij = P_ij (dP_ij - D_i),
// dP_ij = dO_i . v_j (the exact gradient of the masked softmax):
//   dV_j = sum_i P_ij dO_i,   dK_j = scale sum_i dS_ij q_i,   dQ_i = scale sum_j dS_ij k_j,
// summed over the q heads that share a kv head (GQA). As in the forward pass,
// only tiles inside a document's own causal triangle are visited (page "Sample
// Packing: attention problems of long-sequence LLM training", section 5.1
// "FlashAttention").
//
// Three launches:
//   bwd_pre_kernel   D_i = rowsum(dO * O) (fp32) and zeroes the fp32 dQ
//                    accumulator, laid out [Hq][d / 32][T][32]; runs beside the
//                    tile schedule (programmatic dependent launch).
//   attn_bwd_kernel  persistent; a work unit is a (kv head, 128-row kv tile):
//                    K, V stay in shared memory while the CTA walks every (q
//                    head of the group, q tile from the diagonal to the segment
//                    end, upward or downward). Per step, five
//                    tcgen05 MMAs with fp32 accumulation in TMEM:
//                      S^T = K Q^T           region A (P^T is then written over it, bf16)
//                      dP^T = V dO^T         region B
//                      dV += P^T dO          region C (P^T read from TMEM)
//                      dK += dS^T Q          region E (dS^T from shared memory)
//                      dQ_part = dS K        region B (once dP^T has been read), then
//                                            TMA reduce-add into the HBM accumulator.
//   bwd_dq_kernel    dq = scale * accumulator, in the output layout and type.
//
// Warp roles (640 threads: four compute warpgroups, and one for the TMA
// producer, the MMA issuer and two idle warps). Compute warp w works on TMEM
// lanes 32 (w % 4) .. +31 (kv rows; q rows for the dQ read-out):
//   warps 0-7   "P": P^T(i) = exp(S^T(i) * scale - LSE) on one half of the
//               columns of region A, written back into it as bf16 (the P^T
//               columns of a half sit in the first half of that half's S^T
//               columns). Nothing else, so P(i+1) starts as soon as S^T(i+1) is
//               in.
//   warps 8-15  "dS": dS^T(i) = P^T(i) (dP^T(i) - D) into shared memory, then the
//               dQ(i) read-out (two 32 x 32 chunks per warp for d = 128, staged
//               in the spent Q(i) stage and in the dS buffer and added by the TMA
//               engine); at the end of a unit the dV and dK stores.
//   warp 16     TMA producer; warp 17 issues the MMAs in the order
//               dV(i), dK(i), dQ(i), S(i+1), dP(i+1), dV(i+1), ...
#include "internal.h"
#include "ptx.cuh"

#include <type_traits>

namespace spd {
namespace {

constexpr int kThreads = 640;        // 16 compute warps (4 warpgroups) + producer + MMA issuer + 2 idle warps
// Register split (setmaxnreg, per warpgroup): the launch gives 96 per thread
// (640 x 96 = 61440); the warpgroup of the producer / MMA issuer drops to 48, the
// two P warpgroups rise to 112 and the two dS warpgroups to 104:
// 2 x 128 x 112 + 2 x 128 x 104 + 128 x 48 = 61440. Per SM sub-partition (one
// warp of each warpgroup): (112 + 112 + 104 + 104 + 48) x 32 = 15360 <= 16384.
constexpr uint32_t kPRegs = 112, kDsRegs = 104, kControlRegs = 48;
constexpr int kPWarps = 8, kDsWarps = 8;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAtom = 128 * 128;
constexpr int kQStages = 2;   // the per-stage counters below are selected with (index & 1)

template <int D>
struct BwdSmem {
    uint8_t k[D / 64][kAtom];
    uint8_t v[D / 64][kAtom];
    uint8_t q[kQStages][D / 64][kAtom];
    uint8_t dout[kQStages][D / 64][kAtom];
    uint8_t ds[2][kAtom];            // dS^T: [128 kv rows][128 q cols]
    float lse2[2][128];              // LSE * log2(e) of the step's q columns
    float delta[2][128];             // D of the step's q columns
    uint64_t kv_full, kv_empty;
    uint64_t q_full[kQStages], q_empty[kQStages], do_full[kQStages], do_empty[kQStages];
    uint64_t s_full, dp_full, p_full, ds_full, dq_full, dq_free;
    uint64_t acc_full, acc_free;     // unit's MMAs complete / its dV, dK read out
    uint64_t cols_l[2], cols_d[2];   // the step's lse2 / delta written
    uint64_t unit_full[2], unit_empty[2];
    int4 unit[2];                    // work unit in flight: {kv head (-1: no more work), seg_start, seg_end, kv tile}
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ bool wait_drain(uint64_t *bar, uint32_t parity)
{
    uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    return true;
}

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          int *status)
{
    bool w = mbar_wait(bar, parity, abort_flag, status);
    return __all_sync(0xffffffffu, w);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }


// ------------------------------------------------------------------ preprocess
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const uint16_t *__restrict__ out,
                                                      const uint16_t *__restrict__ dout, float *delta,
                                                      float *dq_acc, int32_t T, int32_t Hq)
{
    // 8 threads per (token, head) row; each covers D / 8 elements. A warp
    // takes 4 rows per iteration and every lane runs the same iterations, so
    // the 8-lane shuffles always see a full warp.
    constexpr int kPer = D / 8;
    const long long rows = static_cast<long long>(T) * Hq;
    const int lane = threadIdx.x & 31, sub = lane & 7;
    const long long warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    for (long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w * 4 < rows;
         w += warps) {
        const long long row = w * 4 + (lane >> 3);
        const bool active = row < rows;
        float acc = 0.f;
        if (active) {
            const uint4 *o4 = reinterpret_cast<const uint4 *>(out + row * D + sub * kPer);
            const uint4 *d4 = reinterpret_cast<const uint4 *>(dout + row * D + sub * kPer);
#pragma unroll
            for (int c = 0; c < kPer / 8; ++c) {
                uint4 a = o4[c], b = d4[c];
                const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    acc += bf16_lo(aw[e]) * bf16_lo(bw[e]) + bf16_hi(aw[e]) * bf16_hi(bw[e]);
            }
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        acc += __shfl_xor_sync(0xffffffffu, acc, 4);
        if (!active) continue;
        const long long i = row / Hq;
        const int h = static_cast<int>(row % Hq);
        const long long hi = static_cast<long long>(h) * T + i;
        if (sub == 0) delta[hi] = acc;
    }
    // zero the fp32 dQ accumulator (any layout: Hq * T * D floats)
    float4 *z = reinterpret_cast<float4 *>(dq_acc);
    const long long n4 = rows * (D / 4);
    for (long long x = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; x < n4;
         x += static_cast<long long>(gridDim.x) * blockDim.x)
        z[x] = make_float4(0.f, 0.f, 0.f, 0.f);
    // Launched as a programmatic dependent of the tile schedule, which it does
    // not read: it runs beside it, and does not complete before it, so the main
    // kernel (a plain launch after this one) sees the finished schedule.
    pdl_wait();
}

// ------------------------------------------------------------------ dq convert
template <int D>
__global__ void __launch_bounds__(256) bwd_dq_kernel(const float *__restrict__ dq_acc, void *dq,
                                                     int grad_fp32, float scale, int32_t T, int32_t Hq)
{
    // one thread per 8 consecutive elements of one (token, head) row
    const long long n8 = static_cast<long long>(T) * Hq * (D / 8);
    for (long long x = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; x < n8;
         x += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long row = x / (D / 8);  // token-major row = i * Hq + h
        const int c8 = static_cast<int>(x % (D / 8));
        const long long i = row / Hq;
        const int h = static_cast<int>(row % Hq);
        // accumulator layout [h][d / 32][i][32]
        const int dblk = c8 >> 2, din = (c8 & 3) * 8;
        const float4 *src = reinterpret_cast<const float4 *>(
            dq_acc + ((static_cast<long long>(h) * (D / 32) + dblk) * T + i) * 32 + din);
        float4 a = src[0], b = src[1];
        float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        if (grad_fp32) {
            float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(dq) + row * D + c8 * 8);
            dst[0] = make_float4(v[0] * scale, v[1] * scale, v[2] * scale, v[3] * scale);
            dst[1] = make_float4(v[4] * scale, v[5] * scale, v[6] * scale, v[7] * scale);
        } else {
            uint4 w = make_uint4(pack_bf16x2(v[0] * scale, v[1] * scale), pack_bf16x2(v[2] * scale, v[3] * scale),
                                 pack_bf16x2(v[4] * scale, v[5] * scale), pack_bf16x2(v[6] * scale, v[7] * scale));
            *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(dq) + row * D + c8 * 8) = w;
        }
    }
}

// A work unit in flight: {kv head (-1: no more work), segment start, segment
// end, kv tile | kDescBit}. Kv tile t reads q tiles t .. n - 1 of its segment,
// in ascending order, or in descending order (n - 1 down to t) when kDescBit
// is set: the second kv tile of a scheduled pair walks down, so that the CTAs
// working through one document's pairs touch nearby q tiles at any moment.
constexpr int kDescBit = 1 << 30;
__device__ __forceinline__ int seg_tiles(const int4 &u) { return (u.z - u.y + kTile - 1) / kTile; }
__device__ __forceinline__ int unit_kv_tile(const int4 &u) { return u.w & (kDescBit - 1); }
__device__ __forceinline__ int unit_nq(const int4 &u) { return seg_tiles(u) - unit_kv_tile(u); }
// q tile (inside the segment) of the unit's j-th q-tile step, 0 <= j < unit_nq
__device__ __forceinline__ int unit_q_tile(const int4 &u, int j)
{
    return (u.w & kDescBit) ? seg_tiles(u) - 1 - j : unit_kv_tile(u) + j;
}

// dV (P warps, IS_P) or dK (dS warps) rows of a finished unit's kv tile: the
// calling warp's 32 rows (TMEM lanes 32 quarter ..), d columns [half * D/2,
// half * D/2 + D/2), read from TMEM at `acc`. With bf16 grads and d = 128, a
// quarter that lies wholly inside the segment is converted into the warp's
// staging slot (free once the TMA engine has read the unit's last dQ chunk from
// it) and leaves in one TMA store, so the HBM writes are whole lines; a quarter
// that reaches past the segment end is written by plain stores of its live rows
// (a box must not touch the next segment). Called once per unit.
template <int D, bool IS_P>
__device__ __forceinline__ void store_acc_rows(const AttnBwdArgs &a, uint32_t acc, int4 u, int quarter, int half,
                                            const uint8_t *slot)
{
    const int lane = threadIdx.x & 31;
    const int row0 = u.y + unit_kv_tile(u) * kTile + quarter * 32;
    const int kj = row0 + lane;
    const float mul = IS_P ? 1.f : a.scale;
    if (D == 128 && a.store_tma && row0 + 32 <= u.z) {
        const uint32_t slot_addr = smem_u32(slot);
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            uint32_t v[32];
            tmem_ld32(acc + c * 32, v);
            tmem_wait_ld();
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
                w[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
            // row `lane`, d columns 32c .. 32c+31: 16-byte chunks 4c .. 4c+3, 128-byte swizzle
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
                st_shared_v4(slot_addr + lane * 128 + (((c * 4 + v4) ^ (lane & 7)) << 4), w[4 * v4], w[4 * v4 + 1],
                             w[4 * v4 + 2], w[4 * v4 + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_3d(IS_P ? &a.tm_dv : &a.tm_dk, slot, half * 64, u.x, row0);
            bulk_commit_group();
        }
        return;
    }
    const bool live = kj < u.z;
    const size_t orow = (static_cast<size_t>(kj) * a.Hkv + u.x) * D + half * (D / 2);
    void *base = IS_P ? a.dv : a.dk;
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
        uint32_t v[32];
        tmem_ld32(acc + c * 32, v);
        tmem_wait_ld();
        if (!live) continue;
        if (a.grad_fp32) {
            float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(base) + orow + c * 32);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                dst[e] = make_float4(__uint_as_float(v[4 * e]) * mul, __uint_as_float(v[4 * e + 1]) * mul,
                                     __uint_as_float(v[4 * e + 2]) * mul, __uint_as_float(v[4 * e + 3]) * mul);
        } else {
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(base) + orow + c * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                dst[e] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * e]) * mul, __uint_as_float(v[8 * e + 1]) * mul),
                                    pack_bf16x2(__uint_as_float(v[8 * e + 2]) * mul, __uint_as_float(v[8 * e + 3]) * mul),
                                    pack_bf16x2(__uint_as_float(v[8 * e + 4]) * mul, __uint_as_float(v[8 * e + 5]) * mul),
                                    pack_bf16x2(__uint_as_float(v[8 * e + 6]) * mul, __uint_as_float(v[8 * e + 7]) * mul));
        }
    }
}

// ------------------------------------------------------------------ main kernel

template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_bwd_kernel(const __grid_constant__ AttnBwdArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    BwdSmem<D> &sm = *reinterpret_cast<BwdSmem<D> *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (*reinterpret_cast<volatile int *>(a.status) != 0) return;
    if (smem_u32(smem_raw) & 1023u) {  // swizzled operand atoms need 1024-byte alignment
        if (threadIdx.x == 0) set_status(a.status, kErrTimeout);
        return;
    }
    const int group = a.Hq / a.Hkv;

    if (threadIdx.x == 0) {
        mbar_init(&sm.kv_full, 1);
        mbar_init(&sm.kv_empty, 1);
        for (int s = 0; s < kQStages; ++s) {
            mbar_init(&sm.q_full[s], 1);
            mbar_init(&sm.q_empty[s], kDsWarps);   // the dS warps, once their staged dQ chunks have been read
            mbar_init(&sm.do_full[s], 1);
            mbar_init(&sm.do_empty[s], 1);
        }
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.dp_full, 1);
        mbar_init(&sm.p_full, 32 * kPWarps);
        mbar_init(&sm.ds_full, 32 * kDsWarps);
        mbar_init(&sm.dq_full, 1);
        mbar_init(&sm.dq_free, 32 * kDsWarps);
        mbar_init(&sm.acc_full, 1);
        mbar_init(&sm.acc_free, kDsWarps);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.cols_l[b], 128);
            mbar_init(&sm.cols_d[b], 128);
            mbar_init(&sm.unit_full[b], 1);
            mbar_init(&sm.unit_empty[b], 1 + kPWarps + kDsWarps);  // MMA thread + one lane per compute warp
        }
        mbar_init(&sm.drain, 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 17) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 16 && lane == 0) {
        if (a.store_tma) {
            tma_prefetch_desc(&a.tm_dk);
            tma_prefetch_desc(&a.tm_dv);
        }
        tma_prefetch_desc(&a.tm_q);
        tma_prefetch_desc(&a.tm_k);
        tma_prefetch_desc(&a.tm_v);
        tma_prefetch_desc(&a.tm_do);
        tma_prefetch_desc(&a.tm_dqacc);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    volatile int *abort_flag = &sm.abort_flag;
    constexpr uint32_t kTileBytes = 128 * D * 2;
    constexpr uint32_t kA = 0, kB = 128, kC = 256, kE = 256 + D;

    // Work unit `it` from the two-slot ring, for a whole compute warp.
    auto warp_unit = [&](int it, int4 &d) -> bool {
        const int slot = it & 1;
        if (!warp_wait(&sm.unit_full[slot], (it >> 1) & 1, abort_flag, a.status)) return false;
        d = sm.unit[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.unit_empty[slot]);
        return true;
    };

    if (warp >= 16) {
    setmaxnreg_dec<kControlRegs>();
    if (warp == 16) {
        // ------------------------------------------------------------ producer
        // Takes work units (kv head, pair of kv tiles) from the shared counter in
        // list order (unit_of): the few units much longer than a kv head's share
        // of an SM first, across kv heads; then kv-head-major, so the CTAs of one
        // kv head run together and the Q / dO tiles they share and the dQ rows
        // they add into stay in L2; longest segment first inside a head, a
        // segment's pairs in order. Every pair of a segment costs the same, so the
        // CTAs on one document stay in step, the first tiles walking up and the
        // second ones down through nearby q tiles. Q / dO stream through a
        // 2-stage ring that runs on across units; the next unit's K / V are
        // pulled into L2 as soon as it is taken and copied in once the last MMA
        // reading K has completed.
        if (lane == 0) {
            const int n_tiles = *a.tile_count;
            const int total_units = n_tiles * a.Hkv;
            const int n_long = *a.long_count;
            int gi = 0, kv_loads = 0;
            int last_q[kQStages], last_do[kQStages];
            for (int s = 0; s < kQStages; ++s) last_q[s] = last_do[s] = -1;
            auto load_step = [&](const int4 &d, int nq, int i, int gs) -> bool {
                const int st = gs % kQStages, u = gs / kQStages;
                const int h = d.x * group + i / nq;
                const int q0 = d.y + unit_q_tile(d, i % nq) * kTile;
                if (u > 0 && !mbar_wait(&sm.q_empty[st], (u - 1) & 1, abort_flag, a.status)) return false;
                mbar_arrive_expect_tx(&sm.q_full[st], kTileBytes);
                for (int c = 0; c < D / 64; ++c) tma_load_3d(sm.q[st][c], &a.tm_q, c * 64, h, q0, &sm.q_full[st]);
                if (st) last_q[1] = u;   // constant indices keep the arrays in registers
                else last_q[0] = u;
                if (u > 0 && !mbar_wait(&sm.do_empty[st], (u - 1) & 1, abort_flag, a.status)) return false;
                mbar_arrive_expect_tx(&sm.do_full[st], kTileBytes);
                for (int c = 0; c < D / 64; ++c)
                    tma_load_3d(sm.dout[st][c], &a.tm_do, c * 64, h, q0, &sm.do_full[st]);
                if (st) last_do[1] = u;
                else last_do[0] = u;
                return true;
            };
            bool ok = true;
            int4 pending = make_int4(-1, 0, 0, 0);   // second kv tile of the pair taken last
            for (int it = 0; ok; ++it) {
                const int slot = it & 1;
                if (it >= 2 && !mbar_wait(&sm.unit_empty[slot], ((it >> 1) - 1) & 1, abort_flag, a.status)) break;
                int4 d = make_int4(-1, 0, 0, 0);
                if (pending.x >= 0 && !*abort_flag) {
                    d = pending;
                    pending.x = -1;
                } else {
                    // A scheduled unit is one kv tile, or the pair of kv tiles p and
                    // n - 1 - p of one segment: n + 1 q-tile steps together, the same
                    // for every pair of the segment.
                    const int w = *abort_flag ? total_units : atomicAdd(a.work_counter, 1);
                    if (w < total_units) {
                        int head, idx;
                        unit_of(w, n_tiles, n_long, a.Hkv, head, idx);
                        const Tile tl = a.tiles[idx];
                        const int n = (tl.seg_end - tl.seg_start + kTile - 1) / kTile;
                        d = make_int4(head, tl.seg_start, tl.seg_end, tl.t & ~kSingleTile);
                        if (!(tl.t & kSingleTile))
                            pending = make_int4(head, tl.seg_start, tl.seg_end, (n - 1 - tl.t) | kDescBit);
                    }
                }
                sm.unit[slot] = d;
                mbar_arrive(&sm.unit_full[slot]);
                if (d.x < 0) break;
                const int k0 = d.y + unit_kv_tile(d) * kTile;
                for (int c = 0; c < D / 64; ++c) {
                    tma_prefetch_l2_3d(&a.tm_k, c * 64, d.x, k0);
                    tma_prefetch_l2_3d(&a.tm_v, c * 64, d.x, k0);
                }
                const int nq = unit_nq(d);
                const int nsteps = group * nq;
                if (!load_step(d, nq, 0, gi)) break;
                if (it > 0 && !mbar_wait(&sm.kv_empty, (it - 1) & 1, abort_flag, a.status)) break;
                if (!(a.debug_skip && it == 0)) {   // test hook: kv_full of the first unit never completes
                    mbar_arrive_expect_tx(&sm.kv_full, 2 * kTileBytes);
                    for (int c = 0; c < D / 64; ++c) {
                        tma_load_3d(sm.k[c], &a.tm_k, c * 64, d.x, k0, &sm.kv_full);
                        tma_load_3d(sm.v[c], &a.tm_v, c * 64, d.x, k0, &sm.kv_full);
                    }
                    ++kv_loads;
                }
                for (int i = 1; i < nsteps; ++i)
                    if (!load_step(d, nq, i, gi + i)) { ok = false; break; }
                gi += nsteps;
            }
            if (*abort_flag) {
                // Let the copies still in flight land before the CTA exits.
                if (kv_loads > 0) wait_drain(&sm.kv_full, (kv_loads - 1) & 1);
                for (int s = 0; s < kQStages; ++s) {
                    if (last_q[s] >= 0) wait_drain(&sm.q_full[s], last_q[s] & 1);
                    if (last_do[s] >= 0) wait_drain(&sm.do_full[s], last_do[s] & 1);
                }
            }
        }
    } else if (warp == 17) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_ss = idesc_bf16(128, 128, 0, 0);  // S^T, dP^T
            constexpr uint32_t id_kn = idesc_bf16(128, D, 0, 1);    // dV (A in TMEM), dK
            constexpr uint32_t id_mn = idesc_bf16(128, D, 1, 1);    // dQ
            // base descriptors; the k-steps add a start-address step inside the MMA block
            const uint64_t kd_k = sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);      // K, K-major (S^T A operand)
            const uint64_t kd_v = sdesc_sw128(smem_u32(sm.v[0]), 16, 1024);      // V, K-major (dP^T A operand)
            const uint64_t kd_mn = sdesc_sw128(smem_u32(sm.k[0]), kAtom, 1024);  // K, MN-major (dQ B operand)
            const uint64_t dsd_k = sdesc_sw128(smem_u32(sm.ds[0]), 16, 1024);    // dS^T, K-major (dK A operand)
            const uint64_t dsd_mn = sdesc_sw128(smem_u32(sm.ds[0]), kAtom, 1024); // dS, MN-major (dQ A operand)
            int do_commits[kQStages] = {};
            int kv_commits = 0;
            auto issue_s = [&](int gs) -> bool {   // S^T = K Q^T into A
                const int st = gs % kQStages;
                if (!mbar_wait(&sm.q_full[st], (gs / kQStages) & 1, abort_flag, a.status)) return false;
                tc_fence_after();
                const uint64_t qd = sdesc_sw128(smem_u32(sm.q[st][0]), 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t step = ((kk >> 2) * kAtom + (kk & 3) * 32) >> 4;
                    umma_bf16_step(tmem + kA, kd_k, qd, step, step, id_ss, kk > 0 ? 1u : 0u);
                }
                umma_commit(&sm.s_full);
                return true;
            };
            auto issue_dp = [&](int gs) -> bool {  // dP^T = V dO^T into B, once the previous dQ left B
                const int st = gs % kQStages;
                if (!mbar_wait(&sm.do_full[st], (gs / kQStages) & 1, abort_flag, a.status)) return false;
                if (gs > 0 && !mbar_wait(&sm.dq_free, (gs - 1) & 1, abort_flag, a.status)) return false;
                tc_fence_after();
                const uint64_t dod = sdesc_sw128(smem_u32(sm.dout[st][0]), 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t step = ((kk >> 2) * kAtom + (kk & 3) * 32) >> 4;
                    umma_bf16_step(tmem + kB, kd_v, dod, step, step, id_ss, kk > 0 ? 1u : 0u);
                }
                umma_commit(&sm.dp_full);
                return true;
            };
            bool ok = true;
            int gi = 0;
            for (int it = 0; ok; ++it) {
                const int slot = it & 1;
                if (!mbar_wait(&sm.unit_full[slot], (it >> 1) & 1, abort_flag, a.status)) break;
                const int4 d = sm.unit[slot];
                mbar_arrive(&sm.unit_empty[slot]);
                if (d.x < 0) break;
                const int nsteps = group * unit_nq(d);
                ok = mbar_wait(&sm.kv_full, it & 1, abort_flag, a.status) && issue_s(gi) && issue_dp(gi);
                for (int i = 0; ok && i < nsteps; ++i, ++gi) {
                    const int st = gi % kQStages;
                    const uint32_t ph = gi & 1;
                    // dV += P^T dO: P^T in TMEM over S^T (M = kv, K = q), dO MN-major.
                    // The first step of a unit overwrites dV (accumulate = 0).
                    if (!mbar_wait(&sm.p_full, ph, abort_flag, a.status)) { ok = false; break; }
                    // the first dV of a unit overwrites the last unit's dV: read out by then
                    if (i == 0 && it > 0 && !mbar_wait(&sm.acc_free, (it - 1) & 1, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    {
                        const uint64_t dod = sdesc_sw128(smem_u32(sm.dout[st][0]), kAtom, 1024);
#pragma unroll
                        for (int kk = 0; kk < 128 / 16; ++kk)
                            // P^T q columns 16kk .. 16kk+15 sit at TMEM column 64 (kk / 4) + 8 (kk % 4)
                            umma_bf16_ts_step(tmem + kC, tmem + kA + (kk >> 2) * 64 + (kk & 3) * 8, dod,
                                              kk * (2048 >> 4), id_kn, (i > 0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit(&sm.do_empty[st]);
                    if (st) ++do_commits[1];   // constant indices keep the counts in registers
                    else ++do_commits[0];
                    // dK += dS^T Q (M = kv), dQ_part = dS K (M = q) into B
                    if (!mbar_wait(&sm.ds_full, ph, abort_flag, a.status)) { ok = false; break; }
                    tc_fence_after();
                    {
                        const uint64_t qd_mn = sdesc_sw128(smem_u32(sm.q[st][0]), kAtom, 1024);
#pragma unroll
                        for (int kk = 0; kk < 128 / 16; ++kk)
                            umma_bf16_step(tmem + kE, dsd_k, qd_mn, ((kk >> 2) * kAtom + (kk & 3) * 32) >> 4,
                                           kk * (2048 >> 4), id_kn, (i > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                        for (int kk = 0; kk < 128 / 16; ++kk)
                            umma_bf16_step(tmem + kB, dsd_mn, kd_mn, kk * (2048 >> 4), kk * (2048 >> 4), id_mn,
                                           kk > 0 ? 1u : 0u);
                    }
                    umma_commit(&sm.dq_full);
                    // next step: S^T over P^T (dV ran before it and the dS warps read
                    // P^T before ds_full), then dP^T
                    if (i + 1 < nsteps && !(issue_s(gi + 1) && issue_dp(gi + 1))) { ok = false; break; }
                }
                if (!ok) break;
                umma_commit(&sm.kv_empty);   // K / V fully read: the next unit's may load
                umma_commit(&sm.acc_full);   // dV / dK of the unit final
                ++kv_commits;
            }
            umma_commit(&sm.drain);
            wait_drain(&sm.drain, 0);
            for (int s = 0; s < kQStages; ++s)
                if (do_commits[s] > 0) wait_drain(&sm.do_empty[s], (do_commits[s] - 1) & 1);
            if (kv_commits > 0) wait_drain(&sm.kv_empty, (kv_commits - 1) & 1);
        }
    }
    } else {
        // ------------------------------------------------------------ compute warps
        // One body, instantiated for the P warps and for the dS warps.
        auto compute = [&](auto role) {
        constexpr bool is_p = decltype(role)::value;
        const int w = is_p ? warp : warp - kPWarps;
        const int quarter = w & 3, half = w >> 2;
        const int t = quarter * 32 + lane;                        // kv row / q row = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const int col0 = half * 64;                               // this warp's 64 q columns
        const float sl2 = a.scale_log2;
        const uint64_t sl2_2 = f2_pack(sl2, sl2);
        const uint32_t ds_addr = smem_u32(sm.ds[0]);
        const bool loader = half == 0;                            // loads the step's LSE / D column t
        auto col_term = [&](const int4 &u, int i) -> float {
            const int nq = unit_nq(u);
            const int h = u.x * group + i / nq;
            const int qi = u.y + unit_q_tile(u, i % nq) * kTile + t;
            if (qi >= a.total_tokens) return 0.f;
            const size_t x = static_cast<size_t>(h) * a.total_tokens + qi;
            return is_p ? -a.lse[x] * 1.4426950408889634f : a.delta[x];   // P warps keep -LSE log2 e
        };
        // dS warps' staging slots: A in the step's spent Q stage (d = 128), B in
        // the dS buffer (free once dK / dQ, its readers, have completed).
        auto slot_a = [&](int gs) -> uint8_t * {
            return D == 128 ? sm.q[gs % kQStages][0] + (quarter + 4 * half) * 4096
                            : sm.ds[0] + (quarter + 4 * half) * 4096;
        };
        uint8_t *const slot_b = sm.ds[0] + (quarter + 4 * half) * 4096;
        // Stages one [32 rows][32 cols] chunk of dQ (registers v, d columns
        // 32 chunk ..) in the 128-byte-swizzled layout and lets the TMA engine add
        // it into the accumulator in the background. Rows past the segment carry
        // exact zeros.
        auto dq_stage = [&](const uint32_t (&v)[32], uint8_t *stage, int chunk, int q0, int seg_end, int h) {
            const uint32_t stage_addr = smem_u32(stage);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                st_shared_v4(stage_addr + lane * 128 + ((e ^ (lane & 7)) << 4), v[4 * e], v[4 * e + 1], v[4 * e + 2],
                             v[4 * e + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (q0 + quarter * 32 < seg_end)   // skip a chunk of padding rows only
                    tma_reduce_add_3d(&a.tm_dqacc, stage, 0, q0 + quarter * 32, h * (D / 32) + chunk);
                bulk_commit_group();
            }
        };

        int4 cur;
        bool ok = warp_unit(0, cur);
        float nxt = (ok && loader && cur.x >= 0) ? col_term(cur, 0) : 0.f;
        int gi = 0;
        for (int it = 0; ok && cur.x >= 0; ++it) {
            const int nq = unit_nq(cur);
            const int nsteps = group * nq;
            const int kj = cur.y + unit_kv_tile(cur) * kTile + t;
            for (int i = 0; i < nsteps; ++i, ++gi) {
                const int h = cur.x * group + i / nq;
                const int q0 = cur.y + unit_q_tile(cur, i % nq) * kTile;
                const uint32_t ph = gi & 1;
                float *colbuf = is_p ? sm.lse2[gi & 1] : sm.delta[gi & 1];
                uint64_t *colbar = is_p ? &sm.cols_l[gi & 1] : &sm.cols_d[gi & 1];
                if (loader) {
                    colbuf[t] = nxt;
                    mbar_arrive(colbar);
                    if (i + 1 < nsteps) nxt = col_term(cur, i + 1);
                }
                if (!warp_wait(colbar, (gi >> 1) & 1, abort_flag, a.status)) { ok = false; break; }
                const float4 *CC = reinterpret_cast<const float4 *>(colbuf + col0);
                if constexpr (is_p) {
                    // P^T = exp(S^T * scale - LSE); column col0 + c (q row q0 + col0 + c)
                    // is live for kv row kj iff kj <= q row < seg_end. The P warps do
                    // nothing else, so P of the next step starts as soon as its S^T is in.
                    const int c_lo = kj - q0 - col0, c_hi = cur.z - q0 - col0;
                    const bool full = c_lo <= 0 && c_hi >= 64;
                    if (!warp_wait(&sm.s_full, ph, abort_flag, a.status)) { ok = false; break; }
                    tc_fence_after();
                    // Both S^T chunks are read before P^T is written: P^T columns col0 + 32c ..
                    // +31 (bf16 pairs) go to TMEM columns col0 + 16c .. +15.
                    uint32_t sv2[2][32];
                    tmem_ld64(tmem + lane_off + kA + col0, *reinterpret_cast<uint32_t(*)[64]>(&sv2[0][0]));
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const uint32_t (&sv)[32] = sv2[c];
                        uint32_t pk[16];
#pragma unroll
                        for (int e4 = 0; e4 < 8; ++e4) {
                            const float4 l4 = CC[c * 8 + e4];   // one broadcast load for four columns (-LSE log2 e)
                            const uint64_t lv2[2] = {f2_pack(l4.x, l4.y), f2_pack(l4.z, l4.w)};
#pragma unroll
                            for (int e2 = 0; e2 < 2; ++e2) {
                                const int e = e4 * 2 + e2, col = c * 32 + 2 * e;
                                // the scale and the LSE of a column pair in one packed instruction
                                float p0, p1;
                                f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])),
                                                 sl2_2, lv2[e2]),
                                          p0, p1);
                                p0 = ex2(p0);
                                p1 = ex2(p1);
                                if (!full) {
                                    if (col < c_lo || col >= c_hi) p0 = 0.f;
                                    if (col + 1 < c_lo || col + 1 >= c_hi) p1 = 0.f;
                                }
                                pk[e] = pack_bf16x2(p0, p1);
                            }
                        }
                        tmem_st16(tmem + lane_off + kA + col0 + c * 16, pk);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(&sm.p_full);
                } else {
                    // dS^T = P^T * (dP^T - D); P^T read back from TMEM (bf16), masked entries are 0
                    if (!warp_wait(&sm.dp_full, ph, abort_flag, a.status)) { ok = false; break; }
                    if (!warp_wait(&sm.p_full, ph, abort_flag, a.status)) { ok = false; break; }
                    tc_fence_after();
                    // This warp's staged chunks of the previous step (the dS buffer one and
                    // the Q stage one) must have been read by the TMA engine before dS is
                    // written over the former; the Q stage then goes back to the producer.
                    if (gi > 0) {
                        if (lane == 0) {
                            bulk_wait_group_read0();
                            mbar_arrive(&sm.q_empty[(gi - 1) % kQStages]);
                        }
                        __syncwarp();
                    }
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint32_t dp[32], pv[16];
                        tmem_ld32(tmem + lane_off + kB + col0 + c * 32, dp);
                        tmem_ld16(tmem + lane_off + kA + col0 + c * 16, pv);
                        tmem_wait_ld();
                        uint32_t pk[16];
#pragma unroll
                        for (int e4 = 0; e4 < 8; ++e4) {
                            const float4 d4 = CC[c * 8 + e4];
                            const uint64_t dv2[2] = {f2_pack(d4.x, d4.y), f2_pack(d4.z, d4.w)};
#pragma unroll
                            for (int e2 = 0; e2 < 2; ++e2) {
                                const int e = e4 * 2 + e2;
                                // dS = P (dP - D) for a column pair, two packed instructions
                                float d0, d1;
                                f2_unpack(f2_mul(f2_pack(bf16_lo(pv[e]), bf16_hi(pv[e])),
                                                 f2_sub(f2_pack(__uint_as_float(dp[2 * e]), __uint_as_float(dp[2 * e + 1])),
                                                        dv2[e2])),
                                          d0, d1);
                                pk[e] = pack_bf16x2(d0, d1);
                            }
                        }
                        // row t, q columns col0 + 32c .. +31: atom `half`, 16-byte chunks 4c .. 4c+3
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4) {
                            const int chunk = c * 4 + v4;
                            st_shared_v4(ds_addr + half * kAtom + t * 128 + ((chunk ^ (t & 7)) << 4), pk[4 * v4],
                                         pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
                        }
                    }
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(&sm.ds_full);
                    // dQ read-out: this warp's rows of d columns 32 half (and 32 (half + 2)
                    // for d = 128). Both TMEM loads land before B is released for the next
                    // dP^T; the chunks are then staged and added in the background.
                    if (!warp_wait(&sm.dq_full, ph, abort_flag, a.status)) { ok = false; break; }
                    tc_fence_after();
                    uint32_t va[32], vb[32];
                    tmem_ld32(tmem + lane_off + kB + half * 32, va);
                    if (D == 128) tmem_ld32(tmem + lane_off + kB + (half + 2) * 32, vb);
                    tmem_wait_ld();
                    tc_fence_before();
                    mbar_arrive(&sm.dq_free);
                    dq_stage(va, slot_a(gi), half, q0, cur.z, h);
                    if (D == 128) dq_stage(vb, slot_b, half + 2, q0, cur.z, h);
                }
            }
            if (!ok) break;
            // Take the next unit and start its first column load. The dS warps then
            // read out this unit's dV and dK once all its MMAs have completed
            // (acc_full) and release the accumulators (acc_free) before the next
            // unit's first dV MMA; the P warps go straight on.
            int4 nu;
            if (!warp_unit(it + 1, nu)) { ok = false; break; }
            if (loader && nu.x >= 0) nxt = col_term(nu, 0);
            if constexpr (!is_p) {
                if (!warp_wait(&sm.acc_full, it & 1, abort_flag, a.status)) { ok = false; break; }
                tc_fence_after();
                store_acc_rows<D, true>(a, tmem + lane_off + kC + half * (D / 2), cur, quarter, half, slot_a(gi - 1));
                store_acc_rows<D, false>(a, tmem + lane_off + kE + half * (D / 2), cur, quarter, half, slot_b);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.acc_free);
            }
            cur = nu;
        }
        if (lane == 0) bulk_wait_group0();     // every reduce / store of this warp has landed
        __syncwarp();
        };
        if (warp < kPWarps) {
            setmaxnreg_inc<kPRegs>();
            compute(std::true_type{});
        } else {
            setmaxnreg_inc<kDsRegs>();
            compute(std::false_type{});
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 17) tmem_dealloc(tmem, kTmemCols);
}

template <int D>
cudaError_t launch_bwd_d(const AttnBwdArgs &a, int64_t max_units, cudaStream_t stream)
{
    const int T = a.total_tokens;
    const long long rows = static_cast<long long>(T) * a.Hq;
    {
        long long blocks = (rows * 8 + 255) / 256;
        if (blocks > 152 * 16) blocks = 152 * 16;
        if (blocks < 1) blocks = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(blocks));
        cfg.blockDim = dim3(256);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&cfg, bwd_pre_kernel<D>, a.out, a.dout, a.delta, a.dq_acc, T, a.Hq);
        if (e != cudaSuccess) return e;
    }
    const size_t smem = sizeof(BwdSmem<D>);
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    // Persistent: one CTA per SM takes work units from the shared counter.
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    int64_t grid = max_units * a.Hkv;
    if (grid > sms) grid = sms;
    if (grid > 0) {
        prof_begin(kProfAttnBwd, stream);
        attn_bwd_kernel<D><<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(a);
        prof_end(kProfAttnBwd, stream);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    long long blocks = (rows * (D / 8) + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    bwd_dq_kernel<D><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a.dq_acc, a.dq, a.grad_fp32, a.scale, T, a.Hq);
    return cudaGetLastError();
}

}  // namespace

// max_units: upper bound of the number of kv tiles of one kv head.
cudaError_t launch_attn_bwd(const AttnBwdArgs &a, int head_dim, int64_t max_units, cudaStream_t stream)
{
    if (head_dim == 64) return launch_bwd_d<64>(a, max_units, stream);
    if (head_dim == 128) return launch_bwd_d<128>(a, max_units, stream);
    return cudaErrorInvalidValue;
}

}  // namespace spd
