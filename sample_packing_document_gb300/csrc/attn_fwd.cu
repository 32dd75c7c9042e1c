// Forward attention over packed rows with the per-document causal mask.
//
// One CTA computes two consecutive 128-row q tiles (X = A, B) of one segment
// and one q head: O_X = softmax(S_X) V with S_X = scale * Q_X K^T over the kv
// tiles of the same segment up to X's diagonal (page "Sample Packing: attention
// problems of long-sequence LLM training", section 5.1 "FlashAttention":
// tiles above a document's diagonal are never visited, the diagonal tile is
// the only one that needs the mask). Both tiles share every K / V tile the CTA
// loads. Online softmax in fp32 (running max m, running sum l; O is rescaled
// only when the max grows by more than 2^8, which keeps every partial value
// within fp32 / bf16 range and leaves the result exact up to rounding).
//
// Warp roles (320 threads):
//   warps 0-3 / 4-7  softmax of tile A / B: thread r owns q row r (TMEM lane
//                    r). Reads S_X from TMEM, writes P_X as bf16 back into the
//                    first 64 columns of S_X's TMEM region, rescales O_X in
//                    TMEM when needed, final normalisation and stores.
//   warp 8           TMA producer: Q_A, Q_B once, K / V tiles through a 2-stage ring.
//   warp 9           MMA issuer: S_X(j) = Q_X K_j^T (both operands in shared
//                    memory), O_X += P_X(j) V_j (P from TMEM, V from shared
//                    memory), interleaved A / B so one tile's softmax overlaps
//                    the other tile's MMAs.
// TMEM: S_A / P_A [0,128), S_B / P_B [128,256), O_A [256, 256+d), O_B [384, 384+d).
// Each tile's MMAs run in issue order on the tensor pipe, so S_X(j+1), issued
// after O_X += P_X(j) V_j, never overwrites P_X(j) before it has been read, and
// the commit after S_X(j+1) also covers that P V product (O_X is then stable
// for a rescale).
#include "internal.h"
#include "ptx.cuh"

namespace spd {
namespace {

constexpr int kStages = 2;
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAtom = 128 * 128;  // bytes of one [128 rows][64 bf16] swizzled atom

template <int D>
struct alignas(1024) FwdSmem {
    uint8_t q[2][D / 64][kAtom];
    uint8_t k[kStages][D / 64][kAtom];
    uint8_t v[kStages][D / 64][kAtom];
    uint64_t q_full;
    uint64_t k_full[kStages], v_full[kStages], kv_empty[kStages];
    uint64_t s_full[2], p_full[2], o_done[2];
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

// Bounded wait taken by a whole warp: either every lane goes on or none does,
// so the warp never splits before a .sync.aligned tcgen05 instruction.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          int *status)
{
    bool w = mbar_wait(bar, parity, abort_flag, status);
    return __all_sync(0xffffffffu, w);
}

// D[tmem] (+)= A[tmem] * B[smem]: A (M x K, bf16) sits in TMEM, one row per
// lane, two K elements per 32-bit column.
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ AttnFwdArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    FwdSmem<D> &sm = *reinterpret_cast<FwdSmem<D> *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (*reinterpret_cast<volatile int *>(a.status) != 0) return;
    // Head-major order: the CTAs of one head (and the heads of one kv group)
    // run together, so the K / V tiles they share stay in L2; inside a head the
    // work list is longest-first.
    const int h = blockIdx.x / a.grid_tiles;
    const int unit_idx = blockIdx.x % a.grid_tiles;
    if (unit_idx >= *a.tile_count) return;
    const Tile tl = a.tiles[unit_idx];
    const int n_seg_tiles = (tl.seg_end - tl.seg_start + kTile - 1) / kTile;
    const int tA = tl.t;                          // q tile of A; B is tA + 1 if the segment has it
    const bool has_b = tA + 1 < n_seg_tiles;
    const int n_kv = has_b ? tA + 2 : tA + 1;     // kv tiles the CTA loads
    const int g = h / (a.Hq / a.Hkv);

    if (threadIdx.x == 0) {
        mbar_init(&sm.q_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.k_full[s], 1);
            mbar_init(&sm.v_full[s], 1);
            mbar_init(&sm.kv_empty[s], 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&sm.s_full[x], 1);
            mbar_init(&sm.p_full[x], 128);
            mbar_init(&sm.o_done[x], 1);
        }
        mbar_init(&sm.drain, 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 8 && lane == 0) {
        tma_prefetch_desc(&a.tm_q);
        tma_prefetch_desc(&a.tm_k);
        tma_prefetch_desc(&a.tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    volatile int *abort_flag = &sm.abort_flag;
    constexpr uint32_t kTileBytes = 128 * D * 2;
    const int q0A = tl.seg_start + tA * kTile;

    if (warp == 8) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            mbar_arrive_expect_tx(&sm.q_full, (has_b ? 2 : 1) * kTileBytes);
            for (int x = 0; x < (has_b ? 2 : 1); ++x)
                for (int c = 0; c < D / 64; ++c)
                    tma_load_3d(sm.q[x][c], &a.tm_q, c * 64, h, q0A + x * kTile, &sm.q_full);
            int last_use[kStages];
            for (int s = 0; s < kStages; ++s) last_use[s] = -1;
            for (int j = 0; j < n_kv; ++j) {
                const int st = j % kStages, u = j / kStages;
                if (u > 0 && !mbar_wait(&sm.kv_empty[st], (u - 1) & 1, abort_flag, a.status)) break;
                const int kv0 = tl.seg_start + j * kTile;
                mbar_arrive_expect_tx(&sm.k_full[st], kTileBytes);
                for (int c = 0; c < D / 64; ++c)
                    tma_load_3d(sm.k[st][c], &a.tm_k, c * 64, g, kv0, &sm.k_full[st]);
                mbar_arrive_expect_tx(&sm.v_full[st], kTileBytes);
                for (int c = 0; c < D / 64; ++c)
                    tma_load_3d(sm.v[st][c], &a.tm_v, c * 64, g, kv0, &sm.v_full[st]);
                last_use[st] = u;
            }
            if (*abort_flag) {
                // Let the copies still in flight land before the CTA exits.
                wait_drain(&sm.q_full, 0);
                for (int s = 0; s < kStages; ++s)
                    if (last_use[s] >= 0) {
                        wait_drain(&sm.k_full[s], last_use[s] & 1);
                        wait_drain(&sm.v_full[s], last_use[s] & 1);
                    }
            }
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16(128, 128, 0, 0);
            constexpr uint32_t idesc_o = idesc_bf16(128, D, 0, 1);
            const int n_tile0 = tA + 1, n_tile1 = has_b ? tA + 2 : 0;  // kv tiles each q tile reads
            int empty_commits[kStages] = {};
            auto issue_s = [&](int x, int j) {
                const uint32_t q_addr = smem_u32(sm.q[x][0]);
                const uint32_t k_addr = smem_u32(sm.k[j % kStages][0]);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kAtom + (kk & 3) * 32;
                    umma_bf16(tmem + x * 128, sdesc_sw128(q_addr + off, 16, 1024), sdesc_sw128(k_addr + off, 16, 1024),
                              idesc_s, kk > 0 ? 1u : 0u);
                }
                umma_commit(&sm.s_full[x]);
            };
            auto issue_pv = [&](int x, int j) {
                const uint32_t v_addr = smem_u32(sm.v[j % kStages][0]);
#pragma unroll
                for (int kk = 0; kk < 128 / 16; ++kk)
                    umma_bf16_ts(tmem + 256 + x * 128, tmem + x * 128 + kk * 8, sdesc_sw128(v_addr + kk * 2048, kAtom, 1024),
                                 idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
            };
            bool ok = mbar_wait(&sm.q_full, 0, abort_flag, a.status) &&
                      mbar_wait(&sm.k_full[0], 0, abort_flag, a.status);
            if (ok) {
                tc_fence_after();
                issue_s(0, 0);
                if (n_tile1 > 0) issue_s(1, 0);
            }
            for (int j = 0; ok && j < n_kv; ++j) {
                const int st = j % kStages;
                const bool next_k = j + 1 < n_kv;
                if (!mbar_wait(&sm.v_full[st], (j / kStages) & 1, abort_flag, a.status)) { ok = false; break; }
                if (next_k && !mbar_wait(&sm.k_full[(j + 1) % kStages], ((j + 1) / kStages) & 1, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    const int nt = x ? n_tile1 : n_tile0;
                    if (!ok || j >= nt) continue;
                    if (!mbar_wait(&sm.p_full[x], j & 1, abort_flag, a.status)) { ok = false; continue; }
                    tc_fence_after();
                    issue_pv(x, j);
                    if (j + 1 < nt) issue_s(x, j + 1);   // its commit also covers this P V
                    else umma_commit(&sm.o_done[x]);
                }
                if (!ok) break;
                umma_commit(&sm.kv_empty[st]);
                ++empty_commits[st];
            }
            // Every arrive the tensor core owes this CTA's barriers must land
            // before the CTA exits.
            umma_commit(&sm.drain);
            wait_drain(&sm.drain, 0);
            for (int s = 0; s < kStages; ++s)
                if (empty_commits[s] > 0) wait_drain(&sm.kv_empty[s], (empty_commits[s] - 1) & 1);
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int x = warp >> 2;                      // 0: tile A, 1: tile B
        const int r = threadIdx.x & 127;              // q row within the tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t s_col = x * 128, o_col = 256 + x * 128;
        const int tX = tA + x;
        const int nX = (x == 0) ? tA + 1 : (has_b ? tA + 2 : 0);
        const float sl2 = a.scale_log2;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nX; ++j) {
            if (!warp_wait(&sm.s_full[x], j & 1, abort_flag, a.status)) { ok = false; break; }
            tc_fence_after();
            const bool diag = (j == tX);
            // pass 1: row max, 64 columns per TMEM round trip, 8 independent chains
            float mxs[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) mxs[e] = -INFINITY;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t sv[64];
                tmem_ld32(tmem + lane_off + s_col + c * 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
                tmem_ld32(tmem + lane_off + s_col + c * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
                tmem_wait_ld();
                if (diag) {
#pragma unroll
                    for (int e = 0; e < 64; ++e)
                        if (c * 64 + e <= r) mxs[e & 7] = fmaxf(mxs[e & 7], __uint_as_float(sv[e]));
                } else {
#pragma unroll
                    for (int e = 0; e < 64; ++e) mxs[e & 7] = fmaxf(mxs[e & 7], __uint_as_float(sv[e]));
                }
            }
            const float mx = fmaxf(fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3])),
                                   fmaxf(fmaxf(mxs[4], mxs[5]), fmaxf(mxs[6], mxs[7])));
            const float m_new = fmaxf(m, mx * sl2);
            const bool need = m_new > m + 8.0f;
            if (__any_sync(0xffffffffu, need)) {
                const float m_use = need ? m_new : m;
                const float alpha = ex2(m - m_use);  // 0 when m = -inf
                if (j > 0) {
                    // O_X is stable: the commit that raised s_full covers the last P V.
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tmem + lane_off + o_col + c * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(tmem + lane_off + o_col + c * 32, o);
                    }
                }
                l *= alpha;
                m = m_use;
            }
            // pass 2: P = 2^(S * scale * log2 e - m), written as bf16 over the
            // first 64 columns of S_X's region; P columns 32c..32c+31 only cover
            // S columns already read.
            float sums[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t sv[64];
                tmem_ld32(tmem + lane_off + s_col + c * 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
                tmem_ld32(tmem + lane_off + s_col + c * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
                tmem_wait_ld();
                uint32_t pk[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    float p0 = ex2(__uint_as_float(sv[2 * e]) * sl2 - m);
                    float p1 = ex2(__uint_as_float(sv[2 * e + 1]) * sl2 - m);
                    if (diag) {
                        if (c * 64 + 2 * e > r) p0 = 0.f;
                        if (c * 64 + 2 * e + 1 > r) p1 = 0.f;
                    }
                    sums[e & 3] += p0 + p1;
                    pk[e] = pack_bf16x2(p0, p1);
                }
                tmem_st32(tmem + lane_off + s_col + c * 32, pk);
            }
            const float sum = (sums[0] + sums[1]) + (sums[2] + sums[3]);
            l += sum;
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&sm.p_full[x]);
        }
        if (ok && nX > 0 && warp_wait(&sm.o_done[x], 0, abort_flag, a.status)) {
            tc_fence_after();
            const int qi = q0A + x * kTile + r;
            const bool valid = qi < tl.seg_end;
            const float inv_l = 1.f / l;
            uint16_t *orow = a.out + (static_cast<size_t>(qi) * a.Hq + h) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_off + o_col + c * 32, o);
                tmem_wait_ld();
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    w[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
                if (valid) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
                    for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
                }
            }
            if (valid) a.lse[static_cast<size_t>(h) * a.total_tokens + qi] = (m + log2f(l)) * 0.69314718055994531f;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tmem, kTmemCols);
}

template <int D>
cudaError_t launch_fwd_d(const AttnFwdArgs &a, int64_t grid_units, cudaStream_t stream)
{
    // One CTA per SM: every CTA allocates 512 TMEM columns, so a second
    // resident CTA would only block in tcgen05.alloc.
    size_t smem = sizeof(FwdSmem<D>) + 1024;
    if (smem < 120 * 1024) smem = 120 * 1024;
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    AttnFwdArgs a2 = a;
    a2.grid_tiles = static_cast<int32_t>(grid_units);
    const int64_t grid = grid_units * a.Hq;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
    prof_begin(kProfAttnFwd, stream);
    attn_fwd_kernel<D><<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(a2);
    prof_end(kProfAttnFwd, stream);
    return cudaGetLastError();
}

}  // namespace

// grid_units: upper bound of the number of work units (pairs of q tiles).
cudaError_t launch_attn_fwd(const AttnFwdArgs &a, int head_dim, int64_t grid_units, cudaStream_t stream)
{
    if (head_dim == 64) return launch_fwd_d<64>(a, grid_units, stream);
    if (head_dim == 128) return launch_fwd_d<128>(a, grid_units, stream);
    return cudaErrorInvalidValue;
}

}  // namespace spd
