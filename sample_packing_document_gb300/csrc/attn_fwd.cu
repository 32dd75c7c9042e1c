// Forward attention over packed rows with the per-document causal mask.
//
// One CTA computes one 128-row q tile of one q head: O = softmax(S) V with
// S = scale * Q K^T over the kv tiles 0..t of the same segment (page "Sample
// Packing: attention problems of long-sequence LLM training", section 5.1
// "FlashAttention": tiles above a document's diagonal are never visited, the
// diagonal tile is the only one that needs the mask, tiles below it need
// none). Online softmax in fp32 (running max m, running sum l; O rescaled only
// when the max grows by more than 2^8, which keeps every partial value within
// fp32 / bf16 range and leaves the result exact up to rounding).
//
// Warp roles (192 threads):
//   warps 0-3  softmax: thread r owns q row r = TMEM lane r. Reads S from
//              TMEM, writes P (bf16) to shared memory, rescales O in TMEM,
//              final normalisation and stores.
//   warp 4     TMA producer: Q once, K / V tiles through a 2-stage ring.
//   warp 5     MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM
//              S buffers, O += P_j V_j into the TMEM O accumulator.
// TMEM: S0 columns [0,128), S1 [128,256), O [256, 256 + head_dim).
#include "internal.h"
#include "ptx.cuh"

namespace spd {
namespace {

constexpr int kStages = 2;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAtom = 128 * 128;  // bytes of one [128 rows][64 bf16] swizzled atom

template <int D>
struct alignas(1024) FwdSmem {
    uint8_t q[D / 64][kAtom];
    uint8_t k[kStages][D / 64][kAtom];
    uint8_t v[kStages][D / 64][kAtom];
    uint8_t p[2][kAtom];
    uint64_t q_full;
    uint64_t k_full[kStages], v_full[kStages], kv_empty[kStages];
    uint64_t s_full[2], s_empty[2];
    uint64_t p_full, o_done, drain;
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
    const int tile_idx = blockIdx.x % a.grid_tiles;
    if (tile_idx >= *a.tile_count) return;
    const Tile tl = a.tiles[tile_idx];
    const int q0 = tl.seg_start + tl.t * kTile;
    const int n_kv = tl.t + 1;
    const int g = h / (a.Hq / a.Hkv);

    if (threadIdx.x == 0) {
        mbar_init(&sm.q_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.k_full[s], 1);
            mbar_init(&sm.v_full[s], 1);
            mbar_init(&sm.kv_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.s_full[b], 1);
            mbar_init(&sm.s_empty[b], 128);
        }
        mbar_init(&sm.p_full, 128);
        mbar_init(&sm.o_done, 1);
        mbar_init(&sm.drain, 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
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

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            mbar_arrive_expect_tx(&sm.q_full, kTileBytes);
            for (int c = 0; c < D / 64; ++c) tma_load_3d(sm.q[c], &a.tm_q, c * 64, h, q0, &sm.q_full);
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
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16(128, 128, 0, 0);
            constexpr uint32_t idesc_o = idesc_bf16(128, D, 0, 1);
            const uint32_t q_addr = smem_u32(sm.q[0]);
            const uint32_t p_addr = smem_u32(sm.p[0]);
            int empty_commits[kStages] = {};
            bool ok = mbar_wait(&sm.q_full, 0, abort_flag, a.status);
            auto issue_pv = [&](int jj) -> bool {
                const int st = jj % kStages;
                if (!mbar_wait(&sm.p_full, jj & 1, abort_flag, a.status)) return false;
                if (!mbar_wait(&sm.v_full[st], (jj / kStages) & 1, abort_flag, a.status)) return false;
                tc_fence_after();
                const uint32_t v_addr = smem_u32(sm.v[st][0]);
#pragma unroll
                for (int kk = 0; kk < 128 / 16; ++kk) {
                    uint64_t ad = sdesc_sw128(p_addr + (kk >> 2) * kAtom + (kk & 3) * 32, 16, 1024);
                    uint64_t bd = sdesc_sw128(v_addr + kk * 2048, kAtom, 1024);
                    umma_bf16(tmem + 256, ad, bd, idesc_o, (jj > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(&sm.o_done);
                umma_commit(&sm.kv_empty[st]);
                ++empty_commits[st];
                return true;
            };
            for (int j = 0; ok && j < n_kv; ++j) {
                const int st = j % kStages, sb = j & 1;
                if (!mbar_wait(&sm.k_full[st], (j / kStages) & 1, abort_flag, a.status)) { ok = false; break; }
                if (j >= 2 && !mbar_wait(&sm.s_empty[sb], ((j >> 1) - 1) & 1, abort_flag, a.status)) { ok = false; break; }
                tc_fence_after();
                const uint32_t k_addr = smem_u32(sm.k[st][0]);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    uint64_t ad = sdesc_sw128(q_addr + (kk >> 2) * kAtom + (kk & 3) * 32, 16, 1024);
                    uint64_t bd = sdesc_sw128(k_addr + (kk >> 2) * kAtom + (kk & 3) * 32, 16, 1024);
                    umma_bf16(tmem + sb * 128, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
                }
                umma_commit(&sm.s_full[sb]);
                if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
            }
            if (ok) ok = issue_pv(n_kv - 1);
            // Every arrive the tensor core owes this CTA's barriers must land
            // before the CTA exits.
            umma_commit(&sm.drain);
            wait_drain(&sm.drain, 0);
            for (int s = 0; s < kStages; ++s)
                if (empty_commits[s] > 0) wait_drain(&sm.kv_empty[s], (empty_commits[s] - 1) & 1);
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int r = threadIdx.x;  // q row within the tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const float sl2 = a.scale_log2;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        const uint32_t p_row = smem_u32(sm.p[0]) + r * 128;
        for (int j = 0; j < n_kv; ++j) {
            const int sb = j & 1;
            if (!warp_wait(&sm.s_full[sb], (j >> 1) & 1, abort_flag, a.status)) { ok = false; break; }
            tc_fence_after();
            uint32_t s[128];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                tmem_ld32(tmem + lane_off + sb * 128 + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[c * 32]));
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(&sm.s_empty[sb]);

            float mx = -INFINITY;
            const bool diag = (j == n_kv - 1);
#pragma unroll
            for (int c = 0; c < 128; ++c) {
                float x = __uint_as_float(s[c]) * sl2;
                if (diag && c > r) x = -INFINITY;
                s[c] = __float_as_uint(x);
                mx = fmaxf(mx, x);
            }
            const float m_new = fmaxf(m, mx);
            const bool need = m_new > m + 8.0f;
            const bool warp_need = __any_sync(0xffffffffu, need);
            if (warp_need) {
                const float m_use = need ? m_new : m;
                const float alpha = ex2(m - m_use);  // 0 when m = -inf
                if (j > 0) {
                    if (!warp_wait(&sm.o_done, (j - 1) & 1, abort_flag, a.status)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tmem + lane_off + 256 + c * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(tmem + lane_off + 256 + c * 32, o);
                    }
                    tmem_wait_st();
                }
                l *= alpha;
                m = m_use;
            }
            float sum = 0.f;
            uint32_t pk[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                float p0 = ex2(__uint_as_float(s[2 * c]) - m);
                float p1 = ex2(__uint_as_float(s[2 * c + 1]) - m);
                sum += p0 + p1;
                pk[c] = pack_bf16x2(p0, p1);
            }
            l += sum;
            if (j > 0 && !warp_need) {
                if (!warp_wait(&sm.o_done, (j - 1) & 1, abort_flag, a.status)) { ok = false; break; }
            }
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const uint32_t addr = p_row + (c >> 3) * kAtom + (((c & 7) ^ (r & 7)) << 4);
                st_shared_v4(addr, pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&sm.p_full);
        }
        if (ok && warp_wait(&sm.o_done, (n_kv - 1) & 1, abort_flag, a.status)) {
            tc_fence_after();
            const int qi = q0 + r;
            const bool valid = qi < tl.seg_end;
            const float inv_l = 1.f / l;
            uint16_t *orow = a.out + (static_cast<size_t>(qi) * a.Hq + h) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_off + 256 + c * 32, o);
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
    if (warp == 5) tmem_dealloc(tmem, kTmemCols);
}

template <int D>
cudaError_t launch_fwd_d(const AttnFwdArgs &a, int64_t grid_tiles, cudaStream_t stream)
{
    // One CTA per SM: every CTA allocates 512 TMEM columns, so a second
    // resident CTA would only block in tcgen05.alloc.
    size_t smem = sizeof(FwdSmem<D>) + 1024;
    if (smem < 120 * 1024) smem = 120 * 1024;
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    AttnFwdArgs a2 = a;
    a2.grid_tiles = static_cast<int32_t>(grid_tiles);
    const int64_t grid = grid_tiles * a.Hq;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
    prof_begin(kProfAttnFwd, stream);
    attn_fwd_kernel<D><<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(a2);
    prof_end(kProfAttnFwd, stream);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd(const AttnFwdArgs &a, int head_dim, int64_t grid_tiles, cudaStream_t stream)
{
    if (head_dim == 64) return launch_fwd_d<64>(a, grid_tiles, stream);
    if (head_dim == 128) return launch_fwd_d<128>(a, grid_tiles, stream);
    return cudaErrorInvalidValue;
}

}  // namespace spd
