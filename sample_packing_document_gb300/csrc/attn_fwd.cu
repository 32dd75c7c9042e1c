// Forward attention over packed rows with the per-document causal mask.
//
// A persistent CTA (one per SM) takes work units from a shared counter; a unit
// is two consecutive 128-row q tiles (X = A, B) of one segment and one q head: O_X = softmax(S_X) V with S_X = scale * Q_X K^T over the kv
// tiles of the same segment up to X's diagonal (page "Sample Packing: attention
// problems of long-sequence LLM training", section 5.1 "FlashAttention":
// tiles above a document's diagonal are never visited, the diagonal tile is
// the only one that needs the mask). Both tiles share every K / V tile the CTA
// loads. Online softmax in fp32 (running max m, running sum l; O is rescaled
// only when the max grows by more than 2^8, which keeps every partial value
// within fp32 / bf16 range and leaves the result exact up to rounding).
//
// Warp roles (384 threads; warps 10-11 only complete the third warpgroup):
//   warps 0-3 / 4-7  softmax of tile A / B: thread r owns q row r (TMEM lane
//                    r). Reads the whole S_X row from TMEM into registers once,
//                    writes P_X as bf16 back into the first 64 columns of S_X's
//                    TMEM region, rescales O_X in TMEM when needed, final
//                    normalisation and stores.
//   warp 8           TMA producer: takes the next work unit, loads Q_A, Q_B and
//                    streams the K / V tiles through 2-stage rings that run on
//                    across units, K one tile ahead of V (a K stage frees after
//                    the last S MMA reading it, a step before its V stage).
//   warp 9           MMA issuer: S_X(j) = Q_X K_j^T (both operands in shared
//                    memory), O_X += P_X(j) V_j (P from TMEM, V from shared
//                    memory), interleaved A / B so one tile's softmax overlaps
//                    the other tile's MMAs.
//   warps 10-11      with RoPE only: rotate Q_A, Q_B and every K tile in shared
//                    memory once its copy has landed and before any MMA reads
//                    it (rotate-half form, channel j with j + d/2, angle p *
//                    theta_j, p = the row's position inside its segment), so the
//                    rotated q and k never go through HBM. Without RoPE they idle.
// TMEM: S_A / P_A [0,128), S_B / P_B [128,256), O_A [256, 256+d), O_B [384, 384+d).
// Each tile's MMAs run in issue order on the tensor pipe, so S_X(j+1), issued
// after O_X += P_X(j) V_j, never overwrites P_X(j) before it has been read, and
// the commit after S_X(j+1) also covers that P V product (O_X is then stable
// for a rescale).
#include "internal.h"
#include "ptx.cuh"

namespace spd {
namespace {

constexpr int kStages = 2;   // the per-stage counters below are selected with (index & 1)
constexpr int kThreads = 384;
// Register split (setmaxnreg): the launch gives 168 per thread (384 x 168 = 64512);
// the warpgroup of the producer / MMA issuer drops to 72 and the two softmax
// warpgroups rise to 216 (2 x 128 x 216 + 128 x 72 = 64512), enough to keep a
// whole 128-column S row in registers.
constexpr uint32_t kSoftmaxRegs = 216, kControlRegs = 72;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAtom = 128 * 128;  // bytes of one [128 rows][64 bf16] swizzled atom
constexpr int kRotWarps = 2;           // warps 10-11: RoPE rotation of the Q / K tiles in shared memory

template <int D>
struct alignas(1024) FwdSmem {
    uint8_t q[2][D / 64][kAtom];
    uint8_t k[kStages][D / 64][kAtom];
    uint8_t v[kStages][D / 64][kAtom];
    uint8_t ostage[8][32 * 128];   // per softmax warp: 32 rows x 64 d of O (bf16, 128-byte swizzle)
    uint64_t q_full, q_empty, q_rot;
    uint64_t k_full[kStages], v_full[kStages], k_empty[kStages], v_empty[kStages], k_rot[kStages];
    uint64_t s_full[2], p_full[2], o_done[2], o_free[2];
    uint64_t unit_full[2], unit_empty[2];
    int4 unit[2];               // work unit in flight: {head (-1: no more work), seg_start, seg_end, first tile}
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

struct UnitShape {
    int tA, n_kv;
    bool has_b;
};

__device__ __forceinline__ UnitShape unit_shape(const int4 &u)
{
    UnitShape r;
    const int n_seg_tiles = (u.z - u.y + kTile - 1) / kTile;
    r.tA = u.w;
    r.has_b = r.tA + 1 < n_seg_tiles;
    r.n_kv = r.has_b ? r.tA + 2 : r.tA + 1;
    return r;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ AttnFwdArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    FwdSmem<D> &sm = *reinterpret_cast<FwdSmem<D> *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (*reinterpret_cast<volatile int *>(a.status) != 0) return;

    if (threadIdx.x == 0) {
        mbar_init(&sm.q_full, 1);
        mbar_init(&sm.q_empty, 1);
        mbar_init(&sm.q_rot, kRotWarps);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.k_full[s], 1);
            mbar_init(&sm.v_full[s], 1);
            mbar_init(&sm.k_empty[s], 1);
            mbar_init(&sm.v_empty[s], 1);
            mbar_init(&sm.k_rot[s], kRotWarps);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&sm.s_full[x], 1);
            mbar_init(&sm.p_full[x], 4);      // one arrive per softmax warp
            mbar_init(&sm.o_done[x], 1);
            mbar_init(&sm.o_free[x], 4);
            mbar_init(&sm.unit_full[x], 1);
            // MMA thread + one lane of each softmax warp (+ each rotator warp with RoPE)
            mbar_init(&sm.unit_empty[x], a.rope ? 9 + kRotWarps : 9);
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
        tma_prefetch_desc(&a.tm_o);
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
    const int units_per_head = *a.tile_count;
    const int total_units = units_per_head * a.Hq;
    const int n_long = *a.long_count;

    if (warp >= 8) {
    setmaxnreg_dec<kControlRegs>();
    if (warp == 8) {
        // ------------------------------------------------------------ producer
        // Takes work units from the shared counter in list order (unit_of): the
        // few units much longer than a head's share of an SM first, across heads;
        // then head-major (the CTAs on one head run together, so the K / V tiles
        // they share stay in L2), longest first inside a head.
        if (lane == 0) {
            // K runs one kv tile ahead of V: a K stage frees as soon as the last S
            // MMA reading it has completed (one kv step before its V stage), so the
            // copy of K(n + 2) starts a step earlier than a shared K / V stage would
            // allow. V(n) is issued right after K(n + 1).
            uint32_t kv_iter = 0;              // global index of the next K tile
            int last_k_use[kStages] = {-1, -1}, last_v_use[kStages] = {-1, -1};
            int pend_v = -1, pend_row = 0, pend_g = 0;   // a V tile not yet issued
            int q_loads = 0;
            auto load_v = [&](int n, int row, int g) -> bool {
                const int st = n % kStages, use = n / kStages;
                if (use > 0 && !mbar_wait(&sm.v_empty[st], (use - 1) & 1, abort_flag, a.status)) return false;
                mbar_arrive_expect_tx(&sm.v_full[st], kTileBytes);
                for (int c = 0; c < D / 64; ++c) tma_load_3d(sm.v[st][c], &a.tm_v, c * 64, g, row, &sm.v_full[st]);
                if (st) last_v_use[1] = use;   // constant indices keep the array in registers
                else last_v_use[0] = use;
                return true;
            };
            for (int it = 0;; ++it) {
                const int slot = it & 1;
                if (it >= 2 && !mbar_wait(&sm.unit_empty[slot], ((it >> 1) - 1) & 1, abort_flag, a.status)) break;
                const int u = *abort_flag ? total_units : atomicAdd(a.work_counter, 1);
                int4 d = make_int4(-1, 0, 0, 0);
                if (u < total_units) {
                    int head, idx;
                    unit_of(u, units_per_head, n_long, a.Hq, head, idx);
                    const Tile tl = a.tiles[idx];
                    d = make_int4(head, tl.seg_start, tl.seg_end, tl.t);
                }
                sm.unit[slot] = d;
                mbar_arrive(&sm.unit_full[slot]);
                if (d.x < 0) {
                    if (pend_v >= 0 && !*abort_flag) load_v(pend_v, pend_row, pend_g);   // the last V tile
                    break;
                }
                const UnitShape us = unit_shape(d);
                const int h = d.x, g = h / (a.Hq / a.Hkv);
                const int q0A = d.y + us.tA * kTile;
                // Q_A, Q_B once the previous unit's last S MMA has read them
                if (it > 0 && !mbar_wait(&sm.q_empty, (it - 1) & 1, abort_flag, a.status)) break;
                if (!(a.debug_skip && it == 0)) {   // test hook: q_full of the first unit never completes
                    mbar_arrive_expect_tx(&sm.q_full, (us.has_b ? 2 : 1) * kTileBytes);
                    for (int x = 0; x < (us.has_b ? 2 : 1); ++x)
                        for (int c = 0; c < D / 64; ++c)
                            tma_load_3d(sm.q[x][c], &a.tm_q, c * 64, h, q0A + x * kTile, &sm.q_full);
                    ++q_loads;
                }
                bool ok = true;
                for (int j = 0; j < us.n_kv; ++j, ++kv_iter) {
                    const int st = kv_iter % kStages, use = kv_iter / kStages;
                    if (use > 0 && !mbar_wait(&sm.k_empty[st], (use - 1) & 1, abort_flag, a.status)) { ok = false; break; }
                    const int kv0 = d.y + j * kTile;
                    mbar_arrive_expect_tx(&sm.k_full[st], kTileBytes);
                    for (int c = 0; c < D / 64; ++c)
                        tma_load_3d(sm.k[st][c], &a.tm_k, c * 64, g, kv0, &sm.k_full[st]);
                    if (st) last_k_use[1] = use;
                    else last_k_use[0] = use;
                    if (pend_v >= 0 && !load_v(pend_v, pend_row, pend_g)) { ok = false; break; }
                    pend_v = static_cast<int>(kv_iter);
                    pend_row = kv0;
                    pend_g = g;
                }
                if (!ok) break;
            }
            if (*abort_flag) {
                // Let the copies still in flight land before the CTA exits.
                if (q_loads > 0) wait_drain(&sm.q_full, (q_loads - 1) & 1);
                for (int s = 0; s < kStages; ++s) {
                    if (last_k_use[s] >= 0) wait_drain(&sm.k_full[s], last_k_use[s] & 1);
                    if (last_v_use[s] >= 0) wait_drain(&sm.v_full[s], last_v_use[s] & 1);
                }
            }
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16(128, 128, 0, 0);
            constexpr uint32_t idesc_o = idesc_bf16(128, D, 0, 1);
            uint32_t kv_iter = 0;
            int k_commits[kStages] = {0, 0}, v_commits[kStages] = {0, 0};
            int q_commits = 0;
            uint32_t p_cnt0 = 0, p_cnt1 = 0;      // P tiles consumed, per q tile slot
            uint32_t o_cnt0 = 0, o_cnt1 = 0;      // units that used O_A / O_B
            bool ok = true;
            for (int it = 0; ok; ++it) {
                const int slot = it & 1;
                if (!mbar_wait(&sm.unit_full[slot], (it >> 1) & 1, abort_flag, a.status)) break;
                const int4 d = sm.unit[slot];
                mbar_arrive(&sm.unit_empty[slot]);
                if (d.x < 0) break;
                const UnitShape us = unit_shape(d);
                const int n_tile0 = us.tA + 1, n_tile1 = us.has_b ? us.tA + 2 : 0;  // kv tiles each q tile reads
                int s_left = n_tile0 + n_tile1;   // S MMAs of this unit still to issue
                auto issue_s = [&](int x, int j) {
                    // descriptors of the k-steps differ only in the start address (low field)
                    const uint64_t qd = sdesc_sw128(smem_u32(sm.q[x][0]), 16, 1024);
                    const uint64_t kd = sdesc_sw128(smem_u32(sm.k[(kv_iter + j) % kStages][0]), 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off16 = ((kk >> 2) * kAtom + (kk & 3) * 32) >> 4;
                        umma_bf16_step(tmem + x * 128, qd, kd, off16, off16, idesc_s, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(&sm.s_full[x]);
                    if (--s_left == 0) {             // Q_A / Q_B fully read: next unit may load
                        umma_commit(&sm.q_empty);
                        ++q_commits;
                    }
                };
                auto issue_pv = [&](int x, int j) {
                    const uint64_t vd = sdesc_sw128(smem_u32(sm.v[(kv_iter + j) % kStages][0]), kAtom, 1024);
#pragma unroll
                    for (int kk = 0; kk < 128 / 16; ++kk)
                        umma_bf16_ts_step(tmem + 256 + x * 128, tmem + x * 128 + kk * 8, vd, kk * (2048 >> 4), idesc_o,
                                          (j > 0 || kk > 0) ? 1u : 0u);
                };
                // with RoPE, the operands are ready once rotated in place
                uint64_t *const q_ready = a.rope ? &sm.q_rot : &sm.q_full;
                uint64_t *const k_ready = a.rope ? sm.k_rot : sm.k_full;
                ok = mbar_wait(q_ready, it & 1, abort_flag, a.status) &&
                     mbar_wait(&k_ready[kv_iter % kStages], (kv_iter / kStages) & 1, abort_flag, a.status);
                if (!ok) break;
                tc_fence_after();
                issue_s(0, 0);                        // S regions: the last P V of each tile ran before
                if (n_tile1 > 0) issue_s(1, 0);
                umma_commit(&sm.k_empty[kv_iter % kStages]);   // K(0) read by both tiles' first S
                if (kv_iter % kStages) ++k_commits[1];   // constant indices keep the counts in registers
                else ++k_commits[0];
                for (int j = 0; ok && j < us.n_kv; ++j) {
                    const uint32_t kvj = kv_iter + j;
                    const int st = kvj % kStages;
                    const bool next_k = j + 1 < us.n_kv;
                    if (!mbar_wait(&sm.v_full[st], (kvj / kStages) & 1, abort_flag, a.status)) { ok = false; break; }
                    if (next_k && !mbar_wait(&k_ready[(kvj + 1) % kStages], ((kvj + 1) / kStages) & 1, abort_flag,
                                             a.status)) {
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        const int nt = x ? n_tile1 : n_tile0;
                        if (!ok || j >= nt) continue;
                        uint32_t &pc = x ? p_cnt1 : p_cnt0;
                        if (!mbar_wait(&sm.p_full[x], pc & 1, abort_flag, a.status)) { ok = false; continue; }
                        ++pc;
                        if (j == 0) {                 // O_X must have been read out by the last unit's epilogue
                            const uint32_t oc = x ? o_cnt1 : o_cnt0;
                            if (oc > 0 && !mbar_wait(&sm.o_free[x], (oc - 1) & 1, abort_flag, a.status)) {
                                ok = false;
                                continue;
                            }
                        }
                        tc_fence_after();
                        issue_pv(x, j);
                        if (j + 1 < nt) issue_s(x, j + 1);   // its commit also covers this P V
                        else {
                            umma_commit(&sm.o_done[x]);
                            if (x) ++o_cnt1;
                            else ++o_cnt0;
                        }
                    }
                    if (!ok) break;
                    if (next_k) {                     // K(j + 1) read by every S of this step
                        umma_commit(&sm.k_empty[(kvj + 1) % kStages]);
                        if ((kvj + 1) % kStages) ++k_commits[1];
                        else ++k_commits[0];
                    }
                    umma_commit(&sm.v_empty[st]);     // V(j) read by every P V of this step
                    if (st) ++v_commits[1];
                    else ++v_commits[0];
                }
                kv_iter += us.n_kv;
            }
            // Every arrive the tensor core owes this CTA's barriers must land
            // before the CTA exits.
            umma_commit(&sm.drain);
            wait_drain(&sm.drain, 0);
            for (int s = 0; s < kStages; ++s) {
                if (k_commits[s] > 0) wait_drain(&sm.k_empty[s], (k_commits[s] - 1) & 1);
                if (v_commits[s] > 0) wait_drain(&sm.v_empty[s], (v_commits[s] - 1) & 1);
            }
            if (q_commits > 0) wait_drain(&sm.q_empty, (q_commits - 1) & 1);
        }
    } else if (a.rope) {
        // ------------------------------------------------------------ RoPE rotators
        // 64 threads rotate a [128 rows][D] tile in place: thread tau takes the
        // 16-byte chunk c of the first half of every row r0 + kStride * k (8
        // channel pairs j = 8c .. 8c + 7, each with its partner j + D/2 at the same
        // swizzled offset of the second 64-column atom for D = 128, or chunk c + 4
        // of the same atom for D = 64). The angle of row r is (p0 + r) theta_j for
        // a tile starting p0 tokens into its segment: exact for the thread's first
        // row (64-bit fixed-point phase, as spd_rope computes it), then stepped
        // from row to row by the fixed rotation kStride theta_j.
        constexpr int kCh = D / 16, kStride = 64 / kCh, kRows = 128 / kStride;
        const int tau = threadIdx.x - 320;
        const int c = tau % kCh, r0 = tau / kCh;
        auto exact_cs = [&](uint32_t p, int e, float &cs, float &sn) {
            const uint64_t ph = static_cast<uint64_t>(p) * a.freq[c * 8 + e];   // turns * 2^64, mod 2^64
            const int32_t half_turns = static_cast<int32_t>(static_cast<uint32_t>(ph >> 32));
            sincospif(static_cast<float>(half_turns) * 4.656612873077393e-10f, &sn, &cs);
        };
        float stc[8], sts[8];   // rotation by kStride positions
#pragma unroll
        for (int e = 0; e < 8; ++e) exact_cs(kStride, e, stc[e], sts[e]);
        auto rotate_tile = [&](uint8_t (*tile)[kAtom], int p0) {
            float zc[8], zs[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) exact_cs(static_cast<uint32_t>(p0 + r0), e, zc[e], zs[e]);
            const uint32_t lo_base = smem_u32(tile[0]);
            const uint32_t hi_base = D == 128 ? smem_u32(tile[D / 128]) : lo_base;
#pragma unroll 2
            for (int k = 0; k < kRows; ++k) {
                const int row = r0 + kStride * k;
                const uint32_t lo_addr = lo_base + row * 128 + ((c ^ (row & 7)) << 4);
                const uint32_t hi_addr = hi_base + row * 128 + (((D == 128 ? c : c + 4) ^ (row & 7)) << 4);
                uint32_t lo[4], hi[4], olo[4], ohi[4];
                ld_shared_v4(lo_addr, lo[0], lo[1], lo[2], lo[3]);
                ld_shared_v4(hi_addr, hi[0], hi[1], hi[2], hi[3]);
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const int e0 = 2 * w, e1 = 2 * w + 1;
                    const float x0 = __uint_as_float(lo[w] << 16), x1 = __uint_as_float(lo[w] & 0xffff0000u);
                    const float y0 = __uint_as_float(hi[w] << 16), y1 = __uint_as_float(hi[w] & 0xffff0000u);
                    olo[w] = pack_bf16x2(x0 * zc[e0] - y0 * zs[e0], x1 * zc[e1] - y1 * zs[e1]);
                    ohi[w] = pack_bf16x2(y0 * zc[e0] + x0 * zs[e0], y1 * zc[e1] + x1 * zs[e1]);
                }
                st_shared_v4(lo_addr, olo[0], olo[1], olo[2], olo[3]);
                st_shared_v4(hi_addr, ohi[0], ohi[1], ohi[2], ohi[3]);
#pragma unroll
                for (int e = 0; e < 8; ++e) {   // advance every angle by kStride positions
                    const float nc = zc[e] * stc[e] - zs[e] * sts[e];
                    zs[e] = zs[e] * stc[e] + zc[e] * sts[e];
                    zc[e] = nc;
                }
            }
            fence_proxy_async_smem();   // the tensor core reads these operands next
            __syncwarp();
        };
        uint32_t kv_iter = 0;
        for (int it = 0;; ++it) {
            const int slot = it & 1;
            if (!warp_wait(&sm.unit_full[slot], (it >> 1) & 1, abort_flag, a.status)) break;
            const int4 d = sm.unit[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.unit_empty[slot]);
            if (d.x < 0) break;
            const UnitShape us = unit_shape(d);
            if (!warp_wait(&sm.q_full, it & 1, abort_flag, a.status)) break;
            for (int x = 0; x < (us.has_b ? 2 : 1); ++x) rotate_tile(sm.q[x], (us.tA + x) * kTile);
            if (lane == 0) mbar_arrive(&sm.q_rot);
            bool ok = true;
            for (int j = 0; j < us.n_kv; ++j, ++kv_iter) {
                const int st = kv_iter % kStages;
                if (!warp_wait(&sm.k_full[st], (kv_iter / kStages) & 1, abort_flag, a.status)) { ok = false; break; }
                rotate_tile(sm.k[st], j * kTile);
                if (lane == 0) mbar_arrive(&sm.k_rot[st]);
            }
            if (!ok) break;
        }
    }
    } else {
        setmaxnreg_inc<kSoftmaxRegs>();
        // ------------------------------------------------------------ softmax
        const int x = warp >> 2;                      // 0: tile A, 1: tile B
        const int r = threadIdx.x & 127;              // q row within the tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t s_col = x * 128, o_col = 256 + x * 128;
        const float sl2 = a.scale_log2;
        uint32_t s_cnt = 0, o_cnt = 0;                // S tiles and units this warpgroup consumed
        bool ok = true;
        for (int it = 0; ok; ++it) {
            const int slot = it & 1;
            if (!warp_wait(&sm.unit_full[slot], (it >> 1) & 1, abort_flag, a.status)) break;
            const int4 d = sm.unit[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.unit_empty[slot]);
            if (d.x < 0) break;
            const UnitShape us = unit_shape(d);
            if (x == 1 && !us.has_b) continue;
            const int h = d.x;
            const int tX = us.tA + x;
            const int nX = tX + 1;
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < nX; ++j) {
                if (!warp_wait(&sm.s_full[x], s_cnt & 1, abort_flag, a.status)) { ok = false; break; }
                ++s_cnt;
                tc_fence_after();
                const bool diag = (j == tX);
                // The whole S row (128 columns) is read once into registers.
                uint32_t sv[128];
                tmem_ld128(tmem + lane_off + s_col, sv);
                tmem_wait_ld();
                // row max: 8 independent chains of three-input maxima
                float mxs[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) mxs[e] = -INFINITY;
                if (diag) {
#pragma unroll
                    for (int e = 0; e < 128; ++e)
                        if (e <= r) mxs[e & 7] = fmaxf(mxs[e & 7], __uint_as_float(sv[e]));
                } else {
#pragma unroll
                    for (int e = 0; e < 128; e += 16)
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            mxs[c] = fmax3(mxs[c], __uint_as_float(sv[e + c]), __uint_as_float(sv[e + 8 + c]));
                }
                const float mx = fmaxf(fmax3(mxs[0], mxs[1], mxs[2]), fmax3(mxs[3], mxs[4], fmax3(mxs[5], mxs[6], mxs[7])));
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
                // P = 2^(S * scale * log2 e - m), written as bf16 over the first 64
                // columns of S_X's region (already in registers). Columns go in
                // pairs through the packed fp32 instructions (half the issue slots
                // of scalar ones: the loop is bound by instruction issue).
                const uint64_t sl2_2 = f2_pack(sl2, sl2), negm_2 = f2_pack(-m, -m);
                uint64_t sum2[2] = {0ull, 0ull};   // (0.f, 0.f)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int col = c * 32 + 2 * e;
                        const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(sv[col]), __uint_as_float(sv[col + 1])),
                                                   sl2_2, negm_2);
                        float p0, p1;
                        f2_unpack(x2, p0, p1);
                        p0 = ex2(p0);
                        p1 = ex2(p1);
                        if (diag) {
                            if (col > r) p0 = 0.f;
                            if (col + 1 > r) p1 = 0.f;
                        }
                        sum2[e & 1] = f2_add(sum2[e & 1], f2_pack(p0, p1));
                        pk[e] = pack_bf16x2(p0, p1);
                    }
                    tmem_st16(tmem + lane_off + s_col + c * 16, pk);
                }
                {
                    float a0, a1, b0, b1;
                    f2_unpack(sum2[0], a0, a1);
                    f2_unpack(sum2[1], b0, b1);
                    l += (a0 + a1) + (b0 + b1);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();                 // the warp's P stores are done: one arrive for all 32 lanes
                if (lane == 0) mbar_arrive(&sm.p_full[x]);
            }
            if (!ok) break;
            // epilogue: normalise O_X and store it with the row's LSE. O is read
            // out of TMEM (as bf16) before anything is stored, so the next unit's
            // first P V into O_X waits for the TMEM reads only.
            if (!warp_wait(&sm.o_done[x], o_cnt & 1, abort_flag, a.status)) { ok = false; break; }
            tc_fence_after();
            const int qi = d.y + tX * kTile + r;
            const bool valid = qi < d.z;
            const float inv_l = 1.f / l;
            uint32_t ow[D / 2];   // O row as bf16 pairs
#pragma unroll
            for (int c = 0; c < D / 32; c += 2) {
                uint32_t o[2][32];
                tmem_ld32(tmem + lane_off + o_col + c * 32, o[0]);
                tmem_ld32(tmem + lane_off + o_col + c * 32 + 32, o[1]);
                tmem_wait_ld();
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        ow[(c + h2) * 16 + e] =
                            pack_bf16x2(__uint_as_float(o[h2][2 * e]) * inv_l, __uint_as_float(o[h2][2 * e + 1]) * inv_l);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.o_free[x]);
            if (valid) a.lse[static_cast<size_t>(h) * a.total_tokens + qi] = (m + log2f(l)) * 0.69314718055994531f;
            // A quarter wholly inside the segment leaves through TMA stores of
            // [32 rows][64 d] boxes staged in this warp's slot (whole lines in HBM);
            // a quarter reaching past the segment end is stored row by row (a box
            // must not touch the next segment).
            const int row0 = d.y + tX * kTile + (warp & 3) * 32;
            if (row0 + 32 <= d.z) {
                const uint32_t slot = smem_u32(sm.ostage[warp]);
#pragma unroll
                for (int half = 0; half < D / 64; ++half) {
                    if (lane == 0) bulk_wait_group_read0();   // the slot's last store has been read
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(slot + lane * 128 + ((j ^ (lane & 7)) << 4), ow[half * 32 + 4 * j],
                                     ow[half * 32 + 4 * j + 1], ow[half * 32 + 4 * j + 2], ow[half * 32 + 4 * j + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&a.tm_o, sm.ostage[warp], half * 64, h, row0);
                        bulk_commit_group();
                    }
                }
            } else if (valid) {
                uint4 *dst = reinterpret_cast<uint4 *>(a.out + (static_cast<size_t>(qi) * a.Hq + h) * D);
#pragma unroll
                for (int e = 0; e < D / 8; ++e) dst[e] = make_uint4(ow[4 * e], ow[4 * e + 1], ow[4 * e + 2], ow[4 * e + 3]);
            }
            ++o_cnt;
        }
        if (lane == 0) bulk_wait_group0();   // this warp's O stores have landed
        __syncwarp();
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
    // Persistent: one CTA per SM takes work units from the shared counter.
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    int64_t grid = grid_units * a.Hq;
    if (grid > sms) grid = sms;
    if (grid <= 0) return cudaSuccess;
    prof_begin(kProfAttnFwd, stream);
    attn_fwd_kernel<D><<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(a);
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
