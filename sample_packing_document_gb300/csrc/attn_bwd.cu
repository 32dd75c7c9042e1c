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
//                    accumulator, laid out [Hq][d / 32][T][32].
//   attn_bwd_kernel  one CTA per (128-row kv tile, kv head): K, V stay in shared
//                    memory; the CTA walks every (q head of the group, q tile
//                    from the diagonal to the segment end). Per step, five
//                    tcgen05 MMAs with fp32 accumulation in TMEM:
//                      S^T = K Q^T           region A (P^T is then written over it, bf16)
//                      dP^T = V dO^T         region B
//                      dV += P^T dO          region C (P^T read from TMEM)
//                      dK += dS^T Q          region E (dS^T from shared memory)
//                      dQ_part = dS K        region B (once dP^T has been read), then
//                                            TMA reduce-add into the HBM accumulator.
//   bwd_dq_kernel    dq = scale * accumulator, in the output layout and type.
//
// Warp roles (576 threads). Warp w works on TMEM lanes 32 (w % 4) .. +31 (kv
// rows; q rows for the dQ read-out) and on one half of the columns:
//   warps 0-7   "P": P^T(i) = exp(S^T(i) * scale - LSE) from region A, written
//               back into it as bf16 (the P^T columns of a half sit in the first
//               half of that half's S^T columns); then one 32 x 32 chunk of the
//               dQ(i) read-out, staged in the spent Q(i) stage, and its reduce-add.
//   warps 8-15  "dS": dS^T(i) = P^T(i) (dP^T(i) - D) into shared memory, then one
//               chunk of the dQ(i) read-out, staged in the dS buffer; at the end
//               the dK / dV stores.
//   warp 16     TMA producer; warp 17 issues the MMAs in the order
//              dV(i), dK(i), dQ(i), S(i+1), dP(i+1), dV(i+1), ...
// so P(i+1) is computed while dK(i) / dQ(i) run, dS(i) while dV(i) runs, and the
// dQ(i) read-out while S(i+1) runs.
#include "internal.h"
#include "ptx.cuh"

namespace spd {
namespace {

constexpr int kThreads = 576;        // 16 compute warps + producer + MMA issuer
constexpr int kPWarps = 8, kDsWarps = 8;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAtom = 128 * 128;
constexpr int kQStages = 2;

template <int D>
struct BwdSmem {
    uint8_t k[D / 64][kAtom];
    uint8_t v[D / 64][kAtom];
    uint8_t q[kQStages][D / 64][kAtom];
    uint8_t dout[kQStages][D / 64][kAtom];
    uint8_t ds[2][kAtom];            // dS^T: [128 kv rows][128 q cols]
    float lse2[2][128];              // LSE * log2(e) of the step's q columns
    float delta[2][128];             // D of the step's q columns
    uint64_t kv_full;
    uint64_t q_full[kQStages], q_empty[kQStages], do_full[kQStages], do_empty[kQStages];
    uint64_t s_full, dp_full, p_full, ds_full, dq_full, dq_free;
    uint64_t cols_l[2], cols_d[2];   // the step's lse2 / delta written
    uint64_t fin, drain;
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
    // kv-head-major order: the CTAs of one kv head run together, so the Q / dO
    // tiles they share and the dQ rows they add into stay in L2.
    const int g = blockIdx.x / a.grid_tiles;
    const int tile_idx = blockIdx.x % a.grid_tiles;
    if (tile_idx >= *a.tile_count) return;
    const Tile tl = a.tiles[tile_idx];
    const int group = a.Hq / a.Hkv;
    const int n_seg_tiles = (tl.seg_end - tl.seg_start + kTile - 1) / kTile;
    const int nq = n_seg_tiles - tl.t;   // q tiles t .. n-1
    const int nsteps = group * nq;
    const int k0 = tl.seg_start + tl.t * kTile;

    if (threadIdx.x == 0) {
        mbar_init(&sm.kv_full, 1);
        for (int s = 0; s < kQStages; ++s) {
            mbar_init(&sm.q_full[s], 1);
            mbar_init(&sm.q_empty[s], 4 * (D / 64));  // the P warps that stage dQ there, once it is read
            mbar_init(&sm.do_full[s], 1);
            mbar_init(&sm.do_empty[s], 1);
        }
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.dp_full, 1);
        mbar_init(&sm.p_full, 32 * kPWarps);
        mbar_init(&sm.ds_full, 32 * kDsWarps);
        mbar_init(&sm.dq_full, 1);
        mbar_init(&sm.dq_free, 32 * (kPWarps + kDsWarps));
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.cols_l[b], 128);
            mbar_init(&sm.cols_d[b], 128);
        }
        mbar_init(&sm.fin, 1);
        mbar_init(&sm.drain, 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 17) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 16 && lane == 0) {
        tma_prefetch_desc(&a.tm_q);
        tma_prefetch_desc(&a.tm_k);
        tma_prefetch_desc(&a.tm_v);
        tma_prefetch_desc(&a.tm_do);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    volatile int *abort_flag = &sm.abort_flag;
    constexpr uint32_t kTileBytes = 128 * D * 2;
    constexpr uint32_t kA = 0, kB = 128, kC = 256, kE = 256 + D;

    if (warp == 16) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            mbar_arrive_expect_tx(&sm.kv_full, 2 * kTileBytes);
            for (int c = 0; c < D / 64; ++c) {
                tma_load_3d(sm.k[c], &a.tm_k, c * 64, g, k0, &sm.kv_full);
                tma_load_3d(sm.v[c], &a.tm_v, c * 64, g, k0, &sm.kv_full);
            }
            int last_q[kQStages], last_do[kQStages];
            for (int s = 0; s < kQStages; ++s) last_q[s] = last_do[s] = -1;
            for (int i = 0; i < nsteps; ++i) {
                const int st = i % kQStages, u = i / kQStages;
                const int h = g * group + i / nq;
                const int q0 = tl.seg_start + (tl.t + i % nq) * kTile;
                if (u > 0 && !mbar_wait(&sm.q_empty[st], (u - 1) & 1, abort_flag, a.status)) break;
                mbar_arrive_expect_tx(&sm.q_full[st], kTileBytes);
                for (int c = 0; c < D / 64; ++c) tma_load_3d(sm.q[st][c], &a.tm_q, c * 64, h, q0, &sm.q_full[st]);
                last_q[st] = u;
                if (u > 0 && !mbar_wait(&sm.do_empty[st], (u - 1) & 1, abort_flag, a.status)) break;
                mbar_arrive_expect_tx(&sm.do_full[st], kTileBytes);
                for (int c = 0; c < D / 64; ++c)
                    tma_load_3d(sm.dout[st][c], &a.tm_do, c * 64, h, q0, &sm.do_full[st]);
                last_do[st] = u;
            }
            if (*abort_flag) {
                // Let the copies still in flight land before the CTA exits.
                wait_drain(&sm.kv_full, 0);
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
            const uint32_t k_addr = smem_u32(sm.k[0]), v_addr = smem_u32(sm.v[0]);
            const uint32_t ds_addr = smem_u32(sm.ds[0]);
            int do_commits[kQStages] = {};
            auto issue_s = [&](int i) -> bool {   // S^T(i) = K Q(i)^T into A
                const int st = i % kQStages;
                if (!mbar_wait(&sm.q_full[st], (i / kQStages) & 1, abort_flag, a.status)) return false;
                tc_fence_after();
                const uint32_t q_addr = smem_u32(sm.q[st][0]);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kAtom + (kk & 3) * 32;
                    umma_bf16(tmem + kA, sdesc_sw128(k_addr + off, 16, 1024), sdesc_sw128(q_addr + off, 16, 1024),
                              id_ss, kk > 0 ? 1u : 0u);
                }
                umma_commit(&sm.s_full);
                return true;
            };
            auto issue_dp = [&](int i) -> bool {  // dP^T(i) = V dO(i)^T into B, once dQ(i-1) left B
                const int st = i % kQStages;
                if (!mbar_wait(&sm.do_full[st], (i / kQStages) & 1, abort_flag, a.status)) return false;
                if (i > 0 && !mbar_wait(&sm.dq_free, (i - 1) & 1, abort_flag, a.status)) return false;
                tc_fence_after();
                const uint32_t do_addr = smem_u32(sm.dout[st][0]);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kAtom + (kk & 3) * 32;
                    umma_bf16(tmem + kB, sdesc_sw128(v_addr + off, 16, 1024), sdesc_sw128(do_addr + off, 16, 1024),
                              id_ss, kk > 0 ? 1u : 0u);
                }
                umma_commit(&sm.dp_full);
                return true;
            };
            bool ok = mbar_wait(&sm.kv_full, 0, abort_flag, a.status) && issue_s(0) && issue_dp(0);
            for (int i = 0; ok && i < nsteps; ++i) {
                const int st = i % kQStages;
                const uint32_t ph = i & 1;
                // dV += P^T(i) dO(i): P^T in TMEM over S^T (M = kv, K = q), dO MN-major
                if (!mbar_wait(&sm.p_full, ph, abort_flag, a.status)) { ok = false; break; }
                tc_fence_after();
                {
                    const uint32_t do_addr = smem_u32(sm.dout[st][0]);
#pragma unroll
                    for (int kk = 0; kk < 128 / 16; ++kk)
                        // P^T q columns 16kk .. 16kk+15 sit at TMEM column 64 (kk / 4) + 8 (kk % 4)
                        umma_bf16_ts(tmem + kC, tmem + kA + (kk >> 2) * 64 + (kk & 3) * 8,
                                     sdesc_sw128(do_addr + kk * 2048, kAtom, 1024), id_kn, (i > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(&sm.do_empty[st]);
                ++do_commits[st];
                // dK += dS^T Q(i) (M = kv), dQ_part = dS K (M = q) into B
                if (!mbar_wait(&sm.ds_full, ph, abort_flag, a.status)) { ok = false; break; }
                tc_fence_after();
                {
                    const uint32_t q_addr = smem_u32(sm.q[st][0]);
#pragma unroll
                    for (int kk = 0; kk < 128 / 16; ++kk)
                        umma_bf16(tmem + kE, sdesc_sw128(ds_addr + (kk >> 2) * kAtom + (kk & 3) * 32, 16, 1024),
                                  sdesc_sw128(q_addr + kk * 2048, kAtom, 1024), id_kn, (i > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                    for (int kk = 0; kk < 128 / 16; ++kk)
                        umma_bf16(tmem + kB, sdesc_sw128(ds_addr + kk * 2048, kAtom, 1024),
                                  sdesc_sw128(k_addr + kk * 2048, kAtom, 1024), id_mn, kk > 0 ? 1u : 0u);
                }
                umma_commit(&sm.dq_full);
                // next step: S^T(i+1) over P^T(i) (dV(i) ran before it and the dS warps
                // read P^T(i) before ds_full(i)), then dP^T(i+1)
                if (i + 1 < nsteps && !(issue_s(i + 1) && issue_dp(i + 1))) { ok = false; break; }
            }
            umma_commit(&sm.fin);
            umma_commit(&sm.drain);
            wait_drain(&sm.drain, 0);
            for (int s = 0; s < kQStages; ++s)
                if (do_commits[s] > 0) wait_drain(&sm.do_empty[s], (do_commits[s] - 1) & 1);
        }
    } else if (warp < kPWarps) {
        // ------------------------------------------------------------ P warps
        const int quarter = warp & 3, half = warp >> 2;
        const int t = quarter * 32 + lane;                        // kv row = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const int col0 = half * 64;                               // this warp's 64 q columns
        const float sl2 = a.scale_log2;
        const int kj = k0 + t;
        const bool loader = half == 0;                            // loads the step's LSE column t
        const int my_chunk = half;                                // dQ read-out chunk (d columns 32c..)
        const bool reads_out = my_chunk < D / 64;
        bool ok = true;
        auto col_term = [&](int i) -> float {
            const int h = g * group + i / nq;
            const int qi = tl.seg_start + (tl.t + i % nq) * kTile + t;
            if (qi >= a.total_tokens) return 0.f;
            return a.lse[static_cast<size_t>(h) * a.total_tokens + qi] * 1.4426950408889634f;
        };
        float nxt = loader ? col_term(0) : 0.f;
        for (int i = 0; i < nsteps; ++i) {
            const int h = g * group + i / nq;
            const int q0 = tl.seg_start + (tl.t + i % nq) * kTile;
            if (loader) {
                sm.lse2[i & 1][t] = nxt;
                mbar_arrive(&sm.cols_l[i & 1]);
                if (i + 1 < nsteps) nxt = col_term(i + 1);
            }
            if (!warp_wait(&sm.cols_l[i & 1], (i >> 1) & 1, abort_flag, a.status)) { ok = false; break; }
            const float *L2 = sm.lse2[i & 1] + col0;
            // column col0 + c (q row q0 + col0 + c) is live for kv row kj iff kj <= q row < seg_end
            const int c_lo = kj - q0 - col0, c_hi = tl.seg_end - q0 - col0;
            const bool full = c_lo <= 0 && c_hi >= 64;
            if (!warp_wait(&sm.s_full, i & 1, abort_flag, a.status)) { ok = false; break; }
            tc_fence_after();
            // P^T columns col0 + 32c .. +31 (bf16 pairs) go to TMEM columns col0 + 16c ..
            // +15, inside the S^T columns this warp has already read itself.
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t sv[32];
                tmem_ld32(tmem + lane_off + kA + col0 + c * 32, sv);
                tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int col = c * 32 + 2 * e;
                    float p0 = ex2(__uint_as_float(sv[2 * e]) * sl2 - L2[col]);
                    float p1 = ex2(__uint_as_float(sv[2 * e + 1]) * sl2 - L2[col + 1]);
                    if (!full) {
                        if (col < c_lo || col >= c_hi) p0 = 0.f;
                        if (col + 1 < c_lo || col + 1 >= c_hi) p1 = 0.f;
                    }
                    pk[e] = pack_bf16x2(p0, p1);
                }
                tmem_st16(tmem + lane_off + kA + col0 + c * 16, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&sm.p_full);
            // The Q(i-1) stage held this warp's staged dQ(i-1) chunk: once the TMA
            // engine has read it (it had the whole P computation to do so) the
            // stage goes back to the producer.
            if (i > 0 && reads_out) {
                if (lane == 0) {
                    bulk_wait_group_read0();
                    mbar_arrive(&sm.q_empty[(i - 1) % kQStages]);
                }
                __syncwarp();
            }
            // dQ(i) read-out of one [32 rows][32 cols] chunk, staged in this warp's
            // slice of the Q(i) stage (free once dK(i) completed) in the 128-byte-
            // swizzled layout and added by the TMA engine in the background.
            if (!warp_wait(&sm.dq_full, i & 1, abort_flag, a.status)) { ok = false; break; }
            tc_fence_after();
            if (reads_out) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_off + kB + my_chunk * 32, v);
                tmem_wait_ld();
                const uint8_t *stage = sm.q[i % kQStages][0] + (quarter + 4 * my_chunk) * 4096;
                const uint32_t stage_addr = smem_u32(stage);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    st_shared_v4(stage_addr + lane * 128 + ((e ^ (lane & 7)) << 4), v[4 * e], v[4 * e + 1],
                                 v[4 * e + 2], v[4 * e + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (q0 + quarter * 32 < tl.seg_end)   // skip a chunk of padding rows only
                        tma_reduce_add_3d(&a.tm_dqacc, stage, 0, q0 + quarter * 32, h * (D / 32) + my_chunk);
                    bulk_commit_group();
                }
            }
            tc_fence_before();
            mbar_arrive(&sm.dq_free);
        }
        if (lane == 0) bulk_wait_group0();     // every reduce of this warp has landed
        __syncwarp();
        (void)ok;
    } else {
        // ------------------------------------------------------------ dS warps
        const int w = warp - kPWarps;
        const int quarter = w & 3, half = w >> 2;
        const int t = quarter * 32 + lane;                        // kv row / q row = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t ds_addr = smem_u32(sm.ds[0]);
        const int col0 = half * 64;                               // this warp's 64 q columns
        const int kj = k0 + t;
        const bool loader = half == 0;                            // loads the step's D column t
        const int my_chunk = D / 64 + half;                       // dQ read-out chunk, if any
        const bool reads_out = my_chunk < D / 32;
        bool ok = true;
        auto col_term = [&](int i) -> float {
            const int h = g * group + i / nq;
            const int qi = tl.seg_start + (tl.t + i % nq) * kTile + t;
            if (qi >= a.total_tokens) return 0.f;
            return a.delta[static_cast<size_t>(h) * a.total_tokens + qi];
        };
        float nxt = loader ? col_term(0) : 0.f;
        for (int i = 0; i < nsteps; ++i) {
            const int h = g * group + i / nq;
            const int q0 = tl.seg_start + (tl.t + i % nq) * kTile;
            const uint32_t ph = i & 1;
            if (loader) {
                sm.delta[i & 1][t] = nxt;
                mbar_arrive(&sm.cols_d[i & 1]);
                if (i + 1 < nsteps) nxt = col_term(i + 1);
            }
            if (!warp_wait(&sm.cols_d[i & 1], (i >> 1) & 1, abort_flag, a.status)) { ok = false; break; }
            const float *DD = sm.delta[i & 1] + col0;
            // dS^T = P^T * (dP^T - D); P^T read back from TMEM (bf16), masked entries are 0
            if (!warp_wait(&sm.dp_full, ph, abort_flag, a.status)) { ok = false; break; }
            if (!warp_wait(&sm.p_full, ph, abort_flag, a.status)) { ok = false; break; }
            tc_fence_after();
            // This warp's slice of the dS buffer held its staged dQ(i-1) chunk: it is
            // reusable once the TMA engine has read it (dK(i-1) / dQ(i-1), its other
            // readers, completed before dq_full(i-1)). dP(i) ran meanwhile.
            if (i > 0 && reads_out) {
                if (lane == 0) bulk_wait_group_read0();
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
                for (int e = 0; e < 16; ++e) {
                    const int col = c * 32 + 2 * e;
                    const float d0 = bf16_lo(pv[e]) * (__uint_as_float(dp[2 * e]) - DD[col]);
                    const float d1 = bf16_hi(pv[e]) * (__uint_as_float(dp[2 * e + 1]) - DD[col + 1]);
                    pk[e] = pack_bf16x2(d0, d1);
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

            // dQ(i) read-out of one [32 rows][32 cols] chunk, staged in this warp's
            // slice of the dS buffer (free: dK(i) and dQ(i) completed) in the 128-
            // byte-swizzled layout and added by the TMA engine in the background.
            // Rows past the segment carry exact zeros.
            if (!warp_wait(&sm.dq_full, ph, abort_flag, a.status)) { ok = false; break; }
            tc_fence_after();
            if (reads_out) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_off + kB + my_chunk * 32, v);
                tmem_wait_ld();
                const uint8_t *stage = sm.ds[0] + (quarter + 4 * half) * 4096;
                const uint32_t stage_addr = smem_u32(stage);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    st_shared_v4(stage_addr + lane * 128 + ((e ^ (lane & 7)) << 4), v[4 * e], v[4 * e + 1],
                                 v[4 * e + 2], v[4 * e + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (q0 + quarter * 32 < tl.seg_end)   // skip a chunk of padding rows only
                        tma_reduce_add_3d(&a.tm_dqacc, stage, 0, q0 + quarter * 32, h * (D / 32) + my_chunk);
                    bulk_commit_group();
                }
            }
            tc_fence_before();
            mbar_arrive(&sm.dq_free);
        }
        if (lane == 0) bulk_wait_group0();     // every reduce of this warp has landed
        __syncwarp();
        // dK, dV rows of this tile, d columns [half * D/2, half * D/2 + D/2)
        if (ok && warp_wait(&sm.fin, 0, abort_flag, a.status)) {
            tc_fence_after();
            const bool live = kj < tl.seg_end;
            const size_t orow = (static_cast<size_t>(kj) * a.Hkv + g) * D + half * (D / 2);
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const uint32_t col = (which ? kE : kC) + half * (D / 2);
                const float mul = which ? a.scale : 1.f;
                void *base = which ? a.dk : a.dv;
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_off + col + c * 32, v);
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
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 17) tmem_dealloc(tmem, kTmemCols);
}

template <int D>
cudaError_t launch_bwd_d(const AttnBwdArgs &a, int64_t grid_tiles, cudaStream_t stream)
{
    const int T = a.total_tokens;
    const long long rows = static_cast<long long>(T) * a.Hq;
    {
        long long blocks = (rows * 8 + 255) / 256;
        if (blocks > 152 * 16) blocks = 152 * 16;
        if (blocks < 1) blocks = 1;
        bwd_pre_kernel<D><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a.out, a.dout, a.delta, a.dq_acc, T, a.Hq);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const size_t smem = sizeof(BwdSmem<D>);
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    AttnBwdArgs a2 = a;
    a2.grid_tiles = static_cast<int32_t>(grid_tiles);
    const int64_t grid = grid_tiles * a.Hkv;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
    if (grid > 0) {
        prof_begin(kProfAttnBwd, stream);
        attn_bwd_kernel<D><<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(a2);
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

cudaError_t launch_attn_bwd(const AttnBwdArgs &a, int head_dim, int64_t grid_tiles, cudaStream_t stream)
{
    if (head_dim == 64) return launch_bwd_d<64>(a, grid_tiles, stream);
    if (head_dim == 128) return launch_bwd_d<128>(a, grid_tiles, stream);
    return cudaErrorInvalidValue;
}

}  // namespace spd
