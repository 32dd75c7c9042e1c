// Rotary position embedding with per-document positions, in place on q and k.
//
// The attention-layer pseudo code under Figure 1 of the XTuner page "序列并行"
// ("Sequence parallel") rotates q and k (apply_rotary_pos_emb) right before
// attention; packed documents take their positions from the pack's `indexes`
// (InternEvo page "Data loading and flow", section "Fetching data from the
// Dataloader": position inside the current segment), i.e. they restart at every
// document (page "Sample Packing: attention problems of long-sequence LLM
// training", section 4.1, reset_position_id). Rotate-half form: channel j of a
// head pairs with channel j + d/2 and turns by p * theta_j, theta_j =
// base^(-2j/d); the inverse turns by -p * theta_j (the gradient with respect to
// the input).
//
// The phase is kept exactly: the host passes every frequency as a 64-bit
// fixed-point number of turns per position, F_j = theta_j / (2 pi) * 2^64; the
// wrapping integer product p * F_j is the phase in turns modulo 1 (error
// ~2^-53 turns per position from the fp64 rounding of F_j), whose top 32 bits
// feed sincospif. A float angle p * theta_j would be off by up to p * 2^-24
// radians (1% at p ~ 10^5).
#include "internal.h"
#include "ptx.cuh"

namespace spd {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__global__ void __launch_bounds__(kThreads) rope_kernel(const __grid_constant__ RopeArgs a)
{
    // one thread per (token, group of 8 channel pairs)
    const int groups = a.d / 16;
    const int64_t n = static_cast<int64_t>(a.T) * groups;
    for (int64_t x = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; x < n;
         x += static_cast<int64_t>(gridDim.x) * kThreads) {
        const int tok = static_cast<int>(x / groups), g = static_cast<int>(x % groups);
        const uint64_t p = static_cast<uint32_t>(a.pos[tok]);
        float c[8], s[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint64_t ph = p * a.freq[g * 8 + e];                      // turns * 2^64, mod 2^64
            const int32_t half_turns = static_cast<int32_t>(static_cast<uint32_t>(ph >> 32));
            const float u = static_cast<float>(half_turns) * 4.656612873077393e-10f;  // 2^-31: in [-1, 1)
            sincospif(u, &s[e], &c[e]);                                     // sin / cos of pi u = 2 pi turns
            if (a.inverse) s[e] = -s[e];
        }
        for (int which = 0; which < 2; ++which) {
            uint16_t *base = which ? a.k : a.q;
            const int H = which ? a.Hkv : a.Hq;
            if (!base) continue;
            // four heads at a time: all eight loads are issued before the first
            // store, so a thread keeps 128 bytes in flight
            constexpr int kHeads = 4;
            for (int h0 = 0; h0 < H; h0 += kHeads) {
                uint4 lo4[kHeads], hi4[kHeads];
#pragma unroll
                for (int u = 0; u < kHeads; ++u) {
                    if (h0 + u < H) {
                        const uint16_t *row = base + (static_cast<size_t>(tok) * H + h0 + u) * a.d;
                        lo4[u] = *reinterpret_cast<const uint4 *>(row + g * 8);
                        hi4[u] = *reinterpret_cast<const uint4 *>(row + a.d / 2 + g * 8);
                    }
                }
#pragma unroll
                for (int u = 0; u < kHeads; ++u) {
                    if (h0 + u >= H) break;
                    const uint32_t lo[4] = {lo4[u].x, lo4[u].y, lo4[u].z, lo4[u].w};
                    const uint32_t hi[4] = {hi4[u].x, hi4[u].y, hi4[u].z, hi4[u].w};
                    uint32_t olo[4], ohi[4];
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const float x0 = bf_lo(lo[w]), x1 = bf_hi(lo[w]);     // channels j, j + 1
                        const float y0 = bf_lo(hi[w]), y1 = bf_hi(hi[w]);     // channels j + d/2, j + 1 + d/2
                        const int e0 = 2 * w, e1 = 2 * w + 1;
                        olo[w] = pack_bf16x2(x0 * c[e0] - y0 * s[e0], x1 * c[e1] - y1 * s[e1]);
                        ohi[w] = pack_bf16x2(y0 * c[e0] + x0 * s[e0], y1 * c[e1] + x1 * s[e1]);
                    }
                    uint16_t *row = base + (static_cast<size_t>(tok) * H + h0 + u) * a.d;
                    *reinterpret_cast<uint4 *>(row + g * 8) = make_uint4(olo[0], olo[1], olo[2], olo[3]);
                    *reinterpret_cast<uint4 *>(row + a.d / 2 + g * 8) = make_uint4(ohi[0], ohi[1], ohi[2], ohi[3]);
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_rope(const RopeArgs &a, int num_sms, cudaStream_t stream)
{
    const int64_t n = static_cast<int64_t>(a.T) * (a.d / 16);
    if (n == 0) return cudaSuccess;
    long long blocks = (n + kThreads - 1) / kThreads;
    const long long cap = static_cast<long long>(num_sms > 0 ? num_sms : 1) * 8;
    if (blocks > cap) blocks = cap;
    prof_begin(kProfRope, stream);
    rope_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(a);
    prof_end(kProfRope, stream);
    return cudaGetLastError();
}

}  // namespace spd
