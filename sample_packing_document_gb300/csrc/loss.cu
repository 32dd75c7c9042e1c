// Masked token loss over packed labels (XTuner page "序列并行", section
// "Reduce Loss": the mean token cross-entropy over labels that are not -100,
// with num_tokens = (labels != -100).sum() as the weight of the rank's loss in
// reduce_sequence_parallel_loss). The labels are the pack's (-100 at document
// ends and padding).
//
// loss_row_kernel: one CTA per token row of V bf16 logits, one pass: each thread
// keeps a running (max, sum of 2^(y - max)) over its 16-byte chunks (y = logit *
// log2 e), the CTA combines them, loss = (lse2 - y[label]) * ln 2. With a
// gradient buffer, a second pass over the row (still in L2) writes
// (softmax - onehot(label)) * grad_scale as bf16.
// loss_row_smem_kernel: the same with the row staged in shared memory by one
// bulk copy (vocabularies up to 57344): HBM sees each logit once.
// loss_sum_kernel: one CTA sums the per-token losses in fp64 in a fixed order
// (deterministic) and counts the tokens.
#include "internal.h"
#include "ptx.cuh"

namespace spd {
namespace {

constexpr int kRowThreads = 256, kSumThreads = 1024;
constexpr int32_t kIgnore = -100;
constexpr float kLog2e = 1.4426950408889634f, kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float bf16_to_f(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

// the gradient row of a token that is not counted is zero
__device__ __forceinline__ void zero_row(uint16_t *grow, int V, int tid)
{
    if (!grow) return;
    for (int i = tid; i < V; i += kRowThreads) grow[i] = 0;
}

// (m, s) pairs with s = sum 2^(y - m): combine two partial sums
__device__ __forceinline__ void lse_combine(float &m, float &s, float m2, float s2)
{
    const float mn = fmaxf(m, m2);
    if (mn == -INFINITY) return;
    s = s * ex2(m - mn) + s2 * ex2(m2 - mn);
    m = mn;
}

__global__ void __launch_bounds__(kRowThreads) loss_row_kernel(LossArgs a)
{
    __shared__ float sm_m[kRowThreads / 32], sm_s[kRowThreads / 32];
    __shared__ float row_lse2;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int t = blockIdx.x; t < a.T; t += gridDim.x) {
        const int32_t lab = a.labels[t];
        const uint16_t *row = a.logits + static_cast<size_t>(t) * a.V;
        uint16_t *grow = a.dlogits ? a.dlogits + static_cast<size_t>(t) * a.V : nullptr;
        const bool counted = lab != kIgnore;
        if (counted && (lab < 0 || lab >= a.V)) {   // a label outside the vocabulary
            if (tid == 0) {
                a.token_loss[t] = 0.f;
                if (a.status) atomicExch(a.status, kErrInvalidArg);
            }
            zero_row(grow, a.V, tid);
            continue;
        }
        if (!counted) {
            if (tid == 0) a.token_loss[t] = 0.f;
            zero_row(grow, a.V, tid);
            continue;
        }
        float m = -INFINITY, s = 0.f;
        if (a.vec) {
            for (int i = tid * 8; i < a.V; i += kRowThreads * 8) {
                const uint4 w = *reinterpret_cast<const uint4 *>(row + i);
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
                float y[8], cm = -INFINITY;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    y[2 * e] = __uint_as_float(ww[e] << 16) * kLog2e;
                    y[2 * e + 1] = __uint_as_float(ww[e] & 0xffff0000u) * kLog2e;
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) cm = fmaxf(cm, y[e]);
                float cs = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) cs += ex2(y[e] - cm);
                lse_combine(m, s, cm, cs);
            }
        } else {
            for (int i = tid; i < a.V; i += kRowThreads) lse_combine(m, s, bf16_to_f(row[i]) * kLog2e, 1.f);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
            lse_combine(m, s, m2, s2);
        }
        if (lane == 0) {
            sm_m[warp] = m;
            sm_s[warp] = s;
        }
        __syncthreads();
        if (tid == 0) {
            float M = sm_m[0], S = sm_s[0];
            for (int w = 1; w < kRowThreads / 32; ++w) lse_combine(M, S, sm_m[w], sm_s[w]);
            const float lse2 = M + __log2f(S);
            row_lse2 = lse2;
            a.token_loss[t] = (lse2 - bf16_to_f(row[lab]) * kLog2e) * kLn2;
        }
        __syncthreads();
        if (grow) {
            const float lse2 = row_lse2, sc = a.grad_scale;
            if (a.vec) {
                for (int i = tid * 8; i < a.V; i += kRowThreads * 8) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(row + i);
                    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
                    uint32_t o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j = i + 2 * e;
                        const float p0 = ex2(__uint_as_float(ww[e] << 16) * kLog2e - lse2) - (j == lab ? 1.f : 0.f);
                        const float p1 = ex2(__uint_as_float(ww[e] & 0xffff0000u) * kLog2e - lse2) -
                                         (j + 1 == lab ? 1.f : 0.f);
                        o[e] = pack_bf16x2(p0 * sc, p1 * sc);
                    }
                    *reinterpret_cast<uint4 *>(grow + i) = make_uint4(o[0], o[1], o[2], o[3]);
                }
            } else {
                for (int i = tid; i < a.V; i += kRowThreads) {
                    const float p = ex2(bf16_to_f(row[i]) * kLog2e - lse2) - (i == lab ? 1.f : 0.f);
                    grow[i] = static_cast<uint16_t>(pack_bf16x2(p * sc, 0.f) & 0xffffu);
                }
            }
        }
        __syncthreads();   // sm_m / row_lse2 are reused by the next row
    }
}

// The same with the row staged once in shared memory by a bulk copy (rows of
// at most kSmemRowMax bf16, 16-byte aligned): both passes read shared memory,
// so HBM sees every logit once even when the gradient is written.
constexpr int kSmemRowMax = 56 * 1024;   // 112 KB of bf16: two CTAs per SM

__global__ void __launch_bounds__(kRowThreads) loss_row_smem_kernel(LossArgs a)
{
    extern __shared__ __align__(16) uint8_t smem_row[];
    __shared__ float sm_m[kRowThreads / 32], sm_s[kRowThreads / 32];
    __shared__ float row_lse2;
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint16_t *srow = reinterpret_cast<const uint16_t *>(smem_row);
    const uint32_t row_bytes = static_cast<uint32_t>(a.V) * 2;
    if (tid == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    uint32_t loads = 0;
    int dummy_status = 0;
    bool timed_out = false;
    for (int t = blockIdx.x; t < a.T; t += gridDim.x) {
        const int32_t lab = a.labels[t];
        uint16_t *grow = a.dlogits ? a.dlogits + static_cast<size_t>(t) * a.V : nullptr;
        if (lab == kIgnore || lab < 0 || lab >= a.V) {
            if (tid == 0) {
                a.token_loss[t] = 0.f;
                if (lab != kIgnore && a.status) atomicExch(a.status, kErrInvalidArg);
            }
            zero_row(grow, a.V, tid);
            continue;
        }
        if (tid == 0) {
            mbar_arrive_expect_tx(&bar, row_bytes);
            bulk_load(smem_row, a.logits + static_cast<size_t>(t) * a.V, row_bytes, &bar);
        }
        // bounded wait; a copy that never lands leaves the row's loss at 0
        const bool ok = mbar_wait(&bar, loads & 1, &abort_flag, a.status ? a.status : &dummy_status);
        ++loads;
        if (!__syncthreads_and(ok)) {
            timed_out = true;
            break;
        }
        float m = -INFINITY, s = 0.f;
        for (int i = tid * 8; i < a.V; i += kRowThreads * 8) {
            const uint4 w = *reinterpret_cast<const uint4 *>(srow + i);
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
            float y[8], cm = -INFINITY;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                y[2 * e] = __uint_as_float(ww[e] << 16) * kLog2e;
                y[2 * e + 1] = __uint_as_float(ww[e] & 0xffff0000u) * kLog2e;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) cm = fmaxf(cm, y[e]);
            float cs = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) cs += ex2(y[e] - cm);
            lse_combine(m, s, cm, cs);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
            lse_combine(m, s, m2, s2);
        }
        if (lane == 0) {
            sm_m[warp] = m;
            sm_s[warp] = s;
        }
        __syncthreads();
        if (tid == 0) {
            float M = sm_m[0], S = sm_s[0];
            for (int w = 1; w < kRowThreads / 32; ++w) lse_combine(M, S, sm_m[w], sm_s[w]);
            const float lse2 = M + __log2f(S);
            row_lse2 = lse2;
            a.token_loss[t] = (lse2 - bf16_to_f(srow[lab]) * kLog2e) * kLn2;
        }
        __syncthreads();
        if (grow) {
            const float lse2 = row_lse2, sc = a.grad_scale;
            for (int i = tid * 8; i < a.V; i += kRowThreads * 8) {
                const uint4 w = *reinterpret_cast<const uint4 *>(srow + i);
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
                uint32_t o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = i + 2 * e;
                    const float p0 = ex2(__uint_as_float(ww[e] << 16) * kLog2e - lse2) - (j == lab ? 1.f : 0.f);
                    const float p1 = ex2(__uint_as_float(ww[e] & 0xffff0000u) * kLog2e - lse2) -
                                     (j + 1 == lab ? 1.f : 0.f);
                    o[e] = pack_bf16x2(p0 * sc, p1 * sc);
                }
                *reinterpret_cast<uint4 *>(grow + i) = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
        __syncthreads();   // the next row's copy overwrites the staged row
    }
    // The copy that timed out may still land: its issuing thread waits for it
    // once more (bounded) so the CTA's shared memory outlives it.
    if (timed_out && tid == 0) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&bar, (loads - 1) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
    }
}

__global__ void __launch_bounds__(kSumThreads) loss_sum_kernel(LossArgs a)
{
    __shared__ double sh_s[kSumThreads / 32];
    __shared__ int sh_n[kSumThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    double s = 0.0;
    int n = 0;
    for (int t = tid; t < a.T; t += kSumThreads) {   // fixed order: the sum is reproducible
        s += static_cast<double>(a.token_loss[t]);
        const int32_t lab = a.labels[t];
        n += (lab != kIgnore && lab >= 0 && lab < a.V) ? 1 : 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        s += __shfl_xor_sync(0xffffffffu, s, o);
        n += __shfl_xor_sync(0xffffffffu, n, o);
    }
    if (lane == 0) {
        sh_s[warp] = s;
        sh_n[warp] = n;
    }
    __syncthreads();
    if (tid == 0) {
        double S = 0.0;
        int N = 0;
        for (int w = 0; w < kSumThreads / 32; ++w) {
            S += sh_s[w];
            N += sh_n[w];
        }
        *a.loss_sum = S;
        *a.num_tokens = N;
    }
}

}  // namespace

cudaError_t launch_loss(const LossArgs &a, int num_sms, cudaStream_t stream)
{
    if (a.T > 0) {
        long long blocks = a.T;
        const long long cap = static_cast<long long>(num_sms > 0 ? num_sms : 1) * 8;
        if (blocks > cap) blocks = cap;
        if (a.vec && a.V <= kSmemRowMax) {
            const int smem = a.V * 2;
            cudaError_t e = cudaFuncSetAttribute(loss_row_smem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            prof_begin(kProfLoss, stream);
            loss_row_smem_kernel<<<static_cast<unsigned>(blocks), kRowThreads, smem, stream>>>(a);
            prof_end(kProfLoss, stream);
        } else {
            prof_begin(kProfLoss, stream);
            loss_row_kernel<<<static_cast<unsigned>(blocks), kRowThreads, 0, stream>>>(a);
            prof_end(kProfLoss, stream);
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    loss_sum_kernel<<<1, kSumThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace spd
