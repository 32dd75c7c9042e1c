// spd_varlen_attn_fwd_noalloc: the forward attention for callers that cannot
// allocate device memory (no cudaMalloc, no caching allocator, no workspace
// to pass). Its scratch -- the status word and the tile work list that
// spd_varlen_attn_fwd keeps in the caller's workspace -- lives instead in one
// fixed array of this library's device image.
#include <mutex>

#include "../../include/spd.h"
#include "internal.h"

namespace spd {
namespace {

// Fixed scratch, allocated by the CUDA runtime when the library's device image
// is loaded on a GPU and held until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SPD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
std::mutex g_setup_mu;
void *g_scratch_ptr[kMaxDev];  // device address of g_noalloc_scratch, per device

// Device address of the scratch array on the current device. The first call
// on a device looks it up (cudaGetSymbolAddress with that device current);
// later calls reuse it. Host code must never hand the symbol itself to a
// kernel: on the host it names a stand-in, not the device array.
int scratch_on_current_device(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return SPD_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SPD_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return SPD_OK;
}

}  // namespace
}  // namespace spd

extern "C" int spd_varlen_attn_fwd_noalloc(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                           const int32_t *cu_seqlens, int32_t num_segs, int64_t total_tokens,
                                           int32_t max_seqlen, int Hq, int Hkv, int head_dim,
                                           float softmax_scale, uint16_t *out, float *lse,
                                           int32_t *device_status, spd_stream_t stream)
{
    const size_t need = spd_attn_workspace_size(total_tokens, num_segs, Hq, Hkv, head_dim, 0);
    if (need == 0) {
        // same host checks (and codes) as the workspace entry point
        return spd_varlen_attn_fwd(q, k, v, cu_seqlens, num_segs, total_tokens, max_seqlen, Hq, Hkv, head_dim,
                                   softmax_scale, out, lse, nullptr, 0, stream);
    }
    // Pointer checks of the workspace entry point, made here first so that a
    // bad pointer reports SPD_ERR_INVALID_ARG whatever the problem size.
    auto misaligned = [](const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; };
    if (total_tokens > 0 &&
        (!q || !k || !v || !out || !lse || !cu_seqlens || misaligned(q, 16) || misaligned(k, 16) ||
         misaligned(v, 16) || misaligned(out, 16) || misaligned(lse, 4) || misaligned(cu_seqlens, 4)))
        return SPD_ERR_INVALID_ARG;
    if (need > SPD_NOALLOC_SCRATCH_BYTES) return SPD_ERR_TOO_LARGE;
    void *scratch = nullptr;
    int rc = spd::scratch_on_current_device(&scratch);
    if (rc != SPD_OK) return rc;
    // The scheduler kernel rewrites the status word, the tile count and the
    // whole work list on every call, so nothing left by an earlier call is read.
    rc = spd_varlen_attn_fwd(q, k, v, cu_seqlens, num_segs, total_tokens, max_seqlen, Hq, Hkv, head_dim,
                             softmax_scale, out, lse, scratch, SPD_NOALLOC_SCRATCH_BYTES, stream);
    if (rc != SPD_OK) return rc;
    if (device_status) {
        cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        if (cudaMemcpyAsync(device_status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return SPD_ERR_CUDA;
    }
    return SPD_OK;
}
