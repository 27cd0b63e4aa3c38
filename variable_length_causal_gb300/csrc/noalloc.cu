// noalloc.cu -- vlc_attn_fwd_noalloc: the forward attention call for callers
// that cannot allocate device memory.
//
// Some callers are not allowed to obtain memory per call: code that runs
// inside another runtime's execution hook (a plugin's enqueue function, a
// host callback) where allocating is forbidden or would deadlock on the
// runtime's allocator lock, and long-running services whose device-memory
// budget is fixed at start-up.  They cannot provide the workspace that
// vlc_attn_fwd needs.  This entry point keeps that scratch (work list,
// segment order, RoPE table, device error word) in one file-scope device
// array instead.  The caller still passes inputs and outputs.
//
// Properties a caller must know:
//  - The array holds kNoAllocScratchBytes (8 MiB) on every GPU that loads this
//    library, for the lifetime of the process.  A problem is accepted when the
//    forward's workspace without its optional region (the rotated copy of k)
//    fits; larger ones are rejected with VLC_ERR_WORKSPACE before anything is
//    enqueued.  When the whole workspace fits, k is rotated once into it exactly
//    as vlc_attn_fwd does; otherwise the attention kernel's RoPE warps rotate
//    every staged K tile.
//  - The first call on a device looks up the array's device address with
//    cudaGetSymbolAddress (with that device current) and caches it; make that
//    first call before any stream capture begins.
//  - Every call, on every stream, shares the same array.  Calls whose GPU work
//    overlaps (different streams without ordering between them) race on it and
//    give wrong results; serialise them.  Each call clears the error word
//    itself; the rest of the array is fully rewritten before it is read.
//  - Device-side errors (invalid cu_seqlens, an expired wait) are reported by
//    copying the call's VLC_DEVERR_* bits over the caller's err_out word (if
//    given), in stream order.
//  - No cudaMalloc, cudaFree or other allocating routine is called.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/vlc.h"
#include "internal.h"

namespace vlc {

constexpr size_t kNoAllocScratchBytes = VLC_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (looked up once).
int scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return VLC_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return VLC_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return VLC_OK;
}
}  // namespace

}  // namespace vlc

extern "C" int vlc_attn_fwd_noalloc(const void* q, const void* k, const void* v, const int32_t* cu,
                                    int32_t nseg, int32_t total, int32_t H, int32_t d,
                                    int32_t max_seqlen, float softmax_scale, float rope_theta,
                                    void* o, float* lse, int32_t* err_out, void* stream) {
    if (vlc_workspace_bytes(nseg, total, H, d, max_seqlen, 0) == 0) {
        // invalid or unsupported arguments: the regular entry point's own checks give
        // the status (they reject these before the workspace is looked at, so nothing
        // is enqueued)
        return vlc_attn_fwd(q, k, v, cu, nseg, total, H, d, max_seqlen, softmax_scale, rope_theta, o, lse,
                            nullptr, 0, stream);
    }
    // The scratch must hold the forward's work list, segment order, RoPE table and
    // error word.  If it also holds the optional rotated copy of k (the whole layout
    // fits), the forward uses it; otherwise it rotates the K tiles inside the kernel.
    const size_t need = vlc::ws_layout(nseg, total, H, H, d, max_seqlen, 0).total_min;
    if (need > vlc::kNoAllocScratchBytes) return VLC_ERR_WORKSPACE;
    void* scratch = nullptr;
    const int st = vlc::scratch_for_current_device(&scratch);
    if (st != VLC_OK) return st;
    // The regular entry point does the rest: it clears the error word in the
    // scratch, builds the work list and RoPE table there, and launches.
    const int fst = vlc_attn_fwd(q, k, v, cu, nseg, total, H, d, max_seqlen, softmax_scale,
                                 rope_theta, o, lse, scratch, vlc::kNoAllocScratchBytes, stream);
    if (fst != VLC_OK) return fst;
    // The error word is the first int32 of the scratch; copy it out on the stream.
    if (err_out != nullptr &&
        cudaMemcpyAsync(err_out, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return VLC_ERR_CUDA;
    return VLC_OK;
}
