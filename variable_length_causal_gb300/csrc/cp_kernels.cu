// cp_kernels.cu -- the device steps of the context-parallel split: RoPE by explicit
// positions (a rank's rows keep the positions they had in the whole segment; the
// transposed rotation takes gradients back), the merge of partial attention results
// over disjoint key blocks, and the sum of partial gradients.  Entry points
// vlc_rope_pos, vlc_rope_pos_workspace_bytes, vlc_lse_merge and vlc_sum_parts
// (include/vlc.h); the host partition is in cp.cpp.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "../../include/vlc.h"
#include "attn_common.cuh"
#include "internal.h"

namespace vlc {
namespace cp {

// out[row] = R(pos[row]) x[row] for every head: D/16 threads per row, each owning a
// (lo, hi) pair of 16-byte chunks of every head (the chunk pairing of load_angles and
// rotate_chunks, shared with the backward's prep pass and vlc_rope_qk).  A position
// outside [0, max_pos] raises VLC_DEVERR_POS and zeroes the row.
template <int D>
__global__ void __launch_bounds__(256)
rope_pos_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ pos, uint4* __restrict__ out,
                int64_t rows, int32_t H, int32_t max_pos, const float2* __restrict__ table, int rope,
                bool transpose, int32_t* err) {
    constexpr int TPR = D / 16;
    constexpr int HALF = D / 16;
    const bool il = rope == kRopeInterleaved;
    const int64_t n = rows * TPR;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t row = i / TPR;
        const int c = static_cast<int>(i % TPR);
        const int32_t p = __ldg(pos + row);
        const bool ok = p >= 0 && p <= max_pos;
        if (!ok && c == 0) atomicOr(err, VLC_DEVERR_POS);
        float cs[8], sn[8];
        if (ok) load_angles<D>(table, p, il, c, cs, sn);
        if (transpose) {   // R(p)^T = R(-p): the same cosines, negated sines
#pragma unroll
            for (int e = 0; e < 8; ++e) sn[e] = -sn[e];
        }
        for (int h = 0; h < H; ++h) {
            const int64_t lo = (row * H + h) * (2 * HALF) + c;
            rotate_chunks(x, out, lo, lo + HALF, cs, sn, ok, il);
        }
    }
}

struct MergeParts {
    const uint4* o[VLC_LSE_MERGE_MAX];
    const float* lse[VLC_LSE_MERGE_MAX];
    int n;
};

// One thread per (row, head, 8-column chunk): the parts' LSE values of the row give
// the weights e^{LSE_k - max}; O is the weighted sum of the parts' chunks over the
// weights' total, accumulated in fp32 and rounded once to bf16.
template <int D>
__global__ void __launch_bounds__(256)
lse_merge_kernel(const MergeParts parts, int64_t rows, int32_t H, uint4* __restrict__ o, float* __restrict__ lse) {
    constexpr int CPT = D / 8;   // 16-byte chunks per head row
    const int64_t n = rows * H * CPT;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int c = static_cast<int>(i % CPT);
        const int64_t rh = i / CPT;
        const int h = static_cast<int>(rh % H);
        const int64_t row = rh / H;
        const int64_t li = static_cast<int64_t>(h) * rows + row;
        float l[VLC_LSE_MERGE_MAX];
        float mx = -INFINITY;
#pragma unroll
        for (int k = 0; k < VLC_LSE_MERGE_MAX; ++k) {
            l[k] = k < parts.n ? __ldg(parts.lse[k] + li) : -INFINITY;
            mx = fmaxf(mx, l[k]);
        }
        if (mx == -INFINITY) {   // no part saw a key
            o[i] = make_uint4(0u, 0u, 0u, 0u);
            if (c == 0) lse[li] = -INFINITY;
            continue;
        }
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        float tot = 0.f;
#pragma unroll
        for (int k = 0; k < VLC_LSE_MERGE_MAX; ++k) {
            if (k >= parts.n || l[k] == -INFINITY) continue;
            const float w = expf(l[k] - mx);
            tot += w;
            const uint4 v = __ldg(parts.o[k] + i);
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[2 * e] = fmaf(w, bf16_lo(wv[e]), acc[2 * e]);
                acc[2 * e + 1] = fmaf(w, bf16_hi(wv[e]), acc[2 * e + 1]);
            }
        }
        const float inv = 1.f / tot;
        o[i] = make_uint4(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv),
                          pack_bf16x2(acc[4] * inv, acc[5] * inv), pack_bf16x2(acc[6] * inv, acc[7] * inv));
        if (c == 0) lse[li] = mx + logf(tot);
    }
}

// out = sum of n bf16 arrays, accumulated in fp32 and rounded once (8 elements per thread).
__global__ void __launch_bounds__(256)
sum_parts_kernel(const MergeParts parts, int64_t n16, uint4* __restrict__ out) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
        for (int k = 0; k < parts.n; ++k) {
            const uint4 v = __ldg(parts.o[k] + i);
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[2 * e] += bf16_lo(wv[e]);
                acc[2 * e + 1] += bf16_hi(wv[e]);
            }
        }
        out[i] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                            pack_bf16x2(acc[6], acc[7]));
    }
}

int grid_for(int64_t threads) {
    static int sms = 0;
    if (sms == 0) {
        int dev = 0, n = 0;
        if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
            sms = n;
        if (sms <= 0) sms = 1;
    }
    int64_t blocks = (threads + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    if (blocks > cap) blocks = cap;
    return static_cast<int>(blocks < 1 ? 1 : blocks);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t table_rows_for(int32_t max_pos) { return (static_cast<int64_t>(max_pos) + kTablePad) / kTablePad * kTablePad; }

}  // namespace cp
}  // namespace vlc

extern "C" size_t vlc_rope_pos_workspace_bytes(int32_t max_pos, int32_t d) {
    if (max_pos < 0 || max_pos >= VLC_MAX_SEQLEN || (d != 64 && d != 128)) return 0;
    return 256 + static_cast<size_t>(vlc::cp::table_rows_for(max_pos)) * (d / 2) * sizeof(float2);
}

extern "C" int vlc_rope_pos(const void* x, const int32_t* pos, int32_t rows, int32_t H, int32_t d, int32_t max_pos,
                            float rope_theta, uint32_t flags, void* out, void* ws, size_t ws_bytes, void* stream) {
    using namespace vlc;
    if (x == nullptr || pos == nullptr || out == nullptr || rows < 1 || H < 1) return VLC_ERR_ARG;
    if (flags & ~static_cast<uint32_t>(VLC_ROPE_INTERLEAVED | VLC_ROPE_TRANSPOSE)) return VLC_ERR_ARG;
    if (!(rope_theta > 0.f) || !std::isfinite(rope_theta)) return VLC_ERR_ARG;
    if (d != 64 && d != 128) return VLC_ERR_UNSUPPORTED;
    if (max_pos < 0 || max_pos >= VLC_MAX_SEQLEN) return VLC_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(rows) * H * d > (int64_t(1) << 40)) return VLC_ERR_UNSUPPORTED;
    if (!cp::aligned(x, 16) || !cp::aligned(out, 16)) return VLC_ERR_ARG;
    if (ws == nullptr || !cp::aligned(ws, 256) || ws_bytes < vlc_rope_pos_workspace_bytes(max_pos, d))
        return VLC_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* w = static_cast<uint8_t*>(ws);
    int32_t* err = reinterpret_cast<int32_t*>(w);
    float2* table = reinterpret_cast<float2*>(w + 256);
    const int32_t trows = static_cast<int32_t>(cp::table_rows_for(max_pos));
    if (cudaMemsetAsync(err, 0, sizeof(int32_t), s) != cudaSuccess) return VLC_ERR_CUDA;
    if (launch_rope_table(table, trows, d, static_cast<double>(rope_theta), err, s) != cudaSuccess)
        return VLC_ERR_CUDA;
    const int mode = (flags & VLC_ROPE_INTERLEAVED) ? kRopeInterleaved : kRopeHalf;
    const int64_t threads = static_cast<int64_t>(rows) * (d / 16);
    auto kernel = d == 128 ? cp::rope_pos_kernel<128> : cp::rope_pos_kernel<64>;
    kernel<<<cp::grid_for(threads), 256, 0, s>>>(static_cast<const uint4*>(x), pos, static_cast<uint4*>(out), rows, H,
                                                 max_pos, table, mode, (flags & VLC_ROPE_TRANSPOSE) != 0, err);
    return cudaGetLastError() == cudaSuccess ? VLC_OK : VLC_ERR_CUDA;
}

extern "C" int vlc_sum_parts(const void* const* parts, int32_t nparts, int64_t elems, void* out, void* stream) {
    using namespace vlc;
    if (parts == nullptr || out == nullptr || nparts < 1 || nparts > VLC_LSE_MERGE_MAX || elems < 1 || elems % 8 != 0)
        return VLC_ERR_ARG;
    if (!cp::aligned(out, 16)) return VLC_ERR_ARG;
    cp::MergeParts mp{};
    mp.n = nparts;
    for (int k = 0; k < nparts; ++k) {
        if (parts[k] == nullptr || !cp::aligned(parts[k], 16)) return VLC_ERR_ARG;
        mp.o[k] = static_cast<const uint4*>(parts[k]);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t n16 = elems / 8;
    cp::sum_parts_kernel<<<cp::grid_for(n16), 256, 0, s>>>(mp, n16, static_cast<uint4*>(out));
    return cudaGetLastError() == cudaSuccess ? VLC_OK : VLC_ERR_CUDA;
}

extern "C" int vlc_lse_merge(const void* const* o_parts, const float* const* lse_parts, int32_t nparts, int32_t rows,
                             int32_t H, int32_t d, void* o, float* lse, void* stream) {
    using namespace vlc;
    if (o_parts == nullptr || lse_parts == nullptr || o == nullptr || lse == nullptr || rows < 1 || H < 1 ||
        nparts < 1 || nparts > VLC_LSE_MERGE_MAX)
        return VLC_ERR_ARG;
    if (d != 64 && d != 128) return VLC_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(rows) * H * d > (int64_t(1) << 40)) return VLC_ERR_UNSUPPORTED;
    if (!cp::aligned(o, 16) || !cp::aligned(lse, 4)) return VLC_ERR_ARG;
    cp::MergeParts parts{};
    parts.n = nparts;
    for (int k = 0; k < nparts; ++k) {
        if (o_parts[k] == nullptr || lse_parts[k] == nullptr || !cp::aligned(o_parts[k], 16) ||
            !cp::aligned(lse_parts[k], 4))
            return VLC_ERR_ARG;
        parts.o[k] = static_cast<const uint4*>(o_parts[k]);
        parts.lse[k] = lse_parts[k];
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t threads = static_cast<int64_t>(rows) * H * (d / 8);
    auto kernel = d == 128 ? cp::lse_merge_kernel<128> : cp::lse_merge_kernel<64>;
    kernel<<<cp::grid_for(threads), 256, 0, s>>>(parts, rows, H, static_cast<uint4*>(o), lse);
    return cudaGetLastError() == cudaSuccess ? VLC_OK : VLC_ERR_CUDA;
}
