// ce.cu -- shifted next-token cross-entropy statistics over a packed buffer.
//
// What it computes ("Sequence packing and variable-length attention",
// charlestar, sections "After isolation one cross-boundary prediction pair
// remains" and "Packing should not decide how much a long sample weighs"):
// with pre-shifted labels (label_i = token_{i+1} inside a segment, -100 on each
// segment's last token and on ignored segments), logit row i contributes
// CE_i = ln sum_c exp(z_ic) - z_i,label_i when label_i != -100.  The call returns
// the pack's loss sum and target count, and per segment S_r = sum CE_i and
// n_r = #targets, so the caller picks the denominator (token mean or sample mean).
//
// The work is one pass over the [total, vocab] bf16 logits (HBM-bound):
//   ce_rows_kernel      one CTA per row at a time (grid-stride): 16-byte loads,
//                       an online log-sum-exp in base 2 (one rescale per 8
//                       logits), a CTA reduction, CE_i into the workspace.  Rows
//                       whose label is -100 are not read at all.
//   ce_segments_kernel  one warp per segment: S_r and n_r in a fixed order.
//   ce_total_kernel     one CTA: the pack totals (fp64 accumulation, fixed order).
// Every reduction has a fixed order, so results are bitwise reproducible.
#include <cuda_bf16.h>
#include <algorithm>
#include <cmath>
#include <cstdint>

#include "../../include/vlc.h"
#include "internal.h"

namespace vlc {
namespace ce {

constexpr int kRowThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994530942f;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Merge two partial (max, sum) pairs of a base-2 log-sum-exp.
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
    const float mn = fmaxf(m, m2);
    if (mn == -INFINITY) return;
    s = s * ex2(m - mn) + s2 * ex2(m2 - mn);
    m = mn;
}

template <bool VEC>
__global__ void __launch_bounds__(kRowThreads)
ce_rows_kernel(const __nv_bfloat16* __restrict__ logits, int32_t vocab, int32_t total,
               const int64_t* __restrict__ labels, float* __restrict__ row_loss,
               uint8_t* __restrict__ row_valid, int32_t* __restrict__ err) {
    __shared__ float sm[kRowThreads / 32], ss[kRowThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int64_t i = blockIdx.x; i < total; i += gridDim.x) {
        const int64_t y = __ldg(labels + i);
        const bool in_range = y >= 0 && y < vocab;
        if (!in_range) {   // ignored (or invalid) target: the row is not read
            if (tid == 0) {
                row_loss[i] = 0.f;
                row_valid[i] = 0;
                if (y != -100) atomicOr(err, VLC_DEVERR_LABEL);
            }
            continue;
        }
        const __nv_bfloat16* row = logits + i * static_cast<int64_t>(vocab);
        float m = -INFINITY, s = 0.f;
        if constexpr (VEC) {
            const uint4* r4 = reinterpret_cast<const uint4*>(row);
            const int nvec = vocab >> 3;
#pragma unroll 4
            for (int c = tid; c < nvec; c += kRowThreads) {
                const uint4 u = __ldg(r4 + c);
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
                float x[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    x[2 * e] = __uint_as_float(w[e] << 16) * kLog2e;
                    x[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u) * kLog2e;
                }
                float cm = fmaxf(fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])),
                                 fmaxf(fmaxf(x[4], x[5]), fmaxf(x[6], x[7])));
                if (cm > m) {
                    s = (m == -INFINITY) ? 0.f : s * ex2(m - cm);
                    m = cm;
                }
                if (m != -INFINITY) {   // all -inf so far: nothing to add
                    float a = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) a += ex2(x[e] - m);
                    s += a;
                }
            }
        } else {
            for (int c = tid; c < vocab; c += kRowThreads) {
                const float x = __bfloat162float(row[c]) * kLog2e;
                if (x > m) {
                    s = (m == -INFINITY) ? 0.f : s * ex2(m - x);
                    m = x;
                }
                if (m != -INFINITY) s += ex2(x - m);
            }
        }
        // warp, then CTA reduction of (max, sum)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
            const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
            lse_merge(m, s, m2, s2);
        }
        if (lane == 0) { sm[warp] = m; ss[warp] = s; }
        __syncthreads();
        if (tid == 0) {
            float mm = sm[0], sv = ss[0];
            for (int wi = 1; wi < kRowThreads / 32; ++wi) lse_merge(mm, sv, sm[wi], ss[wi]);
            const float lse = (mm + __log2f(sv)) * kLn2;
            row_loss[i] = lse - __bfloat162float(row[y]);
            row_valid[i] = 1;
        }
        __syncthreads();
    }
}

// One warp per segment: S_r and n_r in a fixed order (lane-strided, then a
// shuffle tree).  Segment bounds are clamped to [0, total] so a bad cu cannot
// send the warp out of the arrays; cu validity bits go to the error word.
__global__ void __launch_bounds__(256)
ce_segments_kernel(const float* __restrict__ row_loss, const uint8_t* __restrict__ row_valid,
                   const int32_t* __restrict__ cu, int32_t nseg, int32_t total,
                   float* __restrict__ seg_loss, int32_t* __restrict__ seg_count,
                   int32_t* __restrict__ err) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t r = gw; r < nseg; r += nw) {
        int64_t a = 0, b = total;
        if (cu != nullptr) {
            const int32_t c0 = __ldg(cu + r), c1 = __ldg(cu + r + 1);
            if (lane == 0) {
                int e = 0;
                if (r == 0 && c0 != 0) e |= VLC_DEVERR_CU_FIRST;
                if (c1 <= c0) e |= VLC_DEVERR_CU_ORDER;
                if (r == nseg - 1 && c1 != total) e |= VLC_DEVERR_CU_TOTAL;
                if (e) atomicOr(err, e);
            }
            a = min(max(static_cast<int64_t>(c0), int64_t(0)), static_cast<int64_t>(total));
            b = min(max(static_cast<int64_t>(c1), a), static_cast<int64_t>(total));
        }
        float sr = 0.f;
        int nr = 0;
        for (int64_t i = a + lane; i < b; i += 32) {
            sr += row_loss[i];
            nr += row_valid[i];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            sr += __shfl_xor_sync(0xffffffffu, sr, o);
            nr += __shfl_xor_sync(0xffffffffu, nr, o);
        }
        if (lane == 0) {
            seg_loss[r] = sr;
            seg_count[r] = nr;
        }
    }
}

__global__ void __launch_bounds__(1024)
ce_total_kernel(const float* __restrict__ seg_loss, const int32_t* __restrict__ seg_count,
                int32_t nseg, float* __restrict__ loss_sum, int64_t* __restrict__ count) {
    __shared__ double sd[32];
    __shared__ long long sc[32];
    double a = 0.0;
    long long n = 0;
    for (int r = threadIdx.x; r < nseg; r += blockDim.x) {
        a += static_cast<double>(seg_loss[r]);
        n += seg_count[r];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        n += __shfl_xor_sync(0xffffffffu, n, o);
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) { sd[warp] = a; sc[warp] = n; }
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        long long c = 0;
        for (int wi = 0; wi < static_cast<int>(blockDim.x >> 5); ++wi) { t += sd[wi]; c += sc[wi]; }
        *loss_sum = static_cast<float>(t);
        *count = c;
    }
}

}  // namespace ce

CeLayout ce_layout(int32_t total, int32_t nseg) {
    CeLayout L{};
    auto align256 = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    size_t off = 0;
    L.header = off;
    off = align256(off + 256);
    L.row_loss = off;
    off = align256(off + sizeof(float) * static_cast<size_t>(total));
    L.row_valid = off;
    off = align256(off + static_cast<size_t>(total));
    L.seg_loss = off;
    off = align256(off + sizeof(float) * static_cast<size_t>(nseg));
    L.seg_count = off;
    off = align256(off + sizeof(int32_t) * static_cast<size_t>(nseg));
    L.total = off;
    return L;
}

cudaError_t launch_shifted_ce(const void* logits, int32_t vocab, int32_t total, const int64_t* labels,
                              const int32_t* cu, int32_t nseg, float* loss_sum, int64_t* count,
                              float* seg_loss, int32_t* seg_count, uint8_t* ws, cudaStream_t s) {
    const CeLayout L = ce_layout(total, nseg);
    int32_t* err = reinterpret_cast<int32_t*>(ws + L.header);
    float* row_loss = reinterpret_cast<float*>(ws + L.row_loss);
    uint8_t* row_valid = ws + L.row_valid;
    float* sl = seg_loss != nullptr ? seg_loss : reinterpret_cast<float*>(ws + L.seg_loss);
    int32_t* sc = seg_count != nullptr ? seg_count : reinterpret_cast<int32_t*>(ws + L.seg_count);
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaError_t e = cudaMemsetAsync(ws + L.header, 0, 256, s);
    if (e != cudaSuccess) return e;
    const int64_t rows_grid = std::min<int64_t>(total, static_cast<int64_t>(sms) * 8);
    const bool vec = (vocab % 8 == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);
    const auto* lg = static_cast<const __nv_bfloat16*>(logits);
    if (vec)
        ce::ce_rows_kernel<true><<<static_cast<int>(rows_grid), ce::kRowThreads, 0, s>>>(
            lg, vocab, total, labels, row_loss, row_valid, err);
    else
        ce::ce_rows_kernel<false><<<static_cast<int>(rows_grid), ce::kRowThreads, 0, s>>>(
            lg, vocab, total, labels, row_loss, row_valid, err);
    const int segs_grid = static_cast<int>(std::min<int64_t>((static_cast<int64_t>(nseg) + 7) / 8,
                                                             static_cast<int64_t>(sms) * 8));
    ce::ce_segments_kernel<<<segs_grid, 256, 0, s>>>(row_loss, row_valid, cu, nseg, total, sl, sc, err);
    ce::ce_total_kernel<<<1, 1024, 0, s>>>(sl, sc, nseg, loss_sum, count);
    return cudaGetLastError();
}

}  // namespace vlc
