// prep.cu -- the integer/metadata kernels of the path:
//   * work-list builder: validates cu_seqlens and emits only in-segment,
//     at-or-below-diagonal tiles ("Sequence packing and variable-length
//     attention", charlestar: validity contract and allow(i,j); "Packing document
//     boundary", operatorworld, pitfall 1: the varlen kernel skips cross-document
//     blocks);
//   * positions and labels: p_i = i - cu_r and pre-shifted labels with -100 at
//     segment ends ("Length grouping, de-padding and packing", M020 section 06);
//   * RoPE cos/sin table for fixed frequencies theta^(-2j/d).
#include <algorithm>
#include <cmath>
#include <cstdint>

#include "../../include/vlc.h"
#include "internal.h"

namespace vlc {

// ============================================================== work list
//
// One CTA of 1024 threads.  Segments are ordered by descending tile count with
// a stable counting sort (histogram over tile counts, exclusive scan from the
// largest count down, then in-order placement warp by warp so that equal
// counts keep their segment order).

constexpr int kWlThreads = 1024;

__device__ __forceinline__ int block_excl_scan(int v, int* warp_sums, int* total_out) {
    // Exclusive scan of one int per thread across the CTA (1024 threads).
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
        int s = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        warp_sums[lane] = s - w;   // exclusive prefix of warp totals
        if (lane == 31) warp_sums[32] = s;
    }
    __syncthreads();
    int r = x - v + warp_sums[warp];
    *total_out = warp_sums[32];
    __syncthreads();
    return r;
}

__device__ __forceinline__ void worklist_body(const WlSpec& spec) {
    const int32_t* __restrict__ cu = spec.cu;
    const int32_t nseg = spec.nseg, total = spec.total, max_seqlen = spec.max_seqlen;
    const int32_t BM = spec.BM, BN = spec.BN;
    const int kind = spec.kind;
    int4* __restrict__ items = spec.items;
    const int64_t cap = spec.cap;
    int32_t* __restrict__ order = spec.order;
    int32_t* __restrict__ seg_base = spec.seg_base;
    int32_t* __restrict__ count = spec.count;
    int32_t* __restrict__ err = spec.err;
    const int32_t* __restrict__ cu_padded = spec.cu_padded;
    const int32_t* __restrict__ cu_kv = spec.cu_kv;
    const int32_t total_kv = spec.total_kv, max_seqlen_kv = spec.max_seqlen_kv;
    extern __shared__ int wl_smem[];
    int* hist = wl_smem;                    // [nbins] counts, then running positions
    __shared__ int warp_sums[33];
    __shared__ int s_err, s_maxlen, s_maxlen_kv;
    const int tid = threadIdx.x;
    const int tile = (kind == VLC_WORKLIST_FWD) ? BM : BN;
    // a segment's item count: its q tiles (forward) or key tiles (backward); keys and
    // values have segments of their own when cu_kv is given (bottom-right aligned)
    const int32_t* const ck = cu_kv != nullptr ? cu_kv : cu;
    const int32_t* const cn = (kind == VLC_WORKLIST_FWD) ? cu : ck;
    const int nbins = ((kind == VLC_WORKLIST_FWD || cu_kv == nullptr ? max_seqlen : max_seqlen_kv) + tile - 1) /
                      tile + 1;

    if (tid == 0) {
        s_err = 0;
        s_maxlen = 0;
        s_maxlen_kv = 0;
    }
    for (int b = tid; b < nbins; b += kWlThreads) hist[b] = 0;
    __syncthreads();

    // ---- 1. validate cu_seqlens
    int local_err = 0, local_max = 0, local_max_kv = 0;
    for (int r = tid; r < nseg; r += kWlThreads) {
        int a = cu[r], b = cu[r + 1];
        if (r == 0 && a != 0) local_err |= VLC_DEVERR_CU_FIRST;
        if (b <= a) local_err |= VLC_DEVERR_CU_ORDER;
        local_max = max(local_max, b - a);
        if (cu_kv != nullptr) {   // key segments start at 0 and are at least as long as the query ones
            const int ka = cu_kv[r], kb = cu_kv[r + 1];
            if (r == 0 && ka != 0) local_err |= VLC_DEVERR_CU_FIRST;
            if (static_cast<int64_t>(kb) - ka < static_cast<int64_t>(b) - a) local_err |= VLC_DEVERR_QKV;
            local_max_kv = max(local_max_kv, kb - ka);
        }
        if (cu_padded != nullptr) {   // slot r holds segment r: it starts at 0 and is long enough
            const int pa = cu_padded[r], pb = cu_padded[r + 1];
            if ((r == 0 && pa != 0) || static_cast<int64_t>(pb) - pa < static_cast<int64_t>(b) - a)
                local_err |= VLC_DEVERR_CU_PADDED;
        }
    }
    if (tid == 0) {
        if (cu_padded == nullptr ? cu[nseg] != total : cu_padded[nseg] != total)
            local_err |= (cu_padded == nullptr ? VLC_DEVERR_CU_TOTAL : VLC_DEVERR_CU_PADDED);
        if (cu_kv != nullptr && cu_kv[nseg] != total_kv) local_err |= VLC_DEVERR_CU_TOTAL;
    }
    if (local_err) atomicOr(&s_err, local_err);
    atomicMax(&s_maxlen, local_max);
    atomicMax(&s_maxlen_kv, local_max_kv);
    __syncthreads();
    if (tid == 0 && s_maxlen != max_seqlen) s_err |= VLC_DEVERR_MAXLEN;
    if (tid == 0 && cu_kv != nullptr && s_maxlen_kv != max_seqlen_kv) s_err |= VLC_DEVERR_MAXLEN;
    __syncthreads();
    if (s_err != 0) {
        if (tid == 0) {
            atomicOr(err, s_err);
            *count = 0;
        }
        return;
    }

    // ---- 2. histogram of tile counts
    for (int r = tid; r < nseg; r += kWlThreads) {
        int n = (cn[r + 1] - cn[r] + tile - 1) / tile;
        atomicAdd(&hist[n], 1);
    }
    __syncthreads();

    // ---- 3. start position of each bin in descending-count order:
    //         start[b] = number of segments with count > b.
    //         Thread t owns bins [t*per, (t+1)*per) counted from the top.
    {
        const int per = (nbins + kWlThreads - 1) / kWlThreads;
        int vals[16];
        int sum = 0;
        for (int i = 0; i < per; ++i) {
            int rb = tid * per + i;          // rank from the top
            int b = nbins - 1 - rb;
            int c = (rb < nbins) ? hist[b] : 0;
            if (i < 16) vals[i] = c;
            sum += c;
        }
        int tot;
        int base = block_excl_scan(sum, warp_sums, &tot);
        for (int i = 0; i < per; ++i) {
            int rb = tid * per + i;
            if (rb < nbins) {
                int b = nbins - 1 - rb;
                hist[b] = base;             // becomes the running position of bin b
                base += vals[i];
            }
        }
    }
    __syncthreads();

    // ---- 4. stable placement, one warp at a time inside each chunk of 1024
    const int lane = tid & 31, warp = tid >> 5;
    for (int c0 = 0; c0 < nseg; c0 += kWlThreads) {
        const int r = c0 + tid;
        const bool valid = r < nseg;
        const int n = valid ? (cn[r + 1] - cn[r] + tile - 1) / tile : -1;
        for (int w = 0; w < kWlThreads / 32; ++w) {
            if (warp == w) {
                unsigned peers = __match_any_sync(0xffffffffu, n);
                int leader = __ffs(peers) - 1;
                int rank = __popc(peers & ((1u << lane) - 1u));
                int base = 0;
                if (valid && lane == leader) {
                    base = hist[n];
                    hist[n] = base + __popc(peers);
                }
                base = __shfl_sync(peers, base, leader);
                if (valid) order[base + rank] = r;
            }
            __syncthreads();
        }
    }
    __syncthreads();

    // ---- 5. item offset of each sorted segment (exclusive scan of tile counts)
    int carry = 0;
    for (int c0 = 0; c0 < nseg; c0 += kWlThreads) {
        const int k = c0 + tid;
        int n = 0;
        if (k < nseg) {
            int r = order[k];
            n = (cn[r + 1] - cn[r] + tile - 1) / tile;
        }
        int tot;
        int ex = block_excl_scan(n, warp_sums, &tot);
        if (k < nseg) seg_base[k] = carry + ex;
        carry += tot;
    }
    if (tid == 0) seg_base[nseg] = carry;
    __syncthreads();

    // ---- 6. items (host guarantees cap >= nseg + total / tile >= carry)
    for (int k = tid; k < nseg; k += kWlThreads) {
        const int r = order[k];
        const int L = cu[r + 1] - cu[r];
        const int Lk = ck[r + 1] - ck[r];
        // queries are the last L of the Lk positions; with every key visible the diagonal
        // lies past the last key
        const int off = spec.all_visible ? Lk : Lk - L;
        const int base = seg_base[k];
        const int n = seg_base[k + 1] - base;
        for (int j = 0; j < n; ++j) {
            int4 it;
            it.x = r;
            if (kind == VLC_WORKLIST_FWD) {
                const int qt = n - 1 - j;
                const int last = min(Lk, min(L, (qt + 1) * BM) + off);   // keys the tile sees
                it.y = qt;
                it.z = 0;
                it.w = (last + BN - 1) / BN;
            } else {
                const int kt = j;
                it.y = kt;
                it.z = max(0, kt * BN - off) / BM;
                it.w = (L + BM - 1) / BM;
            }
            if (base + j < cap) items[base + j] = it;
        }
    }
    if (tid == 0) *count = carry;
}

// ============================================================== padding rows
//
// Padded layouts: the rows [cu_padded[r] + L_r, cu_padded[r+1]) of slot r are
// not tokens.  One block per slot (grid-stride over slots) zeroes them in each
// given bf16 tensor with 16-byte stores (a row is H * d * 2 >= 128 bytes, so a
// slot's padding is one contiguous, aligned byte range) and writes -inf into
// those columns of lse.  Ranges are clamped to [0, total) rows.

__global__ void __launch_bounds__(256)
pad_fill_kernel(const int32_t* __restrict__ cu, const int32_t* __restrict__ cu_padded, int32_t nseg,
                int32_t total, uint4* __restrict__ a, int64_t a_row16, uint4* __restrict__ b,
                int64_t b_row16, uint4* __restrict__ c, int64_t c_row16, float* __restrict__ lse,
                int32_t H, const int32_t* __restrict__ err) {
    if (*err != 0) return;
    for (int r = blockIdx.x; r < nseg; r += gridDim.x) {
        const int64_t p0 = max(static_cast<int64_t>(0),
                               min(static_cast<int64_t>(total),
                                   static_cast<int64_t>(cu_padded[r]) + (cu[r + 1] - cu[r])));
        const int64_t p1 = max(static_cast<int64_t>(0), min(static_cast<int64_t>(total),
                                                            static_cast<int64_t>(cu_padded[r + 1])));
        if (p0 >= p1) continue;   // block-uniform
        uint4* const dst[3] = {a, b, c};
        const int64_t row16[3] = {a_row16, b_row16, c_row16};
#pragma unroll
        for (int t = 0; t < 3; ++t) {
            if (dst[t] == nullptr) continue;
            for (int64_t i = p0 * row16[t] + threadIdx.x; i < p1 * row16[t]; i += blockDim.x)
                dst[t][i] = make_uint4(0u, 0u, 0u, 0u);
        }
        if (lse != nullptr) {
            const int64_t n = p1 - p0;
            for (int64_t i = threadIdx.x; i < n * H; i += blockDim.x) {
                const int64_t h = i / n;
                lse[h * total + p0 + (i - h * n)] = -INFINITY;
            }
        }
    }
}

cudaError_t launch_pad_fill(const int32_t* cu, const int32_t* cu_padded, int32_t nseg, int32_t total,
                            void* a, int64_t a_row_bytes, void* b, int64_t b_row_bytes, void* c,
                            int64_t c_row_bytes, float* lse, int32_t H, const int32_t* err,
                            int num_sms, cudaStream_t s) {
    const int blocks = static_cast<int>(std::min<int64_t>(nseg, 4LL * num_sms));
    pad_fill_kernel<<<blocks, 256, 0, s>>>(cu, cu_padded, nseg, total, static_cast<uint4*>(a),
                                           a_row_bytes / 16, static_cast<uint4*>(b), b_row_bytes / 16,
                                           static_cast<uint4*>(c), c_row_bytes / 16, lse, H, err);
    return cudaGetLastError();
}

// ============================================================== positions + labels
//
// Each warp owns one contiguous run of tokens (a multiple of 128) and walks it
// 128 tokens at a time, 4 consecutive tokens per lane: one binary search over cu
// per warp for the run's first token, then every lane steps forward from the
// warp's current segment (segments are at least one token long, so a lane
// crosses at most a few boundaries).  Token loads and position / label stores are
// 16-byte vectors, and consecutive lanes touch consecutive bytes.

constexpr int kPlThreads = 256;
constexpr int kPlVec = 4;
constexpr int kPlWarpSpan = 32 * kPlVec;   // tokens per warp per step

__global__ void __launch_bounds__(kPlThreads)
positions_labels_kernel(const int32_t* __restrict__ cu, int32_t nseg,
                        const int64_t* __restrict__ tokens, int32_t total,
                        const uint8_t* __restrict__ seg_ignore, int32_t* __restrict__ pos,
                        int64_t* __restrict__ labels, int32_t* __restrict__ err) {
    const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int lane = threadIdx.x & 31;

    if (err != nullptr) {   // validity bits (cheap: nseg reads in total)
        int e = 0;
        for (int64_t r = gtid; r < nseg; r += nthreads) {
            if (r == 0 && cu[0] != 0) e |= VLC_DEVERR_CU_FIRST;
            if (cu[r + 1] <= cu[r]) e |= VLC_DEVERR_CU_ORDER;
        }
        if (gtid == 0 && cu[nseg] != total) e |= VLC_DEVERR_CU_TOTAL;
        if (e) atomicOr(err, e);
    }

    const int64_t nwarps = nthreads >> 5;
    const int64_t gwarp = gtid >> 5;
    const int64_t span = ((static_cast<int64_t>(total) + nwarps - 1) / nwarps + kPlWarpSpan - 1) /
                         kPlWarpSpan * kPlWarpSpan;
    const int64_t begin = gwarp * span;
    const int64_t end = min(static_cast<int64_t>(total), begin + span);
    if (begin >= end) return;   // warp-uniform
    const bool vec_ok = ((reinterpret_cast<uintptr_t>(pos) | reinterpret_cast<uintptr_t>(labels) |
                          reinterpret_cast<uintptr_t>(tokens)) & 15) == 0;

    // largest r in [0, nseg-1] with cu[r] <= begin (clamped; in bounds even for bad cu)
    int rw = 0;
    if (lane == 0) {
        int lo = 0, hi = nseg - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(cu + mid) <= begin) lo = mid; else hi = mid - 1;
        }
        rw = lo;
    }
    rw = __shfl_sync(0xffffffffu, rw, 0);

    for (int64_t base = begin; base < end; base += kPlWarpSpan) {   // warp-uniform trip count
        const int64_t i0 = base + kPlVec * lane;
        int r = rw;
        int32_t seg_start = __ldg(cu + r), seg_end = __ldg(cu + r + 1);
        int64_t tk[kPlVec + 1];
        const bool full = (i0 + kPlVec <= end);
        if (full && vec_ok) {
            const longlong2 a = __ldg(reinterpret_cast<const longlong2*>(tokens + i0));
            const longlong2 b = __ldg(reinterpret_cast<const longlong2*>(tokens + i0) + 1);
            tk[0] = a.x; tk[1] = a.y; tk[2] = b.x; tk[3] = b.y;
        } else {
#pragma unroll
            for (int t = 0; t < kPlVec; ++t) tk[t] = (i0 + t < total) ? __ldg(tokens + i0 + t) : 0;
        }
        tk[kPlVec] = (i0 + kPlVec < total) ? __ldg(tokens + i0 + kPlVec) : 0;
        int32_t p[kPlVec];
        int64_t lab[kPlVec];
#pragma unroll
        for (int t = 0; t < kPlVec; ++t) {
            const int64_t i = i0 + t;
            while (r < nseg - 1 && i >= seg_end) {
                ++r;
                seg_start = seg_end;
                seg_end = __ldg(cu + r + 1);
            }
            const bool ign = seg_ignore != nullptr && __ldg(seg_ignore + r) != 0;
            p[t] = static_cast<int32_t>(i - seg_start);
            lab[t] = (!ign && i + 1 < seg_end) ? tk[t + 1] : -100;
        }
        if (full && vec_ok) {
            *reinterpret_cast<int4*>(pos + i0) = make_int4(p[0], p[1], p[2], p[3]);
            reinterpret_cast<longlong2*>(labels + i0)[0] = make_longlong2(lab[0], lab[1]);
            reinterpret_cast<longlong2*>(labels + i0)[1] = make_longlong2(lab[2], lab[3]);
        } else {
            for (int t = 0; t < kPlVec; ++t)
                if (i0 + t < end) {
                    pos[i0 + t] = p[t];
                    labels[i0 + t] = lab[t];
                }
        }
        rw = __shfl_sync(0xffffffffu, r, 31);   // segment of the last token of this step
    }
}

cudaError_t launch_positions_labels(const int32_t* cu, int32_t nseg, const int64_t* tokens,
                                    int32_t total, const uint8_t* seg_ignore, int32_t* pos,
                                    int64_t* labels, int32_t* err, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // one warp per 128-token step at small sizes; at most 8 resident CTAs per SM, each warp
    // then walks a longer contiguous run
    const int64_t steps = (static_cast<int64_t>(total) + kPlWarpSpan - 1) / kPlWarpSpan;
    int64_t blocks = (steps + kPlThreads / 32 - 1) / (kPlThreads / 32);
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    positions_labels_kernel<<<static_cast<int>(blocks), kPlThreads, 0, s>>>(
        cu, nseg, tokens, total, seg_ignore, pos, labels, err);
    return cudaGetLastError();
}

// ============================================================== RoPE table
//
// table[p][j] = (cos(p w_j), sin(p w_j)), w_j = theta^(-2j/d).  The angle is
// formed in fp64 and reduced to [-pi, pi] in fp64 (one fused multiply-add
// against 2*pi in double), so the fp32 sincos that follows sees a small
// argument; the result is accurate to a few 1e-7 even at p ~ 1e6.
// table2 (optional) holds the same values blocked by four frequencies:
// table2[j/4][p][j%4], so that 32 threads owning 32 consecutive positions read
// 32 consecutive 32-byte pieces (the backward epilogues, one row per thread).

constexpr double kTwoPi = 6.283185307179586476925286766559;

// Rows [0, rows) x frequencies [0, half): table[p][j] = (cos, sin)(p theta^(-2j/d)),
// table2 (optional) the same blocked by four frequencies.  The angle is formed and
// reduced modulo 2 pi in fp64, then sincosf on the reduced fp32 argument.  Block `blk`
// of `nblk` takes a grid-stride share of the rows x half entries.
__device__ __forceinline__ void rope_table_body(const TabSpec& tab, int blk, int nblk) {
    __shared__ double w[256];
    const int half = tab.half;
    for (int j = threadIdx.x; j < half; j += blockDim.x)
        w[j] = exp2(-2.0 * static_cast<double>(j) / static_cast<double>(2 * half) * tab.log2_theta);
    __syncthreads();
    const int64_t n = static_cast<int64_t>(tab.rows) * half;
    for (int64_t idx = static_cast<int64_t>(blk) * blockDim.x + threadIdx.x; idx < n;
         idx += static_cast<int64_t>(nblk) * blockDim.x) {
        const int64_t p = idx / half;
        const int j = static_cast<int>(idx - p * half);
        const double x = static_cast<double>(p) * w[j];
        const double k = rint(x * (1.0 / kTwoPi));
        const double red = fma(-k, kTwoPi, x);
        float sn, cs;
        sincosf(static_cast<float>(red), &sn, &cs);
        tab.table[idx] = make_float2(cs, sn);
        if (tab.table2 != nullptr)
            tab.table2[((static_cast<int64_t>(j >> 2) * tab.rows + p) << 2) + (j & 3)] = make_float2(cs, sn);
    }
}

// One launch for a call's metadata: blocks [0, nwl) build work lists w0 (and w1), the
// remaining blocks fill the RoPE table(s).  The table does not read cu_seqlens, so it
// needs no validation and runs beside the work lists.
__global__ void __launch_bounds__(kWlThreads, 1)
meta_kernel(WlSpec w0, WlSpec w1, int nwl, TabSpec tab) {
    if (static_cast<int>(blockIdx.x) < nwl) {
        worklist_body(blockIdx.x == 0 ? w0 : w1);
        return;
    }
    if (tab.table != nullptr) rope_table_body(tab, blockIdx.x - nwl, gridDim.x - nwl);
}

static int wl_nbins(const WlSpec& w) {
    const int tile = (w.kind == VLC_WORKLIST_FWD) ? w.BM : w.BN;
    return ((w.kind == VLC_WORKLIST_FWD || w.cu_kv == nullptr ? w.max_seqlen : w.max_seqlen_kv) + tile - 1) / tile + 1;
}

cudaError_t launch_meta(const WlSpec* lists, int nwl, const TabSpec* tab, cudaStream_t s) {
    if (nwl < 0 || nwl > 2 || (nwl == 0 && tab == nullptr)) return cudaErrorInvalidValue;
    WlSpec w[2] = {};
    int nbins = 1;
    for (int i = 0; i < nwl; ++i) {
        w[i] = lists[i];
        nbins = std::max(nbins, wl_nbins(w[i]));
    }
    TabSpec tb{};
    int tblocks = 0;
    if (tab != nullptr && tab->table != nullptr) {
        tb = *tab;
        const int64_t n = static_cast<int64_t>(tb.rows) * tb.half;
        tblocks = static_cast<int>(std::min<int64_t>((n + kWlThreads - 1) / kWlThreads, 296));
    }
    const size_t smem = sizeof(int) * static_cast<size_t>(nbins);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(meta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    meta_kernel<<<nwl + tblocks, kWlThreads, smem, s>>>(w[0], w[1], nwl, tb);
    return cudaGetLastError();
}

cudaError_t launch_worklist(const int32_t* cu, int32_t nseg, int32_t total, int32_t max_seqlen,
                            int32_t BM, int32_t BN, int kind, int4* items, int64_t cap,
                            int32_t* order, int32_t* seg_base, int32_t* count, int32_t* err,
                            cudaStream_t s, const int32_t* cu_padded, const int32_t* cu_kv,
                            int32_t total_kv, int32_t max_seqlen_kv) {
    const WlSpec w{cu, nseg, total, max_seqlen, BM, BN, kind, items, cap, order, seg_base, count, err,
                   cu_padded, cu_kv, total_kv, max_seqlen_kv};
    return launch_meta(&w, 1, nullptr, s);
}

TabSpec rope_table_spec(float2* table, int32_t rows, int32_t d, double theta, float2* table2) {
    return TabSpec{table, table2, rows, d / 2, std::log2(theta)};
}

cudaError_t launch_rope_table(float2* table, int32_t rows, int32_t d, double theta,
                              const int32_t* err, cudaStream_t s, float2* table2) {
    (void)err;   // the table reads no input that needs validation
    const TabSpec tb = rope_table_spec(table, rows, d, theta, table2);
    return launch_meta(nullptr, 0, &tb, s);
}

}  // namespace vlc
