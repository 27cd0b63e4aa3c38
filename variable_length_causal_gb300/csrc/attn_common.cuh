// attn_common.cuh -- device helpers shared by the forward and backward
// attention kernels: work-unit decoding, warp-collective bounded waits, the
// 128-byte swizzle address map, and RoPE applied to a staged tile.
#pragma once
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace vlc {

struct Unit {
    int seg, tile, lo, hi, h;   // tile = q tile (forward items) or key tile (backward items)
    int L, row0;                // queries: count and first row
    int Lk, row0k;              // keys / values: count and first row (== L, row0 for self-attention)
    int off;                    // Lk - L: query p sits at position p + off and sees keys 0 .. p + off
};

// Unit u -> (item, head).  Units run over the sorted segments; inside a
// segment head-major, then the segment's items in work-list order.  The
// segment's length comes from cu, its first row from rows (cu itself, or the
// padded offsets of a layout with padding between segments); likewise for the
// keys and values from cu_kv / rows_kv.  KV == false is self-attention: the key
// side equals the query side and is not loaded.
// Executed by a whole warp: the search for the unit's segment probes 32 sorted-
// segment offsets at once and keeps the bracket the ballot points to, so a pack
// of up to 1024 segments is searched in two dependent rounds of loads (32768 in
// three) instead of one round per halving.  Every lane returns the same Unit.
template <bool KV>
__device__ __forceinline__ Unit decode_unit_warp(const int4* __restrict__ items,
                                                 const int32_t* __restrict__ seg_base,
                                                 const int32_t* __restrict__ cu,
                                                 const int32_t* __restrict__ rows,
                                                 const int32_t* __restrict__ cu_kv,
                                                 const int32_t* __restrict__ rows_kv, int nseg, int H, int u) {
    const int64_t HH = H;
    const int lane = threadIdx.x & 31;
    // invariant: H * seg_base[lo] <= u, and the answer lies in [lo, hi]
    int lo = 0, hi = nseg - 1;
    while (lo < hi) {
        const int64_t span = static_cast<int64_t>(hi - lo) + 1;
        const int pr = lo + static_cast<int>((static_cast<int64_t>(lane) * span) >> 5);   // probe 0 is lo
        const bool ok = HH * __ldg(seg_base + pr) <= u;
        const uint32_t m = __ballot_sync(0xffffffffu, ok);
        const int last = 31 - __clz(m);   // probes are non-decreasing, so the ok ones come first
        const int nlo = __shfl_sync(0xffffffffu, pr, last);
        const int nxt = __shfl_sync(0xffffffffu, pr, last < 31 ? last + 1 : 31);
        hi = last < 31 ? nxt - 1 : hi;
        lo = nlo;
    }
    const int base = __ldg(seg_base + lo);
    const int n = __ldg(seg_base + lo + 1) - base;
    const int64_t local = u - HH * base;
    Unit w;
    w.h = static_cast<int>(local / n);
    const int4 it = __ldg(items + base + static_cast<int>(local - static_cast<int64_t>(w.h) * n));
    w.seg = it.x;
    w.tile = it.y;
    w.lo = it.z;
    w.hi = it.w;
    w.L = __ldg(cu + it.x + 1) - __ldg(cu + it.x);
    w.row0 = __ldg(rows + it.x);
    if constexpr (KV) {
        w.Lk = __ldg(cu_kv + it.x + 1) - __ldg(cu_kv + it.x);
        w.row0k = __ldg(rows_kv + it.x);
        w.off = w.Lk - w.L;
    } else {
        w.Lk = w.L;
        w.row0k = w.row0;
        w.off = 0;
    }
    return w;
}

// All 32 lanes poll; succeed together or give up together (ctl as in mbar_wait).
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int* ctl) {
    // the common case first: a completed phase costs one probe and one vote (the limit is read
    // from shared memory only on the slow path, so the probe does not queue behind that load)
    if (__all_sync(0xffffffffu, mbar_test_wait(bar, parity))) return true;
    const uint32_t lim = static_cast<uint32_t>(ctl[1]);
    const bool sleep = lim >= kWaitLimitUs;
    uint64_t t0 = 0;
    const int lane = threadIdx.x & 31;
#pragma unroll 1
    for (int it = 0;; ++it) {
        const bool done = sleep ? mbar_try_wait(bar, parity) : mbar_test_wait(bar, parity);
        if (__all_sync(0xffffffffu, done)) return true;
        int give_up = 0;
        if (lane == 0 && (!sleep || it >= 64)) {
            if (t0 == 0) t0 = globaltimer_ns();
            if (ctl[0]) give_up = 1;
            else if (globaltimer_ns() - t0 > 1000ull * lim) { ctl[0] = 1; give_up = 1; }
        }
        if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
    }
}

// ---------------------------------------------------------------- dynamic unit ring
// A scheduler warp claims work units from a global counter (longest first, so
// CTAs that finish early take the next unit and the units in flight stay a
// contiguous window of the work list), decodes each one (dependent global loads:
// the search over the sorted segments, then the item and the segment's offsets)
// and publishes index and decoded unit in a ring of kRing
// shared-memory slots; every other role consumes the same sequence in order and
// reads the decoded unit from the slot.  The ring depth bounds how far the
// scheduler claims ahead of the slowest role (kRing - 1 units).  A unit index of
// -1 ends the sequence.
constexpr int kRing = 2;
constexpr int kSlotInts = 12;   // unit index + the 10 fields of Unit, padded (16-byte aligned slots)

struct Ring {
    volatile int* slot;     // kRing x kSlotInts ints in shared memory
    uint32_t full0, empty0; // barrier addresses of slot 0 (8-byte stride)
};

// The scheduler as a whole warp: lane 0 claims, every lane takes part in `decode(u)`
// (a warp-collective decode such as decode_unit_warp), lane 0 publishes.
template <class Decode>
__device__ __forceinline__ bool ring_put_warp(const Ring& rg, int n, int* counter, int nunits,
                                              volatile int* abort, Decode&& decode, int& u_out) {
    const int s = n % kRing;
    const int lane = threadIdx.x & 31;
    if (!wait_warp(rg.empty0 + 8u * s, ((n / kRing) & 1) ^ 1, abort)) return false;
    int u = 0;
    if (lane == 0) u = atomicAdd(counter, 1);
    u = __shfl_sync(0xffffffffu, u, 0);
    if (u >= nunits) u = -1;
    Unit w{};
    if (u >= 0) w = decode(u);
    if (lane == 0) {
        const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(const_cast<int*>(rg.slot + s * kSlotInts)));
        const int v[12] = {u, w.seg, w.tile, w.lo, w.hi, w.h, w.L, w.row0, w.Lk, w.row0k, w.off, 0};
#pragma unroll
        for (int q = 0; q < 3; ++q)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a + 16u * q), "r"(v[4 * q]),
                         "r"(v[4 * q + 1]), "r"(v[4 * q + 2]), "r"(v[4 * q + 3])
                         : "memory");
        mbar_arrive(rg.full0 + 8u * s);   // release: waiters see the slot
    }
    __syncwarp();
    u_out = u;
    return true;
}

__device__ __forceinline__ void ring_read(const volatile int* d, int& u, Unit& w) {
    // three 16-byte loads: the slot is read while the tensor pipe's operand reads keep the
    // shared memory busy, so every separate access costs a queueing delay
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(const_cast<int*>(d)));
    int v[12];
#pragma unroll
    for (int q = 0; q < 3; ++q)
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v[4 * q]), "=r"(v[4 * q + 1]), "=r"(v[4 * q + 2]), "=r"(v[4 * q + 3])
                     : "r"(a + 16u * q)
                     : "memory");
    u = v[0];
    w.seg = v[1]; w.tile = v[2]; w.lo = v[3]; w.hi = v[4]; w.h = v[5];
    w.L = v[6]; w.row0 = v[7]; w.Lk = v[8]; w.row0k = v[9]; w.off = v[10];
}

// One consumer thread (a TMA producer or the MMA issuer).
__device__ __forceinline__ bool ring_get(const Ring& rg, int n, volatile int* abort, int& u_out, Unit& w) {
    const int s = n % kRing;
    if (!mbar_wait(rg.full0 + 8u * s, (n / kRing) & 1, abort)) return false;
    ring_read(rg.slot + s * kSlotInts, u_out, w);
    mbar_arrive(rg.empty0 + 8u * s);
    return true;
}

// A whole consumer warp; lane 0 releases the slot once every lane has read it.
__device__ __forceinline__ bool ring_get_warp(const Ring& rg, int n, volatile int* abort, int& u_out, Unit& w);

// 16-byte chunk `ci` (0..7) of row `r` inside a block of rows x 128 bytes with
// the 128-byte swizzle used by both TMA and the MMA descriptors.
__device__ __forceinline__ uint32_t sw128(uint32_t block_base, int r, int ci) {
    return block_base + static_cast<uint32_t>(r) * 128u +
           static_cast<uint32_t>(((ci ^ (r & 7)) & 7) << 4);
}

__device__ __forceinline__ bool ring_get_warp(const Ring& rg, int n, volatile int* abort, int& u_out, Unit& w) {
    const int s = n % kRing;
    if (!wait_warp(rg.full0 + 8u * s, (n / kRing) & 1, abort)) return false;
    ring_read(rg.slot + s * kSlotInts, u_out, w);
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(rg.empty0 + 8u * s);
    return true;
}

// Named barrier among `nthreads` threads (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// RoPE pairings.  Rotate-half (IL = false) rotates columns (j, j + D/2);
// interleaved (IL = true) rotates columns (2j, 2j + 1).  Both use the
// frequencies w_j = theta^(-2j/D) of the table rows table[p][j] = (cos, sin).
//
// A RoPE thread owns two 16-byte chunks of a row: chunk ci and chunk
// ci + D/16 (its "lo" and "hi" chunks, 8 columns each).  Rotate-half pairs
// column c of the lo chunk with the same column of the hi chunk (pairs
// j = 8ci .. 8ci+7); interleaved pairs neighbours inside each chunk (pairs
// 4ci .. 4ci+3 in lo, D/4 + 4ci .. D/4 + 4ci+3 in hi).  For both, the thread
// keeps 8 angles as 4 float2 values so the arithmetic runs on packed pairs:
//   rotate-half  c[q] = (cos w_{8ci+2q}, cos w_{8ci+2q+1})
//   interleaved  c[q] = (cos w_{4ci+q},  cos w_{D/4+4ci+q})
// and likewise s[q] for the sines.
template <int D, bool IL>
__device__ __forceinline__ void rope_load(const float2* __restrict__ row, int ci, float2 c[4], float2 s[4]) {
    if constexpr (!IL) {
        const float4* t4 = reinterpret_cast<const float4*>(row + ci * 8);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 f = __ldg(t4 + q);
            c[q] = make_float2(f.x, f.z);
            s[q] = make_float2(f.y, f.w);
        }
    } else {
        const float4* lo = reinterpret_cast<const float4*>(row + ci * 4);
        const float4* hi = reinterpret_cast<const float4*>(row + D / 4 + ci * 4);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float4 a = __ldg(lo + h), b = __ldg(hi + h);
            c[2 * h] = make_float2(a.x, b.x);
            s[2 * h] = make_float2(a.y, b.y);
            c[2 * h + 1] = make_float2(a.z, b.z);
            s[2 * h + 1] = make_float2(a.w, b.w);
        }
    }
}

// Per-thread RoPE state for rope_tile: this thread always handles the same
// 8 rotation pairs of rows spaced ROWS_PER_IT apart, so the angle steps by the
// constant rotation e^{i * ROWS_PER_IT * w_j}, which is the RoPE table's row
// ROWS_PER_IT.  Loaded once per kernel.
template <int D>
struct RopeStep {
    float2 c[4], s[4], ns[4];   // cos, sin, -sin of the per-step angle (packed as in rope_load)
};

template <int D, bool IL>
__device__ __forceinline__ RopeStep<D> rope_step(const float2* __restrict__ table, int lane) {
    constexpr int half = D / 2;
    constexpr int PAIRS_PER_ROW = half / 8;
    constexpr int ROWS_PER_IT = 32 / PAIRS_PER_ROW;
    RopeStep<D> st;
    rope_load<D, IL>(table + ROWS_PER_IT * half, lane % PAIRS_PER_ROW, st.c, st.s);
#pragma unroll
    for (int q = 0; q < 4; ++q) st.ns[q] = make_float2(-st.s[q].x, -st.s[q].y);
    return st;
}

// Rotate a staged tile of ROWS rows (segment-local positions pos0 + row) in
// place: x' = x cos - y sin, y' = y cos + x sin for each pair (x, y) of the
// pairing IL, computed in fp32 (packed pairs) and rounded to bf16.  Executed
// by 128 threads (4 warps, wr = 0..3).
// A thread reads the cos/sin of its first row from the table and advances the
// angle by complex multiplication with its RopeStep (a few 1e-7 of drift over
// a tile).
// BLK: bytes between the tile's 64-column blocks (ROWS x 128 B for a whole tile; a slice of
// a taller tile passes the taller tile's block size).  gdst (optional): the rotated rows
// r < nvalid are also written to global memory, row r at gdst + r * gstride (bf16, D columns).
template <int D, int ROWS, bool IL, uint32_t BLK = ROWS * 128u>
__device__ __forceinline__ void rope_tile(uint32_t tile, int pos0, const float2* __restrict__ table,
                                          const RopeStep<D>& step, int wr, int lane,
                                          uint8_t* __restrict__ gdst = nullptr, int64_t gstride = 0,
                                          int nvalid = 0) {
    constexpr int half = D / 2;
    constexpr int PAIRS_PER_ROW = half / 8;            // threads per row
    constexpr int ROWS_PER_IT = 32 / PAIRS_PER_ROW;
    constexpr int ROWS_PER_WARP = ROWS / 4;
    const int rsub = lane / PAIRS_PER_ROW;
    const int ci = lane % PAIRS_PER_ROW;
    const int r0 = wr * ROWS_PER_WARP + rsub;
    float2 cs[4], sn[4];   // cos/sin at the current row (packed as in rope_load)
    rope_load<D, IL>(table + static_cast<int64_t>(pos0 + r0) * half, ci, cs, sn);
#pragma unroll 2
    for (int it = 0; it < ROWS_PER_WARP / ROWS_PER_IT; ++it) {
        const int r = r0 + it * ROWS_PER_IT;
        uint32_t lo_addr, hi_addr;
        if constexpr (D == 128) {
            lo_addr = sw128(tile, r, ci);
            hi_addr = sw128(tile + BLK, r, ci);
        } else {
            lo_addr = sw128(tile, r, ci);
            hi_addr = sw128(tile, r, ci + 4);
        }
        uint32_t a[4], b[4];
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]) : "r"(lo_addr));
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]) : "r"(hi_addr));
        uint32_t na[4], nb[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            // (x, y) of the two pairs that share the angles cs[q], sn[q]
            const float2 x = IL ? make_float2(bf16_lo(a[q]), bf16_lo(b[q])) : make_float2(bf16_lo(a[q]), bf16_hi(a[q]));
            const float2 y = IL ? make_float2(bf16_hi(a[q]), bf16_hi(b[q])) : make_float2(bf16_lo(b[q]), bf16_hi(b[q]));
            const float2 nsn = make_float2(-sn[q].x, -sn[q].y);
            const float2 xr = fma2(x, cs[q], mul2(y, nsn));    // x cos - y sin
            const float2 yr = fma2(y, cs[q], mul2(x, sn[q]));  // y cos + x sin
            if constexpr (IL) {
                na[q] = pack_bf16x2(xr.x, yr.x);
                nb[q] = pack_bf16x2(xr.y, yr.y);
            } else {
                na[q] = pack_bf16x2(xr.x, xr.y);
                nb[q] = pack_bf16x2(yr.x, yr.y);
            }
        }
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                     ::"r"(lo_addr), "r"(na[0]), "r"(na[1]), "r"(na[2]), "r"(na[3]) : "memory");
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                     ::"r"(hi_addr), "r"(nb[0]), "r"(nb[1]), "r"(nb[2]), "r"(nb[3]) : "memory");
        if (gdst != nullptr && r < nvalid) {   // the same 16-byte chunks of the row-major row
            uint8_t* row = gdst + r * gstride;
            *reinterpret_cast<uint4*>(row + 16 * ci) = make_uint4(na[0], na[1], na[2], na[3]);
            *reinterpret_cast<uint4*>(row + (D == 128 ? 128 : 64) + 16 * ci) = make_uint4(nb[0], nb[1], nb[2], nb[3]);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {   // advance the angle by ROWS_PER_IT rows
            const float2 c = cs[q], sv = sn[q];
            cs[q] = fma2(c, step.c[q], mul2(sv, step.ns[q]));   // c cos_d - s sin_d
            sn[q] = fma2(sv, step.c[q], mul2(c, step.s[q]));    // s cos_d + c sin_d
        }
    }
}

// ---------------------------------------------------------------- row rotation (HBM passes)
// cs/sn[2e], [2e+1]: angles of the two pairs that the e-th 32-bit words of a
// thread's lo and hi chunks take part in (rotate-half: the pairs at word e's two
// columns; interleaved: word e of lo, word e of hi), at position pos.
template <int D>
__device__ __forceinline__ void load_angles(const float2* __restrict__ table, int64_t pos, bool il, int c,
                                            float cs[8], float sn[8]) {
    if (!il) {
        const float4* t4 = reinterpret_cast<const float4*>(table + pos * (D / 2) + c * 8);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float4 f = __ldg(t4 + e);
            cs[2 * e] = f.x; sn[2 * e] = f.y; cs[2 * e + 1] = f.z; sn[2 * e + 1] = f.w;
        }
    } else {
        const float4* l4 = reinterpret_cast<const float4*>(table + pos * (D / 2) + c * 4);
        const float4* h4 = reinterpret_cast<const float4*>(table + pos * (D / 2) + D / 4 + c * 4);
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
            const float4 f = __ldg(l4 + e2), g = __ldg(h4 + e2);
            cs[4 * e2] = f.x; sn[4 * e2] = f.y; cs[4 * e2 + 1] = g.x; sn[4 * e2 + 1] = g.y;
            cs[4 * e2 + 2] = f.z; sn[4 * e2 + 2] = f.w; cs[4 * e2 + 3] = g.z; sn[4 * e2 + 3] = g.w;
        }
    }
}

// Rotate chunks a0 (lo) and a1 (hi) of one row of src into dst with the angles of
// load_angles; padding rows (real == false) become zeros, so every operand row
// stays finite.
__device__ __forceinline__ void rotate_chunks(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                              int64_t a0, int64_t a1, const float cs[8], const float sn[8],
                                              bool real, bool il) {
    if (!real) {
        dst[a0] = make_uint4(0u, 0u, 0u, 0u);
        dst[a1] = make_uint4(0u, 0u, 0u, 0u);
        return;
    }
    const uint4 x4 = __ldg(src + a0), y4 = __ldg(src + a1);
    const uint32_t xv[4] = {x4.x, x4.y, x4.z, x4.w}, yv[4] = {y4.x, y4.y, y4.z, y4.w};
    uint32_t nx[4], ny[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float c0 = cs[2 * e], s0 = sn[2 * e], c1 = cs[2 * e + 1], s1 = sn[2 * e + 1];
        if (!il) {   // pairs (lo word e, hi word e) at columns 2e and 2e+1
            const float x0 = bf16_lo(xv[e]), x1 = bf16_hi(xv[e]);
            const float y0 = bf16_lo(yv[e]), y1 = bf16_hi(yv[e]);
            nx[e] = pack_bf16x2(fmaf(x0, c0, -y0 * s0), fmaf(x1, c1, -y1 * s1));
            ny[e] = pack_bf16x2(fmaf(y0, c0, x0 * s0), fmaf(y1, c1, x1 * s1));
        } else {     // lo word e and hi word e are pairs of their own
            const float x0 = bf16_lo(xv[e]), y0 = bf16_hi(xv[e]);
            const float x1 = bf16_lo(yv[e]), y1 = bf16_hi(yv[e]);
            nx[e] = pack_bf16x2(fmaf(x0, c0, -y0 * s0), fmaf(y0, c0, x0 * s0));
            ny[e] = pack_bf16x2(fmaf(x1, c1, -y1 * s1), fmaf(y1, c1, x1 * s1));
        }
    }
    dst[a0] = make_uint4(nx[0], nx[1], nx[2], nx[3]);
    dst[a1] = make_uint4(ny[0], ny[1], ny[2], ny[3]);
}

// Largest r in [0, nseg-1] with rows[r] <= tok (clamped, in bounds).
__device__ __forceinline__ int segment_of_row(const int32_t* __restrict__ rows, int nseg, int64_t tok) {
    int a = 0, b = nseg - 1;
    while (a < b) {
        const int mid = (a + b + 1) >> 1;
        if (__ldg(rows + mid) <= tok) a = mid; else b = mid - 1;
    }
    return a;
}

}  // namespace vlc
