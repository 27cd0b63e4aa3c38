// attn_bwd.cu -- backward of the varlen block-diagonal causal attention, sm_103a.
//
// Gradients of sum(O * dO) with the standard softmax-attention derivatives,
// restricted (like the forward) to each segment's allowed pairs
// ("Sequence packing and variable-length attention", charlestar: allow(i,j)
// and the mask applied before the softmax; the page checks Q/K/V gradients by
// finite differences):
//   P = exp(S - LSE),  dV = P^T dO,  dP = dO V^T,  D_i = rowsum(dO_i * O_i),
//   dS = P o (dP - D),  dQ' = scale dS K',  dK' = scale dS^T Q',
//   dQ = R(p)^T dQ',  dK = R(p)^T dK'   (RoPE is orthogonal: its inverse is R(-p)).
//
// Three kernels, no atomics (results are bitwise reproducible):
//   prep_kernel    D = rowsum(dO * O) in fp32, layout [H, total]; with RoPE (on
//                  operands not rotated beforehand) also q' = R(p) q and
//                  k' = R(p) k once into the workspace (bf16).
//   dq_kernel      q-major, one unit = (q tile of 128 rows, head): for every key
//                  step of 128 rows, tcgen05 computes S = Q'K'^T (two TMEM buffers)
//                  and dP = dO V^T; two warpgroups (64 key columns each) form P
//                  as soon as S lands and dS once dP lands, writing dS back packed
//                  over the dP columns; tcgen05 adds dS K' (tensor-memory A
//                  operand) into a TMEM dQ accumulator; epilogue applies scale
//                  and R(p)^T and stores bf16.
//   dkdv_kernel    key-major, one unit = (key tile of 128 rows, head): for every
//                  q step of 128 rows from the diagonal to the segment end,
//                  S^T = K'Q'^T and dP^T = V dO^T into TMEM; two warpgroups (64 q
//                  columns each) form P^T as soon as S^T lands and dS^T once dP^T
//                  lands, writing them back packed into TMEM; tcgen05 accumulates
//                  dV += P^T dO and dK += dS^T Q' (tensor-memory A operands) in
//                  the order dP^T(i) dV(i) S^T(i+1) dK(i) dP^T(i+1), so each math
//                  phase has a two-MMA window; a stager warp prefetches LSE/delta;
//                  four epilogue warps store dV and R(p)^T dK while the math
//                  warps start the next unit.
// Both attention kernels are persistent (one CTA per SM) and warp-specialised:
// warp 0 TMA producer, warp 1 MMA issuer, warp 2 TMEM allocator and then unit
// scheduler (claims and decodes units for every other role), warp 3 V producer
// (dQ pass) or LSE/delta stager (dK/dV pass), warps 4-11 two math warpgroups,
// warps 12-15 (dK/dV pass only) the epilogue warpgroup.  The roles re-split the
// launch's registers with setmaxnreg inside their own branches.  Every wait is
// bounded.
#include <type_traits>
#include <cuda.h>
#include <cmath>
#include <cstdint>

#include "../../include/vlc.h"
#include "attn_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace vlc {

bool make_tmap_thd(CUtensorMap* map, const void* base, int32_t total, int32_t H, int32_t d,
                   int box_rows);

namespace bwd {

constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kDrainNs = 200000000ull;

// ====================================================================== prep
// One pass over the (token, head) rows: D = rowsum(dO * O) in fp32 ([H, total]),
// and with RoPE the rotated q' = R(p) q and k' = R(p) k (bf16, rounded once),
// so the attention passes below read pre-rotated operands.  The rows are the
// total * H query rows followed (with RoPE) by the total_kv * Hkv key rows.
// D/16 threads per row; thread c handles 16-byte chunks c and c + D/16 of the
// row: rotate-half pairs j = 8c .. 8c+7 (columns j and j+D/2), or, with the
// interleaved pairing, pairs 4c .. 4c+3 and D/4 + 4c .. D/4 + 4c+3 (columns 2j
// and 2j+1).  A query of segment r sits at position p + Lk_r - L_r (bottom-right
// alignment; 0 extra for self-attention), a key at its own index.
// SEP == false (self-attention): the row (token, head hh) also rotates key row
// (token, hh) when hh < Hkv, with the same position and angles.  SEP == true
// (keys with segments of their own): key rows follow the query rows as a range
// of their own.
template <int D, bool SEP>
__global__ void __launch_bounds__(256)
prep_kernel(const uint4* __restrict__ dout, const uint4* __restrict__ o, const uint4* __restrict__ q,
            const uint4* __restrict__ k, uint4* __restrict__ qrot, uint4* __restrict__ krot,
            float* __restrict__ delta, const int32_t* __restrict__ cu,
            const int32_t* __restrict__ seg_rows, const int32_t* __restrict__ cu_kv,
            const int32_t* __restrict__ seg_rows_kv, int32_t nseg,
            const float2* __restrict__ table, int32_t total, int32_t H, int32_t Hkv, int32_t total_kv,
            int rope, const int32_t* __restrict__ err) {
    if (*err != 0) return;
    constexpr int TPR = D / 16;        // threads per row
    constexpr int HALF = D / 16;       // uint4 chunks per half row
    const int64_t qrows = static_cast<int64_t>(total) * H;
    const int64_t rows = qrows + (SEP && rope ? static_cast<int64_t>(total_kv) * Hkv : 0);
    const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int c = threadIdx.x % TPR;
    const int64_t per_iter = nthreads / TPR;
    const bool il = rope == kRopeInterleaved;
    for (int64_t first = 0; first < rows; first += per_iter) {   // uniform trip count
        const int64_t row = first + gtid / TPR;
        float acc = 0.f;
        if (row < qrows) {          // query row: D, and q' (self-attention: and k') with RoPE
            const int64_t lo = row * (2 * HALF) + c, hi = lo + HALF;
            const uint4 g0 = __ldg(dout + lo), g1 = __ldg(dout + hi);
            const uint4 o0 = __ldg(o + lo), o1 = __ldg(o + hi);
            const uint32_t gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
            const uint32_t ov[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e)
                acc += bf16_lo(gv[e]) * bf16_lo(ov[e]) + bf16_hi(gv[e]) * bf16_hi(ov[e]);
            if (rope) {
                const int64_t tok = row / H;
                const int a = segment_of_row(seg_rows, nseg, tok);
                const int64_t L = __ldg(cu + a + 1) - __ldg(cu + a);
                const int64_t pos0 = tok - __ldg(seg_rows + a);
                const bool real = pos0 < L;   // rows past the length: padding (padded layouts)
                const int64_t off = SEP ? (__ldg(cu_kv + a + 1) - __ldg(cu_kv + a)) - L : 0;
                float cs[8], sn[8];
                if (real) load_angles<D>(table, pos0 + off, il, c, cs, sn);
                rotate_chunks(q, qrot, lo, hi, cs, sn, real, il);
                if (!SEP) {
                    const int64_t hh = row - tok * H;   // k has only Hkv heads
                    if (hh < Hkv) {
                        const int64_t klo = (tok * Hkv + hh) * (2 * HALF) + c;
                        rotate_chunks(k, krot, klo, klo + HALF, cs, sn, real, il);
                    }
                }
            }
        } else if (SEP && row < rows) {   // key row (RoPE only): k'
            const int64_t kr = row - qrows;
            const int64_t lo = kr * (2 * HALF) + c, hi = lo + HALF;
            const int64_t tok = kr / Hkv;
            const int a = segment_of_row(seg_rows_kv, nseg, tok);
            const int64_t pos0 = tok - __ldg(seg_rows_kv + a);
            const bool real = pos0 < __ldg(cu_kv + a + 1) - __ldg(cu_kv + a);
            float cs[8], sn[8];
            if (real) load_angles<D>(table, pos0, il, c, cs, sn);
            rotate_chunks(k, krot, lo, hi, cs, sn, real, il);
        }
#pragma unroll
        for (int m = TPR / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
        if (row < qrows && c == 0) {
            const int64_t tok = row / H, h = row - tok * H;
            delta[h * total + tok] = acc;
        }
    }
}

// Apply scale and R(p)^T to one row of fp32 gradients held in TMEM columns
// [col0, col0 + D) of this thread's lane, and store it as bf16.  IL selects the
// interleaved pairing (columns 2j, 2j+1), else rotate-half (j, j + D/2).  The two
// math warpgroups share a row: `part` (0 or 1) takes half of the rotation pairs.
// The cos/sin come from the blocked table (tab2[j/4][pos][j%4], tab_rows
// positions): with one row per thread and consecutive rows at consecutive
// positions, each 32-byte load of a warp covers 32 consecutive pieces; a
// sub-chunk's loads are issued before its TMEM loads.  v8: row_out is 32-byte
// aligned (256-bit stores).
template <int D, bool IL>
__device__ __forceinline__ void store_unrotated(uint32_t taddr, const float2* __restrict__ tab2, int tab_rows,
                                                int pos, float scale, bool rope, bool valid,
                                                uint8_t* __restrict__ row_out, bool v8, int part) {
    constexpr int half = D / 2;
    const float2* trow = rope ? tab2 + static_cast<int64_t>(pos) * 4 : nullptr;
    const int64_t jstride = static_cast<int64_t>(tab_rows) * 4;   // float2 per group of 4 frequencies
    if constexpr (IL) {
        // 16-column sub-chunks (8 pairs: two table loads); this part's half of the columns
#pragma unroll
        for (int b = 0; b < D / 32; ++b) {
            const int cb = part * (D / 2) + b * 16;   // first column
            float tb[2][8];
            if (rope) {
                ld_nc_v8(trow + (cb / 8) * jstride, tb[0]);
                ld_nc_v8(trow + (cb / 8 + 1) * jstride, tb[1]);
            }
            uint32_t r[16];
            tmem_ld16(taddr + cb, r);
            tmem_wait_ld();
            uint32_t pk[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {   // pair cb/2 + q at columns cb + 2q, cb + 2q + 1
                float x = __uint_as_float(r[2 * q]) * scale, y = __uint_as_float(r[2 * q + 1]) * scale;
                if (rope) {
                    const float c = tb[q >> 2][2 * (q & 3)], s = tb[q >> 2][2 * (q & 3) + 1];
                    const float u = x * c + y * s, w = y * c - x * s;
                    x = u; y = w;
                }
                pk[q] = pack_bf16x2(x, y);
            }
            if (valid) st_row32(row_out + cb * 2, pk, v8);
        }
    } else {
    // rotate-half: 16-pair sub-chunks (four table loads), pairs [part*half/2, +half/2)
#pragma unroll
    for (int b = 0; b < half / 32; ++b) {
        const int j0 = part * (half / 2) + b * 16;
        float tb[4][8];
        if (rope) {
#pragma unroll
            for (int m = 0; m < 4; ++m) ld_nc_v8(trow + (j0 / 4 + m) * jstride, tb[m]);
        }
        uint32_t lo[16], hi[16];
        tmem_ld16(taddr + j0, lo);
        tmem_ld16(taddr + half + j0, hi);
        tmem_wait_ld();
        uint32_t plo[8], phi[8];
#pragma unroll
        for (int m = 0; m < 4; ++m) {   // pairs j0 + 4m .. +3
            float g[4], h[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                g[q] = __uint_as_float(lo[4 * m + q]) * scale;
                h[q] = __uint_as_float(hi[4 * m + q]) * scale;
                if (rope) {
                    const float c = tb[m][2 * q], s = tb[m][2 * q + 1];
                    const float x = g[q] * c + h[q] * s, y = h[q] * c - g[q] * s;
                    g[q] = x; h[q] = y;
                }
            }
            plo[2 * m] = pack_bf16x2(g[0], g[1]);
            plo[2 * m + 1] = pack_bf16x2(g[2], g[3]);
            phi[2 * m] = pack_bf16x2(h[0], h[1]);
            phi[2 * m + 1] = pack_bf16x2(h[2], h[3]);
        }
        if (valid) {
            st_row32(row_out + j0 * 2, plo, v8);
            st_row32(row_out + (half + j0) * 2, phi, v8);
        }
    }
    }
}

// The same with the row's cos/sin loaded ahead (load_unrot_tables, D/2 floats for this
// part's pairs in sub-chunk order), for a warp that has the registers to hold them while
// it waits for the accumulator.
template <int D, bool IL>
__device__ __forceinline__ void load_unrot_tables(const float2* __restrict__ tab2, int tab_rows, int pos,
                                                  int part, float (&tb)[D / 2]) {
    const float2* trow = tab2 + static_cast<int64_t>(pos) * 4;
    const int64_t jstride = static_cast<int64_t>(tab_rows) * 4;   // float2 per group of 4 frequencies
    if constexpr (IL) {
#pragma unroll
        for (int b = 0; b < D / 32; ++b) {   // 16-column sub-chunks: 8 pairs, two loads
            const int cb = part * (D / 2) + b * 16;
            ld_nc_v8(trow + (cb / 8) * jstride, tb + 16 * b);
            ld_nc_v8(trow + (cb / 8 + 1) * jstride, tb + 16 * b + 8);
        }
    } else {
#pragma unroll
        for (int b = 0; b < D / 64; ++b) {   // 16-pair sub-chunks: four loads
            const int j0 = part * (D / 4) + b * 16;
#pragma unroll
            for (int m = 0; m < 4; ++m) ld_nc_v8(trow + (j0 / 4 + m) * jstride, tb + 32 * b + 8 * m);
        }
    }
}

template <int D, bool IL>
__device__ __forceinline__ void store_unrotated_tb(uint32_t taddr, const float (&tb)[D / 2], float scale, bool rope,
                                                   bool valid, uint8_t* __restrict__ row_out, bool v8, int part) {
    constexpr int half = D / 2;
    if constexpr (IL) {
#pragma unroll
        for (int b = 0; b < D / 32; ++b) {
            const int cb = part * (D / 2) + b * 16;   // first column
            uint32_t r[16];
            tmem_ld16(taddr + cb, r);
            tmem_wait_ld();
            uint32_t pk[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {   // pair cb/2 + q at columns cb + 2q, cb + 2q + 1
                float x = __uint_as_float(r[2 * q]) * scale, y = __uint_as_float(r[2 * q + 1]) * scale;
                if (rope) {
                    const float c = tb[16 * b + 2 * q], s = tb[16 * b + 2 * q + 1];
                    const float u = x * c + y * s, w = y * c - x * s;
                    x = u; y = w;
                }
                pk[q] = pack_bf16x2(x, y);
            }
            if (valid) st_row32(row_out + cb * 2, pk, v8);
        }
    } else {
#pragma unroll
        for (int b = 0; b < half / 32; ++b) {
            const int j0 = part * (half / 2) + b * 16;
            uint32_t lo[16], hi[16];
            tmem_ld16(taddr + j0, lo);
            tmem_ld16(taddr + half + j0, hi);
            tmem_wait_ld();
            uint32_t plo[8], phi[8];
#pragma unroll
            for (int m = 0; m < 4; ++m) {   // pairs j0 + 4m .. +3
                float g[4], h[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    g[q] = __uint_as_float(lo[4 * m + q]) * scale;
                    h[q] = __uint_as_float(hi[4 * m + q]) * scale;
                    if (rope) {
                        const float c = tb[32 * b + 8 * m + 2 * q], s = tb[32 * b + 8 * m + 2 * q + 1];
                        const float x = g[q] * c + h[q] * s, y = h[q] * c - g[q] * s;
                        g[q] = x; h[q] = y;
                    }
                }
                plo[2 * m] = pack_bf16x2(g[0], g[1]);
                plo[2 * m + 1] = pack_bf16x2(g[2], g[3]);
                phi[2 * m] = pack_bf16x2(h[0], h[1]);
                phi[2 * m + 1] = pack_bf16x2(h[2], h[3]);
            }
            if (valid) {
                st_row32(row_out + j0 * 2, plo, v8);
                st_row32(row_out + (half + j0) * 2, phi, v8);
            }
        }
    }
}

// TMEM column of the packed bf16 K-slice k (16 columns of a 64-column step) when
// math warpgroup g owns step columns [32g, 32g + 32) and packs them into TMEM
// columns [32g, 32g + 16) of the step buffer.
__device__ __forceinline__ uint32_t packed_col(int k) { return (k >> 1) * 32 + (k & 1) * 8; }

// ====================================================================== dQ pass
namespace dq {

constexpr int BK = 128;        // key rows per step (N = 128 keeps the MMAs at full rate)
// Register split of the launch's 168 per thread (the launcher checks the count): the
// control warps (TMA, MMA, scheduler, V producer) give theirs to the math warps, which
// then hold the epilogue's cos/sin while they wait for the accumulator.
constexpr uint32_t kLaunchRegsQ = 168, kCtrlRegsQ = 80, kMathRegsQ = 208;
static_assert(128 * kCtrlRegsQ + 256 * kMathRegsQ <= kThreads * kLaunchRegsQ, "register split exceeds the pool");
constexpr int kKStages = 3;   // K(j) is held from S(j) until dQ(j) completes
constexpr int kVStages = 2;

enum : int {
    QD_FULL = 0, QD_EMPTY = 1, QT_FULL = 2, QT_EMPTY = 3,
    K_FULL = 4, K_EMPTY = K_FULL + kKStages, V_FULL = K_EMPTY + kKStages, V_EMPTY = V_FULL + kVStages,
    S_FULL = V_EMPTY + kVStages, S_EMPTY = S_FULL + 1, DP_FULL = S_FULL + 2, DS_FULL = S_FULL + 3,
    ACC_FULL = S_FULL + 4, ACC_EMPTY = ACC_FULL + 1, DRAIN = ACC_FULL + 2,
    UNIT_FULL = ACC_FULL + 3, UNIT_EMPTY = UNIT_FULL + kRing, NUM_BARS = UNIT_EMPTY + kRing
};

template <int D>
struct Layout {
    static constexpr int KB = D / 64;
    static constexpr uint32_t BLK = 128u * 128u;       // 128 rows x 128 B
    static constexpr uint32_t TILE = 128u * D * 2u;
    static constexpr uint32_t Q0 = 0;                          // one staging slot
    static constexpr uint32_t DO0 = TILE;                      // one staging slot
    static constexpr uint32_t K0 = 2 * TILE;                   // kKStages
    static constexpr uint32_t V0 = K0 + kKStages * TILE;       // kVStages
    static constexpr uint32_t BAR0 = V0 + kVStages * TILE;
    static constexpr uint32_t MISC = BAR0 + NUM_BARS * 8;      // tmem slot, abort flag, wait limit, unit ring
    static constexpr uint32_t RING = (MISC + 16 + 15) / 16 * 16;   // 16-byte aligned slots
    static constexpr uint32_t BYTES = RING + 4 * kSlotInts * kRing;
    static constexpr uint32_t ALLOC = BYTES + 1024;
    // TMEM: S at columns 0..127, dP at 128 (the packed bf16 dS of a step overwrites
    // the consumed dP columns), the dQ accumulator at 256, and the unit's Q' and dO
    // (bf16 pairs, one lane per query row) as the A operands of the S and dP MMAs.
    static constexpr uint32_t S_COL = 0, DP_COL = 128, DQ_COL = 256;
    static constexpr uint32_t QT_COL = 256 + D, DOT_COL = 256 + D + D / 2;
    static_assert(DOT_COL + D / 2 <= 512, "TMEM columns");
};

// TMEM column of dS K-slice k (16 key columns): warpgroup g owns key columns
// [64g, 64g + 64) and packs them into dP columns [64g, 64g + 32).
__device__ __forceinline__ uint32_t ds_col(int k) { return (k >> 2) * 64 + (k & 3) * 8; }

// Copy this thread's row of a staged [128 x D] bf16 tile (128-byte swizzle,
// 64-column blocks) into TMEM as bf16 pairs: warpgroup g copies the row's
// columns [D/2 * g, D/2 * (g + 1)) to TMEM columns col0 + [D/4 * g, D/4 * (g + 1)).
template <int D>
__device__ __forceinline__ void stage_row_to_tmem(uint32_t tile, int r, int g, uint32_t taddr_row) {
    constexpr uint32_t BLK = 128u * 128u;
    if constexpr (D == 128) {
        uint32_t v[32];
        const uint32_t blk = tile + g * BLK;
#pragma unroll
        for (int c = 0; c < 8; ++c)
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v[4 * c]), "=r"(v[4 * c + 1]), "=r"(v[4 * c + 2]), "=r"(v[4 * c + 3])
                         : "r"(sw128(blk, r, c)));
        tmem_st32(taddr_row + 32 * g, v);
    } else {
        uint32_t v[16];
#pragma unroll
        for (int c = 0; c < 4; ++c)
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v[4 * c]), "=r"(v[4 * c + 1]), "=r"(v[4 * c + 2]), "=r"(v[4 * c + 3])
                         : "r"(sw128(tile, r, 4 * g + c)));
        tmem_st16(taddr_row + 16 * g, v);
    }
}

template <int D, bool KV>
__global__ void __launch_bounds__(kThreads, 1)
dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
          const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
          const BwdParams p) {
    using LY = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (sbase - smem_u32(smem_raw));
    auto bar = [&](int i) -> uint32_t { return sbase + LY::BAR0 + 8u * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sgen + LY::MISC);
    volatile int* abort = reinterpret_cast<volatile int*>(sgen + LY::MISC + 4);   // [abort flag, wait limit in us]
    const Ring rg{reinterpret_cast<volatile int*>(sgen + LY::RING), bar(UNIT_FULL), bar(UNIT_EMPTY)};
    constexpr int kRingConsumers = 1 + 1 + 1 + 8;   // Q'/dO/K' and V producers, MMA warp, 8 math warps
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    __shared__ int s_skip, s_nunits;
    if (threadIdx.x == 0) {
        s_skip = *reinterpret_cast<volatile int32_t*>(p.err);
        s_nunits = *reinterpret_cast<const volatile int32_t*>(p.count) * p.H;
    }
    __syncthreads();
    if (s_skip != 0) return;
    const int nunits = s_nunits;

    if (threadIdx.x == 0) {
        mbar_init(bar(QD_FULL), 1);
        mbar_init(bar(QD_EMPTY), 8);      // one arrival per math warp once its rows are in TMEM
        mbar_init(bar(QT_FULL), 256);
        mbar_init(bar(QT_EMPTY), 1);
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(bar(K_FULL + i), 1);
            mbar_init(bar(K_EMPTY + i), 1);
        }
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(bar(V_FULL + i), 1);
            mbar_init(bar(V_EMPTY + i), 1);
        }
        mbar_init(bar(S_FULL), 1);
        mbar_init(bar(S_EMPTY), 256);
        mbar_init(bar(DP_FULL), 1);
        mbar_init(bar(DS_FULL), 256);
        mbar_init(bar(ACC_FULL), 1);
        mbar_init(bar(ACC_EMPTY), 256);
        mbar_init(bar(DRAIN), 1);
        for (int i = 0; i < kRing; ++i) {
            mbar_init(bar(UNIT_FULL + i), 1);
            mbar_init(bar(UNIT_EMPTY + i), kRingConsumers);
        }
        abort[0] = 0;
        abort[1] = static_cast<int>(p.wait_limit_us);   // the waits' limit (ctl[1])
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    uint32_t q_issued = 0, k_issued = 0, v_issued = 0;

    if (warp == 0) {
        setmaxnreg_dec<kCtrlRegsQ>();
        if (lane == 0) {   // ---------------------------------------- TMA producer: Q' / dO and K'
            const uint64_t pol_stream = make_l2_policy_evict_first();   // q/dO: once per unit
            const uint64_t pol_keep = make_l2_policy_evict_last();      // K/V: re-read by other units
            uint32_t unit_it = 0, kv = 0;
            bool ok = true;
            for (int n = 0; ok; ++n, ++unit_it) {
                int u;
                Unit w;
                if (!(ok = ring_get(rg, n, abort, u, w)) || u < 0) break;
                // the staging slot frees as soon as the math warps copied the last unit's rows to TMEM
                if (!(ok = mbar_wait(bar(QD_EMPTY), (unit_it & 1) ^ 1, abort))) break;
                mbar_expect_tx(bar(QD_FULL), 2 * LY::TILE);
                const int qrow = w.row0 + w.tile * 128;
#pragma unroll
                for (int kb = 0; kb < LY::KB; ++kb) {
                    tma_load_3d_hint(sbase + LY::Q0 + kb * LY::BLK, &tmQ, kb * 64, w.h, qrow, bar(QD_FULL),
                                     pol_stream);
                    tma_load_3d_hint(sbase + LY::DO0 + kb * LY::BLK, &tmDO, kb * 64, w.h, qrow, bar(QD_FULL),
                                     pol_stream);
                }
                q_issued = unit_it + 1;
                for (int j = 0; j < w.hi && ok; ++j) {
                    const uint32_t nn = kv + j;
                    const int ks = nn % kKStages;
                    if (!(ok = mbar_wait(bar(K_EMPTY + ks), ((nn / kKStages) & 1) ^ 1, abort))) break;
                    mbar_expect_tx(bar(K_FULL + ks), LY::TILE);
#pragma unroll
                    for (int kb = 0; kb < LY::KB; ++kb)
                        tma_load_3d_hint(sbase + LY::K0 + ks * LY::TILE + kb * LY::BLK, &tmK, kb * 64,
                                         w.h / (p.H / p.Hkv), w.row0k + j * BK, bar(K_FULL + ks), pol_keep);
                    k_issued = nn + 1;
                }
                kv += w.hi;
            }
        }
        __syncwarp();
    } else if (warp == 3) {
        setmaxnreg_dec<kCtrlRegsQ>();
        if (lane == 0) {   // ---------------------------------------- TMA producer: V
            const uint64_t pol_keep = make_l2_policy_evict_last();
            uint32_t kv = 0;
            bool ok = true;
            for (int n = 0; ok; ++n) {
                int u;
                Unit w;
                if (!(ok = ring_get(rg, n, abort, u, w)) || u < 0) break;
                for (int j = 0; j < w.hi && ok; ++j) {
                    const uint32_t nn = kv + j;
                    const int vs = nn % kVStages;
                    if (!(ok = mbar_wait(bar(V_EMPTY + vs), ((nn / kVStages) & 1) ^ 1, abort))) break;
                    mbar_expect_tx(bar(V_FULL + vs), LY::TILE);
#pragma unroll
                    for (int kb = 0; kb < LY::KB; ++kb)
                        tma_load_3d_hint(sbase + LY::V0 + vs * LY::TILE + kb * LY::BLK, &tmV, kb * 64,
                                         w.h / (p.H / p.Hkv), w.row0k + j * BK, bar(V_FULL + vs), pol_keep);
                    v_issued = nn + 1;
                }
                kv += w.hi;
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        setmaxnreg_dec<kCtrlRegsQ>();
        {   // ---------------------------------------- MMA issuer (converged warp, one elected lane issues)
            constexpr uint32_t IDESC_S = idesc_bf16_f32(128, BK, false);
            constexpr uint32_t IDESC_DQ = idesc_bf16_f32(128, D, true);
            uint32_t unit_it = 0, kv = 0;
            bool ok = true;
            auto commit = [&](uint32_t b) {
                if (elect_one()) mma_commit(b);
                __syncwarp();
            };
            // S(n) = Q'K'(n)^T: Q' from TMEM, K' from shared memory; the S columns are free
            // once the math warps have read S(n-1)
            auto issue_s = [&](uint32_t nn) -> bool {
                const int ks = nn % kKStages;
                if (!wait_warp(bar(K_FULL + ks), (nn / kKStages) & 1, abort)) return false;
                if (!wait_warp(bar(S_EMPTY), (nn & 1) ^ 1, abort)) return false;
                tc_fence_after();
                const uint64_t kd = smem_desc_sw128(sbase + LY::K0 + ks * LY::TILE, 16, 1024);
                if (elect_one()) {
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t off = ((k >> 2) * LY::BLK + (k & 3) * 32) >> 4;
                        mma_bf16_ts(tmem + LY::S_COL, tmem + LY::QT_COL + 8 * k, kd + off, IDESC_S,
                                    k > 0 ? 1u : 0u);
                    }
                    mma_commit(bar(S_FULL));
                }
                __syncwarp();
                return true;
            };
            // dP(n) = dO V(n)^T: dO from TMEM (the dP columns were last read by dQ(n-1), issued earlier)
            auto issue_dp = [&](uint32_t nn) -> bool {
                const int vs = nn % kVStages;
                if (!wait_warp(bar(V_FULL + vs), (nn / kVStages) & 1, abort)) return false;
                tc_fence_after();
                const uint64_t vd = smem_desc_sw128(sbase + LY::V0 + vs * LY::TILE, 16, 1024);
                if (elect_one()) {
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t off = ((k >> 2) * LY::BLK + (k & 3) * 32) >> 4;
                        mma_bf16_ts(tmem + LY::DP_COL, tmem + LY::DOT_COL + 8 * k, vd + off, IDESC_S,
                                    k > 0 ? 1u : 0u);
                    }
                    mma_commit(bar(DP_FULL));
                    mma_commit(bar(V_EMPTY + vs));
                }
                __syncwarp();
                return true;
            };
            for (int n = 0; ok; ++n, ++unit_it) {
                int u;
                Unit w;
                if (!(ok = ring_get_warp(rg, n, abort, u, w)) || u < 0) break;
                if (!(ok = wait_warp(bar(QT_FULL), unit_it & 1, abort))) break;
                if (!(ok = issue_s(kv))) break;
                if (!(ok = issue_dp(kv))) break;
                for (int j = 0; j < w.hi; ++j) {
                    const uint32_t nn = kv + j;
                    if (j + 1 < w.hi && !(ok = issue_s(nn + 1))) break;
                    if (j == w.hi - 1) commit(bar(QT_EMPTY));   // after the last S / dP of the unit
                    // dQ += dS(n) K'(n): dS packed over the dP columns
                    if (j == 0 && !(ok = wait_warp(bar(ACC_EMPTY), (unit_it & 1) ^ 1, abort))) break;
                    if (!(ok = wait_warp(bar(DS_FULL), nn & 1, abort))) break;
                    tc_fence_after();
                    const int ks = nn % kKStages;
                    const uint64_t kd = smem_desc_sw128(sbase + LY::K0 + ks * LY::TILE, LY::BLK, 1024);
                    if (elect_one()) {
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k)
                            mma_bf16_ts(tmem + LY::DQ_COL, tmem + LY::DP_COL + ds_col(k),
                                        kd + ((k * 16 * 128) >> 4), IDESC_DQ, (j > 0 || k > 0) ? 1u : 0u);
                        mma_commit(bar(K_EMPTY + ks));
                    }
                    __syncwarp();
                    if (j + 1 < w.hi && !(ok = issue_dp(nn + 1))) break;
                }
                if (!ok) break;
                commit(bar(ACC_FULL));
                kv += w.hi;
            }
            commit(bar(DRAIN));
            mbar_wait_limit(bar(DRAIN), 0, kDrainNs);
        }
        __syncwarp();
    } else if (warp == 2) {
        setmaxnreg_dec<kCtrlRegsQ>();
        // ------------------------------------------------------------ unit scheduler (after the
        // TMEM allocation): claims and decodes units ahead of the other roles
        {   // the whole warp: lane 0 claims and publishes, all lanes decode
            auto decode = [&](int u) {
                Unit w = decode_unit_warp<KV>(p.items, p.seg_base, p.cu, p.rows, p.cu_kv, p.rows_kv, p.nseg, p.H, u);
                if (KV && p.keys_all_visible) w.off = w.Lk;   // the diagonal past the last key: no mask
                return w;
            };
            for (int n = 0;; ++n) {
                int u;
                if (!ring_put_warp(rg, n, p.next_q, nunits, abort, decode, u) || u < 0) break;
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        setmaxnreg_inc<kMathRegsQ>();
        // ------------------------------------------------------------ Q'/dO staging, P, dS + epilogue
        const int g = (warp - 4) >> 2;             // math warpgroup: key columns [64g, 64g + 64)
        const int wq = warp & 3;
        const int r = wq * 32 + lane;              // query row = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const float scale_log2 = p.scale * kLog2e;
        const bool v8 = (reinterpret_cast<uintptr_t>(p.dq) & 31) == 0;   // 256-bit row stores
        const int c0 = 64 * g;
        uint32_t unit_it = 0, kv = 0;
        // Copy unit k's Q' and dO rows into TMEM once its tiles have landed and the
        // previous unit's last S / dP MMAs are done; then free the staging slot.
        auto stage = [&](uint32_t k) -> bool {
            if (!wait_warp(bar(QD_FULL), k & 1, abort)) return false;
            if (!wait_warp(bar(QT_EMPTY), (k & 1) ^ 1, abort)) return false;
            tc_fence_after();
            stage_row_to_tmem<D>(sbase + LY::Q0, r, g, tmem + lane_off + LY::QT_COL);
            stage_row_to_tmem<D>(sbase + LY::DO0, r, g, tmem + lane_off + LY::DOT_COL);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(QT_FULL));
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(QD_EMPTY));
            return true;
        };
        int u = -1;
        Unit w{};
        bool ok = ring_get_warp(rg, 0, abort, u, w);
        bool have = ok && u >= 0;
        if (have) ok = have = stage(0);
        // this row's LSE (base 2) and D of a unit; a row past the segment gets lse2 = +inf, so
        // its P is exp2(-inf) = 0 without a mask
        auto row_stats = [&](const Unit& uw, float& l2, float& dd) {
            const int qp = uw.tile * 128 + r;
            l2 = INFINITY;
            dd = 0.f;
            if (qp < uw.L) {
                const int64_t idx = static_cast<int64_t>(uw.h) * p.total + uw.row0 + qp;
                l2 = __ldg(p.lse + idx) * kLog2e;
                dd = __ldg(p.delta + idx);
            }
        };
        float lse2_next = 0.f, dlt_next = 0.f;   // the next unit's, loaded before this unit's epilogue
        if (have) row_stats(w, lse2_next, dlt_next);
        while (have) {
            const int qpos = w.tile * 128 + r;
            const bool valid = qpos < w.L;
            const int rpos = valid ? qpos + w.off : 0;   // RoPE position of the query
            // last key this row sees; the mask applies from key tile j_edge on (the last
            // tile, or the last two when the diagonal is not tile-aligned: off % BK != 0)
            const int lastk = min(qpos + w.off, w.Lk - 1);
            const int j_edge = w.hi - 1 - ((w.off & (BK - 1)) != 0 ? 1 : 0);
            const int64_t tok = static_cast<int64_t>(w.row0) + (valid ? qpos : 0);
            const float lse2 = lse2_next, dlt = dlt_next;
            for (int j = 0; j < w.hi; ++j, ++kv) {
                // ---- phase A: P = exp2(s * scale_log2 - lse2) (masked), kept packed
                if (!(ok = wait_warp(bar(S_FULL), kv & 1, abort))) break;
                tc_fence_after();
                uint32_t sa[32], sb[32];
                tmem_ld32(tmem + lane_off + LY::S_COL + c0, sa);
                tmem_ld32(tmem + lane_off + LY::S_COL + c0 + 32, sb);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(bar(S_EMPTY));
                // diagonal step(s) and the segment tail mask key columns c > lim (scores -> -inf);
                // the other steps take a loop without the compare
                const bool edge = j >= j_edge;
                const int lim = lastk - j * BK;
                const float2 sc2 = make_float2(scale_log2, scale_log2), nl2 = make_float2(-lse2, -lse2);
                uint32_t pp[32];
                auto phase_a = [&](auto masked) {
#pragma unroll
                    for (int e = 0; e < 64; e += 2) {
                        const uint32_t* src = (e < 32) ? sa : sb;
                        const int ee = e & 31;
                        float2 s = make_float2(__uint_as_float(src[ee]), __uint_as_float(src[ee + 1]));
                        if constexpr (decltype(masked)::value) {
                            const int col = c0 + e;
                            if (col > lim) s.x = -INFINITY;
                            if (col + 1 > lim) s.y = -INFINITY;
                        }
                        const float2 x = fma2(s, sc2, nl2);
                        pp[e >> 1] = pack_bf16x2(ex2_approx(x.x), ex2_approx(x.y));
                    }
                };
                if (edge) phase_a(std::true_type{});
                else phase_a(std::false_type{});
                // ---- phase B: dS = P (dP - D), packed over the consumed dP columns
                if (!(ok = wait_warp(bar(DP_FULL), kv & 1, abort))) break;
                tc_fence_after();
                tmem_ld32(tmem + lane_off + LY::DP_COL + c0, sa);
                tmem_ld32(tmem + lane_off + LY::DP_COL + c0 + 32, sb);
                tmem_wait_ld();
                const float2 nd2 = make_float2(-dlt, -dlt);
                uint32_t pk[32];
#pragma unroll
                for (int e = 0; e < 64; e += 2) {
                    const uint32_t* src = (e < 32) ? sa : sb;
                    const int ee = e & 31;
                    const float2 pv = make_float2(bf16_lo(pp[e >> 1]), bf16_hi(pp[e >> 1]));
                    const float2 ds = mul2(pv, add2(make_float2(__uint_as_float(src[ee]),
                                                                __uint_as_float(src[ee + 1])), nd2));
                    pk[e >> 1] = pack_bf16x2(ds.x, ds.y);
                }
                tmem_st32(tmem + lane_off + LY::DP_COL + c0, pk);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(DS_FULL));
            }
            if (!ok) break;
            // cos/sin of this row's rotation pairs, in flight across the staging and the ACC wait
            const bool il = p.use_rope == kRopeInterleaved;
            float tb[D / 2];
            if (p.use_rope) {
                if (il) load_unrot_tables<D, true>(p.table2, p.table_rows, rpos, g, tb);
                else load_unrot_tables<D, false>(p.table2, p.table_rows, rpos, g, tb);
            }
            // stage the next unit before this unit's epilogue, so its first MMAs can start
            Unit w2{};
            int u2 = -1;
            if (!(ok = ring_get_warp(rg, static_cast<int>(unit_it) + 1, abort, u2, w2))) break;
            const bool have_next = u2 >= 0;
            if (have_next) {
                row_stats(w2, lse2_next, dlt_next);   // in flight across the staging and the epilogue
                if (!(ok = stage(unit_it + 1))) break;
            }
            if (!(ok = wait_warp(bar(ACC_FULL), unit_it & 1, abort))) break;
            tc_fence_after();
            {   // both warpgroups: each takes half of the row's rotation pairs
                uint8_t* row_out = reinterpret_cast<uint8_t*>(p.dq) + (tok * p.H + w.h) * static_cast<int64_t>(D) * 2;
                if (il) store_unrotated_tb<D, true>(tmem + lane_off + LY::DQ_COL, tb, p.scale, true, valid, row_out, v8, g);
                else store_unrotated_tb<D, false>(tmem + lane_off + LY::DQ_COL, tb, p.scale, p.use_rope != 0, valid,
                                                  row_out, v8, g);
            }
            tc_fence_before();
            mbar_arrive(bar(ACC_EMPTY));
            w = w2;
            have = have_next;
            ++unit_it;
        }
    }

    __syncthreads();
    if (*abort) {
        // each producer waits (bounded) for the last copy it issued into every slot and stage
        if (warp == 0 && lane == 0) {
            if (q_issued > 0) mbar_wait_limit(bar(QD_FULL), (q_issued - 1) & 1, kDrainNs);
            for (int s2 = 0; s2 < kKStages; ++s2)
                if (k_issued > static_cast<uint32_t>(s2)) {
                    const uint32_t nn = k_issued - 1 - ((k_issued - 1 - s2) % kKStages);
                    mbar_wait_limit(bar(K_FULL + s2), (nn / kKStages) & 1, kDrainNs);
                }
        }
        if (warp == 3 && lane == 0) {
            for (int s2 = 0; s2 < kVStages; ++s2)
                if (v_issued > static_cast<uint32_t>(s2)) {
                    const uint32_t nn = v_issued - 1 - ((v_issued - 1 - s2) % kVStages);
                    mbar_wait_limit(bar(V_FULL + s2), (nn / kVStages) & 1, kDrainNs);
                }
        }
        if (threadIdx.x == 0) atomicOr(p.err, VLC_DEVERR_TIMEOUT);
        __syncthreads();
    }
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace dq

// ====================================================================== dK/dV pass
namespace dkdv {

constexpr int BQ = 128;       // q rows per step (N = 128 keeps the S^T / dP^T MMAs at full rate)
// 4 control warps (TMA, MMA, scheduler, LSE/delta stager), 8 math warps (P^T, dS^T) and 4
// epilogue warps (dV, dK out of TMEM), so that the math warps go on to the next unit while
// the epilogue warps drain the accumulators.  The block's 128 registers per thread are
// re-split at run time: the launcher checks that the kernel was built with exactly 128.
constexpr int kThreadsKV = 512;
constexpr uint32_t kLaunchRegsKV = 65536 / kThreadsKV;
constexpr uint32_t kCtrlRegs = 80, kMathRegs = 144, kEpiRegs = 144;
static_assert(kCtrlRegs % 8 == 0 && kMathRegs % 8 == 0 && kEpiRegs % 8 == 0, "register counts are multiples of 8");
static_assert(kCtrlRegs + 2 * kMathRegs + kEpiRegs <= 4 * kLaunchRegsKV, "register split exceeds the pool");
constexpr int kQStages = 2;
constexpr int kLsedSlots = 3;

enum : int {
    KV_FULL = 0, KV_EMPTY = 1,
    QO_FULL = 2, QO_EMPTY = 2 + kQStages,
    ST_FULL = 2 + 2 * kQStages, DPT_FULL = ST_FULL + 1, PT_FULL = ST_FULL + 2, DST_FULL = ST_FULL + 3,
    LSED_FULL = ST_FULL + 4, LSED_EMPTY = LSED_FULL + kLsedSlots,
    ACC_FULL = LSED_EMPTY + kLsedSlots, ACC_EMPTY = ACC_FULL + 1, DRAIN = ACC_FULL + 2, DV_FULL = ACC_FULL + 3,
    DV_EMPTY = ACC_FULL + 4, UNIT_FULL = ACC_FULL + 5, UNIT_EMPTY = UNIT_FULL + kRing, NUM_BARS = UNIT_EMPTY + kRing
};

template <int D>
struct Layout {
    static constexpr int KB = D / 64;
    static constexpr uint32_t BLK = 128u * 128u;        // 128 rows x 128 B
    static constexpr uint32_t TILE = 128u * D * 2u;
    static constexpr uint32_t K0 = 0;
    static constexpr uint32_t V0 = TILE;
    static constexpr uint32_t Q0 = 2 * TILE;                   // kQStages stages
    static constexpr uint32_t DO0 = Q0 + kQStages * TILE;      // kQStages stages
    static constexpr uint32_t LSED = DO0 + kQStages * TILE;    // kLsedSlots x (128 lse2 + 128 delta)
    static constexpr uint32_t BAR0 = LSED + kLsedSlots * 256 * 4;
    static constexpr uint32_t MISC = BAR0 + NUM_BARS * 8;      // tmem slot, abort flag, wait limit, unit ring
    static constexpr uint32_t RING = (MISC + 16 + 15) / 16 * 16;   // 16-byte aligned slots
    static constexpr uint32_t BYTES = RING + 4 * kSlotInts * kRing;
    static constexpr uint32_t ALLOC = BYTES + 1024;
    // TMEM: S^T at 0, dP^T at 128 (the packed bf16 P^T / dS^T of a step overwrite the
    // consumed S^T / dP^T columns), dV and dK accumulators after them.
    static constexpr uint32_t DPT_COL = 128, DV_COL = 256, DK_COL = 256 + D;
};

template <int D, bool KV>
__global__ void __launch_bounds__(kThreadsKV, 1)
dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
            const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
            const BwdParams p) {
    using LY = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (sbase - smem_u32(smem_raw));
    auto bar = [&](int i) -> uint32_t { return sbase + LY::BAR0 + 8u * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sgen + LY::MISC);
    volatile int* abort = reinterpret_cast<volatile int*>(sgen + LY::MISC + 4);   // [abort flag, wait limit in us]
    const Ring rg{reinterpret_cast<volatile int*>(sgen + LY::RING), bar(UNIT_FULL), bar(UNIT_EMPTY)};
    constexpr int kRingConsumers = 1 + 1 + 1 + 8 + 4;   // TMA producer, MMA warp, LSE/delta stager, 8 math warps,
                                                        // 4 epilogue warps
    float* lsed = reinterpret_cast<float*>(sgen + LY::LSED);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = p.H / p.Hkv;   // query heads per key/value head: a unit runs over all of them

    __shared__ int s_skip, s_nunits;
    if (threadIdx.x == 0) {
        s_skip = *reinterpret_cast<volatile int32_t*>(p.err);
        s_nunits = *reinterpret_cast<const volatile int32_t*>(p.count_k) * p.Hkv;
    }
    __syncthreads();
    if (s_skip != 0) return;
    const int nunits = s_nunits;

    if (threadIdx.x == 0) {
        mbar_init(bar(KV_FULL), 1);
        mbar_init(bar(KV_EMPTY), 1);
        for (int i = 0; i < kQStages; ++i) {
            mbar_init(bar(QO_FULL + i), 1);
            mbar_init(bar(QO_EMPTY + i), 1);
        }
        mbar_init(bar(ST_FULL), 1);
        mbar_init(bar(DPT_FULL), 1);
        mbar_init(bar(PT_FULL), 256);
        mbar_init(bar(DST_FULL), 256);
        for (int i = 0; i < kLsedSlots; ++i) {
            mbar_init(bar(LSED_FULL + i), 1);
            mbar_init(bar(LSED_EMPTY + i), 8);
        }
        mbar_init(bar(ACC_FULL), 1);
        mbar_init(bar(ACC_EMPTY), 128);   // dK columns read by the 4 epilogue warps
        mbar_init(bar(DV_FULL), 1);
        mbar_init(bar(DV_EMPTY), 128);    // dV columns read
        mbar_init(bar(DRAIN), 1);
        for (int i = 0; i < kRing; ++i) {
            mbar_init(bar(UNIT_FULL + i), 1);
            mbar_init(bar(UNIT_EMPTY + i), kRingConsumers);
        }
        abort[0] = 0;
        abort[1] = static_cast<int>(p.wait_limit_us);   // the waits' limit (ctl[1])
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    uint32_t kv_issued = 0, q_issued = 0;

    if (warp == 0) {
        setmaxnreg_dec<kCtrlRegs>();
        if (lane == 0) {   // ---------------------------------------- TMA producer
            const uint64_t pol_stream = make_l2_policy_evict_first();   // K/V: once per unit
            const uint64_t pol_keep = make_l2_policy_evict_last();      // q/dO: re-read by other units
            uint32_t unit_it = 0, qo = 0;
            bool ok = true;
            for (int n = 0; ok; ++n, ++unit_it) {
                int u;
                Unit w;   // w.h: key/value head
                if (!(ok = ring_get(rg, n, abort, u, w)) || u < 0) break;
                if (!(ok = mbar_wait(bar(KV_EMPTY), (unit_it & 1) ^ 1, abort))) break;
                mbar_expect_tx(bar(KV_FULL), 2 * LY::TILE);
                const int krow = w.row0k + w.tile * 128;
#pragma unroll
                for (int kb = 0; kb < LY::KB; ++kb) {
                    tma_load_3d_hint(sbase + LY::K0 + kb * LY::BLK, &tmK, kb * 64, w.h, krow, bar(KV_FULL), pol_stream);
                    tma_load_3d_hint(sbase + LY::V0 + kb * LY::BLK, &tmV, kb * 64, w.h, krow, bar(KV_FULL), pol_stream);
                }
                kv_issued = unit_it + 1;
                const int nq = w.hi - w.lo;
                for (int sq = 0; sq < grp * nq && ok; ++sq, ++qo) {   // every q tile of every query head
                    const int i = w.lo + sq % nq, hq = w.h * grp + sq / nq;
                    const int s = qo % kQStages;
                    if (!(ok = mbar_wait(bar(QO_EMPTY + s), ((qo / kQStages) & 1) ^ 1, abort))) break;
                    mbar_expect_tx(bar(QO_FULL + s), 2 * LY::TILE);
                    const int qrow = w.row0 + i * BQ;
#pragma unroll
                    for (int kb = 0; kb < LY::KB; ++kb) {
                        tma_load_3d_hint(sbase + LY::Q0 + s * LY::TILE + kb * LY::BLK, &tmQ, kb * 64, hq,
                                         qrow, bar(QO_FULL + s), pol_keep);
                        tma_load_3d_hint(sbase + LY::DO0 + s * LY::TILE + kb * LY::BLK, &tmDO, kb * 64, hq,
                                         qrow, bar(QO_FULL + s), pol_keep);
                    }
                    q_issued = qo + 1;
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        setmaxnreg_dec<kCtrlRegs>();
        {   // ---------------------------------------- MMA issuer (converged warp, one elected lane issues)
            constexpr uint32_t IDESC_ST = idesc_bf16_f32(128, BQ, false);
            constexpr uint32_t IDESC_ACC = idesc_bf16_f32(128, D, true);
            uint32_t unit_it = 0, st = 0;
            bool ok = true;
            auto commit = [&](uint32_t b) {
                if (elect_one()) mma_commit(b);
                __syncwarp();
            };
            const uint64_t kd0 = smem_desc_sw128(sbase + LY::K0, 16, 1024);
            const uint64_t vd0 = smem_desc_sw128(sbase + LY::V0, 16, 1024);
            // S^T = K'Q'(step)^T into columns 0..127 (read by dV of the previous step,
            // issued earlier); dP^T = V dO(step)^T into 128..255 (read by dK before).
            auto issue_st = [&](uint32_t sp) -> bool {
                const int s = sp % kQStages;
                if (!wait_warp(bar(QO_FULL + s), (sp / kQStages) & 1, abort)) return false;
                tc_fence_after();
                const uint64_t qd = smem_desc_sw128(sbase + LY::Q0 + s * LY::TILE, 16, 1024);
                if (elect_one()) {
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t off = ((k >> 2) * LY::BLK + (k & 3) * 32) >> 4;
                        mma_bf16_ss(tmem, kd0 + off, qd + off, IDESC_ST, k > 0 ? 1u : 0u);
                    }
                    mma_commit(bar(ST_FULL));
                }
                __syncwarp();
                return true;
            };
            auto issue_dpt = [&](uint32_t sp) {
                const int s = sp % kQStages;
                const uint64_t od = smem_desc_sw128(sbase + LY::DO0 + s * LY::TILE, 16, 1024);
                if (elect_one()) {
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t off = ((k >> 2) * LY::BLK + (k & 3) * 32) >> 4;
                        mma_bf16_ss(tmem + LY::DPT_COL, vd0 + off, od + off, IDESC_ST, k > 0 ? 1u : 0u);
                    }
                    mma_commit(bar(DPT_FULL));
                }
                __syncwarp();
            };
            for (int n = 0; ok; ++n, ++unit_it) {
                int u;
                Unit w;
                if (!(ok = ring_get_warp(rg, n, abort, u, w)) || u < 0) break;
                if (!(ok = wait_warp(bar(KV_FULL), unit_it & 1, abort))) break;
                if (!(ok = issue_st(st))) break;
                issue_dpt(st);
                const int nsteps = grp * (w.hi - w.lo);
                // K and V are read only by S^T and dP^T: once the last step's pair is issued
                // the tiles go back to the producer, which loads the next unit's K/V under the
                // rest of this unit (its last P^T / dS^T, dV and dK MMAs and the epilogue)
                if (nsteps == 1) commit(bar(KV_EMPTY));
                for (int sq = 0; sq < nsteps; ++sq, ++st) {
                    const int s = st % kQStages;
                    const uint64_t qdm = smem_desc_sw128(sbase + LY::Q0 + s * LY::TILE, LY::BLK, 1024);
                    const uint64_t odm = smem_desc_sw128(sbase + LY::DO0 + s * LY::TILE, LY::BLK, 1024);
                    // dV += P^T dO (P^T packed over the S^T columns); the first one overwrites dV,
                    // so the epilogue warps must have read the previous unit's
                    if (sq == 0 && !(ok = wait_warp(bar(DV_EMPTY), (unit_it & 1) ^ 1, abort))) break;
                    if (!(ok = wait_warp(bar(PT_FULL), st & 1, abort))) break;
                    tc_fence_after();
                    if (elect_one()) {
#pragma unroll
                        for (int k = 0; k < BQ / 16; ++k)
                            mma_bf16_ts(tmem + LY::DV_COL, tmem + dq::ds_col(k), odm + ((k * 16 * 128) >> 4),
                                        IDESC_ACC, (sq > 0 || k > 0) ? 1u : 0u);
                    }
                    __syncwarp();
                    // after the unit's last dV MMA the dV epilogue can start under the last dK MMA
                    if (sq + 1 == nsteps) commit(bar(DV_FULL));
                    if (sq + 1 < nsteps && !(ok = issue_st(st + 1))) break;
                    // dK += dS^T Q' (dS^T packed over the dP^T columns)
                    if (sq == 0 && !(ok = wait_warp(bar(ACC_EMPTY), (unit_it & 1) ^ 1, abort))) break;
                    if (!(ok = wait_warp(bar(DST_FULL), st & 1, abort))) break;
                    tc_fence_after();
                    if (elect_one()) {
#pragma unroll
                        for (int k = 0; k < BQ / 16; ++k)
                            mma_bf16_ts(tmem + LY::DK_COL, tmem + LY::DPT_COL + dq::ds_col(k),
                                        qdm + ((k * 16 * 128) >> 4), IDESC_ACC, (sq > 0 || k > 0) ? 1u : 0u);
                        mma_commit(bar(QO_EMPTY + s));
                    }
                    __syncwarp();
                    if (sq + 1 < nsteps) {
                        issue_dpt(st + 1);
                        if (sq + 2 == nsteps) commit(bar(KV_EMPTY));
                    }
                }
                if (!ok) break;
                commit(bar(ACC_FULL));
            }
            commit(bar(DRAIN));
            mbar_wait_limit(bar(DRAIN), 0, kDrainNs);
        }
        __syncwarp();
    } else if (warp == 3) {
        setmaxnreg_dec<kCtrlRegs>();
        // ------------------------------------------------------------ LSE / delta stager
        uint32_t st = 0;
        bool ok = true;
        for (int n = 0; ok; ++n) {
            int u;
            Unit w;
            if (!(ok = ring_get_warp(rg, n, abort, u, w)) || u < 0) break;
            const int nq = w.hi - w.lo;
            for (int sq = 0; sq < grp * nq && ok; ++sq, ++st) {
                const int i = w.lo + sq % nq, hq = w.h * grp + sq / nq;
                const int sl = st % kLsedSlots;
                if (!(ok = wait_warp(bar(LSED_EMPTY + sl), ((st / kLsedSlots) & 1) ^ 1, abort))) break;
                float* dst = lsed + sl * 256;
#pragma unroll
                for (int h4 = 0; h4 < 4; ++h4) {
                    const int q = lane + 32 * h4;
                    const int qq = i * BQ + q;
                    // a column past the segment gets lse2 = +inf: its P^T is exp2(-inf) = 0, so
                    // phase A needs no mask for the segment tail
                    float l2 = INFINITY, dl = 0.f;
                    if (qq < w.L) {
                        const int64_t idx = static_cast<int64_t>(hq) * p.total + w.row0 + qq;
                        l2 = __ldg(p.lse + idx) * kLog2e;
                        dl = __ldg(p.delta + idx);
                    }
                    dst[q] = l2;
                    dst[128 + q] = dl;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(LSED_FULL + sl));
            }
        }
    } else if (warp == 2) {
        setmaxnreg_dec<kCtrlRegs>();
        // ------------------------------------------------------------ unit scheduler (after the
        // TMEM allocation): claims and decodes units ahead of the other roles
        {   // the whole warp: lane 0 claims and publishes, all lanes decode
            auto decode = [&](int u) {
                Unit w = decode_unit_warp<KV>(p.items_k, p.seg_base_k, p.cu, p.rows, p.cu_kv, p.rows_kv, p.nseg, p.Hkv, u);
                if (KV && p.keys_all_visible) w.off = w.Lk;   // the diagonal past the last key: no mask
                return w;
            };
            for (int n = 0;; ++n) {
                int u;
                if (!ring_put_warp(rg, n, p.next_k, nunits, abort, decode, u) || u < 0) break;
            }
        }
        __syncwarp();
    } else if (warp < 12) {
        // ------------------------------------------------------------ P^T, dS^T
        setmaxnreg_inc<kMathRegs>();
        const int g = (warp - 4) >> 2;             // math warpgroup: q columns [64g, 64g + 64)
        const int wq = warp & 3;
        const int r = wq * 32 + lane;              // key row = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const float scale_log2 = p.scale * kLog2e;
        const int c0 = 64 * g;
        uint32_t st = 0;
        bool ok = true;
        for (int n = 0; ok; ++n) {
            int u;
            Unit w;
            if (!(ok = ring_get_warp(rg, n, abort, u, w)) || u < 0) break;
            const int kvpos = w.tile * 128 + r;
            const int nq = w.hi - w.lo;
            for (int sq = 0; sq < grp * nq; ++sq, ++st) {
                const int i = w.lo + sq % nq;
                const int sl = st % kLsedSlots;
                const float* l2s = lsed + sl * 256 + c0;
                const float* dls = lsed + sl * 256 + 128 + c0;
                if (!(ok = wait_warp(bar(LSED_FULL + sl), (st / kLsedSlots) & 1, abort))) break;
                // allowed q columns: kvpos <= i*BQ + col + off (the diagonal; the segment tail
                // comes through lse2 = +inf); only steps whose first column does not see the
                // tile's last key need the mask, and they take a loop of their own
                const bool diag = i * BQ + w.off < w.tile * 128 + 127;
                const int c_lo = kvpos - w.off - i * BQ;
                // ---- phase A: P^T = exp2(s * scale_log2 - lse2) over this group's 64 columns
                if (!(ok = wait_warp(bar(ST_FULL), st & 1, abort))) break;
                tc_fence_after();
                uint32_t pp[32];
                auto phase_a = [&](auto masked) {
                    uint32_t sr0[32], sr1[32];   // both halves in flight before the first wait
                    tmem_ld32(tmem + lane_off + c0, sr0);
                    tmem_ld32(tmem + lane_off + c0 + 32, sr1);
                    tmem_wait_ld();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t* sr = h == 0 ? sr0 : sr1;
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float2 lz = *reinterpret_cast<const float2*>(l2s + 32 * h + e);
                            float2 s = make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1]));
                            if constexpr (decltype(masked)::value) {   // above the diagonal -> -inf
                                const int col = c0 + 32 * h + e;
                                if (col < c_lo) s.x = -INFINITY;
                                if (col + 1 < c_lo) s.y = -INFINITY;
                            }
                            const float2 x = fma2(s, make_float2(scale_log2, scale_log2), make_float2(-lz.x, -lz.y));
                            pp[16 * h + (e >> 1)] = pack_bf16x2(ex2_approx(x.x), ex2_approx(x.y));
                        }
                    }
                };
                if (diag) phase_a(std::true_type{});
                else phase_a(std::false_type{});
                {
                    uint32_t lo[16], hi[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) { lo[e] = pp[e]; hi[e] = pp[16 + e]; }
                    tmem_st16(tmem + lane_off + c0, lo);
                    tmem_st16(tmem + lane_off + c0 + 16, hi);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(PT_FULL));
                // ---- phase B: dS^T = P^T (dP^T - D), packed over the consumed dP^T columns
                if (!(ok = wait_warp(bar(DPT_FULL), st & 1, abort))) break;
                tc_fence_after();
                uint32_t pd[32];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t dr[32];
                    tmem_ld32(tmem + lane_off + LY::DPT_COL + c0 + 32 * h, dr);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float2 dz = *reinterpret_cast<const float2*>(dls + 32 * h + e);
                        const uint32_t pv = pp[16 * h + (e >> 1)];
                        const float2 ds = mul2(make_float2(bf16_lo(pv), bf16_hi(pv)),
                                               make_float2(__uint_as_float(dr[e]) - dz.x,
                                                           __uint_as_float(dr[e + 1]) - dz.y));
                        pd[16 * h + (e >> 1)] = pack_bf16x2(ds.x, ds.y);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(LSED_EMPTY + sl));
                {
                    uint32_t lo[16], hi[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) { lo[e] = pd[e]; hi[e] = pd[16 + e]; }
                    tmem_st16(tmem + lane_off + LY::DPT_COL + c0, lo);
                    tmem_st16(tmem + lane_off + LY::DPT_COL + c0 + 16, hi);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(DST_FULL));
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue: dV, R(p)^T dK
        if constexpr (kEpiRegs > kLaunchRegsKV) setmaxnreg_inc<kEpiRegs>();
        else setmaxnreg_dec<kEpiRegs>();
        const int wq = warp & 3;
        const int r = wq * 32 + lane;              // key row = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const bool v8 = ((reinterpret_cast<uintptr_t>(p.dk) | reinterpret_cast<uintptr_t>(p.dv)) & 31) == 0;
        uint32_t unit_it = 0;
        bool ok = true;
        for (int n = 0; ok; ++n, ++unit_it) {
            int u;
            Unit w;
            if (!(ok = ring_get_warp(rg, n, abort, u, w)) || u < 0) break;
            const int kvpos = w.tile * 128 + r;
            if (!(ok = wait_warp(bar(DV_FULL), unit_it & 1, abort))) break;
            tc_fence_after();
            const bool valid = kvpos < w.Lk;
            const int64_t tok = static_cast<int64_t>(w.row0k) + (valid ? kvpos : 0);
            const int64_t roff = (tok * p.Hkv + w.h) * static_cast<int64_t>(D) * 2;
            // dV: the whole row packed to bf16 first, so its columns go back to the MMA warp
            // before the stores
            uint32_t pv[D / 2];
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t rr[32];
                tmem_ld32(tmem + lane_off + LY::DV_COL + c * 32, rr);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    pv[16 * c + e] = pack_bf16x2(__uint_as_float(rr[2 * e]), __uint_as_float(rr[2 * e + 1]));
            }
            tc_fence_before();
            mbar_arrive(bar(DV_EMPTY));
            if (valid) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c)
                    st_row64(reinterpret_cast<uint8_t*>(p.dv) + roff + c * 64, pv + 16 * c, v8);
            }
            // dK: scale and R(p)^T over all of the row's rotation pairs
            if (!(ok = wait_warp(bar(ACC_FULL), unit_it & 1, abort))) break;
            tc_fence_after();
            {
                uint8_t* row_out = reinterpret_cast<uint8_t*>(p.dk) + roff;
#pragma unroll 1
                for (int part = 0; part < 2; ++part) {
                    if (p.use_rope == kRopeInterleaved)
                        store_unrotated<D, true>(tmem + lane_off + LY::DK_COL, p.table2, p.table_rows, kvpos,
                                                 p.scale, true, valid, row_out, v8, part);
                    else
                        store_unrotated<D, false>(tmem + lane_off + LY::DK_COL, p.table2, p.table_rows, kvpos,
                                                  p.scale, p.use_rope != 0, valid, row_out, v8, part);
                }
            }
            tc_fence_before();
            mbar_arrive(bar(ACC_EMPTY));
        }
    }

    __syncthreads();
    if (*abort) {
        if (warp == 0 && lane == 0) {
            if (kv_issued > 0) mbar_wait_limit(bar(KV_FULL), (kv_issued - 1) & 1, kDrainNs);
            for (int s2 = 0; s2 < kQStages; ++s2)
                if (q_issued > static_cast<uint32_t>(s2)) {
                    const uint32_t nn = q_issued - 1 - ((q_issued - 1 - s2) % kQStages);
                    mbar_wait_limit(bar(QO_FULL + s2), (nn / kQStages) & 1, kDrainNs);
                }
        }
        if (threadIdx.x == 0) atomicOr(p.err, VLC_DEVERR_TIMEOUT);
        __syncthreads();
    }
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace dkdv
}  // namespace bwd

template <int D>
static cudaError_t launch_bwd_d(const BwdParams& p, int num_sms, cudaStream_t s) {
    {
        const bool sep = p.cu_kv != p.cu;   // keys with segments of their own
        const int rot = p.operands_rotated ? kRopeNone : p.use_rope;   // rotation in this pass
        const int64_t rows = static_cast<int64_t>(p.total) * p.H +
                             (sep && rot ? static_cast<int64_t>(p.total_kv) * p.Hkv : 0);
        int64_t blocks = (rows * (D / 16) + 255) / 256;
        if (blocks > static_cast<int64_t>(num_sms) * 8) blocks = static_cast<int64_t>(num_sms) * 8;
        auto prep = sep ? bwd::prep_kernel<D, true> : bwd::prep_kernel<D, false>;
        prep<<<static_cast<int>(blocks), 256, 0, s>>>(
            static_cast<const uint4*>(p.dout), static_cast<const uint4*>(p.o),
            static_cast<const uint4*>(p.q), static_cast<const uint4*>(p.k), static_cast<uint4*>(p.qrot),
            static_cast<uint4*>(p.krot), p.delta, p.cu, p.rows, p.cu_kv, p.rows_kv, p.nseg, p.table, p.total, p.H,
            p.Hkv, p.total_kv, rot, p.err);
    }
    // with RoPE the attention passes read the rotated copies
    const bool rotated_here = p.use_rope && !p.operands_rotated;
    const void* qop = rotated_here ? p.qrot : p.q;
    const void* kop = rotated_here ? p.krot : p.k;
    CUtensorMap q128, do128, k128, v128;
    if (!make_tmap_thd(&q128, qop, p.total, p.H, D, 128) ||
        !make_tmap_thd(&do128, p.dout, p.total, p.H, D, 128) ||
        !make_tmap_thd(&k128, kop, p.total_kv, p.Hkv, D, 128) ||
        !make_tmap_thd(&v128, p.v, p.total_kv, p.Hkv, D, 128))
        return cudaErrorInvalidValue;
    const bool kv = p.cu_kv != p.cu || p.keys_all_visible;   // the instance that reads the unit's offset
    {
        constexpr uint32_t smem = bwd::dq::Layout<D>::ALLOC;
        auto kernel = kv ? bwd::dq::dq_kernel<D, true> : bwd::dq::dq_kernel<D, false>;
        // the warp roles re-split the register pool: valid only at the launch count it assumes
        cudaFuncAttributes fa{};
        cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != static_cast<int>(bwd::dq::kLaunchRegsQ)) return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        kernel<<<num_sms, bwd::kThreads, smem, s>>>(q128, do128, k128, v128, p);
    }
    {
        constexpr uint32_t smem = bwd::dkdv::Layout<D>::ALLOC;
        auto kernel = kv ? bwd::dkdv::dkdv_kernel<D, true> : bwd::dkdv::dkdv_kernel<D, false>;
        // the warp roles re-split the register pool: valid only at the launch count it assumes
        cudaFuncAttributes fa{};
        cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != static_cast<int>(bwd::dkdv::kLaunchRegsKV)) return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        kernel<<<num_sms, bwd::dkdv::kThreadsKV, smem, s>>>(q128, do128, k128, v128, p);
    }
    return cudaGetLastError();
}

cudaError_t launch_attn_bwd(const BwdParams& p, int num_sms, cudaStream_t s) {
    return p.d == 128 ? launch_bwd_d<128>(p, num_sms, s) : launch_bwd_d<64>(p, num_sms, s);
}

}  // namespace vlc
