// attn_fwd.cu -- varlen block-diagonal causal attention, forward, sm_103a.
//
// What it computes ("Sequence packing and variable-length attention",
// charlestar, section "EOS is content; isolation happens before softmax"):
// for every segment r and head h, O = softmax(Q'K'^T * scale + M) V with
// M = -inf where key position > query position, over that segment only; Q', K'
// are q, k rotated by RoPE at the per-segment positions p = i - cu_r
// (section "Positions are reset per segment").  LSE = ln sum exp(scores).
//
// Design (one persistent CTA per SM, 384 threads, warp-specialised):
//   warp 0      TMA producer: Q tile (128 rows) per work unit, K/V tiles
//               (128 rows) per key tile, 128-byte swizzle, 2 stages each.
//   warp 1      MMA issuer (one thread): S = Q'K'^T into TMEM (double buffer),
//               O += P V into TMEM (tcgen05.mma kind::f16, fp32 accumulate).
//   warp 2      TMEM allocator (512 columns).
//   warps 4-7   softmax + epilogue: one thread per query row (= TMEM lane):
//               fp32 online softmax in the exp2 domain, the causal / segment-
//               tail mask only on the last key tile of an item, P (bf16) to
//               shared memory, lazy O rescale, final O / l and LSE.
//   warps 8-11  RoPE: rotate the staged Q and K tiles in shared memory at the
//               segment-local positions, round to bf16, hand them to the MMA.
// A work unit is one (work item, head) pair; the work list (built on the
// device beforehand) only holds in-segment, at-or-below-diagonal tiles.
// Every wait is bounded; on expiry the kernel sets VLC_DEVERR_TIMEOUT, drains
// its own in-flight copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cmath>
#include <cstdint>

#include "../../include/vlc.h"
#include "attn_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace vlc {
namespace fwd {

constexpr int BM = kFwdBM;
constexpr int BN = kFwdBN;
static_assert(BM == 128 && BN == 128, "tile shape fixed by the TMEM lane mapping");
constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;   // log2 units: rescale O only when max grows > 2^8
constexpr float kLn2 = 0.69314718055994530942f;

// barrier slots
enum : int {
    Q_FULL = 0, Q_READY = 2, Q_EMPTY = 4,
    K_FULL = 6, K_READY = 8, K_EMPTY = 10,
    V_FULL = 12, V_EMPTY = 14,
    S_FULL = 16, S_EMPTY = 18,
    P_FULL = 20, PV_DONE = 21, O_EMPTY = 22, DRAIN = 23,
    NUM_BARS = 24
};

template <int D>
struct Layout {
    static constexpr int KB = D / 64;                  // 64-column (128-byte) blocks per row
    static constexpr uint32_t BLK = 128u * 128u;       // one block of 128 rows: 16 KB
    static constexpr uint32_t TILE = 128u * D * 2u;    // a Q/K/V tile
    static constexpr uint32_t Q0 = 0;
    static constexpr uint32_t K0 = Q0 + 2 * TILE;
    static constexpr uint32_t V0 = K0 + 2 * TILE;
    static constexpr uint32_t P0 = V0 + 2 * TILE;
    static constexpr uint32_t PBYTES = 128u * BN * 2u;
    static constexpr uint32_t BAR0 = P0 + PBYTES;
    static constexpr uint32_t MISC = BAR0 + NUM_BARS * 8;
    static constexpr uint32_t BYTES = MISC + 16;
    static constexpr uint32_t ALLOC = BYTES + 1024;    // room to align the base to 1024
    static constexpr uint32_t S_COL = 0;               // S buffers at columns 0 and 128
    static constexpr uint32_t O_COL = 256;             // O at columns 256 .. 256+D
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
    using LY = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (sbase - smem_u32(smem_raw));
    auto bar = [&](int i) -> uint32_t { return sbase + LY::BAR0 + 8u * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sgen + LY::MISC);
    volatile int* abort = reinterpret_cast<volatile int*>(sgen + LY::MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    __shared__ int s_skip, s_nunits;
    if (threadIdx.x == 0) {   // one read, so every thread takes the same branch
        s_skip = *reinterpret_cast<volatile int32_t*>(p.err);
        s_nunits = *reinterpret_cast<const volatile int32_t*>(p.count) * p.H;
    }
    __syncthreads();
    if (s_skip != 0) return;   // invalid cu_seqlens: the whole call is a no-op
    const int nunits = s_nunits;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(Q_FULL + i), 1);
            mbar_init(bar(Q_READY + i), 128);
            mbar_init(bar(Q_EMPTY + i), 1);
            mbar_init(bar(K_FULL + i), 1);
            mbar_init(bar(K_READY + i), 128);
            mbar_init(bar(K_EMPTY + i), 1);
            mbar_init(bar(V_FULL + i), 1);
            mbar_init(bar(V_EMPTY + i), 1);
            mbar_init(bar(S_FULL + i), 1);
            mbar_init(bar(S_EMPTY + i), 128);
        }
        mbar_init(bar(P_FULL), 128);
        mbar_init(bar(PV_DONE), 1);
        mbar_init(bar(O_EMPTY), 128);
        mbar_init(bar(DRAIN), 1);
        *abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // per-role counters kept for the teardown drain
    uint32_t q_issued = 0, kv_issued = 0;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t q_it = 0, kv_it = 0;
            for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
                const Unit w = decode_unit(p.items, p.seg_base, p.cu, p.nseg, p.H, u);
                const int qs = q_it & 1;
                if (!mbar_wait(bar(Q_EMPTY + qs), ((q_it >> 1) & 1) ^ 1, abort)) break;
                mbar_expect_tx(bar(Q_FULL + qs), LY::TILE);
                const uint32_t qdst = sbase + LY::Q0 + qs * LY::TILE;
#pragma unroll
                for (int kb = 0; kb < LY::KB; ++kb)
                    tma_load_3d(qdst + kb * LY::BLK, &tmQ, kb * 64, w.h, w.row0 + w.tile * BM,
                                bar(Q_FULL + qs));
                q_issued = ++q_it;
                bool ok = true;
                for (int j = 0; j < w.hi && ok; ++j) {
                    const int ks = kv_it & 1;
                    const uint32_t ph = ((kv_it >> 1) & 1) ^ 1;
                    const int row = w.row0 + j * BN;
                    if (!(ok = mbar_wait(bar(K_EMPTY + ks), ph, abort))) break;
                    mbar_expect_tx(bar(K_FULL + ks), LY::TILE);
#pragma unroll
                    for (int kb = 0; kb < LY::KB; ++kb)
                        tma_load_3d(sbase + LY::K0 + ks * LY::TILE + kb * LY::BLK, &tmK, kb * 64,
                                    w.h, row, bar(K_FULL + ks));
                    if (!(ok = mbar_wait(bar(V_EMPTY + ks), ph, abort))) {
                        kv_issued = kv_it + 1;   // the K half of this stage is in flight
                        break;
                    }
                    mbar_expect_tx(bar(V_FULL + ks), LY::TILE);
#pragma unroll
                    for (int kb = 0; kb < LY::KB; ++kb)
                        tma_load_3d(sbase + LY::V0 + ks * LY::TILE + kb * LY::BLK, &tmV, kb * 64,
                                    w.h, row, bar(V_FULL + ks));
                    kv_issued = ++kv_it;
                }
                if (!ok) break;
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_bf16_f32(128, BN, false);
            constexpr uint32_t IDESC_O = idesc_bf16_f32(128, D, true);
            uint32_t q_it = 0, kv_it = 0, s_it = 0, pv_it = 0, unit_it = 0;
            bool ok = true;
            auto issue_pv = [&](bool first) -> bool {
                const int vs = pv_it & 1;
                if (first && !mbar_wait(bar(O_EMPTY), (unit_it & 1) ^ 1, abort)) return false;
                if (!mbar_wait(bar(V_FULL + vs), (pv_it >> 1) & 1, abort)) return false;
                if (!mbar_wait(bar(P_FULL), pv_it & 1, abort)) return false;
                tc_fence_after();
                const uint32_t vbase = sbase + LY::V0 + vs * LY::TILE;
                const uint32_t pbase = sbase + LY::P0;
#pragma unroll
                for (int k = 0; k < BN / 16; ++k) {
                    const uint64_t a = smem_desc_sw128(pbase + (k >> 2) * LY::BLK + (k & 3) * 32, 16, 1024);
                    const uint64_t b = smem_desc_sw128(vbase + k * 16 * 128, LY::BLK, 1024);
                    mma_bf16_ss(tmem + LY::O_COL, a, b, IDESC_O, (!first || k > 0) ? 1u : 0u);
                }
                mma_commit(bar(PV_DONE));
                mma_commit(bar(V_EMPTY + vs));
                ++pv_it;
                return true;
            };
            for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
                const Unit w = decode_unit(p.items, p.seg_base, p.cu, p.nseg, p.H, u);
                const int qs = q_it & 1;
                if (!(ok = mbar_wait(bar(Q_READY + qs), (q_it >> 1) & 1, abort))) break;
                const uint32_t qbase = sbase + LY::Q0 + qs * LY::TILE;
                for (int j = 0; j < w.hi; ++j) {
                    const int ks = kv_it & 1;
                    if (!(ok = mbar_wait(bar(K_READY + ks), (kv_it >> 1) & 1, abort))) break;
                    const int sb = s_it & 1;
                    if (!(ok = mbar_wait(bar(S_EMPTY + sb), ((s_it >> 1) & 1) ^ 1, abort))) break;
                    tc_fence_after();
                    const uint32_t kbase = sbase + LY::K0 + ks * LY::TILE;
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t off = (k >> 2) * LY::BLK + (k & 3) * 32;
                        mma_bf16_ss(tmem + LY::S_COL + sb * 128,
                                    smem_desc_sw128(qbase + off, 16, 1024),
                                    smem_desc_sw128(kbase + off, 16, 1024), IDESC_S,
                                    k > 0 ? 1u : 0u);
                    }
                    mma_commit(bar(S_FULL + sb));
                    mma_commit(bar(K_EMPTY + ks));
                    if (j == w.hi - 1) mma_commit(bar(Q_EMPTY + qs));
                    ++s_it;
                    ++kv_it;
                    if (j > 0 && !(ok = issue_pv(j == 1))) break;
                }
                if (!ok) break;
                if (!(ok = issue_pv(w.hi == 1))) break;
                ++q_it;
                ++unit_it;
            }
            // let every issued MMA finish before TMEM can be released
            mma_commit(bar(DRAIN));
            mbar_wait_limit(bar(DRAIN), 0, 200000000ull);
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ softmax + epilogue
        const int wq = warp - 4;
        const int r = wq * 32 + lane;                  // query row in the tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t sP = sbase + LY::P0;
        uint32_t s_it = 0, pv_it = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
            const Unit w = decode_unit(p.items, p.seg_base, p.cu, p.nseg, p.H, u);
            const int qpos = w.tile * BM + r;
            float m_run = 0.f, l_run = 0.f;
            for (int j = 0; j < w.hi; ++j) {
                const int sb = s_it & 1;
                if (!(ok = wait_warp(bar(S_FULL + sb), (s_it >> 1) & 1, abort))) break;
                tc_fence_after();
                float x[BN];
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t rr[32];
                    tmem_ld32(tmem + lane_off + LY::S_COL + sb * 128 + c * 32, rr);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[c * 32 + e] = __uint_as_float(rr[e]);
                }
                tc_fence_before();
                mbar_arrive(bar(S_EMPTY + sb));
                ++s_it;

                // scale to the log2 domain; mask only on the last (diagonal / tail) tile
                // raw scores; the mask only on the last (diagonal / tail) tile.  The max of
                // the raw scores times scale_log2 (> 0) is the max in the log2 domain.
                float mt = -INFINITY;
                if (j == w.hi - 1) {
                    const int lim = min(qpos, w.L - 1) - j * BN;   // allowed key columns: c <= lim
#pragma unroll
                    for (int c = 0; c < BN; ++c) {
                        x[c] = (c <= lim) ? x[c] : -INFINITY;
                        mt = fmaxf(mt, x[c]);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < BN; ++c) mt = fmaxf(mt, x[c]);
                }
                mt *= p.scale_log2;
                float m_use = m_run, alpha = 1.f;
                bool rescale = false;
                if (j == 0) {
                    m_use = mt;
                } else {
                    const bool need = mt > m_run + kRescaleThreshold;
                    rescale = __any_sync(0xffffffffu, need);
                    if (rescale) {
                        m_use = fmaxf(m_run, mt);
                        alpha = ex2_approx(m_run - m_use);
                    }
                }
                float rs = 0.f;
                uint32_t pk[BN / 2];
#pragma unroll
                for (int c = 0; c < BN / 2; ++c) {
                    const float p0 = ex2_approx(fmaf(x[2 * c], p.scale_log2, -m_use));
                    const float p1 = ex2_approx(fmaf(x[2 * c + 1], p.scale_log2, -m_use));
                    rs += p0 + p1;
                    pk[c] = pack_bf16x2(p0, p1);
                }
                // previous P·V must be done: frees the P buffer and makes O stable
                if (pv_it > 0 && !(ok = wait_warp(bar(PV_DONE), (pv_it - 1) & 1, abort))) break;
                if (rescale) {
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t rr[32];
                        const uint32_t ta = tmem + lane_off + LY::O_COL + c * 32;
                        tmem_ld32(ta, rr);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
                        tmem_st32(ta, rr);
                    }
                    tmem_wait_st();
                    l_run *= alpha;
                }
                l_run += rs;
                m_run = m_use;
#pragma unroll
                for (int ci = 0; ci < BN / 8; ++ci) {
                    const uint32_t addr = sw128(sP + (ci >> 3) * LY::BLK, r, ci & 7);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                                 ::"r"(addr), "r"(pk[4 * ci]), "r"(pk[4 * ci + 1]),
                                 "r"(pk[4 * ci + 2]), "r"(pk[4 * ci + 3]) : "memory");
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(bar(P_FULL));
                ++pv_it;
            }
            if (!ok) break;
            // ---- epilogue: O / l -> bf16, LSE
            if (!(ok = wait_warp(bar(PV_DONE), (pv_it - 1) & 1, abort))) break;
            tc_fence_after();
            const bool valid = qpos < w.L;
            const int64_t tok = static_cast<int64_t>(w.row0) + qpos;
            const float inv_l = 1.f / l_run;
            uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) +
                            ((valid ? tok : 0) * p.H + w.h) * static_cast<int64_t>(D) * 2;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t rr[32];
                tmem_ld32(tmem + lane_off + LY::O_COL + c * 32, rr);
                tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    pk[e] = pack_bf16x2(__uint_as_float(rr[2 * e]) * inv_l,
                                        __uint_as_float(rr[2 * e + 1]) * inv_l);
                if (valid) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + c * 64);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                }
            }
            if (valid) p.lse[static_cast<int64_t>(w.h) * p.total + tok] = (m_run + __log2f(l_run)) * kLn2;
            tc_fence_before();
            mbar_arrive(bar(O_EMPTY));
        }
    } else if (warp >= 8) {
        // ------------------------------------------------------------ RoPE on staged Q/K
        const int wr = warp - 8;
        RopeStep<D> step{};
        if (p.use_rope) step = rope_step<D>(p.table, lane);
        uint32_t q_it = 0, kv_it = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
            const Unit w = decode_unit(p.items, p.seg_base, p.cu, p.nseg, p.H, u);
            const int qs = q_it & 1;
            if (!(ok = wait_warp(bar(Q_FULL + qs), (q_it >> 1) & 1, abort))) break;
            if (p.use_rope) rope_tile<D, 128>(sbase + LY::Q0 + qs * LY::TILE, w.tile * BM, p.table, step, wr, lane);
            fence_proxy_async_smem();
            mbar_arrive(bar(Q_READY + qs));
            ++q_it;
            for (int j = 0; j < w.hi; ++j) {
                const int ks = kv_it & 1;
                if (!(ok = wait_warp(bar(K_FULL + ks), (kv_it >> 1) & 1, abort))) break;
                if (p.use_rope) rope_tile<D, 128>(sbase + LY::K0 + ks * LY::TILE, j * BN, p.table, step, wr, lane);
                fence_proxy_async_smem();
                mbar_arrive(bar(K_READY + ks));
                ++kv_it;
            }
        }
    }

    __syncthreads();
    if (*abort) {
        if (warp == 0 && lane == 0) {
            // wait (bounded) for the last copy issued on every stage
            for (int s = 0; s < 2; ++s) {
                if (q_issued > static_cast<uint32_t>(s)) {
                    const uint32_t n = ((q_issued - 1 - s) & ~1u) + s;
                    mbar_wait_limit(bar(Q_FULL + s), (n >> 1) & 1, 200000000ull);
                }
                if (kv_issued > static_cast<uint32_t>(s)) {
                    const uint32_t n = ((kv_issued - 1 - s) & ~1u) + s;
                    mbar_wait_limit(bar(K_FULL + s), (n >> 1) & 1, 200000000ull);
                    mbar_wait_limit(bar(V_FULL + s), (n >> 1) & 1, 200000000ull);
                }
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

}  // namespace fwd

// Encode a [total, H, d] bf16 tensor as a 3-D TMA map with 64 x 1 x 128 boxes.
bool make_tmap_thd(CUtensorMap* map, const void* base, int32_t total, int32_t H, int32_t d,
                   int box_rows);

cudaError_t launch_attn_fwd(const FwdParams& p, int num_sms, cudaStream_t s) {
    CUtensorMap tq, tk, tv;
    if (!make_tmap_thd(&tq, p.q, p.total, p.H, p.d, 128) ||
        !make_tmap_thd(&tk, p.k, p.total, p.H, p.d, 128) ||
        !make_tmap_thd(&tv, p.v, p.total, p.H, p.d, 128))
        return cudaErrorInvalidValue;
    const dim3 grid(num_sms), block(fwd::kThreads);
    if (p.d == 128) {
        constexpr uint32_t smem = fwd::Layout<128>::ALLOC;
        cudaError_t e = cudaFuncSetAttribute(fwd::attn_fwd_kernel<128>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        fwd::attn_fwd_kernel<128><<<grid, block, smem, s>>>(tq, tk, tv, p);
    } else {
        constexpr uint32_t smem = fwd::Layout<64>::ALLOC;
        cudaError_t e = cudaFuncSetAttribute(fwd::attn_fwd_kernel<64>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        fwd::attn_fwd_kernel<64><<<grid, block, smem, s>>>(tq, tk, tv, p);
    }
    return cudaGetLastError();
}

}  // namespace vlc
