// attn_fwd.cu -- varlen block-diagonal causal attention, forward, sm_103a.
//
// What it computes ("Sequence packing and variable-length attention",
// charlestar, section "EOS is content; isolation happens before softmax"):
// for every segment r and head h, O = softmax(Q'K'^T * scale + M) V with
// M = -inf where key position > query position, over that segment only; Q', K'
// are q, k rotated by RoPE at the per-segment positions p = i - cu_r
// (section "Positions are reset per segment").  LSE = ln sum exp(scores).
//
// Design: one persistent CTA per SM, warp-specialised (640 threads; 512 in the
// fallback instance with RoPE warps).  A work unit is (segment, head, block of 256 query
// rows) = two 128-row q tiles that share every K/V tile; the work list holds only
// in-segment, at-or-below-diagonal key tiles, and a q tile stops at its own
// diagonal key tile.  Units are claimed dynamically (longest first) from a global
// counter by a scheduler warp, which decodes each one and hands it to every role
// through a shared-memory ring.
//   warp 0       TMA producer of q tiles (3-slot ring) and K tiles (2 stages),
//                128-byte swizzle; warp 3 the same for V tiles (2 stages).
//   warp 1       MMA issuer (one elected lane of the converged warp), tcgen05.mma
//                kind::f16, fp32 accumulators in TMEM:
//                S_t = Q'_t K'^T (shared-memory operands) and O_t += P_t V with
//                P_t read from TMEM; issue order S0 S1 | PV0(j) S0(j+1)
//                PV1(j) S1(j+1) | ..., so each q tile's softmax overlaps the
//                other tile's MMAs.
//   warp 2       TMEM allocator (512 columns: S/P 0, S/P 1, O 0, O 1), then the
//                unit scheduler.
//   warps 4-11   softmax + epilogue of q tile 0; warps 12-19 the same for q tile 1.
//                A query row (TMEM lane) belongs to two threads of one warp, 64 score
//                columns each (the 16x32bx2 TMEM access shape), so a softmax step per
//                thread is half a row: its maximum comes with the TMEM load (ld.red)
//                and meets the other half's in one shuffle; exp2 and bf16 P written
//                back over the consumed S columns; the causal / segment-tail mask only
//                on a tile's last key tile; lazy O rescale when the row max grows by
//                more than 2^8; epilogue O / l -> bf16 and LSE, half a row per thread.
//   RoPE (segment-local positions): k is rotated once beforehand into the workspace
//                (the k half of the rotation pass) and the warps of q tile 0, which end each
//                unit one key tile ahead of tile 1's, rotate the next unit's two staged q
//                tiles in shared memory before their epilogue.  Without room in the
//                workspace for the rotated k, a fallback instance rotates every staged q
//                and K tile in a RoPE warpgroup (warps 12-15; its softmax warps 4-7 and
//                8-11 hold one query row per thread, 128 scores each: there are no
//                registers left for split rows).
// Every wait is bounded; on expiry the kernel sets VLC_DEVERR_TIMEOUT, drains
// its own in-flight copies and MMAs, frees TMEM and returns.
#include <type_traits>
#include <cuda.h>
#include <cmath>
#include <cstdint>

#include "../../include/vlc.h"
#include "attn_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace vlc {
namespace fwd {

constexpr int BQ = 128;                 // rows per q tile
constexpr int QB = kFwdQB;              // rows per work unit (two q tiles)
constexpr int BN = kFwdBN;              // rows per key tile
static_assert(QB == 2 * BQ && BN == 128, "two 128-row q tiles per unit, 128-row key tiles");
constexpr int kQSlots = 3;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
// Kernel instances by where q and K tiles are rotated:
//   kModePlain  no RoPE, or q, k rotated beforehand (vlc_rope_qk);
//   kModeWarps  a RoPE warpgroup rotates every staged q and K tile (the fallback when the
//               workspace has no room for a rotated copy of k);
//   kModeQRot   k rotated once beforehand into the workspace for every segment, and the
//               q tiles rotated in shared memory by the softmax warps of q tile 0 while
//               they finish the unit before (they end it one key tile ahead of tile 1's).
enum : int { kModePlain = 0, kModeWarps = 1, kModeQRot = 2 };

// Threads: a control warpgroup (producers, MMA issuer, scheduler) and the softmax
// warpgroups; the warpgroups re-split the launch's register pool with setmaxnreg.
//   without RoPE warps: four softmax warpgroups, two per q tile (the two threads of a
//     query row sit in one warp and take 64 score columns each);
//   with RoPE warps: two softmax warpgroups, one thread per query row holding its
//     128 scores, and a RoPE warpgroup (no register room for the split rows).
template <int MODE>
struct Cfg {
    static constexpr bool kWarps = MODE == kModeWarps;
    static constexpr int kSoftWarps = kWarps ? 8 : 16;
    static constexpr int kThreads = 32 * (4 + kSoftWarps + (kWarps ? 4 : 0));   // 512 or 640
    static constexpr uint32_t kLaunchRegs = 65536u / kThreads / 8u * 8u;        // registers per thread at launch
    static constexpr uint32_t kCtrlRegs = kWarps ? 72u : 56u;
    static constexpr uint32_t kRopeRegs = kWarps ? 88u : 0u;
    static constexpr uint32_t kSoftRegs =
        (kThreads * kLaunchRegs - 128u * kCtrlRegs - 128u * kRopeRegs) / (32u * kSoftWarps) / 8u * 8u;
    static_assert(128u * kCtrlRegs + 128u * kRopeRegs + 32u * kSoftWarps * kSoftRegs <= kThreads * kLaunchRegs,
                  "register split exceeds the pool");
    static constexpr uint32_t kTileThreads = 32u * kSoftWarps / 2;   // softmax threads of one q tile
    // threads that rotate a staged q tile and arrive on its Q_READY barrier (a warpgroup)
    static constexpr uint32_t kQReadyCount = 128u;
};
constexpr float kLn2 = 0.69314718055994530942f;

enum : int {
    Q_FULL = 0, Q_READY = 3, Q_EMPTY = 6,
    K_FULL = 9, K_READY = 11, K_EMPTY = 13, V_FULL = 15, V_EMPTY = 17,
    S_FULL = 19, P_FULL = 21, O_FULL = 23, O_EMPTY = 25,
    DRAIN = 27, UNIT_FULL = 28, UNIT_EMPTY = 28 + kRing, NUM_BARS = 28 + 2 * kRing
};

template <int D>
struct Layout {
    static constexpr int KB = D / 64;
    static constexpr uint32_t BLK = 128u * 128u;       // 128 rows x 128 bytes
    static constexpr uint32_t TILE = 128u * D * 2u;
    static constexpr uint32_t Q0 = 0;                  // kQSlots tiles
    static constexpr uint32_t K0 = kQSlots * TILE;     // 2 stages
    static constexpr uint32_t V0 = K0 + 2 * TILE;      // 2 stages
    static constexpr uint32_t BAR0 = V0 + 2 * TILE;
    static constexpr uint32_t MISC = BAR0 + NUM_BARS * 8;   // tmem slot, abort flag, wait limit, unit ring
    static constexpr uint32_t RING = (MISC + 16 + 15) / 16 * 16;   // 16-byte aligned slots
    static constexpr uint32_t BYTES = RING + 4 * kSlotInts * kRing;
    static constexpr uint32_t ALLOC = BYTES + 1024;
    __host__ __device__ static constexpr uint32_t S_COL(int t) { return 128u * t; }   // P_t shares these columns
    __host__ __device__ static constexpr uint32_t O_COL(int t) { return 256u + 128u * t; }
};

// One work unit pairs two adjacent 128-row q tiles of a segment that share every
// K/V tile.  With T = ceil(L / 128) q tiles, unit qb holds tiles (2qb - s, 2qb - s + 1)
// where s = T mod 2, so an odd T leaves tile 0 alone in unit 0 (one key tile of work)
// rather than the last, longest tile.  Slot t of the unit is q tile q0 + t and needs
// the key tiles up to the one holding key (q0 + t + 1) * 128 - 1 + off (its diagonal;
// off = Lk - L is 0 for self-attention, where that is [0, q0 + t + 1)); nk is the
// length of the K/V stream.
struct FUnit {
    Unit w;
    bool has1;
    bool pre;   // K tiles come rotated from p.krot, not rotated in-kernel
    int q0, n0, n1, nk;
    int hkv;   // key/value head of query head w.h
};

template <bool KV>
__device__ __forceinline__ FUnit make_funit(const FwdParams& p, const Unit& w) {
    FUnit f;
    f.w = w;
    const int T = (f.w.L + BQ - 1) / BQ;
    const int s = T & 1;
    const bool lone = (s != 0) && (f.w.tile == 0);
    f.has1 = !lone;
    f.q0 = lone ? 0 : 2 * f.w.tile - s;
    if constexpr (KV) {
        const int nkt = (f.w.Lk + BN - 1) / BN;
        f.n0 = min(nkt, ((f.q0 + 1) * BQ + f.w.off + BN - 1) / BN);
        f.n1 = f.has1 ? min(nkt, ((f.q0 + 2) * BQ + f.w.off + BN - 1) / BN) : 0;
    } else {
        f.n0 = f.q0 + 1;
        f.n1 = f.has1 ? f.q0 + 2 : 0;
    }
    f.nk = f.has1 ? f.n1 : f.n0;
    f.pre = p.krot != nullptr;
    f.hkv = p.Hkv == p.H ? f.w.h : f.w.h / (p.H / p.Hkv);
    return f;
}

// KV: keys and values have segments of their own (bottom-right aligned queries).
template <int D, bool KV, int MODE>
__global__ void __launch_bounds__(Cfg<MODE>::kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmKr,
                const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
    using LY = Layout<D>;
    using CF = Cfg<MODE>;
    constexpr bool ROPE = MODE == kModeWarps;     // the RoPE-warp instance (one thread per row)
    constexpr bool ROTQ = MODE == kModeQRot;      // softmax warps rotate the q tiles
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (sbase - smem_u32(smem_raw));
    auto bar = [&](int i) -> uint32_t { return sbase + LY::BAR0 + 8u * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sgen + LY::MISC);
    volatile int* abort = reinterpret_cast<volatile int*>(sgen + LY::MISC + 4);   // [abort flag, wait limit in us]
    const Ring rg{reinterpret_cast<volatile int*>(sgen + LY::RING), bar(UNIT_FULL), bar(UNIT_EMPTY)};
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Q/K and V producers, MMA warp, the softmax warps, and the 4 RoPE warps when they rotate
    constexpr int kRingConsumers = 1 + 1 + 1 + CF::kSoftWarps + 4;

    __shared__ int s_skip, s_nunits;
    if (threadIdx.x == 0) {   // one read, so every thread takes the same branch
        s_skip = *reinterpret_cast<volatile int32_t*>(p.err);
        s_nunits = *reinterpret_cast<const volatile int32_t*>(p.count) * p.H;
    }
    __syncthreads();
    if (s_skip != 0) return;   // invalid cu_seqlens: the whole call is a no-op
    const int nunits = s_nunits;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kQSlots; ++i) {
            mbar_init(bar(Q_FULL + i), 1);
            mbar_init(bar(Q_READY + i), CF::kQReadyCount);
            mbar_init(bar(Q_EMPTY + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(K_FULL + i), 1);
            mbar_init(bar(K_READY + i), 128);
            mbar_init(bar(K_EMPTY + i), 1);
            mbar_init(bar(V_FULL + i), 1);
            mbar_init(bar(V_EMPTY + i), 1);
            mbar_init(bar(S_FULL + i), 1);
            mbar_init(bar(P_FULL + i), CF::kTileThreads);   // the softmax threads of q tile i
            mbar_init(bar(O_FULL + i), 1);
            mbar_init(bar(O_EMPTY + i), CF::kTileThreads);
        }
        mbar_init(bar(DRAIN), 1);
        for (int i = 0; i < kRing; ++i) {
            mbar_init(bar(UNIT_FULL + i), 1);
            mbar_init(bar(UNIT_EMPTY + i), ROPE && p.use_rope ? kRingConsumers : kRingConsumers - 4);
        }
        abort[0] = 0;
        abort[1] = static_cast<int>(p.wait_limit_us);   // the waits' limit (ctl[1])
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmKr);
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

    uint32_t q_issued = 0, k_issued = 0, kv_issued = 0;   // for the teardown drain

    // Softmax warpgroups hold a whole S row per thread; the producer/MMA/TMEM and
    // RoPE warpgroups give registers up for them (each role sets its budget first).
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        setmaxnreg_dec<CF::kCtrlRegs>();
        if (lane == 0) {
            const uint64_t pol_stream = make_l2_policy_evict_first();   // q: read once
            const uint64_t pol_keep = make_l2_policy_evict_last();      // K/V: read by many units
            uint32_t qm = 0, kvn = 0;
            bool ok = true;
            for (int n = 0; ok; ++n) {
                int u;
                Unit w;
                if (!(ok = ring_get(rg, n, abort, u, w)) || u < 0) break;
                const FUnit f = make_funit<KV>(p, w);
                for (int t = 0; t < 1 + (f.has1 ? 1 : 0) && ok; ++t) {
                    const int slot = qm % kQSlots;
                    if (!(ok = mbar_wait(bar(Q_EMPTY + slot), ((qm / kQSlots) & 1) ^ 1, abort))) break;
                    mbar_expect_tx(bar(Q_FULL + slot), LY::TILE);
                    const int row = f.w.row0 + (f.q0 + t) * BQ;
#pragma unroll
                    for (int kb = 0; kb < LY::KB; ++kb)
                        tma_load_3d_hint(sbase + LY::Q0 + slot * LY::TILE + kb * LY::BLK, &tmQ, kb * 64,
                                         f.w.h, row, bar(Q_FULL + slot), pol_stream);
                    q_issued = ++qm;
                }
                // K tiles only: V tiles come from their own producer (warp 3), so a V
                // load never waits behind a K stage and vice versa.
                for (int j = 0; j < f.nk && ok; ++j) {
                    const uint32_t n = kvn + j;
                    const int ks = n & 1;
                    if (!(ok = mbar_wait(bar(K_EMPTY + ks), ((n >> 1) & 1) ^ 1, abort))) break;
                    mbar_expect_tx(bar(K_FULL + ks), LY::TILE);
#pragma unroll
                    for (int kb = 0; kb < LY::KB; ++kb)
                        tma_load_3d_hint(sbase + LY::K0 + ks * LY::TILE + kb * LY::BLK, f.pre ? &tmKr : &tmK, kb * 64,
                                         f.hkv, f.w.row0k + j * BN, bar(K_FULL + ks), pol_keep);
                    k_issued = n + 1;
                }
                kvn += f.nk;
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs this loop (so descriptors and addresses stay warp-uniform);
        // one elected lane issues every MMA and commit.
        setmaxnreg_dec<CF::kCtrlRegs>();
        {
            constexpr uint32_t IDESC_S = idesc_bf16_f32(128, BN, false);
            constexpr uint32_t IDESC_O = idesc_bf16_f32(128, D, true);
            uint32_t qm = 0, kvn = 0, cnt_p[2] = {0, 0}, cnt_u[2] = {0, 0};
            // without RoPE the staged tiles go straight from the TMA barriers to the MMAs; with
            // the q rotation in the softmax warps the K tiles do (k was rotated beforehand)
            const int qrb = p.use_rope ? Q_READY : Q_FULL, krb = ROPE && p.use_rope ? K_READY : K_FULL;
            bool ok = true;
            auto commit = [&](uint32_t b) {
                if (elect_one()) mma_commit(b);
                __syncwarp();
            };
            // Descriptors are built once per tile; the K-step offsets are added to the
            // start-address field (addresses stay below 2^18, so the field cannot carry).
            auto issue_s = [&](int t, int slot, int ks) {
                const uint64_t qd = smem_desc_sw128(sbase + LY::Q0 + slot * LY::TILE, 16, 1024);
                const uint64_t kd = smem_desc_sw128(sbase + LY::K0 + ks * LY::TILE, 16, 1024);
                if (elect_one()) {
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t off = ((k >> 2) * LY::BLK + (k & 3) * 32) >> 4;
                        mma_bf16_ss(tmem + LY::S_COL(t), qd + off, kd + off, IDESC_S, k > 0 ? 1u : 0u);
                    }
                    mma_commit(bar(S_FULL + t));
                }
                __syncwarp();
            };
            for (int un = 0; ok; ++un) {
                int u;
                Unit uw;
                if (!(ok = ring_get_warp(rg, un, abort, u, uw)) || u < 0) break;
                const FUnit f = make_funit<KV>(p, uw);
                const int n[2] = {f.n0, f.n1};
                const int slot[2] = {static_cast<int>(qm % kQSlots), static_cast<int>((qm + 1) % kQSlots)};
                {   // without RoPE in the kernel each q tile's first S goes as soon as that tile has
                    // landed (the second tile's slot is the last to land; +1% on the short-document
                    // packs); with it both tiles are waited for first (the other order measured up to
                    // 2.5% slower there)
                    constexpr bool kEachTile = MODE == kModePlain;
                    const int ks = kvn & 1;
                    if (!(ok = wait_warp(bar(qrb + slot[0]), (qm / kQSlots) & 1, abort))) break;
                    if (!kEachTile && f.has1 &&
                        !(ok = wait_warp(bar(qrb + slot[1]), ((qm + 1) / kQSlots) & 1, abort)))
                        break;
                    if (!(ok = wait_warp(bar(krb + ks), (kvn >> 1) & 1, abort))) break;
                    tc_fence_after();
                    for (int t = 0; t < 2 && ok; ++t) {
                        if (n[t] == 0) continue;
                        if (kEachTile && t == 1) {
                            if (!(ok = wait_warp(bar(qrb + slot[1]), ((qm + 1) / kQSlots) & 1, abort))) break;
                            tc_fence_after();
                        }
                        issue_s(t, slot[t], ks);
                        if (n[t] == 1) commit(bar(Q_EMPTY + slot[t]));
                    }
                    if (!ok) break;
                    commit(bar(K_EMPTY + ks));
                }
                for (int j = 0; j < f.nk && ok; ++j) {
                    const uint32_t kvj = kvn + j;
                    const int vs = kvj & 1;
                    if (!(ok = wait_warp(bar(V_FULL + vs), (kvj >> 1) & 1, abort))) break;
                    bool k_next = false;
                    for (int t = 0; t < 2 && ok; ++t) {
                        if (j >= n[t]) continue;
                        if (!(ok = wait_warp(bar(P_FULL + t), cnt_p[t] & 1, abort))) break;
                        ++cnt_p[t];
                        if (j == 0 && !(ok = wait_warp(bar(O_EMPTY + t), (cnt_u[t] & 1) ^ 1, abort))) break;
                        tc_fence_after();
                        const uint64_t vd = smem_desc_sw128(sbase + LY::V0 + vs * LY::TILE, LY::BLK, 1024);
                        if (elect_one()) {
#pragma unroll
                            for (int k = 0; k < BN / 16; ++k)
                                mma_bf16_ts(tmem + LY::O_COL(t), tmem + LY::S_COL(t) + 8 * k,
                                            vd + ((k * 16 * 128) >> 4), IDESC_O, (j > 0 || k > 0) ? 1u : 0u);
                            if (j == n[t] - 1) mma_commit(bar(O_FULL + t));
                        }
                        __syncwarp();
                        if (j + 1 < n[t]) {
                            const uint32_t kvn1 = kvj + 1;
                            if (!k_next) {
                                if (!(ok = wait_warp(bar(krb + (kvn1 & 1)), (kvn1 >> 1) & 1, abort))) break;
                                tc_fence_after();
                                k_next = true;
                            }
                            issue_s(t, slot[t], kvn1 & 1);
                            if (j + 1 == n[t] - 1) commit(bar(Q_EMPTY + slot[t]));
                        }
                    }
                    if (!ok) break;
                    commit(bar(V_EMPTY + vs));
                    if (k_next) commit(bar(K_EMPTY + ((kvj + 1) & 1)));
                }
                if (!ok) break;
                kvn += f.nk;
                qm += f.has1 ? 2 : 1;
                ++cnt_u[0];
                if (f.has1) ++cnt_u[1];
            }
            commit(bar(DRAIN));
            mbar_wait_limit(bar(DRAIN), 0, 200000000ull);
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 4 + CF::kSoftWarps) {
        if constexpr (ROPE) {
            // ------------------------------------------------------------ softmax + epilogue, one
            // thread per query row (warps 4-7: q tile 0, 8-11: q tile 1; the RoPE warpgroup's
            // registers leave no room for the split rows below)
            setmaxnreg_inc<CF::kSoftRegs>();
            const int t = (warp - 4) >> 2;             // q tile slot handled by this warpgroup
            const int wq = warp & 3;                   // TMEM lane quadrant
            const int r = wq * 32 + lane;              // query row in the tile = TMEM lane
            const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
            const uint32_t sadr = tmem + lane_off + LY::S_COL(t);
            const uint32_t oadr = tmem + lane_off + LY::O_COL(t);
            const float sl2 = p.scale_log2;
            const bool v8 = (reinterpret_cast<uintptr_t>(p.o) & 31) == 0;   // 256-bit row stores
            uint32_t cnt_s = 0, cnt_u = 0;
            bool ok = true;
            for (int un = 0; ok; ++un) {
                int u;
                Unit uw;
                if (!(ok = ring_get_warp(rg, un, abort, u, uw)) || u < 0) break;
                const FUnit f = make_funit<KV>(p, uw);
                const int nt = t == 0 ? f.n0 : f.n1;
                if (nt == 0) continue;
                const int qpos = (f.q0 + t) * BQ + r;
                float m_run = 0.f, l_run = 0.f;
                for (int j = 0; j < nt; ++j) {
                    if (!(ok = wait_warp(bar(S_FULL + t), cnt_s & 1, abort))) break;
                    ++cnt_s;
                    tc_fence_after();
                    // allowed key columns of this tile: c <= lim.  Only the last tile is masked,
                    // or the last two when the diagonal is not tile-aligned (off % BN != 0)
                    const bool edge = (j == nt - 1) || (KV && j == nt - 2 && (f.w.off & (BN - 1)) != 0);
                    const int lim = edge ? min(qpos + f.w.off, f.w.Lk - 1) - j * BN : BN - 1;
                    // the thread's whole S row (BN fp32 columns) in registers: four loads, one wait
                    uint32_t s[BN];
    #pragma unroll
                    for (int c = 0; c < BN / 32; ++c)
                        tmem_ld32(sadr + c * 32, *reinterpret_cast<uint32_t(*)[32]>(s + c * 32));
                    tmem_wait_ld();
                    if (edge) {   // masked scores -> -inf: they drop out of the max and exp2 gives 0
    #pragma unroll
                        for (int e = 0; e < BN; ++e)
                            if (e > lim) s[e] = 0xff800000u;
                    }
                    // row max of the raw scores: four independent 3-input max chains
                    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    #pragma unroll
                    for (int e = 0; e < BN; e += 8) {
    #pragma unroll
                        for (int q = 0; q < 4; ++q)
                            m4[q] = fmax3(m4[q], __uint_as_float(s[e + 2 * q]), __uint_as_float(s[e + 2 * q + 1]));
                    }
                    const float mt = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]) * sl2;
                    float m_use = m_run, alpha = 1.f;
                    bool rescale = false;
                    if (j == 0) {
                        m_use = mt;
                    } else {
                        rescale = __any_sync(0xffffffffu, mt > m_run + kRescaleThreshold);
                        if (rescale) {
                            m_use = fmaxf(m_run, mt);
                            alpha = ex2_approx(m_run - m_use);
                        }
                    }
                    // P = exp2(s * scale_log2 - m) -> bf16 pairs written over the first BN/2
                    // S columns, each half as soon as it is packed
                    const float2 sc2 = make_float2(sl2, sl2), nm2 = make_float2(-m_use, -m_use);
                    float2 rs2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    #pragma unroll
                    for (int hlf = 0; hlf < 2; ++hlf) {
                        uint32_t pk[BN / 4];
    #pragma unroll
                        for (int e = 0; e < BN / 4; ++e) {
                            const int c = hlf * (BN / 2) + 2 * e;
                            const float2 x = fma2(make_float2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), sc2, nm2);
                            const float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
                            rs2[e & 1] = add2(rs2[e & 1], make_float2(p0, p1));
                            pk[e] = pack_bf16x2(p0, p1);
                        }
                        tmem_st32(sadr + hlf * (BN / 4), pk);
                    }
                    if (rescale) {   // O_t is stable: S_t(j) done implies P_t V(j-1) done
    #pragma unroll 1
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t rr[32];
                            tmem_ld32(oadr + c * 32, rr);
                            tmem_wait_ld();
    #pragma unroll
                            for (int e = 0; e < 32; ++e)
                                rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
                            tmem_st32(oadr + c * 32, rr);
                        }
                        l_run *= alpha;
                    }
                    tmem_wait_st();
                    l_run += (rs2[0].x + rs2[1].x) + (rs2[0].y + rs2[1].y);
                    m_run = m_use;
                    tc_fence_before();
                    mbar_arrive(bar(P_FULL + t));
                }
                if (!ok) break;
                // ---- epilogue: O / l -> bf16, LSE
                if (!(ok = wait_warp(bar(O_FULL + t), cnt_u & 1, abort))) break;
                tc_fence_after();
                const bool valid = qpos < f.w.L;
                const int64_t tok = static_cast<int64_t>(f.w.row0) + qpos;
                const float inv_l = 1.f / l_run;
                uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) +
                                ((valid ? tok : 0) * p.H + f.w.h) * static_cast<int64_t>(D) * 2;
                // read O (two 32-column chunks at a time); the columns are released to the
                // next unit as soon as the last chunk has landed, before packing and storing
    #pragma unroll
                for (int c = 0; c < D / 32; c += 2) {
                    uint32_t ra[32], rb[32];
                    tmem_ld32(oadr + c * 32, ra);
                    tmem_ld32(oadr + c * 32 + 32, rb);
                    tmem_wait_ld();
                    if (c + 2 >= D / 32) {
                        tc_fence_before();
                        mbar_arrive(bar(O_EMPTY + t));
                    }
                    uint32_t pk[32];
    #pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        pk[e] = pack_bf16x2(__uint_as_float(ra[2 * e]) * inv_l, __uint_as_float(ra[2 * e + 1]) * inv_l);
                        pk[16 + e] = pack_bf16x2(__uint_as_float(rb[2 * e]) * inv_l, __uint_as_float(rb[2 * e + 1]) * inv_l);
                    }
                    if (valid) {
                        st_row64(orow + c * 64, pk, v8);
                        st_row64(orow + c * 64 + 64, pk + 16, v8);
                    }
                }
                if (valid)
                    p.lse[static_cast<int64_t>(f.w.h) * p.total + tok] = (m_run + __log2f(l_run)) * kLn2;
                ++cnt_u;
            }
        } else {
            // ------------------------------------------------------------ softmax + epilogue
            // Two warpgroups per q tile.  A warp covers 16 query rows (TMEM lanes) of its
            // quadrant; thread i < 16 takes score columns 0-63 of row i, thread i + 16 columns
            // 64-127 of the same row (the 16x32bx2 access shape), so a row's maximum and sum
            // meet in one shuffle.
            setmaxnreg_inc<CF::kSoftRegs>();
            const int t = (warp - 4) >> 3;             // q tile slot handled by this warp
            const int wq = warp & 3;                   // TMEM lane quadrant (warp % 4)
            const int sub = ((warp - 4) >> 2) & 1;     // which 16 lanes of the quadrant
            const int hf = lane >> 4;                  // which half of the row's columns
            const int r = wq * 32 + sub * 16 + (lane & 15);   // query row in the tile = TMEM lane
            const uint32_t lane_off = static_cast<uint32_t>(wq * 32 + sub * 16) << 16;
            const uint32_t sadr = tmem + lane_off + LY::S_COL(t);
            const uint32_t oadr = tmem + lane_off + LY::O_COL(t);
            constexpr int HC = BN / 2;                 // score columns per thread
            constexpr int HD = D / 2;                  // output columns per thread
            const float sl2 = p.scale_log2;
            const bool v8 = (reinterpret_cast<uintptr_t>(p.o) & 31) == 0;   // 256-bit row stores
            uint32_t cnt_s = 0, cnt_u = 0;
            // With kModeQRot the warps of q tile 0, which finish each unit one key tile before
            // those of q tile 1, rotate the next unit's q tiles in shared memory (warpgroup sub
            // takes tile sub) once they have landed and release them to the MMA warp; the next
            // unit is read from the ring after this unit's last P, before the O wait.  qm counts
            // the q slots of the units before the current one, as the producer and the MMA warp do.
            uint32_t qm = 0;
            auto rotate_q = [&](const FUnit& g, uint32_t qslots) -> bool {
                if constexpr (ROTQ) {
                    if (t != 0 || (sub == 1 && !g.has1)) return true;
                    const uint32_t qs = qslots + sub;
                    if (!wait_warp(bar(Q_FULL + qs % kQSlots), (qs / kQSlots) & 1, abort)) return false;
                    const uint32_t tile = sbase + LY::Q0 + (qs % kQSlots) * LY::TILE;
                    const int pos0 = (g.q0 + sub) * BQ + g.w.off;
                    // with qrot_out the rotated rows of the segment also go to global memory
                    const int64_t gstride = static_cast<int64_t>(p.H) * D * 2;
                    uint8_t* gdst = p.qrot_out == nullptr ? nullptr
                                    : static_cast<uint8_t*>(p.qrot_out) +
                                          (static_cast<int64_t>(g.w.row0) + (g.q0 + sub) * BQ) * gstride +
                                          static_cast<int64_t>(g.w.h) * D * 2;
                    const int nvalid = g.w.L - (g.q0 + sub) * BQ;
                    if (p.use_rope == kRopeInterleaved)
                        rope_tile<D, 128, true>(tile, pos0, p.table, rope_step<D, true>(p.table, lane), wq, lane,
                                                gdst, gstride, nvalid);
                    else
                        rope_tile<D, 128, false>(tile, pos0, p.table, rope_step<D, false>(p.table, lane), wq, lane,
                                                 gdst, gstride, nvalid);
                    fence_proxy_async_smem();
                    mbar_arrive(bar(Q_READY + qs % kQSlots));
                }
                return true;
            };
            int u;
            Unit uw;
            bool ok = ring_get_warp(rg, 0, abort, u, uw);
            if (ok && u >= 0) ok = rotate_q(make_funit<KV>(p, uw), 0);
            for (int un = 0; ok && u >= 0; ++un) {
                const FUnit f = make_funit<KV>(p, uw);
                const uint32_t qm_next = qm + (f.has1 ? 2u : 1u);
                const int nt = t == 0 ? f.n0 : f.n1;
                int u_next;
                Unit w_next;
                if (nt == 0) {
                    if (!(ok = ring_get_warp(rg, un + 1, abort, u_next, w_next))) break;
                    if (u_next >= 0 && !(ok = rotate_q(make_funit<KV>(p, w_next), qm_next))) break;
                    u = u_next;
                    uw = w_next;
                    qm = qm_next;
                    continue;
                }
                const int qpos = (f.q0 + t) * BQ + r;
                float m_run = 0.f, l_run = 0.f;   // l_run: this thread's half of the row sum
                for (int j = 0; j < nt; ++j) {
                    if (!(ok = wait_warp(bar(S_FULL + t), cnt_s & 1, abort))) break;
                    ++cnt_s;
                    tc_fence_after();
                    // allowed key columns of this tile: c <= lim.  Only the last tile is masked,
                    // or the last two when the diagonal is not tile-aligned (off % BN != 0)
                    const bool edge = (j == nt - 1) || (KV && j == nt - 2 && (f.w.off & (BN - 1)) != 0);
                    const int lim = (edge ? min(qpos + f.w.off, f.w.Lk - 1) - j * BN : BN - 1) - hf * HC;
                    // the thread's 64 scores in registers (two loads, one wait); the loads also
                    // return their maxima
                    uint32_t s[HC];
                    float mx0, mx1;
                    tmem_ld32_pair_max<HC>(sadr, *reinterpret_cast<uint32_t(*)[32]>(s), mx0);
                    tmem_ld32_pair_max<HC>(sadr + 32, *reinterpret_cast<uint32_t(*)[32]>(s + 32), mx1);
                    tmem_wait_ld();
                    float mloc = fmaxf(mx0, mx1);
                    if (edge) {   // masked scores -> -inf: they drop out of the max and exp2 gives 0
    #pragma unroll
                        for (int e = 0; e < HC; ++e)
                            if (e > lim) s[e] = 0xff800000u;
                        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    #pragma unroll
                        for (int e = 0; e < HC; e += 8) {
    #pragma unroll
                            for (int q = 0; q < 4; ++q)
                                m4[q] = fmax3(m4[q], __uint_as_float(s[e + 2 * q]), __uint_as_float(s[e + 2 * q + 1]));
                        }
                        mloc = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
                    }
                    const float mt = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 16)) * sl2;
                    float m_use = m_run, alpha = 1.f;
                    bool rescale = false;
                    if (j == 0) {
                        m_use = mt;
                    } else {
                        rescale = __any_sync(0xffffffffu, mt > m_run + kRescaleThreshold);
                        if (rescale) {
                            m_use = fmaxf(m_run, mt);
                            alpha = ex2_approx(m_run - m_use);
                        }
                    }
                    // P = exp2(s * scale_log2 - m) -> 32 bf16 pairs written over the row's
                    // consumed S columns (thread i < 16: columns 0-31, i + 16: columns 32-63)
                    const float2 sc2 = make_float2(sl2, sl2), nm2 = make_float2(-m_use, -m_use);
                    float2 rs2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                    {
                        uint32_t pk[HC / 2];
    #pragma unroll
                        for (int e = 0; e < HC / 2; ++e) {
                            const float2 x = fma2(make_float2(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1])), sc2, nm2);
                            const float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
                            rs2[e & 1] = add2(rs2[e & 1], make_float2(p0, p1));
                            pk[e] = pack_bf16x2(p0, p1);
                        }
                        tmem_st32_pair<HC / 2>(sadr, pk);
                    }
                    if (rescale) {   // O_t is stable: S_t(j) done implies P_t V(j-1) done
    #pragma unroll 1
                        for (int c = 0; c < HD / 32; ++c) {
                            uint32_t rr[32];
                            tmem_ld32_pair<HD>(oadr + c * 32, rr);
                            tmem_wait_ld();
    #pragma unroll
                            for (int e = 0; e < 32; ++e)
                                rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
                            tmem_st32_pair<HD>(oadr + c * 32, rr);
                        }
                        l_run *= alpha;
                    }
                    tmem_wait_st();
                    l_run += (rs2[0].x + rs2[1].x) + (rs2[0].y + rs2[1].y);
                    m_run = m_use;
                    tc_fence_before();
                    mbar_arrive(bar(P_FULL + t));
                }
                if (!ok) break;
                if (!(ok = ring_get_warp(rg, un + 1, abort, u_next, w_next))) break;
                if (u_next >= 0 && !(ok = rotate_q(make_funit<KV>(p, w_next), qm_next))) break;
                // ---- epilogue: O / l -> bf16, LSE
                if (!(ok = wait_warp(bar(O_FULL + t), cnt_u & 1, abort))) break;
                tc_fence_after();
                const bool valid = qpos < f.w.L;
                const int64_t tok = static_cast<int64_t>(f.w.row0) + qpos;
                const float l_row = l_run + __shfl_xor_sync(0xffffffffu, l_run, 16);
                const float inv_l = 1.f / l_row;
                uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) +
                                ((valid ? tok : 0) * p.H + f.w.h) * static_cast<int64_t>(D) * 2 + hf * HD * 2;
                // the thread's half of the O row (columns hf * D/2 ...), all chunks then one wait;
                // the columns go back to the next unit before packing and storing
                uint32_t ro[HD];
    #pragma unroll
                for (int c = 0; c < HD / 32; ++c)
                    tmem_ld32_pair<HD>(oadr + c * 32, *reinterpret_cast<uint32_t(*)[32]>(ro + c * 32));
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(bar(O_EMPTY + t));
    #pragma unroll
                for (int c = 0; c < HD / 32; ++c) {
                    uint32_t pk[16];
    #pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack_bf16x2(__uint_as_float(ro[c * 32 + 2 * e]) * inv_l,
                                            __uint_as_float(ro[c * 32 + 2 * e + 1]) * inv_l);
                    if (valid) st_row64(orow + c * 64, pk, v8);
                }
                if (valid && hf == 0)
                    p.lse[static_cast<int64_t>(f.w.h) * p.total + tok] = (m_run + __log2f(l_row)) * kLn2;
                ++cnt_u;
                u = u_next;
                uw = w_next;
                qm = qm_next;
            }
        }
    } else if (warp >= 4 + CF::kSoftWarps) {
        // ------------------------------------------------------------ RoPE on staged q / K tiles
        // (only in the instance with RoPE)
        if constexpr (ROPE) setmaxnreg_dec<CF::kRopeRegs>();
        const int wr = warp - 4 - CF::kSoftWarps;
        // one copy of the loop per pairing, so neither carries the other's state
        auto run = [&](auto il_tag) {
            constexpr bool IL = decltype(il_tag)::value;
            RopeStep<D> step{};
            if (p.use_rope) step = rope_step<D, IL>(p.table, lane);
            uint32_t qm = 0, kvn = 0;
            bool ok = true;
            for (int un = 0; ok; ++un) {
                int u;
                Unit uw;
                if (!(ok = ring_get_warp(rg, un, abort, u, uw)) || u < 0) break;
                const FUnit f = make_funit<KV>(p, uw);
                for (int t = 0; t < 1 + (f.has1 ? 1 : 0) && ok; ++t) {
                    const int slot = qm % kQSlots;
                    if (!(ok = wait_warp(bar(Q_FULL + slot), (qm / kQSlots) & 1, abort))) break;
                    if (p.use_rope)
                        rope_tile<D, 128, IL>(sbase + LY::Q0 + slot * LY::TILE, (f.q0 + t) * BQ + f.w.off,
                                              p.table, step, wr, lane);
                    fence_proxy_async_smem();
                    mbar_arrive(bar(Q_READY + slot));
                    ++qm;
                }
                for (int j = 0; j < f.nk && ok; ++j) {
                    const int ks = kvn & 1;
                    if (!(ok = wait_warp(bar(K_FULL + ks), (kvn >> 1) & 1, abort))) break;
                    if (p.use_rope && !f.pre)
                        rope_tile<D, 128, IL>(sbase + LY::K0 + ks * LY::TILE, j * BN, p.table, step, wr, lane);
                    fence_proxy_async_smem();
                    mbar_arrive(bar(K_READY + ks));
                    ++kvn;
                }
            }
        };
        if constexpr (ROPE) {
            if (p.use_rope == kRopeInterleaved) run(std::true_type{});
            else run(std::false_type{});
        }   // without RoPE these warps take no units
    } else if (warp == 3) {
        // ------------------------------------------------------------ TMA producer of V tiles
        setmaxnreg_dec<CF::kCtrlRegs>();
        if (lane == 0) {
            const uint64_t pol_keep = make_l2_policy_evict_last();
            uint32_t vn = 0;
            bool ok = true;
            for (int un = 0; ok; ++un) {
                int u;
                Unit uw;
                if (!(ok = ring_get(rg, un, abort, u, uw)) || u < 0) break;
                const FUnit f = make_funit<KV>(p, uw);
                for (int j = 0; j < f.nk && ok; ++j) {
                    const uint32_t n = vn + j;
                    const int vs = n & 1;
                    if (!(ok = mbar_wait(bar(V_EMPTY + vs), ((n >> 1) & 1) ^ 1, abort))) break;
                    mbar_expect_tx(bar(V_FULL + vs), LY::TILE);
#pragma unroll
                    for (int kb = 0; kb < LY::KB; ++kb)
                        tma_load_3d_hint(sbase + LY::V0 + vs * LY::TILE + kb * LY::BLK, &tmV, kb * 64,
                                         f.hkv, f.w.row0k + j * BN, bar(V_FULL + vs), pol_keep);
                    kv_issued = n + 1;
                }
                vn += f.nk;
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ warp 2: TMEM allocator, then
        // the unit scheduler (claims and decodes units ahead of the other roles)
        setmaxnreg_dec<CF::kCtrlRegs>();
        {   // the whole warp: lane 0 claims and publishes, all lanes decode
            auto decode = [&](int u) {
                Unit w = decode_unit_warp<KV>(p.items, p.seg_base, p.cu, p.rows, p.cu_kv, p.rows_kv, p.nseg, p.H, u);
                // all keys visible: the diagonal moves past the last key (query p sees keys up to p + Lk)
                if (KV && p.keys_all_visible) w.off = w.Lk;
                return w;
            };
            for (int n = 0;; ++n) {
                int u;
                if (!ring_put_warp(rg, n, p.next, nunits, abort, decode, u) || u < 0) break;
            }
        }
        __syncwarp();
    }

    __syncthreads();
    if (*abort) {
        // each producer waits (bounded) for the last copy it issued into every slot and stage
        if ((warp == 0 || warp == 3) && lane == 0) {
            for (int s = 0; s < kQSlots; ++s)
                if (q_issued > static_cast<uint32_t>(s)) {
                    const uint32_t n = q_issued - 1 - ((q_issued - 1 - s) % kQSlots);
                    mbar_wait_limit(bar(Q_FULL + s), (n / kQSlots) & 1, 200000000ull);
                }
            for (int s = 0; s < 2; ++s) {
                if (k_issued > static_cast<uint32_t>(s)) {
                    const uint32_t n = ((k_issued - 1 - s) & ~1u) + s;
                    mbar_wait_limit(bar(K_FULL + s), (n >> 1) & 1, 200000000ull);
                }
                if (kv_issued > static_cast<uint32_t>(s)) {
                    const uint32_t n = ((kv_issued - 1 - s) & ~1u) + s;
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
    CUtensorMap tq, tk, tkr, tv;
    if (!make_tmap_thd(&tq, p.q, p.total, p.H, p.d, 128) ||
        !make_tmap_thd(&tk, p.k, p.total_kv, p.Hkv, p.d, 128) ||
        !make_tmap_thd(&tkr, p.krot != nullptr ? p.krot : p.k, p.total_kv, p.Hkv, p.d, 128) ||
        !make_tmap_thd(&tv, p.v, p.total_kv, p.Hkv, p.d, 128))
        return cudaErrorInvalidValue;
    const bool kv = p.cu_kv != p.cu || p.keys_all_visible;
    // RoPE with k rotated beforehand into the workspace: the softmax warps rotate q; RoPE
    // without that copy: the RoPE-warp instance; no RoPE (or operands rotated beforehand)
    const int mode = p.use_rope == kRopeNone ? fwd::kModePlain
                     : (p.krot != nullptr ? fwd::kModeQRot : fwd::kModeWarps);
    using KFn = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, const FwdParams);
    auto pick = [&](auto dtag, auto kvtag) -> KFn {
        constexpr int D = decltype(dtag)::value;
        constexpr bool KVI = decltype(kvtag)::value;
        return mode == fwd::kModePlain  ? fwd::attn_fwd_kernel<D, KVI, fwd::kModePlain>
               : mode == fwd::kModeQRot ? fwd::attn_fwd_kernel<D, KVI, fwd::kModeQRot>
                                        : fwd::attn_fwd_kernel<D, KVI, fwd::kModeWarps>;
    };
    using D128 = std::integral_constant<int, 128>;
    using D64 = std::integral_constant<int, 64>;
    const KFn kernel = p.d == 128 ? (kv ? pick(D128{}, std::true_type{}) : pick(D128{}, std::false_type{}))
                                  : (kv ? pick(D64{}, std::true_type{}) : pick(D64{}, std::false_type{}));
    const int threads = mode == fwd::kModeWarps ? fwd::Cfg<fwd::kModeWarps>::kThreads : fwd::Cfg<fwd::kModePlain>::kThreads;
    const uint32_t regs =
        mode == fwd::kModeWarps ? fwd::Cfg<fwd::kModeWarps>::kLaunchRegs : fwd::Cfg<fwd::kModePlain>::kLaunchRegs;
    const dim3 grid(num_sms), block(threads);
    const uint32_t smem = p.d == 128 ? fwd::Layout<128>::ALLOC : fwd::Layout<64>::ALLOC;
    // The warpgroups re-split the block's register pool at run time, which is only
    // valid if every thread is launched with exactly the planned registers.
    {
        cudaFuncAttributes fa{};
        cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != static_cast<int>(regs)) return cudaErrorInvalidConfiguration;
    }
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kernel<<<grid, block, smem, s>>>(tq, tk, tkr, tv, p);
    return cudaGetLastError();
}


// ---------------------------------------------------------------- q', k' for a whole training step
// R(p) q and R(p) k for every row, once: the forward and backward passes of a step can
// then run on the rotated operands (no in-kernel rotation, no rotation in the
// backward's prep pass).  With H = 0 (no query heads) and the key segments it is the
// forward's k pass: k' for the kernel that rotates only the q tiles.  A block takes a
// contiguous run of tokens, D/16 threads per
// token: each thread loads the cos/sin of its 16-byte chunk pair once per token and
// rotates that chunk pair in every query head and every key head of the token
// (consecutive threads cover consecutive 16-byte chunks of a head row, so a warp reads
// and writes whole 128-byte lines).
namespace fwd {
template <int D>
__global__ void __launch_bounds__(256)
rope_qk_kernel(const uint4* __restrict__ q, const uint4* __restrict__ k, uint4* __restrict__ qrot,
               uint4* __restrict__ krot, const int32_t* __restrict__ cu, const int32_t* __restrict__ rows,
               int32_t nseg, const float2* __restrict__ table, int32_t total, int32_t H, int32_t Hkv, int rope,
               const int32_t* __restrict__ err) {
    if (*err != 0) return;
    constexpr int TPR = D / 16;               // threads per token (16-byte chunk pairs of a head row)
    constexpr int HALF = D / 16;
    constexpr int TOKB = 256 / TPR;           // tokens side by side in a block
    const int c = threadIdx.x % TPR, ts = threadIdx.x / TPR;
    const bool il = rope == kRopeInterleaved;
    // a contiguous run of tokens per block; a thread takes every TOKB-th token of it, so its
    // segment index only moves forward, and loads its chunk pair's cos/sin once per token for
    // all of the token's head rows
    const int64_t per = (static_cast<int64_t>(total) + gridDim.x - 1) / gridDim.x;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * per;
    const int64_t t1 = min(static_cast<int64_t>(total), t0 + per);
    int64_t tok = t0 + ts;
    if (tok >= t1) return;
    int a = segment_of_row(rows, nseg, tok);
    int64_t next = a + 1 < nseg ? __ldg(rows + a + 1) : INT64_MAX;
    for (; tok < t1; tok += TOKB) {
        while (tok >= next) {
            ++a;
            next = a + 1 < nseg ? __ldg(rows + a + 1) : INT64_MAX;
        }
        const int64_t pos0 = tok - __ldg(rows + a);
        const bool real = pos0 < __ldg(cu + a + 1) - __ldg(cu + a);   // rows past a padded segment: zeros
        float cs[8], sn[8];
        if (real) load_angles<D>(table, pos0, il, c, cs, sn);
#pragma unroll 4
        for (int h = 0; h < H; ++h) {
            const int64_t lo = (tok * H + h) * (2 * HALF) + c;
            rotate_chunks(q, qrot, lo, lo + HALF, cs, sn, real, il);
        }
#pragma unroll 4
        for (int h = 0; h < Hkv; ++h) {
            const int64_t lo = (tok * Hkv + h) * (2 * HALF) + c;
            rotate_chunks(k, krot, lo, lo + HALF, cs, sn, real, il);
        }
    }
}
}  // namespace fwd

static cudaError_t launch_rope_rows(const FwdParams& p, const void* q, const void* k, void* qrot, void* krot,
                                    const int32_t* cu, const int32_t* rows, int32_t total, int32_t H, int num_sms,
                                    cudaStream_t s) {
    const int tokb = 256 / (p.d / 16);   // tokens per block pass
    int64_t blocks = (static_cast<int64_t>(total) + tokb - 1) / tokb;
    if (blocks > static_cast<int64_t>(num_sms) * 8) blocks = static_cast<int64_t>(num_sms) * 8;
    if (blocks < 1) blocks = 1;
    auto kernel = p.d == 128 ? fwd::rope_qk_kernel<128> : fwd::rope_qk_kernel<64>;
    kernel<<<static_cast<int>(blocks), 256, 0, s>>>(static_cast<const uint4*>(q), static_cast<const uint4*>(k),
                                                     static_cast<uint4*>(qrot), static_cast<uint4*>(krot), cu, rows,
                                                     p.nseg, p.table, total, H, p.Hkv, p.use_rope, p.err);
    return cudaGetLastError();
}

cudaError_t launch_rope_qk(const FwdParams& p, void* qrot, void* krot, int num_sms, cudaStream_t s) {
    return launch_rope_rows(p, p.q, p.k, qrot, krot, p.cu, p.rows, p.total, p.H, num_sms, s);
}

// k alone (no query heads), over the key segments: the forward's rotated copy of k.
cudaError_t launch_rope_k(const FwdParams& p, void* krot, int num_sms, cudaStream_t s) {
    return launch_rope_rows(p, nullptr, p.k, nullptr, krot, p.cu_kv, p.rows_kv, p.total_kv, 0, num_sms, s);
}

}  // namespace vlc
