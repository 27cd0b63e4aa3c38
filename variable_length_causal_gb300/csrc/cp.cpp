// cp.cpp -- host side of the context-parallel split of a packed buffer: which rows
// each rank of a context-parallel group holds, and which (query chunk, key chunk)
// blocks of the ring it computes.  Declared in include/vlc.h (vlc_cp_partition,
// vlc_cp_block_mode).
//
// "Long-context training: remove padding" (vllbc), failure-modes section: with
// context parallelism the sequence length must be a multiple of
// 2 * context_parallel_size, because of how CP slices it.  "Sequence packing and
// variable-length attention" (charlestar), section on the two ledgers: the shards
// and the communication must follow the global segment boundaries, and ranks are
// balanced by attention work (sum of L^2), not tokens.  Every segment of length L
// is cut into 2 * cp chunks of m = L / (2 cp); rank i holds chunk i (its "low"
// half) and chunk 2 cp - 1 - i (its "high" half) of every segment, so each rank's
// causal work inside every segment is (2 cp - 1) m^2 + m (m + 1), the same for all
// ranks.  A rank's buffer is its low chunks of all segments in segment order, then
// its high chunks: each half is a packed buffer of its own whose segments are the
// chunks (offsets cu_chunk), so a block of the ring is one attention call.
#include <cstdint>

#include "../../include/vlc.h"

extern "C" int vlc_cp_partition(const int32_t* cu, int32_t nseg, int32_t cp, int32_t rank, int64_t* rows,
                                int32_t* pos, int32_t* cu_chunk, int32_t* bad_seg) {
    if (bad_seg != nullptr) *bad_seg = -1;
    if (cu == nullptr || rows == nullptr || pos == nullptr || cu_chunk == nullptr || nseg < 1 || cp < 1 ||
        rank < 0 || rank >= cp || cu[0] != 0)
        return VLC_ERR_ARG;
    const int64_t parts = 2 * static_cast<int64_t>(cp);
    int64_t acc = 0;
    cu_chunk[0] = 0;
    for (int32_t r = 0; r < nseg; ++r) {
        const int64_t L = static_cast<int64_t>(cu[r + 1]) - cu[r];
        if (L < 1) return VLC_ERR_CU_SEQLENS;
        if (L % parts != 0) {
            if (bad_seg != nullptr) *bad_seg = r;
            return VLC_ERR_ARG;
        }
        acc += L / parts;
        cu_chunk[r + 1] = static_cast<int32_t>(acc);
    }
    int64_t o = 0;
    for (int half = 0; half < 2; ++half) {
        const int64_t c = half == 0 ? rank : parts - 1 - rank;   // chunk index inside every segment
        for (int32_t r = 0; r < nseg; ++r) {
            const int64_t m = static_cast<int64_t>(cu_chunk[r + 1]) - cu_chunk[r];
            for (int64_t p = c * m; p < (c + 1) * m; ++p, ++o) {
                rows[o] = static_cast<int64_t>(cu[r]) + p;
                pos[o] = static_cast<int32_t>(p);
            }
        }
    }
    return VLC_OK;
}

extern "C" int vlc_cp_block_mode(int32_t cp, int32_t q_rank, int32_t q_half, int32_t kv_rank, int32_t kv_half) {
    if (cp < 1 || q_rank < 0 || q_rank >= cp || kv_rank < 0 || kv_rank >= cp || (q_half & ~1) || (kv_half & ~1))
        return -1;
    const int32_t cq = q_half == 0 ? q_rank : 2 * cp - 1 - q_rank;
    const int32_t ck = kv_half == 0 ? kv_rank : 2 * cp - 1 - kv_rank;
    if (ck < cq) return VLC_CP_BLOCK_ALL;      // every key of the chunk precedes every query
    if (ck == cq) return VLC_CP_BLOCK_CAUSAL;  // the chunk's own keys: causal
    return VLC_CP_BLOCK_NONE;                  // every key follows every query
}
