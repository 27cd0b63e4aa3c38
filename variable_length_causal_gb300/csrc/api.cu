// api.cu -- the extern "C" boundary declared in include/vlc.h: host-side
// argument checks, workspace layout, TMA descriptor encoding and the launch
// sequence of each call.  No device memory is allocated here.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/vlc.h"
#include "internal.h"

namespace vlc {

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

static int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

WsLayout ws_layout(int32_t nseg, int32_t total, int32_t H, int32_t Hkv, int32_t d,
                   int32_t max_seqlen, int is_bwd, int32_t total_kv, int32_t max_seqlen_kv) {
    WsLayout L{};
    const bool qkv = total_kv >= 0;
    if (!qkv) {
        total_kv = total;
        max_seqlen_kv = max_seqlen;
    }
    const int min_tile = is_bwd ? (kBwdBM < kFwdBM ? kBwdBM : kFwdBM) : kFwdBM;
    const int32_t rows_max = total > total_kv ? total : total_kv;
    L.item_cap = static_cast<int64_t>(nseg) + static_cast<int64_t>(rows_max) / min_tile + 1;
    // RoPE positions reach the last key tile; bottom-right aligned queries of a partial
    // first tile reach up to one tile further
    const int32_t max_pos = max_seqlen > max_seqlen_kv ? max_seqlen : max_seqlen_kv;
    L.table_rows = static_cast<int32_t>(ceil_div64(max_pos, kTablePad) * kTablePad + (qkv ? kTablePad : 0));
    size_t off = 0;
    L.header = off;
    off = align256(off + sizeof(WsHeader));
    L.items = off;
    off = align256(off + sizeof(int4) * static_cast<size_t>(L.item_cap) * (is_bwd ? 2 : 1));
    L.order = off;
    off = align256(off + sizeof(int32_t) * static_cast<size_t>(nseg) * (is_bwd ? 2 : 1));
    L.seg_base = off;
    off = align256(off + sizeof(int32_t) * static_cast<size_t>(nseg + 1) * (is_bwd ? 2 : 1));
    L.table = off;
    off = align256(off + sizeof(float2) * static_cast<size_t>(L.table_rows) * (d / 2));
    L.table2 = L.delta = L.qrot = L.krot = off;
    if (is_bwd) {
        L.table2 = off;
        off = align256(off + sizeof(float2) * static_cast<size_t>(L.table_rows) * (d / 2));
        L.delta = off;
        off = align256(off + sizeof(float) * static_cast<size_t>(H) * total);
        L.qrot = off;
        off = align256(off + static_cast<size_t>(total) * H * d * 2);
        L.krot = off;
        off = align256(off + static_cast<size_t>(total_kv) * Hkv * d * 2);
    }
    L.total_min = off;
    if (!is_bwd) {   // the forward's rotated copy of k, used when the workspace has room
        L.krot = off;
        off = align256(off + static_cast<size_t>(total_kv) * Hkv * d * 2);
    }
    L.total = off;
    return L;
}

// Limit of one bounded wait in the attention kernels (vlc_set_wait_limit_us).
static std::atomic<uint32_t> g_wait_limit_us{kWaitLimitUs};
uint32_t wait_limit_us() { return g_wait_limit_us.load(std::memory_order_relaxed); }

static int num_sms_cached() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n;
    }
    return cache[dev];
}

// ---------------------------------------------------------------- TMA descriptors
static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// [total, H, d] bf16, boxes of 64 (d) x 1 (head) x box_rows (tokens), 128-byte swizzle.
// Rows past `total` read as zeros.
bool make_tmap_thd(CUtensorMap* map, const void* base, int32_t total, int32_t H, int32_t d,
                   int box_rows) {
    auto enc = get_encode();
    if (enc == nullptr) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                          static_cast<cuuint64_t>(total)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                             static_cast<cuuint64_t>(H) * static_cast<cuuint64_t>(d) * 2};
    cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace vlc

using namespace vlc;

static bool aligned(const void* p, size_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// Arguments of one attention call (forward or backward).  cu_kv == nullptr is
// self-attention (keys and values segmented like the queries, total_kv and
// max_seqlen_kv taken from the query side).
struct AttnArgs {
    const void *q, *k, *v, *dout, *o_in;
    const float* lse_in;
    const int32_t *cu, *cu_padded, *cu_kv;
    int32_t nseg, total, total_kv, H, Hkv, d, max_seqlen, max_seqlen_kv;
    float softmax_scale, rope_theta;
    uint32_t flags;
    void* o;
    float* lse;
    void *dq, *dk, *dv;
    void* ws;
    size_t ws_bytes;
    void* stream;
    void *qrot_out, *krot_out;   // forward: also return R(p) q and R(p) k (vlc_attn_fwd_rot)
};

static int check_attn_args(const AttnArgs& a, int is_bwd) {
    if (a.nseg < 1 || a.total < 1 || a.H < 1 || a.max_seqlen < 1) return VLC_ERR_ARG;
    if (a.cu_kv != nullptr && (a.total_kv < 1 || a.max_seqlen_kv < 1)) return VLC_ERR_ARG;
    if (a.Hkv < 1 || a.H % a.Hkv != 0) return VLC_ERR_ARG;
    if (a.flags & ~static_cast<uint32_t>(VLC_ROPE_INTERLEAVED | VLC_QK_ROTATED | VLC_KEYS_ALL_VISIBLE))
        return VLC_ERR_ARG;
    // the backward takes rotated operands for self-attention only (the operands of vlc_rope_qk)
    if (is_bwd && (a.flags & VLC_QK_ROTATED) && a.cu_kv != nullptr) return VLC_ERR_ARG;
    if (a.flags & VLC_KEYS_ALL_VISIBLE) {
        // a block of keys that all precede the queries: separate key segments, and no
        // in-kernel rotation (the positions are not implied by the lengths); the backward
        // returns the gradients with respect to the operands as given (rope_theta == 0)
        if (a.cu_kv == nullptr) return VLC_ERR_ARG;
        if (is_bwd ? a.rope_theta != 0.f : !((a.flags & VLC_QK_ROTATED) || a.rope_theta == 0.f)) return VLC_ERR_ARG;
    }
    if (!(a.rope_theta >= 0.f) || !std::isfinite(a.rope_theta)) return VLC_ERR_ARG;
    if (a.d != 64 && a.d != 128) return VLC_ERR_UNSUPPORTED;
    if (a.max_seqlen > VLC_MAX_SEQLEN || a.max_seqlen_kv > VLC_MAX_SEQLEN) return VLC_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(a.total) * a.H * a.d > (int64_t(1) << 40)) return VLC_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(a.total_kv) * a.Hkv * a.d > (int64_t(1) << 40)) return VLC_ERR_UNSUPPORTED;
    if (a.ws == nullptr || !aligned(a.ws, 256)) return VLC_ERR_WORKSPACE;
    const bool qkv = a.cu_kv != nullptr;
    if (a.ws_bytes < ws_layout(a.nseg, a.total, a.H, a.Hkv, a.d, a.max_seqlen, is_bwd, qkv ? a.total_kv : -1,
                               qkv ? a.max_seqlen_kv : -1).total_min)
        return VLC_ERR_WORKSPACE;
    return VLC_OK;
}

static int rope_mode(float rope_theta, uint32_t flags) {
    if (rope_theta == 0.f) return kRopeNone;
    return (flags & VLC_ROPE_INTERLEAVED) ? kRopeInterleaved : kRopeHalf;
}

static int attn_fwd_impl(AttnArgs a) {
    if (a.q == nullptr || a.k == nullptr || a.v == nullptr || a.cu == nullptr || a.o == nullptr ||
        a.lse == nullptr)
        return VLC_ERR_ARG;
    const bool qkv = a.cu_kv != nullptr;
    if (!qkv) {
        a.total_kv = a.total;
        a.max_seqlen_kv = a.max_seqlen;
    }
    int st = check_attn_args(a, 0);
    if (st != VLC_OK) return st;
    if (!aligned(a.q, 16) || !aligned(a.k, 16) || !aligned(a.v, 16) || !aligned(a.o, 16) || !aligned(a.lse, 4))
        return VLC_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(a.stream);
    const WsLayout L = ws_layout(a.nseg, a.total, a.H, a.Hkv, a.d, a.max_seqlen, 0, qkv ? a.total_kv : -1,
                                 qkv ? a.max_seqlen_kv : -1);
    uint8_t* w = static_cast<uint8_t*>(a.ws);
    WsHeader* hdr = reinterpret_cast<WsHeader*>(w + L.header);
    int4* items = reinterpret_cast<int4*>(w + L.items);
    int32_t* order = reinterpret_cast<int32_t*>(w + L.order);
    int32_t* seg_base = reinterpret_cast<int32_t*>(w + L.seg_base);
    float2* table = reinterpret_cast<float2*>(w + L.table);

    if (cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s) != cudaSuccess) return VLC_ERR_CUDA;
    // operands rotated by vlc_rope_qk: the forward applies no rotation of its own
    const int mode = (a.flags & VLC_QK_ROTATED) ? kRopeNone : rope_mode(a.rope_theta, a.flags);
    {   // the work list and (with RoPE) the cos/sin table in one launch
        const WlSpec wl{a.cu, a.nseg, a.total, a.max_seqlen, kFwdQB, kFwdBN, VLC_WORKLIST_FWD, items,
                        L.item_cap, order, seg_base, &hdr->count, &hdr->err, a.cu_padded, a.cu_kv,
                        a.total_kv, a.max_seqlen_kv, (a.flags & VLC_KEYS_ALL_VISIBLE) ? 1 : 0};
        const TabSpec tab = rope_table_spec(table, L.table_rows, a.d, static_cast<double>(a.rope_theta));
        if (launch_meta(&wl, 1, mode != kRopeNone ? &tab : nullptr, s) != cudaSuccess) return VLC_ERR_CUDA;
    }
    if (a.cu_padded != nullptr &&
        launch_pad_fill(a.cu, a.cu_padded, a.nseg, a.total, a.o, int64_t(a.H) * a.d * 2, nullptr, 0, nullptr,
                        0, a.lse, a.H, &hdr->err, num_sms_cached(), s) != cudaSuccess)
        return VLC_ERR_CUDA;
    FwdParams p{};
    p.q = a.q; p.k = a.k; p.v = a.v; p.o = a.o; p.lse = a.lse; p.cu = a.cu;
    p.rows = a.cu_padded != nullptr ? a.cu_padded : a.cu;
    p.cu_kv = qkv ? a.cu_kv : a.cu;
    p.rows_kv = qkv ? a.cu_kv : p.rows;
    p.items = items; p.seg_base = seg_base; p.count = &hdr->count; p.err = &hdr->err;
    p.next = &hdr->next[0];
    p.table = mode != kRopeNone ? table : nullptr;
    p.nseg = a.nseg; p.total = a.total; p.H = a.H; p.d = a.d; p.Hkv = a.Hkv; p.total_kv = a.total_kv;
    const float scale = a.softmax_scale > 0.f ? a.softmax_scale : 1.0f / std::sqrt(static_cast<float>(a.d));
    p.scale_log2 = scale * 1.4426950408889634f;
    p.use_rope = mode;
    p.wait_limit_us = wait_limit_us();
    p.keys_all_visible = (a.flags & VLC_KEYS_ALL_VISIBLE) ? 1 : 0;
    // k rotated once into the workspace (if it has room) for every segment: the kernel then
    // rotates only the q tiles, in its softmax warps; without the room, its RoPE warps rotate
    // every staged q and K tile
    p.krot = nullptr;
    p.qrot_out = a.qrot_out;
    void* krot = a.krot_out != nullptr ? a.krot_out : (a.ws_bytes >= L.total ? w + L.krot : nullptr);
    if (mode != kRopeNone && krot != nullptr) {
        if (launch_rope_k(p, krot, num_sms_cached(), s) != cudaSuccess) return VLC_ERR_CUDA;
        p.krot = krot;
    }
    if (launch_attn_fwd(p, num_sms_cached(), s) != cudaSuccess) return VLC_ERR_CUDA;
    return VLC_OK;
}

static int attn_bwd_impl(AttnArgs a) {
    if (a.dout == nullptr || a.q == nullptr || a.k == nullptr || a.v == nullptr || a.o_in == nullptr ||
        a.lse_in == nullptr || a.cu == nullptr || a.dq == nullptr || a.dk == nullptr || a.dv == nullptr)
        return VLC_ERR_ARG;
    const bool qkv = a.cu_kv != nullptr;
    if (!qkv) {
        a.total_kv = a.total;
        a.max_seqlen_kv = a.max_seqlen;
    }
    int st = check_attn_args(a, 1);
    if (st != VLC_OK) return st;
    for (const void* ptr : {a.dout, a.q, a.k, a.v, a.o_in, static_cast<const void*>(a.dq),
                            static_cast<const void*>(a.dk), static_cast<const void*>(a.dv)})
        if (!aligned(ptr, 16)) return VLC_ERR_ARG;
    if (!aligned(a.lse_in, 4)) return VLC_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(a.stream);
    const WsLayout L = ws_layout(a.nseg, a.total, a.H, a.Hkv, a.d, a.max_seqlen, 1, qkv ? a.total_kv : -1,
                                 qkv ? a.max_seqlen_kv : -1);
    uint8_t* w = static_cast<uint8_t*>(a.ws);
    WsHeader* hdr = reinterpret_cast<WsHeader*>(w + L.header);
    int4* items_q = reinterpret_cast<int4*>(w + L.items);
    int4* items_k = items_q + L.item_cap;
    int32_t* order = reinterpret_cast<int32_t*>(w + L.order);
    int32_t* seg_base_q = reinterpret_cast<int32_t*>(w + L.seg_base);
    int32_t* seg_base_k = seg_base_q + (a.nseg + 1);
    float2* table = reinterpret_cast<float2*>(w + L.table);

    if (cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s) != cudaSuccess) return VLC_ERR_CUDA;
    const int mode = rope_mode(a.rope_theta, a.flags);
    float2* table2 = reinterpret_cast<float2*>(w + L.table2);
    {   // q-tile items (dQ pass), key-tile items (dK/dV pass) and the cos/sin tables in one launch
        const int allv = (a.flags & VLC_KEYS_ALL_VISIBLE) ? 1 : 0;
        const WlSpec wl[2] = {
            {a.cu, a.nseg, a.total, a.max_seqlen, kFwdBM, kFwdBN, VLC_WORKLIST_FWD, items_q, L.item_cap, order,
             seg_base_q, &hdr->count, &hdr->err, a.cu_padded, a.cu_kv, a.total_kv, a.max_seqlen_kv, allv},
            {a.cu, a.nseg, a.total, a.max_seqlen, kBwdBM, kFwdBN, VLC_WORKLIST_BWD, items_k, L.item_cap,
             order + a.nseg, seg_base_k, &hdr->count2, &hdr->err, a.cu_padded, a.cu_kv, a.total_kv,
             a.max_seqlen_kv, allv}};
        const TabSpec tab = rope_table_spec(table, L.table_rows, a.d, static_cast<double>(a.rope_theta), table2);
        if (launch_meta(wl, 2, mode != kRopeNone ? &tab : nullptr, s) != cudaSuccess) return VLC_ERR_CUDA;
    }
    if (a.cu_padded != nullptr &&
        launch_pad_fill(a.cu, a.cu_padded, a.nseg, a.total, a.dq, int64_t(a.H) * a.d * 2, a.dk,
                        int64_t(a.Hkv) * a.d * 2, a.dv, int64_t(a.Hkv) * a.d * 2, nullptr, a.H, &hdr->err,
                        num_sms_cached(), s) != cudaSuccess)
        return VLC_ERR_CUDA;
    BwdParams p{};
    p.dout = a.dout; p.q = a.q; p.k = a.k; p.v = a.v; p.o = a.o_in; p.lse = a.lse_in;
    p.dq = a.dq; p.dk = a.dk; p.dv = a.dv; p.cu = a.cu;
    p.rows = a.cu_padded != nullptr ? a.cu_padded : a.cu;
    p.cu_kv = qkv ? a.cu_kv : a.cu;
    p.rows_kv = qkv ? a.cu_kv : p.rows;
    p.items = items_q; p.seg_base = seg_base_q; p.count = &hdr->count; p.err = &hdr->err;
    p.items_k = items_k; p.seg_base_k = seg_base_k; p.count_k = &hdr->count2;
    p.next_q = &hdr->next[1];
    p.next_k = &hdr->next[2];
    p.table = mode != kRopeNone ? table : nullptr;
    p.table2 = mode != kRopeNone ? table2 : nullptr;
    p.table_rows = L.table_rows;
    p.delta = reinterpret_cast<float*>(w + L.delta);
    p.qrot = w + L.qrot;
    p.krot = w + L.krot;
    p.nseg = a.nseg; p.total = a.total; p.H = a.H; p.d = a.d; p.Hkv = a.Hkv; p.total_kv = a.total_kv;
    p.scale = a.softmax_scale > 0.f ? a.softmax_scale : 1.0f / std::sqrt(static_cast<float>(a.d));
    p.use_rope = mode;
    p.operands_rotated = (a.flags & VLC_QK_ROTATED) ? 1 : 0;
    p.wait_limit_us = wait_limit_us();
    p.keys_all_visible = (a.flags & VLC_KEYS_ALL_VISIBLE) ? 1 : 0;
    if (launch_attn_bwd(p, num_sms_cached(), s) != cudaSuccess) return VLC_ERR_CUDA;
    return VLC_OK;
}

static AttnArgs fwd_args(const void* q, const void* k, const void* v, const int32_t* cu,
                         const int32_t* cu_padded, const int32_t* cu_kv, int32_t nseg, int32_t total,
                         int32_t total_kv, int32_t H, int32_t H_kv, int32_t d, int32_t max_seqlen,
                         int32_t max_seqlen_kv, float softmax_scale, float rope_theta, uint32_t flags,
                         void* o, float* lse, void* ws, size_t ws_bytes, void* stream) {
    AttnArgs a{};
    a.q = q; a.k = k; a.v = v; a.cu = cu; a.cu_padded = cu_padded; a.cu_kv = cu_kv;
    a.nseg = nseg; a.total = total; a.total_kv = total_kv; a.H = H; a.Hkv = H_kv; a.d = d;
    a.max_seqlen = max_seqlen; a.max_seqlen_kv = max_seqlen_kv;
    a.softmax_scale = softmax_scale; a.rope_theta = rope_theta; a.flags = flags;
    a.o = o; a.lse = lse; a.ws = ws; a.ws_bytes = ws_bytes; a.stream = stream;
    return a;
}

static AttnArgs bwd_args(const void* dout, const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const int32_t* cu, const int32_t* cu_padded, const int32_t* cu_kv,
                         int32_t nseg, int32_t total, int32_t total_kv, int32_t H, int32_t H_kv, int32_t d,
                         int32_t max_seqlen, int32_t max_seqlen_kv, float softmax_scale, float rope_theta,
                         uint32_t flags, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, void* stream) {
    AttnArgs a = fwd_args(q, k, v, cu, cu_padded, cu_kv, nseg, total, total_kv, H, H_kv, d, max_seqlen,
                          max_seqlen_kv, softmax_scale, rope_theta, flags, nullptr, nullptr, ws, ws_bytes,
                          stream);
    a.dout = dout; a.o_in = o; a.lse_in = lse; a.dq = dq; a.dk = dk; a.dv = dv;
    return a;
}

extern "C" {

const char* vlc_status_string(int status) {
    switch (status) {
        case VLC_OK: return "ok";
        case VLC_ERR_ARG: return "invalid argument";
        case VLC_ERR_CU_SEQLENS: return "invalid cu_seqlens / max_seqlen";
        case VLC_ERR_UNSUPPORTED: return "unsupported shape";
        case VLC_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case VLC_ERR_CUDA: return "CUDA error";
        case VLC_ERR_TIMEOUT: return "device wait timed out";
        case VLC_ERR_LABEL: return "label outside [0, vocab) and not -100";
        default: return "unknown status";
    }
}

int vlc_version(void) { return 100; }

void vlc_set_wait_limit_us(uint32_t us) {
    vlc::g_wait_limit_us.store(us == 0 || us > vlc::kWaitLimitUs ? vlc::kWaitLimitUs : us, std::memory_order_relaxed);
}

size_t vlc_workspace_bytes_gqa(int32_t nseg, int32_t total, int32_t H, int32_t H_kv, int32_t d,
                               int32_t max_seqlen, int is_bwd) {
    if (nseg < 1 || total < 1 || H < 1 || H_kv < 1 || H % H_kv != 0 || (d != 64 && d != 128) ||
        max_seqlen < 1 || max_seqlen > VLC_MAX_SEQLEN)
        return 0;
    return ws_layout(nseg, total, H, H_kv, d, max_seqlen, is_bwd ? 1 : 0).total;
}

size_t vlc_workspace_bytes(int32_t nseg, int32_t total, int32_t H, int32_t d, int32_t max_seqlen,
                           int is_bwd) {
    return vlc_workspace_bytes_gqa(nseg, total, H, H, d, max_seqlen, is_bwd);
}

int64_t vlc_worklist_capacity(int32_t nseg, int32_t total, int32_t tile) {
    if (nseg < 1 || total < 1 || tile < 1) return 0;
    return static_cast<int64_t>(nseg) + static_cast<int64_t>(total) / tile + 1;
}

int vlc_build_positions_labels(const int32_t* cu, int32_t nseg, const int64_t* tokens,
                               int32_t total, const uint8_t* seg_ignore, int32_t* pos_out,
                               int64_t* labels_out, int32_t* err_out, void* stream) {
    if (cu == nullptr || tokens == nullptr || pos_out == nullptr || labels_out == nullptr)
        return VLC_ERR_ARG;
    if (nseg < 1 || total < 1) return VLC_ERR_ARG;
    if (!aligned(tokens, 8) || !aligned(pos_out, 4) || !aligned(labels_out, 8)) return VLC_ERR_ARG;
    cudaError_t e = launch_positions_labels(cu, nseg, tokens, total, seg_ignore, pos_out,
                                            labels_out, err_out,
                                            static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? VLC_OK : VLC_ERR_CUDA;
}

int vlc_build_worklist(const int32_t* cu, int32_t nseg, int32_t total, int32_t max_seqlen,
                       int32_t BM, int32_t BN, int kind, int32_t* items_out, int64_t capacity,
                       int32_t* seg_order_out, int32_t* count_out, int32_t* err_out,
                       void* stream) {
    if (cu == nullptr || items_out == nullptr || seg_order_out == nullptr ||
        count_out == nullptr || err_out == nullptr)
        return VLC_ERR_ARG;
    if (nseg < 1 || total < 1 || max_seqlen < 1) return VLC_ERR_ARG;
    if (kind != VLC_WORKLIST_FWD && kind != VLC_WORKLIST_BWD) return VLC_ERR_ARG;
    auto pow2ok = [](int32_t t) { return t >= 16 && t <= 256 && (t & (t - 1)) == 0; };
    if (!pow2ok(BM) || !pow2ok(BN)) return VLC_ERR_ARG;
    if (max_seqlen > VLC_MAX_SEQLEN) return VLC_ERR_UNSUPPORTED;
    const int32_t tile = (kind == VLC_WORKLIST_FWD) ? BM : BN;
    if (ceil_div64(max_seqlen, tile) + 1 > 16384) return VLC_ERR_UNSUPPORTED;
    if (capacity < vlc_worklist_capacity(nseg, total, tile)) return VLC_ERR_WORKSPACE;
    if (!aligned(items_out, 16)) return VLC_ERR_ARG;
    cudaError_t e = launch_worklist(cu, nseg, total, max_seqlen, BM, BN, kind,
                                    reinterpret_cast<int4*>(items_out), capacity, seg_order_out,
                                    seg_order_out + nseg, count_out, err_out,
                                    static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? VLC_OK : VLC_ERR_CUDA;
}

int vlc_attn_fwd_ex(const void* q, const void* k, const void* v, const int32_t* cu,
                    const int32_t* cu_padded, int32_t nseg, int32_t total, int32_t H, int32_t H_kv,
                    int32_t d, int32_t max_seqlen, float softmax_scale, float rope_theta,
                    uint32_t flags, void* o, float* lse, void* ws, size_t ws_bytes, void* stream) {
    return attn_fwd_impl(fwd_args(q, k, v, cu, cu_padded, nullptr, nseg, total, 0, H, H_kv, d, max_seqlen, 0,
                                  softmax_scale, rope_theta, flags, o, lse, ws, ws_bytes, stream));
}

int vlc_attn_fwd_rot(const void* q, const void* k, const void* v, const int32_t* cu, int32_t nseg,
                     int32_t total, int32_t H, int32_t H_kv, int32_t d, int32_t max_seqlen,
                     float softmax_scale, float rope_theta, uint32_t flags, void* o, float* lse,
                     void* qrot, void* krot, void* ws, size_t ws_bytes, void* stream) {
    if (qrot == nullptr || krot == nullptr || !aligned(qrot, 16) || !aligned(krot, 16)) return VLC_ERR_ARG;
    if (!(rope_theta > 0.f) || (flags & ~static_cast<uint32_t>(VLC_ROPE_INTERLEAVED))) return VLC_ERR_ARG;
    AttnArgs a = fwd_args(q, k, v, cu, nullptr, nullptr, nseg, total, 0, H, H_kv, d, max_seqlen, 0, softmax_scale,
                          rope_theta, flags, o, lse, ws, ws_bytes, stream);
    a.qrot_out = qrot;
    a.krot_out = krot;
    return attn_fwd_impl(a);
}

int vlc_attn_fwd_gqa(const void* q, const void* k, const void* v, const int32_t* cu, int32_t nseg,
                     int32_t total, int32_t H, int32_t H_kv, int32_t d, int32_t max_seqlen,
                     float softmax_scale, float rope_theta, void* o, float* lse, void* ws,
                     size_t ws_bytes, void* stream) {
    return vlc_attn_fwd_ex(q, k, v, cu, nullptr, nseg, total, H, H_kv, d, max_seqlen, softmax_scale,
                           rope_theta, 0u, o, lse, ws, ws_bytes, stream);
}

int vlc_attn_fwd(const void* q, const void* k, const void* v, const int32_t* cu, int32_t nseg,
                 int32_t total, int32_t H, int32_t d, int32_t max_seqlen, float softmax_scale,
                 float rope_theta, void* o, float* lse, void* ws, size_t ws_bytes, void* stream) {
    return vlc_attn_fwd_gqa(q, k, v, cu, nseg, total, H, H, d, max_seqlen, softmax_scale, rope_theta,
                            o, lse, ws, ws_bytes, stream);
}

int vlc_attn_bwd_ex(const void* dout, const void* q, const void* k, const void* v, const void* o,
                    const float* lse, const int32_t* cu, const int32_t* cu_padded, int32_t nseg,
                    int32_t total, int32_t H, int32_t H_kv, int32_t d, int32_t max_seqlen,
                    float softmax_scale, float rope_theta, uint32_t flags, void* dq, void* dk,
                    void* dv, void* ws, size_t ws_bytes, void* stream) {
    return attn_bwd_impl(bwd_args(dout, q, k, v, o, lse, cu, cu_padded, nullptr, nseg, total, 0, H, H_kv, d,
                                  max_seqlen, 0, softmax_scale, rope_theta, flags, dq, dk, dv, ws, ws_bytes,
                                  stream));
}

int vlc_attn_bwd_gqa(const void* dout, const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const int32_t* cu, int32_t nseg, int32_t total, int32_t H,
                     int32_t H_kv, int32_t d, int32_t max_seqlen, float softmax_scale,
                     float rope_theta, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                     void* stream) {
    return vlc_attn_bwd_ex(dout, q, k, v, o, lse, cu, nullptr, nseg, total, H, H_kv, d, max_seqlen,
                           softmax_scale, rope_theta, 0u, dq, dk, dv, ws, ws_bytes, stream);
}

int vlc_attn_bwd(const void* dout, const void* q, const void* k, const void* v, const void* o,
                 const float* lse, const int32_t* cu, int32_t nseg, int32_t total, int32_t H,
                 int32_t d, int32_t max_seqlen, float softmax_scale, float rope_theta, void* dq,
                 void* dk, void* dv, void* ws, size_t ws_bytes, void* stream) {
    return vlc_attn_bwd_gqa(dout, q, k, v, o, lse, cu, nseg, total, H, H, d, max_seqlen, softmax_scale,
                            rope_theta, dq, dk, dv, ws, ws_bytes, stream);
}

int vlc_rope_qk(const void* q, const void* k, const int32_t* cu, const int32_t* cu_padded, int32_t nseg,
                int32_t total, int32_t H, int32_t H_kv, int32_t d, int32_t max_seqlen, float rope_theta,
                uint32_t flags, void* qrot, void* krot, void* ws, size_t ws_bytes, void* stream) {
    if (q == nullptr || k == nullptr || cu == nullptr || qrot == nullptr || krot == nullptr) return VLC_ERR_ARG;
    AttnArgs a = fwd_args(q, k, k, cu, cu_padded, nullptr, nseg, total, total, H, H_kv, d, max_seqlen, max_seqlen,
                          0.f, rope_theta, flags, nullptr, nullptr, ws, ws_bytes, stream);
    if (flags & ~static_cast<uint32_t>(VLC_ROPE_INTERLEAVED)) return VLC_ERR_ARG;
    int st = check_attn_args(a, 0);
    if (st != VLC_OK) return st;
    if (!(rope_theta > 0.f)) return VLC_ERR_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(qrot, 16) || !aligned(krot, 16)) return VLC_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const WsLayout L = ws_layout(nseg, total, H, H_kv, d, max_seqlen, 0);
    uint8_t* w = static_cast<uint8_t*>(ws);
    WsHeader* hdr = reinterpret_cast<WsHeader*>(w + L.header);
    float2* table = reinterpret_cast<float2*>(w + L.table);
    if (cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s) != cudaSuccess) return VLC_ERR_CUDA;
    // the work list validates cu (and cu_padded) before anything reads positions; the table,
    // which reads no input, is filled in the same launch
    const int mode = rope_mode(rope_theta, flags);
    {
        const WlSpec wl{cu, nseg, total, max_seqlen, kFwdQB, kFwdBN, VLC_WORKLIST_FWD,
                        reinterpret_cast<int4*>(w + L.items), L.item_cap, reinterpret_cast<int32_t*>(w + L.order),
                        reinterpret_cast<int32_t*>(w + L.seg_base), &hdr->count, &hdr->err, cu_padded, nullptr, 0,
                        0};
        const TabSpec tab = rope_table_spec(table, L.table_rows, d, static_cast<double>(rope_theta));
        if (launch_meta(&wl, 1, &tab, s) != cudaSuccess) return VLC_ERR_CUDA;
    }
    FwdParams p{};
    p.q = q; p.k = k; p.cu = cu;
    p.rows = cu_padded != nullptr ? cu_padded : cu;
    p.err = &hdr->err;
    p.table = table;
    p.nseg = nseg; p.total = total; p.H = H; p.Hkv = H_kv; p.d = d;
    p.use_rope = mode;
    if (launch_rope_qk(p, qrot, krot, num_sms_cached(), s) != cudaSuccess) return VLC_ERR_CUDA;
    return VLC_OK;
}

size_t vlc_workspace_bytes_qkv(int32_t nseg, int32_t total_q, int32_t total_kv, int32_t H, int32_t H_kv,
                               int32_t d, int32_t max_seqlen_q, int32_t max_seqlen_kv, int is_bwd) {
    if (nseg < 1 || total_q < 1 || total_kv < 1 || H < 1 || H_kv < 1 || H % H_kv != 0 ||
        (d != 64 && d != 128) || max_seqlen_q < 1 || max_seqlen_kv < 1 || max_seqlen_q > VLC_MAX_SEQLEN ||
        max_seqlen_kv > VLC_MAX_SEQLEN)
        return 0;
    return ws_layout(nseg, total_q, H, H_kv, d, max_seqlen_q, is_bwd ? 1 : 0, total_kv, max_seqlen_kv).total;
}

int vlc_attn_fwd_qkv(const void* q, const void* k, const void* v, const int32_t* cu_q,
                     const int32_t* cu_kv, int32_t nseg, int32_t total_q, int32_t total_kv, int32_t H,
                     int32_t H_kv, int32_t d, int32_t max_seqlen_q, int32_t max_seqlen_kv,
                     float softmax_scale, float rope_theta, uint32_t flags, void* o, float* lse, void* ws,
                     size_t ws_bytes, void* stream) {
    if (cu_kv == nullptr) return VLC_ERR_ARG;
    return attn_fwd_impl(fwd_args(q, k, v, cu_q, nullptr, cu_kv, nseg, total_q, total_kv, H, H_kv, d,
                                  max_seqlen_q, max_seqlen_kv, softmax_scale, rope_theta, flags, o, lse, ws,
                                  ws_bytes, stream));
}

int vlc_attn_bwd_qkv(const void* dout, const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const int32_t* cu_q, const int32_t* cu_kv, int32_t nseg,
                     int32_t total_q, int32_t total_kv, int32_t H, int32_t H_kv, int32_t d,
                     int32_t max_seqlen_q, int32_t max_seqlen_kv, float softmax_scale, float rope_theta,
                     uint32_t flags, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, void* stream) {
    if (cu_kv == nullptr) return VLC_ERR_ARG;
    return attn_bwd_impl(bwd_args(dout, q, k, v, o, lse, cu_q, nullptr, cu_kv, nseg, total_q, total_kv, H,
                                  H_kv, d, max_seqlen_q, max_seqlen_kv, softmax_scale, rope_theta, flags, dq,
                                  dk, dv, ws, ws_bytes, stream));
}

int vlc_get_error(const void* ws, int32_t* bits_out, void* stream) {
    if (ws == nullptr) return VLC_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t bits = 0;
    if (cudaMemcpyAsync(&bits, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return VLC_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return VLC_ERR_CUDA;
    if (bits_out != nullptr) *bits_out = bits;
    if (bits & VLC_DEVERR_TIMEOUT) return VLC_ERR_TIMEOUT;
    if (bits & VLC_DEVERR_POS) return VLC_ERR_ARG;
    if (bits & ~VLC_DEVERR_LABEL) return VLC_ERR_CU_SEQLENS;
    if (bits != 0) return VLC_ERR_LABEL;
    return VLC_OK;
}

size_t vlc_ce_workspace_bytes(int32_t total, int32_t nseg) {
    if (total < 1 || nseg < 1) return 0;
    return vlc::ce_layout(total, nseg).total;
}

int vlc_shifted_ce(const void* logits, int32_t vocab, int32_t total, const int64_t* labels,
                   const int32_t* cu, int32_t nseg, float* loss_sum, int64_t* target_count,
                   float* seg_loss, int32_t* seg_count, void* ws, size_t ws_bytes, void* stream) {
    if (cu == nullptr) nseg = 1;
    if (logits == nullptr || labels == nullptr || loss_sum == nullptr || target_count == nullptr ||
        vocab < 1 || total < 1 || nseg < 1)
        return VLC_ERR_ARG;
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) != 0 ||
        ws_bytes < vlc_ce_workspace_bytes(total, nseg))
        return VLC_ERR_WORKSPACE;
    const cudaError_t e = vlc::launch_shifted_ce(logits, vocab, total, labels, cu, nseg, loss_sum,
                                                 target_count, seg_loss, seg_count,
                                                 static_cast<uint8_t*>(ws), static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? VLC_OK : VLC_ERR_CUDA;
}

}  // extern "C"
