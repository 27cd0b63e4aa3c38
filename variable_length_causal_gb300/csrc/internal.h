// internal.h -- declarations shared by the C-ABI layer and the kernels.
#pragma once
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace vlc {

constexpr int kFwdBM = 128;   // query rows per tile (dQ pass work list)
constexpr int kFwdQB = 256;   // query rows per forward work unit (two q tiles)
constexpr int kFwdBN = 128;   // key rows per forward tile
constexpr int kBwdBM = 128;   // query rows per backward (key-major pass) step
constexpr int kTablePad = 128;  // RoPE table rows are padded to a multiple of this
constexpr uint32_t kWaitLimitUs = 2000000u;   // default limit of one bounded wait in a kernel (2 s)

// Workspace header (first 256 bytes).
struct WsHeader {
    int32_t err;          // VLC_DEVERR_* bits
    int32_t count;        // work items written by the work-list kernel
    int32_t count2;       // items of the second work list (backward key-major pass)
    int32_t next[3];      // dynamic unit counters of the attention kernels (zeroed per call)
    int32_t pad[58];
};

// Byte offsets of the workspace regions for one problem size.
struct WsLayout {
    size_t header, items, order, seg_base, table, table2, delta, qrot, krot, total;
    size_t total_min;          // forward: the bytes needed without the rotated-k copy (its fallback)
    int64_t item_cap;
    int32_t table_rows;
};

// total_kv / max_seqlen_kv < 0: self-attention (the query sizes).
WsLayout ws_layout(int32_t nseg, int32_t total, int32_t H, int32_t Hkv, int32_t d,
                   int32_t max_seqlen, int is_bwd, int32_t total_kv = -1, int32_t max_seqlen_kv = -1);

// Kernel launchers (return cudaGetLastError()).
cudaError_t launch_positions_labels(const int32_t* cu, int32_t nseg, const int64_t* tokens,
                                    int32_t total, const uint8_t* seg_ignore, int32_t* pos,
                                    int64_t* labels, int32_t* err, cudaStream_t s);

// Arguments of one work-list build (see launch_worklist) and of one RoPE table fill.
struct WlSpec {
    const int32_t* cu;
    int32_t nseg, total, max_seqlen, BM, BN;
    int kind;
    int4* items;
    int64_t cap;
    int32_t* order;
    int32_t* seg_base;
    int32_t* count;
    int32_t* err;
    const int32_t* cu_padded;
    const int32_t* cu_kv;
    int32_t total_kv, max_seqlen_kv;
    int all_visible;   // every key of a segment visible to every query (ranges as if the diagonal were past Lk)
};
struct TabSpec {
    float2* table;
    float2* table2;   // null: no blocked copy
    int32_t rows, half;
    double log2_theta;
};
TabSpec rope_table_spec(float2* table, int32_t rows, int32_t d, double theta, float2* table2 = nullptr);

// One kernel launch for up to two work lists and (tab != null) a RoPE table fill,
// which run side by side in separate blocks.
cudaError_t launch_meta(const WlSpec* lists, int nwl, const TabSpec* tab, cudaStream_t s);

cudaError_t launch_worklist(const int32_t* cu, int32_t nseg, int32_t total, int32_t max_seqlen,
                            int32_t BM, int32_t BN, int kind, int4* items, int64_t cap,
                            int32_t* order, int32_t* seg_base, int32_t* count, int32_t* err,
                            cudaStream_t s, const int32_t* cu_padded = nullptr,
                            const int32_t* cu_kv = nullptr, int32_t total_kv = 0,
                            int32_t max_seqlen_kv = 0);

// Padded layouts: zero the padding rows [cu_padded[r] + L_r, cu_padded[r+1]) of up
// to three bf16 row-major tensors (row_bytes each; null to skip) and set those
// columns of lse ([H, total], null to skip) to -inf.  No-op if *err != 0.
cudaError_t launch_pad_fill(const int32_t* cu, const int32_t* cu_padded, int32_t nseg, int32_t total,
                            void* a, int64_t a_row_bytes, void* b, int64_t b_row_bytes, void* c,
                            int64_t c_row_bytes, float* lse, int32_t H, const int32_t* err,
                            int num_sms, cudaStream_t s);

// table2 (optional): the same values blocked by four frequencies, [d/8][rows][4].
cudaError_t launch_rope_table(float2* table, int32_t rows, int32_t d, double theta,
                              const int32_t* err, cudaStream_t s, float2* table2 = nullptr);

// RoPE modes of FwdParams::use_rope / BwdParams::use_rope.
constexpr int kRopeNone = 0, kRopeHalf = 1, kRopeInterleaved = 2;

struct FwdParams {
    const void* q;
    const void* k;
    const void* v;
    void* o;
    float* lse;
    const int32_t* cu;
    const int32_t* rows;       // [nseg+1] first row of each segment (cu_padded, or cu if unpadded)
    const int32_t* cu_kv;      // [nseg+1] key/value segments (== cu for self-attention)
    const int32_t* rows_kv;    // [nseg+1] first key/value row of each segment (== rows for self-attention)
    const int4* items;
    const int32_t* seg_base;   // [nseg+1] item offsets of the sorted segments
    const int32_t* count;
    int32_t* next;             // unit counter (zeroed before the launch)
    int32_t* err;
    const float2* table;       // RoPE cos/sin [rows][d/2], null if no RoPE
    const void* krot;          // R(p) k of every key row (rotated beforehand), or null
    void* qrot_out;            // with krot: the kernel also writes R(p) q here (bf16 [total, H, d]), or null
    int32_t nseg, total, H, d;
    int32_t Hkv;               // key/value heads; query head h reads head h / (H / Hkv)
    int32_t total_kv;          // key/value rows (== total for self-attention)
    float scale_log2;          // softmax_scale * log2(e)
    int use_rope;              // kRopeNone, kRopeHalf (rotate-half pairs) or kRopeInterleaved
    uint32_t wait_limit_us;    // limit of one bounded wait in the kernel (kWaitLimitUs by default)
    int keys_all_visible;      // 1: every key of a query's key segment is visible (no causal mask;
                               // separate key segments, operands rotated beforehand)
};

cudaError_t launch_attn_fwd(const FwdParams& p, int num_sms, cudaStream_t s);

// R(p) k into krot for every key row, keys at their own positions (0 .. Lk-1 of the key
// segment, p.cu_kv / p.rows_kv; rows past a padded segment's length become zeros): the
// pass of launch_rope_qk with no query heads.  No-op if *err != 0.
cudaError_t launch_rope_k(const FwdParams& p, void* krot, int num_sms, cudaStream_t s);

// R(p) q into qrot and R(p) k into krot for every row (self-attention; rows past
// a segment's length in a padded layout become zeros).  Uses p.q, p.k, p.cu,
// p.rows, p.nseg, p.total, p.H, p.Hkv, p.d, p.table, p.use_rope, p.err.
cudaError_t launch_rope_qk(const FwdParams& p, void* qrot, void* krot, int num_sms, cudaStream_t s);

struct BwdParams {
    const void* dout;
    const void* q;
    const void* k;
    const void* v;
    const void* o;
    const float* lse;
    void* dq;
    void* dk;
    void* dv;
    const int32_t* cu;
    const int32_t* rows;       // [nseg+1] first row of each segment (cu_padded, or cu if unpadded)
    const int32_t* cu_kv;      // [nseg+1] key/value segments (== cu for self-attention)
    const int32_t* rows_kv;    // [nseg+1] first key/value row of each segment (== rows for self-attention)
    const int4* items;         // q-tile items (dQ pass), as in the forward
    const int32_t* seg_base;
    const int32_t* count;
    const int4* items_k;       // key-tile items (dK/dV pass)
    const int32_t* seg_base_k;
    const int32_t* count_k;
    int32_t* next_q;           // unit counters of the dQ and dK/dV passes (zeroed per call)
    int32_t* next_k;
    int32_t* err;
    const float2* table;
    const float2* table2;      // the table blocked by four frequencies: [d/8][table_rows][4]
    int32_t table_rows;
    float* delta;              // [H, total]: rowsum(dO * O)
    void* qrot;                // [total, H, d] bf16: R(p) q (workspace; only with RoPE)
    void* krot;                // [total_kv, Hkv, d] bf16: R(p) k
    int32_t nseg, total, H, d;
    int32_t Hkv;               // key/value heads; query head h reads head h / (H / Hkv)
    int32_t total_kv;          // key/value rows (== total for self-attention)
    float scale;
    int use_rope;              // kRopeHalf / kRopeInterleaved: inputs are rotated in the prep
                               // pass with that pairing, gradients un-rotated; kRopeNone: no RoPE
    int operands_rotated;      // 1: q and k already hold R(p) q, R(p) k; only the gradients are
                               // un-rotated (the prep pass computes D alone)
    uint32_t wait_limit_us;    // limit of one bounded wait in the kernels (kWaitLimitUs by default)
    int keys_all_visible;      // 1: every key of a query's key segment is visible (no causal mask;
                               // separate key segments, no RoPE)
};

// Limit of one bounded wait for the attention kernels launched from now on (the
// process-wide setting of vlc_set_wait_limit_us).
uint32_t wait_limit_us();

cudaError_t launch_attn_bwd(const BwdParams& p, int num_sms, cudaStream_t s);

// Workspace of the shifted cross-entropy call: header (error word), per-row
// losses and valid flags, per-segment sums and counts.
struct CeLayout {
    size_t header, row_loss, row_valid, seg_loss, seg_count, total;
};
CeLayout ce_layout(int32_t total, int32_t nseg);

cudaError_t launch_shifted_ce(const void* logits, int32_t vocab, int32_t total, const int64_t* labels,
                              const int32_t* cu, int32_t nseg, float* loss_sum, int64_t* count,
                              float* seg_loss, int32_t* seg_count, uint8_t* ws, cudaStream_t s);

}  // namespace vlc
