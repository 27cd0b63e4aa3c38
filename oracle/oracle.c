/*
 * oracle.c -- plain, slow fp64 CPU oracle for isolated sequence packing.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header, table or helper with the
 * CUDA library; it is written from the pages' statement of the method.
 *
 * Sources (page title, section):
 *  [CSTAR] "Sequence packing and variable-length attention" (charlestar.github.io)
 *      - "Nine tokens together keep three sample identities": cu_seqlens as a
 *        prefix sum, segment r = [cu_r, cu_{r+1}), local position p_i = i - cu_r,
 *        and the validity contract (cu[0]==0, strictly increasing,
 *        cu[-1]==total, max_seqlen == largest difference, int32 range).
 *      - "EOS is content; isolation happens before softmax":
 *        allow(i,j) = (s_i == s_j) and (p_j <= p_i); additive mask M (0 / -inf)
 *        added to QK^T/sqrt(d) before the softmax, O = softmax(QK^T/sqrt(d)+M) V.
 *      Grouped key/value heads (Hkv dividing H, query head h reading key/value head
 *      h / (H / Hkv)) are this library's extension of the pages' equal-head setting.
 *      - "Positions are reset per segment; the pure-RoPE argument": fixed-frequency
 *        RoPE rotation R(p) with (R(m+c)q)^T (R(n+c)k) = q^T R(n-m) k.
 *      - "After isolation one cross-boundary prediction pair remains": the
 *        pre-shifted label contract (ignore index -100 on each segment's last logit).
 *  [M020] "Length grouping, de-padding and packing" (xuujii ai-infra-kb M020),
 *      section 06 "positions and labels": targets [12,13,ignore,22,ignore].
 *  [COMPASS] "Sequence Packing" (brenchcc llm-compass), "Implementation notes":
 *      padding tail as its own segment whose labels are all -100.
 *  [CSTAR] "After isolation one cross-boundary prediction pair remains" and
 *      "Packing should not decide how much a long sample weighs": the next-token
 *      loss is kept as a sum of per-target cross-entropies plus a count of valid
 *      targets (ignore index -100), per sample and per pack, so the training loop
 *      chooses the denominator (token mean sum S / sum n, or sample mean of S_r / n_r).
 *
 * Everything is computed one segment at a time; there is no tiling, fusion or
 * reordering beyond the definitions above.  Inputs are the raw bf16 bit
 * patterns of q/k/v/dO (exactly representable in fp64); all arithmetic is fp64.
 *
 * "Contract" mode (contract == 1) rounds the RoPE-rotated q', k' to bf16
 * (round to nearest, ties to even) before the contraction, because the tensor
 * cores consume bf16 operands; the pages fix no precision for this step, and
 * exact mode (contract == 0) keeps them in fp64.  Gradients pass through that
 * rounding unchanged (straight-through).  contract == -1 selects exact mode
 * with fp64 input arrays instead of bf16 bit patterns (finite-difference tests).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_ERR_CU_FIRST 1     /* cu[0] != 0 */
#define ORC_ERR_CU_ORDER 2     /* some segment has length <= 0 */
#define ORC_ERR_CU_TOTAL 4     /* cu[nseg] != total */
#define ORC_ERR_MAXLEN 8       /* max_seqlen != largest segment length */
#define ORC_ERR_ARG 16         /* nseg < 1 or total < 1 */

/* ---------------------------------------------------------------- helpers */

/* bf16 bit pattern -> double.  A bf16 value is the upper 16 bits of an IEEE
 * binary32 value, so widening is exact. */
static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 value (8 significant bits, ties to even),
 * returned as a double.  Written from the definition: scale the significand to
 * [128, 256), round to an integer with ties to even, scale back.  Values in
 * the bf16 subnormal range are rounded at the fixed 2^-133 quantum. */
static double round_to_bf16(double x) {
    if (x == 0.0 || !isfinite(x)) return x;
    int e;
    double m = frexp(x, &e);          /* x = m * 2^e, 0.5 <= |m| < 1 */
    int shift = 8;
    if (e - 1 < -126) shift = 8 - ((-126) - (e - 1));   /* subnormal quantum */
    if (shift < 0) return 0.0 * x;
    double s = ldexp(m, shift);
    double r = floor(s);
    double frac = s - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
    return ldexp(r, e - shift);
}

/* RoPE angle for local position p and rotation pair j of a head of size d:
 * phi = p * theta^(-2j/d)  (fixed frequencies, rotate-half pairing). */
static double rope_angle(int64_t p, int j, int d, double theta) {
    return (double)p * pow(theta, -2.0 * (double)j / (double)d);
}

/* Elements of rotation pair j: rotate-half pairing (x_j, x_{j+d/2}) by default;
 * with interleaved != 0 the adjacent pairing (x_{2j}, x_{2j+1}) (the complex-number
 * form of RoFormer, which "Positions are reset per segment" cites; rotate-half is the
 * HF Llama form it also cites).  Both use frequency theta^(-2j/d) for pair j. */
static void rope_pair(int j, int d, int interleaved, int* ia, int* ib) {
    if (interleaved) { *ia = 2 * j; *ib = 2 * j + 1; }
    else { *ia = j; *ib = j + d / 2; }
}

/* Rotate one head vector x[0..d) by R(p):  x'_a = x_a cos - x_b sin,
 * x'_b = x_b cos + x_a sin  for every pair (a, b). */
static void rope_rotate(const double* x, double* out, int64_t p, int d, double theta,
                        int interleaved) {
    int half = d / 2;
    for (int j = 0; j < half; ++j) {
        double phi = rope_angle(p, j, d, theta);
        double c = cos(phi), s = sin(phi);
        int ia, ib;
        rope_pair(j, d, interleaved, &ia, &ib);
        double a = x[ia], b = x[ib];
        out[ia] = a * c - b * s;
        out[ib] = b * c + a * s;
    }
}

/* Transpose rotation R(p)^T = R(-p), used to carry gradients back through RoPE. */
static void rope_rotate_transpose(const double* g, double* out, int64_t p, int d, double theta,
                                  int interleaved) {
    int half = d / 2;
    for (int j = 0; j < half; ++j) {
        double phi = rope_angle(p, j, d, theta);
        double c = cos(phi), s = sin(phi);
        int ia, ib;
        rope_pair(j, d, interleaved, &ia, &ib);
        double a = g[ia], b = g[ib];
        out[ia] = a * c + b * s;
        out[ib] = b * c - a * s;
    }
}

/* ---------------------------------------------------------------- cu_seqlens */

/* Validity contract for cu_seqlens ([CSTAR], "Nine tokens together ..."). */
int orc_validate_cu(const int32_t* cu, int32_t nseg, int32_t total, int32_t max_seqlen) {
    if (nseg < 1 || total < 1) return ORC_ERR_ARG;
    int err = 0;
    if (cu[0] != 0) err |= ORC_ERR_CU_FIRST;
    int64_t longest = 0;
    for (int32_t r = 0; r < nseg; ++r) {
        int64_t len = (int64_t)cu[r + 1] - (int64_t)cu[r];
        if (len <= 0) err |= ORC_ERR_CU_ORDER;
        if (len > longest) longest = len;
    }
    if (cu[nseg] != total) err |= ORC_ERR_CU_TOTAL;
    if (longest != max_seqlen) err |= ORC_ERR_MAXLEN;
    return err;
}

/* Segment index of token i: the r with cu[r] <= i < cu[r+1], found by a
 * plain linear scan (the pages use searchsorted; the answer is the same). */
static int32_t segment_of(const int32_t* cu, int32_t nseg, int64_t i) {
    for (int32_t r = 0; r < nseg; ++r)
        if (i >= cu[r] && i < cu[r + 1]) return r;
    return -1;
}

/* Local positions p_i = i - cu_r and pre-shifted next-token labels:
 * label_i = token_{i+1} when i+1 is still inside segment r, else -100; every
 * label of an ignored segment (a padding tail) is -100. */
void orc_positions_labels(const int32_t* cu, int32_t nseg, const int64_t* tokens,
                          const uint8_t* seg_ignore, int32_t* pos, int64_t* labels) {
    int64_t total = cu[nseg];
    for (int64_t i = 0; i < total; ++i) {
        int32_t r = segment_of(cu, nseg, i);
        if (r < 0) { pos[i] = -1; labels[i] = -100; continue; }   /* invalid cu */
        pos[i] = (int32_t)(i - cu[r]);
        int ignored = seg_ignore != NULL && seg_ignore[r] != 0;
        if (!ignored && i + 1 < cu[r + 1])
            labels[i] = tokens[i + 1];
        else
            labels[i] = -100;
    }
}

/* ---------------------------------------------------------------- work lists */

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* Stable order of segments by descending tile count n_r = ceil(L_r / tile).
 * Plain insertion sort: O(nseg^2) worst case, fine for an oracle. */
static void order_segments(const int32_t* cu, int32_t nseg, int32_t tile, int32_t* order) {
    for (int32_t r = 0; r < nseg; ++r) order[r] = r;
    for (int32_t a = 1; a < nseg; ++a) {
        int32_t x = order[a];
        int64_t nx = ceil_div((int64_t)cu[x + 1] - cu[x], tile);
        int32_t b = a - 1;
        while (b >= 0) {
            int32_t y = order[b];
            int64_t ny = ceil_div((int64_t)cu[y + 1] - cu[y], tile);
            if (ny >= nx) break;        /* keep equal keys in index order */
            order[b + 1] = y;
            --b;
        }
        order[b + 1] = x;
    }
}

/* Forward work list: one item {seg, q_tile, kv_lo, kv_hi} per q tile of BM
 * rows of every segment.  Query row p (local) may see key rows 0..p of its own
 * segment only, so q tile t needs key tiles [0, ceil(min(L, (t+1)BM) / BN)).
 * No item refers to another segment, and no key tile lies wholly above the
 * diagonal.  Order: segments by descending q-tile count (ties by index), and
 * inside a segment q tiles from last to first (longest key range first).
 * Returns the item count, or -1 if cap is too small. */
int64_t orc_worklist_fwd(const int32_t* cu, int32_t nseg, int32_t BM, int32_t BN,
                         int32_t* items, int64_t cap) {
    int32_t* order = (int32_t*)malloc(sizeof(int32_t) * (size_t)nseg);
    order_segments(cu, nseg, BM, order);
    int64_t n = 0;
    for (int32_t k = 0; k < nseg; ++k) {
        int32_t r = order[k];
        int64_t L = (int64_t)cu[r + 1] - cu[r];
        int64_t nq = ceil_div(L, BM);
        for (int64_t t = nq - 1; t >= 0; --t) {
            if (n >= cap) { free(order); return -1; }
            int64_t last_row = (t + 1) * BM < L ? (t + 1) * BM : L;
            items[4 * n + 0] = r;
            items[4 * n + 1] = (int32_t)t;
            items[4 * n + 2] = 0;
            items[4 * n + 3] = (int32_t)ceil_div(last_row, BN);
            ++n;
        }
    }
    free(order);
    return n;
}

/* Backward work list: one item {seg, kv_tile, q_lo, q_hi} per key tile of BN
 * rows.  Key row j (local) is seen by query rows j..L-1, so key tile t is
 * needed by q tiles [floor(t*BN / BM), ceil(L / BM)).  Order: segments by
 * descending key-tile count (ties by index), key tiles first to last. */
int64_t orc_worklist_bwd(const int32_t* cu, int32_t nseg, int32_t BM, int32_t BN,
                         int32_t* items, int64_t cap) {
    int32_t* order = (int32_t*)malloc(sizeof(int32_t) * (size_t)nseg);
    order_segments(cu, nseg, BN, order);
    int64_t n = 0;
    for (int32_t k = 0; k < nseg; ++k) {
        int32_t r = order[k];
        int64_t L = (int64_t)cu[r + 1] - cu[r];
        int64_t nk = ceil_div(L, BN);
        for (int64_t t = 0; t < nk; ++t) {
            if (n >= cap) { free(order); return -1; }
            items[4 * n + 0] = r;
            items[4 * n + 1] = (int32_t)t;
            items[4 * n + 2] = (int32_t)((t * BN) / BM);
            items[4 * n + 3] = (int32_t)ceil_div(L, BM);
            ++n;
        }
    }
    free(order);
    return n;
}

/* ---------------------------------------------------------------- RoPE */

/* Apply R(pos[n]) to rows of x ([n][d] fp64).  Exposed so tests can probe the
 * rotation at arbitrary positions (shift invariance, R(0) = I, ...). */
void orc_rope_rows(const double* x, const int64_t* pos, int64_t n, int32_t d,
                   double theta, int interleaved, double* out) {
    for (int64_t i = 0; i < n; ++i) rope_rotate(x + i * d, out + i * d, pos[i], d, theta, interleaved);
}

/* ---------------------------------------------------------------- attention */

typedef struct {
    const void *q, *k, *v, *dout;       /* q / dO [total][H][d], k / v [total_kv][Hkv][d]: bf16
                                           bits, or fp64 when f64_inputs */
    int f64_inputs;
    const int32_t* cu;                   /* query segments */
    const int32_t* cu_kv;                /* key/value segments (the same array for self-attention) */
    int32_t nseg, total, total_kv, H, Hkv, d;   /* H % Hkv == 0 */
    double scale, theta;                 /* theta == 0: no RoPE */
    int contract;
    int rope_interleaved;                /* pairing of the rotation (rope_pair) */
} orc_problem;

/* Grouped heads: query head h reads key/value head h / (H / Hkv), so each run of
 * H / Hkv consecutive query heads shares one key/value head (Hkv == H is plain
 * multi-head attention). */
static int32_t kv_head(const orc_problem* P, int32_t h) { return h / (P->H / P->Hkv); }

/* Element c of token row i, head h of an input tensor, widened to fp64. */
static double input_elem(const orc_problem* P, const void* x, int64_t i, int32_t h, int c) {
    const int32_t nh = (x == P->k || x == P->v) ? P->Hkv : P->H;
    size_t off = ((size_t)i * nh + h) * P->d + c;
    if (P->f64_inputs) return ((const double*)x)[off];
    return bf16_bits_to_double(((const uint16_t*)x)[off]);
}

/* q' (or k') for token row i of head h: widen, rotate by position p, and round
 * to bf16 in contract mode. */
static void load_rotated(const orc_problem* P, const void* x, int64_t i, int32_t h,
                         int64_t p, double* out) {
    int d = P->d;
    double* tmp = (double*)malloc(sizeof(double) * (size_t)d);
    for (int c = 0; c < d; ++c) tmp[c] = input_elem(P, x, i, h, c);
    if (P->theta != 0.0) {
        rope_rotate(tmp, out, p, d, P->theta, P->rope_interleaved);
        if (P->contract)
            for (int c = 0; c < d; ++c) out[c] = round_to_bf16(out[c]);
    } else {
        memcpy(out, tmp, sizeof(double) * (size_t)d);
    }
    free(tmp);
}

static void load_plain(const orc_problem* P, const void* x, int64_t i, int32_t h, double* out) {
    for (int c = 0; c < P->d; ++c) out[c] = input_elem(P, x, i, h, c);
}

/* One segment r, one head h: Q', dO of its L queries and K', V of its Lk keys in
 * fp64.  Self-attention has Lk == L.  With Lk > L the queries are the last L
 * positions of the segment (bottom-right alignment, the convention for q and kv
 * of different lengths that "Sequence packing and variable-length attention"
 * says differs from the square case): query p sits at position p + off,
 * off = Lk - L, sees keys j <= p + off, and is rotated by that position. */
typedef struct {
    int64_t L, Lk, off, base, base_k;
    double *q, *g;          /* [L][d] */
    double *k, *v;          /* [Lk][d] */
} seg_head;

static void seg_head_load(const orc_problem* P, int32_t r, int32_t h, int want_grad, seg_head* S) {
    int d = P->d;
    S->base = P->cu[r];
    S->L = (int64_t)P->cu[r + 1] - P->cu[r];
    S->base_k = P->cu_kv[r];
    S->Lk = (int64_t)P->cu_kv[r + 1] - P->cu_kv[r];
    S->off = S->Lk - S->L;
    S->q = (double*)malloc(sizeof(double) * (size_t)S->L * d);
    S->g = want_grad ? (double*)malloc(sizeof(double) * (size_t)S->L * d) : NULL;
    S->k = (double*)malloc(sizeof(double) * (size_t)S->Lk * d);
    S->v = (double*)malloc(sizeof(double) * (size_t)S->Lk * d);
    for (int64_t p = 0; p < S->L; ++p) {
        int64_t i = S->base + p;
        load_rotated(P, P->q, i, h, p + S->off, S->q + p * d);
        if (want_grad) load_plain(P, P->dout, i, h, S->g + p * d);
    }
    for (int64_t j = 0; j < S->Lk; ++j) {
        load_rotated(P, P->k, S->base_k + j, kv_head(P, h), j, S->k + j * d);
        load_plain(P, P->v, S->base_k + j, kv_head(P, h), S->v + j * d);
    }
}

static void seg_head_free(seg_head* S) {
    free(S->q); free(S->k); free(S->v); free(S->g);
}

static double dot(const double* a, const double* b, int d) {
    double s = 0.0;
    for (int c = 0; c < d; ++c) s += a[c] * b[c];
    return s;
}

/* Masked softmax row p of one segment-head: scores s_j = q'_p . k'_j * scale
 * for the allowed keys j <= p + off (the -inf entries of the additive mask
 * contribute exp(-inf) = 0 to the normaliser), LSE_p = ln sum_j exp(s_j). */
static double softmax_row(const seg_head* S, int64_t p, int d, double scale, double* s) {
    const int64_t last = p + S->off;
    double m = -INFINITY;
    for (int64_t j = 0; j <= last; ++j) {
        s[j] = dot(S->q + p * d, S->k + j * d, d) * scale;
        if (s[j] > m) m = s[j];
    }
    double z = 0.0;
    for (int64_t j = 0; j <= last; ++j) z += exp(s[j] - m);
    return m + log(z);
}

/* Forward for one row: o[d] = sum_{j<=p+off} exp(s_j - LSE) v_j, returns LSE. */
static double fwd_row(const seg_head* S, int64_t p, int d, double scale, double* s, double* o) {
    double lse = softmax_row(S, p, d, scale, s);
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (int64_t j = 0; j <= p + S->off; ++j) {
        double w = exp(s[j] - lse);
        for (int c = 0; c < d; ++c) o[c] += w * S->v[j * d + c];
    }
    return lse;
}

static orc_problem make_problem(const void* q, const void* k, const void* v,
                                const void* dout, const int32_t* cu, const int32_t* cu_kv,
                                int32_t nseg, int32_t total, int32_t total_kv, int32_t H,
                                int32_t Hkv, int32_t d, double scale, double theta, int contract) {
    orc_problem P;
    P.q = q; P.k = k; P.v = v; P.dout = dout; P.cu = cu;
    P.cu_kv = cu_kv != NULL ? cu_kv : cu;
    /* contract: 1 contract mode, 0 exact mode, -1 exact mode on fp64 inputs; adding 4 (or, for
     * fp64 inputs, passing -5) selects the interleaved RoPE pairing. */
    P.rope_interleaved = 0;
    if (contract >= 0 && (contract & 4)) { P.rope_interleaved = 1; contract &= ~4; }
    else if (contract < 0 && contract != -1) { P.rope_interleaved = 1; contract = -1; }
    P.f64_inputs = contract < 0;   /* contract == -1 selects fp64 inputs, exact mode */
    if (contract < 0) contract = 0;
    P.nseg = nseg; P.total = total; P.total_kv = cu_kv != NULL ? total_kv : total;
    P.H = H; P.Hkv = Hkv; P.d = d;
    P.scale = scale > 0.0 ? scale : 1.0 / sqrt((double)d);
    P.theta = theta; P.contract = contract;
    return P;
}

static void fwd_seg_head(const orc_problem* P, int32_t r, int32_t h, double* o, double* lse);

/* Full forward: o [total][H][d], lse [H][total] (natural log).  cu_kv == NULL is
 * self-attention (keys and values segmented like the queries, total_kv ignored). */
void orc_attn_fwd(const void* q, const void* k, const void* v, const int32_t* cu,
                  const int32_t* cu_kv, int32_t nseg, int32_t total, int32_t total_kv, int32_t H,
                  int32_t Hkv, int32_t d, double scale, double theta, int contract, double* o,
                  double* lse) {
    orc_problem P = make_problem(q, k, v, NULL, cu, cu_kv, nseg, total, total_kv, H, Hkv, d, scale,
                                 theta, contract);
    int64_t nwork = (int64_t)nseg * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t w = 0; w < nwork; ++w) fwd_seg_head(&P, (int32_t)(w / H), (int32_t)(w % H), o, lse);
}

/* One segment-head of the forward: rows of segment r, head h. */
static void fwd_seg_head(const orc_problem* P, int32_t r, int32_t h, double* o, double* lse) {
    seg_head S;
    seg_head_load(P, r, h, 0, &S);
    double* s = (double*)malloc(sizeof(double) * (size_t)(S.Lk > 0 ? S.Lk : 1));
    for (int64_t p = 0; p < S.L; ++p) {
        int64_t i = S.base + p;
        lse[(size_t)h * P->total + i] = fwd_row(&S, p, P->d, P->scale, s, o + ((size_t)i * P->H + h) * P->d);
    }
    free(s);
    seg_head_free(&S);
}

/* Forward restricted to a set of (segment, head) pairs; other entries untouched. */
void orc_attn_fwd_seg_heads(const void* q, const void* k, const void* v, const int32_t* cu,
                            const int32_t* cu_kv, int32_t nseg, int32_t total, int32_t total_kv,
                            int32_t H, int32_t Hkv, int32_t d, double scale, double theta,
                            int contract, const int32_t* segs, const int32_t* heads, int64_t n,
                            double* o, double* lse) {
    orc_problem P = make_problem(q, k, v, NULL, cu, cu_kv, nseg, total, total_kv, H, Hkv, d, scale,
                                 theta, contract);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < n; ++t) fwd_seg_head(&P, segs[t], heads[t], o, lse);
}

/* Sampled forward: the same result for selected (token, head) pairs only,
 * so that full-size problems can be checked row by row. */
void orc_attn_fwd_rows(const void* q, const void* k, const void* v, const int32_t* cu,
                       const int32_t* cu_kv, int32_t nseg, int32_t total, int32_t total_kv,
                       int32_t H, int32_t Hkv, int32_t d, double scale, double theta, int contract,
                       const int64_t* rows, const int32_t* heads, int64_t n, double* o, double* lse) {
    orc_problem P = make_problem(q, k, v, NULL, cu, cu_kv, nseg, total, total_kv, H, Hkv, d, scale,
                                 theta, contract);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < n; ++t) {
        int64_t i = rows[t];
        int32_t h = heads[t];
        int32_t r = segment_of(cu, nseg, i);
        int64_t p = i - cu[r];
        /* only query p and the keys 0..p+off it sees are needed */
        seg_head S;
        S.base = cu[r];
        S.base_k = P.cu_kv[r];
        S.off = ((int64_t)P.cu_kv[r + 1] - P.cu_kv[r]) - ((int64_t)cu[r + 1] - cu[r]);
        S.L = p + 1;
        S.Lk = p + S.off + 1;
        S.q = (double*)malloc(sizeof(double) * (size_t)(p + 1) * d);
        S.k = (double*)malloc(sizeof(double) * (size_t)S.Lk * d);
        S.v = (double*)malloc(sizeof(double) * (size_t)S.Lk * d);
        S.g = NULL;
        load_rotated(&P, q, i, h, p + S.off, S.q + p * d);
        for (int64_t j = 0; j < S.Lk; ++j) {
            load_rotated(&P, k, S.base_k + j, kv_head(&P, h), j, S.k + j * d);
            load_plain(&P, v, S.base_k + j, kv_head(&P, h), S.v + j * d);
        }
        double* s = (double*)malloc(sizeof(double) * (size_t)S.Lk);
        lse[t] = fwd_row(&S, p, d, P.scale, s, o + t * d);
        free(s);
        seg_head_free(&S);
    }
}

/* Backward of one segment and one key/value head (the standard softmax-attention
 * derivatives), for every query head h of its group:
 *   P = exp(S - LSE) on allowed entries, dV = P^T dO, dP = dO V^T,
 *   D_p = sum_j P_pj dP_pj, dS = P o (dP - D), dQ' = scale dS K', dK' = scale dS^T Q',
 * then dQ = R(p + off)^T dQ', dK = R(j)^T dK'; the group's contributions to dK and dV
 * add up (each query head reads the shared K and V).  dq has H heads, dk/dv Hkv. */
static void bwd_seg_kvhead(const orc_problem* P, int32_t r, int32_t hk, double* dq, double* dk,
                           double* dv) {
    int d = P->d;
    const int32_t group = P->H / P->Hkv;
    const int64_t L = (int64_t)P->cu[r + 1] - P->cu[r], base = P->cu[r];
    const int64_t Lk = (int64_t)P->cu_kv[r + 1] - P->cu_kv[r], base_k = P->cu_kv[r];
    const int64_t off = Lk - L;
    const size_t nk = (size_t)(Lk > 0 ? Lk : 1);
    double* gk = (double*)calloc(nk * d, sizeof(double));
    double* gv = (double*)calloc(nk * d, sizeof(double));
    double* gq = (double*)malloc(sizeof(double) * (size_t)L * d);
    double* lse = (double*)malloc(sizeof(double) * (size_t)L);
    double* s = (double*)malloc(sizeof(double) * nk);
    double* pr = (double*)malloc(sizeof(double) * nk);
    double* dp = (double*)malloc(sizeof(double) * nk);
    for (int32_t h = hk * group; h < (hk + 1) * group; ++h) {
        seg_head S;
        seg_head_load(P, r, h, 1, &S);
        for (int64_t p = 0; p < L; ++p) lse[p] = softmax_row(&S, p, d, P->scale, s);
        memset(gq, 0, sizeof(double) * (size_t)L * d);
        for (int64_t p = 0; p < L; ++p) {
            double D = 0.0;
            for (int64_t j = 0; j <= p + off; ++j) {
                pr[j] = exp(dot(S.q + p * d, S.k + j * d, d) * P->scale - lse[p]);
                dp[j] = dot(S.g + p * d, S.v + j * d, d);
                D += pr[j] * dp[j];
            }
            for (int64_t j = 0; j <= p + off; ++j) {
                double ds = pr[j] * (dp[j] - D);
                for (int c = 0; c < d; ++c) {
                    gv[j * d + c] += pr[j] * S.g[p * d + c];
                    gq[p * d + c] += P->scale * ds * S.k[j * d + c];
                    gk[j * d + c] += P->scale * ds * S.q[p * d + c];
                }
            }
        }
        for (int64_t p = 0; p < L; ++p) {
            size_t o2 = ((size_t)(base + p) * P->H + h) * d;
            if (P->theta != 0.0) rope_rotate_transpose(gq + p * d, dq + o2, p + off, d, P->theta, P->rope_interleaved);
            else memcpy(dq + o2, gq + p * d, sizeof(double) * (size_t)d);
        }
        seg_head_free(&S);
    }
    for (int64_t j = 0; j < Lk; ++j) {
        size_t o2 = ((size_t)(base_k + j) * P->Hkv + hk) * d;
        if (P->theta != 0.0) rope_rotate_transpose(gk + j * d, dk + o2, j, d, P->theta, P->rope_interleaved);
        else memcpy(dk + o2, gk + j * d, sizeof(double) * (size_t)d);
        memcpy(dv + o2, gv + j * d, sizeof(double) * (size_t)d);
    }
    free(lse); free(s); free(gq); free(gk); free(gv); free(pr); free(dp);
}

void orc_attn_bwd(const void* dout, const void* q, const void* k, const void* v,
                  const int32_t* cu, const int32_t* cu_kv, int32_t nseg, int32_t total,
                  int32_t total_kv, int32_t H, int32_t Hkv, int32_t d, double scale, double theta,
                  int contract, double* dq, double* dk, double* dv) {
    orc_problem P = make_problem(q, k, v, dout, cu, cu_kv, nseg, total, total_kv, H, Hkv, d, scale,
                                 theta, contract);
    int64_t nwork = (int64_t)nseg * Hkv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t w = 0; w < nwork; ++w)
        bwd_seg_kvhead(&P, (int32_t)(w / Hkv), (int32_t)(w % Hkv), dq, dk, dv);
}

/* Backward restricted to a set of (segment, key/value head) pairs: dq of every
 * query head of each pair's group and dk/dv of the pair; the other rows are left
 * untouched.  Used for sampled checks at full size. */
void orc_attn_bwd_seg_heads(const void* dout, const void* q, const void* k,
                            const void* v, const int32_t* cu, const int32_t* cu_kv, int32_t nseg,
                            int32_t total, int32_t total_kv, int32_t H, int32_t Hkv, int32_t d,
                            double scale, double theta, int contract, const int32_t* segs,
                            const int32_t* heads, int64_t n, double* dq, double* dk, double* dv) {
    orc_problem P = make_problem(q, k, v, dout, cu, cu_kv, nseg, total, total_kv, H, Hkv, d, scale,
                                 theta, contract);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < n; ++t) bwd_seg_kvhead(&P, segs[t], heads[t], dq, dk, dv);
}

/* ---------------------------------------------------------------- shifted cross-entropy
 * [CSTAR] "After isolation one cross-boundary prediction pair remains": with the
 * pre-shifted labels (lab_i = token_{i+1} inside a segment, -100 on its last
 * token and on ignored segments) the loss term of logit row i is the
 * cross-entropy  CE_i = ln(sum_c exp(z_ic)) - z_i,lab_i  for lab_i != -100.
 * [CSTAR] "Packing should not decide how much a long sample weighs": keep the
 * per-segment sums S_r = sum_{i in r} CE_i and counts n_r = #{i in r : lab_i !=
 * -100}, and the pack totals sum_r S_r and sum_r n_r.  Logits are [total, vocab],
 * either bf16 bit patterns (is_f64 == 0) or doubles (is_f64 == 1).  A label
 * outside [0, vocab) other than -100 makes the call return 1 and counts nothing
 * for that row.  cu may be NULL (one segment covering the whole buffer). */
int orc_shifted_ce(const void* logits, int is_f64, int32_t vocab, int32_t total,
                   const int64_t* labels, const int32_t* cu, int32_t nseg, double* loss_sum,
                   int64_t* count, double* seg_loss, int64_t* seg_count) {
    int bad = 0;
    int32_t cu1[2] = {0, total};
    if (cu == NULL) { cu = cu1; nseg = 1; }
    double* row = (double*)calloc((size_t)total, sizeof(double));
    int8_t* ok = (int8_t*)calloc((size_t)total, 1);
#pragma omp parallel for schedule(dynamic, 64) reduction(| : bad)
    for (int64_t i = 0; i < total; ++i) {
        const int64_t y = labels[i];
        if (y == -100) continue;
        if (y < 0 || y >= vocab) { bad = 1; continue; }
        double mx = -INFINITY;
        for (int32_t c = 0; c < vocab; ++c) {
            const int64_t at = i * (int64_t)vocab + c;
            const double z = is_f64 ? ((const double*)logits)[at]
                                    : bf16_bits_to_double(((const uint16_t*)logits)[at]);
            if (z > mx) mx = z;
        }
        double s = 0.0, zy = 0.0;
        for (int32_t c = 0; c < vocab; ++c) {
            const int64_t at = i * (int64_t)vocab + c;
            const double z = is_f64 ? ((const double*)logits)[at]
                                    : bf16_bits_to_double(((const uint16_t*)logits)[at]);
            s += exp(z - mx);
            if (c == y) zy = z;
        }
        row[i] = (mx + log(s)) - zy;
        ok[i] = 1;
    }
    double tot = 0.0;
    int64_t cnt = 0;
    for (int32_t r = 0; r < nseg; ++r) {
        double sr = 0.0;
        int64_t nr = 0;
        for (int64_t i = cu[r]; i < cu[r + 1]; ++i)
            if (ok[i]) { sr += row[i]; ++nr; }
        if (seg_loss) seg_loss[r] = sr;
        if (seg_count) seg_count[r] = nr;
        tot += sr;
        cnt += nr;
    }
    *loss_sum = tot;
    *count = cnt;
    free(row);
    free(ok);
    return bad;
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
