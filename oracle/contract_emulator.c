/*
 * CPU emulator of the fixed fp32 numeric contract "rlk-linlogp-v1".
 *
 * TEST INFRASTRUCTURE ONLY.  Built by oracle/build.py into
 * oracle/libcontract_emulator.so and loaded by oracle/emulator.py.  It
 * shares no source, header, table or constant generator with the CUDA
 * library: every rule below is written again from the contract text.
 *
 * Compile with -ffp-contract=off: the only fused multiply-adds are the
 * explicit fmaf() calls (glibc's fmaf rounds once, as IEEE fusedMultiplyAdd).
 *
 * The pages fix *that* each of these must be pinned, not their values
 * ("vLLM RL-Kernel v0.1.0: ROCm 上でのビット単位のトレーニング-ロールアウト
 * 一貫性", section 数値実行契約: input dependence, split, merge order,
 * precision, rounding, primitives; and the Chinese report "ROCm上实现训练与
 * 推理logprob逐位对齐", section 技术路径：对齐四个关键环节).  The values are
 * this library's own reading:
 *
 *   split      vocabulary tiles of 128 columns; tile j = [128j, min(128j+128, V)).
 *   in-tile    m = max over the tile's real columns; d_c = RN(l_c - m);
 *              e_c = rlk_exp(d_c); s = 128-slot pairwise tree over the column
 *              index (slot pairs (0,1),(2,3),..., then pairs of those, 7
 *              levels); a missing column's slot is absent and its partner
 *              passes through unchanged.
 *   merge      merge(L, R): the operand with the larger m is "hi" (L on a tie),
 *              m = hi.m, s = fma(lo.s, rlk_exp(RN(lo.m - hi.m)), hi.s).
 *   tile tree  recursive bisection of [0, n_tiles): a node [a, b) with two or
 *              more tiles splits at a + ceil((b - a) / 2); value = merge(left, right).
 *   shards     n_shards = 2^d: shard r is the r-th node at depth d; its record
 *              is (m, s) of that node, the target logit if the shard owns
 *              the target (else 0) and the ownership flag.  Records merge
 *              in shard order along the same tree.
 *   finalize   lse = RN(m + rlk_log(s)); logprob = RN(tgt - lse).
 *   exp        Cody-Waite reduction x = n ln2 + r with n = nearest integer
 *              to x log2(e) (computed as fma(x, log2e, 1.5 * 2^23) minus
 *              1.5 * 2^23), r = fma(-n, ln2_hi, x) then fma(-n, ln2_lo, r),
 *              degree-7 Taylor polynomial of e^r in Horner form (coefficients
 *              1/k! rounded to fp32), scaled by 2^n; x < -86 gives +0.
 *   log        s = 2^e f with f in [sqrt(1/2), sqrt(2)]; u = (f-1)/(f+1);
 *              log f = 2u + u^3 (2/3 + u^2 (2/5 + u^2 (2/7 + u^2 (2/9 + u^2 2/11))));
 *              log s = fma(e, ln2_hi, fma(e, ln2_lo, log f)).
 *   inactive   rows with mask 0 give (0, 0) and all-zero shard records.
 *   no owner   an active row whose target lies outside [0, V) gives NaN.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>

#define EMU_TILE 128

static float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* ---- constants, derived here from their definitions (fp32 round-to-nearest) ---- */
static float c_log2e, c_ln2_hi, c_ln2_lo, c_shifter, c_sqrt2;
static float c_taylor[8];   /* 1/k!, k = 0..7 */
static float c_atanh[5];    /* 2/3, 2/5, 2/7, 2/9, 2/11 */
static int c_ready = 0;

static void init_constants(void) {
    if (c_ready) return;
    /* log2(e) and ln 2 to well beyond fp32 precision (long double on x86,
       binary128 on aarch64), then rounded once to fp32 */
    long double ln2 = 0.693147180559945309417232121458176568L;
    long double log2e = 1.442695040888963407359924681001892137L;
    c_log2e = (float)log2e;
    c_ln2_hi = (float)ln2;
    c_ln2_lo = (float)(ln2 - (long double)c_ln2_hi);
    c_shifter = 12582912.0f; /* 1.5 * 2^23 */
    c_sqrt2 = (float)1.414213562373095048801688724209698079L;
    double fact = 1.0;
    for (int k = 0; k < 8; ++k) {
        if (k > 0) fact *= (double)k;
        c_taylor[k] = (float)(1.0 / fact);
    }
    for (int k = 0; k < 5; ++k) c_atanh[k] = (float)(2.0 / (double)(2 * k + 3));
    c_ready = 1;
}

float emu_exp(float x) {
    init_constants();
    if (x < -86.0f) return 0.0f;                    /* also -inf */
    float t = fmaf(x, c_log2e, c_shifter);
    float n = t - c_shifter;                         /* exact: integer-valued */
    int32_t ni = (int32_t)(f2u(t) - f2u(c_shifter));
    float r = fmaf(-n, c_ln2_hi, x);
    r = fmaf(-n, c_ln2_lo, r);
    float p = c_taylor[7];
    for (int k = 6; k >= 0; --k) p = fmaf(p, r, c_taylor[k]);
    float scale = u2f((uint32_t)(ni + 127) << 23);
    return p * scale;
}

float emu_log(float s) {
    init_constants();
    uint32_t b = f2u(s);
    int32_t e = (int32_t)(b >> 23) - 127;
    float f = u2f((b & 0x007FFFFFu) | 0x3F800000u);
    if (f > c_sqrt2) { f = f * 0.5f; e += 1; }
    float u = (f - 1.0f) / (f + 1.0f);
    float u2 = u * u;
    float p = c_atanh[4];
    for (int k = 3; k >= 0; --k) p = fmaf(p, u2, c_atanh[k]);
    float lf = fmaf(p, u * u2, 2.0f * u);
    float ef = (float)e;
    return fmaf(ef, c_ln2_hi, fmaf(ef, c_ln2_lo, lf));
}

void emu_merge(float m1, float s1, float m2, float s2, float* mo, float* so) {
    float mh, sh, ml, sl;
    if (m2 > m1) { mh = m2; sh = s2; ml = m1; sl = s1; }
    else         { mh = m1; sh = s1; ml = m2; sl = s2; }
    *mo = mh;
    *so = fmaf(sl, emu_exp(ml - mh), sh);
}

/* one tile of n (1..128) logits -> (m, s) */
void emu_tile_ms(const float* v, int n, float* mo, float* so) {
    float m = v[0];
    for (int c = 1; c < n; ++c) m = fmaxf(m, v[c]);
    /* 128 slots, absent flag for c >= n */
    float val[EMU_TILE];
    int present[EMU_TILE];
    for (int c = 0; c < EMU_TILE; ++c) {
        present[c] = c < n;
        val[c] = present[c] ? emu_exp(v[c] - m) : 0.0f;
    }
    for (int width = EMU_TILE; width > 1; width /= 2) {
        for (int i = 0; i < width / 2; ++i) {
            int a = 2 * i, b = 2 * i + 1;
            float r;
            int pr;
            if (present[a] && present[b]) { r = val[a] + val[b]; pr = 1; }
            else if (present[a])          { r = val[a]; pr = 1; }
            else if (present[b])          { r = val[b]; pr = 1; }
            else                          { r = 0.0f; pr = 0; }
            val[i] = r;
            present[i] = pr;
        }
    }
    *mo = m;
    *so = val[0];
}

/* value of the bisection-tree node [a, b) over leaves (m[], s[]) */
static void tree_node(const float* m, const float* s, int64_t a, int64_t b, float* mo, float* so) {
    if (b - a == 1) { *mo = m[a]; *so = s[a]; return; }
    int64_t mid = a + (b - a + 1) / 2;
    float ml, sl, mr, sr;
    tree_node(m, s, a, mid, &ml, &sl);
    tree_node(m, s, mid, b, &mr, &sr);
    emu_merge(ml, sl, mr, sr, mo, so);
}

void emu_tree(const float* m, const float* s, int64_t n, float* mo, float* so) {
    tree_node(m, s, 0, n, mo, so);
}

/* tile ranges of the 2^depth nodes at that depth; returns 0 or -1 if too shallow */
int emu_tree_nodes(int64_t n_tiles, int depth, int64_t* begin, int64_t* end) {
    int64_t a[64], b[64];
    int cnt = 1;
    a[0] = 0; b[0] = n_tiles;
    if (depth < 0 || depth > 5) return -1;
    for (int d = 0; d < depth; ++d) {
        int64_t na[64], nb[64];
        for (int i = 0; i < cnt; ++i) {
            if (b[i] - a[i] < 2) return -1;
            int64_t mid = a[i] + (b[i] - a[i] + 1) / 2;
            na[2 * i] = a[i]; nb[2 * i] = mid;
            na[2 * i + 1] = mid; nb[2 * i + 1] = b[i];
        }
        cnt *= 2;
        memcpy(a, na, sizeof(int64_t) * cnt);
        memcpy(b, nb, sizeof(int64_t) * cnt);
    }
    for (int i = 0; i < cnt; ++i) { begin[i] = a[i]; end[i] = b[i]; }
    return 0;
}

/* per-row, per-tile (m, s) of fp32 logits [T][V] -> tm, ts [T][n_tiles] */
void emu_tile_partials(const float* logits, int64_t T, int64_t V, float* tm, float* ts) {
    int64_t nt = (V + EMU_TILE - 1) / EMU_TILE;
    for (int64_t t = 0; t < T; ++t) {
        const float* row = logits + t * V;
        for (int64_t j = 0; j < nt; ++j) {
            int64_t c0 = j * EMU_TILE;
            int n = (int)((V - c0) < EMU_TILE ? (V - c0) : EMU_TILE);
            emu_tile_ms(row + c0, n, tm + t * nt + j, ts + t * nt + j);
        }
    }
}

/*
 * Full contract from fp32 logits [T][V].  Outputs (may be NULL):
 *   out_lp, out_lse [T];
 *   rec_m, rec_s, rec_tgt [n_shards][T], rec_owned [n_shards][T];
 *   root_direct_m/s [T]: the root computed directly over all tiles (no shard
 *   records), for the self-check that both routes give the same bits.
 * Returns 0, or -1 for an unsupported shard count.
 */
int emu_linear_logprob(const float* logits, int64_t T, int64_t V, const int32_t* targets,
                       const uint8_t* active, int n_shards,
                       float* out_lp, float* out_lse,
                       float* rec_m, float* rec_s, float* rec_tgt, uint32_t* rec_owned,
                       float* root_direct_m, float* root_direct_s) {
    int depth = 0;
    while ((1 << depth) < n_shards) ++depth;
    if ((1 << depth) != n_shards || depth > 3) return -1;
    int64_t nt = (V + EMU_TILE - 1) / EMU_TILE;
    int64_t nb[8], ne[8];
    if (emu_tree_nodes(nt, depth, nb, ne) != 0) return -1;
    float* tm = (float*)malloc(sizeof(float) * nt);
    float* ts = (float*)malloc(sizeof(float) * nt);
    for (int64_t t = 0; t < T; ++t) {
        const float* row = logits + t * V;
        int act = active ? (active[t] != 0) : 1;
        if (!act) {
            if (out_lp) out_lp[t] = 0.0f;
            if (out_lse) out_lse[t] = 0.0f;
            for (int r = 0; r < n_shards; ++r) {
                if (rec_m) rec_m[r * T + t] = 0.0f;
                if (rec_s) rec_s[r * T + t] = 0.0f;
                if (rec_tgt) rec_tgt[r * T + t] = 0.0f;
                if (rec_owned) rec_owned[r * T + t] = 0u;
            }
            if (root_direct_m) root_direct_m[t] = 0.0f;
            if (root_direct_s) root_direct_s[t] = 0.0f;
            continue;
        }
        for (int64_t j = 0; j < nt; ++j) {
            int64_t c0 = j * EMU_TILE;
            int n = (int)((V - c0) < EMU_TILE ? (V - c0) : EMU_TILE);
            emu_tile_ms(row + c0, n, tm + j, ts + j);
        }
        float sm[8], ss[8], stg[8];
        int sown[8];
        int64_t tg = targets[t];
        int owners = 0;
        float tgt = 0.0f;
        for (int r = 0; r < n_shards; ++r) {
            tree_node(tm, ts, nb[r], ne[r], &sm[r], &ss[r]);
            int64_t v0 = nb[r] * EMU_TILE;
            int64_t v1 = ne[r] * EMU_TILE < V ? ne[r] * EMU_TILE : V;
            sown[r] = (tg >= v0 && tg < v1);
            stg[r] = sown[r] ? row[tg] : 0.0f;
            if (sown[r]) { owners += 1; tgt = stg[r]; }
            if (rec_m) rec_m[r * T + t] = sm[r];
            if (rec_s) rec_s[r * T + t] = ss[r];
            if (rec_tgt) rec_tgt[r * T + t] = stg[r];
            if (rec_owned) rec_owned[r * T + t] = (uint32_t)sown[r];
        }
        float rm, rs;
        tree_node(sm, ss, 0, n_shards, &rm, &rs);
        if (root_direct_m || root_direct_s) {
            float dm, ds;
            tree_node(tm, ts, 0, nt, &dm, &ds);
            if (root_direct_m) root_direct_m[t] = dm;
            if (root_direct_s) root_direct_s[t] = ds;
        }
        float lse = rm + emu_log(rs);
        float lp = tgt - lse;
        if (owners != 1) { lse = NAN; lp = NAN; }
        if (out_lp) out_lp[t] = lp;
        if (out_lse) out_lse[t] = lse;
    }
    free(tm);
    free(ts);
    return 0;
}

/* log_softmax: out[t][v] = RN(l - lse) with lse from the full tile tree; inactive rows 0 */
int emu_log_softmax(const float* logits, int64_t T, int64_t V, const uint8_t* active,
                    float* out, float* out_lse) {
    int32_t* tg = (int32_t*)calloc((size_t)(T > 0 ? T : 1), sizeof(int32_t));
    int rc = emu_linear_logprob(logits, T, V, tg, active, 1, NULL, out_lse, NULL, NULL, NULL, NULL,
                                NULL, NULL);
    free(tg);
    if (rc != 0) return rc;
    for (int64_t t = 0; t < T; ++t) {
        int act = active ? (active[t] != 0) : 1;
        for (int64_t v = 0; v < V; ++v)
            out[t * V + v] = act ? logits[t * V + v] - out_lse[t] : 0.0f;
    }
    return 0;
}

/* fp32 -> bf16 bits, round to nearest even (finite inputs) */
static uint16_t bf16_rne(float f) {
    uint32_t u = f2u(f);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/*
 * Gradient of sum_t g[t] logprob[t] with respect to the logits, as the
 * backward's first stage writes it: p = rlk_exp(RN(l - lse)),
 * d = RN(1 - p) at the target and -p elsewhere, G = bf16_RN(RN(g * d));
 * inactive rows give +0.  lse is the forward's fp32 log-sum-exp.
 */
void emu_grad_logits(const float* logits, int64_t T, int64_t V, const float* lse,
                     const int32_t* targets, const float* g, const uint8_t* active,
                     uint16_t* out) {
    for (int64_t t = 0; t < T; ++t) {
        int act = active ? (active[t] != 0) : 1;
        for (int64_t v = 0; v < V; ++v) {
            if (!act) { out[t * V + v] = 0; continue; }
            float p = emu_exp(logits[t * V + v] - lse[t]);
            float d = (v == (int64_t)targets[t]) ? 1.0f - p : -p;
            out[t * V + v] = bf16_rne(g[t] * d);
        }
    }
}

/*
 * Strict RMSNorm ("RMSNorm" row of the strict-path table: reduction domain,
 * epsilon, residual add, output boundary), as this library reads it:
 *   x'   = bf16_RN(RN(x + r))                     (residual add, if given)
 *   s    = pairwise tree over nextpow2(H) feature slots of RN(x'_i * x'_i)
 *          (exact products; slots >= H absent)
 *   a    = RN(RN(s / H) + eps)
 *   rstd = rlk_rsqrt(a)
 *   y_i  = bf16_RN(RN(RN(x'_i * rstd) * gamma_i))
 * rlk_rsqrt: seed 0x5f375a86 - (bits(a) >> 1) (Lomont's constant for the
 * classic bit-level inverse-square-root estimate), two Newton steps
 * y <- RN(y * fma(-RN(a/2), RN(y*y), 1.5)), then one in correction form
 * y <- fma(y, fma(-RN(a/2), RN(y*y), 0.5), y).
 */
float emu_rsqrt(float a) {
    uint32_t i = 0x5f375a86u - (f2u(a) >> 1);
    float y = u2f(i);
    float h = 0.5f * a;
    for (int k = 0; k < 2; ++k) {
        float r = y * y;
        float t = fmaf(-h, r, 1.5f);
        y = y * t;
    }
    /* last step in correction form: y + y * (0.5 - h y^2), one rounding for the update */
    float e = fmaf(-h, y * y, 0.5f);
    return fmaf(y, e, y);
}

static float bf16_to_f32(uint16_t b) { return u2f((uint32_t)b << 16); }

void emu_rmsnorm(const uint16_t* x, const uint16_t* res, const uint16_t* gamma, float eps,
                 int64_t T, int64_t H, uint16_t* y, uint16_t* xr_out) {
    int64_t slots = 1;
    while (slots < H) slots *= 2;
    float* q = (float*)malloc(sizeof(float) * (size_t)slots);
    float* xr = (float*)malloc(sizeof(float) * (size_t)H);
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t i = 0; i < H; ++i) {
            float v = bf16_to_f32(x[t * H + i]);
            if (res) {
                uint16_t b = bf16_rne(v + bf16_to_f32(res[t * H + i]));
                if (xr_out) xr_out[t * H + i] = b;
                v = bf16_to_f32(b);
            }
            xr[i] = v;
        }
        for (int64_t i = 0; i < slots; ++i) q[i] = i < H ? xr[i] * xr[i] : 0.0f;
        for (int64_t w = slots; w > 1; w /= 2)
            for (int64_t i = 0; i < w / 2; ++i) q[i] = q[2 * i] + q[2 * i + 1];
        float mean = q[0] / (float)H;
        float rstd = emu_rsqrt(mean + eps);
        for (int64_t i = 0; i < H; ++i)
            y[t * H + i] = bf16_rne((xr[i] * rstd) * bf16_to_f32(gamma[i]));
    }
    free(q);
    free(xr);
}

void emu_rsqrt_sweep(float lo, float hi, double* max_ulp, float* worst_x, int64_t* count);

/* ---- exhaustive accuracy sweeps against fp64 libm (the independent reference) ---- */
static double ulp_err(float y, double z) {
    if (z == 0.0) return y == 0.0f ? 0.0 : INFINITY;
    int ez;
    frexp(z, &ez);                 /* z = f * 2^ez, f in [0.5, 1) */
    int e = ez - 1;                /* binade of z */
    if (e < -126) e = -126;
    double ulp = ldexp(1.0, e - 23);
    return fabs((double)y - z) / ulp;
}

/* sweep all floats x in [lo, hi] (lo <= hi <= 0 or 0 <= lo <= hi) */
void emu_exp_sweep(float lo, float hi, double* max_ulp, float* worst_x, int64_t* count) {
    uint32_t blo = f2u(lo), bhi = f2u(hi);
    int neg = (f2u(hi) >> 31) != 0 || hi == 0.0f;
    uint32_t a, b;
    if (neg) { a = f2u(hi) | 0x80000000u; b = blo; if (a > b) { uint32_t t = a; a = b; b = t; } }
    else { a = blo; b = bhi; }
    double best = 0.0;
    float wx = 0.0f;
    int64_t cnt = 0;
    #pragma omp parallel
    {
        double lbest = 0.0;
        float lwx = 0.0f;
        int64_t lcnt = 0;
        #pragma omp for schedule(static)
        for (int64_t u = (int64_t)a; u <= (int64_t)b; ++u) {
            float x = u2f((uint32_t)u);
            float y = emu_exp(x);
            double z = exp((double)x);
            double err = (x < -86.0f) ? 0.0 : ulp_err(y, z);
            if (err > lbest) { lbest = err; lwx = x; }
            ++lcnt;
        }
        #pragma omp critical
        {
            if (lbest > best) { best = lbest; wx = lwx; }
            cnt += lcnt;
        }
    }
    *max_ulp = best;
    *worst_x = wx;
    *count = cnt;
}

void emu_log_sweep(float lo, float hi, double* max_ulp, float* worst_x, int64_t* count) {
    uint32_t a = f2u(lo), b = f2u(hi);
    double best = 0.0;
    float wx = 0.0f;
    int64_t cnt = 0;
    #pragma omp parallel
    {
        double lbest = 0.0;
        float lwx = 0.0f;
        int64_t lcnt = 0;
        #pragma omp for schedule(static)
        for (int64_t u = (int64_t)a; u <= (int64_t)b; ++u) {
            float x = u2f((uint32_t)u);
            float y = emu_log(x);
            double z = log((double)x);
            double err = ulp_err(y, z);
            if (err > lbest) { lbest = err; lwx = x; }
            ++lcnt;
        }
        #pragma omp critical
        {
            if (lbest > best) { best = lbest; wx = lwx; }
            cnt += lcnt;
        }
    }
    *max_ulp = best;
    *worst_x = wx;
    *count = cnt;
}

/* constants as derived here, for tests that check them against their definitions */
void emu_constants(float* out /* 16 */) {
    init_constants();
    out[0] = c_log2e; out[1] = c_ln2_hi; out[2] = c_ln2_lo; out[3] = c_shifter; out[4] = c_sqrt2;
    for (int k = 0; k < 8; ++k) out[5 + k] = c_taylor[k];
    out[13] = c_atanh[0]; out[14] = c_atanh[1]; out[15] = c_atanh[4];
}

void emu_rsqrt_sweep(float lo, float hi, double* max_ulp, float* worst_x, int64_t* count) {
    uint32_t a = f2u(lo), b = f2u(hi);
    double best = 0.0;
    float wx = 0.0f;
    int64_t cnt = 0;
    #pragma omp parallel
    {
        double lbest = 0.0;
        float lwx = 0.0f;
        int64_t lcnt = 0;
        #pragma omp for schedule(static)
        for (int64_t u = (int64_t)a; u <= (int64_t)b; ++u) {
            float x = u2f((uint32_t)u);
            float y = emu_rsqrt(x);
            double z = 1.0 / sqrt((double)x);
            double err = ulp_err(y, z);
            if (err > lbest) { lbest = err; lwx = x; }
            ++lcnt;
        }
        #pragma omp critical
        {
            if (lbest > best) { best = lbest; wx = lwx; }
            cnt += lcnt;
        }
    }
    *max_ulp = best;
    *worst_x = wx;
    *count = cnt;
}

/* Position-weighted sum of a primitive over the fp32 bit patterns
 * [first, first + count): sum_i (bits(f(x_i)) + 0x9E3779B9) (2 i + 1) mod 2^64,
 * with which 0 or 1: emu_exp, 2: emu_log, 3: emu_rsqrt -- the same sum the
 * library's diagnostic forms on the GPU, where 1 is its two-lane exp. */
uint64_t emu_primitive_hash(int which, uint32_t first, uint64_t count) {
    init_constants();
    uint64_t h = 0;
#pragma omp parallel for reduction(+ : h) schedule(static)
    for (int64_t i = 0; i < (int64_t)count; ++i) {
        const float x = u2f(first + (uint32_t)i);
        const float y = which <= 1 ? emu_exp(x) : which == 2 ? emu_log(x) : emu_rsqrt(x);
        h += ((uint64_t)f2u(y) + 0x9E3779B9ull) * (2ull * (uint64_t)i + 1ull);
    }
    return h;
}
