/*
 * Plain CPU oracle of the decode-batch QKV front.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link
 * or call this file; only tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes (page "vllm.models.muse_spark.nvidia.specialized_decode.
 * cutedsl.attention.qkv_front", module docstring): the QKV + o-gate projection
 * out = x @ W^T (BF16 inputs, FP32 accumulation, rounded to BF16), then for
 * every 64-wide q and k head the weightless RMS norm and the interleaved RoPE,
 * the store of the row, and the insert of each token's K and V into a paged
 * BF16 cache.  The page states the fused kernel writes what "the projection
 * GEMM followed by fused_muse_spark_qknorm_rope_kv_insert" writes, up to the
 * GEMM's summation order, so the oracle is that unfused definition, step by
 * step, with one fixed summation order.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -shared -fPIC.  Every float
 * operation below is a single IEEE binary32 operation in program order.
 *
 * Readings of the pages where they are silent (each also listed in the
 * design notes):
 *   - the projection value is rounded to BF16 before the norm (module
 *     docstring: the owner "rounds to BF16 and runs the epilogue");
 *   - norm then RoPE, with no rounding in between; one rounding to BF16 at the
 *     end of the q/k epilogue;
 *   - RMS norm: u = p / sqrt(mean(p^2) + eps), eps = 1e-6, no weight;
 *   - RoPE pairs (2i, 2i+1); cos in table column i, sin in column 32 + i;
 *     (a, b) -> (a c - b s, b c + a s);
 *   - a negative slot means "no insert" (padding token), silently;
 *   - an out-of-range slot or position is an error: that token's insert (and,
 *     for a bad position, its q and k head outputs) is skipped and the error
 *     bit is returned.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_HEAD_DIM 64        /* qkv_front page, module docstring: "one head (64 output columns)" */
#define ORACLE_Q_PER_KV 8         /* cute_ops page, split_qkv: "q and gate: 8 heads of 64 per KV head" */
#define ORACLE_PAGE_SLOTS 16      /* cute_ops page, attn2 paragraph: cache [pages, num_kv_heads, 16, 128] */
#define ORACLE_SLOT_WIDTH 128     /* K | V per slot: 64 + 64 */
#define ORACLE_EPS 1e-6f

enum { ORACLE_HEAD_Q = 0, ORACLE_HEAD_K = 1, ORACLE_HEAD_V = 2, ORACLE_HEAD_GATE = 3 };
enum { ORACLE_ERR_SLOT = 1, ORACLE_ERR_POSITION = 2, ORACLE_ERR_SHAPE = 4 };

/* ---- BF16 <-> FP32 ------------------------------------------------------ */

/* BF16 is the upper half of an IEEE binary32; widening is exact. */
float oracle_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 to BF16, round-to-nearest, ties to even (IEEE 754
 * roundTiesToEven on the 8-bit significand).  NaN stays NaN (quiet). */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t exp_bits = (u >> 23) & 0xFFu;
    uint32_t man_bits = u & 0x7FFFFFu;
    if (exp_bits == 0xFFu && man_bits != 0) {
        return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN, sign kept */
    }
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xFFFFu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) {
        upper += 1u; /* carries into the exponent: may round up to infinity */
    }
    return (uint16_t)upper;
}

/* ---- step 1: projection GEMM ---------------------------------------------
 * acc[t][n] = sum_k x[t][k] * W[n][k], sequential over k in FP32, each product
 * rounded once and added once (qkv_front page, module docstring: "split-K BF16
 * GEMM ... FP32 accumulate"; the summation order is free, this one is
 * k = 0, 1, ..., K-1). */
void oracle_project_f32(const uint16_t *x, const uint16_t *W, int M, int N, int K, float *acc)
{
    for (int t = 0; t < M; ++t) {
        const uint16_t *xr = x + (size_t)t * K;
        for (int n = 0; n < N; ++n) {
            const uint16_t *wr = W + (size_t)n * K;
            float s = 0.0f;
            for (int k = 0; k < K; ++k) {
                float prod = oracle_bf16_to_f32(xr[k]) * oracle_bf16_to_f32(wr[k]);
                s = s + prod;
            }
            acc[(size_t)t * N + n] = s;
        }
    }
}

/* ---- step 2: which head a 64-column group is ------------------------------
 * cute_ops page, split_qkv: rows are [q | k | v | gate]; q and gate have
 * 8 heads per KV head, k and v one each. */
int oracle_head_kind(int head, int num_kv_heads)
{
    int q_heads = ORACLE_Q_PER_KV * num_kv_heads;
    if (head < q_heads) return ORACLE_HEAD_Q;
    if (head < q_heads + num_kv_heads) return ORACLE_HEAD_K;
    if (head < q_heads + 2 * num_kv_heads) return ORACLE_HEAD_V;
    return ORACLE_HEAD_GATE;
}

/* ---- step 3: weightless RMS norm of one head -------------------------------
 * u_j = p_j / sqrt(mean_j p_j^2 + eps), no learned weight (qkv_front page,
 * module docstring: "the per-head weightless RMS norm").  mean = (sum of
 * squares, sequential in j) / 64; r = 1 / sqrt(mean + eps); u_j = p_j * r. */
void oracle_rms_norm_head(const float *p, float eps, float *u)
{
    float ss = 0.0f;
    for (int j = 0; j < ORACLE_HEAD_DIM; ++j) {
        float sq = p[j] * p[j];
        ss = ss + sq;
    }
    float ms = ss / (float)ORACLE_HEAD_DIM;
    float r = 1.0f / sqrtf(ms + eps);
    for (int j = 0; j < ORACLE_HEAD_DIM; ++j) {
        u[j] = p[j] * r;
    }
}

/* ---- step 4: interleaved RoPE of one head ----------------------------------
 * Pair i is (u_{2i}, u_{2i+1}) (qkv_front page, QkvFrontKernel.finish: each
 * lane owns head columns 2 lane, 2 lane + 1; cute_ops page,
 * unsupported_projection: the rotary table is not neox style).  The fp32 table
 * row of the token's position holds cos in columns 0..31 and sin in 32..63. */
void oracle_rope_head(const float *u, const float *cs_row, float *y)
{
    for (int i = 0; i < ORACLE_HEAD_DIM / 2; ++i) {
        float c = cs_row[i];
        float s = cs_row[ORACLE_HEAD_DIM / 2 + i];
        float a = u[2 * i];
        float b = u[2 * i + 1];
        float ac = a * c, bs = b * s, bc = b * c, as = a * s;
        y[2 * i] = ac - bs;
        y[2 * i + 1] = bc + as;
    }
}

/* ---- step 5: paged K/V insert of one token --------------------------------
 * cute_ops page, attn2 paragraph: cache bf16 [pages, num_kv_heads, 16, 128],
 * K | V per slot.  Slot s lives in page s / 16 at offset s % 16.  KV head g of
 * the token: K half (0..63) = the token's k head g of `out`, V half (64..127)
 * = its v head g. */
void oracle_kv_insert_token(const uint16_t *out_row, int64_t slot, uint16_t *kv_cache,
                            int num_kv_heads)
{
    int64_t page = slot / ORACLE_PAGE_SLOTS;
    int64_t off = slot % ORACLE_PAGE_SLOTS;
    int q_cols = ORACLE_Q_PER_KV * num_kv_heads * ORACLE_HEAD_DIM;
    int kv_cols = num_kv_heads * ORACLE_HEAD_DIM;
    for (int g = 0; g < num_kv_heads; ++g) {
        uint16_t *dst = kv_cache
            + (((size_t)page * num_kv_heads + g) * ORACLE_PAGE_SLOTS + off) * ORACLE_SLOT_WIDTH;
        const uint16_t *k_src = out_row + q_cols + g * ORACLE_HEAD_DIM;
        const uint16_t *v_src = out_row + q_cols + kv_cols + g * ORACLE_HEAD_DIM;
        for (int j = 0; j < ORACLE_HEAD_DIM; ++j) {
            dst[j] = k_src[j];
            dst[ORACLE_HEAD_DIM + j] = v_src[j];
        }
    }
}

/* ---- the whole front ---------------------------------------------------
 * x [M, K], W [N, K] bf16; positions, slots int64 [M]; cos_sin fp32
 * [cos_rows, 64]; out [M, N] bf16; kv_cache bf16 [num_pages, nkv, 16, 128].
 * N must be 18 * 64 * nkv (cute_ops page, split_qkv: 2 * q_width +
 * 2 * kv_width).  Returns 0 or an OR of ORACLE_ERR_* bits.  `acc` is caller
 * scratch of M * N floats. */
int oracle_qkv_front(const uint16_t *x, const uint16_t *W, const int64_t *positions,
                     const int64_t *slots, const float *cos_sin, int64_t cos_rows,
                     uint16_t *out, uint16_t *kv_cache, int64_t num_pages, int M, int N,
                     int K, int num_kv_heads, float *acc)
{
    if (num_kv_heads < 1 || N != 2 * (ORACLE_Q_PER_KV + 1) * num_kv_heads * ORACLE_HEAD_DIM)
        return ORACLE_ERR_SHAPE;
    int err = 0;
    oracle_project_f32(x, W, M, N, K, acc);
    int heads = N / ORACLE_HEAD_DIM;
    float p[ORACLE_HEAD_DIM], u[ORACLE_HEAD_DIM], y[ORACLE_HEAD_DIM];
    for (int t = 0; t < M; ++t) {
        int64_t pos = positions[t];
        int pos_ok = pos >= 0 && pos < cos_rows;
        if (!pos_ok) err |= ORACLE_ERR_POSITION;
        for (int h = 0; h < heads; ++h) {
            const float *a = acc + (size_t)t * N + (size_t)h * ORACLE_HEAD_DIM;
            uint16_t *o = out + (size_t)t * N + (size_t)h * ORACLE_HEAD_DIM;
            for (int j = 0; j < ORACLE_HEAD_DIM; ++j)
                p[j] = oracle_bf16_to_f32(oracle_f32_to_bf16(a[j]));
            int kind = oracle_head_kind(h, num_kv_heads);
            if (kind == ORACLE_HEAD_Q || kind == ORACLE_HEAD_K) {
                if (!pos_ok) continue; /* no table row: the head is left as it was */
                oracle_rms_norm_head(p, ORACLE_EPS, u);
                oracle_rope_head(u, cos_sin + (size_t)pos * ORACLE_HEAD_DIM, y);
                for (int j = 0; j < ORACLE_HEAD_DIM; ++j) o[j] = oracle_f32_to_bf16(y[j]);
            } else {
                for (int j = 0; j < ORACLE_HEAD_DIM; ++j) o[j] = oracle_f32_to_bf16(p[j]);
            }
        }
        int64_t slot = slots[t];
        if (slot < 0) continue; /* padding token: nothing to insert */
        if (slot >= num_pages * ORACLE_PAGE_SLOTS) {
            err |= ORACLE_ERR_SLOT;
            continue;
        }
        if (!pos_ok) continue; /* its k head was not computed */
        oracle_kv_insert_token(out + (size_t)t * N, slot, kv_cache, num_kv_heads);
    }
    return err;
}

/* ---- the unfused epilogue on its own ---------------------------------------
 * fused_muse_spark_qknorm_rope_kv_insert, the kernel the front replaces
 * (qkv_front page, module docstring; cute_ops page, qkv_front paragraph): on a
 * BF16 projection output qkv [T, N] (rows [q | k | v | gate]), in place, every
 * q and k head is normed and rotated and rounded to BF16; v and gate heads are
 * left as they are; each token's k and v heads go into its cache slot.  The
 * same steps as the front after its rounding, for any number of tokens.
 * Returns 0 or an OR of ORACLE_ERR_* bits (same rules as oracle_qkv_front). */
int oracle_qknorm_rope_kv_insert(uint16_t *qkv, const int64_t *positions, const int64_t *slots,
                                 const float *cos_sin, int64_t cos_rows, uint16_t *kv_cache,
                                 int64_t num_pages, int T, int N, int num_kv_heads)
{
    if (num_kv_heads < 1 || N != 2 * (ORACLE_Q_PER_KV + 1) * num_kv_heads * ORACLE_HEAD_DIM)
        return ORACLE_ERR_SHAPE;
    int err = 0;
    int heads = N / ORACLE_HEAD_DIM;
    float p[ORACLE_HEAD_DIM], u[ORACLE_HEAD_DIM], y[ORACLE_HEAD_DIM];
    for (int t = 0; t < T; ++t) {
        int64_t pos = positions[t];
        int pos_ok = pos >= 0 && pos < cos_rows;
        if (!pos_ok) err |= ORACLE_ERR_POSITION;
        uint16_t *row = qkv + (size_t)t * N;
        for (int h = 0; h < heads; ++h) {
            int kind = oracle_head_kind(h, num_kv_heads);
            if (kind != ORACLE_HEAD_Q && kind != ORACLE_HEAD_K) continue;
            if (!pos_ok) continue;
            uint16_t *o = row + (size_t)h * ORACLE_HEAD_DIM;
            for (int j = 0; j < ORACLE_HEAD_DIM; ++j) p[j] = oracle_bf16_to_f32(o[j]);
            oracle_rms_norm_head(p, ORACLE_EPS, u);
            oracle_rope_head(u, cos_sin + (size_t)pos * ORACLE_HEAD_DIM, y);
            for (int j = 0; j < ORACLE_HEAD_DIM; ++j) o[j] = oracle_f32_to_bf16(y[j]);
        }
        int64_t slot = slots[t];
        if (slot < 0) continue;
        if (slot >= num_pages * ORACLE_PAGE_SLOTS) {
            err |= ORACLE_ERR_SLOT;
            continue;
        }
        if (!pos_ok) continue;
        oracle_kv_insert_token(row, slot, kv_cache, num_kv_heads);
    }
    return err;
}

/* ---- the predecessor: the first layer's front -----------------------------
 * Page "vllm.models.muse_spark.nvidia.specialized_decode.cutedsl.boundary.
 * layer_front", class LayerFront: run(x, stream, out, aux) writes
 * stream = x as FP32, aux = stream (when kept), and out = the layer's
 * pre-QKV RMS norm of the stream, in BF16.  x is BF16 or FP32 [rows, 8192].
 * Reading (the page names the norm, not its formula): the RMS norm of the
 * whole row, r = 1 / sqrt(mean_j s_j^2 + eps) with the sum sequential in j,
 * then out_j = bf16((s_j * r) * w_j) with the BF16 weight w widened to FP32
 * (weightless when w is NULL: out_j = bf16(s_j * r)).  The result of this
 * step is what the QKV front reads as x. */
void oracle_layer_front(const void *x, int x_is_f32, const uint16_t *weight, float *stream,
                        float *aux, uint16_t *out, int rows, int hidden, float eps)
{
    for (int t = 0; t < rows; ++t) {
        float *srow = stream + (size_t)t * hidden;
        for (int j = 0; j < hidden; ++j) {
            srow[j] = x_is_f32 ? ((const float *)x)[(size_t)t * hidden + j]
                               : oracle_bf16_to_f32(((const uint16_t *)x)[(size_t)t * hidden + j]);
            if (aux) aux[(size_t)t * hidden + j] = srow[j];
        }
        float ss = 0.0f;
        for (int j = 0; j < hidden; ++j) {
            float sq = srow[j] * srow[j];
            ss = ss + sq;
        }
        float ms = ss / (float)hidden;
        float r = 1.0f / sqrtf(ms + eps);
        for (int j = 0; j < hidden; ++j) {
            float y = srow[j] * r;
            if (weight) y = y * oracle_bf16_to_f32(weight[j]);
            out[(size_t)t * hidden + j] = oracle_f32_to_bf16(y);
        }
    }
}

/* ---- the cache's consumer: attn2 ---------------------------------------------
 * Page "...runtime.cute_ops", attn2 paragraph: paged decode attention of the
 * 8-token verify step (one request: 1 + 7 draft tokens), head_dim 64, 8 query
 * heads per KV head, the bf16 cache [pages, num_kv_heads, 16, 128] (K | V per
 * slot), fused with the attention output's weightless RMS norm and sigmoid
 * gate: the o_proj input.  Context length L >= 8, optional sliding window.
 * Readings (the pages name these, not their formulas):
 *   - request r owns rows 8r .. 8r+7 of qkv; row i is the token at position
 *     L - 8 + i and attends keys j <= L - 8 + i (causal), and with a window W
 *     only keys j > (L - 8 + i) - W;
 *   - key j of request r is slot j % 16 of page block_table[r][j / 16];
 *   - q head h (< 8 nkv) uses KV head h / 8; its gate is gate head h of the
 *     same row ([q | k | v | gate] layout);
 *   - o = softmax(scale q K^T) V, then out = bf16( o / sqrt(mean(o^2) + eps)
 *     * sigmoid(gate) );
 *   - all of it in double here (the pages fix no precision for it).
 * A request with L < 8 or L beyond its block table, or a page index outside
 * the cache, is skipped (its rows untouched) and reported (bit 8). */
enum { ORACLE_ERR_ATTN_REQUEST = 8 };

int oracle_attn2(const uint16_t *qkv, int N, int num_kv_heads, const uint16_t *kv_cache,
                 int64_t num_pages, const int32_t *block_table, int max_blocks,
                 const int32_t *context_lens, int R, int window, double scale, double eps,
                 uint16_t *out)
{
    if (num_kv_heads < 1 || N != 2 * (ORACLE_Q_PER_KV + 1) * num_kv_heads * ORACLE_HEAD_DIM)
        return ORACLE_ERR_SHAPE;
    const int q_heads = ORACLE_Q_PER_KV * num_kv_heads;
    const int gate_col = q_heads * ORACLE_HEAD_DIM + 2 * num_kv_heads * ORACLE_HEAD_DIM;
    const int out_cols = q_heads * ORACLE_HEAD_DIM;
    int err = 0;
    int max_len = 0;
    for (int r = 0; r < R; ++r)
        if (context_lens[r] > max_len) max_len = context_lens[r];
    double *sc = (double *)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    if (!sc) return ORACLE_ERR_SHAPE;
    for (int r = 0; r < R; ++r) {
        const int L = context_lens[r];
        int ok = L >= 8 && (L + ORACLE_PAGE_SLOTS - 1) / ORACLE_PAGE_SLOTS <= max_blocks;
        for (int b = 0; ok && b < (L + ORACLE_PAGE_SLOTS - 1) / ORACLE_PAGE_SLOTS; ++b) {
            int32_t pg = block_table[(size_t)r * max_blocks + b];
            if (pg < 0 || pg >= num_pages) ok = 0;
        }
        if (!ok) {
            err |= ORACLE_ERR_ATTN_REQUEST;
            continue;
        }
        for (int i = 0; i < 8; ++i) {
            const size_t row = (size_t)r * 8 + i;
            const int pos = L - 8 + i;
            const int lo = window > 0 && pos - window + 1 > 0 ? pos - window + 1 : 0;
            for (int h = 0; h < q_heads; ++h) {
                const int g = h / ORACLE_Q_PER_KV;
                const uint16_t *q = qkv + row * N + (size_t)h * ORACLE_HEAD_DIM;
                double m = -INFINITY;
                /* scores, then their maximum */
                for (int j = lo; j <= pos; ++j) {
                    const int32_t pg = block_table[(size_t)r * max_blocks + j / ORACLE_PAGE_SLOTS];
                    const uint16_t *k = kv_cache
                        + (((size_t)pg * num_kv_heads + g) * ORACLE_PAGE_SLOTS + j % ORACLE_PAGE_SLOTS)
                          * ORACLE_SLOT_WIDTH;
                    double d = 0.0;
                    for (int e = 0; e < ORACLE_HEAD_DIM; ++e)
                        d += (double)oracle_bf16_to_f32(q[e]) * (double)oracle_bf16_to_f32(k[e]);
                    sc[j - lo] = scale * d;
                    if (sc[j - lo] > m) m = sc[j - lo];
                }
                double o[ORACLE_HEAD_DIM] = {0};
                double l = 0.0;
                for (int j = lo; j <= pos; ++j) {
                    const int32_t pg = block_table[(size_t)r * max_blocks + j / ORACLE_PAGE_SLOTS];
                    const uint16_t *v = kv_cache
                        + (((size_t)pg * num_kv_heads + g) * ORACLE_PAGE_SLOTS + j % ORACLE_PAGE_SLOTS)
                          * ORACLE_SLOT_WIDTH + ORACLE_HEAD_DIM;
                    const double p = exp(sc[j - lo] - m);
                    l += p;
                    for (int e = 0; e < ORACLE_HEAD_DIM; ++e) o[e] += p * (double)oracle_bf16_to_f32(v[e]);
                }
                double ms = 0.0;
                for (int e = 0; e < ORACLE_HEAD_DIM; ++e) {
                    o[e] /= l;
                    ms += o[e] * o[e];
                }
                ms /= ORACLE_HEAD_DIM;
                const double rn = 1.0 / sqrt(ms + eps);
                const uint16_t *gt = qkv + row * N + gate_col + (size_t)h * ORACLE_HEAD_DIM;
                uint16_t *dst = out + row * out_cols + (size_t)h * ORACLE_HEAD_DIM;
                for (int e = 0; e < ORACLE_HEAD_DIM; ++e) {
                    const double sg = 1.0 / (1.0 + exp(-(double)oracle_bf16_to_f32(gt[e])));
                    dst[e] = oracle_f32_to_bf16((float)(o[e] * rn * sg));
                }
            }
        }
    }
    free(sc);
    return err;
}
