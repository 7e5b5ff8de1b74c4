/*
 * CPU oracle for the multi-adapter (segmented-rank) LoRA hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header or table with the CUDA
 * library.
 *
 * Plain C99, double precision, one token (or one token/expert pair) at a time,
 * in the order the source pages state the computation.  bf16 inputs are
 * widened exactly to double; nothing is rounded back to 16 bits.
 *
 * Sources (page title, section):
 *   [P1] "vLLM-Ascend dynamic LoRA fused operator" (pwwt.cn):
 *        1.1 the two-matmul definition y = y_base + (x A^T) B^T;
 *        2.1 operator inputs (hidden_states, lora_id_map with -1 = none);
 *        2.3 bucketing tokens by lora_id into a segment table;
 *        3.4 id -1 tokens keep their base output unchanged.
 *   [P2] "[SGLang] LoRA + MoE fusion" (secrett2633 blog): stages 1.5 and 3.5
 *        (gate/up delta before the activation, down delta before the final
 *        reduce), LoRAInfo weight shapes, moe_lora_align_block_size.
 *   [P5] "[SGLang] LoRA Layers: QKV, Gate/Up" (secrett2633 blog): stacked
 *        projections, A = (n*r, in), B = (sum of slice widths, r).
 *   [P1] 3.3 the LoRA linear layer: the base matmul of the layer's input with
 *        its weight, plus the LoRA delta (issued beside it or fused with it).
 *   [P5] "VocabParallelEmbeddingWithLoRA": embedding LoRA, A used as an
 *        embedding lookup (rank, vocab) and B as a plain matmul (embed_dim, rank).
 *
 * Readings taken where the pages are silent:
 *   - a per-adapter scale multiplies the expand result (1.0 reproduces [P1]);
 *   - ids >= L or < -1 behave like -1 and are counted as bad;
 *   - segments are in ascending adapter id, tokens ascending inside one,
 *     -1 tokens last in the permutation and in no segment;
 *   - MoE alignment: per adapter, pairs grouped by ascending expert, each
 *     group padded to a multiple of block_m with the sentinel M*topk, unused
 *     block slots carry expert id -1.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Embedding LoRA, [P5] "VocabParallelEmbeddingWithLoRA": for every token t with adapter
 * i = ids[t] in [0, L) and vocabulary id v = vocab[t] in [0, V):
 *   S[j]      = A_i[j, v]                                  (j < r = rank[i]: the lookup)
 *   y[t, n]   = y_base[t, n] + scale[i] * sum_j S[j] * B_i[n, j]
 * A[i]: bf16 [rank[i]][V] row-major; B[i]: bf16 [N][rank[i]].  Tokens with ids[t] == -1, an
 * out-of-range adapter id or an out-of-range vocabulary id copy y_base.  Returns the number of
 * out-of-range adapter or vocabulary ids.
 */
int oracle_embedding_apply(int32_t M, int32_t V, int32_t N, int32_t L, const int32_t *rank, const double *scale,
                           const uint16_t *const *A, const uint16_t *const *B, const int32_t *ids,
                           const int32_t *vocab, const uint16_t *y_base, int64_t ldy, double *y_out)
{
    int bad = 0;
    for (int32_t t = 0; t < M; ++t) {
        for (int32_t n = 0; n < N; ++n) y_out[(int64_t)t * N + n] = bf(y_base[(int64_t)t * ldy + n]);
        const int32_t i = ids[t];
        if (i < 0 || i >= L) {   /* -1: no adapter; anything else out of range is counted */
            if (i != -1) ++bad;
            continue;
        }
        const int32_t v = vocab[t];
        if (v < 0 || v >= V) { ++bad; continue; }
        const int32_t r = rank[i];
        for (int32_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int32_t j = 0; j < r; ++j) acc += bf(A[i][(int64_t)j * V + v]) * bf(B[i][(int64_t)n * r + j]);
            y_out[(int64_t)t * N + n] += scale[i] * acc;
        }
    }
    return bad;
}

/*
 * Base projection of a LoRA linear layer, [P1] 3.3: out[t][n] = sum_k x[t,k] * W[n,k]
 * (x: bf16 [M][ldx], W: bf16 [N][ldw], both K columns used; out: double [M][N]).
 */
void oracle_matmul_bt(int32_t M, int32_t N, int32_t K, const uint16_t *x, int64_t ldx, const uint16_t *W,
                      int64_t ldw, double *out)
{
    for (int32_t t = 0; t < M; ++t) {
        for (int32_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int32_t k = 0; k < K; ++k) acc += bf(x[(int64_t)t * ldx + k]) * bf(W[(int64_t)n * ldw + k]);
            out[(int64_t)t * N + n] = acc;
        }
    }
}

/*
 * Dense LoRA delta, [P1] 1.1 / 2.3 and [P5] stacked layers.
 *
 * For every token t with adapter i = ids[t] in [0, L):
 *   for every output slice s (width slice_n[s], first column off_s):
 *     S[j]        = sum_k x[t,k] * A_i[sa*r + j, k]          (j < r = rank[i])
 *     y[t, off_s+n] = y_base[t, off_s+n] + scale[i] * sum_j S[j] * B_i[off_s+n, j]
 *   where sa = s when A has one row block per slice (n_a == n_slices) and
 *   sa = 0 when all slices share one block (n_a == 1).
 * Tokens with ids[t] == -1 (or out of range) copy y_base.
 *
 * A[i]: bf16 [n_a * rank[i]][K] row-major.  B[i]: bf16 [N][rank[i]] row-major.
 * y_out: double [M][N].  enabled (nullable): adapters with enabled[i] == 0
 * behave like -1.  Returns the number of out-of-range ids.
 */
int oracle_lora_apply(int32_t M, int32_t K, int32_t n_slices, const int32_t *slice_n, int32_t n_a,
                      int32_t L, const int32_t *rank, const double *scale,
                      const uint16_t *const *A, const uint16_t *const *B,
                      const int32_t *ids, const uint8_t *enabled,
                      const uint16_t *x, int64_t ldx, const uint16_t *y_base, int64_t ldy,
                      double *y_out)
{
    int32_t N = 0;
    for (int32_t s = 0; s < n_slices; ++s) N += slice_n[s];
    int bad = 0;
    int32_t r_max = 1;
    for (int32_t i = 0; i < L; ++i) if (rank[i] > r_max) r_max = rank[i];
    double *S = (double *)malloc(sizeof(double) * (size_t)r_max);
    for (int32_t t = 0; t < M; ++t) {
        for (int32_t n = 0; n < N; ++n) y_out[(int64_t)t * N + n] = bf(y_base[(int64_t)t * ldy + n]);
        int32_t i = ids[t];
        if (i == -1) continue;
        if (i < -1 || i >= L) { ++bad; continue; }
        if (enabled && !enabled[i]) continue;
        int32_t r = rank[i];
        int32_t off = 0;
        for (int32_t s = 0; s < n_slices; ++s) {
            int32_t sa = (n_a == 1) ? 0 : s;
            /* shrink: S = x_t A_i^T restricted to row block sa */
            for (int32_t j = 0; j < r; ++j) {
                const uint16_t *arow = A[i] + (int64_t)(sa * r + j) * K;
                double acc = 0.0;
                for (int32_t k = 0; k < K; ++k) acc += bf(x[(int64_t)t * ldx + k]) * bf(arow[k]);
                S[j] = acc;
            }
            /* expand and add: y += scale * S B_i^T over this slice's columns */
            for (int32_t n = off; n < off + slice_n[s]; ++n) {
                const uint16_t *brow = B[i] + (int64_t)n * r;
                double acc = 0.0;
                for (int32_t j = 0; j < r; ++j) acc += S[j] * bf(brow[j]);
                y_out[(int64_t)t * N + n] += scale[i] * acc;
            }
            off += slice_n[s];
        }
    }
    free(S);
    return bad;
}

/*
 * Segment table by bucketing on lora_id, [P1] 2.3.
 *
 * A counting sort: count tokens per bucket (adapter 0..L-1, bucket L for -1,
 * disabled and out-of-range ids), exclusive prefix sum of the counts, then
 * place tokens in ascending t so each bucket keeps original token order.
 * Segments are the non-empty adapter buckets in ascending adapter id:
 * (adapter, start offset into perm, token count).
 * Returns the number of out-of-range ids.
 */
int oracle_build_segments(int32_t M, int32_t L, const int32_t *ids, const uint8_t *enabled,
                          int32_t *perm, int32_t *seg_adapter, int32_t *seg_start, int32_t *seg_len,
                          int32_t *num_segments, int32_t *num_valid)
{
    int bad = 0;
    int64_t *count = (int64_t *)calloc((size_t)L + 1, sizeof(int64_t));
    int64_t *next = (int64_t *)calloc((size_t)L + 1, sizeof(int64_t));
    int32_t *key = (int32_t *)malloc(sizeof(int32_t) * (size_t)(M > 0 ? M : 1));
    for (int32_t t = 0; t < M; ++t) {
        int32_t i = ids[t];
        int32_t b = L;
        if (i >= 0 && i < L) {
            if (!enabled || enabled[i]) b = i;
        } else if (i != -1) {
            ++bad;
        }
        key[t] = b;
        count[b] += 1;
    }
    int64_t run = 0;
    for (int32_t b = 0; b <= L; ++b) { next[b] = run; run += count[b]; }
    for (int32_t t = 0; t < M; ++t) perm[next[key[t]]++] = t;
    int32_t ns = 0;
    int64_t start = 0;
    for (int32_t b = 0; b < L; ++b) {
        if (count[b] > 0) {
            seg_adapter[ns] = b;
            seg_start[ns] = (int32_t)start;
            seg_len[ns] = (int32_t)count[b];
            ++ns;
        }
        start += count[b];
    }
    *num_segments = ns;
    *num_valid = (int32_t)start;
    free(count);
    free(next);
    free(key);
    return bad;
}

/*
 * (adapter, expert) block alignment for the MoE variant, [P2]
 * "MoE LoRA Alignment" (moe_lora_align_block_size).
 *
 * Pairs p = t*topk + k, expert topk_ids[p].  For every adapter l:
 *   for e = 0..E-1 in order:
 *     append every pair p (ascending) with ids[p/topk] == l and topk_ids[p] == e,
 *     then pad with the sentinel M*topk to a multiple of block_m;
 *     every block of that padded group gets expert id e.
 *   num_tokens_post_padded[l] = total padded length; remaining slots of the
 *   [P_max] row hold the sentinel, remaining block ids are -1.
 * Disabled adapters get length 0.  Pairs with an out-of-range expert or
 * adapter id are skipped and counted.  Returns that count.
 */
int oracle_moe_align(int32_t M, int32_t topk, int32_t E, int32_t L, int32_t block_m,
                     const int32_t *ids, const int32_t *topk_ids, const uint8_t *enabled,
                     int32_t P_max, int32_t B_max,
                     int32_t *sorted_ids, int32_t *expert_ids, int32_t *num_tokens_post_padded)
{
    int bad = 0;
    const int32_t P = M * topk;
    const int32_t sentinel = P;
    for (int32_t p = 0; p < P; ++p) {
        int32_t i = ids[p / topk];
        int32_t e = topk_ids[p];
        if ((i < -1 || i >= L) || (i >= 0 && (e < 0 || e >= E))) ++bad;
    }
    for (int32_t l = 0; l < L; ++l) {
        int32_t *row = sorted_ids + (int64_t)l * P_max;
        int32_t *blk = expert_ids + (int64_t)l * B_max;
        for (int32_t q = 0; q < P_max; ++q) row[q] = sentinel;
        for (int32_t b = 0; b < B_max; ++b) blk[b] = -1;
        int32_t pos = 0;
        if (!enabled || enabled[l]) {
            for (int32_t e = 0; e < E; ++e) {
                int32_t cnt = 0;
                for (int32_t p = 0; p < P; ++p) {
                    if (ids[p / topk] == l && topk_ids[p] == e) {
                        row[pos + cnt] = p;
                        ++cnt;
                    }
                }
                int32_t padded = ((cnt + block_m - 1) / block_m) * block_m;
                for (int32_t b = pos / block_m; b < (pos + padded) / block_m; ++b) blk[b] = e;
                pos += padded;
            }
        }
        num_tokens_post_padded[l] = pos;
    }
    return bad;
}

/*
 * MoE LoRA delta for one stage, [P2] stages 1.5 and 3.5.
 *
 * For every pair p = t*topk + k whose token has adapter l = ids[t] in
 * [0, L) (enabled) and whose expert e = topk_ids[p] is in [0, E):
 *   u      = (src_is_token ? src[t] : src[p])        (row of length K)
 *   S[j]   = sum_c u[c] * A_l[ea][j][c]                 ea = (E_A == 1 ? 0 : e)
 *   out[p][n] = cache[p][n] + w * scale[l] * sum_j S[j] * B_l[eb][n][j],  eb likewise
 *   w = topk_weights[p] when given, else 1.
 * Other pairs copy cache.  gate/up: src = hidden states (per token), A shared
 * by the experts, N = 2*intermediate; the result feeds SiLU-mul.  down:
 * src = SiLU-mul output (per pair), B shared, N = hidden; the result feeds the
 * top-k reduce.
 *
 * A[l]: bf16 [E_A][rank[l]][K].  B[l]: bf16 [E_B][N][rank[l]].  out: double [P][N].
 */
int oracle_moe_delta(int32_t M, int32_t topk, int32_t E, int32_t L, int32_t K, int32_t N,
                     const int32_t *rank, const double *scale, int32_t E_A, int32_t E_B,
                     const uint16_t *const *A, const uint16_t *const *B,
                     const int32_t *ids, const int32_t *topk_ids, const uint8_t *enabled,
                     const float *topk_weights, int32_t src_is_token,
                     const uint16_t *src, int64_t ld_src, const uint16_t *cache, int64_t ld_cache,
                     double *out)
{
    int bad = 0;
    const int32_t P = M * topk;
    int32_t r_max = 1;
    for (int32_t i = 0; i < L; ++i) if (rank[i] > r_max) r_max = rank[i];
    double *S = (double *)malloc(sizeof(double) * (size_t)r_max);
    for (int32_t p = 0; p < P; ++p) {
        for (int32_t n = 0; n < N; ++n) out[(int64_t)p * N + n] = bf(cache[(int64_t)p * ld_cache + n]);
        int32_t t = p / topk;
        int32_t l = ids[t];
        int32_t e = topk_ids[p];
        if (l == -1) continue;
        if (l < -1 || l >= L || e < 0 || e >= E) { ++bad; continue; }
        if (enabled && !enabled[l]) continue;
        int32_t r = rank[l];
        const uint16_t *a = A[l] + (int64_t)(E_A == 1 ? 0 : e) * r * K;
        const uint16_t *b = B[l] + (int64_t)(E_B == 1 ? 0 : e) * N * r;
        const uint16_t *u = src + (int64_t)(src_is_token ? t : p) * ld_src;
        for (int32_t j = 0; j < r; ++j) {
            double acc = 0.0;
            for (int32_t c = 0; c < K; ++c) acc += bf(u[c]) * bf(a[(int64_t)j * K + c]);
            S[j] = acc;
        }
        double w = topk_weights ? (double)topk_weights[p] : 1.0;
        for (int32_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int32_t j = 0; j < r; ++j) acc += S[j] * bf(b[(int64_t)n * r + j]);
            out[(int64_t)p * N + n] += w * scale[l] * acc;
        }
    }
    free(S);
    return bad;
}
