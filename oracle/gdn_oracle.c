/*
 * Oracle for the gated delta rule: a plain, slow, float64 CPU recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; it exists so that tests, the smoke check and the CPU
 * baseline in the benchmark can compare the CUDA library against an
 * independent computation of the same definition.  It shares no code with
 * the CUDA sources.
 *
 * What it computes (one independent problem per (sequence, head) pair):
 *
 *   S_0 = state_in[b,h]            (d x d, S[i][j]: i = value index, j = key index)
 *   for t = 0 .. T-1:
 *     alpha = exp(g[b,t,h])        (the gate arrives in the log domain and is
 *                                   exponentiated here)
 *     S <- alpha * S                                   -- gating (decay)
 *     r <- S k_t                                        -- what the memory says for k_t
 *     S <- S + beta_t (v_t - r) k_t^T                   -- delta rule: overwrite
 *     o_t <- S q_t / sqrt(d)                            -- output from the updated state
 *   state_out[b,h] = S
 *
 * which is S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T and
 * o_t = S_t q_t / sqrt(d) written step by step.
 *
 * Sources:
 *   - "Gated Delta Net on AMD: why ROCm stumbles on hybrid-attention LLMs",
 *     section "What Gated Delta Net is, in plain language": the delta rule
 *     overwrites the part of the running summary that new information
 *     contradicts; the gate scales how much of the old summary is kept.
 *   - "marcsun13/ggml-gated-delta-net" model card, section "Ops": one call
 *     covers a whole run of steps, (q, k, v, g, beta, state) -> (out,
 *     final_state); shapes q,k,v (n_seqs, n_tokens, n_heads, head_dim),
 *     g,beta (n_seqs, n_tokens, n_heads), state (n_seqs, n_heads, d, d);
 *     state indexed [value][key], a fresh state is zeros; one key head per
 *     value head; the output carries 1/sqrt(head_dim); g is a log-domain gate.
 *   - same model card, the first contract note under the shape table: with
 *     fewer key heads than value heads, upstream maps value head i to key
 *     head i % n_k_heads (the tiled convention).  q and k then carry n_k_heads
 *     heads; n_k_heads == n_heads is the identity mapping.
 *
 * Option l2norm_qk (the op's fused preprocessing, off by default): q_t and
 * k_t are first replaced by q_t / |q_t| and k_t / |k_t| (Euclidean norm over
 * the head's d components, in double); a zero vector stays zero.  The model
 * card's "Ops" section counts this normalisation among the eager ops that
 * surround the recurrence in a Gated DeltaNet layer, and the synthetic
 * workloads normalise q and k per head this way.
 *
 * Inputs are float32 (bf16 data is upcast exactly by the caller); every
 * operation is done in double.  No blocking, no reordering beyond the
 * definition above, no fast-math.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One (sequence, head) problem.  Element strides are given so the caller can
 * pass the (b, h) slice of a (B, T, H, d) array without copying:
 *   q/k:       token t, component j at [t * qk_stride + j]
 *   v/out:     token t, component i at [t * tok_stride + i]
 *   g/beta:    token t at [t * gate_stride]
 *   state:     S[i][j] at [i * d + j]                                      */
/* x (d floats) as double into y, divided by its Euclidean norm when
 * `normalise` is set (a zero vector stays zero). */
static void load_vec(const float *x, double *y, int d, int normalise)
{
    double ss = 0.0;
    for (int j = 0; j < d; ++j) {
        y[j] = (double)x[j];
        ss += y[j] * y[j];
    }
    if (normalise && ss > 0.0) {
        const double n = sqrt(ss);
        for (int j = 0; j < d; ++j)
            y[j] /= n;
    }
}

static void oracle_one_head(const float *q, const float *k, const float *v,
                            const float *g, const float *beta, long qk_stride,
                            long tok_stride, long gate_stride,
                            const float *state_in, double *out,
                            double *state_out, int T, int d, double *S,
                            double *r, double *qv, double *kv, int l2norm_qk)
{
    const double inv_sqrt_d = 1.0 / sqrt((double)d);
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j)
            S[(size_t)i * d + j] = state_in ? (double)state_in[(size_t)i * d + j] : 0.0;

    for (int t = 0; t < T; ++t) {
        load_vec(q + (size_t)t * qk_stride, qv, d, l2norm_qk);
        load_vec(k + (size_t)t * qk_stride, kv, d, l2norm_qk);
        const double *qt = qv;
        const double *kt = kv;
        const float *vt = v + (size_t)t * tok_stride;
        const double alpha = exp((double)g[(size_t)t * gate_stride]);
        const double b = (double)beta[(size_t)t * gate_stride];

        /* gating: S <- alpha S */
        for (size_t e = 0; e < (size_t)d * d; ++e)
            S[e] *= alpha;
        /* r = S k */
        for (int i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int j = 0; j < d; ++j)
                acc += S[(size_t)i * d + j] * kt[j];
            r[i] = acc;
        }
        /* delta rule: S <- S + beta (v - r) k^T */
        for (int i = 0; i < d; ++i) {
            const double c = b * ((double)vt[i] - r[i]);
            for (int j = 0; j < d; ++j)
                S[(size_t)i * d + j] += c * kt[j];
        }
        /* o = S q / sqrt(d) */
        double *ot = out + (size_t)t * tok_stride;
        for (int i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int j = 0; j < d; ++j)
                acc += S[(size_t)i * d + j] * qt[j];
            ot[i] = acc * inv_sqrt_d;
        }
    }
    memcpy(state_out, S, sizeof(double) * (size_t)d * d);
}

/* Full problem, all (b, h) pairs.  Layouts as on the model card:
 *   q, k         : (B, T, Hk, d) contiguous; value head h reads key head h % Hk
 *   v, out       : (B, T, H, d) contiguous
 *   g, beta      : (B, T, H) contiguous
 *   state_in     : (B, H, d, d) contiguous, [value][key]; NULL means zeros
 *   state_out    : (B, H, d, d) contiguous, [value][key]
 * n_threads <= 0 uses the OpenMP default.  l2norm_qk != 0 normalises q and k
 * first (see the header).  Returns 0, or -1 on bad sizes or an allocation
 * failure (outputs are then unspecified).                                  */
int gdn_oracle_forward(const float *q, const float *k, const float *v,
                       const float *g, const float *beta,
                       const float *state_in, double *out, double *state_out,
                       int B, int T, int H, int Hk, int d, int n_threads,
                       int l2norm_qk)
{
    if (B < 0 || T < 0 || H < 0 || d <= 0 || Hk <= 0 || Hk > (H > 0 ? H : 1))
        return -1;
    const long qk_stride = (long)Hk * d;
    const long tok_stride = (long)H * d;
    const long gate_stride = H;
    const long n_pairs = (long)B * H;
    int failed = 0;
#ifdef _OPENMP
    /* The count applies to this call only: a one-thread call leaves the
     * default for the calls after it unchanged. */
    const int nt = n_threads > 0 ? n_threads : omp_get_max_threads();
#else
    (void)n_threads;
#endif
#pragma omp parallel num_threads(nt)
    {
        double *S = (double *)malloc(sizeof(double) * (size_t)d * d);
        double *r = (double *)malloc(sizeof(double) * (size_t)d * 3);
        if (!S || !r) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (long p = 0; p < n_pairs; ++p) {
            if (!S || !r)
                continue;
            const long b = p / H, h = p % H;
            const size_t in_off = (size_t)b * T * H * d + (size_t)h * d;
            const size_t qk_off = (size_t)b * T * Hk * d + (size_t)(h % Hk) * d;
            const size_t gb_off = (size_t)b * T * H + (size_t)h;
            const size_t st_off = (size_t)p * d * d;
            oracle_one_head(q + qk_off, k + qk_off, v + in_off, g + gb_off,
                            beta + gb_off, qk_stride, tok_stride, gate_stride,
                            state_in ? state_in + st_off : NULL,
                            out + in_off, state_out + st_off, T, d, S, r, r + d,
                            r + 2 * (size_t)d, l2norm_qk);
        }
        free(S);
        free(r);
    }
    return failed ? -1 : 0;
}

/* Number of threads an OpenMP parallel region would use (for reporting). */
int gdn_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
