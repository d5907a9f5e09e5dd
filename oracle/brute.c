/*
 * Brute-force causal chunk attention in long double, for tiny inputs.
 *
 * TEST INFRASTRUCTURE ONLY: it checks the NumPy oracle and is never linked
 * into the product library.
 *
 * Computes Eq. (1) of "VPP: Virtual Pipeline Parallelism for Efficient Chunked
 * Prefill in Long-Context LLM Inference" (English technical review, §2.2),
 * softmax(Q K^T * scale) V, with the causal rule of the same section (token i
 * attends to tokens <= i) for a chunk whose first query sits at absolute
 * position prefix_len (§2.3, chunked prefill).  Every score, exponential and
 * sum is a separate scalar loop; nothing is blocked or reordered.
 *
 * Layouts (row-major, double):
 *   q   [C][Hq][dq]          k [P+C][Hkv][dq]      v [P+C][Hkv][dv]
 *   out [C][Hq][dv]          lse [Hq][C]  (natural log of the denominator)
 * Query head h reads kv head h / (Hq / Hkv).
 * Returns 0 on success, -1 on invalid sizes.
 */
#include <math.h>
#include <stdlib.h>

int brute_causal_chunk_attention(const double *q, const double *k, const double *v,
                                 int C, int P, int Hq, int Hkv, int dq, int dv,
                                 double scale, double *out, double *lse)
{
    if (C < 0 || P < 0 || Hq <= 0 || Hkv <= 0 || dq <= 0 || dv <= 0 || Hq % Hkv != 0)
        return -1;
    int G = Hq / Hkv;
    int T = P + C;
    long double *score = (long double *)malloc(sizeof(long double) * (size_t)(T > 0 ? T : 1));
    if (!score)
        return -1;
    for (int i = 0; i < C; ++i) {
        int pos = P + i; /* keys 0..pos are visible */
        for (int h = 0; h < Hq; ++h) {
            int g = h / G;
            long double mx = -INFINITY;
            for (int j = 0; j <= pos; ++j) {
                long double acc = 0.0L;
                for (int c = 0; c < dq; ++c)
                    acc += (long double)q[((size_t)i * Hq + h) * dq + c] *
                           (long double)k[((size_t)j * Hkv + g) * dq + c];
                score[j] = acc * (long double)scale;
                if (score[j] > mx)
                    mx = score[j];
            }
            long double den = 0.0L;
            for (int j = 0; j <= pos; ++j)
                den += expl(score[j] - mx);
            for (int c = 0; c < dv; ++c) {
                long double num = 0.0L;
                for (int j = 0; j <= pos; ++j)
                    num += expl(score[j] - mx) * (long double)v[((size_t)j * Hkv + g) * dv + c];
                out[((size_t)i * Hq + h) * dv + c] = (double)(num / den);
            }
            lse[(size_t)h * C + i] = (double)(mx + logl(den));
        }
    }
    free(score);
    return 0;
}
