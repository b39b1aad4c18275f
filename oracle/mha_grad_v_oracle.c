/*
 * CPU oracle for the attention gradient with respect to V (test
 * infrastructure only).
 *
 * Page: mha_grad_v.wgsl (meganeura 0.2.0), its Params struct and entry point.
 * Layouts (row-major): Q and dO [q_seq][num_heads][head_dim], K [kv][num_kv_heads]
 * [head_dim], LSE [q_seq][num_heads][2] = (max score, log of the sum of
 * exp(score - max)) from the forward pass, dV [kv][num_kv_heads][head_dim].
 * kv_seq == 0 means causal self-attention with kv = q_seq; otherwise kv = kv_seq.
 * For KV position t and KV head g, with heads_per_kv = num_heads / num_kv_heads:
 *
 *   start = causal ? t : 0,   end = window > 0 ? min(q_seq, t + window) : q_seq,
 *   dV[t][g][:] = sum over pos in [start, end) and head h of group g
 *                 (h = g * heads_per_kv + r) of  P * dO[pos][h][:],
 *   P = exp(min(s - max[pos][h], 0) - logsum[pos][h]),
 *   s = (sum over d of Q[pos][h][d] * K[t][g][d]) / sqrt(head_dim).
 *
 * These functions restate that with plain double loops in the page's order
 * (nothing blocked or fused); nothing here is shared with the CUDA library.
 * oracle_mha_forward_lse_f64 produces the forward statistics that the
 * definition consumes, over the keys each query attends (t <= pos when causal,
 * t > pos - window when windowed): the inputs for consistent test cases.
 * Pins: tests/test_mha_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>

static int check(int q_seq, int kv_seq, int nh, int nkv, int hd) {
    if (q_seq <= 0 || kv_seq < 0 || nh <= 0 || nkv <= 0 || hd <= 0 || nh % nkv != 0) return -1;
    return 0;
}

/* Rows t in [t_begin, t_end) of dV as defined above (dv holds those rows
 * only, from row t_begin).  Returns 0, or -1 for a bad shape or range. */
int oracle_mha_grad_v_rows_f64(const double *q, const double *k, const double *d_out, const double *lse,
                               double *dv, int q_seq, int kv_seq, int num_heads, int num_kv_heads, int head_dim,
                               int window, int t_begin, int t_end) {
    if (check(q_seq, kv_seq, num_heads, num_kv_heads, head_dim) != 0 || window < 0) return -1;
    const int causal = kv_seq == 0;
    const int kv = causal ? q_seq : kv_seq;
    if (t_begin < 0 || t_end > kv || t_begin > t_end) return -1;
    const int hpk = num_heads / num_kv_heads;
    const int64_t q_dim = (int64_t)num_heads * head_dim, kv_dim = (int64_t)num_kv_heads * head_dim;
    const double scale = 1.0 / sqrt((double)head_dim);
    for (int t = t_begin; t < t_end; ++t)
        for (int g = 0; g < num_kv_heads; ++g) {
            const double *kt = k + t * kv_dim + (int64_t)g * head_dim;
            double *out = dv + (t - t_begin) * kv_dim + (int64_t)g * head_dim;
            for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
            const int start = causal ? t : 0;
            int end = q_seq;
            if (window > 0 && t + window < end) end = t + window;
            for (int pos = start; pos < end; ++pos)
                for (int r = 0; r < hpk; ++r) {
                    const int h = g * hpk + r;
                    const double *qp = q + pos * q_dim + (int64_t)h * head_dim;
                    double s = 0.0;
                    for (int d = 0; d < head_dim; ++d) s += qp[d] * kt[d];
                    s *= scale;
                    const double *st = lse + ((int64_t)pos * num_heads + h) * 2;
                    double e = s - st[0];
                    if (e > 0.0) e = 0.0;
                    const double p = exp(e - st[1]);
                    const double *go = d_out + pos * q_dim + (int64_t)h * head_dim;
                    for (int d = 0; d < head_dim; ++d) out[d] += p * go[d];
                }
        }
    return 0;
}

/* dV as defined above, every row.  Returns 0, or -1 for a bad shape. */
int oracle_mha_grad_v_f64(const double *q, const double *k, const double *d_out, const double *lse, double *dv,
                          int q_seq, int kv_seq, int num_heads, int num_kv_heads, int head_dim, int window) {
    const int kv = kv_seq == 0 ? q_seq : kv_seq;
    return oracle_mha_grad_v_rows_f64(q, k, d_out, lse, dv, q_seq, kv_seq, num_heads, num_kv_heads, head_dim,
                                      window, 0, kv < 0 ? 0 : kv);
}

/* Forward statistics (max score, log of sum of exp(score - max)) of every
 * query position and head over the keys it attends: t < kv, and t <= pos when
 * causal, and t > pos - window when window > 0.  A query that attends no key
 * gets (0, 0).  Returns 0, or -1 for a bad shape. */
int oracle_mha_forward_lse_f64(const double *q, const double *k, double *lse, int q_seq, int kv_seq,
                               int num_heads, int num_kv_heads, int head_dim, int window) {
    if (check(q_seq, kv_seq, num_heads, num_kv_heads, head_dim) != 0 || window < 0) return -1;
    const int causal = kv_seq == 0;
    const int kv = causal ? q_seq : kv_seq;
    const int hpk = num_heads / num_kv_heads;
    const int64_t q_dim = (int64_t)num_heads * head_dim, kv_dim = (int64_t)num_kv_heads * head_dim;
    const double scale = 1.0 / sqrt((double)head_dim);
    for (int pos = 0; pos < q_seq; ++pos)
        for (int h = 0; h < num_heads; ++h) {
            const int g = h / hpk;
            const double *qp = q + pos * q_dim + (int64_t)h * head_dim;
            double mx = -INFINITY;
            for (int pass = 0; pass < 2; ++pass) {
                double sum = 0.0;
                for (int t = 0; t < kv; ++t) {
                    if (causal && t > pos) continue;
                    if (window > 0 && t <= pos - window) continue;
                    const double *kt = k + t * kv_dim + (int64_t)g * head_dim;
                    double s = 0.0;
                    for (int d = 0; d < head_dim; ++d) s += qp[d] * kt[d];
                    s *= scale;
                    if (pass == 0) {
                        if (s > mx) mx = s;
                    } else {
                        sum += exp(s - mx);
                    }
                }
                if (pass == 1) {
                    double *st = lse + ((int64_t)pos * num_heads + h) * 2;
                    if (mx == -INFINITY) {
                        st[0] = 0.0;
                        st[1] = 0.0;
                    } else {
                        st[0] = mx;
                        st[1] = log(sum);
                    }
                }
            }
        }
    return 0;
}
