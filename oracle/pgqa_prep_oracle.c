/*
 * CPU oracle, in f64, for the step that precedes paged attention: per-head
 * RMSNorm of the projected Q and K (and, optionally, a weightless RMSNorm of
 * V), rotary position embedding of Q and K, and the paged write of K and V
 * into the [page][nkv][16][hd] pools.  TEST INFRASTRUCTURE ONLY: the library
 * under paged_gqa_decode_attn_gb300/ never links, loads or calls this file,
 * and this file shares no code or header with it.
 *
 * The step is the QK-RMSNorm/RoPE pool write whose device gates pegainfer
 * PR #1002 ("reduce the duplicated CPU operator oracles in the HD256/HD512
 * QK-RoPE smokes") describes: RMSNorm and RoPE over a head vector of hd
 * dims, rotation over the first rotary_dim dims (the "rope-lo" and "rope-hi"
 * halves) with the remaining dims passed through, K and V landing at the
 * paged-KV address of the token's position.  The page gives no formula, so
 * this is the plainest reading, stated once here:
 *
 *   RMSNorm   r = 1 / sqrt(mean_d x_d^2 + eps),  y_d = x_d * r * w_d
 *             (V: y_d = x_d * r, no weight, when norm_v; else y = x)
 *   RoPE      half = rotary_dim / 2; for i < half, f_i = theta^(-2i / rotary_dim),
 *             a = pos * f_i:
 *               y'_i        = y_i cos a - y_{i+half} sin a
 *               y'_{i+half} = y_{i+half} cos a + y_i sin a
 *             dims >= rotary_dim unchanged; V is not rotated
 *   address   page = block_table[off[t] + pos[t]/16] (then page_map[page]),
 *             element ((page*nkv + kh)*16 + pos[t]%16)*hd + d
 *
 * Inputs are bf16 bits (widened exactly to f64), weights bf16 bits.  Results
 * are f64; the test compares the device's bf16 against them within a bound.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static double bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* RMSNorm of one head vector (x: hd bf16), scaled by w (bf16) unless w is NULL. */
static void rms_norm(const uint16_t *x, const uint16_t *w, int hd, double eps, double *y)
{
    double ss = 0.0;
    for (int d = 0; d < hd; ++d) {
        double v = bf16_value(x[d]);
        ss += v * v;
    }
    double r = 1.0 / sqrt(ss / hd + eps);
    for (int d = 0; d < hd; ++d)
        y[d] = bf16_value(x[d]) * r * (w ? bf16_value(w[d]) : 1.0);
}

/* Rotary embedding of y (in place) at position pos over its first rotary_dim dims. */
static void rope(double *y, int rotary_dim, double theta, int pos)
{
    int half = rotary_dim / 2;
    for (int i = 0; i < half; ++i) {
        double f = pow(theta, -2.0 * i / rotary_dim);
        double a = (double)pos * f;
        double c = cos(a), s = sin(a);
        double lo = y[i], hi = y[i + half];
        y[i] = lo * c - hi * s;
        y[i + half] = hi * c + lo * s;
    }
}

/*
 * q_out: [rows][nh][hd], k_out / v_out: [rows][nkv][hd] (f64, the values the
 * step writes); slot: [rows] the element offset of (row, kv head 0, dim 0) in
 * the pool (kv head kh adds kh*16*hd).  Returns 0, or -1 for bad sizes.
 */
int pgqa_prep_oracle(const uint16_t *q_in, const uint16_t *k_in, const uint16_t *v_in, const uint16_t *q_weight,
                     const uint16_t *k_weight, const int32_t *pos, const int32_t *block_table, const int32_t *off,
                     const int32_t *page_map, int rows, int nh, int nkv, int hd, int rotary_dim, double theta,
                     double eps, int norm_v, double *q_out, double *k_out, double *v_out, int64_t *slot)
{
    if (rows < 0 || nh < 1 || nkv < 1 || hd < 2 || rotary_dim < 0 || rotary_dim > hd || rotary_dim % 2)
        return -1;
    for (int t = 0; t < rows; ++t) {
        for (int h = 0; h < nh; ++h) {
            double *y = q_out + ((int64_t)t * nh + h) * hd;
            rms_norm(q_in + ((int64_t)t * nh + h) * hd, q_weight, hd, eps, y);
            rope(y, rotary_dim, theta, pos[t]);
        }
        for (int kh = 0; kh < nkv; ++kh) {
            double *yk = k_out + ((int64_t)t * nkv + kh) * hd;
            rms_norm(k_in + ((int64_t)t * nkv + kh) * hd, k_weight, hd, eps, yk);
            rope(yk, rotary_dim, theta, pos[t]);
            double *yv = v_out + ((int64_t)t * nkv + kh) * hd;
            const uint16_t *xv = v_in + ((int64_t)t * nkv + kh) * hd;
            if (norm_v)
                rms_norm(xv, NULL, hd, eps, yv);
            else
                for (int d = 0; d < hd; ++d)
                    yv[d] = bf16_value(xv[d]);
        }
        int64_t page = block_table[(int64_t)off[t] + pos[t] / 16];
        if (page_map)
            page = page_map[page];
        slot[t] = (page * nkv * 16 + pos[t] % 16) * (int64_t)hd;
    }
    return 0;
}
