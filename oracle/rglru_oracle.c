/*
 * RG-LRU oracle: TEST INFRASTRUCTURE ONLY.
 *
 * A plain, serial-per-channel, float64 CPU statement of what the RG-LRU hot path computes,
 * written from the method's definition and used only to check the CUDA library.  Only the
 * tests, the smoke check and the benchmark's CPU-baseline leg may load it; the product path
 * never does.  It shares no source, header, table or helper with the CUDA library.
 *
 * Method (Fattori comparison page, "the operator fuses" list and "semantic limits" list):
 *   r_t = sigmoid(lr_t)                 recurrence gate        (bullet 1: sigmoid activations)
 *   i_t = sigmoid(li_t)                 input gate             (bullet 1)
 *   log a_t = -8 * r_t * softplus(L)    dynamic decay, c = 8   (bullet 2: softplus(a_param),
 *                                                               dynamic decay; the constant and
 *                                                               its sign are fixed by the
 *                                                               specification, not the page)
 *   m_t = sqrt(1 - a_t^2)               stationary multiplier  (bullet 2)
 *   h_t = a_t h_{t-1} + m_t (i_t x_t)   input-gated write and state-stationary recurrence
 *                                                              (bullets 3 and 4)
 * Canonical mode (same page, "semantic limits" list: segment_pos / reset / initial state and
 * the reset-token normalisation): at a reset token the previous state is dropped
 * (h_{t-1} := 0) and m_t = 1; the state before token 0 is h0.  Restricted mode (the page's
 * benchmark record, "protocol" and "correctness.contract"): zero initial state, no resets,
 * sqrt(1 - a^2) on every token.
 *
 * Gate logits come from block-diagonal projections (Fattori comparison page, first paragraph;
 * benchmark record "protocol.scope"): per gate block `blk` of width k,
 *   lr[., blk*k + j] = sum_i x[., blk*k + i] * Wa[blk][i][j] + ba[blk*k + j]   (W stored (in, out))
 * and the same for li with Wx, bx.
 *
 * The backward is the exact derivative of the loss  L = sum y*dy + sum hT*dhT, derived by
 * hand from the recurrence above (the page's "reverse recurrence and pointwise derivatives"
 * of the custom backward):
 *   g_t   = dy_t + abar_{t+1} g_{t+1},  g_{T-1} = dy_{T-1} + dhT      (total dL/dh_t)
 *   dla_t = abar_t * g_t * (h_{t-1} - u_t abar_t / m_t)  on non-reset tokens, 0 on reset tokens
 *           (u_t = i_t x_t; d a/d la = a, d m/d la = -a^2/m)
 *   dlr_t = dla_t * (-8 softplus(L)) * r_t (1 - r_t)
 *   du_t  = g_t m_t,  dx_t = du_t i_t,  dli_t = du_t x_t i_t (1 - i_t)
 *   dL_w  = sigmoid(L_w) * sum_{b,t} dla_t * (-8 r_t)
 *   dh0   = abar_0 g_0  (canonical; the state before token 0 is h0)
 * Projection backward: dx += dlr Wa^T + dli Wx^T per block, dW = x^T dl per block,
 * db = sum over tokens of dl.
 *
 * Everything is float64.  The per-channel loops run in the order written; channels and
 * rows are independent, so the OpenMP split over them changes no arithmetic.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_CANONICAL 0
#define ORACLE_RESTRICTED 1

static double sigmoid_d(double z) { return 1.0 / (1.0 + exp(-z)); }

/* softplus(z) = log(1 + e^z), written so that large |z| neither overflows nor loses digits. */
static double softplus_d(double z) { return z > 0.0 ? z + log1p(exp(-z)) : log1p(exp(z)); }

/* Reset at (b, t): reset_mask != 0, or segment_pos == 0.  At most one of the two is given. */
static int is_reset(const uint8_t *reset_mask, const int32_t *segment_pos, long bt) {
  if (reset_mask) return reset_mask[bt] != 0;
  if (segment_pos) return segment_pos[bt] == 0;
  return 0;
}

/* Forward of the recurrence.  Arrays are [B, T, W] row-major (W contiguous); Lambda [W];
 * reset_mask / segment_pos [B, T] (nullable); h0 [B, W] (nullable => zeros); hT [B, W]. */
int oracle_forward(int mode, int B, int T, int W, const double *x, const double *lr,
                   const double *li, const double *Lambda, const uint8_t *reset_mask,
                   const int32_t *segment_pos, const double *h0, double *y, double *hT) {
  if (B < 1 || T < 1 || W < 1) return 1;
  const int canonical = (mode == ORACLE_CANONICAL);
  long n_chan = (long)B * W;
#pragma omp parallel for schedule(static)
  for (long bw = 0; bw < n_chan; ++bw) {
    const long b = bw / W, w = bw % W;
    const double sp = softplus_d(Lambda[w]);
    double h = (canonical && h0) ? h0[b * W + w] : 0.0;
    for (long t = 0; t < T; ++t) {
      const long bt = b * T + t;
      const long idx = bt * W + w;
      const double r = sigmoid_d(lr[idx]);
      const double i = sigmoid_d(li[idx]);
      const double la = -8.0 * r * sp;
      const double a = exp(la);
      const int rst = canonical && is_reset(reset_mask, segment_pos, bt);
      const double abar = rst ? 0.0 : a;
      const double m = rst ? 1.0 : sqrt(-expm1(2.0 * la)); /* sqrt(1 - a^2) */
      h = abar * h + m * (i * x[idx]);
      y[idx] = h;
    }
    hT[b * W + w] = h;
  }
  return 0;
}

/* Backward of the recurrence.  dy [B,T,W]; dhT [B,W] nullable (zero); outputs dx, dlr, dli
 * [B,T,W], dLambda [W], dh0 [B,W] (nullable; zero in restricted mode). */
int oracle_backward(int mode, int B, int T, int W, const double *x, const double *lr,
                    const double *li, const double *Lambda, const uint8_t *reset_mask,
                    const int32_t *segment_pos, const double *h0, const double *dy,
                    const double *dhT, double *dx, double *dlr, double *dli, double *dLambda,
                    double *dh0) {
  if (B < 1 || T < 1 || W < 1) return 1;
  const int canonical = (mode == ORACLE_CANONICAL);
  int status = 0;
#pragma omp parallel
  {
    /* Per-thread scratch for one channel's recomputed forward. */
    double *r_s = (double *)malloc(sizeof(double) * (size_t)T * 6);
    int *rst_s = (int *)malloc(sizeof(int) * (size_t)T);
#pragma omp for schedule(static)
    for (long w = 0; w < W; ++w) {
      if (!r_s || !rst_s) {
#pragma omp atomic write
        status = 2;
        continue;
      }
      double *a_s = r_s + T, *m_s = r_s + 2 * (size_t)T, *i_s = r_s + 3 * (size_t)T;
      double *hprev_s = r_s + 4 * (size_t)T, *abar_s = r_s + 5 * (size_t)T;
      const double sp = softplus_d(Lambda[w]);
      double dsp_total = 0.0;
      for (long b = 0; b < B; ++b) {
        /* Recompute the forward for channel (b, w). */
        double h = (canonical && h0) ? h0[b * W + w] : 0.0;
        for (long t = 0; t < T; ++t) {
          const long bt = b * T + t, idx = bt * W + w;
          const double r = sigmoid_d(lr[idx]);
          const double i = sigmoid_d(li[idx]);
          const double la = -8.0 * r * sp;
          const double a = exp(la);
          const int rst = canonical && is_reset(reset_mask, segment_pos, bt);
          r_s[t] = r;
          i_s[t] = i;
          a_s[t] = a;
          rst_s[t] = rst;
          abar_s[t] = rst ? 0.0 : a;
          m_s[t] = rst ? 1.0 : sqrt(-expm1(2.0 * la));
          hprev_s[t] = h;
          h = abar_s[t] * h + m_s[t] * (i * x[idx]);
        }
        /* Reverse recurrence for g = dL/dh and the pointwise derivatives. */
        double g_next = 0.0, dsp_b = 0.0;
        for (long t = T - 1; t >= 0; --t) {
          const long idx = (b * T + t) * W + w;
          double g = dy[idx];
          if (t == T - 1) {
            if (dhT) g += dhT[b * W + w];
          } else {
            g += abar_s[t + 1] * g_next;
          }
          const double r = r_s[t], i = i_s[t], a = a_s[t], m = m_s[t];
          const double u = i * x[idx];
          const double dla = rst_s[t] ? 0.0 : a * g * (hprev_s[t] - u * a / m);
          dlr[idx] = dla * (-8.0 * sp) * r * (1.0 - r);
          const double du = g * m;
          dx[idx] = du * i;
          dli[idx] = du * x[idx] * i * (1.0 - i);
          dsp_b += dla * (-8.0 * r);
          g_next = g;
        }
        if (dh0) dh0[b * W + w] = canonical ? abar_s[0] * g_next : 0.0;
        dsp_total += dsp_b;
      }
      dLambda[w] = sigmoid_d(Lambda[w]) * dsp_total; /* softplus' = sigmoid */
    }
    free(r_s);
    free(rst_s);
  }
  return status;
}

/* Block-diagonal gate projections.  x [B*T, W]; Wa, Wx [nblk, k, k] stored (in, out);
 * ba, bx [W] (nullable => zero); outputs lr, li [B*T, W]. */
int oracle_gate_proj(long BT, int W, int nblk, const double *x, const double *Wa,
                     const double *ba, const double *Wx, const double *bx, double *lr,
                     double *li) {
  if (BT < 1 || W < 1 || nblk < 1 || W % nblk) return 1;
  const int k = W / nblk;
#pragma omp parallel for schedule(static)
  for (long n = 0; n < BT; ++n) {
    const double *xr = x + n * W;
    for (int blk = 0; blk < nblk; ++blk) {
      double *outr = lr + n * W + (long)blk * k;
      double *outi = li + n * W + (long)blk * k;
      for (int j = 0; j < k; ++j) {
        outr[j] = ba ? ba[blk * k + j] : 0.0;
        outi[j] = bx ? bx[blk * k + j] : 0.0;
      }
      for (int i = 0; i < k; ++i) {
        const double xi = xr[blk * k + i];
        const double *wa = Wa + ((long)blk * k + i) * k;
        const double *wx = Wx + ((long)blk * k + i) * k;
        for (int j = 0; j < k; ++j) {
          outr[j] += xi * wa[j];
          outi[j] += xi * wx[j];
        }
      }
    }
  }
  return 0;
}

/* Backward of the projections.  dx [B*T, W] is ACCUMULATED into (dx += dlr Wa^T + dli Wx^T);
 * dWa, dWx [nblk, k, k] and dba, dbx [W] are written. */
int oracle_gate_proj_backward(long BT, int W, int nblk, const double *x, const double *Wa,
                              const double *Wx, const double *dlr, const double *dli,
                              double *dx, double *dWa, double *dba, double *dWx, double *dbx) {
  if (BT < 1 || W < 1 || nblk < 1 || W % nblk) return 1;
  const int k = W / nblk;
  /* dx: rows independent. */
#pragma omp parallel for schedule(static)
  for (long n = 0; n < BT; ++n) {
    for (int blk = 0; blk < nblk; ++blk) {
      const double *gr = dlr + n * W + (long)blk * k;
      const double *gi = dli + n * W + (long)blk * k;
      for (int i = 0; i < k; ++i) {
        const double *wa = Wa + ((long)blk * k + i) * k;
        const double *wx = Wx + ((long)blk * k + i) * k;
        double acc = 0.0;
        for (int j = 0; j < k; ++j) acc += gr[j] * wa[j] + gi[j] * wx[j];
        dx[n * W + (long)blk * k + i] += acc;
      }
    }
  }
  /* dW rows (blk, i) independent; each sums over tokens in order. */
  const long rows = (long)nblk * k;
#pragma omp parallel for schedule(static)
  for (long row = 0; row < rows; ++row) {
    const long blk = row / k, i = row % k;
    double *da = dWa + row * k;
    double *dxw = dWx + row * k;
    for (int j = 0; j < k; ++j) da[j] = dxw[j] = 0.0;
    for (long n = 0; n < BT; ++n) {
      const double xi = x[n * W + blk * k + i];
      const double *gr = dlr + n * W + blk * k;
      const double *gi = dli + n * W + blk * k;
      for (int j = 0; j < k; ++j) {
        da[j] += xi * gr[j];
        dxw[j] += xi * gi[j];
      }
    }
  }
  /* db: per channel, sum over tokens in order. */
#pragma omp parallel for schedule(static)
  for (long w = 0; w < W; ++w) {
    double sa = 0.0, sx = 0.0;
    for (long n = 0; n < BT; ++n) {
      sa += dlr[n * W + w];
      sx += dli[n * W + w];
    }
    dba[w] = sa;
    dbx[w] = sx;
  }
  return 0;
}
