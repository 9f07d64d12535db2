/*
 * Plain CPU oracle of one gated Mixture-of-Experts FFN layer, forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the timed
 * CPU baseline of the benchmark use this file.  It shares no code, header or
 * table with the CUDA library and never calls it.
 *
 * What it computes (per token t; no blocking, fusion or reordering):
 *   1. gate logits   l[t,e] = sum_i x[t,i] * Wg[i,e]           (fp32, see below)
 *   2. softmax       p[t,e] = exp(l[t,e] - max) / sum exp(.)    (double)
 *      top-k         k experts by logit, ties to the lower index
 *      gate weights  top-1: w = p[e1];  top-2: w_j = p_j / (p_1 + p_2)
 *   3. capacity      C = ceil(cf * T / E)   (cf = +infinity: C = T, dropless)
 *      dispatch      assignments (t, j) in token-major order; the rank of an
 *                    assignment is the number of earlier ones to the same
 *                    expert; kept iff rank < C; slots are compact:
 *                    slot = exscan(kept)[e] + rank
 *   4. expert FFN    FFN_e(x) = GeLU_tanh(x W1[e]) W2[e]          (double)
 *   5. combine       out[t] = sum_j [kept] w_j FFN_{e_j}(x_t)
 *                    (+ GeLU_tanh(x_t Wr1) Wr2 for the residual variant)
 *
 * Sources.  Each token goes to experts through a gating function, and the
 * activated parameters per token equal those of the dense model (DeepSpeed-MoE
 * review, "MoE based NLG Model Architecture").  Top-2 sends a token to two
 * experts and sums their outputs; Residual-MoE sums a fixed MLP and one routed
 * expert (same review, "Phenomenon2").  The 'standard' / 'residual' MLP type
 * switch is the one of the DeepSpeed-MoE Inference wiki ("PR-MoE 최적화로 더
 * 낮은 비용").  The pages give no formula for the gate, the capacity, the drop
 * rule or the activation; the readings taken here are: no bias terms; fp32
 * logits from the fp32 fused-multiply-add chain in ascending i starting from
 * +0; selection on logits with ties to the lower index; capacity
 * ceil(cf*T/E) per expert independent of k, with cf*T and /E evaluated in
 * double; dispatch in token-major order; compact slots; dropped assignments
 * contribute zero and top-2 weights are not renormalised after a drop; GeLU is
 * the tanh form 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
 *
 * Precision.  The logits are the canonical fp32 chain acc = fmaf(x_i, Wg_ie,
 * acc) (this file is compiled with -ffp-contract=off), so routing is a plain
 * function of the fp32 inputs.  Everything after the logits is double; the
 * hidden activations stay double.
 *
 * Parity pins (tests): exact-rational replay of the fp32 chain; a stable-sort
 * brute force of the dispatch; dense all-experts brute force of the layer;
 * closed forms (Wg = 0, constant token, x = 0); the E = 1 reduction to a plain
 * MLP; GeLU identities and values.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_F32 0
#define OR_F16 1

/* malloc that stops the process when the host is out of memory (a checker that went on
 * with a null buffer would report garbage as a reference). */
static void* xmalloc(size_t bytes) {
  void* p = malloc(bytes ? bytes : 1);
  if (!p) {
    fprintf(stderr, "oracle: out of host memory (%zu bytes)\n", bytes);
    abort();
  }
  return p;
}

/* IEEE binary16 bit pattern -> double, from the format's definition. */
double oracle_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int ex = (h >> 10) & 31;
  int man = h & 1023;
  double v;
  if (ex == 0) v = ldexp((double)man, -24);
  else if (ex == 31) v = man ? NAN : INFINITY;
  else v = ldexp((double)(man + 1024), ex - 25);
  return sign ? -v : v;
}

static double elem(const void* p, int dtype, size_t i) {
  if (dtype == OR_F16) return oracle_half_to_double(((const uint16_t*)p)[i]);
  return (double)((const float*)p)[i];
}

/* Step 1: fp32 gate logits, the fused-multiply-add chain in ascending i. */
void oracle_gate_logits(const void* x, int x_dtype, const float* Wg, int T, int d, int E,
                        float* logits) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      float acc = 0.0f;
      for (int i = 0; i < d; ++i) {
        float xi = (float)elem(x, x_dtype, (size_t)t * d + i); /* exact: f16 -> f32 */
        acc = fmaf(xi, Wg[(size_t)i * E + e], acc);
      }
      logits[(size_t)t * E + e] = acc;
    }
  }
}

/* Step 2: softmax over E (double) and top-k selection on the logits. */
void oracle_softmax_topk(const float* logits, int T, int E, int k, double* probs /* nullable */,
                         int32_t* topk_idx, double* topk_w) {
  double* p = (double*)xmalloc(sizeof(double) * (size_t)E);
  for (int t = 0; t < T; ++t) {
    const float* l = logits + (size_t)t * E;
    int e1 = 0;
    for (int e = 1; e < E; ++e)
      if (l[e] > l[e1]) e1 = e;                 /* strict: equal logits keep the lower index */
    int e2 = -1;
    if (k == 2) {
      for (int e = 0; e < E; ++e) {
        if (e == e1) continue;
        if (e2 < 0 || l[e] > l[e2]) e2 = e;
      }
    }
    double m = (double)l[e1];
    double s = 0.0;
    for (int e = 0; e < E; ++e) {
      p[e] = exp((double)l[e] - m);
      s += p[e];
    }
    for (int e = 0; e < E; ++e) p[e] /= s;
    if (probs) memcpy(probs + (size_t)t * E, p, sizeof(double) * (size_t)E);
    topk_idx[(size_t)t * k] = e1;
    if (k == 1) {
      topk_w[t] = p[e1];
    } else {
      topk_idx[(size_t)t * 2 + 1] = e2;
      double z = p[e1] + p[e2];
      topk_w[(size_t)t * 2] = p[e1] / z;
      topk_w[(size_t)t * 2 + 1] = p[e2] / z;
    }
  }
  free(p);
}

/*
 * Step 3a: capacity C = ceil(cf * T / E); -1 on bad arguments.  cf = +infinity
 * is the dropless mode: C = T, which no expert can exceed (a token's k experts
 * are distinct), so nothing is dropped.
 */
int oracle_capacity(int T, int E, double cf) {
  if (T < 1 || E < 1 || !(cf > 0.0)) return -1;
  if (isinf(cf)) return T;
  double c = ceil(cf * (double)T / (double)E);
  if (c > 2147483647.0) return -1;
  return (int)c;
}

/*
 * Step 3b: capacity-limited dispatch, token-major.  Outputs counts_raw[E],
 * kept[E], offsets[E+1], perm[S] (S = offsets[E]) and slot_of[T*k] (-1 = dropped).
 * Returns S.
 */
int oracle_dispatch(const int32_t* topk_idx, int T, int E, int k, int C, int32_t* counts_raw,
                    int32_t* kept, int32_t* offsets, int32_t* perm, int32_t* slot_of) {
  int32_t* rank = (int32_t*)xmalloc(sizeof(int32_t) * (size_t)T * k);
  for (int e = 0; e < E; ++e) counts_raw[e] = 0;
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      int e = topk_idx[(size_t)t * k + j];
      rank[(size_t)t * k + j] = counts_raw[e]++;
    }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) {
    kept[e] = counts_raw[e] < C ? counts_raw[e] : C;
    offsets[e + 1] = offsets[e] + kept[e];
  }
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      size_t a = (size_t)t * k + j;
      int e = topk_idx[a];
      if (rank[a] < C) {
        int s = offsets[e] + rank[a];
        slot_of[a] = s;
        perm[s] = t;
      } else {
        slot_of[a] = -1;
      }
    }
  free(rank);
  return offsets[E];
}

/*
 * Step 3b for one shard of a batch that is split over ranks in token order
 * (shard r holds a contiguous run of tokens, after those of shards 0 .. r-1).
 * base[e] = assignments to expert e in the earlier shards.  The assignment's
 * rank in the whole batch is base[e] + its rank within the shard, and the
 * capacity rule of step 3b applies to that rank, with C the whole batch's
 * capacity.  Outputs are those of oracle_dispatch for the shard's own tokens:
 * counts_raw / kept of this shard, compact slots over its kept assignments,
 * perm holding shard-local token indices.  Experts outside [0, E) are not
 * counted and their assignments are dropped.  Returns the shard's S.
 */
int oracle_dispatch_shard(const int32_t* topk_idx, int T, int E, int k, int C,
                          const int32_t* base, int32_t* counts_raw, int32_t* kept,
                          int32_t* offsets, int32_t* perm, int32_t* slot_of) {
  int32_t* rank = (int32_t*)xmalloc(sizeof(int32_t) * ((size_t)T * k + 1));
  for (int e = 0; e < E; ++e) counts_raw[e] = 0;
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      size_t a = (size_t)t * k + j;
      int e = topk_idx[a];
      rank[a] = (e >= 0 && e < E) ? counts_raw[e]++ : -1;
    }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) {
    long long left = (long long)C - base[e];            /* capacity left for this shard */
    if (left < 0) left = 0;
    kept[e] = counts_raw[e] < left ? counts_raw[e] : (int32_t)left;
    offsets[e + 1] = offsets[e] + kept[e];
  }
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      size_t a = (size_t)t * k + j;
      int e = topk_idx[a];
      if (rank[a] >= 0 && (long long)base[e] + rank[a] < C) {
        int s = offsets[e] + rank[a];
        slot_of[a] = s;
        perm[s] = t;
      } else {
        slot_of[a] = -1;
      }
    }
  free(rank);
  return offsets[E];
}

double oracle_gelu(double x) {
  const double c = sqrt(2.0 / M_PI);
  return 0.5 * x * (1.0 + tanh(c * (x + 0.044715 * x * x * x)));
}

/*
 * Step 4: one MLP on one token in double: y = GeLU(x W_in) W_out with
 * W_in [d, f] and W_out [f, d] row-major.  h is caller scratch of length f.
 */
static void mlp_token(const void* x, int x_dtype, size_t x_off, const void* W_in,
                      const void* W_out, int w_dtype, int d, int f, double* h, double* y) {
  for (int j = 0; j < f; ++j) h[j] = 0.0;
  for (int i = 0; i < d; ++i) {
    double xi = elem(x, x_dtype, x_off + i);
    for (int j = 0; j < f; ++j) h[j] += xi * elem(W_in, w_dtype, (size_t)i * f + j);
  }
  for (int j = 0; j < f; ++j) h[j] = oracle_gelu(h[j]);
  for (int m = 0; m < d; ++m) y[m] = 0.0;
  for (int j = 0; j < f; ++j) {
    double hj = h[j];
    for (int m = 0; m < d; ++m) y[m] += hj * elem(W_out, w_dtype, (size_t)j * d + m);
  }
}

void oracle_expert_ffn(const void* x_row, int x_dtype, const void* W1e, const void* W2e,
                       int w_dtype, int d, int f, double* y) {
  double* h = (double*)xmalloc(sizeof(double) * (size_t)f);
  mlp_token(x_row, x_dtype, 0, W1e, W2e, w_dtype, d, f, h, y);
  free(h);
}

/*
 * Step 5 for a list of rows: out[r] = sum_j [slot_of >= 0] w_j FFN_{e_j}(x_t)
 * (+ residual MLP), t = rows[r].  W1[e] / W2[e] point at expert e's [d,f] and
 * [f,d] matrices (entries of experts no listed token uses may be NULL).
 * Wr1/Wr2 are NULL for the standard variant.  Returns 0, or -1 if a needed
 * expert pointer is NULL.
 */
int oracle_combine_rows(const void* x, int x_dtype, int T, int d, int f, int k,
                        const int32_t* topk_idx, const double* topk_w, const int32_t* slot_of,
                        const void* const* W1, const void* const* W2, int w_dtype,
                        const void* Wr1, const void* Wr2, int f_res, const int32_t* rows,
                        int n_rows, double* out) {
  int bad = 0;
  int fmax = f > f_res ? f : f_res;
#pragma omp parallel
  {
    double* h = (double*)xmalloc(sizeof(double) * (size_t)(fmax > 0 ? fmax : 1));
    double* y = (double*)xmalloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
    for (int r = 0; r < n_rows; ++r) {
      int t = rows ? rows[r] : r;
      double* o = out + (size_t)r * d;
      for (int m = 0; m < d; ++m) o[m] = 0.0;
      if (t < 0 || t >= T) continue;
      for (int j = 0; j < k; ++j) {
        size_t a = (size_t)t * k + j;
        if (slot_of[a] < 0) continue;           /* dropped: contributes zero */
        int e = topk_idx[a];
        if (!W1[e] || !W2[e]) {
#pragma omp atomic write
          bad = 1;
          continue;
        }
        mlp_token(x, x_dtype, (size_t)t * d, W1[e], W2[e], w_dtype, d, f, h, y);
        for (int m = 0; m < d; ++m) o[m] += topk_w[a] * y[m];
      }
      if (Wr1 && Wr2 && f_res > 0) {
        mlp_token(x, x_dtype, (size_t)t * d, Wr1, Wr2, w_dtype, d, f_res, h, y);
        for (int m = 0; m < d; ++m) o[m] += y[m];
      }
    }
    free(h);
    free(y);
  }
  return bad ? -1 : 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Thread count of later calls (timing of the oracle on one core and on all cores). */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
