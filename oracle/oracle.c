/*
 * oracle.c — plain, slow, single-threaded fp64 CPU oracle of SANTA++ decode-step attention.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the package smoke check and the benchmark's CPU
 * baseline load this file's library.  It shares no code, header, table or helper with the
 * CUDA path, and the CUDA path never calls it.
 *
 * It follows the method step by step, in the order and notation of the pages:
 *   [ABS] "SANTA++: Sampling Attention through Representative Keys" (arXiv 2609.35629),
 *         abstract: teams, one representative per team scored by the query, sampled teams,
 *         exact attention inside them, reweighting by the inverse inclusion probability.
 *   [EXP] "SANTA++：用代表性 Key 采样把 KV cache 读带宽砍掉 80%" (explainer), section 三
 *         "core method": 1 teams, 2 representative / score / softmax, 3 sample M teams,
 *         4 exact scores in sampled teams, 5 reweight, combine; 3.1 importance sampling.
 * Choices the pages leave open are fixed as follows (each is listed in the design notes):
 *   - teams are contiguous blocks of T tokens (one KV page); the last one may be partial;
 *   - the representative is the mean of the team's valid keys;
 *   - scores carry the 1/sqrt(d) of the in-team attention;
 *   - with grouped-query attention the team probability is the mean over the G query heads
 *     of their per-head softmax, and the sampled set is shared by the group;
 *   - the M draws are i.i.d. with replacement; draw r of unit (b, h) takes word 0 of
 *     Philox4x32-10 with key (lo32(seed), hi32(seed)) and counter (r, h, b, 0), maps it to
 *     u = (x + 0.5) / 2^32 and picks the smallest i with u*Z < C_i (strict), C the running
 *     sum of p in team order and Z = C_{n-1}; the pages fix no arithmetic for this
 *     decision, and it is taken exactly on 62-bit fixed-point probabilities (integer CDF,
 *     floor(u Z) by a 128-bit product), the same way the GPU kernel takes it;
 *   - S is the set of distinct drawn teams and the weight of team i is 1/pi_i with
 *     pi_i = 1 - (1 - p_i)^M, the probability that i is drawn at least once (Horvitz-
 *     Thompson), applied to numerator and denominator alike; the output is their ratio.
 *
 * Data: q [B][Hq][d], k_pool / v_pool [P][Hkv][T][d] in fp32 or bf16 (read exactly into
 * double), page_table [B][max_teams], seq_lens [B].  Every floating-point step is fp64.
 * Build: gcc -O2 -ffp-contract=off (no contraction, so results do not depend on the host);
 * the sampling decision uses unsigned __int128 (gcc, x86-64 and aarch64).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_MAX_TEAMS 16384 /* longest supported sequence, in teams */

typedef struct oracle_problem {
  const void* q;
  const void* k_pool;
  const void* v_pool;
  int dtype;
  const int32_t* page_table;
  const int32_t* seq_lens;
  int64_t num_pages;
  int batch, num_q_heads, num_kv_heads, head_dim, team_size, max_teams;
} oracle_problem;

/* ---------------------------------------------------------------- element access */

/* One stored element as an exact double (bf16 is the top half of an IEEE fp32). */
static double elem(const void* base, int dtype, int64_t idx) {
  float f;
  if (dtype == ORACLE_BF16) {
    uint32_t w = (uint32_t)((const uint16_t*)base)[idx] << 16;
    memcpy(&f, &w, sizeof f);
  } else {
    f = ((const float*)base)[idx];
  }
  return (double)f;
}

double oracle_elem(const void* base, int dtype, int64_t idx) { return elem(base, dtype, idx); }

static int64_t kv_index(const oracle_problem* pr, int64_t page, int h, int t, int k) {
  return ((page * pr->num_kv_heads + h) * (int64_t)pr->team_size + t) * pr->head_dim + k;
}

static double q_elem(const oracle_problem* pr, int b, int hq, int k) {
  return elem(pr->q, pr->dtype, ((int64_t)b * pr->num_q_heads + hq) * pr->head_dim + k);
}

/* Number of teams of sequence b, or -1 if its length is out of range. */
static int num_teams(const oracle_problem* pr, int b) {
  int L = pr->seq_lens[b];
  if (L < 1 || (int64_t)L > (int64_t)pr->max_teams * pr->team_size) return -1;
  return (L + pr->team_size - 1) / pr->team_size;
}

/* Valid tokens of team i of sequence b (the last team may be partial). */
static int team_len(const oracle_problem* pr, int b, int i) {
  int rest = pr->seq_lens[b] - i * pr->team_size;
  return rest < pr->team_size ? rest : pr->team_size;
}

static int64_t team_page(const oracle_problem* pr, int b, int i) {
  return pr->page_table[(int64_t)b * pr->max_teams + i];
}

/* ---------------------------------------------------------------- Philox4x32-10 */
/* Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11):
 * ten rounds of the 4x32 Philox S-box; each round multiplies counter words 0 and 2 by the
 * two round multipliers, and mixes the high halves with words 1, 3 and the round key; the
 * key is bumped by the two Weyl constants before every round after the first. */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    uint64_t p0 = (uint64_t)0xD2511F53u * x0;
    uint64_t p1 = (uint64_t)0xCD9E8D57u * x2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    x0 = hi1 ^ x1 ^ k0;
    x1 = lo1;
    x2 = hi0 ^ x3 ^ k1;
    x3 = lo0;
  }
  out[0] = x0;
  out[1] = x1;
  out[2] = x2;
  out[3] = x3;
}

/* The uniform of draw r of unit (b, h): word 0 of Philox4x32-10 at counter (r, h, b, 0)
 * under key (lo32(seed), hi32(seed)), as (x + 1/2) / 2^32, which is exact in fp64.  (The
 * draws use it exactly, through oracle_draw_point.) */
double oracle_uniform(uint64_t seed, int b, int h, int r) {
  uint32_t ctr[4] = {(uint32_t)r, (uint32_t)h, (uint32_t)b, 0u};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t w[4];
  oracle_philox4x32_10(ctr, key, w);
  return ((double)w[0] + 0.5) / 4294967296.0;
}

/* ---------------------------------------------------------------- step 1-2: representatives */

/* rep[p][h][:] = mean of the page's first fill[p] keys (fill NULL: every page full);
 * a page with no valid key gets the zero vector.  [ABS; EXP 三 step 2, the mean key]
 * Returns 0, or -1 if a fill is out of range. */
int oracle_build_reps(const oracle_problem* pr, const int32_t* page_fill, double* reps) {
  const int d = pr->head_dim, T = pr->team_size;
  for (int64_t p = 0; p < pr->num_pages; ++p) {
    int c = page_fill ? page_fill[p] : T;
    if (c < 0 || c > T) return -1;
    for (int h = 0; h < pr->num_kv_heads; ++h) {
      double* rep = reps + (p * pr->num_kv_heads + h) * d;
      for (int k = 0; k < d; ++k) {
        double sum = 0.0;
        for (int t = 0; t < c; ++t) sum += elem(pr->k_pool, pr->dtype, kv_index(pr, p, h, t, k));
        rep[k] = c > 0 ? sum / (double)c : 0.0;
      }
    }
  }
  return 0;
}

/* ---------------------------------------------------------------- step 2: team probabilities */

/* For unit (b, h): s_{g,i} = q_g . rep_i / sqrt(d) for the G query heads of the group,
 * p_{g,i} = exp(s_{g,i} - max_i s_{g,i}) / sum_i exp(...), p_i = (1/G) sum_g p_{g,i}.
 * scores [G][max_teams] (may be NULL) and p [max_teams] are written for i < n.
 * Returns n, or -1 for a bad seq_len, -2 for a bad page id.  [ABS; EXP 三 step 2] */
int oracle_team_probs(const oracle_problem* pr, const double* reps, int b, int h,
                      double* scores, double* p) {
  const int d = pr->head_dim;
  const int G = pr->num_q_heads / pr->num_kv_heads;
  const int n = num_teams(pr, b);
  if (n < 0) return -1;
  if (n > ORACLE_MAX_TEAMS) return -5;
  for (int i = 0; i < n; ++i) {
    int64_t page = team_page(pr, b, i);
    if (page < 0 || page >= pr->num_pages) return -2;
    p[i] = 0.0;
  }
  const double inv_sqrt_d = 1.0 / sqrt((double)d);
  double* s = (double*)malloc(sizeof(double) * (size_t)n);
  if (!s) return -6;
  for (int g = 0; g < G; ++g) {
    const int hq = h * G + g;
    for (int i = 0; i < n; ++i) {
      const double* rep = reps + (team_page(pr, b, i) * pr->num_kv_heads + h) * d;
      double dot = 0.0;
      for (int k = 0; k < d; ++k) dot += q_elem(pr, b, hq, k) * rep[k];
      s[i] = dot * inv_sqrt_d;
      if (scores) scores[(int64_t)g * pr->max_teams + i] = s[i];
    }
    double m = s[0];
    for (int i = 1; i < n; ++i)
      if (s[i] > m) m = s[i];
    double z = 0.0;
    for (int i = 0; i < n; ++i) z += exp(s[i] - m);
    for (int i = 0; i < n; ++i) p[i] += exp(s[i] - m) / z;
  }
  for (int i = 0; i < n; ++i) p[i] /= (double)G;
  free(s);
  return n;
}

/* ---------------------------------------------------------------- step 3: sampling */

/* Team probability as a 62-bit fixed-point integer: round(p * 2^62), ties away from zero.
 * The CDF is the exact integer running sum of these, so its value does not depend on the
 * order of the additions. */
uint64_t oracle_fixed_prob(double p) {
  return (uint64_t)llround(ldexp(p, 62));
}

/* Inverse-CDF search: the smallest i with t < C[i]; if there is none (t >= C[n-1]), the
 * smallest i with C[i] == C[n-1], i.e. the team that completes the distribution. */
int oracle_cdf_search(const uint64_t* C, int n, uint64_t t) {
  for (int i = 0; i < n; ++i)
    if (t < C[i]) return i;
  for (int i = 0; i < n; ++i)
    if (C[i] == C[n - 1]) return i;
  return n - 1;
}

/* Position of draw r on the integer CDF: t = floor(u * Z) with u = (2x + 1) / 2^33, x the
 * draw's Philox word, computed exactly with a 128-bit product.  t < Z always. */
uint64_t oracle_draw_point(uint64_t seed, int b, int h, int r, uint64_t Z) {
  uint32_t ctr[4] = {(uint32_t)r, (uint32_t)h, (uint32_t)b, 0u};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t w[4];
  oracle_philox4x32_10(ctr, key, w);
  unsigned __int128 prod = (unsigned __int128)(2ull * w[0] + 1ull) * Z;
  return (uint64_t)(prod >> 33);
}

/* M i.i.d. draws from p[0..n) for unit (b, h), 1 <= n <= ORACLE_MAX_TEAMS.
 * [ABS; EXP 三 step 3]  The draw takes u = (x + 1/2) / 2^32 and picks the smallest i with
 * u * Z < C_i, evaluated exactly on the fixed-point CDF (C_i = sum_{k<=i} round(p_k 2^62),
 * Z = C_{n-1}).
 * draws [M] receive team indices; t_out [M] (may be NULL) receives floor(u * Z); cdf [n]
 * (may be NULL) receives C. */
void oracle_draw(const double* p, int n, int M, uint64_t seed, int b, int h, int32_t* draws,
                 uint64_t* t_out, uint64_t* cdf) {
  if (n < 1 || n > ORACLE_MAX_TEAMS) return;
  uint64_t* C = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)n);
  if (!C) return;
  uint64_t run = 0;
  for (int i = 0; i < n; ++i) {
    run += oracle_fixed_prob(p[i]);
    C[i] = run;
  }
  const uint64_t Z = C[n - 1];
  for (int r = 0; r < M; ++r) {
    const uint64_t t = oracle_draw_point(seed, b, h, r, Z);
    draws[r] = oracle_cdf_search(C, n, t);
    if (t_out) t_out[r] = t;
  }
  if (cdf)
    for (int i = 0; i < n; ++i) cdf[i] = C[i];
  free(C);
}

/* S = distinct drawn teams in ascending order, with pi_i = 1 - (1 - p_i)^M evaluated as
 * -expm1(M log1p(-p_i)).  Returns |S|.  [ABS, abstract: the weights 1/pi_i] */
int oracle_select(const int32_t* draws, int M, const double* p, int n, int32_t* sel,
                  double* pi) {
  int count = 0;
  for (int i = 0; i < n; ++i) {
    int hit = 0;
    for (int r = 0; r < M; ++r)
      if (draws[r] == i) hit = 1;
    if (hit) {
      sel[count] = i;
      pi[count] = -expm1((double)M * log1p(-p[i]));
      ++count;
    }
  }
  return count;
}

/* ---------------------------------------------------------------- sampler variants */

/*
 * Beyond the method above, three samplers and a defensive mixture (the build's "next" rows;
 * same arithmetic conventions as the default sampler):
 *   0  i.i.d. draws, Horvitz-Thompson weight 1/pi_i with pi_i = 1 - (1 - q_i)^M (the method);
 *   1  systematic draws, the stratified / systematic variants of [SANTA] ("Stochastic Sparse
 *      Attention for Memory-Bound Inference", abstract) applied to team draws: one uniform
 *      u (the Philox word of draw 0), the M points (r + u) / M, r = 0..M-1, on the CDF of q.
 *      Team i's interval has length q_i and the points are 1/M apart, so it holds at least
 *      one point with probability pi_i = min(1, M q_i); the weight is 1/pi_i;
 *   2  i.i.d. draws with the Hansen-Hurwitz weight c_i / (M q_i), c_i the number of draws
 *      of team i: the per-draw 1/p_i reweighting of [EXP] section 三 step 5.
 * The defensive mixture of [EXP] section 八 (pitfall 4: mix a uniform share into the team
 * distribution so that no weight explodes) samples from q_i = (1 - alpha) p_i + alpha / n;
 * alpha = 0 is the plain method.
 * Every sampler returns, per selected team, recip = 1 / weight, which the attention step
 * uses exactly as it uses pi.
 */
#define ORACLE_SAMPLER_IID_HT 0
#define ORACLE_SAMPLER_SYSTEMATIC 1
#define ORACLE_SAMPLER_IID_HH 2

/* q_i = (1 - alpha) p_i + alpha / n for i < n. */
void oracle_mix(const double* p, int n, double alpha, double* q) {
  for (int i = 0; i < n; ++i) q[i] = (1.0 - alpha) * p[i] + alpha / (double)n;
}

/* Systematic point r on the integer CDF: floor((r Z + t_u) / M) with t_u = floor(u Z) the
 * draw-0 point.  Because r Z is an integer, this equals floor((r + u) Z / M) exactly, so
 * t_r < C_i holds exactly when (r + u) / M * Z < C_i.  t_r < Z. */
uint64_t oracle_systematic_point(uint64_t t_u, int r, int M, uint64_t Z) {
  const unsigned __int128 num = (unsigned __int128)(uint64_t)r * Z + t_u;
  return (uint64_t)(num / (unsigned __int128)(uint64_t)M);
}

/* M systematic draws from q[0..n) for unit (b, h); outputs as oracle_draw. */
void oracle_draw_systematic(const double* q, int n, int M, uint64_t seed, int b, int h,
                            int32_t* draws, uint64_t* t_out, uint64_t* cdf) {
  if (n < 1 || n > ORACLE_MAX_TEAMS) return;
  uint64_t* C = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)n);
  if (!C) return;
  uint64_t run = 0;
  for (int i = 0; i < n; ++i) {
    run += oracle_fixed_prob(q[i]);
    C[i] = run;
  }
  const uint64_t Z = C[n - 1];
  const uint64_t t_u = oracle_draw_point(seed, b, h, 0, Z);
  for (int r = 0; r < M; ++r) {
    const uint64_t t = oracle_systematic_point(t_u, r, M, Z);
    draws[r] = oracle_cdf_search(C, n, t);
    if (t_out) t_out[r] = t;
  }
  if (cdf)
    for (int i = 0; i < n; ++i) cdf[i] = C[i];
  free(C);
}

/* S = distinct drawn teams in ascending order, with recip = 1 / weight of each:
 * sampler 0: 1 - (1 - q_i)^M; sampler 1: min(1, M q_i); sampler 2: M q_i / c_i.
 * Returns |S|, or -1 for an unknown sampler. */
int oracle_select_ex(const int32_t* draws, int M, const double* q, int n, int sampler,
                     int32_t* sel, double* recip) {
  if (sampler < ORACLE_SAMPLER_IID_HT || sampler > ORACLE_SAMPLER_IID_HH) return -1;
  int count = 0;
  for (int i = 0; i < n; ++i) {
    int c = 0;
    for (int r = 0; r < M; ++r)
      if (draws[r] == i) ++c;
    if (!c) continue;
    sel[count] = i;
    if (sampler == ORACLE_SAMPLER_IID_HT)
      recip[count] = -expm1((double)M * log1p(-q[i]));
    else if (sampler == ORACLE_SAMPLER_SYSTEMATIC)
      recip[count] = fmin(1.0, (double)M * q[i]);
    else
      recip[count] = (double)M * q[i] / (double)c;
    ++count;
  }
  return count;
}

/* ---------------------------------------------------------------- steps 4-5: attention */

/* Raw score of token t of team i for query head hq: q . k / sqrt(d). */
static double token_score(const oracle_problem* pr, int b, int hq, int h, int64_t page, int t) {
  double dot = 0.0;
  for (int k = 0; k < pr->head_dim; ++k)
    dot += q_elem(pr, b, hq, k) * elem(pr->k_pool, pr->dtype, kv_index(pr, page, h, t, k));
  return dot / sqrt((double)pr->head_dim);
}

static int check_sel(const oracle_problem* pr, int b, const int32_t* sel, int count) {
  const int n = num_teams(pr, b);
  if (n < 0) return -1;
  for (int c = 0; c < count; ++c) {
    if (sel[c] < 0 || sel[c] >= n) return -3;
    int64_t page = team_page(pr, b, sel[c]);
    if (page < 0 || page >= pr->num_pages) return -2;
  }
  return 0;
}

/* Horvitz-Thompson numerator and denominator with a caller-fixed shift m_g:
 *   num_g = sum_{c} (1/pi_c) sum_{j in team sel[c]} exp(s_j - m_g) v_j   [G][d]
 *   den_g = sum_{c} (1/pi_c) sum_{j in team sel[c]} exp(s_j - m_g)       [G]
 * [ABS; EXP 三 steps 4-5, 3.1].  Returns 0 or a negative error. */
int oracle_num_den(const oracle_problem* pr, int b, int h, const int32_t* sel, const double* pi,
                   int count, const double* shift, double* num, double* den) {
  int err = check_sel(pr, b, sel, count);
  if (err) return err;
  const int d = pr->head_dim;
  const int G = pr->num_q_heads / pr->num_kv_heads;
  for (int g = 0; g < G; ++g) {
    const int hq = h * G + g;
    den[g] = 0.0;
    for (int k = 0; k < d; ++k) num[g * d + k] = 0.0;
    for (int c = 0; c < count; ++c) {
      const int64_t page = team_page(pr, b, sel[c]);
      const int len = team_len(pr, b, sel[c]);
      const double w = 1.0 / pi[c];
      for (int t = 0; t < len; ++t) {
        const double e = exp(token_score(pr, b, hq, h, page, t) - shift[g]);
        den[g] += w * e;
        for (int k = 0; k < d; ++k)
          num[g * d + k] += w * e * elem(pr->v_pool, pr->dtype, kv_index(pr, page, h, t, k));
      }
    }
  }
  return 0;
}

/* The estimate out_g = num_g / den_g, with m_g the largest score among the sampled tokens
 * (it cancels in the ratio and only keeps exp() in range).  out [G][d]. */
int oracle_attend(const oracle_problem* pr, int b, int h, const int32_t* sel, const double* pi,
                  int count, double* out) {
  int err = check_sel(pr, b, sel, count);
  if (err) return err;
  if (count < 1) return -3;
  const int d = pr->head_dim;
  const int G = pr->num_q_heads / pr->num_kv_heads;
  double shift[8] = {0}, den[8] = {0};
  double num[8 * 128] = {0};
  if (G > 8 || d > 128) return -4;
  for (int g = 0; g < G; ++g) {
    double m = -INFINITY;
    for (int c = 0; c < count; ++c) {
      const int64_t page = team_page(pr, b, sel[c]);
      const int len = team_len(pr, b, sel[c]);
      for (int t = 0; t < len; ++t) {
        double s = token_score(pr, b, h * G + g, h, page, t);
        if (s > m) m = s;
      }
    }
    shift[g] = m;
  }
  err = oracle_num_den(pr, b, h, sel, pi, count, shift, num, den);
  if (err) return err;
  for (int g = 0; g < G; ++g)
    for (int k = 0; k < d; ++k) out[g * d + k] = num[g * d + k] / den[g];
  return 0;
}

/* ---------------------------------------------------------------- value-row sampling */

/*
 * Value-row sampling inside the selected teams ([SANTA] "Stochastic Sparse Attention for
 * Memory-Bound Inference", abstract: draw value rows from the post-softmax distribution and
 * gather-add them in place of the full P.V product).  With grouped-query attention one set
 * of rows per team serves the G query heads: rows are drawn from the group-mean in-team
 * distribution r_j = (1/G) sum_g exp(s_gj - m_gi) / Z_gi (m_gi, Z_gi the team's max and sum
 * of exp for head g), and head g weighs a drawn row j by exp(s_gj - m_gi) / r_j.  That is an
 * importance-sampling estimate of sum_j exp(s_gj - m_gi) v_j, unbiased given the team; the
 * denominators Z_gi stay exact.  Row draw k of team i of unit (b, h) takes word 0 of
 * Philox4x32-10 with counter (k, h, b, 1 + i) (team draws use word 3 = 0) and is decided
 * exactly on the 62-bit fixed-point CDF of r, like the team draws.
 */

/* r_j for the valid tokens of team `team` of unit (b, h): r [len].  Returns len or < 0. */
int oracle_vs_row_probs(const oracle_problem* pr, int b, int h, int team, double* r) {
  const int n = num_teams(pr, b);
  if (n < 0) return -1;
  if (team < 0 || team >= n) return -3;
  const int64_t page = team_page(pr, b, team);
  if (page < 0 || page >= pr->num_pages) return -2;
  const int len = team_len(pr, b, team);
  const int G = pr->num_q_heads / pr->num_kv_heads;
  for (int t = 0; t < len; ++t) r[t] = 0.0;
  for (int g = 0; g < G; ++g) {
    double m = -INFINITY, z = 0.0;
    for (int t = 0; t < len; ++t) {
      const double sc = token_score(pr, b, h * G + g, h, page, t);
      if (sc > m) m = sc;
    }
    for (int t = 0; t < len; ++t) z += exp(token_score(pr, b, h * G + g, h, page, t) - m);
    for (int t = 0; t < len; ++t)
      r[t] += exp(token_score(pr, b, h * G + g, h, page, t) - m) / z / (double)G;
  }
  return len;
}

/* Position of row draw k of team `team` on an integer CDF of total Z (as oracle_draw_point,
 * counter (k, h, b, 1 + team)). */
uint64_t oracle_vs_point(uint64_t seed, int b, int h, int team, int k, uint64_t Z) {
  uint32_t ctr[4] = {(uint32_t)k, (uint32_t)h, (uint32_t)b, (uint32_t)(1 + team)};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t w[4];
  oracle_philox4x32_10(ctr, key, w);
  unsigned __int128 prod = (unsigned __int128)(2ull * w[0] + 1ull) * Z;
  return (uint64_t)(prod >> 33);
}

/* S row draws of team `team`: idx [S] token indices; t [S] and C [len] may be NULL.
 * Returns len or < 0. */
int oracle_vs_draw(const oracle_problem* pr, int b, int h, int team, int S, uint64_t seed,
                   int32_t* idx, uint64_t* t_out, uint64_t* cdf) {
  double r[1024];
  if (pr->team_size > 1024) return -4;
  const int len = oracle_vs_row_probs(pr, b, h, team, r);
  if (len <= 0) return len < 0 ? len : -3;
  uint64_t C[1024];
  uint64_t run = 0;
  for (int j = 0; j < len; ++j) {
    run += oracle_fixed_prob(r[j]);
    C[j] = run;
  }
  for (int k = 0; k < S; ++k) {
    const uint64_t t = oracle_vs_point(seed, b, h, team, k, C[len - 1]);
    idx[k] = oracle_cdf_search(C, len, t);
    if (t_out) t_out[k] = t;
  }
  if (cdf)
    for (int j = 0; j < len; ++j) cdf[j] = C[j];
  return len;
}

/* Numerator and denominator with value-row sampling, given the row draws idx [count][S] and
 * a caller-fixed shift m_g:
 *   num_g = sum_c (1/pi_c) (1/S) sum_k exp(s_g,idx - m_g) / r_idx * v_idx   [G][d]
 *   den_g = sum_c (1/pi_c) sum_{j in team} exp(s_gj - m_g)                  [G] (exact)
 * Returns 0 or < 0. */
int oracle_num_den_vs(const oracle_problem* pr, int b, int h, const int32_t* sel,
                      const double* pi, int count, int S, const int32_t* idx,
                      const double* shift, double* num, double* den) {
  int err = check_sel(pr, b, sel, count);
  if (err) return err;
  const int d = pr->head_dim;
  const int G = pr->num_q_heads / pr->num_kv_heads;
  double r[1024];
  if (pr->team_size > 1024) return -4;
  for (int g = 0; g < G; ++g) {
    den[g] = 0.0;
    for (int k = 0; k < d; ++k) num[g * d + k] = 0.0;
  }
  for (int c = 0; c < count; ++c) {
    const int64_t page = team_page(pr, b, sel[c]);
    const int len = oracle_vs_row_probs(pr, b, h, sel[c], r);
    if (len < 0) return len;
    const double w = 1.0 / pi[c];
    for (int g = 0; g < G; ++g) {
      const int hq = h * G + g;
      for (int t = 0; t < len; ++t) den[g] += w * exp(token_score(pr, b, hq, h, page, t) - shift[g]);
      for (int k = 0; k < S; ++k) {
        const int j = idx[c * S + k];
        if (j < 0 || j >= len) return -5;
        const double a = w * exp(token_score(pr, b, hq, h, page, j) - shift[g]) / r[j] / S;
        for (int e = 0; e < d; ++e)
          num[g * d + e] += a * elem(pr->v_pool, pr->dtype, kv_index(pr, page, h, j, e));
      }
    }
  }
  return 0;
}

/* The value-sampled estimate out_g = num_g / den_g (shift: the largest score among the
 * sampled teams' tokens, as oracle_attend); idx [count][S] receives the row draws (may be
 * NULL).  out [G][d].  Returns 0 or < 0. */
int oracle_attend_vs(const oracle_problem* pr, int b, int h, const int32_t* sel,
                     const double* pi, int count, int S, uint64_t seed, int32_t* idx_out,
                     double* out) {
  int err = check_sel(pr, b, sel, count);
  if (err) return err;
  if (count < 1 || S < 1) return -3;
  const int d = pr->head_dim;
  const int G = pr->num_q_heads / pr->num_kv_heads;
  if (G > 8 || d > 128) return -4;
  int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)count * (size_t)S);
  if (!idx) return -6;
  double shift[8], den[8], num[8 * 128];
  for (int g = 0; g < G; ++g) {
    double m = -INFINITY;
    for (int c = 0; c < count; ++c) {
      const int64_t page = team_page(pr, b, sel[c]);
      const int len = team_len(pr, b, sel[c]);
      for (int t = 0; t < len; ++t) {
        const double s = token_score(pr, b, h * G + g, h, page, t);
        if (s > m) m = s;
      }
    }
    shift[g] = m;
  }
  for (int c = 0; c < count && !err; ++c) {
    const int len = oracle_vs_draw(pr, b, h, sel[c], S, seed, idx + (size_t)c * S, 0, 0);
    if (len < 0) err = len;
  }
  if (!err) err = oracle_num_den_vs(pr, b, h, sel, pi, count, S, idx, shift, num, den);
  if (!err) {
    for (int g = 0; g < G; ++g)
      for (int k = 0; k < d; ++k) out[g * d + k] = num[g * d + k] / den[g];
    if (idx_out)
      for (size_t i = 0; i < (size_t)count * S; ++i) idx_out[i] = idx[i];
  }
  free(idx);
  return err;
}

/* Dense softmax attention over every valid token of sequence b, for the G query heads of
 * KV head h: the quantity the estimator targets.  out [G][d]. */
int oracle_dense(const oracle_problem* pr, int b, int h, double* out) {
  const int n = num_teams(pr, b);
  if (n < 0) return -1;
  const int d = pr->head_dim;
  const int G = pr->num_q_heads / pr->num_kv_heads;
  for (int i = 0; i < n; ++i) {
    int64_t page = team_page(pr, b, i);
    if (page < 0 || page >= pr->num_pages) return -2;
  }
  for (int g = 0; g < G; ++g) {
    const int hq = h * G + g;
    double m = -INFINITY;
    for (int i = 0; i < n; ++i)
      for (int t = 0; t < team_len(pr, b, i); ++t) {
        double s = token_score(pr, b, hq, h, team_page(pr, b, i), t);
        if (s > m) m = s;
      }
    double den = 0.0;
    for (int k = 0; k < d; ++k) out[g * d + k] = 0.0;
    for (int i = 0; i < n; ++i) {
      const int64_t page = team_page(pr, b, i);
      for (int t = 0; t < team_len(pr, b, i); ++t) {
        const double e = exp(token_score(pr, b, hq, h, page, t) - m);
        den += e;
        for (int k = 0; k < d; ++k)
          out[g * d + k] += e * elem(pr->v_pool, pr->dtype, kv_index(pr, page, h, t, k));
      }
    }
    for (int k = 0; k < d; ++k) out[g * d + k] /= den;
  }
  return 0;
}

/* ---------------------------------------------------------------- whole step for one unit */

/* Steps 2-5 in order for unit (b, h): team probabilities, M draws, the distinct set with
 * its inclusion probabilities, and the estimate.  draws [M], sel [M], pi [M], p
 * [max_teams], out [G][d].  Returns |S| or a negative error. */
int oracle_decode(const oracle_problem* pr, const double* reps, int M, uint64_t seed, int b,
                  int h, int32_t* draws, int32_t* sel, double* pi, double* p, double* out) {
  int n = oracle_team_probs(pr, reps, b, h, 0, p);
  if (n < 0) return n;
  oracle_draw(p, n, M, seed, b, h, draws, 0, 0);
  int count = oracle_select(draws, M, p, n, sel, pi);
  int err = oracle_attend(pr, b, h, sel, pi, count, out);
  return err ? err : count;
}

/* oracle_decode with a sampler (0, 1, 2 as above) and a defensive mixture alpha in [0, 1]:
 * q [max_teams] receives the sampling distribution, recip [M] the 1 / weight of each
 * selected team.  Returns |S| or a negative error. */
int oracle_decode_ex(const oracle_problem* pr, const double* reps, int M, uint64_t seed, int b,
                     int h, int sampler, double alpha, int32_t* draws, int32_t* sel,
                     double* recip, double* q, double* out) {
  if (!(alpha >= 0.0 && alpha <= 1.0)) return -1;
  int n = oracle_team_probs(pr, reps, b, h, 0, q);
  if (n < 0) return n;
  oracle_mix(q, n, alpha, q);
  if (sampler == ORACLE_SAMPLER_SYSTEMATIC)
    oracle_draw_systematic(q, n, M, seed, b, h, draws, 0, 0);
  else
    oracle_draw(q, n, M, seed, b, h, draws, 0, 0);
  int count = oracle_select_ex(draws, M, q, n, sampler, sel, recip);
  if (count < 0) return count;
  int err = oracle_attend(pr, b, h, sel, recip, count, out);
  return err ? err : count;
}
