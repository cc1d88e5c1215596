/*
 * Gated DeltaNet slot-pool oracle: a plain, slow, double-precision CPU
 * restatement of the per-layer GDN step over a slot-indexed state pool.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or constant with the
 * CUDA library; the two meet only through seeded inputs generated elsewhere.
 *
 * Sources it follows (page title, section):
 *  - "TokenSpeed alcanza 580 tps con Qwen3.5-397B-A17B en GPU"
 *      §"Ciclo de vida de slots": working slot (mutable, updated in place every
 *        decode step) and checkpoint slot (snapshot target);
 *      §"Riesgo de correctitud: estado obsoleto": a reused slot is made safe
 *        only by copy-on-write from a clean checkpoint or by explicit zeroing;
 *      §"Scheduler dual": per-request mamba_pool_indices, state filled during
 *        prefill and updated in place during decode, spec_cache of per-step
 *        conv/SSM snapshots for speculative rollback.
 *  - "构建面向 Agentic 推理的下一代 LLM 推理引擎" (TokenSpeed talk)
 *      §"为什么 Agentic 推理需要新推理引擎": linear-attention state is an SSM
 *        state plus a convolution state.
 *  - The per-token recurrence is not written on the pages.  It follows the
 *    published Gated DeltaNet formulation (Yang, Kautz, Hatamizadeh, "Gated
 *    Delta Networks", ICLR 2025):  S_t = a_t (I - b_t k_t k_t^T) S_{t-1}
 *    + b_t k_t v_t^T,  o_t = S_t^T q_t, with the gate g = -exp(A_log) *
 *    softplus(a + dt_bias), a_t = exp(g), b_t = sigmoid(b), a width-W causal
 *    conv1d + SiLU over the q|k|v channels and an L2 normalisation of q and
 *    k (q additionally scaled by dk^-1/2).  The chunkwise form used only as a
 *    cross-check follows the WY/UT representation of Yang et al.,
 *    "Parallelizing Linear Transformers with the Delta Rule over Sequence
 *    Length", NeurIPS 2024.
 *
 * Conventions (the readings taken where the pages are silent):
 *  - state per V head is stored transposed, St[dv][dk] (row j = column j of
 *    S), so o = St q and the update of row j uses only (k, v_j, q);
 *  - channels are q | k | v, head-major; V head h reads QK head h / (HV/HK);
 *  - conv state holds the last W-1 raw (pre-conv) inputs, oldest first; the
 *    weight index W-1 multiplies the newest input; no bias;
 *  - q_hat = q / sqrt(|q|^2 + 1e-6) / sqrt(dk), k_hat = k / sqrt(|k|^2 + 1e-6);
 *  - slot id -1 is padding: the row is skipped and its outputs are zero; any
 *    other id outside [0, num_slots) is skipped the same way and sets bit 1
 *    of the error word.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_ERR_SLOT_OOB 1u

typedef struct {
  int32_t hk, hv, dk, dv, w;
} orc_dims;

typedef struct {
  double* ssm;  /* [num_slots][hv][dv][dk] */
  double* conv; /* [num_slots][w-1][C]     */
  int32_t num_slots;
} orc_pool;

typedef struct {
  const double* conv_w;  /* [C][w] */
  const double* A_log;   /* [hv]   */
  const double* dt_bias; /* [hv]   */
} orc_params;

static const double ORC_EPS = 1e-6;

static int64_t n_chan(const orc_dims* d) {
  return 2 * (int64_t)d->hk * d->dk + (int64_t)d->hv * d->dv;
}
static int64_t ssm_elems(const orc_dims* d) {
  return (int64_t)d->hv * d->dv * d->dk;
}
static int64_t conv_elems(const orc_dims* d) {
  return (int64_t)(d->w - 1) * n_chan(d);
}

/* 0 = usable slot, 1 = padding (-1), 2 = out of range */
static int slot_class(int32_t id, int32_t num_slots) {
  if (id == -1) return 1;
  if (id < 0 || id >= num_slots) return 2;
  return 0;
}

/* ---- the per-token pieces ------------------------------------------------ */

double orc_silu(double y) { return y / (1.0 + exp(-y)); }
double orc_softplus(double x) { return log1p(exp(x)); }
double orc_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* g = -exp(A_log) * softplus(a + dt_bias) */
double orc_gate_g(double A_log, double dt_bias, double a) {
  return -exp(A_log) * orc_softplus(a + dt_bias);
}

/* out = x / sqrt(sum x^2 + eps) * scale */
void orc_l2norm(int32_t n, const double* x, double scale, double* out) {
  double ss = 0.0;
  for (int32_t i = 0; i < n; ++i) ss += x[i] * x[i];
  double r = 1.0 / sqrt(ss + ORC_EPS);
  for (int32_t i = 0; i < n; ++i) out[i] = x[i] * r * scale;
}

/* Causal conv1d over the window [hist[0..w-2], x] for every channel, then
 * SiLU.  hist is [w-1][C], oldest row first. */
void orc_conv_silu(const orc_dims* d, const double* hist, const double* x,
                   const double* conv_w, double* y) {
  int64_t C = n_chan(d);
  int W = d->w;
  for (int64_t c = 0; c < C; ++c) {
    double acc = 0.0;
    for (int i = 0; i < W - 1; ++i) acc += conv_w[c * W + i] * hist[i * C + c];
    acc += conv_w[c * W + (W - 1)] * x[c];
    y[c] = orc_silu(acc);
  }
}

/* Shift the conv history by one token: drop the oldest, append x. */
static void conv_shift(const orc_dims* d, double* hist, const double* x) {
  int64_t C = n_chan(d);
  for (int i = 0; i + 1 < d->w - 1; ++i)
    memcpy(hist + i * C, hist + (i + 1) * C, sizeof(double) * C);
  if (d->w > 1) memcpy(hist + (int64_t)(d->w - 2) * C, x, sizeof(double) * C);
}

/* Gated delta rule on one head, state stored transposed St[dv][dk]:
 *   u = v - alpha * St k
 *   St <- alpha * St + beta * u k^T
 *   o = St q          (read out from the updated state)
 * Equivalent to S <- alpha (I - beta k k^T) S + beta k v^T, o = S^T q. */
void orc_delta_core(int32_t dk, int32_t dv, double* St, const double* k,
                    const double* v, const double* q, double alpha,
                    double beta, double* o) {
  for (int32_t j = 0; j < dv; ++j) {
    double* row = St + (int64_t)j * dk;
    double sk = 0.0;
    for (int32_t i = 0; i < dk; ++i) sk += row[i] * k[i];
    double u = v[j] - alpha * sk;
    for (int32_t i = 0; i < dk; ++i) row[i] = alpha * row[i] + beta * u * k[i];
    double oj = 0.0;
    for (int32_t i = 0; i < dk; ++i) oj += row[i] * q[i];
    o[j] = oj;
  }
}

/* Features of one token for every head: q_hat, k_hat per QK head, v per V
 * head, and (alpha, beta) per V head.  y is [C] (conv + SiLU output). */
typedef struct {
  double* qh;    /* [hk][dk] */
  double* kh;    /* [hk][dk] */
  double* v;     /* [hv][dv] (points into y) */
  double* g;     /* [hv] */
  double* alpha; /* [hv] */
  double* beta;  /* [hv] */
} orc_feat;

static void token_features(const orc_dims* d, const orc_params* p,
                           const double* y, const double* a_t,
                           const double* b_t, orc_feat* f) {
  double qscale = 1.0 / sqrt((double)d->dk);
  for (int h = 0; h < d->hk; ++h) {
    orc_l2norm(d->dk, y + (int64_t)h * d->dk, qscale, f->qh + (int64_t)h * d->dk);
    orc_l2norm(d->dk, y + (int64_t)(d->hk + h) * d->dk, 1.0,
               f->kh + (int64_t)h * d->dk);
  }
  for (int h = 0; h < d->hv; ++h) {
    f->g[h] = orc_gate_g(p->A_log[h], p->dt_bias[h], a_t[h]);
    f->alpha[h] = exp(f->g[h]);
    f->beta[h] = orc_sigmoid(b_t[h]);
  }
}

/* One token on one slot (conv state and SSM state updated in place).
 * Heads outside [h_lo, h_hi) keep their state and leave o untouched; the
 * conv history always advances for every channel. */
static void token_step(const orc_dims* d, const orc_params* p, double* ssm,
                       double* conv, const double* x, const double* a_t,
                       const double* b_t, double* o, int h_lo, int h_hi,
                       double* work) {
  int64_t C = n_chan(d);
  double* y = work;
  double* qh = y + C;
  double* kh = qh + (int64_t)d->hk * d->dk;
  double* g = kh + (int64_t)d->hk * d->dk;
  double* al = g + d->hv;
  double* be = al + d->hv;
  orc_conv_silu(d, conv, x, p->conv_w, y);
  conv_shift(d, conv, x);
  orc_feat f = {qh, kh, y + 2 * (int64_t)d->hk * d->dk, g, al, be};
  token_features(d, p, y, a_t, b_t, &f);
  int G = d->hv / d->hk;
  for (int h = h_lo; h < h_hi; ++h) {
    int hq = h / G;
    orc_delta_core(d->dk, d->dv, ssm + (int64_t)h * d->dv * d->dk,
                   kh + (int64_t)hq * d->dk, f.v + (int64_t)h * d->dv,
                   qh + (int64_t)hq * d->dk, al[h], be[h],
                   o + (int64_t)h * d->dv);
  }
}

static int64_t work_elems(const orc_dims* d) {
  return n_chan(d) + 2 * (int64_t)d->hk * d->dk + 3 * (int64_t)d->hv;
}

static int check_dims(const orc_dims* d) {
  if (!d || d->hk <= 0 || d->hv <= 0 || d->dk <= 0 || d->dv <= 0 || d->w < 1)
    return 1;
  if (d->hv % d->hk) return 1;
  return 0;
}

static void clamp_heads(const orc_dims* d, int* h_lo, int* h_hi) {
  if (*h_lo < 0) *h_lo = 0;
  if (*h_hi > d->hv || *h_hi < 0) *h_hi = d->hv;
}

/* ---- a0..a6: one decode step over a batch ------------------------------- */
/* qkv [B][C], a,b [B][hv], out [B][hv][dv].  Heads outside [h_lo,h_hi) are
 * not advanced (sampling); pass h_lo=0, h_hi=-1 for all heads. */
int orc_decode_step(const orc_dims* d, orc_pool pool, const orc_params* p,
                    const int32_t* slot_ids, int32_t B, const double* qkv,
                    const double* a, const double* b, double* out,
                    uint32_t* err, int32_t h_lo, int32_t h_hi) {
  if (check_dims(d)) return 1;
  clamp_heads(d, &h_lo, &h_hi);
  int64_t C = n_chan(d), HVDV = (int64_t)d->hv * d->dv;
  int64_t fail = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : fail)
  for (int32_t r = 0; r < B; ++r) {
    int32_t s = slot_ids[r];
    int cls = slot_class(s, pool.num_slots);
    double* o = out + r * HVDV;
    if (cls) {
      if (cls == 2) fail |= ORC_ERR_SLOT_OOB;
      for (int64_t i = 0; i < HVDV; ++i) o[i] = 0.0;
      continue;
    }
    double* work = (double*)malloc(sizeof(double) * work_elems(d));
    token_step(d, p, pool.ssm + s * ssm_elems(d), pool.conv + s * conv_elems(d),
               qkv + r * C, a + (int64_t)r * d->hv, b + (int64_t)r * d->hv, o,
               h_lo, h_hi, work);
    free(work);
  }
  if (err) *err |= (uint32_t)fail;
  return 0;
}

/* ---- a9 / a10: slot copy and zero ---------------------------------------- */
int orc_slot_copy(const orc_dims* d, orc_pool src, orc_pool dst,
                  const int32_t* src_ids, const int32_t* dst_ids, int32_t n,
                  uint32_t* err) {
  if (check_dims(d)) return 1;
  int64_t ns = ssm_elems(d), nc = conv_elems(d);
  for (int32_t i = 0; i < n; ++i) {
    int cs = slot_class(src_ids[i], src.num_slots);
    int cd = slot_class(dst_ids[i], dst.num_slots);
    if (cs == 2 || cd == 2) {
      if (err) *err |= ORC_ERR_SLOT_OOB;
      continue;
    }
    if (cs || cd) continue;
    memmove(dst.ssm + dst_ids[i] * ns, src.ssm + src_ids[i] * ns, sizeof(double) * ns);
    memmove(dst.conv + dst_ids[i] * nc, src.conv + src_ids[i] * nc, sizeof(double) * nc);
  }
  return 0;
}

int orc_slot_zero(const orc_dims* d, orc_pool pool, const int32_t* ids,
                  int32_t n, uint32_t* err) {
  if (check_dims(d)) return 1;
  int64_t ns = ssm_elems(d), nc = conv_elems(d);
  for (int32_t i = 0; i < n; ++i) {
    int c = slot_class(ids[i], pool.num_slots);
    if (c == 2 && err) *err |= ORC_ERR_SLOT_OOB;
    if (c) continue;
    for (int64_t e = 0; e < ns; ++e) pool.ssm[ids[i] * ns + e] = 0.0;
    for (int64_t e = 0; e < nc; ++e) pool.conv[ids[i] * nc + e] = 0.0;
  }
  return 0;
}

/* ---- a7: speculative verify ---------------------------------------------
 * For request r, run T draft tokens from its working slot without touching
 * the working slot; after token t the state (SSM and conv history) is written
 * into spec slot spec_ids[r][t] (-1: not written).  qkv [B][T][C], a,b
 * [B][T][hv], out [B][T][hv][dv]. */
int orc_spec_verify(const orc_dims* d, orc_pool work, orc_pool spec,
                    const orc_params* p, const int32_t* slot_ids,
                    const int32_t* spec_ids, int32_t B, int32_t T,
                    const double* qkv, const double* a, const double* b,
                    double* out, uint32_t* err) {
  if (check_dims(d)) return 1;
  int64_t C = n_chan(d), HVDV = (int64_t)d->hv * d->dv;
  int64_t ns = ssm_elems(d), nc = conv_elems(d);
  int64_t fail = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : fail)
  for (int32_t r = 0; r < B; ++r) {
    int32_t s = slot_ids[r];
    int cls = slot_class(s, work.num_slots);
    if (cls) {
      if (cls == 2) fail |= ORC_ERR_SLOT_OOB;
      for (int64_t i = 0; i < (int64_t)T * HVDV; ++i) out[(int64_t)r * T * HVDV + i] = 0.0;
      continue;
    }
    double* st = (double*)malloc(sizeof(double) * (ns + nc + work_elems(d)));
    double* cv = st + ns;
    double* wk = cv + nc;
    memcpy(st, work.ssm + s * ns, sizeof(double) * ns);
    memcpy(cv, work.conv + s * nc, sizeof(double) * nc);
    for (int32_t t = 0; t < T; ++t) {
      int64_t rt = (int64_t)r * T + t;
      token_step(d, p, st, cv, qkv + rt * C, a + rt * d->hv, b + rt * d->hv,
                 out + rt * HVDV, 0, d->hv, wk);
      int32_t sid = spec_ids[rt];
      int sc = slot_class(sid, spec.num_slots);
      if (sc == 2) fail |= ORC_ERR_SLOT_OOB;
      if (sc) continue;
      memcpy(spec.ssm + sid * ns, st, sizeof(double) * ns);
      memcpy(spec.conv + sid * nc, cv, sizeof(double) * nc);
    }
    free(st);
  }
  if (err) *err |= (uint32_t)fail;
  return 0;
}

/* ---- a7': commit the accepted snapshot ----------------------------------
 * accept_len[r] = L in 0..T.  L >= 1 copies spec slot spec_ids[r][L-1] into
 * the working slot slot_ids[r]; L = 0 keeps the working slot (it already is
 * the rollback state).  L outside 0..T is out of range (error bit, skip). */
int orc_spec_commit(const orc_dims* d, orc_pool spec, orc_pool work,
                    const int32_t* spec_ids, const int32_t* accept_len,
                    const int32_t* slot_ids, int32_t B, int32_t T,
                    uint32_t* err) {
  if (check_dims(d)) return 1;
  for (int32_t r = 0; r < B; ++r) {
    int32_t L = accept_len[r];
    if (L < 0 || L > T) {
      if (err) *err |= ORC_ERR_SLOT_OOB;
      continue;
    }
    if (L == 0) continue;
    int32_t src = spec_ids[(int64_t)r * T + (L - 1)];
    int32_t dst = slot_ids[r];
    orc_slot_copy(d, spec, work, &src, &dst, 1, err);
  }
  return 0;
}

/* ---- index-update commit ------------------------------------------------
 * TokenSpeed talk, "Kernel: 让 MLA 真正跑满 GPU": the accepted draft's state is
 * adopted by updating the request's index rather than by moving data; the
 * Qwen3.5 page, "Scheduler dual": rollback keeps the pre-draft working slot.
 * The snapshots live in the working pool.  For request r, L = accept_len[r]:
 *   L = 0: the working slot stays; freed[r][t] = spec_ids[r][t] for all t.
 *   1 <= L <= T and spec_ids[r][L-1] >= 0: slot_ids[r] becomes
 *     spec_ids[r][L-1]; freed[r][0] = the old working slot and
 *     freed[r][1..T) = the other snapshots in draft order.
 *   anything else: error bit, slot_ids[r] unchanged, freed[r][*] = -1. */
int orc_commit_index(const int32_t* spec_ids, const int32_t* accept_len, int32_t* slot_ids,
                     int32_t* freed, int32_t B, int32_t T, uint32_t* err) {
  if (B < 0 || T < 1) return 1;
  for (int32_t r = 0; r < B; ++r) {
    const int32_t* sp = spec_ids + (int64_t)r * T;
    int32_t* fr = freed + (int64_t)r * T;
    int32_t L = accept_len[r];
    if (L == 0) {
      for (int32_t t = 0; t < T; ++t) fr[t] = sp[t];
      continue;
    }
    if (L < 0 || L > T || sp[L - 1] < 0) {
      if (err) *err |= ORC_ERR_SLOT_OOB;
      for (int32_t t = 0; t < T; ++t) fr[t] = -1;
      continue;
    }
    int32_t k = 0;
    fr[k++] = slot_ids[r];
    for (int32_t t = 0; t < T; ++t)
      if (t != L - 1) fr[k++] = sp[t];
    slot_ids[r] = sp[L - 1];
  }
  return 0;
}

/* ---- state pack / unpack ---------------------------------------------------
 * TokenSpeed Qwen3.5 page, "Disaggregacion Prefill-Decode": slot ids become
 * offsets and the states move as contiguous blocks.  Record i of the staging
 * area holds slot ids[i]: its SSM [hv][dv][dk] (st_ssm + i * ssm elements)
 * and its conv history [W-1][C] (st_conv + i * conv elements).
 * Pack: id -1 gives a zero record; an id outside the pool a zero record and
 * the error bit.  Unpack: record i -> slot ids[i]; -1 is skipped; an id
 * outside the pool is skipped with the error bit. */
int orc_state_pack(const orc_dims* d, orc_pool pool, const int32_t* ids, int32_t n,
                   double* st_ssm, double* st_conv, uint32_t* err) {
  if (check_dims(d)) return 1;
  int64_t ns = ssm_elems(d), nc = conv_elems(d);
  for (int32_t i = 0; i < n; ++i) {
    int c = slot_class(ids[i], pool.num_slots);
    if (c == 2 && err) *err |= ORC_ERR_SLOT_OOB;
    for (int64_t e = 0; e < ns; ++e) st_ssm[i * ns + e] = c ? 0.0 : pool.ssm[ids[i] * ns + e];
    for (int64_t e = 0; e < nc; ++e) st_conv[i * nc + e] = c ? 0.0 : pool.conv[ids[i] * nc + e];
  }
  return 0;
}

int orc_state_unpack(const orc_dims* d, const double* st_ssm, const double* st_conv, orc_pool pool,
                     const int32_t* ids, int32_t n, uint32_t* err) {
  if (check_dims(d)) return 1;
  int64_t ns = ssm_elems(d), nc = conv_elems(d);
  for (int32_t i = 0; i < n; ++i) {
    int c = slot_class(ids[i], pool.num_slots);
    if (c == 2 && err) *err |= ORC_ERR_SLOT_OOB;
    if (c) continue;
    for (int64_t e = 0; e < ns; ++e) pool.ssm[ids[i] * ns + e] = st_ssm[i * ns + e];
    for (int64_t e = 0; e < nc; ++e) pool.conv[ids[i] * nc + e] = st_conv[i * nc + e];
  }
  return 0;
}

/* ---- KDA: the delta rule with a per-key-channel decay --------------------
 * The pages name Kimi Delta Attention (Kimi K3) as the second linear-
 * attention family beside GDN and do not write it.  It follows the published
 * formulation (Kimi Linear, 2025): the scalar decay of the gated delta rule
 * becomes a decay per key channel,
 *   S_t = (I - b_t k_t k_t^T) Diag(a_t) S_{t-1} + b_t k_t v_t^T,  o_t = S_t^T q_t,
 * a_t[c] = exp(g_c), g_c = -exp(A_log[h]) * softplus(a[h][c] + dt_bias[h][c]).
 * In the transposed storage St[dv][dk] (row j = column j of S):
 *   u_j = v_j - sum_i a_i St[j][i] k_i
 *   St[j][i] <- a_i St[j][i] + b u_j k_i
 *   o_j = sum_i St[j][i] q_i   (updated state) */
void orc_kda_core(int32_t dk, int32_t dv, double* St, const double* k, const double* v,
                  const double* q, const double* alpha, double beta, double* o) {
  for (int32_t j = 0; j < dv; ++j) {
    double* row = St + (int64_t)j * dk;
    double sk = 0.0;
    for (int32_t i = 0; i < dk; ++i) sk += alpha[i] * row[i] * k[i];
    double u = v[j] - sk;
    for (int32_t i = 0; i < dk; ++i) row[i] = alpha[i] * row[i] + beta * u * k[i];
    double oj = 0.0;
    for (int32_t i = 0; i < dk; ++i) oj += row[i] * q[i];
    o[j] = oj;
  }
}

/* One KDA token on one slot (conv history and SSM state updated in place):
 * a_t [hv][dk] gate logits, b_t [hv], o [hv][dv].  work: C + 3 dk doubles. */
static void kda_token_step(const orc_dims* d, const orc_params* p, double* ssm, double* conv,
                           const double* x, const double* a_t, const double* b_t, double* o,
                           double* work) {
  int64_t C = n_chan(d);
  int dk = d->dk, G = d->hv / d->hk;
  double *y = work, *qh = y + C, *kh = qh + dk, *al = kh + dk;
  orc_conv_silu(d, conv, x, p->conv_w, y);
  conv_shift(d, conv, x);
  for (int h = 0; h < d->hv; ++h) {
    int hq = h / G;
    orc_l2norm(dk, y + (int64_t)hq * dk, 1.0 / sqrt((double)dk), qh);
    orc_l2norm(dk, y + (int64_t)(d->hk + hq) * dk, 1.0, kh);
    for (int c = 0; c < dk; ++c)
      al[c] = exp(orc_gate_g(p->A_log[h], p->dt_bias[(int64_t)h * dk + c], a_t[(int64_t)h * dk + c]));
    orc_kda_core(dk, d->dv, ssm + (int64_t)h * d->dv * dk, kh,
                 y + 2 * (int64_t)d->hk * dk + (int64_t)h * d->dv, qh, al, orc_sigmoid(b_t[h]),
                 o + (int64_t)h * d->dv);
  }
}

/* KDA decode: as orc_decode_step (same pool, conv, norms, beta), with the
 * gate logits a [B][hv][dk] and dt_bias [hv][dk] per key channel. */
int orc_kda_decode_step(const orc_dims* d, orc_pool pool, const orc_params* p,
                        const int32_t* slot_ids, int32_t B, const double* qkv,
                        const double* a, const double* b, double* out, uint32_t* err) {
  if (check_dims(d)) return 1;
  int64_t C = n_chan(d), HVDV = (int64_t)d->hv * d->dv;
  int64_t fail = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : fail)
  for (int32_t r = 0; r < B; ++r) {
    int32_t s = slot_ids[r];
    int cls = slot_class(s, pool.num_slots);
    double* o = out + r * HVDV;
    if (cls) {
      if (cls == 2) fail |= ORC_ERR_SLOT_OOB;
      for (int64_t i = 0; i < HVDV; ++i) o[i] = 0.0;
      continue;
    }
    double* work = (double*)malloc(sizeof(double) * (C + 3 * (int64_t)d->dk));
    kda_token_step(d, p, pool.ssm + s * ssm_elems(d), pool.conv + s * conv_elems(d), qkv + r * C,
                   a + (int64_t)r * d->hv * d->dk, b + (int64_t)r * d->hv, o, work);
    free(work);
  }
  if (err) *err |= (uint32_t)fail;
  return 0;
}

/* KDA speculative verify: as orc_spec_verify, each draft a KDA token step;
 * a [B][T][hv][dk]. */
int orc_kda_spec_verify(const orc_dims* d, orc_pool work, orc_pool spec, const orc_params* p,
                        const int32_t* slot_ids, const int32_t* spec_ids, int32_t B, int32_t T,
                        const double* qkv, const double* a, const double* b, double* out,
                        uint32_t* err) {
  if (check_dims(d)) return 1;
  int64_t C = n_chan(d), HVDV = (int64_t)d->hv * d->dv;
  int64_t ns = ssm_elems(d), nc = conv_elems(d);
  int64_t fail = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : fail)
  for (int32_t r = 0; r < B; ++r) {
    int32_t s = slot_ids[r];
    int cls = slot_class(s, work.num_slots);
    if (cls) {
      if (cls == 2) fail |= ORC_ERR_SLOT_OOB;
      for (int64_t i = 0; i < (int64_t)T * HVDV; ++i) out[(int64_t)r * T * HVDV + i] = 0.0;
      continue;
    }
    double* st = (double*)malloc(sizeof(double) * (ns + nc + C + 3 * (int64_t)d->dk));
    double* cv = st + ns;
    double* wk = cv + nc;
    memcpy(st, work.ssm + s * ns, sizeof(double) * ns);
    memcpy(cv, work.conv + s * nc, sizeof(double) * nc);
    for (int32_t t = 0; t < T; ++t) {
      int64_t rt = (int64_t)r * T + t;
      kda_token_step(d, p, st, cv, qkv + rt * C, a + rt * d->hv * d->dk, b + rt * d->hv,
                     out + rt * HVDV, wk);
      int32_t sid = spec_ids[rt];
      int sc = slot_class(sid, spec.num_slots);
      if (sc == 2) fail |= ORC_ERR_SLOT_OOB;
      if (sc) continue;
      memcpy(spec.ssm + sid * ns, st, sizeof(double) * ns);
      memcpy(spec.conv + sid * nc, cv, sizeof(double) * nc);
    }
    free(st);
  }
  if (err) *err |= (uint32_t)fail;
  return 0;
}

/* KDA prefill, token by token: the contract of orc_prefill (packed sequences,
 * absolute start positions, block-aligned checkpoints of state and conv
 * history) with every token a KDA token step; a [Ttot][hv][dk]. */
int orc_kda_prefill(const orc_dims* d, orc_pool pool, orc_pool ckpt, const orc_params* p,
                    const int32_t* slot_ids, const int32_t* cu_seqlens, const int64_t* start_pos,
                    int32_t n_seq, const int32_t* ckpt_ids, int32_t max_ckpt, int32_t ckpt_block,
                    const double* qkv, const double* a, const double* b, double* out, uint32_t* err) {
  if (check_dims(d) || ckpt_block <= 0) return 1;
  int64_t C = n_chan(d), HVDV = (int64_t)d->hv * d->dv;
  int64_t ns = ssm_elems(d), nc = conv_elems(d);
  int64_t fail = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : fail)
  for (int32_t n = 0; n < n_seq; ++n) {
    int32_t s = slot_ids[n];
    int64_t t0 = cu_seqlens[n], t1 = cu_seqlens[n + 1];
    int cls = slot_class(s, pool.num_slots);
    if (cls) {
      if (cls == 2) fail |= ORC_ERR_SLOT_OOB;
      for (int64_t i = t0 * HVDV; i < t1 * HVDV; ++i) out[i] = 0.0;
      continue;
    }
    double* ssm = pool.ssm + s * ns;
    double* conv = pool.conv + s * nc;
    double* wk = (double*)malloc(sizeof(double) * (C + 3 * (int64_t)d->dk));
    int64_t p0 = start_pos[n];
    int64_t blk0 = p0 / ckpt_block;
    for (int64_t i = t0; i < t1; ++i) {
      kda_token_step(d, p, ssm, conv, qkv + i * C, a + i * d->hv * d->dk, b + i * d->hv, out + i * HVDV,
                     wk);
      int64_t P = p0 + (i - t0) + 1;
      if (P % ckpt_block) continue;
      int64_t idx = P / ckpt_block - blk0 - 1;
      if (idx < 0 || idx >= max_ckpt) continue;
      int32_t cid = ckpt_ids[(int64_t)n * max_ckpt + idx];
      int cc = slot_class(cid, ckpt.num_slots);
      if (cc == 2) fail |= ORC_ERR_SLOT_OOB;
      if (cc) continue;
      memcpy(ckpt.ssm + cid * ns, ssm, sizeof(double) * ns);
      memcpy(ckpt.conv + cid * nc, conv, sizeof(double) * nc);
    }
    free(wk);
  }
  if (err) *err |= (uint32_t)fail;
  return 0;
}

/* ---- KDA prefill cross-check: the window (chunk) form (double) -----------
 * Same contract as orc_kda_prefill, the state recurrence evaluated one window
 * of `chunk` tokens at a time, windows aligned to absolute positions.  With the
 * per-channel cumulative log decay lb_r[c] = sum_{m<=r} g_m[c] inside the window
 * (r = 0 .. n-1) and, for every state row j (St[j][.]):
 *   A'[r][m] = sum_c k_r[c] k_m[c] e^{lb_r[c] - lb_m[c]}   (r > m)
 *   M[r][m]  = sum_c q_r[c] k_m[c] e^{lb_r[c] - lb_m[c]}   (r >= m)
 *   (I + diag(beta) A') T = diag(beta)
 *   X[r]     = v_r[j] - sum_c St[j][c] k_r[c] e^{lb_r[c]}
 *   Delta[r] = sum_m T[r][m] X[m]
 *   o_r[j]   = sum_c St[j][c] q_r[c] e^{lb_r[c]} + sum_{m<=r} M[r][m] Delta[m]
 *   St'[j][c] = St[j][c] e^{lb_{n-1}[c]} + sum_r Delta[r] k_r[c] e^{lb_{n-1}[c] - lb_r[c]}
 * ckpt_block must be a multiple of chunk. */
int orc_kda_prefill_chunked(const orc_dims* d, orc_pool pool, orc_pool ckpt, const orc_params* p,
                            const int32_t* slot_ids, const int32_t* cu_seqlens, const int64_t* start_pos,
                            int32_t n_seq, const int32_t* ckpt_ids, int32_t max_ckpt, int32_t ckpt_block,
                            int32_t chunk, const double* qkv, const double* a, const double* b, double* out,
                            uint32_t* err) {
  if (check_dims(d) || ckpt_block <= 0 || chunk <= 0 || ckpt_block % chunk) return 1;
  int64_t C = n_chan(d), HVDV = (int64_t)d->hv * d->dv;
  int64_t ns = ssm_elems(d), nc = conv_elems(d);
  int dk = d->dk, dv = d->dv, G = d->hv / d->hk;
  int64_t fail = 0;
  for (int32_t n = 0; n < n_seq; ++n) {
    int32_t s = slot_ids[n];
    int64_t t0 = cu_seqlens[n], t1 = cu_seqlens[n + 1], L = t1 - t0;
    int cls = slot_class(s, pool.num_slots);
    if (cls) {
      if (cls == 2) fail |= ORC_ERR_SLOT_OOB;
      for (int64_t i = t0 * HVDV; i < t1 * HVDV; ++i) out[i] = 0.0;
      continue;
    }
    int64_t p0 = start_pos[n], blk0 = p0 / ckpt_block;
    /* per-token features and the conv history after every token */
    double* fq = (double*)malloc(sizeof(double) * (L + 1) * d->hk * dk);
    double* fk = (double*)malloc(sizeof(double) * (L + 1) * d->hk * dk);
    double* fv = (double*)malloc(sizeof(double) * (L + 1) * d->hv * dv);
    double* fg = (double*)malloc(sizeof(double) * (L + 1) * d->hv * dk);
    double* fb = (double*)malloc(sizeof(double) * (L + 1) * d->hv);
    double* hist_after = (double*)malloc(sizeof(double) * (L + 1) * nc);
    double* conv = pool.conv + s * nc;
    double* y = (double*)malloc(sizeof(double) * C);
    for (int64_t i = 0; i < L; ++i) {
      const double* x = qkv + (t0 + i) * C;
      orc_conv_silu(d, conv, x, p->conv_w, y);
      conv_shift(d, conv, x);
      memcpy(hist_after + i * nc, conv, sizeof(double) * nc);
      for (int hq = 0; hq < d->hk; ++hq) {
        orc_l2norm(dk, y + (int64_t)hq * dk, 1.0 / sqrt((double)dk), fq + (i * d->hk + hq) * dk);
        orc_l2norm(dk, y + (int64_t)(d->hk + hq) * dk, 1.0, fk + (i * d->hk + hq) * dk);
      }
      memcpy(fv + i * d->hv * dv, y + 2 * (int64_t)d->hk * dk, sizeof(double) * d->hv * dv);
      for (int h = 0; h < d->hv; ++h) {
        fb[i * d->hv + h] = orc_sigmoid(b[(t0 + i) * d->hv + h]);
        for (int c = 0; c < dk; ++c)
          fg[(i * d->hv + h) * dk + c] =
              orc_gate_g(p->A_log[h], p->dt_bias[(int64_t)h * dk + c], a[((t0 + i) * d->hv + h) * dk + c]);
      }
    }
    int64_t mc = chunk;
    double* lb = (double*)malloc(sizeof(double) * mc * dk);
    double* Ap = (double*)malloc(sizeof(double) * mc * mc);
    double* Mm = (double*)malloc(sizeof(double) * mc * mc);
    double* Tm = (double*)malloc(sizeof(double) * mc * mc);
    double* X = (double*)malloc(sizeof(double) * mc);
    double* D = (double*)malloc(sizeof(double) * mc);
    double* rowbuf = (double*)malloc(sizeof(double) * dk);
    /* checkpoint rows are written per head as the windows end; the conv history
       of a checkpoint comes from hist_after */
    for (int h = 0; h < d->hv; ++h) {
      int hq = h / G;
      double* St = pool.ssm + s * ns + (int64_t)h * dv * dk;
      int64_t i = 0;
      while (i < L) {
        int64_t pos = p0 + i;
        int64_t wend = (pos / chunk + 1) * chunk;
        int64_t nr = wend - pos;
        if (nr > L - i) nr = L - i;
#define KQ(r) (fk + ((i + (r)) * d->hk + hq) * dk)
#define QQ(r) (fq + ((i + (r)) * d->hk + hq) * dk)
#define GG(r) (fg + ((i + (r)) * d->hv + h) * dk)
        for (int c = 0; c < dk; ++c) {
          double acc = 0.0;
          for (int64_t r = 0; r < nr; ++r) {
            acc += GG(r)[c];
            lb[r * dk + c] = acc;
          }
        }
        for (int64_t r = 0; r < nr; ++r)
          for (int64_t m = 0; m < nr; ++m) {
            double va = 0.0, vm = 0.0;
            if (m <= r)
              for (int c = 0; c < dk; ++c) {
                double f = KQ(m)[c] * exp(lb[r * dk + c] - lb[m * dk + c]);
                va += KQ(r)[c] * f;
                vm += QQ(r)[c] * f;
              }
            Ap[r * nr + m] = m < r ? va : 0.0;
            Mm[r * nr + m] = vm;
          }
        /* (I + diag(beta) A') T = diag(beta), row by row */
        for (int64_t r = 0; r < nr; ++r) {
          double br = fb[(i + r) * d->hv + h];
          for (int64_t c = 0; c < nr; ++c) {
            double v = (r == c) ? br : 0.0;
            for (int64_t m = 0; m < r; ++m) v -= br * Ap[r * nr + m] * Tm[m * nr + c];
            Tm[r * nr + c] = v;
          }
        }
        for (int j = 0; j < dv; ++j) {
          double* row = St + (int64_t)j * dk;
          for (int64_t r = 0; r < nr; ++r) {
            double sk = 0.0;
            for (int c = 0; c < dk; ++c) sk += row[c] * KQ(r)[c] * exp(lb[r * dk + c]);
            X[r] = fv[(i + r) * d->hv * dv + (int64_t)h * dv + j] - sk;
          }
          for (int64_t r = 0; r < nr; ++r) {
            double v = 0.0;
            for (int64_t m = 0; m <= r; ++m) v += Tm[r * nr + m] * X[m];
            D[r] = v;
          }
          for (int64_t r = 0; r < nr; ++r) {
            double sq = 0.0;
            for (int c = 0; c < dk; ++c) sq += row[c] * QQ(r)[c] * exp(lb[r * dk + c]);
            for (int64_t m = 0; m <= r; ++m) sq += Mm[r * nr + m] * D[m];
            out[(t0 + i + r) * HVDV + (int64_t)h * dv + j] = sq;
          }
          for (int c = 0; c < dk; ++c) {
            double last = lb[(nr - 1) * dk + c];
            double v = row[c] * exp(last);
            for (int64_t r = 0; r < nr; ++r) v += D[r] * KQ(r)[c] * exp(last - lb[r * dk + c]);
            rowbuf[c] = v;
          }
          memcpy(row, rowbuf, sizeof(double) * dk);
        }
#undef KQ
#undef QQ
#undef GG
        i += nr;
        /* a block boundary at the window's end */
        int64_t P = p0 + i;
        if (P % ckpt_block == 0) {
          int64_t idx = P / ckpt_block - blk0 - 1;
          if (idx >= 0 && idx < max_ckpt) {
            int32_t cid = ckpt_ids[(int64_t)n * max_ckpt + idx];
            int cc = slot_class(cid, ckpt.num_slots);
            if (cc == 2) fail |= ORC_ERR_SLOT_OOB;
            if (cc == 0) {
              memcpy(ckpt.ssm + cid * ns + (int64_t)h * dv * dk, St, sizeof(double) * dv * dk);
              if (h == 0) memcpy(ckpt.conv + cid * nc, hist_after + (i - 1) * nc, sizeof(double) * nc);
            }
          }
        }
      }
    }
    free(fq); free(fk); free(fv); free(fg); free(fb); free(hist_after); free(y);
    free(lb); free(Ap); free(Mm); free(Tm); free(X); free(D); free(rowbuf);
  }
  if (err) *err |= (uint32_t)fail;
  return 0;
}

/* ---- readout epilogue: gated RMS norm ----------------------------------
 * Not written on the pages.  The published Gated DeltaNet block normalises
 * each head's readout and gates it with a SiLU of a separate projection z:
 * for every (token, V head) row o of dv values,
 *   y = o / sqrt(mean(o^2) + eps) * w * silu(z)
 * with w [dv] a learned weight shared by the heads.  o, z, y are
 * [n_tok][hv][dv]; y may alias o. */
int orc_gated_rmsnorm(const orc_dims* d, const double* o, const double* z, const double* w,
                      double eps, int64_t n_tok, double* y) {
  if (check_dims(d) || n_tok < 0 || eps < 0.0) return 1;
  int64_t rows = n_tok * d->hv, dv = d->dv;
  for (int64_t r = 0; r < rows; ++r) {
    const double* orow = o + r * dv;
    double ss = 0.0;
    for (int64_t j = 0; j < dv; ++j) ss += orow[j] * orow[j];
    double inv = 1.0 / sqrt(ss / (double)dv + eps);
    for (int64_t j = 0; j < dv; ++j)
      y[r * dv + j] = orow[j] * inv * w[j] * orc_silu(z[r * dv + j]);
  }
  return 0;
}

/* ---- a8: prefill, token by token (the plain definition) -----------------
 * Sequence n owns tokens [cu_seqlens[n], cu_seqlens[n+1]) of qkv [Ttot][C]
 * (a,b [Ttot][hv], out [Ttot][hv][dv]); its first token sits at absolute
 * position start_pos[n] and its state lives in slot slot_ids[n].  After the
 * token at absolute position P-1, for every P with P % ckpt_block == 0 and
 * start_pos < P <= end, the slot's state (SSM + conv history) is copied to
 * checkpoint slot ckpt_ids[n][P/ckpt_block - floor(start_pos/ckpt_block) - 1]
 * (entry -1: skipped; index beyond max_ckpt: skipped).  Heads outside
 * [h_lo,h_hi) are not advanced (sampling). */
int orc_prefill(const orc_dims* d, orc_pool pool, orc_pool ckpt,
                const orc_params* p, const int32_t* slot_ids,
                const int32_t* cu_seqlens, const int64_t* start_pos,
                int32_t n_seq, const int32_t* ckpt_ids, int32_t max_ckpt,
                int32_t ckpt_block, const double* qkv, const double* a,
                const double* b, double* out, uint32_t* err, int32_t h_lo,
                int32_t h_hi) {
  if (check_dims(d) || ckpt_block <= 0) return 1;
  clamp_heads(d, &h_lo, &h_hi);
  int64_t C = n_chan(d), HVDV = (int64_t)d->hv * d->dv;
  int64_t ns = ssm_elems(d), nc = conv_elems(d);
  int64_t fail = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : fail)
  for (int32_t n = 0; n < n_seq; ++n) {
    int32_t s = slot_ids[n];
    int64_t t0 = cu_seqlens[n], t1 = cu_seqlens[n + 1];
    int cls = slot_class(s, pool.num_slots);
    if (cls) {
      if (cls == 2) fail |= ORC_ERR_SLOT_OOB;
      for (int64_t i = t0 * HVDV; i < t1 * HVDV; ++i) out[i] = 0.0;
      continue;
    }
    double* ssm = pool.ssm + s * ns;
    double* conv = pool.conv + s * nc;
    double* wk = (double*)malloc(sizeof(double) * work_elems(d));
    int64_t p0 = start_pos[n];
    int64_t blk0 = p0 / ckpt_block;
    for (int64_t i = t0; i < t1; ++i) {
      int64_t pos = p0 + (i - t0);
      token_step(d, p, ssm, conv, qkv + i * C, a + i * d->hv, b + i * d->hv,
                 out + i * HVDV, h_lo, h_hi, wk);
      int64_t P = pos + 1;
      if (P % ckpt_block) continue;
      int64_t idx = P / ckpt_block - blk0 - 1;
      if (idx < 0 || idx >= max_ckpt) continue;
      int32_t cid = ckpt_ids[(int64_t)n * max_ckpt + idx];
      int cc = slot_class(cid, ckpt.num_slots);
      if (cc == 2) fail |= ORC_ERR_SLOT_OOB;
      if (cc) continue;
      memcpy(ckpt.ssm + cid * ns, ssm, sizeof(double) * ns);
      memcpy(ckpt.conv + cid * nc, conv, sizeof(double) * nc);
    }
    free(wk);
  }
  if (err) *err |= (uint32_t)fail;
  return 0;
}

/* ---- a8 cross-check: the chunkwise WY/UT form (double) -------------------
 * Same contract as orc_prefill, but the state recurrence is evaluated one
 * chunk of `chunk` tokens at a time, chunks aligned to absolute positions
 * (multiples of `chunk`).  For a chunk with rows i (tokens), local cumulative
 * log-decay b_i = sum_{j<=i} g_j and Gamma_ij = exp(b_i - b_j) (i >= j):
 *   A = strict_lower(diag(beta) (K K^T (.) Gamma))
 *   T = (I + A)^{-1} diag(beta)          (forward substitution)
 *   W = T diag(e^b) K,   U = T V,   Delta = U - W S0
 *   O = diag(e^b) Q S0 + (Q K^T (.) Gamma (.) lower_incl_diag) Delta
 *   S_end = e^{b_last} S0 + (diag(e^{b_last - b}) K)^T Delta
 * with S = dk x dv.  ckpt_block must be a multiple of chunk. */
int orc_prefill_chunked(const orc_dims* d, orc_pool pool, orc_pool ckpt,
                        const orc_params* p, const int32_t* slot_ids,
                        const int32_t* cu_seqlens, const int64_t* start_pos,
                        int32_t n_seq, const int32_t* ckpt_ids,
                        int32_t max_ckpt, int32_t ckpt_block, int32_t chunk,
                        const double* qkv, const double* a, const double* b,
                        double* out, uint32_t* err) {
  if (check_dims(d) || ckpt_block <= 0 || chunk <= 0 || ckpt_block % chunk) return 1;
  int64_t C = n_chan(d), HVDV = (int64_t)d->hv * d->dv;
  int64_t ns = ssm_elems(d), nc = conv_elems(d);
  int dk = d->dk, dv = d->dv, G = d->hv / d->hk;
  int64_t fail = 0;
  for (int32_t n = 0; n < n_seq; ++n) {
    int32_t s = slot_ids[n];
    int64_t t0 = cu_seqlens[n], t1 = cu_seqlens[n + 1], L = t1 - t0;
    int cls = slot_class(s, pool.num_slots);
    if (cls) {
      if (cls == 2) fail |= ORC_ERR_SLOT_OOB;
      for (int64_t i = t0 * HVDV; i < t1 * HVDV; ++i) out[i] = 0.0;
      continue;
    }
    int64_t p0 = start_pos[n], blk0 = p0 / ckpt_block;
    /* per-token features, and the conv history at every chunk boundary */
    double* feat_q = (double*)malloc(sizeof(double) * (L + 1) * d->hk * dk);
    double* feat_k = (double*)malloc(sizeof(double) * (L + 1) * d->hk * dk);
    double* feat_v = (double*)malloc(sizeof(double) * (L + 1) * d->hv * dv);
    double* feat_g = (double*)malloc(sizeof(double) * (L + 1) * d->hv);
    double* feat_b = (double*)malloc(sizeof(double) * (L + 1) * d->hv);
    double* hist_at = (double*)malloc(sizeof(double) * (L + 1) * nc); /* history before token i */
    double* conv = pool.conv + s * nc;
    double* y = (double*)malloc(sizeof(double) * C);
    double* alpha_tmp = (double*)malloc(sizeof(double) * d->hv);
    for (int64_t i = 0; i < L; ++i) {
      memcpy(hist_at + i * nc, conv, sizeof(double) * nc);
      const double* x = qkv + (t0 + i) * C;
      orc_conv_silu(d, conv, x, p->conv_w, y);
      conv_shift(d, conv, x);
      orc_feat f = {feat_q + i * d->hk * dk, feat_k + i * d->hk * dk, NULL,
                    feat_g + i * d->hv, alpha_tmp, feat_b + i * d->hv};
      token_features(d, p, y, a + (t0 + i) * d->hv, b + (t0 + i) * d->hv, &f);
      memcpy(feat_v + i * d->hv * dv, y + 2 * (int64_t)d->hk * dk, sizeof(double) * d->hv * dv);
    }
    memcpy(hist_at + L * nc, conv, sizeof(double) * nc);

    int64_t maxc = chunk;
    double* S = (double*)malloc(sizeof(double) * dk * dv);     /* S[m][j] */
    double* bcum = (double*)malloc(sizeof(double) * maxc);
    double* A = (double*)malloc(sizeof(double) * maxc * maxc);
    double* Tm = (double*)malloc(sizeof(double) * maxc * maxc);
    double* Wm = (double*)malloc(sizeof(double) * maxc * dk);
    double* Um = (double*)malloc(sizeof(double) * maxc * dv);
    double* Dm = (double*)malloc(sizeof(double) * maxc * dv);
    double* Snew = (double*)malloc(sizeof(double) * dk * dv);

    for (int h = 0; h < d->hv; ++h) {
      int hq = h / G;
      double* St = pool.ssm + s * ns + (int64_t)h * dv * dk;
      for (int m = 0; m < dk; ++m)
        for (int j = 0; j < dv; ++j) S[m * dv + j] = St[(int64_t)j * dk + m];
      int64_t i = 0;
      while (i < L) {
        int64_t pos = p0 + i;
        int64_t cend = (pos / chunk + 1) * chunk; /* absolute end of this chunk */
        int64_t n_r = cend - pos;
        if (n_r > L - i) n_r = L - i;
#define KR(r) (feat_k + (i + (r)) * d->hk * dk + (int64_t)hq * dk)
#define QR(r) (feat_q + (i + (r)) * d->hk * dk + (int64_t)hq * dk)
#define VR(r) (feat_v + (i + (r)) * d->hv * dv + (int64_t)h * dv)
        double acc = 0.0;
        for (int64_t r = 0; r < n_r; ++r) {
          acc += feat_g[(i + r) * d->hv + h];
          bcum[r] = acc;
        }
        for (int64_t r = 0; r < n_r; ++r)
          for (int64_t c = 0; c < n_r; ++c) {
            double v = 0.0;
            if (c < r) {
              double kk = 0.0;
              for (int m = 0; m < dk; ++m) kk += KR(r)[m] * KR(c)[m];
              v = feat_b[(i + r) * d->hv + h] * kk * exp(bcum[r] - bcum[c]);
            }
            A[r * n_r + c] = v;
          }
        /* (I + A) T = diag(beta), row by row */
        for (int64_t r = 0; r < n_r; ++r)
          for (int64_t c = 0; c < n_r; ++c) {
            double v = (r == c) ? feat_b[(i + r) * d->hv + h] : 0.0;
            for (int64_t m = 0; m < r; ++m) v -= A[r * n_r + m] * Tm[m * n_r + c];
            Tm[r * n_r + c] = v;
          }
        for (int64_t r = 0; r < n_r; ++r) {
          for (int m = 0; m < dk; ++m) {
            double v = 0.0;
            for (int64_t c = 0; c < n_r; ++c) v += Tm[r * n_r + c] * exp(bcum[c]) * KR(c)[m];
            Wm[r * dk + m] = v;
          }
          for (int j = 0; j < dv; ++j) {
            double v = 0.0;
            for (int64_t c = 0; c < n_r; ++c) v += Tm[r * n_r + c] * VR(c)[j];
            Um[r * dv + j] = v;
          }
        }
        for (int64_t r = 0; r < n_r; ++r)
          for (int j = 0; j < dv; ++j) {
            double ws = 0.0;
            for (int m = 0; m < dk; ++m) ws += Wm[r * dk + m] * S[m * dv + j];
            Dm[r * dv + j] = Um[r * dv + j] - ws;
          }
        for (int64_t r = 0; r < n_r; ++r) {
          double* o = out + (t0 + i + r) * HVDV + (int64_t)h * dv;
          for (int j = 0; j < dv; ++j) {
            double qs = 0.0;
            for (int m = 0; m < dk; ++m) qs += QR(r)[m] * S[m * dv + j];
            double v = exp(bcum[r]) * qs;
            for (int64_t c = 0; c <= r; ++c) {
              double qk = 0.0;
              for (int m = 0; m < dk; ++m) qk += QR(r)[m] * KR(c)[m];
              v += qk * exp(bcum[r] - bcum[c]) * Dm[c * dv + j];
            }
            o[j] = v;
          }
        }
        double blast = bcum[n_r - 1];
        for (int m = 0; m < dk; ++m)
          for (int j = 0; j < dv; ++j) {
            double v = exp(blast) * S[m * dv + j];
            for (int64_t c = 0; c < n_r; ++c)
              v += exp(blast - bcum[c]) * KR(c)[m] * Dm[c * dv + j];
            Snew[m * dv + j] = v;
          }
        memcpy(S, Snew, sizeof(double) * dk * dv);
#undef KR
#undef QR
#undef VR
        i += n_r;
        int64_t P = p0 + i;
        if (P % ckpt_block == 0) {
          int64_t idx = P / ckpt_block - blk0 - 1;
          if (idx >= 0 && idx < max_ckpt) {
            int32_t cid = ckpt_ids[(int64_t)n * max_ckpt + idx];
            int cc = slot_class(cid, ckpt.num_slots);
            if (cc == 2) fail |= ORC_ERR_SLOT_OOB;
            if (!cc) {
              double* Ct = ckpt.ssm + cid * ns + (int64_t)h * dv * dk;
              for (int m = 0; m < dk; ++m)
                for (int j = 0; j < dv; ++j) Ct[(int64_t)j * dk + m] = S[m * dv + j];
              if (h == 0) memcpy(ckpt.conv + cid * nc, hist_at + i * nc, sizeof(double) * nc);
            }
          }
        }
      }
      for (int m = 0; m < dk; ++m)
        for (int j = 0; j < dv; ++j) St[(int64_t)j * dk + m] = S[m * dv + j];
    }
    free(S); free(bcum); free(A); free(Tm); free(Wm); free(Um); free(Dm); free(Snew);
    free(feat_q); free(feat_k); free(feat_v); free(feat_g); free(feat_b);
    free(hist_at); free(y); free(alpha_tmp);
  }
  if (err) *err |= (uint32_t)fail;
  return 0;
}

int orc_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}
