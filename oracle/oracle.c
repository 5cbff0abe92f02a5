/*
 * ORACLE: plain, slow, obviously correct CPU implementation of the fused
 * mixture-of-experts FFN layer.  Test infrastructure only: it is called by the
 * tests, by the smoke check and by the benchmark's CPU-baseline leg, never by
 * the library.  It shares no code with the CUDA path or with the input
 * generator.
 *
 * What it computes (the layer of "ggml-cuda: overlap the MoE shared expert on
 * a separate stream", ROCm/llama.cpp PR #36, section "What this changes": the
 * diamond join = add(ffn_moe_out, ffn_shexp) whose two branches are forked
 * from the FFN-input norm).  The per-step arithmetic is not printed on that
 * page; it is the plain reading of the layer named there: a router GEMV,
 * softmax over experts, top-k selection renormalised to sum 1, SwiGLU experts,
 * a sigmoid-gated shared expert and the final add.  Everything is accumulated
 * in double, in the natural index order, and rounded to fp32 only where a
 * result leaves the oracle:
 *
 *   logit[t,e] = fp32( sum_h Wr[e,h] * x[t,h] )
 *   top-k      = the k largest fp32 logits; equal logits go to the lower index
 *   p[t,j]     = exp(l_j - l_1) / sum_{i<k} exp(l_i - l_1)      (double)
 *   s[t]       = 1 / (1 + exp(-sum_h g[h] * x[t,h]))            (double)
 *   FFN_e(x)   = Wd_e ( silu(Wg_e x) * (Wu_e x) ),  silu(z) = z / (1 + e^-z)
 *   out[t]     = fp32( sum_{j<k} p[t,j] FFN_{id[t,j]}(x_t) + s[t] FFN_sh(x_t) )
 *
 * The routed sum runs in rank order (slot 0 first) and the shared term is
 * added last, which is the order of add(ffn_moe_out, ffn_shexp).
 *
 * Weight formats read here:
 *   bf16:  row-major [rows, cols] bf16.
 *   4-bit: each row = cols/2 bytes of nibbles (element 2j in the low nibble of
 *          byte j, element 2j+1 in the high nibble) followed by cols/32 fp16
 *          scales; element value = d * (nibble - 8) for its 32-block.
 *   int8:  each row = cols signed bytes q, then one fp32 scale s (little
 *          endian) and 12 bytes of padding; element value = s * q.  With this
 *          format the gate and up projections take an int8 activation, as the
 *          int8 linear of "ggml operator extensions" (sd.cpp integration,
 *          sd.linear_i8.v1) defines it: x is quantised per token,
 *          xs = max|x| / 127 and qx = clamp(round(x / xs), -127, 127) in fp32
 *          (round half away from zero; xs = 0 gives qx = 0), and the
 *          projection is float(int32_dot(W, qx)) * xs * s, the products in
 *          that order in fp32; SwiGLU follows.  The down projection uses the
 *          weights s * q with the fp32 h (in double, like the other formats).
 * Layer layout: router [E,H]; expert e = gate [I,H] | up [I,H] | downT [I,H];
 * shared = gate [Is,H] | up [Is,H] | downT [Is,H]; shared-gate vector [H] bf16.
 * downT is the down projection stored transposed (row i = column i of the
 * [H,I] matrix Wd), so every stored row has H elements and, in the 4-bit
 * format, the blocks of all three matrices run along H.
 *
 * Portable C11 with pthreads; built with -ffp-contract=off.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int32_t T, H, E, top_k, I, Is;
} or_shapes;

/* ---------------------------------------------------------------- */
/* Scalar decoding of the stored formats                             */

double or_bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* IEEE binary16 -> double, written from the format: sign, 5-bit exponent with
 * bias 15, 10-bit fraction; exponent 0 is subnormal (fraction * 2^-24). */
double or_f16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int m = h & 0x3FF;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + m), e - 25);
  return sign ? -v : v;
}

/* fp32 -> bf16 with round to nearest even (used for the normalised
 * activation of the layer stack, which is stored in bf16). */
uint16_t or_float_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
  uint32_t rounding = 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)((u + rounding) >> 16);
}

/* fp32 scale of an int8 row (the 4 bytes after its cols values). */
static float i8_row_scale(const uint8_t* row, int64_t cols) {
  float s;
  memcpy(&s, row + cols, 4);
  return s;
}

/* Value of element c of row r of a weight matrix with `cols` columns. */
static double weight_at(const uint8_t* base, int wfmt, int64_t cols, int64_t r, int64_t c) {
  if (wfmt == 0) {
    const uint16_t* w = (const uint16_t*)base;
    return or_bf16_to_double(w[r * cols + c]);
  }
  if (wfmt == 2) {
    const uint8_t* row = base + r * (cols + 16);
    return (double)i8_row_scale(row, cols) * (double)(int8_t)row[c];
  }
  const uint8_t* row = base + r * (cols * 9 / 16);
  uint8_t byte = row[c / 2];
  int nib = (c & 1) ? (byte >> 4) : (byte & 0x0F);
  const uint8_t* sc = row + cols / 2 + 2 * (c / 32);
  uint16_t dbits = (uint16_t)(sc[0] | (sc[1] << 8));
  return or_f16_to_double(dbits) * (double)(nib - 8);
}

/* Decode one stored row into doubles (test helper). */
void or_decode_row(const uint8_t* base, int wfmt, int64_t cols, int64_t r, double* out) {
  for (int64_t c = 0; c < cols; ++c) out[c] = weight_at(base, wfmt, cols, r, c);
}

static int64_t matrix_bytes(int wfmt, int64_t rows, int64_t cols) {
  return wfmt == 0 ? rows * cols * 2 : wfmt == 1 ? rows * (cols * 9 / 16) : rows * (cols + 16);
}

/* The int8 activation of one row of n values (each an fp32 value): scale
 * xs = fp32(max|x|) / 127 in fp32, q = clamp(roundf(x / xs), -127, 127) with
 * the division in fp32 and rounding half away from zero; xs = 0 gives q = 0. */
void or_quantize_i8(const double* x, int64_t n, int8_t* q, float* scale) {
  float amax = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float a = fabsf((float)x[i]);
    if (a > amax) amax = a;
  }
  float xs = amax / 127.0f;
  for (int64_t i = 0; i < n; ++i) {
    int v = 0;
    if (xs != 0.0f) {
      float r = roundf((float)x[i] / xs);
      v = (int)r;
      if (v > 127) v = 127;
      if (v < -127) v = -127;
    }
    q[i] = (int8_t)v;
  }
  *scale = xs;
}

/* float(int32_dot(W_r, q)) * xs * s_r for row r of an int8 matrix, in fp32,
 * the products in that order; returned as double. */
static double i8_projection(const uint8_t* W, int64_t cols, int64_t r, const int8_t* q, float xs) {
  const uint8_t* row = W + r * (cols + 16);
  int64_t dot = 0;
  for (int64_t c = 0; c < cols; ++c) dot += (int64_t)(int8_t)row[c] * (int64_t)q[c];
  float v = (float)dot;
  v = v * xs;
  v = v * i8_row_scale(row, cols);
  return (double)v;
}

/* Bytes of one expert block (gate | up | downT) with intermediate size `inter`. */
int64_t or_expert_bytes(int wfmt, int64_t H, int64_t inter) {
  return 3 * matrix_bytes(wfmt, inter, H);
}

/* y[r] = sum_c W[r,c] * v[c], in double, c ascending. */
static void matvec(const uint8_t* W, int wfmt, int64_t rows, int64_t cols, const double* v, double* y) {
  for (int64_t r = 0; r < rows; ++r) {
    double acc = 0.0;
    for (int64_t c = 0; c < cols; ++c) acc += weight_at(W, wfmt, cols, r, c) * v[c];
    y[r] = acc;
  }
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* One SwiGLU FFN: y = Wd ( silu(gate x) * (up x) ).  blk points at
 * gate|up|downT; y[c] = sum_i Wd[c,i] h[i] with Wd[c,i] = downT[i,c], in
 * double, i ascending. */
void or_swiglu_ffn(const uint8_t* blk, int wfmt, int64_t H, int64_t inter, const double* x, double* y) {
  double* g = (double*)malloc(sizeof(double) * (size_t)inter);
  double* u = (double*)malloc(sizeof(double) * (size_t)inter);
  const uint8_t* Wg = blk;
  const uint8_t* Wu = blk + matrix_bytes(wfmt, inter, H);
  const uint8_t* WdT = blk + 2 * matrix_bytes(wfmt, inter, H);
  if (wfmt == 2) {
    int8_t* q = (int8_t*)malloc((size_t)H);
    float xs;
    or_quantize_i8(x, H, q, &xs);
    for (int64_t i = 0; i < inter; ++i) {
      g[i] = i8_projection(Wg, H, i, q, xs);
      u[i] = i8_projection(Wu, H, i, q, xs);
    }
    free(q);
  } else {
    matvec(Wg, wfmt, inter, H, x, g);
    matvec(Wu, wfmt, inter, H, x, u);
  }
  for (int64_t i = 0; i < inter; ++i) g[i] = silu(g[i]) * u[i];
  for (int64_t c = 0; c < H; ++c) {
    double acc = 0.0;
    for (int64_t i = 0; i < inter; ++i) acc += weight_at(WdT, wfmt, H, i, c) * g[i];
    y[c] = acc;
  }
  free(g);
  free(u);
}

/* ---------------------------------------------------------------- */
/* Router, top-k and bucketing                                       */

/* logits[e] = fp32(sum_h Wr[e,h] x[h]) for one token. */
void or_router_logits(const uint16_t* router_w, int64_t E, int64_t H, const double* x, float* logits) {
  for (int64_t e = 0; e < E; ++e) {
    double acc = 0.0;
    for (int64_t h = 0; h < H; ++h) acc += or_bf16_to_double(router_w[e * H + h]) * x[h];
    logits[e] = (float)acc;
  }
}

/* The k largest logits, larger first, equal values ordered by lower index;
 * p = softmax restricted to the chosen k (identical to a full softmax followed
 * by zeroing the others and renormalising).  p_out in double. */
void or_topk(const float* logits, int64_t E, int64_t k, int32_t* ids, double* p_out) {
  char* taken = (char*)calloc((size_t)E, 1);
  for (int64_t j = 0; j < k; ++j) {
    int64_t best = -1;
    for (int64_t e = 0; e < E; ++e) {
      if (taken[e]) continue;
      if (best < 0 || logits[e] > logits[best]) best = e; /* strict: the lower index keeps a tie */
    }
    taken[best] = 1;
    ids[j] = (int32_t)best;
  }
  free(taken);
  double l1 = (double)logits[ids[0]];
  double z = 0.0;
  for (int64_t j = 0; j < k; ++j) z += exp((double)logits[ids[j]] - l1);
  for (int64_t j = 0; j < k; ++j) p_out[j] = exp((double)logits[ids[j]] - l1) / z;
}

/* Token -> expert bucketing, written as the plain stable counting sort:
 * counts[e] = #{(t,j): id[t,j] = e}; offsets = exclusive prefix sum (E+1);
 * perm lists the flat indices t*k+j grouped by expert (ascending expert), and
 * token-major, slot-minor inside a group; active = experts with counts > 0,
 * ascending.  Returns U = number of active experts. */
int32_t or_bucketing(const int32_t* ids, int64_t T, int64_t k, int64_t E, int32_t* counts, int32_t* offsets,
                     int32_t* perm, int32_t* active) {
  int64_t pos = 0;
  int32_t U = 0;
  for (int64_t e = 0; e < E; ++e) {
    offsets[e] = (int32_t)pos;
    int32_t c = 0;
    for (int64_t ts = 0; ts < T * k; ++ts) {
      if (ids[ts] == e) {
        perm[pos++] = (int32_t)ts;
        c++;
      }
    }
    counts[e] = c;
    if (c > 0) active[U++] = (int32_t)e;
  }
  offsets[E] = (int32_t)pos;
  return U;
}

/* ---------------------------------------------------------------- */
/* The layer                                                         */

/* The FFNs of a layer call (one per routed (token, slot) and one per token for
 * the shared expert) are evaluated in two phases, each split into tasks of
 * TASK_ROWS rows that any thread may take:
 *   phase 0: h[i] = silu(gate_i . x) * (up_i . x) for rows i of each FFN;
 *   phase 1: y[c] = sum_i downT[i,c] h[i], i ascending, for columns c.
 * Every value is computed by exactly the loops of or_swiglu_ffn (same terms,
 * same order), so the result is bit-identical to calling or_swiglu_ffn per FFN
 * and does not depend on the number of threads. */
#define TASK_ROWS 64

typedef struct {
  const uint8_t* blk;
  int wfmt;
  int64_t H, inter;
  const double* x;
  const int8_t* qx; /* int8 format: the token's int8 activation [H] */
  float xs;         /* and its scale */
  double* h;        /* [inter] */
  double* y;        /* [H] */
} ffn_job;

typedef struct {
  ffn_job* jobs;
  int64_t njobs;
  int64_t* first; /* [njobs + 1]: first task of each job in the current phase */
  int phase;
  int64_t next;
  pthread_mutex_t mu;
} job_queue;

static void run_task(const ffn_job* f, int phase, int64_t r0, int64_t r1) {
  const int64_t mb = matrix_bytes(f->wfmt, f->inter, f->H);
  if (phase == 0) {
    for (int64_t i = r0; i < r1; ++i) {
      double g = 0.0, u = 0.0;
      if (f->wfmt == 2) {
        g = i8_projection(f->blk, f->H, i, f->qx, f->xs);
        u = i8_projection(f->blk + mb, f->H, i, f->qx, f->xs);
      } else {
        for (int64_t c = 0; c < f->H; ++c) g += weight_at(f->blk, f->wfmt, f->H, i, c) * f->x[c];
        for (int64_t c = 0; c < f->H; ++c) u += weight_at(f->blk + mb, f->wfmt, f->H, i, c) * f->x[c];
      }
      f->h[i] = silu(g) * u;
    }
  } else {
    for (int64_t c = r0; c < r1; ++c) {
      double acc = 0.0;
      for (int64_t i = 0; i < f->inter; ++i) acc += weight_at(f->blk + 2 * mb, f->wfmt, f->H, i, c) * f->h[i];
      f->y[c] = acc;
    }
  }
}

static void* ffn_worker(void* arg) {
  job_queue* q = (job_queue*)arg;
  const int64_t ntasks = q->first[q->njobs];
  for (;;) {
    pthread_mutex_lock(&q->mu);
    int64_t k = q->next++;
    pthread_mutex_unlock(&q->mu);
    if (k >= ntasks) break;
    int64_t j = 0;
    while (q->first[j + 1] <= k) ++j;
    const ffn_job* f = &q->jobs[j];
    const int64_t n = q->phase == 0 ? f->inter : f->H;
    const int64_t r0 = (k - q->first[j]) * TASK_ROWS;
    run_task(f, q->phase, r0, r0 + TASK_ROWS < n ? r0 + TASK_ROWS : n);
  }
  return NULL;
}

static void run_jobs(ffn_job* jobs, int64_t njobs, int nthreads) {
  job_queue q;
  q.jobs = jobs;
  q.njobs = njobs;
  q.first = (int64_t*)malloc(sizeof(int64_t) * (size_t)(njobs + 1));
  pthread_mutex_init(&q.mu, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  for (int phase = 0; phase < 2; ++phase) {
    q.phase = phase;
    q.next = 0;
    q.first[0] = 0;
    for (int64_t j = 0; j < njobs; ++j)
      q.first[j + 1] = q.first[j] + ((phase == 0 ? jobs[j].inter : jobs[j].H) + TASK_ROWS - 1) / TASK_ROWS;
    int nt = nthreads;
    if (nt > q.first[njobs]) nt = (int)q.first[njobs];
    pthread_t th[256];
    int created[256];
    for (int t = 1; t < nt; ++t) created[t] = pthread_create(&th[t], NULL, ffn_worker, &q) == 0;
    ffn_worker(&q);
    for (int t = 1; t < nt; ++t)
      if (created[t]) pthread_join(th[t], NULL);
  }
  pthread_mutex_destroy(&q.mu);
  free(q.first);
}

/* Threads a layer call of these shapes would use when offered nthreads. */
int or_threads_used(const or_shapes* s, int nthreads) {
  const int64_t njobs = (int64_t)s->T * s->top_k + s->T;
  const int64_t t0 = ((int64_t)s->T * s->top_k * ((s->I + TASK_ROWS - 1) / TASK_ROWS) +
                      (int64_t)s->T * ((s->Is + TASK_ROWS - 1) / TASK_ROWS));
  const int64_t t1 = njobs * ((s->H + TASK_ROWS - 1) / TASK_ROWS);
  int64_t m = t0 > t1 ? t0 : t1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  return (int)(m < nthreads ? m : nthreads);
}

/*
 * Full layer for T tokens.  act: 0 = x is fp32 [T,H], 1 = x is bf16 [T,H].
 * wfmt: 0 = bf16 experts and shared expert, 1 = 4-bit blocks, 2 = int8 rows.
 * Outputs: out fp32 [T,H]; optional logits fp32 [T,E], ids int32 [T,k],
 * p fp32 [T,k], s fp32 [T].  The result does not depend on nthreads.
 * Returns 0, or -1 on an invalid argument.
 */
int or_moe_ffn(const or_shapes* s, int act, int wfmt, const void* x, const uint16_t* router_w, const uint8_t* expert_w,
               const uint8_t* shexp_w, const uint16_t* shexp_gate_w, int nthreads, float* out, float* logits_out,
               int32_t* ids_out, float* p_out, float* s_out) {
  if (!s || !x || !router_w || !expert_w || !shexp_w || !shexp_gate_w || !out) return -1;
  const int64_t T = s->T, H = s->H, E = s->E, k = s->top_k, I = s->I, Is = s->Is;
  if (T < 0 || H <= 0 || E <= 0 || k <= 0 || k > E || I <= 0 || Is <= 0) return -1;
  if (wfmt == 1 && (H % 32 || I % 32 || Is % 32)) return -1;
  if (wfmt == 2 && H % 16) return -1;
  if (wfmt < 0 || wfmt > 2) return -1;
  if (T == 0) return 0;

  double* xd = (double*)malloc(sizeof(double) * (size_t)(T * H));
  for (int64_t i = 0; i < T * H; ++i)
    xd[i] = act == 0 ? (double)((const float*)x)[i] : or_bf16_to_double(((const uint16_t*)x)[i]);

  float* logits = (float*)malloc(sizeof(float) * (size_t)(T * E));
  int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T * k));
  double* p = (double*)malloc(sizeof(double) * (size_t)(T * k));
  double* sg = (double*)malloc(sizeof(double) * (size_t)T);
  for (int64_t t = 0; t < T; ++t) {
    const double* xt = xd + t * H;
    or_router_logits(router_w, E, H, xt, logits + t * E);
    or_topk(logits + t * E, E, k, ids + t * k, p + t * k);
    double a = 0.0;
    for (int64_t h = 0; h < H; ++h) a += or_bf16_to_double(shexp_gate_w[h]) * xt[h];
    sg[t] = 1.0 / (1.0 + exp(-a));
  }

  /* One job per routed (token, slot) and one per token for the shared expert. */
  const int64_t eb = or_expert_bytes(wfmt, H, I);
  const int64_t njobs = T * k + T;
  const int64_t hmax = I > Is ? I : Is;
  ffn_job* jobs = (ffn_job*)malloc(sizeof(ffn_job) * (size_t)njobs);
  double* y = (double*)malloc(sizeof(double) * (size_t)(njobs * H));
  double* hbuf = (double*)malloc(sizeof(double) * (size_t)(njobs * hmax));
  /* int8 format: each token's activation quantised once, shared by its FFNs */
  int8_t* qx = (int8_t*)malloc((size_t)(T * H));
  float* xs = (float*)malloc(sizeof(float) * (size_t)T);
  for (int64_t t = 0; t < T; ++t) {
    xs[t] = 0.0f;
    if (wfmt == 2) or_quantize_i8(xd + t * H, H, qx + t * H, &xs[t]);
  }
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t j = 0; j < k; ++j) {
      int64_t n = t * k + j;
      jobs[n] = (ffn_job){expert_w + (int64_t)ids[n] * eb, wfmt, H, I, xd + t * H, qx + t * H, xs[t],
                          hbuf + n * hmax, y + n * H};
    }
    int64_t n = T * k + t;
    jobs[n] = (ffn_job){shexp_w, wfmt, H, Is, xd + t * H, qx + t * H, xs[t], hbuf + n * hmax, y + n * H};
  }
  run_jobs(jobs, njobs, nthreads);
  free(hbuf);
  free(qx);
  free(xs);

  for (int64_t t = 0; t < T; ++t) {
    for (int64_t h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int64_t j = 0; j < k; ++j) acc += p[t * k + j] * y[(t * k + j) * H + h];
      acc += sg[t] * y[(T * k + t) * H + h];
      out[t * H + h] = (float)acc;
    }
  }
  if (logits_out) memcpy(logits_out, logits, sizeof(float) * (size_t)(T * E));
  if (ids_out) memcpy(ids_out, ids, sizeof(int32_t) * (size_t)(T * k));
  if (p_out)
    for (int64_t i = 0; i < T * k; ++i) p_out[i] = (float)p[i];
  if (s_out)
    for (int64_t t = 0; t < T; ++t) s_out[t] = (float)sg[t];

  free(xd);
  free(logits);
  free(ids);
  free(p);
  free(sg);
  free(jobs);
  free(y);
  return 0;
}

/* ---------------------------------------------------------------- */
/* Transformer-block form used by the layer stack                    */

/* y = bf16( x / sqrt(mean(x^2) + eps) ), weight 1.0, for one token. */
void or_rmsnorm_bf16(const float* x, int64_t H, double eps, uint16_t* y) {
  double ss = 0.0;
  for (int64_t h = 0; h < H; ++h) ss += (double)x[h] * (double)x[h];
  double inv = 1.0 / sqrt(ss / (double)H + eps);
  for (int64_t h = 0; h < H; ++h) y[h] = or_float_to_bf16((float)((double)x[h] * inv));
}

/*
 * One pre-norm block: xn = bf16(RMSNorm(x_res)); m = fp32(MoE(xn));
 * x_res <- fp32(x_res + m).  The MoE output and the residual add are rounded
 * to fp32 separately.  x_res fp32 [T,H] is updated in place.  Optional ids
 * [T,k] and xn_out bf16 [T,H] report the routing and the normalised input.
 */
int or_block_step(const or_shapes* s, int wfmt, float* x_res, const uint16_t* router_w, const uint8_t* expert_w,
                  const uint8_t* shexp_w, const uint16_t* shexp_gate_w, double eps, int nthreads, int32_t* ids_out,
                  uint16_t* xn_out) {
  const int64_t T = s->T, H = s->H;
  uint16_t* xn = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(T * H));
  float* m = (float*)malloc(sizeof(float) * (size_t)(T * H));
  for (int64_t t = 0; t < T; ++t) or_rmsnorm_bf16(x_res + t * H, H, eps, xn + t * H);
  int rc = or_moe_ffn(s, 1, wfmt, xn, router_w, expert_w, shexp_w, shexp_gate_w, nthreads, m, NULL, ids_out, NULL,
                      NULL);
  if (rc == 0)
    for (int64_t i = 0; i < T * H; ++i) x_res[i] = (float)((double)x_res[i] + (double)m[i]);
  if (xn_out) memcpy(xn_out, xn, sizeof(uint16_t) * (size_t)(T * H));
  free(xn);
  free(m);
  return rc;
}
