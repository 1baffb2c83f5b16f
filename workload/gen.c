/*
 * Seeded synthetic inputs for the sparse-KV reuse decode step.
 *
 * This file holds no part of the method: it draws the per-step top-k token
 * selections, the fp32 queries and the bf16 K/V rows that both the CPU oracle
 * and the CUDA path consume.  Every random number comes from a counter-based
 * SplitMix64 stream (Steele, Lea, Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014), keyed by (seed, purpose, stream index), so any
 * element can be drawn independently and the fill is parallel over threads.
 *
 * Normals use the Box-Muller transform on two uniforms; fp32 -> bf16 uses
 * round-to-nearest-even on the bit pattern.
 *
 * Selection recipe (one chain per (request, kv-head)), after the workloads
 * the AVSG page (arxivdaily 2609.37538, English abstract) and the Spin page
 * (gist.science 2604.26837, section 1) describe: DSA keeps re-selecting a
 * large overlap of ids across decode steps.
 *   forced : a fixed id list (first/last positions) always present;
 *   kept   : each non-forced id of the previous selection, independently with
 *            probability p_keep (p_keep_token between tokens of one MTP
 *            iteration);
 *   fresh  : the rest; floor(zipf_frac * n_fresh) drawn Zipf(s) over the rank
 *            from the end of the context (rank r -> id L - r), then uniform
 *            without replacement; collisions are redrawn;
 *   order  : Fisher-Yates shuffle of the final list.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* Key of one stream: nested mixing of every coordinate. */
static uint64_t stream_key(uint64_t seed, uint64_t purpose, uint64_t a,
                           uint64_t b, uint64_t c) {
  uint64_t k = mix64(seed + GAMMA);
  k = mix64(k ^ mix64(purpose + 1 * GAMMA));
  k = mix64(k ^ mix64(a + 2 * GAMMA));
  k = mix64(k ^ mix64(b + 3 * GAMMA));
  k = mix64(k ^ mix64(c + 4 * GAMMA));
  return k;
}

/* The i-th draw of a stream (i >= 0). */
static inline uint64_t draw(uint64_t key, uint64_t i) {
  return mix64(key + (i + 1) * GAMMA);
}

static inline double to_unit(uint64_t x) { /* [0, 1) with 53 bits */
  return (double)(x >> 11) * (1.0 / 9007199254740992.0);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t b;
  memcpy(&b, &f, 4);
  b += 0x7FFFu + ((b >> 16) & 1u);
  return (uint16_t)(b >> 16);
}

/* ------------------------------------------------------------------ normals */

typedef struct {
  void* out;
  int is_bf16;
  int64_t per_stream, begin, end; /* flat element range [begin, end) */
  uint64_t seed, purpose;
  int64_t stream_base;
} normal_job;

static void* normal_worker(void* arg) {
  normal_job* j = (normal_job*)arg;
  int64_t cur_stream = -1;
  uint64_t key = 0;
  const double two_pi = 6.283185307179586476925286766559;
  for (int64_t e = j->begin; e < j->end; ++e) {
    int64_t s = e / j->per_stream, w = e - s * j->per_stream;
    if (s != cur_stream) {
      cur_stream = s;
      key = stream_key(j->seed, j->purpose, (uint64_t)(j->stream_base + s), 0, 0);
    }
    uint64_t pair = (uint64_t)(w >> 1);
    double u1 = to_unit(draw(key, 2 * pair)), u2 = to_unit(draw(key, 2 * pair + 1));
    double r = sqrt(-2.0 * log(1.0 - u1));
    double z = (w & 1) ? r * sin(two_pi * u2) : r * cos(two_pi * u2);
    float f = (float)z;
    if (j->is_bf16)
      ((uint16_t*)j->out)[e] = f32_to_bf16_rne(f);
    else
      ((float*)j->out)[e] = f;
  }
  return NULL;
}

/* Fill out[nstreams][per_stream] with N(0,1): bf16 bit patterns (is_bf16=1,
 * uint16 storage) or fp32.  Stream s uses key (seed, purpose, stream_base+s). */
int gen_normal(void* out, int is_bf16, int64_t nstreams, int64_t per_stream,
               uint64_t seed, uint64_t purpose, int64_t stream_base, int nthreads) {
  if (!out || nstreams < 0 || per_stream <= 0) return -1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  int64_t total = nstreams * per_stream;
  pthread_t th[256];
  normal_job jobs[256];
  int64_t chunk = (total + nthreads - 1) / nthreads;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    int64_t b = (int64_t)t * chunk, e = b + chunk;
    if (b >= total) break;
    if (e > total) e = total;
    jobs[t] = (normal_job){out, is_bf16, per_stream, b, e, seed, purpose, stream_base};
    if (pthread_create(&th[t], NULL, normal_worker, &jobs[t]) != 0) {
      normal_worker(&jobs[t]);
      th[t] = 0;
    }
    started = t + 1;
  }
  for (int t = 0; t < started; ++t)
    if (th[t]) pthread_join(th[t], NULL);
  return 0;
}

/* --------------------------------------------------------------- selections */

typedef struct {
  int32_t units, num_entries, k, steps, tokens;
  double p_keep, p_keep_token, zipf_frac, zipf_s;
  int32_t num_forced;
  const int32_t* forced;
  uint64_t seed;
  int32_t unit_base; /* unit u draws from the stream of unit unit_base + u */
} sel_params;

typedef struct {
  const sel_params* p;
  int32_t* out;
  const double* cdf; /* Zipf CDF over rank 1..L, or NULL */
  int32_t u_begin, u_end;
  int status;
} sel_job;

#define MAX_TRIES 100000000LL

static int32_t zipf_rank(const double* cdf, int32_t n, double u) {
  /* smallest index i with cdf[i] > u; rank = i + 1 */
  int32_t lo = 0, hi = n - 1;
  while (lo < hi) {
    int32_t mid = lo + (hi - lo) / 2;
    if (cdf[mid] > u) hi = mid; else lo = mid + 1;
  }
  return lo + 1;
}

static void* sel_worker(void* arg) {
  sel_job* j = (sel_job*)arg;
  const sel_params* p = j->p;
  const int32_t L = p->num_entries, k = p->k;
  uint32_t* mark = (uint32_t*)calloc((size_t)L, sizeof(uint32_t));
  if (!mark) { j->status = -2; return NULL; }
  uint32_t stamp = 0;
  for (int32_t u = j->u_begin; u < j->u_end; ++u) {
    const int32_t* prev = NULL;
    for (int32_t t = 0; t < p->steps; ++t) {
      for (int32_t tok = 0; tok < p->tokens; ++tok) {
        int32_t* cur = j->out + (((int64_t)t * p->units + u) * p->tokens + tok) * (int64_t)k;
        uint64_t key = stream_key(p->seed, 4, (uint64_t)(u + p->unit_base), (uint64_t)t,
                                  (uint64_t)tok);
        uint64_t ctr = 0;
        ++stamp;
        if (stamp == 0) { memset(mark, 0, (size_t)L * 4); stamp = 1; }
        int32_t n = 0;
        for (int32_t f = 0; f < p->num_forced && n < k; ++f) {
          int32_t id = p->forced[f];
          if (id < 0 || id >= L || mark[id] == stamp) continue;
          mark[id] = stamp;
          cur[n++] = id;
        }
        if (prev) {
          double pk = tok > 0 ? p->p_keep_token : p->p_keep;
          for (int32_t i = 0; i < k && n < k; ++i) {
            int32_t id = prev[i];
            if (mark[id] == stamp) continue; /* forced: kept without a draw */
            if (to_unit(draw(key, ctr++)) < pk) {
              mark[id] = stamp;
              cur[n++] = id;
            }
          }
        }
        int32_t n_fresh = k - n;
        int32_t n_zipf = j->cdf ? (int32_t)floor(p->zipf_frac * (double)n_fresh) : 0;
        for (int32_t i = 0; i < n_zipf; ++i) {
          int64_t tries = 0;
          int32_t id;
          do {
            if (++tries > MAX_TRIES) { j->status = -3; free(mark); return NULL; }
            id = L - zipf_rank(j->cdf, L, to_unit(draw(key, ctr++)));
          } while (mark[id] == stamp);
          mark[id] = stamp;
          cur[n++] = id;
        }
        while (n < k) {
          int64_t tries = 0;
          int32_t id;
          do {
            if (++tries > MAX_TRIES) { j->status = -3; free(mark); return NULL; }
            id = (int32_t)(to_unit(draw(key, ctr++)) * (double)L);
          } while (mark[id] == stamp);
          mark[id] = stamp;
          cur[n++] = id;
        }
        for (int32_t i = k - 1; i > 0; --i) {
          int32_t r = (int32_t)(to_unit(draw(key, ctr++)) * (double)(i + 1));
          int32_t tmp = cur[i]; cur[i] = cur[r]; cur[r] = tmp;
        }
        prev = cur;
      }
    }
  }
  free(mark);
  return NULL;
}

/* Selections out[steps][units][tokens][k] (int32). Returns 0, or <0 on a bad
 * parameter (-1), allocation failure (-2) or a redraw loop that ran out (-3). */
int gen_selections(int32_t* out, const sel_params* p, int nthreads) {
  if (!out || !p || p->units < 0 || p->num_entries <= 0 || p->k < 0 ||
      p->k > p->num_entries || p->steps < 0 || p->tokens < 1 || p->num_forced < 0 ||
      p->unit_base < 0 ||
      (p->num_forced > 0 && !p->forced))
    return -1;
  if (p->units == 0 || p->steps == 0 || p->k == 0) return 0;
  double* cdf = NULL;
  if (p->zipf_frac > 0.0) {
    const int32_t L = p->num_entries;
    cdf = (double*)malloc((size_t)L * sizeof(double));
    if (!cdf) return -2;
    double acc = 0.0;
    for (int32_t r = 1; r <= L; ++r) { acc += pow((double)r, -p->zipf_s); cdf[r - 1] = acc; }
    for (int32_t r = 0; r < L; ++r) cdf[r] /= acc;
    cdf[L - 1] = 1.0;
  }
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (nthreads > p->units) nthreads = p->units;
  pthread_t th[256];
  sel_job jobs[256];
  int32_t per = (p->units + nthreads - 1) / nthreads;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    int32_t b = t * per, e = b + per;
    if (b >= p->units) break;
    if (e > p->units) e = p->units;
    jobs[t] = (sel_job){p, out, cdf, b, e, 0};
    if (pthread_create(&th[t], NULL, sel_worker, &jobs[t]) != 0) {
      sel_worker(&jobs[t]);
      th[t] = 0;
    }
    started = t + 1;
  }
  int status = 0;
  for (int t = 0; t < started; ++t) {
    if (th[t]) pthread_join(th[t], NULL);
    if (jobs[t].status) status = jobs[t].status;
  }
  free(cdf);
  return status;
}
