/*
 * Threaded generator of synthetic expert weight records.
 *
 * Same generator as synth/__init__.py (splitmix64 as a counter-based stream,
 * Irwin-Hall sum of four 16-bit uniforms scaled in float32, bf16 round to
 * nearest even, FP4 e2m1 codes with e4m3 block scales chosen by nearest value
 * with ties to the even code).  It only produces inputs; none of the MoE
 * layer's arithmetic lives here.  Build with -ffp-contract=off so float
 * operations round exactly like numpy's float32 arithmetic.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { WD_FP32 = 0, WD_BF16 = 1, WD_FP4 = 2 };

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static inline float element(uint64_t base, uint64_t n, float c) {
  uint64_t r = mix64(base + (n + 1) * 0x9E3779B97F4A7C15ull);
  int64_t s = (int64_t)((r & 0xFFFF) + ((r >> 16) & 0xFFFF) + ((r >> 32) & 0xFFFF) + (r >> 48)) - 131070;
  return (float)s * c;
}

static inline uint16_t bf16_rne(float v) {
  uint32_t b;
  memcpy(&b, &v, 4);
  return (uint16_t)((b + 0x7FFFu + ((b >> 16) & 1u)) >> 16);
}

static float e4m3_tab[127];
static pthread_once_t tab_once = PTHREAD_ONCE_INIT;

static void init_tab(void) {
  for (int c = 0; c < 127; ++c) {
    int e = c >> 3, m = c & 7;
    double v;
    if (e == 0) {
      v = (m / 8.0) / 64.0;
    } else {
      v = 1.0 + m / 8.0;
      for (int i = 0; i < e - 7; ++i) v *= 2.0;
      for (int i = 0; i < 7 - e; ++i) v *= 0.5;
    }
    e4m3_tab[c] = (float)v;
  }
}

/* code of the table value nearest to t >= 0, ties to the even code, saturating */
static inline int rne_encode(float t, const float* tab, int n) {
  int last = n - 1;
  int lo = 0, hi = n; /* first index with tab[i] > t */
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (tab[mid] <= t) lo = mid + 1; else hi = mid;
  }
  int c = lo - 1;
  if (c < 0) c = 0;
  if (c >= last) return last;
  float m = (tab[c] + tab[c + 1]) * 0.5f;
  if (t > m || (t == m && (c & 1))) return c + 1;
  return c;
}

/* e2m1 magnitude code nearest to a >= 0: the decision points are the midpoints
 * between neighbouring values {0,.5,1,1.5,2,3,4,6}; a tie goes to the even code. */
static inline int e2m1_rne(float a) {
  return (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) + (a >= 3.5f) + (a > 5.0f);
}

typedef struct {
  uint64_t seed;
  float c;
  int H, I, wdtype;
  int64_t key0, n_keys;
  uint8_t* dst;
  int64_t unit0, unit1; /* units = (key, tensor, row) triples */
} job_t;

static void do_row(const job_t* j, int64_t unit) {
  const int64_t H = j->H, I = j->I, HI = H * I;
  const int64_t rows_per_key = 2 * I + H;
  int64_t kidx = unit / rows_per_key;
  int64_t r = unit % rows_per_key;
  int t, row;
  int64_t K;
  if (r < I) { t = 0; row = (int)r; K = H; }
  else if (r < 2 * I) { t = 1; row = (int)(r - I); K = H; }
  else { t = 2; row = (int)(r - 2 * I); K = I; }
  uint64_t key = (uint64_t)(j->key0 + kidx);
  uint64_t base = mix64((j->seed << 32) ^ key);
  uint64_t n0 = (uint64_t)t * HI + (uint64_t)row * K;
  if (j->wdtype == WD_FP32) {
    int64_t S = 12 * HI;
    float* out = (float*)(j->dst + kidx * S) + n0;
    for (int64_t x = 0; x < K; ++x) out[x] = element(base, n0 + x, j->c);
  } else if (j->wdtype == WD_BF16) {
    int64_t S = 6 * HI;
    uint16_t* out = (uint16_t*)(j->dst + kidx * S) + n0;
    for (int64_t x = 0; x < K; ++x) out[x] = bf16_rne(element(base, n0 + x, j->c));
  } else {
    int64_t S = 3 * HI / 2 + 3 * HI / 16;
    uint8_t* rec = j->dst + kidx * S;
    /* gate codes | up codes | gate scales | up scales | down codes | down scales */
    const int64_t in_t = (int64_t)row * K; /* element offset inside tensor t */
    uint8_t* codes;
    uint8_t* scales;
    if (t < 2) {
      codes = rec + t * (HI / 2) + (in_t >> 1);
      scales = rec + HI + t * (HI / 16) + (in_t >> 4);
    } else {
      codes = rec + HI + HI / 8 + (in_t >> 1);
      scales = rec + HI + HI / 8 + HI / 2 + (in_t >> 4);
    }
    for (int64_t b = 0; b < K / 16; ++b) {
      float v[16];
      float amax = 0.0f;
      for (int x = 0; x < 16; ++x) {
        v[x] = element(base, n0 + b * 16 + x, j->c);
        float a = v[x] < 0 ? -v[x] : v[x];
        if (a > amax) amax = a;
      }
      float tq = amax / 6.0f;
      int sc = rne_encode(tq, e4m3_tab, 127);
      float sv = e4m3_tab[sc];
      scales[b] = (uint8_t)sc;
      for (int x = 0; x < 16; x += 2) {
        uint8_t cd[2];
        for (int h = 0; h < 2; ++h) {
          float w = v[x + h];
          int mag = 0;
          if (sv > 0.0f) {
            float q = w / sv;
            mag = e2m1_rne(q < 0 ? -q : q);
          }
          cd[h] = (uint8_t)(mag | ((w < 0.0f && mag > 0) ? 8 : 0));
        }
        codes[b * 8 + x / 2] = (uint8_t)(cd[0] | (cd[1] << 4));
      }
    }
  }
}

static void* worker(void* arg) {
  const job_t* j = (const job_t*)arg;
  for (int64_t u = j->unit0; u < j->unit1; ++u) do_row(j, u);
  return NULL;
}

/* Fill n_keys records (keys key0 ..) back to back at dst.  Returns 0 on success. */
int synth_records(uint64_t seed, float c, int H, int I, int wdtype, int64_t key0, int64_t n_keys,
                  void* dst, int n_threads) {
  if (H <= 0 || I <= 0 || n_keys < 0 || !dst) return 1;
  if (wdtype == WD_FP4 && ((H % 32) || (I % 32))) return 2;
  if (wdtype < 0 || wdtype > 2) return 3;
  pthread_once(&tab_once, init_tab);
  int64_t units = n_keys * (int64_t)(2 * I + H);
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  if (units < n_threads) n_threads = units > 0 ? (int)units : 1;
  pthread_t th[256];
  job_t jobs[256];
  for (int i = 0; i < n_threads; ++i) {
    jobs[i] = (job_t){seed, c, H, I, wdtype, key0, n_keys, (uint8_t*)dst,
                      units * i / n_threads, units * (i + 1) / n_threads};
  }
  for (int i = 1; i < n_threads; ++i) pthread_create(&th[i], NULL, worker, &jobs[i]);
  worker(&jobs[0]);
  for (int i = 1; i < n_threads; ++i) pthread_join(th[i], NULL);
  return 0;
}
