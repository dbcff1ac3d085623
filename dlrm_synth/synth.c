/*
 * Seeded synthetic inputs for the DLRMv1 forward: counter-based, parallel and
 * reproducible on any host.
 *
 * This file holds only random-number generation. It contains none of the
 * forward's arithmetic (no gather, no dot, no GEMM, no activation), so both the
 * CUDA path's tests and the CPU oracle may consume what it produces.
 *
 * Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014). Element i of stream (seed, stream_id) is
 * mix64(key + (i + 1) * GAMMA), i.e. the i-th output of a SplitMix64 sequence
 * whose state starts at key(seed, stream_id). Any element is computable on its
 * own, so every thread fills its own slice.
 *
 * Distributions:
 *   uniform f32   lo + (hi - lo) * u,  u = top 24 bits * 2^-24 in [0, 1)
 *   normal f32    Box-Muller on elements 2i (u1 in (0,1]) and 2i+1 (u2 in [0,1))
 *   uniform int   floor(u32 * V / 2^32), u32 = top 32 bits, V < 2^32
 *   zipf int      truncated Zipf over ranks 1..V, P(k) ~ k^-s; inverse CDF by
 *                 binary search; rank k is row k-1.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64(mix64(seed ^ 0x243F6A8885A308D3ULL) + stream * GAMMA);
}

static inline uint64_t element(uint64_t key, uint64_t i) {
  return mix64(key + (i + 1) * GAMMA);
}

uint64_t synth_element(uint64_t seed, uint64_t stream, uint64_t i) {
  return element(stream_key(seed, stream), i);
}

/* Element i of the plain SplitMix64 sequence whose state starts at `key`. */
uint64_t synth_raw(uint64_t key, uint64_t i) { return element(key, i); }

typedef struct {
  int kind; /* 0 uniform f32, 1 normal f32, 2 uniform int, 3 zipf int */
  void* out;
  int64_t begin, end;
  uint64_t key;
  double lo, hi;
  int64_t v;
  const double* cdf;
} job_t;

static void* run_job(void* arg) {
  job_t* j = (job_t*)arg;
  const double two_pi = 6.283185307179586476925286766559;
  for (int64_t i = j->begin; i < j->end; ++i) {
    switch (j->kind) {
      case 0: {
        double u = (double)(element(j->key, (uint64_t)i) >> 40) * (1.0 / 16777216.0);
        ((float*)j->out)[i] = (float)(j->lo + (j->hi - j->lo) * u);
        break;
      }
      case 1: {
        uint64_t a = element(j->key, 2 * (uint64_t)i);
        uint64_t b = element(j->key, 2 * (uint64_t)i + 1);
        double u1 = (double)((a >> 11) + 1) * (1.0 / 9007199254740992.0);
        double u2 = (double)(b >> 11) * (1.0 / 9007199254740992.0);
        ((float*)j->out)[i] = (float)(sqrt(-2.0 * log(u1)) * cos(two_pi * u2));
        break;
      }
      case 2: {
        uint64_t u32 = element(j->key, (uint64_t)i) >> 32;
        ((int64_t*)j->out)[i] = (int64_t)((u32 * (uint64_t)j->v) >> 32);
        break;
      }
      case 3: {
        double u = (double)(element(j->key, (uint64_t)i) >> 11) * (1.0 / 9007199254740992.0);
        /* first k with cdf[k] > u */
        int64_t lo = 0, hi = j->v - 1;
        while (lo < hi) {
          int64_t mid = lo + (hi - lo) / 2;
          if (j->cdf[mid] > u) hi = mid; else lo = mid + 1;
        }
        ((int64_t*)j->out)[i] = lo;
        break;
      }
    }
  }
  return NULL;
}

static int run_parallel(job_t proto, int64_t n, int threads) {
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  if (n < 65536) threads = 1;
  pthread_t tid[256];
  job_t jobs[256];
  int64_t chunk = (n + threads - 1) / threads;
  int started = 0;
  for (int t = 0; t < threads; ++t) {
    jobs[t] = proto;
    jobs[t].begin = (int64_t)t * chunk;
    jobs[t].end = jobs[t].begin + chunk < n ? jobs[t].begin + chunk : n;
    if (jobs[t].begin >= jobs[t].end) break;
    if (threads == 1) { run_job(&jobs[t]); continue; }
    if (pthread_create(&tid[t], NULL, run_job, &jobs[t]) != 0) return -1;
    ++started;
  }
  for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
  return 0;
}

int synth_uniform_f32(float* out, int64_t n, uint64_t seed, uint64_t stream, double lo,
                      double hi, int threads) {
  job_t p = {0, out, 0, 0, stream_key(seed, stream), lo, hi, 0, NULL};
  return run_parallel(p, n, threads);
}

int synth_normal_f32(float* out, int64_t n, uint64_t seed, uint64_t stream, int threads) {
  job_t p = {1, out, 0, 0, stream_key(seed, stream), 0, 0, 0, NULL};
  return run_parallel(p, n, threads);
}

int synth_uniform_i64(int64_t* out, int64_t n, uint64_t seed, uint64_t stream, int64_t v,
                      int threads) {
  if (v <= 0 || v > 0xFFFFFFFFLL) return -2;
  job_t p = {2, out, 0, 0, stream_key(seed, stream), 0, 0, v, NULL};
  return run_parallel(p, n, threads);
}

/* cdf: caller-owned buffer of v doubles, filled here (cdf[k] = P(rank <= k+1)). */
int synth_zipf_cdf(double* cdf, int64_t v, double s) {
  if (v <= 0) return -2;
  double acc = 0.0;
  for (int64_t k = 0; k < v; ++k) {
    acc += pow((double)(k + 1), -s);
    cdf[k] = acc;
  }
  for (int64_t k = 0; k < v; ++k) cdf[k] /= acc;
  cdf[v - 1] = 1.0;
  return 0;
}

int synth_zipf_i64(int64_t* out, int64_t n, uint64_t seed, uint64_t stream,
                   const double* cdf, int64_t v, int threads) {
  if (v <= 0) return -2;
  job_t p = {3, out, 0, 0, stream_key(seed, stream), 0, 0, v, cdf};
  return run_parallel(p, n, threads);
}
