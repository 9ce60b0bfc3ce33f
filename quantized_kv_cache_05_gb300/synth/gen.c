/* Seeded synthetic inputs for the quantized-KV decode workloads.
 *
 * This module only draws random numbers: it holds none of the method's
 * arithmetic (no quantization, no scales, no attention).  The CUDA library's
 * tests, its benchmark and the CPU oracle all take their inputs from here.
 *
 * Generator: counter-based.  Stream (seed, tensor, purpose) has the key
 *   key = mix64(mix64(seed + GAMMA) ^ (tensor << 32 | purpose))
 * and its i-th 64-bit draw is mix64(key + (i + 1) * GAMMA), where mix64 is
 * the SplitMix64 output function (Steele, Lea, Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014) and GAMMA = 0x9E3779B97F4A7C15.
 * So element i of any tensor is a pure function of (seed, tensor, i) and any
 * slice can be produced on its own.
 *
 * Normal values: from draw r, u1 = ((r >> 40) + 1) * 2^-24 in (0, 1] and
 * u2 = (r & 0xFFFFFF) * 2^-24 in [0, 1); z = sqrt(-2 ln u1) cos(2 pi u2)
 * (Box-Muller, cosine branch), evaluated in double, rounded to float, then
 * optionally multiplied by an outlier factor in float, then rounded to bf16
 * (round to nearest even).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <pthread.h>
#include <stdlib.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t syn_key(uint64_t seed, uint32_t tensor, uint32_t purpose) {
  return mix64(mix64(seed + GAMMA) ^ (((uint64_t)tensor << 32) | (uint64_t)purpose));
}

uint64_t syn_draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GAMMA); }

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t bias = 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)((u + bias) >> 16);
}

static inline float normal_from_draw(uint64_t r) {
  double u1 = (double)((r >> 40) + 1) * (1.0 / 16777216.0);
  double u2 = (double)(r & 0xFFFFFFULL) * (1.0 / 16777216.0);
  double z = sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
  return (float)z;
}

typedef struct {
  uint64_t key_val, key_out;
  uint64_t offset, lo, hi;
  int D;
  const uint8_t* chan_mask;
  float chan_mult, elem_p, elem_mult;
  uint16_t* out;
} fill_job;

static void* fill_worker(void* arg) {
  const fill_job* j = (const fill_job*)arg;
  for (uint64_t i = j->lo; i < j->hi; ++i) {
    uint64_t g = j->offset + i;
    float v = normal_from_draw(syn_draw(j->key_val, g));
    if (j->chan_mask && j->D > 0 && j->chan_mask[g % (uint64_t)j->D]) v = v * j->chan_mult;
    if (j->elem_p > 0.0f) {
      double u = (double)(syn_draw(j->key_out, g) >> 11) * (1.0 / 9007199254740992.0);
      if (u < (double)j->elem_p) v = v * j->elem_mult;
    }
    j->out[i] = f32_to_bf16_rne(v);
  }
  return NULL;
}

/* Fill out[0..n) with elements offset..offset+n of tensor `tensor`:
 *   N(0,1), times chan_mult where chan_mask[(offset+i) % D] != 0 (if given),
 *   times elem_mult with probability elem_p per element (if elem_p > 0). */
void syn_fill_bf16(uint64_t seed, uint32_t tensor, uint64_t offset, uint64_t n, int D,
                   const uint8_t* chan_mask, float chan_mult, float elem_p, float elem_mult,
                   uint16_t* out, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (n < (uint64_t)nthreads * 65536ULL) nthreads = 1;
  fill_job jobs[256];
  pthread_t th[256];
  for (int t = 0; t < nthreads; ++t) {
    fill_job* j = &jobs[t];
    j->key_val = syn_key(seed, tensor, 0);
    j->key_out = syn_key(seed, tensor, 1);
    j->offset = offset;
    j->lo = n * (uint64_t)t / (uint64_t)nthreads;
    j->hi = n * (uint64_t)(t + 1) / (uint64_t)nthreads;
    j->D = D;
    j->chan_mask = chan_mask;
    j->chan_mult = chan_mult;
    j->elem_p = elem_p;
    j->elem_mult = elem_mult;
    j->out = out;
  }
  if (nthreads == 1) {
    fill_worker(&jobs[0]);
    return;
  }
  for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, fill_worker, &jobs[t]);
  for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
}
