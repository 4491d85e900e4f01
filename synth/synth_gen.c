/* Counter-based random draws for the synthetic inputs of the MoE expert block.
 *
 * One generator: the 32-bit MurmurHash3 finaliser (fmix32, Appleby 2011)
 * applied to a key built from (seed, stream, counter).  Nothing here is part
 * of the block's arithmetic; it only produces inputs.
 *
 * Build: gcc -O2 -shared -fPIC -pthread synth_gen.c -o _synth.so
 */
#include <stdint.h>
#include <stddef.h>
#include <pthread.h>

static inline uint32_t fmix32(uint32_t x) {
  x ^= x >> 16;
  x *= 0x85EBCA6Bu;
  x ^= x >> 13;
  x *= 0xC2B2AE35u;
  x ^= x >> 16;
  return x;
}

static inline uint32_t stream_key(uint32_t seed, uint32_t stream) {
  uint32_t k = seed * 0x9E3779B1u + stream * 0x85EBCA77u;
  return fmix32(fmix32(k) ^ stream);
}

static inline uint32_t hash_at(uint32_t key, uint64_t idx) {
  uint32_t lo = (uint32_t)idx, hi = (uint32_t)(idx >> 32);
  return fmix32(fmix32(lo ^ key) ^ (hi * 0x27D4EB2Fu) ^ (key * 7u));
}

/* out[i] = hash(seed, stream, start + i), i < count */
void synth_hash_range(uint32_t seed, uint32_t stream, uint64_t start, uint64_t count, uint32_t* out) {
  uint32_t key = stream_key(seed, stream);
  for (uint64_t i = 0; i < count; ++i) out[i] = hash_at(key, start + i);
}

/* Integers uniform in [-127, 127] for flat positions start .. start+count-1.
 * One hash feeds two consecutive positions (low / high 16 bits); a 16-bit
 * half h becomes ((h * 255) >> 16) - 127. */
typedef struct {
  uint32_t key;
  uint64_t start, begin, end;
  int8_t* out;
} int8_job_t;

static void* int8_worker(void* p) {
  int8_job_t* j = (int8_job_t*)p;
  for (uint64_t i = j->begin; i < j->end; ++i) {
    uint64_t g = j->start + i;
    uint32_t h = hash_at(j->key, g >> 1);
    uint32_t half = (g & 1) ? (h >> 16) : (h & 0xFFFFu);
    j->out[i] = (int8_t)((int32_t)((half * 255u) >> 16) - 127);
  }
  return NULL;
}

int synth_int8_uniform(uint32_t seed, uint32_t stream, uint64_t start, uint64_t count,
                       int8_t* out, int threads) {
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  if (count < (1u << 20)) threads = 1;
  pthread_t tid[256];
  int joined[256];
  int8_job_t job[256];
  uint32_t key = stream_key(seed, stream);
  uint64_t per = (count + threads - 1) / threads;
  per = (per + 1) & ~(uint64_t)1;
  int launched = 0;
  for (int t = 0; t < threads; ++t) {
    uint64_t b = per * t, e = b + per;
    if (b >= count) break;
    if (e > count) e = count;
    job[t].key = key; job[t].start = start; job[t].begin = b; job[t].end = e; job[t].out = out;
    joined[t] = 0;
    if (pthread_create(&tid[t], NULL, int8_worker, &job[t]) != 0) {
      int8_worker(&job[t]);
      joined[t] = 1;
    }
    launched = t + 1;
  }
  for (int t = 0; t < launched; ++t)
    if (!joined[t]) pthread_join(tid[t], NULL);
  return 0;
}
