/*
 * Seeded synthetic input generator shared by the FP64 oracle tests and the CUDA
 * path's tests and benchmark.  It holds none of the attention method's arithmetic:
 * it only turns (seed, stream, index) into integers, uniforms, N(0,1) draws and
 * their bf16 roundings.
 *
 * Definition (counter-based, so every element can be drawn independently):
 *   mix64(z)            the splitmix64 output finaliser (Steele, Lea & Flood,
 *                       "Fast splittable pseudorandom number generators", 2014):
 *                       z ^= z>>30; z *= 0xBF58476D1CE4E5B9;
 *                       z ^= z>>27; z *= 0x94D049BB133111EB; z ^= z>>31
 *   base(seed, stream)  mix64(seed ^ mix64(stream + 0x632BE59BD9B4E019))
 *   draw(seed,stream,i) mix64(base + (i+1) * 0x9E3779B97F4A7C15)
 *   uniform(x)          (x >> 11) * 2^-53, in [0, 1)
 *   normal pair k       u1 = uniform(draw(2k)), u2 = uniform(draw(2k+1));
 *                       rad = sqrt(-2 ln(1-u1));
 *                       z[2k] = rad cos(2 pi u2), z[2k+1] = rad sin(2 pi u2)
 *                       (Box & Muller, 1958)
 *   bf16(x)             round x to binary32 (nearest-even), then to bfloat16
 *                       (nearest-even on the upper 16 bits)
 *   randint(lo,hi,i)    lo + draw(i) mod (hi-lo+1)
 *
 * The Python module synth/__init__.py restates the same definition in numpy for
 * small sizes; a test checks the two agree bit for bit.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  z ^= z >> 31;
  return z;
}

static inline uint64_t stream_base(uint64_t seed, uint64_t stream) {
  return mix64(seed ^ mix64(stream + 0x632BE59BD9B4E019ull));
}

static inline uint64_t draw_at(uint64_t base, uint64_t i) {
  return mix64(base + (i + 1) * 0x9E3779B97F4A7C15ull);
}

static inline double uniform01(uint64_t x) { return (double)(x >> 11) * 0x1.0p-53; }

static inline uint16_t bf16_rne(double x) {
  float f = (float)x;
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* n raw 64-bit draws */
void synth_draws(uint64_t seed, uint64_t stream, int64_t n, uint64_t* out) {
  uint64_t b = stream_base(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = draw_at(b, (uint64_t)i);
}

/* n integers uniform on [lo, hi] */
void synth_randint(uint64_t seed, uint64_t stream, int64_t n, int64_t lo, int64_t hi, int64_t* out) {
  uint64_t b = stream_base(seed, stream);
  uint64_t span = (uint64_t)(hi - lo + 1);
  for (int64_t i = 0; i < n; ++i) out[i] = lo + (int64_t)(draw_at(b, (uint64_t)i) % span);
}

/* n uniforms on [0, 1) */
void synth_uniform(uint64_t seed, uint64_t stream, int64_t n, double* out) {
  uint64_t b = stream_base(seed, stream);
  for (int64_t i = 0; i < n; ++i) out[i] = uniform01(draw_at(b, (uint64_t)i));
}

/*
 * n bf16 values x[i] = bf16(s * z[i]) with z ~ N(0,1).  When head_scale is not
 * NULL the element index i is read as the flat index of a [T][heads][head_dim]
 * tensor and s = head_scale[(i / head_dim) % heads]; otherwise s = 1.
 */
void synth_normal_bf16(uint64_t seed, uint64_t stream, int64_t n, const double* head_scale,
                       int64_t heads, int64_t head_dim, uint16_t* out) {
  uint64_t b = stream_base(seed, stream);
  int64_t npairs = (n + 1) / 2;
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < npairs; ++k) {
    double u1 = uniform01(draw_at(b, (uint64_t)(2 * k)));
    double u2 = uniform01(draw_at(b, (uint64_t)(2 * k + 1)));
    double rad = sqrt(-2.0 * log(1.0 - u1));
    double ang = 2.0 * M_PI * u2;
    double z[2] = {rad * cos(ang), rad * sin(ang)};
    for (int t = 0; t < 2; ++t) {
      int64_t i = 2 * k + t;
      if (i >= n) break;
      double s = head_scale ? head_scale[(i / head_dim) % heads] : 1.0;
      out[i] = bf16_rne(s * z[t]);
    }
  }
}

/* the same normals in double, unrounded (used only to pin the bf16 rounding) */
void synth_normal_f64(uint64_t seed, uint64_t stream, int64_t n, double* out) {
  uint64_t b = stream_base(seed, stream);
  int64_t npairs = (n + 1) / 2;
  for (int64_t k = 0; k < npairs; ++k) {
    double u1 = uniform01(draw_at(b, (uint64_t)(2 * k)));
    double u2 = uniform01(draw_at(b, (uint64_t)(2 * k + 1)));
    double rad = sqrt(-2.0 * log(1.0 - u1));
    double ang = 2.0 * M_PI * u2;
    out[2 * k] = rad * cos(ang);
    if (2 * k + 1 < n) out[2 * k + 1] = rad * sin(ang);
  }
}
