// Seeded synthetic-input generator shared by the oracle tests, the GPU tests and the bench.
//
// It holds none of the attention / scoring / selection arithmetic: it only turns
// (seed, stream tag, element index) into numbers.  Every element is a pure function of
// its index (counter-based), so any sub-range of a tensor can be regenerated on its own
// and the work splits across threads without changing a single bit of the output.
//
// Generators used, by their published definitions:
//   * SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number generators",
//     OOPSLA 2014; constants as in Vigna's public reference code).  Output number i of a
//     stream whose state starts at s0 is mix(s0 + (i + 1) * golden), so the i-th output is
//     computed directly from i.
//   * Box-Muller (1958) for standard normals, in fp64 with libm log/sqrt/cos/sin.
//   * bf16 = IEEE binary32 rounded to its upper 16 bits with round-to-nearest-even,
//     written here from the definition of the format (value -> fp32 by a C cast, which
//     rounds to nearest even, then fp32 -> bf16 by RNE on the bit pattern).
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>
#include <algorithm>

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

inline uint64_t sm64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Initial SplitMix64 state of the stream (seed, tag).
inline uint64_t stream_base(uint64_t seed, uint64_t tag) {
  return sm64_mix(seed + kGolden * (tag + 1)) ^ sm64_mix(tag * 0xD1B54A32D192ED03ull + 0x1234567ull);
}

// i-th raw 64-bit output of the stream.
inline uint64_t raw(uint64_t base, uint64_t i) { return sm64_mix(base + kGolden * (i + 1)); }

// Uniform in the open interval (0, 1) from the top 53 bits.
inline double unif(uint64_t base, uint64_t i) {
  return (static_cast<double>(raw(base, i) >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

// Standard normal number i of the stream: pair j = i / 2 uses uniforms 2j and 2j+1.
inline double normal(uint64_t base, uint64_t i) {
  const uint64_t j = i >> 1;
  const double u1 = unif(base, 2 * j), u2 = unif(base, 2 * j + 1);
  const double r = std::sqrt(-2.0 * std::log(u1));
  const double a = 6.283185307179586476925286766559 * u2;
  return (i & 1) ? r * std::sin(a) : r * std::cos(a);
}

inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return static_cast<uint16_t>(u >> 16);  // inf/nan: keep
  const uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return static_cast<uint16_t>(u >> 16);
}

template <class F>
void parallel_for(int64_t n, int nthreads, F f) {
  if (nthreads <= 0) nthreads = static_cast<int>(std::max(1u, std::thread::hardware_concurrency()));
  const int64_t min_chunk = 1 << 16;
  int64_t nt = std::min<int64_t>(nthreads, std::max<int64_t>(1, n / min_chunk));
  if (nt <= 1) { f(0, n); return; }
  std::vector<std::thread> th;
  for (int64_t t = 0; t < nt; ++t) {
    const int64_t lo = n * t / nt, hi = n * (t + 1) / nt;
    th.emplace_back([=] { f(lo, hi); });
  }
  for (auto& x : th) x.join();
}

}  // namespace

extern "C" {

// Raw uniforms in (0,1), elements [offset, offset + n) of stream (seed, tag).
void gen_uniform_f64(uint64_t seed, uint64_t tag, int64_t offset, int64_t n, double* out, int nthreads) {
  const uint64_t b = stream_base(seed, tag);
  parallel_for(n, nthreads, [&](int64_t lo, int64_t hi) {
    for (int64_t i = lo; i < hi; ++i) out[i] = unif(b, static_cast<uint64_t>(offset + i));
  });
}

// Standard normals times `scale`, as fp32, elements [offset, offset + n).
void gen_normal_f32(uint64_t seed, uint64_t tag, int64_t offset, int64_t n, double scale, float* out,
                    int nthreads) {
  const uint64_t b = stream_base(seed, tag);
  parallel_for(n, nthreads, [&](int64_t lo, int64_t hi) {
    for (int64_t i = lo; i < hi; ++i)
      out[i] = static_cast<float>(scale * normal(b, static_cast<uint64_t>(offset + i)));
  });
}

// Standard normals as fp64, elements [offset, offset + n).
void gen_normal_f64(uint64_t seed, uint64_t tag, int64_t offset, int64_t n, double* out, int nthreads) {
  const uint64_t b = stream_base(seed, tag);
  parallel_for(n, nthreads, [&](int64_t lo, int64_t hi) {
    for (int64_t i = lo; i < hi; ++i) out[i] = normal(b, static_cast<uint64_t>(offset + i));
  });
}

// Rows of `row_len` standard normals rounded to bf16 (returned as raw uint16 bits).
// Rows [row_offset, row_offset + n_rows) of stream (seed, tag).  When outlier_p > 0 each
// row is multiplied by outlier_scale with probability outlier_p, decided by uniform
// number `row` of the companion stream (seed, tag ^ 0x5A5A5A5A); the product is formed in
// fp64 before rounding.
void gen_rows_bf16(uint64_t seed, uint64_t tag, int64_t row_offset, int64_t n_rows, int row_len,
                   double outlier_p, double outlier_scale, uint16_t* out, int nthreads) {
  const uint64_t b = stream_base(seed, tag);
  const uint64_t bo = stream_base(seed, tag ^ 0x5A5A5A5Aull);
  parallel_for(n_rows, nthreads, [&](int64_t lo, int64_t hi) {
    for (int64_t r = lo; r < hi; ++r) {
      const uint64_t row = static_cast<uint64_t>(row_offset + r);
      double s = 1.0;
      if (outlier_p > 0.0 && unif(bo, row) < outlier_p) s = outlier_scale;
      uint16_t* o = out + r * row_len;
      const uint64_t e0 = row * static_cast<uint64_t>(row_len);
      for (int d = 0; d < row_len; ++d)
        o[d] = f32_to_bf16_rne(static_cast<float>(s * normal(b, e0 + d)));
    }
  });
}

// Converts fp32 values to bf16 bits with round-to-nearest-even (used to round a
// random-walk master copy of an input to the bf16 the kernels read).
void gen_f32_to_bf16(const float* in, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_rne(in[i]);
}

}  // extern "C"
