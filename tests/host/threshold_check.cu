// Host-side check of the quantizer's decision thresholds (kvq::qthr in kvq_quantizer.cuh).
//
// For many groups -- standard-normal groups, groups with outliers, tiny and subnormal ranges,
// magnitudes up to the fp16 maximum, groups straddling zero -- every fp16 value x between the
// group's minimum and maximum must get the same 2-bit code from the thresholds (the number of
// thresholds x reaches) as from the quantizer's definition, clamp(rint(fl(fl(x - z) / s)), 0, 3),
// computed here with plain IEEE fp32 operations.  Prints "checked N values" and exits 0, or
// prints the first mismatch and exits 1.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "kvq_quantizer.cuh"

using namespace kvq::qthr;

static uint64_t rng_state = 0x9E3779B97F4A7C15ull;
static uint64_t next_u64() {  // splitmix64
  uint64_t z = (rng_state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}
static double uniform() { return (next_u64() >> 11) * (1.0 / 9007199254740992.0); }
static double normal() {
  const double u1 = uniform() + 1e-300, u2 = uniform();
  return std::sqrt(-2.0 * std::log(u1)) * std::cos(6.283185307179586 * u2);
}

static uint32_t exact_code(float x, float z, float s) {
  volatile float d = x - z;
  volatile float q = d / s;
  float r = std::rint(q);
  if (r < 0.0f) r = 0.0f;
  if (r > 3.0f) r = 3.0f;
  return (uint32_t)r;
}

static bool ge16(uint16_t a, uint16_t b) { return half_to_float(a) >= half_to_float(b); }

// div_const<L> against the IEEE division for every significand of one binade and for every
// a < 2^-121 (the quotient q turns subnormal below a = L * 2^-126 < 2^-122); while q is normal the
// computation scales exactly with a power of two of a (the remainder a - q*L is a multiple of
// ulp(q), exact even when subnormal, and the last FMA rounds once), so this covers every finite
// a >= 0.  Returns the values checked.
template <int L>
static long long check_div_const() {
  long long n = 0;
  auto one = [&](uint32_t bits) {
    float a;
    std::memcpy(&a, &bits, 4);
    volatile float want = a / (float)L;
    const float got = div_const<L>(a);
    if (std::memcmp(&got, (const void*)&want, 4) != 0) {
      std::printf("div_const<%d> mismatch: a %a got %a want %a\n", L, a, got, (float)want);
      std::exit(1);
    }
    ++n;
  };
  for (uint32_t m = 0; m < (1u << 23); ++m) one(0x3F800000u | m);        // [1, 2)
  for (uint32_t b = 0; b < (6u << 23); ++b) one(b);                      // 0 .. 2^-121 (subnormals included)
  return n;
}

int main() {
  long long checked = check_div_const<3>() + check_div_const<7>() + check_div_const<15>();
  for (int g = 0; g < 4000; ++g) {
    // a group of 32 fp16 values from one of several distributions
    const int kind = g % 8;
    float v[32];
    for (int i = 0; i < 32; ++i) {
      double x;
      switch (kind) {
        case 0: x = normal(); break;
        case 1: x = (i == 7 ? 40.0 + 5.0 * normal() : normal()); break;
        case 2: x = 1e-6 * normal(); break;                            // subnormal fp16 scales
        case 3: x = 1000.0 + 1e-2 * normal(); break;                     // range far below the magnitude
        case 4: x = 60000.0 * (2.0 * uniform() - 1.0); break;            // up to the fp16 maximum
        case 5: x = -3.0 - std::fabs(normal()); break;                   // all negative
        case 6: x = (uniform() < 0.5 ? 1.0 : -1.0) * std::ldexp(1.0, -(int)(uniform() * 30)); break;
        default: x = normal() * std::ldexp(1.0, (int)(uniform() * 20) - 10); break;
      }
      v[i] = half_to_float(float_to_half((float)x));
    }
    float mn = v[0], mx = v[0];
    for (int i = 1; i < 32; ++i) {
      mn = v[i] < mn ? v[i] : mn;
      mx = v[i] > mx ? v[i] : mx;
    }
    uint32_t t[3];
    const uint32_t zs = thresholds2(mn, mx, t);
    const float z = half_to_float((uint16_t)(zs & 0xFFFFu)), s = half_to_float((uint16_t)(zs >> 16));
    if (!(t[0] <= 0xFFFFu && t[1] <= 0xFFFFu && t[2] <= 0xFFFFu)) return 1;
    // every fp16 value from the minimum to the maximum (value order)
    const int lo = ord(float_to_half(mn)), hi = ord(float_to_half(mx));
    for (int o = lo; o <= hi; ++o) {
      const uint16_t xb = (uint16_t)bits_of(o);
      const float x = half_to_float(xb);
      const uint32_t want = s > 0.0f ? exact_code(x, z, s) : 0u;
      const uint32_t got = (uint32_t)ge16(xb, (uint16_t)t[0]) + (uint32_t)ge16(xb, (uint16_t)t[1]) +
                           (uint32_t)ge16(xb, (uint16_t)t[2]);
      if (got != want) {
        std::printf("mismatch: group %d kind %d mn %a mx %a z %a s %a x %a code %u thresholds give %u (t = %04x %04x %04x)\n",
                    g, kind, mn, mx, z, s, x, want, got, t[0], t[1], t[2]);
        return 1;
      }
      ++checked;
    }
  }
  std::printf("checked %lld values\n", checked);
  return 0;
}
