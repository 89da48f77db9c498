// Exhaustive check of the exponent rules of the power-of-two operand scaling
// (fa_scale.cuh): for every non-negative bf16 magnitude, the exponent of a tensor's
// fp16 copy keeps the largest element finite in fp16 and, when it rescales, puts it
// in [2^14, 2^15); for every combination of the largest |dO|, |V|, |delta| exponents
// and head dims, the dS exponent keeps the worst-case |dS| below fp16's 65504 and, when
// it rescales, above 2^11. Built and run by tests/test_host_scale.py; prints
// "ok <checks>" or the first failure (exit 1).
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include "fa_scale.cuh"

using namespace fa;

static long long checks = 0;
static void fail(const char* what, double a, double b, double c, double d) {
  std::printf("FAIL %s: %.17g %.17g %.17g %.17g\n", what, a, b, c, d);
  std::exit(1);
}

static double bits_value(uint32_t b) {
  float f;
  std::memcpy(&f, &b, 4);
  return (double)f;
}

int main() {
  const double FP16_MAX = 65504.0;
  // every non-negative bf16 magnitude as the tensor's largest |x|
  for (uint32_t h = 0; h < 0x8000u; ++h) {
    const uint32_t bits = h << 16;
    const double amax = bits_value(bits);
    const int e = copy_exponent(bits);
    ++checks;
    if (!std::isfinite(amax) || amax == 0.0) {
      if (e != 0) fail("copy_exponent of zero / inf / nan", amax, e, 0, 0);
      continue;
    }
    const double scaled = std::ldexp(amax, e);
    if (scaled > FP16_MAX) fail("copy overflows fp16", amax, e, scaled, 0);
    if (e == 0) {
      if (!(amax >= 0.25 && amax < 32768.0)) fail("unscaled copy outside its window", amax, e, 0, 0);
    } else if (e > -EXP_LIMIT && e < EXP_LIMIT) {
      if (!(scaled >= 16384.0 && scaled < 32768.0)) fail("rescaled copy not in [2^14, 2^15)", amax, e, scaled, 0);
    } else if (e == EXP_LIMIT) {  // the cap: amax at most lands in [2^14, 2^15)
      if (!(scaled < 32768.0)) fail("capped scale-up above 2^15", amax, e, scaled, 0);
    } else {
      fail("scale-down clamp reached for a bf16 value", amax, e, 0, 0);
    }
  }
  // dS exponent: the largest magnitudes of dO, V (floor exponents fg, fv) and delta (fd)
  for (int dv = 16; dv <= 128; dv += 16) {
    int dlog = 0;
    while ((1 << dlog) < dv) ++dlog;
    for (int fg = -133; fg <= 127; fg += 2)
      for (int fv = -133; fv <= 127; fv += 3)
        for (int fd = -140; fd <= 127; fd += 5) {
          // bf16 values with those floor exponents: the largest is (2 - 2^-7) 2^f
          auto top = [](int f) { return std::ldexp(2.0 - 1.0 / 128, f); };
          auto bot = [](int f) { return std::ldexp(1.0, f); };
          auto bits_of = [](int f) {
            const float v = (float)std::ldexp(1.0, f < -126 ? -126 : f);
            uint32_t b;
            std::memcpy(&b, &v, 4);
            return b;
          };
          if (fg < -126 || fv < -126 || fd < -126) continue;  // (subnormal amax: clamp region)
          const int e = ds_exponent(bits_of(fg), bits_of(fv), bits_of(fd), dlog);
          ++checks;
          const double bmax = dv * top(fg) * top(fv) + top(fd);
          const double bmin = std::fmax(dv * bot(fg) * bot(fv), bot(fd));
          if (std::ldexp(bmax, e) >= 32768.0 && e > -EXP_LIMIT)
            fail("dS bound overflows 2^15", fg, fv, fd, e);
          if (e != 0 && e > -EXP_LIMIT && e < EXP_LIMIT && std::ldexp(bmin, e) < 2048.0)
            fail("rescaled dS bound below 2^11", fg, fv, fd, e);
          if (e == 0 && std::ldexp(bmax, e) >= 32768.0) fail("unscaled dS overflows", fg, fv, fd, e);
        }
  }
  std::printf("ok %lld\n", checks);
  return 0;
}
