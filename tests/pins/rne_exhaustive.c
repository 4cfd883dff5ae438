/*
 * Pin for the oracle's fp16 rounding: compare tg_oracle_f32_to_f16 with the host compiler's
 * own binary32 -> _Float16 conversion (libgcc's correctly rounded soft-float routine) over
 * every one of the 2^32 binary32 bit patterns, and tg_oracle_f64_to_f16 with the compiler's
 * binary64 -> _Float16 conversion over a pseudo-random sweep plus constructed near-tie values.
 * NaNs only have to agree on being NaN (payloads are not part of the rounding rule).
 *
 * Usage: rne_exhaustive [stride]   (stride 1 = exhaustive)   exit 0 = all equal
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

uint16_t tg_oracle_f32_to_f16(float x);
uint16_t tg_oracle_f64_to_f16(double x);

static int same(uint16_t a, uint16_t b) {
  int an = ((a & 0x7C00) == 0x7C00) && (a & 0x3FF);
  int bn = ((b & 0x7C00) == 0x7C00) && (b & 0x3FF);
  if (an || bn) return an && bn;
  return a == b;
}

static uint16_t ref16(_Float16 h) {
  uint16_t b;
  memcpy(&b, &h, 2);
  return b;
}

int main(int argc, char** argv) {
  uint64_t stride = argc > 1 ? strtoull(argv[1], NULL, 10) : 1;
  if (stride == 0) stride = 1;
  long long bad32 = 0, bad64 = 0;
#pragma omp parallel for reduction(+ : bad32) schedule(static)
  for (int64_t hi = 0; hi < 65536; ++hi) {
    for (uint64_t lo = 0; lo < 65536; lo += stride) {
      uint32_t u = (uint32_t)((hi << 16) | lo);
      float f;
      memcpy(&f, &u, 4);
      uint16_t got = tg_oracle_f32_to_f16(f);
      uint16_t want = ref16((_Float16)f);
      if (!same(got, want)) {
        if (bad32 < 5)
#pragma omp critical
          fprintf(stderr, "f32 0x%08x: oracle 0x%04x compiler 0x%04x\n", u, got, want);
        bad32++;
      }
    }
  }
  /* binary64: random bit patterns restricted to the interesting exponent band, plus every
     fp16 midpoint +- a few ulps of binary64 */
  uint64_t s = 0x243F6A8885A308D3ull;
  for (long i = 0; i < 20000000; ++i) {
    s ^= s << 13; s ^= s >> 7; s ^= s << 17;
    uint64_t exp = 1023 - 30 + (s >> 58);           /* 2^-30 .. 2^33 */
    uint64_t bits = (s & 0x800FFFFFFFFFFFFFull) | (exp << 52);
    double d;
    memcpy(&d, &bits, 8);
    if (!same(tg_oracle_f64_to_f16(d), ref16((_Float16)d))) {
      if (bad64 < 5) fprintf(stderr, "f64 %a mismatch\n", d);
      bad64++;
    }
  }
  for (uint32_t h = 0; h < 0x7C00; ++h) {
    /* midpoint between h and h+1 (positive), and around it */
    uint16_t a = (uint16_t)h, b = (uint16_t)(h + 1);
    _Float16 ha, hb;
    memcpy(&ha, &a, 2);
    memcpy(&hb, &b, 2);
    double mid = ((double)ha + (double)hb) / 2.0;
    double probes[5] = {mid, nextafter(mid, 0.0), nextafter(mid, INFINITY),
                        nextafter(nextafter(mid, 0.0), 0.0), -mid};
    for (int p = 0; p < 5; ++p) {
      if (!same(tg_oracle_f64_to_f16(probes[p]), ref16((_Float16)probes[p]))) {
        if (bad64 < 10) fprintf(stderr, "f64 probe %a mismatch\n", probes[p]);
        bad64++;
      }
    }
  }
  printf("mismatches f32=%lld f64=%lld\n", bad32, bad64);
  return (bad32 || bad64) ? 1 : 0;
}
