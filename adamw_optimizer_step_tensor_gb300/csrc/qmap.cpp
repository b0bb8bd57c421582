// qmap.cpp -- host construction of the 8-bit and 4-bit code maps and of the
// tables the kernels use to find the nearest code.
//
// Default maps: dynamic-exponent quantisation as described by Dettmers et
// al., "8-bit Optimizers via Block-wise Quantization" (arXiv:2110.02861):
// after the sign bit, E zero bits select the decade 10^-E, a one bit closes
// the run, and the remaining F bits split [0.1, 1] into 2^F equal bins whose
// centres are the representable fractions.  Signed map (first moment):
// E = 0..6, F = 6 - E, both signs; unsigned map (second moment): the sign bit
// becomes a fraction bit, F = 7 - E.  Both add exact 0 and +1.0, giving 256
// values each, stored ascending (the code of a value is its index).
//
// Each value is the rational (2n + 18k + 9) / (20 n 10^E) with n = 2^F, bin k,
// rounded once to the nearest float32 with integer arithmetic only.
//
// 4-bit maps (the format of Li, Chen, Zhu, "Memory Efficient Optimizers with
// 4-bit States", as torchao's 4-bit AdamW uses it): the first moment on the
// same tree with three magnitude bits (E = 0..2, F = 2 - E, both signs, plus
// 0 and +1.0: 16 values), the second moment on k/16, k = 1..16 (no zero).
#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <vector>

#include "internal.h"

namespace adamw {
namespace {

// Nearest float32 (ties to even) of num / (p5 * 2^k), num > 0, result normal.
float round_ratio(uint64_t num, uint64_t p5, int k) {
  int s = 0;
  while (((num << s) / p5) < (1ull << 25)) ++s;       // quotient gets 26 bits
  const uint64_t n = num << s;
  const uint64_t q = n / p5, r = n % p5;
  uint64_t keep = q >> 2;                               // 24 significant bits
  const uint64_t rb = q & 3u;
  if (rb > 2u || (rb == 2u && (r != 0u || (keep & 1u)))) ++keep;
  return std::ldexp(static_cast<float>(keep), 2 - s - k);
}

void dynamic_map(int frac_bits_e0, bool is_signed, int n_exp, int size, float* out) {
  std::vector<float> v = {0.0f, 1.0f};
  uint64_t p5 = 5;                                      // 5^(E+1)
  for (int e = 0; e < n_exp; ++e, p5 *= 5) {
    const int f = frac_bits_e0 - e;
    const uint64_t n = 1ull << f;
    for (uint64_t b = 0; b < n; ++b) {
      // (2n + 18b + 9) / (20 n 10^E) = num / (5^(E+1) * 2^(2 + F + E))
      const float x = round_ratio(2 * n + 18 * b + 9, p5, 2 + f + e);
      v.push_back(x);
      if (is_signed) v.push_back(-x);
    }
  }
  std::sort(v.begin(), v.end());
  std::memcpy(out, v.data(), static_cast<size_t>(size) * sizeof(float));
}

// #{k : thr[k] <= x} over n - 1 ascending thresholds (float comparisons).
int count_le(const float* thr, int n, float x) {
  int c = 0;
  while (c < n - 1 && thr[c] <= x) ++c;
  return c;
}

float bits_to_float(uint32_t b) {
  float f;
  std::memcpy(&f, &b, 4);
  return f;
}

}  // namespace

void default_maps(float smap[256], float umap[256]) {
  dynamic_map(6, true, 7, 256, smap);
  dynamic_map(7, false, 7, 256, umap);
}

void default_maps4(float smap[16], float umap[16]) {
  dynamic_map(2, true, 3, 16, smap);
  for (int k = 0; k < 16; ++k) umap[k] = static_cast<float>(k + 1) / 16.0f;   // exact
}

// Fill one QMapDev from n (16 or 256) ascending finite values.  Returns the
// largest number of thresholds inside one bucket, or -1 if the values are
// unusable.
int build_qmap(const float* value, int n, QMapDev* out) {
  if (n < 2 || n > 256) return -1;
  for (int k = 0; k < n; ++k) {
    if (!std::isfinite(value[k])) return -1;
    if (k > 0 && !(value[k - 1] < value[k])) return -1;
  }
  std::memset(out->value, 0, sizeof(out->value));
  std::memcpy(out->value, value, static_cast<size_t>(n) * sizeof(float));
  // thr[k]: smallest float strictly above the exact midpoint of value[k], value[k+1]
  for (int k = 0; k < n - 1; ++k) {
    const double a = value[k], b = value[k + 1];
    const double s = a + b;
    const double bb = s - a;                            // two-sum: the sum must be exact
    if ((a - (s - bb)) + (b - bb) != 0.0) return -1;
    const double mid = s * 0.5;
    float c = static_cast<float>(mid);
    if (static_cast<double>(c) <= mid) c = std::nextafter(c, INFINITY);
    out->thr[k] = c;
  }
  for (int k = n - 1; k < 256 + kMaxRefine; ++k) out->thr[k] = INFINITY;
  // Normalised values satisfy |x| <= 1, so the last bucket (|x| >= 1.9921875)
  // is reached only by NaN: its lowest code is 0 and, since no threshold
  // compares true against NaN, NaN quantises to code 0.
  int refine = 0;
  for (int k = 0; k < kBuckets; ++k) {
    if (k == kBuckets - 1) {
      out->lo_pos[k] = 0;
      out->lo_neg[k] = 0;
      continue;
    }
    uint32_t lo_bits, hi_bits;
    if (k == 0) {
      lo_bits = 0u;
      hi_bits = (103u << 23) - 1u;
    } else {
      const uint32_t e = 103u + static_cast<uint32_t>(k - 1) / 128u;
      const uint32_t mt = static_cast<uint32_t>(k - 1) % 128u;
      lo_bits = (e << 23) | (mt << 16);
      hi_bits = lo_bits | 0xFFFFu;
    }
    const float lo = bits_to_float(lo_bits), hi = bits_to_float(hi_bits);
    const int pos_lo = count_le(out->thr, n, lo), pos_hi = count_le(out->thr, n, hi);
    const int neg_lo = count_le(out->thr, n, -hi), neg_hi = count_le(out->thr, n, -lo);
    out->lo_pos[k] = static_cast<uint8_t>(pos_lo);
    out->lo_neg[k] = static_cast<uint8_t>(neg_lo);
    refine = std::max(refine, std::max(pos_hi - pos_lo, neg_hi - neg_lo));
  }
  return refine;
}

int zero_code_of(const float* value, int n) {
  for (int k = 0; k < n; ++k)
    if (value[k] == 0.0f) return k;
  return -1;
}

}  // namespace adamw
