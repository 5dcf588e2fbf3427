// softhalf.h -- host-side software FP16 / BF16 arithmetic for the fitter.
//
// The fitter scores candidate programs by replaying them on the CPU with the
// rounding the GPU applies ("Fast Polynomial Transcendentals for LLMs",
// §3.2 steps 3-5 and the deployed packed-FMA order of Fig. 2c).  This file
// implements that rounding with integer arithmetic: an operand is an integer
// significand times a power of two; a fused multiply-add forms the exact sum
// in a 128-bit integer (operands far below the result's last bit collapse to
// a sticky bit) and rounds once, to nearest with ties to even, keeping
// subnormals, overflowing to infinity, and producing 0x7FFF for NaN results.
#pragma once

#include <cmath>
#include <cstdint>
#include <cstring>

namespace polyact {

struct HalfFormat {
  int frac_bits;   // stored significand bits (10 FP16, 7 BF16)
  int exp_bits;    // 5 FP16, 8 BF16
  int bias;        // 15, 127
  uint16_t inf_bits() const { return (uint16_t)(((1u << exp_bits) - 1u) << frac_bits); }
  int emax_field() const { return (1 << exp_bits) - 1; }
  int min_exp() const { return 1 - bias - frac_bits; }   // exponent of the subnormal quantum
};

inline HalfFormat half_format(int dtype) {
  return dtype == 0 ? HalfFormat{10, 5, 15} : HalfFormat{7, 8, 127};
}

constexpr uint16_t kQuietNaN = 0x7FFF;

// Unpacked finite value: (-1)^neg * sig * 2^exp, sig an integer.
struct Unpacked {
  bool neg;
  bool nan;
  bool inf;
  uint64_t sig;
  int exp;
};

inline Unpacked unpack(uint16_t b, const HalfFormat &f) {
  Unpacked u{};
  u.neg = (b >> 15) & 1;
  int e = (b >> f.frac_bits) & f.emax_field();
  uint64_t m = b & ((1u << f.frac_bits) - 1u);
  if (e == f.emax_field()) {
    u.nan = m != 0;
    u.inf = m == 0;
    return u;
  }
  if (e == 0) {
    u.sig = m;
    u.exp = f.min_exp();
  } else {
    u.sig = m | (1ull << f.frac_bits);
    u.exp = e - f.bias - f.frac_bits;
  }
  return u;
}

inline int bit_length(unsigned __int128 v) {
  const uint64_t hi = (uint64_t)(v >> 64), lo = (uint64_t)v;
  if (hi) return 128 - __builtin_clzll(hi);
  if (lo) return 64 - __builtin_clzll(lo);
  return 0;
}

// Round (-1)^neg * (mag + s) * 2^exp to the format, where 0 <= s < 1 is an
// unknown fraction that is non-zero iff `sticky`.  Requires that, whenever
// `sticky` is set, the result's last kept bit lies at least two bits above
// the units of `mag` (the caller guarantees this by aligning with headroom).
inline uint16_t round_pack(bool neg, unsigned __int128 mag, int exp, bool sticky,
                           const HalfFormat &f) {
  const uint16_t sign = neg ? 0x8000 : 0;
  if (mag == 0 && !sticky) return sign;
  const int p = f.frac_bits + 1;
  int top = exp + bit_length(mag) - 1;             // exponent of the leading bit
  int qexp = top - (p - 1);                        // exponent of the last kept bit
  if (qexp < f.min_exp()) qexp = f.min_exp();      // subnormal range: fixed quantum
  int shift = qexp - exp;
  unsigned __int128 q;
  if (shift <= 0) {
    q = mag << (-shift);                           // exact (sticky cannot be set here)
  } else if (shift - 1 >= bit_length(mag)) {
    q = 0;                                         // below half the quantum: to zero
  } else {
    unsigned __int128 rem = mag & ((((unsigned __int128)1) << shift) - 1);
    q = mag >> shift;
    unsigned __int128 halfway = ((unsigned __int128)1) << (shift - 1);
    bool up = rem > halfway || (rem == halfway && (sticky || (q & 1)));
    if (up) q += 1;
  }
  if (q == 0) return sign;
  if (q >> p) {                                    // carried into the next binade
    q >>= 1;
    qexp += 1;
  }
  int field;
  uint64_t frac;
  if (q >> (p - 1)) {
    field = qexp + (p - 1) + f.bias;
    frac = (uint64_t)q - (1ull << (p - 1));
  } else {
    field = 0;
    frac = (uint64_t)q;
  }
  if (field >= f.emax_field()) return sign | f.inf_bits();
  return (uint16_t)(sign | (field << f.frac_bits) | frac);
}

// a * b + c, one rounding.
inline uint16_t soft_fma(uint16_t a, uint16_t b, uint16_t c, int dtype) {
  const HalfFormat f = half_format(dtype);
  Unpacked A = unpack(a, f), B = unpack(b, f), C = unpack(c, f);
  if (A.nan || B.nan || C.nan) return kQuietNaN;
  bool pneg = A.neg != B.neg;
  if (A.inf || B.inf) {
    if ((!A.inf && A.sig == 0) || (!B.inf && B.sig == 0)) return kQuietNaN;  // inf * 0
    if (C.inf && C.neg != pneg) return kQuietNaN;                             // inf - inf
    return (pneg ? 0x8000 : 0) | f.inf_bits();
  }
  if (C.inf) return (C.neg ? 0x8000 : 0) | f.inf_bits();
  uint64_t psig = A.sig * B.sig;
  int pexp = A.exp + B.exp;
  if (psig == 0 && C.sig == 0) {
    // exact zero sum: -0 only when both addends are -0
    return (pneg && C.neg) ? 0x8000 : 0;
  }
  if (psig == 0) return c;                                        // 0 + c = c exactly
  if (C.sig == 0) return round_pack(pneg, psig, pexp, false, f);  // product alone
  // Align both addends to a common exponent with 100 bits of headroom below
  // the larger one; anything below that becomes a sticky bit.
  int hi_exp = pexp > C.exp ? pexp : C.exp;
  int base = hi_exp - 100;
  auto place = [&](uint64_t sig, int e, bool &lost) -> unsigned __int128 {
    if (e >= base) return ((unsigned __int128)sig) << (e - base);
    int sh = base - e;
    if (sh >= 64) {
      lost = sig != 0;
      return 0;
    }
    lost = (sig & ((1ull << sh) - 1)) != 0;
    return (unsigned __int128)(sig >> sh);
  };
  bool lost_p = false, lost_c = false;
  unsigned __int128 P = place(psig, pexp, lost_p);
  unsigned __int128 Cc = place(C.sig, C.exp, lost_c);
  bool sticky = lost_p || lost_c;       // at most one of them can lose bits
  if (pneg == C.neg) return round_pack(pneg, P + Cc, base, sticky, f);
  // opposite signs: magnitude difference; a truncated operand is the smaller
  // one, so the exact magnitude is (big - small_trunc) - frac, i.e.
  // (big - small_trunc - 1) + (1 - frac) when bits were lost.
  bool p_big = P > Cc || (P == Cc && !lost_p);
  unsigned __int128 big = p_big ? P : Cc, small = p_big ? Cc : P;
  bool neg = p_big ? pneg : C.neg;
  if (big == small && !sticky) return 0;                           // exact cancellation: +0
  unsigned __int128 d = big - small;
  if (sticky) d -= 1;
  return round_pack(neg, d, base, sticky, f);
}

inline uint16_t soft_mul(uint16_t a, uint16_t b, int dtype) {
  return soft_fma(a, b, 0x8000, dtype);   // a*b + (-0) == a*b, signed zeros kept
}

inline uint16_t soft_add(uint16_t a, uint16_t b, int dtype) {
  return soft_fma(a, dtype == 0 ? 0x3C00 : 0x3F80, b, dtype);   // a*1 + b
}

// Round a double to the format (nearest-even).
inline uint16_t from_double(double x, int dtype) {
  const HalfFormat f = half_format(dtype);
  if (std::isnan(x)) return kQuietNaN;
  bool neg = std::signbit(x);
  if (std::isinf(x)) return (neg ? 0x8000 : 0) | f.inf_bits();
  if (x == 0) return neg ? 0x8000 : 0;
  uint64_t bits;
  std::memcpy(&bits, &x, 8);
  int e = (int)((bits >> 52) & 0x7FF);
  uint64_t m = bits & ((1ull << 52) - 1);
  uint64_t sig;
  int exp;
  if (e == 0) {
    sig = m;
    exp = -1074;
  } else {
    sig = m | (1ull << 52);
    exp = e - 1075;
  }
  // give the rounding two guard bits of headroom (sticky is never needed:
  // the value is exact)
  return round_pack(neg, ((unsigned __int128)sig) << 2, exp - 2, false, f);
}

inline double to_double(uint16_t b, int dtype) {
  const HalfFormat f = half_format(dtype);
  Unpacked u = unpack(b, f);
  if (u.nan) return std::nan("");
  if (u.inf) return u.neg ? -INFINITY : INFINITY;
  double v = std::ldexp((double)u.sig, u.exp);
  return u.neg ? -v : v;
}

inline bool is_nan_bits(uint16_t b, int dtype) {
  const HalfFormat f = half_format(dtype);
  return (b & 0x7FFF) > f.inf_bits();
}

}  // namespace polyact
