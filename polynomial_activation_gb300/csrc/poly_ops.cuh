// poly_ops.cuh -- the polynomial programs as packed-pair operations.
//
// "Fast Polynomial Transcendentals for LLMs" (arXiv 2610.00049):
//   reduction   t = min(|x|, Lc)                          eq. 2 (sign bit cleared,
//               NaN-propagating packed minimum)
//   Horner      v = c_D; v = fma(v, t, c_j), j = D-1 .. 1 (0 for even forms)
//   rebuild     CO  y = fma(v ^ sign(x), t, 1/2)          eq. 3, sign-bit transfer
//               O   y = (v ^ sign(x)) * t                 odd tanh
//               E   y = v                                  even derivatives (§3.3)
//               HX  y = fma(v, t, x * 1/2), and y = max(x, +0) where |x| > Lc
//                                                          eq. 6 with an exact tail
// Each fma / multiply is one packed instruction rounding once (§3.4).
#pragma once

#include "packed.cuh"
#include "stream_kernel.cuh"

namespace polyact {
namespace dev {

template <int DT, int FORM, int D>
__device__ __forceinline__ uint32_t eval_prog(uint32_t x, const DevProg &p) {
  static_assert(D >= 2 && D <= POLY_MAX_DEGREE, "degree");
  const uint32_t a = x & 0x7FFF7FFFu;
  const uint32_t t = pmin_nan<DT>(a, p.lc);
  constexpr int last = FORM == POLY_FORM_E ? 0 : 1;
  uint32_t v = p.c[D];
#pragma unroll
  for (int j = D - 1; j >= last; --j) v = pfma<DT>(v, t, p.c[j]);
  if constexpr (FORM == POLY_FORM_E) {
    return v;
  } else if constexpr (FORM == POLY_FORM_CO) {
    return pfma<DT>(v ^ (x & 0x80008000u), t, half_pair<DT>());
  } else if constexpr (FORM == POLY_FORM_O) {
    return pmul<DT>(v ^ (x & 0x80008000u), t);
  } else {
    const uint32_t h = pmul<DT>(x, half_pair<DT>());
    const uint32_t y = pfma<DT>(v, t, h);
    const uint32_t m = pgt_mask<DT>(a, p.lc);
    const uint32_t r = pmax<DT>(x, 0u);
    return (y & ~m) | (r & m);
  }
}

struct ProgPair {
  DevProg p1, p2;
};

// y = f(x)
template <int DT, int FORM, int D>
struct OpFwd {
  static constexpr int NIN = 1, NOUT = 1;
  static constexpr bool TWO_D = false;
  using Params = ProgPair;
  __device__ __forceinline__ static void pair(const uint32_t (&a)[1], uint32_t (&b)[1],
                                              const Params &p) {
    b[0] = eval_prog<DT, FORM, D>(a[0], p.p1);
  }
};

// dx = dy * f'(x); inputs (x, dy)
template <int DT, int FORM, int D>
struct OpBwd {
  static constexpr int NIN = 2, NOUT = 1;
  static constexpr bool TWO_D = false;
  using Params = ProgPair;
  __device__ __forceinline__ static void pair(const uint32_t (&a)[2], uint32_t (&b)[1],
                                              const Params &p) {
    b[0] = pmul<DT>(a[1], eval_prog<DT, FORM, D>(a[0], p.p1));
  }
};

// y = s(g) * u; inputs (g, u)
template <int DT, int DS>
struct OpSwigluFwd {
  static constexpr int NIN = 2, NOUT = 1;
  static constexpr bool TWO_D = true;
  using Params = ProgPair;
  __device__ __forceinline__ static void pair(const uint32_t (&a)[2], uint32_t (&b)[1],
                                              const Params &p) {
    b[0] = pmul<DT>(eval_prog<DT, POLY_FORM_HX, DS>(a[0], p.p1), a[1]);
  }
};

// dg = (dy * u) * s'(g), du = dy * s(g); inputs (g, u, dy)
template <int DT, int DS, int DD>
struct OpSwigluBwd {
  static constexpr int NIN = 3, NOUT = 2;
  static constexpr bool TWO_D = true;
  using Params = ProgPair;
  __device__ __forceinline__ static void pair(const uint32_t (&a)[3], uint32_t (&b)[2],
                                              const Params &p) {
    const uint32_t s = eval_prog<DT, POLY_FORM_HX, DS>(a[0], p.p1);
    const uint32_t sd = eval_prog<DT, POLY_FORM_CO, DD>(a[0], p.p2);
    b[0] = pmul<DT>(pmul<DT>(a[2], a[1]), sd);
    b[1] = pmul<DT>(a[2], s);
  }
};

// The paper's deployed B1/B4 rule (§3.3, §5.2.4): recompute the sigmoid
// program p(g) and form SiLU and its derivative algebraically.
// y = (g * p) * u; inputs (g, u)
template <int DT, int DP>
struct OpSwigluSigFwd {
  static constexpr int NIN = 2, NOUT = 1;
  static constexpr bool TWO_D = true;
  using Params = ProgPair;
  __device__ __forceinline__ static void pair(const uint32_t (&a)[2], uint32_t (&b)[1],
                                              const Params &p) {
    const uint32_t pg = eval_prog<DT, POLY_FORM_CO, DP>(a[0], p.p1);
    b[0] = pmul<DT>(pmul<DT>(a[0], pg), a[1]);
  }
};

// s = g p, q = fma(-p, p, p) = p (1 - p), s' = fma(g, q, p);
// dg = (dy * u) * s', du = dy * s; inputs (g, u, dy)
template <int DT, int DP>
struct OpSwigluSigBwd {
  static constexpr int NIN = 3, NOUT = 2;
  static constexpr bool TWO_D = true;
  using Params = ProgPair;
  __device__ __forceinline__ static void pair(const uint32_t (&a)[3], uint32_t (&b)[2],
                                              const Params &p) {
    const uint32_t pg = eval_prog<DT, POLY_FORM_CO, DP>(a[0], p.p1);
    const uint32_t q = pfma<DT>(pg ^ 0x80008000u, pg, pg);
    const uint32_t sd = pfma<DT>(a[0], q, pg);
    b[0] = pmul<DT>(pmul<DT>(a[2], a[1]), sd);
    b[1] = pmul<DT>(a[2], pmul<DT>(a[0], pg));
  }
};

}  // namespace dev
}  // namespace polyact
