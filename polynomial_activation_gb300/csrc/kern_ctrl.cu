// kern_ctrl.cu -- MUFU-native controls with the same memory schedule as the
// polynomial kernels (same streaming kernel, same loads, stores and grid).
//
// The comparison of "Fast Polynomial Transcendentals for LLMs" (§4.2,
// Table 3) is polynomial FMA programs vs. special-function-unit evaluation.
// Two controls are built.
//
// FP32 (POLY_CTRL_FP32): each element widened to FP32, special-function unit
// in FP32:
//   sigmoid  1 / (1 + 2^(-x log2 e))         ex2.approx + rcp.approx
//   tanh     tanh.approx
//   SiLU     e = 2^(-|x| log2 e); (x >= 0 ? x : x e) / (1 + e)
//            (the overflow-safe form keeps the divisor in (1, 2])
//   GELU     x/2 (1 + erf(x / sqrt 2))         erff: no special-function erf
// and backward from x: sigma (1 - sigma), 1 - tanh^2, sigma (1 + x (1 - sigma)),
// Phi + x phi.  One rounding to the target format at the end.
//
// Packed (POLY_CTRL_PACKED): every operation on a packed pair in the target
// format, one tanh.approx.{f16x2,bf16x2} instruction per pair (which the
// special-function unit executes as one operation per element: ncu counts one
// special-function instruction per element, half the FP32 control's two for
// sigmoid and SiLU), through the identities sigma(x) = 1/2 + tanh(x/2)/2 and
// SiLU(x) = h + h tanh(h), h = x/2:
//   tanh     t = tanh(x)
//   sigmoid  t = tanh(x * 1/2);  y = fma(t, 1/2, 1/2)
//   SiLU     h = x * 1/2;  t = tanh(h);  y = fma(h, t, h)
//   GELU     the tanh form h (1 + tanh(z)), z = x (k + k c x^2), k = sqrt(2/pi),
//            c = 0.044715 (within 4.8e-4 of exact GELU, 8.7e-4 for its
//            derivative; no special-function erf exists)
//   backward sigma' = fma(-p, p, p) with p = sigma; tanh' = fma(-t, t, 1);
//            SiLU' = fma(x, fma(-p, p, p), p); GELU' = p + (1 - t^2) h z' with
//            p = fma(t, 1/2, 1/2), z' = k + 3 k c x^2 and x clamped to
//            [-16, 16] (the derivative is 0 or 1 to the target precision
//            beyond; the clamp keeps x^2 finite); dx = dy * derivative
// Each packed instruction rounds once to the target format.  Both controls
// approximate the true function, not the polynomial programs.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "packed.cuh"
#include "stream_kernel.cuh"

namespace polyact {
namespace dev {

__device__ __forceinline__ float ex2a(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcpa(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float tanha(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kInvSqrt2 = 0.70710678118654752f;
constexpr float kInvSqrt2Pi = 0.39894228040143268f;

__device__ __forceinline__ float c_sigmoid(float x) { return rcpa(1.0f + ex2a(-x * kLog2e)); }
__device__ __forceinline__ float c_silu(float x) {
  const float e = ex2a(-fabsf(x) * kLog2e);
  const float r = rcpa(1.0f + e);
  return (x >= 0.0f ? x : x * e) * r;
}
__device__ __forceinline__ float c_Phi(float x) { return 0.5f * (1.0f + erff(x * kInvSqrt2)); }

template <int FN>
__device__ __forceinline__ float c_fwd(float x) {
  if constexpr (FN == POLY_SIGMOID) return c_sigmoid(x);
  else if constexpr (FN == POLY_TANH) return tanha(x);
  else if constexpr (FN == POLY_SILU) return c_silu(x);
  else return x * c_Phi(x);
}

template <int FN>
__device__ __forceinline__ float c_bwd(float x) {
  if constexpr (FN == POLY_SIGMOID) {
    const float s = c_sigmoid(x);
    return s * (1.0f - s);
  } else if constexpr (FN == POLY_TANH) {
    const float t = tanha(x);
    return 1.0f - t * t;
  } else if constexpr (FN == POLY_SILU) {
    const float s = c_sigmoid(x);
    return s * (1.0f + x * (1.0f - s));
  } else {
    return c_Phi(x) + x * (ex2a(-0.5f * x * x * kLog2e) * kInvSqrt2Pi);
  }
}

template <int DT>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (DT == kF16) {
    __half2 h = *reinterpret_cast<__half2 *>(&w);
    return __half22float2(h);
  } else {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  }
}

template <int DT>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (DT == kF16) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
  }
}

struct NoParams {};

template <int DT, int FN>
struct CtrlFwd {
  static constexpr int NIN = 1, NOUT = 1;
  static constexpr bool TWO_D = false;
  using Params = NoParams;
  __device__ __forceinline__ static void pair(const uint32_t (&a)[1], uint32_t (&b)[1],
                                              const Params &) {
    const float2 x = unpack2<DT>(a[0]);
    b[0] = pack2<DT>(c_fwd<FN>(x.x), c_fwd<FN>(x.y));
  }
};

template <int DT, int FN>
struct CtrlBwd {
  static constexpr int NIN = 2, NOUT = 1;
  static constexpr bool TWO_D = false;
  using Params = NoParams;
  __device__ __forceinline__ static void pair(const uint32_t (&a)[2], uint32_t (&b)[1],
                                              const Params &) {
    const float2 x = unpack2<DT>(a[0]), dy = unpack2<DT>(a[1]);
    b[0] = pack2<DT>(dy.x * c_bwd<FN>(x.x), dy.y * c_bwd<FN>(x.y));
  }
};

template <int DT>
struct CtrlSwigluFwd {
  static constexpr int NIN = 2, NOUT = 1;
  static constexpr bool TWO_D = true;
  using Params = NoParams;
  __device__ __forceinline__ static void pair(const uint32_t (&a)[2], uint32_t (&b)[1],
                                              const Params &) {
    const float2 g = unpack2<DT>(a[0]), u = unpack2<DT>(a[1]);
    b[0] = pack2<DT>(c_silu(g.x) * u.x, c_silu(g.y) * u.y);
  }
};

template <int DT>
struct CtrlSwigluBwd {
  static constexpr int NIN = 3, NOUT = 2;
  static constexpr bool TWO_D = true;
  using Params = NoParams;
  __device__ __forceinline__ static void pair(const uint32_t (&a)[3], uint32_t (&b)[2],
                                              const Params &) {
    const float2 g = unpack2<DT>(a[0]), u = unpack2<DT>(a[1]), dy = unpack2<DT>(a[2]);
    const float s0 = c_sigmoid(g.x), s1 = c_sigmoid(g.y);
    const float d0 = s0 * (1.0f + g.x * (1.0f - s0)), d1 = s1 * (1.0f + g.y * (1.0f - s1));
    b[0] = pack2<DT>(dy.x * u.x * d0, dy.y * u.y * d1);
    b[1] = pack2<DT>(dy.x * g.x * s0, dy.y * g.y * s1);
  }
};

// ---- packed target-format control -------------------------------------

template <int DT>
__device__ __forceinline__ uint32_t ptanh_approx(uint32_t x) {
  uint32_t y;
  if constexpr (DT == kF16)
    asm("tanh.approx.f16x2 %0, %1;" : "=r"(y) : "r"(x));
  else
    asm("tanh.approx.bf16x2 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

template <int DT>
__device__ __forceinline__ uint32_t pmax_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  if constexpr (DT == kF16)
    asm("max.NaN.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Constants as packed pairs (FP16 / BF16 bit patterns of the nearest value):
// 1; k = sqrt(2/pi) = 0.79788456; k c = 0.03567741; 3 k c = 0.10703222; 16.
template <int DT>
struct PkConst {
  static constexpr uint32_t one = DT == kF16 ? 0x3C003C00u : 0x3F803F80u;
  static constexpr uint32_t k = DT == kF16 ? 0x3A623A62u : 0x3F4C3F4Cu;
  static constexpr uint32_t kc = DT == kF16 ? 0x28912891u : 0x3D123D12u;
  static constexpr uint32_t k3c = DT == kF16 ? 0x2EDA2EDAu : 0x3DDB3DDBu;
  static constexpr uint32_t sixteen = DT == kF16 ? 0x4C004C00u : 0x41804180u;
};

constexpr uint32_t kSignPair = 0x80008000u;

// sigma(x) = fma(tanh(x / 2), 1/2, 1/2)
template <int DT>
__device__ __forceinline__ uint32_t pk_sigmoid(uint32_t x) {
  const uint32_t t = ptanh_approx<DT>(pmul<DT>(x, half_pair<DT>()));
  return pfma<DT>(t, half_pair<DT>(), half_pair<DT>());
}

// SiLU(x) = h + h tanh(h), h = x / 2; also returns t = tanh(h)
template <int DT>
__device__ __forceinline__ uint32_t pk_silu(uint32_t x, uint32_t &t) {
  const uint32_t h = pmul<DT>(x, half_pair<DT>());
  t = ptanh_approx<DT>(h);
  return pfma<DT>(h, t, h);
}

// sigma' = p (1 - p) = fma(-p, p, p)
template <int DT>
__device__ __forceinline__ uint32_t pk_pq(uint32_t p) {
  return pfma<DT>(p ^ kSignPair, p, p);
}

template <int DT, int FN>
__device__ __forceinline__ uint32_t pk_fwd(uint32_t x) {
  using C = PkConst<DT>;
  if constexpr (FN == POLY_SIGMOID) {
    return pk_sigmoid<DT>(x);
  } else if constexpr (FN == POLY_TANH) {
    return ptanh_approx<DT>(x);
  } else if constexpr (FN == POLY_SILU) {
    uint32_t t;
    return pk_silu<DT>(x, t);
  } else {
    const uint32_t x2 = pmul<DT>(x, x);
    const uint32_t z = pmul<DT>(x, pfma<DT>(x2, C::kc, C::k));
    const uint32_t h = pmul<DT>(x, half_pair<DT>());
    return pfma<DT>(h, ptanh_approx<DT>(z), h);
  }
}

template <int DT, int FN>
__device__ __forceinline__ uint32_t pk_bwd(uint32_t x) {
  using C = PkConst<DT>;
  if constexpr (FN == POLY_SIGMOID) {
    return pk_pq<DT>(pk_sigmoid<DT>(x));
  } else if constexpr (FN == POLY_TANH) {
    const uint32_t t = ptanh_approx<DT>(x);
    return pfma<DT>(t ^ kSignPair, t, C::one);
  } else if constexpr (FN == POLY_SILU) {
    const uint32_t p = pk_sigmoid<DT>(x);
    return pfma<DT>(x, pk_pq<DT>(p), p);
  } else {
    const uint32_t xc = pmin_nan<DT>(pmax_nan<DT>(x, C::sixteen ^ kSignPair), C::sixteen);
    const uint32_t x2 = pmul<DT>(xc, xc);
    const uint32_t t = ptanh_approx<DT>(pmul<DT>(xc, pfma<DT>(x2, C::kc, C::k)));
    const uint32_t p = pfma<DT>(t, half_pair<DT>(), half_pair<DT>());
    const uint32_t a = pfma<DT>(t ^ kSignPair, t, C::one);              // 1 - t^2
    const uint32_t b = pmul<DT>(pmul<DT>(xc, half_pair<DT>()), pfma<DT>(x2, C::k3c, C::k));
    return pfma<DT>(a, b, p);
  }
}

template <int DT, int FN>
struct PkFwd {
  static constexpr int NIN = 1, NOUT = 1;
  static constexpr bool TWO_D = false;
  using Params = NoParams;
  __device__ __forceinline__ static void pair(const uint32_t (&a)[1], uint32_t (&b)[1],
                                              const Params &) {
    b[0] = pk_fwd<DT, FN>(a[0]);
  }
};

template <int DT, int FN>
struct PkBwd {
  static constexpr int NIN = 2, NOUT = 1;
  static constexpr bool TWO_D = false;
  using Params = NoParams;
  __device__ __forceinline__ static void pair(const uint32_t (&a)[2], uint32_t (&b)[1],
                                              const Params &) {
    b[0] = pmul<DT>(a[1], pk_bwd<DT, FN>(a[0]));
  }
};

// y = SiLU(g) * u; inputs (g, u)
template <int DT>
struct PkSwigluFwd {
  static constexpr int NIN = 2, NOUT = 1;
  static constexpr bool TWO_D = true;
  using Params = NoParams;
  __device__ __forceinline__ static void pair(const uint32_t (&a)[2], uint32_t (&b)[1],
                                              const Params &) {
    uint32_t t;
    b[0] = pmul<DT>(pk_silu<DT>(a[0], t), a[1]);
  }
};

// s = SiLU(g), p = fma(t, 1/2, 1/2), s' = fma(g, fma(-p, p, p), p);
// dg = (dy * u) * s', du = dy * s; inputs (g, u, dy)
template <int DT>
struct PkSwigluBwd {
  static constexpr int NIN = 3, NOUT = 2;
  static constexpr bool TWO_D = true;
  using Params = NoParams;
  __device__ __forceinline__ static void pair(const uint32_t (&a)[3], uint32_t (&b)[2],
                                              const Params &) {
    uint32_t t;
    const uint32_t s = pk_silu<DT>(a[0], t);
    const uint32_t p = pfma<DT>(t, half_pair<DT>(), half_pair<DT>());
    const uint32_t sd = pfma<DT>(a[0], pk_pq<DT>(p), p);
    b[0] = pmul<DT>(pmul<DT>(a[2], a[1]), sd);
    b[1] = pmul<DT>(a[2], s);
  }
};

template <int DT, int FN>
static cudaError_t ctrl_fn(int kind, int packed, const Streams &s, const Layout &l,
                           cudaStream_t st) {
  if (packed) {
    if (kind == kActFwd) return launch_op<PkFwd<DT, FN>>(s, l, NoParams{}, st);
    return launch_op<PkBwd<DT, FN>>(s, l, NoParams{}, st);
  }
  if (kind == kActFwd) return launch_op<CtrlFwd<DT, FN>>(s, l, NoParams{}, st);
  return launch_op<CtrlBwd<DT, FN>>(s, l, NoParams{}, st);
}

template <int DT>
static cudaError_t ctrl_dt(int kind, int packed, int fn, const Streams &s, const Layout &l,
                           cudaStream_t st) {
  if (kind == kSwigluFwd)
    return packed ? launch_op<PkSwigluFwd<DT>>(s, l, NoParams{}, st)
                  : launch_op<CtrlSwigluFwd<DT>>(s, l, NoParams{}, st);
  if (kind == kSwigluBwd)
    return packed ? launch_op<PkSwigluBwd<DT>>(s, l, NoParams{}, st)
                  : launch_op<CtrlSwigluBwd<DT>>(s, l, NoParams{}, st);
  switch (fn) {
    case POLY_SIGMOID: return ctrl_fn<DT, POLY_SIGMOID>(kind, packed, s, l, st);
    case POLY_TANH: return ctrl_fn<DT, POLY_TANH>(kind, packed, s, l, st);
    case POLY_SILU: return ctrl_fn<DT, POLY_SILU>(kind, packed, s, l, st);
    case POLY_GELU: return ctrl_fn<DT, POLY_GELU>(kind, packed, s, l, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dev

cudaError_t launch_ctrl(int kind, int dtype, int fn, const Streams &s, const Layout &l,
                        cudaStream_t stream, int variant) {
  const int packed = variant == POLY_CTRL_PACKED;
  return dtype == dev::kF16 ? dev::ctrl_dt<dev::kF16>(kind, packed, fn, s, l, stream)
                            : dev::ctrl_dt<dev::kBF16>(kind, packed, fn, s, l, stream);
}

}  // namespace polyact
