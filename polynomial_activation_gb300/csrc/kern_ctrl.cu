// kern_ctrl.cu -- MUFU-native controls with the same memory schedule as the
// polynomial kernels (same streaming kernel, same loads, stores and grid).
//
// The comparison of "Fast Polynomial Transcendentals for LLMs" (§4.2,
// Table 3) is polynomial FMA programs vs. special-function-unit evaluation.
// These controls evaluate in FP32 with the special-function unit:
//   sigmoid  1 / (1 + 2^(-x log2 e))         ex2.approx + rcp.approx
//   tanh     tanh.approx
//   SiLU     e = 2^(-|x| log2 e); (x >= 0 ? x : x e) / (1 + e)
//            (the overflow-safe form keeps the divisor in (1, 2])
//   GELU     x/2 (1 + erf(x / sqrt 2))         erff: no special-function erf
// and backward from x: sigma (1 - sigma), 1 - tanh^2, sigma (1 + x (1 - sigma)),
// Phi + x phi.  One rounding to the target format at the end.
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

template <int DT, int FN>
static cudaError_t ctrl_fn(int kind, const Streams &s, const Layout &l, cudaStream_t st) {
  if (kind == kActFwd) return launch_op<CtrlFwd<DT, FN>>(s, l, NoParams{}, st);
  return launch_op<CtrlBwd<DT, FN>>(s, l, NoParams{}, st);
}

template <int DT>
static cudaError_t ctrl_dt(int kind, int fn, const Streams &s, const Layout &l,
                           cudaStream_t st) {
  if (kind == kSwigluFwd) return launch_op<CtrlSwigluFwd<DT>>(s, l, NoParams{}, st);
  if (kind == kSwigluBwd) return launch_op<CtrlSwigluBwd<DT>>(s, l, NoParams{}, st);
  switch (fn) {
    case POLY_SIGMOID: return ctrl_fn<DT, POLY_SIGMOID>(kind, s, l, st);
    case POLY_TANH: return ctrl_fn<DT, POLY_TANH>(kind, s, l, st);
    case POLY_SILU: return ctrl_fn<DT, POLY_SILU>(kind, s, l, st);
    case POLY_GELU: return ctrl_fn<DT, POLY_GELU>(kind, s, l, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dev

cudaError_t launch_ctrl(int kind, int dtype, int fn, const Streams &s, const Layout &l,
                        cudaStream_t stream) {
  return dtype == dev::kF16 ? dev::ctrl_dt<dev::kF16>(kind, fn, s, l, stream)
                            : dev::ctrl_dt<dev::kBF16>(kind, fn, s, l, stream);
}

}  // namespace polyact
