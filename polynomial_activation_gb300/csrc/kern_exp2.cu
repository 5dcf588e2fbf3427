// kern_exp2.cu -- exp2 with a polynomial fractional core ("Fast Polynomial
// Transcendentals for LLMs", Appendix B.1, eq. 16-19): x = n + f with
// n = floor(x), f in [0, 1); 2^f from a short packed-FP16 program; 2^n
// rebuilt by adding n to the exponent bits.  FP32 in, FP32 out.
//
// Per element: xc = min(max(x, -126), 128); n = floor(xc); f = xc - n
// (FP32, one rounding); h = f rounded to FP16; the core (one rounding per
// packed op, FP16 constants):
//   D1    p = fma(h, 1, 1)
//   PWL2  p = fma(h, a, 1); m = max(fma(h, 1, -1/2), 0); p = fma(m, b, p)
//   D2    v = fma(b, h, a); p = fma(v, h, 1)
//   D3    v = fma(c3, h, c2); v = fma(v, h, c1); p = fma(v, h, 1)
// then y = bits(float(p)) + (n << 23); NaN in -> 0x7FFFFFFF.  The MUFU
// control computes ex2.approx.ftz.f32(x) with the same memory schedule.
#include <cuda_fp16.h>

#include "launch.h"
#include "packed.cuh"
#include "stream_kernel.cuh"

namespace polyact {
namespace dev {

constexpr int kExp2Threads = 256;

struct Exp2Params {
  uint32_t c[3];   // core constants as duplicated FP16 pairs
};

template <int CORE>
__device__ __forceinline__ uint32_t exp2_core(uint32_t h, const Exp2Params &p) {
  constexpr uint32_t one = 0x3C003C00u, mhalf = 0xB800B800u;
  if constexpr (CORE == POLY_EXP2_D1) {
    return pfma<kF16>(h, one, one);
  } else if constexpr (CORE == POLY_EXP2_PWL2) {
    const uint32_t q = pfma<kF16>(h, p.c[0], one);
    const uint32_t m = pmax<kF16>(pfma<kF16>(h, one, mhalf), 0u);
    return pfma<kF16>(m, p.c[1], q);
  } else if constexpr (CORE == POLY_EXP2_D2) {
    return pfma<kF16>(pfma<kF16>(p.c[1], h, p.c[0]), h, one);
  } else {
    uint32_t v = pfma<kF16>(p.c[2], h, p.c[1]);
    v = pfma<kF16>(v, h, p.c[0]);
    return pfma<kF16>(v, h, one);
  }
}

// Two elements (one packed pair through the core).
template <int CORE>
__device__ __forceinline__ float2 exp2_pair(float x0, float x1, const Exp2Params &p) {
  if constexpr (CORE == POLY_EXP2_MUFU) {
    float y0, y1;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y0) : "f"(x0));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y1) : "f"(x1));
    return make_float2(y0, y1);
  } else {
    const float c0 = fminf(fmaxf(x0, -126.0f), 128.0f), c1 = fminf(fmaxf(x1, -126.0f), 128.0f);
    const float n0 = floorf(c0), n1 = floorf(c1);
    const float f0 = __fsub_rn(c0, n0), f1 = __fsub_rn(c1, n1);
    __half2 h = __floats2half2_rn(f0, f1);                      // low lane = f0
    const uint32_t q = exp2_core<CORE>(*reinterpret_cast<uint32_t *>(&h), p);
    const __half2 qh = *reinterpret_cast<const __half2 *>(&q);
    const float2 pf = __half22float2(qh);
    uint32_t b0 = __float_as_uint(pf.x) + ((uint32_t)(int)n0 << 23);
    uint32_t b1 = __float_as_uint(pf.y) + ((uint32_t)(int)n1 << 23);
    if (x0 != x0) b0 = 0x7FFFFFFFu;
    if (x1 != x1) b1 = 0x7FFFFFFFu;
    return make_float2(__uint_as_float(b0), __uint_as_float(b1));
  }
}

// One-pass grid over n floats: two 16-byte chunks (8 floats) per thread when
// x and y share their address modulo 16, scalar head and tail otherwise.
template <int CORE>
__global__ void __launch_bounds__(kExp2Threads) exp2_kernel(const float *__restrict__ x,
                                                           float *__restrict__ y, int64_t n,
                                                           int vec, Exp2Params p) {
  pdl_wait();
  int64_t head = n;
  if (vec) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(x);
    head = (int64_t)(((16u - (a & 15u)) & 15u) >> 2);
    if (head > n) head = n;
  }
  const int64_t nvec = (n - head) >> 2;
  const int64_t body_end = head + (nvec << 2);
  const int64_t gid = (int64_t)blockIdx.x * kExp2Threads + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * kExp2Threads;
#pragma unroll 1
  for (int64_t base = (int64_t)blockIdx.x * (2 * kExp2Threads) + threadIdx.x; base < nvec;
       base += (int64_t)gridDim.x * (2 * kExp2Threads)) {
    float4 v[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int64_t i = base + u * kExp2Threads;
      if (i < nvec)
        asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(v[u].x), "=f"(v[u].y), "=f"(v[u].z), "=f"(v[u].w)
                     : "l"(x + head + (i << 2)));
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int64_t i = base + u * kExp2Threads;
      if (i < nvec) {
        const float2 a = exp2_pair<CORE>(v[u].x, v[u].y, p);
        const float2 b = exp2_pair<CORE>(v[u].z, v[u].w, p);
        asm volatile("st.global.L1::no_allocate.v4.f32 [%0], {%1, %2, %3, %4};"
                     :
                     : "l"(y + head + (i << 2)), "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y)
                     : "memory");
      }
    }
  }
  const int64_t ntail = n - body_end;
#pragma unroll 1
  for (int64_t i = gid; i < head + ntail; i += stride) {
    const int64_t e = i < head ? i : body_end + (i - head);
    const float xv = x[e];
    y[e] = exp2_pair<CORE>(xv, xv, p).x;
  }
  pdl_release();
}

template <int CORE>
static cudaError_t go(const float *x, float *y, int64_t n, int vec, const Exp2Params &p,
                      cudaStream_t st) {
  const int64_t per_block = (int64_t)kExp2Threads * (vec ? 8 : 1);
  int64_t blocks = (n + per_block - 1) / per_block;
  if (blocks > 0x7FFFFFFF) blocks = 0x7FFFFFFF;
  if (blocks < 1) blocks = 1;
  return launch_pdl(exp2_kernel<CORE>, blocks, kExp2Threads, st, x, y, n, vec, p);
}

}  // namespace dev

cudaError_t launch_exp2(int core, const float *x, float *y, int64_t n, int vec,
                        const uint16_t *c, cudaStream_t stream) {
  dev::Exp2Params p;
  for (int j = 0; j < 3; ++j) p.c[j] = (uint32_t)c[j] * 0x00010001u;
  switch (core) {
    case POLY_EXP2_D1: return dev::go<POLY_EXP2_D1>(x, y, n, vec, p, stream);
    case POLY_EXP2_PWL2: return dev::go<POLY_EXP2_PWL2>(x, y, n, vec, p, stream);
    case POLY_EXP2_D2: return dev::go<POLY_EXP2_D2>(x, y, n, vec, p, stream);
    case POLY_EXP2_D3: return dev::go<POLY_EXP2_D3>(x, y, n, vec, p, stream);
    case POLY_EXP2_MUFU: return dev::go<POLY_EXP2_MUFU>(x, y, n, vec, p, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace polyact
