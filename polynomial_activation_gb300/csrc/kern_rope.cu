// kern_rope.cu -- fused rotary position embedding with paired polynomial
// sine / cosine ("Fast Polynomial Transcendentals for LLMs", Appendix B.2).
//
// Forward reads FP16 Q [B, S, Hq, D] and K [B, S, Hkv, D] and writes the
// rotated tensors transposed to [B, Hq, S, D] and [B, Hkv, S, D]; backward
// reads gradients in the transposed layout, rotates by -theta and writes
// [B, S, H, D].  One thread owns four frequencies (a 16-byte chunk of a
// head: four interleaved complex pairs) of one (batch, position) and up to
// eight heads: it forms the four phases once and reuses the sine / cosine
// across those heads.
//
// Phase: phi = (pos * Delta_i) mod 2^32 (Q0.32 turns); as a signed 32-bit
// value it is a Q31 half-turn coordinate in [-1, 1); beyond +-1/2 it folds
// (sin(pi u) = sin(pi (+-1 - u)), cos changes sign); q = s' >> 16 is the
// signed Q15 coordinate.  Polynomial variant (packed FP16, one rounding per
// operation): u = FP16(q) * 2^-15, w = u * u,
//   sin = (fma(fma(s5, w, s3), w, s1)) * u,
//   cos = fma(fma(fma(c6, w, c4), w, c2), w, 1)   (negated if folded).
// Rotation of (a, b) by (c, s): t = (a s, b s) -> (-(b s), a s);
// out = fma((a, b), (c, c), t).  The MUFU variant takes sin / cos from
// sin.approx / cos.approx of pi u in FP32; the table variant reads FP16
// cos / sin tables [S, D/2] supplied by the caller.  All three share the
// rotation and the memory instructions.
#include <cuda_fp16.h>

#include "launch.h"
#include "packed.cuh"
#include "stream_kernel.cuh"

namespace polyact {
namespace dev {

constexpr int kRopeThreads = 256;
constexpr int kHeadUnroll = 8;
constexpr int kHeadsPerThread = 8;   // heads a thread rotates with one sine / cosine set

__device__ __forceinline__ uint32_t swap_lanes(uint32_t x) { return __byte_perm(x, 0, 0x1032); }
__device__ __forceinline__ uint32_t lane_lo2(uint32_t x) { return __byte_perm(x, 0, 0x1010); }
__device__ __forceinline__ uint32_t lane_hi2(uint32_t x) { return __byte_perm(x, 0, 0x3232); }

// Q15 half-turn coordinate of (pos * delta) mod 2^32 and whether it folded.
__device__ __forceinline__ int q15(uint32_t pos, uint32_t delta, uint32_t &flip) {
  const int32_t s = (int32_t)(pos * delta);            // wraps mod 2^32
  int64_t s2 = s;
  flip = 0;
  if (s > (1 << 30)) {
    s2 = (int64_t(1) << 31) - s;
    flip = 1;
  } else if (s < -(1 << 30)) {
    s2 = -(int64_t(1) << 31) - s;
    flip = 1;
  }
  return (int)(s2 >> 16);
}

__device__ __forceinline__ uint32_t int_pair_to_f16(int q0, int q1) {
  const __half h0 = __int2half_rn(q0), h1 = __int2half_rn(q1);
  const __half2 h = __halves2half2(h0, h1);
  return *reinterpret_cast<const uint32_t *>(&h);
}

// cos, sin pairs (lanes = two frequencies) of the folded coordinates.
template <int VARIANT>
__device__ __forceinline__ void sincos2(int q0, int q1, uint32_t f0, uint32_t f1,
                                        const RopeConsts &k, uint32_t &cs, uint32_t &sn) {
  const uint32_t flipmask = (f0 ? 0x00008000u : 0u) | (f1 ? 0x80000000u : 0u);
  if constexpr (VARIANT == POLY_ROPE_POLY) {
    const uint32_t u = pmul<kF16>(int_pair_to_f16(q0, q1), 0x02000200u);   // * 2^-15
    const uint32_t w = pmul<kF16>(u, u);
    uint32_t v = pfma<kF16>(k.s[2], w, k.s[1]);
    v = pfma<kF16>(v, w, k.s[0]);
    sn = pmul<kF16>(v, u);
    v = pfma<kF16>(k.c[2], w, k.c[1]);
    v = pfma<kF16>(v, w, k.c[0]);
    cs = pfma<kF16>(v, w, 0x3C003C00u) ^ flipmask;
  } else {
    const float t0 = (float)q0 * (3.14159265358979323846f / 32768.0f);
    const float t1 = (float)q1 * (3.14159265358979323846f / 32768.0f);
    float s0, s1, c0, c1;
    asm("sin.approx.f32 %0, %1;" : "=f"(s0) : "f"(t0));
    asm("sin.approx.f32 %0, %1;" : "=f"(s1) : "f"(t1));
    asm("cos.approx.f32 %0, %1;" : "=f"(c0) : "f"(t0));
    asm("cos.approx.f32 %0, %1;" : "=f"(c1) : "f"(t1));
    __half2 hs = __floats2half2_rn(s0, s1), hc = __floats2half2_rn(c0, c1);
    sn = *reinterpret_cast<uint32_t *>(&hs);
    cs = *reinterpret_cast<uint32_t *>(&hc) ^ flipmask;
  }
}

// Rotate one packed complex number x = (a, b) by (c, s) given as duplicated pairs.
__device__ __forceinline__ uint32_t rotate(uint32_t x, uint32_t cc, uint32_t ss) {
  const uint32_t t = swap_lanes(pmul<kF16>(x, ss)) ^ 0x00008000u;   // (-(b s), a s)
  return pfma<kF16>(x, cc, t);
}

__device__ __forceinline__ uint4 ld16(const uint16_t *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st16(uint16_t *p, const uint4 &v) {
  asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1, %2, %3, %4};"
               :
               : "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

template <int VARIANT, int INV>
__global__ void __launch_bounds__(kRopeThreads) rope_kernel(RopeArgs a, RopeConsts k) {
  pdl_wait();
  const int64_t groups = a.head_dim >> 3;                // chunks of 4 frequencies
  const int64_t H = a.hq + a.hkv;
  const int64_t hchunks = (H + kHeadsPerThread - 1) / kHeadsPerThread;
  const int64_t total = a.batch * a.seq * hchunks * groups;
  for (int64_t t = (int64_t)blockIdx.x * kRopeThreads + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * kRopeThreads) {
    int64_t j, hc, b, s;
    if (total <= 0xFFFFFFFFll) {   // 32-bit index arithmetic (the common case)
      const uint32_t t32 = (uint32_t)t, g32 = (uint32_t)groups, h32 = (uint32_t)hchunks;
      const uint32_t r = t32 / g32, bs = r / h32;
      j = t32 - r * g32;
      hc = r - bs * h32;
      b = bs / (uint32_t)a.seq;
      s = bs - (uint32_t)b * (uint32_t)a.seq;
    } else {
      j = t % groups;
      const int64_t r = t / groups;
      hc = r % hchunks;
      const int64_t bs = r / hchunks;
      b = bs / a.seq;
      s = bs - b * a.seq;
    }
    const int64_t h_begin = hc * kHeadsPerThread;
    const int64_t h_end = h_begin + kHeadsPerThread < H ? h_begin + kHeadsPerThread : H;
    // ---- four (cos, sin) pairs for frequencies 4j .. 4j+3
    uint32_t cA, sA, cB, sB;
    if constexpr (VARIANT == POLY_ROPE_TABLE) {
      const uint16_t *ct = a.cos_tab + s * (a.head_dim >> 1) + 4 * j;
      const uint16_t *st = a.sin_tab + s * (a.head_dim >> 1) + 4 * j;
      const uint2 cv = *reinterpret_cast<const uint2 *>(ct);
      const uint2 sv = *reinterpret_cast<const uint2 *>(st);
      cA = cv.x; cB = cv.y; sA = sv.x; sB = sv.y;
    } else {
      const uint32_t pos = (uint32_t)(a.pos_offset + s);
      const uint4 d = *reinterpret_cast<const uint4 *>(a.delta + 4 * j);
      uint32_t f0, f1, f2, f3;
      const int q0 = q15(pos, d.x, f0), q1 = q15(pos, d.y, f1);
      const int q2 = q15(pos, d.z, f2), q3 = q15(pos, d.w, f3);
      sincos2<VARIANT>(q0, q1, f0, f1, k, cA, sA);
      sincos2<VARIANT>(q2, q3, f2, f3, k, cB, sB);
    }
    if constexpr (INV) {
      sA ^= 0x80008000u;
      sB ^= 0x80008000u;
    }
    // ---- every head of this (batch, position): [B, S, H, D] <-> [B, H, S, D]
#pragma unroll 1
    for (int64_t h0 = h_begin; h0 < h_end; h0 += kHeadUnroll) {
      uint4 v[kHeadUnroll];
#pragma unroll
      for (int u = 0; u < kHeadUnroll; ++u) {
        const int64_t h = h0 + u;
        if (h < h_end) {
          const bool isq = h < a.hq;
          const int64_t hh = isq ? h : h - a.hq, nh = isq ? a.hq : a.hkv;
          const uint16_t *base = isq ? a.in_q : a.in_k;
          const int64_t row = INV ? ((b * nh + hh) * a.seq + s) : ((b * a.seq + s) * nh + hh);
          v[u] = ld16(base + row * a.head_dim + 8 * j);
        }
      }
#pragma unroll
      for (int u = 0; u < kHeadUnroll; ++u) {
        const int64_t h = h0 + u;
        if (h < h_end) {
          const bool isq = h < a.hq;
          const int64_t hh = isq ? h : h - a.hq, nh = isq ? a.hq : a.hkv;
          uint16_t *base = isq ? a.out_q : a.out_k;
          const int64_t row = INV ? ((b * a.seq + s) * nh + hh) : ((b * nh + hh) * a.seq + s);
          uint4 o;
          o.x = rotate(v[u].x, lane_lo2(cA), lane_lo2(sA));
          o.y = rotate(v[u].y, lane_hi2(cA), lane_hi2(sA));
          o.z = rotate(v[u].z, lane_lo2(cB), lane_lo2(sB));
          o.w = rotate(v[u].w, lane_hi2(cB), lane_hi2(sB));
          st16(base + row * a.head_dim + 8 * j, o);
        }
      }
    }
  }
  pdl_release();
}

template <int VARIANT>
static cudaError_t rope_go(int inv, const RopeArgs &a, const RopeConsts &k, cudaStream_t st) {
  const int64_t H = a.hq + a.hkv;
  const int64_t total =
      a.batch * a.seq * ((H + kHeadsPerThread - 1) / kHeadsPerThread) * (a.head_dim >> 3);
  int64_t blocks = (total + kRopeThreads - 1) / kRopeThreads;
  if (blocks > 0x7FFFFFFF) blocks = 0x7FFFFFFF;
  if (blocks < 1) blocks = 1;
  if (inv) return launch_pdl(rope_kernel<VARIANT, 1>, blocks, kRopeThreads, st, a, k);
  return launch_pdl(rope_kernel<VARIANT, 0>, blocks, kRopeThreads, st, a, k);
}

}  // namespace dev

cudaError_t launch_rope(int variant, int inv, const RopeArgs &a, const RopeConsts &k,
                        cudaStream_t stream) {
  switch (variant) {
    case POLY_ROPE_POLY: return dev::rope_go<POLY_ROPE_POLY>(inv, a, k, stream);
    case POLY_ROPE_MUFU: return dev::rope_go<POLY_ROPE_MUFU>(inv, a, k, stream);
    case POLY_ROPE_TABLE: return dev::rope_go<POLY_ROPE_TABLE>(inv, a, k, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace polyact
