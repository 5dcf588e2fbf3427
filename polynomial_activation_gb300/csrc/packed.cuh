// packed.cuh -- two-lane FP16 / BF16 arithmetic on 32-bit registers (sm_103a).
//
// Every operation is one PTX instruction on a register holding two 16-bit
// lanes ("Fast Polynomial Transcendentals for LLMs", §3.4: one packed FMA
// advances two Horner chains).  All round to nearest-even once; subnormals
// are kept (no .ftz); the NaN-propagating minimum implements the clamp of
// eq. 2 so that a NaN input stays NaN.
#pragma once

#include <cstdint>

namespace polyact {
namespace dev {

constexpr int kF16 = 0;
constexpr int kBF16 = 1;

template <int DT>
__device__ __forceinline__ uint32_t pfma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  if constexpr (DT == kF16)
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  else
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

template <int DT>
__device__ __forceinline__ uint32_t pmul(uint32_t a, uint32_t b) {
  uint32_t d;
  if constexpr (DT == kF16)
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// min that returns NaN if either lane operand is NaN
template <int DT>
__device__ __forceinline__ uint32_t pmin_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  if constexpr (DT == kF16)
    asm("min.NaN.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else
    asm("min.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

template <int DT>
__device__ __forceinline__ uint32_t pmax(uint32_t a, uint32_t b) {
  uint32_t d;
  if constexpr (DT == kF16)
    asm("max.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// per-lane mask: 0xFFFF where a > b (ordered: false for NaN), else 0
template <int DT>
__device__ __forceinline__ uint32_t pgt_mask(uint32_t a, uint32_t b) {
  uint32_t d;
  if constexpr (DT == kF16)
    asm("set.gt.u32.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else
    asm("set.gt.u32.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

template <int DT>
__device__ __forceinline__ constexpr uint32_t half_pair() {
  return DT == kF16 ? 0x38003800u : 0x3F003F00u;   // (0.5, 0.5)
}

}  // namespace dev
}  // namespace polyact
