// launch.h -- host-side launch interface between the C ABI layer and the
// CUDA translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/polyact.h"

namespace polyact {

// A program as the kernels see it: every coefficient duplicated into both
// lanes of a 32-bit register.
struct DevProg {
  uint32_t c[POLY_MAX_DEGREE + 1];
  uint32_t lc;
};

// Up to three input and two output streams of 16-bit elements.
struct Streams {
  const uint16_t *in0, *in1, *in2;
  uint16_t *out0, *out1;
};

enum LayoutMode { kFlat = 0, kRagged = 1, kStrided = 2 };

// Where the elements are.
//  kFlat:    n contiguous elements; `vec` when every stream sits at the same
//            address modulo 16 (16-byte body, scalar head and tail).
//  kRagged:  rows [seg[0], seg[nseg]) of a [cap_rows, cols] matrix, bounds
//            read on the device; `vec` as for kFlat on the base addresses.
//  kStrided: rows x cols with per-stream leading dimensions; `vec` when every
//            row start is 16-byte aligned and cols % 8 == 0.
struct Layout {
  int mode;
  int vec;
  int64_t n;
  const int32_t *seg;
  int32_t nseg;
  int64_t cap_rows, cols, rows;
  int32_t *status;
  int64_t ld_in[3], ld_out[2];
};

enum Kind { kActFwd = 0, kActBwd = 1, kSwigluFwd = 2, kSwigluBwd = 3 };

// Polynomial programs.  p2 is used by kSwigluBwd of variant 0 only (the SiLU
// derivative); SwiGLU variant 1 takes the sigmoid program in p1.
cudaError_t launch_poly(int kind, int dtype, int form1, int deg1, int deg2, const Streams &s,
                        const Layout &l, const DevProg &p1, const DevProg &p2,
                        cudaStream_t stream, int variant = 0);

// MUFU controls (fn used by kActFwd / kActBwd; variant = POLY_CTRL_*).
cudaError_t launch_ctrl(int kind, int dtype, int fn, const Streams &s, const Layout &l,
                        cudaStream_t stream, int variant);

// Tanh softcap: forward with the odd tanh program, backward with an even
// derivative program; alpha and 1/alpha as target-format bit patterns.
cudaError_t launch_softcap(int bwd, int dtype, int degree, const Streams &s, const Layout &l,
                           const DevProg &p, uint16_t alpha, uint16_t inv_alpha,
                           cudaStream_t stream);

// exp2 with a polynomial fractional core (core = POLY_EXP2_*; c = up to
// three FP16 constants of the core).
cudaError_t launch_exp2(int core, const float *x, float *y, int64_t n, int vec,
                        const uint16_t *c, cudaStream_t stream);

// Fused RoPE (FP16): inputs / outputs in [B, S, H, D] or [B, H, S, D] order.
struct RopeArgs {
  const uint16_t *in_q, *in_k;
  uint16_t *out_q, *out_k;
  const uint32_t *delta;                 // Q0.32 turn increment per frequency
  const uint16_t *cos_tab, *sin_tab;     // table variant: [S, D/2] FP16
  int64_t batch, seq, hq, hkv, head_dim, pos_offset;
};
// FP16 sine (s1, s3, s5) and cosine (c2, c4, c6) coefficients, duplicated pairs.
struct RopeConsts {
  uint32_t s[3], c[3];
};
cudaError_t launch_rope(int variant, int inv, const RopeArgs &a, const RopeConsts &k,
                        cudaStream_t stream);

// Zero the rows of a [cap_rows, cols] 16-bit buffer outside [seg[0], seg[nseg])
// (clamped to [0, cap_rows] on the device, as the ragged kernels do).
cudaError_t launch_zero_outside(uint16_t *out, const int32_t *seg, int32_t nseg,
                                int64_t cap_rows, int64_t cols, cudaStream_t stream);

// Streaming-bandwidth probe: reps passes of out = a (nin 1) or a ^ b (nin 2)
// over nvec 16-byte chunks (every stream 16-byte aligned, 1 <= nvec < 2^31),
// `inflight` (1, 2, 4 or 8) chunks per input in flight per thread.
cudaError_t launch_stream_peak(int nin, int inflight, const uint16_t *a, const uint16_t *b,
                               uint16_t *out, int64_t nvec, int reps, cudaStream_t stream);

// Raw packed instruction over element triples (arithmetic diagnostic).
cudaError_t launch_diag(int op, int dtype, const Streams &s, const Layout &l,
                        cudaStream_t stream);

}  // namespace polyact
