// kern_swiglu.cu -- SwiGLU gate with the polynomial SiLU ("Fast Polynomial
// Transcendentals for LLMs", §3.4 and §5.2.4 eq. 15): forward y = s(g) u,
// backward dg = (dy u) s'(g), du = dy s(g) in one pass, no intermediate
// activation tensor.  One template instance per (format, degree of s,
// degree of s').
#include "poly_ops.cuh"

namespace polyact {
namespace dev {

template <int DT, int DS>
static cudaError_t sw_bwd_dd(int dd, const Streams &s, const Layout &l, const ProgPair &p,
                             cudaStream_t st) {
  switch (dd) {
    case 3: return launch_op<OpSwigluBwd<DT, DS, 3>>(s, l, p, st);
    case 4: return launch_op<OpSwigluBwd<DT, DS, 4>>(s, l, p, st);
    case 5: return launch_op<OpSwigluBwd<DT, DS, 5>>(s, l, p, st);
    case 6: return launch_op<OpSwigluBwd<DT, DS, 6>>(s, l, p, st);
  }
  return cudaErrorInvalidValue;
}

template <int DT, int DS>
static cudaError_t sw_ds(int kind, int dd, const Streams &s, const Layout &l,
                         const ProgPair &p, cudaStream_t st) {
  if (kind == kSwigluFwd) return launch_op<OpSwigluFwd<DT, DS>>(s, l, p, st);
  return sw_bwd_dd<DT, DS>(dd, s, l, p, st);
}

template <int DT>
static cudaError_t sw_dt(int kind, int ds, int dd, const Streams &s, const Layout &l,
                         const ProgPair &p, cudaStream_t st) {
  switch (ds) {
    case 3: return sw_ds<DT, 3>(kind, dd, s, l, p, st);
    case 4: return sw_ds<DT, 4>(kind, dd, s, l, p, st);
    case 5: return sw_ds<DT, 5>(kind, dd, s, l, p, st);
    case 6: return sw_ds<DT, 6>(kind, dd, s, l, p, st);
  }
  return cudaErrorInvalidValue;
}

template <int DT>
static cudaError_t sw_sig_dt(int kind, int dp, const Streams &s, const Layout &l,
                             const ProgPair &p, cudaStream_t st) {
#define POLYACT_SIG(D)                                                        \
  case D:                                                                     \
    return kind == kSwigluFwd ? launch_op<OpSwigluSigFwd<DT, D>>(s, l, p, st) \
                              : launch_op<OpSwigluSigBwd<DT, D>>(s, l, p, st);
  switch (dp) {
    POLYACT_SIG(3)
    POLYACT_SIG(4)
    POLYACT_SIG(5)
    POLYACT_SIG(6)
  }
#undef POLYACT_SIG
  return cudaErrorInvalidValue;
}

// variant 0: direct SiLU program (+ centred SiLU' program in backward);
// variant 1: sigmoid program recomputed, SiLU and SiLU' formed algebraically
// (ds = the sigmoid program's degree, dd unused).
cudaError_t launch_swiglu(int kind, int variant, int dtype, int ds, int dd, const Streams &s,
                          const Layout &l, const ProgPair &p, cudaStream_t st) {
  if (variant == 1)
    return dtype == kF16 ? sw_sig_dt<kF16>(kind, ds, s, l, p, st)
                         : sw_sig_dt<kBF16>(kind, ds, s, l, p, st);
  return dtype == kF16 ? sw_dt<kF16>(kind, ds, dd, s, l, p, st)
                       : sw_dt<kBF16>(kind, ds, dd, s, l, p, st);
}

}  // namespace dev
}  // namespace polyact
