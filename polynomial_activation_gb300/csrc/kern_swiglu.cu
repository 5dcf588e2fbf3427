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

cudaError_t launch_swiglu(int kind, int dtype, int ds, int dd, const Streams &s,
                          const Layout &l, const ProgPair &p, cudaStream_t st) {
  return dtype == kF16 ? sw_dt<kF16>(kind, ds, dd, s, l, p, st)
                       : sw_dt<kBF16>(kind, ds, dd, s, l, p, st);
}

}  // namespace dev
}  // namespace polyact
