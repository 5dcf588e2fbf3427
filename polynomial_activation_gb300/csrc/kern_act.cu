// kern_act.cu -- elementwise forward and backward programs (the isolated
// function sweep of "Fast Polynomial Transcendentals for LLMs", §4.2 and
// Table 3): one template instance per (format, form, degree).
#include "poly_ops.cuh"

namespace polyact {
namespace dev {

template <int DT, int FORM>
static cudaError_t act_deg(int kind, int deg, const Streams &s, const Layout &l,
                           const ProgPair &p, cudaStream_t st) {
  // forward forms: CO, O, HX; backward forms: E, CO
  constexpr bool fwd_ok = FORM != POLY_FORM_E;
  constexpr bool bwd_ok = FORM == POLY_FORM_E || FORM == POLY_FORM_CO;
#define POLYACT_CASE(D)                                                          \
  case D:                                                                        \
    if constexpr (fwd_ok) {                                                      \
      if (kind == kActFwd) return launch_op<OpFwd<DT, FORM, D>>(s, l, p, st);    \
    }                                                                            \
    if constexpr (bwd_ok) {                                                      \
      if (kind == kActBwd) return launch_op<OpBwd<DT, FORM, D>>(s, l, p, st);    \
    }                                                                            \
    return cudaErrorInvalidValue;
  switch (deg) {
    case 2:   // only even programs derived from degree-3 forward programs
      if constexpr (FORM == POLY_FORM_E) {
        if (kind == kActBwd) return launch_op<OpBwd<DT, POLY_FORM_E, 2>>(s, l, p, st);
      }
      return cudaErrorInvalidValue;
    POLYACT_CASE(3)
    POLYACT_CASE(4)
    POLYACT_CASE(5)
    POLYACT_CASE(6)
  }
#undef POLYACT_CASE
  return cudaErrorInvalidValue;
}

template <int DT>
static cudaError_t act_dt(int kind, int form, int deg, const Streams &s, const Layout &l,
                          const ProgPair &p, cudaStream_t st) {
  if (kind == kActFwd) {
    switch (form) {
      case POLY_FORM_CO: return act_deg<DT, POLY_FORM_CO>(kind, deg, s, l, p, st);
      case POLY_FORM_O: return act_deg<DT, POLY_FORM_O>(kind, deg, s, l, p, st);
      case POLY_FORM_HX: return act_deg<DT, POLY_FORM_HX>(kind, deg, s, l, p, st);
    }
  } else {
    switch (form) {
      case POLY_FORM_E: return act_deg<DT, POLY_FORM_E>(kind, deg, s, l, p, st);
      case POLY_FORM_CO: return act_deg<DT, POLY_FORM_CO>(kind, deg, s, l, p, st);
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_act(int kind, int dtype, int form, int deg, const Streams &s,
                       const Layout &l, const ProgPair &p, cudaStream_t st) {
  return dtype == kF16 ? act_dt<kF16>(kind, form, deg, s, l, p, st)
                       : act_dt<kBF16>(kind, form, deg, s, l, p, st);
}

}  // namespace dev
}  // namespace polyact
