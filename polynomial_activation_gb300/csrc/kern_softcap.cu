// kern_softcap.cu -- standalone tanh softcap ("Fast Polynomial
// Transcendentals for LLMs", §2.3 eq. 1 and §3.3 eq. 12):
//   forward   y  = alpha * tanh_program(x * (1/alpha))
//   backward  dx = dy * dtanh_program(x * (1/alpha))   (the scale cancels)
// tanh_program is an odd program, dtanh_program an even one (a direct
// derivative fit or the differentiated forward program).  alpha and 1/alpha
// are target-format constants; every product rounds once.
#include "poly_ops.cuh"

namespace polyact {
namespace dev {

struct SoftcapParams {
  DevProg p;
  uint32_t alpha, inv_alpha;   // duplicated pairs
};

template <int DT, int D>
struct OpSoftcapFwd {
  static constexpr int NIN = 1, NOUT = 1;
  static constexpr bool TWO_D = false;
  using Params = SoftcapParams;
  __device__ __forceinline__ static void pair(const uint32_t (&a)[1], uint32_t (&b)[1],
                                              const Params &p) {
    const uint32_t z = pmul<DT>(a[0], p.inv_alpha);
    b[0] = pmul<DT>(p.alpha, eval_prog<DT, POLY_FORM_O, D>(z, p.p));
  }
};

template <int DT, int D>
struct OpSoftcapBwd {
  static constexpr int NIN = 2, NOUT = 1;
  static constexpr bool TWO_D = false;
  using Params = SoftcapParams;
  __device__ __forceinline__ static void pair(const uint32_t (&a)[2], uint32_t (&b)[1],
                                              const Params &p) {
    const uint32_t z = pmul<DT>(a[0], p.inv_alpha);
    b[0] = pmul<DT>(a[1], eval_prog<DT, POLY_FORM_E, D>(z, p.p));
  }
};

template <int DT>
static cudaError_t softcap_dt(int bwd, int deg, const Streams &s, const Layout &l,
                              const SoftcapParams &p, cudaStream_t st) {
  if (!bwd) {
    switch (deg) {
      case 3: return launch_op<OpSoftcapFwd<DT, 3>>(s, l, p, st);
      case 4: return launch_op<OpSoftcapFwd<DT, 4>>(s, l, p, st);
      case 5: return launch_op<OpSoftcapFwd<DT, 5>>(s, l, p, st);
      case 6: return launch_op<OpSoftcapFwd<DT, 6>>(s, l, p, st);
    }
    return cudaErrorInvalidValue;
  }
  switch (deg) {
    case 2: return launch_op<OpSoftcapBwd<DT, 2>>(s, l, p, st);
    case 3: return launch_op<OpSoftcapBwd<DT, 3>>(s, l, p, st);
    case 4: return launch_op<OpSoftcapBwd<DT, 4>>(s, l, p, st);
    case 5: return launch_op<OpSoftcapBwd<DT, 5>>(s, l, p, st);
    case 6: return launch_op<OpSoftcapBwd<DT, 6>>(s, l, p, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dev

cudaError_t launch_softcap(int bwd, int dtype, int degree, const Streams &s, const Layout &l,
                           const DevProg &p, uint16_t alpha, uint16_t inv_alpha,
                           cudaStream_t stream) {
  dev::SoftcapParams sp{p, (uint32_t)alpha * 0x00010001u, (uint32_t)inv_alpha * 0x00010001u};
  return dtype == dev::kF16 ? dev::softcap_dt<dev::kF16>(bwd, degree, s, l, sp, stream)
                            : dev::softcap_dt<dev::kBF16>(bwd, degree, s, l, sp, stream);
}

}  // namespace polyact
