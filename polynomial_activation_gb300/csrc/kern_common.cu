// kern_common.cu -- launch sizing and the dispatch from the C ABI layer to
// the per-family translation units.
#include <atomic>

#include "poly_ops.cuh"

namespace polyact {
namespace dev {

cudaError_t launch_act(int kind, int dtype, int form, int deg, const Streams &s,
                       const Layout &l, const ProgPair &p, cudaStream_t st);
cudaError_t launch_swiglu(int kind, int variant, int dtype, int ds, int dd, const Streams &s,
                          const Layout &l, const ProgPair &p, cudaStream_t st);

int sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      v = 152;
    cache[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

int64_t grid_for(const Layout &l, int per_thread) {
  int64_t work;
  if (l.mode == kStrided)
    work = l.rows * l.cols;
  else if (l.mode == kRagged)
    work = l.cap_rows * l.cols;   // an upper bound: the row range is on the device
  else
    work = l.n;
  const int64_t per_block = (int64_t)kThreads * per_thread;
  int64_t blocks = (work + per_block - 1) / per_block;
  const int64_t max_blocks = 0x7FFFFFFF;
  if (blocks > max_blocks) blocks = max_blocks;   // the kernels stride past this
  if (blocks < 1) blocks = 1;
  return blocks;
}

template <int DT, int OP>
struct OpDiag {
  static constexpr int NIN = 3, NOUT = 1;
  static constexpr bool TWO_D = false;
  struct Params {};
  __device__ __forceinline__ static void pair(const uint32_t (&a)[3], uint32_t (&b)[1],
                                              const Params &) {
    if constexpr (OP == POLY_DIAG_FMA) b[0] = pfma<DT>(a[0], a[1], a[2]);
    else if constexpr (OP == POLY_DIAG_MUL) b[0] = pmul<DT>(a[0], a[1]);
    else if constexpr (OP == POLY_DIAG_MIN_NAN) b[0] = pmin_nan<DT>(a[0], a[1]);
    else if constexpr (OP == POLY_DIAG_MAX) b[0] = pmax<DT>(a[0], a[1]);
    else b[0] = pgt_mask<DT>(a[0], a[1]);
  }
};

template <int DT>
static cudaError_t diag_dt(int op, const Streams &s, const Layout &l, cudaStream_t st) {
  switch (op) {
    case POLY_DIAG_FMA: return launch_op<OpDiag<DT, POLY_DIAG_FMA>>(s, l, {}, st);
    case POLY_DIAG_MUL: return launch_op<OpDiag<DT, POLY_DIAG_MUL>>(s, l, {}, st);
    case POLY_DIAG_MIN_NAN: return launch_op<OpDiag<DT, POLY_DIAG_MIN_NAN>>(s, l, {}, st);
    case POLY_DIAG_MAX: return launch_op<OpDiag<DT, POLY_DIAG_MAX>>(s, l, {}, st);
    case POLY_DIAG_GT: return launch_op<OpDiag<DT, POLY_DIAG_GT>>(s, l, {}, st);
  }
  return cudaErrorInvalidValue;
}

// Streaming-bandwidth probe (a measurement tool beside the kernels it
// measures): `reps` passes over nvec 16-byte chunks, each writing out = a or
// a ^ b with the kernels' own loads and stores.  Every thread keeps INF
// chunks per input in flight: U of its chunk slots (grid-strided) times ILP
// consecutive passes loaded before any is stored.  Pass r shifts the chunk a
// slot takes by r * rot (mod nvec), so every pass moves each chunk through
// another SM.  With a working set that fits in L2 and enough passes to hide
// one launch's ramp and drain, the rate is the L2 streaming bandwidth of
// 16-byte register-staged accesses with that much in flight; above L2 size
// it is the HBM rate of the same pattern.
template <int NIN, int U, int ILP>
__global__ void __launch_bounds__(kThreads)
    stream_peak_kernel(const uint16_t *a, const uint16_t *b, uint16_t *out, uint32_t nvec,
                       uint32_t rot, int reps) {
  pdl_wait();
  const uint32_t stride = gridDim.x * (uint32_t)kThreads;
  const uint32_t first = blockIdx.x * (uint32_t)kThreads + threadIdx.x;
  uint32_t shift = 0;
#pragma unroll 1
  for (int r = 0; r < reps; r += ILP) {
#pragma unroll 1
    for (uint32_t c = first; c < nvec; c += U * stride) {
      uint32_t k[U][ILP];
      uint4 v[U][ILP][NIN];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t j = c + u * stride;
        uint32_t sh = shift;
#pragma unroll
        for (int q = 0; q < ILP; ++q) {
          k[u][q] = 0xFFFFFFFFu;
          if (j < nvec && r + q < reps) {
            k[u][q] = j + sh < nvec ? j + sh : j + sh - nvec;
            v[u][q][0] = ld_stream(a + (size_t)k[u][q] * 8);
            if constexpr (NIN == 2) v[u][q][1] = ld_stream(b + (size_t)k[u][q] * 8);
          }
          sh += rot;
          if (sh >= nvec) sh -= nvec;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int q = 0; q < ILP; ++q) {
          if (k[u][q] != 0xFFFFFFFFu) {
            uint4 o = v[u][q][0];
            if constexpr (NIN == 2) {
              o.x ^= v[u][q][1].x;
              o.y ^= v[u][q][1].y;
              o.z ^= v[u][q][1].z;
              o.w ^= v[u][q][1].w;
            }
            st_stream(out + (size_t)k[u][q] * 8, o);
          }
        }
      }
    }
#pragma unroll
    for (int q = 0; q < ILP; ++q) {
      shift += rot;
      if (shift >= nvec) shift -= nvec;
    }
  }
  pdl_release();
}

// One launch of a probe instance with as many blocks as the SMs hold at
// once (its register budget decides: more chunks in flight per thread means
// fewer resident threads).
template <int NIN, int U, int ILP>
static cudaError_t stream_peak_launch(const uint16_t *a, const uint16_t *b, uint16_t *out,
                                      uint32_t n, uint32_t rot, int reps, cudaStream_t stream) {
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &per_sm, stream_peak_kernel<NIN, U, ILP>, kThreads, 0);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  return launch_pdl(stream_peak_kernel<NIN, U, ILP>, (int64_t)sm_count() * per_sm, kThreads,
                    stream, a, b, out, n, rot, reps);
}

template <int NIN>
static cudaError_t stream_peak_nin(int inflight, const uint16_t *a, const uint16_t *b,
                                   uint16_t *out, uint32_t n, uint32_t rot, int reps,
                                   cudaStream_t stream) {
  switch (inflight) {
    case 1: return stream_peak_launch<NIN, 1, 1>(a, b, out, n, rot, reps, stream);
    case 2: return stream_peak_launch<NIN, 2, 1>(a, b, out, n, rot, reps, stream);
    case 4: return stream_peak_launch<NIN, 2, 2>(a, b, out, n, rot, reps, stream);
    case 8: return stream_peak_launch<NIN, 2, 4>(a, b, out, n, rot, reps, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dev

cudaError_t launch_stream_peak(int nin, int inflight, const uint16_t *a, const uint16_t *b,
                               uint16_t *out, int64_t nvec, int reps, cudaStream_t stream) {
  const uint32_t n = (uint32_t)nvec;
  const uint32_t rot = ((n / 7u) | 1u) % n;   // n >= 1; shift stays below n
  return nin == 2 ? dev::stream_peak_nin<2>(inflight, a, b, out, n, rot, reps, stream)
                  : dev::stream_peak_nin<1>(inflight, a, b, out, n, rot, reps, stream);
}

cudaError_t launch_diag(int op, int dtype, const Streams &s, const Layout &l,
                        cudaStream_t stream) {
  return dtype == dev::kF16 ? dev::diag_dt<dev::kF16>(op, s, l, stream)
                            : dev::diag_dt<dev::kBF16>(op, s, l, stream);
}

cudaError_t launch_poly(int kind, int dtype, int form1, int deg1, int deg2, const Streams &s,
                        const Layout &l, const DevProg &p1, const DevProg &p2,
                        cudaStream_t stream, int variant) {
  dev::ProgPair pp{p1, p2};
  if (kind == kActFwd || kind == kActBwd)
    return dev::launch_act(kind, dtype, form1, deg1, s, l, pp, stream);
  return dev::launch_swiglu(kind, variant, dtype, deg1, deg2, s, l, pp, stream);
}

}  // namespace polyact
