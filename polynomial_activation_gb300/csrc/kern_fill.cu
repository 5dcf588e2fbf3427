// kern_fill.cu -- zero the rows of a routed-expert [cap_rows, cols] buffer
// that no segment covers: rows outside [seg[0], seg[nseg]), with the same
// clamp to [0, cap_rows] the ragged SwiGLU kernels apply.  A ragged output
// or gradient then reads as zero there, and rows inside the range are left
// for the ragged kernel to write -- one pass over the buffer in total, where
// filling the whole buffer first costs a second one.
//
// The row range is read on the device, so the grid cannot be sized to it:
// a grid of at most eight blocks per SM strides over the elements to zero
// (none at all when the segments cover every row), with 16-byte stores and
// a scalar head and tail of at most seven elements per range.
#include "launch.h"
#include "stream_kernel.cuh"

namespace polyact {
namespace dev {

constexpr int kFillThreads = 256;

// Zero elements [s, e) of p, thread t of nt grid-wide.
__device__ __forceinline__ void zero_range(uint16_t *p, int64_t s, int64_t e, int64_t t,
                                           int64_t nt) {
  if (e <= s) return;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(p + s);
  int64_t a = s + (int64_t)(((16u - (addr & 15u)) & 15u) >> 1);   // first 16-byte boundary
  if (a > e) a = e;
  const int64_t nvec = (e - a) >> 3;
  const int64_t z = a + (nvec << 3);
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  for (int64_t k = t; k < nvec; k += nt) st_stream(p + a + (k << 3), zero);
  const int64_t nh = a - s, ntl = e - z;   // at most 7 each
  if (t < nh)
    p[s + t] = 0;
  else if (t < nh + ntl)
    p[z + (t - nh)] = 0;
}

__global__ void __launch_bounds__(kFillThreads)
    zero_outside_kernel(uint16_t *out, const int32_t *seg, int32_t nseg, int64_t cap_rows,
                        int64_t cols) {
  pdl_wait();
  int64_t lo, hi;
  ragged_rows(seg, nseg, cap_rows, nullptr, lo, hi);
  if (lo > cap_rows) lo = cap_rows;   // offsets past the buffer: an empty range
  if (hi > cap_rows) hi = cap_rows;
  const int64_t t = (int64_t)blockIdx.x * kFillThreads + threadIdx.x;
  const int64_t nt = (int64_t)gridDim.x * kFillThreads;
  zero_range(out, 0, lo * cols, t, nt);
  zero_range(out, hi * cols, cap_rows * cols, t, nt);
  pdl_release();
}

}  // namespace dev

cudaError_t launch_zero_outside(uint16_t *out, const int32_t *seg, int32_t nseg,
                                int64_t cap_rows, int64_t cols, cudaStream_t stream) {
  const int64_t chunks = (cap_rows * cols + 7) >> 3;
  int64_t blocks = (chunks + dev::kFillThreads - 1) / dev::kFillThreads;
  const int64_t most = (int64_t)dev::sm_count() * 8;
  if (blocks > most) blocks = most;
  if (blocks < 1) blocks = 1;
  return dev::launch_pdl(dev::zero_outside_kernel, blocks, dev::kFillThreads, stream, out, seg,
                         nseg, cap_rows, cols);
}

}  // namespace polyact
