// stream_kernel.cuh -- the streaming elementwise kernel shared by every
// entry point (polynomial programs, SwiGLU, MUFU controls).
//
// Each element is independent, so the work is a pure memory stream: HBM (or
// L2) bandwidth bounds it, not arithmetic.  The kernel therefore does
//  * 16-byte loads and stores (8 FP16/BF16 elements = 4 packed pairs per
//    access, "Fast Polynomial Transcendentals for LLMs" §3.4: "one thread
//    loads a 16-byte int4 chunk, reinterprets it as four pairs"), with
//    kUnroll independent chunks per stream in flight per thread;
//  * a grid sized to the resident capacity of the GPU (a multiple of the SM
//    count), striding over the tensor;
//  * a scalar head (up to 7 elements, when the tensors are not 16-byte
//    aligned) and tail (n % 8), evaluated with the same packed instructions
//    on one lane so that every element gets bit-identical arithmetic.
// An operation ("Op") supplies NIN input streams, NOUT output streams and a
// function from NIN packed pairs to NOUT packed pairs.
#pragma once

#include <cstdint>

#include "launch.h"

namespace polyact {
namespace dev {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

// Streaming loads: the data is touched once, keep it out of L1.
__device__ __forceinline__ uint4 ld_stream(const uint16_t *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream(uint16_t *p, const uint4 &v) {
  asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1, %2, %3, %4};"
               :
               : "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ uint16_t ld_one(const uint16_t *p) {
  uint16_t v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

template <class Op>
__device__ __forceinline__ void apply_chunk(const uint4 (&in)[Op::NIN], uint4 (&out)[Op::NOUT],
                                            const typename Op::Params &p) {
  const uint32_t *iw[Op::NIN];
#pragma unroll
  for (int k = 0; k < Op::NIN; ++k) iw[k] = reinterpret_cast<const uint32_t *>(&in[k]);
  uint32_t *ow[Op::NOUT];
#pragma unroll
  for (int k = 0; k < Op::NOUT; ++k) ow[k] = reinterpret_cast<uint32_t *>(&out[k]);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t a[Op::NIN], b[Op::NOUT];
#pragma unroll
    for (int k = 0; k < Op::NIN; ++k) a[k] = iw[k][w];
    Op::pair(a, b, p);
#pragma unroll
    for (int k = 0; k < Op::NOUT; ++k) ow[k][w] = b[k];
  }
}

template <class Op>
__device__ __forceinline__ void apply_one(const uint16_t *const *in, uint16_t *const *out,
                                          int64_t e, const typename Op::Params &p) {
  uint32_t a[Op::NIN], b[Op::NOUT];
#pragma unroll
  for (int k = 0; k < Op::NIN; ++k) {
    uint32_t v = ld_one(in[k] + e);
    a[k] = v | (v << 16);   // same element in both lanes
  }
  Op::pair(a, b, p);
#pragma unroll
  for (int k = 0; k < Op::NOUT; ++k) out[k][e] = (uint16_t)(b[k] & 0xFFFFu);
}

// Flat / ragged: one contiguous range of elements.
template <class Op>
__device__ __forceinline__ void flat_body(const Streams &s, const Layout &l,
                                          const typename Op::Params &p) {
  int64_t n = l.n, head = l.head, off = 0;
  if (l.mode == kRagged) {
    int64_t lo = l.seg[0], hi = l.seg[l.nseg];
    if (lo < 0) lo = 0;
    if (hi > l.cap_rows) hi = l.cap_rows;
    if (hi < lo) hi = lo;
    off = lo * l.cols;
    n = (hi - lo) * l.cols;
    if (l.vec) {
      const uintptr_t a = reinterpret_cast<uintptr_t>(s.in0 + off);
      head = (int64_t)(((16u - (a & 15u)) & 15u) >> 1);
      if (head > n) head = n;
    } else {
      head = n;
    }
    if (l.status != nullptr && blockIdx.x == 0) {
      int bad = 0;
      for (int e = threadIdx.x; e < l.nseg; e += blockDim.x) bad |= l.seg[e] > l.seg[e + 1];
      if (threadIdx.x == 0) bad |= (l.seg[0] != 0) | (l.seg[l.nseg] > l.cap_rows);
      bad = __syncthreads_or(bad);
      if (threadIdx.x == 0) *l.status = bad ? 1 : 0;
    }
  }
  const uint16_t *in[Op::NIN];
  const uint16_t *src[3] = {s.in0, s.in1, s.in2};
#pragma unroll
  for (int k = 0; k < Op::NIN; ++k) in[k] = src[k] + off;
  uint16_t *out[Op::NOUT];
  uint16_t *dst[2] = {s.out0, s.out1};
#pragma unroll
  for (int k = 0; k < Op::NOUT; ++k) out[k] = dst[k] + off;

  const int64_t nvec = l.vec ? (n - head) / 8 : 0;
  const int64_t body_end = head + nvec * 8;
  const int64_t step = (int64_t)gridDim.x * kThreads * kUnroll;
  for (int64_t base = (int64_t)blockIdx.x * kThreads * kUnroll + threadIdx.x; base < nvec;
       base += step) {
    uint4 r[kUnroll][Op::NIN];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = base + u * kThreads;
      if (i < nvec) {
#pragma unroll
        for (int k = 0; k < Op::NIN; ++k) r[u][k] = ld_stream(in[k] + head + i * 8);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = base + u * kThreads;
      if (i < nvec) {
        uint4 o[Op::NOUT];
        apply_chunk<Op>(r[u], o, p);
#pragma unroll
        for (int k = 0; k < Op::NOUT; ++k) st_stream(out[k] + head + i * 8, o[k]);
      }
    }
  }
  const int64_t ntail = n - body_end;
  for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < head + ntail;
       i += (int64_t)gridDim.x * kThreads) {
    const int64_t e = i < head ? i : body_end + (i - head);
    apply_one<Op>(in, out, e, p);
  }
}

// Strided: rows x cols with a leading dimension per stream.
template <class Op>
__device__ __forceinline__ void strided_body(const Streams &s, const Layout &l,
                                             const typename Op::Params &p) {
  const uint16_t *src[3] = {s.in0, s.in1, s.in2};
  uint16_t *dst[2] = {s.out0, s.out1};
  const int64_t gid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  if (l.vec) {
    const int64_t cpr = l.cols / 8;
    const int64_t total = l.rows * cpr;
    for (int64_t c = gid; c < total; c += stride) {
      const int64_t row = c / cpr;
      const int64_t col = (c - row * cpr) * 8;
      uint4 r[Op::NIN], o[Op::NOUT];
#pragma unroll
      for (int k = 0; k < Op::NIN; ++k) r[k] = ld_stream(src[k] + row * l.ld_in[k] + col);
      apply_chunk<Op>(r, o, p);
#pragma unroll
      for (int k = 0; k < Op::NOUT; ++k) st_stream(dst[k] + row * l.ld_out[k] + col, o[k]);
    }
  } else {
    const int64_t total = l.rows * l.cols;
    for (int64_t e = gid; e < total; e += stride) {
      const int64_t row = e / l.cols;
      const int64_t col = e - row * l.cols;
      const uint16_t *in[Op::NIN];
      uint16_t *out[Op::NOUT];
#pragma unroll
      for (int k = 0; k < Op::NIN; ++k) in[k] = src[k] + row * l.ld_in[k];
#pragma unroll
      for (int k = 0; k < Op::NOUT; ++k) out[k] = dst[k] + row * l.ld_out[k];
      apply_one<Op>(in, out, col, p);
    }
  }
}

template <class Op>
__global__ void __launch_bounds__(kThreads) stream_kernel(Streams s, Layout l,
                                                          typename Op::Params p) {
  if (l.mode == kStrided)
    strided_body<Op>(s, l, p);
  else
    flat_body<Op>(s, l, p);
}

// Blocks for a launch: enough to cover the work once, capped at what the
// GPU holds resident (SM count x resident blocks per SM).
int64_t grid_for(const void *kernel, const Layout &l);

template <class Op>
cudaError_t launch_op(const Streams &s, const Layout &l, const typename Op::Params &p,
                      cudaStream_t stream) {
  const void *k = reinterpret_cast<const void *>(&stream_kernel<Op>);
  const int64_t blocks = grid_for(k, l);
  stream_kernel<Op><<<(unsigned)blocks, kThreads, 0, stream>>>(s, l, p);
  return cudaGetLastError();
}

}  // namespace dev
}  // namespace polyact
