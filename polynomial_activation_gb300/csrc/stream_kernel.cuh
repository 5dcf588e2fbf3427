// stream_kernel.cuh -- the streaming elementwise kernel shared by every
// entry point (polynomial programs, SwiGLU, MUFU controls).
//
// Each element is independent, so the work is a pure memory stream: HBM (or
// L2) bandwidth bounds it, not arithmetic.  The kernel therefore does
//  * 16-byte loads and stores (8 FP16/BF16 elements = 4 packed pairs per
//    access, as the paper, "Fast Polynomial Transcendentals for LLMs" §3.4,
//    loads int4 chunks and reinterprets them as four pairs), one or two
//    chunks per stream per thread;
//  * a one-pass grid: every thread owns its chunks, blocks retire and are
//    replaced as fast as the memory system drains them;
//  * a dense kernel for the common cases (flat, or ragged rows of a multiple
//    of 8 columns; every stream 16-byte aligned; fewer than 2^31 elements)
//    with 32-bit indices and no layout branches, which cuts the per-thread
//    instruction count that dominates launches of L2-resident size;
//  * programmatic dependent launch, so that a launch's blocks are scheduled
//    while the previous kernel on the stream drains;
//  * a scalar head (up to the first 16-byte boundary) and tail, evaluated
//    with the same packed instructions on one lane so that every element
//    gets bit-identical arithmetic; inputs whose addresses disagree with the
//    output's modulo 16 bytes are realigned in registers (two aligned
//    16-byte loads and funnel shifts per chunk), and only layouts whose
//    outputs disagree with each other take the scalar path throughout.
// An operation ("Op") supplies NIN input streams, NOUT output streams and a
// function from NIN packed pairs to NOUT packed pairs.
#pragma once

#include <cstdint>

#include "launch.h"

namespace polyact {
namespace dev {

constexpr int kThreads = 256;

// Streaming loads / stores: the data is touched once, keep it out of L1.
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

// Programmatic dependent launch.  pdl_wait() (first thing in every kernel):
// wait until the previous kernel on the stream has completed and its writes
// are visible -- nothing is read before.  pdl_release() (last thing, after the
// stores): this block is done, so the next kernel on the stream may be
// launched once every block of this one has released or exited; its blocks
// are then scheduled while this grid's last stores drain and its completion
// is signalled, instead of after.  Releasing at the end rather than at entry
// keeps the next kernel's blocks from occupying SMs, parked in their own
// wait, while this grid still streams: measured on GB300, 6-25 % off
// launches of 0.5-8 M elements (L2-resident), no change at HBM sizes.  The
// dense kernel releases earlier, right after its loads are issued, where
// that measured faster still: one-input and two-input one-output launches of
// one chunk per thread (below ~1.2 M and ~2.4 M elements) -- 5-22 % off
// 0.25-2.4 M elements.  Everywhere else, and for the three-input SwiGLU
// backward at every size, the release after the stores measured faster
// (8-23 % off 0.25-2 M-element SwiGLU backward launches, 8-18 % off two-input
// launches of two chunks per thread at 2.5-4 M elements).
// Ordering between kernels is unchanged.  (Both are no-ops for a launch
// without the programmatic-serialisation attribute.)
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint16_t ld_one(const uint16_t *p) {
  uint16_t v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// Chunks of 8 elements per stream per thread: two for single-input
// operations, one for multi-input ones (measured on GB300 with a one-pass
// grid: the fastest of 1, 2, 4 and 8 chunks of 16 or 32 bytes at HBM
// sizes).  Smaller calls of the dense kernel, flat, rows or ragged (the
// latter by row capacity), measured over 256 K-268 M elements with
// 256-thread blocks (dense_shape below):
//  * single input: one chunk per thread while two would give fewer than two
//    blocks per SM (below ~1.2 M elements);
//  * two inputs, one output: one chunk per thread while that grid holds at
//    most 8 blocks per SM (below ~2.4 M elements), then two while the
//    two-chunk grid holds at most 16 blocks per SM (~2.4-10 M elements:
//    8-18 % faster at 2.5-4 M for the polynomial programs of 3-5 FMAs, within
//    2 % for the lighter even-form derivatives), one above.
template <class Op>
__host__ __device__ constexpr int chunks_per_thread() {
  return Op::NIN == 1 ? 2 : 1;
}
constexpr int kTwoChunkMaxBlocksPerSm = 16;
constexpr int64_t kRowsTwoOutMax = int64_t(1) << 23;

template <class Op>
__device__ __forceinline__ void apply_chunk(const uint4 (&in)[Op::NIN], uint4 (&out)[Op::NOUT],
                                            const typename Op::Params &p) {
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t a[Op::NIN], b[Op::NOUT];
#pragma unroll
    for (int k = 0; k < Op::NIN; ++k) a[k] = reinterpret_cast<const uint32_t *>(&in[k])[w];
    Op::pair(a, b, p);
#pragma unroll
    for (int k = 0; k < Op::NOUT; ++k) reinterpret_cast<uint32_t *>(&out[k])[w] = b[k];
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

// Row range [lo, hi) of a ragged call: rows [seg[0], seg[nseg]) clamped to
// [0, cap_rows] whatever the offsets say.  If status is given, block 0 also
// records whether the offsets were valid (seg[0] == 0, non-decreasing,
// seg[nseg] <= cap_rows): 0 valid, 1 not.  Every thread of block 0 must call
// this (it synchronises the block).
__device__ __forceinline__ void ragged_rows(const int32_t *seg, int32_t nseg, int64_t cap_rows,
                                            int32_t *status, int64_t &lo, int64_t &hi) {
  lo = seg[0];
  hi = seg[nseg];
  if (lo < 0) lo = 0;
  if (hi > cap_rows) hi = cap_rows;
  if (hi < lo) hi = lo;
  if (status != nullptr && blockIdx.x == 0) {
    int bad = 0;
    for (int e = threadIdx.x; e < nseg; e += blockDim.x) bad |= seg[e] > seg[e + 1];
    if (threadIdx.x == 0) bad |= (seg[0] != 0) | (seg[nseg] > cap_rows);
    bad = __syncthreads_or(bad);
    if (threadIdx.x == 0) *status = bad ? 1 : 0;
  }
}

// Flat / ragged: one contiguous range of elements.  When every stream sits at
// the same address modulo 16 (l.vec), the scalar head runs up to the first
// 16-byte boundary and the body moves 16-byte chunks; otherwise every
// element takes the scalar path.
template <class Op>
__global__ void __launch_bounds__(kThreads) stream_kernel(Streams s, Layout l,
                                                          typename Op::Params p) {
  pdl_wait();
  constexpr int U = chunks_per_thread<Op>();
  int64_t n = l.n, off = 0;
  if (l.mode == kRagged) {
    int64_t lo, hi;
    ragged_rows(l.seg, l.nseg, l.cap_rows, l.status, lo, hi);
    off = lo * l.cols;
    n = (hi - lo) * l.cols;
  }
  const uint16_t *in[Op::NIN];
  const uint16_t *src[3] = {s.in0, s.in1, s.in2};
#pragma unroll
  for (int k = 0; k < Op::NIN; ++k) in[k] = src[k] + off;
  uint16_t *out[Op::NOUT];
  uint16_t *dst[2] = {s.out0, s.out1};
#pragma unroll
  for (int k = 0; k < Op::NOUT; ++k) out[k] = dst[k] + off;

  int64_t head = n;
  if (l.vec) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(in[0]);
    head = (int64_t)(((16u - (a & 15u)) & 15u) >> 1);
    if (head > n) head = n;
  }
  const int64_t nvec = (n - head) >> 3;
  const int64_t body_end = head + (nvec << 3);
#pragma unroll 1
  for (int64_t base = (int64_t)blockIdx.x * (kThreads * U) + threadIdx.x; base < nvec;
       base += (int64_t)gridDim.x * (kThreads * U)) {
    uint4 r[U][Op::NIN];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = base + u * kThreads;
      if (i < nvec) {
#pragma unroll
        for (int k = 0; k < Op::NIN; ++k) r[u][k] = ld_stream(in[k] + head + (i << 3));
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = base + u * kThreads;
      if (i < nvec) {
        uint4 o[Op::NOUT];
        apply_chunk<Op>(r[u], o, p);
#pragma unroll
        for (int k = 0; k < Op::NOUT; ++k) st_stream(out[k] + head + (i << 3), o[k]);
      }
    }
  }
  const int64_t ntail = n - body_end;
#pragma unroll 1
  for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < head + ntail;
       i += (int64_t)gridDim.x * kThreads) {
    const int64_t e = i < head ? i : body_end + (i - head);
    apply_one<Op>(in, out, e, p);
  }
  pdl_release();
}

// Bytes m .. m + 15 (m even, 0..14) of the 32-byte window lo:hi, little
// endian: the 16-byte chunk that starts m bytes into an aligned window.
__device__ __forceinline__ uint4 realign16(const uint4 &lo, const uint4 &hi, uint32_t m) {
  const uint32_t sh = (m & 3u) * 8u;
  uint32_t w0, w1, w2, w3, w4;
  switch (m >> 2) {
    case 0: w0 = lo.x; w1 = lo.y; w2 = lo.z; w3 = lo.w; w4 = hi.x; break;
    case 1: w0 = lo.y; w1 = lo.z; w2 = lo.w; w3 = hi.x; w4 = hi.y; break;
    case 2: w0 = lo.z; w1 = lo.w; w2 = hi.x; w3 = hi.y; w4 = hi.z; break;
    default: w0 = lo.w; w1 = hi.x; w2 = hi.y; w3 = hi.z; w4 = hi.w; break;
  }
  return make_uint4(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh),
                    __funnelshift_r(w2, w3, sh), __funnelshift_r(w3, w4, sh));
}

// Flat / ragged calls whose inputs sit at other addresses modulo 16 than
// the output (a view that starts at an odd element, say), all outputs alike:
// the output moves in aligned 16-byte chunks, and each input chunk is
// assembled from the two aligned 16-byte chunks that straddle it, shifted by
// that input's constant byte offset -- every access stays a 16-byte access
// instead of falling back to one element per load.  The first and the last
// output chunks take the scalar path with the head and tail, so that no
// window reaches outside an input: chunk i reads input bytes from
// floor16(start + 2 (head + 8 i)) >= start + 2 (head - 7) > start (head >= 8)
// to at most start + 2 (head + 8 (i + 2)) <= start + 2 n (i <= nvec - 2 of
// the whole chunks).
template <class Op>
__global__ void __launch_bounds__(kThreads) realign_kernel(Streams s, Layout l,
                                                           typename Op::Params p) {
  pdl_wait();
  constexpr int U = chunks_per_thread<Op>();
  int64_t n = l.n, off = 0;
  if (l.mode == kRagged) {
    int64_t lo, hi;
    ragged_rows(l.seg, l.nseg, l.cap_rows, l.status, lo, hi);
    off = lo * l.cols;
    n = (hi - lo) * l.cols;
  }
  const uint16_t *in[Op::NIN];
  const uint16_t *src[3] = {s.in0, s.in1, s.in2};
#pragma unroll
  for (int k = 0; k < Op::NIN; ++k) in[k] = src[k] + off;
  uint16_t *out[Op::NOUT];
  uint16_t *dst[2] = {s.out0, s.out1};
#pragma unroll
  for (int k = 0; k < Op::NOUT; ++k) out[k] = dst[k] + off;

  const uintptr_t ao = reinterpret_cast<uintptr_t>(out[0]);
  int64_t head = (int64_t)(((16u - (ao & 15u)) & 15u) >> 1) + 8;
  if (head > n) head = n;
  int64_t nvec = ((n - head) >> 3) - 1;
  if (nvec < 0) nvec = 0;
  const int64_t body_end = head + (nvec << 3);
  uint32_t m[Op::NIN];
#pragma unroll
  for (int k = 0; k < Op::NIN; ++k)
    m[k] = (uint32_t)(reinterpret_cast<uintptr_t>(in[k] + head) & 15u);
#pragma unroll 1
  for (int64_t base = (int64_t)blockIdx.x * (kThreads * U) + threadIdx.x; base < nvec;
       base += (int64_t)gridDim.x * (kThreads * U)) {
    uint4 lo[U][Op::NIN], hi[U][Op::NIN];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = base + u * kThreads;
      if (i < nvec) {
#pragma unroll
        for (int k = 0; k < Op::NIN; ++k) {
          const uintptr_t a =
              reinterpret_cast<uintptr_t>(in[k] + head + (i << 3)) & ~uintptr_t(15);
          lo[u][k] = ld_stream(reinterpret_cast<const uint16_t *>(a));
          hi[u][k] = m[k] ? ld_stream(reinterpret_cast<const uint16_t *>(a + 16)) : lo[u][k];
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = base + u * kThreads;
      if (i < nvec) {
        uint4 x[Op::NIN], o[Op::NOUT];
#pragma unroll
        for (int k = 0; k < Op::NIN; ++k) x[k] = realign16(lo[u][k], hi[u][k], m[k]);
        apply_chunk<Op>(x, o, p);
#pragma unroll
        for (int k = 0; k < Op::NOUT; ++k) st_stream(out[k] + head + (i << 3), o[k]);
      }
    }
  }
  const int64_t ntail = n - body_end;
#pragma unroll 1
  for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < head + ntail;
       i += (int64_t)gridDim.x * kThreads) {
    const int64_t e = i < head ? i : body_end + (i - head);
    apply_one<Op>(in, out, e, p);
  }
  pdl_release();
}

// Dense: the common layouts with 32-bit indices, no layout branches and no
// loop (the grid covers the body exactly once).
//   kDenseFlat    n < 2^31 contiguous elements, every stream on a 16-byte
//                 boundary; the last block also evaluates the n mod 8 tail.
//   kDenseRagged  the rows read from the device offsets (cols % 8 == 0 and
//                 cap_rows * cols < 2^31, so every row starts on a 16-byte
//                 boundary and there is no tail); the grid covers cap_rows and
//                 blocks past the last row only return.
//   kDenseRows    rows x cols with a leading dimension per stream, every row
//                 start on a 16-byte boundary and every extent below 2^31
//                 elements (e.g. the gate and up halves of one [T, 2H]
//                 buffer); the row of a chunk comes from a multiply and a
//                 shift instead of a division.
enum DenseMode { kDenseFlat = 0, kDenseRagged = 1, kDenseRows = 2 };
enum ReleaseAt { kReleaseAfterLoads = 1, kReleaseAtEnd = 2 };

struct DenseArgs {
  uint32_t nvec, ntail;            // chunks of 8 elements; flat tail elements
  uint32_t release_at;              // where dependents are released: kRelease*
  const int32_t *seg;              // ragged: device offsets, their count,
  int32_t nseg, cap_rows;          //   the row capacity and the status word
  int32_t *status;
  uint32_t cols;                   // ragged / rows: elements per row
  uint32_t cpr, mul, shift;        // rows: chunks per row and floor(c / cpr) =
                                   //   (c * mul) >> shift for every c < 2^31
  uint32_t ld_in[3], ld_out[2];    // rows: leading dimensions in elements
};

// Division constants for numerators below 2^31 (the round-up reciprocal:
// with l = ceil(log2 d) and m = ceil(2^(31+l) / d), m * d lies in
// [2^(31+l), 2^(31+l) + 2^l), which makes floor(n m / 2^(31+l)) = floor(n / d)).
inline void row_divisor(uint32_t d, uint32_t &mul, uint32_t &shift) {
  uint32_t l = 0;
  while ((uint64_t(1) << l) < d) ++l;
  mul = (uint32_t)(((uint64_t(1) << (31 + l)) + d - 1) / d);
  shift = 31 + l;
}

// Element offset of chunk i (the flat form stays one wide multiply-add).
template <int MODE>
__device__ __forceinline__ size_t chunk_offset(uint32_t i, const DenseArgs &a, uint32_t ld) {
  if constexpr (MODE == kDenseRows) {
    const uint32_t row = (uint32_t)(((uint64_t)i * a.mul) >> a.shift);
    return (size_t)(row * ld + (i - row * a.cpr) * 8);
  } else {
    return (size_t)i * 8;
  }
}

template <class Op, int MODE, int U>
__global__ void __launch_bounds__(kThreads) dense_kernel(Streams s, DenseArgs a,
                                                         typename Op::Params p) {
  pdl_wait();
  const uint16_t *src[3] = {s.in0, s.in1, s.in2};
  uint16_t *dst[2] = {s.out0, s.out1};
  uint32_t nvec = a.nvec;
  if constexpr (MODE == kDenseRagged) {
    int64_t lo, hi;
    ragged_rows(a.seg, a.nseg, a.cap_rows, a.status, lo, hi);
    const size_t off = (size_t)lo * a.cols;
#pragma unroll
    for (int k = 0; k < Op::NIN; ++k) src[k] += off;
#pragma unroll
    for (int k = 0; k < Op::NOUT; ++k) dst[k] += off;
    nvec = (uint32_t)(((uint64_t)(hi - lo) * a.cols) >> 3);
  }
  const uint32_t base = blockIdx.x * (uint32_t)(kThreads * U) + threadIdx.x;
  uint4 r[U][Op::NIN];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const uint32_t i = base + u * kThreads;
    if (i < nvec) {
#pragma unroll
      for (int k = 0; k < Op::NIN; ++k)
        r[u][k] = ld_stream(src[k] + chunk_offset<MODE>(i, a, a.ld_in[k]));
    }
  }
  if (a.release_at == kReleaseAfterLoads) pdl_release();
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const uint32_t i = base + u * kThreads;
    if (i < nvec) {
      uint4 o[Op::NOUT];
      apply_chunk<Op>(r[u], o, p);
#pragma unroll
      for (int k = 0; k < Op::NOUT; ++k)
        st_stream(dst[k] + chunk_offset<MODE>(i, a, a.ld_out[k]), o[k]);
    }
  }
  if (MODE == kDenseFlat && a.ntail != 0 && blockIdx.x == gridDim.x - 1 &&
      threadIdx.x < a.ntail) {
    const uint16_t *in[Op::NIN];
    uint16_t *out[Op::NOUT];
#pragma unroll
    for (int k = 0; k < Op::NIN; ++k) in[k] = src[k];
#pragma unroll
    for (int k = 0; k < Op::NOUT; ++k) out[k] = dst[k];
    apply_one<Op>(in, out, (int64_t)nvec * 8 + threadIdx.x, p);
  }
  if (a.release_at == kReleaseAtEnd) pdl_release();
}

// Strided: rows x cols with a leading dimension per stream (a separate
// kernel so that its index arithmetic does not weigh on the flat path).
template <class Op>
__global__ void __launch_bounds__(kThreads) strided_kernel(Streams s, Layout l,
                                                           typename Op::Params p) {
  pdl_wait();
  const uint16_t *src[3] = {s.in0, s.in1, s.in2};
  uint16_t *dst[2] = {s.out0, s.out1};
  const int64_t gid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  if (l.vec) {
    const int64_t cpr = l.cols >> 3;
    const int64_t total = l.rows * cpr;
#pragma unroll 1
    for (int64_t c = gid; c < total; c += stride) {
      const int64_t row = c / cpr;
      const int64_t col = (c - row * cpr) << 3;
      uint4 r[Op::NIN], o[Op::NOUT];
#pragma unroll
      for (int k = 0; k < Op::NIN; ++k) r[k] = ld_stream(src[k] + row * l.ld_in[k] + col);
      apply_chunk<Op>(r, o, p);
#pragma unroll
      for (int k = 0; k < Op::NOUT; ++k) st_stream(dst[k] + row * l.ld_out[k] + col, o[k]);
    }
  } else {
    const int64_t total = l.rows * l.cols;
#pragma unroll 1
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
  pdl_release();
}

// Blocks for a launch: `per_thread` elements per thread, covering the work
// in one pass (measured on GB300: a one-pass grid streams 8-10 % faster than
// a persistent grid striding over the tensor).
int64_t grid_for(const Layout &l, int per_thread);
// Streaming multiprocessors of the calling thread's current device (cached).
int sm_count();

// Launch with the programmatic-stream-serialisation attribute (see pdl_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), int64_t blocks, int threads, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Chunks per thread and release point of a dense-kernel launch over nvec
// chunks (the rules above chunks_per_thread and pdl_wait).
struct DenseShape {
  int u;
  uint32_t release_at;
};
template <class Op>
DenseShape dense_shape(int64_t nvec) {
  const int64_t sms = sm_count();
  const int64_t one = (nvec + kThreads - 1) / kThreads;             // U = 1 grid
  const int64_t two = (nvec + 2 * kThreads - 1) / (2 * kThreads);   // U = 2 grid
  if constexpr (Op::NIN == 1) {
    if (two < 2 * sms) return {1, kReleaseAfterLoads};
    return {2, kReleaseAtEnd};
  } else if constexpr (Op::NIN == 2 && Op::NOUT == 1) {
    if (one <= 8 * sms) return {1, kReleaseAfterLoads};
    if (two <= kTwoChunkMaxBlocksPerSm * sms) return {2, kReleaseAtEnd};
    return {1, kReleaseAtEnd};
  } else {
    return {1, kReleaseAtEnd};
  }
}

// A dense-kernel launch in the shape dense_shape gives.
template <class Op, int MODE>
cudaError_t launch_dense(cudaStream_t stream, const Streams &s, DenseArgs a,
                         const typename Op::Params &p) {
  const DenseShape sh = dense_shape<Op>(a.nvec);
  a.release_at = sh.release_at;
  const int64_t per = (int64_t)kThreads * sh.u;
  int64_t blocks = ((int64_t)a.nvec + per - 1) / per;
  if (blocks < 1) blocks = 1;
  if constexpr (Op::NIN == 1 || (Op::NIN == 2 && Op::NOUT == 1)) {
    if (sh.u == 2) return launch_pdl(dense_kernel<Op, MODE, 2>, blocks, kThreads, stream, s, a, p);
  }
  return launch_pdl(dense_kernel<Op, MODE, 1>, blocks, kThreads, stream, s, a, p);
}

// Every stream of s starts on a 16-byte boundary (unused streams are null).
inline bool aligned16(const Streams &s) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(s.in0) | reinterpret_cast<uintptr_t>(s.in1) |
                      reinterpret_cast<uintptr_t>(s.in2) | reinterpret_cast<uintptr_t>(s.out0) |
                      reinterpret_cast<uintptr_t>(s.out1);
  return (a & 15u) == 0;
}

// Launch an op on a flat / ragged layout (every op) or, when the op allows
// it (TWO_D), on a strided one.
template <class Op>
cudaError_t launch_op(const Streams &s, const Layout &l, const typename Op::Params &p,
                      cudaStream_t stream) {
  const int64_t lim = int64_t(1) << 31;
  if constexpr (Op::TWO_D) {
    if (l.mode == kStrided) {
      // two-output operations (the SwiGLU backward) keep the strided kernel
      // above 2^23 chunks (67 M elements): within +-2 % of the rows mode at
      // 117 M on GB300, while the rows mode wins below (3-22 % at 4-56 M on
      // fused gate-up halves) and for every single-output operation
      bool fast = l.vec && l.rows * (l.cols >> 3) < (Op::NOUT == 1 ? lim : kRowsTwoOutMax);
      for (int k = 0; k < 3; ++k) fast &= (l.rows - 1) * l.ld_in[k] + l.cols < lim;
      for (int k = 0; k < 2; ++k) fast &= (l.rows - 1) * l.ld_out[k] + l.cols < lim;
      if (fast) {
        DenseArgs a{};
        a.cpr = (uint32_t)(l.cols >> 3);
        a.nvec = (uint32_t)(l.rows * a.cpr);
        row_divisor(a.cpr, a.mul, a.shift);
        for (int k = 0; k < 3; ++k) a.ld_in[k] = (uint32_t)l.ld_in[k];
        for (int k = 0; k < 2; ++k) a.ld_out[k] = (uint32_t)l.ld_out[k];
        return launch_dense<Op, kDenseRows>(stream, s, a, p);
      }
      const int64_t blocks = grid_for(l, l.vec ? 8 : 1);
      return launch_pdl(strided_kernel<Op>, blocks, kThreads, stream, s, l, p);
    }
  }
  if (l.mode == kStrided) return cudaErrorInvalidValue;
  if (l.mode == kFlat && l.n < lim && aligned16(s)) {
    DenseArgs a{};
    a.nvec = (uint32_t)(l.n >> 3);
    a.ntail = (uint32_t)(l.n & 7);
    return launch_dense<Op, kDenseFlat>(stream, s, a, p);
  }
  if (l.mode == kRagged && l.cols % 8 == 0 && l.cap_rows * l.cols < lim && aligned16(s)) {
    DenseArgs a{};
    a.seg = l.seg;
    a.nseg = l.nseg;
    a.cap_rows = (int32_t)l.cap_rows;
    a.status = l.status;
    a.cols = (uint32_t)l.cols;
    // the row range is known on the device only: the grid and shape are the
    // capacity's (the kernel takes its own chunk count from the offsets)
    a.nvec = (uint32_t)((l.cap_rows * l.cols) >> 3);
    return launch_dense<Op, kDenseRagged>(stream, s, a, p);
  }
  // streams that disagree modulo 16 while the outputs agree: realigned
  // 16-byte accesses instead of one element per load
  if (!l.vec && (Op::NOUT == 1 || ((reinterpret_cast<uintptr_t>(s.out0) ^
                                    reinterpret_cast<uintptr_t>(s.out1)) & 15u) == 0)) {
    const int64_t blocks = grid_for(l, 8 * chunks_per_thread<Op>());
    return launch_pdl(realign_kernel<Op>, blocks, kThreads, stream, s, l, p);
  }
  const int64_t blocks = grid_for(l, l.vec ? 8 * chunks_per_thread<Op>() : 1);
  return launch_pdl(stream_kernel<Op>, blocks, kThreads, stream, s, l, p);
}

}  // namespace dev
}  // namespace polyact
