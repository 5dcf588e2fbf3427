// capi.cpp -- the extern "C" boundary of libpolyact (declared in
// include/polyact.h): argument validation, the program registry and the
// dispatch to the CUDA launchers.  Every check happens on the host before any
// CUDA call, so invalid arguments never reach the GPU.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/polyact.h"
#include "fit_internal.h"
#include "launch.h"
#include "softhalf.h"

using namespace polyact;

namespace {

thread_local int t_last_cuda_error = 0;

std::mutex g_reg_mu;
bool g_have[4][2][2];
poly_program g_prog[4][2][2];
std::atomic<int> g_swiglu_variant{POLY_SWIGLU_DIRECT};

bool valid_fn(int fn) { return fn >= POLY_SIGMOID && fn <= POLY_GELU; }
bool valid_dir(int d) { return d == POLY_FWD || d == POLY_BWD; }
bool valid_dtype(int dt) { return dt == POLY_F16 || dt == POLY_BF16; }
bool valid_ctrl(int v) { return v == POLY_CTRL_FP32 || v == POLY_CTRL_PACKED; }
bool valid_swiglu_variant(int v) { return v == POLY_SWIGLU_DIRECT || v == POLY_SWIGLU_SIGMOID; }

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return POLY_OK;
  t_last_cuda_error = (int)e;
  return POLY_ECUDA;
}

// Injected launch failures (poly_debug_fail_launches).
std::mutex g_fail_mu;
int g_fail_pending = 0;
int g_fail_code = 0;

// Runs the launch unless an injected failure is pending, in which case the
// launch is skipped and that failure is reported instead.
template <class Launch>
int launch_status(Launch &&launch) {
  {
    std::lock_guard<std::mutex> lk(g_fail_mu);
    if (g_fail_pending > 0) {
      --g_fail_pending;
      return cuda_status((cudaError_t)g_fail_code);
    }
  }
  return cuda_status(launch());
}

DevProg dev_prog(const poly_program &p) {
  DevProg d;
  std::memset(&d, 0, sizeof(d));
  for (int j = 0; j <= p.degree; ++j) d.c[j] = (uint32_t)p.coef[j] * 0x00010001u;
  d.lc = (uint32_t)p.lc_bits * 0x00010001u;
  return d;
}

int check_program(const poly_program &p) {
  if (!valid_fn(p.fn) || !valid_dir(p.dir) || !valid_dtype(p.dtype)) return POLY_ENOPROG;
  // even programs may have degree 2 (derived from a degree-3 forward program)
  const int min_degree = p.form == POLY_FORM_E ? 2 : POLY_MIN_DEGREE;
  if (p.degree < min_degree || p.degree > POLY_MAX_DEGREE) return POLY_ENOPROG;
  if (p.form != form_of_fn(p.fn, p.dir)) return POLY_ENOPROG;
  if (p.version != POLY_PROGRAM_VERSION) return POLY_ENOPROG;
  const bool even = p.form == POLY_FORM_E;
  if (!even && (p.coef[0] & 0x7FFF) != 0) return POLY_ENOPROG;   // c_0 = f(0) = 0
  // the clamp: a finite positive target-format value, lc its exact value, and
  // no further than one unit past the fit interval (Lc <= Li + 1, §3.2 step 6)
  const double lc = to_double(p.lc_bits, p.dtype);
  if (!std::isfinite(lc) || !(lc > 0.0) || lc != p.lc) return POLY_ENOPROG;
  if (!std::isfinite(p.li) || !(p.li > 0.0) || !(lc <= p.li + 1.0)) return POLY_ENOPROG;
  return POLY_OK;
}

// Largest extent, in elements, that any call accepts (2^46, far beyond the
// memory a GB300 system can address).  Larger sizes, and tensors whose last
// byte would wrap the address space, are rejected, so that no size or span
// computed below can overflow.
constexpr int64_t kMaxElems = int64_t(1) << 46;

// a * b for non-negative sizes, or -1 if it exceeds kMaxElems.
int64_t checked_mul(int64_t a, int64_t b) {
  int64_t r;
  if (a < 0 || b < 0 || __builtin_mul_overflow(a, b, &r) || r > kMaxElems) return -1;
  return r;
}

// Byte span [lo, hi) of a tensor, as rows of `width` bytes whose starts are
// `pitch` bytes apart (one row for a flat tensor); ok is false when its
// extent is too large or its end wraps the address space.
struct Span {
  uintptr_t lo, hi;
  bool ok;
  uintptr_t pitch, width;
};

Span span_bytes(const void *p, int64_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  uintptr_t hi = 0;
  const bool ok = bytes >= 0 && !__builtin_add_overflow(a, (uintptr_t)bytes, &hi);
  return {a, hi, ok, (uintptr_t)bytes, (uintptr_t)bytes};
}

Span span_flat(const void *p, int64_t n) {
  if (n < 0 || n > kMaxElems) return {0, 0, false, 0, 0};
  return span_bytes(p, n * 2);
}

// rows x cols with leading dimension ld (all at most kMaxElems, ld >= cols).
Span span_2d(const void *p, int64_t rows, int64_t cols, int64_t ld) {
  const int64_t body = checked_mul(rows - 1, ld);
  if (body < 0 || cols > kMaxElems || body + cols > kMaxElems) return {0, 0, false, 0, 0};
  Span s = span_bytes(p, (body + cols) * 2);
  if (rows > 1) {
    s.pitch = (uintptr_t)ld * 2;
    s.width = (uintptr_t)cols * 2;
  }
  return s;
}

// Whether two tensors share a byte.  Extents that intersect can still be
// disjoint when both are row sets of the same pitch and one's rows fall in
// the other's gaps (the gate and up halves of one [T, 2H] buffer).
bool overlaps(const Span &a, const Span &b) {
  if (!(a.lo < b.hi && b.lo < a.hi)) return false;
  if (a.pitch == b.pitch && a.pitch > a.width && b.pitch > b.width) {
    const Span &f = a.lo <= b.lo ? a : b;
    const Span &g = a.lo <= b.lo ? b : a;
    const uintptr_t d = (g.lo - f.lo) % f.pitch;
    if (d >= f.width && d + g.width <= f.pitch) return false;
  }
  return true;
}

bool same_view(const Span &a, const Span &b) {
  return a.lo == b.lo && a.hi == b.hi && a.pitch == b.pitch && a.width == b.width;
}

// Every span is valid; outputs may coincide exactly with an input (in
// place), never partially overlap anything, and never overlap each other.
bool aliasing_ok(const Span *in, int nin, const Span *out, int nout) {
  for (int i = 0; i < nin; ++i)
    if (!in[i].ok) return false;
  for (int o = 0; o < nout; ++o)
    if (!out[o].ok) return false;
  for (int o = 0; o < nout; ++o) {
    for (int i = 0; i < nin; ++i) {
      if (!overlaps(out[o], in[i])) continue;
      if (same_view(out[o], in[i])) continue;
      return false;
    }
    for (int o2 = o + 1; o2 < nout; ++o2)
      if (overlaps(out[o], out[o2])) return false;
  }
  return true;
}

bool even_address(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 1u) == 0; }

// Flat layout of n contiguous elements: the 16-byte path needs every stream
// at the same address modulo 16 (the kernel derives the scalar head).
Layout flat_layout(const void *const *ptrs, int np, int64_t n) {
  Layout l;
  std::memset(&l, 0, sizeof(l));
  l.mode = kFlat;
  l.n = n;
  const uintptr_t m = reinterpret_cast<uintptr_t>(ptrs[0]) & 15u;
  l.vec = 1;
  for (int i = 1; i < np; ++i)
    if ((reinterpret_cast<uintptr_t>(ptrs[i]) & 15u) != m) l.vec = 0;
  return l;
}

int registry_get(int fn, int dir, int dtype, poly_program *out) {
  {
    std::lock_guard<std::mutex> lk(g_reg_mu);
    if (g_have[fn][dir][dtype]) {
      *out = g_prog[fn][dir][dtype];
      return POLY_OK;
    }
  }
  poly_program p;
  int st = poly_fit(fn, dir, dtype, poly_default_degree(fn, dir), nullptr, &p);
  if (st != POLY_OK) return st;
  std::lock_guard<std::mutex> lk(g_reg_mu);
  if (!g_have[fn][dir][dtype]) {
    g_prog[fn][dir][dtype] = p;
    g_have[fn][dir][dtype] = true;
  }
  *out = g_prog[fn][dir][dtype];
  return POLY_OK;
}

// Shared validation + layout for the dense 2-D SwiGLU calls.
int swiglu_layout(const void *const *in, const int64_t *ld_in, int nin, void *const *out,
                  const int64_t *ld_out, int nout, int64_t rows, int64_t cols, Layout *l) {
  if (rows < 0 || cols < 0 || rows > kMaxElems || cols > kMaxElems) return POLY_EINVAL;
  for (int i = 0; i < nin; ++i)
    if (ld_in[i] < cols || ld_in[i] > kMaxElems) return POLY_EINVAL;
  for (int i = 0; i < nout; ++i)
    if (ld_out[i] < cols || ld_out[i] > kMaxElems) return POLY_EINVAL;
  if (rows == 0 || cols == 0) return 1;   // nothing to do
  const void *all[5];
  Span si[3], so[2];
  for (int i = 0; i < nin; ++i) {
    if (in[i] == nullptr || !even_address(in[i])) return POLY_EINVAL;
    si[i] = span_2d(in[i], rows, cols, ld_in[i]);
    all[i] = in[i];
  }
  for (int i = 0; i < nout; ++i) {
    if (out[i] == nullptr || !even_address(out[i])) return POLY_EINVAL;
    so[i] = span_2d(out[i], rows, cols, ld_out[i]);
    all[nin + i] = out[i];
  }
  if (!aliasing_ok(si, nin, so, nout)) return POLY_EINVAL;
  bool contiguous = true;
  for (int i = 0; i < nin; ++i) contiguous &= (ld_in[i] == cols) || rows == 1;
  for (int i = 0; i < nout; ++i) contiguous &= (ld_out[i] == cols) || rows == 1;
  if (contiguous) {
    *l = flat_layout(all, nin + nout, rows * cols);
    return POLY_OK;
  }
  std::memset(l, 0, sizeof(*l));
  l->mode = kStrided;
  l->rows = rows;
  l->cols = cols;
  bool vec = (cols % 8) == 0;
  for (int i = 0; i < nin; ++i) {
    l->ld_in[i] = ld_in[i];
    vec &= (reinterpret_cast<uintptr_t>(in[i]) & 15u) == 0 && (ld_in[i] % 8) == 0;
  }
  for (int i = 0; i < nout; ++i) {
    l->ld_out[i] = ld_out[i];
    vec &= (reinterpret_cast<uintptr_t>(out[i]) & 15u) == 0 && (ld_out[i] % 8) == 0;
  }
  l->vec = vec ? 1 : 0;
  return POLY_OK;
}

int ragged_layout(const void *const *in, int nin, void *const *out, int nout,
                  const int32_t *seg_off, int num_segments, int64_t cap_rows, int64_t cols,
                  int32_t *status, Layout *l) {
  if (cap_rows < 0 || cols < 0 || num_segments < 0 || seg_off == nullptr) return POLY_EINVAL;
  if (cap_rows == 0 || cols == 0) return 1;
  const void *all[5];
  Span si[3], so[2];
  const int64_t n = checked_mul(cap_rows, cols);
  if (n < 0) return POLY_EINVAL;
  for (int i = 0; i < nin; ++i) {
    if (in[i] == nullptr || !even_address(in[i])) return POLY_EINVAL;
    si[i] = span_flat(in[i], n);
    all[i] = in[i];
  }
  for (int i = 0; i < nout; ++i) {
    if (out[i] == nullptr || !even_address(out[i])) return POLY_EINVAL;
    so[i] = span_flat(out[i], n);
    all[nin + i] = out[i];
  }
  if (!aliasing_ok(si, nin, so, nout)) return POLY_EINVAL;
  *l = flat_layout(all, nin + nout, n);
  l->mode = kRagged;
  l->seg = seg_off;
  l->nseg = num_segments;
  l->cap_rows = cap_rows;
  l->cols = cols;
  l->status = status;
  return POLY_OK;
}

// Programs of the current SwiGLU variant: the SiLU program (and, for the
// direct backward, the centred SiLU derivative), or the sigmoid program.
int swiglu_programs(int variant, int dtype, bool need_bwd, poly_program *s, poly_program *sd) {
  if (variant == POLY_SWIGLU_SIGMOID) {
    int st = registry_get(POLY_SIGMOID, POLY_FWD, dtype, s);
    *sd = *s;
    return st;
  }
  int st = registry_get(POLY_SILU, POLY_FWD, dtype, s);
  if (st != POLY_OK) return st;
  if (need_bwd) return registry_get(POLY_SILU, POLY_BWD, dtype, sd);
  *sd = *s;
  return POLY_OK;
}

}  // namespace

extern "C" {

const char *poly_status_str(int status) {
  switch (status) {
    case POLY_OK: return "POLY_OK";
    case POLY_EINVAL: return "POLY_EINVAL: invalid argument";
    case POLY_ENOPROG: return "POLY_ENOPROG: inconsistent program descriptor";
    case POLY_ECUDA: return "POLY_ECUDA: CUDA call or kernel launch failed";
    case POLY_ENOFIT: return "POLY_ENOFIT: no candidate passed the fitter's gates";
  }
  return "unknown status";
}

int poly_last_cuda_error(void) { return t_last_cuda_error; }

int poly_abi_version(void) { return 4; }

int poly_debug_fail_launches(int cuda_error, int count) {
  if (cuda_error <= 0 || count < 0) return POLY_EINVAL;
  std::lock_guard<std::mutex> lk(g_fail_mu);
  const int pending = g_fail_pending;
  g_fail_pending = count;
  g_fail_code = cuda_error;
  return pending;
}

int poly_form_of(int fn, int dir) {
  if (!valid_fn(fn) || !valid_dir(dir)) return POLY_EINVAL;
  return form_of_fn(fn, dir);
}

int poly_default_degree(int fn, int dir) {
  if (!valid_fn(fn) || !valid_dir(dir)) return POLY_EINVAL;
  if (dir == POLY_BWD) return 4;
  static const int fwd[4] = {3, 4, 3, 5};
  return fwd[fn];
}

int poly_fit_defaults(poly_fit_opts *o) {
  if (o == nullptr) return POLY_EINVAL;
  o->li_min = 1.0;
  o->li_max = 12.0;
  o->li_step = 0.25;
  o->lc_min = 1.0;
  o->lc_step = 0.25;
  o->n_nodes = 2000;
  o->n_score = 8000;
  o->score_hi = 12.0;
  o->top_k = 0;
  o->lc_refine_ulps = 0;
  return POLY_OK;
}

int poly_fit(int fn, int dir, int dtype, int degree, const poly_fit_opts *opts,
             poly_program *out) {
  if (!valid_fn(fn) || !valid_dir(dir) || !valid_dtype(dtype) || out == nullptr)
    return POLY_EINVAL;
  if (degree < POLY_MIN_DEGREE || degree > POLY_MAX_DEGREE) return POLY_EINVAL;
  poly_fit_opts o;
  if (opts == nullptr)
    poly_fit_defaults(&o);
  else
    o = *opts;
  if (!(o.li_min > 0) || !(o.li_step > 0) || !(o.li_max >= o.li_min) || !(o.lc_min > 0) ||
      !(o.lc_step > 0) || o.n_nodes < degree || o.n_score < 2 || !(o.score_hi > 0) ||
      o.top_k < 0 || o.lc_refine_ulps < 0 || o.lc_refine_ulps > 64 || o.li_max > 1e4 || (o.li_max - o.li_min) / o.li_step > 1e5)
    return POLY_EINVAL;
  return fit_program(fn, dir, dtype, degree, o, out);
}

int poly_derive_program(const poly_program *fwd, poly_program *out) {
  if (fwd == nullptr || out == nullptr) return POLY_EINVAL;
  int st = check_program(*fwd);
  if (st != POLY_OK) return st;
  if (fwd->dir != POLY_FWD || (fwd->form != POLY_FORM_O && fwd->form != POLY_FORM_CO))
    return POLY_EINVAL;
  return derive_program(*fwd, out);
}

int poly_set_program(const poly_program *p) {
  if (p == nullptr) return POLY_EINVAL;
  int st = check_program(*p);
  if (st != POLY_OK) return st;
  std::lock_guard<std::mutex> lk(g_reg_mu);
  g_prog[p->fn][p->dir][p->dtype] = *p;
  g_have[p->fn][p->dir][p->dtype] = true;
  return POLY_OK;
}

int poly_get_program(int fn, int dir, int dtype, poly_program *out) {
  if (!valid_fn(fn) || !valid_dir(dir) || !valid_dtype(dtype) || out == nullptr)
    return POLY_EINVAL;
  return registry_get(fn, dir, dtype, out);
}

int poly_set_swiglu_variant(int variant) {
  if (!valid_swiglu_variant(variant)) return POLY_EINVAL;
  g_swiglu_variant.store(variant);
  return POLY_OK;
}

int poly_get_swiglu_variant(void) { return g_swiglu_variant.load(); }

int poly_reset_programs(void) {
  std::lock_guard<std::mutex> lk(g_reg_mu);
  std::memset(g_have, 0, sizeof(g_have));
  return POLY_OK;
}

// ctrl < 0: the polynomial program; otherwise the MUFU control of that variant.
static int act_call(int ctrl, int kind, int fn, int dtype, const void *x, const void *dy,
                    void *y, int64_t n, poly_stream_t stream) {
  if (!valid_fn(fn) || !valid_dtype(dtype) || n < 0) return POLY_EINVAL;
  if (ctrl >= 0 && !valid_ctrl(ctrl)) return POLY_EINVAL;
  if (n == 0) return POLY_OK;
  const bool bwd = kind == kActBwd;
  if (x == nullptr || y == nullptr || (bwd && dy == nullptr)) return POLY_EINVAL;
  if (!even_address(x) || !even_address(y) || (bwd && !even_address(dy))) return POLY_EINVAL;
  Span si[2] = {span_flat(x, n), span_flat(bwd ? dy : x, n)};
  Span so[1] = {span_flat(y, n)};
  if (!aliasing_ok(si, bwd ? 2 : 1, so, 1)) return POLY_EINVAL;
  const void *ptrs[3] = {x, bwd ? dy : x, y};
  Layout l = flat_layout(ptrs, 3, n);
  Streams s{static_cast<const uint16_t *>(x), static_cast<const uint16_t *>(dy), nullptr,
            static_cast<uint16_t *>(y), nullptr};
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (ctrl >= 0)
    return launch_status([&] { return launch_ctrl(kind, dtype, fn, s, l, cs, ctrl); });
  poly_program p;
  int st = registry_get(fn, bwd ? POLY_BWD : POLY_FWD, dtype, &p);
  if (st != POLY_OK) return st;
  DevProg d = dev_prog(p);
  return launch_status(
      [&] { return launch_poly(kind, dtype, p.form, p.degree, 0, s, l, d, d, cs); });
}

int poly_act_fwd(int fn, int dtype, const void *x, void *y, int64_t n, poly_stream_t stream) {
  return act_call(-1, kActFwd, fn, dtype, x, nullptr, y, n, stream);
}

int poly_act_bwd(int fn, int dtype, const void *x, const void *dy, void *dx, int64_t n,
                 poly_stream_t stream) {
  return act_call(-1, kActBwd, fn, dtype, x, dy, dx, n, stream);
}

int poly_ctrl_act_fwd(int fn, int dtype, const void *x, void *y, int64_t n,
                      poly_stream_t stream) {
  return act_call(POLY_CTRL_FP32, kActFwd, fn, dtype, x, nullptr, y, n, stream);
}

int poly_ctrl_act_bwd(int fn, int dtype, const void *x, const void *dy, void *dx, int64_t n,
                      poly_stream_t stream) {
  return act_call(POLY_CTRL_FP32, kActBwd, fn, dtype, x, dy, dx, n, stream);
}

int poly_ctrl_act_fwd_v(int variant, int fn, int dtype, const void *x, void *y, int64_t n,
                        poly_stream_t stream) {
  if (!valid_ctrl(variant)) return POLY_EINVAL;
  return act_call(variant, kActFwd, fn, dtype, x, nullptr, y, n, stream);
}

int poly_ctrl_act_bwd_v(int variant, int fn, int dtype, const void *x, const void *dy, void *dx,
                        int64_t n, poly_stream_t stream) {
  if (!valid_ctrl(variant)) return POLY_EINVAL;
  return act_call(variant, kActBwd, fn, dtype, x, dy, dx, n, stream);
}

// ctrl < 0: the polynomial rule `variant`; otherwise the MUFU control `ctrl`.
static int swiglu_call(int ctrl, int variant, bool bwd, int dtype, const void *g, const void *u,
                       const void *dy, void *o0, void *o1, int64_t rows, int64_t cols,
                       const int64_t *ld_in, const int64_t *ld_out, poly_stream_t stream) {
  if (!valid_dtype(dtype)) return POLY_EINVAL;
  if (ctrl >= 0 ? !valid_ctrl(ctrl) : !valid_swiglu_variant(variant)) return POLY_EINVAL;
  const void *in[3] = {g, u, dy};
  void *out[2] = {o0, o1};
  Layout l;
  int st = swiglu_layout(in, ld_in, bwd ? 3 : 2, out, ld_out, bwd ? 2 : 1, rows, cols, &l);
  if (st == 1) return POLY_OK;
  if (st != POLY_OK) return st;
  Streams s{static_cast<const uint16_t *>(g), static_cast<const uint16_t *>(u),
            static_cast<const uint16_t *>(dy), static_cast<uint16_t *>(o0),
            static_cast<uint16_t *>(o1)};
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const int kind = bwd ? kSwigluBwd : kSwigluFwd;
  if (ctrl >= 0)
    return launch_status([&] { return launch_ctrl(kind, dtype, POLY_SILU, s, l, cs, ctrl); });
  poly_program ps, pd;
  st = swiglu_programs(variant, dtype, bwd, &ps, &pd);
  if (st != POLY_OK) return st;
  return launch_status([&] {
    return launch_poly(kind, dtype, ps.form, ps.degree, pd.degree, s, l, dev_prog(ps),
                       dev_prog(pd), cs, variant);
  });
}

int poly_swiglu_fwd_v(int variant, int dtype, const void *g, const void *u, void *y,
                      int64_t rows, int64_t cols, int64_t ldg, int64_t ldu, int64_t ldy,
                      poly_stream_t stream) {
  const int64_t li[3] = {ldg, ldu, cols}, lo[2] = {ldy, cols};
  return swiglu_call(-1, variant, false, dtype, g, u, nullptr, y, nullptr, rows, cols, li, lo,
                     stream);
}

int poly_swiglu_bwd_v(int variant, int dtype, const void *g, const void *u, const void *dy,
                      void *dg, void *du, int64_t rows, int64_t cols, int64_t ldg, int64_t ldu,
                      int64_t lddy, int64_t lddg, int64_t lddu, poly_stream_t stream) {
  const int64_t li[3] = {ldg, ldu, lddy}, lo[2] = {lddg, lddu};
  return swiglu_call(-1, variant, true, dtype, g, u, dy, dg, du, rows, cols, li, lo, stream);
}

int poly_swiglu_fwd(int dtype, const void *g, const void *u, void *y, int64_t rows,
                    int64_t cols, int64_t ldg, int64_t ldu, int64_t ldy, poly_stream_t stream) {
  return poly_swiglu_fwd_v(g_swiglu_variant.load(), dtype, g, u, y, rows, cols, ldg, ldu, ldy,
                           stream);
}

int poly_swiglu_bwd(int dtype, const void *g, const void *u, const void *dy, void *dg, void *du,
                    int64_t rows, int64_t cols, int64_t ldg, int64_t ldu, int64_t lddy,
                    int64_t lddg, int64_t lddu, poly_stream_t stream) {
  return poly_swiglu_bwd_v(g_swiglu_variant.load(), dtype, g, u, dy, dg, du, rows, cols, ldg,
                           ldu, lddy, lddg, lddu, stream);
}

int poly_ctrl_swiglu_fwd_v(int variant, int dtype, const void *g, const void *u, void *y,
                           int64_t rows, int64_t cols, int64_t ldg, int64_t ldu, int64_t ldy,
                           poly_stream_t stream) {
  if (!valid_ctrl(variant)) return POLY_EINVAL;
  const int64_t li[3] = {ldg, ldu, cols}, lo[2] = {ldy, cols};
  return swiglu_call(variant, 0, false, dtype, g, u, nullptr, y, nullptr, rows, cols, li, lo,
                     stream);
}

int poly_ctrl_swiglu_bwd_v(int variant, int dtype, const void *g, const void *u, const void *dy,
                           void *dg, void *du, int64_t rows, int64_t cols, int64_t ldg,
                           int64_t ldu, int64_t lddy, int64_t lddg, int64_t lddu,
                           poly_stream_t stream) {
  if (!valid_ctrl(variant)) return POLY_EINVAL;
  const int64_t li[3] = {ldg, ldu, lddy}, lo[2] = {lddg, lddu};
  return swiglu_call(variant, 0, true, dtype, g, u, dy, dg, du, rows, cols, li, lo, stream);
}

int poly_ctrl_swiglu_fwd(int dtype, const void *g, const void *u, void *y, int64_t rows,
                         int64_t cols, int64_t ldg, int64_t ldu, int64_t ldy,
                         poly_stream_t stream) {
  return poly_ctrl_swiglu_fwd_v(POLY_CTRL_FP32, dtype, g, u, y, rows, cols, ldg, ldu, ldy,
                                stream);
}

int poly_ctrl_swiglu_bwd(int dtype, const void *g, const void *u, const void *dy, void *dg,
                         void *du, int64_t rows, int64_t cols, int64_t ldg, int64_t ldu,
                         int64_t lddy, int64_t lddg, int64_t lddu, poly_stream_t stream) {
  return poly_ctrl_swiglu_bwd_v(POLY_CTRL_FP32, dtype, g, u, dy, dg, du, rows, cols, ldg, ldu,
                                lddy, lddg, lddu, stream);
}

static int ragged_call(int variant, bool bwd, int dtype, const void *g, const void *u,
                       const void *dy, void *o0, void *o1, const int32_t *seg_off,
                       int num_segments, int64_t cap_rows, int64_t cols, int32_t *status,
                       poly_stream_t stream) {
  if (!valid_dtype(dtype) || !valid_swiglu_variant(variant)) return POLY_EINVAL;
  const void *in[3] = {g, u, dy};
  void *out[2] = {o0, o1};
  Layout l;
  int st = ragged_layout(in, bwd ? 3 : 2, out, bwd ? 2 : 1, seg_off, num_segments, cap_rows,
                         cols, status, &l);
  if (st == 1) return POLY_OK;
  if (st != POLY_OK) return st;
  poly_program ps, pd;
  st = swiglu_programs(variant, dtype, bwd, &ps, &pd);
  if (st != POLY_OK) return st;
  Streams s{static_cast<const uint16_t *>(g), static_cast<const uint16_t *>(u),
            static_cast<const uint16_t *>(dy), static_cast<uint16_t *>(o0),
            static_cast<uint16_t *>(o1)};
  return launch_status([&] {
    return launch_poly(bwd ? kSwigluBwd : kSwigluFwd, dtype, ps.form, ps.degree, pd.degree, s,
                       l, dev_prog(ps), dev_prog(pd), reinterpret_cast<cudaStream_t>(stream),
                       variant);
  });
}

int poly_swiglu_fwd_ragged_v(int variant, int dtype, const void *g, const void *u, void *y,
                             const int32_t *seg_off, int num_segments, int64_t cap_rows,
                             int64_t cols, int32_t *status, poly_stream_t stream) {
  return ragged_call(variant, false, dtype, g, u, nullptr, y, nullptr, seg_off, num_segments,
                     cap_rows, cols, status, stream);
}

int poly_swiglu_bwd_ragged_v(int variant, int dtype, const void *g, const void *u,
                             const void *dy, void *dg, void *du, const int32_t *seg_off,
                             int num_segments, int64_t cap_rows, int64_t cols, int32_t *status,
                             poly_stream_t stream) {
  return ragged_call(variant, true, dtype, g, u, dy, dg, du, seg_off, num_segments, cap_rows,
                     cols, status, stream);
}

int poly_swiglu_fwd_ragged(int dtype, const void *g, const void *u, void *y,
                           const int32_t *seg_off, int num_segments, int64_t cap_rows,
                           int64_t cols, int32_t *status, poly_stream_t stream) {
  return poly_swiglu_fwd_ragged_v(g_swiglu_variant.load(), dtype, g, u, y, seg_off,
                                  num_segments, cap_rows, cols, status, stream);
}

int poly_swiglu_bwd_ragged(int dtype, const void *g, const void *u, const void *dy, void *dg,
                           void *du, const int32_t *seg_off, int num_segments, int64_t cap_rows,
                           int64_t cols, int32_t *status, poly_stream_t stream) {
  return poly_swiglu_bwd_ragged_v(g_swiglu_variant.load(), dtype, g, u, dy, dg, du, seg_off,
                                  num_segments, cap_rows, cols, status, stream);
}

int poly_ragged_zero_outside(void *out, const int32_t *seg_off, int num_segments,
                             int64_t cap_rows, int64_t cols, poly_stream_t stream) {
  if (seg_off == nullptr || num_segments < 0 || cap_rows < 0 || cols < 0) return POLY_EINVAL;
  if (cap_rows == 0 || cols == 0) return POLY_OK;
  const int64_t n = checked_mul(cap_rows, cols);
  if (n < 0 || out == nullptr || !even_address(out) || !span_flat(out, n).ok) return POLY_EINVAL;
  return launch_status([&] {
    return launch_zero_outside(static_cast<uint16_t *>(out), seg_off, num_segments, cap_rows,
                               cols, reinterpret_cast<cudaStream_t>(stream));
  });
}

// Shared part of the softcap calls: alpha must give finite, non-zero
// target-format constants alpha and 1/alpha (1/alpha formed in FP64, then
// rounded once).
static int softcap_call(bool bwd, int dtype, double alpha, const void *x, const void *dy,
                        void *out, int64_t n, poly_stream_t stream) {
  if (!valid_dtype(dtype) || n < 0 || !(alpha > 0) || !std::isfinite(alpha)) return POLY_EINVAL;
  const uint16_t a = from_double(alpha, dtype), ia = from_double(1.0 / alpha, dtype);
  auto usable = [&](uint16_t b) {
    const double v = to_double(b, dtype);
    return std::isfinite(v) && v != 0.0;
  };
  if (!usable(a) || !usable(ia)) return POLY_EINVAL;
  if (n == 0) return POLY_OK;
  if (x == nullptr || out == nullptr || (bwd && dy == nullptr)) return POLY_EINVAL;
  if (!even_address(x) || !even_address(out) || (bwd && !even_address(dy))) return POLY_EINVAL;
  Span si[2] = {span_flat(x, n), span_flat(bwd ? dy : x, n)};
  Span so[1] = {span_flat(out, n)};
  if (!aliasing_ok(si, bwd ? 2 : 1, so, 1)) return POLY_EINVAL;
  const void *ptrs[3] = {x, bwd ? dy : x, out};
  Layout l = flat_layout(ptrs, 3, n);
  poly_program p;
  int st = registry_get(POLY_TANH, bwd ? POLY_BWD : POLY_FWD, dtype, &p);
  if (st != POLY_OK) return st;
  Streams s{static_cast<const uint16_t *>(x), static_cast<const uint16_t *>(dy), nullptr,
            static_cast<uint16_t *>(out), nullptr};
  return launch_status([&] {
    return launch_softcap(bwd ? 1 : 0, dtype, p.degree, s, l, dev_prog(p), a, ia,
                          reinterpret_cast<cudaStream_t>(stream));
  });
}

int poly_softcap_fwd(int dtype, double alpha, const void *x, void *y, int64_t n,
                     poly_stream_t stream) {
  return softcap_call(false, dtype, alpha, x, nullptr, y, n, stream);
}

int poly_softcap_bwd(int dtype, double alpha, const void *x, const void *dy, void *dx, int64_t n,
                     poly_stream_t stream) {
  return softcap_call(true, dtype, alpha, x, dy, dx, n, stream);
}

// FP16 constants of each exp2 core, from the paper's printed parameters
// (Appendix B.1 eq. 17-19); PWL2's b = 2 (1 - a) and D2's 1 - a are formed
// in FP64 (D2's from the already rounded a, which keeps p(1) = 2 exact).
static void exp2_constants(int core, uint16_t *c) {
  c[0] = c[1] = c[2] = 0;
  if (core == POLY_EXP2_PWL2) {
    const double a = 0.7980513010;
    c[0] = from_double(a, POLY_F16);
    c[1] = from_double(2.0 * (1.0 - a), POLY_F16);
  } else if (core == POLY_EXP2_D2) {
    c[0] = from_double(0.6602339719, POLY_F16);
    c[1] = from_double(1.0 - to_double(c[0], POLY_F16), POLY_F16);
  } else if (core == POLY_EXP2_D3) {
    c[0] = from_double(0.6951461434, POLY_F16);
    c[1] = from_double(0.2275643945, POLY_F16);
    c[2] = from_double(0.0771190897, POLY_F16);
  }
}

static int exp2_call(int core, const float *x, float *y, int64_t n, poly_stream_t stream) {
  if (core < POLY_EXP2_D1 || core > POLY_EXP2_MUFU || n < 0) return POLY_EINVAL;
  if (n == 0) return POLY_OK;
  if (x == nullptr || y == nullptr) return POLY_EINVAL;
  if ((reinterpret_cast<uintptr_t>(x) & 3u) || (reinterpret_cast<uintptr_t>(y) & 3u))
    return POLY_EINVAL;
  if (n > kMaxElems) return POLY_EINVAL;
  Span si[1] = {span_bytes(x, n * 4)};
  Span so[1] = {span_bytes(y, n * 4)};
  if (!aliasing_ok(si, 1, so, 1)) return POLY_EINVAL;
  const int vec = ((reinterpret_cast<uintptr_t>(x) ^ reinterpret_cast<uintptr_t>(y)) & 15u) == 0;
  uint16_t c[3];
  exp2_constants(core, c);
  return launch_status(
      [&] { return launch_exp2(core, x, y, n, vec, c, reinterpret_cast<cudaStream_t>(stream)); });
}

int poly_exp2(int core, const float *x, float *y, int64_t n, poly_stream_t stream) {
  if (core == POLY_EXP2_MUFU) return POLY_EINVAL;   // the control has its own entry point
  return exp2_call(core, x, y, n, stream);
}

int poly_ctrl_exp2(const float *x, float *y, int64_t n, poly_stream_t stream) {
  return exp2_call(POLY_EXP2_MUFU, x, y, n, stream);
}

namespace {
std::once_flag g_sincos_once;
uint16_t g_sin16[3], g_cos16[3];
void sincos_init() { std::call_once(g_sincos_once, [] { fit_sincos(g_sin16, g_cos16); }); }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

int poly_rope_programs(uint16_t *sin_coef, uint16_t *cos_coef) {
  if (sin_coef == nullptr || cos_coef == nullptr) return POLY_EINVAL;
  sincos_init();
  for (int j = 0; j < 3; ++j) {
    sin_coef[j] = g_sin16[j];
    cos_coef[j] = g_cos16[j];
  }
  return POLY_OK;
}

int poly_rope_turn_increments(int head_dim, double base, uint32_t *out) {
  if (head_dim <= 0 || (head_dim & 1) || !(base > 1.0) || !std::isfinite(base) || !out)
    return POLY_EINVAL;
  for (int i = 0; i < head_dim / 2; ++i) {
    const double omega = std::pow(base, -2.0 * i / head_dim);
    out[i] = (uint32_t)std::llround(omega * 4294967296.0 / (2.0 * M_PI));
  }
  return POLY_OK;
}

static int rope_call(int inv, int variant, const void *q, const void *k, void *q_out,
                     void *k_out, const uint32_t *delta, const void *cos_tab,
                     const void *sin_tab, int64_t batch, int64_t seq, int64_t hq, int64_t hkv,
                     int64_t head_dim, int64_t pos_offset, poly_stream_t stream) {
  if (variant < POLY_ROPE_POLY || variant > POLY_ROPE_TABLE) return POLY_EINVAL;
  if (batch < 0 || seq < 0 || hq < 0 || hkv < 0 || head_dim <= 0 || (head_dim & 7) ||
      pos_offset < 0 || pos_offset > (int64_t(1) << 32) || seq > kMaxElems ||
      pos_offset + seq > (int64_t(1) << 32))
    return POLY_EINVAL;
  if (batch == 0 || seq == 0 || hq + hkv == 0) return POLY_OK;
  const int64_t rows = checked_mul(batch, seq);
  const int64_t nq = checked_mul(checked_mul(rows, hq), head_dim);
  const int64_t nk = checked_mul(checked_mul(rows, hkv), head_dim);
  const int64_t ntab = checked_mul(seq, head_dim / 2);
  if (rows < 0 || nq < 0 || nk < 0 || ntab < 0 || hq > kMaxElems || hkv > kMaxElems)
    return POLY_EINVAL;
  Span si[4], so[2];
  int nin = 0, nout = 0;
  if (hq > 0) {
    if (!q || !q_out || !aligned16(q) || !aligned16(q_out)) return POLY_EINVAL;
    si[nin++] = span_flat(q, nq);
    so[nout++] = span_flat(q_out, nq);
  }
  if (hkv > 0) {
    if (!k || !k_out || !aligned16(k) || !aligned16(k_out)) return POLY_EINVAL;
    si[nin++] = span_flat(k, nk);
    so[nout++] = span_flat(k_out, nk);
  }
  if (variant == POLY_ROPE_TABLE) {
    if (!cos_tab || !sin_tab || !aligned16(cos_tab) || !aligned16(sin_tab)) return POLY_EINVAL;
    si[nin++] = span_flat(cos_tab, ntab);
    si[nin++] = span_flat(sin_tab, ntab);
  } else if (!delta || !aligned16(delta)) {
    return POLY_EINVAL;
  }
  for (int i = 0; i < nin; ++i)
    if (!si[i].ok) return POLY_EINVAL;
  for (int o = 0; o < nout; ++o)
    if (!so[o].ok) return POLY_EINVAL;
  // transposed layouts: an output may not touch any input, nor the other output
  for (int o = 0; o < nout; ++o) {
    for (int i = 0; i < nin; ++i)
      if (overlaps(so[o], si[i])) return POLY_EINVAL;
    for (int o2 = o + 1; o2 < nout; ++o2)
      if (overlaps(so[o], so[o2])) return POLY_EINVAL;
  }
  sincos_init();
  RopeConsts kc;
  for (int j = 0; j < 3; ++j) {
    kc.s[j] = (uint32_t)g_sin16[j] * 0x00010001u;
    kc.c[j] = (uint32_t)g_cos16[j] * 0x00010001u;
  }
  RopeArgs a{static_cast<const uint16_t *>(q), static_cast<const uint16_t *>(k),
             static_cast<uint16_t *>(q_out), static_cast<uint16_t *>(k_out), delta,
             static_cast<const uint16_t *>(cos_tab), static_cast<const uint16_t *>(sin_tab),
             batch, seq, hq, hkv, head_dim, pos_offset};
  return launch_status(
      [&] { return launch_rope(variant, inv, a, kc, reinterpret_cast<cudaStream_t>(stream)); });
}

int poly_rope_fwd(int variant, const void *q, const void *k, void *q_out, void *k_out,
                  const uint32_t *delta, const void *cos_tab, const void *sin_tab,
                  int64_t batch, int64_t seq, int64_t hq, int64_t hkv, int64_t head_dim,
                  int64_t pos_offset, poly_stream_t stream) {
  return rope_call(0, variant, q, k, q_out, k_out, delta, cos_tab, sin_tab, batch, seq, hq, hkv,
                   head_dim, pos_offset, stream);
}

int poly_rope_bwd(int variant, const void *dq, const void *dk, void *dq_out, void *dk_out,
                  const uint32_t *delta, const void *cos_tab, const void *sin_tab,
                  int64_t batch, int64_t seq, int64_t hq, int64_t hkv, int64_t head_dim,
                  int64_t pos_offset, poly_stream_t stream) {
  return rope_call(1, variant, dq, dk, dq_out, dk_out, delta, cos_tab, sin_tab, batch, seq, hq,
                   hkv, head_dim, pos_offset, stream);
}

int poly_diag_stream_peak(int nin, int inflight, const void *a, const void *b, void *out,
                          int64_t n, int reps, poly_stream_t stream) {
  if ((nin != 1 && nin != 2) || n < 0 || (n & 7) || reps < 1 || reps > (1 << 20))
    return POLY_EINVAL;
  if (inflight != 1 && inflight != 2 && inflight != 4 && inflight != 8) return POLY_EINVAL;
  if ((n >> 3) >= (int64_t(1) << 31)) return POLY_EINVAL;
  if (n == 0) return POLY_OK;
  if (nin == 1) b = a;
  if (a == nullptr || b == nullptr || out == nullptr) return POLY_EINVAL;
  if (!aligned16(a) || !aligned16(b) || !aligned16(out)) return POLY_EINVAL;
  const Span si[2] = {span_flat(a, n), span_flat(b, n)};
  const Span so = span_flat(out, n);
  if (!si[0].ok || !si[1].ok || !so.ok) return POLY_EINVAL;
  for (int i = 0; i < 2; ++i)
    if (overlaps(so, si[i])) return POLY_EINVAL;
  return launch_status([&] {
    return launch_stream_peak(nin, inflight, static_cast<const uint16_t *>(a),
                              static_cast<const uint16_t *>(b), static_cast<uint16_t *>(out),
                              n >> 3, reps, reinterpret_cast<cudaStream_t>(stream));
  });
}

int poly_diag_packed(int op, int dtype, const void *a, const void *b, const void *c, void *out,
                     int64_t n, poly_stream_t stream) {
  if (op < POLY_DIAG_FMA || op > POLY_DIAG_GT || !valid_dtype(dtype) || n < 0)
    return POLY_EINVAL;
  if (n == 0) return POLY_OK;
  if (op == POLY_DIAG_FMA && c == nullptr) return POLY_EINVAL;
  if (c == nullptr) c = a;   // only FMA reads c
  if (a == nullptr || b == nullptr || out == nullptr) return POLY_EINVAL;
  if (!even_address(a) || !even_address(b) || !even_address(c) || !even_address(out))
    return POLY_EINVAL;
  Span si[3] = {span_flat(a, n), span_flat(b, n), span_flat(c, n)};
  Span so[1] = {span_flat(out, n)};
  if (!aliasing_ok(si, 3, so, 1)) return POLY_EINVAL;
  const void *ptrs[4] = {a, b, c, out};
  Layout l = flat_layout(ptrs, 4, n);
  Streams s{static_cast<const uint16_t *>(a), static_cast<const uint16_t *>(b),
            static_cast<const uint16_t *>(c), static_cast<uint16_t *>(out), nullptr};
  return launch_status(
      [&] { return launch_diag(op, dtype, s, l, reinterpret_cast<cudaStream_t>(stream)); });
}

}  // extern "C"
