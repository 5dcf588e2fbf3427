/*
 * polyact.h -- C ABI of libpolyact: packed-polynomial activation programs for
 * GB300 (sm_103a).
 *
 * Method: "Fast Polynomial Transcendentals for LLMs" (arXiv 2610.00049).
 * Sigmoid, tanh, SiLU and exact GELU (and the derivatives used in backward)
 * are replaced by short range-reduced polynomial programs evaluated with
 * packed two-lane FP16 / BF16 FMAs (§3.1 analytic reduction, §3.4 packed
 * CUDA programs), standalone or fused into a SwiGLU gate (§3.4, §5.2.4
 * eq. 15).  A host-side constrained fitter builds the programs (§3.2).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Status: every function returns an int; POLY_OK (0) on success, a
 *   negative POLY_E* code otherwise (poly_status_str names it).  No function
 *   throws, aborts or prints.
 * - Ownership: the caller owns every buffer.  The library never allocates,
 *   frees or synchronises device memory.
 * - Device calls (poly_act_*, poly_swiglu_*, poly_ragged_zero_outside,
 *   poly_softcap_*, poly_exp2, poly_rope_*, poly_ctrl_*, poly_diag_packed,
 *   poly_diag_stream_peak)
 *   take addresses the GPU can reach -- device memory, or, on systems with
 *   coherent host access such as
 *   GB300's NVLink-C2C, pinned host memory (the kernels then stream it over
 *   the link with no staging copy) -- and a CUDA stream (poly_stream_t is
 *   layout-compatible with cudaStream_t; NULL = the legacy default stream).
 *   Kernels run on the calling thread's current device.  They validate the
 *   arguments on the host, enqueue one kernel and return without waiting.
 *   Several host threads may call them at once (each launch carries its
 *   program as a kernel parameter; nothing is shared between launches).
 *   A launch failure is reported as POLY_ECUDA (the CUDA error is consumed
 *   and available through poly_last_cuda_error).
 * - Tensors hold 16-bit elements (FP16 or BF16 bit patterns), contiguous
 *   unless leading dimensions are given.  Any 2-byte alignment is accepted:
 *   16-byte-aligned data takes the 128-bit vector path, a scalar head and
 *   tail cover the rest, and inputs that sit at other addresses modulo 16
 *   than the output are realigned in registers (still 16-byte accesses).
 *   Odd addresses -> POLY_EINVAL.  Exceptions, stated
 *   at each call: poly_exp2 works on FP32 (4-byte aligned), the RoPE calls
 *   on FP16 with 16-byte-aligned tensors.
 * - n == 0 (or rows == 0 / cols == 0) is a valid no-op: POLY_OK, no launch.
 * - Sizes: a tensor extent above 2^46 elements, a leading dimension or size
 *   factor above that, or a tensor whose last byte would wrap the address
 *   space -> POLY_EINVAL (no size computation can overflow).
 * - Aliasing: an output may be exactly the same view as an input (in
 *   place).  An output sharing any byte with another tensor otherwise ->
 *   POLY_EINVAL.  Views that share no element may interleave: row sets of
 *   the same leading dimension whose rows fall in each other's gaps (the
 *   gate and up halves of one [T, 2H] buffer, ld = 2H) are accepted.
 * - Arithmetic: every packed FMA / multiply rounds once to the target format,
 *   to nearest-even, with subnormals kept; a NaN result is 0x7FFF.  Outputs
 *   are bit-exact functions of the inputs and the installed program.
 */
#ifndef POLYACT_H
#define POLYACT_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *poly_stream_t;

/* Target formats (§3.4: FP16 for the isolated sweep, BF16 in integrations). */
enum { POLY_F16 = 0, POLY_BF16 = 1 };

/* Functions.  Forward evaluates the function, backward its derivative. */
enum { POLY_SIGMOID = 0, POLY_TANH = 1, POLY_SILU = 2, POLY_GELU = 3 };
enum { POLY_FWD = 0, POLY_BWD = 1 };

/* Reduction forms (§3.1 eq. 2-6, §3.3 eq. 9), with t = min(|x|, Lc):
 *   POLY_FORM_CO  centred odd  y = 1/2 + sign(x) t (c1 + c2 t + ... + cD t^(D-1))
 *                 sigmoid forward; SiLU' and GELU' backward
 *   POLY_FORM_O   odd          y = sign(x) t (c1 + ... + cD t^(D-1))      tanh forward
 *   POLY_FORM_E   even         y = c0 + c1 t + ... + cD t^D          sigmoid', tanh'
 *   POLY_FORM_HX  x/2 + even   y = x/2 + t (c1 + ... + cD t^(D-1)) for |x| <= Lc,
 *                              y = max(x, +0) for |x| > Lc           SiLU, GELU forward
 * The form is fixed by (fn, dir). */
enum { POLY_FORM_CO = 0, POLY_FORM_O = 1, POLY_FORM_E = 2, POLY_FORM_HX = 3 };

enum {
  POLY_OK = 0,
  POLY_EINVAL = -1,   /* bad enum, null pointer with work to do, bad size,
                         misaligned (odd) address, partial aliasing          */
  POLY_ENOPROG = -2,  /* program descriptor inconsistent (form/degree/dtype) */
  POLY_ECUDA = -3,    /* a CUDA call or kernel launch failed                 */
  POLY_ENOFIT = -4    /* the fitter found no candidate passing its gates     */
};

#define POLY_MIN_DEGREE 3
#define POLY_MAX_DEGREE 6
#define POLY_PROGRAM_VERSION 1u

/* One accepted program (§3.2).  Plain data; copy freely. */
typedef struct poly_program {
  int32_t fn, dir, dtype, form, degree;
  uint16_t coef[POLY_MAX_DEGREE + 1]; /* c_0..c_D, target-format bit patterns;
                                         c_0 = f(0) (0 for CO/O/HX forms)    */
  uint16_t lc_bits;                   /* runtime clamp Lc in the target format */
  double li;                          /* fit interval [0, Li] of eq. 7-8       */
  double lc;                          /* Lc as a number                        */
  double search_score;                /* split-rounding max abs error, §3.2 step 6 */
  double deployed_score;              /* same grid, deployed (fused) order     */
  double stated_max_abs_err;          /* max over every finite input of
                                         |program - FP64 function|            */
  double table2;                      /* Table 2 metric: real arithmetic on
                                         20,001 points over [-Lc, Lc]          */
  int32_t rank;                       /* split-score rank of the accepted one  */
  uint32_t version;                   /* POLY_PROGRAM_VERSION                  */
} poly_program;

/* Search options of the fitter (§3.2 steps 1-7).  poly_fit_defaults fills:
 * Li in {1, 1.25, ..., 12}; Lc in {1, 1.25, ..., Li + 1}; 2,000 Chebyshev
 * nodes; 8,000 score points over [0, 12]; top_k = 0 (every gated candidate is
 * re-scored in deployed order; k > 0 keeps the k best by split-order score);
 * lc_refine_ulps = 0 (k > 0 also re-scores each finalist with its clamp moved
 * by 1..k target-format ulps either way, at most 64). */
typedef struct poly_fit_opts {
  double li_min, li_max, li_step;
  double lc_min, lc_step;
  int32_t n_nodes;
  int32_t n_score;
  double score_hi;
  int32_t top_k;
  int32_t lc_refine_ulps;
} poly_fit_opts;

/* ---- status / metadata ------------------------------------------------ */

/* Static string naming a status code (never NULL). */
const char *poly_status_str(int status);
/* The CUDA error code behind the last POLY_ECUDA on this thread (0 if none). */
int poly_last_cuda_error(void);
/* Library ABI version (bumped when an entry point, signature or struct
 * changes or is added). */
int poly_abi_version(void);
/* Form of (fn, dir) or POLY_EINVAL. */
int poly_form_of(int fn, int dir);
/* Degree of the default program of (fn, dir): sigmoid D3, tanh D4, SiLU D3,
 * GELU D5 forward; D4 for every derivative.  POLY_EINVAL on bad enums. */
int poly_default_degree(int fn, int dir);

/* ---- fitter (host only, no CUDA) ---------------------------------------- */

/* Fill *opts with the defaults listed above.  POLY_EINVAL if opts is NULL. */
int poly_fit_defaults(poly_fit_opts *opts);

/* Run the constrained fit and search of §3.2 for (fn, dir, dtype, degree):
 * eq. 8 endpoint-constrained least squares in FP64 for every Li, coefficients
 * rounded to the target format, every Lc <= Li + 1 replayed with one rounding
 * per multiply and per add, scored as max abs error over the score grid and
 * gated (finite; exact P(0) = f(0); range for sigmoid/tanh/sigma'/tanh';
 * monotone real-arithmetic replay for functions monotone on t >= 0); the
 * candidates (top_k of them if top_k > 0) are re-scored in the deployed fused
 * order and gated again, and the one with the smallest deployed-order error
 * (exact ties: the smaller Table 2 metric, then the smaller Li, then the
 * smaller Lc) is written to *out.  opts NULL = defaults.  Deterministic.
 * Host memory only.  Thread-safe (concurrent calls give what lone calls give).
 * Returns POLY_EINVAL (bad enum, degree outside [3, 6], bad opts, out NULL)
 * or POLY_ENOFIT (no candidate passed). */
int poly_fit(int fn, int dir, int dtype, int degree, const poly_fit_opts *opts,
             poly_program *out);

/* ---- program registry ---------------------------------------------------- */

/* Install *p as the program used for (p->fn, p->dir, p->dtype) by later
 * calls.  Validates enums, form, degree, version, that c_0 matches the form,
 * and the clamp: lc_bits must decode to a finite positive value equal to lc,
 * with Lc <= Li + 1 (li finite and positive).  POLY_ENOPROG if inconsistent.
 * Thread-safe. */
int poly_set_program(const poly_program *p);

/* Copy the installed program for (fn, dir, dtype) into *out.  If none is
 * installed yet, the default-degree program is fitted (poly_fit with default
 * options, tens to hundreds of milliseconds of host time) and installed
 * first.  Thread-safe. */
int poly_get_program(int fn, int dir, int dtype, poly_program *out);

/* Forget every installed program (defaults are re-fitted on next use). */
int poly_reset_programs(void);

/* Differentiated-polynomial backward (§3.3: B2 "differentiates its D4 tanh
 * program and evaluates the resulting D3 program").  From an odd or
 * centred-odd forward program y = [1/2 +] sign(x) (c_1 t + ... + c_D t^D)
 * write to *out the even backward program of degree D - 1 with
 * coefficients (j + 1) c_(j+1), each rounded once to the target format, the
 * same clamp (beyond Lc it keeps its value at Lc) and its own stated bound
 * against the true derivative.  Install it with poly_set_program to use it
 * in poly_act_bwd / poly_softcap_bwd in place of the direct derivative fit.
 * Host only.  POLY_EINVAL for a NULL pointer or a program that is not an odd
 * or centred-odd forward program; POLY_ENOPROG for an inconsistent one.
 * Direct fits are the default because they are 4-7x more accurate (the
 * paper: "backward has its own error profile"). */
int poly_derive_program(const poly_program *fwd, poly_program *out);

/* ---- elementwise programs (§5.1.1, Table 3) ------------------------------ */

/* y[i] = program_fwd(fn, dtype)(x[i]) for i < n.  x, y: device, n elements.
 * y == x allowed.  Uses the installed (or default) forward program. */
int poly_act_fwd(int fn, int dtype, const void *x, void *y, int64_t n,
                 poly_stream_t stream);

/* dx[i] = dy[i] * program_bwd(fn, dtype)(x[i]) (one rounding) -- the direct
 * derivative fit evaluated from x (§4.2).  dx may equal x or dy. */
int poly_act_bwd(int fn, int dtype, const void *x, const void *dy, void *dx,
                 int64_t n, poly_stream_t stream);

/* ---- SwiGLU gate (§3.4, §5.2.4 eq. 15) ------------------------------------
 * Two rules, chosen per call by the _v entry points (variant argument), or
 * process-wide for the plain entry points by poly_set_swiglu_variant:
 * POLY_SWIGLU_DIRECT (default): s = installed SiLU forward program (HX form),
 *   s' = installed SiLU backward program (CO form, the centred SiLU
 *   derivative of eq. 9).
 *   Forward:   y  = s(g) * u
 *   Backward:  dg = (dy * u) * s'(g),   du = dy * s(g)
 * POLY_SWIGLU_SIGMOID: the rule the paper deploys in B1/B4 (§3.3, §5.2.4):
 *   p = installed sigmoid forward program, s = g * p,
 *   s' = p + g p (1 - p) evaluated as q = fma(-p, p, p), s' = fma(g, q, p).
 *   Forward:   y  = (g * p) * u
 *   Backward:  dg = (dy * u) * s',      du = dy * (g * p)
 * Every product and fma rounds once.
 * Dense: row-major [rows, cols] with leading dimensions (elements, >= cols).
 */
enum { POLY_SWIGLU_DIRECT = 0, POLY_SWIGLU_SIGMOID = 1 };
/* Select the SwiGLU rule used by later calls of the plain (non-_v) SwiGLU
 * entry points (thread-safe, process-wide; callers on different streams that
 * want different rules use the _v entry points instead).  POLY_EINVAL for an
 * unknown variant. */
int poly_set_swiglu_variant(int variant);
/* The current SwiGLU rule. */
int poly_get_swiglu_variant(void);

int poly_swiglu_fwd(int dtype, const void *g, const void *u, void *y,
                    int64_t rows, int64_t cols, int64_t ldg, int64_t ldu,
                    int64_t ldy, poly_stream_t stream);
int poly_swiglu_bwd(int dtype, const void *g, const void *u, const void *dy,
                    void *dg, void *du, int64_t rows, int64_t cols, int64_t ldg,
                    int64_t ldu, int64_t lddy, int64_t lddg, int64_t lddu,
                    poly_stream_t stream);
/* The same calls with the rule as an argument (POLY_SWIGLU_DIRECT or
 * POLY_SWIGLU_SIGMOID; anything else -> POLY_EINVAL).  Nothing process-wide
 * is read, so concurrent callers may use different rules. */
int poly_swiglu_fwd_v(int variant, int dtype, const void *g, const void *u, void *y,
                      int64_t rows, int64_t cols, int64_t ldg, int64_t ldu, int64_t ldy,
                      poly_stream_t stream);
int poly_swiglu_bwd_v(int variant, int dtype, const void *g, const void *u, const void *dy,
                      void *dg, void *du, int64_t rows, int64_t cols, int64_t ldg,
                      int64_t ldu, int64_t lddy, int64_t lddg, int64_t lddu,
                      poly_stream_t stream);

/* Ragged routed-expert SwiGLU: the rows of all experts are packed without
 * padding into [cap_rows, cols] tensors (leading dimension cols); expert e
 * owns rows [seg_off[e], seg_off[e+1]).  seg_off is a DEVICE int32 array of
 * num_segments + 1 entries, read by the kernel (no host synchronisation):
 * rows [max(seg_off[0], 0), min(seg_off[num_segments], cap_rows)) are
 * processed, nothing else is touched.  status: optional device int32; when
 * non-NULL the kernel writes 0 if seg_off is valid (seg_off[0] == 0,
 * non-decreasing, seg_off[num_segments] <= cap_rows) and 1 otherwise. */
int poly_swiglu_fwd_ragged(int dtype, const void *g, const void *u, void *y,
                           const int32_t *seg_off, int num_segments,
                           int64_t cap_rows, int64_t cols, int32_t *status,
                           poly_stream_t stream);
int poly_swiglu_bwd_ragged(int dtype, const void *g, const void *u,
                           const void *dy, void *dg, void *du,
                           const int32_t *seg_off, int num_segments,
                           int64_t cap_rows, int64_t cols, int32_t *status,
                           poly_stream_t stream);
/* The ragged calls with the rule as an argument, as poly_swiglu_fwd_v. */
int poly_swiglu_fwd_ragged_v(int variant, int dtype, const void *g, const void *u, void *y,
                             const int32_t *seg_off, int num_segments, int64_t cap_rows,
                             int64_t cols, int32_t *status, poly_stream_t stream);
int poly_swiglu_bwd_ragged_v(int variant, int dtype, const void *g, const void *u,
                             const void *dy, void *dg, void *du, const int32_t *seg_off,
                             int num_segments, int64_t cap_rows, int64_t cols,
                             int32_t *status, poly_stream_t stream);

/* Zero the rows of a [cap_rows, cols] buffer of 16-bit elements (any format:
 * +0 is all-zero bits) that the ragged calls above leave untouched: rows
 * outside [max(seg_off[0], 0), min(seg_off[num_segments], cap_rows)), the
 * range read on the device as those calls read it (empty when the offsets
 * cross or start past the buffer: every row is zeroed then).  Paired with a ragged
 * call on the same stream (in either order) it gives an output or gradient
 * that reads as zero outside the segments, writing each row once instead of
 * filling the whole buffer first; when the segments cover every row it
 * writes nothing.  out: device (or pinned host) memory, 2-byte aligned.
 * POLY_EINVAL if seg_off or out is NULL (with work to do), num_segments,
 * cap_rows or cols is negative, or the extent is too large (Sizes rule). */
int poly_ragged_zero_outside(void *out, const int32_t *seg_off, int num_segments,
                             int64_t cap_rows, int64_t cols, poly_stream_t stream);

/* ---- tanh softcap (§2.3 eq. 1; §3.3 eq. 12) -------------------------------
 * softcap_alpha(x) = alpha tanh(x / alpha), the attention-logit softcap.
 * Forward:   z = x * A_inv,  y = A * tanh_program(z)
 * Backward:  z = x * A_inv,  dx = dy * dtanh_program(z)     (alpha cancels)
 * with A = alpha and A_inv = 1/alpha (formed in FP64) rounded once to the
 * target format; every product rounds once.  tanh_program is the installed
 * tanh forward program, dtanh_program the installed tanh backward program
 * (the direct derivative fit by default, or one from poly_derive_program).
 * POLY_EINVAL if alpha is not finite and > 0 or if A or A_inv would be zero
 * or infinite in the target format; otherwise the conventions of
 * poly_act_fwd / poly_act_bwd. */
int poly_softcap_fwd(int dtype, double alpha, const void *x, void *y, int64_t n,
                     poly_stream_t stream);
int poly_softcap_bwd(int dtype, double alpha, const void *x, const void *dy, void *dx,
                     int64_t n, poly_stream_t stream);

/* ---- exp2 with a polynomial fractional core (Appendix B.1, eq. 16-19) -----
 * y[i] = 2^x[i] for FP32 x, y (device addresses, n elements, y == x allowed):
 * xc = min(max(x, -126), 128); n = floor(xc); f = xc - n (FP32, one
 * rounding); h = f rounded to FP16; p = core(h) in packed FP16 arithmetic
 * (one rounding per operation); y = float(p) scaled by 2^n through its
 * exponent bits; NaN in -> 0x7FFFFFFF; x < -126 gives 2^-126.
 * Cores (constants rounded to FP16 from the paper's parameters):
 *   POLY_EXP2_D1    p = 1 + f                                   one FMA
 *   POLY_EXP2_PWL2  p = 1 + a f + b max(f - 1/2, 0), a = 0.7980513010,
 *                   b = 2 (1 - a) -> 0.7978515625, 0.40380859375 (eq. 17)
 *   POLY_EXP2_D2    p = 1 + a f + (1 - a) f^2, a = 0.6602339719 (eq. 18)
 *   POLY_EXP2_D3    FA4's cubic (eq. 19)
 *   order: PWL2 p = fma(h, a, 1), m = max(fma(h, 1, -1/2), 0), p = fma(m, b, p);
 *          D2 p = fma(fma(b, h, a), h, 1); D3 Horner from the top coefficient.
 * POLY_EINVAL for an unknown core, n < 0, NULL or misaligned (not 4-byte)
 * pointers, or partial overlap. */
enum { POLY_EXP2_D1 = 0, POLY_EXP2_PWL2 = 1, POLY_EXP2_D2 = 2, POLY_EXP2_D3 = 3,
       POLY_EXP2_MUFU = 4 };
int poly_exp2(int core, const float *x, float *y, int64_t n, poly_stream_t stream);

/* ---- fused RoPE with paired polynomial sine / cosine (Appendix B.2) -------
 * FP16 only.  Frequencies omega_i = base^(-2i/D), i < D/2, act on the
 * interleaved pairs (x_2i, x_2i+1) as complex numbers.  The caller passes
 * delta: a DEVICE array of D/2 Q0.32 turn increments
 * Delta_i = round(omega_i 2^32 / 2 pi) (poly_rope_turn_increments fills one
 * on the host).  At position p = pos_offset + s the phase is
 * (p Delta_i) mod 2^32; as a signed value it is a Q31 half-turn coordinate,
 * folded into [-1/2, 1/2] half-turns (sin(pi u) = sin(pi (+-1 - u)), cosine
 * negated), then truncated to the signed Q15 coordinate q.
 * Variants:
 *   POLY_ROPE_POLY   u = FP16(q) 2^-15, w = u u, sin = fma(fma(s5, w, s3), w, s1) u,
 *                    cos = fma(fma(fma(c6, w, c4), w, c2), w, 1) (packed FP16,
 *                    one rounding per op; D5 sine and D6 cosine fitted as in
 *                    eq. 7-8 with the end value at u = 1/2 exact)
 *   POLY_ROPE_MUFU   sin.approx / cos.approx of pi u in FP32, rounded to FP16
 *   POLY_ROPE_TABLE  cos_tab / sin_tab: DEVICE FP16 [S, D/2]; row s serves
 *                    position pos_offset + s (delta may be NULL)
 * Rotation of (a, b) by (c, s): out = (fma(a, c, -(b s)), fma(b, c, a s)).
 * Forward: q [B, S, Hq, D], k [B, S, Hkv, D] -> q_out [B, Hq, S, D],
 *          k_out [B, Hkv, S, D].
 * Backward: the same call shape with gradients in [B, H, S, D] in and
 *          [B, S, H, D] out, rotated by -theta.
 * Contiguous tensors; every pointer 16-byte aligned; head_dim a multiple of 8;
 * hq or hkv may be 0 (its pointers then unused); outputs may not overlap any
 * input; pos_offset + seq <= 2^32.  POLY_EINVAL otherwise. */
enum { POLY_ROPE_POLY = 0, POLY_ROPE_MUFU = 1, POLY_ROPE_TABLE = 2 };
int poly_rope_fwd(int variant, const void *q, const void *k, void *q_out, void *k_out,
                  const uint32_t *delta, const void *cos_tab, const void *sin_tab,
                  int64_t batch, int64_t seq, int64_t hq, int64_t hkv, int64_t head_dim,
                  int64_t pos_offset, poly_stream_t stream);
int poly_rope_bwd(int variant, const void *dq, const void *dk, void *dq_out, void *dk_out,
                  const uint32_t *delta, const void *cos_tab, const void *sin_tab,
                  int64_t batch, int64_t seq, int64_t hq, int64_t hkv, int64_t head_dim,
                  int64_t pos_offset, poly_stream_t stream);
/* Host: out[i] = round(base^(-2i/head_dim) 2^32 / 2 pi), i < head_dim / 2.
 * POLY_EINVAL unless head_dim is positive and even, base > 1, out non-NULL. */
int poly_rope_turn_increments(int head_dim, double base, uint32_t *out);
/* Host: the FP16 bit patterns of the sine (s1, s3, s5) and cosine
 * (c2, c4, c6) coefficients the POLY_ROPE_POLY variant uses. */
int poly_rope_programs(uint16_t *sin_coef, uint16_t *cos_coef);

/* ---- MUFU-native controls (same signatures and memory schedule) ----------
 * The comparators of §4.2 / Table 3: the same functions on the
 * special-function unit instead of polynomial programs.  Two variants:
 *
 * POLY_CTRL_FP32 (the plain poly_ctrl_* calls): each element widened to
 * FP32: sigmoid = rcp.approx(1 + ex2.approx(-x log2 e)); tanh = tanh.approx;
 * SiLU = the overflow-safe form e = 2^(-|x| log2 e),
 * y = (x >= 0 ? x : x e) * rcp.approx(1 + e); exact GELU = x/2 (1 + erff(x /
 * sqrt 2)) (no special-function erf exists; erff is a CUDA-core polynomial).
 * Backward: sigma (1 - sigma), 1 - tanh^2, sigma (1 + x (1 - sigma)),
 * Phi + x phi, all recomputed from x.  One rounding to the target format.
 *
 * POLY_CTRL_PACKED (the _v calls): packed two-lane arithmetic in the target
 * format with one tanh.approx.{f16x2,bf16x2} instruction per pair -- one
 * special-function operation per element, against two for the FP32 control's
 * sigmoid and SiLU (GB300's special-function unit is twice GB200's,
 * Approximating Softmax in Pretrained LLMs, Appendix B.5): tanh = tanh.approx(x); sigmoid =
 * fma(t, 1/2, 1/2), t = tanh.approx(x * 1/2); SiLU = fma(h, t, h) with
 * h = x * 1/2, t = tanh.approx(h); GELU in the tanh form h (1 + tanh(z)),
 * z = x (k + k c x^2), k = sqrt(2/pi), c = 0.044715 (within 4.8e-4 of exact
 * GELU).  Backward: sigma' = fma(-p, p, p), tanh' = fma(-t, t, 1),
 * SiLU' = fma(x, fma(-p, p, p), p), GELU' = fma(1 - t^2, h z', p) with x
 * clamped to [-16, 16] and z' = k + 3 k c x^2; dx = dy * derivative.  SwiGLU:
 * y = SiLU(g) * u; dg = (dy * u) * SiLU'(g), du = dy * SiLU(g).  Every
 * operation rounds once to the target format.  Infinite inputs are outside
 * both controls' domain (the backward controls give NaN at +-inf).
 *
 * Results approximate the true function, not the polynomial programs. */
enum { POLY_CTRL_FP32 = 0, POLY_CTRL_PACKED = 1 };
int poly_ctrl_act_fwd(int fn, int dtype, const void *x, void *y, int64_t n,
                      poly_stream_t stream);
int poly_ctrl_act_bwd(int fn, int dtype, const void *x, const void *dy,
                      void *dx, int64_t n, poly_stream_t stream);
int poly_ctrl_swiglu_fwd(int dtype, const void *g, const void *u, void *y,
                         int64_t rows, int64_t cols, int64_t ldg, int64_t ldu,
                         int64_t ldy, poly_stream_t stream);
int poly_ctrl_swiglu_bwd(int dtype, const void *g, const void *u,
                         const void *dy, void *dg, void *du, int64_t rows,
                         int64_t cols, int64_t ldg, int64_t ldu, int64_t lddy,
                         int64_t lddg, int64_t lddu, poly_stream_t stream);
/* The controls with the variant as an argument (POLY_EINVAL for another). */
int poly_ctrl_act_fwd_v(int variant, int fn, int dtype, const void *x, void *y, int64_t n,
                        poly_stream_t stream);
int poly_ctrl_act_bwd_v(int variant, int fn, int dtype, const void *x, const void *dy,
                        void *dx, int64_t n, poly_stream_t stream);
int poly_ctrl_swiglu_fwd_v(int variant, int dtype, const void *g, const void *u, void *y,
                           int64_t rows, int64_t cols, int64_t ldg, int64_t ldu, int64_t ldy,
                           poly_stream_t stream);
int poly_ctrl_swiglu_bwd_v(int variant, int dtype, const void *g, const void *u,
                           const void *dy, void *dg, void *du, int64_t rows, int64_t cols,
                           int64_t ldg, int64_t ldu, int64_t lddy, int64_t lddg,
                           int64_t lddu, poly_stream_t stream);
/* 2^x by ex2.approx.ftz.f32 on the special-function unit, same memory
 * schedule and validation as poly_exp2. */
int poly_ctrl_exp2(const float *x, float *y, int64_t n, poly_stream_t stream);

/* ---- arithmetic diagnostic ------------------------------------------------
 * Runs one raw packed instruction over n element triples so that the
 * target-format arithmetic the programs rely on (one rounding per FMA or
 * multiply, nearest-even, subnormals kept, NaN results 0x7FFF, §3.2 Fig. 2c
 * and §3.4) can be checked against an independent model, element by element:
 *   POLY_DIAG_FMA     out = a * b + c        (fma.rn.{f16x2,bf16x2})
 *   POLY_DIAG_MUL     out = a * b            (mul.rn)
 *   POLY_DIAG_MIN_NAN out = min(a, b), NaN if either is NaN
 *   POLY_DIAG_MAX     out = max(a, b)
 *   POLY_DIAG_GT      out = 0xFFFF if a > b (ordered) else 0
 * a, b, c, out: device arrays of n 16-bit elements (c unused except by FMA,
 * may be NULL otherwise).  Same validation and status codes as above. */
enum { POLY_DIAG_FMA = 0, POLY_DIAG_MUL = 1, POLY_DIAG_MIN_NAN = 2, POLY_DIAG_MAX = 3,
       POLY_DIAG_GT = 4 };
int poly_diag_packed(int op, int dtype, const void *a, const void *b, const void *c,
                     void *out, int64_t n, poly_stream_t stream);

/* ---- streaming-bandwidth probe (a measurement tool; no counterpart in the
 * paper, which states its L2 and HBM regimes (§4.2) but no peaks) ---------
 * reps passes of out[i] = a[i] (nin = 1) or a[i] ^ b[i] (nin = 2, bitwise)
 * over n 16-bit elements, with the 16-byte loads and stores of the
 * streaming kernels; every thread keeps `inflight` (1, 2, 4 or 8) 16-byte
 * chunks per input in flight, from as many 256-thread blocks as the SMs hold
 * at once for that register budget, and pass r assigns each chunk to another
 * thread than pass r - 1 did.
 * The rate reps * n * 2 * (nin + 1) bytes / time is the L2 streaming
 * bandwidth of that access pattern when a, b and out fit in L2 and the
 * launch spans many passes, and its HBM rate when they do not.  a, b, out:
 * device memory, 16-byte aligned; out overlaps neither input; n a multiple of
 * 8 below 2^34; 1 <= reps <= 2^20; b unused (may be NULL) for nin = 1.
 * POLY_EINVAL otherwise; n == 0 is a no-op. */
int poly_diag_stream_peak(int nin, int inflight, const void *a, const void *b, void *out,
                          int64_t n, int reps, poly_stream_t stream);

/* ---- failure injection (host only; no counterpart in the paper) ----------
 * poly_debug_fail_launches: the next `count` kernel launches, from any entry
 * point above, are not enqueued; each of those calls returns POLY_ECUDA and
 * sets poly_last_cuda_error() to `cuda_error`, exactly as a failed launch
 * would.  Validation still runs first, and calls that launch nothing (n == 0,
 * invalid arguments) do not consume a failure.  This lets a caller's handling
 * of launch failures be tested without faulting a GPU.  Process-wide and
 * thread-safe; count == 0 clears pending failures.  Returns the number of
 * failures that were still pending, or POLY_EINVAL (cuda_error <= 0 or
 * count < 0). */
int poly_debug_fail_launches(int cuda_error, int count);

#ifdef __cplusplus
}
#endif

#endif /* POLYACT_H */
