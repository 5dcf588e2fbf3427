// fit_internal.h -- declarations shared by the fitter and the C ABI layer.
#pragma once

#include <cstdint>

#include "../../include/polyact.h"

namespace polyact {

double fn_value(int fn, int dir, double x);
int form_of_fn(int fn, int dir);
double residual_at_zero(int fn, int dir);
uint16_t replay_one(int form, const uint16_t *coef, int degree, uint16_t lc, uint16_t x,
                    int dtype, bool fused);
double replay_real(int form, const double *c, int degree, double lc, double x);
void fit_coefficients(int fn, int dir, int degree, double li, int n_nodes, double *c);
int fit_program(int fn, int dir, int dtype, int degree, const poly_fit_opts &o,
                poly_program *out);
int derive_program(const poly_program &fwd, poly_program *out);
// FP16 RoPE programs: s = (s1, s3, s5), c = (c2, c4, c6).
void fit_sincos(uint16_t *s, uint16_t *c);

}  // namespace polyact
