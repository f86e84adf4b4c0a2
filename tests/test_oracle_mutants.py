"""The pins are strong enough: each plausible mistake, planted in a temporary copy
of the oracle's C source (on the CPU, never on the GPU), makes at least one pin
fail.  The real oracle source is never modified."""
import os

import pytest

import oracle
from oracle_pins import PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text in oracle.c, replacement, which occurrence: index or "all")
MUTANTS = [
    ("sigma_convention_2sigma2",
     "return exp(-sq_dist(xi, yj, D) / (sigma * sigma));",
     "return exp(-sq_dist(xi, yj, D) / (2.0 * sigma * sigma));", 0),
    ("exponent_sign",
     "return exp(-sq_dist(xi, yj, D) / (sigma * sigma));",
     "return exp(sq_dist(xi, yj, D) / (sigma * sigma));", 0),
    ("abs_instead_of_square", "s += diff * diff;", "s += fabs(diff);", 0),
    ("dropped_last_coordinate",
     "for (int d = 0; d < D; ++d) {\n        double diff = xi[d] - yj[d];",
     "for (int d = 0; d < D - 1; ++d) {\n        double diff = xi[d] - yj[d];", 0),
    ("sum_drops_signal", "double term = k * b[j * E + e];", "double term = k;", 0),
    ("sum_ignores_column", "double term = k * b[j * E + e];", "double term = k * b[j * E];", 0),
    ("sum_drops_last_point",
     "for (int64_t j = 0; j < N; ++j) {\n                double k = gauss(x + i * D, y + j * D, D, sigma);\n                double term",
     "for (int64_t j = 0; j < N - 1; ++j) {\n                double k = gauss(x + i * D, y + j * D, D, sigma);\n                double term", 0),
    ("compensation_sign", "*comp += (*sum - t) + v;", "*comp += (*sum - t) - v;", 0),
    ("lse_weight_sign_second_pass",
     "/ (sigma * sigma) + w[j * E + e];", "/ (sigma * sigma) - w[j * E + e];", 1),
    ("lse_drops_max", "L[i * E + e] = m + log(s + c);", "L[i * E + e] = log(s + c);", 0),
    ("lse_sigma_not_squared",
     "-sq_dist(x + i * D, y + j * D, D) / (sigma * sigma) + w",
     "-sq_dist(x + i * D, y + j * D, D) / (sigma) + w", "all"),
    ("grad_factor", "-(2.0 / (sigma * sigma)) * k", "-(1.0 / (sigma * sigma)) * k", 0),
    ("grad_direction", "double diff = x[i * D + d] - y[j * D + d];",
     "double diff = y[j * D + d] - x[i * D + d];", 0),
    ("grad_drops_signal", "beta += g[i * E + e] * b[j * E + e];", "beta += g[i * E + e];", 0),
    ("grad_wrong_row_of_g", "beta += g[i * E + e] * b[j * E + e];", "beta += g[e] * b[j * E + e];", 0),
    ("grad_y_sign", "double term = (2.0 / (sigma * sigma)) * k * beta * diff;",
     "double term = -(2.0 / (sigma * sigma)) * k * beta * diff;", 0),
    ("grad_y_drops_signal", "beta += g[i * E + e] * b[j * E + e];", "beta += g[i * E + e];", 1),
    ("grad_y_wrong_row_of_b", "beta += g[i * E + e] * b[j * E + e];", "beta += g[i * E + e] * b[e];", 1),
    ("grad_y_drops_last_row",
     "for (int64_t i = 0; i < M; ++i) {\n                double k = gauss(x + i * D, y + j * D, D, sigma);\n                double beta",
     "for (int64_t i = 0; i < M - 1; ++i) {\n                double k = gauss(x + i * D, y + j * D, D, sigma);\n                double beta", 0),
    ("grad_b_drops_kernel", "double term = gauss(x + i * D, y + j * D, D, sigma) * g[i * E + e];",
     "double term = g[i * E + e];", 0),
    ("grad_b_wrong_column", "double term = gauss(x + i * D, y + j * D, D, sigma) * g[i * E + e];",
     "double term = gauss(x + i * D, y + j * D, D, sigma) * g[i * E];", 0),
    ("grad_b_uses_j_row_of_g", "double term = gauss(x + i * D, y + j * D, D, sigma) * g[i * E + e];",
     "double term = gauss(x + i * D, y + j * D, D, sigma) * g[(j % M) * E + e];", 0),
    ("laplace_without_sqrt", "case 1: return exp(-sqrt(q) / sigma);", "case 1: return exp(-q / sigma);", 0),
    ("laplace_sigma_squared", "case 1: return exp(-sqrt(q) / sigma);",
     "case 1: return exp(-sqrt(q) / (sigma * sigma));", 0),
    ("cauchy_drops_one", "case 2: return 1.0 / (1.0 + q / (sigma * sigma));",
     "case 2: return 1.0 / (q / (sigma * sigma) + 1e-300);", 0),
    ("cauchy_sigma_not_squared", "case 2: return 1.0 / (1.0 + q / (sigma * sigma));",
     "case 2: return 1.0 / (1.0 + q / sigma);", 0),
    ("imq_without_sqrt", "case 3: return 1.0 / sqrt(1.0 + q / (sigma * sigma));",
     "case 3: return 1.0 / (1.0 + q / (sigma * sigma));", 0),
    ("maxmin_ties_keep_last", "int better = sense > 0 ? f > best : f < best;",
     "int better = sense > 0 ? f >= best : f <= best;", 0),
    ("maxmin_min_is_max", "int better = sense > 0 ? f > best : f < best;", "int better = f > best;", 0),
    ("maxmin_runner_not_shifted", "                    runner = best;\n", "", 0),
    ("maxmin_drops_signal",
     "double f = radial_kernel(kind, sq_dist(x + i * D, y + j * D, D), sigma) * b[j * E + e];",
     "double f = radial_kernel(kind, sq_dist(x + i * D, y + j * D, D), sigma);", 0),
    ("ranges_end_inclusive", "j < redranges_j[2 * r + 1]; ++j)", "j <= redranges_j[2 * r + 1] && j < N; ++j)", 0),
    ("ranges_slice_start_off_by_one", "int64_t r0 = c == 0 ? 0 : slices_i[c - 1], r1 = slices_i[c];",
     "int64_t r0 = slices_i[c] - 1, r1 = slices_i[c];", 0),
    ("ranges_ties_keep_scan_order", "int same_lower = f == best && bj >= 0 && j < bj;", "int same_lower = 0;", 0),
    ("ranges_uncovered_max_zero", "val[i] = red == 0 ? 0.0 : (red > 0 ? -INFINITY : INFINITY);",
     "val[i] = 0.0;", 0),
    ("knn_tie_highest_index", "(d1 == d2 && j1 < j2)", "(d1 == d2 && j1 > j2)", 0),
    ("knn_largest_first", "return d1 < d2 ||", "return d1 > d2 ||", 0),
    ("knn_next_is_kth", "next[i] = (K < n) ? bd[K] : INFINITY;",
     "next[i] = (K < n) ? bd[K - 1] : INFINITY;", 0),
    ("knn_fill_zero", "idx[i * K + k] = (k < n) ? bj[k] : -1;",
     "idx[i * K + k] = (k < n) ? bj[k] : 0;", 0),
]


def _mutate(src, old, new, which):
    n = src.count(old)
    assert n >= 1, f"mutation anchor not found in oracle.c: {old!r}"
    if which == "all":
        return src.replace(old, new)
    assert which < n, f"anchor {old!r} occurs {n} times"
    pos = -1
    for _ in range(which + 1):
        pos = src.index(old, pos + 1)
    return src[:pos] + new + src[pos + len(old):]


@pytest.mark.parametrize("name,old,new,which", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, which):
    with open(SRC) as f:
        src = f.read()
    mutated = _mutate(src, old, new, which)
    assert mutated != src
    c = tmp_path / f"{name}.c"
    c.write_text(mutated)
    so = oracle.build(str(c), str(tmp_path / f"lib{name}.so"))
    orc = oracle.Oracle(so)
    caught = []
    for pin in PINS:
        try:
            pin(orc)
        except AssertionError:
            caught.append(pin.__name__)
            break
    assert caught, f"mutant {name} passes every pin"
