"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch every one of them.  The committed oracle is never modified: each case
edits the C source text in memory and compiles it into a temporary library.
"""
import os

import pytest

import oracle as oracle_pkg
from oracle_pins import failing_pins

# (name, original text, replacement): each a single plausible slip.
MUTANTS = [
    ("no_score_scale", "    s *= scale;\n    s -= alibi", "    s -= alibi"),
    ("alibi_sign", "    s -= alibi * fabs((double)(r - j));", "    s += alibi * fabs((double)(r - j));"),
    ("alibi_no_abs", "    s -= alibi * fabs((double)(r - j));", "    s -= alibi * (double)(r - j);"),
    ("bmask_ignored", "    if (bmask && !bmask[(size_t)(r / 128) * nb + j / 128]) {",
     "    if (0) {"),
    ("bmask_transposed", "    if (bmask && !bmask[(size_t)(r / 128) * nb + j / 128]) {",
     "    if (bmask && !bmask[(size_t)(j / 128) * nb + r / 128]) {"),
    ("bmask_block_64", "    if (bmask && !bmask[(size_t)(r / 128) * nb + j / 128]) {",
     "    if (bmask && !bmask[(size_t)(r / 128) * nb + (j / 64 < nb ? j / 64 : nb - 1)]) {"),
    ("decode_alibi_top_aligned", "      s -= J->alibi * fabs((double)(J->Nk - J->Nq + i - j));",
     "      s -= J->alibi * fabs((double)(i - j));"),
    ("no_max_shift", "p[j] = exp(p[j] - mx);", "p[j] = exp(p[j]);"),
    ("causal_off_by_one", "int ncols = causal ? r + 1 : N;",
     "int ncols = causal ? (r > 0 ? r : 1) : N;"),
    ("lse_log2", "return mx + log(z);", "return mx + log2(z);"),
    ("ds_sign", "dp[j] = p[j] * (dp[j] - D);", "dp[j] = p[j] * (dp[j] + D);"),
    ("ds_missing_d", "dp[j] = p[j] * (dp[j] - D);", "dp[j] = p[j] * dp[j];"),
    ("dq_no_scale", "for (int c = 0; c < d; ++c) dqr[c] *= J->scale;", ""),
    ("dk_transposed_operand", "dkj[c] += ds * qr[c];", "dkj[c] += ds * dor[c];"),
    ("dv_wrong_operand", "dvj[c] += pv * dor[c];", "dvj[c] += pv * qr[c];"),
    ("dp_wrong_index", "const double* vj = J->v + (size_t)j * d;\n      double s = 0.0;\n      for (int c = 0; c < d; ++c) s += dor[c] * vj[c];",
     "const double* vj = J->v + (size_t)j * d;\n      double s = 0.0;\n      for (int c = 0; c < d; ++c) s += dor[c] * vj[d - 1 - c];"),
    ("online_no_acc_rescale", "for (int c = 0; c < d; ++c) acc[c] *= a_old;", ""),
    ("online_garbled_l_update", "double l_new = a_old * l + a_blk * lj;",
     "double l_new = a_old * l + lj;"),
    ("online_no_fj_rescale", "for (int t = 0; t < w; ++t) x[t] *= a_blk; /* f_j rescale */", ""),
    ("decode_causal_top_aligned", "int ncols = J->causal ? J->Nk - J->Nq + i + 1 : J->Nk;",
     "int ncols = J->causal ? i + 1 : J->Nk;"),
    ("decode_causal_off_by_one", "int ncols = J->causal ? J->Nk - J->Nq + i + 1 : J->Nk;",
     "int ncols = J->causal ? J->Nk - J->Nq + i : J->Nk;"),
    ("decode_no_normalise", "const double pj = p[j] / z;", "const double pj = p[j];"),
    ("dropout_no_rescale",
     "      if (J->dr) pj = dropout_keep(J->dr, r, j) ? pj * (256.0 / J->dr->t) : 0.0;",
     "      if (J->dr) pj = dropout_keep(J->dr, r, j) ? pj : 0.0;"),
    ("dropout_rescale_by_p", "? pj * (256.0 / J->dr->t) : 0.0;",
     "? pj / (1.0 - J->dr->t / 256.0) : 0.0;"),
    ("dropout_dp_not_dropped",
     "      if (J->dr) s = dropout_keep(J->dr, r, j) ? s * (256.0 / J->dr->t) : 0.0;\n", ""),
    ("dropout_dv_not_dropped",
     "      if (J->dr) pv = dropout_keep(J->dr, r, j) ? pv * (256.0 / J->dr->t) : 0.0;\n", ""),
    ("dropout_head_ignored", "(unsigned int)(j / 16), dr->head, dr->offset}",
     "(unsigned int)(j / 16), 0u, dr->offset}"),
    ("dropout_byte_order", "unsigned int byte = (x[b / 4] >> (8 * (b % 4))) & 0xFFu;",
     "unsigned int byte = (x[b % 4] >> (8 * (b / 4))) & 0xFFu;"),
    ("dropout_keep_ge", "  return byte < (unsigned int)dr->t;", "  return byte >= (unsigned int)dr->t;"),
    ("dropout_threshold_trunc", "int t = (int)floor(256.0 * (1.0 - p) + 0.5);",
     "int t = (int)(256.0 * (1.0 - p));"),
    ("philox_output_order", "    x1 = lo1;", "    x1 = lo0;"),
    ("philox_no_key_bump", "    k0 += (W0);", "    k0 += 0;"),
    ("philox32_multiplier", "0xD2511F53u", "0xD2511F55u"),
    ("philox32_weyl", "0xBB67AE85u", "0xBB67AE87u"),
    ("philox32_nine_rounds", "for (int round = 0; round < 10; ++round)",
     "for (int round = 0; round < 9; ++round)"),
]


@pytest.fixture(scope="module")
def source():
    with open(oracle_pkg.SRC) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(source, tmp_path, name, old, new):
    assert source.count(old) == 1, f"mutation site for {name} not unique"
    lib = oracle_pkg.build_from_text(source.replace(old, new), str(tmp_path))
    mutant = oracle_pkg.Oracle(lib)
    bad = failing_pins(mutant, first_only=True)
    assert bad, f"planted mistake {name} passed every pin"
    os.remove(lib)
