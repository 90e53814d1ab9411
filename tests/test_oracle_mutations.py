"""Plant plausible mistakes in a copy of the oracle and check that the pins catch them.

Each mutation rewrites one line of ``oracle/attention_oracle.c`` in a temporary
copy (a dropped term, a wrong sign, a wrong index, an off-by-one mask), builds
it with gcc and runs the pin checks of ``test_oracle.py`` against it.  Every
mutant must fail at least one pin; the unmodified source must pass all of them.
"""
import os
import shutil

import numpy as np
import pytest

import oracle
from tests.golden import fixtures

MUTATIONS = {
    "lse_drops_scale": ("*lse_out = s * m + log(l);", "*lse_out = m + log(l);"),
    "exponent_sign": ("double w = exp(s * (x[j] - m));", "double w = exp(s * (m - x[j]));"),
    "spread_drops_abs": ("spread[c] += p * fabs(vj[c] - o_row[c]);",
                         "spread[c] += p * (vj[c] - o_row[c]);"),
    "causal_off_by_one": ("int64_t end = i + 1 + (mask == 2 ? Nk - Nq : 0);",
                          "int64_t end = i + (mask == 2 ? Nk - Nq : 0);"),
    "bottom_right_offset_sign": ("int64_t end = i + 1 + (mask == 2 ? Nk - Nq : 0);",
                                 "int64_t end = i + 1 + (mask == 2 ? Nq - Nk : 0);"),
    "no_normalisation": ("for (int64_t c = 0; c < d; ++c) o_row[c] /= l;",
                         "for (int64_t c = 0; c < d; ++c) o_row[c] /= 1.0;"),
    "wrong_value_row": ("l += w;\n        const double* vj = v + j * d;",
                        "l += w;\n        const double* vj = v + (nvalid - 1 - j) * d;"),
    "score_uses_wrong_key": ("const double* kj = k + j * d;",
                             "const double* kj = k + (j == 0 ? 0 : j - 1) * d;"),
    "recurrence_drops_alpha_on_l": ("l *= alpha;", "l *= 1.0;"),
    "recurrence_drops_alpha_on_u": ("for (int64_t c = 0; c < d; ++c) u[c] *= alpha;",
                                    "for (int64_t c = 0; c < d; ++c) u[c] *= 1.0;"),
    "recurrence_alpha_sign": ("alpha = exp(scale * (m - m_new));",
                              "alpha = exp(scale * (m_new - m));"),
    "recurrence_weights_use_old_max": ("double w = exp(scale * (x[j - j0] - m_new));",
                                       "double w = exp(scale * (x[j - j0] - m));"),
    "fp16_exponent_bias": ("mag = ldexp((double)(frac + 1024), expo - 25);",
                           "mag = ldexp((double)(frac + 1024), expo - 24);"),
    "bf16_fraction_width": ("mag = ldexp((double)(frac + 128), expo - 134);",
                            "mag = ldexp((double)(frac + 64), expo - 133);"),
}


def _pins(lib) -> list:
    """Run the pin checks against `lib`; return the names of those that fail."""
    failed = []
    ex = fixtures.load("worked_example.txt")
    cz = fixtures.load("worked_example_causal.txt")

    def check(name, ok):
        if not ok:
            failed.append(name)

    o, lse = oracle.attention(ex["Q"], ex["K"], ex["V"], ex["scale"], lib=lib)
    check("worked_plain", np.allclose(o, ex["O"], atol=1e-14)
          and np.allclose(lse, ex["LSE"], atol=1e-14))
    o, lse = oracle.attention(ex["Q"], ex["K"], ex["V"], cz["scale"], True, lib=lib)
    check("worked_causal", np.allclose(o, cz["O"], atol=1e-14)
          and np.allclose(lse, cz["LSE"], atol=1e-14))
    br = fixtures.load("worked_example_bottom_right.txt")
    o, lse = oracle.attention(ex["Q"], ex["K"], ex["V"], br["scale"], oracle.BOTTOM_RIGHT, lib=lib)
    check("worked_bottom_right", np.allclose(o, br["O"], atol=1e-14)
          and np.allclose(lse, br["LSE"], atol=1e-14))
    o, lse, tr = oracle.blocked_head(ex["Q"], ex["K"], ex["V"], ex["scale"], False, 2,
                                     trace=True, lib=lib)
    check("worked_recurrence", np.allclose(tr["l"][1], ex["l1"], atol=1e-14)
          and np.allclose(tr["u"][1], ex["U1"], atol=1e-14)
          and np.allclose(o, ex["O"], atol=1e-14))
    rng = np.random.default_rng(1)
    ok = True
    for n in (3, 6):
        q, k, v = (rng.standard_normal((n, 3)) for _ in range(3))
        for causal in (False, True):
            o_ref, l_ref = oracle.attention(q, k, v, 0.7, causal, lib=lib)
            for bn in (1, 2, n):
                o2, l2 = oracle.blocked_head(q, k, v, 0.7, causal, bn, lib=lib)
                ok &= np.allclose(o2, o_ref, atol=1e-12) and np.allclose(l2, l_ref, atol=1e-12)
    check("blocked_vs_plain", ok)
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        ref16 = bits.view(np.float16).astype(np.float64)
        refb = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    d16 = oracle.decode16(bits, oracle.FP16, lib=lib)
    db = oracle.decode16(bits, oracle.BF16, lib=lib)
    check("decode16", np.array_equal(d16, ref16, equal_nan=True)
          and np.array_equal(db, refb, equal_nan=True))
    from online_softmax_tiling_gb300 import synth
    v = synth.round_to_bits(np.array([[[[1.0, -2.0], [3.0, 0.5]]]]), oracle.FP16)
    z = np.zeros((1, 1, 2, 2), np.uint16)
    _, _, sp = oracle.attention_rows16(z, z, v, oracle.FP16, 1.0, False, [0, 1],
                                       with_spread=True, lib=lib)
    check("spread_closed_form", np.allclose(sp, [[1.0, 1.25], [1.0, 1.25]], atol=1e-15))
    return failed


def _build_variant(tmp_path, name, old, new):
    src = open(oracle.SOURCE, encoding="utf-8").read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new), encoding="utf-8")
    return oracle.build(str(path), str(tmp_path / f"lib{name}.so"), force=True)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_unmodified_oracle_passes_all_pins():
    assert _pins(oracle.load()) == []


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTATIONS[name]
    lib = oracle.load(_build_variant(tmp_path, name, old, new))
    assert _pins(lib), f"mutation {name} passed every pin"
