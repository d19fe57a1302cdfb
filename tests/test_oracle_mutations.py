"""Planted mistakes in the oracle: each case compiles a copy of the oracle's C source with one
plausible mistake (a wrong tie rule, an off-by-one exponent or E8M0 code, a flipped margin sign, a
window that forgets its history or a NaN, a block amax over part of its block, a scale read from the
wrong row or K block, a column-wise copy in the wrong order, a subnormal decoded one binade off, a
statistic that counts zeros, a cast that drops its scale) and checks that the pin written for that
function fails on it.
The same pins pass on the real oracle in their own modules, so together they show that the pins
are sharp enough to catch that class of mistake."""
import contextlib

import pytest

import oracle as o
import test_oracle_alternatives as alternative_pins
import test_oracle_bias as bias_pins
import test_oracle_codec as codec_pins
import test_oracle_f32cast as f32cast_pins
import test_oracle_history_gemm as history_gemm_pins
import test_oracle_quant as quant_pins
import test_oracle_stats as stats_pins


@contextlib.contextmanager
def _mutant(tmp_path, old, new):
    src = open(o._SRC).read()
    assert src.count(old) == 1, old
    path = tmp_path / "fp8_oracle.c"
    path.write_text(src.replace(old, new))
    o.lib()  # the real oracle is loaded (and built) before it is swapped out
    saved = (o._SRC, o._LIB, o._lib)
    o._SRC, o._LIB, o._lib = str(path), str(tmp_path / "liboracle.so"), None
    try:
        o.lib()
        yield o
    finally:
        o._SRC, o._LIB, o._lib = saved


MUTANTS = {
    "ties round away from even": (
        "else c = (lo & 1) ? hi : lo;", "else c = hi;",
        lambda m: codec_pins.test_midpoints_tie_to_even(m, 0)),
    "subnormals decoded one binade low": (
        "v = ldexp((double)m, 1 - bias - mb);", "v = ldexp((double)m, -bias - mb);",
        lambda m: codec_pins.test_decode_matches_torch_all_codes(m, 0)),
    "compute_bias rounds instead of flooring": (
        "long e = (long)(x - 1) - (long)margin;", "long e = (long)x - (long)margin;",
        lambda m: bias_pins.test_bracket_property(m, 0)),
    "margin added instead of subtracted": (
        "long e = (long)(x - 1) - (long)margin;", "long e = (long)(x - 1) + (long)margin;",
        lambda m: bias_pins.test_margin_shift(m, 1, 2)),
    "history window forgets all but its first entry": (
        "int64_t n = *pos < L ? *pos : L;", "int64_t n = 1;",
        lambda m: history_gemm_pins.test_history_window_invariant(m, 4, 0, 0)),
    "sampled product: block scale of B read from row 0": (
        "\n        for (int64_t k = 0; k < K; ++k) {\n"
        "            double a = fp8o_decode(A[m * lda + k], fa) * operand_scale(ga, sfa, m, k, K);\n"
        "            double b = fp8o_decode(B[n * ldb + k], fb) * operand_scale(gb, sfb, n, k, K);",
        "\n        for (int64_t k = 0; k < K; ++k) {\n"
        "            double a = fp8o_decode(A[m * lda + k], fa) * operand_scale(ga, sfa, m, k, K);\n"
        "            double b = fp8o_decode(B[n * ldb + k], fb) * operand_scale(gb, sfb, 0, k, K);",
        lambda m: history_gemm_pins.test_gemm_exact_block(m, 1, 1)),
    "whole product: block scale of B read from row 0": (
        "                double b = fp8o_decode(B[n * ldb + k], fb) * operand_scale(gb, sfb, n, k, K);",
        "                double b = fp8o_decode(B[n * ldb + k], fb) * operand_scale(gb, sfb, 0, k, K);",
        lambda m: history_gemm_pins.test_gemm_full_exact_block(m, 1, 1)),
    "whole product: MX scale of A from the wrong K block": (
        "                double a = fp8o_decode(A[m * lda + k], fa) * operand_scale(ga, sfa, m, k, K);",
        "                double a = fp8o_decode(A[m * lda + k], fa) * operand_scale(ga, sfa, m, k ^ 32, K);",
        lambda m: history_gemm_pins.test_gemm_full_exact_block(m, 3, 3)),
    "amax drops a NaN": (
        "            if (isnan(a) || a > m) m = a;", "            if (a > m) m = a;",
        lambda m: quant_pins.test_amax_matches_numpy(m)),
    "history window drops a NaN": (
        "if (isnan(hist[i]) || hist[i] > m) m = hist[i];", "if (hist[i] > m) m = hist[i];",
        lambda m: history_gemm_pins.test_history_nan_stays_in_window(m)),
    "128x128 block amax taken over its first row only": (
        "float amax = amax_of(x + i0 * rs + j0 * cs, ni, nj, rs, cs);", "float amax = amax_of(x + i0 * rs + j0 * cs, 1, nj, rs, cs);",
        lambda m: quant_pins.test_block_quant_brute_force(m, 2, 0, (130, 96))),
    "E8M0 code off by one": (
        "sf_e8m0[b] = (uint8_t)(127 - e);", "sf_e8m0[b] = (uint8_t)(128 - e);",
        lambda m: quant_pins.test_block_quant_brute_force(m, 3, 0, (3, 160))),
    "OCP bias one binade off": (
        "long e = (long)(fmt == FMT_E4M3 ? 8 : 15) - (long)(x - 1) - (long)margin;",
        "long e = (long)(fmt == FMT_E4M3 ? 8 : 15) - (long)x - (long)margin;",
        lambda m: alternative_pins.test_ocp_hand_values(m, 0, 448.0, 0)),
    "ratio scale through a rounded reciprocal": (
        "(float)fmt_max(fmt) / a;", "(float)fmt_max(fmt) * (1.0f / a);",
        lambda m: alternative_pins.test_ratio_scale_correctly_rounded(m, 0)),
    "flush-to-zero count includes the zeros": (
        "if (xv != 0.0f && (fp8o_encode(v, fmt) & 0x7F) == 0) ++und;", "if ((fp8o_encode(v, fmt) & 0x7F) == 0) ++und;",
        lambda m: stats_pins.test_nan_and_zero_count_in_neither(m)),
    "fp32 cast ignores its scale": (
        "        float p = x[i] * s;", "        float p = x[i];",
        lambda m: f32cast_pins.test_matches_torch_in_range(m, 0, 0.3)),
    "column-wise copy written in reverse row order": (
        "if (q_col) q_col[j * rows + i] = (uint8_t)code;", "if (q_col) q_col[j * rows + (rows - 1 - i)] = (uint8_t)code;",
        lambda m: quant_pins.test_tensor_quant_brute_force(m, 0)),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pin_catches_planted_mistake(tmp_path, name):
    old, new, pin = MUTANTS[name]
    with _mutant(tmp_path, old, new) as m:
        with pytest.raises(AssertionError):
            pin(m)
    pin(o)  # and the real oracle passes the same pin


# The bf16 rounding and the output-cast bracket are Python functions of the oracle: the mistake is
# planted in the function's own source, which is executed in the oracle module's namespace.
PY_MUTANTS = {
    "bf16 rounding truncates": (
        "round_bf16", "r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16", "r = (u >> 16) << 16",
        lambda m: history_gemm_pins.test_round_bf16_matches_torch(m)),
    "output-cast bracket starts at the nearest code": (
        "gemm_quantize_bracket", "return codes(y_ref - tol), codes(y_ref + tol), codes(y_ref)",
        "return codes(y_ref), codes(y_ref + tol), codes(y_ref)",
        lambda m: history_gemm_pins.test_gemm_quantize_bracket_brute_force(m, 0)),
}


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_pin_catches_planted_mistake_in_python(monkeypatch, name):
    import inspect
    import textwrap
    fn, old, new, pin = PY_MUTANTS[name]
    src = textwrap.dedent(inspect.getsource(getattr(o, fn)))
    assert src.count(old) == 1, old
    ns = dict(vars(o))
    exec(compile(src.replace(old, new), f"<mutant {fn}>", "exec"), ns)
    monkeypatch.setattr(o, fn, ns[fn])
    with pytest.raises(AssertionError):
        pin(o)
    monkeypatch.undo()
    pin(o)
