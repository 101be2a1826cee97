"""Planted mistakes: each copy of the oracle below carries one plausible
error (a dropped term, a wrong sign or index, reversed taps, a misplaced
epsilon, ...).  The pin suite, run against that copy in a child process,
must fail.  Mistakes are planted in a temporary copy of the C source on the
CPU; the real oracle is never modified."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "kda_oracle.c")

MUTANTS = {
    "dropped_beta_k_v_term": (
        "- beta * k[i] * u[j] + beta * k[i] * v[j];", "- beta * k[i] * u[j];"),
    "wrong_sign_on_erase": (
        "- beta * k[i] * u[j] + beta * k[i] * v[j];", "+ beta * k[i] * u[j] + beta * k[i] * v[j];"),
    "decay_on_value_index": (
        "S[(size_t)i * V + j] *= alpha[i];", "S[(size_t)i * V + j] *= alpha[j % K];"),
    "l2_eps_outside_sqrt": (
        "double inv = 1.0 / sqrt(ss + eps);", "double inv = 1.0 / (sqrt(ss) + eps);"),
    "rms_eps_outside_sqrt": (
        "double r = 1.0 / sqrt(ss / (double)V + eps);", "double r = 1.0 / (sqrt(ss / (double)V) + eps);"),
    "reversed_conv_taps": (
        "wt[t] = (double)wc[(int64_t)t * D_c", "wt[t] = (double)wc[(int64_t)(W - 1 - t) * D_c"),
    "conv_state_shift_wrong_end": ("CS(W - 2) = xin;", "CS(0) = xin;"),
    "gate_silu_not_sigmoid": (
        "* w[j] * kda_oracle_sigmoid(gate[j]);", "* w[j] * kda_oracle_silu(gate[j]);"),
    "q_scale_from_value_dim": (
        "1.0 / sqrt((double)K);", "1.0 / sqrt((double)V);"),
    "slot_zero_not_padding": ("if (s <= 0 || s >= p->num_slots) {", "if (s < 0 || s >= p->num_slots) {"),
    "bf16_ties_away": (
        "if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;",
        "if (rem >= 0.5) fl += 1.0;"),
    "gate_drops_dt_bias": (
        "if (p->dt_bias) z += (double)p->dt_bias[(int64_t)h * K + i];", "(void)0;"),
    "gate_uses_A_log_not_exp": (
        "if (lower_bound < 0.0) return lower_bound * kda_oracle_sigmoid(exp(A_log) * z);",
        "if (lower_bound < 0.0) return lower_bound * kda_oracle_sigmoid(A_log * z);"),
    "sd_layout_taps_newest_first": (
        "#define CS(t) cs0[ch * cs_ch + (int64_t)(t) * cs_t]",
        "#define CS(t) cs0[ch * cs_ch + (int64_t)(p->conv_state_sd ? (W - 2 - (t)) : (t)) * cs_t]"),
    "readout_skips_last_key": (
        "for (int i = 0; i < K; ++i) acc += S[(size_t)i * V + j] * q[i];",
        "for (int i = 0; i < K - 1; ++i) acc += S[(size_t)i * V + j] * q[i];"),
    # prefill (token loop of the varlen batch)
    "prefill_window_not_slid": ("          wm[W - 2] = xin;\n", ""),
    "prefill_state_reloaded_every_token": (
        "    /* 1. conv + SiLU with the window, then slide the window */",
        "    for (int64_t e = 0; e < (int64_t)K * V; ++e) S[e] = (double)Sg[e];"),
    "prefill_final_window_not_stored": (
        "      for (int t = 0; t < W - 1; ++t) cs0[ch * cs_ch + t * cs_t] = win[(size_t)m * (W - 1) + t];",
        "      (void)0;"),
    "prefill_beta_of_first_token": (
        "kda_oracle_bf16_to_f64(p->beta[(int64_t)r * H + h]);",
        "kda_oracle_bf16_to_f64(p->beta[(int64_t)r0 * H + h]);"),
    "prefill_slot_zero_not_padding": (
        "if (s < 1 || s >= p->num_slots) { /* padding or out of range */",
        "if (s < 0 || s >= p->num_slots) { /* padding or out of range */"),
    "prefill_q_scale_from_value_dim": ("pow((double)K, -0.5);", "pow((double)V, -0.5);"),
    "prefill_gate_drops_dt_bias": (
        "        if (p->dt_bias) zz += (double)p->dt_bias[(int64_t)h * K + i];", "        (void)zz;"),
    "prefill_gate_beta_not_activated": ("      beta = kda_oracle_sigmoid(beta);\n    } else {", "    } else {"),
    "prefill_sd_taps_newest_first": (
        "  const int64_t cs_t = p->conv_state_sd ? C : 1;\n  /* window",
        "  const int64_t cs_t = p->conv_state_sd ? -C : 1;\n  cs0 += p->conv_state_sd ? (W - 2) * C : 0;\n  /* window"),
    "prefill_decay_of_previous_token": (
        "alpha[i] = exp((double)p->g[((int64_t)r * H + h) * K + i]);",
        "alpha[i] = exp((double)p->g[((int64_t)(r > r0 ? r - 1 : r) * H + h) * K + i]);"),
    # multi-token (speculative) decode
    "multi_window_not_slid": ("        for (int k = 0; k < W - 2; ++k) wm[k] = wm[k + 1];\n        wm[W - 2] = xin;\n", ""),
    "multi_state_reread_every_token": (
        "    const int32_t dst = p->dst_slots[r];",
        "    const int32_t dst = p->dst_slots[r];\n    for (int64_t e = 0; e < (int64_t)K * V; ++e) S[e] = (double)S_src[e];"),
    "multi_window_stored_to_source": (
        "uint16_t* cs_dst = p->conv_state + (int64_t)dst * C * (W - 1);",
        "uint16_t* cs_dst = p->conv_state + (int64_t)src * C * (W - 1);"),
    "multi_slot_zero_not_absent": (
        "if (dst <= 0 || dst >= p->num_slots) { /* absent token */",
        "if (dst < 0 || dst >= p->num_slots) { /* absent token */"),
    "multi_decay_of_first_token": (
        "alpha[i] = exp((double)p->g[(r * H + h) * K + i]);",
        "alpha[i] = exp((double)p->g[((int64_t)n * T * H + h) * K + i]);"),
    "multi_padding_source_processed": (
        "if (src <= 0 || src >= p->num_slots) { /* padding or out-of-range sequence */",
        "if (src < 0 || src >= p->num_slots) { /* padding or out-of-range sequence */"),
}

PIN_FILES = ("test_oracle_pins.py", "test_prefill_oracle_pins.py", "test_multi_oracle_pins.py")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    (tmp_path / "kda_oracle.c").write_text(src.replace(old, new))
    hdr = os.path.join(ROOT, "oracle", "kda_oracle.h")
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                    "-I", os.path.dirname(hdr), str(tmp_path / "kda_oracle.c"), "-o", str(so), "-lm"],
                   check=True)
    env = dict(os.environ, KDA_ORACLE_SO=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        *[os.path.join(ROOT, "tests", f) for f in PIN_FILES]],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    # exit code 1 = some test failed (not a crash, not a collection error)
    assert r.returncode == 1, f"mutant {name} survived or crashed:\n{r.stdout[-2000:]}\n{r.stderr[-2000:]}"
