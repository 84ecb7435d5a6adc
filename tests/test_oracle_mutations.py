"""The oracle's pins must be sharp: each planted mistake below (a transposed
operand, a flipped sign, a dropped term, a wrong index, a reversed tap order,
a misplaced epsilon, truncation instead of rounding) is compiled into a copy of
the oracle on the CPU, and the pin suite must fail against every copy."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "gdn_oracle.c")

MUTATIONS = {
    "transposed_product": ("sm += S[(size_t)i * dk + l] * M[(size_t)l * dk + j];",
                           "sm += S[(size_t)l * dk + j] * M[(size_t)i * dk + l];"),
    "beta_sign_in_M": ("- beta * khat[l] * khat[j]", "+ beta * khat[l] * khat[j]"),
    "alpha_dropped": ("alpha * sm + beta", "sm + beta"),
    "outer_product_indices": ("beta * v[i] * khat[j]", "beta * v[j % dv] * khat[i % dk]"),
    "output_from_old_state": ("acc += S_new[(size_t)i * dk + j] * qhat[j];",
                              "acc += S[(size_t)i * dk + j] * qhat[j];"),
    "conv_taps_reversed": ("pre += w[(size_t)c * W + j] * win[(size_t)j * C + c];",
                           "pre += w[(size_t)c * W + (W - 2 - j)] * win[(size_t)j * C + c];"),
    "eps_outside_sqrt": ("1.0 / sqrt(ss + eps)", "1.0 / (sqrt(ss) + eps)"),
    "q_scale_missing": ("1.0 / sqrt((double)dk), qhat", "1.0, qhat"),
    "softplus_sign": ("return log1p(exp(x));", "return log1p(exp(-x));"),
    "gqa_interleaved": ("int g = h / group;", "int g = h % hk;"),
    "sigmoid_sign": ("return 1.0 / (1.0 + exp(-b));", "return 1.0 / (1.0 + exp(b));"),
    "dt_bias_dropped": ("gdn_oracle_softplus(a + dt_bias)", "gdn_oracle_softplus(a)"),
    "window_not_shifted": ("new_win[(size_t)j * C + c] = win[(size_t)(j + 1) * C + c];",
                           "new_win[(size_t)j * C + c] = win[(size_t)j * C + c];"),
    "bf16_truncates": ("nearbyint(x / spacing)", "trunc(x / spacing)"),
    "padding_writes_null": ("if (rs == 0) {\n            row_ok[r] = 0;",
                            "if (0) {\n            row_ok[r] = 0;"),
    # many tokens a sequence
    "prefill_state_not_carried": ("memcpy(S, S_new, sizeof(double) * head_elems);", ""),
    "prefill_tokens_reversed": ("for (int t = cu_seqlens[r]; t < cu_seqlens[r + 1]; ++t) {\n            gdn_oracle_head(",
                                "for (int t = cu_seqlens[r + 1] - 1; t >= cu_seqlens[r]; --t) {\n            gdn_oracle_head("),
    "verify_one_token_slot": ("pool + (size_t)token_slot[t] * slot_elems", "pool + (size_t)token_slot[cu_seqlens[r]] * slot_elems"),
    "prefill_twin_writes_read_slot": ("int ws = write_slot ? write_slot[r] : rs;", "int ws = rs;"),
    "conv_prefill_window_not_carried": ("memcpy(win, new_win, sizeof(double) * slot_elems);", ""),
    "copy_slots_may_write_null": ("dst[i] <= 0 || dst[i] >= num_slots", "dst[i] < 0 || dst[i] >= num_slots"),
    # the layer's composition: rounding, activation forwarding, in-place window
    "layer_rounding_dropped": ("y[(size_t)r * C + c] = act_bf16 ? gdn_oracle_round_bf16(t) : gdn_oracle_round_f32(t);",
                               "y[(size_t)r * C + c] = t;"),
    "layer_silu_not_forwarded": ("keep_in_place ? NULL : write_slot, w, bias, silu, y);",
                                 "keep_in_place ? NULL : write_slot, w, bias, 0, y);"),
    "layer_window_to_twin_in_place": ("keep_in_place ? NULL : write_slot, w, bias, silu, y);",
                                      "write_slot, w, bias, silu, y);"),
    "copy_slots_reversed": ("pool[(size_t)dst[i] * slot_elems + e] = pool[(size_t)src[i] * slot_elems + e];",
                            "pool[(size_t)src[i] * slot_elems + e] = pool[(size_t)dst[i] * slot_elems + e];"),
}
PIN_FILES = ["test_oracle_pins.py", "test_oracle_prefill_pins.py"]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    src = open(SRC).read()
    old, new = MUTATIONS[name]
    assert old in src, f"mutation site for {name} not found"
    cfile = tmp_path / "mut.c"
    cfile.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", str(so),
                    str(cfile), "-lm"], check=True)
    env = dict(os.environ, GDN_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        *[os.path.join(ROOT, "tests", f) for f in PIN_FILES]],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch {name}:\n{r.stdout[-2000:]}"
