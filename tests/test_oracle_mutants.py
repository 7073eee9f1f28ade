"""Each plausible mistake planted in a copy of the oracle (compiled on the CPU) fails a pin.

This shows that the pins constrain every step of the oracle's arithmetic: a dropped term, a
wrong sign, a wrong index or a missing rounding step is caught.
"""

import os
import subprocess

import pytest

import oracle
import oracle_pins

MUTANTS = {
    "delta_sign": ("delta[c] = beta[s] * (vr - acc);", "delta[c] = beta[s] * (acc - vr);"),
    "retrieve_without_decay": ("float a = kv[w] * d[w];", "float a = kv[w];"),
    "write_without_decay": ("fmaf(kv[w], delta[c], decayed)", "fmaf(kv[w], delta[c], rows[(int64_t)w * hd + c])"),
    "write_without_weight": ("fmaf(kv[w], delta[c], decayed)", "(decayed + delta[c])"),
    "k_val_unrounded": ("kv[w] = round_to_bank(k_val[s * W + w], bank_dtype);", "kv[w] = k_val[s * W + w];"),
    "q_val_unrounded": ("float qv = round_to_bank(q_val[s * R + r], bank_dtype);", "float qv = q_val[s * R + r];"),
    "v_unrounded": ("float vr = round_to_bank(v[s * hd + c], bank_dtype);", "float vr = v[s * hd + c];"),
    "shared_gate_index": ("g[s * G + (G == 1 ? 0 : w)]", "g[s * G]"),
    "gate_single_precision_exp": ("d[w] = (float)exp((double)g[s * G + (G == 1 ? 0 : w)]);",
                                  "d[w] = expf(g[s * G + (G == 1 ? 0 : w)]);"),
    "bf16_round_half_up": ("u += 0x7fffu + ((u >> 16) & 1u);", "u += 0x8000u;"),
    "seq_reuses_token0": ("const char* kit = (const char*)k_idx + (size_t)(t * n_streams * W) * ies;",
                          "const char* kit = (const char*)k_idx;"),
    "gather_blocked_groups": ("for (int n = gi; n < width; n += groups) {",
                              "for (int n = gi * ((width + groups - 1) / groups); n < width && "
                              "n < (gi + 1) * ((width + groups - 1) / groups); ++n) {"),
    "gather_padding_stash_kept": ("memset(dst, 0, (size_t)hd * bes);", "(void)dst;"),
    "gather_op1_uses_op0_weights": ("const void* w = o == 0 ? w0 : w1;", "const void* w = w0;"),
    "kpos_padding_written": ("        if ((int)(t % chunk) >= v_t) continue; /* padding: stores nothing */",
                             "        (void)v_t;"),
    "kpos_row_of_entry_0": ("            int64_t slot = load_index(idx0, idx_dtype, t * width0 + n);\n            if (check && (slot",
                            "            int64_t slot = load_index(idx0, idx_dtype, t * width0);\n            if (check && (slot"),
    "gather_padding_not_zeroed": ("for (int64_t c = 0; c < hd; ++c) out[t * hd + c] = 0.0f;",
                                  "for (int64_t c = 0; c < hd; ++c) out[t * hd + c] = out[t * hd + c];"),
}


@pytest.fixture(scope="module")
def source():
    with open(oracle.SOURCE) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, f"mutation site for {name} not found exactly once"
    src = tmp_path / f"{name}.c"
    src.write_text(source.replace(old, new))
    lib = str(tmp_path / f"lib{name}.so")
    subprocess.run(oracle.build_command(str(src), lib), check=True)
    orc = oracle.Oracle(lib)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, oracle.OracleError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
