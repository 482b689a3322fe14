"""The oracle's pins catch plausible mistakes (no GPU).

Each case plants one slip in a temporary copy of the oracle's C source -- a top-left
causal mask, the wrong grouped-query head map, a dropped softmax scale, a log-sum-exp
without its max, an inverted merge weight, V read from K, a mis-decoded bf16 -- builds
it, and checks that the pin suite in test_oracle.py fails against it.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "fa_oracle.c")

MUTATIONS = {
    "top_left_causal": ("long lim = i + J->Sk - J->Sq + 1; /* bottom-right", "long lim = i + 1; /* bottom-right"),
    "window_left_off_by_one": ("long lim = i + J->Sk - J->Sq - J->win_left;",
                               "long lim = i + J->Sk - J->Sq - J->win_left + 1;"),
    "gqa_modulo": ("long hk = h / g; /* grouped-query head map */", "long hk = h % J->Hkv;"),
    "dropped_scale": ("s_buf[t] = scale * dot;", "s_buf[t] = dot;"),
    "lse_without_max": ("*lse = m + log(l);", "*lse = log(l);"),
    "merge_weight_inverted": ("double w = exp(lse_parts[s] - total);",
                              "double w = exp(total - lse_parts[s]);"),
    "v_read_from_k": ("o[d] += p * load_elem(v, dtype, vbase + d);",
                      "o[d] += p * load_elem(k, dtype, vbase + d);"),
    "paged_table_stride": ("const long pg = block_table[b * max_pages + j / page_size];",
                           "const long pg = block_table[b + j / page_size];"),
    "bf16_decode_shift": ("uint32_t u = (uint32_t)h << 16;", "uint32_t u = (uint32_t)h << 15;"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_fail_on_planted_mistake(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no host C compiler")
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutant = tmp_path / "fa_oracle_mutant.c"
    mutant.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", str(lib), str(mutant),
                    "-lpthread", "-lm"], check=True)
    env = dict(os.environ, FA_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutation {name}:\n{r.stdout[-2000:]}"
