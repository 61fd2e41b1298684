"""Plants plausible mistakes in a temporary copy of the oracle (on the CPU) and checks that
the pins in test_oracle_pins.py catch each one.  The committed oracle is never modified."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "gqa_head_mapping": (
        "int G = pr->num_q_heads / pr->num_kv_heads;\n    return (int64_t)branch_of_token(pr, qt)"
        " * pr->num_kv_heads + h / G;",
        "int G = pr->num_q_heads / pr->num_kv_heads; (void)G;\n    return (int64_t)"
        "branch_of_token(pr, qt) * pr->num_kv_heads + h % pr->num_kv_heads;"),
    "causal_off_by_one": ("if (pos[c] > p_i) break;", "if (pos[c] >= p_i) break;"),
    "missing_scale": ("s[c] = pr->scale * acc;", "s[c] = acc;"),
    "wrong_log_base": ("double L = m + log(sum);", "double L = m + log2(sum);"),
    "slot_ignores_tok_begin": (
        "int64_t slot = (sg[1] + t) % P;\n            const uint16_t *kr",
        "int64_t slot = (t) % P;\n            const uint16_t *kr"),
    "drop_bit_ignored": (
        "visible = (int)((w >> (j % 32)) & 1u);\n            }\n            if (!visible) continue;",
        "visible = (int)((w >> (j % 32)) & 1u); (void)visible;\n            }\n"),
    "value_row_from_keys": ("vc[n_vis * D + d] = widen_bf16(vr[d]);",
                            "vc[n_vis * D + d] = widen_bf16(kr[d]); (void)vr;"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_oracle_mistake(name, tmp_path):
    before, after = MUTATIONS[name]
    src = open(os.path.join(ROOT, "oracle", "fork_attn_oracle.c")).read()
    assert before in src
    ignore = shutil.ignore_patterns("*.so", "__pycache__")
    for d in ("oracle", "tests", "shared_prefix_paged_attn_b300"):
        shutil.copytree(os.path.join(ROOT, d), tmp_path / d, ignore=ignore)
    (tmp_path / "oracle" / "fork_attn_oracle.c").write_text(src.replace(before, after))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py"], cwd=tmp_path, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode != 0, f"planted mistake {name} went unnoticed:\n{r.stdout[-2000:]}"
    assert " failed" in r.stdout
