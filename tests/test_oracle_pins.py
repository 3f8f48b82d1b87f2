"""The CPU oracle against what the pages and the mathematics fix (no GPU).

Every pin in tests/pins.py runs against the oracle as built.  The mutation
tests then compile copies of oracle.c with one plausible mistake planted each
(a dropped term, a wrong index, a flipped sign, a reversed order, a wrong
bias...) and check that some pin fails for every one of them.
"""
import json
import os
import subprocess
import sys

import pytest

import oracle
from tests import pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, olib):
    pin(olib)


# (name, exact text in oracle.c, replacement, pins expected to catch it)
MUTANTS = [
    ("plan_cursor_not_advanced", "cursor[e] += 1;", ";",
     [pins.pin_plan_hand_example, pins.pin_plan_bruteforce]),
    ("plan_scan_inclusive", "off[e + 1] = off[e] + cnt[e];", "off[e + 1] = off[e] + cnt[e] + (e == 0);",
     [pins.pin_plan_hand_example, pins.pin_plan_bruteforce]),
    ("plan_invalid_not_marked", "tok_map[i] = -1;\n            }\n        }\n    }\n    free(cursor);\n    *n_invalid",
     "tok_map[i] = 0;\n            }\n        }\n    }\n    free(cursor);\n    *n_invalid",
     [pins.pin_plan_hand_example, pins.pin_plan_bruteforce]),
    ("plan_reverse_tokens", "for (int64_t s = 0; s < S; ++s) {\n        for (int k = 0; k < K; ++k) {\n            int64_t i = s * K + k;\n            int32_t e",
     "for (int64_t s = S - 1; s >= 0; --s) {\n        for (int k = 0; k < K; ++k) {\n            int64_t i = s * K + k;\n            int32_t e",
     [pins.pin_plan_hand_example, pins.pin_plan_bruteforce]),
    ("plan_src_is_token", "packed_src[row] = (int32_t)i;", "packed_src[row] = (int32_t)s;",
     [pins.pin_plan_hand_example, pins.pin_plan_bruteforce]),
    ("group_rep_last_not_first", "if (group_of(topk_idx[s * K + kp], E, group_size) == g)\n                    first = 0;",
     "if (group_of(topk_idx[s * K + kp], E, group_size) == g && 0)\n                    first = 0;",
     [pins.pin_group_plan_bruteforce, pins.pin_group_plan_invariants]),
    ("group_map_wrong_token", "grp_tok_map[r * K + k2] = (g2 == g) ? tok_map[s * K + k2] : -1;",
     "grp_tok_map[r * K + k2] = (g2 == g) ? tok_map[s * K + k] : -1;",
     [pins.pin_group_plan_bruteforce, pins.pin_dispatch_dedup]),
    ("dispatch_wrong_source_row", "memcpy(packed + row * row_bytes, rows + s * row_bytes",
     "memcpy(packed + row * row_bytes, rows + (s ^ 1) * row_bytes",
     [pins.pin_dispatch_scatter, pins.pin_combine_identity_telescopes]),
    ("combine_drops_last_k", "for (int k = 0; k < K; ++k) {\n                int64_t row = tok_map[s * K + k];",
     "for (int k = 0; k < K - 1; ++k) {\n                int64_t row = tok_map[s * K + k];",
     [pins.pin_combine_identity_telescopes, pins.pin_combine_exact_rational]),
    ("combine_reverse_k", "for (int k = 0; k < K; ++k) {\n                int64_t row = tok_map[s * K + k];",
     "for (int k = K - 1; k >= 0; --k) {\n                int64_t row = tok_map[s * K + k];",
     [pins.pin_combine_k_order]),
    ("combine_weight_index", "float term = w[s * K + k] * load_elem(y, in_dt, row * H + j);\n                acc = acc + term;\n            }\n            store_elem(out",
     "float term = w[k] * load_elem(y, in_dt, row * H + j);\n                acc = acc + term;\n            }\n            store_elem(out",
     [pins.pin_combine_identity_telescopes, pins.pin_combine_exact_rational]),
    ("combine_sign", "acc = acc + term;\n            }\n            store_elem(out",
     "acc = acc - term;\n            }\n            store_elem(out",
     [pins.pin_combine_identity_telescopes]),
    ("combine_transposed_y", "load_elem(y, in_dt, row * H + j);\n                acc = acc + term;\n            }\n            store_elem(out",
     "load_elem(y, in_dt, j * H + row);\n                acc = acc + term;\n            }\n            store_elem(out",
     [pins.pin_combine_identity_telescopes, pins.pin_combine_exact_rational]),
    ("dedup_stage2_weighted", "acc = acc + gtok[r * H + j];", "acc = acc + w[s * K + k] * gtok[r * H + j];",
     [pins.pin_combine_dedup_closed_forms]),
    ("fold_counts_unused_entries", "if (map[s * K + k] >= 0)\n                    acc = acc + w[s * K + i];",
     "if (map[s * K + k] >= -1)\n                    acc = acc + w[s * K + i];",
     [pins.pin_combine_fold_direct_map]),
    ("fold_sums_other_weights", "acc = acc + w[s * K + i];", "acc = acc + w[s * K + k];",
     [pins.pin_combine_fold_group_rows, pins.pin_combine_fold_direct_map]),
    ("fold_unweighted_still_weights", "acc = acc + (weighted ? w[s * K + k] * v : v);",
     "acc = acc + w[s * K + k] * v;",
     [pins.pin_combine_fold_group_rows, pins.pin_combine_fold_direct_map]),
    ("fold_weighted_ignores_weights", "acc = acc + (weighted ? w[s * K + k] * v : v);",
     "acc = acc + v;", [pins.pin_combine_fold_weighted_telescopes]),
    ("bf16_ties_away", "if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u)))",
     "if (rest >= 0x8000u)", [pins.pin_bf16_rounding]),
    ("bf16_truncates", "keep += 1u;", ";", [pins.pin_bf16_rounding, pins.pin_combine_exact_rational]),
    ("e4m3_bias_8", "pow(2.0, ex - 7)", "pow(2.0, ex - 8)", [pins.pin_e4m3_table]),
    ("e4m3_subnormal_exp", "pow(2.0, -6)", "pow(2.0, -7)", [pins.pin_e4m3_table]),
    ("expert_scale_wrong_expert", "* c[e]);", "* c[e == 0 ? 0 : e - 1]);",
     [pins.pin_expert_stages, pins.pin_combine_expert_scale_closed_form]),
    ("dequant_wrong_block", "scales[r * nb + j / block]", "scales[r * nb + j % nb]",
     [pins.pin_expert_stages]),
    ("capacity_keeps_late_entries", "if (slot < capacity) {", "if (slot < capacity + (s > 0)) {",
     [pins.pin_plan_capacity_bruteforce, pins.pin_plan_capacity_hand_example]),
    ("capacity_cnt_uncapped", "cnt[e] = (int32_t)(seen[e] < capacity ? seen[e] : capacity);",
     "cnt[e] = (int32_t)seen[e];", [pins.pin_plan_capacity_bruteforce]),
    ("e4m3_encode_ties_up", "code = (lo & 1) ? (uint8_t)(lo + 1) : lo;  /* tie: even mantissa */",
     "code = (uint8_t)(lo + 1);", [pins.pin_e4m3_encode]),
    ("e4m3_encode_overflow_to_nan", "if (a >= 448.0)\n        return (uint8_t)(sign | 0x7e);",
     "if (a >= 448.0)\n        return (uint8_t)(sign | 0x7f);", [pins.pin_e4m3_encode]),
    ("quant_scale_off_by_max", "float scale = (amax > 0.0f) ? amax / 448.0f : 1.0f;",
     "float scale = (amax > 0.0f) ? amax / 240.0f : 1.0f;", [pins.pin_quant_fp8_rule]),
    ("quant_multiplies", "q[s * H + b * block + j] = oracle_f32_to_e4m3(v / scale);",
     "q[s * H + b * block + j] = oracle_f32_to_e4m3(v * (1.0f / scale));", [pins.pin_quant_fp8_rule]),
]


@pytest.mark.parametrize("name,old,new,catchers", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, catchers, tmp_path):
    src = open(oracle._SRC).read()
    assert src.count(old) >= 1, f"anchor for mutant {name} not found in oracle.c"
    mutated = src.replace(old, new, 1)
    assert mutated != src
    csrc = tmp_path / "mutant.c"
    csrc.write_text(mutated)
    so = tmp_path / "libmutant.so"
    oracle.build(str(csrc), str(so))
    # run the pins in a child process so that a mutant which corrupts memory
    # cannot take the test session down with it
    script = (
        "import json, sys\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "import oracle\n"
        "from tests import pins\n"
        f"lib = oracle.load({str(so)!r})\n"
        "caught = []\n"
        f"for name in {[c.__name__ for c in catchers]!r}:\n"
        "    try:\n"
        "        getattr(pins, name)(lib)\n"
        "    except AssertionError:\n"
        "        caught.append(name)\n"
        "print(json.dumps(caught))\n")
    r = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, f"mutant {name}: child exited {r.returncode}: {r.stderr[-2000:]}"
    caught = json.loads(r.stdout.strip().splitlines()[-1])
    assert caught, f"mutant {name} passed every pin it should fail"
