"""Runs a battery of the oracle's pins against one build of oracle.c and
prints, as the last line, a JSON object {pin name: "pass" | "fail: ..."}.

  python tests/oracle_pin_battery.py PATH_TO_SHARED_LIBRARY

The pins are the functions of test_oracle.py and test_oracle_tables.py,
called directly with fixed arguments; each raises AssertionError when the
build gets its case wrong.  test_oracle_mutation.py runs this script once per
altered copy of the source, each in a process of its own.
"""
import json
import os
import sys
import traceback

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import oracle  # noqa: E402
import test_oracle as to  # noqa: E402
import test_oracle_tables as tt  # noqa: E402
from oracle import MASK_BLOCK, MASK_CAUSAL, MASK_NONE, MASK_SLIDING  # noqa: E402

PINS = [
    ("finite differences, sliding window + sink, GQA",
     to.test_finite_differences, (MASK_SLIDING, True, (2, 4, 2, 9, 9))),
    ("finite differences, block mask + sink", to.test_finite_differences,
     (MASK_BLOCK, True, (1, 2, 1, 13, 13))),
    ("finite differences, causal, GQA", to.test_finite_differences,
     (MASK_CAUSAL, False, (2, 4, 2, 9, 9))),
    ("torch SDPA, no mask + sink", to.test_against_torch_sdpa, (MASK_NONE, True)),
    ("torch SDPA, causal + sink", to.test_against_torch_sdpa, (MASK_CAUSAL, True)),
    ("torch SDPA, sliding window + sink", to.test_against_torch_sdpa, (MASK_SLIDING, True)),
    ("torch SDPA, block mask", to.test_against_torch_sdpa, (MASK_BLOCK, False)),
    ("single visible key", to.test_single_visible_key_closed_form, ()),
    ("sink = -inf is no sink", to.test_sink_minus_inf_is_no_sink, ()),
    ("all-ones block mask is dense", to.test_all_ones_block_mask_equals_dense, ()),
    ("block expansion is the token mask", to.test_block_expansion_equals_token_mask, ()),
    ("column sum of dV, sink", to.test_dv_column_sum, (True,)),
    ("column sum of dV, no sink", to.test_dv_column_sum, (False,)),
    ("shift invariance, sink", to.test_shift_invariance_ties_dsink_to_ds, (True,)),
    ("visible-pair closed forms", to.test_visible_count_closed_forms, ()),
    ("select tables brute force", tt.test_select_tables_brute_force,
     (250, 330, 48, 80, 64, 128)),
    ("select tables brute force, blocks starting on a tile's last row / key",
     tt.test_select_tables_brute_force, (300, 400, 63, 127, 64, 128)),
    ("runbook tile-to-block mapping", tt.test_divisible_mapping_from_runbook, ()),
    ("mask transpose is a permute", tt.test_mask_transpose_is_permute, ()),
]


def main(path):
    oracle.use_library(path)
    out = {}
    for name, fn, args in PINS:
        try:
            fn(*args)
            out[name] = "pass"
        except Exception as e:  # a wrong result, or a shape the build broke
            out[name] = "fail: " + (str(e).splitlines() or [type(e).__name__])[0][:120]
        except BaseException:
            out[name] = "fail: " + traceback.format_exc().splitlines()[-1][:120]
    print(json.dumps(out))


if __name__ == "__main__":
    main(sys.argv[1])
