"""Plant plausible mistakes in copies of the oracle and check that the pins
catch every one (CPU only).  Each mutation is a textual edit of oracle.c that
must match exactly once; the mutant is compiled into a temporary library and
the full pin set is run against it: at least one pin has to fail."""
import os

import pytest

from oracle import build as obuild
from oracle import oracle as orc
from tests import oracle_pins

MUTATIONS = {
    "causal_off_by_one": ("long long hi = qpos + 1;", "long long hi = qpos;"),
    "top_left_causal": ("long long prefix = (long long)seq_lens[s] - q_len;",
                        "long long prefix = 0;"),
    "gqa_head_map": ("int kvh = h / group;", "int kvh = h % num_kv_heads;"),
    "dropped_scale": ("scores[t] = scale * acc + bias;", "scores[t] = acc + bias;"),
    "slot_reversed": ("return (long long)page * block_size + (j % block_size);",
                      "return (long long)page * block_size + (block_size - 1 - j % block_size);"),
    "keys_read_from_values": ("acc += qrow[d] * widen(kc,", "acc += qrow[d] * widen(vc,"),
    "lse_without_max": ("*lse = mx + log(denom);", "*lse = log(denom);"),
    "merge_uniform_weights": ("double w = exp(partial_lse[p] - m) / denom;",
                              "double w = 1.0 / num_parts;"),
    "mla_value_offset": ("(size_t)dk, 0, (size_t)dk, 0, block_table,",
                         "(size_t)dk, 0, (size_t)dk, (size_t)rope_dim, block_table,"),
    "bf16_widening": ("[idx]) << 16;", "[idx]) << 15;"),
    "window_off_by_one": ("lo = qpos - sliding_window + 1;", "lo = qpos - sliding_window;"),
    "alibi_sign": (": -slope * dist;", ": slope * dist;"),
    "alibi_sqrt_ignored": ("bias_sqrt ? -slope * sqrt(dist) :", "bias_sqrt ? -slope * dist :"),
    "alibi_slope_per_kv_head": ("alibi_slopes[h] : 0.0", "alibi_slopes[h / group] : 0.0"),
    "denominator_dropped_term": ("for (long long t = 0; t < n; ++t) {\n    scores[t] = exp(",
                                 "for (long long t = 1; t < n; ++t) {\n    scores[t] = exp("),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, tmp_path):
    src = open(obuild.SRC).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"mutation {name!r} no longer matches the oracle source"
    mutant_src = tmp_path / "oracle_mutant.c"
    mutant_src.write_text(src.replace(old, new))
    lib_path = obuild.build(str(mutant_src), str(tmp_path / "liboracle_mutant.so"))
    lib = orc.load(lib_path)
    failures = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except Exception as exc:  # a failed assertion or an oracle error
            failures.append((pin.__name__, type(exc).__name__))
    assert failures, f"no pin detects mutation {name!r}"


def test_unmutated_copy_passes(tmp_path):
    src = open(obuild.SRC).read()
    p = tmp_path / "oracle_copy.c"
    p.write_text(src)
    lib = orc.load(obuild.build(str(p), str(tmp_path / "liboracle_copy.so")))
    for pin in oracle_pins.ALL_PINS:
        pin(lib)
