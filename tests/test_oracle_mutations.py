"""The oracle's pins have power: planting a plausible mistake in the oracle
(a copy of its C source, built in a temporary directory, on the CPU) makes at
least one pin fail.  Each mutant is loaded in place of the real oracle
library for the duration of one check and the real one is restored after.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
import test_oracle_attention as TA
import test_oracle_stree as TS
import test_oracle_tree as TT
import test_oracle_verify as TV

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text in oracle.c, replacement, pins expected to catch it)
MUTANTS = [
    ("gqa head mapping h % Hkv", "const int kvh = h / G;", "const int kvh = h % Hkv;",
     [TA.test_gqa_head_mapping]),
    ("tree mask transposed", "mask[(size_t)t * T + (j - L)]", "mask[(size_t)(j - L) * T + t]",
     [lambda o: TA.test_tree_node_equals_attention_over_its_own_path(o, "random")]),
    ("last prefix slot dropped", "int allowed = (j < L) ? 1", "int allowed = (j < L - 1) ? 1",
     [TA.test_single_query_is_plain_decode_attention]),
    ("softmax scale dropped", "scores[j] = scale * acc;", "scores[j] = acc;",
     [TA.test_single_query_is_plain_decode_attention]),
    ("accept comparison reversed", "if (!(uq < p))", "if (!(uq > p))",
     [lambda o: TV.test_enumeration_emitted_token_is_target_distribution(o, 0)]),
    ("residual replaced by p", "r[v] = diff > 0.0 ? diff : 0.0;",
     "r[v] = row_prob(trow, dtype, v, mt, stt);",
     [lambda o: TV.test_enumeration_emitted_token_is_target_distribution(o, 0)]),
    ("bonus drawn from the previous row",
     "const char *trow = (const char *)target + ((size_t)b * (N + 1) + a) * V * esz;",
     "const char *trow = (const char *)target + ((size_t)b * (N + 1) + (a == N ? N - 1 : a)) * V * esz;",
     [lambda o: TV.test_enumeration_emitted_token_is_target_distribution(o, 0)]),
    ("inverse CDF off by one", "            y = kk;\n            break;",
     "            y = kk + 1 < V ? kk + 1 : kk;\n            break;",
     [TV.test_chi_square_v64]),
    ("greedy compares with own argmax", "tok[i] == amax[par[i]]", "tok[i] == amax[i]",
     [lambda o: TT.test_greedy_matches_brute_force(o, 0)]),
    ("greedy tie takes the largest index", "depth[i] > depth[best]", "depth[i] >= depth[best]",
     [TT.test_exhaustive_tiny_trees]),
    ("argmax tie takes the last index", "if (x > m) {", "if (x >= m) {",
     [TV.test_row_stats_argmax_ties_take_smallest_index]),
    ("siblings tested against p (no residual update)", "                    c += n;",
     "                    c += 0.0;", [lambda o: TS.test_first_token_follows_target_at_root(3, 1.0)]),
    ("residual normaliser dropped from the sibling test",
     "const double lhs = (double)u_accept[(size_t)b * T + v] * qu[x] * n;",
     "const double lhs = (double)u_accept[(size_t)b * T + v] * qu[x];",
     [lambda o: TS.test_first_token_follows_target_at_root(3, 3.0)]),
    ("residual constant carried from the parent node", "            c = 0.0;\n            int next = -1;",
     "            int next = -1;", [lambda o: TS.test_later_tokens_follow_target_below_the_root()]),
    ("tree's final draw from p after rejections",
     "w[k] = c == 0.0 ? pu[k] : (d > 0.0 ? d : 0.0);", "w[k] = pu[k];",
     [lambda o: TS.test_chain_tree_equals_chain_rule(64, 4, 300, "f32", 1),
      lambda o: TS.test_first_token_follows_target_at_root(1, 1.0)]),
    ("compaction copies from the wrong slot",
     "k_in + base + (size_t)(L + src) * D", "k_in + base + (size_t)(L + d) * D",
     [TT.test_compaction_invariants]),
]


@pytest.mark.parametrize("name,old,new,checks", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, checks):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site not unique: {old!r}"
    mut_c = tmp_path / "mutant.c"
    mut_c.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-shared", "-fPIC",
                           str(mut_c), "-o", str(so), "-lm"])
    real = oracle.lib()
    mutant = ctypes.CDLL(str(so))
    for fn in ("orc_ancestor_mask", "orc_tree_attention", "orc_row_stats", "orc_verify_chain",
               "orc_verify_tree_greedy", "orc_verify_tree_stochastic", "orc_compact_kv"):
        getattr(mutant, fn).argtypes = getattr(real, fn).argtypes
        getattr(mutant, fn).restype = getattr(real, fn).restype
    caught = 0
    try:
        oracle._lib = mutant
        for check in checks:
            try:
                check(oracle)
            except (AssertionError, ValueError):
                caught += 1
    finally:
        oracle._lib = real
    assert caught == len(checks), f"mutant '{name}' survived"
