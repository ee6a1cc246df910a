"""The pins catch plausible mistakes: each case plants one mistake in a copy of
the oracle's C source, builds it, and checks that a named pin fails."""
import os
import subprocess
import tempfile

import pytest

import oracle
from tests import test_oracle_attention as TA
from tests import test_oracle_cache as TC
from tests import test_oracle_sparse as TS

SRC = os.path.join(os.path.dirname(oracle.__file__), "pkv_oracle.c")

MUTANTS = [
    ("gqa head map h % Hkv", "int kvh = h / g;", "int kvh = h % J->num_kv_heads;",
     lambda: TA.test_oracle_matches_sdpa(*TA.CASES[1])),
    ("verify mask off by one", "int vis = ctx - J->q_len + j + 1;", "int vis = ctx - J->q_len + j;",
     lambda: TA.test_oracle_matches_sdpa(*TA.CASES[4])),
    ("scale dropped", "x[t - t0] = J->scale * dot;", "x[t - t0] = dot;",
     lambda: TA.test_oracle_matches_sdpa(*TA.CASES[0])),
    ("block offset t/bs", "size_t row = ((size_t)pb * bs + (size_t)(t % bs)) * H + kvh;\n    if (J->cache_kind == OC_K8V4) {\n        size_t meta",
     "size_t row = ((size_t)pb * bs + (size_t)(t / bs % bs)) * H + kvh;\n    if (J->cache_kind == OC_K8V4) {\n        size_t meta",
     lambda: TA.test_oracle_matches_sdpa(*TA.CASES[0])),
    ("nibble order swapped", "int c = (d % 2 == 0) ? (byte & 0x0f) : (byte >> 4);",
     "int c = (d % 2 == 0) ? (byte >> 4) : (byte & 0x0f);",
     TC.test_k8v4_attention_matches_sdpa_over_independent_dequant),
    ("ties away from zero", "clampf(rintf(kv[d] / s), -127.0f, 127.0f)",
     "clampf(roundf(kv[d] / s), -127.0f, 127.0f)", TC.test_quantiser_worked_example_ties_to_even),
    ("lse weight drops l_p", "double w = l[p] * exp(m[p] - M);", "double w = exp(m[p] - M);",
     lambda: TA.test_split_partials_and_reduce_equal_single_pass(32)),
    ("softmax max not subtracted in weights", "double w = exp(x[t - t0] - m);", "double w = exp(x[t - t0]);",
     lambda: TA.test_split_partials_and_reduce_equal_single_pass(16)),
    ("dequant gather drops the V zero", "double vv = (double)c * sv + zv;", "double vv = (double)c * sv;",
     lambda: TC.test_dequant_gather_matches_numpy_torch_rounding("bf16")),
    ("dequant gather reads the neighbour token's scales",
     "size_t meta = ((size_t)pb * H + (size_t)h) * block_size + (size_t)off;",
     "size_t meta = ((size_t)pb * H + (size_t)h) * block_size + (size_t)(off ^ 1);",
     lambda: TC.test_dequant_gather_matches_numpy_torch_rounding("f16")),
    ("window one token short", "if (J->window > 0 && ctx > J->window) lo = ctx - J->window;",
     "if (J->window > 0 && ctx > J->window) lo = ctx - J->window + 1;",
     lambda: TA.test_window_matches_sdpa_over_the_last_tokens(*TA.WINDOW_CASES[0])),
    ("window per draft row", "if (J->window > 0 && ctx > J->window) lo = ctx - J->window;",
     "if (J->window > 0 && vis > J->window) lo = vis - J->window;",
     lambda: TA.test_window_matches_sdpa_over_the_last_tokens(*TA.WINDOW_CASES[2])),
    ("sparse page token offset", "int t = p * bs + o;", "int t = p * bs + o + 1;",
     lambda: TS.test_sparse_matches_sdpa_over_listed_pages(*TS.CASES[0])),
    ("sparse repeated page kept", "if (p < 0 || p >= npages || p <= last) continue;",
     "if (p < 0 || p >= npages || p < last) continue;", TS.test_bad_entries_are_skipped),
]


@pytest.mark.parametrize("name,old,new,pin", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pin_catches_planted_mistake(name, old, new, pin):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "mut.c")
        so = os.path.join(d, "mut.so")
        open(c, "w").write(src.replace(old, new))
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-pthread", "-o", so, c, "-lm"])
        prev = oracle.use_library(so)
        try:
            with pytest.raises(AssertionError):
                pin()
        finally:
            oracle.restore_library(prev)
