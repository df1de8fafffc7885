"""The automatic kernel choice against the measured variant table.

``profiles/variant_sweep.json`` (written on a GB300 by ``bench.py --sweep``)
holds, for every BF16 configuration (M, N, K) in both weight forms, the
per-call time of every variant, and for every INT4 / MXFP8 / NVFP4
configuration the time of every weight-format kernel.  The choice the library
makes for each of them (``swiglu_select_variant``,
``swiglu_select_weight_kernel``, host-only, on the table's SM count) must be
within 5 % of the best measured one.  The page's method rests on such a
choice: two kernels, each best in its own regime (page "Riepilogo Tecnico ...
Inferenza Efficiente di LLM", sections "Metodologia" and "Risultati").
"""
import json
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TABLE = os.path.join(ROOT, "profiles", "variant_sweep.json")

# The BF16 configurations the benchmark and the parity tests use: (N, K, Ms)
BF16_CONFIGS = [(4864, 896, (64, 128, 512, 2048, 8192)), (18944, 3584, (256, 1024, 2048, 4096)),
                (29568, 8192, (2048, 8192, 16384))]


@pytest.fixture(scope="module")
def table():
    with open(TABLE) as f:
        return json.load(f)


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import swiglu_gemm_transformer_gb300 as sg
    return sg


def test_table_covers_every_configuration(table):
    assert table["sm_count"] == 152          # GB300; the host-only choice assumes it too
    have = {(e["N"], e["K"], e["M"], e["form"]) for e in table["entries"] if e["kind"] == "bf16"}
    for N, K, Ms in BF16_CONFIGS:
        for M in Ms:
            for form in ("separate", "interleaved"):
                assert (N, K, M, form) in have, (N, K, M, form)
    assert any(e["kind"] == "w4" for e in table["entries"])
    assert any(e["kind"] == "mx" for e in table["entries"])


def test_choice_within_5_percent_of_best(table, lib):
    sg = lib
    slow = []
    for e in table["entries"]:
        us = e["us"]
        best = min(us, key=us.get)
        if e["kind"] == "bf16":
            chosen = sg.variant_name(sg.swiglu_select_variant(e["M"], e["N"], e["K"],
                                                              e["form"] == "interleaved"))
        else:
            chosen = sg.WEIGHT_KERNELS[sg.swiglu_select_weight_kernel(e["M"], e["N"])]
        if us[chosen] > 1.05 * us[best]:
            slow.append((e["workload"], e["form"], e["M"], chosen, us[chosen], best, us[best]))
    assert not slow, slow
