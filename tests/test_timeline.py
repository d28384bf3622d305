"""Host logic of the per-kernel timeline (eagle_speculative_decoding_step_gb300/timeline.py)
on a synthetic block log: launches are rebuilt from blocks, steps end at a verifier,
and each launch is charged the wall time it adds along the sequence."""
import numpy as np

from eagle_speculative_decoding_step_gb300 import timeline as tl


def _log(blocks):
    """blocks: (kernel id, grid, block index, start ns, end ns) in recording order."""
    a = np.zeros(tl.LOG_WORDS, dtype=np.uint64)
    a[0] = len(blocks)
    for i, (k, g, b, s, e) in enumerate(blocks):
        a[8 + 4 * i:8 + 4 * i + 4] = [s, 0, e, k | (g << 8) | (b << 32)]
    return a.view(np.int64)


GEMM, NORM, GREEDY = 1, 9, 18


def test_launches_group_blocks_by_grid_in_start_order():
    blocks = [(GEMM, 2, 0, 100, 500), (GEMM, 2, 1, 110, 520),          # launch 1
              (NORM, 1, 0, 400, 700),                                    # overlaps (early launch)
              (GEMM, 2, 1, 800, 1200), (GEMM, 2, 0, 790, 1100)]          # launch 2, blocks out of order
    ls = tl.launches(_log(blocks))
    assert [(l["name"].split()[0], l["start"], l["end"], l["blocks"]) for l in ls] == [
        ("tc_kernel", 100, 520, 2), ("resnorm_kernel", 400, 700, 1), ("tc_kernel", 790, 1200, 2)]
    # tail: last block end minus the median block end
    assert [l["tail"] for l in ls] == [10, 0, 50]


def test_attribution_splits_the_step_span_along_the_sequence():
    step = [{"name": "a", "start": 0, "end": 100}, {"name": "b", "start": 50, "end": 130},
            {"name": "a", "start": 140, "end": 200}, {"name": "c", "start": 150, "end": 190}]
    per, span = tl.attribute(step)
    assert span == 200
    assert per["a"]["charged_ns"] == 100 + 60 + 0 and per["a"]["launches"] == 2
    assert per["b"]["charged_ns"] == 30
    assert per["c"]["charged_ns"] == 0          # finished inside a's second launch
    # the charged times add up to the span minus the idle gap 130..140
    assert sum(d["charged_ns"] for d in per.values()) == span - 10


def test_last_step_is_between_the_last_two_verifiers():
    ls = [{"name": n, "start": i, "end": i + 1} for i, n in enumerate(
        ["x", "verify_greedy_kernel", "y", "z", "verify_greedy_kernel", "w", "verify_greedy_kernel"])]
    assert [l["name"] for l in tl.last_step(ls)] == ["w", "verify_greedy_kernel"]
    md = tl.markdown(tl.last_step(ls))
    assert "| `w` | 1 |" in md and "2 launches" in md


def test_names_cover_the_kernel_ids_of_the_instrumented_build():
    import os
    import re
    src = open(os.path.join(os.path.dirname(tl.__file__), "csrc", "common.cuh")).read()
    body = re.search(r"enum TLKernel : unsigned \{([^}]*)\}", src).group(1)
    ids = [x.strip().split("=")[0].strip() for x in body.split(",") if x.strip()]
    assert len(ids) == len(tl.NAMES) - 1
    # the enum's order matches the names (kTLTc -> tc_kernel, ..., kTLGather -> gather_rows_kernel)
    assert ids[0] == "kTLTc" and tl.NAMES[1].startswith("tc_kernel")
    assert ids[-1] == "kTLGather" and tl.NAMES[-1] == "gather_rows_kernel"
    assert ids[ids.index("kTLRejection")] and tl.NAMES[ids.index("kTLRejection") + 1] == "verify_rejection_kernel"
