"""The C-ABI library loads and exports every symbol include/eaglespec.h declares;
host-side argument checks reject bad calls before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest

from eagle_speculative_decoding_step_gb300 import binding as lib
from eagle_speculative_decoding_step_gb300 import build, configs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "eaglespec.h")


@pytest.fixture(scope="module")
def so():
    build.build()
    return lib.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(spec_[a-z_0-9]+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ["spec_fc_fuse", "spec_draft_layer", "spec_lm_head", "spec_lowrank_candidates",
                 "spec_tree_expand", "spec_verify_greedy", "spec_verify_rejection", "spec_workspace_bytes",
                 "spec_get_device_error"]:
        assert want in names


def test_library_exports_every_declared_symbol(so):
    for name in declared_functions():
        assert hasattr(so, name), name
        assert name in lib.EXPORTS, "binding lacks " + name


def test_status_strings(so):
    assert so.spec_status_string(0) == b"ok"
    assert b"workspace" in so.spec_status_string(-8)
    assert so.spec_version() >= 1


def test_workspace_queries(so):
    for name in configs.ORDER:
        w = configs.WORKLOADS[name]
        d = lib.make_desc(w)
        n = lib.spec_workspace_bytes(d, w.rows_max, w.max_ctx)
        assert n > 0 and n % 256 == 0
        assert lib.spec_verify_workspace_bytes(w.B, w.verify_rows, w.V) > 0
    bad = lib.make_desc(configs.WORKLOADS["tiny"])
    bad.n_kv_heads = 3                       # 4 q heads not a multiple of 3
    assert lib.spec_workspace_bytes(bad, 1, 64) == 0
    assert lib.spec_tree_state_bytes(1, 8, 5, 31) > 0


FAKE = 4096    # non-null, never dereferenced: every call below fails its host checks first


def _status(fn, *args):
    return getattr(lib.load(), fn)(*args)


def test_host_checks_reject_before_launch(so):
    w = configs.WORKLOADS["llama8b_chain"]
    d = lib.make_desc(w)
    wt = lib.Weights()
    # NULL arguments
    assert _status("spec_fc_fuse", ctypes.byref(d), ctypes.byref(wt), None, None, 4, None, 0, None) == -1
    # bad row count
    wt.fc = FAKE
    assert _status("spec_fc_fuse", ctypes.byref(d), ctypes.byref(wt), FAKE, FAKE, 0, FAKE, 0, None) == -2
    # workspace too small
    assert _status("spec_fc_fuse", ctypes.byref(d), ctypes.byref(wt), FAKE, FAKE, 4, FAKE, 16, None) == -8
    # misaligned activation
    assert _status("spec_fc_fuse", ctypes.byref(d), ctypes.byref(wt), FAKE + 2, FAKE, 4, FAKE, 1 << 40, None) == -9
    # unsupported window (< 64 keys)
    d2 = lib.make_desc(w)
    d2.window = 10
    assert _status("spec_fc_fuse", ctypes.byref(d2), ctypes.byref(wt), FAKE, FAKE, 4, FAKE, 1 << 40, None) == -2
    # lm head: k out of range
    wt.lm_head = FAKE
    assert _status("spec_lm_head", ctypes.byref(d), ctypes.byref(wt), FAKE, 4, 9, FAKE, 0, FAKE, None, None,
                   FAKE, 1 << 40, None) == -2
    # low-rank head on a model without one
    assert _status("spec_lowrank_candidates", ctypes.byref(d), ctypes.byref(wt), FAKE, 4, 1, None, None, FAKE, None,
                   0, FAKE, 1 << 40, None) == -3
    # verifiers
    assert _status("spec_verify_greedy", 2, 70, 100, FAKE, FAKE, None, 0, FAKE, FAKE, None, None, None, None,
                   FAKE, 1 << 40, None) == -4            # more than 64 rows per request
    assert _status("spec_verify_greedy", 2, 6, 100, FAKE, FAKE, None, 0, FAKE, FAKE, None, None, None, None,
                   FAKE, 8, None) == -8                  # workspace too small
    assert _status("spec_verify_rejection", 2, 0, 100, FAKE, FAKE, FAKE, None, None, 0, 0, FAKE, FAKE, None, FAKE,
                   1 << 40, None) == -2
    # tree capacity
    io = lib.TreeIO(*([FAKE] * 11))
    assert _status("spec_tree_expand", 1, 8, 1, 9, 31, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(io), None) == -4
    assert _status("spec_tree_expand", 1, 4, 1, 3, 64, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(io), None) == -4
    assert _status("spec_tree_expand", 1, 4, 0, 3, 8, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(io), None) == -1
