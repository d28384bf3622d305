"""GPU parity of spec_decode_metadata: the page's printed example and random ragged batches."""
import json
import os

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_step_gb300 import binding as lib
from oracle import metadata

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _run(cu, nd, ids):
    R = len(cu)
    S = int(np.sum(nd))
    i32 = dict(dtype=torch.int32, device="cuda")
    o = [torch.full((R,), -9, **i32), torch.full((S + R,), -9, **i32), torch.full((max(S, 1),), -9, **i32),
         torch.full((R,), -9, **i32), torch.full((max(S, 1),), -9, **i32)]
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    d = lambda a: torch.from_numpy(np.asarray(a, dtype=np.int32)).cuda()  # noqa: E731
    lib.spec_decode_metadata(R, d(cu), d(nd), o[0], o[1], o[2], o[3], input_ids=d(ids), draft_token_ids=o[4], ws=ws)
    torch.cuda.synchronize()
    assert lib.spec_get_device_error(ws) == 0
    return [x.cpu().numpy() for x in o], S


def test_printed_example():
    g = json.load(open(os.path.join(GOLDEN, "spec_decode_metadata.json")))
    ids = np.arange(209) + 7
    (cu_nd, li, ti, bi, di), S = _run(g["cu_num_scheduled_tokens"], g["num_draft_tokens"], ids)
    assert cu_nd.tolist() == g["cu_num_draft_tokens"]
    assert li.tolist() == g["logits_indices"]
    assert ti[:S].tolist() == g["target_logits_indices"]
    assert bi.tolist() == g["bonus_logits_indices"]


@pytest.mark.parametrize("R", [1, 37, 1024, 3000])
def test_random_ragged(R):
    g = np.random.default_rng(R)
    nd = g.integers(0, 8, size=R)
    sched = nd + 1 + g.integers(0, 50, size=R)
    cu = np.cumsum(sched)
    ids = g.integers(0, 100000, size=int(cu[-1]))
    ref = metadata.spec_decode_metadata(cu, nd, ids)
    (cu_nd, li, ti, bi, di), S = _run(cu, nd, ids)
    np.testing.assert_array_equal(cu_nd, ref["cu_num_draft_tokens"])
    np.testing.assert_array_equal(li, ref["logits_indices"])
    np.testing.assert_array_equal(ti[:S], ref["target_logits_indices"])
    np.testing.assert_array_equal(bi, ref["bonus_logits_indices"])
    np.testing.assert_array_equal(di[:S], ref["draft_token_ids"])
