"""GPU parity of spec_tree_expand against the oracle (exact: same fp32 inputs)."""
import numpy as np
import pytest
import torch

from eagle_speculative_decoding_step_gb300 import binding as lib
from oracle import tree
from gpu_helpers import dev

pytestmark = pytest.mark.gpu


def _topk_inputs(g, rows, k, V, ties=False):
    ids = np.stack([g.choice(V, size=k, replace=False) for _ in range(rows)]).astype(np.int32)
    lp = -np.sort(g.exponential(1.0, size=(rows, k)).astype(np.float32), axis=1)
    if ties:
        lp[:, 1] = lp[:, 0]                        # equal scores inside a row
        lp[::2] = lp[0]                            # equal rows
    return ids, lp.astype(np.float32)


@pytest.mark.parametrize("B,k,D,N,ties", [(1, 8, 5, 31, False), (3, 4, 4, 20, True), (2, 1, 6, 6, False),
                                          (2, 3, 1, 3, False), (1, 16, 2, 63, True)])
def test_tree_expand_parity(B, k, D, N, ties):
    g = np.random.default_rng(B * 100 + k * 10 + D)
    V = 50000
    ctx = np.array([100 + 7 * b for b in range(B)], dtype=np.int32)
    root = g.integers(0, V, size=B).astype(np.int32)
    st = tree.tree_init(B, k, D, N, root, ctx)
    i32 = dict(dtype=torch.int32, device="cuda")
    f = [torch.zeros(B * k, **i32) for _ in range(3)]
    fmask = torch.zeros(B * k, dtype=torch.int64, device="cuda")
    fsrc = torch.zeros(B * k, **i32)
    t = [torch.zeros(B, N + 1, **i32) for _ in range(4)]
    tscore = torch.zeros(B, N + 1, dtype=torch.float32, device="cuda")
    tmask = torch.zeros(B, N + 1, dtype=torch.int64, device="cuda")
    io = lib.make_tree_io(f[0], f[1], f[2], fmask, fsrc, t[0], t[1], t[2], t[3], tscore, tmask)
    state = torch.zeros(lib.spec_tree_state_bytes(B, k, D, N), dtype=torch.uint8, device="cuda")
    dctx, droot = dev(ctx), dev(root)
    for d in range(1, D + 1):
        rows = B if d == 1 else B * k
        ids, lp = _topk_inputs(g, rows, k, V, ties)
        ref = tree.tree_expand(st, d, ids, lp)
        dids, dlp = dev(ids), dev(lp)
        lib.spec_tree_expand(B, k, d, D, N, dctx, droot, dids, dlp, state, io)
        torch.cuda.synchronize()
        if d < D:
            np.testing.assert_array_equal(f[0].cpu().numpy(), ref["tok"])
            np.testing.assert_array_equal(f[1].cpu().numpy(), ref["pos"])
            np.testing.assert_array_equal(f[2].cpu().numpy(), ref["kv_idx"])
            np.testing.assert_array_equal(fmask.cpu().numpy().astype(np.uint64),
                                          np.array(ref["mask"], dtype=np.uint64))
            np.testing.assert_array_equal(fsrc.cpu().numpy(), ref["hid_src"])
        else:
            np.testing.assert_array_equal(t[0].cpu().numpy(), ref["tok"])
            np.testing.assert_array_equal(t[1].cpu().numpy(), ref["parent"])
            np.testing.assert_array_equal(t[2].cpu().numpy(), ref["depth"])
            np.testing.assert_array_equal(t[3].cpu().numpy(), ref["pos"])
            np.testing.assert_array_equal(tscore.cpu().numpy(), ref["score"])
            np.testing.assert_array_equal(tmask.cpu().numpy().astype(np.uint64),
                                          np.array(ref["mask"], dtype=np.uint64))


def test_tree_expand_rejects_oversized_tree():
    io = lib.TreeIO()
    with pytest.raises(lib.SpecError):
        lib.spec_tree_expand(1, 8, 1, 9, 31, 0, 0, 0, 0, 0, io)        # 1 + 8*8 > 64 draft entries
    with pytest.raises(lib.SpecError):
        lib.spec_tree_expand(1, 4, 1, 3, 64, 0, 0, 0, 0, 0, io)        # total + 1 > 64
