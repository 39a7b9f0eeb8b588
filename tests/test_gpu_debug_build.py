"""The TPA_DEBUG build, libtpa_debug.so (GPU).

Its kernels check every metadata index they read from a tree view before
using it as an address.  On a well-formed tree it gives the release
library's results bit for bit and reports no error.  On a view whose device
blob was edited (a child position that does not follow its parent, a
sequence position beyond the tree) it skips the bad accesses and reports
TPA_ERR_INVALID_ARG through tpa_sync_status.  The edited values still lie
inside the metadata arrays, so even unchecked code would not have read
outside them.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from synth import random_small_sequences
from _pipeline import pack_and_upload, random_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    import prefix_shared_tree_attention_gb300 as tpa
    from prefix_shared_tree_attention_gb300._abi import debug_lib
    tpa.lib()
    tpa.device_check()
    return tpa, debug_lib()


def _logprobs(L, view, logits, outs):
    return L.tpa_tree_logprobs_entropy(C.byref(view), logits.data_ptr(), logits.stride(0), 0, logits.shape[1],
                                       *[o.data_ptr() for o in outs], torch.cuda.current_stream().cuda_stream)


def test_debug_build_matches_release(libs):
    tpa, D = libs
    rng = np.random.default_rng(61)
    seqs = random_small_sequences(rng, 9, 200, 3, min_len=2)
    T = 256
    tree, dtree, mask = pack_and_upload(tpa, seqs, T)
    B, N, rows = tree.n_trees, tree.info.total_seq_tokens, tree.info.total_tree_tokens
    logits = (2 * torch.randn((rows, 512), generator=torch.Generator().manual_seed(6))).to(torch.bfloat16).cuda()
    rel = [torch.empty(s, device="cuda") for s in ((B, T), (B, T), (N,), (N,))]
    dbg = [torch.empty(s, device="cuda") for s in ((B, T), (B, T), (N,), (N,))]
    assert _logprobs(tpa.lib(), dtree.view, logits, rel) == 0
    assert _logprobs(D, dtree.view, logits, dbg) == 0
    # the block mask and the forward through the debug library too
    dmask = tpa.BlockMask(B, T, "cuda")
    assert D.tpa_block_classify(C.byref(dtree.view), C.byref(dmask.view), None) == 0
    (q, k, v, _), _ = random_inputs(B, T, 4, 2, 64, 5)
    o_rel, lse_rel = tpa.tree_attn_fwd(dtree, mask, q, k, v)
    o_dbg, lse_dbg = torch.empty_like(o_rel), torch.empty_like(lse_rel)
    assert D.tpa_tree_attn_fwd(C.byref(dtree.view), C.byref(dmask.view), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                               o_dbg.data_ptr(), lse_dbg.data_ptr(), 4, 2, 64, 0.0, None) == 0
    assert D.tpa_sync_status(None) == 0 and tpa.lib().tpa_sync_status(None) == 0
    assert all(torch.equal(a, b) for a, b in zip(rel, dbg))
    assert torch.equal(o_rel, o_dbg) and torch.equal(lse_rel, lse_dbg)
    assert all(torch.equal(dmask.arrays()[k_], mask.arrays()[k_]) for k_ in ("cls", "q_ptr", "q_idx", "k_ptr"))


def test_debug_build_reports_bad_view_indices(libs):
    tpa, D = libs
    seqs = [[1, 2, 3, 4, 5], [1, 2, 7, 8], [1, 9]]
    T = 256
    tree, dtree, mask = pack_and_upload(tpa, seqs, T)
    B, N, rows = tree.n_trees, tree.info.total_seq_tokens, tree.info.total_tree_tokens
    arr = tree.arrays()
    n0 = int(arr["n_tokens"][0])
    base = dtree.buf.data_ptr()

    def poke(ptr_field: int, index: int, value: int):
        off = ptr_field - base + 4 * index
        dtree.buf[off:off + 4].view(torch.int32).fill_(value)

    # the root's first child entry now names position 0 (not after its parent),
    # and a token of the first sequence sits at a padding position (< T)
    c_first = int(arr["child_off"][0][0])
    poke(dtree.view.child_pos, c_first, 0)
    poke(dtree.view.seq_pos, 2, n0 + 3)
    logits = torch.randn((rows, 64)).to(torch.bfloat16).cuda()
    outs = [torch.zeros(s, device="cuda") for s in ((B, T), (B, T), (N,), (N,))]
    assert _logprobs(D, dtree.view, logits, outs) == 0
    assert D.tpa_sync_status(None) == -1       # TPA_ERR_INVALID_ARG, read once ...
    assert D.tpa_sync_status(None) == 0        # ... and cleared
