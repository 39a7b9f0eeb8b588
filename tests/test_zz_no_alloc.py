"""The workspace-free backward entry point (GPU).

tpa_tree_attn_bwd_noalloc serves callers that cannot give the library a
device workspace (runtimes whose memory pool owns the whole device, C callers
without an allocator): it draws its scratch from a fixed array inside the
library. These tests call it through the C ABI and compare it with the
regular tpa_tree_attn_bwd on the same inputs, twice in a row with different
inputs (the shared array keeps the previous call's contents, which must not
leak into the next result), for fp32 and bf16 gradients, and check that a
problem too large for the array is refused. This file is collected last on
purpose.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from synth import random_small_sequences
from _pipeline import assert_attn_close, pack_and_upload, random_inputs

pytestmark = pytest.mark.gpu

GRAD = {torch.float32: 0, torch.bfloat16: 1}


@pytest.fixture(scope="module")
def tpa():
    import prefix_shared_tree_attention_gb300 as tpa
    tpa.lib()
    tpa.device_check()
    return tpa


def _noalloc(tpa, dtree, mask, q, k, v, o, lse, do, grad_dtype):
    hq, hkv, d = q.shape[2], k.shape[2], q.shape[3]
    dq, dk, dv = (torch.empty(x.shape, dtype=grad_dtype, device=x.device) for x in (q, k, v))
    rc = tpa.lib().tpa_tree_attn_bwd_noalloc(
        C.byref(dtree.view), C.byref(mask.view), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
        lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), hq, hkv, d, 0.0,
        GRAD[grad_dtype], torch.cuda.current_stream().cuda_stream)
    assert rc == 0, tpa.lib().tpa_status_string(rc)
    return dq, dk, dv


@pytest.mark.parametrize("grad_dtype", [torch.float32, torch.bfloat16])
def test_noalloc_matches_workspace_entry_point(tpa, grad_dtype):
    rng = np.random.default_rng(33)
    seqs = random_small_sequences(rng, 10, 300, 3, min_len=1)
    T, hq, hkv, d = 512, 4, 2, 128
    tree, dtree, mask = pack_and_upload(tpa, seqs, T)
    for call, seed in enumerate((101, 202)):       # two calls in a row, different inputs
        (q, k, v, do), _ = random_inputs(tree.n_trees, T, hq, hkv, d, seed)
        o, lse = tpa.tree_attn_fwd(dtree, mask, q, k, v)
        ref = tpa.tree_attn_bwd(dtree, mask, q, k, v, o, lse, do, grad_dtype=grad_dtype)
        got = _noalloc(tpa, dtree, mask, q, k, v, o, lse, do, grad_dtype)
        tpa.sync_status()
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            assert g.dtype == grad_dtype
            assert_attn_close(g.float(), r.float(), f"call {call} {name}")
        # no key column of this tree is long enough to be split into items that
        # add into their rows, so the two entry points agree bit for bit
        assert all(torch.equal(g, r) for g, r in zip(got, ref))


def test_noalloc_refuses_oversized_problem(tpa):
    # 1 tree x 65536 positions x 128 query heads needs 32 MiB of scratch (D alone)
    tree, dtree, mask = pack_and_upload(tpa, [[1, 2, 3]], 65536)
    buf = torch.zeros(1024, dtype=torch.float32, device="cuda")
    p = buf.data_ptr()
    rc = tpa.lib().tpa_tree_attn_bwd_noalloc(C.byref(dtree.view), C.byref(mask.view), p, p, p, p, p, p, p, p, p,
                                             128, 128, 128, 0.0, 0, None)
    assert tpa.lib().tpa_status_string(rc) == b"TPA_ERR_BUFFER_TOO_SMALL"
    tpa.sync_status()
