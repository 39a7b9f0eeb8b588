"""Bounded waits on the GPU, tested without a fault.

Every wait in the attention kernels gives up after a clock-bounded limit,
raises the CTA's abort flag and sets the translation unit's device status
word; the kernel then returns.  ``tpa_wait_probe`` runs that same wait on an
mbarrier: completed first (the wait succeeds) or never arrived at (the wait
runs out after a few milliseconds).  The host must see TPA_ERR_DEVICE_TIMEOUT
exactly once, and the context must stay usable: an attention forward and
backward afterwards still match the oracle.
"""
import time

import numpy as np
import pytest

import oracle
from synth import random_small_sequences
from _pipeline import assert_attn_close, pack_and_upload, random_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tpa():
    import prefix_shared_tree_attention_gb300 as tpa
    tpa.lib()
    tpa.device_check()
    return tpa


def test_completed_wait_reports_ok(tpa):
    tpa.sync_status()
    tpa.wait_probe(10_000_000, arrive=True)
    tpa.sync_status()


def test_wait_that_runs_out_is_reported_once_and_context_stays_usable(tpa):
    tpa.sync_status()
    t0 = time.perf_counter()
    tpa.wait_probe(3_000_000, arrive=False)  # ~3 ms bound
    with pytest.raises(tpa.TpaError) as err:
        tpa.sync_status()
    elapsed = time.perf_counter() - t0
    assert err.value.name == "TPA_ERR_DEVICE_TIMEOUT"
    assert elapsed < 5.0, f"the bounded wait took {elapsed:.2f} s"
    tpa.sync_status()  # reading the status cleared it

    # the context still runs the attention correctly
    rng = np.random.default_rng(91)
    T = 256
    seqs = random_small_sequences(rng, 5, 200, 3, min_len=1)
    pk = oracle.tree_pack(seqs, T)
    tree, dtree, mask = pack_and_upload(tpa, seqs, T)
    (q, k, v, do), (qc, kc, vc, doc) = random_inputs(tree.n_trees, T, 4, 2, 128, 91)
    o, lse = tpa.tree_attn_fwd(dtree, mask, q, k, v)
    dq, dk, dv = tpa.tree_attn_bwd(dtree, mask, q, k, v, o, lse, do)
    tpa.sync_status()
    for b, t in enumerate(pk.trees):
        O, _ = oracle.attn_forward(t, qc[b], kc[b], vc[b], t_pad=T)
        dQ, dK, dV = oracle.attn_backward(t, qc[b], kc[b], vc[b], doc[b], t_pad=T)
        assert_attn_close(o[b], O, f"O tree {b}")
        assert_attn_close(dq[b], dQ, f"dQ tree {b}")
        assert_attn_close(dk[b], dK, f"dK tree {b}")
        assert_attn_close(dv[b], dV, f"dV tree {b}")


def test_probe_rejects_bad_limits(tpa):
    for bad in (0, 20_000_000_000):
        with pytest.raises(tpa.TpaError) as err:
            tpa.wait_probe(bad, arrive=True)
        assert err.value.name == "TPA_ERR_INVALID_ARG"
