"""prefix_shared_tree_attention_gb300 — tree training's hot path on GB300.

A thin Python binding over libtpa (include/tpa.h): argument marshalling and
torch-owned device memory only; every step runs in the library (the C++
packer on the host, CUDA kernels for sm_103a on the device). Functions keep
the C names without the ``tpa_`` prefix:

    tree = tree_pack(seqs, max_tokens_per_mb)           # host trie packer
    tree = tree_pack_padded(input_ids, attention_mask, max_tokens_per_mb)  # from a padded batch
    dtree = tree.upload(device)                         # metadata -> HBM
    mask = block_classify(dtree)                        # 128x128 tile classes + CSR
    dense = dense_mask(dtree)                           # [B, T, T] ancestor mask (Megatron-style)
    o, lse = tree_attn_fwd(dtree, mask, q, k, v)
    dq, dk, dv = tree_attn_bwd(dtree, mask, q, k, v, o, lse, dout)
    pos_logp, pos_ent, seq_logp, seq_ent = tree_logprobs_entropy(dtree, logits)
    pos_logp, pos_ent, seq_logp, seq_ent = lm_head_logprobs_entropy(dtree, hidden, weight)  # no logits tensor
    group_of, n_groups, algo = balance(weights, capacity, min_groups, 1, "kk")  # trees -> ranks
    metrics = packing_metrics(weights, group_of, n_groups, capacity)
"""
from ._abi import BLOCK_SIZE, LOGITS_COMPACT, LOGITS_PADDED, STATUS, TpaError, lib  # noqa: F401
from .api import (  # noqa: F401
    BlockMask, DeviceTree, Tree, balance, block_classify, dense_mask, device_check, extract_sequences,
    lm_head_logprobs_entropy, lm_head_workspace_bytes, packing_metrics, sync_status, tree_attn_bwd,
    tree_pack_padded,
    tree_attn_bwd_workspace_bytes, tree_attn_fwd, tree_logprobs_entropy, tree_pack, wait_probe,
)
