"""CPU oracle for prefix-shared tree attention — TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct restatement of what the tree-training
method computes, written from the AReaL "树训练" (tree training) page:

* ``pack``      — trie construction by first-fit-decreasing insertion,
                  linear-chain compression and the flattened preorder layout
                  (§树构建过程 steps 2-3, §数据结构 ``TrieNode``), plus
                  ``tree_token_ratio`` (§指标和监控).
* ``mask``      — the dense ancestor-or-self mask ("a token only attends to
                  its ancestors", §树构建过程 diagram) built by walking parent
                  links, and the 128x128 block classes derived from it by
                  counting (§注意力机制, BLOCK_SIZE 128).
* ``attention`` — fp64 masked softmax attention forward and its analytic
                  backward, computed node by node over each node's root path.
* ``logprobs``  — fp64 per-sequence log-probabilities and entropies gathered
                  from the packed tree rows (§对数概率计算).
* ``lm_head``   — fp64 logits rows from hidden states and the LM-head
                  weight, for the fused LM-head log-prob path.
* ``extract``   — step 1 of tree building: real tokens of padded rows from
                  ``input_ids`` and ``attention_mask``.
* ``balance``   — FFD and KK allocation of weighted items (trees or
                  sequences) to micro-batches / ranks and the packing metrics,
                  from the blog post "AReaL 序列打包算法 FFD 与 KK".

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package. It shares no code with the CUDA library and
never imports it; the product path never calls it.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against facts fixed independently of this code (the page's worked example,
closed forms, brute force over tiny inputs, and reductions to library causal
attention / textbook formulas). The one reading that the pages do not pin is
first-fit (creation order) versus lightest-fit tree choice; see ``pack``.
"""
from .pack import OraclePacking, OracleTree, tree_pack, PackError  # noqa: F401
from .mask import dense_mask, block_classes, block_csr  # noqa: F401
from .attention import attn_forward, attn_backward, attn_rows  # noqa: F401
from .logprobs import sequence_logprobs_entropy, position_logprobs_entropy  # noqa: F401
from .balance import ffd_allocate, kk_allocate, packing_metrics, BalanceError  # noqa: F401
from .extract import extract_sequences  # noqa: F401
from .lm_head import LazyLogits  # noqa: F401
