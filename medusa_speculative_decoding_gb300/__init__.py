"""GB300 (sm_103a) hot path of the Medusa decode step.

The computation lives in libmedusa_gb300.so (hand-written CUDA kernels behind
the C ABI of include/medusa.h); this package is its thin Python binding:

  heads_topk          Medusa heads h + SiLU(W1 h + b1) -> W2, per-head top-k
  heads_topk_static   the same without a workspace (library-owned scratch)
  sparse_tree_paths   the most accurate rank tuples (host)
  tree_layout         node table, ancestor mask and paths of a tree (host)
  build_tree          candidate tokens of the tree nodes
  tree_attention      ancestor-masked attention of all candidates in one pass
  verify_accept_tree  greedy / typical acceptance, longest accepted branch
  verify_accept_tree_sample  typical acceptance, next token drawn from the
                      best node's softmax
  verify_project_tree the same as verify_accept_tree from the tree's hidden states: lm_head projection
                      on the tensor cores, reduced without writing the logits
  verify_accept_chain speculative-sampling acceptance with k + 1 tokens
  kv_compact          keep the accepted branch's KV rows and hidden state
  device_status       raises if a bounded device wait gave up (MEDUSA_ERR_TIMEOUT)
  set_wait_limit      test hook: the tensor-core kernels' wait limit
"""
from ._native import MedusaError, lib  # noqa: F401
from .api import (build_tree, device_status, heads_topk, heads_topk_static, heads_topk_workspace,  # noqa: F401
                  kv_compact, set_wait_limit,
                  sparse_tree_paths, tree_attention, tree_attention_workspace, tree_layout,
                  verify_accept_chain, verify_accept_tree, verify_accept_workspace,
                  verify_accept_tree_sample, verify_chain_workspace, verify_project_tree,
                  verify_project_workspace, verify_sample_workspace)
