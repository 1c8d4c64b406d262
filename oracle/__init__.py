"""CPU fp64 oracle for context-parallel causal attention — TEST INFRASTRUCTURE.

This package is the checker, not the product. Only the test suite, the smoke
check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may
import it. It shares no code with the CUDA path: it never imports the
``context_blockwise_causal_gb300`` package and that package never imports it.

Contents
--------
``attention``        plain softmax attention (and its gradients) over the
                     uncut, natural-order sequence, straight from the
                     definition; fp64 throughout.
``context_parallel`` the zigzag split into 2*cp half-chunks, the per-rank
                     block steps with their masks, and the log-sum-exp
                     correction/merge of partial results — an independent
                     second route to the same numbers, used to pin the first.

Sources (web pages; cited by title and section):
  [MLM-CP]   "大模型面试宝典 · Megatron-LM 篇", question 3 "Context Parallel 篇",
             sub-questions 3.1–3.5.
  [Practice] "超大规模集群下大语言模型训练实操指南", section "CP 与其他技术结合".
  [M019]     "Megatron 面试题（一）：模型抽象与训练数据流", item M019
             (two-stage global-max / global-sum log-sum-exp).
  [M014]     same page, item M014 (GQA head grouping).

Every function is pinned by a CPU test in tests/test_oracle.py (hand-computed
values, closed forms, a library attention routine, finite differences and the
equality of the two routes); none is "parity unpinned".
"""
from .attention import attention_forward, attention_backward, softmax_scale  # noqa: F401
from .context_parallel import (  # noqa: F401
    zigzag_chunks,
    zigzag_global_index,
    cp_step_plan,
    block_attention,
    lse_merge,
    cp_step_partials,
    cp_attention_forward,
)
from .rope import rope_angles, rope_apply, natural_positions, rank_local_positions  # noqa: F401
from .varlen import varlen_attention_forward, varlen_attention_backward  # noqa: F401
