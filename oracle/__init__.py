"""Plain, slow, fp64 CPU oracle of the dynamic draft-tree hot path.

THIS PACKAGE IS TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it. The product path
(``dynamic_draft_tree_gb300``) never imports it and shares no code with it.

What it restates, and from where (page titles, sections):

* EAGLE-2 ("EAGLE-2 完全拆解：动态草稿树如何让投机解码上下文感知"):
  - §"置信度为什么可以近似接受率": draft confidence c = softmax probability of
    the drafted token.
  - §"value 公式": node value V_i = product of confidences on the root path;
    kept in log form, value(child) = value(parent) + log c.
  - §"扩展阶段": expand the top-k nodes of the newest layer by value; each
    expanded node contributes its top-K vocabulary children.
  - §"重排阶段": rerank all nodes by value, take top-m, ties toward shallower
    nodes, giving a connected subtree; flatten it and build the ancestor-only
    attention mask.
  - §"先把投机解码的账本摆清楚" and §"无损性为什么没有被动态树破坏":
    speculative-sampling acceptance min(1, p/q) with residual
    norm(max(0, p - q)); greedy decoding is deterministic. ``sampled``
    applies the same rule to children drawn from the draft distribution
    without replacement (each sibling against the distribution it was drawn
    from).
* CAST ("Inference-Cost-Aware Dynamic Tree Construction ..."), §关键设计 1-4:
  cost lookup table with the grid quantiser select(c), width pruning by
  marginal utility against C1, depth pruning with the FIFO ratio buffer
  against C2, verify-count selection against C3.
* EAGLE-2, §"一段更贴近实现的流程" (after verification): ``kv`` commits the root's and the accepted
  positions' temporary KV rows to the cache, in path order, and discards the rest.
* Graft ("Draft Less, Retrieve More"), the three-step method description:
  confidence checkpoints c_d = exp(max_j S_{d,j}) against tau_d, retrieval
  x_u = M[x_{F(u)}, r_u] over a template, hybrid flatten to K_max tokens,
  online refresh of M rows with the target's top-k successors.

Readings where the pages are silent or garbled are listed in each module's
docstring. Every function is written for clarity, not speed.

Functions whose result is not fixed by an independent pin say
"parity unpinned" in their docstring: ``graft.retrieve`` (the template shape).
"""


