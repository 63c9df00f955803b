"""One draft-tree round as a sequence of libdt calls (orchestration only, no arithmetic).

Call order (EAGLE-2 page §"一段更贴近实现的流程"; CAST page §关键设计 2-4; Graft page
steps (1)-(3)):

  reset -> [frontier -> draft rows -> expand -> prune]* -> (verify count) -> rerank
  -> (retrieve) -> meta -> target rows -> verify -> (M refresh)

By default a layer's expansion, its pruning and the next frontier are one call
(dt_expand_prune_select, two kernels), and CAST's verify count and rerank are one call; with
``fused=False`` every step is its own call. Graft's root-anchored retrieval is issued on a second
stream right after the reset (it needs the root tokens and M only) and joined before the tree is
flattened, so it runs beside the draft layers; a tail-anchored one follows the rerank. A block
drafter (Graft with ``block``) builds all draft layers with one dt_block_expand call.

The draft and target model forwards are outside the library: ``draft_rows(d,
frontier_token)`` must return the logits tensor [B][F][V] of layer d (row f =
the draft row of frontier slot f), or for a block drafter, called once with d = 0,
the block's rows [B][L][V]; ``target_rows(meta)`` the tensor
[B][P][V] (row i = the target's next-token row after position i). Every call
is asynchronous on the current stream; no host synchronisation happens inside
a round, so a round can be captured in a CUDA graph.
"""
import torch

from . import (Handle, Meta, Template, make_prune_params, make_prune_out, dt_tree_reset, dt_select_frontier,
               dt_expand_layer, dt_expand_prune_select, dt_cast_prune, dt_cast_prune_select, dt_cast_verify_rerank, dt_rerank, dt_graft_retrieve, dt_build_tree_meta, dt_verify, dt_verify_rows,
               dt_verify_accept, dt_adj_update, dt_block_expand, dt_expand_layer_sampled, dt_verify_sampled,
               DT_GREEDY, DT_SAMPLE, DT_VERIFY_PACKED,
               DT_POLICY_CAST_WIDTH_DEPTH, DT_POLICY_CAST_VERIFY, DT_POLICY_GRAFT_CHECKPOINT, DT_POLICY_NONE,
               DT_ANCHOR_ROOT, DT_ANCHOR_TAIL)


class RoundRunner:
    """Device buffers and call sequence of one round for a policy ('eagle' | 'cast' | 'graft')."""

    def __init__(self, policy, B, V, K, k, D, P, D_path, m, dtype, T=0, cast=None, cast_tables=None,
                 graft=None, template=None, flags=0, device="cuda", fused=True, packed=False, block=False,
                 draw=False):
        """``fused``: each layer's expansion, pruning and next frontier as one call
        (dt_expand_prune_select), and CAST's verify count + rerank as one (dt_cast_verify_rerank),
        instead of the separate calls. ``packed``: the target rows are padding-free
        (DT_VERIFY_PACKED): ``target_rows`` returns them at meta.row_off[b] + i. ``block`` (Graft):
        the D draft layers come from a block drafter's rows in one dt_block_expand call. ``draw``
        (EAGLE-2 with T = 1): sampled drafts, the children drawn from the draft rows
        (dt_expand_layer_sampled), every drawn node verified (dt_verify_sampled); ``draft_rows`` must
        then return views of one [D][B][k][V] buffer, layer d at index d - 1, which is handed to the
        verify as ``self.draft_rows``."""
        self.fused = fused
        self.packed = packed
        self.block = block
        self.draw = draw
        self.draft_rows = None
        self.policy, self.B, self.V, self.K, self.k, self.D = policy, B, V, K, k, D
        self.P, self.D_path, self.T = P, D_path, T
        self.h = Handle(B, V, K, k, D, P, dtype, flags)
        i32 = dict(dtype=torch.int32, device=device)
        self.frontier_token = torch.full((B, k), -1, **i32)
        per_req = policy == "cast" and bool((cast or {}).get("per_request", False))
        self.width = torch.full((B if per_req else 1,), k, **i32)
        self.stop = torch.zeros((B,), **i32)
        self.stage = torch.full((B,), -1, **i32)
        self.m_dev = torch.full((B if policy == "graft" or per_req else 1,), m, **i32)
        self.m_cap = m
        self.selected = torch.empty((B, m), **i32)
        self.meta = Meta(B, P, D_path, device)
        self.accept_len = torch.empty((B,), **i32)
        self.accept_path = torch.empty((B, D_path), **i32)
        self.bonus = torch.empty((B,), **i32)
        self.pos_offset = torch.zeros((B,), **i32)
        self.top8 = None
        self.params = None
        self.prune_out = None
        if policy == "cast":
            S_T, S_D = cast_tables
            self.S_T = torch.as_tensor(S_T, dtype=torch.float64, device=device).contiguous()
            self.S_D = torch.as_tensor(S_D, dtype=torch.float64, device=device).contiguous()
            self.cast = cast
        if policy == "graft":
            self.graft = graft
            self.R_cap = graft["K_total"]
            anchor = DT_ANCHOR_TAIL if graft.get("anchor", "root") == "tail" else DT_ANCHOR_ROOT
            self.template = Template(*template, anchor=anchor)
            self.ret_anchor = torch.zeros((B,), **i32)
            self.retrieve_stream = torch.cuda.Stream(device=device) if anchor == DT_ANCHOR_ROOT else None
            self.retrieved = torch.cuda.Event() if anchor == DT_ANCHOR_ROOT else None
            self.ret_token = torch.empty((B, self.R_cap), **i32)
            self.ret_parent = torch.empty((B, self.R_cap), **i32)
            self.ret_count = torch.empty((B,), **i32)
            self.top8 = torch.empty((B, P, 8), **i32)
            self.params = make_prune_params(ckpt_layers=graft["ckpt_layers"], tau=graft["tau"],
                                            k_draft=graft["k_draft"], K_total=graft["K_total"], D_max=D)
            self.prune_out = make_prune_out(stop=self.stop, m=self.m_dev, stage=self.stage)

    def set_n0(self, n0):
        c = self.cast
        self.params = make_prune_params(S_T=self.S_T, S_D=self.S_D, L=c["L"], n0=n0, C1=c["C1"], C2=c["C2"],
                                        C3=c["C3"], R=c["R"], width_cap=c["width_cap"], m_cap=c["m_cap"],
                                        D_max=self.D, per_request=bool(c.get("per_request", False)))
        self.prune_out = make_prune_out(width=self.width, stop=self.stop)
        self.verify_out = make_prune_out(m=self.m_dev)

    def run(self, roots, draft_rows, target_rows, seed=0, rnd=0, M=None, n0=0, timing=None):
        """Launch one round; returns nothing (outputs live in this object's tensors).

        ``timing`` (optional): an object with ``start(kind)`` and ``stop(kind)``; the composite
        calls are then issued as their parts (dt_expand_layer + the pruning / frontier calls,
        dt_verify_rows + dt_verify_accept: the same kernels) and each part is bracketed by
        start/stop with kind "expand", "prune_select", "verify_rows" or "verify_accept", e.g. to
        record events around them.
        """
        h = self.h
        pol = self.policy
        if pol == "cast":
            self.set_n0(n0)
        if pol == "graft":  # the checkpoints only ever set stop; CAST writes every entry, EAGLE none
            self.stop.zero_()
        policy = {"cast": DT_POLICY_CAST_WIDTH_DEPTH, "graft": DT_POLICY_GRAFT_CHECKPOINT}.get(pol, DT_POLICY_NONE)
        width = None if pol == "cast" else self.width
        dt_tree_reset(h, roots)
        tail = pol == "graft" and self.template.anchor == DT_ANCHOR_TAIL
        if pol == "graft" and not tail:  # root-centred retrieval beside the draft layers (Graft step (2))
            main = torch.cuda.current_stream()
            self.retrieve_stream.wait_stream(main)
            with torch.cuda.stream(self.retrieve_stream):
                dt_graft_retrieve(h, M, self.template, self.R_cap, self.ret_token, self.ret_parent, self.ret_count,
                                  ret_anchor=self.ret_anchor)
                self.retrieved.record(self.retrieve_stream)
        if self.block:  # a block drafter: every draft layer from one set of rows, gated per position
            rows = draft_rows(0, None)
            if timing is not None:
                timing.start("expand")
            dt_block_expand(h, rows, self.D, self.params, self.prune_out)
            if timing is not None:
                timing.stop("expand")
        else:
            dt_select_frontier(h, None, None, self.frontier_token)  # layer 0 = {root}: the root in slot 0
        for d in range(1, 0 if self.block else self.D + 1):
            F = 1 if d == 1 else self.k
            if d > 1 and not self.fused:
                dt_select_frontier(h, self.width, self.stop, self.frontier_token)
            logits = draft_rows(d, self.frontier_token)
            if self.draw:  # sampled drafts: draws from every frontier row, no pruning (EAGLE-2 frontier)
                if timing is not None:
                    timing.start("expand")
                dt_expand_layer_sampled(h, logits, self.k, seed, rnd)
                if timing is not None:
                    timing.stop("expand")
                if d < self.D:
                    dt_select_frontier(h, self.width, None, self.frontier_token)
                continue
            if not self.fused:
                dt_expand_layer(h, logits, F)
                if pol in ("cast", "graft"):
                    dt_cast_prune(h, policy, self.params, self.prune_out)
            elif timing is not None:  # the kernels of dt_expand_prune_select, as separate calls
                timing.start("expand")
                dt_expand_layer(h, logits, F)
                timing.stop("expand")
                timing.start("prune_select")
                if pol == "cast":
                    if d < self.D:
                        dt_cast_prune_select(h, self.params, self.prune_out, self.frontier_token)
                    else:
                        dt_cast_prune(h, policy, self.params, self.prune_out)
                else:
                    if pol == "graft":
                        dt_cast_prune(h, policy, self.params, self.prune_out)
                    if d < self.D:
                        dt_select_frontier(h, self.width, self.stop if pol == "graft" else None,
                                           self.frontier_token)
                timing.stop("prune_select")
            else:
                dt_expand_prune_select(h, logits, F, policy, self.params, self.prune_out, width, self.frontier_token)
        if pol == "cast" and self.fused:  # verify count and the rerank to it
            dt_cast_verify_rerank(h, self.params, self.verify_out, self.selected)
        else:
            if pol == "cast":
                dt_cast_prune(h, DT_POLICY_CAST_VERIFY, self.params, self.verify_out)
            dt_rerank(h, self.m_dev, self.m_cap, self.selected)
        if pol == "graft":
            if tail:
                dt_graft_retrieve(h, M, self.template, self.R_cap, self.ret_token, self.ret_parent, self.ret_count,
                                  selected=self.selected, m_cap=self.m_cap, ret_anchor=self.ret_anchor)
            else:
                torch.cuda.current_stream().wait_event(self.retrieved)
            dt_build_tree_meta(h, self.selected, self.m_cap, self.meta, self.pos_offset, self.ret_token,
                               self.ret_parent, self.ret_count, self.R_cap, ret_anchor=self.ret_anchor,
                               K_total=self.graft["K_total"])
        else:
            dt_build_tree_meta(h, self.selected, self.m_cap, self.meta, self.pos_offset)
        logits = target_rows(self.meta)
        mode = (DT_SAMPLE if self.T == 1 else DT_GREEDY) | (DT_VERIFY_PACKED if self.packed else 0)
        if self.draw:
            if timing is not None:
                timing.start("verify_sampled")
            dt_verify_sampled(h, self.meta, logits, self.draft_rows, seed, rnd, self.accept_len, self.accept_path,
                              self.bonus, packed=self.packed)
            if timing is not None:
                timing.stop("verify_sampled")
        elif timing is not None:
            timing.start("verify_rows")
            dt_verify_rows(h, self.meta, logits, mode, self.top8 is not None)
            timing.stop("verify_rows")
            timing.start("verify_accept")
            dt_verify_accept(h, self.meta, logits, mode, seed, rnd, self.accept_len, self.accept_path, self.bonus,
                             self.top8)
            timing.stop("verify_accept")
        else:
            dt_verify(h, self.meta, logits, mode, seed, rnd, self.accept_len, self.accept_path, self.bonus,
                      self.top8)
        if pol == "graft":
            dt_adj_update(h, M, self.meta, self.top8)
