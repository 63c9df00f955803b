"""GB300 dynamic draft-tree hot path: Python binding of the libdt C ABI.

Every function here has the name of the C entry point it calls and only
marshals arguments (torch CUDA tensors -> device pointers, the current CUDA
stream); all work runs in libdt's sm_103a kernels. See include/dt.h for the
semantics, layouts and error behaviour of each call.
"""
import ctypes

import torch

from ._lib import (lib, check, DtError, DtConfig, DtTreeView, DtPruneParams, DtPruneOut, DtTemplate,  # noqa
                   DtTreeMeta, EXPORTS, DT_OK, DT_ERR_ARG, DT_ERR_CUDA, DT_ERR_DEVICE,
                   DT_ERR_DEVICE_TIMEOUT, DT_BF16, DT_F32, DT_GREEDY, DT_SAMPLE, DT_VERIFY_PACKED,
                   DT_POLICY_CAST_WIDTH_DEPTH, DT_POLICY_CAST_VERIFY, DT_POLICY_GRAFT_CHECKPOINT, DT_POLICY_NONE,
                   DT_DEV_BAD_LOGITS, DT_DEV_BAD_TOKEN, DT_DEV_BAD_TREE, DT_DEV_TIMEOUT, DT_DEV_INTERNAL, DT_DEV_KV_FULL,
                   DT_FLAG_TEST_TIMEOUT, DT_ANCHOR_ROOT, DT_ANCHOR_TAIL, LIB_PATH)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensor required")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor required")
    return t.data_ptr()


def _stream(stream=None):
    return (stream if stream is not None else torch.cuda.current_stream()).cuda_stream


class Handle:
    """An open libdt handle (one draft tree in flight) and its configuration."""

    def __init__(self, B_max, V, K, W, D_max, P_max, dtype=DT_BF16, flags=0):
        self.cfg = DtConfig(B_max, V, K, W, D_max, P_max, dtype, flags)
        self.h = ctypes.c_void_p()
        check(lib.dt_create(ctypes.byref(self.cfg), ctypes.byref(self.h)))

    def close(self):
        if self.h:
            check(lib.dt_destroy(self.h))
            self.h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class _DevArray:
    """Zero-copy view of a library-owned device array, for torch.as_tensor."""

    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (ptr, False), "version": 3, "strides": None}


def dt_create(B_max, V, K, W, D_max, P_max, dtype=DT_BF16, flags=0):
    return Handle(B_max, V, K, W, D_max, P_max, dtype, flags)


def dt_destroy(h):
    h.close()


def dt_get_tree(h):
    """The tree arrays as torch tensors viewing the handle's workspace (valid until the next call)."""
    v = DtTreeView()
    check(lib.dt_get_tree(h.h, ctypes.byref(v)))
    Bm, N, D, LW, W = h.cfg.B_max, v.N, v.D_max, v.LW, v.W

    def view(ptr, shape, ts):
        return torch.as_tensor(_DevArray(ptr, shape, ts), device="cuda")

    return dict(B=v.B, K=v.K, W=W, D_max=D, N=N, LW=LW, depth=v.depth,
                token=view(v.token, (Bm, N), "<i4"), parent=view(v.parent, (Bm, N), "<i4"),
                node_depth=view(v.node_depth, (Bm, N), "<i4"), logc=view(v.logc, (Bm, N), "<f4"),
                value=view(v.value, (Bm, N), "<f4"),
                layer_order=view(v.layer_order, (Bm, D + 1, LW), "<i4"),
                layer_count=view(v.layer_count, (Bm, D + 1), "<i4"),
                frontier=view(v.frontier, (Bm, W), "<i4"),
                frontier_count=view(v.frontier_count, (Bm,), "<i4"))


def dt_get_status(h, stream=None):
    """Synchronises the stream; returns the device status bits (0 = clean)."""
    bits = ctypes.c_int32(0)
    rc = lib.dt_get_status(h.h, _stream(stream), ctypes.byref(bits))
    if rc not in (DT_OK, DT_ERR_DEVICE, DT_ERR_DEVICE_TIMEOUT):
        check(rc)
    return bits.value


def dt_clear_status(h, stream=None):
    check(lib.dt_clear_status(h.h, _stream(stream)))


def dt_tree_reset(h, root_token, stream=None):
    check(lib.dt_tree_reset(h.h, root_token.numel(), _ptr(root_token), _stream(stream)))


def dt_select_frontier(h, width=None, stop=None, frontier_token=None, stream=None):
    wl = 0 if width is None else width.numel()
    check(lib.dt_select_frontier(h.h, _ptr(width), wl, _ptr(stop), _ptr(frontier_token), _stream(stream)))


def dt_expand_layer(h, logits, F, ld=None, stream=None):
    ld = logits.shape[-1] if ld is None else ld
    check(lib.dt_expand_layer(h.h, _ptr(logits), ld, F, _stream(stream)))


def dt_expand_prune_select(h, logits, F, policy, params=None, out=None, width=None, frontier_token=None, ld=None,
                           stream=None):
    """Expansion, then the policy's pruning (DT_POLICY_NONE: none), then the next frontier."""
    ld = logits.shape[-1] if ld is None else ld
    wl = 0 if width is None else width.numel()
    check(lib.dt_expand_prune_select(h.h, _ptr(logits), ld, F, policy,
                                     None if params is None else ctypes.byref(params),
                                     None if out is None else ctypes.byref(out), _ptr(width), wl,
                                     _ptr(frontier_token), _stream(stream)))


def dt_cast_prune(h, policy, params, out, stream=None):
    check(lib.dt_cast_prune(h.h, policy, ctypes.byref(params), ctypes.byref(out), _stream(stream)))


def dt_cast_prune_select(h, params, out, frontier_token=None, stream=None):
    """CAST width/depth pruning of the newest layer, then the next layer's frontier, in one launch."""
    check(lib.dt_cast_prune_select(h.h, ctypes.byref(params), ctypes.byref(out), _ptr(frontier_token),
                                   _stream(stream)))


def dt_cast_verify_rerank(h, params, out, selected, stream=None):
    """CAST verify count, then the rerank to that count (selected [B][m_cap]), in two launches."""
    check(lib.dt_cast_verify_rerank(h.h, ctypes.byref(params), ctypes.byref(out), _ptr(selected),
                                    _stream(stream)))


def dt_rerank(h, m, m_cap, selected, stream=None):
    ml = 0 if m is None else m.numel()
    check(lib.dt_rerank(h.h, _ptr(m), ml, m_cap, _ptr(selected), _stream(stream)))


def dt_graft_retrieve(h, M, template, R_cap, ret_token, ret_parent, ret_count, selected=None, m_cap=0,
                      ret_anchor=None, stream=None):
    """Retrieval envelope from M; a tail-anchored template needs ``selected`` / ``m_cap``."""
    check(lib.dt_graft_retrieve(h.h, _ptr(M), ctypes.byref(template.c), R_cap, _ptr(selected), m_cap,
                                _ptr(ret_token), _ptr(ret_parent), _ptr(ret_count), _ptr(ret_anchor),
                                _stream(stream)))


def dt_build_tree_meta(h, selected, m_cap, meta, pos_offset=None, ret_token=None, ret_parent=None,
                       ret_count=None, R_cap=0, ret_anchor=None, K_total=0, stream=None):
    check(lib.dt_build_tree_meta(h.h, _ptr(selected), m_cap, _ptr(ret_token), _ptr(ret_parent),
                                 _ptr(ret_count), _ptr(ret_anchor), R_cap, K_total, _ptr(pos_offset),
                                 ctypes.byref(meta.c), _stream(stream)))


def dt_expand_layer_sampled(h, logits, F, seed, round_, ld=None, stream=None):
    """dt_expand_layer with the children drawn from softmax(row) without replacement (Philox draws)."""
    ld = logits.shape[-1] if ld is None else ld
    check(lib.dt_expand_layer_sampled(h.h, _ptr(logits), ld, F, seed, round_, _stream(stream)))


def dt_verify_sampled(h, meta, logits, draft_rows, seed, round_, accept_len, accept_path, bonus, packed=False,
                      ld=None, ld_d=None, stream=None):
    """Verify of sampled drafts: draft_rows is the [D_max][B][W][V] buffer the layers were drawn from."""
    ld = logits.shape[-1] if ld is None else ld
    ld_d = draft_rows.shape[-1] if ld_d is None else ld_d
    check(lib.dt_verify_sampled(h.h, ctypes.byref(meta.c), _ptr(logits), ld, DT_VERIFY_PACKED if packed else 0,
                                _ptr(draft_rows), ld_d, seed, round_, _ptr(accept_len), _ptr(accept_path),
                                _ptr(bonus), _stream(stream)))


def dt_block_expand(h, logits, L, params=None, out=None, ld=None, stream=None):
    """Draft layers 1..L from a block drafter's rows [B][L][V] (one call; Graft gates with params)."""
    ld = logits.shape[-1] if ld is None else ld
    check(lib.dt_block_expand(h.h, _ptr(logits), ld, L, None if params is None else ctypes.byref(params),
                              None if out is None else ctypes.byref(out), _stream(stream)))


def dt_verify(h, meta, logits, mode, seed, round_, accept_len, accept_path, bonus, top8=None, ld=None,
              stream=None):
    ld = logits.shape[-1] if ld is None else ld
    check(lib.dt_verify(h.h, ctypes.byref(meta.c), _ptr(logits), ld, mode, seed, round_, _ptr(accept_len),
                        _ptr(accept_path), _ptr(bonus), _ptr(top8), _stream(stream)))


def dt_verify_rows(h, meta, logits, mode, with_top8=False, ld=None, stream=None):
    """Streaming half of dt_verify (one read of every used target row)."""
    ld = logits.shape[-1] if ld is None else ld
    check(lib.dt_verify_rows(h.h, ctypes.byref(meta.c), _ptr(logits), ld, mode, 1 if with_top8 else 0,
                             _stream(stream)))


def dt_verify_accept(h, meta, logits, mode, seed, round_, accept_len, accept_path, bonus, top8=None, ld=None,
                     stream=None):
    """Acceptance half of dt_verify (after dt_verify_rows)."""
    ld = logits.shape[-1] if ld is None else ld
    check(lib.dt_verify_accept(h.h, ctypes.byref(meta.c), _ptr(logits), ld, mode, seed, round_, _ptr(accept_len),
                               _ptr(accept_path), _ptr(bonus), _ptr(top8), _stream(stream)))


def dt_adj_update(h, M, meta, top8, stream=None):
    check(lib.dt_adj_update(h.h, _ptr(M), ctypes.byref(meta.c), _ptr(top8), _stream(stream)))


def dt_commit_kv(h, tmp_kv, cache, cache_len, accept_len, accept_path, row_off=None, P=None, stream=None):
    """Append the root's and the accepted positions' KV rows to each request's cache.

    tmp_kv [B][P][...] and cache [B][L_max][...] are device tensors whose trailing dimensions form
    one row (contiguous, a multiple of 16 bytes); cache_len [B] int32 is updated in place. With
    ``row_off`` ([B+1] int32 device, dt_tree_meta.row_off) tmp_kv is packed: [rows][...], the row of
    position i of request b being row_off[b] + i; P (positions per request of the tree) is then
    required."""
    packed = row_off is not None
    lead = 1 if packed else 2
    if tmp_kv.dim() < lead + 1 or cache.dim() < 3:
        raise ValueError("tmp_kv needs [B][positions][row...] ([rows][row...] packed), cache [B][L_max][row...]")
    esz = tmp_kv.element_size()
    row0 = tmp_kv[0] if packed else tmp_kv[0, 0]
    row_bytes = row0.numel() * esz
    if cache[0, 0].numel() * cache.element_size() != row_bytes:
        raise ValueError("tmp_kv and cache rows differ in size")
    if not row0.is_contiguous() or not cache[0, 0].is_contiguous():
        raise ValueError("KV rows must be contiguous")
    for t in (tmp_kv, cache):
        if not t.is_cuda:
            raise ValueError("device tensor required")
    if packed:
        if P is None:
            raise ValueError("P is required with row_off")
        pos_stride, req_stride = tmp_kv.stride(0) * esz, 0
    else:
        P = tmp_kv.shape[1]
        pos_stride, req_stride = tmp_kv.stride(1) * esz, tmp_kv.stride(0) * esz
    check(lib.dt_commit_kv(h.h, tmp_kv.data_ptr(), pos_stride, req_stride, P,
                           cache.data_ptr(), cache.stride(1) * cache.element_size(),
                           cache.stride(0) * cache.element_size(), cache.shape[1], row_bytes, _ptr(cache_len),
                           _ptr(accept_len), _ptr(accept_path), accept_path.shape[-1], _ptr(row_off),
                           _stream(stream)))


def dt_row_topk_static(logits, K, logp, ids, V=None, status=None, stream=None):
    """Row log-softmax top-K with no handle and no allocation: logits [rows][ld] (bf16 or fp32),
    logp [rows][K] fp32 and ids [rows][K] int32 caller-owned; status an int32 device word or None."""
    ld = logits.shape[-1]
    rows = logits.numel() // ld
    V = ld if V is None else V
    if logits.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("logits must be bfloat16 or float32")
    if logp.dtype != torch.float32 or ids.dtype != torch.int32 or logp.numel() < rows * K or ids.numel() < rows * K:
        raise ValueError("logp must be float32 and ids int32, each with rows*K elements")
    dtype = DT_BF16 if logits.dtype == torch.bfloat16 else DT_F32
    check(lib.dt_row_topk_static(_ptr(logits), ld, rows, V, K, dtype, _ptr(logp), _ptr(ids), _ptr(status),
                                 _stream(stream)))


class Meta:
    """Caller-owned device arrays of a flattened verify tree (dt_tree_meta)."""

    def __init__(self, B, P, D_path, device="cuda"):
        i32 = dict(dtype=torch.int32, device=device)
        self.P, self.D_path = P, D_path
        self.tokens = torch.empty((B, P), **i32)
        self.parents = torch.empty((B, P), **i32)
        self.depth = torch.empty((B, P), **i32)
        self.node_id = torch.empty((B, P), **i32)
        self.mask = torch.empty((B, P, P), dtype=torch.uint8, device=device)
        self.position_ids = torch.empty((B, P), **i32)
        self.retrieve = torch.empty((B, P, D_path), **i32)
        self.n_leaves = torch.empty((B,), **i32)
        self.n_pos = torch.empty((B,), **i32)
        self.row_off = torch.empty((B + 1,), **i32)
        self.c = DtTreeMeta(P, D_path, *[_ptr(t) for t in (self.tokens, self.parents, self.depth, self.node_id,
                                                            self.mask, self.position_ids, self.retrieve,
                                                            self.n_leaves, self.n_pos, self.row_off)])

    def numpy(self):
        return {k: getattr(self, k).cpu().numpy() for k in
                ("tokens", "parents", "depth", "node_id", "mask", "position_ids", "retrieve", "n_leaves",
                 "n_pos", "row_off")}


def make_prune_params(S_T=None, S_D=None, L=512.0, n0=0, C1=0.0, C2=0.0, C3=0.0, R=3, width_cap=1, m_cap=1,
                      D_max=1, ckpt_layers=(), tau=(), k_draft=(), K_total=0, per_request=False):
    """dt_prune_params from device tables (float64 tensors [M_rows][N_cols]) and scalars."""
    p = DtPruneParams()
    p.S_T = _ptr(S_T)
    p.S_D = _ptr(S_D)
    if S_T is not None:
        p.M_rows, p.N_cols = S_T.shape
    p.L, p.n0, p.C1, p.C2, p.C3, p.R = L, n0, C1, C2, C3, R
    p.width_cap, p.m_cap, p.D_max = width_cap, m_cap, D_max
    p.n_ckpt = len(ckpt_layers)
    for i, (c, t, k) in enumerate(zip(ckpt_layers, tau, k_draft)):
        p.ckpt_layer[i], p.tau[i], p.k_draft[i] = c, t, k
    p.K_total = K_total
    p.per_request = 1 if per_request else 0
    return p


def make_prune_out(width=None, stop=None, m=None, stage=None):
    return DtPruneOut(_ptr(width), _ptr(stop), _ptr(m), _ptr(stage))


class Template:
    """Host-side retrieval template (parent, rank) in breadth-first order, hanging from the root or
    (anchor DT_ANCHOR_TAIL) from the deepest kept draft node."""

    def __init__(self, parent, rank, anchor=DT_ANCHOR_ROOT):
        self.n = len(parent)
        self.anchor = anchor
        self._p = (ctypes.c_int32 * max(1, self.n))(*parent)
        self._r = (ctypes.c_int32 * max(1, self.n))(*rank)
        self.c = DtTemplate(self.n, ctypes.cast(self._p, ctypes.c_void_p), ctypes.cast(self._r, ctypes.c_void_p),
                            anchor)
