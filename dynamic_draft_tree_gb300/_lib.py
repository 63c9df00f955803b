"""ctypes binding of libdt.so: the same entry points as include/dt.h, argument marshalling only.

Tensors are torch CUDA tensors; their device pointers and the current CUDA
stream are handed to the C ABI. Every computation runs in the library's
kernels. Importing this module fails loudly when libdt.so is missing.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdt.so")

DT_OK, DT_ERR_ARG, DT_ERR_CUDA, DT_ERR_DEVICE, DT_ERR_DEVICE_TIMEOUT = 0, -1, -2, -3, -4
DT_BF16, DT_F32 = 0, 1
DT_GREEDY, DT_SAMPLE = 0, 1
DT_VERIFY_PACKED = 2
DT_POLICY_CAST_WIDTH_DEPTH, DT_POLICY_CAST_VERIFY, DT_POLICY_GRAFT_CHECKPOINT, DT_POLICY_NONE = 0, 1, 2, 3
DT_DEV_BAD_LOGITS, DT_DEV_BAD_TOKEN, DT_DEV_BAD_TREE, DT_DEV_TIMEOUT, DT_DEV_INTERNAL = 1, 2, 4, 8, 16
DT_DEV_KV_FULL = 32
DT_FLAG_TEST_TIMEOUT = 1
DT_ANCHOR_ROOT, DT_ANCHOR_TAIL = 0, 1

EXPORTS = ["dt_last_error_string", "dt_create", "dt_destroy", "dt_get_tree", "dt_get_status",
           "dt_clear_status", "dt_tree_reset", "dt_select_frontier", "dt_expand_layer", "dt_cast_prune",
           "dt_rerank", "dt_graft_retrieve", "dt_build_tree_meta", "dt_verify", "dt_adj_update",
           "dt_row_topk_static", "dt_cast_prune_select",
           "dt_cast_verify_rerank", "dt_expand_prune_select", "dt_verify_rows", "dt_verify_accept",
           "dt_commit_kv", "dt_block_expand", "dt_expand_layer_sampled", "dt_verify_sampled"]

c_i32p = ctypes.c_void_p
vp = ctypes.c_void_p


class DtConfig(ctypes.Structure):
    _fields_ = [("B_max", ctypes.c_int32), ("V", ctypes.c_int32), ("K", ctypes.c_int32),
                ("W", ctypes.c_int32), ("D_max", ctypes.c_int32), ("P_max", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("flags", ctypes.c_int32)]


class DtTreeView(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("K", ctypes.c_int32), ("W", ctypes.c_int32),
                ("D_max", ctypes.c_int32), ("N", ctypes.c_int32), ("LW", ctypes.c_int32),
                ("depth", ctypes.c_int32), ("token", vp), ("parent", vp), ("node_depth", vp),
                ("logc", vp), ("value", vp), ("layer_order", vp), ("layer_count", vp),
                ("frontier", vp), ("frontier_count", vp)]


class DtPruneParams(ctypes.Structure):
    _fields_ = [("S_T", vp), ("S_D", vp), ("M_rows", ctypes.c_int32), ("N_cols", ctypes.c_int32),
                ("L", ctypes.c_double), ("n0", ctypes.c_int64), ("C1", ctypes.c_double),
                ("C2", ctypes.c_double), ("C3", ctypes.c_double), ("R", ctypes.c_int32),
                ("width_cap", ctypes.c_int32), ("m_cap", ctypes.c_int32), ("D_max", ctypes.c_int32),
                ("n_ckpt", ctypes.c_int32), ("ckpt_layer", ctypes.c_int32 * 16),
                ("tau", ctypes.c_double * 16), ("k_draft", ctypes.c_int32 * 16),
                ("K_total", ctypes.c_int32), ("per_request", ctypes.c_int32)]


class DtPruneOut(ctypes.Structure):
    _fields_ = [("width", vp), ("stop", vp), ("m", vp), ("stage", vp)]


class DtTemplate(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int32), ("parent", vp), ("rank", vp), ("anchor", ctypes.c_int32)]


class DtTreeMeta(ctypes.Structure):
    _fields_ = [("P", ctypes.c_int32), ("D_path", ctypes.c_int32), ("tokens", vp), ("parents", vp),
                ("depth", vp), ("node_id", vp), ("mask", vp), ("position_ids", vp),
                ("retrieve", vp), ("n_leaves", vp), ("n_pos", vp), ("row_off", vp)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libdt.so not found at {LIB_PATH}: build it with __graft_entry__.build() "
                          "(there is no fallback implementation)")
    lib = ctypes.CDLL(LIB_PATH)
    I = ctypes.c_int
    sig = {
        "dt_last_error_string": ([], ctypes.c_char_p),
        "dt_create": ([ctypes.POINTER(DtConfig), ctypes.POINTER(vp)], I),
        "dt_destroy": ([vp], I),
        "dt_get_tree": ([vp, ctypes.POINTER(DtTreeView)], I),
        "dt_get_status": ([vp, vp, ctypes.POINTER(ctypes.c_int32)], I),
        "dt_clear_status": ([vp, vp], I),
        "dt_tree_reset": ([vp, ctypes.c_int32, vp, vp], I),
        "dt_select_frontier": ([vp, vp, ctypes.c_int32, vp, vp, vp], I),
        "dt_expand_layer": ([vp, vp, ctypes.c_int64, ctypes.c_int32, vp], I),
        "dt_cast_prune": ([vp, ctypes.c_int32, ctypes.POINTER(DtPruneParams), ctypes.POINTER(DtPruneOut), vp], I),
        "dt_rerank": ([vp, vp, ctypes.c_int32, ctypes.c_int32, vp, vp], I),
        "dt_graft_retrieve": ([vp, vp, ctypes.POINTER(DtTemplate), ctypes.c_int32, vp, ctypes.c_int32,
                               vp, vp, vp, vp, vp], I),
        "dt_build_tree_meta": ([vp, vp, ctypes.c_int32, vp, vp, vp, vp, ctypes.c_int32, ctypes.c_int32, vp,
                                ctypes.POINTER(DtTreeMeta), vp], I),
        "dt_expand_layer_sampled": ([vp, vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64, ctypes.c_uint64, vp], I),
        "dt_verify_sampled": ([vp, ctypes.POINTER(DtTreeMeta), vp, ctypes.c_int64, ctypes.c_int32, vp, ctypes.c_int64,
                               ctypes.c_uint64, ctypes.c_uint64, vp, vp, vp, vp], I),
        "dt_block_expand": ([vp, vp, ctypes.c_int64, ctypes.c_int32, ctypes.POINTER(DtPruneParams),
                             ctypes.POINTER(DtPruneOut), vp], I),
        "dt_verify": ([vp, ctypes.POINTER(DtTreeMeta), vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64,
                       ctypes.c_uint64, vp, vp, vp, vp, vp], I),
        "dt_adj_update": ([vp, vp, ctypes.POINTER(DtTreeMeta), vp, vp], I),
        "dt_cast_prune_select": ([vp, ctypes.POINTER(DtPruneParams), ctypes.POINTER(DtPruneOut), vp, vp], I),
        "dt_expand_prune_select": ([vp, vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                    ctypes.POINTER(DtPruneParams), ctypes.POINTER(DtPruneOut), vp, ctypes.c_int32,
                                    vp, vp], I),
        "dt_verify_rows": ([vp, ctypes.POINTER(DtTreeMeta), vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, vp], I),
        "dt_verify_accept": ([vp, ctypes.POINTER(DtTreeMeta), vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64,
                              ctypes.c_uint64, vp, vp, vp, vp, vp], I),
        "dt_commit_kv": ([vp, vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, vp, ctypes.c_int64, ctypes.c_int64,
                          ctypes.c_int32, ctypes.c_int64, vp, vp, vp, ctypes.c_int32, vp, vp], I),
        "dt_cast_verify_rerank": ([vp, ctypes.POINTER(DtPruneParams), ctypes.POINTER(DtPruneOut), vp, vp], I),
        "dt_row_topk_static": ([vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                vp, vp, vp, vp], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


lib = _load()


class DtError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"libdt error {code}: {msg}")
        self.code = code


def check(rc):
    if rc != DT_OK:
        raise DtError(rc, lib.dt_last_error_string().decode(errors="replace"))
    return rc
