"""Seeded synthetic logits for the draft-tree workloads (inputs only; no tree arithmetic).

The draft and target model forwards are outside the hot path; this module
stands in for them with counter-hashed rows. The host (``synth_cpu.c``) and
device (``synth_gpu.cu``) implementations follow the one definition below and
are checked bit for bit against each other. Both the oracle harness and the
GPU harness take their rows from here; nothing here knows about trees.

Definition (all integer arithmetic mod 2^64):

* mix64 = the SplitMix64 output function (Steele, Lea, Flood 2014);
  hk(a, x) = mix64(a ^ mix64(x + 0x9E3779B97F4A7C15)).
* Row key r = hk(hk(hk(hk(seed, salt), b), depthkey), ctx): request b, the
  depth key of the row and the token ``ctx`` whose next-token row it is.
* Noise of token v on lane L (0 = draft, 1 = the target's extra lane): the sum
  of the twelve 16-bit fields of mix64(r ^ (v<<3 | L<<2 | j)), j = 0..2, minus
  393210 (an integer Irwin-Hall sum with variance ~65536^2).
  Draft noise = I_0 * fp32(sigma/65536); target noise =
  (4*I_0 + 3*I_1) * fp32(sigma/(5*65536)), i.e. 0.8 z_draft + 0.6 z'.
* kind 0 (normal + peak): peak token = mix64(r ^ PEAK_SALT) mod V, height =
  lo_b + (hi_b - lo_b) * u24 * 2^-24 with u24 from mix64(src ^ HEIGHT_SALT) >> 40,
  src = r (per row) or hk(hk(seed, salt), b) (per request); the height is
  added to the peak token only. Draft and target rows of the same key share
  the peak and the height.
* kind 1 (Zipf): rank(v) = (a*v + c) mod V with a coprime to V and c from the
  key; x_v = -s * ln_table[rank] + noise, ln_table[k] = fp32(ln(k + 1)) built
  once on the host. kind 2: the Zipf row of kind 1 with the permutation shifted so that
  the peak token of kind 0 has rank 0, plus that peak's height.
* Every fp32 step rounds once (no fused multiply-add); bf16 output rounds to
  nearest even from the fp32 value.
"""

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
CPU_LIB = os.path.join(HERE, "libsynth_cpu.so")
GPU_LIB = os.path.join(HERE, "libsynth_gpu.so")

DRAFT, TARGET = 0, 1
BF16, F32 = 0, 1


class SpecC(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("V", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("height_per_request", ctypes.c_int32), ("sigma", ctypes.c_float),
                ("zipf_s", ctypes.c_float), ("peak_lo", ctypes.c_void_p),
                ("peak_hi", ctypes.c_void_p), ("ln_table", ctypes.c_void_p),
                ("salts", ctypes.c_void_p)]


def _fresh(lib, src):
    """lib exists, is newer than src and is an ELF file for this machine."""
    import platform

    want = {"x86_64": 62, "aarch64": 183, "arm64": 183}.get(platform.machine())
    if not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(src):
        return False
    with open(lib, "rb") as f:
        head = f.read(20)
    return head[:4] == b"\x7fELF" and int.from_bytes(head[18:20], "little") == want


def build_cpu(force=False):
    src = os.path.join(HERE, "synth_cpu.c")
    if force or not _fresh(CPU_LIB, src):
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                               "-o", CPU_LIB, src, "-lm"])


def build_gpu(force=False, arch="103a"):
    src = os.path.join(HERE, "synth_gpu.cu")
    if force or not _fresh(GPU_LIB, src):
        subprocess.check_call(["nvcc", "-O3", f"-gencode=arch=compute_{arch},code=sm_{arch}",
                               "-lineinfo", "-Xcompiler", "-fPIC", "-shared", "-o", GPU_LIB, src])


_cpu = None
_gpu = None


def _cpu_lib():
    global _cpu
    if _cpu is None:
        build_cpu()
        lib = ctypes.CDLL(CPU_LIB)
        lib.synth_gen_rows.argtypes = [ctypes.POINTER(SpecC), ctypes.c_uint64, ctypes.c_uint64,
                                       ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                       ctypes.c_int64, ctypes.c_int32]
        lib.synth_root_token.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64,
                                         ctypes.c_int32]
        lib.synth_root_token.restype = ctypes.c_int32
        lib.synth_zipf_table.argtypes = [ctypes.c_int32, ctypes.c_void_p]
        _cpu = lib
    return _cpu


def _gpu_lib():
    global _gpu
    if _gpu is None:
        if not os.path.exists(GPU_LIB):
            raise RuntimeError("libsynth_gpu.so is not built; run __graft_entry__.build()")
        lib = ctypes.CDLL(GPU_LIB)
        lib.synth_gen_rows_gpu.argtypes = [ctypes.POINTER(SpecC), ctypes.c_uint64, ctypes.c_uint64,
                                           ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p]
        lib.synth_gen_rows_gpu.restype = ctypes.c_int
        lib.synth_host_device_ptr.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)]
        lib.synth_host_device_ptr.restype = ctypes.c_int
        lib.synth_gather_spans_gpu.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]
        lib.synth_gather_spans_gpu.restype = ctypes.c_int
        _gpu = lib
    return _gpu


def zipf_table(V):
    out = np.empty(V, np.float32)
    _cpu_lib().synth_zipf_table(V, out.ctypes.data)
    return out


def root_tokens(seed, salt, B, V):
    lib = _cpu_lib()
    return np.array([lib.synth_root_token(seed, salt, b, V) for b in range(B)], np.int32)


class Spec:
    """Row recipe for one workload. ``peak_lo``/``peak_hi`` are per request."""

    def __init__(self, V, dtype=BF16, kind=0, sigma=2 ** 0.5, peak_lo=None, peak_hi=None,
                 height_per_request=False, zipf_s=1.1, B=1):
        self.V, self.dtype, self.kind, self.sigma = V, dtype, kind, sigma
        self.height_per_request = height_per_request
        self.zipf_s = zipf_s
        lo = np.zeros(B, np.float32) if peak_lo is None else np.asarray(peak_lo, np.float32)
        hi = np.zeros(B, np.float32) if peak_hi is None else np.asarray(peak_hi, np.float32)
        if lo.size == 1 and B > 1:
            lo = np.full(B, lo.item(), np.float32)
        if hi.size == 1 and B > 1:
            hi = np.full(B, hi.item(), np.float32)
        self.peak_lo, self.peak_hi = lo, hi
        self.ln_table = zipf_table(V) if kind != 0 else np.zeros(1, np.float32)
        self._dev = None

    @property
    def np_dtype(self):
        return np.uint16 if self.dtype == BF16 else np.float32

    def c_struct_host(self, salts=None):
        return SpecC(self.kind, self.V, self.dtype, int(self.height_per_request), self.sigma,
                     self.zipf_s, self.peak_lo.ctypes.data, self.peak_hi.ctypes.data,
                     self.ln_table.ctypes.data, None if salts is None else salts.ctypes.data)

    def c_struct_device(self, torch, salts_dev=None):
        if self._dev is None:
            self._dev = [torch.from_numpy(self.peak_lo).cuda(), torch.from_numpy(self.peak_hi).cuda(),
                         torch.from_numpy(self.ln_table).cuda()]
        lo, hi, ln = self._dev
        return SpecC(self.kind, self.V, self.dtype, int(self.height_per_request), self.sigma,
                     self.zipf_s, lo.data_ptr(), hi.data_ptr(), ln.data_ptr(),
                     None if salts_dev is None else salts_dev.data_ptr())


def gen_rows_cpu(spec, seed, salt, stream, ctx, depth=None, depth_add=0, rows_per_b=1, b0=0, salts=None):
    """Rows for contexts ``ctx`` (int32 [R]); returns raw bits (uint16 for bf16) or fp32, [R][V].

    Row rr belongs to request b0 + rr // rows_per_b. Rows whose ctx is negative are zeros.
    ``salts`` (uint64 [B], optional) replaces ``salt`` per request.
    """
    ctx = np.ascontiguousarray(ctx, np.int32).ravel()
    R = ctx.size
    out = np.zeros((R, spec.V), spec.np_dtype)
    dptr = None
    if depth is not None:
        depth = np.ascontiguousarray(depth, np.int32).ravel()
        dptr = depth.ctypes.data
    if salts is not None:
        salts = np.ascontiguousarray(salts, np.uint64)
    st = spec.c_struct_host(salts)
    _cpu_lib().synth_gen_rows(ctypes.byref(st), seed, salt, stream, ctx.ctypes.data, dptr,
                              depth_add, rows_per_b, b0, out.ctypes.data, spec.V, R)
    return out


def gen_rows_gpu(torch, spec, seed, salt, stream, ctx_dev, out_dev, ld, depth_dev=None, depth_add=0,
                 rows_per_b=1, cuda_stream=None, salts_dev=None, row_req_dev=None):
    """Device rows into ``out_dev`` (row rr at element rr*ld); ctx/depth are device int32 tensors;
    ``salts_dev`` (device int64 [B], optional) replaces ``salt`` per request; row rr belongs to
    request rr // rows_per_b, or to ``row_req_dev[rr]`` (device int32 [R]) when given (packed rows)."""
    st = spec.c_struct_device(torch, salts_dev)
    cs = (cuda_stream or torch.cuda.current_stream()).cuda_stream
    R = ctx_dev.numel()
    rc = _gpu_lib().synth_gen_rows_gpu(ctypes.byref(st), seed, salt, stream, ctx_dev.data_ptr(),
                                       None if depth_dev is None else depth_dev.data_ptr(), depth_add,
                                       rows_per_b, None if row_req_dev is None else row_req_dev.data_ptr(),
                                       out_dev.data_ptr(), ld, R, cs)
    if rc != 0:
        raise RuntimeError(f"synth_gen_rows_gpu failed ({rc})")


def host_device_ptr(t):
    """Device address of a pinned host tensor's storage (its mapping for kernels), or None when the
    memory is not mapped for the device."""
    dev = ctypes.c_void_p()
    if _gpu_lib().synth_host_device_ptr(ctypes.c_void_p(t.data_ptr()), ctypes.byref(dev)) != 0 or not dev.value:
        return None
    return int(dev.value)


def gather_spans_gpu(torch, spans_dev, blocks, cuda_stream=None):
    """Moves host bytes to the device with a kernel: spans_dev is a device int64 tensor [n][3] of
    (source address for the device, destination address, bytes)."""
    cs = (cuda_stream or torch.cuda.current_stream()).cuda_stream
    rc = _gpu_lib().synth_gather_spans_gpu(spans_dev.data_ptr(), spans_dev.shape[0], blocks, cs)
    if rc != 0:
        raise RuntimeError(f"synth_gather_spans_gpu failed ({rc})")


def bf16_bits_to_f64(bits):
    """Exact widening of bf16 bit patterns to float64."""
    b = np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def to_f64(rows, dtype):
    return bf16_bits_to_f64(rows) if dtype == BF16 else np.asarray(rows, np.float32).astype(np.float64)


def packed_row_map(torch, row_off, tokens, depth):
    """Per-row inputs of a padding-free target batch, on the device (graph-capturable, no sync).

    row_off [B+1] (dt_tree_meta.row_off), tokens/depth [B][P] (the verify tree): for every row j of a
    [B*P] buffer, the request b with row_off[b] <= j < row_off[b+1], the context token tokens[b][j -
    row_off[b]] and its depth; rows past row_off[B] get token -1 (not generated). Returns int32
    (row_req, ctx, depth) of length B*P."""
    B, P = tokens.shape
    j = torch.arange(B * P, device=tokens.device, dtype=torch.int64)
    off = row_off.to(torch.int64)
    b = torch.searchsorted(off[1:].contiguous(), j, right=True).clamp_(max=B - 1)
    i = (j - off[b]).clamp_(0, P - 1)
    valid = j < off[B]
    ctx = torch.where(valid, tokens[b, i], torch.full_like(j, -1, dtype=tokens.dtype))
    dep = torch.where(valid, depth[b, i], torch.zeros_like(j, dtype=depth.dtype))
    return b.to(torch.int32), ctx.to(torch.int32).contiguous(), dep.to(torch.int32).contiguous()
