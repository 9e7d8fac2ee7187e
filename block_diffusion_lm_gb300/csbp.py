"""ctypes binding of libcsbp (include/csbp.h): argument marshalling only.

Every step of the attention path runs in the library's kernels; PyTorch is
used here only to own device memory and to name the current CUDA stream.
There is no fallback: if libcsbp.so is missing or fails to load, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcsbp.so")
INCLUDE = os.path.join(os.path.dirname(_PKG), "include")
HEADER = os.path.join(INCLUDE, "csbp.h")

OK = 0
STATUS = {0: "CSBP_OK", -1: "CSBP_ERR_INVALID", -2: "CSBP_ERR_UNSUPPORTED",
          -3: "CSBP_ERR_WORKSPACE", -4: "CSBP_ERR_CUDA", -5: "CSBP_ERR_TIMEOUT",
          -6: "CSBP_ERR_CAPACITY", -7: "CSBP_ERR_DEVICE"}


class CsbpError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")


class Problem(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("L", ctypes.c_int32), ("M", ctypes.c_int32),
                ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("d", ctypes.c_int32),
                ("P", ctypes.c_int32), ("tile_q", ctypes.c_int32), ("tile_kv", ctypes.c_int32),
                ("has_clean_queries", ctypes.c_int32), ("scale", ctypes.c_float),
                ("window", ctypes.c_int32), ("clean_causal", ctypes.c_int32),
                ("bwd_chunk", ctypes.c_int32), ("per_rank", ctypes.c_int32),
                ("rank", ctypes.c_int32)]


class Inputs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("q_clean", "k_clean", "v_clean", "q_corr", "k_corr", "v_corr")] + [
                    ("stride_tok", ctypes.c_int64 * 6), ("stride_batch", ctypes.c_int64 * 6)]


class CeProblem(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int64), ("d_model", ctypes.c_int32), ("vocab", ctypes.c_int32),
                ("chunk_rows", ctypes.c_int32), ("head_grad", ctypes.c_int32),
                ("grad_scale", ctypes.c_float)]


class ScheduleInfo(ctypes.Structure):
    _fields_ = [("n_fwd_tasks", ctypes.c_int32), ("n_fwd_segments", ctypes.c_int32),
                ("n_bwd_tasks", ctypes.c_int32), ("n_bwd_segments", ctypes.c_int32),
                ("tile_pairs", ctypes.c_int64), ("bytes", ctypes.c_int64),
                ("problem_key", ctypes.c_uint64)]


_lib = None
_lib_path = LIB_PATH
DEBUG_LIB_PATH = os.path.join(_PKG, "libcsbp_debug.so")


def use_library(path: str = LIB_PATH) -> None:
    """Bind later calls to the library at `path` (e.g. the debug build,
    DEBUG_LIB_PATH, whose kernels check their work-list records)."""
    global _lib, _lib_path
    _lib, _lib_path = None, path


def lib():
    """Load the bound library, libcsbp.so by default (raises if it was not
    built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_lib_path):
            raise RuntimeError(f"{_lib_path} not built: run block_diffusion_lm_gb300.build.build()")
        L = ctypes.CDLL(_lib_path)
        P = ctypes.POINTER
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        L.csbp_block_schedule.argtypes = [P(Problem), P(i32), P(i32), vp, i64, P(ScheduleInfo)]
        L.csbp_workspace_bytes.argtypes = [P(Problem), ctypes.c_int]
        L.csbp_workspace_bytes.restype = sz
        L.csbp_attn_fwd.argtypes = [P(Problem), P(Inputs), vp, P(ScheduleInfo), vp, vp, vp, vp,
                                    sz, vp]
        L.csbp_attn_bwd.argtypes = [P(Problem), P(Inputs), vp, P(ScheduleInfo), vp, vp, vp, vp,
                                    vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.csbp_attn_bwd_noalloc.argtypes = [P(Problem), P(Inputs), vp, P(ScheduleInfo), vp, vp,
                                            vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.csbp_attn_bwd_noalloc.restype = ctypes.c_int
        L.csbp_e4m3_to_bf16.argtypes = [vp, ctypes.c_float, vp, i64, vp]
        L.csbp_e4m3_to_bf16.restype = ctypes.c_int
        L.csbp_attn_bwd_noalloc_status.argtypes = [vp]
        L.csbp_attn_bwd_noalloc_status.restype = ctypes.c_int
        L.csbp_lse_merge.argtypes = [i32, P(vp), P(vp), i64, i32, i32, vp, vp, vp]
        L.csbp_check_status.argtypes = [vp, vp]
        L.csbp_status_string.argtypes = [ctypes.c_int]
        L.csbp_status_string.restype = ctypes.c_char_p
        L.csbp_version.restype = i32
        L.csbp_kernel_timing.argtypes = [i32]
        L.csbp_kernel_timing_read.argtypes = [P(ctypes.c_double), P(i32), P(ctypes.c_double),
                                              P(i32)]
        L.csbp_kernel_timing_read_kind.argtypes = [i32, P(ctypes.c_double), P(i32)]
        L.csbp_wait_selftest.argtypes = [i64, vp, vp]
        L.csbp_ce_workspace_bytes.argtypes = [P(CeProblem)]
        L.csbp_ce_workspace_bytes.restype = sz
        L.csbp_vocab_ce.argtypes = [P(CeProblem), vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        for fn in ("csbp_block_schedule", "csbp_attn_fwd", "csbp_attn_bwd", "csbp_lse_merge",
                   "csbp_check_status", "csbp_kernel_timing", "csbp_kernel_timing_read",
                   "csbp_kernel_timing_read_kind", "csbp_vocab_ce", "csbp_wait_selftest"):
            getattr(L, fn).restype = ctypes.c_int
        _lib = L
    return _lib


def header_functions():
    """Names of the functions the headers under include/ declare."""
    names = set()
    for h in sorted(os.listdir(INCLUDE)):
        if h.endswith(".h"):
            with open(os.path.join(INCLUDE, h)) as f:
                text = f.read()
            names.update(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(csbp_\w+)\s*\(", text, re.M))
    return sorted(names)


def _check(fn, status):
    if status != OK:
        raise CsbpError(fn, status)


def make_problem(batch, L, M, Hq, Hkv, d, P=1, has_clean_queries=True, scale=None,
                 tile=128, window=0, clean_causal=False, bwd_chunk=0, rank=None) -> Problem:
    """rank=None: every query row; rank=r: only the rows CSBP rank r of P owns."""
    return Problem(batch, L, M, Hq, Hkv, d, P, tile, tile, 1 if has_clean_queries else 0,
                   float(scale if scale is not None else d ** -0.5), int(window),
                   1 if clean_causal else 0, int(bwd_chunk), 0 if rank is None else 1,
                   0 if rank is None else int(rank))


def block_schedule(problem: Problem):
    """Host work list: returns (block_owner, chunk_owner, words[int32], info)."""
    info = ScheduleInfo()
    B = problem.L // problem.M if problem.M > 0 else 0
    bo = np.zeros(max(B, 1), np.int32)
    co = np.zeros(max(2 * problem.P, 1), np.int32)
    st = lib().csbp_block_schedule(ctypes.byref(problem),
                                   bo.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                   co.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                   None, 0, ctypes.byref(info))
    if st != -6:
        _check("csbp_block_schedule", st)
    words = np.zeros(info.bytes // 4, np.int32)
    st = lib().csbp_block_schedule(ctypes.byref(problem),
                                   bo.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                   co.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                   words.ctypes.data_as(ctypes.c_void_p), words.nbytes,
                                   ctypes.byref(info))
    _check("csbp_block_schedule", st)
    return bo[:B], co[:2 * problem.P], words, info


def kernel_timing(enable: bool) -> None:
    """Start (clearing the record) or stop event timing of the main kernels."""
    _check("csbp_kernel_timing", lib().csbp_kernel_timing(1 if enable else 0))


def kernel_timing_read():
    """(fwd_kernel_ms, n_fwd, bwd_kernel_ms, n_bwd) summed over the record."""
    fm, bm = ctypes.c_double(), ctypes.c_double()
    fn, bn = ctypes.c_int32(), ctypes.c_int32()
    _check("csbp_kernel_timing_read",
           lib().csbp_kernel_timing_read(ctypes.byref(fm), ctypes.byref(fn), ctypes.byref(bm),
                                         ctypes.byref(bn)))
    return fm.value, fn.value, bm.value, bn.value


def kernel_timing_read_kind(kind: int):
    """(ms, launches) of one timer kind: 0 fwd, 1 bwd, 2 CE logits GEMM,
    3 CE row kernel, 4 CE dH GEMM, 5 CE dW GEMM."""
    ms, n = ctypes.c_double(), ctypes.c_int32()
    _check("csbp_kernel_timing_read_kind",
           lib().csbp_kernel_timing_read_kind(kind, ctypes.byref(ms), ctypes.byref(n)))
    return ms.value, n.value


def workspace_bytes(problem: Problem, which: int) -> int:
    return int(lib().csbp_workspace_bytes(ctypes.byref(problem), which))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


class _Checks:
    """Refuse tensors the library would misread: the C ABI sees only
    pointers, so dtype, shape and contiguity of every argument are checked
    first, then (in `done`) that all of them are on a CUDA device."""

    def __init__(self, fn):
        self.fn = fn
        self.seen = []

    def tensor(self, name, t, dtype, shape, required=True, strided=False):
        """`strided`: token and batch strides are free (the library takes
        them); heads and features must still be contiguous."""
        fn = self.fn
        if t is None:
            if required:
                raise ValueError(f"{fn}: {name} is required")
            return
        if t.dtype != dtype:
            raise ValueError(f"{fn}: {name} must be {dtype}, got {t.dtype}")
        if shape is not None and tuple(t.shape) != tuple(shape):
            raise ValueError(f"{fn}: {name} must have shape {tuple(shape)}, "
                             f"got {tuple(t.shape)}")
        if strided:
            if t.stride(3) != 1 or (t.shape[2] > 1 and t.stride(2) != t.shape[3]):
                raise ValueError(f"{fn}: {name} must have contiguous heads and features "
                                 f"(strides [..., d, 1]), got {tuple(t.stride())}")
            # a zero stride means "contiguous" to the library, so a broadcast
            # (expanded) batch or token dimension would be misread
            if any(t.shape[i] > 1 and t.stride(i) == 0 for i in (0, 1)):
                raise ValueError(f"{fn}: {name} has a broadcast (stride-0) batch or token "
                                 f"dimension; materialise it first")
            row = t.shape[2] * t.shape[3]
            if t.shape[1] > 1 and (t.stride(1) < row or t.stride(1) % 8):
                raise ValueError(f"{fn}: {name} token stride {t.stride(1)} must be >= H*d = "
                                 f"{row} and a multiple of 8")
            if t.shape[0] > 1 and (t.stride(0) < t.shape[1] * max(t.stride(1), row)
                                   or t.stride(0) % 8):
                raise ValueError(f"{fn}: {name} batch entries must not interleave (batch "
                                 f"stride >= L x token stride, a multiple of 8); make a "
                                 f"sequence-first layout batch-first")
        elif not t.is_contiguous():
            raise ValueError(f"{fn}: {name} must be contiguous")
        self.seen.append((name, t))

    def attn(self, problem, tensors):
        """q/o/dq/dO bf16 [batch][L][Hq][d], k/v/dk/dv bf16 [batch][L][Hkv][d],
        lse fp32 [batch][2][Hq][L]; clean-query tensors are optional when the
        problem has no clean queries."""
        import torch
        q = (problem.batch, problem.L, problem.Hq, problem.d)
        kv = (problem.batch, problem.L, problem.Hkv, problem.d)
        for name, t in tensors.items():
            if name == "lse":
                self.tensor(name, t, torch.float32, (problem.batch, 2, problem.Hq, problem.L))
                continue
            key_side = name.startswith(("k_", "v_", "dk_", "dv_"))
            optional = not key_side and name.endswith("_clean") and not problem.has_clean_queries
            self.tensor(name, t, torch.bfloat16, kv if key_side else q, required=not optional,
                        strided=name in _INPUT_NAMES)

    def done(self):
        for name, t in self.seen:
            if not t.is_cuda:
                raise ValueError(f"{self.fn}: {name} must be a CUDA tensor")


_INPUT_NAMES = ("q_clean", "k_clean", "v_clean", "q_corr", "k_corr", "v_corr")


def _inputs(inputs):
    """csbp_inputs from a dict of [batch][L][H][d] tensors: pointers, and the
    token / batch strides of each (0 where a dimension has one entry)."""
    ts = [inputs.get(n) for n in _INPUT_NAMES]
    tok = [0 if t is None or t.shape[1] == 1 else t.stride(1) for t in ts]
    bat = [0 if t is None or t.shape[0] == 1 else t.stride(0) for t in ts]
    return Inputs(*(_ptr(t) for t in ts), (ctypes.c_int64 * 6)(*tok),
                  (ctypes.c_int64 * 6)(*bat))


def _stream_ptr(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def attn_fwd(problem, inputs: dict, work_dev, info, o_clean, o_corr, lse, workspace, stream=None):
    import torch
    c = _Checks("csbp_attn_fwd")
    c.attn(problem, {**{n: inputs.get(n) for n in _INPUT_NAMES},
                     "o_clean": o_clean, "o_corr": o_corr, "lse": lse})
    c.tensor("work", work_dev, torch.int32, None)
    c.tensor("workspace", workspace, torch.uint8, None)
    c.done()
    inp = _inputs(inputs)
    st = lib().csbp_attn_fwd(ctypes.byref(problem), ctypes.byref(inp), _ptr(work_dev),
                             ctypes.byref(info), _ptr(o_clean), _ptr(o_corr), _ptr(lse),
                             _ptr(workspace), workspace.numel() * workspace.element_size(),
                             _stream_ptr(stream))
    _check("csbp_attn_fwd", st)


def _check_bwd(c, problem, inputs, work_dev, o_clean, o_corr, lse, do_clean, do_corr, grads):
    import torch
    names = ("dq_clean", "dq_corr", "dk_clean", "dv_clean", "dk_corr", "dv_corr")
    c.attn(problem, {**{n: inputs.get(n) for n in _INPUT_NAMES},
                     "o_clean": o_clean, "o_corr": o_corr, "lse": lse,
                     "do_clean": do_clean, "do_corr": do_corr,
                     **{n: grads.get(n) for n in names}})
    c.tensor("work", work_dev, torch.int32, None)


def attn_bwd(problem, inputs: dict, work_dev, info, o_clean, o_corr, lse, do_clean, do_corr,
             grads: dict, workspace, stream=None):
    import torch
    c = _Checks("csbp_attn_bwd")
    _check_bwd(c, problem, inputs, work_dev, o_clean, o_corr, lse, do_clean, do_corr, grads)
    c.tensor("workspace", workspace, torch.uint8, None)
    c.done()
    inp = _inputs(inputs)
    st = lib().csbp_attn_bwd(ctypes.byref(problem), ctypes.byref(inp), _ptr(work_dev),
                             ctypes.byref(info), _ptr(o_clean), _ptr(o_corr), _ptr(lse),
                             _ptr(do_clean), _ptr(do_corr), _ptr(grads.get("dq_clean")),
                             _ptr(grads["dq_corr"]), _ptr(grads["dk_clean"]),
                             _ptr(grads["dv_clean"]), _ptr(grads["dk_corr"]),
                             _ptr(grads["dv_corr"]), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _check("csbp_attn_bwd", st)


def attn_bwd_noalloc(problem, inputs: dict, work_dev, info, o_clean, o_corr, lse, do_clean,
                     do_corr, grads: dict, stream=None):
    """csbp_attn_bwd_noalloc: the backward with the library's own fixed
    scratch instead of a caller workspace (for callers that cannot allocate
    device memory; calls on one device must not overlap)."""
    c = _Checks("csbp_attn_bwd_noalloc")
    _check_bwd(c, problem, inputs, work_dev, o_clean, o_corr, lse, do_clean, do_corr, grads)
    c.done()
    inp = _inputs(inputs)
    st = lib().csbp_attn_bwd_noalloc(ctypes.byref(problem), ctypes.byref(inp), _ptr(work_dev),
                                     ctypes.byref(info), _ptr(o_clean), _ptr(o_corr), _ptr(lse),
                                     _ptr(do_clean), _ptr(do_corr), _ptr(grads.get("dq_clean")),
                                     _ptr(grads["dq_corr"]), _ptr(grads["dk_clean"]),
                                     _ptr(grads["dv_clean"]), _ptr(grads["dk_corr"]),
                                     _ptr(grads["dv_corr"]), _stream_ptr(stream))
    _check("csbp_attn_bwd_noalloc", st)


def attn_bwd_noalloc_status(stream=None):
    """csbp_attn_bwd_noalloc_status: synchronise the stream and raise if a
    device wait of the last allocation-free backward gave up."""
    _check("csbp_attn_bwd_noalloc_status", lib().csbp_attn_bwd_noalloc_status(_stream_ptr(stream)))


def e4m3_to_bf16(x, scale: float, out=None, stream=None):
    """csbp_e4m3_to_bf16: decode fp8 E4M3 bytes (a torch uint8 or
    float8_e4m3fn CUDA tensor) times `scale` into bf16 (out: bf16 tensor of
    the same shape, allocated if None)."""
    import torch
    c = _Checks("csbp_e4m3_to_bf16")
    if x is None or x.dtype not in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
        raise ValueError("csbp_e4m3_to_bf16: x must be a uint8 or float8_e4m3fn tensor")
    if not x.is_contiguous():
        raise ValueError("csbp_e4m3_to_bf16: x must be contiguous")
    if out is None:
        out = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
    c.tensor("out", out, torch.bfloat16, tuple(x.shape))
    c.seen.append(("x", x))
    c.done()
    _check("csbp_e4m3_to_bf16", lib().csbp_e4m3_to_bf16(_ptr(x), float(scale), _ptr(out),
                                                        x.numel(), _stream_ptr(stream)))
    return out


def lse_merge(o_parts, lse_parts, o_out, lse_out, stream=None):
    """o_parts: list of fp32 [rows, Hq, d] device tensors; lse_parts: list of
    fp32 [Hq, rows]; o_out bf16 [rows, Hq, d]; lse_out fp32 [Hq, rows]."""
    import torch
    c = _Checks("csbp_lse_merge")
    n = len(o_parts)
    if n < 1 or len(lse_parts) != n:
        raise ValueError("csbp_lse_merge: needs one LSE part per output part, at least one")
    rows, Hq, d = o_parts[0].shape
    for s, (o, z) in enumerate(zip(o_parts, lse_parts)):
        c.tensor(f"o_parts[{s}]", o, torch.float32, (rows, Hq, d))
        c.tensor(f"lse_parts[{s}]", z, torch.float32, (Hq, rows))
    c.tensor("o_out", o_out, torch.bfloat16, (rows, Hq, d))
    c.tensor("lse_out", lse_out, torch.float32, (Hq, rows))
    c.done()
    op = (ctypes.c_void_p * n)(*[t.data_ptr() for t in o_parts])
    zp = (ctypes.c_void_p * n)(*[t.data_ptr() for t in lse_parts])
    st = lib().csbp_lse_merge(n, op, zp, rows, Hq, d, _ptr(o_out), _ptr(lse_out),
                              _stream_ptr(stream))
    _check("csbp_lse_merge", st)


def wait_selftest(budget_ns, workspace, stream=None):
    """Launch the hang-guard self-test (a bounded wait that must give up)."""
    _check("csbp_wait_selftest",
           lib().csbp_wait_selftest(int(budget_ns), _ptr(workspace), _stream_ptr(stream)))


def check_status(workspace, stream=None):
    st = lib().csbp_check_status(_ptr(workspace), _stream_ptr(stream))
    _check("csbp_check_status", st)


class BlockDiffusionAttention:
    """Owns the device work list and workspaces of one problem shape.

    forward(t) / backward(t, o) take dicts of bf16 [batch, L, H, d] CUDA
    tensors (keys as in `inputs.make_inputs`) and return fresh outputs.
    """

    def __init__(self, batch, L, M, Hq, Hkv, d, P=1, has_clean_queries=True, scale=None,
                 device="cuda", window=0, clean_causal=False, bwd_chunk=0, rank=None):
        import torch
        self.problem = make_problem(batch, L, M, Hq, Hkv, d, P, has_clean_queries, scale,
                                    window=window, clean_causal=clean_causal,
                                    bwd_chunk=bwd_chunk, rank=rank)
        bo, co, words, info = block_schedule(self.problem)
        self.block_owner, self.chunk_owner, self.info = bo, co, info
        self.work_host = words
        self.work_dev = torch.from_numpy(words).to(device)
        self.ws_fwd = torch.zeros(workspace_bytes(self.problem, 0), dtype=torch.uint8, device=device)
        self.ws_bwd = torch.zeros(workspace_bytes(self.problem, 1), dtype=torch.uint8, device=device)
        self.device = device
        self.shape = (batch, L, Hq, d)
        self.kv_shape = (batch, L, Hkv, d)
        self.has_clean = has_clean_queries

    def alloc_outputs(self):
        import torch
        b, L, Hq, d = self.shape
        o_clean = torch.empty(self.shape, dtype=torch.bfloat16, device=self.device) if self.has_clean else None
        o_corr = torch.empty(self.shape, dtype=torch.bfloat16, device=self.device)
        lse = torch.full((b, 2, Hq, L), float("nan"), dtype=torch.float32, device=self.device)
        return o_clean, o_corr, lse

    def alloc_grads(self):
        import torch
        g = {k: torch.empty(self.kv_shape, dtype=torch.bfloat16, device=self.device)
             for k in ("dk_clean", "dv_clean", "dk_corr", "dv_corr")}
        g["dq_corr"] = torch.empty(self.shape, dtype=torch.bfloat16, device=self.device)
        g["dq_clean"] = (torch.empty(self.shape, dtype=torch.bfloat16, device=self.device)
                         if self.has_clean else None)
        return g

    def forward(self, t, out=None, stream=None):
        o_clean, o_corr, lse = out if out is not None else self.alloc_outputs()
        attn_fwd(self.problem, t, self.work_dev, self.info, o_clean, o_corr, lse, self.ws_fwd,
                 stream)
        return o_clean, o_corr, lse

    def backward(self, t, fwd_out, grads=None, stream=None):
        o_clean, o_corr, lse = fwd_out
        g = grads if grads is not None else self.alloc_grads()
        attn_bwd(self.problem, t, self.work_dev, self.info, o_clean, o_corr, lse,
                 t.get("do_clean"), t["do_corr"], g, self.ws_bwd, stream)
        return g

    def check(self, stream=None):
        check_status(self.ws_fwd, stream)
        check_status(self.ws_bwd, stream)


# ------------------------------------------------------------ vocabulary loss
def make_ce_problem(rows, d_model, vocab, chunk_rows=0, head_grad=True, grad_scale=1.0):
    return CeProblem(int(rows), int(d_model), int(vocab), int(chunk_rows),
                     1 if head_grad else 0, float(grad_scale))


def ce_workspace_bytes(problem: CeProblem) -> int:
    return int(lib().csbp_ce_workspace_bytes(ctypes.byref(problem)))


def vocab_ce(problem, h, w, target, loss, lse, dh, dw, workspace, stream=None):
    import torch
    c = _Checks("csbp_vocab_ce")
    N, Dm, V = problem.rows, problem.d_model, problem.vocab
    c.tensor("h", h, torch.bfloat16, (N, Dm))
    c.tensor("w", w, torch.bfloat16, (V, Dm))
    c.tensor("target", target, torch.int32, (N,))
    c.tensor("loss", loss, torch.float32, (N,))
    c.tensor("lse", lse, torch.float32, (N,))
    c.tensor("dh", dh, torch.bfloat16, (N, Dm))
    if problem.head_grad:
        c.tensor("dw", dw, torch.float32, (V, Dm))
    elif dw is not None:
        raise ValueError("csbp_vocab_ce: dw must be None for a frozen head")
    c.tensor("workspace", workspace, torch.uint8, None)
    c.done()
    st = lib().csbp_vocab_ce(ctypes.byref(problem), _ptr(h), _ptr(w), _ptr(target), _ptr(loss),
                             _ptr(lse), _ptr(dh), _ptr(dw), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _check("csbp_vocab_ce", st)


class VocabCrossEntropy:
    """Owns the workspace of one LM-head cross-entropy shape.

    __call__(h, w, target) takes bf16 h [N, Dm], bf16 w [V, Dm] and int32
    target [N] on the GPU and returns (loss [N], lse [N], dh [N, Dm] bf16,
    dw [V, Dm] fp32 or None for a frozen head).
    """

    def __init__(self, rows, d_model, vocab, chunk_rows=0, head_grad=True, grad_scale=1.0,
                 device="cuda"):
        import torch
        self.problem = make_ce_problem(rows, d_model, vocab, chunk_rows, head_grad, grad_scale)
        n = ce_workspace_bytes(self.problem)
        if n == 0:
            raise CsbpError("csbp_ce_workspace_bytes", -1)
        self.ws = torch.zeros(n, dtype=torch.uint8, device=device)
        self.device = device

    def alloc_outputs(self):
        import torch
        p = self.problem
        loss = torch.empty(p.rows, dtype=torch.float32, device=self.device)
        lse = torch.empty(p.rows, dtype=torch.float32, device=self.device)
        dh = torch.empty((p.rows, p.d_model), dtype=torch.bfloat16, device=self.device)
        dw = (torch.empty((p.vocab, p.d_model), dtype=torch.float32, device=self.device)
              if p.head_grad else None)
        return loss, lse, dh, dw

    def __call__(self, h, w, target, out=None, stream=None):
        loss, lse, dh, dw = out if out is not None else self.alloc_outputs()
        vocab_ce(self.problem, h, w, target, loss, lse, dh, dw, self.ws, stream)
        return loss, lse, dh, dw

    def check(self, stream=None):
        check_status(self.ws, stream)
