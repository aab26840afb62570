"""Thin Python binding of the C ABI in include/decode_attn.h (argument marshalling only).

Every step of the computation runs in the CUDA library libdecode_attn.so; this module
only converts arguments and raises DecodeAttnError for non-zero return codes. PyTorch is
used for device memory and streams. If the library has not been built this module raises
on first use: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

from . import build as _build

DA_F32, DA_F16, DA_BF16 = 0, 1, 2
DA_SOFTMAX_SYNC, DA_SOFTMAX_UNIFIED, DA_SOFTMAX_UNIFIED_LOCAL = 0, 1, 2
ERRORS = {0: "DA_OK", -1: "DA_ERR_INVALID_ARG", -2: "DA_ERR_UNSUPPORTED",
          -3: "DA_ERR_WORKSPACE_TOO_SMALL", -4: "DA_ERR_BAD_BLOCK_TABLE", -5: "DA_ERR_CUDA",
          -6: "DA_ERR_DEVICE_TIMEOUT", -7: "DA_ERR_BAD_SEQ_LEN", -8: "DA_ERR_HISTOGRAM_RANGE",
          -9: "DA_ERR_RANGE_TOO_WIDE"}
DA_ERR_RANGE_TOO_WIDE = -9
MAX_HIST_BINS = 32768
DTYPE_CODES = {"f32": DA_F32, "f16": DA_F16, "bf16": DA_BF16}
MODE_CODES = {"sync": DA_SOFTMAX_SYNC, "unified": DA_SOFTMAX_UNIFIED,
              "unified_local": DA_SOFTMAX_UNIFIED_LOCAL}


class DecodeAttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {ERRORS.get(code, code)}: {decode_attn_strerror(code)}")


class da_problem(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int),
        ("num_q_heads", ctypes.c_int),
        ("num_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("paged", ctypes.c_int),
        ("page_size", ctypes.c_int),
        ("max_blocks_per_seq", ctypes.c_int),
        ("num_physical_blocks", ctypes.c_int),
        ("max_seq_len", ctypes.c_int),
        ("qkv_dtype", ctypes.c_int),
        ("out_dtype", ctypes.c_int),
        ("mode", ctypes.c_int),
        ("unified_max", ctypes.c_float),
        ("range_lo", ctypes.c_float),
        ("range_hi", ctypes.c_float),
        ("validate", ctypes.c_int),
        ("num_sms", ctypes.c_int),
        ("kv_fp8", ctypes.c_int),
        ("k_scale", ctypes.c_float),
        ("v_scale", ctypes.c_float),
        ("debug_stall_stage", ctypes.c_int),
    ]


class da_plan_info(ctypes.Structure):
    _fields_ = [
        ("grid_ctas", ctypes.c_int),
        ("num_splits", ctypes.c_int),
        ("unit_tokens", ctypes.c_int),
        ("stage_tokens", ctypes.c_int),
        ("stages", ctypes.c_int),
        ("recompute_splits", ctypes.c_int),
        ("max_splits", ctypes.c_int),
        ("workspace_bytes", ctypes.c_size_t),
        ("smem_bytes", ctypes.c_size_t),
        ("split_tokens", ctypes.c_int),
        ("split_tokens_min", ctypes.c_int),
        ("kv_heads_per_group", ctypes.c_int),
    ]


class da_stats(ctypes.Structure):
    _fields_ = [
        ("grid_ctas", ctypes.c_int),
        ("num_splits", ctypes.c_int),
        ("rows_flagged", ctypes.c_longlong),
        ("splits_flagged", ctypes.c_longlong),
        ("recompute_launched", ctypes.c_int),
        ("split_tokens", ctypes.c_int),
        ("split_tokens_min", ctypes.c_int),
    ]


class da_run_args(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p),
        ("k_cache", ctypes.c_void_p),
        ("v_cache", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("seq_lens", ctypes.c_void_p),
        ("scale", ctypes.c_float),
        ("num_splits", ctypes.c_int),
        ("out", ctypes.c_void_p),
        ("out_lse", ctypes.c_void_p),
        ("row_flags", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("cuda_stream", ctypes.c_void_p),
        ("stats", ctypes.POINTER(da_stats)),
        ("split_event_begin", ctypes.c_void_p),
        ("split_event_end", ctypes.c_void_p),
    ]


_lib = None
P = ctypes.c_void_p


def library_path() -> str:
    return _build.LIB


def lib():
    """Load libdecode_attn.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(path)
        L.decode_attn_plan.argtypes = [ctypes.POINTER(da_problem), ctypes.c_int,
                                       ctypes.POINTER(P), ctypes.POINTER(ctypes.c_size_t)]
        L.decode_attn_plan_info.argtypes = [P, ctypes.POINTER(da_plan_info)]
        L.decode_attn_workspace_init.argtypes = [P, P, ctypes.c_size_t, P]
        L.decode_attn_run.argtypes = [P, P, P, P, P, P, ctypes.c_float, ctypes.c_int, P, P, P,
                                      P, ctypes.c_size_t, P, ctypes.POINTER(da_stats)]
        L.decode_attn_run_ex.argtypes = [P, ctypes.POINTER(da_run_args)]
        L.decode_attn_run_static.argtypes = [P, P, P, P, P, P, ctypes.c_float, ctypes.c_int, P,
                                             P, P, P, ctypes.POINTER(da_stats)]
        L.decode_attn_check_status.argtypes = [P, P, P]
        L.decode_attn_debug_gather.argtypes = [P, P, P, P, P]
        L.decode_attn_logit_histogram.argtypes = [P, P, P, P, P, ctypes.c_float, ctypes.c_float,
                                                  ctypes.c_float, ctypes.c_int, P, P]
        F = ctypes.POINTER(ctypes.c_float)
        L.decode_attn_choose_phi.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), ctypes.c_int,
                                             ctypes.c_float, ctypes.c_float, ctypes.c_double,
                                             ctypes.c_float, F, F, F]
        L.decode_attn_destroy.argtypes = [P]
        L.decode_attn_destroy.restype = None
        L.decode_attn_strerror.argtypes = [ctypes.c_int]
        L.decode_attn_strerror.restype = ctypes.c_char_p
        L.decode_attn_abi_version.argtypes = []
        for name in ("decode_attn_plan", "decode_attn_plan_info", "decode_attn_workspace_init",
                     "decode_attn_run", "decode_attn_run_ex", "decode_attn_run_static",
                     "decode_attn_check_status",
                     "decode_attn_debug_gather", "decode_attn_logit_histogram",
                     "decode_attn_choose_phi",
                     "decode_attn_abi_version"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(rc: int, where: str):
    if rc != 0:
        raise DecodeAttnError(rc, where)


def header_symbols() -> list:
    """Entry points declared in include/decode_attn.h."""
    path = os.path.join(_build.INCLUDE, "decode_attn.h")
    with open(path) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(decode_attn_[a-z_]+)\s*\(", text)))


# ---- the C entry points, same names ---------------------------------------------------------
def decode_attn_abi_version() -> int:
    return lib().decode_attn_abi_version()


def decode_attn_strerror(code: int) -> str:
    return lib().decode_attn_strerror(code).decode()


def decode_attn_plan(problem: da_problem, num_splits: int = 0):
    """Returns (plan handle, workspace bytes)."""
    plan = P()
    ws = ctypes.c_size_t()
    _check(lib().decode_attn_plan(ctypes.byref(problem), num_splits, ctypes.byref(plan),
                                  ctypes.byref(ws)), "decode_attn_plan")
    return plan, ws.value


def decode_attn_plan_info(plan) -> da_plan_info:
    info = da_plan_info()
    _check(lib().decode_attn_plan_info(plan, ctypes.byref(info)), "decode_attn_plan_info")
    return info


def decode_attn_workspace_init(plan, workspace: int, workspace_bytes: int, stream: int = 0):
    _check(lib().decode_attn_workspace_init(plan, workspace, workspace_bytes, stream or None),
           "decode_attn_workspace_init")


def decode_attn_run(plan, q: int, k_cache: int, v_cache: int, block_table: Optional[int],
                    seq_lens: int, scale: float, num_splits: int, out: int,
                    out_lse: Optional[int], row_flags: Optional[int], workspace: int,
                    workspace_bytes: int, stream: int = 0, want_stats: bool = False):
    """Pointers are integers (device addresses). Returns da_stats when want_stats."""
    st = da_stats() if want_stats else None
    _check(lib().decode_attn_run(plan, q, k_cache, v_cache, block_table or None, seq_lens,
                                 scale, num_splits, out, out_lse or None, row_flags or None,
                                 workspace, workspace_bytes, stream or None,
                                 ctypes.byref(st) if st is not None else None),
           "decode_attn_run")
    return st


def decode_attn_run_ex(plan, args: da_run_args):
    _check(lib().decode_attn_run_ex(plan, ctypes.byref(args)), "decode_attn_run_ex")


def decode_attn_run_static(plan, q: int, k_cache: int, v_cache: int, block_table: Optional[int],
                           seq_lens: int, scale: float, num_splits: int, out: int,
                           out_lse: Optional[int], row_flags: Optional[int], stream: int = 0,
                           want_stats: bool = False):
    """decode_attn_run on the library's fixed per-device scratch: for callers that cannot
    allocate a workspace. Pointers are integers (device addresses); nothing is allocated
    here either. Returns da_stats when want_stats."""
    st = da_stats() if want_stats else None
    _check(lib().decode_attn_run_static(plan, q, k_cache, v_cache, block_table or None,
                                        seq_lens, scale, num_splits, out, out_lse or None,
                                        row_flags or None, stream or None,
                                        ctypes.byref(st) if st is not None else None),
           "decode_attn_run_static")
    return st


def decode_attn_check_status(plan, workspace: int, stream: int = 0):
    _check(lib().decode_attn_check_status(plan, workspace, stream or None),
           "decode_attn_check_status")


def decode_attn_debug_gather(plan, block_table: Optional[int], seq_lens: int, offsets_out: int,
                             stream: int = 0):
    _check(lib().decode_attn_debug_gather(plan, block_table or None, seq_lens, offsets_out,
                                          stream or None), "decode_attn_debug_gather")


def decode_attn_logit_histogram(plan, q: int, k_cache: int, block_table: Optional[int],
                                seq_lens: int, scale: float, lo: float, hi: float, nbins: int,
                                counts: int, stream: int = 0):
    """Accumulate the histogram of one step's scaled logits into the device uint64 buffer
    `counts` ([nbins + 2]: below lo, the nbins bins of [lo, hi), at or above hi)."""
    _check(lib().decode_attn_logit_histogram(plan, q, k_cache, block_table or None, seq_lens,
                                             scale, lo, hi, nbins, counts, stream or None),
           "decode_attn_logit_histogram")


def decode_attn_choose_phi(counts, lo: float, hi: float, coverage: float = 0.9999,
                           max_width: float = float("inf")):
    """(phi, x_lo, x_hi, applies) from a host histogram (a sequence of nbins + 2 counts).
    applies is False when the covered range is wider than max_width (the unified max should
    not be used for this data); other failures raise."""
    n = len(counts) - 2
    if n < 1:
        raise ValueError("a histogram holds at least one bin and the two outer counts")
    arr = (ctypes.c_ulonglong * len(counts))(*[int(c) for c in counts])
    phi, x_lo, x_hi = ctypes.c_float(), ctypes.c_float(), ctypes.c_float()
    rc = lib().decode_attn_choose_phi(arr, n, lo, hi, coverage, max_width, ctypes.byref(phi),
                                      ctypes.byref(x_lo), ctypes.byref(x_hi))
    if rc not in (0, DA_ERR_RANGE_TOO_WIDE):
        _check(rc, "decode_attn_choose_phi")
    return phi.value, x_lo.value, x_hi.value, rc == 0


def decode_attn_destroy(plan):
    lib().decode_attn_destroy(plan)


def make_problem(*, batch, num_q_heads, num_kv_heads, head_dim, qkv_dtype, out_dtype, paged=False,
                 page_size=16, max_blocks_per_seq=0, num_physical_blocks=0, max_seq_len=0,
                 mode="sync", unified_max=0.0, range_lo=-64.0, range_hi=64.0, validate=False,
                 num_sms=0, kv_dtype=None, k_scale=1.0, v_scale=1.0,
                 debug_stall_stage=0) -> da_problem:
    """kv_dtype=None: K / V stored as qkv_dtype; "e4m3": an FP8 cache of codes standing for
    code * k_scale and code * v_scale (q stays qkv_dtype, which must be bf16)."""
    if kv_dtype not in (None, qkv_dtype, "e4m3"):
        raise ValueError("K / V are stored as qkv_dtype or as e4m3")
    fp8 = kv_dtype == "e4m3"
    return da_problem(batch, num_q_heads, num_kv_heads, head_dim, int(bool(paged)), page_size,
                      max_blocks_per_seq, num_physical_blocks, max_seq_len,
                      DTYPE_CODES[qkv_dtype], DTYPE_CODES[out_dtype], MODE_CODES[mode],
                      unified_max, range_lo, range_hi, int(bool(validate)), num_sms, int(fp8),
                      k_scale if fp8 else 1.0, v_scale if fp8 else 1.0, int(debug_stall_stage))


# ---- torch-facing convenience (marshalling only) -------------------------------------------
class DecodeAttention:
    """A plan plus its workspace on the current CUDA device.

    run() takes torch tensors already on the device, passes their addresses and the
    current stream to decode_attn_run, and returns (out, lse, row_flags)."""

    def __init__(self, problem: da_problem, num_splits: int = 0, device=None):
        import torch
        self.problem = problem
        self.plan, self.workspace_bytes = decode_attn_plan(problem, num_splits)
        self.info = decode_attn_plan_info(self.plan)
        from .workloads import TORCH_DTYPES
        names = {v: k for k, v in DTYPE_CODES.items()}
        self._qkv_dtype = TORCH_DTYPES[names[problem.qkv_dtype]]
        self._out_dtype = TORCH_DTYPES[names[problem.out_dtype]]
        self.device = torch.device(device) if device is not None else torch.device("cuda")
        # a zero-filled workspace needs no decode_attn_workspace_init call
        self.workspace = torch.zeros(self.workspace_bytes, dtype=torch.uint8, device=self.device)

    def __del__(self):
        plan = getattr(self, "plan", None)
        if plan is not None and _lib is not None:
            decode_attn_destroy(plan)
            self.plan = None

    def run(self, q, k_cache, v_cache, block_table, seq_lens, scale: float, num_splits: int = -1,
            out=None, out_lse=None, row_flags=None, stream=None, want_stats: bool = False,
            split_events=None):
        import torch
        pr = self.problem
        qkv = self._qkv_dtype
        # an FP8 cache holds E4M3 codes: torch.float8_e4m3fn, or their bytes as uint8
        kv_ok = (torch.uint8, torch.float8_e4m3fn) if pr.kv_fp8 else (qkv,)
        for name, t, ok in (("q", q, (qkv,)), ("k_cache", k_cache, kv_ok),
                            ("v_cache", v_cache, kv_ok)):
            if t.device.type != "cuda" or t.dtype not in ok or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous CUDA tensor of {ok}")
        if seq_lens.dtype != torch.int32 or seq_lens.device.type != "cuda":
            raise ValueError("seq_lens must be an int32 CUDA tensor")
        if block_table is not None and (block_table.dtype != torch.int32 or
                                        not block_table.is_contiguous()):
            raise ValueError("block_table must be a contiguous int32 CUDA tensor")
        B, H = pr.batch, pr.num_q_heads
        if out is None:
            out = torch.empty((B, H, pr.head_dim), dtype=self._out_dtype, device=q.device)
        if out_lse is None:
            out_lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
        if row_flags is None:
            row_flags = torch.empty((B, H), dtype=torch.uint8, device=q.device)
        s = stream if stream is not None else torch.cuda.current_stream(q.device)
        st = da_stats() if want_stats else None
        args = da_run_args(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                           None if block_table is None else block_table.data_ptr(),
                           seq_lens.data_ptr(), float(scale), num_splits, out.data_ptr(),
                           out_lse.data_ptr(), row_flags.data_ptr(), self.workspace.data_ptr(),
                           self.workspace_bytes, s.cuda_stream or None,
                           ctypes.pointer(st) if st is not None else None,
                           split_events[0].cuda_event if split_events else None,
                           split_events[1].cuda_event if split_events else None)
        decode_attn_run_ex(self.plan, args)
        if want_stats:
            return out, out_lse, row_flags, st
        return out, out_lse, row_flags
