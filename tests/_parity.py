"""Helpers shared by the parity tests: run the CUDA path and the CPU oracle on the same
seeded inputs and compare them.

Tolerance. The bar of max |error| <= 2e-3 and, per (b, h) row, ||error||_2 / ||ref||_2 <= 1e-3
(absolute when ||ref||_2 < 1e-6) applies to the kernels' FP32 result: a run with an fp32
output is compared with the unrounded float64 oracle. A 16-bit output cannot meet a 1e-3
relative bound against the exact result (rounding alone costs ~1.7e-3 in bf16), so a bf16 /
fp16 output is checked in two ways:
  - faithful rounding: |got - ref| below one ulp of the output format at ref (plus 1e-5
    absolute, for values near zero where the FP32 accumulation error exceeds the format's
    spacing);
  - the rounding mode: the kernels round their FP32 value to nearest even, so wherever the
    float64 value lies farther than the FP32 path's error bound from a rounding midpoint,
    the output must equal the float64 value rounded to nearest even, exactly. Only elements
    within that bound of a midpoint (a few percent at most) may round either way.
The log-sum-exp is an FP32 result too: it must match the oracle's within LSE_REL * max(1,
|lse|), about a hundred FP32 ulps, far below what losing any one split would change.
"""
import math

import numpy as np
import torch

import oracle
from decode_attention_attn_gb300 import binding, workloads
from decode_attention_attn_gb300.harness import DeviceInputs, problem_for  # noqa: F401

MAX_ABS = 2e-3
MAX_REL_L2 = 1e-3
# Error bound of the FP32 path, relative to |ref| + the row's RMS: the band around a rounding
# midpoint inside which a 16-bit output may round either way.
FP32_REL = 2e-5
# Largest fraction of a 16-bit output that may lie in such a band (else the check is vacuous).
MAX_MIDPOINT_FRACTION = 0.5
LSE_REL = 1e-5


def oracle_shape(inp: workloads.Inputs):
    w = inp.wl
    return oracle.make_shape(batch=w.batch, num_q_heads=w.num_q_heads,
                             num_kv_heads=w.num_kv_heads, head_dim=w.head_dim, dtype=w.dtype,
                             paged=w.paged, page_size=w.page_size,
                             max_blocks_per_seq=inp.max_blocks_per_seq,
                             max_seq_len=inp.max_seq_len,
                             num_physical_blocks=inp.num_physical_blocks, kv_dtype=w.kv_dtype,
                             k_scale=inp.k_scale, v_scale=inp.v_scale)


def run_oracle(inp: workloads.Inputs, rows=None, nthreads=None, phi=None, lo=None, hi=None):
    w = inp.wl
    bt = None if inp.block_table is None else inp.block_table.numpy()
    return oracle.decode_attn(
        oracle_shape(inp), workloads.bits(inp.q), workloads.bits(inp.k_cache),
        workloads.bits(inp.v_cache), bt, inp.seq_lens.numpy(), w.scale,
        w.phi if phi is None else phi, w.range_lo if lo is None else lo,
        w.range_hi if hi is None else hi, rows=rows,
        nthreads=oracle.host_threads() if nthreads is None else nthreads)


def run_gpu(dev: DeviceInputs, mode=None, num_splits=None, out_dtype=None, plan_splits=None,
            validate=False, want_stats=False, phi=None, lo=None, hi=None, attn=None, num_sms=0):
    inp = dev.inp
    w = inp.wl
    if attn is None:
        ns = w.num_splits if plan_splits is None else plan_splits
        attn = binding.DecodeAttention(
            problem_for(inp, mode, out_dtype, validate, phi, lo, hi, num_sms), ns)
    res = attn.run(dev.q, dev.k, dev.v, dev.bt, dev.sl, w.scale,
                   -1 if num_splits is None else num_splits, want_stats=want_stats)
    torch.cuda.synchronize()
    return res


def ulp(x: np.ndarray, out_dtype: str) -> np.ndarray:
    """Spacing of the 16-bit output format at |x| (subnormal spacing below the normal range)."""
    mant = {"bf16": 7, "f16": 10}[out_dtype]
    emin = {"bf16": -126, "f16": -14}[out_dtype]
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** emin)))
    return 2.0 ** (e - mant)


def round_nearest_even(x: np.ndarray, out_dtype: str):
    """float64 x rounded once, to nearest even, to the 16-bit format (as float64), and the
    distance of x from the nearest rounding midpoint. Exact: x / spacing is exact (a power of
    two) and np.rint rounds halves to even. Values stay far inside both formats' range."""
    x = np.asarray(x, dtype=np.float64)
    sp = ulp(x, out_dtype)
    y = x / sp
    r = np.rint(y) * sp
    mid = np.abs(np.abs(y - np.floor(y)) - 0.5) * sp
    return r, mid


def compare(out_gpu: torch.Tensor, ref: np.ndarray, out_dtype: str, where=""):
    """Assert the tolerance bar; returns (max_abs, max_rel_l2) against the unrounded oracle."""
    got = out_gpu.detach().to("cpu", torch.float64).numpy().reshape(ref.shape)
    assert np.isfinite(got).all(), f"{where}: non-finite output"
    err = got - ref
    max_abs = float(np.max(np.abs(err))) if err.size else 0.0
    rn = np.linalg.norm(ref.reshape(-1, ref.shape[-1]), axis=1)
    en = np.linalg.norm(err.reshape(-1, err.shape[-1]), axis=1)
    rel = np.where(rn < 1e-6, en, en / np.maximum(rn, 1e-300))
    max_rel = float(rel.max()) if rel.size else 0.0
    if out_dtype == "f32":
        assert max_abs <= MAX_ABS, f"{where}: max abs error {max_abs:.3e} > {MAX_ABS}"
        assert max_rel <= MAX_REL_L2, f"{where}: max row rel-L2 {max_rel:.3e} > {MAX_REL_L2}"
    else:
        bound = ulp(np.maximum(np.abs(ref), np.abs(got)), out_dtype) + 1e-5
        bad = np.abs(err) > bound
        assert not bad.any(), (f"{where}: {int(bad.sum())} elements are not a faithful "
                               f"{out_dtype} rounding (worst |err|/ulp "
                               f"{float(np.max(np.abs(err) / bound)):.3f})")
        rne, mid = round_nearest_even(ref, out_dtype)
        rms = (rn / math.sqrt(ref.shape[-1])).reshape(ref.shape[:-1] + (1,))
        band = mid <= FP32_REL * (np.abs(ref) + rms)
        frac = float(band.mean()) if band.size else 0.0
        assert frac <= MAX_MIDPOINT_FRACTION, (
            f"{where}: {frac:.3f} of the elements lie near a rounding midpoint")
        wrong = (got != rne) & ~band
        assert not wrong.any(), (f"{where}: {int(wrong.sum())} elements are not the float64 "
                                 f"result rounded to nearest even (of {band.size - int(band.sum())}"
                                 f" away from a midpoint)")
    return max_abs, max_rel


def compare_lse(lse_gpu: torch.Tensor, ref_lse: np.ndarray, where="", tol=LSE_REL):
    """The natural-log LSE against the oracle's: -inf exactly where the oracle has it, else
    within tol * max(1, |lse|)."""
    got = lse_gpu.detach().cpu().numpy().astype(np.float64).reshape(ref_lse.shape)
    inf = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(got), inf), f"{where}: -inf pattern of lse differs"
    if (~inf).any():
        d = np.abs(got[~inf] - ref_lse[~inf])
        lim = tol * np.maximum(1.0, np.abs(ref_lse[~inf]))
        assert np.all(d <= lim), f"{where}: lse error {d.max():.3e} (bound {lim.min():.3e})"
    return float(np.max(np.abs(got[~inf] - ref_lse[~inf]))) if (~inf).any() else 0.0


def margin_ok(margin: np.ndarray, eps=1e-3):
    """Rows whose flag decision is far from flipping (GPU logits are FP32, oracle's float64)."""
    return margin > eps
