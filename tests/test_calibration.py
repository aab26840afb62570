"""Calibration of phi: the logit histogram (GPU) and the host-side choice of phi.

"FlashDecoding++: Faster Large Language Model Inference on GPUs", "The Overflow and Precision
Problem: Choosing phi" and Fig. 5: profile the scaled logits as a histogram, take the range
holding more than 99.99% of them, and set phi to its lower bound; a range too wide for one
constant (OPT-6.7B) means the unified max is not used.

The CPU tests pin decode_attn_choose_phi to order statistics of the data (the first value
that may not be dropped from either tail fixes the covered bins) and to a small histogram
worked by hand. The GPU tests compare the device histogram bin by bin with one built from
the float64 logits of the oracle, then run the unified softmax with the phi read off it.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from decode_attention_attn_gb300 import binding, workloads

import _parity

W = workloads


# ---- host: decode_attn_choose_phi ---------------------------------------------------------
def _bin_indices(x, lo, hi, nbins):
    """Histogram slot of each value in float64: 0 below lo, 1 + i for bin i, nbins + 1 at
    or above hi (the layout the library documents)."""
    w = (hi - lo) / nbins
    idx = np.floor((np.asarray(x, np.float64) - lo) / w)
    return np.where(idx < 0, 0, np.where(idx >= nbins, nbins + 1, idx + 1)).astype(np.int64)


def _histogram(x, lo, hi, nbins):
    return np.bincount(_bin_indices(x, lo, hi, nbins), minlength=nbins + 2)


def test_choose_phi_on_a_hand_worked_histogram():
    # 4 bins of width 1 over [0, 4); 1 value below, bins 2 / 10 / 10 / 3, none above: 26.
    counts = [1, 2, 10, 10, 3, 0]
    # coverage 0.8: at most floor(0.1 * 26) = 2 values may go on each side; the lower tail
    # (1 below, then bin 0 of 2 -> 3) keeps bin 0; the upper tail (bin 3 of 3) keeps bin 3.
    assert binding.decode_attn_choose_phi(counts, 0.0, 4.0, 0.8) == (0.0, 0.0, 4.0, True)
    # coverage 0.5: 6 per side: 1 + 2 = 3 dropped below (bin 1 starts the range), 3 above
    # (bin 2 ends it): [1, 3), phi = 1.
    assert binding.decode_attn_choose_phi(counts, 0.0, 4.0, 0.5) == (1.0, 1.0, 3.0, True)
    # the same range, wider than allowed: reported, with applies False
    assert binding.decode_attn_choose_phi(counts, 0.0, 4.0, 0.5, max_width=1.5) == \
        (1.0, 1.0, 3.0, False)
    # coverage 1: nothing may be dropped, and one value lies below the histogram's range
    with pytest.raises(binding.DecodeAttnError) as e:
        binding.decode_attn_choose_phi(counts, 0.0, 4.0, 1.0)
    assert e.value.code == -8   # DA_ERR_HISTOGRAM_RANGE


@pytest.mark.parametrize("coverage", [0.9999, 0.999, 0.95, 1.0])
def test_choose_phi_matches_order_statistics(coverage):
    """With k = floor((1 - coverage) N / 2) values allowed out per side, the sorted value
    s[k] must be kept, so the range starts at the edge of its bin, and ends at the top edge
    of the bin of s[N - 1 - k]."""
    rng = np.random.default_rng(41)
    x = rng.standard_normal(200_001) * 1.3 + 0.4
    x[:7] = [-5.5, -5.2, 6.0, 6.4, 0.0, 1e-9, 3.7]   # a few in the tails
    lo, hi, nbins = -8.0, 8.0, 1600
    w = (hi - lo) / nbins
    phi, x_lo, x_hi, applies = binding.decode_attn_choose_phi(
        _histogram(x, lo, hi, nbins), lo, hi, coverage)
    assert applies
    s = np.sort(x)
    k = int(math.floor((1.0 - coverage) * x.size / 2.0))
    want_lo = lo + math.floor((s[k] - lo) / w) * w
    want_hi = lo + (math.floor((s[x.size - 1 - k] - lo) / w) + 1) * w
    # bin edges rounded outwards to fp32
    assert want_lo - 1e-6 <= x_lo <= want_lo and want_hi <= x_hi <= want_hi + 1e-6
    assert phi == x_lo
    kept = np.count_nonzero((x >= x_lo) & (x < x_hi))
    assert kept >= coverage * x.size
    # the range is the narrowest bin-aligned one: one bin less on either side drops too many
    assert np.count_nonzero(x < x_lo + w - 1e-9) > k
    assert np.count_nonzero(x >= x_hi - w + 1e-9) > k


def test_choose_phi_flags_a_wide_range():
    """Fig. 5's OPT-6.7B case: logits over hundreds of units do not fit one constant."""
    rng = np.random.default_rng(42)
    x = rng.uniform(-400.0, 300.0, 50_000)
    phi, x_lo, x_hi, applies = binding.decode_attn_choose_phi(
        _histogram(x, -512.0, 512.0, 1024), -512.0, 512.0, 0.9999, max_width=60.0)
    assert not applies and x_hi - x_lo > 600.0 and phi == x_lo


def test_choose_phi_rejects_bad_arguments():
    counts = [0, 5, 5, 0]
    for args in [(counts, 1.0, 1.0, 0.9), (counts, 0.0, 1.0, 0.0), (counts, 0.0, 1.0, 1.5),
                 (counts, 0.0, float("nan"), 0.9), ([0, 0, 0, 0], 0.0, 1.0, 0.9)]:
        with pytest.raises(binding.DecodeAttnError) as e:
            binding.decode_attn_choose_phi(*args)
        assert e.value.code == -1
    with pytest.raises(binding.DecodeAttnError):
        binding.decode_attn_choose_phi(counts, 0.0, 1.0, 0.9, max_width=0.0)
    with pytest.raises(ValueError):
        binding.decode_attn_choose_phi([1], 0.0, 1.0)
    # the histogram's top slot counts values at or above hi: more than a tail there fails
    with pytest.raises(binding.DecodeAttnError) as e:
        binding.decode_attn_choose_phi([0, 5, 5, 3], 0.0, 1.0, 0.9)
    assert e.value.code == -8


# ---- GPU: decode_attn_logit_histogram -------------------------------------------------------
HIST_LO, HIST_HI, HIST_BINS = -6.0, 6.0, 480

# The pages' workloads, and small cases for the other groups, head dims and storage types,
# with ragged and empty sequences
CALIB_CASES = [
    W.TINY, W.MHA_4K, W.GQA_32K, W.PAGED_B64,
    W.Workload("calib_g8_d64_bf16_paged", 3, 16, 2, 64, "bf16", "bf16", lens=(700, 1, 33),
               paged=True, page_size=32),
    W.Workload("calib_g2_d64_f16", 3, 4, 2, 64, "f16", "f16", lens=(0, 1029, 77)),
    W.Workload("calib_g8_d128_f32", 2, 8, 1, 128, "f32", "f32", lens=(513, 1)),
    W.Workload("calib_g4_d64_bf16", 2, 8, 2, 64, "bf16", "bf16", lens=(2000, 999)),
    # FP8 (E4M3) caches: the logits of the codes times k_scale
    W.GQA_32K_FP8,
    W.Workload("calib_g8_d64_e4m3_paged", 3, 16, 2, 64, "bf16", "bf16", lens=(700, 1, 33),
               paged=True, page_size=32, kv_dtype="e4m3"),
]


def _oracle_logits(inp):
    bt = None if inp.block_table is None else inp.block_table.numpy()
    return oracle.logits(_parity.oracle_shape(inp), W.bits(inp.q), W.bits(inp.k_cache), bt,
                         inp.seq_lens.numpy(), inp.wl.scale)


def _device_histogram(attn, dev, scale, lo=HIST_LO, hi=HIST_HI, nbins=HIST_BINS, counts=None,
                      calls=1):
    if counts is None:
        counts = torch.zeros(nbins + 2, dtype=torch.int64, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(calls):
        binding.decode_attn_logit_histogram(
            attn.plan, dev.q.data_ptr(), dev.k.data_ptr(),
            None if dev.bt is None else dev.bt.data_ptr(), dev.sl.data_ptr(), scale, lo, hi,
            nbins, counts.data_ptr(), stream)
    torch.cuda.synchronize()
    return counts


def _check_counts(got, x, lo=HIST_LO, hi=HIST_HI, nbins=HIST_BINS, reps=1):
    """Bin by bin: the device places every logit away from a bin edge where the float64
    logit falls. A logit within tol of an edge may fall on either side: tol bounds the
    error of the fp32 dot product (a dozen roundings of partial sums no larger than
    scale * sum_i |q_i k_i|, about 7 for these N(0, 1) inputs) and of the fp32 bin index."""
    got = np.asarray(got, np.int64)
    tol = 2e-5 * (1.0 + np.abs(x))
    b_lo = _bin_indices(x - tol, lo, hi, nbins)
    b_hi = _bin_indices(x + tol, lo, hi, nbins)
    assert np.all(b_hi - b_lo <= 1)       # tol is far below a bin width
    sure = b_lo == b_hi
    certain = np.bincount(b_lo[sure], minlength=nbins + 2) * reps
    # an edge value may land in either of its two slots
    possible = (np.bincount(b_lo[~sure], minlength=nbins + 2) +
                np.bincount(b_hi[~sure], minlength=nbins + 2)) * reps
    assert got.sum() == x.size * reps, (got.sum(), x.size * reps)
    assert np.all(got >= certain), np.nonzero(got < certain)
    assert np.all(got <= certain + possible), np.nonzero(got > certain + possible)
    assert (~sure).sum() <= max(10, x.size // 200)   # edge values are rare
    return sure


@pytest.mark.gpu
@pytest.mark.parametrize("wl", CALIB_CASES, ids=[w.name for w in CALIB_CASES])
def test_logit_histogram_matches_oracle(wl):
    inp = W.generate(wl)
    dev = _parity.DeviceInputs(inp)
    attn = binding.DecodeAttention(_parity.problem_for(inp, mode="sync"), 0)
    counts = _device_histogram(attn, dev, wl.scale).cpu().numpy()
    x = _oracle_logits(inp)
    _check_counts(counts, x)


@pytest.mark.gpu
def test_logit_histogram_accumulates_and_counts_the_tails():
    """Two calls add up; a narrow [lo, hi) puts the rest in the two outer slots; a single
    bin holds everything in range."""
    inp = W.generate(W.PAGED_B64.replace(batch=8))
    dev = _parity.DeviceInputs(inp)
    attn = binding.DecodeAttention(_parity.problem_for(inp, mode="sync"), 0)
    x = _oracle_logits(inp)
    counts = _device_histogram(attn, dev, inp.wl.scale, calls=2).cpu().numpy()
    _check_counts(counts, x, reps=2)
    counts = _device_histogram(attn, dev, inp.wl.scale, lo=-0.5, hi=0.25, nbins=3).cpu().numpy()
    _check_counts(counts, x, lo=-0.5, hi=0.25, nbins=3)
    counts = _device_histogram(attn, dev, inp.wl.scale, lo=-1.0, hi=1.0, nbins=1).cpu().numpy()
    _check_counts(counts, x, lo=-1.0, hi=1.0, nbins=1)


@pytest.mark.gpu
def test_logit_histogram_skips_pages_outside_the_pool():
    """A block-table entry outside the pool: its page's tokens are not counted, while the other
    pages of the same 64-token item are. The page is each sequence's last, so the expected
    counts are the oracle's over the sequences cut at that page's first token."""
    wl = W.Workload("calib_bad_pages", 3, 8, 2, 128, "bf16", "bf16", lens=(200, 77, 1000),
                    paged=True, page_size=16)
    inp = W.generate(wl, offset=4)
    dev = _parity.DeviceInputs(inp)
    attn = binding.DecodeAttention(_parity.problem_for(inp, mode="sync"), 0)
    cut = inp.seq_lens.clone()
    for b, n in enumerate(inp.seq_lens.tolist()):
        last = (n - 1) // wl.page_size
        dev.bt[b, last] = inp.num_physical_blocks + 3 if b != 1 else -7
        cut[b] = last * wl.page_size
    counts = _device_histogram(attn, dev, wl.scale).cpu().numpy()
    bt = inp.block_table.numpy()
    x = oracle.logits(_parity.oracle_shape(inp), W.bits(inp.q), W.bits(inp.k_cache), bt,
                      cut.numpy(), wl.scale)
    _check_counts(counts, x)


@pytest.mark.gpu
def test_logit_histogram_rejects_bad_arguments():
    inp = W.generate(W.TINY)
    dev = _parity.DeviceInputs(inp)
    attn = binding.DecodeAttention(_parity.problem_for(inp, mode="sync"), 0)
    counts = torch.zeros(8, dtype=torch.int64, device="cuda")
    L = binding.lib()
    base = [attn.plan, dev.q.data_ptr(), dev.k.data_ptr(), None, dev.sl.data_ptr(), 0.125]
    for lo, hi, nbins in [(1.0, 1.0, 6), (0.0, 1.0, 0), (0.0, 1.0, binding.MAX_HIST_BINS + 1),
                          (0.0, float("inf"), 6)]:
        assert L.decode_attn_logit_histogram(*base, lo, hi, nbins, counts.data_ptr(), None) == -1
    # a block table for a contiguous cache, a misaligned K pointer
    assert L.decode_attn_logit_histogram(attn.plan, dev.q.data_ptr(), dev.k.data_ptr(),
                                         dev.sl.data_ptr(), dev.sl.data_ptr(), 0.125, 0.0, 1.0,
                                         6, counts.data_ptr(), None) == -1
    assert L.decode_attn_logit_histogram(attn.plan, dev.q.data_ptr(), dev.k.data_ptr() + 4,
                                         None, dev.sl.data_ptr(), 0.125, 0.0, 1.0, 6,
                                         counts.data_ptr(), None) == -1
    torch.cuda.synchronize()
    assert int(counts.sum()) == 0   # nothing ran


@pytest.mark.gpu
@pytest.mark.parametrize("wl", [W.GQA_32K, W.PAGED_B64], ids=["gqa32k", "paged"])
@pytest.mark.parametrize("mode", ["unified", "unified_local"])
def test_calibrated_phi_drives_the_unified_softmax(wl, mode):
    """Calibrate on two draws of the workload, read phi off the histogram (coverage 99.99%),
    then run the unified softmax on a third draw with phi and the covered range as the flag
    interval: every row with a logit outside [x_lo, x_hi] (from the oracle's float64
    logits) is flagged and no other, and the outputs match the oracle."""
    counts = None
    for offset in (0, 1):
        inp = W.generate(wl, offset)
        dev = _parity.DeviceInputs(inp)
        attn = binding.DecodeAttention(_parity.problem_for(inp, mode="sync"), 0)
        counts = _device_histogram(attn, dev, wl.scale, counts=counts)
    counts = counts.cpu().numpy()
    phi, x_lo, x_hi, applies = binding.decode_attn_choose_phi(counts, HIST_LO, HIST_HI, 0.9999,
                                                              max_width=64.0)
    assert applies and phi == x_lo
    # the N(0, 1)-like logits of these workloads: the same range the oracle's logits give
    x01 = np.concatenate([_oracle_logits(W.generate(wl, o)) for o in (0, 1)])
    ref = binding.decode_attn_choose_phi(_histogram(x01, HIST_LO, HIST_HI, HIST_BINS),
                                         HIST_LO, HIST_HI, 0.9999)
    w = (HIST_HI - HIST_LO) / HIST_BINS
    assert abs(x_lo - ref[1]) <= w + 1e-6 and abs(x_hi - ref[2]) <= w + 1e-6

    inp = W.generate(wl, 2)
    dev = _parity.DeviceInputs(inp)
    lo, hi = 0.0, float(np.float32(x_hi) - np.float32(phi))
    res = _parity.run_gpu(dev, mode=mode, out_dtype="f32", phi=phi, lo=lo, hi=hi)
    out, flags = res[0], res[2]
    x = _oracle_logits(inp)
    # the expected flag of each row, from its float64 logits; rows with a logit within tol
    # of a bound (where the device's x - phi may fall either way: the tensor-core path holds
    # q * scale as a pair of bf16 values, about 16 significant bits) are not compared
    tol = 1e-4 * (1.0 + np.abs(x))
    out_sure = (x + tol < x_lo) | (x - tol > x_lo + hi)
    near = ~out_sure & ((x - tol < x_lo) | (x + tol > x_lo + hi))
    B, Hq = wl.batch, wl.num_q_heads
    lens = inp.seq_lens.numpy().astype(np.int64)
    row = np.repeat(np.arange(B * Hq), np.repeat(lens, Hq))
    want = np.bincount(row, weights=out_sure, minlength=B * Hq) > 0
    unsure = (np.bincount(row, weights=near, minlength=B * Hq) > 0) & ~want
    got = flags.cpu().numpy().reshape(-1).astype(bool)
    assert np.array_equal(got[~unsure], want[~unsure])
    assert want.sum() > 0          # long rows: some logits fall outside the 99.99% range
    ref_out = _parity.run_oracle(inp, phi=phi, lo=lo, hi=hi)[0]
    _parity.compare(out, ref_out, "f32", where=f"{wl.name} {mode} calibrated phi")
