"""FP8 (E4M3) K / V caches against the float64 oracle.

"FlashAttention and inference kernels", "A paged decode attention kernel (with GQA)": the KV
cache is BF16 or FP8, converted on read. The caches here are the seeded N(0, 1) draws of the
bf16 workloads quantised with one scale per tensor (decode_attention_attn_gb300.workloads);
the oracle reads the same codes and scales (its decoding is pinned in test_oracle_pins.py).
The tensor-core consumers convert every code exactly, so the bar is the one of the bf16
caches: the oracle's result on the quantised cache, not on the unquantised draw.
"""
import numpy as np
import pytest
import torch

import _parity
from decode_attention_attn_gb300 import binding, build as lib_build, workloads

W = workloads


def _check(dev, ref, ref_lse, mode, out_dtype=None, num_splits=None, plan_splits=None, where="",
           num_sms=0):
    od = out_dtype or dev.inp.wl.out_dtype
    out, lse, flags = _parity.run_gpu(dev, mode=mode, out_dtype=od, num_splits=num_splits,
                                      plan_splits=plan_splits, num_sms=num_sms)
    _parity.compare(out, ref.reshape(out.shape), od, where=f"{where} {mode} {od}")
    _parity.compare_lse(lse, ref_lse.reshape(lse.shape), where=f"{where} {mode}")
    return out, lse, flags


@pytest.fixture(scope="module")
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib_build.build()
    binding.lib()
    torch.cuda.set_device(0)


@pytest.fixture(scope="module")
def gqa32k_fp8(_gpu):
    inp = W.generate(W.GQA_32K_FP8)
    return _parity.DeviceInputs(inp), _parity.run_oracle(inp)


@pytest.fixture(scope="module")
def paged64_fp8(_gpu):
    inp = W.generate(W.PAGED_B64_FP8)
    return _parity.DeviceInputs(inp), _parity.run_oracle(inp)


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["sync", "unified", "unified_local"])
def test_gqa_32k_fp8(gqa32k_fp8, mode):
    """One KV head per split-kernel group at this size (4 packed groups would spread over 38
    CTAs each); the packed form of the same step is checked as well."""
    dev, (ref, ref_lse, ref_flag, margin) = gqa32k_fp8
    plan = binding.DecodeAttention(_parity.problem_for(dev.inp, mode=mode), 0)
    assert plan.info.kv_heads_per_group == 1
    _check(dev, ref, ref_lse, mode, out_dtype="f32", num_sms=16, where="gqa32k fp8 packed")
    out, lse, flags = _check(dev, ref, ref_lse, mode, where="gqa32k fp8")
    _check(dev, ref, ref_lse, mode, out_dtype="f32", where="gqa32k fp8 fp32-out")
    _check(dev, ref, ref_lse, mode, num_splits=16, plan_splits=16, out_dtype="f32",
           where="gqa32k fp8 S=16")
    if mode != "sync":
        assert _parity.margin_ok(margin).all()
        assert np.array_equal(flags.cpu().numpy().ravel(), ref_flag)


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["sync", "unified", "unified_local"])
def test_paged_batch64_fp8(paged64_fp8, mode):
    """The paged batch packs pairs of KV heads (256 packed groups on 152 SMs)."""
    dev, (ref, ref_lse, ref_flag, margin) = paged64_fp8
    plan = binding.DecodeAttention(_parity.problem_for(dev.inp, mode=mode), 0)
    assert plan.info.kv_heads_per_group == 2
    _check(dev, ref, ref_lse, mode, where="paged b64 fp8")
    _check(dev, ref, ref_lse, mode, out_dtype="f32", where="paged b64 fp8 fp32-out")
    _check(dev, ref, ref_lse, mode, num_splits=4, plan_splits=4, out_dtype="f32",
           where="paged b64 fp8 S=4")


EDGE_LENS = (0, 1, 15, 16, 17, 63, 64, 65, 127, 129, 1000, 1024 + 7)


@pytest.mark.gpu
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("page_size", [0, 16, 32])
def test_fp8_edge_sweep(_gpu, head_dim, group, page_size):
    """Ragged and empty sequences, tails of every stage and page position, both head dims and
    groups, contiguous and paged caches, every mode and split choice. Groups of 4 run twice:
    planned for the device (one KV head per split-kernel group at this size) and for 32 SMs,
    where the plan packs the two KV heads into one group."""
    paged = page_size > 0
    wl = W.Workload(f"fp8_edge_{head_dim}_{group}_{page_size}", len(EDGE_LENS), 2 * group, 2,
                    head_dim, "bf16", "bf16", lens=EDGE_LENS, paged=paged,
                    page_size=page_size or 16, max_seq_len=0 if paged else 1024 + 9,
                    kv_dtype="e4m3")
    inp = W.generate(wl, offset=5 * group + head_dim + page_size)
    dev = _parity.DeviceInputs(inp)
    ref, ref_lse, _, _ = _parity.run_oracle(inp)
    for sms in ((0, 32) if group == 4 else (0,)):
        packed = binding.DecodeAttention(_parity.problem_for(inp, num_sms=sms), 0)
        assert packed.info.kv_heads_per_group == (2 if sms else 1)
        for i, mode in enumerate(("sync", "unified", "unified_local")):
            for ns in ((0, 3), (1, 7), (0, 2))[i]:
                for od in ("bf16", "f32"):
                    _check(dev, ref, ref_lse, mode, out_dtype=od, num_splits=ns, plan_splits=ns,
                           num_sms=sms, where=f"fp8 edge d{head_dim} G{group} page={page_size} "
                                              f"S={ns} sms={sms}")


@pytest.mark.gpu
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("page_size", [0, 16])
def test_fp8_group4_odd_kv_heads(_gpu, head_dim, page_size):
    """Groups of 4 query heads over an odd number of KV heads: the last KV head has no partner,
    so the plan keeps one KV head per group (the packed pairs cover an even count)."""
    paged = page_size > 0
    wl = W.Workload(f"fp8_odd_{head_dim}_{page_size}", 3, 12, 3, head_dim, "bf16", "bf16",
                    lens=(1000, 65, 0), paged=paged, page_size=page_size or 16,
                    max_seq_len=0 if paged else 1030, kv_dtype="e4m3")
    inp = W.generate(wl, offset=11 + head_dim + page_size)
    dev = _parity.DeviceInputs(inp)
    ref, ref_lse, _, _ = _parity.run_oracle(inp)
    for mode in ("sync", "unified", "unified_local"):
        for ns in (0, 3):
            _check(dev, ref, ref_lse, mode, out_dtype="f32", num_splits=ns, plan_splits=ns,
                   where=f"fp8 odd kv heads d{head_dim} page={page_size} S={ns}")


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["unified", "unified_local"])
def test_fp8_forced_fallback(_gpu, mode):
    """A narrow range flags every row: the recompute (or the split-local switch) runs over
    the FP8 tiles, with the same flags as the oracle's."""
    wl = W.GQA_32K_FP8.replace(name="fp8_forced", seq_len=5000, mode=mode)
    inp = W.generate(wl, offset=9)
    dev = _parity.DeviceInputs(inp)
    phi, lo, hi = 0.0, -0.25, 0.25
    ref, ref_lse, ref_flag, margin = _parity.run_oracle(inp, phi=phi, lo=lo, hi=hi)
    assert ref_flag.all() and _parity.margin_ok(margin).all()
    for sms in (0, 16):   # one KV head per group, then packed pairs (planned for 16 SMs)
        attn = binding.DecodeAttention(
            _parity.problem_for(inp, mode=mode, phi=phi, lo=lo, hi=hi, num_sms=sms), 0)
        assert attn.info.kv_heads_per_group == (2 if sms else 1)
        out, lse, flags, st = _parity.run_gpu(dev, want_stats=True, attn=attn)
        where = f"fp8 forced fallback sms={sms}"
        _parity.compare(out, ref.reshape(out.shape), "bf16", where=where)
        _parity.compare_lse(lse, ref_lse.reshape(lse.shape), where=where)
        assert flags.cpu().numpy().all() and st.rows_flagged == 32


@pytest.mark.gpu
def test_fp8_extreme_codes(_gpu):
    """Caches made of the format's corner codes: zeros of both signs, the subnormals, the
    smallest normal and the largest value 448, with scales far from 1."""
    wl = W.Workload("fp8_codes", 2, 8, 2, 128, "bf16", "f32", lens=(300, 77), kv_dtype="e4m3")
    inp = W.generate(wl, offset=3)
    g = torch.Generator().manual_seed(77)
    corner = torch.tensor([0x00, 0x80, 0x01, 0x81, 0x07, 0x87, 0x08, 0x88, 0x7E, 0xFE, 0x38],
                          dtype=torch.uint8)
    for t in (inp.k_cache, inp.v_cache):
        pick = torch.randint(0, corner.numel(), t.shape, generator=g)
        keep = torch.rand(t.shape, generator=g) < 0.5
        t.copy_(torch.where(keep, t, corner[pick]))
    inp.k_scale, inp.v_scale = 2.0 ** -8 * 3, 2.0 ** -9 * 0.7   # |k| <= 5.25, |v| <= 0.62
    dev = _parity.DeviceInputs(inp)
    ref, ref_lse, _, _ = _parity.run_oracle(inp)
    for mode in ("sync", "unified", "unified_local"):
        _check(dev, ref, ref_lse, mode, out_dtype="f32", where="fp8 corner codes")


@pytest.mark.gpu
def test_fp8_cache_as_float8_tensor(_gpu):
    """DecodeAttention accepts the cache as torch.float8_e4m3fn as well as its bytes."""
    inp = W.generate(W.Workload("fp8_view", 1, 4, 1, 64, "bf16", "f32", seq_len=333,
                                kv_dtype="e4m3"))
    dev = _parity.DeviceInputs(inp)
    ref, _, _, _ = _parity.run_oracle(inp)
    attn = binding.DecodeAttention(_parity.problem_for(inp, mode="sync"), 0)
    out, _, _ = attn.run(dev.q, dev.k.view(torch.float8_e4m3fn), dev.v.view(torch.float8_e4m3fn),
                         None, dev.sl, inp.wl.scale)
    torch.cuda.synchronize()
    _parity.compare(out, ref.reshape(out.shape), "f32", where="float8 view")
