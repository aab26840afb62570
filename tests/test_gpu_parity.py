"""GPU parity: the CUDA path (through the C ABI) against the float64 CPU oracle.

All inputs are seeded and synthetic (decode_attention_attn_gb300.workloads). Outputs are
compared element by element under the bar in _parity.py; integer results (gather offsets,
row flags) are compared bit-exactly.
"""
import math

import numpy as np
import pytest
import torch

import _parity
import oracle
from decode_attention_attn_gb300 import binding, build as lib_build, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib_build.build()
    binding.lib()
    torch.cuda.set_device(0)


def _check(dev, ref, ref_lse, mode, out_dtype=None, num_splits=None, plan_splits=None, where=""):
    w = dev.inp.wl
    od = out_dtype or w.out_dtype
    out, lse, flags = _parity.run_gpu(dev, mode=mode, out_dtype=od, num_splits=num_splits,
                                      plan_splits=plan_splits)
    _parity.compare(out, ref.reshape(out.shape), od, where=f"{where} {mode} {od}")
    _parity.compare_lse(lse, ref_lse.reshape(lse.shape), where=f"{where} {mode}")
    return out, lse, flags


# ---- the five named workloads at full size ------------------------------------------------
def test_tiny_fp32_four_splits():
    inp = workloads.generate(workloads.TINY)
    dev = _parity.DeviceInputs(inp)
    ref, ref_lse, ref_flag, margin = _parity.run_oracle(inp)
    for mode in ("sync", "unified"):
        for ns in (None, 0, 1, 4):
            _check(dev, ref, ref_lse, mode, num_splits=ns, where=f"tiny splits={ns}")


def test_mha_fp16_split256():
    inp = workloads.generate(workloads.MHA_4K)
    dev = _parity.DeviceInputs(inp)
    ref, ref_lse, _, _ = _parity.run_oracle(inp)
    for mode in ("sync", "unified"):
        _check(dev, ref, ref_lse, mode, where="mha fp16 S=16")
        _check(dev, ref, ref_lse, mode, out_dtype="f32", where="mha fp32-out")
        _check(dev, ref, ref_lse, mode, num_splits=0, where="mha balanced")


@pytest.fixture(scope="module")
def gqa32k():
    inp = workloads.generate(workloads.GQA_32K)
    return _parity.DeviceInputs(inp), _parity.run_oracle(inp)


@pytest.mark.parametrize("mode", ["sync", "unified", "unified_local"])
def test_gqa_32k_bf16(gqa32k, mode):
    dev, (ref, ref_lse, ref_flag, margin) = gqa32k
    out, lse, flags = _check(dev, ref, ref_lse, mode, where="gqa32k heuristic")
    _check(dev, ref, ref_lse, mode, out_dtype="f32", where="gqa32k fp32-out")
    _check(dev, ref, ref_lse, mode, num_splits=128, plan_splits=128, where="gqa32k S=128")
    if mode == "unified":
        assert _parity.margin_ok(margin).all()
        assert np.array_equal(flags.cpu().numpy().ravel(), ref_flag)


@pytest.fixture(scope="module")
def paged64():
    inp = workloads.generate(workloads.PAGED_B64)
    return _parity.DeviceInputs(inp), _parity.run_oracle(inp)


@pytest.mark.parametrize("mode", ["sync", "unified", "unified_local"])
def test_paged_batch64_bf16(paged64, mode):
    dev, (ref, ref_lse, ref_flag, margin) = paged64
    out, lse, flags = _check(dev, ref, ref_lse, mode, where="paged b64 heuristic")
    _check(dev, ref, ref_lse, mode, out_dtype="f32", where="paged b64 fp32-out")
    _check(dev, ref, ref_lse, mode, num_splits=4, plan_splits=4, where="paged b64 S=4")
    _check(dev, ref, ref_lse, mode, num_splits=4, plan_splits=4, out_dtype="f32",
           where="paged b64 S=4 fp32-out")
    if mode == "unified":
        assert _parity.margin_ok(margin).all()
        assert np.array_equal(flags.cpu().numpy().ravel(), ref_flag)


def test_unified_stress_128k():
    inp = workloads.generate(workloads.STRESS_128K)
    dev = _parity.DeviceInputs(inp)
    ref, ref_lse, ref_flag, margin = _parity.run_oracle(inp)
    assert _parity.margin_ok(margin).all(), "a flag decision lies within 1e-3 of a bound"
    out, lse, flags, st = _parity.run_gpu(dev, mode="unified", want_stats=True)
    _parity.compare(out, ref.reshape(out.shape), "bf16", where="stress unified")
    _parity.compare_lse(lse, ref_lse.reshape(lse.shape), where="stress unified")
    got_flags = flags.cpu().numpy().ravel()
    assert np.array_equal(got_flags, ref_flag)
    assert st.rows_flagged == int(ref_flag.sum()) and st.recompute_launched == 1
    assert st.splits_flagged >= 1
    out32, _, _ = _parity.run_gpu(dev, mode="unified", out_dtype="f32")
    _parity.compare(out32, ref.reshape(out32.shape), "f32", where="stress unified fp32-out")
    out_s, lse_s, flags_s = _parity.run_gpu(dev, mode="sync")
    _parity.compare(out_s, ref.reshape(out_s.shape), "bf16", where="stress sync")
    assert not flags_s.cpu().numpy().any()
    # split-local fallback: the same flags, the same results, and no second pass
    out_l, lse_l, flags_l, st_l = _parity.run_gpu(dev, mode="unified_local", want_stats=True)
    _parity.compare(out_l, ref.reshape(out_l.shape), "bf16", where="stress unified_local")
    _parity.compare_lse(lse_l, ref_lse.reshape(lse_l.shape), where="stress unified_local")
    assert np.array_equal(flags_l.cpu().numpy().ravel(), ref_flag)
    assert st_l.rows_flagged == int(ref_flag.sum()) and st_l.recompute_launched == 0
    out_l32, _, _ = _parity.run_gpu(dev, mode="unified_local", out_dtype="f32")
    _parity.compare(out_l32, ref.reshape(out_l32.shape), "f32", where="stress unified_local f32")


# ---- edge sweep: group sizes, head dims, dtypes, layouts, ragged lengths, splits -------------
EDGE_LENS = (0, 1, 15, 16, 17, 63, 64, 65, 255, 256, 257, 1000)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_edge_sweep(dtype, head_dim, group):
    case = 0
    for paged in (False, True):
        wl = workloads.Workload(f"edge_{dtype}_{head_dim}_{group}_{paged}", len(EDGE_LENS),
                                2 * group, 2, head_dim, dtype, dtype, lens=EDGE_LENS,
                                paged=paged, page_size=16, max_seq_len=1024 + 7 if not paged else 0)
        inp = workloads.generate(wl, offset=group + 3 * head_dim)
        dev = _parity.DeviceInputs(inp)
        ref, ref_lse, _, _ = _parity.run_oracle(inp)
        for mode in ("sync", "unified", "unified_local"):
            ns = (0, 1, 3, 7)[case % 4]
            case += 1
            for od in ((dtype, "f32") if dtype != "f32" else ("f32",)):
                _check(dev, ref, ref_lse, mode, out_dtype=od, num_splits=ns, plan_splits=ns,
                       where=f"edge {dtype} d{head_dim} G{group} paged={paged} S={ns}")


@pytest.mark.parametrize("group", [1, 4])
@pytest.mark.parametrize("paged", [False, True])
def test_step_with_fewer_units_than_ctas(group, paged):
    """The grid is sized from the cache capacity (8192 tokens here) but this step holds a few
    dozen 16-token units, fewer than the CTAs: balanced shares must still put each group's
    pieces on consecutive CTAs, so that the merge finds every partial it counts."""
    lens = (40, 0, 100, 0, 1)
    wl = workloads.Workload(f"sparse_G{group}_paged{paged}", len(lens), 2 * group, 2, 128,
                            "bf16", "bf16", lens=lens, paged=paged, page_size=16,
                            max_seq_len=0 if paged else 8192)
    inp = workloads.generate(wl, offset=11 + group)
    if paged:   # a wide table: the capacity, not the lengths, sizes the grid
        bt = torch.full((len(lens), 512), -1, dtype=torch.int32)
        bt[:, :inp.block_table.shape[1]] = inp.block_table
        inp.block_table, inp.max_blocks_per_seq = bt, 512
    dev = _parity.DeviceInputs(inp)
    ref, ref_lse, _, _ = _parity.run_oracle(inp)
    attn = binding.DecodeAttention(_parity.problem_for(inp), 0)
    assert attn.info.grid_ctas >= 100   # this step has fewer than 100 units, cost units included
    for mode in ("sync", "unified"):
        for od in ("bf16", "f32"):
            _check(dev, ref, ref_lse, mode, out_dtype=od, num_splits=0, plan_splits=0,
                   where=f"sparse G{group} paged={paged}")


@pytest.mark.parametrize("group,head_dim", [(1, 128), (4, 64), (8, 64), (8, 128)])
def test_merge_of_many_pieces(group, head_dim):
    """100 uniform splits per group: the in-kernel merge takes its partials in several blocks
    (more pieces than one block holds for every elements-per-thread width), and the last
    splits of each sequence are empty."""
    wl = workloads.Workload(f"many_G{group}_d{head_dim}", 1, 2 * group, 2, head_dim, "bf16",
                            "bf16", seq_len=8192, num_splits=100)
    inp = workloads.generate(wl, offset=5 * group + head_dim)
    dev = _parity.DeviceInputs(inp)
    ref, ref_lse, _, _ = _parity.run_oracle(inp)
    for mode in ("sync", "unified"):
        for od in ("bf16", "f32"):
            _check(dev, ref, ref_lse, mode, out_dtype=od, num_splits=100, plan_splits=100,
                   where=f"many pieces G{group} d{head_dim}")


@pytest.mark.parametrize("page_size", [8, 16, 32, 64, 128])
def test_page_sizes(page_size):
    wl = workloads.PAGED_B64.replace(name=f"pages{page_size}", batch=6, page_size=page_size,
                                     lens=(1, 100, 700, 2049, 64, 129))
    inp = workloads.generate(wl, offset=page_size)
    dev = _parity.DeviceInputs(inp)
    ref, ref_lse, _, _ = _parity.run_oracle(inp)
    for mode in ("sync", "unified"):
        for ns in (0, 5):
            for od in ("bf16", "f32"):
                _check(dev, ref, ref_lse, mode, out_dtype=od, num_splits=ns, plan_splits=ns,
                       where=f"page {page_size} S={ns}")


# ---- integer exactness: gather offsets --------------------------------------------------------
@pytest.mark.parametrize("paged", [False, True])
def test_gather_offsets_bit_exact(paged):
    wl = workloads.PAGED_B64.replace(name="gather", batch=5, lens=(0, 1, 17, 300, 1024),
                                     paged=paged, max_seq_len=0 if paged else 1100)
    inp = workloads.generate(wl)
    dev = _parity.DeviceInputs(inp)
    attn = binding.DecodeAttention(_parity.problem_for(inp), 0)
    T = inp.max_blocks_per_seq * wl.page_size if paged else inp.max_seq_len
    offs = torch.empty((wl.batch, wl.num_kv_heads, T), dtype=torch.int64, device="cuda")
    binding.decode_attn_debug_gather(attn.plan, None if dev.bt is None else dev.bt.data_ptr(),
                                     dev.sl.data_ptr(), offs.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    want = oracle.gather_offsets(_parity.oracle_shape(inp),
                                 None if inp.block_table is None else inp.block_table.numpy(),
                                 inp.seq_lens.numpy())
    assert np.array_equal(offs.cpu().numpy(), want)


# ---- overflow detection and synchronised recompute ------------------------------------------
@pytest.mark.parametrize("mode", ["unified", "unified_local"])
def test_forced_fallback_every_row(mode):
    wl = workloads.GQA_32K.replace(name="forced", seq_len=5000, mode=mode)
    inp = workloads.generate(wl, offset=9)
    dev = _parity.DeviceInputs(inp)
    phi, lo, hi = 0.0, -0.25, 0.25        # N(0,1) logits: every row leaves the range
    ref, ref_lse, ref_flag, margin = _parity.run_oracle(inp, phi=phi, lo=lo, hi=hi)
    assert ref_flag.all() and _parity.margin_ok(margin).all()
    narrow = binding.DecodeAttention(_parity.problem_for(inp, mode=mode, phi=phi, lo=lo, hi=hi), 0)
    out, lse, flags, st = _parity.run_gpu(dev, want_stats=True, attn=narrow)
    _parity.compare(out, ref.reshape(out.shape), "bf16", where="forced fallback")
    _parity.compare_lse(lse, ref_lse.reshape(lse.shape), where="forced fallback")
    assert flags.cpu().numpy().all() and st.rows_flagged == 32
    # the same workspace then serves an unflagged run (the flagged list was reset)
    wide = binding.DecodeAttention(_parity.problem_for(inp, mode=mode), 0)
    assert wide.workspace_bytes == narrow.workspace_bytes
    wide.workspace = narrow.workspace
    ref2, ref_lse2, _, _ = _parity.run_oracle(inp)
    out2, lse2, flags2, st2 = _parity.run_gpu(dev, want_stats=True, attn=wide)
    _parity.compare(out2, ref2.reshape(out2.shape), "bf16", where="after fallback")
    assert st2.rows_flagged == 0 and not flags2.cpu().numpy().any()


def test_some_rows_flagged_in_a_paged_batch():
    """A few K rows point along one query head's direction, so exactly those rows (a head in
    each of two groups of different sequences, two heads of one of them) leave [lo, hi]: the
    list holds only their groups, the recompute covers them, the other groups keep their
    unified results, and the flags are exact per row."""
    wl = workloads.Workload("someflags", 6, 32, 8, 128, "bf16", "bf16", lens=(900, 3000, 17, 2500, 640, 1),
                            paged=True, page_size=16, mode="unified")
    inp = workloads.generate(wl, offset=21)
    G, P = 4, 16
    # (sequence, kv head, token, head within the group)
    plant = [(1, 2, 100, 1), (3, 5, 2000, 3), (3, 5, 7, 0)]
    for b, kvh, t, hg in plant:
        qh = inp.q[b, kvh * G + hg].float()
        row = inp.block_table[b, t // P].item()
        inp.k_cache[row, t % P, kvh] = (12.0 * qh / qh.norm()).to(torch.bfloat16)
    phi, lo, hi = 0.0, -30.0, 8.0
    dev = _parity.DeviceInputs(inp)
    ref, ref_lse, ref_flag, margin = _parity.run_oracle(inp, phi=phi, lo=lo, hi=hi)
    flagged = {(b, kvh * G + hg) for b, kvh, _, hg in plant}
    got_rows = {(int(i) // 32, int(i) % 32) for i in np.flatnonzero(ref_flag)}
    assert flagged <= got_rows and len(got_rows) <= 8   # the planted rows, a few neighbours at most
    assert _parity.margin_ok(margin).all()
    for mode, od in (("unified", "bf16"), ("unified", "f32"), ("unified_local", "bf16"),
                     ("unified_local", "f32")):
        out, lse, flags, st = _parity.run_gpu(dev, mode=mode, out_dtype=od, want_stats=True,
                                              phi=phi, lo=lo, hi=hi)
        _parity.compare(out, ref.reshape(out.shape), od, where=f"some rows flagged {mode} {od}")
        _parity.compare_lse(lse, ref_lse.reshape(lse.shape), where="some rows flagged")
        assert np.array_equal(flags.cpu().numpy().ravel().astype(bool), ref_flag.astype(bool))
        assert st.rows_flagged == int(ref_flag.sum())


def test_underflow_injection_is_flagged_and_finite():
    # every logit far below phi + lo: the unified exponentials would underflow to zero
    wl = workloads.Workload("underflow", 1, 4, 1, 128, "bf16", "bf16", seq_len=700,
                            mode="unified")
    inp = workloads.generate(wl)
    u = torch.randn(128, generator=torch.Generator().manual_seed(3))
    u = u / u.norm()
    inp.k_cache[:] = (u * 3.0 + 0.05 * inp.k_cache.float()).to(torch.bfloat16)
    inp.q[:] = (-60.0 * u).to(torch.bfloat16)          # logits ~ -60 * 3 / sqrt(128) * |u|^2
    dev = _parity.DeviceInputs(inp)
    ref, ref_lse, ref_flag, margin = _parity.run_oracle(inp, phi=0.0, lo=-10.0, hi=10.0)
    assert ref_flag.all() and _parity.margin_ok(margin).all()
    for mode in ("unified", "unified_local"):
        out, lse, flags = _parity.run_gpu(dev, mode=mode, phi=0.0, lo=-10.0, hi=10.0)
        _parity.compare(out, ref.reshape(out.shape), "bf16", where=f"underflow {mode}")
        _parity.compare_lse(lse, ref_lse.reshape(lse.shape), where=f"underflow {mode}")
        assert flags.cpu().numpy().all()


# ---- validation findings ------------------------------------------------------------------
def test_bad_block_table_is_reported_not_read():
    wl = workloads.PAGED_B64.replace(name="badtable", batch=3, lens=(40, 300, 17))
    inp = workloads.generate(wl)
    inp.block_table[1, 5] = -1                          # inside sequence 1's length
    inp.block_table[2, 0] = inp.num_physical_blocks + 5
    dev = _parity.DeviceInputs(inp)
    with pytest.raises(binding.DecodeAttnError) as e:
        _parity.run_gpu(dev, validate=True)
    assert e.value.code == -4
    # without validate the run completes and check_status reports it afterwards
    attn = binding.DecodeAttention(_parity.problem_for(inp), 0)
    _parity.run_gpu(dev, attn=attn)
    with pytest.raises(binding.DecodeAttnError) as e:
        binding.decode_attn_check_status(attn.plan, attn.workspace.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream)
    assert e.value.code == -4
    binding.decode_attn_check_status(attn.plan, attn.workspace.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)   # cleared
    # sequence 0 does not touch the bad entries: its rows are still exact
    ref, ref_lse, _, _ = _parity.run_oracle(inp, rows=list(range(wl.num_q_heads)))
    out, _, _ = _parity.run_gpu(dev)
    _parity.compare(out[0], ref.reshape(out[0].shape), "bf16", where="bad table, clean seq")


def test_pipeline_timeout_is_reported_and_cleared():
    """The bounded-wait path, without a fault: a test hook makes CTA 0's producer leave its
    first ring stage unarmed and unfilled and shortens every wait to 2 ms, so its consumers'
    wait runs out. The run reports DA_ERR_DEVICE_TIMEOUT (validate), the status word of a run
    without validate reads once and is cleared by decode_attn_check_status, and the same
    workspace then serves an ordinary run exactly."""
    wl = workloads.GQA_32K.replace(name="timeout", seq_len=4096)
    inp = workloads.generate(wl)
    dev = _parity.DeviceInputs(inp)
    prob = _parity.problem_for(inp, validate=True)
    prob.debug_stall_stage = 1
    with pytest.raises(binding.DecodeAttnError) as e:
        binding.DecodeAttention(prob, 0).run(dev.q, dev.k, dev.v, dev.bt, dev.sl, wl.scale)
    assert e.value.code == -6   # DA_ERR_DEVICE_TIMEOUT
    prob = _parity.problem_for(inp)
    prob.debug_stall_stage = 1
    stalled = binding.DecodeAttention(prob, 0)
    stalled.run(dev.q, dev.k, dev.v, dev.bt, dev.sl, wl.scale)
    stream = torch.cuda.current_stream().cuda_stream
    with pytest.raises(binding.DecodeAttnError) as e:
        binding.decode_attn_check_status(stalled.plan, stalled.workspace.data_ptr(), stream)
    assert e.value.code == -6
    binding.decode_attn_check_status(stalled.plan, stalled.workspace.data_ptr(), stream)
    plain = binding.DecodeAttention(_parity.problem_for(inp), 0)
    assert plain.workspace_bytes == stalled.workspace_bytes
    plain.workspace = stalled.workspace   # the workspace the timed-out runs used
    out, lse, _ = plain.run(dev.q, dev.k, dev.v, dev.bt, dev.sl, wl.scale)
    torch.cuda.synchronize()
    ref, ref_lse, _, _ = _parity.run_oracle(inp)
    _parity.compare(out, ref.reshape(out.shape), wl.out_dtype, where="after a timeout")
    _parity.compare_lse(lse, ref_lse.reshape(lse.shape), where="after a timeout")


def test_bad_seq_len_is_reported():
    wl = workloads.GQA_32K.replace(name="badlen", batch=2, seq_len=256)
    inp = workloads.generate(wl)
    dev = _parity.DeviceInputs(inp)
    dev.sl[1] = 257                                    # above the 256-token capacity
    with pytest.raises(binding.DecodeAttnError) as e:
        _parity.run_gpu(dev, validate=True)
    assert e.value.code == -7


# ---- determinism and workspace reuse --------------------------------------------------------
def test_runs_are_bitwise_deterministic(paged64):
    dev, _ = paged64
    attn = binding.DecodeAttention(_parity.problem_for(dev.inp, mode="unified"), 0)
    outs = [_parity.run_gpu(dev, attn=attn) for _ in range(3)]
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert torch.equal(a, b)


def test_one_workspace_across_split_choices(gqa32k):
    dev, (ref, ref_lse, _, _) = gqa32k
    attn = binding.DecodeAttention(_parity.problem_for(dev.inp, mode="unified"), 16)
    for ns in (-1, 0, 16, 1, 3, 0, -1):
        out, lse, _ = _parity.run_gpu(dev, attn=attn, num_splits=ns)
        _parity.compare(out, ref.reshape(out.shape), "bf16", where=f"reuse S={ns}")
        _parity.compare_lse(lse, ref_lse.reshape(lse.shape), where=f"reuse S={ns}")
