"""decode_attn_run_static: the entry point for callers that cannot allocate a device workspace.

Such callers include a server whose device memory is all reserved for its KV-cache pool, a
process under a device-memory cap, a decode loop that cannot pay for the device-wide
synchronisation that cudaMalloc / cudaFree may cause, and C code with no device allocator.
The entry point runs the same kernels as decode_attn_run, on a fixed scratch region that
the library reserves per device. Each case below checks, on two consecutive calls, that its
results match decode_attn_run with a caller workspace on the same inputs within the parity
tolerance, and the float64 CPU oracle within the same tolerance, and that the calls made no
allocation through PyTorch's allocator. The cases run one after another, so each call also
follows runs of other plans on the same scratch.
"""
import ctypes

import pytest
import torch

from decode_attention_attn_gb300 import binding, workloads

import _parity

W = workloads
CASES = [
    (W.PAGED_B64, "unified"),
    (W.GQA_32K, "sync"),
    (W.STRESS_128K, "unified"),   # flagged rows: exercises the recompute pass and its list
    (W.MHA_4K, "sync"),           # uniform splits (the plan's default for this workload)
    (W.PAGED_B64_FP8, "unified_local"),   # an FP8 cache
]


@pytest.mark.gpu
@pytest.mark.parametrize("wl,mode", CASES, ids=[f"{w.name}-{m}" for w, m in CASES])
def test_static_scratch_matches_workspace_run(wl, mode):
    inp = W.generate(wl)
    dev = _parity.DeviceInputs(inp)
    oracle_out, oracle_lse, _, _ = _parity.run_oracle(inp)
    attn = binding.DecodeAttention(_parity.problem_for(inp, mode=mode, out_dtype="f32"),
                                   wl.num_splits)
    assert attn.info.workspace_bytes <= 8 << 20
    ref_out, ref_lse, ref_flags = attn.run(dev.q, dev.k, dev.v, dev.bt, dev.sl, wl.scale)
    torch.cuda.synchronize()
    ref = ref_out.double().cpu().numpy()
    out = torch.empty_like(ref_out)
    lse = torch.empty_like(ref_lse)
    flags = torch.empty_like(ref_flags)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        flags.fill_(7)
        # PyTorch's allocator counts every allocation it serves; the call must add none (the
        # library itself allocates nothing, which this cannot see, but it would show a torch
        # allocation hidden in the binding)
        torch.cuda.synchronize()
        allocations = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
        binding.decode_attn_run_static(
            attn.plan, dev.q.data_ptr(), dev.k.data_ptr(), dev.v.data_ptr(),
            None if dev.bt is None else dev.bt.data_ptr(), dev.sl.data_ptr(), wl.scale, -1,
            out.data_ptr(), lse.data_ptr(), flags.data_ptr(), stream)
        torch.cuda.synchronize()
        assert torch.cuda.memory_stats().get("allocation.all.allocated", 0) == allocations
        where = f"{wl.name} {mode} call {call}"
        _parity.compare(out, ref, "f32", where=where)
        _parity.compare_lse(lse, ref_lse.double().cpu().numpy(), where=where)
        assert torch.equal(flags, ref_flags), f"{where}: row flags differ"
        _parity.compare(out, oracle_out.reshape(ref.shape), "f32", where=where + " vs oracle")
        _parity.compare_lse(lse, oracle_lse.reshape(ref_lse.shape), where=where + " vs oracle")
    if mode == "unified" and wl.outlier_frac > 0:
        assert int(ref_flags.sum()) > 0   # the recompute pass really ran in this case


@pytest.mark.gpu
def test_static_scratch_reports_device_findings_through_stats():
    """A caller of the static entry point sees device findings (here block-table entries
    outside the page pool) through the stats it asks for."""
    wl = W.PAGED_B64.replace(name="static_badtable", batch=3, lens=(40, 300, 17))
    inp = W.generate(wl)
    inp.block_table[1, 5] = -1
    inp.block_table[2, 0] = inp.num_physical_blocks + 5
    dev = _parity.DeviceInputs(inp)
    attn = binding.DecodeAttention(_parity.problem_for(inp), 0)
    out = torch.empty((wl.batch, wl.num_q_heads, wl.head_dim), dtype=torch.bfloat16,
                      device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    with pytest.raises(binding.DecodeAttnError) as e:
        binding.decode_attn_run_static(
            attn.plan, dev.q.data_ptr(), dev.k.data_ptr(), dev.v.data_ptr(), dev.bt.data_ptr(),
            dev.sl.data_ptr(), wl.scale, -1, out.data_ptr(), None, None, stream, want_stats=True)
    assert e.value.code == -4   # DA_ERR_BAD_BLOCK_TABLE
    # the next call clears the region's status: a clean table reports nothing
    good = W.generate(wl)
    dev_good = _parity.DeviceInputs(good)
    st = binding.decode_attn_run_static(
        attn.plan, dev_good.q.data_ptr(), dev_good.k.data_ptr(), dev_good.v.data_ptr(),
        dev_good.bt.data_ptr(), dev_good.sl.data_ptr(), wl.scale, -1, out.data_ptr(), None, None,
        stream, want_stats=True)
    assert st.split_tokens >= st.split_tokens_min > 0


def test_static_scratch_rejects_oversize_plan():
    """A plan whose workspace exceeds the fixed scratch is refused before anything runs."""
    prob = binding.make_problem(batch=4096, num_q_heads=32, num_kv_heads=8, head_dim=128,
                                qkv_dtype="bf16", out_dtype="bf16", max_seq_len=1024,
                                num_sms=152)
    plan, ws = binding.decode_attn_plan(prob, 0)
    try:
        assert ws > 8 << 20
        fake = 1 << 20   # aligned non-null addresses: the size check comes first
        rc = binding.lib().decode_attn_run_static(plan, fake, fake, fake, None, fake,
                                                  ctypes.c_float(0.088), -1, fake, None, None,
                                                  None, None)
        assert rc == -3, binding.ERRORS.get(rc, rc)   # DA_ERR_WORKSPACE_TOO_SMALL
    finally:
        binding.decode_attn_destroy(plan)
