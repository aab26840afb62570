"""Glue between the seeded workloads and the C ABI, shared by bench.py and the tests.

It holds none of the attention arithmetic and never touches the CPU oracle: it maps a
workload's shape onto a da_problem and copies a workload's tensors to the device once.
"""
from __future__ import annotations

from . import binding, workloads


def problem_for(inp: workloads.Inputs, mode=None, out_dtype=None, validate=False, phi=None,
                lo=None, hi=None, num_sms=0):
    """The da_problem describing `inp` (its shape, storage types and unified-max constants)."""
    w = inp.wl
    return binding.make_problem(
        batch=w.batch, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
        head_dim=w.head_dim, qkv_dtype=w.dtype, out_dtype=out_dtype or w.out_dtype,
        paged=w.paged, page_size=w.page_size, max_blocks_per_seq=inp.max_blocks_per_seq,
        num_physical_blocks=inp.num_physical_blocks, max_seq_len=inp.max_seq_len,
        mode=mode or w.mode, unified_max=w.phi if phi is None else phi,
        range_lo=w.range_lo if lo is None else lo, range_hi=w.range_hi if hi is None else hi,
        validate=validate, num_sms=num_sms, kv_dtype=w.kv_dtype, k_scale=inp.k_scale,
        v_scale=inp.v_scale)


class DeviceInputs:
    """The workload's tensors copied to the GPU once."""

    def __init__(self, inp: workloads.Inputs, device="cuda"):
        self.inp = inp
        self.q = inp.q.to(device)
        self.k = inp.k_cache.to(device)
        self.v = inp.v_cache.to(device)
        self.bt = None if inp.block_table is None else inp.block_table.to(device)
        self.sl = inp.seq_lens.to(device)
