"""Host-side tests of the C ABI (CPU only: no call here reaches CUDA).

Plans are made with an explicit SM count (da_problem.num_sms), so planning never queries a
device, and every run below fails argument validation before anything is enqueued.
"""
import ctypes
import os
import math

import numpy as np
import pytest
import torch

from decode_attention_attn_gb300 import binding, build as lib_build, workloads


@pytest.fixture(scope="module")
def L():
    lib_build.build()
    return binding.lib()


def _prob(**kw):
    base = dict(batch=1, num_q_heads=32, num_kv_heads=8, head_dim=128, qkv_dtype="bf16",
                out_dtype="bf16", max_seq_len=32768, num_sms=152)
    base.update(kw)
    return binding.make_problem(**base)


def test_library_exports_every_header_symbol(L):
    names = binding.header_symbols()
    assert "decode_attn_plan" in names and "decode_attn_run" in names
    for n in names:
        assert hasattr(L, n), f"{n} declared in decode_attn.h but not exported"


def test_abi_version_and_strerror(L):
    assert binding.decode_attn_abi_version() == 4
    for code in binding.ERRORS:
        assert binding.decode_attn_strerror(code)
    assert "unknown" in binding.decode_attn_strerror(-99)


@pytest.mark.parametrize("kw,code", [
    (dict(num_q_heads=32, num_kv_heads=6), -1),          # H_q % H_kv != 0
    (dict(num_q_heads=24, num_kv_heads=8), -2),          # group 3 not built
    (dict(num_q_heads=32, num_kv_heads=2), -2),          # group 16 not built
    (dict(head_dim=96), -2),
    (dict(qkv_dtype="bf16", max_seq_len=0), -1),
    (dict(batch=0), -1),
    (dict(paged=True, page_size=12, max_blocks_per_seq=8, num_physical_blocks=8), -2),
    (dict(paged=True, page_size=4, max_blocks_per_seq=8, num_physical_blocks=8), -2),
    (dict(paged=True, page_size=16, max_blocks_per_seq=0, num_physical_blocks=8), -1),
    (dict(paged=True, page_size=16, max_blocks_per_seq=8, num_physical_blocks=1 << 27), -1),
    (dict(batch=70000, max_seq_len=32768), -1),          # B * max_seq_len >= 2^31
    (dict(mode="unified", range_lo=5.0, range_hi=5.0), -1),
    (dict(mode="unified", unified_max=math.inf), -1),
    (dict(mode="unified_local", range_lo=1.0, range_hi=-1.0), -1),
    (dict(num_sms=-1), -1),
    # FP8 caches: bf16 q, finite positive scales
    (dict(kv_dtype="e4m3", k_scale=0.0), -1),
    (dict(kv_dtype="e4m3", v_scale=-1.0), -1),
    (dict(kv_dtype="e4m3", k_scale=math.inf), -1),
    (dict(kv_dtype="e4m3", v_scale=math.nan), -1),
    (dict(kv_dtype="e4m3", qkv_dtype="f16", out_dtype="f16"), -2),
    (dict(debug_stall_stage=-1), -1),
])
def test_plan_rejects_bad_problems(L, kw, code):
    with pytest.raises(binding.DecodeAttnError) as e:
        binding.decode_attn_plan(_prob(**kw), 0)
    assert e.value.code == code


@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_fp8_plans_for_every_group(L, group):
    plan, _ = binding.decode_attn_plan(_prob(kv_dtype="e4m3", num_q_heads=8 * group,
                                             num_kv_heads=8), 0)
    binding.decode_attn_destroy(plan)


def test_plan_rejects_a_bad_fp8_flag(L):
    prob = _prob()
    prob.kv_fp8 = 2
    with pytest.raises(binding.DecodeAttnError) as e:
        binding.decode_attn_plan(prob, 0)
    assert e.value.code == -1


def test_fp8_plan_packs_kv_head_pairs_on_large_steps(L):
    """FP8 caches with groups of 4 query heads over pairs of KV heads: the split kernel takes a
    pair at once where the step is large (four packed groups per SM, or 128 MiB of cache), so
    that its 64-token stage holds as many bytes as a bf16 stage of one KV head and a balanced
    share covers half as many tokens of a group. The 32K GQA step (67 MB) keeps one KV head
    per group, with half-size stages and a deeper pipeline; so does an odd KV-head count."""
    fp8 = dict(kv_dtype="e4m3", k_scale=0.01, v_scale=0.02)
    paged = dict(batch=64, paged=True, page_size=16, max_blocks_per_seq=512,
                 num_physical_blocks=20000, max_seq_len=0)
    cases = {"bf16": _prob(), "32k": _prob(**fp8), "128k": _prob(max_seq_len=131072, **fp8),
             "paged": _prob(**paged, **fp8), "odd": _prob(num_q_heads=12, num_kv_heads=3, **fp8),
             "odd_paged": _prob(**paged, num_q_heads=12, num_kv_heads=3, **fp8),
             "few_sms": _prob(num_sms=16, **fp8)}
    info = {}
    for k, prob in cases.items():
        plan, _ = binding.decode_attn_plan(prob, 0)
        info[k] = binding.decode_attn_plan_info(plan)
        binding.decode_attn_destroy(plan)
    hp = {k: i.kv_heads_per_group for k, i in info.items()}
    assert hp == {"bf16": 1, "32k": 1, "128k": 2, "paged": 2, "odd": 1, "odd_paged": 1,
                  "few_sms": 2}
    for k, i in info.items():
        assert i.stage_tokens == 64 and i.smem_bytes <= 232448
    assert info["32k"].stages > info["bf16"].stages
    assert info["128k"].stages >= 5
    # a packed share: half the tokens of a pair that carries twice the bytes per token
    s16, _ = binding.decode_attn_plan(_prob(max_seq_len=131072), 0)
    i16 = binding.decode_attn_plan_info(s16)
    binding.decode_attn_destroy(s16)
    assert abs(2 * info["128k"].split_tokens - i16.split_tokens) <= 64


def test_plan_rejects_an_unknown_softmax_mode(L):
    prob = _prob()
    prob.mode = 3
    with pytest.raises(binding.DecodeAttnError) as e:
        binding.decode_attn_plan(prob, 0)
    assert e.value.code == -1


def test_plan_choices_for_the_named_workloads(L):
    # 32K GQA: balanced shares over all 152 SMs, a deep pipeline within 227 KB
    plan, ws = binding.decode_attn_plan(_prob(), 0)
    info = binding.decode_attn_plan_info(plan)
    assert info.grid_ctas == 152 and info.num_splits == 0
    assert info.stages >= 4 and info.smem_bytes <= 232448
    assert info.unit_tokens == 16 and info.stage_tokens == 64
    assert info.recompute_splits == 19            # ceil(152 SMs / 8 groups)
    binding.decode_attn_destroy(plan)
    # tiny: explicit 4 uniform splits -> 4 CTAs
    plan, _ = binding.decode_attn_plan(_prob(num_q_heads=1, num_kv_heads=1, head_dim=64,
                                             qkv_dtype="f32", out_dtype="f32", max_seq_len=256), 4)
    info = binding.decode_attn_plan_info(plan)
    assert info.num_splits == 4 and info.grid_ctas == 4
    binding.decode_attn_destroy(plan)
    # paged batch of 64: balanced; a page of 32 makes the split unit 32
    plan, _ = binding.decode_attn_plan(_prob(batch=64, paged=True, page_size=32,
                                             max_blocks_per_seq=256, num_physical_blocks=9000,
                                             max_seq_len=0), 0)
    info = binding.decode_attn_plan_info(plan)
    assert info.num_splits == 0 and info.grid_ctas == 152 and info.unit_tokens == 32
    binding.decode_attn_destroy(plan)
    # a batch too large to keep lengths in shared memory falls back to uniform splits
    plan, _ = binding.decode_attn_plan(_prob(batch=4096, max_seq_len=512), 0)
    info = binding.decode_attn_plan_info(plan)
    assert info.num_splits >= 1
    binding.decode_attn_destroy(plan)


def test_small_problem_does_not_spread_below_min_share(L):
    # one group of 256 tokens = 16 units of 16 -> at most 2 CTAs of >= 8 units
    plan, _ = binding.decode_attn_plan(_prob(num_q_heads=4, num_kv_heads=1, max_seq_len=256), 0)
    assert binding.decode_attn_plan_info(plan).grid_ctas == 2
    binding.decode_attn_destroy(plan)


def test_workspace_holds_the_split_partials(L):
    # Flash-Decoding's "Hardware Execution Topology and Memory Traffic" sizes the partial
    # outputs of B=1, H=32, S=128, d=128 at 1.05 MB in 16-bit floats; this library keeps them
    # in FP32, so exactly twice that, plus small per-group bookkeeping.
    plan, ws = binding.decode_attn_plan(_prob(num_kv_heads=32, max_seq_len=32768), 128)
    part_o = 1 * 32 * 128 * 128 * 2 * 2
    assert part_o == 2 * 1048576
    assert part_o <= ws <= part_o + 96 * 1024
    binding.decode_attn_destroy(plan)


def test_plan_reports_the_split_size(L):
    # 32K GQA on 152 SMs: 8 groups of 32768 tokens over 152 balanced shares, 19 per group, so
    # every split holds about 32768 / 19 tokens, in whole 16-token units
    plan, _ = binding.decode_attn_plan(_prob(max_seq_len=32768), 0)
    info = binding.decode_attn_plan_info(plan)
    assert info.num_splits == 0 and info.grid_ctas == 152
    assert info.split_tokens % 16 == 0 and info.split_tokens_min % 16 == 0
    assert 32768 // 19 - 16 * 13 <= info.split_tokens_min <= info.split_tokens <= 32768 // 19 + 32
    binding.decode_attn_destroy(plan)
    # uniform splits: roundup(ceil(4096 / 16), 16) = 256 tokens each
    plan, _ = binding.decode_attn_plan(_prob(num_kv_heads=32, max_seq_len=4096), 16)
    info = binding.decode_attn_plan_info(plan)
    assert (info.split_tokens, info.split_tokens_min) == (256, 256)
    binding.decode_attn_destroy(plan)
    plan, _ = binding.decode_attn_plan(_prob(max_seq_len=1000), 3)
    info = binding.decode_attn_plan_info(plan)
    assert (info.split_tokens, info.split_tokens_min) == (336, 328)
    binding.decode_attn_destroy(plan)


def test_run_rejects_bad_arguments_before_any_cuda_call(L):
    plan, ws = binding.decode_attn_plan(_prob(max_seq_len=1024), 0)
    A = 0x100000   # aligned fake device addresses: never dereferenced, validation fails first
    good = dict(q=A, k_cache=A, v_cache=A, block_table=None, seq_lens=A, scale=0.1,
                num_splits=-1, out=A, out_lse=A, row_flags=A, workspace=A, workspace_bytes=ws)

    def call(**kw):
        args = dict(good)
        args.update(kw)
        with pytest.raises(binding.DecodeAttnError) as e:
            binding.decode_attn_run(plan, **args)
        return e.value.code

    assert call(q=0) == -1
    assert call(seq_lens=0) == -1
    assert call(out=0) == -1
    assert call(workspace=0) == -1
    assert call(block_table=A) == -1                 # contiguous problem given a table
    assert call(q=A + 8) == -1                       # q not 16-byte aligned
    assert call(k_cache=A + 4) == -1
    assert call(workspace=A + 16) == -1              # workspace not 256-byte aligned
    assert call(out_lse=A + 2) == -1
    assert call(scale=float("nan")) == -1
    assert call(num_splits=-2) == -1
    assert call(workspace_bytes=ws - 1) == -3
    info = binding.decode_attn_plan_info(plan)
    assert call(num_splits=info.max_splits + 1) == -3
    binding.decode_attn_destroy(plan)
    pplan, pws = binding.decode_attn_plan(_prob(paged=True, page_size=16, max_blocks_per_seq=64,
                                                num_physical_blocks=64, max_seq_len=0), 0)
    with pytest.raises(binding.DecodeAttnError) as e:   # paged problem without a table
        binding.decode_attn_run(pplan, A, A, A, None, A, 0.1, -1, A, A, A, A, pws)
    assert e.value.code == -1
    binding.decode_attn_destroy(pplan)


def test_workspace_init_and_debug_gather_validate_arguments(L):
    plan, ws = binding.decode_attn_plan(_prob(max_seq_len=1024), 0)
    with pytest.raises(binding.DecodeAttnError) as e:
        binding.decode_attn_workspace_init(plan, 0x100000, ws - 1)
    assert e.value.code == -3
    with pytest.raises(binding.DecodeAttnError) as e:
        binding.decode_attn_workspace_init(plan, 0x100008, ws)
    assert e.value.code == -1
    with pytest.raises(binding.DecodeAttnError) as e:
        binding.decode_attn_debug_gather(plan, 0x100000, 0x100000, 0x100000)
    assert e.value.code == -1
    binding.decode_attn_destroy(plan)


# ---- the synthetic workload recipe ---------------------------------------------------------
def test_paged_workload_recipe():
    wl = workloads.PAGED_B64.replace(batch=8)
    inp = workloads.generate(wl)
    lens = inp.seq_lens.numpy()
    assert lens.min() >= 512 and lens.max() <= 8192
    pages = (lens + 15) // 16
    table = inp.block_table.numpy()
    used = np.concatenate([table[b, :pages[b]] for b in range(8)])
    assert sorted(used.tolist()) == list(range(inp.num_physical_blocks))   # each page once
    for b in range(8):
        assert (table[b, pages[b]:] == -1).all()
    assert inp.k_cache.shape == (inp.num_physical_blocks, 16, 8, 128)
    assert inp.kv_bytes() == int(lens.sum()) * 8 * 2 * 128 * 2


def test_full_paged_workload_lengths_are_seeded():
    lens = workloads.sequence_lengths(workloads.PAGED_B64)
    assert len(lens) == 64 and min(lens) >= 512 and max(lens) <= 8192
    assert lens == workloads.sequence_lengths(workloads.PAGED_B64)


def test_stress_workload_outlier_rows():
    wl = workloads.STRESS_128K.replace(seq_len=4096)
    inp = workloads.generate(wl)
    assert inp.outlier_rows == round(0.005 * 8 * 4096)
    norms = inp.k_cache.float().norm(dim=-1)[0]           # [tokens, kv heads]
    big = (norms > 200).sum().item()                      # |40 * N(0, I_128)| ~ 450
    assert big == inp.outlier_rows


def test_kv_cache_bytes_per_token_matches_the_handbook():
    # "FlashAttention and inference kernels", "Inference: prefill and decode": 32 layers,
    # 8 KV heads, d = 128, BF16 -> 128 KB of KV cache per token.
    wl = workloads.GQA_32K.replace(seq_len=1)
    inp = workloads.generate(wl)
    assert inp.kv_bytes() * 32 == 128 * 1024


def test_plain_c_program_uses_the_abi(L, tmp_path):
    """tests/c_abi_host.c, compiled with gcc against include/decode_attn.h alone and linked to
    the library: the boundary needs neither Python nor CUDA headers on the caller's side."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    here = os.path.dirname(os.path.abspath(__file__))
    lib = binding.library_path()
    exe = str(tmp_path / "c_abi_host")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I" + lib_build.INCLUDE,
                    os.path.join(here, "c_abi_host.c"), lib, "-Wl,-rpath," + os.path.dirname(lib),
                    "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    lines = r.stdout.splitlines()
    assert lines[-1] == "ok"
    bf16 = next(x for x in lines if x.startswith("bf16 ")).split()
    fp8 = next(x for x in lines if x.startswith("fp8 ")).split()
    assert int(bf16[2]) == int(fp8[2]) == 152                # grid_ctas
    assert int(fp8[4]) >= int(bf16[4])                       # stages: FP8 tiles are smaller
    assert int(bf16[12]) == int(fp8[12]) == 1                # 32K GQA: one KV head per group
