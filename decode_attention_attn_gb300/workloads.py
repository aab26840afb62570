"""Seeded synthetic decode-attention workloads.

This module only draws inputs and describes shapes; it holds none of the attention
arithmetic. The same tensors feed the CUDA path and the CPU oracle in the tests and in
bench.py.

Recipe (every draw from a torch CPU generator, values i.i.d. N(0, 1) in fp32, then one
round-to-nearest-even cast to the storage dtype):
  q seed 1, K seed 2, V seed 3 (the seed convention of "FlashAttention and inference
  kernels", "A paged decode attention kernel (with GQA)"), sequence lengths seed 4,
  outlier K rows seed 5, block-table permutation seed 7 (physical pages assigned to the
  sequences' logical pages in a shuffled order, in sequence order, -1 past the end).

The five named workloads have the shapes of the pages' models: Llama2-7B-shaped MHA
(32 heads of 128), a GQA model with 32 query heads over 8 KV heads, and a tiny case.

FP8 caches (kv_dtype "e4m3"): K and V are drawn as above in fp32, then each tensor is
quantised with one scale, max |x| / 448 (448 is the largest E4M3 value), to E4M3 codes by
PyTorch's float8_e4m3fn cast (round to nearest even); the cache holds the code bytes and the
scales (as fp32 numbers) travel with the inputs. q stays bf16.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

SEED_Q, SEED_K, SEED_V, SEED_LENS, SEED_OUTLIERS, SEED_PERM = 1, 2, 3, 4, 5, 7

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2, "e4m3": 1}
E4M3_MAX = 448.0


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: str                      # q / K / V storage: "f32", "f16", "bf16"
    out_dtype: str
    seq_len: int = 0                # every sequence this long (when len_range is None)
    len_range: Optional[tuple] = None   # inclusive uniform range of per-sequence lengths
    paged: bool = False
    page_size: int = 16
    num_splits: int = 0             # 0: the library's heuristic; >0: that many splits
    mode: str = "sync"              # "sync", "unified" or "unified_local"
    phi: float = -3.9               # unified max constant (natural-log units)
    range_lo: float = -64.0         # closed in-range interval on (x - phi)
    range_hi: float = 64.0
    outlier_frac: float = 0.0       # fraction of K rows (kv head, token) scaled
    outlier_scale: float = 40.0
    lens: Optional[tuple] = None    # explicit per-sequence lengths (overrides the above)
    max_seq_len: int = 0            # contiguous capacity per sequence (0: max length)
    kv_dtype: Optional[str] = None  # None: K / V stored as dtype; "e4m3": an FP8 cache

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def kv_storage(self) -> str:
        return self.kv_dtype or self.dtype

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads the pages' models suggest (tiny, Llama2-7B MHA, 32K GQA, paged batch,
# unified-max stress).
TINY = Workload("tiny_b1_h1_d64_n256_f32", 1, 1, 1, 64, "f32", "f32", seq_len=256, num_splits=4)
MHA_4K = Workload("mha_b1_h32_d128_n4096_f16", 1, 32, 32, 128, "f16", "f16", seq_len=4096,
                  num_splits=16)
GQA_32K = Workload("gqa_b1_h32kv8_d128_n32768_bf16", 1, 32, 8, 128, "bf16", "bf16",
                   seq_len=32768)
PAGED_B64 = Workload("paged_b64_h32kv8_d128_n512to8192_bf16", 64, 32, 8, 128, "bf16", "bf16",
                     len_range=(512, 8192), paged=True, page_size=16)
STRESS_128K = Workload("unified_stress_b1_h32kv8_d128_n131072_bf16", 1, 32, 8, 128, "bf16",
                       "bf16", seq_len=131072, mode="unified", outlier_frac=0.005)

# The 32K GQA and paged workloads over FP8 (E4M3) caches: the same draws, quantised.
GQA_32K_FP8 = GQA_32K.replace(name="gqa_b1_h32kv8_d128_n32768_e4m3", kv_dtype="e4m3")
PAGED_B64_FP8 = PAGED_B64.replace(name="paged_b64_h32kv8_d128_n512to8192_e4m3", kv_dtype="e4m3")

WORKLOADS = {w.name: w for w in (TINY, MHA_4K, GQA_32K, PAGED_B64, STRESS_128K, GQA_32K_FP8,
                                 PAGED_B64_FP8)}
ALIASES = {"tiny": TINY.name, "mha": MHA_4K.name, "gqa32k": GQA_32K.name,
           "paged": PAGED_B64.name, "stress": STRESS_128K.name,
           "gqa32k_fp8": GQA_32K_FP8.name, "paged_fp8": PAGED_B64_FP8.name}


def get(name: str) -> Workload:
    return WORKLOADS[ALIASES.get(name, name)]


@dataclasses.dataclass
class Inputs:
    wl: Workload
    q: torch.Tensor                 # [B, Hq, d]
    k_cache: torch.Tensor           # [B, T, Hkv, d] or [nblocks, page, Hkv, d]
    v_cache: torch.Tensor
    block_table: Optional[torch.Tensor]   # int32 [B, max_blocks] (paged)
    seq_lens: torch.Tensor          # int32 [B]
    max_seq_len: int                # contiguous capacity (0 when paged)
    max_blocks_per_seq: int         # paged table width (0 when contiguous)
    num_physical_blocks: int
    outlier_rows: int = 0
    k_scale: float = 1.0            # FP8 caches: the value of code 1 (an fp32 number)
    v_scale: float = 1.0

    def kv_bytes(self) -> int:
        """Algorithmic K+V bytes of one step: sum_b N_b * H_kv * 2 * d * sizeof."""
        w = self.wl
        return int(self.seq_lens.to(torch.int64).sum()) * w.num_kv_heads * 2 * w.head_dim * \
            ELEM_BYTES[w.kv_storage]


def _gen(seed: int, offset: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(seed + 1000003 * offset)
    return g


def _normal(shape, seed, offset, dtype) -> torch.Tensor:
    x = torch.randn(shape, generator=_gen(seed, offset), dtype=torch.float32)
    return x.to(TORCH_DTYPES[dtype])


def sequence_lengths(wl: Workload, offset: int = 0) -> list:
    if wl.lens is not None:
        return [int(n) for n in wl.lens]
    if wl.len_range is not None:
        lo, hi = wl.len_range
        return torch.randint(lo, hi + 1, (wl.batch,), generator=_gen(SEED_LENS, offset)).tolist()
    return [wl.seq_len] * wl.batch


def generate(wl: Workload, offset: int = 0) -> Inputs:
    """Draw the workload's inputs. `offset` selects an independent draw of the same shape."""
    lens = sequence_lengths(wl, offset)
    B, Hkv, d = wl.batch, wl.num_kv_heads, wl.head_dim
    q = _normal((B, wl.num_q_heads, d), SEED_Q, offset, wl.dtype)
    if wl.paged:
        P = wl.page_size
        pages = [(n + P - 1) // P for n in lens]
        total = sum(pages)
        width = max(pages) if pages else 0
        perm = torch.randperm(total, generator=_gen(SEED_PERM, offset)).to(torch.int32)
        table = torch.full((B, max(width, 1)), -1, dtype=torch.int32)
        nxt = 0
        for b, np_ in enumerate(pages):
            table[b, :np_] = perm[nxt:nxt + np_]
            nxt += np_
        kv_shape = (total, P, Hkv, d)
        block_table, max_blocks, nblocks, cap = table, max(width, 1), total, 0
    else:
        cap = wl.max_seq_len or (max(lens) if lens else 0)
        kv_shape = (B, cap, Hkv, d)
        block_table, max_blocks, nblocks = None, 0, 0
    k32 = torch.randn(kv_shape, generator=_gen(SEED_K, offset), dtype=torch.float32)
    n_out = 0
    if wl.outlier_frac > 0:
        # Scale a seeded fraction of K rows: a row is one (kv head, token) key vector of
        # length d, drawn without replacement over the sequence's tokens.
        assert B == 1 and not wl.paged, "outlier injection is defined for one contiguous sequence"
        n_tok = lens[0]
        n_out = int(round(wl.outlier_frac * Hkv * n_tok))
        pick = torch.randperm(Hkv * n_tok, generator=_gen(SEED_OUTLIERS, offset))[:n_out]
        tok, head = pick // Hkv, pick % Hkv
        k32[0, tok, head, :] *= wl.outlier_scale
    if wl.kv_dtype == "e4m3":
        k, k_scale = quantize_e4m3(k32)
        del k32
        v, v_scale = quantize_e4m3(torch.randn(kv_shape, generator=_gen(SEED_V, offset),
                                               dtype=torch.float32))
        return Inputs(wl, q, k, v, block_table, torch.tensor(lens, dtype=torch.int32), cap,
                      max_blocks, nblocks, n_out, k_scale, v_scale)
    k = k32.to(TORCH_DTYPES[wl.dtype])
    del k32
    v = _normal(kv_shape, SEED_V, offset, wl.dtype)
    return Inputs(wl, q, k, v, block_table, torch.tensor(lens, dtype=torch.int32), cap,
                  max_blocks, nblocks, n_out)


def quantize_e4m3(x: torch.Tensor):
    """(E4M3 code bytes as uint8, scale): one fp32 scale for the tensor, max |x| / 448."""
    amax = float(x.abs().max()) if x.numel() else 0.0
    scale = float(np.float32(amax / E4M3_MAX)) if amax > 0 else 1.0
    codes = (x / scale).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale


def input_digest(inp: Inputs) -> dict:
    """The first 16 hex digits of the SHA-256 of each input tensor's stored bytes, so that a
    measurement names the exact inputs it ran on."""
    import hashlib
    out = {}
    for name in ("q", "k_cache", "v_cache", "block_table", "seq_lens"):
        t = getattr(inp, name)
        if t is not None:
            out[name] = hashlib.sha256(bits(t).tobytes()).hexdigest()[:16]
    return out


def bits(t: torch.Tensor) -> np.ndarray:
    """The tensor's storage as numpy: float32 for fp32, uint16 bit patterns for fp16/bf16,
    the code bytes (uint8) of an FP8 cache."""
    t = t.contiguous()
    if t.dtype == torch.float32:
        return t.numpy()
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return t.view(torch.uint8).numpy()
    return t.view(torch.int16).numpy().view(np.uint16)
