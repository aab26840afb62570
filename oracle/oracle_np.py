"""An independent NumPy restatement of decode attention, for tiny shapes only.

TEST INFRASTRUCTURE ONLY (same rule as the C oracle). It exists to pin the C oracle:
it is written separately from it and shares no code with it. It decodes storage with
NumPy's own conversions, walks rows and tokens with explicit Python loops, and
evaluates the max-shifted softmax of "Flash-Decoding: Mathematical Foundations,
Split-KV Parallelism, Online Softmax Reduction, and Serving Latency Optimization",
section "The Single-Token Generation Bottleneck", through the block table of
"FlashAttention and inference kernels", section "PagedAttention".
"""
import math

import numpy as np


def decode(bits, dtype):
    """float64 values of fp32 / fp16 / bf16 storage, by NumPy's own conversions, and of
    e4m3 codes by PyTorch's float8_e4m3fn (NumPy has no 8-bit float)."""
    a = np.asarray(bits)
    if dtype == "e4m3":
        import torch
        codes = torch.from_numpy(np.ascontiguousarray(a.astype(np.uint8)))
        return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    if dtype == "f32":
        return a.astype(np.float32).astype(np.float64)
    if dtype == "f16":
        return a.astype(np.uint16).view(np.float16).astype(np.float64)
    if dtype == "bf16":
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def reference(q_bits, k_bits, v_bits, dtype, seq_lens, scale, *, num_kv_heads, paged=False,
              page_size=16, block_table=None, phi=0.0, range_lo=-math.inf, range_hi=math.inf,
              kv_dtype=None, k_scale=1.0, v_scale=1.0):
    """q: [B, Hq, d]; k, v: [B, T, Hkv, d] (contiguous) or [nblocks, page, Hkv, d] (paged).
    kv_dtype="e4m3": k, v are FP8 codes standing for code * k_scale, code * v_scale.

    Returns (out [B, Hq, d], lse [B, Hq], flag [B, Hq])."""
    q = decode(q_bits, dtype)
    if kv_dtype == "e4m3":
        k = decode(k_bits, "e4m3") * k_scale
        v = decode(v_bits, "e4m3") * v_scale
    else:
        k = decode(k_bits, dtype)
        v = decode(v_bits, dtype)
    B, Hq, d = q.shape
    group = Hq // num_kv_heads
    out = np.zeros((B, Hq, d))
    lse = np.full((B, Hq), -math.inf)
    flag = np.zeros((B, Hq), np.uint8)
    for b in range(B):
        n = int(seq_lens[b])
        for h in range(Hq):
            kvh = h // group
            keys, vals = [], []
            for t in range(n):
                if paged:
                    blk = int(block_table[b][t // page_size])
                    keys.append(k[blk, t % page_size, kvh])
                    vals.append(v[blk, t % page_size, kvh])
                else:
                    keys.append(k[b, t, kvh])
                    vals.append(v[b, t, kvh])
            if n == 0:
                continue
            x = [scale * float(np.dot(q[b, h], kk)) for kk in keys]
            m = max(x)
            w = [math.exp(xi - m) for xi in x]
            denom = sum(w)
            acc = np.zeros(d)
            for wi, vv in zip(w, vals):
                acc = acc + wi * vv
            out[b, h] = acc / denom
            lse[b, h] = m + math.log(denom)
            flag[b, h] = int(any((xi - phi) < range_lo or (xi - phi) > range_hi for xi in x))
    return out, lse, flag
