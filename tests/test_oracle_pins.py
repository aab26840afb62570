"""Pins for the float64 CPU oracle (all CPU-only).

Each test ties the oracle to something other than itself: a value the pages print for a
worked example (tests/golden/), a closed form, an invariant the pages state, a library
conversion, or an independent NumPy brute force. A plausible slip in the oracle (a
dropped term, a wrong sign or index, a transposed operand, the wrong head mapping, the
wrong log base, an open instead of closed range) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import oracle_np
from decode_attention_attn_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _scalar_problem(scores, values):
    """d = 1, one row: q = [1], K = scores, V = values, scale 1 -> logits equal the scores."""
    n = len(scores)
    shape = oracle.make_shape(batch=1, num_q_heads=1, num_kv_heads=1, head_dim=1, dtype="f32",
                              max_seq_len=n)
    q = np.ones((1, 1, 1), np.float32)
    k = np.asarray(scores, np.float32).reshape(1, n, 1, 1)
    v = np.asarray(values, np.float32).reshape(1, n, 1, 1)
    return shape, q, k, v, np.array([n], np.int32)


# ---------------------------------------------------------------------------------------
# Worked examples printed on the pages
# ---------------------------------------------------------------------------------------
def test_handbook_exercise1_final_and_direct_sum():
    g = _golden("handbook_exercise1_online_softmax.json")
    scores = [s for tile in g["tiles"] for s in tile]
    shape, q, k, v, lens = _scalar_problem(scores, g["v"])
    out, lse, _, _ = oracle.decode_attn(shape, q, k, v, None, lens, 1.0)
    tol = g["printed_abs_tolerance"]
    assert abs(out[0, 0] - g["printed"]["final"]) <= tol["final"]
    # the page's "directly" line: the weights e^x sum to 178.6, i.e. lse = ln(178.6)
    assert abs(math.exp(lse[0]) - g["printed"]["direct_weight_sum"]) <= tol["direct_weight_sum"]


def test_handbook_exercise1_tile_states_and_merge():
    g = _golden("handbook_exercise1_online_softmax.json")
    scores = [s for tile in g["tiles"] for s in tile]
    shape, q, k, v, lens = _scalar_problem(scores, g["v"])
    tol = g["printed_abs_tolerance"]
    o1, m1, l1, L1 = oracle.split_partial(shape, q, k, v, None, 0, 0, [0, 1], 1.0)
    p1 = g["printed"]["after_tile1"]
    assert m1 == p1["m"]
    assert abs(l1 - p1["l"]) <= tol["l"]
    assert abs(o1[0] * l1 - p1["O_unnormalised"]) <= tol["O_unnormalised"]
    o2, m2, l2, L2 = oracle.split_partial(shape, q, k, v, None, 0, 0, [2, 3], 1.0)
    o, lse = oracle.lse_merge(np.stack([o1, o2]), [m1, m2], [l1, l2])
    p2 = g["printed"]["after_tile2"]
    # state after the second tile, relative to m' = 5 (the merged maximum)
    assert max(m1, m2) == p2["m"]
    l_merged = math.exp(lse - p2["m"])
    assert abs(l_merged - p2["l"]) <= tol["l"]
    assert abs(o[0] * l_merged - p2["O_unnormalised"]) <= tol["O_unnormalised"]
    assert abs(o[0] - g["printed"]["final"]) <= tol["final"]
    oa, lsea = oracle.lse_merge_alpha(np.stack([o1, o2]), [L1, L2])
    assert abs(oa[0] - o[0]) < 1e-12 and abs(lsea - lse) < 1e-12


def test_fig6_flags_boundaries_and_partitions():
    g = _golden("fdpp_fig6_unified_max_flags.json")
    phi, a, b = g["phi"], g["a"], g["b"]
    for case in g["cases"]:
        vals = case["values"]
        shape, q, k, v, lens = _scalar_problem(vals, [1.0, 2.0, 3.0, 4.0])
        out, lse, flag, margin = oracle.decode_attn(shape, q, k, v, None, lens, 1.0, phi, a, b)
        assert flag[0] == case["flag"], case["name"]
        # the recompute is the synchronised softmax: its reference point is max(y)
        o_s, m_s, l_s, L_s = oracle.split_partial(shape, q, k, v, None, 0, 0, [0, 1, 2, 3], 1.0)
        assert m_s == case["max"]
        split = len(g["partition"][0])
        uo, ulse, uflag, nflag = oracle.unified_row(shape, q, k, v, None, lens, 0, 0, 1.0, phi,
                                                    a, b, split_tokens=split)
        assert uflag == case["flag"]
        assert nflag == sum(case["partition_flags"])
        if not case["flag"]:
            # unflagged: the unified (Eq. 4) and synchronised results agree
            assert abs(uo[0] - out[0, 0]) < 1e-12 and abs(ulse - lse[0]) < 1e-12
    # on-boundary elements (y: 3 - 6 = -3 and 9 - 6 = 3) leave zero margin but no flag
    shape, q, k, v, lens = _scalar_problem([3.0, 6.0, 9.0, 6.0], [1.0, 2.0, 3.0, 4.0])
    _, _, flag, margin = oracle.decode_attn(shape, q, k, v, None, lens, 1.0, phi, a, b)
    assert flag[0] == 0 and margin[0] == 0.0


# ---------------------------------------------------------------------------------------
# Independent brute force on tiny shapes
# ---------------------------------------------------------------------------------------
def _tiny_case(rng, dtype, paged, B, Hq, Hkv, d, lens, page_size, adversarial):
    def draw(shape):
        x = rng.standard_normal(shape).astype(np.float32)
        if adversarial:
            x *= rng.choice([1.0, 30.0, 300.0], size=shape).astype(np.float32)
        t = torch.from_numpy(x).to(workloads.TORCH_DTYPES[dtype])
        return workloads.bits(t)

    q = draw((B, Hq, d))
    if paged:
        pages = [(n + page_size - 1) // page_size for n in lens]
        total = max(sum(pages), 1) + 2            # two spare physical blocks
        perm = rng.permutation(total).astype(np.int32)
        width = max(max(pages), 1)
        table = np.full((B, width), -1, np.int32)
        nxt = 0
        for b, np_ in enumerate(pages):
            table[b, :np_] = perm[nxt:nxt + np_]
            nxt += np_
        kshape = (total, page_size, Hkv, d)
        shape = oracle.make_shape(batch=B, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
                                  dtype=dtype, paged=True, page_size=page_size,
                                  max_blocks_per_seq=width, num_physical_blocks=total)
    else:
        table = None
        cap = max(max(lens), 1) + 3
        kshape = (B, cap, Hkv, d)
        shape = oracle.make_shape(batch=B, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
                                  dtype=dtype, max_seq_len=cap)
    k, v = draw(kshape), draw(kshape)
    return shape, q, k, v, table, np.asarray(lens, np.int32)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("adversarial", [False, True])
def test_brute_force_tiny(dtype, paged, adversarial):
    rng = np.random.default_rng(11 + 7 * paged + 3 * adversarial)
    for B, Hq, Hkv, d, page in [(1, 1, 1, 1, 1), (2, 4, 2, 3, 4), (2, 4, 1, 8, 16), (3, 6, 3, 5, 2)]:
        lens = list(rng.integers(0, 41, size=B))
        lens[0] = max(lens[0], 1)
        shape, q, k, v, table, sl = _tiny_case(rng, dtype, paged, B, Hq, Hkv, d, lens, page,
                                               adversarial)
        scale = 1.0 / math.sqrt(d)
        out, lse, flag, _ = oracle.decode_attn(shape, q, k, v, table, sl, scale, 0.5, -2.0, 2.0)
        ref_o, ref_l, ref_f = oracle_np.reference(q, k, v, dtype, sl, scale, num_kv_heads=Hkv,
                                                  paged=paged, page_size=page, block_table=table,
                                                  phi=0.5, range_lo=-2.0, range_hi=2.0)
        np.testing.assert_allclose(out, ref_o.reshape(-1, d), rtol=1e-11, atol=1e-12)
        finite = np.isfinite(ref_l.ravel())
        np.testing.assert_allclose(lse[finite], ref_l.ravel()[finite], rtol=1e-12, atol=1e-12)
        assert np.all(np.isneginf(lse[~finite]))
        np.testing.assert_array_equal(flag, ref_f.ravel())


# ---------------------------------------------------------------------------------------
# Invariants of the split-KV merge (Flash-Decoding: "The Rescaling and Online Softmax
# Reduction Algorithm"; any partition merges to the unsplit result)
# ---------------------------------------------------------------------------------------
def _random_problem(seed, dtype="bf16", n=200, d=16, Hq=4, Hkv=2, paged=True, page=16):
    rng = np.random.default_rng(seed)
    return _tiny_case(rng, dtype, paged, 1, Hq, Hkv, d, [n], page, False)


def test_single_split_equals_unsplit():
    shape, q, k, v, table, sl = _random_problem(1)
    out, lse, _, _ = oracle.decode_attn(shape, q, k, v, table, sl, 0.25)
    for h in range(shape.num_q_heads):
        o_s, m_s, l_s, L_s = oracle.split_partial(shape, q, k, v, table, 0, h,
                                                  np.arange(sl[0]), 0.25)
        np.testing.assert_allclose(o_s, out[h], rtol=1e-13, atol=1e-15)
        assert abs(L_s - lse[h]) < 1e-12
        o, l = oracle.lse_merge(o_s[None], [m_s], [l_s])
        np.testing.assert_allclose(o, out[h], rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("seed", [2, 3, 4])
def test_any_partition_merges_to_unsplit(seed):
    shape, q, k, v, table, sl = _random_problem(seed, n=257)
    rng = np.random.default_rng(100 + seed)
    out, lse, _, _ = oracle.decode_attn(shape, q, k, v, table, sl, 0.3)
    n = int(sl[0])
    for trial in range(6):
        if trial % 2 == 0:   # contiguous splits, some possibly empty
            cuts = np.sort(rng.integers(0, n + 1, size=rng.integers(1, 9)))
            bounds = [0, *cuts.tolist(), n]
            parts = [np.arange(bounds[i], bounds[i + 1]) for i in range(len(bounds) - 1)]
        else:                # arbitrary disjoint subsets covering every token
            lab = rng.integers(0, 5, size=n)
            parts = [np.flatnonzero(lab == j) for j in range(6)]   # label 5 stays empty
        for h in range(shape.num_q_heads):
            res = [oracle.split_partial(shape, q, k, v, table, 0, h, p, 0.3) for p in parts]
            o_s = np.stack([r[0] for r in res])
            o, l = oracle.lse_merge(o_s, [r[1] for r in res], [r[2] for r in res])
            oa, la = oracle.lse_merge_alpha(o_s, [r[3] for r in res])
            np.testing.assert_allclose(o, out[h], rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(oa, out[h], rtol=1e-12, atol=1e-14)
            assert abs(l - lse[h]) < 1e-12 and abs(la - lse[h]) < 1e-12


def test_all_empty_merge_is_zero_and_neg_inf():
    o, lse = oracle.lse_merge(np.zeros((3, 4)), [-math.inf] * 3, [0.0] * 3)
    assert np.all(o == 0) and lse == -math.inf
    o, lse = oracle.lse_merge_alpha(np.zeros((3, 4)), [-math.inf] * 3)
    assert np.all(o == 0) and lse == -math.inf


# ---------------------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------------------
def test_constant_v_rows_give_that_v():
    rng = np.random.default_rng(5)
    n, d, cap = 300, 8, 300
    shape = oracle.make_shape(batch=1, num_q_heads=2, num_kv_heads=1, head_dim=d, dtype="f32",
                              max_seq_len=cap)
    q = (rng.standard_normal((1, 2, d)) * 20).astype(np.float32)    # very peaked logits
    k = rng.standard_normal((1, cap, 1, d)).astype(np.float32)
    row = rng.standard_normal(d).astype(np.float32)
    v = np.broadcast_to(row, (1, cap, 1, d)).copy()
    out, _, _, _ = oracle.decode_attn(shape, q, k, v, None, np.array([n], np.int32), 1.0)
    np.testing.assert_allclose(out, np.stack([row, row]).astype(np.float64), rtol=1e-14, atol=1e-15)


def test_uniform_logits_give_mean_v_and_ln_n():
    rng = np.random.default_rng(6)
    n, d = 123, 8
    shape = oracle.make_shape(batch=1, num_q_heads=1, num_kv_heads=1, head_dim=d, dtype="f32",
                              max_seq_len=n)
    q = np.zeros((1, 1, d), np.float32)
    k = rng.standard_normal((1, n, 1, d)).astype(np.float32)
    v = rng.standard_normal((1, n, 1, d)).astype(np.float32)
    out, lse, _, _ = oracle.decode_attn(shape, q, k, v, None, np.array([n], np.int32), 0.7)
    np.testing.assert_allclose(out[0], v[0, :n, 0].astype(np.float64).mean(axis=0), rtol=1e-12,
                               atol=1e-14)
    assert abs(lse[0] - math.log(n)) < 1e-13     # natural log, not log2


def test_one_hot_logit_through_shuffled_pages_and_gqa_mapping():
    """A large logit at one known token per KV head selects that token's V row.

    Pins the block-table gather (the token is found at slot t % page of physical block
    table[t / page]) and the GQA head mapping kv_head = h / (H_q / H_kv): query heads 0, 1
    share KV head 0 and heads 2, 3 share KV head 1 (a mapping h % H_kv would pair 0 with 2).
    """
    rng = np.random.default_rng(8)
    P, n, d, Hq, Hkv = 4, 37, 8, 4, 2
    pages = (n + P - 1) // P
    total = pages + 3
    perm = rng.permutation(total).astype(np.int32)
    table = perm[:pages].reshape(1, pages)
    shape = oracle.make_shape(batch=1, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, dtype="f32",
                              paged=True, page_size=P, max_blocks_per_seq=pages,
                              num_physical_blocks=total)
    u = rng.standard_normal(d).astype(np.float32)
    u /= np.linalg.norm(u)
    q = np.broadcast_to(u, (1, Hq, d)).copy()
    k = (rng.standard_normal((total, P, Hkv, d)) * 0.01).astype(np.float32)
    v = rng.standard_normal((total, P, Hkv, d)).astype(np.float32)
    targets = {0: 29, 1: 6}            # KV head -> its one-hot token
    c = 60.0
    for kvh, t in targets.items():
        k[table[0, t // P], t % P, kvh] = c * u
    out, lse, _, _ = oracle.decode_attn(shape, q, k, v, table, np.array([n], np.int32), 1.0)
    for h in range(Hq):
        kvh = h // (Hq // Hkv)
        t = targets[kvh]
        want = v[table[0, t // P], t % P, kvh].astype(np.float64)
        x_star = float(np.dot(u.astype(np.float64), (c * u).astype(np.float32).astype(np.float64)))
        # every other logit is below 0.01 * sqrt(d) * 5 < 1 in magnitude: gap > 58
        assert np.max(np.abs(out[h] - want)) < n * math.exp(-(x_star - 1.0)) * 10
        assert abs(lse[h] - x_star) < n * math.exp(-(x_star - 1.0))


def test_unified_equals_synchronised_when_unflagged():
    shape, q, k, v, table, sl = _random_problem(9, n=180)
    out, lse, flag, _ = oracle.decode_attn(shape, q, k, v, table, sl, 0.25, -3.9, -64, 64)
    assert not flag.any()
    for h in range(shape.num_q_heads):
        for split in (0, 7, 64):
            uo, ulse, uflag, nflag = oracle.unified_row(shape, q, k, v, table, sl, 0, h, 0.25,
                                                        -3.9, -64.0, 64.0, split_tokens=split)
            assert uflag == 0 and nflag == 0
            np.testing.assert_allclose(uo, out[h], rtol=1e-12, atol=1e-14)
            assert abs(ulse - lse[h]) < 1e-12


def test_unified_overflow_is_flagged():
    """x - phi far above hi: the unified form would overflow; the oracle flags the row."""
    shape, q, k, v, lens = _scalar_problem([1.0, 900.0, 2.0], [1.0, 2.0, 3.0])
    out, lse, flag, margin = oracle.decode_attn(shape, q, k, v, None, lens, 1.0, 0.0, -64, 64)
    assert flag[0] == 1 and margin[0] == 900.0 - 64.0
    assert abs(out[0, 0] - 2.0) < 1e-12 and abs(lse[0] - 900.0) < 1e-12
    uo, ulse, uflag, nflag = oracle.unified_row(shape, q, k, v, None, lens, 0, 0, 1.0, 0.0,
                                                -64.0, 64.0, split_tokens=2)
    assert uflag == 1 and nflag == 1
    assert not np.isfinite(uo[0])     # e^900 overflows float64: why the row is recomputed


def test_underflow_is_flagged():
    """All logits far below phi: every exponential underflows; the lower bound flags it."""
    shape, q, k, v, lens = _scalar_problem([-900.0, -901.0], [1.0, 3.0])
    out, lse, flag, _ = oracle.decode_attn(shape, q, k, v, None, lens, 1.0, 0.0, -64, 64)
    assert flag[0] == 1 and np.isfinite(out).all()
    w = 1.0 / (1.0 + math.exp(-1.0))
    assert abs(out[0, 0] - (w * 1.0 + (1 - w) * 3.0)) < 1e-12


def test_empty_row():
    shape, q, k, v, _ = _scalar_problem([1.0, 2.0], [3.0, 4.0])
    out, lse, flag, margin = oracle.decode_attn(shape, q, k, v, None, np.array([0], np.int32), 1.0)
    assert out[0, 0] == 0.0 and lse[0] == -math.inf and flag[0] == 0 and margin[0] == math.inf


# ---------------------------------------------------------------------------------------
# Exact decoding and gather offsets against library routines
# ---------------------------------------------------------------------------------------
def test_fp16_and_bf16_decoding_matches_library_conversions():
    allbits = np.arange(65536, dtype=np.uint16)
    for dtype, lib_vals in (
        ("f16", allbits.view(np.float16).astype(np.float64)),
        ("bf16", torch.from_numpy(allbits.view(np.int16)).view(torch.bfloat16)
         .to(torch.float64).numpy()),
    ):
        got = np.array([oracle.load(dtype, allbits, i) for i in range(65536)])
        nan = np.isnan(lib_vals)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan], lib_vals[~nan])
        assert np.array_equal(np.signbit(got[~nan]), np.signbit(lib_vals[~nan]))


def test_gather_offsets_match_ravel_multi_index():
    rng = np.random.default_rng(12)
    B, Hkv, d, P = 3, 2, 8, 4
    lens = np.array([5, 0, 13], np.int32)
    pages = (lens + P - 1) // P
    total = int(pages.sum()) + 1
    perm = rng.permutation(total).astype(np.int32)
    width = int(pages.max())
    table = np.full((B, width), -1, np.int32)
    nxt = 0
    for b in range(B):
        table[b, :pages[b]] = perm[nxt:nxt + pages[b]]
        nxt += pages[b]
    shape = oracle.make_shape(batch=B, num_q_heads=2 * Hkv, num_kv_heads=Hkv, head_dim=d,
                              dtype="bf16", paged=True, page_size=P, max_blocks_per_seq=width,
                              num_physical_blocks=total)
    offs = oracle.gather_offsets(shape, table, lens)
    cache_shape = (total, P, Hkv, d)
    for b in range(B):
        for kvh in range(Hkv):
            for t in range(width * P):
                want = (np.ravel_multi_index((table[b, t // P], t % P, kvh, 0), cache_shape)
                        if t < lens[b] else -1)
                assert offs[b, kvh, t] == want
    cshape = oracle.make_shape(batch=B, num_q_heads=Hkv, num_kv_heads=Hkv, head_dim=d,
                               dtype="bf16", max_seq_len=16)
    offs = oracle.gather_offsets(cshape, None, lens)
    for b in range(B):
        for kvh in range(Hkv):
            for t in range(16):
                want = (np.ravel_multi_index((b, t, kvh, 0), (B, 16, Hkv, d))
                        if t < lens[b] else -1)
                assert offs[b, kvh, t] == want


def test_out_of_pool_block_table_entry_is_rejected():
    shape = oracle.make_shape(batch=1, num_q_heads=1, num_kv_heads=1, head_dim=2, dtype="f32",
                              paged=True, page_size=2, max_blocks_per_seq=2,
                              num_physical_blocks=2)
    q = np.ones((1, 1, 2), np.float32)
    k = np.ones((2, 2, 1, 2), np.float32)
    table = np.array([[1, 5]], np.int32)
    with pytest.raises(ValueError):
        oracle.decode_attn(shape, q, k, k, table, np.array([4], np.int32), 1.0)
    out, _, _, _ = oracle.decode_attn(shape, q, k, k, table, np.array([2], np.int32), 1.0)
    assert np.all(out == 1.0)


# ---------------------------------------------------------------------------------------
# The logit values behind the choice of phi ("FlashDecoding++", Fig. 5)
# ---------------------------------------------------------------------------------------
def test_logits_of_one_hot_keys_are_single_products():
    """K row t = c_t e_(t mod d): the scaled logit of head h is scale * c_t * q[h, t mod d]."""
    rng = np.random.default_rng(31)
    d, Hq, Hkv, n = 8, 4, 2, 11
    shape = oracle.make_shape(batch=1, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, dtype="f32",
                              max_seq_len=n)
    q = rng.standard_normal((1, Hq, d)).astype(np.float32)
    c = rng.standard_normal(n).astype(np.float32)
    k = np.zeros((1, n, Hkv, d), np.float32)
    for t in range(n):
        k[0, t, :, t % d] = c[t]
    x = oracle.logits(shape, q, k, None, np.array([n], np.int32), 0.5)
    assert x.shape == (Hq * n,)
    for h in range(Hq):
        for t in range(n):
            assert x[h * n + t] == 0.5 * float(c[t]) * float(q[0, h, t % d])


@pytest.mark.parametrize("paged", [False, True])
def test_logits_agree_with_the_attention_oracle(paged):
    """Each row's logits reproduce the (separately pinned) attention oracle: their
    log-sum-exp is its lse, row by row, in the documented order; in the paged case that
    also ties them to the block-table gather the attention oracle uses."""
    rng = np.random.default_rng(32)
    lens = [5, 0, 23, 9]
    shape, q, k, v, table, sl = _tiny_case(rng, "bf16", paged, 4, 4, 2, 16, lens, 4, False)
    x = oracle.logits(shape, q, k, table, sl, 0.3)
    out, lse, _, _ = oracle.decode_attn(shape, q, k, v, table, sl, 0.3)
    at = 0
    for b, n in enumerate(lens):
        for h in range(4):
            r = b * 4 + h
            xs = x[at:at + n]
            at += n
            if n == 0:
                assert lse[r] == -math.inf
                continue
            m = xs.max()
            assert abs(m + math.log(np.exp(xs - m).sum()) - lse[r]) < 1e-12
    assert at == x.size


# ---------------------------------------------------------------------------------------
# FP8 (E4M3) K / V caches ("FlashAttention and inference kernels", "A paged decode
# attention kernel (with GQA)": the cache is BF16 or FP8, converted on read)
# ---------------------------------------------------------------------------------------
def test_e4m3_decoding_matches_library_conversion_and_hand_values():
    codes = np.arange(256, dtype=np.uint8)
    got = np.array([oracle.load("e4m3", codes, i) for i in range(256)])
    lib_vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(lib_vals)
    assert np.array_equal(np.isnan(got), nan) and list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.array_equal(got[~nan], lib_vals[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(lib_vals[~nan]))
    # by hand from the format: 1.0, the largest value, the smallest normal and subnormal,
    # a subnormal with two mantissa bits, negative zero
    for c, want in [(0x38, 1.0), (0x7E, 448.0), (0x08, 2.0 ** -6), (0x01, 2.0 ** -9),
                    (0x06, 6 * 2.0 ** -9), (0xB8, -1.0), (0x3D, 1.625)]:
        assert got[c] == want, (hex(c), got[c], want)
    assert got[0x80] == 0.0 and np.signbit(got[0x80])


def _fp8_codes(rng, shape):
    """Random E4M3 codes, every one but the two NaNs possible."""
    mag = rng.integers(0, 0x7F, size=shape)
    return (mag | (rng.integers(0, 2, size=shape) << 7)).astype(np.uint8)


def _tiny_fp8_case(rng, paged, B, Hq, Hkv, d, lens, page, k_scale, v_scale):
    shape, q, _, _, table, sl = _tiny_case(rng, "bf16", paged, B, Hq, Hkv, d, lens, page, False)
    if paged:
        kshape = (shape.num_physical_blocks, page, Hkv, d)
    else:
        kshape = (B, shape.max_seq_len, Hkv, d)
    shape.kv_e4m3, shape.k_scale, shape.v_scale = 1, k_scale, v_scale
    return shape, q, _fp8_codes(rng, kshape), _fp8_codes(rng, kshape), table, sl


@pytest.mark.parametrize("paged", [False, True])
def test_brute_force_tiny_fp8_kv(paged):
    rng = np.random.default_rng(51 + paged)
    for B, Hq, Hkv, d, page in [(1, 1, 1, 1, 1), (2, 4, 2, 3, 4), (2, 8, 1, 8, 16)]:
        lens = list(rng.integers(0, 41, size=B))
        lens[0] = max(lens[0], 1)
        ks, vs = 0.0137, 0.21
        shape, q, k, v, table, sl = _tiny_fp8_case(rng, paged, B, Hq, Hkv, d, lens, page, ks, vs)
        scale = 1.0 / math.sqrt(d)
        out, lse, flag, _ = oracle.decode_attn(shape, q, k, v, table, sl, scale, 0.5, -2.0, 2.0)
        ref_o, ref_l, ref_f = oracle_np.reference(q, k, v, "bf16", sl, scale, num_kv_heads=Hkv,
                                                  paged=paged, page_size=page, block_table=table,
                                                  phi=0.5, range_lo=-2.0, range_hi=2.0,
                                                  kv_dtype="e4m3", k_scale=ks, v_scale=vs)
        np.testing.assert_allclose(out, ref_o.reshape(-1, d), rtol=1e-11, atol=1e-12)
        finite = np.isfinite(ref_l.ravel())
        np.testing.assert_allclose(lse[finite], ref_l.ravel()[finite], rtol=1e-12, atol=1e-12)
        np.testing.assert_array_equal(flag, ref_f.ravel())


def test_fp8_scales_act_linearly():
    """Doubling k_scale is doubling the softmax scale (the logits are scale * k_scale *
    q . code); doubling v_scale doubles the output and leaves the lse alone. Both by powers
    of two, so the results agree bit for bit."""
    rng = np.random.default_rng(53)
    shape, q, k, v, table, sl = _tiny_fp8_case(rng, True, 2, 4, 2, 16, [37, 20], 8, 0.01, 0.3)
    base = oracle.decode_attn(shape, q, k, v, table, sl, 0.25)
    shape.k_scale = 0.02
    twice_k = oracle.decode_attn(shape, q, k, v, table, sl, 0.125)
    assert np.array_equal(base[0], twice_k[0]) and np.array_equal(base[1], twice_k[1])
    shape.k_scale, shape.v_scale = 0.01, 0.6
    twice_v = oracle.decode_attn(shape, q, k, v, table, sl, 0.25)
    assert np.array_equal(2.0 * base[0], twice_v[0]) and np.array_equal(base[1], twice_v[1])


def test_oracle_rejects_bad_fp8_shapes():
    rng = np.random.default_rng(54)
    shape, q, k, v, table, sl = _tiny_fp8_case(rng, False, 1, 2, 1, 8, [5], 4, 0.1, 0.2)
    for field, bad in (("kv_e4m3", 2), ("k_scale", math.nan), ("v_scale", math.inf)):
        saved = getattr(shape, field)
        setattr(shape, field, bad)
        with pytest.raises(ValueError):
            oracle.decode_attn(shape, q, k, v, table, sl, 0.5)
        setattr(shape, field, saved)
    oracle.decode_attn(shape, q, k, v, table, sl, 0.5)   # restored: accepted


def test_fp8_workload_quantisation():
    """The FP8 recipe: one scale per tensor, max |x| / 448, so the largest code is 448 and
    code * scale stays within E4M3's half-ulp (2^-4 relative, or 2^-10 * scale absolute for
    subnormals) of the fp32 draw."""
    x = torch.randn((3, 40, 2, 16), generator=torch.Generator().manual_seed(5))
    codes, scale = workloads.quantize_e4m3(x)
    assert codes.dtype == torch.uint8 and scale == float(np.float32(x.abs().max() / 448.0))
    vals = codes.view(torch.float8_e4m3fn).to(torch.float64)
    assert vals.abs().max() == 448.0
    err = (vals * scale - x.double()).abs()
    bound = torch.maximum(x.double().abs() * 2.0 ** -4, torch.full_like(err, 2.0 ** -10 * scale))
    assert bool((err <= bound * (1 + 1e-6)).all())
