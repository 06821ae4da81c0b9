"""Pins of the CPU oracle against what the pages and mathematics fix.

Each test checks the oracle against something other than itself: the values
printed in the pages' worked example, closed forms, brute force on tiny
inputs, special cases that reduce to a library routine (numpy matmul / sort,
scipy's logistic), and exact invariants.  None needs a GPU.
"""
import itertools
import math
from pathlib import Path

import numpy as np
import pytest
from scipy.special import expit

import oracle
import synth

GOLDEN = Path(__file__).parent / "golden"


def _golden(name):
    out = {}
    for line in (GOLDEN / name).read_text().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        k, *v = line.split()
        out[k] = v
    return out


# --- int4 storage format ("25GB 内存上运行 GLM 5.2 744B", section 06) --------

def test_unpack_matches_printed_worked_example():
    g = _golden("int4_unpack_gate_proj.txt")
    raw = np.array([int(b, 16) for b in g["first_bytes"]], dtype=np.uint8)
    q = oracle.unpack_int4(raw, 2 * raw.size)
    # the page prints the low nibbles: they are the even-indexed elements
    assert q[0::2].tolist() == [int(v) for v in g["low_nibbles"]]


def test_size_identity_from_printed_tensor():
    g = _golden("int4_unpack_gate_proj.txt")
    rows, nbytes, cols = int(g["rows"][0]), int(g["packed_bytes"][0]), int(g["implied_cols"][0])
    assert rows * ((cols + 1) // 2) == nbytes
    assert nbytes * 2 // rows == cols


def test_nibble_order_low_first():
    # byte 0x4B: low nibble 0xB -> element 0 = 11 - 8 = 3; high nibble 4 -> element 1 = -4
    assert oracle.unpack_int4(np.array([0x4B], np.uint8), 2).tolist() == [3, -4]
    # stored value 8 is zero; 0 is -8; 15 is 7
    assert oracle.unpack_int4(np.array([0x88, 0xF0], np.uint8), 4).tolist() == [0, 0, -8, 7]


def test_expert_bytes_match_the_pages_19MB_figure():
    # one GLM-5.2 expert: gate/up [2048, 6144], down [6144, 2048], int4 + per-row f32 scale
    b = synth.slab_bytes(6144, 2048) + 4 * synth.scale_count(6144, 2048)
    assert b == 18_915_328
    assert abs(b / 1e6 - 19) < 0.2
    # per-expert bytes of the other layer shapes (b_exp = 2 I ceil(H/2) + H ceil(I/2) + 4 (2I + H))
    assert synth.slab_bytes(256, 128) + 4 * synth.scale_count(256, 128) == 51_200
    assert synth.slab_bytes(2048, 1024) + 4 * synth.scale_count(2048, 1024) == 3_162_112
    assert synth.slab_bytes(2048, 512) + 4 * synth.scale_count(2048, 512) == 1_585_152


def test_quantize_roundtrip_exact_on_integer_rows():
    rng = np.random.default_rng(7)
    O, I = 6, 33
    q = rng.integers(-7, 8, size=(O, I))
    q[:, 0] = 7            # amax = 7 * s0 so the quantiser's scale is s0 exactly
    s0 = 2.0 ** -rng.integers(3, 9, size=O)
    w = (q * s0[:, None]).astype(np.float32)
    q4, s = oracle.quantize_int4(w)
    assert np.array_equal(s, s0.astype(np.float32))
    for o in range(O):
        assert oracle.unpack_int4(q4[o], I).tolist() == q[o].tolist()
    # I odd: the pad nibble of the last byte is stored as 8 (value 0)
    assert np.all(q4[:, -1] >> 4 == 8)


def test_quantize_rounds_half_to_even_and_clips():
    # amax = 7 -> s = 1: rint(2.5)=2, rint(3.5)=4, rint(-2.5)=-2, rint(0.5)=0
    w = np.array([[2.5, 3.5, -2.5, 0.5, 7.0, -6.5]], np.float32)
    q4, s = oracle.quantize_int4(w)
    assert s[0] == 1.0
    assert oracle.unpack_int4(q4[0], 6).tolist() == [2, 4, -2, 0, 7, -6]
    # all-zero row: scale floor 1e-8, every stored nibble 8
    q4, s = oracle.quantize_int4(np.zeros((1, 4), np.float32))
    assert s[0] == np.float32(1e-8) and q4.tolist() == [[0x88, 0x88]]


# --- SwiGLU expert (section 11 / section 04) ---------------------------------

def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(1.0) == pytest.approx(1.0 / (1.0 + math.e ** -1), rel=1e-15)
    assert oracle.silu(-1.0) == pytest.approx(-1.0 / (1.0 + math.e), rel=1e-15)
    assert oracle.silu(40.0) == pytest.approx(40.0, rel=1e-15)
    for v in (-7.5, -0.3, 0.2, 3.0):
        assert oracle.silu(v) == pytest.approx(v * expit(v), rel=1e-14)


def _pack(q_rows):
    """Pack integer rows in [-8, 7] by hand (stored q+8, even element low)."""
    q = np.asarray(q_rows)
    O, n = q.shape
    out = np.full((O, (n + 1) // 2), 0x88, np.uint8)
    for o in range(O):
        for i in range(n):
            b = out[o, i // 2]
            if i % 2 == 0:
                out[o, i // 2] = (b & 0xF0) | (q[o, i] + 8)
            else:
                out[o, i // 2] = (b & 0x0F) | ((q[o, i] + 8) << 4)
    return out


def test_expert_hand_2x2():
    # H = I = 2.  gate q = [[1,0],[0,-1]] sg=[1,.5]; up q = [[2,1],[-3,0]] su=[1,2];
    # down q = [[1,1],[-1,2]] sd=[1,.25]; x = [1, 2].
    # g = [1, -1], u = [4, -6], h = [4 silu(1), -6 silu(-1)] = [2.92423431452, 1.61364852822]
    # d = [h0 + h1, (-h0 + 2 h1)/4] = [4.53788284274, 0.0757656854800]
    slab = np.concatenate([_pack([[1, 0], [0, -1]]).ravel(), _pack([[2, 1], [-3, 0]]).ravel(),
                           _pack([[1, 1], [-1, 2]]).ravel()])
    scale = np.array([1, .5, 1, 2, 1, .25], np.float32)
    d, h = oracle.expert(2, 2, slab, scale, np.array([1.0, 2.0]))
    assert h == pytest.approx([2.9242343145200196, 1.6136485282199706], rel=1e-13)
    assert d == pytest.approx([4.53788284273999, 0.07576568547998022], rel=1e-12)


def _dequant(q4, scale, O, n):
    q = np.stack([oracle.unpack_int4(q4[o], n) for o in range(O)]).astype(np.float64)
    return q * scale.astype(np.float64)[:, None]


def _dense_swiglu(H, I, slab, scale, x):
    rb = (H + 1) // 2
    g4 = slab[:I * rb].reshape(I, rb)
    u4 = slab[I * rb:2 * I * rb].reshape(I, rb)
    d4 = slab[2 * I * rb:].reshape(H, (I + 1) // 2)
    Wg = _dequant(g4, scale[:I], I, H)
    Wu = _dequant(u4, scale[I:2 * I], I, H)
    Wd = _dequant(d4, scale[2 * I:], H, I)
    g = Wg @ x
    return Wd @ (g * expit(g) * (Wu @ x))


@pytest.mark.parametrize("H,I", [(64, 32), (7, 5), (32, 96)])
def test_expert_equals_dense_swiglu(H, I):
    rng = np.random.default_rng(H * 100 + I)
    slab = rng.integers(0, 256, synth.slab_bytes(H, I), dtype=np.uint8)
    if H % 2:   # pad nibbles hold 8
        rb = (H + 1) // 2
        m = slab[:2 * I * rb].reshape(2 * I, rb)
        m[:, -1] = (m[:, -1] & 0x0F) | 0x80
    if I % 2:
        d = slab[2 * I * ((H + 1) // 2):].reshape(H, (I + 1) // 2)
        d[:, -1] = (d[:, -1] & 0x0F) | 0x80
    scale = rng.uniform(0.005, 0.02, 2 * I + H).astype(np.float32)
    x = rng.standard_normal(H)
    d, _ = oracle.expert(H, I, slab, scale, x)
    np.testing.assert_allclose(d, _dense_swiglu(H, I, slab, scale, x), rtol=1e-10, atol=1e-12)


# --- int8 per-row experts (reader.mx section 03, the OLMoE engine) -------------------

def test_int8_quantize_roundtrip_exact_on_integer_rows():
    rng = np.random.default_rng(41)
    O, I = 6, 40
    k = rng.integers(-127, 128, (O, I))
    k[:, 0] = 127                                  # amax / 127 is the power-of-two scale
    s = 2.0 ** rng.integers(-12, -4, O)
    q, sc = oracle.quantize_int8((k * s[:, None]).astype(np.float32))
    assert np.array_equal(q, k.astype(np.int8))
    np.testing.assert_array_equal(sc, s.astype(np.float32))
    q0, s0 = oracle.quantize_int8(np.zeros((2, 8), np.float32))   # zero rows: scale floor 1e-8
    assert not q0.any() and np.all(s0 == np.float32(1e-8))


def _int8_slab(rng, H, I):
    return rng.integers(-128, 128, 3 * I * H).astype(np.int8).view(np.uint8)


@pytest.mark.parametrize("H,I", [(64, 32), (7, 5)])
def test_int8_expert_equals_dense_swiglu(H, I):
    rng = np.random.default_rng(H + 7 * I)
    slab = _int8_slab(rng, H, I)
    scale = rng.uniform(0.005, 0.02, 2 * I + H).astype(np.float32)
    x = rng.standard_normal(H)
    q = slab.view(np.int8).astype(np.float64)
    Wg = q[:I * H].reshape(I, H) * scale[:I, None]
    Wu = q[I * H:2 * I * H].reshape(I, H) * scale[I:2 * I, None]
    Wd = q[2 * I * H:].reshape(H, I) * scale[2 * I:, None]
    g = Wg @ x
    want = Wd @ (g * expit(g) * (Wu @ x))
    d, _ = oracle.expert(H, I, slab, scale, x, fmt=oracle.FORMAT_INT8)
    np.testing.assert_allclose(d, want, rtol=1e-10, atol=1e-12)


def test_int8_and_int4_agree_on_int4_values():
    # the same integer weights in [-8, 7] stored in both formats give the same expert exactly
    rng = np.random.default_rng(5)
    H, I = 16, 8
    vals = [rng.integers(-8, 8, (I, H)), rng.integers(-8, 8, (I, H)), rng.integers(-8, 8, (H, I))]
    def pack4(m):
        m = m + 8
        return (m[:, 0::2] | (m[:, 1::2] << 4)).astype(np.uint8).ravel()
    slab4 = np.concatenate([pack4(v) for v in vals])
    slab8 = np.concatenate([v.astype(np.int8).ravel() for v in vals]).view(np.uint8)
    scale = rng.uniform(0.005, 0.02, 2 * I + H).astype(np.float32)
    x = rng.standard_normal(H)
    d4, h4 = oracle.expert(H, I, slab4, scale, x)
    d8, h8 = oracle.expert(H, I, slab8, scale, x, fmt=oracle.FORMAT_INT8)
    assert np.array_equal(d4, d8) and np.array_equal(h4, h8)


def test_int8_layer_single_expert_and_shared_format():
    rng = np.random.default_rng(9)
    H, I = 24, 16
    slab = _int8_slab(rng, H, I)
    scale = rng.uniform(0.005, 0.02, 2 * I + H).astype(np.float32)
    sh = _int8_slab(rng, H, I)
    shs = rng.uniform(0.005, 0.02, 2 * I + H).astype(np.float32)
    x = rng.standard_normal(H)
    W = rng.normal(0, 0.1, (1, H)).astype(np.float32)
    cfg = oracle.make_cfg(H, 1, 1, I, 1, I, routed_scale=2.5, expert_format=oracle.FORMAT_INT8,
                          shared_format=oracle.FORMAT_INT8)
    ref = oracle.LayerRef(cfg, W, np.zeros(1, np.float32), [slab], [scale], sh, shs)
    y, idx, w, _ = ref.token(x)
    d, _ = oracle.expert(H, I, slab, scale, x, fmt=oracle.FORMAT_INT8)
    ds, _ = oracle.expert(H, I, sh, shs, x, fmt=oracle.FORMAT_INT8)
    np.testing.assert_allclose(y, w[0] * d + ds, rtol=1e-12, atol=1e-14)
    assert w[0] == pytest.approx(2.5, rel=1e-15)


# --- int4 affine group-64 (Edge0 article, section 三) -----------------------------------

def test_g64_expert_bytes_match_the_pages_1_77MB_figure():
    # 35B-class expert (H 2048, I 512): int4 payload plus one float16 (scale, bias) per 64
    b = synth.slab_bytes(2048, 512, 2) + 4 * synth.scale_count(2048, 512, 2)
    assert b == 1_572_864 + 196_608 == 1_769_472
    assert round(b / 1e6, 2) == 1.77


def _g64_pairs(s, b):
    s16, b16 = np.asarray(s, np.float16), np.asarray(b, np.float16)
    return (s16.view(np.uint16).astype(np.uint32) | (b16.view(np.uint16).astype(np.uint32) << 16)).view(np.float32)


def _g64_dense(slab, pairs, O, n):
    q = np.zeros((O, n))
    q[:, 0::2] = (slab.reshape(O, n // 2) & 15)
    q[:, 1::2] = (slab.reshape(O, n // 2) >> 4)
    u = pairs.view(np.uint32)
    s = (u & 0xFFFF).astype(np.uint16).view(np.float16).astype(np.float64).reshape(O, n // 64)
    b = (u >> 16).astype(np.uint16).view(np.float16).astype(np.float64).reshape(O, n // 64)
    return q * np.repeat(s, 64, 1) + np.repeat(b, 64, 1)


def test_g64_expert_equals_dense_swiglu():
    rng = np.random.default_rng(17)
    H, I = 128, 64
    slab = rng.integers(0, 256, synth.slab_bytes(H, I, 2), dtype=np.uint8)
    ng = [I * H // 64, I * H // 64, H * I // 64]
    s = rng.uniform(0.005, 0.02, sum(ng))
    pairs = _g64_pairs(s, -s * rng.uniform(7.5, 8.5, sum(ng)))
    x = rng.standard_normal(H)
    o1, o2 = I * H // 2, 2 * I * H // 2
    Wg = _g64_dense(slab[:o1], pairs[:ng[0]], I, H)
    Wu = _g64_dense(slab[o1:o2], pairs[ng[0]:ng[0] + ng[1]], I, H)
    Wd = _g64_dense(slab[o2:], pairs[ng[0] + ng[1]:], H, I)
    g = Wg @ x
    want = Wd @ (g * expit(g) * (Wu @ x))
    d, _ = oracle.expert(H, I, slab, pairs, x, fmt=oracle.FORMAT_G64)
    np.testing.assert_allclose(d, want, rtol=1e-10, atol=1e-12)


def test_g64_with_bias_minus_8s_is_the_symmetric_int4_expert():
    # u - 8 = q: with b = -8 s in every group of a row, affine = symmetric int4 with scale s
    rng = np.random.default_rng(23)
    H, I = 128, 64
    slab = rng.integers(0, 256, synth.slab_bytes(H, I), dtype=np.uint8)
    row_s = np.float16(rng.uniform(0.005, 0.02, 2 * I + H)).astype(np.float32)   # f16-exact scales
    per_row = np.concatenate([np.repeat(row_s[:I], H // 64), np.repeat(row_s[I:2 * I], H // 64),
                              np.repeat(row_s[2 * I:], I // 64)])
    pairs = _g64_pairs(per_row, -8 * per_row)
    x = rng.standard_normal(H)
    d4, h4 = oracle.expert(H, I, slab, row_s, x)
    dg, hg = oracle.expert(H, I, slab, pairs, x, fmt=oracle.FORMAT_G64)
    np.testing.assert_allclose(hg, h4, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(dg, d4, rtol=1e-12, atol=1e-14)


# --- router (section 11; Edge0 section 七) ------------------------------------

def _route_scores(c_values, K, x=None):
    """Route with W = 0, so sigmoid = 0.5 everywhere and selection score = 0.5 + b."""
    E = len(c_values)
    H = 4
    cfg = oracle.make_cfg(H, E, K, 8, routed_scale=1.0)
    W = np.zeros((E, H), np.float32)
    b = (np.asarray(c_values, np.float64) - 0.5).astype(np.float32)
    return oracle.route(cfg, W, b, np.ones(H) if x is None else x)


def test_topk_equals_best_subset_bruteforce():
    rng = np.random.default_rng(3)
    for trial in range(40):
        E = int(rng.integers(2, 9))
        K = int(rng.integers(1, E + 1))
        c = rng.uniform(-1, 1, E).astype(np.float32)
        idx, _, margin, sc = _route_scores(c, K)
        choice = sc[2]
        best = max(itertools.combinations(range(E), K), key=lambda S: sum(choice[list(S)]))
        assert sorted(idx.tolist()) == sorted(best)
        assert all(choice[idx[i]] >= choice[idx[i + 1]] for i in range(K - 1))
        if K < E:
            srt = np.sort(choice)[::-1]
            assert margin == srt[K - 1] - srt[K]
        else:
            assert margin == math.inf


def test_topk_ties_lowest_index_wins():
    c = [0.0, 0.2, 0.2, 0.1, 0.2]
    assert _route_scores(c, 1)[0].tolist() == [1]
    assert _route_scores(c, 2)[0].tolist() == [1, 2]
    assert _route_scores(c, 3)[0].tolist() == [1, 2, 4]
    assert _route_scores(c, 4)[0].tolist() == [1, 2, 4, 3]
    assert _route_scores([0.3] * 6, 4)[0].tolist() == [0, 1, 2, 3]


def test_topk_e_equals_k_selects_all():
    idx, _, margin, _ = _route_scores([0.1, 0.4, -0.2, 0.3], 4)
    assert idx.tolist() == [1, 3, 0, 2] and margin == math.inf


def test_zero_bias_is_topk_of_logits_and_weights_use_unbiased_sigmoid():
    rng = np.random.default_rng(11)
    E, H, K, s = 32, 48, 4, 2.5
    W = rng.normal(0, 0.3, (E, H)).astype(np.float32)
    x = rng.standard_normal(H)
    logits = W.astype(np.float64) @ x
    cfg = oracle.make_cfg(H, E, K, 8, routed_scale=s)
    idx, w, _, _ = oracle.route(cfg, W, np.zeros(E, np.float32), x)
    assert idx.tolist() == np.argsort(-logits, kind="stable")[:K].tolist()
    sig = expit(logits)
    np.testing.assert_allclose(w, s * sig[idx] / (sig[idx].sum() + 1e-20), rtol=1e-12)
    assert w.sum() == pytest.approx(s, rel=1e-12)
    # a bias that keeps the same selection leaves the weights unchanged
    b = np.zeros(E, np.float32)
    b[idx] = 0.75
    idx2, w2, _, _ = oracle.route(cfg, W, b, x)
    assert sorted(idx2.tolist()) == sorted(idx.tolist())
    np.testing.assert_allclose(np.sort(w2), np.sort(w), rtol=1e-14)
    # a bias can change the selection; weights are still the plain sigmoid
    b = np.zeros(E, np.float32)
    lo = np.argsort(logits)[:K]
    b[lo] = 5.0
    idx3, w3, _, _ = oracle.route(cfg, W, b, x)
    assert sorted(idx3.tolist()) == sorted(lo.tolist())
    np.testing.assert_allclose(w3, s * sig[idx3] / (sig[idx3].sum() + 1e-20), rtol=1e-12)
    # without renormalisation the weight is s * sigmoid
    cfg0 = oracle.make_cfg(H, E, K, 8, routed_scale=s, norm_topk=0)
    idx0, w0, _, _ = oracle.route(cfg0, W, np.zeros(E, np.float32), x)
    np.testing.assert_allclose(w0, s * sig[idx0], rtol=1e-12)


def test_invalid_group_config_rejected():
    W, b, x = np.zeros((8, 4), np.float32), np.zeros(8, np.float32), np.ones(4)
    for kw in (dict(n_group=3),                          # E not a multiple of n_group
               dict(n_group=4, topk_group=0),
               dict(n_group=4, topk_group=5),
               dict(n_group=4, topk_group=1, K=3),      # K > topk_group * E / n_group
               dict(n_group=2, topk_group=1, score_func=oracle.SCORE_SOFTMAX),
               dict(score_func=2)):
        args = dict(K=2)
        args.update(kw)
        K = args.pop("K")
        cfg = oracle.make_cfg(4, 8, K, 8, **args)
        with pytest.raises(ValueError):
            oracle.route(cfg, W, b, x)


# --- routing variants (Edge0 section 七; reader.mx section 03, the OLMoE engine) -------

def _route_grouped(bias, K, n_group, topk_group):
    E, H = len(bias), 4
    cfg = oracle.make_cfg(H, E, K, 8, routed_scale=1.0, n_group=n_group, topk_group=topk_group)
    return oracle.route(cfg, np.zeros((E, H), np.float32), np.asarray(bias, np.float32), np.ones(H))


def test_group_limited_hand_cases():
    g = _golden("route_group_limited.txt")
    w = np.array([float(v) for v in g["w"]])
    for case in ("a", "b"):
        bias = [float(v) for v in g[case + "_bias"]]
        idx, wt, margin, sc = _route_grouped(bias, 3, 4, 2)
        assert idx.tolist() == [int(v) for v in g[case + "_idx"]], case
        np.testing.assert_allclose(wt, w, rtol=1e-12)
        assert margin == pytest.approx(float(g[case + "_margin"][0]), abs=1e-6), case
        # experts of the dropped groups carry -inf
        kept = {e // 2 for e in idx.tolist()}
        assert all((sc[2][e] == -np.inf) == (e // 2 not in kept) for e in range(8)) or case == "b"
    idx, _, _, _ = _route_grouped([float(v) for v in g["a_bias"]], 3, 1, 1)
    assert idx.tolist() == [int(v) for v in g["a_idx_ungrouped"]]


def test_group_ties_keep_lower_groups():
    idx, _, margin, _ = _route_grouped([0.1] * 8, 3, 4, 2)
    assert idx.tolist() == [0, 1, 2] and margin == 0.0


def test_grouping_that_keeps_everything_is_plain_topk():
    rng = np.random.default_rng(21)
    for _ in range(30):
        bias = rng.uniform(-0.3, 0.3, 16)
        ref, wref, _, _ = _route_grouped(bias, 5, 1, 1)
        for n_group, topk_group in ((4, 4), (16, 16), (16, 5), (16, 7)):
            # all groups kept; or groups of one expert with at least K kept: the top-K survive
            idx, w, _, _ = _route_grouped(bias, 5, n_group, topk_group)
            assert idx.tolist() == ref.tolist() and np.array_equal(w, wref)


def _softmax_case(seed, E=24, H=40, K=5):
    rng = np.random.default_rng(seed)
    W = rng.normal(0, 0.4, (E, H)).astype(np.float32)
    x = rng.standard_normal(H)
    b = rng.uniform(-0.5, 0.5, E).astype(np.float32)
    return W, b, x, W.astype(np.float64) @ x


@pytest.mark.parametrize("norm_topk", [1, 0])
def test_softmax_topk_matches_scipy_softmax(norm_topk):
    from scipy.special import softmax
    for seed in range(10):
        W, b, x, logits = _softmax_case(seed)
        E, H, K, s = W.shape[0], W.shape[1], 5, 1.75
        cfg = oracle.make_cfg(H, E, K, 8, routed_scale=s, norm_topk=norm_topk,
                              score_func=oracle.SCORE_SOFTMAX)
        idx, w, margin, sc = oracle.route(cfg, W, b, x)
        g = softmax(logits)
        assert margin > 1e-9
        assert idx.tolist() == np.argsort(-g, kind="stable")[:K].tolist()
        np.testing.assert_allclose(sc[1], g, rtol=1e-12)
        want = s * g[idx] / g[idx].sum() if norm_topk else s * g[idx]
        np.testing.assert_allclose(w, want, rtol=1e-12)
        # the bias plays no part in the softmax family
        idx0, w0, _, _ = oracle.route(cfg, W, np.zeros_like(b), x)
        assert idx0.tolist() == idx.tolist() and np.array_equal(w0, w)


def test_softmax_all_selected_weights_sum_to_scale():
    W, b, x, logits = _softmax_case(3, E=6, K=6)
    for norm in (1, 0):
        cfg = oracle.make_cfg(W.shape[1], 6, 6, 8, routed_scale=2.0, norm_topk=norm,
                              score_func=oracle.SCORE_SOFTMAX)
        _, w, margin, _ = oracle.route(cfg, W, b, x)
        assert w.sum() == pytest.approx(2.0, rel=1e-13) and margin == math.inf


def test_softmax_is_shift_invariant():
    # a constant added to every logit (here: a column of W against x_h = 1) changes nothing
    W, b, x, _ = _softmax_case(5, E=12, H=16, K=3)
    x = x.copy()
    x[0] = 1.0
    W = W.copy()
    W[:, 0] = 0.0               # so that the shifted column is exact in float32
    W2 = W.copy()
    W2[:, 0] = 0.375
    cfg = oracle.make_cfg(16, 12, 3, 8, routed_scale=1.0, score_func=oracle.SCORE_SOFTMAX)
    i1, w1, _, _ = oracle.route(cfg, W, b, x)
    i2, w2, _, _ = oracle.route(cfg, W2, b, x)
    assert i1.tolist() == i2.tolist()
    np.testing.assert_allclose(w1, w2, rtol=1e-12)


# --- whole layer ---------------------------------------------------------------

def _small_layer(H=64, E=6, K=2, I=32, I_sh=48, s=2.5, seed=5, shared=True):
    rng = np.random.default_rng(seed)
    W = rng.normal(0, 0.1, (E, H)).astype(np.float32)
    b = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    slabs = [rng.integers(0, 256, synth.slab_bytes(H, I), dtype=np.uint8) for _ in range(E)]
    scales = [rng.uniform(0.005, 0.02, 2 * I + H).astype(np.float32) for _ in range(E)]
    sh = rng.integers(0, 256, synth.slab_bytes(H, I_sh), dtype=np.uint8) if shared else None
    shs = rng.uniform(0.005, 0.02, 2 * I_sh + H).astype(np.float32) if shared else None
    cfg = oracle.make_cfg(H, E, K, I, int(shared), I_sh if shared else 0, routed_scale=s)
    return cfg, W, b, slabs, scales, sh, shs


def test_single_expert_layer_is_scaled_dense_swiglu():
    H, I, s = 64, 32, 2.5
    cfg, W, b, slabs, scales, _, _ = _small_layer(H=H, E=1, K=1, I=I, s=s, shared=False)
    L = oracle.LayerRef(cfg, W, b, slabs, scales)
    x = np.random.default_rng(1).standard_normal(H)
    y, idx, w, _ = L.token(x)
    assert idx.tolist() == [0] and w[0] == pytest.approx(s, rel=1e-15)
    np.testing.assert_allclose(y, s * _dense_swiglu(H, I, slabs[0], scales[0], x), rtol=1e-10)


def test_shared_only_is_dense_swiglu():
    H, I_sh = 64, 48
    cfg, W, b, slabs, scales, sh, shs = _small_layer(H=H, I_sh=I_sh, s=0.0)
    L = oracle.LayerRef(cfg, W, b, slabs, scales, sh, shs)
    x = np.random.default_rng(2).standard_normal(H)
    y, _, w, _ = L.token(x)
    assert np.all(w == 0)
    np.testing.assert_allclose(y, _dense_swiglu(H, I_sh, sh, shs, x), rtol=1e-10)


def test_layer_is_weighted_sum_plus_shared():
    H, I, I_sh, K, s = 64, 32, 48, 2, 2.5
    cfg, W, b, slabs, scales, sh, shs = _small_layer(H=H, I=I, I_sh=I_sh, K=K, s=s)
    L = oracle.LayerRef(cfg, W, b, slabs, scales, sh, shs)
    x = np.random.default_rng(4).standard_normal(H)
    y, idx, w, _ = L.token(x)
    ref = sum(w[k] * _dense_swiglu(H, I, slabs[idx[k]], scales[idx[k]], x) for k in range(K))
    ref = ref + _dense_swiglu(H, I_sh, sh, shs, x)
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-12)


def test_doubling_down_scales_doubles_output_exactly():
    H, I, I_sh = 64, 32, 48
    cfg, W, b, slabs, scales, sh, shs = _small_layer(H=H, I=I, I_sh=I_sh)
    x = np.random.default_rng(6).standard_normal(H)
    y1, *_ = oracle.LayerRef(cfg, W, b, slabs, scales, sh, shs).token(x)
    sc2 = [s.copy() for s in scales]
    for s in sc2:
        s[2 * I:] *= 2
    shs2 = shs.copy()
    shs2[2 * I_sh:] *= 2
    y2, *_ = oracle.LayerRef(cfg, W, b, slabs, sc2, sh, shs2).token(x)
    assert np.array_equal(y2, 2 * y1)


def test_forced_selection_rescored():
    cfg, W, b, slabs, scales, sh, shs = _small_layer()
    L = oracle.LayerRef(cfg, W, b, slabs, scales, sh, shs)
    x = np.random.default_rng(8).standard_normal(cfg.H)
    y, idx, w, _ = L.token(x)
    yf, idxf, wf, _ = L.token(x, forced_idx=idx)
    assert np.array_equal(y, yf) and np.array_equal(w, wf)
    other = np.array([idx[1], idx[0]], np.int32)     # same set, other order
    yo, _, wo, _ = L.token(x, forced_idx=other)
    np.testing.assert_allclose(yo, y, rtol=1e-12)


def test_missing_selected_expert_is_an_error():
    cfg, W, b, slabs, scales, sh, shs = _small_layer()
    L = oracle.LayerRef(cfg, W, b, [None] * cfg.E, [None] * cfg.E, sh, shs)
    with pytest.raises(ValueError):
        L.token(np.ones(cfg.H))


def test_rmsnorm_closed_form():
    out = oracle.rmsnorm(np.array([3.0, 4.0]), 0.0)
    np.testing.assert_allclose(out, np.array([3.0, 4.0]) / math.sqrt(12.5), rtol=1e-15)
    x = np.random.default_rng(9).standard_normal(100) * 3
    eps = 1e-5
    out = oracle.rmsnorm(x, eps)
    ms = np.mean(x * x)
    assert np.mean(out * out) == pytest.approx(ms / (ms + eps), rel=1e-12)


def test_prenorm_residual_layer():
    cfg, W, b, slabs, scales, sh, shs = _small_layer()
    x = np.random.default_rng(10).standard_normal(cfg.H) * 4
    y_plain, *_ = oracle.LayerRef(cfg, W, b, slabs, scales, sh, shs).token(oracle.rmsnorm(x, 1e-5))
    cfg_r = oracle.make_cfg(cfg.H, cfg.E, cfg.K, cfg.I, 1, cfg.I_shared, routed_scale=2.5,
                            prenorm_residual=1, rms_eps=1e-5)
    y_res, *_ = oracle.LayerRef(cfg_r, W, b, slabs, scales, sh, shs).token(x)
    np.testing.assert_allclose(y_res, x + y_plain, rtol=1e-13, atol=1e-13)
    # with nothing routed and no shared expert the residual stream is unchanged
    cfg_0 = oracle.make_cfg(cfg.H, cfg.E, cfg.K, cfg.I, 0, 0, routed_scale=0.0,
                            prenorm_residual=1)
    y0, *_ = oracle.LayerRef(cfg_0, W, b, slabs, scales).token(x)
    assert np.array_equal(y0, x)


def test_forward_loops_tokens():
    cfg, W, b, slabs, scales, sh, shs = _small_layer()
    L = oracle.LayerRef(cfg, W, b, slabs, scales, sh, shs)
    X = np.random.default_rng(12).standard_normal((5, cfg.H)).astype(np.float32)
    Y, I_, Wt, M = L.forward(X)
    for t in range(5):
        y, idx, w, m = L.token(X[t].astype(np.float64))
        assert np.array_equal(Y[t], y) and np.array_equal(I_[t], idx) and M[t] == m
