"""Pins of the CPU oracle against what the definition and the mathematics fix.

Each test ties the oracle to something other than itself: an exhaustive library
conversion, a hand-worked fixture (tests/golden/), a closed form, a textbook routine
(numpy matmul / scipy softmax) the layer reduces to in a special case, brute force on
tiny inputs, or an invariant of the definition.
"""
import math
import os

import numpy as np
import pytest
from scipy.special import softmax

import oracle
import syngen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def silu(t: float) -> float:
    return t / (1.0 + math.exp(-t))


def f16(v: float) -> int:
    return int(np.float16(v).view(np.uint16))


def bf16(v: float) -> int:
    return syngen.f32_to_bf16(v)


# ---- conversions --------------------------------------------------------------

def test_half_to_double_exhaustive_vs_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    ours = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(ours[~nan], ref[~nan])
    # signed zero preserved
    assert math.copysign(1.0, oracle.half_to_double(0x8000)) == -1.0


def test_bf16_to_float_exhaustive():
    bits = np.arange(65536, dtype=np.uint32)
    ref = (bits << 16).view(np.float32)
    ours = np.array([oracle.bf16_to_float(int(b)) for b in bits], np.float32)
    nan = np.isnan(ref)
    np.testing.assert_array_equal(ours.view(np.uint32)[~nan], ref.view(np.uint32)[~nan])


# ---- router order -------------------------------------------------------------

def _read_kv(path):
    d = {}
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if line:
            k, *v = line.split()
            d.setdefault(k, []).append(v)
    return d


def test_canonical_order_golden():
    d = _read_kv(os.path.join(GOLDEN, "canonical_order.txt"))
    H = int(d["H"][0][0])
    x = np.ones(H, np.float32)
    x[0] = float(d["x0"][0][0])
    w = np.ones(H, np.float32)
    got = oracle.canonical_logit(w, x)
    assert float(got) == float(d["expect"][0][0])
    assert float(got) != float(np.float32(2 ** 24))  # not the sequential order


def test_canonical_logit_within_fp32_bound_of_exact_dot():
    rng = np.random.default_rng(5)
    for H in (128, 512, 2048):
        w = (rng.standard_normal(H) * 0.02).astype(np.float32)
        x = rng.standard_normal(H).astype(np.float32)
        got = float(oracle.canonical_logit(w, x))
        exact = float(np.dot(w.astype(np.float64), x.astype(np.float64)))
        # H/32 fmas per lane then 5 additions: error <= gamma_{H/32+5} * sum |w x|
        n = H // 32 + 5
        bound = n * 2.0 ** -24 / (1 - n * 2.0 ** -24) * float(np.abs(w.astype(np.float64) * x).sum())
        assert abs(got - exact) <= bound


def test_canonical_logit_is_lane_structured():
    # a single nonzero product lands exactly, wherever it sits
    H = 256
    for h in (0, 1, 4, 127, 128, 255):
        w = np.zeros(H, np.float32)
        x = np.zeros(H, np.float32)
        w[h], x[h] = 3.0, -0.5
        assert float(oracle.canonical_logit(w, x)) == -1.5


# ---- hand-worked layer ----------------------------------------------------------

def _worked_layer():
    d = _read_kv(os.path.join(GOLDEN, "worked_layer.txt"))
    H, E, k, I, R = (int(v) for v in d["dims"][0])
    x = np.zeros(H, np.float32)
    for h, v in d["x"]:
        x[int(h)] = float(v)
    xb = np.array([[bf16(float(v)) for v in x]], np.uint16)
    router = np.zeros((E, H), np.float32)
    for e, h, v in d["router"]:
        router[int(e), int(h)] = float(v)
    ew = syngen.ExpertW(
        qg=np.zeros((E, I, H), np.int8), sg=np.full((E, I, H // 32), f16(1.0), np.uint16),
        qu=np.zeros((E, I, H), np.int8), su=np.full((E, I, H // 32), f16(1.0), np.uint16),
        qd=np.zeros((E, H, I), np.int8), sd=np.full((E, H, I // 32), f16(1.0), np.uint16))
    for e, mat, row, col, code, scale in d["q"]:
        e, row, col, code = int(e), int(row), int(col), int(code)
        if mat == "gate":
            ew.qg[e, row, col] = code
            ew.sg[e, row, col // 32] = f16(float(scale))
        elif mat == "up":
            ew.qu[e, row, col] = code
            ew.su[e, row, col // 32] = f16(float(scale))
        else:
            ew.qd[e, row, col] = code
            ew.sd[e, row, col // 32] = f16(float(scale))
    return d, (H, E, k, I, R), router, xb, ew


def test_worked_layer_golden():
    d, (H, E, k, I, R), router, xb, ew = _worked_layer()
    rt = oracle.route(router, xb, k)
    assert rt.ids[0].tolist() == [int(v) for v in d["expect_ids"][0]]
    np.testing.assert_array_equal(rt.w[0], [float(v) for v in d["expect_w"][0]])
    assert rt.union.tolist() == sorted(int(v) for v in d["expect_ids"][0])
    out = oracle.layer(router, xb, k, np.arange(E), ew)
    expect = np.zeros(H)
    for o, c, a, b in d["expect_out"]:
        expect[int(o)] = float(c) + float(a) * silu(8.0) + float(b) * silu(-128.0)
    np.testing.assert_allclose(out[0], expect, rtol=1e-14, atol=1e-300)
    # the dense brute force agrees
    np.testing.assert_allclose(oracle.layer_dense(router, xb, k, ew)[0], expect, rtol=1e-14, atol=1e-300)


def test_worked_layer_catches_swapped_gate_up():
    # silu(v) * g instead of silu(g) * v would give 0.5*(-silu(6)*64) at o5
    d, dims, router, xb, ew = _worked_layer()
    out = oracle.layer(router, xb, 2, np.arange(4), ew)
    assert abs(out[0, 5] - (-192.0 - 0.5 * silu(8.0))) < 1e-12
    assert abs(out[0, 5] - (-0.5 * 64 * silu(6.0))) > 1.0


# ---- special cases reducing to textbook routines --------------------------------

def _rand_experts(rng, E, H, I, zero=False):
    def q(shape):
        return np.zeros(shape, np.int8) if zero else rng.integers(-8, 8, shape, dtype=np.int8)

    def s(shape):
        return (np.abs(rng.standard_normal(shape)) * 0.02).astype(np.float16).view(np.uint16)
    return syngen.ExpertW(q((E, I, H)), s((E, I, H // 32)), q((E, I, H)), s((E, I, H // 32)),
                          q((E, H, I)), s((E, H, I // 32)))


def _dense(qa, sa):
    """Dequantize [rows][K] codes with [rows][K/32] fp16 scales (numpy, float64)."""
    sc = sa.view(np.float16).astype(np.float64)
    return qa.astype(np.float64) * np.repeat(sc, 32, axis=1)


def test_single_expert_is_plain_swiglu_mlp():
    rng = np.random.default_rng(11)
    H, I = 256, 96
    ew = _rand_experts(rng, 1, H, I)
    router = (rng.standard_normal((1, H)) * 0.02).astype(np.float32)
    xb = np.array([[bf16(float(v)) for v in rng.standard_normal(H)] for _ in range(3)], np.uint16)
    out = oracle.layer(router, xb, 1, [0], ew)
    x = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    Wg, Wu, Wd = _dense(ew.qg[0], ew.sg[0]), _dense(ew.qu[0], ew.su[0]), _dense(ew.qd[0], ew.sd[0])
    g, v = x @ Wg.T, x @ Wu.T
    ref = (g / (1 + np.exp(-g)) * v) @ Wd.T
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_one_hot_row_and_single_codes_closed_form():
    """A one-hot row meeting one nonzero gate code, one up code and one down code: the
    layer reduces to one product chain, out[o] = sd * qd * silu(sg * qg * a) * (su * qu * a),
    and every other output is exactly zero (silu(0) * 0)."""
    rng = np.random.default_rng(5)
    H, I = 256, 64
    j0, i0, o0, a = 77, 41, 200, 1.5
    ew = _rand_experts(rng, 1, H, I, zero=True)
    ew.qg[0, i0, j0], ew.sg[0, i0, j0 // 32] = 3, f16(0.25)
    ew.qu[0, i0, j0], ew.su[0, i0, j0 // 32] = -2, f16(0.5)
    ew.qd[0, o0, i0], ew.sd[0, o0, i0 // 32] = 5, f16(0.125)
    row = np.zeros(H, np.uint16)
    row[j0] = bf16(a)
    out = oracle.layer(np.zeros((1, H), np.float32), row[None, :], 1, [0], ew)
    g, v = 0.25 * 3 * a, 0.5 * -2 * a
    want = 0.125 * 5 * silu(g) * v
    assert abs(out[0, o0] - want) <= 1e-12 * abs(want)
    rest = np.delete(out[0], o0)
    assert (rest == 0).all()


def test_expert_ffn_matches_single_expert_layer():
    rng = np.random.default_rng(21)
    H, I = 128, 64
    ew = _rand_experts(rng, 1, H, I)
    router = np.zeros((1, H), np.float32)
    xb = np.array([[bf16(float(v)) for v in rng.standard_normal(H)]], np.uint16)
    y = oracle.expert_ffn(xb[0], ew, 0)
    np.testing.assert_array_equal(y, oracle.layer(router, xb, 1, [0], ew)[0])


def test_k_equals_e_is_full_softmax():
    rng = np.random.default_rng(12)
    E, H = 8, 512
    router = (rng.standard_normal((E, H)) * 0.02).astype(np.float32)
    xb = np.array([[bf16(float(v)) for v in rng.standard_normal(H)] for _ in range(4)], np.uint16)
    rt = oracle.route(router, xb, E)
    for r in range(4):
        p = softmax(rt.logits[r].astype(np.float64))
        np.testing.assert_allclose(rt.w[r], p[rt.ids[r]], rtol=1e-14)
        assert sorted(rt.ids[r].tolist()) == list(range(E))
    assert rt.union.tolist() == list(range(E))


def test_topk_two_closed_form_weights():
    # two picks with logits l1 >= l2: w1 = 1 / (1 + exp(l2 - l1))
    H, E = 128, 4
    router = np.zeros((E, H), np.float32)
    router[0, 0], router[1, 0], router[2, 0], router[3, 0] = 0.25, 1.5, -1.0, 0.75
    x = np.zeros(H, np.float32)
    x[0] = 2.0
    xb = np.array([[bf16(float(v)) for v in x]], np.uint16)
    rt = oracle.route(router, xb, 2)
    assert rt.ids[0].tolist() == [1, 3]
    l1, l2 = 3.0, 1.5
    assert abs(rt.w[0, 0] - 1 / (1 + math.exp(l2 - l1))) < 1e-16
    assert abs(rt.w[0, 1] - 1 / (1 + math.exp(l1 - l2))) < 1e-16


# ---- routing brute force, ties, sums ---------------------------------------------

def test_topk_matches_brute_force_sort():
    rng = np.random.default_rng(13)
    for E, k, H, R in [(8, 2, 512, 4), (16, 5, 256, 3), (64, 8, 128, 2), (33, 7, 128, 1)]:
        router = (rng.standard_normal((E, H)) * 0.02).astype(np.float32)
        xb = np.array([[bf16(float(v)) for v in rng.standard_normal(H)] for _ in range(R)], np.uint16)
        rt = oracle.route(router, xb, k)
        for r in range(R):
            order = sorted(range(E), key=lambda e: (-float(rt.logits[r, e]), e))
            assert rt.ids[r].tolist() == order[:k]
        assert rt.union.tolist() == sorted(set(rt.ids.flatten().tolist()))


def test_forced_ties_pick_lower_id():
    rng = np.random.default_rng(14)
    E, H = 8, 256
    router = (rng.standard_normal((E, H)) * 0.02).astype(np.float32)
    x = rng.standard_normal(H)
    xb = np.array([[bf16(float(v)) for v in x]], np.uint16)
    xf = (xb.astype(np.uint32) << 16).view(np.float32)[0]
    # make experts 5 and 2 identical and dominant; 6 identical to 1 (a tie lower down)
    big = (np.sign(xf) * 0.05).astype(np.float32)
    router[5] = big
    router[2] = big
    router[6] = router[1]
    rt = oracle.route(router, xb, 4)
    assert rt.ids[0, 0] == 2 and rt.ids[0, 1] == 5
    assert rt.logits[0, 2] == rt.logits[0, 5]
    assert rt.w[0, 0] == rt.w[0, 1]
    if 1 in rt.ids[0] and 6 in rt.ids[0]:
        assert list(rt.ids[0]).index(1) < list(rt.ids[0]).index(6)
    # all-zero router: every logit is 0, the picks are 0..k-1
    rt0 = oracle.route(np.zeros((E, H), np.float32), xb, 3)
    assert rt0.ids[0].tolist() == [0, 1, 2]
    np.testing.assert_allclose(rt0.w[0], [1 / 3] * 3, rtol=1e-15)


def test_weights_sum_to_one():
    cfg = syngen.CONFIGS["tiny"].with_(rows=4, row_sigma=0.5)
    for layer in range(3):
        rt = oracle.route(syngen.router(cfg, layer), syngen.rows(cfg, layer), cfg.top_k)
        np.testing.assert_allclose(rt.w.sum(axis=1), 1.0, atol=1e-15)
        assert (np.diff(rt.w, axis=1) <= 0).all()  # rank order = descending weight


# ---- invariants on generated layers ------------------------------------------------

@pytest.fixture(scope="module")
def tiny4():
    cfg = syngen.CONFIGS["tiny"].with_(rows=4, row_sigma=0.5)
    router = syngen.router(cfg, 0)
    xb = syngen.rows(cfg, 0)
    ew = syngen.experts_stacked(cfg, 0, range(cfg.experts), threads=1)
    return cfg, router, xb, ew


def test_dense_brute_force_equals_union_evaluation(tiny4):
    cfg, router, xb, ew = tiny4
    out = oracle.layer(router, xb, cfg.top_k, np.arange(cfg.experts), ew)
    dense = oracle.layer_dense(router, xb, cfg.top_k, ew)
    np.testing.assert_allclose(out, dense, rtol=1e-12, atol=1e-12 * np.abs(dense).max())


def test_row_independence_bitwise(tiny4):
    cfg, router, xb, ew = tiny4
    out = oracle.layer(router, xb, cfg.top_k, np.arange(cfg.experts), ew)
    for r in range(xb.shape[0]):
        alone = oracle.layer(router, xb[r:r + 1].copy(), cfg.top_k, np.arange(cfg.experts), ew)
        np.testing.assert_array_equal(alone[0], out[r])


def test_row_permutation_equivariance(tiny4):
    cfg, router, xb, ew = tiny4
    out = oracle.layer(router, xb, cfg.top_k, np.arange(cfg.experts), ew)
    perm = np.array([2, 0, 3, 1])
    outp = oracle.layer(router, xb[perm].copy(), cfg.top_k, np.arange(cfg.experts), ew)
    np.testing.assert_array_equal(outp, out[perm])


def test_union_and_unique_bytes(tiny4):
    cfg, router, xb, ew = tiny4
    rt = oracle.route(router, xb, cfg.top_k)
    picked = set()
    for r in range(xb.shape[0]):
        picked |= set(int(e) for e in rt.ids[r])
    assert rt.union.tolist() == sorted(picked)
    # per-expert packed bytes printed for the workloads (three H x I matrices at 18 B per
    # 32 weights): 221,184 B for the tiny layer, 2,654,208 B for the 35B-A3B-shaped one,
    # 1,769,472 B for the 512-expert one
    assert oracle.unique_expert_bytes(512, 256, 1) == 221_184
    assert oracle.unique_expert_bytes(2048, 768, 1) == 2_654_208
    assert oracle.unique_expert_bytes(2048, 512, 1) == 1_769_472
    assert oracle.unique_expert_bytes(2048, 768, 8) == 21_233_664  # 8 unique experts, one row
    assert oracle.unique_expert_bytes(cfg.hidden, cfg.inter, len(picked)) == len(picked) * 221_184


def test_all_zero_codes_give_zero(tiny4):
    cfg, router, xb, _ = tiny4
    ew0 = _rand_experts(np.random.default_rng(0), cfg.experts, cfg.hidden, cfg.inter, zero=True)
    out = oracle.layer(router, xb, cfg.top_k, np.arange(cfg.experts), ew0)
    assert (out == 0).all()


def test_down_scale_linearity(tiny4):
    cfg, router, xb, ew = tiny4
    out = oracle.layer(router, xb, cfg.top_k, np.arange(cfg.experts), ew)
    sd2 = (ew.sd.view(np.float16).astype(np.float32) * 2).astype(np.float16).view(np.uint16)
    ew2 = syngen.ExpertW(ew.qg, ew.sg, ew.qu, ew.su, ew.qd, np.ascontiguousarray(sd2))
    out2 = oracle.layer(router, xb, cfg.top_k, np.arange(cfg.experts), ew2)
    np.testing.assert_array_equal(out2, 2 * out)


def test_missing_expert_is_reported(tiny4):
    cfg, router, xb, ew = tiny4
    rt = oracle.route(router, xb, cfg.top_k)
    keep = [e for e in range(cfg.experts) if e != rt.union[0]]
    sub = syngen.ExpertW(*(np.ascontiguousarray(getattr(ew, f)[keep]) for f in ("qg", "sg", "qu", "su", "qd", "sd")))
    with pytest.raises(KeyError):
        oracle.layer(router, xb, cfg.top_k, keep, sub)


def test_bad_dims_rejected():
    with pytest.raises(ValueError):
        oracle.route(np.zeros((4, 100), np.float32), np.zeros((1, 100), np.uint16), 2)  # H % 128
    with pytest.raises(ValueError):
        oracle.route(np.zeros((4, 128), np.float32), np.zeros((1, 128), np.uint16), 5)  # k > E


def test_generated_full_size_layer_routes_sanely():
    cfg = syngen.CONFIGS["a3b_r4"]
    rt = oracle.route(syngen.router(cfg, 0), syngen.rows(cfg, 0), cfg.top_k)
    assert rt.ids.shape == (4, 8)
    assert cfg.top_k <= rt.union.size <= 32
    assert (rt.gap64 >= 0).all()


def test_fp64_shadow_gap_on_known_logits():
    """The shadow gap is the exact (fp64) difference between the k-th and (k+1)-th
    largest logit.  A one-hot row x = e_3 makes every logit exactly Wr[e][3]; with the
    column set to distinct powers of two (and ties) the gaps are known in closed form."""
    E, H = 8, 128
    router = np.zeros((E, H), np.float32)
    router[:, 3] = [0.5, -1.0, 0.25, 2.0, 0.125, 0.25, -0.5, 1.0]   # descending: 2, 1, .5, .25, .25, .125, ...
    xb = np.zeros((1, H), np.uint16)
    xb[0, 3] = bf16(1.0)
    gaps = {1: 2.0 - 1.0, 2: 1.0 - 0.5, 3: 0.5 - 0.25, 4: 0.25 - 0.25, 5: 0.25 - 0.125, 7: -0.5 - (-1.0)}
    for k, want in gaps.items():
        rt = oracle.route(router, xb, k)
        assert rt.gap64[0] == want, (k, rt.gap64[0], want)
    assert np.isinf(oracle.route(router, xb, E).gap64[0])  # k = E: nothing left out
    # a gap below fp32 resolution stays visible in fp64: logits 1 + 2^-30 and 1
    r2 = np.zeros((2, H), np.float32)
    r2[0, 0], r2[0, 1] = 1.0, 2.0 ** -30
    r2[1, 0] = 1.0
    x2 = np.zeros((1, H), np.uint16)
    x2[0, 0] = x2[0, 1] = bf16(1.0)
    rt2 = oracle.route(r2, x2, 1)
    assert rt2.gap64[0] == 2.0 ** -30


# ---- routing tail skip (Avalon README, "Numbers": experts that every token of a
# verification routes only at rank 7 or lower are skipped) ---------------------------

def _ranked_router(row_logits):
    """Router whose logits for one-hot row r (x = e_r) are exactly row_logits[r]:
    Wr[e][r] = row_logits[r][e], zero elsewhere, H = 128."""
    R, E = len(row_logits), len(row_logits[0])
    H = 128
    router = np.zeros((E, H), np.float32)
    for r in range(R):
        for e in range(E):
            router[e, r] = row_logits[r][e]
    xb = np.zeros((R, H), np.uint16)
    for r in range(R):
        xb[r, r] = bf16(1.0)
    return router, xb


# Hand-built ranks (k = 4).  Row 0 ranks experts 0, 1, 2, 3 (1-based ranks 1..4); row 1
# ranks 0, 1, 4, 5.  So expert 2 and 4 are only ever rank 3, experts 3 and 5 only rank 4.
TAIL_LOGITS_A = [[8.0, 7.0, 6.0, 5.0, 1.0, 0.5, 0.0, -1.0],
                 [8.0, 7.0, 0.0, -1.0, 6.0, 5.0, -2.0, -3.0]]
# Row 1 now ranks 0, 3, 1, 4: expert 3 is rank 4 in row 0 but rank 2 in row 1.
TAIL_LOGITS_B = [[8.0, 7.0, 6.0, 5.0, 1.0, 0.5, 0.0, -1.0],
                 [8.0, 7.0, 0.0, 7.5, 6.0, -1.0, -2.0, -3.0]]


@pytest.mark.parametrize("tail, union", [(0, [0, 1, 2, 3, 4, 5]), (5, [0, 1, 2, 3, 4, 5]),
                                         (4, [0, 1, 2, 4]), (3, [0, 1]), (2, [0]), (1, [])])
def test_tail_skip_union_hand_built(tail, union):
    router, xb = _ranked_router(TAIL_LOGITS_A)
    rt = oracle.route(router, xb, 4, tail)
    np.testing.assert_array_equal(rt.ids, [[0, 1, 2, 3], [0, 1, 4, 5]])
    assert rt.union.tolist() == union
    for r in range(2):
        for j in range(4):
            assert rt.keep[r, j] == (rt.ids[r, j] in union)


def test_tail_skip_keeps_an_expert_ranked_high_by_any_row():
    router, xb = _ranked_router(TAIL_LOGITS_B)
    rt = oracle.route(router, xb, 4, 3)
    np.testing.assert_array_equal(rt.ids, [[0, 1, 2, 3], [0, 3, 1, 4]])
    # expert 3: rank 4 in row 0, rank 2 in row 1 -> kept; 2 and 4 are only rank 3
    assert rt.union.tolist() == [0, 1, 3]
    np.testing.assert_array_equal(rt.keep, [[1, 1, 0, 1], [1, 1, 1, 0]])


def test_tail_skip_weights_are_not_renormalised():
    router, xb = _ranked_router(TAIL_LOGITS_A)
    full = oracle.route(router, xb, 4, 0)
    skip = oracle.route(router, xb, 4, 3)
    np.testing.assert_array_equal(full.w, skip.w)
    # row 0's kept weights are the first two softmax terms of logits 8, 7, 6, 5
    ex = np.exp(np.array([8.0, 7.0, 6.0, 5.0]) - 8.0)
    np.testing.assert_allclose(skip.w[0, :2], ex[:2] / ex.sum(), rtol=1e-15)


def test_tail_skip_layer_equals_dense_with_dropped_gates(tiny4):
    cfg, router, xb, ew = tiny4
    for tail in (1, 2, 3):
        rt = oracle.route(router, xb, cfg.top_k, tail)
        out = oracle.layer(router, xb, cfg.top_k, np.arange(cfg.experts), ew, tail)
        dense = oracle.layer_dense(router, xb, cfg.top_k, ew, tail)
        scale = max(np.abs(dense).max(), 1e-30)
        np.testing.assert_allclose(out, dense, rtol=1e-12, atol=1e-12 * scale)
        if tail == 1:
            assert rt.union.size == 0
            assert not out.any()
    # a threshold past k drops nothing: bitwise the plain layer
    plain = oracle.layer(router, xb, cfg.top_k, np.arange(cfg.experts), ew)
    past = oracle.layer(router, xb, cfg.top_k, np.arange(cfg.experts), ew, cfg.top_k + 1)
    np.testing.assert_array_equal(plain, past)


def test_tail_skip_union_grows_with_threshold():
    cfg = syngen.CONFIGS["a3b_r4"]
    router = syngen.router(cfg, 0)
    xb = syngen.rows(cfg, 0)
    sizes = [oracle.route(router, xb, cfg.top_k, t).union.size for t in range(1, cfg.top_k + 2)]
    assert sizes[0] == 0 and all(a <= b for a, b in zip(sizes, sizes[1:]))
    assert sizes[-1] == oracle.route(router, xb, cfg.top_k).union.size
