"""Pins for the CPU oracle: every oracle function is checked against something
other than itself -- values the pages print, closed forms, exact rational
brute force on tiny shapes, and library routines (torch's BF16 conversion,
numpy's float32 view).  CPU only."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from split_w4a16_quantized_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _torch_bf16_bits(x64):
    """Library rounding: float64 -> float32 (exact for the values used) -> BF16."""
    x32 = np.asarray(x64, np.float64).astype(np.float32)
    assert np.array_equal(x32.astype(np.float64), np.asarray(x64, np.float64))
    return torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bits_to_f64(b):
    return inputs.bf16_bits_to_f32(b).astype(np.float64)


def _bf16_bits(v):
    return int(_torch_bf16_bits(np.array([v]))[0])


# ---- number formats --------------------------------------------------------

def test_bf16_value_all_finite_patterns():
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref32 = (b.astype(np.uint32) << 16).view(np.float32)
    fin = np.isfinite(ref32)
    ref = np.where(fin, ref32, 0).astype(np.float64)
    got = oracle.bf16_value(b)
    assert np.array_equal(got[fin], ref[fin])


def test_bf16_round_matches_torch_rne():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(200000).astype(np.float32).astype(np.float64)
    x *= np.exp2(rng.integers(-60, 60, x.size)).astype(np.float64)
    assert np.array_equal(oracle.bf16_round(x), _torch_bf16_bits(x))


def test_bf16_round_ties_to_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: the even neighbour is 1.
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 (odd) and 1 + 2^-6 (even).
    x = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 0.0, -0.0, 3.0])
    got = oracle.bf16_round(x)
    assert list(got) == [0x3F80, 0x3F82, 0xBF80, 0x0000, 0x8000, 0x4040]


# ---- unpack ----------------------------------------------------------------

def test_unpack_fixed_words():
    Wq = np.array([[0x76543210, 0xFEDCBA98]], np.uint32)
    assert list(oracle.unpack(Wq, 16)[0]) == list(range(16))


def test_unpack_single_nibbles():
    for j in range(8):
        q = oracle.unpack(np.array([[1 << (4 * j)]], np.uint32), 8)[0]
        assert list(q) == [1 if i == j else 0 for i in range(8)]
        q = oracle.unpack(np.array([[0xF << (4 * j)]], np.uint32), 8)[0]
        assert list(q) == [15 if i == j else 0 for i in range(8)]


def test_unpack_inverts_generator_packing():
    p = inputs.make_w4a16(1, 512, 37, seed=3)
    assert np.array_equal(oracle.unpack(p["Wq"], 512), p["q"])


# ---- dequant ---------------------------------------------------------------

def test_dequant_matches_library_rounding():
    p = inputs.make_w4a16(1, 768, 50, seed=4)
    G = 768 // 128
    s = np.repeat(_bits_to_f64(p["scales"]), 128, axis=1)
    b = np.repeat(_bits_to_f64(p["biases"]), 128, axis=1)
    exact = s * p["q"].astype(np.float64) + b
    assert np.array_equal(oracle.dequant(p["Wq"], p["scales"], p["biases"], 768),
                          _torch_bf16_bits(exact))
    assert G == 6


def test_dequant_group_index():
    # scale_g = 2^-g, q = 1, bias 0: every element of group g dequantizes to 2^-g
    Kred, G = 512, 4
    Wq = np.full((1, Kred // 8), 0x11111111, np.uint32)
    scales = np.array([[_bf16_bits(2.0 ** -g) for g in range(G)]], np.uint16)
    biases = np.zeros((1, G), np.uint16)
    w = _bits_to_f64(oracle.dequant(Wq, scales, biases, Kred))[0]
    assert np.array_equal(w, np.repeat(2.0 ** -np.arange(G), 128))


# ---- the matmul ------------------------------------------------------------

def _exact_qmm(p):
    """Exact rational C = A @ W^T with W rounded to BF16 by torch."""
    Kred = p["Kred"]
    a = _bits_to_f64(p["A"])
    s = np.repeat(_bits_to_f64(p["scales"]), 128, axis=1)
    b = np.repeat(_bits_to_f64(p["biases"]), 128, axis=1)
    w = _bits_to_f64(_torch_bf16_bits(s * p["q"].astype(np.float64) + b))
    M, N = a.shape[0], w.shape[0]
    C = [[sum((Fraction(a[m, k]) * Fraction(w[n, k]) for k in range(Kred)), Fraction(0))
          for n in range(N)] for m in range(M)]
    mag = np.abs(a) @ np.abs(w).T
    return C, mag


@pytest.mark.parametrize("M,Kred,Nout,seed", [(1, 128, 1, 0), (2, 128, 5, 1), (3, 256, 4, 2),
                                              (3, 256, 5, 3)])
def test_qmm_exact_brute_force(M, Kred, Nout, seed):
    p = inputs.make_w4a16(M, Kred, Nout, seed=seed)
    C = oracle.qmm(p["A"], p["Wq"], p["scales"], p["biases"], threads=2)
    exact, mag = _exact_qmm(p)
    for m in range(M):
        for n in range(Nout):
            assert abs(Fraction(C[m, n]) - exact[m][n]) <= Fraction(mag[m, n]) * Fraction(1, 2 ** 45)


def test_qmm_closed_form_constant_rows():
    # q = c_n, scale = s_n, bias = b_n on row n: C[m, n] = BF16(s_n c_n + b_n) * sum_k A[m, k]
    M, Kred, Nout = 4, 384, 6
    c = np.array([0, 3, 7, 8, 12, 15])
    Wq = np.array([[int(ci) * 0x11111111] * (Kred // 8) for ci in c], np.uint32)
    sv = np.array([0.0078125, 0.01171875, 0.015625, 0.005859375, 0.009765625, 0.0185546875])
    bv = np.array([-0.0625, -0.09375, -0.125, -0.046875, -0.078125, -0.1484375])
    scales = np.repeat(_torch_bf16_bits(sv)[:, None], 3, axis=1)
    biases = np.repeat(_torch_bf16_bits(bv)[:, None], 3, axis=1)
    a_bits = inputs.f32_to_bf16_bits(np.random.default_rng(5).standard_normal((M, Kred)))
    C = oracle.qmm(a_bits, Wq, scales, biases, threads=1)
    wv = _bits_to_f64(_torch_bf16_bits(_bits_to_f64(scales[:, 0]) * c + _bits_to_f64(biases[:, 0])))
    rowsum = [math.fsum(r) for r in _bits_to_f64(a_bits)]
    for m in range(M):
        for n in range(Nout):
            assert C[m, n] == pytest.approx(wv[n] * rowsum[m], rel=1e-13, abs=1e-13)


def test_qmm_identity_weights():
    # one-hot q rows (q[n, n] = 1), scale 1, bias 0: C = A[:, :Nout] exactly
    Kred, Nout, M = 128, 100, 7
    q = np.zeros((Nout, Kred), np.uint8)
    q[np.arange(Nout), np.arange(Nout)] = 1
    Wq = inputs.pack_nibbles(q)
    scales = np.full((Nout, 1), 0x3F80, np.uint16)
    biases = np.zeros((Nout, 1), np.uint16)
    a = inputs.make_w4a16(M, Kred, 1, seed=6)["A"]
    C = oracle.qmm(a, Wq, scales, biases, threads=1)
    assert np.array_equal(C, _bits_to_f64(a)[:, :Nout])


def test_qmm_one_hot_activations_give_transposed_weights():
    # A = identity [Kred, Kred]: C[m, n] = w[n, m], which pins operand order
    p = inputs.make_w4a16(1, 256, 9, seed=7)
    eye = np.where(np.eye(256, dtype=bool), np.uint16(0x3F80), np.uint16(0))
    C = oracle.qmm(eye, p["Wq"], p["scales"], p["biases"], threads=2)
    w = _bits_to_f64(oracle.dequant(p["Wq"], p["scales"], p["biases"], 256))
    assert np.array_equal(C, w.T)


def test_qmm_sampled_matches_full():
    p = inputs.make_w4a16(9, 640, 33, seed=8)
    C = oracle.qmm(p["A"], p["Wq"], p["scales"], p["biases"], threads=2)
    rows, cols = np.array([0, 4, 8]), np.array([0, 1, 17, 32])
    S = oracle.qmm_sampled(p["A"], p["Wq"], p["scales"], p["biases"], rows, cols, threads=2)
    assert np.array_equal(S, C[np.ix_(rows, cols)])


# ---- partition emulation ---------------------------------------------------

def test_partitioned_split1_is_rounded_exact():
    p = inputs.make_w4a16(5, 1280, 40, seed=9)
    C64 = oracle.qmm(p["A"], p["Wq"], p["scales"], p["biases"], threads=2)
    for mode in (0, 1):
        C, _ = oracle.qmm_partitioned(p["A"], p["Wq"], p["scales"], p["biases"], 1, mode)
        # bf16_round is itself pinned against torch's rounding above
        assert np.array_equal(C, oracle.bf16_round(C64))


def test_partition_boundaries_follow_groups():
    # activations nonzero only in group g: only the partition holding g gets a nonzero plane
    Kred, G, s = 1280, 10, 5
    p = inputs.make_w4a16(2, Kred, 8, seed=10)
    for g in range(G):
        a = np.zeros((2, Kred), np.uint16)
        a[:, g * 128:(g + 1) * 128] = p["A"][:, g * 128:(g + 1) * 128]
        _, P = oracle.qmm_partitioned(a, p["Wq"], p["scales"], p["biases"], s, 1,
                                      with_partials=True)
        nonzero = [bool(np.any(P[i] != 0)) for i in range(s)]
        assert nonzero == [i == g // (G // s) for i in range(s)]


def plane_sum_case():
    """M = 1, Nout = 1, Kred = 384, split 3: partition p holds one group whose
    only nonzero product is A[0, 128p] * w[0, 128p] = v_p, with
    (v_0, v_1, v_2) = (1, 2^-8, 2^-30), all exact in BF16.  The chapter's
    reduce adds the planes in FP32 in ascending order: 1 + 2^-8 is exact, and
    adding 2^-30 (below half an FP32 ulp of 1) leaves it there; 1 + 2^-8 is the
    midpoint between the BF16 neighbours 1 and 1 + 2^-7, and round-to-even
    gives 1.  The exact sum lies above that midpoint and rounds to 1 + 2^-7."""
    A = np.zeros((1, 384), np.uint16)
    A[0, [0, 128, 256]] = 0x3F80
    q = np.zeros((1, 384), np.uint8)
    q[0, [0, 128, 256]] = 1
    scales = np.array([[0x3F80, 0x3B80, 0x3080]], np.uint16)  # 1, 2^-8, 2^-30
    return {"A": A, "Wq": inputs.pack_nibbles(q), "scales": scales,
            "biases": np.zeros((1, 3), np.uint16)}


def test_partitioned_planes_are_added_in_fp32():
    p = plane_sum_case()
    C, planes = oracle.qmm_partitioned(p["A"], p["Wq"], p["scales"], p["biases"], 3, 0,
                                       with_partials=True)
    assert planes[:, 0, 0].tolist() == [1.0, 2.0 ** -8, 2.0 ** -30]
    assert int(C[0, 0]) == 0x3F80  # FP32 ascending sum, one BF16 rounding: 1
    # the fp64 result of the same planes rounds the other way
    C64 = oracle.qmm(p["A"], p["Wq"], p["scales"], p["biases"])
    assert C64[0, 0] == 1 + 2.0 ** -8 + 2.0 ** -30
    assert int(oracle.bf16_round(C64)[0, 0]) == 0x3F81
    # FP32 planes (partial_mode 1) take the same sum
    C32, _ = oracle.qmm_partitioned(p["A"], p["Wq"], p["scales"], p["biases"], 3, 1)
    assert int(C32[0, 0]) == 0x3F80


def test_partitioned_error_bound():
    p = inputs.make_w4a16(8, 2560, 64, seed=11)
    C64 = oracle.qmm(p["A"], p["Wq"], p["scales"], p["biases"], threads=2)
    for s in (2, 4, 5, 10):
        C, P = oracle.qmm_partitioned(p["A"], p["Wq"], p["scales"], p["biases"], s, 0,
                                      with_partials=True)
        got = oracle.bf16_value(C)
        # BF16 keeps 8 significant bits: each rounding is off by at most 2^-8 relative
        bound = 2.0 ** -8 * (np.abs(P).sum(axis=0) + np.abs(C64)) + 2.0 ** -20 * np.abs(P).sum(axis=0)
        assert np.all(np.abs(got - C64) <= bound + 1e-30)
        assert np.allclose(P.sum(axis=0), C64, rtol=0, atol=2.0 ** -8 * np.abs(P).sum(axis=0).max())


def test_partitioned_sampled_matches_full():
    p = inputs.make_w4a16(7, 1280, 45, seed=16)
    rows, cols = np.array([0, 3, 6]), np.array([1, 2, 30, 44])
    for s in (1, 2, 5, 10):
        for mode in (0, 1):
            C, _ = oracle.qmm_partitioned(p["A"], p["Wq"], p["scales"], p["biases"], s, mode)
            S = oracle.qmm_partitioned_sampled(p["A"], p["Wq"], p["scales"], p["biases"], rows,
                                               cols, s, mode)
            assert np.array_equal(S, C[np.ix_(rows, cols)])
        _, P = oracle.qmm_partitioned(p["A"], p["Wq"], p["scales"], p["biases"], s, 0,
                                      with_partials=True)
        _, Ps = oracle.qmm_partitioned_sampled(p["A"], p["Wq"], p["scales"], p["biases"], rows,
                                               cols, s, 0, with_partials=True)
        assert np.array_equal(Ps, np.moveaxis(P, 0, 2)[np.ix_(rows, cols)])


def test_partitioned_rejects_split_beyond_the_groups():
    p = inputs.make_w4a16(1, 2560, 4, seed=12)
    with pytest.raises(ValueError):
        oracle.qmm_partitioned(p["A"], p["Wq"], p["scales"], p["biases"], 21, 0)
    with pytest.raises(ValueError):
        oracle.qmm_partitioned(p["A"], p["Wq"], p["scales"], p["biases"], 0, 0)


@pytest.mark.parametrize("G,s", [(10, 3), (10, 4), (10, 7), (11, 2), (20, 6), (7, 7), (20, 13)])
def test_near_equal_partition_boundaries(G, s):
    # a split that does not divide G: slices in order, the first G mod s one
    # group longer; activations nonzero only in group g light up one plane
    lengths = [G // s + 1] * (G % s) + [G // s] * (s - G % s)
    owner = [i for i, n in enumerate(lengths) for _ in range(n)]
    assert len(owner) == G
    p = inputs.make_w4a16(2, 128 * G, 8, seed=17)
    for g in range(G):
        a = np.zeros((2, 128 * G), np.uint16)
        a[:, g * 128:(g + 1) * 128] = p["A"][:, g * 128:(g + 1) * 128]
        _, P = oracle.qmm_partitioned(a, p["Wq"], p["scales"], p["biases"], s, 1,
                                      with_partials=True)
        nonzero = [bool(np.any(P[i] != 0)) for i in range(s)]
        assert nonzero == [i == owner[g] for i in range(s)], (g, nonzero)


@pytest.mark.parametrize("split", list(range(1, 12)))
def test_near_equal_partitions_cover_every_group(split):
    # integer weights (scale 1, bias 0) and integer activations: every plane is
    # an exact FP32 sum, so the planes add up to C64 exactly and C = BF16(C64);
    # a dropped or doubled group breaks the first equality
    rng = np.random.default_rng(18)
    G = 11
    M, Kred, Nout = 3, 128 * G, 5
    q = rng.integers(0, 16, (Nout, Kred)).astype(np.uint32)
    Wq = np.zeros((Nout, Kred // 8), np.uint32)
    for j in range(8):
        Wq |= q[:, j::8] << (4 * j)
    scales = np.full((Nout, G), _bf16_bits(1.0), np.uint16)
    biases = np.zeros((Nout, G), np.uint16)
    A = inputs.f32_to_bf16_bits(rng.integers(-2, 3, (M, Kred)).astype(np.float32))
    C64 = oracle.qmm(A, Wq, scales, biases, threads=2)
    assert np.array_equal(C64, _bits_to_f64(A) @ q.T.astype(np.float64))
    C, P = oracle.qmm_partitioned(A, Wq, scales, biases, split, 1, with_partials=True)
    if split > 1:
        assert np.array_equal(P.sum(axis=0), C64)
        assert all(np.any(P[i] != 0) for i in range(split))
    assert np.array_equal(C, oracle.bf16_round(C64))


# ---- policy and waves ------------------------------------------------------

def test_plan_pages_stated_schedules():
    gold = _golden("splitk_policy_pages.json")
    pol = gold["policy"]
    for c in gold["cases"]:
        s = oracle.splitk_plan(c["M"], c["Kred"], c["Nout"], pol["bm"], pol["bn"],
                               pol["target"], pol["cap"], pol["min_k"])
        assert s == c["split"], c


def _plan_property(M, Kred, Nout, bm, bn, target, cap, min_k):
    """The largest s >= 2 that divides Kred/128 and stays within every bound, else 1."""
    base = math.ceil(M / bm) * math.ceil(Nout / bn)
    ok = [s for s in range(2, Kred // 128 + 1)
          if (Kred // 128) % s == 0 and s <= cap and s * base <= target and s * min_k <= Kred]
    return max(ok) if ok else 1


def test_plan_matches_divisor_formulation():
    rng = np.random.default_rng(13)
    for _ in range(3000):
        M = int(rng.integers(1, 3000))
        Kred = 128 * int(rng.integers(1, 101))
        Nout = int(rng.integers(1, 12000))
        bm, bn = int(rng.choice([8, 16, 32, 64, 128])), int(rng.choice([32, 64, 128, 256]))
        target = int(rng.integers(0, 2000))
        cap = int(rng.integers(1, 33))
        min_k = 128 * int(rng.integers(1, 9))
        assert oracle.splitk_plan(M, Kred, Nout, bm, bn, target, cap, min_k) == \
            _plan_property(M, Kred, Nout, bm, bn, target, cap, min_k)


def _plan_near_equal_property(M, Kred, Nout, bm, bn, target, cap, min_k):
    """Among the splits within every bound (no divisibility), those whose
    longest partition, ceil(G/s) groups, is shortest; the smallest of them."""
    G = Kred // 128
    base = math.ceil(M / bm) * math.ceil(Nout / bn)
    ok = [s for s in range(1, G + 1)
          if s == 1 or (s <= cap and s * base <= target and s * min_k <= Kred)]
    best = min(-(-G // s) for s in ok)
    return min(s for s in ok if -(-G // s) == best)


def test_plan_near_equal_fuzz():
    rng = np.random.default_rng(19)
    agree = 0
    for _ in range(3000):
        M = int(rng.integers(1, 3000))
        Kred = 128 * int(rng.integers(1, 101))
        Nout = int(rng.integers(1, 12000))
        bm, bn = int(rng.choice([8, 16, 32, 64, 128])), int(rng.choice([32, 64, 128, 256]))
        target = int(rng.integers(0, 2000))
        cap = int(rng.integers(1, 33))
        min_k = 128 * int(rng.integers(1, 9))
        s = oracle.splitk_plan_near_equal(M, Kred, Nout, bm, bn, target, cap, min_k)
        assert s == _plan_near_equal_property(M, Kred, Nout, bm, bn, target, cap, min_k)
        d = oracle.splitk_plan(M, Kred, Nout, bm, bn, target, cap, min_k)
        # the divisor rule never splits further, and agrees when s divides G
        assert d <= s
        if (Kred // 128) % s == 0:
            assert d == s
            agree += 1
    assert agree > 100


def test_plan_near_equal_takes_the_models_best_one_wave_split():
    # the Split-K page's model: 16 output tiles, the largest split whose
    # blocks fit one wave -- 6 on 108 SMs, 8 on 132 -- for k = 16384 (128
    # groups), which 6 does not divide
    gold = _golden("splitk_waves_model.json")
    M, Nout = gold["output"]
    bm, bn = gold["tile"]
    for arch in ("a100", "h100"):
        s = oracle.splitk_plan_near_equal(M, 16384, Nout, bm, bn, gold[arch]["sms"], 16)
        assert s == gold[arch]["best_split_one_wave"]
    # the divisor rule stops at 4 on the A100 (128 groups)
    assert oracle.splitk_plan(M, 16384, Nout, bm, bn, gold["a100"]["sms"], 16) == 4


def test_waves_model_table():
    gold = _golden("splitk_waves_model.json")
    tiles = (gold["output"][0] // gold["tile"][0]) * (gold["output"][1] // gold["tile"][1])
    assert tiles == gold["tiles"]
    a = gold["a100"]
    for r in a["rows"]:
        assert tiles * r["split"] == r["blocks"]
        assert oracle.waves(tiles, r["split"], a["sms"]) == r["waves"]
    best = max(s for s in range(1, 64) if oracle.waves(tiles, s, a["sms"]) == 1)
    assert best == a["best_split_one_wave"]
    assert round(1 - tiles / a["sms"], 2) == a["idle_fraction_unsplit"]
    h = gold["h100"]
    best = max(s for s in range(1, 64) if oracle.waves(tiles, s, h["sms"]) == 1)
    assert best == h["best_split_one_wave"] and tiles * best == h["blocks"]


# ---- copy / compute overlap schedule --------------------------------------

def test_overlap_model_page_example():
    gold = _golden("overlap_model.json")
    c = gold["compute_heavy"]
    t = (c["t_load"], c["t_comp"], c["t_store"])
    for out_reuse in (False, True):
        T1 = oracle.overlap_schedule(c["tiles"], 1, *t, out_reuse=out_reuse)
        T2 = oracle.overlap_schedule(c["tiles"], 2, *t, out_reuse=out_reuse)
        T3 = oracle.overlap_schedule(c["tiles"], 3, *t, out_reuse=out_reuse)
        assert (T1, T2) == (c["T_one_buffer"], c["T_two_buffers"])
        assert round(T1 / T2, 2) == c["speedup"]
        assert gold["third_buffer_same_as_two_with_fixed_times"] and T3 == T2


def test_overlap_closed_forms():
    rng = np.random.default_rng(23)
    for _ in range(300):
        n = int(rng.integers(1, 40))
        tl, tc, ts = (float(x) for x in rng.integers(1, 50, 3))
        # one buffer: loads and computes alternate and the last store follows
        # (the page's T_1, for stores no slower than a load plus a compute);
        # slower stores queue behind the first compute instead
        T1 = oracle.overlap_schedule(n, 1, tl, tc, ts)
        if ts <= tl + tc:
            assert T1 == n * (tl + tc) + ts
        assert T1 == max(n * (tl + tc) + ts, tl + tc + n * ts)
        b = int(rng.integers(2, 6))
        hi = max(tl, tc, ts)
        # compute slowest: after the first load the compute engine never waits
        if tc == hi:
            assert oracle.overlap_schedule(n, b, tl, tc, ts) == tl + n * tc + ts
        # copy-in slowest: the loads run back to back and set the pace
        if tl == hi:
            assert oracle.overlap_schedule(n, b, tl, tc, ts) == n * tl + tc + ts


def _time_stepped(n, b, tl, tc, ts, out_reuse):
    """Integer-time simulation: at every tick each engine starts its next tile
    if it is idle and the tile's inputs are ready (a different procedure from
    the oracle's per-tile recurrence)."""
    INF = float("inf")
    end = {e: [INF] * n for e in ("l", "c", "s")}
    nxt = {"l": 0, "c": 0, "s": 0}
    busy_until = {"l": 0, "c": 0, "s": 0}
    t = 0
    while nxt["s"] < n:
        i = nxt["l"]
        if i < n and busy_until["l"] <= t and (i < b or end["c"][i - b] <= t):
            end["l"][i] = t + tl[i]; busy_until["l"] = end["l"][i]; nxt["l"] += 1
        i = nxt["c"]
        if i < n and busy_until["c"] <= t and end["l"][i] <= t and \
                (not out_reuse or i < b or end["s"][i - b] <= t):
            end["c"][i] = t + tc[i]; busy_until["c"] = end["c"][i]; nxt["c"] += 1
        i = nxt["s"]
        if i < n and busy_until["s"] <= t and end["c"][i] <= t:
            end["s"][i] = t + ts[i]; busy_until["s"] = end["s"][i]; nxt["s"] += 1
        if nxt["s"] == n:
            break
        t += 1
    return max(end["s"])


def test_overlap_schedule_matches_a_time_stepped_simulation():
    rng = np.random.default_rng(24)
    for _ in range(400):
        n = int(rng.integers(1, 12))
        b = int(rng.integers(1, 5))
        tl, tc, ts = (rng.integers(1, 8, n).astype(float) for _ in range(3))
        for out_reuse in (False, True):
            T, ev = oracle.overlap_schedule(n, b, tl, tc, ts, out_reuse=out_reuse,
                                            with_events=True)
            assert T == _time_stepped(n, b, tl, tc, ts, out_reuse)
            assert np.all(ev[:, 1] - ev[:, 0] == tl) and np.all(ev[:, 5] - ev[:, 4] == ts)


def test_overlap_more_buffers_never_hurt_and_help_only_with_varying_times():
    rng = np.random.default_rng(25)
    helped = False
    for _ in range(300):
        n = int(rng.integers(2, 20))
        tl, tc, ts = (rng.integers(1, 10, n).astype(float) for _ in range(3))
        Ts = [oracle.overlap_schedule(n, b, tl, tc, ts) for b in (1, 2, 3, 4)]
        assert all(a >= b for a, b in zip(Ts, Ts[1:]))
        helped |= Ts[2] < Ts[1]
    assert helped  # some varying-time schedule gains from a third buffer


# ---- split-KV decode attention ---------------------------------------------

def _attn_problem(B, Hq, Hkv, Lmax, D, seed, lens=None):
    rng = np.random.default_rng(seed)
    q = inputs.f32_to_bf16_bits(rng.standard_normal((B, Hq, D)).astype(np.float32))
    K = inputs.f32_to_bf16_bits(rng.standard_normal((B, Hkv, Lmax, D)).astype(np.float32))
    V = inputs.f32_to_bf16_bits(rng.standard_normal((B, Hkv, Lmax, D)).astype(np.float32))
    if lens is None:
        lens = rng.integers(1, Lmax + 1, B)
    return q, K, V, np.asarray(lens, np.int32)


def test_attention_matches_a_library_softmax():
    from scipy.special import softmax
    for (B, Hq, Hkv, Lmax, D) in [(1, 1, 1, 1, 8), (2, 4, 2, 9, 16), (3, 8, 1, 33, 32)]:
        q, K, V, lens = _attn_problem(B, Hq, Hkv, Lmax, D, seed=B + Lmax)
        O = oracle.decode_attention(q, K, V, lens, threads=2)
        qf, Kf, Vf = _bits_to_f64(q), _bits_to_f64(K), _bits_to_f64(V)
        for b in range(B):
            for h in range(Hq):
                g = h // (Hq // Hkv)
                L = lens[b]
                p = softmax(Kf[b, g, :L] @ qf[b, h] / np.sqrt(D))
                assert np.allclose(O[b, h], p @ Vf[b, g, :L], rtol=0, atol=1e-12)


def test_attention_closed_forms():
    B, Hq, Hkv, Lmax, D = 2, 4, 2, 40, 16
    q, K, V, lens = _attn_problem(B, Hq, Hkv, Lmax, D, seed=30, lens=[40, 23])
    Vf = _bits_to_f64(V)
    # every key of a sequence equal: uniform weights, the mean of the valid V rows
    Ku = np.repeat(K[:, :, :1, :], Lmax, axis=2)
    O = oracle.decode_attention(q, Ku, V, lens, threads=2)
    for b in range(B):
        for h in range(Hq):
            g = h // 2
            assert np.allclose(O[b, h], Vf[b, g, :lens[b]].mean(axis=0), rtol=0, atol=1e-12)
    # a constant V per KV head: every query head reads its own group's value
    Vc = np.zeros_like(V)
    for g in range(Hkv):
        Vc[:, g] = _bf16_bits(float(g + 1))
    O = oracle.decode_attention(q, K, Vc, lens, threads=2)
    for h in range(Hq):
        assert np.all(O[:, h] == h // (Hq // Hkv) + 1)
    # one key aligned with the query and far longer wins: O -> that key's V row
    qs = np.full((1, 1, D), _bf16_bits(1.0), np.uint16)
    Kd = np.zeros((1, 1, 16, D), np.uint16)
    Kd[0, 0, 5] = _bf16_bits(8.0)            # score 8 * D / sqrt(D) = 32; the rest 0
    Vd = V[:1, :1, :16]
    O = oracle.decode_attention(qs, Kd, Vd, [16], threads=1)
    bound = 15 * np.exp(-32.0) * np.abs(_bits_to_f64(Vd)).max() * 2
    assert np.all(np.abs(O[0, 0] - _bits_to_f64(Vd)[0, 0, 5]) <= bound)


def test_attention_ignores_positions_past_the_length():
    q, K, V, lens = _attn_problem(3, 4, 4, 30, 16, seed=31, lens=[30, 7, 1])
    O = oracle.decode_attention(q, K, V, lens, threads=2)
    K2, V2 = K.copy(), V.copy()
    for b, L in enumerate(lens):
        K2[b, :, L:] = _bf16_bits(100.0)
        V2[b, :, L:] = _bf16_bits(-1000.0)
    assert np.array_equal(O, oracle.decode_attention(q, K2, V2, lens, threads=2))


def test_attention_shift_invariance():
    # adding one vector t to every key shifts all scores of a query by q.t:
    # the softmax, and O, stay the same (integer values keep K + t exact)
    rng = np.random.default_rng(32)
    B, H, L, D = 2, 3, 25, 16
    q = inputs.f32_to_bf16_bits(rng.integers(-3, 4, (B, H, D)).astype(np.float32))
    Kf = rng.integers(-3, 4, (B, H, L, D)).astype(np.float32)
    K = inputs.f32_to_bf16_bits(Kf)
    K2 = inputs.f32_to_bf16_bits(Kf + rng.integers(-5, 6, (1, 1, 1, D)).astype(np.float32))
    V = inputs.f32_to_bf16_bits(rng.standard_normal((B, H, L, D)).astype(np.float32))
    lens = np.array([25, 11], np.int32)
    O1 = oracle.decode_attention(q, K, V, lens, scale=0.1, threads=2)
    O2 = oracle.decode_attention(q, K2, V, lens, scale=0.1, threads=2)
    assert np.allclose(O1, O2, rtol=0, atol=1e-12)


@pytest.mark.parametrize("chunk", [1, 3, 7, 16, 64, 1000])
def test_split_kv_lse_merge_is_exact_and_the_naive_merge_is_not(chunk):
    q, K, V, lens = _attn_problem(3, 8, 2, 64, 32, seed=33, lens=[64, 45, 9])
    O = oracle.decode_attention(q, K, V, lens, threads=2)
    Os = oracle.decode_attention_split(q, K, V, lens, chunk, "lse", threads=2)
    assert np.allclose(Os, O, rtol=0, atol=1e-12)
    On = oracle.decode_attention_split(q, K, V, lens, chunk, "naive", threads=2)
    if chunk < 64:  # more than one chunk somewhere: the naive mean is wrong
        assert np.abs(On - O).max() > 1e-3
    else:
        assert np.allclose(On, O, rtol=0, atol=1e-12)


def test_attention_split_factor():
    rng = np.random.default_rng(34)
    for _ in range(2000):
        B, Hkv = int(rng.integers(1, 65)), int(rng.integers(1, 17))
        Lmax, sms = int(rng.integers(1, 40000)), int(rng.integers(1, 200))
        bps, mc = int(rng.integers(1, 5)), int(rng.integers(1, 2049))
        S = oracle.attention_splits(B, Hkv, Lmax, sms, bps, mc)
        # the smallest S whose grid reaches the target, unless the chunk floor binds
        cap = max(1, Lmax // mc)
        want = next(s for s in range(1, 10 ** 6) if s * B * Hkv >= sms * bps)
        assert S == min(want, cap) and S >= 1
        if S > 1:
            assert Lmax // S >= mc


# ---- dense GEMM ------------------------------------------------------------

def test_gemm_exact_brute_force():
    d = inputs.make_dense(3, 4, 96, seed=14)
    C = oracle.gemm(d["A"], d["W"], threads=1)
    a, w = _bits_to_f64(d["A"]), _bits_to_f64(d["W"])
    for m in range(3):
        for n in range(4):
            exact = sum((Fraction(a[m, k]) * Fraction(w[n, k]) for k in range(96)), Fraction(0))
            assert abs(Fraction(C[m, n]) - exact) <= Fraction(float(np.abs(a[m]) @ np.abs(w[n]))) \
                * Fraction(1, 2 ** 45)


@pytest.mark.parametrize("split", [1, 2, 4, 6, 7, 9, 12, 16])
def test_gemm_partitioned_covers_every_tile(split):
    # integer-valued operands: every partial and sum is exact, so C = BF16(C64)
    # for any split; a dropped or doubled k-tile would change the result
    rng = np.random.default_rng(15)
    K = 64 * 37
    a = inputs.f32_to_bf16_bits(rng.integers(-2, 3, (5, K)).astype(np.float32))
    w = inputs.f32_to_bf16_bits(rng.integers(-2, 3, (6, K)).astype(np.float32))
    C64 = oracle.gemm(a, w, threads=2)
    C = oracle.gemm_partitioned(a, w, split, ktile=64, threads=2)
    assert np.array_equal(C, oracle.bf16_round(C64))
    ones = np.full((1, K), 0x3F80, np.uint16)
    assert oracle.bf16_value(oracle.gemm_partitioned(ones, ones, split, 64))[0, 0] == \
        oracle.bf16_value(oracle.bf16_round(np.array([float(K)])))[0]


# ---- group plan (the grouped call's opt-in split plan) ------------------------

def _tc_tiles(M):
    """The tcgen05 kernel table: tiles of 16/32/64/128/256 activation rows x 128 columns."""
    for bm in (16, 32, 64, 128):
        if M <= bm:
            return bm, 128
    return 256, 128


def test_group_plan_single_call_by_hand():
    # k at M = 32: 8 tiles of 20 groups on 152 SMs, one tile per SM each step.
    # A tile costs 3 + 0.40 * (its groups); planes 2 * s * 32 * 1024 * 2 B at 3 TB/s.
    # s=1: 3 + 8.0 = 11.0; s=2: 3 + 4.0 + 0.0874 = 7.0874; s=4: 5.0 + 0.1748;
    # s=5: 4.6 + 0.2185; s=10: 3.8 + 0.4369 = 4.2369; 20 is over the cap of 16.
    trace = []
    s = oracle.group_plan([(32, 2560, 1024)], _tc_tiles, 152, trace=trace)
    assert s == [10]
    assert [t[0] for t in trace] == [[1], [2], [4], [5], [10]]
    plane = lambda k: k * 32 * 1024 * 2 * 2 / 3.0e6
    want = [11.0, 7.0 + plane(2), 5.0 + plane(4), 4.6 + plane(5), 3.8 + plane(10)]
    assert np.allclose([t[1] for t in trace], want, rtol=0, atol=1e-12)


def test_group_plan_wave_tail_by_hand():
    # down at M = 2048: 160 tiles of 256 rows on 152 SMs.
    # s=1: tiles of 3 + 76 * 0.6 = 48.6; eight SMs run two -> 97.2.
    # s=2: 320 tiles of 3 + 38 * 0.6 = 25.8; sixteen SMs run three -> 77.4,
    #      plus planes 2 * 2048 * 2560 * 2 * 2 B / 3e6 = 13.98 -> 91.38 (kept).
    # s=4: 640 tiles of 14.4, five rounds -> 72.0 + 27.96 = 99.96 (not kept).
    trace = []
    assert oracle.group_plan([(2048, 9728, 2560)], _tc_tiles, 152, trace=trace) == [2]
    planes = 2 * 2048 * 2560 * 2 * 2 / 3.0e6
    assert np.isclose(trace[0][1], 97.2) and np.isclose(trace[1][1], 77.4 + planes)
    # o at M = 2048: 160 tiles of 3 + 32 * 0.6 = 22.2 -> 44.4; split 2 gives
    # 320 tiles of 12.6 (three rounds, 37.8) plus 13.98 of planes: not kept.
    assert oracle.group_plan([(2048, 4096, 2560)], _tc_tiles, 152) == [1]


def test_group_plan_agrees_with_the_chapter_policy_on_single_calls():
    # For one call that under-fills the GPU the plan ends where the chapter's
    # occupancy rule does (the workload's shapes at M = 32 and 128).
    for M in (32, 128):
        for name, (Kred, Nout) in inputs.PROJECTIONS.items():
            bm, bn = _tc_tiles(M)
            pol = oracle.splitk_plan(M, Kred, Nout, bm, bn, 152, 16)
            assert oracle.group_plan([(M, Kred, Nout)], _tc_tiles, 152) == [pol], (M, name)


def test_group_plan_on_a_full_group():
    shapes = lambda M: [(M,) + inputs.PROJECTIONS[n] for n in inputs.PROJECTIONS]
    # the seven projections already fill the GPU together: only down, whose
    # partitions are the longest, splits; nothing splits at M = 2048
    assert oracle.group_plan(shapes(32), _tc_tiles, 152) == [1, 1, 1, 1, 1, 1, 4]
    assert oracle.group_plan(shapes(128), _tc_tiles, 152) == [1, 1, 1, 1, 1, 1, 2]
    assert oracle.group_plan(shapes(2048), _tc_tiles, 152) == [1] * 7


def test_group_plan_invariants():
    rng = np.random.default_rng(11)
    for _ in range(40):
        n = int(rng.integers(1, 8))
        M = int(rng.choice([1, 4, 16, 32, 64, 128, 300]))
        shapes = [(M, 128 * int(rng.integers(1, 100)), int(rng.integers(1, 6000)))
                  for _ in range(n)]
        near = bool(rng.integers(0, 2))
        trace = []
        s = oracle.group_plan(shapes, _tc_tiles, 152, near_equal=near, trace=trace)
        costs = [t[1] for t in trace]
        assert all(b < a for a, b in zip(costs, costs[1:]))  # every kept move lowers the cost
        for (m, K, N), v in zip(shapes, s):
            G = K // 128
            assert 1 <= v <= min(16, G)
            assert near or G % v == 0
            if m <= 8:
                assert v == 1 or K // v >= 512
    # ties between equally long calls go to the lower index
    assert oracle.group_plan([(32, 2560, 1024), (32, 2560, 1024)], _tc_tiles, 152)[0] >= \
        oracle.group_plan([(32, 2560, 1024), (32, 2560, 1024)], _tc_tiles, 152)[1]


def test_group_plan_own_launch_keeps_the_single_call_split():
    # A call that runs in a launch of its own is not planned with the others:
    # it keeps the chapter's occupancy split under its own policy, whatever
    # the calls beside it, and the shared launch is planned as if it were
    # absent.
    lean = (16, 64, 304, 16, 128)
    own = lambda M: lean if M <= 32 else None
    shapes = [(16, 2560, 1024), (16, 9728, 2560), (128, 2560, 1024), (128, 9728, 2560)]
    s = oracle.group_plan(shapes, _tc_tiles, 152, own_launch=own)
    assert s[0] == oracle.splitk_plan(16, 2560, 1024, *lean) == 10
    assert s[1] == oracle.splitk_plan(16, 9728, 2560, *lean) == 4
    assert s[2:] == oracle.group_plan(shapes[2:], _tc_tiles, 152)
    ne = oracle.group_plan(shapes[:2], _tc_tiles, 152, near_equal=True, own_launch=own)
    assert ne == [oracle.splitk_plan_near_equal(16, 2560, 1024, *lean),
                  oracle.splitk_plan_near_equal(16, 9728, 2560, *lean)]
