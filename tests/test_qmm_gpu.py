"""GPU parity tests: the CUDA path through the C ABI against the CPU oracle.

Tolerances, per element:
  BF16 partial planes (split > 1): |C_gpu - C_emu| <= 0.02 * max(1, |C_emu|),
      C_emu = the oracle's partition emulation (same split, each partition's
      fp64 sum rounded to BF16, planes added in FP32, one BF16 cast) -- the
      arithmetic the chapter specifies for the split path; and, against the
      fp64 C64, the bound that arithmetic implies: 2^-8 per BF16 rounding of
      every plane and of C.
  FP32 partial planes or split 1: |C_gpu - C64| <= 0.008 * max(1, |C64|).
Unpacking, dequantized weights, split plans and the reduce are bit-exact.
"""
import ctypes

import time

import numpy as np
import pytest
import torch

import oracle
from split_w4a16_quantized_gb300 import build, inputs
from split_w4a16_quantized_gb300 import qmm as Q

pytestmark = pytest.mark.gpu

TOL_BF16, TOL_F32 = 0.02, 0.008
NAN_BF16 = 0x7FC0
CANARY = 64


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()


KERNELS = {"default": Q.QMM_KERNELS_DEFAULT, "mma": Q.QMM_KERNELS_MMA_SYNC,
           "tc": Q.QMM_KERNELS_TCGEN05, "lean": Q.QMM_KERNELS_LEAN}


@pytest.fixture(params=["mma", "tc", "lean"])
def family(request):
    """Run the test once per kernel family table; check the status word after."""
    prev = Q.qmm_set_kernels(KERNELS[request.param])
    Q.qmm_kernel_status(clear=True)
    yield request.param
    try:
        assert Q.qmm_kernel_status(clear=True) == 0, "a bounded wait ran out in a kernel"
    finally:
        Q.qmm_set_kernels(prev)


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def _val(bits: np.ndarray) -> np.ndarray:
    return inputs.bf16_bits_to_f32(bits).astype(np.float64)


def _tol(split: int, partial_dtype: int) -> float:
    return TOL_BF16 if split > 1 and partial_dtype == Q.QMM_PARTIAL_BF16 else TOL_F32


def _assert_close(got_bits, ref64, tol, what=""):
    got = _val(got_bits)
    assert np.all(np.isfinite(got)), "non-finite output " + what
    err = np.abs(got - ref64)
    lim = tol * np.maximum(1.0, np.abs(ref64))
    bad = np.argwhere(err > lim)
    assert bad.size == 0, "%s: %d elements out of tolerance, first %s err %g lim %g" % (
        what, len(bad), bad[0], err[tuple(bad[0])], lim[tuple(bad[0])])


def _ulp_bf16(x):
    """One BF16 unit in the last place at |x| (8 significant bits); 0 at 0."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, 2.0 ** (e - 7), 0.0)


def _assert_emulated(got_bits, emu_bits, planes, what):
    """Within 0.02 * max(1, |C_emu|) of the partition emulation, widened per
    element by one BF16 ulp of each partial plane (planes: [..., split]): the
    GPU forms each partition sum in FP32 in its own order, so when the exact
    sum sits within FP32 error of a BF16 rounding boundary the plane may round
    to the other neighbour -- a one-ulp step that, for planes much larger than
    their sum, exceeds 0.02 * max(1, |C|) on its own."""
    emu = _val(emu_bits)
    got = _val(got_bits)
    assert np.all(np.isfinite(got)), "non-finite output " + what
    lim = TOL_BF16 * np.maximum(1.0, np.abs(emu)) + _ulp_bf16(planes).sum(axis=-1)
    err = np.abs(got - emu)
    bad = np.argwhere(err > lim)
    assert bad.size == 0, "%s: %d elements out of tolerance, first %s err %g lim %g" % (
        what, len(bad), bad[0], err[tuple(bad[0])], lim[tuple(bad[0])])


def _check_full(p, got_bits, split, dt, C64, what=""):
    """Whole-output parity of one call (see the module docstring)."""
    if split > 1 and dt == Q.QMM_PARTIAL_BF16:
        emu, planes = oracle.qmm_partitioned(p["A"], p["Wq"], p["scales"], p["biases"], split, 0,
                                             with_partials=True)
        _assert_emulated(got_bits, emu, np.moveaxis(planes, 0, -1),
                         what + " vs BF16-partial emulation")
        bound = 2.0 ** -8 * (1 + 2.0 ** -7) * (np.abs(planes).sum(axis=0) + np.abs(C64)) \
            + 1e-4 * np.maximum(1.0, np.abs(C64))
        err = np.abs(_val(got_bits) - C64)
        assert np.all(err <= bound), what + ": error above the BF16-partial bound, max excess %g" \
            % (err - bound).max()
    else:
        _assert_close(got_bits, C64, TOL_F32, what)


def _check_sampled(p, got_bits, split, dt, rows, cols, what=""):
    got = got_bits[np.ix_(rows, cols)]
    if split > 1 and dt == Q.QMM_PARTIAL_BF16:
        emu, planes = oracle.qmm_partitioned_sampled(p["A"], p["Wq"], p["scales"], p["biases"],
                                                     rows, cols, split, 0, with_partials=True)
        _assert_emulated(got, emu, planes, what + " vs BF16-partial emulation")
    else:
        ref = oracle.qmm_sampled(p["A"], p["Wq"], p["scales"], p["biases"], rows, cols)
        _assert_close(got, ref, TOL_F32, what)


def _run(d, M, Nout, split_req=0, pol=None, partial_dtype=Q.QMM_PARTIAL_BF16,
         plan=Q.qmm_splitk_plan):
    """Call qmm_w4a16_g128 into a NaN-filled C with a canary tail; returns (C bits, split).
    plan: the split plan of the partition rule in force."""
    Kred = d["A"].shape[1]
    if split_req == 0:
        p = pol or Q.qmm_policy_preset(Q.QMM_PRESET_GB300, M)
        split = plan(M, Kred, Nout, p)
    else:
        split = split_req
    nbytes = Q.qmm_splitk_workspace_bytes(M, Nout, split, partial_dtype)
    ws = torch.full((max(nbytes, 16) // 2,), float("nan"), dtype=torch.bfloat16, device="cuda")
    buf = torch.full((M * Nout + CANARY,), 0, dtype=torch.int16, device="cuda")
    buf.fill_(NAN_BF16)
    C = buf[:M * Nout].view(torch.bfloat16).view(M, Nout)
    used = Q.qmm_w4a16_g128(d["A"], d["Wq"], d["scales"], d["biases"], C, split_req=split_req,
                            pol=pol, workspace=ws if nbytes else None, partial_dtype=partial_dtype)
    torch.cuda.synchronize()
    assert np.all(buf[M * Nout:].cpu().numpy() == np.int16(NAN_BF16)), "canary overwritten"
    assert used == split
    return _bits(C), used


# ---- probes: bit-exact -----------------------------------------------------

@pytest.mark.parametrize("Nout,Kred", [(1000, 2560), (37, 256), (16, 128)])
def test_unpack_probe_bit_exact(Nout, Kred):
    p = inputs.make_w4a16(1, Kred, Nout, seed=31)
    d = Q.to_device(p)
    q = torch.empty((Nout, Kred), dtype=torch.uint8, device="cuda")
    Q.qmm_unpack_probe(d["Wq"], Kred, q)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), oracle.unpack(p["Wq"], Kred))


@pytest.mark.parametrize("Nout,Kred", [(1000, 2560), (37, 256)])
def test_dequant_probe_bit_exact(Nout, Kred):
    p = inputs.make_w4a16(1, Kred, Nout, seed=32)
    d = Q.to_device(p)
    w = torch.empty((Nout, Kred), dtype=torch.bfloat16, device="cuda")
    Q.qmm_dequant_probe(d["Wq"], d["scales"], d["biases"], Kred, w)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(w), oracle.dequant(p["Wq"], p["scales"], p["biases"], Kred))


def _mixed_scales(Nout, G, rng):
    """BF16 scale and bias bits spanning both dequant paths: magnitudes from
    2^-12 to 2^-1 (the subnormal-nibble path serves |scale| < 2^-5), both
    signs, exact zeros, and the two exponents on either side of the switch
    (largest below 2^-5 and 2^-5 itself)."""
    mag = 2.0 ** rng.uniform(-12, -1, (Nout, G))
    sgn = np.where(rng.random((Nout, G)) < 0.2, -1.0, 1.0)
    sc = inputs.f32_to_bf16_bits((mag * sgn).astype(np.float32))
    sc[rng.random((Nout, G)) < 0.05] = 0
    sc[0, 0], sc[1 % Nout, 0] = 0x3CFF, 0x3D00  # 0.0311 (last fast) and 2^-5 (first slow)
    bias = inputs.f32_to_bf16_bits((rng.normal(0, 0.05, (Nout, G))).astype(np.float32))
    return sc, bias


@pytest.mark.parametrize("Nout,Kred", [(1000, 2560), (37, 256)])
def test_dequant_probe_both_paths_bit_exact(Nout, Kred):
    rng = np.random.default_rng(33)
    p = inputs.make_w4a16(1, Kred, Nout, seed=33)
    p["scales"], p["biases"] = _mixed_scales(Nout, Kred // 128, rng)
    d = Q.to_device(p)
    w = torch.empty((Nout, Kred), dtype=torch.bfloat16, device="cuda")
    Q.qmm_dequant_probe(d["Wq"], d["scales"], d["biases"], Kred, w)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(w), oracle.dequant(p["Wq"], p["scales"], p["biases"], Kred))


@pytest.mark.parametrize("M", [1, 8, 16, 32, 64])
def test_mixed_scale_ranges_against_oracle(family, M):
    """Whole calls whose groups mix scales on both sides of the
    subnormal-nibble limit: the lean kernel takes the two-step dequant for a
    group of a CTA as soon as one of its rows needs it, the other kernels
    decide per scale, so every mix appears."""
    rng = np.random.default_rng(34 + M)
    Kred, Nout = 1280, 200
    p = inputs.make_w4a16(M, Kred, Nout, seed=34 + M)
    p["scales"], p["biases"] = _mixed_scales(Nout, Kred // 128, rng)
    d = Q.to_device(p)
    C64 = oracle.qmm(p["A"], p["Wq"], p["scales"], p["biases"])
    for split_req in (1, 2, 5):
        for dt in (Q.QMM_PARTIAL_BF16, Q.QMM_PARTIAL_F32):
            got, s = _run(d, M, Nout, split_req, partial_dtype=dt)
            _check_full(p, got, s, dt, C64, "M=%d req=%d dt=%d" % (M, split_req, dt))


# ---- the K-projection at M = 16 (policy vs unsplit) ------------------------

@pytest.mark.parametrize("M", [1, 16, 40, 128, 300])
def test_one_hot_weights_copy_activations(family, M):
    # q[n, k] = 1 at k = n, scale 1, bias 0: C = A[:, :Nout] exactly, which
    # pins the k order and the row/column mapping of every kernel family
    Kred, Nout = 256, 200
    q = np.zeros((Nout, Kred), np.uint8)
    q[np.arange(Nout), np.arange(Nout)] = 1
    prob = inputs.make_w4a16(M, Kred, Nout, seed=40)
    prob["Wq"] = inputs.pack_nibbles(q)
    prob["scales"] = np.full((Nout, 2), 0x3F80, np.uint16)
    prob["biases"] = np.zeros((Nout, 2), np.uint16)
    d = Q.to_device(prob)
    for split_req in (1, 2):
        got, _ = _run(d, M, Nout, split_req, partial_dtype=Q.QMM_PARTIAL_F32)
        assert np.array_equal(got, prob["A"][:, :Nout]), "split %d" % split_req


@pytest.mark.parametrize("partial_dtype", [Q.QMM_PARTIAL_BF16, Q.QMM_PARTIAL_F32])
def test_k_projection_m16_policy_and_unsplit(partial_dtype):
    Kred, Nout = inputs.PROJECTIONS["k"]
    p = inputs.make_w4a16(16, Kred, Nout, seed=0)
    d = Q.to_device(p)
    C64 = oracle.qmm(p["A"], p["Wq"], p["scales"], p["biases"])
    got, s = _run(d, 16, Nout, 0, partial_dtype=partial_dtype)
    assert s > 1, "an under-filled grid must split"
    _check_full(p, got, s, partial_dtype, C64, "policy")
    got1, s1 = _run(d, 16, Nout, 1)
    assert s1 == 1
    _assert_close(got1, C64, TOL_F32, "unsplit")


@pytest.mark.parametrize("name,splits", [("k", [2, 4, 5, 10, 20]), ("o", [2, 4, 8, 16, 32]),
                                         ("down", [2, 4, 19, 38, 76])])
def test_forced_splits(family, name, splits):
    Kred, Nout = inputs.PROJECTIONS[name]
    p = inputs.make_w4a16(16, Kred, Nout, seed=1)
    d = Q.to_device(p)
    C64 = oracle.qmm(p["A"], p["Wq"], p["scales"], p["biases"])
    for s in splits:
        for dt in (Q.QMM_PARTIAL_BF16, Q.QMM_PARTIAL_F32):
            got, used = _run(d, 16, Nout, s, partial_dtype=dt)
            _check_full(p, got, s, dt, C64, "%s s=%d dt=%d" % (name, s, dt))


# ---- every kernel family, ragged tiles -------------------------------------

@pytest.mark.parametrize("M", [1, 3, 8, 9, 16, 17, 31, 32, 33, 64, 65, 100, 128, 129, 300])
def test_families_ragged(family, M):
    Kred, Nout = 1280, 1000  # Nout = 1000: partial last column tile
    p = inputs.make_w4a16(M, Kred, Nout, seed=100 + M)
    d = Q.to_device(p)
    C64 = oracle.qmm(p["A"], p["Wq"], p["scales"], p["biases"])
    for split_req in (0, 1, 2, 5, 10):
        for dt in (Q.QMM_PARTIAL_BF16, Q.QMM_PARTIAL_F32):
            got, s = _run(d, M, Nout, split_req, partial_dtype=dt)
            _check_full(p, got, s, dt, C64, "M=%d req=%d dt=%d" % (M, split_req, dt))


def test_odd_output_width_scalar_stores():
    M, Kred, Nout = 5, 512, 77
    p = inputs.make_w4a16(M, Kred, Nout, seed=7)
    d = Q.to_device(p)
    C64 = oracle.qmm(p["A"], p["Wq"], p["scales"], p["biases"])
    for split_req in (1, 2, 4):
        got, s = _run(d, M, Nout, split_req)
        _check_full(p, got, s, Q.QMM_PARTIAL_BF16, C64, "req=%d" % split_req)


def test_minimum_shape():
    p = inputs.make_w4a16(1, 128, 1, seed=8)
    d = Q.to_device(p)
    got, s = _run(d, 1, 1, 0)
    _assert_close(got, oracle.qmm(p["A"], p["Wq"], p["scales"], p["biases"]), TOL_F32)


# ---- the projection workloads at full size, sampled ------------------------

def _sample(M, Nout, rng):
    rows = np.unique(np.concatenate([[0, M - 1], rng.integers(0, M, 6)]))
    cols = np.unique(np.concatenate([[0, Nout - 1], rng.integers(0, Nout, 126)]))
    return rows, cols


@pytest.mark.parametrize("M", [16, 32, 64, 128, 2048])
@pytest.mark.parametrize("name", list(inputs.PROJECTIONS) + ["ragged"])
def test_projection_full_size_sampled(name, M):
    Kred, Nout = inputs.RAGGED if name == "ragged" else inputs.PROJECTIONS[name]
    p = inputs.make_w4a16(M, Kred, Nout, seed=0)
    d = Q.to_device(p)
    rng = np.random.default_rng(M * 7 + Nout)
    rows, cols = _sample(M, Nout, rng)
    got, s = _run(d, M, Nout, 0)
    _check_sampled(p, got, s, Q.QMM_PARTIAL_BF16, rows, cols, "policy s=%d" % s)
    got1, _ = _run(d, M, Nout, 1)
    _check_sampled(p, got1, 1, Q.QMM_PARTIAL_BF16, rows, cols, "unsplit")
    # properties at every element: the split and the unsplit control agree up to
    # the BF16-partial rounding noise (aggregate) and never differ grossly
    a, b = _val(got), _val(got1)
    assert np.all(np.isfinite(a)) and np.all(np.isfinite(b))
    assert np.linalg.norm(a - b) <= 0.01 * np.linalg.norm(b), "split vs unsplit (L2)"
    assert np.all(np.abs(a - b) <= 0.25 * np.maximum(1.0, np.abs(b))), "split vs unsplit (max)"


CENSUS = [("k", 16)] + [(n, M) for M in (32, 128) for n in inputs.PROJECTIONS] + \
    [(n, M) for M in (1, 4, 8) for n in ("k", "o", "down")]


@pytest.mark.parametrize("name,M", CENSUS)
def test_plain_bar_census(name, M):
    """The plain bar |C_gpu - C64| <= 0.02 * max(1, |C64|) on the config inputs
    (seed 0) at the policy split.  With BF16 partial planes the chapter's own
    arithmetic misses it where the planes are much larger than C (one BF16
    rounding of a plane of magnitude 8 is 2^-6 already): the oracle's partition
    emulation misses it there too.  So: wherever the emulation meets the bar
    with room for the GPU's one-ulp plane differences, the GPU meets it; every
    element the GPU leaves outside is one the method itself leaves outside
    (within that room); and the whole output meets the emulation bar."""
    Kred, Nout = inputs.PROJECTIONS[name]
    p = inputs.make_w4a16(M, Kred, Nout, seed=0)
    got, s = _run(Q.to_device(p), M, Nout, 0)
    C64 = oracle.qmm(p["A"], p["Wq"], p["scales"], p["biases"])
    if s == 1:
        _assert_close(got, C64, TOL_F32, "%s M=%d unsplit" % (name, M))
        return
    lim = TOL_BF16 * np.maximum(1.0, np.abs(C64))
    gerr = np.abs(_val(got) - C64)
    emu, planes = oracle.qmm_partitioned(p["A"], p["Wq"], p["scales"], p["biases"], s, 0,
                                         with_partials=True)
    eerr = np.abs(_val(emu) - C64)
    room = _ulp_bf16(planes).sum(axis=0) + _ulp_bf16(C64)
    sure = eerr + room <= lim
    assert np.all(gerr[sure] <= lim[sure]), "plain bar missed where the method meets it"
    out = gerr > lim
    assert np.all(eerr[out] + room[out] > lim[out]), "a miss the method does not share"
    # the census itself (elements outside the plain bar): GPU against emulation
    assert abs(int(out.sum()) - int((eerr > lim).sum())) <= max(2, int(0.02 * (eerr > lim).sum()))
    _check_full(p, got, s, Q.QMM_PARTIAL_BF16, C64, "%s M=%d s=%d" % (name, M, s))


@pytest.mark.parametrize("name,M,req", [("gate", 2048, 0), ("down", 2048, Q.QMM_SPLIT_PLANNED),
                                        ("down", 128, 0)])
def test_full_size_every_element(name, M, req):
    """Every output element at full size against the oracle: the fall-back
    shape (gate, M = 2048, unsplit), down at M = 2048 at the group plan's
    split, and down at M = 128 at the policy's split."""
    Kred, Nout = inputs.PROJECTIONS[name]
    p = inputs.make_w4a16(M, Kred, Nout, seed=3)
    d = Q.to_device(p)
    s_want = Q.qmm_group_plan([(M, Kred, Nout)])[0] if req else 0
    got, s = _run(d, M, Nout, req if not req else s_want)
    C64 = oracle.qmm(p["A"], p["Wq"], p["scales"], p["biases"])
    _check_full(p, got, s, Q.QMM_PARTIAL_BF16, C64, "%s M=%d s=%d" % (name, M, s))
    if name == "gate":
        assert s == 1


def test_fallback_shape_runs_the_unsplit_kernel_exactly():
    # base grid already fills the target: the policy must pick split 1 and the
    # result must be bit-identical to the unsplit control
    Kred, Nout = inputs.PROJECTIONS["gate"]
    M = 2048
    p = inputs.make_w4a16(M, Kred, Nout, seed=2)
    d = Q.to_device(p)
    for pol in (Q.qmm_policy_preset(Q.QMM_PRESET_PAGES), None):
        got, s = _run(d, M, Nout, 0, pol=pol)
        assert s == 1
        got1, _ = _run(d, M, Nout, 1)
        assert np.array_equal(got, got1)


@pytest.mark.parametrize("M", [1, 4, 8])
@pytest.mark.parametrize("name", ["k", "o", "down"])
def test_decode_regime(family, name, M):
    Kred, Nout = inputs.PROJECTIONS[name]
    p = inputs.make_w4a16(M, Kred, Nout, seed=3)
    d = Q.to_device(p)
    C64 = oracle.qmm(p["A"], p["Wq"], p["scales"], p["biases"])
    got, s = _run(d, M, Nout, 0)
    assert Kred // s >= 512, "decode splits keep >= 512 reduction elements"
    _check_full(p, got, s, Q.QMM_PARTIAL_BF16, C64, "s=%d" % s)


def test_deterministic(family):
    Kred, Nout = inputs.PROJECTIONS["k"]
    p = inputs.make_w4a16(32, Kred, Nout, seed=4)
    d = Q.to_device(p)
    a, _ = _run(d, 32, Nout, 0)
    b, _ = _run(d, 32, Nout, 0)
    assert np.array_equal(a, b)


# ---- the reduce on its own: bit-exact --------------------------------------

@pytest.mark.parametrize("split", [1, 2, 3, 7, 16])
@pytest.mark.parametrize("M,Nout", [(16, 1024), (5, 77), (3, 8)])
@pytest.mark.parametrize("dt", [Q.QMM_PARTIAL_BF16, Q.QMM_PARTIAL_F32])
def test_reduce_bit_exact(split, M, Nout, dt):
    rng = np.random.default_rng(split * 1000 + M + Nout)
    planes = rng.standard_normal((split, M, Nout)).astype(np.float32) * 4
    if dt == Q.QMM_PARTIAL_BF16:
        bits = inputs.f32_to_bf16_bits(planes)
        planes = inputs.bf16_bits_to_f32(bits)
        dev = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    else:
        dev = torch.from_numpy(planes).cuda()
    acc = np.zeros((M, Nout), np.float32)
    for p in range(split):  # FP32, ascending partition
        acc = (acc + planes[p]).astype(np.float32)
    want = inputs.f32_to_bf16_bits(acc)
    C = torch.empty((M, Nout), dtype=torch.bfloat16, device="cuda")
    Q.qmm_splitk_reduce(dev, dt, split, M, Nout, C)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(C), want)


# ---- the partition kernel on its own: planes against the oracle -----------

def _partition(d, M, Nout, split, dt):
    tdt = torch.float32 if dt == Q.QMM_PARTIAL_F32 else torch.bfloat16
    planes = torch.full((split, M, Nout), float("nan"), dtype=tdt, device="cuda")
    Q.qmm_w4a16_g128_partition(d["A"], d["Wq"], d["scales"], d["biases"], planes, split, dt)
    torch.cuda.synchronize()
    return planes


def test_plane_sum_rounds_as_the_fp32_reduce(family):
    """Planes 1, 2^-8 and 2^-30 (one group each): the chapter's FP32 ascending
    sum ties at 1 + 2^-8 and rounds to 1, where the exact sum would round to
    1 + 2^-7 (the oracle case of the same name), for the separate reduce and
    the fused one."""
    A = np.zeros((1, 384), np.uint16)
    A[0, [0, 128, 256]] = 0x3F80
    q = np.zeros((1, 384), np.uint8)
    q[0, [0, 128, 256]] = 1
    p = {"A": A, "Wq": inputs.pack_nibbles(q),
         "scales": np.array([[0x3F80, 0x3B80, 0x3080]], np.uint16),
         "biases": np.zeros((1, 3), np.uint16)}
    want, _ = oracle.qmm_partitioned(p["A"], p["Wq"], p["scales"], p["biases"], 3, 0)
    assert int(want[0, 0]) == 0x3F80
    d = Q.to_device(p)
    got, s = _run(d, 1, 1, 3)
    assert s == 3 and int(got[0, 0]) == 0x3F80
    prev = Q.qmm_set_reduce(Q.QMM_REDUCE_FUSED)
    try:
        nb = Q.qmm_splitk_workspace_bytes(1, 1, 3, Q.QMM_PARTIAL_BF16)
        ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")  # fused counters start at zero
        got = _call_with(d, 1, 1, 3, Q.QMM_PARTIAL_BF16, ws)
        assert int(got[0, 0]) == 0x3F80
    finally:
        Q.qmm_set_reduce(prev)


@pytest.mark.parametrize("M,Nout", [(40, 1000), (128, 256), (3, 136)])
@pytest.mark.parametrize("split", [1, 2, 5, 20])
@pytest.mark.parametrize("dt", [Q.QMM_PARTIAL_BF16, Q.QMM_PARTIAL_F32])
def test_partition_planes(family, M, Nout, split, dt):
    """Each plane is the partition's sum rounded once (BF16 or FP32) -- the
    oracle's partition emulation of that plane.  The kernel accumulates in
    FP32 in its own order, so a BF16 plane may sit one BF16 ulp away (the
    FP32 sum and the exact one on either side of a rounding boundary); both
    kinds also get 2^-10 * max(1, |plane|) for the FP32 accumulation.  A
    dropped, doubled or misplaced 128-group moves a plane by far more."""
    p = inputs.make_w4a16(M, 2560, Nout, seed=50 + split + M)
    d = Q.to_device(p)
    got = _partition(d, M, Nout, split, dt).float().cpu().numpy().astype(np.float64)
    mode = 1 if dt == Q.QMM_PARTIAL_F32 else 0
    _, want = oracle.qmm_partitioned(p["A"], p["Wq"], p["scales"], p["biases"], split, mode,
                                     with_partials=True)
    assert np.all(np.isfinite(got)), "a plane element was not written"
    lim = 2.0 ** -10 * np.maximum(1.0, np.abs(want))
    if dt == Q.QMM_PARTIAL_BF16:
        lim = lim + _ulp_bf16(want)
    err = np.abs(got - want)
    bad = np.argwhere(err > lim)
    assert bad.size == 0, "%d plane elements out of tolerance, first %s err %g lim %g" % (
        len(bad), bad[0], err[tuple(bad[0])], lim[tuple(bad[0])])


@pytest.mark.parametrize("name,M", [("k", 16), ("down", 128), ("ragged", 33)])
@pytest.mark.parametrize("dt", [Q.QMM_PARTIAL_BF16, Q.QMM_PARTIAL_F32])
def test_partition_then_reduce_is_the_call(family, name, M, dt):
    """qmm_w4a16_g128 at a split s > 1 is the partition kernel followed by the
    reduce on the same planes: bitwise the same C."""
    Kred, Nout = inputs.PROJECTIONS[name] if name != "ragged" else inputs.RAGGED
    p = inputs.make_w4a16(M, Kred, Nout, seed=60 + M)
    d = Q.to_device(p)
    pol = Q.qmm_policy_preset(Q.QMM_PRESET_GB300, M)
    split = Q.qmm_splitk_plan(M, Kred, Nout, pol)
    assert split > 1
    whole, used = _run(d, M, Nout, 0, partial_dtype=dt)
    assert used == split
    planes = _partition(d, M, Nout, split, dt)
    C = torch.empty((M, Nout), dtype=torch.bfloat16, device="cuda")
    Q.qmm_splitk_reduce(planes, dt, split, M, Nout, C)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(C), whole)


def test_partition_argument_errors():
    d = Q.to_device(inputs.make_w4a16(8, 256, 64, seed=1))
    small = torch.empty((2, 8, 63), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(Q.QmmError) as e:
        Q.qmm_w4a16_g128_partition(d["A"], d["Wq"], d["scales"], d["biases"], small, 2)
    assert e.value.code == Q.QMM_EWORKSPACE
    ok = torch.empty((3, 8, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(Q.QmmError) as e:  # 3 does not divide G = 2
        Q.qmm_w4a16_g128_partition(d["A"], d["Wq"], d["scales"], d["biases"], ok, 3)
    assert e.value.code == Q.QMM_ESHAPE
    prev = Q.qmm_set_partitions(Q.QMM_PARTITIONS_NEAR_EQUAL)
    try:
        with pytest.raises(Q.QmmError) as e:  # near-equal: 3 > G = 2 is still refused
            Q.qmm_w4a16_g128_partition(d["A"], d["Wq"], d["scales"], d["biases"], ok, 3)
        assert e.value.code == Q.QMM_ESHAPE
        d3 = Q.to_device(inputs.make_w4a16(8, 640, 64, seed=1))  # G = 5: split 3 is fine
        Q.qmm_w4a16_g128_partition(d3["A"], d3["Wq"], d3["scales"], d3["biases"], ok, 3)
        torch.cuda.synchronize()
    finally:
        Q.qmm_set_partitions(prev)


# ---- static weights: the early start overlaps the previous kernel -----------

@pytest.mark.parametrize("pdl", [True, False])
def test_weights_static_back_to_back(pdl):
    """Calls launched back to back on one stream, with the static-weights
    promise, so each partition kernel loads and dequantizes weights while
    the kernel before it is still running.  Each result must match the
    oracle exactly as without the promise."""
    shapes = [("k", 16), ("gate", 32), ("down", 128), ("k", 16), ("ragged", 33)]
    probs = []
    for j, (name, M) in enumerate(shapes):
        Kred, Nout = inputs.RAGGED if name == "ragged" else inputs.PROJECTIONS[name]
        p = inputs.make_w4a16(M, Kred, Nout, seed=70 + j)
        probs.append((p, Q.to_device(p), M, Nout))
    prev_w, prev_p = Q.qmm_set_weights_static(True), Q.qmm_set_pdl(pdl)
    try:
        outs = []
        for p, d, M, Nout in probs:
            C, used = Q.w4a16_matmul(d["A"], d["Wq"], d["scales"], d["biases"])
            outs.append((C, used))
        torch.cuda.synchronize()
        assert Q.qmm_kernel_status(clear=True) == 0
    finally:
        Q.qmm_set_weights_static(prev_w)
        Q.qmm_set_pdl(prev_p)
    rng = np.random.default_rng(5)
    for (p, d, M, Nout), (C, used) in zip(probs, outs):
        rows, cols = _sample(M, Nout, rng)
        _check_sampled(p, _bits(C), used, Q.QMM_PARTIAL_BF16, rows, cols,
                       "static weights M=%d Nout=%d" % (M, Nout))


# ---- dense BF16 split-K GEMM -----------------------------------------------

@pytest.fixture(scope="module")
def dense512():
    d = inputs.make_dense(512, 512, 16384, seed=0)
    return d, oracle.gemm(d["A"], d["W"])


def _dense_dev(d):
    f = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return f(d["A"]), f(d["W"])


@pytest.mark.parametrize("split", [1, 2, 4, 6, 8, 9, 12, 16])
def test_dense_gemm_splits(family, dense512, split):
    d, C64 = dense512
    A, W = _dense_dev(d)
    C = torch.empty((512, 512), dtype=torch.bfloat16, device="cuda")
    nb = Q.qmm_gemm_workspace_bytes(512, 512, split)
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda") if nb else None
    Q.qmm_gemm_bf16_splitk(A, W, C, split, ws)
    torch.cuda.synchronize()
    _assert_close(_bits(C), C64, TOL_F32, "s=%d" % split)


@pytest.mark.parametrize("split", [1, 3, 10])
def test_dense_gemm_ragged(family, split):
    d = inputs.make_dense(200, 130, 640, seed=5)
    C64 = oracle.gemm(d["A"], d["W"])
    A, W = _dense_dev(d)
    C = torch.empty((200, 130), dtype=torch.bfloat16, device="cuda")
    nb = Q.qmm_gemm_workspace_bytes(200, 130, split)
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda") if nb else None
    Q.qmm_gemm_bf16_splitk(A, W, C, split, ws)
    torch.cuda.synchronize()
    _assert_close(_bits(C), C64, TOL_F32, "s=%d" % split)


# ---- error codes with real device buffers ----------------------------------

@pytest.mark.parametrize("name,M", [("down", 2048), ("o", 2048), ("k", 32), ("down", 128)])
def test_planned_split_request(name, M):
    """split_req = QMM_SPLIT_PLANNED dispatches the group plan's split for the
    call alone, with the bits of that split forced."""
    Kred, Nout = inputs.PROJECTIONS[name]
    p = inputs.make_w4a16(M, Kred, Nout, seed=7)
    d = Q.to_device(p)
    want = Q.qmm_group_plan([(M, Kred, Nout)])[0]
    C, used = Q.w4a16_matmul(d["A"], d["Wq"], d["scales"], d["biases"],
                             split_req=Q.QMM_SPLIT_PLANNED)
    C2, used2 = Q.w4a16_matmul(d["A"], d["Wq"], d["scales"], d["biases"], split_req=want)
    torch.cuda.synchronize()
    assert Q.qmm_kernel_status(clear=True) == 0
    assert used == used2 == want
    assert np.array_equal(_bits(C), _bits(C2))
    if M <= 128:  # under-filled calls: the chapter policy's split
        pol = Q.qmm_policy_preset(Q.QMM_PRESET_GB300, M)
        assert want == Q.qmm_splitk_plan(M, Kred, Nout, pol)
    rows, cols = _sample(M, Nout, np.random.default_rng(4))
    _check_sampled(p, _bits(C), used, Q.QMM_PARTIAL_BF16, rows, cols, "planned split")


def test_bounded_wait_runs_out_and_reports():
    """A wait that nothing completes gives up after its limit: the status word
    reports it, nothing traps, and the context stays usable (a matmul right
    after is correct)."""
    assert Q.qmm_kernel_status(clear=True) == 0
    t0 = time.monotonic()
    Q.qmm_wait_timeout_probe()
    torch.cuda.synchronize()
    took = time.monotonic() - t0
    assert Q.qmm_kernel_status(clear=True) == 1
    assert 0.5 < took < 30.0, took
    assert Q.qmm_kernel_status(clear=True) == 0  # cleared
    M, (Kred, Nout) = 16, inputs.PROJECTIONS["k"]
    p = inputs.make_w4a16(M, Kred, Nout, seed=5)
    d = Q.to_device(p)
    C, split = Q.w4a16_matmul(d["A"], d["Wq"], d["scales"], d["biases"])
    torch.cuda.synchronize()
    assert Q.qmm_kernel_status(clear=True) == 0
    rows, cols = _sample(M, Nout, np.random.default_rng(3))
    _check_sampled(p, _bits(C), split, Q.QMM_PARTIAL_BF16, rows, cols, "after a timed-out wait")


def test_error_codes_on_device():
    Kred, Nout, M = 2560, 1024, 16
    p = inputs.make_w4a16(M, Kred, Nout, seed=9)
    d = Q.to_device(p)
    C = torch.empty((M, Nout), dtype=torch.bfloat16, device="cuda")
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(Q.QmmError) as e:
        Q.qmm_w4a16_g128(d["A"], d["Wq"], d["scales"], d["biases"], C, split_req=4, workspace=small)
    assert e.value.code == Q.QMM_EWORKSPACE
    with pytest.raises(Q.QmmError) as e:
        Q.qmm_w4a16_g128(d["A"], d["Wq"], d["scales"], d["biases"], C, split_req=3)
    assert e.value.code == Q.QMM_ESHAPE
    lib = Q.lib()
    rc = lib.qmm_w4a16_g128(ctypes.c_void_p(d["A"].data_ptr() + 2), ctypes.c_void_p(d["Wq"].data_ptr()),
                            ctypes.c_void_p(d["scales"].data_ptr()), ctypes.c_void_p(d["biases"].data_ptr()),
                            ctypes.c_void_p(C.data_ptr()), M, Kred, Nout, 1, None, None, 0, 0, None, None)
    assert rc == Q.QMM_EALIGN


# ---- fused last-CTA reduce: the same C as the separate reduce ---------------

def _call_with(d, M, Nout, split, dt, ws):
    C = torch.full((M, Nout), float("nan"), dtype=torch.bfloat16, device="cuda")
    used = Q.qmm_w4a16_g128(d["A"], d["Wq"], d["scales"], d["biases"], C, split_req=split,
                            workspace=ws, partial_dtype=dt)
    torch.cuda.synchronize()
    assert used == split
    return _bits(C)


@pytest.mark.parametrize("name,M,split", [("k", 16, 10), ("gate", 32, 2), ("down", 128, 4),
                                          ("ragged", 33, 10), ("odd", 5, 2), ("k", 300, 4),
                                          ("down", 8, 4), ("ragged", 16, 5), ("o", 1, 8)])
@pytest.mark.parametrize("dt", [Q.QMM_PARTIAL_BF16, Q.QMM_PARTIAL_F32])
@pytest.mark.parametrize("kernels", ["tc", "lean"])
def test_fused_reduce_bitwise_equals_kernel_reduce(name, M, split, dt, kernels):
    """QMM_REDUCE_FUSED adds the planes in the partition kernel's last CTA of
    each tile: same planes, same FP32 ascending sum, so the same bits as the
    separate reduce, and within the chapter's tolerance of the oracle.  Three
    calls on one workspace also check that every call leaves the tile
    counters at zero."""
    if name == "odd":
        Kred, Nout = 256, 77          # scalar path of the fused reduce
    else:
        Kred, Nout = inputs.RAGGED if name == "ragged" else inputs.PROJECTIONS[name]
    p = inputs.make_w4a16(M, Kred, Nout, seed=90 + M)
    d = Q.to_device(p)
    prev_k = Q.qmm_set_kernels(KERNELS[kernels])
    try:
        prev = Q.qmm_set_reduce(Q.QMM_REDUCE_KERNEL)
        nb = Q.qmm_splitk_workspace_bytes(M, Nout, split, dt)
        ref = _call_with(d, M, Nout, split, dt, torch.empty(max(nb, 16), dtype=torch.uint8,
                                                            device="cuda"))
        Q.qmm_set_reduce(Q.QMM_REDUCE_FUSED)
        nbf = Q.qmm_splitk_workspace_bytes(M, Nout, split, dt)
        assert nbf > nb  # the counters follow the planes
        ws = torch.zeros(nbf, dtype=torch.uint8, device="cuda")
        for _ in range(3):
            got = _call_with(d, M, Nout, split, dt, ws)
            assert np.array_equal(got, ref)
        assert Q.qmm_kernel_status(clear=True) == 0
        C64 = oracle.qmm(p["A"], p["Wq"], p["scales"], p["biases"])
        _check_full(p, got, split, dt, C64, "fused %s M=%d s=%d" % (name, M, split))
    finally:
        Q.qmm_set_reduce(prev)
        Q.qmm_set_kernels(prev_k)


def test_fused_reduce_with_the_static_scratch():
    d = Q.to_device(inputs.make_w4a16(32, 2560, 1024, seed=99))
    prev = Q.qmm_set_reduce(Q.QMM_REDUCE_KERNEL)
    try:
        C1 = torch.empty((32, 1024), dtype=torch.bfloat16, device="cuda")
        C2 = torch.empty_like(C1)
        Q.qmm_w4a16_g128_noalloc(d["A"], d["Wq"], d["scales"], d["biases"], C1, split_req=10)
        Q.qmm_set_reduce(Q.QMM_REDUCE_FUSED)
        for _ in range(2):
            Q.qmm_w4a16_g128_noalloc(d["A"], d["Wq"], d["scales"], d["biases"], C2, split_req=10)
            torch.cuda.synchronize()
            assert np.array_equal(_bits(C1), _bits(C2))
    finally:
        Q.qmm_set_reduce(prev)


# ---- near-equal partitions (QMM_PARTITIONS_NEAR_EQUAL) ----------------------

NE_PLAN = Q.qmm_splitk_plan_near_equal


@pytest.fixture
def near_equal():
    prev = Q.qmm_set_partitions(Q.QMM_PARTITIONS_NEAR_EQUAL)
    try:
        yield
    finally:
        Q.qmm_set_partitions(prev)


@pytest.mark.parametrize("M", [16, 128])
@pytest.mark.parametrize("name,splits", [("k", [3, 6, 7, 9, 13, 16, 19]), ("o", [3, 5, 7, 9, 31]),
                                         ("down", [3, 5, 7, 9, 13, 75])])
def test_near_equal_forced_splits(family, near_equal, name, splits, M):
    """Splits that do not divide the group count: the first G mod s partitions
    hold one group more.  Against the oracle's emulation of that cut."""
    Kred, Nout = inputs.PROJECTIONS[name]
    p = inputs.make_w4a16(M, Kred, Nout, seed=110 + M)
    d = Q.to_device(p)
    C64 = oracle.qmm(p["A"], p["Wq"], p["scales"], p["biases"])
    for s in splits:
        for dt in (Q.QMM_PARTIAL_BF16, Q.QMM_PARTIAL_F32):
            got, used = _run(d, M, Nout, s, partial_dtype=dt, plan=NE_PLAN)
            _check_full(p, got, s, dt, C64, "%s M=%d s=%d dt=%d" % (name, M, s, dt))


@pytest.mark.parametrize("M", [1, 9, 17, 33, 65, 129, 300])
def test_near_equal_families_ragged(family, near_equal, M):
    # G = 10 and Nout = 1000: every short last stage (one to three groups on
    # the narrow tiles) and a partial last column tile
    Kred, Nout = 1280, 1000
    p = inputs.make_w4a16(M, Kred, Nout, seed=120 + M)
    d = Q.to_device(p)
    C64 = oracle.qmm(p["A"], p["Wq"], p["scales"], p["biases"])
    for split_req in (0, 3, 4, 6, 7, 9):
        got, s = _run(d, M, Nout, split_req, plan=NE_PLAN)
        _check_full(p, got, s, Q.QMM_PARTIAL_BF16, C64, "M=%d req=%d" % (M, split_req))


@pytest.mark.parametrize("M", [16, 32, 64, 128])
@pytest.mark.parametrize("name", list(inputs.PROJECTIONS) + ["ragged"])
def test_near_equal_policy_full_size_sampled(near_equal, name, M):
    Kred, Nout = inputs.RAGGED if name == "ragged" else inputs.PROJECTIONS[name]
    p = inputs.make_w4a16(M, Kred, Nout, seed=0)
    d = Q.to_device(p)
    pol = Q.qmm_policy_preset(Q.QMM_PRESET_GB300, M)
    got, s = _run(d, M, Nout, 0, plan=NE_PLAN)
    assert s == NE_PLAN(M, Kred, Nout, pol) >= Q.qmm_splitk_plan(M, Kred, Nout, pol)
    rows, cols = _sample(M, Nout, np.random.default_rng(M * 11 + Nout))
    _check_sampled(p, got, s, Q.QMM_PARTIAL_BF16, rows, cols, "near-equal policy s=%d" % s)


@pytest.mark.parametrize("name,M,splits", [("k", 32, [2, 5, 10]), ("down", 128, [2, 4]),
                                           ("ragged", 33, [4, 10])])
def test_near_equal_dividing_split_is_the_equal_cut(family, name, M, splits):
    """With a split that divides G both rules cut the same partitions: the
    same bits from either mode."""
    Kred, Nout = inputs.RAGGED if name == "ragged" else inputs.PROJECTIONS[name]
    d = Q.to_device(inputs.make_w4a16(M, Kred, Nout, seed=130 + M))
    for s in splits:
        a, _ = _run(d, M, Nout, s)
        prev = Q.qmm_set_partitions(Q.QMM_PARTITIONS_NEAR_EQUAL)
        try:
            b, _ = _run(d, M, Nout, s, plan=NE_PLAN)
        finally:
            Q.qmm_set_partitions(prev)
        assert np.array_equal(a, b), "s=%d" % s


@pytest.mark.parametrize("M,Nout", [(40, 1000), (3, 136)])
@pytest.mark.parametrize("split", [3, 7, 13])
@pytest.mark.parametrize("dt", [Q.QMM_PARTIAL_BF16, Q.QMM_PARTIAL_F32])
def test_near_equal_partition_planes(family, near_equal, M, Nout, split, dt):
    """Each plane against the oracle's plane of the near-equal cut (the
    tolerance of test_partition_planes)."""
    p = inputs.make_w4a16(M, 2560, Nout, seed=140 + split + M)
    d = Q.to_device(p)
    got = _partition(d, M, Nout, split, dt).float().cpu().numpy().astype(np.float64)
    mode = 1 if dt == Q.QMM_PARTIAL_F32 else 0
    _, want = oracle.qmm_partitioned(p["A"], p["Wq"], p["scales"], p["biases"], split, mode,
                                     with_partials=True)
    assert np.all(np.isfinite(got)), "a plane element was not written"
    lim = 2.0 ** -10 * np.maximum(1.0, np.abs(want))
    if dt == Q.QMM_PARTIAL_BF16:
        lim = lim + _ulp_bf16(want)
    err = np.abs(got - want)
    bad = np.argwhere(err > lim)
    assert bad.size == 0, "%d plane elements out of tolerance, first %s err %g lim %g" % (
        len(bad), bad[0], err[tuple(bad[0])], lim[tuple(bad[0])])


@pytest.mark.parametrize("name,M,split", [("k", 32, 16), ("down", 128, 7), ("ragged", 33, 7)])
def test_near_equal_fused_reduce_and_static_scratch(near_equal, name, M, split):
    """The fused last-CTA reduce and the allocation-free entry point under
    the near-equal rule: the same bits as the separate reduce with a caller
    workspace."""
    Kred, Nout = inputs.RAGGED if name == "ragged" else inputs.PROJECTIONS[name]
    dt = Q.QMM_PARTIAL_BF16
    d = Q.to_device(inputs.make_w4a16(M, Kred, Nout, seed=150 + M))
    prev_k = Q.qmm_set_kernels(Q.QMM_KERNELS_TCGEN05)
    prev = Q.qmm_set_reduce(Q.QMM_REDUCE_KERNEL)
    try:
        nb = Q.qmm_splitk_workspace_bytes(M, Nout, split, dt)
        ref = _call_with(d, M, Nout, split, dt, torch.empty(nb, dtype=torch.uint8, device="cuda"))
        C = torch.empty((M, Nout), dtype=torch.bfloat16, device="cuda")
        used = Q.qmm_w4a16_g128_noalloc(d["A"], d["Wq"], d["scales"], d["biases"], C,
                                        split_req=split)
        torch.cuda.synchronize()
        assert used == split and np.array_equal(_bits(C), ref)
        Q.qmm_set_reduce(Q.QMM_REDUCE_FUSED)
        ws = torch.zeros(Q.qmm_splitk_workspace_bytes(M, Nout, split, dt), dtype=torch.uint8,
                         device="cuda")
        for _ in range(2):
            assert np.array_equal(_call_with(d, M, Nout, split, dt, ws), ref)
        assert Q.qmm_kernel_status(clear=True) == 0
    finally:
        Q.qmm_set_reduce(prev)
        Q.qmm_set_kernels(prev_k)


def test_near_equal_weights_static_back_to_back(near_equal):
    """Back-to-back policy calls with the static-weights early start under
    the near-equal rule (o and down split 7 ways)."""
    shapes = [("k", 32), ("down", 128), ("o", 32), ("k", 128), ("ragged", 33)]
    probs = []
    for j, (name, M) in enumerate(shapes):
        Kred, Nout = inputs.RAGGED if name == "ragged" else inputs.PROJECTIONS[name]
        p = inputs.make_w4a16(M, Kred, Nout, seed=160 + j)
        probs.append((p, Q.to_device(p), M, Nout))
    prev_w = Q.qmm_set_weights_static(True)
    try:
        outs = [Q.w4a16_matmul(d["A"], d["Wq"], d["scales"], d["biases"])
                for p, d, M, Nout in probs]
        torch.cuda.synchronize()
        assert Q.qmm_kernel_status(clear=True) == 0
    finally:
        Q.qmm_set_weights_static(prev_w)
    rng = np.random.default_rng(6)
    for (p, d, M, Nout), (C, used) in zip(probs, outs):
        pol = Q.qmm_policy_preset(Q.QMM_PRESET_GB300, M)
        assert used == NE_PLAN(M, p["A"].shape[1], Nout, pol)
        rows, cols = _sample(M, Nout, rng)
        _check_sampled(p, _bits(C), used, Q.QMM_PARTIAL_BF16, rows, cols,
                       "near-equal static weights M=%d Nout=%d" % (M, Nout))


# ---- streaming host activations (qmm_w4a16_g128_stream) ---------------------

STREAM_SHAPES = [("k", 16), ("down", 128), ("ragged", 33), ("gate", 32), ("k", 300), ("o", 64)]


def _stream_chunks(seed0):
    chunks, probs = [], []
    for j, (name, M) in enumerate(STREAM_SHAPES):
        Kred, Nout = inputs.RAGGED if name == "ragged" else inputs.PROJECTIONS[name]
        p = inputs.make_w4a16(M, Kred, Nout, seed=seed0 + j)
        d = Q.to_device(p)
        A_host = torch.from_numpy(p["A"].view(np.int16)).view(torch.bfloat16).pin_memory()
        C_host = torch.full((M, Nout), float("nan"), dtype=torch.bfloat16).pin_memory()
        chunks.append({"A": A_host, "C": C_host, "Wq": d["Wq"], "scales": d["scales"],
                       "biases": d["biases"]})
        probs.append((p, d, M, Nout))
    return chunks, probs


@pytest.mark.parametrize("buffers", [1, 2, 3, 8])
@pytest.mark.parametrize("streams", ["three", "one"])
def test_stream_executor_equals_the_calls(buffers, streams):
    """Each chunk's host output is bitwise the output of qmm_w4a16_g128 on the
    same inputs, for any buffer count, on three streams or on one; a second
    run on the same arena (and the library's reused events) gives the same."""
    chunks, probs = _stream_chunks(170)
    calls = Q.stream_calls(chunks)
    nbytes = Q.qmm_stream_arena_bytes(calls, buffers)
    assert nbytes > 0
    arena = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    if streams == "three":
        s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    else:
        s_in = s_comp = s_out = torch.cuda.current_stream()
    refs = []
    for p, d, M, Nout in probs:
        C, used = Q.w4a16_matmul(d["A"], d["Wq"], d["scales"], d["biases"])
        refs.append((_bits(C), used))
    for rep in range(2):
        for c in chunks:
            c["C"].fill_(float("nan"))
        used = Q.qmm_w4a16_g128_stream(calls, buffers, arena, s_in, s_comp, s_out)
        s_out.synchronize()
        torch.cuda.synchronize()
        for j, (c, (ref, ref_used)) in enumerate(zip(chunks, refs)):
            assert used[j] == ref_used
            assert np.array_equal(c["C"].view(torch.int16).numpy().view(np.uint16), ref), \
                "chunk %d rep %d" % (j, rep)
    # and one chunk against the oracle directly
    p, d, M, Nout = probs[1]
    rows, cols = _sample(M, Nout, np.random.default_rng(7))
    got = chunks[1]["C"].view(torch.int16).numpy().view(np.uint16)
    _check_sampled(p, got, used[1], Q.QMM_PARTIAL_BF16, rows, cols, "streamed down M=128")
    assert Q.qmm_kernel_status(clear=True) == 0


def test_stream_executor_under_near_equal_and_fused_reduce():
    """Near-equal partitions and the fused reduce inside the pipeline: the same
    bits as the separate reduce's calls (the arena zeroed once, as a fused
    workspace must be)."""
    chunks, probs = _stream_chunks(180)
    prev_p = Q.qmm_set_partitions(Q.QMM_PARTITIONS_NEAR_EQUAL)
    prev_k = Q.qmm_set_kernels(Q.QMM_KERNELS_TCGEN05)
    prev_r = Q.qmm_set_reduce(Q.QMM_REDUCE_KERNEL)
    try:
        refs = []
        for p, d, M, Nout in probs:
            C, used = Q.w4a16_matmul(d["A"], d["Wq"], d["scales"], d["biases"])
            refs.append((_bits(C), used))
        Q.qmm_set_reduce(Q.QMM_REDUCE_FUSED)
        calls = Q.stream_calls(chunks)
        arena = torch.zeros(Q.qmm_stream_arena_bytes(calls, 2), dtype=torch.uint8, device="cuda")
        used = Q.qmm_w4a16_g128_stream(calls, 2, arena, torch.cuda.Stream(), torch.cuda.Stream(),
                                       torch.cuda.Stream())
        torch.cuda.synchronize()
        for j, (c, (ref, ref_used)) in enumerate(zip(chunks, refs)):
            assert used[j] == ref_used
            assert np.array_equal(c["C"].view(torch.int16).numpy().view(np.uint16), ref), j
        assert Q.qmm_kernel_status(clear=True) == 0
    finally:
        Q.qmm_set_kernels(prev_k)
        Q.qmm_set_reduce(prev_r)
        Q.qmm_set_partitions(prev_p)


def test_stream_executor_refuses_a_small_arena():
    chunks, _ = _stream_chunks(190)
    calls = Q.stream_calls(chunks[:2])
    nbytes = Q.qmm_stream_arena_bytes(calls, 2)
    # one more buffer adds one slot: the largest A and C, each rounded to 256 bytes
    r256 = lambda x: -(-x // 256) * 256
    slot = r256(max(c["A"].numel() * 2 for c in chunks[:2])) + \
        r256(max(c["C"].numel() * 2 for c in chunks[:2]))
    assert nbytes - Q.qmm_stream_arena_bytes(calls, 1) == slot
    small = torch.empty(nbytes - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(Q.QmmError) as e:
        Q.qmm_w4a16_g128_stream(calls, 2, small)
    assert e.value.code == Q.QMM_EWORKSPACE


# ---- several independent calls in few launches (qmm_w4a16_g128_grouped) -----

def _group_problems(shapes, seed0):
    probs = []
    for j, (name, M) in enumerate(shapes):
        if name == "odd":
            Kred, Nout = 256, 77
        else:
            Kred, Nout = inputs.RAGGED if name == "ragged" else inputs.PROJECTIONS[name]
        p = inputs.make_w4a16(M, Kred, Nout, seed=seed0 + j)
        d = Q.to_device(p)
        d["C"] = torch.full((M, Nout), float("nan"), dtype=torch.bfloat16, device="cuda")
        probs.append((p, d))
    return probs


def _grouped_vs_calls(probs, dt=Q.QMM_PARTIAL_BF16):
    refs = []
    for p, d in probs:
        M, Nout = d["C"].shape
        C = torch.empty((M, Nout), dtype=torch.bfloat16, device="cuda")
        nb = Q.qmm_splitk_workspace_bytes(M, Nout, 16, dt)  # room for any split
        ws = torch.zeros(max(nb, 16) + (64 << 10), dtype=torch.uint8, device="cuda")
        used = Q.qmm_w4a16_g128(d["A"], d["Wq"], d["scales"], d["biases"], C, workspace=ws,
                                partial_dtype=dt)
        refs.append((_bits(C), used))
    calls = Q.group_calls([d for _, d in probs])
    nb = Q.qmm_group_workspace_bytes(calls, dt)
    ws = torch.full((max(nb, 16) // 2 + 8,), float("nan"), dtype=torch.bfloat16, device="cuda")
    used = Q.qmm_w4a16_g128_grouped(calls, ws if nb else None, dt)
    torch.cuda.synchronize()
    assert Q.qmm_kernel_status(clear=True) == 0
    for j, ((p, d), (ref, ref_used)) in enumerate(zip(probs, refs)):
        assert used[j] == ref_used, j
        assert np.array_equal(_bits(d["C"]), ref), "call %d" % j
    return used


GROUP_SHAPES = [(n, M) for M in (32, 128) for n in inputs.PROJECTIONS] + \
    [("ragged", 33), ("odd", 5), ("k", 16), ("down", 300), ("q", 8), ("ragged", 1)]


@pytest.fixture(params=["tiles", "persistent"])
def grouped_schedule(request):
    """Both schedules of the grouped call's partition launches: one CTA per
    tile, or one CTA per SM walking the tiles (qmm_set_grouped_schedule)."""
    prev = Q.qmm_set_grouped_schedule(Q.QMM_GROUPED_PERSISTENT if request.param == "persistent"
                                      else Q.QMM_GROUPED_TILES)
    yield request.param
    Q.qmm_set_grouped_schedule(prev)


@pytest.mark.parametrize("rule", ["equal", "near-equal"])
@pytest.mark.parametrize("dt", [Q.QMM_PARTIAL_BF16, Q.QMM_PARTIAL_F32])
def test_grouped_equals_the_calls(family, grouped_schedule, rule, dt):
    """Each C of the grouped call is bitwise its own call's C: the same CTA
    body, ring depth aside, and the same ordered FP32 reduce."""
    prev = Q.qmm_set_partitions(Q.QMM_PARTITIONS_NEAR_EQUAL if rule == "near-equal"
                                else Q.QMM_PARTITIONS_EQUAL)
    try:
        probs = _group_problems(GROUP_SHAPES, 200)
        used = _grouped_vs_calls(probs, dt)
        assert max(used) > 1 and min(used) == 1
    finally:
        Q.qmm_set_partitions(prev)
    # and one call against the oracle directly
    p, d = probs[13]  # down M=128
    M, Nout = d["C"].shape
    rows, cols = _sample(M, Nout, np.random.default_rng(8))
    _check_sampled(p, _bits(d["C"]), used[13], dt, rows, cols, "grouped down M=128")


def test_grouped_more_calls_than_one_launch_holds(grouped_schedule):
    # 20 calls of one tile width: two partition launches and two reduce launches
    shapes = [("k", 32), ("v", 32), ("q", 32), ("odd", 20), ("ragged", 31)] * 4
    probs = _group_problems(shapes, 230)
    _grouped_vs_calls(probs)


@pytest.mark.parametrize("pdl", [True, False])
def test_grouped_with_static_weights(grouped_schedule, pdl):
    prev_w, prev_p = Q.qmm_set_weights_static(True), Q.qmm_set_pdl(pdl)
    try:
        probs = _group_problems(GROUP_SHAPES, 260)
        _grouped_vs_calls(probs)
        # twice back to back on one stream: the second group's early weight
        # work overlaps the first group's last kernel
        calls = Q.group_calls([d for _, d in probs])
        ws = torch.zeros(Q.qmm_group_workspace_bytes(calls), dtype=torch.uint8, device="cuda")
        first = [_bits(d["C"]) for _, d in probs]
        for _ in range(3):
            Q.qmm_w4a16_g128_grouped(calls, ws)
        torch.cuda.synchronize()
        assert all(np.array_equal(_bits(d["C"]), f) for (_, d), f in zip(probs, first))
    finally:
        Q.qmm_set_weights_static(prev_w)
        Q.qmm_set_pdl(prev_p)


@pytest.mark.parametrize("dt", [Q.QMM_PARTIAL_BF16, Q.QMM_PARTIAL_F32])
def test_group_plan_equals_the_calls_at_the_planned_splits(grouped_schedule, dt):
    """Under QMM_GROUP_PLAN_GROUP each C is bitwise qmm_w4a16_g128's C with
    split_req = the planned split, the splits reported are the plan, and the
    workspace holds exactly the planned planes."""
    probs = _group_problems(GROUP_SHAPES, 340)
    shapes = [(d["C"].shape[0], d["A"].shape[1], d["C"].shape[1]) for _, d in probs]
    prev = Q.qmm_set_group_plan(Q.QMM_GROUP_PLAN_GROUP)
    try:
        plan = Q.qmm_group_plan(shapes, 0, dt)
        assert max(plan) > 1 and min(plan) == 1
        refs = []
        for (p, d), sp in zip(probs, plan):
            M, Nout = d["C"].shape
            C = torch.empty((M, Nout), dtype=torch.bfloat16, device="cuda")
            nb = Q.qmm_splitk_workspace_bytes(M, Nout, sp, dt)
            ws = torch.zeros(max(nb, 16) + (64 << 10), dtype=torch.uint8, device="cuda")
            assert Q.qmm_w4a16_g128(d["A"], d["Wq"], d["scales"], d["biases"], C, split_req=sp,
                                    workspace=ws, partial_dtype=dt) == sp
            refs.append(_bits(C))
        calls = Q.group_calls([d for _, d in probs])
        nb = Q.qmm_group_workspace_bytes(calls, dt)
        elem = 4 if dt == Q.QMM_PARTIAL_F32 else 2
        assert nb == sum(-(-(sp * M * N * elem) // 256) * 256
                         for sp, (M, _, N) in zip(plan, shapes) if sp > 1)
        ws = torch.full((max(nb, 16) // 2 + 8,), float("nan"), dtype=torch.bfloat16, device="cuda")
        used = Q.qmm_w4a16_g128_grouped(calls, ws if nb else None, dt)
        torch.cuda.synchronize()
        assert Q.qmm_kernel_status(clear=True) == 0
        assert used == plan
        for j, ((p, d), ref) in enumerate(zip(probs, refs)):
            assert np.array_equal(_bits(d["C"]), ref), "call %d" % j
    finally:
        Q.qmm_set_group_plan(prev)
    # one planned call against the oracle directly (down at M = 128, split 2 or the plan's)
    p, d = probs[13]
    M, Nout = d["C"].shape
    rows, cols = _sample(M, Nout, np.random.default_rng(9))
    _check_sampled(p, _bits(d["C"]), used[13], dt, rows, cols, "group plan down M=128")


@pytest.mark.parametrize("shapes", [
    [("k", 32)],                                    # fewer tiles than SMs: one each
    [("odd", 3), ("odd", 40), ("ragged", 1), ("k", 8), ("odd", 129)] * 3,
    [("down", 128), ("odd", 7), ("gate", 32), ("ragged", 64)],
    [("q", 48), ("down", 40), ("odd", 64), ("k", 33), ("o", 60)],  # 64-row tiles
])
def test_persistent_grouped_tile_lists(shapes):
    """The persistent schedule on short and mixed tile lists: partitions of
    one or two groups (phantom positions in every stage), ragged rows and
    columns, more and fewer tiles than SMs; each C bitwise its own call's."""
    prev = Q.qmm_set_grouped_schedule(Q.QMM_GROUPED_PERSISTENT)
    try:
        probs = _group_problems(shapes, 310)
        _grouped_vs_calls(probs)
        _grouped_vs_calls(probs, Q.QMM_PARTIAL_F32)
    finally:
        Q.qmm_set_grouped_schedule(prev)


def test_grouped_argument_errors():
    probs = _group_problems([("k", 32), ("down", 128)], 290)
    calls = Q.group_calls([d for _, d in probs])
    nb = Q.qmm_group_workspace_bytes(calls)
    assert nb > 0
    with pytest.raises(Q.QmmError) as e:
        Q.qmm_w4a16_g128_grouped(calls, torch.empty(nb - 256, dtype=torch.uint8, device="cuda"))
    assert e.value.code == Q.QMM_EWORKSPACE
    with pytest.raises(Q.QmmError) as e:
        Q.qmm_w4a16_g128_grouped(calls, None)
    assert e.value.code == Q.QMM_EWORKSPACE
    # only unsplit calls need no workspace
    big = _group_problems([("gate", 2048)], 295)
    c1 = Q.group_calls([d for _, d in big])
    assert Q.qmm_group_workspace_bytes(c1) == 0
    assert Q.qmm_w4a16_g128_grouped(c1, None) == [1]


# ---- split-KV decode attention (qmm_decode_attention) ------------------------
#
# Tolerance, per element: |O_gpu - O64| <= 2^-8 |O64| + 1e-4.  The GPU forms
# scores, weights and sums in FP32 (relative error ~1e-6 here) and rounds O
# to BF16 once (2^-9 relative); 1e-4 covers the FP32 sums of up to ~10^4
# weighted rows for the small |O| of long, flat softmaxes.

def _attention(prob, splits_req=0, scale=0.0):
    d = Q.attention_to_device(prob)
    B, Hq, D = prob["q"].shape
    O = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    S = splits_req or Q.qmm_decode_attention_splits(B, Hq, prob["K"].shape[1], prob["K"].shape[2])
    nb = Q.qmm_decode_attention_workspace_bytes(B, Hq, D, S)
    ws = torch.full((max(nb, 16) // 4,), float("nan"), dtype=torch.float32, device="cuda")
    used = Q.qmm_decode_attention(d["q"], d["K"], d["V"], d["lens"], O, scale, splits_req,
                                  ws if nb else None)
    torch.cuda.synchronize()
    assert used == S
    assert Q.qmm_kernel_status(clear=True) == 0
    return _bits(O).reshape(B, Hq, D), used


def _assert_attention(got_bits, O64, what=""):
    got = _val(got_bits)
    assert np.all(np.isfinite(got)), "non-finite output " + what
    lim = 2.0 ** -8 * np.abs(O64) + 1e-4
    err = np.abs(got - O64)
    bad = np.argwhere(err > lim)
    assert bad.size == 0, "%s: %d elements out of tolerance, first %s err %g lim %g" % (
        what, len(bad), bad[0], err[tuple(bad[0])], lim[tuple(bad[0])])


@pytest.mark.parametrize("B,Hq,Hkv,Lmax,D", [(1, 1, 1, 1, 64), (2, 4, 2, 100, 128),
                                             (3, 32, 8, 777, 128), (4, 8, 1, 64, 64),
                                             (2, 16, 8, 2049, 128), (5, 8, 4, 300, 64)])
def test_attention_splits_against_oracle(B, Hq, Hkv, Lmax, D):
    """Split factors 1, 2, 4, 8, a non-power-of-two one and the plan's, on
    ragged lengths, against the fp64 definition."""
    prob = inputs.make_attention(B, Hq, Hkv, Lmax, D, seed=300 + Lmax)
    O64 = oracle.decode_attention(prob["q"], prob["K"], prob["V"], prob["lens"])
    for S in (0, 1, 2, 3, 4, 7, 8):
        got, used = _attention(prob, S)
        _assert_attention(got, O64, "S=%d (used %d)" % (S, used))


def test_attention_edge_lengths_and_scale():
    # single positions, full length, a length just past a tile, empty splits
    B, Hq, Hkv, Lmax, D = 6, 8, 2, 200, 128
    prob = inputs.make_attention(B, Hq, Hkv, Lmax, D, seed=310,
                                 lens=[1, 200, 65, 64, 63, 129])
    for scale in (0.0, 0.05):
        O64 = oracle.decode_attention(prob["q"], prob["K"], prob["V"], prob["lens"],
                                      scale=scale or None)
        for S in (1, 2, 5, 16):  # 16 splits of 200 positions: most are empty
            got, _ = _attention(prob, S, scale)
            _assert_attention(got, O64, "scale=%g S=%d" % (scale, S))


def test_attention_dominant_key_and_uniform_keys():
    # closed forms through the GPU path: a dominant key returns its V row,
    # equal keys return the mean of the valid V rows
    B, Hq, Hkv, Lmax, D = 2, 4, 4, 300, 128
    prob = inputs.make_attention(B, Hq, Hkv, Lmax, D, seed=320, lens=[300, 150])
    prob["K"][:] = prob["K"][:, :, :1, :]
    O64 = oracle.decode_attention(prob["q"], prob["K"], prob["V"], prob["lens"])
    Vf = _val(prob["V"])
    for b, L in enumerate(prob["lens"]):
        assert np.allclose(O64[b], Vf[b, :, :L].mean(axis=1), atol=1e-12)
    for S in (1, 3):
        got, _ = _attention(prob, S)
        _assert_attention(got, O64, "uniform S=%d" % S)


def test_attention_workload_full_size():
    """The bench workload: Qwen3-4B heads (32 query, 8 KV, dim 128), 32
    sequences with lengths mixed in [1024, 8192], the plan's split."""
    h = inputs.ATTENTION_HEADS
    prob = inputs.make_attention(32, h["Hq"], h["Hkv"], 8192, h["D"], seed=0, lmin=1024)
    O64 = oracle.decode_attention(prob["q"], prob["K"], prob["V"], prob["lens"])
    got, used = _attention(prob, 0)
    assert used == Q.qmm_decode_attention_splits(32, 32, 8, 8192)
    _assert_attention(got, O64, "workload S=%d" % used)
    again, _ = _attention(prob, 0)
    assert np.array_equal(got, again), "not deterministic"


def test_attention_errors_on_device():
    prob = inputs.make_attention(2, 8, 2, 100, 128, seed=330)
    d = Q.attention_to_device(prob)
    O = torch.empty((2, 8, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(Q.QmmError) as e:
        Q.qmm_decode_attention(d["q"], d["K"], d["V"], d["lens"], O, splits_req=4)
    assert e.value.code == Q.QMM_EWORKSPACE
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(Q.QmmError) as e:
        Q.qmm_decode_attention(d["q"], d["K"], d["V"], d["lens"], O, splits_req=4,
                               workspace=small)
    assert e.value.code == Q.QMM_EWORKSPACE


# ---- per-call options ---------------------------------------------------------

def test_options_two_threads_on_the_gpu():
    """Two threads call qmm_w4a16_g128_ex on the same inputs under different
    partition rules (down at M = 128: split 4 equal, 7 near-equal) while the
    process-wide rule flips: each thread's result is bitwise the one its own
    rule gives alone, and within tolerance of the oracle at that split."""
    import threading
    M, (Kred, Nout) = 128, inputs.PROJECTIONS["down"]
    p = inputs.make_w4a16(M, Kred, Nout, seed=71)
    d = Q.to_device(p)
    rules = (Q.QMM_PARTITIONS_EQUAL, Q.QMM_PARTITIONS_NEAR_EQUAL)
    opts = {r: Q.qmm_options(partitions=r) for r in rules}
    wsb = max(Q.qmm_splitk_workspace_bytes(M, Nout, 16, options=o) for o in opts.values())

    def call(rule, stream):
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        C = torch.empty((M, Nout), dtype=torch.bfloat16, device="cuda")
        with torch.cuda.stream(stream):
            s = Q.qmm_w4a16_g128(d["A"], d["Wq"], d["scales"], d["biases"], C, workspace=ws,
                                 stream=stream, options=opts[rule])
        stream.synchronize()
        return _bits(C), s

    base = {r: call(r, torch.cuda.Stream()) for r in rules}
    assert base[rules[0]][1] == 4 and base[rules[1]][1] == 7
    for r in rules:
        got, s = base[r]
        _check_sampled(p, got, s, Q.QMM_PARTIAL_BF16, np.arange(0, M, 9),
                       np.arange(0, Nout, 37), "options rule %d" % r)
    errors = []
    stop = threading.Event()

    def worker(rule):
        try:
            st = torch.cuda.Stream()
            for _ in range(20):
                got, s = call(rule, st)
                if s != base[rule][1] or not np.array_equal(got, base[rule][0]):
                    errors.append("rule %d: split %d, bits differ" % (rule, s))
                    return
        except Exception as e:  # reported by the assertion below
            errors.append("rule %d: %r" % (rule, e))

    def flipper():
        i = 0
        while not stop.is_set():
            Q.qmm_set_partitions(i & 1)
            i += 1

    prev = Q.qmm_set_partitions(Q.QMM_PARTITIONS_EQUAL)
    try:
        f = threading.Thread(target=flipper)
        ws_ = [threading.Thread(target=worker, args=(r,)) for r in rules]
        f.start()
        for t in ws_:
            t.start()
        for t in ws_:
            t.join()
        stop.set()
        f.join()
    finally:
        Q.qmm_set_partitions(prev)
    assert not errors


# ---- balanced split (QMM_SPLIT_BALANCED) ----------------------------------------

@pytest.mark.parametrize("name", ["down", "o"])
def test_balanced_split_rows(name):
    """The balanced split of a call with a partial last wave (160 tiles on 152
    SMs): rows [0, head) are bitwise the unsplit call's, rows [head, M)
    bitwise those of a call on those rows alone at the tail's split, and both
    ranges agree with the oracle on sampled elements."""
    M, (Kred, Nout) = 2048, inputs.PROJECTIONS[name]
    p = inputs.make_w4a16(M, Kred, Nout, seed=81)
    d = Q.to_device(p)
    split, bm, bn, head = Q.qmm_call_plan(M, Kred, Nout, Q.QMM_SPLIT_BALANCED, with_head=True)
    assert 0 < head < M and head % bm == 0 and split > 1
    nbytes = Q.qmm_call_workspace_bytes(M, Kred, Nout, Q.QMM_SPLIT_BALANCED)
    assert nbytes == split * (M - head) * Nout * 2
    ws = torch.full((nbytes // 2,), float("nan"), dtype=torch.bfloat16, device="cuda")
    C = torch.empty((M, Nout), dtype=torch.bfloat16, device="cuda")
    used = Q.qmm_w4a16_g128(d["A"], d["Wq"], d["scales"], d["biases"], C,
                            split_req=Q.QMM_SPLIT_BALANCED, workspace=ws)
    assert used == split
    C1 = torch.empty_like(C)
    Q.qmm_w4a16_g128(d["A"], d["Wq"], d["scales"], d["biases"], C1, split_req=1)
    At = d["A"][head:].contiguous()
    Ct = torch.empty((M - head, Nout), dtype=torch.bfloat16, device="cuda")
    wt = torch.empty(Q.qmm_splitk_workspace_bytes(M - head, Nout, split), dtype=torch.uint8,
                     device="cuda")
    Q.qmm_w4a16_g128(At, d["Wq"], d["scales"], d["biases"], Ct, split_req=split, workspace=wt)
    torch.cuda.synchronize()
    got = _bits(C)
    assert np.array_equal(got[:head], _bits(C1)[:head]), "head rows differ from the unsplit call"
    assert np.array_equal(got[head:], _bits(Ct)), "tail rows differ from the tail call"
    cols = np.arange(3, Nout, 97)
    _check_sampled(p, got, 1, Q.QMM_PARTIAL_BF16, np.arange(0, head, 211), cols, "head")
    pt = dict(p, A=p["A"][head:])
    _check_sampled(pt, got[head:], split, Q.QMM_PARTIAL_BF16, np.arange(0, M - head, 17), cols,
                   "tail")


def test_balanced_split_without_a_partial_wave_is_the_planned_split():
    # gate at M = 2048: 608 tiles, four full waves on 152 SMs: nothing to cut
    M, (Kred, Nout) = 2048, inputs.PROJECTIONS["gate"]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    s, _, _, head = Q.qmm_call_plan(M, Kred, Nout, Q.QMM_SPLIT_BALANCED, with_head=True)
    if (M // 256) * (Nout // 128) % sms == 0:
        assert head == 0
    assert s == Q.qmm_call_plan(M, Kred, Nout, Q.QMM_SPLIT_PLANNED)[0] or head > 0


@pytest.mark.parametrize("name,M", [("k", 2048), ("k", 1024), ("q", 512), ("o", 256),
                                    ("gate", 129)])
def test_balanced_split_narrow_tile(name, M):
    """Where the wide tile leaves no full wave, the balanced split may take the
    128-row tile at its own split (see the plan): the whole output matches the
    oracle, and each full 128-row slice is bitwise the slice called alone
    (M = 128 takes the same kernel) at that split."""
    Kred, Nout = inputs.PROJECTIONS[name]
    p = inputs.make_w4a16(M, Kred, Nout, seed=83 + M)
    d = Q.to_device(p)
    split, bm, bn, head = Q.qmm_call_plan(M, Kred, Nout, Q.QMM_SPLIT_BALANCED, with_head=True)
    if (bm, bn) == Q.qmm_kernel_tile(M):
        pytest.skip("the wide tile is kept on this device")
    assert (bm, bn, head) == (128, 128, 0) and Q.qmm_kernel_tile(128) == (128, 128)
    nbytes = Q.qmm_call_workspace_bytes(M, Kred, Nout, Q.QMM_SPLIT_BALANCED)
    assert nbytes == (Q.qmm_splitk_workspace_bytes(M, Nout, split) if split > 1 else 0)
    ws = torch.full((max(nbytes, 16) // 2,), float("nan"), dtype=torch.bfloat16, device="cuda")
    C = torch.full((M, Nout), float("nan"), dtype=torch.bfloat16, device="cuda")
    used = Q.qmm_w4a16_g128(d["A"], d["Wq"], d["scales"], d["biases"], C,
                            split_req=Q.QMM_SPLIT_BALANCED, workspace=ws)
    assert used == split
    torch.cuda.synchronize()
    got = _bits(C)
    C64 = oracle.qmm(p["A"], p["Wq"], p["scales"], p["biases"])
    _check_full(p, got, split, Q.QMM_PARTIAL_BF16, C64, "%s M=%d narrow tile" % (name, M))
    wt = torch.empty(max(16, Q.qmm_splitk_workspace_bytes(128, Nout, split)), dtype=torch.uint8,
                     device="cuda")
    for r0 in range(0, M - 127, 128 * 5):
        Cs = torch.empty((128, Nout), dtype=torch.bfloat16, device="cuda")
        Q.qmm_w4a16_g128(d["A"][r0:r0 + 128].contiguous(), d["Wq"], d["scales"], d["biases"], Cs,
                         split_req=split, workspace=wt)
        torch.cuda.synchronize()
        assert np.array_equal(got[r0:r0 + 128], _bits(Cs)), "rows %d.. differ" % r0


@pytest.mark.parametrize("name,M", [("o", 2048), ("k", 2048), ("down", 16)])
def test_wrapper_sizes_the_workspace_of_every_plan(name, M):
    """w4a16_matmul allocates the workspace the library's plan needs for any
    split request; its C is bitwise the explicit call's."""
    Kred, Nout = inputs.PROJECTIONS[name]
    d = Q.to_device(inputs.make_w4a16(M, Kred, Nout, seed=87))
    for req in (0, Q.QMM_SPLIT_PLANNED, Q.QMM_SPLIT_BALANCED):
        C, used = Q.w4a16_matmul(d["A"], d["Wq"], d["scales"], d["biases"], split_req=req)
        ws = torch.empty(max(16, Q.qmm_call_workspace_bytes(M, Kred, Nout, req)),
                         dtype=torch.uint8, device="cuda")
        C2 = torch.empty_like(C)
        used2 = Q.qmm_w4a16_g128(d["A"], d["Wq"], d["scales"], d["biases"], C2, split_req=req,
                                 workspace=ws)
        torch.cuda.synchronize()
        assert used == used2 == Q.qmm_call_plan(M, Kred, Nout, req)[0]
        assert np.array_equal(_bits(C), _bits(C2)), (name, M, req)


# ---- cluster reduce (QMM_REDUCE_CLUSTER) ----------------------------------------

@pytest.mark.parametrize("name,M,split,dt", [
    ("k", 32, 10, Q.QMM_PARTIAL_BF16), ("q", 32, 4, Q.QMM_PARTIAL_BF16),
    ("down", 128, 4, Q.QMM_PARTIAL_BF16), ("ragged", 33, 5, Q.QMM_PARTIAL_BF16),
    ("k", 100, 10, Q.QMM_PARTIAL_F32), ("o", 64, 8, Q.QMM_PARTIAL_F32),
])
def test_cluster_reduce_equals_the_reduce_kernel(name, M, split, dt):
    """The cluster reduce gives C bit for bit as the planes and the reduce
    kernel do; where every cluster of the call fits the device at once it
    takes the cluster path, which writes no plane (the workspace keeps its
    NaN fill)."""
    Kred, Nout = inputs.RAGGED if name == "ragged" else inputs.PROJECTIONS[name]
    p = inputs.make_w4a16(M, Kred, Nout, seed=91 + M)
    d = Q.to_device(p)
    nbytes = Q.qmm_splitk_workspace_bytes(M, Nout, split, dt)
    prev = Q.qmm_set_kernels(Q.QMM_KERNELS_TCGEN05)
    try:
        outs = {}
        for mode in (Q.QMM_REDUCE_KERNEL, Q.QMM_REDUCE_CLUSTER):
            ws = torch.full((nbytes // 2,), float("nan"), dtype=torch.bfloat16, device="cuda")
            C = torch.full((M, Nout), float("nan"), dtype=torch.bfloat16, device="cuda")
            s = Q.qmm_w4a16_g128(d["A"], d["Wq"], d["scales"], d["biases"], C, split_req=split,
                                 workspace=ws, partial_dtype=dt,
                                 options=Q.qmm_options(reduce=mode))
            torch.cuda.synchronize()
            assert s == split
            outs[mode] = (_bits(C), bool(torch.isnan(ws.float()).all()))
        assert Q.qmm_kernel_status(clear=True) == 0
    finally:
        Q.qmm_set_kernels(prev)
    assert np.array_equal(outs[Q.QMM_REDUCE_CLUSTER][0], outs[Q.QMM_REDUCE_KERNEL][0])
    assert not outs[Q.QMM_REDUCE_KERNEL][1]  # the reduce kernel's planes are in the workspace
    if (name, M) in (("k", 32), ("q", 32), ("down", 128)):
        assert outs[Q.QMM_REDUCE_CLUSTER][1], "expected the cluster path (no planes written)"
    rows, cols = np.arange(0, M, 7), np.arange(1, Nout, 41)
    _check_sampled(p, outs[Q.QMM_REDUCE_CLUSTER][0], split, dt, rows, cols, "cluster reduce")


def test_cluster_reduce_under_the_default_table_and_static_weights():
    """The step's calls (M = 32 and 128, policy splits) under the cluster
    reduce, static weights and programmatic launch, back to back on one
    stream: every C bit for bit the reduce kernel's."""
    calls = [(n, M) for M in (32, 128) for n in ("q", "k", "o", "gate", "down")]
    probs = {c: inputs.make_w4a16(c[1], *inputs.PROJECTIONS[c[0]], seed=5) for c in calls}
    devs = {c: Q.to_device(probs[c]) for c in calls}
    ws = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    res = {}
    prev = Q.qmm_set_weights_static(True)
    try:
        for mode in (Q.QMM_REDUCE_KERNEL, Q.QMM_REDUCE_CLUSTER):
            opt = Q.qmm_options(reduce=mode)
            Cs = {}
            for c in calls:
                M, (Kred, Nout) = c[1], inputs.PROJECTIONS[c[0]]
                Cs[c] = torch.empty((M, Nout), dtype=torch.bfloat16, device="cuda")
                Q.qmm_w4a16_g128(devs[c]["A"], devs[c]["Wq"], devs[c]["scales"],
                                 devs[c]["biases"], Cs[c], workspace=ws, options=opt)
            torch.cuda.synchronize()
            res[mode] = {c: _bits(Cs[c]) for c in calls}
        assert Q.qmm_kernel_status(clear=True) == 0
    finally:
        Q.qmm_set_weights_static(prev)
    for c in calls:
        assert np.array_equal(res[Q.QMM_REDUCE_CLUSTER][c], res[Q.QMM_REDUCE_KERNEL][c]), c


@pytest.mark.parametrize("name,M,split,dt", [
    ("k", 16, 5, Q.QMM_PARTIAL_BF16), ("down", 8, 4, Q.QMM_PARTIAL_BF16),
    ("ragged", 1, 10, Q.QMM_PARTIAL_BF16), ("o", 16, 16, Q.QMM_PARTIAL_F32),
])
def test_cluster_reduce_lean_family(name, M, split, dt):
    """The lean family (few activation rows) under the cluster reduce: C bit
    for bit the reduce kernel's (through the cluster path where the device
    holds all of the call's clusters at once, else the reduce kernel), and
    the oracle on a sample."""
    Kred, Nout = inputs.RAGGED if name == "ragged" else inputs.PROJECTIONS[name]
    p = inputs.make_w4a16(M, Kred, Nout, seed=17 + M)
    d = Q.to_device(p)
    nbytes = Q.qmm_splitk_workspace_bytes(M, Nout, split, dt)
    outs = {}
    for mode in (Q.QMM_REDUCE_KERNEL, Q.QMM_REDUCE_CLUSTER):
        ws = torch.full((nbytes // 2,), float("nan"), dtype=torch.bfloat16, device="cuda")
        C = torch.full((M, Nout), float("nan"), dtype=torch.bfloat16, device="cuda")
        s = Q.qmm_w4a16_g128(d["A"], d["Wq"], d["scales"], d["biases"], C, split_req=split,
                             workspace=ws, partial_dtype=dt,
                             options=Q.qmm_options(reduce=mode, kernels=Q.QMM_KERNELS_DEFAULT))
        torch.cuda.synchronize()
        assert s == split
        outs[mode] = (_bits(C), bool(torch.isnan(ws.float()).all()))
    assert Q.qmm_kernel_status(clear=True) == 0
    assert np.array_equal(outs[Q.QMM_REDUCE_CLUSTER][0], outs[Q.QMM_REDUCE_KERNEL][0])
    if (name, M) == ("k", 16):  # 32 clusters of 5: every one fits the device at once
        assert outs[Q.QMM_REDUCE_CLUSTER][1], "expected the cluster path (no planes written)"
    _check_sampled(p, outs[Q.QMM_REDUCE_CLUSTER][0], split, dt, np.arange(M),
                   np.arange(0, Nout, 29), "lean cluster reduce")
