"""Host-side checks of the C-ABI library (CPU only): it builds, loads and
exports every entry point include/qmm.h declares; the split plan is
bit-exact against the oracle's; argument errors come back as codes before any
CUDA work."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
from split_w4a16_quantized_gb300 import build, inputs
from split_w4a16_quantized_gb300 import qmm as Q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
M_LIST = [1, 2, 4, 8, 9, 16, 17, 32, 33, 64, 100, 128, 129, 256, 2048, 4096]
SHAPES = list(inputs.PROJECTIONS.values()) + [inputs.RAGGED]


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()


def _declared():
    text = open(os.path.join(ROOT, "include", "qmm.h")).read()
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(qmm_\w+)\s*\(", text, re.M)))


def test_exports_every_declared_symbol():
    names = _declared()
    assert "qmm_w4a16_g128" in names and "qmm_splitk_plan" in names and "qmm_splitk_reduce" in names
    lib = ctypes.CDLL(Q.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(Q._SIGS), "binding and header disagree"


def test_strerror_codes():
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert Q.qmm_strerror(code) != "unknown error"
    assert Q.qmm_strerror(7) == "unknown error"


def test_pages_preset_values():
    p = Q.qmm_policy_preset(Q.QMM_PRESET_PAGES)
    assert p.as_tuple() == (32, 32, 320, 16, 128)


@pytest.mark.parametrize("sms", [148, 152])
def test_gb300_preset(sms):
    for M in M_LIST:
        p = Q.qmm_policy_preset(Q.QMM_PRESET_GB300, M, sms)
        assert (p.bm, p.bn) == Q.qmm_kernel_tile(M)
        assert p.target_blocks % sms == 0 and p.target_blocks >= sms
        assert p.min_k_per_split == (512 if M <= 8 else 128)


def _policies():
    out = [Q.qmm_policy_preset(Q.QMM_PRESET_PAGES)]
    for sms in (108, 132, 148, 152):
        out += [Q.qmm_policy_preset(Q.QMM_PRESET_GB300, M, sms) for M in (1, 16, 32, 128)]
    return out


def test_plan_bit_exact_against_oracle_on_workload_shapes():
    for pol in _policies():
        for M in M_LIST:
            for Kred, Nout in SHAPES:
                got = Q.qmm_splitk_plan(M, Kred, Nout, pol)
                assert got == oracle.splitk_plan(M, Kred, Nout, *pol.as_tuple()), (pol, M, Kred, Nout)


def test_plan_bit_exact_against_oracle_fuzz():
    rng = np.random.default_rng(21)
    for _ in range(20000):
        M = int(rng.integers(1, 5000))
        Kred = 128 * int(rng.integers(1, 129))
        Nout = int(rng.integers(1, 20000))
        pol = Q.qmm_policy(int(rng.integers(1, 257)), int(rng.integers(1, 257)),
                           int(rng.integers(0, 5000)), int(rng.integers(1, 65)),
                           128 * int(rng.integers(1, 17)))
        assert Q.qmm_splitk_plan(M, Kred, Nout, pol) == \
            oracle.splitk_plan(M, Kred, Nout, *pol.as_tuple())


def test_plan_near_equal_bit_exact_against_oracle():
    for pol in _policies():
        for M in M_LIST:
            for Kred, Nout in SHAPES:
                got = Q.qmm_splitk_plan_near_equal(M, Kred, Nout, pol)
                assert got == oracle.splitk_plan_near_equal(M, Kred, Nout, *pol.as_tuple())
                assert got >= Q.qmm_splitk_plan(M, Kred, Nout, pol)
    rng = np.random.default_rng(22)
    for _ in range(20000):
        M = int(rng.integers(1, 5000))
        Kred = 128 * int(rng.integers(1, 129))
        Nout = int(rng.integers(1, 20000))
        pol = Q.qmm_policy(int(rng.integers(1, 257)), int(rng.integers(1, 257)),
                           int(rng.integers(0, 5000)), int(rng.integers(1, 65)),
                           128 * int(rng.integers(1, 17)))
        assert Q.qmm_splitk_plan_near_equal(M, Kred, Nout, pol) == \
            oracle.splitk_plan_near_equal(M, Kred, Nout, *pol.as_tuple())


def test_gb300_near_equal_splits_of_the_workload():
    # 152 SMs, one CTA each: the divisor rule leaves o and down at 4 ways
    # (80 CTAs); near-equal partitions take 7 (140 CTAs, the longest
    # partition 11 of 76 groups instead of 19, and 5 of 32 instead of 8).
    # k/v stay at 10: 16 partitions of 20 groups still leave one of 2.
    got = {}
    for M in (32, 128):
        pol = Q.qmm_policy_preset(Q.QMM_PRESET_GB300, M, 152)
        for name, (Kred, Nout) in inputs.PROJECTIONS.items():
            got[name, M] = (Q.qmm_splitk_plan(M, Kred, Nout, pol),
                            Q.qmm_splitk_plan_near_equal(M, Kred, Nout, pol))
    for M in (32, 128):
        assert got["down", M] == (4, 7) and got["o", M] == (4, 7)
        assert got["k", M] == (10, 10) and got["v", M] == (10, 10)
        assert got["q", M] == (4, 4) and got["gate", M] == (2, 2) and got["up", M] == (2, 2)


def test_partition_rule_switch():
    assert Q.qmm_set_partitions(Q.QMM_PARTITIONS_NEAR_EQUAL) == Q.QMM_PARTITIONS_EQUAL
    assert Q.qmm_set_partitions(Q.QMM_PARTITIONS_EQUAL) == Q.QMM_PARTITIONS_NEAR_EQUAL
    assert Q.lib().qmm_set_partitions(2) == Q.QMM_EINVAL
    assert Q.lib().qmm_set_partitions(-1) == Q.QMM_EINVAL
    with pytest.raises(Q.QmmError):
        Q.qmm_set_partitions(5)


def test_plan_errors():
    pol = Q.qmm_policy_preset(Q.QMM_PRESET_PAGES)
    s = ctypes.c_int(0)
    lib = Q.lib()
    assert lib.qmm_splitk_plan(16, 2500, 1024, ctypes.byref(pol), ctypes.byref(s)) == Q.QMM_ESHAPE
    assert lib.qmm_splitk_plan(0, 2560, 1024, ctypes.byref(pol), ctypes.byref(s)) == Q.QMM_EINVAL
    assert lib.qmm_splitk_plan(16, 2560, 1024, None, ctypes.byref(s)) == Q.QMM_EINVAL
    bad = Q.qmm_policy(32, 32, 320, 16, 100)
    assert lib.qmm_splitk_plan(16, 2560, 1024, ctypes.byref(bad), ctypes.byref(s)) == Q.QMM_EINVAL
    for plan in (lib.qmm_splitk_plan_near_equal,):
        assert plan(16, 2500, 1024, ctypes.byref(pol), ctypes.byref(s)) == Q.QMM_ESHAPE
        assert plan(0, 2560, 1024, ctypes.byref(pol), ctypes.byref(s)) == Q.QMM_EINVAL
        assert plan(16, 2560, 1024, None, ctypes.byref(s)) == Q.QMM_EINVAL
        assert plan(16, 2560, 1024, ctypes.byref(bad), ctypes.byref(s)) == Q.QMM_EINVAL
        assert plan(16, 2560, 1024, ctypes.byref(pol), None) == Q.QMM_EINVAL


def test_workspace_bytes():
    assert Q.qmm_splitk_workspace_bytes(16, 1024, 1) == 0
    assert Q.qmm_splitk_workspace_bytes(16, 1024, 10) == 10 * 16 * 1024 * 2
    assert Q.qmm_splitk_workspace_bytes(16, 1024, 10, Q.QMM_PARTIAL_F32) == 10 * 16 * 1024 * 4
    assert Q.qmm_splitk_workspace_bytes(16, 1024, 10, 7) == 0
    assert Q.qmm_gemm_workspace_bytes(512, 512, 6) == 6 * 512 * 512 * 4
    assert Q.qmm_gemm_workspace_bytes(512, 512, 1) == 0


def test_argument_errors_before_any_cuda_work():
    # fake, never-dereferenced addresses: every call must fail validation first
    lib = Q.lib()
    P = ctypes.c_void_p
    a, w, s, b, c = P(0x10000), P(0x20000), P(0x30000), P(0x40000), P(0x50000)
    call = lambda *x: lib.qmm_w4a16_g128(*x)
    assert call(None, w, s, b, c, 16, 2560, 1024, 0, None, None, 0, 0, None, None) == Q.QMM_EINVAL
    assert call(a, w, s, b, c, 0, 2560, 1024, 0, None, None, 0, 0, None, None) == Q.QMM_EINVAL
    assert call(a, w, s, b, c, 16, 2500, 1024, 0, None, None, 0, 0, None, None) == Q.QMM_ESHAPE
    assert call(a, w, s, b, c, 16, 2560, 1024, 0, None, None, 0, 5, None, None) == Q.QMM_EINVAL
    # negative split requests other than QMM_SPLIT_PLANNED / BALANCED are rejected
    assert call(a, w, s, b, c, 16, 2560, 1024, -3, None, None, 0, 0, None, None) == Q.QMM_EINVAL
    # (a planned or balanced split request passes validation and then needs the device)
    for req in (Q.QMM_SPLIT_PLANNED, Q.QMM_SPLIT_BALANCED):
        assert call(a, w, s, b, c, 16, 2560, 1024, req, None, None, 0, 0, None,
                    None) in (Q.QMM_ENODEV, Q.QMM_EWORKSPACE)
    assert call(P(0x10002), w, s, b, c, 16, 2560, 1024, 0, None, None, 0, 0, None, None) == \
        Q.QMM_EALIGN
    assert call(a, w, P(0x30001), b, c, 16, 2560, 1024, 0, None, None, 0, 0, None, None) == \
        Q.QMM_EALIGN
    assert lib.qmm_splitk_reduce(None, 0, 2, 16, 16, c, None) == Q.QMM_EINVAL
    assert lib.qmm_splitk_reduce(a, 0, 2, 16, 16, P(0x50008), None) == Q.QMM_EALIGN
    assert lib.qmm_gemm_bf16_splitk(a, w, c, 512, 512, 1000, 2, None, 0, None) == Q.QMM_ESHAPE
    assert lib.qmm_gemm_bf16_splitk(a, w, c, 512, 512, 1024, 17, None, 0, None) == Q.QMM_ESHAPE


def test_noalloc_checks_match_the_main_entry_point():
    # fake, never-dereferenced addresses: the allocation-free call runs the
    # checks of qmm_w4a16_g128 in the same order and returns the same codes
    lib = Q.lib()
    P = ctypes.c_void_p
    a, w, s, b, c = P(0x10000), P(0x20000), P(0x30000), P(0x40000), P(0x50000)
    bad = Q.qmm_policy(0, 32, 152, 16, 128)  # bm < 1
    main = lambda A, M, split, pol: lib.qmm_w4a16_g128(A, w, s, b, c, M, 2560, 1024, split, pol,
                                                       None, 0, 0, None, None)
    noalloc = lambda A, M, split, pol: lib.qmm_w4a16_g128_noalloc(A, w, s, b, c, M, 2560, 1024,
                                                                  split, pol, 0, None, None)
    cases = [
        (a, 16, 2, ctypes.byref(bad)),         # invalid policy with a forced split
        (a, 16, 0, ctypes.byref(bad)),         # invalid policy with the policy split
        (a, 16, -3, None),                     # negative request other than the named ones
        (P(0x10002), 2048, 20, None),          # misaligned A, planes far beyond the buffer
        (P(0x10002), 16, Q.QMM_SPLIT_PLANNED, None),
    ]
    for A, M, split, pol in cases:
        assert noalloc(A, M, split, pol) == main(A, M, split, pol), (M, split)
    assert noalloc(a, 16, 2, ctypes.byref(bad)) == Q.QMM_EINVAL
    # the balanced split needs a grouped launch and is not offered here
    assert noalloc(a, 16, Q.QMM_SPLIT_BALANCED, None) == Q.QMM_EINVAL
    assert noalloc(P(0x10002), 2048, 20, None) == Q.QMM_EALIGN
    # valid arguments without a usable device: no device, before the limit
    # check and the address lookup
    if not torch.cuda.is_available():
        assert noalloc(a, 2048, 20, None) == Q.QMM_ENODEV
        assert noalloc(a, 16, Q.QMM_SPLIT_PLANNED, None) == Q.QMM_ENODEV


def test_overlap_schedule_bit_exact_against_oracle():
    rng = np.random.default_rng(26)
    for _ in range(2000):
        n = int(rng.integers(1, 30))
        b = int(rng.integers(1, 6))
        t = [rng.random(n) * float(rng.choice([1.0, 10.0, 100.0])) for _ in range(3)]
        if rng.random() < 0.3:
            t = [np.full(n, float(rng.integers(0, 9))) for _ in range(3)]
        for out_reuse in (False, True):
            T, ev = Q.qmm_overlap_schedule(n, b, *t, out_reuse=out_reuse, with_events=True)
            To, evo = oracle.overlap_schedule(n, b, *t, out_reuse=out_reuse, with_events=True)
            assert T == To and np.array_equal(ev, evo)


def test_overlap_schedule_errors():
    lib = Q.lib()
    D = ctypes.POINTER(ctypes.c_double)
    one = (ctypes.c_double * 1)(1.0)
    neg = (ctypes.c_double * 1)(-1.0)
    T = ctypes.c_double()
    assert lib.qmm_overlap_schedule(0, 1, one, one, one, 0, ctypes.byref(T), None) == Q.QMM_EINVAL
    assert lib.qmm_overlap_schedule(1, 0, one, one, one, 0, ctypes.byref(T), None) == Q.QMM_EINVAL
    assert lib.qmm_overlap_schedule(1, 1, neg, one, one, 0, ctypes.byref(T), None) == Q.QMM_EINVAL
    assert lib.qmm_overlap_schedule(1, 1, one, one, one, 2, ctypes.byref(T), None) == Q.QMM_EINVAL
    assert lib.qmm_overlap_schedule(1, 1, None, one, one, 0, ctypes.byref(T), None) == Q.QMM_EINVAL
    assert lib.qmm_overlap_schedule(1, 1, one, one, one, 0, None, None) == Q.QMM_EINVAL
    assert lib.qmm_overlap_schedule(1, 1, one, one, one, 0, ctypes.byref(T), None) == Q.QMM_OK
    assert T.value == 3.0


def test_stream_executor_argument_errors_before_any_cuda_work():
    lib = Q.lib()
    P = ctypes.c_void_p
    ok = Q.qmm_stream_call(0x1000, 0x2000, 0x30000, 0x40000, 0x50000, 16, 2560, 1024)
    calls = (Q.qmm_stream_call * 1)(ok)
    arena = P(0x100000)
    run = lambda c, n, b, a: lib.qmm_w4a16_g128_stream(c, n, b, a, 1 << 30, None, None, None,
                                                       None)
    assert run(None, 1, 2, arena) == Q.QMM_EINVAL
    assert run(calls, 0, 2, arena) == Q.QMM_EINVAL
    assert run(calls, 1, 0, arena) == Q.QMM_EINVAL
    assert run(calls, 1, 2, None) == Q.QMM_EINVAL
    assert run(calls, 1, 2, P(0x100010)) == Q.QMM_EALIGN
    bad = (Q.qmm_stream_call * 2)(ok, Q.qmm_stream_call(0x1000, 0x2000, 0x30000, 0x40000,
                                                          0x50000, 16, 2500, 1024))
    assert run(bad, 2, 2, arena) == Q.QMM_ESHAPE          # the second chunk's Kred
    bad[1] = Q.qmm_stream_call(0x1000, None, 0x30000, 0x40000, 0x50000, 16, 2560, 1024)
    assert run(bad, 2, 2, arena) == Q.QMM_EINVAL
    bad[1] = Q.qmm_stream_call(0x1000, 0x2000, 0x30004, 0x40000, 0x50000, 16, 2560, 1024)
    assert run(bad, 2, 2, arena) == Q.QMM_EALIGN
    assert lib.qmm_stream_arena_bytes(None, 1, 1) == 0
    assert lib.qmm_stream_arena_bytes(calls, 1, 0) == 0


def test_grouped_argument_errors_before_any_cuda_work():
    lib = Q.lib()
    P = ctypes.c_void_p
    ok = Q.qmm_group_call(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 16, 2560, 1024)
    run = lambda c, n, dt=0: lib.qmm_w4a16_g128_grouped(c, n, P(0x100000), 1 << 30, dt, None,
                                                         None)
    one = (Q.qmm_group_call * 1)(ok)
    assert run(None, 1) == Q.QMM_EINVAL
    assert run(one, 0) == Q.QMM_EINVAL
    assert run(one, 1, 7) == Q.QMM_EINVAL
    two = (Q.qmm_group_call * 2)(ok, Q.qmm_group_call(0x10000, 0x20000, 0x30000, 0x40000,
                                                      0x50000, 16, 2500, 1024))
    assert run(two, 2) == Q.QMM_ESHAPE                    # the second call's Kred
    two[1] = Q.qmm_group_call(0x10000, 0x20000, 0x30000, 0x40000, None, 16, 2560, 1024)
    assert run(two, 2) == Q.QMM_EINVAL
    two[1] = Q.qmm_group_call(0x10002, 0x20000, 0x30000, 0x40000, 0x50000, 16, 2560, 1024)
    assert run(two, 2) == Q.QMM_EALIGN
    two[1] = Q.qmm_group_call(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0, 2560, 1024)
    assert run(two, 2) == Q.QMM_EINVAL
    assert lib.qmm_group_workspace_bytes(None, 1, 0) == 0
    assert lib.qmm_group_workspace_bytes(two, 2, 0) == 0


def test_attention_splits_bit_exact_against_oracle():
    rng = np.random.default_rng(27)
    for _ in range(5000):
        B, Hkv = int(rng.integers(1, 65)), int(rng.choice([1, 2, 4, 8, 16]))
        qg = int(rng.choice([1, 2, 4, 8]))
        Lmax, sms = int(rng.integers(1, 40000)), int(rng.integers(1, 200))
        got = Q.qmm_decode_attention_splits(B, Hkv * qg, Hkv, Lmax, sms)
        want = oracle.attention_splits(B, Hkv, Lmax, sms, 4, 512)
        assert got == want
    # the workload: 32 sequences x 8 KV heads on 152 SMs, 4 blocks per SM
    assert Q.qmm_decode_attention_splits(32, 32, 8, 8192, 152) == 3
    assert Q.qmm_decode_attention_workspace_bytes(32, 32, 128, 2) == 32 * 32 * 2 * 130 * 4
    assert Q.qmm_decode_attention_workspace_bytes(32, 32, 128, 1) == 0


def test_attention_argument_errors_before_any_cuda_work():
    lib = Q.lib()
    P = ctypes.c_void_p
    q, k, v, ln, o = P(0x10000), P(0x20000), P(0x30000), P(0x40000), P(0x50000)
    run = lambda *a: lib.qmm_decode_attention(*a)
    ok = (q, k, v, ln, o, 2, 32, 8, 100, 128, 0.0, 0, None, 0, None, None)
    bad = lambda i, x: tuple(x if j == i else a for j, a in enumerate(ok))
    assert run(*bad(0, None)) == Q.QMM_EINVAL
    assert run(*bad(3, None)) == Q.QMM_EINVAL
    assert run(*bad(5, 0)) == Q.QMM_EINVAL
    assert run(*bad(6, 30)) == Q.QMM_EINVAL          # Hq not a multiple of Hkv
    assert run(*bad(9, 96)) == Q.QMM_ESHAPE          # D
    assert run(*bad(6, 48)) == Q.QMM_ESHAPE          # 6 query heads per KV head
    assert run(*bad(11, -1)) == Q.QMM_EINVAL
    assert run(*bad(0, P(0x10008))) == Q.QMM_EALIGN
    assert run(*bad(3, P(0x40002))) == Q.QMM_EALIGN
    s = ctypes.c_int()
    assert lib.qmm_decode_attention_splits(0, 32, 8, 100, 152, ctypes.byref(s)) == Q.QMM_EINVAL
    assert lib.qmm_decode_attention_splits(1, 30, 8, 100, 152, ctypes.byref(s)) == Q.QMM_EINVAL


def test_fused_reduce_workspace_holds_the_counters():
    from split_w4a16_quantized_gb300 import qmm as Q
    prev_k = Q.qmm_set_kernels(Q.QMM_KERNELS_TCGEN05)
    prev = Q.qmm_set_reduce(Q.QMM_REDUCE_FUSED)
    try:
        # planes, rounded up to 256 bytes, 256 bytes of slack, the fixed counter area
        planes = 4 * 128 * 2560 * 2
        assert Q.qmm_splitk_workspace_bytes(128, 2560, 4, Q.QMM_PARTIAL_BF16) == \
            (planes + 255) // 256 * 256 + 256 + 32768
        assert Q.qmm_splitk_workspace_bytes(128, 2560, 1, Q.QMM_PARTIAL_BF16) == 0
        Q.qmm_set_kernels(Q.QMM_KERNELS_MMA_SYNC)  # the separate reduce: planes only
        assert Q.qmm_splitk_workspace_bytes(128, 2560, 4, Q.QMM_PARTIAL_BF16) == planes
        with pytest.raises(Q.QmmError):
            Q.qmm_set_reduce(7)
    finally:
        Q.qmm_set_reduce(prev)
        Q.qmm_set_kernels(prev_k)


def test_grouped_schedule_setting():
    from split_w4a16_quantized_gb300 import qmm as Q
    prev = Q.qmm_set_grouped_schedule(Q.QMM_GROUPED_PERSISTENT)
    assert prev == Q.QMM_GROUPED_PERSISTENT  # the default (no other test leaves it changed)
    try:
        assert Q.qmm_set_grouped_schedule(Q.QMM_GROUPED_TILES) == Q.QMM_GROUPED_PERSISTENT
        assert Q.qmm_set_grouped_schedule(Q.QMM_GROUPED_TILES) == Q.QMM_GROUPED_TILES
        with pytest.raises(Q.QmmError):
            Q.qmm_set_grouped_schedule(2)
    finally:
        Q.qmm_set_grouped_schedule(prev)


def test_group_plan_bit_exact_against_the_oracle():
    """qmm_group_plan equals the oracle's restatement of the rule on the
    workload's groups and on seeded random groups (both partition rules, both
    plane types, several SM counts).  The tile of each M is the library's
    kernel table, the same on both sides."""
    import oracle
    from split_w4a16_quantized_gb300 import inputs
    from split_w4a16_quantized_gb300 import qmm as Q
    tiles = lambda M: Q.qmm_kernel_tile(M)
    cases = [[(M,) + inputs.PROJECTIONS[n] for n in inputs.PROJECTIONS]
             for M in (1, 4, 8, 16, 32, 64, 128, 2048)]
    rng = np.random.default_rng(21)
    for _ in range(60):
        n = int(rng.integers(1, 17))
        Ms = rng.choice([1, 3, 8, 16, 20, 32, 40, 64, 100, 128, 129, 512], size=n)
        cases.append([(int(M), 128 * int(rng.integers(1, 129)), int(rng.integers(1, 12000)))
                      for M in Ms])
    prev = Q.qmm_set_partitions(Q.QMM_PARTITIONS_EQUAL)
    try:
        for k, shapes in enumerate(cases):
            near = k % 3 == 2
            dt = Q.QMM_PARTIAL_F32 if k % 4 == 3 else Q.QMM_PARTIAL_BF16
            sms = (152, 132, 108)[k % 3]
            Q.qmm_set_partitions(Q.QMM_PARTITIONS_NEAR_EQUAL if near else Q.QMM_PARTITIONS_EQUAL)
            got = Q.qmm_group_plan(shapes, sms, dt)
            own = lambda M: None if Q.qmm_kernel_grouped(M) else \
                Q.qmm_policy_preset(Q.QMM_PRESET_GB300, M, sms).as_tuple()
            want = oracle.group_plan(shapes, tiles, sms, near_equal=near,
                                     partial_bytes=4 if dt == Q.QMM_PARTIAL_F32 else 2,
                                     own_launch=own)
            assert got == want, (k, shapes, got, want)
    finally:
        Q.qmm_set_partitions(prev)


def test_group_plan_setting():
    from split_w4a16_quantized_gb300 import qmm as Q
    prev = Q.qmm_set_group_plan(Q.QMM_GROUP_PLAN_GROUP)
    assert prev == Q.QMM_GROUP_PLAN_CALLS  # the default
    try:
        assert Q.qmm_set_group_plan(Q.QMM_GROUP_PLAN_CALLS) == Q.QMM_GROUP_PLAN_GROUP
        with pytest.raises(Q.QmmError):
            Q.qmm_set_group_plan(5)
        with pytest.raises(Q.QmmError):
            Q.qmm_group_plan([(32, 100, 1024)], 152)   # Kred not a multiple of 128
        with pytest.raises(Q.QmmError):
            Q.qmm_group_plan([(0, 2560, 1024)], 152)
    finally:
        Q.qmm_set_group_plan(prev)


def test_group_plan_falls_back_to_the_policy_on_huge_launches():
    """A launch of more than 65536 tiles is not planned: each call keeps the
    chapter's policy split for the given SM count (host only, no device)."""
    from split_w4a16_quantized_gb300 import qmm as Q
    shapes = [(16384, 2560, 16384)] * 9 + [(16384, 2560, 1024)]  # 64 x 128 tiles each
    got = Q.qmm_group_plan(shapes, 152)
    want = [Q.qmm_splitk_plan(M, K, N, Q.qmm_policy_preset(Q.QMM_PRESET_GB300, M, 152))
            for M, K, N in shapes]
    assert got == want
    # exactly the limit unsplit is planned; a split would pass the limit, so
    # none is made
    assert Q.qmm_group_plan([(16384, 2560, 16384)] * 8, 152) == [1] * 8
    # a call of another tile width is planned in its own launch: k at M = 16
    # beside them splits as it would alone (the chapter policy's split)
    alone = Q.qmm_group_plan([(16, 2560, 1024)], 152)
    assert alone[0] > 1
    assert Q.qmm_group_plan([(16384, 2560, 16384)] * 8 + [(16, 2560, 1024)], 152) == [1] * 8 + alone


# ---- per-call options -------------------------------------------------------

def test_options_init_and_binding_default():
    o = Q.qmm_options()
    Q.lib().qmm_options_init(ctypes.byref(o))
    assert all(getattr(o, f) == Q.QMM_OPT_DEFAULT for f in Q._OPTION_FIELDS)
    Q.lib().qmm_options_init(None)  # no-op


@pytest.mark.parametrize("field,bad", [("kernels", 4), ("partitions", 2), ("reduce", 3),
                                       ("weights_static", 2), ("pdl", -2),
                                       ("grouped_schedule", 2), ("group_plan", 5)])
def test_options_out_of_range_rejected_first(field, bad):
    o = Q.qmm_options(**{field: bad})
    s = ctypes.c_int(0)
    # rejected before the shape check (Kred 100 would be QMM_ESHAPE)
    rc = Q.lib().qmm_call_plan(16, 100, 1024, 0, None, 0, 152, ctypes.byref(o),
                               ctypes.byref(s), None, None, None)
    assert rc == Q.QMM_EINVAL
    assert Q.lib().qmm_splitk_workspace_bytes_ex(16, 1024, 4, 0, ctypes.byref(o)) == 0
    # and before any device pointer is looked at
    rc = Q.lib().qmm_w4a16_g128_ex(None, None, None, None, None, 16, 2560, 1024, 0, None, None,
                                   0, 0, None, None, ctypes.byref(o))
    assert rc == Q.QMM_EINVAL


def test_options_override_the_process_settings_for_one_call():
    prev = Q.qmm_set_partitions(Q.QMM_PARTITIONS_EQUAL)
    try:
        eq = Q.qmm_call_plan(128, 9728, 2560, num_sms=152)
        ne = Q.qmm_call_plan(128, 9728, 2560, num_sms=152,
                             options=Q.qmm_options(partitions=Q.QMM_PARTITIONS_NEAR_EQUAL))
        pol = Q.qmm_policy_preset(Q.QMM_PRESET_GB300, 128, 152)
        assert eq[0] == Q.qmm_splitk_plan(128, 9728, 2560, pol) == 4
        assert ne[0] == Q.qmm_splitk_plan_near_equal(128, 9728, 2560, pol) == 7
        # the process setting is untouched by the call
        assert Q.qmm_set_partitions(Q.QMM_PARTITIONS_EQUAL) == Q.QMM_PARTITIONS_EQUAL
        Q.qmm_set_partitions(Q.QMM_PARTITIONS_NEAR_EQUAL)
        assert Q.qmm_call_plan(128, 9728, 2560, num_sms=152)[0] == 7
        assert Q.qmm_call_plan(128, 9728, 2560, num_sms=152,
                               options=Q.qmm_options(partitions=Q.QMM_PARTITIONS_EQUAL))[0] == 4
    finally:
        Q.qmm_set_partitions(prev)
    # the kernel table picks the tile; the fused reduce adds its counter area
    assert Q.qmm_call_plan(32, 2560, 9728, num_sms=152,
                           options=Q.qmm_options(kernels=Q.QMM_KERNELS_MMA_SYNC))[1:] == \
        (32, 128)
    plain = Q.qmm_splitk_workspace_bytes(128, 1024, 10)
    fused = Q.qmm_splitk_workspace_bytes(128, 1024, 10,
                                         options=Q.qmm_options(reduce=Q.QMM_REDUCE_FUSED))
    assert plain == 10 * 128 * 1024 * 2 and fused > plain


def test_options_two_threads_get_their_own_rule():
    """Two threads plan the same call under different partition rules while
    the process-wide rule is a third party's: each always gets its own."""
    import threading
    want = {Q.QMM_PARTITIONS_EQUAL: 4, Q.QMM_PARTITIONS_NEAR_EQUAL: 7}
    errors = []
    barrier = threading.Barrier(3)

    def worker(rule):
        o = Q.qmm_options(partitions=rule)
        barrier.wait()
        for _ in range(2000):
            if Q.qmm_call_plan(128, 9728, 2560, num_sms=152, options=o)[0] != want[rule]:
                errors.append(rule)
                return

    def flipper():
        barrier.wait()
        for i in range(2000):
            Q.qmm_set_partitions(i & 1)

    prev = Q.qmm_set_partitions(Q.QMM_PARTITIONS_EQUAL)
    try:
        ts = [threading.Thread(target=worker, args=(r,)) for r in want] + \
            [threading.Thread(target=flipper)]
        for t in ts:
            t.start()
        for t in ts:
            t.join()
    finally:
        Q.qmm_set_partitions(prev)
    assert not errors


# ---- balanced split plan -------------------------------------------------------

@pytest.mark.parametrize("sms", [148, 152])
@pytest.mark.parametrize("name", sorted(inputs.PROJECTIONS))
@pytest.mark.parametrize("M", [300, 1000, 2048, 4096])
def test_balanced_plan_structure(sms, name, M):
    """QMM_SPLIT_BALANCED cuts only calls with a partial last wave, at whole row
    tiles that fit the full waves, and splits the tail at a split the
    partition rule accepts; the workspace holds exactly the tail's planes."""
    Kred, Nout = inputs.PROJECTIONS[name]
    s, bm, bn, head = Q.qmm_call_plan(M, Kred, Nout, Q.QMM_SPLIT_BALANCED, num_sms=sms,
                                      with_head=True)
    rt, ct = -(-M // bm), -(-Nout // bn)
    G = Kred // 128
    ws = Q.qmm_call_workspace_bytes(M, Kred, Nout, Q.QMM_SPLIT_BALANCED, num_sms=sms)
    planned = Q.qmm_call_plan(M, Kred, Nout, Q.QMM_SPLIT_PLANNED, num_sms=sms)[0]
    wide = Q.qmm_kernel_tile(M)
    if head == 0:
        if (bm, bn) == wide:
            assert s == planned
        else:
            # the next narrower tile at the occupancy rule's split for it: no
            # larger than the wide tile's, and one wave
            assert (bm, bn) == (wide[0] // 2, wide[1])
            assert -(-M // wide[0]) * ct <= sms
            assert s == oracle.splitk_plan(M, Kred, Nout, bm, bn, sms, 16)
            assert s <= planned and rt * ct * s <= sms
        assert ws == Q.qmm_splitk_workspace_bytes(M, Nout, s)
        return
    tiles = rt * ct
    assert tiles > sms and tiles % sms != 0
    assert head % bm == 0 and 0 < head < M
    assert (head // bm) * ct <= tiles // sms * sms
    assert 1 <= s <= min(16, G) and G % s == 0
    assert ws == (s * (M - head) * Nout * 2 if s > 1 else 0)


def test_balanced_plan_cuts_the_wave_tail_of_down_and_o():
    for name in ("down", "o"):
        Kred, Nout = inputs.PROJECTIONS[name]
        s, bm, _, head = Q.qmm_call_plan(2048, Kred, Nout, Q.QMM_SPLIT_BALANCED, num_sms=152,
                                         with_head=True)
        # 8 x 20 tiles of 256 x 128: 7 row tiles fill the first wave
        assert (bm, head) == (256, 1792) and s > 1
    # no partial wave (gate: 608 = 4 x 152) or no full wave (k: 64 tiles): no cut
    for name in ("gate", "k"):
        Kred, Nout = inputs.PROJECTIONS[name]
        assert Q.qmm_call_plan(2048, Kred, Nout, Q.QMM_SPLIT_BALANCED, num_sms=152,
                               with_head=True)[3] == 0


@pytest.mark.parametrize("name,M,want", [
    # k at M = 2048: 64 wide tiles at split 2 become 128 narrow tiles unsplit
    ("k", 2048, (1, 128, 128, 0)), ("k", 1024, (2, 128, 128, 0)),
    ("q", 512, (1, 128, 128, 0)), ("gate", 256, (1, 128, 128, 0)),
    ("o", 256, (2, 128, 128, 0)),
    # narrow tiles that would not fit one wave (160 > 152), or a full wave: wide
    ("o", 1024, (1, 256, 128, 0)), ("gate", 2048, (1, 256, 128, 0)),
    ("q", 2048, (1, 256, 128, 0)),
    # the long reduction of down: twice the dequant per multiply-add costs
    # more than the planes and the reduce launch the narrow tile saves
    ("down", 512, (2, 256, 128, 0)), ("down", 129, (4, 256, 128, 0)),
])
def test_balanced_plan_narrow_tile(name, M, want):
    Kred, Nout = inputs.PROJECTIONS[name]
    got = Q.qmm_call_plan(M, Kred, Nout, Q.QMM_SPLIT_BALANCED, num_sms=152, with_head=True)
    assert got == want


# ---- binding argument checks (no device needed) ---------------------------------

def _host_args(M=4, Kred=256, Nout=16):
    return (torch.zeros((M, Kred), dtype=torch.bfloat16),
            torch.zeros((Nout, Kred // 8), dtype=torch.int32),
            torch.zeros((Nout, Kred // 128), dtype=torch.bfloat16),
            torch.zeros((Nout, Kred // 128), dtype=torch.bfloat16),
            torch.zeros((M, Nout), dtype=torch.bfloat16))


@pytest.mark.parametrize("fn", [Q.qmm_w4a16_g128, Q.qmm_w4a16_g128_noalloc])
def test_binding_rejects_host_and_mistyped_tensors(fn):
    """The per-call entry points check every tensor before the library is
    called: a host tensor, a wrong dtype, a non-contiguous view and
    inconsistent shapes are named errors, not a launch."""
    A, Wq, s, b, C = _host_args()
    with pytest.raises(TypeError, match="A must be a CUDA tensor"):
        fn(A, Wq, s, b, C)
    with pytest.raises(ValueError, match="inconsistent shapes"):
        fn(A, Wq, s[:8], b, C)
    with pytest.raises(ValueError, match="inconsistent shapes"):
        fn(A, Wq, s, b, C[:, :8])


def test_binding_pointer_check_reports_the_failed_condition():
    # the one-expression check falls back to the detailed one for its message
    A = torch.zeros((4, 8), dtype=torch.float32)
    with pytest.raises(TypeError, match="x must be a CUDA tensor"):
        Q._ptr(A, (torch.bfloat16,), "x")
    with pytest.raises(TypeError, match="y must be a CUDA tensor"):
        Q._ptr(object(), (torch.bfloat16,), "y")
