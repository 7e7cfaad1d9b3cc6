"""Allocation-free entry point: qmm_w4a16_g128_noalloc keeps the split-K
partial planes in the library's fixed device buffer.

Two consecutive calls of different shapes and splits reuse the same buffer.
Each must equal qmm_w4a16_g128 with a caller workspace bit for bit, because
the kernels, split and partial dtype are the same.  A call whose planes
exceed the buffer must be refused before anything is launched.  This file is
collected last so that it runs both alone and after every other GPU test.
"""
import numpy as np
import pytest
import torch

from split_w4a16_quantized_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def Q():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from split_w4a16_quantized_gb300 import build, qmm
    build.build()
    return qmm


def _problem(Q, M, Kred, Nout, seed):
    return Q.to_device(inputs.make_w4a16(M, Kred, Nout, seed=seed))


def _with_workspace(Q, d, split, partial_dtype):
    M, Nout = d["A"].shape[0], d["Wq"].shape[0]
    C = torch.empty((M, Nout), dtype=torch.bfloat16, device=d["A"].device)
    nbytes = Q.qmm_splitk_workspace_bytes(M, Nout, split, partial_dtype)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=d["A"].device)
    used = Q.qmm_w4a16_g128(d["A"], d["Wq"], d["scales"], d["biases"], C, split_req=split,
                            workspace=ws, partial_dtype=partial_dtype)
    return C, used


def _no_alloc(Q, d, split_req, partial_dtype):
    M, Nout = d["A"].shape[0], d["Wq"].shape[0]
    C = torch.full((M, Nout), float("nan"), dtype=torch.bfloat16, device=d["A"].device)
    used = Q.qmm_w4a16_g128_noalloc(d["A"], d["Wq"], d["scales"], d["biases"], C,
                                    split_req=split_req, partial_dtype=partial_dtype)
    return C, used


def _bits(C):
    return C.view(torch.int16).cpu().numpy()


def test_scratch_size(Q):
    assert Q.qmm_static_scratch_bytes() == 8 << 20


@pytest.mark.parametrize("partial_dtype", ["bf16", "f32"])
def test_two_consecutive_calls_match_workspace_path(Q, partial_dtype):
    pd = Q.QMM_PARTIAL_BF16 if partial_dtype == "bf16" else Q.QMM_PARTIAL_F32
    # k projection at M = 128 (policy split, 10 planes) then gate at M = 32
    # (2 planes, another plane size): the second call overwrites the first's
    # planes in the shared buffer
    d1 = _problem(Q, 128, 2560, 1024, seed=11)
    d2 = _problem(Q, 32, 2560, 9728, seed=12)
    C1, s1 = _no_alloc(Q, d1, 0, pd)
    C2, s2 = _no_alloc(Q, d2, 0, pd)
    torch.cuda.synchronize()
    assert s1 > 1 and s2 > 1
    assert Q.qmm_splitk_workspace_bytes(128, 1024, s1, pd) <= Q.qmm_static_scratch_bytes()
    R1, r1 = _with_workspace(Q, d1, s1, pd)
    R2, r2 = _with_workspace(Q, d2, s2, pd)
    torch.cuda.synchronize()
    assert (r1, r2) == (s1, s2)
    assert Q.qmm_kernel_status(clear=True) == 0
    np.testing.assert_array_equal(_bits(C1), _bits(R1))
    np.testing.assert_array_equal(_bits(C2), _bits(R2))


def test_forced_split_and_unsplit(Q):
    d = _problem(Q, 64, 4096, 2560, seed=13)
    C4, s4 = _no_alloc(Q, d, 4, Q.QMM_PARTIAL_BF16)
    C1, s1 = _no_alloc(Q, d, 1, Q.QMM_PARTIAL_BF16)
    R4, _ = _with_workspace(Q, d, 4, Q.QMM_PARTIAL_BF16)
    R1, _ = _with_workspace(Q, d, 1, Q.QMM_PARTIAL_BF16)
    torch.cuda.synchronize()
    assert (s4, s1) == (4, 1)
    np.testing.assert_array_equal(_bits(C4), _bits(R4))
    np.testing.assert_array_equal(_bits(C1), _bits(R1))


def test_planes_beyond_the_buffer_are_refused(Q):
    # M = 2048, Nout = 1024, split 4 with BF16 partials: 16 MiB of planes
    d = _problem(Q, 2048, 2560, 1024, seed=14)
    assert Q.qmm_splitk_workspace_bytes(2048, 1024, 4, Q.QMM_PARTIAL_BF16) > \
        Q.qmm_static_scratch_bytes()
    C = torch.full((2048, 1024), 7.0, dtype=torch.bfloat16, device=d["A"].device)
    with pytest.raises(Q.QmmError) as e:
        Q.qmm_w4a16_g128_noalloc(d["A"], d["Wq"], d["scales"], d["biases"], C, split_req=4)
    assert e.value.code == Q.QMM_EWORKSPACE
    torch.cuda.synchronize()
    assert bool((C == 7.0).all())  # nothing was launched
    # a forced split that does not divide G is a shape error, as in qmm_w4a16_g128
    with pytest.raises(Q.QmmError) as e:
        Q.qmm_w4a16_g128_noalloc(d["A"], d["Wq"], d["scales"], d["biases"], C, split_req=3)
    assert e.value.code == Q.QMM_ESHAPE


def test_planned_split_matches_workspace_path(Q):
    # QMM_SPLIT_PLANNED resolves to the group plan's split for the call alone,
    # as qmm_w4a16_g128 resolves it; the planes then go to the fixed buffer
    d = _problem(Q, 128, 9728, 2560, seed=15)
    C = torch.full((128, 2560), float("nan"), dtype=torch.bfloat16, device=d["A"].device)
    used = Q.qmm_w4a16_g128_noalloc(d["A"], d["Wq"], d["scales"], d["biases"], C,
                                    split_req=Q.QMM_SPLIT_PLANNED)
    nbytes = Q.qmm_splitk_workspace_bytes(128, 2560, max(used, 1), Q.QMM_PARTIAL_BF16)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=d["A"].device)
    R = torch.empty_like(C)
    ref = Q.qmm_w4a16_g128(d["A"], d["Wq"], d["scales"], d["biases"], R,
                           split_req=Q.QMM_SPLIT_PLANNED, workspace=ws)
    torch.cuda.synchronize()
    assert used == ref == Q.qmm_group_plan([(128, 9728, 2560)])[0]
    np.testing.assert_array_equal(_bits(C), _bits(R))
