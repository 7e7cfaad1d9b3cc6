"""CPU oracle for the split-K W4A16-g128 projection matmul (test infrastructure).

Only the tests, the smoke check and the bench's CPU-baseline leg use this
package; the library under ``split_w4a16_quantized_gb300`` never imports it and
shares no code with it.  The arithmetic lives in ``qmm_oracle.c`` (plain C,
fp64); this module compiles it with gcc and wraps it with ctypes.  The one
exception is the group plan (``group_plan``), the grouped call's opt-in split
rule, which is restated here in plain Python.

Sources the oracle follows (cited per function in the C file):
  * tiny-llm book, "Week 2 Day 7: Split-K Prefill" (Tasks 2-4)
  * gpu-kernels-explained, "Split-K, streams and overlap" (Concept sections;
    Maths, Overlap and Split-K; A100 table)
  * "Optimize Prefill vs Decode Kernels" (Required reasoning process, steps 4
    and 5; Correctness requirements: the split-KV log-sum-exp merge)

Parity pins: every function here is checked by ``tests/test_oracle.py``
against values the pages print, closed forms, exact rational brute force on
tiny shapes and library routines; none is "parity unpinned".  The group plan
is this library's rule, not the pages', so no printed value exists for it.
Its pins are list-schedule outcomes derived by hand (the wave tail of down at
M = 2048), agreement with the chapter's independently implemented policy on
single under-filled calls, and invariants (every kept move lowers the
estimate; splits stay valid).
"""
from __future__ import annotations

import ctypes
import heapq
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmm_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libqmm_oracle.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off keeps every a*b+c a separately rounded multiply and add on
# both x86-64 and aarch64, so the oracle gives the same bits on both hosts.
_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, OpenMP when available).  Returns the .so path."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    base = ["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        sig = {
            "oracle_bf16_round": [P, I64, P],
            "oracle_bf16_value": [P, I64, P],
            "oracle_unpack": [P, I64, I64, P],
            "oracle_dequant": [P, P, P, I64, I64, P],
            "oracle_qmm": [P, P, P, P, I64, I64, I64, P, I],
            "oracle_qmm_sampled": [P, P, P, P, I64, I64, I64, P, I64, P, I64, P, I],
            "oracle_qmm_partitioned": [P, P, P, P, I64, I64, I64, I, I, P, P, I],
            "oracle_qmm_partitioned_sampled": [P, P, P, P, I64, I64, I64, P, I64, P, I64, I, I,
                                               P, P, I],
            "oracle_splitk_plan": [I64, I64, I64, I64, I64, I64, I64, I64, P],
            "oracle_splitk_plan_near_equal": [I64, I64, I64, I64, I64, I64, I64, I64, P],
            "oracle_waves": [I64, I64, I64],
            "oracle_overlap_schedule": [I64, I64, P, P, P, I, P, P],
            "oracle_decode_attention": [P, P, P, P, I64, I64, I64, I64, I64, ctypes.c_double, P,
                                        I],
            "oracle_decode_attention_split": [P, P, P, P, I64, I64, I64, I64, I64,
                                              ctypes.c_double, I64, I, P, I],
            "oracle_attention_splits": [I64, I64, I64, I64, I64, I64, P],
            "oracle_gemm": [P, P, I64, I64, I64, P, I],
            "oracle_gemm_partitioned": [P, P, I64, I64, I64, I64, I, P, I],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = I64 if name == "oracle_waves" else I
        _lib = lib
        return lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def _check(rc, what):
    if rc != 0:
        raise ValueError("%s failed (%d)" % (what, rc))


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- number formats ------------------------------------------------------

def bf16_round(x) -> np.ndarray:
    """Round float64 values to BF16 (nearest, ties to even); returns bits."""
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    _check(_load().oracle_bf16_round(_ptr(x), x.size, _ptr(out)), "bf16_round")
    return out


def bf16_value(b) -> np.ndarray:
    """BF16 bits -> float64 (exact)."""
    b = _c(b, np.uint16)
    out = np.empty(b.shape, np.float64)
    _load().oracle_bf16_value(_ptr(b), b.size, _ptr(out))
    return out


# ---- W4A16-g128 ----------------------------------------------------------

def unpack(Wq, Kred: int) -> np.ndarray:
    Wq = _c(Wq, np.uint32)
    nout = Wq.shape[0]
    q = np.empty((nout, Kred), np.uint8)
    _check(_load().oracle_unpack(_ptr(Wq), nout, Kred, _ptr(q)), "unpack")
    return q


def dequant(Wq, scales, biases, Kred: int) -> np.ndarray:
    """BF16 bits of w[n,k] = BF16(scale*q + bias) [Nout, Kred]."""
    Wq, scales, biases = _c(Wq, np.uint32), _c(scales, np.uint16), _c(biases, np.uint16)
    nout = Wq.shape[0]
    w = np.empty((nout, Kred), np.uint16)
    _check(_load().oracle_dequant(_ptr(Wq), _ptr(scales), _ptr(biases), nout, Kred, _ptr(w)),
           "dequant")
    return w


def qmm(A, Wq, scales, biases, threads: int | None = None) -> np.ndarray:
    """fp64 C = A @ W^T [M, Nout]."""
    A, Wq = _c(A, np.uint16), _c(Wq, np.uint32)
    scales, biases = _c(scales, np.uint16), _c(biases, np.uint16)
    M, Kred = A.shape
    nout = Wq.shape[0]
    C = np.empty((M, nout), np.float64)
    _check(_load().oracle_qmm(_ptr(A), _ptr(Wq), _ptr(scales), _ptr(biases), M, Kred, nout,
                              _ptr(C), threads or default_threads()), "qmm")
    return C


def qmm_sampled(A, Wq, scales, biases, rows, cols, threads: int | None = None) -> np.ndarray:
    """fp64 C[rows][:, cols] computed element by element."""
    A, Wq = _c(A, np.uint16), _c(Wq, np.uint32)
    scales, biases = _c(scales, np.uint16), _c(biases, np.uint16)
    rows, cols = _c(rows, np.int64), _c(cols, np.int64)
    M, Kred = A.shape
    nout = Wq.shape[0]
    out = np.empty((rows.size, cols.size), np.float64)
    _check(_load().oracle_qmm_sampled(_ptr(A), _ptr(Wq), _ptr(scales), _ptr(biases), M, Kred,
                                      nout, _ptr(rows), rows.size, _ptr(cols), cols.size,
                                      _ptr(out), threads or default_threads()), "qmm_sampled")
    return out


def qmm_partitioned(A, Wq, scales, biases, split: int, partial_mode: int = 0,
                    with_partials: bool = False, threads: int | None = None):
    """Partition emulation: returns (C bf16 bits [M,Nout], partial planes or None).
    A split that does not divide Kred/128 takes near-equal partitions (the first
    G mod split ones hold one group more)."""
    A, Wq = _c(A, np.uint16), _c(Wq, np.uint32)
    scales, biases = _c(scales, np.uint16), _c(biases, np.uint16)
    M, Kred = A.shape
    nout = Wq.shape[0]
    C = np.empty((M, nout), np.uint16)
    P = np.empty((split, M, nout), np.float64) if with_partials else None
    _check(_load().oracle_qmm_partitioned(
        _ptr(A), _ptr(Wq), _ptr(scales), _ptr(biases), M, Kred, nout, split, partial_mode,
        _ptr(C), _ptr(P) if P is not None else None, threads or default_threads()),
        "qmm_partitioned")
    return C, P


def qmm_partitioned_sampled(A, Wq, scales, biases, rows, cols, split: int,
                            partial_mode: int = 0, with_partials: bool = False,
                            threads: int | None = None):
    """Partition emulation at sampled elements: BF16 bits [len(rows), len(cols)],
    and with_partials the plane values [len(rows), len(cols), split]."""
    A, Wq = _c(A, np.uint16), _c(Wq, np.uint32)
    scales, biases = _c(scales, np.uint16), _c(biases, np.uint16)
    rows, cols = _c(rows, np.int64), _c(cols, np.int64)
    M, Kred = A.shape
    nout = Wq.shape[0]
    out = np.empty((rows.size, cols.size), np.uint16)
    planes = np.empty((rows.size, cols.size, split), np.float64) if with_partials else None
    _check(_load().oracle_qmm_partitioned_sampled(
        _ptr(A), _ptr(Wq), _ptr(scales), _ptr(biases), M, Kred, nout, _ptr(rows), rows.size,
        _ptr(cols), cols.size, split, partial_mode, _ptr(out),
        _ptr(planes) if planes is not None else None, threads or default_threads()),
        "qmm_partitioned_sampled")
    return (out, planes) if with_partials else out


def splitk_plan(M, Kred, Nout, bm, bn, target, cap, min_k=128) -> int:
    s = ctypes.c_int(0)
    _check(_load().oracle_splitk_plan(M, Kred, Nout, bm, bn, target, cap, min_k,
                                      ctypes.byref(s)), "splitk_plan")
    return s.value


def splitk_plan_near_equal(M, Kred, Nout, bm, bn, target, cap, min_k=128) -> int:
    """The plan for near-equal partitions: the fewest partitions that reach the
    shortest longest partition within the policy's bounds."""
    s = ctypes.c_int(0)
    _check(_load().oracle_splitk_plan_near_equal(M, Kred, Nout, bm, bn, target, cap, min_k,
                                                 ctypes.byref(s)), "splitk_plan_near_equal")
    return s.value


def waves(tiles, split, sms) -> int:
    r = _load().oracle_waves(tiles, split, sms)
    if r < 0:
        raise ValueError("waves: bad arguments")
    return int(r)


def overlap_schedule(n, buffers, t_load, t_comp, t_store, out_reuse=False,
                     with_events=False):
    """Finish time of n tiles through copy-in, compute and copy-out engines with
    `buffers` buffers; times are scalars (every tile alike) or length-n arrays.
    with_events also returns the [n, 6] start/end times."""
    t = [np.ascontiguousarray(np.broadcast_to(np.asarray(x, np.float64), (n,)))
         for x in (t_load, t_comp, t_store)]
    T = ctypes.c_double(0.0)
    ev = np.empty((n, 6), np.float64) if with_events else None
    _check(_load().oracle_overlap_schedule(n, buffers, _ptr(t[0]), _ptr(t[1]), _ptr(t[2]),
                                           int(bool(out_reuse)), ctypes.byref(T),
                                           _ptr(ev) if ev is not None else None),
           "overlap_schedule")
    return (T.value, ev) if with_events else T.value


# ---- split-KV decode attention -----------------------------------------------

def _attn_args(q, K, V, lens):
    q, K, V = _c(q, np.uint16), _c(K, np.uint16), _c(V, np.uint16)
    lens = _c(lens, np.int32)
    B, Hq, D = q.shape
    _, Hkv, Lmax, _ = K.shape
    assert K.shape == V.shape == (B, Hkv, Lmax, D) and lens.shape == (B,)
    return q, K, V, lens, B, Hq, Hkv, Lmax, D


def decode_attention(q, K, V, lens, scale=None, threads: int | None = None) -> np.ndarray:
    """fp64 O [B, Hq, D] of one query token per sequence over its KV history
    (K, V BF16 bits [B, Hkv, Lmax, D]; lens [B]); scale defaults to 1/sqrt(D)."""
    q, K, V, lens, B, Hq, Hkv, Lmax, D = _attn_args(q, K, V, lens)
    O = np.empty((B, Hq, D), np.float64)
    sc = 1.0 / np.sqrt(D) if scale is None else float(scale)
    _check(_load().oracle_decode_attention(_ptr(q), _ptr(K), _ptr(V), _ptr(lens), B, Hq, Hkv,
                                           Lmax, D, sc, _ptr(O), threads or default_threads()),
           "decode_attention")
    return O


def decode_attention_split(q, K, V, lens, chunk: int, merge: str = "lse", scale=None,
                           threads: int | None = None) -> np.ndarray:
    """The split-KV algorithm in fp64: chunks of `chunk` positions merged with
    the log-sum-exp correction (merge="lse") or naively ("naive")."""
    q, K, V, lens, B, Hq, Hkv, Lmax, D = _attn_args(q, K, V, lens)
    O = np.empty((B, Hq, D), np.float64)
    sc = 1.0 / np.sqrt(D) if scale is None else float(scale)
    _check(_load().oracle_decode_attention_split(
        _ptr(q), _ptr(K), _ptr(V), _ptr(lens), B, Hq, Hkv, Lmax, D, sc, chunk,
        {"lse": 0, "naive": 1}[merge], _ptr(O), threads or default_threads()),
        "decode_attention_split")
    return O


def attention_splits(B, Hkv, Lmax, sms, blocks_per_sm, min_chunk) -> int:
    s = ctypes.c_int(0)
    _check(_load().oracle_attention_splits(B, Hkv, Lmax, sms, blocks_per_sm, min_chunk,
                                           ctypes.byref(s)), "attention_splits")
    return s.value


# ---- dense BF16 GEMM -----------------------------------------------------

def gemm(A, W, threads: int | None = None) -> np.ndarray:
    A, W = _c(A, np.uint16), _c(W, np.uint16)
    M, K = A.shape
    N = W.shape[0]
    C = np.empty((M, N), np.float64)
    _check(_load().oracle_gemm(_ptr(A), _ptr(W), M, N, K, _ptr(C),
                               threads or default_threads()), "gemm")
    return C


def gemm_partitioned(A, W, split: int, ktile: int = 64, threads: int | None = None):
    A, W = _c(A, np.uint16), _c(W, np.uint16)
    M, K = A.shape
    N = W.shape[0]
    C = np.empty((M, N), np.uint16)
    _check(_load().oracle_gemm_partitioned(_ptr(A), _ptr(W), M, N, K, ktile, split, _ptr(C),
                                           threads or default_threads()), "gemm_partitioned")
    return C


# ---- group plan ---------------------------------------------------------------
#
# The grouped call's opt-in split plan.  The pages motivate it: split-K only
# pays while SMs would otherwise idle (gpu-kernels-explained, "Split-K, streams
# and overlap", the wave model).  The cost model and its constants are this
# library's own, and the oracle restates them as the rule's definition.

GROUP_PLAN_TILE_US = 3.0           # fixed cost of one CTA tile
GROUP_PLAN_PLANE_BYTES_PER_US = 3.0e6


def group_plan_group_us(bm: int) -> float:
    """Time of one 128-group of a tile, by tile width (activation rows)."""
    if bm <= 32:
        return 0.40
    if bm <= 64:
        return 0.45
    if bm <= 128:
        return 0.55
    return 0.60


def group_plan_cost(shapes, tiles, splits, bm, sms, partial_bytes=2):
    """Estimated time (us) of one launch: the CTA tiles of every call, longest
    first, each placed on the SM that frees first, plus the partial planes
    written and read back."""
    durations = []
    planes = 0.0
    for (M, Kred, Nout), t, s in zip(shapes, tiles, splits):
        G = Kred // 128
        longest = -(-G // s)
        durations.append((GROUP_PLAN_TILE_US + longest * group_plan_group_us(bm), t * s))
        if s > 1:
            planes += float(s) * M * Nout * 2 * partial_bytes / GROUP_PLAN_PLANE_BYTES_PER_US
    durations.sort(key=lambda x: -x[0])  # stable: equal durations keep call order
    free = [0.0] * sms
    heapq.heapify(free)
    span = 0.0
    for d, count in durations:
        for _ in range(count):
            t = heapq.heappop(free) + d
            heapq.heappush(free, t)
            span = max(span, t)
    return span + planes


def group_plan(shapes, tiles_of, sms, near_equal=False, partial_bytes=2, cap=16,
               decode_max_m=8, decode_min_k=512, trace=None, own_launch=None):
    """Splits for calls of shapes [(M, Kred, Nout)], where tiles_of(M) gives
    the (bm, bn) tile of the kernel that serves M.  The calls of one tile width
    share a launch.  Per launch, every call starts unsplit.  Then, repeatedly,
    the call with the longest partition (lowest index on ties) moves to its
    next valid split.  The move is kept only if it lowers group_plan_cost, and
    the descent ends at the first move that does not, or when that call has no
    larger valid split.  Valid splits follow the chapter's single-call rule: at
    most cap and G, at least decode_min_k reduction elements per partition for
    M <= decode_max_m, and dividing G unless near_equal.  trace, if a list,
    receives (splits, cost) after every kept move, per launch.  (The library
    also makes no move that takes a launch over 65536 tiles.)

    own_launch(M), if given, returns None for a call that shares its tile
    width's launch, or the policy (bm, bn, target, cap, min_k) of a call that
    runs in a launch of its own: such a call is not planned with the others
    and keeps the chapter's single-call split under that policy (the
    near-equal plan when near_equal)."""
    splits = [1] * len(shapes)
    widths = []
    for M, _, _ in shapes:
        if tiles_of(M)[0] not in widths:
            widths.append(tiles_of(M)[0])
    for bm in widths:
        idx = [i for i, (M, _, _) in enumerate(shapes) if tiles_of(M)[0] == bm]
        if own_launch is not None and own_launch(shapes[idx[0]][0]) is not None:
            plan = splitk_plan_near_equal if near_equal else splitk_plan
            for i in idx:
                M, Kred, Nout = shapes[i]
                pbm, pbn, target, pcap, min_k = own_launch(M)
                splits[i] = plan(M, Kred, Nout, pbm, pbn, target, pcap, min_k)
            continue
        part = [shapes[i] for i in idx]
        tiles = []
        for M, Kred, Nout in part:
            tbm, tbn = tiles_of(M)
            tiles.append(-(-M // tbm) * -(-Nout // tbn))
        s = [1] * len(part)
        cost = group_plan_cost(part, tiles, s, bm, sms, partial_bytes)
        if trace is not None:
            trace.append((list(s), cost))
        while True:
            lengths = [-(-(K // 128) // si) for (_, K, _), si in zip(part, s)]
            top = lengths.index(max(lengths))
            M, Kred, _ = part[top]
            G = Kred // 128
            min_k = decode_min_k if M <= decode_max_m else 128
            smax = min(cap, G, max(1, Kred // min_k))
            nxt = next((v for v in range(s[top] + 1, smax + 1) if near_equal or G % v == 0), None)
            if nxt is None:
                break
            t = list(s)
            t[top] = nxt
            c2 = group_plan_cost(part, tiles, t, bm, sms, partial_bytes)
            if not c2 < cost:
                break
            s, cost = t, c2
            if trace is not None:
                trace.append((list(s), cost))
        for i, v in zip(idx, s):
            splits[i] = v
    return splits
