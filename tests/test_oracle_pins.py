"""Pins for the CPU oracle: closed forms, invariants, brute force, library
special cases and hand-worked fixtures.  None of these retypes the oracle's
own formula; each is chosen so that a plausible slip in the oracle (a dropped
stage, a swapped index, a transposed operand, a wrong sign) fails at least one.
"""
import json
import math
import os

import numpy as np
import pytest
from scipy.special import expit, softmax

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(20261202)


def rand_case(rows, cols, zero_stages=()):
    codes = rng.integers(0, 256, size=(rows, cols // 8, 3), dtype=np.uint8)
    cb = rng.normal(0, 1, size=(3, 256, 8)).astype(np.float32)
    for s in zero_stages:
        cb[s] = 0
    return codes, cb


# ------------------------------------------------------------ RVQ decode

def test_golden_tiny_example():
    g = json.load(open(os.path.join(GOLDEN, "rvq_tiny.json")))
    cb = np.zeros((3, 256, 8), np.float32)
    cb[0, 3] = g["codebook_nonzero"]["stage0_entry3"]
    cb[1, 5] = g["codebook_nonzero"]["stage1_entry5"]
    cb[2, 7] = g["codebook_nonzero"]["stage2_entry7"]
    codes = np.array(g["codes_row_chunk_stage"], np.uint8)
    x = np.array(g["x"], np.float64)
    y = oracle.rvq_gemv(codes, cb, g["rows"], g["cols"], x)[0]
    assert y.tolist() == g["y"]
    lut = oracle.rvq_lut_build(cb, x, g["cols"])
    for j, s, k, v in g["lut_entries_chunk_stage_entry_value"]:
        assert lut[j, s, k] == v
    assert oracle.rvq_lut_gemv(codes, lut, g["rows"], g["cols"]).tolist() == g["y"]


@pytest.mark.parametrize("rows,cols", [(1, 8), (3, 16), (16, 64), (7, 40)])
def test_lut_formulation_equals_explicit_dequant(rows, cols):
    """Brute force: explicit decode + dot product == sum of table lookups."""
    codes, cb = rand_case(rows, cols)
    x = rng.normal(size=cols)
    y_def = oracle.rvq_gemv(codes, cb, rows, cols, x)[0]
    y_lut = oracle.rvq_lut_gemv(codes, oracle.rvq_lut_build(cb, x, cols), rows, cols)
    np.testing.assert_allclose(y_lut, y_def, rtol=1e-12, atol=1e-12 * np.abs(y_def).max())


def test_zeroed_later_stages_is_single_stage_vq():
    """With stage-2/3 codebooks zero, the stage-2/3 codes cannot matter and the
    result is bit-identical whatever they are."""
    rows, cols = 32, 64
    codes, cb = rand_case(rows, cols, zero_stages=(1, 2))
    x = rng.normal(size=cols)
    y1 = oracle.rvq_gemv(codes, cb, rows, cols, x)
    codes2 = codes.copy()
    codes2[:, :, 1:] = rng.integers(0, 256, size=codes2[:, :, 1:].shape)
    y2 = oracle.rvq_gemv(codes2, cb, rows, cols, x)
    assert np.array_equal(y1, y2)


def test_single_chunk_single_stage_is_matmul():
    """cols = 8, row r coded by stage-1 entry r, other stages zero: the matrix
    is the stage-1 codebook itself, so y = C1 @ x (numpy matmul)."""
    codes = np.zeros((256, 1, 3), np.uint8)
    codes[:, 0, 0] = np.arange(256)
    codes[:, 0, 1:] = rng.integers(0, 256, size=(256, 2))
    cb = np.zeros((3, 256, 8), np.float32)
    cb[0] = rng.normal(size=(256, 8))
    x = rng.normal(size=(3, 8))
    y = oracle.rvq_gemv(codes, cb, 256, 8, x)
    np.testing.assert_allclose(y, x @ cb[0].astype(np.float64).T, rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(oracle.rvq_dequant(codes, cb, 256, 8), cb[0].astype(np.float64))


@pytest.mark.parametrize("stage", [0, 1, 2])
def test_closed_form_code_count(stage):
    """One-hot codebook: C_s[k*] = all ones, everything else zero, x = 1.
    Then y[r] = 8 * #{chunks j : code(r, j, s) == k*} exactly."""
    rows, cols, kstar = 24, 256, 17
    codes = rng.integers(0, 256, size=(rows, cols // 8, 3), dtype=np.uint8)
    codes[::3, ::2, stage] = kstar          # make matches frequent
    cb = np.zeros((3, 256, 8), np.float32)
    cb[stage, kstar] = 1.0
    y = oracle.rvq_gemv(codes, cb, rows, cols, np.ones(cols))[0]
    expect = 8 * (codes[:, :, stage] == kstar).sum(axis=1)
    assert np.array_equal(y, expect.astype(np.float64))


def test_decode_codes_back_from_one_hot_inputs():
    """C_s[k][i] = k * 256^s * 2^i (exact in fp32).  With x one-hot at column
    8j+i, y[r] / 2^i must spell code(r,j,0) + 256 code(r,j,1) + 65536 code(r,j,2):
    pins row/column orientation, chunk index, dimension index and stage order."""
    rows, cols = 16, 48
    codes = rng.integers(0, 256, size=(rows, cols // 8, 3), dtype=np.uint8)
    k = np.arange(256, dtype=np.float64)
    cb = np.empty((3, 256, 8), np.float32)
    for s in range(3):
        for i in range(8):
            cb[s, :, i] = k * 256.0 ** s * 2.0 ** i
    assert np.array_equal(cb.astype(np.float64)[2, :, 7], k * 65536 * 128)
    for col in [0, 5, 8, 19, 47]:
        x = np.zeros(cols)
        x[col] = 1.0
        y = oracle.rvq_gemv(codes, cb, rows, cols, x)[0]
        j, i = divmod(col, 8)
        v = (y / 2.0 ** i).astype(np.int64)
        assert np.array_equal(v.astype(np.float64) * 2.0 ** i, y)
        assert np.array_equal(v & 255, codes[:, j, 0])
        assert np.array_equal((v >> 8) & 255, codes[:, j, 1])
        assert np.array_equal(v >> 16, codes[:, j, 2])


def test_linearity_in_x():
    rows, cols = 20, 96
    codes, cb = rand_case(rows, cols)
    x1, x2 = rng.normal(size=cols), rng.normal(size=cols)
    a, b = 0.75, -2.5
    y = oracle.rvq_gemv(codes, cb, rows, cols, np.stack([x1, x2, a * x1 + b * x2]))
    np.testing.assert_allclose(y[2], a * y[0] + b * y[1], rtol=1e-12, atol=1e-12)


def test_codebook_relabelling_is_invisible():
    """Permuting each stage's codebook entries and relabelling the codes the
    same way gives a bit-identical result: codes act only as indices."""
    rows, cols = 16, 64
    codes, cb = rand_case(rows, cols)
    x = rng.normal(size=cols)
    cb2, codes2 = np.empty_like(cb), np.empty_like(codes)
    for s in range(3):
        perm = rng.permutation(256)
        cb2[s, perm] = cb[s]
        codes2[:, :, s] = perm[codes[:, :, s]]
    assert np.array_equal(oracle.rvq_gemv(codes, cb, rows, cols, x),
                          oracle.rvq_gemv(codes2, cb2, rows, cols, x))


def test_stage_swap_together_is_invisible():
    """Swapping stages 0 and 2 in both codes and codebooks changes only the
    addition order: a stage-index mismatch between codes and codebooks fails."""
    rows, cols = 16, 64
    codes, cb = rand_case(rows, cols)
    x = rng.normal(size=cols)
    y = oracle.rvq_gemv(codes, cb, rows, cols, x)
    y2 = oracle.rvq_gemv(codes[:, :, ::-1], cb[::-1], rows, cols, x)
    np.testing.assert_allclose(y2, y, rtol=1e-14, atol=1e-14)
    # and swapping only the codes does change the result
    y3 = oracle.rvq_gemv(codes[:, :, ::-1], cb, rows, cols, x)
    assert not np.allclose(y3, y)


def test_every_code_byte_matters_and_only_those():
    """3 * rows * cols / 8 bytes: each one influences its own row only, and
    bytes after the array are never read."""
    rows, cols = 8, 32
    codes, cb = rand_case(rows, cols)
    x = rng.normal(size=cols)
    assert codes.nbytes == 3 * rows * cols // 8
    base = oracle.rvq_gemv(codes, cb, rows, cols, x)[0]
    for flat in range(codes.size):
        c2 = codes.copy().reshape(-1)
        c2[flat] ^= 0x5A
        y = oracle.rvq_gemv(c2.reshape(codes.shape), cb, rows, cols, x)[0]
        r = flat // (3 * cols // 8)
        diff = np.nonzero(y != base)[0]
        assert diff.tolist() == [r]
    # embed in a larger buffer with garbage after it: same result
    lib = oracle._load()
    big = np.concatenate([codes.reshape(-1), rng.integers(0, 256, 4096, dtype=np.uint8)])
    y = np.empty(rows)
    xs = np.ascontiguousarray(x)
    lib.oracle_rvq_gemv(big.ctypes.data, cb.ctypes.data, rows, cols, xs.ctypes.data, 1,
                        y.ctypes.data)
    assert np.array_equal(y, base)


# ---------------------------------------------------------------- router

def test_route_golden_ties():
    g = json.load(open(os.path.join(GOLDEN, "route_ties.json")))
    for case in g["cases"]:
        lg = np.array([case["logits"]], np.float32)
        idx, w, rc = oracle.route(lg, case["k"])
        assert rc == 0
        assert idx[0].tolist() == case["idx"]
        np.testing.assert_allclose(w[0], np.array(case["w"], np.float32), rtol=1e-7, atol=0)


def test_route_matches_full_sort_and_softmax():
    n, E, k = 64, 64, 8
    lg = rng.normal(size=(n, E)).astype(np.float32)
    lg[3, 10] = lg[3, 20] = lg[3].max() + 1  # a tie at the top
    lg[5, :] = np.round(lg[5, :])             # many ties
    idx, w, rc = oracle.route(lg, k)
    assert rc == 0
    for t in range(n):
        order = np.lexsort((np.arange(E), -lg[t].astype(np.float64)))
        assert idx[t].tolist() == order[:k].tolist()
        np.testing.assert_allclose(w[t], softmax(lg[t, order[:k]].astype(np.float64)),
                                   rtol=2e-7, atol=1e-9)
    np.testing.assert_allclose(w.astype(np.float64).sum(axis=1), 1.0, atol=1e-6)
    assert (np.diff(w, axis=1) <= 0).all()  # selection order is descending weight


def test_route_k_equals_E_is_full_softmax():
    n, E = 5, 16
    lg = rng.normal(size=(n, E)).astype(np.float32)
    idx, w, _ = oracle.route(lg, E)
    for t in range(n):
        assert sorted(idx[t].tolist()) == list(range(E))
        full = softmax(lg[t].astype(np.float64))
        np.testing.assert_allclose(w[t], full[idx[t]], rtol=2e-7, atol=1e-9)


def test_route_k1_is_argmax_and_shift_invariant():
    lg = rng.normal(size=(40, 32)).astype(np.float32)
    idx, w, _ = oracle.route(lg, 1)
    assert idx[:, 0].tolist() == np.argmax(lg, axis=1).tolist()
    assert (w == 1.0).all()
    idx2, w2, _ = oracle.route(lg + np.float32(8.0), 4)
    idx3, w3, _ = oracle.route(lg, 4)
    assert np.array_equal(idx2, idx3)
    np.testing.assert_allclose(w2, w3, rtol=1e-5)


def test_route_flags_non_finite():
    lg = np.zeros((2, 8), np.float32)
    lg[1, 3] = np.nan
    assert oracle.route(lg, 2)[2] == -1
    lg[1, 3] = np.inf
    assert oracle.route(lg, 2)[2] == -1


# -------------------------------------------------------------- grouping

def test_group_golden():
    g = json.load(open(os.path.join(GOLDEN, "group_tiny.json")))
    offsets, pairs = oracle.group(np.array(g["topk_idx"], np.int32), g["E"])
    assert offsets.tolist() == g["offsets"]
    assert pairs.tolist() == g["pairs"]


@pytest.mark.parametrize("n,E,k", [(1, 64, 8), (37, 64, 8), (300, 256, 16)])
def test_group_invariants(n, E, k):
    """The invariants fix the output uniquely: every (token, slot) once, in
    its expert's segment, segments in expert order, tokens ascending."""
    lg = rng.normal(size=(n, E)).astype(np.float32)
    idx, _, _ = oracle.route(lg, k)
    offsets, pairs = oracle.group(idx, E)
    assert offsets[0] == 0 and offsets[-1] == n * k
    assert (np.diff(offsets) >= 0).all()
    assert sorted(pairs.tolist()) == list(range(n * k))
    flat = idx.reshape(-1)
    for e in range(E):
        seg = pairs[offsets[e]:offsets[e + 1]]
        assert (flat[seg] == e).all()
        assert (np.diff(seg // k) > 0).all()
        assert len(seg) == (flat == e).sum()


# ------------------------------------------------------------ expert FFN

def test_swiglu_values():
    assert oracle.swiglu(0.0, 5.0) == 0.0
    for g in [-30.0, -2.0, -0.5, 0.25, 3.0, 40.0]:
        assert math.isclose(oracle.swiglu(g, 1.5), g * expit(g) * 1.5, rel_tol=1e-15)
    v = oracle.swiglu(-1000.0, 1.0)
    assert v == 0.0 and math.copysign(1.0, v) == -1.0
    assert oracle.swiglu(1000.0, 2.0) == 2000.0


def _ffn_case(d, f):
    gate = rand_case(f, d)
    up = rand_case(f, d)
    down = rand_case(d, f)
    return gate, up, down


def test_ffn_is_down_of_swiglu_of_gate_up():
    """Composition check with library routines on the (pinned) dense decode."""
    d, f = 32, 16
    gate, up, down = _ffn_case(d, f)
    x = rng.normal(size=d) * 0.1
    Wg = oracle.rvq_dequant(*gate, f, d)
    Wu = oracle.rvq_dequant(*up, f, d)
    Wd = oracle.rvq_dequant(*down, d, f)
    g, u = Wg @ x, Wu @ x
    expect = Wd @ (g * expit(g) * u)
    y, h = oracle.expert_ffn(gate, up, down, d, f, x, want_h=True)
    np.testing.assert_allclose(h, g * expit(g) * u, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(y, expect, rtol=1e-11, atol=1e-12 * np.abs(expect).max())
    # gate and up are not interchangeable: swapping them changes the output
    y_sw = oracle.expert_ffn(up, gate, down, d, f, x)
    assert not np.allclose(y_sw, y)


def test_ffn_zero_up_or_gate_gives_zero():
    d, f = 16, 8
    gate, up, down = _ffn_case(d, f)
    x = rng.normal(size=d)
    up0 = (up[0], np.zeros_like(up[1]))
    gate0 = (gate[0], np.zeros_like(gate[1]))
    assert (oracle.expert_ffn(gate, up0, down, d, f, x) == 0).all()
    assert (oracle.expert_ffn(gate0, up, down, d, f, x) == 0).all()


# --------------------------------------------------------------- combine

def test_combine_zero_weights_is_residual_and_matches_einsum():
    n, k, d = 4, 3, 16
    y = rng.normal(size=(n * k, d))
    res = rng.normal(size=(n, d))
    assert np.array_equal(oracle.combine(y, np.zeros((n, k), np.float32), res), res)
    w = rng.random((n, k)).astype(np.float32)
    out = oracle.combine(y, w, res)
    expect = res + np.einsum("tk,tkd->td", w.astype(np.float64), y.reshape(n, k, d))
    np.testing.assert_allclose(out, expect, rtol=1e-14, atol=1e-14)
    one = np.zeros((n, k), np.float32)
    one[:, 1] = 1.0
    assert np.array_equal(oracle.combine(y, one, res), res + y.reshape(n, k, d)[:, 1])


def test_moe_layer_is_composition_of_steps():
    n, E, k, d, f = 3, 8, 2, 16, 8
    experts = {e: _ffn_case(d, f) for e in range(E)}
    wr = rng.normal(size=(E, d)).astype(np.float32)
    x = rng.normal(size=(n, d))
    r = oracle.moe_layer(lambda e: experts[e], wr, x, k, d, f)
    lg = oracle.router_logits(wr, x)
    np.testing.assert_allclose(lg, x @ wr.astype(np.float64).T, rtol=1e-13, atol=1e-13)
    idx, w, _ = oracle.route(lg.astype(np.float32), k)
    assert np.array_equal(r["idx"], idx) and np.array_equal(r["w"], w)
    y = np.stack([oracle.expert_ffn(*experts[int(idx[t, s])], d, f, x[t])
                  for t in range(n) for s in range(k)])
    assert np.array_equal(r["y_pair"], y)
    assert np.array_equal(r["out"], oracle.combine(y, w, x))


def test_router_bias_is_added():
    E, d = 6, 16
    wr = rng.normal(size=(E, d)).astype(np.float32)
    b = rng.normal(size=E).astype(np.float32)
    x = rng.normal(size=(2, d))
    np.testing.assert_allclose(oracle.router_logits(wr, x, b) - oracle.router_logits(wr, x),
                               np.broadcast_to(b.astype(np.float64), (2, E)), atol=1e-13)


# ------------------------------------------------------------ rms norm (stack)

def test_rms_norm_closed_forms():
    """Constant rows map to +-1/sqrt(1 + eps/c^2); a row of +-a values has unit
    RMS after the norm; a one-hot row scales to sqrt(d) (eps = 0)."""
    d = 64
    c = np.array([[3.0] * d, [-0.5] * d])
    y = oracle.rms_norm(c, eps=0.0)
    assert np.allclose(y[0], 1.0, rtol=0, atol=1e-15) and np.allclose(y[1], -1.0, rtol=0, atol=1e-15)
    y = oracle.rms_norm(np.array([[2.0] * d]), eps=0.25)
    assert np.allclose(y, 2.0 / np.sqrt(4.0 + 0.25), rtol=1e-15, atol=0)
    onehot = np.zeros((1, d))
    onehot[0, 5] = 7.0
    y = oracle.rms_norm(onehot, eps=0.0)
    assert abs(y[0, 5] - np.sqrt(d)) < 1e-12 and np.count_nonzero(y) == 1


def test_rms_norm_invariants():
    """Unit mean square for eps = 0, invariance to positive scaling, odd
    symmetry, rows independent of each other."""
    rng = np.random.default_rng(5)
    x = rng.normal(size=(6, 96)) * rng.uniform(0.1, 50, size=(6, 1))
    y = oracle.rms_norm(x, eps=0.0)
    assert np.allclose((y * y).mean(axis=1), 1.0, rtol=1e-13)
    assert np.allclose(oracle.rms_norm(3.7 * x, eps=0.0), y, rtol=1e-13)
    assert np.allclose(oracle.rms_norm(-x, eps=0.0), -y, rtol=0, atol=0)
    assert np.allclose(oracle.rms_norm(x[2:3], eps=0.0), y[2:3], rtol=0, atol=0)


# ------------------------------------------------------------ record checksum

def test_crc32_check_value():
    """The catalogued check value of CRC-32/ISO-HDLC: the nine ASCII bytes
    "123456789" give 0xCBF43926."""
    assert oracle.crc32(b"123456789") == 0xCBF43926
    assert oracle.crc32(b"") == 0


@pytest.mark.parametrize("n", [1, 7, 128, 4096, 100003])
def test_crc32_matches_zlib(n):
    """Library special case: zlib's crc32 is the same code."""
    import zlib
    data = np.random.default_rng(n).integers(0, 256, size=n, dtype=np.uint8)
    assert oracle.crc32(data) == zlib.crc32(data.tobytes())


def test_crc32_sees_every_single_bit_flip():
    data = np.random.default_rng(5).integers(0, 256, size=3000, dtype=np.uint8)
    ref = oracle.crc32(data)
    for pos in (0, 1, 1499, 2998, 2999):
        for bit in (0, 3, 7):
            d = data.copy()
            d[pos] ^= np.uint8(1 << bit)
            assert oracle.crc32(d) != ref


# ------------------------------------------------------------ offline encoder

def _prototype_matrix():
    """96 x 64 weights whose 768 sub-vectors cycle through 256 distinct
    prototypes P[p] = (p + 1) * (1..8) / 1024 (exact in fp32 and in the
    encoder's 2^-32 fixed point)."""
    P = ((np.arange(256)[:, None] + 1) * (np.arange(8)[None, :] + 1) / 1024.0).astype(np.float32)
    sub = P[np.arange(768) % 256]
    return sub.reshape(96, 64), P


def test_encode_recovers_prototypes_exactly():
    """Closed form: the initial codebook takes sub-vectors 3k (N = 768), i.e.
    P[3k mod 256], all distinct since 3 is odd; every sub-vector matches one
    codeword exactly (code 171 p mod 256, 171 = 3^-1 mod 256), the means of
    identical members are exact, the residual is zero, and the later stages
    get zero codebooks and code 0 (ties to the lower index)."""
    w, P = _prototype_matrix()
    codes, cb = oracle.rvq_encode(w, 3)
    i = np.arange(768).reshape(96, 8)
    assert np.array_equal(codes[..., 0], (171 * (i % 256)) % 256)
    assert np.array_equal(codes[..., 1:], np.zeros((96, 8, 2), np.uint8))
    assert np.array_equal(cb[0], P[(3 * np.arange(256)) % 256])
    assert not cb[1:].any()
    deq = (cb[0][codes[..., 0]] + cb[1][codes[..., 1]] + cb[2][codes[..., 2]]).reshape(96, 64)
    assert np.array_equal(deq, w)


def _stage_distortion(w, codes, cb, stages):
    r = w.reshape(-1, 8).astype(np.float64)
    c = codes.reshape(-1, 3)
    for s in range(stages):
        r = r - cb[s][c[:, s]].astype(np.float64)
    return float((r ** 2).sum())


def test_encode_lloyd_rounds_never_increase_distortion():
    w = np.random.default_rng(11).normal(0, 0.02, size=(64, 512)).astype(np.float32)
    d = [_stage_distortion(w, *oracle.rvq_encode(w, it), 1) for it in (0, 1, 2, 4)]
    assert all(b <= a * (1 + 1e-6) for a, b in zip(d, d[1:])), d
    assert d[-1] < d[0]
    full = _stage_distortion(w, *oracle.rvq_encode(w, 2), 3)
    assert full < _stage_distortion(w, *oracle.rvq_encode(w, 2), 1)


def test_encode_codes_are_nearest_codewords():
    """Every stage's code is a nearest codeword of that stage's residual
    (checked in double: its distance is within fp32 rounding of the least)."""
    w = np.random.default_rng(12).normal(0, 0.02, size=(32, 256)).astype(np.float32)
    codes, cb = oracle.rvq_encode(w, 2)
    r = w.reshape(-1, 8).astype(np.float32)
    c = codes.reshape(-1, 3)
    for s in range(3):
        dist = ((r[:, None, :].astype(np.float64) - cb[s][None].astype(np.float64)) ** 2).sum(-1)
        got = dist[np.arange(len(r)), c[:, s]]
        assert np.all(got <= dist.min(1) * (1 + 1e-5) + 1e-12)
        r = r - cb[s][c[:, s]]
