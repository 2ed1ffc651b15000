"""Pins for the f64 checker in ``oracle/`` against facts that do not come
from the checker itself: hand-packed words, closed forms, the quantizer
round-trip bound, exact rational brute force on tiny shapes, and the
constant-per-expert case that exposes a mis-gathered index (mlxcel PR #1562,
What changed: f64 dense per-expert reference and constant-per-expert case).
"""

import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "packed_words.txt")


def _golden_words():
    out = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            out.append((int(parts[0]), int(parts[1], 16), [int(t) for t in parts[2:]]))
    return out


def _bf16(v):
    return synth.f32_to_bf16_bits(np.asarray(v, dtype=np.float32))


def _bf16_exact(v):
    """bf16 bits of v, asserting that v is exactly representable."""
    h = _bf16(v)
    assert np.all(synth.bf16_bits_to_f32(h) == np.asarray(v, dtype=np.float32))
    return h


# ---------------------------------------------------------------- unpacking


@pytest.mark.parametrize("bits,word,codes", _golden_words())
def test_hand_packed_word_unpacks(bits, word, codes):
    per = 32 // bits
    assert len(codes) == per
    # One row of 64 codes: the word in slot 3, zeros elsewhere.
    K = 64
    w = np.zeros((1, K * bits // 32), dtype=np.uint32)
    w[0, 3] = word
    q = oracle.unpack(w, 1, K, bits)
    assert list(q[0, 3 * per:4 * per]) == codes
    assert int(q.sum()) == sum(codes)


@pytest.mark.parametrize("bits,word,codes", _golden_words())
def test_hand_packed_word_dequantises(bits, word, codes):
    # s = 1, b = 0 turns the codes into weights; s = 0.5, b = -3 checks both
    # terms of s*q + b.
    K = 64
    per = 32 // bits
    w = np.zeros((1, K * bits // 32), dtype=np.uint32)
    w[0, 0] = word
    for s, b in ((1.0, 0.0), (0.5, -3.0)):
        wh = oracle.dequant(w, _bf16_exact([[s]]), _bf16_exact([[b]]), 1, K, bits)
        assert list(wh[0, :per]) == [s * c + b for c in codes]
        assert np.all(wh[0, per:] == b)


def _golden_streams():
    out = []
    path = os.path.join(os.path.dirname(__file__), "golden", "packed_streams.txt")
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, codes = line.split(":")
            bits, words = head.split()
            out.append((int(bits), [int(t, 16) for t in words.split(",")],
                        [int(t) for t in codes.split()]))
    return out


@pytest.mark.parametrize("bits,words,codes", _golden_streams())
def test_hand_packed_stream_unpacks(bits, words, codes):
    # 3- and 6-bit rows whose codes straddle words, placed as the second
    # unit of a 64-code row with zeros elsewhere
    K = 64
    w = np.zeros((1, K * bits // 32), dtype=np.uint32)
    n0 = len(words)
    w[0, n0:2 * n0] = words
    q = oracle.unpack(w, 1, K, bits)
    per_unit = len(codes)
    assert list(q[0, per_unit:2 * per_unit]) == codes
    assert int(q.sum()) == sum(codes)
    # the input generator's packer writes the same words from the codes
    qq = np.zeros((1, K), np.uint8)
    qq[0, per_unit:2 * per_unit] = codes
    assert np.array_equal(synth.pack_codes(qq, bits), w)
    # and the hex-digit reading of the test agrees
    assert _row_codes(w[0], K, bits) == list(q[0])


@pytest.mark.parametrize("bits,words,codes", _golden_streams())
def test_hand_packed_stream_dequantises(bits, words, codes):
    K = 64
    w = np.zeros((1, K * bits // 32), dtype=np.uint32)
    w[0, :len(words)] = words
    wh = oracle.dequant(w, _bf16_exact([[0.5]]), _bf16_exact([[-3.0]]), 1, K, bits)
    assert list(wh[0, :len(codes)]) == [0.5 * c - 3.0 for c in codes]
    assert np.all(wh[0, len(codes):] == -3.0)


def test_packer_matches_golden_words():
    # The input generator's packer writes the golden words from their codes.
    for bits, word, codes in _golden_words():
        packed = synth.pack_codes(np.array([codes], dtype=np.uint8), bits)
        assert int(packed[0, 0]) == word


@pytest.mark.parametrize("bits", [2, 3, 4, 6, 8])
def test_one_hot_x_selects_weight(bits):
    # x = e_k picks out w^[n, k]: pins nibble order, word order across k and
    # the group index at the 63/64 boundary.
    rng = np.random.default_rng(5)
    N, K = 3, 192
    q = rng.integers(0, 1 << bits, size=(N, K), dtype=np.uint8)
    w = synth.pack_codes(q, bits)
    s_vals = np.array([[0.5, 0.25, 2.0], [1.0, 0.125, 4.0], [0.0625, 8.0, 1.5]], np.float32)
    b_vals = np.array([[-1.0, 3.0, 0.5], [2.0, -0.75, 0.0], [1.25, -2.0, 6.0]], np.float32)
    s, b = _bf16_exact(s_vals), _bf16_exact(b_vals)
    for k in (0, 1, 7, 8, 31, 63, 64, 65, 127, 128, 191):
        x = np.zeros((1, K), dtype=np.float32)
        x[0, k] = 1.0
        y, _ = oracle.qmm(_bf16_exact(x), w, s, b, 1, K, N, bits)
        g = k // 64
        want = s_vals[:, g].astype(np.float64) * q[:, k] + b_vals[:, g]
        assert np.array_equal(y[0], want), k


# ------------------------------------------------------------- closed forms


@pytest.mark.parametrize("bits", [2, 3, 4, 6, 8])
def test_zero_scale_gives_bias_times_row_sum(bits):
    rng = np.random.default_rng(7)
    M, N, K = 3, 5, 256
    x = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
    q = rng.integers(0, 1 << bits, size=(N, K), dtype=np.uint8)
    c = (np.arange(N, dtype=np.float32) + 1.0) / 8.0
    s = _bf16_exact(np.zeros((N, K // 64), np.float32))
    b = _bf16_exact(np.repeat(c[:, None], K // 64, axis=1))
    y, bnd = oracle.qmm(_bf16_exact(x), synth.pack_codes(q, bits), s, b, M, K, N, bits)
    want = x.sum(axis=1, dtype=np.float64)[:, None] * c[None, :].astype(np.float64)
    assert np.array_equal(y, want)
    assert np.array_equal(bnd, np.abs(x).sum(axis=1, dtype=np.float64)[:, None] * c[None, :])


@pytest.mark.parametrize("bits", [2, 3, 4, 6, 8])
def test_all_max_codes(bits):
    rng = np.random.default_rng(8)
    M, N, K = 2, 4, 128
    x = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
    q = np.full((N, K), (1 << bits) - 1, dtype=np.uint8)
    w = synth.pack_codes(q, bits)
    assert np.all(w == 0xFFFFFFFF)
    s = _bf16_exact(np.ones((N, K // 64), np.float32))
    b = _bf16_exact(np.zeros((N, K // 64), np.float32))
    y, _ = oracle.qmm(_bf16_exact(x), w, s, b, M, K, N, bits)
    want = ((1 << bits) - 1) * x.sum(axis=1, dtype=np.float64)
    assert np.array_equal(y, np.repeat(want[:, None], N, axis=1))


def test_alternating_group_scales_pin_group_boundary():
    # Group g has s = 2^g, b = -g; with x = 1 and q = 1 the sum is
    # 64 * sum_g (2^g - g), which moves if any k is charged to the wrong group.
    K, N, bits = 256, 2, 4
    ng = K // 64
    q = np.ones((N, K), dtype=np.uint8)
    s = _bf16_exact(np.tile([2.0 ** g for g in range(ng)], (N, 1)))
    b = _bf16_exact(np.tile([-float(g) for g in range(ng)], (N, 1)))
    x = _bf16_exact(np.ones((1, K), np.float32))
    y, _ = oracle.qmm(x, synth.pack_codes(q, bits), s, b, 1, K, N, bits)
    assert np.all(y == 64 * sum(2.0 ** g - g for g in range(ng)))
    # Shift one code across the 63/64 boundary: only group 0 vs 1 sees it.
    q2 = q.copy()
    q2[:, 63] = 0
    q2[:, 64] = 2
    y2, _ = oracle.qmm(x, synth.pack_codes(q2, bits), s, b, 1, K, N, bits)
    assert np.all(y2 - y == -1.0 + 2.0)


# ------------------------------------------------------ quantizer round trip


@pytest.mark.parametrize("bits", [2, 3, 4, 6, 8])
def test_round_trip_exact_bound_on_representable_grid(bits):
    # Groups whose min and (max - min)/(2^bits - 1) are exact in bf16: the
    # dequantised weight is within s/2 of the original, exactly.
    rng = np.random.default_rng(11)
    L = (1 << bits) - 1
    N, K = 6, 256
    ng = K // 64
    step = 2.0 ** rng.integers(-9, -5, size=(N, ng))
    lo = rng.integers(-64, 0, size=(N, ng)) * 2.0 ** -8
    u = rng.random((N, ng, 64)) * L
    u[:, :, 0] = 0.0
    u[:, :, 1] = L
    W = (lo[:, :, None] + u * step[:, :, None]).reshape(N, K).astype(np.float32)
    qw = synth.quantize(W, bits)
    s = synth.bf16_bits_to_f32(qw.scales).astype(np.float64)
    b = synth.bf16_bits_to_f32(qw.biases).astype(np.float64)
    Wg = W.astype(np.float64).reshape(N, ng, 64)
    assert np.array_equal(b, Wg.min(axis=2))
    assert np.array_equal(s, (Wg.max(axis=2) - Wg.min(axis=2)) / L)
    wh = oracle.dequant(qw.w, qw.scales, qw.biases, N, K, bits).reshape(N, ng, 64)
    err = np.abs(Wg - wh)
    assert np.all(err <= s[:, :, None] / 2 * (1 + 1e-12))
    # and the codes the checker unpacks are the quantizer's codes
    assert np.array_equal(oracle.unpack(qw.w, N, K, bits), qw.q)


@pytest.mark.parametrize("bits", [2, 3, 4, 6, 8])
def test_round_trip_bound_gaussian_weights(bits):
    # W ~ N(0, 0.02): with bf16-rounded s and b the error bound gains the
    # amount by which the stored [b, b + L*s] range misses [min, max].
    L = (1 << bits) - 1
    N, K = 64, 512
    W = synth.dense_weights(N, K, seed=0)
    qw = synth.quantize(W, bits)
    ng = K // 64
    s = synth.bf16_bits_to_f32(qw.scales).astype(np.float64)[:, :, None]
    b = synth.bf16_bits_to_f32(qw.biases).astype(np.float64)[:, :, None]
    Wg = W.astype(np.float64).reshape(N, ng, 64)
    mn = Wg.min(axis=2, keepdims=True)
    mx = Wg.max(axis=2, keepdims=True)
    slack = np.maximum(0, b - mn) + np.maximum(0, mx - (b + L * s))
    wh = oracle.dequant(qw.w, qw.scales, qw.biases, N, K, bits).reshape(N, ng, 64)
    err = np.abs(Wg - wh)
    assert np.all(err <= s / 2 + slack + 1e-15)
    # the plain s/2 bound holds for every weight inside the stored range
    inside = (Wg >= b) & (Wg <= b + L * s)
    assert np.all(err[inside] <= (s / 2 + 1e-15 + 0 * Wg)[inside])


def test_flat_group_dequantises_to_bias():
    W = np.full((2, 128), 0.0123, dtype=np.float32)
    qw = synth.quantize(W, 4)
    assert np.all(qw.scales == 0) and np.all(qw.q == 0)
    wh = oracle.dequant(qw.w, qw.scales, qw.biases, 2, 128, 4)
    assert np.all(wh == synth.bf16_bits_to_f32(qw.biases[0, 0]))


# --------------------------------------------- exact rational brute force


def _hex_unpack(word, bits):
    """Codes of one word, lowest k first, read from its hex digits."""
    digits = "%08x" % word
    if bits == 2:
        # each hex digit holds two codes: its low two bits first
        out = []
        for d in reversed(digits):
            v = int(d, 16)
            out += [v % 4, v // 4]
        return out
    if bits == 4:
        return [int(d, 16) for d in reversed(digits)]
    return [int(digits[i:i + 2], 16) for i in (6, 4, 2, 0)]


def _row_codes(words, K, bits):
    """Codes of one packed row, read as a bit string built from the hex
    digits of its words: word 0 first, each word's lowest digit first, each
    digit's lowest bit first; code k is bits [k*bits, k*bits + bits)."""
    bitstring = []
    for word in words:
        for d in reversed("%08x" % int(word)):
            v = int(d, 16)
            bitstring += [(v >> i) & 1 for i in range(4)]
    return [sum(bitstring[k * bits + i] << i for i in range(bits)) for k in range(K)]


def _bf16_fraction(h):
    # the bf16 pattern is the top half of an IEEE binary32
    return Fraction(struct.unpack("<f", struct.pack("<I", int(h) << 16))[0])


def _brute(x, w, s, b, M, K, N, bits, group=64):
    y = [[Fraction(0)] * N for _ in range(M)]
    for n in range(N):
        codes = _row_codes(w[n], K, bits)
        wrow = [_bf16_fraction(s[n, k // group]) * codes[k] + _bf16_fraction(b[n, k // group])
                for k in range(K)]
        for m in range(M):
            y[m][n] = sum((_bf16_fraction(x[m, k]) * wrow[k] for k in range(K)), Fraction(0))
    return y


@pytest.mark.parametrize("bits", [2, 3, 4, 6, 8])
@pytest.mark.parametrize("M,N,K", [(1, 1, 64), (2, 3, 64), (4, 4, 128), (3, 2, 128)])
def test_brute_force_exact(bits, M, N, K):
    seed = 100 * bits + 10 * M + N + K
    W = synth.dense_weights(N, K, seed=seed)
    qw = synth.quantize(W, bits)
    x = synth.activations(M, K, seed=seed + 1)
    y, bnd = oracle.qmm(x, qw.w, qw.scales, qw.biases, M, K, N, bits)
    exact = _brute(x, qw.w, qw.scales, qw.biases, M, K, N, bits)
    for m in range(M):
        for n in range(N):
            e = float(exact[m][n])
            # f64 summation error is far below 1e-12 of the magnitude bound
            assert abs(y[m, n] - e) <= 1e-12 * bnd[m, n] + 1e-300, (m, n)


def test_brute_force_exhaustive_codes_4bit():
    # Every 4-bit code value at every nibble position of a word.
    K, N = 64, 16
    q = np.array([[(n + k) % 16 for k in range(K)] for n in range(N)], dtype=np.uint8)
    w = synth.pack_codes(q, 4)
    s = _bf16_exact(np.full((N, 1), 0.25, np.float32))
    b = _bf16_exact(np.full((N, 1), -1.5, np.float32))
    x = synth.activations(2, K, seed=3)
    y, _ = oracle.qmm(x, w, s, b, 2, K, N, 4)
    exact = _brute(x, w, s, b, 2, K, N, 4)
    for m in range(2):
        for n in range(N):
            assert abs(y[m, n] - float(exact[m][n])) <= 1e-13


# ------------------------------------------------------- contraction layout


@pytest.mark.parametrize("bits", [2, 3, 4, 6, 8])
def test_qmm_is_x_times_dequant_transposed(bits):
    # Special case reducing to a library matmul: y = x . W^T with W^ built
    # from the exact per-element formula (written here with the hex unpack).
    M, N, K = 5, 7, 192
    W = synth.dense_weights(N, K, seed=21)
    qw = synth.quantize(W, bits)
    x = synth.activations(M, K, seed=22)
    codes = np.array([_row_codes(qw.w[n], K, bits) for n in range(N)], dtype=np.float64)
    s = synth.bf16_bits_to_f32(qw.scales).astype(np.float64)
    b = synth.bf16_bits_to_f32(qw.biases).astype(np.float64)
    wh = codes * np.repeat(s, 64, axis=1) + np.repeat(b, 64, axis=1)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    y, bnd = oracle.qmm(x, qw.w, qw.scales, qw.biases, M, K, N, bits)
    assert np.allclose(y, xf @ wh.T, rtol=0, atol=1e-12)
    assert np.allclose(bnd, np.abs(xf) @ np.abs(wh).T, rtol=0, atol=1e-12)
    yv, _ = oracle.qmv(x[2], qw.w, qw.scales, qw.biases, K, N, bits)
    assert np.array_equal(yv, y[2])


# ---------------------------------------------------- sorted-MoE variant


def test_constant_per_expert_catches_misgather():
    # w^_e[n, k] = c_{e,n} (s = 0, b = c), distinct per (e, n); x integer so
    # every sum is exact: y[r, n] = c_{e(r), n} * sum_k x[src(r), k].
    E, N, K, T, top_k = 6, 5, 128, 9, 3
    expert_ids, row_src = synth.routing(T, E, top_k, seed=2)
    B = T * top_k
    rng = np.random.default_rng(4)
    x = rng.integers(-4, 5, size=(T, K)).astype(np.float32)
    # (e + 1)/2 + n/16 is exact in bf16 and distinct for n < 8
    c = np.array([[(e + 1) / 2.0 + n / 16.0 for n in range(N)] for e in range(E)])
    cb = _bf16_exact(c)
    s = np.zeros((E, N, K // 64), np.uint16)
    b = np.repeat(cb[:, :, None], K // 64, axis=2)
    w = rng.integers(0, 2 ** 32, size=(E, N, K // 8), dtype=np.uint64).astype(np.uint32)
    y, _ = oracle.gather_qmm(_bf16_exact(x), w, s, b, expert_ids, row_src, T, B, E, K, N, 4)
    xs = x.sum(axis=1, dtype=np.float64)
    want = c[expert_ids] * xs[row_src][:, None]
    assert np.array_equal(y, want)
    # the per-(e, n) constants are distinct, so a wrong expert, a wrong source
    # row or swapped n would change the answer
    assert len(np.unique(c)) == E * N


def test_gather_single_expert_equals_qmm_on_gathered_rows():
    E, N, K, T = 1, 6, 128, 5
    W = synth.dense_weights(N, K, seed=31)
    qw = synth.quantize(W, 4)
    x = synth.activations(T, K, seed=32)
    row_src = np.array([3, 0, 4, 4, 1, 2, 0], dtype=np.int32)
    B = len(row_src)
    ids = np.zeros(B, np.int32)
    y, _ = oracle.gather_qmm(x, qw.w[None], qw.scales[None], qw.biases[None], ids, row_src,
                             T, B, E, K, N, 4)
    ref, _ = oracle.qmm(x[row_src], qw.w, qw.scales, qw.biases, B, K, N, 4)
    assert np.array_equal(y, ref)


def test_gather_matches_per_expert_qmm():
    E, N, K, T, top_k, bits = 4, 3, 128, 6, 2, 8
    ids, src = synth.routing(T, E, top_k, seed=40)
    B = T * top_k
    qws = [synth.quantize(synth.dense_weights(N, K, seed=41 + e), bits) for e in range(E)]
    w = np.stack([q.w for q in qws])
    s = np.stack([q.scales for q in qws])
    b = np.stack([q.biases for q in qws])
    x = synth.activations(T, K, seed=45)
    y, bnd = oracle.gather_qmm(x, w, s, b, ids, src, T, B, E, K, N, bits)
    for r in range(B):
        ref, rb = oracle.qmm(x[src[r]][None], w[ids[r]], s[ids[r]], b[ids[r]], 1, K, N, bits)
        assert np.array_equal(y[r], ref[0]) and np.array_equal(bnd[r], rb[0])


def test_gather_out_of_range_expert_row_is_zero():
    E, N, K = 2, 3, 64
    qw = synth.quantize(synth.dense_weights(N, K, seed=1), 4)
    w = np.stack([qw.w, qw.w])
    s = np.stack([qw.scales, qw.scales])
    b = np.stack([qw.biases, qw.biases])
    x = synth.activations(3, K, seed=2)
    ids = np.array([0, 1, 7], np.int32)
    y, _ = oracle.gather_qmm(x, w, s, b, ids, None, 3, 3, E, K, N, 4)
    assert np.all(y[2] == 0)


def test_points_match_full_results():
    E, N, K, T, top_k = 3, 4, 128, 5, 2
    ids, src = synth.routing(T, E, top_k, seed=50)
    B = T * top_k
    qws = [synth.quantize(synth.dense_weights(N, K, seed=51 + e), 4) for e in range(E)]
    w = np.stack([q.w for q in qws])
    s = np.stack([q.scales for q in qws])
    b = np.stack([q.biases for q in qws])
    x = synth.activations(T, K, seed=55)
    y, bnd = oracle.gather_qmm(x, w, s, b, ids, src, T, B, E, K, N, 4)
    rows = np.array([0, 3, B - 1, 5], np.int64)
    cols = np.array([1, 0, 3, 2], np.int64)
    yp, bp = oracle.points(x, w, s, b, rows, cols, K, N, 4, expert_ids=ids, row_src=src, E=E)
    assert np.array_equal(yp, y[rows, cols]) and np.array_equal(bp, bnd[rows, cols])
    # and without expert ids it is qmm
    y2, _ = oracle.qmm(x, w[0], s[0], b[0], T, K, N, 4)
    yp2, _ = oracle.points(x, w[0], s[0], b[0], np.array([4, 0]), np.array([3, 2]), K, N, 4)
    assert np.array_equal(yp2, y2[[4, 0], [3, 2]])


def test_routing_recipe():
    ids, src = synth.routing(573, 128, 8, seed=2)
    assert ids.shape == (4584,) and src.shape == (4584,)
    assert np.all(np.diff(ids) >= 0)
    # each token appears top_k times, with distinct experts
    assert np.all(np.bincount(src, minlength=573) == 8)
    pairs = set(zip(src.tolist(), ids.tolist()))
    assert len(pairs) == 4584


# ---- the affine encoder (binary32 decisions)

def test_quantize_hand_example_exact_grid():
    # values -1 + 0.25 * (j % 16): min -1, max 2.75, range/15 = 0.25 exactly,
    # so every code is j % 16 and the stored scale/bias are 0.25 and -1
    j = np.arange(64)
    W = (-1.0 + 0.25 * (j % 16)).astype(np.float32)[None, :]
    for bits in (4, 8):
        codes, s, b = oracle.quantize(W, bits)
        step = 0.25 if bits == 4 else 3.75 / 255
        assert s[0, 0] == synth.f32_to_bf16_bits(np.float32(step))
        assert b[0, 0] == 0xBF80  # -1.0
        q = oracle.unpack(codes, 1, 64, bits)[0]
        if bits == 4:
            assert np.array_equal(q, j % 16)
        else:
            s_f = float(np.asarray(synth.bf16_bits_to_f32(s)).reshape(-1)[0])
            assert np.array_equal(q, np.clip(np.rint((W[0] + 1.0) / s_f), 0, 255))


def test_quantize_flat_group_and_signed_zero():
    W = np.zeros((2, 128), np.float32)
    W[0, :64] = 0.3
    W[0, 64:] = -0.0          # a group of negative zeros
    W[1, :64] = -0.0
    W[1, 64:] = np.where(np.arange(64) % 2 == 0, 0.0, -0.0).astype(np.float32)
    codes, s, b = oracle.quantize(W, 4)
    assert np.all(s == 0) and np.all(codes == 0)
    assert b[0, 0] == synth.f32_to_bf16_bits(np.float32(0.3))
    assert b[0, 1] == 0 and b[1, 0] == 0 and b[1, 1] == 0   # -0 is read as +0


@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("bits", [2, 3, 4, 6, 8])
def test_quantize_round_trip_bound(bits, group):
    rng = np.random.default_rng(31 + bits)
    W = (rng.standard_normal((48, 1024)) * 0.02).astype(np.float32)
    codes, s, b = oracle.quantize(W, bits, group)
    assert s.shape == (48, 1024 // group)
    w_hat = oracle.dequant(codes, s, b, 48, 1024, bits, group)
    s_f = np.repeat(synth.bf16_bits_to_f32(s).astype(np.float64), group, axis=1)
    Wg = W.reshape(48, 1024 // group, group).astype(np.float64)
    mag = np.repeat(np.abs(Wg).max(axis=2), group, axis=1)
    # half a step; the stored scale is the exact step rounded to bf16 (relative
    # error <= 2^-9), so the top of the range can sit up to levels * 2^-9
    # steps past the last code; plus the bf16 rounding of the bias (the group
    # minimum)
    levels = (1 << bits) - 1
    assert np.all(np.abs(W - w_hat) <= (0.5 + levels * 2.0 ** -9) * s_f + 2.0 ** -8 * mag + 1e-12)
    # and within plain half a step away from the clamped ends
    inner = (W > np.repeat(Wg.min(axis=2), group, axis=1) + 2 * s_f) & \
            (W < np.repeat(Wg.max(axis=2), group, axis=1) - 2 * s_f)
    assert np.all(np.abs(W - w_hat)[inner] <= 0.5 * s_f[inner] * (1 + 1e-6) + 1e-12)


@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("bits", [2, 3, 4, 6, 8])
def test_quantize_agrees_with_float64_encoder(bits, group):
    # synth.quantize takes the same decisions in float64 (numpy): away from
    # exact ties the two encoders must agree on every code, scale and bias
    rng = np.random.default_rng(41 + bits)
    W = (rng.standard_normal((96, 2048)) * 0.02).astype(np.float32)
    codes, s, b = oracle.quantize(W, bits, group)
    qw = synth.quantize(W, bits, group)
    assert np.array_equal(s, qw.scales) and np.array_equal(b, qw.biases)
    q = oracle.unpack(codes, 96, 2048, bits)
    # a quotient within binary32 rounding of a half-way point may round the
    # other way in float32 (ties to even there): such codes may differ by one
    s_f = np.repeat(synth.bf16_bits_to_f32(s).astype(np.float64), group, axis=1)
    b_f = np.repeat(synth.bf16_bits_to_f32(b).astype(np.float64), group, axis=1)
    t = np.where(s_f > 0, (W.astype(np.float64) - b_f) / np.where(s_f > 0, s_f, 1.0), 0.0)
    near_tie = np.abs(t - np.floor(t) - 0.5) < 1e-5
    assert np.array_equal(q[~near_tie], qw.q[~near_tie])
    assert np.all(np.abs(q[near_tie].astype(int) - qw.q[near_tie].astype(int)) <= 1)
    assert near_tie.mean() < 1e-3


# ---- group sizes 32 and 128 (issue #1536, Diagnosis item 4: the group size
# is a parameter of the stored format; 32 and 128 sit on either side of 64)


def _group_sb(N, ng):
    """Exact, pairwise distinct scale and bias per (row, group)."""
    g = np.arange(ng)[None, :]
    n = np.arange(N)[:, None]
    s_vals = (2.0 ** ((n + g) % 7 - 4)).astype(np.float32)
    b_vals = ((g + 1) * 0.125 * np.where(n % 2 == 0, 1.0, -1.0) + n).astype(np.float32)
    return s_vals, b_vals


@pytest.mark.parametrize("group", [32, 128])
@pytest.mark.parametrize("bits", [2, 3, 4, 6, 8])
def test_one_hot_x_selects_weight_group_sizes(bits, group):
    # x = e_k picks out w^[n, k] = s[n, k/G] q + b[n, k/G]: a k charged to
    # the neighbouring group reads another (s, b) pair
    rng = np.random.default_rng(60 + bits + group)
    N, K = 3, 384
    ng = K // group
    q = rng.integers(0, 1 << bits, size=(N, K), dtype=np.uint8)
    w = synth.pack_codes(q, bits)
    s_vals, b_vals = _group_sb(N, ng)
    s, b = _bf16_exact(s_vals), _bf16_exact(b_vals)
    for k in sorted({0, 1, group - 1, group, group + 1, 2 * group - 1, 2 * group, K - 1}):
        x = np.zeros((1, K), dtype=np.float32)
        x[0, k] = 1.0
        y, _ = oracle.qmm(_bf16_exact(x), w, s, b, 1, K, N, bits, group)
        g = k // group
        want = s_vals[:, g].astype(np.float64) * q[:, k] + b_vals[:, g]
        assert np.array_equal(y[0], want), k


@pytest.mark.parametrize("group", [32, 128])
def test_alternating_group_scales_pin_group_boundary_sizes(group):
    # Group g has s = 2^g, b = -g; with x = 1 and q = 1 the sum is
    # G * sum_g (2^g - g); moving one unit of code from k = G-1 to k = G
    # changes it by s_1 - s_0 = 1, and by a different amount if either k
    # sits in the wrong group.
    K, N, bits = 512, 2, 4
    ng = K // group
    q = np.ones((N, K), dtype=np.uint8)
    s = _bf16_exact(np.tile([2.0 ** g for g in range(ng)], (N, 1)))
    b = _bf16_exact(np.tile([-float(g) for g in range(ng)], (N, 1)))
    x = _bf16_exact(np.ones((1, K), np.float32))
    y, _ = oracle.qmm(x, synth.pack_codes(q, bits), s, b, 1, K, N, bits, group)
    assert np.all(y == group * sum(2.0 ** g - g for g in range(ng)))
    q2 = q.copy()
    q2[:, group - 1] = 0
    q2[:, group] = 2
    y2, _ = oracle.qmm(x, synth.pack_codes(q2, bits), s, b, 1, K, N, bits, group)
    assert np.all(y2 - y == 1.0)


@pytest.mark.parametrize("group", [32, 128])
@pytest.mark.parametrize("bits", [2, 3, 4, 6, 8])
@pytest.mark.parametrize("M,N,K", [(1, 2, 128), (2, 3, 256)])
def test_brute_force_exact_group_sizes(bits, group, M, N, K):
    seed = 7 * group + 100 * bits + 10 * M + N + K
    W = synth.dense_weights(N, K, seed=seed)
    qw = synth.quantize(W, bits, group)
    x = synth.activations(M, K, seed=seed + 1)
    y, bnd = oracle.qmm(x, qw.w, qw.scales, qw.biases, M, K, N, bits, group)
    exact = _brute(x, qw.w, qw.scales, qw.biases, M, K, N, bits, group)
    for m in range(M):
        for n in range(N):
            assert abs(y[m, n] - float(exact[m][n])) <= 1e-12 * bnd[m, n] + 1e-300, (m, n)


@pytest.mark.parametrize("group", [32, 128])
def test_gather_group_sizes_constant_per_expert(group):
    # s = 0, b = c_{e,n} per group: y[r, n] = c_{e(r),n} * sum_k x[src(r), k]
    # exactly, whatever the group size, and the group count per row is K/G
    E, N, K, T = 3, 4, 256, 5
    ng = K // group
    rng = np.random.default_rng(70 + group)
    x = rng.integers(-4, 5, size=(T, K)).astype(np.float32)
    c = ((np.arange(E)[:, None] + 1) / 4.0 + np.arange(N)[None, :] / 64.0).astype(np.float32)
    w = np.zeros((E, N, K // 8), np.uint32)
    s = _bf16_exact(np.zeros((E, N, ng), np.float32))
    b = _bf16_exact(np.repeat(c[:, :, None], ng, axis=2))
    ids = np.array([0, 0, 1, 2, 2, 2], np.int32)
    src = np.array([4, 1, 0, 3, 2, 0], np.int32)
    y, _ = oracle.gather_qmm(_bf16_exact(x), w, s, b, ids, src, T, 6, E, K, N, 4, group)
    want = x.sum(axis=1, dtype=np.float64)[src][:, None] * c[ids].astype(np.float64)
    assert np.array_equal(y, want)


@pytest.mark.parametrize("group", [32, 128])
def test_quantize_hand_example_group_sizes(group):
    # the exact grid -1 + 0.25 * (j % 16) repeats inside every group of 32
    # or 128, so every group stores s = 0.25, b = -1 and codes j % 16
    K = 256
    j = np.arange(K)
    W = (-1.0 + 0.25 * (j % 16)).astype(np.float32)[None, :]
    codes, s, b = oracle.quantize(W, 4, group)
    assert s.shape == (1, K // group)
    assert np.all(s == synth.f32_to_bf16_bits(np.float32(0.25)))
    assert np.all(b == 0xBF80)
    assert np.array_equal(oracle.unpack(codes, 1, K, 4)[0], j % 16)
    # a single group's range change moves only that group's pair
    W2 = W.copy()
    W2[0, group + 3] = 5.0
    _, s2, b2 = oracle.quantize(W2, 4, group)
    changed = np.nonzero(s2[0] != s[0])[0]
    assert list(changed) == [1]
    assert np.array_equal(b2, b)


# ---- the [K, N] operand layout (PR #1562, What changed: both operand
# layouts): row k holds the codes of every output n, groups run along n


def _kn_case(K, N, bits, group, seed):
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 1 << bits, size=(K, N), dtype=np.uint8)
    w = synth.pack_codes(q, bits)                      # [K, N*bits/32]
    g = np.arange(N // group)[None, :]
    k = np.arange(K)[:, None]
    s_vals = (2.0 ** ((k + 2 * g) % 6 - 5)).astype(np.float32)
    b_vals = ((g + 1) * 0.25 - (k % 3) * 0.5).astype(np.float32)
    return q, w, s_vals, b_vals


@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("bits", [2, 4, 8])
def test_kn_one_hot_selects_weight(bits, group):
    # x = e_k picks row k: y[n] = s[k, n/G] q[k, n] + b[k, n/G], so a code
    # read from the wrong row or column, or a scale from the wrong (row,
    # group), shows
    K, N = 7, 384
    q, w, s_vals, b_vals = _kn_case(K, N, bits, group, 80 + bits + group)
    s, b = _bf16_exact(s_vals), _bf16_exact(b_vals)
    for k in range(K):
        x = np.zeros((1, K), np.float32)
        x[0, k] = 1.0
        y, _ = oracle.qmm_kn(_bf16_exact(x), w, s, b, 1, K, N, bits, group)
        gidx = np.arange(N) // group
        want = s_vals[k, gidx].astype(np.float64) * q[k] + b_vals[k, gidx]
        assert np.array_equal(y[0], want), k


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_kn_uniform_scales_equal_transposed_layout(bits):
    # with one scale and bias everywhere the two layouts hold the same
    # matrix: the [K, N] result equals the [N, K] result on the transposed
    # codes
    rng = np.random.default_rng(90 + bits)
    M, K, N = 3, 128, 192
    q = rng.integers(0, 1 << bits, size=(K, N), dtype=np.uint8)
    x = synth.activations(M, K, seed=91)
    y_kn, b_kn = oracle.qmm_kn(x, synth.pack_codes(q, bits),
                               _bf16_exact(np.full((K, N // 64), 0.125, np.float32)),
                               _bf16_exact(np.full((K, N // 64), -0.5, np.float32)),
                               M, K, N, bits)
    y_nk, b_nk = oracle.qmm(x, synth.pack_codes(np.ascontiguousarray(q.T), bits),
                            _bf16_exact(np.full((N, K // 64), 0.125, np.float32)),
                            _bf16_exact(np.full((N, K // 64), -0.5, np.float32)),
                            M, K, N, bits)
    assert np.array_equal(y_kn, y_nk)
    assert np.array_equal(b_kn, b_nk)


@pytest.mark.parametrize("group", [32, 64])
def test_kn_zero_scale_closed_form(group):
    # s = 0: y[m, n] = sum_k x[m, k] b[k, n/G], exact for integer x
    rng = np.random.default_rng(95)
    M, K, N = 2, 40, 128
    x = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
    bv = (rng.integers(-8, 9, size=(K, N // group)) / 4.0).astype(np.float32)
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    y, _ = oracle.qmm_kn(_bf16_exact(x), synth.pack_codes(q, 4),
                         _bf16_exact(np.zeros((K, N // group), np.float32)), _bf16_exact(bv),
                         M, K, N, 4, group)
    want = x.astype(np.float64) @ np.repeat(bv, group, axis=1).astype(np.float64)
    assert np.array_equal(y, want)


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("group", [32, 64])
def test_kn_brute_force_exact(bits, group):
    M, K, N = 2, 5, 64
    q, w, s_vals, b_vals = _kn_case(K, N, bits, group, 97 + bits)
    s, b = _bf16_exact(s_vals), _bf16_exact(b_vals)
    x = synth.activations(M, K, seed=98)
    y, bnd = oracle.qmm_kn(x, w, s, b, M, K, N, bits, group)
    for n in range(N):
        col = [_row_codes(w[k], N, bits)[n] for k in range(K)]
        for m in range(M):
            exact = sum((_bf16_fraction(x[m, k]) *
                         (_bf16_fraction(s[k, n // group]) * col[k] +
                          _bf16_fraction(b[k, n // group])) for k in range(K)), Fraction(0))
            assert abs(y[m, n] - float(exact)) <= 1e-12 * bnd[m, n] + 1e-300, (m, n)


def test_quantize_writes_golden_stream_words():
    # weights on an exact grid whose codes are known: the encoder's packing of
    # straddling 3- and 6-bit codes must give the hand-packed words
    streams = {(b, tuple(c)): w for b, w, c in _golden_streams()}
    j = np.arange(64)
    # 3-bit: -1 + 0.25 * (j % 8): min -1, range / 7 = 0.25 exactly, codes j % 8
    W3 = (-1.0 + 0.25 * (j % 8)).astype(np.float32)[None, :]
    codes, s, b = oracle.quantize(W3, 3)
    assert s[0, 0] == synth.f32_to_bf16_bits(np.float32(0.25)) and b[0, 0] == 0xBF80
    want = streams[(3, tuple(list(range(8)) * 4))]
    assert list(codes[0, :3]) == want and list(codes[0, 3:6]) == want
    # 6-bit: -1 + 0.0625 * j: range / 63 = 0.0625 exactly, codes j
    W6 = (-1.0 + 0.0625 * j).astype(np.float32)[None, :]
    codes, s, b = oracle.quantize(W6, 6)
    assert s[0, 0] == synth.f32_to_bf16_bits(np.float32(0.0625)) and b[0, 0] == 0xBF80
    assert list(codes[0, :3]) == streams[(6, tuple(range(16)))]
