"""Pins of the fp64 oracle against facts that do not come from the oracle itself: the pages'
structural constants, the OCP MX FP4/E8M0 code tables, hand-worked examples, exact rational
arithmetic, closed forms and brute force on tiny inputs. CPU only."""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for ln in f:
            ln = ln.strip()
            if ln and not ln.startswith("#"):
                yield ln.split()


# ---------------------------------------------------------------------------------------------
# structural constants (Lighthouse 八.3 / 八.7, blog.tulong.co 技术架构创新 1)
# ---------------------------------------------------------------------------------------------
def test_structural_constants_and_entry_counts():
    c = {f[0]: int(f[1]) for f in _lines("structural_constants.txt")}
    assert c["csa_block_m"] == 4 and c["hca_block_m"] == 128 and c["sliding_window"] == 128
    assert math.lcm(c["csa_block_m"], c["hca_block_m"]) == c["cache_block"]
    for N in (2048, 131072, 1048576):
        assert O.entry_count(N, c["csa_block_m"]) == N // 4
        assert O.entry_count(N, c["hca_block_m"]) == N // 128
    # a partial trailing block is not an entry
    assert O.entry_count(131, 4) == 32 and O.entry_count(127, 128) == 0


# ---------------------------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------------------------
def _e2m1_bitfield(code):
    """Independent decode of one e2m1 code from its bit fields (sign, 2-bit exponent with bias
    1, 1-bit mantissa; exponent 0 is subnormal)."""
    s, e, mt = code >> 3, (code >> 1) & 3, code & 1
    mag = Fraction(mt, 2) if e == 0 else Fraction(2) ** (e - 1) * (1 + Fraction(mt, 2))
    return -mag if s else mag


def test_e2m1_table_and_nibble_order():
    table = {}
    for f in _lines("e2m1_codes.txt"):
        if f[0] == "byte":
            b = int(f[1], 16)
            got = O.e2m1_unpack(np.array([b], np.uint8), 2)
            assert list(got) == [float(f[2]), float(f[3])]
        elif f[0] == "scale":
            assert O.ue8m0_to_f64(np.array([int(f[1])]))[0] == float(f[2])
        else:
            table[int(f[0], 16)] = float(f[1])
    assert len(table) == 16
    for code, v in table.items():
        assert float(_e2m1_bitfield(code)) == v
        byte = np.array([code | (code << 4)], np.uint8)
        assert list(O.e2m1_unpack(byte, 2)) == [v, v]
    with pytest.raises(ValueError):
        O.ue8m0_to_f64(np.array([255]))


def _bf16_rne_rational(x: Fraction) -> int:
    """Round a positive rational to bf16 by exhaustive neighbour search: find the two bf16
    values bracketing x and take the nearer, the even mantissa on a tie."""
    assert x >= 0
    if x == 0:
        return 0
    e = math.floor(math.log2(x))
    while Fraction(2) ** e > x:
        e -= 1
    while Fraction(2) ** (e + 1) <= x:
        e += 1
    ulp = Fraction(2) ** (e - 7)
    lo_m = math.floor(x / ulp)           # 128 .. 255
    lo, hi = lo_m * ulp, (lo_m + 1) * ulp
    if x - lo < hi - x or (x - lo == hi - x and lo_m % 2 == 0):
        m, ee = lo_m, e
    else:
        m, ee = lo_m + 1, e
        if m == 256:
            m, ee = 128, e + 1
    return ((ee + 127) << 7) | (m - 128)


def test_bf16_rne_hand_values():
    for f in _lines("bf16_rounding.txt"):
        expr, bits = f[0], int(f[1], 16)
        val = Fraction(eval(expr.replace("^", "**"), {"__builtins__": {}}))  # sums of powers of 2
        got = int(O.f64_to_bf16_rne(np.array([float(val)]))[0])
        assert got == bits, (expr, hex(got))
        assert _bf16_rne_rational(val) == bits
    assert int(O.f64_to_bf16_rne(np.array([-0.0]))[0]) == 0
    assert O.bf16_to_f64(np.array([0x3F80, 0xC000, 0x0001], np.uint16)).tolist() == \
        [1.0, -2.0, 2.0 ** -133]


def test_bf16_rne_against_exact_rounding():
    rng = np.random.default_rng(7)
    bits = rng.integers(0x00800000, 0x7F000000, size=3000, dtype=np.uint32)
    # force many exact ties and near-ties
    bits[:1000] = (bits[:1000] & ~np.uint32(0xFFFF)) | np.uint32(0x8000)
    bits[1000:1500] = (bits[1000:1500] & ~np.uint32(0xFFFF)) | np.uint32(0x7FFF)
    x = bits.view(np.float32).astype(np.float64)
    got = O.f64_to_bf16_rne(x)
    for xi, g in zip(x, got):
        assert int(g) == _bf16_rne_rational(Fraction(float(xi)))


# ---------------------------------------------------------------------------------------------
# pooling (R1, R2)
# ---------------------------------------------------------------------------------------------
def test_pooling_closed_forms():
    rng = np.random.default_rng(1)
    raw = rng.standard_normal((64, 8))
    w = rng.standard_normal(64)
    # m = 1: every entry is its token
    assert np.array_equal(O.compress(raw, w, 1), raw)
    # equal logits: block mean
    np.testing.assert_allclose(O.compress(raw, np.full(64, 0.3), 4),
                               raw.reshape(16, 4, 8).mean(axis=1), rtol=0, atol=1e-15)
    # m = 2: logistic weights
    ent = O.compress(raw, w, 2)
    for j in range(32):
        p0 = 1.0 / (1.0 + math.exp(w[2 * j + 1] - w[2 * j]))
        np.testing.assert_allclose(ent[j], p0 * raw[2 * j] + (1 - p0) * raw[2 * j + 1],
                                   rtol=0, atol=1e-14)
    # weights are positive and sum to one; a constant block pools to the constant
    p = O.pooling_weights(w.reshape(16, 4))
    assert np.all(p > 0) and np.allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-15)
    const = np.tile(np.arange(8.0), (64, 1))
    np.testing.assert_allclose(O.compress(const, w, 8), const[:8], atol=1e-14)
    # partial trailing block dropped
    assert O.compress(raw[:10], w[:10], 4).shape == (2, 8)
    # large logits do not overflow
    big = O.compress(raw[:4], np.array([1000.0, 999.0, -1000.0, 0.0]), 4)
    assert np.all(np.isfinite(big))


# ---------------------------------------------------------------------------------------------
# indexer (R6) and top-k (R7)
# ---------------------------------------------------------------------------------------------
def _pack(bytes_hex, d_I):
    b = [int(x, 16) for x in bytes_hex]
    return np.array(b + [0] * (d_I // 2 - len(b)), np.uint8)


def _worked_example():
    q_codes, q_scales, k_codes, k_scales = [], [], [], []
    scores, topk = {}, {}
    for f in _lines("indexer_worked_example.txt"):
        if f[0] == "qhead":
            q_scales.append([int(f[3])]); q_codes.append(_pack(f[5:], 32))
        elif f[0] == "key":
            k_scales.append([int(f[3])]); k_codes.append(_pack(f[5:], 32))
        elif f[0] == "score":
            scores[int(f[1])] = (float(f[2]), int(f[3], 16))
        elif f[0] == "topk":
            topk[int(f[1])] = [int(x) for x in f[2:]]
    return (np.stack(q_codes), np.array(q_scales, np.uint8), np.stack(k_codes),
            np.array(k_scales, np.uint8), scores, topk)


def test_indexer_worked_example():
    qc, qs, kc, ks, scores, topk = _worked_example()
    s = O.index_scores(qc, qs, kc, ks, 32)
    sb = O.f64_to_bf16_rne(s)
    for j, (v, bits) in scores.items():
        assert s[j] == v and int(sb[j]) == bits
    for k, want in topk.items():
        idx, cnt = O.topk_select(sb, len(s), k)
        assert idx.tolist() == want and cnt == min(k, len(s))


def _brute_index_score(qc, qs, kc, ks, d_I):
    """Exact rational score from the raw nibbles with integer arithmetic only."""
    H = qc.shape[0]
    total = Fraction(0)
    for h in range(H):
        dot = Fraction(0)
        for i in range(d_I):
            qn = (int(qc[h, i // 2]) >> (4 * (i % 2))) & 0xF
            kn = (int(kc[i // 2]) >> (4 * (i % 2))) & 0xF
            sc = Fraction(2) ** (int(qs[h, i // 32]) - 127 + int(ks[i // 32]) - 127)
            dot += _e2m1_bitfield(qn) * _e2m1_bitfield(kn) * sc
        total += max(dot, Fraction(0))
    return total


@pytest.mark.parametrize("d_I,H_I", [(32, 2), (64, 4)])
def test_index_scores_bruteforce(d_I, H_I):
    rng = np.random.default_rng(d_I + H_I)
    E = 24
    qc = rng.integers(0, 256, (H_I, d_I // 2), dtype=np.uint8)
    qs = rng.integers(123, 128, (H_I, d_I // 32), dtype=np.uint8)
    kc = rng.integers(0, 256, (E, d_I // 2), dtype=np.uint8)
    ks = rng.integers(123, 128, (E, d_I // 32), dtype=np.uint8)
    s = O.index_scores(qc, qs, kc, ks, d_I)
    for j in range(E):
        assert Fraction(float(s[j])) == _brute_index_score(qc, qs, kc[j], ks[j], d_I)


def test_index_scores_exact_at_worst_case():
    # all codes +-6 with scale 1: the largest magnitude the configurations allow
    d_I, H_I = 64, 4
    qc = np.full((H_I, d_I // 2), 0x77, np.uint8)
    qs = np.full((H_I, 2), 127, np.uint8)
    kc = np.stack([np.full(d_I // 2, 0x77, np.uint8), np.full(d_I // 2, 0xFF, np.uint8),
                   np.full(d_I // 2, 0x11, np.uint8)])
    ks = np.array([[127, 127], [127, 127], [123, 123]], np.uint8)
    s = O.index_scores(qc, qs, kc, ks, d_I)
    assert s[0] == 4 * 64 * 36 and s[1] == 0.0
    assert s[2] == 4 * 64 * 3 * 2.0 ** -4                      # 6 * 0.5 * 2^-4 per element
    assert int(O.f64_to_bf16_rne(s[:1])[0]) == 0x4610


def _valid_topk(vals, chosen, k):
    """Characterisation of R7 by pairwise comparison (no sorting): every chosen entry beats
    every unchosen one on (score desc, index asc), and the count is min(k, n)."""
    n = len(vals)
    if len(chosen) != min(k, n):
        return False
    rest = [j for j in range(n) if j not in chosen]
    return all(vals[i] > vals[j] or (vals[i] == vals[j] and i < j) for i in chosen for j in rest)


def test_topk_bruteforce_with_ties():
    rng = np.random.default_rng(3)
    for trial in range(300):
        n = int(rng.integers(0, 9))
        k = int(rng.integers(1, 10))
        # few distinct values -> many ties; include 0 (the ReLU floor)
        vals = rng.choice([0.0, 0.5, 1.0, 3.0, 19.5], size=n)
        bits = O.f64_to_bf16_rne(vals) if n else np.zeros(0, np.uint16)
        idx, cnt = O.topk_select(bits, n, k)
        chosen = [int(i) for i in idx[:cnt]]
        assert idx[cnt:].tolist() == [-1] * (k - cnt)
        assert chosen == sorted(chosen)
        assert _valid_topk(vals, set(chosen), k)
        # exactly one subset satisfies the characterisation
        sols = [c for c in itertools.combinations(range(n), min(k, n))
                if _valid_topk(vals, set(c), k)]
        assert sols == [tuple(chosen)]


def test_visibility_rule():
    # R3: entry j visible to t iff (j+1)m-1 <= t
    m, E = 4, 10
    for t in range(0, 50):
        n = O.visible_entries(t, m, E)
        for j in range(E):
            assert (j < n) == ((j + 1) * m - 1 <= t)
    assert O.visible_entries(2, 4, 10) == 0 and O.visible_entries(3, 4, 10) == 1


# ---------------------------------------------------------------------------------------------
# attention (R4, R5, R8, R9) against brute force
# ---------------------------------------------------------------------------------------------
def _brute_attention(q, keys, values):
    """Pure-Python softmax attention of one head."""
    if not keys:
        return [0.0] * len(values[0]) if values else None
    logits = [sum(a * b for a, b in zip(q, k)) for k in keys]
    mx = max(logits)
    ex = [math.exp(l - mx) for l in logits]
    z = sum(ex)
    return [sum(ex[n] * values[n][c] for n in range(len(keys))) / z for c in range(len(values[0]))]


def _rand_seq(rng, N, H, d, d_I=32, H_I=2, m=1):
    bf = lambda a: O.f64_to_bf16_rne(a.astype(np.float32).astype(np.float64))
    q = bf(rng.standard_normal((N, H, d)) / math.sqrt(d))
    k = bf(rng.standard_normal((N, d)))
    v = bf(rng.standard_normal((N, d)))
    w = rng.standard_normal(N)
    E = N // m
    idx = dict(qi_codes=rng.integers(0, 256, (N, H_I, d_I // 2), dtype=np.uint8),
               qi_scales=rng.integers(123, 128, (N, H_I, d_I // 32), dtype=np.uint8),
               ki_codes=rng.integers(0, 256, (E, d_I // 2), dtype=np.uint8),
               ki_scales=rng.integers(123, 128, (E, d_I // 32), dtype=np.uint8))
    return q, k, v, w, idx


def test_csa_reduces_to_causal_attention():
    """I3: with m=1, k >= N and W=0, CSA is ordinary causal attention."""
    rng = np.random.default_rng(11)
    N, H, d = 12, 2, 8
    q, k, v, w, ix = _rand_seq(rng, N, H, d)
    res = O.csa_layer_seq(q, k, v, w, **ix, m=1, W=0, k=N + 3, d_I=32, q_pos0=0)
    qf, kf, vf = O.bf16_to_f64(q), O.bf16_to_f64(k), O.bf16_to_f64(v)
    for t in range(N):
        for h in range(H):
            want = _brute_attention(list(qf[t, h]), [list(kf[u]) for u in range(t + 1)],
                                    [list(vf[u]) for u in range(t + 1)])
            np.testing.assert_allclose(res["out"][t, h], want, rtol=0, atol=1e-12)
        assert res["cnt"][t] == t + 1


def test_window_only_is_sliding_window_attention():
    """With a block longer than the context nothing is visible, and CSA/HCA reduce to
    sliding-window attention over [t-W+1, t]."""
    rng = np.random.default_rng(12)
    N, H, d, W = 20, 2, 8, 5
    q, k, v, w, ix = _rand_seq(rng, N, H, d, m=32)
    res_c = O.csa_layer_seq(q, k, v, w, **ix, m=32, W=W, k=4, d_I=32, q_pos0=0)
    res_h = O.hca_layer_seq(q, k, v, w, m=32, W=W, q_pos0=0)
    qf, kf, vf = O.bf16_to_f64(q), O.bf16_to_f64(k), O.bf16_to_f64(v)
    for t in range(N):
        lo = max(0, t - W + 1)
        for h in range(H):
            want = _brute_attention(list(qf[t, h]), [list(kf[u]) for u in range(lo, t + 1)],
                                    [list(vf[u]) for u in range(lo, t + 1)])
            np.testing.assert_allclose(res_c["out"][t, h], want, rtol=0, atol=1e-12)
            np.testing.assert_allclose(res_h["out"][t, h], want, rtol=0, atol=1e-12)


def test_csa_with_full_k_equals_dense_over_entries():
    """I4: when k covers every visible entry, CSA equals dense (HCA-style) attention over the
    same entries plus window."""
    rng = np.random.default_rng(13)
    N, H, d, m, W = 64, 2, 8, 4, 6
    q, k, v, w, ix = _rand_seq(rng, N, H, d, m=m)
    c = O.csa_layer_seq(q, k, v, w, **ix, m=m, W=W, k=N, d_I=32, q_pos0=0)
    h = O.hca_layer_seq(q, k, v, w, m=m, W=W, q_pos0=0)
    assert np.array_equal(c["out"], h["out"]) and np.array_equal(c["lse"], h["lse"])


def test_entries_and_window_are_not_deduplicated():
    """R5: an entry built from one token (m=1) and the same token in the window both count."""
    q = np.array([[1.0, 0.0]])
    keys_e = np.array([[0.5, 0.0]]); vals_e = np.array([[1.0, 2.0]])
    raw_k = np.array([[0.5, 0.0]]); raw_v = np.array([[1.0, 2.0]])
    out, lse = O.csa_attend_one(q, keys_e, vals_e, [0], 1, raw_k, raw_v, 0, 1)
    np.testing.assert_allclose(lse, [0.5 + math.log(2.0)], rtol=0, atol=1e-15)
    np.testing.assert_allclose(out, [[1.0, 2.0]], atol=1e-15)


def test_softmax_rows_sum_to_one_and_empty_set():
    rng = np.random.default_rng(14)
    q = rng.standard_normal((4, 16)) * 3
    keys = rng.standard_normal((33, 16)) * 3
    p = O.attention_weights(q, keys)
    assert np.all(np.abs(p.sum(axis=1) - 1.0) < 1e-12)
    out, lse = O.attend(q, keys[:0], np.zeros((0, 5)))
    assert np.all(out == 0) and np.all(np.isneginf(lse))
    # lse definition
    _, lse2 = O.attend(q, keys, rng.standard_normal((33, 5)))
    np.testing.assert_allclose(lse2, np.log(np.exp(q @ keys.T).sum(axis=1)), rtol=1e-13)


def test_csa_layer_topk_visible_and_sorted():
    rng = np.random.default_rng(15)
    N, H, d, m, W, k = 64, 2, 8, 4, 4, 5
    q, kk, v, w, ix = _rand_seq(rng, N, H, d, m=m)
    res = O.csa_layer_seq(q, kk, v, w, **ix, m=m, W=W, k=k, d_I=32, q_pos0=0)
    for t in range(N):
        n_vis = O.visible_entries(t, m, N // m)
        cnt = res["cnt"][t]
        assert cnt == min(k, n_vis)
        sel = res["idx"][t][:cnt]
        assert np.all(np.diff(sel) > 0) and (cnt == 0 or sel[-1] < n_vis)
        assert np.all(res["idx"][t][cnt:] == -1)


# ---------------------------------------------------------------------------------------------
# R14: the indexer's own compressed keys, MX FP4 conversion (OCP MX v1.0, section 6.3)
# ---------------------------------------------------------------------------------------------
def _mx_fixture():
    rounds, blocks = [], []
    for line in open(os.path.join(GOLDEN, "mx_fp4_conversion.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        if line.startswith("round "):
            _, y, c = line.split()
            rounds.append((float(y), int(c, 16)))
        else:
            head, _, tail = line.partition("|")
            _, rest, scale, rest_code = head.split()
            vals = [tuple(t.split(":")) for t in tail.split()]
            blocks.append((float(rest), int(scale), int(rest_code, 16),
                           [(float(v), int(c, 16)) for v, c in vals]))
    return rounds, blocks


def test_mx_fp4_element_rounding_worked_values():
    rounds, _ = _mx_fixture()
    y = np.array([r[0] for r in rounds])
    np.testing.assert_array_equal(O.e2m1_round(y), np.array([r[1] for r in rounds], np.uint8))


def test_mx_fp4_block_conversion_worked_examples():
    _, blocks = _mx_fixture()
    for rest, scale, rest_code, vals in blocks:
        x = np.full(32, rest)
        for i, (v, _) in enumerate(vals):
            x[i] = v
        codes, scales = O.mx_fp4_quantize(x[None, :])
        nib = np.stack([codes[0] & 0xF, codes[0] >> 4], axis=-1).reshape(32)
        assert int(scales[0, 0]) == scale, (rest, vals, int(scales[0, 0]))
        want = [c for _, c in vals] + [rest_code] * (32 - len(vals))
        np.testing.assert_array_equal(nib, np.array(want, np.uint8), err_msg=str((rest, vals)))


def test_mx_fp4_every_element_is_a_nearest_grid_point():
    """Property of the conversion for random blocks spanning many binades: every dequantized
    element is a grid point no farther from V/X than any other grid point (saturated elements
    sit at +-6), and the block maximum lands in [4, 8) X, the top binade of the grid."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((400, 64)) * np.ldexp(1.0, rng.integers(-20, 20, (400, 1)))
    x[::7, 3] = 0.0
    codes, scales = O.mx_fp4_quantize(x)
    X = np.repeat(O.ue8m0_to_f64(scales), 32, axis=-1)
    deq = O.mx_fp4_dequant(codes, scales, 64)
    y = x / X
    grid = np.concatenate([-O.E2M1_MAGNITUDES[::-1], O.E2M1_MAGNITUDES])
    d_best = np.abs(y[..., None] - grid).min(axis=-1)
    d_got = np.abs(y - deq / X)
    sat = np.abs(y) > 6.0
    assert np.all(d_got[~sat] <= d_best[~sat])
    assert np.all(np.abs(deq[sat] / X[sat]) == 6.0)
    amax = np.abs(x.reshape(400, 2, 32)).max(axis=-1)
    ratio = amax / O.ue8m0_to_f64(scales)
    assert np.all((ratio >= 4.0) & (ratio < 8.0))


def test_mx_fp4_grid_values_round_trip():
    """Blocks whose values already lie on the e2m1 grid times 2^e, with a maximum of 4 or 6
    times 2^e, convert back to themselves exactly."""
    rng = np.random.default_rng(6)
    for e in (-10, -2, 0, 3):
        vals = O.E2M1_MAGNITUDES[rng.integers(0, 8, (50, 32))] * \
            np.where(rng.random((50, 32)) < 0.5, -1.0, 1.0)
        vals[:, 0] = rng.choice([4.0, 6.0, -6.0], 50)
        x = np.ldexp(vals, e)
        codes, scales = O.mx_fp4_quantize(x)
        assert np.all(scales == 127 + e)
        np.testing.assert_array_equal(O.mx_fp4_dequant(codes, scales, 32), x + 0.0)


def test_bf16_rounding_paths_agree():
    """The direct float64 -> bf16 rounding used for pooled index keys agrees with the fp32-bit
    rounding of the index-score path on every fp32 value, ties included."""
    rng = np.random.default_rng(7)
    f = (rng.integers(0x00800000, 0x7F000000, 20000, dtype=np.uint32)).view(np.float32)
    f = np.concatenate([f, -f, np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 0.0], np.float32)])
    x = f.astype(np.float64)
    np.testing.assert_array_equal(O.f64_to_bf16_rne_any(x), O.f64_to_bf16_rne(x))


def test_index_key_entries_block_one_equals_direct_conversion():
    """With m = 1 every entry is its raw row (the weights of one token are 1), so the compressed
    index keys are the MX FP4 conversion of the raw bf16 rows themselves; with equal logits an
    entry is the block mean."""
    rng = np.random.default_rng(8)
    xi = O.f64_to_bf16_rne_any(rng.standard_normal((12, 64)))
    codes, scales, pb, _ = O.index_key_entries(xi, rng.standard_normal(12), 1)
    c2, s2 = O.mx_fp4_quantize(O.bf16_to_f64(xi))
    np.testing.assert_array_equal(pb, xi)
    np.testing.assert_array_equal(codes, c2)
    np.testing.assert_array_equal(scales, s2)
    _, _, _, pooled = O.index_key_entries(xi, np.zeros(12), 4)
    np.testing.assert_allclose(pooled, O.bf16_to_f64(xi).reshape(3, 4, 64).mean(axis=1),
                               rtol=0, atol=1e-15)


def test_index_key_entries_follow_the_dominant_logit():
    """The pooling weights are a softmax over the block's logits: a token whose logit exceeds
    the others' by 60 takes all the weight (to 1e-26), so its raw row is the pooled key."""
    rng = np.random.default_rng(9)
    xi = O.f64_to_bf16_rne_any(rng.standard_normal((16, 64)))
    logits = np.full(16, -30.0)
    pick = rng.integers(0, 4, 4)
    logits[np.arange(4) * 4 + pick] = 30.0
    codes, scales, pb, pooled = O.index_key_entries(xi, logits, 4)
    np.testing.assert_allclose(pooled, O.bf16_to_f64(xi)[np.arange(4) * 4 + pick], rtol=1e-20,
                               atol=1e-20)
    np.testing.assert_array_equal(pb, xi[np.arange(4) * 4 + pick])


def test_topk_on_real_values_bruteforce():
    """The real-valued selector (FP32 scores) against the characterisation by brute force, with
    signed zeros and values that differ below BF16 resolution; on BF16-representable values it
    agrees with the BF16 selector."""
    rng = np.random.default_rng(4)
    for trial in range(300):
        n = int(rng.integers(0, 9))
        k = int(rng.integers(1, 10))
        vals = rng.choice([0.0, -0.0, 1.0, 1.0 + 2.0 ** -20, 1.0 + 2.0 ** -21, 3.0, -2.0], size=n)
        idx, cnt = O.topk_select_values(vals, n, k)
        chosen = [int(i) for i in idx[:cnt]]
        assert idx[cnt:].tolist() == [-1] * (k - cnt)
        sols = [c for c in itertools.combinations(range(n), min(k, n))
                if _valid_topk(vals + 0.0, set(c), k)]
        assert sols == [tuple(chosen)]
        b = rng.choice([0.0, 0.5, 1.0, 3.0, -1.5], size=n)
        bits = O.f64_to_bf16_rne(b) if n else np.zeros(0, np.uint16)
        i1, c1 = O.topk_select(bits, n, k)
        i2, c2 = O.topk_select_values(b, n, k)
        assert c1 == c2 and np.array_equal(i1, i2)
