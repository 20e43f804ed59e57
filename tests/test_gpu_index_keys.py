"""Parity of the indexer's own compressed keys and of the MX FP4 query conversion (through the C
ABI) with the fp64 oracle.

The conversion from bf16 values is integer work and is compared bit for bit. The pooled index
key is rounded to bf16 from the kernel's fp32 sum and from the oracle's fp64 sum; the two can
differ where the exact pooled value lies within the fp32 error of a bf16 rounding boundary. The
kernel's fp32 error is bounded by its arithmetic (IEEE division, expf within 2 ulp), to first
order in u = 2^-24, with A the largest distance of a block's logit from its maximum and
L = ceil(log2 m):
  - e_i = expf(fl(w_i - max)): the rounded argument gives A u, expf's 2 ulp 4 u (relative);
  - the sum of the m weights over a shuffle tree: every weight passes at most L roundings
    (partners beyond the m lanes add exact zeros), so the sum carries (4 + A + L) u;
  - the reciprocal and the product e_i * (1 / sum): 2 u; each p_i is within (10 + 2A + L) u;
  - the m fused multiply-adds of sum_i p_i x_i: m u of sum_i p_i |x_i|.
In all |kernel - exact| <= (m + L + 10 + 2A) u sum_i p_i |x_i|; the test allows one u more for
the second-order terms. An element whose exact value +- that bound rounds to another bf16 value
is ambiguous. Every other element must match exactly: a block without an ambiguous
element is compared bit for bit, and a block with one must equal the conversion of some
admissible choice of its ambiguous elements, the rest fixed. The tests also require ambiguous
elements to stay rare (a few percent), so the comparison is exact almost everywhere."""
import itertools

import numpy as np
import pytest
import torch

import long_context_compressed_pooling_b300 as csa
import oracle as O
from synth import LayerShape, generate_layer, index_key_rows
from _helpers import bits, npy

pytestmark = pytest.mark.gpu
DEV = "cuda"
U = 2.0 ** -24


@pytest.fixture(autouse=True)
def _clean_status():
    if torch.cuda.is_available():
        csa.device_status(reset=True)
    yield
    if torch.cuda.is_available():
        assert csa.device_status(reset=True) == 0


def _nibbles(codes):
    c = np.asarray(codes, np.uint8)
    return np.stack([c & 0xF, c >> 4], axis=-1).reshape(c.shape[:-1] + (2 * c.shape[-1],))


# ---------------------------------------------------------------------------------------------
# MX FP4 conversion of bf16 rows (bit-exact)
# ---------------------------------------------------------------------------------------------
def _special_rows(d, rng):
    """Rows that exercise the rule's edges: zero blocks, -0, bf16 subnormals, huge values,
    values exactly on rounding midpoints, maxima on powers of two, saturation."""
    rows = []
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    for e in (-130, -20, -3, 0, 7, 100):
        for top in (4.0, 6.0, 5.0, 7.75):
            r = np.ldexp(rng.choice(np.concatenate([mids, -mids, O.E2M1_MAGNITUDES]), d), e)
            r[::32] = np.ldexp(top, e)  # the block maximum
            rows.append(r)
    z = np.zeros(d)
    z[1::2] = -0.0
    rows.append(z)
    tiny = np.full(d, 2.0 ** -133)
    tiny[5] = -(2.0 ** -130)
    rows.append(tiny)
    rows.append(np.full(d, 3.0e38))
    return np.stack(rows)


@pytest.mark.parametrize("d", [32, 64, 128])
def test_quantize_mxfp4_bitexact(d):
    rng = np.random.default_rng(d)
    gauss = rng.standard_normal((3000, d)) * np.ldexp(1.0, rng.integers(-30, 30, (3000, 1)))
    # the special rows keep their signed zeros and bf16 subnormals: their bit patterns are the
    # upper halves of the fp32 values (truncation is fine, they are only inputs)
    f32 = _special_rows(d, rng).astype(np.float32)
    xb = np.concatenate([O.f64_to_bf16_rne_any(gauss),
                         (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)])
    x = torch.from_numpy(xb.view(np.int16)).to(DEV).view(torch.bfloat16).reshape(-1, d)
    codes, scales = csa.quantize_mxfp4(x)
    ref_c, ref_s = O.mx_fp4_quantize(O.bf16_to_f64(xb))
    np.testing.assert_array_equal(npy(scales), ref_s)
    np.testing.assert_array_equal(npy(codes), ref_c)


def test_quantize_mxfp4_query_layout():
    """Index queries [B, Nq, H_I, d_I] convert row by row into the indexer's input layout."""
    s = LayerShape("csa", B=2, N=64, Nq=5, q_pos0=59, H=8, d=64, m=4, W=8, k=4, H_I=4, d_I=64,
                   q_scale=0.125, compress_begin=0)
    x = generate_layer(s, seed=3, device=DEV)["q"][..., :64].contiguous()  # any bf16 rows
    codes, scales = csa.quantize_mxfp4(x)
    assert codes.shape == (2, 5, 8, 32) and scales.shape == (2, 5, 8, 2)
    ref_c, ref_s = O.mx_fp4_quantize(O.bf16_to_f64(bits(x)))
    np.testing.assert_array_equal(npy(codes), ref_c)
    np.testing.assert_array_equal(npy(scales), ref_s)


# ---------------------------------------------------------------------------------------------
# pooled index keys (bit-exact outside the fp32 ambiguity of the bf16 rounding)
# ---------------------------------------------------------------------------------------------
def _check_seq_keys(codes_g, scales_g, xi_bits, logits, m, j0, j1, what):
    """Compares entries [j0, j1) of one sequence; returns the number of ambiguous elements."""
    codes_o, scales_o, pb_o, pooled = O.index_key_entries(xi_bits, logits, m)
    E, d = pooled.shape
    w = np.asarray(logits, np.float64)[: E * m].reshape(E, m)
    a = np.abs(w - w.max(axis=1, keepdims=True)).max(axis=1)
    p = O.pooling_weights(w)
    mag = np.einsum("ji,jid->jd", p, np.abs(O.bf16_to_f64(xi_bits)[: E * m].reshape(E, m, d)))
    L = int(np.ceil(np.log2(m))) if m > 1 else 0
    delta = ((m + L + 11 + 2 * a) * U)[:, None] * mag
    lo = O.f64_to_bf16_rne_any(pooled - delta)
    hi = O.f64_to_bf16_rne_any(pooled + delta)
    amb = (lo != pb_o) | (hi != pb_o)                      # [E, d]
    ng, no = _nibbles(codes_g), _nibbles(codes_o)
    n_amb = 0
    for j in range(j0, j1):
        for blk in range(d // 32):
            sl = slice(32 * blk, 32 * blk + 32)
            got = (int(scales_g[j, blk]), tuple(ng[j, sl]))
            if not amb[j, sl].any():
                assert got == (int(scales_o[j, blk]), tuple(no[j, sl])), f"{what} entry {j} block {blk}"
                continue
            pos = np.nonzero(amb[j, sl])[0]
            n_amb += len(pos)
            assert len(pos) <= 10, f"{what}: too many ambiguous elements in entry {j}"
            choices = [sorted({int(lo[j, 32 * blk + i]), int(pb_o[j, 32 * blk + i]),
                               int(hi[j, 32 * blk + i])}) for i in pos]
            ok = False
            for combo in itertools.product(*choices):
                vb = pb_o[j, sl].copy()
                vb[pos] = combo
                c, sc = O.mx_fp4_quantize(O.bf16_to_f64(vb)[None, :])
                if got == (int(sc[0, 0]), tuple(_nibbles(c)[0])):
                    ok = True
                    break
            assert ok, f"{what} entry {j} block {blk}: no admissible rounding gives the kernel's codes"
    return n_amb


@pytest.mark.parametrize("B,N,d_I,m,tok_begin", [
    (2, 1000, 64, 4, 0),      # 250 entries, several warps per CTA, grid-stride
    (1, 4096, 128, 4, 1024),  # entries from 256 on only: the rest must stay untouched
    (3, 302, 32, 4, 0),       # d_I = 32 (one element per lane), ragged trailing block
    (1, 512, 64, 1, 0),       # m = 1: the keys are the raw rows converted
    (2, 640, 64, 32, 64),     # m = 32: one lane per token
    (1, 97, 128, 8, 0),       # 12 entries
])
def test_compress_index_keys_matches_oracle(B, N, d_I, m, tok_begin):
    s = LayerShape("csa", B=B, N=N, Nq=1, q_pos0=N - 1, H=8, d=64, m=m, W=8, k=4, H_I=4,
                   d_I=d_I, q_scale=0.125, compress_begin=tok_begin)
    xi = index_key_rows(s, seed=N + m, device=DEV)
    logits = generate_layer(s, seed=N + m, device=DEV, skip=("q", "k_raw", "v_raw"))["logits"]
    E = N // m
    kc = torch.full((B, E, d_I // 2), 0x5A, dtype=torch.uint8, device=DEV)
    ks = torch.full((B, E, d_I // 32), 0xA5, dtype=torch.uint8, device=DEV)
    csa.compress_index_keys(xi, logits, m, kc, ks, tok_begin=tok_begin)
    kcn, ksn = npy(kc), npy(ks)
    j0 = tok_begin // m
    assert np.all(kcn[:, :j0] == 0x5A) and np.all(ksn[:, :j0] == 0xA5)
    n_amb = 0
    for b in range(B):
        n_amb += _check_seq_keys(kcn[b], ksn[b], bits(xi[b]), npy(logits[b]), m, j0, E,
                                 f"b={b}")
    assert n_amb <= 0.05 * B * (E - j0) * d_I, n_amb


def test_layer_pair_writes_the_chunk_index_keys():
    """A prefill chunk whose layer call pools its own index keys: the cached prefix keys come
    from a standalone call, the layer writes the chunk's entries (poisoned before), and the
    result equals the standalone conversion of the whole sequence; the layer's top-k equals
    the standalone indexer's top-k on those keys; the keys match the oracle."""
    B, N, Nq, m, k, W, d_I = 1, 4096, 256, 4, 64, 32, 64
    q0 = N - Nq
    s = LayerShape("csa", B=B, N=N, Nq=Nq, q_pos0=q0, H=64, d=128, m=m, W=W, k=k, H_I=4,
                   d_I=d_I, q_scale=1.0 / np.sqrt(128), compress_begin=q0)
    x = generate_layer(s, seed=11, device=DEV)
    xi = index_key_rows(s, seed=11, device=DEV)
    E = N // m
    full_c, full_s = csa.compress_index_keys(xi, x["logits"], m)
    kc, ks = full_c.clone(), full_s.clone()
    kc[:, q0 // m:] = 0x77
    ks[:, q0 // m:] = 0x33
    k_cmp = torch.empty((B, E, 128), dtype=torch.bfloat16, device=DEV)
    v_cmp = torch.empty_like(k_cmp)
    csa.compress(x["k_raw"], x["v_raw"], x["logits"], m, k_cmp, v_cmp, tok_end=q0)
    out = torch.empty_like(x["q"])
    idx = torch.empty((B, Nq, k), dtype=torch.int32, device=DEV)
    cnt = torch.empty((B, Nq), dtype=torch.int32, device=DEV)
    layer = dict(q=x["q"], k_raw=x["k_raw"], v_raw=x["v_raw"], logits=x["logits"],
                 qi_codes=x["qi_codes"], qi_scales=x["qi_scales"], ki_codes=kc, ki_scales=ks,
                 k_cmp=k_cmp, v_cmp=v_cmp, out=out, topk_idx=idx, topk_cnt=cnt, xi_raw=xi,
                 m=m, W=W, k=k, q_pos0=q0, compress_begin=q0)
    csa.layer_pair(layer, None)
    torch.cuda.synchronize()
    assert torch.equal(kc, full_c) and torch.equal(ks, full_s)
    i2, c2, _ = csa.index_topk(x["qi_codes"], x["qi_scales"], kc, ks, q0, m, k)
    assert torch.equal(i2, idx) and torch.equal(c2, cnt)
    n_amb = _check_seq_keys(npy(kc[0]), npy(ks[0]), bits(xi[0]), npy(x["logits"][0]), m, 0, E,
                            "layer pair")
    assert n_amb <= 0.05 * E * d_I


@pytest.mark.parametrize("B,N,Nq", [(2, 65536, 2048), (16, 131072, 1)])
def test_layer_pair_scores_the_keys_it_just_pooled(B, N, Nq):
    """The layer pools the index keys of its new blocks in one launch and scores them in the
    next, which may start before the pooling has finished: the key tiles the pooling writes must
    be read only after it completes. The new keys are poisoned (tiny scales) before every one of
    several repeated calls; a call that scored a poisoned key would select differently from the
    standalone indexer run afterwards on the finished keys."""
    m, k, W, d_I = 4, 256, 128, 64
    q0 = N - Nq
    cb = (q0 // m) * m if Nq > 1 else N - m
    s = LayerShape("csa", B=B, N=N, Nq=Nq, q_pos0=q0, H=64, d=128, m=m, W=W, k=k, H_I=4,
                   d_I=d_I, q_scale=1.0 / np.sqrt(128), compress_begin=cb)
    x = generate_layer(s, seed=23 + Nq, device=DEV)
    xi = index_key_rows(s, seed=23 + Nq, device=DEV)
    E = N // m
    j0 = cb // m
    full_c, full_s = csa.compress_index_keys(xi, x["logits"], m)
    kc, ks = full_c.clone(), full_s.clone()
    k_cmp = torch.empty((B, E, 128), dtype=torch.bfloat16, device=DEV)
    v_cmp = torch.empty_like(k_cmp)
    csa.compress(x["k_raw"], x["v_raw"], x["logits"], m, k_cmp, v_cmp, tok_end=cb)
    out = torch.empty_like(x["q"])
    idx = torch.empty((B, Nq, k), dtype=torch.int32, device=DEV)
    cnt = torch.empty((B, Nq), dtype=torch.int32, device=DEV)
    layer = dict(q=x["q"], k_raw=x["k_raw"], v_raw=x["v_raw"], logits=x["logits"],
                 qi_codes=x["qi_codes"], qi_scales=x["qi_scales"], ki_codes=kc, ki_scales=ks,
                 k_cmp=k_cmp, v_cmp=v_cmp, out=out, topk_idx=idx, topk_cnt=cnt, xi_raw=xi,
                 m=m, W=W, k=k, q_pos0=q0, compress_begin=cb)
    ref_i, ref_c, _ = csa.index_topk(x["qi_codes"], x["qi_scales"], full_c, full_s, q0, m, k)
    step = csa.PreparedLayerPair(layer, None)
    for rep in range(6):
        kc[:, j0:] = 0x77
        ks[:, j0:] = 0x01
        step()
        torch.cuda.synchronize()
        assert torch.equal(kc, full_c) and torch.equal(ks, full_s), rep
        assert torch.equal(idx, ref_i) and torch.equal(cnt, ref_c), rep
