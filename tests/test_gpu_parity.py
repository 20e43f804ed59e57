"""Parity of the CUDA path (through the C ABI) with the fp64 oracle on seeded inputs, at sizes
the oracle finishes in seconds that still span several tiles with ragged tails."""
import numpy as np
import pytest
import torch

import long_context_compressed_pooling_b300 as csa
import oracle as O
from synth import LayerShape, generate_layer
from _helpers import (ATT_MAX_ABS, ATT_REL_L2, assert_attention_close, assert_entries_close,
                      assert_lse_close, bits, f64, npy)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _clean_status():
    if torch.cuda.is_available():
        csa.device_status(reset=True)
    yield
    if torch.cuda.is_available():
        assert csa.device_status(reset=True) == 0


def _shape(kind, B, N, Nq, q_pos0, H, d, m, W, k=0, H_I=0, d_I=0, q_scale=None):
    return LayerShape(kind, B=B, N=N, Nq=Nq, q_pos0=q_pos0, H=H, d=d, m=m, W=W, k=k, H_I=H_I,
                      d_I=d_I, q_scale=1.0 / np.sqrt(d) if q_scale is None else q_scale,
                      compress_begin=0)


# ---------------------------------------------------------------------------------------------
# compressor
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("d,m,N", [(64, 4, 1000), (128, 4, 515), (128, 128, 1000), (128, 1, 50),
                                   (256, 16, 300), (128, 8, 4096)])
def test_compress_matches_oracle(d, m, N):
    s = _shape("hca", 2, N, 1, N - 1, 8, d, m, 8)
    x = generate_layer(s, seed=100 + d + m, device=DEV, skip=("q",))
    E = N // m
    kc = torch.full((2, E, d), 7.0, dtype=torch.bfloat16, device=DEV)
    vc = torch.full((2, E, d), 7.0, dtype=torch.bfloat16, device=DEV)
    csa.compress(x["k_raw"], x["v_raw"], x["logits"], m, kc, vc)
    for b in range(2):
        w = npy(x["logits"][b])
        assert_entries_close(bits(kc[b]), O.compress(f64(x["k_raw"][b]), w, m), f"K b={b}")
        assert_entries_close(bits(vc[b]), O.compress(f64(x["v_raw"][b]), w, m), f"V b={b}")


def test_compress_partial_range_touches_only_its_entries():
    d, m, N = 128, 4, 256
    s = _shape("csa", 3, N, 1, N - 1, 8, d, m, 8, k=4, H_I=4, d_I=64)
    x = generate_layer(s, seed=5, device=DEV, skip=("q",))
    E = N // m
    kc = torch.full((3, E, d), 7.0, dtype=torch.bfloat16, device=DEV)
    vc = kc.clone()
    csa.compress(x["k_raw"], x["v_raw"], x["logits"], m, kc, vc, tok_begin=12, tok_end=30)
    # entries 3..6 (tokens 12..27) are written; token 28,29 form no complete block
    touched = np.zeros(E, bool)
    touched[3:7] = True
    for b in range(3):
        ref = O.compress(f64(x["k_raw"][b]), npy(x["logits"][b]), m)
        assert_entries_close(bits(kc[b])[touched], ref[touched])
        assert np.all(f64(kc[b])[~touched] == 7.0)


# ---------------------------------------------------------------------------------------------
# indexer + top-k (bit-exact)
# ---------------------------------------------------------------------------------------------
INDEX_CASES = [
    # B, Nq, q_pos0, N, m, H_I, d_I, k
    (3, 1, 1199, 1200, 4, 4, 64, 16),    # decode, every entry visible, 3 ragged tiles
    (2, 1, 800, 1200, 4, 4, 64, 64),     # decode, partial visibility
    (2, 1, 1199, 1200, 4, 4, 64, 512),   # k above the visible count: padding
    (2, 150, 50, 200, 4, 2, 32, 8),      # prefill, config-1 indexer shape, ragged query groups
    (1, 70, 500, 600, 4, 4, 64, 24),     # prefill chunk, several query groups
    (2, 9, 1500, 2048, 4, 8, 64, 32),    # 8 indexer heads
    (1, 5, 95, 128, 1, 1, 32, 7),        # block size 1, one head
    (1, 12, 60000, 64000, 4, 4, 64, 100),  # prefill, ~120 tiles per CTA: the copy ring wraps
    (4, 1, 1048575, 1048576, 4, 4, 64, 512),  # decode at 1M: ~28 tiles per CTA, ring wraps
    (3, 1, 159999, 160000, 4, 4, 64, 300),  # decode: CTAs span two sequences, ragged tiles
]


@pytest.mark.parametrize("B,Nq,q_pos0,N,m,H_I,d_I,k", INDEX_CASES)
def test_index_scores_and_topk_bitexact(B, Nq, q_pos0, N, m, H_I, d_I, k):
    s = _shape("csa", B, N, Nq, q_pos0, 8, 64, m, 8, k=k, H_I=H_I, d_I=d_I)
    x = generate_layer(s, seed=7 * Nq + k, device=DEV, skip=("q", "k_raw", "v_raw", "logits"))
    E = N // m
    idx, cnt, sc = csa.index_topk(x["qi_codes"], x["qi_scales"], x["ki_codes"], x["ki_scales"],
                                  q_pos0, m, k, want_scores=True)
    idx, cnt, scb = npy(idx), npy(cnt), bits(sc)
    qc, qs, kc, ks = (npy(x[n]) for n in ("qi_codes", "qi_scales", "ki_codes", "ki_scales"))
    for b in range(B):
        for i in range(Nq):
            t = q_pos0 + i
            nv = O.visible_entries(t, m, E)
            ref = O.f64_to_bf16_rne(O.index_scores(qc[b, i], qs[b, i], kc[b, :nv], ks[b, :nv], d_I))
            assert np.array_equal(scb[b, i, :nv], ref), (b, i)
            ridx, rcnt = O.topk_select(ref, nv, k)
            assert cnt[b, i] == rcnt, (b, i)
            assert np.array_equal(idx[b, i], ridx), (b, i)


def _tie_scores(rng, shape):
    vals = np.array([0x0000, 0x8000, 0x3F80, 0x3F81, 0x4040, 0xBF80, 0x419C, 0x0001, 0x7F7F],
                    np.uint16)
    return vals[rng.integers(0, len(vals), size=shape)]


@pytest.mark.parametrize("E,Nq,q_pos0,m,k", [(300, 4, 1196, 4, 50), (64, 3, 100, 1, 64),
                                             (5000, 2, 19999, 4, 700), (60000, 1, 239999, 4, 300),
                                             (1000, 1, 3999, 4, 999),
                                             (6000, 150, 23850, 4, 100),   # one CTA, 2 rounds
                                             (300000, 1, 1199999, 4, 2048),  # cluster of 10
                                             (600000, 1, 2399999, 4, 2048),  # staged chunks
                                             (32768, 1, 131071, 4, 512),     # cluster of 8
                                             (262144, 1, 1048575, 4, 2048),  # cluster of 16
                                             (33001, 1, 132007, 4, 400),     # odd rows, C = 9
                                             (40000, 5, 159000, 4, 300),     # C = 10, 5 rows
                                             (5000, 3, 4094, 1, 40),   # CTAs past the row end
                                             (20000, 300, 79700, 4, 2048)])  # 600 one-CTA rows
def test_topk_ties_and_negative_scores(E, Nq, q_pos0, m, k):
    rng = np.random.default_rng(E + k)
    sc_np = _tie_scores(rng, (2, Nq, E))
    sc = torch.from_numpy(sc_np.view(np.int16)).to(DEV).view(torch.bfloat16)
    idx, cnt = csa.topk(sc, q_pos0, m, k)
    idx, cnt = npy(idx), npy(cnt)
    for b in range(2):
        for i in range(Nq):
            nv = O.visible_entries(q_pos0 + i, m, E)
            ridx, rcnt = O.topk_select(sc_np[b, i], nv, k)
            assert cnt[b, i] == rcnt and np.array_equal(idx[b, i], ridx), (b, i)


@pytest.mark.parametrize("Nq", [150, 300])
@pytest.mark.parametrize("kind", ["spread", "sampled_high", "few_values"])
def test_topk_many_rows_one_cta_each(kind, Nq):
    """Rows of one CTA each, 32768 keys (150 and 300 rows): ordinary scores, the largest scores
    on every 32nd position, and only five distinct values (huge tie groups); top-k lists
    bit-exact."""
    rng = np.random.default_rng({"spread": 1, "sampled_high": 2, "few_values": 3}[kind] + Nq)
    B, E, m, k = 1, 32768, 4, 2048
    q_pos0 = E * m - Nq  # the rows see 32731 .. 32768 entries
    if kind == "spread":
        vals = rng.gamma(4.0, 2.0, size=(B, Nq, E)).astype(np.float32)
    elif kind == "sampled_high":
        vals = rng.uniform(0.0, 1.0, size=(B, Nq, E)).astype(np.float32)
        vals[:, :, ::32] += 100.0  # the positions one thread's first key comes from
    else:
        vals = rng.choice(np.array([0.0, 0.5, 1.0, 2.0, 3.0], np.float32), size=(B, Nq, E))
    sc_np = O.f64_to_bf16_rne(vals.astype(np.float64))
    sc = torch.from_numpy(sc_np.view(np.int16)).to(DEV).view(torch.bfloat16)
    idx, cnt = csa.topk(sc, q_pos0, m, k)
    idx, cnt = npy(idx), npy(cnt)
    for i in range(Nq):
        nv = O.visible_entries(q_pos0 + i, m, E)
        ridx, rcnt = O.topk_select(sc_np[0, i], nv, k)
        assert cnt[0, i] == rcnt and np.array_equal(idx[0, i], ridx), i


# ---------------------------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------------------------
ATT_CASES = [
    # B, Nq, q_pos0, N, H, d, m, W, k
    (2, 5, 251, 256, 64, 128, 4, 16, 8),     # prefill-like rows, 64 heads
    (3, 1, 1023, 1024, 64, 128, 4, 128, 64), # decode: split-K over the key list
    (1, 40, 0, 40, 8, 64, 4, 64, 6),         # config-1 shape from position 0 (early rows empty)
    (2, 3, 700, 703, 16, 64, 4, 5, 100),     # k above visible, short window
    (1, 2, 4000, 4096, 128, 128, 4, 128, 40),  # two head groups
    (16, 1, 4095, 4096, 64, 128, 4, 128, 512),  # decode batch 16: 10-CTA cluster merge
    (1, 1, 32767, 32768, 64, 128, 4, 128, 8192),  # 65 splits: two merge batches per warp
    (1, 1, 32767, 32768, 16, 64, 4, 64, 4096),    # d = 64, workspace merge
    # d = 64 prefill: several query tokens per CTA (64 / Hp of them)
    (2, 37, 900, 1000, 4, 64, 4, 32, 20),    # 16 tokens per CTA, last group partial, 2 sequences
    (1, 9, 2000, 2048, 12, 64, 4, 16, 50),   # 12 heads padded to 16: 4 tokens per CTA
    (1, 2, 4000, 4096, 128, 64, 4, 128, 40),  # two 64-head groups, one token per CTA
    # d = 128 prefill, persistent CTAs (one per SM) walking several tokens each
    (2, 300, 1700, 2000, 64, 128, 4, 100, 300),  # 600 tokens of 4 key chunks, ragged last chunk
    (1, 500, 100, 700, 64, 128, 4, 40, 150),    # 1-2 chunks per token, counts vary by token
    (1, 200, 1000, 1200, 128, 128, 4, 64, 100),  # two head groups: 400 (token, group) items
]


def _run_csa(B, Nq, q_pos0, N, H, d, m, W, k, seed):
    s = _shape("csa", B, N, Nq, q_pos0, H, d, m, W, k=k, H_I=4, d_I=64)
    x = generate_layer(s, seed=seed, device=DEV)
    E = N // m
    kc = torch.empty((B, E, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.empty_like(kc)
    csa.compress(x["k_raw"], x["v_raw"], x["logits"], m, kc, vc)
    idx, cnt, _ = csa.index_topk(x["qi_codes"], x["qi_scales"], x["ki_codes"], x["ki_scales"],
                                 q_pos0, m, k)
    out, lse = csa.csa_attend(x["q"], kc, vc, idx, cnt, x["k_raw"], x["v_raw"], W, q_pos0,
                              want_lse=True)
    return x, kc, vc, idx, cnt, out, lse


@pytest.mark.parametrize("B,Nq,q_pos0,N,H,d,m,W,k", ATT_CASES)
def test_csa_attend_matches_oracle(B, Nq, q_pos0, N, H, d, m, W, k):
    x, kc, vc, idx, cnt, out, lse = _run_csa(B, Nq, q_pos0, N, H, d, m, W, k, seed=N + k)
    qb, kr, vr = bits(x["q"]), bits(x["k_raw"]), bits(x["v_raw"])
    for b in range(B):
        # attention alone, on the GPU's bf16 entries
        kcf, vcf = f64(kc[b]), f64(vc[b])
        for i in range(Nq):
            t = q_pos0 + i
            o, l = O.csa_attend_one(O.bf16_to_f64(qb[b, i]), kcf, vcf, npy(idx[b, i]),
                                    int(cnt[b, i]), O.bf16_to_f64(kr[b]), O.bf16_to_f64(vr[b]),
                                    t, W)
            assert_attention_close(f64(out[b, i]), o, f"b={b} i={i}")
            assert_lse_close(npy(lse[b, i]), l, f"b={b} i={i}")
        # whole layer against the oracle's own fp64 pooling and top-k
        ref = O.csa_layer_seq(qb[b], kr[b], vr[b], npy(x["logits"][b]), npy(x["qi_codes"][b]),
                              npy(x["qi_scales"][b]), npy(x["ki_codes"][b]),
                              npy(x["ki_scales"][b]), m=m, W=W, k=k, d_I=64, q_pos0=q_pos0)
        assert np.array_equal(npy(idx[b]), ref["idx"]) and np.array_equal(npy(cnt[b]), ref["cnt"])
        assert_attention_close(f64(out[b]), ref["out"], f"layer b={b}")


def test_csa_attend_tokens_without_keys_persistent():
    """Persistent CTAs walking tokens of which some have no key (no window, t < 3 sees no
    entry) and most have one to a few: every token's output and log-sum-exp against the oracle
    on the GPU's bf16 entries; keyless tokens give zeros and -inf. (The whole-layer comparison
    with the oracle's fp64 pooling does not apply here: a token with one key outputs that entry,
    so its error is the entry's own bf16 rounding, up to ~2^-9 of values near 3.)"""
    B, Nq, q_pos0, N, H, d, m, W, k = 1, 300, 0, 300, 64, 128, 4, 0, 64
    x, kc, vc, idx, cnt, out, lse = _run_csa(B, Nq, q_pos0, N, H, d, m, W, k, seed=N + k)
    qb, kr, vr = bits(x["q"]), bits(x["k_raw"]), bits(x["v_raw"])
    kcf, vcf = f64(kc[0]), f64(vc[0])
    for i in range(Nq):
        o, l = O.csa_attend_one(O.bf16_to_f64(qb[0, i]), kcf, vcf, npy(idx[0, i]),
                                int(cnt[0, i]), O.bf16_to_f64(kr[0]), O.bf16_to_f64(vr[0]),
                                q_pos0 + i, W)
        assert_attention_close(f64(out[0, i]), o, f"i={i}")
        assert_lse_close(npy(lse[0, i]), l, f"i={i}")
    for i in range(3):
        assert int(cnt[0, i]) == 0
        assert not f64(out[0, i]).any() and np.all(np.isneginf(npy(lse[0, i])))


HCA_CASES = [
    # B, Nq, q_pos0, N, H, d, m, W
    (2, 3, 1021, 1024, 64, 128, 128, 16),
    (3, 1, 8191, 8192, 64, 128, 128, 128),   # decode, split-K over 64 entries + window
    (1, 50, 0, 300, 8, 64, 128, 64),         # config-1 shape: no entry visible for t < 127
    (1, 4, 996, 1000, 64, 64, 4, 0),         # no window at all
    (2, 1, 131071, 131072, 64, 128, 128, 128),  # 9 splits per token: cluster merge
    (1, 1, 262143, 262144, 64, 128, 128, 128),  # 17 splits: workspace merge
    (1, 160, 3840, 4000, 64, 128, 4, 128),   # dense prefill rows: ~9 key chunks per CTA
    (2, 21, 4000, 4200, 4, 64, 128, 128),    # d = 64, 16 tokens per CTA, 2 sequences
    (1, 70, 9000, 9100, 16, 64, 4, 100),     # d = 64, 4 tokens per CTA, ~19 key chunks
    (1, 300, 3700, 4000, 64, 128, 4, 128),   # persistent CTAs: 2-3 tokens of 8-9 chunks each
    (1, 400, 0, 400, 64, 128, 4, 0),         # persistent, no window: early tokens see no key
]


@pytest.mark.parametrize("B,Nq,q_pos0,N,H,d,m,W", HCA_CASES)
def test_hca_attend_matches_oracle(B, Nq, q_pos0, N, H, d, m, W):
    s = _shape("hca", B, N, Nq, q_pos0, H, d, m, W)
    x = generate_layer(s, seed=N + W, device=DEV)
    E = N // m
    kc = torch.empty((B, E, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.empty_like(kc)
    csa.compress(x["k_raw"], x["v_raw"], x["logits"], m, kc, vc)
    out, lse = csa.hca_attend(x["q"], kc, vc, m, x["k_raw"], x["v_raw"], W, q_pos0, want_lse=True)
    qb, kr, vr = bits(x["q"]), bits(x["k_raw"]), bits(x["v_raw"])
    for b in range(B):
        ref = O.hca_layer_seq(qb[b], kr[b], vr[b], npy(x["logits"][b]), m=m, W=W, q_pos0=q_pos0,
                              k_cmp=f64(kc[b]), v_cmp=f64(vc[b]))
        assert_attention_close(f64(out[b]), ref["out"], f"b={b}")
        assert_lse_close(npy(lse[b]), ref["lse"], f"b={b}")
        ref2 = O.hca_layer_seq(qb[b], kr[b], vr[b], npy(x["logits"][b]), m=m, W=W, q_pos0=q_pos0)
        assert_attention_close(f64(out[b]), ref2["out"], f"layer b={b}")


@pytest.mark.parametrize("B,Nq,q_pos0,N,m,W", [(1, 160, 3840, 4000, 4, 128),
                                               (2, 1, 65535, 65536, 128, 128)])
def test_hca_attend_large_logits(B, Nq, q_pos0, N, m, W):
    # Unscaled queries: logits spread over tens of nats, so the running maximum keeps rising
    # across key chunks and the partial outputs are rescaled many times. The softmax is then
    # nearly one-hot and outputs reach |o| ~ 4-5, where one bf16 rounding of the output alone is
    # up to 2^-6 (above the workloads' 1e-2 max-abs bar, which holds for their 1/sqrt(d)-scaled
    # queries), so each element gets 1e-2 plus one bf16 rounding (2^-8 relative) of its value.
    H, d = 64, 128
    s = _shape("hca", B, N, Nq, q_pos0, H, d, m, W, q_scale=1.0)
    x = generate_layer(s, seed=17 + N, device=DEV)
    E = N // m
    kc = torch.empty((B, E, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.empty_like(kc)
    csa.compress(x["k_raw"], x["v_raw"], x["logits"], m, kc, vc)
    out, lse = csa.hca_attend(x["q"], kc, vc, m, x["k_raw"], x["v_raw"], W, q_pos0, want_lse=True)
    qb, kr, vr = bits(x["q"]), bits(x["k_raw"]), bits(x["v_raw"])
    for b in range(B):
        ref = O.hca_layer_seq(qb[b], kr[b], vr[b], npy(x["logits"][b]), m=m, W=W, q_pos0=q_pos0,
                              k_cmp=f64(kc[b]), v_cmp=f64(vc[b]))
        got = f64(out[b])
        err = np.abs(got - ref["out"])
        lim = ATT_MAX_ABS + np.abs(ref["out"]) * 2.0 ** -8
        assert np.all(err <= lim), f"b={b}: worst excess {float(np.max(err - lim)):.3e}"
        rel = np.linalg.norm(got - ref["out"]) / np.linalg.norm(ref["out"])
        assert rel <= ATT_REL_L2, f"b={b}: rel_l2={rel:.3e}"
        assert_lse_close(npy(lse[b]), ref["lse"], f"b={b}")


def test_empty_key_set_gives_zero_and_neg_inf():
    # W = 0 and queries before the first complete block: nothing to attend to
    B, Nq, N, H, d, m = 1, 3, 64, 8, 64, 4
    s = _shape("hca", B, N, Nq, 0, H, d, m, 0)
    x = generate_layer(s, seed=3, device=DEV)
    kc = torch.empty((B, N // m, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.empty_like(kc)
    csa.compress(x["k_raw"], x["v_raw"], x["logits"], m, kc, vc)
    out, lse = csa.hca_attend(x["q"], kc, vc, m, x["k_raw"], x["v_raw"], 0, 0, want_lse=True)
    assert torch.all(out.float() == 0) and torch.all(torch.isneginf(lse))


def test_bad_topk_index_is_flagged_and_skipped_packed_d64():
    # d = 64 prefill (8 tokens per CTA): a bad index of one token is flagged and left out of that
    # token's softmax only
    B, Nq, q_pos0, N, H, d, m, W, k = 1, 5, 251, 256, 8, 64, 4, 8, 4
    x, kc, vc, idx, cnt, out, lse = _run_csa(B, Nq, q_pos0, N, H, d, m, W, k, seed=11)
    bad = idx.clone()
    bad[0, 2, 1] = N // m + 5                     # out of range
    out2, _ = csa.csa_attend(x["q"], kc, vc, bad, cnt, x["k_raw"], x["v_raw"], W, q_pos0)
    flags = csa.device_status(reset=True)
    assert flags & 0x1
    for i in range(Nq):
        sel = npy(idx[0, i])
        if i == 2:
            sel = sel[np.array([0, 2, 3])]
        o, _ = O.csa_attend_one(f64(x["q"][0, i]), f64(kc[0]), f64(vc[0]), sel, len(sel),
                                f64(x["k_raw"][0]), f64(x["v_raw"][0]), q_pos0 + i, W)
        assert_attention_close(f64(out2[0, i]), o, f"i={i}")


def test_bad_topk_index_is_flagged_and_skipped():
    B, Nq, q_pos0, N, H, d, m, W, k = 1, 1, 255, 256, 64, 128, 4, 8, 4
    x, kc, vc, idx, cnt, out, lse = _run_csa(B, Nq, q_pos0, N, H, d, m, W, k, seed=9)
    bad = idx.clone()
    bad[0, 0, 1] = N // m + 5                     # out of range
    out2, _ = csa.csa_attend(x["q"], kc, vc, bad, cnt, x["k_raw"], x["v_raw"], W, q_pos0)
    flags = csa.device_status(reset=True)
    assert flags & 0x1
    keep = np.array([0, 2, 3])
    sel = npy(idx[0, 0])[keep]
    o, _ = O.csa_attend_one(f64(x["q"][0, 0]), f64(kc[0]), f64(vc[0]), sel, len(sel),
                            f64(x["k_raw"][0]), f64(x["v_raw"][0]), q_pos0, W)
    assert_attention_close(f64(out2[0, 0]), o)


# ---------------------------------------------------------------------------------------------
# the layer pair on the tiny prefill workload (full oracle comparison)
# ---------------------------------------------------------------------------------------------
def test_tiny_pair_prefill_full_oracle():
    from synth import get_config
    wl = get_config("tiny_pair_prefill_2k")
    cs, hs = wl.layer("csa"), wl.layer("hca")
    xc = generate_layer(cs, wl.seed, 0, device=DEV)
    xh = generate_layer(hs, wl.seed, 1, device=DEV)
    c = dict(xc, m=cs.m, W=cs.W, k=cs.k, q_pos0=cs.q_pos0, compress_begin=0,
             k_cmp=torch.empty((1, cs.E, cs.d), dtype=torch.bfloat16, device=DEV),
             v_cmp=torch.empty((1, cs.E, cs.d), dtype=torch.bfloat16, device=DEV),
             out=torch.empty_like(xc["q"]), lse=torch.empty((1, cs.Nq, cs.H), device=DEV),
             topk_idx=torch.empty((1, cs.Nq, cs.k), dtype=torch.int32, device=DEV),
             topk_cnt=torch.empty((1, cs.Nq), dtype=torch.int32, device=DEV),
             scores=torch.zeros((1, cs.Nq, cs.E), dtype=torch.bfloat16, device=DEV))
    h = dict(xh, m=hs.m, W=hs.W, q_pos0=hs.q_pos0, compress_begin=0,
             k_cmp=torch.empty((1, hs.E, hs.d), dtype=torch.bfloat16, device=DEV),
             v_cmp=torch.empty((1, hs.E, hs.d), dtype=torch.bfloat16, device=DEV),
             out=torch.empty_like(xh["q"]), lse=torch.empty((1, hs.Nq, hs.H), device=DEV))
    csa.layer_pair(c, h)
    torch.cuda.synchronize()
    rc = O.csa_layer_seq(bits(xc["q"][0]), bits(xc["k_raw"][0]), bits(xc["v_raw"][0]),
                         npy(xc["logits"][0]), npy(xc["qi_codes"][0]), npy(xc["qi_scales"][0]),
                         npy(xc["ki_codes"][0]), npy(xc["ki_scales"][0]), m=cs.m, W=cs.W, k=cs.k,
                         d_I=cs.d_I, q_pos0=0)
    assert np.array_equal(npy(c["topk_idx"][0]), rc["idx"])
    assert np.array_equal(npy(c["topk_cnt"][0]), rc["cnt"])
    scb = bits(c["scores"][0])
    for i, sref in enumerate(rc["scores"]):
        assert np.array_equal(scb[i, :len(sref)], sref), i
    assert_attention_close(f64(c["out"][0]), rc["out"], "csa")
    assert_lse_close(npy(c["lse"][0]), rc["lse"], "csa lse")
    rh = O.hca_layer_seq(bits(xh["q"][0]), bits(xh["k_raw"][0]), bits(xh["v_raw"][0]),
                         npy(xh["logits"][0]), m=hs.m, W=hs.W, q_pos0=0)
    assert_attention_close(f64(h["out"][0]), rh["out"], "hca")
    assert_lse_close(npy(h["lse"][0]), rh["lse"], "hca lse")
