"""FP32 index scores and the selector over them (the selection the BF16 scores replace), against
the fp64 oracle: the FP32 scores are exact, so they and the selection are compared bit for bit."""
import numpy as np
import pytest
import torch

import long_context_compressed_pooling_b300 as csa
import oracle as O
from synth import LayerShape, generate_layer
from _helpers import bits, npy

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _clean_status():
    if torch.cuda.is_available():
        csa.device_status(reset=True)
    yield
    if torch.cuda.is_available():
        assert csa.device_status(reset=True) == 0


@pytest.mark.parametrize("B,Nq,q_pos0,N,m,H_I,d_I,k", [
    (3, 1, 1199, 1200, 4, 4, 64, 16),       # decode, ragged tiles
    (1, 70, 500, 600, 4, 4, 64, 24),        # prefill rows, partial visibility
    (2, 9, 1500, 2048, 4, 8, 64, 32),       # 8 indexer heads
    (2, 150, 50, 200, 4, 2, 32, 8),         # d_I = 32
    (2, 1, 131071, 131072, 4, 4, 64, 512),  # decode at 128K: cluster rows
])
def test_fp32_scores_and_selection_match_oracle(B, Nq, q_pos0, N, m, H_I, d_I, k):
    s = LayerShape("csa", B=B, N=N, Nq=Nq, q_pos0=q_pos0, H=8, d=64, m=m, W=8, k=k, H_I=H_I,
                   d_I=d_I, q_scale=0.125, compress_begin=0)
    x = generate_layer(s, seed=N + Nq, device=DEV, skip=("q", "k_raw", "v_raw", "logits"))
    sb, sf = csa.index_scores(x["qi_codes"], x["qi_scales"], x["ki_codes"], x["ki_scales"],
                              q_pos0, m)
    idx, cnt = csa.topk_f32(sf, q_pos0, m, k)
    idx_b, cnt_b = csa.topk(sb, q_pos0, m, k)
    sbn, sfn, idn, cn = bits(sb), npy(sf), npy(idx), npy(cnt)
    qc, qs, kc, ks = (npy(x[n]) for n in ("qi_codes", "qi_scales", "ki_codes", "ki_scales"))
    E = N // m
    for b in range(B):
        for i in range(Nq):
            nv = O.visible_entries(q_pos0 + i, m, E)
            ref = O.index_scores(qc[b, i], qs[b, i], kc[b, :nv], ks[b, :nv], d_I)
            np.testing.assert_array_equal(sfn[b, i, :nv].astype(np.float64), ref, err_msg=str((b, i)))
            assert np.all(sfn[b, i, nv:] == 0)                  # invisible entries untouched
            np.testing.assert_array_equal(sbn[b, i, :nv], O.f64_to_bf16_rne(ref))
            ridx, rcnt = O.topk_select_values(ref, nv, k)
            assert cn[b, i] == rcnt and np.array_equal(idn[b, i], ridx), (b, i)
    # the BF16 selection on the same call's BF16 scores is the csa_topk one
    i2, c2, _ = csa.index_topk(x["qi_codes"], x["qi_scales"], x["ki_codes"], x["ki_scales"],
                               q_pos0, m, k)
    assert torch.equal(i2, idx_b) and torch.equal(c2, cnt_b)


def _tie_values(rng, shape):
    """Few distinct FP32 values, several of them sharing their upper 16 bits (the BF16-truncated
    part) and differing below it, plus signed zeros and negatives."""
    vals = np.array([0.0, -0.0, 1.0, 1.0 + 2 ** -20, 1.0 + 2 ** -22, 1.0 + 2 ** -10,
                     3.0, 3.0 + 2 ** -18, -1.5, 1e-30, 7.5], np.float32)
    return vals[rng.integers(0, len(vals), size=shape)]


@pytest.mark.parametrize("E,Nq,q_pos0,m,k", [
    (300, 4, 1196, 4, 50),          # one CTA per row, ties at the threshold
    (6000, 150, 23850, 4, 100),     # 150 rows: one 1024-thread CTA each
    (32768, 1, 131071, 4, 512),     # cluster of 8
    (262144, 1, 1048575, 4, 2048),  # cluster of 16
    (300000, 1, 1199999, 4, 2048),  # cluster of 10, 1024 x 32 keys per CTA
    (33001, 1, 132007, 4, 400),     # odd row length: unaligned rows load key by key
    (5000, 3, 4094, 1, 40),         # CTAs past the row end
    (1000, 2, 3999, 4, 999),        # k close to the row length
])
def test_topk_f32_ties_and_signed_values(E, Nq, q_pos0, m, k):
    rng = np.random.default_rng(E + k)
    sc = _tie_values(rng, (2, Nq, E))
    idx, cnt = csa.topk_f32(torch.from_numpy(sc).to(DEV), q_pos0, m, k)
    idx, cnt = npy(idx), npy(cnt)
    for b in range(2):
        for i in range(Nq):
            nv = O.visible_entries(q_pos0 + i, m, E)
            ridx, rcnt = O.topk_select_values(sc[b, i].astype(np.float64), nv, k)
            assert cnt[b, i] == rcnt and np.array_equal(idx[b, i], ridx), (b, i)


def test_topk_f32_wide_spread_takes_the_radix_path():
    """Scores spread over many octaves, so the k-th largest lies far below the maximum (the
    near-max band of the coarse keys holds fewer than k): the exact radix select decides."""
    rng = np.random.default_rng(1)
    sc = (rng.standard_normal((3, 2, 20000)) * np.exp2(rng.integers(-40, 40, (3, 2, 20000))))
    sc = sc.astype(np.float32)
    idx, cnt = csa.topk_f32(torch.from_numpy(sc).to(DEV), 79999, 4, 3000)
    idx = npy(idx)
    for b in range(3):
        for i in range(2):
            ridx, _ = O.topk_select_values(sc[b, i].astype(np.float64), 20000, 3000)
            assert np.array_equal(idx[b, i], ridx), (b, i)
